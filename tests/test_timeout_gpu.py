"""Failure detection on the GPU without a fault: every on-chip wait of the
kernels is bounded, and a kernel whose wait runs out reports MLA_DEV_TIMEOUT,
drains the copies and MMAs it has already issued, releases its tensor memory
and returns.  These tests shorten the limit (mla_set_wait_limit_ns) so that
waits run out, check the status bit and that the call returns, and then check
that the next call with the normal limit is correct."""
import numpy as np
import pytest
import torch

from oracle import mla_oracle as O
from sparse_latent_attention_decode_b300 import synth
from tests import parity_util as U

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from sparse_latent_attention_decode_b300 import mla


class _ShortWaits:
    """Every kernel launched inside polls its waits without suspending and
    gives up after a few microseconds."""

    def __enter__(self):
        self.prev = mla.set_wait_limit_ns(1)
        return self

    def __exit__(self, *exc):
        mla.set_wait_limit_ns(self.prev)
        return False


def _status():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


def test_limit_setting_round_trips():
    prev = mla.set_wait_limit_ns(12345)
    try:
        assert mla.set_wait_limit_ns(prev) == 12345
    finally:
        mla.set_wait_limit_ns(prev)
    assert prev == 2_000_000_000


def test_projection_wait_runs_out_then_next_call_is_correct():
    M, N, K = 64, 7168, 16384                       # the wo shape: a long weight stream per CTA
    x, w = synth.make_linear_inputs(101, M, N, K)
    dx, dw = x.cuda(), w.cuda()
    st = _status()
    with _ShortWaits():
        mla.mla_linear_bf16(dx, dw, dev_status=st)
        torch.cuda.synchronize()                    # the call returns
    assert int(st.item()) & mla.MLA_DEV_TIMEOUT
    st2 = _status()
    y = mla.mla_linear_bf16(dx, dw, dev_status=st2)
    torch.cuda.synchronize()
    assert int(st2.item()) == 0
    cols = np.random.default_rng(1).choice(N, 256, replace=False)
    xd, wd = synth.to_f64(x), synth.to_f64(w)[cols]
    ref = O.linear(xd, wd)
    mag = O.linear(np.abs(xd), np.abs(wd))
    assert np.all(np.abs(y.cpu().double().numpy()[:, cols] - ref) <= 2e-6 * mag)


def test_absorption_wait_runs_out_then_next_call_is_correct():
    B = 64
    t = synth.make_inputs(synth.small_workload(B, [4096] * B, k=1, K=1, S_cap=4096), seed=103)
    d = {k: v.cuda() for k, v in t.items()}
    cis = mla.rope_freqs_init()
    st = _status()
    with _ShortWaits():
        mla.mla_absorb_q(d["q_nope"], d["q_pe"], cis, d["end_pos"], d["wkv_b"], dev_status=st)
        torch.cuda.synchronize()
    assert int(st.item()) & mla.MLA_DEV_TIMEOUT
    st2 = _status()
    q_lat = mla.mla_absorb_q(d["q_nope"], d["q_pe"], cis, d["end_pos"], d["wkv_b"], dev_status=st2)
    torch.cuda.synchronize()
    assert int(st2.item()) == 0
    x = U.oracle_inputs(t)
    U.assert_attn_close(synth.to_f64(q_lat.cpu()), U.oracle_q_lat(x, list(range(B))), "absorb after timeout")


def test_decode_step_wait_runs_out_then_next_step_is_correct():
    # absorption, the two-CTA attention kernel (gather, DSMEM exchange, MMAs)
    # and the up-projection, all with waits that run out
    B, K = 8, 1024
    t = synth.make_inputs(synth.small_workload(B, [2048] * B, k=K, K=K, S_cap=2048), seed=105)
    d = {k: v.cuda() for k, v in t.items()}
    args = (d["q_nope"], d["q_pe"], d["kv_cache"], d["pe_cache"], d["wkv_b"], d["topk_idx"], d["end_pos"])
    step = mla.DecodeStep(B, K)
    with _ShortWaits():
        step(*args)
        torch.cuda.synchronize()
    assert int(step.status.item()) & mla.MLA_DEV_TIMEOUT
    step.status.zero_()
    out = step(*args)
    torch.cuda.synchronize()
    step.check_status()
    x = U.oracle_inputs(t)
    U.assert_attn_close(out.cpu().numpy(), U.oracle_out(x, list(range(B))), "step after timeout")
