"""The workspace-free decode entry point (mla_sparse_decode_static_ws).

It serves callers that cannot allocate device memory: its scratch is a fixed
array inside the library.  These tests call it through the C ABI and check
that it returns, bit for bit, what mla_sparse_decode (caller-supplied
workspace) returns, and that both agree with the float64 oracle, on two calls
in a row, so that what one call leaves in the shared array cannot leak into
the next.  The file is named to be collected last."""
import ctypes

import pytest
import torch

from sparse_latent_attention_decode_b300 import synth
from tests import parity_util as U

if torch.cuda.is_available():
    from sparse_latent_attention_decode_b300 import mla


def _q_lat(d):
    cis = mla.rope_freqs_init()
    return mla.mla_absorb_q(d["q_nope"], d["q_pe"], cis, d["end_pos"], d["wkv_b"])


@pytest.mark.gpu
@pytest.mark.parametrize("with_wkv_b", [True, False], ids=["head_outputs", "latent_o"])
def test_static_workspace_matches_caller_workspace_on_two_calls(with_wkv_b):
    scale = mla.softmax_scale()
    # first call: 3 sequences in one unit each; second call: one sequence whose
    # selection is split over several units (partials live in the scratch)
    cases = [dict(B=3, ep=[700, 513, 260], k=256, K=300, S=704, seed=21),
             dict(B=1, ep=[1001], k=1001, K=1001, S=1024, seed=22)]
    for c in cases:
        t = synth.make_inputs(synth.small_workload(c["B"], c["ep"], k=c["k"], K=c["K"], S_cap=c["S"]),
                              seed=c["seed"])
        d = {n: v.cuda() for n, v in t.items()}
        q_lat = _q_lat(d)
        w = d["wkv_b"] if with_wkv_b else None
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        ref = mla.mla_sparse_decode(q_lat, d["kv_cache"], d["pe_cache"], d["topk_idx"], d["end_pos"], scale,
                                    wkv_b=w)
        got = mla.mla_sparse_decode_static_ws(q_lat, d["kv_cache"], d["pe_cache"], d["topk_idx"], d["end_pos"],
                                              scale, wkv_b=w, dev_status=st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        # the same kernels on the same inputs: bit-identical to the caller-workspace call
        assert torch.equal(got, ref), "static workspace differs from caller workspace"
        # and, independently, within the tolerance of the float64 oracle
        x = U.oracle_inputs(t)
        bs = list(range(c["B"]))
        ora = U.oracle_out(x, bs) if with_wkv_b else U.oracle_o_lat(x, bs, q_lat=synth.to_f64(q_lat.cpu()))
        U.assert_attn_close(got.cpu().numpy(), ora, "static workspace vs oracle")


def test_static_workspace_rejects_sizes_beyond_its_capacity():
    from sparse_latent_attention_decode_b300 import mla as binding
    lib = binding._lib
    need = lib.mla_sparse_decode_workspace_size(4096, 2048)
    assert need > (32 << 20)
    p = ctypes.c_void_p(0x10000)   # never dereferenced: the size check fails first
    rc = lib.mla_sparse_decode_static_ws(p, p, p, 16, p, 2048, p, 4096, 1.0, p, p, None, None)
    assert rc == -3
