"""GPU parity: every entry point of the C ABI against the float64 oracle on
identical seeded inputs.  Needs a B300 (sm_103a)."""
import numpy as np
import pytest
import torch

from oracle import mla_oracle as O
from sparse_latent_attention_decode_b300 import synth
from tests import parity_util as U

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from sparse_latent_attention_decode_b300 import mla


def _dev(t):
    return {k: v.cuda() for k, v in t.items()}


class _PerSeq:
    """Widen one sequence of a large host tensor to float64 on demand."""

    def __init__(self, t):
        self.t = t

    def __getitem__(self, b):
        return synth.to_f64(self.t[b])


def _oracle_view(t):
    x = {k: synth.to_f64(v) for k, v in t.items() if k not in ("kv_cache", "pe_cache")}
    x["kv_cache"] = _PerSeq(t["kv_cache"])
    x["pe_cache"] = _PerSeq(t["pe_cache"])
    return x


# ----------------------------------------------------------------- RoPE
def test_rope_table_matches_oracle():
    cis = mla.rope_freqs_init().cpu().double().numpy()
    ora = O.freqs_cis(np.arange(16384), U.INV_FREQ)
    assert np.abs(cis[..., 0] - ora.real).max() <= 2e-7
    assert np.abs(cis[..., 1] - ora.imag).max() <= 2e-7


def test_rope_table_without_yarn_and_short_table():
    p = mla.rope_params(max_seq_len=4096)
    cis = mla.rope_freqs_init(p).cpu().double().numpy()
    ora = O.freqs_cis(np.arange(4096), O.yarn_inv_freq(max_seq_len=4096))
    assert np.abs(cis[..., 0] - ora.real).max() <= 2e-7
    assert np.abs(cis[..., 1] - ora.imag).max() <= 2e-7


def test_rope_apply_matches_oracle():
    g = torch.Generator().manual_seed(7)
    end = torch.tensor([1, 2, 1001, 4096, 8191, 16384], dtype=torch.int32)
    q_pe = torch.randn(6, 128, 64, generator=g).to(torch.bfloat16)
    cis = mla.rope_freqs_init()
    got = mla.mla_rope_apply(q_pe.cuda(), cis, end.cuda()).cpu().double().numpy()
    x = synth.to_f64(q_pe)
    ora = O.rope_for_batch(x, end.numpy(), U.INV_FREQ)
    U.assert_rope_close(got, ora, x, "rope")


def test_rope_apply_reports_bad_position():
    cis = mla.rope_freqs_init()
    q_pe = torch.ones(2, 128, 64, dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = mla.mla_rope_apply(q_pe, cis, torch.tensor([0, 16385], dtype=torch.int32, device="cuda"), dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & mla.MLA_DEV_BAD_POSITION
    assert torch.all(out == 0)


@pytest.mark.parametrize("n_heads", [1, 64, 128])
@pytest.mark.parametrize("interleaved", [True, False])
def test_rope_apply_layout_matches_oracle(n_heads, interleaved):
    g = torch.Generator().manual_seed(17 + n_heads)
    end = torch.tensor([1, 2, 333, 4097, 12000, 16384, 7], dtype=torch.int32)
    x = torch.randn(7, n_heads, 64, generator=g).to(torch.bfloat16)
    cis = mla.rope_freqs_init()
    got = mla.mla_rope_apply_layout(x.cuda(), cis, end.cuda(), interleaved).cpu().double().numpy()
    xd = synth.to_f64(x)
    ora = O.rope_for_positions(xd, end.numpy(), U.INV_FREQ, interleaved=interleaved)
    U.assert_rope_close(got, ora, xd, f"rope layout {interleaved}", interleaved=interleaved)


def test_rope_apply_layout_interleaved_equals_query_rope():
    g = torch.Generator().manual_seed(5)
    end = torch.tensor([3, 16000], dtype=torch.int32, device="cuda")
    x = torch.randn(2, 128, 64, generator=g).to(torch.bfloat16).cuda()
    cis = mla.rope_freqs_init()
    a = mla.mla_rope_apply_layout(x, cis, end, True)
    b = mla.mla_rope_apply(x, cis, end)
    assert torch.equal(a, b)


def test_rope_apply_layout_reports_bad_position():
    cis = mla.rope_freqs_init()
    x = torch.ones(2, 64, 64, dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = mla.mla_rope_apply_layout(x, cis, torch.tensor([16385, 5], dtype=torch.int32, device="cuda"), False,
                                    dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & mla.MLA_DEV_BAD_POSITION
    assert torch.all(out[0] == 0) and torch.any(out[1] != 0)


def test_rope_apply_layout_rejects_bad_arguments():
    cis = mla.rope_freqs_init()
    x = torch.ones(1, 64, 64, dtype=torch.bfloat16, device="cuda")
    out = torch.empty(1, 64, 64, dtype=torch.float32, device="cuda")
    end = torch.ones(1, dtype=torch.int32, device="cuda")
    st = mla._lib.mla_rope_apply_layout(mla._ptr(x), mla._ptr(cis), cis.shape[0], mla._ptr(end), 1, 64, 2,
                                        mla._ptr(out), None, mla._stream(x.device))
    assert st != 0
    st = mla._lib.mla_rope_apply_layout(mla._ptr(x), mla._ptr(cis), cis.shape[0], mla._ptr(end), 1, 0, 1,
                                        mla._ptr(out), None, mla._stream(x.device))
    assert st != 0


# ----------------------------------------------------------------- absorb / up-projection
@pytest.mark.parametrize("B", [1, 3, 64, 130])
def test_absorb_matches_oracle(B):
    t = synth.make_inputs(synth.small_workload(B, [8] * B, k=1, K=1, S_cap=8), seed=11)
    # positions spread over the whole rotary table
    t["end_pos"] = torch.tensor([1 + (977 * b) % 16384 for b in range(B)], dtype=torch.int32)
    d = _dev(t)
    cis = mla.rope_freqs_init()
    q_lat = mla.mla_absorb_q(d["q_nope"], d["q_pe"], cis, d["end_pos"], d["wkv_b"]).cpu()
    x = U.oracle_inputs(t)
    ora = U.oracle_q_lat(x, list(range(B)))
    got = synth.to_f64(q_lat)
    U.assert_attn_close(got[..., :512], ora[..., :512], "absorbed q")
    U.assert_attn_close(got[..., 512:], ora[..., 512:], "rotated q_pe")
    # each element is the bf16 rounding of an fp32 sum: within 2^-8 relative
    assert np.all(np.abs(got - ora) <= 2.0 ** -8 * np.abs(ora) + 1e-6 * np.abs(ora).max())


@pytest.mark.parametrize("B", [1, 5, 64])
def test_out_up_matches_oracle(B):
    g = torch.Generator().manual_seed(13)
    o = torch.randn(B, 128, 512, generator=g)
    t = synth.make_inputs(synth.small_workload(1, [4], k=1, K=1, S_cap=4), seed=2)
    got = mla.mla_out_up(o.cuda(), t["wkv_b"].cuda()).cpu().double().numpy()
    ora = O.out_up(o.double().numpy(), synth.to_f64(t["wkv_b"]))
    U.assert_attn_close(got, ora, "out_up")


# ----------------------------------------------------------------- attention, small cases
SMALL = [
    # (B, end_pos, k, K, S_cap, selection)
    (1, [8], 8, 8, 8, "uniform"),
    (3, [600, 333, 37], 300, 300, 600, "uniform"),          # ragged tail: K not a multiple of 32
    (2, [1000, 1000], 1000, 1000, 1024, "all"),
    (4, [2100, 1500, 2048, 700], 1100, 1100, 2112, "recent_half"),
    (2, [5000, 4097], 2048, 2048, 5000, "uniform"),
    (3, [1000, 70, 3000], 2048, 2048, 3000, "uniform"),    # rows mostly padding: units cut short or left empty
    (40, [4096] * 40, 4096, 4096, 4096, "uniform"),        # one unit of 4096 entries (16-bit staged positions)
    (2, [70000, 65600], 3000, 3000, 70000, "uniform"),     # a cache of 70,000 rows: 32-bit staged positions
    # few splits merged by the up-projection from bf16 partials (the largest share of their rounding)
    (1, [150], 150, 150, 256, "all"),                       # three units, the last one ragged
    (2, [128, 100], 128, 128, 256, "uniform"),              # two units per row, two rows
]


@pytest.mark.parametrize("case", SMALL, ids=[f"B{c[0]}_K{c[3]}" for c in SMALL])
def test_sparse_decode_small_matches_oracle(case):
    B, ep, k, K, S, sel = case
    t = synth.make_inputs(synth.small_workload(B, ep, k=k, K=K, S_cap=S, selection=sel), seed=3)
    d = _dev(t)
    x = U.oracle_inputs(t)
    # a rotary table long enough for the positions (its frequencies do not depend on its length)
    params = mla.rope_params(max_seq_len=S) if S > 16384 else None
    step = mla.DecodeStep(B, K, params=params)
    out = step(d["q_nope"], d["q_pe"], d["kv_cache"], d["pe_cache"], d["wkv_b"], d["topk_idx"], d["end_pos"])
    torch.cuda.synchronize()
    step.check_status()
    U.assert_attn_close(out.cpu().numpy(), U.oracle_out(x, list(range(B))), "head outputs")
    # the attention stage alone, with the GPU's own bf16 query
    o = mla.mla_sparse_decode(step.q_lat, d["kv_cache"], d["pe_cache"], d["topk_idx"], d["end_pos"], step.scale)
    q_gpu = synth.to_f64(step.q_lat.cpu())
    U.assert_attn_close(o.cpu().numpy(), U.oracle_o_lat(x, list(range(B)), q_lat=q_gpu), "latent o")


@pytest.mark.parametrize("growth", ["flat", "step", "ramp"])
def test_many_blocks_per_unit_and_rescaled_maximum(growth):
    # 80 sequences (one unit each: no split) x 640 selected keys = 10 key blocks
    # per unit, more than the gather pipeline has stages.  "step" scales the
    # cache rows of the second half of each selection by 3, "ramp" by
    # 1 + 0.35 * block index: later blocks raise the running maximum, which
    # forces the rescaling of the accumulated output.
    B, S, K = 80, 700, 640
    t = synth.make_inputs(synth.small_workload(B, [S] * B, k=K, K=K, S_cap=S), seed=31)
    if growth != "flat":
        for b in range(B):
            sel = t["topk_idx"][b].long()
            for j in range(K // 64):
                f = (3.0 if j >= 5 else 1.0) if growth == "step" else 1.0 + 0.35 * j
                rows = sel[64 * j: 64 * (j + 1)]
                t["kv_cache"][b, rows] = (t["kv_cache"][b, rows].float() * f).to(torch.bfloat16)
                t["pe_cache"][b, rows] = (t["pe_cache"][b, rows].float() * f).to(torch.bfloat16)
    d = _dev(t)
    step = mla.DecodeStep(B, K)
    out = step(d["q_nope"], d["q_pe"], d["kv_cache"], d["pe_cache"], d["wkv_b"], d["topk_idx"], d["end_pos"])
    torch.cuda.synchronize()
    step.check_status()
    x = U.oracle_inputs(t)
    bs = [0, 1, 39, 79]
    U.assert_attn_close(out.cpu().numpy()[bs], U.oracle_out(x, bs), f"many blocks ({growth})")


def _scaled_case(q_scale, row_scale, seed=91):
    B, S, K = 3, 2048, 1024
    t = synth.make_inputs(synth.small_workload(B, [2048, 1500, 1100], k=K, K=K, S_cap=S), seed=seed)
    t["q_nope"] = (t["q_nope"].float() * q_scale).to(torch.bfloat16)
    t["q_pe"] = (t["q_pe"].float() * q_scale).to(torch.bfloat16)
    g = torch.Generator().manual_seed(seed + 1)
    for b in range(B):
        sel = t["topk_idx"][b].long()
        rows = sel[torch.randperm(K, generator=g)[:6]]
        t["kv_cache"][b, rows] = (t["kv_cache"][b, rows].float() * row_scale).to(torch.bfloat16)
        t["pe_cache"][b, rows] = (t["pe_cache"][b, rows].float() * row_scale).to(torch.bfloat16)
    d = _dev(t)
    step = mla.DecodeStep(B, K)
    out = step(d["q_nope"], d["q_pe"], d["kv_cache"], d["pe_cache"], d["wkv_b"], d["topk_idx"], d["end_pos"])
    torch.cuda.synchronize()
    x = U.oracle_inputs(t)
    # the largest partial score either CTA of a pair sends (from the GPU's own bf16 query)
    q = synth.to_f64(step.q_lat.cpu())
    big = 0.0
    for b in range(B):
        e = int(x["end_pos"][b])
        sel = x["topk_idx"][b][(x["topk_idx"][b] >= 0) & (x["topk_idx"][b] < e)].astype(np.int64)
        kv, pe = x["kv_cache"][b][sel], x["pe_cache"][b][sel]
        for r in range(2):
            part = q[b, :, 256 * r:256 * r + 256] @ kv[:, 256 * r:256 * r + 256].T + \
                q[b, :, 512 + 32 * r:512 + 32 * r + 32] @ pe[:, 32 * r:32 * r + 32].T
            big = max(big, float(np.abs(part).max()))
    return step, out, x, big, B, d


@pytest.mark.parametrize("q_scale", [4.0, 8.0, 16.0])
def test_large_scores_and_peaked_softmax(q_scale):
    # Each CTA of a pair sends its partial scores (half of the 576-wide dot
    # product) to the other as fp16.  Scaling the query drives the partial
    # scores to hundreds (logits up to ~110) and the softmax towards a few
    # dominant keys; the result must stay within the tolerance and the status
    # word clear while every partial is within the exchange's stated range.
    # The query enters the attention as bf16 (q_lat), whose rounding moves a
    # logit by ~2^-9 of its size; that error belongs to the query's dtype, so
    # the attention stage is compared with the GPU's own bf16 q_lat as input.
    step, out, x, big, B, d = _scaled_case(q_scale, 1.0)
    assert 150.0 < big <= 2048.0
    assert int(step.status.item()) == 0
    assert np.all(np.isfinite(out.cpu().numpy()))
    o = mla.mla_sparse_decode(step.q_lat, d["kv_cache"], d["pe_cache"], d["topk_idx"], d["end_pos"], step.scale)
    q_gpu = synth.to_f64(step.q_lat.cpu())
    U.assert_attn_close(o.cpu().numpy(), U.oracle_o_lat(x, list(range(B)), q_lat=q_gpu), f"large scores x{q_scale}")


@pytest.mark.parametrize("q_scale,row_scale", [(16.0, 8.0), (1024.0, 64.0)], ids=["beyond_range", "beyond_fp16"])
def test_partial_scores_beyond_the_exchange_range_are_reported(q_scale, row_scale):
    # a partial above 2048 (and one above fp16's 65504) sets MLA_DEV_SCORE_RANGE
    step, out, x, big, B, _ = _scaled_case(q_scale, row_scale)
    assert big > 2048.0
    assert int(step.status.item()) & mla.MLA_DEV_SCORE_RANGE


def test_padding_out_of_range_and_empty_rows():
    B, S = 3, 512
    t = synth.make_inputs(synth.small_workload(B, [512, 300, 200], k=100, K=160, S_cap=S), seed=5)
    topk = t["topk_idx"].clone()
    topk[0, 100:130] = torch.tensor([-5, 512, 513, 10 ** 6, -1] * 6, dtype=torch.int32)
    topk[1, 100:] = 300 + torch.arange(60, dtype=torch.int32)   # all >= end_pos[1] = 300
    topk[2, :] = -1       # nothing selected
    t["topk_idx"] = topk
    d = _dev(t)
    x = U.oracle_inputs(t)
    step = mla.DecodeStep(B, 160)
    out = step(d["q_nope"], d["q_pe"], d["kv_cache"], d["pe_cache"], d["wkv_b"], d["topk_idx"], d["end_pos"])
    torch.cuda.synchronize()
    step.check_status()
    got = out.cpu().numpy()
    assert np.all(got[2] == 0.0)
    U.assert_attn_close(got[:2], U.oracle_out(x, [0, 1]), "padded rows")


def test_nan_poisoned_unselected_rows_do_not_leak():
    B, S = 2, 700
    t = synth.make_inputs(synth.small_workload(B, [700, 650], k=200, K=200, S_cap=S), seed=6)
    x = U.oracle_inputs(t)
    want = U.oracle_out(x, [0, 1])
    for b in range(B):
        keep = torch.zeros(S, dtype=torch.bool)
        keep[t["topk_idx"][b].long()] = True
        t["kv_cache"][b][~keep] = float("nan")
        t["pe_cache"][b][~keep] = float("nan")
    d = _dev(t)
    step = mla.DecodeStep(B, 200)
    out = step(d["q_nope"], d["q_pe"], d["kv_cache"], d["pe_cache"], d["wkv_b"], d["topk_idx"], d["end_pos"])
    torch.cuda.synchronize()
    U.assert_attn_close(out.cpu().numpy(), want, "NaN-poisoned cache")


def test_selection_order_does_not_matter():
    B = 2
    t = synth.make_inputs(synth.small_workload(B, [900, 900], k=512, K=512, S_cap=900), seed=8)
    d = _dev(t)
    step = mla.DecodeStep(B, 512)
    a = step(d["q_nope"], d["q_pe"], d["kv_cache"], d["pe_cache"], d["wkv_b"], d["topk_idx"], d["end_pos"]).clone()
    perm = torch.randperm(512, generator=torch.Generator().manual_seed(1))
    b = step(d["q_nope"], d["q_pe"], d["kv_cache"], d["pe_cache"], d["wkv_b"], d["topk_idx"][:, perm.cuda()].contiguous(),
             d["end_pos"])
    torch.cuda.synchronize()
    U.assert_attn_close(b.cpu().numpy(), a.cpu().numpy().astype(np.float64), "permuted selection")


def _expected_dup(topk, end_pos, T):
    """Plain set logic: does some row repeat a position it can see?"""
    n = end_pos.shape[0]
    rows = topk.reshape(n * T, -1)
    for r in range(n * T):
        b, s = divmod(r, T)
        ep = int(end_pos[b])
        e = ep - T + s + 1
        if ep < T:
            continue
        valid = [int(t) for t in rows[r] if 0 <= int(t) < e]
        if len(valid) != len(set(valid)):
            return True
    return False


def test_check_selection_flags_repeated_visible_positions_only():
    S = 100

    def run(topk, end_pos, T=1):
        tk = torch.tensor(topk, dtype=torch.int32).cuda()
        ep = torch.tensor(end_pos, dtype=torch.int32).cuda()
        st = mla.mla_check_selection(tk, ep, S)
        torch.cuda.synchronize()
        return int(st.item())

    # distinct positions; padding (negative, at or beyond end_pos) repeated freely
    assert run([[0, 5, 99, -1, -1, 7], [3, 49, 50, 50, 60, -7]], [100, 50]) == 0
    # a repeated position that the row sees
    assert run([[0, 5, 99, -1, -1, 7], [3, 49, 3, 50, 60, -7]], [100, 50]) == mla.MLA_DEV_DUPLICATE_INDEX
    # at the edge of the visible range: end_pos - 1 repeated is flagged, end_pos repeated is not
    assert run([[9, 9, 0]], [10]) == mla.MLA_DEV_DUPLICATE_INDEX
    assert run([[10, 10, 0]], [10]) == 0
    # multi-token: token 0 of a two-token sequence does not see position end_pos - 1, token 1 does
    tk = [[[39, 39, 1], [2, 3, 4]]]
    assert run(tk, [40], T=2) == 0
    tk = [[[2, 3, 4], [39, 39, 1]]]
    assert run(tk, [40], T=2) == mla.MLA_DEV_DUPLICATE_INDEX
    # a sequence with a bad end_pos is skipped and reported as the decode reports it
    assert run([[1, 1, 2], [4, 5, 6]], [0, 100]) == mla.MLA_DEV_BAD_END_POS
    # random rows against plain set logic (rows of up to 2048 entries, a third of them repeating a position)
    g = np.random.default_rng(11)
    for trial in range(40):
        n, T, K = int(g.integers(1, 5)), int(g.integers(1, 3)), int(g.choice([3, 64, 2048]))
        end_pos = g.integers(T, S + 1, size=n)
        topk = np.empty((n, T, K), dtype=np.int64)
        for b in range(n):
            for t in range(T):
                row = g.permutation(np.arange(-5, S + 5))[:K] if K <= S + 10 else g.integers(-5, S + 5, size=K)
                if K <= S + 10 and g.random() < 0.33:
                    row[int(g.integers(0, K))] = row[int(g.integers(0, K))]
                topk[b, t] = row
        got = run(topk.tolist(), end_pos.tolist(), T=T)
        want = mla.MLA_DEV_DUPLICATE_INDEX if _expected_dup(topk, end_pos, T) else 0
        assert got == want, (trial, n, T, K)


def test_check_selection_at_the_largest_cache():
    # the bitmap spans the whole visible range of the largest cache the check accepts
    S = mla.CHECK_MAX_S_CAP
    tk = torch.tensor([[S - 1, 0, S // 2, S - 1]], dtype=torch.int32).cuda()
    ep = torch.tensor([S], dtype=torch.int32).cuda()
    assert int(mla.mla_check_selection(tk, ep, S).item()) == mla.MLA_DEV_DUPLICATE_INDEX
    tk[0, 3] = S - 2
    assert int(mla.mla_check_selection(tk, ep, S).item()) == 0


def test_single_key_and_bad_end_pos_status():
    B, S = 3, 64
    t = synth.make_inputs(synth.small_workload(B, [64, 64, 64], k=1, K=1, S_cap=S), seed=9)
    t["end_pos"] = torch.tensor([64, 0, 65], dtype=torch.int32)   # 0 and > S_cap are invalid
    d = _dev(t)
    step = mla.DecodeStep(B, 1)
    out = step(d["q_nope"], d["q_pe"], d["kv_cache"], d["pe_cache"], d["wkv_b"], d["topk_idx"], d["end_pos"])
    torch.cuda.synchronize()
    st = int(step.status.item())
    assert st & mla.MLA_DEV_BAD_END_POS
    got = out.cpu().numpy()
    assert np.all(got[1] == 0.0) and np.all(got[2] == 0.0)
    x = U.oracle_inputs(t)
    tk = int(t["topk_idx"][0, 0])
    w_uv = x["wkv_b"].reshape(128, 256, 512)[:, 128:, :]
    want = np.einsum("hdc,c->hd", w_uv, x["kv_cache"][0][tk])
    U.assert_attn_close(got[0], want, "single key")


# ----------------------------------------------------------------- the named workloads, full size
@pytest.mark.parametrize("name", synth.WORKLOADS)
def test_named_workload_matches_oracle_on_every_sequence(name):
    # the step as bench.py times it (DecodeStep: absorb, attention with its
    # split policy, up-projection), compared with the oracle on every
    # sequence of the batch, each sequence checked on its own
    wl = synth.workload(name)
    t = synth.make_inputs(wl, seed=0)
    d = _dev(t)
    step = mla.DecodeStep(wl.B, wl.row_stride())
    out = step(d["q_nope"], d["q_pe"], d["kv_cache"], d["pe_cache"], d["wkv_b"], d["topk_idx"], d["end_pos"])
    torch.cuda.synchronize()
    step.check_status()
    got = out.cpu().numpy()
    del d
    assert np.all(np.isfinite(got))
    x = _oracle_view(t)
    for b0 in range(0, wl.B, 16):
        bs = list(range(b0, min(wl.B, b0 + 16)))
        ora = U.oracle_out(x, bs)
        for j, b in enumerate(bs):
            U.assert_attn_close(got[b], ora[j], f"{name}, sequence {b}")


# ----------------------------------------------------------------- fp8 wkv_b
def _assert_bits_equal(got_bf16, want_f64):
    got = got_bf16.cpu().to(torch.float64).numpy()
    nan = np.isnan(want_f64)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want_f64[~nan])
    # the sign of zero is part of the bit pattern
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(want_f64[~nan]))


def test_dequant_wkv_b_is_bit_exact():
    codes, scale = synth.make_fp8_weight(21)
    got = mla.mla_weight_dequant_fp8(codes.cuda(), scale.cuda())
    _assert_bits_equal(got, O.dequant_to_bf16(codes.numpy(), scale.numpy(), 128))


@pytest.mark.parametrize("rows,cols,block", [(200, 300, 128), (130, 528, 128), (64, 96, 64), (7, 33, 1),
                                             (1, 16, 128), (257, 512, 32), (3, 5, 4)])
def test_dequant_ragged_shapes_and_blocks(rows, cols, block):
    codes, scale = synth.make_fp8_weight(rows * 7 + cols, rows=rows, cols=cols, block=block, name="ragged")
    got = mla.mla_weight_dequant_fp8(codes.cuda(), scale.cuda(), block=block)
    _assert_bits_equal(got, O.dequant_to_bf16(codes.numpy(), scale.numpy(), block))


def test_dequant_every_code_including_nan_and_signed_zero():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8).reshape(16, 16)
    scale = torch.tensor([[0.75]], dtype=torch.float32)
    got = mla.mla_weight_dequant_fp8(codes.cuda(), scale.cuda(), block=16)
    _assert_bits_equal(got, O.dequant_to_bf16(codes.numpy(), scale.numpy(), 16))


def test_dequant_unaligned_output_takes_the_scalar_path():
    codes, scale = synth.make_fp8_weight(4, rows=40, cols=128, block=128)
    buf = torch.empty(40 * 128 + 1, dtype=torch.bfloat16, device="cuda")
    out = buf[1:].view(40, 128)                   # 2-byte offset: not 16-byte aligned
    mla.mla_weight_dequant_fp8(codes.cuda(), scale.cuda(), out=out)
    _assert_bits_equal(out, O.dequant_to_bf16(codes.numpy(), scale.numpy(), 128))


def test_decode_with_fp8_wkv_b_matches_oracle():
    B = 3
    t = synth.make_inputs(synth.small_workload(B, [700, 64, 1001], k=256, K=256, S_cap=1024), seed=29)
    codes, scale = synth.make_fp8_weight(29)
    d = _dev(t)
    d["wkv_b"] = mla.mla_weight_dequant_fp8(codes.cuda(), scale.cuda())
    step = mla.DecodeStep(B, 256)
    out = step(d["q_nope"], d["q_pe"], d["kv_cache"], d["pe_cache"], d["wkv_b"], d["topk_idx"], d["end_pos"])
    torch.cuda.synchronize()
    step.check_status()
    x = U.oracle_inputs(t)
    x["wkv_b"] = O.dequant_to_bf16(codes.numpy(), scale.numpy(), 128)
    U.assert_attn_close(out.cpu().numpy(), U.oracle_out(x, list(range(B))), "decode with fp8 wkv_b")


# ----------------------------------------------------------------- captured step
def test_one_sequence_step_merges_its_splits_in_the_up_projection():
    # B = 1: the selection is split over many units and the up-projection
    # merges the partials itself (no combine kernel)
    B, K = 1, 4096
    t = synth.make_inputs(synth.small_workload(B, [4096], k=K, K=K, S_cap=4096, selection="all"), seed=43)
    d = _dev(t)
    step = mla.DecodeStep(B, K)
    with mla.ProfileHook() as hook:
        out = step(d["q_nope"], d["q_pe"], d["kv_cache"], d["pe_cache"], d["wkv_b"], d["topk_idx"], d["end_pos"])
        torch.cuda.synchronize()
    step.check_status()
    assert hook.launches == 3                     # absorb, attention, up-projection
    x = U.oracle_inputs(t)
    U.assert_attn_close(out.cpu().numpy(), U.oracle_out(x, [0]), "one sequence, split merged in the up-projection")


def test_captured_step_replays_the_eager_step_exactly():
    B, K = 5, 512
    t = synth.make_inputs(synth.small_workload(B, [900, 512, 1000, 64, 777], k=K, K=K, S_cap=1024), seed=41)
    d = _dev(t)
    args = (d["q_nope"], d["q_pe"], d["kv_cache"], d["pe_cache"], d["wkv_b"], d["topk_idx"], d["end_pos"])
    step = mla.DecodeStep(B, K)
    with mla.ProfileHook() as hook:
        eager = step(*args).clone()
    g = mla.CapturedStep(step, *args)
    # absorb, attention, split combine (5 sequences do not fill the GPU: their
    # selections are split), up-projection
    assert g.kernels_per_replay == hook.launches == 4
    d["q_nope"].mul_(-1)                      # new inputs in the captured buffers
    out = g().clone()
    torch.cuda.synchronize()
    step.check_status()
    x = U.oracle_inputs(t)
    x["q_nope"] = -x["q_nope"]
    U.assert_attn_close(out.cpu().numpy(), U.oracle_out(x, list(range(B))), "captured step, new inputs")
    d["q_nope"].mul_(-1)
    assert torch.equal(g().clone(), eager)


# ----------------------------------------------------------------- cache append
def _append_case(B, T, S_cap, end, seed):
    g = torch.Generator().manual_seed(seed)
    kv_a = (torch.randn(B, T, 576, generator=g) * 2.5).to(torch.bfloat16)
    w = (1.0 + 0.1 * torch.randn(512, generator=g)).to(torch.bfloat16).float()
    kv = torch.full((B, S_cap, 512), 7.0, dtype=torch.bfloat16)
    pe = torch.full((B, S_cap, 64), 7.0, dtype=torch.bfloat16)
    return kv_a, w, kv, pe, torch.tensor(end, dtype=torch.int32)


@pytest.mark.parametrize("B,T,S_cap,end", [(1, 1, 16, [1]), (4, 1, 1024, [1, 2, 1000, 1024]),
                                           (3, 4, 4096, [4, 4096, 1234]), (130, 2, 64, [2 + b % 62 for b in range(130)])])
def test_cache_append_matches_oracle(B, T, S_cap, end):
    kv_a, w, kv, pe, end_pos = _append_case(B, T, S_cap, end, seed=B * 13 + T)
    cis = mla.rope_freqs_init()
    dkv, dpe = kv.cuda(), pe.cuda()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    mla.mla_cache_append(kv_a.cuda(), w.cuda(), cis, end_pos.cuda(), dkv, dpe, eps=1e-6, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    pos, lat, rot = O.cache_rows(synth.to_f64(kv_a), w.double().numpy(), 1e-6, end_pos.numpy(), U.INV_FREQ)
    got_kv, got_pe = dkv.cpu(), dpe.cpu()
    written = torch.zeros(B, S_cap, dtype=torch.bool)
    for b in range(B):
        for s in range(T):
            p = int(pos[b, s])
            written[b, p] = True
            gl = got_kv[b, p].double().numpy()
            # bf16 rounding of the fp32 result: half an ulp (2^-8 relative) plus fp32 error
            assert np.all(np.abs(gl - lat[b, s]) <= 2.0 ** -8 * np.abs(lat[b, s]) + 1e-5), (b, s)
            gr = got_pe[b, p].double().numpy()
            pair = np.repeat(np.hypot(rot[b, s, 0::2], rot[b, s, 1::2]), 2)
            assert np.all(np.abs(gr - rot[b, s]) <= 2.0 ** -8 * np.abs(rot[b, s]) + 1e-5 * pair), (b, s)
    # nothing else was touched
    assert torch.all(got_kv[~written] == 7.0) and torch.all(got_pe[~written] == 7.0)


def test_cache_append_then_decode_reads_the_new_rows():
    B, S_cap, K = 2, 512, 128
    t = synth.make_inputs(synth.small_workload(B, [300, 511], k=K, K=K, S_cap=S_cap), seed=43)
    kv_a, w, _, _, _ = _append_case(B, 1, S_cap, [1, 1], seed=44)
    end_pos = t["end_pos"] + 1                    # one new token per sequence
    t["topk_idx"][:, 0] = end_pos - 1             # the new token is selected
    d = _dev(t)
    cis = mla.rope_freqs_init()
    mla.mla_cache_append(kv_a.cuda(), w.cuda(), cis, end_pos.cuda(), d["kv_cache"], d["pe_cache"])
    step = mla.DecodeStep(B, K)
    out = step(d["q_nope"], d["q_pe"], d["kv_cache"], d["pe_cache"], d["wkv_b"], d["topk_idx"], end_pos.cuda())
    torch.cuda.synchronize()
    step.check_status()
    x = U.oracle_inputs(t)
    x["end_pos"] = end_pos.numpy().astype(np.int64)
    # the oracle reads the appended rows the GPU wrote (bf16, checked above)
    x["kv_cache"] = synth.to_f64(d["kv_cache"].cpu())
    x["pe_cache"] = synth.to_f64(d["pe_cache"].cpu())
    U.assert_attn_close(out.cpu().numpy(), U.oracle_out(x, list(range(B))), "decode after append")


def test_cache_append_reports_and_skips_bad_positions():
    kv_a, w, kv, pe, _ = _append_case(3, 2, 64, [2, 2, 2], seed=5)
    dkv, dpe = kv.cuda(), pe.cuda()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    cis = mla.rope_freqs_init(mla.rope_params(max_seq_len=32))
    end = torch.tensor([1, 65, 40], dtype=torch.int32, device="cuda")   # < T, > S_cap, beyond the table
    mla.mla_cache_append(kv_a.cuda(), w.cuda(), cis, end, dkv, dpe, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == mla.MLA_DEV_BAD_END_POS | mla.MLA_DEV_BAD_POSITION
    assert torch.all(dkv.cpu() == 7.0) and torch.all(dpe.cpu() == 7.0)


# ----------------------------------------------------------------- multi-token decode
TOKENS = [
    # (end_pos per sequence, T, k, K)
    ([300, 41], 2, 40, 40),
    ([1000, 64, 777], 4, 256, 256),
    ([2048, 1500], 3, 1100, 1100),       # several splits per query row
    ([5, 9, 600, 4096] * 5, 2, 300, 320),  # 40 query rows, ragged K tail
    ([1500], 2, 1100, 1100),             # two query rows of one sequence: splits merged in the up-projection
]


@pytest.mark.parametrize("case", TOKENS, ids=[f"n{len(c[0])}_T{c[1]}_K{c[3]}" for c in TOKENS])
def test_multi_token_decode_matches_oracle(case):
    ends, T, k, K = case
    S = max(ends)
    wl = synth.small_workload(len(ends), ends, k=k, K=K, S_cap=S)
    t = synth.make_token_inputs(wl, T, seed=47)
    d = _dev(t)
    cis = mla.rope_freqs_init()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    q_lat = mla.mla_absorb_q_tokens(d["q_nope"], d["q_pe"], cis, d["end_pos"], d["wkv_b"], dev_status=st)
    out = mla.mla_sparse_decode_tokens(q_lat, d["kv_cache"], d["pe_cache"], d["topk_idx"], d["end_pos"], U.SCALE,
                                       wkv_b=d["wkv_b"], dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    x = U.oracle_inputs(t)
    ora = O.decode_tokens(x["q_nope"], x["q_pe"], x["kv_cache"], x["pe_cache"], x["wkv_b"], x["topk_idx"],
                          x["end_pos"], U.INV_FREQ, U.SCALE)
    U.assert_attn_close(out.cpu().numpy().reshape(-1, 128, 128), ora.reshape(-1, 128, 128), "multi-token")


def test_multi_token_decode_at_full_context_on_sampled_sequences():
    # the multi-token row as bench.py times it: 32 sequences x 2 query tokens over a
    # 16384-row cache, a top-2048 selection per token; compared with the oracle on
    # sampled sequences (both tokens of each), the rest checked for finiteness
    n, T, K = 32, 2, 2048
    wl = synth.small_workload(n, [16384] * n, k=K, K=K, S_cap=16384)
    t = synth.make_token_inputs(wl, T, seed=59, threads=16)
    d = _dev(t)
    cis = mla.rope_freqs_init()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    q_lat = mla.mla_absorb_q_tokens(d["q_nope"], d["q_pe"], cis, d["end_pos"], d["wkv_b"], dev_status=st)
    out = mla.mla_sparse_decode_tokens(q_lat, d["kv_cache"], d["pe_cache"], d["topk_idx"], d["end_pos"], U.SCALE,
                                       wkv_b=d["wkv_b"], dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    got = out.cpu()
    assert torch.isfinite(got).all()
    bs = [0, 17, 31]
    x = {k: synth.to_f64(t[k][bs]) for k in ("q_nope", "q_pe", "kv_cache", "pe_cache", "topk_idx", "end_pos")}
    ora = O.decode_tokens(x["q_nope"], x["q_pe"], x["kv_cache"], x["pe_cache"], synth.to_f64(t["wkv_b"]),
                          x["topk_idx"], x["end_pos"], U.INV_FREQ, U.SCALE)
    U.assert_attn_close(got[bs].numpy().reshape(-1, 128, 128), ora.reshape(-1, 128, 128), "multi-token, full context")


def test_multi_token_one_token_equals_the_single_token_entry():
    B, K = 6, 512
    t = synth.make_inputs(synth.small_workload(B, [900, 512, 1000, 64, 777, 1], k=K, K=K, S_cap=1024), seed=53)
    d = _dev(t)
    cis = mla.rope_freqs_init()
    q1 = mla.mla_absorb_q(d["q_nope"], d["q_pe"], cis, d["end_pos"], d["wkv_b"])
    qt = mla.mla_absorb_q_tokens(d["q_nope"][:, None], d["q_pe"][:, None], cis, d["end_pos"], d["wkv_b"])
    assert torch.equal(q1, qt[:, 0])
    o1 = mla.mla_sparse_decode(q1, d["kv_cache"], d["pe_cache"], d["topk_idx"], d["end_pos"], U.SCALE, wkv_b=d["wkv_b"])
    ot = mla.mla_sparse_decode_tokens(qt, d["kv_cache"], d["pe_cache"], d["topk_idx"][:, None], d["end_pos"], U.SCALE,
                                      wkv_b=d["wkv_b"])
    assert torch.equal(o1, ot[:, 0])


def test_multi_token_bad_end_pos_is_reported():
    wl = synth.small_workload(2, [3, 100], k=3, K=3, S_cap=100)
    t = synth.make_token_inputs(wl, 4, seed=2)
    d = _dev(t)
    cis = mla.rope_freqs_init()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    q_lat = mla.mla_absorb_q_tokens(d["q_nope"], d["q_pe"], cis, d["end_pos"], d["wkv_b"], dev_status=st)
    out = mla.mla_sparse_decode_tokens(q_lat, d["kv_cache"], d["pe_cache"], d["topk_idx"], d["end_pos"], U.SCALE,
                                       wkv_b=d["wkv_b"], dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & mla.MLA_DEV_BAD_END_POS       # end_pos 3 < T = 4
    assert torch.all(out[0] == 0) and torch.any(out[1] != 0)


# ----------------------------------------------------------------- projections (wkv_a, wo)
def _assert_linear_close(got, x, w, cols=None, bf16_out=False):
    xd, wd = synth.to_f64(x), synth.to_f64(w)
    if cols is not None:
        wd = wd[cols]
        got = got[:, cols]
    ref = O.linear(xd, wd)
    mag = O.linear(np.abs(xd), np.abs(wd))       # sum_k |x w|: the scale of fp32 accumulation error
    g = got.cpu().double().numpy()
    tol = 2e-6 * mag + (2.0 ** -8 * np.abs(ref) if bf16_out else 0.0)
    assert np.all(np.abs(g - ref) <= tol), float(np.max(np.abs(g - ref) / np.maximum(mag, 1e-30)))


@pytest.mark.parametrize("M,N,K", [(1, 576, 7168), (64, 576, 7168), (3, 200, 72), (17, 129, 1024),
                                   (300, 256, 128), (64, 1024, 16384), (256, 128, 64)])
def test_linear_matches_oracle(M, N, K):
    x, w = synth.make_linear_inputs(M * 31 + N, M, N, K)
    got = mla.mla_linear_bf16(x.cuda(), w.cuda())
    torch.cuda.synchronize()
    _assert_linear_close(got, x, w)


def test_linear_wo_full_size_sampled_columns_and_bf16_output():
    M, N, K = 64, 7168, 16384
    x, w = synth.make_linear_inputs(61, M, N, K)
    dx, dw = x.cuda(), w.cuda()
    y = mla.mla_linear_bf16(dx, dw)
    yb = mla.mla_linear_bf16(dx, dw, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    cols = np.random.default_rng(0).choice(N, 384, replace=False)
    cols = np.concatenate([cols, [0, 127, 128, N - 1]])
    _assert_linear_close(y, x, w, cols)
    _assert_linear_close(yb, x, w, cols, bf16_out=True)
    assert torch.equal(yb, y.to(torch.bfloat16))     # one rounding of the same fp32 sums
    assert torch.equal(y, mla.mla_linear_bf16(dx, dw))   # reproducible


def test_decode_bf16_output_feeds_the_output_projection():
    B, K, dim = 4, 256, 1024
    t = synth.make_inputs(synth.small_workload(B, [500, 256, 1000, 3], k=K, K=K, S_cap=1024), seed=67)
    d = _dev(t)
    cis = mla.rope_freqs_init()
    q_lat = mla.mla_absorb_q(d["q_nope"], d["q_pe"], cis, d["end_pos"], d["wkv_b"])
    out32 = mla.mla_sparse_decode_tokens(q_lat[:, None], d["kv_cache"], d["pe_cache"], d["topk_idx"][:, None],
                                         d["end_pos"], U.SCALE, wkv_b=d["wkv_b"])
    out16 = mla.mla_sparse_decode_tokens(q_lat[:, None], d["kv_cache"], d["pe_cache"], d["topk_idx"][:, None],
                                         d["end_pos"], U.SCALE, wkv_b=d["wkv_b"], out_dtype=torch.bfloat16)
    o16 = mla.mla_sparse_decode_tokens(q_lat[:, None], d["kv_cache"], d["pe_cache"], d["topk_idx"][:, None],
                                       d["end_pos"], U.SCALE, out_dtype=torch.bfloat16)
    o32 = mla.mla_sparse_decode(q_lat, d["kv_cache"], d["pe_cache"], d["topk_idx"], d["end_pos"], U.SCALE)
    _, wo = synth.make_linear_inputs(68, 1, dim, 128 * 128, name="wo")
    y = mla.mla_linear_bf16(out16.reshape(B, -1), wo.cuda())
    torch.cuda.synchronize()
    assert torch.equal(out16, out32.to(torch.bfloat16))
    # the latent o in bf16 is the attention's own bf16 rounding (the combine or the epilogue)
    assert torch.allclose(o16[:, 0].float(), o32, rtol=2 ** -8, atol=1e-6)
    x = U.oracle_inputs(t)
    heads = U.oracle_out(x, list(range(B)))
    ora = O.output_projection(O.round_to_bf16(heads), synth.to_f64(wo))
    mag = O.output_projection(np.abs(heads), np.abs(synth.to_f64(wo)))
    err = np.abs(y.cpu().double().numpy() - ora)
    # the head outputs carry the attention tolerance (relative to their size)
    # before the projection; the projection adds fp32 accumulation error
    assert np.all(err <= 5e-3 * mag + 1e-4), float(np.max(err / np.maximum(mag, 1e-30)))


def test_host_buffer_step_matches_oracle_eager_and_captured():
    # the end-to-end path bench.py times: pinned host inputs in, head outputs back
    B, K = 3, 256
    t = synth.make_inputs(synth.small_workload(B, [700, 256, 1000], k=K, K=K, S_cap=1024), seed=71)
    d = _dev(t)
    h = {k: t[k].pin_memory() for k in ("q_nope", "q_pe", "topk_idx", "end_pos")}
    hs = mla.HostDecodeStep(B, K)
    out = hs.run(h["q_nope"], h["q_pe"], h["topk_idx"], h["end_pos"], d["kv_cache"], d["pe_cache"], d["wkv_b"])
    torch.cuda.synchronize()
    hs.check_status()
    assert out.device.type == "cpu" and out.is_pinned()
    x = U.oracle_inputs(t)
    U.assert_attn_close(out.numpy(), U.oracle_out(x, list(range(B))), "host-buffer step")
    eager = out.clone()
    g = mla.CapturedStep(hs.run, h["q_nope"], h["q_pe"], h["topk_idx"], h["end_pos"], d["kv_cache"],
                         d["pe_cache"], d["wkv_b"])
    h["q_nope"].mul_(-1)                      # new inputs in the captured host buffers
    g()
    torch.cuda.synchronize()                  # the result is copied back asynchronously
    got = g.out.clone()
    x["q_nope"] = -x["q_nope"]
    U.assert_attn_close(got.numpy(), U.oracle_out(x, list(range(B))), "captured host-buffer step")
    h["q_nope"].mul_(-1)
    g()
    torch.cuda.synchronize()
    assert torch.equal(g.out, eager)
    # the same inputs in one packed pinned buffer, copied in at once: the same bits
    packed = torch.zeros(mla.HostDecodeStep.packed_bytes(B, K), dtype=torch.uint8).pin_memory()
    for view, name in zip(mla.HostDecodeStep.packed_inputs(packed, B, K), ("q_nope", "q_pe", "topk_idx", "end_pos")):
        view.copy_(h[name])
    hs2 = mla.HostDecodeStep(B, K)
    got = hs2.run_packed(packed, d["kv_cache"], d["pe_cache"], d["wkv_b"])
    torch.cuda.synchronize()
    hs2.check_status()
    assert torch.equal(got, eager)


def test_host_pipeline_steps_each_match_their_inputs():
    B, K, n = 2, 128, 5
    t = synth.make_inputs(synth.small_workload(B, [400, 300], k=K, K=K, S_cap=512), seed=73)
    d = _dev(t)
    pipe = mla.HostDecodePipeline(B, K)
    ins, outs, keep = [], [], []                 # keep: the pinned inputs stay alive until finish()
    hp, ht, he = t["q_pe"].pin_memory(), t["topk_idx"].pin_memory(), t["end_pos"].pin_memory()
    for i in range(n):
        f = float(i + 1) * (-1) ** i              # a different query per step
        q = (t["q_nope"].float() * f).to(torch.bfloat16)
        ins.append(q)
        keep.append(q.pin_memory())
        outs.append(torch.empty(B, 128, 128, dtype=torch.float32).pin_memory())
        pipe.submit(keep[-1], hp, ht, he, d["kv_cache"], d["pe_cache"], d["wkv_b"], outs[-1])
    pipe.finish()
    torch.cuda.synchronize()
    pipe.check_status()
    x = U.oracle_inputs(t)
    for i in range(n):
        x["q_nope"] = synth.to_f64(ins[i])
        U.assert_attn_close(outs[i].numpy(), U.oracle_out(x, list(range(B))), f"pipeline step {i}")


def test_maximum_batch_of_query_rows():
    # B = 4096 query rows (the ABI's limit): absorption and up-projection take
    # 32 passes of 128 sequences, the attention grid 8192 CTAs; short caches
    B, S, K = 4096, 64, 64
    t = synth.make_inputs(synth.small_workload(B, [1 + (37 * b) % 64 for b in range(B)], k=40, K=K, S_cap=S),
                          seed=83, threads=16)
    d = _dev(t)
    step = mla.DecodeStep(B, K)
    out = step(d["q_nope"], d["q_pe"], d["kv_cache"], d["pe_cache"], d["wkv_b"], d["topk_idx"], d["end_pos"])
    torch.cuda.synchronize()
    step.check_status()
    got = out.cpu().numpy()
    x = U.oracle_inputs(t)
    bs = [0, 1, 127, 128, 129, 2047, 2048, 4094, 4095] + list(range(1000, 4096, 331))
    U.assert_attn_close(got[bs], U.oracle_out(x, bs), "B=4096 sampled sequences")
    with pytest.raises(mla.MLAError):
        mla.DecodeStep(B + 1, K)                # one row past the limit: no workspace size


def test_captured_host_pipeline_steps_match_their_inputs():
    # the end-to-end path bench.py times: each step one graph replay that copies
    # the step's pinned host inputs in and its bf16 head outputs back
    B, K, n = 3, 256, 5
    t = synth.make_inputs(synth.small_workload(B, [700, 256, 1000], k=K, K=K, S_cap=1024), seed=77)
    d = _dev(t)
    pipe = mla.CapturedHostPipeline(B, K, d["kv_cache"], d["pe_cache"], d["wkv_b"])
    x = U.oracle_inputs(t)
    for i in range(n):
        f = float(i + 1) * (-1) ** i              # a different query per step
        h = pipe.host_inputs(i)
        h["q_nope"].copy_((t["q_nope"].float() * f).to(torch.bfloat16))
        for name in ("q_pe", "topk_idx", "end_pos"):
            h[name].copy_(t[name])
        pipe.submit()
        pipe.finish()
        torch.cuda.synchronize()
        pipe.check_status()
        out = pipe.host_output(i)
        assert out.dtype == torch.bfloat16 and out.is_pinned()
        x["q_nope"] = synth.to_f64(h["q_nope"])
        ora = U.oracle_out(x, list(range(B)))
        # bf16 head outputs: the attention tolerance plus one bf16 rounding
        got = out.double().numpy()
        U.assert_attn_close(got, ora, f"captured pipeline step {i}")


def test_fused_decode_step_matches_the_oracle_chain():
    # one new token per sequence, from its hidden state to the block output:
    # wkv_a projection -> cache append -> absorption -> attention with the
    # up-projection -> wo projection, eager and captured in one graph
    B, K, S, dim = 4, 256, 1024, 1024
    ends = [301, 513, 1001, 4]                    # counts the new token
    t = synth.make_inputs(synth.small_workload(B, ends, k=K, K=K, S_cap=S), seed=97)
    t["topk_idx"][:, 0] = t["end_pos"] - 1          # the new token is selected
    x, wkv_a = synth.make_linear_inputs(98, B, 576, dim, name="wkv_a")
    _, wo = synth.make_linear_inputs(99, 1, dim, 128 * 128, name="wo")
    g = torch.Generator().manual_seed(100)
    norm_w = (1.0 + 0.1 * torch.randn(512, generator=g)).to(torch.bfloat16).float()
    d = _dev(t)
    kv0, pe0 = d["kv_cache"].clone(), d["pe_cache"].clone()
    dx, dwa, dwo, dnw = x.cuda(), wkv_a.cuda(), wo.cuda(), norm_w.cuda()
    step = mla.FusedDecodeStep(B, K, dim)
    args = (dx, d["q_nope"], d["q_pe"], d["kv_cache"], d["pe_cache"], dwa, dnw, d["wkv_b"], dwo, d["topk_idx"],
            d["end_pos"])
    y = step(*args).clone()
    torch.cuda.synchronize()
    step.check_status()
    # the oracle chain, rounding to bf16 where the path stores bf16 (the kv_a
    # projection, the cache rows, the head outputs)
    xo = U.oracle_inputs(t)
    kv_a = O.round_to_bf16(O.linear(synth.to_f64(x), synth.to_f64(wkv_a)))
    pos, lat, rot = O.cache_rows(kv_a[:, None], norm_w.double().numpy(), 1e-6, xo["end_pos"], U.INV_FREQ)
    kvc, pec = xo["kv_cache"].copy(), xo["pe_cache"].copy()
    for b in range(B):
        kvc[b, pos[b, 0]] = O.round_to_bf16(lat[b, 0])
        pec[b, pos[b, 0]] = O.round_to_bf16(rot[b, 0])
    heads = O.decode_step(xo["q_nope"], xo["q_pe"], kvc, pec, xo["wkv_b"], xo["topk_idx"], xo["end_pos"],
                          U.INV_FREQ, U.SCALE)
    wod = synth.to_f64(wo)
    ora = O.output_projection(O.round_to_bf16(heads), wod)
    mag = O.output_projection(np.abs(heads), np.abs(wod))
    err = np.abs(y.cpu().double().numpy() - ora)
    # the attention tolerance carried through wo: an element of a sequence's
    # head outputs may be off by 2e-2 of that sequence's largest head output,
    # and the errors sum to at most 5e-3 of the outputs' magnitude; plus the
    # bf16 rounding of y (2^-9 relative)
    maxh = np.abs(heads).reshape(B, -1).max(axis=1)
    bound = 2e-2 * maxh[:, None] * np.abs(wod).sum(axis=1)[None, :] + 2.0 ** -8 * np.abs(ora) + 1e-4
    assert np.all(err <= bound), float(np.max(err / bound))
    assert err.sum() / mag.sum() <= 5e-3 + 2.0 ** -9, float(err.sum() / mag.sum())
    # the same step captured in one CUDA graph replays to the same result
    d["kv_cache"].copy_(kv0)
    d["pe_cache"].copy_(pe0)
    gstep = mla.CapturedStep(step, *args)
    d["kv_cache"].copy_(kv0)
    d["pe_cache"].copy_(pe0)
    yg = gstep().clone()
    torch.cuda.synchronize()
    step.check_status()
    assert torch.equal(yg, y)
    assert gstep.kernels_per_replay >= 5
