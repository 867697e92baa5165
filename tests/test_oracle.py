"""Pins of the float64 oracle against facts that do not come from the oracle
itself: values printed or fixed by the pages, closed forms, invariants,
brute force on a toy, and special cases that reduce to something simpler.

CPU only (no GPU needed)."""
import math
import os

import numpy as np
import pytest
import torch

from oracle import mla_oracle as O
from sparse_latent_attention_decode_b300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_pairs(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, v = line.split()
            vals[k] = v
    return vals


ARGS = _read_pairs("model_args_defaults.txt")
ROPE_KW = dict(rope_dim=int(ARGS["qk_rope_head_dim"]), rope_theta=float(ARGS["rope_theta"]),
               rope_factor=float(ARGS["rope_factor"]), beta_fast=float(ARGS["beta_fast"]),
               beta_slow=float(ARGS["beta_slow"]), original_seq_len=int(ARGS["original_seq_len"]),
               max_seq_len=int(ARGS["max_seq_len"]))


def _f64(t):
    return synth.to_f64(t)


# ---------------------------------------------------------------- frequencies
def test_yarn_correction_range_matches_hand_derivation():
    g = _read_pairs("yarn_inv_freq_closed_form.txt")
    low, high = O.yarn_correction_range(32, 1, 64, 10000.0, 4096)
    assert (low, high) == (int(g["low"]), int(g["high"]))


def test_yarn_inv_freq_closed_form_values():
    g = _read_pairs("yarn_inv_freq_closed_form.txt")
    f = O.yarn_inv_freq(**ROPE_KW)
    assert f.shape == (32,)
    for k, v in g.items():
        if k in ("low", "high"):
            continue
        assert f[int(k)] == pytest.approx(float(v), rel=1e-14), k


def test_yarn_inv_freq_piecewise_closed_form_all_pairs():
    # unchanged below the ramp, divided by the factor above it, linear blend between
    f = O.yarn_inv_freq(**ROPE_KW)
    for i in range(32):
        base = 10.0 ** (-i / 8.0)
        if i <= 10:
            want = base
        elif i >= 23:
            want = base / 40.0
        else:
            want = base * ((i - 10) / 520.0 + (23 - i) / 13.0)
        assert f[i] == pytest.approx(want, rel=1e-13), i


def test_no_yarn_when_context_not_extended():
    kw = dict(ROPE_KW, max_seq_len=4096)
    f = O.yarn_inv_freq(**kw)
    np.testing.assert_allclose(f, 10.0 ** (-np.arange(32) / 8.0), rtol=1e-14)


def test_softmax_scale_closed_form():
    g = _read_pairs("softmax_scale_closed_form.txt")
    assert O.softmax_scale() == pytest.approx(float(g["softmax_scale"]), rel=1e-15)
    assert O.softmax_scale(max_seq_len=4096) == pytest.approx(float(g["softmax_scale_no_yarn"]), rel=1e-15)
    assert O.softmax_scale(max_seq_len=4096) == pytest.approx(1.0 / math.sqrt(192.0), rel=1e-15)


# ---------------------------------------------------------------- RoPE
def test_rope_unit_vector_lands_on_cos_sin_interleaved():
    # e_{2i} rotated by angle th must become (cos th, sin th) in slots (2i, 2i+1):
    # pins the interleaved pairing and the sign of the rotation
    f = O.yarn_inv_freq(**ROPE_KW)
    t = 16383
    for i in (0, 5, 10, 17, 31):
        x = np.zeros(64)
        x[2 * i] = 1.0
        y = O.rope_interleaved(x, O.freqs_cis([t], f)[0])
        th = t * f[i]
        assert y[2 * i] == pytest.approx(math.cos(th), abs=1e-12)
        assert y[2 * i + 1] == pytest.approx(math.sin(th), abs=1e-12)
        rest = np.delete(y, [2 * i, 2 * i + 1])
        assert np.all(rest == 0.0)
        # the odd slot rotates the other way round: e_{2i+1} -> (-sin, cos)
        x = np.zeros(64)
        x[2 * i + 1] = 1.0
        y = O.rope_interleaved(x, O.freqs_cis([t], f)[0])
        assert y[2 * i] == pytest.approx(-math.sin(th), abs=1e-12)
        assert y[2 * i + 1] == pytest.approx(math.cos(th), abs=1e-12)


def test_rope_preserves_pair_norms_and_identity_at_zero():
    rng = np.random.default_rng(0)
    f = O.yarn_inv_freq(**ROPE_KW)
    x = rng.standard_normal((7, 128, 64))
    pos = np.array([0, 1, 999, 1000, 4095, 8191, 16383])
    y = O.rope_interleaved(x, O.freqs_cis(pos, f)[:, None, :])
    nx = np.hypot(x[..., 0::2], x[..., 1::2])
    ny = np.hypot(y[..., 0::2], y[..., 1::2])
    np.testing.assert_allclose(ny, nx, rtol=1e-13)
    np.testing.assert_array_equal(y[0], x[0])


def test_rope_composition_law():
    f = O.yarn_inv_freq(**ROPE_KW)
    a, b = 1234, 15000 - 1234
    ca, cb, cab = O.freqs_cis([a], f)[0], O.freqs_cis([b], f)[0], O.freqs_cis([a + b], f)[0]
    np.testing.assert_allclose(ca * cb, cab, atol=1e-11)


def test_rope_low_pairs_rotate_by_unscaled_frequency():
    # pairs i <= 10 sit below the YaRN ramp: angle = t * 10000^(-i/32)
    f = O.yarn_inv_freq(**ROPE_KW)
    t = 16383
    c = O.freqs_cis([t], f)[0]
    for i in range(11):
        th = t * 10000.0 ** (-i / 32.0)
        assert c[i] == pytest.approx(complex(math.cos(th), math.sin(th)), abs=1e-10)


# ---------------------------------------------------------------- attention
def _small_case(B=2, end_pos=(300, 257), k=100, S_cap=320, seed=1, selection="uniform"):
    wl = synth.small_workload(B, list(end_pos), k=k, K=k, S_cap=S_cap, selection=selection)
    t = synth.make_inputs(wl, seed=seed)
    return wl, {n: _f64(v) for n, v in t.items()}


def test_worked_example_shapes():
    g = _read_pairs("worked_example_p1000.txt")
    wl = synth.workload("p1000_b1")
    assert wl.end_pos[0] == int(g["keys_read"]) == int(g["cached_positions"]) + 1
    x = {n: _f64(v) for n, v in synth.make_inputs(wl).items()}
    f = O.yarn_inv_freq(**ROPE_KW)
    q_lat = O.q_latent(x["q_nope"], x["q_pe"], x["wkv_b"], x["end_pos"], f)
    assert q_lat.shape == (1, int(g["heads"]), int(g["q_width"]))
    assert x["kv_cache"].shape[-1] + x["pe_cache"].shape[-1] == int(g["k_width"])
    _, p = O.attend_one(q_lat[0, :, :512], q_lat[0, :, 512:], x["kv_cache"][0], x["pe_cache"][0],
                        x["topk_idx"][0], int(x["end_pos"][0]), O.softmax_scale(), return_probs=True)
    assert p.shape == (int(g["heads"]), int(g["keys_read"]))


def test_softmax_rows_sum_to_one():
    wl, x = _small_case()
    f = O.yarn_inv_freq(**ROPE_KW)
    q_lat = O.q_latent(x["q_nope"], x["q_pe"], x["wkv_b"], x["end_pos"], f)
    for b in range(wl.B):
        _, p = O.attend_one(q_lat[b, :, :512], q_lat[b, :, 512:], x["kv_cache"][b], x["pe_cache"][b],
                            x["topk_idx"][b], wl.end_pos[b], O.softmax_scale(), return_probs=True)
        np.testing.assert_allclose(p.sum(axis=1), 1.0, atol=1e-12)
        unsel = np.ones(wl.end_pos[b], bool)
        unsel[x["topk_idx"][b][x["topk_idx"][b] >= 0]] = False
        assert np.all(p[:, unsel] == 0.0)


def test_absorbed_equals_naive_non_absorbed_at_p1000():
    # the pages' worked example (1001 keys, all selected): absorbing W_UK into the
    # query and W_UV into the output must equal ordinary per-head attention over
    # keys/values expanded from the latent cache
    wl = synth.workload("p1000_b1")
    x = {n: _f64(v) for n, v in synth.make_inputs(wl).items()}
    f = O.yarn_inv_freq(**ROPE_KW)
    s = O.softmax_scale()
    out = O.decode_step(x["q_nope"], x["q_pe"], x["kv_cache"], x["pe_cache"], x["wkv_b"],
                        x["topk_idx"], x["end_pos"], f, s)
    q_pe_rot = O.rope_for_batch(x["q_pe"], x["end_pos"], f)
    naive = O.naive_attention_one(x["q_nope"][0], q_pe_rot[0], x["kv_cache"][0], x["pe_cache"][0],
                                  x["wkv_b"], x["topk_idx"][0], 1001, s)
    np.testing.assert_allclose(out[0], naive, rtol=0, atol=1e-12 * np.abs(naive).max())


def test_absorbed_equals_naive_with_sparse_selection():
    wl, x = _small_case(B=1, end_pos=(300,), k=37)
    f = O.yarn_inv_freq(**ROPE_KW)
    s = O.softmax_scale()
    out = O.decode_step(x["q_nope"], x["q_pe"], x["kv_cache"], x["pe_cache"], x["wkv_b"],
                        x["topk_idx"], x["end_pos"], f, s)
    q_pe_rot = O.rope_for_batch(x["q_pe"], x["end_pos"], f)
    naive = O.naive_attention_one(x["q_nope"][0], q_pe_rot[0], x["kv_cache"][0], x["pe_cache"][0],
                                  x["wkv_b"], x["topk_idx"][0], 300, s)
    np.testing.assert_allclose(out[0], naive, rtol=0, atol=1e-12 * np.abs(naive).max())


def test_brute_force_toy_4_heads_8_keys():
    rng = np.random.default_rng(3)
    q_lat = rng.standard_normal((128, 576))
    kv = rng.standard_normal((8, 512))
    pe = rng.standard_normal((8, 64))
    topk = np.array([6, 1, -1, 3, 7, 0, 8, 4])   # -1 and 8 are padding for end_pos = 8
    s = O.softmax_scale()
    o = O.attend_one(q_lat[:, :512], q_lat[:, 512:], kv, pe, topk, 8, s)
    bf = O.brute_force_toy(q_lat, kv, pe, topk, 8, s, heads=range(4))
    for h in range(4):
        np.testing.assert_allclose(o[h], bf[h], rtol=0, atol=1e-13)


def test_single_selected_key_gives_value_projection_of_that_row():
    wl, x = _small_case(B=1, end_pos=(300,), k=1)
    f = O.yarn_inv_freq(**ROPE_KW)
    out = O.decode_step(x["q_nope"], x["q_pe"], x["kv_cache"], x["pe_cache"], x["wkv_b"],
                        x["topk_idx"], x["end_pos"], f, O.softmax_scale())
    t = int(x["topk_idx"][0][0])
    w_uv = x["wkv_b"].reshape(128, 256, 512)[:, 128:, :]
    want = np.einsum("hdc,c->hd", w_uv, x["kv_cache"][0][t])
    np.testing.assert_allclose(out[0], want, rtol=0, atol=1e-12 * np.abs(want).max())


def test_zero_query_averages_selected_rows():
    wl, x = _small_case(B=1, end_pos=(300,), k=50)
    x["q_nope"][:] = 0.0
    x["q_pe"][:] = 0.0
    f = O.yarn_inv_freq(**ROPE_KW)
    out = O.decode_step(x["q_nope"], x["q_pe"], x["kv_cache"], x["pe_cache"], x["wkv_b"],
                        x["topk_idx"], x["end_pos"], f, O.softmax_scale())
    sel = x["topk_idx"][0]
    mean = x["kv_cache"][0][sel].mean(axis=0)
    w_uv = x["wkv_b"].reshape(128, 256, 512)[:, 128:, :]
    want = np.einsum("hdc,c->hd", w_uv, mean)
    np.testing.assert_allclose(out[0], want, rtol=0, atol=1e-12 * np.abs(want).max())


def test_permutation_duplicates_padding_and_nan_poison():
    wl, x = _small_case(B=1, end_pos=(300,), k=64)
    f = O.yarn_inv_freq(**ROPE_KW)
    s = O.softmax_scale()
    q_lat = O.q_latent(x["q_nope"], x["q_pe"], x["wkv_b"], x["end_pos"], f)
    args = (q_lat[0, :, :512], q_lat[0, :, 512:], x["kv_cache"][0], x["pe_cache"][0])
    row = x["topk_idx"][0]
    base = O.attend_one(*args, row, 300, s)
    perm = np.random.default_rng(5).permutation(row)
    np.testing.assert_allclose(O.attend_one(*args, perm, 300, s), base, rtol=0, atol=1e-14)
    dup = np.concatenate([row, row[:10], [-1, -7, 300, 10 ** 6]])
    np.testing.assert_allclose(O.attend_one(*args, dup, 300, s), base, rtol=0, atol=1e-14)
    kv = x["kv_cache"][0].copy()
    pe = x["pe_cache"][0].copy()
    unsel = np.ones(kv.shape[0], bool)
    unsel[row] = False
    kv[unsel] = np.nan
    pe[unsel] = np.nan
    # scores of unselected keys are NaN here, so compute through the selected rows only
    sub = O.attend_one(args[0], args[1], kv[row], pe[row], np.arange(64), 64, s)
    np.testing.assert_allclose(sub, base, rtol=0, atol=1e-13)


def test_sparse_equals_dense_over_gathered_subcache():
    wl, x = _small_case(B=1, end_pos=(300,), k=80)
    f = O.yarn_inv_freq(**ROPE_KW)
    s = O.softmax_scale()
    q_lat = O.q_latent(x["q_nope"], x["q_pe"], x["wkv_b"], x["end_pos"], f)
    row = x["topk_idx"][0]
    base = O.attend_one(q_lat[0, :, :512], q_lat[0, :, 512:], x["kv_cache"][0], x["pe_cache"][0], row, 300, s)
    # plain dense softmax attention (no mask) over the gathered rows
    kv = x["kv_cache"][0][row]
    pe = x["pe_cache"][0][row]
    sc = (q_lat[0, :, :512] @ kv.T + q_lat[0, :, 512:] @ pe.T) * s
    p = np.exp(sc - sc.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    np.testing.assert_allclose(p @ kv, base, rtol=0, atol=1e-13)


def test_empty_selection_gives_zero():
    wl, x = _small_case(B=1, end_pos=(300,), k=10)
    row = np.full(10, -1)
    f = O.yarn_inv_freq(**ROPE_KW)
    q_lat = O.q_latent(x["q_nope"], x["q_pe"], x["wkv_b"], x["end_pos"], f)
    o = O.attend_one(q_lat[0, :, :512], q_lat[0, :, 512:], x["kv_cache"][0], x["pe_cache"][0], row, 300,
                     O.softmax_scale())
    assert np.all(o == 0.0)


# ------------------------------------------------- planted mistakes must be caught
def test_pins_catch_swapped_weight_halves(monkeypatch):
    wl, x = _small_case(B=1, end_pos=(300,), k=37)
    f = O.yarn_inv_freq(**ROPE_KW)
    s = O.softmax_scale()
    q_pe_rot = O.rope_for_batch(x["q_pe"], x["end_pos"], f)
    naive = O.naive_attention_one(x["q_nope"][0], q_pe_rot[0], x["kv_cache"][0], x["pe_cache"][0],
                                  x["wkv_b"], x["topk_idx"][0], 300, s)
    real_split = O.split_wkv_b
    monkeypatch.setattr(O, "split_wkv_b", lambda w: real_split(w)[::-1])
    bad = O.decode_step(x["q_nope"], x["q_pe"], x["kv_cache"], x["pe_cache"], x["wkv_b"],
                        x["topk_idx"], x["end_pos"], f, s)
    monkeypatch.setattr(O, "split_wkv_b", real_split)
    assert np.abs(bad[0] - naive).max() > 1e-3 * np.abs(naive).max()


def test_pins_catch_non_interleaved_pairing(monkeypatch):
    def half_split(x, cis):
        z = x[..., :32] + 1j * x[..., 32:]
        y = z * cis
        return np.concatenate([y.real, y.imag], axis=-1)
    monkeypatch.setattr(O, "rope_interleaved", half_split)
    with pytest.raises(AssertionError):
        test_rope_unit_vector_lands_on_cos_sin_interleaved()


# ------------------------------------------------- half-split (indexer) rotary layout
def test_half_split_rope_unit_vectors():
    # e_i (i < 32) becomes cos at slot i and sin at slot i + 32; e_(i+32) becomes
    # -sin at slot i and cos at slot i + 32 (multiplication by exp(j theta))
    f = O.yarn_inv_freq(**ROPE_KW)
    t = 4095
    cis = O.freqs_cis([t], f)[0]
    for i in (0, 5, 10, 11, 23, 31):
        th = t * f[i]
        e = np.zeros(64)
        e[i] = 1.0
        y = O.rope_half_split(e, cis)
        want = np.zeros(64)
        want[i], want[i + 32] = math.cos(th), math.sin(th)
        assert np.allclose(y, want, atol=1e-13)
        e = np.zeros(64)
        e[i + 32] = 1.0
        y = O.rope_half_split(e, cis)
        want = np.zeros(64)
        want[i], want[i + 32] = -math.sin(th), math.cos(th)
        assert np.allclose(y, want, atol=1e-13)


def test_half_split_rope_is_the_interleaved_rotation_of_the_regrouped_pairs():
    # moving feature i + 32 next to feature i turns the half-split layout into the
    # interleaved one; the rotation must commute with that regrouping
    rng = np.random.default_rng(3)
    x = rng.standard_normal((5, 64, 64))
    f = O.yarn_inv_freq(**ROPE_KW)
    cis = O.freqs_cis(np.arange(5) * 1000 + 7, f)[:, None, :]
    inter = np.empty_like(x)
    inter[..., 0::2], inter[..., 1::2] = x[..., :32], x[..., 32:]
    y_int = O.rope_interleaved(inter, cis)
    back = np.concatenate([y_int[..., 0::2], y_int[..., 1::2]], axis=-1)
    assert np.allclose(O.rope_half_split(x, cis), back, atol=1e-12)
    # pair norms (x[i], x[i+32]) are preserved, position 0 is the identity
    y = O.rope_half_split(x, cis)
    assert np.allclose(np.hypot(y[..., :32], y[..., 32:]), np.hypot(x[..., :32], x[..., 32:]), atol=1e-12)
    assert np.allclose(O.rope_half_split(x, O.freqs_cis([0], f)[0]), x, atol=1e-15)


def test_rope_for_positions_selects_the_layout():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((3, 64, 64))
    end = np.array([1, 2049, 16384])
    f = O.yarn_inv_freq(**ROPE_KW)
    cis = O.freqs_cis(end - 1, f)[:, None, :]
    assert np.array_equal(O.rope_for_positions(x, end, f, interleaved=True), O.rope_interleaved(x, cis))
    assert np.array_equal(O.rope_for_positions(x, end, f, interleaved=False), O.rope_half_split(x, cis))
    assert np.array_equal(O.rope_for_positions(x, end, f), O.rope_for_batch(x, end, f))


def test_pins_catch_interleaved_pairing_in_the_half_split_layout(monkeypatch):
    monkeypatch.setattr(O, "rope_half_split", O.rope_interleaved)
    with pytest.raises(AssertionError):
        test_half_split_rope_unit_vectors()


# ----------------------------------------------------------------- fp8 weights
def test_e4m3_decode_matches_torch_for_every_code():
    codes = np.arange(256)
    got = O.e4m3_decode(codes)
    ref = torch.tensor(codes, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(got[~np.isnan(got)], ref[~np.isnan(ref)])
    # sign of zero
    assert np.signbit(got[0x80]) and not np.signbit(got[0x00])


def test_e4m3_decode_closed_form_codes():
    # values fixed by the format: bias 7, 3 mantissa bits, no infinities
    want = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 / 8 * 2.0 ** -6, 0x08: 2.0 ** -6, 0x38: 1.0, 0x39: 1.125,
            0x40: 2.0, 0x7E: 448.0, 0xFE: -448.0, 0xB8: -1.0, 0x30: 0.5}
    got = O.e4m3_decode(list(want))
    assert np.array_equal(got, np.array(list(want.values())))
    assert np.isnan(O.e4m3_decode([0x7F, 0xFF])).all()


def test_dequant_block_maps_tiles_to_their_multiplier():
    # ragged 200 x 300 with block 128: a 2 x 3 grid of distinct powers of two
    scale = np.array([[1.0, 2.0, 4.0], [8.0, 16.0, 32.0]])
    codes = np.full((200, 300), 0x38)            # every code is 1.0
    w = O.dequant_block_fp8(codes, scale, block=128)
    for r, c in [(0, 0), (127, 127), (128, 0), (0, 128), (199, 299), (127, 256), (128, 255)]:
        assert w[r, c] == scale[r // 128, c // 128]
    codes = np.full((4, 6), 0xC0)                # -2.0, block 2: grid 2 x 3
    w = O.dequant_block_fp8(codes, np.arange(1, 7, dtype=np.float64).reshape(2, 3), block=2)
    assert np.array_equal(w, -2.0 * np.repeat(np.repeat(np.arange(1, 7).reshape(2, 3), 2, 0), 2, 1))


def test_round_to_bf16_matches_torch_and_breaks_ties_to_even():
    x = np.random.default_rng(1).standard_normal(50000).astype(np.float32) * 3.0
    ref = torch.tensor(x).to(torch.bfloat16).double().numpy()
    assert np.array_equal(O.round_to_bf16(x.astype(np.float64)), ref)
    ulp = 2.0 ** -7
    assert O.round_to_bf16(1 + ulp / 2) == 1.0                 # tie, 1.0 is even
    assert O.round_to_bf16(1 + 3 * ulp / 2) == 1 + 2 * ulp     # tie, rounds up to even
    assert O.round_to_bf16(-(1 + 3 * ulp / 2)) == -(1 + 2 * ulp)
    assert O.round_to_bf16(2 - ulp / 4) == 2.0                 # carries into the next binade


def test_dequant_to_bf16_is_within_the_rounding_bound_of_the_exact_product():
    codes, scale = synth.make_fp8_weight(3, rows=300, cols=260, block=128)
    exact = O.dequant_block_fp8(codes.numpy(), scale.numpy().astype(np.float64), block=128)
    b16 = O.dequant_to_bf16(codes.numpy(), scale.numpy(), block=128)
    # half a bf16 ulp (2^-8 relative at most) plus the float32 rounding before it
    assert np.all(np.abs(b16 - exact) <= (2.0 ** -8 + 2.0 ** -23) * np.abs(exact))
    # every result is a bf16 value
    assert np.array_equal(b16, O.round_to_bf16(b16))


def test_fp8_synth_weight_spans_the_code_range():
    codes, scale = synth.make_fp8_weight(0, rows=256, cols=512)
    v = O.e4m3_decode(codes.numpy())
    assert not np.isnan(v).any()
    assert np.abs(v).max() == 448.0 and (np.abs(v) < 2.0 ** -6).any()     # saturated and subnormal codes
    assert scale.shape == (2, 4) and (scale > 0).all()


# ----------------------------------------------------------------- cache append
U_INV_FREQ = O.yarn_inv_freq()

def test_rms_norm_worked_values_and_invariants():
    got = O.rms_norm(np.array([3.0, 4.0]), np.array([1.0, 2.0]), 0.0)
    # mean of squares 12.5: 3 / sqrt(12.5) and 2 * 4 / sqrt(12.5)
    assert np.allclose(got, [0.848528137423857, 2.262741699796952], rtol=0, atol=1e-15)
    x = np.random.default_rng(2).standard_normal((5, 512))
    y = O.rms_norm(x, np.ones(512), 0.0)
    assert np.allclose(np.mean(y * y, axis=-1), 1.0, rtol=0, atol=1e-13)        # unit RMS
    assert np.allclose(O.rms_norm(7.5 * x, np.ones(512), 0.0), y, rtol=1e-14)  # scale invariance
    assert np.array_equal(O.rms_norm(np.zeros(512), np.ones(512), 1e-6), np.zeros(512))
    c = O.rms_norm(np.full(512, -0.25), np.full(512, 3.0), 0.0)
    assert np.allclose(c, -3.0, rtol=1e-15)


def test_cache_rows_positions_and_rotary_key_properties():
    rng = np.random.default_rng(4)
    B, T = 2, 3
    kv_a = rng.standard_normal((B, T, 576))
    w = rng.standard_normal(512)
    pos, lat, rot = O.cache_rows(kv_a, w, 1e-6, [5, 10], U_INV_FREQ)
    assert np.array_equal(pos, [[2, 3, 4], [7, 8, 9]])
    assert np.allclose(lat, O.rms_norm(kv_a[..., :512], w, 1e-6))
    # a rotation: norms of the rotary key are kept
    assert np.allclose(np.linalg.norm(rot, axis=-1), np.linalg.norm(kv_a[..., 512:], axis=-1), rtol=1e-13)
    # a query and a key rotated at positions p and t score by p - t alone
    q = rng.standard_normal(64)
    k = kv_a[0, 0, 512:]
    def score(p, t):
        qr = O.rope_for_positions(q[None, None, :], [p + 1], U_INV_FREQ)[0, 0]
        kr = O.cache_rows(np.concatenate([np.ones(512), k])[None, None, :], w, 1e-6, [t + 1], U_INV_FREQ)[2][0, 0]
        return qr @ kr
    assert abs(score(4, 4) - q @ k) < 1e-12
    assert abs(score(9000, 8990) - score(10, 0)) < 1e-9
    assert abs(score(9000, 8990) - score(10, 1)) > 1e-6


def test_same_position_pin_catches_a_key_rotated_in_the_other_layout():
    rng = np.random.default_rng(6)
    q, k = rng.standard_normal(64), rng.standard_normal(64)
    cis = O.freqs_cis(np.array([99]), U_INV_FREQ)[0]
    qr = O.rope_for_positions(q[None, None, :], [100], U_INV_FREQ)[0, 0]
    kr_good = O.cache_rows(np.concatenate([np.ones(512), k])[None, None, :], np.ones(512), 0.0, [100],
                           U_INV_FREQ)[2][0, 0]
    kr_bad = O.rope_half_split(k, cis)
    assert abs(qr @ kr_good - q @ k) < 1e-12
    assert abs(qr @ kr_bad - q @ k) > 1e-3


# ----------------------------------------------------------------- multi-token decode
def _tok_case(T, seed=9, end=(300, 41)):
    wl = synth.small_workload(len(end), list(end), k=40, K=40, S_cap=320)
    t = synth.make_token_inputs(wl, T, seed=seed)
    return {k: synth.to_f64(v) for k, v in t.items()}


def test_one_token_decode_is_the_single_token_step():
    x = _tok_case(1)
    got = O.decode_tokens(x["q_nope"], x["q_pe"], x["kv_cache"], x["pe_cache"], x["wkv_b"], x["topk_idx"],
                          x["end_pos"], U_INV_FREQ, O.softmax_scale())
    ref = O.decode_step(x["q_nope"][:, 0], x["q_pe"][:, 0], x["kv_cache"], x["pe_cache"], x["wkv_b"],
                        x["topk_idx"][:, 0], x["end_pos"], U_INV_FREQ, O.softmax_scale())
    assert np.allclose(got[:, 0], ref, rtol=1e-12, atol=1e-12)


def test_each_token_is_a_single_token_step_at_its_own_position():
    T = 4
    x = _tok_case(T)
    got = O.decode_tokens(x["q_nope"], x["q_pe"], x["kv_cache"], x["pe_cache"], x["wkv_b"], x["topk_idx"],
                          x["end_pos"], U_INV_FREQ, O.softmax_scale())
    for s in range(T):
        ep = x["end_pos"] - T + s + 1
        ref = O.decode_step(x["q_nope"][:, s], x["q_pe"][:, s], x["kv_cache"], x["pe_cache"], x["wkv_b"],
                            x["topk_idx"][:, s], ep, U_INV_FREQ, O.softmax_scale())
        assert np.allclose(got[:, s], ref, rtol=1e-12, atol=1e-12), s


def test_multi_token_outputs_are_causal():
    T = 3
    x = _tok_case(T, end=(60,))
    x["topk_idx"][0, :, :3] = [57, 58, 59]               # every token selects the three new positions
    args = lambda: (x["q_nope"], x["q_pe"], x["kv_cache"], x["pe_cache"], x["wkv_b"], x["topk_idx"],
                    x["end_pos"], U_INV_FREQ, O.softmax_scale())
    before = O.decode_tokens(*args())
    x["kv_cache"][0, 59] *= -3.0                          # the last token's own row
    x["pe_cache"][0, 59] += 1.0
    after = O.decode_tokens(*args())
    assert np.array_equal(before[0, :2], after[0, :2])    # tokens at 57 and 58 cannot see position 59
    assert not np.allclose(before[0, 2], after[0, 2])


def test_position_pin_catches_tokens_placed_at_the_last_position(monkeypatch):
    # plant: every token placed at end_pos - 1 (no causal mask, one rotation)
    T = 3
    x = _tok_case(T, end=(60,))
    x["topk_idx"][0, :, :3] = [57, 58, 59]
    monkeypatch.setattr(O, "token_positions", lambda end_pos, T: int(end_pos) - 1 + 0 * np.arange(T))
    got = O.decode_tokens(x["q_nope"], x["q_pe"], x["kv_cache"], x["pe_cache"], x["wkv_b"], x["topk_idx"],
                          x["end_pos"], U_INV_FREQ, O.softmax_scale())
    ref = O.decode_step(x["q_nope"][:, 0], x["q_pe"][:, 0], x["kv_cache"], x["pe_cache"], x["wkv_b"],
                        x["topk_idx"][:, 0], x["end_pos"] - T + 1, U_INV_FREQ, O.softmax_scale())
    assert not np.allclose(got[:, 0], ref, rtol=1e-12, atol=1e-12)


# ----------------------------------------------------------------- projections
def test_linear_against_loops_on_a_non_square_case():
    rng = np.random.default_rng(8)
    x, w = rng.standard_normal((3, 5)), rng.standard_normal((4, 5))
    want = np.array([[sum(x[m, k] * w[n, k] for k in range(5)) for n in range(4)] for m in range(3)])
    assert np.allclose(O.linear(x, w), want, rtol=1e-14, atol=1e-14)


def test_output_projection_flattens_head_major():
    heads = np.zeros((1, 128, 128))
    heads[0, 3, 7] = 1.0                       # head 3, feature 7 -> input column 3*128 + 7
    wo = np.zeros((5, 128 * 128))
    wo[2, 3 * 128 + 7] = 2.5
    wo[4, 7 * 128 + 3] = 9.0                   # the transposed position must not be picked up
    assert np.array_equal(O.output_projection(heads, wo), [[0, 0, 2.5, 0, 0]])
