"""Float64 CPU oracle for one decode step of absorbed, top-k-sparse latent attention.

TEST INFRASTRUCTURE ONLY.  This module exists to check the CUDA library; the
product never imports it.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may use it.  It shares
no code with the CUDA path: it takes plain numpy arrays (the seeded inputs,
already rounded to bf16 by the input generator and widened to float64) and
returns float64 arrays.

Everything is written as the plain definition the pages state, in float64, with
numpy's einsum / exp / cos / sin as the only library steps.  Sources (the five
DeepSeek-V3.2-Exp atlas pages):

* "Transformer blocks", RoPE coefficients panel, excerpt ``rope`` and excerpt
  ``model-args``: the frequency table and its YaRN blend, and the default
  arguments (max_seq_len 16384, original_seq_len 4096, rope_theta 1e4,
  rope_factor 40, beta_fast 32, beta_slow 1, mscale 1).
* "Rotated query part", excerpt ``apply-rope``: interleaved pair rotation.
* "Query heads", excerpt ``mla-init``: the softmax scale and its mscale factor.
* "Rotated query part" / "Query content heads" / "Attention weights", excerpt
  ``mla-decode``: absorption, scores, selection mask, softmax, PV and the
  value up-projection.

The pages omit the bodies of the two YaRN helpers (``find_correction_range``,
``linear_ramp_factor``); the closed forms used below are the standard YaRN
definitions, spelled out in ``yarn_inv_freq``.

Readings where the pages are silent (each is also listed in the design notes):
* per-sequence position: the query of sequence b sits at ``end_pos[b] - 1``
  (the Attention weights page: P cached positions, L = P + 1 keys read);
* selection entries that are negative or >= end_pos[b] are padding and are
  ignored; a sequence with nothing selected yields an all-zero output (the
  pages' softmax over an all -inf row would give NaN);
* the selection is a set (the mask is built by a scatter), so repeated indices
  count once.
"""
from __future__ import annotations

import math

import numpy as np

# Shapes of the attention block (Query heads page, excerpt mla-init; Attention
# weights page header: 128 heads, 576 = 512 latent + 64 rotary).
N_HEADS = 128
D_NOPE = 128
D_ROPE = 64
D_V = 128
KV_LORA = 512
D_QK = D_NOPE + D_ROPE  # 192


# --------------------------------------------------------------------------
# fp8 weights: e4m3 decoding and block dequantisation ("Rotated query part"
# page, excerpt mla-decode: weight_dequant(wkv_b.weight, wkv_b.scale), called
# once and kept as the wkv_b of the absorbed path).  The pages name the call
# only; the format is read as OCP FP8 E4M3 (sign, 4 exponent bits with bias 7,
# 3 mantissa bits, no infinities, S.1111.111 = NaN) with one multiplier per
# block x block tile.
# --------------------------------------------------------------------------
def e4m3_decode(codes) -> np.ndarray:
    """Value of each 8-bit E4M3 code, from the format's definition:
    exponent field 0 -> (-1)^s * m/8 * 2^-6 (subnormal); S.1111.111 -> NaN;
    otherwise (-1)^s * (1 + m/8) * 2^(e-7)."""
    c = np.asarray(codes, dtype=np.int64) & 0xFF
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    normal = (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0)
    sub = (m / 8.0) * 2.0 ** -6
    v = sign * np.where(e == 0, sub, normal)
    return np.where((c & 0x7F) == 0x7F, np.nan, v)


def dequant_block_fp8(codes, scale, block: int = 128) -> np.ndarray:
    """Exact dequantised weight: e4m3(codes[r, c]) * scale[r // block, c // block]
    in float64 (the product of a 4-bit and a 24-bit significand is exact)."""
    codes = np.asarray(codes)
    rows, cols = codes.shape
    s = np.asarray(scale, dtype=np.float64)
    assert s.shape == (-(-rows // block), -(-cols // block))
    s_full = np.repeat(np.repeat(s, block, axis=0), block, axis=1)[:rows, :cols]
    return e4m3_decode(codes) * s_full


def round_to_bf16(x) -> np.ndarray:
    """Round to the nearest bfloat16 (8 significant bits), ties to even, for
    values in the normal range; NaN stays NaN."""
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)                  # x = m * 2^e, 0.5 <= |m| < 1
    r = np.ldexp(np.rint(np.ldexp(m, 8)), e - 8)   # np.rint: ties to even
    return np.where(np.isfinite(x), r, x)


def dequant_to_bf16(codes, scale, block: int = 128) -> np.ndarray:
    """The bf16 weight the decode consumes.  The rounding decides a bit
    pattern, so it is taken in the precision of the library's dequantisation:
    the code times the multiplier rounded to float32, then to bf16."""
    codes = np.asarray(codes)
    rows, cols = codes.shape
    s = np.asarray(scale, dtype=np.float32)
    s_full = np.repeat(np.repeat(s, block, axis=0), block, axis=1)[:rows, :cols]
    p32 = e4m3_decode(codes).astype(np.float32) * s_full      # IEEE float32 product
    return round_to_bf16(p32.astype(np.float64))


# --------------------------------------------------------------------------
# a1: frequency table (Transformer blocks page, excerpts rope + model-args)
# --------------------------------------------------------------------------
def yarn_correction_dim(num_rotations: float, dim: int, base: float, original_seq_len: int) -> float:
    """Feature index whose wavelength completes ``num_rotations`` turns over the
    original context: dim * ln(L0 / (2*pi*n)) / (2 * ln(base)).  Standard YaRN
    definition (the helper body is omitted on the pages)."""
    return dim * math.log(original_seq_len / (num_rotations * 2.0 * math.pi)) / (2.0 * math.log(base))


def yarn_correction_range(beta_fast: float, beta_slow: float, dim: int, base: float,
                          original_seq_len: int) -> tuple[int, int]:
    """(low, high): floor / ceil of the correction dims, clamped to [0, dim-1]."""
    low = math.floor(yarn_correction_dim(beta_fast, dim, base, original_seq_len))
    high = math.ceil(yarn_correction_dim(beta_slow, dim, base, original_seq_len))
    return max(low, 0), min(high, dim - 1)


def yarn_inv_freq(rope_dim: int = 64, rope_theta: float = 10000.0, rope_factor: float = 40.0,
                  beta_fast: float = 32.0, beta_slow: float = 1.0, original_seq_len: int = 4096,
                  max_seq_len: int = 16384) -> np.ndarray:
    """Per-pair angular frequency f'_i, i = 0 .. rope_dim/2 - 1, in float64.

    f_i = 1 / theta^(2i / rope_dim).  When max_seq_len exceeds the original
    context, blend with the interpolated f_i / factor through the linear ramp
    r_i = clamp((i - low) / (high - low), 0, 1):  smooth = 1 - r,
    f'_i = f_i / factor * (1 - smooth) + f_i * smooth.
    """
    half = rope_dim // 2
    i = np.arange(half, dtype=np.float64)
    freqs = 1.0 / (rope_theta ** (2.0 * i / rope_dim))
    if max_seq_len > original_seq_len:
        low, high = yarn_correction_range(beta_fast, beta_slow, rope_dim, rope_theta, original_seq_len)
        hi = float(high)
        if low == high:
            hi += 0.001
        ramp = np.clip((i - low) / (hi - low), 0.0, 1.0)
        smooth = 1.0 - ramp
        freqs = freqs / rope_factor * (1.0 - smooth) + freqs * smooth
    return freqs


def freqs_cis(positions, inv_freq: np.ndarray) -> np.ndarray:
    """cis[t, i] = exp(j * t * f'_i) as complex128, for the given positions."""
    t = np.asarray(positions, dtype=np.float64)
    return np.exp(1j * np.outer(t, inv_freq))


# --------------------------------------------------------------------------
# a2: interleaved rotary embedding (Rotated query part, excerpt apply-rope)
# --------------------------------------------------------------------------
def rope_interleaved(x: np.ndarray, cis: np.ndarray) -> np.ndarray:
    """Rotate adjacent pairs (x[..., 2i], x[..., 2i+1]) as the complex number
    x[2i] + j x[2i+1] times cis[..., i].  ``cis`` broadcasts against x's leading
    dims with the pair axis last."""
    z = x[..., 0::2] + 1j * x[..., 1::2]
    y = z * cis
    out = np.empty(x.shape, dtype=np.float64)
    out[..., 0::2] = y.real
    out[..., 1::2] = y.imag
    return out


def rope_half_split(x: np.ndarray, cis: np.ndarray) -> np.ndarray:
    """The indexer's layout (apply-rope with interleaved=False, Rotated query
    part page): feature i and feature i + d/2 form the complex number
    x[i] + j x[i + d/2], which is multiplied by cis[..., i]; the real parts are
    written back to the first half and the imaginary parts to the second."""
    d2 = x.shape[-1] // 2
    z = x[..., :d2] + 1j * x[..., d2:]
    y = z * cis
    return np.concatenate([y.real, y.imag], axis=-1)


def rope_for_positions(x: np.ndarray, end_pos: np.ndarray, inv_freq: np.ndarray, interleaved: bool = True):
    """Rotate x [B, n_heads, 64] of each sequence at position end_pos[b] - 1, in
    the interleaved (query) or half-split (indexer) layout."""
    pos = np.asarray(end_pos, dtype=np.int64) - 1
    cis = freqs_cis(pos, inv_freq)[:, None, :]
    return rope_interleaved(x, cis) if interleaved else rope_half_split(x, cis)


# --------------------------------------------------------------------------
# softmax scale (Query heads page, excerpt mla-init)
# --------------------------------------------------------------------------
def softmax_scale(qk_head_dim: int = D_QK, max_seq_len: int = 16384, original_seq_len: int = 4096,
                  mscale: float = 1.0, rope_factor: float = 40.0) -> float:
    """qk_head_dim^-0.5, times mscale_y^2 with mscale_y = 0.1*mscale*ln(factor) + 1
    when the context is extended beyond the original length."""
    s = qk_head_dim ** -0.5
    if max_seq_len > original_seq_len:
        m = 0.1 * mscale * math.log(rope_factor) + 1.0
        s = s * m * m
    return s


# --------------------------------------------------------------------------
# a3: key absorption (mla-decode excerpt, first einsum)
# --------------------------------------------------------------------------
def split_wkv_b(wkv_b: np.ndarray):
    """wkv_b [H*256, 512] viewed [H, 256, 512]: rows 0..127 of each head are the
    key half W_UK, rows 128..255 the value half W_UV.  H follows the array (the
    step is independent per head, so a block of consecutive heads is a valid
    input)."""
    w = wkv_b.reshape(-1, D_NOPE + D_V, KV_LORA)
    return w[:, :D_NOPE, :], w[:, D_NOPE:, :]


def absorb(q_nope: np.ndarray, wkv_b: np.ndarray) -> np.ndarray:
    """q~[b,h,c] = sum_d q_nope[b,h,d] * W_UK[h,d,c]."""
    w_uk, _ = split_wkv_b(wkv_b)
    return np.einsum("bhd,hdc->bhc", q_nope, w_uk)


# --------------------------------------------------------------------------
# a4..a7: masked scores, softmax, PV (mla-decode excerpt)
# --------------------------------------------------------------------------
def selection_mask(topk_row: np.ndarray, end_pos: int) -> np.ndarray:
    """0 on the selected positions of [0, end_pos), -inf elsewhere (a scatter of
    zeros into a -inf row; padding entries outside [0, end_pos) are dropped)."""
    mask = np.full(end_pos, -np.inf)
    idx = np.asarray(topk_row, dtype=np.int64)
    idx = idx[(idx >= 0) & (idx < end_pos)]
    mask[idx] = 0.0
    return mask


def attend_one(q_abs: np.ndarray, q_pe_rot: np.ndarray, kv: np.ndarray, pe: np.ndarray,
               topk_row: np.ndarray, end_pos: int, scale: float, return_probs: bool = False):
    """One sequence: scores over all end_pos cached keys, selection mask added,
    softmax over keys, probability-weighted sum of the latent rows.

    q_abs [H,512], q_pe_rot [H,64], kv [>=end_pos,512], pe [>=end_pos,64].
    Returns o [H,512] (and the probabilities [H,end_pos] when asked)."""
    kv = kv[:end_pos]
    pe = pe[:end_pos]
    scores = (q_abs @ kv.T + q_pe_rot @ pe.T) * scale
    mask = selection_mask(topk_row, end_pos)
    if not np.isfinite(mask).any():
        o = np.zeros((q_abs.shape[0], kv.shape[1]))
        return (o, np.zeros_like(scores)) if return_probs else o
    sel = np.isfinite(mask)
    scores = scores + mask[None, :]
    m = scores[:, sel].max(axis=1, keepdims=True)
    e = np.zeros_like(scores)
    e[:, sel] = np.exp(scores[:, sel] - m)
    p = e / e.sum(axis=1, keepdims=True)
    # unselected keys carry probability exactly 0; restricting the product to the
    # selected rows keeps non-finite data in unselected rows out of the result
    o = p[:, sel] @ kv[sel]
    return (o, p) if return_probs else o


# --------------------------------------------------------------------------
# a8: value up-projection (mla-decode excerpt, last einsum)
# --------------------------------------------------------------------------
def out_up(o_lat: np.ndarray, wkv_b: np.ndarray) -> np.ndarray:
    """out[b,h,d] = sum_c o[b,h,c] * W_UV[h,d,c]."""
    _, w_uv = split_wkv_b(wkv_b)
    return np.einsum("bhc,hdc->bhd", o_lat, w_uv)


# --------------------------------------------------------------------------
# the whole step
# --------------------------------------------------------------------------
def rope_for_batch(q_pe: np.ndarray, end_pos: np.ndarray, inv_freq: np.ndarray) -> np.ndarray:
    """Rotate each sequence's q_pe [B,H,64] at its own position end_pos[b] - 1."""
    pos = np.asarray(end_pos, dtype=np.int64) - 1
    cis = freqs_cis(pos, inv_freq)  # [B,32]
    return rope_interleaved(q_pe, cis[:, None, :])


def q_latent(q_nope: np.ndarray, q_pe: np.ndarray, wkv_b: np.ndarray, end_pos: np.ndarray,
             inv_freq: np.ndarray) -> np.ndarray:
    """[absorbed q~ | rotated q_pe] -> [B,H,576]."""
    return np.concatenate([absorb(q_nope, wkv_b), rope_for_batch(q_pe, end_pos, inv_freq)], axis=-1)


def decode_step(q_nope, q_pe, kv_cache, pe_cache, wkv_b, topk_idx, end_pos, inv_freq, scale,
                batches=None):
    """Full step for the listed sequences: RoPE, absorb, sparse attention,
    value up-projection.  Returns out [len(batches),H,128]."""
    bs = list(range(q_nope.shape[0])) if batches is None else list(batches)
    q_lat = q_latent(q_nope[bs], q_pe[bs], wkv_b, np.asarray(end_pos)[bs], inv_freq)
    o = np.stack([attend_one(q_lat[j, :, :KV_LORA], q_lat[j, :, KV_LORA:], kv_cache[b], pe_cache[b],
                             topk_idx[b], int(end_pos[b]), scale) for j, b in enumerate(bs)])
    return out_up(o, wkv_b)


# --------------------------------------------------------------------------
# Projections on either side of the attention ("Query heads" page, excerpt
# mla-init: wkv_a = Linear(dim, 512 + 64), wo = RowParallelLinear(128 * 128,
# dim); "Attention weights" page, excerpt mla-output: wo(x.flatten(2))).  A
# Linear layer without bias: y = x . W^T with W stored [out, in].
# --------------------------------------------------------------------------
def linear(x: np.ndarray, w: np.ndarray) -> np.ndarray:
    return np.asarray(x, dtype=np.float64) @ np.asarray(w, dtype=np.float64).T


def output_projection(heads: np.ndarray, wo: np.ndarray) -> np.ndarray:
    """heads [B,128,128] flattened to [B,16384] (head-major), times wo^T."""
    return linear(heads.reshape(heads.shape[0], -1), wo)


# --------------------------------------------------------------------------
# Multi-token decode: T query tokens per sequence.  The "Attention weights"
# page notes that the causal mask is added to the selection before the
# softmax; the plain reading for T tokens is that token s of sequence b sits at
# position end_pos[b] - T + s, has its own selection row, and sees a key t only
# if t is selected AND t <= its position.
# --------------------------------------------------------------------------
def token_positions(end_pos: int, T: int) -> np.ndarray:
    return int(end_pos) - T + np.arange(T)


def attend_tokens(q_abs: np.ndarray, q_pe_rot: np.ndarray, kv: np.ndarray, pe: np.ndarray,
                  topk_rows: np.ndarray, end_pos: int, scale: float) -> np.ndarray:
    """T tokens of one sequence: q_abs [T,H,512], q_pe_rot [T,H,64],
    topk_rows [T,K].  Scores over all end_pos keys plus the index mask (0 on
    each token's selection, -inf elsewhere) plus the causal mask (-inf on keys
    after the token's position), softmax over keys, PV.  Returns [T,H,512]."""
    T = q_abs.shape[0]
    kv, pe = kv[:end_pos], pe[:end_pos]
    scores = (np.einsum("shc,tc->sht", q_abs, kv) + np.einsum("shr,tr->sht", q_pe_rot, pe)) * scale
    index_mask = np.full((T, end_pos), -np.inf)
    for s in range(T):
        idx = np.asarray(topk_rows[s], dtype=np.int64)
        idx = idx[(idx >= 0) & (idx < end_pos)]
        index_mask[s, idx] = 0.0
    pos = token_positions(end_pos, T)
    causal = np.where(np.arange(end_pos)[None, :] <= pos[:, None], 0.0, -np.inf)
    mask = index_mask + causal                         # [T, end_pos]
    out = np.zeros((T, q_abs.shape[1], kv.shape[1]))
    for s in range(T):
        sel = np.isfinite(mask[s])
        if not sel.any():
            continue                                   # nothing visible: zeros
        z = scores[s][:, sel]
        p = np.exp(z - z.max(axis=1, keepdims=True))
        p /= p.sum(axis=1, keepdims=True)
        out[s] = p @ kv[sel]
    return out


def decode_tokens(q_nope, q_pe, kv_cache, pe_cache, wkv_b, topk_idx, end_pos, inv_freq, scale, batches=None):
    """Full step for T tokens per sequence: q_nope [n,T,H,128], q_pe [n,T,H,64],
    topk_idx [n,T,K], end_pos [n] (cached tokens including the T new ones).
    Returns out [len(batches),T,H,128]."""
    bs = list(range(q_nope.shape[0])) if batches is None else list(batches)
    T = q_nope.shape[1]
    res = []
    for b in bs:
        pos = token_positions(end_pos[b], T)
        q_abs = absorb(q_nope[b], wkv_b)                                   # [T,H,512]
        cis = freqs_cis(pos, inv_freq)[:, None, :]
        q_rot = rope_interleaved(q_pe[b], cis)                             # [T,H,64]
        o = attend_tokens(q_abs, q_rot, kv_cache[b], pe_cache[b], topk_idx[b], int(end_pos[b]), scale)
        res.append(out_up(o, wkv_b))
    return np.stack(res)


# --------------------------------------------------------------------------
# Cache append ("Query heads" page, excerpt mla-init and its prose: wkv_a
# emits the 512 latent features and the 64-wide rotary key, kv_norm is an
# RMSNorm of the latent; "Attention weights" page, excerpt mla-decode: the
# caches are read up to end_pos).  The write itself is not printed; token s of
# T new tokens sits at position end_pos - T + s.  RMSNorm is taken in its
# standard form x * w / sqrt(mean(x^2) + eps) (its body is not on the pages).
# --------------------------------------------------------------------------
def rms_norm(x: np.ndarray, w: np.ndarray, eps: float) -> np.ndarray:
    x = np.asarray(x, dtype=np.float64)
    return x * np.asarray(w, dtype=np.float64) / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)


def cache_rows(kv_a: np.ndarray, kv_norm_w: np.ndarray, eps: float, end_pos, inv_freq: np.ndarray):
    """The rows the append writes: (positions [B, T], latent rows [B, T, 512],
    rotary rows [B, T, 64]), unrounded float64."""
    B, T = kv_a.shape[0], kv_a.shape[1]
    pos = np.asarray(end_pos, dtype=np.int64)[:, None] - T + np.arange(T)[None, :]
    latent = rms_norm(kv_a[..., :KV_LORA], kv_norm_w, eps)
    cis = freqs_cis(pos.reshape(-1), inv_freq).reshape(B, T, -1)
    rot = rope_interleaved(kv_a[..., KV_LORA:], cis)
    return pos, latent, rot


# --------------------------------------------------------------------------
# independent formulations used only to pin the oracle
# --------------------------------------------------------------------------
def naive_attention_one(q_nope_b, q_pe_rot_b, kv, pe, wkv_b, topk_row, end_pos, scale):
    """Non-absorbed multi-head attention for one sequence: per head expand the
    latent rows into keys [W_UK kv ; pe] and values W_UV kv, then ordinary
    masked softmax attention.  The absorbed path must agree with this."""
    w_uk, w_uv = split_wkv_b(wkv_b)
    kv = kv[:end_pos]
    pe = pe[:end_pos]
    mask = selection_mask(topk_row, end_pos)
    out = np.zeros((N_HEADS, D_V))
    for h in range(N_HEADS):
        k_h = np.concatenate([kv @ w_uk[h].T, pe], axis=1)       # [T,192]
        v_h = kv @ w_uv[h].T                                      # [T,128]
        q_h = np.concatenate([q_nope_b[h], q_pe_rot_b[h]])        # [192]
        s = k_h @ q_h * scale + mask
        s = s - s.max()
        p = np.exp(s)
        p = p / p.sum()
        out[h] = p @ v_h
    return out


def brute_force_toy(q_lat_b, kv, pe, topk_row, end_pos, scale, heads):
    """Scalar loops over (head, key, feature) for a handful of heads and keys:
    the slow, obviously correct form of scores -> softmax -> PV."""
    sel = sorted({int(t) for t in topk_row if 0 <= int(t) < end_pos})
    res = {}
    for h in heads:
        scores = []
        for t in sel:
            acc = 0.0
            for c in range(KV_LORA):
                acc += float(q_lat_b[h][c]) * float(kv[t][c])
            for r in range(D_ROPE):
                acc += float(q_lat_b[h][KV_LORA + r]) * float(pe[t][r])
            scores.append(acc * scale)
        mx = max(scores)
        ex = [math.exp(s - mx) for s in scores]
        tot = sum(ex)
        o = [0.0] * KV_LORA
        for w, t in zip(ex, sel):
            for c in range(KV_LORA):
                o[c] += (w / tot) * float(kv[t][c])
        res[h] = o
    return res
