"""Tolerances and oracle helpers shared by the GPU parity tests.

Tolerances (stated by the decode step's accuracy target):
* RoPE (fp32 path): every output element within 1e-5 of the oracle, relative
  to the norm of its (x[2i], x[2i+1]) pair.
* bf16-in / fp32-accumulate results (q_lat, o, head outputs):
  max|gpu - oracle| <= 2e-2 * max|oracle|  and
  sum|gpu - oracle| / sum|oracle| <= 5e-3 over the compared tensor.
"""
import numpy as np

from oracle import mla_oracle as O
from sparse_latent_attention_decode_b300 import synth

MAX_REL = 2e-2
MEAN_REL = 5e-3
ROPE_REL = 1e-5


def attn_errors(gpu, ora):
    gpu = np.asarray(gpu, dtype=np.float64)
    ora = np.asarray(ora, dtype=np.float64)
    d = np.abs(gpu - ora)
    scale = np.abs(ora).max()
    return d.max() / max(scale, 1e-300), d.sum() / max(np.abs(ora).sum(), 1e-300)


def assert_attn_close(gpu, ora, what=""):
    gpu = np.asarray(gpu, dtype=np.float64)
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite GPU output"
    mx, mean = attn_errors(gpu, ora)
    assert mx <= MAX_REL and mean <= MEAN_REL, f"{what}: max-rel {mx:.3e}, mean-rel {mean:.3e}"
    return mx, mean


def assert_rope_close(gpu, ora, x, what="", interleaved=True):
    """Error of each rotated feature relative to the norm of the pair it
    belongs to: (2i, 2i+1) interleaved, (i, i+32) half-split."""
    gpu = np.asarray(gpu, dtype=np.float64)
    if interleaved:
        pair = np.repeat(np.hypot(x[..., 0::2], x[..., 1::2]), 2, axis=-1)
    else:
        d2 = x.shape[-1] // 2
        half = np.hypot(x[..., :d2], x[..., d2:])
        pair = np.concatenate([half, half], axis=-1)
    err = np.abs(gpu - ora) / np.maximum(pair, 1e-30)
    assert err.max() <= ROPE_REL, f"{what}: rope rel err {err.max():.3e}"
    return err.max()


def oracle_inputs(t: dict) -> dict:
    return {k: synth.to_f64(v) for k, v in t.items()}


INV_FREQ = O.yarn_inv_freq()
SCALE = O.softmax_scale()


def oracle_q_lat(x, batches):
    return O.q_latent(x["q_nope"][batches], x["q_pe"][batches], x["wkv_b"], x["end_pos"][batches], INV_FREQ)


def oracle_o_lat(x, batches, q_lat=None):
    """o for the listed sequences; q_lat (if given) is the query to attend with
    (e.g. the GPU's bf16 q_lat, so the attention stage is compared alone)."""
    if q_lat is None:
        q_lat = oracle_q_lat(x, batches)
    return np.stack([O.attend_one(q_lat[j, :, :512], q_lat[j, :, 512:], x["kv_cache"][b], x["pe_cache"][b],
                                  x["topk_idx"][b], int(x["end_pos"][b]), SCALE)
                     for j, b in enumerate(batches)])


def oracle_out(x, batches):
    return O.decode_step(x["q_nope"], x["q_pe"], x["kv_cache"], x["pe_cache"], x["wkv_b"], x["topk_idx"],
                         x["end_pos"], INV_FREQ, SCALE, batches=batches)
