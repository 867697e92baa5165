"""Thin ctypes binding over the C ABI of ``libmla_decode.so`` (include/mla_decode.h).

Argument marshalling only: every step of the decode runs in the library's CUDA
kernels.  PyTorch supplies device memory and the current stream.  If the
library has not been built, importing this module raises; there is no
fallback path.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmla_decode.so")

N_HEADS, D_NOPE, D_ROPE, D_V, KV_LORA, Q_LAT = 128, 128, 64, 128, 512, 576
QK_HEAD_DIM = D_NOPE + D_ROPE

MLA_OK = 0
MLA_DEV_BAD_END_POS = 1
MLA_DEV_BAD_POSITION = 2
MLA_DEV_TIMEOUT = 4
MLA_DEV_SCORE_RANGE = 8
MLA_DEV_DUPLICATE_INDEX = 16
CHECK_MAX_S_CAP = 1 << 20


class MLAError(RuntimeError):
    """A library call returned a non-zero status."""


class RopeParams(ctypes.Structure):
    _fields_ = [("rope_dim", ctypes.c_int32), ("max_seq_len", ctypes.c_int32),
                ("original_seq_len", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("rope_theta", ctypes.c_double), ("rope_factor", ctypes.c_double),
                ("beta_fast", ctypes.c_double), ("beta_slow", ctypes.c_double),
                ("mscale", ctypes.c_double)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with "
                          "`python -m sparse_latent_attention_decode_b300.build`")
    lib = ctypes.CDLL(LIB_PATH)
    P, I, Z, F, D = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_float, ctypes.c_double
    sig = {
        "mla_rope_params_default": (None, [ctypes.POINTER(RopeParams)]),
        "mla_softmax_scale": (D, [ctypes.POINTER(RopeParams), I]),
        "rope_freqs_init": (I, [P, ctypes.POINTER(RopeParams), P]),
        "mla_rope_apply": (I, [P, P, I, P, I, P, P, P]),
        "mla_rope_apply_layout": (I, [P, P, I, P, I, I, I, P, P, P]),
        "mla_absorb_q": (I, [P, P, P, I, P, P, I, P, P, P]),
        "mla_sparse_decode_workspace_size": (Z, [I, I]),
        "mla_sparse_decode": (I, [P, P, P, I, P, I, P, I, F, P, P, P, Z, P, P]),
        "mla_out_up": (I, [P, P, I, P, P]),
        "mla_status_string": (ctypes.c_char_p, [I]),
        "mla_profile_hook": (I, [P, P, P]),
        "mla_sparse_decode_static_ws": (I, [P, P, P, I, P, I, P, I, F, P, P, P, P]),
        "mla_weight_dequant_fp8": (I, [P, P, I, I, I, P, P]),
        "mla_cache_append": (I, [P, P, F, P, I, P, I, I, P, P, I, P, P]),
        "mla_absorb_q_tokens": (I, [P, P, P, I, P, P, I, I, P, P, P]),
        "mla_sparse_decode_tokens": (I, [P, P, P, I, P, I, P, I, I, F, P, P, I, P, Z, P, P]),
        "mla_linear_workspace_size": (Z, [I, I, I]),
        "mla_linear_bf16": (I, [P, P, I, I, I, P, P, P, Z, P, P]),
        "mla_set_wait_limit_ns": (ctypes.c_uint64, [ctypes.c_uint64]),
        "mla_check_selection": (I, [P, I, P, I, I, I, P, P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_lib = _load()

EXPORTED = ("mla_rope_params_default", "mla_softmax_scale", "rope_freqs_init", "mla_rope_apply", "mla_rope_apply_layout",
            "mla_absorb_q", "mla_sparse_decode_workspace_size", "mla_sparse_decode", "mla_out_up",
            "mla_status_string", "mla_profile_hook", "mla_sparse_decode_static_ws", "mla_weight_dequant_fp8",
            "mla_cache_append", "mla_absorb_q_tokens", "mla_sparse_decode_tokens",
            "mla_linear_workspace_size", "mla_linear_bf16", "mla_set_wait_limit_ns", "mla_check_selection")
STATIC_WS_BYTES = 32 << 20


def set_wait_limit_ns(ns: int) -> int:
    """Limit of the kernels' bounded on-chip waits (process-wide); returns the
    previous limit.  See mla_set_wait_limit_ns in include/mla_decode.h."""
    return int(_lib.mla_set_wait_limit_ns(int(ns)))


def status_string(code: int) -> str:
    return _lib.mla_status_string(int(code)).decode()


def _check(code: int, what: str):
    if code != MLA_OK:
        raise MLAError(f"{what}: {status_string(code)} (code {code})")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _need(t, name, dtype, shape=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def rope_params(max_seq_len: int = 16384, original_seq_len: int = 4096, rope_theta: float = 10000.0,
                rope_factor: float = 40.0, beta_fast: float = 32.0, beta_slow: float = 1.0,
                mscale: float = 1.0) -> RopeParams:
    p = RopeParams()
    _lib.mla_rope_params_default(ctypes.byref(p))
    p.max_seq_len, p.original_seq_len = max_seq_len, original_seq_len
    p.rope_theta, p.rope_factor = rope_theta, rope_factor
    p.beta_fast, p.beta_slow, p.mscale = beta_fast, beta_slow, mscale
    return p


def softmax_scale(params: RopeParams | None = None, qk_head_dim: int = QK_HEAD_DIM) -> float:
    p = params if params is not None else rope_params()
    return float(_lib.mla_softmax_scale(ctypes.byref(p), qk_head_dim))


def rope_freqs_init(params: RopeParams | None = None, device="cuda", out=None) -> torch.Tensor:
    """Rotary table [max_seq_len, 32, 2] fp32 of (cos, sin)."""
    p = params if params is not None else rope_params()
    if out is None:
        out = torch.empty(p.max_seq_len, D_ROPE // 2, 2, dtype=torch.float32, device=device)
    _need(out, "cis", torch.float32, (p.max_seq_len, D_ROPE // 2, 2))
    _check(_lib.rope_freqs_init(_ptr(out), ctypes.byref(p), _stream(out.device)), "rope_freqs_init")
    return out


def mla_rope_apply(q_pe, cis, end_pos, out=None, dev_status=None) -> torch.Tensor:
    B = q_pe.shape[0]
    _need(q_pe, "q_pe", torch.bfloat16, (B, N_HEADS, D_ROPE))
    _need(cis, "cis", torch.float32)
    _need(end_pos, "end_pos", torch.int32, (B,))
    if out is None:
        out = torch.empty(B, N_HEADS, D_ROPE, dtype=torch.float32, device=q_pe.device)
    _need(out, "q_pe_rot", torch.float32, (B, N_HEADS, D_ROPE))
    _check(_lib.mla_rope_apply(_ptr(q_pe), _ptr(cis), cis.shape[0], _ptr(end_pos), B, _ptr(out),
                               _ptr(dev_status), _stream(q_pe.device)), "mla_rope_apply")
    return out


def mla_rope_apply_layout(x, cis, end_pos, interleaved: bool, out=None, dev_status=None) -> torch.Tensor:
    """Rotary embedding of x [B, n_heads, 64] (bf16) at end_pos - 1, interleaved
    pairs (query layout) or half-split pairs (indexer layout); fp32 result."""
    B, n_heads = x.shape[0], x.shape[1]
    _need(x, "x", torch.bfloat16, (B, n_heads, D_ROPE))
    _need(cis, "cis", torch.float32)
    _need(end_pos, "end_pos", torch.int32, (B,))
    if out is None:
        out = torch.empty(B, n_heads, D_ROPE, dtype=torch.float32, device=x.device)
    _need(out, "out", torch.float32, (B, n_heads, D_ROPE))
    _check(_lib.mla_rope_apply_layout(_ptr(x), _ptr(cis), cis.shape[0], _ptr(end_pos), B, n_heads,
                                      1 if interleaved else 0, _ptr(out), _ptr(dev_status), _stream(x.device)),
           "mla_rope_apply_layout")
    return out


def mla_absorb_q(q_nope, q_pe, cis, end_pos, wkv_b, out=None, dev_status=None) -> torch.Tensor:
    B = q_nope.shape[0]
    _need(q_nope, "q_nope", torch.bfloat16, (B, N_HEADS, D_NOPE))
    _need(q_pe, "q_pe", torch.bfloat16, (B, N_HEADS, D_ROPE))
    _need(cis, "cis", torch.float32)
    _need(end_pos, "end_pos", torch.int32, (B,))
    _need(wkv_b, "wkv_b", torch.bfloat16, (N_HEADS * (D_NOPE + D_V), KV_LORA))
    if out is None:
        out = torch.empty(B, N_HEADS, Q_LAT, dtype=torch.bfloat16, device=q_nope.device)
    _need(out, "q_lat", torch.bfloat16, (B, N_HEADS, Q_LAT))
    _check(_lib.mla_absorb_q(_ptr(q_nope), _ptr(q_pe), _ptr(cis), cis.shape[0], _ptr(end_pos), _ptr(wkv_b), B,
                             _ptr(out), _ptr(dev_status), _stream(q_nope.device)), "mla_absorb_q")
    return out


def mla_weight_dequant_fp8(w, scale, block: int = 128, out=None) -> torch.Tensor:
    """bf16 [rows, cols] from e4m3 codes w [rows, cols] (uint8 or float8_e4m3fn)
    and fp32 block multipliers scale [ceil(rows/block), ceil(cols/block)]."""
    if isinstance(w, torch.Tensor) and w.dtype == torch.float8_e4m3fn:
        w = w.view(torch.uint8)
    rows, cols = w.shape
    _need(w, "w", torch.uint8, (rows, cols))
    _need(scale, "scale", torch.float32, ((rows + block - 1) // block, (cols + block - 1) // block))
    if out is None:
        out = torch.empty(rows, cols, dtype=torch.bfloat16, device=w.device)
    _need(out, "out", torch.bfloat16, (rows, cols))
    _check(_lib.mla_weight_dequant_fp8(_ptr(w), _ptr(scale), rows, cols, block, _ptr(out), _stream(w.device)),
           "mla_weight_dequant_fp8")
    return out


def mla_cache_append(kv_a, kv_norm_w, cis, end_pos, kv_cache, pe_cache, eps: float = 1e-6,
                     dev_status=None) -> None:
    """Write the T new tokens of each sequence (kv_a [B, T, 576] bf16, the wkv_a
    output) into kv_cache [B, S_cap, 512] / pe_cache [B, S_cap, 64] at
    positions end_pos - T .. end_pos - 1: RMSNorm of the latent, rotation of
    the rotary key."""
    B, T = kv_a.shape[0], kv_a.shape[1]
    S_cap = kv_cache.shape[1]
    _need(kv_a, "kv_a", torch.bfloat16, (B, T, Q_LAT))
    _need(kv_norm_w, "kv_norm_w", torch.float32, (KV_LORA,))
    _need(cis, "cis", torch.float32)
    _need(end_pos, "end_pos", torch.int32, (B,))
    _need(kv_cache, "kv_cache", torch.bfloat16, (B, S_cap, KV_LORA))
    _need(pe_cache, "pe_cache", torch.bfloat16, (B, S_cap, D_ROPE))
    _check(_lib.mla_cache_append(_ptr(kv_a), _ptr(kv_norm_w), float(eps), _ptr(cis), cis.shape[0], _ptr(end_pos),
                                 B, T, _ptr(kv_cache), _ptr(pe_cache), S_cap, _ptr(dev_status),
                                 _stream(kv_a.device)), "mla_cache_append")


def mla_absorb_q_tokens(q_nope, q_pe, cis, end_pos, wkv_b, out=None, dev_status=None) -> torch.Tensor:
    """mla_absorb_q for T tokens per sequence: q_nope [n, T, 128, 128],
    q_pe [n, T, 128, 64]; token s of sequence b is rotated at end_pos[b] - T + s."""
    n, T = q_nope.shape[0], q_nope.shape[1]
    _need(q_nope, "q_nope", torch.bfloat16, (n, T, N_HEADS, D_NOPE))
    _need(q_pe, "q_pe", torch.bfloat16, (n, T, N_HEADS, D_ROPE))
    _need(cis, "cis", torch.float32)
    _need(end_pos, "end_pos", torch.int32, (n,))
    _need(wkv_b, "wkv_b", torch.bfloat16, (N_HEADS * (D_NOPE + D_V), KV_LORA))
    if out is None:
        out = torch.empty(n, T, N_HEADS, Q_LAT, dtype=torch.bfloat16, device=q_nope.device)
    _need(out, "q_lat", torch.bfloat16, (n, T, N_HEADS, Q_LAT))
    _check(_lib.mla_absorb_q_tokens(_ptr(q_nope), _ptr(q_pe), _ptr(cis), cis.shape[0], _ptr(end_pos), _ptr(wkv_b),
                                    n, T, _ptr(out), _ptr(dev_status), _stream(q_nope.device)),
           "mla_absorb_q_tokens")
    return out


def mla_sparse_decode_tokens(q_lat, kv_cache, pe_cache, topk_idx, end_pos, softmax_scale, wkv_b=None, out=None,
                             workspace=None, dev_status=None, out_dtype=torch.float32) -> torch.Tensor:
    """mla_sparse_decode for T tokens per sequence: q_lat [n, T, 128, 576],
    topk_idx [n, T, K]; token s of sequence b sees its selected positions up to
    end_pos[b] - T + s.  Returns [n, T, 128, 128] (or [n, T, 128, 512]) in
    out_dtype (float32 or bfloat16)."""
    if out_dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("out_dtype must be torch.float32 or torch.bfloat16")
    n, T, K = topk_idx.shape
    S_cap = kv_cache.shape[1]
    _need(q_lat, "q_lat", torch.bfloat16, (n, T, N_HEADS, Q_LAT))
    _need(kv_cache, "kv_cache", torch.bfloat16, (n, S_cap, KV_LORA))
    _need(pe_cache, "pe_cache", torch.bfloat16, (n, S_cap, D_ROPE))
    _need(topk_idx, "topk_idx", torch.int32, (n, T, K))
    _need(end_pos, "end_pos", torch.int32, (n,))
    if wkv_b is not None:
        _need(wkv_b, "wkv_b", torch.bfloat16, (N_HEADS * (D_NOPE + D_V), KV_LORA))
    width = D_V if wkv_b is not None else KV_LORA
    if out is None:
        out = torch.empty(n, T, N_HEADS, width, dtype=out_dtype, device=q_lat.device)
    _need(out, "out", out_dtype, (n, T, N_HEADS, width))
    if workspace is None:
        workspace = torch.empty(workspace_size(n * T, K), dtype=torch.uint8, device=q_lat.device)
    _check(_lib.mla_sparse_decode_tokens(_ptr(q_lat), _ptr(kv_cache), _ptr(pe_cache), S_cap, _ptr(topk_idx), K,
                                         _ptr(end_pos), n, T, float(softmax_scale), _ptr(wkv_b), _ptr(out),
                                         1 if out_dtype == torch.bfloat16 else 0,
                                         _ptr(workspace), workspace.numel(), _ptr(dev_status),
                                         _stream(q_lat.device)), "mla_sparse_decode_tokens")
    return out


def linear_workspace_size(M: int, N: int, K: int) -> int:
    n = int(_lib.mla_linear_workspace_size(M, N, K))
    if n == 0:
        raise MLAError(f"linear workspace size undefined for M={M}, N={N}, K={K}")
    return n


def mla_linear_bf16(x, w, out_dtype=torch.float32, out=None, workspace=None, dev_status=None) -> torch.Tensor:
    """Y = X . W^T for x [M, K] and w [N, K] (bf16), fp32 accumulation; the
    result [M, N] is float32 or bfloat16."""
    M, K = x.shape
    N = w.shape[0]
    _need(x, "x", torch.bfloat16, (M, K))
    _need(w, "w", torch.bfloat16, (N, K))
    if out_dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("out_dtype must be torch.float32 or torch.bfloat16")
    if out is None:
        out = torch.empty(M, N, dtype=out_dtype, device=x.device)
    _need(out, "out", out_dtype, (M, N))
    if workspace is None:
        workspace = torch.empty(linear_workspace_size(M, N, K), dtype=torch.uint8, device=x.device)
    f32 = out if out_dtype == torch.float32 else None
    b16 = out if out_dtype == torch.bfloat16 else None
    _check(_lib.mla_linear_bf16(_ptr(x), _ptr(w), M, N, K, _ptr(f32), _ptr(b16), _ptr(workspace), workspace.numel(),
                                _ptr(dev_status), _stream(x.device)), "mla_linear_bf16")
    return out


def workspace_size(B: int, K: int) -> int:
    n = int(_lib.mla_sparse_decode_workspace_size(B, K))
    if n == 0:
        raise MLAError(f"workspace size undefined for B={B}, K={K}")
    return n


def mla_sparse_decode(q_lat, kv_cache, pe_cache, topk_idx, end_pos, softmax_scale, wkv_b=None, out=None,
                      workspace=None, dev_status=None) -> torch.Tensor:
    """Latent attention over the selected rows; with wkv_b the result is the
    head output [B,128,128], without it the normalised latent o [B,128,512]."""
    B, K = topk_idx.shape
    S_cap = kv_cache.shape[1]
    _need(q_lat, "q_lat", torch.bfloat16, (B, N_HEADS, Q_LAT))
    _need(kv_cache, "kv_cache", torch.bfloat16, (B, S_cap, KV_LORA))
    _need(pe_cache, "pe_cache", torch.bfloat16, (B, S_cap, D_ROPE))
    _need(topk_idx, "topk_idx", torch.int32, (B, K))
    _need(end_pos, "end_pos", torch.int32, (B,))
    if wkv_b is not None:
        _need(wkv_b, "wkv_b", torch.bfloat16, (N_HEADS * (D_NOPE + D_V), KV_LORA))
    width = D_V if wkv_b is not None else KV_LORA
    if out is None:
        out = torch.empty(B, N_HEADS, width, dtype=torch.float32, device=q_lat.device)
    _need(out, "out", torch.float32, (B, N_HEADS, width))
    if workspace is None:
        workspace = torch.empty(workspace_size(B, K), dtype=torch.uint8, device=q_lat.device)
    _check(_lib.mla_sparse_decode(_ptr(q_lat), _ptr(kv_cache), _ptr(pe_cache), S_cap, _ptr(topk_idx), K,
                                  _ptr(end_pos), B, float(softmax_scale), _ptr(wkv_b), _ptr(out),
                                  _ptr(workspace), workspace.numel(), _ptr(dev_status),
                                  _stream(q_lat.device)), "mla_sparse_decode")
    return out


def mla_sparse_decode_static_ws(q_lat, kv_cache, pe_cache, topk_idx, end_pos, softmax_scale, wkv_b=None, out=None,
                                dev_status=None) -> torch.Tensor:
    """mla_sparse_decode for callers that cannot allocate a workspace: the
    library's own fixed device array (STATIC_WS_BYTES) serves as scratch.
    Calls that overlap on the GPU share that array and must not race."""
    B, K = topk_idx.shape
    S_cap = kv_cache.shape[1]
    _need(q_lat, "q_lat", torch.bfloat16, (B, N_HEADS, Q_LAT))
    _need(kv_cache, "kv_cache", torch.bfloat16, (B, S_cap, KV_LORA))
    _need(pe_cache, "pe_cache", torch.bfloat16, (B, S_cap, D_ROPE))
    _need(topk_idx, "topk_idx", torch.int32, (B, K))
    _need(end_pos, "end_pos", torch.int32, (B,))
    if wkv_b is not None:
        _need(wkv_b, "wkv_b", torch.bfloat16, (N_HEADS * (D_NOPE + D_V), KV_LORA))
    width = D_V if wkv_b is not None else KV_LORA
    if out is None:
        out = torch.empty(B, N_HEADS, width, dtype=torch.float32, device=q_lat.device)
    _need(out, "out", torch.float32, (B, N_HEADS, width))
    _check(_lib.mla_sparse_decode_static_ws(_ptr(q_lat), _ptr(kv_cache), _ptr(pe_cache), S_cap, _ptr(topk_idx), K,
                                            _ptr(end_pos), B, float(softmax_scale), _ptr(wkv_b), _ptr(out),
                                            _ptr(dev_status), _stream(q_lat.device)), "mla_sparse_decode_static_ws")
    return out


def mla_out_up(o_lat, wkv_b, out=None) -> torch.Tensor:
    B = o_lat.shape[0]
    _need(o_lat, "o_lat", torch.float32, (B, N_HEADS, KV_LORA))
    _need(wkv_b, "wkv_b", torch.bfloat16, (N_HEADS * (D_NOPE + D_V), KV_LORA))
    if out is None:
        out = torch.empty(B, N_HEADS, D_V, dtype=torch.float32, device=o_lat.device)
    _need(out, "out", torch.float32, (B, N_HEADS, D_V))
    _check(_lib.mla_out_up(_ptr(o_lat), _ptr(wkv_b), B, _ptr(out), _stream(o_lat.device)), "mla_out_up")
    return out


def mla_check_selection(topk_idx, end_pos, S_cap: int, dev_status=None) -> torch.Tensor:
    """Flags a position repeated among the valid entries of a selection row
    (MLA_DEV_DUPLICATE_INDEX in the returned int32 status word; read it after
    synchronising).  topk_idx [B, K] (one token per sequence) or [n, T, K];
    end_pos [B] or [n]; S_cap is the cache capacity the selection indexes."""
    if topk_idx.dim() == 2:
        n, K = topk_idx.shape
        T = 1
    else:
        n, T, K = topk_idx.shape
    _need(topk_idx, "topk_idx", torch.int32)
    _need(end_pos, "end_pos", torch.int32, (n,))
    if dev_status is None:
        dev_status = torch.zeros(1, dtype=torch.int32, device=topk_idx.device)
    _need(dev_status, "dev_status", torch.int32, (1,))
    _check(_lib.mla_check_selection(_ptr(topk_idx), K, _ptr(end_pos), n, T, int(S_cap), _ptr(dev_status),
                                    _stream(topk_idx.device)), "mla_check_selection")
    return dev_status


class ProfileHook:
    """Context manager around the library's per-thread profiling hook: counts
    the kernels the library enqueues and (optionally) records a pair of CUDA
    events around the attention kernel of each mla_sparse_decode call."""

    def __init__(self, ev_start=None, ev_stop=None):
        self.count = ctypes.c_int64(0)
        self.ev_start, self.ev_stop = ev_start, ev_stop

    def set_events(self, ev_start, ev_stop):
        self.ev_start, self.ev_stop = ev_start, ev_stop
        self._arm()

    def _arm(self):
        s = ctypes.c_void_p(self.ev_start.cuda_event) if self.ev_start is not None else None
        e = ctypes.c_void_p(self.ev_stop.cuda_event) if self.ev_stop is not None else None
        _lib.mla_profile_hook(s, e, ctypes.byref(self.count))

    def __enter__(self):
        self._arm()
        return self

    def __exit__(self, *exc):
        _lib.mla_profile_hook(None, None, None)
        return False

    @property
    def launches(self) -> int:
        return int(self.count.value)


class CapturedStep:
    """A callable captured once into a CUDA graph and then replayed: one graph
    launch per step instead of one host call per kernel, so that the host never
    paces the device.  Every tensor the callable touches must stay allocated
    (the graph holds their addresses); ``out`` is what the captured call
    returned, refreshed by each replay.  The library kernels keep their
    programmatic-dependent-launch chaining inside the graph."""

    def __init__(self, fn, *args, warmup: int = 2):
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            for _ in range(warmup):
                fn(*args)
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with ProfileHook() as hook:
            with torch.cuda.graph(self.graph):
                self.out = fn(*args)
        self.kernels_per_replay = hook.launches

    def __call__(self):
        self.graph.replay()
        return self.out


class DecodeStep:
    """One decode step with its buffers held: absorb (RoPE fused) -> sparse
    attention -> value up-projection, three library calls on the current
    stream.  The caches and wkv_b are resident device state; the per-step
    inputs are the query parts, the selection and end_pos."""

    def __init__(self, B: int, K: int, device="cuda", params: RopeParams | None = None,
                 out_dtype=torch.float32):
        if out_dtype not in (torch.float32, torch.bfloat16):
            raise TypeError("out_dtype must be torch.float32 or torch.bfloat16")
        self.B, self.K, self.device = B, K, torch.device(device)
        self.params = params if params is not None else rope_params()
        self.scale = softmax_scale(self.params)
        self.cis = rope_freqs_init(self.params, device=self.device)
        self.q_lat = torch.empty(B, N_HEADS, Q_LAT, dtype=torch.bfloat16, device=self.device)
        self.out = torch.empty(B, N_HEADS, D_V, dtype=out_dtype, device=self.device)
        self.workspace = torch.empty(workspace_size(B, K), dtype=torch.uint8, device=self.device)
        self.status = torch.zeros(1, dtype=torch.int32, device=self.device)

    def __call__(self, q_nope, q_pe, kv_cache, pe_cache, wkv_b, topk_idx, end_pos):
        mla_absorb_q(q_nope, q_pe, self.cis, end_pos, wkv_b, out=self.q_lat, dev_status=self.status)
        if self.out.dtype == torch.float32:
            return mla_sparse_decode(self.q_lat, kv_cache, pe_cache, topk_idx, end_pos, self.scale, wkv_b=wkv_b,
                                     out=self.out, workspace=self.workspace, dev_status=self.status)
        out = mla_sparse_decode_tokens(self.q_lat[:, None], kv_cache, pe_cache, topk_idx[:, None], end_pos,
                                       self.scale, wkv_b=wkv_b, out=self.out[:, None], workspace=self.workspace,
                                       dev_status=self.status, out_dtype=torch.bfloat16)
        return out[:, 0]

    def check_status(self):
        v = int(self.status.item())
        if v:
            raise MLAError(f"device status: {status_string(v)} (bits {v})")


class HostDecodeStep(DecodeStep):
    """End-to-end step from host buffers: per-step inputs are copied from
    pinned host memory to the device, the three library calls run, and the
    head outputs are copied back into a pinned host buffer."""

    def __init__(self, B: int, K: int, device="cuda", params: RopeParams | None = None,
                 out_dtype=torch.float32):
        super().__init__(B, K, device, params, out_dtype)
        dev = self.device
        # the per-step inputs live in one device buffer (see packed_inputs), so that a
        # caller holding them in one pinned buffer of the same layout copies them at once
        self.d_packed = torch.empty(self.packed_bytes(B, K), dtype=torch.uint8, device=dev)
        self.d_q_nope, self.d_q_pe, self.d_topk, self.d_end = self.packed_inputs(self.d_packed, B, K)
        self.h_out = torch.empty(B, N_HEADS, D_V, dtype=out_dtype).pin_memory()

    @staticmethod
    def _packed_layout(B: int, K: int):
        sizes = (B * N_HEADS * D_NOPE * 2, B * N_HEADS * D_ROPE * 2, B * K * 4, B * 4)
        offs, o = [], 0
        for n in sizes:
            offs.append(o)
            o += (n + 255) // 256 * 256
        return offs, o

    @staticmethod
    def packed_bytes(B: int, K: int) -> int:
        """Bytes of one buffer holding a step's inputs (q_nope, q_pe, topk_idx,
        end_pos, each at a 256-byte aligned offset)."""
        return HostDecodeStep._packed_layout(B, K)[1]

    @staticmethod
    def packed_inputs(buf: torch.Tensor, B: int, K: int):
        """Views (q_nope, q_pe, topk_idx, end_pos) into a uint8 buffer of
        packed_bytes(B, K) bytes, host or device."""
        offs, _ = HostDecodeStep._packed_layout(B, K)
        q_nope = buf[offs[0]:offs[0] + B * N_HEADS * D_NOPE * 2].view(torch.bfloat16).view(B, N_HEADS, D_NOPE)
        q_pe = buf[offs[1]:offs[1] + B * N_HEADS * D_ROPE * 2].view(torch.bfloat16).view(B, N_HEADS, D_ROPE)
        topk = buf[offs[2]:offs[2] + B * K * 4].view(torch.int32).view(B, K)
        end = buf[offs[3]:offs[3] + B * 4].view(torch.int32)
        return q_nope, q_pe, topk, end

    def h2d_bytes(self):
        return sum(t.numel() * t.element_size() for t in (self.d_q_nope, self.d_q_pe, self.d_topk, self.d_end))

    def d2h_bytes(self):
        return self.h_out.numel() * self.h_out.element_size()

    def run(self, h_q_nope, h_q_pe, h_topk, h_end, kv_cache, pe_cache, wkv_b):
        self.d_q_nope.copy_(h_q_nope, non_blocking=True)
        self.d_q_pe.copy_(h_q_pe, non_blocking=True)
        self.d_topk.copy_(h_topk, non_blocking=True)
        self.d_end.copy_(h_end, non_blocking=True)
        out = self(self.d_q_nope, self.d_q_pe, kv_cache, pe_cache, wkv_b, self.d_topk, self.d_end)
        self.h_out.copy_(out, non_blocking=True)
        return self.h_out

    def run_packed(self, h_packed, kv_cache, pe_cache, wkv_b):
        """run() with the inputs in one pinned buffer laid out by packed_inputs:
        one host-to-device copy instead of four."""
        self.d_packed.copy_(h_packed, non_blocking=True)
        out = self(self.d_q_nope, self.d_q_pe, kv_cache, pe_cache, wkv_b, self.d_topk, self.d_end)
        self.h_out.copy_(out, non_blocking=True)
        return self.h_out


class HostDecodePipeline:
    """Decode steps from pinned host buffers with the transfers overlapped:
    the inputs of step i go up on one copy stream and the outputs of step i-1
    come back on another while the device computes.  Two device buffer sets
    alternate; every step still copies its own inputs in and its own head
    outputs out.  ``submit`` enqueues one step and returns at once; read an
    output buffer only after ``finish`` (or after the step two submissions
    later has been submitted and ``finish`` has run)."""

    def __init__(self, B: int, K: int, device="cuda", params: RopeParams | None = None):
        self.device = torch.device(device)
        self.steps = [HostDecodeStep(B, K, self.device, params) for _ in range(2)]
        self.h2d = torch.cuda.Stream(self.device)
        self.d2h = torch.cuda.Stream(self.device)
        self.in_ready = [torch.cuda.Event() for _ in range(2)]
        self.computed = [torch.cuda.Event() for _ in range(2)]
        self.copied_out = [torch.cuda.Event() for _ in range(2)]
        self.count = 0

    def h2d_bytes(self):
        return self.steps[0].h2d_bytes()

    def d2h_bytes(self):
        return self.steps[0].d2h_bytes()

    def submit(self, h_q_nope, h_q_pe, h_topk, h_end, kv_cache, pe_cache, wkv_b, h_out):
        i, k = self.count, self.count % 2
        st = self.steps[k]
        compute = torch.cuda.current_stream(self.device)
        with torch.cuda.stream(self.h2d):
            if i >= 2:
                self.h2d.wait_event(self.computed[k])      # step i-2 has read these device inputs
            st.d_q_nope.copy_(h_q_nope, non_blocking=True)
            st.d_q_pe.copy_(h_q_pe, non_blocking=True)
            st.d_topk.copy_(h_topk, non_blocking=True)
            st.d_end.copy_(h_end, non_blocking=True)
            self.in_ready[k].record(self.h2d)
        compute.wait_event(self.in_ready[k])
        if i >= 2:
            compute.wait_event(self.copied_out[k])          # step i-2's outputs have left the device buffer
        out = st(st.d_q_nope, st.d_q_pe, kv_cache, pe_cache, wkv_b, st.d_topk, st.d_end)
        self.computed[k].record(compute)
        with torch.cuda.stream(self.d2h):
            self.d2h.wait_event(self.computed[k])
            h_out.copy_(out, non_blocking=True)
            self.copied_out[k].record(self.d2h)
        self.count += 1

    def finish(self):
        """Make the current stream wait for every submitted step's copies."""
        compute = torch.cuda.current_stream(self.device)
        for k in range(min(self.count, 2)):
            compute.wait_event(self.copied_out[k])

    def check_status(self):
        for st in self.steps:
            st.check_status()


class CapturedHostPipeline:
    """End-to-end decode steps from pinned host buffers, each step one CUDA
    graph replay: the graph copies the step's query parts, selection and
    end_pos in from one pinned host buffer (one copy), runs absorption, attention and
    up-projection, and copies the head outputs back into pinned host memory.
    Two buffer sets, each with its own graph and stream, alternate, so that
    one step's transfers overlap the other's compute, and the host makes one
    call per step (a slow host does not pace the device).

    Fill ``host_inputs(i)`` before ``submit(i)``; read ``host_output(i)``
    after ``finish()``.  Step i uses buffer set i % 2: do not refill it
    before the step two submissions earlier has finished (``finish``)."""

    def __init__(self, B: int, K: int, kv_cache, pe_cache, wkv_b, device="cuda",
                 params: RopeParams | None = None, out_dtype=torch.bfloat16):
        self.device = torch.device(device)
        self.steps, self.h_in, self.graphs, self.streams = [], [], [], []
        for _ in range(2):
            st = HostDecodeStep(B, K, self.device, params, out_dtype)
            # the step's inputs in one pinned buffer: one host-to-device copy per step
            packed = torch.zeros(HostDecodeStep.packed_bytes(B, K), dtype=torch.uint8).pin_memory()
            q_nope, q_pe, topk, end = HostDecodeStep.packed_inputs(packed, B, K)
            topk.fill_(-1)
            end.fill_(1)
            h = {"q_nope": q_nope, "q_pe": q_pe, "topk_idx": topk, "end_pos": end}
            g = CapturedStep(st.run_packed, packed, kv_cache, pe_cache, wkv_b)
            self.steps.append(st)
            self.h_in.append(h)
            self.graphs.append(g)
            self.streams.append(torch.cuda.Stream(self.device))
        self.count = 0

    def host_inputs(self, i: int) -> dict:
        return self.h_in[i % 2]

    def host_output(self, i: int) -> torch.Tensor:
        return self.steps[i % 2].h_out

    def h2d_bytes(self):
        return self.steps[0].d_packed.numel()

    def d2h_bytes(self):
        return self.steps[0].d2h_bytes()

    def submit(self):
        k = self.count % 2
        with torch.cuda.stream(self.streams[k]):
            self.graphs[k]()
        self.count += 1

    def finish(self):
        """Make the current stream wait for every submitted step."""
        cur = torch.cuda.current_stream(self.device)
        for s in self.streams:
            cur.wait_stream(s)

    def check_status(self):
        for st in self.steps:
            st.check_status()


class FusedDecodeStep:
    """The attention block's decode step for one new token per sequence, from
    the token's hidden state to the block's output, as five library calls on
    the current stream (capture it with CapturedStep to make it one launch):

        kv_a = x . wkv_a^T                       (mla_linear_bf16, bf16 out)
        cache rows at end_pos - 1                (mla_cache_append: RMSNorm of
                                                  the latent, rotation of the
                                                  rotary key)
        q_lat = [q_nope . W_UK | rope(q_pe)]     (mla_absorb_q)
        heads = softmax over the selection . V, up-projected (mla_sparse_decode_tokens, bf16 out)
        y = heads.flatten . wo^T                 (mla_linear_bf16)

    x [B, dim] bf16 (the normalised hidden state), wkv_a [576, dim],
    kv_norm_w [512] fp32, wo [dim, 16384] bf16; the query parts q_nope / q_pe
    come from the query path, which needs trained weights and is not part of
    this library.  end_pos counts the new token (its row is written at
    end_pos - 1 before the attention reads the caches)."""

    def __init__(self, B: int, K: int, dim: int, device="cuda", params: RopeParams | None = None,
                 eps: float = 1e-6):
        self.B, self.K, self.dim, self.eps = B, K, dim, eps
        self.device = torch.device(device)
        self.params = params if params is not None else rope_params()
        self.scale = softmax_scale(self.params)
        self.cis = rope_freqs_init(self.params, device=self.device)
        dev = self.device
        self.kv_a = torch.empty(B, Q_LAT, dtype=torch.bfloat16, device=dev)
        self.q_lat = torch.empty(B, N_HEADS, Q_LAT, dtype=torch.bfloat16, device=dev)
        self.heads = torch.empty(B, 1, N_HEADS, D_V, dtype=torch.bfloat16, device=dev)
        self.y = torch.empty(B, dim, dtype=torch.bfloat16, device=dev)
        self.ws_attn = torch.empty(workspace_size(B, K), dtype=torch.uint8, device=dev)
        self.ws_a = torch.empty(linear_workspace_size(B, Q_LAT, dim), dtype=torch.uint8, device=dev)
        self.ws_o = torch.empty(linear_workspace_size(B, dim, N_HEADS * D_V), dtype=torch.uint8, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)

    def __call__(self, x, q_nope, q_pe, kv_cache, pe_cache, wkv_a, kv_norm_w, wkv_b, wo, topk_idx, end_pos):
        mla_linear_bf16(x, wkv_a, out_dtype=torch.bfloat16, out=self.kv_a, workspace=self.ws_a,
                        dev_status=self.status)
        mla_cache_append(self.kv_a[:, None], kv_norm_w, self.cis, end_pos, kv_cache, pe_cache, eps=self.eps,
                         dev_status=self.status)
        mla_absorb_q(q_nope, q_pe, self.cis, end_pos, wkv_b, out=self.q_lat, dev_status=self.status)
        mla_sparse_decode_tokens(self.q_lat[:, None], kv_cache, pe_cache, topk_idx[:, None], end_pos, self.scale,
                                 wkv_b=wkv_b, out=self.heads, workspace=self.ws_attn, dev_status=self.status,
                                 out_dtype=torch.bfloat16)
        return mla_linear_bf16(self.heads.view(self.B, N_HEADS * D_V), wo, out_dtype=torch.bfloat16, out=self.y,
                               workspace=self.ws_o, dev_status=self.status)

    def check_status(self):
        v = int(self.status.item())
        if v:
            raise MLAError(f"device status: {status_string(v)} (bits {v})")
