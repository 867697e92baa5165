"""Seeded synthetic inputs for the sparse latent attention decode step.

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic.  Both the CUDA path (tests, bench) and the float64 oracle
consume what it returns.

Every random tensor is drawn on the CPU from ``torch.Generator`` streams keyed
by (seed, tensor name, sequence), so that the values of one sequence can be
regenerated without drawing the whole batch.  Floating-point tensors are drawn
in float32 and rounded to bf16 (round-to-nearest-even); consumers that need
float64 widen the bf16 values exactly.

Value distributions (the workloads of the decode step): q_nope, q_pe, the
latent cache and the rotary cache ~ N(0, 1); wkv_b ~ N(0, std 512^-0.5).
Cache rows at or beyond a sequence's end_pos are never read by the step and are
left at zero unless ``fill_tail`` is set.
"""
from __future__ import annotations

import concurrent.futures as _cf
import dataclasses
import hashlib

import torch

N_HEADS = 128
D_NOPE = 128
D_ROPE = 64
D_V = 128
KV_LORA = 512
S_CAP_DEFAULT = 16384


def _gen(seed: int, name: str, b: int = 0) -> torch.Generator:
    h = hashlib.blake2b(f"{seed}/{name}/{b}".encode(), digest_size=8).digest()
    return torch.Generator("cpu").manual_seed(int.from_bytes(h, "little") & ((1 << 63) - 1))


def _randn_bf16(shape, g: torch.Generator, std: float = 1.0) -> torch.Tensor:
    x = torch.randn(shape, generator=g, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(torch.bfloat16)


@dataclasses.dataclass
class Workload:
    """Shape recipe of one decode-step workload.

    end_pos: per-sequence number of cached keys (the query sits at end_pos-1).
    selection: "all" (every cached key selected), "uniform" (k distinct keys
    uniform without replacement), or "recent_half" (the most recent positions
    plus uniform draws over the rest, see ``draw_topk``).
    k: selected count per sequence (None = end_pos); K: row stride of topk_idx.
    """
    name: str
    B: int
    end_pos: list
    selection: str
    k: int | None = None
    K: int | None = None
    S_cap: int = S_CAP_DEFAULT

    def k_of(self, b: int) -> int:
        e = self.end_pos[b]
        return e if self.k is None else min(self.k, e)

    def row_stride(self) -> int:
        if self.K is not None:
            return self.K
        return max(self.k_of(b) for b in range(self.B))


def _ragged_end_pos(seed: int, B: int, lo: int, hi: int) -> list:
    g = _gen(seed, "end_pos")
    return [int(v) for v in torch.randint(lo, hi + 1, (B,), generator=g)]


def workload(name: str, seed: int = 0) -> Workload:
    """The named workloads of the decode step (all with a 16384-row cache)."""
    if name == "p1000_b1":          # the pages' worked example: P=1000 cached, 1001 keys
        return Workload(name, 1, [1001], "all")
    if name == "sparse_b32_ctx4096_top2048":
        return Workload(name, 32, [4096] * 32, "uniform", k=2048, K=2048)
    if name == "sparse_b64_ctx16384_top2048":
        return Workload(name, 64, [16384] * 64, "uniform", k=2048, K=2048)
    if name == "ragged_b128_ctx1024to8192_top2048":
        return Workload(name, 128, _ragged_end_pos(seed, 128, 1024, 8192), "recent_half", k=2048, K=2048)
    if name == "dense_b16_ctx16384":
        return Workload(name, 16, [16384] * 16, "all")
    if name == "dense_b1_ctx16384":
        return Workload(name, 1, [16384], "all")
    raise KeyError(name)


WORKLOADS = ["p1000_b1", "sparse_b32_ctx4096_top2048", "sparse_b64_ctx16384_top2048",
             "ragged_b128_ctx1024to8192_top2048", "dense_b16_ctx16384", "dense_b1_ctx16384"]


def draw_topk(seed: int, b: int, end_pos: int, k: int, selection: str) -> torch.Tensor:
    """k distinct positions of [0, end_pos) for sequence b, in a random order.

    "all": every position.  "uniform": without replacement.  "recent_half": the
    min(k/2, 512) most recent positions plus the remainder drawn without
    replacement from the older ones; when k == end_pos this is every position.
    """
    g = _gen(seed, "topk", b)
    if selection == "all" or k >= end_pos:
        sel = torch.arange(end_pos, dtype=torch.int64)
    elif selection == "uniform":
        sel = torch.randperm(end_pos, generator=g)[:k]
    elif selection == "recent_half":
        n_recent = min(k // 2, 512)
        recent = torch.arange(end_pos - n_recent, end_pos, dtype=torch.int64)
        older = torch.randperm(end_pos - n_recent, generator=g)[: k - n_recent]
        sel = torch.cat([recent, older])
    else:
        raise ValueError(selection)
    perm = torch.randperm(sel.numel(), generator=g)
    return sel[perm].to(torch.int32)


def make_inputs(wl: Workload, seed: int = 0, fill_tail: bool = False, threads: int = 8) -> dict:
    """Host tensors for one workload: q_nope [B,128,128], q_pe [B,128,64],
    kv_cache [B,S_cap,512], pe_cache [B,S_cap,64], wkv_b [128*256,512] (bf16),
    topk_idx [B,K] and end_pos [B] (int32; topk rows padded with -1)."""
    B, S = wl.B, wl.S_cap
    K = wl.row_stride()
    q_nope = torch.empty(B, N_HEADS, D_NOPE, dtype=torch.bfloat16)
    q_pe = torch.empty(B, N_HEADS, D_ROPE, dtype=torch.bfloat16)
    kv = torch.zeros(B, S, KV_LORA, dtype=torch.bfloat16)
    pe = torch.zeros(B, S, D_ROPE, dtype=torch.bfloat16)
    topk = torch.full((B, K), -1, dtype=torch.int32)

    def one(b):
        q_nope[b] = _randn_bf16((N_HEADS, D_NOPE), _gen(seed, "q_nope", b))
        q_pe[b] = _randn_bf16((N_HEADS, D_ROPE), _gen(seed, "q_pe", b))
        rows = S if fill_tail else wl.end_pos[b]
        kv[b, :rows] = _randn_bf16((rows, KV_LORA), _gen(seed, "kv_cache", b))
        pe[b, :rows] = _randn_bf16((rows, D_ROPE), _gen(seed, "pe_cache", b))
        sel = draw_topk(seed, b, wl.end_pos[b], wl.k_of(b), wl.selection)
        topk[b, : sel.numel()] = sel

    with _cf.ThreadPoolExecutor(max_workers=max(1, threads)) as ex:
        list(ex.map(one, range(B)))
    wkv_b = _randn_bf16((N_HEADS * (D_NOPE + D_V), KV_LORA), _gen(seed, "wkv_b"), std=KV_LORA ** -0.5)
    end_pos = torch.tensor(wl.end_pos, dtype=torch.int32)
    return dict(q_nope=q_nope, q_pe=q_pe, kv_cache=kv, pe_cache=pe, wkv_b=wkv_b,
                topk_idx=topk, end_pos=end_pos)


def make_token_inputs(wl: Workload, T: int, seed: int = 0, threads: int = 8) -> dict:
    """make_inputs for T query tokens per sequence (multi-token decode):
    q_nope [B,T,128,128], q_pe [B,T,128,64] and topk_idx [B,T,K]; each token
    draws its own selection over all end_pos[b] cached positions (positions
    after the token's own are left in, as an indexer run before the causal
    mask would), the caches, wkv_b and end_pos are those of make_inputs."""
    t = make_inputs(wl, seed, threads=threads)
    B, K = wl.B, wl.row_stride()
    q_nope = torch.empty(B, T, N_HEADS, D_NOPE, dtype=torch.bfloat16)
    q_pe = torch.empty(B, T, N_HEADS, D_ROPE, dtype=torch.bfloat16)
    topk = torch.full((B, T, K), -1, dtype=torch.int32)
    for b in range(B):
        q_nope[b] = _randn_bf16((T, N_HEADS, D_NOPE), _gen(seed, "tok/q_nope", b))
        q_pe[b] = _randn_bf16((T, N_HEADS, D_ROPE), _gen(seed, "tok/q_pe", b))
        for s in range(T):
            sel = draw_topk(seed + 7919 * (s + 1), b, wl.end_pos[b], wl.k_of(b), wl.selection)
            topk[b, s, : sel.numel()] = sel
    t.update(q_nope=q_nope, q_pe=q_pe, topk_idx=topk)
    return t


def make_linear_inputs(seed: int, M: int, N: int, K: int, name: str = "linear"):
    """Token rows x [M, K] ~ N(0, 1) and a weight w [N, K] ~ N(0, K^-1/2), both
    bf16: the shapes of wkv_a (N = 576, K = dim) and wo (N = dim, K = 16384)."""
    x = _randn_bf16((M, K), _gen(seed, name + "/x"))
    w = _randn_bf16((N, K), _gen(seed, name + "/w"), std=K ** -0.5)
    return x, w


def make_fp8_weight(seed: int, rows: int = N_HEADS * (D_NOPE + D_V), cols: int = KV_LORA, block: int = 128,
                    name: str = "wkv_b_fp8"):
    """A block-scaled fp8 weight: e4m3 codes [rows, cols] (uint8) and fp32
    multipliers [ceil(rows/block), ceil(cols/block)].

    Codes are N(0, 112) draws clamped to the e4m3 range +-448 and rounded to
    e4m3 by torch's cast (so every tile spans most of the code range, as a
    per-tile absmax quantisation leaves it); multipliers are
    4 * 512^-0.5 / 448 * exp(N(0, 0.25^2)) per tile, so that the dequantised
    weight has about the spread of the bf16 wkv_b.  No code is NaN."""
    g = _gen(seed, name)
    x = torch.randn(rows, cols, generator=g, dtype=torch.float32).mul_(112.0).clamp_(-448.0, 448.0)
    codes = x.to(torch.float8_e4m3fn).view(torch.uint8)
    sr, sc = -(-rows // block), -(-cols // block)
    z = torch.randn(sr, sc, generator=_gen(seed, name + "/scale"), dtype=torch.float32)
    scale = torch.exp(z * 0.25) * (4.0 * KV_LORA ** -0.5 / 448.0)
    return codes.contiguous(), scale.to(torch.float32).contiguous()


def small_workload(B: int, end_pos, k=None, K=None, S_cap: int = 1024, selection: str = "uniform",
                   name: str = "small") -> Workload:
    """A reduced workload with the same distributions, for tests."""
    ep = list(end_pos) if hasattr(end_pos, "__iter__") else [int(end_pos)] * B
    return Workload(name, B, ep, selection, k=k, K=K, S_cap=S_cap)


def to_f64(t: torch.Tensor):
    """Exact widening of a bf16 / int tensor to a float64 / int64 numpy array."""
    if t.dtype == torch.bfloat16:
        return t.to(torch.float64).numpy()
    return t.numpy().astype("int64")
