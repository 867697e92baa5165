#!/usr/bin/env python
"""Benchmark of one decode step of absorbed, top-k-sparse latent attention.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--configs all|none|NAME,...] [--impl ours|reference]

A step is the whole path for one batch: RoPE + key absorption
(mla_absorb_q), then scores / softmax / PV / value up-projection
(mla_sparse_decode with wkv_b).  Inputs are seeded synthetic tensors already
resident in HBM; the step is captured once in a CUDA graph and each timed
step is one replay.  The timed steps rotate over four input sets (the
workload's tensors and three device copies of them: caches, wkv_b, query
parts, selection), so that consecutive steps share no buffer and each step's
working set (its gathered rows and wkv_b, 180 MB at the headline workload)
is larger than the 126 MB L2; they run back to back, as a decode loop runs
them, timed by CUDA events around chunks of consecutive replays.  The same
replays are also timed one at a time with L2 flushed before each (a 256 MiB
buffer written, then another read) and events around each replay
(``ms_per_step_flushed``): that figure carries, besides the step, the
launch-to-event overhead of a single launch, about 5-7 us on this system
even for an empty kernel.

The headline line is the workload named by --workload (B=64, 16384 cached
positions, top-2048); its ``configs`` object carries the same measurement
for every named workload (the pages' P=1000 example at B=1, B=32 at 4096
positions, B=64 at 16384, the ragged B=128 batch, dense B=16 and dense B=1),
each with the attention kernel's time, its algorithmic bytes and FLOPs and
its fraction of the slower of its two bounds (HBM bytes at the measured copy
peak, FLOPs at the measured bf16 tensor peak).

With N > 1 each rank runs an independent replica on its own batch (different
seed): no collective on the data path, weak scaling; a barrier and a
max-over-ranks reduction bracket the timing.  Launched without torchrun,
``--gpus N`` (N > 1) starts the N ranks itself through torch.distributed.run.

The line printed by rank 0 also carries: the end-to-end figure through the
host-buffer API (each step's pinned host inputs copied in and bf16 head
outputs copied back, one CUDA-graph replay per step, transfers overlapped
across steps by CapturedHostPipeline), the
float64 oracle timed on a bounded sample on the host cores (cpu_baseline),
GPU clocks sampled through NVML while the timed steps and an untimed soak of
the same graph around them run, and the number of library kernels launched
in the timed region.

--impl reference times the float64 CPU oracle (the only reference this path
has) on the same workload: each step is one sequence of the batch.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

METRIC = "decode query-tokens/sec and achieved HBM GB/s, % of roofline (sparse MLA)"
UNIT = "tokens/s"
DEFAULT_WORKLOAD = "sparse_b64_ctx16384_top2048"
ROW_BYTES = (512 + 64) * 2          # one gathered cache row (latent + rotary), bf16
FLUSH_BYTES = 256 << 20             # > 126 MB L2
FALLBACK_HBM_GBS = 6400.0
FALLBACK_BF16_TFLOPS = 1800.0
REF_HEADS = 64                     # heads per reference-arm step (a bounded sample of one query token)


# ----------------------------------------------------------------- distributed plumbing
def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def dist_init(world: int, backend: str):
    if world > 1:
        import torch.distributed as dist
        if not dist.is_initialized():
            dist.init_process_group(backend=backend)


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, device=None) -> float:
    """Largest value of x over all ranks (control plane only)."""
    if world == 1:
        return float(x)
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_seed(rank: int, base: int = 0) -> int:
    """Each rank draws an independent batch of the same shape."""
    return base + 1000003 * rank


# ----------------------------------------------------------------- clocks
class _Nvml:
    """The few read-only NVML queries the clock record needs, called through
    ctypes on the driver's libnvidia-ml (no Python binding required)."""

    CLOCK_SM = 1

    def __init__(self):
        import ctypes
        self.c = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        rc = self.lib.nvmlInit_v2()
        if rc != 0:
            raise RuntimeError(f"nvmlInit_v2 returned {rc}")
        self.reasons = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons

    def handle(self, bus_id: str, index: int):
        h = self.c.c_void_p()
        if self.lib.nvmlDeviceGetHandleByPciBusId_v2(bus_id.encode(), self.c.byref(h)) == 0:
            return h
        if self.lib.nvmlDeviceGetHandleByIndex_v2(self.c.c_uint(index), self.c.byref(h)) == 0:
            return h
        raise RuntimeError(f"no NVML handle for {bus_id} / index {index}")

    def sample(self, h):
        u = self.c.c_uint()
        m = self.c.c_uint()
        r = self.c.c_ulonglong()
        p = self.c.c_uint()
        if self.lib.nvmlDeviceGetClockInfo(h, self.CLOCK_SM, self.c.byref(u)) != 0:
            raise RuntimeError("nvmlDeviceGetClockInfo failed")
        self.lib.nvmlDeviceGetMaxClockInfo(h, self.CLOCK_SM, self.c.byref(m))
        self.reasons(h, self.c.byref(r))
        self.lib.nvmlDeviceGetPowerUsage(h, self.c.byref(p))
        return int(u.value), int(m.value), int(r.value), p.value / 1000.0


class ClockSampler:
    """SM clock, its maximum, power and the clock-event reasons of the bench
    GPU, read through NVML (queries only) every 20 ms by a background thread.
    Only samples taken while a window is open (open_window / close_window)
    are kept: the timed steps and the untimed soak of the same graph that
    brackets them."""

    # NVML clock-event reason bits
    REASONS = (("sw_power_cap", 0x4), ("hw_slowdown", 0x8), ("sw_thermal_slowdown", 0x20),
               ("hw_thermal_slowdown", 0x40), ("hw_power_brake_slowdown", 0x80))

    def __init__(self, device_index: int, period_s: float = 0.02):
        import threading
        self.period = period_s
        self.samples = []
        self.errors = []
        self.window = False
        self.stop_flag = threading.Event()
        self.thread = None
        self.nvml = None
        self.handle = None
        try:
            self.nvml = _Nvml()
            props = torch.cuda.get_device_properties(device_index)
            bus = (f"{getattr(props, 'pci_domain_id', 0):08X}:{props.pci_bus_id:02X}:"
                   f"{getattr(props, 'pci_device_id', 0):02X}.0")
            idx = device_index
            visible = os.environ.get("CUDA_VISIBLE_DEVICES", "")
            ids = [v.strip() for v in visible.split(",") if v.strip()]
            if ids and all(v.isdigit() for v in ids) and device_index < len(ids):
                idx = int(ids[device_index])
            self.handle = self.nvml.handle(bus, idx)
        except Exception as e:
            self.errors.append(f"nvml: {e}")
            self.nvml = None
        if self.nvml is not None:
            self.thread = threading.Thread(target=self._run, daemon=True)
            self.thread.start()

    def _run(self):
        while not self.stop_flag.is_set():
            if self.window:
                try:
                    sm, mx, rs, pw = self.nvml.sample(self.handle)
                    self.samples.append((time.time(), sm, mx, rs, pw))
                except Exception as e:
                    if len(self.errors) < 4:
                        self.errors.append(f"sample: {e}")
            time.sleep(self.period)

    def open_window(self):
        self.window = True

    def close_window(self):
        self.window = False

    def summary(self) -> dict:
        self.stop_flag.set()
        if self.thread is not None:
            self.thread.join(timeout=2)
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "source": "nvml",
                    "errors": self.errors}
        sm = [x[1] for x in self.samples]
        mx = [x[2] for x in self.samples]
        reasons = sorted({name for x in self.samples for name, bit in self.REASONS if x[3] & bit})
        return {"sm_mhz": statistics.median(sm), "sm_mhz_min": min(sm), "sm_max_mhz": max(mx),
                "reasons": reasons, "samples": len(self.samples),
                "power_w_max": max(x[4] for x in self.samples),
                "seconds": self.samples[-1][0] - self.samples[0][0], "source": "nvml (libnvidia-ml), every 20 ms",
                "window": "the timed steps and an untimed soak of the same graph around them",
                **({"errors": self.errors} if self.errors else {})}


# ----------------------------------------------------------------- helpers
def read_stream_gbs(dev, n_bytes: int = 2 << 30, reps: int = 10) -> float:
    """Read-only HBM stream for context beside the copy peak (which counts read
    and write bytes): PyTorch's sum over a 2 GiB buffer, mean of `reps` runs."""
    x = torch.ones(n_bytes // 4, dtype=torch.float32, device=dev)
    for _ in range(3):
        x.sum()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record()
    for _ in range(reps):
        x.sum()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / reps
    del x
    return n_bytes / (ms * 1e-3) / 1e9


def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        return json.load(open(p))
    except Exception:
        return {}


TRAFFIC_SUMMARY = os.path.join(ROOT, "profiles", "attn_kernel_sparse_b64_ctx16384_top2048.md")
KERNEL_SOURCES = [os.path.join(ROOT, "sparse_latent_attention_decode_b300", "csrc", f)
                  for f in ("attn.cu", "tc05.cuh", "common.cuh")]


def kernel_source_digest() -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        h.update(open(f, "rb").read())
    return h.hexdigest()


def traffic_record() -> float | None:
    """DRAM bytes (read + write) per launch of the attention kernel, from the
    committed ncu summary, if that summary was taken on the kernel sources as
    they are now (its `kernel_source_sha256:` line); else None."""
    try:
        text = open(TRAFFIC_SUMMARY).read()
    except OSError:
        return None
    sha = re.search(r"^kernel_source_sha256:\s*([0-9a-f]{64})", text, re.M)
    val = re.search(r"^dram_bytes_per_launch:\s*([0-9.eE+]+)", text, re.M)
    if not sha or not val or sha.group(1) != kernel_source_digest():
        return None
    return float(val.group(1))


def selected_rows(topk: torch.Tensor, end_pos: torch.Tensor) -> int:
    e = end_pos.view(-1, 1).to(topk.device)
    return int(((topk >= 0) & (topk < e)).sum().item())


def oracle_sample(t: dict, wl, budget_s: float, max_seqs: int | None = None):
    """Time the float64 oracle's full step on sequences 0, 1, ... (cycling over
    the batch) until the budget is used (at least one; at most max_seqs).
    Returns (sequence-steps, seconds)."""
    from oracle import mla_oracle as O
    from sparse_latent_attention_decode_b300 import synth
    inv = O.yarn_inv_freq()
    scale = O.softmax_scale()
    wkv = synth.to_f64(t["wkv_b"])
    done, spent = 0, 0.0
    limit = None if max_seqs is None else max_seqs
    while (limit is None or done < limit) and (done == 0 or spent < budget_s):
        b = done % wl.B
        x = {k: synth.to_f64(t[k][b:b + 1]) for k in ("q_nope", "q_pe", "kv_cache", "pe_cache", "topk_idx",
                                                     "end_pos")}
        t0 = time.perf_counter()
        O.decode_step(x["q_nope"], x["q_pe"], x["kv_cache"], x["pe_cache"], wkv, x["topk_idx"], x["end_pos"],
                      inv, scale)
        spent += time.perf_counter() - t0
        done += 1
    return done, spent


# ----------------------------------------------------------------- our arm
class L2Flush:
    """Evicts L2 before a timed launch: writes a 256 MiB buffer (> the 126 MB
    L2), then reads a second one, so that the lines left in L2 are clean and
    none of the flush's dirty lines is written back during the timed work."""

    def __init__(self, dev):
        self.w = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
        self.r = torch.ones(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        self.acc = torch.empty((), dtype=torch.float32, device=dev)

    def __call__(self, i: int = 0):
        self.w.fill_(i & 0xFF)
        torch.sum(self.r, dim=0, out=self.acc)


def time_single_kernel(fn, n: int, flush) -> float:
    """Mean device time (ms) of fn(), which enqueues one library kernel on the
    current stream, with L2 flushed before each launch."""
    for i in range(3):
        flush(i)
        fn()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * n)]
    torch.cuda.synchronize()
    for i in range(n):
        flush((i + 5) & 0xFF)
        ev[2 * i].record()
        fn()
        ev[2 * i + 1].record()
    torch.cuda.synchronize()
    return statistics.mean(ev[2 * i].elapsed_time(ev[2 * i + 1]) for i in range(n))


def measure_next_rows(mla, synth, dev, flush, seed: int, n: int = 50) -> dict:
    """The entry points beyond the decode step, each on its own workload:
    algorithmic bytes per launch and the event-timed launch duration."""
    out = {}
    # half-split RoPE of an indexer-shaped query: 64 sequences x 64 heads x 64
    B, nh = 64, 64
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(B, nh, 64, generator=g).to(torch.bfloat16).to(dev)
    end = torch.randint(1, 16385, (B,), generator=g, dtype=torch.int32).to(dev)
    cis = mla.rope_freqs_init(device=dev)
    y = torch.empty(B, nh, 64, dtype=torch.float32, device=dev)
    ms = time_single_kernel(lambda: mla.mla_rope_apply_layout(x, cis, end, False, out=y), n, flush)
    nbytes = B * nh * 64 * (2 + 4) + B * 32 * 8 + B * 4
    out["rope_half_split"] = {"workload": f"B={B} x {nh} heads x 64, end_pos uniform in [1, 16384]",
                              "kernel_ms": ms, "alg_bytes_per_launch": nbytes,
                              "achieved_gbs": nbytes / (ms * 1e-3) / 1e9}
    # fp8 wkv_b dequantisation: 32768 x 512 e4m3 codes, 128 x 128 tiles
    codes, scale = synth.make_fp8_weight(seed)
    codes, scale = codes.to(dev), scale.to(dev)
    w = torch.empty(codes.shape, dtype=torch.bfloat16, device=dev)
    ms = time_single_kernel(lambda: mla.mla_weight_dequant_fp8(codes, scale, out=w), n, flush)
    nbytes = codes.numel() * 3 + scale.numel() * 4
    out["weight_dequant_fp8"] = {"workload": "wkv_b 32768 x 512 e4m3, fp32 scale per 128 x 128 tile",
                                 "kernel_ms": ms, "alg_bytes_per_launch": nbytes,
                                 "achieved_gbs": nbytes / (ms * 1e-3) / 1e9}
    del codes, scale, w
    # cache append of one new token for 64 sequences (RMSNorm + rotary key)
    S_app = 4096
    kv_a = torch.randn(B, 1, 576, generator=g).to(torch.bfloat16).to(dev)
    norm_w = torch.ones(512, dtype=torch.float32, device=dev)
    kvc = torch.zeros(B, S_app, 512, dtype=torch.bfloat16, device=dev)
    pec = torch.zeros(B, S_app, 64, dtype=torch.bfloat16, device=dev)
    end_a = torch.randint(1, S_app + 1, (B,), generator=g, dtype=torch.int32).to(dev)
    ms = time_single_kernel(lambda: mla.mla_cache_append(kv_a, norm_w, cis, end_a, kvc, pec), n, flush)
    nbytes = B * (576 * 2 + 512 * 2 + 64 * 2 + 32 * 8 + 4) + 512 * 4
    out["cache_append"] = {"workload": f"B={B}, 1 token each, S_cap {S_app}", "kernel_ms": ms,
                           "alg_bytes_per_launch": nbytes, "achieved_gbs": nbytes / (ms * 1e-3) / 1e9}
    del kvc, pec
    # the projections around the attention; the model width 7168 is the
    # DeepSeek-V3 value (the pages leave dim out)
    for name, (M, N, K) in (("linear_wkv_a", (B, 576, 7168)), ("linear_wo", (B, 7168, 128 * 128))):
        x, w = synth.make_linear_inputs(seed, M, N, K, name=name)
        x, w = x.to(dev), w.to(dev)
        y = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
        ws = torch.empty(mla.linear_workspace_size(M, N, K), dtype=torch.uint8, device=dev)
        ms = time_single_kernel(lambda: mla.mla_linear_bf16(x, w, out_dtype=torch.bfloat16, out=y, workspace=ws),
                                n, flush)
        nbytes = (N * K + M * K + M * N) * 2
        out[name] = {"workload": f"M={M} tokens, N={N}, K={K}, bf16 in and out (weight and split-K reduction "
                                 f"in one timed call)", "kernel_ms": ms, "alg_bytes_per_launch": nbytes,
                     "achieved_gbs": nbytes / (ms * 1e-3) / 1e9}
        del x, w, y, ws
    return out


def measure_multi_token(mla, step, d, B, K, rows, flush, n: int = 50) -> dict:
    """Multi-token decode over the bench caches: B/2 sequences x 2 query tokens
    (the step's own q_lat and selections regrouped), the attention kernel
    timed alone by the library's events around it."""
    n_seq, T = B // 2, 2
    q = step.q_lat.view(n_seq, T, 128, 576)
    top = d["topk_idx"].view(n_seq, T, K)
    end = d["end_pos"][:n_seq].contiguous()
    kv, pe = d["kv_cache"][:n_seq], d["pe_cache"][:n_seq]
    out = torch.empty(n_seq, T, 128, 128, dtype=torch.float32, device=q.device)
    ws = torch.empty(mla.workspace_size(n_seq * T, K), dtype=torch.uint8, device=q.device)
    call = lambda: mla.mla_sparse_decode_tokens(q, kv, pe, top, end, step.scale, wkv_b=d["wkv_b"], out=out,
                                                workspace=ws)
    for i in range(3):
        call()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * n)]
    for e in ev:
        e.record()
    torch.cuda.synchronize()
    with mla.ProfileHook() as hook:
        for i in range(n):
            flush((i + 13) & 0xFF)
            hook.set_events(ev[2 * i], ev[2 * i + 1])
            call()
    torch.cuda.synchronize()
    ms = statistics.mean(ev[2 * i].elapsed_time(ev[2 * i + 1]) for i in range(n))
    # selected rows a token can see: its selection minus positions after it
    pos = end[:, None].long() - T + torch.arange(T, device=q.device)[None, :]
    vis = int(((top >= 0) & (top.long() <= pos[:, :, None])).sum().item())
    nbytes = vis * ROW_BYTES
    return {"workload": f"{n_seq} sequences x {T} tokens, end_pos {int(end[0])}, top-{K} per token, causal",
            "kernel_ms": ms, "alg_bytes_per_launch": nbytes, "achieved_gbs": nbytes / (ms * 1e-3) / 1e9}


FLOP_PER_ROW = 128 * (576 + 512) * 2   # scores (K=576) and PV (N=512) of all heads for one selected row


def roofline(alg_bytes: int, flops: int, ms: float, hbm_gbs: float, tflops: float) -> dict:
    """The slower of the kernel's two bounds (HBM bytes at the copy peak,
    FLOPs at the bf16 tensor peak) and the fraction of it the kernel reaches."""
    t_hbm = alg_bytes / (hbm_gbs * 1e9)
    t_tc = flops / (tflops * 1e12)
    sec = ms * 1e-3
    if t_hbm >= t_tc:
        return {"bound": "hbm", "achieved": alg_bytes / sec / 1e9, "peak": hbm_gbs, "unit": "GB/s",
                "frac": t_hbm / sec, "ideal_ms": t_hbm * 1e3, "other_bound_ms": t_tc * 1e3}
    return {"bound": "tensor", "achieved": flops / sec / 1e12, "peak": tflops, "unit": "TFLOP/s",
            "frac": t_tc / sec, "ideal_ms": t_tc * 1e3, "other_bound_ms": t_hbm * 1e3}


def timed_chunks(fn, n: int, chunks: int = 20) -> list:
    """Per-call device time (ms) of n back-to-back calls of fn(i), measured by
    CUDA events around consecutive chunks of calls (no synchronisation inside)."""
    per = max(1, n // chunks)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(n // per + 2)]
    ev[0].record()
    k, done = 0, 0
    while done < n:
        m = min(per, n - done)
        for i in range(done, done + m):
            fn(i)
        done += m
        k += 1
        ev[k].record()
    torch.cuda.synchronize()
    out = []
    done = 0
    for c in range(k):
        m = min(per, n - done)
        out.append((ev[c].elapsed_time(ev[c + 1]) / m, m))
        done += m
    return out


def measure_workload(mla, synth, name: str, dev, flush, args, rank: int, world: int, peaks: dict,
                     clocks=None, soak_s: float = 0.0):
    """One named workload.

    The step: R = --rotate input sets -- the workload's tensors and R-1 device
    copies of them (caches, wkv_b, query parts, selection, end_pos), each with
    its own captured step -- so that consecutive steps share no buffer and
    each step's working set (its gathered rows plus wkv_b) is larger than L2.
    The timed steps replay the sets in turn, back to back, timed by CUDA events
    around chunks of consecutive replays.  The same replays are also timed one
    at a time with L2 flushed before each (events around every replay).

    The attention kernel: back-to-back launches of the step's own attention
    call (bf16 latent output, no up-projection) over the rotating sets, when
    that call is the attention kernel alone (no split combine); and, for every
    workload, one launch at a time with L2 flushed before it (library events
    right around the kernel inside the step)."""
    wl = synth.workload(name, seed=replica_seed(rank, args.seed))
    t = synth.make_inputs(wl, seed=replica_seed(rank, args.seed))
    d = {k: v.to(dev) for k, v in t.items()}
    ROTATE = max(1, args.rotate)
    sets = [d] + [{k: v.clone() for k, v in d.items()} for _ in range(ROTATE - 1)]
    B, K = wl.B, wl.row_stride()
    rows = selected_rows(d["topk_idx"], d["end_pos"])
    argsets = [(s_["q_nope"], s_["q_pe"], s_["kv_cache"], s_["pe_cache"], s_["wkv_b"], s_["topk_idx"],
                s_["end_pos"]) for s_ in sets]
    steps = [mla.DecodeStep(B, K, device=dev) for _ in range(ROTATE)]
    graphs = [mla.CapturedStep(steps[r], *argsets[r]) for r in range(ROTATE)]
    step, graph, args_dev = steps[0], graphs[0], argsets[0]
    for i in range(max(args.warmup, ROTATE)):
        graphs[i % ROTATE]()
    torch.cuda.synchronize()
    for r in range(1, ROTATE):
        assert torch.equal(graphs[r].out, graphs[0].out), "rotating input sets disagree"

    # ---- the timed steps: back-to-back replays over the rotating sets; an
    # untimed soak of the same replays around them keeps the clocks sampled
    def soak():
        t_end = time.perf_counter() + soak_s
        while time.perf_counter() < t_end:
            for i in range(50):
                graphs[i % ROTATE]()
            torch.cuda.synchronize()

    if clocks is not None:
        clocks.open_window()
        soak()
    barrier(world)
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    chunks = timed_chunks(lambda i: graphs[i % ROTATE](), args.steps)
    wall = time.perf_counter() - t_wall
    barrier(world)
    if clocks is not None:
        soak()
        clocks.close_window()
    for st_ in steps:
        st_.check_status()
    ms = sum(c * m for c, m in chunks) / args.steps
    ms_max = max_over_ranks(ms, world, dev)

    # ---- the same steps one at a time, L2 flushed before each
    n_fl = max(3, min(args.steps, args.flushed_steps))
    st = [torch.cuda.Event(enable_timing=True) for _ in range(2 * n_fl)]
    for i in range(n_fl):
        flush(i + 7)
        st[2 * i].record()
        graphs[i % ROTATE]()
        st[2 * i + 1].record()
    torch.cuda.synchronize()
    step_fl = [st[2 * i].elapsed_time(st[2 * i + 1]) for i in range(n_fl)]

    # ---- the attention kernel alone, back to back over the rotating sets
    att_out = [torch.empty(B, 1, 128, 512, dtype=torch.bfloat16, device=dev) for _ in range(ROTATE)]
    att_ws = [torch.empty(mla.workspace_size(B, K), dtype=torch.uint8, device=dev) for _ in range(ROTATE)]

    def att(i):
        r = i % ROTATE
        s_ = sets[r]
        mla.mla_sparse_decode_tokens(steps[r].q_lat[:, None], s_["kv_cache"], s_["pe_cache"], s_["topk_idx"][:, None],
                                     s_["end_pos"], step.scale, out=att_out[r], workspace=att_ws[r],
                                     out_dtype=torch.bfloat16)

    with mla.ProfileHook() as h:
        att(0)
    kern_b2b = None
    n_kern = max(3, min(args.steps, args.kernel_steps))
    if h.launches == 1:
        for i in range(ROTATE):
            att(i)
        torch.cuda.synchronize()
        kc = timed_chunks(att, n_kern)
        kern_b2b = sum(c * m for c, m in kc) / n_kern

    # ---- the attention kernel alone, one launch at a time: CUDA events recorded
    # by the library on the launching stream right before and after it, L2 flushed
    kt = [torch.cuda.Event(enable_timing=True) for _ in range(2 * n_kern)]
    for ev in kt:       # the library re-records these on the launching stream; a first record
        ev.record()     # through torch marks them recorded for torch's elapsed_time()
    torch.cuda.synchronize()
    with mla.ProfileHook() as khook:
        for i in range(n_kern):
            flush(i + 11)
            khook.set_events(kt[2 * i], kt[2 * i + 1])
            step(*args_dev)
    torch.cuda.synchronize()
    step.check_status()
    kern_all = [kt[2 * i].elapsed_time(kt[2 * i + 1]) for i in range(n_kern)]
    kern_iso = statistics.mean(kern_all)
    kern = kern_b2b if kern_b2b is not None else kern_iso

    hbm = float(peaks.get("hbm_gbs") or FALLBACK_HBM_GBS)
    tf = float(peaks.get("bf16_tflops") or FALLBACK_BF16_TFLOPS)
    alg_bytes = rows * ROW_BYTES
    flops = rows * FLOP_PER_ROW
    step_bytes = alg_bytes + d["wkv_b"].numel() * 2
    rec = {
        "workload": name, "batch": B, "topk_row": K,
        "end_pos": wl.end_pos[0] if len(set(wl.end_pos)) == 1 else f"{min(wl.end_pos)}..{max(wl.end_pos)}",
        "selection": wl.selection, "selected_rows": rows,
        "ms_per_step": ms_max, "ms_per_step_median": statistics.median(c for c, _ in chunks),
        "tokens_per_s": world * B / (ms_max * 1e-3),
        "ms_per_step_flushed": statistics.mean(step_fl), "ms_per_step_flushed_median": statistics.median(step_fl),
        "kernel_ms": kern,
        "kernel_timing": ("back-to-back launches over the rotating input sets, events around chunks"
                          if kern_b2b is not None else
                          "one launch at a time, L2 flushed, library events around the kernel (the attention "
                          "call also runs a split combine, so it is not timed back to back)"),
        "kernel_ms_isolated": kern_iso, "kernel_ms_isolated_median": statistics.median(kern_all),
        "alg_bytes_per_launch": alg_bytes, "flops_per_launch": flops,
        "roofline": roofline(alg_bytes, flops, kern, hbm, tf),
        "roofline_isolated": roofline(alg_bytes, flops, kern_iso, hbm, tf),
        "step_roofline": {"bytes": step_bytes, "ideal_ms": step_bytes / (hbm * 1e9) * 1e3,
                          "frac": step_bytes / (hbm * 1e9) * 1e3 / ms_max,
                          "note": "gathered rows x 1152 B + one read of wkv_b, at the copy peak"},
        "launches_per_step": graph.kernels_per_replay, "wall_s_timed_region": wall,
    }
    del graphs[1:], steps[1:], sets[1:], att_out, att_ws
    return rec, d, t, wl, step, graph


def measure_fused_step(mla, synth, d, B, K, rows, flush, seed: int, n: int = 50, dim: int = 7168) -> dict:
    """The attention block's whole decode step for one new token per sequence
    (FusedDecodeStep: wkv_a projection, cache append, absorption, attention
    with the up-projection, wo projection) on the bench caches, captured in
    one CUDA graph; each replay timed with L2 flushed before it.  The model
    width 7168 is the DeepSeek-V3 value (the pages leave dim out)."""
    dev = d["kv_cache"].device
    x, wkv_a = synth.make_linear_inputs(seed + 11, B, 576, dim, name="fused/wkv_a")
    _, wo = synth.make_linear_inputs(seed + 12, 1, dim, 128 * 128, name="fused/wo")
    x, wkv_a, wo = x.to(dev), wkv_a.to(dev), wo.to(dev)
    norm_w = torch.ones(512, dtype=torch.float32, device=dev)
    step = mla.FusedDecodeStep(B, K, dim, device=dev)
    g = mla.CapturedStep(step, x, d["q_nope"], d["q_pe"], d["kv_cache"], d["pe_cache"], wkv_a, norm_w, d["wkv_b"],
                         wo, d["topk_idx"], d["end_pos"])
    for i in range(3):
        flush(i)
        g()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * n)]
    torch.cuda.synchronize()
    for i in range(n):
        flush(i + 17)
        ev[2 * i].record()
        g()
        ev[2 * i + 1].record()
    torch.cuda.synchronize()
    step.check_status()
    ms = statistics.mean(ev[2 * i].elapsed_time(ev[2 * i + 1]) for i in range(n))
    nbytes = (wkv_a.numel() + wo.numel() + d["wkv_b"].numel() + x.numel()) * 2 + rows * ROW_BYTES + \
        B * (576 * 2 + 1152) + B * dim * 2
    return {"workload": f"B={B} new tokens, dim {dim}, top-{K} over the bench caches: wkv_a -> cache append -> "
                        f"absorb -> attention + up-projection -> wo, one graph replay",
            "kernel_ms": ms, "kernels_per_step": g.kernels_per_replay, "alg_bytes_per_launch": nbytes,
            "achieved_gbs": nbytes / (ms * 1e-3) / 1e9}


def run_ours(args):
    from sparse_latent_attention_decode_b300 import mla, synth

    rank, world, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (no CPU fallback)")
    torch.cuda.set_device(local)
    dist_init(world, "nccl")
    dev = torch.device("cuda", local)
    flush = L2Flush(dev)
    peaks = measured_peaks()
    peak_src = "measured" if peaks.get("hbm_gbs") else "fallback"
    clocks = ClockSampler(local)

    names = [args.workload]
    if args.configs == "all":
        names += [n for n in synth.WORKLOADS if n != args.workload]
    elif args.configs not in ("none", ""):
        names += [n for n in args.configs.split(",") if n and n != args.workload]

    configs = {}
    head = None
    for name in names:
        is_head = name == args.workload
        rec, d, t, wl, step, graph = measure_workload(mla, synth, name, dev, flush, args, rank, world, peaks,
                                                      clocks=clocks if is_head else None,
                                                      soak_s=args.clock_soak if is_head else 0.0)
        configs[name] = rec
        if is_head:
            head = (rec, d, t, wl, step, graph)
        else:
            del d, t, step, graph
            torch.cuda.empty_cache()
    clk = clocks.summary()
    rec, d, t, wl, step, graph = head
    B, K = wl.B, wl.row_stride()

    # ---- end to end through the host-buffer API: every step copies its inputs
    # in from pinned host memory and its head outputs (bf16, the dtype the
    # output projection takes) back; each step is one replay of a CUDA graph
    # holding the copies and the three library calls, and two buffer sets on
    # two streams alternate so that one step's transfers overlap the other's
    # compute.  No L2 flush here: the caches the step gathers from (1.2 GB)
    # are far larger than L2.
    pipe = mla.CapturedHostPipeline(B, K, d["kv_cache"], d["pe_cache"], d["wkv_b"], device=dev)
    for k in range(2):
        for name in ("q_nope", "q_pe", "topk_idx", "end_pos"):
            pipe.host_inputs(k)[name].copy_(t[name])
    for i in range(args.warmup):
        pipe.submit()
    pipe.finish()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    cur = torch.cuda.current_stream(dev)
    e0.record()
    for st_ in pipe.streams:
        st_.wait_stream(cur)
    for i in range(args.steps):
        pipe.submit()
    pipe.finish()
    e1.record()
    torch.cuda.synchronize()
    barrier(world)
    pipe.check_status()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, world, dev)

    next_rows = measure_next_rows(mla, synth, dev, flush, args.seed, n=args.next_steps)
    next_rows["fused_step"] = measure_fused_step(mla, synth, d, B, K, rec["selected_rows"], flush, args.seed,
                                                 n=args.next_steps)
    if B % 2 == 0:
        next_rows["multi_token_decode"] = measure_multi_token(mla, step, d, B, K, rec["selected_rows"], flush,
                                                              n=args.next_steps)

    if rank != 0:
        return None

    hbm = float(peaks.get("hbm_gbs") or FALLBACK_HBM_GBS)
    read_peak = read_stream_gbs(dev)
    traffic = traffic_record()
    roof = dict(rec["roofline"])
    roof.update({"kernel": "mla_sparse_decode attention kernel", "traffic": traffic,
                 "peak_source": f"{peak_src} hbm_gbs / bf16_tflops (burst: the kernel is timed alone)",
                 "alg_bytes_per_launch": rec["alg_bytes_per_launch"], "flops_per_launch": rec["flops_per_launch"],
                 "kernel_ms": rec["kernel_ms"], "kernel_timing": rec["kernel_timing"],
                 "isolated": {"kernel_ms": rec["kernel_ms_isolated"],
                              "frac": rec["roofline_isolated"]["frac"],
                              "timing": "one launch at a time, L2 flushed, events right around the kernel"},
                 "read_stream_gbs": read_peak,
                 "frac_of_read_stream": rec["alg_bytes_per_launch"] / (rec["kernel_ms"] * 1e-3) / 1e9 / read_peak})

    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        n, secs = oracle_sample(t, wl, budget_s=args.cpu_budget)
        cpu = {"value": n / secs, "unit": UNIT, "cores": len(os.sched_getaffinity(0)), "kind": "oracle",
               "sample": f"{n} sequence-steps of the {args.workload} batch (sequences taken in order, "
                         f"cycling over the {B} of the batch); float64 numpy, full step per sequence (RoPE, "
                         f"absorb, masked scores over all end_pos keys, softmax, PV, up-projection); {secs:.1f} s"}

    ms_max = rec["ms_per_step"]
    line = {
        "metric": METRIC, "value": world * B / (ms_max * 1e-3), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max,
        "ms_per_step_median": rec["ms_per_step_median"], "ms_per_step_flushed": rec["ms_per_step_flushed"],
        "ms_per_step_flushed_median": rec["ms_per_step_flushed_median"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": args.workload, "batch_per_gpu": B, "global_batch": world * B,
                   "end_pos": rec["end_pos"], "topk_row": K, "selected_rows_per_gpu": rec["selected_rows"],
                   "S_cap": wl.S_cap, "heads": 128, "kv_lora": 512, "rope_dim": 64,
                   "l2": f"inputs larger than L2: the timed steps rotate over {args.rotate} input sets (the "
                         f"workload's tensors and {args.rotate - 1} device copies), consecutive steps share no "
                         "buffer; ms_per_step_flushed: "
                         "one step at a time with L2 flushed before each (256 MiB written, then 256 MiB read)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "e2e": {"value": world * B / (e2e_ms * 1e-3), "unit": UNIT, "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": pipe.h2d_bytes(), "d2h_bytes_per_step": pipe.d2h_bytes(),
                "out_dtype": "bf16",
                "path": "CapturedHostPipeline: each step one graph replay (pinned host inputs copied in, three "
                        "library calls, head outputs copied back); two buffer sets on two streams overlap one "
                        "step's copies with the other's compute; no L2 flush (the caches exceed L2)"},
        "roofline": roof,
        "step_roofline": rec["step_roofline"],
        "configs": {k: v for k, v in configs.items()},
        "cpu_baseline": cpu,
        "next_rows": {k: dict(v, frac=v["achieved_gbs"] / hbm) for k, v in next_rows.items()},
        "clocks": clk,
        "gpu_launches": rec["launches_per_step"] * args.steps,
        "wall_s_timed_region": rec["wall_s_timed_region"],
    }
    return line


# ----------------------------------------------------------------- reference arm (the oracle)
def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return None
    from sparse_latent_attention_decode_b300 import synth
    wl = synth.workload(args.workload, seed=replica_seed(0, args.seed))
    t = synth.make_inputs(wl, seed=replica_seed(0, args.seed))
    from oracle import mla_oracle as O
    inv, scale = O.yarn_inv_freq(), O.softmax_scale()
    wkv = synth.to_f64(t["wkv_b"])
    n_total = args.warmup + args.steps
    times = []
    for i in range(n_total):
        # one step: one sequence of the batch, one block of REF_HEADS consecutive
        # heads (the step is independent per head), cycling over both
        b = i % wl.B
        h0 = (i // wl.B * REF_HEADS) % 128
        x = {k: synth.to_f64(t[k][b:b + 1]) for k in ("kv_cache", "pe_cache", "topk_idx", "end_pos")}
        qn = synth.to_f64(t["q_nope"][b:b + 1, h0:h0 + REF_HEADS])
        qp = synth.to_f64(t["q_pe"][b:b + 1, h0:h0 + REF_HEADS])
        w = wkv[h0 * 256:(h0 + REF_HEADS) * 256]
        t0 = time.perf_counter()
        O.decode_step(qn, qp, x["kv_cache"], x["pe_cache"], w, x["topk_idx"], x["end_pos"], inv, scale)
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    sec = statistics.mean(times) * (128 / REF_HEADS)   # seconds per query token (all 128 heads)
    v = 1.0 / sec
    return {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": args.workload, "batch_per_step": 1, "heads_per_step": REF_HEADS,
                       "S_cap": wl.S_cap,
                       "note": "float64 CPU oracle; value = query tokens/s scaled from the head sample"},
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": len(os.sched_getaffinity(0)), "kind": "oracle",
                             "sample": f"per step one sequence of {args.workload} and {REF_HEADS} of its 128 heads "
                                       f"(cycling), {args.steps} steps; time scaled by 128/{REF_HEADS} to one "
                                       f"query token"},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def spawn_ranks(argv, n: int) -> int:
    """Start n ranks of this script through torch.distributed.run on this
    node (rendezvous on 127.0.0.1); returns the launcher's exit code."""
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
           "--master-addr=127.0.0.1", f"--master-port={port}", os.path.abspath(__file__), *argv]
    return subprocess.call(cmd)


def main(argv=None):
    argv = list(sys.argv[1:] if argv is None else argv)
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000, help="timed steps per workload")
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--rotate", type=int, default=4,
                    help="input sets the timed steps rotate over (1: one set, e.g. for a profiler capture)")
    ap.add_argument("--flushed-steps", type=int, default=200,
                    help="steps also timed one at a time with L2 flushed before each")
    ap.add_argument("--kernel-steps", type=int, default=200,
                    help="extra steps in which the attention kernel alone is timed")
    ap.add_argument("--next-steps", type=int, default=50,
                    help="timed launches per added entry point (next_rows)")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, help="the headline workload")
    ap.add_argument("--configs", default="all",
                    help="workloads measured besides the headline: all, none, or a comma-separated list")
    ap.add_argument("--clock-soak", type=float, default=1.0,
                    help="seconds of untimed replays before and after the headline's timed steps, "
                         "during which the clocks are sampled too")
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle time for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)
    args.warmup = max(args.warmup, 3)   # timing rule: at least 3 untimed warm-up steps
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        # started without torchrun: one process per GPU, launched from here
        raise SystemExit(spawn_ranks(argv, args.gpus))
    line = run_reference(args) if args.impl == "reference" else run_ours(args)
    if line is not None:
        print(json.dumps(line), flush=True)
    rank, world, _ = dist_env()
    if world > 1:
        import torch.distributed as dist
        if dist.is_initialized():
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
