#!/usr/bin/env python
"""Benchmark of one decode step of absorbed, top-k-sparse latent attention.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is the whole path for one batch: RoPE + key absorption
(mla_absorb_q), then scores / softmax / PV / value up-projection
(mla_sparse_decode with wkv_b).  Inputs are seeded synthetic tensors already
resident in HBM; the step is captured once in a CUDA graph and each timed
step is one replay; L2 is flushed (a 256 MiB write) before every timed step
and each step is timed with its own CUDA events on the launching stream.

With N > 1 (torchrun, one process per GPU) each rank runs an independent
replica on its own batch (different seed): no collective on the data path,
weak scaling; a barrier and a max-over-ranks reduction bracket the timing.

The line printed by rank 0 also carries: the end-to-end figure through the
host-buffer API (each step's pinned host inputs copied in and head outputs
copied back, transfers overlapped across steps by HostDecodePipeline), the
roofline of the attention kernel, the float64 oracle timed on a bounded sample
on the host cores (cpu_baseline), GPU clocks sampled during the timed region,
and the number of library kernels launched in the timed region.

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
import tempfile
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
class ClockSampler:
    """nvidia-smi samples (100 ms) of the bench GPU; only samples taken
    between mark_start() and mark_stop() (the timed region) are kept."""

    FIELDS = ("timestamp,index,pci.bus_id,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.path = None
        self.t0 = self.t1 = None
        try:
            props = torch.cuda.get_device_properties(device_index)
            self.bus = f"{props.pci_bus_id:02X}:{props.pci_device_id:02X}."
        except Exception:
            self.bus = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "100", "-f", self.path],
                                         stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
            time.sleep(0.6)   # let the sampler come up before the timed region
        except Exception:
            self.proc = None

    def mark_start(self):
        self.t0 = time.time()

    def mark_stop(self):
        self.t1 = time.time()

    def stop(self) -> dict | None:
        if self.proc is None:
            return None
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        import datetime
        rows = []
        try:
            for line in open(self.path):
                f = [x.strip() for x in line.split(",")]
                if len(f) < 11:
                    continue
                try:
                    ts = datetime.datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                except ValueError:
                    continue
                if self.t0 is not None and not (self.t0 <= ts <= (self.t1 or ts)):
                    continue
                rows.append(f[1:])
        finally:
            os.unlink(self.path)
        mine = [r for r in rows if self.bus and self.bus in r[1].upper()]
        if mine or len({r[0] for r in rows}) > 1:
            rows = mine
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[2]) for r in rows if num(r[2]) is not None]
        mx = [num(r[3]) for r in rows if num(r[3]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[6 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


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
def time_single_kernel(fn, n: int, flush) -> float:
    """Mean device time (ms) of fn(), which enqueues one library kernel on the
    current stream, with L2 flushed before each launch."""
    for i in range(3):
        flush.fill_(i)
        fn()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * n)]
    torch.cuda.synchronize()
    for i in range(n):
        flush.fill_((i + 5) & 0xFF)
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
            flush.fill_((i + 13) & 0xFF)
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


def run_ours(args):
    from sparse_latent_attention_decode_b300 import mla, synth

    rank, world, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (no CPU fallback)")
    torch.cuda.set_device(local)
    dist_init(world, "nccl")
    dev = torch.device("cuda", local)

    wl = synth.workload(args.workload, seed=replica_seed(rank, args.seed))
    t = synth.make_inputs(wl, seed=replica_seed(rank, args.seed))
    d = {k: v.to(dev) for k, v in t.items()}
    B, K = wl.B, wl.row_stride()
    rows = selected_rows(d["topk_idx"], d["end_pos"])
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    step = mla.DecodeStep(B, K, device=dev)
    args_dev = (d["q_nope"], d["q_pe"], d["kv_cache"], d["pe_cache"], d["wkv_b"], d["topk_idx"], d["end_pos"])

    # ---- device-resident inputs: the timed steps, each one replay of the step
    # captured in a CUDA graph (kernels chained by programmatic dependent
    # launch, nothing recorded between them)
    graph = mla.CapturedStep(step, *args_dev)
    for i in range(args.warmup):
        flush.fill_(i & 0xFF)
        graph()
    torch.cuda.synchronize()
    st = [torch.cuda.Event(enable_timing=True) for _ in range(2 * args.steps)]
    clocks = ClockSampler(local)
    clocks.start()
    barrier(world)
    torch.cuda.synchronize()
    clocks.mark_start()
    t_wall = time.perf_counter()
    for i in range(args.steps):
        flush.fill_((i + 7) & 0xFF)
        st[2 * i].record()
        graph()
        st[2 * i + 1].record()
    launches = graph.kernels_per_replay * args.steps
    torch.cuda.synchronize()
    barrier(world)
    wall = time.perf_counter() - t_wall
    clocks.mark_stop()
    clk = clocks.stop()
    step.check_status()
    step_ms = [st[2 * i].elapsed_time(st[2 * i + 1]) for i in range(args.steps)]
    ms = statistics.mean(step_ms)
    ms_max = max_over_ranks(ms, world, dev)
    ms_median = statistics.median(step_ms)

    # ---- the attention kernel alone: CUDA events recorded by the library on
    # the launching stream right before and after it (these steps are not the
    # timed ones: an event between two kernels separates them)
    n_kern = min(args.steps, args.kernel_steps)
    kt = [torch.cuda.Event(enable_timing=True) for _ in range(2 * n_kern)]
    for ev in kt:       # the library re-records these on the launching stream; a first record
        ev.record()     # through torch marks them recorded for torch's elapsed_time()
    torch.cuda.synchronize()
    with mla.ProfileHook() as khook:
        for i in range(n_kern):
            flush.fill_((i + 11) & 0xFF)
            khook.set_events(kt[2 * i], kt[2 * i + 1])
            step(*args_dev)
    torch.cuda.synchronize()
    step.check_status()
    kern = statistics.mean(kt[2 * i].elapsed_time(kt[2 * i + 1]) for i in range(n_kern))

    # ---- end to end through the host-buffer API: every step copies its inputs
    # in from pinned host memory and its head outputs back; the pipeline
    # overlaps step i's transfers with its neighbours' compute.  No L2 flush
    # here: the caches the step gathers from (1.2 GB) are far larger than L2.
    h = {k: t[k].pin_memory() for k in ("q_nope", "q_pe", "topk_idx", "end_pos")}
    pipe = mla.HostDecodePipeline(B, K, device=dev)
    h_outs = [torch.empty(B, 128, 128, dtype=torch.float32).pin_memory() for _ in range(2)]
    hargs = (h["q_nope"], h["q_pe"], h["topk_idx"], h["end_pos"], d["kv_cache"], d["pe_cache"], d["wkv_b"])
    for i in range(args.warmup):
        pipe.submit(*hargs, h_outs[i % 2])
    pipe.finish()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    e0.record()
    for i in range(args.steps):
        pipe.submit(*hargs, h_outs[i % 2])
    pipe.finish()
    e1.record()
    torch.cuda.synchronize()
    barrier(world)
    pipe.check_status()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, world, dev)

    next_rows = measure_next_rows(mla, synth, dev, flush, args.seed, n=args.next_steps)
    if B % 2 == 0:
        next_rows["multi_token_decode"] = measure_multi_token(mla, step, d, B, K, rows, flush, n=args.next_steps)

    if rank != 0:
        return None

    peaks = measured_peaks()
    hbm = peaks.get("hbm_gbs")
    peak_src = "measured" if hbm else "fallback"
    hbm = float(hbm) if hbm else FALLBACK_HBM_GBS
    alg_bytes = rows * ROW_BYTES
    achieved = alg_bytes / (kern * 1e-3) / 1e9
    read_peak = read_stream_gbs(dev)
    # the whole step's ideal time: the gathered rows plus one read of wkv_b
    step_bytes = alg_bytes + d["wkv_b"].numel() * 2
    step_ideal_ms = step_bytes / (hbm * 1e9) * 1e3
    traffic = traffic_record()

    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        n, secs = oracle_sample(t, wl, budget_s=args.cpu_budget)
        cpu = {"value": n / secs, "unit": UNIT, "cores": len(os.sched_getaffinity(0)), "kind": "oracle",
               "sample": f"{n} sequence-steps of the {args.workload} batch (sequences taken in order, "
                         f"cycling over the {B} of the batch); float64 numpy, full step per sequence (RoPE, "
                         f"absorb, masked scores over all end_pos keys, softmax, PV, up-projection); {secs:.1f} s"}

    line = {
        "metric": METRIC, "value": world * B / (ms_max * 1e-3), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max, "ms_per_step_median": ms_median,
        "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": args.workload, "batch_per_gpu": B, "global_batch": world * B,
                   "end_pos": (wl.end_pos[0] if len(set(wl.end_pos)) == 1 else
                               f"{min(wl.end_pos)}..{max(wl.end_pos)}"),
                   "topk_row": K, "selected_rows_per_gpu": rows, "S_cap": wl.S_cap, "heads": 128,
                   "kv_lora": 512, "rope_dim": 64, "l2": "flushed by a 256 MiB write before each step",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "e2e": {"value": world * B / (e2e_ms * 1e-3), "unit": UNIT, "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": pipe.h2d_bytes(), "d2h_bytes_per_step": pipe.d2h_bytes(),
                "path": "HostDecodePipeline: per-step copies in and out, overlapped across steps; no L2 flush "
                        "(the caches exceed L2)"},
        "roofline": {"bound": "hbm", "kernel": "mla_sparse_decode attention kernel",
                     "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                     "peak_source": f"{peak_src} hbm_gbs", "traffic": traffic,
                     "alg_bytes_per_launch": alg_bytes, "kernel_ms": kern,
                     "read_stream_gbs": read_peak, "frac_of_read_stream": achieved / read_peak},
        "step_roofline": {"bytes": step_bytes, "ideal_ms": step_ideal_ms, "frac": step_ideal_ms / ms_max,
                          "note": "gathered rows x 1152 B + one read of wkv_b, at the copy peak"},
        "cpu_baseline": cpu,
        "next_rows": {k: dict(v, frac=v["achieved_gbs"] / hbm) for k, v in next_rows.items()},
        "clocks": clk,
        "gpu_launches": launches,
        "wall_s_timed_region": wall,
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


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4000,
                    help="timed steps (long enough for several clock samples)")
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--kernel-steps", type=int, default=200,
                    help="extra steps in which the attention kernel alone is timed")
    ap.add_argument("--next-steps", type=int, default=50,
                    help="timed launches per added entry point (next_rows)")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle time for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)
    args.warmup = max(args.warmup, 3)   # timing rule: at least 3 untimed warm-up steps
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
