"""Benchmark of the DSA indexer decode step on GB300.

One step = the whole hot path over one batch: paged_mqa_logits_metadata ->
fp8_fp4_paged_mqa_logits -> top_k_per_row, on the 40-request x ~120K-context
varlen speculative-decode workload (FP8 e4m3 q and keys, H = 64, D = 128,
block_kv = 64, 1..6 rows per request, top-k 2048) unless --workload says
otherwise.  Inputs are synthetic and seeded (workloads.config).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
    python bench.py --dcp-world R [--dcp-interleave I]
    python bench.py --logits-budget BYTES
    python bench.py --workload prefill

Prints one JSON line (rank 0).  `value` is device time per step with inputs
resident in HBM, the step (three kernels) replayed from a CUDA graph as a
serving loop runs it (`direct_launch_value`: the same steps launched call by
call); `e2e` is the same step through the C ABI from pinned host
buffers, with the per-step host->device input copies and the device->host
read of the top-k indices inside the timed region.  `--impl reference` times
the CPU oracle (the only other implementation of the method here) on a
bounded sample of the same workload and scales it to one step.

`--dcp-world R` times decode context parallelism on one GPU instead: each of
R ranks' steps (metadata, logits and top-k over its 1/R of every request's
keys, then the candidate pack) run in turn, the packs are stacked by a
device copy where R GPUs would all-gather them, and the merge kernel gives
the global top-k, which is checked against the unsharded step's.  It prints
one JSON line of per-rank and merge kernel times.

`--logits-budget BYTES` times the step as the one native call
dsa_indexer_decode_topk, its rows in slices whose logits fit BYTES (each
slice with its own schedule, one reused scratch), beside the same call
unsliced, and checks that both give the same top-k.

`--workload prefill` times the prefill step over the paged cache (row tags
-> lengths and requests, schedule, logits, top-k) on a chunk of 2 x 4096
rows of two 8192-token prompts; its roofline is the FP8 tensor rate.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import math
import os
import re
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = ("indexer decode µs/step + HBM GB/s (% roofline), 40 req × 120K ctx varlen")
PAGES_CONTEXT = ("pages: sm100_paged_mqa_logits 214.304 us -> 51.808 us (varlen) on an SM100 GPU, "
                 "GLM-5.3-Flash, 120K context, batch 40, 5 speculative steps (nsys); "
                 "another machine and kernel-only")
FP8_PEAK_RATIO = 2.0  # nominal dense fp8 : bf16 tensor rate
FP4_PER_FP8 = 3.0     # nominal dense fp4 : fp8 tensor rate of the part (13.5 : 4.5 PFLOP/s)


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="varlen",
                    choices=["tiny", "plain", "mtp", "varlen", "fp4_varlen", "mxfp4_varlen", "prefill"])
    ap.add_argument("--e2e-steps", type=int, default=500)
    ap.add_argument("--cpu-budget-s", type=float, default=12.0,
                    help="seconds of oracle work for the cpu_baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the per_config block (the other decode workloads, timed the same way)")
    ap.add_argument("--dcp-world", type=int, default=0,
                    help="time the decode-context-parallel step instead: the workload's keys split "
                         "over this many ranks, every rank emulated in turn on this GPU")
    ap.add_argument("--dcp-interleave", type=int, default=1)
    ap.add_argument("--logits-budget", type=int, default=0,
                    help="time the whole step as one native call whose rows run in slices "
                         "whose logits fit this many bytes")
    return ap.parse_args()


def max_over_ranks(x, device, world):
    """The largest of every rank's x (a float); x itself with one rank."""
    if world <= 1:
        return x
    import torch
    t = torch.tensor([float(x)], device=device, dtype=torch.float64)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


def workload_desc(name, wl):
    T = wl.num_rows
    fmt = ["FP8 e4m3", "FP4 e2m1 + e4m3/16 + fp32/token", "MXFP4 e2m1 + ue8m0/32"][wl.kv_format]
    qf = "MXFP4 e2m1 + ue8m0/32" if wl.q_scale is not None else "e4m3"
    return (f"{name}: B={len(wl.request_lens)} requests, context {min(wl.request_lens)}.."
            f"{max(wl.request_lens)}, rows/request {min(wl.rows_per_request)}.."
            f"{max(wl.rows_per_request)} (T={T}), q {qf}, keys {fmt}, H=64, D=128, "
            f"block_kv=64, top-k {wl.topk}, logits {'fp32' if wl.logits_dtype == 0 else 'bf16'}")


def algorithmic_bytes(wl):
    """Bytes the logits kernel must move once: keys + scales per group, logits, q, w, tables."""
    import workloads as W
    ctx = wl.context_lens.cpu().tolist()
    ind = None if wl.indices is None else wl.indices.cpu().tolist()
    per_tok = {W.KV_FP8: 132, W.KV_FP4: 76, W.KV_MXFP4: 68}[wl.kv_format]  # values + scales a token
    logit_b = 4 if wl.logits_dtype == W.LOGITS_F32 else 2
    # groups = runs of equal request ids, at most 8 rows
    key_bytes = 0
    bt_bytes = 0
    t = 0
    T = len(ctx)
    while t < T:
        u = t + 1
        while u < T and ind is not None and ind[u] == ind[t] and u - t < 8:
            u += 1
        lmax = max(max(ctx[t:u]), 0)
        key_bytes += lmax * per_tok
        bt_bytes += (lmax + 63) // 64 * 4
        t = u
    logits_bytes = sum(max(c, 0) for c in ctx) * logit_b
    q_bytes = T * 64 * 128 if wl.q_scale is None else T * 64 * (64 + 4)
    small = q_bytes + T * 64 * 4 + T * 4 * 2 + bt_bytes
    flops = 2 * 64 * 128 * sum(max(c, 0) for c in ctx)
    return key_bytes, logits_bytes, small, flops


def kernel_source_sha(kernel_file):
    """Hash of a kernel's source file and the headers it includes."""
    csrc = os.path.join(ROOT, "sparse_attention_indexer_paged_gb300", "csrc")
    h = hashlib.sha256()
    for f in (kernel_file, "ptx.cuh", "common.cuh"):
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def profile_traffic(kernel_file, summary_name):
    """dram bytes per launch from the committed ncu summary, if it matches the current source."""
    path = os.path.join(ROOT, "profiles", summary_name)
    try:
        text = open(path).read()
        sha = kernel_source_sha(kernel_file)
        m = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
        s = re.search(r"source_sha256_16:\s*([0-9a-f]+)", text)
        if m and s and s.group(1) == sha:
            return float(m.group(1))
    except OSError:
        pass
    return None


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        # raw samples (the JSON line carries their summary): DSA_CLOCKS_DIR, else the temp dir
        import tempfile
        out_dir = os.environ.get("DSA_CLOCKS_DIR", tempfile.gettempdir())
        self.path = os.path.join(out_dir, f"dsa_clocks_rank{gpu_index}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm.sort()
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def measure_fp8_peak(dev):
    """Dense e4m3 tensor throughput on this GPU, TFLOP/s: a cuBLASLt FP8 GEMM
    (torch._scaled_mm, 8192^3, bf16 out) timed as a burst after warm-up, the
    way the bf16 peak beside it was measured.  None if the GEMM is unavailable."""
    import torch
    try:
        n = 8192
        a = torch.randn(n, n, device=dev).to(torch.float8_e4m3fn)
        b = torch.randn(n, n, device=dev).to(torch.float8_e4m3fn).t()
        one = torch.tensor(1.0, device=dev)
        f = lambda: torch._scaled_mm(a, b, scale_a=one, scale_b=one, out_dtype=torch.bfloat16)  # noqa: E731
        for _ in range(5):
            f()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = 20
        e0.record()
        for _ in range(reps):
            f()
        e1.record()
        torch.cuda.synchronize()
        sec = e0.elapsed_time(e1) * 1e-3 / reps
        del a, b
        return round(2 * n ** 3 / sec / 1e12, 1)
    except Exception:
        return None


def fp8_peak_tflops(dev, bf16_tf):
    """(TFLOP/s, how it was obtained) of the dense FP8 tensor rate."""
    m = measure_fp8_peak(dev)
    if m is not None:
        return m, "measured in this run: cuBLASLt e4m3 GEMM 8192^3 (torch._scaled_mm), burst"
    return bf16_tf * FP8_PEAK_RATIO, f"bf16 peak x {FP8_PEAK_RATIO} (nominal fp8:bf16 ratio; the FP8 GEMM was unavailable)"


def tensor_peak(kv_format, fp8_tf, fp8_src, bf16_tf):
    """(TFLOP/s, how it was obtained) of the tensor rate the logits
    contraction runs at for this key format: FP8 keys (kind::f8f6f4) the FP8
    GEMM figure; FP4 keys (dequantised to f16 tiles, kind::f16) the measured
    bf16 GEMM (f16 and bf16 share a rate); MXFP4 (block-scaled kind::mxf4)
    the FP8 figure times the nominal fp4:fp8 ratio."""
    import workloads as W
    if kv_format == W.KV_FP4:
        return bf16_tf, "bf16 GEMM peak (MEASURED_PEAKS.json bf16_tflops): the FP4 kernel's MMAs are kind::f16"
    if kv_format == W.KV_MXFP4:
        return round(fp8_tf * FP4_PER_FP8, 1), f"FP8 peak x {FP4_PER_FP8} (nominal fp4:fp8 ratio; kind::mxf4 MMAs)"
    return fp8_tf, fp8_src


def measure_config(name, dev, K=200, KB=100, fp8_tf=None, fp8_src="", bf16_tf=None, hbm_gbs=None):
    """One decode workload timed as the headline is: the three-kernel step
    replayed from a CUDA graph (K replays), then a per-kernel event loop (KB
    steps); the logits kernel's achieved GB/s against the bytes it must move."""
    import torch
    import sparse_attention_indexer_paged_gb300 as dsa
    import workloads as W
    wl = W.config(name, device=dev)
    T, S = wl.num_rows, dsa.device_num_sms()
    sched = torch.empty(dsa.schedule_words(S, T), dtype=torch.int32, device=dev)
    ldt = torch.float32 if wl.logits_dtype == W.LOGITS_F32 else torch.bfloat16
    logits = torch.empty((T, wl.logits_stride), dtype=ldt, device=dev)
    idx = torch.empty((T, wl.topk), dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    gs = torch.cuda.Stream(device=dev)

    def run(ev=None):
        # the binding launches on the current stream: gs
        with torch.cuda.stream(gs):
            if ev is not None:
                ev[0].record(gs)
            dsa.paged_mqa_logits_metadata(wl.context_lens, wl.indices, S, out=sched, kv_format=wl.kv_format)
            if ev is not None:
                ev[1].record(gs)
            dsa.fp8_fp4_paged_mqa_logits(wl.q, wl.kv_cache, wl.weights, wl.context_lens, wl.block_table, sched,
                                         indices=wl.indices, kv_format=wl.kv_format, logits_dtype=wl.logits_dtype,
                                         logits_stride=wl.logits_stride, num_sms=S, status=status, out=logits,
                                         q_scale=wl.q_scale)
            if ev is not None:
                ev[2].record(gs)
            dsa.top_k_per_row(logits, None, wl.context_lens, wl.topk, out=idx, status=status)
            if ev is not None:
                ev[3].record(gs)

    gs.wait_stream(torch.cuda.current_stream(dev))
    for _ in range(3):
        run()
    gs.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=gs, capture_error_mode="relaxed"):
        run()
    with torch.cuda.stream(gs):
        for _ in range(5):
            g.replay()
        gs.synchronize()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(gs)
        for _ in range(K):
            g.replay()
        t1.record(gs)
    gs.synchronize()
    step_us = t0.elapsed_time(t1) * 1e3 / K
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(KB)]
    for i in range(KB):
        run(evs[i])
    gs.synchronize()
    kus = [sum(e[j].elapsed_time(e[j + 1]) for e in evs) * 1e3 / KB for j in range(3)]
    assert int(status.item()) == 0, dsa.status_string(int(status.item()))
    key_b, logit_b, small_b, flops = algorithmic_bytes(wl)
    alg = key_b + logit_b + small_b
    t_mem = alg / (hbm_gbs * 1e9)
    tc_tf, tc_src = tensor_peak(wl.kv_format, fp8_tf, fp8_src, bf16_tf)
    t_tc = flops / (tc_tf * 1e12)
    achieved = alg / (kus[1] * 1e-6) / 1e9
    res = {
        "workload": workload_desc(name, wl),
        "step_us": round(step_us, 3),
        "kernels_us": {"metadata": round(kus[0], 3), "logits": round(kus[1], 3), "top_k": round(kus[2], 3)},
        "logits_algorithmic_bytes": alg,
        "logits_achieved_gbs": round(achieved, 1),
        "logits_roofline_frac": round(achieved / hbm_gbs, 4),
        "logits_bound": "hbm" if t_mem >= t_tc else "tensor",
        "tensor_peak_tflops": tc_tf,
        "tensor_peak_source": tc_src,
        "tensor_frac": round(flops / (kus[1] * 1e-6) / 1e12 / tc_tf, 4),
        "bound_us": round(max(t_mem, t_tc) * 1e6, 2),
        "logits_frac_of_bound": round(max(t_mem, t_tc) / (kus[1] * 1e-6), 4),
        "step_roofline_frac": round(max(t_mem, t_tc) / (step_us * 1e-6), 4),
        "steps": K,
    }
    del wl, logits, idx, sched, g
    torch.cuda.empty_cache()
    return res


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def run_ours(args, rank, world, local):
    import torch
    import sparse_attention_indexer_paged_gb300 as dsa
    import workloads as W

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    dsa.build()
    L = dsa.lib()
    wl = W.config(args.workload, device=dev)          # per-rank replica (weak scaling)
    T = wl.num_rows
    S = dsa.device_num_sms()
    stream = torch.cuda.current_stream(dev)
    sp = ctypes.c_void_p(stream.cuda_stream)
    sched = torch.empty(dsa.schedule_words(S, T), dtype=torch.int32, device=dev)
    ldt = torch.float32 if wl.logits_dtype == 0 else torch.bfloat16
    logits = torch.empty((T, wl.logits_stride), dtype=ldt, device=dev)
    idx = torch.empty((T, wl.topk), dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    P = lambda t: ctypes.c_void_p(t.data_ptr()) if t is not None else None  # noqa: E731

    mx = wl.kv_format == W.KV_MXFP4
    logits_fn = L.dsa_mxfp4_paged_mqa_logits if mx else L.dsa_fp8_fp4_paged_mqa_logits

    def make_calls(q, w, ctx, ind, bt, out_idx, qs=None, strm=None):
        sp_ = sp if strm is None else strm
        meta = (P(ctx), P(ind), T, 64, S, wl.kv_format, P(sched), sp_)  # groups sized for the key format
        # MXFP4 keys: the MXFP4 entry point with the q scales; else the key format
        head = (P(q), P(qs), P(wl.kv_cache), wl.page_stride, wl.num_pages) if mx else \
               (P(q), P(wl.kv_cache), wl.page_stride, wl.num_pages, wl.kv_format)
        lg = head + (P(w), P(ctx), P(bt), bt.stride(0), P(ind), P(sched), S, P(logits), wl.logits_dtype,
                     wl.logits_stride, T, 64, 128, 64, P(status), sp_)
        tk = (P(logits), wl.logits_dtype, wl.logits_stride, None, P(ctx), T, wl.topk,
              P(out_idx), out_idx.stride(0), P(status), sp_)
        return meta, lg, tk

    meta, lg, tk = make_calls(wl.q, wl.weights, wl.context_lens, wl.indices, wl.block_table, idx, wl.q_scale)

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        r1 = L.dsa_paged_mqa_logits_metadata_for_keys(*meta)
        if ev is not None:
            ev[1].record(stream)
        r2 = logits_fn(*lg)
        if ev is not None:
            ev[2].record(stream)
        r3 = L.dsa_top_k_per_row(*tk)
        if ev is not None:
            ev[3].record(stream)
        return r1 | r2 | r3

    for _ in range(max(args.warmup, 3)):
        assert step() == 0
    torch.cuda.synchronize()
    assert int(status.item()) == 0, dsa.status_string(int(status.item()))

    K = args.steps
    # The step as a CUDA graph (metadata, logits and top-k captured once on a
    # stream of their own): how a serving loop runs a decode step.
    gstream = torch.cuda.Stream(device=dev)
    gsp = ctypes.c_void_p(gstream.cuda_stream)
    meta_g, lg_g, tk_g = meta[:-1] + (gsp,), lg[:-1] + (gsp,), tk[:-1] + (gsp,)

    def gstep():
        return L.dsa_paged_mqa_logits_metadata_for_keys(*meta_g) | logits_fn(*lg_g) | L.dsa_top_k_per_row(*tk_g)

    gstream.wait_stream(stream)
    with torch.cuda.stream(gstream):
        for _ in range(3):
            assert gstep() == 0
    gstream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=gstream, capture_error_mode="relaxed"):
        assert gstep() == 0
    with torch.cuda.stream(gstream):
        for _ in range(max(args.warmup, 3)):
            graph.replay()
    torch.cuda.synchronize()

    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    d0, d1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    # timed: K graph replays (the value), then K directly launched steps
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with torch.cuda.stream(gstream):
        t0.record(gstream)
        for _ in range(K):
            graph.replay()
        t1.record(gstream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    d0.record(stream)
    for _ in range(K):
        step()
    d1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop()
    assert int(status.item()) == 0, dsa.status_string(int(status.item()))
    ms_step = max_over_ranks(t0.elapsed_time(t1) / K, dev, world)
    direct_ms = max_over_ranks(d0.elapsed_time(d1) / K, dev, world)
    # per-kernel breakdown: a separate loop with events between the kernels
    KB = min(K, 500)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(KB)]
    for i in range(KB):
        step(evs[i])
    torch.cuda.synchronize()
    meta_ms = sum(e[0].elapsed_time(e[1]) for e in evs) / KB
    logit_ms = sum(e[1].elapsed_time(e[2]) for e in evs) / KB
    topk_ms = sum(e[2].elapsed_time(e[3]) for e in evs) / KB
    assert int(status.item()) == 0, dsa.status_string(int(status.item()))

    # ---- end to end through the C ABI from pinned host buffers.  Every step
    # copies its inputs host -> device and reads its result back; a serving
    # loop overlaps step i's kernels with step i+1's input copy and step
    # i-1's result copy, so device inputs and outputs are double buffered
    # and three streams are ordered by events.
    # A step's inputs travel as one copy: they sit at 256-byte-aligned offsets
    # of one pinned host buffer and of one device buffer per set.  The kernels
    # of each set run as a CUDA graph on a compute stream of their own.
    parts = [("q", wl.q), ("w", wl.weights), ("ctx", wl.context_lens), ("bt", wl.block_table)]
    if wl.indices is not None:
        parts.append(("ind", wl.indices))
    if wl.q_scale is not None:
        parts.append(("qs", wl.q_scale))
    layout, off = {}, 0
    for name, t in parts:
        layout[name] = (off, t)
        off = (off + t.numel() * t.element_size() + 255) // 256 * 256
    blob_bytes = off

    def blob_view(blob, name):
        o, t = layout[name]
        return blob[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape)

    hblob = torch.zeros(blob_bytes, dtype=torch.uint8).pin_memory()
    for name, t in parts:
        blob_view(hblob, name).copy_(t.cpu())
    hidx = [torch.empty((T, wl.topk), dtype=torch.int32).pin_memory() for _ in range(2)]
    s_in, s_out, s_cmp = (torch.cuda.Stream(device=dev) for _ in range(3))
    csp = ctypes.c_void_p(s_cmp.cuda_stream)
    sets = []
    for _ in range(2):
        dblob = torch.empty(blob_bytes, dtype=torch.uint8, device=dev)
        dv = {name: blob_view(dblob, name) for name, _ in parts}
        didx = torch.empty_like(idx)
        calls = make_calls(dv["q"], dv["w"], dv["ctx"], dv.get("ind"), dv["bt"], didx, dv.get("qs"), strm=csp)
        dblob.copy_(hblob)
        torch.cuda.synchronize()
        m, lgc, tkc = calls
        with torch.cuda.stream(s_cmp):
            assert (L.dsa_paged_mqa_logits_metadata_for_keys(*m) | logits_fn(*lgc) | L.dsa_top_k_per_row(*tkc)) == 0
        s_cmp.synchronize()
        graph_set = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph_set, stream=s_cmp, capture_error_mode="relaxed"):
            assert (L.dsa_paged_mqa_logits_metadata_for_keys(*m) | logits_fn(*lgc) | L.dsa_top_k_per_row(*tkc)) == 0
        sets.append(dict(dblob=dblob, didx=didx, graph=graph_set))
    h2d_bytes = blob_bytes
    d2h_bytes = hidx[0].numel() * hidx[0].element_size()
    ev_ready = [torch.cuda.Event() for _ in range(2)]     # inputs of the set copied in
    ev_done = [torch.cuda.Event() for _ in range(2)]      # kernels of the set finished
    ev_out = [torch.cuda.Event() for _ in range(2)]       # result of the set copied out
    for e in ev_done + ev_out:
        e.record(stream)

    def e2e_step(i):
        st = sets[i % 2]
        s_in.wait_event(ev_done[i % 2])       # the kernels that read this set are done
        with torch.cuda.stream(s_in):
            st["dblob"].copy_(hblob, non_blocking=True)
        ev_ready[i % 2].record(s_in)
        s_cmp.wait_event(ev_ready[i % 2])
        s_cmp.wait_event(ev_out[i % 2])       # its previous result was copied out
        with torch.cuda.stream(s_cmp):
            st["graph"].replay()
        ev_done[i % 2].record(s_cmp)
        s_out.wait_event(ev_done[i % 2])
        with torch.cuda.stream(s_out):
            hidx[i % 2].copy_(st["didx"], non_blocking=True)
        ev_out[i % 2].record(s_out)
        return 0

    for i in range(4):
        assert e2e_step(i) == 0
    torch.cuda.synchronize()
    assert torch.equal(hidx[0], idx.cpu()) and torch.equal(hidx[1], idx.cpu()), \
        "e2e result differs from the device-resident run"
    KE = args.e2e_steps
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    for i in range(KE):
        e2e_step(i)
    e1.record(s_out)   # after the last result copy, which follows the last step's kernels
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / KE, dev, world)
    # the same step with nothing overlapped (copy in, kernels, copy out, all
    # on one stream): the per-step latency a single request stream sees
    st0 = sets[0]

    def serial_step():
        with torch.cuda.stream(s_cmp):
            st0["dblob"].copy_(hblob, non_blocking=True)
            st0["graph"].replay()
            hidx[0].copy_(st0["didx"], non_blocking=True)
        return 0

    for _ in range(3):
        assert serial_step() == 0
    torch.cuda.synchronize()
    e0.record(s_cmp)
    for _ in range(KE):
        serial_step()
    e1.record(s_cmp)
    torch.cuda.synchronize()
    e2e_serial_ms = max_over_ranks(e0.elapsed_time(e1) / KE, dev, world)

    # ---- roofline of the dominant kernel (logits)
    hbm_gbs, bf16_tf, peak_src = peaks()
    key_b, logit_b, small_b, flops = algorithmic_bytes(wl)
    alg_bytes = key_b + logit_b + small_b
    achieved = alg_bytes / (logit_ms * 1e-3) / 1e9
    fp8_tf, fp8_src = fp8_peak_tflops(dev, bf16_tf)
    tc_tf, tc_src = tensor_peak(wl.kv_format, fp8_tf, fp8_src, bf16_tf)
    t_mem = alg_bytes / (hbm_gbs * 1e9)
    t_tc = flops / (tc_tf * 1e12)
    traffic = profile_traffic("logits.cu", f"logits_{args.workload}_ncu.md")
    step_bytes = alg_bytes + logit_b + T * wl.topk * 4   # + top-k re-read of logits and index write
    result = {
        "metric": METRIC,
        "value": round(ms_step * 1e3, 3),
        "unit": "us/step",
        "n_gpus": world,
        "steps": K,
        "warmup": max(args.warmup, 3),  # warm-ups actually run
        "ms_per_step": round(ms_step, 6),
        "higher_is_better": False,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": ["fp8_e4m3", "fp4_e2m1+fp8_e4m3", "mxfp4_e2m1+ue8m0"][wl.kv_format],
        "data": "synthetic (seeded workloads.config; no dataset or weights)",
        "config": {
            "workload": workload_desc(args.workload, wl),
            "seed": wl.seed,
            "rows": T,
            "global_batch": len(wl.request_lens) * world,
            "seq_len": max(wl.request_lens),
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
            "l2": "inputs larger than L2: key pool %.0f MB resident in HBM vs 129 MB L2; no flush"
                  % (wl.kv_cache.numel() / 1e6),
            "num_sms": S,
        },
        "kernels_us": {"metadata": round(meta_ms * 1e3, 3), "logits": round(logit_ms * 1e3, 3),
                       "top_k": round(topk_ms * 1e3, 3)},
        "hbm_gbs": round(step_bytes / (ms_step * 1e-3) / 1e9, 1),
        "roofline": {
            "kernel": "logits",
            "bound": "hbm" if t_mem >= t_tc else "tensor",
            "achieved": round(achieved, 1),
            "peak": hbm_gbs,
            "unit": "GB/s",
            "frac": round(achieved / hbm_gbs, 4),
            "traffic": traffic,
            "algorithmic_bytes": alg_bytes,
            "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)" if peak_src == "measured"
                           else "fallback 6.8 TB/s",
            "tensor_frac_of_fp8_peak": round(flops / (logit_ms * 1e-3) / 1e12 / fp8_tf, 4),
            "fp8_peak_tflops": fp8_tf,
            "fp8_peak_source": fp8_src,
            "tensor_peak_tflops": tc_tf,
            "tensor_peak_source": tc_src,
            "tensor_frac": round(flops / (logit_ms * 1e-3) / 1e12 / tc_tf, 4),
            "bound_us": round(max(t_mem, t_tc) * 1e6, 2),
            "step_roofline_frac": round(max(t_mem, t_tc) / (ms_step * 1e-3), 4),
        },
        "e2e": {"value": round(e2e_ms * 1e3, 3), "unit": "us/step",
                "h2d_bytes_per_step": h2d_bytes, "d2h_bytes_per_step": d2h_bytes, "serialized_value": round(e2e_serial_ms * 1e3, 3), "pipelining": "step i kernels overlap step i+1 input copy and step i-1 result copy; a step's inputs are one copy from a pinned staging buffer and its kernels one CUDA graph replay"},
        "launch": "value: the step (metadata, logits, top-k) captured once as a CUDA graph and "
                  "replayed K times; direct_launch_value: the same K steps launched one call at a time",
        "direct_launch_value": round(direct_ms * 1e3, 3),
        "gpu_launches": 6 * K,
        "clocks": clk,
        "context": PAGES_CONTEXT,
    }
    if rank == 0 and not args.no_per_config:
        # the other decode configurations, each timed the same way (graph
        # replays, per-kernel events) with its own roofline
        others = [c for c in ("plain", "mtp", "varlen", "fp4_varlen", "mxfp4_varlen") if c != args.workload]
        result["per_config"] = {c: measure_config(c, dev, fp8_tf=fp8_tf, fp8_src=fp8_src, bf16_tf=bf16_tf,
                                                  hbm_gbs=hbm_gbs) for c in others}
    if rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(wl.to("cpu"), args.cpu_budget_s)
    if world > 1:
        torch.distributed.destroy_process_group()
    return result


# ---------------------------------------------------------------------------
# decode context parallelism, the ranks emulated in turn on one GPU
# ---------------------------------------------------------------------------

def run_dcp(args, local):
    import torch
    import sparse_attention_indexer_paged_gb300 as dsa
    import workloads as W

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dsa.build()
    L = dsa.lib()
    R, inter = args.dcp_world, args.dcp_interleave
    base = W.config(args.workload)
    shards = [W.dcp_shard(base, r, R, inter).to(dev) for r in range(R)]
    glob = base.to(dev)
    T, k, S = glob.num_rows, glob.topk, dsa.device_num_sms()
    stream = torch.cuda.current_stream(dev)
    sp = ctypes.c_void_p(stream.cuda_stream)
    P = lambda t: ctypes.c_void_p(t.data_ptr()) if t is not None else None  # noqa: E731
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    ldt = torch.float32 if glob.logits_dtype == 0 else torch.bfloat16

    def calls(wl, r):
        sched = torch.empty(dsa.schedule_words(S, T), dtype=torch.int32, device=dev)
        logits = torch.empty((T, wl.logits_stride), dtype=ldt, device=dev)
        idx = torch.empty((T, k), dtype=torch.int32, device=dev)
        packed = torch.empty((T, k, 2), dtype=torch.float32, device=dev)
        meta = (P(wl.context_lens), P(wl.indices), T, 64, S, wl.kv_format, P(sched), sp)
        lg = (P(wl.q), P(wl.kv_cache), wl.page_stride, wl.num_pages, wl.kv_format, P(wl.weights),
              P(wl.context_lens), P(wl.block_table), wl.block_table.stride(0), P(wl.indices), P(sched), S,
              P(logits), wl.logits_dtype, wl.logits_stride, T, 64, 128, 64, P(status), sp)
        tk = (P(logits), wl.logits_dtype, wl.logits_stride, None, P(wl.context_lens), T, k, P(idx),
              idx.stride(0), P(status), sp)
        pk = (P(logits), wl.logits_dtype, wl.logits_stride, P(idx), idx.stride(0), T, k, r, R, inter,
              P(packed), sp)
        return dict(keep=(sched, logits, idx), packed=packed, meta=meta, lg=lg, tk=tk, pk=pk)

    ranks = [calls(sh, r) for r, sh in enumerate(shards)]
    gathered = torch.empty((R, T, k, 2), dtype=torch.float32, device=dev)
    merged = torch.empty((T, k), dtype=torch.int32, device=dev)
    mg = (P(gathered), R, T, k, P(merged), merged.stride(0), sp)
    ref = calls(glob, 0)

    def step(ev=None):
        rc = 0
        for r, c in enumerate(ranks):
            if ev is not None:
                ev[r][0].record(stream)
            rc |= L.dsa_paged_mqa_logits_metadata_for_keys(*c["meta"])
            if ev is not None:
                ev[r][1].record(stream)
            rc |= L.dsa_fp8_fp4_paged_mqa_logits(*c["lg"])
            if ev is not None:
                ev[r][2].record(stream)
            rc |= L.dsa_top_k_per_row(*c["tk"])
            if ev is not None:
                ev[r][3].record(stream)
            rc |= L.dsa_dcp_pack_topk(*c["pk"])
            if ev is not None:
                ev[r][4].record(stream)
        for r, c in enumerate(ranks):      # where R GPUs would all-gather
            gathered[r].copy_(c["packed"])
        if ev is not None:
            ev[R][0].record(stream)
        rc |= L.dsa_dcp_merge_topk(*mg)
        if ev is not None:
            ev[R][1].record(stream)
        return rc

    # the unsharded step, for the exactness check
    assert (L.dsa_paged_mqa_logits_metadata_for_keys(*ref["meta"]) | L.dsa_fp8_fp4_paged_mqa_logits(*ref["lg"])
            | L.dsa_top_k_per_row(*ref["tk"])) == 0
    for _ in range(max(args.warmup, 3)):
        assert step() == 0
    torch.cuda.synchronize()
    assert int(status.item()) == 0, dsa.status_string(int(status.item()))
    exact = bool(torch.equal(merged, ref["keep"][2]))

    K = args.steps
    evs = [[[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(R + 1)] for _ in range(K)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    torch.cuda.synchronize()
    t0.record(stream)
    for i in range(K):
        step(evs[i])
    t1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    assert int(status.item()) == 0, dsa.status_string(int(status.item()))

    def avg(r, a, b):
        return sum(e[r][a].elapsed_time(e[r][b]) for e in evs) / K * 1e3

    per_rank = [dict(metadata=round(avg(r, 0, 1), 3), logits=round(avg(r, 1, 2), 3),
                     top_k=round(avg(r, 2, 3), 3), pack=round(avg(r, 3, 4), 3), step=round(avg(r, 0, 4), 3))
                for r in range(R)]
    merge_us = avg(R, 0, 1)
    crit = max(x["step"] for x in per_rank) + merge_us
    hbm_gbs, _, peak_src = peaks()
    merge_bytes = R * T * k * 8 + T * k * 4
    merge_gbs = merge_bytes / (merge_us * 1e-6) / 1e9
    return {
        "metric": "indexer DCP decode µs/step on the critical path (slowest rank's step + merge; "
                  "the all-gather not timed: one GPU)",
        "value": round(crit, 3),
        "unit": "us/step",
        "higher_is_better": False,
        "n_gpus": 1,
        "steps": K,
        "warmup": max(args.warmup, 3),  # warm-ups actually run
        "dtype": "e4m3 x e4m3 -> f32" if glob.kv_format == 0 else "e4m3 x e2m1 -> f32",
        "data": "synthetic",
        "config": {"workload": f"{args.workload} split over {R} DCP ranks (interleave {inter})",
                   "shape": workload_desc(args.workload, base), "rows": T, "num_sms": S,
                   "emulation": "ranks run in turn on one GPU; packs stacked by device copies"},
        "exact_vs_unsharded": exact,
        "kernels_us": {"per_rank": per_rank, "merge": round(merge_us, 3)},
        "all_ranks_serial_us": round(t0.elapsed_time(t1) / K * 1e3, 3),
        "merge_roofline": {"bound": "hbm", "algorithmic_bytes": merge_bytes, "achieved": round(merge_gbs, 1),
                           "peak": hbm_gbs, "unit": "GB/s", "frac": round(merge_gbs / hbm_gbs, 4),
                           "peak_source": peak_src},
        "gpu_launches": (4 * R + 1) * K,
        "clocks": clk,
    }


# ---------------------------------------------------------------------------
# prefill over the paged cache
# ---------------------------------------------------------------------------

def run_prefill(args, local):
    import torch
    import sparse_attention_indexer_paged_gb300 as dsa
    import workloads as W

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dsa.build()
    L = dsa.lib()
    wl = W.config(args.workload)
    pf = W.prefill_view(wl).to(dev)
    T, B, k, S = pf.num_rows, pf.num_requests, pf.topk, dsa.device_num_sms()
    stream = torch.cuda.current_stream(dev)
    sp = ctypes.c_void_p(stream.cuda_stream)
    P = lambda t: ctypes.c_void_p(t.data_ptr()) if t is not None else None  # noqa: E731
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    ctx = torch.empty(T, dtype=torch.int32, device=dev)
    req = torch.empty(T, dtype=torch.int32, device=dev)
    sched = torch.empty(dsa.schedule_words(S, T), dtype=torch.int32, device=dev)
    ldt = torch.float32 if pf.logits_dtype == 0 else torch.bfloat16
    logits = torch.empty((T, pf.logits_stride), dtype=ldt, device=dev)
    idx = torch.empty((T, k), dtype=torch.int32, device=dev)
    rows_a = (P(pf.cu_seqlen_ks), P(pf.cu_seqlen_ke), T, P(pf.local_cu_seq_lens), B, P(ctx), P(req), P(status), sp)
    meta_a = (P(ctx), P(req), T, 64, S, pf.kv_format, P(sched), sp)
    lg_a = (P(pf.q), P(pf.q_scale), P(pf.kv_cache), pf.page_stride, int(pf.kv_cache.shape[0]), pf.kv_format, P(pf.weights),
            P(ctx), P(req), P(pf.block_table), pf.block_table.stride(0), B, P(sched), S, P(logits),
            pf.logits_dtype, pf.logits_stride, T, 64, 128, 64, P(status), sp)
    tk_a = (P(logits), pf.logits_dtype, pf.logits_stride, None, P(ctx), T, k, P(idx), idx.stride(0), P(status), sp)

    def step(ev=None):
        rc = 0
        calls = ((L.dsa_prefill_rows, rows_a), (L.dsa_paged_mqa_logits_metadata_for_keys, meta_a),
                 (L.dsa_prefill_mqa_logits, lg_a), (L.dsa_top_k_per_row, tk_a))
        for i, (fn, a) in enumerate(calls):
            if ev is not None:
                ev[i].record(stream)
            rc |= fn(*a)
        if ev is not None:
            ev[4].record(stream)
        return rc

    for _ in range(max(args.warmup, 3)):
        assert step() == 0
    torch.cuda.synchronize()
    assert int(status.item()) == 0, dsa.status_string(int(status.item()))
    K = args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(K)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    torch.cuda.synchronize()
    t0.record(stream)
    for i in range(K):
        step(evs[i])
    t1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    assert int(status.item()) == 0, dsa.status_string(int(status.item()))
    ms = t0.elapsed_time(t1) / K
    names = ("prefill_rows", "metadata", "logits", "top_k")
    us = {n: sum(e[i].elapsed_time(e[i + 1]) for e in evs) / K * 1e3 for i, n in enumerate(names)}
    hbm_gbs, bf16_tf, peak_src = peaks()
    fp8_tf, fp8_src = fp8_peak_tflops(dev, bf16_tf)
    lens = ctx.cpu().to(torch.int64)
    flops = int(lens.sum()) * 64 * 128 * 2
    achieved = flops / (us["logits"] * 1e-6) / 1e12
    return {
        "metric": "indexer prefill µs/step over the paged cache (rows, schedule, logits, top-k)",
        "value": round(ms * 1e3, 3),
        "unit": "us/step",
        "higher_is_better": False,
        "n_gpus": 1,
        "steps": K,
        "warmup": max(args.warmup, 3),  # warm-ups actually run
        "dtype": "e4m3 x e4m3 -> f32" if pf.kv_format == 0 else "e4m3 x e2m1 -> f32",
        "data": "synthetic",
        "config": {"workload": "prefill: 2 requests x 8192-token prompts, their last 4096 tokens as rows "
                               "(T=8192, causal lengths 4097..8192), q and keys e4m3, H=64, D=128, "
                               "top-k 2048, fp32 logits", "rows": T, "num_sms": S},
        "kernels_us": {n: round(v, 3) for n, v in us.items()},
        "roofline": {"kernel": "logits", "bound": "tensor", "achieved": round(achieved, 1),
                     "peak": fp8_tf, "unit": "TFLOP/s", "frac": round(achieved / fp8_tf, 4),
                     "flops": flops, "traffic": profile_traffic("logits.cu", "logits_prefill_ncu.md"),
                     "peak_source": fp8_src},
        "gpu_launches": 4 * K,
        "clocks": clk,
    }


# ---------------------------------------------------------------------------
# the step in row slices under a logits budget
# ---------------------------------------------------------------------------

def run_chunked(args, local):
    import torch
    import sparse_attention_indexer_paged_gb300 as dsa
    import workloads as W

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dsa.build()
    L = dsa.lib()
    wl = W.config(args.workload, device=dev)
    T, k, S = wl.num_rows, wl.topk, dsa.device_num_sms()
    stream = torch.cuda.current_stream(dev)
    sp = ctypes.c_void_p(stream.cuda_stream)
    P = lambda t: ctypes.c_void_p(t.data_ptr()) if t is not None else None  # noqa: E731
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    eb = 4 if wl.logits_dtype == 0 else 2

    def plan(budget):
        sb, sw = dsa.indexer_decode_scratch(T, wl.logits_dtype, wl.logits_stride, budget, S)
        scr = torch.empty(sb, dtype=torch.uint8, device=dev)
        sched = torch.empty(sw, dtype=torch.int32, device=dev)
        out = torch.empty((T, k), dtype=torch.int32, device=dev)
        a = (P(wl.q), P(wl.q_scale), P(wl.kv_cache), wl.page_stride, wl.num_pages, wl.kv_format, P(wl.weights),
             P(wl.context_lens), P(wl.block_table), wl.block_table.stride(0), P(wl.indices), T, 64, 128, 64,
             S, wl.logits_dtype, wl.logits_stride, budget, P(scr), sb, P(sched), sw, k, P(out), out.stride(0),
             P(status), sp)
        return dict(args=a, keep=(scr, sched), out=out, scratch_bytes=sb)

    runs = {"sliced": plan(args.logits_budget), "one_pass": plan(0)}
    res = {}
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    for name, r in runs.items():
        for _ in range(max(args.warmup, 3)):
            assert L.dsa_indexer_decode_topk(*r["args"]) == 0
        torch.cuda.synchronize()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for _ in range(args.steps):
            L.dsa_indexer_decode_topk(*r["args"])
        t1.record(stream)
        torch.cuda.synchronize()
        res[name] = t0.elapsed_time(t1) / args.steps * 1e3
    clk = clocks.stop()
    assert int(status.item()) == 0, dsa.status_string(int(status.item()))
    same = bool(torch.equal(runs["sliced"]["out"], runs["one_pass"]["out"]))
    ranges = dsa.decode_chunk_ranges(T, wl.logits_stride * eb // 2, args.logits_budget)
    return {
        "metric": "indexer decode µs/step as one native call, rows in slices under a logits budget",
        "value": round(res["sliced"], 3),
        "unit": "us/step",
        "higher_is_better": False,
        "n_gpus": 1,
        "steps": args.steps,
        "warmup": max(args.warmup, 3),  # warm-ups actually run
        "dtype": "e4m3 x e4m3 -> f32" if wl.kv_format == 0 else "e4m3 x e2m1 -> f32",
        "data": "synthetic",
        "config": {"workload": args.workload, "shape": workload_desc(args.workload, wl), "rows": T,
                   "logits_budget_bytes": args.logits_budget, "slices": ranges or [[0, T]],
                   "scratch_bytes": runs["sliced"]["scratch_bytes"],
                   "one_pass_scratch_bytes": runs["one_pass"]["scratch_bytes"], "num_sms": S},
        "one_pass_us": round(res["one_pass"], 3),
        "same_topk_as_one_pass": same,
        "gpu_launches": 3 * max(1, len(ranges)) * args.steps,
        "clocks": clk,
    }


# ---------------------------------------------------------------------------
# the oracle timed on the host cores
# ---------------------------------------------------------------------------

def _oracle_sample(wl, rows, cols):
    """Oracle logits (no bound) + top-k of `rows` restricted to the first `cols` columns."""
    import numpy as np
    import oracle
    ctx = wl.context_lens.clone()
    ctx[rows] = torch_min(ctx[rows], cols)
    t0 = time.perf_counter()
    lg, _ = oracle.paged_mqa_logits(wl.q, wl.kv_cache, wl.page_stride, wl.kv_format, wl.weights,
                                    ctx, wl.block_table, int(max(cols, 1)),
                                    rows=np.array(rows, dtype=np.int32), with_bound=False,
                                    q_scale=wl.q_scale)
    oracle.top_k_per_row(lg, ctx.numpy()[rows], wl.topk)
    return time.perf_counter() - t0, int(sum(int(ctx[r]) for r in rows))


def torch_min(x, c):
    import torch
    return torch.clamp(x, max=int(c))


def cpu_baseline(wl, budget_s):
    """Time the oracle on a bounded sample of rows, scaled to one full step."""
    total_cols = int(sum(max(int(c), 0) for c in wl.context_lens))
    T = wl.num_rows
    t1, c1 = _oracle_sample(wl, [0], int(wl.context_lens[0]))
    per_col = t1 / max(c1, 1)
    n = max(1, min(T, int(budget_s / max(t1, 1e-6))))
    rows = sorted(set(int(round(i * (T - 1) / max(n - 1, 1))) for i in range(n)))
    ts, cs = _oracle_sample(wl, rows, max(int(wl.context_lens.max()), 1))
    per_col = ts / max(cs, 1)
    us_step = per_col * total_cols * 1e6
    return {"value": round(us_step, 1), "unit": "us/step", "cores": os.cpu_count(),
            "kind": "oracle",
            "sample": f"{len(rows)} of {T} rows, all their columns ({cs} of {total_cols} "
                      f"row-columns): fp64 logits + stable top-k, scaled by row-columns"}


def run_reference(args, rank, world):
    """--impl reference: the CPU oracle as it stands, timed over whole steps.

    Each step is the oracle's fp64 logits and stable top-k of every row over
    all its columns.  When the requested steps would not finish within a few
    minutes, every step (warm-up and timed) runs the same evenly spaced subset
    of rows instead, the value is scaled by row-columns, and the line says so.
    """
    if rank != 0:
        return None
    import workloads as W
    wl = W.config(args.workload)
    total_cols = int(sum(max(int(c), 0) for c in wl.context_lens))
    T = wl.num_rows
    budget_s = 180.0
    probe_rows = list(range(0, T, max(1, T // 16)))[:16]
    t_probe, c_probe = _oracle_sample(wl, probe_rows, max(int(wl.context_lens.max()), 1))
    est_full = t_probe / max(c_probe, 1) * total_cols
    n_steps = args.steps + args.warmup
    if n_steps * est_full <= budget_s:
        rows = list(range(T))
    else:
        n = max(8, min(T, int(T * budget_s / (n_steps * est_full))))
        rows = sorted(set(int(round(i * (T - 1) / max(n - 1, 1))) for i in range(n)))
    cols = max(int(wl.context_lens.max()), 1)
    for _ in range(args.warmup):
        _oracle_sample(wl, rows, cols)
    spent, done = 0.0, 0
    for _ in range(args.steps):
        dt, c = _oracle_sample(wl, rows, cols)
        spent += dt
        done += c
    us_step = spent / max(done, 1) * total_cols * 1e6
    if len(rows) == T:
        sample = (f"every step is a whole step: oracle fp64 logits + stable top-k of all {T} rows over all "
                  f"their columns ({total_cols} row-columns); {args.warmup} warm-up and {args.steps} timed steps")
    else:
        sample = (f"every step runs the same {len(rows)} of {T} rows over all their columns ({done // max(args.steps, 1)} "
                  f"of {total_cols} row-columns), scaled to a whole step by row-columns, so that "
                  f"{args.warmup} + {args.steps} steps fit about {budget_s:.0f} s")
    return {"impl": "reference", "metric": METRIC, "value": round(us_step, 1), "unit": "us/step",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(us_step / 1e3, 3), "higher_is_better": False, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded workloads.config)",
            "config": {"workload": workload_desc(args.workload, wl), "seed": wl.seed},
            "timed_s": round(spent, 2),
            "cpu_baseline": {"value": round(us_step, 1), "unit": "us/step",
                             "cores": os.cpu_count(), "kind": "oracle", "sample": sample},
            "e2e": {"value": round(us_step, 1), "unit": "us/step", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    args = parse()
    rank, world, local = dist_env()
    if args.impl == "reference":
        res = run_reference(args, rank, world)
    elif args.workload == "prefill":
        assert world == 1, "the prefill bench runs in one process"
        res = run_prefill(args, local)
    elif args.logits_budget > 0:
        assert world == 1, "the sliced step runs in one process"
        res = run_chunked(args, local)
    elif args.dcp_world > 0:
        assert world == 1, "the DCP emulation runs in one process"
        res = run_dcp(args, local)
    else:
        res = run_ours(args, rank, world, local)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
