"""Benchmark: SageAttention-style quantized attention on one GB300 per rank.

One step = one pass of the whole hot path on device-resident BF16 inputs:
the quantization prologue (one persistent kernel, after a memset of its
work counters) and the tcgen05 attention kernel, through the library's C ABI
(``sage_sageattn``). The workload is the
video-diffusion-sized self-attention B=1, H=28, S=16384, D=128 with smooth_k
on (synthetic, seeded; Q/K ~ N(0, 1.5^2) with 1% of entries x8, V ~ N(0, 1)).

Printed metric: attention TOPS = 4*B*H*S^2*D / step time (whole step,
prologue included). The JSON line also carries the attention kernel alone
(``attention_kernel``) and the prologue's HBM bandwidth (``prologue``), each
against the measured peaks, the CPU oracle's throughput on a bounded sample
(``cpu_baseline``) and the end-to-end rate with host buffers (``e2e``).

``--impl reference`` times the CPU oracle (the only reference this method
has) on a bounded sample of the same workload.
"""

from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "B1_H28_S16384"
METRIC = "attention TOPS at B1 H28 S16k D128 (frac of INT8/FP8 peak); prologue HBM GB/s"


def bench_config(world=1, strong=False):
    """The workload named in both arms' JSON lines."""
    par = (f"heads split over {world} ranks (strong scaling, no exchange)" if strong
           else f"replicas x{world} (heads are independent)")
    return {"workload": WORKLOAD, "B": 1, "H": 28, "S": 16384, "D": 128, "smooth_k": True, "layout": "NHD",
            "l2": "step inputs (3 x 117 MB) larger than L2; per-kernel and per-config times with a 2xL2 scrub "
                  "written before each rep",
            "parallelism": par}


# DRAM traffic of one attention launch at this workload (dram__bytes_read.sum +
# dram__bytes_write.sum from one ncu capture of the kernel), with the SHA-256
# prefix of the kernel's source file the capture was taken on: reported only
# while the source still matches.
ATTN_TRAFFIC = {"bytes": 293839872 + 94373888, "source_sha256": "971d9f9a64063f6d"}
PROLOGUE_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def attention_traffic():
    """The recorded per-launch DRAM traffic of the attention kernel, or None
    once its source differs from the one the counters were taken on."""
    import hashlib

    path = os.path.join(ROOT, "quantized_attention_fp64_gb300", "csrc", "attention_tc.cu")
    with open(path, "rb") as f:
        digest = hashlib.sha256(f.read()).hexdigest()
    return ATTN_TRAFFIC["bytes"] if digest.startswith(ATTN_TRAFFIC["source_sha256"]) else None


def prologue_bytes(B, H, S, D):
    """Algorithmic prologue bytes: bf16 Q, K, V read once; int8 Q/K and e4m3 V
    codes, the scales and the key mean written once."""
    s_pad = -(-S // 128) * 128
    return 6 * B * S * H * D + 3 * B * H * s_pad * D + 2 * 4 * B * H * (s_pad // 32) + 2 * 4 * B * H * D


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    return dict(PROLOGUE_FALLBACK), "fallback"


def attention_peak(peaks):
    """Dense peak of the attention kernel's two contractions: QK^T runs as
    fp16 x fp16 (same rate as bf16), PV as e4m3 (2x the bf16 rate); they do
    equal work, so the combined peak is their harmonic mean."""
    p16 = peaks["bf16_tflops"]
    p8 = 2.0 * p16
    return 2.0 / (1.0 / p16 + 1.0 / p8), p16, p8


def dist_setup(n_gpus):
    from quantized_attention_fp64_gb300 import dist

    return dist.setup()


def barrier(world):
    from quantized_attention_fp64_gb300 import dist

    dist.barrier(world)


def max_over_ranks(x, world):
    from quantized_attention_fp64_gb300 import dist

    return dist.max_over_ranks(x, world)


class ClockSampler:
    """nvidia-smi samples of the SM clock and throttle reasons during timing."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        try:
            with open(self.path) as f:
                for line in f:
                    parts = [p.strip() for p in line.split(",")]
                    if len(parts) < 9:
                        continue
                    try:
                        sm.append(float(parts[1]))
                        mx.append(float(parts[2]))
                    except ValueError:
                        continue
                    for n, v in zip(names, parts[5:9]):
                        if v.lower() == "active":
                            reasons.add(n)
            os.unlink(self.path)
        except OSError:
            pass
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        sm.sort()
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": max(mx), "reasons": sorted(reasons), "samples": len(sm)}


def cpu_oracle_sample(rows=1024, seed=3, heads=1):
    """Times the oracle (as it stands) on a bounded sample of the workload:
    for each of ``heads`` heads, the full prologue of that head plus the
    emulated attention of ``rows`` of its query rows against all 16384 keys.
    The step time is extrapolated to all 28 heads (the prologue's share scales
    with heads, the attention's with query rows). Returns attention-op
    throughput in TOPS and a description."""
    import numpy as np

    from oracle import attention_emulated, e4m3_decode, quantize_head
    from quantized_attention_fp64_gb300.workloads import WORKLOADS, make_qkv

    w = WORKLOADS[WORKLOAD]
    q, k, v = make_qkv(w, "cpu")
    t_pro = t_att = 0.0
    for h in range(heads):
        qh, kh, vh = (t[0, :, h, :].float().numpy() for t in (q, k, v))
        sel = np.arange(w.S) if rows >= w.S else np.sort(
            np.random.default_rng(seed + h).choice(w.S, rows, replace=False))
        t0 = time.perf_counter()
        r = quantize_head(qh, kh, vh, True)
        t1 = time.perf_counter()
        attention_emulated(r["q_codes"], r["k_codes"], e4m3_decode(r["v_codes"]), r["q_scale"], r["k_scale"],
                           r["v_scale"], 1.0 / math.sqrt(128.0), rows=sel)
        t2 = time.perf_counter()
        t_pro += t1 - t0
        t_att += t2 - t1
    n_rows = min(rows, w.S)
    head_time = (t_pro + t_att * (w.S / n_rows)) / heads   # one full head of one step
    value = 4.0 * w.S * w.S * 128 / head_time / 1e12
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    return {
        "value": value, "unit": "TOPS", "cores": cores, "kind": "oracle",
        "sample": f"{heads} head(s) of {WORKLOAD}: full prologue ({t_pro:.2f} s) + emulated attention of "
                  f"{n_rows} query rows x {w.S} keys per head ({t_att:.2f} s), extrapolated to the step's "
                  f"{w.H} heads x {w.S} rows; numpy, BLAS threads up to {cores}",
        "attention_ops_sampled": 4.0 * heads * n_rows * w.S * 128, "seconds": t_pro + t_att,
    }


def cold_time(torch, fn, scrub, reps=7):
    """Median device time of one call of fn with L2 cold: fn is captured in
    a one-call CUDA graph; before each rep a buffer of twice the L2 size is
    written (untimed), then CUDA events on the launching stream bracket the
    graph replay. The scrub keeps the GPU busy while the host enqueues the
    events and the replay, so no host time falls between them."""
    import statistics

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            fn()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    times = []
    for r in range(reps):
        scrub.fill_(r & 0xFF)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        g.replay()
        b.record(stream)
        b.synchronize()
        times.append(a.elapsed_time(b) / 1e3)
    return statistics.median(times)


# The configurations the pages' workloads are stood in for by (the five
# synthetic shapes, config 2 with smooth_k on and off) and the 80-head case
# past 2^31 bytes per tensor: (workload, smooth_k, oracle heads, oracle rows).
CONFIGS = [("B1_H2_S256", False, 2, 256), ("B2_H8_S1024", True, 4, 256), ("B2_H8_S1024", False, 4, 256),
           ("B1_H28_S4096", True, 3, 256), ("B1_H28_S16384", True, 3, 256), ("B1_H28_S131072", True, 1, 128),
           ("B1_H80_S131072", True, 1, 128)]


def config_rows(torch, peaks, scrub, sm):
    """Per configuration: the prologue (sage_quantize) and the attention
    kernel timed with L2 cold, against the measured peaks; the accuracy of
    sampled rows of sampled heads against the oracle (its emulation of the
    quantized method and exact fp64 attention); and the oracle's own time on
    that sample, extrapolated to the whole configuration."""
    import numpy as np

    from oracle.tensors import attention_from_codes, exact_head, quantize_tensors
    from quantized_attention_fp64_gb300 import sageattn
    from quantized_attention_fp64_gb300.api import alloc_bundle, attention, quantize
    from quantized_attention_fp64_gb300.workloads import WORKLOADS, make_qkv

    p_att = attention_peak(peaks)[0]
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    rows_out = []
    for name, smooth, n_heads, n_rows in CONFIGS:
        w = WORKLOADS[name]
        B, H, S = w.B, w.H, w.S
        q, k, v = make_qkv(w, "cuda")
        qz = alloc_bundle(B, S, H, q.device)
        out = torch.empty_like(q)
        t_pro = cold_time(torch, lambda: quantize(q, k, v, "NHD", smooth, out=qz), scrub)
        t_att = cold_time(torch, lambda: attention(qz, sm, out=out), scrub)
        o = sageattn(q, k, v, sm_scale=sm, smooth_k=smooth)
        torch.cuda.synchronize()
        pb = prologue_bytes(B, H, S, 128)
        ops = float(w.attention_ops)
        # sampled heads (first, middle, last) and rows (seeded), as host arrays
        heads = sorted({(bb, hh) for bb, hh in [(0, 0), (B - 1, H - 1), (B // 2, H // 2), (0, H // 3)]})[:n_heads]
        rows = np.sort(np.random.default_rng(17).choice(S, min(S, n_rows), replace=False))
        qs, ks, vs = (torch.stack([t[bb, :, hh] for bb, hh in heads], dim=1)[None].float().cpu().numpy()
                      for t in (q, k, v))
        got = torch.stack([o[bb, :, hh] for bb, hh in heads], dim=1).float().cpu().numpy()[rows]
        t0 = time.perf_counter()
        ref = quantize_tensors(qs, ks, vs, "NHD", smooth)
        t1 = time.perf_counter()
        emu = np.stack([attention_from_codes(ref, S, sm, 0, i, rows=rows) for i in range(len(heads))], axis=1)
        t2 = time.perf_counter()
        exact = np.stack([exact_head(qs, ks, vs, "NHD", sm, 0, i, rows=rows) for i in range(len(heads))], axis=1)
        err = np.abs(got.astype(np.float64) - emu)

        def cos(a, b):
            a, b = np.asarray(a, np.float64).ravel(), np.asarray(b, np.float64).ravel()
            return float(a @ b / (np.linalg.norm(a) * np.linalg.norm(b)))

        n_pairs = len(heads)
        cpu_full = (t1 - t0) * (B * H / n_pairs) + (t2 - t1) * (B * H * S / (n_pairs * len(rows)))
        rows_out.append({
            "workload": name, "smooth_k": smooth,
            "prologue_ms": t_pro * 1e3, "prologue_gbs": pb / t_pro / 1e9,
            "prologue_frac_of_hbm": pb / t_pro / 1e9 / peaks["hbm_gbs"],
            "attention_ms": t_att * 1e3, "attention_tops": ops / t_att / 1e12,
            "attention_frac_of_peak": ops / t_att / 1e12 / p_att,
            "accuracy": {"cos_vs_exact": cos(got, exact), "cos_emulation_vs_exact": cos(emu, exact),
                         "max_abs_vs_emulation": float(err.max()), "mean_abs_vs_emulation": float(err.mean()),
                         "sample": f"{n_pairs} (batch, head) pairs x {len(rows)} query rows"},
            "cpu_oracle": {"sample_seconds": t2 - t0, "extrapolated_seconds": cpu_full, "cores": cores,
                           "sample": f"prologue of {n_pairs} heads + emulated attention of {len(rows)} rows each",
                           "gpu_speedup": cpu_full / (t_pro + t_att)},
            "timing": "median of 7, CUDA events around a one-call graph replay, 2xL2 scrub before each rep"})
        del q, k, v, qz, out, o
        torch.cuda.empty_cache()
    return rows_out


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    times = []
    base = None
    for i in range(args.warmup + args.steps):
        b = cpu_oracle_sample(rows=args.ref_rows, seed=3 + i)
        if i >= args.warmup:
            times.append(b)
        base = b
    val = sum(t["value"] for t in times) / len(times)
    line = {
        "impl": "reference", "metric": METRIC, "value": val, "unit": "TOPS",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * 4.0 * 28 * 16384 ** 2 * 128 / (val * 1e12), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "int8/e4m3 codes, fp32 softmax (numpy emulation)",
        "data": "synthetic", "config": bench_config(args.gpus),
        "cpu_baseline": {k: base[k] for k in ("kind", "cores", "sample")} | {"value": val, "unit": "TOPS"},
        "e2e": {"value": val, "unit": "TOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def run_profile(args):
    """One prologue and one attention call on a named workload, for ncu."""
    import torch

    from quantized_attention_fp64_gb300 import _build
    from quantized_attention_fp64_gb300.api import attention, quantize
    from quantized_attention_fp64_gb300.workloads import WORKLOADS, make_qkv

    _build.build()
    torch.cuda.set_device(0)
    w = WORKLOADS[args.workload]
    q, k, v = make_qkv(w, "cuda")
    for _ in range(args.warmup + 1):
        qz = quantize(q, k, v, "NHD", w.smooth_k)
        attention(qz, 1.0 / math.sqrt(float(w.D)), is_causal=args.causal)
    torch.cuda.synchronize()
    print(f"profiled {args.workload}" + (" (causal)" if args.causal else ""))
    return 0


def short_call_latency(torch, sageattn, sm):
    """Short calls (a few hundred tokens, where the host work and the kernel
    launches dominate): the latency of one sageattn call at a time, from
    CUDA events around the call (host marshalling, the cluster prologue and
    the attention kernel) and from the wall clock including a synchronize,
    beside torch's bf16 scaled_dot_product_attention timed the same way.
    Also the first call of a fresh process (library load included)."""
    import statistics

    from quantized_attention_fp64_gb300.workloads import custom, make_qkv

    def one_at_a_time(fn, reps=50, warm=10):
        for _ in range(warm):
            fn()
        torch.cuda.synchronize()
        ev, wall = [], []
        for _ in range(reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            t0 = time.perf_counter()
            a.record()
            fn()
            b.record()
            b.synchronize()
            wall.append((time.perf_counter() - t0) * 1e6)
            ev.append(a.elapsed_time(b) * 1e3)
        return statistics.median(ev), statistics.median(wall)

    rows = []
    for (b_, h_, s_) in ((1, 28, 256), (1, 28, 512), (1, 28, 1024), (2, 8, 1024)):
        qs, ks, vs = make_qkv(custom(b_, h_, s_, seed_index=5000 + s_, k_offset_std=2.0), "cuda")
        qt, kt, vt = (x.transpose(1, 2) for x in (qs, ks, vs))
        ours_ev, ours_wall = one_at_a_time(lambda: sageattn(qs, ks, vs, sm_scale=sm))
        ref_ev, ref_wall = one_at_a_time(
            lambda: torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=sm))
        rows.append({"workload": f"B{b_}_H{h_}_S{s_}", "sageattn_us": round(ours_ev, 2),
                     "sageattn_wall_us": round(ours_wall, 2), "sdpa_bf16_us": round(ref_ev, 2),
                     "sdpa_bf16_wall_us": round(ref_wall, 2), "ratio": round(ours_ev / ref_ev, 3)})
    code = ("import time, torch\n"
            "from quantized_attention_fp64_gb300.workloads import custom, make_qkv\n"
            "q, k, v = make_qkv(custom(1, 28, 256, seed_index=5256), 'cuda')\n"
            "torch.cuda.synchronize()\n"
            "t0 = time.perf_counter()\n"
            "from quantized_attention_fp64_gb300 import sageattn\n"
            "sageattn(q, k, v)\n"
            "torch.cuda.synchronize()\n"
            "print(time.perf_counter() - t0)\n")
    first = None
    try:
        r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True, timeout=300)
        if r.returncode == 0:
            first = float(r.stdout.strip().splitlines()[-1])
    except (subprocess.SubprocessError, ValueError):
        first = None
    return {"timing": "one call at a time: median of 50 (CUDA events around the call; wall clock with a "
                      "synchronize)", "reference": "torch.nn.functional.scaled_dot_product_attention, bf16",
            "rows": rows, "first_call_s": first,
            "first_call_note": "fresh process, B1 H28 S256: library load, module load and the call"}


def run_gpu(args):
    import torch

    from quantized_attention_fp64_gb300 import _build, device_error, dist, sageattn, workspace_size
    from quantized_attention_fp64_gb300.api import alloc_bundle, attention, quantize

    _build.build()
    rank, world, local = dist_setup(args.gpus)
    peaks, peak_kind = load_peaks()
    from quantized_attention_fp64_gb300.workloads import WORKLOADS, make_qkv

    w = WORKLOADS[WORKLOAD]
    B, H, S, D = w.B, w.H, w.S, 128
    strong = args.strong and world > 1
    ops_total = float(w.attention_ops)
    q, k, v = make_qkv(w, "cuda")
    out = torch.empty_like(q)
    sm = 1.0 / math.sqrt(128.0)
    stream = torch.cuda.current_stream()
    if strong:
        # this rank's block of heads (strided views of the full tensors: each
        # rank holds the whole input, as after a broadcast, and computes its
        # heads; no exchange)
        h0, h1 = dist.head_shard(H, rank, world)
        qb, kb, vb = (dist.head_block(t, rank, world) for t in (q, k, v))
        out_b = torch.empty((B, S, h1 - h0, D), dtype=torch.bfloat16, device="cuda")
        ws = torch.empty(workspace_size(B, S, h1 - h0, D), dtype=torch.uint8, device="cuda")

        def step():
            sageattn(qb, kb, vb, tensor_layout="NHD", sm_scale=sm, out=out_b, workspace=ws)
    else:
        ws = torch.empty(workspace_size(B, S, H, D), dtype=torch.uint8, device="cuda")

        def step():
            sageattn(q, k, v, tensor_layout="NHD", sm_scale=sm, out=out, workspace=ws)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if device_error() != 0:
        raise RuntimeError("device error word set during warm-up")

    # --- timed region: K whole steps
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
    barrier(world)
    t_step = max_over_ranks(e0.elapsed_time(e1) / 1e3 / args.steps, world)
    clocks = clk.summary()
    # whole-job attention ops per step: the full workload split over the ranks
    # (strong), or one workload per rank (weak)
    job_ops = ops_total if strong else world * ops_total

    # --- per-kernel timing on the launching stream (the benchmark workload):
    # each kernel alone, replayed from a CUDA graph of n_k back-to-back calls
    # (warm: K and V of one head are re-read from L2 by every unit anyway),
    # and once more with L2 cold (a 2xL2 scrub before each single call)
    qz = alloc_bundle(B, S, H, q.device)
    scratch = torch.empty(max(1, workspace_size(B, S, H, D)), dtype=torch.uint8, device="cuda")
    n_k = max(args.steps, 5)

    def graph_time(fn):
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            fn()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side):
                for _ in range(n_k):
                    fn()
        torch.cuda.current_stream().wait_stream(side)
        g.replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        g.replay()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / 1e3 / n_k

    l2 = torch.cuda.get_device_properties(torch.cuda.current_device()).L2_cache_size
    scrub = torch.empty(2 * l2, dtype=torch.uint8, device="cuda")
    t_pro = graph_time(lambda: quantize(q, k, v, "NHD", True, out=qz, scratch=scratch))
    t_att = graph_time(lambda: attention(qz, sm, out=out))
    t_pro_cold = cold_time(torch, lambda: quantize(q, k, v, "NHD", True, out=qz, scratch=scratch), scrub)
    t_att_cold = cold_time(torch, lambda: attention(qz, sm, out=out), scrub)
    # the causal mask (sage_attention_ex): the kernel skips the key tiles a
    # query tile cannot see, so it does the visible half of the work
    t_att_causal = graph_time(lambda: attention(qz, sm, out=out, is_causal=True))
    ops_causal = 4.0 * B * H * D * (S * (S + 1) / 2)
    # head dimension 64 at the same size (the pages' second workload): the
    # plain three-kernel prologue and the D = 64 attention kernel
    w64 = WORKLOADS["B1_H28_S16384_D64"]
    q64, k64, v64 = make_qkv(w64, "cuda")
    qz64 = alloc_bundle(w64.B, w64.S, w64.H, q64.device, 64)
    out64 = torch.empty_like(q64)
    sm64 = 1.0 / math.sqrt(64.0)
    t_pro64 = graph_time(lambda: quantize(q64, k64, v64, "NHD", True, out=qz64))
    t_att64 = graph_time(lambda: attention(qz64, sm64, out=out64))
    del q64, k64, v64, qz64, out64
    if device_error() != 0:
        raise RuntimeError("device error word set during timing")
    configs = config_rows(torch, peaks, scrub, sm) if (rank == 0 and not args.no_configs) else None
    short_calls = short_call_latency(torch, sageattn, sm) if rank == 0 else None

    # --- end to end through the C ABI with pinned host buffers: every step
    # copies the inputs in and the output back (sage_sageattn_host, whose
    # head groups' copies overlap the other groups' kernels)
    from quantized_attention_fp64_gb300 import host_workspace_size, sageattn_host

    if strong:
        qh, kh, vh = (t.contiguous().cpu().pin_memory() for t in (qb, kb, vb))
        hb = h1 - h0
    else:
        qh, kh, vh = (t.cpu().pin_memory() for t in (q, k, v))
        hb = H
    oh = torch.empty(qh.shape, dtype=torch.bfloat16, pin_memory=True)
    ws_host = torch.empty(host_workspace_size(B, S, hb, D), dtype=torch.uint8, device="cuda")

    def e2e_step():
        sageattn_host(qh, kh, vh, tensor_layout="NHD", sm_scale=sm, out=oh, workspace=ws_host)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    step()  # the device path's result (out last held a causal timing run)
    torch.cuda.synchronize()
    if not torch.equal(oh, (out_b if strong else out).cpu()):
        raise RuntimeError("host-buffer path disagrees with the device path")
    barrier(world)
    ee0, ee1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ee0.record(stream)
    for _ in range(args.steps):
        e2e_step()
    ee1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    t_e2e = max_over_ranks(ee0.elapsed_time(ee1) / 1e3 / args.steps, world)
    del ws_host

    n_elem = B * S * hb * D
    s_pad = -(-S // 128) * 128
    pro_bytes = prologue_bytes(B, H, S, D)
    # sage_quantize also writes the fp16 copies of the Q/K codes the tensor
    # cores read (sm_103a has no int8 MMA kind)
    pro_moved = pro_bytes + 4 * B * H * s_pad * D
    p_att, p16, p8 = attention_peak(peaks)
    att_tflops = ops_total / t_att / 1e12
    line = {
        "metric": METRIC,
        "value": job_ops / t_step / 1e12,
        "unit": "TOPS",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": t_step * 1e3,
        "higher_is_better": True,
        "scaling": "strong" if strong else "weak",
        "vs_baseline": None,
        "dtype": "int8 QK (exact on fp16 tensor cores), e4m3 PV, fp32 softmax",
        "data": "synthetic",
        "config": bench_config(world, strong),
        "roofline": {"kernel": "attention_tc", "bound": "tensor", "achieved": att_tflops, "peak": p_att,
                     "unit": "TFLOP/s", "frac": att_tflops / p_att, "traffic": attention_traffic(),
                     "traffic_unit": "bytes per launch (DRAM read + write, one ncu capture of this source)",
                     "peak_note": f"harmonic mean of fp16 {p16:.1f} and e4m3 {p8:.1f} TFLOP/s "
                                  f"({peak_kind} bf16 burst: the kernel is timed alone; e4m3 = 2x nominal ratio)"},
        "attention_kernel": {"ms": t_att * 1e3, "tflops": att_tflops, "frac_of_peak": att_tflops / p_att,
                             "cold_l2_ms": t_att_cold * 1e3,
                             "cold_l2_frac_of_peak": ops_total / t_att_cold / 1e12 / p_att},
        "attention_kernel_causal": {"ms": t_att_causal * 1e3, "visible_ops": ops_causal,
                                    "tflops": ops_causal / t_att_causal / 1e12,
                                    "frac_of_peak": ops_causal / t_att_causal / 1e12 / p_att},
        "prologue": {"ms": t_pro * 1e3, "call": "sage_quantize", "algorithmic_bytes": pro_bytes,
                     "gbs": pro_bytes / t_pro / 1e9, "frac_of_hbm": pro_bytes / t_pro / 1e9 / peaks["hbm_gbs"],
                     "cold_l2_ms": t_pro_cold * 1e3, "cold_l2_gbs": pro_bytes / t_pro_cold / 1e9,
                     "cold_l2_frac_of_hbm": pro_bytes / t_pro_cold / 1e9 / peaks["hbm_gbs"],
                     "bytes_written_and_read": pro_moved, "gbs_moved": pro_moved / t_pro / 1e9,
                     "peak_gbs": peaks["hbm_gbs"], "bound": "hbm"},
        "head_dim_64": {"workload": "B1_H28_S16384_D64", "attention_ms": t_att64 * 1e3,
                        "attention_tflops": float(w64.attention_ops) / t_att64 / 1e12,
                        "attention_frac_of_peak": float(w64.attention_ops) / t_att64 / 1e12 / p_att,
                        "prologue_ms": t_pro64 * 1e3,
                        "prologue_gbs": 9 * w64.B * w64.H * w64.S * 64 / t_pro64 / 1e9,
                        "prologue_frac_of_hbm": 9 * w64.B * w64.H * w64.S * 64 / t_pro64 / 1e9 / peaks["hbm_gbs"]},
        "configs": configs,
        "short_calls": short_calls,
        "e2e": {"value": job_ops / t_e2e / 1e12, "unit": "TOPS", "h2d_bytes_per_step": 3 * 2 * n_elem,
                "d2h_bytes_per_step": 2 * n_elem, "ms_per_step": t_e2e * 1e3,
                "call": "sage_sageattn_host (pinned host q, k, v, out; head groups' copies overlap the kernels)"},
        # per step: the prologue kernel and the attention kernel (plus one
        # cudaMemsetAsync of the prologue's counters, not a kernel of ours)
        "gpu_launches": 2 * args.steps,
        "clocks": clocks,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_oracle_sample(rows=args.cpu_rows, heads=args.cpu_heads)
    if rank == 0:
        print(json.dumps(line))
    dist.teardown(world)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--ref-rows", type=int, default=1024, help="query rows per --impl reference step")
    ap.add_argument("--cpu-rows", type=int, default=16384, help="query rows per head of the cpu_baseline sample")
    ap.add_argument("--cpu-heads", type=int, default=2, help="heads of the cpu_baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true", help="skip the per-configuration table")
    ap.add_argument("--strong", action="store_true",
                    help="with N > 1: split the workload's heads over the ranks (strong scaling) instead of "
                         "running one replica per rank")
    ap.add_argument("--profile", action="store_true", help="run one prologue + attention on --workload and exit")
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--causal", action="store_true", help="with --profile: the attention call with the causal mask")
    args = ap.parse_args()
    if args.profile:
        return run_profile(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
