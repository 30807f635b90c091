"""Benchmark of the W4A16 GEMM hot path on one GB300 (or N replicas).

Headline (``value``): one step = the whole decode-shaped sweep of an 8B-class
decoder layer: the four layer shapes (K, N) = (4096, 6144), (4096, 4096),
(4096, 28672), (14336, 4096) times M in {1, 4, 16}, asymmetric int4, group
128, fp16 activations and output, fp32 accumulation: 12 GEMM launches through
the C-ABI library, with the packed weights (offline repack, timed separately)
and the activations resident in HBM.  Weight copies are rotated so that no
launch finds its weights in L2 (distinct weight bytes per step exceed the L2
size; even and odd steps use disjoint copy sets).  All timed steps are one
CUDA graph timed with CUDA events on the launch stream.

Per-config block (``configs``): every (shape, M) problem of the decode,
prefill, 70B-class and symmetric-G64 workloads, each timed on its own as a
CUDA graph of 50 launches over rotated weight copies (more than 3x the L2),
replayed 10 times (median and min), with TFLOP/s, weight GB/s and the
fraction of the roofline that bounds it (HBM on the algorithmic bytes for
small M, the dense 16-bit tensor-core peak for large M, the larger of the two
times in between).  The dominant kernel's ``roofline`` entry uses these
per-problem times.

Prints one JSON line (rank 0).  ``--impl reference`` times the CPU oracle
(numpy dequant + float64 matmul) on the host cores on a column sample of the
decode workload instead.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "decode_8b"
CONFIG_WORKLOADS = ("decode_8b", "prefill_8b", "class_70b", "sym_g64")
GRAPH_LAUNCHES = 50      # launches per per-problem graph
GRAPH_REPEATS = 10       # timed replays per problem (median and min)


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0,
                    help="target CPU time of the oracle baseline sample")
    ap.add_argument("--no-tune", action="store_true",
                    help="skip tm_tune (variant selection from measured throughput); use the "
                         "table in TM_TUNE_CACHE or the built-in rule")
    ap.add_argument("--warm-replays", type=int, default=0,
                    help="untimed graph replays before the timed one (0: as many as fit in 1.5 s)")
    ap.add_argument("--case", type=str, default=None,
                    help="K,N,M: time one decode-format problem instead of the sweep (for profiling)")
    ap.add_argument("--case-fmt", choices=["w4", "int8", "fp8", "w4_g32"], default="w4",
                    help="with --case: the weight format")
    ap.add_argument("--variant", type=str, default=None,
                    help="with --case: kernel:block_m:split_k:dq_warps (default: tuned/auto)")
    ap.add_argument("--reps", type=int, default=6, help="with --case: launches")
    ap.add_argument("--configs", type=str, default=",".join(CONFIG_WORKLOADS),
                    help="workloads of the per-problem block ('' to skip it)")
    ap.add_argument("--formats", type=str, default="int8,fp8,w4_g32",
                    help="non-default weight formats to time beside the configs ('' skips)")
    ap.add_argument("--attn-case", type=str, default=None,
                    help="one decode-attention case name:case[:chunk_tiles], repeated --reps times")
    ap.add_argument("--attention", type=str, default=",".join(("attn_8b_kv8", "attn_8b_kv4")),
                    help="decode-attention workloads to time beside the configs ('' skips)")
    ap.add_argument("--config-cpu-seconds", type=float, default=1.0,
                    help="CPU time of the oracle sample per shape in the per-config block")
    return ap.parse_args()


# ------------------------------------------------------------------ helpers
def weight_bytes(K: int, N: int, group: int, symmetric: bool) -> float:
    """Algorithmic weight bytes: 4-bit codes + 16-bit scale (+ 4-bit zero) per group."""
    per_group = 2.0 + (0.0 if symmetric else 0.5)
    return K * N / 2 + (K / group) * N * per_group


def problem_bytes(M: int, K: int, N: int, group: int, symmetric: bool) -> float:
    """Algorithmic bytes of one GEMM: weights + A (fp16) + C (fp16)."""
    return weight_bytes(K, N, group, symmetric) + 2.0 * M * K + 2.0 * M * N


def max_over_ranks(x: float, world: int, device=None) -> float:
    """The largest value of x over all ranks (a job takes as long as its
    slowest rank).  device: where the reduction tensor lives (the GPU for
    NCCL, None for gloo)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(units_per_rank: float, world: int, seconds: float) -> float:
    """Whole-job throughput: every rank processes units_per_rank (weak
    scaling), all ranks together in `seconds` (the slowest rank's time)."""
    return world * units_per_rank / seconds


def recorded_traffic(ent: dict, source_hash: str, ran: list) -> int | None:
    """Measured DRAM bytes per launch of the dominant kernel: the mean of the
    recorded captures of the problems that ran with it, ran = [(K, N, M,
    variant dict)], each captured with the same kernel sources and variant.
    None if the sources changed or any problem has no capture."""
    if not ran or ent.get("source_hash") != source_hash:
        return None
    rec = {(x["case"], x.get("variant")): x["dram_read"] + x["dram_write"]
           for x in ent.get("per_problem", [])}
    got = [rec.get((f"{K},{N},{M}", f"{v['kernel']}:{v['block_m']}:{v['split_k']}:{v['dq_warps']}"))
           for K, N, M, v in ran]
    if any(x is None for x in got):
        return None
    return round(sum(got) / len(got))


def kernel_source_hash(files: list | None = None) -> str:
    """Hash of the kernel sources under csrc/: the named files (a kernel's own
    translation unit and the headers it includes), else every file."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "w4a16_gemm_gb300", "csrc")
    for f in sorted(files if files else os.listdir(csrc)):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def load_peaks() -> tuple[dict, str]:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return json.load(f), "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def gpu_id(dev) -> str:
    """nvidia-smi -i selector of a torch device (its UUID when torch exposes it)."""
    import torch

    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return str(dev.index or 0)


class ClockSampler:
    """nvidia-smi clocks/throttle sampling in the background (200 ms period)."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,utilization.gpu,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.rows: list[list[str]] = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append([x.strip() for x in line.split(",")])

    def stop(self) -> dict | None:
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        rows = [r for r in self.rows if len(r) >= 10]
        if not rows:
            return None

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        loaded = [r for r in rows if (num(r[4]) or 0) > 0] or rows
        sm = [num(r[1]) for r in loaded if num(r[1]) is not None]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in loaded:
            for name, v in zip(names, r[6:10]):
                if v.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": num(loaded[0][2]), "reasons": sorted(reasons),
                "samples": len(rows), "samples_under_load": len(loaded)}


# ------------------------------------------------------- per-problem timing
def roofline_terms(M: int, K: int, N: int, group: int, symmetric: bool, seconds: float,
                   peaks: dict) -> dict:
    """Roofline of one GEMM: t_hbm = algorithmic bytes / HBM peak, t_tc =
    2MNK / 16-bit tensor-core peak (burst: each problem is timed on its own);
    frac = max(t_hbm, t_tc) / measured time.  bound: 'hbm' for M <= 16,
    'tensor' for M >= 2048, 'both' in between (both fractions reported)."""
    t_hbm = problem_bytes(M, K, N, group, symmetric) / (peaks["hbm_gbs"] * 1e9)
    t_tc = 2.0 * M * N * K / (peaks["bf16_tflops"] * 1e12)
    bound = "hbm" if M <= 16 else "tensor" if M >= 2048 else "both"
    return {"bound": bound, "frac_hbm": round(t_hbm / seconds, 4), "frac_tc": round(t_tc / seconds, 4),
            "frac": round(max(t_hbm, t_tc) / seconds, 4)}


def graph_time(launch, stream, launches: int, repeats: int) -> list[float]:
    """Seconds per launch of `launch(i)`, i = 0..launches-1, captured in one
    CUDA graph and replayed `repeats` times (CUDA events on the launch stream)."""
    import torch

    with torch.cuda.stream(stream):
        for i in range(3):
            launch(i)
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(launches):
            launch(i)
    out = []
    with torch.cuda.stream(stream):
        g.replay()
        stream.synchronize()
        for _ in range(repeats):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            g.replay()
            e1.record(stream)
            e1.synchronize()
            out.append(e0.elapsed_time(e1) * 1e-3 / launches)
    del g
    return out


def variant_name(v: dict, dtype: str = "f16", wbits: int = 4) -> str:
    if v["kernel"] == "gemv":
        if wbits == 8:
            return f"gemv8_kernel<{dtype},{v['block_m']}>"
        if v["dq_warps"] == 1:
            return f"gemv_mma_kernel<{dtype},{v['block_m'] // 8}>"
        return f"gemv_kernel<{dtype},{v['block_m']}>"
    if v["kernel"] == "decode_mma":
        return f"decode_mma_kernel<{dtype},{v['block_m'] // 8}{',8' if wbits == 8 else ''}>"
    if v["kernel"] == "tc_decode":
        return f"tc_decode_kernel<{dtype},{v['block_m']},{v['dq_warps']}>"
    return f"tc_gemm_kernel<{dtype},{v['block_m']},{v['dq_warps']}{',8' if wbits == 8 else ''}>"


def oracle_problem_seconds(qw, a_bits, M: int, budget_s: float) -> tuple[float, str]:
    """CPU oracle time of one full (M, K, N) problem, measured on a column
    sample (all K) and a row sample and extrapolated linearly: dequant time
    scales with the columns, the float64 matmul with rows x columns."""
    import numpy as np

    import oracle

    K, N = qw.q.shape
    rows = min(M, 64)
    ncols = 128
    while True:
        cols = slice(0, ncols)
        z = None if qw.zeros is None else qw.zeros[:, cols]
        t0 = time.perf_counter()
        w = oracle.dequant_bits(qw.q[:, cols], qw.scales[:, cols], z, qw.group, qw.dtype)
        t1 = time.perf_counter()
        oracle.gemm_ref(a_bits[:rows], w, qw.dtype)
        t2 = time.perf_counter()
        if t2 - t0 >= budget_s / 4 or ncols >= N:
            break
        ncols = min(N, ncols * 4)
    full = (t1 - t0) * (N / ncols) + (t2 - t1) * (M / rows) * (N / ncols)
    kind = "measured" if (ncols >= N and rows >= M) else "extrapolated"
    return full, f"{kind} from {rows} rows x {ncols} columns"


def config_sweep(wl_name: str, dev, stream, peaks: dict, tune: bool, cpu_budget_s: float) -> dict:
    """Times every (shape, M) of one workload as a graph of GRAPH_LAUNCHES
    launches over rotated weight copies; the CPU oracle on a bounded sample
    of each problem beside it."""
    import math

    import torch

    from w4a16_gemm_gb300 import binding, synth

    wl = synth.WORKLOADS[wl_name]
    dt = torch.float16 if wl.dtype == "f16" else torch.bfloat16
    L2 = torch.cuda.get_device_properties(dev).L2_cache_size
    problems = []
    cpu_s_total, cpu_notes = 0.0, []
    for si, (K, N) in enumerate(wl.shapes):
        qw = synth.weight(wl_name, si)
        p = binding.to_device(qw, dev)
        wb = weight_bytes(K, N, wl.group, wl.symmetric)
        R = min(64, math.ceil(3 * L2 / wb) + 1)
        Ws = [binding.pack(p.q, p.scales, p.zeros, qw.group) for _ in range(R)]
        del p
        if tune:
            binding.tune(Ws[0], list(wl.ms))
        for M in wl.ms:
            a = synth.activations(wl_name, si, M)
            A = binding.acts_to_device(a, dt, dev)
            C = torch.empty((M, N), dtype=dt, device=dev)
            v = binding.select(Ws[0], M)
            ts = graph_time(lambda i: binding.gemm(A, Ws[i % R], out=C, stream=stream), stream,
                            GRAPH_LAUNCHES, GRAPH_REPEATS)
            binding.poll_error(stream)
            t_med, t_min = statistics.median(ts), min(ts)
            rec = {"K": K, "N": N, "M": M, "variant": v, "kernel": variant_name(v, wl.dtype),
                   "us": round(t_med * 1e6, 3), "us_min": round(t_min * 1e6, 3),
                   "tflops": round(2.0 * M * N * K / t_med / 1e12, 2),
                   "weight_gbs": round(wb / t_med / 1e9, 1),
                   "bytes": problem_bytes(M, K, N, wl.group, wl.symmetric)}
            rec.update(roofline_terms(M, K, N, wl.group, wl.symmetric, t_med, peaks))
            if cpu_budget_s > 0:
                t_cpu, how = oracle_problem_seconds(qw, a, M, cpu_budget_s)
                rec["cpu_oracle_s"] = round(t_cpu, 3)
                cpu_s_total += t_cpu
                cpu_notes.append(how)
            problems.append(rec)
            del A, C
        for w in Ws:
            w.free()
        del Ws, qw
        torch.cuda.synchronize()
    t_gpu = sum(r["us"] for r in problems) * 1e-6
    flops = sum(2.0 * r["M"] * r["N"] * r["K"] for r in problems)
    wbytes = sum(weight_bytes(r["K"], r["N"], wl.group, wl.symmetric) for r in problems)
    out = {"problems": problems,
           "tflops": round(flops / t_gpu / 1e12, 2), "weight_gbs": round(wbytes / t_gpu / 1e9, 1),
           "seconds_per_pass": round(t_gpu, 6)}
    for bound in ("hbm", "tensor", "both"):
        fr = [r["frac"] for r in problems if r["bound"] == bound]
        if fr:
            out[f"frac_{bound}_min"] = min(fr)
            out[f"frac_{bound}_median"] = round(statistics.median(fr), 4)
    if cpu_budget_s > 0:
        extrap = any("extrapolated" in n for n in cpu_notes)
        out["cpu_baseline"] = {
            "value": round(flops / cpu_s_total / 1e12, 6), "unit": "TFLOP/s",
            "weight_gbs": round(wbytes / cpu_s_total / 1e9, 4), "cores": cpu_cores(), "kind": "oracle",
            "sample": ("extrapolated: " if extrap else "") +
                      "per problem, numpy dequant (RNE) of a column sample over all K and a float64 "
                      "matmul of a row sample, scaled linearly to the full problem"}
    return out


FORMAT_SHAPES = ((4096, 6144), (4096, 4096), (4096, 28672), (14336, 4096))
FORMAT_DECODE_MS = (1, 16)
FORMAT_PREFILL = (4096, 4096, 2048)     # K, N, M (bf16)


def format_weight_bytes(fmt: str, K: int, N: int) -> float:
    """Algorithmic weight bytes of the non-default formats (group 128 unless
    named): int8 = 8-bit code + 16-bit scale + 8-bit zero per group; fp8 =
    8-bit code + 16-bit scale; w4_g32 = 4-bit code + 16-bit scale + 4-bit zero
    per group of 32."""
    if fmt == "int8":
        return K * N * (1.0 + 3.0 / 128)
    if fmt == "fp8":
        return K * N * (1.0 + 2.0 / 128)
    return K * N * (0.5 + 2.5 / 32)


def _format_weight(fmt: str, K: int, N: int, dt, dev, gen):
    """A seeded random weight of the format: uniform codes (FP8 codes with the
    two NaN patterns replaced by 1.0), scales of either sign in [2e-4, 2e-3],
    uniform zeros."""
    import torch

    from w4a16_gemm_gb300 import binding

    G = 32 if fmt == "w4_g32" else 128
    hi = 16 if fmt == "w4_g32" else 256
    q = torch.randint(0, hi, (K, N), dtype=torch.uint8, device=dev, generator=gen)
    s = torch.rand((K // G, N), device=dev, generator=gen) * 1.8e-3 + 2e-4
    s = (s * (torch.randint(0, 2, s.shape, device=dev, generator=gen) * 2 - 1)).to(dt)
    if fmt == "fp8":
        q[(q == 0x7F) | (q == 0xFF)] = 0x38
        return binding.pack_fp8(q, s, G)
    z = torch.randint(0, hi, (K // G, N), dtype=torch.uint8, device=dev, generator=gen)
    if fmt == "int8":
        return binding.pack_w8(q, s, z, G)
    return binding.pack(q, s, z, G)


def formats_sweep(fmts: list, dev, stream, peaks: dict, tune: bool) -> dict:
    """Times the non-default weight formats the way the configs are timed (graph
    of GRAPH_LAUNCHES launches over rotated weight copies): the decode shapes at
    M in FORMAT_DECODE_MS (fp16) and one prefill problem (bf16)."""
    import math

    import torch

    from w4a16_gemm_gb300 import binding

    L2 = torch.cuda.get_device_properties(dev).L2_cache_size
    gen = torch.Generator(device=dev)
    out = {}
    for fmt in fmts:
        cases = [(K, N, FORMAT_DECODE_MS, torch.float16, "f16") for K, N in FORMAT_SHAPES]
        cases.append((FORMAT_PREFILL[0], FORMAT_PREFILL[1], (FORMAT_PREFILL[2],), torch.bfloat16, "bf16"))
        problems = []
        for K, N, ms, dt, dname in cases:
            gen.manual_seed(1000 + K * 7 + N)
            wb = format_weight_bytes(fmt, K, N)
            R = min(64, math.ceil(3 * L2 / wb) + 1)
            Ws = [_format_weight(fmt, K, N, dt, dev, gen) for _ in range(R)]
            if tune:
                binding.tune(Ws[0], list(ms))
            for M in ms:
                A = torch.randn((M, K), device=dev, generator=gen).to(dt)
                C = torch.empty((M, N), dtype=dt, device=dev)
                v = binding.select(Ws[0], M)
                ts = graph_time(lambda i: binding.gemm(A, Ws[i % R], out=C, stream=stream), stream,
                                GRAPH_LAUNCHES, GRAPH_REPEATS)
                binding.poll_error(stream)
                t = statistics.median(ts)
                t_hbm = (wb + 2.0 * M * K + 2.0 * M * N) / (peaks["hbm_gbs"] * 1e9)
                t_tc = 2.0 * M * N * K / (peaks["bf16_tflops"] * 1e12)
                problems.append({"K": K, "N": N, "M": M, "dtype": dname, "variant": v,
                                 "kernel": variant_name(v, dname, 4 if fmt == "w4_g32" else 8), "us": round(t * 1e6, 3),
                                 "us_min": round(min(ts) * 1e6, 3),
                                 "tflops": round(2.0 * M * N * K / t / 1e12, 2),
                                 "weight_gbs": round(wb / t / 1e9, 1),
                                 "bound": "hbm" if M <= 16 else "tensor",
                                 "frac": round(max(t_hbm, t_tc) / t, 4)})
                del A, C
            for w in Ws:
                w.free()
            del Ws
            torch.cuda.synchronize()
        out[fmt] = {"problems": problems,
                    "weight_bytes": {"int8": "K*N*(1 + 3/128)", "fp8": "K*N*(1 + 2/128)",
                                     "w4_g32": "K*N*(1/2 + 2.5/32)"}[fmt]}
    return out


ATTN_NAMES = ("attn_8b_kv8", "attn_8b_kv4")


def attn_kv_bytes(lens, Hkv: int, D: int, bits: int) -> float:
    """Algorithmic cache bytes of one decode-attention step: per cached token
    and KV head, K and V codes (D * bits / 8 bytes each) with a 16-bit scale
    and an 8-bit zero each."""
    return float(sum(int(n) for n in lens)) * Hkv * (2 * D * bits / 8 + 2 * 3)


def attention_sweep(names: list, dev, stream, peaks: dict, cpu_budget_s: float) -> dict:
    """Times decode attention over the low-bit KV cache for every (batch,
    length mix) case of each workload, graph of GRAPH_LAUNCHES launches over
    rotated cache copies (> 3x L2 when one copy is smaller), median of
    GRAPH_REPEATS replays; HBM roofline on the algorithmic bytes (cache +
    Q + O).  The cache is drawn on the device (uniform codes and zeros,
    per-token scales uniform in the workload's range); the CPU oracle is
    timed on one sequence of each case."""
    import torch

    from w4a16_gemm_gb300 import binding, synth

    L2 = torch.cuda.get_device_properties(dev).L2_cache_size
    out = {}
    for name in names:
        wl = synth.ATTN_WORKLOADS[name]
        cases = []
        for ci, (B, _) in enumerate(wl.cases):
            c = attn_case_inputs(name, ci, dev, L2)
            copies, q, o, lens, lens_np, R = c["copies"], c["q"], c["o"], c["lens"], c["lens_np"], c["R"]
            L_max, kvb, alloc, sm = c["L_max"], c["kv_bytes"], c["alloc"], c["sm_scale"]
            plan = binding.attn_decode_plan(B, wl.Hq, wl.Hkv, L_max, wl.bits, q.dtype)
            ts = graph_time(lambda i: binding.attn_decode(q, lens=lens, kv_bits=wl.bits, sm_scale=sm, out=o,
                                                          stream=stream, **copies[i % R]),
                            stream, GRAPH_LAUNCHES, GRAPH_REPEATS)
            binding.poll_error(stream)
            t = statistics.median(ts)
            tot = kvb + 2.0 * 2 * B * wl.Hq * wl.D
            rec = {"B": B, "lens": f"{int(lens_np.min())}..{int(lens_np.max())} (sum {int(lens_np.sum())})",
                   "L_max": L_max, "us": round(t * 1e6, 3), "us_min": round(min(ts) * 1e6, 3),
                   "kv_gbs": round(kvb / t / 1e9, 1), "bytes": round(tot),
                   "frac_hbm": round(tot / t / 1e9 / peaks["hbm_gbs"], 4),
                   "chunk_tiles": plan["chunk_tiles"], "grid": plan["grid"], "copies": R,
                   "device_bytes_per_copy": alloc}
            if cpu_budget_s > 0:
                rec["cpu_oracle_s_one_seq"] = round(_attn_oracle_one(copies[0], q, lens_np, wl, sm), 4)
            cases.append(rec)
            del c, copies, q, o, lens
            torch.cuda.synchronize()
        t_all = sum(c["us"] for c in cases) * 1e-6
        b_all = sum(c["bytes"] for c in cases)
        out[name] = {"cases": cases, "kernel": f"attn_decode_kernel<{wl.dtype},{wl.bits}>",
                     "layout": f"Hq={wl.Hq} Hkv={wl.Hkv} D={wl.D}, {wl.bits}-bit KV, {wl.dtype}",
                     "gbs_over_cases": round(b_all / t_all / 1e9, 1),
                     "frac_hbm_over_cases": round(b_all / t_all / 1e9 / peaks["hbm_gbs"], 4)}
    return out


def attn_case_inputs(name: str, ci: int, dev, L2: int, copies: int | None = None) -> dict:
    """Device inputs of case ci of an attention workload: the cache drawn on
    the device (uniform codes and zeros, per-token scales uniform in the
    workload's range), in enough rotated copies that the copies together
    exceed 3x L2 (unless `copies` is given), N(0, 1) queries, the seeded
    length mix."""
    import math

    import torch

    from w4a16_gemm_gb300 import synth

    wl = synth.ATTN_WORKLOADS[name]
    B = wl.cases[ci][0]
    dt = torch.float16 if wl.dtype == "f16" else torch.bfloat16
    width = wl.D * wl.bits // 8
    zhi = 256 if wl.bits == 8 else 16
    lo, hi = (0.004, 0.012) if wl.bits == 8 else (0.06, 0.2)
    lens_np = synth.attn_lens(name, ci)
    L_max = int(-(-int(lens_np.max()) // 64) * 64)
    gen = torch.Generator(device=dev)
    gen.manual_seed(9000 + 10 * ci + wl.bits)
    kvb = attn_kv_bytes(lens_np, wl.Hkv, wl.D, wl.bits)
    R = copies or (min(64, math.ceil(3 * L2 / kvb) + 1) if kvb < 3 * L2 else 1)

    def cache():
        shp = (B, wl.Hkv, L_max)
        return dict(
            k_cache=torch.randint(0, 256, shp + (width,), dtype=torch.uint8, device=dev, generator=gen),
            v_cache=torch.randint(0, 256, shp + (width,), dtype=torch.uint8, device=dev, generator=gen),
            k_scale=(torch.rand(shp, device=dev, generator=gen) * (hi - lo) + lo).to(dt),
            v_scale=(torch.rand(shp, device=dev, generator=gen) * (hi - lo) + lo).to(dt),
            k_zero=torch.randint(0, zhi, shp, dtype=torch.uint8, device=dev, generator=gen),
            v_zero=torch.randint(0, zhi, shp, dtype=torch.uint8, device=dev, generator=gen))

    q = torch.randn((B, wl.Hq, wl.D), device=dev, generator=gen).to(dt)
    return {"copies": [cache() for _ in range(R)], "q": q, "o": torch.empty_like(q),
            "lens": torch.from_numpy(lens_np).to(dev), "lens_np": lens_np, "R": R, "L_max": L_max,
            "kv_bytes": kvb, "alloc": B * wl.Hkv * L_max * (2 * width + 6), "sm_scale": 1.0 / math.sqrt(wl.D)}


def run_attn_case(args) -> dict:
    """One decode-attention case, repeated eagerly over rotated cache copies
    (a small case for ncu captures): --attn-case name:case[:chunk_tiles]."""
    import torch

    from w4a16_gemm_gb300 import binding, build, synth

    build.build()
    parts = args.attn_case.split(":")
    name, ci = parts[0], int(parts[1])
    ct = int(parts[2]) if len(parts) > 2 else 0
    wl = synth.ATTN_WORKLOADS[name]
    L2 = torch.cuda.get_device_properties(0).L2_cache_size
    c = attn_case_inputs(name, ci, torch.device("cuda"), L2, copies=2)

    def launch(i):
        binding.attn_decode(c["q"], lens=c["lens"], kv_bits=wl.bits, sm_scale=c["sm_scale"], out=c["o"],
                            chunk_tiles=ct, **c["copies"][i % 2])

    for i in range(2):
        launch(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(args.reps):
        launch(i)
    e1.record()
    torch.cuda.synchronize()
    binding.poll_error()
    us = e0.elapsed_time(e1) * 1e3 / args.reps
    return {"metric": "decode attention KV GB/s (single case)", "value": round(c["kv_bytes"] / us / 1e3, 1),
            "unit": "GB/s", "case": {"workload": name, "case": ci, "B": int(len(c["lens_np"])),
                                     "L_max": c["L_max"], "chunk_tiles": ct},
            "us_per_launch": round(us, 2), "kv_bytes": c["kv_bytes"],
            "note": "eager launches, 2 rotated cache copies; for profiling, not the headline"}


def _attn_oracle_one(c, q, lens_np, wl, sm) -> float:
    """Seconds of the CPU oracle for the first sequence of a case."""
    import numpy as np

    from oracle import attention

    n = int(lens_np[0])
    h = lambda t: t[:1, :, :n].contiguous().view(torch_int16()).cpu().numpy().view(np.uint16)
    u = lambda t: t[:1, :, :n].contiguous().cpu().numpy()
    qb = q[:1].contiguous().view(torch_int16()).cpu().numpy().view(np.uint16)
    t0 = time.perf_counter()
    attention.attn_decode_ref(qb, u(c["k_cache"]), h(c["k_scale"]), u(c["k_zero"]), u(c["v_cache"]),
                              h(c["v_scale"]), u(c["v_zero"]), lens_np[:1], wl.bits, wl.dtype, sm)
    return time.perf_counter() - t0


def torch_int16():
    import torch

    return torch.int16


# ---------------------------------------------------------------- our arm
def run_ours(args, rank: int, world: int):
    import numpy as np
    import torch

    from w4a16_gemm_gb300 import binding, build, synth

    build.build()
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    wl = synth.WORKLOADS[WORKLOAD]
    dt = torch.float16
    L2 = torch.cuda.get_device_properties(dev).L2_cache_size

    # inputs: quantized weights (synthetic, seeded), packed once per copy
    shapes = list(wl.shapes)
    problems = []          # (shape_idx, M)
    for si in range(len(shapes)):
        for M in wl.ms:
            problems.append((si, M))
    n_sets = 2
    packed = {}            # (set, shape_idx, M) -> PackedW4
    acts, outs = {}, {}
    pack_times = {}
    dev_inputs = {}
    for si, (K, N) in enumerate(shapes):
        qw = synth.weight(WORKLOAD, si)
        p = binding.to_device(qw, dev)
        dev_inputs[si] = p
        for s in range(n_sets):
            for M in wl.ms:
                packed[(s, si, M)] = binding.pack(p.q, p.scales, p.zeros, qw.group)
        # time the offline repack (a1) on its own
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        ev0.record()
        tmp = binding.pack(p.q, p.scales, p.zeros, qw.group)
        ev1.record()
        torch.cuda.synchronize()
        pack_times[si] = ev0.elapsed_time(ev1) * 1e-3
        tmp.free()
        for M in wl.ms:
            acts[(si, M)] = binding.acts_to_device(synth.activations(WORKLOAD, si, M), dt, dev)
            outs[(si, M)] = torch.empty((M, N), dtype=dt, device=dev)
    del dev_inputs
    torch.cuda.synchronize()

    if not args.no_tune:
        for si in range(len(shapes)):
            binding.tune(packed[(0, si, wl.ms[0])], list(wl.ms))

    variants = {(si, M): binding.select(packed[(0, si, M)], M) for si, M in problems}

    stream = torch.cuda.Stream(device=dev)

    def launch_step(step: int):
        s = step % n_sets
        for si, M in problems:
            binding.gemm(acts[(si, M)], packed[(s, si, M)], out=outs[(si, M)], stream=stream)

    # warm-up (also sizes the split-K workspace of this stream outside capture)
    with torch.cuda.stream(stream):
        for w in range(max(args.warmup, 3)):
            launch_step(w)
    torch.cuda.synchronize()
    binding.poll_error(stream)

    K_steps = args.steps
    # all K timed steps back to back in one graph (the `value` timing)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for k in range(K_steps):
            launch_step(k)
    # clock-sampled warm replays, then the timed replay
    sampler = ClockSampler(gpu_id(dev))
    sampler.start()
    # graphs replay on the current stream: make it the launch stream
    with torch.cuda.stream(stream):
        if args.warm_replays > 0:
            for _ in range(args.warm_replays):
                graph.replay()
            torch.cuda.synchronize()
        else:
            t_end = time.time() + 1.5
            while time.time() < t_end:
                graph.replay()
                torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        graph.replay()
        t1.record(stream)
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        elapsed = t0.elapsed_time(t1) * 1e-3
    clocks = sampler.stop()
    binding.poll_error(stream)
    del graph

    # whole-job numbers
    wbytes_step = sum(weight_bytes(*shapes[si], wl.group, wl.symmetric) for si, M in problems)
    flops_step = sum(2.0 * M * shapes[si][0] * shapes[si][1] for si, M in problems)
    elapsed = max_over_ranks(elapsed, world, dev)
    value = job_rate(K_steps * wbytes_step, world, elapsed) / 1e9
    ms_per_step = elapsed / K_steps * 1e3

    # end to end through the public API with host buffers (pinned), copies timed
    a_host = {k: v.cpu().pin_memory() for k, v in acts.items()}
    c_host = {k: torch.empty(v.shape, dtype=dt).pin_memory() for k, v in outs.items()}
    h2d = sum(v.numel() * 2 for v in a_host.values())
    d2h = sum(v.numel() * 2 for v in c_host.values())
    a_dev = {k: torch.empty_like(v) for k, v in acts.items()}
    with torch.cuda.stream(stream):
        e_steps = max(10, K_steps // 4)
        for w in range(3):
            for si, M in problems:
                a_dev[(si, M)].copy_(a_host[(si, M)], non_blocking=True)
                binding.gemm(a_dev[(si, M)], packed[(w % n_sets, si, M)], out=outs[(si, M)], stream=stream)
                c_host[(si, M)].copy_(outs[(si, M)], non_blocking=True)
        stream.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for k in range(e_steps):
            for si, M in problems:
                a_dev[(si, M)].copy_(a_host[(si, M)], non_blocking=True)
                binding.gemm(a_dev[(si, M)], packed[(k % n_sets, si, M)], out=outs[(si, M)],
                             stream=stream)
                c_host[(si, M)].copy_(outs[(si, M)], non_blocking=True)
        e1.record(stream)
        stream.synchronize()
    e2e_s = max_over_ranks(e0.elapsed_time(e1) * 1e-3, world, dev)
    e2e_value = job_rate(e_steps * wbytes_step, world, e2e_s) / 1e9
    for w in packed.values():
        w.free()
    del packed, acts, outs, a_dev, a_host, c_host
    torch.cuda.synchronize()

    # per-problem block: every (shape, M) of each workload, graph of 50 launches each
    peaks, peak_src = load_peaks()
    configs = {}
    for name in [x for x in args.configs.split(",") if x]:
        configs[name] = config_sweep(name, dev, stream, peaks, tune=not args.no_tune,
                                     cpu_budget_s=args.config_cpu_seconds if rank == 0 else 0.0)

    formats = None
    fmts = [x for x in args.formats.split(",") if x]
    if fmts:
        formats = formats_sweep(fmts, dev, stream, peaks, tune=not args.no_tune)

    attention = None
    anames = [x for x in args.attention.split(",") if x]
    if anames:
        attention = attention_sweep(anames, dev, stream, peaks,
                                    cpu_budget_s=args.config_cpu_seconds if rank == 0 else 0.0)

    # roofline of the dominant kernel of the headline step: the variant with the
    # most time per step, from the per-problem graph timings of the decode sweep
    roof = None
    dec = configs.get(WORKLOAD)
    if dec is not None:
        per = {}
        for r in dec["problems"]:
            rec = per.setdefault(r["kernel"], [0.0, 0.0, 0, []])
            rec[0] += r["us"] * 1e-6
            rec[1] += r["bytes"]
            rec[2] += 1
            rec[3].append((r["K"], r["N"], r["M"], r["variant"]))
        dom = max(per, key=lambda k: per[k][0])
        tot_s, tot_b, n_l, ran = per[dom]
        achieved = tot_b / tot_s / 1e9
        traffic = None
        tp = os.path.join(ROOT, "profiles", "traffic.json")
        if os.path.exists(tp):
            with open(tp) as f:
                ent = json.load(f).get(WORKLOAD, {})
            traffic = recorded_traffic(ent, kernel_source_hash(ent.get("source_files")), ran)
        roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4), "traffic": traffic,
                "kernel": dom, "problems": n_l, "avg_launch_us": round(tot_s / n_l * 1e6, 3),
                "algorithmic_bytes_per_launch": round(tot_b / n_l),
                "duration_source": f"median of {GRAPH_REPEATS} replays of a CUDA graph of "
                                   f"{GRAPH_LAUNCHES} launches per problem (rotated weight copies)",
                "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)" if peak_src == "measured"
                else "fallback 6.8 TB/s"}

    line = {
        "metric": "W4A16 GEMM weight GB/s, 8B-class decode sweep (4 layer shapes x M in {1,4,16})",
        "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": K_steps,
        "warmup": max(args.warmup, 3), "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
        "data": "synthetic (seeded N(0,1) fp16 activations; N(0,0.02) weights RTN-quantized to int4)",
        "config": {"workload": "decode_8b: (K,N) in (4096,6144),(4096,4096),(4096,28672),(14336,4096); "
                               "M in {1,4,16}; asym uint4 G=128 fp16 scales; fp16 in/out, fp32 accumulate",
                   "launches_per_step": len(problems),
                   "l2": f"inputs larger than L2: {n_sets} disjoint weight-copy sets, "
                         f"{wbytes_step / 1e6:.0f} MB distinct weights per step vs L2 {L2 / 1e6:.0f} MB",
                   "timing": "one CUDA graph of all timed steps, CUDA events on the launch stream",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "tflops": round(world * K_steps * flops_step / elapsed / 1e12, 4),
        "roofline": roof,
        "e2e": {"value": round(e2e_value, 1), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e_steps,
                "how": "eager C-ABI calls via the Python binding; A copied from pinned host, C copied back, every call"},
        "gpu_launches": K_steps * len(problems),
        "clocks": clocks,
        "pack": {"seconds_per_shape": {f"{shapes[si][0]}x{shapes[si][1]}": round(t * 1e6, 1)
                                       for si, t in pack_times.items()},
                 "unit": "us", "note": "offline repack (tm_pack_w4), timed once per shape"},
        "variants": {f"{shapes[si][0]}x{shapes[si][1]}xM{M}": variants[(si, M)] for si, M in problems},
        "configs": configs,
        "formats": formats,
        "attention": attention,
        "peaks": {"hbm_gbs": peaks["hbm_gbs"], "tensor_tflops": peaks["bf16_tflops"], "source": peak_src},
    }
    return line


# ------------------------------------------------------------- the oracle
def oracle_sample_step(col_frac: float):
    """Runs the oracle on a column sample of every problem of one step.

    Returns (seconds, weight bytes processed)."""
    import numpy as np

    import oracle
    from w4a16_gemm_gb300 import synth

    wl = synth.WORKLOADS[WORKLOAD]
    total_t, total_b = 0.0, 0.0
    for si, (K, N) in enumerate(wl.shapes):
        qw = _ORACLE_CACHE.get(si)
        if qw is None:
            qw = synth.weight(WORKLOAD, si)
            _ORACLE_CACHE[si] = qw
        ncols = max(16, int(N * col_frac))
        cols = slice(0, ncols)
        for M in wl.ms:
            a = _ORACLE_ACTS.setdefault((si, M), synth.activations(WORKLOAD, si, M))
            t0 = time.perf_counter()
            w = oracle.dequant_bits(qw.q[:, cols], qw.scales[:, cols], qw.zeros[:, cols], qw.group, qw.dtype)
            c = oracle.gemm_ref(a, w, qw.dtype)
            total_t += time.perf_counter() - t0
            total_b += weight_bytes(K, ncols, qw.group, False)
            del w, c
    return total_t, total_b


_ORACLE_CACHE: dict = {}
_ORACLE_ACTS: dict = {}


def cpu_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_baseline(target_s: float) -> dict:
    probe_t, _ = oracle_sample_step(1 / 256)
    frac = min(1.0, max(1 / 256, (target_s / max(probe_t, 1e-3)) / 256))
    t, b = oracle_sample_step(frac)
    return {"value": round(b / t / 1e9, 4), "unit": "GB/s", "cores": cpu_cores(), "kind": "oracle",
            "sample": f"all 12 problems of one decode_8b step restricted to the first "
                      f"{frac * 100:.2f}% of the N columns; numpy dequant (RNE) + float64 matmul; "
                      f"{t:.1f} s of CPU time"}


def run_reference(args) -> dict:
    K_steps, W = args.steps, args.warmup
    probe_t, _ = oracle_sample_step(1 / 256)
    budget = 120.0
    per_step_target = budget / max(1, K_steps + W)
    frac = min(1.0, max(1 / 1024, (per_step_target / max(probe_t, 1e-3)) / 256))
    for _ in range(W):
        oracle_sample_step(frac)
    t_tot, b_tot = 0.0, 0.0
    for _ in range(K_steps):
        t, b = oracle_sample_step(frac)
        t_tot += t
        b_tot += b
    value = b_tot / t_tot / 1e9
    sample = (f"each step: all 12 decode_8b problems restricted to the first {frac * 100:.3f}% "
              f"of the N columns; numpy dequant (RNE) + float64 matmul")
    return {
        "impl": "reference",
        "metric": "W4A16 GEMM weight GB/s, 8B-class decode sweep (4 layer shapes x M in {1,4,16})",
        "value": round(value, 4), "unit": "GB/s", "n_gpus": 1, "steps": K_steps, "warmup": W,
        "ms_per_step": round(t_tot / K_steps * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (same seeded inputs as the GPU arm)",
        "config": {"workload": "decode_8b (column sample), CPU oracle on the host cores"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cpu_cores(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def run_case(args) -> dict:
    """One problem of the decode format, repeated (a small case for ncu captures)."""
    import torch

    from w4a16_gemm_gb300 import binding, build, synth

    build.build()
    K, N, M = (int(x) for x in args.case.split(","))
    qw, a = synth.random_problem(1, M, K, N)
    if args.case_fmt == "w4":
        p = binding.to_device(qw)
        Ws = [binding.pack(p.q, p.scales, p.zeros, qw.group) for _ in range(4)]
    else:
        gen = torch.Generator(device="cuda")
        gen.manual_seed(5)
        Ws = [_format_weight(args.case_fmt, K, N, torch.float16, torch.device("cuda"), gen) for _ in range(4)]
    A = binding.acts_to_device(a, torch.float16)
    C = torch.empty((M, N), dtype=torch.float16, device="cuda")
    cfg = None
    if args.variant:
        k, bm, sk, dq = args.variant.split(":")
        cfg = dict(kernel=k, block_m=int(bm), split_k=int(sk), dq_warps=int(dq))
    elif not args.no_tune:
        binding.tune(Ws[0], [M])
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for i in range(2):
        binding.gemm(A, Ws[i % 4], out=C, config=cfg)
    torch.cuda.synchronize()
    e0.record()
    for i in range(args.reps):
        binding.gemm(A, Ws[i % 4], out=C, config=cfg)
    e1.record()
    torch.cuda.synchronize()
    binding.poll_error()
    us = e0.elapsed_time(e1) * 1e3 / args.reps
    wb = weight_bytes(K, N, 128, False) if args.case_fmt == "w4" else format_weight_bytes(args.case_fmt, K, N)
    return {"metric": "W4A16 GEMM weight GB/s (single problem)", "value": round(wb / us / 1e3, 1),
            "unit": "GB/s", "case": {"K": K, "N": N, "M": M, "format": args.case_fmt}, "us_per_launch": round(us, 2),
            "variant": cfg if cfg else binding.select(Ws[0], M),
            "note": "eager launches, 4 rotated weight copies; for profiling, not the headline"}


def main():
    args = parse()
    if args.attn_case:
        print(json.dumps(run_attn_case(args)), flush=True)
        return
    if args.case:
        print(json.dumps(run_case(args)), flush=True)
        return
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return
    if world > 1:
        import torch
        import torch.distributed as dist

        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        dist.init_process_group("nccl")
    line = run_ours(args, rank, world)
    if rank == 0:
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(args.cpu_seconds)
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
