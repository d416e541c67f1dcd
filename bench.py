#!/usr/bin/env python3
"""Benchmark of the Dion3 / Gram Newton-Schulz hot path on GB300 (one process per GPU).

Headline step (the whole hot path): one Dion3 step over the two megabatches of a 7B dense
model's hidden matrices -- 128 x (4096 x 4096) and 96 x (4096 x 11008) -- with f = 1/4
(k = 1024 rows), mu = 0.95, eta = 0.01 (eta' = 0.02), l1 row selection, T = 5 with the
Jordan triple (3.4445, -4.7750, 2.0315), restarts after iterations 2 and 4, Gram iterates in
float16.  State: W fp32 N(0, 0.02), M fp32 starting at zero, G bf16 low-rank-plus-noise
(seed 4000 + matrix index + 10^6 * set), two pre-generated G sets alternating step by step.
All inputs are resident in HBM (65 GB per step, far larger than the 129 MB L2).

The JSON line also carries:
  phases       device time per phase (CUDA events recorded by the library on its stream),
  roofline     for the dominant phase's kernel,
  e2e          the same step fed from pinned HOST memory (G copied in, selected rows copied
               out, every step),
  gram_ns      Gram Newton-Schulz matrices/s on the 7B megabatches (bf16, f = 1, restarts 2,4),
  sym_gemm     the symmetric-GEMM sweep (TFLOP/s on n^2 k useful FLOPs, vs torch.matmul),
  cpu_baseline the float64 oracle on a bounded sample of the same step.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "Gram-NS matrices/s & Dion3 step ms per megabatch; sym-GEMM TFLOP/s vs bf16 peak"
JORDAN = (3.4445, -4.7750, 2.0315)
T_ITERS = 5
ABC = [JORDAN] * T_ITERS
RESTARTS = (2, 4)
MEGABATCHES = [(128, 4096, 4096), (96, 4096, 11008)]  # (batch, n, m): attention and MLP shapes
F = (1, 4)
MU, ETA = 0.95, 0.01
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# Pass C with the decay carried: reads M[S,:] (fp32) and writes X_S (fp16); M[S,:] is not written.
GATHER_BYTES = 6.0
DECAY_NOTE = ("M[S,:] <- mu M[S,:] of each step is applied by the next step's momentum pass "
              "(dion3_step_carry: same fp32 roundings, bit-identical state; pass C skips its write of M[S,:])")
WORKLOAD = ("dion3_step f=1/4 on 7B dense shapes: megabatches 128x4096x4096 + 96x4096x11008 "
            "(k=1024, alpha'=4 and 10.75), T=5 Jordan triple, restarts after 2 and 4, mu=0.95, eta=0.01, l1 "
            "selection, fp16 Gram iterates, W/M fp32, G bf16")


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-sub", action="store_true", help="skip the Gram-NS and sym-GEMM sub-measurements")
    ap.add_argument("--no-cpu", action="store_true", help="skip the oracle CPU baseline")
    ap.add_argument("--case", choices=["gram_small", "gram_mid", "gram_mid_mlp", "step_small", "step_small_mlp",
                                       "sym_gemm", "sym_small", "moe", "moe_gram", "moe_w2_cols", "fp32"],
                    default=None,
                    help="run one small profiling case (a few GB, inputs larger than L2) instead of the bench")
    return ap.parse_args()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(PEAKS_FALLBACK), "fallback"


def gram_flops(k: int, m: int, T: int = T_ITERS, restarts=RESTARTS) -> int:
    """(4T + 3a - 3) k^3 + r * 3 (a - 1) k^3 with a = m / k, in exact integers (useful FLOPs)."""
    r = len(restarts)
    return (4 * T - 3) * k ** 3 + 3 * m * k * k + r * 3 * (m * k * k - k ** 3)


def gram_chain_products(k: int, m: int, T: int = T_ITERS, restarts=RESTARTS, es: int = 2):
    """(useful FLOPs, algorithmic DRAM bytes) of each product of one matrix's Gram-NS chain in a
    Dion3 step, in launch order (k > 128: separate products; 16-bit iterates of es bytes; the
    last product is the fused W update, which reads and writes k fp32 rows of W)."""
    xxt = (k * k * m, (k * m + k * k) * es)            # X X^T: reads X, writes R
    poly = (k ** 3, 2 * k * k * es)                     # a I + b R + c R^2: reads R, writes Z
    prod = (k ** 3, 3 * k * k * es)                     # Q Z, R Z, (R Z) Z: two in, one out
    qx = (2 * k * k * m, (k * k + 2 * k * m) * es)      # restart: reads Q, X; writes X
    wupd = (2 * k * k * m, (k * k + k * m) * es + 8 * k * m)
    seq, q_identity = [xxt], True
    for t in range(1, T + 1):
        seq.append(poly)
        if q_identity:
            q_identity = False
        else:
            seq.append(prod)
        if t in restarts:
            seq += [qx, xxt]
            q_identity = True
        elif t < T:
            seq += [prod, prod]
    seq.append(wupd)
    return seq


def gram_chain_bound_ms(mbs, tc_peak_tflops: float, hbm_gbs: float) -> float:
    """Attainable time of the product chains of megabatches [(B, n, m)]: each product takes at
    least its useful FLOPs at the tensor peak and its algorithmic bytes at the copy bandwidth."""
    total = 0.0
    for B, n, m in mbs:
        for f, b in gram_chain_products(k_rows(n), m):
            total += max(B * f / (tc_peak_tflops * 1e12), B * b / (hbm_gbs * 1e9))
    return total * 1e3


def k_rows(n: int) -> int:
    return -((-n * F[0]) // F[1])


def sample_indices(B: int):
    """Matrices 0, B/2 and B-1 of a megabatch: the oracle's timing and parity sample."""
    return sorted({0, B // 2, B - 1})


def clock_at_max(clk) -> bool:
    """True when the sampled median SM clock is within 3% of the maximum."""
    try:
        return float(clk["sm_mhz"]) >= 0.97 * float(clk["sm_max_mhz"])
    except (KeyError, TypeError, ValueError):
        return False


def time_variant_steps(torch, d3, mbs, ws, status, K, workload, **kw):
    """K carried steps of both megabatches with one option changed (same state chain)."""
    if K <= 0:
        return None
    for s in range(2):   # the first step applies the previous variant's pending decay
        for x in mbs:
            carried_step(d3, x, s % 2, ws, status, **kw)
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    for s in range(K):
        for x in mbs:
            carried_step(d3, x, s % 2, ws, status, **kw)
    t1.record()
    torch.cuda.synchronize()
    return {"workload": workload, "ms_per_step": t0.elapsed_time(t1) / K, "steps": K,
            "device_status": int(status.item())}


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, index: int):
        self.path = tempfile.mktemp(prefix="clocks_", suffix=".csv")
        self.proc = None
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-i", str(index), "-lms", "200"], stdout=self.fh, stderr=subprocess.DEVNULL)
        except OSError as e:
            self.err = str(e)

    def stop(self):
        if self.proc is None:
            return {"error": getattr(self, "err", "nvidia-smi unavailable")}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        sm, smax, reasons = [], [], set()
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for name, val in zip(self.NAMES, parts[5:9]):
                    if val.lower().startswith("active"):
                        reasons.add(name)
        os.unlink(self.path)
        if not sm:
            return {"error": "no samples"}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------- ranks
def rank_seed_offset(rank: int) -> int:
    """Each rank draws its own megabatches (weak scaling): seeds are shifted by 10^5 per rank,
    more than any seed range a single rank uses."""
    return 10 ** 5 * rank


def combine_over_ranks(torch, dist, ms_rank: float, world: int, device) -> tuple[float, float]:
    """(slowest rank's ms per step, whole-job ms per megabatch step).  Every rank processes its
    own megabatches in the same time window, so the job finishes `world` steps' worth of
    megabatches in the slowest rank's time."""
    if dist is not None and world > 1:
        t = torch.tensor([ms_rank], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms_rank = float(t.item())
    return ms_rank, ms_rank / world


# ----------------------------------------------------------------------------- inputs
def step_inputs(torch, synthetic, dev, rank: int):
    mbs = []
    idx0 = 0
    for (B, n, m) in MEGABATCHES:
        W = torch.empty((B, n, m), dtype=torch.float32, device=dev)
        for i in range(B):
            W[i].copy_(synthetic.gaussian((n, m), seed=5000 + idx0 + i + rank_seed_offset(rank), std=0.02,
                                          device=dev))
        M = torch.zeros((B, n, m), dtype=torch.float32, device=dev)
        Gs = []
        for s in range(2):
            G = torch.empty((B, n, m), dtype=torch.bfloat16, device=dev)
            for i in range(B):
                synthetic.lowrank_plus_noise(n, m, 4000 + idx0 + i + 10 ** 6 * s + rank_seed_offset(rank),
                                             dtype=torch.bfloat16, device=dev, out=G[i])
            Gs.append(G)
        sel = torch.empty((B, k_rows(n)), dtype=torch.int32, device=dev)
        mbs.append({"B": B, "n": n, "m": m, "W": W, "M": M, "Gs": Gs, "sel": sel})
        idx0 += B
    return mbs


def carried_step(d3, x, slot, ws, status, events=None, f=F, norm_p=1, compute=None):
    """One step of megabatch x; its decay of M[S,:] is left to the next call (x["carried"])."""
    import torch

    d3.step(x["W"], x["M"], x["Gs"][slot], f=f, mu=MU, eta=ETA, norm_p=norm_p, abc=ABC, restart_after=RESTARTS,
            compute=torch.float16 if compute is None else compute, sel_out=x["sel"], workspace=ws, status=status,
            events=events,
            carry=(x["sel"], MU) if x.get("carried") else None, defer=True)
    x["carried"] = True


# ----------------------------------------------------------------------------- ours
def run_ours(args):
    import torch

    import matrix_orthogonalizing_optimizer_syrk_gb300 as d3
    import synthetic
    from matrix_orthogonalizing_optimizer_syrk_gb300 import _build

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0:
        _build.build()
    if dist is not None:
        dist.barrier()
    d3.lib()
    peaks, peaks_kind = load_peaks()

    mbs = step_inputs(torch, synthetic, dev, rank)
    # matrix 0 of each megabatch before any step: the oracle sample (timed on the host) and the
    # inputs of the bench's own parity check
    want_cpu = rank == 0 and world == 1 and not args.no_cpu
    samples = [(x["B"], [(i, x["W"][i].cpu().numpy().copy(), x["Gs"][0][i].float().cpu().numpy())
                         for i in sample_indices(x["B"])]) for x in mbs] if want_cpu else None
    ws_bytes = max(d3.workspace_bytes_step(x["B"], x["n"], x["m"], F[0], F[1], p, torch.float16, len(RESTARTS))
                   for x in mbs for p in (1, 2))   # l1 for the headline, l2 for the step_l2_selection figure
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)

    def one_step(s_idx, events=None):
        for gi, x in enumerate(mbs):
            carried_step(d3, x, s_idx % 2, ws, status, None if events is None else events[gi])

    for s in range(args.warmup):
        one_step(s)
    torch.cuda.synchronize()

    K = args.steps
    phase_ev = [[[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in mbs] for _ in range(K)]
    for step_evs in phase_ev:
        for evs in step_evs:
            for e in evs:
                e.record()  # creates the event handle the library records into
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    time.sleep(0.3)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    t0.record()
    for s in range(K):
        one_step(args.warmup + s, phase_ev[s])
    t1.record()
    torch.cuda.synchronize()
    wall1 = time.perf_counter()
    if dist is not None:
        dist.barrier()
    clk = clocks.stop()
    ms_total = t0.elapsed_time(t1)
    ms_rank, ms_job = combine_over_ranks(torch, dist, ms_total / K, world, dev)
    dev_status = int(status.item())
    # the same step with rows ranked by their L2 norm (exact sums of squares), as the
    # benchmark configuration words it; same state chain, same number of steps
    step_l2 = time_variant_steps(torch, d3, mbs, ws, status, K, "the headline step with norm_p=2 (rows ranked by "
                                 "exact sums of squares, i.e. by row L2 norm), same megabatches and state chain",
                                 norm_p=2)
    step_bf16 = time_variant_steps(torch, d3, mbs, ws, status, K, "the headline step with bfloat16 Gram iterates "
                                   "(fp32 accumulation), same megabatches and state chain", compute=torch.bfloat16)

    # phase split (sum over steps, per megabatch)
    names = ["momentum_keys", "select", "gather", "gram_ns_products"]
    per_mb = []
    for gi, x in enumerate(mbs):
        acc = [0.0] * 4
        for s in range(K):
            evs = phase_ev[s][gi]
            for p in range(4):
                acc[p] += evs[p].elapsed_time(evs[p + 1])
        per_mb.append([a / K for a in acc])  # ms per step
    hbm = float(peaks.get("hbm_gbs", PEAKS_FALLBACK["hbm_gbs"]))
    tc_sus = float(peaks.get("bf16_tflops_sustained", PEAKS_FALLBACK["bf16_tflops_sustained"]))
    bytesA = sum(10.0 * x["B"] * x["n"] * x["m"] for x in mbs)
    bytesC = sum(GATHER_BYTES * x["B"] * k_rows(x["n"]) * x["m"] for x in mbs)
    flops = sum(float(x["B"] * gram_flops(k_rows(x["n"]), x["m"])) for x in mbs)
    ph = {n: sum(pm[i] for pm in per_mb) for i, n in enumerate(names)}
    # the chain's attainable time: per product, the slower of its tensor and HBM times
    bound_ms = gram_chain_bound_ms([(x["B"], x["n"], x["m"]) for x in mbs], tc_sus, hbm)
    phases = {
        "momentum_keys": {"ms": ph["momentum_keys"], "GB/s": bytesA / ph["momentum_keys"] / 1e6,
                          "frac_hbm": bytesA / ph["momentum_keys"] / 1e6 / hbm,
                          "algorithmic_bytes": bytesA},
        "select": {"ms": ph["select"]},
        "gather": {"ms": ph["gather"], "GB/s": bytesC / ph["gather"] / 1e6, "frac_hbm": bytesC / ph["gather"] / 1e6 / hbm,
                   "algorithmic_bytes": bytesC},
        "gram_ns_products": {"ms": ph["gram_ns_products"], "TFLOP/s": flops / ph["gram_ns_products"] / 1e9,
                             "frac_tensor_sustained": flops / ph["gram_ns_products"] / 1e9 / tc_sus,
                             "useful_flops": flops,
                             "attainable_ms": bound_ms,
                             "frac_of_attainable": bound_ms / ph["gram_ns_products"]},
        "per_megabatch_ms": [{"shape": f"{x['B']}x{x['n']}x{x['m']}", "ms": sum(pm)} for x, pm in zip(mbs, per_mb)],
    }
    dominant = max(names, key=lambda n: ph[n])
    launches_per_mb = d3.step_launch_count(T_ITERS, RESTARTS, k_rows(MEGABATCHES[0][1]), carry=True)
    if dominant == "gram_ns_products":
        n_launch = sum(d3.gram_core_launch_count(T_ITERS, RESTARTS, k_rows(x["n"])) for x in mbs)
        achieved = flops / ph[dominant] / 1e9
        tc_burst = float(peaks.get("bf16_tflops", PEAKS_FALLBACK["bf16_tflops"]))
        # The burst peak was measured at the maximum SM clock, the sustained one at the clock a
        # seconds-long GEMM loop settles to under the power cap: take the one whose clock this
        # run saw.
        at_max = clock_at_max(clk)
        peak = tc_burst if at_max else tc_sus
        roof = {"kernel": "tc_gemm_kernel (all tcgen05 GEMM launches of the Gram-NS chain)", "bound": "tensor",
                "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                "peak_source": (f"{peaks_kind} bf16_tflops (burst; the run's median SM clock was at its maximum)"
                                if at_max else f"{peaks_kind} bf16_tflops_sustained (the run's SM clock sat below "
                                               f"its maximum)") + "; fp16 dense rate = bf16 dense rate",
                "frac_of_burst": achieved / tc_burst, "frac_of_sustained": achieved / tc_sus,
                "launches_per_step": n_launch, "per_launch_work": flops / n_launch}
    else:
        kernel_bytes = bytesA if dominant == "momentum_keys" else bytesC
        achieved = kernel_bytes / ph[dominant] / 1e6
        roof = {"kernel": dominant, "bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                "frac": achieved / hbm, "peak_source": f"{peaks_kind} hbm_gbs",
                "launches_per_step": len(mbs), "per_launch_work": kernel_bytes / len(mbs)}
    roof["traffic"] = recorded_traffic(roof["kernel"])

    line = {
        "metric": METRIC,
        "value": ms_job,
        "unit": "ms per megabatch step (both 7B shape groups)",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": ms_rank,
        "higher_is_better": False,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "fp16",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "megabatches": [f"{b}x{n}x{m}" for b, n, m in MEGABATCHES],
                   "l2": "inputs larger than L2 (about 65 GB touched per step)", "state": "W, M fp32; G bf16",
                   "gram_iterates": "float16 (the paper's precision), fp32 accumulation",
                   "error_feedback": DECAY_NOTE,
                   "parallelism": f"replica per GPU x{world} (independent megabatches, no collective)"},
        "roofline": roof,
        "phases": phases,
        "step_l2_selection": step_l2,
        "step_bf16_iterates": step_bf16,
        "gpu_launches": K * len(mbs) * launches_per_mb,
        "clocks": clk,
        "device_status": dev_status,
        "wall_s_timed": wall1 - wall0,
    }

    # end to end: G from pinned host memory, selected rows back to the host, every step
    line["e2e"] = run_e2e(torch, d3, mbs, ws, status, args, dev, dist)

    del mbs, ws
    torch.cuda.empty_cache()
    if rank == 0 and not args.no_sub:
        line["gram_ns"] = bench_gram_ns(torch, d3, synthetic, dev, peaks, peaks_kind)
        line["sym_gemm"] = bench_sym_gemm(torch, d3, synthetic, dev, peaks, peaks_kind)
        line["moe_step"] = bench_moe_step(torch, d3, synthetic, dev, peaks, peaks_kind)
        line["moe_w2_columns"] = bench_moe_w2_cols(torch, d3, synthetic, dev)
        line["gram_ns_fp32"] = bench_gram_fp32(torch, d3, synthetic, dev)
    if rank == 0 and world == 1 and not args.no_cpu:
        line["cpu_baseline"], line["parity"] = cpu_baseline_and_parity(torch, d3, dev, samples)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


def recorded_traffic(kernel: str):
    """dram read+write bytes per launch from the committed ncu summary, if it was taken on the
    current source of that kernel (matched by a hash of its source file); else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    entry = rec.get(kernel)
    if not entry:
        return None
    src = os.path.join(ROOT, "matrix_orthogonalizing_optimizer_syrk_gb300", "csrc", entry["source"])
    try:
        with open(src, "rb") as f:
            h = hashlib.sha256(f.read()).hexdigest()[:16]
    except OSError:
        return None
    return entry["bytes_per_launch"] if h == entry.get("source_sha256_16") else None


def run_e2e(torch, d3, mbs, ws, status, args, dev, dist):
    """The step fed from pinned host memory: every step copies its G (both megabatches) host to
    device and reads its selected rows back.  Copies run on their own stream into the device
    G buffer the previous step is not using, so step t+1's copy overlaps step t's compute; the
    timed region holds every step's copy, compute and read-back."""
    host_G = [x["Gs"][0].to("cpu").pin_memory() for x in mbs]
    host_sel = [torch.empty(x["sel"].shape, dtype=torch.int32).pin_memory() for x in mbs]
    h2d = sum(g.numel() * g.element_size() for g in host_G)
    d2h = sum(s.numel() * s.element_size() for s in host_sel)
    comp = torch.cuda.current_stream()
    copy = torch.cuda.Stream()
    K = max(1, args.steps)
    copied = [torch.cuda.Event() for _ in range(K + 1)]
    computed = [torch.cuda.Event() for _ in range(K + 1)]

    def enqueue_copy(t):
        slot = t % 2
        if t >= 2:
            copy.wait_event(computed[t - 2])  # step t-2 has finished reading this buffer
        with torch.cuda.stream(copy):
            for x, hg in zip(mbs, host_G):
                x["Gs"][slot].copy_(hg, non_blocking=True)
        copied[t].record(copy)

    def enqueue_step(t):
        comp.wait_event(copied[t])
        for x, hs in zip(mbs, host_sel):
            carried_step(d3, x, t % 2, ws, status)
            hs.copy_(x["sel"], non_blocking=True)
        computed[t].record(comp)

    # warm-up pass through the same pipeline (untimed)
    enqueue_copy(0)
    enqueue_step(0)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(comp)
    copy.wait_event(t0)
    enqueue_copy(0)
    for t in range(K):
        if t + 1 < K:
            enqueue_copy(t + 1)
        enqueue_step(t)
    t1.record(comp)
    torch.cuda.synchronize()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    _, ms_job = combine_over_ranks(torch, dist, t0.elapsed_time(t1) / K, world, dev)
    return {"value": ms_job, "unit": "ms per megabatch step (both 7B shape groups)",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "path": "G copied from pinned host memory on a copy stream (step t+1's copy overlaps step t), "
                    "dion3_step_carry (decay carried) through the C ABI, selected rows copied back every step"}


def _time_calls(torch, fn, reps, flush=None):
    ts = []
    for _ in range(reps):
        if flush is not None:
            flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b))
    return statistics.median(ts)


def bench_gram_ns(torch, d3, synthetic, dev, peaks, peaks_kind):
    """Gram NS on the 7B megabatches (f = 1): bf16 momenta, fp16 iterates, restarts after 2, 4."""
    out = {"workload": "gram_ns on 128x4096x4096 + 96x4096x11008 bf16 low-rank+noise, T=5 Jordan, restarts 2,4, "
                       "fp16 iterates", "batches": []}
    total_ms, total_flops = 0.0, 0.0
    idx0 = 0
    for (B, n, m) in MEGABATCHES:
        X = torch.empty((B, n, m), dtype=torch.bfloat16, device=dev)
        for i in range(B):
            synthetic.lowrank_plus_noise(n, m, 3000 + idx0 + i, dtype=torch.bfloat16, device=dev, out=X[i])
        idx0 += B
        O = torch.empty_like(X)
        ws = torch.empty(max(d3.workspace_bytes_gram_ns(B, n, m, torch.bfloat16, c, len(RESTARTS))
                             for c in (torch.float16, torch.bfloat16)), dtype=torch.uint8, device=dev)
        fn = lambda: d3.gram_ns(X, ABC, RESTARTS, compute=torch.float16, out=O, workspace=ws)  # noqa: E731
        fn()
        torch.cuda.synchronize()
        ms = _time_calls(torch, fn, 3)
        fl = float(B * gram_flops(n, m))
        entry = {"shape": f"{B}x{n}x{m}", "ms": ms, "matrices_per_s": B / ms * 1e3, "TFLOP/s": fl / ms / 1e9}
        # the same batch with bfloat16 iterates, and with the paper's single restart (after iteration 2)
        for name, compute, rs in (("bf16_iterates", torch.bfloat16, RESTARTS),
                                  ("restart_after_2_only", torch.float16, (2,))):
            f2 = lambda: d3.gram_ns(X, ABC, rs, compute=compute, out=O, workspace=ws)  # noqa: E731
            f2()
            torch.cuda.synchronize()
            ms2 = _time_calls(torch, f2, 3)
            fl2 = float(B * gram_flops(n, m, restarts=rs))
            entry[name] = {"restarts": list(rs), "iterates": str(compute).replace("torch.", ""), "ms": ms2,
                           "matrices_per_s": B / ms2 * 1e3, "TFLOP/s": fl2 / ms2 / 1e9}
        if n == m:
            # alpha = 1: the standard Newton-Schulz fallback on the same batch (T (3 alpha + 1) n^3 FLOPs)
            ws2 = torch.empty(d3.workspace_bytes_ns_standard(B, n, m, torch.float16), dtype=torch.uint8, device=dev)
            fn2 = lambda: d3.ns_standard(X, ABC, compute=torch.float16, out=O, workspace=ws2)  # noqa: E731
            fn2()
            torch.cuda.synchronize()
            ms2 = _time_calls(torch, fn2, 3)
            fl2 = float(B * T_ITERS * (3 * m / n + 1) * n ** 3)
            entry["ns_standard_fallback"] = {"ms": ms2, "matrices_per_s": B / ms2 * 1e3, "TFLOP/s": fl2 / ms2 / 1e9}
            del ws2
        out["batches"].append(entry)
        total_ms += ms
        total_flops += fl
        del X, O, ws
        torch.cuda.empty_cache()
    peak = float(peaks.get("bf16_tflops", PEAKS_FALLBACK["bf16_tflops"]))
    out["matrices_per_s"] = sum(b for b, _, _ in MEGABATCHES) / total_ms * 1e3
    out["TFLOP/s"] = total_flops / total_ms / 1e9
    for name in ("bf16_iterates", "restart_after_2_only"):
        ms_v = sum(e[name]["ms"] for e in out["batches"])
        out[name] = {"matrices_per_s": sum(b for b, _, _ in MEGABATCHES) / ms_v * 1e3, "ms": ms_v}
    out["frac_tensor_burst"] = out["TFLOP/s"] / peak
    out["peak_source"] = f"{peaks_kind} bf16_tflops"
    return out


def bench_moe_step(torch, d3, synthetic, dev, peaks, peaks_kind):
    """Dion3 step on a fine-grained MoE megabatch: 16 layers x 64 experts x {w1, w3, w2 oriented}
    = 3072 matrices of 768 x 2048, f = 1/8 (k = 96, alpha' = 21.3), restarts after 2 and 4."""
    B, n, m = 3072, 768, 2048
    fk = (1, 8)
    k = -((-n * fk[0]) // fk[1])
    W = synthetic.gaussian((B, n, m), seed=6000, std=0.02, device=dev)
    M = torch.zeros((B, n, m), dtype=torch.float32, device=dev)
    Gs = [synthetic.lowrank_batch(B, n, m, base_seed=5000 + 10 ** 6 * s, dtype=torch.bfloat16, device=dev)
          for s in range(2)]
    ws = torch.empty(d3.workspace_bytes_step(B, n, m, fk[0], fk[1], 1, torch.float16, len(RESTARTS)),
                     dtype=torch.uint8, device=dev)
    sel = torch.empty((B, k), dtype=torch.int32, device=dev)
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
    for e in evs:
        e.record()
    state = {"s": 0}

    def fn(events=None):
        d3.step(W, M, Gs[state["s"] % 2], f=fk, mu=MU, eta=ETA, norm_p=1, abc=ABC, restart_after=RESTARTS,
                compute=state.get("compute", torch.float16), sel_out=sel, workspace=ws, events=events,
                carry=(sel, MU) if state["s"] > 0 else None, defer=True)
        state["s"] += 1

    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    ms = _time_calls(torch, fn, 5)
    fn(evs)
    torch.cuda.synchronize()
    ph = [evs[i].elapsed_time(evs[i + 1]) for i in range(4)]
    # the same carried step with bfloat16 Gram iterates (the configuration's precision word)
    state["compute"] = torch.bfloat16
    for _ in range(2):
        fn()
    torch.cuda.synchronize()
    ms_bf16 = _time_calls(torch, fn, 5)
    hbm = float(peaks.get("hbm_gbs", PEAKS_FALLBACK["hbm_gbs"]))
    bytes_a = 10.0 * B * n * m
    bytes_c = GATHER_BYTES * B * k * m
    out = {"workload": "dion3_step f=1/8 on 3072 x 768x2048 (MoE experts), T=5 Jordan, restarts 2,4, fp16 iterates, "
                       "decay of M[S] carried",
           "ms": ms, "ms_bf16_iterates": ms_bf16,
           "phases_ms": {"momentum_keys": ph[0], "select": ph[1], "gather": ph[2], "gram_ns_products": ph[3]},
           "momentum_frac_hbm": bytes_a / ph[0] / 1e6 / hbm,
           "hbm_floor_ms": (bytes_a + bytes_c) / hbm / 1e6,
           "peak_source": f"{peaks_kind} hbm_gbs"}
    del W, M, Gs, ws
    torch.cuda.empty_cache()
    return out


def bench_moe_w2_cols(torch, d3, synthetic, dev):
    """The 1024 MoE w2 matrices in their stored layout (2048 x 768, short side = columns), f = 1/8:
    dion3_step_cols, beside dion3_step on the same matrices oriented (768 x 2048)."""
    B, m, n = 1024, 2048, 768
    fk = (1, 8)
    out = {"workload": "MoE w2: 1024 x (2048 x 768) stored, f=1/8 (k=96 columns), T=5 Jordan, restarts 2,4, "
                       "fp16 iterates"}
    for name, shape, fn_name in (("columns_stored_2048x768", (B, m, n), "step_cols"),
                                 ("rows_oriented_768x2048", (B, n, m), "step")):
        W = synthetic.gaussian(shape, seed=6100, std=0.02, device=dev)
        M = torch.zeros(shape, dtype=torch.float32, device=dev)
        G = synthetic.lowrank_batch(B, shape[1], shape[2], base_seed=6200, dtype=torch.bfloat16, device=dev)
        fn = getattr(d3, fn_name)
        call = lambda: fn(W, M, G, f=fk, mu=MU, eta=ETA, abc=ABC, restart_after=RESTARTS)  # noqa: E731
        for _ in range(3):
            call()
        torch.cuda.synchronize()
        out[name + "_ms"] = _time_calls(torch, call, 5)
        del W, M, G
        torch.cuda.empty_cache()
    return out


def bench_gram_fp32(torch, d3, synthetic, dev):
    """fp32 Gram NS on one 256 x 1024 N(0,1) matrix from seed 0, restart after 2 (latency)."""
    X = synthetic.gaussian((256, 1024), seed=0, device="cpu").to(dev)
    X = X / X.norm()
    ws = torch.empty(d3.workspace_bytes_gram_ns(1, 256, 1024, torch.float32, torch.float32, 1), dtype=torch.uint8,
                     device=dev)
    O = torch.empty_like(X)
    fn = lambda: d3.gram_ns(X, ABC, (2,), compute=torch.float32, out=O, workspace=ws)  # noqa: E731
    fn()
    torch.cuda.synchronize()
    ms = _time_calls(torch, fn, 20)
    # the same call captured once in a CUDA graph and replayed (no per-launch host work)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        fn()
    graph.replay()
    torch.cuda.synchronize()
    ms_g = _time_calls(torch, graph.replay, 20)
    return {"workload": "gram_ns fp32 (FFMA) 256x1024, T=5 Jordan, restart after 2", "us": ms * 1e3,
            "matrices_per_s": 1e3 / ms, "cuda_graph_us": ms_g * 1e3}


def bench_sym_gemm(torch, d3, synthetic, dev, peaks, peaks_kind):
    """D = A A^T (+ C): n in {1024..8192}, k in {n, 4n}; TFLOP/s on n^2 k useful FLOPs; L2 flushed."""
    peak = float(peaks.get("bf16_tflops", PEAKS_FALLBACK["bf16_tflops"]))
    flush_buf = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    flush = lambda: flush_buf.fill_(1)  # noqa: E731
    rows = []
    for n in (1024, 2048, 4096, 8192):
        for kmul in (1, 4):
            k = n * kmul
            A = synthetic.gaussian((n, k), seed=2000 + n + k, std=k ** -0.5, dtype=torch.bfloat16, device=dev)
            C = synthetic.symmetric_gaussian(n, seed=2100 + n, dtype=torch.bfloat16, device=dev)
            D = torch.empty((n, n), dtype=torch.bfloat16, device=dev)
            for beta in (0.0, 1.0):
                ours = lambda: d3.sym_gemm(A, C=C if beta else None, beta=beta, out=D)  # noqa: E731
                if beta:
                    ref = lambda: torch.addmm(C, A, A.T, out=D)  # noqa: E731
                else:
                    ref = lambda: torch.matmul(A, A.T, out=D)  # noqa: E731
                ours()
                ref()
                torch.cuda.synchronize()
                t_ours = _time_calls(torch, ours, 5, flush)
                t_ref = _time_calls(torch, ref, 5, flush)
                tf = n * n * k / t_ours / 1e9
                rows.append({"n": n, "k": k, "beta": beta, "ms": t_ours, "TFLOP/s": tf, "frac": tf / peak,
                             "torch_matmul_ms": t_ref, "speedup_vs_torch_matmul": t_ref / t_ours})
            del A, C, D
    head = [r for r in rows if r["n"] == 8192 and r["k"] == 32768 and r["beta"] == 0.0][0]
    return {"workload": "sym_gemm bf16, fp32 accumulate, n in {1024,2048,4096,8192}, k in {n,4n}, beta in {0,1}",
            "headline": {"n": 8192, "k": 32768, "TFLOP/s": head["TFLOP/s"], "frac": head["frac"]},
            "peak": peak, "peak_source": f"{peaks_kind} bf16_tflops (kernel timed alone)", "sweep": rows}


# ----------------------------------------------------------------------------- CPU oracle
def cpu_sample_inputs(synthetic, torch, which: int):
    """Sample `which` (0, 1, 2 -> matrix 0, B/2, B-1) of each megabatch at the first timed step's
    state (M = 0), built on the host with the bench's seeds."""
    import numpy as np

    out = []
    idx0 = 0
    for (B, n, m) in MEGABATCHES:
        i = sample_indices(B)[which]
        W = synthetic.gaussian((n, m), seed=5000 + idx0 + i, std=0.02, device="cpu").numpy()
        G = synthetic.lowrank_plus_noise(n, m, 4000 + idx0 + i, dtype=torch.bfloat16, device="cpu").float().numpy()
        out.append((B, W, np.zeros((n, m), np.float32), G))
        idx0 += B
    return out


def oracle_step_ms(samples) -> float:
    """Oracle time for one Dion3 step of every megabatch, extrapolated from one matrix of each."""
    import oracle

    total = 0.0
    for B, W, M, G in samples:
        t0 = time.perf_counter()
        oracle.dion3_step(W, M, G, F[0], F[1], mu=MU, eta=ETA, norm_p=1, abc=ABC, restart_after=RESTARTS)
        total += (time.perf_counter() - t0) * B
    return total * 1e3


def cpu_baseline_and_parity(torch, d3, dev, samples):
    """The oracle's Dion3 step on matrices 0, B/2 and B-1 of each megabatch (their first-step
    inputs, as generated on the device), timed on the host cores; the mean time per matrix of a
    megabatch is scaled by its size (extrapolated).  Parity: matrix 0 of each megabatch runs two
    steps (the second with the same G) through the C ABI as the timed loop runs them (batch 1,
    decay of M[S,:] carried into the second step's momentum pass and applied at the end),
    compared with the oracle's two plain steps."""
    import numpy as np

    import oracle

    total = 0.0
    checks = []
    per_matrix_s = {}
    for B, picks in samples:
        times = []
        for j, (i, W0, G0) in enumerate(picks):
            n, m = W0.shape
            M0 = np.zeros((n, m), np.float32)
            t0 = time.perf_counter()
            W1, M1, S, _ = oracle.dion3_step(W0, M0, G0, F[0], F[1], mu=MU, eta=ETA, norm_p=1, abc=ABC,
                                             restart_after=RESTARTS)
            times.append(time.perf_counter() - t0)
            if j != 0:
                continue
            W2, M2, S2, _ = oracle.dion3_step(W1, M1, G0, F[0], F[1], mu=MU, eta=ETA, norm_p=1, abc=ABC,
                                              restart_after=RESTARTS)
            Wd = torch.from_numpy(W0).to(dev).unsqueeze(0).contiguous()
            Md = torch.zeros((1, n, m), dtype=torch.float32, device=dev)
            Gd = torch.from_numpy(G0).to(device=dev, dtype=torch.bfloat16).unsqueeze(0).contiguous()
            status = torch.zeros(1, dtype=torch.int32, device=dev)
            x = {"W": Wd, "M": Md, "Gs": [Gd, Gd], "sel": torch.empty((1, k_rows(n)), dtype=torch.int32, device=dev)}
            carried_step(d3, x, 0, None, status)
            sel1 = x["sel"][0].cpu().numpy()
            Wd1 = Wd[0].double().cpu().numpy()
            carried_step(d3, x, 1, None, status)
            d3.decay_rows(Md, x["sel"], MU)
            torch.cuda.synchronize()
            rel = lambda got, ref: float(np.linalg.norm(got - ref) / np.linalg.norm(ref))  # noqa: E731
            checks.append({"shape": f"{n}x{m}",
                           "rows_selected_equal": bool(np.array_equal(sel1, S) and
                                                       np.array_equal(x["sel"][0].cpu().numpy(), S2)),
                           "M_bit_exact": bool(np.array_equal(Md[0].cpu().numpy().view(np.uint32),
                                                              M2.view(np.uint32))),
                           "dW_rel_frob": max(rel(Wd1 - W0, W1 - W0), rel(Wd[0].double().cpu().numpy() - Wd1, W2 - W1)),
                           "device_status": int(status.item())})
            del Wd, Md, Gd, x
        per_matrix_s[f"{B}x{picks[0][1].shape[0]}x{picks[0][1].shape[1]}"] = times
        total += statistics.mean(times) * B
    base = {"value": total * 1e3, "unit": "ms per megabatch step (both 7B shape groups)",
            "cores": len(os.sched_getaffinity(0)), "kind": "oracle", "extrapolated": True,
            "sample": "one oracle Dion3 step (float64, exact keys) on matrices 0, B/2 and B-1 of each megabatch "
                      "(4096x4096 and 4096x11008, first-step inputs, M=0); the mean time per matrix is scaled by the "
                      "megabatch sizes 128 and 96 (extrapolated)",
            "seconds_per_matrix": per_matrix_s}
    parity = {"against": "two oracle steps on matrix 0 of each megabatch (the cpu_baseline sample's inputs, G "
                         "used twice), run through the C ABI with batch 1 as the timed loop runs them (carried "
                         "decay, applied at the end); rows of both steps, M after both, worst dW of the two",
              "tolerance": {"rows": "bit-exact", "M": "bit-exact", "dW_rel_frob": 3e-2}, "checks": checks}
    return base, parity


def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import torch

    import synthetic

    samples = [cpu_sample_inputs(synthetic, torch, j) for j in range(3)]
    for w in range(args.warmup):
        oracle_step_ms(samples[w % 3])
    t0 = time.perf_counter()
    vals = [oracle_step_ms(samples[s % 3]) for s in range(max(1, args.steps))]
    wall = time.perf_counter() - t0
    v = statistics.mean(vals)
    cores = len(os.sched_getaffinity(0))
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "ms per megabatch step (both 7B shape groups)",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": v, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "megabatches": [f"{b}x{n}x{m}" for b, n, m in MEGABATCHES]},
        "cpu_baseline": {"value": v, "unit": "ms per megabatch step (both 7B shape groups)", "cores": cores,
                         "kind": "oracle", "extrapolated": True,
                         "sample": "step s: one oracle Dion3 step on matrix 0, B/2 or B-1 (s mod 3) of each "
                                   "megabatch, scaled by 128 and 96 (extrapolated); value = mean over the steps"},
        "e2e": {"value": v, "unit": "ms per megabatch step (both 7B shape groups)", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "wall_s_timed": wall,
    }
    print(json.dumps(line), flush=True)


def run_case(args):
    """Small, self-contained workloads for ncu captures (prints timings, not a bench line)."""
    import torch

    import matrix_orthogonalizing_optimizer_syrk_gb300 as d3
    import synthetic
    from matrix_orthogonalizing_optimizer_syrk_gb300 import _build

    _build.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    out = {"case": args.case}
    if args.case == "gram_small":
        B, n, m = 16, 1024, 4096  # 128 MB of bf16 input
        X = synthetic.lowrank_batch(B, n, m, base_seed=7000, dtype=torch.bfloat16, device=dev)
        fn = lambda: d3.gram_ns(X, ABC, RESTARTS, compute=torch.float16)  # noqa: E731
    elif args.case in ("gram_mid", "gram_mid_mlp"):
        # the 7B step's product chain on 72 of its selected-row matrices (k = 1024, fp16 X_S read in
        # place): every launch's working set is larger than L2 (each k x k buffer 144 MB), so its
        # DRAM bytes per matrix carry over to the full megabatches (ncu traffic captures)
        B, n, m = 72, 1024, (4096 if args.case == "gram_mid" else 11008)
        X = synthetic.lowrank_batch(B, n, m, base_seed=7050, dtype=torch.float16, device=dev)
        O = torch.empty_like(X)
        ws = torch.empty(d3.workspace_bytes_gram_ns(B, n, m, torch.float16, torch.float16, len(RESTARTS)),
                         dtype=torch.uint8, device=dev)
        fn = lambda: d3.gram_ns(X, ABC, RESTARTS, compute=torch.float16, out=O, workspace=ws)  # noqa: E731
    elif args.case in ("step_small", "step_small_mlp"):
        # 16 x 4096 x 4096 (1 GB of W and of M, 0.5 GB of G) or 8 x 4096 x 11008 (1.4 GB of W and of M)
        B, n, m = (16, 4096, 4096) if args.case == "step_small" else (8, 4096, 11008)
        W = synthetic.gaussian((B, n, m), seed=7100, std=0.02, device=dev)
        M = torch.zeros((B, n, m), dtype=torch.float32, device=dev)
        G = synthetic.lowrank_batch(B, n, m, base_seed=7200, dtype=torch.bfloat16, device=dev)
        x = {"W": W, "M": M, "Gs": [G], "sel": torch.empty((B, k_rows(n)), dtype=torch.int32, device=dev)}
        fn = lambda: carried_step(d3, x, 0, None, None)  # noqa: E731
    elif args.case == "moe":
        B, n, m = 3072, 768, 2048  # the MoE megabatch at full size (launch-list captures only)
        W = synthetic.gaussian((B, n, m), seed=7400, std=0.02, device=dev)
        M = torch.zeros((B, n, m), dtype=torch.float32, device=dev)
        G = synthetic.lowrank_batch(B, n, m, base_seed=7500, dtype=torch.bfloat16, device=dev)
        x = {"W": W, "M": M, "Gs": [G], "sel": torch.empty((B, 96), dtype=torch.int32, device=dev)}
        fn = lambda: carried_step(d3, x, 0, None, None, f=(1, 8))  # noqa: E731
    elif args.case == "moe_gram":
        B, n, m = 768, 96, 2048  # a quarter of the MoE megabatch's selected rows, 302 MB of bf16
        X = synthetic.lowrank_batch(B, n, m, base_seed=7600, dtype=torch.bfloat16, device=dev)
        fn = lambda: d3.gram_ns(X, ABC, RESTARTS, compute=torch.float16)  # noqa: E731
    elif args.case == "moe_w2_cols":
        B, m, n = 1024, 2048, 768  # the MoE w2 matrices in their stored layout, column selection
        W = synthetic.gaussian((B, m, n), seed=7700, std=0.02, device=dev)
        M = torch.zeros((B, m, n), dtype=torch.float32, device=dev)
        G = synthetic.lowrank_batch(B, m, n, base_seed=7800, dtype=torch.bfloat16, device=dev)
        fn = lambda: d3.step_cols(W, M, G, f=(1, 8), mu=MU, eta=ETA, abc=ABC, restart_after=RESTARTS)  # noqa: E731
    elif args.case == "sym_small":
        # the small corner of the symmetric-GEMM sweep, each shape ours then torch.matmul (cuBLAS),
        # with a 256 MB L2 flush before every call
        flush_buf = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
        calls = []
        for n, k in ((1024, 1024), (1024, 4096), (2048, 2048), (2048, 8192)):
            A = synthetic.gaussian((n, k), seed=2000 + n + k, std=k ** -0.5, dtype=torch.bfloat16, device=dev)
            D = torch.empty((n, n), dtype=torch.bfloat16, device=dev)
            calls.append((f"{n}x{k}", A, D))

        def fn():
            for _, A, D in calls:
                flush_buf.fill_(1)
                d3.sym_gemm(A, out=D)
                flush_buf.fill_(1)
                torch.matmul(A, A.T, out=D)
        for name, A, D in calls:
            ours = lambda: d3.sym_gemm(A, out=D)  # noqa: E731
            ref = lambda: torch.matmul(A, A.T, out=D)  # noqa: E731
            ours()
            ref()
            torch.cuda.synchronize()
            out[name] = {"ours_us": 1e3 * _time_calls(torch, ours, 10, lambda: flush_buf.fill_(1)),
                         "torch_matmul_us": 1e3 * _time_calls(torch, ref, 10, lambda: flush_buf.fill_(1))}
    elif args.case == "fp32":
        X = synthetic.gaussian((256, 1024), seed=0, device="cpu").to(dev)
        fn = lambda: d3.gram_ns(X, ABC, (2,), compute=torch.float32)  # noqa: E731
    else:
        n, k = 8192, 16384  # 256 MB of bf16 input
        A = synthetic.gaussian((n, k), seed=7300, std=k ** -0.5, dtype=torch.bfloat16, device=dev)
        D = torch.empty((n, n), dtype=torch.bfloat16, device=dev)
        fn = lambda: d3.sym_gemm(A, out=D)  # noqa: E731
    fn()
    torch.cuda.synchronize()
    out["ms"] = _time_calls(torch, fn, 2)
    print(json.dumps(out), flush=True)


def main():
    args = parse_args()
    if args.case:
        run_case(args)
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
