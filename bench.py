"""Throughput of the per-token 4x4 Birkhoff projection on GB300.

One step = one forward pass (X -> P, Newton on the reduced dual) followed by
one backward pass (P, dP -> dX, implicit differentiation) over T = 2^26
tokens of X ~ N(0,1) fp32 (the throughput-sweep workload at its largest
size), inputs resident in HBM.  Every tensor is 4.3 GB, far larger than the
129 MB L2, so no flush is needed between steps.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  With --gpus N > 1 (launched by torchrun) each
rank projects its own 2^26 tokens (weak scaling, no collective on the data
path); the reported time is the maximum over ranks.
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

METRIC = "4×4 Birkhoff proj tokens/s fwd & fwd+bwd at 2^26 tokens; % of roofline"
LOG2_T = 26
SIGMA = 1.0
BYTES_FWD_F32 = 128  # X read + P written per token
BYTES_BWD_F32 = 192  # P, dP read + dX written per token
PEAKS_PATH = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_HBM_GBS = 6800.0
KERNEL_SOURCES = ["b4_device.cuh", "b4_math.cuh", "b4_kernels.cuh", "b4_queue.cuh", "b4_launch.cuh",
                  "b4_types.h", "k_forward.cu", "k_backward.cu"]
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "dram_traffic.txt")


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "birkhoff_projection_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def hbm_peak():
    try:
        with open(PEAKS_PATH) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def recorded_traffic():
    """Per-token DRAM bytes of each kernel from the committed ncu summary, if it
    was taken on the current kernel sources (else None)."""
    try:
        lines = open(TRAFFIC_FILE).read().splitlines()
    except OSError:
        return None
    out, src = {}, None
    for ln in lines:
        parts = ln.split()
        if len(parts) >= 2 and parts[0] == "kernel_source_hash":
            src = parts[1]
        if len(parts) >= 3 and parts[0] == "dram_bytes_per_token":
            out[parts[1]] = float(parts[2])
    if src != kernel_source_hash():
        return None
    return out


ISSUE_FILE = os.path.join(ROOT, "profiles", "issue_counts.txt")


def recorded_issue_counts():
    """Warp instructions per 32 tokens of each kernel, from the committed ncu
    summary, if it was taken on the current kernel sources (else {})."""
    try:
        lines = open(ISSUE_FILE).read().splitlines()
    except OSError:
        return {}
    out, src = {}, None
    for ln in lines:
        parts = ln.split()
        if len(parts) >= 2 and parts[0] == "kernel_source_hash":
            src = parts[1]
        if len(parts) >= 3 and parts[0] == "warp_inst_per_32_tokens":
            out[parts[1]] = float(parts[2])
    return out if src == kernel_source_hash() else {}


def issue_ceiling(inst_per_32: float, nsm: int, sm_mhz: float) -> float:
    """Tokens/s at which instruction issue alone would bind: every SM issues
    one warp instruction per clock on each of its 4 schedulers."""
    return nsm * 4 * sm_mhz * 1e6 * 32.0 / inst_per_32


def cpu_model() -> str:
    """The host CPU's model name (lscpu or /proc/cpuinfo)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.lower().startswith("model name"):
                return ln.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for ln in open("/proc/cpuinfo"):
            if ln.lower().startswith(("model name", "cpu model")):
                return ln.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform

    return platform.processor() or platform.machine()


class ClockSampler:
    """nvidia-smi samples (200 ms) while the timed region runs."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.out = ""

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        self.out = self.proc.stdout.read()

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self._t.join(timeout=5)

    def summary(self, t0=None, t1=None):
        """Median SM clock and the throttle reasons seen; restricted to samples
        inside [t0, t1] (host wall clock) when any fall there."""
        import datetime

        rows = []
        for ln in self.out.strip().splitlines():
            p = [x.strip() for x in ln.split(",")]
            if len(p) < 9:
                continue
            try:
                ts = datetime.datetime.strptime(p[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((ts, float(p[1]), float(p[2]), p[5:9]))
            except ValueError:
                continue
        inside = [r for r in rows if t0 is not None and t0 <= r[0] <= t1]
        window = "timed region"
        if not inside:
            inside, window = rows, "warm-up and timed region"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, _, r in inside for i in range(4)
                          if r[i].lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in inside),
                "sm_max_mhz": max(r[2] for r in inside), "reasons": reasons,
                "samples": len(inside), "window": window}


def max_over_ranks(x: float, dist=None, device=None) -> float:
    """Maximum of x over the ranks of the process group (x itself alone)."""
    if dist is None or not dist.is_initialized():
        return x
    import torch

    t = torch.tensor([x], dtype=torch.float64, device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tokens_per_s(tokens_per_rank: int, world: int, steps: int, max_total_ms: float) -> float:
    """Weak scaling: every rank projects its own tokens each step; the job's
    throughput is all ranks' tokens over the slowest rank's time."""
    return world * tokens_per_rank * steps / (max_total_ms * 1e-3)


def cpu_baseline(X_host, G_host, target_s: float = 12.0, single_s: float = 3.0):
    """The float64 oracle (Newton forward + implicit backward) on the host
    cores, on a bounded prefix of the same tokens; then on one core."""
    import oracle

    oracle.build()

    def timed(n):
        t0 = time.perf_counter()
        P = oracle.project64(X_host[:n])
        oracle.backward64(P, G_host[:n])
        return time.perf_counter() - t0

    n = 1 << 16
    dt = timed(n)
    n = int(min(X_host.shape[0], max(n, n * target_s / max(dt, 1e-3))))
    dt = timed(n)
    cores = oracle.num_threads()
    prev = oracle.set_num_threads(1)
    try:
        n1 = 1 << 12
        dt1 = timed(n1)
        n1 = int(min(X_host.shape[0], max(n1, n1 * single_s / max(dt1, 1e-4))))
        dt1 = timed(n1)
    finally:
        oracle.set_num_threads(prev)
    return {"value": n / dt, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "cpu_model": cpu_model(),
            "single_core": {"value": n1 / dt1, "unit": "tokens/s", "cores": 1,
                            "sample": "first %d tokens, %.1f s" % (n1, dt1)},
            "sample": "first %d tokens of the workload, float64 Newton forward + implicit "
                      "backward, %.1f s" % (n, dt)}


def evals_stats(b4, X):
    """Mean evaluations per token and the mean over consecutive 32-token
    groups of their maximum (what one warp of one-token-per-thread lanes
    waits for), from the kernel's own per-token counts."""
    _, ev, nonconv = b4.forward(X, return_stats=True)
    T = ev.numel() // 32 * 32
    wmax = ev.reshape(-1)[:T].reshape(-1, 32).amax(1).float().mean()
    return {"mean_evals": float(ev.float().mean()), "warp32_max_evals": float(wmax),
            "nonconverged": int(nonconv.item())}


def hard_configs(b4, workloads, dev, X, G, P, dX, peak, reps=10):
    """Device times of the other workloads beside the headline (inputs
    resident; each larger than L2 or rotated over copies that are):
    the fused fp32 pass and 20-iteration Sinkhorn-Knopp on the headline
    tokens; forward and forward + backward at T = 2^26, sigma = 10; the
    large-magnitude workload (2^20 tokens); the bf16 mHC batch (2^24)."""
    import torch

    T = X.shape[0]
    out = {}
    tf = time_device(lambda i: b4._fused_pass(X, G, P, dX), reps, dev)
    out["fused_f32_sigma1"] = {"tokens": T, "ms": tf, "tokens_per_s": T / (tf * 1e-3),
                               "gbs": 256 * T / (tf * 1e-3) / 1e9,
                               "hbm_frac": 256 * T / (tf * 1e-3) / 1e9 / peak,
                               "bytes_per_token": 256}
    ts = time_device(lambda i: b4.sinkhorn(X, 20, out=P), reps, dev)
    tfw = time_device(lambda i: b4.forward(X, out=P), reps, dev)
    out["sinkhorn20_f32_sigma1"] = {"tokens": T, "ms": ts, "tokens_per_s": T / (ts * 1e-3),
                                    "newton_forward_ms": tfw,
                                    "gbs": 128 * T / (ts * 1e-3) / 1e9}
    # sigma = 10 at the same size
    X10, G10 = workloads.sweep(T.bit_length() - 1, 10.0, device=dev)
    f10 = time_device(lambda i: b4.forward(X10, out=P), reps, dev)

    def fb10(i):
        b4.forward(X10, out=P)
        b4.backward(G10, P=P, out=dX)

    fb = time_device(fb10, reps, dev)
    st = evals_stats(b4, X10)
    bound_f = 128 * T / (peak * 1e9) * 1e3
    bound_fb = 320 * T / (peak * 1e9) * 1e3
    out["sigma10"] = dict(st, tokens=T, fwd_ms=f10, fwd_bwd_ms=fb,
                          fwd_tokens_per_s=T / (f10 * 1e-3), fwd_bwd_tokens_per_s=T / (fb * 1e-3),
                          fwd_hbm_frac=bound_f / f10, fwd_bwd_hbm_frac=bound_fb / fb)
    del X10, G10
    # large magnitude, 2^20 tokens (67 MB per tensor): four copies rotate
    X3, G3 = workloads.large_magnitude(device=dev)
    sets = [(X3.clone(), G3.clone(), torch.empty_like(X3), torch.empty_like(X3)) for _ in range(4)]
    T3 = X3.shape[0]
    f3 = time_device(lambda i: b4.forward(sets[i % 4][0], out=sets[i % 4][2]), 4 * reps, dev)

    def fb3(i):
        x, g, p, d = sets[i % 4]
        b4.forward(x, out=p)
        b4.backward(g, P=p, out=d)

    fb3t = time_device(fb3, 4 * reps, dev)
    out["large_magnitude"] = dict(evals_stats(b4, X3), tokens=T3, fwd_ms=f3, fwd_bwd_ms=fb3t,
                                  fwd_tokens_per_s=T3 / (f3 * 1e-3),
                                  fwd_bwd_tokens_per_s=T3 / (fb3t * 1e-3),
                                  fwd_hbm_frac=128 * T3 / (f3 * 1e-3) / 1e9 / peak,
                                  fwd_bwd_hbm_frac=320 * T3 / (fb3t * 1e-3) / 1e9 / peak,
                                  input_sets=4)
    del sets, X3, G3
    # bf16 mHC batch, 2^24 tokens (537 MB per tensor)
    Xb, Gb = workloads.mhc_batch(device=dev)
    Tb = Xb.numel() // 16
    Pb, dXb = torch.empty_like(Xb), torch.empty_like(Xb)
    tfu = time_device(lambda i: b4._fused_pass(Xb, Gb, Pb, dXb), reps, dev)

    def sepb(i):
        b4.forward(Xb, out=Pb)
        b4.backward(Gb, P=Pb, out=dXb)

    tsep = time_device(sepb, reps, dev)
    tfb = time_device(lambda i: b4.forward(Xb, out=Pb), reps, dev)
    out["mhc_bf16"] = dict(evals_stats(b4, Xb.reshape(Tb, 4, 4)), tokens=Tb, fused_ms=tfu,
                           fused_tokens_per_s=Tb / (tfu * 1e-3),
                           fused_hbm_frac=128 * Tb / (tfu * 1e-3) / 1e9 / peak,
                           separate_ms=tsep, separate_hbm_frac=160 * Tb / (tsep * 1e-3) / 1e9 / peak,
                           fwd_ms=tfb, fwd_hbm_frac=64 * Tb / (tfb * 1e-3) / 1e9 / peak)
    del Xb, Gb, Pb, dXb
    torch.cuda.empty_cache()
    return out


def run_reference(args):
    """The reference arm: the float64 oracle as it stands, on host cores."""
    import numpy as np

    import oracle
    from birkhoff_projection_gb300 import workloads

    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    oracle.build()
    n = 1 << 18  # tokens per step: a bounded sample of the workload
    X, G = workloads.sweep(18, SIGMA)  # same distribution, host generator
    x = X.double().numpy()
    g = G.double().numpy()
    for _ in range(args.warmup):
        oracle.backward64(oracle.project64(x), g)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.backward64(oracle.project64(x), g)
    dt = time.perf_counter() - t0
    value = n * args.steps / dt
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "impl": "reference",
        "config": {"workload": "sweep T=2^26 sigma=1 fwd+bwd (host sample of 2^18 tokens per step)",
                   "tokens": 1 << LOG2_T, "sigma": SIGMA},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": oracle.num_threads(),
                         "kind": "oracle", "sample": "2^18 tokens per step, float64 Newton "
                                                     "forward + implicit backward"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--log2-tokens", type=int, default=LOG2_T)
    ap.add_argument("--schedule", choices=["default", "queue", "lane", "lanes4"], default="default",
                    help="token schedule of the Newton passes (birkhoff4_opts.schedule)")
    ap.add_argument("--sigma", type=float, default=SIGMA,
                    help="logit scale of the timed workload (the headline is sigma = 1)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-hard", action="store_true",
                    help="skip the other workloads' device times (sigma 10, large magnitude, bf16 mHC, "
                         "fused fp32, Sinkhorn-20)")
    ap.add_argument("--sweep", action="store_true",
                    help="throughput sweep T = 2^12..2^26, sigma 1 and 10 (one JSON line each)")
    ap.add_argument("--mhc", action="store_true",
                    help="bf16 mHC batch [64,32,8192,4,4]: fused and separate passes")
    ap.add_argument("--eot", action="store_true",
                    help="streaming entropic OT: n = m = 65536 points, d = 64 and 512, both precisions")
    ap.add_argument("--nxn", action="store_true",
                    help="n x n kernels, n = 2..8, 1 GiB of fp32 X per n (one JSON line each)")
    ap.add_argument("--nxn-n", type=int, default=None, help="with --nxn: this n only")
    ap.add_argument("--nxn-mib", type=int, default=1024, help="with --nxn: MiB of fp32 X per n")
    ap.add_argument("--eot-profile", choices=["update", "transport", "hvp"],
                    help="profiling target (not a measurement): three calls of one streaming "
                         "EOT op on seeded clouds, n = m = --eot-n points of dimension --eot-d")
    ap.add_argument("--eot-n", type=int, default=16384)
    ap.add_argument("--eot-d", type=int, default=64)
    args = ap.parse_args()
    if args.impl == "reference":
        return run_reference(args)
    if args.eot_profile:
        return run_eot_profile(args)
    if args.sweep or args.mhc or args.nxn or args.eot:
        return run_extra(args)

    import numpy as np
    import torch

    import birkhoff_projection_gb300 as b4
    from birkhoff_projection_gb300 import workloads

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    warmup = max(args.warmup, 3)

    X, G = workloads.sweep(args.log2_tokens, args.sigma, device=dev, shard=rank)
    T = X.shape[0]
    P = torch.empty_like(X)
    dX = torch.empty_like(X)
    stream = torch.cuda.current_stream(dev)

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        b4.forward(X, out=P, schedule=args.schedule)
        if ev is not None:
            ev[1].record(stream)
        b4.backward(G, P=P, out=dX)
        if ev is not None:
            ev[2].record(stream)

    # evaluation counts of this input (outside the timed region)
    _, evals, nonconv = b4.forward(X, return_stats=True, schedule=args.schedule)
    mean_evals = float(evals.float().mean())
    del evals
    torch.cuda.synchronize(dev)

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    with ClockSampler(local) as clk:
        for _ in range(warmup):
            step()
        torch.cuda.synchronize(dev)
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize(dev)
        t0 = time.time()
        for k in range(args.steps):
            step(evs[k])
        torch.cuda.synchronize(dev)
        t1 = time.time()
        if dist is not None:
            dist.barrier()
        time.sleep(0.1)  # let the sampler flush its last line
    wall = t1 - t0
    fwd_ms = [e[0].elapsed_time(e[1]) for e in evs]
    bwd_ms = [e[1].elapsed_time(e[2]) for e in evs]
    total_ms = evs[0][0].elapsed_time(evs[-1][2])
    total_ms = max_over_ranks(total_ms, dist, dev)
    ms_step = total_ms / args.steps
    value = whole_job_tokens_per_s(T, world, args.steps, total_ms)
    fwd_avg = statistics.mean(fwd_ms)
    bwd_avg = statistics.mean(bwd_ms)
    peak, peak_kind = hbm_peak()
    fwd_gbs = BYTES_FWD_F32 * T / (fwd_avg * 1e-3) / 1e9
    bwd_gbs = BYTES_BWD_F32 * T / (bwd_avg * 1e-3) / 1e9
    traffic = recorded_traffic()
    dominant = "forward" if fwd_avg >= bwd_avg else "backward"
    dom = {"forward": (fwd_gbs, BYTES_FWD_F32, "forward_f32"),
           "backward": (bwd_gbs, BYTES_BWD_F32, "backward_f32")}[dominant]
    tr = None if traffic is None or dom[2] not in traffic else traffic[dom[2]] * T

    # MUFU ceiling: measured ex2 rate against the evaluations this input needed
    mufu = (ctypes_probe(b4, dev))
    mufu_per_token = 20.0 + (mean_evals - 1.0) * 12.0
    clocks = clk.summary(t0, t1)

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return

    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": "sweep T=2^%d sigma=%g fp32, forward + backward"
                               % (args.log2_tokens, args.sigma),
                   "tokens_per_gpu": T, "sigma": args.sigma,
                   "l2": "inputs larger than L2 (%.1f GB per tensor, L2 129 MB)" % (T * 64 / 1e9)},
        "fwd": {"tokens_per_s": world * T / (fwd_avg * 1e-3), "ms": fwd_avg, "gbs": fwd_gbs,
                "hbm_frac": fwd_gbs / peak, "mean_evals": mean_evals,
                "nonconverged": int(nonconv.item())},
        "bwd": {"tokens_per_s": world * T / (bwd_avg * 1e-3), "ms": bwd_avg, "gbs": bwd_gbs,
                "hbm_frac": bwd_gbs / peak},
        "roofline": {"bound": "hbm", "kernel": dominant, "achieved": dom[0], "peak": peak,
                     "peak_kind": peak_kind, "unit": "GB/s", "frac": dom[0] / peak,
                     "traffic": tr, "algorithmic_bytes": dom[1] * T},
        "roofline_fwd_bwd": {
            "hbm_bound_tokens_per_s": peak * 1e9 / (BYTES_FWD_F32 + BYTES_BWD_F32),
            "frac": value / world / (peak * 1e9 / (BYTES_FWD_F32 + BYTES_BWD_F32))},
        "mufu": {"ex2_per_s": mufu, "ops_per_token_fwd": mufu_per_token,
                 "bound_tokens_per_s": (mufu / mufu_per_token) if mufu else None},
        "gpu_launches": 2 * args.steps,
        "clocks": clocks,
        "wall_s": wall,
    }
    if not args.no_e2e:
        # two public host-memory paths: the kernel reading and writing pinned
        # host memory itself (zero copy) and chunked copies on the copy
        # engines; the faster is the e2e figure, the other is reported beside it
        mapped = e2e_mapped(b4, X, G, dev, steps=3)
        copies = e2e_host(b4, X, G, dev, steps=3)
        best, other = (mapped, copies) if mapped["value"] >= copies["value"] else (copies, mapped)
        best["other_path"] = {k: other[k] for k in ("api", "value", "ms_per_step", "host_link_gbs")}
        ceiling = host_link_ceiling(dev)
        best["link_ceiling"] = ceiling
        best["link_frac"] = best["host_link_gbs"] / ceiling["both_gbs"]
        line["e2e"] = best
    if not args.no_hard:
        line["hard_configs"] = hard_configs(b4, workloads, dev, X, G, P, dX, peak)
    counts = recorded_issue_counts()
    nsm = torch.cuda.get_device_properties(dev).multi_processor_count
    mhz = clocks.get("sm_mhz") or 2070.0
    line["issue_ceiling"] = {
        k: {"warp_inst_per_32_tokens": v, "ceiling_tokens_per_s": issue_ceiling(v, nsm, mhz)}
        for k, v in counts.items()} or None
    # achieved tokens/s of each counted kernel against its issue ceiling
    achieved = {"forward_f32_sigma1": T / (fwd_avg * 1e-3), "backward_f32_sigma1": T / (bwd_avg * 1e-3)}
    hard = line.get("hard_configs") or {}
    if "sigma10" in hard:
        achieved["forward_f32_sigma10"] = hard["sigma10"]["fwd_tokens_per_s"]
    if "mhc_bf16" in hard:
        achieved["fused_bf16_mhc"] = hard["mhc_bf16"]["fused_tokens_per_s"]
    for k, v in achieved.items():
        if counts.get(k):
            ic = line["issue_ceiling"][k]
            ic["achieved_frac"] = v / ic["ceiling_tokens_per_s"]
    if not args.no_cpu_baseline:
        idx = slice(0, 1 << 22)
        line["cpu_baseline"] = cpu_baseline(X[idx].double().cpu().numpy(),
                                            G[idx].double().cpu().numpy())
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def time_device(fn, reps, dev):
    """Median CUDA-event time (ms) of fn() on the current stream; inputs
    resident; for sizes below 2x L2 the caller rotates among input sets."""
    import torch

    s = torch.cuda.current_stream(dev)
    for _ in range(3):
        fn(0)
    torch.cuda.synchronize(dev)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(reps + 1)]
    ev[0].record(s)
    for i in range(reps):
        fn(i)
        ev[i + 1].record(s)
    torch.cuda.synchronize(dev)
    t = sorted(ev[i].elapsed_time(ev[i + 1]) for i in range(reps))
    return t[len(t) // 2]


def run_extra(args):
    """Extra measurement lines: the throughput sweep, the bf16 mHC batch and
    the n x n kernels, streaming entropic OT."""
    import torch

    import birkhoff_projection_gb300 as b4
    from birkhoff_projection_gb300 import workloads

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    if args.sweep:
        for sigma in workloads.SWEEP_SIGMAS:
            for lg in workloads.SWEEP_LOG2_T:
                T = 1 << lg
                # rotate among enough input sets to exceed 2x L2 in total
                nsets = max(1, -(-2 * l2 // (T * 64 * 2)))
                sets = []
                for k in range(min(nsets, 64)):
                    X, G = workloads.sweep(lg, sigma, device=dev, shard=k)
                    sets.append((X, G, torch.empty_like(X), torch.empty_like(X)))
                fw = lambda i: b4.forward(sets[i % len(sets)][0], out=sets[i % len(sets)][2])

                def fb(i):
                    X, G, P, dX = sets[i % len(sets)]
                    b4.forward(X, out=P)
                    b4.backward(G, P=P, out=dX)

                reps = max(20, min(2000, (1 << 27) // T))
                tf = time_device(fw, reps, dev)
                tfb = time_device(fb, reps, dev)
                # the same work replayed from a CUDA graph of 16 calls (no
                # host launch cost between kernels)
                graphs = {}
                for key, f in (("fwd", fw), ("fwd_bwd", fb)):
                    g = torch.cuda.CUDAGraph()
                    with torch.cuda.graph(g):
                        for i in range(16):
                            f(i)
                    graphs[key] = time_device(lambda i, g=g: g.replay(), max(5, reps // 16), dev) / 16
                _, ev, _ = b4.forward(sets[0][0], return_stats=True)
                print(json.dumps({"sweep": True, "log2_tokens": lg, "sigma": sigma,
                                  "input_sets": len(sets), "fwd_ms": tf, "fwd_bwd_ms": tfb,
                                  "fwd_tokens_per_s": T / (tf * 1e-3),
                                  "fwd_bwd_tokens_per_s": T / (tfb * 1e-3),
                                  "fwd_gbs": 128 * T / (tf * 1e-3) / 1e9,
                                  "fwd_bwd_gbs": 320 * T / (tfb * 1e-3) / 1e9,
                                  "graph_fwd_ms": graphs["fwd"], "graph_fwd_bwd_ms": graphs["fwd_bwd"],
                                  "graph_fwd_tokens_per_s": T / (graphs["fwd"] * 1e-3),
                                  "graph_fwd_bwd_tokens_per_s": T / (graphs["fwd_bwd"] * 1e-3),
                                  "mean_evals": float(ev.float().mean())}), flush=True)
                del sets
                torch.cuda.empty_cache()
    if args.mhc:
        Xb, Gb = workloads.mhc_batch(device=dev)
        T = Xb.numel() // 16
        P = torch.empty_like(Xb)
        dX = torch.empty_like(Xb)
        tfused = time_device(lambda i: b4._fused_pass(Xb, Gb, P, dX), 20, dev)

        def sep(i):
            b4.forward(Xb, out=P)
            b4.backward(Gb, P=P, out=dX)

        tsep = time_device(sep, 20, dev)
        tf = time_device(lambda i: b4.forward(Xb, out=P), 20, dev)
        print(json.dumps({"mhc_bf16": True, "tokens": T, "fused_ms": tfused,
                          "fused_tokens_per_s": T / (tfused * 1e-3),
                          "fused_gbs": 128 * T / (tfused * 1e-3) / 1e9,
                          "separate_ms": tsep, "separate_tokens_per_s": T / (tsep * 1e-3),
                          "separate_gbs": 160 * T / (tsep * 1e-3) / 1e9,
                          "fwd_ms": tf, "fwd_gbs": 64 * T / (tf * 1e-3) / 1e9}), flush=True)
    if args.eot:
        run_eot(dev)
    if args.nxn:
        peak, peak_kind = hbm_peak()
        for n in (range(2, 9) if args.nxn_n is None else [args.nxn_n]):
            T = (args.nxn_mib << 18) // (n * n)  # MiB of fp32 X
            g = torch.Generator(device=dev).manual_seed(11 + n)
            X = torch.randn(T, n, n, device=dev, generator=g)
            G = torch.randn(T, n, n, device=dev, generator=g)
            P = torch.empty_like(X)
            dX = torch.empty_like(X)
            tf = time_device(lambda i: b4.forward_nxn(X, out=P), 10, dev)
            tb = time_device(lambda i: b4.backward_nxn(G, P=P, out=dX), 10, dev)
            fw_gbs = 8 * n * n * T / (tf * 1e-3) / 1e9
            bw_gbs = 12 * n * n * T / (tb * 1e-3) / 1e9
            print(json.dumps({"nxn": n, "tokens": T, "sigma": 1.0, "fwd_ms": tf, "bwd_ms": tb,
                              "fwd_tokens_per_s": T / (tf * 1e-3),
                              "bwd_tokens_per_s": T / (tb * 1e-3),
                              "fwd_gbs": fw_gbs, "bwd_gbs": bw_gbs,
                              "hbm_peak_gbs": peak, "peak_kind": peak_kind,
                              "fwd_frac": fw_gbs / peak, "bwd_frac": bw_gbs / peak}), flush=True)
            del X, G, P, dX
            torch.cuda.empty_cache()


def tf32_peak():
    """Dense TF32 tensor peak: the measured bf16 burst peak times the nominal
    TF32 / BF16 ratio (1.1 / 2.25 PFLOP/s)."""
    try:
        with open(PEAKS_PATH) as f:
            return float(json.load(f)["bf16_tflops"]) * 1.1 / 2.25, "measured bf16 x 1.1/2.25"
    except (OSError, KeyError, ValueError):
        return 1900.0 * 1.1 / 2.25, "fallback bf16 x 1.1/2.25"


def lib_tr_bytes(n, m, d):
    from birkhoff_projection_gb300 import lib

    return lib().eot_transport_workspace_bytes(n, m, d)


def run_eot(dev):
    """Streaming EOT lines: time per Sinkhorn iteration (two potential
    updates) at n = m = 65536, from the difference of 1 + K and 1 iterations
    (the one-off repacking of the clouds cancels)."""
    import torch

    from birkhoff_projection_gb300 import eot, workloads

    n, m = workloads.EOT_SIZES["bench"]
    eps = workloads.EOT_EPS
    peak, peak_kind = tf32_peak()
    for d in workloads.EOT_DIMS:
        X, Y, la, lb = workloads.eot_clouds(n, m, d, seed=0, device=dev)
        for passes in (eot.TF32, eot.TF32X3):
            ws = torch.empty(eot.workspace_bytes(n, m, d, passes), dtype=torch.uint8, device=dev)
            K = 10 if d <= 128 else 4
            f = torch.zeros(n, device=dev)
            g = torch.zeros(m, device=dev)
            t1 = time_device(lambda i: eot.sinkhorn(X, Y, la, lb, eps, 1, passes, f, g, ws), 5, dev)
            tk = time_device(lambda i: eot.sinkhorn(X, Y, la, lb, eps, 1 + K, passes, f, g, ws), 5, dev)
            it_ms = (tk - t1) / K
            upd_ms = it_ms / 2
            alg = 2.0 * n * m * d / (upd_ms * 1e-3) / 1e12
            tensor = alg * passes * (-(-d // 32) * 32) / d
            print(json.dumps({"eot": True, "n": n, "m": m, "d": d, "passes": passes, "eps": eps,
                              "ms_per_iteration": it_ms, "ms_per_update": upd_ms,
                              "algorithmic_tflops": alg, "tensor_tflops": tensor,
                              "tf32_peak_tflops": peak, "peak_kind": peak_kind,
                              "frac_of_tensor_peak": tensor / peak,
                              "ex2_per_update": n * m,
                              "f_finite": bool(torch.isfinite(f).all())}), flush=True)
            del ws
        # transport application (pi Y, row masses, gradient) at the potentials
        # of one f update
        f = eot.update(X, Y, torch.zeros(m, device=dev), lb, eps)
        g = torch.zeros(m, device=dev)
        ws = torch.empty(lib_tr_bytes(n, m, d), dtype=torch.uint8, device=dev)
        tt = time_device(lambda i: eot.transport(X, Y, f, g, la, lb, eps, want_grad=True,
                                                 workspace=ws), 5, dev)
        d_pad = -(-d // 32) * 32
        slices = -(-d_pad // 256)  # value coordinates per launch: 256
        alg = 4.0 * n * m * d / (tt * 1e-3) / 1e12
        # S = Q K^T runs as TF32 once per slice; P V as f16 (kind::f16) once
        s_flops = 2.0 * n * m * d_pad * slices
        pv_flops = 2.0 * n * m * d_pad
        f16_peak = peak * 2.25 / 1.1  # the measured bf16 rate; f16 is nominally the same
        t_ideal = (s_flops / peak + pv_flops / f16_peak) / 1e12 * 1e3
        print(json.dumps({"eot_transport": True, "n": n, "m": m, "d": d, "eps": eps,
                          "ms": tt, "algorithmic_tflops": alg, "value_slices": slices,
                          "s_dtype": "tf32", "pv_dtype": "f16",
                          "tf32_peak_tflops": peak, "f16_peak_tflops": f16_peak,
                          "roofline_ms": t_ideal, "frac_of_roofline": t_ideal / tt}), flush=True)
        del ws
        del X, Y
        torch.cuda.empty_cache()
    # Hessian-vector product (20 CG steps) at n = m = 16384, d = 64
    nh = 16384
    X, Y, la, lb = workloads.eot_clouds(nh, nh, 64, seed=0, device=dev)
    f, g = eot.sinkhorn(X, Y, la, lb, eps, 20)
    V = torch.randn(nh, 64, device=dev)
    ws = torch.empty(eot.lib().eot_hvp_workspace_bytes(nh, nh, 64), dtype=torch.uint8, device=dev)
    th = time_device(lambda i: eot.hvp(X, Y, f, g, la, lb, V, eps, cg_iters=20, workspace=ws), 3, dev)
    print(json.dumps({"eot_hvp": True, "n": nh, "m": nh, "d": 64, "eps": eps, "cg_iters_max": 20,
                      "ms": th, "plan_passes_max": 2 * 20 + 4,
                      "note": "CG stops on the device once converged; later passes exit at once"}),
          flush=True)


def run_eot_profile(args):
    """Three calls of one streaming EOT op, for an ncu capture of its kernel
    (update: lse_kernel; transport: transport_kernel, one launch per 256
    value coordinates; hvp: the plan passes of 5 CG steps)."""
    import torch

    from birkhoff_projection_gb300 import eot, workloads

    dev = torch.device("cuda:0")
    n = m = args.eot_n
    d = args.eot_d
    eps = workloads.EOT_EPS
    X, Y, la, lb = workloads.eot_clouds(n, m, d, seed=0, device=dev)
    g = torch.zeros(m, device=dev)
    if args.eot_profile == "update":
        ws = torch.empty(eot.workspace_bytes(n, m, d, eot.TF32), dtype=torch.uint8, device=dev)
        calls = [lambda: eot.update(X, Y, g, lb, eps, passes=eot.TF32, workspace=ws)] * 3
    elif args.eot_profile == "transport":
        f = eot.update(X, Y, g, lb, eps)
        ws = torch.empty(lib_tr_bytes(n, m, d), dtype=torch.uint8, device=dev)
        calls = [lambda: eot.transport(X, Y, f, g, la, lb, eps, workspace=ws)] * 3
    else:
        f, g = eot.sinkhorn(X, Y, la, lb, eps, 20)
        V = torch.randn(n, d, device=dev, generator=torch.Generator(device=dev).manual_seed(1))
        ws = torch.empty(eot.lib().eot_hvp_workspace_bytes(n, m, d), dtype=torch.uint8, device=dev)
        calls = [lambda: eot.hvp(X, Y, f, g, la, lb, V, eps, cg_iters=5, workspace=ws)] * 3
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    for c in calls:
        c()
    torch.cuda.synchronize(dev)
    print(json.dumps({"eot_profile": args.eot_profile, "n": n, "m": m, "d": d, "calls": len(calls),
                      "wall_s": time.perf_counter() - t0, "note": "profiling target, not a measurement"}),
          flush=True)


def ctypes_probe(b4, dev):
    """MUFU ex2 operations per second on this GPU (microbenchmark)."""
    import ctypes

    import torch

    L = b4.lib()
    out = (ctypes.c_float * 2)()
    nsm = torch.cuda.get_device_properties(dev).multi_processor_count
    s = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    L.birkhoff4_mufu_probe(out, nsm * 8, 256, s)  # warm-up
    if L.birkhoff4_mufu_probe(out, nsm * 8, 4096, s) != 0 or out[0] <= 0:
        return None
    return float(out[1]) / (float(out[0]) * 1e-3)


def bind_to_gpu_numa_node(dev) -> str:
    """Run this process on the host cores of the GPU's NUMA node, so pinned
    host buffers (first-touched here) sit next to the GPU's host link."""
    import torch

    try:
        p = torch.cuda.get_device_properties(dev)
        bus = "%04x:%02x:%02x.0" % (p.pci_domain_id, p.pci_bus_id, p.pci_device_id)
        node = int(open("/sys/bus/pci/devices/%s/numa_node" % bus).read())
        if node < 0:
            return "no NUMA affinity reported"
        cpus = open("/sys/devices/system/node/node%d/cpulist" % node).read().strip()
        sel = set()
        for part in cpus.split(","):
            a, _, b = part.partition("-")
            sel.update(range(int(a), int(b or a) + 1))
        os.sched_setaffinity(0, sel)
        return "node %d (%d cores)" % (node, len(sel))
    except (OSError, ValueError, AttributeError) as e:
        return "unbound (%s)" % type(e).__name__


def e2e_mapped(b4, X, G, dev, steps=3):
    """The step on host-resident tokens without copies
    (birkhoff4_forward_backward_mapped): the kernel reads pinned host X and dP
    and writes P and dX back to pinned host memory over the host link; every
    byte crosses the link inside the timed region."""
    import torch

    numa = bind_to_gpu_numa_node(dev)
    T = X.shape[0]
    Xh = torch.empty(X.shape, dtype=X.dtype, pin_memory=True)
    Gh = torch.empty(G.shape, dtype=G.dtype, pin_memory=True)
    Ph = torch.empty(X.shape, dtype=X.dtype, pin_memory=True)
    dXh = torch.empty(X.shape, dtype=X.dtype, pin_memory=True)
    Xh.copy_(X)
    Gh.copy_(G)
    b4.forward_backward_mapped(Xh, Gh, Ph, dXh, device=dev)
    torch.cuda.synchronize(dev)
    s = torch.cuda.current_stream(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    for _ in range(steps):
        b4.forward_backward_mapped(Xh, Gh, Ph, dXh, device=dev)
    e1.record(s)
    e1.synchronize()
    ms = e0.elapsed_time(e1) / steps
    nbytes = X.numel() * X.element_size()
    return {"value": T / (ms * 1e-3), "unit": "tokens/s", "h2d_bytes_per_step": 2 * nbytes,
            "d2h_bytes_per_step": 2 * nbytes, "ms_per_step": ms, "steps": steps,
            "host_link_gbs": 4 * nbytes / (ms * 1e-3) / 1e9,
            "api": "birkhoff4_forward_backward_mapped (zero copy, fused pass)", "numa": numa}


def host_link_ceiling(dev, nbytes=1 << 30, reps=3):
    """What the host link itself moves: copy-engine copies of `nbytes`
    between pinned host memory and the device, one direction at a time and
    both at once (two streams).  The e2e step moves as many bytes each way,
    so `both_gbs` is its ceiling."""
    import torch

    n = nbytes // 4
    a = torch.ones(n, dtype=torch.float32, pin_memory=True)
    b = torch.empty(n, dtype=torch.float32, pin_memory=True)
    da = torch.empty(n, dtype=torch.float32, device=dev)
    db = torch.ones(n, dtype=torch.float32, device=dev)
    s1, s2 = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    cur = torch.cuda.current_stream(dev)

    def timed(h2d, d2h):
        best = float("inf")
        for _ in range(reps):
            torch.cuda.synchronize(dev)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(cur)
            s1.wait_event(e0)
            s2.wait_event(e0)
            if h2d:
                with torch.cuda.stream(s1):
                    da.copy_(a, non_blocking=True)
            if d2h:
                with torch.cuda.stream(s2):
                    b.copy_(db, non_blocking=True)
            cur.wait_stream(s1)
            cur.wait_stream(s2)
            e1.record(cur)
            e1.synchronize()
            best = min(best, e0.elapsed_time(e1))
        return (int(h2d) + int(d2h)) * nbytes / (best * 1e-3) / 1e9

    return {"h2d_gbs": timed(True, False), "d2h_gbs": timed(False, True),
            "both_gbs": timed(True, True), "bytes_per_direction": nbytes,
            "method": "cudaMemcpyAsync pinned<->device, best of %d" % reps}


def e2e_host(b4, X, G, dev, steps=3, nstreams=4, chunk=1 << 21):
    """The same step through the C ABI with host buffers
    (birkhoff4_forward_backward_host): pinned host X and dP in, P and dX out,
    streamed in chunks over `nstreams` streams; every copy is inside the
    timed region."""
    import torch

    numa = bind_to_gpu_numa_node(dev)
    T = X.shape[0]
    Xh = torch.empty(X.shape, dtype=X.dtype, pin_memory=True)
    Gh = torch.empty(G.shape, dtype=G.dtype, pin_memory=True)
    Ph = torch.empty(X.shape, dtype=X.dtype, pin_memory=True)
    dXh = torch.empty(X.shape, dtype=X.dtype, pin_memory=True)
    Xh.copy_(X)
    Gh.copy_(G)
    streams = [torch.cuda.Stream(device=dev) for _ in range(nstreams)]
    ws = b4.host_workspace(dev, X.dtype, chunk_tokens=chunk, nstreams=nstreams)
    b4.forward_backward_host(Xh, Gh, Ph, dXh, device=dev, workspace=ws, streams=streams)
    torch.cuda.synchronize(dev)
    s = torch.cuda.current_stream(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    for _ in range(steps):
        b4.forward_backward_host(Xh, Gh, Ph, dXh, device=dev, workspace=ws, streams=streams)
    e1.record(s)
    e1.synchronize()
    ms = e0.elapsed_time(e1) / steps
    nbytes = X.numel() * X.element_size()
    return {"value": T / (ms * 1e-3), "unit": "tokens/s", "h2d_bytes_per_step": 2 * nbytes,
            "d2h_bytes_per_step": 2 * nbytes, "ms_per_step": ms, "steps": steps,
            "host_link_gbs": 4 * nbytes / (ms * 1e-3) / 1e9,
            "api": "birkhoff4_forward_backward_host (fused pass, chunks of %d tokens, %d streams)"
                   % (chunk, nstreams), "numa": numa}


if __name__ == "__main__":
    main()
