"""Benchmark: per-tensor FP8 E4M3 quantize -> scaled GEMM at M = N = K = 8192.

One step is one pass of the whole path over one batch: quantise A (8192^2
fp32, N(0,1) with 0.1% +-50 sigma outliers) and B (N(0,0.02), same outlier
rule) to E4M3 on the device (amax -> scale -> cast), then the scaled GEMM
with FP32 accumulation and BF16 output.  Inputs are generated once (seeded),
copied to HBM before timing.  `value` is 2*M*N*K / (time of one whole step),
in TFLOP/s.  The roofline object describes the GEMM kernel: `achieved` from
CUDA events around each GEMM launch over the timed steps, `achieved_isolated`
from the same kernel timed one step at a time before them.  By default
consecutive steps are pipelined: the HBM-bound quantisation of step i+1 runs
on a second stream while the tensor-bound GEMM of step i runs (codes and
scales double-buffered); every step still does all of its work, and the
serial schedule's time is reported beside it (--schedule serial times it
alone).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

With --impl reference the CPU oracle (test infrastructure under oracle/) is
timed on the host cores on a bounded sample of the same workload.  Under
torchrun each rank runs an independent replica on its own GPU (no data
exchange); rank 0 prints one JSON line.
"""

import argparse
import datetime
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

METRIC = ("FP8 E4M3 GEMM TFLOP/s (% of GB300 dense FP8 peak) at 8192³; "
          "quantize GB/s")
N_SIZE = 8192
FLOPS = 2.0 * N_SIZE ** 3
QUANT_BYTES_PER_ELEM = 9          # amax pass reads 4 B, cast pass reads 4 B + writes 1 B
E2E_REPEATS = 5                   # separate timed runs of the end-to-end loop (median reported)
GEMM_BYTES = 2 * N_SIZE * N_SIZE + 2 * N_SIZE * N_SIZE   # A, B codes + C bf16
FP8_OVER_BF16 = 4.5 / 2.25        # nominal dense FP8 : BF16 tensor ratio
NOMINAL_FP8_TFLOPS = 4500.0       # nominal dense FP8 tensor rate of one GB300
SUSTAINED_MIN_MS = 2000.0         # timed regions this long are rated against the sustained peak
NOMINAL_HBM_GBS = 8000.0          # GB300 HBM3e, nominal (~8 TB/s)
WORKLOAD = ("per-tensor E4M3 quantize(A), quantize(B) + scaled GEMM, "
            "M=N=K=8192, A~N(0,1), B~N(0,0.02), 0.1% +-50sigma outliers, seed 0")
WORKLOAD_DELAYED = ("per-tensor E4M3 delayed-scaling quantize(A), quantize(B) (scale from "
                    "the amax recorded at the previous step, one pass) + scaled GEMM, "
                    "M=N=K=8192, A~N(0,1), B~N(0,0.02), 0.1% +-50sigma outliers, seed 0")
GEMM_SOURCES = ["precision_linear_algebra_gb300/csrc/gemm.cu",
                "precision_linear_algebra_gb300/csrc/ptx.cuh"]
QUANT_SOURCES = ["precision_linear_algebra_gb300/csrc/quantize.cu"]


def _dist_env():
    return int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")), \
        int(os.environ.get("LOCAL_RANK", "0"))


def max_over_ranks(x, device=None):
    """max of a per-rank float over all ranks (identity when not distributed).

    The only collective of the replica benchmark: each rank times its own
    replica and the job's time is the slowest rank's."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return p["hbm_gbs"], p["bf16_tflops"], p.get("bf16_tflops_sustained"), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


def _src_hash(paths):
    """Hash of the sources' code: // comments and blank lines are left out,
    so that an edit of comments alone does not retire a profile."""
    h = hashlib.sha256()
    for p in paths:
        with open(os.path.join(ROOT, p), encoding="utf-8") as f:
            for line in f:
                code = line.split("//", 1)[0].rstrip()
                if code:
                    h.update(code.encode("utf-8") + b"\n")
    return h.hexdigest()[:16]


def _profile_traffic(name, paths):
    """dram bytes per launch recorded in profiles/<name>.md, if the kernel
    source is unchanged since the capture (its hash is stored there)."""
    path = os.path.join(ROOT, "profiles", name + ".md")
    try:
        fields = {}
        for line in open(path):
            if line.startswith("<!--") and "=" in line:
                for kv in line.strip("<!-> \n").split(";"):
                    if "=" in kv:
                        k, v = kv.split("=", 1)
                        fields[k.strip()] = v.strip()
        if fields.get("source_sha256") == _src_hash(paths):
            return float(fields["traffic_bytes_per_launch"])
    except Exception:
        pass
    return None


def _parse_nvsmi_time(ts):
    """Epoch seconds of an nvidia-smi timestamp ("2026/12/03 07:25:22.123",
    local time), or None."""
    try:
        return datetime.datetime.strptime(ts, "%Y/%m/%d %H:%M:%S.%f").timestamp()
    except ValueError:
        return None


_CLOCK_REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]


def _summarise_clocks(rows, window=None):
    """Median SM clock, maximum clock and active reasons of sampled rows
    [time, index, sm, max, power, active, hw, hw_thermal, sw_thermal,
    sw_power_cap].  With window = (t0, t1) (epoch seconds) only the samples
    taken inside it count; when none is (a region shorter than the sampling
    interval) all samples do, and the summary says so."""
    sel = rows
    in_region = None
    if window is not None:
        t0, t1 = window
        sel = [r for r in rows if r[0] is not None and t0 - 0.05 <= r[0] <= t1 + 0.05]
        in_region = len(sel)
        if not sel:
            sel = rows
    sm = [float(r[2]) for r in sel if r[2].replace(".", "").isdigit()]
    mx = [float(r[3]) for r in sel if r[3].replace(".", "").isdigit()]
    reasons = sorted({_CLOCK_REASONS[i] for r in sel for i in range(4)
                      if r[6 + i].lower() == "active"})
    out = {"sm_mhz": statistics.median(sm) if sm else None,
           "sm_max_mhz": max(mx) if mx else None,
           "reasons": reasons, "samples": len(sel)}
    if window is not None:
        out["samples_in_timed_region"] = in_region
        out["window"] = ("timed region" if in_region else
                         "whole sampling period (the timed region was shorter than "
                         "the 100 ms sampling interval)")
    return out


class ClockSampler:
    """nvidia-smi clocks/throttle reasons sampled around the timed region."""
    QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.rows = []
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.QUERY,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 10:
                self.rows.append([_parse_nvsmi_time(parts[0])] + parts[1:])

    def stop(self, window=None):
        """Stop sampling; summarise the samples inside window = (t0, t1)
        (epoch seconds), if given."""
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        return _summarise_clocks(self.rows, window)


def _per_op(W, phases, alu_peak, fp8_peak):
    """Each GEMM of a multi-GEMM step on its own: mean CUDA-event time of its
    launches over the timed steps, TFLOP/s and fractions of the ALU and FP8
    peaks (launches are recorded in step order, one per operation)."""
    ops = W.get("per_op")
    durs = (phases.get("launches") or {}).get("gemm") or []
    if not ops or not durs or len(durs) % len(ops):
        return None
    out = {}
    for i, (name, flops) in enumerate(ops):
        ms = statistics.mean(durs[i::len(ops)])
        tf = flops / (ms * 1e-3) / 1e12
        out[name] = {"ms": ms, "tflops": tf, "frac": tf / alu_peak,
                     "frac_of_fp8_peak": tf / fp8_peak}
    return out


def _alu_promotion_peak(torch, dev):
    """Ceiling of the 32x32 block-scaled GEMM on the CUDA cores, in GEMM
    TFLOP/s: each output needs one FP32 FMA per 32-wide K block (64 GEMM
    FLOP per FMA), at 128 FP32 FMAs per SM per clock (four sub-partitions of
    32 lanes; a packed fma.rn.f32x2 issues at half the rate, so it does not
    raise this), on every SM at the maximum SM clock."""
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    mhz = None
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            mhz = float(json.load(f).get("sm_max_mhz"))
    except Exception:
        pass
    src = "MEASURED_PEAKS.json sm_max_mhz"
    if not mhz:
        mhz, src = 2070.0, "the maximum SM clock of the part"
    peak = 64.0 * 128 * sms * mhz * 1e6 / 1e12
    return peak, ("CUDA-core promotion ceiling: 128 FP32 FMA per SM per clock x %d SMs x "
                  "%.0f MHz (%s) x 64 GEMM FLOP per FMA (one FMA per output per 32-wide "
                  "K block); the tensor-core work of the same GEMM takes half as long"
                  % (sms, mhz, src))


def _peak_regime(ms_total, clocks, have_sustained, graph_replayed):
    """Which measured peak rates the dominant kernel of a timed region:
    (True, why) for the sustained figure -- it comes from a seconds-long
    loop, so it applies only to a timed region that long -- else (False,
    why) for the burst figure.  Power-capped clocks in a short region do not
    switch the figure (they are reported in the clocks record)."""
    if graph_replayed or not have_sustained:
        return False, "burst: %s" % ("CUDA graph replay" if graph_replayed
                                     else "no sustained figure measured")
    if ms_total >= SUSTAINED_MIN_MS:
        return True, "sustained: timed region %.0f ms >= %.0f ms" % (ms_total, SUSTAINED_MIN_MS)
    capped = "sw_power_cap" in (clocks.get("reasons") or [])
    return False, "burst: timed region %.0f ms%s" % (
        ms_total, " (sw_power_cap active, median SM clock %s MHz)" % clocks.get("sm_mhz")
        if capped else ", clocks not power-capped")


def _median_min_per_step(xs, steps):
    """[median, min] over the steps of the per-step sums of a phase's
    consecutive interval durations (xs holds steps x k of them), or None."""
    if not xs or steps <= 0 or len(xs) % steps:
        return None
    k = len(xs) // steps
    per_step = [sum(xs[i * k:(i + 1) * k]) for i in range(steps)]
    return [statistics.median(per_step), min(per_step)]


_SLOWDOWNS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown")


def _clocks_invalid(clocks):
    """True for a timed region that saw a hardware or thermal slowdown, or
    whose median SM clock sat below 3/4 of the maximum with no reason active
    (a leftover clock lock).  The power cap alone is normal under a dense
    GEMM and keeps the run valid."""
    reasons = clocks.get("reasons") or []
    if any(r in _SLOWDOWNS for r in reasons):
        return True
    sm, mx = clocks.get("sm_mhz"), clocks.get("sm_max_mhz")
    return bool(not reasons and sm and mx and sm < 0.75 * mx)


# ------------------------------------------------------------ CPU oracle arm
def _oracle_inputs(seed=0):
    from precision_linear_algebra_gb300 import workloads
    return workloads.square_outliers(N_SIZE, seed=seed)


def _oracle_sample(A, B, rows_q, rows_g, cols_g):
    """Time the oracle on a bounded sample of one step; return the estimated
    time of a full step (s) and the wall time spent.

    Sample: per-tensor quantisation of the first rows_q rows of A and of B,
    then the GEMM outputs C[0:rows_g, 0:cols_g] (full K) from those codes."""
    import numpy as np
    import oracle
    t0 = time.perf_counter()
    qa, _, sa = oracle.quantize_pertensor(A[:rows_q])
    qb, _, sb = oracle.quantize_pertensor(B[:rows_q])
    t_q = time.perf_counter() - t0
    rg = np.arange(rows_g) % rows_q
    cg = np.arange(cols_g) % rows_q
    t1 = time.perf_counter()
    oracle.gemm_pertensor(qa, qb, sa, sb, rows=rg, cols=cg)
    t_g = time.perf_counter() - t1
    est = t_q * (N_SIZE / rows_q) + t_g * (N_SIZE * N_SIZE / (rows_g * cols_g))
    return est, t_q + t_g


def run_reference(args):
    world, rank, _ = _dist_env()
    if rank != 0:
        return
    threads = os.cpu_count() or 1
    # One step = quantise rows_q rows of A and of B, then rows_g rows of the
    # GEMM; sized so that warm-up + steps stay within a few minutes.
    A, B = _oracle_inputs()
    budget_s = 150.0
    per_step = budget_s / max(1, args.steps + args.warmup)
    rows_q = int(min(N_SIZE, max(8, 400 * per_step)))
    rows_g = int(min(N_SIZE, max(1, 128 * per_step)))
    cols_g = int(min(N_SIZE, max(8, 1024 * per_step)))
    for _ in range(args.warmup):
        _oracle_sample(A, B, rows_q, rows_g, cols_g)
    ests, walls = [], []
    for _ in range(args.steps):
        e, w = _oracle_sample(A, B, rows_q, rows_g, cols_g)
        ests.append(e)
        walls.append(w)
    est = statistics.median(ests)
    value = FLOPS / est / 1e12
    sample = ("each step: oracle quantize of %d rows of A and of B (of 8192) and oracle "
              "GEMM of a %d x %d output block (K 8192); step time scaled to the full "
              "8192^3 step by element and output counts" % (rows_q, rows_g, cols_g))
    # A step of this arm is the bounded sample: ms_per_step is its wall
    # time; the full-step estimate behind `value` is reported beside it.
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": statistics.median(walls) * 1e3,
            "ms_per_full_step_estimate": est * 1e3,
            "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD,
                       "parallelism": "replicas" if world > 1 else "single GPU",
                       "M": N_SIZE, "N": N_SIZE, "K": N_SIZE,
                       "l2": "inputs 2 x 268 MB fp32 > 129 MB L2; no flush"},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads,
                             "kind": "oracle", "cpu_model": _cpu_model(), "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def _timed(f, *a, **k):
    t0 = time.perf_counter()
    out = f(*a, **k)
    return out, time.perf_counter() - t0


def _oracle_sample_workload(workload, linears=""):
    """Time the oracle on a bounded sample of one step of `workload`; return
    (estimated seconds for the full step, wall seconds timed, description).
    Quantisation is scaled by element counts and GEMMs by output counts (the
    oracle's cost per output is proportional to K)."""
    import numpy as np
    import oracle
    from precision_linear_algebra_gb300 import workloads
    if workload in ("pertensor8192", "pertensor8192_delayed"):
        A, B = _oracle_inputs()
        if workload == "pertensor8192":
            est, wall = _oracle_sample(A, B, 4096, 1024, 4096)
            return est, wall, ("oracle quantize of 4096 rows of A and of B + oracle GEMM of a "
                               "1024 x 4096 output block of the 8192^3 workload")
        rq, rg, cg = 4096, 1024, 4096
        prev_a, prev_b = oracle.amax_fp32(A[:rq]), oracle.amax_fp32(B[:rq])
        (qa, _, sa), t1 = _timed(oracle.quantize_pertensor_delayed, A[:rq], prev_a)
        (qb, _, sb), t2 = _timed(oracle.quantize_pertensor_delayed, B[:rq], prev_b)
        _, t3 = _timed(oracle.gemm_pertensor, qa, qb, sa, sb, rows=np.arange(rg) % rq,
                       cols=np.arange(cg) % rq)
        est = (t1 + t2) * (N_SIZE / rq) + t3 * (N_SIZE * N_SIZE / (rg * cg))
        return est, t1 + t2 + t3, ("oracle delayed-scaling quantize of 4096 rows of A and of B "
                                   "+ oracle GEMM of a 1024 x 4096 output block of the 8192^3 "
                                   "workload")
    if workload.startswith("square"):
        n = int(workload[len("square"):])
        A, B = workloads.square(n, seed=0)
        rq = n if n <= 1024 else 2048
        rg = n if n <= 1024 else 1024
        fmt = _SQUARE_OPTS["fmt"]
        (qa, _, sa), t1 = _timed(oracle.quantize_pertensor, A[:rq], fmt)
        (qb, _, sb), t2 = _timed(oracle.quantize_pertensor, B, fmt)
        _, t3 = _timed(oracle.gemm_pertensor, qa, qb, sa, sb, rows=np.arange(rg),
                       a_fmt=fmt, b_fmt=fmt)
        est = t1 * (n / rq) + t2 + t3 * (n / rg)
        if rq == n and rg == n:
            desc = "oracle quantize of A and B + oracle GEMM, the whole %d^3 step" % n
        else:
            desc = ("oracle quantize of %d rows of A and all of B + oracle GEMM of %d output "
                    "rows (of %d)" % (rq, rg, n))
        return est, t1 + t2 + t3, desc
    if workload == "blockscaled":
        names = linears.split(",") if linears else ["qkv", "attn_out", "gate_up", "down"]
        est = wall = 0.0
        for name in names:
            X, W = workloads.transformer_linear(name, seed=0)
            (M, K), N = X.shape, W.shape[0]
            (qx, sx), t1 = _timed(oracle.quantize_blockwise_32x32, X[:1024])
            (qw, sw), t2 = _timed(oracle.quantize_blockwise_32x32, W[:1024])
            _, t3 = _timed(oracle.gemm_blockscaled_32x32, qx, qw, sx, sw,
                           rows=np.arange(256), cols=np.arange(1024))
            est += t1 * (M / 1024) + t2 * (N / 1024) + t3 * (M * N / (256 * 1024))
            wall += t1 + t2 + t3
            del X, W
        return est, wall, ("per linear: oracle block quantize of 1024 rows of the activations "
                           "and of the weights + oracle block-scaled GEMM of a 256 x 1024 output "
                           "block (full K)")
    if workload == "grouped":
        counts, offs, X, W = workloads.moe_layer(seed=0)
        E, N, K = W.shape
        Mt = int(offs[-1])
        (qx, _, sx), t1 = _timed(oracle.quantize_pertensor, X[:4096])
        (qw, _, sw), t2 = _timed(oracle.quantize_pertensor, W[0][:4096])
        _, t3 = _timed(oracle.gemm_pertensor, qx, qw, sx, sw, rows=np.arange(1024),
                       cols=np.arange(4096))
        est = (t1 + t2) * ((Mt * K + E * N * K) / (8192 * K)) + t3 * (Mt * N / (1024 * 4096))
        return est, t1 + t2 + t3, ("oracle per-tensor quantize of 4096 activation rows and "
                                   "4096 weight rows + oracle GEMM of a 1024 x 4096 output "
                                   "block of expert 0 (K 4096)")
    if workload == "attention":
        batch, heads, seq, hd, sampled = 2, 64, 2048, 128, 16
        E = batch * heads
        g = np.random.default_rng(0)
        wall = 0.0
        for _ in range(sampled):
            Q = workloads.normal(g, (seq, hd))
            Kh = workloads.normal(g, (seq, hd))
            P = g.random((seq, seq), dtype=np.float32) / np.float32(seq)
            Vt = workloads.normal(g, (hd, seq))
            qQ, _, sQ = oracle.quantize_pertensor(Q)
            qK, _, sK = oracle.quantize_pertensor(Kh)
            qP, _, sP = oracle.quantize_pertensor(P)
            qV, _, sV = oracle.quantize_pertensor(Vt)
            _, t1 = _timed(oracle.gemm_pertensor, qQ, qK, sQ, sK)
            _, t2 = _timed(oracle.gemm_pertensor, qP, qV, sP, sV)
            wall += t1 + t2
        return wall * E / sampled, wall, (
            "oracle GEMMs of %d heads (of %d): Q K^T (2048 x 2048, K 128) and P V (2048 x 128, "
            "K 2048); set-up quantisation not timed" % (sampled, E))
    raise ValueError(workload)


def _cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo), or None."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return None


def _cpu_baseline_subprocess(flops, workload="pertensor8192", linears=""):
    """The oracle on the host cores, run in a child process so that its BLAS
    threads are set explicitly; about 10-30 s of CPU work on a sample of the
    workload's step, scaled to the whole step."""
    threads = os.cpu_count() or 1
    env = dict(os.environ, OPENBLAS_NUM_THREADS=str(threads), OMP_NUM_THREADS=str(threads),
               MKL_NUM_THREADS=str(threads))
    code = ("import json,sys; sys.path.insert(0, %r); import bench; "
            "bench._SQUARE_OPTS.update(fmt=%r); "
            "e, w, d = bench._oracle_sample_workload(%r, %r); print(json.dumps([e, w, d]))"
            % (ROOT, _SQUARE_OPTS["fmt"], workload, linears))
    try:
        out = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True,
                             text=True, timeout=600)
        est, wall, desc = json.loads(out.stdout.strip().splitlines()[-1])
    except Exception as exc:  # reported, not fatal
        return {"value": None, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                "sample": "failed: %s" % exc}
    return {"value": flops / est / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "cpu_model": _cpu_model(), "ms_per_step": est * 1e3,
            "sample": "%s (%.1f s wall), scaled to one full step by element and output counts"
                      % (desc, wall)}


# ------------------------------------------------------------------ GPU arm
class _Phases:
    """CUDA events around the phases of a step ('quant', 'gemm'), on the
    launching stream; durations are summed per phase per step."""

    def __init__(self, torch, stream):
        self.torch, self.stream = torch, stream
        self.events = []
        self.on = False

    def mark(self, phase, stream=None):
        """Record an event on `stream` (default: the launching stream); call
        once before and once after the phase's launches."""
        if self.on:
            e = self.torch.cuda.Event(enable_timing=True)
            e.record(self.stream if stream is None else stream)
            self.events.append((phase, e))

    def collect(self):
        out = {}
        for ph, ds in self.durations().items():
            out[ph] = sum(ds)
        self.events = []
        return out

    def durations(self):
        """Each bracketed interval's duration (ms), per phase, in order."""
        out = {}
        for (ph, e0), (_, e1) in zip(self.events[0::2], self.events[1::2]):
            out.setdefault(ph, []).append(e0.elapsed_time(e1))
        return out


def busy_warmup(step, torch, seconds):
    """Run untimed steps for at least `seconds` of wall time (synchronising
    every few steps), so that the timed region starts at settled clocks."""
    t0 = time.time()
    while time.time() - t0 < seconds:
        for _ in range(4):
            step()
        torch.cuda.synchronize()


def _workload_pertensor(fl, torch, dev, sptr, ph, delayed=False):
    """The 8192^3 step.  delayed=True quantises each operand in one pass with
    the scale of the amax it recorded at the previous step (delayed scaling);
    the two amax words of each operand alternate between steps."""
    from precision_linear_algebra_gb300 import workloads
    A_np, B_np = workloads.square_outliers(N_SIZE, seed=0)
    A = torch.from_numpy(A_np).to(dev)
    B = torch.from_numpy(B_np).to(dev)
    qa = torch.empty((N_SIZE, N_SIZE), dtype=torch.uint8, device=dev)
    qb = torch.empty_like(qa)
    amax = torch.empty(2, dtype=torch.float32, device=dev)
    scale = torch.empty(2, dtype=torch.float32, device=dev)
    C = torch.empty((N_SIZE, N_SIZE), dtype=torch.bfloat16, device=dev)
    P = lambda t, i=0: t.data_ptr() + i * t.element_size()
    # amax history for delayed scaling: hist[2 * operand + parity]
    hist = torch.empty(4, dtype=torch.float32, device=dev)

    def quant(x, q, amax_t, amax_i, scale_t, scale_i, s, operand, parity):
        if delayed:
            fl.fp8_quantize_pertensor_delayed(
                P(x), N_SIZE, N_SIZE, N_SIZE, P(q), N_SIZE, P(hist, 2 * operand + (parity ^ 1)),
                P(hist, 2 * operand + parity), P(scale_t, scale_i), 0, s)
        else:
            fl.fp8_quantize_pertensor(P(x), N_SIZE, N_SIZE, N_SIZE, P(q), N_SIZE,
                                      P(amax_t, amax_i), P(scale_t, scale_i), s)

    if delayed:
        # seed the history with the current amax of each operand
        for operand, x in enumerate((A, B)):
            for parity in (0, 1):
                fl.fp8_quantize_pertensor(P(x), N_SIZE, N_SIZE, N_SIZE, P(qa), N_SIZE,
                                          P(hist, 2 * operand + parity), P(scale, 0), sptr)
    counter = [0]

    def step():
        parity = counter[0] & 1
        counter[0] += 1
        ph.mark("quant")
        quant(A, qa, amax, 0, scale, 0, sptr, 0, parity)
        quant(B, qb, amax, 1, scale, 1, sptr, 1, parity)
        ph.mark("quant")
        ph.mark("gemm")
        fl.fp8_gemm(P(qa), N_SIZE, P(qb), N_SIZE, P(C), N_SIZE, N_SIZE, N_SIZE, N_SIZE,
                    P(scale, 0), P(scale, 1), sptr)
        ph.mark("gemm")

    # Pipelined schedule: step i+1's quantisation (HBM-bound) runs on its own
    # stream while step i's GEMM (tensor-bound) runs on another.  Codes and
    # scales are double-buffered; events order quantize(i) before GEMM(i)
    # and GEMM(i) before quantize(i+2), which reuses its buffers.
    main = torch.cuda.current_stream(dev)
    sq, sg = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    qa2 = [qa, torch.empty_like(qa)]
    qb2 = [qb, torch.empty_like(qb)]
    amax2 = torch.empty(4, dtype=torch.float32, device=dev)
    scale2 = torch.empty(4, dtype=torch.float32, device=dev)
    qdone = [torch.cuda.Event(), torch.cuda.Event()]
    gdone = [torch.cuda.Event(), torch.cuda.Event()]

    def pbegin():
        for e in qdone + gdone:
            e.record(main)
        sq.wait_stream(main)
        sg.wait_stream(main)

    def pstep(i):
        b = i & 1
        sq.wait_event(gdone[b])
        ph.mark("quant", sq)
        quant(A, qa2[b], amax2, 2 * b, scale2, 2 * b, sq.cuda_stream, 0, b)
        quant(B, qb2[b], amax2, 2 * b + 1, scale2, 2 * b + 1, sq.cuda_stream, 1, b)
        ph.mark("quant", sq)
        qdone[b].record(sq)
        sg.wait_event(qdone[b])
        ph.mark("gemm", sg)
        fl.fp8_gemm(P(qa2[b]), N_SIZE, P(qb2[b]), N_SIZE, P(C), N_SIZE, N_SIZE, N_SIZE,
                    N_SIZE, P(scale2, 2 * b), P(scale2, 2 * b + 1), sg.cuda_stream)
        ph.mark("gemm", sg)
        gdone[b].record(sg)

    def pend():
        main.wait_stream(sq)
        main.wait_stream(sg)

    # Pipelined end to end: step i's fp32 inputs come from pinned host memory
    # (A and B on two copy streams), its C goes back to a pinned host buffer
    # on a third; host->device copies of step i+1, compute of step i and the
    # device->host copy of step i-1 overlap.  Device inputs and host outputs
    # are double-buffered; events keep every buffer from being overwritten
    # while still in use.
    e2e = {}

    def ebegin(host_inputs, host_outputs2):
        A_h, B_h = host_inputs
        C_h2 = host_outputs2[0]
        if not e2e:
            e2e.update(A=[A, torch.empty_like(A)], B=[B, torch.empty_like(B)],
                       C=[C, torch.empty_like(C)],
                       sa=torch.cuda.Stream(dev), sb=torch.cuda.Stream(dev),
                       so=torch.cuda.Stream(dev),
                       loaded=[torch.cuda.Event(), torch.cuda.Event()],
                       quantized=[torch.cuda.Event(), torch.cuda.Event()],
                       computed=[torch.cuda.Event(), torch.cuda.Event()],
                       stored=[torch.cuda.Event(), torch.cuda.Event()])
        e2e.update(A_h=A_h, B_h=B_h, C_h=C_h2)
        for k in ("loaded", "quantized", "computed", "stored"):
            for ev in e2e[k]:
                ev.record(main)
        for st in (e2e["sa"], e2e["sb"], e2e["so"], sq, sg):
            st.wait_stream(main)

    def estep(i):
        b = i & 1
        E = e2e
        # inputs: buffer b is free once quantize(i-2) has read it
        E["sa"].wait_event(E["quantized"][b])
        E["sb"].wait_event(E["quantized"][b])
        with torch.cuda.stream(E["sa"]):
            E["A"][b].copy_(E["A_h"], non_blocking=True)
        with torch.cuda.stream(E["sb"]):
            E["B"][b].copy_(E["B_h"], non_blocking=True)
        ev_a, ev_b = torch.cuda.Event(), torch.cuda.Event()
        ev_a.record(E["sa"])
        ev_b.record(E["sb"])
        # quantize (codes double-buffered as in the device-resident pipeline)
        sq.wait_event(ev_a)
        sq.wait_event(ev_b)
        sq.wait_event(gdone[b])
        quant(E["A"][b], qa2[b], amax2, 2 * b, scale2, 2 * b, sq.cuda_stream, 0, b)
        quant(E["B"][b], qb2[b], amax2, 2 * b + 1, scale2, 2 * b + 1, sq.cuda_stream, 1, b)
        E["quantized"][b].record(sq)
        qdone[b].record(sq)
        # GEMM into C[b] once the D2H of step i-2 has drained it
        sg.wait_event(qdone[b])
        sg.wait_event(E["stored"][b])
        fl.fp8_gemm(P(qa2[b]), N_SIZE, P(qb2[b]), N_SIZE, P(E["C"][b]), N_SIZE, N_SIZE,
                    N_SIZE, N_SIZE, P(scale2, 2 * b), P(scale2, 2 * b + 1), sg.cuda_stream)
        gdone[b].record(sg)
        E["computed"][b].record(sg)
        # result back to the host
        E["so"].wait_event(E["computed"][b])
        with torch.cuda.stream(E["so"]):
            E["C_h"][b].copy_(E["C"][b], non_blocking=True)
        E["stored"][b].record(E["so"])

    def eend():
        for st in (e2e["sa"], e2e["sb"], e2e["so"], sq, sg):
            main.wait_stream(st)

    def crosscheck(iters=20):
        """cuBLASLt through torch._scaled_mm on the same codes and scales
        (a library comparison point, not part of the step): its TFLOP/s
        over `iters` back-to-back calls, this library's GEMM timed the same
        way beside it, and the fraction of cuBLASLt's BF16 outputs equal to
        this library's bit for bit."""
        step()
        torch.cuda.synchronize()
        a8 = qa.view(torch.float8_e4m3fn)
        b8 = qb.view(torch.float8_e4m3fn).t()          # [K][N], column-major
        sa_t, sb_t = scale[0:1], scale[1:2]
        ref = torch._scaled_mm(a8, b8, sa_t, sb_t, out_dtype=torch.bfloat16)
        for _ in range(3):
            torch._scaled_mm(a8, b8, sa_t, sb_t, out_dtype=torch.bfloat16)
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(main)
        for _ in range(iters):
            torch._scaled_mm(a8, b8, sa_t, sb_t, out_dtype=torch.bfloat16)
        t1.record(main)
        torch.cuda.synchronize()
        ms = t0.elapsed_time(t1) / iters
        same = (ref.view(torch.int16) == C.view(torch.int16)).float().mean().item()

        def ours():
            fl.fp8_gemm(P(qa), N_SIZE, P(qb), N_SIZE, P(C), N_SIZE, N_SIZE, N_SIZE,
                        N_SIZE, P(scale, 0), P(scale, 1), sptr)
        for _ in range(3):
            ours()
        t0.record(main)
        for _ in range(iters):
            ours()
        t1.record(main)
        torch.cuda.synchronize()
        ms_ours = t0.elapsed_time(t1) / iters
        return {"what": "torch._scaled_mm (cuBLASLt) FP8 E4M3, per-tensor scales, BF16 out, "
                        "same codes; library comparison point, not a target",
                "tflops": FLOPS / (ms * 1e-3) / 1e12, "ms": ms, "iters": iters,
                "bitwise_equal_fraction": same,
                "this_library_back_to_back_ms": ms_ours,
                "this_library_back_to_back_tflops": FLOPS / (ms_ours * 1e-3) / 1e12}

    return dict(step=step, pipeline=(pbegin, pstep, pend), e2e_pipeline=(ebegin, estep, eend),
                crosscheck=None if delayed else crosscheck,
                flops=FLOPS, launches=3 if delayed else 5,
                workload=WORKLOAD_DELAYED if delayed else WORKLOAD,
                quant_bytes_per_elem=5 if delayed else QUANT_BYTES_PER_ELEM,
                config={"M": N_SIZE, "N": N_SIZE, "K": N_SIZE,
                        "l2": "inputs 2 x 268 MB fp32 > 129 MB L2; no flush"},
                inputs=[(A, A_np), (B, B_np)], outputs=[C],
                quant_elems=2 * N_SIZE * N_SIZE, gemm_label="gemm_e4m3_pair_kernel<false>",
                gemm_bytes=GEMM_BYTES, profile=("gemm_e4m3_pertensor_8192", GEMM_SOURCES),
                qprofile=(("quantize_pertensor_delayed_8192" if delayed
                           else "quantize_pertensor_8192"), QUANT_SOURCES))


# Options of the square workloads (set from the command line).
_SQUARE_OPTS = {"fmt": "e4m3", "gemm_variant": 0}
_FMT_CODES = {"e4m3": 0, "e5m2": 1}


def _workload_square(n):
    """Per-tensor quantize(A), quantize(B) + GEMM at M = N = K = n (N(0,1)
    inputs), in the format --fmt.  The small sizes are launch-bound, so the
    timed step replays one CUDA graph holding the step's launches."""

    def build(fl, torch, dev, sptr, ph):
        f = _FMT_CODES[_SQUARE_OPTS["fmt"]]
        from precision_linear_algebra_gb300 import workloads
        A_np, B_np = workloads.square(n, seed=0)
        A = torch.from_numpy(A_np).to(dev)
        B = torch.from_numpy(B_np).to(dev)
        qa = torch.empty((n, n), dtype=torch.uint8, device=dev)
        qb = torch.empty_like(qa)
        amax = torch.empty(2, dtype=torch.float32, device=dev)
        scale = torch.empty(2, dtype=torch.float32, device=dev)
        C = torch.empty((n, n), dtype=torch.bfloat16, device=dev)
        P = lambda t, i=0: t.data_ptr() + i * t.element_size()

        def quant(stream_ptr):
            fl.fp8_quantize_pertensor_ex(P(A), n, n, n, P(qa), n, P(amax, 0), P(scale, 0),
                                         f, stream_ptr)
            fl.fp8_quantize_pertensor_ex(P(B), n, n, n, P(qb), n, P(amax, 1), P(scale, 1),
                                         f, stream_ptr)

        def gemm(stream_ptr):
            fl.fp8_gemm_ex(P(qa), n, P(qb), n, P(C), n, n, n, n, P(scale, 0), P(scale, 1),
                           f, f, stream_ptr)

        def launches(stream_ptr):
            quant(stream_ptr)
            gemm(stream_ptr)

        def launches_forked(main_s, side_s):
            # The two quantisations are independent: B's runs on a side
            # stream forked from and joined back into the main one, so the
            # captured graph holds them as parallel branches.
            fork = torch.cuda.Event()
            fork.record(main_s)
            side_s.wait_event(fork)
            fl.fp8_quantize_pertensor_ex(P(A), n, n, n, P(qa), n, P(amax, 0), P(scale, 0),
                                         f, main_s.cuda_stream)
            fl.fp8_quantize_pertensor_ex(P(B), n, n, n, P(qb), n, P(amax, 1), P(scale, 1),
                                         f, side_s.cuda_stream)
            join = torch.cuda.Event()
            join.record(side_s)
            main_s.wait_event(join)
            gemm(main_s.cuda_stream)

        def step():
            ph.mark("quant")
            quant(sptr)
            ph.mark("quant")
            ph.mark("gemm")
            gemm(sptr)
            ph.mark("gemm")

        # One step captured as a CUDA graph (after a warm-up on a side stream,
        # so that one-time library set-up happens outside the capture).
        cap = torch.cuda.Stream(dev)
        cap.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(cap):
            launches(cap.cuda_stream)
        torch.cuda.current_stream(dev).wait_stream(cap)
        torch.cuda.synchronize()
        side = torch.cuda.Stream(dev)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=cap):
            launches_forked(cap, side)
        torch.cuda.synchronize()
        # Kernels per step: tensors of at most 512K floats take the one-launch
        # quantiser, larger ones amax + cast.
        per_operand = 1 if n * n <= (1 << 19) else 2
        return dict(step=step, graph=graph, flops=2.0 * n ** 3, launches=2 * per_operand + 1,
                    workload=("per-tensor %s quantize(A), quantize(B) + scaled GEMM, "
                              "M=N=K=%d, A, B ~ N(0,1), seed 0; one CUDA graph per step, the two "
                              "quantisations as parallel branches"
                              % (_SQUARE_OPTS["fmt"].upper(), n)),
                    config={"M": n, "N": n, "K": n, "format": _SQUARE_OPTS["fmt"],
                            "gemm_variant": _SQUARE_OPTS["gemm_variant"],
                            "l2": ("L2-resident inputs (%d KB fp32); no flush" % (8 * n * n // 1024)
                                   if 8 * n * n < 64 << 20 else
                                   "inputs 2 x %d MB fp32; no flush" % (4 * n * n >> 20))},
                    inputs=[(A, A_np), (B, B_np)], outputs=[C], quant_elems=2 * n * n,
                    gemm_label=("gemm_e4m3_kernel<256,4,false>" if _SQUARE_OPTS["gemm_variant"] == 1
                                else "gemm_e4m3_pair_kernel<false>"),
                    gemm_bytes=4 * n * n,
                    profile=("gemm_e4m3_square_%d" % n, GEMM_SOURCES),
                    qprofile=("quantize_square_%d" % n, QUANT_SOURCES))
    return build


def _workload_blockscaled(fl, torch, dev, sptr, ph, linears=("qkv", "attn_out", "gate_up", "down")):
    from precision_linear_algebra_gb300 import workloads
    items = []
    flops = 0.0
    qelems = 0
    gbytes = 0
    for name in linears:
        X_np, W_np = workloads.transformer_linear(name, seed=0)
        M, K = X_np.shape
        N = W_np.shape[0]
        X = torch.from_numpy(X_np).to(dev)
        W = torch.from_numpy(W_np).to(dev)
        qx = torch.empty((M, K), dtype=torch.uint8, device=dev)
        qw = torch.empty((N, K), dtype=torch.uint8, device=dev)
        sx = torch.empty(((M + 31) // 32, (K + 31) // 32), dtype=torch.float32, device=dev)
        sw = torch.empty(((N + 31) // 32, (K + 31) // 32), dtype=torch.float32, device=dev)
        C = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        items.append((M, N, K, X, W, qx, qw, sx, sw, C, X_np, W_np))
        flops += 2.0 * M * N * K
        qelems += M * K + N * K
        gbytes += M * K + N * K + 2 * M * N + 4 * (sx.numel() + sw.numel())

    def run(xs, ws, cs, s, mark=True):
        for (M, N, K, _, _, qx, qw, sx, sw, _, _, _), X, W, C in zip(items, xs, ws, cs):
            if mark:
                ph.mark("quant")
            fl.fp8_quantize_blockwise_32x32(X.data_ptr(), M, K, K, qx.data_ptr(), K,
                                            sx.data_ptr(), sx.stride(0), s)
            fl.fp8_quantize_blockwise_32x32(W.data_ptr(), N, K, K, qw.data_ptr(), K,
                                            sw.data_ptr(), sw.stride(0), s)
            if mark:
                ph.mark("quant")
                ph.mark("gemm")
            fl.fp8_gemm_blockscaled_32x32(qx.data_ptr(), K, qw.data_ptr(), K, C.data_ptr(), N,
                                          M, N, K, sx.data_ptr(), sx.stride(0),
                                          sw.data_ptr(), sw.stride(0), s)
            if mark:
                ph.mark("gemm")

    def step():
        run([it[3] for it in items], [it[4] for it in items], [it[9] for it in items], sptr)

    # Pipelined end to end, as for the 8192^3 workload: step i's fp32
    # activations and weights come from pinned host memory on a copy stream,
    # its outputs go back on another; the host->device copies of step i+1,
    # the compute of step i (one stream, so codes and scales need no second
    # copy) and the device->host copies of step i-1 overlap.  Device inputs
    # and outputs are double-buffered.
    main = torch.cuda.current_stream(dev)
    nl = len(items)
    e2e = {}

    def ebegin(host_inputs, host_outputs2):
        if not e2e:
            e2e.update(
                X=[[it[3] for it in items], [torch.empty_like(it[3]) for it in items]],
                W=[[it[4] for it in items], [torch.empty_like(it[4]) for it in items]],
                C=[[it[9] for it in items], [torch.empty_like(it[9]) for it in items]],
                si=torch.cuda.Stream(dev), sc=torch.cuda.Stream(dev),
                so=torch.cuda.Stream(dev),
                computed=[torch.cuda.Event(), torch.cuda.Event()],
                stored=[torch.cuda.Event(), torch.cuda.Event()])
        e2e.update(X_h=host_inputs[:nl], W_h=host_inputs[nl:], C_h=host_outputs2)
        for k in ("computed", "stored"):
            for ev in e2e[k]:
                ev.record(main)
        for st in (e2e["si"], e2e["sc"], e2e["so"]):
            st.wait_stream(main)

    def estep(i):
        b = i & 1
        T = e2e
        # inputs: buffer b is free once the compute of step i-2 has read it
        T["si"].wait_event(T["computed"][b])
        with torch.cuda.stream(T["si"]):
            for d, h in zip(T["X"][b] + T["W"][b], T["X_h"] + T["W_h"]):
                d.copy_(h, non_blocking=True)
        loaded = torch.cuda.Event()
        loaded.record(T["si"])
        # compute into C[b] once the device->host copies of step i-2 have read it
        T["sc"].wait_event(loaded)
        T["sc"].wait_event(T["stored"][b])
        run(T["X"][b], T["W"][b], T["C"][b], T["sc"].cuda_stream, mark=False)
        T["computed"][b].record(T["sc"])
        T["so"].wait_event(T["computed"][b])
        with torch.cuda.stream(T["so"]):
            for k in range(nl):
                T["C_h"][k][b].copy_(T["C"][b][k], non_blocking=True)
        T["stored"][b].record(T["so"])

    def eend():
        for st in (e2e["si"], e2e["sc"], e2e["so"]):
            main.wait_stream(st)

    return dict(step=step, e2e_pipeline=(ebegin, estep, eend),
                flops=flops, launches=12, quant_bytes_per_elem=5, gemm_bound="alu",
                per_op=[(name, 2.0 * it[0] * it[1] * it[2]) for name, it in zip(linears, items)],
                workload=("32x32 block-scaled E4M3: block-quantize activations [4096][K] ~ N(0,1) "
                          "and weights [N][K] ~ N(0,0.02), then the block-scaled GEMM, for the "
                          "four 70B-class linears qkv (10240,8192), attn_out (8192,8192), gate_up "
                          "(57344,8192), down (8192,28672); seed 0"),
                config={"M": 4096, "linears": ",".join(linears),
                        "l2": "inputs 4.3 GB fp32 > 129 MB L2; no flush"},
                inputs=[(it[3], it[10]) for it in items] + [(it[4], it[11]) for it in items],
                outputs=[it[9] for it in items], quant_elems=qelems,
                gemm_label="gemm_e4m3_block32_kernel", gemm_bytes=gbytes,
                profile=("gemm_e4m3_block32_transformer", ["precision_linear_algebra_gb300/csrc/gemm_block32.cu",
                                                           "precision_linear_algebra_gb300/csrc/ptx.cuh"]),
                qprofile=("quantize_block32_transformer", QUANT_SOURCES))


def _workload_grouped(fl, torch, dev, sptr, ph):
    from precision_linear_algebra_gb300 import workloads
    counts, offs, X_np, W_np = workloads.moe_layer(seed=0)
    E, N, K = W_np.shape
    Mt = int(offs[-1])
    X = torch.from_numpy(X_np).to(dev)
    W = torch.from_numpy(W_np).to(dev)
    qx = torch.empty((Mt, K), dtype=torch.uint8, device=dev)
    qw = torch.empty((E, N, K), dtype=torch.uint8, device=dev)
    amax = torch.empty(2 * E, dtype=torch.float32, device=dev)
    sx = torch.empty(E, dtype=torch.float32, device=dev)
    sw = torch.empty(E, dtype=torch.float32, device=dev)
    d_off = torch.from_numpy(offs.astype("int32")).to(dev)
    C = torch.empty((Mt, N), dtype=torch.bfloat16, device=dev)
    P = lambda t, i=0: t.data_ptr() + i * t.element_size()

    # Codes and scales are double-buffered for the pipelined schedule.
    qx2 = [qx, torch.empty_like(qx)]
    qw2 = [qw, torch.empty_like(qw)]
    amax2 = [amax, torch.empty_like(amax)]
    sx2 = [sx, torch.empty_like(sx)]
    sw2 = [sw, torch.empty_like(sw)]
    # Activations: current scaling (their own amax, two passes).  Weights do
    # not change between steps, so each step quantises them in one pass with
    # the amax recorded at the previous step (delayed scaling), which is the
    # current amax: the codes and scales are those of current scaling.  The
    # two amax words of each expert alternate between steps (hist_w[parity]).
    hist_w = torch.empty((2, E), dtype=torch.float32, device=dev)
    for e in range(E):
        for parity in (0, 1):
            fl.fp8_quantize_pertensor(P(W) + e * N * K * 4, N, K, K, P(qw) + e * N * K, K,
                                      P(hist_w[parity], e), P(sw, e), sptr)
    counter = [0]

    def quant(b, s, Xd=X, Wd=W):
        parity = counter[0] & 1
        counter[0] += 1
        # every expert's activation rows in one call, the offsets read on
        # the device (as the grouped GEMM reads them)
        fl.fp8_quantize_pertensor_grouped(P(Xd), E, d_off.data_ptr(), Mt, K, K, P(qx2[b]), K,
                                          P(amax2[b]), P(sx2[b]), s)
        for e in range(E):
            fl.fp8_quantize_pertensor_delayed(
                P(Wd) + e * N * K * 4, N, K, K, P(qw2[b]) + e * N * K, K,
                P(hist_w[parity ^ 1], e), P(hist_w[parity], e), P(sw2[b], e), 0, s)

    def gemm(b, s, Cd=C):
        fl.fp8_grouped_gemm(E, d_off.data_ptr(), Mt, P(qx2[b]), K, P(qw2[b]), K, N * K, P(Cd),
                            N, N, K, P(sx2[b]), P(sw2[b]), s)

    def step():
        ph.mark("quant")
        quant(0, sptr)
        ph.mark("quant")
        ph.mark("gemm")
        gemm(0, sptr)
        ph.mark("gemm")

    # Pipelined schedule, as for the 8192^3 workload: step i+1's
    # quantisation on one stream while step i's grouped GEMM runs on another;
    # events order quantize(i) before GEMM(i) and GEMM(i) before
    # quantize(i+2), which reuses its buffers.
    main = torch.cuda.current_stream(dev)
    sq, sg = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    qdone = [torch.cuda.Event(), torch.cuda.Event()]
    gdone = [torch.cuda.Event(), torch.cuda.Event()]

    def pbegin():
        for ev in qdone + gdone:
            ev.record(main)
        sq.wait_stream(main)
        sg.wait_stream(main)

    def pstep(i):
        b = i & 1
        sq.wait_event(gdone[b])
        ph.mark("quant", sq)
        quant(b, sq.cuda_stream)
        ph.mark("quant", sq)
        qdone[b].record(sq)
        sg.wait_event(qdone[b])
        ph.mark("gemm", sg)
        gemm(b, sg.cuda_stream)
        ph.mark("gemm", sg)
        gdone[b].record(sg)

    def pend():
        main.wait_stream(sq)
        main.wait_stream(sg)

    # Pipelined end to end, as for the 8192^3 workload: step i's activations
    # and weights come from pinned host memory on two copy streams, its C
    # goes back on a third; the host->device copies of step i+1, compute of
    # step i and the device->host copy of step i-1 overlap (the link carries
    # both directions at once).  Device inputs and C are double-buffered.
    e2e = {}

    def ebegin(host_inputs, host_outputs2):
        X_h, W_h = host_inputs
        C_h2 = host_outputs2[0]
        if not e2e:
            e2e.update(X=[X, torch.empty_like(X)], W=[W, torch.empty_like(W)],
                       C=[C, torch.empty_like(C)],
                       sx=torch.cuda.Stream(dev), sw=torch.cuda.Stream(dev),
                       so=torch.cuda.Stream(dev),
                       quantized=[torch.cuda.Event(), torch.cuda.Event()],
                       computed=[torch.cuda.Event(), torch.cuda.Event()],
                       stored=[torch.cuda.Event(), torch.cuda.Event()])
        e2e.update(X_h=X_h, W_h=W_h, C_h=C_h2)
        for k in ("quantized", "computed", "stored"):
            for ev in e2e[k]:
                ev.record(main)
        for st in (e2e["sx"], e2e["sw"], e2e["so"], sq, sg):
            st.wait_stream(main)

    def estep(i):
        b = i & 1
        T = e2e
        # inputs: buffer b is free once quantize(i-2) has read it
        T["sx"].wait_event(T["quantized"][b])
        T["sw"].wait_event(T["quantized"][b])
        with torch.cuda.stream(T["sx"]):
            T["X"][b].copy_(T["X_h"], non_blocking=True)
        with torch.cuda.stream(T["sw"]):
            T["W"][b].copy_(T["W_h"], non_blocking=True)
        ev_x, ev_w = torch.cuda.Event(), torch.cuda.Event()
        ev_x.record(T["sx"])
        ev_w.record(T["sw"])
        sq.wait_event(ev_x)
        sq.wait_event(ev_w)
        sq.wait_event(gdone[b])
        quant(b, sq.cuda_stream, T["X"][b], T["W"][b])
        T["quantized"][b].record(sq)
        qdone[b].record(sq)
        # GEMM into C[b] once the device->host copy of step i-2 has read it
        sg.wait_event(qdone[b])
        sg.wait_event(T["stored"][b])
        gemm(b, sg.cuda_stream, T["C"][b])
        gdone[b].record(sg)
        T["computed"][b].record(sg)
        T["so"].wait_event(T["computed"][b])
        with torch.cuda.stream(T["so"]):
            T["C_h"][b].copy_(T["C"][b], non_blocking=True)
        T["stored"][b].record(T["so"])

    def eend():
        for st in (e2e["sx"], e2e["sw"], e2e["so"], sq, sg):
            main.wait_stream(st)

    return dict(step=step, pipeline=(pbegin, pstep, pend), e2e_pipeline=(ebegin, estep, eend),
                flops=2.0 * Mt * N * K,
                launches=2 + E + 1,
                workload=("grouped MoE E4M3: 8 experts, K 4096, N 14336, 8192 tokens top-2 "
                          "(16384 rows, Dirichlet(1) counts %s), per-expert per-tensor quantize "
                          "of activations (current scaling, all experts in one grouped call) and "
                          "weights (one pass with the amax recorded at the previous step; the "
                          "weights do not change, so codes and scales equal current scaling's), "
                          "one grouped GEMM launch; seed 0"
                          % list(map(int, counts))),
                config={"experts": E, "N": N, "K": K, "rows": Mt,
                        "l2": "inputs 2.1 GB fp32 > 129 MB L2; no flush"},
                inputs=[(X, X_np), (W, W_np)], outputs=[C], quant_elems=Mt * K + E * N * K,
                quant_bytes=QUANT_BYTES_PER_ELEM * Mt * K + 5 * E * N * K,
                gemm_label="gemm_e4m3_pair_kernel<true>",
                gemm_bytes=Mt * K + E * N * K + 2 * Mt * N,
                profile=("gemm_e4m3_grouped_moe", GEMM_SOURCES),
                qprofile=None)


def _workload_attention(fl, torch, dev, sptr, ph, batch=2, heads=64, seq=2048, hd=128):
    """The two GEMMs of non-causal FP8 multi-head attention, one group per
    (batch, head): scores = Q K^T (K = head_dim) and out = P V (K = seq, V
    given transposed).  Q, K, P and V are quantised to E4M3 per head once,
    at set-up (the quantiser is measured by the other workloads); a step is
    the two grouped GEMM launches.  Softmax is not part of this path: P is a
    seeded stand-in for the probabilities."""
    import numpy as np
    from precision_linear_algebra_gb300 import workloads
    E = batch * heads
    g = np.random.default_rng(0)
    Q_np = workloads.normal(g, (E * seq, hd))
    K_np = workloads.normal(g, (E, seq, hd))
    P_np = g.random((E * seq, seq), dtype=np.float32) / np.float32(seq)
    Vt_np = workloads.normal(g, (E, hd, seq))
    qQ = torch.empty(Q_np.shape, dtype=torch.uint8, device=dev)
    qK = torch.empty(K_np.shape, dtype=torch.uint8, device=dev)
    qP = torch.empty(P_np.shape, dtype=torch.uint8, device=dev)
    qV = torch.empty(Vt_np.shape, dtype=torch.uint8, device=dev)
    amax = torch.empty(4 * E, dtype=torch.float32, device=dev)
    sc = torch.empty(4 * E, dtype=torch.float32, device=dev)
    Pp = lambda t, i=0: t.data_ptr() + i * t.element_size()
    for arr, q, k4, rows, cols in ((Q_np, qQ, 0, seq, hd), (K_np, qK, 1, seq, hd),
                                   (P_np, qP, 2, seq, seq), (Vt_np, qV, 3, hd, seq)):
        x = torch.from_numpy(arr).to(dev)
        for e in range(E):
            fl.fp8_quantize_pertensor(Pp(x, e * rows * cols), rows, cols, cols,
                                      Pp(q, e * rows * cols), cols, Pp(amax, k4 * E + e),
                                      Pp(sc, k4 * E + e), sptr)
        torch.cuda.synchronize()
        del x
    offs = torch.arange(E + 1, dtype=torch.int32, device=dev) * seq
    S = torch.empty((E * seq, seq), dtype=torch.bfloat16, device=dev)
    O = torch.empty((E * seq, hd), dtype=torch.bfloat16, device=dev)

    def run(q4, so, s):
        q_Q, q_K, q_P, q_V = q4
        S_, O_ = so
        fl.fp8_grouped_gemm(E, offs.data_ptr(), E * seq, Pp(q_Q), hd, Pp(q_K), hd, seq * hd,
                            Pp(S_), seq, seq, hd, Pp(sc, 0), Pp(sc, E), s)
        fl.fp8_grouped_gemm(E, offs.data_ptr(), E * seq, Pp(q_P), seq, Pp(q_V), seq, hd * seq,
                            Pp(O_), hd, hd, seq, Pp(sc, 2 * E), Pp(sc, 3 * E), s)

    def step():
        ph.mark("quant")
        ph.mark("quant")
        ph.mark("gemm")
        run((qQ, qK, qP, qV), (S, O), sptr)
        ph.mark("gemm")

    # Pipelined end to end: step i+1's codes go to the device on one copy
    # stream while step i's two GEMMs run and step i-1's scores and outputs
    # come back on another; device codes, S and O are double-buffered.
    main = torch.cuda.current_stream(dev)
    e2e = {}

    def ebegin(host_inputs, host_outputs2):
        if not e2e:
            e2e.update(Q=[[qQ, qK, qP, qV], [torch.empty_like(t) for t in (qQ, qK, qP, qV)]],
                       R=[[S, O], [torch.empty_like(S), torch.empty_like(O)]],
                       si=torch.cuda.Stream(dev), sc=torch.cuda.Stream(dev),
                       so=torch.cuda.Stream(dev),
                       computed=[torch.cuda.Event(), torch.cuda.Event()],
                       stored=[torch.cuda.Event(), torch.cuda.Event()])
        e2e.update(H=host_inputs, R_h=host_outputs2)
        for k in ("computed", "stored"):
            for ev in e2e[k]:
                ev.record(main)
        for st in (e2e["si"], e2e["sc"], e2e["so"]):
            st.wait_stream(main)

    def estep(i):
        b = i & 1
        T = e2e
        T["si"].wait_event(T["computed"][b])
        with torch.cuda.stream(T["si"]):
            for d, h in zip(T["Q"][b], T["H"]):
                d.copy_(h, non_blocking=True)
        loaded = torch.cuda.Event()
        loaded.record(T["si"])
        T["sc"].wait_event(loaded)
        T["sc"].wait_event(T["stored"][b])
        run(T["Q"][b], T["R"][b], T["sc"].cuda_stream)
        T["computed"][b].record(T["sc"])
        T["so"].wait_event(T["computed"][b])
        with torch.cuda.stream(T["so"]):
            for k in range(2):
                T["R_h"][k][b].copy_(T["R"][b][k], non_blocking=True)
        T["stored"][b].record(T["so"])

    def eend():
        for st in (e2e["si"], e2e["sc"], e2e["so"]):
            main.wait_stream(st)

    flops = 2.0 * 2 * E * seq * seq * hd
    codes = [(qQ, qQ.cpu().numpy()), (qK, qK.cpu().numpy()), (qP, qP.cpu().numpy()),
             (qV, qV.cpu().numpy())]
    return dict(step=step, e2e_pipeline=(ebegin, estep, eend),
                flops=flops, launches=2, gemm_bound="hbm",
                workload=("FP8 attention GEMMs (scores = Q K^T, out = P V), non-causal, batch %d x "
                          "%d heads, seq %d, head_dim %d, E4M3 inputs with per-head scales "
                          "(quantised at set-up); two grouped launches per step; seed 0"
                          % (batch, heads, seq, hd)),
                config={"batch": batch, "heads": heads, "seq": seq, "head_dim": hd,
                        "l2": "operands 0.64 GB + outputs 1.14 GB > 129 MB L2; no flush"},
                inputs=codes, outputs=[S, O], quant_elems=1,
                gemm_label="gemm_e4m3_pair_kernel<true>",
                gemm_bytes=qQ.numel() + qK.numel() + qP.numel() + qV.numel() + 2 * (S.numel() + O.numel()),
                profile=("gemm_e4m3_attention", GEMM_SOURCES),
                qprofile=None)


WORKLOADS = {"pertensor8192": _workload_pertensor,
             "pertensor8192_delayed": (lambda fl, torch, dev, sptr, ph:
                                       _workload_pertensor(fl, torch, dev, sptr, ph, delayed=True)),
             "blockscaled": _workload_blockscaled,
             "grouped": _workload_grouped, "attention": _workload_attention,
             "square256": _workload_square(256),
             "square1024": _workload_square(1024),
             "square4096": _workload_square(4096)}


def run_gpu(args):
    import torch
    import precision_linear_algebra_gb300 as fl
    from precision_linear_algebra_gb300 import build

    world, rank, local_rank = _dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if rank == 0 or not os.path.exists(build.LIB_PATH):
        build.build()
    if world > 1:
        dist.barrier()
    fl.load()
    _SQUARE_OPTS.update(fmt=args.fmt, gemm_variant=args.gemm_variant)
    if args.workload.startswith("square") and args.gemm_variant:
        fl.fp8la_set_gemm_variant(args.gemm_variant)
    stream = torch.cuda.current_stream(dev)
    sptr = stream.cuda_stream
    ph = _Phases(torch, stream)
    if args.workload == "blockscaled" and args.linears:
        W = _workload_blockscaled(fl, torch, dev, sptr, ph, tuple(args.linears.split(",")))
    else:
        W = WORKLOADS[args.workload](fl, torch, dev, sptr, ph)
    step = W["step"]

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    # Then keep the GPU busy until its clocks have settled: on a GPU that was
    # idle, the first half second or so runs a few per cent below the
    # maximum SM clock (2002 against 2070 MHz was seen, 7 % off the step).
    busy_warmup(step, torch, args.warmup_seconds)
    if fl.fp8_get_device_status(sptr) != 0:
        raise RuntimeError("device status reports a timeout during warm-up")

    # Per-phase kernel durations, measured live on the launching stream.
    q_ms, g_ms = [], []
    ph.on = True
    for _ in range(min(args.steps, 50)):
        step()
        torch.cuda.synchronize()
        d = ph.collect()
        q_ms.append(d["quant"])
        g_ms.append(d["gemm"])
    ph.on = False

    visible = [v for v in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if v]
    gpu_index = visible[local_rank] if local_rank < len(visible) else local_rank
    pipelined = args.schedule == "pipelined" and "pipeline" in W
    graph = W.get("graph")

    def timed_region():
        """The timed steps (and, when pipelined, the serial schedule before
        them), with the SM clocks sampled throughout."""
        sampler = ClockSampler(gpu_index)
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        sampler.start()
        # the sampler's first rows take a moment; the GPU stays busy meanwhile
        busy_warmup(step, torch, 0.3)
        serial_ms = None
        if pipelined:
            # The serial schedule too, for reference (same steps, one stream).
            s0 = torch.cuda.Event(enable_timing=True)
            s1 = torch.cuda.Event(enable_timing=True)
            s0.record(stream)
            for _ in range(args.steps):
                step()
            s1.record(stream)
            torch.cuda.synchronize()
            serial_ms = s0.elapsed_time(s1) / args.steps
            pbegin, pstep, pend = W["pipeline"]
            pbegin()
            for i in range(max(3, args.warmup)):
                pstep(i)
            pend()
            torch.cuda.synchronize()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        # Every launch of the timed steps is bracketed by CUDA events on
        # its own stream (not possible inside a replayed graph).
        ph.events = []
        ph.on = graph is None
        torch.cuda.synchronize()
        t_start = time.time()
        t0.record(stream)
        if graph is not None:
            for _ in range(args.steps):
                graph.replay()
        elif pipelined:
            pbegin, pstep, pend = W["pipeline"]
            pbegin()
            for i in range(args.steps):
                pstep(i)
            pend()
        else:
            for _ in range(args.steps):
                step()
        t1.record(stream)
        torch.cuda.synchronize()
        t_end = time.time()
        ph.on = False
        clocks = sampler.stop(window=(t_start, t_end))
        if world > 1:
            dist.barrier()
        per_launch = ph.durations()
        phases = {k: v / args.steps for k, v in ph.collect().items()}
        phases["launches"] = per_launch
        return t0.elapsed_time(t1), serial_ms, clocks, phases

    ms_total, serial_ms, clocks, phases = timed_region()
    # A run that saw a hardware or thermal slowdown, or SM clocks far below
    # their maximum with no reason given (a clock lock left by someone else),
    # is not a valid measurement: it is taken once more, and the line says so.
    if max_over_ranks(1.0 if _clocks_invalid(clocks) else 0.0, dev) > 0:
        first = clocks
        ms_total, serial_ms, clocks, phases = timed_region()
        clocks["remeasured"] = {"first_reasons": first["reasons"],
                                "first_sm_mhz": first["sm_mhz"]}
    if fl.fp8_get_device_status(sptr) != 0:
        raise RuntimeError("device status reports a timeout in the timed region")
    if world > 1:
        ms_total = max_over_ranks(ms_total, dev)
    ms_step = ms_total / args.steps
    value = world * W["flops"] / (ms_step * 1e-3) / 1e12

    # End to end through the public API, host buffers: pinned H2D of the
    # step's fp32 inputs, the step's calls, D2H of the outputs, every step.
    hosts = [(d, torch.from_numpy(h).pin_memory()) for d, h in W["inputs"]]
    outs = [(o, torch.empty(o.shape, dtype=o.dtype).pin_memory()) for o in W["outputs"]]
    e2e_steps = max(3, min(args.steps, 30))
    e2e_pipelined = args.schedule == "pipelined" and "e2e_pipeline" in W

    def e2e_step():
        for d, h in hosts:
            d.copy_(h, non_blocking=True)
        step()
        for o, h in outs:
            h.copy_(o, non_blocking=True)

    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)

    def time_serial():
        e0.record(stream)
        for _ in range(e2e_steps):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / e2e_steps

    # The host link is shared with other work on the machine, so each
    # schedule is timed in E2E_REPEATS separate runs of e2e_steps steps and
    # the median run is reported (all runs are listed in the JSON line).
    e2e_serial_runs, e2e_runs = [], []
    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    if e2e_pipelined:
        ebegin, estep, eend = W["e2e_pipeline"]
        outs2 = [[h, torch.empty_like(h).pin_memory()] for _, h in outs]
        host_inputs = [h for _, h in hosts]
        e2e_serial_runs = [time_serial() for _ in range(E2E_REPEATS)]
        ebegin(host_inputs, outs2)
        for i in range(3):
            estep(i)
        eend()
        torch.cuda.synchronize()
        for _ in range(E2E_REPEATS):
            e0.record(stream)
            ebegin(host_inputs, outs2)
            for i in range(e2e_steps):
                estep(i)
            eend()
            e1.record(stream)
            torch.cuda.synchronize()
            e2e_runs.append(e0.elapsed_time(e1) / e2e_steps)
    else:
        e2e_runs = [time_serial() for _ in range(E2E_REPEATS)]
    e2e_equal = None
    if e2e_pipelined:
        # The host copies of the last pipelined step's outputs against the
        # device outputs of a plain step on the same inputs, bit for bit.
        step()
        torch.cuda.synchronize()
        e2e_equal = True
        for k, (o, _) in enumerate(outs):
            last = outs2[k][(e2e_steps - 1) & 1]
            dev_out = o.cpu()
            e2e_equal = e2e_equal and bool(torch.equal(last.view(torch.int16),
                                                       dev_out.view(torch.int16)))
            del dev_out
    e2e_ms = statistics.median(e2e_runs)
    e2e_serial_ms = statistics.median(e2e_serial_runs) if e2e_serial_runs else None
    if world > 1:
        e2e_ms = max_over_ranks(e2e_ms, dev)
    h2d = sum(h.numel() * h.element_size() for _, h in hosts)
    d2h = sum(h.numel() * h.element_size() for _, h in outs)

    hbm, bf16_burst, bf16_sust, peak_src = _peaks()
    fp8_peak = bf16_burst * FP8_OVER_BF16
    # The measured sustained figure comes from a seconds-long loop under the
    # power cap; it is the denominator when the timed region itself lasts
    # that long, or when the clocks sampled during it show the power cap
    # holding the SM clock below its maximum.  Other timed regions (and
    # kernels timed alone) are rated against the burst figure.
    in_loop, peak_regime = _peak_regime(ms_total, clocks, bf16_sust is not None,
                                        graph is not None)
    alu_peak, alu_src = _alu_promotion_peak(torch, dev)
    fp8_loop_peak = (bf16_sust if in_loop else bf16_burst) * FP8_OVER_BF16

    crosscheck = None
    if W.get("crosscheck") is not None and rank == 0:
        try:
            crosscheck = W["crosscheck"]()
        except Exception as e:                       # reported, never fatal
            crosscheck = {"error": "%s: %s" % (type(e).__name__, e)}
    # Kernel durations per step: over the timed steps from the events around
    # each launch on its own stream; with a replayed graph (no events inside
    # it) from the per-phase loop that ran before the timed region, which is
    # also reported for every workload as the kernels' isolated timing.
    g_iso = statistics.mean(g_ms)
    q_iso = statistics.mean(q_ms)
    if graph is None:
        g_avg = phases.get("gemm", g_iso)
        q_avg = phases.get("quant", q_iso)
        timing = ("CUDA events around each launch, on its own stream, over the timed steps"
                  + ("; pipelined, so each GEMM runs beside the next step's quantisation"
                     if pipelined else ""))
    else:
        g_avg, q_avg = g_iso, q_iso
        timing = ("CUDA events around each phase in a loop of single steps before the timed "
                  "region (the timed steps replay one CUDA graph)")
    qbpe = W.get("quant_bytes_per_elem", QUANT_BYTES_PER_ELEM)
    # algorithmic bytes of one step's quantisation (a workload whose
    # operands are quantised at different byte counts gives the total)
    qbytes = W.get("quant_bytes", qbpe * W["quant_elems"])

    def tflops(ms):
        return W["flops"] / (ms * 1e-3) / 1e12

    def gemm_gbs_of(ms):
        return W["gemm_bytes"] / (ms * 1e-3) / 1e9

    def quant_gbs_of(ms):
        if args.workload == "attention" or ms <= 1e-6:
            return None                                            # quantised at set-up
        return qbytes / (ms * 1e-3) / 1e9

    gemm_tflops, gemm_gbs, quant_gbs = tflops(g_avg), gemm_gbs_of(g_avg), quant_gbs_of(q_avg)
    quant_gbs_iso = quant_gbs_of(q_iso)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "warmup_busy_s": args.warmup_seconds,
            "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "e4m3 (fp32 accumulate, bf16 out)", "data": "synthetic",
            "config": dict({"workload": W["workload"],
                            "parallelism": "replicas" if world > 1 else "single GPU"},
                           **W["config"]),
            "roofline": ({"bound": "tensor", "achieved": gemm_tflops, "peak": fp8_loop_peak,
                          "unit": "TFLOP/s", "frac": gemm_tflops / fp8_loop_peak,
                          "traffic": _profile_traffic(*W["profile"]),
                          "kernel": W["gemm_label"], "timing": timing,
                          "peak_source": "%s bf16 %s %.1f x nominal fp8/bf16 ratio 2"
                                         % (peak_src, "sustained" if in_loop else "burst",
                                            bf16_sust if in_loop else bf16_burst),
                          "timed_region_ms": ms_total,
                          "peak_regime": peak_regime,
                          "frac_of_burst": gemm_tflops / fp8_peak,
                          "frac_of_nominal_fp8": gemm_tflops / NOMINAL_FP8_TFLOPS,
                          "achieved_isolated": tflops(g_iso),
                          "peak_isolated": fp8_peak,
                          "frac_isolated": tflops(g_iso) / fp8_peak,
                          "frac_isolated_of_nominal_fp8": tflops(g_iso) / NOMINAL_FP8_TFLOPS,
                          "nominal_fp8_tflops": NOMINAL_FP8_TFLOPS,
                          "library_crosscheck": crosscheck}
                         if W.get("gemm_bound", "tensor") == "tensor" else
                         {"bound": "alu", "achieved": gemm_tflops, "peak": alu_peak,
                          "unit": "TFLOP/s", "frac": gemm_tflops / alu_peak,
                          "traffic": _profile_traffic(*W["profile"]),
                          "kernel": W["gemm_label"], "timing": timing,
                          "peak_source": alu_src, "timed_region_ms": ms_total,
                          "tensor_peak": fp8_peak,
                          "frac_of_fp8_peak": gemm_tflops / fp8_peak,
                          "frac_of_nominal_fp8": gemm_tflops / NOMINAL_FP8_TFLOPS,
                          "achieved_isolated": tflops(g_iso),
                          "frac_isolated": tflops(g_iso) / alu_peak,
                          "frac_isolated_of_fp8_peak": tflops(g_iso) / fp8_peak,
                          "per_op": _per_op(W, phases, alu_peak, fp8_peak)}
                         if W.get("gemm_bound") == "alu" else
                         {"bound": "hbm", "achieved": gemm_gbs, "peak": hbm, "unit": "GB/s",
                          "frac": gemm_gbs / hbm,
                          "traffic": _profile_traffic(*W["profile"]),
                          "kernel": W["gemm_label"], "timing": timing,
                          "algorithmic_bytes_per_step": W["gemm_bytes"],
                          "peak_source": "%s copy bandwidth" % peak_src,
                          "tflops": gemm_tflops,
                          "frac_of_fp8_peak": gemm_tflops / fp8_peak,
                          "achieved_isolated": gemm_gbs_of(g_iso),
                          "frac_isolated": gemm_gbs_of(g_iso) / hbm}),
            "roofline_quantize": {"bound": "hbm", "achieved": quant_gbs, "peak": hbm,
                                  "unit": "GB/s",
                                  "frac": quant_gbs / hbm if quant_gbs else None,
                                  "frac_of_nominal_hbm": (quant_gbs / NOMINAL_HBM_GBS
                                                          if quant_gbs else None),
                                  "nominal_hbm_gbs": NOMINAL_HBM_GBS,
                                  "traffic": (_profile_traffic(*W["qprofile"])
                                              if W.get("qprofile") else None),
                                  "algorithmic_bytes_per_elem": qbytes / W["quant_elems"], "timing": timing,
                                  "achieved_isolated": quant_gbs_iso,
                                  "frac_isolated": (quant_gbs_iso / hbm
                                                    if quant_gbs_iso else None)},
            "breakdown": {"gemm_ms": g_avg, "quantize_ms": q_avg,
                          "gemm_ms_median_min": _median_min_per_step(
                              phases.get("launches", {}).get("gemm"), args.steps),
                          "gemm_ms_isolated": g_iso, "quantize_ms_isolated": q_iso,
                          "gemm_tflops": gemm_tflops, "quantize_gbs": quant_gbs,
                          "schedule": ("cuda graph" if graph is not None else
                                       "pipelined" if pipelined else "serial"),
                          "serial_ms_per_step": serial_ms if pipelined else ms_step,
                          "serial_value": (world * W["flops"] / (serial_ms * 1e-3) / 1e12
                                           if pipelined else value)},
            "e2e": {"value": world * W["flops"] / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "ms_per_step": e2e_ms,
                    "schedule": "pipelined" if e2e_pipelined else "serial",
                    "serial_ms_per_step": e2e_serial_ms if e2e_pipelined else e2e_ms,
                    "runs_ms_per_step": e2e_runs,
                    "serial_runs_ms_per_step": e2e_serial_runs or e2e_runs,
                    "pipelined_output_equals_device": e2e_equal},
            "gpu_launches": W["launches"] * args.steps * (len(args.linears.split(",")) / 4.0
                                                           if args.workload == "blockscaled"
                                                           and args.linears else 1),
            "clocks": clocks,
        }
        if args.workload != "pertensor8192":
            line["workload_kind"] = args.workload
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = _cpu_baseline_subprocess(W["flops"], args.workload,
                                                            args.linears)
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--warmup-seconds", type=float, default=1.0,
                    help="after the warm-up steps, keep running untimed steps for this long "
                         "(wall time) so that the timed region starts at settled clocks")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", default="pertensor8192", choices=sorted(WORKLOADS),
                    help="pertensor8192 is the headline line; the others measure the "
                         "block-scaled and grouped variants")
    ap.add_argument("--schedule", default="pipelined", choices=["pipelined", "serial"],
                    help="pipelined (default): step i+1's quantisation overlaps step i's GEMM "
                         "on a second stream; serial: one stream, steps back to back")
    ap.add_argument("--fmt", default="e4m3", choices=sorted(_FMT_CODES),
                    help="square* workloads: FP8 format of both operands")
    ap.add_argument("--gemm-variant", type=int, default=0, choices=[0, 1, 2],
                    help="square* workloads: GEMM kernel (0 by shape, 1 single CTA, 2 CTA pair)")
    ap.add_argument("--linears", default="",
                    help="blockscaled only: comma list of qkv,attn_out,gate_up,down "
                         "(default: all four)")
    args = ap.parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
