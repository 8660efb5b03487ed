"""Benchmark: per-tensor FP8 E4M3 quantize -> scaled GEMM at M = N = K = 8192.

One step is one pass of the whole path over one batch: quantise A (8192^2
fp32, N(0,1) with 0.1% +-50 sigma outliers) and B (N(0,0.02), same outlier
rule) to E4M3 on the device (amax -> scale -> cast), then the scaled GEMM
with FP32 accumulation and BF16 output.  Inputs are generated once (seeded),
copied to HBM before timing.  `value` is 2*M*N*K / (time of one whole step),
in TFLOP/s; the roofline object describes the GEMM kernel alone.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

With --impl reference the CPU oracle (test infrastructure under oracle/) is
timed on the host cores on a bounded sample of the same workload.  Under
torchrun each rank runs an independent replica on its own GPU (no data
exchange); rank 0 prints one JSON line.
"""

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

METRIC = ("FP8 E4M3 GEMM TFLOP/s (% of GB300 dense FP8 peak) at 8192³; "
          "quantize GB/s")
N_SIZE = 8192
FLOPS = 2.0 * N_SIZE ** 3
QUANT_BYTES_PER_ELEM = 9          # amax pass reads 4 B, cast pass reads 4 B + writes 1 B
GEMM_BYTES = 2 * N_SIZE * N_SIZE + 2 * N_SIZE * N_SIZE   # A, B codes + C bf16
FP8_OVER_BF16 = 4.5 / 2.25        # nominal dense FP8 : BF16 tensor ratio
WORKLOAD = ("per-tensor E4M3 quantize(A), quantize(B) + scaled GEMM, "
            "M=N=K=8192, A~N(0,1), B~N(0,0.02), 0.1% +-50sigma outliers, seed 0")
GEMM_SOURCES = ["precision_linear_algebra_gb300/csrc/gemm.cu",
                "precision_linear_algebra_gb300/csrc/ptx.cuh"]
QUANT_SOURCES = ["precision_linear_algebra_gb300/csrc/quantize.cu"]


def _dist_env():
    return int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")), \
        int(os.environ.get("LOCAL_RANK", "0"))


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return p["hbm_gbs"], p["bf16_tflops"], p.get("bf16_tflops_sustained"), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


def _src_hash(paths):
    h = hashlib.sha256()
    for p in paths:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
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


class ClockSampler:
    """nvidia-smi clocks/throttle reasons sampled while the timed region runs."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
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
            if len(parts) >= 9:
                self.rows.append(parts)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = self.rows
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


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
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": est * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def _cpu_baseline_subprocess():
    """The oracle on the host cores, run in a child process so that its BLAS
    threads are set explicitly; about 10-30 s of CPU work."""
    threads = os.cpu_count() or 1
    env = dict(os.environ, OPENBLAS_NUM_THREADS=str(threads), OMP_NUM_THREADS=str(threads),
               MKL_NUM_THREADS=str(threads))
    code = ("import json,sys; sys.path.insert(0, %r); import bench; "
            "A, B = bench._oracle_inputs(); "
            "e, w = bench._oracle_sample(A, B, 1024, 256, 2048); print(json.dumps([e, w]))" % ROOT)
    try:
        out = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True,
                             text=True, timeout=300)
        est, wall = json.loads(out.stdout.strip().splitlines()[-1])
    except Exception as exc:  # reported, not fatal
        return {"value": None, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                "sample": "failed: %s" % exc}
    return {"value": FLOPS / est / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": "oracle quantize of 1024 rows of A and of B + oracle GEMM of a 256 x 2048 "
                      "output block of the 8192^3 workload (%.1f s wall), scaled to one full "
                      "step by element and output counts" % wall}


# ------------------------------------------------------------------ GPU arm
def run_gpu(args):
    import numpy as np
    import torch
    import precision_linear_algebra_gb300 as fl
    from precision_linear_algebra_gb300 import build, workloads

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

    A_np, B_np = workloads.square_outliers(N_SIZE, seed=0)
    A = torch.from_numpy(A_np).to(dev)
    B = torch.from_numpy(B_np).to(dev)
    qa = torch.empty((N_SIZE, N_SIZE), dtype=torch.uint8, device=dev)
    qb = torch.empty_like(qa)
    amax = torch.empty(2, dtype=torch.float32, device=dev)
    scale = torch.empty(2, dtype=torch.float32, device=dev)
    C = torch.empty((N_SIZE, N_SIZE), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream(dev)
    sptr = stream.cuda_stream
    P = lambda t, i=0: t.data_ptr() + i * t.element_size()

    ev_q = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    ev_g = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    q_ms, g_ms = [], []

    def step(record=False):
        if record:
            ev_q[0].record(stream)
        fl.fp8_quantize_pertensor(P(A), N_SIZE, N_SIZE, N_SIZE, P(qa), N_SIZE,
                                  P(amax, 0), P(scale, 0), sptr)
        fl.fp8_quantize_pertensor(P(B), N_SIZE, N_SIZE, N_SIZE, P(qb), N_SIZE,
                                  P(amax, 1), P(scale, 1), sptr)
        if record:
            ev_q[1].record(stream)
            ev_g[0].record(stream)
        fl.fp8_gemm(P(qa), N_SIZE, P(qb), N_SIZE, P(C), N_SIZE, N_SIZE, N_SIZE, N_SIZE,
                    P(scale, 0), P(scale, 1), sptr)
        if record:
            ev_g[1].record(stream)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    if fl.fp8_get_device_status(sptr) != 0:
        raise RuntimeError("device status reports a timeout during warm-up")

    # Per-kernel durations, measured live on the launching stream.
    for _ in range(min(args.steps, 50)):
        step(record=True)
        torch.cuda.synchronize()
        q_ms.append(ev_q[0].elapsed_time(ev_q[1]))
        g_ms.append(ev_g[0].elapsed_time(ev_g[1]))

    visible = [v for v in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if v]
    sampler = ClockSampler(visible[local_rank] if local_rank < len(visible) else local_rank)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.3)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(args.steps):
        step()
    t1.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    if world > 1:
        dist.barrier()
    ms_total = t0.elapsed_time(t1)
    if fl.fp8_get_device_status(sptr) != 0:
        raise RuntimeError("device status reports a timeout in the timed region")
    if world > 1:
        tt = torch.tensor([ms_total], device=dev)
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        ms_total = tt.item()
    ms_step = ms_total / args.steps
    value = world * FLOPS / (ms_step * 1e-3) / 1e12

    # End to end through the public API, host buffers: pinned H2D of the
    # step's fp32 inputs, the three calls, D2H of C, every step.
    A_h = torch.from_numpy(A_np).pin_memory()
    B_h = torch.from_numpy(B_np).pin_memory()
    C_h = torch.empty((N_SIZE, N_SIZE), dtype=torch.bfloat16).pin_memory()
    e2e_steps = max(3, min(args.steps, 30))

    def e2e_step():
        A.copy_(A_h, non_blocking=True)
        B.copy_(B_h, non_blocking=True)
        step()
        C_h.copy_(C, non_blocking=True)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    if world > 1:
        tt = torch.tensor([e2e_ms], device=dev)
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        e2e_ms = tt.item()

    hbm, bf16_burst, bf16_sust, peak_src = _peaks()
    fp8_peak = bf16_burst * FP8_OVER_BF16
    g_avg = statistics.mean(g_ms)
    q_avg = statistics.mean(q_ms) / 2.0          # per operand
    gemm_tflops = FLOPS / (g_avg * 1e-3) / 1e12
    quant_gbs = QUANT_BYTES_PER_ELEM * N_SIZE * N_SIZE / (q_avg * 1e-3) / 1e9
    traffic = _profile_traffic("gemm_e4m3_pertensor_8192", GEMM_SOURCES)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "e4m3 (fp32 accumulate, bf16 out)", "data": "synthetic",
            "config": {"workload": WORKLOAD, "M": N_SIZE, "N": N_SIZE, "K": N_SIZE,
                       "parallelism": "replicas" if world > 1 else "single GPU",
                       "l2": "inputs 2 x 268 MB fp32 > 129 MB L2; no flush"},
            "roofline": {"bound": "tensor", "achieved": gemm_tflops, "peak": fp8_peak,
                         "unit": "TFLOP/s", "frac": gemm_tflops / fp8_peak,
                         "traffic": traffic,
                         "kernel": "gemm_e4m3_kernel<256,4,false>",
                         "peak_source": "%s bf16 burst %.1f x nominal fp8/bf16 ratio 2"
                                        % (peak_src, bf16_burst),
                         "frac_of_sustained": (gemm_tflops / (bf16_sust * FP8_OVER_BF16)
                                               if bf16_sust else None)},
            "roofline_quantize": {"bound": "hbm", "achieved": quant_gbs, "peak": hbm,
                                  "unit": "GB/s", "frac": quant_gbs / hbm,
                                  "traffic": _profile_traffic("quantize_pertensor_8192",
                                                              QUANT_SOURCES),
                                  "algorithmic_bytes_per_elem": QUANT_BYTES_PER_ELEM},
            "breakdown": {"gemm_ms": g_avg, "quantize_ms_per_operand": q_avg,
                          "gemm_tflops": gemm_tflops, "quantize_gbs": quant_gbs},
            "e2e": {"value": world * FLOPS / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                    "h2d_bytes_per_step": 2 * 4 * N_SIZE * N_SIZE,
                    "d2h_bytes_per_step": 2 * N_SIZE * N_SIZE,
                    "ms_per_step": e2e_ms},
            "gpu_launches": 5 * args.steps,
            "clocks": clocks,
        }
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = _cpu_baseline_subprocess()
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
