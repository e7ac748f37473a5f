"""Benchmark of the FP32 SGEMM path on GB300: prints ONE JSON line.

A step is one sgemm_f32 call, C = alpha * A * B + beta * C, on the 8192^3 workload
(A, B uniform[-1, 1), C N(0, 1), seed 3, alpha = 0.5, beta = 2). Inputs (805 MB) are larger
than the 129 MB L2, so no flush is needed between steps. C is updated in place each step;
with beta = 2 its magnitude doubles per step, which stays far from overflow for the step
counts used here and does not change the work.

value   = 2 M N K x steps x ranks / (max over ranks of the CUDA-event time of the steps)
e2e     = the same metric through sgemm_f32_host: A, B, C in pinned host memory, each step
          copying them to the device and C back (the library overlaps the copies of row
          blocks with the GEMMs of their neighbours), all inside the timed region
roofline: FP32 FFMA pipe ("alu"): SMs x 128 lanes x 2 FLOP x max SM clock
cpu_baseline: the CPU FP64 oracle on a bounded sample of rows of the same workload.

`--impl reference` times that oracle instead (the only reference this study has: the
pages ship no library), on the same workload and metric.

Launch: python bench.py [--gpus N --steps K --warmup W]; for N > 1 under
torch.distributed.run, one independent replica per GPU (the problem does not shard).
"""
from __future__ import annotations

import argparse
import json
import re
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from workloads import BY_NAME, CONFIGS, HEADLINE, workload_inputs  # noqa: E402

METRIC = "SGEMM TFLOPS (2MNK/t) at 4096³ and 8192³; fraction of GB300 FP32 peak"
UNIT = "TFLOP/s"
FP32_LANES_PER_SM = 128  # Blackwell SM: 4 partitions x 32 FP32 lanes


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=HEADLINE.name)
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=30.0,
                    help="target CPU time of the oracle sample (the headline's whole product "
                         "takes about 27 s on the GPU box's 16 cores: then every row is checked)")
    ap.add_argument("--no-variants", action="store_true",
                    help="skip the separately reported tensor-core 3xTF32 variant")
    ap.add_argument("--variant", type=int, default=-1,
                    help="force a tile configuration (profiling / tuning); -1 = automatic")
    ap.add_argument("--split", type=int, default=0,
                    help="force the split-K layout (see sgemm_f32_forced); 0 = automatic")
    return ap.parse_args()


TRAFFIC_FILE = os.path.join(ROOT, "profiles", "sgemm_ffma_traffic.json")
CSRC = os.path.join(ROOT, "dense_fp32_matrix_08_gb300", "csrc")
KERNEL_TU = "sgemm_tma.cu"  # the dominant kernel's translation unit
KERNEL_HOST = ("sgemm_plan.h", "sgemm_api.cu")  # the host code that plans and launches it


def kernel_sources():
    """The files the dominant GEMM kernel and its launch come from: its translation unit with
    every local header it includes, transitively, and the planning/launch host files."""
    seen, todo = [], [KERNEL_TU]
    while todo:
        fn = todo.pop(0)
        if fn in seen or not os.path.exists(os.path.join(CSRC, fn)):
            continue
        seen.append(fn)
        with open(os.path.join(CSRC, fn)) as f:
            todo += re.findall(r'^\s*#\s*include\s+"([^"/]+)"', f.read(), re.M)
    return sorted(set(seen) | set(KERNEL_HOST))


def kernel_source_hash() -> str:
    """sha256 over kernel_sources(): a recorded ncu traffic figure is only reported while
    this hash matches the one it was taken with (changes to other kernels leave it valid)."""
    import hashlib
    h = hashlib.sha256()
    for fn in kernel_sources():
        h.update(fn.encode())
        with open(os.path.join(CSRC, fn), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def git_sha():
    """The checked-out commit, or None where the tree is a copy without .git."""
    import subprocess
    try:
        out = subprocess.run(["git", "rev-parse", "HEAD"], cwd=ROOT, capture_output=True,
                             text=True, timeout=10)
        return out.stdout.strip() or None if out.returncode == 0 else None
    except (OSError, subprocess.SubprocessError):
        return None


def recorded_traffic(workload: str, plan: dict):
    """DRAM bytes per launch of the GEMM kernel from the committed ncu capture, or None if
    it was taken on another workload, plan or kernel source."""
    try:
        with open(TRAFFIC_FILE) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    for r in rec.get("captures", []):
        if (r.get("workload") == workload and r.get("source_sha256") == kernel_source_hash()
                and all(r.get("plan", {}).get(k) == plan.get(k)
                        for k in ("variant", "split", "main_tiles"))):
            return r["dram_bytes_read"] + r["dram_bytes_write"]
    return None


# ------------------------------------------------------------------------------------
# distributed plumbing (replicas only: barrier and max-over-ranks timing)

class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist
            backend = "nccl" if torch.cuda.is_available() else "gloo"
            if backend == "nccl":
                torch.cuda.set_device(self.local)
            dist.init_process_group(backend)
            self.pg = dist

    def barrier(self):
        if self.pg:
            if torch.cuda.is_available():
                self.pg.barrier(device_ids=[self.local])
            else:
                self.pg.barrier()

    def max(self, x: float) -> float:
        if not self.pg:
            return x
        dev = "cuda" if torch.cuda.is_available() else "cpu"
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


def replica_throughput(flops_per_step: float, steps: int, world: int, t_max: float) -> float:
    """Whole-job TFLOP/s of `world` independent replicas, each doing `steps` steps of
    `flops_per_step`, timed by the slowest rank (t_max seconds)."""
    return flops_per_step * steps * world / t_max / 1e12


# ------------------------------------------------------------------------------------
# clock sampling during the timed region

REASON_COLS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]


class ClockSampler:
    def __init__(self, bus_id: str | None):
        self.bus_id = bus_id
        self.proc = None
        self.lines: list[str] = []
        self.th = None

    def start(self):
        q = ("pci.bus_id,clocks.sm,clocks.max.sm,power.draw,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={q}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                text=True)
        except OSError:
            self.proc = None
            return
        self.th = threading.Thread(target=self._read, daemon=True)
        self.th.start()
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict | None:
        if not self.proc:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.th:
            self.th.join(timeout=2)
        rows = []
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 8:
                continue
            if self.bus_id and self.bus_id.lower() not in f[0].lower():
                continue
            try:
                rows.append((float(f[1]), float(f[2]), float(f[3]), f[4:8]))
            except ValueError:
                continue
        if not rows:
            return None
        power = [r[2] for r in rows]
        loaded = [r for r in rows if r[2] >= 0.5 * max(power)] or rows
        reasons = sorted({REASON_COLS[i] for r in loaded for i, v in enumerate(r[3])
                          if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in loaded),
                "sm_max_mhz": max(r[1] for r in rows), "reasons": reasons,
                "samples": len(loaded), "power_w_max": max(power)}


def bus_id_of(dev: int) -> str | None:
    try:
        p = torch.cuda.get_device_properties(dev)
        return f"{p.pci_bus_id:02X}:{p.pci_device_id:02X}."
    except Exception:
        return None


def max_sm_clock_mhz() -> float:
    try:
        out = subprocess.run(["nvidia-smi", "--query-gpu=clocks.max.sm",
                              "--format=csv,noheader,nounits"], capture_output=True,
                             text=True, timeout=30).stdout.split()
        return float(out[0])
    except Exception:
        return 2070.0  # GB300 maximum SM clock


def host_link_gbs(h: torch.Tensor, stream) -> dict:
    """Plain copy rates between the pinned host tensor `h` and the device, measured right
    after the end-to-end leg (5 copies each way, CUDA events): the host link the e2e
    figure depends on, which differs between machines and with the host's other load."""
    d = torch.empty_like(h, device="cuda")
    n = h.numel() * h.element_size()
    out = {}
    with torch.cuda.stream(stream):
        for name, dst, src in (("h2d_GBs", d, h), ("d2h_GBs", h, d)):
            dst.copy_(src, non_blocking=True)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(5):
                dst.copy_(src, non_blocking=True)
            e1.record(stream)
            e1.synchronize()
            out[name] = round(5 * n / (e0.elapsed_time(e1) * 1e-3) / 1e9, 1)
    del d
    out["bytes_per_copy"] = n
    return out


def cpu_model() -> str:
    """The host CPU's model name (lscpu), for the CPU baseline's record."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=30).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform
    return platform.processor() or platform.machine()


# ------------------------------------------------------------------------------------
# CPU oracle leg

def cpu_oracle_sample(w, A, B, C, seconds: float, rows_hint: int | None = None):
    """Time the oracle on a bounded set of rows; returns (TFLOP/s, rows, seconds, R, S)."""
    import oracle
    rng = np.random.default_rng(12345)
    # the oracle spreads rows over its threads: probe with two rows per thread, so that
    # the per-row time it measures is the one the full sample runs at
    probe = np.sort(rng.choice(w.M, size=min(w.M, 2 * oracle.threads()), replace=False))
    t0 = time.perf_counter()
    oracle.sgemm_f64_rows(A, B, C, w.alpha, w.beta, probe)
    dt = max(time.perf_counter() - t0, 1e-6)
    nrows = rows_hint or int(max(1, min(w.M, seconds / (dt / len(probe)))))
    if not rows_hint and nrows >= 0.75 * w.M:
        nrows = w.M  # within a third over the budget: check the whole product
    rows = np.sort(rng.choice(w.M, size=nrows, replace=False))
    t0 = time.perf_counter()
    R, S = oracle.sgemm_f64_rows(A, B, C, w.alpha, w.beta, rows)
    t = time.perf_counter() - t0
    return 2.0 * nrows * w.N * w.K / t / 1e12, rows, t, R, S, oracle.threads()


def reference_arm(args, dist: Dist):
    """`--impl reference`: the CPU FP64 oracle timed on the host cores."""
    if dist.rank != 0:
        return
    w = BY_NAME[args.workload]
    A, B, C = workload_inputs(w)
    per_step = max(1.0, min(6.0, 150.0 / max(1, args.steps + args.warmup)))
    _, rows, _, _, _, cores = cpu_oracle_sample(w, A, B, C, per_step)
    import oracle
    for _ in range(args.warmup):
        oracle.sgemm_f64_rows(A, B, C, w.alpha, w.beta, rows)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.sgemm_f64_rows(A, B, C, w.alpha, w.beta, rows)
    t = time.perf_counter() - t0
    value = 2.0 * len(rows) * w.N * w.K * args.steps / t / 1e12
    sample = (f"{len(rows)} of {w.M} output rows (all {w.N} columns, full K={w.K}) per "
              f"step, FP64 accumulation")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 0,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * t / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": _config(w),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "cpu_model": cpu_model(), "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def _config(w, sets=1, in_bytes=0):
    l2 = ("inputs larger than L2 (no flush needed)" if sets == 1 else
          f"inputs {in_bytes / 1e6:.0f} MB < 2x L2: steps rotate over {sets} device copies "
          f"({sets * in_bytes / 1e6:.0f} MB), so each step reads them from HBM (no flush)")
    return {"workload": f"sgemm {w.M}x{w.N}x{w.K} fp32 row-major packed, A,B "
                        f"{w.ab_dist} C {w.c_dist} seed {w.seed}, alpha={w.alpha} "
                        f"beta={w.beta}",
            "M": w.M, "N": w.N, "K": w.K, "alpha": w.alpha, "beta": w.beta,
            "parallelism": "replicas (one independent problem per GPU)",
            "l2": l2}


# ------------------------------------------------------------------------------------

# Dense TF32 tensor peak from the measured bf16 peak and the nominal TF32 : bf16 ratio
# (1.1 : 2.25 PFLOP/s dense on GB300).
TF32_OVER_BF16 = 1.1 / 2.25
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")


def hbm_peak_gbs():
    try:
        with open(PEAKS_FILE) as f:
            return float(json.load(f)["hbm_gbs"]), "of measured (MEASURED_PEAKS.json copy)"
    except (OSError, ValueError, KeyError):
        return 6800.0, "of fallback (6.8 TB/s)"


def tf32_peak_tflops():
    try:
        with open(PEAKS_FILE) as f:
            pk = json.load(f)
        return pk["bf16_tflops"] * TF32_OVER_BF16, "of measured (bf16 burst x 1.1/2.25)"
    except (OSError, ValueError, KeyError):
        return 1900.0 * TF32_OVER_BF16, "of fallback (1.9 PFLOP/s bf16 x 1.1/2.25)"


def tensor_core_variant(sg, args, stream, w, dA, dB, dC, C0):
    """The 3xTF32 tensor-core variant on the same workload, reported separately: FP32-
    equivalent TFLOP/s (2MNK/t, split passes included) and its tensor roofline (3 TF32
    products per multiply-add against the TF32 peak)."""
    M, N, K = w.M, w.N, w.K
    s_handle = stream.cuda_stream
    dC.copy_(C0)

    def step():
        rc = sg.lib.sgemm_f32_3xtf32(M, N, K, w.alpha, dA.data_ptr(), K, dB.data_ptr(), N,
                                     w.beta, dC.data_ptr(), N, s_handle)
        if rc != 0:
            raise RuntimeError(f"sgemm_f32_3xtf32 returned {rc}")

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
        t = time_steps(step, args.steps, stream)
    rc, status = sg.sgemm_f32_3xtf32_status()
    value = w.flops * args.steps / t / 1e12
    peak, basis = tf32_peak_tflops()
    return {"value": value, "unit": UNIT, "ms_per_step": 1e3 * t / args.steps,
            "launches_per_step": 3, "device_status": status,
            "roofline": {"bound": "tensor", "achieved": 3 * value, "peak": peak,
                         "unit": "TFLOP/s", "frac": 3 * value / peak, "peak_basis": basis,
                         "note": "achieved counts the 3 TF32 products per multiply-add; "
                                 "the time includes the hi/lo split passes"}}


def minimal_workspace_variant(sg, args, stream, w, dA, dB, dC, C0, plan):
    """The same product through sgemm_f32_ws given only the smallest workspace it runs with
    (sgemm_f32_workspace_size_min: the split-K partial tiles, no A^T copy). The plan is the
    default one with A transposed in shared memory by the same kernel's twin configuration,
    so the result must be bitwise the default call's, which this leg checks once."""
    M, N, K = w.M, w.N, w.K
    s_handle = stream.cuda_stream
    rc, nbytes = sg.sgemm_f32_workspace_size_min(M, N, K, K, N, N)
    if rc != 0:
        raise RuntimeError(f"sgemm_f32_workspace_size_min returned {rc}")
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=dC.device)

    def step():
        rc = sg.lib.sgemm_f32_ws(M, N, K, w.alpha, dA.data_ptr(), K, dB.data_ptr(), N,
                                 w.beta, dC.data_ptr(), N, ws.data_ptr(), nbytes, s_handle)
        if rc != 0:
            raise RuntimeError(f"sgemm_f32_ws returned {rc}")

    ref = C0.to(dC.device)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        rc = sg.lib.sgemm_f32(M, N, K, w.alpha, dA.data_ptr(), K, dB.data_ptr(), N, w.beta,
                              ref.data_ptr(), N, s_handle)
        if rc != 0:
            raise RuntimeError(f"sgemm_f32 returned {rc}")
        dC.copy_(C0)
        step()
    stream.synchronize()
    bitwise = bool(torch.equal(dC, ref))
    del ref
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
        t = time_steps(step, args.steps, stream)
    rc, status = sg.sgemm_f32_status()
    value = w.flops * args.steps / t / 1e12
    with_copy = plan["ws_bytes"] is not None and nbytes < plan["ws_bytes"]
    return {"value": value, "unit": UNIT, "ms_per_step": 1e3 * t / args.steps,
            "api": "sgemm_f32_ws with sgemm_f32_workspace_size_min bytes",
            "ws_bytes": nbytes, "default_ws_bytes": plan["ws_bytes"],
            "launches_per_step": plan["launches"] - 1 if with_copy else plan["launches"],
            "bitwise_equal_to_default": bitwise, "device_status": status}


def time_steps(fn, steps, stream, per_step=None):
    """Seconds for `steps` calls of fn enqueued back to back on `stream` (CUDA events on
    both sides). With a list `per_step`, an event after every call also gives each step's
    milliseconds (no synchronisation in between, so the total is unchanged)."""
    start = torch.cuda.Event(enable_timing=True)
    marks = []
    start.record(stream)
    for _ in range(steps):
        fn()
        if per_step is not None:
            marks.append(torch.cuda.Event(enable_timing=True))
            marks[-1].record(stream)
    end = torch.cuda.Event(enable_timing=True)
    end.record(stream)
    end.synchronize()
    if per_step is not None:
        prev = start
        for m in marks:
            per_step.append(round(prev.elapsed_time(m), 3))
            prev = m
    return start.elapsed_time(end) / 1e3


def recorded_share(workload: str, plan: dict):
    """The GEMM kernel's share of the step's GPU time from the committed ncu launch list,
    or None if it was taken on another workload, plan or kernel source."""
    try:
        with open(TRAFFIC_FILE) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    for r in rec.get("captures", []):
        if (r.get("workload") == workload and r.get("source_sha256") == kernel_source_hash()
                and "kernel_share" in r
                and all(r.get("plan", {}).get(k) == plan.get(k)
                        for k in ("variant", "split", "main_tiles"))):
            return r["kernel_share"]
    return None


def parity_rows(got, rows, R, S, C0, beta):
    """Elementwise check of sampled output rows against the oracle's R and S (the bound
    |C - R| <= 1e-4 (S + |beta c|), NaN failing)."""
    got = np.asarray(got, dtype=np.float64)
    c = C0.numpy()[rows].astype(np.float64)
    tol = 1e-4 * (S + np.abs(np.float64(np.float32(beta)) * c))
    err = np.abs(got - R)
    ok = bool(np.all(err <= tol))  # NaN compares false
    return {"rows": int(len(rows)), "max_err_over_tol": float(np.nanmax(err / tol)), "ok": ok}


def config_leg(sg, w, args, stream, peak, l2_bytes):
    """One more configuration on the automatic plan, timed like the headline: its first call
    (pristine C) checked against the oracle on 64 sampled rows, then `args.steps` calls after
    `args.warmup`, on rotating device copies when the inputs are under twice the L2. Calls
    shorter than 200 us are also replayed from a CUDA graph of max(40, copies) calls, which
    takes the host's launch cost out of the per-call time."""
    import oracle
    M, N, K = w.M, w.N, w.K
    A, B, C0 = workload_inputs(w)
    in_bytes = 4 * (M * K + K * N + M * N)
    sets = 1 if in_bytes >= 2 * l2_bytes else min(1024, -(-2 * l2_bytes // in_bytes))
    dA, dB, dC = A.cuda(), B.cuda(), C0.cuda()
    copies = [(dA, dB, dC)] + [(dA.clone(), dB.clone(), dC.clone()) for _ in range(sets - 1)]
    s_handle = stream.cuda_stream
    plan = sg.sgemm_f32_plan(M, N, K, K, N, N, w.alpha, w.beta, 0)
    calls = [0]

    def step():
        xA, xB, xC = copies[calls[0] % sets]
        calls[0] += 1
        rc = sg.lib.sgemm_f32(M, N, K, w.alpha, xA.data_ptr(), K, xB.data_ptr(), N, w.beta,
                              xC.data_ptr(), N, s_handle)
        if rc != 0:
            raise RuntimeError(f"sgemm_f32 returned {rc} on {w.name}")

    with torch.cuda.stream(stream):
        step()
    stream.synchronize()
    rng = np.random.default_rng(w.seed + 7)
    rows = np.unique(np.concatenate([[0, M - 1], rng.choice(M, size=min(M, 62),
                                                            replace=False)]))
    R, S = oracle.sgemm_f64_rows(A, B, C0, w.alpha, w.beta, rows)
    parity = parity_rows(dC[torch.as_tensor(rows, device="cuda")].cpu().numpy(), rows, R, S,
                         C0, w.beta)
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
        t = time_steps(step, args.steps, stream)
    per_call = t / args.steps
    rec = {"value": w.flops / per_call / 1e12, "unit": UNIT, "ms_per_call": 1e3 * per_call,
           "timing": "stream: back-to-back calls, CUDA events"}
    if per_call < 200e-6:
        graph_calls = max(40, sets)  # every rotating copy captured: the replay reads HBM
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g, stream=stream):
                for _ in range(graph_calls):
                    step()
            for _ in range(3):
                g.replay()
            start = torch.cuda.Event(enable_timing=True)
            end = torch.cuda.Event(enable_timing=True)
            reps = 5
            start.record(stream)
            for _ in range(reps):
                g.replay()
            end.record(stream)
            end.synchronize()
        per_call = start.elapsed_time(end) / 1e3 / (reps * graph_calls)
        rec.update({"value": w.flops / per_call / 1e12, "ms_per_call": 1e3 * per_call,
                    "timing": f"CUDA graph of {graph_calls} calls replayed {reps} times, "
                              f"CUDA events",
                    "stream_value": w.flops / (t / args.steps) / 1e12})
        del g
    alg_bytes = 4.0 * (M * K + K * N + M * N * (2 if w.beta != 0.0 else 1))
    hbm, hbm_basis = hbm_peak_gbs()
    gbs = alg_bytes / per_call / 1e9
    rec.update({
        "frac": rec["value"] / peak, "frac_basis": "of the FP32 peak (derived, as headline)",
        "alg_gbs": gbs, "hbm_frac": gbs / hbm, "hbm_basis": hbm_basis,
        "bound": "hbm" if w.flops / alg_bytes < peak * 1e12 / (hbm * 1e9) else "alu",
        "plan": {k: plan[k] for k in ("variant", "split", "main_tiles", "launches",
                                      "ws_bytes")},
        "parity": parity,
        "l2": ("inputs larger than 2x L2 (no flush needed)" if sets == 1 else
               f"inputs {in_bytes / 1e6:.1f} MB: calls rotate over {sets} device copies "
               f"({sets * in_bytes / 1e6:.0f} MB), so each call reads them from HBM"),
    })
    del copies
    torch.cuda.empty_cache()
    return rec


def our_arm(args, dist: Dist):
    import dense_fp32_matrix_08_gb300 as sg

    dev = dist.local if dist.world > 1 else 0
    torch.cuda.set_device(dev)
    w = BY_NAME[args.workload]
    M, N, K = w.M, w.N, w.K
    A, B, C0 = workload_inputs(w)
    stream = torch.cuda.Stream()
    s_handle = stream.cuda_stream
    dA, dB, dC = A.cuda(), B.cuda(), C0.cuda()
    # Inputs smaller than twice the L2 rotate over enough device copies that each step
    # reads its operands from HBM, not from the previous step's L2 lines.
    in_bytes = 4 * (M * K + K * N + M * N)
    l2_bytes = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or (129 << 20)
    sets = 1 if in_bytes >= 2 * l2_bytes else min(64, -(-2 * l2_bytes // in_bytes))
    copies = [(dA, dB, dC)] + [(dA.clone(), dB.clone(), dC.clone()) for _ in range(sets - 1)]
    calls = [0]
    torch.cuda.synchronize()

    plan = sg.sgemm_f32_plan(M, N, K, K, N, N, w.alpha, w.beta, 0)
    assert plan["status"] == 0, plan
    forced = args.variant >= 0 or args.split != 0
    if forced:
        plan = {"status": 0, "variant": args.variant, "split": args.split, "main_tiles": None,
                "launches": 2 if args.split not in (0, 1) else 1, "ws_bytes": None}

    def step():
        xA, xB, xC = copies[calls[0] % sets]
        calls[0] += 1
        if forced:
            rc = sg.lib.sgemm_f32_forced(M, N, K, w.alpha, xA.data_ptr(), K, xB.data_ptr(), N,
                                         w.beta, xC.data_ptr(), N, args.variant, args.split,
                                         s_handle)
        else:
            rc = sg.lib.sgemm_f32(M, N, K, w.alpha, xA.data_ptr(), K, xB.data_ptr(), N,
                                  w.beta, xC.data_ptr(), N, s_handle)
        if rc != 0:
            raise RuntimeError(f"sgemm_f32 returned {rc}")

    # first call on the pristine C: kept for the oracle check in the CPU-baseline leg
    with torch.cuda.stream(stream):
        step()
    stream.synchronize()
    first_rows = None

    cpu = None
    if dist.rank == 0 and not args.no_cpu_baseline:
        tf, rows, t, R, S, cores = cpu_oracle_sample(w, A, B, C0, args.cpu_seconds)
        e2e_rows, e2e_R, e2e_S = rows, R, S
        got = dC[torch.as_tensor(rows, device="cuda")].cpu().numpy().astype(np.float64)
        tol = 1e-4 * (S + np.abs(np.float32(w.beta) * C0.numpy()[rows].astype(np.float64)))
        err = np.abs(got - R)
        what = (f"all {M} output rows (the whole product)" if len(rows) == M else
                f"{len(rows)} random output rows of {M}")
        cpu = {"value": tf, "unit": UNIT, "cores": cores, "kind": "oracle",
               "cpu_model": cpu_model(),
               "sample": f"{what} (all {N} columns, full K={K}), FP64, {t:.1f} s",
               "parity": {"rows": len(rows), "max_err_over_tol": float(np.max(err / tol)),
                          "ok": bool(np.all(err <= tol))}}
    del first_rows

    for _ in range(args.warmup):
        with torch.cuda.stream(stream):
            step()
    stream.synchronize()

    sampler = ClockSampler(bus_id_of(dev))
    sampler.start()
    dist.barrier()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        elapsed = time_steps(step, args.steps, stream)
    torch.cuda.synchronize()
    dist.barrier()
    clocks = sampler.stop()
    t_max = dist.max(elapsed)
    flops = 2.0 * M * N * K
    value = replica_throughput(flops, args.steps, dist.world, t_max)
    ms = 1e3 * t_max / args.steps

    # dominant kernel: with a single-launch plan the step time is the kernel's duration
    props = torch.cuda.get_device_properties(dev)
    max_mhz = (clocks or {}).get("sm_max_mhz") or max_sm_clock_mhz()
    peak = props.multi_processor_count * FP32_LANES_PER_SM * 2 * max_mhz * 1e6 / 1e12
    achieved = flops * args.steps / elapsed / 1e12
    roof = {"bound": "alu", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
            "frac": achieved / peak, "traffic": recorded_traffic(w.name, plan),
            "traffic_unit": "bytes per launch (ncu dram__bytes_read.sum + "
                            "dram__bytes_write.sum of the GEMM kernel)",
            "peak_basis": f"{props.multi_processor_count} SMs x {FP32_LANES_PER_SM} FP32 "
                          f"lanes x 2 FLOP x {max_mhz:.0f} MHz (max SM clock)",
            "kernel_launches_per_step": plan["launches"],
            "achieved_basis": "2MNK per step over the whole step's time (every launch of "
                              "the step: A^T copy, GEMM kernel, split-K finish); the GEMM "
                              "kernel alone is kernel_share of it (ncu launch list)"}
    share = recorded_share(w.name, plan)
    if share:
        roof["kernel_share"] = share
        roof["kernel_achieved"] = achieved / share
    if clocks and clocks.get("sm_mhz"):
        roof["frac_at_sampled_clock"] = achieved / (peak * clocks["sm_mhz"] / max_mhz)
    # below the FP32/HBM ridge (the thin shapes) the roofline is HBM: algorithmic bytes
    # (A, B, C read when beta != 0, C write) per second against the measured copy bandwidth
    alg_bytes = 4.0 * (M * K + K * N + M * N * (2 if w.beta != 0.0 else 1))
    hbm, hbm_basis = hbm_peak_gbs()
    if flops / alg_bytes < peak * 1e12 / (hbm * 1e9):
        gbs = alg_bytes * args.steps / elapsed / 1e9
        roof = {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s",
                "frac": gbs / hbm, "traffic": recorded_traffic(w.name, plan),
                "traffic_unit": roof["traffic_unit"], "peak_basis": hbm_basis,
                "algorithmic_bytes_per_step": alg_bytes,
                "kernel_launches_per_step": plan["launches"],
                "fp32": {"achieved": achieved, "peak": peak, "unit": "TFLOP/s"}}

    # the derived FP32 peak's measured counterpart: the library's FFMA2 pipe probe, timed
    # after (outside) the timed region
    probe = sg.sgemm_f32_fma_probe(1 << 17, 5)
    if probe["status"] == 0 and probe["tflops"] > 0:
        fp32 = roof.get("fp32", roof)
        fp32["fp32_probe"] = {
            "tflops": probe["tflops"], "ms_per_launch": probe["ms"],
            "frac_of_derived_peak": probe["tflops"] / peak,
            "what": "sgemm_f32_fma_probe: SMs x 8 CTAs x 256 threads, 8 independent "
                    "fma.rn.f32x2 chains per thread on broadcast operand pairs, 2^17 "
                    "iterations; median of 5 launches (CUDA events), run after the timed "
                    "region"}
        fp32["frac_of_probe"] = achieved / probe["tflops"]

    # end to end: host buffers in pinned memory through the library's host-buffer entry
    # point; the copies in and out are inside the timed region
    e2e = None
    if args.e2e_steps > 0:
        hA, hB, hC = A.pin_memory(), B.pin_memory(), C0.pin_memory()

        def e2e_step():
            rc = sg.lib.sgemm_f32_host(M, N, K, w.alpha, hA.data_ptr(), K, hB.data_ptr(), N,
                                       w.beta, hC.data_ptr(), N, s_handle)
            if rc != 0:
                raise RuntimeError(f"sgemm_f32_host returned {rc}")

        e2e_parity = None
        with torch.cuda.stream(stream):
            e2e_step()  # on the pristine C: its sampled rows are checked against the oracle
            stream.synchronize()
            if cpu is not None:
                e2e_parity = parity_rows(hC[torch.as_tensor(e2e_rows)].numpy(), e2e_rows,
                                         e2e_R, e2e_S, C0, w.beta)
            e2e_step()
            stream.synchronize()
            dist.barrier()
            e2e_steps_ms = []
            e2e_t = time_steps(e2e_step, args.e2e_steps, stream, e2e_steps_ms)
        e2e_t = dist.max(e2e_t)
        e2e = {"value": replica_throughput(flops, args.e2e_steps, dist.world, e2e_t),
               "unit": UNIT, "api": "sgemm_f32_host (pinned host buffers)",
               "h2d_bytes_per_step": 4 * (M * K + K * N + M * N),
               "d2h_bytes_per_step": 4 * M * N, "ms_per_step": 1e3 * e2e_t / args.e2e_steps,
               "parity": e2e_parity, "host_link": host_link_gbs(hC, stream),
               "step_ms": e2e_steps_ms}

    secondary = {}
    if not args.no_secondary and w.name == HEADLINE.name:
        for w2 in CONFIGS:
            if w2.name != HEADLINE.name:
                secondary[w2.name] = config_leg(sg, w2, args, stream, peak, l2_bytes)

    variants = {}
    if not args.no_variants:
        variants["3xtf32_tensor_core"] = tensor_core_variant(sg, args, stream, w, dA, dB, dC, C0)
        if not forced:
            variants["minimal_workspace"] = minimal_workspace_variant(sg, args, stream, w, dA,
                                                                      dB, dC, C0, plan)

    if dist.rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": dist.world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32", "data": "synthetic", "config": _config(w, sets, in_bytes),
            "roofline": roof, "cpu_baseline": cpu, "e2e": e2e, "clocks": clocks,
            "gpu_launches": plan["launches"] * args.steps,
            "plan": {k: plan[k] for k in ("variant", "split", "main_tiles", "launches",
                                          "ws_bytes")},
            "source_sha256": kernel_source_hash(), "git_sha": git_sha(),
            "impl": "ours",
        }
        if secondary:
            line["secondary"] = secondary
        if variants:
            line["variants"] = variants
        print(json.dumps(line), flush=True)


def main():
    args = parse()
    dist = Dist()
    try:
        if args.impl == "reference":
            reference_arm(args, dist)
        else:
            our_arm(args, dist)
    finally:
        dist.close()


if __name__ == "__main__":
    main()
