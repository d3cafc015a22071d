#!/usr/bin/env python
"""Benchmark: GEMM TFLOP/s (2MNK / t) of C = A x B, row-major, on GB300.

One step is one call of the library's C entry point on one batch of
synthetic input resident in HBM (dispatch, optional re-pitch, the GEMM
kernel with its loads, MMAs and epilogue).  The headline line times the
TF32 tensor-core path at M = N = K = 8192; the same run also times every
other mode (FP32 SIMT and 3xTF32 at 8192^3; BF16, FP16, FP8 E4M3 / E5M2
and TF32 at the 16384 x 14336 x 4096 transformer-layer shape) and reports them under
"modes".  Inputs are larger than L2 (129 MB), so no flush is needed.  The
small workloads (64^3, 1024^3, ragged 1000 x 1013 x 997) are timed per mode
under "small", with L2 warm (CUDA-graph replay) and with L2 flushed before
each call.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--mode tf32|3xtf32|simt|bf16|fp16|e4m3|e5m2]
  python bench.py --impl reference ...   # the CPU oracle, timed on host cores

Multi-GPU (launched by torch.distributed.run): every rank runs its own
replica (GEMM has no exchange step here); value = all ranks' flops / the
slowest rank's time.
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "GEMM TFLOP/s (2MNK/t) at 8192³ per mode; % of FP32/TF32/BF16 dense peak"
UNIT = "TFLOP/s"
# Nominal dense tensor rates (PFLOP/s): the ratio converts the measured BF16
# peak into peaks for the other tensor-core types.
NOMINAL_PF = {"bf16": 2.25, "tf32": 1.1, "fp8": 4.5}
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                  "sm_max_mhz": 2070.0}


# ---------------------------------------------------------------- helpers
def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawTextHelpFormatter)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=50)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--mode", choices=["tf32", "3xtf32", "simt", "bf16", "fp16", "e4m3", "e5m2"],
                   default="tf32")
    p.add_argument("--no-modes", action="store_true", help="headline only, skip the per-mode table")
    p.add_argument("--no-cpu", action="store_true", help="skip the CPU-oracle baseline")
    p.add_argument("--cpu-seconds", type=float, default=10.0)
    p.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg")
    p.add_argument("--layout", choices=["NN", "NT", "TN", "TT"], default="NN",
                   help="operand layout of the headline: T = that operand is stored transposed "
                        "(A as K x M, B as N x K)")
    p.add_argument("--shape", default=None,
                   help="M,N,K: time the headline mode on a seeded uniform[-1,1) workload of this "
                        "shape instead of the benchmark workload (profiling runs)")
    p.add_argument("--quick", action="store_true",
                   help="smoke run: every workload of the configuration once (1 timed step, 3 "
                        "warm-up, no CPU baseline, no end-to-end leg, 2 steps per mode)")
    a = p.parse_args(argv)
    if a.quick:
        a.steps, a.warmup, a.no_cpu, a.no_e2e = 1, 3, True, True
    if a.warmup < 3:
        p.error("--warmup must be >= 3")
    if a.steps < 1:
        p.error("--steps must be >= 1")
    return a


def workload_for(mode, transformer=False, shape=None):
    from dense_gemm_f32_gb300 import inputs

    if shape:
        M, N, K = (int(x) for x in shape.split(","))
        return inputs.Workload(f"uniform {M}x{N}x{K}", M, N, K, 3, "uniform", bf16=(mode == "bf16"),
                               fp16=(mode == "fp16"),
                               fp8=mode if mode in ("e4m3", "e5m2") else "")

    if mode == "bf16":
        return inputs.TRANSFORMER_BF16
    if mode == "fp16":
        return inputs.TRANSFORMER_F16
    if mode == "e4m3":
        return inputs.TRANSFORMER_E4M3
    if mode == "e5m2":
        return inputs.TRANSFORMER_E5M2
    return inputs.TRANSFORMER_F32 if transformer else inputs.SQUARE_8192


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS if k in d}, "measured"
    except (OSError, ValueError, KeyError):
        return dict(FALLBACK_PEAKS), "fallback"


def mode_peak(mode, peaks, num_sms, measured=None):
    """(bound, peak TFLOP/s, how) for a mode's kernel timed in a short loop.

    BF16 / FP16: the driver's measured cuBLAS BF16 burst.  TF32 (and 3xTF32,
    whose MMA work is three TF32 products) and FP8: cuBLAS's own TF32 and FP8
    rates measured in this run (`measured`, best of 10 at 8192^3), else the
    BF16 burst scaled by the nominal dense-rate ratio.  SIMT: the FFMA peak,
    SMs x 128 lanes x 2 flop x the maximum SM clock."""
    measured = measured or {}
    if mode == "simt":
        mhz = peaks.get("sm_max_mhz", 2070.0)
        return "alu", num_sms * 128 * 2 * mhz * 1e6 / 1e12, (
            f"{num_sms} SMs x 128 FP32 lanes x 2 flop x {mhz:.0f} MHz")
    bf16 = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    if mode == "bf16":
        return "tensor", bf16, "measured cuBLAS bf16 burst (MEASURED_PEAKS)"
    if mode == "fp16":
        return "tensor", bf16, ("measured cuBLAS bf16 burst (MEASURED_PEAKS; fp16 and bf16 share "
                                "the nominal rate)")
    key = "fp8" if mode in ("e4m3", "e5m2") else "tf32"
    if measured.get(key):
        what = ("torch._scaled_mm E4M3 8192^3" if key == "fp8" else
                "torch.matmul fp32 8192^3 with TF32 allowed")
        return "tensor", measured[key], f"measured in this run: cuBLAS {what}, best of 10"
    return "tensor", nominal_peak(mode, peaks), (
        f"fallback: measured bf16 burst x nominal {key}/bf16 ratio "
        f"{NOMINAL_PF[key] / NOMINAL_PF['bf16']:.4f}")


def nominal_peak(mode, peaks):
    """The BF16 burst scaled by the nominal dense-rate ratio (a secondary
    figure next to the measured TF32 / FP8 peaks)."""
    bf16 = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    key = "fp8" if mode in ("e4m3", "e5m2") else "tf32" if mode in ("tf32", "3xtf32") else "bf16"
    return bf16 * NOMINAL_PF[key] / NOMINAL_PF["bf16"]


def measure_tensor_peaks(device, reps=10):
    """cuBLAS's TF32 and FP8 (E4M3) rates at 8192^3 on this GPU, the best of
    `reps` back-to-back calls after 3 warm-up calls: the roofline denominators
    of the TF32 and FP8 modes.  A failed measurement is recorded, not raised."""
    import torch

    out, errors = {}, {}
    n = 8192
    flops = 2.0 * n ** 3
    g = torch.Generator(device="cpu").manual_seed(12)
    A = (2 * torch.rand(n, n, generator=g) - 1).to(device)
    B = (2 * torch.rand(n, n, generator=g) - 1).to(device)

    def best(fn):
        # back to back, one event between consecutive calls (no host launch
        # gap inside a timed interval), the fastest interval
        for _ in range(3):
            fn()
        torch.cuda.synchronize(device)
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(reps + 1)]
        ev[0].record()
        for i in range(reps):
            fn()
            ev[i + 1].record()
        torch.cuda.synchronize(device)
        return flops / (min(ev[i].elapsed_time(ev[i + 1]) for i in range(reps)) * 1e-3) / 1e12

    prev = torch.backends.cuda.matmul.allow_tf32
    try:
        torch.backends.cuda.matmul.allow_tf32 = True
        C = torch.empty(n, n, device=device)
        out["tf32"] = best(lambda: torch.matmul(A, B, out=C))
    except Exception as e:  # noqa: BLE001 -- recorded in the line instead
        errors["tf32"] = f"{type(e).__name__}: {e}"
    finally:
        torch.backends.cuda.matmul.allow_tf32 = prev
    try:
        A8 = A.to(torch.float8_e4m3fn)
        B8 = B.t().contiguous().t().to(torch.float8_e4m3fn)  # column-major, as cuBLAS wants
        one = torch.tensor(1.0, device=device)
        out["fp8"] = best(lambda: torch._scaled_mm(A8, B8, scale_a=one, scale_b=one,
                                                   out_dtype=torch.float32))
    except Exception as e:  # noqa: BLE001
        errors["fp8"] = f"{type(e).__name__}: {e}"
    if errors:
        out["errors"] = errors
    return out


def kernel_name(mode, M, N, num_sms):
    """The kernel the library runs for this mode and shape: the CTA-pair
    tensor-core kernel once there are 256 x 256 tiles for at least a quarter
    of the SMs, else the single-CTA one (the library's own rule)."""
    if mode == "simt":  # B stored K x N, 16-byte aligned rows: the TMA ring kernel
        return "sgemm_ring_kernel (TMA ring)"
    pair_tiles = ((M + 255) // 256) * ((N + 255) // 256)
    return "tc2_gemm_kernel (CTA pair)" if pair_tiles * 4 >= num_sms else "tc_gemm_kernel"


def source_sha(mode):
    """Hash of the sources of a mode's kernel: a recorded traffic figure
    applies only while it matches."""
    csrc = os.path.join(ROOT, "dense_gemm_f32_gb300", "csrc")
    files = (["simt.cu", "ptx.cuh", "tmap.cuh"] if mode == "simt"
             else ["tc.cu", "ptx.cuh", "tf32_split.cuh", "tmap.cuh"])
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:12]


# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) per launch of the
# dominant kernel, from one ncu capture each (--clock-control none, one
# launch), keyed by (mode, workload); `sha` is source_sha(mode) of the sources
# the capture ran, so a figure goes stale (null in the line) as soon as the
# kernel changes.  The summaries of these captures are in profiles/.
_NCU = ("ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum,gpu__time_duration.sum "
        "--clock-control none -k regex:{k} -s 3 -c 1 python bench.py --mode {m} --steps 3 "
        "--warmup 3 --no-modes --no-cpu --no-e2e")
_WHERE = "one GB300 of the pool, 2026-12-02, after the same command exited 0 without ncu"
RECORDED_TRAFFIC = {
    ("tf32", "square-8192 fp32"): {
        "bytes": 2044077312 + 259028480, "sha": "8caeb4a95d22", "kernel": "tc2_gemm_kernel<TF32>",
        "read": 2044077312, "write": 259028480, "command": _NCU.format(k="tc2_gemm", m="tf32"),
        "where": _WHERE},
    ("3xtf32", "square-8192 fp32"): {
        "bytes": 4320433408 + 262098944, "sha": "8caeb4a95d22",
        "kernel": "tc2_gemm_kernel<3xTF32> (lo parts loaded too)", "read": 4320433408,
        "write": 262098944, "command": _NCU.format(k="tc2_gemm", m="3xtf32"), "where": _WHERE},
    ("bf16", "transformer-layer 16384x14336x4096 bf16"): {
        "bytes": 972379392 + 907912960, "sha": "8caeb4a95d22", "kernel": "tc2_gemm_kernel<BF16>",
        "read": 972379392, "write": 907912960, "command": _NCU.format(k="tc2_gemm", m="bf16"),
        "where": _WHERE},
    ("e4m3", "transformer-layer 16384x14336x4096 e4m3"): {
        "bytes": 315256832 + 888218880, "sha": "8caeb4a95d22",
        "kernel": "tc2_gemm_kernel<E4M3> (B stored N x K after the transpose launch)",
        "read": 315256832, "write": 888218880, "command": _NCU.format(k="tc2_gemm", m="e4m3"),
        "where": _WHERE},
    ("simt", "square-8192 fp32"): {
        "bytes": 2853867520 + 262399232, "sha": "cb63087d890a", "kernel": "sgemm_ring_kernel",
        "read": 2853867520, "write": 262399232, "command": _NCU.format(k="sgemm_ring", m="simt"),
        "where": _WHERE},
}


def recorded_traffic(mode, workload_name, table=None):
    """(bytes per launch, provenance) for a mode's kernel on a workload, or
    (None, why) when nothing was recorded for the current sources."""
    table = RECORDED_TRAFFIC if table is None else table
    rec = table.get((mode, workload_name))
    if rec is None:
        return None, "no ncu capture recorded for this kernel and workload"
    if rec["sha"] != source_sha(mode):
        return None, f"stale: recorded for sources {rec['sha']}, now {source_sha(mode)}"
    return float(rec["bytes"]), {k: v for k, v in rec.items() if k != "bytes"}


class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons in the background."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.file = None
        self.t0 = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        self.t0 = time.time()
        return self

    def rows(self):
        """Samples so far (the sampler keeps running)."""
        if self.proc is None:
            return []
        time.sleep(0.12)  # let nvidia-smi write the samples of the window just ended
        self.file.flush()
        with open(self.file.name) as f:
            return self._parse(f)

    def stop(self):
        rows = []
        if self.proc is None:
            return rows
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = self._parse(self.file)
        self.file.close()
        os.unlink(self.file.name)
        return rows

    @staticmethod
    def _parse(lines):
        rows = []
        for ln in lines:
            c = [x.strip() for x in ln.split(",")]
            if len(c) < 9:
                continue
            try:
                ts = time.mktime(time.strptime(c[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                frac = float("0." + c[0].split(".")[1]) if "." in c[0] else 0.0
                rows.append({"t": ts + frac, "sm": float(c[1]), "max": float(c[2]),
                             "reasons": {"hw_slowdown": c[5], "hw_thermal_slowdown": c[6],
                                         "sw_thermal_slowdown": c[7], "sw_power_cap": c[8]}})
            except ValueError:
                continue
        return rows


# Throttle reasons that void a measurement (sw_power_cap is kept and noted).
REJECT_REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown")


def rejected(clocks):
    """Why a timed window's clock record voids it: a rejecting throttle
    reason, or SM clocks far below their maximum with no reason (a leftover
    clock lock).  None when the window is usable."""
    bad = [r for r in clocks.get("reasons", []) if r in REJECT_REASONS]
    if bad:
        return ",".join(bad)
    sm, mx = clocks.get("sm_mhz"), clocks.get("sm_max_mhz")
    if sm and mx and sm < 0.8 * mx and not clocks.get("reasons"):
        return f"sm clock {sm:.0f} of {mx:.0f} MHz with no reason"
    return None


def summarize_clocks(rows, windows):
    """Median SM clock and active throttle reasons over samples inside any of
    the timed windows (wall-clock (start, end) pairs)."""
    if not rows:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                "note": "nvidia-smi unavailable"}
    inside = [r for r in rows if any(a - 0.05 <= r["t"] <= b + 0.05 for a, b in windows)]
    note = "samples inside the timed regions"
    if not inside:
        lo = min(a for a, _ in windows) - 1.0
        hi = max(b for _, b in windows) + 1.0
        inside = [r for r in rows if lo <= r["t"] <= hi]
        note = "no sample fell inside a timed region; samples within 1 s of them"
    if not inside:
        inside, note = rows, "all samples of the run"
    reasons = sorted({k for r in inside for k, v in r["reasons"].items()
                      if v.lower() in ("active", "1", "yes")})
    return {"sm_mhz": statistics.median(r["sm"] for r in inside),
            "sm_max_mhz": max(r["max"] for r in inside), "reasons": reasons,
            "samples": len(inside), "note": note}


def aggregate(median_ms, total_ms, world, flops_per_rank, steps, all_max):
    """Whole-job numbers from this rank's timed steps: all ranks' flops over
    the slowest rank's median step (`value`, `ms_per_step`), and over the
    slowest rank's bracketed total of the K steps (`value_from_total`).
    `all_max` reduces a float by max over ranks."""
    med = all_max(median_ms)
    tot = all_max(total_ms)
    return {"ms_per_step": med, "ms_total": tot,
            "value": world * flops_per_rank / (med * 1e-3) / 1e12,
            "value_from_total": world * flops_per_rank * steps / (tot * 1e-3) / 1e12}


# ------------------------------------------------------------- distributed
class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None

    def init(self, backend):
        if self.world > 1:
            import torch.distributed as dist

            dist.init_process_group(backend=backend)
            self.pg = dist

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, x, device=None):
        if not self.pg:
            return x
        import torch

        t = torch.tensor([float(x)], dtype=torch.float64, device=device)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


# ----------------------------------------------------------------- CPU arm
def cpu_oracle_rate(seconds, chunk=8):
    """The oracle as it stands, on the host cores, over the first rows of the
    8192^3 workload until `seconds` have passed.  (TFLOP/s, rows, threads, s)"""
    import numpy as np

    import oracle
    from dense_gemm_f32_gb300 import inputs

    w = inputs.SQUARE_8192
    A, B = inputs.make(w)
    An, Bn = A.numpy(), B.numpy()
    threads = oracle.max_threads()
    done, t0 = 0, time.perf_counter()
    while True:
        rows = np.arange(done, done + chunk) % w.M
        oracle.gemm_rows(An, Bn, rows, with_abs=False)
        done += chunk
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    flops = 2.0 * done * w.N * w.K
    return flops / el / 1e12, done, threads, el


def cpu_oracle_small():
    """Seconds the oracle (C only) takes on the three small workloads, on one
    host thread and on all of them."""
    import oracle
    from dense_gemm_f32_gb300 import inputs

    out, nmax = {}, oracle.max_threads()
    try:
        for w in (inputs.SQUARE_64, inputs.SQUARE_1024, inputs.RAGGED_1000):
            A, B = inputs.make(w)
            An, Bn = A.float().numpy(), B.float().numpy()
            row = {}
            for n in sorted({1, nmax}):
                oracle.set_threads(n)
                t0 = time.perf_counter()
                oracle.gemm(An, Bn)
                row[f"s_{n}_thread{'s' if n > 1 else ''}"] = round(time.perf_counter() - t0, 4)
            out[w.name] = row
    finally:
        oracle.set_threads(nmax)
    return out


def run_reference(args, dist):
    """--impl reference: the CPU oracle timed as the reference arm."""
    if dist.rank != 0:
        return 0
    import numpy as np

    import oracle
    from dense_gemm_f32_gb300 import inputs

    w = inputs.SQUARE_8192
    A, B = inputs.make(w)
    An, Bn = A.numpy(), B.numpy()
    rows_per_step = 16
    threads = oracle.max_threads()
    nxt = 0

    def step():
        nonlocal nxt
        rows = (np.arange(rows_per_step) + nxt) % w.M
        nxt += rows_per_step
        oracle.gemm_rows(An, Bn, rows, with_abs=False)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    el = time.perf_counter() - t0
    flops = 2.0 * rows_per_step * w.N * w.K * args.steps
    value = flops / el / 1e12
    sample = (f"{rows_per_step} full rows of C (all {w.N} columns, K={w.K}) per step of the "
              f"{w.name} workload, FP64 accumulation")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": el * 1e3 / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded uniform[-1,1))",
            "config": {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "mode": "cpu-oracle"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------- GPU arm
def device_inputs(w, mode, device):
    import dense_gemm_f32_gb300 as dg
    from dense_gemm_f32_gb300 import inputs

    A, B = inputs.make(w)
    want = dg.input_dtype(mode)
    if A.dtype != want:  # a float32 workload timed in a narrower mode
        A, B = A.float().to(want), B.float().to(want)
    return A, B, A.to(device), B.to(device)


def l2_flush_buffer(device):
    """A float32 buffer of twice the L2 size: writing it evicts A, B and C."""
    import torch

    l2 = getattr(torch.cuda.get_device_properties(device), "L2_cache_size", 0) or (129 << 20)
    return torch.empty(2 * l2 // 4, dtype=torch.float32, device=device)


def time_device(mode, Ad, Bd, C, steps, warmup, dist, device, ta=False, tb=False, flush=None):
    """Device time of `steps` calls on inputs resident in HBM.  Without
    `flush` the calls run back to back and are timed by one event between
    each pair of calls; with it (inputs smaller than L2) the buffer is
    rewritten before every call, outside that call's event pair."""
    import torch

    import dense_gemm_f32_gb300 as dg

    stream = torch.cuda.current_stream(device)
    for _ in range(warmup):
        dg.matmul(Ad, Bd, mode=mode, out=C, trans_a=ta, trans_b=tb)
    torch.cuda.synchronize(device)
    dist.barrier()
    torch.cuda.synchronize(device)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    ev_end = [torch.cuda.Event(enable_timing=True) for _ in range(steps)] if flush is not None else None
    n0 = dg.dgemm_kernel_launches()
    w0 = time.time()
    for i in range(steps):
        if flush is not None:
            flush.zero_()
        ev[i].record(stream)
        dg.matmul(Ad, Bd, mode=mode, out=C, trans_a=ta, trans_b=tb)
        if flush is not None:
            ev_end[i].record(stream)
    ev[steps].record(stream)
    torch.cuda.synchronize(device)
    w1 = time.time()
    dist.barrier()
    torch.cuda.synchronize(device)
    launches = dg.dgemm_kernel_launches() - n0
    if flush is None:
        per = [ev[i].elapsed_time(ev[i + 1]) for i in range(steps)]
        total = ev[0].elapsed_time(ev[steps])
    else:
        per = [ev[i].elapsed_time(ev_end[i]) for i in range(steps)]
        total = sum(per)
    return {"ms_total": total, "per_step_ms": per, "launches": launches, "window": (w0, w1),
            "flushed": None if flush is None else True}


def cublas_same_run(mode, Ad, Bd, device, steps=10):
    """cuBLAS (through torch) on a mode's operands, timed the same way (median
    of `steps` event-timed calls after 3 warm-up calls): a comparator for the
    roofline fraction, not part of the library.  Returns (ms, None), or
    (None, why) for a mode cuBLAS has no counterpart of (3xTF32) or a call
    that fails."""
    import torch

    if mode == "3xtf32":
        return None, "no cuBLAS counterpart (split-precision TF32)"
    prev = torch.backends.cuda.matmul.allow_tf32
    try:
        if mode in ("tf32", "simt"):
            torch.backends.cuda.matmul.allow_tf32 = mode == "tf32"
            fn = lambda: Ad @ Bd  # noqa: E731
        elif mode in ("bf16", "fp16"):
            fn = lambda: torch.mm(Ad, Bd, out_dtype=torch.float32)  # noqa: E731
        elif mode in ("e4m3", "e5m2"):
            Bt = Bd.t().contiguous().t()  # column-major B, as cuBLAS's FP8 kernels want
            one = torch.tensor(1.0, device=device)
            fn = lambda: torch._scaled_mm(Ad, Bt, scale_a=one, scale_b=one,  # noqa: E731
                                          out_dtype=torch.float32)
        else:
            return None, f"unknown mode {mode}"
        for _ in range(3):
            fn()
        torch.cuda.synchronize(device)
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
        for i in range(steps):
            ev[i].record()
            fn()
        ev[steps].record()
        torch.cuda.synchronize(device)
        return statistics.median(ev[i].elapsed_time(ev[i + 1]) for i in range(steps)), None
    except Exception as e:  # noqa: BLE001 -- a comparator must never fail the bench
        return None, f"{type(e).__name__}: {e}"
    finally:
        torch.backends.cuda.matmul.allow_tf32 = prev


def cublas_entry(flops, ours_tflops, ms, why):
    """The cuBLAS comparator's entry in the line: its rate and ours over it,
    or why there is none."""
    if ms is None:
        return {"tflops": None, "why": why}
    tf = flops / (ms * 1e-3) / 1e12
    return {"tflops": round(tf, 1), "frac_of_cublas": round(ours_tflops / tf, 4)}


def time_graph(mode, Ad, Bd, C, device, calls=20, replays=7):
    """Device time per call of `calls` back-to-back calls captured in one CUDA
    graph (no host launch gaps; L2 warm after the first call): the median over
    `replays` replays, each timed by its own event pair, so that one replay
    caught in a clock dip does not move the figure."""
    import torch

    import dense_gemm_f32_gb300 as dg

    st = torch.cuda.Stream(device)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(st):
        dg.matmul(Ad, Bd, mode=mode, out=C)
        st.synchronize()
        with torch.cuda.graph(g, stream=st):
            for _ in range(calls):
                dg.matmul(Ad, Bd, mode=mode, out=C)
    g.replay()
    torch.cuda.synchronize(device)
    cur = torch.cuda.current_stream(device)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(replays + 1)]
    ev[0].record(cur)
    for i in range(replays):
        g.replay()
        ev[i + 1].record(cur)
    torch.cuda.synchronize(device)
    per = [ev[i].elapsed_time(ev[i + 1]) for i in range(replays)]
    return statistics.median(per) * 1e3 / calls


SMALL_MODES = ("simt", "tf32", "3xtf32", "bf16", "fp16", "e4m3", "e5m2")


def time_small(device, dist, steps=20):
    """The small workloads of the benchmark configuration (64^3, 1024^3 and
    the ragged 1000 x 1013 x 997), every mode: microseconds per call with L2
    warm (graph replay of back-to-back calls) and with L2 flushed before each
    call (event pair per call)."""
    import torch

    from dense_gemm_f32_gb300 import inputs

    flush = l2_flush_buffer(device)
    out, windows = {}, []
    for w in (inputs.SQUARE_64, inputs.SQUARE_1024, inputs.RAGGED_1000):
        for m in SMALL_MODES:
            _, _, Ad, Bd = device_inputs(w, m, device)
            C = torch.empty((w.M, w.N), dtype=torch.float32, device=device)
            try:
                warm = time_graph(m, Ad, Bd, C, device)
            except RuntimeError as e:  # capture refused: report, keep going
                warm = None
                print(f"graph timing of {m}@{w.name} failed: {e}", file=sys.stderr)
            r = time_device(m, Ad, Bd, C, steps, 3, dist, device, flush=flush)
            windows.append(r["window"])
            cold = statistics.median(r["per_step_ms"]) * 1e3
            out[f"{m}@{w.name}"] = {
                "us_warm": None if warm is None else round(warm, 2),
                "us_l2_flushed": round(cold, 2),
                "tflops_warm": None if warm is None else round(w.flops / warm / 1e6, 2),
                "tflops_l2_flushed": round(w.flops / cold / 1e6, 2)}
    del flush
    torch.cuda.empty_cache()
    return out, windows


def time_e2e(mode, A, B, steps, warmup, dist, device):
    """Same metric through the public API with host buffers.  Every step
    copies its A and B from pinned host memory to the device, runs the GEMM
    and copies its C back to pinned host memory.  Steps are pipelined on
    three streams with two device buffer sets: the uploads of step i+1 and
    the read-back of step i-1 overlap the GEMM of step i."""
    import torch

    import dense_gemm_f32_gb300 as dg

    Ah, Bh = A.pin_memory(), B.pin_memory()
    M, N = A.shape[0], B.shape[1]
    Ch = [torch.empty((M, N), dtype=torch.float32).pin_memory() for _ in range(2)]
    Ad = [torch.empty_like(Ah, device=device) for _ in range(2)]
    Bd = [torch.empty_like(Bh, device=device) for _ in range(2)]
    Cd = [torch.empty((M, N), dtype=torch.float32, device=device) for _ in range(2)]
    s_up, s_mm, s_down = (torch.cuda.Stream(device) for _ in range(3))
    ev = lambda: torch.cuda.Event()  # noqa: E731
    up_done = [ev(), ev()]      # inputs of buffer b uploaded
    mm_done = [ev(), ev()]      # GEMM on buffer b finished
    down_done = [ev(), ev()]    # C of buffer b copied back
    for b in range(2):          # all buffers start free
        down_done[b].record(s_down)
        mm_done[b].record(s_mm)

    def run(n):
        for i in range(n):
            b = i & 1
            s_up.wait_event(mm_done[b])           # buffer b's inputs no longer in use
            with torch.cuda.stream(s_up):
                Ad[b].copy_(Ah, non_blocking=True)
                Bd[b].copy_(Bh, non_blocking=True)
            up_done[b].record(s_up)
            s_mm.wait_event(up_done[b])
            s_mm.wait_event(down_done[b])         # buffer b's C already read back
            dg.matmul(Ad[b], Bd[b], mode=mode, out=Cd[b], stream=s_mm)
            mm_done[b].record(s_mm)
            s_down.wait_event(mm_done[b])
            with torch.cuda.stream(s_down):
                Ch[b].copy_(Cd[b], non_blocking=True)
            down_done[b].record(s_down)

    run(warmup)
    torch.cuda.synchronize(device)
    dist.barrier()
    torch.cuda.synchronize(device)
    t0 = time.perf_counter()
    run(steps)
    torch.cuda.synchronize(device)
    ms = (time.perf_counter() - t0) * 1e3
    dist.barrier()
    h2d = Ah.numel() * Ah.element_size() + Bh.numel() * Bh.element_size()
    d2h = Ch[0].numel() * Ch[0].element_size()
    return ms, h2d, d2h


def run_ours(args, dist):
    import torch

    import dense_gemm_f32_gb300 as dg
    from dense_gemm_f32_gb300 import build

    build.build()
    dg.load()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (there is no CPU fallback)")
    device = torch.device("cuda", dist.local_rank)
    torch.cuda.set_device(device)
    dist.init("nccl" if dist.world > 1 else "gloo")
    props = torch.cuda.get_device_properties(device)
    num_sms = props.multi_processor_count
    peaks, peak_src = load_peaks()
    sampler = ClockSampler(dist.local_rank).start()

    # ---- headline
    mode = args.mode
    w = workload_for(mode, shape=args.shape)
    A, B, Ad, Bd = device_inputs(w, mode, device)
    ta, tb = args.layout[0] == "T", args.layout[1] == "T"
    if ta:  # store the transposed operands (A as K x M, B as N x K)
        Ad = Ad.t().contiguous()
    if tb:
        Bd = Bd.t().contiguous()
    C = torch.empty((w.M, w.N), dtype=torch.float32, device=device)
    in_bytes = Ad.numel() * Ad.element_size() + Bd.numel() * Bd.element_size() + C.numel() * 4
    l2 = getattr(props, "L2_cache_size", 0) or (129 << 20)
    flush = l2_flush_buffer(device) if in_bytes < 2 * l2 else None
    r = time_device(mode, Ad, Bd, C, args.steps, args.warmup, dist, device, ta, tb, flush=flush)
    # A window whose clock record shows a rejecting throttle reason (or a
    # clock lock) is measured once more; every rank takes the same decision.
    why = rejected(summarize_clocks(sampler.rows(), [r["window"]]))
    remeasured = None
    if dist.max(1.0 if why else 0.0, device) > 0:
        remeasured = why or "another rank's window"
        r = time_device(mode, Ad, Bd, C, args.steps, args.warmup, dist, device, ta, tb, flush=flush)
    del flush
    agg = aggregate(statistics.median(r["per_step_ms"]), r["ms_total"], dist.world, w.flops,
                    args.steps, lambda x: dist.max(x, device))
    windows = [r["window"]]
    launches_per_step = r["launches"] / args.steps
    mean_launch_ms = statistics.mean(r["per_step_ms"])

    # ---- this GPU's cuBLAS TF32 and FP8 rates: the denominators of those modes
    measured = measure_tensor_peaks(device) if not args.quick else {}
    bound, peak, peak_how = mode_peak(mode, peaks, num_sms, measured)
    achieved = w.flops / (mean_launch_ms * 1e-3) / 1e12
    traffic, traffic_src = recorded_traffic(mode, w.name)
    roofline = {"bound": bound, "achieved": achieved, "peak": peak, "unit": UNIT,
                "frac": achieved / peak, "traffic": traffic, "traffic_source": traffic_src,
                "kernel": kernel_name(mode, w.M, w.N, num_sms),
                "peak_source": f"{peak_src}: {peak_how}",
                "per_launch_flops": w.flops, "launches_per_step": launches_per_step,
                "achieved_from": "2MNK / mean per-launch device time (CUDA events, timed steps)"}
    if bound == "tensor":
        roofline["peak_nominal_ratio"] = round(nominal_peak(mode, peaks), 1)
        roofline["frac_of_nominal_ratio"] = round(achieved / nominal_peak(mode, peaks), 4)
    if measured.get("errors"):
        roofline["peak_measure_errors"] = measured["errors"]

    # ---- cuBLAS on the same operands (comparator for the roofline fraction)
    cublas_head = (None, "not timed")
    if not args.quick and not ta and not tb and dist.world == 1:
        cublas_head = cublas_same_run(mode, Ad, Bd, device)
        # like with like: our median step against cuBLAS's median call
        median_tflops = w.flops / (statistics.median(r["per_step_ms"]) * 1e-3) / 1e12
        roofline["cublas_same_run"] = cublas_entry(w.flops, median_tflops, *cublas_head)

    # ---- end to end through the public API with host buffers
    e2e_line = None
    del Ad, Bd, C
    torch.cuda.empty_cache()
    if not args.no_e2e:
        e2e_steps = max(3, min(args.steps, 20))
        e2e_ms, h2d, d2h = time_e2e(mode, A, B, e2e_steps, 3, dist, device)
        e2e = aggregate(e2e_ms / e2e_steps, e2e_ms, dist.world, w.flops, e2e_steps,
                        lambda x: dist.max(x, device))
        e2e_line = {"value": e2e["value_from_total"], "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h}
    torch.cuda.empty_cache()

    # ---- every other mode, same clocking, each with cuBLAS on its operands
    modes = {}
    if not args.no_modes:
        table = [("simt", False), ("tf32", False), ("3xtf32", False), ("bf16", True),
                 ("fp16", True), ("e4m3", True), ("e5m2", True), ("tf32", True)]
        for m, tr in table:
            wm = workload_for(m, transformer=tr)
            if m == mode and wm.name == w.name:
                per = r["per_step_ms"]
                cub = cublas_head
            else:
                _, _, Adm, Bdm = device_inputs(wm, m, device)
                Cm = torch.empty((wm.M, wm.N), dtype=torch.float32, device=device)
                steps_m = 2 if args.quick else max(20, min(args.steps, 30))
                rm = time_device(m, Adm, Bdm, Cm, steps_m, 3, dist, device)
                windows.append(rm["window"])
                per = rm["per_step_ms"]
                cub = ((None, "not timed") if args.quick or dist.world > 1
                       else cublas_same_run(m, Adm, Bdm, device))
                del Adm, Bdm, Cm
                torch.cuda.empty_cache()
            bm, pm, how = mode_peak(m, peaks, num_sms, measured)
            med = statistics.median(per)
            tfl = wm.flops / (med * 1e-3) / 1e12
            e = {"tflops_median": round(tfl, 2), "bound": bm, "peak": round(pm, 1),
                 "frac": round(tfl / pm, 4), "peak_source": how, "ms_median": round(med, 4),
                 "ms_min": round(min(per), 4), "ms_max": round(max(per), 4), "steps": len(per),
                 "cublas_same_run": cublas_entry(wm.flops, tfl, *cub)}
            if m == "3xtf32":  # three TF32 products per product: the tensor pipe's share
                e["mma_frac"] = round(3 * tfl / pm, 4)
            if m == "simt":
                e["kernel"] = kernel_name(m, wm.M, wm.N, num_sms)
            modes[f"{m}@{wm.name}"] = e
    small = {}
    if not args.no_modes and not args.shape:
        small, sw = time_small(device, dist)
        windows += sw
    clocks = summarize_clocks(sampler.stop(), windows)

    # ---- CPU oracle baseline (rank 0, N = 1 only)
    cpu = None
    if not args.no_cpu and dist.world == 1:
        v, rows, threads, secs = cpu_oracle_rate(args.cpu_seconds)
        cpu = {"value": v, "unit": UNIT, "cores": threads, "kind": "oracle",
               "sample": f"first {rows} full rows of C of the {inputs_name()} workload "
                         f"({secs:.1f} s, FP64 accumulation, OpenMP over rows)",
               "small_workloads": cpu_oracle_small()}

    if dist.rank == 0:
        line = {
            "metric": METRIC, "value": agg["value"], "unit": UNIT, "n_gpus": dist.world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": agg["ms_per_step"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": {"tf32": "tf32", "3xtf32": "3xtf32", "simt": "f32", "bf16": "bf16",
                      "fp16": "fp16", "e4m3": "fp8-e4m3", "e5m2": "fp8-e5m2"}[mode],
            "data": "synthetic (seeded, shapes and distributions of the workload)",
            "config": {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "mode": mode,
                       "layout": f"row-major, compact leading dimensions, op(A) op(B) = "
                                 f"{args.layout}",
                       "l2": ("inputs larger than L2 (no flush needed)" if r.get("flushed") is None
                              else "L2 flushed (2 x L2 bytes written) before every timed call"),
                       "parallelism": "replicas" if dist.world > 1 else "single GPU",
                       "remeasured": remeasured},
            "roofline": roofline,
            "cpu_baseline": cpu,
            "e2e": e2e_line,
            "gpu_launches": r["launches"],
            "clocks": clocks,
            "modes": modes,
            "small": small,
            "step_ms": {"median": statistics.median(r["per_step_ms"]),
                        "min": min(r["per_step_ms"]), "max": max(r["per_step_ms"]),
                        "mean": mean_launch_ms, "total_of_k_steps": agg["ms_total"],
                        "value_from_total": agg["value_from_total"],
                        "value_is": "whole-job TFLOP/s over the median of the K timed steps"},
            "measured_peaks_this_run": {k: (round(v, 1) if isinstance(v, float) else v)
                                        for k, v in measured.items()},
        }
        print(json.dumps(line), flush=True)
    st, where = dg.dgemm_watchdog_status(torch.cuda.current_stream(device).cuda_stream)
    dist.close()
    if st != dg.OK:
        print(f"watchdog tripped at site {where:#x}", file=sys.stderr)
        return 1
    return 0


def inputs_name():
    from dense_gemm_f32_gb300 import inputs

    return inputs.SQUARE_8192.name


def main(argv=None):
    args = parse_args(argv)
    dist = Dist()
    if args.impl == "reference":
        return run_reference(args, dist)
    return run_ours(args, dist)


if __name__ == "__main__":
    sys.exit(main())
