"""Benchmark of the POET-X transformed linear on B300: one JSON line.

A step is one pass of the whole hot path on one batch: the Cayley-Neumann
blocks of both sides, the forward y = R (W0 (P x)) and the backward to dX and
the packed skew gradients, on the square 2048-wide layer (d_in = d_out = 2048,
8 + 8 blocks of b = 256, n = 3, 8192 bf16 tokens).  ``value`` is tokens/s with
the inputs resident in HBM; ``e2e`` is the same step through the C ABI with
host buffers (pinned host -> device copies of x and dy, device -> host copies
of y, dX and both skew gradients inside the timed region).

Usage:  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl poetx|reference]
For N > 1 launch one rank per GPU with torch.distributed.run; each rank runs
its own batch (weak scaling) and the packed skew gradients are all-reduced,
the data-parallel exchange of the method.
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from orthogonal_equivalence_neumann_b300 import TransformedLinear, _lib, dp, inputs  # noqa: E402

METRIC = "transformed-linear tokens/s (fwd+bwd) and Cayley-Neumann blocks/s; % of roofline"
CASE = inputs.SQUARE_2048
ROTATE = 4            # input sets cycled over the steps: 4 x (x + dy) = 268 MB > 126 MB L2
CPU_SAMPLE_FRACTION = 0.25   # cpu_baseline: 3 sampled steps of a quarter step each
REF_BUDGET_S = 90.0          # reference arm: wall time of warm-up plus timed oracle steps

# Peak of the fp32 FFMA pipes: 148 SMs x 128 lanes x 2 flop x 2.032 GHz.
ALU_FP32_PEAK_TFLOPS = 148 * 128 * 2 * 2.032e9 / 1e12


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0,
            "source": "fallback"}


def kernel_work(case):
    """Algorithmic work per launch of each kernel for one step of `case`:
    name -> (bound, flops per launch, bytes per launch)."""
    T, di, do, bi, bo, n = case.T, case.d_in, case.d_out, case.b_in, case.b_out, case.n
    es = 2 if case.dtype == "bf16" else 4
    nbi, nbo = di // bi, do // bo
    gemm_flops = 2.0 * T * di * do
    gemm_bytes = es * (T * di + di * do + T * do)
    blk_flops = (2.0 * T * di * bi + 2.0 * T * do * bo) / 2      # mean over the P and R sides
    blk_bytes = es * (2 * T * di + 2 * T * do) / 2
    dq_flops = (2.0 * T * di * bi + 2.0 * T * do * bo) / 2
    dq_bytes = es * (2 * T * di + 2 * T * do) / 2 + 4 * (di * bi + do * bo) / 2
    cnp_f = (2.0 * n * bi ** 3 * nbi + 2.0 * n * bo ** 3 * nbo) / 2
    cnp_fb = 4 * (nbi * bi * (bi - 1) / 2 + nbo * bo * (bo - 1) / 2) / 2 + es * (nbi * bi * bi + nbo * bo * bo) / 2
    cnpb_f = 3 * cnp_f
    cnpb_b = 4 * (nbi * bi * bi + nbo * bo * bo) / 2 + 8 * (nbi * bi * (bi - 1) / 2 + nbo * bo * (bo - 1) / 2) / 2
    nbb = nbi * bi * bi + nbo * bo * bo                 # entries of all blocks of both sides
    npk = nbi * bi * (bi - 1) / 2 + nbo * bo * (bo - 1) / 2  # packed parameters of both sides
    return {
        "gemm_simt": ("alu", gemm_flops, gemm_bytes),
        "block_apply_simt": ("alu", blk_flops, blk_bytes),
        "dq_simt": ("alu", dq_flops, dq_bytes),
        "cnp_fwd_simt": ("alu", cnp_f, cnp_fb),
        "cnp_bwd_simt": ("alu", cnpb_f, cnpb_b),
        # tensor-core path (one launch per product; the CNP kernels serve both sides)
        "tc_gemm_nt": ("tensor", gemm_flops, gemm_bytes),
        "tc_gemm_nn": ("tensor", gemm_flops, gemm_bytes),
        "tc_blockapply_gather": ("hbm", blk_flops, blk_bytes),
        "tc_blockapply_scatter": ("hbm", blk_flops, blk_bytes),
        "tc_cluster_gather": ("hbm", blk_flops, blk_bytes),
        "tc_cluster_scatter": ("hbm", blk_flops, blk_bytes),
        "tc_plain_apply": ("hbm", blk_flops, blk_bytes),
        "tc_dq": ("hbm", dq_flops, dq_bytes),
        "tc_cluster_dq": ("hbm", dq_flops, dq_bytes),
        "tc_permute_cols": ("hbm", 0.0, es * (T * di + T * do)),
        "tc_cnp_tile": ("tensor", 2 * cnp_f, 4 * npk + 2 * nbb),
        "tc_cnp_tile_f32": ("tensor", 2 * cnp_f, 4 * npk + 4 * nbb),
        "tc_cnp_unpack": ("hbm", 0.0, 4 * npk + 2 * nbb),
        "tc_cnp_fwd": ("tensor", 2 * cnp_f, 2 * nbb + 2 * nbb),
        "tc_cnp_unpack_f32": ("hbm", 0.0, 4 * npk + 4 * nbb),
        "tc_cnp_fwd_f32": ("tensor", 2 * cnp_f, 4 * nbb + 4 * nbb),
        "tc_cnp_bwd_prep": ("hbm", 0.0, 4 * npk + 4 * nbb + 3 * 2 * nbb),
        "tc_cnp_bwd": ("tensor", 2 * cnpb_f, 3 * 2 * nbb + 4 * nbb + 4 * npk),
    }


def step_flops(case):
    T, di, do, bi, bo, n = case.T, case.d_in, case.d_out, case.b_in, case.b_out, case.n
    fwd = 2.0 * T * di * do + 2.0 * T * di * bi + 2.0 * T * do * bo
    bwd = fwd + 2.0 * T * di * bi + 2.0 * T * do * bo
    return fwd + bwd


def sources_sha(srcs):
    """sha1[:12] over the concatenated contents of comma-separated source paths."""
    h = hashlib.sha1()
    for src in srcs.split(","):
        path = os.path.join(ROOT, src)
        if not os.path.exists(path):
            return None
        h.update(open(path, "rb").read())
    return h.hexdigest()[:12]


def read_traffic(kernel):
    """Per-launch DRAM bytes of `kernel` from the committed ncu summary, if the
    kernel's sources are unchanged since the capture (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(p):
        return None
    for line in open(p):
        parts = line.split("#", 1)[0].split()
        if len(parts) == 4 and parts[0] == kernel:
            srcs, sha, nbytes = parts[1], parts[2], parts[3]
            if sources_sha(srcs) == sha:
                return float(nbytes)
    return None


class _CtypesNvml:
    """The few read-only NVML queries the clock sampler makes, bound with
    ctypes to the driver's libnvidia-ml when the pynvml module is absent."""
    NVML_CLOCK_SM = 1

    def __init__(self):
        import ctypes
        self._c = ctypes
        self._lib = ctypes.CDLL("libnvidia-ml.so.1")

    def _check(self, rc, what):
        if rc != 0:
            raise RuntimeError("%s returned %d" % (what, rc))

    def nvmlInit(self):
        self._check(self._lib.nvmlInit_v2(), "nvmlInit_v2")

    def _handle(self, fn, arg):
        h = self._c.c_void_p()
        self._check(fn(arg, self._c.byref(h)), fn.__name__)
        return h

    def nvmlDeviceGetHandleByPciBusId(self, bus):
        return self._handle(self._lib.nvmlDeviceGetHandleByPciBusId_v2, self._c.c_char_p(bus))

    def nvmlDeviceGetHandleByIndex(self, i):
        return self._handle(self._lib.nvmlDeviceGetHandleByIndex_v2, self._c.c_uint(i))

    def _clock(self, fn, h, kind):
        v = self._c.c_uint()
        self._check(fn(h, self._c.c_int(kind), self._c.byref(v)), fn.__name__)
        return v.value

    def nvmlDeviceGetClockInfo(self, h, kind):
        return self._clock(self._lib.nvmlDeviceGetClockInfo, h, kind)

    def nvmlDeviceGetMaxClockInfo(self, h, kind):
        return self._clock(self._lib.nvmlDeviceGetMaxClockInfo, h, kind)

    def nvmlDeviceGetCurrentClocksEventReasons(self, h):
        v = self._c.c_ulonglong()
        fn = getattr(self._lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self._lib.nvmlDeviceGetCurrentClocksThrottleReasons
        self._check(fn(h, self._c.byref(v)), "clock event reasons")
        return v.value


class ClockSampler:
    """SM clock and clock-event reasons sampled during the timed region.

    Reads NVML (the library nvidia-smi reports from) every few milliseconds
    from a background thread, so that even a short timed region gets samples;
    falls back to `nvidia-smi -lms` when NVML cannot be loaded.  Read-only:
    no GPU setting is changed."""
    REASONS = (("hw_slowdown", 0x8), ("hw_thermal_slowdown", 0x40),
               ("sw_thermal_slowdown", 0x20), ("sw_power_cap", 0x4),
               ("hw_power_brake_slowdown", 0x80))

    def __init__(self, gpu_index, period_s=0.002):
        self.gpu = gpu_index
        self.period = period_s
        self.samples = []       # (sm_mhz, reasons bitmask)
        self.max_mhz = None
        self._stop = None
        self._thread = None
        self.source = None

    def _loop(self, nv, h):
        while not self._stop.is_set():
            try:
                sm = nv.nvmlDeviceGetClockInfo(h, nv.NVML_CLOCK_SM)
                rs = nv.nvmlDeviceGetCurrentClocksEventReasons(h)
                self.samples.append((float(sm), int(rs)))
            except Exception:
                pass
            self._stop.wait(self.period)

    def __enter__(self):
        import threading
        try:
            try:
                import pynvml as nv
            except ImportError:
                nv = _CtypesNvml()
            nv.nvmlInit()
            h = None
            try:   # the NVML device of this CUDA device, by PCI address
                p = torch.cuda.get_device_properties(self.gpu)
                bus = "%08X:%02X:%02X.0" % (p.pci_domain_id, p.pci_bus_id, p.pci_device_id)
                h = nv.nvmlDeviceGetHandleByPciBusId(bus.encode())
            except Exception:
                h = nv.nvmlDeviceGetHandleByIndex(self.gpu)
            self.max_mhz = float(nv.nvmlDeviceGetMaxClockInfo(h, nv.NVML_CLOCK_SM))
            self._stop = threading.Event()
            self._thread = threading.Thread(target=self._loop, args=(nv, h), daemon=True)
            self._thread.start()
            self.source = "nvml"
        except Exception as e:   # NVML unusable here: sample through nvidia-smi instead
            self.nvml_error = repr(e)[:200]
            self._thread = None
            self._smi_start()
        return self

    def _smi_start(self):
        fields = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active")
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + fields,
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.proc.stdout.readline()    # running before the timed region starts
            self.source = "nvidia-smi"
        except OSError:
            self.proc = None

    def __exit__(self, *a):
        if self._thread is not None:
            self._stop.set()
            self._thread.join(timeout=5)
            return
        if getattr(self, "proc", None) is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            for line in out.splitlines():
                f = [x.strip() for x in line.split(",")]
                try:
                    self.samples.append((float(f[1]), int(f[4], 16)))
                    self.max_mhz = float(f[2])
                except (ValueError, IndexError):
                    continue

    def summary(self):
        sm = [s for s, _ in self.samples]
        reasons = sorted({nm for _, r in self.samples for nm, bit in self.REASONS if r & bit})
        out = {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": self.max_mhz,
               "reasons": reasons, "samples": len(sm), "source": self.source}
        if getattr(self, "nvml_error", None):
            out["nvml_error"] = self.nvml_error
        return out


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v, world):
    return dp.max_over_ranks(v) if world > 1 else v


def allreduce_grads(layer, world):
    """The data-parallel exchange: sum the packed skew gradients over ranks."""
    if world > 1:
        dp.allreduce_dtheta(layer.dtheta_P, layer.dtheta_R)


class OracleSample:
    """The CPU oracle (as it stands) on a proportional sample of the step.

    A fraction f of one step of `case`: f*T tokens of the forward and the
    backward (through the oracle's unmerged-weight, four-permutation path with
    the layer's Cayley-Neumann blocks), and f*(nb_P + nb_R) block
    Cayley-Neumann forward+backward evaluations (whole blocks, carried over
    from step to step by a credit counter), so each sampled step is the same
    mix of work as a full step, scaled by f.  Inputs are converted to float64
    once, outside the timing."""

    def __init__(self, case, inp):
        import oracle
        self.o = oracle
        self.case = case
        self.x = inp["x"].float().double().numpy()
        self.dy = inp["dy"].float().double().numpy()
        self.W0 = inp["W0"].float().double().numpy()
        self.thP = inp["theta_P"].double().numpy()
        self.thR = inp["theta_R"].double().numpy()
        self.pin = inp["perm_in"].numpy()
        self.pout = inp["perm_out"].numpy()
        self.QP = oracle.cnp(self.thP, case.b_in, case.n)
        self.QR = oracle.cnp(self.thR, case.b_out, case.n)
        self.dQP = np.zeros_like(self.QP)
        self.dQR = np.zeros_like(self.QR)
        self.credit = 0.0
        self.next_block = 0
        self.tok = 0

    def step(self, f):
        """Run one sampled step; returns (seconds, tokens credited = f*T)."""
        c, o = self.case, self.o
        nbi, nbo = c.d_in // c.b_in, c.d_out // c.b_out
        T_s = max(1, int(round(f * c.T)))
        t0 = time.perf_counter()
        self.credit += f * (nbi + nbo)
        while self.credit >= 1.0:
            j = self.next_block % (nbi + nbo)
            if j < nbi:
                th, b, dQ = self.thP[j:j + 1], c.b_in, self.dQP[j:j + 1]
            else:
                th, b, dQ = self.thR[j - nbi:j - nbi + 1], c.b_out, self.dQR[j - nbi:j - nbi + 1]
            o.cnp(th, b, c.n)
            o.cnp_backward(th, b, c.n, dQ)
            self.next_block += 1
            self.credit -= 1.0
        lo = self.tok % c.T
        hi = min(c.T, lo + T_s)
        x, dy = self.x[lo:hi], self.dy[lo:hi]
        o.forward(x, self.W0, self.QP, self.QR, self.pin, self.pout)
        _, self.dQP, self.dQR = o.backward(x, dy, self.W0, self.QP, self.QR, self.pin, self.pout)
        self.tok = hi % c.T
        return time.perf_counter() - t0, (hi - lo) * 1.0


def host_cores():
    return int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))


def run_reference(args, world, rank):
    """The reference arm: the CPU oracle, each step a proportional sample of the
    step sized so that warm-up plus timed steps take about REF_BUDGET_S."""
    if rank != 0:
        return
    inp = inputs.make_linear_inputs(CASE)
    smp = OracleSample(CASE, inp)
    cal_f = 1.0 / 64
    t_cal, _ = smp.step(cal_f)
    f = min(1.0 / 8, cal_f * REF_BUDGET_S / max(1, args.steps + args.warmup) / max(t_cal, 1e-6))
    f = max(f, 1.0 / CASE.T)
    for _ in range(args.warmup):
        smp.step(f)
    total, toks = 0.0, 0.0
    for _ in range(args.steps):
        dt, n = smp.step(f)
        total += dt
        toks += n
    value = toks / total
    sample = ("oracle on %.4g of each step: %d of %d tokens fwd+bwd and the matching share "
              "of the %d block Cayley-Neumann fwd+bwd, f64" % (
                  f, max(1, int(round(f * CASE.T))), CASE.T,
                  CASE.d_in // CASE.b_in + CASE.d_out // CASE.b_out))
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(world),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": host_cores(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def workload_config(world):
    return {"workload": "square_d2048_b256_n3_T8192 (POET-X transformed linear fwd+bwd)",
            "d_in": CASE.d_in, "d_out": CASE.d_out, "b": CASE.b_in, "n": CASE.n,
            "tokens_per_gpu": CASE.T, "global_batch_tokens": CASE.T * world,
            "parallelism": "dp%d" % world,
            "l2": "inputs rotate over %d sets of x and dy (%d MB > 126 MB L2)" % (
                ROTATE, ROTATE * 2 * CASE.T * CASE.d_in * 2 // 2 ** 20)}


def cnp_roofline_point(b, out_bytes, n, nblocks, seconds, peaks):
    """Roofline of one Cayley-Neumann generation call: algorithmic bytes (packed
    theta in, Q out) and flops (n products of b x b x b per block) against the
    measured HBM peak and the peak of the unit the products run on: bf16 Q on
    the bf16 tensor cores; fp32 Q on the tensor cores as three MMA chains of
    fp16 parts per product (so a third of the 16-bit peak)."""
    byts = nblocks * (4 * (b * (b - 1) // 2) + out_bytes * b * b)
    flops = nblocks * 2.0 * n * b ** 3
    t_hbm = byts / (peaks["hbm_gbs"] * 1e9)
    out = {"gbs": round(byts / seconds / 1e9, 1), "tflops": round(flops / seconds / 1e12, 2),
           "hbm_frac": round(t_hbm / seconds, 4)}
    if out_bytes == 2:
        unit, peak = "tensor", peaks["bf16_tflops"]
    else:
        unit, peak = "tensor_split3", peaks["bf16_tflops"] / 3
    t_c = flops / (peak * 1e12)
    out["bound"] = "hbm" if t_hbm >= t_c else unit
    out["frac"] = round(max(t_hbm, t_c) / seconds, 4)
    return out


def cnp_points(dev, peaks):
    """Cayley-Neumann generation throughput at 4096 blocks, n = 3, sigma = 1e-2,
    and each point's roofline fraction."""
    out, roof = {}, {}
    for b in (32, 64, 128, 256):
        th = inputs.make_theta(4096, b, 1e-2, inputs.sweep_seed(b, 1e-2, 3)).to(dev)
        for dt, nm in ((torch.float32, "f32"), (torch.bfloat16, "bf16")):
            Q = torch.empty(4096, b, b, dtype=dt, device=dev)
            for _ in range(2):
                _lib.poetx_cayley_neumann(th, b, 3, Q)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            reps = 5
            torch.cuda.synchronize()
            e0.record()
            for _ in range(reps):
                _lib.poetx_cayley_neumann(th, b, 3, Q)
            e1.record()
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1) / reps
            out["b%d_%s" % (b, nm)] = round(4096 / (ms * 1e-3))
            roof["b%d_%s" % (b, nm)] = cnp_roofline_point(b, Q.element_size(), 3, 4096, ms * 1e-3,
                                                          peaks)
        del th, Q
    return out, roof


def fold_point(lay, dev, peaks):
    """End-of-inner-loop fold W0_new = R W0 P (poetx_fold_w0) at the layer's
    shape, into a scratch matrix (the layer is left as it is)."""
    need = _lib.poetx_fold_workspace_bytes(lay.d_out, lay.d_in, lay.b_in, lay.b_out, lay.dtype)
    ws = torch.empty(need, dtype=torch.uint8, device=dev)
    out = torch.empty_like(lay.W0m)
    lay.cayley_neumann()

    def fold():
        _lib.poetx_fold_w0(lay.W0m, lay.Q_P, lay.Q_R, lay.perm_in, lay.perm_out, lay.b_in,
                           lay.b_out, out, ws)

    for _ in range(3):
        fold()
    reps = 10
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record()
    for _ in range(reps):
        fold()
    e1.record()
    torch.cuda.synchronize()
    us = 1e3 * e0.elapsed_time(e1) / reps
    es = lay.W0m.element_size()
    alg = es * (2 * lay.d_out * lay.d_in + lay.d_in * lay.b_in + lay.d_out * lay.b_out)
    gbs = alg / (us * 1e-6) / 1e9
    del ws, out
    return {"us": round(us, 2), "algorithmic_bytes": alg, "achieved_gbs": round(gbs, 1),
            "frac": round(gbs / peaks["hbm_gbs"], 4),
            "passes": "two scattered block applies and two transposes",
            "note": "the weight and the intermediate fit in L2 at this shape"}


def xq_point(case, inp, lay, xs, dys, y, dX, dev):
    """POET-XQ at the bench shape: the weight kept as INT8 codes + per-row
    scales, dequantised into the workspace by every forward and backward.
    Eager steps of the XQ layer beside eager steps of the bf16 layer (same
    inputs, same loop), and the dequantisation alone."""
    xq = TransformedLinear(inp["W0"].to(dev), inp["theta_P"], inp["theta_R"], inp["perm_in"],
                           inp["perm_out"], case.b_in, case.b_out, case.n, T_max=case.T,
                           save_z=True, device=dev, w0_int8=True)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def timed(fn, reps):
        for k in range(3):
            fn(k)
        torch.cuda.synchronize()
        e0.record()
        for k in range(reps):
            fn(k)
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps

    reps = 20
    ms_xq = timed(lambda k: xq.step(xs[k % len(xs)], dys[k % len(dys)], y, dX), reps)
    ms_bf16 = timed(lambda k: lay.step(xs[k % len(xs)], dys[k % len(dys)], y, dX), reps)
    Wd = torch.empty(case.d_out, case.d_in, dtype=torch.bfloat16, device=dev)
    us_deq = 1e3 * timed(lambda k: _lib.poetx_dequantize_w0(xq.W0q, xq.w0_scale, Wd), 50)
    out = {"ms_per_step_eager": round(ms_xq, 4), "bf16_ms_per_step_eager": round(ms_bf16, 4),
           "dequantize_us": round(us_deq, 2),
           "resident_w0_bytes": xq.W0q.numel() + 4 * xq.w0_scale.numel(),
           "bf16_w0_bytes": 2 * case.d_out * case.d_in}
    del xq, Wd
    return out


def config_points(dev, peaks, reps=20):
    """Graph-replayed steps of the workloads' other layer shapes: the MLP
    up-projection 2048 -> 5632 (b = 128, 16384 tokens) and the three linear
    shapes of the 1B-style stack (b = 256, 8192 tokens).  Each shape cycles
    ROTATE input sets, so the inputs of consecutive replays do not sit in L2.
    Measured after the headline; a failure here is reported in place of these
    numbers."""
    out = {}
    try:
        st = inputs.stack_cases(layers=1)
        cases = [("upproj_2048x5632_b128_T16384", inputs.UPPROJ), ("stack_qkvo_2048x2048", st[0]),
                 ("stack_gate_up_2048x5632", st[4]), ("stack_down_5632x2048", st[6])]
        for name, case in cases:
            inp = inputs.make_linear_inputs(case)
            lay = TransformedLinear(inp["W0"].to(dev), inp["theta_P"], inp["theta_R"],
                                    inp["perm_in"], inp["perm_out"], case.b_in, case.b_out, case.n,
                                    T_max=case.T, save_z=True, device=dev)
            gen = torch.Generator(device=dev).manual_seed(977)
            xs = [inp["x"].to(dev)] + [torch.randn(case.T, case.d_in, generator=gen, device=dev).to(
                torch.bfloat16) for _ in range(ROTATE - 1)]
            dys = [inp["dy"].to(dev)] + [torch.randn(case.T, case.d_out, generator=gen,
                                                     device=dev).to(torch.bfloat16)
                                         for _ in range(ROTATE - 1)]
            y = torch.empty(case.T, case.d_out, dtype=torch.bfloat16, device=dev)
            dX = torch.empty(case.T, case.d_in, dtype=torch.bfloat16, device=dev)
            graphs = [lay.capture_step(xs[k], dys[k], y, dX) for k in range(ROTATE)]
            for g in graphs:
                g.replay()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for k in range(reps):
                graphs[k % ROTATE].replay()
            e1.record()
            torch.cuda.synchronize()
            _lib.poetx_stream_status()
            ms = e0.elapsed_time(e1) / reps
            fl = step_flops(case)
            out[name] = {"ms_per_step": round(ms, 4), "tokens_per_s": round(case.T / (ms * 1e-3)),
                         "tflops": round(fl / (ms * 1e-3) / 1e12, 1),
                         "frac_of_bf16_peak": round(fl / (ms * 1e-3) / 1e12 / peaks["bf16_tflops"], 4)}
            del lay, graphs, xs, dys, y, dX
            torch.cuda.empty_cache()
        out["stack_16_layers"] = stack_point(dev, peaks)
    except Exception as e:   # noqa: BLE001 -- reported, the headline stands
        out["error"] = repr(e)[:300]
    return out


def link_bandwidth(dev, mb=64, reps=10):
    """Pinned host <-> device copy bandwidth of this GPU's link, measured alone:
    one direction at a time, then both at once on two streams (as the
    end-to-end loop moves them), GB/s from CUDA events."""
    n = mb << 20
    h_src = torch.empty(n, dtype=torch.uint8).pin_memory()
    h_dst = torch.empty(n, dtype=torch.uint8).pin_memory()
    d_a = torch.empty(n, dtype=torch.uint8, device=dev)
    d_b = torch.empty(n, dtype=torch.uint8, device=dev)
    s1, s2 = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)

    def timed(st, fn):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        fn()
        torch.cuda.synchronize()
        e0.record(st)
        for _ in range(reps):
            fn()
        e1.record(st)
        torch.cuda.synchronize()
        return n * reps / (e0.elapsed_time(e1) * 1e-3) / 1e9

    with torch.cuda.stream(s1):
        h2d = timed(s1, lambda: d_a.copy_(h_src, non_blocking=True))
        d2h = timed(s1, lambda: h_dst.copy_(d_b, non_blocking=True))
    # both directions at once: each stream's own events over the same interval
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    ev[0].record(s1)
    ev[2].record(s2)
    for _ in range(reps):
        with torch.cuda.stream(s1):
            d_a.copy_(h_src, non_blocking=True)
        with torch.cuda.stream(s2):
            h_dst.copy_(d_b, non_blocking=True)
    ev[1].record(s1)
    ev[3].record(s2)
    torch.cuda.synchronize()
    c_h2d = n * reps / (ev[0].elapsed_time(ev[1]) * 1e-3) / 1e9
    c_d2h = n * reps / (ev[2].elapsed_time(ev[3]) * 1e-3) / 1e9
    del h_src, h_dst, d_a, d_b
    return {"h2d_gbs": round(h2d, 1), "d2h_gbs": round(d2h, 1), "concurrent_h2d_gbs": round(c_h2d, 1),
            "concurrent_d2h_gbs": round(c_d2h, 1), "copy_mb": mb}


def stack_point(dev, peaks, steps=3):
    """The 1B-style stack measured as one training step: 16 layers x 7 linears
    (q, k, v, o 2048 -> 2048; gate, up 2048 -> 5632; down 5632 -> 2048), i.e.
    112 layers each with its own frozen weight (1.64 GB of W0 in all),
    parameters and permutations, and a fresh synthetic activation per linear
    (seeded device draws with the workload's distributions).  One step = the
    Cayley-Neumann blocks and forward of every linear in order, then the
    backward of every linear in reverse order (each keeps its own z), captured
    into one CUDA graph and replayed; the linears share one workspace."""
    cases = inputs.stack_cases()
    bf = torch.bfloat16
    gen = torch.Generator(device=dev).manual_seed(2468)
    cpu = torch.Generator().manual_seed(2469)
    need = max(_lib.poetx_workspace_bytes(c.T, c.d_in, c.d_out, c.b_in, c.b_out, bf) for c in cases)
    ws = torch.empty(need, dtype=torch.uint8, device=dev)
    lays, xs, dys = [], [], []
    for c in cases:
        W0 = (torch.randn(c.d_out, c.d_in, generator=gen, device=dev) * c.d_in ** -0.5).to(bf)
        thP = torch.randn(c.d_in // c.b_in, c.b_in * (c.b_in - 1) // 2, generator=gen,
                          device=dev) * c.sigma
        thR = torch.randn(c.d_out // c.b_out, c.b_out * (c.b_out - 1) // 2, generator=gen,
                          device=dev) * c.sigma
        pi = torch.randperm(c.d_in, generator=cpu).to(torch.int32)
        po = torch.randperm(c.d_out, generator=cpu).to(torch.int32)
        lays.append(TransformedLinear(W0, thP, thR, pi, po, c.b_in, c.b_out, c.n, T_max=c.T,
                                      save_z=True, device=dev, workspace=ws))
        xs.append(torch.randn(c.T, c.d_in, generator=gen, device=dev).to(bf))
        dys.append(torch.randn(c.T, c.d_out, generator=gen, device=dev).to(bf))
    outs = {d: torch.empty(cases[0].T, d, dtype=bf, device=dev) for d in (2048, 5632)}

    def step():
        for lay, x in zip(lays, xs):
            lay.cayley_neumann()
            lay.forward(x, outs[lay.d_out])
        for lay, x, dy in zip(reversed(lays), reversed(xs), reversed(dys)):
            lay.backward(x, dy, outs[lay.d_in])

    side = torch.cuda.Stream(device=dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream(dev).wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, capture_error_mode="relaxed"):
        step()
    graph.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        graph.replay()
    e1.record()
    torch.cuda.synchronize()
    _lib.poetx_stream_status()
    ms = e0.elapsed_time(e1) / steps
    fl = sum(step_flops(c) for c in cases)
    w0_bytes = sum(2 * c.d_in * c.d_out for c in cases)
    del graph, lays, xs, dys, outs, ws
    torch.cuda.empty_cache()
    return {"ms_per_step": round(ms, 3), "tokens_per_s": round(cases[0].T / (ms * 1e-3)),
            "tflops": round(fl / (ms * 1e-3) / 1e12, 1),
            "frac_of_bf16_peak": round(fl / (ms * 1e-3) / 1e12 / peaks["bf16_tflops"], 4),
            "linears": len(cases), "w0_bytes": w0_bytes, "steps": steps,
            "measured": "one CUDA graph: forward of the 112 linears in order, then their "
                        "backward in reverse order"}


def run_poetx(args, world, rank, local):
    dev = torch.device("cuda", local)
    peaks = load_peaks()
    case = CASE
    inp = inputs.make_linear_inputs(case)
    lay = TransformedLinear(inp["W0"].to(dev), inp["theta_P"], inp["theta_R"], inp["perm_in"],
                            inp["perm_out"], case.b_in, case.b_out, case.n, T_max=case.T,
                            save_z=True, device=dev)
    # rotating input sets: set 0 is the seeded draw; the others are seeded device draws
    gen = torch.Generator(device=dev).manual_seed(4242 + rank)
    xs = [inp["x"].to(dev)] + [torch.randn(case.T, case.d_in, generator=gen, device=dev).to(
        torch.bfloat16) for _ in range(ROTATE - 1)]
    dys = [inp["dy"].to(dev)] + [torch.randn(case.T, case.d_out, generator=gen, device=dev).to(
        torch.bfloat16) for _ in range(ROTATE - 1)]
    y = torch.empty(case.T, case.d_out, dtype=torch.bfloat16, device=dev)
    dX = torch.empty(case.T, case.d_in, dtype=torch.bfloat16, device=dev)

    def step(k):
        lay.step(xs[k % ROTATE], dys[k % ROTATE], y, dX)
        allreduce_grads(lay, world)

    for k in range(args.warmup):
        step(k)
    _lib.poetx_stream_status()
    torch.cuda.synchronize()

    # ---------------- CUDA graphs: one step per input set, and a profiled copy of each
    # (event pairs around every kernel, recorded as graph nodes) for the per-kernel
    # durations; the profiled copies run as the last steps of the timed region.
    graphs = [lay.capture_step(xs[k], dys[k], y, dX) for k in range(ROTATE)]
    torch.cuda.synchronize()
    n0 = _lib.poetx_launch_count()
    _lib.poetx_profile_report()   # drop anything recorded so far
    _lib.poetx_profile_enable(True)
    pgraphs = [lay.capture_step(xs[k], dys[k], y, dX, warm=False) for k in range(ROTATE)]
    _lib.poetx_profile_enable(False)
    launches_per_step = (_lib.poetx_launch_count() - n0) / ROTATE
    torch.cuda.synchronize()
    for g in graphs + pgraphs:   # first replays upload the graphs (the profiled copies'
        g.replay()               # event pairs are read after their replays in the timed region)
    torch.cuda.synchronize()
    n_prof = min(ROTATE, args.steps)

    def gstep(k, prof):
        (pgraphs if prof else graphs)[k % ROTATE].replay()
        allreduce_grads(lay, world)

    # ---------------- timed region (device-resident inputs)
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        barrier(world)
        torch.cuda.synchronize()
        torch.cuda.nvtx.range_push("poetx_timed")
        e0.record(stream)
        for k in range(args.steps - n_prof):
            gstep(k, False)
        for k in range(args.steps - n_prof, args.steps):
            gstep(k, True)
        e1.record(stream)
        torch.cuda.nvtx.range_pop()
        torch.cuda.synchronize()
        barrier(world)
    _lib.poetx_stream_status()
    launches = launches_per_step * args.steps
    ms = max_over_ranks(e0.elapsed_time(e1), world)
    ms_per_step = ms / args.steps
    value = world * case.T * args.steps / (ms * 1e-3)
    timing_src = "event nodes around each kernel in the last %d graph replays of the timed region" % n_prof
    try:
        prof = _lib.poetx_profile_report()
    except Exception:   # events recorded by graph nodes not readable: an eager profiled pass
        timing_src = "event pairs around each kernel in %d eager steps after the timed region" % ROTATE
        _lib.poetx_profile_enable(True)
        for k in range(ROTATE):
            step(k)
        _lib.poetx_profile_enable(False)
        prof = _lib.poetx_profile_report()

    # ---------------- roofline of the dominant kernel
    work = kernel_work(case)
    dom = max(prof.items(), key=lambda kv: kv[1][1])
    dname, (dcnt, dms) = dom
    bound, flops, nbytes = work.get(dname, ("alu", float("nan"), float("nan")))
    avg_s = dms / dcnt * 1e-3
    if bound == "tensor":
        peak = peaks["bf16_tflops"]
        achieved, unit = flops / avg_s / 1e12, "TFLOP/s"
    elif bound == "hbm":
        peak = peaks["hbm_gbs"]
        achieved, unit = nbytes / avg_s / 1e9, "GB/s"
    else:
        peak = ALU_FP32_PEAK_TFLOPS
        achieved, unit = flops / avg_s / 1e12, "TFLOP/s"
    total_ms = sum(v[1] for v in prof.values())
    roofline = {"bound": bound, "kernel": dname, "achieved": round(achieved, 2),
                "peak": round(peak, 1), "unit": unit, "frac": round(achieved / peak, 4),
                "traffic": read_traffic(dname),
                "peak_source": "fp32 FFMA 148x128x2x2.032GHz" if bound == "alu" else peaks["source"],
                "share": round(dms / total_ms, 4) if total_ms else None,
                "timing": timing_src,
                "kernels": {k: {"launches": v[0], "us_per_launch": round(v[1] / v[0] * 1e3, 2)}
                            for k, v in prof.items()}}

    # ---------------- end to end through host buffers
    # Every step's inputs come from pinned host memory and every step's results
    # (y, dX, both skew gradients) go back to it, inside the timed region; as a
    # training loop would, the copies run on their own streams with two device
    # buffer sets, so step k's upload and step k-1's download overlap step k's
    # compute (the compute calls are the public API's, eager).
    NB = 2
    h_x = [t.cpu().pin_memory() for t in xs[:2]]
    h_dy = [t.cpu().pin_memory() for t in dys[:2]]
    d_x = [torch.empty_like(xs[0]) for _ in range(NB)]
    d_dy = [torch.empty_like(dys[0]) for _ in range(NB)]
    d_y = [torch.empty_like(y) for _ in range(NB)]
    d_dX = [torch.empty_like(dX) for _ in range(NB)]
    d_tp = [torch.empty_like(lay.dtheta_P) for _ in range(NB)]
    d_tr = [torch.empty_like(lay.dtheta_R) for _ in range(NB)]
    h_y = [torch.empty(y.shape, dtype=y.dtype).pin_memory() for _ in range(NB)]
    h_dX = [torch.empty(dX.shape, dtype=dX.dtype).pin_memory() for _ in range(NB)]
    h_tp = [torch.empty(lay.dtheta_P.shape, dtype=torch.float32).pin_memory() for _ in range(NB)]
    h_tr = [torch.empty(lay.dtheta_R.shape, dtype=torch.float32).pin_memory() for _ in range(NB)]
    copy_in = torch.cuda.Stream(device=dev)
    copy_out = torch.cuda.Stream(device=dev)
    in_ready = [torch.cuda.Event() for _ in range(NB)]
    computed = [torch.cuda.Event() for _ in range(NB)]
    out_done = [torch.cuda.Event() for _ in range(NB)]

    def upload(k):
        b = k % NB
        with torch.cuda.stream(copy_in):
            copy_in.wait_event(computed[b])       # step k - NB is done with these buffers
            d_x[b].copy_(h_x[k % 2], non_blocking=True)
            d_dy[b].copy_(h_dy[k % 2], non_blocking=True)
            in_ready[b].record(copy_in)

    # the compute of a step is the same captured graph as in the timed region,
    # one per device buffer set
    egraphs = [lay.capture_step(d_x[b], d_dy[b], d_y[b], d_dX[b]) for b in range(NB)]

    def e2e_step(k):
        b = k % NB
        stream.wait_event(in_ready[b])
        stream.wait_event(out_done[b])            # step k - NB's results have left
        egraphs[b].replay()
        allreduce_grads(lay, world)
        d_tp[b].copy_(lay.dtheta_P, non_blocking=True)
        d_tr[b].copy_(lay.dtheta_R, non_blocking=True)
        computed[b].record(stream)
        with torch.cuda.stream(copy_out):
            copy_out.wait_event(computed[b])
            h_y[b].copy_(d_y[b], non_blocking=True)
            h_dX[b].copy_(d_dX[b], non_blocking=True)
            h_tp[b].copy_(d_tp[b], non_blocking=True)
            h_tr[b].copy_(d_tr[b], non_blocking=True)
            out_done[b].record(copy_out)

    def e2e_run(n):
        copy_in.wait_stream(stream)
        upload(0)
        for k in range(n):
            if k + 1 < n:
                upload(k + 1)
            e2e_step(k)
        stream.wait_stream(copy_out)
        stream.wait_stream(copy_in)

    e2e_run(2)
    torch.cuda.synchronize()
    barrier(world)
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    e2e_run(args.steps)
    f1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    e2e_ms = max_over_ranks(f0.elapsed_time(f1), world)
    h2d = (d_x[0].numel() + d_dy[0].numel()) * 2
    d2h = (y.numel() + dX.numel()) * 2 + 4 * (h_tp[0].numel() + h_tr[0].numel())
    link = link_bandwidth(dev)
    # the bound the host link alone sets: both directions overlapped with the compute
    t_link = max(h2d / (link["concurrent_h2d_gbs"] * 1e9), d2h / (link["concurrent_d2h_gbs"] * 1e9))
    e2e = {"value": world * case.T * args.steps / (e2e_ms * 1e-3), "unit": "tokens/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
           "copies": "pinned host buffers; uploads and downloads on their own streams, "
                     "double-buffered; compute as the captured step graph",
           "link": link, "link_bound_tokens_per_s": round(case.T / t_link),
           "frac_of_link_bound": round(world * case.T * args.steps / (e2e_ms * 1e-3) /
                                       (world * case.T / t_link), 4)}

    cnp, cnp_roof = cnp_points(dev, peaks) if rank == 0 else (None, None)
    fold = fold_point(lay, dev, peaks) if rank == 0 else None
    xq = xq_point(case, inp, lay, xs, dys, y, dX, dev) if rank == 0 else None
    cfgs = config_points(dev, peaks) if rank == 0 and world == 1 else None

    # ---------------- CPU oracle baseline (rank 0, N = 1 only)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        smp = OracleSample(case, inp)
        secs, toks = 0.0, 0.0
        for _ in range(3):
            dt, n = smp.step(CPU_SAMPLE_FRACTION)
            secs += dt
            toks += n
        cpu = {"value": toks / secs, "unit": "tokens/s", "cores": host_cores(), "kind": "oracle",
               "sample": "3 x %.2f of one step (%d tokens fwd+bwd and the matching share of the "
                         "block Cayley-Neumann fwd+bwd each), f64, %.1f s"
                         % (CPU_SAMPLE_FRACTION, int(CPU_SAMPLE_FRACTION * case.T), secs)}

    if rank == 0:
        flops = step_flops(case)
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic", "config": workload_config(world),
            "step_tflops": round(flops / (ms_per_step * 1e-3) / 1e12 / 1, 2),
            "step_frac_of_bf16_peak": round(flops / (ms_per_step * 1e-3) / 1e12 / peaks["bf16_tflops"], 4),
            "cnp_blocks_per_s": cnp, "cnp_roofline": cnp_roof, "fold_w0": fold, "xq": xq, "other_shapes": cfgs, "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": int(launches), "clocks": clk.summary(),
        }
        print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="poetx", choices=["poetx", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    world, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        if not torch.cuda.is_available():
            raise SystemExit("bench.py: no CUDA device (the library has no CPU path)")
        run_poetx(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
