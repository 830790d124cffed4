"""Benchmark: dense tensor-core GEMM on one GB300 (BF16 and FP8 E4M3).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

A step is one call of the library on the headline workload, the BF16
4096 x 4096 x 4096 GEMM (A, B ~ N(0,1) rounded to BF16, BF16 output), the
square problem of "Tensor Cores: Matrix Instructions, Swizzling and FP8,
Measured" (Step 2).  One step's inputs (67 MB) would fit in the 129 MB L2, so
the steps cycle through enough copies of the inputs (5) that every step reads
operands that are not in L2.  The K timed steps run back to back from one
CUDA graph, between one pair of CUDA events.  The metric is
TFLOPS = 2*M*N*K / time.

Rank 0 prints one JSON line.  With N > 1 (torchrun) every rank runs its own
replica of the workload (GEMMs shard without any exchange; "replicas only"),
times are maxed over ranks, and value = all ranks' FLOPs / that time.

--impl reference times the CPU oracle (the plain FP64 reference of the same
GEMM) on the host cores, on a bounded sample of output tiles per step.
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_BF16_TFLOPS = 1900.0
FP8_OVER_BF16 = 2.0   # nominal dense ratio (4.5 / 2.25 PFLOP/s)


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def kernel_source_sha(files=None):
    """sha256 over CUDA sources (all of csrc/, or the named files), to tell
    whether a stored ncu figure is still current."""
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "tensor_core_dense_gb300", "csrc")
    for name in sorted(files or os.listdir(csrc)):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()


def stored_traffic(summary="gemm_tn2_bf16_4096.md"):
    """DRAM bytes per launch from the committed ncu summary, or None when the
    summary is missing or was taken on different kernel sources."""
    path = os.path.join(ROOT, "profiles", summary)
    try:
        fields = {}
        with open(path) as f:
            for line in f:
                if ":" in line and line.strip().startswith(
                        ("source_sha256", "source_files", "traffic_bytes")):
                    k, v = line.split(":", 1)
                    fields[k.strip()] = v.strip().strip("`")
        files = fields.get("source_files", "").split() or None
        if fields.get("source_sha256") != kernel_source_sha(files):
            return None
        return int(fields["traffic_bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        return None


def peaks():
    try:
        with open(PEAKS_FILE) as f:
            p = json.load(f)
        return float(p["bf16_tflops"]), float(p.get("hbm_gbs", 6800.0)), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_BF16_TFLOPS, 6800.0, "fallback"


def sustained_peak():
    """The measured bf16 rate of a seconds-long GEMM loop under the power cap."""
    try:
        with open(PEAKS_FILE) as f:
            return float(json.load(f)["bf16_tflops_sustained"])
    except (OSError, KeyError, ValueError):
        return None


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi clock / throttle-reason samples every `ms` milliseconds."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_id: str, ms: int = 50):
        self.proc = None
        self.t0 = time.time()
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", device_id, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(ms)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return []
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = []
        for line in out.splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                mask = int(f[4], 16)
            except ValueError:
                mask = 0
            try:
                rows.append(dict(sm=float(f[1]), max=float(f[2]),
                                 power=float(f[3]) if f[3] not in ("[N/A]", "") else 0.0,
                                 hw=f[5], hw_thermal=f[6], sw_thermal=f[7], sw_power=f[8],
                                 mask=mask))
            except ValueError:
                continue
        return rows

    # every clock-event reason bit the driver defines, for the raw masks
    REASON_BITS = ((0x1, "gpu_idle"), (0x2, "applications_clocks_setting"),
                   (0x4, "sw_power_cap"), (0x8, "hw_slowdown"), (0x10, "sync_boost"),
                   (0x20, "sw_thermal_slowdown"), (0x40, "hw_thermal_slowdown"),
                   (0x80, "hw_power_brake_slowdown"), (0x100, "display_clock_setting"))

    @staticmethod
    def summary(rows):
        """Median SM clock and the throttle reasons seen: `reasons` the four the
        timing rules act on, `reasons_mask` the OR of every raw reason mask
        sampled and `other_reasons` its remaining bits by name."""
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        reasons = set()
        mask = 0
        for r in rows:
            for k, name in (("hw", "hw_slowdown"), ("hw_thermal", "hw_thermal_slowdown"),
                            ("sw_thermal", "sw_thermal_slowdown"), ("sw_power", "sw_power_cap")):
                if r[k].lower().startswith("active"):
                    reasons.add(name)
            mask |= int(r.get("mask", 0))
        other = sorted(name for bit, name in ClockSampler.REASON_BITS
                       if mask & bit and name not in reasons and
                       name not in ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                                    "sw_power_cap"))
        return {"sm_mhz": statistics.median(r["sm"] for r in rows),
                "sm_max_mhz": max(r["max"] for r in rows),
                "power_w_max": max(r["power"] for r in rows),
                "reasons": sorted(reasons), "reasons_mask": hex(mask),
                "other_reasons": other, "samples": len(rows),
                **({"mem_mhz_min": min(r["mem"] for r in rows),
                    "mem_mhz_max": max(r["mem"] for r in rows)}
                   if all("mem" in r for r in rows) else {})}


class NvmlSampler:
    """SM clock, power and clock-event reasons read through NVML (the driver's
    libnvidia-ml, read-only queries) every `ms` milliseconds on a thread, only
    while started: sized for timed regions of a few milliseconds, which an
    nvidia-smi process started beside the run cannot resolve.  Rows have the
    ClockSampler layout."""

    SW_POWER_CAP, HW_SLOWDOWN, SW_THERMAL, HW_THERMAL = 0x4, 0x8, 0x20, 0x40

    def __init__(self, device_uuid: str, ms: float = 1.0):
        import ctypes
        self.ms = ms
        self.rows = []
        self.thread = None
        self.running = False
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.lib = lib
        self.h = ctypes.c_void_p()
        if lib.nvmlDeviceGetHandleByUUID(device_uuid.encode(), ctypes.byref(self.h)) != 0:
            raise OSError("no NVML handle for " + device_uuid)
        self.reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons")
        mx = ctypes.c_uint()
        lib.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(mx))  # 1 = NVML_CLOCK_SM
        self.max_mhz = float(mx.value)

    def _sample(self):
        import ctypes
        c, pw, rs, mc = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong(), ctypes.c_uint()
        self.lib.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(c))
        self.lib.nvmlDeviceGetClockInfo(self.h, 2, ctypes.byref(mc))  # 2 = NVML_CLOCK_MEM
        self.lib.nvmlDeviceGetPowerUsage(self.h, ctypes.byref(pw))
        self.reasons_fn(self.h, ctypes.byref(rs))
        act = lambda bit: "Active" if rs.value & bit else "Not Active"  # noqa: E731
        self.rows.append(dict(sm=float(c.value), max=self.max_mhz, power=pw.value / 1000.0,
                              hw=act(self.HW_SLOWDOWN), hw_thermal=act(self.HW_THERMAL),
                              sw_thermal=act(self.SW_THERMAL), sw_power=act(self.SW_POWER_CAP),
                              mask=int(rs.value), mem=float(mc.value)))

    def _loop(self):
        while self.running:
            self._sample()
            time.sleep(self.ms / 1000.0)

    def start(self):
        import threading
        self.running = True
        self.thread = threading.Thread(target=self._loop, daemon=True)
        self.thread.start()

    def stop(self):
        self.running = False
        if self.thread is not None:
            self.thread.join()
        self._sample()  # at least one sample, taken right at the end of the region
        return self.rows


# -------------------------------------------------------------- our path

def _dist_init(args):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
    return world, rank, local


def _barrier_max(value, world):
    """Max of a float over ranks (and a barrier)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64,
                     device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_tflops(flops_per_step, steps, max_total_ms, world):
    """Whole-job throughput: every rank ran `steps` steps of `flops_per_step`;
    the job took the slowest rank's time."""
    return world * flops_per_step * steps / (max_total_ms * 1e-3) / 1e12


def _barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def device_tensors(w):
    import numpy as np
    import torch
    A = torch.from_numpy(w.A.view(np.int16)).cuda().view(torch.bfloat16) if w.kind == "bf16" \
        else torch.from_numpy(w.A).cuda()
    B = torch.from_numpy(w.B.view(np.int16)).cuda().view(torch.bfloat16) if w.kind == "bf16" \
        else torch.from_numpy(w.B).cuda()
    return A, B


def make_call(w, A, B, D, C=None, sa=None, sb=None):
    """A zero-argument closure that enqueues the library call on the current stream."""
    import torch

    import tensor_core_dense_gb300 as tcg
    if w.kind == "bf16":
        def call():
            tcg.gemm_bf16(A, B, D, C, alpha=w.alpha, beta=w.beta,
                          stream=torch.cuda.current_stream())
    elif w.kind == "fp8_mx":
        def call():
            tcg.gemm_mxfp8(A, B, sa, sb, D, C, a_format=w.a_fp8, b_format=w.b_fp8,
                           alpha=w.alpha, beta=w.beta, stream=torch.cuda.current_stream())
    else:
        mode = tcg.SCALE_TENSOR if w.kind == "fp8_tensor" else tcg.SCALE_BLOCK128

        def call():
            tcg.gemm_fp8_e4m3(A, B, sa, sb, D, C, mode=mode, alpha=w.alpha, beta=w.beta,
                              stream=torch.cuda.current_stream())
    return call


def l2_bytes():
    import torch
    try:
        return int(torch.cuda.get_device_properties(torch.cuda.current_device()).L2_cache_size)
    except (AttributeError, RuntimeError):
        return 129 << 20


def rotation_count(input_bytes):
    """Copies of the inputs to cycle through so no step finds its operands in
    L2: enough that 2x the L2 size streams by between two uses of a copy."""
    l2 = l2_bytes()
    if input_bytes >= 2 * l2:
        return 1
    return -(-2 * l2 // max(1, input_bytes)) + 1


class Rotation:
    """R device copies of a workload's inputs and outputs, with one library
    call closure per copy."""

    def __init__(self, w, copies=None):
        import numpy as np
        import torch
        inb = w.A.nbytes + w.B.nbytes + (w.C.nbytes if w.C is not None else 0)
        self.input_bytes = inb
        self.copies = copies or rotation_count(inb)
        self.calls = []
        self.tensors = []
        for _ in range(self.copies):
            A, B = device_tensors(w)
            D = torch.empty((w.M, w.N), dtype=torch.bfloat16 if w.out == "bf16" else torch.float32,
                            device="cuda")
            C = None
            if w.C is not None:
                C = torch.from_numpy(w.C.view(np.int16)).cuda().view(torch.bfloat16)
            if w.kind == "fp8_mx":  # E8M0 scale bytes
                sa, sb = torch.from_numpy(w.a_sf).cuda(), torch.from_numpy(w.b_sf).cuda()
            else:
                sa = torch.from_numpy(w.a_scale).cuda() if w.a_scale is not None else None
                sb = torch.from_numpy(w.b_scale).cuda() if w.b_scale is not None else None
            self.tensors.append((A, B, C, D, sa, sb))
            self.calls.append(make_call(w, A, B, D, C, sa, sb))

    def step(self, i):
        self.calls[i % self.copies]()

    def describe(self):
        mb = self.input_bytes / 1e6
        if self.copies == 1:
            return f"inputs larger than L2: {mb:.0f} MB per step (L2 {l2_bytes() / 1e6:.0f} MB)"
        return (f"inputs larger than L2: {self.copies} copies of the {mb:.0f} MB inputs are "
                f"cycled ({self.copies * mb:.0f} MB > L2 {l2_bytes() / 1e6:.0f} MB), so no step "
                f"finds its operands in L2")


def time_graph(rot, steps, warmup, sampler=None, replays=1, world=1):
    """Time `steps` back-to-back calls (cycling the copies) replayed from one
    CUDA graph, `replays` times; returns (list of ms per replay, kernel
    launches inside the graph, graph).  Each replay is bracketed by a barrier
    and a device synchronisation; a sampler (start/stop) runs around the timed
    replays only."""
    import torch

    import tensor_core_dense_gb300 as tcg
    for i in range(warmup):
        rot.step(i)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    n0 = tcg.launch_count()
    with torch.cuda.graph(g, stream=side):
        for i in range(steps):
            rot.step(i)
    launches = tcg.launch_count() - n0
    torch.cuda.synchronize()
    g.replay()  # one untimed replay
    torch.cuda.synchronize()
    times = []
    if sampler is not None:
        sampler.start()
    for _ in range(replays):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        _barrier(world)
        torch.cuda.synchronize()
        e0.record()
        g.replay()
        e1.record()
        torch.cuda.synchronize()
        _barrier(world)
        times.append(e0.elapsed_time(e1))
    if sampler is not None:
        sampler.stop()
    return times, launches, g


def isa_peak_tflops(sms, sm_mhz, fp8=False):
    """Dense tensor-core rate the instruction set allows at a clock: 8,192
    BF16 (16,384 FP8) FLOP per SM per clock x SMs x clock.  The per-SM figure
    is the B200 datasheet's, inferred in "How Blackwell's Tensor Memory
    Actually Works" (peak arithmetic); on GB300 ncu's tensor-pipe counter
    gives the same rate (about 8,200 BF16 and 16,400 FP8 FLOP/clk/SM)."""
    if not sms or not sm_mhz:
        return None
    return (16384.0 if fp8 else 8192.0) * sms * sm_mhz * 1e6 / 1e12


def add_peak_fractions(o, peak_bf16, sms, sm_mhz):
    """Adds to a GEMM workload's result `o` its fraction of the measured peak
    of its input type (FP8 -- per-tensor, block-scaled or microscaled -- at
    FP8_OVER_BF16 times the BF16 figure) and of the instruction-set rate at
    the sampled clock."""
    fp8 = "fp8" in o["workload"]
    if fp8:
        o["frac_of_fp8_peak"] = round(o["tflops"] / (peak_bf16 * FP8_OVER_BF16), 4)
    else:
        o["frac_of_bf16_peak"] = round(o["tflops"] / peak_bf16, 4)
    isa_o = isa_peak_tflops(sms, sm_mhz, fp8=fp8)
    if isa_o:
        o["frac_of_isa_peak_at_clock"] = round(o["tflops"] / isa_o, 4)
    return o


SECONDARY = ("bf16_256", "fp8_4096", "bf16_mlp", "fp8_skinny_16", "fp8_skinny_64",
             "fp8_skinny_128", "fp8_block_4096", "bf16_skinny_16", "mxfp8_4096")

# The FP8 quantiser on the operands the FP8 workloads cast: (seed, tensor id,
# rows, cols, granularity, outlier probability).  The values are the FP32
# tensors synth.workloads quantises on the host for fp8_4096 (A, per tensor)
# and fp8_skinny_M (A in 1 x 128 blocks, the 8192 x 8192 B in 128 x 128).
QUANT = {
    "quant_tensor_4096": (3, 1, 4096, 4096, "tensor", 0.0),
    "quant_row128_128": (5, 1, 128, 8192, "row128", 0.01),
    "quant_block128_8192": (5, 2, 8192, 8192, "block128", 0.01),
}


class QuantRotation:
    """Device copies of one quantiser workload (FP32 X, codes, scales), with
    one library call closure per copy, cycled so no call finds X in L2."""

    def __init__(self, name):
        import torch

        import synth
        import tensor_core_dense_gb300 as tcg
        seed, tensor, rows, cols, gran, outl = QUANT[name]
        x = synth.values_f32(seed, tensor, rows, cols, out_prob=outl, out_factor=50.0)
        self.rows, self.cols, self.granularity = rows, cols, gran
        mode = {"tensor": tcg.QUANT_TENSOR, "row128": tcg.QUANT_ROW128,
                "block128": tcg.QUANT_BLOCK128}[gran]
        nscale = tcg.quant_scale_count(rows, cols, mode)
        self.input_bytes = x.nbytes
        self.output_bytes = rows * cols + 4 * nscale
        self.copies = rotation_count(self.input_bytes + self.output_bytes)
        X0 = torch.from_numpy(x).cuda()
        self.calls, self.tensors = [], []
        for i in range(self.copies):
            X = X0 if i == 0 else X0.clone()
            Q = torch.empty((rows, cols), dtype=torch.uint8, device="cuda")
            S = torch.empty((nscale,), dtype=torch.float32, device="cuda")
            self.tensors.append((X, Q, S))
            self.calls.append(
                lambda X=X, Q=Q, S=S: tcg.quantize_e4m3(X, Q, S, mode=mode,
                                                        stream=torch.cuda.current_stream()))

    def step(self, i):
        self.calls[i % self.copies]()


def quant_config(name, steps, warmup, hbm_peak):
    """One quantiser workload: algorithmic bytes (X read once, codes and scales
    written once) per call over the mean call time."""
    rot = QuantRotation(name)
    times, launches, g = time_graph(rot, steps, warmup, replays=3)
    ms = statistics.median(times) / steps
    nbytes = rot.input_bytes + rot.output_bytes
    gbs = nbytes / (ms * 1e-3) / 1e9
    out = {"workload": name, "rows": rot.rows, "cols": rot.cols,
           "granularity": rot.granularity, "input": "f32", "us": round(ms * 1e3, 2),
           "gbs": round(gbs, 1), "frac_of_hbm": round(gbs / hbm_peak, 4),
           "kernels_per_call": launches // steps, "copies": rot.copies}
    del rot, g
    return out


def secondary_configs(steps=50, warmup=5, names=SECONDARY, size=None):
    """The other workloads, timed the same way (context beside the main line);
    size = (M, N, K) overrides a workload's shape (profiling a smaller case of
    the same kernel)."""
    import torch

    import synth.workloads as W
    out = []
    for name in names:
        if name in QUANT:
            out.append(quant_config(name, steps, warmup, peaks()[1]))
            torch.cuda.empty_cache()
            continue
        w = W.make(name) if size is None else W.make(name, M=size[0], N=size[1], K=size[2])
        rot = Rotation(w)
        times, _, g = time_graph(rot, steps, warmup, replays=3)
        ms = statistics.median(times) / steps
        out_bytes = w.M * w.N * (2 if w.out == "bf16" else 4)
        nbytes = rot.input_bytes + out_bytes
        nbytes += (w.a_scale.nbytes if w.a_scale is not None else 0) + (
            w.b_scale.nbytes if w.b_scale is not None else 0)
        nbytes += (w.a_sf.nbytes if w.a_sf is not None else 0) + (
            w.b_sf.nbytes if w.b_sf is not None else 0)
        out.append({"workload": name, "M": w.M, "N": w.N, "K": w.K,
                    "tflops": round(w.flops / (ms * 1e-3) / 1e12, 1),
                    "gbs": round(nbytes / (ms * 1e-3) / 1e9, 1), "us": round(ms * 1e3, 2),
                    "copies": rot.copies})
        del rot, g
        torch.cuda.empty_cache()
    return out


# Workloads the CPU baseline times, with their share of its time budget.
CPU_BASELINE = ("bf16_256", "bf16_4096", "fp8_4096", "bf16_mlp", "fp8_skinny_16",
                "fp8_skinny_64", "fp8_skinny_128")


def _oracle_tiles(w, tiles, cores):
    """The oracle as it stands on output tiles of a workload (values unused)."""
    import oracle
    in_type = oracle.IN_BF16 if w.kind == "bf16" else oracle.IN_E4M3
    mode = {"bf16": oracle.SCALE_NONE, "fp8_tensor": oracle.SCALE_TENSOR,
            "fp8_block": oracle.SCALE_BLOCK128}[w.kind]
    c_type = oracle.C_BF16 if (w.C is not None and w.C.dtype.name == "uint16") else oracle.C_F32
    return oracle.gemm(w.M, w.N, w.K, w.A, w.lda, w.B, w.ldb, in_type=in_type, scale_mode=mode,
                       a_scale=w.a_scale, b_scale=w.b_scale, C=w.C,
                       ldc=(w.C.shape[1] if w.C is not None else 0), c_type=c_type,
                       alpha=w.alpha, beta=w.beta, tiles=tiles, nthreads=cores)


def cpu_baseline_config(w, seconds, cores):
    """Oracle wall time on a fixed tile set of one workload: the whole output
    when it is small, else 128 x 128 tiles led by the first and the last tile
    (then seeded ones, the parity tests' sampler), in batches of one tile per
    core until about `seconds` have passed.  The full-output time is an
    extrapolation from the sampled rate."""
    import synth.workloads as W
    if w.M * w.N <= 256 * 256:
        tiles = [(0, 0, w.M, w.N)]
    else:
        tiles = W.sample_tiles(w.M, w.N, n=4096, size=128, seed=0)
    done_flops, t_used, ntiles = 0, 0.0, 0
    while ntiles < len(tiles) and (ntiles == 0 or t_used < seconds):
        batch = tiles[ntiles:ntiles + cores]
        t0 = time.perf_counter()
        _oracle_tiles(w, batch, cores)
        t_used += time.perf_counter() - t0
        done_flops += sum(2 * r * c * w.K for _, _, r, c in batch)
        ntiles += len(batch)
    rate = done_flops / t_used
    return {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "tiles": ntiles,
            "tile": "whole output" if len(tiles) == 1 else "128x128, first and last included",
            "wall_s": round(t_used, 3), "gflops_fp64": round(rate / 1e9, 3),
            "full_output_s_extrapolated": round(w.flops / rate, 1)}


def cpu_baseline_sample(w_main, seconds=24.0):
    """The oracle as it stands, timed on the host cores on every configured
    workload (see cpu_baseline_config); `value` is its rate on the headline
    workload in TFLOPS of FP64 reference work."""
    import oracle
    import synth.workloads as W
    cores = oracle.default_threads()
    per = []
    for name in CPU_BASELINE:
        w = w_main if name == w_main.name else W.make(name)
        per.append(cpu_baseline_config(w, seconds / len(CPU_BASELINE), cores))
    main = next(p for p in per if p["workload"] == w_main.name)
    return {"value": round(main["gflops_fp64"] / 1e3, 6), "unit": "TFLOPS", "cores": cores,
            "kind": "oracle",
            "sample": (f"{main['tiles']} output tiles of 128x128 (first and last included) of "
                       f"the {w_main.M}x{w_main.N}x{w_main.K} BF16 GEMM, FP64, "
                       f"{main['wall_s']:.1f} s; per_config lists every workload"),
            "per_config": per}


def run_ours(args):
    import numpy as np
    import torch

    import synth.workloads as W
    import tensor_core_dense_gb300 as tcg

    world, rank, local = _dist_init(args)
    torch.cuda.set_device(local)
    tcg.lib()
    w = W.make("bf16_4096")
    rot = Rotation(w)

    dev_uuid = str(torch.cuda.get_device_properties(local).uuid)
    smi_id = dev_uuid if dev_uuid.startswith("GPU-") else f"GPU-{dev_uuid}"
    # clocks during the timed replay: NVML polled every millisecond (the
    # region lasts milliseconds), else nvidia-smi around the whole run
    try:
        nvml = NvmlSampler(smi_id)
        sampler = None
    except (OSError, AttributeError):
        nvml = None
        sampler = ClockSampler(smi_id)
    # W warm-up steps, capture of the K timed steps, then R timed replays of
    # them, each with a barrier and a synchronize on both sides; the median
    # replay is the measurement
    _barrier(world)
    times, launches, graph = time_graph(rot, args.steps, args.warmup, nvml,
                                        replays=args.replays, world=world)
    _barrier(world)
    clocks = ClockSampler.summary(nvml.rows if nvml is not None else sampler.stop())
    clocks["source"] = ("nvml, 1 ms, timed replays only" if nvml is not None
                        else "nvidia-smi, 50 ms")
    assert tcg.last_device_status() == tcg.OK
    del graph

    total_ms = _barrier_max(statistics.median(times), world)
    ms_per_step = total_ms / args.steps
    value = aggregate_tflops(w.flops, args.steps, total_ms, world)
    replay_info = {"n": len(times), "statistic": "median",
                   "ms": [round(t, 4) for t in times],
                   "tflops_min": round(aggregate_tflops(w.flops, args.steps, max(times), world), 2),
                   "tflops_max": round(aggregate_tflops(w.flops, args.steps, min(times), world), 2)}

    # end to end through the public API with host buffers: every step copies
    # its A and B in from pinned host memory, runs the GEMM and copies D out.
    # Consecutive steps overlap on three streams (H2D, compute, D2H) over two
    # device slots, as a caller streaming batches would run it; events keep a
    # slot's inputs and output from being overwritten while still in use.
    slots = [(rot.tensors[i], rot.calls[i]) for i in range(2)]
    ha = torch.from_numpy(w.A.view(np.int16)).pin_memory()
    hb = torch.from_numpy(w.B.view(np.int16)).pin_memory()
    hds = [torch.empty((w.M, w.N), dtype=torch.int16).pin_memory() for _ in range(2)]
    s_in, s_gemm, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev = {k: [torch.cuda.Event() for _ in range(2)] for k in ("in", "gemm", "out")}
    e2e_steps = min(args.steps, 50)
    started = [False, False]

    def e2e_step(i):
        k = i % 2
        (A, B, _, D, _, _), call = slots[k]
        if started[k]:
            s_in.wait_event(ev["gemm"][k])       # the GEMM two steps back has read A, B
        with torch.cuda.stream(s_in):
            A.view(torch.int16).copy_(ha, non_blocking=True)
            B.view(torch.int16).copy_(hb, non_blocking=True)
            ev["in"][k].record(s_in)
        s_gemm.wait_event(ev["in"][k])
        if started[k]:
            s_gemm.wait_event(ev["out"][k])      # D two steps back has been copied out
        with torch.cuda.stream(s_gemm):
            call()
            ev["gemm"][k].record(s_gemm)
        s_out.wait_event(ev["gemm"][k])
        with torch.cuda.stream(s_out):
            hds[k].copy_(D.view(torch.int16), non_blocking=True)
            ev["out"][k].record(s_out)
        started[k] = True

    for i in range(4):
        e2e_step(i)
    torch.cuda.synchronize()
    _barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    cur = torch.cuda.current_stream()
    e0.record(cur)
    for st in (s_in, s_gemm, s_out):
        st.wait_event(e0)
    for i in range(e2e_steps):
        e2e_step(i)
    for st in (s_in, s_gemm, s_out):
        cur.wait_stream(st)
    e1.record(cur)
    torch.cuda.synchronize()
    e2e_ms = _barrier_max(e0.elapsed_time(e1), world)
    A, B, _, D, _, _ = slots[0][0]
    e2e_value = world * w.flops * e2e_steps / (e2e_ms * 1e-3) / 1e12

    peak_bf16, _, peak_src = peaks()
    achieved = w.flops / (ms_per_step * 1e-3) / 1e12
    sms = torch.cuda.get_device_properties(local).multi_processor_count
    isa = isa_peak_tflops(sms, clocks.get("sm_mhz"))
    region_ms = sum(times)
    line = {
        "metric": "GEMM TFLOPS (BF16, FP8 E4M3) on 1 GB300; % of dense tensor-core peak",
        "value": round(value, 2),
        "unit": "TFLOPS",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": "bf16_4096: BF16 GEMM M=N=K=4096, A,B ~ N(0,1) rounded to BF16, "
                               "BF16 output, alpha=1, beta=0",
                   "M": w.M, "N": w.N, "K": w.K, "parallelism": f"replicas x{world}",
                   "l2": rot.describe(),
                   "timing": f"K back-to-back library calls captured in one CUDA graph; "
                             f"{args.replays} replays, each between a CUDA-event pair with a "
                             f"barrier and a synchronize on both sides; value from the median "
                             f"replay"},
        "roofline": {"bound": "tensor", "achieved": round(achieved, 2),
                     "peak": peak_bf16, "unit": "TFLOP/s",
                     "frac": round(achieved / peak_bf16, 4),
                     "peak_source": f"{peak_src} bf16_tflops (burst: cuBLAS-class GEMM "
                                    f"throughput measured on this pool)",
                     "frac_of_sustained": (round(achieved / sustained_peak(), 4)
                                           if sustained_peak() and region_ms >= 100.0
                                           else None),
                     "isa_peak_at_clock": round(isa, 1) if isa else None,
                     "frac_of_isa_peak_at_clock": round(achieved / isa, 4) if isa else None,
                     "isa_peak_source": (f"8192 BF16 FLOP/clk/SM x {sms} SMs x the median SM "
                                         f"clock sampled during the timed replays"),
                     "kernel": "gemm_tn2_kernel<bf16,bf16 out> (CTA pair)",
                     "traffic": stored_traffic() if args.traffic is None else args.traffic},
        "gpu_launches": launches,
        "replays": replay_info,
        "clocks": clocks,
        "e2e": {"value": round(e2e_value, 2), "unit": "TFLOPS",
                "h2d_bytes_per_step": int(w.A.nbytes + w.B.nbytes),
                "d2h_bytes_per_step": int(D.numel() * 2),
                "method": "public API with pinned host buffers; each step's H2D, GEMM and "
                          "D2H overlap the neighbouring steps' on three streams (two "
                          "device slots)"},
    }
    del rot, A, B, D
    torch.cuda.empty_cache()
    if rank == 0 and not args.no_secondary:
        line["other_configs"] = secondary_configs(names=SECONDARY + tuple(QUANT))
        for o in line["other_configs"]:
            if o["workload"] not in QUANT:
                add_peak_fractions(o, peak_bf16, sms, clocks.get("sm_mhz"))
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_sample(w)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ---------------------------------------------------------------- reference

def run_reference(args):
    """The CPU oracle as it stands, on rank 0, one bounded sample per step."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import numpy as np

    import oracle
    import synth.workloads as W
    w = W.make("bf16_4096")
    cores = oracle.default_threads()
    rng = np.random.default_rng(1)

    def tiles(n, size):
        return [(int(rng.integers(0, w.M // size)) * size, int(rng.integers(0, w.N // size)) * size,
                 size, size) for _ in range(n)]

    # size each step so the whole run stays within about two minutes
    t0 = time.perf_counter()
    oracle.gemm(w.M, w.N, w.K, w.A, w.lda, w.B, w.ldb, tiles=tiles(cores, 32), nthreads=cores)
    t_tile = max(time.perf_counter() - t0, 1e-4)
    budget = 120.0 / max(1, args.steps + args.warmup)
    per_step = max(1, int(budget / t_tile)) * cores
    step_flops = per_step * 2 * 32 * 32 * w.K
    for _ in range(args.warmup):
        oracle.gemm(w.M, w.N, w.K, w.A, w.lda, w.B, w.ldb, tiles=tiles(per_step, 32),
                    nthreads=cores)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.gemm(w.M, w.N, w.K, w.A, w.lda, w.B, w.ldb, tiles=tiles(per_step, 32),
                    nthreads=cores)
    dt = time.perf_counter() - t0
    value = step_flops * args.steps / dt / 1e12
    sample = (f"{per_step} output tiles of 32x32 (K={w.K}) per step of the 4096^3 BF16 GEMM, "
              f"FP64 oracle")
    line = {
        "impl": "reference",
        "metric": "GEMM TFLOPS (BF16, FP8 E4M3) on 1 GB300; % of dense tensor-core peak",
        "value": round(value, 6), "unit": "TFLOPS", "n_gpus": int(os.environ.get("WORLD_SIZE", 1)),
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "bf16_4096: BF16 GEMM M=N=K=4096, A,B ~ N(0,1) rounded to BF16, "
                               "BF16 output, alpha=1, beta=0",
                   "M": w.M, "N": w.N, "K": w.K},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOPS", "cores": cores,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 6), "unit": "TFLOPS", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--replays", type=int, default=5,
                    help="timed replays of the K-step graph; the median is reported")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-secondary", action="store_true", help="skip the other workloads")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--traffic", type=float, default=None,
                    help="DRAM bytes per launch of the timed kernel from an ncu capture")
    ap.add_argument("--only", choices=SECONDARY + tuple(QUANT), default=None,
                    help="time one secondary workload alone (for profiling); prints its line")
    ap.add_argument("--size", default=None,
                    help="with --only: M,N,K overriding the workload's shape")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.only:
        import torch
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        size = tuple(int(x) for x in args.size.split(",")) if args.size else None
        print(json.dumps(secondary_configs(args.steps, args.warmup, (args.only,), size)[0]))
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
