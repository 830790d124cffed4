"""Seeded synthetic inputs for the GEMM workloads (no GEMM arithmetic here).

Both the CUDA library's tests/benchmark and the CPU oracle consume what this
module produces; it imports neither.  The generator is counter based
(SplitMix64 keyed by seed and tensor id, indexed by the element's logical
position), so any element can be regenerated alone; see ``synth.c``.

Workload recipes (value distributions of the pages' workloads):

* ``uniform`` in [-1, 1) rounded to BF16 -- the 4,096^3 test's inputs
  ("Tensor Cores: Matrix Instructions, Swizzling and FP8, Measured", Step 2);
* ``normal(mu, sd)`` rounded to BF16, or quantised to E4M3 with an FP32 scale
  amax/448 per tensor, per 1 x 128 row block or per 128 x 128 block
  ("Tensor cores and low precision": scale so the largest magnitude sits at
  448, then cast);
* normal with rare outliers: each element independently, with probability p,
  multiplied by a factor.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libsynth.so")
_lock = threading.Lock()
_lib = None

UNIFORM, NORMAL = 0, 1


class _Dist(ctypes.Structure):
    _fields_ = [("dist", ctypes.c_int32), ("pad_", ctypes.c_int32), ("p0", ctypes.c_double),
                ("p1", ctypes.c_double), ("out_prob", ctypes.c_double),
                ("out_factor", ctypes.c_double)]


def build(force: bool = False) -> str:
    with _lock:
        if (not force and os.path.exists(_LIB_PATH)
                and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
            return _LIB_PATH
        os.makedirs(_BUILD, exist_ok=True)
        tmp = f"{_LIB_PATH}.{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                               "-ffp-contract=off", "-fno-fast-math", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
        return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        vp, i64, u64 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64
        lib.synth_key.restype = u64
        lib.synth_key.argtypes = [u64, u64]
        lib.synth_draw.restype = u64
        lib.synth_draw.argtypes = [u64, u64]
        for name in ("synth_fill_f32", "synth_fill_bf16"):
            getattr(lib, name).argtypes = [ctypes.POINTER(_Dist), u64, u64, i64, i64, i64, vp,
                                           ctypes.c_int]
            getattr(lib, name).restype = None
        for name in ("synth_quant_e4m3_tensor", "synth_quant_e4m3_rowblock",
                     "synth_quant_e4m3_block128"):
            getattr(lib, name).argtypes = [vp, i64, i64, i64, vp, vp]
            getattr(lib, name).restype = None
        for name in ("synth_to_bf16_array", "synth_to_e4m3_array", "synth_to_e5m2_array"):
            getattr(lib, name).argtypes = [vp, i64, vp]
            getattr(lib, name).restype = None
        _lib = lib
    return _lib


def _threads():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def _dist(kind, p0, p1, out_prob=0.0, out_factor=1.0):
    return _Dist(kind, 0, float(p0), float(p1), float(out_prob), float(out_factor))


def values_f32(seed, tensor, rows, cols, *, dist="normal", p0=0.0, p1=1.0,
               out_prob=0.0, out_factor=1.0) -> np.ndarray:
    """rows x cols float32 values of the given distribution."""
    kind = NORMAL if dist == "normal" else UNIFORM
    out = np.empty((rows, cols), dtype=np.float32)
    d = _dist(kind, p0, p1, out_prob, out_factor)
    _load().synth_fill_f32(ctypes.byref(d), seed, tensor, rows, cols, cols, out.ctypes.data,
                           _threads())
    return out


def bf16(seed, tensor, rows, cols, *, ld=None, dist="normal", p0=0.0, p1=1.0) -> np.ndarray:
    """rows x ld uint16 BF16 patterns; columns >= cols (padding) are zero."""
    ld = cols if ld is None else ld
    out = np.zeros((rows, ld), dtype=np.uint16)
    kind = NORMAL if dist == "normal" else UNIFORM
    d = _dist(kind, p0, p1)
    _load().synth_fill_bf16(ctypes.byref(d), seed, tensor, rows, cols, ld, out.ctypes.data,
                            _threads())
    return out


def _quant(name, x, ld, nscales):
    rows, cols = x.shape
    ld = cols if ld is None else ld
    q = np.zeros((rows, ld), dtype=np.uint8)
    s = np.empty(max(nscales, 1), dtype=np.float32)
    x = np.ascontiguousarray(x, dtype=np.float32)
    getattr(_load(), name)(x.ctypes.data, rows, cols, ld, q.ctypes.data, s.ctypes.data)
    return q, s[:nscales]


def e4m3_tensor(x, ld=None):
    """Per-tensor FP8: (q uint8 rows x ld, scale float32[1])."""
    return _quant("synth_quant_e4m3_tensor", x, ld, 1)


def e4m3_rowblock(x, ld=None):
    """1 x 128 blocks: (q, scale[kb*rows + r])."""
    rows, cols = x.shape
    return _quant("synth_quant_e4m3_rowblock", x, ld, ((cols + 127) // 128) * rows)


def e4m3_block128(x, ld=None):
    """128 x 128 blocks: (q, scale[nb*KB + kb])."""
    rows, cols = x.shape
    return _quant("synth_quant_e4m3_block128", x, ld,
                  ((rows + 127) // 128) * ((cols + 127) // 128))


def to_bf16(x) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    _load().synth_to_bf16_array(x.ctypes.data, x.size, out.ctypes.data)
    return out


def to_e4m3(x) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint8)
    _load().synth_to_e4m3_array(x.ctypes.data, x.size, out.ctypes.data)
    return out


def to_e5m2(x) -> np.ndarray:
    """float32 -> E5M2 bytes, nearest even, saturating at +-57344."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint8)
    _load().synth_to_e5m2_array(x.ctypes.data, x.size, out.ctypes.data)
    return out


def draw(seed, tensor, ctr) -> int:
    """Raw 64-bit draw `ctr` of stream (seed, tensor)."""
    lib = _load()
    return int(lib.synth_draw(lib.synth_key(seed, tensor), ctr))


# ------------------------------------------------------------- microscaling

def mx_tile_sf(exps, K):
    """E8M0 scale bytes exps[r, kb] (one per row and 32-wide K block) laid out
    as the library reads them: tiles of 128 rows x 4 K blocks, 512 bytes
    each, tile (r // 128, kb // 4) at ((r // 128) * KT + kb // 4) * 512 with
    KT = ceil(ceil(K / 32) / 4); inside a tile, row r % 32 takes 16 bytes,
    (r // 32) % 4 picks 4 of them and kb % 4 the byte.  Padding rows and
    blocks hold 127 (scale 1).  Built by reshaping, not by index arithmetic."""
    exps = np.asarray(exps, dtype=np.uint8)
    rows = exps.shape[0]
    KB = -(-K // 32)
    RT, KT = -(-rows // 128), -(-KB // 4)
    pad = np.full((RT * 128, KT * 4), 127, dtype=np.uint8)
    pad[:rows, :KB] = exps[:, :KB]
    # axes (row tile, (r // 32) % 4, r % 32, K tile, kb % 4) -> tile-major order
    return np.ascontiguousarray(pad.reshape(RT, 4, 32, KT, 4).transpose(0, 3, 2, 1, 4)).ravel()


def mx_quant(x, ld=None, fmt="e4m3"):
    """Microscaled FP8 of a rows x K float32 matrix: per row and 32-wide K
    block an E8M0 exponent e and codes FP8(x / 2^(e - 127)), saturating.
    e = floor(log2(amax)) - emax + 127 with emax = 8 for E4M3 (448 = 1.75 *
    2^8) and 15 for E5M2, so the block's largest magnitude lands in the
    format's top binade (the microscaling recipe); an all-zero block takes
    e = 127.  Returns (q uint8 rows x ld, exps uint8 rows x ceil(K/32))."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    rows, K = x.shape
    ld = K if ld is None else ld
    KB = -(-K // 32)
    xp = np.zeros((rows, KB * 32), np.float32)
    xp[:, :K] = x
    amax = np.abs(xp.reshape(rows, KB, 32)).max(axis=2)
    _, ex = np.frexp(amax)                         # amax = m * 2^ex, 0.5 <= m < 1
    emax = 8 if fmt == "e4m3" else 15
    e = np.where(amax > 0, ex - 1 - emax + 127, 127)
    e = np.clip(e, 0, 254).astype(np.uint8)
    scaled = np.ldexp(xp.reshape(rows, KB, 32),
                      -(e.astype(np.int32) - 127)[:, :, None]).reshape(rows, KB * 32)[:, :K]
    q = np.zeros((rows, ld), np.uint8)
    q[:, :K] = to_e4m3(scaled) if fmt == "e4m3" else to_e5m2(scaled)
    return q, e
