"""CPU oracle for D = alpha*A*B + beta*C with BF16 / FP8 E4M3 operands.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline / reference legs may import this package.  The
product path (``tensor_core_dense_gb300``) never imports it and has no CPU
fallback.

The arithmetic lives in ``oracle.c`` (plain C, FP64 accumulation, exact
decoding of the BF16 and E4M3 bit patterns); this module only compiles it
with gcc and marshals numpy arrays.  Sources and readings:

* the operation D = A*B + C, A M x K, B K x N ("Tensor Cores: Matrix
  Instructions, Swizzling and FP8, Measured", Step 1), with B stored N x K,
  K contiguous (same page, Step 2);
* BF16 = 1/8/7 bits ("Tensor Cores", "Precision: FP16, BF16, TF32, FP8");
* E4M3 = 1/4/3 bits, no infinity, max normal 448, hence bias 7; E5M2 = 1/5/2
  bits, IEEE special values, max normal 57,344, hence bias 15 ("Tensor cores
  and low precision", the FP8 paragraph);
* FP8 scale factors applied after the product ("Tensor cores and low
  precision", the scaling paragraph), per tensor or per 128-wide K block;
* the FP8 quantiser that produces those scales and codes: scale = amax / 448
  per tensor, per 1 x 128 row block or per 128 x 128 block ("Tensor cores and
  low precision", the scaling paragraph; "Tensor Cores", "Precision: FP16,
  BF16, TF32, FP8": scaling factors per tensor, per row or per block).

Every function here is pinned by ``tests/test_oracle.py`` against facts the
pages fix, closed forms, library routines (torch's bfloat16 / float8_e4m3fn
conversions) and exact brute force; none is "parity unpinned".
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

IN_BF16, IN_E4M3 = 0, 1
Q_TENSOR, Q_ROW128, Q_BLOCK128 = 0, 1, 2
SCALE_NONE, SCALE_TENSOR, SCALE_BLOCK128, SCALE_MX32 = 0, 1, 2, 3
C_BF16, C_F32 = 0, 1
FP8_E4M3, FP8_E5M2 = 0, 1


class _Args(ctypes.Structure):
    _fields_ = [
        ("M", ctypes.c_int64),
        ("N", ctypes.c_int64),
        ("K", ctypes.c_int64),
        ("in_type", ctypes.c_int32),
        ("scale_mode", ctypes.c_int32),
        ("A", ctypes.c_void_p),
        ("lda", ctypes.c_int64),
        ("B", ctypes.c_void_p),
        ("ldb", ctypes.c_int64),
        ("a_scale", ctypes.c_void_p),
        ("b_scale", ctypes.c_void_p),
        ("C", ctypes.c_void_p),
        ("ldc", ctypes.c_int64),
        ("c_type", ctypes.c_int32),
        ("pad_", ctypes.c_int32),
        ("alpha", ctypes.c_double),
        ("beta", ctypes.c_double),
        ("a_fp8", ctypes.c_int32),
        ("b_fp8", ctypes.c_int32),
        ("a_sf", ctypes.c_void_p),
        ("b_sf", ctypes.c_void_p),
    ]


def build(force: bool = False) -> str:
    """Compile oracle.c into _build/liboracle.so (portable C, no -march)."""
    with _lock:
        if (not force and os.path.exists(_LIB_PATH)
                and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
            return _LIB_PATH
        os.makedirs(_BUILD, exist_ok=True)
        tmp = f"{_LIB_PATH}.{os.getpid()}.tmp"
        subprocess.check_call([
            "gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
            "-ffp-contract=off", "-fno-fast-math", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
        return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        lib.orc_bf16_decode.restype = ctypes.c_double
        lib.orc_bf16_decode.argtypes = [ctypes.c_uint16]
        lib.orc_e4m3_decode.restype = ctypes.c_double
        lib.orc_e4m3_decode.argtypes = [ctypes.c_uint8]
        for name in ("orc_bf16_decode_array", "orc_bf16_encode_array",
                     "orc_e4m3_decode_array", "orc_e4m3_encode_array",
                     "orc_e5m2_decode_array", "orc_e5m2_encode_array",
                     "orc_e8m0_decode_array", "orc_cast_bf16_array"):
            getattr(lib, name).argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p]
            getattr(lib, name).restype = None
        lib.orc_gemm_tiles.argtypes = [ctypes.POINTER(_Args), ctypes.c_int64, ctypes.c_void_p,
                                       ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
        lib.orc_gemm_tiles.restype = ctypes.c_int
        i64 = ctypes.c_int64
        lib.orc_quant_fp8.argtypes = [ctypes.c_void_p, ctypes.c_int32, i64, i64, i64,
                                      ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p, i64,
                                      ctypes.c_void_p]
        lib.orc_quant_fp8.restype = ctypes.c_int
        lib.orc_mx_sf_offset.argtypes = [i64, i64, i64]
        lib.orc_mx_sf_offset.restype = i64
        _lib = lib
    return _lib


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data


def _elementwise(name, x, in_dtype, out_dtype):
    x = np.ascontiguousarray(x, dtype=in_dtype)
    out = np.empty(x.shape, dtype=out_dtype)
    getattr(_load(), name)(_ptr(x), x.size, _ptr(out))
    return out


def bf16_decode(bits) -> np.ndarray:
    """BF16 bit patterns (uint16) -> float64 values."""
    return _elementwise("orc_bf16_decode_array", bits, np.uint16, np.float64)


def bf16_encode(x) -> np.ndarray:
    """float32 values -> BF16 bit patterns, round to nearest even."""
    return _elementwise("orc_bf16_encode_array", x, np.float32, np.uint16)


def e4m3_decode(bits) -> np.ndarray:
    """E4M3 bytes -> float64 values (NaN for S.1111.111)."""
    return _elementwise("orc_e4m3_decode_array", bits, np.uint8, np.float64)


def e5m2_decode(bits) -> np.ndarray:
    """E5M2 bytes -> float64 values (+-inf for S.11111.00, NaN for other S.11111.xx)."""
    return _elementwise("orc_e5m2_decode_array", bits, np.uint8, np.float64)


def e5m2_encode(x) -> np.ndarray:
    """float32 values -> E5M2 bytes, nearest even, saturating at +-57344."""
    return _elementwise("orc_e5m2_encode_array", x, np.float32, np.uint8)


def e4m3_encode(x) -> np.ndarray:
    """float32 values -> E4M3 bytes, nearest even, saturating at +-448."""
    return _elementwise("orc_e4m3_encode_array", x, np.float32, np.uint8)


def e8m0_decode(bits) -> np.ndarray:
    """E8M0 bytes -> float64 values 2^(e - 127) (NaN for 0xFF)."""
    return _elementwise("orc_e8m0_decode_array", bits, np.uint8, np.float64)


def mx_sf_bytes(rows, K) -> int:
    """Bytes of one operand's MX scales: ceil(rows/128) x ceil(ceil(K/32)/4)
    tiles of 512 bytes."""
    return -(-rows // 128) * -(-(-(-K // 32)) // 4) * 512


def mx_sf_offset(r, kb, K) -> int:
    """Byte offset of the scale of row r, 32-wide K block kb (oracle.c's
    orc_mx_sf_offset, the tiled layout)."""
    return int(_load().orc_mx_sf_offset(int(r), int(kb), -(-(-(-K // 32)) // 4)))


def cast_bf16(v) -> np.ndarray:
    """The BF16 output expected for FP64 values v: v -> FP32 -> BF16 (nearest even)."""
    return _elementwise("orc_cast_bf16_array", v, np.float64, np.uint16)


def default_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def gemm(M, N, K, A, lda, B, ldb, *, in_type=IN_BF16, scale_mode=SCALE_NONE,
         a_scale=None, b_scale=None, C=None, ldc=0, c_type=C_F32, alpha=1.0, beta=0.0,
         tiles=None, nthreads=None, a_fp8=FP8_E4M3, b_fp8=FP8_E4M3, a_sf=None, b_sf=None):
    """Reference values and error bounds for D = alpha*A*B + beta*C.

    A: flat uint16 (BF16) or uint8 (FP8) array, element (i, k) at A[i*lda + k];
       with in_type=IN_E4M3 the bytes are E4M3 or E5M2 per a_fp8 / b_fp8.
    B: same dtype, element (k, j) at B[j*ldb + k] (N x K, K contiguous).
    C: flat uint16 (c_type=C_BF16) or float32 (C_F32) array, (i, j) at C[i*ldc + j];
       not read when beta == 0.
    a_scale / b_scale: float32 arrays (scale_mode TENSOR: one value each;
       BLOCK128: a_scale[kb*M + i], b_scale[nb*ceil(K/128) + kb]).
    a_sf / b_sf: scale_mode MX32: uint8 E8M0 scales per 32-wide K block, in
       the tiled layout of oracle.c (mx_sf_bytes(M, K) / mx_sf_bytes(N, K)).
    tiles: None for the whole M x N output, else a list of (i0, j0, mi, nj).

    Returns (v, bound): FP64 arrays.  For tiles=None each is M x N; otherwise a
    list of mi x nj arrays, one per tile.  bound = |alpha| * sum_k |a_ik * b_kj|.
    """
    lib = _load()
    in_np = np.uint16 if in_type == IN_BF16 else np.uint8
    A = np.ascontiguousarray(A, dtype=in_np).ravel()
    B = np.ascontiguousarray(B, dtype=in_np).ravel()
    if K > 0:
        if M > 0 and A.size < (M - 1) * lda + K:
            raise ValueError("A too small")
        if N > 0 and B.size < (N - 1) * ldb + K:
            raise ValueError("B too small")
    if C is not None:
        C = np.ascontiguousarray(C, dtype=np.uint16 if c_type == C_BF16 else np.float32).ravel()
        if M > 0 and N > 0 and C.size < (M - 1) * ldc + N:
            raise ValueError("C too small")
    elif beta != 0.0:
        raise ValueError("C required when beta != 0")
    if scale_mode in (SCALE_TENSOR, SCALE_BLOCK128):
        a_scale = np.ascontiguousarray(a_scale, dtype=np.float32).ravel()
        b_scale = np.ascontiguousarray(b_scale, dtype=np.float32).ravel()
        if scale_mode == SCALE_BLOCK128:
            KB = (K + 127) // 128
            if a_scale.size < KB * M or b_scale.size < ((N + 127) // 128) * KB:
                raise ValueError("scale arrays too small")
    else:
        a_scale = b_scale = None
    if scale_mode == SCALE_MX32:
        a_scale = b_scale = None
        a_sf = np.ascontiguousarray(a_sf, dtype=np.uint8).ravel()
        b_sf = np.ascontiguousarray(b_sf, dtype=np.uint8).ravel()
        if a_sf.size < mx_sf_bytes(M, K) or b_sf.size < mx_sf_bytes(N, K):
            raise ValueError("MX scale arrays too small")
    else:
        a_sf = b_sf = None
    args = _Args(M, N, K, in_type, scale_mode, _ptr(A), lda, _ptr(B), ldb,
                 _ptr(a_scale), _ptr(b_scale), _ptr(C), ldc, c_type, 0,
                 float(alpha), float(beta), int(a_fp8), int(b_fp8), _ptr(a_sf), _ptr(b_sf))
    whole = tiles is None
    if whole:
        tiles = [(0, 0, M, N)]
    t = np.ascontiguousarray(np.array(tiles, dtype=np.int64).reshape(-1, 4))
    total = int((t[:, 2] * t[:, 3]).sum()) if len(t) else 0
    v = np.empty(max(total, 1), dtype=np.float64)
    bound = np.empty(max(total, 1), dtype=np.float64)
    rc = lib.orc_gemm_tiles(ctypes.byref(args), len(t), _ptr(t), _ptr(v), _ptr(bound),
                            int(nthreads or default_threads()))
    if rc != 0:
        raise ValueError("oracle rejected the arguments")
    outs_v, outs_b, o = [], [], 0
    for (_, _, mi, nj) in t.tolist():
        outs_v.append(v[o:o + mi * nj].reshape(mi, nj))
        outs_b.append(bound[o:o + mi * nj].reshape(mi, nj))
        o += mi * nj
    if whole:
        return outs_v[0], outs_b[0]
    return outs_v, outs_b


def quantize_e4m3(x, mode, *, ldq=None):
    """FP8 E4M3 quantisation (quantize_fp8 with fmt=FP8_E4M3)."""
    return quantize_fp8(x, mode, FP8_E4M3, ldq=ldq)


def quantize_fp8(x, mode, fmt, *, ldq=None):
    """FP8 quantisation of a 2-D array x (float32 values, or uint16 BF16 bit
    patterns) with scale = amax / 448 (FP8_E4M3) or amax / 57344 (FP8_E5M2)
    per block (``oracle.c``, orc_quant_fp8).

    mode: Q_TENSOR (scale[0]), Q_ROW128 (scale[kb*rows + r]) or Q_BLOCK128
    (scale[rb*ceil(cols/128) + kb]).  Returns (q, scale): q is a rows x ldq
    uint8 array (columns >= cols stay zero), scale a float32 array.
    """
    if x.dtype == np.uint16:
        x_type = 1
    else:
        x_type = 0
        x = np.asarray(x, dtype=np.float32)
    x = np.ascontiguousarray(x)
    rows, cols = x.shape
    ldq = cols if ldq is None else ldq
    KB, RB = (cols + 127) // 128, (rows + 127) // 128
    n = {Q_TENSOR: 1, Q_ROW128: KB * rows, Q_BLOCK128: RB * KB}[mode]
    q = np.zeros((rows, ldq), dtype=np.uint8)
    s = np.zeros(max(n, 1), dtype=np.float32)
    rc = _load().orc_quant_fp8(_ptr(x), x_type, rows, cols, cols, mode, int(fmt), _ptr(q), ldq,
                               _ptr(s))
    if rc != 0:
        raise ValueError("oracle rejected the quantiser arguments")
    return q, s[:n]
