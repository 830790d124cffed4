"""Python binding for libtcgemm.so, the sm_103a tensor-core GEMM library.

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI of ``include/tcgemm.h``.  PyTorch provides device
memory and streams.  There is no CPU fallback: if the compiled library is
missing, importing the binding's entry points raises.

    D = alpha * A @ B.T + beta * C      (A: M x K, B: N x K, both K-major)

The entry points keep the C names: ``gemm_bf16``, ``gemm_fp8_e4m3``, ``gemm_fp8``
(E4M3 / E5M2 per operand), ``gemm_mxfp8`` (E8M0 scales per 32-wide K block,
applied by the tensor core) and the FP8 quantiser ``quantize_e4m3`` that
produces the FP8 GEMM's codes and scales.
"""

from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libtcgemm.so")

OK, ERR_INVALID_ARG, ERR_ALIGNMENT, ERR_UNSUPPORTED, ERR_CUDA, ERR_TIMEOUT = range(6)
OUT_BF16, OUT_F32 = 0, 1
SCALE_TENSOR, SCALE_BLOCK128 = 0, 1
IN_F32, IN_BF16 = 0, 1
FP8_E4M3, FP8_E5M2 = 0, 1
QUANT_TENSOR, QUANT_ROW128, QUANT_BLOCK128 = 0, 1, 2

# Every symbol include/tcgemm.h declares.
EXPORTS = ("gemm_bf16", "gemm_fp8_e4m3", "gemm_fp8", "gemm_mxfp8", "gemm_fp8_e4m3_block_noalloc",
           "quantize_e4m3", "quantize_fp8", "tcg_status_string", "tcg_last_device_status", "tcg_launch_count",
           "tcg_debug_timeout_probe")

_lib = None


class TcgError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} (status {status})")


def lib():
    """The loaded C library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(
                f"{LIB_PATH} is missing: build it with tensor_core_dense_gb300.build.build() "
                "(or __graft_entry__.build()); there is no CPU fallback")
        L = ctypes.CDLL(LIB_PATH)
        i64, vp, f32, i32 = ctypes.c_int64, ctypes.c_void_p, ctypes.c_float, ctypes.c_int
        L.gemm_bf16.argtypes = [i64, i64, i64, vp, i64, vp, i64, vp, i64, vp, i64, i32, f32, f32,
                                vp]
        L.gemm_bf16.restype = i32
        L.gemm_fp8_e4m3.argtypes = [i64, i64, i64, vp, i64, vp, i64, vp, vp, i32, vp, i64, vp,
                                    i64, i32, f32, f32, vp]
        L.gemm_fp8_e4m3.restype = i32
        L.gemm_fp8.argtypes = [i64, i64, i64, vp, i64, i32, vp, i64, i32, vp, vp, i32, vp, i64,
                               vp, i64, i32, f32, f32, vp]
        L.gemm_fp8.restype = i32
        L.gemm_mxfp8.argtypes = [i64, i64, i64, vp, i64, i32, vp, i64, i32, vp, vp, vp, i64,
                                 vp, i64, i32, f32, f32, vp]
        L.gemm_mxfp8.restype = i32
        L.quantize_e4m3.argtypes = [i64, i64, vp, i64, i32, i32, vp, i64, vp, vp]
        L.quantize_e4m3.restype = i32
        L.quantize_fp8.argtypes = [i64, i64, vp, i64, i32, i32, i32, vp, i64, vp, vp]
        L.quantize_fp8.restype = i32
        L.tcg_status_string.argtypes = [i32]
        L.tcg_status_string.restype = ctypes.c_char_p
        L.tcg_last_device_status.argtypes = [vp]
        L.tcg_last_device_status.restype = i32
        L.tcg_debug_timeout_probe.argtypes = [vp]
        L.tcg_debug_timeout_probe.restype = i32
        L.tcg_launch_count.argtypes = []
        L.tcg_launch_count.restype = ctypes.c_uint64
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().tcg_status_string(int(status)).decode()


def launch_count() -> int:
    """Kernels launched by the library in this process."""
    return int(lib().tcg_launch_count())


def _stream_handle(stream):
    if stream is None:
        import torch
        stream = torch.cuda.current_stream()
    return getattr(stream, "cuda_stream", stream) or None


def last_device_status(stream=None) -> int:
    """Synchronise the stream; return (and clear) the device status word."""
    return int(lib().tcg_last_device_status(_stream_handle(stream)))


# ------------------------------------------------------------ raw entry points

def gemm_bf16_raw(M, N, K, A, lda, B, ldb, C, ldc, D, ldd, out_dtype, alpha, beta,
                  stream) -> int:
    """The C call with integer device pointers; returns the status code."""
    return int(lib().gemm_bf16(M, N, K, A, lda, B, ldb, C, ldc, D, ldd, out_dtype,
                               float(alpha), float(beta), stream))


def gemm_fp8_e4m3_raw(M, N, K, A, lda, B, ldb, a_scale, b_scale, mode, C, ldc, D, ldd,
                      out_dtype, alpha, beta, stream) -> int:
    return int(lib().gemm_fp8_e4m3(M, N, K, A, lda, B, ldb, a_scale, b_scale, mode, C, ldc, D,
                                   ldd, out_dtype, float(alpha), float(beta), stream))


def gemm_fp8_raw(M, N, K, A, lda, a_format, B, ldb, b_format, a_scale, b_scale, mode, C, ldc,
                 D, ldd, out_dtype, alpha, beta, stream) -> int:
    return int(lib().gemm_fp8(M, N, K, A, lda, a_format, B, ldb, b_format, a_scale, b_scale,
                              mode, C, ldc, D, ldd, out_dtype, float(alpha), float(beta),
                              stream))


def gemm_mxfp8_raw(M, N, K, A, lda, a_format, B, ldb, b_format, a_sf, b_sf, C, ldc, D, ldd,
                   out_dtype, alpha, beta, stream) -> int:
    return int(lib().gemm_mxfp8(M, N, K, A, lda, a_format, B, ldb, b_format, a_sf, b_sf, C,
                                ldc, D, ldd, out_dtype, float(alpha), float(beta), stream))


def quantize_e4m3_raw(rows, cols, X, ldx, x_dtype, mode, Q, ldq, scale, stream) -> int:
    return int(lib().quantize_e4m3(rows, cols, X, ldx, x_dtype, mode, Q, ldq, scale, stream))


def quantize_fp8_raw(rows, cols, X, ldx, x_dtype, fmt, mode, Q, ldq, scale, stream) -> int:
    return int(lib().quantize_fp8(rows, cols, X, ldx, x_dtype, fmt, mode, Q, ldq, scale, stream))


# --------------------------------------------------------------- tensor API

def _ld(t, rows_name):
    """Leading dimension in elements.  A single-row matrix never uses its row
    pitch, so it gets the smallest 16-byte-multiple pitch >= its width."""
    if t.dim() != 2:
        raise ValueError(f"{rows_name} must be 2-D")
    if t.size(1) > 1 and t.stride(1) != 1:
        raise ValueError(f"{rows_name} must have a contiguous last dimension")
    if t.size(0) > 1:
        return t.stride(0)
    step = max(1, 16 // t.element_size())
    return max(step, -(-t.size(1) // step) * step)


def _out_dtype(D):
    import torch
    if D.dtype == torch.bfloat16:
        return OUT_BF16
    if D.dtype == torch.float32:
        return OUT_F32
    raise ValueError("D must be bfloat16 or float32")


def _ptr(t):
    return None if t is None else t.data_ptr()


def _beta(C, beta, what):
    """beta as given; a non-zero beta needs a C to scale (the C call would
    return ERR_INVALID_ARG for a NULL C)."""
    if C is None and float(beta) != 0.0:
        raise ValueError(f"{what}: beta = {beta} needs C")
    return beta


def gemm_bf16(A, B, D, C=None, *, alpha=1.0, beta=0.0, stream=None):
    """D = alpha * A @ B.T + beta * C on the GPU (BF16 A, B; D/C BF16 or FP32)."""
    import torch
    if A.dtype != torch.bfloat16 or B.dtype != torch.bfloat16:
        raise ValueError("A and B must be bfloat16")
    M, K = A.shape
    N = B.shape[0]
    if B.shape[1] != K or tuple(D.shape) != (M, N):
        raise ValueError("shape mismatch")
    if C is not None and (tuple(C.shape) != (M, N) or C.dtype != D.dtype):
        raise ValueError("C must match D")
    st = gemm_bf16_raw(M, N, K, _ptr(A), _ld(A, "A"), _ptr(B), _ld(B, "B"), _ptr(C),
                       _ld(C, "C") if C is not None else 0, _ptr(D), _ld(D, "D"), _out_dtype(D),
                       alpha, _beta(C, beta, "gemm_bf16"), _stream_handle(stream))
    if st != OK:
        raise TcgError(st, "gemm_bf16")
    return D


def _fp8_format(t, given, name):
    import torch
    if t.dtype == torch.float8_e5m2:
        fmt = FP8_E5M2
    elif t.dtype == torch.float8_e4m3fn:
        fmt = FP8_E4M3
    elif t.dtype == torch.uint8:
        fmt = FP8_E4M3 if given is None else given
    else:
        raise ValueError(f"{name} must hold FP8 bytes")
    if given is not None and given != fmt:
        raise ValueError(f"{name}: format {given} does not match dtype {t.dtype}")
    return fmt


def gemm_fp8(A, B, a_scale, b_scale, D, C=None, *, mode=SCALE_TENSOR, a_format=None,
             b_format=None, alpha=1.0, beta=0.0, stream=None):
    """D = alpha * (sa.A) @ (sb.B).T + beta * C with FP8 A, B: float8_e4m3fn /
    float8_e5m2 tensors, or uint8 with a_format / b_format (default E4M3), and
    FP32 scale tensors on the device (layouts in include/tcgemm.h)."""
    import torch
    af, bf = _fp8_format(A, a_format, "A"), _fp8_format(B, b_format, "B")
    if a_scale.dtype != torch.float32 or b_scale.dtype != torch.float32:
        raise ValueError("scales must be float32")
    M, K = A.shape
    N = B.shape[0]
    if B.shape[1] != K or tuple(D.shape) != (M, N):
        raise ValueError("shape mismatch")
    if C is not None and (tuple(C.shape) != (M, N) or C.dtype != D.dtype):
        raise ValueError("C must match D")
    st = gemm_fp8_raw(M, N, K, _ptr(A), _ld(A, "A"), af, _ptr(B), _ld(B, "B"), bf, _ptr(a_scale),
                      _ptr(b_scale), mode, _ptr(C), _ld(C, "C") if C is not None else 0, _ptr(D),
                      _ld(D, "D"), _out_dtype(D), alpha, _beta(C, beta, "gemm_fp8"),
                      _stream_handle(stream))
    if st != OK:
        raise TcgError(st, "gemm_fp8")
    return D


def gemm_fp8_e4m3(A, B, a_scale, b_scale, D, C=None, *, mode=SCALE_TENSOR, alpha=1.0,
                  beta=0.0, stream=None):
    """D = alpha * (sa.A) @ (sb.B).T + beta * C with E4M3 A, B (uint8 or float8_e4m3fn)
    and FP32 scale tensors on the device (layouts in include/tcgemm.h)."""
    import torch
    for t, n in ((A, "A"), (B, "B")):
        if t.dtype not in (torch.uint8, torch.float8_e4m3fn):
            raise ValueError(f"{n} must hold E4M3 bytes")
    if a_scale.dtype != torch.float32 or b_scale.dtype != torch.float32:
        raise ValueError("scales must be float32")
    M, K = A.shape
    N = B.shape[0]
    if B.shape[1] != K or tuple(D.shape) != (M, N):
        raise ValueError("shape mismatch")
    if C is not None and (tuple(C.shape) != (M, N) or C.dtype != D.dtype):
        raise ValueError("C must match D")
    st = gemm_fp8_e4m3_raw(M, N, K, _ptr(A), _ld(A, "A"), _ptr(B), _ld(B, "B"), _ptr(a_scale),
                           _ptr(b_scale), mode, _ptr(C), _ld(C, "C") if C is not None else 0,
                           _ptr(D), _ld(D, "D"), _out_dtype(D), alpha,
                           _beta(C, beta, "gemm_fp8_e4m3"), _stream_handle(stream))
    if st != OK:
        raise TcgError(st, "gemm_fp8_e4m3")
    return D


def mx_scale_bytes(rows, K):
    """Bytes of one operand's E8M0 scales for gemm_mxfp8: ceil(rows/128) x
    ceil(K/128) tiles of 512 bytes."""
    return -(-rows // 128) * -(-K // 128) * 512


def gemm_mxfp8(A, B, a_sf, b_sf, D, C=None, *, a_format=None, b_format=None, alpha=1.0,
               beta=0.0, stream=None):
    """D = alpha * sum_kb SFA * SFB * (A @ B.T over 32-wide K blocks) + beta * C
    with FP8 A, B (float8_e4m3fn / float8_e5m2, or uint8 with a_format /
    b_format) and E8M0 scale bytes a_sf, b_sf (uint8 or float8_e8m0fnu
    tensors on the device, tiled layout in include/tcgemm.h)."""
    import torch
    af, bf = _fp8_format(A, a_format, "A"), _fp8_format(B, b_format, "B")
    M, K = A.shape
    N = B.shape[0]
    if B.shape[1] != K or tuple(D.shape) != (M, N):
        raise ValueError("shape mismatch")
    for t, n, rows in ((a_sf, "a_sf", M), (b_sf, "b_sf", N)):
        if t.dtype not in (torch.uint8, getattr(torch, "float8_e8m0fnu", torch.uint8)):
            raise ValueError(f"{n} must hold E8M0 bytes")
        if not t.is_contiguous() or t.numel() < mx_scale_bytes(rows, K):
            raise ValueError(f"{n} must be contiguous with mx_scale_bytes({rows}, K) bytes")
    if C is not None and (tuple(C.shape) != (M, N) or C.dtype != D.dtype):
        raise ValueError("C must match D")
    st = gemm_mxfp8_raw(M, N, K, _ptr(A), _ld(A, "A"), af, _ptr(B), _ld(B, "B"), bf,
                        _ptr(a_sf), _ptr(b_sf), _ptr(C), _ld(C, "C") if C is not None else 0,
                        _ptr(D), _ld(D, "D"), _out_dtype(D), alpha,
                        _beta(C, beta, "gemm_mxfp8"), _stream_handle(stream))
    if st != OK:
        raise TcgError(st, "gemm_mxfp8")
    return D


def quant_scale_count(rows, cols, mode):
    """Number of FP32 scales quantize_e4m3 writes for a rows x cols input."""
    kb, rb = -(-cols // 128), -(-rows // 128)
    return {QUANT_TENSOR: 1, QUANT_ROW128: rows * kb, QUANT_BLOCK128: rb * kb}[mode]


def quantize_e4m3(X, Q, scale, *, mode=QUANT_TENSOR, stream=None):
    """FP8 E4M3 codes into Q (uint8 or float8_e4m3fn, rows x >=cols) and
    dequantisation scales into `scale` (float32, quant_scale_count values) for
    the float32 or bfloat16 matrix X (layouts in include/tcgemm.h)."""
    return quantize_fp8(X, Q, scale, mode=mode, fmt=FP8_E4M3, stream=stream)


def quantize_fp8(X, Q, scale, *, mode=QUANT_TENSOR, fmt=FP8_E4M3, stream=None):
    """quantize_e4m3 with the encoding chosen: FP8_E4M3 (scale amax/448) or
    FP8_E5M2 (scale amax/57344); Q may be uint8 or the matching float8 dtype."""
    import torch
    if X.dtype == torch.float32:
        x_dtype = IN_F32
    elif X.dtype == torch.bfloat16:
        x_dtype = IN_BF16
    else:
        raise ValueError("X must be float32 or bfloat16")
    if Q.dtype not in (torch.uint8, torch.float8_e4m3fn, torch.float8_e5m2):
        raise ValueError("Q must hold bytes")
    if scale.dtype != torch.float32 or not scale.is_contiguous():
        raise ValueError("scale must be a contiguous float32 tensor")
    rows, cols = X.shape
    if Q.shape[0] != rows or Q.shape[1] < cols:
        raise ValueError("Q must be rows x (>= cols)")
    if scale.numel() < quant_scale_count(rows, cols, mode):
        raise ValueError("scale too small")
    st = quantize_fp8_raw(rows, cols, _ptr(X), _ld(X, "X"), x_dtype, fmt, mode, _ptr(Q),
                          _ld(Q, "Q"), _ptr(scale), _stream_handle(stream))
    if st != OK:
        raise TcgError(st, "quantize_fp8")
    return Q, scale
