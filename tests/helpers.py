"""Shared test helpers: running a workload through the library, and comparing
its output with the oracle under the stated tolerances.

Tolerances (per element, D compared before the output cast, i.e. from an FP32
output of the same kernel):
    BF16 inputs:  |D - v| <= 2^-14 * bound + 1e-6          + c_term
    FP8 inputs:   |D - v| <= 2^-10 * bound                  + c_term
where v is the oracle's FP64 value, bound = |alpha| * sum_k |a_ik b_kj| (with
the dequantisation scales), and c_term = 2^-22 * (|v| + |beta c_ij|) covers the
FP32 evaluation of alpha*acc + beta*c, a step the per-product bound does not
describe.  A BF16 output is accepted when it lies within one BF16 ulp of v
beyond that tolerance.
"""

from __future__ import annotations

import numpy as np

import oracle

TOL_BF16 = 2.0 ** -14
TOL_FP8 = 2.0 ** -10


def tolerance(kind, v, bound, beta=0.0, c=None):
    rel = TOL_BF16 if kind == "bf16" else TOL_FP8
    tol = rel * bound + 2.0 ** -22 * np.abs(v)
    if kind == "bf16":
        tol = tol + 1e-6
    if c is not None and beta != 0.0:
        tol = tol + 2.0 ** -22 * np.abs(beta * c)
    return tol


def bf16_ulp(x):
    """Spacing of BF16 numbers at |x| (8 significant bits)."""
    ax = np.maximum(np.abs(x), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(ax)) - 7)


def check_f32(kind, got, v, bound, beta=0.0, c=None, what=""):
    tol = tolerance(kind, v, bound, beta, c)
    err = np.abs(got.astype(np.float64) - v)
    bad = ~(err <= tol)
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} outside tolerance; first at {tuple(i)}: "
            f"got {got[tuple(i)]!r} want {v[tuple(i)]!r} tol {tol[tuple(i)]!r}")
    return float((err / np.maximum(tol, 1e-300)).max()) if err.size else 0.0


def check_bf16(kind, got_bits, v, bound, beta=0.0, c=None, what=""):
    got = oracle.bf16_decode(got_bits)
    tol = tolerance(kind, v, bound, beta, c) + bf16_ulp(v)
    err = np.abs(got - v)
    bad = ~(err <= tol)
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} BF16 outputs outside tolerance; first at "
            f"{tuple(i)}: got {got[tuple(i)]!r} want {v[tuple(i)]!r}")
    return float((err / np.maximum(tol, 1e-300)).max()) if err.size else 0.0


def oracle_for(w, tiles=None, C_override=None, nthreads=None):
    """Oracle values and bounds for a synth.workloads.Workload."""
    in_type = oracle.IN_BF16 if w.kind == "bf16" else oracle.IN_E4M3
    mode = {"bf16": oracle.SCALE_NONE, "fp8_tensor": oracle.SCALE_TENSOR,
            "fp8_block": oracle.SCALE_BLOCK128, "fp8_mx": oracle.SCALE_MX32}[w.kind]
    C = w.C if C_override is None else C_override
    c_type = oracle.C_BF16 if (C is not None and C.dtype == np.uint16) else oracle.C_F32
    return oracle.gemm(w.M, w.N, w.K, w.A, w.lda, w.B, w.ldb, in_type=in_type, scale_mode=mode,
                       a_scale=w.a_scale, b_scale=w.b_scale, C=C,
                       ldc=(C.shape[1] if C is not None else 0), c_type=c_type, alpha=w.alpha,
                       beta=w.beta, tiles=tiles, nthreads=nthreads, a_fp8=w.a_fp8,
                       b_fp8=w.b_fp8, a_sf=w.a_sf, b_sf=w.b_sf)


def c_values(C):
    """Decoded C (float64) for tolerance terms."""
    if C is None:
        return None
    if C.dtype == np.uint16:
        return oracle.bf16_decode(C)
    return C.astype(np.float64)


# ------------------------------------------------------------- GPU side

def to_device(arr, dtype=None):
    import torch
    if arr is None:
        return None
    if arr.dtype == np.uint16:
        t = torch.from_numpy(np.ascontiguousarray(arr).view(np.int16))
        return t.cuda().view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(arr)).cuda()


def run(w, out=None, C=None, alpha=None, beta=None, stream=None, D=None):
    """Run a workload through the library; returns D on the device."""
    import torch

    import tensor_core_dense_gb300 as tcg
    out = out or w.out
    alpha = w.alpha if alpha is None else alpha
    beta = w.beta if beta is None else beta
    if C is None:
        C = w.C
    A = to_device(w.A)
    B = to_device(w.B)
    dt = torch.bfloat16 if out == "bf16" else torch.float32
    Cd = None
    if C is not None and beta != 0.0:
        Cd = to_device(C)
        if Cd.dtype != dt:
            Cd = Cd.to(dt)
        Cd = Cd[:, :w.N]
    if D is None:  # rows padded to a 16-byte pitch, as the library requires
        step = 8 if dt == torch.bfloat16 else 4
        D = torch.empty((w.M, -(-w.N // step) * step), dtype=dt, device="cuda")[:, :w.N]
    if w.kind == "bf16":
        tcg.gemm_bf16(A[:, :w.K], B[:, :w.K], D, Cd, alpha=alpha, beta=beta, stream=stream)
    elif w.kind == "fp8_mx":
        tcg.gemm_mxfp8(A[:, :w.K], B[:, :w.K], to_device(w.a_sf), to_device(w.b_sf), D, Cd,
                       a_format=w.a_fp8, b_format=w.b_fp8, alpha=alpha, beta=beta,
                       stream=stream)
    else:
        mode = tcg.SCALE_TENSOR if w.kind == "fp8_tensor" else tcg.SCALE_BLOCK128
        if w.a_fp8 == 0 and w.b_fp8 == 0:
            tcg.gemm_fp8_e4m3(A[:, :w.K], B[:, :w.K], to_device(w.a_scale),
                              to_device(w.b_scale), D, Cd, mode=mode, alpha=alpha, beta=beta,
                              stream=stream)
        else:
            tcg.gemm_fp8(A[:, :w.K], B[:, :w.K], to_device(w.a_scale), to_device(w.b_scale), D,
                         Cd, mode=mode, a_format=w.a_fp8, b_format=w.b_fp8, alpha=alpha,
                         beta=beta, stream=stream)
    return D


def d_to_host(D):
    import torch
    torch.cuda.synchronize()
    if D.dtype == torch.bfloat16:
        return D.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    return D.contiguous().cpu().numpy()


def sample_tiles(M, N, n=16, size=128, seed=0):
    """Output tiles for sampled parity: the first and last tiles plus seeded
    random ones (all clipped to the matrix); the same tiles bench.py's CPU
    baseline times."""
    from synth.workloads import sample_tiles as _tiles
    return _tiles(M, N, n=n, size=size, seed=seed)
