"""GPU parity of the microscaled FP8 GEMM (gemm_mxfp8) against the oracle.

The block-scaled MMA of "How Blackwell's Tensor Memory Actually Works"
("Quantization became an allocation problem"): one E8M0 scale per row and
32-wide K block of A and of B, applied by the tensor core.  Bit-exact cases
use small-integer codes and power-of-two scales that differ per (row, block),
so every misplaced scale, block or byte changes bits; the others compare
microscaled N(0, 1) data with outliers at the FP8 tolerance.
"""

from __future__ import annotations

import numpy as np
import pytest

import synth
import synth.workloads as W
from helpers import (c_values, check_bf16, check_f32, d_to_host, oracle_for, run, sample_tiles,
                     to_device)

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import tensor_core_dense_gb300 as tcg
    tcg.lib()
    yield
    assert tcg.last_device_status() == tcg.OK


def _pad(n, step):
    return -(-n // step) * step


def mx_case(M, N, K, seed, out="f32", alpha=1.0, beta=0.0, a_fmt=0, b_fmt=0, outliers=0.01):
    w = W.Workload(f"mx_{M}x{N}x{K}", M, N, K, "fp8_mx", out, alpha=alpha, beta=beta)
    fmt = {0: "e4m3", 1: "e5m2"}
    ld = _pad(K, 16)
    w.A, ea = synth.mx_quant(synth.values_f32(seed, 1, M, K, out_prob=outliers, out_factor=50.0),
                             ld=ld, fmt=fmt[a_fmt])
    w.B, eb = synth.mx_quant(synth.values_f32(seed, 2, N, K, out_prob=outliers, out_factor=50.0),
                             ld=ld, fmt=fmt[b_fmt])
    w.a_sf, w.b_sf = synth.mx_tile_sf(ea, K), synth.mx_tile_sf(eb, K)
    w.a_fp8, w.b_fp8 = a_fmt, b_fmt
    if beta != 0.0:
        if out == "bf16":
            w.C = synth.bf16(seed, 3, M, N, ld=_pad(N, 8))
        else:
            w.C = np.zeros((M, _pad(N, 4)), np.float32)
            w.C[:, :N] = synth.values_f32(seed, 3, M, N)
    return w


def check_full(w, D):
    v, bound = oracle_for(w)
    got = d_to_host(D)[:, :w.N]
    c = c_values(w.C)[:, :w.N] if w.C is not None else None
    if got.dtype == np.uint16:
        return check_bf16("fp8", got, v, bound, w.beta, c, what=w.name)
    return check_f32("fp8", got, v, bound, w.beta, c, what=w.name)


@pytest.mark.parametrize("M,N,K", [(256, 256, 256), (300, 520, 384), (1000, 700, 1111),
                                   (128, 256, 128), (520, 260, 4096), (1, 1, 32), (37, 3, 100)])
def test_mx_scale_indexing_bit_exact(M, N, K):
    """Codes -3..3 and scales 2^-2..2^2 that depend on (row, block): all sums
    are exact in FP32, so the output must equal the oracle bit for bit."""
    rng = np.random.default_rng(M + 3 * N + K)
    KB = -(-K // 32)
    ld = _pad(K, 16)
    ints = np.array([-3, -2, -1, 0, 1, 2, 3], np.float32)
    a = np.zeros((M, ld), np.float32)
    b = np.zeros((N, ld), np.float32)
    a[:, :K] = rng.choice(ints, size=(M, K))
    b[:, :K] = rng.choice(ints, size=(N, K))
    ea = np.array([[125 + (3 * i + kb) % 5 for kb in range(KB)] for i in range(M)], np.uint8)
    eb = np.array([[125 + (5 * j + 2 * kb) % 5 for kb in range(KB)] for j in range(N)], np.uint8)
    w = W.Workload("mx_exact", M, N, K, "fp8_mx", "f32")
    w.A, w.B = synth.to_e4m3(a), synth.to_e4m3(b)
    w.a_sf, w.b_sf = synth.mx_tile_sf(ea, K), synth.mx_tile_sf(eb, K)
    v, _ = oracle_for(w)
    assert np.array_equal(d_to_host(run(w)).astype(np.float64), v)


# Shapes that take each branch of the pair schedule (whole waves, a tail cut
# into halves, small grids), ragged M, N and K, both output types, beta.
@pytest.mark.parametrize("M,N,K", [(256, 256, 512), (257, 300, 1000), (512, 1024, 4096),
                                   (2048, 2560, 1024), (777, 3000, 1111), (100, 4096, 256)])
@pytest.mark.parametrize("out,beta", [("f32", 0.0), ("bf16", 0.0), ("bf16", 1.0)])
def test_mx_shapes(M, N, K, out, beta):
    w = mx_case(M, N, K, seed=M + 5 * N + K, out=out, beta=beta, alpha=0.5)
    check_full(w, run(w))


# Units of one to three K steps (a step is 4 scale blocks, 128 K values) on
# many tiles per pair: every step is also its unit's first or last.
@pytest.mark.parametrize("M,N,K", [(4096, 2560, 32), (4096, 2560, 128), (4096, 2560, 256),
                                   (3000, 2600, 352)])
def test_mx_one_to_three_step_units(M, N, K):
    w = mx_case(M, N, K, seed=M + N + K, out="f32")
    check_full(w, run(w))


@pytest.mark.parametrize("a_fmt,b_fmt", [(1, 1), (0, 1), (1, 0)])
def test_mx_e5m2_operands(a_fmt, b_fmt):
    w = mx_case(384, 640, 768, seed=90 + 2 * a_fmt + b_fmt, a_fmt=a_fmt, b_fmt=b_fmt)
    check_full(w, run(w))


def test_mx_in_place_and_determinism():
    w = mx_case(600, 1000, 1024, seed=95, out="bf16", beta=-0.75)
    import tensor_core_dense_gb300 as tcg
    D = to_device(w.C)[:, :w.N].clone()
    A, B = to_device(w.A)[:, :w.K], to_device(w.B)[:, :w.K]
    sa, sb = to_device(w.a_sf), to_device(w.b_sf)
    tcg.gemm_mxfp8(A, B, sa, sb, D, D, alpha=w.alpha, beta=w.beta)
    check_full(w, D)
    d1 = d_to_host(run(w))
    d2 = d_to_host(run(w))
    assert np.array_equal(d1, d2)


def test_mx_output_guard_bands_untouched():
    w = mx_case(300, 260, 384, seed=96, out="f32")
    step = 4
    ldd = _pad(w.N, step) + 2 * step
    big = torch.full((w.M + 2, ldd), float("nan"), dtype=torch.float32, device="cuda")
    sentinel = big.clone()
    D = big[1:w.M + 1, step:step + w.N]
    run(w, D=D)
    torch.cuda.synchronize()
    mask = torch.ones_like(big, dtype=torch.bool)
    mask[1:w.M + 1, step:step + w.N] = False
    assert torch.equal(big[mask].view(torch.int32), sentinel[mask].view(torch.int32))
    check_full(w, D)


def test_mx_4096_cubed_sampled():
    """The benchmark's microscaled workload at full size, in its launch
    configuration, on 16 seeded 128 x 128 tiles (first and last included)."""
    w = W.make("mxfp8_4096")
    for out in ("f32", "bf16"):
        D = run(w, out=out)
        tiles = sample_tiles(w.M, w.N, n=16)
        vs, bs = oracle_for(w, tiles=tiles)
        got = d_to_host(D)
        for (i0, j0, mi, nj), v, b in zip(tiles, vs, bs):
            g = got[i0:i0 + mi, j0:j0 + nj]
            if out == "bf16":
                check_bf16("fp8", g, v, b, what=f"mx 4096 {i0},{j0}")
            else:
                check_f32("fp8", g, v, b, what=f"mx 4096 {i0},{j0}")
