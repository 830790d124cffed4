"""GPU parity: the CUDA library (through its C ABI) against the CPU oracle.

Small and ragged shapes are compared element by element on the whole output;
the full-size workloads on seeded samples of 128 x 128 output tiles, in the
same launch configuration the benchmark times.  Bit-exact cases use inputs
whose products and sums are exact in FP32 (small integers, power-of-two
scales), so any indexing or scale-placement error changes bits.
"""

from __future__ import annotations

import numpy as np
import pytest

import oracle
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


def bf16_case(M, N, K, seed, out="f32", alpha=1.0, beta=0.0, dist="normal"):
    w = W.Workload(f"bf16_{M}x{N}x{K}", M, N, K, "bf16", out, alpha=alpha, beta=beta)
    kw = dict(dist="uniform", p0=-1, p1=1) if dist == "uniform" else {}
    w.A = synth.bf16(seed, 1, M, K, ld=_pad(K, 8), **kw)
    w.B = synth.bf16(seed, 2, N, K, ld=_pad(K, 8), **kw)
    if beta != 0.0:
        if out == "bf16":
            w.C = synth.bf16(seed, 3, M, N, ld=_pad(N, 8))
        else:
            w.C = np.zeros((M, _pad(N, 4)), np.float32)
            w.C[:, :N] = synth.values_f32(seed, 3, M, N)
    return w


def fp8_case(M, N, K, seed, mode, out="f32", alpha=1.0, beta=0.0, outliers=0.0):
    kind = "fp8_tensor" if mode == "tensor" else "fp8_block"
    w = W.Workload(f"fp8_{mode}_{M}x{N}x{K}", M, N, K, kind, out, alpha=alpha, beta=beta)
    xa = synth.values_f32(seed, 1, M, K, out_prob=outliers, out_factor=50.0)
    xb = synth.values_f32(seed, 2, N, K, out_prob=outliers, out_factor=50.0)
    if mode == "tensor":
        w.A, w.a_scale = synth.e4m3_tensor(xa, ld=_pad(K, 16))
        w.B, w.b_scale = synth.e4m3_tensor(xb, ld=_pad(K, 16))
    else:
        w.A, w.a_scale = synth.e4m3_rowblock(xa, ld=_pad(K, 16))
        w.B, w.b_scale = synth.e4m3_block128(xb, ld=_pad(K, 16))
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
    kind = "bf16" if w.kind == "bf16" else "fp8"
    if got.dtype == np.uint16:
        return check_bf16(kind, got, v, bound, w.beta, c, what=w.name)
    return check_f32(kind, got, v, bound, w.beta, c, what=w.name)


# ------------------------------------------------------------------ BF16

def test_bf16_256_full_output():
    """256^3, uniform [-1, 1), FP32 output, beta = 0: every output checked."""
    w = W.make("bf16_256")
    check_full(w, run(w))


BF16_SHAPES = [(1, 1, 1), (1, 8, 8), (7, 13, 50), (128, 256, 64), (129, 257, 65),
               (255, 511, 200), (300, 200, 1000), (64, 1000, 136), (1000, 48, 72),
               (384, 768, 4096)]


@pytest.mark.parametrize("M,N,K", BF16_SHAPES)
@pytest.mark.parametrize("out,beta", [("f32", 0.0), ("bf16", 0.0), ("f32", -0.5), ("bf16", 1.0)])
def test_bf16_shapes(M, N, K, out, beta):
    w = bf16_case(M, N, K, seed=M * 7 + N * 3 + K, out=out, alpha=1.25 if beta else 1.0,
                  beta=beta)
    check_full(w, run(w))


# Shapes that take each branch of the scheduler on a 152-SM GB300: a partial
# last wave cut into quarter tiles (160 tiles), half tiles (54 tiles), kept
# whole (256 tiles: 104 left over), and small grids cut into quarters (BF16
# and FP8).
@pytest.mark.parametrize("M,N,K,kind", [(2048, 2560, 1024, "bf16"), (1100, 1300, 700, "bf16"),
                                        (1000, 1000, 2048, "fp8"), (300, 600, 8192, "bf16"),
                                        (4096, 2560, 512, "fp8"), (2048, 4096, 512, "bf16")])
@pytest.mark.parametrize("out,beta", [("f32", 0.0), ("bf16", 1.0)])
def test_tail_schedules(M, N, K, kind, out, beta):
    if kind == "bf16":
        w = bf16_case(M, N, K, seed=M + 2 * N + K, out=out, beta=beta)
    else:
        w = fp8_case(M, N, K, seed=M + 2 * N + K, mode="tensor", out=out, beta=beta)
    check_full(w, run(w))


# Both dense kernels on every kind of shape: the one-SM 128 x 256 kernel and
# the CTA-pair 256 x 256 kernel (the library picks one by shape; TCG_KERNEL
# forces either).
@pytest.mark.parametrize("kernel", ["1cta", "2cta"])
@pytest.mark.parametrize("M,N,K,kind,out,beta", [
    (1, 8, 8, "bf16", "f32", 0.0), (129, 257, 65, "bf16", "bf16", 1.0),
    (1000, 1000, 2048, "fp8", "bf16", 0.0), (2048, 2560, 1024, "bf16", "f32", -0.5),
    (4096, 2560, 512, "fp8", "f32", 0.0), (777, 3000, 1111, "bf16", "bf16", 1.0),
    (2048, 4096, 512, "bf16", "f32", 0.0), (3, 3000, 1000, "fp8", "bf16", 1.0),
    (5, 1000, 4100, "bf16", "f32", 0.0), (12, 700, 2000, "fp8", "f32", 0.0)])
def test_dense_kernels_both_paths(monkeypatch, kernel, M, N, K, kind, out, beta):
    monkeypatch.setenv("TCG_KERNEL", kernel)
    if kind == "bf16":
        w = bf16_case(M, N, K, seed=M + N + 5 * K, out=out, beta=beta)
    else:
        w = fp8_case(M, N, K, seed=M + N + 5 * K, mode="tensor", out=out, beta=beta)
    check_full(w, run(w))


# M <= 128 BF16 and per-tensor FP8 on the swap-AB skinny kernel (the library
# routes decode-sized shapes there; TCG_KERNEL=skinny forces it): ragged M,
# N and K, the cluster-pair split, whole tiles per CTA (more N tiles than
# half the SMs), beta*C, both output types.
@pytest.mark.parametrize("M,N,K", [(1, 8, 8), (7, 13, 50), (16, 1000, 1024), (33, 300, 2000),
                                   (64, 8192, 1024), (100, 2048, 3000), (128, 256, 64),
                                   (128, 20000, 512)])
@pytest.mark.parametrize("kind", ["bf16", "fp8"])
@pytest.mark.parametrize("out,beta", [("f32", 0.0), ("bf16", 1.0)])
def test_dense_small_m_on_skinny_kernel(monkeypatch, M, N, K, kind, out, beta):
    monkeypatch.setenv("TCG_KERNEL", "skinny")
    if kind == "bf16":
        w = bf16_case(M, N, K, seed=M + 3 * N + K, out=out, alpha=0.75, beta=beta)
    else:
        w = fp8_case(M, N, K, seed=M + 3 * N + K, mode="tensor", out=out, beta=beta)
    check_full(w, run(w))


# Units one or two K steps long (a step is 128 bytes of K) on many tiles per
# CTA or pair: every step is also its unit's first or last, so the MMA
# thread's test of the next step is skipped or falls on the next unit's first
# stage, and tiles change every step or two.
@pytest.mark.parametrize("kernel", ["1cta", "2cta"])
@pytest.mark.parametrize("M,N,K,kind", [(4096, 2560, 64, "bf16"), (4096, 2560, 128, "bf16"),
                                        (3000, 2600, 40, "bf16"), (4096, 2560, 128, "fp8"),
                                        (4096, 2560, 256, "fp8"), (3000, 2600, 100, "fp8")])
def test_one_and_two_step_units(monkeypatch, kernel, M, N, K, kind):
    monkeypatch.setenv("TCG_KERNEL", kernel)
    if kind == "bf16":
        w = bf16_case(M, N, K, seed=M + N + K, out="f32")
    else:
        w = fp8_case(M, N, K, seed=M + N + K, mode="tensor", out="f32")
    check_full(w, run(w))


# The skinny kernel with K ranges of one or two steps per CTA: BF16 and
# per-tensor FP8 (its one-scale form), and block-scaled FP8 at Mp = 64 (the
# issue block) and Mp = 128 (the plain wait order).
@pytest.mark.parametrize("M,K,kind", [(16, 64, "bf16"), (128, 128, "bf16"), (64, 128, "tensor"),
                                      (128, 256, "tensor"), (64, 128, "block"),
                                      (64, 256, "block"), (128, 128, "block"),
                                      (128, 256, "block")])
def test_skinny_one_and_two_step_ranges(monkeypatch, M, K, kind):
    if kind == "bf16":
        monkeypatch.setenv("TCG_KERNEL", "skinny")
        w = bf16_case(M, 8192, K, seed=M + K, out="f32")
    elif kind == "tensor":
        monkeypatch.setenv("TCG_KERNEL", "skinny")
        w = fp8_case(M, 8192, K, seed=M + K, mode="tensor", out="f32")
    else:
        w = fp8_case(M, 8192, K, seed=M + K, mode="block", out="f32", outliers=0.01)
    check_full(w, run(w))


def test_dense_small_m_skinny_deterministic(monkeypatch):
    monkeypatch.setenv("TCG_KERNEL", "skinny")
    w = bf16_case(64, 3000, 8192, seed=8, out="f32")
    d1, d2 = d_to_host(run(w)), d_to_host(run(w))
    assert np.array_equal(d1.view(np.uint32), d2.view(np.uint32))


def test_tail_schedule_deterministic():
    w = bf16_case(1100, 1300, 4096, seed=4, out="f32")
    d1, d2 = d_to_host(run(w)), d_to_host(run(w))
    assert np.array_equal(d1.view(np.uint32), d2.view(np.uint32))


def test_bf16_one_hot_indexing_bit_exact():
    """A has one 1 per row at column pi(i): the product is exactly B[j, pi(i)], so
    D[i, j] = fp32(alpha * B[j, pi(i)] + beta * C[i, j]) bit for bit (alpha, beta
    powers of two: the only rounding is the final FP32 sum), for padded
    leading dimensions and ragged tiles."""
    M, N, K = 333, 517, 700
    lda, ldb = 712, 704
    rng = np.random.default_rng(3)
    pi = rng.integers(0, K, size=M)
    a = np.zeros((M, lda), np.float32)
    a[np.arange(M), pi] = 1.0
    w = W.Workload("onehot", M, N, K, "bf16", "f32", alpha=2.0, beta=0.5)
    w.A = synth.to_bf16(a)
    w.B = synth.bf16(9, 2, N, K, ld=ldb)
    w.C = np.zeros((M, 520), np.float32)
    w.C[:, :N] = rng.integers(-64, 64, size=(M, N)).astype(np.float32)
    got = d_to_host(run(w))[:, :N].astype(np.float64)
    b = oracle.bf16_decode(w.B).reshape(N, ldb)
    want = (2.0 * b[:, pi].T + 0.5 * w.C[:, :N]).astype(np.float32).astype(np.float64)
    assert np.array_equal(got, want)


def test_bf16_all_ones_equals_k():
    M, N, K = 130, 260, 4000
    ones = synth.to_bf16(np.ones((max(M, N), K), np.float32))
    w = W.Workload("ones", M, N, K, "bf16", "f32")
    w.A, w.B = ones[:M], ones[:N]
    assert (d_to_host(run(w)) == K).all()


def test_k_zero_gives_beta_c():
    import tensor_core_dense_gb300 as tcg
    M, N = 37, 64
    C = torch.randn(M, N, device="cuda")
    D = torch.full((M, N), float("nan"), device="cuda")
    A = torch.empty((M, 0), dtype=torch.bfloat16, device="cuda")
    B = torch.empty((N, 0), dtype=torch.bfloat16, device="cuda")
    st = tcg.gemm_bf16_raw(M, N, 0, A.data_ptr(), 8, B.data_ptr(), 8, C.data_ptr(), N,
                           D.data_ptr(), N, tcg.OUT_F32, 1.0, -2.0,
                           torch.cuda.current_stream().cuda_stream)
    assert st == tcg.OK
    torch.cuda.synchronize()
    assert torch.equal(D, -2.0 * C)


# ------------------------------------------------------------ FP8 per tensor

FP8_SHAPES = [(1, 16, 32), (128, 256, 128), (200, 300, 1000), (513, 700, 384),
              (256, 1024, 4096)]


@pytest.mark.parametrize("M,N,K", FP8_SHAPES)
@pytest.mark.parametrize("out,beta", [("f32", 0.0), ("bf16", 0.0), ("bf16", 1.0)])
def test_fp8_tensor_shapes(M, N, K, out, beta):
    w = fp8_case(M, N, K, seed=M + N + K, mode="tensor", out=out, beta=beta)
    check_full(w, run(w))


def test_fp8_tensor_scales_bit_exact():
    """Small-integer E4M3 codes with power-of-two scales: D is exact in FP32."""
    M, N, K = 150, 270, 512
    rng = np.random.default_rng(5)
    ints = np.array([-4, -3, -2, -1, 0, 1, 2, 3, 4], np.float32)
    w = W.Workload("fp8_exact", M, N, K, "fp8_tensor", "f32", alpha=1.0)
    w.A = synth.to_e4m3(rng.choice(ints, size=(M, K)))
    w.B = synth.to_e4m3(rng.choice(ints, size=(N, K)))
    w.a_scale = np.array([2.0 ** -3], np.float32)
    w.b_scale = np.array([2.0 ** 5], np.float32)
    v, _ = oracle_for(w)
    assert np.array_equal(d_to_host(run(w)).astype(np.float64), v)


# ------------------------------------------------------- FP8 block, skinny M

SKINNY = [(1, 128, 128), (16, 300, 200), (17, 1024, 4096), (64, 2000, 1000),
          (100, 1024, 4096), (128, 256, 8192), (128, 4096, 1024),
          # N tiles in [SMs/3, SMs/2]: each tile's K range is cut in two and the
          # halves are joined by a cluster of two CTAs (odd and even K blocks)
          (5, 7000, 1000), (33, 6528, 384), (100, 8100, 256), (128, 9728, 1152)]


@pytest.mark.parametrize("M,N,K", SKINNY)
@pytest.mark.parametrize("out,beta", [("f32", 0.0), ("bf16", 0.0), ("bf16", -1.0)])
def test_fp8_block_skinny_shapes(M, N, K, out, beta):
    w = fp8_case(M, N, K, seed=3 * M + N + K, mode="block", out=out, beta=beta, outliers=0.01)
    check_full(w, run(w))


@pytest.mark.parametrize("M,N,K,kernel", [
    (5, 260, 300, None), (64, 1024, 4096, None), (128, 2048, 2048, None), (20, 8192, 640, None),
    (300, 260, 384, "2cta"), (256, 4096, 512, "2cta"), (520, 2300, 1100, "2cta"),
    (300, 260, 384, "skinny"), (256, 4096, 512, "skinny")])
def test_fp8_block_scale_indexing_bit_exact(monkeypatch, M, N, K, kernel):
    """Power-of-two block scales that depend on (row, K block) and (N block,
    K block) with small-integer codes: every misplaced scale changes bits."""
    if kernel:
        monkeypatch.setenv("TCG_KERNEL", kernel)
    KB, NB = (K + 127) // 128, (N + 127) // 128
    rng = np.random.default_rng(M + N)
    ints = np.array([-3, -2, -1, 0, 1, 2, 3], np.float32)
    w = W.Workload("fp8_block_exact", M, N, K, "fp8_block", "f32")
    ldk = _pad(K, 16)
    a = np.zeros((M, ldk), np.float32)
    b = np.zeros((N, ldk), np.float32)
    a[:, :K] = rng.choice(ints, size=(M, K))
    b[:, :K] = rng.choice(ints, size=(N, K))
    w.A, w.B = synth.to_e4m3(a), synth.to_e4m3(b)
    w.a_scale = np.array([2.0 ** ((i % 3) - 1 + (kb % 2)) for kb in range(KB) for i in range(M)],
                         np.float32)
    w.b_scale = np.array([2.0 ** ((nb + kb) % 2) for nb in range(NB) for kb in range(KB)],
                         np.float32)
    v, _ = oracle_for(w)
    assert np.array_equal(d_to_host(run(w)).astype(np.float64), v)


# M > 128, on both kernels that take it: the pair-tile kernel (256 x 256
# tiles; halves at the tail; whole waves plus a split tail at 2560 x 2048) and
# the skinny kernel with A in chunks of 128 rows (the general split, the
# cluster pair at 64 tiles, unsplit tiles at 128 tiles).
@pytest.mark.parametrize("kernel", ["2cta", "skinny"])
@pytest.mark.parametrize("M,N,K", [(129, 256, 512), (300, 1000, 1024), (256, 4096, 512),
                                   (1024, 2048, 1536), (777, 3000, 2200), (2560, 2048, 512),
                                   (513, 130, 4100)])
@pytest.mark.parametrize("out,beta", [("f32", 0.0), ("bf16", 1.0)])
def test_fp8_block_scaled_large_m(monkeypatch, kernel, M, N, K, out, beta):
    monkeypatch.setenv("TCG_KERNEL", kernel)
    w = fp8_case(M, N, K, seed=M + 3 * N + K, mode="block", out=out, beta=beta, outliers=0.01)
    check_full(w, run(w))


def test_fp8_block_alternating_schedules():
    """A call with many tiles (whole tiles per CTA), one with few (K split
    over clusters), then the first shape again: all correct."""
    many = fp8_case(600, 4096, 1024, seed=91, mode="block", out="f32", outliers=0.01)
    few = fp8_case(16, 1000, 2048, seed=92, mode="block", out="f32", outliers=0.01)
    for w in (many, few, many, few):
        check_full(w, run(w))


def test_fp8_block_scaled_4096_cubed_sampled():
    w = fp8_case(4096, 4096, 4096, seed=17, mode="block", out="bf16", outliers=0.01)
    _sampled(w, out="f32")
    _sampled(w, out="bf16")


@pytest.mark.parametrize("M,N", [(64, 4096), (16, 8192), (600, 2048), (4096, 4096)])
def test_fp8_block_skinny_deterministic(M, N):
    w = fp8_case(M, N, 4096, seed=11, mode="block", out="f32", outliers=0.01)
    d1 = d_to_host(run(w))
    d2 = d_to_host(run(w))
    assert np.array_equal(d1.view(np.uint32), d2.view(np.uint32))


# ------------------------------------------------------------ full workloads

def _sampled(w, out, ntiles=16):
    D = run(w, out=out)
    tiles = sample_tiles(w.M, w.N, n=ntiles)
    vs, bs = oracle_for(w, tiles=tiles)
    got = d_to_host(D)
    kind = "bf16" if w.kind == "bf16" else "fp8"
    worst = 0.0
    for (i0, j0, mi, nj), v, b in zip(tiles, vs, bs):
        g = got[i0:i0 + mi, j0:j0 + nj]
        c = c_values(w.C[i0:i0 + mi, j0:j0 + nj]) if w.C is not None else None
        if g.dtype == np.uint16:
            worst = max(worst, check_bf16(kind, g, v, b, w.beta, c, what=f"{w.name} {i0},{j0}"))
        else:
            worst = max(worst, check_f32(kind, g, v, b, w.beta, c, what=f"{w.name} {i0},{j0}"))
    del D
    torch.cuda.empty_cache()
    return worst


@pytest.mark.parametrize("name", ["bf16_4096", "fp8_4096", "bf16_mlp", "fp8_block_4096",
                                  "bf16_skinny_16"])
def test_full_size_sampled(name):
    w = W.make(name)
    _sampled(w, out="f32")   # pre-cast check with the same kernel
    _sampled(w, out=w.out)   # the workload's own output type


@pytest.mark.parametrize("M", [16, 64, 128])
def test_skinny_full_size_sampled(M):
    w = W.make(f"fp8_skinny_{M}")
    for out in ("f32", "bf16"):
        D = run(w, out=out)
        tiles = [(0, j0, M, 128) for j0 in (0, 128, 4096, 8064)] + [
            (0, int(j), M, 128) for j in np.random.default_rng(M).integers(0, 63, 4) * 128]
        vs, bs = oracle_for(w, tiles=tiles)
        got = d_to_host(D)
        for (i0, j0, mi, nj), v, b in zip(tiles, vs, bs):
            g = got[i0:i0 + mi, j0:j0 + nj]
            if out == "f32":
                check_f32("fp8", g, v, b, what=f"{w.name} {j0}")
            else:
                check_bf16("fp8", g, v, b, what=f"{w.name} {j0}")


def test_launch_counter_and_status():
    import tensor_core_dense_gb300 as tcg
    n0 = tcg.launch_count()
    w = bf16_case(64, 64, 64, seed=1)
    run(w)
    torch.cuda.synchronize()
    assert tcg.launch_count() == n0 + 1
    assert tcg.last_device_status() == tcg.OK


# --------------------------------------------------------- E5M2 operands

FMTS = [(1, 1), (0, 1), (1, 0)]  # (A, B): 0 = E4M3, 1 = E5M2


def fp8_fmt_case(M, N, K, seed, mode, a_fmt, b_fmt, out="f32", beta=0.0):
    """FP8 operands in the given encodings: N(0,1) values with 1% outliers x50,
    cast with a scale that puts the largest magnitudes near the format's top
    (448 or 57344), per tensor or in the 1 x 128 / 128 x 128 block layouts."""
    w = W.Workload(f"fp8_{a_fmt}{b_fmt}_{mode}_{M}x{N}x{K}", M, N, K,
                   "fp8_tensor" if mode == "tensor" else "fp8_block", out, beta=beta)
    w.a_fp8, w.b_fp8 = a_fmt, b_fmt
    ldk = _pad(K, 16)
    KB, MB, NB = (K + 127) // 128, 1, (N + 127) // 128

    def cast(x, fmt, scale_el):
        q = np.zeros((x.shape[0], ldk), np.uint8)
        y = (x / scale_el).astype(np.float32)
        q[:, :K] = synth.to_e5m2(y) if fmt == 1 else synth.to_e4m3(y)
        return q

    top = {0: 448.0, 1: 57344.0}
    xa = synth.values_f32(seed, 1, M, K, out_prob=0.01, out_factor=50.0)
    xb = synth.values_f32(seed, 2, N, K, out_prob=0.01, out_factor=50.0)
    if mode == "tensor":
        sa = np.array([np.abs(xa).max() / top[a_fmt]], np.float32)
        sb = np.array([np.abs(xb).max() / top[b_fmt]], np.float32)
        w.A, w.B = cast(xa, a_fmt, sa[0]), cast(xb, b_fmt, sb[0])
    else:
        kb = np.arange(K) // 128
        sa2 = np.stack([np.abs(xa[:, kb == j]).max(1) for j in range(KB)]) / top[a_fmt]  # KB x M
        sb2 = np.array([[np.abs(xb[n * 128:(n + 1) * 128][:, kb == j]).max() for j in range(KB)]
                        for n in range(NB)]) / top[b_fmt]  # NB x KB
        sa2 = np.maximum(sa2, 1e-30).astype(np.float32)
        sb2 = np.maximum(sb2, 1e-30).astype(np.float32)
        w.A = cast(xa, a_fmt, sa2.T[:, kb])
        w.B = cast(xb, b_fmt, np.repeat(sb2, 128, axis=0)[:N][:, kb])
        sa, sb = sa2.ravel(), sb2.ravel()
    w.a_scale, w.b_scale = sa, sb
    if beta != 0.0:
        if out == "bf16":
            w.C = synth.bf16(seed, 3, M, N, ld=_pad(N, 8))
        else:
            w.C = np.zeros((M, _pad(N, 4)), np.float32)
            w.C[:, :N] = synth.values_f32(seed, 3, M, N)
    return w


@pytest.mark.parametrize("kernel", ["1cta", "2cta"])
@pytest.mark.parametrize("a_fmt,b_fmt", FMTS)
@pytest.mark.parametrize("M,N,K,out,beta", [(200, 300, 520, "f32", 0.0),
                                            (640, 512, 1024, "bf16", 1.0)])
def test_fp8_e5m2_tensor_scaled(monkeypatch, kernel, a_fmt, b_fmt, M, N, K, out, beta):
    monkeypatch.setenv("TCG_KERNEL", kernel)
    w = fp8_fmt_case(M, N, K, seed=M + K + 7 * a_fmt + b_fmt, mode="tensor", a_fmt=a_fmt,
                     b_fmt=b_fmt, out=out, beta=beta)
    check_full(w, run(w))


@pytest.mark.parametrize("a_fmt,b_fmt", FMTS)
@pytest.mark.parametrize("M,N,K", [(16, 1000, 1024), (100, 8192, 512), (128, 384, 2048)])
def test_fp8_e5m2_block_scaled_skinny(a_fmt, b_fmt, M, N, K):
    w = fp8_fmt_case(M, N, K, seed=M + N + K + 7 * a_fmt + b_fmt, mode="block", a_fmt=a_fmt,
                     b_fmt=b_fmt)
    check_full(w, run(w))


@pytest.mark.parametrize("a_fmt,b_fmt", FMTS)
@pytest.mark.parametrize("M,N,K", [(300, 700, 1000), (1024, 1024, 2048)])
def test_fp8_e5m2_block_scaled_pair(a_fmt, b_fmt, M, N, K):
    w = fp8_fmt_case(M, N, K, 7 * M + N, "block", a_fmt, b_fmt)
    check_full(w, run(w))


@pytest.mark.parametrize("a_fmt,b_fmt", FMTS)
def test_fp8_e5m2_small_integers_bit_exact(a_fmt, b_fmt):
    """Small integers (exact in both encodings) with power-of-two scales: the
    FP32 accumulation is exact, so a format mix-up changes bits."""
    M, N, K = 130, 260, 384
    rng = np.random.default_rng(5 + a_fmt + 2 * b_fmt)
    ints = np.array([-6, -5, -3, -2, -1, 0, 1, 2, 3, 5, 6], np.float32)
    ldk = _pad(K, 16)
    a = np.zeros((M, ldk), np.float32)
    b = np.zeros((N, ldk), np.float32)
    a[:, :K] = rng.choice(ints, size=(M, K))
    b[:, :K] = rng.choice(ints, size=(N, K))
    enc = {0: synth.to_e4m3, 1: synth.to_e5m2}
    w = W.Workload("fp8_int_exact", M, N, K, "fp8_tensor", "f32")
    w.a_fp8, w.b_fp8 = a_fmt, b_fmt
    w.A, w.B = enc[a_fmt](a), enc[b_fmt](b)
    w.a_scale = np.array([2.0 ** -2], np.float32)
    w.b_scale = np.array([2.0 ** 3], np.float32)
    v, _ = oracle_for(w)
    for kern in ("1cta", "2cta"):
        import os
        os.environ["TCG_KERNEL"] = kern
        try:
            assert np.array_equal(d_to_host(run(w)).astype(np.float64), v), kern
        finally:
            del os.environ["TCG_KERNEL"]


# ------------------------------------------------------------- guard bands

@pytest.mark.parametrize("case", ["bf16_1cta", "bf16_2cta", "fp8_tensor", "fp8_block",
                                  "fp8_block_pair", "fp8_block_large_m"])
def test_output_guard_bands_untouched(monkeypatch, case):
    """D is a view into a larger buffer filled with a sentinel: the kernels
    write exactly the M x N view (no row, column or padding outside it)."""
    if case.startswith("bf16"):
        monkeypatch.setenv("TCG_KERNEL", case.split("_")[1])
        w = bf16_case(300, 200, 96, seed=51, out="f32")
    elif case == "fp8_tensor":
        w = fp8_case(300, 260, 128, seed=52, mode="tensor", out="bf16")
    elif case == "fp8_block":
        w = fp8_case(20, 300, 256, seed=53, mode="block", out="f32")
    elif case == "fp8_block_large_m":
        w = fp8_case(300, 260, 384, seed=55, mode="block", out="bf16", beta=1.0)
    else:
        w = fp8_case(100, 8192, 256, seed=54, mode="block", out="bf16")
    dt = torch.float32 if w.out == "f32" else torch.bfloat16
    step = 4 if dt == torch.float32 else 8
    ldd = _pad(w.N, step) + 2 * step
    big = torch.full((w.M + 2, ldd), float("nan"), dtype=dt, device="cuda")
    sentinel = big.clone()
    D = big[1:w.M + 1, step:step + w.N]
    run(w, D=D)
    torch.cuda.synchronize()
    mask = torch.ones_like(big, dtype=torch.bool)
    mask[1:w.M + 1, step:step + w.N] = False
    outside = big[mask].view(torch.int16 if dt == torch.bfloat16 else torch.int32)
    expect = sentinel[mask].view(torch.int16 if dt == torch.bfloat16 else torch.int32)
    assert torch.equal(outside, expect), "a kernel wrote outside D"
    check_full(w, D)


# ------------------------------------------------------------ maximum sizes

def test_bf16_output_beyond_2_31_elements():
    """A 65,536 x 40,960 output (2.7e9 elements, 5.4 GB of BF16): row and
    column offsets past 2^31 elements, checked on the corner tiles."""
    M, N, K = 65536, 40960, 16
    w = W.Workload("bf16_huge_mn", M, N, K, "bf16", "bf16")
    w.A = synth.bf16(61, 1, M, K)
    w.B = synth.bf16(61, 2, N, K)
    D = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    run(w, D=D)
    torch.cuda.synchronize()
    tiles = [(0, 0, 128, 128), (M - 128, N - 128, 128, 128), (M - 100, 0, 100, 128),
             (0, N - 100, 128, 100), (40000, 20000, 128, 128)]
    vs, bs = oracle_for(w, tiles=tiles)
    for (i0, j0, mi, nj), v, b in zip(tiles, vs, bs):
        got = D[i0:i0 + mi, j0:j0 + nj].contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
        check_bf16("bf16", got, v, b, what=f"huge {i0},{j0}")
    del D
    torch.cuda.empty_cache()


# D = alpha*A*B + beta*D in place (C and D the same array, which the ABI
# allows when ldc == ldd): every kernel reads an output's C value in the thread
# that then writes it, once.
@pytest.mark.parametrize("case", ["bf16_1cta", "bf16_2cta", "fp8_tensor", "fp8_skinny",
                                  "fp8_skinny_split", "fp8_block_pair", "k0"])
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_d_aliases_c_in_place(monkeypatch, case, out):
    if case.startswith("bf16"):
        monkeypatch.setenv("TCG_KERNEL", case.split("_")[1])
        w = bf16_case(300, 520, 200, seed=71, out=out, alpha=0.5, beta=-1.5)
    elif case == "fp8_tensor":
        w = fp8_case(300, 520, 256, seed=72, mode="tensor", out=out, beta=2.0)
    elif case == "fp8_skinny":
        w = fp8_case(40, 8192, 512, seed=73, mode="block", out=out, beta=1.0)
    elif case == "fp8_skinny_split":
        w = fp8_case(64, 1000, 4096, seed=74, mode="block", out=out, beta=1.0)
    elif case == "fp8_block_pair":
        w = fp8_case(600, 1000, 1024, seed=75, mode="block", out=out, beta=-0.75)
    else:
        w = bf16_case(100, 72, 0, seed=76, out=out, beta=3.0)
        w.A = np.zeros((100, 8), np.uint16)
        w.B = np.zeros((72, 8), np.uint16)
    dt = torch.bfloat16 if out == "bf16" else torch.float32
    step = 8 if out == "bf16" else 4
    D = torch.empty((w.M, _pad(w.N, step)), dtype=dt, device="cuda")[:, :w.N]
    cdev = to_device(w.C)
    D.copy_(cdev[:, :w.N].to(dt))
    import tensor_core_dense_gb300 as tcg
    A, B = to_device(w.A), to_device(w.B)
    if w.kind == "bf16":
        tcg.gemm_bf16(A[:, :w.K], B[:, :w.K], D, D, alpha=w.alpha, beta=w.beta)
    else:
        mode = tcg.SCALE_TENSOR if w.kind == "fp8_tensor" else tcg.SCALE_BLOCK128
        tcg.gemm_fp8_e4m3(A[:, :w.K], B[:, :w.K], to_device(w.a_scale), to_device(w.b_scale), D,
                          D, mode=mode, alpha=w.alpha, beta=w.beta)
    if w.K == 0:
        got = d_to_host(D)
        c = c_values(w.C)[:, :w.N]
        want = (np.float64(w.beta) * c).astype(np.float32)
        if out == "bf16":
            assert np.array_equal(got, synth.to_bf16(want)[:, :w.N])
        else:
            assert np.array_equal(got, want)
        return
    check_full(w, D)


def _block_case_device(w):
    A, B = to_device(w.A)[:, :w.K], to_device(w.B)[:, :w.K]
    return A, B, to_device(w.a_scale), to_device(w.b_scale)


def test_block_scaled_concurrent_streams_independent():
    """Block-scaled skinny calls past the cluster-join sizes (more N tiles
    than SMs: whole tiles per CTA) on two streams with no ordering between
    them, enqueued back to back so their kernels can overlap: each matches
    the oracle.  The regular entry point keeps no state on the device, so
    nothing is shared between the calls."""
    import tensor_core_dense_gb300 as tcg
    cases = [fp8_case(32, 20000, 1024, seed=71, mode="block", out="f32", outliers=0.01),
             fp8_case(16, 28672, 2048, seed=72, mode="block", out="f32", outliers=0.01)]
    dev = [_block_case_device(w) for w in cases]
    Ds = [torch.full((w.M, w.N), float("nan"), device="cuda") for w in cases]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    torch.cuda.synchronize()
    for rep in range(3):
        for w, (A, B, sa, sb), D, st in zip(cases, dev, Ds, streams):
            tcg.gemm_fp8_e4m3(A, B, sa, sb, D, mode=tcg.SCALE_BLOCK128, stream=st)
    torch.cuda.synchronize()
    for w, D in zip(cases, Ds):
        v, b = oracle_for(w)
        check_f32("fp8", d_to_host(D), v, b, what=f"stream {w.M}x{w.N}x{w.K}")
    assert tcg.last_device_status() == tcg.OK


def test_block_scaled_whole_tiles_in_a_graph():
    """The same whole-tile form captured in a CUDA graph and replayed twice:
    the call does not allocate (an allocation would break the capture), the
    replays leave the device's free memory unchanged, and each replay
    matches the oracle."""
    import tensor_core_dense_gb300 as tcg
    w = fp8_case(32, 20000, 1024, seed=73, mode="block", out="bf16", outliers=0.01)
    A, B, sa, sb = _block_case_device(w)
    D = torch.empty((w.M, w.N), dtype=torch.bfloat16, device="cuda")
    tcg.gemm_fp8_e4m3(A, B, sa, sb, D, mode=tcg.SCALE_BLOCK128)  # kernel loaded
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        tcg.gemm_fp8_e4m3(A, B, sa, sb, D, mode=tcg.SCALE_BLOCK128, stream=side)
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    v, b = oracle_for(w)
    for _ in range(2):
        D.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        check_bf16("fp8", d_to_host(D), v, b, what="graph replay")
    assert torch.cuda.mem_get_info()[0] == free0
    assert tcg.last_device_status() == tcg.OK


def test_fp8_block_pair_output_beyond_2_31_elements():
    """Block-scaled FP8 on the pair-tile kernel with a 65,600 x 32,768 output
    (2.15e9 elements, 4.3 GB of BF16) and a ragged last tile row: output and
    scale offsets past 2^31, checked on the corner tiles."""
    M, N, K = 65600, 32768, 256
    w = fp8_case(M, N, K, seed=63, mode="block", out="bf16", outliers=0.01)
    D = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    run(w, D=D)
    torch.cuda.synchronize()
    tiles = [(0, 0, 128, 128), (M - 128, N - 128, 128, 128), (M - 64, 0, 64, 128),
             (0, N - 128, 128, 128), (40000, 20000, 128, 128)]
    vs, bs = oracle_for(w, tiles=tiles)
    for (i0, j0, mi, nj), v, b in zip(tiles, vs, bs):
        got = D[i0:i0 + mi, j0:j0 + nj].contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
        check_bf16("fp8", got, v, b, what=f"huge block {i0},{j0}")
    del D
    torch.cuda.empty_cache()


def test_fp8_block_skinny_a_million_columns():
    """N = 1,000,000 (7,813 N tiles, more than the SMs: contiguous ranges of
    whole tiles per CTA), ragged last tile."""
    M, N, K = 16, 1_000_000, 256
    w = fp8_case(M, N, K, seed=62, mode="block", out="bf16", outliers=0.01)
    D = run(w)
    torch.cuda.synchronize()
    tiles = [(0, 0, M, 128), (0, N - 64, M, 64), (0, 500_032, M, 128)]
    vs, bs = oracle_for(w, tiles=tiles)
    for (i0, j0, mi, nj), v, b in zip(tiles, vs, bs):
        got = D[:, j0:j0 + nj].contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
        check_bf16("fp8", got, v, b, what=f"1M columns {j0}")
