"""Pins for the oracle's microscaled FP8 mode (SCALE_MX32), no GPU.

The block-scaled MMA of "How Blackwell's Tensor Memory Actually Works"
("Quantization became an allocation problem") computes D = C + (A x SFA)(B x
SFB) with one scale factor per 32 elements along K, for the MX formats an
E8M0 byte: a bare power-of-two exponent.  What pins the oracle here:

* E8M0 decoding against torch's float8_e8m0fnu conversion for all 256 codes,
  and the facts the format has (no sign, doubling per code, 0xFF = NaN);
* the tiled scale layout: the oracle's C index function against the input
  generator's independent numpy construction, on every (row, block) of
  ragged shapes;
* exact rational brute force on random tiny shapes (E4M3 and E5M2 codes,
  random exponents per row and block, alpha, beta and C), with the scales
  taken from dense per-(row, block) arrays, not from the tiled buffer;
* closed forms: all-ones operands give sum over blocks of 32 * 2^(ea + eb).
"""

from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import synth


def test_e8m0_decode_matches_torch_for_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e8m0_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    assert np.isnan(ours[255]) and np.isnan(ref[255])
    assert np.array_equal(ours[:255], ref[:255])


def test_e8m0_facts():
    v = oracle.e8m0_decode(np.arange(255, dtype=np.uint8))
    assert (v > 0).all()                       # no sign bit, no zero
    assert np.array_equal(v[1:] / v[:-1], np.full(254, 2.0))   # one binade per code
    assert v[127] == 1.0                       # the microscaling bias, 127
    assert np.isnan(oracle.e8m0_decode(np.array([255], np.uint8))[0])


@pytest.mark.parametrize("rows,K", [(1, 32), (5, 100), (128, 128), (129, 130), (300, 700),
                                    (256, 4096)])
def test_tiled_layout_oracle_index_matches_generator(rows, K):
    KB = -(-K // 32)
    rng = np.random.default_rng(rows + K)
    exps = rng.integers(0, 255, size=(rows, KB)).astype(np.uint8)
    tiled = synth.mx_tile_sf(exps, K)
    assert tiled.size == oracle.mx_sf_bytes(rows, K)
    for r in range(rows):
        for kb in range(KB):
            assert tiled[oracle.mx_sf_offset(r, kb, K)] == exps[r, kb], (r, kb)


def _exact_mx(M, N, K, a, b, ea, eb, alpha=1, beta=0, c=None):
    out = [[Fraction(0)] * N for _ in range(M)]
    for i in range(M):
        for j in range(N):
            s = Fraction(0)
            for k in range(K):
                kb = k // 32
                s += a[i][k] * b[j][k] * Fraction(2) ** (int(ea[i, kb]) + int(eb[j, kb]) - 254)
            v = Fraction(alpha) * s
            if beta != 0:
                v += Fraction(beta) * c[i][j]
            out[i][j] = v
    return out


def _rows(vals, rows, cols, ld):
    return [[Fraction(float(vals[r * ld + k])) for k in range(cols)] for r in range(rows)]


def _codes(rng, fmt, rows, K):
    q = rng.integers(0, 256, size=(rows, K)).astype(np.uint8)
    if fmt == 1:
        q[(q & 0x7C) == 0x7C] = 0x3C   # no E5M2 inf / NaN
    else:
        q[(q & 0x7F) == 0x7F] = 0x38   # no E4M3 NaN
    return q


@pytest.mark.parametrize("seed,a_fp8,b_fp8", [(0, 0, 0), (1, 0, 0), (2, 1, 1), (3, 0, 1),
                                               (4, 1, 0), (5, 0, 0)])
def test_mx_brute_force_exact(seed, a_fp8, b_fp8):
    rng = np.random.default_rng(100 + seed)
    M, N = int(rng.integers(1, 6)), int(rng.integers(1, 7))
    K = int(rng.integers(1, 200))
    if seed == 5:
        M, N, K = 130, 3, 70    # rows past one 128-row scale tile
    KB = -(-K // 32)
    qa, qb = _codes(rng, a_fp8, M, K), _codes(rng, b_fp8, N, K)
    ea = rng.integers(110, 145, size=(M, KB)).astype(np.uint8)
    eb = rng.integers(110, 145, size=(N, KB)).astype(np.uint8)
    c = synth.values_f32(seed, 3, M, N)
    alpha, beta = 1.25, -0.5
    v, bound = oracle.gemm(M, N, K, qa, K, qb, K, in_type=oracle.IN_E4M3,
                           scale_mode=oracle.SCALE_MX32, a_sf=synth.mx_tile_sf(ea, K),
                           b_sf=synth.mx_tile_sf(eb, K), C=c, ldc=N, c_type=oracle.C_F32,
                           alpha=alpha, beta=beta, a_fp8=a_fp8, b_fp8=b_fp8)
    dec = {0: oracle.e4m3_decode, 1: oracle.e5m2_decode}
    a = _rows(dec[a_fp8](qa.ravel()), M, K, K)
    b = _rows(dec[b_fp8](qb.ravel()), N, K, K)
    cf = _rows(c.astype(np.float64).ravel(), M, N, N)
    ex = _exact_mx(M, N, K, a, b, ea, eb, alpha, beta, cf)
    for i in range(M):
        for j in range(N):
            bnd = Fraction(alpha) * sum(
                abs(a[i][k] * b[j][k]) * Fraction(2) ** (int(ea[i, k // 32]) + int(eb[j, k // 32])
                                                         - 254) for k in range(K))
            # E4M3 block sums are exact; E5M2 ones within FP64 rounding
            assert abs(Fraction(v[i, j]) - ex[i][j]) <= Fraction(K + 2, 2 ** 52) * (
                bnd + abs(Fraction(beta) * cf[i][j]) * 2), (i, j)
            assert abs(Fraction(bound[i, j]) - bnd) <= Fraction(K + 2, 2 ** 52) * bnd


def test_mx_e4m3_block_sums_are_exact():
    # E4M3 products and their 32-term sums are exact in FP64, and the scale is
    # a power of two: without alpha/beta the oracle's value is the exact one
    rng = np.random.default_rng(9)
    M, N, K = 4, 5, 160
    KB = K // 32
    qa, qb = _codes(rng, 0, M, K), _codes(rng, 0, N, K)
    ea = rng.integers(120, 135, size=(M, KB)).astype(np.uint8)
    eb = rng.integers(120, 135, size=(N, KB)).astype(np.uint8)
    v, _ = oracle.gemm(M, N, K, qa, K, qb, K, in_type=oracle.IN_E4M3,
                       scale_mode=oracle.SCALE_MX32, a_sf=synth.mx_tile_sf(ea, K),
                       b_sf=synth.mx_tile_sf(eb, K))
    ex = _exact_mx(M, N, K, _rows(oracle.e4m3_decode(qa.ravel()), M, K, K),
                   _rows(oracle.e4m3_decode(qb.ravel()), N, K, K), ea, eb)
    assert all(Fraction(v[i, j]) == ex[i][j] for i in range(M) for j in range(N))


@pytest.mark.parametrize("K", [32, 96, 100, 4096])
def test_mx_all_ones_closed_form(K):
    # E4M3 0x38 = 1.0: D = sum over blocks of (block length) * 2^(ea + eb - 254)
    M, N = 3, 4
    KB = -(-K // 32)
    A = np.full((M, K), 0x38, np.uint8)
    B = np.full((N, K), 0x38, np.uint8)
    ea = np.array([[127 + (kb % 3) - i for kb in range(KB)] for i in range(M)], np.uint8)
    eb = np.array([[127 - (kb % 2) + j for kb in range(KB)] for j in range(N)], np.uint8)
    v, bound = oracle.gemm(M, N, K, A, K, B, K, in_type=oracle.IN_E4M3,
                           scale_mode=oracle.SCALE_MX32, a_sf=synth.mx_tile_sf(ea, K),
                           b_sf=synth.mx_tile_sf(eb, K))
    for i in range(M):
        for j in range(N):
            want = sum(min(32, K - 32 * kb) * 2.0 ** ((kb % 3) - i - (kb % 2) + j)
                       for kb in range(KB))
            assert v[i, j] == want and bound[i, j] == want


def test_mx_nan_scale_propagates_and_quantiser_round_trip():
    # the 0xFF scale code is NaN and poisons exactly its rows' outputs
    M, N, K = 2, 2, 64
    A = np.full((M, K), 0x38, np.uint8)
    ea = np.full((M, 2), 127, np.uint8)
    ea[1, 1] = 255
    eb = np.full((N, 2), 127, np.uint8)
    v, _ = oracle.gemm(M, N, K, A, K, A, K, in_type=oracle.IN_E4M3,
                       scale_mode=oracle.SCALE_MX32, a_sf=synth.mx_tile_sf(ea, K),
                       b_sf=synth.mx_tile_sf(eb, K))
    assert np.array_equal(v[0], [64.0, 64.0]) and np.isnan(v[1]).all()
    # the generator's microscaling quantiser: every block's largest magnitude
    # decodes into E4M3's top binade [256, 448], and decode(q) * 2^(e-127)
    # reconstructs x within half an E4M3 step (or saturates at 448 * scale)
    x = synth.values_f32(4, 1, 8, 256, out_prob=0.01, out_factor=50.0)
    q, e = synth.mx_quant(x)
    d = oracle.e4m3_decode(q.ravel()).reshape(q.shape)
    top = np.abs(d).reshape(8, 8, 32).max(axis=2)
    assert ((top >= 256) & (top <= 448)).all()
    s = np.exp2(e.astype(np.float64) - 127).repeat(32, axis=1)
    rec = d * s
    step = np.exp2(np.floor(np.log2(np.maximum(np.abs(x) / s, 2.0 ** -6))) - 3) * s
    inside = np.abs(d) < 448
    assert (np.abs(rec - x)[inside] <= 0.5 * step[inside]).all()
    assert (np.abs(x / s)[~inside] >= 448 - 16).all()   # saturated: at or past 448
