"""Pins for the CPU oracle (runs without a GPU).

Each test ties the oracle to something other than itself: facts the pages
print (tests/golden/), library implementations of the same number formats
(torch's bfloat16 and float8_e4m3fn conversions), closed forms, and exact
brute force with Python rationals on tiny shapes.
"""

import math
import os
import random
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


# ----------------------------------------------------------------- E4M3 codec

def test_e4m3_facts_from_the_pages():
    facts = {r[0]: r[1] for r in _golden("e4m3_format.txt")}
    codes = np.arange(256, dtype=np.uint8)
    vals = oracle.e4m3_decode(codes)
    finite = vals[np.isfinite(vals)]
    assert finite.max() == float(facts["e4m3_max_normal"]) == 448.0
    assert -finite.min() == 448.0
    assert not np.isinf(vals).any()                     # no infinities
    assert np.isnan(vals).sum() == 2                     # only S.1111.111
    assert np.isnan(vals[0x7F]) and np.isnan(vals[0xFF])
    assert vals[0x7E] == 448.0
    # 1 + 4 + 3 bits: 2^4 binades of 2^3 mantissas per sign
    assert int(facts["e4m3_exponent_bits"]) + int(facts["e4m3_mantissa_bits"]) + 1 == 8


def test_e5m2_facts_from_the_pages():
    facts = {r[0]: r[1] for r in _golden("e4m3_format.txt")}
    codes = np.arange(256, dtype=np.uint8)
    vals = oracle.e5m2_decode(codes)
    finite = vals[np.isfinite(vals)]
    assert finite.max() == float(facts["e5m2_max_normal"]) == 57344.0 == -finite.min()
    # IEEE specials kept: infinities at S.11111.00, NaN at S.11111.{01,10,11}
    assert int(facts["e5m2_has_infinity"]) == 1
    assert vals[0x7C] == np.inf and vals[0xFC] == -np.inf
    assert np.isnan(vals).sum() == 6 and all(np.isnan(vals[c]) for c in (0x7D, 0x7E, 0x7F))
    assert int(facts["e5m2_exponent_bits"]) + int(facts["e5m2_mantissa_bits"]) + 1 == 8
    # bias 15: 1.0 is 0.01111.00, the smallest subnormal 2^-16
    assert vals[0x3C] == 1.0 and vals[0x01] == 2.0 ** -16 and vals[0x04] == 2.0 ** -14
    assert (np.diff(vals[:0x7C]) > 0).all()


def test_e5m2_decode_matches_torch_float8_e5m2_for_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e5m2).to(torch.float64).numpy()
    got = oracle.e5m2_decode(codes)
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    m = ~np.isnan(ref)
    assert np.array_equal(ref[m], got[m]) and np.array_equal(np.signbit(ref[m]), np.signbit(got[m]))


def test_e5m2_oracle_encoder_round_trip_torch_and_saturation():
    codes = np.array([c for c in range(256) if np.isfinite(oracle.e5m2_decode(
        np.array([c], np.uint8)))[0]], dtype=np.uint8)
    assert np.array_equal(oracle.e5m2_encode(oracle.e5m2_decode(codes).astype(np.float32)), codes)
    x = (np.random.default_rng(5).standard_normal(1 << 22) *
         np.exp2(np.random.default_rng(6).integers(-24, 16, 1 << 22))).astype(np.float32)
    x = x[np.abs(x) < 61440.0]
    ref = torch.from_numpy(x).to(torch.float8_e5m2).view(torch.uint8).numpy()
    assert np.array_equal(oracle.e5m2_encode(x), ref)
    big = np.array([57344.0, 61439.0, 61440.0, 1e9, np.inf], np.float32)
    assert (oracle.e5m2_encode(big) == 0x7B).all() and (oracle.e5m2_encode(-big) == 0xFB).all()
    # midpoints between neighbours round to the even code
    pos = oracle.e5m2_decode(np.arange(0, 0x7B, dtype=np.uint8))
    mids = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)
    got = oracle.e5m2_encode(mids).astype(int)
    assert ((got % 2) == 0).all() and (np.abs(got - np.arange(0, 0x7A)) <= 1).all()


def test_e5m2_generator_encoder_against_torch_and_decode():
    # the input generator's E5M2 encoder (test inputs only): round trip of every
    # finite code, nearest-even on 4M random values (torch's cast agrees inside
    # the finite range), saturation at +-57344 where torch overflows to inf
    codes = np.array([c for c in range(256) if np.isfinite(oracle.e5m2_decode(
        np.array([c], np.uint8)))[0]], dtype=np.uint8)
    assert np.array_equal(synth.to_e5m2(oracle.e5m2_decode(codes).astype(np.float32)), codes)
    x = (np.random.default_rng(3).standard_normal(1 << 22) *
         np.exp2(np.random.default_rng(4).integers(-20, 16, 1 << 22))).astype(np.float32)
    x = x[np.abs(x) < 61440.0]
    ref = torch.from_numpy(x).to(torch.float8_e5m2).view(torch.uint8).numpy()
    assert np.array_equal(synth.to_e5m2(x), ref)
    big = np.array([57344.0, 60000.0, 61440.0, 1e9, np.inf], np.float32)
    assert (synth.to_e5m2(big) == 0x7B).all() and (synth.to_e5m2(-big) == 0xFB).all()


def test_e4m3_decode_matches_torch_float8_for_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = oracle.e4m3_decode(codes)
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    m = ~np.isnan(ref)
    assert np.array_equal(ref[m], got[m])
    assert np.array_equal(np.signbit(ref[m]), np.signbit(got[m]))  # -0 kept


def test_e4m3_decode_monotone_and_subnormal_step():
    v = oracle.e4m3_decode(np.arange(0, 0x7F, dtype=np.uint8))
    assert (np.diff(v) > 0).all()
    assert v[1] == 2.0 ** -9 and v[8] == 2.0 ** -6 and v[0x38] == 1.0
    neg = oracle.e4m3_decode(np.arange(0x80, 0xFF, dtype=np.uint8))
    assert np.array_equal(neg, -v)


def test_e4m3_encode_round_trip_and_saturation():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    vals = oracle.e4m3_decode(codes).astype(np.float32)
    assert np.array_equal(oracle.e4m3_encode(vals), codes)
    sat = np.array([448.0, 449.0, 464.0, 465.0, 480.0, 1e6, np.inf], dtype=np.float32)
    assert (oracle.e4m3_encode(sat) == 0x7E).all()
    assert (oracle.e4m3_encode(-sat) == 0xFE).all()
    assert oracle.e4m3_encode(np.array([np.nan], dtype=np.float32))[0] in (0x7F, 0xFF)


def test_e4m3_encode_midpoints_round_to_even():
    pos = oracle.e4m3_decode(np.arange(0, 0x7E, dtype=np.uint8))
    mids = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)  # exact in FP32
    enc = oracle.e4m3_encode(mids)
    lo = np.arange(0, 0x7D, dtype=np.uint8)
    expect = np.where(lo % 2 == 0, lo, lo + 1).astype(np.uint8)
    assert np.array_equal(enc, expect)


def test_e4m3_encode_matches_torch_and_the_input_generator():
    rng = np.random.default_rng(0)
    # every 2^9-th FP32 pattern of magnitude below 448 plus random values
    bits = np.arange(0, 0x43E00000, 512, dtype=np.uint32)
    x = np.concatenate([bits.view(np.float32), -bits.view(np.float32),
                        rng.normal(0, 50, 200_000).astype(np.float32).clip(-448, 448)])
    got = oracle.e4m3_encode(x)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(got, ref)
    assert np.array_equal(got, synth.to_e4m3(x))


# ----------------------------------------------------------------- BF16 codec

def test_bf16_decode_matches_torch_for_all_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16)
    ref = ref.to(torch.float64).numpy()
    got = oracle.bf16_decode(bits)
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(ref[~nan], got[~nan])


def test_bf16_encode_matches_torch_round_trip_and_ties():
    rng = np.random.default_rng(1)
    x = np.concatenate([
        rng.standard_normal(500_000).astype(np.float32),
        (rng.standard_normal(100_000) * 1e30).astype(np.float32),
        np.array([3.3895314e38, 3.4028235e38, -3.4028235e38, 1e-40, -0.0, np.inf], np.float32)])
    got = oracle.bf16_encode(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, ref)
    assert np.array_equal(got, synth.to_bf16(x))
    # round trip of every non-NaN pattern
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = oracle.bf16_decode(bits)
    keep = ~np.isnan(vals)
    assert np.array_equal(oracle.bf16_encode(vals[keep].astype(np.float32)), bits[keep])
    # ties: 1 + 2^-8 sits halfway between 1 and 1 + 2^-7 -> even (1.0)
    ties = np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8], dtype=np.float32)
    assert list(oracle.bf16_decode(oracle.bf16_encode(ties))) == [1.0, 1 + 2 ** -6]


# -------------------------------------------------------------- GEMM, exact

def _exact_gemm(M, N, K, a, b, alpha=1, beta=0, c=None, sa=None, sb=None, block=False):
    """Brute force with rationals: a[i][k], b[j][k] are Fractions (decoded)."""
    KB = (K + 127) // 128
    out = [[Fraction(0)] * N for _ in range(M)]
    for i in range(M):
        for j in range(N):
            s = Fraction(0)
            for k in range(K):
                p = a[i][k] * b[j][k]
                if block:
                    p *= Fraction(float(sa[(k // 128) * M + i])) * Fraction(
                        float(sb[(j // 128) * KB + k // 128]))
                elif sa is not None:
                    p *= Fraction(float(sa[0])) * Fraction(float(sb[0]))
                s += p
            v = Fraction(alpha) * s
            if beta != 0:
                v += Fraction(beta) * c[i][j]
            out[i][j] = v
    return out


def _frac_rows(vals, rows, cols, ld):
    return [[Fraction(float(vals[r * ld + c])) for c in range(cols)] for r in range(rows)]


def test_m16n8k16_worked_example_all_128_outputs_exact():
    facts = {r[0]: r[1:] for r in _golden("mma_m16n8k16_example.txt")}
    m, n, k = int(facts["m"][0]), int(facts["n"][0]), int(facts["k"][0])
    assert 2 * m * n * k == int(facts["flops"][0])
    rng = np.random.default_rng(16)
    ai = rng.integers(-8, 9, size=(m, k))
    bi = rng.integers(-8, 9, size=(k, n))           # K x N as on the page
    A = synth.to_bf16(ai.astype(np.float32))
    Bt = synth.to_bf16(bi.T.copy().astype(np.float32))  # stored N x K
    v, bound = oracle.gemm(m, n, k, A, k, Bt, k)
    ref = ai @ bi
    assert v.shape == (16, 8) and ref.size == int(facts["outputs"][0])
    assert np.array_equal(v, ref.astype(np.float64))
    assert np.array_equal(bound, (np.abs(ai)[:, :, None] * np.abs(bi)[None]).sum(1))


def test_fragment_lane_facts_agree_between_the_two_pages():
    facts = _golden("mma_m16n8k16_example.txt")
    for r in facts:
        if r[0] == "lane_of":
            row, col, lane = map(int, r[1:])
            assert 4 * (row % 8) + col // 2 == lane
        if r[0] == "lane_holds":
            lane = int(r[1])
            held = {tuple(map(int, x.split(","))) for x in r[2:]}
            assert held == {(row, col) for row in range(16) for col in range(8)
                            if 4 * (row % 8) + col // 2 == lane}


@pytest.mark.parametrize("seed", range(6))
def test_bf16_brute_force_tiny_shapes(seed):
    rng = random.Random(seed)
    M, N, K = rng.randint(1, 9), rng.randint(1, 9), rng.randint(1, 20)
    lda, ldb, ldc = K + rng.randint(0, 3), K + rng.randint(0, 3), N + rng.randint(0, 2)
    A = synth.bf16(seed, 1, M, K, ld=lda, dist="uniform", p0=-1, p1=1).ravel()
    B = synth.bf16(seed, 2, N, K, ld=ldb, dist="uniform", p0=-1, p1=1).ravel()
    C = synth.values_f32(seed, 3, M, ldc).ravel()
    alpha, beta = 0.75, -1.5
    v, bound = oracle.gemm(M, N, K, A, lda, B, ldb, C=C, ldc=ldc, c_type=oracle.C_F32,
                           alpha=alpha, beta=beta)
    a = _frac_rows(oracle.bf16_decode(A), M, K, lda)
    b = _frac_rows(oracle.bf16_decode(B), N, K, ldb)
    c = _frac_rows(C.astype(np.float64), M, N, ldc)
    ex = _exact_gemm(M, N, K, a, b, alpha, beta, c)
    for i in range(M):
        for j in range(N):
            bnd = sum(abs(a[i][k] * b[j][k]) for k in range(K)) * Fraction(alpha)
            assert abs(Fraction(v[i, j]) - ex[i][j]) <= Fraction(K + 2, 2 ** 52) * (
                bnd + abs(c[i][j]) * 2)
            assert Fraction(bound[i, j]) == bnd  # exact: few 16-bit products


def test_fp8_block_scale_indexing_exact():
    """Block mode with power-of-two scales: every index error changes bits."""
    M, N, K = 5, 260, 300
    KB, NB = (K + 127) // 128, (N + 127) // 128
    rng = np.random.default_rng(7)
    qa = rng.integers(0, 256, size=(M, K)).astype(np.uint8)
    qb = rng.integers(0, 256, size=(N, K)).astype(np.uint8)
    qa[(qa & 0x7F) >= 0x78] = 0x38  # avoid NaN codes and huge values
    qb[(qb & 0x7F) >= 0x78] = 0x40
    sa = np.array([2.0 ** ((i % 7) - 3 + (kb % 5)) for kb in range(KB) for i in range(M)],
                  dtype=np.float32)
    sb = np.array([2.0 ** ((nb + kb) % 4) for nb in range(NB) for kb in range(KB)],
                  dtype=np.float32)
    v, _ = oracle.gemm(M, N, K, qa, K, qb, K, in_type=oracle.IN_E4M3,
                       scale_mode=oracle.SCALE_BLOCK128, a_scale=sa, b_scale=sb)
    a = _frac_rows(oracle.e4m3_decode(qa.ravel()), M, K, K)
    b = _frac_rows(oracle.e4m3_decode(qb.ravel()), N, K, K)
    ex = _exact_gemm(M, N, K, a, b, sa=sa, sb=sb, block=True)
    for i in range(M):
        for j in range(N):
            assert Fraction(v[i, j]) == ex[i][j], (i, j)


def test_fp8_tensor_scale_exact():
    M, N, K = 4, 6, 64
    rng = np.random.default_rng(8)
    qa = (rng.integers(0, 0x77, size=(M, K)).astype(np.uint8)
          | (rng.integers(0, 2, (M, K)) << 7).astype(np.uint8))
    qb = rng.integers(0, 0x77, size=(N, K)).astype(np.uint8)
    sa, sb = np.array([2.0 ** -3], np.float32), np.array([2.0 ** 5], np.float32)
    v, _ = oracle.gemm(M, N, K, qa, K, qb, K, in_type=oracle.IN_E4M3,
                       scale_mode=oracle.SCALE_TENSOR, a_scale=sa, b_scale=sb)
    a = _frac_rows(oracle.e4m3_decode(qa.ravel()), M, K, K)
    b = _frac_rows(oracle.e4m3_decode(qb.ravel()), N, K, K)
    ex = _exact_gemm(M, N, K, a, b, sa=sa, sb=sb)
    assert all(Fraction(v[i, j]) == ex[i][j] for i in range(M) for j in range(N))


@pytest.mark.parametrize("a_fp8,b_fp8", [(1, 1), (0, 1), (1, 0)])
@pytest.mark.parametrize("mode", ["tensor", "block"])
def test_e5m2_operands_exact_rational(a_fp8, b_fp8, mode):
    # E5M2 (and mixed E4M3 x E5M2) operands against exact rational sums:
    # within FP64 rounding of the block sums (E5M2's wider exponent range can
    # take a 128-term sum past 53 bits), scales applied per block
    M, N, K = 3, 140, 260
    KB, NB = (K + 127) // 128, (N + 127) // 128
    rng = np.random.default_rng(10 + 3 * a_fp8 + b_fp8)

    def codes(fmt, rows):
        q = rng.integers(0, 256, size=(rows, K)).astype(np.uint8)
        if fmt == 1:
            q[(q & 0x7C) == 0x7C] = 0x3C   # no inf/NaN codes
        else:
            q[(q & 0x7F) == 0x7F] = 0x38
        return q
    qa, qb = codes(a_fp8, M), codes(b_fp8, N)
    dec = {0: oracle.e4m3_decode, 1: oracle.e5m2_decode}
    if mode == "tensor":
        sa, sb, sm = np.array([2.0 ** -7], np.float32), np.array([3.0], np.float32), \
            oracle.SCALE_TENSOR
    else:
        sa = np.exp2(rng.integers(-4, 4, KB * M)).astype(np.float32)
        sb = (np.exp2(rng.integers(-4, 4, NB * KB)) * 1.5).astype(np.float32)
        sm = oracle.SCALE_BLOCK128
    v, bound = oracle.gemm(M, N, K, qa, K, qb, K, in_type=oracle.IN_E4M3, scale_mode=sm,
                           a_scale=sa, b_scale=sb, a_fp8=a_fp8, b_fp8=b_fp8)
    a = _frac_rows(dec[a_fp8](qa.ravel()), M, K, K)
    b = _frac_rows(dec[b_fp8](qb.ravel()), N, K, K)
    ex = _exact_gemm(M, N, K, a, b, sa=sa, sb=sb, block=(mode == "block"))
    for i in range(M):
        for j in range(N):
            assert abs(Fraction(v[i, j]) - ex[i][j]) <= Fraction(K + 2, 2 ** 52) * Fraction(
                bound[i, j]), (i, j)
    # and the format matters: decoding as E4M3 gives another result
    v2, _ = oracle.gemm(M, N, K, qa, K, qb, K, in_type=oracle.IN_E4M3, scale_mode=sm,
                        a_scale=sa, b_scale=sb)
    assert not np.array_equal(v, v2)


# ------------------------------------------------------------ closed forms

def test_identity_gives_b_transposed_exactly():
    n, N = 48, 37
    A = synth.to_bf16(np.eye(n, dtype=np.float32))
    B = synth.bf16(3, 2, N, n)                     # N x K
    v, _ = oracle.gemm(n, N, n, A, n, B, n)
    assert np.array_equal(v, oracle.bf16_decode(B).reshape(N, n).T)


@pytest.mark.parametrize("K", [1, 7, 128, 1000, 8192])
def test_all_ones_equals_k(K):
    M, N = 3, 5
    ones = synth.to_bf16(np.ones((max(M, N), K), np.float32))
    v, bound = oracle.gemm(M, N, K, ones[:M], K, ones[:N], K)
    assert (v == K).all() and (bound == K).all()
    q = np.full((max(M, N), K), 0x38, np.uint8)    # E4M3 1.0
    sa, sb = np.array([2.0 ** 3], np.float32), np.array([2.0 ** -5], np.float32)
    v8, _ = oracle.gemm(M, N, K, q[:M], K, q[:N], K, in_type=oracle.IN_E4M3,
                        scale_mode=oracle.SCALE_TENSOR, a_scale=sa, b_scale=sb)
    assert (v8 == K * 2.0 ** -2).all()


def test_alpha_beta_closed_form_and_k_zero():
    M, N, K = 4, 6, 32
    ones = synth.to_bf16(np.ones((8, K), np.float32))
    cvals = np.arange(M * N, dtype=np.float32).reshape(M, N) - 7
    Cb = synth.to_bf16(cvals)
    v, _ = oracle.gemm(M, N, K, ones, K, ones, K, C=Cb, ldc=N, c_type=oracle.C_BF16,
                       alpha=0.5, beta=-2.0)
    assert np.array_equal(v, 0.5 * K - 2.0 * cvals)
    v0, b0 = oracle.gemm(M, N, 0, ones, K, ones, K, C=Cb, ldc=N, c_type=oracle.C_BF16,
                         alpha=3.0, beta=1.0)
    assert np.array_equal(v0, cvals) and (b0 == 0).all()


def test_beta_zero_ignores_c_even_nan():
    M, N, K = 2, 3, 4
    ones = synth.to_bf16(np.ones((4, K), np.float32))
    C = np.full(M * N, np.nan, np.float32)
    v, _ = oracle.gemm(M, N, K, ones, K, ones, K, C=C, ldc=N, beta=0.0)
    assert (v == K).all()


def test_tiles_match_whole_output_and_thread_count():
    M, N, K = 70, 90, 50
    A = synth.bf16(11, 1, M, K)
    B = synth.bf16(11, 2, N, K)
    full, fb = oracle.gemm(M, N, K, A, K, B, K, nthreads=1)
    tiles = [(0, 0, 16, 16), (64, 80, 6, 10), (5, 7, 1, 1), (10, 0, 60, 90)]
    vs, bs = oracle.gemm(M, N, K, A, K, B, K, tiles=tiles, nthreads=3)
    for (i0, j0, mi, nj), v, b in zip(tiles, vs, bs):
        assert np.array_equal(v, full[i0:i0 + mi, j0:j0 + nj])
        assert np.array_equal(b, fb[i0:i0 + mi, j0:j0 + nj])


def test_output_cast_is_nearest_even_of_fp32():
    # the value goes through FP32 first (the kernel's accumulator type): a
    # difference below FP32's precision is lost before the BF16 rounding
    v = np.array([1.0, 1 + 2 ** -8, 1 + 2 ** -8 + 2 ** -20, 1 + 2 ** -8 + 2 ** -30,
                  -3.0e38 * 10, 0.0], np.float64)
    got = oracle.bf16_decode(oracle.cast_bf16(v))
    assert got[0] == 1.0 and got[1] == 1.0 and got[2] == 1.0 + 2 ** -7 and got[3] == 1.0
    assert np.isinf(got[4]) and got[4] < 0 and got[5] == 0.0


def test_flop_formula_matches_the_pages():
    for M, N, K, f in _golden("flop_counts.txt"):
        flops = 2 * int(M) * int(N) * int(K)
        if "e9" in f:
            assert round(flops / 1e9, 1) == float(f) / 1e9
        else:
            assert flops == int(f)


def test_bf16_error_bound_sanity_against_float32_gemm():
    """An FP32 GEMM of the same inputs sits inside the BF16 tolerance of the
    oracle, and a one-ulp perturbation of a large entry is caught by it."""
    M, N, K = 64, 64, 512
    A = synth.bf16(2, 1, M, K)
    B = synth.bf16(2, 2, N, K)
    v, bound = oracle.gemm(M, N, K, A, K, B, K)
    af = oracle.bf16_decode(A).reshape(M, K).astype(np.float32)
    bf = oracle.bf16_decode(B).reshape(N, K).astype(np.float32)
    d32 = (torch.from_numpy(af) @ torch.from_numpy(bf).T).double().numpy()
    tol = 2.0 ** -14 * bound + 1e-6
    assert (np.abs(d32 - v) <= tol).all()
    bad = d32.copy()
    i, j = np.unravel_index(np.argmax(np.abs(v)), v.shape)
    bad[i, j] = v[i, j] + 2 * tol[i, j]
    assert not (np.abs(bad - v) <= tol).all()
    assert math.isfinite(float(v.sum()))


# ------------------------------------------------------------------ quantiser
#
# The FP8 recipe ("Tensor cores and low precision", scaling paragraph): scale
# so the largest magnitude sits at 448, cast, remove the scale after the
# product; scales per tensor, per row (1 x 128) or per block (128 x 128)
# ("Tensor Cores", "Precision: FP16, BF16, TF32, FP8").

Q_MODES = (oracle.Q_TENSOR, oracle.Q_ROW128, oracle.Q_BLOCK128)
# per format: decoder, largest normal (the quantiser's target), its code,
# torch's dtype, half a step relative to |x| for normals, half the subnormal step
FMT = {oracle.FP8_E4M3: (oracle.e4m3_decode, 448.0, 0x7E, "float8_e4m3fn", 2.0 ** -4, 2.0 ** -10),
       oracle.FP8_E5M2: (oracle.e5m2_decode, 57344.0, 0x7B, "float8_e5m2", 2.0 ** -3, 2.0 ** -17)}
Q_SHAPES = [(1, 1), (3, 130), (128, 128), (130, 257), (257, 384), (64, 1000)]


def _block_ids(rows, cols, mode):
    """Scale index of every element, from the layouts the GEMM reads."""
    r = np.arange(rows)[:, None]
    c = np.arange(cols)[None, :]
    KB = (cols + 127) // 128
    if mode == oracle.Q_TENSOR:
        return np.zeros((rows, cols), dtype=np.int64)
    if mode == oracle.Q_ROW128:
        return (c // 128) * rows + r
    return (r // 128) * KB + (c // 128)


def _nblocks(rows, cols, mode):
    KB, RB = (cols + 127) // 128, (rows + 127) // 128
    return {oracle.Q_TENSOR: 1, oracle.Q_ROW128: rows * KB, oracle.Q_BLOCK128: RB * KB}[mode]


@pytest.mark.parametrize("fmt", list(FMT))
@pytest.mark.parametrize("mode", Q_MODES)
@pytest.mark.parametrize("rows,cols", Q_SHAPES)
@pytest.mark.parametrize("bf16_in", [False, True])
def test_quant_power_of_two_blocks_reproduce_codes_and_scales(mode, rows, cols, bf16_in, fmt):
    # X = decode(code) * 2^p_block with the format's largest magnitude (448 or
    # 57344) in every block: the scale is exactly 2^p_block and every code
    # comes back unchanged.  A wrong block geometry, scale index, missing |.|
    # or misplaced division changes bits.
    dec, top, topcode, _, _, _ = FMT[fmt]
    rng = np.random.default_rng(rows * 1000 + cols + 7 * mode + 97 * fmt)
    codes = rng.integers(0, 256, size=(rows, cols)).astype(np.uint8)
    if fmt == oracle.FP8_E4M3:
        codes[(codes & 0x7F) == 0x7F] = 0x3A
    else:
        codes[(codes & 0x7C) == 0x7C] = 0x3A    # no E5M2 inf / NaN codes
    ids = _block_ids(rows, cols, mode)
    nb = _nblocks(rows, cols, mode)
    p = rng.integers(-20, 21, size=nb)
    flat_ids = ids.ravel()
    for b in range(nb):  # one +-448 per block, at a random member
        members = np.flatnonzero(flat_ids == b)
        codes.flat[rng.choice(members)] = rng.choice([topcode, topcode | 0x80])
    x = (dec(codes) * np.exp2(p[ids])).astype(np.float32)
    if bf16_in:  # E4M3 values times powers of two are exact in BF16
        xin = oracle.bf16_encode(x)
        assert np.array_equal(oracle.bf16_decode(xin).astype(np.float32), x)
    else:
        xin = x
    q, s = oracle.quantize_fp8(xin, mode, fmt)
    assert np.array_equal(s, np.exp2(p).astype(np.float32))
    assert np.array_equal(q, codes)


@pytest.mark.parametrize("fmt", list(FMT))
@pytest.mark.parametrize("mode", Q_MODES)
def test_quant_block_maximum_lands_on_448_and_zero_block_scale_one(mode, fmt):
    dec, top, _, _, _, _ = FMT[fmt]
    rows, cols = 300, 520
    x = synth.values_f32(11, 1, rows, cols, out_prob=0.01, out_factor=50.0)
    x[:128, :128] = 0.0          # an all-zero 128 x 128 block (and 1 x 128 blocks)
    if mode == oracle.Q_TENSOR:
        x[:, :] = x * 3.0
    q, s = oracle.quantize_fp8(x, mode, fmt)
    ids = _block_ids(rows, cols, mode)
    dq = np.abs(dec(q))
    for b in range(_nblocks(rows, cols, mode)):
        m = ids == b
        amax = np.abs(x[m]).max()
        if amax == 0.0:
            assert s[b] == 1.0 and (q[m] == 0).all()
        else:
            assert dq[m].max() == top                        # the largest sits at the top
            assert abs(float(s[b]) * top / float(amax) - 1.0) < 2.0 ** -23


@pytest.mark.parametrize("fmt", list(FMT))
@pytest.mark.parametrize("mode", Q_MODES)
def test_quant_reconstruction_within_half_an_e4m3_step(mode, fmt):
    # |decode(q) * s - x| <= half a quantum: 2^-4 (E4M3) or 2^-3 (E5M2) of |x|
    # for normal codes, half the subnormal step (times s) below the smallest
    # normal; plus the FP32 division's rounding.
    dec, _, _, _, rel, sub = FMT[fmt]
    rows, cols = 256, 384
    x = synth.values_f32(12, 1, rows, cols, out_prob=0.01, out_factor=50.0).astype(np.float32)
    q, s = oracle.quantize_fp8(x, mode, fmt)
    sel = s[_block_ids(rows, cols, mode)].astype(np.float64)
    err = np.abs(dec(q) * sel - x.astype(np.float64))
    bound = rel * np.abs(x) * (1 + 2.0 ** -20) + sub * sel
    assert (err <= bound).all()
    # and it is not trivially loose: most elements sit well inside it
    assert np.median(err / bound) < 0.6


@pytest.mark.parametrize("fmt", list(FMT))
@pytest.mark.parametrize("mode", Q_MODES)
def test_quant_matches_torch_division_and_float8_cast(mode, fmt):
    # Given the scales, each code is torch's FP32 division followed by torch's
    # float8_e4m3fn / float8_e5m2 conversion; the scales are amax / top of
    # numpy's max.
    _, top, _, tdt, _, _ = FMT[fmt]
    rows, cols = 200, 700
    x = synth.values_f32(13, 1, rows, cols, out_prob=0.01, out_factor=50.0)
    q, s = oracle.quantize_fp8(x, mode, fmt)
    ids = _block_ids(rows, cols, mode)
    amax = np.zeros(_nblocks(rows, cols, mode), dtype=np.float32)
    np.maximum.at(amax, ids.ravel(), np.abs(x).ravel())
    assert np.array_equal(s, (torch.from_numpy(amax) / top).numpy())
    y = torch.from_numpy(x) / torch.from_numpy(s[ids])
    ref = y.to(getattr(torch, tdt)).view(torch.uint8).numpy()
    assert np.array_equal(q, ref)


@pytest.mark.parametrize("mode,fn", [(oracle.Q_TENSOR, synth.e4m3_tensor),
                                     (oracle.Q_ROW128, synth.e4m3_rowblock),
                                     (oracle.Q_BLOCK128, synth.e4m3_block128)])
def test_quant_matches_the_input_generators_quantiser(mode, fn):
    x = synth.values_f32(14, 2, 384, 1152, out_prob=0.01, out_factor=50.0)
    q, s = oracle.quantize_e4m3(x, mode, ldq=1168)
    q2, s2 = fn(x, ld=1168)
    assert np.array_equal(s, s2) and np.array_equal(q, q2)


def test_quant_special_values():
    # NaN entries are skipped by amax and stored as the canonical NaN 0x7F;
    # -0 keeps its sign; an infinite amax gives scale inf, finite values -> +-0
    # and inf/inf -> NaN.
    x = np.array([[1.0, np.nan, -0.0, -448.0 * 4, 2.0 ** -40]], dtype=np.float32)
    q, s = oracle.quantize_e4m3(x, oracle.Q_TENSOR)
    assert s[0] == 4.0
    assert q.tolist() == [[oracle.e4m3_encode(np.float32([0.25]))[0], 0x7F, 0x80, 0xFE, 0x00]]
    xi = np.array([[1.0, -2.0, np.inf, -np.inf]], dtype=np.float32)
    q, s = oracle.quantize_e4m3(xi, oracle.Q_TENSOR)
    assert np.isinf(s[0]) and q.tolist() == [[0x00, 0x80, 0x7F, 0x7F]]
    # amax so small that amax / 448 underflows to zero: scale 1, codes 0
    xt = np.array([[2.0 ** -149, -(2.0 ** -149)]], dtype=np.float32)
    q, s = oracle.quantize_e4m3(xt, oracle.Q_TENSOR)
    assert s[0] == 1.0 and q.tolist() == [[0x00, 0x80]]
    # empty inputs
    q, s = oracle.quantize_e4m3(np.zeros((0, 5), np.float32), oracle.Q_TENSOR)
    assert s.tolist() == [1.0] and q.shape == (0, 5)
    q, s = oracle.quantize_e4m3(np.zeros((4, 0), np.float32), oracle.Q_ROW128)
    assert s.size == 0


@pytest.mark.parametrize("mode", Q_MODES)
def test_quant_bf16_input_equals_fp32_input_of_the_same_values(mode):
    bits = synth.bf16(15, 1, 130, 300, p1=3.0)
    q1, s1 = oracle.quantize_e4m3(bits, mode)
    q2, s2 = oracle.quantize_e4m3(oracle.bf16_decode(bits).astype(np.float32), mode)
    assert np.array_equal(q1, q2) and np.array_equal(s1, s2)
