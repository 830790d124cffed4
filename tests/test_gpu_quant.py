"""GPU parity of the FP8 quantiser (quantize_e4m3, through the C ABI) against
the oracle's quantiser: codes and scales must be bit-identical (the scale is
an FP32 division of the block maximum by 448 and each code an FP32 division
rounded to E4M3, so both sides take every decision in the same precision).

Covered: the three granularities x FP32/BF16 input on small, ragged
(columns not a multiple of 4 or 128, rows not a multiple of 16 or 128),
padded-pitch and full-size shapes; special values (NaN, +-0, +-Inf, FP32
subnormals, all-zero blocks, E4M3 rounding ties); bytes and scales outside
the output left untouched; run-to-run determinism of the per-tensor path.
"""

from __future__ import annotations

import numpy as np
import pytest

import oracle
import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

MODES = {"tensor": oracle.Q_TENSOR, "row128": oracle.Q_ROW128, "block128": oracle.Q_BLOCK128}


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


def gpu_quant(x, mode, *, ldx=None, ldq=None, reps=1, fmt=0):
    """Quantise x (float32 values or uint16 BF16 bits, rows x cols) on the GPU
    from a buffer with row pitch ldx into one with pitch ldq; returns (q, s,
    q_pad, s_extra): codes rows x cols, the scales, the untouched padding
    columns and the sentinel scales after the last one."""
    import tensor_core_dense_gb300 as tcg
    rows, cols = x.shape
    bf16 = x.dtype == np.uint16
    ldx = ldx or _pad(max(cols, 1), 8 if bf16 else 4)
    ldq = ldq or _pad(max(cols, 1), 16)
    host = np.zeros((rows, ldx), dtype=x.dtype)
    host[:, :cols] = x
    if bf16:
        X = torch.from_numpy(host.view(np.int16)).cuda().view(torch.bfloat16)
    else:
        X = torch.from_numpy(host).cuda()
    Q = torch.full((rows, ldq), 0xAB, dtype=torch.uint8, device="cuda")
    n = tcg.quant_scale_count(rows, cols, mode)
    S = torch.full((n + 4,), float("nan"), dtype=torch.float32, device="cuda")
    for _ in range(reps):
        if fmt == 0:
            tcg.quantize_e4m3(X[:, :cols], Q[:, :cols], S, mode=mode)
        else:
            tcg.quantize_fp8(X[:, :cols], Q[:, :cols], S, mode=mode, fmt=fmt)
    torch.cuda.synchronize()
    q = Q.cpu().numpy()
    s = S.cpu().numpy()
    return q[:, :cols], s[:n], q[:, cols:], s[n:]


def check(x, mode_name, fmt=0, **kw):
    mode = MODES[mode_name]
    q_ref, s_ref = oracle.quantize_fp8(x, mode, fmt)
    q, s, q_pad, s_extra = gpu_quant(x, mode, fmt=fmt, **kw)
    assert np.array_equal(s.view(np.uint32), s_ref.view(np.uint32)), (
        f"scales differ at {np.flatnonzero(s.view(np.uint32) != s_ref.view(np.uint32))[:8]}")
    if not np.array_equal(q, q_ref):
        i = tuple(np.argwhere(q != q_ref)[0])
        raise AssertionError(f"{int((q != q_ref).sum())} codes differ; first at {i}: "
                             f"got {q[i]:#04x} want {q_ref[i]:#04x} (x = {x[i]!r})")
    assert (q_pad == 0xAB).all(), "bytes beyond the last column were written"
    assert np.isnan(s_extra).all(), "scales beyond the last block were written"


SHAPES = [(1, 1), (3, 130), (5, 131), (17, 129), (128, 128), (130, 257), (257, 384),
          (16, 8192), (300, 1030)]


@pytest.mark.parametrize("mode", list(MODES))
@pytest.mark.parametrize("rows,cols", SHAPES)
def test_fp32_shapes(mode, rows, cols):
    x = synth.values_f32(21, 1, rows, cols, out_prob=0.01, out_factor=50.0)
    check(x, mode)


@pytest.mark.parametrize("mode", list(MODES))
@pytest.mark.parametrize("rows,cols", SHAPES)
def test_bf16_shapes(mode, rows, cols):
    x = synth.bf16(22, 1, rows, cols, p1=2.0)
    check(x, mode)


@pytest.mark.parametrize("mode", list(MODES))
def test_padded_pitches(mode):
    x = synth.values_f32(23, 1, 140, 200, out_prob=0.01, out_factor=50.0)
    check(x, mode, ldx=260, ldq=272)
    xb = synth.bf16(23, 2, 140, 200)
    check(xb, mode, ldx=264, ldq=256)


@pytest.mark.parametrize("mode", list(MODES))
def test_special_values(mode):
    rng = np.random.default_rng(5)
    x = np.zeros((256, 512), np.float32)
    x[:, :384] = synth.values_f32(24, 1, 256, 384)
    x[:128, 384:] = synth.values_f32(24, 2, 128, 128) * np.float32(1e-20)  # scale ~2^-75
    x[128:, 384:] = synth.values_f32(24, 3, 128, 128) * np.float32(1e30)   # scale ~2^90
    x[:128, :128] = 0.0                                  # an all-zero block
    x[0, 200] = np.nan
    x[130, 5] = -0.0
    x[131, 6:10] = [2.0 ** -149, -(2.0 ** -130), 2.0 ** -126, -(2.0 ** -140)]
    x[200, 300] = np.inf
    x[201, 301] = -np.inf
    x[250, 130:140] = np.nan
    # NaNs of both signs and with payloads must all come out as 0x7F
    x[251, 131:135] = np.array([0xFFC00000, 0x7F800001, 0xFF812345, 0x7FFFFFFF],
                               np.uint32).view(np.float32)
    x[140, 140:200] = -1e-30                             # rounds to -0
    x[160:170, 260:270] = rng.choice([1e-38, -3e-39, 5e-40], size=(10, 10))
    check(x.astype(np.float32), mode)


def _near_midpoint_blocks(seed, rows, cols, fmt=0):
    """Rows of 1 x 128 blocks, each with its own non-power-of-two maximum and
    127 values x whose quotients x / s lie within 3 FP32 units of a midpoint
    between neighbouring E4M3 (or E5M2) values, normal and subnormal."""
    rng = np.random.default_rng(seed)
    if fmt == 0:
        pos, top = oracle.e4m3_decode(np.arange(0, 0x7F, dtype=np.uint8)), 448.0
    else:
        pos, top = oracle.e5m2_decode(np.arange(0, 0x7C, dtype=np.uint8)), 57344.0
    mids = (pos[:-1] + pos[1:]) / 2
    x = np.zeros((rows, cols), np.float32)
    for r in range(rows):
        for kb in range(cols // 128):
            amax = np.float32(top * rng.uniform(0.5, 2.0) * 2.0 ** int(rng.integers(-40, 40)))
            sc = np.float32(amax / np.float32(top))
            vals = (rng.choice(mids, 127) * np.float64(sc)).astype(np.float32)
            vals = (vals.view(np.int32) + rng.integers(-3, 4, 127).astype(np.int32)).view(
                np.float32) * rng.choice(np.array([-1.0, 1.0], np.float32), 127)
            block = np.concatenate([[amax], vals]).astype(np.float32)
            rng.shuffle(block)
            x[r, kb * 128:(kb + 1) * 128] = block
    return x


@pytest.mark.parametrize("mode", list(MODES))
def test_division_near_e4m3_midpoints(mode):
    # Where FP32 -> E4M3 rounding is decided within an FP32 unit or two, the
    # GPU's quotient must be the correctly rounded one, as the oracle's IEEE
    # FP32 division is.
    check(_near_midpoint_blocks(31, 96, 1024), mode)


def test_rounding_ties_and_saturation_edge():
    # amax = 448 exactly, so s = 1 and every quotient is x itself: midpoints
    # between neighbouring E4M3 values (normal and subnormal) must round to
    # the even code, as the oracle's integer encoder does.
    pos = oracle.e4m3_decode(np.arange(0, 0x7F, dtype=np.uint8))
    mids = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)
    vals = np.concatenate([mids, -mids, pos.astype(np.float32), [448.0, -448.0]])
    cols = 512
    x = np.zeros((2, cols), np.float32)
    x.flat[:vals.size] = vals
    for mode in MODES:
        check(x, mode)


@pytest.mark.parametrize("mode", list(MODES))
def test_zero_and_constant_blocks(mode):
    x = np.zeros((130, 260), np.float32)
    check(x, mode)
    x[:, :] = -3.0
    check(x, mode)


def test_tensor_mode_is_deterministic_and_rewrites_its_scale():
    x = synth.values_f32(25, 1, 512, 1024, out_prob=0.01, out_factor=50.0)
    q1, s1, _, _ = gpu_quant(x, oracle.Q_TENSOR, reps=3)
    q2, s2, _, _ = gpu_quant(x, oracle.Q_TENSOR)
    assert np.array_equal(q1, q2) and np.array_equal(s1, s2)
    check(x, "tensor")


def test_empty_inputs():
    import tensor_core_dense_gb300 as tcg
    S = torch.full((2,), float("nan"), dtype=torch.float32, device="cuda")
    assert tcg.quantize_e4m3_raw(0, 64, None, 0, tcg.IN_F32, tcg.QUANT_TENSOR, None, 0,
                                 S.data_ptr(), None) == tcg.OK
    torch.cuda.synchronize()
    assert S[0].item() == 1.0 and np.isnan(S[1].item())
    for mode in (tcg.QUANT_ROW128, tcg.QUANT_BLOCK128):
        assert tcg.quantize_e4m3_raw(64, 0, None, 0, tcg.IN_F32, mode, None, 0, None,
                                     None) == tcg.OK


# Full size, in the configuration the benchmark times: the 4096 x 4096 FP8
# operands quantised per tensor, and the skinny FP8 GEMM's operands (A rows x
# 8192 in 1 x 128 blocks, the 8192 x 8192 weight in 128 x 128 blocks).
@pytest.mark.parametrize("mode,rows,cols,in_dtype", [
    ("tensor", 4096, 4096, "f32"), ("tensor", 4096, 4096, "bf16"),
    ("row128", 128, 8192, "f32"), ("row128", 4096, 4096, "bf16"),
    ("block128", 8192, 8192, "f32"), ("block128", 4096, 4096, "bf16"),
])
def test_full_size(mode, rows, cols, in_dtype):
    if in_dtype == "f32":
        x = synth.values_f32(26, 2, rows, cols, out_prob=0.01, out_factor=50.0)
    else:
        x = synth.bf16(26, 2, rows, cols)
    check(x, mode)


@pytest.mark.parametrize("mode", list(MODES))
def test_beyond_2_31_elements(mode):
    """A 40,000 x 65,664 FP32 matrix (2.6e9 elements, 10.5 GB): a seeded
    40-row slab repeated down the rows on the device; the last (partial) row
    blocks and all of their scales are checked against the oracle."""
    import tensor_core_dense_gb300 as tcg
    R, C, SLAB = 40000, 65664, 40
    slab = synth.values_f32(71, 1, SLAB, C, out_prob=0.01, out_factor=50.0)
    X = torch.from_numpy(slab).cuda().repeat(R // SLAB, 1)
    Q = torch.empty((R, C), dtype=torch.uint8, device="cuda")
    n = tcg.quant_scale_count(R, C, MODES[mode])
    S = torch.empty((n,), dtype=torch.float32, device="cuda")
    tcg.quantize_e4m3(X, Q, S, mode=MODES[mode])
    torch.cuda.synchronize()
    del X
    r0 = (R // 128) * 128                          # the last, 64-row block
    host = slab[np.arange(r0, R) % SLAB]
    KB = (C + 127) // 128
    if mode == "tensor":
        q_ref, s_ref = oracle.quantize_e4m3(slab, MODES[mode])
        q_ref = q_ref[np.arange(r0, R) % SLAB]
        s_got = S.cpu().numpy()
    else:
        q_ref, s_ref = oracle.quantize_e4m3(host, MODES[mode])
        if mode == "block128":
            s_got = S[(R // 128) * KB:].cpu().numpy()
        else:  # scale[kb * R + r] for the last rows
            s_got = S.view(KB, R)[:, r0:].contiguous().cpu().numpy().ravel()
    assert np.array_equal(s_got.view(np.uint32), s_ref.view(np.uint32))
    assert np.array_equal(Q[r0:].cpu().numpy(), q_ref)
    del Q, S
    torch.cuda.empty_cache()


# ---------------------------------------------------------------- E5M2 codes

@pytest.mark.parametrize("mode", list(MODES))
@pytest.mark.parametrize("rows,cols", [(1, 1), (5, 131), (130, 257), (16, 8192), (300, 1030)])
def test_e5m2_shapes(mode, rows, cols):
    check(synth.values_f32(81, 1, rows, cols, out_prob=0.01, out_factor=50.0), mode, fmt=1)
    check(synth.bf16(82, 1, rows, cols, p1=2.0), mode, fmt=1)


@pytest.mark.parametrize("mode", list(MODES))
def test_e5m2_division_near_midpoints_and_specials(mode):
    check(_near_midpoint_blocks(83, 64, 1024, fmt=1), mode, fmt=1)
    x = synth.values_f32(84, 1, 256, 384)
    x[:128, :128] = 0.0
    x[3, 200:204] = np.array([0x7FC00000, 0xFFC00000, 0x7F800001, 0xFF812345],
                             np.uint32).view(np.float32)
    x[130, 5] = -0.0
    x[140, 140:200] = -1e-30
    x[200, 300] = np.inf
    check(x, mode, fmt=1)


def test_e5m2_full_size_block_scaled_weight():
    check(synth.values_f32(85, 2, 8192, 8192, out_prob=0.01, out_factor=50.0), "block128", fmt=1)
