"""How many significant bits the tcgen05 accumulator keeps, measured through
the library.

The probe of "Tensor Cores: Matrix Instructions, Swizzling and FP8, Measured"
(Step 5) sets the accumulator to 2^e and adds a product 1 x 1; FP32 keeps
2^e + 1 exactly up to e = 23.  On Ada the FP8 instruction lost the 1 from
e = 14 on (about 14 significant bits), which is why FP8 GEMMs promote partial
sums to FP32 every so often.  Here the 2^e comes from products placed at the
start of K and the 1 x 1 product either in the same tcgen05.mma instruction,
in the next instruction of the same stage, or in the next K stage (another
shared-memory buffer), for BF16 (kind::f16) and E4M3 (kind::f8f6f4), on both
dense kernels.  The FP32 output of D[0, 0] is compared with 2^e + 1.
"""

import numpy as np
import pytest

import synth
import synth.workloads as W
from helpers import d_to_host, run

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _probe(kind, e, where, M, N):
    """D[0, 0] for accumulator 2^e plus one product 1 at K offset `where`."""
    if kind == "bf16":
        K = 128
        a = np.zeros((M, K), np.float32)
        b = np.zeros((N, K), np.float32)
        a[0, 0], b[0, 0] = 2.0 ** (e // 2), 2.0 ** (e - e // 2)
        a[0, where], b[0, where] = 1.0, 1.0
        w = W.Workload("probe", M, N, K, "bf16", "f32")
        w.A, w.B = synth.to_bf16(a), synth.to_bf16(b)
    else:
        K = 256
        a = np.zeros((M, K), np.float32)
        b = np.zeros((N, K), np.float32)
        if e <= 16:
            ea = min(e, 8)
            a[0, 0], b[0, 0] = 2.0 ** ea, 2.0 ** (e - ea)
        else:                                  # 2^(e-16) products of 2^8 x 2^8
            n = 2 ** (e - 16)
            a[0, :n], b[0, :n] = 256.0, 256.0
        a[0, where], b[0, where] = 1.0, 1.0
        w = W.Workload("probe", M, N, K, "fp8_tensor", "f32")
        w.A, w.B = synth.to_e4m3(a), synth.to_e4m3(b)
        w.a_scale = np.ones(1, np.float32)
        w.b_scale = np.ones(1, np.float32)
    return float(d_to_host(run(w))[0, 0])


def _largest_exact(kind, where, es, M, N):
    best = None
    for e in es:
        if _probe(kind, e, where, M, N) == 2.0 ** e + 1.0:
            best = e
        else:
            break
    return best


# (kind, K offset of the 1 x 1 product, what that offset means)
CASES = [("bf16", 1, "same instruction"), ("bf16", 16, "next instruction"),
         ("bf16", 64, "next stage"), ("fp8", 31, "same instruction"),
         ("fp8", 32, "next instruction"), ("fp8", 128, "next stage")]


@pytest.mark.parametrize("kernel,M,N", [("1cta", 128, 128), ("2cta", 256, 256)])
@pytest.mark.parametrize("kind,where,label", CASES)
def test_accumulator_bits(monkeypatch, capsys, kernel, M, N, kind, where, label):
    monkeypatch.setenv("TCG_KERNEL", kernel)
    # FP8: 2^e for e > 16 is 2^(e-16) products of 256 x 256 before the 1 x 1
    # product, so the placement bounds e (16 products fit before K offset 31,
    # 32 before the next instruction, 128 before the next stage)
    top = 23 if kind == "bf16" else {31: 20, 32: 21, 128: 23}[where]
    best = _largest_exact(kind, where, range(8, top + 1), M, N)
    with capsys.disabled():
        print(f"\naccumulator probe {kernel} {kind} (+1 in the {label}): largest e with "
              f"2^e + 1 exact = {best}")
    if kind == "bf16":
        assert best == 23      # a full FP32 accumulator
    else:
        # GB300 loses nothing up to the largest e each placement can express
        # (the pages found about 14 bits on Ada).  The per-tensor FP8 path
        # accumulates all of K in Tensor Memory without promotion because of
        # this, so anything short of the top of the range is a failure.
        assert best == top
