"""The GEMM workloads, built from the seeded generator (inputs only).

Each workload is the synthetic stand-in for one of the pages' problems:

* ``bf16_256``    BF16 256^3, uniform [-1, 1), FP32 output, beta = 0 -- the
                  4,096^3 test's value recipe at a size the oracle computes
                  whole ("Tensor Cores: Matrix Instructions, Swizzling and FP8,
                  Measured", Step 2);
* ``bf16_4096``   BF16 4096^3, N(0, 1), BF16 output -- that page's headline
                  square problem;
* ``fp8_4096``    FP8 E4M3 4096^3, N(0, 1) quantised per tensor (scale
                  amax / 448), BF16 output ("Tensor cores and low precision",
                  FP8 scaling);
* ``bf16_mlp``    BF16 M=8192, N=28672, K=8192: N(0, 1) activations, N(0, 0.02)
                  weights, a BF16 N(0, 1) residual C with alpha = beta = 1 -- an
                  LLM MLP projection (prefill);
* ``fp8_skinny_M`` FP8 E4M3 M in {16, 64, 128}, N = K = 8192, N(0, 1) with 1%
                  outliers x 50, 1 x 128 scales for A and 128 x 128 for B -- a
                  decode-sized batch ("How Blackwell's Tensor Memory Actually
                  Works", "What this does to serving economics");
* ``mxfp8_4096``  microscaled FP8 4096^3: N(0, 1) with 1% outliers x 50, E4M3
                  codes with one E8M0 scale per row and 32-wide K block of A
                  and of B (the microscaling recipe), BF16 output -- the
                  hardware block scaling of the same page, "Quantization
                  became an allocation problem".

Tensor ids: A = 1, B = 2, C = 3.  Seeds as listed below.
"""

from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from . import bf16, e4m3_block128, e4m3_rowblock, e4m3_tensor, mx_quant, mx_tile_sf, values_f32


@dataclass
class Workload:
    name: str
    M: int
    N: int
    K: int
    kind: str            # "bf16" | "fp8_tensor" | "fp8_block" | "fp8_mx"
    out: str             # "bf16" | "f32"
    alpha: float = 1.0
    beta: float = 0.0
    A: np.ndarray = None  # rows x lda (uint16 BF16 bits or uint8 E4M3)
    B: np.ndarray = None  # N x ldb
    C: np.ndarray = None  # M x ldc (uint16 or float32), or None
    a_scale: np.ndarray = None
    b_scale: np.ndarray = None
    meta: dict = field(default_factory=dict)
    a_fp8: int = 0        # FP8 encodings of A and B: 0 = E4M3, 1 = E5M2
    b_fp8: int = 0
    a_sf: np.ndarray = None  # fp8_mx: E8M0 scale bytes of A and B, tiled layout
    b_sf: np.ndarray = None

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K

    @property
    def lda(self):
        return self.A.shape[1]

    @property
    def ldb(self):
        return self.B.shape[1]


NAMES = ("bf16_256", "bf16_4096", "fp8_4096", "bf16_mlp", "fp8_skinny_16", "fp8_skinny_64",
         "fp8_skinny_128", "fp8_block_4096", "bf16_skinny_16", "mxfp8_4096")


def make(name: str, *, M=None, N=None, K=None) -> Workload:
    """Build a named workload (sizes may be overridden for scaled-down tests)."""
    if name == "bf16_256":
        M, N, K = M or 256, N or 256, K or 256
        w = Workload(name, M, N, K, "bf16", "f32")
        w.A = bf16(1, 1, M, K, dist="uniform", p0=-1.0, p1=1.0)
        w.B = bf16(1, 2, N, K, dist="uniform", p0=-1.0, p1=1.0)
        return w
    if name == "bf16_4096":
        M, N, K = M or 4096, N or 4096, K or 4096
        w = Workload(name, M, N, K, "bf16", "bf16")
        w.A = bf16(2, 1, M, K)
        w.B = bf16(2, 2, N, K)
        return w
    if name == "fp8_4096":
        M, N, K = M or 4096, N or 4096, K or 4096
        w = Workload(name, M, N, K, "fp8_tensor", "bf16")
        w.A, sa = e4m3_tensor(values_f32(3, 1, M, K))
        w.B, sb = e4m3_tensor(values_f32(3, 2, N, K))
        w.a_scale, w.b_scale = sa, sb
        return w
    if name == "bf16_mlp":
        M, N, K = M or 8192, N or 28672, K or 8192
        w = Workload(name, M, N, K, "bf16", "bf16", alpha=1.0, beta=1.0)
        w.A = bf16(4, 1, M, K)
        w.B = bf16(4, 2, N, K, p1=0.02)
        w.C = bf16(4, 3, M, N)
        return w
    if name == "bf16_skinny_16":
        # a decode-sized BF16 GEMM: 16 rows of activations against an 8192^2 weight
        M, N, K = M or 16, N or 8192, K or 8192
        w = Workload(name, M, N, K, "bf16", "bf16")
        w.A = bf16(7, 1, M, K)
        w.B = bf16(7, 2, N, K, p1=0.02)
        return w
    if name == "fp8_block_4096":
        # the block scaling of the skinny workload on a square 4096^3 problem
        M, N, K = M or 4096, N or 4096, K or 4096
        w = Workload(name, M, N, K, "fp8_block", "bf16")
        w.A, w.a_scale = e4m3_rowblock(values_f32(6, 1, M, K, out_prob=0.01, out_factor=50.0))
        w.B, w.b_scale = e4m3_block128(values_f32(6, 2, N, K, out_prob=0.01, out_factor=50.0))
        return w
    if name == "mxfp8_4096":
        M, N, K = M or 4096, N or 4096, K or 4096
        w = Workload(name, M, N, K, "fp8_mx", "bf16")
        w.A, ea = mx_quant(values_f32(8, 1, M, K, out_prob=0.01, out_factor=50.0))
        w.B, eb = mx_quant(values_f32(8, 2, N, K, out_prob=0.01, out_factor=50.0))
        w.a_sf, w.b_sf = mx_tile_sf(ea, K), mx_tile_sf(eb, K)
        return w
    if name.startswith("fp8_skinny_"):
        M = M or int(name.rsplit("_", 1)[1])
        N, K = N or 8192, K or 8192
        w = Workload(name, M, N, K, "fp8_block", "bf16")
        w.A, w.a_scale = e4m3_rowblock(values_f32(5, 1, M, K, out_prob=0.01, out_factor=50.0))
        w.B, w.b_scale = e4m3_block128(values_f32(5, 2, N, K, out_prob=0.01, out_factor=50.0))
        return w
    raise KeyError(name)


def sample_tiles(M, N, n=16, size=128, seed=0):
    """Output tiles (i0, j0, rows, cols) for sampled checks and timings: the
    first and the last tile plus seeded random ones, all clipped to the
    matrix, first and last tile leading.  Tile selection only: no values."""
    rng = np.random.default_rng(seed)
    first, last = (0, 0), (max(0, M - size), max(0, N - size))
    tiles = {first, last}
    while len(tiles) < n:
        i0 = int(rng.integers(0, max(1, M - size + 1)))
        j0 = int(rng.integers(0, max(1, N - size + 1)))
        tiles.add((i0, j0))
        if len(tiles) >= max(1, M - size + 1) * max(1, N - size + 1):
            break  # every position taken (tiny matrices)
    order = [first] + ([last] if last != first else []) + sorted(tiles - {first, last})
    return [(i0, j0, min(size, M - i0), min(size, N - j0)) for i0, j0 in order]

