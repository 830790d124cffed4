"""The allocation-free block-scaled FP8 entry point, checked against the
oracle.

gemm_fp8_e4m3_block_noalloc is meant for callers that may not let a library
allocate device memory: programs capturing CUDA graphs, latency-bound loops
that cannot take the synchronisation an allocation can cause, and programs
whose memory manager owns all of device memory.  It keeps its split-K
scratch in a fixed array inside the library.  This file is collected last so
that a run stopping at the first failure has already run every other test; it
also passes on its own in a fresh process.
"""

import ctypes

import pytest

import synth
from helpers import c_values, check_bf16, check_f32, d_to_host, oracle_for, to_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _noalloc_fn():
    import tensor_core_dense_gb300 as tcg
    f = tcg.lib().gemm_fp8_e4m3_block_noalloc
    i64, vp, f32, i32 = ctypes.c_int64, ctypes.c_void_p, ctypes.c_float, ctypes.c_int
    f.argtypes = [i64, i64, i64, vp, i64, vp, i64, vp, vp, vp, i64, vp, i64, i32, f32, f32, vp]
    f.restype = i32
    return f


def _case(M, N, K, seed, out, beta):
    import synth.workloads as W
    w = W.Workload("noalloc", M, N, K, "fp8_block", out, beta=beta)
    ldk = -(-K // 16) * 16  # 16-byte row pitch for a ragged K
    w.A, w.a_scale = synth.e4m3_rowblock(synth.values_f32(seed, 1, M, K, out_prob=0.01,
                                                          out_factor=50.0), ld=ldk)
    w.B, w.b_scale = synth.e4m3_block128(synth.values_f32(seed, 2, N, K, out_prob=0.01,
                                                          out_factor=50.0), ld=ldk)
    if beta != 0.0:
        w.C = synth.bf16(seed, 3, M, N) if out == "bf16" else synth.values_f32(seed, 3, M, N)
    return w


# M <= 128 runs the skinny kernel: its cluster joins (tiles in three: 4096,
# 2048 columns; in two: 8192) need no scratch, more N tiles than SMs (20000
# columns) use the fixed scratch; M > 128 the pair-tile kernel, which needs
# none (the regular entry point may pick the chunked skinny kernel for the
# same shape: 300 x 1000).
@pytest.mark.parametrize("M,N,K,out,beta", [(64, 4096, 4096, "f32", 0.0),
                                            (16, 8192, 8192, "bf16", 0.0),
                                            (100, 2048, 3000, "bf16", -1.0),
                                            (128, 8192, 8192, "f32", 0.0),
                                            (32, 20000, 1024, "f32", 1.0),
                                            (300, 1000, 1024, "bf16", 1.0),
                                            (1024, 2048, 2048, "f32", 0.0)])
def test_noalloc_matches_oracle_twice(M, N, K, out, beta):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import tensor_core_dense_gb300 as tcg
    fn = _noalloc_fn()
    w = _case(M, N, K, seed=M + N, out=out, beta=beta)
    A, B = to_device(w.A)[:, :K], to_device(w.B)[:, :K]
    ldk = w.lda
    sa, sb = to_device(w.a_scale), to_device(w.b_scale)
    dt = torch.float32 if out == "f32" else torch.bfloat16
    C = to_device(w.C) if w.C is not None else None
    if C is not None and C.dtype != dt:
        C = C.to(dt)
    v, bound = oracle_for(w)
    c = c_values(w.C)
    stream = torch.cuda.current_stream().cuda_stream
    out_code = tcg.OUT_F32 if out == "f32" else tcg.OUT_BF16
    for call in range(2):  # the second call reuses the scratch the first one left
        D = torch.full((M, N), float("nan"), dtype=dt, device="cuda")
        st = fn(M, N, K, A.data_ptr(), ldk, B.data_ptr(), ldk, sa.data_ptr(), sb.data_ptr(),
                C.data_ptr() if C is not None else None, N, D.data_ptr(), N, out_code, 1.0,
                beta, stream)
        assert st == tcg.OK, tcg.status_string(st)
        got = d_to_host(D)
        what = f"noalloc {M}x{N}x{K} {out} call {call}"
        if out == "bf16":
            check_bf16("fp8", got, v, bound, beta, c, what=what)
        else:
            check_f32("fp8", got, v, bound, beta, c, what=what)
    assert tcg.last_device_status() == tcg.OK


def test_noalloc_rejects_problems_beyond_its_scratch():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import tensor_core_dense_gb300 as tcg
    fn = _noalloc_fn()
    # The buffers below are far smaller than the problem, so this call must be
    # refused by the host before anything is launched.  Its tile counters
    # alone (one 4-byte word per 128 columns of N: 64 MiB here) exceed the
    # 32 MiB array, whatever the partial-sum layout.  Check that arithmetic
    # here first, so a change to the scratch sizing fails this test instead
    # of launching a kernel over undersized buffers.
    M, N, K = 128, (1 << 31) - 128, 8192
    counter_bytes = -(-N // 128) * 4
    assert counter_bytes > 32 << 20, "this rejection case no longer exceeds the scratch array"
    A = torch.zeros((M, K), dtype=torch.uint8, device="cuda")
    sa = torch.ones(M * (K // 128), device="cuda")
    D = torch.empty((M, 16), dtype=torch.float32, device="cuda")
    st = fn(M, N, K, A.data_ptr(), K, A.data_ptr(), K, sa.data_ptr(), sa.data_ptr(), None, 0,
            D.data_ptr(), N, tcg.OUT_F32, 1.0, 0.0, torch.cuda.current_stream().cuda_stream)
    assert st == tcg.ERR_UNSUPPORTED
