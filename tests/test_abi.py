"""The C-ABI library without a GPU: it builds, loads, exports every symbol
include/tcgemm.h declares, and rejects bad arguments on the host before any
CUDA call (so these run on a machine with no GPU)."""

import ctypes
import os
import re
import shutil

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = []
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if h.endswith(".h"):
            text = open(os.path.join(ROOT, "include", h)).read()
            names += re.findall(r"^(?:tcg_status|const char\*|uint64_t)\s+(\w+)\s*\(", text, re.M)
    return names


@pytest.fixture(scope="module")
def tcg():
    if shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"):
        pytest.skip("nvcc not available")
    from tensor_core_dense_gb300 import build
    build.build()
    import tensor_core_dense_gb300 as t
    t.lib()
    return t


def test_exports_every_declared_symbol(tcg):
    names = _declared()
    assert set(names) >= {"gemm_bf16", "gemm_fp8_e4m3", "tcg_status_string",
                          "tcg_last_device_status"}
    raw = ctypes.CDLL(tcg.LIB_PATH)
    for n in names:
        assert hasattr(raw, n), n
    assert set(names) == set(tcg.EXPORTS)


def test_status_strings(tcg):
    for code in range(6):
        assert tcg.status_string(code)
    assert tcg.status_string(99) == "unknown status"


A, B, C, D = 0x10000, 0x20000, 0x30000, 0x40000   # never dereferenced: validation fails first


@pytest.mark.parametrize("args,want", [
    ((-1, 8, 8, A, 8, B, 8, None, 0, D, 8, 0, 1.0, 0.0), 1),      # negative M
    ((8, 8, 8, A, 4, B, 8, None, 0, D, 8, 0, 1.0, 0.0), 1),       # lda < K
    ((8, 8, 8, A, 8, B, 8, None, 0, None, 8, 0, 1.0, 0.0), 1),    # D NULL
    ((8, 8, 8, A, 8, B, 8, None, 0, D, 8, 0, 1.0, 1.0), 1),       # beta != 0 without C
    ((8, 8, 8, None, 8, B, 8, None, 0, D, 8, 0, 1.0, 0.0), 1),    # A NULL
    ((8, 8, 8, A + 2, 8, B, 8, None, 0, D, 8, 0, 1.0, 0.0), 2),   # A misaligned
    ((8, 8, 12, A, 12, B, 16, None, 0, D, 8, 0, 1.0, 0.0), 2),    # lda*2 not 16-byte multiple
    ((8, 9, 8, A, 8, B, 8, None, 0, D, 9, 0, 1.0, 0.0), 2),       # ldd*2 not 16-byte multiple
    ((8, 8, 8, A, 8, B, 8, None, 0, D, 8, 7, 1.0, 0.0), 3),       # bad out dtype
    ((0, 8, 8, None, 0, None, 0, None, 0, None, 0, 0, 1.0, 0.0), 0),  # empty: no-op
    ((8, 0, 8, None, 0, None, 0, None, 0, None, 0, 0, 1.0, 0.0), 0),
])
def test_bf16_host_validation(tcg, args, want):
    assert tcg.gemm_bf16_raw(*args, None) == want


@pytest.mark.parametrize("args,want", [
    ((8, 8, 16, A, 16, B, 16, None, None, 0, None, 0, D, 8, 0, 1.0, 0.0), 1),  # no scales
    ((8, 8, 16, A, 16, B, 16, A, B, 5, None, 0, D, 8, 0, 1.0, 0.0), 3),        # bad mode
    ((8, 8, 24, A, 24, B, 32, A, B, 0, None, 0, D, 8, 0, 1.0, 0.0), 2),        # lda not x16
    ((8, 8, 16, A, 8, B, 16, A, B, 0, None, 0, D, 8, 0, 1.0, 0.0), 1),         # lda < K
])
def test_fp8_host_validation(tcg, args, want):
    assert tcg.gemm_fp8_e4m3_raw(*args, None) == want


def test_binding_refuses_without_library(monkeypatch, tmp_path):
    import tensor_core_dense_gb300 as t
    monkeypatch.setattr(t, "_lib", None)
    monkeypatch.setattr(t, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(ImportError):
        t.lib()


X, Q, S = 0x10000, 0x20000, 0x30000   # never dereferenced: validation fails first


@pytest.mark.parametrize("args,want", [
    ((-1, 8, X, 8, 0, 0, Q, 16, S), 1),        # negative rows
    ((8, 8, X, 4, 0, 0, Q, 16, S), 1),         # ldx < cols
    ((8, 8, X, 8, 0, 0, Q, 4, S), 1),          # ldq < cols
    ((8, 8, None, 8, 0, 0, Q, 16, S), 1),      # X NULL
    ((8, 8, X, 8, 0, 1, None, 16, S), 1),      # Q NULL
    ((8, 8, X, 8, 0, 2, Q, 16, None), 1),      # scale NULL
    ((8, 8, X + 4, 8, 0, 0, Q, 16, S), 2),     # X misaligned
    ((8, 6, X, 6, 0, 0, Q, 16, S), 2),         # ldx*4 not a multiple of 16
    ((8, 4, X, 4, 1, 0, Q, 16, S), 2),         # BF16: ldx*2 not a multiple of 16
    ((8, 8, X, 8, 0, 0, Q, 8, S), 2),          # ldq not a multiple of 16
    ((8, 8, X, 8, 0, 0, Q + 1, 16, S), 2),     # Q misaligned
    ((8, 8, X, 8, 0, 0, Q, 16, S + 2), 2),     # scale misaligned
    ((8, 8, X, 8, 5, 0, Q, 16, S), 3),         # bad input dtype
    ((8, 8, X, 8, 0, 7, Q, 16, S), 3),         # bad mode
    ((0, 8, None, 0, 0, 1, None, 0, None), 0),  # empty, row blocks: no-op
    ((8, 0, None, 0, 0, 2, None, 0, None), 0),  # empty, 128 x 128 blocks: no-op
    ((0, 8, None, 0, 0, 0, None, 0, None), 1),  # empty per-tensor writes scale[0]: needs it
])
def test_quant_host_validation(tcg, args, want):
    assert tcg.quantize_e4m3_raw(*args, None) == want



def test_quant_fp8_format_validation(tcg):
    # an unknown FP8 format is refused before anything runs
    assert tcg.quantize_fp8_raw(8, 8, X, 8, 0, 7, 0, Q, 16, S, None) == 3


def test_binding_refuses_beta_without_c():
    # the tensor API must not turn a non-zero beta into 0 when C is missing:
    # it raises before reaching the library (CPU tensors, nothing launched)
    torch = pytest.importorskip("torch")
    import tensor_core_dense_gb300 as t
    A = torch.zeros((16, 16), dtype=torch.bfloat16)
    D = torch.zeros((16, 16), dtype=torch.float32)
    with pytest.raises(ValueError, match="needs C"):
        t.gemm_bf16(A, A, D, None, beta=1.0)
    A8 = torch.zeros((16, 16), dtype=torch.uint8)
    s = torch.ones(1, dtype=torch.float32)
    with pytest.raises(ValueError, match="needs C"):
        t.gemm_fp8_e4m3(A8, A8, s, s, D, None, beta=-2.0)
    with pytest.raises(ValueError, match="needs C"):
        t.gemm_fp8(A8, A8, s, s, D, None, beta=0.5)


@pytest.mark.parametrize("args,want", [
    ((8, 8, 16, A, 16, 0, B, 16, 0, None, B, None, 0, D, 8, 0, 1.0, 0.0), 1),   # no A scales
    ((8, 8, 16, A, 16, 0, B, 16, 0, A, B + 8, None, 0, D, 8, 0, 1.0, 0.0), 2),  # B scales misaligned
    ((8, 8, 16, A, 16, 2, B, 16, 0, A, B, None, 0, D, 8, 0, 1.0, 0.0), 3),      # bad A format
    ((8, 8, 24, A, 24, 0, B, 32, 0, A, B, None, 0, D, 8, 0, 1.0, 0.0), 2),      # lda not x16
    ((8, 8, 16, A, 16, 0, B, 16, 0, A, B, None, 0, D, 8, 0, 1.0, 1.0), 1),      # beta, no C
    ((0, 8, 16, None, 0, 0, None, 0, 0, None, None, None, 0, None, 0, 0, 1.0, 0.0), 0),
])
def test_mxfp8_host_validation(tcg, args, want):
    assert tcg.gemm_mxfp8_raw(*args, None) == want
