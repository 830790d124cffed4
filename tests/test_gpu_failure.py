"""The bounded-wait failure path on the GPU.

Every mbarrier wait in the library's kernels gives up after a time limit,
records TCG_ERR_TIMEOUT in a device status word and lets the kernel return,
instead of spinning forever on a shared GPU.  tcg_debug_timeout_probe runs
that wait against an mbarrier nothing signals; the test checks the status is
reported once, then cleared, and that the context still computes correctly.
No kernel here traps, faults or hangs: the wait is bounded by construction.
"""

from __future__ import annotations

import time

import numpy as np
import pytest

import synth
import synth.workloads as W
from helpers import check_f32, d_to_host, oracle_for, run

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import tensor_core_dense_gb300 as tcg
    tcg.lib()
    yield


def test_bounded_wait_reports_timeout_and_context_survives():
    import tensor_core_dense_gb300 as tcg
    stream = torch.cuda.current_stream().cuda_stream
    assert tcg.last_device_status() == tcg.OK          # nothing pending
    t0 = time.monotonic()
    assert tcg.lib().tcg_debug_timeout_probe(stream) == tcg.OK
    assert tcg.last_device_status() == tcg.ERR_TIMEOUT  # synchronises, reads, clears
    waited = time.monotonic() - t0
    assert 1.0 < waited < 60.0, waited                  # the 2 s limit, not forever
    assert tcg.last_device_status() == tcg.OK           # reported once
    # the context is intact: a GEMM after the timeout is still right
    w = W.Workload("after_timeout", 130, 200, 96, "bf16", "f32")
    w.A = synth.bf16(41, 1, 130, 96)
    w.B = synth.bf16(41, 2, 200, 96)
    v, b = oracle_for(w)
    check_f32("bf16", d_to_host(run(w)), v, b, what="GEMM after a timeout")
    assert tcg.last_device_status() == tcg.OK
