"""The bounded waits of the TMA-fed kernels, made to run out on purpose (GPU).

QGEMM_OPT_DEBUG_STALL has one role of every following launch wait on a barrier that nothing
arrives at; with QGEMM_OPT_WAIT_LIMIT_US lowered, that wait runs out within milliseconds. The
call must then end by itself: qgemm_status reports QGEMM_ERR_TIMEOUT (and clears the word), the
copies and MMAs already issued were drained and the tensor memory released, so the next normal
call on the same context returns the same bits as before. No wait here is unbounded and nothing
faults: the stalled wait is the library's ordinary bounded wait.

A host-side simulated launch failure (QGEMM_OPT_FAULT_INJECT) is checked here too, on real
buffers: the failing call enqueues nothing and leaves its output untouched.
"""
import numpy as np
import pytest
import torch

import weight_quantized_gemm_gb300 as qg
from weight_quantized_gemm_gb300 import synth
from tests._util import ensure_built, torch_dtype, torch_from
from tests.test_gpu_decode import gpu_pack

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def built():
    ensure_built()


def _layer(M, K, N, mode, block, a_dtype):
    w = synth.Workload("t", M, K, N, mode, block, a_dtype, synth.BF16, 3, 4)
    A = torch_from(synth.make_activations(w), a_dtype)
    Bp, T = gpu_pack(synth.make_weights(w), mode, block)
    wsb = qg.qgemm_workspace_bytes(M, K, N, mode, block, a_dtype, synth.BF16)
    ws = torch.empty(max(wsb, 16), dtype=torch.uint8, device=DEV)

    def run(C=None):
        if C is None:
            C = torch.full((M, N), float("nan"), dtype=torch_dtype(synth.BF16), device=DEV)
        qg.qgemm_run(M, K, N, mode, block, A, a_dtype, Bp, T, C, synth.BF16, ws, wsb)
        return C
    return run


# the tensor-core kernel (Int4 prefill; W4A8 after its activation pass) and the TMA-fed decode
# kernel (M = 1 and M = 12: one and two column tiles)
CASES = [(256, 1024, 1024, 1, 64, synth.F16), (64, 1024, 512, 3, 0, synth.BF16),
         (1, 4096, 4096, 1, 64, synth.BF16), (12, 2048, 1024, 2, 0, synth.F16)]


@pytest.mark.parametrize("M,K,N,mode,block,a_dtype", CASES)
def test_wait_runs_out_then_next_call_is_exact(M, K, N, mode, block, a_dtype):
    run = _layer(M, K, N, mode, block, a_dtype)
    ref = run()
    assert qg.qgemm_status() == 0
    ref = ref.float().cpu().numpy()
    assert np.all(np.isfinite(ref))
    prev_wait = qg.qgemm_set_option(qg.OPT_WAIT_LIMIT_US, 2000)
    prev_stall = qg.qgemm_set_option(qg.OPT_DEBUG_STALL, 1)
    try:
        run()
        assert qg.qgemm_status() == -6            # QGEMM_ERR_TIMEOUT
        assert "bounded wait" in qg.qgemm_last_error()
    finally:
        qg.qgemm_set_option(qg.OPT_DEBUG_STALL, prev_stall)
        qg.qgemm_set_option(qg.OPT_WAIT_LIMIT_US, prev_wait)
    assert qg.qgemm_status() == 0                 # the word was cleared
    for _ in range(2):                            # tensor memory and barriers are usable again
        got = run()
        assert qg.qgemm_status() == 0
        assert np.array_equal(got.float().cpu().numpy(), ref)


def test_injected_launch_failure_enqueues_nothing():
    M, K, N = 1, 2048, 1024
    run = _layer(M, K, N, 1, 64, synth.BF16)
    ref = run().float().cpu().numpy()
    prev = qg.qgemm_set_option(qg.OPT_FAULT_INJECT, 2)
    try:
        first = run()                             # counted, runs normally
        C = torch.full((M, N), float("nan"), dtype=torch_dtype(synth.BF16), device=DEV)
        with pytest.raises(qg.QgemmError) as ei:
            run(C)
        assert ei.value.code == -5 and "simulated launch failure" in str(ei.value)
        assert qg.qgemm_get_option(qg.OPT_FAULT_INJECT) == 0
    finally:
        qg.qgemm_set_option(qg.OPT_FAULT_INJECT, prev)
    torch.cuda.synchronize()
    assert np.array_equal(first.float().cpu().numpy(), ref)
    assert torch.isnan(C.float()).all()           # the failed call wrote nothing
    assert qg.qgemm_status() == 0
    third = run()
    assert np.array_equal(third.float().cpu().numpy(), ref)
