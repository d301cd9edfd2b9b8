"""qgemm_run_noalloc: the same layer as qgemm_run, with the library's built-in scratch array in
place of a caller workspace.

It exists for callers that cannot give the library device memory of their own -- an engine
plugin that must not allocate in its execution path, a latency-critical loop that cannot call
an allocator, a plain C host with no device allocator. The test checks, through the C ABI,
that two calls in a row give the same results as qgemm_run with a caller workspace (within the
tolerance used everywhere else), and that a call needing more scratch than the array holds is
refused before anything runs. It packs its own weights, so it passes alone or after the rest
of the suite; the file name keeps it last in collection order.
"""
import numpy as np
import pytest
import torch

import weight_quantized_gemm_gb300 as qg
from weight_quantized_gemm_gb300 import synth
from tests._util import check_close, ensure_built, to_numpy_values, torch_dtype, torch_from

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def built():
    ensure_built()


def _prepare(w: synth.Workload):
    A = torch_from(synth.make_activations(w), w.a_dtype)
    Wd = torch.from_numpy(synth.make_weights(w)).to(DEV)
    Bp = torch.empty(qg.qgemm_packed_bytes(w.K, w.N, w.mode), dtype=torch.uint8, device=DEV)
    T = torch.empty(qg.qgemm_table_bytes(w.K, w.N, w.mode, w.block) // 4, dtype=torch.float32, device=DEV)
    qg.qgemm_pack(Wd, w.K, w.N, w.mode, w.block, 0, Bp, T)
    return A, Bp, T


@pytest.mark.parametrize("w", [
    # decode with K split across thread blocks (small N): scratch holds the float32 partial sums
    synth.Workload("decode_splitk", 2, 4096, 64, synth.MODE_INT4, 64, synth.BF16, synth.BF16, 3, 4),
    # W4A8: scratch holds the activation codes, row scales and row sums
    synth.Workload("w4a8_small", 64, 1024, 256, synth.MODE_W4A8, 0, synth.BF16, synth.BF16, 5, 6),
], ids=lambda w: w.name)
def test_noalloc_matches_run_twice(w):
    need = qg.qgemm_workspace_bytes(w.M, w.K, w.N, w.mode, w.block, w.a_dtype, w.c_dtype)
    assert 0 < need <= qg.NOALLOC_SCRATCH_BYTES
    A, Bp, T = _prepare(w)
    ref = torch.empty((w.M, w.N), dtype=torch_dtype(w.c_dtype), device=DEV)
    ws = torch.empty(need, dtype=torch.uint8, device=DEV)
    qg.qgemm_run(w.M, w.K, w.N, w.mode, w.block, A, w.a_dtype, Bp, T, ref, w.c_dtype, ws, need)
    torch.cuda.synchronize()
    R = to_numpy_values(ref, w.c_dtype)
    for _ in range(2):
        out = torch.full((w.M, w.N), float("nan"), dtype=torch_dtype(w.c_dtype), device=DEV)
        qg.qgemm_run_noalloc(w.M, w.K, w.N, w.mode, w.block, A, w.a_dtype, Bp, T, out, w.c_dtype)
        assert qg.qgemm_status() == 0
        check_close(to_numpy_values(out, w.c_dtype), R, w.a_dtype, w.c_dtype, f"noalloc {w.name}")


def test_noalloc_cuts_tensor_core_splits():
    """The tensor-core path's split-K partials are optional scratch: M = 128, N = 4096, K = 4096
    prefers 4 splits (8 MiB of partials), the built-in array holds 2; the call runs with 2."""
    import oracle
    w = synth.Workload("prefill_splitk", 128, 4096, 4096, synth.MODE_INT4, 64, synth.BF16, synth.BF16, 7, 8)
    need = qg.qgemm_workspace_bytes(w.M, w.K, w.N, w.mode, w.block, w.a_dtype, w.c_dtype)
    assert need == 4 * w.M * w.N * 4 > qg.NOALLOC_SCRATCH_BYTES
    A_np, W_np = synth.make_activations(w), synth.make_weights(w)
    ref = oracle.reference_layer(w.mode, w.block, A_np, w.a_dtype, W_np, 0)
    A, Bp, T = _prepare(w)
    out = torch.full((w.M, w.N), float("nan"), dtype=torch_dtype(w.c_dtype), device=DEV)
    qg.qgemm_run_noalloc(w.M, w.K, w.N, w.mode, w.block, A, w.a_dtype, Bp, T, out, w.c_dtype)
    assert qg.qgemm_status() == 0
    check_close(to_numpy_values(out, w.c_dtype), ref["R"], w.a_dtype, w.c_dtype, "noalloc split-K")


def test_noalloc_refuses_oversized_call():
    # W4A8 at M = 2048, K = 4096 needs ~16.8 MB of scratch, more than the built-in array
    w = synth.Workload("w4a8_big", 2048, 4096, 128, synth.MODE_W4A8, 0, synth.BF16, synth.BF16, 0, 1)
    assert qg.qgemm_workspace_bytes(w.M, w.K, w.N, w.mode, 0, w.a_dtype, w.c_dtype) > qg.NOALLOC_SCRATCH_BYTES
    A = torch.zeros((w.M, w.K), dtype=torch.bfloat16, device=DEV)
    Bp = torch.zeros(w.N * w.K // 2, dtype=torch.uint8, device=DEV)
    T = torch.zeros(w.N * 2, dtype=torch.float32, device=DEV)
    C = torch.full((w.M, w.N), float("nan"), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(qg.QgemmError) as e:
        qg.qgemm_run_noalloc(w.M, w.K, w.N, w.mode, 0, A, w.a_dtype, Bp, T, C, w.c_dtype)
    assert e.value.code == -4
    torch.cuda.synchronize()
    assert torch.isnan(C.float()).all()     # nothing was launched
