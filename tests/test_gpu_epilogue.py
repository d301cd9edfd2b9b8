"""GPU parity of the fused epilogue (qgemm_run_fused: C = act(A x dequant(B) + bias) + residual)
against the CPU oracle, through the C ABI, on every kernel path: the decode kernels (one column,
one and two 8-row tiles, K split across blocks), the exact float32 kernel, the tensor-core kernel
with and without K-splits, and W4A8. The bar is the layer's own (2e-3 normwise for 16-bit
activations, 1e-5 for float32, plus half an output ulp)."""
import numpy as np
import pytest
import torch

import oracle
import weight_quantized_gemm_gb300 as qg
from weight_quantized_gemm_gb300 import synth
from tests._util import check_close, ensure_built, to_numpy_values, torch_dtype, torch_from
from tests.test_gpu_decode import CANARY, gpu_pack

pytestmark = pytest.mark.gpu
DEV = "cuda"
ACTS = [qg.ACT_NONE, qg.ACT_RELU, qg.ACT_SILU, qg.ACT_GELU_TANH]


@pytest.fixture(scope="module", autouse=True)
def built():
    ensure_built()


def fused_case(M, K, N, mode, block, a_dtype, c_dtype, act, with_bias, residual, seed=3):
    """residual: None, "separate" or "inplace" (the residual is C itself)."""
    w = synth.Workload("t", M, K, N, mode, block, a_dtype, c_dtype, seed, seed + 1)
    A_np, W_np = synth.make_activations(w), synth.make_weights(w)
    w_dtype = a_dtype if mode == 0 else 0
    ref = oracle.reference_layer(mode, block, A_np, a_dtype, W_np, w_dtype)
    bias_np = synth.normal64(N, seed + 2, stream=4, std=0.5).astype(np.float32) if with_bias else None
    res_np = synth.encode(synth.normal64(M * N, seed + 3, stream=5).reshape(M, N), c_dtype) if residual else None
    R = oracle.epilogue(ref["R"], bias_np, act, None if res_np is None else oracle.values(res_np, c_dtype))

    Bp, T = gpu_pack(W_np, mode, block, w_dtype)
    A = torch_from(A_np, a_dtype)
    flat = torch.full((M * N + CANARY,), float("nan"), dtype=torch_dtype(c_dtype), device=DEV)
    C = flat[: M * N].view(M, N)
    res = None
    if residual == "inplace":
        C.copy_(torch_from(res_np, c_dtype))
        res = C
    elif residual == "separate":
        res = torch_from(res_np, c_dtype)
    bias = None if bias_np is None else torch.from_numpy(bias_np).to(DEV)
    wsb = qg.qgemm_workspace_bytes(M, K, N, mode, block, a_dtype, c_dtype)
    ws = torch.empty(max(wsb, 16), dtype=torch.uint8, device=DEV)
    qg.qgemm_run_fused(M, K, N, mode, block, A, a_dtype, Bp, T, bias, act, res, C, c_dtype, ws, wsb)
    assert qg.qgemm_status() == 0
    assert torch.isnan(flat[M * N:]).all(), "write past the end of C"
    return check_close(to_numpy_values(C, c_dtype), R, a_dtype, c_dtype,
                       f"M{M} K{K} N{N} mode{mode} act{act} bias{with_bias} res{residual}")


# every activation, with bias and a separate residual, on each path
PATHS = [
    (1, 1024, 300, 1, 64, synth.BF16, synth.BF16),      # decode, one column
    (4, 512, 257, 2, 0, synth.F16, synth.F16),          # decode, one 8-row tile
    (12, 1024, 200, 1, 128, synth.BF16, synth.BF16),    # decode, two 8-row tiles
    (3, 4096, 64, 1, 64, synth.BF16, synth.BF16),       # decode with K split across blocks
    (5, 256, 96, 1, 64, synth.F32, synth.F32),          # exact float32 kernel
    (64, 2560, 512, 1, 64, synth.F16, synth.BF16),      # tensor cores, K split across blocks
    (300, 256, 136, 2, 64, synth.BF16, synth.BF16),     # tensor cores, ragged 256-row tiles
    (40, 512, 130, 0, 0, synth.F16, synth.F16),         # tensor cores, float mode
    (40, 512, 96, 3, 0, synth.BF16, synth.BF16),        # W4A8
]


@pytest.mark.parametrize("act", ACTS)
@pytest.mark.parametrize("M,K,N,mode,block,a_dtype,c_dtype", PATHS)
def test_fused_epilogue(M, K, N, mode, block, a_dtype, c_dtype, act):
    fused_case(M, K, N, mode, block, a_dtype, c_dtype, act, True, "separate")


@pytest.mark.parametrize("M,K,N,mode,block,a_dtype,c_dtype", PATHS)
def test_fused_epilogue_parts(M, K, N, mode, block, a_dtype, c_dtype):
    """Bias alone, residual alone (in place: the residual is C), and nothing (= qgemm_run)."""
    fused_case(M, K, N, mode, block, a_dtype, c_dtype, qg.ACT_NONE, True, None)
    fused_case(M, K, N, mode, block, a_dtype, c_dtype, qg.ACT_SILU, False, "inplace")
    fused_case(M, K, N, mode, block, a_dtype, c_dtype, qg.ACT_NONE, False, None)


def test_fused_epilogue_f32_output_of_16bit_path():
    fused_case(33, 1024, 200, 1, 64, synth.F16, synth.F32, qg.ACT_GELU_TANH, True, "separate")



def test_fused_epilogue_residual_after_long_k():
    """Tensor cores without K-splits over many stages: the residual tile's TMA load into the
    staging area must wait for the last use of every ring slot it overwrites (int4 on 256-row
    tiles, and W4A8 on 128-row tiles with two sub-stages per stage)."""
    prev = qg.qgemm_set_option(qg.OPT_SPLIT_K, 0)
    try:
        fused_case(200, 4096, 384, 1, 64, synth.F16, synth.BF16, qg.ACT_SILU, True, "separate")
        fused_case(200, 4096, 384, 1, 64, synth.F16, synth.BF16, qg.ACT_NONE, False, "inplace")
        fused_case(100, 2048, 256, 3, 0, synth.BF16, synth.BF16, qg.ACT_GELU_TANH, True, "inplace")
    finally:
        qg.qgemm_set_option(qg.OPT_SPLIT_K, prev)
