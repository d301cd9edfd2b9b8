"""The next W4A8 layer's activation step fused into the producing layer (GPU).

qgemm_run_fused_quant writes C as qgemm_run_fused does and the activation codes of C; they must
equal, bit for bit, the oracle's activation quantization of C's stored values. The W4A8 layer fed
with those codes (qgemm_run_w4a8_codes) must give exactly what qgemm_run gives on C. Cases cover
the tensor-core route (epilogue row maxima, ragged tiles, a shape that would otherwise split K,
the W4A8 producer) and the routes that run the standalone pass (decode, float32 activations).
"""
import numpy as np
import pytest
import torch

import oracle
import weight_quantized_gemm_gb300 as qg
from weight_quantized_gemm_gb300 import synth
from tests._util import check_close, ensure_built, to_numpy_values, torch_dtype, torch_from
from tests.test_gpu_decode import gpu_pack

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def built():
    ensure_built()


CASES = [
    # M, K, N, mode, block, a_dtype, c_dtype, act, bias
    (256, 1024, 512, 1, 64, synth.F16, synth.BF16, 0, False),
    (300, 512, 256, 3, 0, synth.BF16, synth.BF16, 2, True),      # W4A8 producer, ragged row tile
    (130, 1024, 192, 2, 0, synth.BF16, synth.F16, 3, True),      # ragged channel tile (N = 128 + 64)
    (64, 2560, 1024, 1, 64, synth.F16, synth.BF16, 1, False),    # split K otherwise
    (8, 1024, 512, 1, 64, synth.BF16, synth.BF16, 0, True),      # decode: standalone pass
    (40, 512, 256, 1, 64, synth.F32, synth.F32, 0, False),       # float32: standalone pass
]


@pytest.mark.parametrize("M,K,N,mode,block,a_dtype,c_dtype,act,bias", CASES)
def test_fused_quant_codes_and_consumer(M, K, N, mode, block, a_dtype, c_dtype, act, bias):
    w = synth.Workload("t", M, K, N, mode, block, a_dtype, c_dtype, 5, 6)
    A_np, W_np = synth.make_activations(w), synth.make_weights(w)
    ref = oracle.reference_layer(mode, block, A_np, a_dtype, W_np)
    b_np = synth.normal64(N, 9, stream=4, std=0.5).astype(np.float32) if bias else None
    R = oracle.epilogue(ref["R"], b_np, act)
    Bp, T = gpu_pack(W_np, mode, block)
    A = torch_from(A_np, a_dtype)
    bias_t = None if b_np is None else torch.from_numpy(b_np).to(DEV)
    C = torch.full((M, N), float("nan"), dtype=torch_dtype(c_dtype), device=DEV)
    qa = torch.full((M, N), 999.0, dtype=torch.float16, device=DEV)
    asc = torch.full((M,), -1.0, dtype=torch.float32, device=DEV)
    rs = torch.full((M,), -7, dtype=torch.int32, device=DEV)
    wsb = qg.qgemm_fused_quant_workspace_bytes(M, K, N, mode, block, a_dtype, c_dtype)
    ws = torch.empty(max(wsb, 16), dtype=torch.uint8, device=DEV)
    qg.qgemm_run_fused_quant(M, K, N, mode, block, A, a_dtype, Bp, T, bias_t, act, None, C, c_dtype, qa, asc, rs,
                             ws, wsb)
    torch.cuda.synchronize()
    assert qg.qgemm_status() == 0
    got = to_numpy_values(C, c_dtype)
    check_close(got, R, a_dtype if a_dtype != synth.F32 or mode == 3 else synth.F32, c_dtype, "layer")
    # the codes: the oracle's activation quantization of C as stored
    qa_r, s_r, rs_r = oracle.act_quant(got.astype(np.float32))
    assert np.array_equal(qa.float().cpu().numpy(), qa_r.astype(np.float32))
    assert np.array_equal(asc.cpu().numpy(), s_r)
    assert np.array_equal(rs.cpu().numpy(), rs_r)

    # the consumer: a W4A8 layer K2 = N -> N2 from the codes equals qgemm_run on C
    N2 = 136
    w2 = synth.Workload("t2", M, N, N2, 3, 0, c_dtype, synth.BF16, 7, 8)
    Bp2, T2 = gpu_pack(synth.make_weights(w2), 3, 0)
    out_codes = torch.full((M, N2), float("nan"), dtype=torch.bfloat16, device=DEV)
    wsb2 = qg.qgemm_w4a8_codes_workspace_bytes(M, N, N2, 0)
    qg.qgemm_run_w4a8_codes(M, N, N2, 0, qa, asc, rs, Bp2, T2, None, 0, None, out_codes, synth.BF16,
                            torch.empty(max(wsb2, 16), dtype=torch.uint8, device=DEV), wsb2)
    out_plain = torch.full((M, N2), float("nan"), dtype=torch.bfloat16, device=DEV)
    wsb3 = qg.qgemm_workspace_bytes(M, N, N2, 3, 0, c_dtype, synth.BF16)
    qg.qgemm_run(M, N, N2, 3, 0, C, c_dtype, Bp2, T2, out_plain, synth.BF16,
                 torch.empty(max(wsb3, 16), dtype=torch.uint8, device=DEV), wsb3)
    torch.cuda.synchronize()
    assert torch.equal(out_codes.view(torch.int16), out_plain.view(torch.int16))


def test_fused_quant_long_rows_zero_and_tiny_rows():
    """Rows of 4096 codes from 32 channel tiles, with a fused residual. Rows 3 and 5 have zero
    activations, so there C is the residual exactly: zero in row 3 (scale 0, codes 0), tiny values
    in row 5 whose scale max|C| / 127 is a subnormal float32."""
    M, K, N = 200, 512, 4096
    w = synth.Workload("t", M, K, N, 1, 64, synth.BF16, synth.BF16, 11, 12)
    A_np, W_np = synth.make_activations(w).copy(), synth.make_weights(w)
    A_np[3] = 0
    A_np[5] = 0
    res64 = synth.normal64(M * N, 13, stream=5).reshape(M, N)
    res64[3] = 0.0
    res64[5] *= 1e-37
    res_np = synth.encode(res64, synth.BF16)
    Bp, T = gpu_pack(W_np, 1, 64)
    A, res = torch_from(A_np, synth.BF16), torch_from(res_np, synth.BF16)
    C = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
    qa = torch.empty((M, N), dtype=torch.float16, device=DEV)
    asc = torch.empty(M, dtype=torch.float32, device=DEV)
    rs = torch.empty(M, dtype=torch.int32, device=DEV)
    wsb = qg.qgemm_fused_quant_workspace_bytes(M, K, N, 1, 64, synth.BF16, synth.BF16)
    qg.qgemm_run_fused_quant(M, K, N, 1, 64, A, synth.BF16, Bp, T, None, 0, res, C, synth.BF16, qa, asc, rs,
                             torch.empty(wsb, dtype=torch.uint8, device=DEV), wsb)
    torch.cuda.synchronize()
    got = to_numpy_values(C, synth.BF16).astype(np.float32)
    assert not got[3].any()
    assert np.array_equal(got[5], oracle.values(res_np[5], synth.BF16).astype(np.float32))
    assert 0 < np.abs(got[5]).max() / np.float32(127) < np.finfo(np.float32).tiny
    qa_r, s_r, rs_r = oracle.act_quant(got)
    assert np.array_equal(qa.float().cpu().numpy(), qa_r.astype(np.float32))
    assert np.array_equal(asc.cpu().numpy(), s_r)
    assert np.array_equal(rs.cpu().numpy(), rs_r)
