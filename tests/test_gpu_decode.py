"""GPU parity of weight packing and the decode path (M <= 16, and M > 16 where the tensor-core
kernel does not apply) against the CPU oracle, through the C ABI.

Bars: packed weights and tables bit-exact; outputs within 2e-3 (16-bit activations) or 1e-5
(float32 activations) normwise, plus half an output ulp for 16-bit outputs."""
import numpy as np
import pytest
import torch

import oracle
import weight_quantized_gemm_gb300 as qg
from weight_quantized_gemm_gb300 import synth
from tests._util import check_close, ensure_built, table_rows, to_numpy_values, torch_dtype, torch_from

pytestmark = pytest.mark.gpu
DEV = "cuda"
CANARY = 1024   # elements of guard band after every output


@pytest.fixture(scope="module", autouse=True)
def built():
    ensure_built()


def gpu_pack(W: np.ndarray, mode: int, block: int, w_dtype: int = 0):
    K, N = W.shape
    Wd = torch.from_numpy(np.ascontiguousarray(W)).to(DEV)
    pb = qg.qgemm_packed_bytes(K, N, mode, w_dtype)
    tb = qg.qgemm_table_bytes(K, N, mode, block)
    Bp = torch.empty(pb, dtype=torch.uint8, device=DEV)
    T = torch.empty(tb // 4, dtype=torch.float32, device=DEV) if tb else None
    qg.qgemm_pack(Wd, K, N, mode, block, w_dtype, Bp, T)
    torch.cuda.synchronize()
    return Bp, T


def gpu_run(M, K, N, mode, block, A_np, a_dtype, Bp, T, c_dtype, ws_bytes=None):
    """qgemm_run with the workspace qgemm_workspace_bytes asks for, or with ws_bytes of it."""
    A = torch_from(A_np, a_dtype)
    # NaN-poisoned output followed by a guard band: every output must be written, nothing after it
    flat = torch.full((M * N + CANARY,), float("nan"), dtype=torch_dtype(c_dtype), device=DEV)
    C = flat[: M * N].view(M, N)
    wsb = qg.qgemm_workspace_bytes(M, K, N, mode, block, a_dtype, c_dtype) if ws_bytes is None else ws_bytes
    ws = torch.empty(wsb + 4096, dtype=torch.uint8, device=DEV).fill_(0xA5) if wsb else None
    qg.qgemm_run(M, K, N, mode, block, A, a_dtype, Bp, T, C, c_dtype, ws, wsb)
    assert qg.qgemm_status() == 0
    tail = flat[M * N:]
    assert torch.isnan(tail).all(), "write past the end of C"
    if ws is not None:
        assert (ws[wsb:] == 0xA5).all(), "write past the end of the workspace"
    return to_numpy_values(C, c_dtype)


def layer_case(M, K, N, mode, block, a_dtype, c_dtype, a_seed=1, w_seed=2, W=None):
    w = synth.Workload("t", M, K, N, mode, block, a_dtype, c_dtype, a_seed, w_seed)
    A_np = synth.make_activations(w)
    W_np = synth.make_weights(w) if W is None else W
    w_dtype = a_dtype if mode == 0 else 0
    ref = oracle.reference_layer(mode, block, A_np, a_dtype, W_np, w_dtype)
    Bp, T = gpu_pack(W_np, mode, block, w_dtype)
    if mode == 0:
        got_bp = Bp.cpu().numpy().view(ref["Bp"].dtype).reshape(ref["Bp"].shape)
    else:
        got_bp = Bp.cpu().numpy().reshape(ref["Bp"].shape)
    assert np.array_equal(got_bp, ref["Bp"]), "packed weights differ from the oracle"
    if mode != 0:
        assert np.array_equal(table_rows(T.cpu().numpy(), N, ref["T"].shape[1]), ref["T"]), "table differs from the oracle"
    got = gpu_run(M, K, N, mode, block, A_np, a_dtype, Bp, T, c_dtype)
    return check_close(got, ref["R"], a_dtype, c_dtype, f"M{M} K{K} N{N} mode{mode} b{block}")


FORMATS = [(1, 64), (1, 128), (2, 0), (2, 64), (0, 0)]


@pytest.mark.parametrize("mode,block", FORMATS)
@pytest.mark.parametrize("a_dtype", [synth.F16, synth.BF16])
@pytest.mark.parametrize("M,K,N", [(1, 64, 1), (3, 256, 31), (8, 512, 257), (9, 1024, 100), (16, 256, 48),
                                   (5, 4096, 80), (17, 192, 33)])
def test_decode_parity(mode, block, a_dtype, M, K, N):
    if block and K % block:
        pytest.skip("block does not divide K")
    layer_case(M, K, N, mode, block, a_dtype, a_dtype)


@pytest.mark.parametrize("c_dtype", [synth.F32, synth.F16, synth.BF16])
def test_decode_output_dtypes(c_dtype):
    layer_case(4, 1024, 300, 1, 64, synth.BF16, c_dtype)


@pytest.mark.parametrize("mode,block", FORMATS)
@pytest.mark.parametrize("M,K,N", [(4, 256, 512), (1, 128, 33), (13, 512, 65)])
def test_f32_activations(mode, block, M, K, N):
    if block and K % block:
        pytest.skip("block does not divide K")
    layer_case(M, K, N, mode, block, synth.F32, synth.F32)


def test_constant_groups_and_zero_rows():
    """Degenerate cases: blocks with hi == lo (scale 0) and all-zero activation rows."""
    K, N = 256, 40
    W = synth.make_weights(synth.Workload("t", 1, K, N, 1, 64, 1, 1, 0, 3))
    W[64:128, :7] = 0.25
    W[:, 9] = -1.5
    for mode, block in [(1, 64), (2, 0)]:
        layer_case(6, K, N, mode, block, synth.F16, synth.F16, W=W.copy())


# ---------------------------------------------------------------- the pages' workloads at full size
def test_int4_b64_f32_m4_k256_n512():
    w = synth.WORKLOADS["int4_b64_m4_k256_n512_f32"]
    err = layer_case(w.M, w.K, w.N, w.mode, w.block, w.a_dtype, w.c_dtype, w.a_seed, w.w_seed)
    assert err <= 1e-5


def test_int4_b64_decode_m1_k4096_n11008():
    w = synth.WORKLOADS["int4_b64_decode_m1_k4096_n11008_bf16"]
    layer_case(w.M, w.K, w.N, w.mode, w.block, w.a_dtype, w.c_dtype, w.a_seed, w.w_seed)


@pytest.mark.parametrize("M", synth.INT8_M_SWEEP)
def test_int8_b0_page_fill_m_sweep(M):
    w = synth.WORKLOADS["int8_b0_k4096_n4096_f16"]
    W = synth.make_weights(w)
    layer_case(M, w.K, w.N, w.mode, w.block, w.a_dtype, w.c_dtype, w.a_seed, w.w_seed, W=W)


@pytest.mark.parametrize("mode,block", [(1, 64), (2, 0), (0, 0)])
@pytest.mark.parametrize("M,N,K", [(6400, 32, 64), (1024, 128, 256)])
def test_page_gemm_check_shapes(mode, block, M, N, K):
    """The two shapes the Vulkan GEMM page checks against float64 (M x N x K)."""
    layer_case(M, K, N, mode, block, synth.F16, synth.F16)


def test_split_k_path_deterministic():
    """Small N splits K across thread blocks; two runs give identical bits."""
    M, K, N = 2, 4096, 64
    assert qg.qgemm_workspace_bytes(M, K, N, 1, 64, 2, 2) > 0
    layer_case(M, K, N, 1, 64, synth.BF16, synth.BF16)
    w = synth.Workload("t", M, K, N, 1, 64, 2, 2, 1, 2)
    A_np, W_np = synth.make_activations(w), synth.make_weights(w)
    Bp, T = gpu_pack(W_np, 1, 64)
    a = gpu_run(M, K, N, 1, 64, A_np, 2, Bp, T, 2)
    b = gpu_run(M, K, N, 1, 64, A_np, 2, Bp, T, 2)
    assert np.array_equal(a, b)


def test_pack_full_size_w4a8_weights():
    w = synth.WORKLOADS["w4a8_m2048_k4096_n14336"]
    W = synth.make_weights(w)
    q, T = oracle.quantize(W, w.K, 15)
    Bp, Tg = gpu_pack(W, 3, 0)
    assert np.array_equal(Bp.cpu().numpy().reshape(w.N, w.K // 2), oracle.pack(q, 4))
    assert np.array_equal(table_rows(Tg.cpu().numpy(), w.N, 1), T)


# ---------------------------------------------------------------- W4A8 activation step
@pytest.mark.parametrize("a_dtype", [synth.BF16, synth.F16, synth.F32])
def test_act_quant_bit_exact(a_dtype):
    M, K = 2048, 4096
    w = synth.Workload("t", M, K, 1, 3, 0, a_dtype, 2, 0, 0)
    A_np = synth.make_activations(w)
    A_np = A_np.copy()
    A_np[17] = 0                                           # a zero row: scale 0, codes 0
    # rows of tiny values (with zeros among them) whose scale max|a| / 127 is a subnormal float32,
    # where a reciprocal of the scale overflows; f16 cannot hold such values, so its tiny rows
    # sit at the bottom of its own range instead
    base = oracle.values(A_np[40], a_dtype)
    tiny_rows = ((33, 1e-38), (34, 2e-40)) if a_dtype != synth.F16 else ((33, 1e-6), (34, 2e-7))
    for row, tiny in tiny_rows:
        x = base * tiny
        x[::5] = 0.0
        A_np[row] = synth.encode(x, a_dtype)
    A32_rows = oracle.values(A_np, a_dtype).astype(np.float32)
    assert A32_rows[33].any() and A32_rows[34].any()
    if a_dtype != synth.F16:
        assert np.abs(A32_rows[33]).max() / np.float32(127) < np.finfo(np.float32).tiny
    qa_r, s_r, rs_r = oracle.act_quant(A32_rows)
    A = torch_from(A_np, a_dtype)
    qa = torch.empty((M, K), dtype=torch.int8, device=DEV)
    s = torch.empty(M, dtype=torch.float32, device=DEV)
    rs = torch.empty(M, dtype=torch.int32, device=DEV)
    qg.qgemm_act_quant(M, K, A, a_dtype, qa, s, rs)
    torch.cuda.synchronize()
    assert np.array_equal(qa.cpu().numpy(), qa_r)
    assert np.array_equal(s.cpu().numpy(), s_r)
    assert np.array_equal(rs.cpu().numpy(), rs_r)


def test_launch_overlap_chained_layers_bit_identical():
    """With QGEMM_OPT_LAUNCH_OVERLAP each decode call may start before the previous kernel ends;
    it must still read A (here: the previous layer's output) only after that kernel is done.
    Four chained layers (square, K = N) give identical bits with and without the option."""
    K = N = 2048
    layers = []
    for i in range(4):
        w = synth.Workload("t", 1, K, N, 1, 64, synth.BF16, synth.BF16, 1, 10 + i, w_std=0.04)
        layers.append(gpu_pack(synth.make_weights(w), 1, 64))
    A0 = torch_from(synth.make_activations(synth.Workload("t", 1, K, N, 1, 64, 2, 2, 3, 0)), synth.BF16)
    wsb = qg.qgemm_workspace_bytes(1, K, N, 1, 64, 2, 2)     # N = 2048 also exercises split-K
    assert wsb > 0
    ws = torch.empty(wsb, dtype=torch.uint8, device=DEV)

    def chain():
        x = A0
        outs = []
        for Bp, T in layers:
            y = torch.empty((1, N), dtype=torch.bfloat16, device=DEV)
            qg.qgemm_run(1, K, N, 1, 64, x, 2, Bp, T, y, 2, ws, wsb)
            outs.append(y)
            x = y
        torch.cuda.synchronize()
        return [o.float().cpu().numpy() for o in outs]

    prev = qg.qgemm_set_option(qg.OPT_LAUNCH_OVERLAP, 0)
    try:
        ref = chain()
        qg.qgemm_set_option(qg.OPT_LAUNCH_OVERLAP, 1)
        for _ in range(3):
            got = chain()
            for a, b in zip(ref, got):
                assert np.array_equal(a, b)
        # inside a CUDA graph as well
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            x = A0
            outs = []
            with torch.cuda.graph(g, stream=s):
                for Bp, T in layers:
                    y = torch.empty((1, N), dtype=torch.bfloat16, device=DEV)
                    qg.qgemm_run(1, K, N, 1, 64, x, 2, Bp, T, y, 2, ws, wsb, stream=s)
                    outs.append(y)
                    x = y
        g.replay()
        torch.cuda.synchronize()
        for a, o in zip(ref, outs):
            assert np.array_equal(a, o.float().cpu().numpy())
    finally:
        qg.qgemm_set_option(qg.OPT_LAUNCH_OVERLAP, prev)


# ---------------------------------------------------------------- packed-weight files
@pytest.mark.parametrize("mode,block,M", [(1, 64, 1), (2, 0, 40), (0, 0, 3)])
def test_weight_file_round_trip_on_device(tmp_path, mode, block, M):
    """qgemm_save from device buffers, qgemm_load into fresh ones: the same bytes, and the
    layer run on the loaded weights gives exactly the output of the original ones."""
    K, N = 512, 200
    w = synth.Workload("t", M, K, N, mode, block, synth.BF16, synth.BF16, 1, 2)
    A_np, W_np = synth.make_activations(w), synth.make_weights(w)
    w_dtype = synth.BF16 if mode == 0 else 0
    Bp, T = gpu_pack(W_np, mode, block, w_dtype)
    path = str(tmp_path / "layer.qgw")
    qg.qgemm_save(path, K, N, mode, block, w_dtype, Bp, T)
    info = qg.qgemm_load_info(path)
    assert info == {"K": K, "N": N, "mode": mode, "block": block, "w_dtype": w_dtype}
    Bp2 = torch.zeros_like(Bp)
    T2 = None if T is None else torch.zeros_like(T)
    qg.qgemm_load(path, Bp2, T2)
    torch.cuda.synchronize()
    assert torch.equal(Bp2, Bp) and (T is None or torch.equal(T2, T))
    got1 = gpu_run(M, K, N, mode, block, A_np, synth.BF16, Bp, T, synth.BF16)
    got2 = gpu_run(M, K, N, mode, block, A_np, synth.BF16, Bp2, T2, synth.BF16)
    assert np.array_equal(got1, got2)
