"""GPU parity of the tensor-core (tcgen05) path against the CPU oracle, through the C ABI:
prefill for M > 16 with 16-bit activations in every weight format, and W4A8 (int32
accumulators bit-exact, rescaled output within the bar)."""
import numpy as np
import pytest
import torch

import oracle
import weight_quantized_gemm_gb300 as qg
from weight_quantized_gemm_gb300 import synth
from tests._util import check_close, ensure_built, table_rows, to_numpy_values, torch_dtype, torch_from
from tests.test_gpu_decode import gpu_pack, gpu_run, layer_case

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def built():
    ensure_built()


# ---------------------------------------------------------------- prefill
@pytest.mark.parametrize("mode,block", [(1, 64), (1, 128), (2, 0), (2, 64), (0, 0)])
@pytest.mark.parametrize("a_dtype", [synth.F16, synth.BF16])
@pytest.mark.parametrize("M,K,N", [(17, 64, 1), (64, 256, 128), (100, 512, 257), (256, 192, 130), (300, 1024, 96)])
def test_prefill_parity(mode, block, a_dtype, M, K, N):
    if block and K % block:
        pytest.skip("block does not divide K")
    layer_case(M, K, N, mode, block, a_dtype, a_dtype)


@pytest.mark.parametrize("c_dtype", [synth.F32, synth.F16, synth.BF16])
def test_prefill_output_dtypes(c_dtype):
    layer_case(130, 512, 200, 1, 64, synth.F16, c_dtype)


# ---------------------------------------------------------------- split-K (mid-sized M)
# Shapes with fewer 128-channel x BN-row tiles than SMs split K across blocks: each split adds its
# stages into float32 partial sums, a second kernel adds the splits in order and rounds once.
@pytest.mark.parametrize("M,K,N,mode,block,a_dtype,splits", [
    (40, 1088, 130, 1, 64, synth.F16, 2),      # splits of 8 and 9 stages; rows not 16-byte multiples
    (64, 2560, 4096, 1, 64, synth.F16, 4),     # partials stored by TMA
    (96, 1600, 1000, 2, 0, synth.BF16, 3),     # uneven splits (8, 8, 9), per-channel int8
    (48, 2048, 384, 1, 128, synth.BF16, 4),    # bf16 hi/lo weight parts, K-blocks across splits
    (33, 1024, 256, 0, 0, synth.BF16, 2),      # float mode
    (256, 2048, 256, 2, 0, synth.BF16, 4),     # Int8-Block0 codes path: the offset term in split 0 only
])
def test_prefill_split_k(M, K, N, mode, block, a_dtype, splits):
    # Int8-Block0 row sums (the codes path: bf16, M >= 256)
    rows = -(-M * 4 // 256) * 256 if (mode == 2 and block == 0 and a_dtype == synth.BF16 and M >= 256) else 0
    assert qg.qgemm_workspace_bytes(M, K, N, mode, block, a_dtype, a_dtype) == rows + splits * M * N * 4
    layer_case(M, K, N, mode, block, a_dtype, a_dtype)


def test_prefill_split_k_less_workspace():
    """Less scratch than asked for: fewer splits (3 of 5, then none), each result within the bar."""
    M, K, N, mode, block = 64, 2560, 512, 1, 64
    w = synth.Workload("t", M, K, N, mode, block, synth.F16, synth.F16, 3, 4)
    A_np, W_np = synth.make_activations(w), synth.make_weights(w)
    ref = oracle.reference_layer(mode, block, A_np, synth.F16, W_np, 0)
    Bp, T = gpu_pack(W_np, mode, block)
    full = qg.qgemm_workspace_bytes(M, K, N, mode, block, synth.F16, synth.F16)
    assert full == 5 * M * N * 4
    for wsb in (full, 3 * M * N * 4 + 100, M * N * 4 + 4, 0):
        got = gpu_run(M, K, N, mode, block, A_np, synth.F16, Bp, T, synth.F16, ws_bytes=wsb)
        check_close(got, ref["R"], synth.F16, synth.F16, f"workspace {wsb}")
    prev = qg.qgemm_set_option(qg.OPT_SPLIT_K, 0)
    try:
        got = gpu_run(M, K, N, mode, block, A_np, synth.F16, Bp, T, synth.F16)
        check_close(got, ref["R"], synth.F16, synth.F16, "split-K off")
    finally:
        qg.qgemm_set_option(qg.OPT_SPLIT_K, prev)


def _sampled_case(w: synth.Workload, npts: int = 4096, seed: int = 0):
    """Full-size layer on the GPU, checked at sampled (m, n) points against the oracle."""
    A_np = synth.make_activations(w)
    W_np = synth.make_weights(w)
    blk = w.K if w.block == 0 else w.block
    q, T = oracle.quantize(W_np, blk, oracle.QMAX[w.mode])
    Bp, Tg = gpu_pack(W_np, w.mode, w.block)
    assert np.array_equal(Bp.cpu().numpy().reshape(w.N, -1), oracle.pack(q, oracle.NBITS[w.mode]))
    assert np.array_equal(table_rows(Tg.cpu().numpy(), w.N, T.shape[1]), T)
    got = gpu_run(w.M, w.K, w.N, w.mode, w.block, A_np, w.a_dtype, Bp, Tg, w.c_dtype)
    rng = np.random.default_rng(seed)
    mi = rng.integers(0, w.M, npts)
    ni = rng.integers(0, w.N, npts)
    mi[:4] = [0, w.M - 1, 0, w.M - 1]
    ni[:4] = [0, w.N - 1, w.N - 1, 0]
    R = oracle.gemm_points(oracle.values(A_np, w.a_dtype), q, T, blk, mi, ni)
    return check_close(got[mi, ni], R, w.a_dtype, w.c_dtype, w.name)


def test_int4_b64_prefill_m1024_k4096_n4096():
    _sampled_case(synth.WORKLOADS["int4_b64_prefill_m1024_k4096_n4096"])


def test_float_f16_gemm_full_size_sampled():
    w = synth.WORKLOADS["float_f16_m2048_k4096_n14336"]
    A_np = synth.make_activations(w)
    W_np = synth.make_weights(w)
    Bp, _ = gpu_pack(W_np, 0, 0, synth.F16)
    got = gpu_run(w.M, w.K, w.N, 0, 0, A_np, w.a_dtype, Bp, None, w.c_dtype)
    Wt = oracle.pack_float(W_np, synth.F16)
    assert np.array_equal(Bp.cpu().numpy().view(np.float16).reshape(w.N, w.K), Wt)
    rng = np.random.default_rng(1)
    mi, ni = rng.integers(0, w.M, 2048), rng.integers(0, w.N, 2048)
    R = oracle.dense_points(oracle.values(A_np, w.a_dtype), oracle.values(Wt, synth.F16), mi, ni)
    check_close(got[mi, ni], R, w.a_dtype, w.c_dtype, w.name)


# ---------------------------------------------------------------- W4A8
def _w4a8_inputs(M, K, N, a_dtype=synth.BF16, seed=0):
    w = synth.Workload("t", M, K, N, synth.MODE_W4A8, 0, a_dtype, synth.BF16, seed, seed + 1)
    return w, synth.make_activations(w), synth.make_weights(w)


def _gpu_w4a8_acc(qa_np, Bp, M, K, N):
    qa = torch.from_numpy(qa_np).to(DEV)
    acc = torch.full((M, N), -7, dtype=torch.int32, device=DEV)
    wsb = qg.qgemm_w4a8_acc_workspace_bytes(M, K)
    ws = torch.empty(wsb, dtype=torch.uint8, device=DEV)
    qg.qgemm_w4a8_acc(M, K, N, qa, Bp, acc, ws, wsb)
    assert qg.qgemm_status() == 0
    return acc.cpu().numpy()


@pytest.mark.parametrize("M,K,N", [(1, 64, 8), (17, 256, 33), (200, 1024, 300), (64, 4096, 128)])
def test_w4a8_acc_bit_exact(M, K, N):
    w, A_np, W_np = _w4a8_inputs(M, K, N)
    q, T = oracle.quantize(W_np, K, 15)
    qa, s, rs = oracle.act_quant(oracle.values(A_np, w.a_dtype).astype(np.float32))
    Bp, _ = gpu_pack(W_np, 3, 0)
    acc = _gpu_w4a8_acc(qa, Bp, M, K, N)
    assert np.array_equal(acc, oracle.w4a8_acc(qa, q))


def test_w4a8_acc_extreme_codes_exact():
    """Largest magnitudes the format allows: |qa| = 127 and q = 15 on every k (acc = +-127*15*K)."""
    M, K, N = 4, 4096, 16
    qa = np.full((M, K), 127, dtype=np.int8)
    qa[1] = -127
    qa[2, ::2] = -127
    qa[3] = np.where(np.arange(K) % 3 == 0, 127, -1).astype(np.int8)
    W = np.zeros((K, N), dtype=np.float32)
    W[0, :] = -1.0
    W[1:, :] = 1.0                               # codes: 0 at k = 0, 15 elsewhere
    q, _ = oracle.quantize(W, K, 15)
    Bp, _ = gpu_pack(W, 3, 0)
    acc = _gpu_w4a8_acc(qa, Bp, M, K, N)
    assert np.array_equal(acc, oracle.w4a8_acc(qa, q))


@pytest.mark.parametrize("K,N", [(8832, 40), (16448, 40), (8832, 42)])
def test_w4a8_acc_extreme_codes_long_k_exact(K, N):
    """K past 8808: the extreme sums 127 * 15 * K exceed 2^24, so one float32 accumulation would
    round them; the library runs K-chunks that are each exact and adds them in int32 (N = 42:
    rows that are no whole number of 16-byte units, added element by element)."""
    M = 5
    qa = np.full((M, K), 127, dtype=np.int8)
    qa[1] = -127
    qa[2, ::2] = -127
    qa[3] = np.where(np.arange(K) % 3 == 0, 127, -1).astype(np.int8)
    qa[4] = np.where(np.arange(K) % 7 == 0, -127, 126).astype(np.int8)
    W = np.ones((K, N), dtype=np.float32)
    W[0, :] = -1.0                               # codes: 0 at k = 0, 15 elsewhere
    W[1, ::3] = -1.0
    q, _ = oracle.quantize(W, K, 15)
    Bp, _ = gpu_pack(W, 3, 0)
    ref = oracle.w4a8_acc(qa, q)
    assert np.abs(ref).max() > 2 ** 24
    acc = _gpu_w4a8_acc(qa, Bp, M, K, N)
    assert np.array_equal(acc, ref)
    acc = _gpu_w4a8_acc(qa, Bp, M, K, N)         # twice: the chunks add into a cleared array
    assert np.array_equal(acc, ref)


@pytest.mark.parametrize("M,K,N", [(3, 8832, 40), (130, 8832, 136)])
@pytest.mark.parametrize("a_dtype", [synth.BF16, synth.F32])
def test_w4a8_layer_long_k(M, K, N, a_dtype):
    """The W4A8 layer with K past the exact range of one float32 accumulation (int32 K-chunks,
    then the rescale): against the oracle's integer path."""
    w, A_np, W_np = _w4a8_inputs(M, K, N, a_dtype)
    ref = oracle.reference_layer(3, 0, A_np, a_dtype, W_np)
    Bp, T = gpu_pack(W_np, 3, 0)
    got = gpu_run(M, K, N, 3, 0, A_np, a_dtype, Bp, T, synth.BF16)
    check_close(got, ref["R"], a_dtype if a_dtype != synth.F32 else synth.BF16, synth.BF16, "w4a8 long K")


@pytest.mark.parametrize("M,K,N", [(1, 128, 40), (33, 512, 100), (300, 1024, 257)])
@pytest.mark.parametrize("a_dtype", [synth.BF16, synth.F16, synth.F32])
def test_w4a8_layer(M, K, N, a_dtype):
    w, A_np, W_np = _w4a8_inputs(M, K, N, a_dtype)
    ref = oracle.reference_layer(3, 0, A_np, a_dtype, W_np)
    Bp, T = gpu_pack(W_np, 3, 0)
    got = gpu_run(M, K, N, 3, 0, A_np, a_dtype, Bp, T, synth.BF16)
    check_close(got, ref["R"], a_dtype if a_dtype != synth.F32 else synth.BF16, synth.BF16, "w4a8")


def test_w4a8_m2048_k4096_n14336_sampled():
    w = synth.WORKLOADS["w4a8_m2048_k4096_n14336"]
    A_np = synth.make_activations(w)
    W_np = synth.make_weights(w)
    q, T = oracle.quantize(W_np, w.K, 15)
    qa, s, rs = oracle.act_quant(oracle.values(A_np, w.a_dtype).astype(np.float32))
    Bp, Tg = gpu_pack(W_np, 3, 0)
    # int32 accumulators: bit-exact at sampled points
    acc = _gpu_w4a8_acc(qa, Bp, w.M, w.K, w.N)
    rng = np.random.default_rng(2)
    mi, ni = rng.integers(0, w.M, 4096), rng.integers(0, w.N, 4096)
    acc_ref = oracle.w4a8_acc_points(qa, q, mi, ni)
    assert np.array_equal(acc[mi, ni], acc_ref)
    # the layer: every output of 24 sampled rows, expected values from the oracle's own integer
    # GEMM and rescale
    got = gpu_run(w.M, w.K, w.N, 3, 0, A_np, w.a_dtype, Bp, Tg, w.c_dtype)
    rows = np.sort(rng.choice(w.M, 24, replace=False))
    acc_rows = oracle.w4a8_acc(qa[rows], q)
    assert np.array_equal(acc[rows], acc_rows)
    R = oracle.w4a8_out(acc_rows, s[rows], rs[rows], T)
    check_close(got[rows], R, w.a_dtype, w.c_dtype, w.name)


@pytest.mark.parametrize("M,K,N,block", [(1, 256, 40, 64), (40, 512, 96, 64), (300, 1024, 130, 128), (64, 2048, 256, 64)])
@pytest.mark.parametrize("a_dtype", [synth.BF16, synth.F16])
def test_w4a8_block_weights_layer(M, K, N, block, a_dtype):
    """W4A8 with block-quantized weights against the oracle's per-block integer rescale."""
    w, A_np, W_np = _w4a8_inputs(M, K, N, a_dtype)
    ref = oracle.reference_layer(3, block, A_np, a_dtype, W_np)
    Bp, T = gpu_pack(W_np, 3, block)
    assert np.array_equal(Bp.cpu().numpy().reshape(N, -1), ref["Bp"])
    assert np.array_equal(table_rows(T.cpu().numpy(), N, K // block), ref["T"])
    got = gpu_run(M, K, N, 3, block, A_np, a_dtype, Bp, T, synth.BF16)
    check_close(got, ref["R"], a_dtype, synth.BF16, f"w4a8 block {block}")


# ---------------------------------------------------------------- persistent tiles
# Blocks that run several tiles stage each output tile in ring slots that the pipeline reserves
# after the tile's last stage. These cases run more tiles than the GPU has SMs, with a short wait
# bound so that a pipeline that stalls fails within seconds instead of running out every wait.
@pytest.fixture
def short_waits():
    prev = qg.qgemm_set_option(qg.OPT_WAIT_LIMIT_US, 200000)
    yield
    qg.qgemm_set_option(qg.OPT_WAIT_LIMIT_US, prev)
    assert qg.qgemm_status() == 0


def test_w4a8_long_k_many_tiles_exact(short_waits):
    """The down-projection of the FFN pair, 2048 x 14336 -> 4096: int32 accumulator tiles (two
    K-chunks added in int32) staged over two of the ring's three slots, 256 tiles on at most one
    block per SM. Bit-exact at sampled points and on whole sampled rows."""
    M, K, N = 2048, 14336, 4096
    w, A_np, W_np = _w4a8_inputs(M, K, N, seed=5)
    q, T = oracle.quantize(W_np, K, 15)
    qa, s, rs = oracle.act_quant(oracle.values(A_np, w.a_dtype).astype(np.float32))
    Bp, Tg = gpu_pack(W_np, 3, 0)
    acc = _gpu_w4a8_acc(qa, Bp, M, K, N)
    rng = np.random.default_rng(7)
    mi, ni = rng.integers(0, M, 4096), rng.integers(0, N, 4096)
    assert np.array_equal(acc[mi, ni], oracle.w4a8_acc_points(qa, q, mi, ni))
    rows = np.sort(rng.choice(M, 8, replace=False))
    acc_rows = oracle.w4a8_acc(qa[rows], q)
    assert np.array_equal(acc[rows], acc_rows)
    got = gpu_run(M, K, N, 3, 0, A_np, w.a_dtype, Bp, Tg, synth.BF16)
    assert qg.qgemm_status() == 0
    check_close(got[rows], oracle.w4a8_out(acc_rows, s[rows], rs[rows], T), w.a_dtype, synth.BF16, "w4a8 long K")


@pytest.mark.parametrize("M,K,N,block,a_dtype", [
    (2048, 4096, 14336, 0, synth.BF16),    # W4A8, 896 tiles of 256 rows
    (1536, 1024, 2560, 64, synth.F16),     # Int4 prefill, 120 tiles: fewer than the SMs
    (4096, 512, 4096, 64, synth.F16),      # Int4 prefill, short K (4 stages) over 512 tiles
])
def test_fused_epilogue_many_tiles(short_waits, M, K, N, block, a_dtype):
    """Bias, activation and a residual tile brought in by TMA where the output is staged, on
    blocks that run several tiles (rows sampled against the oracle)."""
    mode = 3 if block == 0 else 1
    w = synth.Workload("t", M, K, N, mode, block, a_dtype, synth.BF16, 11, 12)
    A_np, W_np = synth.make_activations(w), synth.make_weights(w)
    bias_np = synth.normal64(N, 13, stream=4, std=0.5).astype(np.float32)
    res_np = synth.encode(synth.normal64(M * N, 14, stream=5).reshape(M, N), synth.BF16)
    Bp, T = gpu_pack(W_np, mode, block)
    A = torch_from(A_np, a_dtype)
    C = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=DEV)
    res = torch_from(res_np, synth.BF16)
    bias = torch.from_numpy(bias_np).to(DEV)
    wsb = qg.qgemm_workspace_bytes(M, K, N, mode, block, a_dtype, synth.BF16)
    ws = torch.empty(max(wsb, 16), dtype=torch.uint8, device=DEV)
    prev = qg.qgemm_set_option(qg.OPT_SPLIT_K, 0)
    try:
        qg.qgemm_run_fused(M, K, N, mode, block, A, a_dtype, Bp, T, bias, qg.ACT_SILU, res, C, synth.BF16, ws, wsb)
        assert qg.qgemm_status() == 0
    finally:
        qg.qgemm_set_option(qg.OPT_SPLIT_K, prev)
    rows = np.sort(np.random.default_rng(3).choice(M, 6, replace=False))
    got = to_numpy_values(C, synth.BF16)[rows]
    assert np.all(np.isfinite(got))
    ref = oracle.reference_layer(mode, block, A_np[rows], a_dtype, W_np)
    R = oracle.epilogue(ref["R"], bias_np, qg.ACT_SILU, oracle.values(res_np, synth.BF16)[rows])
    check_close(got, R, a_dtype, synth.BF16, f"fused many tiles mode {mode}")
