"""Pins for the CPU oracle: each test checks it against something other than itself.

The pages print no quantized worked example, so the pins are: the Int8-Block0 closed form of
the benchmark page's own weight fill, exact dyadic cases whose result is known by
construction and recomputed with Python/numpy integers, library routines for the special
cases that reduce to them (GEMV, float GEMM, bf16 rounding), and the invariants the
asymmetric scheme implies. Each is chosen so that a plausible slip in the oracle (a dropped
offset term, a wrong sign, a transposed operand, a wrong index order, truncation instead of
rounding) fails at least one of them.
"""
import os

import numpy as np
import pytest
import torch

import oracle
from weight_quantized_gemm_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _golden_rows(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]


# ------------------------------------------------------------------ Int8-Block0 closed form
def test_int8_block0_page_fill_closed_form():
    """Benchmark page «为什么用 Conv1x1 来测 GEMM»: fill ((i % 127) - 63)/1000 over the
    {ic, oc} = {K, N} weight, Int8-Block0. Every channel's table entry and every code is
    fixed by the fill formula alone (golden file written by exact rational arithmetic)."""
    K = N = 4096
    W = synth.mnn_fill(K, N)
    q, T = oracle.quantize(W, 0, 255)
    assert T.shape == (N, 1, 2)
    lo = np.float32(-63) / np.float32(1000)
    hi = np.float32(63) / np.float32(1000)
    assert np.all(T[:, 0, 0] == lo)                     # offset = channel minimum, same in every row
    # scale * 255 recovers hi - lo to within one float32 rounding of the division
    assert np.allclose(T[:, 0, 1].astype(np.float64) * 255, float(hi) - float(lo), rtol=2 ** -23, atol=0)
    allowed = {}
    for r, codes in _golden_rows("int8_block0_mnn_fill.txt"):
        allowed[int(r)] = [int(c) for c in codes.split("|")]
    k = np.arange(K, dtype=np.int64)[None, :]
    n = np.arange(N, dtype=np.int64)[:, None]
    resid = (k * N + n) % 127                           # flat index i = k*N + n of the [K][N] weight
    exact = np.array([allowed[r][0] for r in range(127)])
    alt = np.array([allowed[r][-1] for r in range(127)])
    ok = (q == exact[resid]) | (q == alt[resid])
    assert ok.all()
    # the three half-way residues are the only ones where neighbours are tolerated
    assert sum(len(v) > 1 for v in allowed.values()) == 3


# ------------------------------------------------------------------ exact dyadic cases
def _dyadic_case(M, K, N, block, qmax, rng, e=9, f=6):
    """Weights on the grid lo + j * 2^-e with both j = 0 and j = qmax in every block, so that
    quantization is exact (q = j, scale = 2^-e, offset = lo); activations are integers * 2^-f."""
    nb = K // block
    j = rng.integers(0, qmax + 1, size=(N, nb, block))
    j[:, :, 0] = 0
    j[:, :, 1] = qmax
    for n in range(N):                                   # shuffle the positions of the extremes
        for b in range(nb):
            rng.shuffle(j[n, b])
    L = rng.integers(-3 * qmax, 2 * qmax, size=(N, nb))  # lo = L * 2^-e
    W_int = (j + L[:, :, None]).reshape(N, K)            # W[k][n] * 2^e, transposed
    W = (W_int.T.astype(np.float64) * 2.0 ** -e).astype(np.float32)
    A_int = rng.integers(-40, 41, size=(M, K))
    A = A_int.astype(np.float64) * 2.0 ** -f
    return W, A, A_int, W_int, j.reshape(N, K), L


@pytest.mark.parametrize("M,N,K,block,qmax", [
    (3, 5, 64, 64, 15), (8, 7, 128, 64, 15), (4, 6, 128, 128, 255), (2, 3, 64, 64, 255),
])
def test_dyadic_exact_small(M, N, K, block, qmax):
    rng = np.random.default_rng(1234 + M * 7 + N)
    W, A, A_int, W_int, j, L = _dyadic_case(M, K, N, block, qmax, rng)
    q, T = oracle.quantize(W, block, qmax)
    assert np.array_equal(q, j)
    assert np.all(T[:, :, 1] == np.float32(2.0 ** -9))
    assert np.array_equal(T[:, :, 0], (L * 2.0 ** -9).astype(np.float32))
    R = oracle.gemm(A, oracle.dequant(q, T, block))
    # brute force in Python integers: R * 2^(e+f) = sum_k A_int[m][k] * W_int[n][k]
    for m in range(M):
        for n in range(N):
            s = sum(int(A_int[m, k]) * int(W_int[n, k]) for k in range(K))
            assert R[m, n] == s * 2.0 ** -15
    # and the point version agrees
    mi, ni = np.meshgrid(np.arange(M), np.arange(N), indexing="ij")
    P = oracle.gemm_points(A, q, T, block, mi.ravel(), ni.ravel())
    assert np.array_equal(P, R.ravel())


@pytest.mark.parametrize("M,N,K", [(6400, 32, 64), (1024, 128, 256)])
@pytest.mark.parametrize("block,qmax", [(64, 15), (0, 255)])
def test_dyadic_exact_page_gemm_shapes(M, N, K, block, qmax):
    """The two GEMM shapes the Vulkan GEMM page checks against float64 (M x N x K)."""
    shapes = {(int(a), int(b), int(c)) for a, b, c, _ in _golden_rows("gemm_check_shapes.txt")}
    assert (M, N, K) in shapes
    blk = K if block == 0 else block
    rng = np.random.default_rng(M + N + K + blk)
    W, A, A_int, W_int, j, L = _dyadic_case(M, K, N, blk, qmax, rng)
    q, T = oracle.quantize(W, blk, qmax)
    assert np.array_equal(q, j)
    R = oracle.gemm(A, oracle.dequant(q, T, blk))
    exact = (A_int.astype(np.int64) @ W_int.T.astype(np.int64)).astype(np.float64) * 2.0 ** -15
    assert np.array_equal(R, exact)


# ------------------------------------------------------------------ library special cases
def test_gemv_matches_numpy():
    """M = 1 reduces to a matrix-vector product (numpy float64 as the library routine)."""
    w = synth.Workload("t", 1, 512, 300, 1, 64, synth.BF16, synth.BF16, 3, 4)
    A = synth.make_activations(w)
    W = synth.make_weights(w)
    q, T = oracle.quantize(W, 64, 15)
    Bt = oracle.dequant(q, T, 64)
    a = oracle.values(A, synth.BF16)
    R = oracle.gemm(a, Bt)
    ref = Bt @ a[0]
    assert np.allclose(R[0], ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())


def test_float_gemm_matches_torch_f64():
    w = synth.Workload("t", 33, 256, 65, 0, 0, synth.F16, synth.F16, 5, 6)
    A = synth.make_activations(w)
    W = synth.make_weights(w)
    Wt = oracle.pack_float(W, synth.F16)
    R = oracle.gemm(oracle.values(A, synth.F16), oracle.values(Wt, synth.F16))
    ref = torch.from_numpy(A.astype(np.float64)) @ torch.from_numpy(Wt.astype(np.float64)).T
    assert np.allclose(R, ref.numpy(), rtol=1e-12, atol=1e-12)
    Pt = oracle.dense_points(oracle.values(A, synth.F16), oracle.values(Wt, synth.F16), [0, 32, 7], [0, 64, 9])
    assert np.allclose(Pt, R[[0, 32, 7], [0, 64, 9]], rtol=1e-14)


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(7)
    x = rng.standard_normal((37, 41)).astype(np.float32)
    # plant exact ties: low 16 bits = 0x8000, with both parities of bit 16
    u = x.view(np.uint32)
    u[::3] = (u[::3] & np.uint32(0xFFFF0000)) | np.uint32(0x8000)
    got = oracle.pack_float(x, synth.BF16)
    ref = torch.from_numpy(x.T.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, ref)
    got16 = oracle.pack_float(x, synth.F16)
    assert np.array_equal(got16, torch.from_numpy(x.T.copy()).to(torch.float16).numpy())


# ------------------------------------------------------------------ invariants of the scheme
@pytest.mark.parametrize("K,N,block,qmax", [(256, 512, 64, 15), (4096, 64, 0, 255), (512, 96, 128, 15)])
def test_quantize_invariants(K, N, block, qmax):
    w = synth.Workload("t", 1, K, N, 1, block, synth.F32, synth.F32, 0, 11)
    W = synth.make_weights(w)
    blk = K if block == 0 else block
    q, T = oracle.quantize(W, blk, qmax)
    nb = K // blk
    G = W.T.reshape(N, nb, blk)                      # groups of the weight, channel-major
    Q = q.reshape(N, nb, blk)
    assert q.max() <= qmax
    assert np.array_equal(T[:, :, 0], G.min(axis=2))                       # offset = group min
    # the min element codes 0 and the max element codes qmax
    assert np.all(np.take_along_axis(Q, G.argmin(axis=2)[..., None], 2) == 0)
    assert np.all(np.take_along_axis(Q, G.argmax(axis=2)[..., None], 2) == qmax)
    s = T[:, :, 1].astype(np.float64)
    rng_ = G.max(axis=2).astype(np.float64) - G.min(axis=2).astype(np.float64)
    assert np.allclose(s * qmax, rng_, rtol=2 ** -22, atol=0)
    recon = Q * s[..., None] + T[:, :, 0:1].astype(np.float64)
    err = np.abs(recon - G.astype(np.float64))
    bound = s[..., None] / 2 * (1 + 2 ** -20) + 4 * np.finfo(np.float32).eps * (np.abs(G) + np.abs(T[:, :, 0:1]))
    assert np.all(err <= bound)


def test_constant_group_reconstructs_exactly():
    W = np.full((128, 3), 0.125, dtype=np.float32)
    W[64:, 1] = -2.5
    q, T = oracle.quantize(W, 64, 15)
    assert np.all(q == 0)
    assert np.all(T[:, :, 1] == 0)
    Bt = oracle.dequant(q, T, 64)
    assert np.array_equal(Bt, W.T.astype(np.float64))


def test_pack_nibble_order_and_roundtrip():
    K = 64
    q = (np.arange(K) % 16).astype(np.uint8)[None, :].repeat(3, 0)
    Bp = oracle.pack(q, 4)
    assert list(Bp[0, :8]) == [0x10, 0x32, 0x54, 0x76, 0x98, 0xBA, 0xDC, 0xFE]
    rng = np.random.default_rng(3)
    r = rng.integers(0, 16, size=(5, 96)).astype(np.uint8)
    assert np.array_equal(oracle.unpack(oracle.pack(r, 4), 96, 4), r)
    r8 = rng.integers(0, 256, size=(5, 96)).astype(np.uint8)
    assert np.array_equal(oracle.pack(r8, 8), r8)


# ------------------------------------------------------------------ W4A8
def test_act_quant_invariants():
    w = synth.Workload("t", 37, 320, 1, 3, 0, synth.BF16, synth.BF16, 9, 0)
    A = oracle.values(synth.make_activations(w), synth.BF16).astype(np.float32)
    A[5] = 0.0                                           # an all-zero row quantizes to zeros
    qa, s, rs = oracle.act_quant(A)
    assert np.abs(qa.astype(np.int32)).max() <= 127
    assert s[5] == 0 and np.all(qa[5] == 0) and rs[5] == 0
    amax = np.abs(A).max(axis=1)
    assert np.allclose(s.astype(np.float64) * 127, amax, rtol=2 ** -23)
    idx = np.abs(A).argmax(axis=1)
    hit = qa[np.arange(37), idx].astype(np.int32)
    assert np.all(np.abs(hit[np.arange(37) != 5]) == 127)
    assert np.array_equal(rs, qa.astype(np.int64).sum(axis=1))
    err = np.abs(qa * s[:, None].astype(np.float64) - A)
    # half a step, plus the float32 rounding of the quotient a / as (|a / as| <= 127)
    assert np.all(err <= s[:, None].astype(np.float64) * (0.5 + 128 * 2.0 ** -23))


def test_w4a8_exact_grid_equals_float_gemm():
    """Activations on the grid j * 2^-e with row max 127 * 2^-e quantize exactly, so the W4A8
    rescale must equal the float GEMM of the same (dequantized) weights; the int32
    accumulators are checked against numpy int64 arithmetic."""
    rng = np.random.default_rng(21)
    M, K, N = 9, 256, 13
    A_int = rng.integers(-127, 128, size=(M, K))
    A_int[:, 0] = 127 * np.where(rng.random(M) < 0.5, -1, 1)
    A = (A_int * 2.0 ** -7).astype(np.float32)
    W = synth.normal64(K * N, 5, 2, 0.02).astype(np.float32).reshape(K, N)
    q, T = oracle.quantize(W, K, 15)
    qa, s, rs = oracle.act_quant(A)
    assert np.array_equal(qa.astype(np.int64), A_int)
    assert np.all(s == np.float32(2.0 ** -7))
    acc = oracle.w4a8_acc(qa, q)
    assert np.array_equal(acc.astype(np.int64), A_int.astype(np.int64) @ q.T.astype(np.int64))
    R = oracle.w4a8_out(acc, s, rs, T)
    ref = oracle.gemm(A.astype(np.float64), oracle.dequant(q, T, K))
    assert np.allclose(R, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())
    pts = oracle.w4a8_acc_points(qa, q, [0, 8, 3], [12, 0, 5])
    assert np.array_equal(pts, acc[[0, 8, 3], [12, 0, 5]])


def test_w4a8_block_weights_pins():
    """W4A8 with block-64 weights: on the exact activation grid the block rescale equals the float
    GEMM of the dequantized block weights (a wrong block index, scale, offset or row sum fails
    it); with one block over K it is the per-channel rescale exactly; a 2-row brute force in
    Python integers checks the block sums."""
    rng = np.random.default_rng(33)
    M, K, N, blk = 7, 256, 11, 64
    A_int = rng.integers(-127, 128, size=(M, K))
    A_int[:, 5] = 127
    A = (A_int * 2.0 ** -6).astype(np.float32)
    W = synth.normal64(K * N, 8, 2, 0.02).astype(np.float32).reshape(K, N)
    q, T = oracle.quantize(W, blk, 15)
    qa, s, rs = oracle.act_quant(A)
    assert np.array_equal(qa.astype(np.int64), A_int) and np.all(s == np.float32(2.0 ** -6))
    R = oracle.w4a8_block_out(qa, s, q, T, blk)
    ref = oracle.gemm(A.astype(np.float64), oracle.dequant(q, T, blk))
    assert np.allclose(R, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())
    qK, TK = oracle.quantize(W, K, 15)
    acc = oracle.w4a8_acc(qa, qK)
    assert np.array_equal(oracle.w4a8_block_out(qa, s, qK, TK, K), oracle.w4a8_out(acc, s, rs, TK))
    for m, n in [(0, 0), (6, 10)]:
        tot = 0.0
        for b in range(K // blk):
            ks = range(b * blk, (b + 1) * blk)
            a_q = sum(int(qa[m, k]) * int(q[n, k]) for k in ks)
            r_s = sum(int(qa[m, k]) for k in ks)
            tot += float(T[n, b, 1]) * a_q + float(T[n, b, 0]) * r_s
        assert abs(R[m, n] - float(s[m]) * tot) <= 1e-12 * max(1.0, abs(R[m, n]))


def test_reference_layer_modes_consistent():
    """The whole-layer helper wires the steps in the order the pages give."""
    for mode, block in [(1, 64), (2, 0), (3, 0), (3, 64)]:
        w = synth.Workload("t", 5, 128, 24, mode, block, synth.BF16, synth.BF16, 1, 2)
        A = synth.make_activations(w)
        W = synth.make_weights(w)
        out = oracle.reference_layer(mode, block, A, synth.BF16, W)
        assert out["R"].shape == (5, 24)
        assert out["Bp"].shape == (24, 128 * oracle.NBITS[mode] // 8)


# ------------------------------------------------------------------ flop convention
def test_flop_convention_reproduces_page():
    """Benchmark page «测量流程» / «输出格式解读»: GFLOPS = 2*M*K*N / (ms * 1e6)."""
    for label, M, K, N, ms, g in _golden_rows("mnn_gemmspeed_printed.txt"):
        w = synth.Workload(label, int(M), int(K), int(N), 0, 0, 0, 0, 0, 0)
        # the printed ms is rounded to 3 decimals: the printed GFLOPS must lie in the range
        # that the unrounded time allows (plus the 2-decimal rounding of the GFLOPS itself)
        lo = w.flops / ((float(ms) + 5e-4) * 1e6) - 0.005
        hi = w.flops / ((float(ms) - 5e-4) * 1e6) + 0.005
        assert lo <= float(g) <= hi, (label, lo, g, hi)
        # a different convention (1*M*K*N, or 1e9 in place of 1e6 per ms) misses by 2x / 1000x
        assert not (lo <= 2 * float(g) <= hi)


# ------------------------------------------------------------------ output epilogue
def test_epilogue_pins():
    """act(R + bias) + residual (Adreno 750 pull request: accumulators kept until bias, residual
    and activation). Each activation against an independent routine or identity, bias and
    residual as exact adds, and the reading of the order (activation before the residual)."""
    sp = pytest.importorskip("scipy.special")
    rng = np.random.default_rng(7)
    R = rng.normal(0.0, 3.0, (9, 33))
    bias = rng.normal(0.0, 1.0, 33).astype(np.float32)
    res = rng.normal(0.0, 1.0, (9, 33))
    x = R + bias.astype(np.float64)
    assert np.array_equal(oracle.epilogue(R), R)
    assert np.array_equal(oracle.epilogue(R, bias, oracle.ACT_NONE, res), x + res)
    assert np.array_equal(oracle.epilogue(R, bias, oracle.ACT_RELU), np.maximum(x, 0.0))
    # SiLU against scipy's logistic function
    np.testing.assert_allclose(oracle.epilogue(R, bias, oracle.ACT_SILU), x * sp.expit(x), rtol=1e-14, atol=1e-300)
    # tanh-form GELU: g(x) - g(-x) = x exactly (the tanh part is odd), g(0) = 0, and within the
    # form's known 4.8e-4 of the exact x * Phi(x); a wrong constant (0.04 for 0.044715,
    # sqrt(pi/2) or 2/pi for sqrt(2/pi)) or a dropped cube misses that bound by 6x or more
    t = np.linspace(-8.0, 8.0, 4001).reshape(1, -1)
    g = oracle.epilogue(t, None, oracle.ACT_GELU_TANH)
    gm = oracle.epilogue(-t, None, oracle.ACT_GELU_TANH)
    np.testing.assert_allclose(g - gm, t, rtol=0, atol=1e-13)
    assert oracle.epilogue(np.zeros((1, 1)), None, oracle.ACT_GELU_TANH)[0, 0] == 0.0
    assert np.abs(g - t * sp.ndtr(t)).max() < 5e-4
    # the order: ReLU(-2) + 5 = 5 (not ReLU(-2 + 5) = 3)
    assert oracle.epilogue(np.full((1, 1), -2.0), None, oracle.ACT_RELU, np.full((1, 1), 5.0))[0, 0] == 5.0
    with pytest.raises(ValueError):
        oracle.epilogue(R, None, 7)
