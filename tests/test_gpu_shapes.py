"""GPU parity beyond the five workloads, through the C ABI:

- the MNN GemmSpeed shape grid (benchmark page "MNN GemmSpeed 基准测试实战", «默认测试尺寸»):
  (K, N) in {(2560, 4096), (2560, 1024), (4096, 2560), (2560, 9728), (9728, 2560)} x
  M in {8, 32, 128, 512}, for Int4-Block64, Int8-Block0 and float weights, f16 activations and
  output (the page's fp16 precision), checked against the oracle at sampled outputs; M = 8 runs on
  the decode kernel, the rest on the tensor-core kernel;
- the N partition: output channels split into shards, each packed and run on its own, give the
  unsharded result bit for bit (the way a multi-GPU run would split the layer, with no exchange).
"""
import functools

import numpy as np
import pytest
import torch

import oracle
import weight_quantized_gemm_gb300 as qg
from weight_quantized_gemm_gb300 import synth
from tests._util import check_close, ensure_built
from tests.test_gpu_decode import gpu_pack, gpu_run

pytestmark = pytest.mark.gpu

MNN_KN = [(2560, 4096), (2560, 1024), (4096, 2560), (2560, 9728), (9728, 2560)]
MNN_M = [8, 32, 128, 512]
FORMATS = [(synth.MODE_INT4, 64), (synth.MODE_INT8, 0), (synth.MODE_FLOAT, 0)]


@pytest.fixture(scope="module", autouse=True)
def built():
    ensure_built()


@functools.lru_cache(maxsize=2)
def _weights(K: int, N: int) -> np.ndarray:
    return synth.make_weights(synth.Workload("grid", 1, K, N, synth.MODE_INT4, 64, synth.F16, synth.F16, 0, 11))


@functools.lru_cache(maxsize=4)
def _packed(K: int, N: int, mode: int, block: int):
    """GPU-packed weights plus what the oracle needs for sampled outputs."""
    W = _weights(K, N)
    if mode == synth.MODE_FLOAT:
        Bp, T = gpu_pack(W, mode, 0, synth.F16)
        return Bp, T, ("dense", oracle.values(oracle.pack_float(W, synth.F16), synth.F16))
    Bp, T = gpu_pack(W, mode, block)
    q, Tq = oracle.quantize(W, K if block == 0 else block, oracle.QMAX[mode])
    return Bp, T, ("quant", q, Tq)


@pytest.mark.parametrize("K,N", MNN_KN, ids=lambda v: str(v))
@pytest.mark.parametrize("mode,block", FORMATS, ids=["int4_b64", "int8_b0", "float"])
@pytest.mark.parametrize("M", MNN_M)
def test_mnn_shape_grid(K, N, mode, block, M):
    w = synth.Workload("grid", M, K, N, mode, block, synth.F16, synth.F16, 5, 11)
    A_np = synth.make_activations(w)
    Bp, T, ref = _packed(K, N, mode, block)
    got = gpu_run(M, K, N, mode, block, A_np, synth.F16, Bp, T, synth.F16)
    rng = np.random.default_rng(K * 7 + N + M)
    npts = 512
    mi, ni = rng.integers(0, M, npts), rng.integers(0, N, npts)
    mi[:2], ni[:2] = [0, M - 1], [0, N - 1]
    A64 = oracle.values(A_np, synth.F16)
    if ref[0] == "dense":
        R = oracle.dense_points(A64, ref[1], mi, ni)
    else:
        R = oracle.gemm_points(A64, ref[1], ref[2], K if block == 0 else block, mi, ni)
    check_close(got[mi, ni], R, synth.F16, synth.F16, f"M{M} K{K} N{N} mode{mode}")


@pytest.mark.parametrize("M,K,N,mode,block,a_dtype", [
    (1, 4096, 11008, synth.MODE_INT4, 64, synth.BF16),     # decode (TMA-fed kernel)
    (4, 4096, 8192, synth.MODE_INT8, 0, synth.F16),        # decode, per-channel table
    (12, 4096, 8192, synth.MODE_INT4, 64, synth.BF16),     # decode, 9 <= M <= 16 (split K, same factor)
    (256, 2048, 4096, synth.MODE_INT4, 64, synth.F16),     # tensor-core prefill
    (64, 1024, 2048, synth.MODE_W4A8, 0, synth.BF16),      # W4A8
], ids=["decode_m1", "decode_int8_m4", "decode_m12", "prefill", "w4a8"])
def test_n_shards_reassemble_bit_exact(M, K, N, mode, block, a_dtype):
    w = synth.Workload("shard", M, K, N, mode, block, a_dtype, a_dtype, 21, 22)
    A_np = synth.make_activations(w)
    W = synth.make_weights(w)
    Bp, T = gpu_pack(W, mode, block)
    full = gpu_run(M, K, N, mode, block, A_np, a_dtype, Bp, T, a_dtype)
    # shard boundaries on 16-channel groups (the table's grouping); the shapes keep each shard's
    # decode K-split factor equal to the unsharded one, so the summation order is the same
    cuts = [0, N // 2 - (N // 2) % 16, N]
    parts = []
    for n0, n1 in zip(cuts[:-1], cuts[1:]):
        Bs, Ts = gpu_pack(np.ascontiguousarray(W[:, n0:n1]), mode, block)
        parts.append(gpu_run(M, K, n1 - n0, mode, block, A_np, a_dtype, Bs, Ts, a_dtype))
    assert np.array_equal(np.concatenate(parts, axis=1), full)
