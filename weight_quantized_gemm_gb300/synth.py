"""Seeded synthetic inputs for the weight-quantized linear layer.

This module only draws numbers and decodes/encodes number formats. It holds none of the
quantization or GEMM arithmetic, so the GPU path and the CPU oracle can both be fed the very
same bytes from here without sharing any of the method.

Generator: a counter-based SplitMix64 stream (Steele, Lea and Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014; the finaliser constants are the published
ones), 53-bit uniforms, and the Box-Muller transform in float64. Each (seed, stream) pair
is an independent stream, and element i of a stream does not depend on the array shape.

Workload recipes follow the benchmark page "MNN GemmSpeed 基准测试实战" (sections
«为什么用 Conv1x1 来测 GEMM» for the weight fill, «默认测试尺寸与 M 的含义» for the shape grid)
and the five workloads the library is measured on.
"""
from __future__ import annotations

import dataclasses

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_MIX1 = np.uint64(0xBF58476D1CE4E5B9)
_MIX2 = np.uint64(0x94D049BB133111EB)
_STREAM = np.uint64(0xD1B54A32D192ED03)

# number-format codes shared with the C ABI (same values as include/qgemm.h)
F32, F16, BF16 = 0, 1, 2
DTYPE_NAMES = {F32: "f32", F16: "f16", BF16: "bf16"}


def _splitmix_finalise(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _MIX1
    z = (z ^ (z >> np.uint64(27))) * _MIX2
    return z ^ (z >> np.uint64(31))


def uniform64(n: int, seed: int, stream: int = 0, start: int = 0) -> np.ndarray:
    """n uniforms in [0, 1) with 53 random bits: element i is a pure function of (seed, stream, start+i)."""
    with np.errstate(over="ignore"):
        key = _splitmix_finalise(np.array([np.uint64(seed) * _GOLDEN ^ np.uint64(stream) * _STREAM],
                                          dtype=np.uint64))[0]
        ctr = np.arange(start + 1, start + n + 1, dtype=np.uint64)
        z = _splitmix_finalise(key + ctr * _GOLDEN)
    return (z >> np.uint64(11)).astype(np.float64) * (1.0 / 9007199254740992.0)


def normal64(n: int, seed: int, stream: int = 0, std: float = 1.0) -> np.ndarray:
    """n draws of N(0, std^2) in float64 (Box-Muller over consecutive uniform pairs)."""
    m = (n + 1) // 2
    u = uniform64(2 * m, seed, stream)
    u1, u2 = 1.0 - u[0::2], u[1::2]  # u1 in (0, 1]: log is finite
    r = np.sqrt(-2.0 * np.log(u1))
    z = np.empty(2 * m, dtype=np.float64)
    z[0::2] = r * np.cos(2.0 * np.pi * u2)
    z[1::2] = r * np.sin(2.0 * np.pi * u2)
    return z[:n] * std


# ---------------------------------------------------------------- number formats
def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (round to nearest, ties to even), as uint16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def encode(x64: np.ndarray, dtype: int) -> np.ndarray:
    """float64 values -> storage array of the given format (bf16 as uint16 bits)."""
    if dtype == F32:
        return x64.astype(np.float32)
    if dtype == F16:
        return x64.astype(np.float16)
    if dtype == BF16:
        return f32_to_bf16_bits(x64.astype(np.float32))
    raise ValueError(f"unknown dtype code {dtype}")


def decode(arr: np.ndarray, dtype: int) -> np.ndarray:
    """storage array (bf16 as uint16 bits) -> exact float64 values."""
    if dtype == BF16:
        return bf16_bits_to_f32(arr).astype(np.float64)
    return np.asarray(arr).astype(np.float64)


def mnn_fill(K: int, N: int) -> np.ndarray:
    """The benchmark page's deterministic weight fill: ((i % 127) - 63) / 1000 over the flat
    index i of the row-major {ic, oc} = [K][N] weight, computed as float32 division."""
    i = np.arange(K * N, dtype=np.int64)
    num = ((i % 127) - 63).astype(np.float32)
    return (num / np.float32(1000.0)).reshape(K, N)


# ---------------------------------------------------------------- workloads
MODE_FLOAT, MODE_INT4, MODE_INT8, MODE_W4A8 = 0, 1, 2, 3
MODE_NAMES = {MODE_FLOAT: "float", MODE_INT4: "int4", MODE_INT8: "int8", MODE_W4A8: "w4a8"}


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    M: int
    K: int
    N: int
    mode: int
    block: int          # 0 = whole K (Block0)
    a_dtype: int
    c_dtype: int
    a_seed: int
    w_seed: int
    w_std: float = 0.02
    w_fill: str = "normal"   # "normal" or "mnn" (the page's ((i % 127) - 63)/1000 fill)
    w_dtype: int = F16        # float mode only: 16-bit type of the packed weight copy

    @property
    def flops(self) -> float:
        return 2.0 * self.M * self.K * self.N


def make_activations(w: Workload, M: int | None = None) -> np.ndarray:
    """A [M][K] in the workload's storage format (stream 1 of the activation seed)."""
    M = w.M if M is None else M
    return encode(normal64(M * w.K, w.a_seed, stream=1).reshape(M, w.K), w.a_dtype)


def make_weights(w: Workload) -> np.ndarray:
    """W [K][N] float32 (stream 2 of the weight seed, or the page's fill)."""
    if w.w_fill == "mnn":
        return mnn_fill(w.K, w.N)
    return normal64(w.K * w.N, w.w_seed, stream=2, std=w.w_std).astype(np.float32).reshape(w.K, w.N)


WORKLOADS = {
    # Int4-Block64, fp32 activations and output
    "int4_b64_m4_k256_n512_f32": Workload("int4_b64_m4_k256_n512_f32", 4, 256, 512, MODE_INT4, 64,
                                          F32, F32, a_seed=0, w_seed=0),
    # decode GEMV of a 7B-class FFN up-projection
    "int4_b64_decode_m1_k4096_n11008_bf16": Workload("int4_b64_decode_m1_k4096_n11008_bf16", 1, 4096, 11008,
                                                     MODE_INT4, 64, BF16, BF16, a_seed=0, w_seed=0),
    # Int8-Block0 with the page's weight fill, M swept over {1, 2, 4, 8, 16}
    "int8_b0_k4096_n4096_f16": Workload("int8_b0_k4096_n4096_f16", 16, 4096, 4096, MODE_INT8, 0,
                                        F16, F16, a_seed=0, w_seed=0, w_fill="mnn"),
    # prefill
    "int4_b64_prefill_m1024_k4096_n4096": Workload("int4_b64_prefill_m1024_k4096_n4096", 1024, 4096, 4096,
                                                   MODE_INT4, 64, F16, BF16, a_seed=1, w_seed=0),
    # W4A8 with per-channel INT4 weights
    "w4a8_m2048_k4096_n14336": Workload("w4a8_m2048_k4096_n14336", 2048, 4096, 14336, MODE_W4A8, 0,
                                        BF16, BF16, a_seed=0, w_seed=0),
    # the fp16 float GEMM of the same shape, run alongside the W4A8 one
    "float_f16_m2048_k4096_n14336": Workload("float_f16_m2048_k4096_n14336", 2048, 4096, 14336, MODE_FLOAT, 0,
                                             F16, F16, a_seed=0, w_seed=0, w_dtype=F16),
}
INT8_M_SWEEP = (1, 2, 4, 8, 16)
