"""CPU oracle for the weight-quantized linear layer (TEST INFRASTRUCTURE ONLY).

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py``
may import this package. The library's GPU path never does, and this package never imports
the library: the two share nothing but the seeded inputs drawn by
``weight_quantized_gemm_gb300.synth`` (which holds no quantization or GEMM arithmetic).

The arithmetic lives in ``qgemm_oracle.c`` (plain loops, float64 accumulation, float32
quantization decisions); this module compiles it with gcc and marshals numpy arrays.
Cited passages: the benchmark page "MNN GemmSpeed 基准测试实战", sections
«为什么用 Conv1x1 来测 GEMM» (GEMM shape, asymmetric [offset, scale] blocks, Int8-Block0,
Int4-Block64, oc x blockNum table) and «测试用例与注册机制» (W4A8).

Parity status of each function is recorded in the test suite's pins; every function here is
pinned (closed forms, exact dyadic cases, brute force, invariants), none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qgemm_oracle.c")
_LIBDIR = os.path.join(_HERE, "_lib")
_LIB = os.path.join(_LIBDIR, "liborc.so")
_lock = threading.Lock()
_lib = None

F32, F16, BF16 = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile the oracle (gcc, -O2 -fopenmp -ffp-contract=off, no fast-math)."""
    with _lock:
        if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
            return _LIB
        os.makedirs(_LIBDIR, exist_ok=True)
        tmp = _LIB + f".{os.getpid()}.tmp"
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
               "-shared", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
        return _LIB


def _load():
    global _lib
    if _lib is None:
        path = build()
        lib = ctypes.CDLL(path)
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        I = ctypes.c_int
        sigs = {
            "orc_set_threads": [I],
            "orc_quantize": [P, I64, I64, I64, I, P, P],
            "orc_pack": [P, I64, I64, I, P],
            "orc_unpack": [P, I64, I64, I, P],
            "orc_dequant": [P, P, I64, I64, I64, P],
            "orc_gemm": [I64, I64, I64, P, P, P],
            "orc_gemm_points": [I64, I64, I64, P, P, P, I64, P, P, P],
            "orc_dense_points": [I64, P, P, I64, P, P, P],
            "orc_to_bf16_t": [P, I64, I64, P],
            "orc_act_quant": [I64, I64, P, P, P, P],
            "orc_w4a8_acc": [I64, I64, I64, P, P, P],
            "orc_w4a8_acc_points": [I64, P, P, I64, P, P, P],
            "orc_w4a8_out": [I64, I64, P, P, P, P, P],
            "orc_epilogue": [I64, I64, P, P, I, P],
            "orc_w4a8_block_out": [I64, I64, I64, I64, P, P, P, P, P],
        }
        for name, args in sigs.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = I
        _lib = lib
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def _check(rc: int, what: str):
    if rc != 0:
        raise ValueError(f"oracle {what} failed with code {rc}")


def set_threads(n: int = 0) -> int:
    """Set the OpenMP thread count (0 keeps the current one); returns the count in use."""
    return _load().orc_set_threads(n)


# ---------------------------------------------------------------- quantize / pack
def quantize(W: np.ndarray, block: int, qmax: int):
    """W [K][N] float32 -> (q [N][K] uint8 codes, T [N][K/block][2] float32 {offset, scale})."""
    W = np.ascontiguousarray(W, dtype=np.float32)
    K, N = W.shape
    block = K if block == 0 else block
    q = np.empty((N, K), dtype=np.uint8)
    T = np.empty((N, K // block, 2), dtype=np.float32)
    _check(_load().orc_quantize(_p(W), K, N, block, qmax, _p(q), _p(T)), "quantize")
    return q, T


def pack(q: np.ndarray, nbits: int) -> np.ndarray:
    q = np.ascontiguousarray(q, dtype=np.uint8)
    N, K = q.shape
    Bp = np.empty((N, K * nbits // 8), dtype=np.uint8)
    _check(_load().orc_pack(_p(q), K, N, nbits, _p(Bp)), "pack")
    return Bp


def unpack(Bp: np.ndarray, K: int, nbits: int) -> np.ndarray:
    Bp = np.ascontiguousarray(Bp, dtype=np.uint8)
    N = Bp.shape[0]
    q = np.empty((N, K), dtype=np.uint8)
    _check(_load().orc_unpack(_p(Bp), K, N, nbits, _p(q)), "unpack")
    return q


def dequant(q: np.ndarray, T: np.ndarray, block: int) -> np.ndarray:
    """codes + table -> Bt [N][K] float64 (the transpose of the dequantized B[K][N])."""
    q = np.ascontiguousarray(q, dtype=np.uint8)
    T = np.ascontiguousarray(T, dtype=np.float32)
    N, K = q.shape
    block = K if block == 0 else block
    Bt = np.empty((N, K), dtype=np.float64)
    _check(_load().orc_dequant(_p(q), _p(T), K, N, block, _p(Bt)), "dequant")
    return Bt


def pack_float(W: np.ndarray, w_dtype: int) -> np.ndarray:
    """Float mode: W [K][N] float32 -> 16-bit copy transposed to [N][K] (bf16 as uint16 bits).
    float16 uses numpy's round-to-nearest-even conversion; bfloat16 is rounded in C."""
    W = np.ascontiguousarray(W, dtype=np.float32)
    K, N = W.shape
    if w_dtype == F16:
        return np.ascontiguousarray(W.T.astype(np.float16))
    if w_dtype == BF16:
        out = np.empty((N, K), dtype=np.uint16)
        _check(_load().orc_to_bf16_t(_p(W), K, N, _p(out)), "to_bf16")
        return out
    if w_dtype == F32:
        return np.ascontiguousarray(W.T)
    raise ValueError(w_dtype)


def values(stored: np.ndarray, dtype: int) -> np.ndarray:
    """Exact float64 values of a stored array (bf16 given as uint16 bit patterns)."""
    if dtype == BF16:
        return (np.ascontiguousarray(stored, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(
            np.float32).astype(np.float64)
    return np.asarray(stored).astype(np.float64)


# ---------------------------------------------------------------- GEMM
def gemm(A64: np.ndarray, Bt: np.ndarray) -> np.ndarray:
    """R = A x B in float64 with A [M][K] and Bt = B^T [N][K]."""
    A64 = np.ascontiguousarray(A64, dtype=np.float64)
    Bt = np.ascontiguousarray(Bt, dtype=np.float64)
    M, K = A64.shape
    N = Bt.shape[0]
    R = np.empty((M, N), dtype=np.float64)
    _check(_load().orc_gemm(M, K, N, _p(A64), _p(Bt), _p(R)), "gemm")
    return R


def gemm_points(A64: np.ndarray, q: np.ndarray, T: np.ndarray, block: int, m_idx, n_idx) -> np.ndarray:
    A64 = np.ascontiguousarray(A64, dtype=np.float64)
    q = np.ascontiguousarray(q, dtype=np.uint8)
    T = np.ascontiguousarray(T, dtype=np.float32)
    N, K = q.shape
    block = K if block == 0 else block
    mi = np.ascontiguousarray(m_idx, dtype=np.int64)
    ni = np.ascontiguousarray(n_idx, dtype=np.int64)
    out = np.empty(mi.shape[0], dtype=np.float64)
    _check(_load().orc_gemm_points(K, N, block, _p(A64), _p(q), _p(T), mi.shape[0], _p(mi), _p(ni), _p(out)),
           "gemm_points")
    return out


def dense_points(A64: np.ndarray, Bt: np.ndarray, m_idx, n_idx) -> np.ndarray:
    A64 = np.ascontiguousarray(A64, dtype=np.float64)
    Bt = np.ascontiguousarray(Bt, dtype=np.float64)
    mi = np.ascontiguousarray(m_idx, dtype=np.int64)
    ni = np.ascontiguousarray(n_idx, dtype=np.int64)
    out = np.empty(mi.shape[0], dtype=np.float64)
    _check(_load().orc_dense_points(A64.shape[1], _p(A64), _p(Bt), mi.shape[0], _p(mi), _p(ni), _p(out)),
           "dense_points")
    return out


# ---------------------------------------------------------------- W4A8
def act_quant(A32: np.ndarray):
    """A [M][K] float32 -> (qa int8 [M][K], as float32 [M], rowsum int32 [M])."""
    A32 = np.ascontiguousarray(A32, dtype=np.float32)
    M, K = A32.shape
    qa = np.empty((M, K), dtype=np.int8)
    s = np.empty(M, dtype=np.float32)
    rs = np.empty(M, dtype=np.int32)
    _check(_load().orc_act_quant(M, K, _p(A32), _p(qa), _p(s), _p(rs)), "act_quant")
    return qa, s, rs


def w4a8_acc(qa: np.ndarray, q: np.ndarray) -> np.ndarray:
    qa = np.ascontiguousarray(qa, dtype=np.int8)
    q = np.ascontiguousarray(q, dtype=np.uint8)
    M, K = qa.shape
    N = q.shape[0]
    acc = np.empty((M, N), dtype=np.int32)
    _check(_load().orc_w4a8_acc(M, K, N, _p(qa), _p(q), _p(acc)), "w4a8_acc")
    return acc


def w4a8_acc_points(qa: np.ndarray, q: np.ndarray, m_idx, n_idx) -> np.ndarray:
    qa = np.ascontiguousarray(qa, dtype=np.int8)
    q = np.ascontiguousarray(q, dtype=np.uint8)
    mi = np.ascontiguousarray(m_idx, dtype=np.int64)
    ni = np.ascontiguousarray(n_idx, dtype=np.int64)
    out = np.empty(mi.shape[0], dtype=np.int32)
    _check(_load().orc_w4a8_acc_points(qa.shape[1], _p(qa), _p(q), mi.shape[0], _p(mi), _p(ni), _p(out)),
           "w4a8_acc_points")
    return out


def w4a8_out(acc: np.ndarray, s: np.ndarray, rowsum: np.ndarray, T: np.ndarray) -> np.ndarray:
    acc = np.ascontiguousarray(acc, dtype=np.int32)
    s = np.ascontiguousarray(s, dtype=np.float32)
    rowsum = np.ascontiguousarray(rowsum, dtype=np.int32)
    T = np.ascontiguousarray(T, dtype=np.float32).reshape(-1, 2)
    M, N = acc.shape
    R = np.empty((M, N), dtype=np.float64)
    _check(_load().orc_w4a8_out(M, N, _p(acc), _p(s), _p(rowsum), _p(T), _p(R)), "w4a8_out")
    return R


ACT_NONE, ACT_RELU, ACT_SILU, ACT_GELU_TANH = 0, 1, 2, 3


def epilogue(R: np.ndarray, bias=None, act: int = ACT_NONE, residual=None) -> np.ndarray:
    """act(R + bias) + residual in float64 (a new array). bias: float32 [N]; residual: the
    residual's values (float64-convertible) [M][N]. Reading of the Adreno 750 pull request's
    "before bias, residual and activation": activation first, then the residual."""
    out = np.array(R, dtype=np.float64, order="C", copy=True)
    M, N = out.shape
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    r = None if residual is None else np.ascontiguousarray(residual, dtype=np.float64)
    _check(_load().orc_epilogue(M, N, _p(out), None if b is None else _p(b), act, None if r is None else _p(r)),
           "epilogue")
    return out


def w4a8_block_out(qa: np.ndarray, s: np.ndarray, q: np.ndarray, T: np.ndarray, block: int) -> np.ndarray:
    """W4A8 with block-quantized weights: as * sum_b (ws_b * block integer GEMM + off_b * block
    row sum), float64. qa [M][K] int8, s [M], q [N][K] codes, T [N][K/block][2]."""
    qa = np.ascontiguousarray(qa, dtype=np.int8)
    s = np.ascontiguousarray(s, dtype=np.float32)
    q = np.ascontiguousarray(q, dtype=np.uint8)
    T = np.ascontiguousarray(T, dtype=np.float32)
    M, K = qa.shape
    N = q.shape[0]
    R = np.empty((M, N), dtype=np.float64)
    _check(_load().orc_w4a8_block_out(M, K, N, block, _p(qa), _p(s), _p(q), _p(T), _p(R)), "w4a8_block_out")
    return R


# ---------------------------------------------------------------- whole layer
QMAX = {1: 15, 2: 255, 3: 15}     # mode -> largest code (INT4, INT8, W4A8 weights)
NBITS = {1: 4, 2: 8, 3: 4}


def reference_layer(mode: int, block: int, A_stored: np.ndarray, a_dtype: int, W: np.ndarray,
                    w_dtype: int = F16):
    """The whole layer for a small case: returns a dict with the packed weights, the table and
    the float64 result R (and for W4A8 the activation codes and the int32 accumulators)."""
    K = W.shape[0]
    out = {}
    if mode == 0:
        Wt = pack_float(W, w_dtype)
        out["Bp"] = Wt
        out["R"] = gemm(values(A_stored, a_dtype), values(Wt, w_dtype))
        return out
    blk = K if block == 0 else block
    q, T = quantize(W, blk, QMAX[mode])
    out.update(q=q, T=T, Bp=pack(q, NBITS[mode]))
    if mode == 3:
        A32 = values(A_stored, a_dtype).astype(np.float32)
        qa, s, rs = act_quant(A32)
        out.update(qa=qa, a_scale=s, rowsum=rs)
        if blk == K:   # per channel: one integer GEMM, rescaled per channel
            acc = w4a8_acc(qa, q)
            out.update(acc=acc, R=w4a8_out(acc, s, rs, T))
        else:          # per K-block: integer GEMMs per block, rescaled per block
            out.update(R=w4a8_block_out(qa, s, q, T, blk))
        return out
    out["R"] = gemm(values(A_stored, a_dtype), dequant(q, T, blk))
    return out
