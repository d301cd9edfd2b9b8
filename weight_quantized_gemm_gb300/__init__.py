"""Python binding of libqgemm (include/qgemm.h): the same entry points, argument marshalling only.

Every compute step runs in the library's CUDA kernels; this module only turns torch tensors
into device pointers and the current CUDA stream into a cudaStream_t. It never falls back to
a CPU or PyTorch implementation: if the compiled library is missing, importing the binding
functions raises.

Build the library with ``__graft_entry__.build()`` (or ``python -m weight_quantized_gemm_gb300._build``).
"""
from __future__ import annotations

import ctypes
import os

__all__ = [
    "QgemmError", "load", "qgemm_packed_bytes", "qgemm_table_bytes", "qgemm_workspace_bytes", "qgemm_pack",
    "qgemm_run", "qgemm_act_quant", "qgemm_w4a8_acc", "qgemm_w4a8_acc_workspace_bytes", "qgemm_status", "qgemm_error_string", "qgemm_last_error",
    "qgemm_set_option", "qgemm_get_option", "OPT_LAUNCH_OVERLAP", "OPT_DECODE_MAX_M", "OPT_SPLIT_K", "OPT_WAIT_LIMIT_US", "OPT_DEBUG_STALL", "OPT_FAULT_INJECT", "qgemm_run_fused", "qgemm_save", "qgemm_load_info", "qgemm_load", "ACT_NONE", "ACT_RELU", "ACT_SILU", "ACT_GELU_TANH", "qgemm_run_noalloc", "NOALLOC_SCRATCH_BYTES", "qgemm_run_fused_quant",
    "qgemm_fused_quant_workspace_bytes", "qgemm_run_w4a8_codes", "qgemm_w4a8_codes_workspace_bytes",
    "MODE_FLOAT", "MODE_INT4", "MODE_INT8", "MODE_W4A8", "F32", "F16", "BF16", "LIB_PATH",
]

MODE_FLOAT, MODE_INT4, MODE_INT8, MODE_W4A8 = 0, 1, 2, 3
OPT_LAUNCH_OVERLAP = 1
OPT_DECODE_MAX_M = 2
OPT_SPLIT_K = 3
OPT_WAIT_LIMIT_US = 4
OPT_DEBUG_STALL = 5
OPT_FAULT_INJECT = 6
ACT_NONE, ACT_RELU, ACT_SILU, ACT_GELU_TANH = 0, 1, 2, 3
NOALLOC_SCRATCH_BYTES = 4 << 20
F32, F16, BF16 = 0, 1, 2
OK = 0
ERRORS = {-1: "QGEMM_ERR_ARG", -2: "QGEMM_ERR_UNSUPPORTED", -3: "QGEMM_ERR_ALIGN", -4: "QGEMM_ERR_WORKSPACE",
          -5: "QGEMM_ERR_CUDA", -6: "QGEMM_ERR_TIMEOUT", -7: "QGEMM_ERR_IO"}

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_lib", "libqgemm.so")
_lib = None

# exported symbol -> (argtypes, restype)
_P, _I, _SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
SIGNATURES = {
    "qgemm_packed_bytes": ([_I, _I, _I, _I], _SZ),
    "qgemm_table_bytes": ([_I, _I, _I, _I], _SZ),
    "qgemm_workspace_bytes": ([_I, _I, _I, _I, _I, _I, _I], _SZ),
    "qgemm_pack": ([_P, _I, _I, _I, _I, _I, _P, _P, _P], _I),
    "qgemm_run": ([_I, _I, _I, _I, _I, _P, _I, _P, _P, _P, _I, _P, _SZ, _P], _I),
    "qgemm_run_fused": ([_I, _I, _I, _I, _I, _P, _I, _P, _P, _P, _I, _P, _P, _I, _P, _SZ, _P], _I),
    "qgemm_act_quant": ([_I, _I, _P, _I, _P, _P, _P, _P], _I),
    "qgemm_w4a8_acc": ([_I, _I, _I, _P, _P, _P, _P, _SZ, _P], _I),
    "qgemm_w4a8_acc_workspace_bytes": ([_I, _I], _SZ),
    "qgemm_status": ([_P], _I),
    "qgemm_run_noalloc": ([_I, _I, _I, _I, _I, _P, _I, _P, _P, _P, _I, _P], _I),
    "qgemm_run_fused_quant": ([_I, _I, _I, _I, _I, _P, _I, _P, _P, _P, _I, _P, _P, _I, _P, _P, _P, _P, _SZ, _P], _I),
    "qgemm_fused_quant_workspace_bytes": ([_I, _I, _I, _I, _I, _I, _I], _SZ),
    "qgemm_run_w4a8_codes": ([_I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _I, _P, _P, _I, _P, _SZ, _P], _I),
    "qgemm_w4a8_codes_workspace_bytes": ([_I, _I, _I, _I], _SZ),
    "qgemm_save": ([ctypes.c_char_p, _I, _I, _I, _I, _I, _P, _P, _I, _P], _I),
    "qgemm_load_info": ([ctypes.c_char_p] + [ctypes.POINTER(ctypes.c_int)] * 5, _I),
    "qgemm_load": ([ctypes.c_char_p, _P, _SZ, _P, _SZ, _I, _P], _I),
    "qgemm_set_option": ([_I, _I], _I),
    "qgemm_get_option": ([_I], _I),
    "qgemm_error_string": ([_I], ctypes.c_char_p),
    "qgemm_last_error": ([], ctypes.c_char_p),
}


class QgemmError(RuntimeError):
    def __init__(self, code: int, fn: str):
        self.code = code
        detail = load().qgemm_last_error().decode(errors="replace")
        super().__init__(f"{fn}: {ERRORS.get(code, code)}: {detail}")


def load():
    """Load the compiled library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"libqgemm is not built ({LIB_PATH} missing); run __graft_entry__.build()")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (args, res) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
    return _lib


def _ptr(x):
    """Device (or host) address of a tensor, an int address, or None."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    return x.ctypes.data      # a numpy array (host memory)


def _on_device(*xs) -> int:
    """1 if the given buffers (torch tensors or numpy arrays; None ignored) are on the GPU, 0 if
    on the host; mixed placements are an error."""
    where = {bool(getattr(x, "is_cuda", False)) for x in xs if x is not None}
    if len(where) > 1:
        raise ValueError("Bp and T must both be device tensors or both host buffers")
    return int(where.pop()) if where else 0


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(rc: int, fn: str):
    if rc != OK:
        raise QgemmError(rc, fn)


# ---------------------------------------------------------------- sizes
def qgemm_packed_bytes(K: int, N: int, mode: int, w_dtype: int = F16) -> int:
    return load().qgemm_packed_bytes(K, N, mode, w_dtype)


def qgemm_table_bytes(K: int, N: int, mode: int, block: int) -> int:
    return load().qgemm_table_bytes(K, N, mode, block)


def qgemm_workspace_bytes(M: int, K: int, N: int, mode: int, block: int, a_dtype: int, c_dtype: int) -> int:
    return load().qgemm_workspace_bytes(M, K, N, mode, block, a_dtype, c_dtype)


# ---------------------------------------------------------------- compute
def qgemm_pack(W, K: int, N: int, mode: int, block: int, w_dtype: int, Bp, T, stream=None) -> None:
    _check(load().qgemm_pack(_ptr(W), K, N, mode, block, w_dtype, _ptr(Bp), _ptr(T), _stream(stream)), "qgemm_pack")


def qgemm_save(path: str, K: int, N: int, mode: int, block: int, w_dtype: int, Bp, T, stream=None) -> None:
    """Writes a packed layer (qgemm_pack's Bp and T, device tensors or host buffers) to `path`."""
    dev = _on_device(Bp, T)
    _check(load().qgemm_save(os.fsencode(path), K, N, mode, block, w_dtype, _ptr(Bp), _ptr(T), dev,
                             _stream(stream) if dev else None), "qgemm_save")


def qgemm_load_info(path: str) -> dict:
    """The shape and format of a packed-weight file: {K, N, mode, block, w_dtype}."""
    vals = [ctypes.c_int() for _ in range(5)]
    _check(load().qgemm_load_info(os.fsencode(path), *[ctypes.byref(v) for v in vals]), "qgemm_load_info")
    return dict(zip(("K", "N", "mode", "block", "w_dtype"), (v.value for v in vals)))


def qgemm_load(path: str, Bp, T, stream=None) -> None:
    """Reads a packed-weight file into Bp and T (device tensors or host buffers, large enough)."""
    nbytes = lambda x: 0 if x is None else (x.numel() * x.element_size() if hasattr(x, "numel") else x.nbytes)
    dev = _on_device(Bp, T)
    _check(load().qgemm_load(os.fsencode(path), _ptr(Bp), nbytes(Bp), _ptr(T), nbytes(T), dev,
                             _stream(stream) if dev else None), "qgemm_load")


def qgemm_run(M: int, K: int, N: int, mode: int, block: int, A, a_dtype: int, Bp, T, C, c_dtype: int,
              workspace=None, workspace_bytes: int | None = None, stream=None) -> None:
    if workspace_bytes is None:
        workspace_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().qgemm_run(M, K, N, mode, block, _ptr(A), a_dtype, _ptr(Bp), _ptr(T), _ptr(C), c_dtype,
                            _ptr(workspace), workspace_bytes, _stream(stream)), "qgemm_run")


def qgemm_run_fused(M: int, K: int, N: int, mode: int, block: int, A, a_dtype: int, Bp, T, bias, act: int, residual,
                    C, c_dtype: int, workspace=None, workspace_bytes: int | None = None, stream=None) -> None:
    """C = act(A x dequant(Bp, T) + bias) + residual (see qgemm.h); bias / residual may be None."""
    if workspace_bytes is None:
        workspace_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().qgemm_run_fused(M, K, N, mode, block, _ptr(A), a_dtype, _ptr(Bp), _ptr(T), _ptr(bias), act,
                                  _ptr(residual), _ptr(C), c_dtype, _ptr(workspace), workspace_bytes, _stream(stream)),
           "qgemm_run_fused")


def qgemm_run_noalloc(M: int, K: int, N: int, mode: int, block: int, A, a_dtype: int, Bp, T, C, c_dtype: int,
                      stream=None) -> None:
    """qgemm_run with the library's built-in scratch instead of a caller workspace (see qgemm.h)."""
    _check(load().qgemm_run_noalloc(M, K, N, mode, block, _ptr(A), a_dtype, _ptr(Bp), _ptr(T), _ptr(C), c_dtype,
                                    _stream(stream)), "qgemm_run_noalloc")


def qgemm_fused_quant_workspace_bytes(M: int, K: int, N: int, mode: int, block: int, a_dtype: int,
                                      c_dtype: int) -> int:
    return load().qgemm_fused_quant_workspace_bytes(M, K, N, mode, block, a_dtype, c_dtype)


def qgemm_run_fused_quant(M: int, K: int, N: int, mode: int, block: int, A, a_dtype: int, Bp, T, bias, act: int,
                          residual, C, c_dtype: int, qa_next, as_next, rowsum_next, workspace=None,
                          workspace_bytes: int | None = None, stream=None) -> None:
    """The layer (as qgemm_run_fused) plus the next W4A8 layer's activation codes of C (see qgemm.h)."""
    if workspace_bytes is None:
        workspace_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().qgemm_run_fused_quant(M, K, N, mode, block, _ptr(A), a_dtype, _ptr(Bp), _ptr(T), _ptr(bias), act,
                                        _ptr(residual), _ptr(C), c_dtype, _ptr(qa_next), _ptr(as_next),
                                        _ptr(rowsum_next), _ptr(workspace), workspace_bytes, _stream(stream)),
           "qgemm_run_fused_quant")


def qgemm_w4a8_codes_workspace_bytes(M: int, K: int, N: int, block: int) -> int:
    return load().qgemm_w4a8_codes_workspace_bytes(M, K, N, block)


def qgemm_run_w4a8_codes(M: int, K: int, N: int, block: int, qa, a_scale, rowsum, Bp, T, bias, act: int, residual,
                         C, c_dtype: int, workspace=None, workspace_bytes: int | None = None, stream=None) -> None:
    """A W4A8 layer from activation codes (exact f16), row scales and code sums (see qgemm.h)."""
    if workspace_bytes is None:
        workspace_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().qgemm_run_w4a8_codes(M, K, N, block, _ptr(qa), _ptr(a_scale), _ptr(rowsum), _ptr(Bp), _ptr(T),
                                       _ptr(bias), act, _ptr(residual), _ptr(C), c_dtype, _ptr(workspace),
                                       workspace_bytes, _stream(stream)), "qgemm_run_w4a8_codes")


def qgemm_act_quant(M: int, K: int, A, a_dtype: int, qa, a_scale, rowsum, stream=None) -> None:
    _check(load().qgemm_act_quant(M, K, _ptr(A), a_dtype, _ptr(qa), _ptr(a_scale), _ptr(rowsum), _stream(stream)),
           "qgemm_act_quant")


def qgemm_w4a8_acc_workspace_bytes(M: int, K: int) -> int:
    return load().qgemm_w4a8_acc_workspace_bytes(M, K)


def qgemm_w4a8_acc(M: int, K: int, N: int, qa, Bp, acc, workspace=None, workspace_bytes: int | None = None,
                   stream=None) -> None:
    if workspace_bytes is None:
        workspace_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().qgemm_w4a8_acc(M, K, N, _ptr(qa), _ptr(Bp), _ptr(acc), _ptr(workspace), workspace_bytes,
                                 _stream(stream)), "qgemm_w4a8_acc")


def qgemm_status(stream=None) -> int:
    return load().qgemm_status(_stream(stream))


def qgemm_set_option(option: int, value: int) -> int:
    rc = load().qgemm_set_option(option, value)
    if rc < 0:
        raise QgemmError(rc, "qgemm_set_option")
    return rc


def qgemm_get_option(option: int) -> int:
    rc = load().qgemm_get_option(option)
    if rc < 0:
        raise QgemmError(rc, "qgemm_get_option")
    return rc


def qgemm_error_string(code: int) -> str:
    return load().qgemm_error_string(code).decode()


def qgemm_last_error() -> str:
    return load().qgemm_last_error().decode(errors="replace")
