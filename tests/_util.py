"""Shared test helpers: tolerance rule, tensor marshalling, library build."""
from __future__ import annotations

import os
import re

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qgemm.h")

# Floating-point bar: normwise relative error max|g - R| / max|R| <= TOL, where R is the
# float64 oracle. For 16-bit outputs the output's own rounding (half an ulp of R_i in the
# output format) is allowed on top, element by element: bf16's unit roundoff 2^-8 alone is
# larger than the 2e-3 bar.
TOL = {0: 1e-5, 1: 2e-3, 2: 2e-3}     # by activation dtype: f32, f16, bf16
MANT_BITS = {0: 23, 1: 10, 2: 7}       # by output dtype
MIN_EXP = {0: -126, 1: -14, 2: -126}


def table_rows(T_flat, N: int, nb: int) -> np.ndarray:
    """The library's {offset, scale} table, stored in 16-channel groups [ceil(N/16)][nb][16][2],
    as [N][nb][2]; asserts that the padding channels of the last group are zero."""
    G = (N + 15) // 16
    t = np.asarray(T_flat).reshape(G, nb, 16, 2).transpose(0, 2, 1, 3).reshape(G * 16, nb, 2)
    assert not t[N:].any(), "padding channels of the table are not zero"
    return t[:N]


def half_ulp(R: np.ndarray, c_dtype: int) -> np.ndarray:
    a = np.abs(R)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, MIN_EXP[c_dtype])
    return 0.5 * np.exp2(e - MANT_BITS[c_dtype])


def check_close(got: np.ndarray, R: np.ndarray, a_dtype: int, c_dtype: int, what: str = "") -> float:
    """Asserts the bar and returns the measured normwise error."""
    got = np.asarray(got, dtype=np.float64)
    assert got.shape == R.shape, (got.shape, R.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    scale = max(float(np.abs(R).max()), 1e-30)
    diff = np.abs(got - R)
    err = float(diff.max() / scale)
    allow = TOL[a_dtype] * scale + (half_ulp(R, c_dtype) if c_dtype != 0 else 0.0)
    bad = diff > allow
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {bad.size} outside the bar; normwise err {err:.3e}, "
                           f"worst at {np.unravel_index(np.argmax(diff - allow), R.shape)}")
    return err


def header_functions() -> list[str]:
    src = open(HEADER).read()
    return re.findall(r"^\s*(?:const\s+)?(?:int|size_t|char\s*\*|const char\s*\*)\s*\*?\s*(qgemm_\w+)\s*\(", src,
                      flags=re.M)


def torch_from(arr: np.ndarray, dtype_code: int, device: str = "cuda"):
    """numpy storage array (bf16 as uint16 bits) -> torch tensor of the right dtype."""
    import torch
    if dtype_code == 2:
        t = torch.from_numpy(np.ascontiguousarray(arr).view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(arr))
    return t.to(device)


def to_numpy_values(t, dtype_code: int) -> np.ndarray:
    """torch tensor -> exact float64 values."""
    import torch
    if dtype_code == 2:
        return (t.cpu().view(torch.int16).numpy().view(np.uint16).astype(np.uint32) << 16).view(
            np.float32).astype(np.float64)
    return t.cpu().numpy().astype(np.float64)


def torch_dtype(code: int):
    import torch
    return {0: torch.float32, 1: torch.float16, 2: torch.bfloat16}[code]


def ensure_built():
    from weight_quantized_gemm_gb300 import _build
    return _build.build()
