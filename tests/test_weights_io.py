"""Packed-weight files (qgemm_save / qgemm_load_info / qgemm_load), host buffers only: no GPU.

The file carries the packed layer byte for byte plus a header; these tests pin the header
layout, the CRC-32 against zlib's (an independent implementation of the same checksum), the
round trip, and every way a file can be wrong (foreign, truncated, extended, corrupt,
inconsistent), each of which must leave the destination untouched."""
import os
import struct
import zlib

import numpy as np
import pytest

import oracle
import weight_quantized_gemm_gb300 as qg
from weight_quantized_gemm_gb300 import synth
from tests._util import ensure_built


@pytest.fixture(scope="module", autouse=True)
def built():
    ensure_built()


def _packed(K, N, mode, block, seed=0):
    """A packed layer made by the oracle (the file format does not care who packed it)."""
    w = synth.Workload("t", 1, K, N, mode, block, synth.F16, synth.F16, seed, seed + 1)
    W = synth.make_weights(w)
    if mode == 0:
        Bp = np.ascontiguousarray(oracle.pack_float(W, synth.F16)).view(np.uint8).reshape(-1)
        return Bp, None
    q, T = oracle.quantize(W, K if block == 0 else block, oracle.QMAX[mode])
    Bp = oracle.pack(q, oracle.NBITS[mode]).reshape(-1)
    nb = T.shape[1]
    # the library's grouped table layout [ceil(N/16)][nb][16][2], zero padding channels
    G = (N + 15) // 16
    Tg = np.zeros((G * 16, nb, 2), np.float32)
    Tg[:N] = T
    Tg = np.ascontiguousarray(Tg.reshape(G, 16, nb, 2).transpose(0, 2, 1, 3)).reshape(-1)
    assert Tg.nbytes == qg.qgemm_table_bytes(K, N, mode, block)
    return np.ascontiguousarray(Bp), Tg


@pytest.mark.parametrize("K,N,mode,block", [(256, 40, 1, 64), (512, 33, 2, 0), (128, 24, 0, 0), (192, 17, 3, 0)])
def test_round_trip_and_header(tmp_path, K, N, mode, block):
    Bp, T = _packed(K, N, mode, block)
    assert Bp.nbytes == qg.qgemm_packed_bytes(K, N, mode, synth.F16 if mode == 0 else 0)
    path = str(tmp_path / "layer.qgw")
    w_dtype = synth.F16 if mode == 0 else 0
    qg.qgemm_save(path, K, N, mode, block, w_dtype, Bp, T)
    raw = open(path, "rb").read()
    payload = Bp.tobytes() + (b"" if T is None else T.tobytes())
    assert len(raw) == 64 + len(payload) and raw[64:] == payload
    magic, ver, hdr, k, n, m, b, wd, crc, pb, tb, rsv = struct.unpack("<8sII5iIQQQ", raw[:64])
    assert (magic, ver, hdr) == (b"QGEMMW\x00\x01", 1, 64)
    assert (k, n, m, b, wd, pb, tb, rsv) == (K, N, mode, block, w_dtype, Bp.nbytes, 0 if T is None else T.nbytes, 0)
    assert crc == zlib.crc32(payload)
    assert qg.qgemm_load_info(path) == {"K": K, "N": N, "mode": mode, "block": block, "w_dtype": w_dtype}
    Bp2 = np.zeros_like(Bp)
    T2 = None if T is None else np.zeros_like(T)
    qg.qgemm_load(path, Bp2, T2)
    assert np.array_equal(Bp2, Bp)
    assert T is None or np.array_equal(T2, T)


def test_bad_files_leave_destination_untouched(tmp_path):
    K, N, mode, block = 256, 40, 1, 64
    Bp, T = _packed(K, N, mode, block, seed=5)
    path = str(tmp_path / "good.qgw")
    qg.qgemm_save(path, K, N, mode, block, 0, Bp, T)
    good = open(path, "rb").read()

    def expect_io_error(data, what):
        p = str(tmp_path / "bad.qgw")
        with open(p, "wb") as f:
            f.write(data)
        Bp2 = np.full_like(Bp, 0xA5)
        T2 = np.full_like(T, 7.0)
        with pytest.raises(qg.QgemmError) as e:
            qg.qgemm_load(p, Bp2, T2)
        assert e.value.code == -7, what
        assert (Bp2 == 0xA5).all() and (T2 == 7.0).all(), f"{what}: destination written"

    flip = bytearray(good)
    flip[64 + 100] ^= 0x10
    expect_io_error(bytes(flip), "corrupt payload")
    expect_io_error(good[:-1], "truncated")
    expect_io_error(good + b"\0", "trailing byte")
    expect_io_error(b"NOTQGEMM" + good[8:], "foreign magic")
    hdr = bytearray(good)
    hdr[20:24] = struct.pack("<i", N + 16)      # N that does not match the stored sizes
    expect_io_error(bytes(hdr), "inconsistent header")
    with pytest.raises(qg.QgemmError) as e:
        qg.qgemm_load_info(str(tmp_path / "missing.qgw"))
    assert e.value.code == -7
    # destination smaller than the file's Bp
    with pytest.raises(qg.QgemmError) as e:
        qg.qgemm_load(path, np.zeros(Bp.nbytes - 16, np.uint8), T)
    assert e.value.code == -1


def test_save_rejects_invalid_shape(tmp_path):
    lib = qg.load()
    p = os.fsencode(str(tmp_path / "x.qgw"))
    buf = np.zeros(1 << 16, np.uint8)
    assert lib.qgemm_save(p, 100, 8, 1, 64, 0, buf.ctypes.data, buf.ctypes.data, 0, None) < 0    # K % 64
    assert lib.qgemm_save(p, 256, 8, 1, 64, 0, None, buf.ctypes.data, 0, None) == -1            # null Bp
    assert lib.qgemm_save(p, 256, 8, 1, 64, 0, buf.ctypes.data, None, 0, None) == -1            # null T
    assert lib.qgemm_save(None, 256, 8, 1, 64, 0, buf.ctypes.data, buf.ctypes.data, 0, None) == -1
    assert not os.path.exists(str(tmp_path / "x.qgw"))
