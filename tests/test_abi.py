"""The C ABI without a GPU: the library loads, exports every function include/qgemm.h
declares, sizes are right, and every argument check returns its code before any launch."""
import ctypes
import subprocess

import pytest

from tests._util import header_functions, ensure_built

import weight_quantized_gemm_gb300 as qg


@pytest.fixture(scope="module", autouse=True)
def built():
    ensure_built()


def test_exports_every_declared_symbol():
    names = header_functions()
    assert {"qgemm_pack", "qgemm_run", "qgemm_workspace_bytes", "qgemm_status"} <= set(names)
    lib = ctypes.CDLL(qg.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", qg.LIB_PATH], capture_output=True, text=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
    assert set(names) <= exported
    assert set(names) == set(qg.SIGNATURES)          # the binding covers exactly the header


def test_sizes():
    assert qg.qgemm_packed_bytes(4096, 11008, qg.MODE_INT4) == 4096 * 11008 // 2
    assert qg.qgemm_table_bytes(4096, 11008, qg.MODE_INT4, 64) == 11008 * 64 * 8
    assert qg.qgemm_table_bytes(256, 200, qg.MODE_INT4, 64) == 208 * 4 * 8    # channels padded to 16
    assert qg.qgemm_packed_bytes(4096, 4096, qg.MODE_INT8) == 4096 * 4096
    assert qg.qgemm_table_bytes(4096, 4096, qg.MODE_INT8, 0) == 4096 * 8
    assert qg.qgemm_packed_bytes(256, 512, qg.MODE_FLOAT, qg.F16) == 256 * 512 * 2
    assert qg.qgemm_packed_bytes(256, 512, qg.MODE_FLOAT, qg.F32) == 256 * 512 * 4
    assert qg.qgemm_table_bytes(256, 512, qg.MODE_FLOAT, 0) == 0
    assert qg.qgemm_packed_bytes(100, 512, qg.MODE_INT4) == 0           # K % 64 != 0
    assert qg.qgemm_table_bytes(256, 512, qg.MODE_INT4, 96) == 0       # block not a multiple of 64
    # W4A8: qa (M*K bytes), scales and row sums, each 256-byte aligned
    assert qg.qgemm_workspace_bytes(2048, 4096, 14336, qg.MODE_W4A8, 0, qg.BF16, qg.BF16) == 2 * 2048 * 4096 + 2 * 8192
    assert qg.qgemm_w4a8_acc_workspace_bytes(2048, 4096) == 2 * 2048 * 4096
    # W4A8, per-channel weights and K past 8808 (one float32 accumulation no longer exact): the
    # K-chunks' int32 accumulators [M][N] follow
    assert qg.qgemm_workspace_bytes(16, 8832, 40, qg.MODE_W4A8, 0, qg.BF16, qg.BF16) == (
        2 * 16 * 8832 + 2 * 256 + (-(-16 * 40 * 4 // 256)) * 256)
    assert qg.qgemm_workspace_bytes(16, 8768, 40, qg.MODE_W4A8, 0, qg.BF16, qg.BF16) == 2 * 16 * 8768 + 2 * 256
    # block-quantized W4A8 weights multiply float weights: no int32 chunks
    assert qg.qgemm_workspace_bytes(16, 8832, 40, qg.MODE_W4A8, 64, qg.BF16, qg.BF16) == 2 * 16 * 8832 + 2 * 256
    # decode with a large N needs no scratch; a small N splits K across blocks
    assert qg.qgemm_workspace_bytes(1, 4096, 11008, qg.MODE_INT4, 64, qg.BF16, qg.BF16) == 0
    assert qg.qgemm_workspace_bytes(1, 4096, 512, qg.MODE_INT4, 64, qg.BF16, qg.BF16) > 0


FAKE = 1 << 40          # 16-byte aligned addresses that are never dereferenced (calls fail first)


@pytest.mark.parametrize("args,code", [
    (dict(K=100), -2),                      # K % 64
    (dict(block=96), -2),                   # block not a multiple of 64
    (dict(block=128, K=192), -2),           # K % block
    (dict(mode=7), -1),
    (dict(a_dtype=5), -1),
    (dict(c_dtype=-1), -1),
    (dict(M=-1), -1),
    (dict(K=0), -1),
    (dict(A=0), -1),
    (dict(T=0), -1),
    (dict(C=FAKE + 8), -3),                 # misaligned
    (dict(Bp=FAKE + 1), -3),
    (dict(mode=3, block=0, ws=0, ws_bytes=0), -4),   # W4A8 needs scratch for the activation codes
    (dict(N=512, ws=0, ws_bytes=0), -4),    # small N: split-K scratch needed
    (dict(M=1 << 21), -2),                  # beyond the launch limit
])
def test_run_rejects_before_launch(args, code):
    a = dict(M=1, K=4096, N=11008, mode=1, block=64, A=FAKE, a_dtype=2, Bp=FAKE, T=FAKE, C=FAKE, c_dtype=2,
             ws=FAKE, ws_bytes=0, stream=0)
    a.update(args)
    rc = qg.load().qgemm_run(a["M"], a["K"], a["N"], a["mode"], a["block"], a["A"], a["a_dtype"], a["Bp"], a["T"],
                             a["C"], a["c_dtype"], a["ws"], a["ws_bytes"], a["stream"])
    assert rc == code, qg.qgemm_last_error()
    assert qg.qgemm_last_error() != ""


def test_empty_calls_are_noops():
    lib = qg.load()
    assert lib.qgemm_run(0, 4096, 64, 1, 64, None, 2, None, None, None, 2, None, 0, None) == 0
    assert lib.qgemm_run(4, 4096, 0, 1, 64, None, 2, None, None, None, 2, None, 0, None) == 0
    assert lib.qgemm_act_quant(0, 4096, None, 2, None, None, None, None) == 0
    assert lib.qgemm_pack(None, 4096, 0, 1, 64, 0, None, None, None) == 0


def test_pack_and_aux_reject():
    lib = qg.load()
    assert lib.qgemm_pack(FAKE, 4096, 64, 1, 64, 0, FAKE, None, None) == -1          # null T
    assert lib.qgemm_pack(FAKE + 4, 4096, 64, 1, 64, 0, FAKE, FAKE, None) == -3      # misaligned W
    assert lib.qgemm_pack(FAKE, 4096, 64, 0, 0, 9, FAKE, None, None) == -1           # bad w_dtype
    assert lib.qgemm_pack(FAKE, 4096, 64, 3, 96, 0, FAKE, FAKE, None) == -2          # block not a multiple of 64
    assert lib.qgemm_act_quant(4, 100, FAKE, 2, FAKE, FAKE, FAKE, None) == -2
    assert lib.qgemm_act_quant(4, 128, FAKE, 2, FAKE + 2, FAKE, FAKE, None) == -3
    assert lib.qgemm_w4a8_acc(4, 128, 8, FAKE, None, FAKE, FAKE, 1 << 20, None) == -1
    assert lib.qgemm_w4a8_acc(4, 128, 8, FAKE, FAKE, FAKE, FAKE, 16, None) == -4      # workspace too small
    # K whose int32 accumulators could overflow (127 * 15 * K > 2^31 - 1)
    big_k = (2147483647 // (127 * 15) // 64 + 1) * 64
    assert lib.qgemm_w4a8_acc(4, big_k, 8, FAKE, FAKE, FAKE, FAKE, 1 << 40, None) == -2
    assert lib.qgemm_w4a8_acc(4, big_k - 64, 8, FAKE, None, FAKE, FAKE, 1 << 40, None) == -1   # passes the K check
    assert lib.qgemm_run(4, big_k, 8, 3, 0, FAKE, 2, FAKE, FAKE, FAKE, 2, FAKE, 1 << 40, None) == -2


def test_options():
    assert qg.qgemm_get_option(qg.OPT_LAUNCH_OVERLAP) == 0
    assert qg.qgemm_set_option(qg.OPT_LAUNCH_OVERLAP, 1) == 0
    assert qg.qgemm_get_option(qg.OPT_LAUNCH_OVERLAP) == 1
    assert qg.qgemm_set_option(qg.OPT_LAUNCH_OVERLAP, 0) == 1
    assert qg.load().qgemm_set_option(qg.OPT_LAUNCH_OVERLAP, 2) == -1
    assert qg.qgemm_get_option(qg.OPT_DECODE_MAX_M) == 16
    ws16 = qg.qgemm_workspace_bytes(32, 4096, 256, qg.MODE_INT4, 64, qg.BF16, qg.BF16)
    assert qg.qgemm_set_option(qg.OPT_DECODE_MAX_M, 64) == 16     # M = 32 now runs on the decode kernels
    assert qg.qgemm_workspace_bytes(32, 4096, 256, qg.MODE_INT4, 64, qg.BF16, qg.BF16) != ws16
    assert qg.qgemm_set_option(qg.OPT_DECODE_MAX_M, 16) == 64
    assert qg.load().qgemm_set_option(qg.OPT_DECODE_MAX_M, 8) == -1
    assert qg.load().qgemm_set_option(qg.OPT_DECODE_MAX_M, 2048) == -1
    # the tensor-core path's split-K partials: M = 64, N = 4096 gives 32 tiles of 128 channels x
    # 64 rows, so K = 2560 (40 stages of 64) is split 4 ways to fill one wave of 152 SMs
    assert qg.qgemm_get_option(qg.OPT_SPLIT_K) == 1
    assert qg.qgemm_workspace_bytes(64, 2560, 4096, qg.MODE_INT4, 64, qg.F16, qg.F16) == 4 * 64 * 4096 * 4
    assert qg.qgemm_workspace_bytes(64, 256, 4096, qg.MODE_INT4, 64, qg.F16, qg.F16) == 0       # 4 stages: no split
    assert qg.qgemm_workspace_bytes(1024, 4096, 4096, qg.MODE_INT4, 64, qg.F16, qg.F16) == 0    # 128 tiles already
    assert qg.qgemm_set_option(qg.OPT_SPLIT_K, 0) == 1
    assert qg.qgemm_workspace_bytes(64, 2560, 4096, qg.MODE_INT4, 64, qg.F16, qg.F16) == 0
    assert qg.qgemm_set_option(qg.OPT_SPLIT_K, 1) == 0
    assert qg.load().qgemm_set_option(qg.OPT_SPLIT_K, 2) == -1
    assert qg.load().qgemm_set_option(99, 0) == -1
    assert qg.load().qgemm_get_option(99) == -1


def test_error_strings():
    for code, name in qg.ERRORS.items():
        assert qg.qgemm_error_string(code) == name
    assert qg.qgemm_error_string(0) == "QGEMM_OK"


def test_fused_epilogue_argument_checks():
    """qgemm_run_fused validates its epilogue before anything is launched."""
    lib = qg.load()
    FAKE = 1 << 20
    run = lib.qgemm_run_fused
    assert run(4, 128, 8, 1, 64, FAKE, 2, FAKE, FAKE, None, 9, None, FAKE, 2, None, 0, None) == -1      # unknown act
    assert run(4, 128, 8, 1, 64, FAKE, 2, FAKE, FAKE, None, -1, None, FAKE, 2, None, 0, None) == -1
    assert run(4, 128, 8, 1, 64, FAKE, 2, FAKE, FAKE, FAKE + 4, 0, None, FAKE, 2, None, 0, None) == -3  # bias
    assert run(4, 128, 8, 1, 64, FAKE, 2, FAKE, FAKE, None, 0, FAKE + 2, FAKE, 2, None, 0, None) == -3  # residual
    assert run(0, 128, 8, 1, 64, None, 2, None, None, None, 3, None, None, 2, None, 0, None) == 0      # empty call


def test_binding_fails_loudly_without_library(monkeypatch):
    """No CPU fallback: with the compiled library absent, the binding raises instead of computing."""
    monkeypatch.setattr(qg, "_lib", None)
    monkeypatch.setattr(qg, "LIB_PATH", "/nonexistent/libqgemm.so")
    with pytest.raises(ImportError):
        qg.load()
    with pytest.raises(ImportError):
        qg.qgemm_workspace_bytes(64, 4096, 4096, qg.MODE_INT4, 64, qg.F16, qg.F16)


@pytest.mark.parametrize("M", [17, 24, 64, 100, 128, 200, 256, 512, 1024])
@pytest.mark.parametrize("K,N", [(1024, 4096), (2560, 1024), (4096, 2560), (2560, 9728), (9728, 2560), (4096, 14336)])
def test_tensor_core_split_rule(M, K, N):
    """The tensor-core path's K-split, read off the workspace size: the splits fill at most one
    wave of 152 SMs, each keeps at least 8 stages of 64, 256-row tiles split 3 or more ways only,
    and Int8-Block0 with bf16 and M >= 256 adds its row sums in front."""
    bn = 64 if M <= 64 else (128 if M <= 128 else 256)
    tiles = -(-N // 128) * -(-M // bn)
    for mode, block, a_dtype in [(qg.MODE_INT4, 64, qg.F16), (qg.MODE_INT8, 0, qg.BF16), (qg.MODE_FLOAT, 0, qg.F16)]:
        ws = qg.qgemm_workspace_bytes(M, K, N, mode, block, a_dtype, qg.BF16)
        rows = -(-M * 4 // 256) * 256 if (mode == qg.MODE_INT8 and a_dtype == qg.BF16 and M >= 256) else 0
        part = ws - rows
        assert part % (M * N * 4) == 0
        splits = part // (M * N * 4)
        if splits:
            assert 2 <= splits <= 152 // tiles and splits <= (K // 64) // 8
            assert bn < 256 or 152 // tiles >= 3      # 256-row tiles: only when 3+ splits fit in a wave
        else:
            want = min(152 // tiles, (K // 64) // 8)
            assert want < (3 if bn >= 256 else 2)


def test_fault_injection_simulates_a_launch_failure():
    """QGEMM_OPT_FAULT_INJECT: the n-th compute call reports QGEMM_ERR_CUDA without launching;
    rejected calls do not count. Each case sets n = 1, so no call here reaches a launch."""
    lib = qg.load()
    assert qg.qgemm_get_option(qg.OPT_FAULT_INJECT) == 0
    run = lambda M, K: lib.qgemm_run(M, K, 11008, 1, 64, FAKE, 2, FAKE, FAKE, FAKE, 2, FAKE, 0, None)
    try:
        assert qg.qgemm_set_option(qg.OPT_FAULT_INJECT, 1) == 0
        assert run(1, 100) == -2                           # rejected first: not counted
        assert qg.qgemm_get_option(qg.OPT_FAULT_INJECT) == 1
        assert run(1, 4096) == -5
        assert "simulated launch failure" in qg.qgemm_last_error()
        assert qg.qgemm_get_option(qg.OPT_FAULT_INJECT) == 0
        assert run(0, 4096) == 0                           # empty calls launch nothing and are not counted
        cases = [
            lambda: lib.qgemm_pack(FAKE, 4096, 64, 1, 64, 0, FAKE, FAKE, None),
            lambda: lib.qgemm_act_quant(4, 128, FAKE, 2, FAKE, FAKE, FAKE, None),
            lambda: lib.qgemm_w4a8_acc(4, 128, 8, FAKE, FAKE, FAKE, FAKE, 1 << 20, None),
            lambda: lib.qgemm_run_fused(4, 128, 8, 1, 64, FAKE, 2, FAKE, FAKE, None, 2, None, FAKE, 2, None, 0, None),
        ]
        for call in cases:
            qg.qgemm_set_option(qg.OPT_FAULT_INJECT, 1)
            assert call() == -5
            assert "simulated launch failure" in qg.qgemm_last_error()
        qg.qgemm_set_option(qg.OPT_FAULT_INJECT, 1)
        with pytest.raises(qg.QgemmError) as ei:          # the binding raises it like any failure
            qg.qgemm_run(1, 4096, 11008, 1, 64, FAKE, 2, FAKE, FAKE, FAKE, 2, FAKE, 0, stream=0)
        assert ei.value.code == -5
        assert lib.qgemm_set_option(qg.OPT_FAULT_INJECT, -1) == -1
    finally:
        qg.qgemm_set_option(qg.OPT_FAULT_INJECT, 0)


def test_fault_injection_from_environment():
    code = ("import weight_quantized_gemm_gb300 as qg; "
            "print(qg.qgemm_get_option(qg.OPT_FAULT_INJECT))")
    import os
    import sys
    env = dict(os.environ, QGEMM_FAULT_INJECT="3")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    out = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env, cwd=root)
    assert out.returncode == 0, out.stderr
    assert out.stdout.strip() == "3"


def test_wait_limit_and_stall_options():
    assert qg.qgemm_get_option(qg.OPT_WAIT_LIMIT_US) == 1000000
    assert qg.qgemm_set_option(qg.OPT_WAIT_LIMIT_US, 500) == 1000000
    assert qg.qgemm_set_option(qg.OPT_WAIT_LIMIT_US, 1000000) == 500
    assert qg.load().qgemm_set_option(qg.OPT_WAIT_LIMIT_US, 0) == -1
    assert qg.load().qgemm_set_option(qg.OPT_WAIT_LIMIT_US, 1000001) == -1
    assert qg.qgemm_get_option(qg.OPT_DEBUG_STALL) == 0
    assert qg.qgemm_set_option(qg.OPT_DEBUG_STALL, 1) == 0
    assert qg.qgemm_set_option(qg.OPT_DEBUG_STALL, 0) == 1
    assert qg.load().qgemm_set_option(qg.OPT_DEBUG_STALL, 2) == -1


def test_fused_quant_sizes_and_checks():
    lib = qg.load()
    # tensor-core route: the per-tile row maxima [ceil(N/128)][M] float32 after the layer's scratch
    assert qg.qgemm_fused_quant_workspace_bytes(256, 1024, 512, qg.MODE_INT4, 64, qg.F16, qg.BF16) == 4 * 256 * 4
    w4 = 2 * 64 * 1024 + 2 * 256
    assert qg.qgemm_fused_quant_workspace_bytes(64, 1024, 512, qg.MODE_W4A8, 0, qg.BF16, qg.BF16) == w4 + 4 * 64 * 4
    # decode path: the standalone activation pass on C needs nothing beyond the layer's own scratch
    assert (qg.qgemm_fused_quant_workspace_bytes(8, 4096, 11008, qg.MODE_INT4, 64, qg.BF16, qg.BF16) ==
            qg.qgemm_workspace_bytes(8, 4096, 11008, qg.MODE_INT4, 64, qg.BF16, qg.BF16))
    assert qg.qgemm_fused_quant_workspace_bytes(256, 1024, 520, qg.MODE_INT4, 64, qg.F16, qg.BF16) == 0   # N % 64
    run = lib.qgemm_run_fused_quant
    args = lambda **kw: [kw.get(k, v) for k, v in dict(
        M=256, K=1024, N=512, mode=1, block=64, A=FAKE, a_dtype=1, Bp=FAKE, T=FAKE, bias=None, act=0, res=None,
        C=FAKE, c_dtype=2, qa=FAKE, asc=FAKE, rs=FAKE, ws=FAKE, wsb=1 << 20, stream=None).items()]
    assert run(*args(N=520)) == -2                     # the next layer's K must be a multiple of 64
    assert run(*args(qa=None)) == -1
    assert run(*args(rs=FAKE + 4)) == -3
    assert run(*args(wsb=16)) == -4
    assert run(*args(M=0, A=None, C=None)) == 0
    # the consumer's int32 accumulators when K needs exact chunks
    assert qg.qgemm_w4a8_codes_workspace_bytes(16, 8832, 40, 0) == -(-16 * 40 * 4 // 256) * 256
    assert qg.qgemm_w4a8_codes_workspace_bytes(16, 4096, 40, 0) == 0
    codes = lib.qgemm_run_w4a8_codes
    assert codes(4, 128, 8, 0, FAKE, None, FAKE, FAKE, FAKE, None, 0, None, FAKE, 2, None, 0, None) == -1
    assert codes(4, 8832, 8, 0, FAKE, FAKE, FAKE, FAKE, FAKE, None, 0, None, FAKE, 2, None, 0, None) == -4
