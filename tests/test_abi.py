"""C-ABI surface checks that need no GPU: the library loads, exports every
declared symbol, and rejects bad arguments before any launch."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "bt.h")


@pytest.fixture(scope="module")
def bt():
    from dequant_gemv_gemm_bt_b300 import build
    build.build()
    from dequant_gemv_gemm_bt_b300 import bt as mod
    return mod


def declared_symbols():
    txt = open(HEADER).read()
    return sorted(set(re.findall(r"^BT_API\s+[\w\s\*]+?\b(bt_\w+)\s*\(", txt, flags=re.M)))


def test_header_declares_the_entry_points():
    syms = declared_symbols()
    for name in ("bt_qgemv", "bt_qgemm", "bt_moe_qgemm", "bt_status_string", "bt_last_device_error"):
        assert name in syms


def test_library_exports_every_declared_symbol(bt):
    for name in declared_symbols():
        assert hasattr(bt.lib, name), name
    assert set(declared_symbols()) == set(bt.EXPORTS)


def test_status_strings(bt):
    for s in range(6):
        assert bt.bt_status_string(s).startswith("BT_")
    assert "unknown" in bt.bt_status_string(99)


def test_set_option_validation(bt):
    assert bt.lib.bt_set_option(99, 1) == bt.BT_ERR_INVALID_ARG
    assert bt.lib.bt_set_option(bt.BT_OPT_PDL, -1) == bt.BT_ERR_INVALID_ARG
    assert bt.lib.bt_set_option(bt.BT_OPT_PDL, 0) == bt.BT_OK


# Fake, 16-byte-aligned device addresses: validation must reject before any CUDA call.
A = 0x7F0000000000
W = (A, A + 4096, A + 8192)


def gemv(bt, codes=W[0], scales=W[1], biases=W[2], bits=4, g=64, n=128, k=256, x=A + 16384, xd=0, y=A + 32768, yd=2):
    return bt.lib.bt_qgemv(codes, scales, biases, bits, g, n, k, x, xd, y, yd, None)


@pytest.mark.parametrize("kw,expect", [
    (dict(codes=None), 1), (dict(scales=None), 1), (dict(x=None), 1), (dict(y=None), 1),
    (dict(bits=7), 2), (dict(bits=1), 2), (dict(bits=12), 2), (dict(g=16), 2), (dict(g=96), 2), (dict(g=256), 2),
    (dict(bits=16, codes=None), 1), (dict(biases=None), 1), (dict(g=128, k=192), 1),
    (dict(n=0), 1), (dict(k=0), 1), (dict(n=-3), 1), (dict(k=100), 1), (dict(k=64 * 1024), 2),
    (dict(codes=A + 4), 3), (dict(x=A + 8), 3), (dict(xd=2), 1), (dict(yd=7), 1),
])
def test_qgemv_rejects_before_launch(bt, kw, expect):
    assert gemv(bt, **kw) == expect


def test_qgemm_and_moe_validation(bt):
    L = bt.lib
    assert L.bt_qgemm(*W, 4, 64, 0, 128, 256, A, 1, A, 1, None) == 1          # M = 0
    assert L.bt_qgemm(*W, 3, 64, 4, 128, 200, A, 1, A, 1, None) == 1          # K % 64
    assert L.bt_qgemm(*W, 7, 64, 4, 128, 256, A, 1, A, 1, None) == 2          # bits
    assert L.bt_moe_qgemm(*W, 4, 64, 0, 128, 256, A, 4, None, A, 1, A, 1, None) == 1   # E = 0
    assert L.bt_moe_qgemm(*W, 4, 64, 8, 128, 256, None, 4, None, A, 1, A, 1, None) == 1  # offsets
    assert L.bt_moe_qgemm(*W, 4, 64, 8, 128, 256, A, -1, None, A, 1, A, 1, None) == 1   # rows < 0
    assert L.bt_moe_qgemm(*W, 4, 64, 8, 128, 256, A, 0, None, A, 1, A, 1, None) == 0    # no rows: no-op
    assert L.bt_moe_route(A, 4, 0, 8, A, A, A, None, None) == 1                 # top_k = 0
    assert L.bt_moe_route(A, 4, 2, 0, A, A, A, None, None) == 1                 # E = 0
    assert L.bt_moe_route(A, 4, 2, 8, None, A, A, None, None) == 1
    assert L.bt_swiglu(A, 1, 4, 0, A, 1, None) == 1
    assert L.bt_moe_combine(A, 1, A, A, 4, 0, 128, A, 1, None) == 1


def test_pass_validation(bt):
    """bt_pass_create checks every stage before any CUDA call; NULL handles are refused."""
    L = bt.lib
    out = ctypes.c_void_p(7)
    assert L.bt_pass_create(None, 1, 4, 64, 1, 0, 2, ctypes.byref(out)) == 1
    assert out.value is None                                                   # *pass cleared
    prob = (bt.GemmProblem * 1)(bt.GemmProblem(A, A, A, A, A, 128, 256))
    stage = (bt.PassStage * 1)(bt.PassStage(ctypes.cast(prob, ctypes.POINTER(bt.GemmProblem)), 1))
    assert L.bt_pass_create(stage, 1, 4, 64, 1, 0, 2, None) == 1               # no out pointer
    assert L.bt_pass_create(stage, 0, 4, 64, 1, 0, 2, ctypes.byref(out)) == 1  # no stages
    assert L.bt_pass_create(stage, 1, 7, 64, 1, 0, 2, ctypes.byref(out)) == 2  # bits
    assert L.bt_pass_create(stage, 1, 4, 64, 0, 0, 2, ctypes.byref(out)) == 1  # M = 0
    assert L.bt_pass_create(stage, 1, 4, 64, 1, 2, 2, ctypes.byref(out)) == 1  # x dtype f32
    prob[0].n = 0
    assert L.bt_pass_create(stage, 1, 4, 64, 1, 0, 2, ctypes.byref(out)) == 1  # n = 0
    assert out.value is None
    assert L.bt_pass_run(None, None) == 1
    L.bt_pass_destroy(None)
