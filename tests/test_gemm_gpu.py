"""Dequant-GEMM (M > 1) on the GPU against the fp64 oracle, through the C ABI."""
import numpy as np
import pytest

import oracle.bt_oracle as O
from helpers import assert_close, half_tensor, make_case, out_to_f64, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from dequant_gemv_gemm_bt_b300 import bt
    return torch, bt


def run(env, qw, xb, xdtype, out_dtype, path=0):
    torch, bt = env
    codes, scales, biases = to_dev(qw, torch)
    x = half_tensor(xb, xdtype, torch)
    od = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[out_dtype]
    try:
        bt.bt_set_option(bt.BT_OPT_GEMM_PATH, path)
        y = bt.bt_qgemm(codes, scales, biases, qw.bits, x, out_dtype=od)
    finally:
        bt.bt_set_option(bt.BT_OPT_GEMM_PATH, 0)
    torch.cuda.synchronize()
    return out_to_f64(y, torch)


@pytest.mark.parametrize("bits", (2, 3, 4, 6, 8))
@pytest.mark.parametrize("m,n,k", [(2, 130, 256), (17, 300, 1024), (64, 257, 512), (128, 384, 3072), (130, 200, 192)])
def test_qgemm_matches_oracle(env, bits, m, n, k):
    qw, x = make_case("gemm", n, k, bits, m=m, xdtype="bf16")
    y = run(env, qw, x, "bf16", "bf16")
    y_ref, a = O.qgemm(qw.codes, qw.scales, qw.biases, bits, O.decode_bf16(x))
    assert_close(y, y_ref, a, "bf16", f"b={bits} m={m} n={n} k={k}")


@pytest.mark.parametrize("path", [1, 2])
@pytest.mark.parametrize("m", [2, 16, 33, 64, 127, 128, 129, 256, 512])
def test_qgemm_paths_q4(env, path, m):
    qw, x = make_case("gemm-path", 640, 1024, 4, m=m, xdtype="bf16")
    y = run(env, qw, x, "bf16", "bf16", path=path)
    y_ref, a = O.qgemm(qw.codes, qw.scales, qw.biases, 4, O.decode_bf16(x))
    assert_close(y, y_ref, a, "bf16", f"path={path} m={m}")


# Every output type is held to its own bound: fp32 outputs to 1e-3*A (the
# tensor-core path feeds bf16 X products split hi + lo weight tiles), 16-bit
# outputs to 8e-3*A.
@pytest.mark.parametrize("xdtype,out", [("f16", "f32"), ("bf16", "f32"), ("f16", "f16"), ("bf16", "bf16")])
@pytest.mark.parametrize("path", [1, 2])
def test_qgemm_dtypes(env, xdtype, out, path):
    qw, x = make_case("gemm-dt", 256, 1024, 4, m=96, xdtype=xdtype)
    y = run(env, qw, x, xdtype, out, path=path)
    y_ref, a = O.qgemm(qw.codes, qw.scales, qw.biases, 4, O.decode_half(x, xdtype))
    assert_close(y, y_ref, a, out, f"{xdtype}->{out} path {path}")


@pytest.mark.parametrize("bits", (2, 4, 6, 8))
@pytest.mark.parametrize("k", (128, 256, 1024, 3072))
def test_qgemm_tc_bf16_x_f32_out_meets_f32_bound(env, bits, k):
    """bf16 X, fp32 Y on the tensor cores at short and long K: a bf16 weight alone
    (8 significant bits) would miss 1e-3*A at small K; the hi + lo tiles meet it."""
    qw, x = make_case("gemm-f32", 300, k, bits, m=80, xdtype="bf16")
    y = run(env, qw, x, "bf16", "f32", path=2)
    y_ref, a = O.qgemm(qw.codes, qw.scales, qw.biases, bits, O.decode_bf16(x))
    assert_close(y, y_ref, a, "f32", f"bf16->f32 b={bits} k={k}")


def test_qgemm_m1_is_gemv(env):
    qw, x = make_case("gemm-m1", 500, 1024, 4, m=1, xdtype="f16")
    y = run(env, qw, x, "f16", "f32")
    y_ref, a = O.qgemm(qw.codes, qw.scales, qw.biases, 4, O.decode_f16(x))
    assert_close(y, y_ref, a, "f32", "M=1")


def test_qgemm_deterministic(env):
    qw, x = make_case("gemm-det", 512, 2048, 4, m=128, xdtype="bf16")
    assert np.array_equal(run(env, qw, x, "bf16", "bf16"), run(env, qw, x, "bf16", "bf16"))


@pytest.mark.parametrize("splits", [1, 2, 3, 5, 8])
@pytest.mark.parametrize("m", [40, 128, 300])
def test_qgemm_tc_k_split(env, splits, m):
    """Tensor-core path with K split over a cluster (partials reduced in shared memory)."""
    torch, bt = env
    qw, x = make_case("gemm-split", 333, 3072, 4, m=m, xdtype="bf16")
    try:
        bt.bt_set_option(bt.BT_OPT_GEMM_SPLITS, splits)
        y = run(env, qw, x, "bf16", "f32", path=2)
        y2 = run(env, qw, x, "bf16", "f32", path=2)
    finally:
        bt.bt_set_option(bt.BT_OPT_GEMM_SPLITS, 0)
    assert np.array_equal(y, y2), "split-K result is not deterministic"
    y_ref, a = O.qgemm(qw.codes, qw.scales, qw.biases, 4, O.decode_bf16(x))
    assert_close(y, y_ref, a, "f32", f"splits={splits} m={m}")


@pytest.mark.parametrize("bits,m,n,k", [(3, 128, 384, 3072), (3, 64, 256, 1024), (4, 96, 256, 64 * 5),
                                        (4, 128, 256, 64 * 63), (4, 64, 512, 16384), (2, 128, 256, 32768)])
def test_qgemm_tc_q3_odd_groups_long_k(env, bits, m, n, k):
    """3-bit codes (stages hold aligned 48-byte K-block pairs), odd group counts, and
    K beyond 192 groups (split over a cluster so each CTA stages at most 192) on the
    tensor cores, fp32 output at 1e-3*A."""
    torch, bt = env
    assert bt.bt_plan_gemm(bits, m, n, k)["path"] == "tc"
    qw, x = make_case("gemm-tc-ext", n, k, bits, m=m, xdtype="bf16")
    y = run(env, qw, x, "bf16", "f32", path=2)
    assert bt.bt_last_device_error() == bt.BT_OK
    y_ref, a = O.qgemm(qw.codes, qw.scales, qw.biases, bits, O.decode_bf16(x))
    assert_close(y, y_ref, a, "f32", f"tc b={bits} m={m} n={n} k={k}")
