"""Format variants on the GPU against the fp64 oracle, through the C ABI: group
sizes 32 and 128 (besides 64), 5-bit codes, and fp16 weights (bits = 16, no
scale or bias) -- the Q2..FP16 range of the BaseRT pages."""
import numpy as np
import pytest

import oracle.bt_oracle as O
from dequant_gemv_gemm_bt_b300 import synth
from helpers import assert_close, half_tensor, out_to_f64, to_dev

pytestmark = pytest.mark.gpu
WIDTHS = (2, 3, 4, 5, 6, 8, 16)


@pytest.fixture(scope="module")
def env():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from dequant_gemv_gemm_bt_b300 import bt
    return torch, bt


def case(tag, n, k, bits, g, m=1, xdtype="f16"):
    r = synth.rng_for("test", "formats", tag, n, k, bits, g, m, xdtype)
    qw = synth.make_qweight(r, n, k, bits, group_size=g)
    x = synth.draw_activations(r, m, k, xdtype)
    return qw, x


def dev_w(qw, torch):
    c, s, b = to_dev(qw, torch)
    return (c, None, None) if qw.bits == 16 else (c, s, b)


@pytest.mark.parametrize("bits", WIDTHS)
@pytest.mark.parametrize("g", (32, 64, 128))
@pytest.mark.parametrize("n,k", [(333, 1024), (70, 3072), (9, 256)])
def test_gemv_formats(env, bits, g, n, k):
    torch, bt = env
    qw, x = case("gemv", n, k, bits, g)
    y = bt.bt_qgemv(*dev_w(qw, torch), bits, half_tensor(x[0], "f16", torch), group_size=g)
    y_ref, a = O.qgemv(qw.codes, qw.scales, qw.biases, bits, O.decode_f16(x[0]), group_size=g)
    assert_close(out_to_f64(y, torch), y_ref, a, "f32", f"GEMV b={bits} g={g} n={n} k={k}")


@pytest.mark.parametrize("bits", WIDTHS)
@pytest.mark.parametrize("g", (32, 128))
def test_gemv_formats_bf16_x(env, bits, g):
    torch, bt = env
    qw, x = case("gemv-bf16", 301, 2048, bits, g, xdtype="bf16")
    y = bt.bt_qgemv(*dev_w(qw, torch), bits, half_tensor(x[0], "bf16", torch), group_size=g)
    y_ref, a = O.qgemv(qw.codes, qw.scales, qw.biases, bits, O.decode_bf16(x[0]), group_size=g)
    assert_close(out_to_f64(y, torch), y_ref, a, "f32", f"GEMV bf16 b={bits} g={g}")


@pytest.mark.parametrize("bits", (4, 5, 16))
@pytest.mark.parametrize("g", (32, 128))
def test_gemv_batched_mixed_k_formats(env, bits, g):
    torch, bt = env
    r = synth.rng_for("test", "formats-batched", bits, g)
    probs, cases = [], []
    for k in (1024, 2048, 3072, 512, 1024, 8192, 256):
        n = int(r.integers(1, 600))
        qw = synth.make_qweight(r, n, k, bits, group_size=g)
        x16 = synth.draw_activations(r, 1, k, "f16")
        y = torch.full((n,), float("nan"), dtype=torch.float32, device="cuda")
        probs.append((*dev_w(qw, torch), half_tensor(x16[0], "f16", torch), y))
        cases.append((qw, x16))
    bt.bt_qgemv_batched(probs, bits, group_size=g)
    torch.cuda.synchronize()
    assert bt.bt_last_device_error() == bt.BT_OK
    for (qw, x16), pr in zip(cases, probs):
        y_ref, a = O.qgemv(qw.codes, qw.scales, qw.biases, bits, O.decode_f16(x16[0]), group_size=g)
        assert_close(out_to_f64(pr[4], torch), y_ref, a, "f32", f"batched b={bits} g={g} k={qw.k}")


@pytest.mark.parametrize("bits", WIDTHS)
@pytest.mark.parametrize("g", (32, 128))
@pytest.mark.parametrize("path", [1, 2])
@pytest.mark.parametrize("out", ["bf16", "f32"])
def test_gemm_formats(env, bits, g, path, out):
    """M = 96 on the CUDA-core tile (path 1) and on the tensor cores (path 2, where the
    shape allows: widths 2/4/6/8; the others run the tile)."""
    torch, bt = env
    qw, x = case("gemm", 260, 1024, bits, g, m=96, xdtype="bf16")
    od = {"bf16": torch.bfloat16, "f32": torch.float32}[out]
    try:
        bt.bt_set_option(bt.BT_OPT_GEMM_PATH, path)
        y = bt.bt_qgemm(*dev_w(qw, torch), bits, half_tensor(x, "bf16", torch), group_size=g, out_dtype=od)
        torch.cuda.synchronize()
    finally:
        bt.bt_set_option(bt.BT_OPT_GEMM_PATH, 0)
    y_ref, a = O.qgemm(qw.codes, qw.scales, qw.biases, bits, O.decode_bf16(x), group_size=g)
    assert_close(out_to_f64(y, torch), y_ref, a, out, f"GEMM b={bits} g={g} path={path} -> {out}")


@pytest.mark.parametrize("g,k,splits", [(32, 2048, 4), (128, 3072, 3), (128, 8192, 8)])
def test_gemm_tc_k_split_formats(env, g, k, splits):
    """Tensor-core K split across a cluster with groups of 32 and 128: every split's
    staged parameter range starts on a group boundary."""
    torch, bt = env
    qw, x = case("gemm-split", 384, k, 4, g, m=128, xdtype="bf16")
    try:
        bt.bt_set_option(bt.BT_OPT_GEMM_SPLITS, splits)
        y = bt.bt_qgemm(*dev_w(qw, torch), 4, half_tensor(x, "bf16", torch), group_size=g, out_dtype=torch.float32)
        torch.cuda.synchronize()
    finally:
        bt.bt_set_option(bt.BT_OPT_GEMM_SPLITS, 0)
    y_ref, a = O.qgemm(qw.codes, qw.scales, qw.biases, 4, O.decode_bf16(x), group_size=g)
    assert_close(out_to_f64(y, torch), y_ref, a, "f32", f"split g={g} k={k}")


def stack(ws):
    return tuple(np.stack([getattr(w, f) for w in ws]) for f in ("codes", "scales", "biases"))


@pytest.mark.parametrize("bits,g", [(4, 128), (5, 32), (16, 64), (6, 32)])
@pytest.mark.parametrize("path", [0, 1, 2])
def test_moe_grouped_formats(env, bits, g, path):
    torch, bt = env
    r = synth.rng_for("test", "formats-moe", bits, g)
    e, n, k = 6, 256, 1024
    w = stack([synth.make_qweight(r, n, k, bits, group_size=g) for _ in range(e)])
    offsets = np.array([0, 3, 3, 40, 41, 41, 97], dtype=np.int32)
    xb = synth.draw_activations(r, 97, k, "bf16")
    dw = [torch.from_numpy(w[0].view(np.int32)).cuda(), torch.from_numpy(w[1].view(np.float16)).cuda(),
          torch.from_numpy(w[2].view(np.float16)).cuda()]
    if bits == 16:
        dw[1] = dw[2] = None
    try:
        bt.bt_set_option(bt.BT_OPT_GEMM_PATH, path)
        y = bt.bt_moe_qgemm(*dw, bits, torch.from_numpy(offsets).cuda(), half_tensor(xb, "bf16", torch),
                            group_size=g, out_dtype=torch.float32)
        torch.cuda.synchronize()
    finally:
        bt.bt_set_option(bt.BT_OPT_GEMM_PATH, 0)
    assert bt.bt_last_device_error() == bt.BT_OK
    y_ref, a = O.moe_qgemm(*w, bits, offsets, O.decode_bf16(xb), group_size=g)
    assert_close(out_to_f64(y, torch), y_ref, a, "f32", f"MoE b={bits} g={g} path={path}")


def test_fp16_weights_one_hot_column(env):
    """bits = 16: a one-hot x returns the stored fp16 weight column exactly."""
    torch, bt = env
    qw, _ = case("fp16-onehot", 515, 1024, 16, 64)
    codes = to_dev(qw, torch)[0]
    w = O.dequant_weight(qw.codes, qw.scales, qw.biases, 16, 1024)
    for col in (0, 1, 31, 32, 513, 1023):
        x = np.zeros((1024,), dtype=np.float16)
        x[col] = 1.0
        y = bt.bt_qgemv(codes, None, None, 16, half_tensor(x.view(np.uint16), "f16", torch))
        np.testing.assert_array_equal(out_to_f64(y, torch), w[:, col])
