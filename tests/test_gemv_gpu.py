"""Dequant-GEMV (M = 1) on the GPU against the fp64 oracle, through the C ABI."""
import numpy as np
import pytest

import oracle.bt_oracle as O
from helpers import assert_close, half_tensor, make_case, out_to_f64, to_dev

pytestmark = pytest.mark.gpu
BITS = (2, 3, 4, 6, 8)


@pytest.fixture(scope="module")
def env():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from dequant_gemv_gemm_bt_b300 import bt
    return torch, bt


def run(env, qw, x16, xdtype, out_dtype):
    torch, bt = env
    codes, scales, biases = to_dev(qw, torch)
    x = half_tensor(x16[0], xdtype, torch)
    od = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[out_dtype]
    y = bt.bt_qgemv(codes, scales, biases, qw.bits, x, out_dtype=od)
    torch.cuda.synchronize()
    return out_to_f64(y, torch)


@pytest.mark.parametrize("bits", BITS)
@pytest.mark.parametrize("n,k", [(1, 64), (7, 128), (333, 1024), (2085, 1024), (515, 3072), (260, 8192)])
def test_qgemv_matches_oracle(env, bits, n, k):
    qw, x = make_case("gemv", n, k, bits)
    y = run(env, qw, x, "f16", "f32")
    y_ref, a = O.qgemv(qw.codes, qw.scales, qw.biases, bits, O.decode_f16(x[0]))
    assert_close(y, y_ref, a, "f32", f"b={bits} n={n} k={k}")


@pytest.mark.parametrize("bits", BITS)
@pytest.mark.parametrize("xdtype,out", [("bf16", "f32"), ("f16", "bf16"), ("bf16", "f16")])
def test_qgemv_dtypes(env, bits, xdtype, out):
    qw, x = make_case("gemv-dt", 301, 2048, bits, xdtype=xdtype)
    y = run(env, qw, x, xdtype, out)
    y_ref, a = O.qgemv(qw.codes, qw.scales, qw.biases, bits, O.decode_half(x[0], xdtype))
    assert_close(y, y_ref, a, out, f"b={bits} {xdtype}->{out}")


@pytest.mark.parametrize("k", [64, 1024, 16384, 32768])
def test_qgemv_k_extremes(env, k):
    for bits in (3, 4):
        qw, x = make_case("gemv-k", 41, k, bits)
        y = run(env, qw, x, "f16", "f32")
        y_ref, a = O.qgemv(qw.codes, qw.scales, qw.biases, bits, O.decode_f16(x[0]))
        assert_close(y, y_ref, a, "f32", f"b={bits} k={k}")


def test_qgemv_single_q4_workload_and_determinism(env):
    """The single Q4 GEMV workload: N=2048, K=1024, fp16 x, fp32 y."""
    torch, bt = env
    qw, x = make_case("c1", 2048, 1024, 4)
    y1 = run(env, qw, x, "f16", "f32")
    y2 = run(env, qw, x, "f16", "f32")
    assert np.array_equal(y1, y2), "GEMV is not bitwise deterministic"
    y_ref, a = O.qgemv(qw.codes, qw.scales, qw.biases, 4, O.decode_f16(x[0]))
    assert_close(y1, y_ref, a, "f32", "N=2048 K=1024 Q4")


@pytest.mark.parametrize("bits", BITS)
def test_qgemv_one_hot_returns_column(env, bits):
    torch, bt = env
    n, k = 517, 1024
    qw, _ = make_case("onehot", n, k, bits)
    w = O.dequant_weight(qw.codes, qw.scales, qw.biases, bits, k)
    for col in (0, 31, 32, 63, 64, 777, 1023):
        x = np.zeros((1, k), dtype=np.float16)
        x[0, col] = 1.0
        y = run(env, qw, x.view(np.uint16), "f16", "f32")
        np.testing.assert_allclose(y, w[:, col], rtol=0, atol=1e-5)


def test_qgemv_lm_head_sampled(env):
    """Full-size lm_head GEMV (N=151936, K=1024, Q4) checked on sampled rows."""
    torch, bt = env
    from dequant_gemv_gemm_bt_b300 import synth
    r = synth.rng_for("test", "lm_head")
    qw = synth.make_qweight(r, 151936, 1024, 4)
    x = synth.draw_activations(r, 1, 1024, "f16")
    y = run(env, qw, x, "f16", "f32")
    rows = np.unique(np.concatenate([np.arange(0, 64), np.arange(151936 - 64, 151936),
                                     r.integers(0, 151936, 2000)]))
    y_ref, a = O.qgemv(qw.codes, qw.scales, qw.biases, 4, O.decode_f16(x[0]), rows=rows)
    assert_close(y[rows], y_ref, a, "f32", "lm_head sampled rows")


def test_qgemv_pdl_and_const_weights(env):
    torch, bt = env
    qw, x = make_case("pdl", 1200, 2048, 4)
    y_ref, a = O.qgemv(qw.codes, qw.scales, qw.biases, 4, O.decode_f16(x[0]))
    try:
        bt.bt_set_option(bt.BT_OPT_PDL, 1)
        bt.bt_set_option(bt.BT_OPT_CONST_WEIGHTS, 1)
        ys = [run(env, qw, x, "f16", "f32") for _ in range(3)]
    finally:
        bt.bt_set_option(bt.BT_OPT_PDL, 0)
        bt.bt_set_option(bt.BT_OPT_CONST_WEIGHTS, 0)
    for y in ys:
        assert_close(y, y_ref, a, "f32", "pdl")


def test_qgemv_generic_path_matches_fast(env):
    torch, bt = env
    for bits in (2, 3, 4, 6, 8):
        qw, x = make_case("generic", 300, 1024, bits)
        y_fast = run(env, qw, x, "f16", "f32")
        try:
            bt.bt_set_option(bt.BT_OPT_GEMV_GENERIC, 1)
            y_gen = run(env, qw, x, "f16", "f32")
        finally:
            bt.bt_set_option(bt.BT_OPT_GEMV_GENERIC, 0)
        y_ref, a = O.qgemv(qw.codes, qw.scales, qw.biases, bits, O.decode_f16(x[0]))
        assert_close(y_gen, y_ref, a, "f32", "generic")
        assert_close(y_fast, y_ref, a, "f32", "fast")


@pytest.mark.parametrize("k", [1024, 3072, 8192])
def test_device_wait_timeout_is_reported(env, k):
    """A stage that is never filled makes the consumers' bounded waits expire;
    the call reports BT_ERR_TIMEOUT and the context stays usable.  K = 3072 and
    8192 split each row over 4 and 8 warps that meet at named barriers: warps
    that gave up still reach every barrier, so none is left waiting."""
    torch, bt = env
    qw, x = make_case("timeout", 4000, k, 4)
    codes, scales, biases = to_dev(qw, torch)
    xt = half_tensor(x[0], "f16", torch)
    assert bt.bt_last_device_error() == bt.BT_OK
    try:
        bt.bt_set_option(bt.BT_OPT_WAIT_TIMEOUT_US, 20000)
        bt.bt_set_option(bt.BT_OPT_TEST_DROP_STAGE, 1)
        bt.bt_qgemv(codes, scales, biases, 4, xt)
        assert bt.bt_last_device_error() == bt.BT_ERR_TIMEOUT
    finally:
        bt.bt_set_option(bt.BT_OPT_TEST_DROP_STAGE, 0)
        bt.bt_set_option(bt.BT_OPT_WAIT_TIMEOUT_US, 4000000)
    assert bt.bt_last_device_error() == bt.BT_OK
    y = run(env, qw, x, "f16", "f32")
    y_ref, a = O.qgemv(qw.codes, qw.scales, qw.biases, 4, O.decode_f16(x[0]))
    assert_close(y, y_ref, a, "f32", "after timeout")


def test_device_wait_timeout_mixed_k_batch(env):
    """The same expiry in a mixed-K batch, whose CTAs also meet at the barrier
    taken when the K split changes between problems."""
    torch, bt = env
    from dequant_gemv_gemm_bt_b300 import synth
    r = synth.rng_for("test", "timeout-mixed")
    probs, cases = [], []
    for k in (3072, 1024, 2048, 1024, 3072):
        qw = synth.make_qweight(r, 900, k, 4)
        x16 = synth.draw_activations(r, 1, k, "f16")
        codes, scales, biases = to_dev(qw, torch)
        y = torch.empty(900, dtype=torch.float32, device="cuda")
        probs.append((codes, scales, biases, half_tensor(x16[0], "f16", torch), y))
        cases.append((qw, x16))
    assert bt.bt_last_device_error() == bt.BT_OK
    try:
        bt.bt_set_option(bt.BT_OPT_WAIT_TIMEOUT_US, 20000)
        bt.bt_set_option(bt.BT_OPT_TEST_DROP_STAGE, 1)
        bt.bt_qgemv_batched(probs, 4)
        assert bt.bt_last_device_error() == bt.BT_ERR_TIMEOUT
    finally:
        bt.bt_set_option(bt.BT_OPT_TEST_DROP_STAGE, 0)
        bt.bt_set_option(bt.BT_OPT_WAIT_TIMEOUT_US, 4000000)
    bt.bt_qgemv_batched(probs, 4)
    torch.cuda.synchronize()
    assert bt.bt_last_device_error() == bt.BT_OK
    for (qw, x16), pr in zip(cases, probs):
        y_ref, a = O.qgemv(qw.codes, qw.scales, qw.biases, 4, O.decode_f16(x16[0]))
        assert_close(out_to_f64(pr[4], torch), y_ref, a, "f32", f"after timeout k={qw.k}")


@pytest.mark.parametrize("bits", BITS)
@pytest.mark.parametrize("k,count", [(1024, 7), (2048, 3), (3072, 29), (1024, 192)])
def test_qgemv_batched_matches_oracle(env, bits, k, count):
    """Independent GEMVs of one K in a single launch, ragged row counts."""
    torch, bt = env
    from dequant_gemv_gemm_bt_b300 import synth
    r = synth.rng_for("test", "batched", bits, k, count)
    ns = [int(v) for v in r.integers(1, 700, count)]
    ns[0] = 1
    cases, probs = [], []
    for i, n in enumerate(ns):
        qw = synth.make_qweight(r, n, k, bits)
        x16 = synth.draw_activations(r, 1, k, "f16")
        codes, scales, biases = to_dev(qw, torch)
        x = half_tensor(x16[0], "f16", torch)
        y = torch.full((n,), float("nan"), dtype=torch.float32, device="cuda")
        probs.append((codes, scales, biases, x, y))
        cases.append((qw, x16))
    bt.bt_qgemv_batched(probs, bits)
    torch.cuda.synchronize()
    assert bt.bt_last_device_error() == bt.BT_OK
    for (qw, x16), pr in zip(cases, probs):
        y_ref, a = O.qgemv(qw.codes, qw.scales, qw.biases, bits, O.decode_f16(x16[0]))
        assert_close(out_to_f64(pr[4], torch), y_ref, a, "f32", f"batched b={bits} n={qw.n}")


def test_qgemv_batched_rejects_bad_tables(env):
    torch, bt = env
    qw, x16 = make_case("batched-bad", 64, 1024, 4)
    codes, scales, biases = to_dev(qw, torch)
    x = half_tensor(x16[0], "f16", torch)
    y = torch.empty(64, device="cuda")
    with pytest.raises(bt.BTError):
        bt.bt_qgemv_batched([(codes, scales, biases, x, y)] * 257, 4)      # over the table capacity
    x2 = torch.zeros(2048, dtype=torch.float16, device="cuda")
    with pytest.raises(ValueError):
        bt.bt_qgemv_batched([(codes, scales, biases, x, y), (codes, scales, biases, x2, y)], 4)   # x/codes K differ
    assert bt.bt_last_device_error() == bt.BT_OK


def test_qgemv_batched_beyond_one_launch(env):
    """A mixed-K batch with k = 16384 (above what one batched launch stages) runs
    one launch per problem and still matches the oracle."""
    torch, bt = env
    cases, probs = [], []
    for tag, n, k in (("a", 64, 1024), ("b", 37, 16384), ("c", 300, 2048)):
        qw, x16 = make_case("batched-split-" + tag, n, k, 4)
        y = torch.full((n,), float("nan"), device="cuda")
        probs.append((*to_dev(qw, torch), half_tensor(x16[0], "f16", torch), y))
        cases.append((qw, x16))
    bt.bt_qgemv_batched(probs, 4)
    torch.cuda.synchronize()
    assert bt.bt_last_device_error() == bt.BT_OK
    for (qw, x16), pr in zip(cases, probs):
        y_ref, a = O.qgemv(qw.codes, qw.scales, qw.biases, 4, O.decode_f16(x16[0]))
        assert_close(out_to_f64(pr[4], torch), y_ref, a, "f32", f"batched fallback k={qw.k}")


@pytest.mark.parametrize("bits", BITS)
def test_qgemv_batched_mixed_k(env, bits):
    """Problems of different K in one launch (the warps sharing a row change between
    problems), in an order that alternates K so every CTA crosses several changes."""
    torch, bt = env
    from dequant_gemv_gemm_bt_b300 import synth
    r = synth.rng_for("test", "batched-mixed", bits)
    ks = [1024, 2048, 64, 3072, 1024, 8192, 576, 2048, 128, 1024, 4096, 3072] * 3
    cases, probs = [], []
    for i, k in enumerate(ks):
        n = int(r.integers(1, 900))
        qw = synth.make_qweight(r, n, k, bits)
        x16 = synth.draw_activations(r, 1, k, "f16")
        codes, scales, biases = to_dev(qw, torch)
        y = torch.full((n,), float("nan"), dtype=torch.float32, device="cuda")
        probs.append((codes, scales, biases, half_tensor(x16[0], "f16", torch), y))
        cases.append((qw, x16))
    bt.bt_qgemv_batched(probs, bits)
    torch.cuda.synchronize()
    assert bt.bt_last_device_error() == bt.BT_OK
    for (qw, x16), pr in zip(cases, probs):
        y_ref, a = O.qgemv(qw.codes, qw.scales, qw.biases, bits, O.decode_f16(x16[0]))
        assert_close(out_to_f64(pr[4], torch), y_ref, a, "f32", f"mixed b={bits} n={qw.n} k={qw.k}")


# One Llama-3.2-1B-shaped layer (hidden 2048): q/o 2048->2048, k/v 2048->512,
# gate/up 2048->8192, down 8192->2048 -- the bit-width sweep's projections.
LLAMA1B_LAYER = (("q", 2048, 2048), ("k", 512, 2048), ("v", 512, 2048), ("o", 2048, 2048),
                 ("gate", 8192, 2048), ("up", 8192, 2048), ("down", 2048, 8192))


@pytest.mark.parametrize("bits", BITS)
def test_qgemv_llama1b_layer_all_bits(env, bits):
    """Every projection of one full-size layer, batched per K as a decode pass runs them."""
    torch, bt = env
    from dequant_gemv_gemm_bt_b300 import synth
    r = synth.rng_for("test", "llama1b-layer", bits)
    cases = []
    for name, n, k in LLAMA1B_LAYER:
        qw = synth.make_qweight(r, n, k, bits)
        x16 = synth.draw_activations(r, 1, k, "f16")
        codes, scales, biases = to_dev(qw, torch)
        y = torch.full((n,), float("nan"), dtype=torch.float32, device="cuda")
        cases.append((name, qw, x16, (codes, scales, biases, half_tensor(x16[0], "f16", torch), y)))
    for k in (2048, 8192):
        bt.bt_qgemv_batched([c[3] for c in cases if c[1].k == k], bits)
    torch.cuda.synchronize()
    assert bt.bt_last_device_error() == bt.BT_OK
    for name, qw, x16, pr in cases:
        y_ref, a = O.qgemv(qw.codes, qw.scales, qw.biases, bits, O.decode_f16(x16[0]))
        assert_close(out_to_f64(pr[4], torch), y_ref, a, "f32", f"llama1b {name} b={bits}")


# ------------------------------------------------ the tensor-pipe GEMV (4-bit codes, fp16 x)
def run_opt(env, qw, x16, out_dtype="f32", cuda_core=False, shape=0):
    """The tensor-pipe kernel wherever it applies (kernel shape `shape`), or the CUDA-core kernel."""
    torch, bt = env
    try:
        bt.bt_set_option(bt.BT_OPT_GEMV_CUDA_CORE, 1 if cuda_core else 0)
        bt.bt_set_option(bt.BT_OPT_GEMV_TENSOR_PIPE, 2 if cuda_core else 1)
        bt.bt_set_option(bt.BT_OPT_GEMV_MMA_SHAPE, shape)
        return run(env, qw, x16, "f16", out_dtype)
    finally:
        bt.bt_set_option(bt.BT_OPT_GEMV_CUDA_CORE, 0)
        bt.bt_set_option(bt.BT_OPT_GEMV_TENSOR_PIPE, 0)
        bt.bt_set_option(bt.BT_OPT_GEMV_MMA_SHAPE, 0)


# kernel shapes: 0 the default diagonal consumer; 5, 6, 7 the four-column consumer
# (8 warps, 8 warps x 2 CTAs, 16 warps), which takes K multiples of 256 only
SHAPES = [0, 5, 6, 7]


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("n,k", [(16, 64), (8, 128), (24, 256), (1000, 1024), (2056, 2048), (520, 3072),
                                 (264, 4096), (136, 8192), (40, 576), (8, 512), (3000, 1280)])
def test_tensor_pipe_gemv_matches_oracle(env, n, k, shape):
    """16-row MMA tiles with ragged last tiles, K split over 1..8 warps, odd group counts."""
    torch, bt = env
    try:
        bt.bt_set_option(bt.BT_OPT_GEMV_TENSOR_PIPE, 1)
        assert bt.bt_plan_gemv(4, n, k)["tensor_pipe"] in (1, 2)
    finally:
        bt.bt_set_option(bt.BT_OPT_GEMV_TENSOR_PIPE, 0)
    qw, x = make_case("mma-gemv", n, k, 4)
    y = run_opt(env, qw, x, shape=shape)
    y_ref, a = O.qgemv(qw.codes, qw.scales, qw.biases, 4, O.decode_f16(x[0]))
    assert_close(y, y_ref, a, "f32", f"tensor pipe shape {shape} n={n} k={k}")
    if shape == 0:
        y_cc = run_opt(env, qw, x, cuda_core=True)
        assert_close(y_cc, y_ref, a, "f32", f"CUDA core n={n} k={k}")
    assert np.array_equal(y, run_opt(env, qw, x, shape=shape)), "tensor-pipe GEMV is not bitwise deterministic"


@pytest.mark.parametrize("shape", [0, 5])
@pytest.mark.parametrize("out", ["bf16", "f16"])
def test_tensor_pipe_gemv_output_dtypes(env, out, shape):
    qw, x = make_case("mma-gemv-dt", 1032, 2048, 4)
    y = run_opt(env, qw, x, out, shape=shape)
    y_ref, a = O.qgemv(qw.codes, qw.scales, qw.biases, 4, O.decode_f16(x[0]))
    assert_close(y, y_ref, a, out, f"tensor pipe shape {shape} -> {out}")


@pytest.mark.parametrize("shape", [0, 5])
def test_tensor_pipe_gemv_lm_head_sampled(env, shape):
    torch, bt = env
    from dequant_gemv_gemm_bt_b300 import synth
    r = synth.rng_for("test", "mma-lm-head")
    qw = synth.make_qweight(r, 151936, 1024, 4)
    x = synth.draw_activations(r, 1, 1024, "f16")
    y = run_opt(env, qw, x, shape=shape)
    rows = np.unique(np.concatenate([np.arange(0, 80), np.arange(151936 - 80, 151936), r.integers(0, 151936, 2000)]))
    y_ref, a = O.qgemv(qw.codes, qw.scales, qw.biases, 4, O.decode_f16(x[0]), rows=rows)
    assert_close(y[rows], y_ref, a, "f32", "tensor pipe lm_head")


@pytest.mark.parametrize("shape,ks", [
    (0, [1024, 3072, 2048, 128, 8192, 1024, 4096, 576, 3072, 64, 2048, 1024] * 3),
    (5, [1024, 3072, 2048, 256, 8192, 1024, 4096, 512, 3072, 768, 2048, 1024] * 3),
    (6, [1024, 3072, 2048, 256, 4096, 1024, 4096, 512, 3072, 768, 2048, 1024] * 3),   # 2 CTAs: K <= 4096 fits
    (7, [1024, 3072, 2048, 256, 8192, 1024, 4096, 512, 3072, 768, 2048, 1024] * 3)])
def test_tensor_pipe_batched_mixed_k(env, shape, ks):
    """One tensor-pipe launch over problems whose K split changes between neighbours
    (every CTA meets the barrier that re-stages x for a new problem)."""
    torch, bt = env
    from dequant_gemv_gemm_bt_b300 import synth
    r = synth.rng_for("test", "mma-batched", shape)
    shapes = [(8 * int(r.integers(1, 200)), k) for k in ks]
    bt.bt_set_option(bt.BT_OPT_GEMV_TENSOR_PIPE, 1)
    bt.bt_set_option(bt.BT_OPT_GEMV_MMA_SHAPE, shape)
    p, _ = bt.bt_plan_gemv_batch(4, shapes)
    assert p["tensor_pipe"] == (2 if shape >= 5 else 1)
    cases, probs = [], []
    for n, k in shapes:
        qw = synth.make_qweight(r, n, k, 4)
        x16 = synth.draw_activations(r, 1, k, "f16")
        codes, scales, biases = to_dev(qw, torch)
        y = torch.full((n,), float("nan"), dtype=torch.float32, device="cuda")
        probs.append((codes, scales, biases, half_tensor(x16[0], "f16", torch), y))
        cases.append((qw, x16))
    try:
        bt.bt_qgemv_batched(probs, 4)
        torch.cuda.synchronize()
    finally:
        bt.bt_set_option(bt.BT_OPT_GEMV_TENSOR_PIPE, 0)
        bt.bt_set_option(bt.BT_OPT_GEMV_MMA_SHAPE, 0)
    assert bt.bt_last_device_error() == bt.BT_OK
    for (qw, x16), pr in zip(cases, probs):
        y_ref, a = O.qgemv(qw.codes, qw.scales, qw.biases, 4, O.decode_f16(x16[0]))
        assert_close(out_to_f64(pr[4], torch), y_ref, a, "f32", f"tensor-pipe batch n={qw.n} k={qw.k}")
