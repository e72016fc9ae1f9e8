"""The small-token tensor-pipe kernel (mma.sync, tokens as the MMA's N) on the GPU
against the fp64 oracle, through the C ABI: dense products of 2..32 rows and grouped
expert products with a few rows per expert, fp16 and bf16 x, every output type held
to its own bound (1e-3*A for fp32, 8e-3*A for 16-bit outputs)."""
import numpy as np
import pytest

import oracle.bt_oracle as O
from dequant_gemv_gemm_bt_b300 import synth
from helpers import assert_close, half_tensor, make_case, out_to_f64, to_dev
from test_moe_fused_gpu import check_h, swiglu_bound

pytestmark = pytest.mark.gpu
OUT = {"f32": "float32", "bf16": "bfloat16", "f16": "float16"}


@pytest.fixture(scope="module")
def env():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from dequant_gemv_gemm_bt_b300 import bt
    return torch, bt


def forced(bt, fn):
    """Run fn with the small-token kernel forced (BT_OPT_GEMM_PATH = 3)."""
    try:
        bt.bt_set_option(bt.BT_OPT_GEMM_PATH, 3)
        return fn()
    finally:
        bt.bt_set_option(bt.BT_OPT_GEMM_PATH, 0)


def dense(env, m, n, k, xdtype, out, tag="small"):
    torch, bt = env
    xt_dtype = torch.bfloat16 if xdtype == "bf16" else torch.float16
    if forced(bt, lambda: bt.bt_plan_gemm(4, m, n, k, x_dtype=xt_dtype))["path"] != "mma":
        pytest.skip("x of these rows exceeds the kernel's staging")
    qw, x = make_case(tag, n, k, 4, m=m, xdtype=xdtype)
    codes, scales, biases = to_dev(qw, torch)
    xt = half_tensor(x, xdtype, torch)
    y = forced(bt, lambda: bt.bt_qgemm(codes, scales, biases, 4, xt, out_dtype=getattr(torch, OUT[out])))
    torch.cuda.synchronize()
    assert bt.bt_last_device_error() == bt.BT_OK
    y_ref, a = O.qgemm(qw.codes, qw.scales, qw.biases, 4, O.decode_half(x, xdtype))
    return out_to_f64(y, torch), y_ref, a


@pytest.mark.parametrize("xdtype", ["f16", "bf16"])
@pytest.mark.parametrize("m", [2, 3, 7, 8, 9, 15, 16])
@pytest.mark.parametrize("n,k", [(264, 256), (1032, 768), (200, 2048), (3072, 3072)])
def test_small_dense_matches_oracle(env, xdtype, m, n, k):
    y, y_ref, a = dense(env, m, n, k, xdtype, "f32")
    assert_close(y, y_ref, a, "f32", f"small m={m} n={n} k={k} {xdtype}")


@pytest.mark.parametrize("m,n,k", [(5, 264, 256), (8, 16384, 3072), (16, 1032, 768)])
def test_small_dense_eight_warps(env, m, n, k):
    torch, bt = env
    bt.bt_set_option(bt.BT_OPT_GEMM_SMALL_WARPS, 8)
    try:
        y, y_ref, a = dense(env, m, n, k, "bf16", "f32", tag="small-8w")
    finally:
        bt.bt_set_option(bt.BT_OPT_GEMM_SMALL_WARPS, 0)
    assert_close(y, y_ref, a, "f32", f"small 8 warps m={m} n={n} k={k}")


@pytest.mark.parametrize("xdtype,out", [("f16", "f16"), ("bf16", "bf16"), ("bf16", "f32"), ("f16", "bf16")])
def test_small_dense_out_dtypes(env, xdtype, out):
    y, y_ref, a = dense(env, 12, 520, 1024, xdtype, out, tag="small-dt")
    assert_close(y, y_ref, a, out, f"{xdtype}->{out}")


@pytest.mark.parametrize("m", [17, 24, 32])
def test_small_dense_forced_up_to_32_rows(env, m):
    """Up to four n8 token tiles in one staging of x (forced; the default takes the
    tensor cores above 16 rows)."""
    y, y_ref, a = dense(env, m, 512, 1024, "bf16", "f32", tag="small-32")
    assert_close(y, y_ref, a, "f32", f"small m={m}")


def test_small_dense_is_deterministic(env):
    torch, bt = env
    qw, x = make_case("small-det", 1536, 2048, 4, m=10, xdtype="bf16")
    codes, scales, biases = to_dev(qw, torch)
    xt = half_tensor(x, "bf16", torch)
    ys = [forced(bt, lambda: bt.bt_qgemm(codes, scales, biases, 4, xt, out_dtype=torch.float32)) for _ in range(3)]
    torch.cuda.synchronize()
    for y in ys[1:]:
        assert torch.equal(y, ys[0])


def stacked(r, e, n, k):
    ws = [synth.make_qweight(r, n, k, 4) for _ in range(e)]
    return (np.stack([w.codes for w in ws]), np.stack([w.scales for w in ws]), np.stack([w.biases for w in ws]))


def dev_stack(w, torch):
    return (torch.from_numpy(w[0].view(np.int32)).cuda(), torch.from_numpy(w[1].view(np.float16)).cuda(),
            torch.from_numpy(w[2].view(np.float16)).cuda())


@pytest.mark.parametrize("xdtype", ["f16", "bf16"])
@pytest.mark.parametrize("gather", [False, True])
@pytest.mark.parametrize("warps", [0, 8])
def test_small_grouped_row_counts(env, xdtype, gather, warps):
    """Experts with 0, 1, 7, 8, 9, 16, 17, 33 and 70 rows: partial n8 tiles, several
    tiles, and experts with more rows than one staging of x holds (walked in chunks);
    16 consumer warps (the default) and 8."""
    torch, bt = env
    bt.bt_set_option(bt.BT_OPT_GEMM_SMALL_WARPS, warps)
    try:
        grouped_row_counts(env, xdtype, gather)
    finally:
        bt.bt_set_option(bt.BT_OPT_GEMM_SMALL_WARPS, 0)


def grouped_row_counts(env, xdtype, gather):
    torch, bt = env
    r = synth.rng_for("test", "small-grouped", xdtype, gather)
    counts = [0, 1, 7, 8, 9, 16, 0, 17, 33, 70]
    e, n, k = len(counts), 264, 1024
    w = stacked(r, e, n, k)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    rows = int(offsets[-1])
    if gather:
        xb = synth.draw_activations(r, 50, k, xdtype)
        row_index = r.integers(0, 50, size=rows).astype(np.int32)
        xg = O.decode_half(xb, xdtype)[row_index]
        ri = torch.from_numpy(row_index).cuda()
    else:
        xb = synth.draw_activations(r, rows, k, xdtype)
        xg = O.decode_half(xb, xdtype)
        ri = None
    y = forced(bt, lambda: bt.bt_moe_qgemm(*dev_stack(w, torch), 4, torch.from_numpy(offsets).cuda(),
                                           half_tensor(xb, xdtype, torch), x_row_index=ri, total_rows=rows,
                                           out_dtype=torch.float32))
    torch.cuda.synchronize()
    assert bt.bt_last_device_error() == bt.BT_OK
    y_ref, a = O.moe_qgemm(*w, 4, offsets, xg)
    assert_close(out_to_f64(y, torch), y_ref, a, "f32", f"small grouped {xdtype} gather={gather}")


def test_small_grouped_swiglu(env):
    """Interleaved gate/up rows: the SwiGLU epilogue pairs rows 2i, 2i+1 (lanes 4 apart)."""
    torch, bt = env
    r = synth.rng_for("test", "small-swiglu")
    counts = [3, 0, 9, 16, 1, 12]
    e, n, k = len(counts), 2 * 136, 768
    w = stacked(r, e, n, k)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    rows = int(offsets[-1])
    xb = synth.draw_activations(r, rows, k, "bf16")
    h = forced(bt, lambda: bt.bt_moe_qgemm_swiglu(*dev_stack(w, torch), 4, torch.from_numpy(offsets).cuda(),
                                                  half_tensor(xb, "bf16", torch), out_dtype=torch.float32))
    torch.cuda.synchronize()
    assert bt.bt_last_device_error() == bt.BT_OK
    y_ref, a = O.moe_qgemm(*w, 4, offsets, O.decode_bf16(xb))
    h_ref, bound = swiglu_bound(y_ref, a, O.RTOL["f32"], 2.0 ** -24)
    check_h(out_to_f64(h, torch), h_ref, bound, "small grouped swiglu")


def test_small_grouped_default_takes_mma_for_moe_prefill(env):
    """The Qwen3-30B-shaped prefill (128 tokens x top-8 over 128 experts, ~8 rows per
    expert) takes the small-token kernel by default, and matches the oracle per element."""
    torch, bt = env
    r = synth.rng_for("test", "small-moe-prefill")
    e, n, k, t, top_k = 128, 1536, 2048, 128, 8
    assert bt.bt_plan_gemm(4, t * top_k, n, k, num_experts=e)["path"] == "mma"
    w = stacked(r, e, n, k)
    ids, _ = synth.draw_routing(r, t, e, top_k)
    off, order = O.route_sort(ids, e)
    xb = synth.draw_activations(r, t, k, "bf16")
    row_index = (order // top_k).astype(np.int32)
    y = bt.bt_moe_qgemm(*dev_stack(w, torch), 4, torch.from_numpy(off.astype(np.int32)).cuda(),
                        half_tensor(xb, "bf16", torch), x_row_index=torch.from_numpy(row_index).cuda(),
                        out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert bt.bt_last_device_error() == bt.BT_OK
    y_ref, a = O.moe_qgemm(*w, 4, off, O.decode_bf16(xb)[row_index])
    assert_close(out_to_f64(y, torch), y_ref, a, "f32", "Qwen3-30B-shaped gate|up, M=128")


@pytest.mark.parametrize("m", [1, 2, 3, 4, 5, 8, 12, 16, 20])
@pytest.mark.parametrize("xdtype", ["f16", "bf16"])
def test_qgemm_batched_matches_oracle(env, m, xdtype):
    """Several products of the same M in one call: one small-token launch for
    M <= 16 (the batched GEMV at M = 1, one launch per product above 16), each
    problem with its own K and N."""
    torch, bt = env
    shapes = [(264, 256), (1032, 1024), (96, 3072), (520, 768), (2048, 1024), (16, 2048)]
    probs, cases = [], []
    for i, (n, k) in enumerate(shapes):
        qw, x = make_case(f"qgemm-batched-{i}", n, k, 4, m=m, xdtype=xdtype)
        c, s, b = to_dev(qw, torch)
        y = torch.full((m, n), float("nan"), device="cuda")
        probs.append((c, s, b, half_tensor(x, xdtype, torch), y))
        cases.append((qw, x))
    bt.bt_qgemm_batched(probs, 4)
    torch.cuda.synchronize()
    assert bt.bt_last_device_error() == bt.BT_OK
    for (qw, x), pr in zip(cases, probs):
        y_ref, a = O.qgemm(qw.codes, qw.scales, qw.biases, 4, O.decode_half(x, xdtype))
        assert_close(out_to_f64(pr[4], torch), y_ref, a, "f32", f"batched m={m} n={qw.n} k={qw.k}")


@pytest.mark.parametrize("m", [2, 3, 4, 5, 8])
@pytest.mark.parametrize("out", ["f32", "f16", "bf16"])
def test_qgemm_batched_few_tokens_on_the_gemv(env, out, m):
    """M = 2..8 with fp16 x and every K a multiple of 256: one launch of the
    batched GEMV's four-column consumer (two tokens x four groups, four tokens
    x two groups or eight tokens x one group in the MMA's columns; M = 3 and 5
    leave token slots empty), with ragged 16-row tiles, mixed K up to 8192, a
    long problem spanning many CTAs, and bitwise-repeatable results."""
    torch, bt = env
    shapes = [(1000, 1024), (2056, 2048), (520, 3072), (264, 8192), (40000, 1024), (8, 512)]
    probs, cases = [], []
    odt = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[out]
    for i, (n, k) in enumerate(shapes):
        qw, x = make_case(f"qgemm-two-{i}", n, k, 4, m=m, xdtype="f16")
        c, s, b = to_dev(qw, torch)
        y = torch.full((m, n), float("nan"), device="cuda", dtype=odt)
        probs.append((c, s, b, half_tensor(x, "f16", torch), y))
        cases.append((qw, x))
    bt.bt_qgemm_batched(probs, 4)
    torch.cuda.synchronize()
    assert bt.bt_last_device_error() == bt.BT_OK
    first = [pr[4].clone() for pr in probs]
    for (qw, x), pr in zip(cases, probs):
        rows = None if qw.n <= 4096 else np.unique(np.linspace(0, qw.n - 1, 600).astype(np.int64))
        y_ref, a = O.qgemm(qw.codes, qw.scales, qw.biases, 4, O.decode_half(x, "f16"), rows=rows)
        y = out_to_f64(pr[4], torch)
        assert_close(y if rows is None else y[:, rows], y_ref, a, out, f"m={m} n={qw.n} k={qw.k}")
    for pr in probs:
        pr[4].fill_(float("nan"))
    bt.bt_qgemm_batched(probs, 4)
    torch.cuda.synchronize()
    for f, pr in zip(first, probs):
        assert torch.equal(f, pr[4]), "few-token GEMV is not bitwise repeatable"


@pytest.mark.parametrize("m", [2, 3, 8])
def test_qgemm_batched_few_tokens_fallback(env, m):
    """A table with a K that is not a multiple of 256 (576) cannot take the
    few-token GEMV: the call falls back (one product per launch) with the same
    results."""
    torch, bt = env
    shapes = [(264, 576), (1032, 1024)]
    probs, cases = [], []
    for i, (n, k) in enumerate(shapes):
        qw, x = make_case(f"qgemm-few-fb-{i}", n, k, 4, m=m, xdtype="f16")
        c, s, b = to_dev(qw, torch)
        y = torch.full((m, n), float("nan"), device="cuda")
        probs.append((c, s, b, half_tensor(x, "f16", torch), y))
        cases.append((qw, x))
    bt.bt_qgemm_batched(probs, 4)
    torch.cuda.synchronize()
    assert bt.bt_last_device_error() == bt.BT_OK
    for (qw, x), pr in zip(cases, probs):
        y_ref, a = O.qgemm(qw.codes, qw.scales, qw.biases, 4, O.decode_half(x, "f16"))
        assert_close(out_to_f64(pr[4], torch), y_ref, a, "f32", f"fallback m={m} n={qw.n} k={qw.k}")


def test_qgemm_batched_more_than_one_launch(env):
    """130 problems: more than one launch's table (120), results as one call."""
    torch, bt = env
    probs, cases = [], []
    for i in range(130):
        n, k = (8 + 8 * (i % 5), 256 * (1 + i % 3))
        n = max(n, 16)
        qw, x = make_case(f"qgemm-batched-many-{i}", n, k, 4, m=3, xdtype="f16")
        c, s, b = to_dev(qw, torch)
        y = torch.full((3, n), float("nan"), device="cuda")
        probs.append((c, s, b, half_tensor(x, "f16", torch), y))
        cases.append((qw, x))
    bt.bt_qgemm_batched(probs, 4)
    torch.cuda.synchronize()
    assert bt.bt_last_device_error() == bt.BT_OK
    for (qw, x), pr in zip(cases, probs):
        y_ref, a = O.qgemm(qw.codes, qw.scales, qw.biases, 4, O.decode_half(x, "f16"))
        assert_close(out_to_f64(pr[4], torch), y_ref, a, "f32", f"batched n={qw.n} k={qw.k}")
