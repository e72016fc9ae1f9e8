"""Grouped expert product and the MoE layer steps on the GPU against the oracle."""
import numpy as np
import pytest

import oracle.bt_oracle as O
from dequant_gemv_gemm_bt_b300 import synth
from helpers import assert_close, half_tensor, out_to_f64, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from dequant_gemv_gemm_bt_b300 import bt
    return torch, bt


def stacked(r, e, n, k, bits):
    ws = [synth.make_qweight(r, n, k, bits) for _ in range(e)]
    return (np.stack([w.codes for w in ws]), np.stack([w.scales for w in ws]), np.stack([w.biases for w in ws]))


def dev_stack(w, torch):
    return (torch.from_numpy(w[0].view(np.int32)).cuda(), torch.from_numpy(w[1].view(np.float16)).cuda(),
            torch.from_numpy(w[2].view(np.float16)).cuda())


@pytest.mark.parametrize("tokens,e,top_k", [(0, 8, 2), (1, 128, 8), (5, 7, 3), (128, 128, 8), (1000, 64, 4)])
def test_route_matches_oracle_bit_exact(env, tokens, e, top_k):
    torch, bt = env
    r = synth.rng_for("test", "route", tokens, e, top_k)
    ids, _ = synth.draw_routing(r, tokens, e, top_k)
    ids_t = torch.from_numpy(ids).cuda()
    off, pidx, prow, ptok = bt.bt_moe_route(ids_t, e, with_token=True)
    assert bt.bt_last_device_error() == bt.BT_OK
    np.testing.assert_array_equal(ptok.cpu().numpy(), pidx.cpu().numpy() // top_k)
    off_ref, order = O.route_sort(ids, e)
    np.testing.assert_array_equal(off.cpu().numpy(), off_ref)
    np.testing.assert_array_equal(pidx.cpu().numpy(), order)
    inv = np.empty_like(order)
    inv[order] = np.arange(order.size)
    np.testing.assert_array_equal(prow.cpu().numpy(), inv)


def test_route_rejects_bad_ids_on_device(env):
    torch, bt = env
    ids = torch.tensor([[0, 1], [5, 9]], dtype=torch.int32, device="cuda")   # 9 >= E
    off, pidx, prow = bt.bt_moe_route(ids, 8)
    assert bt.bt_last_device_error() == bt.BT_ERR_INVALID_ARG
    assert off.cpu().numpy()[-1] == 3
    assert bt.bt_last_device_error() == bt.BT_OK


@pytest.mark.parametrize("bits", (3, 4, 8))
@pytest.mark.parametrize("path", [0, 1, 2])
def test_moe_qgemm_grouped(env, bits, path):
    torch, bt = env
    r = synth.rng_for("test", "moe", bits)
    e, n, k = 6, 200, 512
    w = stacked(r, e, n, k, bits)
    offsets = np.array([0, 3, 3, 40, 41, 41, 97], dtype=np.int32)    # empty experts 1 and 4, one-row expert 3
    xb = synth.draw_activations(r, 97, k, "bf16")
    try:
        bt.bt_set_option(bt.BT_OPT_GEMM_PATH, path)
        y = bt.bt_moe_qgemm(*dev_stack(w, torch), bits, torch.from_numpy(offsets).cuda(),
                            half_tensor(xb, "bf16", torch), out_dtype=torch.bfloat16)
    finally:
        bt.bt_set_option(bt.BT_OPT_GEMM_PATH, 0)
    y_ref, a = O.moe_qgemm(*w, bits, offsets, O.decode_bf16(xb))
    assert_close(out_to_f64(y, torch), y_ref, a, "bf16", f"bits={bits} path={path}")


@pytest.mark.parametrize("bits", (3, 4, 6))
def test_moe_qgemm_gather_decode(env, bits):
    """Decode: one token, 8 distinct experts, rows gathered from the same x row."""
    torch, bt = env
    r = synth.rng_for("test", "moe-decode") if bits == 4 else synth.rng_for("test", "moe-decode", bits)
    e, n, k = 16, 384, 2048
    w = stacked(r, e, n, k, bits)
    ids, _ = synth.draw_routing(r, 1, e, 8)
    off, order = O.route_sort(ids, e)
    x16 = synth.draw_activations(r, 1, k, "f16")
    row_index = (order // 8).astype(np.int32)
    y = bt.bt_moe_qgemm(*dev_stack(w, torch), bits, torch.from_numpy(off.astype(np.int32)).cuda(),
                        half_tensor(x16, "f16", torch), x_row_index=torch.from_numpy(row_index).cuda(),
                        out_dtype=torch.float32)
    y_ref, a = O.moe_qgemm(*w, bits, off, O.decode_f16(x16)[row_index])
    assert_close(out_to_f64(y, torch), y_ref, a, "f32", "decode gather")


def test_swiglu_and_combine(env):
    torch, bt = env
    r = synth.rng_for("test", "swiglu")
    rows, inter = 37, 96
    a = r.standard_normal((rows, 2 * inter)).astype(np.float32)
    h = bt.bt_swiglu(torch.from_numpy(a).cuda(), out_dtype=torch.float32).cpu().numpy()
    want = O.silu(a[:, :inter].astype(np.float64)) * a[:, inter:]
    np.testing.assert_allclose(h, want, rtol=2e-6, atol=1e-6)
    tokens, top_k, hidden = 9, 3, 130
    yg = r.standard_normal((tokens * top_k, hidden)).astype(np.float32)
    gates = r.random((tokens, top_k)).astype(np.float32)
    perm = r.permutation(tokens * top_k).astype(np.int32)
    out = bt.bt_moe_combine(torch.from_numpy(yg).cuda(), torch.from_numpy(gates).cuda(),
                            torch.from_numpy(perm).cuda(), top_k, out_dtype=torch.float32).cpu().numpy()
    want = np.einsum("ts,tsh->th", gates.astype(np.float64), yg[perm].reshape(tokens, top_k, hidden))
    np.testing.assert_allclose(out, want, rtol=1e-5, atol=1e-5)


def run_layer_and_check(torch, bt, r, tokens, e, hdim, idim, top_k, bits, gu, down):
    """route -> gate|up (one grouped product, gathered rows) -> SwiGLU -> down ->
    combine on the GPU, each stage compared element by element with the oracle
    fed the GPU's own input to that stage (tolerances do not compound): routing
    bit-exact, products at the bound of their output type, SwiGLU at the bound
    of h's type against |h|, the fp32 combine at 1e-3 * sum |g * y|."""
    ids, gates = synth.draw_routing(r, tokens, e, top_k)
    xdt, tdt = ("f16", torch.float16) if tokens == 1 else ("bf16", torch.bfloat16)
    odt = "f16" if tokens == 1 else "bf16"
    xb = synth.draw_activations(r, tokens, hdim, xdt)
    x = half_tensor(xb, xdt, torch)
    off, pidx, prow, ptok = bt.bt_moe_route(torch.from_numpy(ids).cuda(), e, with_token=True)
    y_gu = bt.bt_moe_qgemm(*dev_stack(gu, torch), bits, off, x, x_row_index=ptok, out_dtype=tdt)
    h = bt.bt_swiglu(y_gu, out_dtype=tdt)
    y_d = bt.bt_moe_qgemm(*dev_stack(down, torch), bits, off, h, out_dtype=tdt)
    out = bt.bt_moe_combine(y_d, torch.from_numpy(gates).cuda(), prow, top_k, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert bt.bt_last_device_error() == bt.BT_OK
    off_ref, order = O.route_sort(ids, e)
    np.testing.assert_array_equal(off.cpu().numpy(), off_ref)
    np.testing.assert_array_equal(pidx.cpu().numpy(), order)
    gu_ref, gu_a = O.moe_qgemm(*gu, bits, off_ref, O.decode_half(xb, xdt)[order // top_k])
    y_gu_h = out_to_f64(y_gu, torch)
    assert_close(y_gu_h, gu_ref, gu_a, odt, "gate|up")
    h_ref, h_a = O.swiglu(y_gu_h)
    h_h = out_to_f64(h, torch)
    assert_close(h_h, h_ref, h_a, odt, "SwiGLU")
    d_ref, d_a = O.moe_qgemm(*down, bits, off_ref, h_h)
    y_d_h = out_to_f64(y_d, torch)
    assert_close(y_d_h, d_ref, d_a, odt, "down")
    out_ref, out_a = O.moe_combine(y_d_h, gates, order, top_k)
    assert_close(out_to_f64(out, torch), out_ref, out_a, "f32", "combine")
    return ids, gates, xb, out


@pytest.mark.parametrize("tokens", [1, 24])
def test_moe_layer_end_to_end(env, tokens):
    """A small layer stage by stage, then the whole layer against the fp64
    layer with every stage exact, under a bound derived from the rounding of
    the 16-bit intermediates."""
    torch, bt = env
    r = synth.rng_for("test", "moe-layer", tokens)
    e, hdim, idim, top_k, bits = 16, 256, 128, 4, 4
    gate_w, up_w, down_w = stacked(r, e, idim, hdim, bits), stacked(r, e, idim, hdim, bits), stacked(r, e, hdim, idim, bits)
    gu = tuple(np.concatenate([g, u], axis=1) for g, u in zip(gate_w, up_w))
    ids, gates, xb, out = run_layer_and_check(torch, bt, r, tokens, e, hdim, idim, top_k, bits, gu, down_w)
    xf = O.decode_half(xb, "f16" if tokens == 1 else "bf16")
    out_ref, h_ref, off_ref, order = O.moe_layer(xf, ids, gates, gate_w, up_w, down_w, bits)
    # Whole-layer bound, propagated to first order from the per-stage bounds the
    # staged checks hold (eps = 8e-3 of each product's A for 16-bit outputs, u16
    # the rounding of the stored h and Y_down): for h = silu(a) * b,
    #   dh <= |silu'(a)| |b| eps A_a + |silu(a)| eps A_b + u16 |h|,
    # then through the down product and the combine, with 50% slack for the
    # second-order terms.
    eps, u16 = 8e-3, (2.0 ** -11 if tokens == 1 else 2.0 ** -8)
    xg = xf[order // top_k]
    ga, ga_a = O.moe_qgemm(*gate_w, bits, off_ref, xg)
    ub, ub_a = O.moe_qgemm(*up_w, bits, off_ref, xg)
    sig = 1.0 / (1.0 + np.exp(-ga))
    dsilu = np.abs(sig * (1.0 + ga * (1.0 - sig)))
    dh = dsilu * np.abs(ub) * eps * ga_a + np.abs(O.silu(ga)) * eps * ub_a + u16 * np.abs(h_ref)
    _, prop = O.moe_qgemm(*down_w, bits, off_ref, dh)          # sum_i |W_down| dh_i
    d_exact, d_a = O.moe_qgemm(*down_w, bits, off_ref, h_ref)
    bound_rows = prop + eps * d_a + u16 * np.abs(d_exact)
    bound, _ = O.moe_combine(bound_rows, np.abs(gates), order, top_k)
    err = np.abs(out.cpu().numpy() - out_ref)
    lim = 1.5 * bound + 1e-5
    assert np.all(err <= lim), f"layer: worst err/bound {np.max(err / lim):.3g}"


@pytest.mark.parametrize("tokens", [1, 128])
def test_moe_layer_qwen3_30b_shapes(env, tokens):
    """Expert layer at the Qwen3-30B-A3B shapes (hidden 2048, 128 experts, gate/up
    2048->768, down 768->2048, top-8), every stage compared element by element."""
    torch, bt = env
    r = synth.rng_for("test", "moe30b", tokens)
    e, hdim, idim, top_k, bits = 128, 2048, 768, 8, 4
    gu = stacked(r, e, 2 * idim, hdim, bits)
    down = stacked(r, e, hdim, idim, bits)
    run_layer_and_check(torch, bt, r, tokens, e, hdim, idim, top_k, bits, gu, down)


@pytest.mark.parametrize("path", [1, 2])
def test_moe_qgemm_gather_prefill_paths(env, path):
    """Gathered rows (x_row_index) on both the CUDA-core and tensor-core grouped paths."""
    torch, bt = env
    r = synth.rng_for("test", "moe-gather", path)
    e, n, k, bits, t, top_k = 12, 256, 1024, 4, 40, 3
    w = stacked(r, e, n, k, bits)
    ids, _ = synth.draw_routing(r, t, e, top_k)
    off, order = O.route_sort(ids, e)
    xb = synth.draw_activations(r, t, k, "bf16")
    row_index = (order // top_k).astype(np.int32)
    try:
        bt.bt_set_option(bt.BT_OPT_GEMM_PATH, path)
        y = bt.bt_moe_qgemm(*dev_stack(w, torch), bits, torch.from_numpy(off.astype(np.int32)).cuda(),
                            half_tensor(xb, "bf16", torch), x_row_index=torch.from_numpy(row_index).cuda(),
                            out_dtype=torch.float32)
    finally:
        bt.bt_set_option(bt.BT_OPT_GEMM_PATH, 0)
    y_ref, a = O.moe_qgemm(*w, bits, off, O.decode_bf16(xb)[row_index])
    assert_close(out_to_f64(y, torch), y_ref, a, "f32", f"gather path {path}")
