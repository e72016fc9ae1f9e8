"""Fused expert-layer steps on the GPU against the fp64 oracle, through the C ABI:
the grouped gate|up product with the SwiGLU epilogue (every path), and the
routed-pair products that need no sort (decode)."""
import numpy as np
import pytest

import oracle.bt_oracle as O
from dequant_gemv_gemm_bt_b300 import synth
from helpers import assert_close, half_tensor, out_to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from dequant_gemv_gemm_bt_b300 import bt
    return torch, bt


def stacked(r, e, n, k, bits, g=64):
    ws = [synth.make_qweight(r, n, k, bits, group_size=g) for _ in range(e)]
    return tuple(np.stack([getattr(w, f) for w in ws]) for f in ("codes", "scales", "biases"))


def interleave(gate, up):
    """Gate/up weights [E][I][.] -> one [E][2I][.] matrix, row 2i = gate i, row 2i+1 = up i."""
    return tuple(np.stack([a, b], axis=2).reshape(a.shape[0], 2 * a.shape[1], a.shape[2]) for a, b in zip(gate, up))


def dev(w, torch):
    return (torch.from_numpy(w[0].view(np.int32)).cuda(), torch.from_numpy(w[1].view(np.float16)).cuda(),
            torch.from_numpy(w[2].view(np.float16)).cuda())


def swiglu_bound(y_ref, a_ref, rtol, u16):
    """Per-element bound of h = silu(gate) * up computed from a gate|up product whose
    elements are each within rtol * A of the exact ones, propagated to first order,
    plus the rounding u16 of the stored h.  y_ref/a_ref: [R, 2I] interleaved."""
    g, u = y_ref[:, 0::2], y_ref[:, 1::2]
    ag, au = a_ref[:, 0::2], a_ref[:, 1::2]
    sig = 1.0 / (1.0 + np.exp(-g))
    dsilu = np.abs(sig * (1.0 + g * (1.0 - sig)))
    h = O.silu(g) * u
    return h, 1.5 * rtol * (dsilu * np.abs(u) * ag + np.abs(O.silu(g)) * au) + u16 * np.abs(h) + 1e-5


def check_h(h_gpu, h_ref, bound, what):
    err = np.abs(h_gpu - h_ref)
    assert np.all(err <= bound), f"{what}: worst err/bound {np.max(err / bound):.3g}"


@pytest.mark.parametrize("bits", (3, 4, 8))
@pytest.mark.parametrize("path", [0, 1, 2, 3])
@pytest.mark.parametrize("hdt", ["bf16", "f32"])
def test_grouped_gate_up_swiglu(env, bits, path, hdt):
    torch, bt = env
    r = synth.rng_for("test", "fused-swiglu", bits)
    e, inter, k = 6, 96, 512
    gu = interleave(stacked(r, e, inter, k, bits), stacked(r, e, inter, k, bits))
    offsets = np.array([0, 3, 3, 40, 41, 41, 97], dtype=np.int32)      # empty experts, a one-row expert
    xb = synth.draw_activations(r, 97, k, "bf16")
    od = {"bf16": torch.bfloat16, "f32": torch.float32}[hdt]
    try:
        bt.bt_set_option(bt.BT_OPT_GEMM_PATH, path)
        h = bt.bt_moe_qgemm_swiglu(*dev(gu, torch), bits, torch.from_numpy(offsets).cuda(),
                                   half_tensor(xb, "bf16", torch), out_dtype=od)
        torch.cuda.synchronize()
    finally:
        bt.bt_set_option(bt.BT_OPT_GEMM_PATH, 0)
    assert bt.bt_last_device_error() == bt.BT_OK
    y_ref, a_ref = O.moe_qgemm(*gu, bits, offsets, O.decode_bf16(xb))
    rtol = O.RTOL["f32"] if hdt == "f32" else O.RTOL["bf16"]
    h_ref, bound = swiglu_bound(y_ref, a_ref, rtol, 2.0 ** -8 if hdt == "bf16" else 2.0 ** -24)
    check_h(out_to_f64(h, torch), h_ref, bound, f"swiglu b={bits} path={path} -> {hdt}")


def test_grouped_gate_up_swiglu_decode_gemv(env):
    """One row per routed expert (decode): the GEMV path with the epilogue."""
    torch, bt = env
    r = synth.rng_for("test", "fused-swiglu-decode")
    e, inter, k = 16, 384, 2048
    gu = interleave(stacked(r, e, inter, k, 4), stacked(r, e, inter, k, 4))
    ids, _ = synth.draw_routing(r, 1, e, 8)
    off, order = O.route_sort(ids, e)
    x16 = synth.draw_activations(r, 1, k, "f16")
    row_index = (order // 8).astype(np.int32)
    h = bt.bt_moe_qgemm_swiglu(*dev(gu, torch), 4, torch.from_numpy(off.astype(np.int32)).cuda(),
                               half_tensor(x16, "f16", torch), x_row_index=torch.from_numpy(row_index).cuda(),
                               out_dtype=torch.float16)
    torch.cuda.synchronize()
    assert bt.bt_last_device_error() == bt.BT_OK
    assert bt.bt_plan_gemm(4, 8, 2 * inter, k, num_experts=e, x_dtype=torch.float16)["path"] == "gemv"
    y_ref, a_ref = O.moe_qgemm(*gu, 4, off, O.decode_f16(x16)[row_index])
    h_ref, bound = swiglu_bound(y_ref, a_ref, O.RTOL["f32"], 2.0 ** -11)
    check_h(out_to_f64(h, torch), h_ref, bound, "decode swiglu")


def pairs_ref(w, bits, ids, xf):
    top_k = ids.shape[1]
    ys, As = [], []
    for pr, ex in enumerate(ids.reshape(-1)):
        y, a = O.qgemv(w[0][ex], w[1][ex], w[2][ex], bits, xf[pr // top_k])
        ys.append(y)
        As.append(a)
    return np.array(ys), np.array(As)


@pytest.mark.parametrize("tokens", [1, 3])
@pytest.mark.parametrize("bits", (4, 6))
def test_routed_pairs(env, tokens, bits):
    torch, bt = env
    r = synth.rng_for("test", "pairs", tokens, bits)
    e, n, k = 16, 520, 1024
    w = stacked(r, e, n, k, bits)
    ids, _ = synth.draw_routing(r, tokens, e, 8)
    x16 = synth.draw_activations(r, tokens, k, "f16")
    y = bt.bt_moe_qgemv_pairs(*dev(w, torch), bits, torch.from_numpy(ids).cuda(), half_tensor(x16, "f16", torch),
                              out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert bt.bt_last_device_error() == bt.BT_OK
    y_ref, a = pairs_ref(w, bits, ids, O.decode_f16(x16))
    assert_close(out_to_f64(y, torch), y_ref, a, "f32", f"pairs T={tokens} b={bits}")


@pytest.mark.parametrize("tokens", [1, 2])
def test_routed_pairs_swiglu(env, tokens):
    torch, bt = env
    r = synth.rng_for("test", "pairs-swiglu", tokens)
    e, inter, k = 16, 384, 2048
    gu = interleave(stacked(r, e, inter, k, 4), stacked(r, e, inter, k, 4))
    ids, _ = synth.draw_routing(r, tokens, e, 8)
    x16 = synth.draw_activations(r, tokens, k, "f16")
    h = bt.bt_moe_qgemv_pairs(*dev(gu, torch), 4, torch.from_numpy(ids).cuda(), half_tensor(x16, "f16", torch),
                              swiglu=True, out_dtype=torch.float16)
    torch.cuda.synchronize()
    assert bt.bt_last_device_error() == bt.BT_OK
    y_ref, a_ref = pairs_ref(gu, 4, ids, O.decode_f16(x16))
    h_ref, bound = swiglu_bound(y_ref, a_ref, O.RTOL["f32"], 2.0 ** -11)
    check_h(out_to_f64(h, torch), h_ref, bound, f"pairs swiglu T={tokens}")


def test_routed_pairs_bad_id_is_reported(env):
    torch, bt = env
    r = synth.rng_for("test", "pairs-bad")
    w = stacked(r, 4, 64, 256, 4)
    ids = torch.tensor([[0, 9]], dtype=torch.int32, device="cuda")      # 9 >= E
    x16 = synth.draw_activations(r, 1, 256, "f16")
    y = torch.full((2, 64), 7.0, dtype=torch.float32, device="cuda")
    bt.bt_moe_qgemv_pairs(*dev(w, torch), 4, ids, half_tensor(x16, "f16", torch), y)
    assert bt.bt_last_device_error() == bt.BT_ERR_INVALID_ARG
    assert torch.all(y[1] == 7.0)                                        # the bad pair's row is not written
    y_ref, a = pairs_ref(w, 4, np.array([[0]]), O.decode_f16(x16))
    assert_close(out_to_f64(y[:1], torch), y_ref, a, "f32", "good pair")
    assert bt.bt_last_device_error() == bt.BT_OK


def down_combine_ref(w, bits, ids, gates, hf):
    """Oracle: each pair's down product, then the gate-weighted combine; A = sum_s |g| A_pair."""
    top_k = ids.shape[1]
    ys, As = [], []
    for pr, ex in enumerate(ids.reshape(-1)):
        y, a = O.qgemv(w[0][ex], w[1][ex], w[2][ex], bits, hf[pr])
        ys.append(y)
        As.append(a)
    ys, As = np.array(ys), np.array(As)
    out, _ = O.moe_combine(ys, gates, np.arange(ids.size), top_k)
    a_tot, _ = O.moe_combine(As, np.abs(gates), np.arange(ids.size), top_k)
    return out, a_tot


@pytest.mark.parametrize("tokens", [1, 4])
@pytest.mark.parametrize("hdt", ["f16", "bf16"])
def test_down_combine(env, tokens, hdt):
    """Qwen3-30B-A3B-shaped down product of each token's 8 experts (768 -> 2048) with the
    gate-weighted combine in the kernel, against the oracle's per-pair products and combine."""
    torch, bt = env
    r = synth.rng_for("test", "down-combine", tokens, hdt)
    e, hid, inter, top_k = 128, 2048, 768, 8
    down = stacked(r, e, hid, inter, 4)
    ids, gates = synth.draw_routing(r, tokens, e, top_k)
    hb = synth.draw_activations(r, tokens * top_k, inter, hdt)
    out = bt.bt_moe_down_combine(*dev(down, torch), 4, torch.from_numpy(ids).cuda(), torch.from_numpy(gates).cuda(),
                                 half_tensor(hb, hdt, torch), out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert bt.bt_last_device_error() == bt.BT_OK
    out_ref, a = down_combine_ref(down, 4, ids, gates, O.decode_half(hb, hdt))
    assert_close(out_to_f64(out, torch), out_ref, a, "f32", f"down+combine T={tokens} h={hdt}")
    again = bt.bt_moe_down_combine(*dev(down, torch), 4, torch.from_numpy(ids).cuda(),
                                   torch.from_numpy(gates).cuda(), half_tensor(hb, hdt, torch),
                                   out_dtype=torch.float32)
    assert torch.equal(out, again), "down+combine is not deterministic"


def test_down_combine_bad_id_is_reported(env):
    torch, bt = env
    r = synth.rng_for("test", "down-combine-bad")
    e, hid, inter, top_k = 8, 256, 128, 2
    down = stacked(r, e, hid, inter, 4)
    ids = np.array([[1, 3], [2, 99]], dtype=np.int32)                  # token 1 routes to a missing expert
    gates = np.array([[0.25, 0.75], [0.5, 0.5]], dtype=np.float32)
    hb = synth.draw_activations(r, 4, inter, "f16")
    out = torch.full((2, hid), 7.0, dtype=torch.float32, device="cuda")
    bt.bt_moe_down_combine(*dev(down, torch), 4, torch.from_numpy(ids).cuda(), torch.from_numpy(gates).cuda(),
                           half_tensor(hb, "f16", torch), out)
    assert bt.bt_last_device_error() == bt.BT_ERR_INVALID_ARG
    assert torch.all(out[1] == 7.0)
    out_ref, a = down_combine_ref(down, 4, ids[:1], gates[:1], O.decode_f16(hb[:2]))
    assert_close(out_to_f64(out[:1], torch), out_ref, a, "f32", "good token")
    assert bt.bt_last_device_error() == bt.BT_OK


def test_decode_layer_in_two_launches(env):
    """Qwen3-30B-A3B-shaped expert layer for one decode token as two launches, no
    routing sort: routed pairs with the SwiGLU epilogue (gate|up), then the fused
    down + combine; each stage checked element by element with the oracle fed the
    GPU's own input to that stage."""
    torch, bt = env
    r = synth.rng_for("test", "decode-layer-2")
    e, hid, inter, top_k = 128, 2048, 768, 8
    gu = interleave(stacked(r, e, inter, hid, 4), stacked(r, e, inter, hid, 4))
    down = stacked(r, e, hid, inter, 4)
    ids, gates = synth.draw_routing(r, 1, e, top_k)
    x16 = synth.draw_activations(r, 1, hid, "f16")
    ids_t = torch.from_numpy(ids).cuda()
    h = bt.bt_moe_qgemv_pairs(*dev(gu, torch), 4, ids_t, half_tensor(x16, "f16", torch), swiglu=True,
                              out_dtype=torch.float16)
    out = bt.bt_moe_down_combine(*dev(down, torch), 4, ids_t, torch.from_numpy(gates).cuda(), h,
                                 out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert bt.bt_last_device_error() == bt.BT_OK
    y_ref, a_ref = pairs_ref(gu, 4, ids, O.decode_f16(x16))
    h_ref, bound = swiglu_bound(y_ref, a_ref, O.RTOL["f32"], 2.0 ** -11)
    h_gpu = out_to_f64(h, torch)
    check_h(h_gpu, h_ref, bound, "layer SwiGLU")
    out_ref, a = down_combine_ref(down, 4, ids, gates, h_gpu)
    assert_close(out_to_f64(out, torch), out_ref, a, "f32", "layer down+combine")
