"""Pins of the fp64 oracle and of the layout writer against things other than themselves.

Each check is chosen so that a plausible slip in the oracle (a dropped bias
term, a wrong sign, a shifted bit, a transposed operand, a wrong group index)
fails at least one of them; ``test_planted_mistakes_are_caught`` plants such
slips in a copy of the oracle and confirms it.
"""
from fractions import Fraction
import os

import numpy as np
import pytest

from dequant_gemv_gemm_bt_b300 import synth
import oracle.bt_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "layout_fixtures.txt")
BITS = (2, 3, 4, 6, 8)


# ------------------------------------------------------------------ fixtures
def load_layout_fixtures():
    out = []
    cur = None
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, _, rest = line.partition(" ")
        if key == "fixture":
            cur = {"name": rest, "group": 64}
        elif key == "group":
            cur["group"] = int(rest)
        elif key == "bits":
            cur["bits"] = int(rest)
        elif key == "codes":
            kind, _, spec = rest.partition(" ")
            q = np.zeros(cur["group"], dtype=np.int64)
            if kind == "ramp":
                q = np.arange(cur["group"]) % int(spec)
            else:
                for item in spec.split():
                    j, v = item.split(":")
                    q[int(j)] = int(v)
            cur["codes"] = q
        elif key == "words":
            cur["words"] = np.array([int(h, 16) for h in rest.split()], dtype=np.uint32)
        elif key == "end":
            out.append(cur)
    return out


def brute_force_unpack(words: np.ndarray, bits: int, k: int):
    """Bit-by-bit from the little-endian byte array, pure Python."""
    by = bytes(np.ascontiguousarray(words, dtype="<u4").tobytes())
    out = []
    for j in range(k):
        v = 0
        for i in range(bits):
            t = j * bits + i
            bit = (by[t // 8] >> (t % 8)) & 1
            v |= bit << i
        out.append(v)
    return out


def frac_f16(u16) -> Fraction:
    """Exact rational value of an fp16 bit pattern, decoded field by field."""
    u = int(u16)
    sign = -1 if u >> 15 else 1
    e = (u >> 10) & 0x1F
    m = u & 0x3FF
    assert e != 31
    if e == 0:
        return sign * Fraction(m, 1 << 24)
    return sign * Fraction(1024 + m, 1) * Fraction(2) ** (e - 25)


def frac_bf16(u16) -> Fraction:
    u = int(u16)
    sign = -1 if u >> 15 else 1
    e = (u >> 7) & 0xFF
    m = u & 0x7F
    assert e != 255
    if e == 0:
        return sign * Fraction(m, 1) * Fraction(2) ** (-133)
    return sign * Fraction(128 + m, 1) * Fraction(2) ** (e - 134)


# --------------------------------------------------------------- layout pins
@pytest.mark.parametrize("fx", load_layout_fixtures(), ids=lambda f: f["name"])
def test_layout_fixture(fx):
    bits, q, words, g = fx["bits"], fx["codes"], fx["words"], fx["group"]
    assert words.size == g * bits // 32
    packed = synth.pack_codes(q[None, :], bits, g)
    np.testing.assert_array_equal(packed[0], words)
    np.testing.assert_array_equal(O.unpack_codes(words[None, :], bits, g, g)[0], q)
    assert brute_force_unpack(words, bits, g) == list(q)


@pytest.mark.parametrize("bits", (2, 3, 4, 5, 6, 8))
@pytest.mark.parametrize("g", (32, 128))
def test_brute_force_exact_other_group_sizes(bits, g):
    """Exact rational y = sum_k (s q + b) x at group sizes 32 and 128 (and 5-bit codes):
    each code read bit by bit, its group's fp16 scale and bias decoded field by field."""
    r = synth.rng_for("pins", "brute-g", bits, g)
    n, k = 3, 2 * g
    qw = synth.make_qweight(r, n, k, bits, group_size=g)
    x16 = synth.draw_activations(r, 1, k, "f16")[0]
    y, a = O.qgemv(qw.codes, qw.scales, qw.biases, bits, O.decode_f16(x16), group_size=g)
    for row in range(n):
        q = brute_force_unpack(qw.codes[row], bits, k)
        assert max(q) < 2 ** bits
        exact = sum((frac_f16(qw.scales[row, j // g]) * q[j] + frac_f16(qw.biases[row, j // g])) * frac_f16(x16[j])
                    for j in range(k))
        assert abs(y[row] - float(exact)) <= 1e-12 * max(1.0, a[row])


def test_fp16_weights_hand_example():
    """bits = 16: the codes are fp16 weights, two per word, low half first; no scale or bias."""
    words = np.array([[0x40003C00, 0x3800C000]], dtype=np.uint32)    # weights 1.0, 2.0, -2.0, 0.5
    x = np.array([1.0, 0.5, 0.25, -4.0])
    y, a = O.qgemv(words, None, None, 16, x, group_size=4)
    assert y[0] == 1.0 + 1.0 - 0.5 - 2.0 and a[0] == 1.0 + 1.0 + 0.5 + 2.0


def test_fp16_weights_brute_force():
    r = synth.rng_for("pins", "fp16-w")
    qw = synth.make_qweight(r, 4, 128, 16)
    x16 = synth.draw_activations(r, 1, 128, "f16")[0]
    y, _ = O.qgemv(qw.codes, qw.scales, qw.biases, 16, O.decode_f16(x16))
    halves = qw.codes.astype("<u4").view(np.uint16).reshape(4, 128)
    for row in range(4):
        exact = sum(frac_f16(halves[row, j]) * frac_f16(x16[j]) for j in range(128))
        assert abs(y[row] - float(exact)) <= 1e-12


@pytest.mark.parametrize("bits", BITS)
def test_all_ones_words_give_qmax(bits):
    words = np.full((3, 2 * bits * 2), 0xFFFFFFFF, dtype=np.uint32)
    q = O.unpack_codes(words, bits, 128)
    assert np.all(q == 2**bits - 1)


@pytest.mark.parametrize("bits", BITS)
def test_codes_in_range_and_brute_unpack(bits):
    r = synth.rng_for("pins", "range", bits)
    qw = synth.make_qweight(r, 5, 192, bits)
    q = O.unpack_codes(qw.codes, bits, 192)
    assert q.min() >= 0 and q.max() <= 2**bits - 1
    for n in range(5):
        assert brute_force_unpack(qw.codes[n], bits, 192) == list(q[n])


# --------------------------------------------------------- brute-force exact
@pytest.mark.parametrize("bits", BITS)
@pytest.mark.parametrize("k", [64, 128])
def test_brute_force_exact(bits, k):
    r = synth.rng_for("pins", "brute", bits, k)
    n = 7
    qw = synth.make_qweight(r, n, k, bits)
    x16 = synth.draw_activations(r, 1, k, "f16")[0]
    y, a = O.qgemv(qw.codes, qw.scales, qw.biases, bits, O.decode_f16(x16))
    xs = [frac_f16(v) for v in x16]
    for row in range(n):
        q = brute_force_unpack(qw.codes[row], bits, k)
        acc = Fraction(0)
        absacc = Fraction(0)
        for j in range(k):
            g = j // 64
            w = frac_f16(qw.scales[row, g]) * q[j] + frac_f16(qw.biases[row, g])
            acc += w * xs[j]
            absacc += abs(w * xs[j])
        assert abs(y[row] - float(acc)) <= 1e-12 * float(absacc) + 1e-300
        assert abs(a[row] - float(absacc)) <= 1e-12 * float(absacc)


def test_bf16_decode_exact():
    r = synth.rng_for("pins", "bf16")
    xb = synth.draw_activations(r, 1, 256, "bf16")[0]
    got = O.decode_bf16(xb)
    want = [float(frac_bf16(v)) for v in xb]
    np.testing.assert_array_equal(got, np.array(want))


def test_bf16_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    r = synth.rng_for("pins", "bf16-round")
    a = r.standard_normal(4096).astype(np.float32)
    a[:4] = [1.0 + 2**-8, 1.0 + 3 * 2**-8, -(1.0 + 2**-8), 0.0]  # ties to even
    want = torch.from_numpy(a).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(synth.f32_to_bf16_bits(a), want)


# ------------------------------------------------------------- invariants
@pytest.mark.parametrize("bits", BITS)
def test_one_hot_returns_column(bits):
    r = synth.rng_for("pins", "onehot", bits)
    n, k = 9, 192
    qw = synth.make_qweight(r, n, k, bits)
    w = O.dequant_weight(qw.codes, qw.scales, qw.biases, bits, k)
    for col in (0, 63, 64, 100, 191):
        x = np.zeros(k)
        x[col] = 1.0
        y, _ = O.qgemv(qw.codes, qw.scales, qw.biases, bits, x)
        np.testing.assert_array_equal(y, w[:, col])


@pytest.mark.parametrize("bits", BITS)
def test_grid_exact_roundtrip(bits):
    r = synth.rng_for("pins", "grid", bits)
    n, k = 6, 256
    w, q_true, s, beta = synth.grid_exact_weights(r, n, k, bits)
    q, s16, b16 = synth.quantize(w, bits)
    np.testing.assert_array_equal(q, q_true)
    np.testing.assert_array_equal(O.decode_f16(s16), s.astype(np.float64))
    np.testing.assert_array_equal(O.decode_f16(b16), beta.astype(np.float64))
    codes = synth.pack_codes(q, bits)
    np.testing.assert_array_equal(O.unpack_codes(codes, bits, k), q_true)
    wd = O.dequant_weight(codes, s16, b16, bits, k)
    np.testing.assert_array_equal(wd, w.astype(np.float64))


@pytest.mark.parametrize("bits", BITS)
def test_closed_form_all_qmax(bits):
    r = synth.rng_for("pins", "qmax", bits)
    n, k = 4, 320
    g = k // 64
    codes = np.full((n, k * bits // 32), 0xFFFFFFFF, dtype=np.uint32)
    s16 = synth.f32_to_f16_bits(r.uniform(0.001, 0.01, (n, g)))
    b16 = synth.f32_to_f16_bits(r.uniform(-0.05, 0.0, (n, g)))
    y, _ = O.qgemv(codes, s16, b16, bits, np.ones(k))
    want = (64 * (O.decode_f16(s16) * (2**bits - 1) + O.decode_f16(b16))).sum(axis=1)
    np.testing.assert_allclose(y, want, rtol=1e-14, atol=0)


@pytest.mark.parametrize("bits", BITS)
def test_closed_form_zero_scale(bits):
    r = synth.rng_for("pins", "s0", bits)
    n, k = 4, 256
    g = k // 64
    qw = synth.make_qweight(r, n, k, bits)
    s16 = np.zeros((n, g), dtype=np.uint16)
    x = O.decode_f16(synth.draw_activations(r, 1, k, "f16")[0])
    y, _ = O.qgemv(qw.codes, s16, qw.biases, bits, x)
    want = (O.decode_f16(qw.biases) * x.reshape(g, 64).sum(axis=1)[None, :]).sum(axis=1)
    np.testing.assert_allclose(y, want, rtol=1e-13, atol=1e-15)


def test_constant_group_quantizes_to_bias():
    w = np.full((2, 128), 0.0123, dtype=np.float32)
    for bits in BITS:
        q, s16, b16 = synth.quantize(w, bits)
        assert np.all(q == 0) and np.all(s16 == 0)
        wd = O.dequant_weight(synth.pack_codes(q, bits), s16, b16, bits, 128)
        np.testing.assert_array_equal(wd, np.float64(np.float16(0.0123)))


@pytest.mark.parametrize("bits", BITS)
def test_factored_form_matches_matmul(bits):
    """The per-group factored form s*sum(q x) + b*sum(x) equals the matmul definition."""
    r = synth.rng_for("pins", "factored", bits)
    m, n, k = 3, 11, 384
    g = k // 64
    qw = synth.make_qweight(r, n, k, bits)
    x = O.decode_bf16(synth.draw_activations(r, m, k, "bf16"))
    y, a = O.qgemm(qw.codes, qw.scales, qw.biases, bits, x)
    q = O.unpack_codes(qw.codes, bits, k).reshape(n, g, 64).astype(np.float64)
    xs = x.reshape(m, g, 64)
    qx = np.einsum("ngj,mgj->mng", q, xs)
    sx = xs.sum(axis=2)
    y2 = (O.decode_f16(qw.scales)[None] * qx + O.decode_f16(qw.biases)[None] * sx[:, None, :]).sum(2)
    np.testing.assert_allclose(y, y2, rtol=1e-12, atol=1e-12)
    assert np.all(a >= np.abs(y) - 1e-12)


def test_quantizer_error_bound():
    """Min/max quantization error is at most half a step (plus fp16 parameter rounding)."""
    r = synth.rng_for("pins", "qerr")
    w = synth.draw_weights(r, 16, 512)
    for bits in BITS:
        q, s16, b16 = synth.quantize(w, bits)
        wd = O.dequant_weight(synth.pack_codes(q, bits), s16, b16, bits, 512)
        step = np.repeat(O.decode_f16(s16), 64, axis=1)
        err = np.abs(wd - w.astype(np.float64))
        assert np.all(err <= 0.5 * step + 2e-3 * np.abs(w) + 1e-7)


# ------------------------------------------------------------------ MoE pins
def test_route_sort_stable_and_offsets():
    ids = np.array([[3, 0], [0, 2], [3, 1], [2, 0]])
    offsets, order = O.route_sort(ids, 5)
    np.testing.assert_array_equal(offsets, [0, 3, 4, 6, 8, 8])
    # expert 0: pairs (0,1)=1, (1,0)=2, (3,1)=7; expert 1: (2,1)=5; expert 2: 3, 6; expert 3: 0, 4
    np.testing.assert_array_equal(order, [1, 2, 7, 5, 3, 6, 0, 4])


def test_moe_qgemm_matches_per_expert_and_empty_experts():
    r = synth.rng_for("pins", "moe")
    e, n, k, bits = 4, 6, 128, 4
    ws = [synth.make_qweight(r, n, k, bits) for _ in range(e)]
    codes = np.stack([w.codes for w in ws])
    sc = np.stack([w.scales for w in ws])
    bi = np.stack([w.biases for w in ws])
    offsets = np.array([0, 2, 2, 5, 5])  # experts 1 and 3 empty
    x = O.decode_bf16(synth.draw_activations(r, 5, k, "bf16"))
    y, _ = O.moe_qgemm(codes, sc, bi, bits, offsets, x)
    for ex, (lo, hi) in enumerate(zip(offsets[:-1], offsets[1:])):
        if hi > lo:
            y_e, _ = O.qgemm(ws[ex].codes, ws[ex].scales, ws[ex].biases, bits, x[lo:hi])
            np.testing.assert_array_equal(y[lo:hi], y_e)


def test_moe_layer_single_slot_reduces_to_dense_chain():
    r = synth.rng_for("pins", "moe-layer")
    e, hdim, idim, bits, t = 3, 128, 64, 4, 5

    def stack(n, k):
        ws = [synth.make_qweight(r, n, k, bits) for _ in range(e)]
        return (np.stack([w.codes for w in ws]), np.stack([w.scales for w in ws]),
                np.stack([w.biases for w in ws]))
    gw, uw, dw = stack(idim, hdim), stack(idim, hdim), stack(hdim, idim)
    ids = np.array([[1], [0], [1], [2], [1]])
    gates = np.ones((t, 1))
    x = O.decode_bf16(synth.draw_activations(r, t, hdim, "bf16"))
    out, _, _, _ = O.moe_layer(x, ids, gates, gw, uw, dw, bits)
    for tok in range(t):
        ex = ids[tok, 0]
        g, _ = O.qgemv(gw[0][ex], gw[1][ex], gw[2][ex], bits, x[tok])
        u, _ = O.qgemv(uw[0][ex], uw[1][ex], uw[2][ex], bits, x[tok])
        hv = g / (1 + np.exp(-g)) * u
        d, _ = O.qgemv(dw[0][ex], dw[1][ex], dw[2][ex], bits, hv)
        np.testing.assert_allclose(out[tok], d, rtol=1e-12, atol=1e-14)


def test_routing_draw_is_distinct_and_normalized():
    r = synth.rng_for("pins", "routing")
    ids, gates = synth.draw_routing(r, 64, 128, 8)
    for row in ids:
        assert len(set(row.tolist())) == 8
    np.testing.assert_allclose(gates.sum(axis=1), 1.0, rtol=1e-6)


# ------------------------------------------------------- planted mistakes
def test_planted_mistakes_are_caught(monkeypatch):
    """Mutated oracles must fail the brute-force / invariant pins."""
    r = synth.rng_for("pins", "mutants")
    bits, n, k = 3, 5, 128
    qw = synth.make_qweight(r, n, k, bits)
    x = O.decode_f16(synth.draw_activations(r, 1, k, "f16")[0])
    y_good, a_good = O.qgemv(qw.codes, qw.scales, qw.biases, bits, x)

    def brute(row):
        q = brute_force_unpack(qw.codes[row], bits, k)
        return float(sum((frac_f16(qw.scales[row, j // 64]) * q[j] + frac_f16(qw.biases[row, j // 64]))
                         * Fraction(float(x[j])) for j in range(k)))
    want = np.array([brute(i) for i in range(n)])
    assert np.allclose(y_good, want, rtol=1e-12, atol=1e-14)

    real_unpack = O.unpack_codes
    real_deq = O.dequantize
    mutants = {
        "msb_first": lambda c, b, kk, g=64: real_unpack(c, b, kk, g)[:, ::-1].copy(),
        "dropped_bias": None,
        "wrong_group": None,
    }

    def deq_no_bias(q, s, b, g=64):
        return real_deq(q, s, np.zeros_like(b), g)

    def deq_shifted_group(q, s, b, g=64):
        return real_deq(q, np.roll(s, 1, axis=1), b, g)

    caught = 0
    for name in mutants:
        with monkeypatch.context() as mp:
            if name == "msb_first":
                mp.setattr(O, "unpack_codes", mutants[name])
            elif name == "dropped_bias":
                mp.setattr(O, "dequantize", deq_no_bias)
            else:
                mp.setattr(O, "dequantize", deq_shifted_group)
            y_bad, _ = O.qgemv(qw.codes, qw.scales, qw.biases, bits, x)
            if not np.allclose(y_bad, want, rtol=1e-9, atol=1e-12):
                caught += 1
    assert caught == len(mutants)


def silu_pins_hold(f) -> bool:
    """Values of x*sigma(x) fixed by the logistic function itself, not by a formula."""
    ln3 = np.log(3.0)
    x = np.linspace(-20.0, 20.0, 81)
    return bool(f(np.array([0.0]))[0] == 0.0
                and np.allclose(f(np.array([ln3, -ln3])), [0.75 * ln3, -0.25 * ln3], rtol=1e-15, atol=0)  # sigma(ln 3) = 3/4
                and np.allclose(f(-x), f(x) - x, rtol=1e-12, atol=1e-12)   # x*s(-x) = x*s(x) - x
                and np.allclose(f(np.array([60.0])), [60.0], rtol=1e-15, atol=0)   # s(x) -> 1
                and abs(f(np.array([-60.0]))[0]) < 1e-20)                  # s(x) -> 0


def test_silu_closed_forms():
    assert silu_pins_hold(O.silu)


def test_planted_silu_mistakes_are_caught():
    mutants = [lambda v: v / (1.0 + np.exp(v)),          # sign slip in the exponent
               lambda v: 1.0 / (1.0 + np.exp(-v)),       # sigmoid without the factor v
               lambda v: v * np.tanh(v),                 # a different gate
               lambda v: v / (1.0 + np.exp(-2.0 * v))]   # wrong slope
    assert not any(silu_pins_hold(f) for f in mutants)


def test_moe_combine_is_the_gate_weighted_sum_of_single_slot_layers():
    """Top-2 layer = g0 * layer(e0 alone) + g1 * layer(e1 alone); the single-slot layer is
    pinned to the dense chain above.  Also: slot order does not matter, gates act linearly."""
    r = synth.rng_for("pins", "moe-combine")
    e, hdim, idim, bits, t = 4, 128, 64, 4, 6

    def stack(n, k):
        ws = [synth.make_qweight(r, n, k, bits) for _ in range(e)]
        return (np.stack([w.codes for w in ws]), np.stack([w.scales for w in ws]),
                np.stack([w.biases for w in ws]))
    gw, uw, dw = stack(idim, hdim), stack(idim, hdim), stack(hdim, idim)
    ids, gates = synth.draw_routing(r, t, e, 2)
    gates = gates.astype(np.float64)
    x = O.decode_bf16(synth.draw_activations(r, t, hdim, "bf16"))
    out, _, _, _ = O.moe_layer(x, ids, gates, gw, uw, dw, bits)
    ones = np.ones((t, 1))
    s0, _, _, _ = O.moe_layer(x, ids[:, :1], ones, gw, uw, dw, bits)
    s1, _, _, _ = O.moe_layer(x, ids[:, 1:], ones, gw, uw, dw, bits)
    np.testing.assert_allclose(out, gates[:, :1] * s0 + gates[:, 1:] * s1, rtol=1e-12, atol=1e-14)
    swapped, _, _, _ = O.moe_layer(x, ids[:, ::-1], gates[:, ::-1], gw, uw, dw, bits)
    np.testing.assert_allclose(swapped, out, rtol=1e-12, atol=1e-14)
    scaled, _, _, _ = O.moe_layer(x, ids, 3.0 * gates, gw, uw, dw, bits)
    np.testing.assert_allclose(scaled, 3.0 * out, rtol=1e-12, atol=1e-14)


def test_moe_combine_hand_example():
    """Two tokens, top-2, rows placed out of pair order: each output is the
    gate-weighted sum of the rows its pairs were placed at (values by hand)."""
    y = np.array([[1.0, 2.0], [3.0, 4.0], [5.0, 6.0], [7.0, 8.0]])
    pair_index = np.array([2, 0, 3, 1])            # grouped row r holds pair pair_index[r]
    gates = np.array([[0.5, 0.25], [2.0, -1.0]])
    out, a = O.moe_combine(y, gates, pair_index, 2)
    # token 0: pairs 0 (row 1) and 1 (row 3); token 1: pairs 2 (row 0) and 3 (row 2)
    np.testing.assert_array_equal(out, [[3.25, 4.0], [-3.0, -2.0]])
    np.testing.assert_array_equal(a, [[3.25, 4.0], [7.0, 10.0]])


def test_swiglu_matches_silu_of_gate_times_up():
    gu = np.array([[0.0, np.log(3.0), 2.0, -1.0], [1.0, -2.0, 0.5, 4.0]])
    h, a = O.swiglu(gu)
    np.testing.assert_allclose(h[0], [0.0, -0.75 * np.log(3.0)], rtol=1e-15, atol=0)   # silu(ln 3) = 3/4 ln 3
    np.testing.assert_allclose(h[1], [0.5 * O.silu(np.array([1.0]))[0], 4.0 * O.silu(np.array([-2.0]))[0]],
                               rtol=1e-15)
    np.testing.assert_array_equal(a, np.abs(h))


def test_planted_combine_mistakes_are_caught(monkeypatch):
    """A combine that drops the gates or takes one slot only fails the pin above."""
    real = O.moe_layer

    def drop_gates(x, ids, gates, *a, **k):
        return real(x, ids, np.ones_like(gates), *a, **k)

    def first_slot(x, ids, gates, *a, **k):
        out, h, off, pidx = real(x, ids[:, :1], gates[:, :1], *a, **k)
        return out, h, off, pidx

    for bad in (drop_gates, first_slot):
        with monkeypatch.context() as mp:
            mp.setattr(O, "moe_layer", bad)
            with pytest.raises(AssertionError):
                test_moe_combine_is_the_gate_weighted_sum_of_single_slot_layers()


# ---------------------------------------------------------- the pass criterion
def test_pass_criterion_is_per_element():
    """|y - y_ref| <= rtol*A + 1e-5 element by element, with rtol 1e-3 for fp32
    outputs and 8e-3 for 16-bit outputs, and a NaN never passes."""
    assert O.RTOL["f32"] == 1e-3 and O.RTOL["bf16"] == 8e-3 and O.ATOL == 1e-5
    y_ref = np.array([1.0, -2.0, 0.0, 5.0])
    a = np.array([10.0, 4.0, 0.0, 1000.0])
    assert O.within_tolerance(y_ref.copy(), y_ref, a, "f32") == (True, 0.0)
    bound = 1e-3 * a + 1e-5
    for i in range(4):
        for scale, ok in ((0.99, True), (1.01, False)):
            for sign in (1.0, -1.0):
                y = y_ref.copy()
                y[i] += sign * scale * bound[i]
                got_ok, ratio = O.within_tolerance(y, y_ref, a, "f32")
                assert got_ok is ok and abs(ratio - scale) < 1e-6
    # a large A on one element does not loosen another's bound
    y = y_ref.copy()
    y[2] = 2e-5
    assert not O.within_tolerance(y, y_ref, a, "f32")[0]
    assert O.within_tolerance(y, y_ref, a * 0 + 1.0, "f32")[0]          # 2e-5 <= 1e-3*1 + 1e-5
    # 16-bit outputs take the wider bound
    y = y_ref.copy()
    y[0] += 0.05                                                        # 5e-3 * A: fails fp32, passes bf16
    assert not O.within_tolerance(y, y_ref, a, "f32")[0]
    assert O.within_tolerance(y, y_ref, a, "bf16")[0]
    y = y_ref.copy()
    y[1] = np.nan
    assert not O.within_tolerance(y, y_ref, a, "f32")[0]
    y = y_ref.copy()
    y[3] = np.inf
    assert not O.within_tolerance(y, y_ref, a, "f32")[0]
