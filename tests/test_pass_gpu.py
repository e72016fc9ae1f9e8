"""The decode pass object (bt_pass_create / bt_pass_run) on the GPU against the
fp64 oracle: chains of stages where a stage reads what the one before it wrote,
run several times over the same buffers with new inputs written in between
(the first run launches directly, later runs replay the recorded CUDA graph).
Each product is checked against the oracle on the input it actually read."""
import numpy as np
import pytest

import oracle.bt_oracle as O
from dequant_gemv_gemm_bt_b300 import synth
from helpers import assert_close, out_to_f64, to_dev

pytestmark = pytest.mark.gpu

# (name, n, k, input): "x0" is the pass input, anything else names the product whose y it reads
CHAIN = [
    [("q", 2048, 1024, "x0"), ("kv", 1024, 1024, "x0"), ("head", 4096, 1024, "x0")],
    [("o", 1024, 2048, "q"), ("gu", 3072, 1024, "kv")],
    [("down", 1024, 3072, "gu"), ("tail", 512, 1024, "o")],
]


@pytest.fixture(scope="module")
def env():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from dequant_gemv_gemm_bt_b300 import bt
    return torch, bt


def bits_of(t, torch):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def build_chain(torch, m, tag):
    weights, outs = {}, {}
    x0 = torch.empty((m, 1024), dtype=torch.float16, device="cuda")
    for stage in CHAIN:
        for name, n, k, _ in stage:
            qw = synth.make_qweight(synth.rng_for("pass", tag, name, n, k), n, k, 4)
            weights[name] = (qw, to_dev(qw, torch))
            outs[name] = torch.empty((m, n), dtype=torch.float16, device="cuda")
    bufs = dict(outs, x0=x0)
    stages = [[(*weights[name][1], bufs[src], outs[name]) for name, _, _, src in stage] for stage in CHAIN]
    return weights, bufs, stages


def check_chain(torch, weights, bufs, what):
    for stage in CHAIN:
        for name, _, _, src in stage:
            qw = weights[name][0]
            x = O.decode_half(bits_of(bufs[src], torch), "f16")
            assert np.isfinite(x).all(), f"{what}: input of {name} is not finite"
            y_ref, a = O.qgemm(qw.codes, qw.scales, qw.biases, 4, x)
            assert_close(out_to_f64(bufs[name], torch), y_ref, a, "f16", f"{what} {name}")


def new_input(torch, bufs, m, seed):
    x = synth.draw_activations(synth.rng_for("pass-x", m, seed), m, 1024, "f16")
    bufs["x0"].copy_(torch.from_numpy(x.view(np.int16)).view(torch.float16))


@pytest.mark.parametrize("pdl", [0, 1])
@pytest.mark.parametrize("m", [1, 2, 4, 24])
def test_pass_chain_runs_match_oracle(env, m, pdl):
    """Three dependent stages: M = 1 on the batched GEMV, M = 2 and 4 on its
    few-token forms, M = 24 one tensor-core product per launch; with and
    without PDL (and the constant-weights prefetch that PDL allows)."""
    torch, bt = env
    weights, bufs, stages = build_chain(torch, m, f"chain{m}")
    dp = bt.bt_pass_create(stages, 4)
    bt.bt_set_option(bt.BT_OPT_PDL, pdl)   # the first run records the options in force
    bt.bt_set_option(bt.BT_OPT_CONST_WEIGHTS, pdl)
    try:
        for run in range(4):
            new_input(torch, bufs, m, run)
            for name, t in bufs.items():   # a stage that read a stale or unwritten buffer shows NaN
                if name != "x0":
                    t.fill_(float("nan"))
            dp.run()
            torch.cuda.synchronize()
            assert bt.bt_last_device_error() == bt.BT_OK
            check_chain(torch, weights, bufs, f"m={m} pdl={pdl} run {run}")
    finally:
        bt.bt_set_option(bt.BT_OPT_PDL, 0)
        bt.bt_set_option(bt.BT_OPT_CONST_WEIGHTS, 0)
        dp.close()


@pytest.mark.parametrize("m,count", [(1, 300), (4, 130)])
def test_pass_stage_beyond_one_launch(env, m, count):
    """A stage with more products than one launch's table (256 GEMV problems, 120
    small-token problems) takes several launches inside the recorded graph."""
    torch, bt = env
    shapes = [(64, 256), (136, 512), (8, 1024), (264, 256)]
    ws = []
    for i, (n, k) in enumerate(shapes):
        qw = synth.make_qweight(synth.rng_for("pass-many", i, n, k), n, k, 4)
        ws.append((qw, to_dev(qw, torch)))
    xs, ys, probs = [], [], []
    for i in range(count):
        qw, dev = ws[i % len(shapes)]
        x = synth.draw_activations(synth.rng_for("pass-many-x", m, i), m, qw.k, "f16")
        xt = torch.from_numpy(x.view(np.int16)).cuda().view(torch.float16)
        yt = torch.empty((m, qw.n), dtype=torch.float32, device="cuda")
        xs.append(x)
        ys.append(yt)
        probs.append((*dev, xt, yt))
    dp = bt.bt_pass_create([probs], 4)
    try:
        for run in range(2):
            for yt in ys:
                yt.fill_(float("nan"))
            dp.run()
            torch.cuda.synchronize()
            assert bt.bt_last_device_error() == bt.BT_OK
            for i in range(count):
                qw = ws[i % len(shapes)][0]
                y_ref, a = O.qgemm(qw.codes, qw.scales, qw.biases, 4, O.decode_half(xs[i], "f16"))
                assert_close(out_to_f64(ys[i], torch), y_ref, a, "f32", f"run {run} product {i}")
    finally:
        dp.close()


def test_pass_run_on_side_stream_and_errors(env):
    """Runs on a caller stream; a destroyed pass is refused by the binding, a pass
    with a bad product is refused at creation."""
    torch, bt = env
    weights, bufs, stages = build_chain(torch, 1, "side")
    dp = bt.bt_pass_create(stages, 4)
    s = torch.cuda.Stream()
    for run in range(2):
        new_input(torch, bufs, 1, 10 + run)
        s.wait_stream(torch.cuda.current_stream())
        dp.run(stream=s)
        s.synchronize()
        check_chain(torch, weights, bufs, f"side stream run {run}")
    dp.close()
    with pytest.raises(ValueError):
        bt.bt_pass_run(dp)
    shifted = torch.empty(2048 + 1, dtype=torch.float16, device="cuda")[1:].view(1, 2048)   # not 16-byte aligned
    bad = [list(stages[0]), [(*stages[1][0][:3], shifted, stages[1][0][4])]]
    with pytest.raises((ValueError, RuntimeError)):
        bt.bt_pass_create(bad, 4)
