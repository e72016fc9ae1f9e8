"""Shared test helpers: seeded inputs on host and device, oracle comparisons."""
import numpy as np

from dequant_gemv_gemm_bt_b300 import synth
import oracle.bt_oracle as O


def to_dev(qw, torch):
    """Packed weight (numpy) -> torch CUDA tensors (codes int32, scales/biases float16)."""
    codes = torch.from_numpy(qw.codes.view(np.int32)).cuda()
    scales = torch.from_numpy(qw.scales.view(np.float16)).cuda()
    biases = torch.from_numpy(qw.biases.view(np.float16)).cuda()
    return codes, scales, biases


def half_tensor(bits_u16, dtype, torch):
    t = torch.from_numpy(np.ascontiguousarray(bits_u16).view(np.int16)).cuda()
    return t.view(torch.float16 if dtype == "f16" else torch.bfloat16)


def out_to_f64(y, torch):
    return y.float().cpu().numpy().astype(np.float64)


def make_case(tag, n, k, bits, m=1, xdtype="f16"):
    r = synth.rng_for("test", tag, n, k, bits, m, xdtype)
    qw = synth.make_qweight(r, n, k, bits)
    x = synth.draw_activations(r, m, k, xdtype)
    return qw, x


def assert_close(y, y_ref, a, out_dtype, what=""):
    ok, ratio = O.within_tolerance(y, y_ref, a, out_dtype)
    assert ok, f"{what}: worst |err|/bound = {ratio:.3g}"
    return ratio
