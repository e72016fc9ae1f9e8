"""The Python binding checks every tensor against the sizes it passes to libbt
(no GPU needed): the C entry points take bare pointers, so a buffer smaller than
its sizes would otherwise reach a kernel.  CPU tensors with valid shapes get
through every size check and stop at the device check, so each case below
reads the message that stopped it."""
import pytest
import torch

CUDA = "must be a CUDA tensor"


@pytest.fixture(scope="module")
def bt():
    from dequant_gemv_gemm_bt_b300 import build
    build.build()
    from dequant_gemv_gemm_bt_b300 import bt as mod
    return mod


def weight(n, k, bits, experts=None):
    lead = () if experts is None else (experts,)
    return (torch.zeros(lead + (n, k * bits // 32), dtype=torch.int32),
            torch.zeros(lead + (n, k // 64), dtype=torch.float16),
            torch.zeros(lead + (n, k // 64), dtype=torch.float16))


def stopped_by(fn, text):
    with pytest.raises(ValueError) as e:
        fn()
    assert text in str(e.value), str(e.value)


@pytest.mark.parametrize("bits", (2, 3, 4, 6, 8))
def test_gemv_sizes(bt, bits):
    w = weight(300, 1024, bits)
    x = torch.zeros(1024, dtype=torch.float16)
    stopped_by(lambda: bt.bt_qgemv(*w, bits, x), CUDA)
    stopped_by(lambda: bt.bt_qgemv(*w, bits, x.view(1, 1024)), CUDA)
    stopped_by(lambda: bt.bt_qgemv(*w, bits, torch.zeros(2048, dtype=torch.float16)), "codes hold")
    stopped_by(lambda: bt.bt_qgemv(*w, bits, torch.zeros(2, 1024, dtype=torch.float16)), "one row")
    stopped_by(lambda: bt.bt_qgemv(w[0], w[1][:, :8], w[2], bits, x), "scales/biases must be")
    stopped_by(lambda: bt.bt_qgemv(w[0], w[1], w[2][:299], bits, x), "scales/biases must be")
    stopped_by(lambda: bt.bt_qgemv(*w, bits, x, torch.empty(299)), "too few")
    stopped_by(lambda: bt.bt_qgemv(w[0].float(), w[1], w[2], bits, x), "int32/uint32")
    stopped_by(lambda: bt.bt_qgemv(w[0], w[1].float(), w[2], bits, x), "16-bit")
    stopped_by(lambda: bt.bt_qgemv(w[0][None], w[1], w[2], bits, x), "2-D")


def test_gemm_sizes(bt):
    w = weight(256, 512, 4)
    x = torch.zeros(96, 512, dtype=torch.bfloat16)
    stopped_by(lambda: bt.bt_qgemm(*w, 4, x), CUDA)
    stopped_by(lambda: bt.bt_qgemm(*w, 4, x, torch.empty(96, 256, dtype=torch.bfloat16)), CUDA)
    stopped_by(lambda: bt.bt_qgemm(*w, 4, x, torch.empty(96, 255, dtype=torch.bfloat16)), "too few")
    stopped_by(lambda: bt.bt_qgemm(*w, 4, torch.zeros(512, dtype=torch.bfloat16)), "[M, K]")
    stopped_by(lambda: bt.bt_qgemm(*w, 4, torch.zeros(96, 1024, dtype=torch.bfloat16)), "codes hold")
    # row slices of a concatenated weight (q|k|v) are whole weights of their own
    big = weight(5120, 3072, 4)
    stopped_by(lambda: bt.bt_qgemm(big[0][3072:4096], big[1][3072:4096], big[2][3072:4096], 4,
                                   torch.zeros(128, 3072, dtype=torch.bfloat16)), CUDA)


def test_grouped_sizes(bt):
    w = weight(200, 512, 4, experts=6)
    off = torch.tensor([0, 3, 3, 40, 41, 41, 97], dtype=torch.int32)
    x = torch.zeros(97, 512, dtype=torch.bfloat16)
    stopped_by(lambda: bt.bt_moe_qgemm(*w, 4, off, x), CUDA)
    stopped_by(lambda: bt.bt_moe_qgemm(*w, 4, off.long(), x), "int32")
    stopped_by(lambda: bt.bt_moe_qgemm(*w, 4, off[:6], x), "needs 7")
    stopped_by(lambda: bt.bt_moe_qgemm(*w, 4, off, x, total_rows=98), "x holds 97 rows")
    stopped_by(lambda: bt.bt_moe_qgemm(*w, 4, off, x, torch.empty(97, 199)), "too few")
    stopped_by(lambda: bt.bt_moe_qgemm(*weight(200, 512, 4), 4, off, x), "3-D")
    # decode gather: one x row, eight routed rows
    wd = weight(384, 2048, 4, experts=16)
    off16 = torch.zeros(17, dtype=torch.int32)
    xd = torch.zeros(1, 2048, dtype=torch.float16)
    idx = torch.zeros(8, dtype=torch.int32)
    stopped_by(lambda: bt.bt_moe_qgemm(*wd, 4, off16, xd, x_row_index=idx), CUDA)
    stopped_by(lambda: bt.bt_moe_qgemm(*wd, 4, off16, xd, x_row_index=idx, total_rows=9), "needs 9")


def test_batched_sizes(bt):
    probs = []
    for n, k in ((64, 1024), (32, 2048), (7, 3072)):
        w = weight(n, k, 4)
        probs.append((*w, torch.zeros(k, dtype=torch.float16), torch.empty(n)))
    stopped_by(lambda: bt.bt_qgemv_batched(probs, 4), CUDA)
    bad = list(probs)
    bad[1] = probs[1][:4] + (torch.empty(31),)
    stopped_by(lambda: bt.bt_qgemv_batched(bad, 4), "problem 1")
    bad = list(probs)
    bad[2] = (probs[2][0], probs[2][1][:, :1]) + probs[2][2:]
    stopped_by(lambda: bt.bt_qgemv_batched(bad, 4), "problem 2: scales/biases")
    bad = list(probs)
    bad[2] = probs[2][:3] + (probs[2][3].bfloat16(), probs[2][4])
    stopped_by(lambda: bt.bt_qgemv_batched(bad, 4), "problem 2: every problem must share")


def test_routing_swiglu_combine_sizes(bt):
    ids = torch.zeros(5, 4, dtype=torch.int32)
    stopped_by(lambda: bt.bt_moe_route(ids, 16), CUDA)
    stopped_by(lambda: bt.bt_moe_route(ids, 16, with_token=True), CUDA)
    stopped_by(lambda: bt.bt_moe_route(ids.long(), 16), "int32")
    stopped_by(lambda: bt.bt_moe_route(ids, 16, offsets=torch.empty(16, dtype=torch.int32)), "needs 17")
    stopped_by(lambda: bt.bt_moe_route(ids, 16, pair_row=torch.empty(19, dtype=torch.int32)), "needs 20")
    a = torch.zeros(37, 192)
    stopped_by(lambda: bt.bt_swiglu(a), CUDA)
    stopped_by(lambda: bt.bt_swiglu(torch.zeros(37, 191)), "2*I")
    stopped_by(lambda: bt.bt_swiglu(a, torch.empty(37, 95)), "too few")
    yg = torch.zeros(27, 130)
    gates = torch.zeros(9, 3)
    prow = torch.zeros(27, dtype=torch.int32)
    stopped_by(lambda: bt.bt_moe_combine(yg, gates, prow, 3), CUDA)
    stopped_by(lambda: bt.bt_moe_combine(yg, gates.double(), prow, 3), "float32")
    stopped_by(lambda: bt.bt_moe_combine(yg, gates, prow, 4), "float32 [T, top_k]")
    stopped_by(lambda: bt.bt_moe_combine(yg, gates, prow[:26], 3), "needs 27")
    stopped_by(lambda: bt.bt_moe_combine(yg[:26], gates, prow, 3), "needs 27")
    stopped_by(lambda: bt.bt_moe_combine(yg, gates, prow, 3, torch.empty(9, 129)), "too few")
