"""Host-side GEMV launch heuristics (no GPU): invariants of every plan.

The planner maps (bits, N, K, problems, SM count) to a warp split, rows in
flight, pipeline geometry and grid.  These checks hold for any shape, so a
bad heuristic change is caught on CPU before it reaches a device.
"""
import bisect

import pytest

KMAX_SMEM = 227 * 1024
SM_SMEM = 228 * 1024


@pytest.fixture(scope="module")
def bt():
    from dequant_gemv_gemm_bt_b300 import build
    build.build()
    from dequant_gemv_gemm_bt_b300 import bt as mod
    return mod


def per_row(bits, k):
    return k * bits // 8 + 4 * (k // 64)


def check_plan(p, bits, n, k, problems, sms):
    assert p["feasible"] == 1
    if p["tensor_pipe"]:
        return check_tensor_pipe_plan(p, bits, n, k, problems, sms)
    kw, cpl, ri, rb = p["kw"], p["cpl"], p["ri"], p["rows_per_unit"]
    assert kw in (1, 2, 4, 8) and 8 % kw == 0                      # row groups tile the 8 consumer warps
    assert 32 * kw * cpl >= k // 32                                # every 32-code chunk has a lane
    assert ri in (1, 2, 4, 8)
    assert rb % ri == 0 and rb >= ri
    assert p["stage_bytes"] >= rb * per_row(bits, k)                # a unit fits its stage
    assert p["stage_bytes"] % 128 == 0
    assert p["stages"] >= 2
    assert p["smem_bytes"] <= KMAX_SMEM
    assert p["smem_bytes"] * p["ctas_per_sm"] <= SM_SMEM            # the resident CTAs fit the SM
    units = -(-n // rb) * problems
    assert p["num_units"] == units
    assert p["grid"] == min(units, sms * p["ctas_per_sm"])


def check_tensor_pipe_plan(p, bits, n, k, problems, sms):
    """The tensor-pipe kernel: 16-row MMA tiles, each warp's K slice at most 32
    groups (whole blocks of four groups for the four-column consumer), whole
    tiles per unit, one CTA per SM."""
    g = k // 64
    kw, rb = p["kw"], p["rows_per_unit"]
    assert bits == 4 and k <= 8192
    cols4 = p["tensor_pipe"] == 2
    split_units = g // 4 if cols4 else g                            # K is split in blocks or in groups
    if cols4:
        assert k % 256 == 0
    assert kw in (1, 2, 4, 8) and -(-g // kw) <= 32                 # at most 32 groups per warp
    assert kw <= max(1, split_units)
    tiles_per_sm = max(1, (-(-n * problems // sms)) // 16)
    if kw > 1 and -(-g // (kw // 2)) <= 32:                        # split further only to give idle warps work
        assert (kw // 2) * tiles_per_sm < 8 and kw <= split_units
    assert p["ri"] == 16 and rb % 16 == 0 and rb >= 16
    assert rb <= max(16, -(-n // 16) * 16)
    assert p["stage_bytes"] >= rb * per_row(bits, k) and p["stage_bytes"] % 128 == 0
    assert p["stages"] >= 2 and p["ctas_per_sm"] == 1
    # ring + barriers + row-group partials + x sums + permuted x (192 B per group) fit one CTA
    assert p["smem_bytes"] >= p["stages"] * p["stage_bytes"] + g * 192
    assert p["smem_bytes"] <= KMAX_SMEM
    units = -(-n // rb) * problems
    assert p["num_units"] == units
    assert p["grid"] == min(units, sms)
    assert (n * g * 2) % 16 == 0 and (n * k // 2) % 16 == 0         # every unit moves in 16-byte pieces


@pytest.fixture()
def tensor_pipe(bt):
    """Plans with the tensor-pipe GEMV taken wherever it applies (not only for small launches)."""
    bt.bt_set_option(bt.BT_OPT_GEMV_TENSOR_PIPE, 1)
    yield
    bt.bt_set_option(bt.BT_OPT_GEMV_TENSOR_PIPE, 0)


@pytest.fixture()
def cuda_core(bt):
    """Plans of the CUDA-core GEMV kernel (the tensor-pipe one switched off)."""
    bt.bt_set_option(bt.BT_OPT_GEMV_CUDA_CORE, 1)
    yield
    bt.bt_set_option(bt.BT_OPT_GEMV_CUDA_CORE, 0)


@pytest.mark.parametrize("k", (64, 128, 576, 1024, 2048, 3072, 4096, 8192))
@pytest.mark.parametrize("n", (16, 64, 333, 1024, 151936))
def test_tensor_pipe_plan_invariants(bt, tensor_pipe, k, n):
    p = bt.bt_plan_gemv(4, n, k)
    g = k // 64
    if (n * g * 2) % 16 or (n * k // 2) % 16:
        assert p["tensor_pipe"] == 0                                # a ragged unit could not move by bulk copy
    elif -(-n // 16) >= 8 * 148 and k % 256 == 0 and k <= 4096:
        assert p["tensor_pipe"] == 2                                # large launch: the four-column consumer
    else:
        assert p["tensor_pipe"] == 1
    check_plan(p, 4, n, k, 1, 148)


def test_tensor_pipe_applies_to_4_bit_fp16_dense_only(bt, tensor_pipe):
    import torch
    assert bt.bt_plan_gemv(4, 4096, 1024)["tensor_pipe"] == 1       # a few tiles per SM: the diagonal consumer
    assert bt.bt_plan_gemv(4, 65536, 1024)["tensor_pipe"] == 2      # many: the four-column consumer
    assert bt.bt_plan_gemv(4, 65536, 1088)["tensor_pipe"] == 1      # 17 groups: the diagonal consumer
    assert bt.bt_plan_gemv(4, 4096, 16384)["tensor_pipe"] == 0       # K above 8192
    assert bt.bt_plan_gemv(4, 4096, 1024, x_dtype=torch.bfloat16)["tensor_pipe"] == 0
    for bits in (2, 3, 6, 8):
        assert bt.bt_plan_gemv(bits, 4096, 1024)["tensor_pipe"] == 0
    p = bt.bt_plan_gemv(4, 151936, 1024)
    assert p["kw"] == 1 and p["grid"] == 148
    assert {k: bt.bt_plan_gemv(4, 65536, k)["kw"] for k in (1024, 2048, 3072, 4096, 8192)} == \
        {1024: 1, 2048: 1, 3072: 2, 4096: 2, 8192: 4}
    p = bt.bt_plan_gemv(4, 2048, 1024)                              # the single N=2048 GEMV: one tile per CTA
    assert p["kw"] == 8 and p["rows_per_unit"] == 16 and p["grid"] == 128
    try:
        bt.bt_set_option(bt.BT_OPT_GEMV_CUDA_CORE, 1)
        assert bt.bt_plan_gemv(4, 4096, 1024)["tensor_pipe"] == 0
    finally:
        bt.bt_set_option(bt.BT_OPT_GEMV_CUDA_CORE, 0)


def test_tensor_pipe_default_rule(bt):
    """Default rule: the diagonal consumer for launches of at most one 16-row tile
    per SM (the single N=2048 GEMV), the four-column consumer for launches of at
    least eight tiles per SM whose every K is a multiple of 256 and at most 4096,
    the CUDA-core kernel for the rest."""
    assert bt.bt_plan_gemv(4, 2048, 1024)["tensor_pipe"] == 1
    assert bt.bt_plan_gemv(4, 148 * 16, 1024)["tensor_pipe"] == 1
    assert bt.bt_plan_gemv(4, 148 * 16 + 16, 1024)["tensor_pipe"] == 0   # a few tiles per SM
    assert bt.bt_plan_gemv(4, 148 * 128 - 16, 1024)["tensor_pipe"] == 0
    assert bt.bt_plan_gemv(4, 148 * 128, 1024)["tensor_pipe"] == 2        # a tile per consumer warp
    assert bt.bt_plan_gemv(4, 151936, 1024)["tensor_pipe"] == 2
    assert bt.bt_plan_gemv(4, 151936, 1088)["tensor_pipe"] == 0     # 17 groups per row
    assert bt.bt_plan_gemv(4, 151936, 4096)["tensor_pipe"] == 2
    assert bt.bt_plan_gemv(4, 151936, 8192)["tensor_pipe"] == 0     # x of K = 8192 leaves small stages
    assert bt.bt_plan_gemv(6, 151936, 1024)["tensor_pipe"] == 0     # 4-bit codes only
    p, _ = bt.bt_plan_gemv_batch(4, QWEN06_LAYER * 28 + [(151936, 1024)])
    assert p["tensor_pipe"] == 2
    p, _ = bt.bt_plan_gemv_batch(4, QWEN06_LAYER * 28 + [(151936, 1088)])
    assert p["tensor_pipe"] == 0
    try:
        bt.bt_set_option(bt.BT_OPT_GEMV_TENSOR_PIPE, 2)
        assert bt.bt_plan_gemv(4, 2048, 1024)["tensor_pipe"] == 0
    finally:
        bt.bt_set_option(bt.BT_OPT_GEMV_TENSOR_PIPE, 0)


@pytest.mark.parametrize("bits", (2, 3, 4, 6, 8))
@pytest.mark.parametrize("k", (64, 128, 576, 1024, 2048, 3072, 4096, 8192, 16384))
@pytest.mark.parametrize("n", (1, 7, 333, 1024, 151936))
def test_single_plan_invariants(bt, bits, k, n):
    for cc in (0, 1):
        bt.bt_set_option(bt.BT_OPT_GEMV_CUDA_CORE, cc)
        try:
            single_plan_invariants(bt, bits, k, n)
        finally:
            bt.bt_set_option(bt.BT_OPT_GEMV_CUDA_CORE, 0)


def single_plan_invariants(bt, bits, k, n):
    for xdt, name in ((None, "f16"), ("bf16", "bf16")):
        import torch
        dt = torch.float16 if xdt is None else torch.bfloat16
        if k > 16384 and (bits in (3, 6) or name == "bf16"):
            continue
        p = bt.bt_plan_gemv(bits, n, k, x_dtype=dt, sms=148)
        check_plan(p, bits, n, k, 1, 148)


def test_one_chunk_per_lane_up_to_8192(bt, cuda_core):
    for k in (1024, 2048, 3072, 8192):
        p = bt.bt_plan_gemv(4, 151936, k)
        assert p["cpl"] == 1 and p["ctas_per_sm"] == 2
        assert p["kw"] == {1024: 1, 2048: 2, 3072: 4, 8192: 8}[k]
    p = bt.bt_plan_gemv(4, 151936, 16384)
    assert p["cpl"] == 2 and p["kw"] == 8 and p["ctas_per_sm"] == 1


def test_k_limits_per_bit_width(bt):
    """Two chunks per lane (K <= 16384) for 3- and 6-bit codes and for bf16 x; four (K <= 32768)
    for 2/4/8-bit codes with fp16 x.  Beyond that a single product runs on the CUDA-core tile."""
    import torch
    for bits in (2, 3, 4, 6, 8):
        assert bt.bt_plan_gemv(bits, 4096, 16384)["feasible"] == 1
        wide = bits in (2, 4, 8)
        p = bt.bt_plan_gemv(bits, 4096, 32768)
        assert p["feasible"] == (1 if wide else 0)
        assert bt.bt_plan_gemm(bits, 1, 4096, 32768, x_dtype=torch.float16)["path"] == ("gemv" if wide else "simt")
        p = bt.bt_plan_gemv(bits, 4096, 32768, x_dtype=torch.bfloat16)
        assert p["feasible"] == 0


def test_rows_in_flight_shrink_for_small_problems(bt, cuda_core):
    assert bt.bt_plan_gemv(4, 151936, 1024)["ri"] == 8
    p = bt.bt_plan_gemv(4, 4096, 1024)                             # 28 rows per SM: 2 rows in flight
    assert p["ri"] == 2 and p["ctas_per_sm"] == 3


def test_tuning_options_steer_the_plan(bt, cuda_core):
    try:
        bt.bt_set_option(bt.BT_OPT_GEMV_MAX_CPL, 4)
        assert bt.bt_plan_gemv(4, 4096, 2048)["cpl"] == 2
        bt.bt_set_option(bt.BT_OPT_GEMV_MAX_CPL, 0)
        bt.bt_set_option(bt.BT_OPT_GEMV_RI, 2)
        p = bt.bt_plan_gemv(4, 4096, 1024)
        assert p["ri"] == 2 and p["ctas_per_sm"] == 3
        check_plan(p, 4, 4096, 1024, 1, 148)
    finally:
        bt.bt_set_option(bt.BT_OPT_GEMV_MAX_CPL, 0)
        bt.bt_set_option(bt.BT_OPT_GEMV_RI, 0)


QWEN06_LAYER = [(2048, 1024), (1024, 1024), (1024, 1024), (1024, 2048), (3072, 1024), (3072, 1024), (1024, 3072)]


def unit_partition(geoms, grid):
    """Host restatement of the kernel's work split.  Unit b of a problem starts at
    work cost_begin + b*rb*w (work = rows x w: warps per row on the CUDA-core
    kernel, quantization groups per row on the tensor-pipe one); CTA i takes the units
    from the first one starting at or after C*i//grid up to the first one starting
    at or after C*(i+1)//grid.  Returns each CTA's work and the total."""
    starts, costs = [], []
    c = 0
    for n, kw, rb in geoms:
        for b in range(-(-n // rb)):
            starts.append(c + b * rb * kw)
            costs.append(min(rb, n - b * rb) * kw)
        c += n * kw
    total = c

    def unit_at(cost):
        return bisect.bisect_left(starts, cost)

    load, covered = [], 0
    for i in range(grid):
        u0, u1 = unit_at(total * i // grid), unit_at(total * (i + 1) // grid)
        assert u0 == covered                                          # ranges are contiguous and disjoint
        covered = u1
        load.append(sum(costs[u0:u1]))
    assert covered == len(starts)                                     # every unit has a CTA
    return load, total


def test_decode_pass_batch_plan_on_the_tensor_pipe(bt, tensor_pipe):
    """The Qwen3-0.6B-shaped pass as one tensor-pipe launch: K split 1/1/2 for
    K = 1024/2048/3072, whole 16-row tiles per unit, and the work-balanced split
    of units over one CTA per SM."""
    shapes = QWEN06_LAYER * 28 + [(151936, 1024)]
    p, geo = bt.bt_plan_gemv_batch(4, shapes)
    assert p["feasible"] == 1 and p["tensor_pipe"] == 2 and p["ctas_per_sm"] == 1 and p["ri"] == 16
    for (n, k), (kw, rb) in zip(shapes, geo):
        assert kw == {1024: 1, 2048: 1, 3072: 2}[k]
        assert rb % 16 == 0 and rb * per_row(4, k) <= p["stage_bytes"]
    assert p["stages"] >= 2 and p["smem_bytes"] <= KMAX_SMEM
    assert p["smem_bytes"] >= p["stages"] * p["stage_bytes"] + 48 * 192   # x of the largest K (48 groups)
    assert p["num_units"] == sum(-(-n // rb) for (n, _), (_, rb) in zip(shapes, geo))
    assert p["grid"] == 148
    load, total = unit_partition([(n, k // 64, rb) for (n, k), (_, rb) in zip(shapes, geo)], p["grid"])
    assert max(load) <= 1.1 * total / p["grid"]


def test_decode_pass_batch_plan_and_work_split(bt, cuda_core):
    """The same pass on the CUDA-core kernel."""
    shapes = QWEN06_LAYER * 28 + [(151936, 1024)]
    p, geo = bt.bt_plan_gemv_batch(4, shapes)
    assert p["feasible"] == 1 and p["cpl"] == 1 and p["ri"] == 8 and p["ctas_per_sm"] == 2
    for (n, k), (kw, rb) in zip(shapes, geo):
        assert kw == {1024: 1, 2048: 2, 3072: 4}[k]
        assert rb % (p["ri"] * (8 // kw)) == 0 or rb >= n              # whole row batches of every row group
        assert rb * per_row(4, k) <= p["stage_bytes"]
    assert p["smem_bytes"] * p["ctas_per_sm"] <= SM_SMEM
    assert p["num_units"] == sum(-(-n // rb) for (n, _), (_, rb) in zip(shapes, geo))
    load, total = unit_partition([(n, kw, rb) for (n, _), (kw, rb) in zip(shapes, geo)], p["grid"])
    mean = total / p["grid"]
    assert max(load) <= 1.1 * mean                                    # work, not unit count, is balanced


def test_mixed_batch_plan_infeasible_above_8192(bt):
    # one launch cannot hold a mixed batch with k > 8192 (bt_qgemv_batched then
    # runs one launch per problem)
    p, _ = bt.bt_plan_gemv_batch(4, [(64, 1024), (64, 16384)])
    assert p["feasible"] == 0
    with pytest.raises(bt.BTError):
        bt.bt_plan_gemv_batch(4, [(64, 100)])                       # K not a multiple of the group size


# ---------------------------------------------------------------- dense / grouped GEMM plans

SPLIT_CANDIDATES = (1, 2, 3, 4, 6, 8)


def test_gemm_path_choice(bt):
    assert bt.bt_plan_gemm(4, 1, 4096, 4096)["path"] == "gemv"
    for m in (2, 8):
        assert bt.bt_plan_gemm(4, m, 4096, 4096)["path"] == "mma"       # a few tokens: the weight-streaming kernel
    for m in (9, 15):
        assert bt.bt_plan_gemm(4, m, 4096, 4096)["path"] == "tc"
    assert bt.bt_plan_gemm(3, 2, 4096, 4096)["path"] == "tc"            # small-token kernel: 4-bit codes only
    assert bt.bt_plan_gemm(3, 8, 4096, 64 * 3)["path"] == "simt"        # Q3 K = 192: 72-byte rows, neither kernel
    for m in (16, 128, 4096):
        assert bt.bt_plan_gemm(4, m, 4096, 4096)["path"] == "tc"
    assert bt.bt_plan_gemm(3, 128, 4096, 4096)["path"] == "tc"          # Q3: stages hold aligned K-block pairs
    assert bt.bt_plan_gemm(3, 128, 4096, 64 * 63)["path"] == "simt"     # Q3 row of 24*63 B: no 16-B TMA stride
    assert bt.bt_plan_gemm(4, 128, 4096, 64 * 63)["path"] == "tc"       # odd group count
    p = bt.bt_plan_gemm(4, 128, 16384, 64 * 256)                        # 256 groups: more than one CTA stages
    assert p["path"] == "tc" and p["feasible"] == 1 and p["splits"] >= 2
    assert bt.bt_plan_gemm(4, 128, 16384, 32768)["splits"] >= 3          # 512 groups: at most 192 per split
    assert bt.bt_plan_gemm(2, 128, 4096, 64 * 2)["path"] == "tc"        # Q2 row of 32 B: TMA stride ok


@pytest.mark.parametrize("bits", (2, 4, 6, 8))
@pytest.mark.parametrize("m", (16, 33, 64, 100, 128, 129, 512, 2048))
@pytest.mark.parametrize("n,k", ((1024, 3072), (3072, 3072), (5120, 3072), (16384, 3072), (3072, 8192),
                                 (2048, 768), (4096, 128), (151936, 1024)))
def test_dense_tc_plan_invariants(bt, bits, m, n, k):
    sms = 148
    try:
        bt.bt_set_option(bt.BT_OPT_GEMM_PATH, 2)   # at M = 16 the small-token kernel would take 4-bit codes
        p = bt.bt_plan_gemm(bits, m, n, k, sms=sms)
    finally:
        bt.bt_set_option(bt.BT_OPT_GEMM_PATH, 0)
    assert p["path"] == "tc" and p["feasible"] == 1
    bn = p["bn"]
    assert bn == next((w for w in (32, 64, 128) if m <= w), 256)      # narrowest token tile that covers M
    assert p["grid_x"] == -(-n // 128) and p["grid_y"] == -(-m // bn)
    sp, kb = p["splits"], k // 64
    assert sp in SPLIT_CANDIDATES and p["grid_z"] == sp
    tiles = p["grid_x"] * p["grid_y"]
    if sp > 1:
        assert kb // sp >= 4 and tiles * sp <= sms * 85 // 100
    for bigger in (c for c in SPLIT_CANDIDATES if c > sp):              # the largest split that fits one wave
        assert kb // bigger < 4 or tiles * bigger > sms * 85 // 100
    assert p["k_blocks"] * sp >= kb and p["k_blocks"] <= -(-kb // sp) + 2   # near-even, even-aligned split
    assert 2 <= p["stages"] <= 12
    assert p["smem_bytes"] <= 227 * 1024


def test_prefill_gate_up_matches_the_captured_launch(bt):
    # The ncu capture of the Llama-3.2-3B-shaped gate|up launch (N=16384, K=3072,
    # M=128, Q4, bf16) recorded grid 128 x 1 x 1 and 210.2 kB of dynamic shared memory.
    p = bt.bt_plan_gemm(4, 128, 16384, 3072)
    assert (p["grid_x"], p["grid_y"], p["grid_z"]) == (128, 1, 1)
    assert p["smem_bytes"] == 210208


@pytest.mark.parametrize("m", (129, 256, 1024, 4096))
@pytest.mark.parametrize("experts", (8, 64, 128))
def test_grouped_tc_plan(bt, m, experts):
    try:
        bt.bt_set_option(bt.BT_OPT_GEMM_PATH, 2)
        p = bt.bt_plan_gemm(4, m, 1536, 2048, num_experts=experts)
    finally:
        bt.bt_set_option(bt.BT_OPT_GEMM_PATH, 0)
    assert p["path"] == "tc" and p["feasible"] == 1 and p["splits"] == 1
    mean = -(-m // experts)
    assert p["bn"] == next((w for w in (16, 32, 64) if mean <= w), 128)
    # (expert, token tile) slots: every expert's partial tile plus the full tiles
    assert p["grid_y"] == -(-m // p["bn"]) + min(experts, m)
    assert p["grid_x"] == 1536 // 128


def test_grouped_small_batches_run_the_gemv(bt):
    import torch
    assert bt.bt_plan_gemm(4, 0, 1536, 2048, num_experts=128)["path"] == "none"
    p = bt.bt_plan_gemm(4, 8, 1536, 2048, num_experts=128, x_dtype=torch.float16)
    assert p["path"] == "gemv"                                         # one row per routed expert: decode
    assert bt.bt_plan_gemm(4, 129, 1536, 2048, num_experts=128)["path"] == "mma"
    assert bt.bt_plan_gemm(4, 16 * 128, 1536, 2048, num_experts=128)["path"] == "mma"
    assert bt.bt_plan_gemm(4, 16 * 128 + 1, 1536, 2048, num_experts=128)["path"] == "tc"   # > 16 rows per expert


def small_expect(m, n, k, experts, nw, sms=148):
    """The small-token kernel's geometry restated for nw consumer warps: token tiles
    from the rows per weight, shrunk while x and its group sums exceed 112 KiB; row
    blocks of 16 * nw rows (one K box per stage), halved (and the boxes per stage
    doubled) while there are fewer row blocks than SMs, up to 8 boxes."""
    g = k // 64
    xts = g * 128 + 64
    t8 = -(-m // 8) if experts == 0 else min(4, max(1, (3 * -(-m // experts) // 2 + 7) // 8))
    while t8 > 1 and 8 * t8 * xts + 8 * t8 * g * 4 > 112 * 1024:
        t8 -= 1
    kw = 1
    while kw < 8 and -(-n // (16 * nw // kw)) * max(1, experts) < sms:
        kw *= 2
    rb = 16 * nw // kw
    return t8, kw, rb, min(-(-n // rb) * max(1, experts), sms)


@pytest.mark.parametrize("m,n,k,experts", [(1024, 1536, 2048, 128), (1024, 2048, 768, 128), (300, 1536, 2048, 128),
                                           (2, 4096, 4096, 0), (8, 3072, 3072, 0), (7, 1024, 3072, 0),
                                           (5, 151936, 1024, 0), (8, 16384, 3072, 0), (200, 512, 256, 16)])
@pytest.mark.parametrize("warps", [0, 8, 16])
def test_small_token_plan(bt, m, n, k, experts, warps):
    try:
        bt.bt_set_option(bt.BT_OPT_GEMM_SMALL_WARPS, warps)
        p = bt.bt_plan_gemm(4, m, n, k, num_experts=experts)
    finally:
        bt.bt_set_option(bt.BT_OPT_GEMM_SMALL_WARPS, 0)
    assert p["path"] == "mma" and p["feasible"] == 1
    nw = p["rows_per_unit"] * p["splits"] // 16          # rows per block x boxes per stage / 16
    assert nw == (warps or 16) or (warps == 0 and nw == 8)
    if warps == 0 and p["bn"] > 16:
        assert nw == 8                                                 # 3-4 token tiles: the 8-warp kernel
    t8, kw, rb, grid = small_expect(m, n, k, experts, nw)
    assert (p["bn"], p["splits"], p["rows_per_unit"], p["grid_x"]) == (8 * t8, kw, rb, grid)
    if experts == 0:
        assert p["bn"] >= m                                            # every dense row in one staging of x
    assert 2 <= p["stages"] <= 16 and p["smem_bytes"] <= 227 * 1024


def test_small_token_plan_limits(bt):
    assert bt.bt_plan_gemm(4, 8, 1004, 2048)["path"] != "mma"          # N not a multiple of 8
    assert bt.bt_plan_gemm(4, 8, 1024, 64 * 5)["path"] != "mma"        # K not a multiple of 256
    assert bt.bt_plan_gemm(8, 8, 1024, 2048)["path"] != "mma"          # 4-bit codes only
    assert bt.bt_plan_gemm(4, 33, 1024, 1024)["path"] == "tc"          # more than 8 dense rows
    try:
        bt.bt_set_option(bt.BT_OPT_GEMM_PATH, 3)
        assert bt.bt_plan_gemm(4, 32, 1024, 1024)["path"] == "mma"     # forced: up to 32 rows where x fits
        assert bt.bt_plan_gemm(4, 32, 1024, 4096)["path"] == "tc"      # 32 rows of x at K=4096 do not
    finally:
        bt.bt_set_option(bt.BT_OPT_GEMM_PATH, 0)


def test_gemm_plan_at_m1_is_the_gemv_plan(bt):
    import torch
    for n, k in ((4096, 4096), (151936, 1024), (1024, 3072)):
        g = bt.bt_plan_gemm(4, 1, n, k, x_dtype=torch.float16)
        v = bt.bt_plan_gemv(4, n, k, x_dtype=torch.float16)
        assert g["path"] == "gemv" and g["grid_x"] == v["grid"] and g["smem_bytes"] == v["smem_bytes"]


def test_gemm_options_steer_the_plan(bt):
    try:
        bt.bt_set_option(bt.BT_OPT_GEMM_PATH, 1)
        assert bt.bt_plan_gemm(4, 512, 4096, 4096)["path"] == "simt"
        bt.bt_set_option(bt.BT_OPT_GEMM_PATH, 2)
        assert bt.bt_plan_gemm(4, 4, 4096, 4096)["path"] == "tc"
        bt.bt_set_option(bt.BT_OPT_GEMM_PATH, 0)
        bt.bt_set_option(bt.BT_OPT_GEMM_SPLITS, 8)
        assert bt.bt_plan_gemm(4, 128, 16384, 3072)["splits"] == 8
        assert bt.bt_plan_gemm(4, 128, 4096, 64 * 6)["splits"] == 3   # at least two K blocks per split
    finally:
        bt.bt_set_option(bt.BT_OPT_GEMM_PATH, 0)
        bt.bt_set_option(bt.BT_OPT_GEMM_SPLITS, 0)


def test_gemm_plan_rejects_bad_sizes(bt):
    for args in ((4, 0, 64, 64), (4, 16, 0, 64), (4, 16, 64, 100), (4, 16, 64, -64)):
        with pytest.raises(bt.BTError):
            bt.bt_plan_gemm(*args)
    with pytest.raises(bt.BTError):
        bt.bt_plan_gemm(7, 16, 64, 64)
    with pytest.raises(bt.BTError):
        bt.bt_plan_gemm(4, 16, 64, 64 * 1024)                          # K above 32768
