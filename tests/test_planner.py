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


@pytest.mark.parametrize("bits", (2, 3, 4, 6, 8))
@pytest.mark.parametrize("k", (64, 128, 576, 1024, 2048, 3072, 4096, 8192, 16384))
@pytest.mark.parametrize("n", (1, 7, 333, 1024, 151936))
def test_single_plan_invariants(bt, bits, k, n):
    for xdt, name in ((None, "f16"), ("bf16", "bf16")):
        import torch
        dt = torch.float16 if xdt is None else torch.bfloat16
        if k > 16384 and (bits in (3, 6) or name == "bf16"):
            continue
        p = bt.bt_plan_gemv(bits, n, k, x_dtype=dt, sms=148)
        check_plan(p, bits, n, k, 1, 148)


def test_one_chunk_per_lane_up_to_8192(bt):
    for k in (1024, 2048, 3072, 8192):
        p = bt.bt_plan_gemv(4, 151936, k)
        assert p["cpl"] == 1 and p["ctas_per_sm"] == 2
        assert p["kw"] == {1024: 1, 2048: 2, 3072: 4, 8192: 8}[k]
    p = bt.bt_plan_gemv(4, 151936, 16384)
    assert p["cpl"] == 2 and p["kw"] == 8 and p["ctas_per_sm"] == 1


def test_rows_in_flight_shrink_for_small_problems(bt):
    assert bt.bt_plan_gemv(4, 151936, 1024)["ri"] == 8
    p = bt.bt_plan_gemv(4, 4096, 1024)                             # 28 rows per SM: 2 rows in flight
    assert p["ri"] == 2 and p["ctas_per_sm"] == 3


def test_tuning_options_steer_the_plan(bt):
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
    work cost_begin + b*rb*kw (work = rows x warps per row); CTA i takes the units
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


def test_decode_pass_batch_plan_and_work_split(bt):
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


def test_mixed_batch_rejects_k_above_8192(bt):
    p, _ = bt.bt_plan_gemv_batch(4, [(64, 1024), (64, 16384)])
    assert p["feasible"] == 0
    with pytest.raises(bt.BTError):
        bt.bt_plan_gemv_batch(4, [(64, 100)])                       # K not a multiple of the group size
