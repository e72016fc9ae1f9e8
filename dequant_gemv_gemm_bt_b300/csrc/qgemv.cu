// Dequant-GEMV launch planning: per-shape choice of K split, rows in flight per
// warp, rows per pipeline stage and pipeline depth, keyed on (N, K, bits,
// problems) and the SM count.  BaseRT pages, gist.science "Metodologia"
// (kernel choice and threadgroup sizes picked per chip and core count).
#include "qgemv.cuh"

namespace bt {

cudaError_t launch_gemv_b2(const GemvParams&, const GemvPlan&, bt_dtype, const GemvBatch<kBatchCap>*, cudaStream_t);
cudaError_t launch_gemv_b3(const GemvParams&, const GemvPlan&, bt_dtype, const GemvBatch<kBatchCap>*, cudaStream_t);
cudaError_t launch_gemv_b4(const GemvParams&, const GemvPlan&, bt_dtype, const GemvBatch<kBatchCap>*, cudaStream_t);
cudaError_t launch_gemv_b6(const GemvParams&, const GemvPlan&, bt_dtype, const GemvBatch<kBatchCap>*, cudaStream_t);
cudaError_t launch_gemv_b8(const GemvParams&, const GemvPlan&, bt_dtype, const GemvBatch<kBatchCap>*, cudaStream_t);

namespace {
constexpr int kMaxNW = 8;               // consumer warps per CTA (as in the kernel)
constexpr int kStageBudget = 48 * 1024;
constexpr int kRingBudget = 176 * 1024;
constexpr size_t kMaxSmem = 227 * 1024;   // opt-in dynamic shared memory per block on sm_100/sm_103
}  // namespace

GemvPlan plan_gemv(int bits, bool fast, int N, int K, int problems, int num_experts, int sms) {
  GemvPlan pl{};
  pl.fast = fast;
  const int nchunks = K / 32;
  // Chunks of 32 codes per lane: the kernels exist for up to 4 (fast path) or 2
  // (generic).  One chunk per lane, with K split over up to 8 warps, measured
  // fastest on B300 at every K up to 8192: it keeps x in 32 registers, so two
  // CTAs (16 consumer warps) fit per SM, and the cross-warp partial sums are
  // cheap next to the latency hidden (e.g. Q4 K=8192: 3.7 vs 2.3 TB/s with 4
  // chunks per lane; K=3072 still gains with a quarter of its lanes idle).
  // 3 or 4 chunks per lane exist for the fast path of bits 2/4/8 only
  const bool wide = fast && (bits == 2 || bits == 4 || bits == 8);
  const int cpl_cap = wide ? 4 : 2;
  const int want_cpl = opts().gemv_max_cpl > 0 ? std::min(opts().gemv_max_cpl, cpl_cap) : 1;
  int kw = 1;
  while (kw < kMaxNW && (nchunks + 32 * kw - 1) / (32 * kw) > want_cpl) kw *= 2;
  int cpl = (nchunks + 32 * kw - 1) / (32 * kw);
  int nw = kMaxNW;
  if (kw > nw) {            // more than one chunk per lane: only 8 warps, so split K at most 8 ways
    kw = nw;
    cpl = (nchunks + 32 * kw - 1) / (32 * kw);
  }
  pl.kw = kw;
  pl.cpl = cpl;
  // the kernels exist for up to 4 chunks per lane on the fast path of bits 2/4/8 and 2 otherwise
  pl.feasible = cpl <= cpl_cap && kw <= nw && nw % kw == 0 && K <= 16 * 1024 * (wide ? 2 : 1);
  if (!pl.feasible) return pl;
  const int rw = nw / kw;
  const int G = K / kGroup;
  const int row_bytes = K * bits / 8;
  const int per_row = row_bytes + 4 * G;
  // smallest row multiple that keeps every bulk copy a multiple of 16 bytes (a power of two)
  int m = 1;
  while (((m * row_bytes) & 15) || ((m * G * 2) & 15)) m *= 2;
  // rows in flight per warp: as many as the stage budget and the per-SM row count allow
  const long long rows_total = (long long)N * problems;
  const long long per_sm = std::max<long long>(1, (rows_total + sms - 1) / sms);
  // rows in flight per warp: 8 with one chunk per lane (the 8-row lane reduction
  // takes 9 shuffles; decode pass 4.18 vs 3.81 TB/s with 4 rows), fewer as x
  // slices take more registers
  int ri = pl.cpl == 1 ? 8 : (pl.cpl == 2 ? 2 : 1);
  if (opts().gemv_ri > 0) ri = pl.cpl == 1 ? std::min(8, opts().gemv_ri) : std::min(ri, opts().gemv_ri);
  int stage_budget = opts().gemv_stage_kb > 0 ? opts().gemv_stage_kb * 1024 : kStageBudget;
  while (ri > 1 && ((long long)ri * rw * per_row > stage_budget || ri * rw > std::max<long long>(rw, per_sm))) ri /= 2;
  pl.ri = ri;
  const int ctas_per_sm = gemv_ctas_per_sm(pl.cpl, ri);   // must match the kernel's launch bounds
  // two stages of every resident CTA fit the SM's shared memory
  stage_budget = std::min<int>(stage_budget, (int)((kMaxSmem / ctas_per_sm - 1024) / 2));
  const int unit = std::max(ri * rw, m);
  int rb = unit * std::max(1, stage_budget / (unit * per_row));
  const long long want = ((per_sm + unit - 1) / unit) * unit;
  rb = (int)std::min<long long>(rb, std::max<long long>(unit, want));
  rb = std::min(rb, ((N + unit - 1) / unit) * unit);
  pl.rows_per_unit = rb;
  pl.row_bytes = row_bytes;
  const int stage = (rb * per_row + 127) / 128 * 128;
  pl.stage_bytes = stage;
  int stages = std::max(2, std::min(8, (kRingBudget / ctas_per_sm) / stage));
  if (opts().gemv_stages >= 2) stages = std::min(8, opts().gemv_stages);
  pl.stages = stages;
  pl.units_per_problem = (N + rb - 1) / rb;
  pl.num_units = (long long)pl.units_per_problem * problems;
  pl.grid = (int)std::min<long long>(pl.num_units, (long long)sms * ctas_per_sm);
  auto smem_for = [&](int st) {
    return (size_t)st * stage + 2 * st * sizeof(uint64_t) + (size_t)nw * 2 * ri * sizeof(float) +
           (size_t)(num_experts + 1) * sizeof(int);
  };
  while (pl.stages > 2 && smem_for(pl.stages) > kMaxSmem / ctas_per_sm) --pl.stages;
  pl.smem = smem_for(pl.stages);
  if (pl.smem > kMaxSmem) pl.feasible = false;
  return pl;
}

GemvPlan plan_gemv_batch(int bits, bool fast, GemvBatch<kBatchCap>& batch, int sms) {
  GemvPlan pl{};
  pl.fast = fast;
  pl.feasible = false;
  pl.cpl = 1;
  // rows in flight per warp: 8 unless some problem's row group would overflow a stage
  int ri = opts().gemv_ri > 0 ? std::min(8, opts().gemv_ri) : 8;
  int stage_budget = opts().gemv_stage_kb > 0 ? opts().gemv_stage_kb * 1024 : kStageBudget;
  for (int i = 0; i < batch.count; ++i) {
    const GemvProblem& q = batch.prob[i];
    if (q.k <= 0 || q.k % kGroup || q.k > 8 * 32 * 32) return pl;   // one chunk per lane needs K <= 8192
    const int nchunks = q.k / 32;
    int kw = 1;
    while (32 * kw < nchunks) kw *= 2;
    const int per_row = q.k * bits / 8 + 4 * (q.k / kGroup);
    while (ri > 1 && ri * (kMaxNW / kw) * per_row > stage_budget) ri /= 2;
  }
  const int ctas_per_sm = gemv_ctas_per_sm(1, ri);   // one chunk per lane (the kernel's launch bounds)
  // two stages of every resident CTA fit the SM's shared memory
  stage_budget = std::min<int>(stage_budget, (int)((kMaxSmem / ctas_per_sm - 1024) / 2));
  int stage = 0;
  for (int i = 0; i < batch.count; ++i) {
    GemvProblem& q = batch.prob[i];
    const int nchunks = q.k / 32;
    int kw = 1;
    while (32 * kw < nchunks) kw *= 2;
    q.kw = kw;
    q.g = q.k / kGroup;
    q.row_bytes = q.k * bits / 8;
    const int per_row = q.row_bytes + 4 * q.g;
    int m = 1;
    while (((m * q.row_bytes) & 15) || ((m * q.g * 2) & 15)) m *= 2;
    const int unit = std::max(ri * (kMaxNW / kw), m);
    int rb = unit * std::max(1, stage_budget / (unit * per_row));
    rb = std::min(rb, ((q.n + unit - 1) / unit) * unit);
    q.rb = rb;
    stage = std::max(stage, (rb * per_row + 127) / 128 * 128);
  }
  pl.ri = ri;
  pl.kw = batch.prob[0].kw;
  pl.rows_per_unit = batch.prob[0].rb;
  pl.row_bytes = batch.prob[0].row_bytes;
  pl.stage_bytes = stage;
  int stages = std::max(2, std::min(8, (kRingBudget / ctas_per_sm) / stage));
  if (opts().gemv_stages >= 2) stages = std::min(8, opts().gemv_stages);
  auto smem_for = [&](int st) {
    return (size_t)st * stage + 2 * st * sizeof(uint64_t) + (size_t)kMaxNW * 2 * ri * sizeof(float) + sizeof(int);
  };
  while (stages > 2 && smem_for(stages) > kMaxSmem / ctas_per_sm) --stages;
  pl.stages = stages;
  pl.smem = smem_for(stages);
  pl.grid = sms * ctas_per_sm;   // trimmed to the unit count at launch
  pl.feasible = pl.smem <= kMaxSmem;
  return pl;
}

cudaError_t launch_gemv(GemvParams& p, const GemvPlan& pl, int bits, bt_dtype xd, bt_dtype yd, cudaStream_t st,
                        GemvBatch<kBatchCap>* batch) {
  p.rows_per_unit = pl.rows_per_unit;
  p.row_bytes = pl.row_bytes;
  p.stage_bytes = pl.stage_bytes;
  p.stages = pl.stages;
  p.kw = pl.kw;
  p.units_per_problem = pl.units_per_problem;
  p.num_units = pl.num_units;
  p.y_dtype = yd;
  GemvPlan plb = pl;
  if (batch) {   // per-problem row blocks and their running offsets
    long long u = 0, cost = 0;
    for (int i = 0; i < batch->count; ++i) {
      GemvProblem& q = batch->prob[i];
      if (q.k == 0) {   // one K for the whole batch: the plan's geometry
        q.k = p.K;
        q.g = p.G;
        q.row_bytes = pl.row_bytes;
        q.kw = pl.kw;
        q.rb = pl.rows_per_unit;
      }
      q.units = (q.n + q.rb - 1) / q.rb;
      q.unit_begin = u;
      u += q.units;
      // CTAs take equal shares of work, not of units: a row split over kw warps
      // costs kw times a one-warp row (measured: K=2048 ~2.2x, K=3072 ~4x K=1024)
      q.cost_begin = cost;
      cost += (long long)q.n * q.kw;
    }
    p.total_cost = cost;
    p.num_units = u;
    plb.num_units = u;
    plb.grid = (int)std::min<long long>(u, (long long)sm_count() * gemv_ctas_per_sm(pl.cpl, pl.ri));
  }
  if (p.num_units == 0) return cudaSuccess;
  switch (bits) {
    case 2: return launch_gemv_b2(p, plb, xd, batch, st);
    case 3: return launch_gemv_b3(p, plb, xd, batch, st);
    case 4: return launch_gemv_b4(p, plb, xd, batch, st);
    case 6: return launch_gemv_b6(p, plb, xd, batch, st);
    default: return launch_gemv_b8(p, plb, xd, batch, st);
  }
}

}  // namespace bt
