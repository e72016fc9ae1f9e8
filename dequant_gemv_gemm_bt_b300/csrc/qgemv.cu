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
cudaError_t launch_gemv_b5(const GemvParams&, const GemvPlan&, bt_dtype, const GemvBatch<kBatchCap>*, cudaStream_t);
cudaError_t launch_gemv_b8(const GemvParams&, const GemvPlan&, bt_dtype, const GemvBatch<kBatchCap>*, cudaStream_t);
cudaError_t launch_gemv_b16(const GemvParams&, const GemvPlan&, bt_dtype, const GemvBatch<kBatchCap>*, cudaStream_t);
cudaError_t launch_gemv_mma_b4(const GemvParams&, const GemvPlan&, const GemvBatch<kBatchCap>*, cudaStream_t);

namespace {
constexpr int kMaxNW = 8;               // consumer warps per CTA (as in the kernel)
constexpr int kStageBudget = 48 * 1024;
constexpr int kRingBudget = 176 * 1024;
constexpr size_t kMaxSmem = 227 * 1024;   // opt-in dynamic shared memory per block on sm_100/sm_103
}  // namespace

GemvPlan plan_gemv(int bits, bool fast, int N, int K, int problems, int num_experts, int sms, int group,
                   bool pair_rows, int nseg) {
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
  const int o_gemv_max_cpl = opts().gemv_max_cpl.load();
  const int want_cpl = o_gemv_max_cpl > 0 ? std::min(o_gemv_max_cpl, cpl_cap) : 1;
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
  const int G = param_groups(bits, K, group);
  const int row_bytes = K * bits / 8;
  const int per_row = row_bytes + 4 * G;
  // smallest row multiple that keeps every bulk copy a multiple of 16 bytes (a power of two);
  // with K segments every segment is its own copy
  int m = 1;
  while (((m * (row_bytes / nseg)) & 15) || ((m * (G / nseg) * 2) & 15)) m *= 2;
  // rows in flight per warp: as many as the stage budget and the per-SM row count allow
  const long long rows_total = (long long)N * problems;
  const long long per_sm = std::max<long long>(1, (rows_total + sms - 1) / sms);
  // rows in flight per warp: 8 with one chunk per lane (the 8-row lane reduction
  // takes 9 shuffles; decode pass 4.18 vs 3.81 TB/s with 4 rows), fewer as x
  // slices take more registers
  int ri = pl.cpl == 1 ? 8 : (pl.cpl == 2 ? 2 : 1);
  const int o_gemv_ri = opts().gemv_ri.load();
  if (o_gemv_ri > 0) ri = pl.cpl == 1 ? std::min(8, o_gemv_ri) : std::min(ri, o_gemv_ri);
  const int o_gemv_stage_kb = opts().gemv_stage_kb.load();
  int stage_budget = o_gemv_stage_kb > 0 ? o_gemv_stage_kb * 1024 : kStageBudget;
  const int ri_min = pair_rows ? 2 : 1;   // the SwiGLU epilogue pairs rows 2i, 2i+1
  while (ri > ri_min &&
         ((long long)ri * rw * per_row > stage_budget || ri * rw > std::max<long long>(rw, per_sm)))
    ri /= 2;
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
  const int o_gemv_stages = opts().gemv_stages.load();
  if (o_gemv_stages >= 2) stages = std::min(8, o_gemv_stages);
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

// ---------------------------------------------------------- tensor-pipe GEMV
// Geometry of one problem on the tensor-pipe kernel: K split over kw warps so
// that each warp's slice holds at most 32 groups (2048 codes), 16-row tiles,
// units of whole tiles up to the stage budget (and no more tiles than the
// problem's share of one SM).  Returns false when the kernel does not apply.
MmaShape mma_shape(int cfg) {
  switch (cfg) {
    case 1: return {8, 1, 2};
    case 2: return {8, 1, 1};
    case 3: return {16, 1, 1};
    case 4: return {8, 2, 1};
    case 5: return {8, 1, 1, true};
    case 6: return {8, 2, 1, true};
    case 7: return {16, 1, 1, true};
    default: return {8, 1, 2};
  }
}

namespace {
// dynamic shared memory one CTA may take when `ctas` CTAs share an SM (228 KB,
// 1 KB of it reserved per CTA), less the kernel's static shared memory (128 B,
// with room to spare)
constexpr size_t kMmaStaticSmem = 512;
size_t mma_smem_limit(int ctas) {
  return (ctas == 1 ? 227 * 1024 : (228 * 1024) / ctas - 1024) - kMmaStaticSmem;
}

bool mma_applies(int bits, bool fast, int N, int K, int group) {
  if (opts().gemv_cuda_core.load() || bits != 4 || group != 64 || !fast || K > kMmaMaxK || K % kGroup) return false;
  if (opts().gemv_tensor_pipe.load() == 2) return false;
  const int G = K / kGroup, row_bytes = K * bits / 8;
  // every unit, the ragged last one included, must move in 16-byte pieces
  return ((long long)N * G * 2) % 16 == 0 && ((long long)N * row_bytes) % 16 == 0;
}

// Which launches take the tensor pipe, and with which consumer, by default.
// Measured on B300:
//  * a launch of at most one 16-row tile per SM: the diagonal consumer, whose
//    warps then split K down to one group each (single Q4 GEMV N=2048 K=1024:
//    2.72 vs 3.44 us on the CUDA-core kernel);
//  * launches of at least eight tiles per SM (one per consumer warp) with every
//    K a multiple of 256 and at most 4096: the four-column consumer with two
//    large stages (Qwen3-0.6B-shaped decode pass: 4.63-4.68 vs 4.07 TB/s on the
//    CUDA-core kernel; the diagonal consumer 3.69).  With K = 8192 in the launch
//    the x of the longest row leaves smaller stages (Llama-1B-shaped pass at
//    Q4: 4.20 vs 4.31 TB/s on the CUDA-core kernel);
//  * the launches in between (a few tiles per SM, which would leave consumer
//    warps of the four-column kernel idle) and other large launches: the
//    CUDA-core kernel.
// BT_OPT_GEMV_TENSOR_PIPE 1 forces the tensor pipe wherever it applies, 2
// disables it; BT_OPT_GEMV_MMA_SHAPE forces a kernel shape.
bool mma_small_launch(long long rows, int sms) { return (rows + 15) / 16 <= sms; }

// The shape a tensor-pipe launch takes; nw == 0: the launch stays on the CUDA-core kernel.
MmaShape pick_shape(long long rows, int sms, bool all_k_by_4, int g_max) {
  const int cfg = opts().gemv_mma_cfg.load();
  if (cfg != 0) {
    const MmaShape sh = mma_shape(cfg);
    return sh.cols4 && !all_k_by_4 ? mma_shape(0) : sh;
  }
  if (mma_small_launch(rows, sms)) return mma_shape(0);
  if (all_k_by_4 && g_max <= 64 && (rows + 15) / 16 >= 8LL * sms) return mma_shape(5);
  if (opts().gemv_tensor_pipe.load() == 1) return mma_shape(0);
  return MmaShape{0, 0, 0, false};
}

struct MmaGeom {
  int kw, rb, row_bytes, per_row;
};

// per_sm_rows: the launch's rows per SM.  When those fill fewer 16-row tiles
// than the CTA has warps, K is split further (down to one group per warp), so
// that every warp has work (e.g. the single N=2048 GEMV: one tile per CTA,
// eight warps on two groups each).
MmaGeom mma_geom(int bits, int N, int K, long long per_sm_rows, int stage_budget, int nw, bool cols4 = false) {
  MmaGeom m{};
  const int G = K / kGroup;
  m.row_bytes = K * bits / 8;
  m.per_row = m.row_bytes + 4 * G;
  const int tile = 16 * m.per_row;
  const long long tiles_per_sm = std::max<long long>(1, per_sm_rows / 16);
  const int split_units = cols4 ? G / 4 : G;   // the four-column consumer splits K in blocks of four groups
  const int o_gemv_mma_ks = opts().gemv_mma_ks.load();
  const int ks_max = o_gemv_mma_ks > 0 ? o_gemv_mma_ks : 32;
  int kw = 1;
  while (kw < nw && (G + kw - 1) / kw > ks_max) kw *= 2;
  while (kw < nw && kw * tiles_per_sm < nw && 2 * kw <= split_units) kw *= 2;
  while (kw > 1 && kw > split_units) kw /= 2;
  m.kw = kw;
  long long tiles = std::max(1, stage_budget / tile);
  tiles = std::min<long long>(tiles, std::max<long long>(1, (per_sm_rows + 15) / 16));
  tiles = std::min<long long>(tiles, (N + 15) / 16);
  m.rb = (int)(16 * tiles);
  return m;
}

// Shared memory of one CTA: ring, barriers, row-group partials, x sums, permuted x.
size_t mma_smem(int stages, int stage, int g_max, int nw, int* xsum_bytes) {
  const int xsb = (g_max * 4 + 15) / 16 * 16;
  if (xsum_bytes) *xsum_bytes = xsb;
  return (size_t)stages * stage + 2 * stages * sizeof(uint64_t) + (size_t)nw * 2 * 16 * sizeof(float) + xsb +
         (size_t)g_max * 192;
}

int mma_stage_budget(const MmaShape& sh, int g_max) {
  const int o_gemv_mma_stage_kb = opts().gemv_mma_stage_kb.load();
  if (o_gemv_mma_stage_kb > 0) return o_gemv_mma_stage_kb * 1024;
  if (sh.cols4) {
    // the four-column consumer streams fastest from two stages as large as fit
    // beside the x of the longest K (decode pass on B300: 4.68 TB/s at 108 KiB
    // stages, 4.47 at 96, 3.86 at 48; three stages of 64 KiB 4.45)
    const long long room = (long long)mma_smem_limit(sh.ctas) - (long long)mma_smem(2, 0, g_max, sh.nw, nullptr);
    return (int)std::max<long long>(16 * 1024, std::min<long long>(112 * 1024, room / 2 / 1024 * 1024));
  }
  return sh.ctas == 1 ? 48 * 1024 : 24 * 1024;
}

int mma_stages(int stage, int g_max, const MmaShape& sh) {
  int stages = 8;
  while (stages > 2 && mma_smem(stages, stage, g_max, sh.nw, nullptr) > mma_smem_limit(sh.ctas)) --stages;
  const int o_gemv_stages = opts().gemv_stages.load();
  if (o_gemv_stages >= 2) stages = std::min(8, o_gemv_stages);
  return stages;
}

void set_shape(GemvPlan& pl, const MmaShape& sh) {
  pl.mma_nw = sh.nw;
  pl.mma_ctas = sh.ctas;
  pl.mma_unroll = sh.unroll;
  pl.mma_cols4 = sh.cols4;
}

}  // namespace

GemvPlan plan_gemv_mma(int bits, bool fast, int N, int K, int problems, int num_experts, int sms, int group) {
  GemvPlan pl{};
  pl.fast = fast;
  pl.mma = true;
  pl.cpl = 1;
  pl.ri = 16;
  if (num_experts || !mma_applies(bits, fast, N, K, group)) return pl;
  const MmaShape sh = pick_shape((long long)N * problems, sms, (K / kGroup) % 4 == 0, K / kGroup);
  if (sh.nw == 0) return pl;
  set_shape(pl, sh);
  const long long per_sm = std::max<long long>(1, ((long long)N * problems + sms - 1) / sms);
  const MmaGeom m = mma_geom(bits, N, K, per_sm / sh.ctas, mma_stage_budget(sh, K / kGroup), sh.nw, sh.cols4);
  pl.kw = m.kw;
  pl.rows_per_unit = m.rb;
  pl.row_bytes = m.row_bytes;
  pl.stage_bytes = (m.rb * m.per_row + 127) / 128 * 128;
  const int G = K / kGroup;
  pl.stages = mma_stages(pl.stage_bytes, G, sh);
  pl.units_per_problem = (N + m.rb - 1) / m.rb;
  pl.num_units = (long long)pl.units_per_problem * problems;
  pl.grid = (int)std::min<long long>(pl.num_units, (long long)sms * sh.ctas);
  pl.smem = mma_smem(pl.stages, pl.stage_bytes, G, sh.nw, nullptr);
  pl.feasible = pl.smem <= mma_smem_limit(sh.ctas) && pl.stages >= 2;
  return pl;
}

GemvPlan plan_gemv_batch_mma(int bits, bool fast, GemvBatch<kBatchCap>& batch, int sms, int group, int tokens) {
  GemvPlan pl{};
  pl.fast = fast;
  pl.mma = true;
  pl.cpl = 1;
  pl.ri = 16;
  long long rows = 0;
  int g_max = 0;
  for (int i = 0; i < batch.count; ++i) {
    const GemvProblem& q = batch.prob[i];
    if (q.k <= 0 || !mma_applies(bits, fast, q.n, q.k, group)) return pl;
    rows += q.n;
    g_max = std::max(g_max, q.k / kGroup);
  }
  bool all_k_by_4 = true;
  for (int i = 0; i < batch.count; ++i) all_k_by_4 = all_k_by_4 && (batch.prob[i].k / kGroup) % 4 == 0;
  // several tokens per problem: the four-column consumer only (tokens and groups share its columns)
  const MmaShape sh = tokens >= 2 ? (all_k_by_4 ? mma_shape(5) : MmaShape{0, 0, 0, false})
                                  : pick_shape(rows, sms, all_k_by_4, g_max);
  if (sh.nw == 0 || tokens < 1 || tokens > 8) return pl;
  set_shape(pl, sh);
  const int gx = g_max * token_slots(tokens);   // the staged x (and its group sums) of every token
  const long long per_sm = std::max<long long>(1, (rows + sms - 1) / sms);
  int stage = 0;
  for (int i = 0; i < batch.count; ++i) {
    GemvProblem& q = batch.prob[i];
    const MmaGeom m = mma_geom(bits, q.n, q.k, per_sm / sh.ctas, mma_stage_budget(sh, gx), sh.nw, sh.cols4);
    q.kw = tokens >= 2 ? 1 : m.kw;   // the multi-token consumers keep whole rows in one warp (no K split)
    q.g = q.k / kGroup;
    q.row_bytes = m.row_bytes;
    q.rb = m.rb;
    stage = std::max(stage, (m.rb * m.per_row + 127) / 128 * 128);
  }
  pl.kw = batch.prob[0].kw;
  pl.rows_per_unit = batch.prob[0].rb;
  pl.row_bytes = batch.prob[0].row_bytes;
  pl.stage_bytes = stage;
  pl.stages = mma_stages(stage, gx, sh);
  pl.smem = mma_smem(pl.stages, stage, gx, sh.nw, nullptr);
  pl.grid = sms * sh.ctas;   // trimmed to the unit count at launch
  pl.feasible = pl.smem <= mma_smem_limit(sh.ctas) && pl.stages >= 2;
  return pl;
}

GemvPlan plan_gemv_batch(int bits, bool fast, GemvBatch<kBatchCap>& batch, int sms, int group) {
  GemvPlan pl{};
  pl.fast = fast;
  pl.feasible = false;
  pl.cpl = 1;
  // rows in flight per warp: 8 unless some problem's row group would overflow a stage
  const int o_gemv_ri = opts().gemv_ri.load();
  int ri = o_gemv_ri > 0 ? std::min(8, o_gemv_ri) : 8;
  const int o_gemv_stage_kb = opts().gemv_stage_kb.load();
  int stage_budget = o_gemv_stage_kb > 0 ? o_gemv_stage_kb * 1024 : kStageBudget;
  for (int i = 0; i < batch.count; ++i) {
    const GemvProblem& q = batch.prob[i];
    if (q.k <= 0 || q.k % group || q.k > 8 * 32 * 32) return pl;   // one chunk per lane needs K <= 8192
    const int nchunks = q.k / 32;
    int kw = 1;
    while (32 * kw < nchunks) kw *= 2;
    const int per_row = q.k * bits / 8 + 4 * param_groups(bits, q.k, group);
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
    q.g = param_groups(bits, q.k, group);
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
  const int o_gemv_stages = opts().gemv_stages.load();
  if (o_gemv_stages >= 2) stages = std::min(8, o_gemv_stages);
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
      // CTAs take equal shares of work, not of units.  On the CUDA-core kernel a
      // row split over kw warps costs kw times a one-warp row (measured: K=2048
      // ~2.2x, K=3072 ~4x K=1024); on the tensor-pipe kernel a row costs its
      // groups (every warp's share of a row is whole groups, and the measured
      // per-SM busy time with the kw weighting varied from 0.64 to 0.96 of the
      // launch on the decode pass).
      q.cw = pl.mma ? std::max(1, q.g) : q.kw;
      q.cost_begin = cost;
      cost += (long long)q.n * q.cw;
    }
    p.total_cost = cost;
    p.num_units = u;
    plb.num_units = u;
    plb.grid = (int)std::min<long long>(u, (long long)sm_count() * gemv_ctas_per_sm(pl.cpl, pl.ri));
  }
  if (p.num_units == 0) return cudaSuccess;
  if (pl.mma) {
    int g_max = p.G;
    if (batch)
      for (int i = 0; i < batch->count; ++i) g_max = std::max(g_max, batch->prob[i].g);
    p.tokens = std::max(1, p.tokens);
    p.tok_groups = g_max;
    mma_smem(pl.stages, pl.stage_bytes, g_max * token_slots(p.tokens), pl.mma_nw, &p.xsum_bytes);
    plb.grid = (int)std::min<long long>(p.num_units, (long long)sm_count() * pl.mma_ctas);
    return launch_gemv_mma_b4(p, plb, batch, st);
  }
  switch (bits) {
    case 2: return launch_gemv_b2(p, plb, xd, batch, st);
    case 3: return launch_gemv_b3(p, plb, xd, batch, st);
    case 4: return launch_gemv_b4(p, plb, xd, batch, st);
    case 5: return launch_gemv_b5(p, plb, xd, batch, st);
    case 6: return launch_gemv_b6(p, plb, xd, batch, st);
    case 16: return launch_gemv_b16(p, plb, xd, batch, st);
    default: return launch_gemv_b8(p, plb, xd, batch, st);
  }
}

}  // namespace bt
