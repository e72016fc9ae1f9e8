// C ABI of libbt: argument validation, per-shape launch heuristics and the
// device error word.  Every product is computed by the kernels in this
// library; nothing here computes on the host.
#include <algorithm>
#include <cstdlib>
#include <memory>
#include <mutex>
#include <utility>
#include <vector>

#include "bt_common.cuh"
#include "moe.cuh"
#include "qgemm.cuh"
#include "qgemv.cuh"

namespace bt {

__device__ unsigned g_device_error = 0;

LaunchOpts& opts() {
  static LaunchOpts o;
  return o;
}

namespace {
std::mutex g_mu;
std::vector<unsigned*> g_err_ptr;   // per device
std::vector<int> g_sms;

int current_device() {
  int d = 0;
  cudaGetDevice(&d);
  return d;
}
}  // namespace

unsigned* device_error_word() {
  const int d = current_device();
  std::lock_guard<std::mutex> lk(g_mu);
  if ((int)g_err_ptr.size() <= d) g_err_ptr.resize(d + 1, nullptr);
  if (!g_err_ptr[d]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_device_error) != cudaSuccess) return nullptr;
    g_err_ptr[d] = static_cast<unsigned*>(ptr);
  }
  return g_err_ptr[d];
}

int sm_count() {
  const int d = current_device();
  std::lock_guard<std::mutex> lk(g_mu);
  if ((int)g_sms.size() <= d) g_sms.resize(d + 1, 0);
  if (!g_sms[d]) {
    int v = 0;
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, d);
    g_sms[d] = v > 0 ? v : 1;
  }
  return g_sms[d];
}

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
// 2..8-bit affine codes, and 16 = fp16 weights (no scale or bias)
bool bits_ok(int b) { return b == 2 || b == 3 || b == 4 || b == 5 || b == 6 || b == 8 || b == 16; }
bool group_ok(int g) { return g == 32 || g == 64 || g == 128; }
int group_shift(int g) { return g == 32 ? 0 : (g == 64 ? 1 : 2); }
bool half_dtype(bt_dtype d) { return d == BT_F16 || d == BT_BF16; }
bool out_dtype(bt_dtype d) { return d == BT_F16 || d == BT_BF16 || d == BT_F32; }

bt_status check_weights(const uint32_t* codes, const uint16_t* scales, const uint16_t* biases, int bits,
                        int group_size, int N, int K) {
  const bool params = bits != 16;   // fp16 weights carry no scale or bias (they may be NULL)
  if (!codes || (params && (!scales || !biases))) return BT_ERR_INVALID_ARG;
  if (N <= 0 || K <= 0) return BT_ERR_INVALID_ARG;
  if (!bits_ok(bits) || !group_ok(group_size)) return BT_ERR_UNSUPPORTED;
  if (K % group_size) return BT_ERR_INVALID_ARG;
  if (K > kMaxK) return BT_ERR_UNSUPPORTED;
  if (!aligned16(codes) || (params && (!aligned16(scales) || !aligned16(biases)))) return BT_ERR_MISALIGNED;
  return BT_OK;
}

bt_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) e = cudaGetLastError();
  else cudaGetLastError();
  return e == cudaSuccess ? BT_OK : BT_ERR_CUDA;
}

// Which kernel family runs a product of M rows: the GEMV (one row, or a grouped
// launch with no more rows than experts), the small-token tensor-pipe kernel
// (dense M <= 8, or grouped with at most 16 rows per expert on average), the
// tensor cores (any other supported shape) or the CUDA-core tile.  num_experts == 0: dense product.  BT_OPT_GEMM_PATH forces
// 1 (CUDA-core tile), 2 (tensor cores) or 3 (small-token kernel) where the shape
// allows.
enum GemmPath { kPathNone = 0, kPathGemv = 1, kPathSimt = 2, kPathTc = 3, kPathMma = 4 };
GemmPath gemm_path(int bits, int M, int N, int K, int num_experts, int group, int sms) {
  const int forced = opts().gemm_path;
  if (num_experts == 0 && M == 1 && forced != 3) return kPathGemv;
  if (num_experts > 0 && M == 0) return kPathNone;
  if (num_experts > 0 && M <= num_experts && forced == 0) return kPathGemv;
  const bool mma_ok = plan_gemm_small(bits, M, N, K, group, num_experts, sms).feasible;
  const bool tc_ok = tc_shape_ok(bits, K, group, num_experts > 0);
  if (forced == 1) return kPathSimt;
  if (forced == 2) return tc_ok ? kPathTc : kPathSimt;
  if (forced == 3 && mma_ok) return kPathMma;
  if (num_experts > 0) {
    if (mma_ok && ((long long)M + num_experts - 1) / num_experts <= 16) return kPathMma;
    return tc_ok ? kPathTc : kPathSimt;
  }
  // dense: one n8 token tile on the small-token kernel; the tensor cores from 9 rows
  if (mma_ok && M <= 8) return kPathMma;
  if (tc_ok) return kPathTc;
  return mma_ok ? kPathMma : kPathSimt;
}

// fp16 x takes the magic-number fast path at every bit width (BT_OPT_GEMV_GENERIC
// forces the generic one); bits decides only how many chunks per lane exist.
bool gemv_fast_path(int bits, bt_dtype xd) {
  return xd == BT_F16 && !opts().gemv_generic && bits != 5;   // 5-bit codes have no fp16 pair schedule
}

// How the problems of a GEMV launch map to experts and rows (all empty: dense).
struct RowMap {
  const int32_t* offsets = nullptr;     // grouped rows: expert of row r from the offsets
  const int32_t* row_index = nullptr;   // grouped rows: x row of row r
  int num_experts = 0;
  const int32_t* pair_ids = nullptr;    // routed pairs: expert of problem r, x row r / top_k
  int top_k = 0;
  int swiglu = 0;                       // SwiGLU epilogue over interleaved gate/up rows
};

bt_status run_gemv(const uint32_t* codes, const uint16_t* scales, const uint16_t* biases, int bits, int group,
                   int N, int K, const void* x, bt_dtype xd, void* y, bt_dtype yd, int problems, const RowMap& rm,
                   cudaStream_t stream) {
  const int32_t* offsets = rm.offsets;
  const int32_t* row_index = rm.row_index;
  const int num_experts = rm.num_experts;
  GemvParams p{};
  p.codes = codes;
  p.scales = scales;
  p.biases = biases;
  p.x = x;
  p.y = y;
  p.N = N;
  p.K = K;
  p.G = param_groups(bits, K, group);
  p.gshift = group_shift(group);
  p.moe_offsets = offsets;
  p.row_index = row_index;
  p.num_experts = (offsets || rm.pair_ids) ? num_experts : 0;
  p.pair_ids = rm.pair_ids;
  p.top_k = rm.top_k;
  p.swiglu = rm.swiglu;
  p.total_rows = problems;
  p.err = device_error_word();
  p.timeout_ns = opts().wait_timeout_ns;
  p.const_weights = opts().pdl && opts().const_weights;
  p.drop_stage = opts().test_drop_stage.exchange(0);
  GemvPlan pl{};
  if (!rm.pair_ids && !rm.swiglu)
    pl = plan_gemv_mma(bits, gemv_fast_path(bits, xd), N, K, problems, p.num_experts, sm_count(), group);
  if (!pl.feasible)
    pl = plan_gemv(bits, gemv_fast_path(bits, xd), N, K, problems, offsets ? num_experts : 0, sm_count(), group,
                   rm.swiglu != 0);
  if (!pl.feasible && rm.pair_ids) return BT_ERR_UNSUPPORTED;   // routed pairs run on the GEMV only
  if (!pl.feasible) {
    // no GEMV kernel holds this K slice in registers: the CUDA-core tile computes the same product
    GemmParams g{};
    g.codes = codes; g.scales = scales; g.biases = biases; g.x = x; g.y = y;
    g.M = problems; g.N = N; g.K = K;
    g.group = group;
    g.offsets = offsets;
    g.row_index = row_index;
    g.num_experts = num_experts;
    g.swiglu = rm.swiglu;
    g.err = p.err;
    g.timeout_ns = p.timeout_ns;
    return cuda_status(launch_gemm_simt(g, bits, xd, yd, stream));
  }
  return cuda_status(launch_gemv(p, pl, bits, xd, yd, stream));
}

// Grouped expert product (optionally with the SwiGLU epilogue): the GEMV for at
// most one row per expert, else the tensor cores or the CUDA-core tile.
bt_status moe_grouped(const uint32_t* codes, const uint16_t* scales, const uint16_t* biases, int bits,
                      int group_size, int num_experts, int N, int K, const int32_t* expert_offsets, int total_rows,
                      const int32_t* x_row_index, const void* x, bt_dtype x_dtype, void* y, bt_dtype y_dtype,
                      int swiglu, cudaStream_t stream) {
  bt_status s = check_weights(codes, scales, biases, bits, group_size, N, K);
  if (s != BT_OK) return s;
  if (num_experts <= 0 || num_experts > 4096 || total_rows < 0 || !expert_offsets || !x || !y ||
      !half_dtype(x_dtype) || !out_dtype(y_dtype))
    return BT_ERR_INVALID_ARG;
  if (!aligned16(x)) return BT_ERR_MISALIGNED;
  const GemmPath path = gemm_path(bits, total_rows, N, K, num_experts, group_size, sm_count());
  if (path == kPathNone) return BT_OK;
  if (path == kPathGemv) {
    RowMap rm;
    rm.offsets = expert_offsets;
    rm.row_index = x_row_index;
    rm.num_experts = num_experts;
    rm.swiglu = swiglu;
    return run_gemv(codes, scales, biases, bits, group_size, N, K, x, x_dtype, y, y_dtype, total_rows, rm, stream);
  }
  GemmParams p{};
  p.codes = codes; p.scales = scales; p.biases = biases; p.x = x; p.y = y;
  p.M = total_rows; p.N = N; p.K = K;
  p.group = group_size;
  p.swiglu = swiglu;
  p.offsets = expert_offsets;
  p.row_index = x_row_index;
  p.num_experts = num_experts;
  p.err = device_error_word();
  p.timeout_ns = opts().wait_timeout_ns;
  if (path == kPathMma && small_supported(bits, p)) return cuda_status(launch_gemm_small(p, bits, x_dtype, y_dtype, stream));
  if ((path == kPathTc || path == kPathMma) && tc_supported(bits, K, total_rows, p))
    return cuda_status(launch_gemm_tc_grouped(p, bits, x_dtype, y_dtype, stream));
  return cuda_status(launch_gemm_simt(p, bits, x_dtype, y_dtype, stream));
}

}  // namespace
}  // namespace bt

using namespace bt;

namespace {
void fill_plan(const bt::GemvPlan& pl, bt_gemv_plan* out) {
  out->feasible = pl.feasible ? 1 : 0;
  out->tensor_pipe = pl.mma ? (pl.mma_cols4 ? 2 : 1) : 0;
  out->kw = pl.kw;
  out->cpl = pl.cpl;
  out->ri = pl.ri;
  out->rows_per_unit = pl.rows_per_unit;
  out->stage_bytes = pl.stage_bytes;
  out->stages = pl.stages;
  out->ctas_per_sm = pl.mma ? pl.mma_ctas : bt::gemv_ctas_per_sm(pl.cpl, pl.ri);
  out->grid = pl.grid;
  out->num_units = pl.num_units;
  out->smem_bytes = (int64_t)pl.smem;
}
}  // namespace

extern "C" {

const char* bt_status_string(bt_status s) {
  switch (s) {
    case BT_OK: return "BT_OK";
    case BT_ERR_INVALID_ARG: return "BT_ERR_INVALID_ARG: invalid argument";
    case BT_ERR_UNSUPPORTED: return "BT_ERR_UNSUPPORTED: unsupported bits, group size or size";
    case BT_ERR_MISALIGNED: return "BT_ERR_MISALIGNED: pointer not 16-byte aligned";
    case BT_ERR_CUDA: return "BT_ERR_CUDA: CUDA call or launch failed";
    case BT_ERR_TIMEOUT: return "BT_ERR_TIMEOUT: a device-side wait expired";
  }
  return "unknown bt_status";
}

bt_status bt_plan_gemv(int bits, bt_dtype x_dtype, int N, int K, int problems, int sms, bt_gemv_plan* plan) {
  if (!plan || N <= 0 || K <= 0 || K % kGroup || problems <= 0 || sms <= 0 || !half_dtype(x_dtype))
    return BT_ERR_INVALID_ARG;
  if (!bits_ok(bits) || K > kMaxK) return BT_ERR_UNSUPPORTED;
  GemvPlan pl = plan_gemv_mma(bits, gemv_fast_path(bits, x_dtype), N, K, problems, 0, sms);
  if (!pl.feasible) pl = plan_gemv(bits, gemv_fast_path(bits, x_dtype), N, K, problems, 0, sms);
  fill_plan(pl, plan);
  return BT_OK;
}

bt_status bt_plan_gemv_batch(int bits, bt_dtype x_dtype, const int32_t* n, const int32_t* k, int count, int sms,
                             bt_gemv_plan* plan, int32_t* kw, int32_t* rows_per_unit) {
  if (!plan || !n || !k || count < 1 || sms <= 0 || !half_dtype(x_dtype)) return BT_ERR_INVALID_ARG;
  if (count > kBatchCap || !bits_ok(bits)) return BT_ERR_UNSUPPORTED;
  GemvBatch<kBatchCap> batch;
  batch.count = count;
  long long units = 0;
  for (int i = 0; i < count; ++i) {
    if (n[i] <= 0 || k[i] <= 0 || k[i] % kGroup) return BT_ERR_INVALID_ARG;
    batch.prob[i] = GemvProblem{};
    batch.prob[i].n = n[i];
    batch.prob[i].k = k[i];
  }
  GemvPlan pl = plan_gemv_batch_mma(bits, gemv_fast_path(bits, x_dtype), batch, sms);
  if (!pl.feasible) pl = plan_gemv_batch(bits, gemv_fast_path(bits, x_dtype), batch, sms);
  if (pl.feasible) {
    for (int i = 0; i < count; ++i) {
      units += (batch.prob[i].n + batch.prob[i].rb - 1) / batch.prob[i].rb;
      if (kw) kw[i] = batch.prob[i].kw;
      if (rows_per_unit) rows_per_unit[i] = batch.prob[i].rb;
    }
    pl.num_units = units;
    pl.grid = (int)std::min<long long>(units, (long long)sms * (pl.mma ? pl.mma_ctas : gemv_ctas_per_sm(pl.cpl, pl.ri)));
  }
  fill_plan(pl, plan);
  return BT_OK;
}

bt_status bt_plan_gemm(int bits, bt_dtype x_dtype, int M, int N, int K, int num_experts, int sms, bt_gemm_plan* plan) {
  if (!plan || M < 0 || (M == 0 && num_experts == 0) || N <= 0 || K <= 0 || K % kGroup || num_experts < 0 ||
      num_experts > 4096 || sms <= 0 || !half_dtype(x_dtype))
    return BT_ERR_INVALID_ARG;
  if (!bits_ok(bits) || K > kMaxK) return BT_ERR_UNSUPPORTED;
  *plan = bt_gemm_plan{};
  GemmPath path = gemm_path(bits, M, N, K, num_experts, 64, sms);
  GemmGeometry g;
  if (path == kPathGemv) {
    GemvPlan pl = plan_gemv_mma(bits, gemv_fast_path(bits, x_dtype), N, K, num_experts ? M : 1, num_experts, sms);
    if (!pl.feasible) pl = plan_gemv(bits, gemv_fast_path(bits, x_dtype), N, K, num_experts ? M : 1, num_experts, sms);
    if (pl.feasible) {
      g.feasible = true;
      g.stages = pl.stages;
      g.grid_x = pl.grid;
      g.grid_y = g.grid_z = 1;
      g.smem = (long long)pl.smem;
    } else {
      path = kPathSimt;   // run_gemv hands shapes no GEMV kernel holds to the CUDA-core tile
    }
  }
  if (path == kPathMma) {
    const SmallGeometry sg = plan_gemm_small(bits, M, N, K, 64, num_experts, sms);
    g.feasible = sg.feasible;
    g.bn = 8 * sg.t8;
    g.splits = sg.kw;
    g.stages = sg.stages;
    g.grid_x = sg.grid;
    g.grid_y = g.grid_z = 1;
    g.smem = sg.smem;
    plan->rows_per_unit = sg.rb;
  }
  if (path == kPathTc) g = plan_gemm_tc_geometry(bits, M, N, K, num_experts, sms);
  if (path == kPathSimt) g = plan_gemm_simt_geometry(M, N, num_experts);
  plan->path = path;
  plan->feasible = (path == kPathNone || g.feasible) ? 1 : 0;
  plan->bn = g.bn;
  plan->splits = g.splits;
  plan->stages = g.stages;
  plan->k_blocks = g.k_blocks;
  plan->grid_x = g.grid_x;
  plan->grid_y = g.grid_y;
  plan->grid_z = g.grid_z;
  plan->smem_bytes = g.smem;
  return BT_OK;
}

bt_status bt_set_option(bt_option option, long long value) {
  if (value < 0) return BT_ERR_INVALID_ARG;
  switch (option) {
    case BT_OPT_PDL: opts().pdl = value != 0; return BT_OK;
    case BT_OPT_CONST_WEIGHTS: opts().const_weights = value != 0; return BT_OK;
    case BT_OPT_WAIT_TIMEOUT_US: opts().wait_timeout_ns = (unsigned long long)value * 1000ull; return BT_OK;
    case BT_OPT_TEST_DROP_STAGE: opts().test_drop_stage = value != 0; return BT_OK;
    case BT_OPT_GEMV_GENERIC: opts().gemv_generic = value != 0; return BT_OK;
    case BT_OPT_GEMV_STAGES: opts().gemv_stages = (int)value; return BT_OK;
    case BT_OPT_GEMM_PATH: opts().gemm_path = (int)value; return BT_OK;
    case BT_OPT_GEMM_SPLITS: opts().gemm_splits = (int)std::min<long long>(value, 8); return BT_OK;
    case BT_OPT_GEMV_MAX_CPL: opts().gemv_max_cpl = (int)std::min<long long>(value, 4); return BT_OK;
    case BT_OPT_GEMV_RI: opts().gemv_ri = value >= 8 ? 8 : value >= 4 ? 4 : (value >= 2 ? 2 : (int)value); return BT_OK;
    case BT_OPT_GEMV_STAGE_KB: opts().gemv_stage_kb = value == 0 ? 0 : (int)std::max(4LL, std::min(value, 96LL)); return BT_OK;
    case BT_OPT_GEMV_CUDA_CORE: opts().gemv_cuda_core = value != 0; return BT_OK;
    case BT_OPT_GEMV_MMA_STAGE_KB: opts().gemv_mma_stage_kb = value == 0 ? 0 : (int)std::max(8LL, std::min(value, 112LL)); return BT_OK;
    case BT_OPT_GEMV_MMA_SHAPE: opts().gemv_mma_cfg = (int)std::min(value, 7LL); return BT_OK;
    case BT_OPT_GEMV_TENSOR_PIPE: opts().gemv_tensor_pipe = (int)std::min(value, 2LL); return BT_OK;
    case BT_OPT_GEMM_DEQ_WARPS: opts().gemm_deq_warps = (int)value; return BT_OK;
    case BT_OPT_GEMM_SMALL_WARPS: opts().gemm_small_warps = (int)value; return BT_OK;
    case BT_OPT_GEMV_MMA_GROUPS: opts().gemv_mma_ks = value == 0 ? 0 : (int)std::max(1LL, std::min(value, 64LL)); return BT_OK;
  }
  return BT_ERR_INVALID_ARG;
}

bt_status bt_last_device_error(cudaStream_t stream) {
  if (cudaStreamSynchronize(stream) != cudaSuccess) {
    cudaGetLastError();
    return BT_ERR_CUDA;
  }
  unsigned v = 0;
  if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof(v)) != cudaSuccess) return BT_ERR_CUDA;
  if (v) {
    const unsigned zero = 0;
    if (cudaMemcpyToSymbol(g_device_error, &zero, sizeof(zero)) != cudaSuccess) return BT_ERR_CUDA;
  }
  if (v & kErrTimeout) return BT_ERR_TIMEOUT;
  if (v & kErrBadArg) return BT_ERR_INVALID_ARG;
  return BT_OK;
}

bt_status bt_qgemv(const uint32_t* codes, const uint16_t* scales, const uint16_t* biases, int bits,
                   int group_size, int N, int K, const void* x, bt_dtype x_dtype, void* y, bt_dtype y_dtype,
                   cudaStream_t stream) {
  bt_status s = check_weights(codes, scales, biases, bits, group_size, N, K);
  if (s != BT_OK) return s;
  if (!x || !y || !half_dtype(x_dtype) || !out_dtype(y_dtype)) return BT_ERR_INVALID_ARG;
  if (!aligned16(x)) return BT_ERR_MISALIGNED;
  return run_gemv(codes, scales, biases, bits, group_size, N, K, x, x_dtype, y, y_dtype, 1, RowMap{}, stream);
}

namespace bt {
// A validated and planned batched GEMV (no launch).  The run-time fields of p
// (error word, wait bound, PDL weight hint, test hook) are set at each launch.
struct PreparedGemv {
  GemvBatch<kBatchCap> batch;
  GemvParams p;
  GemvPlan pl;
};

bt_status prepare_gemv_batch(const bt_gemv_problem* problems, int count, int bits, int group_size, int K,
                             bt_dtype x_dtype, bt_dtype y_dtype, PreparedGemv& g, int tokens = 1) {
  if (!problems || count < 1 || K < 0) return BT_ERR_INVALID_ARG;
  if (count > kBatchCap) return BT_ERR_UNSUPPORTED;
  if (!half_dtype(x_dtype) || !out_dtype(y_dtype)) return BT_ERR_INVALID_ARG;
  const bool mixed = K == 0;
  long long rows = 0;
  int max_n = 0;
  for (int i = 0; i < count; ++i) {
    const bt_gemv_problem& q = problems[i];
    const int kq = mixed ? q.k : K;
    bt_status s = check_weights(q.codes, q.scales, q.biases, bits, group_size, q.n, kq);
    if (s != BT_OK) return s;
    if (!q.x || !q.y) return BT_ERR_INVALID_ARG;
    if (!aligned16(q.x)) return BT_ERR_MISALIGNED;
    rows += q.n;
    max_n = std::max(max_n, q.n);
  }
  GemvBatch<kBatchCap>& batch = g.batch;
  batch.count = count;
  for (int i = 0; i < count; ++i) {
    GemvProblem& b = batch.prob[i];
    b = GemvProblem{};
    b.codes = problems[i].codes;
    b.scales = problems[i].scales;
    b.biases = problems[i].biases;
    b.x = problems[i].x;
    b.y = problems[i].y;
    b.n = problems[i].n;
    b.k = mixed ? problems[i].k : 0;   // 0: the launch plan's K and geometry
  }
  g.p = GemvParams{};
  g.p.tokens = tokens;
  g.p.K = K;
  g.p.G = param_groups(bits, K, group_size);
  g.p.gshift = group_shift(group_size);
  g.p.N = max_n;
  const bool fast = gemv_fast_path(bits, x_dtype);
  GemvPlan& pl = g.pl;
  if (tokens >= 2) {   // several x rows per problem: the tensor-pipe kernel's four-column consumer or nothing
    pl = mixed ? plan_gemv_batch_mma(bits, fast, batch, sm_count(), group_size, tokens) : GemvPlan{};
  } else if (mixed) {
    pl = plan_gemv_batch_mma(bits, fast, batch, sm_count(), group_size);
    if (!pl.feasible) pl = plan_gemv_batch(bits, fast, batch, sm_count(), group_size);
  } else {
    const int problems_equiv = (int)std::max<long long>(1, (rows + max_n - 1) / max_n);
    // the tensor-pipe kernel needs every problem's units (its ragged last one too) 16-byte aligned
    bool all_mma = true;
    for (int i = 0; i < count && all_mma; ++i)
      all_mma = plan_gemv_mma(bits, fast, problems[i].n, K, 1, 0, sm_count(), group_size).feasible;
    pl = all_mma ? plan_gemv_mma(bits, fast, max_n, K, problems_equiv, 0, sm_count(), group_size) : GemvPlan{};
    if (!pl.feasible) pl = plan_gemv(bits, fast, max_n, K, problems_equiv, 0, sm_count(), group_size);
  }
  return BT_OK;
}

// Launches a prepared batch; a batch no single launch holds (a row group or K
// beyond one launch's staging) runs each problem as its own bt_qgemv, which
// accepts every shape the checks passed.
bt_status run_prepared_gemv(const PreparedGemv& g, const bt_gemv_problem* problems, int count, int bits,
                            int group_size, int K, bt_dtype x_dtype, bt_dtype y_dtype, cudaStream_t stream) {
  if (!g.pl.feasible) {
    for (int i = 0; i < count; ++i) {
      const bt_gemv_problem& q = problems[i];
      const bt_status st = run_gemv(q.codes, q.scales, q.biases, bits, group_size, q.n, K == 0 ? q.k : K, q.x,
                                    x_dtype, q.y, y_dtype, 1, RowMap{}, stream);
      if (st != BT_OK) return st;
    }
    return BT_OK;
  }
  GemvParams p = g.p;
  p.err = device_error_word();
  p.timeout_ns = opts().wait_timeout_ns;
  p.const_weights = opts().pdl && opts().const_weights;
  p.drop_stage = opts().test_drop_stage.exchange(0);
  GemvBatch<kBatchCap> batch = g.batch;
  return cuda_status(launch_gemv(p, g.pl, bits, x_dtype, y_dtype, stream, &batch));
}
}  // namespace bt

bt_status bt_qgemv_batched(const bt_gemv_problem* problems, int count, int bits, int group_size, int K,
                           bt_dtype x_dtype, bt_dtype y_dtype, cudaStream_t stream) {
  std::unique_ptr<PreparedGemv> g(new PreparedGemv);
  const bt_status s = prepare_gemv_batch(problems, count, bits, group_size, K, x_dtype, y_dtype, *g);
  if (s != BT_OK) return s;
  return run_prepared_gemv(*g, problems, count, bits, group_size, K, x_dtype, y_dtype, stream);
}

bt_status bt_qgemm(const uint32_t* codes, const uint16_t* scales, const uint16_t* biases, int bits,
                   int group_size, int M, int N, int K, const void* x, bt_dtype x_dtype, void* y,
                   bt_dtype y_dtype, cudaStream_t stream) {
  bt_status s = check_weights(codes, scales, biases, bits, group_size, N, K);
  if (s != BT_OK) return s;
  if (M <= 0 || !x || !y || !half_dtype(x_dtype) || !out_dtype(y_dtype)) return BT_ERR_INVALID_ARG;
  if (!aligned16(x)) return BT_ERR_MISALIGNED;
  const GemmPath path = gemm_path(bits, M, N, K, 0, group_size, sm_count());
  if (path == kPathGemv)
    return run_gemv(codes, scales, biases, bits, group_size, N, K, x, x_dtype, y, y_dtype, 1, RowMap{}, stream);
  GemmParams p{};
  p.codes = codes; p.scales = scales; p.biases = biases; p.x = x; p.y = y;
  p.M = M; p.N = N; p.K = K;
  p.group = group_size;
  p.err = device_error_word();
  p.timeout_ns = opts().wait_timeout_ns;
  if (path == kPathMma && small_supported(bits, p)) return cuda_status(launch_gemm_small(p, bits, x_dtype, y_dtype, stream));
  if (path == kPathTc && tc_supported(bits, K, M, p))
    return cuda_status(launch_gemm_tc(p, bits, x_dtype, y_dtype, stream));
  return cuda_status(launch_gemm_simt(p, bits, x_dtype, y_dtype, stream));
}

namespace bt {
// One launch of a batched product list (or, where no single launch holds a
// chunk, one launch per product), prepared once and launched many times.
struct PassStep {
  enum Kind { kGemv, kSmall, kEach } kind = kEach;
  std::unique_ptr<PreparedGemv> gemv;
  SmallBatchPrepared* small = nullptr;
  std::vector<bt_gemv_problem> gp;     // kGemv: the chunk, for the per-problem fallback
  std::vector<bt_gemm_problem> each;   // kEach: the chunk
  PassStep() = default;
  PassStep(PassStep&& o) noexcept
      : kind(o.kind), gemv(std::move(o.gemv)), small(std::exchange(o.small, nullptr)), gp(std::move(o.gp)),
        each(std::move(o.each)) {}
  PassStep(const PassStep&) = delete;
  ~PassStep() {
    if (small) free_gemm_small_batched(small);
  }
};

bt_status check_gemm_list(const bt_gemm_problem* problems, int count, int bits, int group_size, int M,
                          bt_dtype x_dtype, bt_dtype y_dtype) {
  if (!problems || count < 1 || M < 1 || !half_dtype(x_dtype) || !out_dtype(y_dtype)) return BT_ERR_INVALID_ARG;
  for (int i = 0; i < count; ++i) {
    const bt_gemm_problem& q = problems[i];
    bt_status s = check_weights(q.codes, q.scales, q.biases, bits, group_size, q.n, q.k);
    if (s != BT_OK) return s;
    if (!q.x || !q.y) return BT_ERR_INVALID_ARG;
    if (!aligned16(q.x)) return BT_ERR_MISALIGNED;
  }
  return BT_OK;
}

// Splits a checked product list into launches: M = 1 takes the batched GEMV
// (kBatchCap problems per launch); up to 16 rows take the small-token kernel
// (where a single product of 9..16 rows would take the tensor cores, a table
// of them is launch-bound); the rest run one product per launch.
bt_status plan_steps(const bt_gemm_problem* problems, int count, int bits, int group_size, int M, bt_dtype x_dtype,
                     bt_dtype y_dtype, std::vector<PassStep>& steps) {
  if (M == 1) {
    for (int i0 = 0; i0 < count; i0 += kBatchCap) {
      const int c = std::min(kBatchCap, count - i0);
      PassStep st;
      st.kind = PassStep::kGemv;
      st.gp.resize((size_t)c);
      for (int i = 0; i < c; ++i) {
        const bt_gemm_problem& q = problems[i0 + i];
        st.gp[i] = bt_gemv_problem{q.codes, q.scales, q.biases, q.x, q.y, q.n, q.k};
      }
      st.gemv.reset(new PreparedGemv);
      const bt_status s = prepare_gemv_batch(st.gp.data(), c, bits, group_size, 0, x_dtype, y_dtype, *st.gemv);
      if (s != BT_OK) return s;
      steps.push_back(std::move(st));
    }
    return BT_OK;
  }
  const int forced = opts().gemm_path;
  if (M >= 2 && M <= 8 && forced == 0 && bits == 4 && group_size == 64 && x_dtype == BT_F16) {
    // two to eight tokens: the batched GEMV's four-column consumer reads and
    // unpacks each weight once for all of them (tokens share the MMA's
    // columns with the groups), where it applies
    std::vector<PassStep> two;
    bool ok = true;
    for (int i0 = 0; i0 < count && ok; i0 += kBatchCap) {
      const int c = std::min(kBatchCap, count - i0);
      PassStep st;
      st.kind = PassStep::kGemv;
      st.gp.resize((size_t)c);
      for (int i = 0; i < c; ++i) {
        const bt_gemm_problem& q = problems[i0 + i];
        st.gp[i] = bt_gemv_problem{q.codes, q.scales, q.biases, q.x, q.y, q.n, q.k};
      }
      st.gemv.reset(new PreparedGemv);
      ok = prepare_gemv_batch(st.gp.data(), c, bits, group_size, 0, x_dtype, y_dtype, *st.gemv, M) == BT_OK &&
           st.gemv->pl.feasible;
      two.push_back(std::move(st));
    }
    if (ok) {
      for (PassStep& st : two) steps.push_back(std::move(st));
      return BT_OK;
    }
  }
  const bool small_ok = (forced == 0 && M <= 16) || forced == 3;
  for (int i0 = 0; i0 < count; i0 += small::kBatchLaunchCap) {
    const int c = std::min(small::kBatchLaunchCap, count - i0);
    PassStep st;
    st.each.assign(problems + i0, problems + i0 + c);
    std::vector<GemmProblem> gp((size_t)c);
    for (int i = 0; i < c; ++i) {
      const bt_gemm_problem& q = problems[i0 + i];
      gp[i] = GemmProblem{q.codes, q.scales, q.biases, q.x, q.y, q.n, q.k};
    }
    if (small_ok && small_batch_supported(gp.data(), c, M, bits, group_size)) {
      st.small = prepare_gemm_small_batched(gp.data(), c, M, x_dtype, y_dtype);
      if (!st.small) return BT_ERR_INVALID_ARG;
      st.kind = PassStep::kSmall;
    }
    steps.push_back(std::move(st));
  }
  return BT_OK;
}

bt_status run_steps(const std::vector<PassStep>& steps, int bits, int group_size, int M, bt_dtype x_dtype,
                    bt_dtype y_dtype, cudaStream_t stream) {
  for (const PassStep& st : steps) {
    bt_status s = BT_OK;
    if (st.kind == PassStep::kGemv) {
      s = run_prepared_gemv(*st.gemv, st.gp.data(), (int)st.gp.size(), bits, group_size, 0, x_dtype, y_dtype, stream);
    } else if (st.kind == PassStep::kSmall) {
      s = cuda_status(run_gemm_small_batched(st.small, device_error_word(), opts().wait_timeout_ns, stream));
    } else {
      for (const bt_gemm_problem& q : st.each) {
        s = bt_qgemm(q.codes, q.scales, q.biases, bits, group_size, M, q.n, q.k, q.x, x_dtype, q.y, y_dtype, stream);
        if (s != BT_OK) break;
      }
    }
    if (s != BT_OK) return s;
  }
  return BT_OK;
}
}  // namespace bt

bt_status bt_qgemm_batched(const bt_gemm_problem* problems, int count, int bits, int group_size, int M,
                           bt_dtype x_dtype, bt_dtype y_dtype, cudaStream_t stream) {
  bt_status s = check_gemm_list(problems, count, bits, group_size, M, x_dtype, y_dtype);
  if (s != BT_OK) return s;
  std::vector<PassStep> steps;
  s = plan_steps(problems, count, bits, group_size, M, x_dtype, y_dtype, steps);
  if (s != BT_OK) return s;
  return run_steps(steps, bits, group_size, M, x_dtype, y_dtype, stream);
}

// ------------------------------------------------------------------ decode pass
struct bt_pass {
  int device = 0;
  int bits = 0, group = 0, M = 0;
  bt_dtype xd = BT_F16, yd = BT_F32;
  std::vector<std::vector<bt::PassStep>> stages;
  cudaStream_t capture = nullptr;
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
  bool ran = false;
  ~bt_pass() {
    if (exec) cudaGraphExecDestroy(exec);
    if (graph) cudaGraphDestroy(graph);
    if (capture) cudaStreamDestroy(capture);
  }
};

bt_status bt_pass_create(const bt_pass_stage* stages, int num_stages, int bits, int group_size, int M,
                         bt_dtype x_dtype, bt_dtype y_dtype, bt_pass** pass) {
  if (!pass) return BT_ERR_INVALID_ARG;
  *pass = nullptr;
  if (!stages || num_stages < 1) return BT_ERR_INVALID_ARG;
  for (int s = 0; s < num_stages; ++s) {   // every check before any CUDA call
    const bt_status st = check_gemm_list(stages[s].problems, stages[s].count, bits, group_size, M, x_dtype, y_dtype);
    if (st != BT_OK) return st;
  }
  std::unique_ptr<bt_pass> ps(new bt_pass);
  if (cudaGetDevice(&ps->device) != cudaSuccess) return BT_ERR_CUDA;
  ps->bits = bits;
  ps->group = group_size;
  ps->M = M;
  ps->xd = x_dtype;
  ps->yd = y_dtype;
  ps->stages.resize((size_t)num_stages);
  for (int s = 0; s < num_stages; ++s) {
    const bt_status st =
        plan_steps(stages[s].problems, stages[s].count, bits, group_size, M, x_dtype, y_dtype, ps->stages[s]);
    if (st != BT_OK) return st;
  }
  *pass = ps.release();
  return BT_OK;
}

namespace {
bt_status run_stages(const bt_pass& ps, cudaStream_t stream) {
  for (const std::vector<bt::PassStep>& st : ps.stages) {
    const bt_status s = run_steps(st, ps.bits, ps.group, ps.M, ps.xd, ps.yd, stream);
    if (s != BT_OK) return s;
  }
  return BT_OK;
}

// Records the pass into a CUDA graph on a stream of its own.  Runs after one
// eager pass, so every kernel is loaded and every per-device setting is made
// before the capture begins.
bt_status record_pass(bt_pass& ps) {
  if (cudaStreamCreateWithFlags(&ps.capture, cudaStreamNonBlocking) != cudaSuccess) return BT_ERR_CUDA;
  if (cudaStreamBeginCapture(ps.capture, cudaStreamCaptureModeThreadLocal) != cudaSuccess) return BT_ERR_CUDA;
  const bt_status s = run_stages(ps, ps.capture);
  cudaGraph_t g = nullptr;
  const cudaError_t e = cudaStreamEndCapture(ps.capture, &g);
  if (s != BT_OK) {
    if (g) cudaGraphDestroy(g);
    return s;
  }
  if (e != cudaSuccess) return BT_ERR_CUDA;
  ps.graph = g;
  if (cudaGraphInstantiate(&ps.exec, g, 0) != cudaSuccess) {
    ps.exec = nullptr;
    return BT_ERR_CUDA;
  }
  return BT_OK;
}
}  // namespace

bt_status bt_pass_run(bt_pass* pass, cudaStream_t stream) {
  if (!pass) return BT_ERR_INVALID_ARG;
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess) return BT_ERR_CUDA;
  if (d != pass->device) return BT_ERR_INVALID_ARG;
  if (!pass->ran) {   // first run: eager launches, then the recording
    const bt_status s = run_stages(*pass, stream);
    if (s != BT_OK) return s;
    pass->ran = true;
    return record_pass(*pass);
  }
  if (!pass->exec) return BT_ERR_CUDA;
  return cuda_status(cudaGraphLaunch(pass->exec, stream));
}

void bt_pass_destroy(bt_pass* pass) { delete pass; }

bt_status bt_moe_qgemm(const uint32_t* codes, const uint16_t* scales, const uint16_t* biases, int bits,
                       int group_size, int num_experts, int N, int K, const int32_t* expert_offsets,
                       int total_rows, const int32_t* x_row_index, const void* x, bt_dtype x_dtype, void* y,
                       bt_dtype y_dtype, cudaStream_t stream) {
  return moe_grouped(codes, scales, biases, bits, group_size, num_experts, N, K, expert_offsets, total_rows,
                     x_row_index, x, x_dtype, y, y_dtype, 0, stream);
}

bt_status bt_moe_qgemm_swiglu(const uint32_t* codes, const uint16_t* scales, const uint16_t* biases, int bits,
                              int group_size, int num_experts, int N, int K, const int32_t* expert_offsets,
                              int total_rows, const int32_t* x_row_index, const void* x, bt_dtype x_dtype, void* h,
                              bt_dtype h_dtype, cudaStream_t stream) {
  if (N % 2) return BT_ERR_INVALID_ARG;
  return moe_grouped(codes, scales, biases, bits, group_size, num_experts, N, K, expert_offsets, total_rows,
                     x_row_index, x, x_dtype, h, h_dtype, 1, stream);
}

bt_status bt_moe_qgemv_pairs(const uint32_t* codes, const uint16_t* scales, const uint16_t* biases, int bits,
                             int group_size, int num_experts, int N, int K, const int32_t* topk_ids, int tokens,
                             int top_k, const void* x, bt_dtype x_dtype, void* y, bt_dtype y_dtype, int swiglu,
                             cudaStream_t stream) {
  bt_status s = check_weights(codes, scales, biases, bits, group_size, N, K);
  if (s != BT_OK) return s;
  if (num_experts <= 0 || num_experts > 4096 || tokens < 0 || top_k < 1 || top_k > 32 || !x || !y || !topk_ids ||
      !half_dtype(x_dtype) || !out_dtype(y_dtype) || (swiglu && N % 2))
    return BT_ERR_INVALID_ARG;
  if (!aligned16(x)) return BT_ERR_MISALIGNED;
  if ((long long)tokens * top_k > (1LL << 30)) return BT_ERR_UNSUPPORTED;
  if (tokens == 0) return BT_OK;
  RowMap rm;
  rm.pair_ids = topk_ids;
  rm.top_k = top_k;
  rm.num_experts = num_experts;
  rm.swiglu = swiglu ? 1 : 0;
  return run_gemv(codes, scales, biases, bits, group_size, N, K, x, x_dtype, y, y_dtype, tokens * top_k, rm, stream);
}

bt_status bt_moe_down_combine(const uint32_t* codes, const uint16_t* scales, const uint16_t* biases, int bits,
                              int group_size, int num_experts, int N, int K, const int32_t* topk_ids,
                              const float* gates, int tokens, int top_k, const void* h, bt_dtype h_dtype,
                              void* out, bt_dtype o_dtype, cudaStream_t stream) {
  bt_status s = check_weights(codes, scales, biases, bits, group_size, N, K);
  if (s != BT_OK) return s;
  if (num_experts <= 0 || num_experts > 4096 || tokens < 0 || top_k < 1 || top_k > 32 || !topk_ids || !gates ||
      !h || !out || !half_dtype(h_dtype) || !out_dtype(o_dtype))
    return BT_ERR_INVALID_ARG;
  if (!aligned16(h)) return BT_ERR_MISALIGNED;
  if (tokens == 0) return BT_OK;
  // every segment copy (one expert's rows) must start and end on 16 bytes
  const long long seg_rb = (long long)K * bits / 8, seg_pb = 2LL * param_groups(bits, K, group_size);
  if ((N * seg_rb) % 16 || (N * seg_pb) % 16 || (long long)top_k * K > kMaxK) return BT_ERR_UNSUPPORTED;
  const int ktot = top_k * K;
  GemvParams p{};
  p.codes = codes;
  p.scales = scales;
  p.biases = biases;
  p.x = h;
  p.y = out;
  p.N = N;
  p.K = ktot;
  p.G = param_groups(bits, ktot, group_size);
  p.gshift = group_shift(group_size);
  p.num_experts = num_experts;
  p.seg_ids = topk_ids;
  p.seg_gates = gates;
  p.nseg = top_k;
  p.seg_k = K;
  p.err = device_error_word();
  p.timeout_ns = opts().wait_timeout_ns;
  p.const_weights = opts().pdl && opts().const_weights;
  p.drop_stage = opts().test_drop_stage.exchange(0);
  const GemvPlan pl = plan_gemv(bits, gemv_fast_path(bits, h_dtype), N, ktot, tokens, 0, sm_count(), group_size,
                                false, top_k);
  if (!pl.feasible) return BT_ERR_UNSUPPORTED;
  return cuda_status(launch_gemv(p, pl, bits, h_dtype, o_dtype, stream));
}

bt_status bt_moe_route(const int32_t* topk_ids, int tokens, int top_k, int num_experts, int32_t* expert_offsets,
                       int32_t* pair_index, int32_t* pair_row, int32_t* pair_token, cudaStream_t stream) {
  if (tokens < 0 || top_k < 1 || top_k > 32 || num_experts < 1 || num_experts > 4096) return BT_ERR_INVALID_ARG;
  if (!expert_offsets || (tokens > 0 && (!topk_ids || !pair_index || !pair_row))) return BT_ERR_INVALID_ARG;
  if ((long long)tokens * top_k > (1LL << 30)) return BT_ERR_UNSUPPORTED;
  return cuda_status(launch_moe_route(topk_ids, tokens, top_k, num_experts, expert_offsets, pair_index, pair_row,
                                      pair_token, stream));
}

bt_status bt_swiglu(const void* gate_up, bt_dtype in_dtype, int rows, int inter, void* h, bt_dtype h_dtype,
                    cudaStream_t stream) {
  if (rows < 0 || inter <= 0 || !out_dtype(in_dtype) || !out_dtype(h_dtype)) return BT_ERR_INVALID_ARG;
  if (rows > 0 && (!gate_up || !h)) return BT_ERR_INVALID_ARG;
  return cuda_status(launch_swiglu(gate_up, in_dtype, rows, inter, h, h_dtype, stream));
}

bt_status bt_moe_combine(const void* y_grouped, bt_dtype y_dtype, const float* gates, const int32_t* pair_row,
                         int tokens, int top_k, int hidden, void* out, bt_dtype out_dtype_, cudaStream_t stream) {
  if (tokens < 0 || top_k < 1 || top_k > 32 || hidden <= 0 || !out_dtype(y_dtype) || !out_dtype(out_dtype_))
    return BT_ERR_INVALID_ARG;
  if (tokens > 65535) return BT_ERR_UNSUPPORTED;
  if (tokens > 0 && (!y_grouped || !gates || !pair_row || !out)) return BT_ERR_INVALID_ARG;
  return cuda_status(launch_combine(y_grouped, y_dtype, gates, pair_row, tokens, top_k, hidden, out, out_dtype_,
                                    stream));
}

}  // extern "C"
