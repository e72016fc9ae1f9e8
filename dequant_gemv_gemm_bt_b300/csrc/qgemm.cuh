// Dequant-GEMM launch description (dense and grouped by expert).
#pragma once
#include <cuda.h>

#include <algorithm>

#include "bt_common.cuh"

namespace bt {

// Y[m, n] = sum_k X[row(m), k] * w_deq_{e(m)}[n, k] for m < M.
// Dense: offsets == nullptr, one weight, row(m) = m.
// Grouped: rows [offsets[e], offsets[e+1]) use expert e; row(m) = row_index[m] when given.
struct GemmParams {
  const uint32_t* codes;
  const uint16_t* scales;
  const uint16_t* biases;
  const void* x;
  void* y;
  int M, N, K;
  int group;                 // quantization group size along K: 32, 64 or 128
  int swiglu;                // epilogue: rows 2i/2i+1 are gate_i/up_i; Y is [M, N/2], silu(gate) * up
  const int32_t* offsets;
  const int32_t* row_index;
  int num_experts;
  unsigned* err;
  unsigned long long timeout_ns;
};

cudaError_t launch_gemm_simt(const GemmParams& p, int bits, bt_dtype xd, bt_dtype yd, cudaStream_t st);
// The tensor-core path's limits on bits, K and group size (pointers are checked by tc_supported).
bool tc_shape_ok(int bits, int K, int group = 64, bool grouped = false);
bool tc_supported(int bits, int K, int M, const GemmParams& p);
cudaError_t launch_gemm_tc(const GemmParams& p, int bits, bt_dtype xd, bt_dtype yd, cudaStream_t st);
cudaError_t launch_gemm_tc_grouped(const GemmParams& p, int bits, bt_dtype xd, bt_dtype yd, cudaStream_t st);

// Launch geometry of one product, computed on the host only: the same choices
// the launchers make, for inspection and tests.
struct GemmGeometry {
  bool feasible = false;
  int bn = 0;            // token-tile width (the MMA's N on the tensor-core path)
  int splits = 1;        // K split (CTAs per cluster)
  int stages = 0;        // TMA ring depth
  int k_blocks = 0;      // largest number of 64-wide K blocks one split walks
  int grid_x = 0, grid_y = 0, grid_z = 0;
  long long smem = 0;    // dynamic shared memory per CTA
};
// num_experts == 0: dense product of M rows; > 0: grouped, M rows in total.
GemmGeometry plan_gemm_tc_geometry(int bits, int M, int N, int K, int num_experts, int sms);
GemmGeometry plan_gemm_simt_geometry(int M, int N, int num_experts);
// Token-tile width of a grouped tensor-core launch: the mean rows per expert, 16..128.
int grouped_bn(int M, int num_experts);

// Small token counts on the tensor pipe (qgemm_mma.cu): 4-bit codes, groups of
// 64, tokens as the N of mma.sync m16n8k16, each weight read from HBM once for
// every token of its problem (all M rows of a dense product, or one expert's rows).
struct SmallGeometry {
  bool feasible = false;
  int t8 = 0;            // n8 token tiles per pass: up to 8 * t8 tokens share one staging of x
  int nw = 0;            // consumer warps per CTA (8 or 16)
  int kw = 0;            // consumer warps splitting one 16-row tile's K range
  int rb = 0;            // weight rows per unit (one TMA ring stage)
  int stages = 0;        // ring depth
  int grid = 0;          // persistent CTAs (units beyond are walked in turn)
  long long smem = 0;    // dynamic shared memory per CTA
};
// num_experts == 0: dense product of M rows (M <= 32); > 0: grouped, M rows in total.
SmallGeometry plan_gemm_small(int bits, int M, int N, int K, int group, int num_experts, int sms);
// Shape limits plus the pointer alignment the TMA and 8-byte parameter copies need.
bool small_supported(int bits, const GemmParams& p);
cudaError_t launch_gemm_small(const GemmParams& p, int bits, bt_dtype xd, bt_dtype yd, cudaStream_t st);

// Several dense small-token products of the same M in one launch (at most
// small::kBatchLaunchCap problems per launch).
namespace small {
constexpr int kBatchLaunchCap = 120;
}
struct GemmProblem {
  const uint32_t* codes;
  const uint16_t* scales;
  const uint16_t* biases;
  const void* x;   // [M][K]
  void* y;         // [M][N]
  int N, K;
};
SmallGeometry plan_gemm_small_batched(const GemmProblem* probs, int count, int M, int sms);
bool small_batch_supported(const GemmProblem* probs, int count, int M, int bits, int group);
cudaError_t launch_gemm_small_batched(const GemmProblem* probs, int count, int M, bt_dtype xd, bt_dtype yd,
                                      unsigned* err, unsigned long long timeout_ns, cudaStream_t st);
// The same, prepared once (plan and tensor maps) and launched many times.
struct SmallBatchPrepared;
SmallBatchPrepared* prepare_gemm_small_batched(const GemmProblem* probs, int count, int M, bt_dtype xd, bt_dtype yd);
cudaError_t run_gemm_small_batched(const SmallBatchPrepared* pb, unsigned* err, unsigned long long timeout_ns,
                                   cudaStream_t st);
void free_gemm_small_batched(SmallBatchPrepared* pb);

namespace tc {
// cuTensorMapEncodeTiled from the driver (null if unavailable).
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_fn();
}  // namespace tc

}  // namespace bt
