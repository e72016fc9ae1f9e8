// Dequant-GEMV launch description shared by the dense and grouped-expert entry points.
#pragma once
#include <algorithm>
#include "bt_common.cuh"

namespace bt {

// One launch streams `problems` independent GEMVs of the same [N, K] shape.
// Dense: one problem.  Grouped experts at one row per expert (decode): problem
// r is grouped row r, whose expert is found from the device offsets.
struct GemvParams {
  const uint32_t* codes;
  const uint16_t* scales;
  const uint16_t* biases;
  const void* x;
  void* y;
  int N, K, G;
  // plan
  int rows_per_unit, row_bytes, stage_bytes, stages, kw, units_per_problem;
  long long num_units;
  long long total_cost;   // batched launches: work of all problems (rows x warps per row)
  // grouped experts (null offsets = dense)
  bt_dtype y_dtype;
  const int32_t* moe_offsets;
  const int32_t* row_index;
  int num_experts;
  int total_rows;
  // control
  unsigned* err;
  unsigned long long timeout_ns;
  int const_weights;
  int drop_stage;
  // tensor-pipe kernel: shared-memory bytes reserved for the per-group x sums
  int xsum_bytes;
  // quantization group of 32-code chunk c is c >> gshift (group size 32 << gshift)
  int gshift;
  // routed pairs (decode without a sort): problem r is pair r of a [tokens, top_k]
  // routing, expert pair_ids[r], x row r / top_k, output row r
  const int32_t* pair_ids;
  int top_k;
  // SwiGLU epilogue: weight rows interleaved (2i gate_i, 2i+1 up_i); the output
  // row holds N/2 values h_i = silu(gate_i . x) * (up_i . x)
  int swiglu;
  // K-segmented problems (expert down products summed into each token's output):
  // problem t's K is nseg segments of seg_k codes; segment s uses expert
  // seg_ids[t*nseg + s] and x segment seg_gates[t*nseg + s] * x[t*nseg + s]
  // (x holds the nseg rows of a token back to back).  N, G and row_bytes above
  // are then the totals over the segments.
  const int32_t* seg_ids;
  const float* seg_gates;
  int nseg, seg_k;
  // tensor-pipe kernel, four-column consumer: tokens (x rows) per problem, 1
  // or 2 (x and y of a problem are then [tokens, K] and [tokens, N]), and the
  // stride in groups between the tokens' staged x
  int tokens;
  int tok_groups;
};

// Batched launches: many independent GEMVs of the same bits and dtypes, each
// with its own weight, x, y, N and (mixed-K batches) K; the table travels in
// the kernel parameters.  Each problem carries its own row geometry: K, groups,
// row bytes, warps per row (kw) and rows per pipeline unit (rb).
constexpr int kBatchCap = 256;
struct GemvProblem {
  const uint32_t* codes;
  const uint16_t* scales;
  const uint16_t* biases;
  const void* x;
  void* y;
  int n;
  int k, g, row_bytes, kw, rb;
  int cw;             // work of one row for the CTA split: kw (CUDA-core kernel) or g (tensor-pipe kernel)
  int units;          // row blocks of this problem (rb rows each)
  long long unit_begin;
  long long cost_begin;   // work of the problems before this one (rows x cw)
};
template <int CAP> struct GemvBatch {
  int count;
  GemvProblem prob[CAP];
};

struct GemvPlan {
  bool fast;
  bool mma;        // the tensor-pipe kernel (qgemv_mma.cuh) rather than the CUDA-core one
  int mma_nw, mma_ctas, mma_unroll;   // its consumer warps per CTA, CTAs per SM, steps per loop iteration
  bool mma_cols4;  // its four-column consumer (four groups per MMA; needs K % 256 == 0)
  bool feasible;   // false: no GEMV kernel fits this shape (the caller uses the CUDA-core tile)
  int kw, cpl, ri, rows_per_unit, row_bytes, stage_bytes, stages, units_per_problem, grid;
  long long num_units;
  size_t smem;
};

// CTAs per SM the kernel is built for (its launch bounds): one x chunk per lane
// runs 2 CTAs with 4 rows in flight per warp, 3 with 2 or fewer; else 1.
inline int gemv_ctas_per_sm(int cpl, int ri) { return cpl == 1 ? (ri <= 2 ? 3 : 2) : 1; }

// Tensor-pipe GEMV: K limit and the kernel shapes that exist (consumer warps
// per CTA, CTAs per SM, steps per loop iteration), chosen by configuration id.
constexpr int kMmaMaxK = 8192;
struct MmaShape {
  int nw, ctas, unroll;
  bool cols4;   // four-column consumer: each MMA covers four quantization groups of 16 rows
};
MmaShape mma_shape(int cfg);   // cfg 0: the default shape

// Quantization groups per row whose scale and bias the kernels read: K / group,
// or 0 for fp16 weights (bits = 16), which have none.
inline int param_groups(int bits, int K, int group) { return bits == 16 ? 0 : K / group; }

// pair_rows: the launch's epilogue combines rows 2i and 2i+1 (SwiGLU), so at
// least two rows are in flight per warp.
GemvPlan plan_gemv(int bits, bool fast, int N, int K, int problems, int num_experts, int sms, int group = 64,
                   bool pair_rows = false, int nseg = 1);
// The tensor-pipe kernel's plan for the same arguments (infeasible when it does
// not apply: 4-bit codes, fp16 x, dense, K <= 8192, every unit 16-byte aligned).
GemvPlan plan_gemv_mma(int bits, bool fast, int N, int K, int problems, int num_experts, int sms,
                       int group = 64);
// One launch over problems of several K (each K <= 8192, one chunk per lane):
// fills every problem's geometry in `batch` and returns the launch plan
// (stage size covering the largest unit); infeasible when the problems need
// different kernel shapes.
GemvPlan plan_gemv_batch(int bits, bool fast, GemvBatch<kBatchCap>& batch, int sms, int group = 64);
// Staged x copies the tensor-pipe kernel keeps for `tokens` tokens per problem
// (its variants take 1, 2 or 4).
inline int token_slots(int tokens) { return tokens <= 1 ? 1 : (tokens == 2 ? 2 : (tokens <= 4 ? 4 : 8)); }
// tokens = 2..8: every problem has that many x rows and y rows (the four-column
// consumer with two tokens x four groups, four tokens x two groups or eight
// tokens x one group in the MMA's columns); infeasible unless every K is a
// multiple of 256.
GemvPlan plan_gemv_batch_mma(int bits, bool fast, GemvBatch<kBatchCap>& batch, int sms, int group = 64,
                             int tokens = 1);
cudaError_t launch_gemv(GemvParams& p, const GemvPlan& pl, int bits, bt_dtype xd, bt_dtype yd,
                        cudaStream_t stream, GemvBatch<kBatchCap>* batch = nullptr);

}  // namespace bt
