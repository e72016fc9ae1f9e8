// Dequant-GEMM launch description (dense and grouped by expert).
#pragma once
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
bool tc_shape_ok(int bits, int K, int group = 64);
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

}  // namespace bt
