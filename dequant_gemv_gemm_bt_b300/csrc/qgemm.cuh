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
  const int32_t* offsets;
  const int32_t* row_index;
  int num_experts;
  unsigned* err;
  unsigned long long timeout_ns;
};

cudaError_t launch_gemm_simt(const GemmParams& p, int bits, bt_dtype xd, bt_dtype yd, cudaStream_t st);
bool tc_supported(int bits, int K, int M, const GemmParams& p);
cudaError_t launch_gemm_tc(const GemmParams& p, int bits, bt_dtype xd, bt_dtype yd, cudaStream_t st);
cudaError_t launch_gemm_tc_grouped(const GemmParams& p, int bits, bt_dtype xd, bt_dtype yd, cudaStream_t st);

}  // namespace bt
