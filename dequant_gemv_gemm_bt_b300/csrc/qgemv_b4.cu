// Dequant-GEMV kernels for 4-bit codes (instantiations of qgemv_impl.cuh and,
// for the tensor-pipe path, qgemv_mma.cuh).
#include "qgemv_impl.cuh"
#include "qgemv_mma.cuh"

namespace bt {
cudaError_t launch_gemv_b4(const GemvParams& p, const GemvPlan& pl, bt_dtype xd, const GemvBatch<kBatchCap>* b,
                           cudaStream_t st) {
  return gemv::launch_bits<4>(p, pl, xd, b, st);
}
cudaError_t launch_gemv_mma_b4(const GemvParams& p, const GemvPlan& pl, const GemvBatch<kBatchCap>* b,
                               cudaStream_t st) {
  return gemv::launch_mma_bits<4>(p, pl, b, st);
}
}  // namespace bt
