// Dequant-GEMV kernels for 6-bit codes (instantiations of qgemv_impl.cuh).
#include "qgemv_impl.cuh"

namespace bt {
cudaError_t launch_gemv_b6(const GemvParams& p, const GemvPlan& pl, bt_dtype xd, const GemvBatch<kBatchCap>* b,
                           cudaStream_t st) {
  return gemv::launch_bits<6>(p, pl, xd, b, st);
}
}  // namespace bt
