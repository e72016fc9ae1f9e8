// Dequant-GEMV kernels for 5-bit codes (generic unpack path) (instantiations of qgemv_impl.cuh).
#include "qgemv_impl.cuh"

namespace bt {
cudaError_t launch_gemv_b5(const GemvParams& p, const GemvPlan& pl, bt_dtype xd, const GemvBatch<kBatchCap>* b,
                            cudaStream_t st) {
  return gemv::launch_bits<5>(p, pl, xd, b, st);
}
}  // namespace bt
