// Dequant-GEMV kernels for fp16 weights (bits = 16) (instantiations of qgemv_impl.cuh).
#include "qgemv_impl.cuh"

namespace bt {
cudaError_t launch_gemv_b16(const GemvParams& p, const GemvPlan& pl, bt_dtype xd, const GemvBatch<kBatchCap>* b,
                            cudaStream_t st) {
  return gemv::launch_bits<16>(p, pl, xd, b, st);
}
}  // namespace bt
