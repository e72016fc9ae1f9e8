// Dequant-GEMV kernels for 8-bit codes (instantiations of qgemv_impl.cuh).
#include "qgemv_impl.cuh"

namespace bt {
cudaError_t launch_gemv_b8(const GemvParams& p, const GemvPlan& pl, bt_dtype xd, cudaStream_t st) {
  return gemv::launch_bits<8>(p, pl, xd, st);
}
cudaError_t launch_gemv_reg_b8(const GemvParams& p, const GemvPlan& pl, bt_dtype xd, cudaStream_t st) {
  return gemv::launch_reg_bits<8>(p, pl, xd, st);
}
}  // namespace bt
