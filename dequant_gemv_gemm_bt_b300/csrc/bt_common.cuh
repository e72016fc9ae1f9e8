// Shared device helpers for libbt: half types, mbarrier / bulk-copy / PDL PTX
// wrappers, bounded waits and the device error word.
#pragma once
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <atomic>

#include "../../include/bt.h"

namespace bt {

// ------------------------------------------------------------------ limits
constexpr int kGroup = 64;        // quantization group along K
constexpr int kMaxK = 32768;

// Device error word: bit 0 = a bounded wait expired, bit 1 = bad device-side argument.
constexpr unsigned kErrTimeout = 1u;
constexpr unsigned kErrBadArg = 2u;

// One process-wide tuning value: bt_set_option may run on one host thread while
// another launches, so every read and write is a relaxed atomic (each value is
// read once per launch; no ordering between values is needed).
template <class T>
struct Opt {
  std::atomic<T> v;
  constexpr Opt(T x) : v(x) {}
  T load() const { return v.load(std::memory_order_relaxed); }
  operator T() const { return load(); }
  Opt& operator=(T x) {
    v.store(x, std::memory_order_relaxed);
    return *this;
  }
  T exchange(T x) { return v.exchange(x, std::memory_order_relaxed); }
};

struct LaunchOpts {
  Opt<bool> pdl{false};
  Opt<bool> const_weights{false};
  Opt<unsigned long long> wait_timeout_ns{4000000000ull};
  Opt<int> test_drop_stage{0};   // test hook: the next GEMV launch leaves one stage unfilled
  Opt<bool> gemv_generic{false}; // tuning: force the generic unpack path
  Opt<int> gemv_stages{0};       // tuning: pipeline depth override (0 = heuristic)
  Opt<int> gemm_path{0};         // tuning: 0 = heuristic, 1 = CUDA-core tile, 2 = tensor-core tile
  Opt<int> gemm_splits{0};       // tuning: tensor-core GEMM K split (0 = heuristic)
  Opt<int> gemv_max_cpl{0};      // tuning: GEMV chunks per lane before splitting K over warps (0 = heuristic)
  Opt<int> gemv_stage_kb{0};     // tuning: GEMV stage size in KiB (0 = heuristic)
  Opt<int> gemv_ri{0};           // tuning: GEMV rows in flight per warp (0 = heuristic)
  Opt<int> gemv_cuda_core{0};    // tuning: 1 = GEMV on the CUDA-core kernel even where the tensor-pipe one applies
  Opt<int> gemv_tensor_pipe{0};  // tuning: tensor-pipe GEMV 0 = by launch size, 1 = wherever it applies, 2 = never
  Opt<int> gemv_mma_stage_kb{0}; // tuning: tensor-pipe GEMV stage size in KiB (0 = heuristic)
  Opt<int> gemv_mma_cfg{0};      // tuning: tensor-pipe GEMV kernel shape (0 = default, 1..4)
  Opt<int> gemv_mma_ks{0};       // tuning: most quantization groups per warp in the tensor-pipe GEMV (0 = heuristic)
  Opt<int> gemm_deq_warps{0};    // tuning: tensor-core GEMM dequant warps per CTA, 8 or 16 (0 = 16 dense, 8 grouped)
  Opt<int> gemm_small_warps{0};  // tuning: small-token kernel consumer warps, 8 or 16 (0 = 16 where it fits)
};
LaunchOpts& opts();
unsigned* device_error_word();   // device address of the error word (current device)
int sm_count();                  // multiprocessors of the current device

// ------------------------------------------------------------ small device utils
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void set_device_error(unsigned* err, unsigned bits) {
  if (err) atomicOr(err, bits);
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

// One bounded probe of an mbarrier phase; the thread may be suspended in
// hardware for up to ~0.5 ms while the phase is incomplete, so waiting warps
// do not spin on the issue slots.
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(500000u)
      : "memory");
  return ok != 0;
}

// Bounded wait on an mbarrier phase.  Returns false (and sets the error word)
// when `timeout_ns` of global time pass without the phase completing.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, unsigned long long timeout_ns,
                                          unsigned* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (globaltimer_ns() - t0 > timeout_ns) {
      set_device_error(err, kErrTimeout);
      return false;
    }
  }
}

// ----------------------------------------------------- bulk (TMA 1-D) copies
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// global -> shared, completes `bytes` transactions on `bar`.  dst, src 16-B aligned, bytes % 16 == 0.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// 16-byte asynchronous copy global -> shared through L1 (no TMA engine), and an
// mbarrier arrive that fires once all of this thread's prior cp.async copies landed.
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_mbar_arrive_noinc(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// ---------------------------------------------------- programmatic dependent launch
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ----------------------------------------------------------------- halves
// Raises a kernel's dynamic shared-memory limit to the most the device allows
// next to the kernel's static shared memory, once per device, so the limit is
// not rewritten on every launch whose size differs from the previous one.
inline cudaError_t raise_smem_limit(const void* fn, std::atomic<uint64_t>& done) {
  int d = 0;
  cudaError_t e = cudaGetDevice(&d);
  if (e != cudaSuccess) return e;
  const uint64_t bit = d < 64 ? (uint64_t{1} << d) : 0;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  int mx = 0;
  e = cudaDeviceGetAttribute(&mx, cudaDevAttrMaxSharedMemoryPerBlockOptin, d);
  if (e != cudaSuccess) return e;
  cudaFuncAttributes fa;
  e = cudaFuncGetAttributes(&fa, fn);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, mx - (int)fa.sharedSizeBytes);
  if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_release);
  return e;
}

// (a & m) | c as one LOP3.  Written as a C++ expression with two constants the
// compiler emits two logic instructions; in the dequant loops that doubles the
// ALU-pipe work per code pair.
__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t m, uint32_t c) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(m), "r"(c));
  return d;
}

template <bt_dtype D> struct HalfT;
template <> struct HalfT<BT_F16> { using T = __half; };
template <> struct HalfT<BT_BF16> { using T = __nv_bfloat16; };

__device__ __forceinline__ float half_bits_to_float(uint16_t v, bt_dtype d) {
  if (d == BT_F16) return __half2float(__ushort_as_half(v));
  return __uint_as_float(static_cast<uint32_t>(v) << 16);
}

template <bt_dtype D> __device__ __forceinline__ float to_f32(uint16_t v) {
  if constexpr (D == BT_F16) return __half2float(__ushort_as_half(v));
  else return __uint_as_float(static_cast<uint32_t>(v) << 16);
}

template <bt_dtype D> __device__ __forceinline__ void store_out(void* base, size_t i, float v) {
  if constexpr (D == BT_F32) static_cast<float*>(base)[i] = v;
  else if constexpr (D == BT_F16) static_cast<__half*>(base)[i] = __float2half_rn(v);
  else static_cast<__nv_bfloat16*>(base)[i] = __float2bfloat16_rn(v);
}

}  // namespace bt
