// Tensor-core dequant-GEMM (tcgen05 / TMEM / TMA) for prefill, M >= 16.
// BaseRT pages, thetesserapress.com "BaseRT claims fastest Apple Silicon
// inference", section "What BaseRT does differently" (prefill, M > 1, runs a
// GEMM that expands the codes in its inner loop; full-precision weights never
// reach memory) and section "Where the wins land" (dense prefill keeps the
// matrix units busy); gist.science "Metodologia" (tiled GEMM on the matrix
// units).
//
// Layout of one CTA tile (swap-AB: weights are the MMA's M side):
//   D[n, m] = sum_k W_deq[n0 + n, k] * X[m0 + m, k],  n < 128, m < BN
//   A = dequantized weight tile, 128 x 64 (one quantization group) per K
//       block, bf16/f16, written by the dequant warps straight into a tensor
//       memory slot (tcgen05.st; lane = weight row, column j = k 2j, 2j+1) and
//       read from there by the MMA, so it never passes through shared memory;
//   B = X tile, BN x 64, loaded by TMA with 128-byte swizzle (shared memory);
//   D = fp32 accumulator in tensor memory (128 lanes x BN columns).
// Warp roles: warp 0 issues TMA loads of the packed codes and of X; warp 1
// owns the tensor-memory allocation and one of its threads issues
// tcgen05.mma; warps 2..9 dequantize, warp w for the rows of TMEM lanes
// 32*(w%4), and then drain the accumulator to global memory.
//
// Dequantization and its rounding.  The codes become exact fp16 "1024 + q"
// pairs (one LOP3 per pair).  With fp16 X the weight is s*q + b from one
// f16x2 FMA of the exact integer (one rounding, to fp16).  With bf16 X each
// weight is formed in fp32 from the exact fp16 scale, w = s*(1024+q) + b',
// b' = b - 1024*s (the product is exact and the FMA rounds once), then
// rounded once to bf16.  A bf16 weight keeps 8 significant bits, so when Y is
// fp32 the kernel also writes the residual w - bf16(w) as a second bf16 A
// tile and issues the MMAs of both (A = hi + lo carries 16 bits), which keeps
// the fp32 output within its 1e-3 relative bound at any K.
//
// The per-row fp16 scales/biases of the CTA's K range are staged in shared
// memory once, with cp.async, before the main loop.  All waits are bounded.
#include <cuda.h>

#include <cstring>

#include "bt_common.cuh"
#include "qgemm.cuh"

namespace bt {
namespace tc {

constexpr int BM = 128;                  // weight rows per tile (MMA M)
constexpr int BK = 64;                   // K per stage = one quantization group
// Codes bytes per weight row in one stage: one K block (8*BITS bytes), except
// for 3-bit codes, whose 24-byte K block is not the multiple of 16 bytes that a
// TMA box row needs: their stage holds the aligned pair of K blocks (48 bytes,
// starting at an even K block) and the dequant warps read the half at hand.
template <int BITS> constexpr int kRowBox = BITS == 3 ? 48 : 8 * BITS;
template <int BITS> __host__ __device__ __forceinline__ int box_x(int g) { return BITS == 3 ? (g & ~1) * 24 : g * 8 * BITS; }
template <int BITS> __device__ __forceinline__ int box_off(int g) { return BITS == 3 ? (g & 1) * 24 : 0; }
// Dequantizing warps: 8 cover one K block (4 TMEM lane quadrants x 2 halves of
// the 64 codes); with 16, two such sets take alternating K blocks, so one set's
// wait -> load -> dequant -> TMEM store chain overlaps the other's.
template <int DW> constexpr int kThreadsT = (2 + DW) * 32;
// A ring in tensor memory: the dequant warps write each K block's 128 x 64 bf16
// A tile into one of the A slots (column j holds k = 2j, 2j+1 of the row in
// that lane; a split slot holds the hi tile in columns 0..31 and the lo tile
// in 32..63) and the MMA reads it from there, so A never passes through
// shared memory (whose bandwidth the MMA's B operand and the TMA writes
// already need).
constexpr int kAStages = 4;
template <int BN> constexpr int acc_cols() { return BN < 32 ? 32 : BN; }
// Columns of one A slot: 32 (64 bf16/f16 k values), or 64 when the slot holds
// the hi and lo bf16 tiles of a split weight.
template <bool SPLIT> constexpr int a_slot_cols() { return SPLIT ? 64 : 32; }
// A slots in use: split tiles at narrow token widths take 3 slots, so that the
// allocation stays within 256 columns and two CTAs still fit an SM's TMEM.
template <int BN, bool SPLIT> constexpr int a_stages() { return (SPLIT && BN <= 64) ? 3 : kAStages; }
template <int BN, bool SPLIT> constexpr int tmem_cols() {
  constexpr int need = acc_cols<BN>() + a_stages<BN, SPLIT>() * a_slot_cols<SPLIT>();
  return need <= 32 ? 32 : need <= 64 ? 64 : need <= 128 ? 128 : need <= 256 ? 256 : 512;
}

struct TcParams {
  int M, N, K, G;          // G = K / 64: K blocks
  int GQ;                  // quantization groups per row (K / group size)
  int gshift;              // group of 32-code half h of K block kb: (2*kb + h) >> gshift
  int splits;              // CTAs of a cluster splitting K (gridDim.z); 1 = no split
  int gc_max;              // most quantization groups any split stages
  int stages;              // TMA ring depth (X tile + packed codes per K block)
  int astages;             // A ring depth (TMEM slots of dequantized weight tiles)
  int bn;
  uint32_t stage_bytes, x_bytes, c_bytes;   // stage_bytes: one TMA-ring slot
  const uint16_t* scales;
  const uint16_t* biases;
  void* y;
  bt_dtype y_dtype;
  int swiglu;                 // epilogue: rows 2i/2i+1 = gate_i/up_i -> Y [M, N/2] = silu(gate) * up
  unsigned* err;
  unsigned long long timeout_ns;
  // grouped experts
  const void* x;              // X base (grouped mode loads rows with cp.async)
  const int32_t* offsets;     // [E+1] device
  const int32_t* row_index;   // [total_rows] device or null
  int num_experts;
};

// ------------------------------------------------------------------ PTX
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int c0, int c1, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int c0, int c1, int c2,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::
          "r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
      : "memory");
}

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row core
// groups 1024 bytes apart (tile base 1024-byte aligned).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)1 << 16;              // leading byte offset (unused for swizzled K-major)
  d |= (uint64_t)(1024 >> 4) << 32;    // stride byte offset
  d |= (uint64_t)1 << 46;              // descriptor version
  d |= (uint64_t)2 << 61;              // 128-byte swizzle
  return d;
}

// Instruction descriptor, kind::f16: fp32 accumulate, A and B both bf16 or both
// f16, both K-major, M = 128, N = n.
__host__ __device__ constexpr uint32_t make_idesc(bool bf16, int n) {
  return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) | ((uint32_t)(n >> 3) << 17) |
         ((uint32_t)(BM >> 4) << 24);
}

// D (TMEM) [+]= A (TMEM) x B (shared memory descriptor).
__device__ __forceinline__ void mma_f16_ta(uint32_t tmem_d, uint32_t tmem_a, uint64_t bdesc, uint32_t idesc,
                                           uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(
          tmem_d),
      "r"(tmem_a), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 16 consecutive 32-bit columns of this thread's TMEM lane (warp-wide, lanes of the warp's quarter).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
        "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t map_to_rank(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
__device__ __forceinline__ void st_cluster_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared::cluster.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
               : "memory");
}

__device__ __forceinline__ uint32_t lds32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ uint16_t lds16(uint32_t a) {
  uint16_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ void lds128(uint32_t a, uint32_t& x, uint32_t& y, uint32_t& z, uint32_t& w) {
  asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];" : "=r"(x), "=r"(y), "=r"(z), "=r"(w) : "r"(a));
}
__device__ __forceinline__ float4 lds128f(uint32_t a) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(a));
  return v;
}


// ------------------------------------------------------------------ dequant math
// Half-precision pair arithmetic (the fp16-X path).
__device__ __forceinline__ uint32_t hsub2_f16(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t hfma2_f16(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}
// fp16 "1024 + q" in both halves of a word: exact for every code below 1024.
constexpr uint32_t kMagic16 = 0x64006400u;

// Both halves of an fp16 pair h = (1024 + q0, 1024 + q1) as weights in fp32:
// w = s*(1024 + q) + bf with bf = b - 1024*s.  The product of two fp16 values
// is exact in fp32 and the FMA rounds once (fma.rn.f32.f16: fp16 factors, fp32
// addend and result).
__device__ __forceinline__ void pair_to_f32(uint32_t h, uint16_t s16, float bf, float& w0, float& w1) {
  asm("{\n .reg .f16 a, b, s;\n mov.b32 {a, b}, %2;\n mov.b16 s, %3;\n"
      " fma.rn.f32.f16 %0, s, a, %4;\n fma.rn.f32.f16 %1, s, b, %4;\n}\n"
      : "=f"(w0), "=f"(w1)
      : "r"(h), "h"(s16), "f"(bf));
}
// Two fp32 values -> one bf16 pair (lo in bits 0..15), each rounded once.
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}
// The weight pair (w0, w1) for the A tile: bf16 hi = round(w), and with SPLIT
// the residual lo = round(w - hi), so that hi + lo holds w to 16 bits.
template <bool SPLIT>
__device__ __forceinline__ void emit_bf16(float w0, float w1, uint32_t& hi, uint32_t& lo) {
  hi = pack_bf16(w0, w1);
  if constexpr (SPLIT) {
    const float h0 = __uint_as_float(hi << 16), h1 = __uint_as_float(hi & 0xFFFF0000u);
    lo = pack_bf16(w0 - h0, w1 - h1);
  }
}

// Generic: code j (bits j*B.. of a little-endian word array) as an integer.
template <int B, int NW>
__device__ __forceinline__ uint32_t code_at(const uint32_t (&w)[NW], int j) {
  const int bit = j * B, wi = bit >> 5, off = bit & 31;
  uint32_t q = w[wi] >> off;
  if (off + B > 32) q |= w[wi + 1] << (32 - off);
  return q & ((1u << B) - 1u);
}

// The 16 code pairs of this thread's 32 codes as fp16 (1024 + q) pairs, in
// the order they are written: pair i holds codes (p_lo[i], p_hi[i]) of the
// chunk; `kord` tells whether pair i already holds codes (2i, 2i+1).
// Q4: per word, (q0,q4) (q1,q5) (q2,q6) (q3,q7) from one LOP3 each.
template <int BITS>
__device__ __forceinline__ void code_pairs(const uint32_t (&w)[BITS], uint32_t (&h)[16]) {
  if constexpr (BITS == 4) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      h[4 * c + 0] = lop3_and_or(w[c], 0x000F000Fu, kMagic16);         // (q0, q4)
      h[4 * c + 1] = lop3_and_or(w[c] >> 4, 0x000F000Fu, kMagic16);    // (q1, q5)
      h[4 * c + 2] = lop3_and_or(w[c] >> 8, 0x000F000Fu, kMagic16);    // (q2, q6)
      h[4 * c + 3] = lop3_and_or(w[c] >> 12, 0x000F000Fu, kMagic16);   // (q3, q7)
    }
  } else if constexpr (BITS == 8) {
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      h[2 * c] = prmt(w[c], kMagic16, 0x7170u);       // (q0, q1): bytes 0, 1 under 0x64 high bytes
      h[2 * c + 1] = prmt(w[c], kMagic16, 0x7372u);   // (q2, q3)
    }
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const uint32_t lo = code_at<BITS, BITS>(w, 2 * i), hi = code_at<BITS, BITS>(w, 2 * i + 1);
      uint32_t pr;
      asm("lop3.b32 %0, %1, %2, %3, 0xFE;" : "=r"(pr) : "r"(lo), "r"(hi << 16), "r"(kMagic16));   // lo | hi<<16 | M
      h[i] = pr;
    }
  }
}

// Dequantize this thread's 32 codes of one row into 16 pairs in k order
// (out[j] holds k = 2j, 2j+1): the A tile's 16 TMEM columns.  With SPLIT
// (bf16 only) `lo` receives the residual tile.
template <int BITS, bool BF16, bool SPLIT>
__device__ __forceinline__ void deq32(const uint32_t (&w)[BITS], uint16_t s16, uint16_t b16, uint32_t (&out)[16],
                                      uint32_t (&lo)[16]) {
  uint32_t h[16];
  code_pairs<BITS>(w, h);
  if constexpr (BF16) {
    const float s = __half2float(__ushort_as_half(s16));
    const float bf = __half2float(__ushort_as_half(b16)) - 1024.f * s;   // exact for min/max-quantized groups
    if constexpr (BITS == 4) {
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        float f[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) pair_to_f32(h[4 * c + i], s16, bf, f[i], f[i + 4]);   // codes i, i+4
#pragma unroll
        for (int j = 0; j < 4; ++j) emit_bf16<SPLIT>(f[2 * j], f[2 * j + 1], out[4 * c + j], lo[4 * c + j]);
      }
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        float f0, f1;
        pair_to_f32(h[i], s16, bf, f0, f1);
        emit_bf16<SPLIT>(f0, f1, out[i], lo[i]);
      }
    }
  } else {
    // fp16: the exact integer pair times s plus b, one rounding per weight
    const uint32_t s2 = (uint32_t)s16 | ((uint32_t)s16 << 16), b2 = (uint32_t)b16 | ((uint32_t)b16 << 16);
    uint32_t d[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) d[i] = hfma2_f16(hsub2_f16(h[i], kMagic16), s2, b2);
    if constexpr (BITS == 4) {
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const uint32_t* e = d + 4 * c;   // (q0,q4) (q1,q5) (q2,q6) (q3,q7)
        out[4 * c + 0] = prmt(e[0], e[1], 0x5410u);
        out[4 * c + 1] = prmt(e[2], e[3], 0x5410u);
        out[4 * c + 2] = prmt(e[0], e[1], 0x7632u);
        out[4 * c + 3] = prmt(e[2], e[3], 0x7632u);
      }
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) out[i] = d[i];
    }
  }
}

__device__ __forceinline__ void store_y(const TcParams& p, size_t i, float v) {
  if (p.y_dtype == BT_F32) store_out<BT_F32>(p.y, i, v);
  else if (p.y_dtype == BT_BF16) store_out<BT_BF16>(p.y, i, v);
  else store_out<BT_F16>(p.y, i, v);
}

// ------------------------------------------------------------------ kernel
template <int BITS, bool BF16, int BN, bool GROUPED, bool SPLIT, int DW>
__global__ void __launch_bounds__(kThreadsT<DW>, 1)
    qgemm_tc_kernel(const __grid_constant__ CUtensorMap map_codes, const __grid_constant__ CUtensorMap map_x,
                    const TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = p.stages;
  // K blocks of this split: boundaries rounded to even group indices (scale pairs
  // are staged with 4-byte copies)
  const int split = blockIdx.z;
  const int kb_lo = split == 0 ? 0 : ((split * p.G) / p.splits) & ~1;
  const int kb_hi = split == p.splits - 1 ? p.G : (((split + 1) * p.G) / p.splits) & ~1;
  const int KB = kb_hi - kb_lo;
  // quantization groups staged for this CTA (its K range starts on an even K
  // block, so on a group boundary for groups of 32, 64 and 128 codes)
  const int gq_lo = (2 * kb_lo) >> p.gshift;
  const int Gc = ((2 * kb_hi + (1 << p.gshift) - 1) >> p.gshift) - gq_lo;
  // shared memory: [TMA ring: S x (X tile | codes)][scales][biases][barriers]; the A ring is in TMEM
  const int SA = p.astages;   // A slots in use (<= kAStages, < S)
  uint8_t* tring = smem;
  uint16_t* sS = reinterpret_cast<uint16_t*>(tring + (size_t)S * p.stage_bytes);  // [128][Gc]
  uint16_t* sB = sS + BM * p.gc_max;                                               // [128][Gc]
  uint64_t* bars = reinterpret_cast<uint64_t*>(
      (reinterpret_cast<uintptr_t>(sB + BM * p.gc_max) + 7) & ~uintptr_t(7));
  uint64_t* full = bars;             // [S] X + codes landed
  uint64_t* empty = bars + S;        // [S] MMAs reading the slot's X done
  uint64_t* afull = bars + 2 * S;    // [SA] A tile written
  uint64_t* tmem_full = afull + kAStages;
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(tmem_full + 1);
  volatile int* fail = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int n0 = blockIdx.x * BM;
  int m0 = blockIdx.y * BN;     // first grouped/dense row of the tile
  int m_end = p.M;              // one past its last valid row
  int expert = 0;
  constexpr int kTmemCols = tmem_cols<BN, SPLIT>();
  constexpr uint32_t kACol0 = acc_cols<BN>();   // first column of the A slots
  constexpr uint32_t kASlot = a_slot_cols<SPLIT>();

  if constexpr (GROUPED) {
    // Tile blockIdx.y of the expert-major list of (expert, BN-row tile) pairs;
    // tiles past the end of the list exit before touching anything.
    __shared__ int s_tile[3];
    pdl_wait();   // offsets come from the routing kernel
    if (threadIdx.x < 32) {
      const int E = p.num_experts;
      int base = 0, found = -1;
      for (int e0 = 0; e0 < E && found < 0; e0 += 32) {
        const int e = e0 + (int)threadIdx.x;
        int cnt = 0, lo = 0;
        if (e < E) {
          lo = max(0, __ldg(p.offsets + e));
          cnt = max(0, min(__ldg(p.offsets + e + 1), p.M) - lo);
        }
        const int tiles = (cnt + BN - 1) / BN;
        int incl = tiles;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int v = __shfl_up_sync(0xffffffffu, incl, o);
          if (threadIdx.x >= (unsigned)o) incl += v;
        }
        const int excl = base + incl - tiles;
        const bool mine = tiles > 0 && (int)blockIdx.y >= excl && (int)blockIdx.y < excl + tiles;
        const unsigned hit = __ballot_sync(0xffffffffu, mine);
        if (hit) {
          found = 0;
          if (mine) {
            s_tile[0] = e;
            s_tile[1] = lo + ((int)blockIdx.y - excl) * BN;
            s_tile[2] = lo + cnt;
          }
        }
        base += __shfl_sync(0xffffffffu, incl, 31);
      }
      if (threadIdx.x == 0 && found < 0) s_tile[0] = -1;
    }
    __syncthreads();
    if (s_tile[0] < 0) return;
    expert = s_tile[0];
    m0 = s_tile[1];
    m_end = s_tile[2];
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], GROUPED ? 33 : 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < SA; ++a) {
      mbar_init(&afull[a], 8);   // one arrive per warp of the set that dequantized the K block
    }
    mbar_init(tmem_full, 1);
    *fail = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(const_cast<uint32_t*>(tmem_slot))),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_launch_dependents();

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    if constexpr (!GROUPED) {
      if (lane == 0) {
        pdl_wait();
        int s = 0;
        uint32_t ph = 0;
        int issued = 0;
        for (int kb = 0; kb < KB; ++kb) {
          if (kb >= S && !mbar_wait(&empty[s], ph ^ 1u, p.timeout_ns, p.err)) { *fail = 1; break; }
          if (*fail) break;
          uint8_t* st = tring + (size_t)s * p.stage_bytes;
          mbar_arrive_expect_tx(&full[s], p.c_bytes + p.x_bytes);
          const int g = kb_lo + kb;
          tma_load_2d(st + p.x_bytes, &map_codes, box_x<BITS>(g), n0, &full[s]);
          tma_load_2d(st, &map_x, g * BK, m0, &full[s]);
          ++issued;
          if (++s == S) { s = 0; ph ^= 1u; }
        }
        if (*fail) {   // let copies in flight land before shared memory is released
          for (int j = issued > S ? issued - S : 0; j < issued; ++j)
            mbar_wait(&full[j % S], (uint32_t)((j / S) & 1), p.timeout_ns, p.err);
        }
      }
    } else {
      // codes: one 3-D TMA box per stage (expert plane); X: the tile's rows,
      // gathered with 16-byte cp.async straight into the swizzled layout
      const uint16_t* xg = static_cast<const uint16_t*>(p.x);
      int s = 0;
      uint32_t ph = 0;
      int issued = 0;
      bool ok = true;
      for (int kb = 0; kb < KB; ++kb) {
        if (kb >= S) {
          bool w = true;
          if (lane == 0) w = mbar_wait(&empty[s], ph ^ 1u, p.timeout_ns, p.err);
          if (!__shfl_sync(0xffffffffu, (int)w, 0)) { ok = false; break; }
        }
        uint8_t* st = tring + (size_t)s * p.stage_bytes;
        const int g = kb_lo + kb;
        if (lane == 0) {
          mbar_arrive_expect_tx(&full[s], p.c_bytes);
          tma_load_3d(st + p.x_bytes, &map_codes, box_x<BITS>(g), n0, expert, &full[s]);
        }
        for (int i = lane; i < BN * 8; i += 32) {
          const int row = i >> 3, ch = i & 7;
          const int gr = m0 + row;
          uint8_t* dst = st + row * 128 + ((ch ^ (row & 7)) << 4);
          if (gr < m_end) {
            const int src = p.row_index ? __ldg(p.row_index + gr) : gr;
            cp_async16(dst, xg + (size_t)src * p.K + (size_t)g * BK + ch * 8);
          } else {
            *reinterpret_cast<uint4*>(dst) = make_uint4(0u, 0u, 0u, 0u);
          }
        }
        cp_async_mbar_arrive_noinc(&full[s]);
        ++issued;
        if (++s == S) { s = 0; ph ^= 1u; }
      }
      if (!ok) {
        *fail = 1;
        cp_async_wait_all();
        if (lane == 0)
          for (int j = issued > S ? issued - S : 0; j < issued; ++j)
            mbar_wait(&full[j % S], (uint32_t)((j / S) & 1), p.timeout_ns, p.err);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = make_idesc(BF16, BN);
      int s = 0, a = 0;
      uint32_t ph = 0, aph = 0;
      for (int kb = 0; kb < KB; ++kb) {
        // The dequant warps arrive on afull only after their own wait on this
        // K block's stage, so the stage's X tile has landed too.  (Each wait or
        // tcgen05 instruction costs this single thread ~60-100 cycles, and it
        // is the one that feeds the tensor core.)
        if (!mbar_wait(&afull[a], aph, p.timeout_ns, p.err)) {
          *fail = 1;
          break;
        }
        tc_fence_after();
        if constexpr (GROUPED) fence_proxy_async();   // X rows written by cp.async / zero fill are read by the tensor core
        const uint32_t a_tmem = tmem_base + kACol0 + (uint32_t)a * kASlot;
        const uint64_t bdesc = sw128_desc(smem_u32(tring) + (uint32_t)(s * p.stage_bytes));
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk) {   // 16 elements: 8 TMEM columns of A, 32 bytes of B per MMA step
          mma_f16_ta(tmem_base, a_tmem + (uint32_t)(kk * 8), bdesc + (uint64_t)(kk * 2), idesc, (kb | kk) != 0);
          if constexpr (SPLIT)   // the residual tile against the same X columns
            mma_f16_ta(tmem_base, a_tmem + 32u + (uint32_t)(kk * 8), bdesc + (uint64_t)(kk * 2), idesc, 1u);
        }
        mma_commit(&empty[s]);   // frees the TMA stage, and the A slot for K block kb + SA
        if (++s == S) { s = 0; ph ^= 1u; }
        if (++a == SA) { a = 0; aph ^= 1u; }
      }
      mma_commit(tmem_full);   // arrives once every MMA issued above has completed
    }
  } else {
    // ---------------------------------------------------------------- dequant warps
    const int t = threadIdx.x - 64;        // 0..32*DW-1
    // warp w may access TMEM lanes 32*(w%4)..: it dequantizes those 32 rows, the
    // first four warps the low 32 codes of each K block, the last four the high 32
    // warp w accesses TMEM lanes 32*(w%4)..: it dequantizes those 32 rows; h selects
    // the low or high 32 codes of a K block, grp which K blocks (kb % (DW/8))
    const int r = 32 * (warp & 3) + lane, h = ((warp - 2) >> 2) & 1, grp = (warp - 2) >> 3;
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
    // stage this CTA's scales and biases: rows n0..n0+127, groups gq_lo..+Gc
    const size_t row0 = ((size_t)expert * p.N + n0) * p.GQ;   // first staged parameter of the tile
    if (Gc == p.GQ && n0 + BM <= p.N &&
        (((reinterpret_cast<uintptr_t>(p.scales + row0) | reinterpret_cast<uintptr_t>(p.biases + row0)) & 15u) == 0)) {
      // whole rows: the tile's parameters are one contiguous block per array, laid
      // out as in shared memory, so they move in 16-byte pieces
      const uint8_t* gs = reinterpret_cast<const uint8_t*>(p.scales + row0);
      const uint8_t* gb = reinterpret_cast<const uint8_t*>(p.biases + row0);
      for (int i = t; i < BM * Gc * 2 / 16; i += DW * 32) {
        cp_async16(reinterpret_cast<uint8_t*>(sS) + i * 16, gs + i * 16);
        cp_async16(reinterpret_cast<uint8_t*>(sB) + i * 16, gb + i * 16);
      }
    } else {
      // part of a row (K split) or the ragged last rows: one parameter at a time
      for (int i = t; i < BM * Gc; i += DW * 32) {
        const int rr = i / Gc, gg = i % Gc;
        const int n = n0 + rr;
        uint16_t sv = 0, bv = 0;
        if (n < p.N) {
          const size_t off = ((size_t)expert * p.N + n) * p.GQ + gq_lo + gg;
          sv = __ldg(p.scales + off);
          bv = __ldg(p.biases + off);
        }
        sS[rr * Gc + gg] = sv;
        sB[rr * Gc + gg] = bv;
      }
    }
    cp_async_wait_all();
    asm volatile("bar.sync 1, %0;" ::"r"(DW * 32) : "memory");
    const uint32_t sS_a = smem_u32(sS), sB_a = smem_u32(sB);

    constexpr int NG = DW / 8;   // sets of dequant warps, taking K blocks in turn
    // Ring positions advance by NG per iteration (no division in the loop):
    // (s, ph) = stage and phase of K block kb, a = its A slot, (sp, pp) = stage
    // and phase of K block kb - SA (negative indices wrap to phase 1; they are
    // never waited on).  S >= 2 >= NG and SA < S.
    int s = grp, a = grp % SA, sp = grp - SA;
    uint32_t ph = 0, pp = 0;
    if (sp < 0) { sp += S; pp = 1; }
    for (int kb = grp; kb < KB; kb += NG) {
      if (!mbar_wait(&full[s], ph, p.timeout_ns, p.err)) { *fail = 1; break; }
      if (kb >= SA) {
        // The commit of K block kb - SA frees this A slot.  empty[] of its stage
        // completes once per use; its next completion needs K block kb - SA + S
        // > kb, whose MMA cannot run before this K block's A tile exists, so the
        // phase awaited here is the one of K block kb - SA.
        if (!mbar_wait(&empty[sp], pp, p.timeout_ns, p.err)) { *fail = 1; break; }
      }
      const uint32_t st = smem_u32(tring) + (uint32_t)(s * p.stage_bytes);
      const uint32_t caddr = st + p.x_bytes + r * kRowBox<BITS> + box_off<BITS>(kb_lo + kb) + h * (4 * BITS);
      uint32_t w[BITS];
      if constexpr (BITS == 4) {
        lds128(caddr, w[0], w[1], w[2], w[3]);
      } else if constexpr (BITS == 8) {
        lds128(caddr, w[0], w[1], w[2], w[3]);
        lds128(caddr + 16, w[4], w[5], w[6], w[7]);
      } else {
#pragma unroll
        for (int i = 0; i < BITS; ++i) w[i] = lds32(caddr + 4 * i);
      }
      const int gq = ((2 * (kb_lo + kb) + h) >> p.gshift) - gq_lo;   // this thread's 32 codes' group
      const uint16_t s16 = lds16(sS_a + (uint32_t)(r * Gc + gq) * 2);
      const uint16_t b16 = lds16(sB_a + (uint32_t)(r * Gc + gq) * 2);
      uint32_t v[16], vlo[16];
      deq32<BITS, BF16, SPLIT>(w, s16, b16, v, vlo);
      const uint32_t slot = tmem_base + lane_base + kACol0 + (uint32_t)a * kASlot + (uint32_t)(16 * h);
      tmem_st16(slot, v);
      if constexpr (SPLIT) tmem_st16(slot + 32u, vlo);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&afull[a]);
      s += NG;
      if (s >= S) { s -= S; ph ^= 1u; }
      sp += NG;
      if (sp >= S) { sp -= S; pp ^= 1u; }
      a += NG;
      while (a >= SA) a -= SA;
    }

  }

  // ------------------------------------------------------------------ epilogue
  // Warps 2..DW+1 drain the accumulator: warp w reads TMEM lanes 32*(w%4).. (the
  // tile rows it may access) and every (DW/4)-th 16-column chunk.  With a K split
  // the partial tiles meet in distributed shared memory first: chunk c belongs
  // to cluster rank c % splits, every rank sends its partial of that chunk to
  // the owner's receive slot [sender], and the owner sums the slots in rank
  // order (deterministic) and stores.
  const bool epi = warp >= 2;
  bool ok = true;
  if (epi) {
    ok = mbar_wait(tmem_full, 0, p.timeout_ns, p.err) && !*fail;
    tc_fence_after();
  }
  const int q = warp & 3;
  const int col_sel = (warp - 2) >> 2;   // this warp's share of the 16-column chunks
  constexpr int kColSets = DW / 4;
  const int row = 32 * q + lane;
  const int n = n0 + row;
  const uint32_t taddr_row = tmem_base + ((uint32_t)(32 * q) << 16);
  if (p.splits == 1) {
    if (epi) {
      for (int c0 = 16 * col_sel; c0 < BN; c0 += 16 * kColSets) {
        uint32_t v[16];
        tmem_ld16(taddr_row + (uint32_t)c0, v);
        if (p.swiglu) {
          // gate row (even TMEM lane) and its up row (the next lane, same warp)
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float gt = __uint_as_float(v[j]);
            const float up = __shfl_xor_sync(0xffffffffu, gt, 1);
            const int m = m0 + c0 + j;
            if (ok && !(row & 1) && n < p.N && m < m_end)
              store_y(p, (size_t)m * (p.N / 2) + (n >> 1), gt / (1.f + expf(-gt)) * up);
          }
        } else if (ok && n < p.N) {
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int m = m0 + c0 + j;
            if (m < m_end) store_y(p, (size_t)m * p.N + n, __uint_as_float(v[j]));
          }
        }
      }
    }
  } else {
    const int R = p.splits;
    constexpr int kChunks = BN / 16;
    const int owned_max = (kChunks + R - 1) / R;
    // receive area (reuses the pipeline stages): [R senders][128 rows][owned_max * 16] fp32
    float* recv = reinterpret_cast<float*>(smem);
    const uint32_t recv_s = smem_u32(recv);
    tc_fence_before();
    cluster_sync_all();            // every CTA of the cluster is past its main loop
    tc_fence_after();
    if (epi) {
      for (int c0 = 16 * col_sel; c0 < BN; c0 += 16 * kColSets) {
        uint32_t v[16];
        tmem_ld16(taddr_row + (uint32_t)c0, v);
        const int chunk = c0 >> 4, owner = chunk % R, slot = chunk / R;
        const uint32_t local = recv_s + (uint32_t)((((split * BM) + row) * owned_max + slot) * 16 * 4);
        const uint32_t remote = map_to_rank(local, (uint32_t)owner);
#pragma unroll
        for (int j = 0; j < 16; j += 4) st_cluster_v4(remote + j * 4, v[j], v[j + 1], v[j + 2], v[j + 3]);
      }
    }
    cluster_sync_all();            // every partial is in its owner's receive area
    if (epi && ok && n < p.N) {
      for (int slot = col_sel; slot < owned_max; slot += kColSets) {
        const int chunk = slot * R + split;
        if (chunk >= kChunks) break;
        float acc[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) acc[j] = 0.f;
        for (int sdr = 0; sdr < R; ++sdr) {
          const uint32_t src = recv_s + (uint32_t)((((sdr * BM) + row) * owned_max + slot) * 16 * 4);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float4 f = lds128f(src + 16 * j);
            acc[4 * j] += f.x; acc[4 * j + 1] += f.y; acc[4 * j + 2] += f.z; acc[4 * j + 3] += f.w;
          }
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int m = m0 + chunk * 16 + j;
          if (m < m_end) store_y(p, (size_t)m * p.N + n, acc[j]);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(kTmemCols)
                 : "memory");
  }
}

// ------------------------------------------------------------------ host side
// Dequant warps per CTA.  Default: 16 for dense launches (one CTA per SM, so
// more warps hide the dequant latency) and 8 for grouped ones (narrow expert
// tiles run two CTAs per SM, which 18 warps' registers would not allow).
// BT_OPT_GEMM_DEQ_WARPS = 8 or 16 forces either.
inline int tc_dequant_warps(bool grouped) {
  const int o = opts().gemm_deq_warps;
  if (o == 8 || o == 16) return o;
  return grouped ? 8 : 16;
}

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  return fn;
}

// Shared memory of one CTA for a given K split (mirrors the layout in the kernel).
// Quantization groups of K blocks [lo, hi) (lo even) with groups of 32 << gshift codes.
inline int groups_in(int lo, int hi, int gshift) {
  return ((2 * hi + (1 << gshift) - 1) >> gshift) - ((2 * lo) >> gshift);
}

template <int BITS, int BN, bool GROUPED>
size_t tc_smem_bytes(int K, int splits, int* stages_out, int* k_blocks_out = nullptr, int gshift = 1) {
  const int G_all = K / BK;
  int kb_max = 0, gq_max = 0;
  for (int z = 0; z < splits; ++z) {
    const int lo = z == 0 ? 0 : ((z * G_all) / splits) & ~1;
    const int hi = z == splits - 1 ? G_all : (((z + 1) * G_all) / splits) & ~1;
    if (hi - lo < 1) return 0;
    kb_max = std::max(kb_max, hi - lo);
    gq_max = std::max(gq_max, groups_in(lo, hi, gshift));
  }
  const uint32_t x_bytes = BN * BK * 2, c_bytes = BM * kRowBox<BITS>;
  const uint32_t stage_bytes = (x_bytes + c_bytes + 1023u) & ~1023u;
  const size_t params_bytes = (size_t)2 * BM * gq_max * sizeof(uint16_t);
  const size_t fixed = 1024 + params_bytes + 8 + (size_t)(2 * 12 + 2 * kAStages + 1) * 8 + 16;
  const size_t budget = (GROUPED && BN <= 32) ? 112 * 1024 : 222 * 1024;
  int stages = (int)((budget - std::min(budget, fixed)) / stage_bytes);
  stages = std::max(2, std::min(12, stages));
  const int chunks = BN / 16, owned_max = (chunks + splits - 1) / splits;
  const size_t recv_bytes = splits > 1 ? (size_t)splits * BM * owned_max * 16 * 4 : 0;
  while ((size_t)stages * stage_bytes < recv_bytes) ++stages;
  if (stages_out) *stages_out = stages;
  if (k_blocks_out) *k_blocks_out = kb_max;
  return fixed + (size_t)stages * stage_bytes;
}

// K split for a dense launch: minimize waves x (K blocks per split + fixed cost),
// where waves come from how many clusters of that size fit on the device at once.
int choose_splits(int tiles, int K, int sms, int group);

template <int BITS, bool BF16, int BN, bool GROUPED, bool SPLIT, int DW>
cudaError_t launch_tc_t(const GemmParams& gp, bt_dtype yd, int splits, cudaStream_t st) {
  if (splits <= 0) splits = GROUPED ? 1 : choose_splits(((gp.N + BM - 1) / BM) * ((gp.M + BN - 1) / BN), gp.K, sm_count(), gp.group);
  EncodeTiledFn enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  const int row_bytes = gp.K * BITS / 8;
  CUtensorMap mc, mx;
  memset(&mx, 0, sizeof(mx));
  if constexpr (GROUPED) {
    cuuint64_t dims[3] = {(cuuint64_t)row_bytes, (cuuint64_t)gp.N, (cuuint64_t)gp.num_experts};
    cuuint64_t strides[2] = {(cuuint64_t)row_bytes, (cuuint64_t)row_bytes * gp.N};
    cuuint32_t box[3] = {(cuuint32_t)kRowBox<BITS>, (cuuint32_t)BM, 1};
    cuuint32_t es[3] = {1, 1, 1};
    if (enc(&mc, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint32_t*>(gp.codes), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  } else {
    cuuint64_t dims[2] = {(cuuint64_t)row_bytes, (cuuint64_t)gp.N};
    cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
    cuuint32_t box[2] = {(cuuint32_t)kRowBox<BITS>, (cuuint32_t)BM};
    cuuint32_t es[2] = {1, 1};
    if (enc(&mc, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint32_t*>(gp.codes), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  if constexpr (!GROUPED) {
    cuuint64_t dims[2] = {(cuuint64_t)gp.K, (cuuint64_t)gp.M};
    cuuint64_t strides[1] = {(cuuint64_t)gp.K * 2};
    cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)BN};
    cuuint32_t es[2] = {1, 1};
    if (enc(&mx, BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
            const_cast<void*>(gp.x), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  TcParams p{};
  p.M = gp.M;
  p.N = gp.N;
  p.K = gp.K;
  p.G = gp.K / BK;
  p.GQ = gp.K / gp.group;
  p.gshift = gp.group == 32 ? 0 : (gp.group == 64 ? 1 : 2);
  p.splits = splits;
  int gc_max = 0;
  for (int z = 0; z < splits; ++z) {   // same split boundaries as the kernel
    const int lo = z == 0 ? 0 : ((z * p.G) / splits) & ~1;
    const int hi = z == splits - 1 ? p.G : (((z + 1) * p.G) / splits) & ~1;
    if (hi - lo < 1) return cudaErrorInvalidValue;
    gc_max = std::max(gc_max, groups_in(lo, hi, p.gshift));
  }
  p.gc_max = gc_max;
  p.bn = BN;
  p.x_bytes = BN * BK * 2;
  p.c_bytes = BM * kRowBox<BITS>;
  p.stage_bytes = (p.x_bytes + p.c_bytes + 1023u) & ~1023u;
  p.scales = gp.scales;
  p.biases = gp.biases;
  p.y = gp.y;
  p.y_dtype = yd;
  p.swiglu = gp.swiglu;
  p.err = gp.err;
  p.timeout_ns = gp.timeout_ns;
  p.x = gp.x;
  p.offsets = gp.offsets;
  p.row_index = gp.row_index;
  p.num_experts = gp.num_experts;
  int stages = 0;
  const size_t smem = tc_smem_bytes<BITS, BN, GROUPED>(gp.K, splits, &stages, nullptr, p.gshift);
  if (smem == 0) return cudaErrorInvalidValue;
  p.stages = stages;
  p.astages = std::min(a_stages<BN, SPLIT>(), stages - 1);   // the dequant waits rely on S > SA
  if (smem > 227 * 1024) return cudaErrorInvalidValue;
  auto k = qgemm_tc_kernel<BITS, BF16, BN, GROUPED, SPLIT, DW>;
  static std::atomic<uint64_t> smem_raised{0};
  cudaError_t e = raise_smem_limit(reinterpret_cast<const void*>(k), smem_raised);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  // grouped: an upper bound on the (expert, tile) list, sum over experts of ceil(rows / BN)
  const long long ytiles = GROUPED ? (long long)(gp.M + BN - 1) / BN + std::min(gp.num_experts, gp.M)
                                   : (gp.M + BN - 1) / BN;
  if (ytiles > 65535) return cudaErrorInvalidValue;
  cfg.gridDim = dim3((gp.N + BM - 1) / BM, (unsigned)ytiles, splits);
  cfg.blockDim = dim3(kThreadsT<DW>);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = opts().pdl ? 1 : 0;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 1;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = splits;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, k, mc, mx, p);
}

// K split for a dense launch.  Measured on B300: launches whose CTA count
// stays at or below ~85% of the SMs run in one wave with room for cluster
// placement, while fuller grids of split clusters spill into a second wave and
// lose more than the split gains.  So: the largest split (1, 2, 3, 4, 6, 8,
// keeping >= 4 K blocks per split) with tiles x split <= 0.85 x SMs.
int choose_splits(int tiles, int K, int sms, int group) {
  const int kb = K / BK;
  // each split stages at most 192 quantization groups of parameters
  const int gq = K / group;
  const int need = (gq + 191) / 192;
  int min_sp = 1;
  for (int sp : {1, 2, 3, 4, 6, 8})
    if (sp >= need) { min_sp = sp; break; }
  const int forced = opts().gemm_splits;
  if (forced > 0) return std::max(min_sp, std::min(forced, kb / 2));
  const int limit = (sms * 85) / 100;
  int best = 1;
  for (int sp : {2, 3, 4, 6, 8})
    if (kb / sp >= 4 && tiles * sp <= limit) best = sp;
  return std::max(best, min_sp);
}

template <int BITS, bool BF16, bool SPLIT, int DW>
cudaError_t launch_tc_bn_dw(const GemmParams& gp, bt_dtype yd, int bn, int splits, cudaStream_t st) {
  switch (bn) {
    case 32: return launch_tc_t<BITS, BF16, 32, false, SPLIT, DW>(gp, yd, splits, st);
    case 64: return launch_tc_t<BITS, BF16, 64, false, SPLIT, DW>(gp, yd, splits, st);
    case 128: return launch_tc_t<BITS, BF16, 128, false, SPLIT, DW>(gp, yd, splits, st);
    default: return launch_tc_t<BITS, BF16, 256, false, SPLIT, DW>(gp, yd, splits, st);
  }
}

template <int BITS, bool BF16, bool SPLIT>
cudaError_t launch_tc_bn(const GemmParams& gp, bt_dtype yd, int bn, int splits, cudaStream_t st) {
  if (tc_dequant_warps(false) == 8) return launch_tc_bn_dw<BITS, BF16, SPLIT, 8>(gp, yd, bn, splits, st);
  return launch_tc_bn_dw<BITS, BF16, SPLIT, 16>(gp, yd, bn, splits, st);
}

// bf16 X with fp32 Y takes the split (hi + lo) A tiles; every other pairing the
// single tile (fp16 A is exact to one fp16 rounding; bf16 Y rounds coarser
// than a bf16 weight).
template <int BITS>
cudaError_t launch_tc_bits(const GemmParams& gp, bt_dtype xd, bt_dtype yd, int bn, int splits, cudaStream_t st) {
  if (xd == BT_BF16) {
    if (yd == BT_F32) return launch_tc_bn<BITS, true, true>(gp, yd, bn, splits, st);
    return launch_tc_bn<BITS, true, false>(gp, yd, bn, splits, st);
  }
  return launch_tc_bn<BITS, false, false>(gp, yd, bn, splits, st);
}


template <int BITS, bool BF16, bool SPLIT, int DW>
cudaError_t launch_tc_grouped_bn_dw(const GemmParams& gp, bt_dtype yd, int bn, cudaStream_t st) {
  switch (bn) {
    case 16: return launch_tc_t<BITS, BF16, 16, true, SPLIT, DW>(gp, yd, 1, st);
    case 32: return launch_tc_t<BITS, BF16, 32, true, SPLIT, DW>(gp, yd, 1, st);
    case 64: return launch_tc_t<BITS, BF16, 64, true, SPLIT, DW>(gp, yd, 1, st);
    default: return launch_tc_t<BITS, BF16, 128, true, SPLIT, DW>(gp, yd, 1, st);
  }
}

template <int BITS, bool BF16, bool SPLIT>
cudaError_t launch_tc_grouped_bn(const GemmParams& gp, bt_dtype yd, int bn, cudaStream_t st) {
  if (tc_dequant_warps(true) == 8) return launch_tc_grouped_bn_dw<BITS, BF16, SPLIT, 8>(gp, yd, bn, st);
  return launch_tc_grouped_bn_dw<BITS, BF16, SPLIT, 16>(gp, yd, bn, st);
}

template <int BITS>
cudaError_t launch_tc_grouped_bits(const GemmParams& gp, bt_dtype xd, bt_dtype yd, int bn, cudaStream_t st) {
  if (xd == BT_BF16) {
    if (yd == BT_F32) return launch_tc_grouped_bn<BITS, true, true>(gp, yd, bn, st);
    return launch_tc_grouped_bn<BITS, true, false>(gp, yd, bn, st);
  }
  return launch_tc_grouped_bn<BITS, false, false>(gp, yd, bn, st);
}

// Host-only geometry of one tensor-core launch: the shared memory, ring depth
// and grid that launch_tc_t computes for the same arguments.
template <int BITS, int BN, bool GROUPED>
GemmGeometry geometry_t(int M, int N, int K, int num_experts, int splits) {
  GemmGeometry g;
  g.bn = BN;
  g.splits = splits;
  int stages = 0, kb = 0;
  const size_t smem = tc_smem_bytes<BITS, BN, GROUPED>(K, splits, &stages, &kb);
  const long long ytiles = GROUPED ? (long long)(M + BN - 1) / BN + std::min(num_experts, M) : (M + BN - 1) / BN;
  g.stages = stages;
  g.k_blocks = kb;
  g.smem = (long long)smem;
  g.grid_x = (N + BM - 1) / BM;
  g.grid_y = (int)std::min<long long>(ytiles, 1LL << 30);
  g.grid_z = splits;
  g.feasible = smem != 0 && smem <= 227 * 1024 && ytiles <= 65535;
  return g;
}

template <int BITS>
GemmGeometry geometry_bits(int bn, int M, int N, int K, int num_experts, int splits) {
  if (num_experts > 0) {
    switch (bn) {
      case 16: return geometry_t<BITS, 16, true>(M, N, K, num_experts, 1);
      case 32: return geometry_t<BITS, 32, true>(M, N, K, num_experts, 1);
      case 64: return geometry_t<BITS, 64, true>(M, N, K, num_experts, 1);
      default: return geometry_t<BITS, 128, true>(M, N, K, num_experts, 1);
    }
  }
  switch (bn) {
    case 32: return geometry_t<BITS, 32, false>(M, N, K, 0, splits);
    case 64: return geometry_t<BITS, 64, false>(M, N, K, 0, splits);
    case 128: return geometry_t<BITS, 128, false>(M, N, K, 0, splits);
    default: return geometry_t<BITS, 256, false>(M, N, K, 0, splits);
  }
}

}  // namespace tc

int grouped_bn(int M, int num_experts) {
  const int avg = (M + num_experts - 1) / num_experts;
  if (avg <= 16) return 16;
  if (avg <= 32) return 32;
  if (avg <= 64) return 64;
  return 128;
}

// Grouped experts: token tiles sized to the mean rows per expert (the MMA's N
// runs 16..128), one CTA per (expert, 128 weight rows, token tile).
cudaError_t launch_gemm_tc_grouped(const GemmParams& gp, int bits, bt_dtype xd, bt_dtype yd, cudaStream_t st) {
  const int bn = grouped_bn(gp.M, gp.num_experts);
  switch (bits) {
    case 2: return tc::launch_tc_grouped_bits<2>(gp, xd, yd, bn, st);
    case 3: return tc::launch_tc_grouped_bits<3>(gp, xd, yd, bn, st);
    case 4: return tc::launch_tc_grouped_bits<4>(gp, xd, yd, bn, st);
    case 6: return tc::launch_tc_grouped_bits<6>(gp, xd, yd, bn, st);
    default: return tc::launch_tc_grouped_bits<8>(gp, xd, yd, bn, st);
  }
}


bool tc_shape_ok(int bits, int K, int group, bool grouped) {
  if (!(bits == 2 || bits == 3 || bits == 4 || bits == 6 || bits == 8)) return false;
  // the CTA's scales/biases are staged whole in shared memory, at most 192 groups:
  // dense launches split a longer K over a cluster, grouped ones run one CTA per tile
  if (K / group > (grouped ? 192 : 8 * 192)) return false;
  if (((size_t)K * bits / 8) % 16) return false;    // TMA row stride
  return true;
}

bool tc_supported(int bits, int K, int M, const GemmParams& gp) {
  if (!tc_shape_ok(bits, K, gp.group, gp.offsets != nullptr)) return false;
  if ((reinterpret_cast<uintptr_t>(gp.x) & 15) || (reinterpret_cast<uintptr_t>(gp.codes) & 15)) return false;
  (void)M;
  return true;
}

// Tile width and K split: token tiles of up to 256 columns; clusters of up to
// 8 CTAs split K so that tiles x splits covers the SMs (each split keeps at
// least 4 K blocks).
void plan_gemm_tc(int M, int N, int K, int sms, int& bn, int& splits) {
  bn = 256;
  if (M <= 32) bn = 32;
  else if (M <= 64) bn = 64;
  else if (M <= 128) bn = 128;
  splits = 0;   // chosen per instantiation from cluster occupancy (choose_splits)
  (void)N; (void)K; (void)sms;
}

GemmGeometry plan_gemm_tc_geometry(int bits, int M, int N, int K, int num_experts, int sms) {
  int bn = 0, splits = 1;
  if (num_experts > 0) {
    bn = grouped_bn(M, num_experts);
  } else {
    plan_gemm_tc(M, N, K, sms, bn, splits);
    splits = tc::choose_splits(((N + tc::BM - 1) / tc::BM) * ((M + bn - 1) / bn), K, sms, 64);
  }
  switch (bits) {
    case 2: return tc::geometry_bits<2>(bn, M, N, K, num_experts, splits);
    case 3: return tc::geometry_bits<3>(bn, M, N, K, num_experts, splits);
    case 4: return tc::geometry_bits<4>(bn, M, N, K, num_experts, splits);
    case 6: return tc::geometry_bits<6>(bn, M, N, K, num_experts, splits);
    default: return tc::geometry_bits<8>(bn, M, N, K, num_experts, splits);
  }
}

cudaError_t launch_gemm_tc(const GemmParams& gp, int bits, bt_dtype xd, bt_dtype yd, cudaStream_t st) {
  int bn, splits;
  plan_gemm_tc(gp.M, gp.N, gp.K, sm_count(), bn, splits);
  switch (bits) {
    case 2: return tc::launch_tc_bits<2>(gp, xd, yd, bn, splits, st);
    case 3: return tc::launch_tc_bits<3>(gp, xd, yd, bn, splits, st);
    case 4: return tc::launch_tc_bits<4>(gp, xd, yd, bn, splits, st);
    case 6: return tc::launch_tc_bits<6>(gp, xd, yd, bn, splits, st);
    default: return tc::launch_tc_bits<8>(gp, xd, yd, bn, splits, st);
  }
}

}  // namespace bt
