// Device code of the dequant-GEMV (M = 1, decode) and its batched form for
// mixture-of-experts decode.  BaseRT pages, thetesserapress.com "BaseRT claims
// fastest Apple Silicon inference", section "What BaseRT does differently": a
// GEMV of its own for M = 1, which expands the codes inside its inner loop, so
// the bytes it reads fall in proportion to the bits per weight.
//
// Design (B300):
//  * Persistent CTAs, each streaming a contiguous range of row blocks ("units")
//    through a shared-memory ring filled by 1-D bulk copies (TMA) issued by one
//    producer thread; weights are read exactly once, with an L2 evict-first hint.
//  * Each consumer lane owns a fixed K-slice of x in registers (loaded once per
//    problem), so shared-memory traffic is only the packed codes and the fp16
//    scale/bias of each row.
//  * Per group the product is factored as s * sum(q*x) + b * sum(x); sum(x) per
//    slice is precomputed, so the bias costs one FMA per 32 codes.
//  * Fast path (fp16 x, every bit width): codes become fp16 "1024 + c*q" with
//    one LOP3 / PRMT per two codes and are multiplied into fp32 accumulators
//    with mixed-precision FMA (one instruction at FFMA rate on sm_103); each
//    class's accumulator starts at minus its sum of 1024*x, which removes the
//    offset.  Bits 2/4/8 pair codes within a word; bits 3/6, whose codes
//    cross words, follow searched schedules of shifted windows
//    (qgemv_stream.h).  Generic path (bf16 x): funnel-shift extraction, exact
//    int->float via the 2^23 magic, fp32 FMA.
//  * A warp works on RI rows at once (independent FMA chains), reduces the RI
//    partials across lanes with a transpose-style shuffle tree (9 shuffles for
//    8 rows) and, when one warp covers a whole row, stores y directly with no
//    block-wide barrier.  When K is split over several warps the partials meet
//    in shared memory behind a named barrier of that row group.  No atomics:
//    results are bitwise deterministic.
//  * Batched launches carry each problem's row geometry (K, warps per row,
//    rows per unit), so one launch covers problems of different K; CTAs take
//    equal shares of work (rows x warps per row).
#pragma once
#include <type_traits>
#include <utility>

#include "bt_common.cuh"
#include "qgemv.cuh"
#include "qgemv_stream.h"

namespace bt {

namespace gemv {

// ------------------------------------------------------------ shared loads
__device__ __forceinline__ uint32_t lds32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t a) {
  uint2 v;
  asm volatile("ld.shared.v2.b32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
  return v;
}
__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
  return v;
}
__device__ __forceinline__ uint16_t lds16(uint32_t a) {
  uint16_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(a));
  return v;
}

// Load the BITS words of one 32-code chunk (4*BITS bytes) from shared or global memory.
template <int BITS, bool SMEM>
__device__ __forceinline__ void load_chunk(uint32_t saddr, const uint8_t* gptr, uint32_t (&w)[BITS]) {
  if constexpr (SMEM) {
    if constexpr (BITS == 4) {
      uint4 v = lds128(saddr); w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
    } else if constexpr (BITS == 8) {
      uint4 a = lds128(saddr), b = lds128(saddr + 16);
      w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w; w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
    } else if constexpr (BITS == 2) {
      uint2 v = lds64(saddr); w[0] = v.x; w[1] = v.y;
    } else if constexpr (BITS == 6) {
#pragma unroll
      for (int i = 0; i < 3; ++i) { uint2 v = lds64(saddr + 8 * i); w[2 * i] = v.x; w[2 * i + 1] = v.y; }
    } else if constexpr (BITS == 16) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        uint4 v = lds128(saddr + 16 * i); w[4 * i] = v.x; w[4 * i + 1] = v.y; w[4 * i + 2] = v.z; w[4 * i + 3] = v.w;
      }
    } else {
#pragma unroll
      for (int i = 0; i < BITS; ++i) w[i] = lds32(saddr + 4 * i);
    }
  } else {
    if constexpr (BITS == 4) {
      uint4 v = __ldg(reinterpret_cast<const uint4*>(gptr)); w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
    } else if constexpr (BITS == 8) {
      uint4 a = __ldg(reinterpret_cast<const uint4*>(gptr)), b = __ldg(reinterpret_cast<const uint4*>(gptr) + 1);
      w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w; w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
    } else if constexpr (BITS == 2 || BITS == 6) {
#pragma unroll
      for (int i = 0; i < BITS / 2; ++i) {
        uint2 v = __ldg(reinterpret_cast<const uint2*>(gptr) + i); w[2 * i] = v.x; w[2 * i + 1] = v.y;
      }
    } else if constexpr (BITS == 16) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        uint4 v = __ldg(reinterpret_cast<const uint4*>(gptr) + i);
        w[4 * i] = v.x; w[4 * i + 1] = v.y; w[4 * i + 2] = v.z; w[4 * i + 3] = v.w;
      }
    } else {
#pragma unroll
      for (int i = 0; i < BITS; ++i) w[i] = __ldg(reinterpret_cast<const uint32_t*>(gptr) + i);
    }
  }
}

// ------------------------------------------------------------ fast path math
// acc += x_lo * h.lo + x_hi * h.hi (one accumulator; two dependent FMAs).
__device__ __forceinline__ void fma_pair(float& acc, uint16_t x_lo, uint16_t x_hi, uint32_t hp) {
  asm("{\n .reg .f16 ha, hb;\n mov.b32 {ha, hb}, %3;\n"
      " fma.rn.f32.f16 %0, %1, ha, %0;\n fma.rn.f32.f16 %0, %2, hb, %0;\n}\n"
      : "+f"(acc) : "h"(x_lo), "h"(x_hi), "r"(hp));
}

// acc_lo += x_lo * h.lo and acc_hi += x_hi * h.hi (two accumulators).
__device__ __forceinline__ void fma_pair2(float& acc_lo, float& acc_hi, uint16_t x_lo, uint16_t x_hi, uint32_t hp) {
  asm("{\n .reg .f16 ha, hb;\n mov.b32 {ha, hb}, %4;\n"
      " fma.rn.f32.f16 %0, %2, ha, %0;\n fma.rn.f32.f16 %1, %3, hb, %1;\n}\n"
      : "+f"(acc_lo), "+f"(acc_hi) : "h"(x_lo), "h"(x_hi), "r"(hp));
}
// acc += x * h.lo, or x * h.hi when HIGH (a half that carries a code alone).
template <bool HIGH>
__device__ __forceinline__ void fma_half(float& acc, uint16_t x, uint32_t hp) {
  if constexpr (HIGH)
    asm("{\n .reg .f16 ha, hb;\n mov.b32 {ha, hb}, %2;\n fma.rn.f32.f16 %0, %1, hb, %0;\n}\n"
        : "+f"(acc) : "h"(x), "r"(hp));
  else
    asm("{\n .reg .f16 ha, hb;\n mov.b32 {ha, hb}, %2;\n fma.rn.f32.f16 %0, %1, ha, %0;\n}\n"
        : "+f"(acc) : "h"(x), "r"(hp));
}

__device__ __forceinline__ uint32_t lop_mask_or(uint32_t w, uint32_t mask) {
  return lop3_and_or(w, mask, 0x64006400u);
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// Number of distinct "classes" (power-of-two multipliers c in 1024 + c*q) per bits.
template <int BITS> struct FastClasses;
template <> struct FastClasses<2> { static constexpr int n = 5; };
template <> struct FastClasses<4> { static constexpr int n = 2; };
template <> struct FastClasses<8> { static constexpr int n = 1; };
template <> struct FastClasses<3> { static constexpr int n = StreamLayout<3>::n_classes; };
template <> struct FastClasses<6> { static constexpr int n = StreamLayout<6>::n_classes; };
template <> struct FastClasses<16> { static constexpr int n = 1; };
template <int BITS> constexpr bool kStreamBits = (BITS == 3 || BITS == 6);
// 5-bit codes have no fp16 pair schedule: they take the generic path.  16 is
// the fp16-weight format: the "codes" are the weights themselves.
template <int BITS> constexpr bool kHasFast = BITS != 5;
// widths whose fast path has kernels with three or four x chunks per lane
template <int BITS> constexpr bool kWideBits = BITS == 2 || BITS == 4 || BITS == 8;

// For each fp16x2 code pair of a word: the positions (within the word) of its
// low-half and high-half codes, and its class.
template <int BITS> struct FastLayout;

// Q4: per word, pairs (q0,q4) c=1, (q1,q5) c=16, (q2,q6) c=1, (q3,q7) c=16.
template <> struct FastLayout<4> {
  static constexpr int pairs_per_word = 4;
  __device__ static constexpr int pos(int pair, int half) { return pair + 4 * half; }
  __device__ static constexpr int cls(int pair) { return (pair & 1) ? 1 : 0; }
  __device__ static constexpr float mult(int c) { return c ? 16.f : 1.f; }
};
// Q2: per word, pairs (q_j, q_{j+8}) for j = 0..7; pairs 0..4 come from w with
// classes 1,4,16,64,256 and pairs 5..7 from w >> 10 with classes 1,4,16.
template <> struct FastLayout<2> {
  static constexpr int pairs_per_word = 8;
  __device__ static constexpr int pos(int pair, int half) { return pair + 8 * half; }
  __device__ static constexpr int cls(int pair) { return pair < 5 ? pair : pair - 5; }
  __device__ static constexpr float mult(int c) {
    return c == 0 ? 1.f : c == 1 ? 4.f : c == 2 ? 16.f : c == 3 ? 64.f : 256.f;
  }
};
// Q8: per word, pairs (q0,q1) and (q2,q3), class 1.
template <> struct FastLayout<8> {
  static constexpr int pairs_per_word = 2;
  __device__ static constexpr int pos(int pair, int half) { return 2 * pair + half; }
  __device__ static constexpr int cls(int) { return 0; }
  __device__ static constexpr float mult(int) { return 1.f; }
};

// One word's code pairs as fp16x2 "1024 + c*q" values.
template <int BITS>
__device__ __forceinline__ void fast_pairs(uint32_t w, uint32_t (&h)[FastLayout<BITS>::pairs_per_word]) {
  if constexpr (BITS == 4) {
    const uint32_t w8 = w >> 8;
    h[0] = lop_mask_or(w, 0x000F000Fu);
    h[1] = lop_mask_or(w, 0x00F000F0u);
    h[2] = lop_mask_or(w8, 0x000F000Fu);
    h[3] = lop_mask_or(w8, 0x00F000F0u);
  } else if constexpr (BITS == 2) {
    const uint32_t w10 = w >> 10;
    h[0] = lop_mask_or(w, 0x00030003u);
    h[1] = lop_mask_or(w, 0x000C000Cu);
    h[2] = lop_mask_or(w, 0x00300030u);
    h[3] = lop_mask_or(w, 0x00C000C0u);
    h[4] = lop_mask_or(w, 0x03000300u);
    h[5] = lop_mask_or(w10, 0x00030003u);
    h[6] = lop_mask_or(w10, 0x000C000Cu);
    h[7] = lop_mask_or(w10, 0x00300030u);
  } else {
    h[0] = prmt(w, 0x64646464u, 0x4140u);
    h[1] = prmt(w, 0x64646464u, 0x4342u);
  }
}

// ------------------------------------------------------------ x slices
// Per chunk a lane keeps: the x values (layout depends on the path), sum(x)
// over the chunk (for the bias term) and, on the fast path, the offset sum
// per class c the starting value -sum_{j in c} 1024 * x_j of that class's
// accumulator, which removes the fp16 magic as the codes are accumulated.
template <int BITS, bool FAST> struct XSlice;

template <int BITS> struct XSlice<BITS, true> {
  uint16_t xh[32];   // fp16 x values of the chunk, one per register
  float xsum;
  float zc[FastClasses<BITS>::n];
};
template <int BITS> struct XSlice<BITS, false> {
  float xv[32];
  float xsum;
};

// ---- bits 3 and 6: the searched code-pair schedules of qgemv_stream.h.
// One schedule entry: its source window of the chunk's stream, one LOP3 and
// the FMAs of its one or two codes into their classes.
template <int BITS, int I>
__device__ __forceinline__ void stream_step(const uint32_t (&w)[BITS], const uint16_t (&xh)[32],
                                            float (&acc)[StreamLayout<BITS>::n_classes]) {
  using L = StreamLayout<BITS>;
  constexpr StreamPair P = L::pair(I);
  constexpr int wi = P.t / 32, sh = P.t % 32;
  uint32_t src;
  if constexpr (sh == 0) src = w[wi];
  else if constexpr (wi + 1 < BITS) src = __funnelshift_r(w[wi], w[wi + 1], sh);
  else src = w[wi] >> sh;
  const uint32_t h = lop3_and_or(src, stream_mask<BITS>(P), 0x64006400u);
  if constexpr (P.lo >= 0 && P.hi >= 0) {
    if constexpr (L::cls(P.olo) == L::cls(P.ohi)) fma_pair(acc[L::cls(P.olo)], xh[P.lo], xh[P.hi], h);
    else fma_pair2(acc[L::cls(P.olo)], acc[L::cls(P.ohi)], xh[P.lo], xh[P.hi], h);
  } else if constexpr (P.lo >= 0) {
    fma_half<false>(acc[L::cls(P.olo)], xh[P.lo], h);
  } else {
    fma_half<true>(acc[L::cls(P.ohi)], xh[P.hi], h);
  }
}

template <int BITS, int... I>
__device__ __forceinline__ void stream_steps(const uint32_t (&w)[BITS], const uint16_t (&xh)[32],
                                             float (&acc)[StreamLayout<BITS>::n_classes],
                                             std::integer_sequence<int, I...>) {
  (stream_step<BITS, I>(w, xh, acc), ...);
}

// x sum of the chunk and each class's seed: minus 1024 times the x of its codes.
template <int BITS, int I>
__device__ __forceinline__ void stream_seed(const uint16_t (&xh)[32], float (&zc)[StreamLayout<BITS>::n_classes]) {
  using L = StreamLayout<BITS>;
  constexpr StreamPair P = L::pair(I);
  if constexpr (P.lo >= 0) zc[L::cls(P.olo)] -= 1024.f * __half2float(__ushort_as_half(xh[P.lo]));
  if constexpr (P.hi >= 0) zc[L::cls(P.ohi)] -= 1024.f * __half2float(__ushort_as_half(xh[P.hi]));
}

template <int BITS, int... I>
__device__ __forceinline__ void stream_seeds(XSlice<BITS, true>& s, std::integer_sequence<int, I...>) {
  float zc[StreamLayout<BITS>::n_classes];
#pragma unroll
  for (int c = 0; c < StreamLayout<BITS>::n_classes; ++c) zc[c] = 0.f;
  (stream_seed<BITS, I>(s.xh, zc), ...);
  float xsum = 0.f;
#pragma unroll
  for (int j = 0; j < 32; ++j) xsum += __half2float(__ushort_as_half(s.xh[j]));
  s.xsum = xsum;
#pragma unroll
  for (int c = 0; c < StreamLayout<BITS>::n_classes; ++c) s.zc[c] = zc[c];
}

template <int BITS>
__device__ __forceinline__ float chunk_dot_stream(const uint32_t (&w)[BITS], const XSlice<BITS, true>& s) {
  using L = StreamLayout<BITS>;
  float acc[L::n_classes];
#pragma unroll
  for (int c = 0; c < L::n_classes; ++c) acc[c] = s.zc[c];
  stream_steps<BITS>(w, s.xh, acc, std::make_integer_sequence<int, L::n_pairs>{});
  float t = acc[0];
#pragma unroll
  for (int c = 1; c < L::n_classes; ++c) t = fmaf(acc[c], 1.f / float(1 << L::offset(c)), t);
  return t;
}

template <int BITS, bt_dtype XD>
__device__ __forceinline__ void load_x_fast(XSlice<BITS, true>& s, const uint16_t* xk, float xscale = 1.f) {
  // xk: 32 consecutive x values (16-B aligned) of this chunk
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint4 q = __ldg(reinterpret_cast<const uint4*>(xk) + i);
    const uint32_t u[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      s.xh[8 * i + 2 * j] = u[j] & 0xFFFF;
      s.xh[8 * i + 2 * j + 1] = u[j] >> 16;
    }
  }
  if (xscale != 1.f) {   // a gate-weighted x segment: xscale * x, rounded to fp16 once
#pragma unroll
    for (int j = 0; j < 32; ++j)
      s.xh[j] = __half_as_ushort(__float2half_rn(xscale * __half2float(__ushort_as_half(s.xh[j]))));
  }
  if constexpr (BITS == 16) {
    s.xsum = 0.f;   // fp16 weights: no bias term
  } else if constexpr (kStreamBits<BITS>) {
    stream_seeds<BITS>(s, std::make_integer_sequence<int, StreamLayout<BITS>::n_pairs>{});
  } else {
  using L = FastLayout<BITS>;
  constexpr int codes_per_word = 32 / BITS;
  constexpr int NC = FastClasses<BITS>::n;
  float xsum = 0.f;
  float zc[NC];
#pragma unroll
  for (int c = 0; c < NC; ++c) zc[c] = 0.f;
#pragma unroll
  for (int wd = 0; wd < BITS; ++wd) {
#pragma unroll
    for (int p = 0; p < L::pairs_per_word; ++p) {
      const float x0 = __half2float(__ushort_as_half(s.xh[wd * codes_per_word + L::pos(p, 0)]));
      const float x1 = __half2float(__ushort_as_half(s.xh[wd * codes_per_word + L::pos(p, 1)]));
      xsum += x0 + x1;
      zc[L::cls(p)] -= (x0 + x1) * 1024.f;
    }
  }
  s.xsum = xsum;
#pragma unroll
  for (int c = 0; c < NC; ++c) s.zc[c] = zc[c];
  }
}

template <int BITS, bt_dtype XD>
__device__ __forceinline__ void load_x_generic(XSlice<BITS, false>& s, const uint16_t* xk, float xscale = 1.f) {
  float xsum = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint4 q = __ldg(reinterpret_cast<const uint4*>(xk) + i);
    const uint32_t u[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      s.xv[8 * i + 2 * j] = xscale * to_f32<XD>(u[j] & 0xFFFF);
      s.xv[8 * i + 2 * j + 1] = xscale * to_f32<XD>(u[j] >> 16);
    }
  }
#pragma unroll
  for (int j = 0; j < 32; ++j) xsum += s.xv[j];
  s.xsum = xsum;
}

// sum_j q_j * x_j over one chunk (fast path, bits 2/4/8: pairs within a word).
template <int BITS>
__device__ __forceinline__ float chunk_dot_words(const uint32_t (&w)[BITS], const XSlice<BITS, true>& s) {
  using L = FastLayout<BITS>;
  constexpr int NC = FastClasses<BITS>::n;
  constexpr int codes_per_word = 32 / BITS;
  float acc[NC];
#pragma unroll
  for (int c = 0; c < NC; ++c) acc[c] = s.zc[c];
#pragma unroll
  for (int wd = 0; wd < BITS; ++wd) {
    uint32_t h[L::pairs_per_word];
    fast_pairs<BITS>(w[wd], h);
#pragma unroll
    for (int p = 0; p < L::pairs_per_word; ++p)
      fma_pair(acc[L::cls(p)], s.xh[wd * codes_per_word + L::pos(p, 0)], s.xh[wd * codes_per_word + L::pos(p, 1)],
               h[p]);
  }
  float t = acc[0];
#pragma unroll
  for (int c = 1; c < NC; ++c) t = fmaf(acc[c], 1.f / L::mult(c), t);
  return t;
}

// fp16 weights: sum_j w_j * x_j with the mixed fp16 x fp16 -> fp32 FMA, two chains.
__device__ __forceinline__ float chunk_dot_f16w(const uint32_t (&w)[16], const XSlice<16, true>& s) {
  float a0 = 0.f, a1 = 0.f;
#pragma unroll
  for (int i = 0; i < 16; i += 2) {
    fma_pair(a0, s.xh[2 * i], s.xh[2 * i + 1], w[i]);
    fma_pair(a1, s.xh[2 * i + 2], s.xh[2 * i + 3], w[i + 1]);
  }
  return a0 + a1;
}

// sum_j q_j * x_j over one chunk (fast path).
template <int BITS>
__device__ __forceinline__ float chunk_dot_fast(const uint32_t (&w)[BITS], const XSlice<BITS, true>& s) {
  if constexpr (BITS == 16) return chunk_dot_f16w(w, s);
  else if constexpr (kStreamBits<BITS>) return chunk_dot_stream<BITS>(w, s);
  else return chunk_dot_words<BITS>(w, s);
}

// sum_j q_j * x_j over one chunk (generic path, any bits).
template <int BITS>
__device__ __forceinline__ float chunk_dot_generic(const uint32_t (&w)[BITS], const XSlice<BITS, false>& s) {
  if constexpr (BITS == 16) {   // fp16 weights
    float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      acc0 = fmaf(s.xv[2 * i], __half2float(__ushort_as_half((uint16_t)(w[i] & 0xFFFFu))), acc0);
      acc1 = fmaf(s.xv[2 * i + 1], __half2float(__ushort_as_half((uint16_t)(w[i] >> 16))), acc1);
    }
    return acc0 + acc1;
  }
  constexpr uint32_t mask = (1u << (BITS & 15)) - 1u;
  float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const int bit = j * BITS, wi = bit >> 5, off = bit & 31;
    const uint32_t sh = off + BITS <= 32 ? (w[wi] >> off) : __funnelshift_r(w[wi], w[wi + 1], off);
    const float qf = __uint_as_float(lop3_and_or(sh, mask, 0x4B000000u)) - 8388608.f;
    if (j & 1) acc1 = fmaf(s.xv[j], qf, acc1);
    else acc0 = fmaf(s.xv[j], qf, acc0);
  }
  return acc0 + acc1;
}

// ------------------------------------------------------- problem -> expert / rows
// Grouped row `prob` belongs to the expert e with off[e] <= prob < off[e+1]
// (offsets cached in shared memory); -1 when no expert holds it.
__device__ __forceinline__ int problem_expert(const GemvParams& p, const int* offs, int prob) {
  if (p.pair_ids) {   // routed pair: its expert id, or -1 (and a device error) when out of range
    const int e = __ldg(p.pair_ids + prob);
    if (e >= 0 && e < p.num_experts) return e;
    set_device_error(p.err, kErrBadArg);
    return -1;
  }
  if (!p.moe_offsets) return 0;
  int lo = 0, hi = p.num_experts;   // invariant: offs[lo] <= prob, answer in [lo, hi)
  if (prob < offs[0] || prob >= offs[p.num_experts]) return -1;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (offs[mid] <= prob) lo = mid; else hi = mid;
  }
  return lo;
}
__device__ __forceinline__ int problem_xrow(const GemvParams& p, int prob) {
  if (p.pair_ids) return prob / p.top_k;
  if (!p.moe_offsets) return 0;
  return p.row_index ? __ldg(p.row_index + prob) : prob;
}
__device__ __forceinline__ int problem_yrow(const GemvParams& p, int prob) {
  return (p.moe_offsets || p.pair_ids) ? prob : 0;
}


// --------------------------------------------------------------- the kernel
// Consumer warps per CTA: 8, plus one producer warp.  One x chunk per lane
// (CPL = 1) fits two CTAs per SM (16 consumer warps, up to 112 registers) with
// four or eight rows in flight per warp, or three CTAs (24 consumer warps, up
// to 75 registers) with two; more chunks per lane keep x in more registers and
// run one CTA per SM.
template <int CPL, int RI> struct Warps {
  static constexpr int kNW = 8;
  static constexpr int kThreads = (kNW + 1) * 32;
  static constexpr int kMinBlocks = CPL == 1 ? (RI <= 2 ? 3 : 2) : 1;
};

// Sum RI per-row partials over the 32 lanes with a transpose-style tree.  On
// return, `row` is the row in [0, RI) whose full sum this lane holds; lanes
// with (lane & (32/RI - 1)) == 0 are the first holder of each row.
template <int RI>
__device__ __forceinline__ float reduce_rows(const float (&part)[RI], int lane, int& row) {
  if constexpr (RI == 8) {
    // 9 shuffles for 8 rows: halve the row set at lane bits 16, 8 and 4, then sum
    const bool b16 = lane & 16, b8 = lane & 8, b4 = lane & 4;
    float a[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float keep = b16 ? part[4 + i] : part[i], give = b16 ? part[i] : part[4 + i];
      a[i] = keep + __shfl_xor_sync(0xffffffffu, give, 16);
    }
    float c[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const float keep = b8 ? a[2 + i] : a[i], give = b8 ? a[i] : a[2 + i];
      c[i] = keep + __shfl_xor_sync(0xffffffffu, give, 8);
    }
    float e = b4 ? c[1] : c[0];
    const float f = b4 ? c[0] : c[1];
    e += __shfl_xor_sync(0xffffffffu, f, 4);
    e += __shfl_xor_sync(0xffffffffu, e, 2);
    e += __shfl_xor_sync(0xffffffffu, e, 1);
    row = ((lane >> 4) & 1) * 4 + ((lane >> 3) & 1) * 2 + ((lane >> 2) & 1);
    return e;
  } else if constexpr (RI == 4) {
    const bool hi = lane & 16;
    float a0 = hi ? part[2] : part[0], a1 = hi ? part[3] : part[1];
    const float b0 = hi ? part[0] : part[2], b1 = hi ? part[1] : part[3];
    a0 += __shfl_xor_sync(0xffffffffu, b0, 16);
    a1 += __shfl_xor_sync(0xffffffffu, b1, 16);
    const bool m = lane & 8;
    float c = m ? a1 : a0;
    const float d = m ? a0 : a1;
    c += __shfl_xor_sync(0xffffffffu, d, 8);
    c += __shfl_xor_sync(0xffffffffu, c, 4);
    c += __shfl_xor_sync(0xffffffffu, c, 2);
    c += __shfl_xor_sync(0xffffffffu, c, 1);
    row = ((lane >> 4) & 1) * 2 + ((lane >> 3) & 1);
    return c;
  } else if constexpr (RI == 2) {
    const bool hi = lane & 16;
    float a = hi ? part[1] : part[0];
    const float b = hi ? part[0] : part[1];
    a += __shfl_xor_sync(0xffffffffu, b, 16);
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
    row = (lane >> 4) & 1;
    return a;
  } else {
    float a = part[0];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
    row = 0;
    return a;
  }
}

__device__ __forceinline__ void store_yv(const GemvParams& p, void* y, size_t i, float v) {
  if (p.y_dtype == BT_F32) store_out<BT_F32>(y, i, v);
  else if (p.y_dtype == BT_BF16) store_out<BT_BF16>(y, i, v);
  else store_out<BT_F16>(y, i, v);
}

// One GEMV problem as the kernel sees it: weight rows, x row, y row.
struct ProbView {
  const uint8_t* codes;      // row 0 of this problem's packed weight
  const uint16_t* scales;
  const uint16_t* biases;
  const uint16_t* x;         // this problem's x (K halves)
  void* y;                   // output base
  size_t y0;                 // element index of this problem's row 0 in y
  int n;                     // rows of the problem
  int units;                 // row blocks of the problem
  int k, g, row_bytes;       // row geometry: codes per row, groups per row, packed bytes per row
  int kw;                    // warps that share one row (K split)
  int rb;                    // rows per pipeline unit
  bool valid;                // false: a grouped row that no expert holds (skipped)
  int nseg, seg_rb, seg_g;   // K segments (1 unless segmented), bytes and groups of one segment's row
};

template <bool BATCH, bool SEG = false>
__device__ __forceinline__ ProbView resolve(const GemvParams& p, const GemvBatch<BATCH ? kBatchCap : 1>& batch,
                                            const int* offs, int prob) {
  ProbView v;
  if constexpr (BATCH) {
    const GemvProblem& q = batch.prob[prob];
    v.codes = reinterpret_cast<const uint8_t*>(q.codes);
    v.scales = q.scales;
    v.biases = q.biases;
    v.x = static_cast<const uint16_t*>(q.x);
    v.y = q.y;
    v.y0 = 0;
    v.n = q.n;
    v.units = q.units;
    v.k = q.k;
    v.g = q.g;
    v.row_bytes = q.row_bytes;
    v.kw = q.kw;
    v.rb = q.rb;
    v.valid = true;
    v.nseg = 1;
    v.seg_rb = q.row_bytes;
    v.seg_g = q.g;
  } else if constexpr (SEG) {
    // segmented token problem: the weights' bases are expert 0's (the producer adds
    // each segment's expert plane); x is the token's nseg rows back to back
    v.codes = reinterpret_cast<const uint8_t*>(p.codes);
    v.scales = p.scales;
    v.biases = p.biases;
    v.x = static_cast<const uint16_t*>(p.x) + (size_t)prob * p.K;
    v.y = p.y;
    v.y0 = (size_t)prob * p.N;
    v.n = p.N;
    v.units = p.units_per_problem;
    v.k = p.K;
    v.g = p.G;
    v.row_bytes = p.row_bytes;
    v.kw = p.kw;
    v.rb = p.rows_per_unit;
    v.nseg = p.nseg;
    v.seg_rb = p.row_bytes / p.nseg;
    v.seg_g = p.G / p.nseg;
    bool ok = true;   // every segment's expert id in range (each thread checks all of them)
    for (int s = 0; s < p.nseg; ++s) {
      const int e = __ldg(p.seg_ids + (size_t)prob * p.nseg + s);
      ok = ok && e >= 0 && e < p.num_experts;
    }
    if (!ok) set_device_error(p.err, kErrBadArg);
    v.valid = ok;
  } else {
    const int e = problem_expert(p, offs, prob);
    const size_t e_rows = (size_t)(e < 0 ? 0 : e) * p.N;
    v.codes = reinterpret_cast<const uint8_t*>(p.codes) + e_rows * p.row_bytes;
    v.scales = p.scales + e_rows * p.G;
    v.biases = p.biases + e_rows * p.G;
    v.x = static_cast<const uint16_t*>(p.x) + (size_t)problem_xrow(p, prob) * p.K;
    v.y = p.y;
    v.y0 = (size_t)problem_yrow(p, prob) * (p.swiglu ? p.N / 2 : p.N);
    v.n = p.N;
    v.units = p.units_per_problem;
    v.k = p.K;
    v.g = p.G;
    v.row_bytes = p.row_bytes;
    v.kw = p.kw;
    v.rb = p.rows_per_unit;
    v.valid = e >= 0;
    v.nseg = 1;
    v.seg_rb = p.row_bytes;
    v.seg_g = p.G;
  }
  return v;
}

// Rows of a unit are staged by bulk copies only when every copy starts on a
// 16-byte boundary and moves a multiple of 16 bytes; otherwise the consumers
// read that unit straight from global memory.
__device__ __forceinline__ bool unit_bulk(const GemvParams& p, const ProbView& v, int row0, int rows) {
  const uintptr_t c0 = reinterpret_cast<uintptr_t>(v.codes) + (size_t)row0 * v.row_bytes;
  const uintptr_t s0 = reinterpret_cast<uintptr_t>(v.scales + (size_t)row0 * v.g);
  const uintptr_t b0 = reinterpret_cast<uintptr_t>(v.biases + (size_t)row0 * v.g);
  const size_t cb = (size_t)rows * v.row_bytes, sb = (size_t)rows * v.g * 2;
  return ((c0 | s0 | b0 | cb | sb) & 15u) == 0;
}

// First problem whose unit range contains unit u (batched launches).
template <bool BATCH>
__device__ __forceinline__ void first_unit(const GemvParams& p, const GemvBatch<BATCH ? kBatchCap : 1>& batch,
                                           long long u, int& prob, int& blk) {
  if constexpr (BATCH) {
    int lo = 0, hi = batch.count;   // unit_begin[lo] <= u
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (batch.prob[mid].unit_begin <= u) lo = mid; else hi = mid;
    }
    prob = lo;
    blk = (int)(u - batch.prob[lo].unit_begin);
  } else {
    prob = (int)(u / p.units_per_problem);
    blk = (int)(u - (long long)prob * p.units_per_problem);
  }
}

// Batched launches: the first unit whose work starts at or after `c`, so that
// CTA i takes the units starting in its equal share of the launch's work.
__device__ __forceinline__ long long unit_at_cost(const GemvParams& p, const GemvBatch<kBatchCap>& batch,
                                                  long long c) {
  if (c >= p.total_cost) return p.num_units;
  int lo = 0, hi = batch.count;   // last problem with cost_begin <= c
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (batch.prob[mid].cost_begin <= c) lo = mid; else hi = mid;
  }
  const GemvProblem& q = batch.prob[lo];
  const long long uc = (long long)q.rb * q.cw;
  const long long blk = (c - q.cost_begin + uc - 1) / uc;
  if (blk < q.units) return q.unit_begin + blk;
  return lo + 1 < batch.count ? batch.prob[lo + 1].unit_begin : p.num_units;
}

template <int BITS, bt_dtype XD, int CPL, bool FAST, int RI, bool BATCH, bool SEG>
__global__ void __launch_bounds__(Warps<CPL, RI>::kThreads, Warps<CPL, RI>::kMinBlocks)
    qgemv_kernel(const GemvParams p, const __grid_constant__ GemvBatch<BATCH ? kBatchCap : 1> batch) {
  constexpr int kNW = Warps<CPL, RI>::kNW;
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = p.stages;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)S * p.stage_bytes);
  uint64_t* empty = full + S;
  float* red = reinterpret_cast<float*>(empty + S);        // [kNW/KW][2][RI][KW] = kNW*2*RI floats
  int* offs = reinterpret_cast<int*>(red + kNW * 2 * RI);  // [E+1] when grouped
  // Set once any wait of this CTA has expired: from then on every warp skips
  // its waits, loads and stores but still walks the loop and reaches every
  // named barrier its row group and the CTA execute, so no partner is left
  // waiting at a barrier that cannot time out.
  __shared__ volatile int s_fail;

  // contiguous range of units for this CTA
  long long u_begin, u_end;
  if constexpr (BATCH) {
    u_begin = unit_at_cost(p, batch, p.total_cost * blockIdx.x / gridDim.x);
    u_end = unit_at_cost(p, batch, p.total_cost * (blockIdx.x + 1) / gridDim.x);
  } else {
    u_begin = p.num_units * blockIdx.x / gridDim.x;
    u_end = p.num_units * (blockIdx.x + 1) / gridDim.x;
  }

  // full[s]: one arrive.expect_tx for the bulk copy of the codes plus one
  // cp.async-tracked arrive from each producer lane (scales and biases).
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) { mbar_init(&full[s], 33); mbar_init(&empty[s], kNW); }
    s_fail = 0;
    fence_mbar_init();
  }
  if (p.moe_offsets) {
    pdl_wait();   // offsets come from the routing kernel
    for (int i = threadIdx.x; i <= p.num_experts; i += blockDim.x) offs[i] = __ldg(p.moe_offsets + i);
  }
  __syncthreads();
  pdl_launch_dependents();

  if (u_begin >= u_end) return;

  if (warp == kNW) {
    // ------------------------------------------------------------ producer
    // Lane 0 moves a unit's packed codes with one bulk copy (large copies keep
    // the copy engine streaming); all 32 lanes move its fp16 scales and biases
    // with 16-byte cp.async, whose completion the same mbarrier tracks.
    if (!p.const_weights || p.pair_ids) pdl_wait();   // routed pairs: expert ids may come from the previous kernel
    const uint64_t pol = l2_policy_evict_first();
    int prob, blk;
    first_unit<BATCH>(p, batch, u_begin, prob, blk);
    ProbView v = resolve<BATCH, SEG>(p, batch, offs, prob);
    int s = 0;
    uint32_t ph = 0;
    long long it = 0;
    bool ok = true;
    for (long long u = u_begin; u < u_end; ++u, ++it) {
      if (blk == v.units) { blk = 0; ++prob; v = resolve<BATCH, SEG>(p, batch, offs, prob); }
      if (it >= S) {
        bool w = true;
        if (lane == 0) w = mbar_wait(&empty[s], ph ^ 1u, p.timeout_ns, p.err);
        if (!__shfl_sync(0xffffffffu, (int)w, 0)) { ok = false; s_fail = 1; break; }
      }
      const int RB = v.rb, row_bytes = v.row_bytes, G = v.g;
      const int row0 = blk * RB;
      const int rows = min(RB, v.n - row0);
      const bool drop = p.drop_stage && blockIdx.x == 0 && it == 0;   // test hook: never fill this stage
      if constexpr (SEG) if (!drop) {
        // K segments: one bulk copy of each segment's rows (from its expert's plane)
        // and its parameters; the host plans every copy 16-byte aligned
        if (v.valid) {
          const uint32_t segc = (uint32_t)rows * v.seg_rb, segs = (uint32_t)rows * v.seg_g * 2;
          uint8_t* st = smem + (size_t)s * p.stage_bytes;
          uint8_t* ss = st + (size_t)RB * row_bytes;
          uint8_t* sbb = ss + (size_t)RB * G * 2;
          if (lane == 0) mbar_arrive_expect_tx(&full[s], segc * v.nseg);
          for (int sg = 0; sg < v.nseg; ++sg) {
            const size_t er = (size_t)__ldg(p.seg_ids + (size_t)prob * v.nseg + sg) * v.n + row0;
            if (lane == 0)
              bulk_g2s(st + (size_t)sg * RB * v.seg_rb, v.codes + er * v.seg_rb, segc, &full[s], pol);
            const uint8_t* gs = reinterpret_cast<const uint8_t*>(v.scales + er * v.seg_g);
            const uint8_t* gb = reinterpret_cast<const uint8_t*>(v.biases + er * v.seg_g);
            uint8_t* ds = ss + (size_t)sg * RB * v.seg_g * 2;
            uint8_t* db = sbb + (size_t)sg * RB * v.seg_g * 2;
            for (uint32_t o = lane * 16u; o < segs; o += 32u * 16u) {
              cp_async16(ds + o, gs + o);
              cp_async16(db + o, gb + o);
            }
          }
          cp_async_mbar_arrive_noinc(&full[s]);
        } else {
          mbar_arrive(&full[s]);
          if (lane == 0) mbar_arrive(&full[s]);
        }
      }
      if constexpr (!SEG) if (!drop) {
        if (v.valid && unit_bulk(p, v, row0, rows)) {
          const uint32_t cbytes = (uint32_t)rows * row_bytes, sbytes = (uint32_t)rows * G * 2;
          uint8_t* st = smem + (size_t)s * p.stage_bytes;
          if (lane == 0) {
            mbar_arrive_expect_tx(&full[s], cbytes);
            bulk_g2s(st, v.codes + (size_t)row0 * row_bytes, cbytes, &full[s], pol);
          }
          const uint8_t* gs = reinterpret_cast<const uint8_t*>(v.scales + (size_t)row0 * G);
          const uint8_t* gb = reinterpret_cast<const uint8_t*>(v.biases + (size_t)row0 * G);
          uint8_t* ss = st + (size_t)RB * row_bytes;
          uint8_t* sbb = ss + (size_t)RB * G * 2;
          for (uint32_t o = lane * 16u; o < sbytes; o += 32u * 16u) {
            cp_async16(ss + o, gs + o);
            cp_async16(sbb + o, gb + o);
          }
          cp_async_mbar_arrive_noinc(&full[s]);
        } else {
          mbar_arrive(&full[s]);
          if (lane == 0) mbar_arrive(&full[s]);
        }
      }
      ++blk;
      if (++s == S) { s = 0; ph ^= 1u; }
    }
    if (!ok) {
      // drain copies still in flight before this CTA's shared memory goes away
      cp_async_wait_all();
      if (lane == 0) {
        const long long issued = it;
        for (long long j = (issued > S ? issued - S : 0); j < issued; ++j)   // failure path only
          mbar_wait(&full[j % S], (uint32_t)((j / S) & 1), p.timeout_ns, p.err);
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  // KW warps share a row (K split), RW row groups per CTA; both follow the
  // problem, so they are set when a unit of a new problem starts.
  int KW = 0, RW = 0, kw = 0, rg = 0, nchunks = 0;
  const bool writer = (lane & (32 / RI - 1)) == 0;
  pdl_wait();   // activations (and offsets) may come from the previous kernel

  XSlice<BITS, FAST> xs[CPL];
  // per x chunk of this lane: byte offset of its codes in a staged row of the
  // unit and index of its parameters (one segment: c * chunk bytes and the
  // chunk's group; K segments: inside its segment's block of the stage)
  int coff[CPL], poff[CPL];
  bool dead = false;   // this warp gave up on a wait, or saw another warp of the CTA give up
  int rbuf = 0;
  int prob, blk;
  first_unit<BATCH>(p, batch, u_begin, prob, blk);
  ProbView v;
  int cur_prob = -1;
  int s = 0;
  uint32_t ph = 0;
  for (long long u = u_begin; u < u_end; ++u) {
    if (cur_prob >= 0 && blk == v.units) { blk = 0; ++prob; }
    if (prob != cur_prob) {
      cur_prob = prob;
      v = resolve<BATCH, SEG>(p, batch, offs, prob);
      if (v.kw != KW) {
        if (v.kw < 1 || kNW % v.kw) {   // never planned so; refuse rather than spin
          if (threadIdx.x == 0) set_device_error(p.err, kErrBadArg);
          return;
        }
        // The row groups change: every consumer warp leaves the previous
        // problem's row-group barriers before any warp uses the new ones.
        if (KW != 0) asm volatile("bar.sync 15, %0;" ::"r"(kNW * 32) : "memory");
        KW = v.kw;
        RW = kNW / KW;
        kw = warp % KW;
        rg = warp / KW;
        rbuf = 0;
      }
      nchunks = v.k / 32;
      const int cps = SEG ? nchunks / v.nseg : nchunks;   // 32-code chunks per segment
#pragma unroll
      for (int i = 0; i < CPL; ++i) {
        const int c = (i * KW + kw) * 32 + lane;
        if (c < nchunks) {
          float xscale = 1.f;
          if constexpr (SEG) {
            const int sg = c / cps, cc = c - sg * cps;
            coff[i] = sg * v.rb * v.seg_rb + cc * (4 * BITS);
            poff[i] = sg * v.rb * v.seg_g + (cc >> p.gshift);
            xscale = __ldg(p.seg_gates + (size_t)prob * v.nseg + sg);
          }
          if constexpr (FAST) load_x_fast<BITS, XD>(xs[i], v.x + (size_t)c * 32, xscale);
          else load_x_generic<BITS, XD>(xs[i], v.x + (size_t)c * 32, xscale);
        }
      }
    }
    if (!dead && (s_fail || !mbar_wait(&full[s], ph, p.timeout_ns, p.err))) {
      dead = true;
      s_fail = 1;
    }
    const int RB = v.rb, row_bytes = v.row_bytes, G = v.g;
    const int row0 = blk * RB;
    const int rows = min(RB, v.n - row0);
    const bool tma = v.valid && (SEG || unit_bulk(p, v, row0, rows));
    // row strides of codes (bytes) and parameters (halves) in a staged unit
    const int crs = SEG ? v.seg_rb : row_bytes, prs = SEG ? v.seg_g : G;
    const uint32_t st = smem_u32(smem + (size_t)s * p.stage_bytes);
    const uint32_t st_sc = st + RB * row_bytes, st_bi = st_sc + RB * G * 2;
    const uint8_t* g_codes = v.codes + (size_t)row0 * row_bytes;
    const uint16_t* g_sc = v.scales + (size_t)row0 * G;
    const uint16_t* g_bi = v.biases + (size_t)row0 * G;
    const size_t ybase = v.y0 + (p.swiglu ? row0 / 2 : row0);

    const int nb = (rows + RI - 1) / RI;
    // The row batches of this unit.  Instantiated per (rows need clamping, unit
    // staged in shared memory), chosen once per unit, so the common case -- a
    // full unit in shared memory -- has no per-row bounds or source branches.
    // LIVE = false walks the same batches and barriers without touching memory
    // (a warp after an expired wait).
    auto batches = [&](auto clamp_tag, auto staged_tag, auto live_tag) {
      constexpr bool CLAMP = decltype(clamp_tag)::value;
      constexpr bool STAGED = decltype(staged_tag)::value;
      constexpr bool LIVE = decltype(live_tag)::value;
    for (int bi = rg; bi < nb; bi += RW) {
      const int r0 = bi * RI;
      float part[RI];
#pragma unroll
      for (int j = 0; j < RI; ++j) part[j] = 0.f;
#pragma unroll
      for (int i = 0; i < CPL; ++i) {
        const int c = (i * KW + kw) * 32 + lane;
        if (LIVE && c < nchunks) {
          uint32_t w[RI][BITS];
          float sc[RI], bs[RI];
          const int co = SEG ? coff[i] : c * (4 * BITS);   // this chunk's codes in a staged row
          const int po = SEG ? poff[i] : (c >> p.gshift);   // and its parameters' index
#pragma unroll
          for (int j = 0; j < RI; ++j) {
            const int r = CLAMP ? min(r0 + j, rows - 1) : r0 + j;
            if constexpr (STAGED) {
              load_chunk<BITS, true>(st + co + r * crs, nullptr, w[j]);
              if constexpr (BITS != 16) {
                sc[j] = to_f32<BT_F16>(lds16(st_sc + (po + r * prs) * 2));
                bs[j] = to_f32<BT_F16>(lds16(st_bi + (po + r * prs) * 2));
              }
            } else {   // one segment only (segmented units are always staged)
              load_chunk<BITS, false>(0, g_codes + (size_t)r * crs + co, w[j]);
              if constexpr (BITS != 16) {
                sc[j] = to_f32<BT_F16>(__ldg(g_sc + (size_t)r * prs + po));
                bs[j] = to_f32<BT_F16>(__ldg(g_bi + (size_t)r * prs + po));
              }
            }
          }
#pragma unroll
          for (int j = 0; j < RI; ++j) {
            float t;
            if constexpr (FAST) t = chunk_dot_fast<BITS>(w[j], xs[i]);
            else t = chunk_dot_generic<BITS>(w[j], xs[i]);
            if constexpr (BITS == 16) part[j] += t;   // fp16 weights: no scale or bias
            else part[j] = fmaf(sc[j], t, fmaf(bs[j], xs[i].xsum, part[j]));
          }
        }
      }
      int rj;
      const float val = reduce_rows<RI>(part, lane, rj);
      const int r = r0 + rj;
      // Store a row's result; with the SwiGLU epilogue the gate row (even) takes
      // its up row (odd, the lane 32/RI away) and stores silu(gate) * up.
      auto emit = [&](float y) {
        if (!BATCH && p.swiglu) {
          if constexpr (RI >= 2) {
            const float up = __shfl_xor_sync(0xffffffffu, y, 32 / RI);
            if (LIVE && writer && !(rj & 1) && r < rows && v.valid)
              store_yv(p, v.y, ybase + (r >> 1), y / (1.f + expf(-y)) * up);
          } else if (threadIdx.x == 0) {
            set_device_error(p.err, kErrBadArg);   // never planned: row pairs need two rows in flight
          }
        } else if (LIVE && writer && r < rows && v.valid) {
          store_yv(p, v.y, ybase + r, y);
        }
      };
      if (KW == 1) {
        emit(val);
      } else {
        float* rb = red + (size_t)((rg * 2 + rbuf) * RI) * KW;   // [RI][KW]
        if (writer) rb[rj * KW + kw] = val;
        asm volatile("bar.sync %0, %1;" ::"r"(1 + rg), "r"(KW * 32) : "memory");
        if (kw == 0) {   // warp-uniform: the whole warp sums (the SwiGLU shuffle needs every lane)
          float acc = 0.f;
          for (int j = 0; j < KW; ++j) acc += rb[rj * KW + j];
          emit(acc);
        }
        rbuf ^= 1;
      }
    }
    };
    using yes = std::integral_constant<bool, true>;
    using no = std::integral_constant<bool, false>;
    if (dead || (SEG && !v.valid)) {   // nothing to read: walk the batches and barriers only
      batches(yes{}, no{}, no{});
    } else if (tma) {
      if (rows == nb * RI) batches(no{}, yes{}, yes{});
      else batches(yes{}, yes{}, yes{});
    } else {
      batches(yes{}, no{}, yes{});
    }
    // A warp that gave up does not arrive: the producer's own bounded wait on
    // this stage then expires and it drains its copies.
    __syncwarp();
    if (!dead && lane == 0) mbar_arrive(&empty[s]);
    ++blk;
    if (++s == S) { s = 0; ph ^= 1u; }
  }
}

// ------------------------------------------------------------------ launch
template <int BITS, bt_dtype XD, int CPL, bool FAST, int RI, bool BATCH, bool SEG>
cudaError_t launch_t(const GemvParams& p, const GemvBatch<kBatchCap>* batch, int grid, size_t smem,
                     cudaStream_t stream) {
  auto k = qgemv_kernel<BITS, XD, CPL, FAST, RI, BATCH, SEG>;
  static std::atomic<uint64_t> smem_raised{0};
  cudaError_t e = raise_smem_limit(reinterpret_cast<const void*>(k), smem_raised);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(Warps<CPL, RI>::kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = opts().pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if constexpr (BATCH) {
    return cudaLaunchKernelEx(&cfg, k, p, *batch);
  } else {
    GemvBatch<1> none{};
    return cudaLaunchKernelEx(&cfg, k, p, none);
  }
}

template <int BITS, bt_dtype XD, int CPL, bool FAST, bool BATCH, bool SEG>
cudaError_t launch_ri(const GemvParams& p, const GemvPlan& pl, const GemvBatch<kBatchCap>* b, cudaStream_t st) {
  switch (pl.ri) {
    case 8:
      if constexpr (CPL == 1) return launch_t<BITS, XD, CPL, FAST, 8, BATCH, SEG>(p, b, pl.grid, pl.smem, st);
      [[fallthrough]];
    case 4: return launch_t<BITS, XD, CPL, FAST, 4, BATCH, SEG>(p, b, pl.grid, pl.smem, st);
    case 2: return launch_t<BITS, XD, CPL, FAST, 2, BATCH, SEG>(p, b, pl.grid, pl.smem, st);
    default: return launch_t<BITS, XD, CPL, FAST, 1, BATCH, SEG>(p, b, pl.grid, pl.smem, st);
  }
}

template <int BITS, bt_dtype XD, bool FAST, bool BATCH, bool SEG>
cudaError_t launch_cpl(const GemvParams& p, const GemvPlan& pl, const GemvBatch<kBatchCap>* b, cudaStream_t st) {
  switch (pl.cpl) {
    case 1: return launch_ri<BITS, XD, 1, FAST, BATCH, SEG>(p, pl, b, st);
    case 2: return launch_ri<BITS, XD, 2, FAST, BATCH, SEG>(p, pl, b, st);
    // three or four chunks per lane: fast path of bits 2/4/8 only (K up to 32768)
    case 3: if constexpr (FAST && kWideBits<BITS> && !SEG) return launch_ri<BITS, XD, 3, FAST, BATCH, SEG>(p, pl, b, st); else break;
    case 4: if constexpr (FAST && kWideBits<BITS> && !SEG) return launch_ri<BITS, XD, 4, FAST, BATCH, SEG>(p, pl, b, st); else break;
  }
  return cudaErrorInvalidValue;
}

template <int BITS, bool BATCH, bool SEG>
cudaError_t launch_bits_b(const GemvParams& p, const GemvPlan& pl, bt_dtype xd, const GemvBatch<kBatchCap>* b,
                          cudaStream_t st) {
  if (xd == BT_F16) {
    if constexpr (kHasFast<BITS>)
      if (pl.fast) return launch_cpl<BITS, BT_F16, true, BATCH, SEG>(p, pl, b, st);
    return launch_cpl<BITS, BT_F16, false, BATCH, SEG>(p, pl, b, st);
  }
  return launch_cpl<BITS, BT_BF16, false, BATCH, SEG>(p, pl, b, st);
}

// K-segmented token problems (a fused down product + combine) run their own
// instantiations, so the others carry none of the segment bookkeeping.
template <int BITS>
cudaError_t launch_bits(const GemvParams& p, const GemvPlan& pl, bt_dtype xd, const GemvBatch<kBatchCap>* b,
                        cudaStream_t st) {
  if (b) return launch_bits_b<BITS, true, false>(p, pl, xd, b, st);
  if (p.seg_ids) return launch_bits_b<BITS, false, true>(p, pl, xd, nullptr, st);
  return launch_bits_b<BITS, false, false>(p, pl, xd, nullptr, st);
}

}  // namespace gemv
}  // namespace bt

