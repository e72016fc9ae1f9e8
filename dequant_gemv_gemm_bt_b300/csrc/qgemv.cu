// Dequant-GEMV (M = 1, decode) and its batched form for mixture-of-experts
// decode.  BaseRT pages, thetesserapress.com "BaseRT claims fastest Apple
// Silicon inference", section "What BaseRT does differently": a dedicated GEMV
// for M = 1 whose memory traffic scales with the compression ratio because the
// weights are dequantized inside the compute loop.
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
//  * Fast path (fp16 x, bits 2/4/8): codes become fp16 "1024 + c*q" with one
//    LOP3 / PRMT per two codes and are multiplied into fp32 accumulators with
//    mixed-precision FMA; the 1024 offset is removed with a precomputed sum.
//    Generic path (bits 3/6, or bf16 x): funnel-shift extraction, exact
//    int->float via the 2^23 magic, fp32 FMA.
//  * Lanes split K; the per-row partials are reduced with warp shuffles and,
//    when several warps split one row, through shared memory.  No atomics:
//    results are bitwise deterministic.
#include "bt_common.cuh"
#include "qgemv.cuh"

namespace bt {

namespace {

constexpr int kConsumerWarps = 8;
constexpr int kThreads = (kConsumerWarps + 1) * 32;

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
    } else {
#pragma unroll
      for (int i = 0; i < BITS; ++i) w[i] = __ldg(reinterpret_cast<const uint32_t*>(gptr) + i);
    }
  }
}

// ------------------------------------------------------------ fast path math
// acc += x.lo * h.lo + x.hi * h.hi, fp16 operands, fp32 accumulation.
__device__ __forceinline__ void fma2_mixed(float& acc, uint32_t xp, uint32_t hp) {
  asm("{\n .reg .f16 xa, xb, ha, hb;\n mov.b32 {xa, xb}, %1;\n mov.b32 {ha, hb}, %2;\n"
      " fma.rn.f32.f16 %0, xa, ha, %0;\n fma.rn.f32.f16 %0, xb, hb, %0;\n}\n"
      : "+f"(acc) : "r"(xp), "r"(hp));
}

__device__ __forceinline__ uint32_t lop_mask_or(uint32_t w, uint32_t mask) {
  return (w & mask) | 0x64006400u;   // one LOP3
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

// Class multiplier of the code at chunk position j (fast path), and the order
// in which x halves are packed so that x pair i lines up with code pair i.
template <int BITS> struct FastLayout;

// Q4: per word, pairs (q0,q4) c=1, (q1,q5) c=16, (q2,q6) c=1, (q3,q7) c=16.
template <> struct FastLayout<4> {
  static constexpr int pairs_per_word = 4;
  __device__ static constexpr int pos(int pair, int half) {  // code index within word
    return (pair == 0 ? 0 : pair == 1 ? 1 : pair == 2 ? 2 : 3) + 4 * half;
  }
  __device__ static constexpr int cls(int pair) { return (pair & 1) ? 1 : 0; }
  __device__ static constexpr float mult(int c) { return c ? 16.f : 1.f; }
};
// Q2: per word, pairs (q_j, q_{j+8}) for j = 0..7; classes 4^(j mod 5 pattern).
template <> struct FastLayout<2> {
  static constexpr int pairs_per_word = 8;
  __device__ static constexpr int pos(int pair, int half) { return pair + 8 * half; }
  // pairs 0..4 come from w with classes 1,4,16,64,256; pairs 5..7 from w>>10 with 1,4,16
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
// Z = sum_j 1024 * x_j / c_j that removes the fp16 magic.
template <int BITS, bool FAST> struct XSlice;

template <int BITS> struct XSlice<BITS, true> {
  uint32_t xp[16];   // fp16 x pairs in fast-layout order
  float xsum, z;
};
template <int BITS> struct XSlice<BITS, false> {
  float xv[32];
  float xsum;
};

template <int BITS, bt_dtype XD>
__device__ __forceinline__ void load_x_fast(XSlice<BITS, true>& s, const uint16_t* xk) {
  // xk: 32 consecutive x values (16-B aligned) of this chunk
  uint16_t v[32];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint4 q = __ldg(reinterpret_cast<const uint4*>(xk) + i);
    const uint32_t u[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) { v[8 * i + 2 * j] = u[j] & 0xFFFF; v[8 * i + 2 * j + 1] = u[j] >> 16; }
  }
  using L = FastLayout<BITS>;
  constexpr int codes_per_word = 32 / BITS;
  float xsum = 0.f, z = 0.f;
#pragma unroll
  for (int wd = 0; wd < BITS; ++wd) {
#pragma unroll
    for (int p = 0; p < L::pairs_per_word; ++p) {
      const int j0 = wd * codes_per_word + L::pos(p, 0);
      const int j1 = wd * codes_per_word + L::pos(p, 1);
      s.xp[wd * L::pairs_per_word + p] = static_cast<uint32_t>(v[j0]) | (static_cast<uint32_t>(v[j1]) << 16);
      const float x0 = __half2float(__ushort_as_half(v[j0])), x1 = __half2float(__ushort_as_half(v[j1]));
      xsum += x0 + x1;
      z += (x0 + x1) * (1024.f / L::mult(L::cls(p)));
    }
  }
  s.xsum = xsum;
  s.z = z;
}

template <int BITS, bt_dtype XD>
__device__ __forceinline__ void load_x_generic(XSlice<BITS, false>& s, const uint16_t* xk) {
  float xsum = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint4 q = __ldg(reinterpret_cast<const uint4*>(xk) + i);
    const uint32_t u[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      s.xv[8 * i + 2 * j] = to_f32<XD>(u[j] & 0xFFFF);
      s.xv[8 * i + 2 * j + 1] = to_f32<XD>(u[j] >> 16);
    }
  }
#pragma unroll
  for (int j = 0; j < 32; ++j) xsum += s.xv[j];
  s.xsum = xsum;
}

// sum_j q_j * x_j over one chunk (fast path).
template <int BITS>
__device__ __forceinline__ float chunk_dot_fast(const uint32_t (&w)[BITS], const XSlice<BITS, true>& s) {
  using L = FastLayout<BITS>;
  constexpr int NC = FastClasses<BITS>::n;
  float acc[NC];
#pragma unroll
  for (int c = 0; c < NC; ++c) acc[c] = 0.f;
#pragma unroll
  for (int wd = 0; wd < BITS; ++wd) {
    uint32_t h[L::pairs_per_word];
    fast_pairs<BITS>(w[wd], h);
#pragma unroll
    for (int p = 0; p < L::pairs_per_word; ++p) fma2_mixed(acc[L::cls(p)], s.xp[wd * L::pairs_per_word + p], h[p]);
  }
  float t = acc[0];
#pragma unroll
  for (int c = 1; c < NC; ++c) t = fmaf(acc[c], 1.f / L::mult(c), t);
  return t - s.z;
}

// sum_j q_j * x_j over one chunk (generic path, any bits).
template <int BITS>
__device__ __forceinline__ float chunk_dot_generic(const uint32_t (&w)[BITS], const XSlice<BITS, false>& s) {
  constexpr uint32_t mask = (1u << BITS) - 1u;
  float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const int bit = j * BITS, wi = bit >> 5, off = bit & 31;
    uint32_t q;
    if (off + BITS <= 32) q = (w[wi] >> off) & mask;
    else q = __funnelshift_r(w[wi], w[wi + 1], off) & mask;
    const float qf = __uint_as_float(0x4B000000u | q) - 8388608.f;
    if (j & 1) acc1 = fmaf(s.xv[j], qf, acc1);
    else acc0 = fmaf(s.xv[j], qf, acc0);
  }
  return acc0 + acc1;
}

// ------------------------------------------------------- problem -> expert / rows
// Grouped row `prob` belongs to the expert e with off[e] <= prob < off[e+1]
// (offsets cached in shared memory); -1 when no expert holds it.
__device__ __forceinline__ int problem_expert(const GemvParams& p, const int* offs, int prob) {
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
  if (!p.moe_offsets) return 0;
  return p.row_index ? __ldg(p.row_index + prob) : prob;
}
__device__ __forceinline__ int problem_yrow(const GemvParams& p, int prob) { return p.moe_offsets ? prob : 0; }

// A unit's rows are staged by bulk copies only when every copy starts on a
// 16-byte boundary and moves a multiple of 16 bytes; otherwise the consumers
// read that unit straight from global memory.
__device__ __forceinline__ bool unit_uses_bulk(const GemvParams& p, size_t wrow, int rows) {
  const size_t c0 = wrow * (size_t)p.row_bytes, s0 = wrow * (size_t)p.G * 2;
  const size_t cb = (size_t)rows * p.row_bytes, sb = (size_t)rows * p.G * 2;
  return ((c0 | s0 | cb | sb) & 15u) == 0;
}

// --------------------------------------------------------------- the kernel
template <int BITS, bt_dtype XD, bt_dtype YD, int CPL, bool FAST>
__global__ void __launch_bounds__(kThreads, 1) qgemv_kernel(const GemvParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = p.stages;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)S * p.stage_bytes);
  uint64_t* empty = full + S;
  float* red = reinterpret_cast<float*>(empty + S);   // [2][RB][KW]
  volatile int* abort_flag = reinterpret_cast<volatile int*>(red + 2 * p.rows_per_unit * p.kw);

  // contiguous range of units for this CTA
  const long long U = p.num_units;
  const long long u_begin = U * blockIdx.x / gridDim.x;
  const long long u_end = U * (blockIdx.x + 1) / gridDim.x;

  int* offs = const_cast<int*>(reinterpret_cast<volatile int*>(abort_flag)) + 4;   // [E+1] when grouped
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], kConsumerWarps); }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (p.moe_offsets) {
    pdl_wait();   // offsets come from the routing kernel
    for (int i = threadIdx.x; i <= p.num_experts; i += blockDim.x) offs[i] = __ldg(p.moe_offsets + i);
  }
  __syncthreads();
  pdl_launch_dependents();

  const int RB = p.rows_per_unit;
  const int row_bytes = p.row_bytes;
  const int G = p.G;

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      if (!p.const_weights || p.moe_offsets) pdl_wait();
      const uint64_t pol = l2_policy_evict_first();
      long long it = 0;
      bool ok = true;
      for (long long u = u_begin; u < u_end && ok; ++u, ++it) {
        const int s = (int)(it % S);
        const uint32_t ph = (uint32_t)((it / S) & 1);
        if (it >= S && !mbar_wait(&empty[s], ph ^ 1u, p.timeout_ns, p.err)) { ok = false; break; }
        const int prob = (int)(u / p.units_per_problem);
        const int blk = (int)(u % p.units_per_problem);
        const int row0 = blk * RB;
        const int rows = min(RB, p.N - row0);
        const int e = problem_expert(p, offs, prob);
        const uint32_t cbytes = (uint32_t)rows * row_bytes, sbytes = (uint32_t)rows * G * 2;
        const size_t wrow = (size_t)(e < 0 ? 0 : e) * p.N + row0;
        const bool tma = unit_uses_bulk(p, wrow, rows);
        if (p.drop_stage && blockIdx.x == 0 && it == 0) continue;   // test hook: never fill this stage
        if (tma && e >= 0) {
          uint8_t* st = smem + (size_t)s * p.stage_bytes;
          mbar_arrive_expect_tx(&full[s], cbytes + 2 * sbytes);
          bulk_g2s(st, reinterpret_cast<const uint8_t*>(p.codes) + wrow * row_bytes, cbytes, &full[s], pol);
          bulk_g2s(st + (size_t)RB * row_bytes, p.scales + wrow * G, sbytes, &full[s], pol);
          bulk_g2s(st + (size_t)RB * row_bytes + (size_t)RB * G * 2, p.biases + wrow * G, sbytes, &full[s], pol);
        } else {
          mbar_arrive(&full[s]);
        }
      }
      if (!ok) {
        // drain copies still in flight before this CTA's shared memory goes away
        *abort_flag = 1;
        const long long issued = it;
        for (long long j = (issued > S ? issued - S : 0); j < issued; ++j)
          mbar_wait(&full[j % S], (uint32_t)((j / S) & 1), p.timeout_ns, p.err);
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int KW = p.kw;
  const int RW = kConsumerWarps / KW;
  const int kw = warp % KW, rg = warp / KW;
  const int nchunks = p.K / 32;
  pdl_wait();   // activations (and offsets) may come from the previous kernel

  XSlice<BITS, FAST> xs[CPL];
  int cur_prob = -1;
  int cur_expert = -1;
  int buf = 0;
  long long it = 0;
  for (long long u = u_begin; u < u_end; ++u, ++it) {
    const int prob = (int)(u / p.units_per_problem);
    const int blk = (int)(u % p.units_per_problem);
    if (prob != cur_prob) {
      cur_prob = prob;
      cur_expert = problem_expert(p, offs, prob);
      const int xrow = problem_xrow(p, prob);
      const uint16_t* xb = static_cast<const uint16_t*>(p.x) + (size_t)xrow * p.K;
#pragma unroll
      for (int i = 0; i < CPL; ++i) {
        const int c = (i * KW + kw) * 32 + lane;
        if (c < nchunks) {
          if constexpr (FAST) load_x_fast<BITS, XD>(xs[i], xb + (size_t)c * 32);
          else load_x_generic<BITS, XD>(xs[i], xb + (size_t)c * 32);
        }
      }
    }
    const int s = (int)(it % S);
    const uint32_t ph = (uint32_t)((it / S) & 1);
    if (!mbar_wait(&full[s], ph, p.timeout_ns, p.err)) return;
    const int row0 = blk * RB;
    const int rows = min(RB, p.N - row0);
    const size_t wrow = (size_t)(cur_expert < 0 ? 0 : cur_expert) * p.N + row0;
    const bool tma = unit_uses_bulk(p, wrow, rows) && cur_expert >= 0;
    const uint32_t st = smem_u32(smem + (size_t)s * p.stage_bytes);
    const uint32_t st_sc = st + RB * row_bytes, st_bi = st_sc + RB * G * 2;
    const uint8_t* g_codes = reinterpret_cast<const uint8_t*>(p.codes) + wrow * row_bytes;
    const uint16_t* g_sc = p.scales + wrow * G;
    const uint16_t* g_bi = p.biases + wrow * G;
    float* redb = red + buf * RB * KW;

    for (int r = rg; r < rows; r += RW) {
      float part = 0.f;
#pragma unroll
      for (int i = 0; i < CPL; ++i) {
        const int c = (i * KW + kw) * 32 + lane;
        if (c < nchunks) {
          uint32_t w[BITS];
          float sc, bi;
          if (tma) {
            load_chunk<BITS, true>(st + r * row_bytes + c * (4 * BITS), nullptr, w);
            sc = to_f32<BT_F16>(lds16(st_sc + (r * G + (c >> 1)) * 2));
            bi = to_f32<BT_F16>(lds16(st_bi + (r * G + (c >> 1)) * 2));
          } else {
            load_chunk<BITS, false>(0, g_codes + (size_t)r * row_bytes + c * (4 * BITS), w);
            sc = to_f32<BT_F16>(__ldg(g_sc + (size_t)r * G + (c >> 1)));
            bi = to_f32<BT_F16>(__ldg(g_bi + (size_t)r * G + (c >> 1)));
          }
          float t;
          if constexpr (FAST) t = chunk_dot_fast<BITS>(w, xs[i]);
          else t = chunk_dot_generic<BITS>(w, xs[i]);
          part = fmaf(sc, t, fmaf(bi, xs[i].xsum, part));
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
      if (lane == 0) redb[r * KW + kw] = part;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
    asm volatile("bar.sync 1, %0;" ::"r"(kConsumerWarps * 32) : "memory");
    if (cur_expert >= 0) {
      for (int t = threadIdx.x; t < rows; t += kConsumerWarps * 32) {
        float acc = 0.f;
        for (int j = 0; j < KW; ++j) acc += redb[t * KW + j];
        store_out<YD>(p.y, (size_t)problem_yrow(p, prob) * p.N + row0 + t, acc);
      }
    }
    buf ^= 1;
  }
}

// ------------------------------------------------------------------ launch
template <int BITS, bt_dtype XD, bt_dtype YD, int CPL, bool FAST>
cudaError_t launch_t(const GemvParams& p, int grid, size_t smem, cudaStream_t stream) {
  auto k = qgemv_kernel<BITS, XD, YD, CPL, FAST>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = opts().pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k, p);
}

template <int BITS, bt_dtype XD, bt_dtype YD, bool FAST>
cudaError_t launch_cpl(const GemvParams& p, int cpl, int grid, size_t smem, cudaStream_t st) {
  switch (cpl) {
    case 1: return launch_t<BITS, XD, YD, 1, FAST>(p, grid, smem, st);
    case 2: return launch_t<BITS, XD, YD, 2, FAST>(p, grid, smem, st);
    case 3: return launch_t<BITS, XD, YD, 3, FAST>(p, grid, smem, st);
    default: return launch_t<BITS, XD, YD, 4, FAST>(p, grid, smem, st);
  }
}

template <int BITS, bt_dtype XD, bt_dtype YD>
cudaError_t launch_bits(const GemvParams& p, int cpl, int grid, size_t smem, cudaStream_t st) {
  constexpr bool kFast = (XD == BT_F16) && (BITS == 2 || BITS == 4 || BITS == 8);
  if (opts().gemv_generic) return launch_cpl<BITS, XD, YD, false>(p, cpl, grid, smem, st);
  return launch_cpl<BITS, XD, YD, kFast>(p, cpl, grid, smem, st);
}

template <bt_dtype XD, bt_dtype YD>
cudaError_t launch_xy(const GemvParams& p, int bits, int cpl, int grid, size_t smem, cudaStream_t st) {
  switch (bits) {
    case 2: return launch_bits<2, XD, YD>(p, cpl, grid, smem, st);
    case 3: return launch_bits<3, XD, YD>(p, cpl, grid, smem, st);
    case 4: return launch_bits<4, XD, YD>(p, cpl, grid, smem, st);
    case 6: return launch_bits<6, XD, YD>(p, cpl, grid, smem, st);
    default: return launch_bits<8, XD, YD>(p, cpl, grid, smem, st);
  }
}

template <bt_dtype XD>
cudaError_t launch_x(const GemvParams& p, int bits, bt_dtype yd, int cpl, int grid, size_t smem, cudaStream_t st) {
  switch (yd) {
    case BT_F32: return launch_xy<XD, BT_F32>(p, bits, cpl, grid, smem, st);
    case BT_BF16: return launch_xy<XD, BT_BF16>(p, bits, cpl, grid, smem, st);
    default: return launch_xy<XD, BT_F16>(p, bits, cpl, grid, smem, st);
  }
}

}  // namespace

GemvPlan plan_gemv(int bits, int N, int K, int problems, int num_experts, int sms) {
  GemvPlan pl{};
  const int nchunks = K / 32;
  int kw = 1;
  while (kw < kConsumerWarps && (nchunks + 32 * kw - 1) / (32 * kw) > 4) kw *= 2;
  pl.kw = kw;
  pl.cpl = (nchunks + 32 * kw - 1) / (32 * kw);
  const int G = K / kGroup;
  const int row_bytes = K * bits / 8;
  const int per_row = row_bytes + 4 * G;
  // smallest row multiple that keeps every bulk copy a multiple of 16 bytes
  int m = 1;
  while (((m * row_bytes) & 15) || ((m * G * 2) & 15)) ++m;
  int rb = std::max(m, (24576 / per_row) / m * m);
  // spread small problems over the machine
  const long long rows_total = (long long)N * problems;
  const int want = (int)std::max<long long>(m, ((rows_total + sms - 1) / sms + m - 1) / m * m);
  rb = std::min(rb, want);
  rb = std::min(rb, std::max(m, 64 / m * m));
  rb = std::min(rb, ((N + m - 1) / m) * m);
  pl.rows_per_unit = rb;
  pl.row_bytes = row_bytes;
  int stage = rb * per_row;
  stage = (stage + 127) / 128 * 128;
  pl.stage_bytes = stage;
  int stages = std::max(2, std::min(8, (96 * 1024) / stage));
  if (opts().gemv_stages > 0) stages = opts().gemv_stages;
  pl.stages = stages;
  pl.units_per_problem = (N + rb - 1) / rb;
  pl.num_units = (long long)pl.units_per_problem * problems;
  pl.grid = (int)std::min<long long>(pl.num_units, (long long)sms);
  pl.smem = (size_t)stages * stage + 2 * stages * sizeof(uint64_t) + 2 * rb * kw * sizeof(float) + 16 +
             (size_t)(num_experts + 1) * sizeof(int);
  return pl;
}

cudaError_t launch_gemv(GemvParams& p, const GemvPlan& pl, int bits, bt_dtype xd, bt_dtype yd, cudaStream_t st) {
  p.rows_per_unit = pl.rows_per_unit;
  p.row_bytes = pl.row_bytes;
  p.stage_bytes = pl.stage_bytes;
  p.stages = pl.stages;
  p.kw = pl.kw;
  p.units_per_problem = pl.units_per_problem;
  p.num_units = pl.num_units;
  if (pl.num_units == 0) return cudaSuccess;
  if (xd == BT_F16) return launch_x<BT_F16>(p, bits, yd, pl.cpl, pl.grid, pl.smem, st);
  return launch_x<BT_BF16>(p, bits, yd, pl.cpl, pl.grid, pl.smem, st);
}

}  // namespace bt
