// Dequant-GEMM for a few tokens per weight (M = 2..32 dense rows, or the ~8 rows
// an expert receives in a grouped prefill launch) on the tensor pipe.  BaseRT
// pages, thetesserapress.com "BaseRT claims fastest Apple Silicon inference",
// section "What BaseRT does differently" (more than one token: a GEMM; the codes
// are expanded inside the product, no dequantized weight is stored) and section
// "Where the wins land, and where they don't" (expert layers and short batches
// wait on memory: every weight byte should cross HBM once per launch).
//
// At these sizes a weight row meets only a few tokens, so the product is bound
// by reading the packed codes, not by arithmetic.  The kernel therefore streams
// each weight tile once and multiplies it by every token of its problem:
//  * Persistent CTAs walk row blocks (rb = 128 / kw weight rows of one problem,
//    for one staging of x).  Warp 8 fills a ring of stages, each one TMA copy of
//    kw 128-byte K boxes x rb rows with the 128-byte swizzle (the codes viewed as
//    [box][row][128 B]), plus the boxes' fp16 scales and biases with 8-byte
//    cp.async into rows padded so that eight rows' loads hit eight different
//    bank pairs.
//  * Consumer warp (rt, kw) owns rows 16 rt .. 16 rt + 15 of every row block and
//    box kw of every stage; it accumulates over all the block's stages, and the
//    kw warps of a tile meet in shared memory once per row block.
//  * The A operand of mma.sync m16n8k16 comes straight from the codes: ldmatrix
//    gives each lane one word (8 codes) of rows g and g+8, and one AND (fp16 x:
//    codes as exact subnormals q*2^-24, the odd pairs as 16q*2^-24) or one LOP3
//    (bf16 x: 128 + q) turns a word into four operand pairs.
//  * B is x: the problem's tokens, permuted to that pair order (and for fp16 the
//    odd pairs divided by 16), written once per problem into shared memory with
//    each token's group sums.  Token j of n8 tile i is column j of the MMA.
//  * Per quantization group the four MMAs' D (16 rows x 8 tokens) is folded into
//    fp32 accumulators as s*D + b*sum(x) (bf16: (b - 128 s)*sum(x)).
#include <cuda.h>

#include <cstring>
#include <memory>

#include "qgemm.cuh"
#include "qgemv_mma.cuh"

namespace bt {
namespace small {

using gemv::ldmatrix_x4;
using gemv::launder;
using gemv::lds128_nv;
using gemv::prmt;

// Consumer warps per CTA (NW, 8 or 16) are a template parameter; the producer
// is warp NW.
template <int NW> constexpr int kThreadsT = (NW + 1) * 32;
constexpr int kMaxT8 = 4;                        // at most 32 tokens per staging of x
constexpr uint32_t kBox = 128;                   // bytes of a row per TMA box (the swizzle span)

struct SmallParams {
  int M, N, K, G;              // M: dense rows, or grouped rows in total; G = K / 64
  int kw;                      // warps sharing a 16-row tile: each takes one 128-byte K box of a stage
  int rb;                      // weight rows per row block (16 * NW / kw)
  int upp;                     // row blocks per problem
  int kchunks;                 // stages per row block: ceil(nbox / kw)
  int nbox;                    // 128-byte K boxes per row (4 groups each)
  int stages;
  uint32_t stage_bytes;        // one ring slot: codes (kw boxes x rb rows x 128 B), then scales, then biases
  uint32_t code_bytes;         // kw * rb * 128
  uint32_t pstride;            // bytes between two rows' staged parameters
  int tok_chunk;               // tokens per staging of x (8 * t8)
  uint32_t x_tok_stride;       // bytes between two tokens' staged x (G * 128 + 64)
  uint32_t xsum_off;           // staged group sums, [G][tok_chunk] fp32, after the staged x
  uint32_t red_off;            // K-split partials
  uint32_t bar_off;            // mbarriers
  const uint16_t* scales;
  const uint16_t* biases;
  const uint16_t* x;           // [rows][K] fp16 or bf16
  const int32_t* row_index;    // grouped: x row of grouped row r (or null: row r)
  const int32_t* offsets;      // grouped: [E + 1]; null: dense
  int num_experts;
  void* y;
  bt_dtype y_dtype;
  int swiglu;                  // rows 2i / 2i+1 are gate_i / up_i; Y is [rows][N / 2]
  int const_weights;           // PDL: weights may be read before the previous kernel ends
  unsigned* err;
  unsigned long long timeout_ns;
};

// A batch of dense problems in one launch (a decode step of several tokens):
// each with its own codes (tensor map), parameters, x [M][K] and y [M][N].
struct SmallProblem {
  CUtensorMap map;             // codes viewed as [box][row][128 B]
  const uint16_t* scales;
  const uint16_t* biases;
  const uint16_t* x;
  void* y;
  int N, K;
};
constexpr int kSmallBatchCap = kBatchLaunchCap;   // 256 bytes per entry: the table fits the 32 KB of kernel parameters
template <int CAP> struct SmallBatch {
  SmallProblem prob[CAP];
  int count;
};

// What the kernel needs of one problem.
struct PView {
  const CUtensorMap* map;
  const uint16_t* scales;
  const uint16_t* biases;
  const uint16_t* x;
  void* y;
  int N, K, G, upp, kchunks;
  uint32_t xts;                // bytes between two tokens' staged x
};

template <bool BATCH, class Tab>
__device__ __forceinline__ PView view(const SmallParams& p, const CUtensorMap* map, const Tab& tab, int e) {
  if constexpr (BATCH) {
    const SmallProblem& q = tab.prob[e];
    const int G = q.K >> 6;
    return PView{&q.map, q.scales, q.biases, q.x, q.y, q.N, q.K, G, (q.N + p.rb - 1) / p.rb,
                 ((q.K >> 8) + p.kw - 1) / p.kw, (uint32_t)G * 128u + 64u};
  } else {
    return PView{map, p.scales, p.biases, p.x, p.y, p.N, p.K, p.G, p.upp, p.kchunks, p.x_tok_stride};
  }
}

// One stage (rb rows x kw 128-byte K boxes from box0) in one TMA copy.  The codes
// are viewed as [box][row][128 bytes] (dense) or [expert][box][row][128 bytes]
// (grouped), so shared memory receives the stage's box b at b * rb * 128, each
// 128-byte row with its 16-byte chunks swizzled by the row index mod 8.
__device__ __forceinline__ void tma_unit_3d(uint32_t dst, const CUtensorMap* map, int row0, int box0,
                                            uint64_t* bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, "
      "%3, %4}], [%5], %6;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(row0), "r"(box0), "r"(smem_u32(bar)), "l"(pol)
      : "memory");
}
__device__ __forceinline__ void tma_unit_4d(uint32_t dst, const CUtensorMap* map, int row0, int box0, int e,
                                            uint64_t* bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, "
      "%3, %4, %5}], [%6], %7;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(row0), "r"(box0), "r"(e), "r"(smem_u32(bar)), "l"(pol)
      : "memory");
}
__device__ __forceinline__ void cp_async8(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ uint2 lds64_nv(uint32_t a) {
  uint2 v;
  asm("ld.shared.v2.b32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
  return v;
}
__device__ __forceinline__ float2 lds64f_nv(uint32_t a) {
  float2 v;
  asm("ld.shared.v2.f32 {%0,%1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(a));
  return v;
}

template <bool BF16>
__device__ __forceinline__ void mma(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                    uint32_t b1) {
  if constexpr (BF16)
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  else
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// One word of 8 four-bit codes (code j in bits 4j..4j+3) -> four A pairs, codes
// (0,4) (1,5) (2,6) (3,7).  fp16: exact subnormals q*2^-24, the (1,5) and (3,7)
// pairs scaled by 16 (their x is staged divided by 16).  bf16: 128 + q, all pairs
// unscaled (the 128 comes back out through the bias term).
template <bool BF16>
__device__ __forceinline__ void a_pairs(uint32_t w, uint32_t (&p)[4]) {
  if constexpr (BF16) {
    constexpr uint32_t M = 0x000F000Fu, MG = 0x43004300u;
    p[0] = lop3_and_or(w, M, MG);
    p[1] = lop3_and_or(w >> 4, M, MG);
    p[2] = lop3_and_or(w >> 8, M, MG);
    p[3] = lop3_and_or(w >> 12, M, MG);
  } else {
    const uint32_t w8 = w >> 8;
    p[0] = w & 0x000F000Fu;
    p[1] = w & 0x00F000F0u;
    p[2] = w8 & 0x000F000Fu;
    p[3] = w8 & 0x00F000F0u;
  }
}

// Rows of problem e (dense: the M rows; grouped: expert e's rows, clamped to M).
template <bool GROUPED>
__device__ __forceinline__ void problem_rows(const SmallParams& p, int e, int& lo, int& cnt) {
  if constexpr (GROUPED) {
    lo = max(0, __ldg(p.offsets + e));
    cnt = max(0, min(__ldg(p.offsets + e + 1), p.M) - lo);
  } else {
    lo = 0;
    cnt = p.M;
  }
}

// Units of the walk: (problem, token chunk, row block).  Problem e contributes
// chunks(e) * upp(e) units, chunks(e) = ceil(rows of e / tok_chunk).
template <bool BATCH, class Tab>
__device__ __forceinline__ int upp_of(const SmallParams& p, const Tab& tab, int e) {
  if constexpr (BATCH) return (tab.prob[e].N + p.rb - 1) / p.rb;
  else return p.upp;
}
template <bool GROUPED, bool BATCH, class Tab>
__device__ __forceinline__ int problem_units(const SmallParams& p, const Tab& tab, int e) {
  int lo, cnt;
  problem_rows<GROUPED>(p, e, lo, cnt);
  return ((cnt + p.tok_chunk - 1) / p.tok_chunk) * upp_of<BATCH>(p, tab, e);
}

// Warp-collective: total units of the launch.
template <bool GROUPED, bool BATCH, class Tab>
__device__ long long count_units(const SmallParams& p, const Tab& tab) {
  if constexpr (BATCH) {
    long long total = 0;
    for (int e = 0; e < tab.count; ++e) total += problem_units<GROUPED, BATCH>(p, tab, e);
    return total;
  }
  if constexpr (!GROUPED) return problem_units<GROUPED, BATCH>(p, tab, 0);
  const int lane = threadIdx.x & 31;
  long long total = 0;
  for (int base = 0; base < p.num_experts; base += 32) {
    const int e = base + lane;
    long long c = e < p.num_experts ? problem_units<GROUPED, BATCH>(p, tab, e) : 0;
#pragma unroll
    for (int o = 16; o; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
    total += c;
  }
  return total;
}

// Grouped launches weigh an expert's units by the n8 token tiles it multiplies
// (a unit's work is a fixed part per K group plus a part per tile), so that the
// CTAs' contiguous shares of the walk take similar time.
template <bool GROUPED, bool BATCH, class Tab>
__device__ __forceinline__ long long unit_weight(const SmallParams& p, const Tab& tab, int e) {
  int lo, cnt;
  problem_rows<GROUPED>(p, e, lo, cnt);
  return 5 + 2 * ((min(cnt, p.tok_chunk) + 7) >> 3);
}

// Warp-collective (grouped): the index of the first unit whose weighted start is
// at or after `c` (the number of units when there is none).
template <bool GROUPED, bool BATCH, class Tab>
__device__ long long unit_at_cost(const SmallParams& p, const Tab& tab, long long c) {
  const int lane = threadIdx.x & 31;
  long long units_before = 0, cost_before = 0;
  for (int base = 0; base < p.num_experts; base += 32) {
    const int e = base + lane;
    const long long n = e < p.num_experts ? problem_units<GROUPED, BATCH>(p, tab, e) : 0;
    const long long w = e < p.num_experts ? unit_weight<GROUPED, BATCH>(p, tab, e) : 1;
    const long long cost = n * w;
    long long ci = cost, ni = n;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long tc = __shfl_up_sync(0xffffffffu, ci, o);
      const long long tn = __shfl_up_sync(0xffffffffu, ni, o);
      if (lane >= o) { ci += tc; ni += tn; }
    }
    const long long c0 = cost_before + ci - cost;   // weighted start of this lane's expert
    const unsigned hit = __ballot_sync(0xffffffffu, n > 0 && c < c0 + cost);
    if (hit) {
      const int src = __ffs(hit) - 1;
      const long long sc0 = __shfl_sync(0xffffffffu, c0, src);
      const long long sw = __shfl_sync(0xffffffffu, w, src);
      const long long su0 = units_before + __shfl_sync(0xffffffffu, ni - n, src);
      return su0 + (c > sc0 ? (c - sc0 + sw - 1) / sw : 0);
    }
    cost_before += __shfl_sync(0xffffffffu, ci, 31);
    units_before += __shfl_sync(0xffffffffu, ni, 31);
  }
  return units_before;
}

// Warp-collective (grouped): the weighted size of the walk.
template <bool GROUPED, bool BATCH, class Tab>
__device__ long long count_cost(const SmallParams& p, const Tab& tab) {
  const int lane = threadIdx.x & 31;
  long long total = 0;
  for (int base = 0; base < p.num_experts; base += 32) {
    const int e = base + lane;
    long long c = e < p.num_experts ? problem_units<GROUPED, BATCH>(p, tab, e) * unit_weight<GROUPED, BATCH>(p, tab, e)
                                    : 0;
#pragma unroll
    for (int o = 16; o; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
    total += c;
  }
  return total;
}

// Warp-collective: the problem holding unit u and the unit's place in it.
template <bool GROUPED, bool BATCH, class Tab>
__device__ void locate(const SmallParams& p, const Tab& tab, long long u, int& e, int& ch, int& blk) {
  e = 0;
  if constexpr (BATCH) {
    while (e + 1 < tab.count && u >= problem_units<GROUPED, BATCH>(p, tab, e)) {
      u -= problem_units<GROUPED, BATCH>(p, tab, e);
      ++e;
    }
  } else if constexpr (GROUPED) {
    const int lane = threadIdx.x & 31;
    for (int base = 0; base < p.num_experts; base += 32) {
      const int ee = base + lane;
      const long long c = ee < p.num_experts ? problem_units<GROUPED, BATCH>(p, tab, ee) : 0;
      long long incl = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const long long t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
      }
      const unsigned hit = __ballot_sync(0xffffffffu, c > 0 && u < incl && u >= incl - c);
      if (hit) {
        const int src = __ffs(hit) - 1;
        e = base + src;
        u -= __shfl_sync(0xffffffffu, incl - c, src);
        break;
      }
      u -= __shfl_sync(0xffffffffu, incl, 31);
    }
  }
  const int upp = upp_of<BATCH>(p, tab, e);
  ch = (int)(u / upp);
  blk = (int)(u - (long long)ch * upp);
}

// The unit after (e, ch, blk).
template <bool GROUPED, bool BATCH, class Tab>
__device__ __forceinline__ void advance(const SmallParams& p, const Tab& tab, int& e, int& ch, int& blk) {
  const int upp = upp_of<BATCH>(p, tab, e);
  if (++blk < upp) return;
  blk = 0;
  if (++ch * upp < problem_units<GROUPED, BATCH>(p, tab, e)) return;
  ch = 0;
  if constexpr (GROUPED) {
    do {
      ++e;
    } while (e < p.num_experts && problem_units<GROUPED, BATCH>(p, tab, e) == 0);
  } else {
    ++e;
  }
}

// Stage the x of rows first..first+ntok-1 of the problem (zeros up to npad) in
// B-fragment order: slot (token, group v, chunk c, lane t), 16 bytes at
// token * x_tok_stride + v * 128 + c * 64 + t * 16, holds the x of codes
// 64v + 32c + 8t + (0,4) (1,5) (2,6) (3,7); with fp16 the (1,5) and (3,7) pairs
// are divided by 16.  xsum[v][token] = sum of token's x over group v (fp32).
// Each thread issues kInFlight independent 16-byte loads before using any, so a
// staging costs a few L2 round trips rather than one per slot.
constexpr int kInFlight = 8;

template <bool BF16, bool GROUPED, int NW>
__device__ void stage_x(const SmallParams& p, const PView& pv, uint32_t xs, float* xsum, int first, int ntok,
                        int npad, int ctid) {
  constexpr int kStep = NW * 32;
  const int lane = ctid & 31;
  const int per_tok = pv.G * 8;
  const int items = npad * per_tok;
  for (int base = ctid - lane; base < items; base += kInFlight * kStep) {
    uint4 raw[kInFlight];
#pragma unroll
    for (int u = 0; u < kInFlight; ++u) {
      const int idx = base + u * kStep + lane;
      raw[u] = make_uint4(0u, 0u, 0u, 0u);
      const int tok = idx / per_tok;
      if (idx < items && tok < ntok) {
        const int rem = idx - tok * per_tok;
        const int v = rem >> 3, c = (rem >> 2) & 1, t = rem & 3;
        int row = first + tok;
        if constexpr (GROUPED) {
          if (p.row_index) row = __ldg(p.row_index + row);
        }
        raw[u] = __ldg(reinterpret_cast<const uint4*>(pv.x + (size_t)row * pv.K + (size_t)v * 64 + c * 32 + t * 8));
      }
    }
#pragma unroll
    for (int u = 0; u < kInFlight; ++u) {
      const int idx = base + u * kStep + lane;
      const int tok = idx / per_tok, rem = idx - tok * per_tok;
      const uint4 r = raw[u];   // halves j = 0..7: x at codes 8t + j (zeros past the last token)
      uint4 o;
      o.x = prmt(r.x, r.z, 0x5410u);   // (x0, x4)
      o.y = prmt(r.x, r.z, 0x7632u);   // (x1, x5)
      o.z = prmt(r.y, r.w, 0x5410u);   // (x2, x6)
      o.w = prmt(r.y, r.w, 0x7632u);   // (x3, x7)
      float part;
      if constexpr (BF16) {
        const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&r.x));
        const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&r.y));
        const float2 cc = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&r.z));
        const float2 d = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&r.w));
        part = ((a.x + a.y) + (b.x + b.y)) + ((cc.x + cc.y) + (d.x + d.y));
      } else {
        const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&r.x));
        const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&r.y));
        const float2 cc = __half22float2(*reinterpret_cast<const __half2*>(&r.z));
        const float2 d = __half22float2(*reinterpret_cast<const __half2*>(&r.w));
        part = ((a.x + a.y) + (b.x + b.y)) + ((cc.x + cc.y) + (d.x + d.y));
        const __half2 sixteenth = __float2half2_rn(0.0625f);
        const __half2 h1 = __hmul2(*reinterpret_cast<const __half2*>(&o.y), sixteenth);
        const __half2 h3 = __hmul2(*reinterpret_cast<const __half2*>(&o.w), sixteenth);
        o.y = *reinterpret_cast<const uint32_t*>(&h1);
        o.w = *reinterpret_cast<const uint32_t*>(&h3);
      }
      if (idx < items) {
        const int v = rem >> 3, c = (rem >> 2) & 1, t = rem & 3;
        const uint32_t dst = xs + (uint32_t)tok * pv.xts + (uint32_t)(v * 128 + c * 64 + t * 16);
        asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(dst), "r"(o.x), "r"(o.y), "r"(o.z), "r"(o.w)
                     : "memory");
      }
      part += __shfl_xor_sync(0xffffffffu, part, 1);
      part += __shfl_xor_sync(0xffffffffu, part, 2);
      part += __shfl_xor_sync(0xffffffffu, part, 4);
      if (idx < items && (idx & 7) == 0) xsum[(rem >> 3) * p.tok_chunk + tok] = part;
    }
  }
}

__device__ __forceinline__ void store_y(const SmallParams& p, void* y, size_t i, float v) {
  if (p.y_dtype == BT_F32) store_out<BT_F32>(y, i, v);
  else if (p.y_dtype == BT_BF16) store_out<BT_BF16>(y, i, v);
  else store_out<BT_F16>(y, i, v);
}

template <bool BF16, int T8, bool GROUPED, int NW, bool BATCH>
__global__ void __launch_bounds__(kThreadsT<NW>, 1)
    qgemm_small_kernel(const __grid_constant__ CUtensorMap map_codes, const SmallParams p,
                       const __grid_constant__ SmallBatch<BATCH ? kSmallBatchCap : 1> batch) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = p.stages;
  const uint32_t ring = smem_u32(smem);
  const uint32_t xs0 = ring + (uint32_t)S * p.stage_bytes;
  float* xsum = reinterpret_cast<float*>(smem + p.xsum_off);
  float* red = reinterpret_cast<float*>(smem + p.red_off);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + p.bar_off);
  uint64_t* empty = full + S;
  __shared__ volatile int s_fail;

  // the CTA's share of the row-block units; every unit is kchunks ring stages
  long long u_begin, u_end;
  if constexpr (GROUPED) {
    const long long C = count_cost<GROUPED, BATCH>(p, batch);
    u_begin = unit_at_cost<GROUPED, BATCH>(p, batch, C * blockIdx.x / gridDim.x);
    u_end = unit_at_cost<GROUPED, BATCH>(p, batch, C * (blockIdx.x + 1) / gridDim.x);
  } else {
    const long long U = count_units<GROUPED, BATCH>(p, batch);
    u_begin = U * blockIdx.x / gridDim.x;
    u_end = U * (blockIdx.x + 1) / gridDim.x;
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 33);
      mbar_init(&empty[s], NW);
    }
    s_fail = 0;
    fence_mbar_init();
  }
  __syncthreads();
  pdl_launch_dependents();
  if (u_begin >= u_end) return;
  int e, ch, blk;
  locate<GROUPED, BATCH>(p, batch, u_begin, e, ch, blk);

  if (warp == NW) {
    // ------------------------------------------------------------ producer
    if (!p.const_weights) pdl_wait();
    const uint64_t pol = l2_policy_evict_first();
    const int gps = 4 * p.kw;   // quantization groups per stage
    int s = 0;
    uint32_t ph = 0;
    long long it = 0;
    bool ok = true;
    for (long long u = u_begin; u < u_end && ok; ++u) {
      const PView pv = view<BATCH>(p, &map_codes, batch, e);
      const int row0 = blk * p.rb;
      const int rows = min(p.rb, pv.N - row0);
      for (int kc = 0; kc < pv.kchunks; ++kc, ++it) {
        if (it >= S) {
          bool w = true;
          if (lane == 0) w = mbar_wait(&empty[s], ph ^ 1u, p.timeout_ns, p.err);
          if (!__shfl_sync(0xffffffffu, (int)w, 0)) { ok = false; s_fail = 1; break; }
        }
        const uint32_t st = ring + (uint32_t)s * p.stage_bytes;
        if (lane == 0) {
          mbar_arrive_expect_tx(&full[s], p.code_bytes);
          if constexpr (GROUPED) tma_unit_4d(st, pv.map, row0, kc * p.kw, e, &full[s], pol);
          else tma_unit_3d(st, pv.map, row0, kc * p.kw, &full[s], pol);
        }
        // scales / biases of groups [kc * gps, +gps) for the block's rows: 8-byte pieces of 4 groups
        const int g0 = kc * gps;
        const int pieces = min(gps, pv.G - g0) >> 2;
        const size_t prow0 = ((size_t)(GROUPED ? e : 0) * pv.N + row0) * pv.G + g0;
        const uint32_t sdst = st + p.code_bytes, bdst = sdst + (uint32_t)p.rb * p.pstride;
        for (int i = lane; i < rows * pieces; i += 32) {
          const int r = i / pieces, j = i - r * pieces;
          const size_t off = prow0 + (size_t)r * pv.G + 4 * j;
          cp_async8(sdst + (uint32_t)r * p.pstride + 8u * j, pv.scales + off);
          cp_async8(bdst + (uint32_t)r * p.pstride + 8u * j, pv.biases + off);
        }
        cp_async_mbar_arrive_noinc(&full[s]);
        if (++s == S) { s = 0; ph ^= 1u; }
      }
      advance<GROUPED, BATCH>(p, batch, e, ch, blk);
    }
    if (!ok) {
      cp_async_wait_all();
      if (lane == 0)
        for (long long j = (it > S ? it - S : 0); j < it; ++j)   // failure path only
          mbar_wait(&full[j % S], (uint32_t)((j / S) & 1), p.timeout_ns, p.err);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  // warp (rt, kw): rows [16 rt, 16 rt + 16) of each row block, K box kw of each stage
  const int g = lane >> 2, tq = lane & 3;
  const int KW = p.kw, rt = warp / KW, kw = warp - rt * KW;
  const int r_lo = rt * 16;
  const int ld_row = (lane & 7) + ((lane >> 3) & 1) * 8; // tile row whose address this lane gives ldmatrix
  const uint32_t ld_c = (uint32_t)(lane >> 4);           // which 32-code half of a group it addresses
  const uint32_t box_off = (uint32_t)kw * (uint32_t)p.rb * kBox;
  uint32_t xs = xs0, xsa = smem_u32(xsum);
  bool dead = false;
  int s = 0;
  uint32_t ph = 0;
  int staged_e = -1, staged_ch = -1, rbuf = 0;
  pdl_wait();   // x comes from the previous kernel
  for (long long u = u_begin; u < u_end; ++u) {
    const PView pv = view<BATCH>(p, &map_codes, batch, e);
    int plo, pcnt;
    problem_rows<GROUPED>(p, e, plo, pcnt);
    const int first = plo + ch * p.tok_chunk;
    const int ntok = min(p.tok_chunk, pcnt - ch * p.tok_chunk);
    const int nt = (ntok + 7) >> 3;
    const int row0 = blk * p.rb;
    const int rows = min(p.rb, pv.N - row0);
    if (staged_e != e || staged_ch != ch) {
      // every consumer is done with the previous x before it is replaced
      asm volatile("bar.sync 15, %0;" ::"r"(NW * 32) : "memory");
      if (!dead) stage_x<BF16, GROUPED, NW>(p, pv, xs0, xsum, first, ntok, nt * 8, (int)threadIdx.x);
      asm volatile("bar.sync 15, %0;" ::"r"(NW * 32) : "memory");
      staged_e = e;
      staged_ch = ch;
      xs = launder(xs0);
      xsa = launder(smem_u32(xsum));
    }
    float acc[T8][4];
#pragma unroll
    for (int i = 0; i < T8; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
    const bool live_rows = r_lo < rows;   // this warp's tile has rows in the block
    for (int kc = 0; kc < pv.kchunks; ++kc) {
      if (!dead && (s_fail || !mbar_wait(&full[s], ph, p.timeout_ns, p.err))) {
        dead = true;
        s_fail = 1;
      }
      const int vb = (kc * KW + kw) * 4;   // first group of this warp's box
      if (!dead && live_rows && vb < pv.G) {
        const uint32_t st = launder(ring + (uint32_t)s * p.stage_bytes);   // after the wait
        const int R = r_lo + ld_row;
        const uint32_t ldb = st + box_off + (uint32_t)R * kBox;
        const uint32_t swz = (uint32_t)(R & 7);
        const int ra = r_lo + g, rb2 = ra + 8;
        const uint32_t ps = st + p.code_bytes + (uint32_t)kw * 8u;
        const uint32_t pb = ps + (uint32_t)p.rb * p.pstride;
        // scales / biases of the box's 4 groups for rows g and g + 8
        const uint2 s4a = lds64_nv(ps + (uint32_t)ra * p.pstride), s4b = lds64_nv(ps + (uint32_t)rb2 * p.pstride);
        const uint2 b4a = lds64_nv(pb + (uint32_t)ra * p.pstride), b4b = lds64_nv(pb + (uint32_t)rb2 * p.pstride);
        const uint32_t xb = xs + (uint32_t)g * pv.xts + (uint32_t)(tq * 16);
        const uint32_t xsb = xsa + (uint32_t)(2 * tq) * 4u;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int v = vb + j;
          uint32_t r[4];
          ldmatrix_x4(ldb + ((((uint32_t)(j << 1) | ld_c) ^ swz) << 4), r);
          uint32_t pa[4], pbq[4], pc[4], pd[4];
          a_pairs<BF16>(r[0], pa);    // row g, codes 0..31 of the group (word tq: codes 8tq..8tq+7)
          a_pairs<BF16>(r[1], pbq);   // row g + 8
          a_pairs<BF16>(r[2], pc);    // row g, codes 32..63
          a_pairs<BF16>(r[3], pd);    // row g + 8
          const float sa = to_f32<BT_F16>((uint16_t)(((j < 2) ? s4a.x : s4a.y) >> (16 * (j & 1))));
          const float sb = to_f32<BT_F16>((uint16_t)(((j < 2) ? s4b.x : s4b.y) >> (16 * (j & 1))));
          float ba = to_f32<BT_F16>((uint16_t)(((j < 2) ? b4a.x : b4a.y) >> (16 * (j & 1))));
          float bb = to_f32<BT_F16>((uint16_t)(((j < 2) ? b4b.x : b4b.y) >> (16 * (j & 1))));
          float ka, kb;   // multipliers of D
          if constexpr (BF16) {
            ka = sa;
            kb = sb;
            ba = fmaf(-128.f, sa, ba);   // D counted 128 + q
            bb = fmaf(-128.f, sb, bb);
          } else {
            ka = sa * 16777216.f;        // D counted q * 2^-24
            kb = sb * 16777216.f;
          }
#pragma unroll
          for (int i8 = 0; i8 < T8; ++i8) {
            if (i8 < nt) {
              const uint32_t xa = xb + (uint32_t)(8 * i8) * pv.xts + (uint32_t)v * 128u;
              const uint4 b1 = lds128_nv(xa), b2 = lds128_nv(xa + 64u);
              float d0[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f};
              mma<BF16>(d0, pa[0], pbq[0], pa[1], pbq[1], b1.x, b1.y);
              mma<BF16>(d1, pc[0], pd[0], pc[1], pd[1], b2.x, b2.y);
              mma<BF16>(d0, pa[2], pbq[2], pa[3], pbq[3], b1.z, b1.w);
              mma<BF16>(d1, pc[2], pd[2], pc[3], pd[3], b2.z, b2.w);
              const float2 xv = lds64f_nv(xsb + (uint32_t)(v * p.tok_chunk + 8 * i8) * 4u);
              acc[i8][0] = fmaf(ka, d0[0] + d1[0], fmaf(ba, xv.x, acc[i8][0]));
              acc[i8][1] = fmaf(ka, d0[1] + d1[1], fmaf(ba, xv.y, acc[i8][1]));
              acc[i8][2] = fmaf(kb, d0[2] + d1[2], fmaf(bb, xv.x, acc[i8][2]));
              acc[i8][3] = fmaf(kb, d0[3] + d1[3], fmaf(bb, xv.y, acc[i8][3]));
            }
          }
        }
      }
      __syncwarp();
      if (!dead && lane == 0) mbar_arrive(&empty[s]);
      if (++s == S) { s = 0; ph ^= 1u; }
    }
    if (KW > 1) {
      // the tile's KW warps meet once per row block, lane-major; the buffer
      // alternates so a warp one block ahead never overwrites unread values
      constexpr int kVals = 4 * T8;
      float* mine = red + (size_t)(((rt * 2 + rbuf) * KW + kw) * kVals) * 32;
#pragma unroll
      for (int i = 0; i < T8; ++i)
#pragma unroll
        for (int c = 0; c < 4; ++c) mine[(i * 4 + c) * 32 + lane] = acc[i][c];
      asm volatile("bar.sync %0, %1;" ::"r"(1 + rt), "r"(KW * 32) : "memory");
      if (kw == 0) {
        const float* all = red + (size_t)((rt * 2 + rbuf) * KW * kVals) * 32;
#pragma unroll
        for (int i = 0; i < T8; ++i)
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            float sum = 0.f;
            for (int k = 0; k < KW; ++k) sum += all[(size_t)(k * kVals + i * 4 + c) * 32 + lane];
            acc[i][c] = sum;
          }
      }
      rbuf ^= 1;
    }
    if (kw == 0) {
#pragma unroll
      for (int i8 = 0; i8 < T8; ++i8) {
        if (i8 < nt) {
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int row = r_lo + g + ((c >> 1) << 3);
            const int tok = 8 * i8 + 2 * tq + (c & 1);
            const float val = acc[i8][c];
            if (p.swiglu) {
              // gate row 2i (even g) and its up row 2i + 1 sit in lanes 4 apart
              const float up = __shfl_xor_sync(0xffffffffu, val, 4);
              if (!dead && !(g & 1) && row < rows && tok < ntok)
                store_y(p, pv.y, (size_t)(first + tok) * (pv.N / 2) + ((row0 + row) >> 1),
                        val / (1.f + expf(-val)) * up);
            } else if (!dead && row < rows && tok < ntok) {
              store_y(p, pv.y, (size_t)(first + tok) * pv.N + row0 + row, val);
            }
          }
        }
      }
    }
    advance<GROUPED, BATCH>(p, batch, e, ch, blk);
  }
}

// ------------------------------------------------------------------ host side
constexpr int kMaxStages = 16;
constexpr size_t kXBudget = 112 * 1024;      // staged x + group sums
constexpr size_t kSmemMax = 226 * 1024;     // dynamic, leaving room for the static fail flag

struct Layout {
  SmallGeometry geo;
  int nbox = 0, kchunks = 0;
  uint32_t pstride = 0, stage_bytes = 0, code_bytes = 0, x_tok_stride = 0;
  uint32_t xsum_off = 0, red_off = 0, bar_off = 0;
};

inline uint32_t align_up(size_t v, size_t a) { return (uint32_t)((v + a - 1) / a * a); }

Layout plan_layout(int bits, int M, int N, int K, int group, int num_experts, int sms, int nw) {
  Layout L;
  SmallGeometry& g = L.geo;
  if (bits != 4 || group != 64 || K < 256 || K % 256 || K > kMaxK || N < 16 || N % 8 || M < 1 || num_experts < 0)
    return L;
  if (num_experts == 0 && M > 8 * kMaxT8) return L;
  const int G = K / 64, row_bytes = K / 2;
  L.nbox = row_bytes / (int)kBox;
  L.x_tok_stride = (uint32_t)G * 128u + 64u;   // odd multiple of 64: tokens g, g+1 in different banks
  int t8;
  if (num_experts == 0) {
    t8 = (M + 7) / 8;
  } else {
    const int mean = (M + num_experts - 1) / num_experts;   // rows per expert
    t8 = std::min(kMaxT8, std::max(1, (3 * mean / 2 + 7) / 8));
  }
  auto x_bytes = [&](int t) { return (size_t)8 * t * L.x_tok_stride + (size_t)8 * t * G * 4; };
  while (t8 > 1 && x_bytes(t8) > kXBudget) --t8;
  if (x_bytes(t8) > kXBudget || (num_experts == 0 && 8 * t8 < M)) return L;
  // K boxes per stage (= warps per 16-row tile): one (the most rows per block)
  // while the row blocks alone give every SM one, else more boxes over fewer rows
  const long long problems = std::max(1, num_experts);
  int kw = 1;
  while (kw < 8 && (long long)((N + 16 * nw / kw - 1) / (16 * nw / kw)) * problems < sms) kw *= 2;
  const int rb = 16 * nw / kw;
  if (rb > 256) return L;   // TMA box rows
  // parameter rows (4 groups per box) padded to an odd multiple of 8 bytes: eight
  // rows' 8-byte loads land in eight different bank pairs
  L.pstride = 8u * (uint32_t)(kw + ((kw % 2 == 0) ? 1 : 2));
  L.kchunks = (L.nbox + kw - 1) / kw;
  L.code_bytes = (uint32_t)(kw * rb * (int)kBox);
  L.stage_bytes = align_up((size_t)L.code_bytes + (size_t)2 * rb * L.pstride, 1024);
  const size_t red = kw > 1 ? (size_t)2 * nw * 4 * t8 * 32 * 4 : 0;
  const size_t xb = (size_t)8 * t8 * L.x_tok_stride;
  const size_t xsum = align_up((size_t)8 * t8 * G * 4, 16);
  const size_t fixed = 1024 + xb + xsum + red + 2 * 8 * kMaxStages;
  if (fixed + 2 * (size_t)L.stage_bytes > kSmemMax) return L;
  const int stages = (int)std::min<size_t>(kMaxStages, (kSmemMax - fixed) / L.stage_bytes);
  L.xsum_off = (uint32_t)(stages * (size_t)L.stage_bytes + xb);
  L.red_off = (uint32_t)(L.xsum_off + xsum);
  L.bar_off = (uint32_t)(L.red_off + red);
  g.t8 = t8;
  g.nw = nw;
  g.kw = kw;
  g.rb = rb;
  g.stages = stages;
  const long long units = (long long)((N + rb - 1) / rb) * problems;
  g.grid = (int)std::min<long long>(units, sms);
  g.smem = (long long)L.bar_off + 2 * 8 * stages + 1024;
  g.feasible = true;
  return L;
}

template <bool BATCH> using TabT = SmallBatch<BATCH ? kSmallBatchCap : 1>;

template <bool BF16, int T8, bool GROUPED, int NW, bool BATCH>
cudaError_t launch_t(const CUtensorMap& map, const SmallParams& p, const TabT<BATCH>& tab, int grid, size_t smem,
                     cudaStream_t st) {
  auto k = qgemm_small_kernel<BF16, T8, GROUPED, NW, BATCH>;
  static std::atomic<uint64_t> smem_raised{0};
  cudaError_t e = raise_smem_limit(reinterpret_cast<const void*>(k), smem_raised);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreadsT<NW>);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = opts().pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k, map, p, tab);
}

template <bool BF16, bool GROUPED, int NW, bool BATCH>
cudaError_t launch_x(const CUtensorMap& map, const SmallParams& p, const TabT<BATCH>& tab, int t8, int grid,
                     size_t smem, cudaStream_t st) {
  switch (t8) {
    case 1: return launch_t<BF16, 1, GROUPED, NW, BATCH>(map, p, tab, grid, smem, st);
    case 2: return launch_t<BF16, 2, GROUPED, NW, BATCH>(map, p, tab, grid, smem, st);
    case 3: return launch_t<BF16, 3, GROUPED, NW, BATCH>(map, p, tab, grid, smem, st);
    default: return launch_t<BF16, 4, GROUPED, NW, BATCH>(map, p, tab, grid, smem, st);
  }
}

template <bool BF16, bool GROUPED, bool BATCH>
cudaError_t launch_nw(const CUtensorMap& map, const SmallParams& p, const TabT<BATCH>& tab, const SmallGeometry& g,
                      cudaStream_t st) {
  if (g.nw == 16) return launch_x<BF16, GROUPED, 16, BATCH>(map, p, tab, g.t8, g.grid, (size_t)g.smem, st);
  return launch_x<BF16, GROUPED, 8, BATCH>(map, p, tab, g.t8, g.grid, (size_t)g.smem, st);
}

// Consumer warps: BT_OPT_GEMM_SMALL_WARPS = 8 or 16 forces either; by default
// 16 where that layout fits shared memory and takes at most two n8 token tiles
// (with three or four the 16-warp kernel, held to 96 registers, spills), else 8.
Layout plan_any(int bits, int M, int N, int K, int group, int num_experts, int sms) {
  const int forced = opts().gemm_small_warps;
  if (forced == 8 || forced == 16) return plan_layout(bits, M, N, K, group, num_experts, sms, forced);
  Layout L = plan_layout(bits, M, N, K, group, num_experts, sms, 16);
  if (!L.geo.feasible || L.geo.t8 > 2) {
    const Layout L8 = plan_layout(bits, M, N, K, group, num_experts, sms, 8);
    if (L8.geo.feasible) L = L8;
  }
  return L;
}

}  // namespace small

SmallGeometry plan_gemm_small(int bits, int M, int N, int K, int group, int num_experts, int sms) {
  return small::plan_any(bits, M, N, K, group, num_experts, sms).geo;
}

bool small_supported(int bits, const GemmParams& p) {
  const auto a16 = [](const void* q) { return (reinterpret_cast<uintptr_t>(q) & 15u) == 0; };
  const auto a8 = [](const void* q) { return (reinterpret_cast<uintptr_t>(q) & 7u) == 0; };
  return bits == 4 && p.group == 64 && a16(p.codes) && a8(p.scales) && a8(p.biases) && a16(p.x) &&
         plan_gemm_small(bits, p.M, p.N, p.K, p.group, p.offsets ? p.num_experts : 0, sm_count()).feasible;
}

namespace small {
// The codes of one weight (or E stacked experts) viewed as [E][box][row][128 B]:
// dim 0 the 128 bytes of a box row, dim 1 the rows (stride row_bytes), dim 2 the
// K boxes (stride 128), dim 3 the experts; a box is one stage (rb rows, kw boxes).
bool encode_codes_map(CUtensorMap* map, const uint32_t* codes, int N, int K, int experts, int rb, int kw) {
  tc::EncodeTiledFn enc = tc::encode_fn();
  if (!enc) return false;
  memset(map, 0, sizeof(*map));
  const int row_bytes = K / 2;
  const cuuint32_t elem[4] = {1, 1, 1, 1};
  const cuuint64_t dims[4] = {kBox, (cuuint64_t)N, (cuuint64_t)(row_bytes / (int)kBox), (cuuint64_t)std::max(1, experts)};
  const cuuint64_t strides[3] = {(cuuint64_t)row_bytes, kBox, (cuuint64_t)row_bytes * N};
  const cuuint32_t box[4] = {kBox, (cuuint32_t)rb, (cuuint32_t)kw, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, experts > 0 ? 4 : 3, const_cast<uint32_t*>(codes), dims, strides, box,
             elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

SmallParams make_params(const Layout& L, int M, bt_dtype yd, unsigned* err, unsigned long long timeout_ns) {
  SmallParams p{};
  p.M = M;
  p.rb = L.geo.rb;
  p.kw = L.geo.kw;
  p.kchunks = L.kchunks;
  p.stages = L.geo.stages;
  p.stage_bytes = L.stage_bytes;
  p.code_bytes = L.code_bytes;
  p.pstride = L.pstride;
  p.nbox = L.nbox;
  p.tok_chunk = 8 * L.geo.t8;
  p.x_tok_stride = L.x_tok_stride;
  p.xsum_off = L.xsum_off;
  p.red_off = L.red_off;
  p.bar_off = L.bar_off;
  p.y_dtype = yd;
  p.const_weights = opts().pdl && opts().const_weights;
  p.err = err;
  p.timeout_ns = timeout_ns;
  return p;
}
}  // namespace small

cudaError_t launch_gemm_small(const GemmParams& gp, int bits, bt_dtype xd, bt_dtype yd, cudaStream_t st) {
  using namespace small;
  const bool grouped = gp.offsets != nullptr;
  const Layout L = plan_any(bits, gp.M, gp.N, gp.K, gp.group, grouped ? gp.num_experts : 0, sm_count());
  if (!L.geo.feasible) return cudaErrorInvalidValue;
  CUtensorMap map;
  if (!encode_codes_map(&map, gp.codes, gp.N, gp.K, grouped ? gp.num_experts : 0, L.geo.rb, L.geo.kw))
    return cudaErrorInvalidValue;
  SmallParams p = make_params(L, gp.M, yd, gp.err, gp.timeout_ns);
  p.N = gp.N;
  p.K = gp.K;
  p.G = gp.K / 64;
  p.upp = (gp.N + L.geo.rb - 1) / L.geo.rb;
  p.scales = gp.scales;
  p.biases = gp.biases;
  p.x = static_cast<const uint16_t*>(gp.x);
  p.row_index = gp.row_index;
  p.offsets = gp.offsets;
  p.num_experts = grouped ? gp.num_experts : 1;
  p.y = gp.y;
  p.swiglu = gp.swiglu;
  const bool bf = xd == BT_BF16;
  static const TabT<false> none{};
  if (grouped)
    return bf ? launch_nw<true, true, false>(map, p, none, L.geo, st) : launch_nw<false, true, false>(map, p, none, L.geo, st);
  return bf ? launch_nw<true, false, false>(map, p, none, L.geo, st) : launch_nw<false, false, false>(map, p, none, L.geo, st);
}

// Several dense problems of the same M in one launch.  The layout is planned for
// the rows of all problems together and the largest K; every problem must fit
// the kernel's limits (4-bit codes, groups of 64, K a multiple of 256, N a
// multiple of 8, 16-byte aligned codes and x, 8-byte aligned parameters).
SmallGeometry plan_gemm_small_batched(const GemmProblem* probs, int count, int M, int sms) {
  if (count < 1 || count > small::kSmallBatchCap) return SmallGeometry{};
  long long rows = 0;
  int kmax = 0;
  for (int i = 0; i < count; ++i) {
    const GemmProblem& q = probs[i];
    if (!plan_gemm_small(4, M, q.N, q.K, 64, 0, sms).feasible) return SmallGeometry{};
    rows += q.N;
    kmax = std::max(kmax, q.K);
  }
  if (rows > (1LL << 30)) return SmallGeometry{};
  SmallGeometry g = small::plan_any(4, M, (int)rows, kmax, 64, 0, sms).geo;
  if (g.feasible) {
    long long units = 0;
    for (int i = 0; i < count; ++i) units += (probs[i].N + g.rb - 1) / g.rb;
    g.grid = (int)std::min<long long>(units, sms);
  }
  return g;
}

bool small_batch_supported(const GemmProblem* probs, int count, int M, int bits, int group) {
  if (bits != 4 || group != 64) return false;
  const auto a16 = [](const void* q) { return (reinterpret_cast<uintptr_t>(q) & 15u) == 0; };
  const auto a8 = [](const void* q) { return (reinterpret_cast<uintptr_t>(q) & 7u) == 0; };
  for (int i = 0; i < count; ++i)
    if (!a16(probs[i].codes) || !a16(probs[i].x) || !a8(probs[i].scales) || !a8(probs[i].biases)) return false;
  return plan_gemm_small_batched(probs, count, M, sm_count()).feasible;
}

struct SmallBatchPrepared {
  small::Layout L;
  small::TabT<true> tab;
  small::SmallParams p;
  bool bf16;
};

SmallBatchPrepared* prepare_gemm_small_batched(const GemmProblem* probs, int count, int M, bt_dtype xd, bt_dtype yd) {
  using namespace small;
  if (count < 1 || count > kSmallBatchCap) return nullptr;
  long long rows = 0;
  int kmax = 0;
  for (int i = 0; i < count; ++i) {
    rows += probs[i].N;
    kmax = std::max(kmax, probs[i].K);
  }
  std::unique_ptr<SmallBatchPrepared> pb(new SmallBatchPrepared);
  pb->L = plan_any(4, M, (int)rows, kmax, 64, 0, sm_count());
  if (!pb->L.geo.feasible) return nullptr;
  pb->L.geo.grid = plan_gemm_small_batched(probs, count, M, sm_count()).grid;
  if (pb->L.geo.grid < 1) return nullptr;
  memset(&pb->tab, 0, sizeof(pb->tab));
  pb->tab.count = count;
  for (int i = 0; i < count; ++i) {
    const GemmProblem& q = probs[i];
    SmallProblem& d = pb->tab.prob[i];
    if (!encode_codes_map(&d.map, q.codes, q.N, q.K, 0, pb->L.geo.rb, pb->L.geo.kw)) return nullptr;
    d.scales = q.scales;
    d.biases = q.biases;
    d.x = static_cast<const uint16_t*>(q.x);
    d.y = q.y;
    d.N = q.N;
    d.K = q.K;
  }
  pb->p = make_params(pb->L, M, yd, nullptr, 0);
  pb->p.num_experts = 1;
  pb->bf16 = xd == BT_BF16;
  return pb.release();
}

cudaError_t run_gemm_small_batched(const SmallBatchPrepared* pb, unsigned* err, unsigned long long timeout_ns,
                                   cudaStream_t st) {
  using namespace small;
  SmallParams p = pb->p;
  p.err = err;
  p.timeout_ns = timeout_ns;
  p.const_weights = opts().pdl && opts().const_weights;
  CUtensorMap unused;
  memset(&unused, 0, sizeof(unused));
  return pb->bf16 ? launch_nw<true, false, true>(unused, p, pb->tab, pb->L.geo, st)
                  : launch_nw<false, false, true>(unused, p, pb->tab, pb->L.geo, st);
}

void free_gemm_small_batched(SmallBatchPrepared* pb) { delete pb; }

cudaError_t launch_gemm_small_batched(const GemmProblem* probs, int count, int M, bt_dtype xd, bt_dtype yd,
                                      unsigned* err, unsigned long long timeout_ns, cudaStream_t st) {
  std::unique_ptr<SmallBatchPrepared> pb(prepare_gemm_small_batched(probs, count, M, xd, yd));
  if (!pb) return cudaErrorInvalidValue;
  return run_gemm_small_batched(pb.get(), err, timeout_ns, st);
}

}  // namespace bt
