// Dequant-GEMV (M = 1, decode) with the dot products on the tensor pipe
// (mma.sync m16n8k16, fp16 in, fp32 accumulate).  BaseRT pages,
// thetesserapress.com "BaseRT claims fastest Apple Silicon inference", section
// "What BaseRT does differently" (a GEMV of its own for M = 1 that expands the
// codes in its inner loop) and section "Where the wins land, and where they
// don't" (large-model decode waits on memory bandwidth: the kernel must keep
// up with HBM, so the contraction leaves the FMA pipe).
//
// What stays from the CUDA-core GEMV (qgemv_impl.cuh): persistent CTAs, one
// producer warp filling a shared-memory ring with one bulk copy per unit of
// rows (codes) plus 16-byte cp.async of the unit's scales and biases, batched
// problem tables, the K split over warps of a row group with a named-barrier
// reduction, and the fail flag that keeps every warp on its barriers after an
// expired wait.
//
// What changes is the consumer.  A warp takes a tile of 16 weight rows and its
// K slice, one quantization group (64 codes, two 16-byte chunks per row at
// 4 bits) per step:
//  * ldmatrix.x4 gives lane (g = lane/4, t = lane%4) word t of one chunk of
//    rows g and g+8, for two chunks: 8 codes per word.
//  * One AND per code pair turns a word into fp16 values q * 2^-24 (codes 0/4)
//    and 16q * 2^-24 (codes 1/5), and with one shift codes 2/6 and 3/7: fp16
//    subnormals whose products with fp16 x are exact in the fp32 accumulator.
//    These are the MMA's A fragments, so no dequantized weight exists anywhere.
//  * The MMA's B operand is x, permuted to the pair order above and with the
//    x of the 16q codes divided by 16, written once per problem into shared
//    memory with the group sums of x.
//  * Lane group g works on group u ^ g of its slice at step u (u mod ks when
//    the slice is not a multiple of 8 groups), so the eight rows one ldmatrix
//    phase reads start in eight different 16-byte bank slots, and B column g
//    holds exactly the x of lane group g's group: the results sit on the
//    diagonal D[g][g], D[g+8][g], in lane (g, g/2).
//  * Per step and row the holder lane adds s * 2^24 * D + b * sum(x) of that
//    group in fp32; rows split over KW warps meet in shared memory.
//
// The four-column consumer (COLS4; K a multiple of 256) keeps every lane's
// results: one MMA covers 16 rows of FOUR groups of a block.  K-pair t of the
// MMA (A registers a0/a1 for the first code pair, a2/a3 for the second) holds
// the codes of block group t, so lane (g, t) reads rows g and g+8 of group t;
// B column j holds the x of group j in its own two k-pairs (j and j + 4) and
// zero elsewhere, so D[r][j] is row r's dot product with group j, for all 16
// rows and the four columns at once.  Only the lanes (j, j) supply x; the
// others pass zeros.  Sixteen MMAs cover a block (64 codes of each group); the
// epilogue then applies each (row, group)'s scale and bias once per block.
#pragma once
#include "qgemv_impl.cuh"

namespace bt {
namespace gemv {

constexpr int kMmaRows = 16;   // rows per tile (the MMA's M)

// The MMA and the shared-memory fragment loads are plain (non-volatile) asm,
// so the compiler may interleave two independent steps; their addresses derive
// from values passed through launder() after the wait or barrier that makes
// the data valid, so no load can be moved above it.
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
      : "r"(addr));
}
__device__ __forceinline__ uint4 lds128_nv(uint32_t a) {
  uint4 v;
  asm("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
  return v;
}
__device__ __forceinline__ uint16_t lds16_nv(uint32_t a) {
  uint16_t v;
  asm("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ float lds32f_nv(uint32_t a) {
  float v;
  asm("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(a));
  return v;
}
// A value the compiler must treat as produced here (volatile, memory clobber).
__device__ __forceinline__ uint32_t launder(uint32_t v) {
  uint32_t r;
  asm volatile("mov.b32 %0, %1;" : "=r"(r) : "r"(v) : "memory");
  return r;
}

// Shared-memory address of the permuted x of (group v, chunk c, lane slot t):
// 16 bytes, groups 192 bytes apart, so that lane groups on neighbouring groups
// read different bank halves.
constexpr int kXGroupBytes = 192;
// The four-token consumer's lanes read two neighbouring groups of one token in
// one phase: 160 bytes apart they fall in different bank slots.
constexpr int kXGroupBytes4 = 160;
__device__ __forceinline__ uint32_t xslot(uint32_t xs, int v, int c, int t, int gbytes = kXGroupBytes) {
  return xs + (uint32_t)(v * gbytes + c * 64 + t * 16);
}

// Permuted, prescaled x of one problem (K values) and its group sums, written
// by all consumer threads: slot (v, c, t) holds, for the 8 x values j = 0..7 at
// k = 64v + 32c + 8t + j, the pairs (x0, x4) (x1/16, x5/16) (x2, x6) (x3/16, x7/16)
// -- the B fragments of the two MMAs of that chunk.
__device__ __forceinline__ void prep_x(uint32_t xs, float* xsum, const uint16_t* x, int G, int ctid, int nthreads,
                                       int gbytes = kXGroupBytes) {
  const int lane = ctid & 31;
  for (int base = ctid - lane; base < G * 8; base += nthreads) {
    const int idx = base + lane;
    float part = 0.f;
    if (idx < G * 8) {
      const int v = idx >> 3, c = (idx >> 2) & 1, t = idx & 3;
      const uint4 raw = __ldg(reinterpret_cast<const uint4*>(x + (size_t)v * 64 + c * 32 + t * 8));
      const __half2 x01 = *reinterpret_cast<const __half2*>(&raw.x), x23 = *reinterpret_cast<const __half2*>(&raw.y);
      const __half2 x45 = *reinterpret_cast<const __half2*>(&raw.z), x67 = *reinterpret_cast<const __half2*>(&raw.w);
      const __half2 sixteenth = __float2half2_rn(0.0625f);
      const __half2 p04 = __lows2half2(x01, x45), p15 = __hmul2(__highs2half2(x01, x45), sixteenth);
      const __half2 p26 = __lows2half2(x23, x67), p37 = __hmul2(__highs2half2(x23, x67), sixteenth);
      uint4 o;
      o.x = *reinterpret_cast<const uint32_t*>(&p04);
      o.y = *reinterpret_cast<const uint32_t*>(&p15);
      o.z = *reinterpret_cast<const uint32_t*>(&p26);
      o.w = *reinterpret_cast<const uint32_t*>(&p37);
      asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(xslot(xs, v, c, t, gbytes)), "r"(o.x), "r"(o.y), "r"(o.z),
                   "r"(o.w)
                   : "memory");
      const float2 f01 = __half22float2(x01), f23 = __half22float2(x23), f45 = __half22float2(x45),
                   f67 = __half22float2(x67);
      part = ((f01.x + f01.y) + (f23.x + f23.y)) + ((f45.x + f45.y) + (f67.x + f67.y));
    }
    part += __shfl_xor_sync(0xffffffffu, part, 1);
    part += __shfl_xor_sync(0xffffffffu, part, 2);
    part += __shfl_xor_sync(0xffffffffu, part, 4);
    if (idx < G * 8 && (idx & 7) == 0) xsum[idx >> 3] = part;
  }
}

// Four fp16x2 A pairs of one word of 8 four-bit codes: (q0,q4) (q1,q5)*16
// (q2,q6) (q3,q7)*16 as subnormals q * 2^-24.
__device__ __forceinline__ void pairs_q4(uint32_t w, uint32_t (&p)[4]) {
  const uint32_t w8 = w >> 8;
  p[0] = w & 0x000F000Fu;
  p[1] = w & 0x00F000F0u;
  p[2] = w8 & 0x000F000Fu;
  p[3] = w8 & 0x00F000F0u;
}

__device__ __forceinline__ uint32_t u4_at(const uint4& v, int i) {
  return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
}
__device__ __forceinline__ uint32_t lds32_nv(uint32_t a) {
  uint32_t v;
  asm("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ float2 lds64f_nv(uint32_t a) {
  float2 v;
  asm("ld.shared.v2.f32 {%0,%1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(a));
  return v;
}
__device__ __forceinline__ float2 half2_bits_to_float2(uint32_t v) {
  return __half22float2(*reinterpret_cast<const __half2*>(&v));
}

template <int NW> struct MmaWarps {
  static constexpr int kThreads = (NW + 1) * 32;
};

template <int BITS, int NW, int CTAS, int UNROLL, bool BATCH, bool COLS4, int TOK = 1>
__global__ void __launch_bounds__(MmaWarps<NW>::kThreads, CTAS)
    qgemv_mma_kernel(const GemvParams p, const __grid_constant__ GemvBatch<BATCH ? kBatchCap : 1> batch) {
  static_assert(BITS == 4, "tensor-pipe GEMV: 4-bit codes");
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = p.stages;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)S * p.stage_bytes);
  uint64_t* empty = full + S;
  float* red = reinterpret_cast<float*>(empty + S);          // [row group][2][KW][16]: NW * 2 * 16 floats
  float* xsum = red + NW * 2 * kMmaRows;                      // [G] group sums of x
  uint8_t* xs_ptr = reinterpret_cast<uint8_t*>(xsum) + p.xsum_bytes;   // permuted x, 128 B per group
  __shared__ volatile int s_fail;

  long long u_begin, u_end;
  if constexpr (BATCH) {
    u_begin = unit_at_cost(p, batch, p.total_cost * blockIdx.x / gridDim.x);
    u_end = unit_at_cost(p, batch, p.total_cost * (blockIdx.x + 1) / gridDim.x);
  } else {
    u_begin = p.num_units * blockIdx.x / gridDim.x;
    u_end = p.num_units * (blockIdx.x + 1) / gridDim.x;
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) { mbar_init(&full[s], 33); mbar_init(&empty[s], NW); }
    s_fail = 0;
    fence_mbar_init();
  }
  __syncthreads();
  pdl_launch_dependents();
  if (u_begin >= u_end) return;

  if (warp == NW) {
    // ------------------------------------------------------------ producer
    if (!p.const_weights) pdl_wait();
    const uint64_t pol = l2_policy_evict_first();
    int prob, blk;
    first_unit<BATCH>(p, batch, u_begin, prob, blk);
    ProbView v = resolve<BATCH>(p, batch, nullptr, prob);
    int s = 0;
    uint32_t ph = 0;
    long long it = 0;
    bool ok = true;
    for (long long u = u_begin; u < u_end; ++u, ++it) {
      if (blk == v.units) { blk = 0; ++prob; v = resolve<BATCH>(p, batch, nullptr, prob); }
      if (it >= S) {
        bool w = true;
        if (lane == 0) w = mbar_wait(&empty[s], ph ^ 1u, p.timeout_ns, p.err);
        if (!__shfl_sync(0xffffffffu, (int)w, 0)) { ok = false; s_fail = 1; break; }
      }
      const int RB = v.rb, row_bytes = v.row_bytes, G = v.g;
      const int row0 = blk * RB;
      const int rows = min(RB, v.n - row0);
      const bool drop = p.drop_stage && blockIdx.x == 0 && it == 0;   // test hook: never fill this stage
      if (!drop) {
        if (unit_bulk(p, v, row0, rows)) {
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
          // the host plans only 16-byte aligned units; anything else is refused
          if (lane == 0) set_device_error(p.err, kErrBadArg);
          mbar_arrive(&full[s]);
          if (lane == 0) mbar_arrive(&full[s]);
        }
      }
      ++blk;
      if (++s == S) { s = 0; ph ^= 1u; }
    }
    if (!ok) {
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
  const int g = lane >> 2, tq = lane & 3;
  const bool holder = tq == (g >> 1);       // holds D[g][g] and D[g+8][g]
  const int ld_row = (lane & 7) + ((lane >> 3) & 1) * 8;   // tile row whose address this lane gives ldmatrix
  const int ld_g = lane & 7;                // lane group of that row
  const int ld_second = lane >> 4;          // 0: the row's first chunk of a group, 1: its second
  const uint32_t xs0 = smem_u32(xs_ptr), xsum0 = smem_u32(xsum);
  uint32_t xs = xs0, xsa = xsum0;   // laundered after each x re-staging
  int KW = 0, RW = 0, kw = 0, rg = 0;
  bool dead = false;
  int rbuf = 0;
  int prob, blk;
  first_unit<BATCH>(p, batch, u_begin, prob, blk);
  ProbView v;
  int cur_prob = -1;
  int tcount = 0;   // tiles of the current problem this CTA has passed
  int s = 0;
  uint32_t ph = 0;
  pdl_wait();   // x comes from the previous kernel
  for (long long u = u_begin; u < u_end; ++u) {
    if (cur_prob >= 0 && blk == v.units) { blk = 0; ++prob; }
    if (prob != cur_prob) {
      cur_prob = prob;
      v = resolve<BATCH>(p, batch, nullptr, prob);
      // every consumer has finished the previous problem's tiles: x can be replaced
      asm volatile("bar.sync 15, %0;" ::"r"(NW * 32) : "memory");
      if (v.kw < 1 || NW % v.kw) {   // never planned so; refuse rather than spin
        if (threadIdx.x == 0) set_device_error(p.err, kErrBadArg);
        return;
      }
      KW = v.kw;
      RW = NW / KW;
      kw = warp % KW;
      rg = warp / KW;
      rbuf = 0;
      tcount = 0;
      if (!dead) {
#pragma unroll
        for (int tk = 0; tk < TOK; ++tk)   // one staged x per token, tok_groups groups apart
          if (tk < p.tokens)
            prep_x(xs0 + (uint32_t)(tk * p.tok_groups * kXGroupBytes + (TOK == 8 ? (tk & 1) * 16 : 0)),
                   xsum + tk * p.tok_groups,
                   v.x + (size_t)tk * v.k, v.g, threadIdx.x, NW * 32, TOK == 4 ? kXGroupBytes4 : kXGroupBytes);
      }
      asm volatile("bar.sync 15, %0;" ::"r"(NW * 32) : "memory");
      xs = launder(xs0);
      xsa = launder(xsum0);
    }
    if (!dead && (s_fail || !mbar_wait(&full[s], ph, p.timeout_ns, p.err))) {
      dead = true;
      s_fail = 1;
    }
    dead = __any_sync(0xffffffffu, dead);   // warp-uniform: the MMAs and shuffles below need every lane
    const int RB = v.rb, row_bytes = v.row_bytes, G = v.g;
    const int row0 = blk * RB;
    const int rows = min(RB, v.n - row0);
    const uint32_t st = launder(smem_u32(smem + (size_t)s * p.stage_bytes));   // after the wait
    const uint32_t st_sc = st + RB * row_bytes, st_bi = st_sc + RB * G * 2;
    const int ntiles = (rows + kMmaRows - 1) / kMmaRows;
    // this warp's K slice: groups [gs0, gs0 + ks)
    const int KS = (G + KW - 1) / KW;
    const int gs0 = kw * KS;
    const int ks = max(0, min(KS, G - gs0));
    const size_t ybase = v.y0 + row0;
    // tiles t of this unit with (tcount + t) % RW == rg
    int t = (rg - tcount + RW * kMmaRows) & (RW - 1);   // RW = NW / KW is a power of two
    if constexpr (COLS4 && TOK == 8) {
      // Five to eight tokens (KW = 1): an MMA covers 16 rows of ONE group and
      // eight tokens.  K-pairs t and t + 4 of lane (g, t) hold words 2t and
      // 2t + 1 of the group (four MMAs: word 2t + w, first or second code pair
      // of each half-word pair), so the lane reads 8 bytes of rows g and g + 8;
      // B column c holds token c's x, supplied by lanes (c, *).  Lane (g, t)
      // holds tokens 2t and 2t + 1 for rows g and g + 8.
      const bool live = g < p.tokens;   // a lane supplying an empty token slot keeps zeros
      // odd tokens' x sits 16 bytes into each group slot: the two tokens of a
      // load phase then fall in different bank slots
      const uint32_t xlane = (uint32_t)(g * p.tok_groups * kXGroupBytes + (g & 1) * 16 + tq * 32);
      const uint32_t xs0t = (uint32_t)(2 * tq * p.tok_groups * 4), xs1t = xs0t + (uint32_t)(p.tok_groups * 4);
      uint4 xr[2] = {make_uint4(0u, 0u, 0u, 0u), make_uint4(0u, 0u, 0u, 0u)};
      for (; t < ntiles; t += RW) {
        const int r0 = t * kMmaRows;
        const int ra = min(r0 + g, rows - 1), rb = min(r0 + g + 8, rows - 1);
        float ds[4] = {0.f, 0.f, 0.f, 0.f}, bx[4] = {0.f, 0.f, 0.f, 0.f};   // (ra, 2t) (ra, 2t+1) (rb, 2t) (rb, 2t+1)
        if (!dead) {
          for (int gi = 0; gi < G; ++gi) {
            const uint32_t off = (uint32_t)(gi * 32 + tq * 8);
            uint32_t wa[2], wb[2];
            asm("ld.shared.v2.b32 {%0,%1}, [%2];" : "=r"(wa[0]), "=r"(wa[1]) : "r"(st + (uint32_t)(ra * row_bytes) + off));
            asm("ld.shared.v2.b32 {%0,%1}, [%2];" : "=r"(wb[0]), "=r"(wb[1]) : "r"(st + (uint32_t)(rb * row_bytes) + off));
            if (live) {
              xr[0] = lds128_nv(xs + xlane + (uint32_t)(gi * kXGroupBytes));
              xr[1] = lds128_nv(xs + xlane + (uint32_t)(gi * kXGroupBytes + 16));
            }
            float dc[2][4] = {};
#pragma unroll
            for (int w = 0; w < 2; ++w) {
              uint32_t pa[4], pb[4];
              pairs_q4(wa[w], pa);
              pairs_q4(wb[w], pb);
              const uint32_t a0[4] = {pa[0], pb[0], pa[1], pb[1]};
              mma16816(dc[0], a0, xr[w].x, xr[w].y);
              const uint32_t a1[4] = {pa[2], pb[2], pa[3], pb[3]};
              mma16816(dc[1], a1, xr[w].z, xr[w].w);
            }
            const uint32_t po_a = (uint32_t)((ra * G + gi) * 2), po_b = (uint32_t)((rb * G + gi) * 2);
            const float sa = to_f32<BT_F16>(lds16_nv(st_sc + po_a)), sb = to_f32<BT_F16>(lds16_nv(st_sc + po_b));
            const float ba = to_f32<BT_F16>(lds16_nv(st_bi + po_a)), bb = to_f32<BT_F16>(lds16_nv(st_bi + po_b));
            const float x0 = lds32f_nv(xsa + xs0t + (uint32_t)(gi * 4)), x1 = lds32f_nv(xsa + xs1t + (uint32_t)(gi * 4));
            ds[0] = fmaf(sa, dc[0][0] + dc[1][0], ds[0]);
            ds[1] = fmaf(sa, dc[0][1] + dc[1][1], ds[1]);
            ds[2] = fmaf(sb, dc[0][2] + dc[1][2], ds[2]);
            ds[3] = fmaf(sb, dc[0][3] + dc[1][3], ds[3]);
            bx[0] = fmaf(ba, x0, bx[0]);
            bx[1] = fmaf(ba, x1, bx[1]);
            bx[2] = fmaf(bb, x0, bx[2]);
            bx[3] = fmaf(bb, x1, bx[3]);
          }
        }
        const int ya = r0 + g, yb = r0 + g + 8;
        if (!dead) {
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const int tk = 2 * tq + j;
            if (tk < p.tokens) {
              const size_t yt = ybase + (size_t)tk * v.n;
              if (ya < rows) store_yv(p, v.y, yt + ya, fmaf(ds[j], 16777216.f, bx[j]));
              if (yb < rows) store_yv(p, v.y, yt + yb, fmaf(ds[2 + j], 16777216.f, bx[2 + j]));
            }
          }
        }
      }
      t = ntiles;
    } else if constexpr (COLS4 && TOK == 4) {
      // Four tokens (p.tokens = 3 or 4; KW = 1): an MMA covers 16 rows of TWO
      // groups.  K-pairs t and t + 4 of lane (g, t) hold half t % 2 of block
      // group t / 2 (its words 4 (t % 2) .. + 3; first and second code pair of a
      // word), so the lane reads 16 bytes of rows g and g + 8.  B column c
      // holds the x of token c / 2 and group c % 2 in the k-pairs of that group:
      // lanes (c, t) with t / 2 == c % 2 supply it.  Lane (g, t) then holds
      // token t's dot products with both groups for rows g and g + 8.
      const int nb2 = G >> 1;   // blocks of two groups
      const bool prov = (tq >> 1) == (g & 1) && (g >> 1) < p.tokens;
      const uint32_t xlane = (uint32_t)((g >> 1) * p.tok_groups * kXGroupBytes + (g & 1) * kXGroupBytes4 +
                                        (tq & 1) * 64);
      const uint32_t xsum_tok = (uint32_t)(tq * p.tok_groups * 4);
      uint4 xr[4];
#pragma unroll
      for (int w = 0; w < 4; ++w) xr[w] = make_uint4(0u, 0u, 0u, 0u);
      for (; t < ntiles; t += RW) {
        const int r0 = t * kMmaRows;
        const int ra = min(r0 + g, rows - 1), rb = min(r0 + g + 8, rows - 1);
        float dsa = 0.f, dsb = 0.f, bxa = 0.f, bxb = 0.f;   // token tq, rows ra and rb
        const uint32_t lo = (uint32_t)((tq >> 1) * 32 + (tq & 1) * 16);
        const uint32_t ca0 = st + (uint32_t)(ra * row_bytes) + lo, cb0 = st + (uint32_t)(rb * row_bytes) + lo;
        const uint32_t pa0 = (uint32_t)(ra * G * 2), pb0 = (uint32_t)(rb * G * 2);
        if (!dead) {
          for (int bi = 0; bi < nb2; ++bi) {
            const int grp = bi * 2;   // first group of the block
            const uint4 wa = lds128_nv(ca0 + (uint32_t)(grp * 32));
            const uint4 wb = lds128_nv(cb0 + (uint32_t)(grp * 32));
            if (prov) {
#pragma unroll
              for (int w = 0; w < 4; ++w) xr[w] = lds128_nv(xs + xlane + (uint32_t)(grp * kXGroupBytes4 + w * 16));
            }
            float dc[4][4] = {};
#pragma unroll
            for (int w = 0; w < 4; ++w) {
              uint32_t pa[4], pb[4];
              pairs_q4(u4_at(wa, w), pa);
              pairs_q4(u4_at(wb, w), pb);
              const uint32_t a0[4] = {pa[0], pb[0], pa[1], pb[1]};
              mma16816(dc[(w & 1) * 2], a0, xr[w].x, xr[w].y);
              const uint32_t a1[4] = {pa[2], pb[2], pa[3], pb[3]};
              mma16816(dc[(w & 1) * 2 + 1], a1, xr[w].z, xr[w].w);
            }
            // D[ra][2t], D[ra][2t+1], D[rb][2t], D[rb][2t+1]: token t, groups grp, grp + 1
            const uint32_t po_a = pa0 + (uint32_t)(grp * 2), po_b = pb0 + (uint32_t)(grp * 2);
            const float2 sa = half2_bits_to_float2(lds32_nv(st_sc + po_a));
            const float2 sb = half2_bits_to_float2(lds32_nv(st_sc + po_b));
            const float2 ba = half2_bits_to_float2(lds32_nv(st_bi + po_a));
            const float2 bb = half2_bits_to_float2(lds32_nv(st_bi + po_b));
            const float2 xsv = lds64f_nv(xsa + xsum_tok + (uint32_t)(grp * 4));
            float d[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) d[i] = (dc[0][i] + dc[1][i]) + (dc[2][i] + dc[3][i]);
            dsa = fmaf(sa.x, d[0], fmaf(sa.y, d[1], dsa));
            dsb = fmaf(sb.x, d[2], fmaf(sb.y, d[3], dsb));
            bxa = fmaf(ba.x, xsv.x, fmaf(ba.y, xsv.y, bxa));
            bxb = fmaf(bb.x, xsv.x, fmaf(bb.y, xsv.y, bxb));
          }
        }
        const int ya = r0 + g, yb = r0 + g + 8;
        if (!dead && tq < p.tokens) {
          const size_t yt = ybase + (size_t)tq * v.n;
          if (ya < rows) store_yv(p, v.y, yt + ya, fmaf(dsa, 16777216.f, bxa));
          if (yb < rows) store_yv(p, v.y, yt + yb, fmaf(dsb, 16777216.f, bxb));
        }
      }
      t = ntiles;
    } else if constexpr (COLS4) {
      // this warp's K slice in blocks of four groups: [kb0, kb0 + nb)
      const int B4 = G >> 2;
      const int KSB = (B4 + KW - 1) / KW;
      const int kb0 = kw * KSB;
      const int nb = max(0, min(KSB, B4 - kb0));
      // B column c holds the x of token c / 4 (TOK = 2; token 0 only for TOK = 1), group c % 4 of
      // the block: lanes (c, c % 4) supply it.  Lane (g, t) holds columns 2t, 2t + 1: token t / 2,
      // groups 2 (t % 2) and 2 (t % 2) + 1.
      const bool prov = TOK == 2 ? (g & 3) == tq : g == tq;
      const int tl = tq & 1;          // with TOK = 1, lanes t = 2, 3 mirror t = 0, 1 (results unused)
      const int tok = TOK == 2 ? (tq >> 1) : 0;
      const uint32_t xtok = TOK == 2 ? (uint32_t)((g >> 2) * p.tok_groups * kXGroupBytes) : 0u;
      const uint32_t xsum_tok = (uint32_t)(tok * p.tok_groups * 4);
      // x fragments: the lanes (j, j) load theirs per block; every other lane keeps zeros
      uint4 xr[8];
#pragma unroll
      for (int w = 0; w < 8; ++w) xr[w] = make_uint4(0u, 0u, 0u, 0u);
      for (; t < ntiles; t += RW) {
        const int r0 = t * kMmaRows;
        const int ra = min(r0 + g, rows - 1), rb = min(r0 + g + 8, rows - 1);
        float dsa = 0.f, dsb = 0.f, bxa = 0.f, bxb = 0.f;   // sum s*D and sum b*sum(x), rows ra and rb
        const uint32_t ca0 = st + (uint32_t)(ra * row_bytes + tq * 32), cb0 = st + (uint32_t)(rb * row_bytes + tq * 32);
        const uint32_t pa0 = (uint32_t)(ra * G * 2), pb0 = (uint32_t)(rb * G * 2);
        if (!dead) {
          for (int bi = 0; bi < nb; ++bi) {
            const int grp = (kb0 + bi) * 4;   // first group of the block
            const uint32_t ca = ca0 + (uint32_t)(grp * 32);
            const uint32_t cb = cb0 + (uint32_t)(grp * 32);
            const uint4 wa0 = lds128_nv(ca), wa1 = lds128_nv(ca + 16);
            const uint4 wb0 = lds128_nv(cb), wb1 = lds128_nv(cb + 16);
            const uint32_t xg = xs + xtok + (uint32_t)((grp + (g & 3)) * kXGroupBytes);   // inside the block for every lane
            if (prov) {
#pragma unroll
              for (int w = 0; w < 8; ++w) xr[w] = lds128_nv(xg + (uint32_t)(w * 16));
            }
            // four independent accumulator chains of four MMAs each
            float dc[4][4] = {};
#pragma unroll
            for (int w = 0; w < 8; ++w) {
              uint32_t pa[4], pb[4];
              pairs_q4(u4_at(w < 4 ? wa0 : wa1, w & 3), pa);   // row ra, group grp + t, word w
              pairs_q4(u4_at(w < 4 ? wb0 : wb1, w & 3), pb);   // row rb
              const uint32_t a0[4] = {pa[0], pb[0], pa[1], pb[1]};
              mma16816(dc[(w & 1) * 2], a0, xr[w].x, xr[w].y);
              const uint32_t a1[4] = {pa[2], pb[2], pa[3], pb[3]};
              mma16816(dc[(w & 1) * 2 + 1], a1, xr[w].z, xr[w].w);
            }
            float d0[4], d1[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              d0[i] = dc[0][i] + dc[1][i];
              d1[i] = dc[2][i] + dc[3][i];
            }
            // D[ra][2t], D[ra][2t+1], D[rb][2t], D[rb][2t+1]: groups gp, gp + 1
            const int gp = grp + 2 * tl;
            const uint32_t po_a = pa0 + (uint32_t)(gp * 2), po_b = pb0 + (uint32_t)(gp * 2);
            const float2 sa = half2_bits_to_float2(lds32_nv(st_sc + po_a));
            const float2 sb = half2_bits_to_float2(lds32_nv(st_sc + po_b));
            const float2 ba = half2_bits_to_float2(lds32_nv(st_bi + po_a));
            const float2 bb = half2_bits_to_float2(lds32_nv(st_bi + po_b));
            const float2 xsv = lds64f_nv(xsa + xsum_tok + (uint32_t)(gp * 4));
            dsa = fmaf(sa.x, d0[0] + d1[0], fmaf(sa.y, d0[1] + d1[1], dsa));
            dsb = fmaf(sb.x, d0[2] + d1[2], fmaf(sb.y, d0[3] + d1[3], dsb));
            bxa = fmaf(ba.x, xsv.x, fmaf(ba.y, xsv.y, bxa));
            bxb = fmaf(bb.x, xsv.x, fmaf(bb.y, xsv.y, bxb));
          }
        }
        float acc_a = fmaf(dsa, 16777216.f, bxa), acc_b = fmaf(dsb, 16777216.f, bxb);
        acc_a += __shfl_xor_sync(0xffffffffu, acc_a, 1);   // the two lanes of one token
        acc_b += __shfl_xor_sync(0xffffffffu, acc_b, 1);
        const bool holder4 = TOK == 2 ? (tq & 1) == 0 : tq == 0;
        const int ya = r0 + g, yb = r0 + g + 8;
        if (TOK == 2) {   // KW == 1 (planned so): each token's rows go out directly
          const size_t yt = ybase + (size_t)tok * v.n;
          if (!dead && holder4) {
            if (ya < rows) store_yv(p, v.y, yt + ya, acc_a);
            if (yb < rows) store_yv(p, v.y, yt + yb, acc_b);
          }
        } else if (KW == 1) {
          if (!dead && holder4) {
            if (ya < rows) store_yv(p, v.y, ybase + ya, acc_a);
            if (yb < rows) store_yv(p, v.y, ybase + yb, acc_b);
          }
        } else {
          float* rbp = red + (size_t)((rg * 2 + rbuf) * KW) * kMmaRows;   // [KW][16]
          if (holder4) {
            rbp[kw * kMmaRows + g] = acc_a;
            rbp[kw * kMmaRows + g + 8] = acc_b;
          }
          asm volatile("bar.sync %0, %1;" ::"r"(1 + rg), "r"(KW * 32) : "memory");
          if (!dead && kw == 0 && holder4) {
            float sa = 0.f, sb = 0.f;
            for (int j = 0; j < KW; ++j) {
              sa += rbp[j * kMmaRows + g];
              sb += rbp[j * kMmaRows + g + 8];
            }
            if (ya < rows) store_yv(p, v.y, ybase + ya, sa);
            if (yb < rows) store_yv(p, v.y, ybase + yb, sb);
          }
          rbuf ^= 1;
        }
      }
      t = ntiles;   // the diagonal consumer's loop below does nothing
    }
    for (; t < ntiles; t += RW) {
      const int r0 = t * kMmaRows;
      float acc_a = 0.f, acc_b = 0.f;   // rows r0 + g, r0 + g + 8 (meaningful on holder lanes)
      if (!dead && ks > 0) {
        const int lr = min(r0 + ld_row, rows - 1);
        const uint32_t ld_base = st + (uint32_t)(lr * row_bytes) + (uint32_t)(((ld_g >> 2) ^ ld_second) << 4) +
                                 (uint32_t)(gs0 * 32);
        const int ra = min(r0 + g, rows - 1), rb = min(r0 + g + 8, rows - 1);
        const uint32_t pbase = (uint32_t)(gs0 * 2);
        const uint32_t sc_a = st_sc + (uint32_t)(ra * G) * 2 + pbase, sc_b = st_sc + (uint32_t)(rb * G) * 2 + pbase;
        const uint32_t bi_a = st_bi + (uint32_t)(ra * G) * 2 + pbase, bi_b = st_bi + (uint32_t)(rb * G) * 2 + pbase;
        const int h = (g >> 2) & 1;       // chunk this lane group reads first
        const uint32_t x1 = xs + (uint32_t)(gs0 * kXGroupBytes + h * 64 + tq * 16);
        const uint32_t x2 = xs + (uint32_t)(gs0 * kXGroupBytes + (h ^ 1) * 64 + tq * 16);
        const uint32_t xsb = xsa + (uint32_t)(gs0 * 4);
        // One step: the slice's group vl for the ldmatrix row, vc for this lane
        // group (the same rotation seen from the two lane mappings).
        auto step = [&](int vl, int vc) {
          uint32_t r[4];
          ldmatrix_x4(ld_base + (uint32_t)(vl * 32), r);
          const uint4 b1 = lds128_nv(x1 + (uint32_t)(vc * kXGroupBytes));
          const uint4 b2 = lds128_nv(x2 + (uint32_t)(vc * kXGroupBytes));
          const uint32_t po = (uint32_t)(vc * 2);
          const uint16_t sa = lds16_nv(sc_a + po), sb = lds16_nv(sc_b + po);
          const uint16_t ba = lds16_nv(bi_a + po), bb = lds16_nv(bi_b + po);
          const float xsv = lds32f_nv(xsb + (uint32_t)(vc * 4));
          uint32_t pa[4], pb[4], pc[4], pd[4];
          pairs_q4(r[0], pa);   // row g, first chunk
          pairs_q4(r[1], pb);   // row g + 8, first chunk
          pairs_q4(r[2], pc);   // row g, second chunk
          pairs_q4(r[3], pd);   // row g + 8, second chunk
          float d[4] = {0.f, 0.f, 0.f, 0.f};
          const uint32_t a0[4] = {pa[0], pb[0], pa[1], pb[1]};
          mma16816(d, a0, b1.x, b1.y);
          const uint32_t a1[4] = {pa[2], pb[2], pa[3], pb[3]};
          mma16816(d, a1, b1.z, b1.w);
          const uint32_t a2[4] = {pc[0], pd[0], pc[1], pd[1]};
          mma16816(d, a2, b2.x, b2.y);
          const uint32_t a3[4] = {pc[2], pd[2], pc[3], pd[3]};
          mma16816(d, a3, b2.z, b2.w);
          const float da = (g & 1) ? d[1] : d[0], db = (g & 1) ? d[3] : d[2];
          acc_a = fmaf(to_f32<BT_F16>(sa) * 16777216.f, da, fmaf(to_f32<BT_F16>(ba), xsv, acc_a));
          acc_b = fmaf(to_f32<BT_F16>(sb) * 16777216.f, db, fmaf(to_f32<BT_F16>(bb), xsv, acc_b));
        };
        if ((ks & 7) == 0) {
          // step j visits group j ^ lane group: a permutation of every aligned block
          // of 8 groups, with the eight rows of an ldmatrix phase in eight bank slots
          if constexpr (UNROLL == 2) {
            for (int j = 0; j < ks; j += 2) {
              step(j ^ ld_g, j ^ g);
              step((j + 1) ^ ld_g, (j + 1) ^ g);
            }
          } else {
            for (int j = 0; j < ks; ++j) step(j ^ ld_g, j ^ g);
          }
        } else {
          int vl = ld_g % ks, vc = g % ks;
          for (int j = 0; j < ks; ++j) {
            step(vl, vc);
            if (++vl == ks) vl = 0;
            if (++vc == ks) vc = 0;
          }
        }
      }
      const int ya = r0 + g, yb = r0 + g + 8;
      if (KW == 1) {
        if (!dead && holder) {
          if (ya < rows) store_yv(p, v.y, ybase + ya, acc_a);
          if (yb < rows) store_yv(p, v.y, ybase + yb, acc_b);
        }
      } else {
        float* rbp = red + (size_t)((rg * 2 + rbuf) * KW) * kMmaRows;   // [KW][16]
        if (holder) {
          rbp[kw * kMmaRows + g] = acc_a;
          rbp[kw * kMmaRows + g + 8] = acc_b;
        }
        asm volatile("bar.sync %0, %1;" ::"r"(1 + rg), "r"(KW * 32) : "memory");
        if (!dead && kw == 0 && holder) {
          float sa = 0.f, sb = 0.f;
          for (int j = 0; j < KW; ++j) {
            sa += rbp[j * kMmaRows + g];
            sb += rbp[j * kMmaRows + g + 8];
          }
          if (ya < rows) store_yv(p, v.y, ybase + ya, sa);
          if (yb < rows) store_yv(p, v.y, ybase + yb, sb);
        }
        rbuf ^= 1;
      }
    }
    tcount += ntiles;
    __syncwarp();
    if (!dead && lane == 0) mbar_arrive(&empty[s]);
    ++blk;
    if (++s == S) { s = 0; ph ^= 1u; }
  }
}

template <int BITS, int NW, int CTAS, int UNROLL, bool BATCH, bool COLS4, int TOK = 1>
cudaError_t launch_mma_t(const GemvParams& p, const GemvBatch<kBatchCap>* batch, int grid, size_t smem,
                         cudaStream_t stream) {
  auto k = qgemv_mma_kernel<BITS, NW, CTAS, UNROLL, BATCH, COLS4, TOK>;
  static std::atomic<uint64_t> smem_raised{0};
  cudaError_t e = raise_smem_limit(reinterpret_cast<const void*>(k), smem_raised);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(MmaWarps<NW>::kThreads);
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

template <int BITS, int NW, int CTAS, int UNROLL, bool COLS4 = false>
cudaError_t launch_mma_shape(const GemvParams& p, const GemvPlan& pl, const GemvBatch<kBatchCap>* b,
                             cudaStream_t st) {
  if (b) return launch_mma_t<BITS, NW, CTAS, UNROLL, true, COLS4>(p, b, pl.grid, pl.smem, st);
  return launch_mma_t<BITS, NW, CTAS, UNROLL, false, COLS4>(p, nullptr, pl.grid, pl.smem, st);
}

template <int BITS>
cudaError_t launch_mma_bits(const GemvParams& p, const GemvPlan& pl, const GemvBatch<kBatchCap>* b,
                            cudaStream_t st) {
  if (pl.mma_cols4 && p.tokens >= 2) {   // several tokens per problem: the batched 8-warp shape only
    if (!b || pl.mma_nw != 8 || pl.mma_ctas != 1 || p.tokens > 8) return cudaErrorInvalidValue;
    if (p.tokens == 2) return launch_mma_t<BITS, 8, 1, 1, true, true, 2>(p, b, pl.grid, pl.smem, st);
    if (p.tokens <= 4) return launch_mma_t<BITS, 8, 1, 1, true, true, 4>(p, b, pl.grid, pl.smem, st);
    return launch_mma_t<BITS, 8, 1, 1, true, true, 8>(p, b, pl.grid, pl.smem, st);
  }
  if (pl.mma_cols4) {
    if (pl.mma_nw == 16) return launch_mma_shape<BITS, 16, 1, 1, true>(p, pl, b, st);
    if (pl.mma_ctas == 2) return launch_mma_shape<BITS, 8, 2, 1, true>(p, pl, b, st);
    return launch_mma_shape<BITS, 8, 1, 1, true>(p, pl, b, st);
  }
  if (pl.mma_nw == 16) return launch_mma_shape<BITS, 16, 1, 1>(p, pl, b, st);
  if (pl.mma_ctas == 2) return launch_mma_shape<BITS, 8, 2, 1>(p, pl, b, st);
  if (pl.mma_unroll == 1) return launch_mma_shape<BITS, 8, 1, 1>(p, pl, b, st);
  return launch_mma_shape<BITS, 8, 1, 2>(p, pl, b, st);
}

}  // namespace gemv
}  // namespace bt
