// CUDA-core dequant-GEMM tile: the small-M and fallback path for M > 1, dense
// and grouped by expert.  BaseRT pages, thetesserapress.com "What BaseRT does
// differently" (a GEMM for prefill, M > 1, that dequantizes in its inner loop).
//
// A CTA owns a [32 tokens x 64 weight rows] output tile.  Per K step of 64
// codes it stages the step's packed words of its 64 weight rows in shared
// memory with the (scale, bias) of each 32-code half (groups of 32, 64 or 128),
// dequantizes them there into fp32 (w = s*q + b, or the fp16 weight itself for
// bits = 16; never written to global memory), stages the matching x tile as
// fp32 and accumulates with fp32 FMA.  Grouped mode walks the device offsets to find
// which expert and which rows a CTA's token tile covers.
#include "bt_common.cuh"
#include "qgemm.cuh"

namespace bt {
namespace {

constexpr int TM = 32, TN = 64, TK = 64, NT = 256;

template <int BITS, bt_dtype XD, bt_dtype YD>
__global__ void __launch_bounds__(NT) qgemm_simt_kernel(const GemmParams p) {
  __shared__ float xs[TM][TK + 1];
  __shared__ float ws[TN][TK + 1];
  __shared__ uint32_t wwords[TN][2 * BITS + 1];
  __shared__ float wsb[TN][2][2];   // (scale, bias) of each 32-code half of the K step
  __shared__ int tile_info[3];   // expert, m0, m_end

  pdl_launch_dependents();
  pdl_wait();
  const int tid = threadIdx.x;
  const int n0 = blockIdx.x * TN;
  if (tid == 0) {
    int e = -1, m0 = 0, m1 = 0;
    const int tile = blockIdx.y;
    if (!p.offsets) {
      e = 0; m0 = tile * TM; m1 = min(m0 + TM, p.M);
      if (m0 >= p.M) e = -1;
    } else {
      int acc = 0;
      for (int ex = 0; ex < p.num_experts; ++ex) {
        const int lo = __ldg(p.offsets + ex), hi = __ldg(p.offsets + ex + 1);
        const int cnt = max(0, min(hi, p.M) - max(lo, 0));
        const int nt = (cnt + TM - 1) / TM;
        if (tile < acc + nt) { e = ex; m0 = max(lo, 0) + (tile - acc) * TM; m1 = min(m0 + TM, min(hi, p.M)); break; }
        acc += nt;
      }
    }
    tile_info[0] = e; tile_info[1] = m0; tile_info[2] = m1;
  }
  __syncthreads();
  const int e = tile_info[0], m0 = tile_info[1], m1 = tile_info[2];
  if (e < 0) return;

  const int row_words = p.K * BITS / 32;
  const int G = p.K / TK;                 // K steps of 64 codes
  const int GQ = p.K / p.group;           // quantization groups per row
  const int tx = tid % 64, ty = tid / 64;
  float acc[TM / 4];
#pragma unroll
  for (int i = 0; i < TM / 4; ++i) acc[i] = 0.f;
  const uint16_t* xb = static_cast<const uint16_t*>(p.x);

  for (int g = 0; g < G; ++g) {
    // stage x tile
    for (int i = tid; i < TM * TK; i += NT) {
      const int mi = i / TK, kk = i % TK;
      const int m = m0 + mi;
      float v = 0.f;
      if (m < m1) {
        const int xr = p.row_index ? __ldg(p.row_index + m) : m;
        v = to_f32<XD>(xb[(size_t)xr * p.K + (size_t)g * TK + kk]);
      }
      xs[mi][kk] = v;
    }
    // stage packed words, scale and bias of the group for the 64 weight rows
    for (int i = tid; i < TN * 2 * BITS; i += NT) {
      const int ni = i / (2 * BITS), wi = i % (2 * BITS);
      const int n = n0 + ni;
      wwords[ni][wi] = (n < p.N) ? __ldg(p.codes + ((size_t)e * p.N + n) * row_words + (size_t)g * 2 * BITS + wi) : 0u;
    }
    if constexpr (BITS != 16) {   // fp16 weights have no scale or bias
      if (tid < 2 * TN) {
        const int ni = tid >> 1, half = tid & 1;
        const int n = n0 + ni;
        const int gq = (g * TK + half * 32) / p.group;   // quantization group of this half of the step
        float s = 0.f, b = 0.f;
        if (n < p.N) {
          s = to_f32<BT_F16>(__ldg(p.scales + ((size_t)e * p.N + n) * GQ + gq));
          b = to_f32<BT_F16>(__ldg(p.biases + ((size_t)e * p.N + n) * GQ + gq));
        }
        wsb[ni][half][0] = s;
        wsb[ni][half][1] = b;
      }
    }
    __syncthreads();
    // dequantize into shared fp32
    for (int i = tid; i < TN * TK; i += NT) {
      const int ni = i / TK, j = i % TK;
      const int bit = j * BITS, wi = bit >> 5, off = bit & 31;
      uint32_t q = wwords[ni][wi] >> off;
      if (off + BITS > 32) q |= wwords[ni][wi + 1] << (32 - off);
      q &= (1u << BITS) - 1u;
      if constexpr (BITS == 16) ws[ni][j] = __half2float(__ushort_as_half((uint16_t)q));   // fp16 weight
      else ws[ni][j] = fmaf(wsb[ni][j >> 5][0], (float)q, wsb[ni][j >> 5][1]);
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < TK; ++kk) {
      const float wv = ws[tx][kk];
#pragma unroll
      for (int i = 0; i < TM / 4; ++i) acc[i] = fmaf(xs[ty + 4 * i][kk], wv, acc[i]);
    }
    __syncthreads();
  }
  const int n = n0 + tx;
  if (p.swiglu) {
    // gate row (even tx) and its up row (tx + 1: the next lane of the same warp)
#pragma unroll
    for (int i = 0; i < TM / 4; ++i) {
      const float up = __shfl_xor_sync(0xffffffffu, acc[i], 1);
      const int m = m0 + ty + 4 * i;
      if (!(tx & 1) && n < p.N && m < m1)
        store_out<YD>(p.y, (size_t)m * (p.N / 2) + (n >> 1), acc[i] / (1.f + expf(-acc[i])) * up);
    }
  } else if (n < p.N) {
#pragma unroll
    for (int i = 0; i < TM / 4; ++i) {
      const int m = m0 + ty + 4 * i;
      if (m < m1) store_out<YD>(p.y, (size_t)m * p.N + n, acc[i]);
    }
  }
}

template <int BITS, bt_dtype XD, bt_dtype YD>
cudaError_t launch_simt_t(const GemmParams& p, int tiles, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((p.N + TN - 1) / TN, tiles);
  cfg.blockDim = dim3(NT);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = opts().pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, qgemm_simt_kernel<BITS, XD, YD>, p);
}

template <bt_dtype XD, bt_dtype YD>
cudaError_t launch_simt_xy(const GemmParams& p, int bits, int tiles, cudaStream_t st) {
  switch (bits) {
    case 2: return launch_simt_t<2, XD, YD>(p, tiles, st);
    case 3: return launch_simt_t<3, XD, YD>(p, tiles, st);
    case 4: return launch_simt_t<4, XD, YD>(p, tiles, st);
    case 5: return launch_simt_t<5, XD, YD>(p, tiles, st);
    case 6: return launch_simt_t<6, XD, YD>(p, tiles, st);
    case 16: return launch_simt_t<16, XD, YD>(p, tiles, st);
    default: return launch_simt_t<8, XD, YD>(p, tiles, st);
  }
}

template <bt_dtype XD>
cudaError_t launch_simt_x(const GemmParams& p, int bits, bt_dtype yd, int tiles, cudaStream_t st) {
  switch (yd) {
    case BT_F32: return launch_simt_xy<XD, BT_F32>(p, bits, tiles, st);
    case BT_BF16: return launch_simt_xy<XD, BT_BF16>(p, bits, tiles, st);
    default: return launch_simt_xy<XD, BT_F16>(p, bits, tiles, st);
  }
}

}  // namespace

GemmGeometry plan_gemm_simt_geometry(int M, int N, int num_experts) {
  GemmGeometry g;
  long long tiles = (M + TM - 1) / TM;   // the same count as launch_gemm_simt
  if (num_experts > 0) tiles += std::min<long long>(num_experts, M);
  g.bn = TM;
  g.grid_x = (N + TN - 1) / TN;
  g.grid_y = (int)std::min<long long>(tiles, 1LL << 30);
  g.grid_z = 1;
  g.feasible = tiles <= 65535;
  return g;
}

cudaError_t launch_gemm_simt(const GemmParams& p, int bits, bt_dtype xd, bt_dtype yd, cudaStream_t st) {
  // token tiles: dense ceil(M/32); grouped at most ceil(M/32) + one partial tile per expert
  long long tiles = (p.M + TM - 1) / TM;
  if (p.offsets) tiles += std::min<long long>(p.num_experts, p.M);
  if (tiles == 0) return cudaSuccess;
  if (tiles > 65535) return cudaErrorInvalidConfiguration;
  if (xd == BT_F16) return launch_simt_x<BT_F16>(p, bits, yd, (int)tiles, st);
  return launch_simt_x<BT_BF16>(p, bits, yd, (int)tiles, st);
}

}  // namespace bt
