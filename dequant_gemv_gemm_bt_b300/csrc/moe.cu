// Mixture-of-experts steps around the grouped expert product: routing (stable
// counting sort of (token, slot) pairs by expert), SwiGLU between the gate/up
// and down products, and the gate-weighted combine.  BaseRT pages,
// thetesserapress.com "Where the wins land, and where they don't" (the MoE
// prefill lead, credited to code paths that do not fork on which experts a
// token picked): the routing here is data (offsets and an index list), and the
// products run as one grouped launch.
#include "bt_common.cuh"
#include "moe.cuh"

namespace bt {
namespace {

constexpr int kRouteThreads = 1024;

// One CTA: histogram, exclusive scan, then a stable scatter that walks the
// pairs in order, 1024 at a time, one warp at a time within a chunk.
__global__ void __launch_bounds__(kRouteThreads) moe_route_kernel(const int32_t* ids, int pairs, int E, int top_k,
                                                                  int32_t* offsets, int32_t* pair_index,
                                                                  int32_t* pair_row, int32_t* pair_token,
                                                                  unsigned* err) {
  extern __shared__ int cursor[];   // [E]
  __shared__ int warp_tot[32];
  pdl_launch_dependents();
  pdl_wait();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int e = tid; e < E; e += blockDim.x) cursor[e] = 0;
  __syncthreads();
  for (int i = tid; i < pairs; i += blockDim.x) {
    const int e = __ldg(ids + i);
    if (e >= 0 && e < E) atomicAdd(&cursor[e], 1);
    else set_device_error(err, kErrBadArg);
  }
  __syncthreads();
  // exclusive scan of cursor[0..E) -> offsets; each thread owns a contiguous run
  const int per = (E + blockDim.x - 1) / blockDim.x;
  const int e0 = min(E, tid * per), e1 = min(E, e0 + per);
  int local = 0;
  for (int e = e0; e < e1; ++e) local += cursor[e];
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = warp_tot[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += v;
    }
    warp_tot[lane] = w;   // inclusive per-warp totals
  }
  __syncthreads();
  int run = (warp ? warp_tot[warp - 1] : 0) + incl - local;
  for (int e = e0; e < e1; ++e) {
    const int c = cursor[e];
    offsets[e] = run;
    cursor[e] = run;
    run += c;
  }
  if (tid == blockDim.x - 1) offsets[E] = run;
  __syncthreads();
  // stable scatter
  for (int base = 0; base < pairs; base += blockDim.x) {
    const int i = base + tid;
    const int e = (i < pairs) ? __ldg(ids + i) : -1;
    const bool valid = e >= 0 && e < E;
    for (int w = 0; w < 32; ++w) {
      if (warp == w) {
        const unsigned act = __ballot_sync(0xffffffffu, valid);
        const unsigned peers = __match_any_sync(0xffffffffu, valid ? e : -1) & act;
        const int rank = __popc(peers & ((1u << lane) - 1u));
        const int pos = valid ? cursor[e] + rank : -1;
        __syncwarp();
        if (valid) {
          pair_index[pos] = i;
          if (pair_token) pair_token[pos] = i / top_k;
          if (rank == 0) cursor[e] += __popc(peers);
        }
        if (i < pairs) pair_row[i] = pos;
      }
      __syncthreads();
    }
  }
}

template <bt_dtype ID, bt_dtype OD>
__global__ void swiglu_kernel(const void* in, int rows, int inter, void* out) {
  pdl_launch_dependents();
  pdl_wait();
  const long long total = (long long)rows * inter;
  for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
       idx += (long long)gridDim.x * blockDim.x) {
    const long long r = idx / inter, i = idx % inter;
    float g, u;
    if constexpr (ID == BT_F32) {
      g = static_cast<const float*>(in)[r * 2 * inter + i];
      u = static_cast<const float*>(in)[r * 2 * inter + inter + i];
    } else {
      g = to_f32<ID>(static_cast<const uint16_t*>(in)[r * 2 * inter + i]);
      u = to_f32<ID>(static_cast<const uint16_t*>(in)[r * 2 * inter + inter + i]);
    }
    const float h = g / (1.f + expf(-g)) * u;
    store_out<OD>(out, idx, h);
  }
}

template <bt_dtype YD, bt_dtype OD>
__global__ void combine_kernel(const void* yg, const float* gates, const int32_t* pair_row, int tokens,
                               int top_k, int hidden, void* out) {
  pdl_launch_dependents();
  pdl_wait();
  const int t = blockIdx.y;
  for (int h = blockIdx.x * blockDim.x + threadIdx.x; h < hidden; h += gridDim.x * blockDim.x) {
    float acc = 0.f;
    for (int s = 0; s < top_k; ++s) {
      const int r = __ldg(pair_row + (size_t)t * top_k + s);
      if (r < 0 || r >= tokens * top_k) continue;
      float v;
      if constexpr (YD == BT_F32) v = static_cast<const float*>(yg)[(size_t)r * hidden + h];
      else v = to_f32<YD>(static_cast<const uint16_t*>(yg)[(size_t)r * hidden + h]);
      acc = fmaf(__ldg(gates + (size_t)t * top_k + s), v, acc);
    }
    store_out<OD>(out, (size_t)t * hidden + h, acc);
  }
}

cudaLaunchConfig_t cfg_for(dim3 grid, dim3 block, size_t smem, cudaStream_t st, cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = opts().pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

template <bt_dtype ID>
cudaError_t swiglu_o(const void* in, int rows, int inter, void* out, bt_dtype od, cudaStream_t st) {
  cudaLaunchAttribute attr[1];
  const long long total = (long long)rows * inter;
  const int blocks = (int)std::min<long long>((total + 255) / 256, 4LL * sm_count());
  cudaLaunchConfig_t cfg = cfg_for(dim3(blocks), dim3(256), 0, st, attr);
  switch (od) {
    case BT_F32: return cudaLaunchKernelEx(&cfg, swiglu_kernel<ID, BT_F32>, in, rows, inter, out);
    case BT_BF16: return cudaLaunchKernelEx(&cfg, swiglu_kernel<ID, BT_BF16>, in, rows, inter, out);
    default: return cudaLaunchKernelEx(&cfg, swiglu_kernel<ID, BT_F16>, in, rows, inter, out);
  }
}

template <bt_dtype YD>
cudaError_t combine_o(const void* yg, const float* gates, const int32_t* pair_row, int tokens, int top_k,
                      int hidden, void* out, bt_dtype od, cudaStream_t st) {
  cudaLaunchAttribute attr[1];
  const int bx = std::max(1, std::min((hidden + 255) / 256, 16));
  cudaLaunchConfig_t cfg = cfg_for(dim3(bx, tokens), dim3(256), 0, st, attr);
  switch (od) {
    case BT_F32: return cudaLaunchKernelEx(&cfg, combine_kernel<YD, BT_F32>, yg, gates, pair_row, tokens, top_k, hidden, out);
    case BT_BF16: return cudaLaunchKernelEx(&cfg, combine_kernel<YD, BT_BF16>, yg, gates, pair_row, tokens, top_k, hidden, out);
    default: return cudaLaunchKernelEx(&cfg, combine_kernel<YD, BT_F16>, yg, gates, pair_row, tokens, top_k, hidden, out);
  }
}

}  // namespace

cudaError_t launch_moe_route(const int32_t* ids, int tokens, int top_k, int E, int32_t* offsets,
                             int32_t* pair_index, int32_t* pair_row, int32_t* pair_token, cudaStream_t st) {
  cudaLaunchAttribute attr[1];
  const size_t smem = (size_t)E * sizeof(int);
  static std::atomic<uint64_t> smem_raised{0};
  cudaError_t e = raise_smem_limit(reinterpret_cast<const void*>(moe_route_kernel), smem_raised);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = cfg_for(dim3(1), dim3(kRouteThreads), smem, st, attr);
  return cudaLaunchKernelEx(&cfg, moe_route_kernel, ids, tokens * top_k, E, top_k, offsets, pair_index, pair_row,
                            pair_token, device_error_word());
}

cudaError_t launch_swiglu(const void* in, bt_dtype id, int rows, int inter, void* out, bt_dtype od,
                          cudaStream_t st) {
  if ((long long)rows * inter == 0) return cudaSuccess;
  switch (id) {
    case BT_F32: return swiglu_o<BT_F32>(in, rows, inter, out, od, st);
    case BT_BF16: return swiglu_o<BT_BF16>(in, rows, inter, out, od, st);
    default: return swiglu_o<BT_F16>(in, rows, inter, out, od, st);
  }
}

cudaError_t launch_combine(const void* yg, bt_dtype yd, const float* gates, const int32_t* pair_row, int tokens,
                           int top_k, int hidden, void* out, bt_dtype od, cudaStream_t st) {
  if (tokens == 0) return cudaSuccess;
  switch (yd) {
    case BT_F32: return combine_o<BT_F32>(yg, gates, pair_row, tokens, top_k, hidden, out, od, st);
    case BT_BF16: return combine_o<BT_BF16>(yg, gates, pair_row, tokens, top_k, hidden, out, od, st);
    default: return combine_o<BT_F16>(yg, gates, pair_row, tokens, top_k, hidden, out, od, st);
  }
}

}  // namespace bt
