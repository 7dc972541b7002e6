// Router logits: logits[t, e] = sum_h x[t, h] Wr[h, e] (+ offset[t, e]).
//
// "Support moe_dropless_fallback=layer on the ragged all-to-all MoE path"
// (MaxText pull request 5920), section How: the overflow check is computed
// from the router's top-k, i.e. downstream of the router's dense
// projection of the tokens onto the experts.  The product accumulates in
// float32 and the logits are float32, the input of moe_route.
//
// Three forms:
//  * bf16 layers with H % 64 == 0 and E % 128 == 0: the grouped tcgen05
//    GEMM (gmm_tc.cu, one group of T rows, 128-column float32 tiles),
//    because at the DeepSeek-V3 layer's size it is a 30 GFLOP contraction;
//    batches whose 128 x 128 tiles leave SMs idle split the reduction over
//    a cluster instead when that is faster (router_tc.cu);
//  * E <= 64 otherwise (the fp32 tiny layer, E = 16 of the small layer): a
//    CUDA-core kernel in which a warp takes a few tokens at a time and its
//    lanes stride over 16-byte words of their rows, each lane keeping the
//    partial sums of its tokens for every expert; Wr is staged in shared
//    memory as float32 in a layout with an odd stride, so that the 32
//    lanes hit 32 distinct banks; the partial sums are then reduced over
//    the warp with xor shuffles in a fixed order;
//  * everything else (E > 64 and no multiple of 128): a CUDA-core kernel
//    in which a CTA of 256 threads takes 16 tokens and 256 experts; x is
//    staged in shared memory 64 columns at a time, each thread accumulates
//    its expert's 16 logits over h in order, reading Wr rows coalesced
//    across the experts.
#include <cuda_bf16.h>

#include "internal.h"

namespace moe {
namespace {

constexpr int kTok = 16;   // tokens per CTA
constexpr int kCols = 256; // experts per CTA (one per thread)
constexpr int kHStep = 64; // x columns staged per round

__device__ __forceinline__ float load_as_f32(const float* p) { return *p; }
__device__ __forceinline__ float load_as_f32(const __nv_bfloat16* p) {
  return __bfloat162float(*p);
}

template <typename TX>
__global__ void __launch_bounds__(kCols) router_simt_kernel(
    const TX* __restrict__ x, const TX* __restrict__ wr,
    const float* __restrict__ offset, float* __restrict__ logits, int T,
    int H, int E) {
  __shared__ float xs[kTok][kHStep];
  const int t0 = blockIdx.x * kTok;
  const int e = blockIdx.y * kCols + threadIdx.x;
  float acc[kTok];
#pragma unroll
  for (int i = 0; i < kTok; ++i) acc[i] = 0.0f;
  for (int h0 = 0; h0 < H; h0 += kHStep) {
    const int hn = min(kHStep, H - h0);
    for (int i = threadIdx.x; i < kTok * kHStep; i += kCols) {
      const int r = i / kHStep, c = i - r * kHStep;
      const int t = t0 + r;
      xs[r][c] = (t < T && c < hn)
                     ? load_as_f32(x + static_cast<long long>(t) * H + h0 + c)
                     : 0.0f;
    }
    __syncthreads();
    if (e < E) {
      for (int c = 0; c < hn; ++c) {
        const float w = load_as_f32(wr + static_cast<long long>(h0 + c) * E + e);
#pragma unroll
        for (int i = 0; i < kTok; ++i) acc[i] = fmaf(xs[i][c], w, acc[i]);
      }
    }
    __syncthreads();
  }
  if (e >= E) return;
#pragma unroll
  for (int i = 0; i < kTok; ++i) {
    const int t = t0 + i;
    if (t >= T) break;
    const long long o = static_cast<long long>(t) * E + e;
    logits[o] = acc[i] + (offset ? offset[o] : 0.0f);
  }
}

constexpr int kWarpCta = 256;             // 8 warps
constexpr int kGroupUnroll = 4;           // row groups per lane in flight
constexpr int kWrSmem = 96 * 1024;        // bytes of staged Wr rows

// Staged Wr layout: rows in groups of V (the x elements of one 16-byte
// load); group g holds [e][j] = Wr[V g + j][e] (e < E, j < V) as float32 at
// g * gld, gld = V E + 1.  gld is odd, so the 32 lanes, each reading the
// same (e, j) of one of 32 consecutive groups, hit 32 distinct banks.
__host__ __device__ __forceinline__ int wr_gld(int E, int V) {
  return V * E + 1;
}

// Row groups staged per chunk: a multiple of 32 (a whole lane stride).
__host__ __device__ __forceinline__ int wr_groups(int E, int V) {
  return (kWrSmem / (4 * wr_gld(E, V))) & ~31;
}

__device__ __forceinline__ void unpack(const uint4& raw, float (&v)[8]) {
  const __nv_bfloat16* b = reinterpret_cast<const __nv_bfloat16*>(&raw);
#pragma unroll
  for (int j = 0; j < 8; ++j) v[j] = __bfloat162float(b[j]);
}

__device__ __forceinline__ void unpack(const uint4& raw, float (&v)[4]) {
  v[0] = __uint_as_float(raw.x);
  v[1] = __uint_as_float(raw.y);
  v[2] = __uint_as_float(raw.z);
  v[3] = __uint_as_float(raw.w);
}

// E <= 64 (H is a multiple of V = 16 / sizeof(TX) in a valid config, as
// rows are whole 16-byte words): a warp takes TPW tokens,
// lane l the row groups l, l + 32, ... of each staged chunk, one 16-byte
// load of x per token and group; each lane keeps TPW x EMAX partial sums,
// reduced over the warp with xor shuffles at the end.
template <typename TX, int EMAX>
__global__ void __launch_bounds__(kWarpCta) router_warp_kernel(
    const TX* __restrict__ x, const TX* __restrict__ wr,
    const float* __restrict__ offset, float* __restrict__ logits, int T,
    int H, int E) {
  constexpr int TPW = EMAX >= 32 ? 1 : 32 / EMAX;  // tokens per warp
  constexpr int V = 16 / sizeof(TX);
  extern __shared__ float ws[];                    // [groups][gld]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gld = wr_gld(E, V), groups = wr_groups(E, V);
  const int t0 = (blockIdx.x * (kWarpCta / 32) + warp) * TPW;
  float acc[TPW][EMAX];
#pragma unroll
  for (int i = 0; i < TPW; ++i)
#pragma unroll
    for (int e = 0; e < EMAX; ++e) acc[i][e] = 0.0f;
  for (int hc = 0; hc < H; hc += groups * V) {
    const int hn = min(groups * V, H - hc);  // a multiple of V
    __syncthreads();  // the previous chunk's readers are done
    // 16-byte loads of Wr (the chunk starts on a 16-byte boundary: Wr is
    // 16-byte aligned and hc is a multiple of 32 V rows); a tail of fewer
    // than V elements goes element by element
    const TX* wc = wr + static_cast<long long>(hc) * E;
    const int n = hn * E, nv = n / V;
    for (int q = threadIdx.x; q < nv; q += kWarpCta) {
      const uint4 raw = __ldg(reinterpret_cast<const uint4*>(wc) + q);
      float v[V];
      unpack(raw, v);
      int r = (q * V) / E, e = q * V - r * E;
#pragma unroll
      for (int u = 0; u < V; ++u) {
        ws[(r / V) * gld + e * V + r % V] = v[u];
        if (++e == E) {
          e = 0;
          ++r;
        }
      }
    }
    for (int q = nv * V + threadIdx.x; q < n; q += kWarpCta) {
      const int r = q / E, e = q - r * E;
      ws[(r / V) * gld + e * V + r % V] = load_as_f32(wc + q);
    }
    __syncthreads();
    const int gn = hn / V;
    for (int gb = lane; gb < gn; gb += 32 * kGroupUnroll) {
      float xv[kGroupUnroll][TPW][V];
#pragma unroll
      for (int u = 0; u < kGroupUnroll; ++u) {
        const int g = gb + 32 * u;
#pragma unroll
        for (int i = 0; i < TPW; ++i) {
          uint4 raw = make_uint4(0, 0, 0, 0);
          if (g < gn && t0 + i < T)
            raw = __ldg(reinterpret_cast<const uint4*>(
                x + static_cast<long long>(t0 + i) * H + hc + g * V));
          unpack(raw, xv[u][i]);
        }
      }
#pragma unroll
      for (int u = 0; u < kGroupUnroll; ++u) {
        const int g = gb + 32 * u;
        if (g < gn) {
          const float* w = ws + g * gld;
#pragma unroll
          for (int e = 0; e < EMAX; ++e) {
            if (e < E) {
#pragma unroll
              for (int j = 0; j < V; ++j) {
                const float we = w[e * V + j];
#pragma unroll
                for (int i = 0; i < TPW; ++i)
                  acc[i][e] = fmaf(xv[u][i][j], we, acc[i][e]);
              }
            }
          }
        }
      }
    }
  }
#pragma unroll
  for (int i = 0; i < TPW; ++i) {
    const int t = t0 + i;
#pragma unroll
    for (int e = 0; e < EMAX; ++e) {
      if (e >= E) break;
      float v = acc[i][e];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (t < T && lane == (e & 31)) {
        const long long q = static_cast<long long>(t) * E + e;
        logits[q] = v + (offset ? offset[q] : 0.0f);
      }
    }
  }
}

template <typename TX, int EMAX>
cudaError_t launch_warp(const moe_config_t& c, const void* x, const void* wr,
                        const float* offset, float* logits, cudaStream_t s) {
  constexpr int TPW = EMAX >= 32 ? 1 : 32 / EMAX;
  constexpr int V = 16 / sizeof(TX);
  constexpr int per_cta = (kWarpCta / 32) * TPW;
  const int grid = (c.T + per_cta - 1) / per_cta;
  const size_t smem =
      static_cast<size_t>(wr_groups(c.E, V)) * wr_gld(c.E, V) * 4;
  const cudaError_t err = cudaFuncSetAttribute(
      router_warp_kernel<TX, EMAX>,
      cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  router_warp_kernel<TX, EMAX><<<grid, kWarpCta, smem, s>>>(
      static_cast<const TX*>(x), static_cast<const TX*>(wr), offset, logits,
      c.T, c.H, c.E);
  return cudaGetLastError();
}

template <typename TX>
cudaError_t launch_warp_any(const moe_config_t& c, const void* x,
                            const void* wr, const float* offset,
                            float* logits, cudaStream_t s) {
  if (c.E <= 8) return launch_warp<TX, 8>(c, x, wr, offset, logits, s);
  if (c.E <= 16) return launch_warp<TX, 16>(c, x, wr, offset, logits, s);
  if (c.E <= 32) return launch_warp<TX, 32>(c, x, wr, offset, logits, s);
  return launch_warp<TX, 64>(c, x, wr, offset, logits, s);
}

}  // namespace

cudaError_t launch_router(const moe_config_t& c, const void* x,
                          const void* w_router, const float* offset,
                          float* logits, int32_t* status, cudaStream_t s) {
  if (c.T == 0) return cudaSuccess;
  if (router_tc_supported(c) && aligned16(logits) &&
      (offset == nullptr || aligned16(offset)))
    return launch_router_tc(c, x, w_router, offset, logits, status, s);
  // a valid config's rows of x are a whole number of 16-byte words
  if (c.E <= 64)
    return c.dtype == MOE_F32
               ? launch_warp_any<float>(c, x, w_router, offset, logits, s)
               : launch_warp_any<__nv_bfloat16>(c, x, w_router, offset,
                                                logits, s);
  const dim3 grid((c.T + kTok - 1) / kTok, (c.E + kCols - 1) / kCols);
  if (c.dtype == MOE_F32)
    router_simt_kernel<float><<<grid, kCols, 0, s>>>(
        static_cast<const float*>(x), static_cast<const float*>(w_router),
        offset, logits, c.T, c.H, c.E);
  else
    router_simt_kernel<__nv_bfloat16><<<grid, kCols, 0, s>>>(
        static_cast<const __nv_bfloat16*>(x),
        static_cast<const __nv_bfloat16*>(w_router), offset, logits, c.T,
        c.H, c.E);
  return cudaGetLastError();
}

}  // namespace moe

using namespace moe;

extern "C" moe_status_t moe_router_logits(const moe_config_t* cfg,
                                          const void* x, const void* w_router,
                                          const float* logit_offset,
                                          float* logits, int32_t* status_word,
                                          moe_stream_t stream) {
  const moe_status_t st = moe_validate_config(cfg);
  if (st != MOE_OK) return st;
  if (cfg->T == 0) return MOE_OK;
  if (x == nullptr || w_router == nullptr || logits == nullptr ||
      !aligned16(x) || !aligned16(w_router) ||
      (reinterpret_cast<uintptr_t>(logits) & 3u) != 0 ||
      (logit_offset != nullptr &&
       (reinterpret_cast<uintptr_t>(logit_offset) & 3u) != 0))
    return MOE_ERR_INVALID_ARG;
  const cudaError_t e = launch_router(*cfg, x, w_router, logit_offset, logits,
                                      status_word, stream);
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
