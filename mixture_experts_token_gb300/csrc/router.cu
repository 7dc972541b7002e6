// Router logits: logits[t, e] = sum_h x[t, h] Wr[h, e] (+ offset[t, e]).
//
// "Support moe_dropless_fallback=layer on the ragged all-to-all MoE path"
// (MaxText pull request 5920), section How: the overflow check is computed
// from the router's top-k, i.e. downstream of the router's dense
// projection of the tokens onto the experts.  The product accumulates in
// float32 and the logits are float32, the input of moe_route.
//
// Two forms:
//  * bf16 layers with H % 64 == 0 and E % 128 == 0: the grouped tcgen05
//    GEMM (gmm_tc.cu, one group of T rows, 128-column float32 tiles),
//    because at the DeepSeek-V3 layer's size it is a 30 GFLOP contraction;
//    batches whose 128 x 128 tiles leave SMs idle split the reduction over
//    a cluster instead when that is faster (router_tc.cu);
//  * everything else (the fp32 tiny layer, E = 16 of the small layer):
//    this CUDA-core kernel.  A CTA of 256 threads takes 16 tokens and 256
//    experts; x is staged in shared memory 64 columns at a time, each
//    thread accumulates its expert's 16 logits over h in order, reading Wr
//    rows coalesced across the experts.
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

}  // namespace

cudaError_t launch_router(const moe_config_t& c, const void* x,
                          const void* w_router, const float* offset,
                          float* logits, int32_t* status, cudaStream_t s) {
  if (c.T == 0) return cudaSuccess;
  if (router_tc_supported(c) && aligned16(logits) &&
      (offset == nullptr || aligned16(offset)))
    return launch_router_tc(c, x, w_router, offset, logits, status, s);
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
