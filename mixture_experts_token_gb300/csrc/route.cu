// Router top-k and combine weights, one warp per token.
//
// "Support moe_dropless_fallback=layer on the ragged all-to-all MoE path"
// (MaxText pull request 5920), section How: the overflow check is computed
// from the router's top-k.  The pages do not fix the tie rule or the
// weights; here equal logits go to the lower expert index, and the weights
// are the softmax over all E logits read at the chosen experts (renorm = 0)
// or the softmax over the k chosen logits (renorm = 1).
//
// Each lane holds E/32 logits (lane-strided, so the loads are coalesced) as
// 64-bit keys: the float's order-preserving bit image in the high word and
// the complemented expert index in the low word.  The largest key is the
// largest logit, lowest index first; k rounds of a butterfly max pick the
// experts in rank order.  Keys are never 0, so 0 marks a taken slot.
#include <math.h>

#include "internal.h"

namespace moe {
namespace {

__device__ __forceinline__ uint32_t ordered_bits(float f) {
  uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float from_ordered_bits(uint32_t o) {
  uint32_t u = (o & 0x80000000u) ? (o & 0x7fffffffu) : ~o;
  return __uint_as_float(u);
}

__device__ __forceinline__ uint64_t make_key(float f, int e) {
  return (static_cast<uint64_t>(ordered_bits(f)) << 32) |
         static_cast<uint64_t>(0xffffffffu - static_cast<uint32_t>(e));
}

__device__ __forceinline__ uint64_t warp_max_u64(uint64_t v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    uint64_t w = __shfl_xor_sync(0xffffffffu, v, o);
    v = w > v ? w : v;
  }
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

template <int EPL>  // logits per lane, ceil(E / 32) rounded up to a template
__global__ void __launch_bounds__(256) route_kernel(
    const float* __restrict__ logits, int T, int E, int k, int renorm,
    int32_t* __restrict__ topk_idx, float* __restrict__ topk_w,
    int32_t* __restrict__ status) {
  const int lane = threadIdx.x & 31;
  const long long t = (static_cast<long long>(blockIdx.x) * blockDim.x +
                       threadIdx.x) >> 5;
  if (t >= T) return;
  const float* row = logits + t * static_cast<long long>(E);

  float v[EPL];
  uint64_t key[EPL];
  bool bad = false;
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = i * 32 + lane;
    if (e < E) {
      float f = __ldg(row + e);
      if (!isfinite(f)) {
        bad = true;
        f = -INFINITY;
      }
      if (f == 0.0f) f = 0.0f;  // -0 and +0 compare equal: one key
      v[i] = f;
      key[i] = make_key(f, e);
    } else {
      v[i] = -INFINITY;
      key[i] = 0;
    }
  }

  // k rounds of arg-max; lane j keeps the j-th pick.
  int my_e = 0;
  float my_v = -INFINITY;
  for (int j = 0; j < k; ++j) {
    uint64_t best = 0;
#pragma unroll
    for (int i = 0; i < EPL; ++i) best = key[i] > best ? key[i] : best;
    best = warp_max_u64(best);
    const int e = static_cast<int>(0xffffffffu - static_cast<uint32_t>(best));
#pragma unroll
    for (int i = 0; i < EPL; ++i)
      if (i * 32 + lane == e) key[i] = 0;
    if (lane == j) {
      my_e = e;
      my_v = from_ordered_bits(static_cast<uint32_t>(best >> 32));
    }
  }

  // The largest finite logit is the first pick's value when it is finite.
  const float m = __shfl_sync(0xffffffffu, my_v, 0);
  float w = 0.0f;
  if (m != -INFINITY) {
    float part = 0.0f;
    if (renorm) {
      part = (lane < k) ? expf(my_v - m) : 0.0f;
    } else {
#pragma unroll
      for (int i = 0; i < EPL; ++i) part += expf(v[i] - m);
    }
    const float denom = warp_sum(part);
    w = expf(my_v - m) / denom;
  }
  if (lane < k) {
    topk_idx[t * k + lane] = my_e;
    topk_w[t * k + lane] = w;
  }
  if (__any_sync(0xffffffffu, bad) && lane == 0 && status != nullptr)
    atomicOr(status, MOE_DEV_NONFINITE);
}

}  // namespace

cudaError_t launch_route(const moe_config_t& c, const float* logits,
                         int32_t* topk_idx, float* topk_w, int32_t* status,
                         cudaStream_t s) {
  if (c.T == 0) return cudaSuccess;
  const int threads = 256;
  const long long warps = c.T;
  const unsigned blocks =
      static_cast<unsigned>((warps * 32 + threads - 1) / threads);
  const int epl = (c.E + 31) / 32;
#define MOE_ROUTE_CASE(N)                                              \
  if (epl <= N) {                                                      \
    route_kernel<N><<<blocks, threads, 0, s>>>(logits, c.T, c.E, c.k,  \
                                               c.renorm, topk_idx,     \
                                               topk_w, status);        \
    return cudaGetLastError();                                         \
  }
  MOE_ROUTE_CASE(1)
  MOE_ROUTE_CASE(2)
  MOE_ROUTE_CASE(4)
  MOE_ROUTE_CASE(8)
  MOE_ROUTE_CASE(16)
  MOE_ROUTE_CASE(32)
#undef MOE_ROUTE_CASE
  return cudaErrorInvalidValue;
}

}  // namespace moe
