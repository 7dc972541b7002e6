// Weighted combine (unpermute): y[t] = sum_j w[t,j] * y_sorted[row_of[t,j]].
//
// "MoE ring-of-experts: TC Pallas ring all-gather for the combine backward +
// x_sorted remat save" (MaxText pull request 4969), section What: the
// combine reduces the expert outputs of a token back to one row (a
// psum_scatter across shards in the ring variant; a gather here, where all
// shards share one GPU).  Dropped rows (row_of = -1) contribute nothing.
//
// One CTA per token, or per (token, column slice) when there are too few
// tokens to keep every SM busy (a fallback chunk of 128 tokens, say): the
// row's 16-byte chunks are then split into `splits` contiguous slices, one
// CTA each, so that the k row loads of a token are spread over several SMs.
// Each thread owns a few 16-byte column chunks, issues
// the k row loads of a chunk back to back (the slot loop is unrolled to a
// compile-time bound so the loads overlap), accumulates in fp32 in slot
// order j = 0..k-1 (deterministic: no atomics), and stores once.
// Algorithmic traffic: R_kept*H*b read + T*H*b written.
// With null weights every kept row counts once: the permute's transpose,
// dx[t] = sum_j dx_sorted[row_of[t,j]], in the backward pass.
#include <cuda_bf16.h>

#include <algorithm>

#include "internal.h"

namespace moe {
namespace {

constexpr int kThreads = 128;
constexpr int kUnroll = 4;

template <typename T>
struct Vec;
template <>
struct Vec<float> {
  static constexpr int N = 4;
  __device__ static void load(const int4& q, float* f) {
    f[0] = __int_as_float(q.x);
    f[1] = __int_as_float(q.y);
    f[2] = __int_as_float(q.z);
    f[3] = __int_as_float(q.w);
  }
  __device__ static int4 store(const float* f) {
    return make_int4(__float_as_int(f[0]), __float_as_int(f[1]),
                     __float_as_int(f[2]), __float_as_int(f[3]));
  }
};
template <>
struct Vec<__nv_bfloat16> {
  static constexpr int N = 8;
  __device__ static void load(const int4& q, float* f) {
    const uint32_t u[4] = {static_cast<uint32_t>(q.x),
                           static_cast<uint32_t>(q.y),
                           static_cast<uint32_t>(q.z),
                           static_cast<uint32_t>(q.w)};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = __uint_as_float(u[i] << 16);
      f[2 * i + 1] = __uint_as_float(u[i] & 0xffff0000u);
    }
  }
  __device__ static int4 store(const float* f) {
    uint32_t u[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __nv_bfloat162 p = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
      u[i] = *reinterpret_cast<uint32_t*>(&p);
    }
    return make_int4(static_cast<int>(u[0]), static_cast<int>(u[1]),
                     static_cast<int>(u[2]), static_cast<int>(u[3]));
  }
};

template <typename T, int KMAX>
__global__ void __launch_bounds__(kThreads) combine_kernel(
    const int4* __restrict__ ys, const int32_t* __restrict__ row_of,
    const float* __restrict__ topk_w, int k, int n16, int per_split,
    int4* __restrict__ y) {
  using V = Vec<T>;
  __shared__ int rows[KMAX];
  __shared__ float wts[KMAX];
  const int t = blockIdx.x, tid = threadIdx.x;
  if (tid < KMAX) {
    const bool on = tid < k;
    rows[tid] = on ? row_of[static_cast<long long>(t) * k + tid] : -1;
    wts[tid] = !on ? 0.0f
                   : topk_w ? topk_w[static_cast<long long>(t) * k + tid]
                            : 1.0f;
  }
  __syncthreads();
  const int begin = blockIdx.y * per_split;
  const int end = min(n16, begin + per_split);
  for (int c0 = begin + tid; c0 < end; c0 += kThreads * kUnroll) {
    float acc[kUnroll][V::N];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u)
#pragma unroll
      for (int i = 0; i < V::N; ++i) acc[u][i] = 0.0f;
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      const int r = rows[j];
      if (r < 0) continue;
      const float w = wts[j];
      const int4* src = ys + static_cast<long long>(r) * n16;
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int c = c0 + u * kThreads;
        if (c < end) {
          float f[V::N];
          V::load(__ldg(src + c), f);
#pragma unroll
          for (int i = 0; i < V::N; ++i) acc[u][i] = fmaf(w, f[i], acc[u][i]);
        }
      }
    }
    int4* dst = y + static_cast<long long>(t) * n16;
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int c = c0 + u * kThreads;
      if (c < end) dst[c] = V::store(acc[u]);
    }
  }
}

// CTAs per token: enough that the grid holds about kCtasPerSm CTAs per SM,
// but no slice narrower than one pass of the CTA's threads.
constexpr int kCtasPerSm = 4;

int combine_splits(int T, int n16) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
          cudaSuccess)
    return 1;
  const int want = (kCtasPerSm * sms + T - 1) / T;
  return std::max(1, std::min(want, n16 / kThreads));
}

template <typename T>
cudaError_t launch_typed(const moe_config_t& c, const void* ys,
                         const int32_t* row_of, const float* w, void* y,
                         cudaStream_t s) {
  const int n16 = c.H * static_cast<int>(sizeof(T)) / 16;
  const int splits = combine_splits(c.T, n16);
  const int per = (n16 + splits - 1) / splits;
  const dim3 grid(static_cast<unsigned>(c.T), static_cast<unsigned>(splits));
  const int4* src = static_cast<const int4*>(ys);
  int4* dst = static_cast<int4*>(y);
#define MOE_COMBINE_CASE(KM)                                            \
  if (c.k <= KM) {                                                      \
    combine_kernel<T, KM><<<grid, kThreads, 0, s>>>(src, row_of, w, c.k, \
                                                    n16, per, dst);     \
    return cudaGetLastError();                                          \
  }
  MOE_COMBINE_CASE(1)
  MOE_COMBINE_CASE(2)
  MOE_COMBINE_CASE(4)
  MOE_COMBINE_CASE(8)
  MOE_COMBINE_CASE(16)
  MOE_COMBINE_CASE(32)
#undef MOE_COMBINE_CASE
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_combine(const moe_config_t& c, const void* y_sorted,
                           const int32_t* row_of, const float* topk_w,
                           void* y, cudaStream_t s) {
  if (c.T == 0) return cudaSuccess;
  if (c.dtype == MOE_F32)
    return launch_typed<float>(c, y_sorted, row_of, topk_w, y, s);
  return launch_typed<__nv_bfloat16>(c, y_sorted, row_of, topk_w, y, s);
}

}  // namespace moe
