// Regrouping of the backward's rows for the weight-gradient GEMMs.
//
// The layer backward leaves every pass's rows in its own row range (one
// range per chunk of the fallback).  The weight gradient of expert e sums
// over its rows of every pass.  This copies x_sorted, dg, du, h and
// dy_sorted into one group-major layout: group g holds the rows of every
// range in range order, starts on a 16-row boundary, and its pad rows up to
// the next boundary are zero.  The weight-gradient GEMM then sees one row
// range per expert, and every block of it is a whole number of K=16 steps
// whose rows are either the group's own or zeros, so it issues no clearing
// stores of its own.
//
// Kernel 1 (one CTA): out_off[g] = exclusive scan of roundup16(rows of g).
// Kernel 2: one warp per destination row: find its group (binary search) and
// its source range, copy the five rows with 16-byte loads and stores, or
// write zeros for a pad row.  Given per-row combine weights, the output
// gradient rows are scaled by their weight on the way (the layer backward
// keeps them unscaled until here).  Algorithmic traffic: the rows of the five
// buffers read once and written once.
#include <cuda_bf16.h>

#include "internal.h"

namespace moe {
namespace {

constexpr int kRegroupThreads = 1024;

struct RegroupParams {
  const int32_t* off[kMaxRegroupSegments];  // [G+1] per range
  int base[kMaxRegroupSegments];            // first row of the range
  int n_seg;
  int G;
};

__device__ __forceinline__ int rows_of(const RegroupParams& p, int g) {
  int n = 0;
  for (int s = 0; s < p.n_seg; ++s)
    n += __ldg(p.off[s] + g + 1) - __ldg(p.off[s] + g);
  return n;
}

__global__ void __launch_bounds__(kRegroupThreads)
    regroup_offsets_kernel(RegroupParams p, int32_t* __restrict__ out_off) {
  __shared__ int wsum[kRegroupThreads / 32];
  const int g = threadIdx.x, lane = g & 31, w = g >> 5;
  const int v = g < p.G ? (rows_of(p, g) + 15) & ~15 : 0;
  int inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += n;
  }
  if (lane == 31) wsum[w] = inc;
  __syncthreads();
  if (w == 0) {
    int x = wsum[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += n;
    }
    wsum[lane] = x;  // inclusive over warps
  }
  __syncthreads();
  const int before = (w > 0 ? wsum[w - 1] : 0) + inc - v;
  if (g < p.G) out_off[g] = before;
  if (g == p.G - 1) out_off[p.G] = before + v;
}

__device__ __forceinline__ void copy_row(const uint4* __restrict__ src,
                                         uint4* __restrict__ dst, int n16,
                                         int lane, bool zero) {
  const uint4 z = make_uint4(0, 0, 0, 0);
  for (int c = lane; c < n16; c += 32) dst[c] = zero ? z : __ldg(src + c);
}

// dst = bf16(w * src) for one bf16 row (the combine backward's scaling of
// an output-gradient row by its combine weight).
__device__ __forceinline__ void scale_row_bf16(const uint4* __restrict__ src,
                                               uint4* __restrict__ dst,
                                               int n16, int lane, float w) {
  for (int c = lane; c < n16; c += 32) {
    const uint4 q = __ldg(src + c);
    const uint32_t in[4] = {q.x, q.y, q.z, q.w};
    uint32_t out[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __nv_bfloat162 pr = __floats2bfloat162_rn(
          w * __uint_as_float(in[i] << 16),
          w * __uint_as_float(in[i] & 0xffff0000u));
      out[i] = *reinterpret_cast<uint32_t*>(&pr);
    }
    dst[c] = make_uint4(out[0], out[1], out[2], out[3]);
  }
}

__global__ void __launch_bounds__(256) regroup_rows_kernel(
    RegroupParams p, const int32_t* __restrict__ out_off, const uint4* xs,
    const uint4* dg, const uint4* du, const uint4* h, const uint4* dys,
    uint4* xs2, uint4* dg2, uint4* du2, uint4* h2, uint4* dys2, int h16,
    int f16, const float* __restrict__ w_row) {
  const int lane = threadIdx.x & 31;
  const long long warp =
      (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const long long n_warps =
      (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  const int total = __ldg(out_off + p.G);
  for (long long d = warp; d < total; d += n_warps) {
    const int row = static_cast<int>(d);
    int lo = 0, hi = p.G - 1;  // largest g with out_off[g] <= row
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (__ldg(out_off + mid) <= row)
        lo = mid;
      else
        hi = mid - 1;
    }
    const int g = lo;
    int local = row - __ldg(out_off + g);
    int src = -1;
    for (int s = 0; s < p.n_seg; ++s) {
      const int a = __ldg(p.off[s] + g), n = __ldg(p.off[s] + g + 1) - a;
      if (local < n) {
        src = p.base[s] + a + local;
        break;
      }
      local -= n;
    }
    const bool zero = src < 0;  // a pad row
    const long long sr = zero ? 0 : src;
    copy_row(xs + sr * h16, xs2 + d * h16, h16, lane, zero);
    if (w_row != nullptr && !zero)
      scale_row_bf16(dys + sr * h16, dys2 + d * h16, h16, lane,
                     __ldg(w_row + sr));
    else
      copy_row(dys + sr * h16, dys2 + d * h16, h16, lane, zero);
    copy_row(dg + sr * f16, dg2 + d * f16, f16, lane, zero);
    copy_row(du + sr * f16, du2 + d * f16, f16, lane, zero);
    copy_row(h + sr * f16, h2 + d * f16, f16, lane, zero);
  }
}

}  // namespace

cudaError_t launch_regroup(const moe_config_t& c, int G,
                           const WgradSegment* seg, int n_seg,
                           int64_t rows_out, const void* xs,
                           const void* dg, const void* du, const void* h,
                           const void* dys, void* xs2, void* dg2, void* du2,
                           void* h2, void* dys2, int32_t* out_off,
                           cudaStream_t s, const float* w_row) {
  if (n_seg < 1 || n_seg > kMaxRegroupSegments || G < 1 ||
      G > kRegroupThreads || (w_row != nullptr && c.dtype != MOE_BF16))
    return cudaErrorInvalidValue;
  RegroupParams p{};
  for (int i = 0; i < n_seg; ++i) {
    p.off[i] = seg[i].group_offsets;
    p.base[i] = seg[i].first_row;
  }
  p.n_seg = n_seg;
  p.G = G;
  regroup_offsets_kernel<<<1, kRegroupThreads, 0, s>>>(p, out_off);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess ||
      (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount,
                                  dev)) != cudaSuccess)
    return e;
  const int eb = elem_bytes(c.dtype);
  const unsigned blocks = static_cast<unsigned>(
      std::min<int64_t>(static_cast<int64_t>(sms) * 8,
                        std::max<int64_t>(1, (rows_out + 7) / 8)));
  regroup_rows_kernel<<<blocks, 256, 0, s>>>(
      p, out_off, static_cast<const uint4*>(xs), static_cast<const uint4*>(dg),
      static_cast<const uint4*>(du), static_cast<const uint4*>(h),
      static_cast<const uint4*>(dys), static_cast<uint4*>(xs2),
      static_cast<uint4*>(dg2), static_cast<uint4*>(du2),
      static_cast<uint4*>(h2), static_cast<uint4*>(dys2), c.H * eb / 16,
      c.F * eb / 16, w_row);
  return cudaGetLastError();
}

}  // namespace moe
