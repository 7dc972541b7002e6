// Backward pass: the bandwidth-bound steps (combine and route backward) and
// the fp32 (CUDA-core) grouped FFN backward.
//
// "Support moe_dropless_fallback=layer on the ragged all-to-all MoE path"
// (MaxText pull request 5920), section Tests: with the layer fallback the
// outputs and the gradients match the dropless model; section How: the
// fallback's backward recomputes one chunk at a time and accumulates the
// expert-weight gradients over chunks.
//
// combine backward, per routed row r = (t, j):
//   dy_sorted[r] = w[t,j] * dy[t],   dtopk_w[t,j] = <dy[t], y_sorted[r]>
// One CTA per token reads dy[t] once with 16-byte loads, writes the k
// scaled copies and reduces the k dot products in fp32 (fixed order: per
// thread over its column chunks, then a fixed tree), so the result is
// deterministic.
// route backward: w = softmax over all logits read at the chosen experts:
//   dlogits[e] = p_e * (dp_e - sum_j w_j dw_j),  dp_e = sum_j [idx_j=e] dw_j
// renorm (softmax over the k chosen): dlogits[idx_j] = w_j (dw_j - sum w dw).
#include <cuda_bf16.h>
#include <math.h>

#include "internal.h"

namespace moe {
namespace {

constexpr int kThreads = 128;

__device__ __forceinline__ void load8(const int4& q, float* f, bool bf16) {
  if (bf16) {
    const uint32_t u[4] = {static_cast<uint32_t>(q.x),
                           static_cast<uint32_t>(q.y),
                           static_cast<uint32_t>(q.z),
                           static_cast<uint32_t>(q.w)};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = __uint_as_float(u[i] << 16);
      f[2 * i + 1] = __uint_as_float(u[i] & 0xffff0000u);
    }
  } else {
    f[0] = __int_as_float(q.x);
    f[1] = __int_as_float(q.y);
    f[2] = __int_as_float(q.z);
    f[3] = __int_as_float(q.w);
  }
}

__device__ __forceinline__ int4 store8(const float* f, bool bf16) {
  if (bf16) {
    uint32_t u[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __nv_bfloat162 p = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
      u[i] = *reinterpret_cast<uint32_t*>(&p);
    }
    return make_int4(static_cast<int>(u[0]), static_cast<int>(u[1]),
                     static_cast<int>(u[2]), static_cast<int>(u[3]));
  }
  return make_int4(__float_as_int(f[0]), __float_as_int(f[1]),
                   __float_as_int(f[2]), __float_as_int(f[3]));
}

template <bool BF16, int KMAX>
__global__ void __launch_bounds__(kThreads) combine_backward_kernel(
    const int4* __restrict__ dy, const int4* __restrict__ ys,
    const int32_t* __restrict__ row_of, const float* __restrict__ topk_w,
    int k, int n16, int4* __restrict__ dys, float* __restrict__ dtopk_w) {
  constexpr int V = BF16 ? 8 : 4;
  __shared__ int rows[KMAX];
  __shared__ float wts[KMAX];
  __shared__ float red[kThreads / 32][KMAX];
  const int t = blockIdx.x, tid = threadIdx.x;
  if (tid < KMAX) {
    const bool on = tid < k;
    rows[tid] = on ? row_of[static_cast<long long>(t) * k + tid] : -1;
    wts[tid] = on ? topk_w[static_cast<long long>(t) * k + tid] : 0.0f;
  }
  __syncthreads();
  float dot[KMAX];
#pragma unroll
  for (int j = 0; j < KMAX; ++j) dot[j] = 0.0f;
  const int4* src = dy + static_cast<long long>(t) * n16;
  for (int c = tid; c < n16; c += kThreads) {
    float d[V];
    load8(__ldg(src + c), d, BF16);
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      const int r = rows[j];
      if (r < 0) continue;
      float y[V], o[V];
      load8(__ldg(ys + static_cast<long long>(r) * n16 + c), y, BF16);
#pragma unroll
      for (int i = 0; i < V; ++i) {
        dot[j] = fmaf(d[i], y[i], dot[j]);
        o[i] = wts[j] * d[i];
      }
      dys[static_cast<long long>(r) * n16 + c] = store8(o, BF16);
    }
  }
  const int lane = tid & 31, w = tid >> 5;
#pragma unroll
  for (int j = 0; j < KMAX; ++j) {
    float v = dot[j];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0) red[w][j] = v;
  }
  __syncthreads();
  if (tid < k) {
    float v = 0.0f;
#pragma unroll
    for (int q = 0; q < kThreads / 32; ++q) v += red[q][tid];
    dtopk_w[static_cast<long long>(t) * k + tid] = rows[tid] >= 0 ? v : 0.0f;
  }
}

template <int EPL>
__global__ void __launch_bounds__(256) route_backward_kernel(
    const float* __restrict__ logits, const int32_t* __restrict__ idx,
    const float* __restrict__ dw, int T, int E, int k, int renorm,
    float* __restrict__ dlogits) {
  const int lane = threadIdx.x & 31;
  const long long t = (static_cast<long long>(blockIdx.x) * blockDim.x +
                       threadIdx.x) >> 5;
  if (t >= T) return;
  const float* row = logits + t * static_cast<long long>(E);
  float* out = dlogits + t * static_cast<long long>(E);
  // this lane's slot j < k: chosen expert and its dw
  const int my_e = lane < k ? idx[t * k + lane] : -1;
  const float my_dw = lane < k ? dw[t * k + lane] : 0.0f;
  float v[EPL];
  float m = -INFINITY;
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = i * 32 + lane;
    float f = e < E ? __ldg(row + e) : -INFINITY;
    if (!isfinite(f)) f = -INFINITY;
    v[i] = f;
    m = fmaxf(m, f);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if (m == -INFINITY) {  // no finite logit: zero weights, zero gradient
#pragma unroll
    for (int i = 0; i < EPL; ++i)
      if (i * 32 + lane < E) out[i * 32 + lane] = 0.0f;
    return;
  }
  if (renorm) {
    // w_j over the chosen logits
    const float lj = my_e >= 0 ? __ldg(row + my_e) : -INFINITY;
    const float lc = isfinite(lj) ? lj : -INFINITY;
    float mk = lc;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
      mk = fmaxf(mk, __shfl_xor_sync(0xffffffffu, mk, o));
    const float ex = (my_e >= 0 && mk != -INFINITY) ? expf(lc - mk) : 0.0f;
    float den = ex;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
      den += __shfl_xor_sync(0xffffffffu, den, o);
    const float wj = den > 0.0f ? ex / den : 0.0f;
    float s = wj * my_dw;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
#pragma unroll
    for (int i = 0; i < EPL; ++i)
      if (i * 32 + lane < E) out[i * 32 + lane] = 0.0f;
    __syncwarp();
    if (my_e >= 0) out[my_e] += wj * (my_dw - s);
    return;
  }
  float part = 0.0f;
#pragma unroll
  for (int i = 0; i < EPL; ++i) part += expf(v[i] - m);
  float den = part;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
  // S = sum_j w_j dw_j with w_j = p at the chosen expert
  const float wj =
      my_e >= 0 ? expf((isfinite(__ldg(row + my_e)) ? __ldg(row + my_e)
                                                    : -INFINITY) - m) / den
                : 0.0f;
  float s = wj * my_dw;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = i * 32 + lane;
    float dp = 0.0f;
    for (int j = 0; j < k; ++j) {
      const int ej = __shfl_sync(0xffffffffu, my_e, j);
      const float dj = __shfl_sync(0xffffffffu, my_dw, j);
      if (ej == e) dp += dj;
    }
    if (e < E) out[e] = expf(v[i] - m) / den * (dp - s);
  }
}

// ------------------------------------------------- fp32 FFN backward ---
__device__ __forceinline__ int group_of_row(const int32_t* off, int G, int r) {
  int lo = 0, hi = G - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(off + mid) <= r)
      lo = mid;
    else
      hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ float silu_f(float z) {
  return z / (1.0f + expf(-z));
}

__device__ __forceinline__ float silu_grad_f(float z) {
  const float s = 1.0f / (1.0f + expf(-z));
  return s * (1.0f + z * (1.0f - s));
}

// g, u, h of every routed row (thread per (row, f)).
__global__ void gemm1_saved_f32(const float* __restrict__ xs,
                                const int32_t* __restrict__ off, int G,
                                const int32_t* __restrict__ gexp, int H, int F,
                                const float* __restrict__ wg,
                                const float* __restrict__ wu,
                                float* __restrict__ g, float* __restrict__ u,
                                float* __restrict__ h) {
  const int R = __ldg(off + G);
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x +
                      threadIdx.x;
  if (i >= static_cast<long long>(R) * F) return;
  const int r = static_cast<int>(i / F), f = static_cast<int>(i % F);
  const int grp = group_of_row(off, G, r);
  const int e = gexp ? max(__ldg(gexp + grp), 0) : grp;
  float a = 0.0f, b = 0.0f;
  for (int q = 0; q < H; ++q) {
    const float xv = __ldg(xs + static_cast<long long>(r) * H + q);
    const long long w = (static_cast<long long>(e) * H + q) * F + f;
    a = fmaf(xv, __ldg(wg + w), a);
    b = fmaf(xv, __ldg(wu + w), b);
  }
  g[i] = a;
  u[i] = b;
  h[i] = silu_f(a) * b;
}

// dg, du from dh = dy_sorted Wd^T (thread per (row, f)).
__global__ void dgrad2_swiglu_f32(const float* __restrict__ dys,
                                  const int32_t* __restrict__ off, int G,
                                  const int32_t* __restrict__ gexp, int H,
                                  int F, const float* __restrict__ wd,
                                  const float* __restrict__ g,
                                  const float* __restrict__ u,
                                  float* __restrict__ dg,
                                  float* __restrict__ du) {
  const int R = __ldg(off + G);
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x +
                      threadIdx.x;
  if (i >= static_cast<long long>(R) * F) return;
  const int r = static_cast<int>(i / F), f = static_cast<int>(i % F);
  const int grp = group_of_row(off, G, r);
  const int e = gexp ? max(__ldg(gexp + grp), 0) : grp;
  float dh = 0.0f;
  for (int q = 0; q < H; ++q)
    dh = fmaf(__ldg(dys + static_cast<long long>(r) * H + q),
              __ldg(wd + (static_cast<long long>(e) * F + f) * H + q), dh);
  const float gv = g[i], uv = u[i];
  dg[i] = dh * uv * silu_grad_f(gv);
  du[i] = dh * silu_f(gv);
}

// dx_sorted = dg Wg^T + du Wu^T (thread per (row, h)).
__global__ void dgrad1_f32(const float* __restrict__ dg,
                           const float* __restrict__ du,
                           const int32_t* __restrict__ off, int G,
                           const int32_t* __restrict__ gexp, int H, int F,
                           const float* __restrict__ wg,
                           const float* __restrict__ wu,
                           float* __restrict__ dxs) {
  const int R = __ldg(off + G);
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x +
                      threadIdx.x;
  if (i >= static_cast<long long>(R) * H) return;
  const int r = static_cast<int>(i / H), hh = static_cast<int>(i % H);
  const int grp = group_of_row(off, G, r);
  const int e = gexp ? max(__ldg(gexp + grp), 0) : grp;
  float acc = 0.0f;
  for (int f = 0; f < F; ++f) {
    const long long w = (static_cast<long long>(e) * H + hh) * F + f;
    acc = fmaf(__ldg(dg + static_cast<long long>(r) * F + f), __ldg(wg + w),
               acc);
    acc = fmaf(__ldg(du + static_cast<long long>(r) * F + f), __ldg(wu + w),
               acc);
  }
  dxs[i] = acc;
}

// dW[e][a][b] (+)= sum_{rows of e} P[r][a] Q[r][b] (thread per (e, a, b)).
// Groups mapped to expert e (duplicates) all add into dW[e], in group order.
__global__ void wgrad_f32(const float* __restrict__ P, int A,
                          const float* __restrict__ Q, int Bn,
                          const int32_t* __restrict__ off, int G,
                          const int32_t* __restrict__ gexp, int E,
                          int accumulate, float* __restrict__ dw) {
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x +
                      threadIdx.x;
  if (i >= static_cast<long long>(E) * A * Bn) return;
  const int e = static_cast<int>(i / (static_cast<long long>(A) * Bn));
  const long long rem = i % (static_cast<long long>(A) * Bn);
  const int a = static_cast<int>(rem / Bn), b = static_cast<int>(rem % Bn);
  float acc = accumulate ? dw[i] : 0.0f;
  for (int grp = 0; grp < G; ++grp) {
    const int we = gexp ? __ldg(gexp + grp) : grp;
    if (we != e) continue;
    const int r0 = __ldg(off + grp), r1 = __ldg(off + grp + 1);
    for (int r = r0; r < r1; ++r)
      acc = fmaf(__ldg(P + static_cast<long long>(r) * A + a),
                 __ldg(Q + static_cast<long long>(r) * Bn + b), acc);
  }
  dw[i] = acc;
}

unsigned blocks_for(long long n, int t) {
  return static_cast<unsigned>((n + t - 1) / t);
}

// The layer backward's form of the combine backward: each kept row gets its
// token's output gradient unscaled, dy_rows[r] = dy[t], and its combine
// weight w_row[r] = topk_w[t, j]; the weight is applied later (to dh in the
// down-projection dgrad, to the rows of dWd in the regroup), so that the
// dgrad GEMM yields dh_u = dy[t] Wd^T, whose dot with h is the weight's
// gradient dy[t] . (h Wd) without recomputing y_sorted.  One CTA per token.
__global__ void __launch_bounds__(kThreads) gather_dy_rows_kernel(
    const int4* __restrict__ dy, const int32_t* __restrict__ row_of,
    const float* __restrict__ topk_w, int k, int n16,
    int4* __restrict__ dy_rows, float* __restrict__ w_row) {
  const long long t = blockIdx.x;
  const int4* src = dy + t * n16;
  for (int j = 0; j < k; ++j) {
    const int r = __ldg(row_of + t * k + j);
    if (r < 0) continue;
    if (threadIdx.x == 0) w_row[r] = __ldg(topk_w + t * k + j);
    int4* dst = dy_rows + static_cast<long long>(r) * n16;
    for (int c = threadIdx.x; c < n16; c += kThreads) dst[c] = __ldg(src + c);
  }
}

// dtopk_w[t, j] = sum over the dgrad's column tiles q (in order) of
// row_dot[r * n_parts + q] for the kept row r of pick (t, j); 0 if dropped.
__global__ void dtopk_from_row_dots_kernel(const int32_t* __restrict__ row_of,
                                           const float* __restrict__ row_dot,
                                           int n_parts, long long n,
                                           float* __restrict__ dtopk_w) {
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x +
                      threadIdx.x;
  if (i >= n) return;
  const int r = __ldg(row_of + i);
  float v = 0.0f;
  if (r >= 0) {
    const float* d = row_dot + static_cast<long long>(r) * n_parts;
    for (int q = 0; q < n_parts; ++q) v += __ldg(d + q);
  }
  dtopk_w[i] = v;
}

}  // namespace

cudaError_t launch_gather_dy_rows(const moe_config_t& c, const void* dy,
                                  const int32_t* row_of, const float* topk_w,
                                  void* dy_rows, float* w_row,
                                  cudaStream_t s) {
  if (c.T == 0) return cudaSuccess;
  gather_dy_rows_kernel<<<c.T, kThreads, 0, s>>>(
      static_cast<const int4*>(dy), row_of, topk_w, c.k,
      c.H * elem_bytes(c.dtype) / 16, static_cast<int4*>(dy_rows), w_row);
  return cudaGetLastError();
}

cudaError_t launch_dtopk_from_row_dots(const moe_config_t& c,
                                       const int32_t* row_of,
                                       const float* row_dot, int n_parts,
                                       float* dtopk_w, cudaStream_t s) {
  const long long n = static_cast<long long>(c.T) * c.k;
  if (n == 0) return cudaSuccess;
  dtopk_from_row_dots_kernel<<<blocks_for(n, 256), 256, 0, s>>>(
      row_of, row_dot, n_parts, n, dtopk_w);
  return cudaGetLastError();
}

cudaError_t launch_combine_backward(const moe_config_t& c, const void* dy,
                                    const void* y_sorted,
                                    const int32_t* row_of,
                                    const float* topk_w, void* dy_sorted,
                                    float* dtopk_w, cudaStream_t s) {
  if (c.T == 0) return cudaSuccess;
  const bool bf = c.dtype == MOE_BF16;
  const int n16 = c.H * elem_bytes(c.dtype) / 16;
  const int4* a = static_cast<const int4*>(dy);
  const int4* b = static_cast<const int4*>(y_sorted);
  int4* o = static_cast<int4*>(dy_sorted);
#define MOE_CB_CASE(KM)                                                     \
  if (c.k <= KM) {                                                          \
    if (bf)                                                                 \
      combine_backward_kernel<true, KM><<<c.T, kThreads, 0, s>>>(           \
          a, b, row_of, topk_w, c.k, n16, o, dtopk_w);                      \
    else                                                                    \
      combine_backward_kernel<false, KM><<<c.T, kThreads, 0, s>>>(          \
          a, b, row_of, topk_w, c.k, n16, o, dtopk_w);                      \
    return cudaGetLastError();                                              \
  }
  MOE_CB_CASE(1)
  MOE_CB_CASE(2)
  MOE_CB_CASE(4)
  MOE_CB_CASE(8)
  MOE_CB_CASE(16)
  MOE_CB_CASE(32)
#undef MOE_CB_CASE
  return cudaErrorInvalidValue;
}

cudaError_t launch_route_backward(const moe_config_t& c, const float* logits,
                                  const int32_t* topk_idx,
                                  const float* dtopk_w, float* dlogits,
                                  cudaStream_t s) {
  if (c.T == 0) return cudaSuccess;
  const unsigned blocks = blocks_for(static_cast<long long>(c.T) * 32, 256);
  const int epl = (c.E + 31) / 32;
#define MOE_RB_CASE(N)                                                       \
  if (epl <= N) {                                                            \
    route_backward_kernel<N><<<blocks, 256, 0, s>>>(                         \
        logits, topk_idx, dtopk_w, c.T, c.E, c.k, c.renorm, dlogits);        \
    return cudaGetLastError();                                               \
  }
  MOE_RB_CASE(1)
  MOE_RB_CASE(2)
  MOE_RB_CASE(4)
  MOE_RB_CASE(8)
  MOE_RB_CASE(16)
  MOE_RB_CASE(32)
#undef MOE_RB_CASE
  return cudaErrorInvalidValue;
}

cudaError_t launch_gmm_saved_f32(const moe_config_t& c, const Groups& g,
                                 const void* xs, const int32_t* off,
                                 const void* wg, const void* wu, void* gbuf,
                                 void* ubuf, void* h, cudaStream_t s) {
  const long long n = static_cast<long long>(c.T) * c.k * c.F;
  if (n == 0) return cudaSuccess;
  gemm1_saved_f32<<<blocks_for(n, 256), 256, 0, s>>>(
      static_cast<const float*>(xs), off, g.n, g.map, c.H, c.F,
      static_cast<const float*>(wg), static_cast<const float*>(wu),
      static_cast<float*>(gbuf), static_cast<float*>(ubuf),
      static_cast<float*>(h));
  return cudaGetLastError();
}

cudaError_t launch_down_dgrad_f32(const moe_config_t& c, const Groups& g,
                                  const int32_t* off, const void* wd,
                                  const void* gbuf, const void* ubuf,
                                  const void* dys, void* dg, void* du,
                                  cudaStream_t s) {
  const long long rows = static_cast<long long>(c.T) * c.k;
  if (rows == 0) return cudaSuccess;
  dgrad2_swiglu_f32<<<blocks_for(rows * c.F, 256), 256, 0, s>>>(
      static_cast<const float*>(dys), off, g.n, g.map, c.H, c.F,
      static_cast<const float*>(wd), static_cast<const float*>(gbuf),
      static_cast<const float*>(ubuf), static_cast<float*>(dg),
      static_cast<float*>(du));
  return cudaGetLastError();
}

cudaError_t launch_gate_up_dgrad_f32(const moe_config_t& c, const Groups& g,
                                     const int32_t* off, const void* wg,
                                     const void* wu, const void* dg,
                                     const void* du, void* dxs,
                                     cudaStream_t s) {
  const long long rows = static_cast<long long>(c.T) * c.k;
  if (rows == 0) return cudaSuccess;
  dgrad1_f32<<<blocks_for(rows * c.H, 256), 256, 0, s>>>(
      static_cast<const float*>(dg), static_cast<const float*>(du), off, g.n,
      g.map, c.H, c.F, static_cast<const float*>(wg),
      static_cast<const float*>(wu), static_cast<float*>(dxs));
  return cudaGetLastError();
}

cudaError_t launch_wgrad_f32(const moe_config_t& c, const Groups& g,
                             const WgradSegment* seg, int n_seg,
                             const void* xs, const void* dg, const void* du,
                             const void* h, const void* dys, float* dwg,
                             float* dwu, float* dwd, int flags,
                             int parts, cudaStream_t s) {
  const bool accumulate = (flags & kWgradAccumulate) != 0;
  const long long nw = static_cast<long long>(c.E) * c.H * c.F;
  const bool gu = (parts & kWgradGateUp) != 0;
  const bool dn = (parts & kWgradDown) != 0;
  if (n_seg == 0 && !accumulate) {
    const size_t bytes = static_cast<size_t>(nw) * sizeof(float);
    cudaError_t e = cudaSuccess;
    if (gu) e = cudaMemsetAsync(dwg, 0, bytes, s);
    if (gu && e == cudaSuccess) e = cudaMemsetAsync(dwu, 0, bytes, s);
    if (dn && e == cudaSuccess) e = cudaMemsetAsync(dwd, 0, bytes, s);
    return e;
  }
  const float* X = static_cast<const float*>(xs);
  const float* DG = static_cast<const float*>(dg);
  const float* DU = static_cast<const float*>(du);
  const float* Hs = static_cast<const float*>(h);
  const float* DY = static_cast<const float*>(dys);
  for (int i = 0; i < n_seg; ++i) {
    const long long r0 = seg[i].first_row;
    const int acc = (accumulate || i > 0) ? 1 : 0;
    const int32_t* off = seg[i].group_offsets;
    if (dn)  // the buffers of a part left out may be null
      wgrad_f32<<<blocks_for(nw, 256), 256, 0, s>>>(
          Hs + r0 * c.F, c.F, DY + r0 * c.H, c.H, off, g.n, g.map, c.E, acc,
          dwd);
    if (gu) {
      const float* xr = X + r0 * c.H;
      wgrad_f32<<<blocks_for(nw, 256), 256, 0, s>>>(
          xr, c.H, DG + r0 * c.F, c.F, off, g.n, g.map, c.E, acc, dwg);
      wgrad_f32<<<blocks_for(nw, 256), 256, 0, s>>>(
          xr, c.H, DU + r0 * c.F, c.F, off, g.n, g.map, c.E, acc, dwu);
    }
  }
  return cudaGetLastError();
}

}  // namespace moe
