// Grouped SwiGLU expert FFN in fp32 on CUDA cores (dtype MOE_F32).
//
// TF32 tensor-core math rounds operands to 10 mantissa bits, which cannot
// meet a 1e-4 relative error bound on fp32 layers, so the fp32 path uses
// FMA.  Row r of the expert-sorted input belongs to the expert e with
// group_offsets[e] <= r < group_offsets[e+1] ("Moe dynamic redundancy"
// (MaxText pull request 4760), review of get_gmm_for_local_experts: a
// grouped matmul over ragged group_sizes).
//
// Tiles of 32 output columns x 32 rows: the weight tile of a k-slab is
// shared by the rows of one expert through shared memory, and each thread
// accumulates 4 rows of one column.  A tile that straddles two experts is
// split per row (each row reads its own expert's weights from L2).
#include "internal.h"

namespace moe {
namespace {

constexpr int BN = 32;   // columns per tile (threadIdx.x)
constexpr int BR = 32;   // rows per tile (8 threadIdx.y x 4)
constexpr int KS = 32;   // k-slab

__device__ __forceinline__ int expert_of_row(const int32_t* off, int E,
                                             int r) {
  // largest e in [0, E) with off[e] <= r
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(off + mid) <= r)
      lo = mid;
    else
      hi = mid - 1;
  }
  return lo;
}

// MODE 0: h = silu(x Wg) * (x Wu)  (N = F, K = H)
// MODE 1: y = h Wd                 (N = H, K = F)
template <int MODE>
__global__ void __launch_bounds__(256) gmm_f32_kernel(
    const float* __restrict__ a, const int32_t* __restrict__ off, int E,
    const int32_t* __restrict__ group_expert, int K, int N,
    const float* __restrict__ w0, const float* __restrict__ w1,
    float* __restrict__ out, int rows_alloc) {
  __shared__ float sa[BR][KS + 1];
  const int R = __ldg(off + E);
  const int tx = threadIdx.x, ty = threadIdx.y;
  const int n = blockIdx.x * BN + tx;
  for (int r0 = blockIdx.y * BR; r0 < R && r0 < rows_alloc;
       r0 += gridDim.y * BR) {
    float g[4] = {0, 0, 0, 0}, u[4] = {0, 0, 0, 0};
    int rr[4], ee[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      rr[q] = r0 + ty + 8 * q;
      const int g = rr[q] < R ? expert_of_row(off, E, rr[q]) : 0;
      ee[q] = group_expert ? max(__ldg(group_expert + g), 0) : g;
    }
    for (int k0 = 0; k0 < K; k0 += KS) {
      __syncthreads();
      for (int i = ty * BN + tx; i < BR * KS; i += 256) {
        const int rl = i / KS, kl = i % KS;
        const int r = r0 + rl, kk = k0 + kl;
        sa[rl][kl] = (r < R && kk < K)
                         ? __ldg(a + static_cast<long long>(r) * K + kk)
                         : 0.0f;
      }
      __syncthreads();
      if (n < N) {
        const int kend = min(KS, K - k0);
        for (int kl = 0; kl < kend; ++kl) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const long long widx =
                (static_cast<long long>(ee[q]) * K + k0 + kl) * N + n;
            const float av = sa[ty + 8 * q][kl];
            g[q] = fmaf(av, __ldg(w0 + widx), g[q]);
            if (MODE == 0) u[q] = fmaf(av, __ldg(w1 + widx), u[q]);
          }
        }
      }
    }
    if (n < N) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        if (rr[q] >= R) continue;
        float v = g[q];
        if (MODE == 0) v = g[q] / (1.0f + expf(-g[q])) * u[q];
        out[static_cast<long long>(rr[q]) * N + n] = v;
      }
    }
  }
}

}  // namespace

cudaError_t launch_gmm1_f32(const moe_config_t& c, const Groups& g,
                            const void* x_sorted,
                            const int32_t* group_offsets, const void* w_gate,
                            const void* w_up, void* h, cudaStream_t s) {
  const long long rows = static_cast<long long>(c.T) * c.k;
  if (rows == 0) return cudaSuccess;
  const dim3 block(BN, 8);
  const unsigned gy = static_cast<unsigned>(
      std::min<long long>((rows + BR - 1) / BR, 65535));
  const dim3 g1((c.F + BN - 1) / BN, gy);
  gmm_f32_kernel<0><<<g1, block, 0, s>>>(
      static_cast<const float*>(x_sorted), group_offsets, g.n, g.map, c.H,
      c.F, static_cast<const float*>(w_gate), static_cast<const float*>(w_up),
      static_cast<float*>(h), static_cast<int>(rows));
  return cudaGetLastError();
}

cudaError_t launch_gmm2_f32(const moe_config_t& c, const Groups& g,
                            const void* h, const int32_t* group_offsets,
                            const void* w_down, void* y_sorted,
                            cudaStream_t s) {
  const long long rows = static_cast<long long>(c.T) * c.k;
  if (rows == 0) return cudaSuccess;
  const dim3 block(BN, 8);
  const unsigned gy = static_cast<unsigned>(
      std::min<long long>((rows + BR - 1) / BR, 65535));
  const dim3 g2((c.H + BN - 1) / BN, gy);
  gmm_f32_kernel<1><<<g2, block, 0, s>>>(
      static_cast<const float*>(h), group_offsets, g.n, g.map, c.F, c.H,
      static_cast<const float*>(w_down), nullptr,
      static_cast<float*>(y_sorted), static_cast<int>(rows));
  return cudaGetLastError();
}

}  // namespace moe
