// Grouped SwiGLU expert FFN in fp32 on CUDA cores (dtype MOE_F32).
//
// TF32 tensor-core math rounds operands to 10 mantissa bits, which cannot
// meet a 1e-4 relative error bound on fp32 layers, so the fp32 path uses
// FMA.  Row r of the expert-sorted input belongs to the expert e with
// group_offsets[e] <= r < group_offsets[e+1] ("Moe dynamic redundancy"
// (MaxText pull request 4760), review of get_gmm_for_local_experts: a
// grouped matmul over ragged group_sizes).
//
// Tiles of 32 output columns x 32 rows; each thread accumulates 4 rows of
// one column, over k in ascending order.  For each k-slab, the slab of the
// input rows is staged in shared memory, then, for each group with rows in
// the tile (the rows are sorted, so those groups are consecutive; usually
// one or two), that group's expert's weight slab, with coalesced loads, and
// the rows of that group accumulate it.  A row's sum runs over k in the
// same order wherever its tile starts, so it gets the same bits.
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
  constexpr int kW1 = MODE == 0 ? 1 : 0;  // slot of the up weights
  __shared__ float sw[kW1 + 1][KS][BN];
  const int R = __ldg(off + E);
  const int tx = threadIdx.x, ty = threadIdx.y;
  const int n = blockIdx.x * BN + tx;
  for (int r0 = blockIdx.y * BR; r0 < R && r0 < rows_alloc;
       r0 += gridDim.y * BR) {
    float g[4] = {0, 0, 0, 0}, u[4] = {0, 0, 0, 0};
    int rr[4], gg[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      rr[q] = r0 + ty + 8 * q;
      gg[q] = rr[q] < R ? expert_of_row(off, E, rr[q]) : -1;
    }
    // the groups of the tile's rows: consecutive, as the rows are sorted
    const int gfirst = expert_of_row(off, E, r0);
    const int glast = expert_of_row(off, E, min(r0 + BR, R) - 1);
    for (int k0 = 0; k0 < K; k0 += KS) {
      const int kend = min(KS, K - k0);
      __syncthreads();
      for (int i = ty * BN + tx; i < BR * KS; i += 256) {
        const int rl = i / KS, kl = i % KS;
        const int r = r0 + rl, kk = k0 + kl;
        sa[rl][kl] = (r < R && kk < K)
                         ? __ldg(a + static_cast<long long>(r) * K + kk)
                         : 0.0f;
      }
      for (int grp = gfirst; grp <= glast; ++grp) {
        if (__ldg(off + grp + 1) == __ldg(off + grp)) continue;  // empty
        const int ex = group_expert ? max(__ldg(group_expert + grp), 0) : grp;
        if (grp != gfirst) __syncthreads();  // the previous group's readers
        for (int i = ty * BN + tx; i < KS * BN; i += 256) {
          const int kl = i / BN, nl = i % BN;
          const int kk = k0 + kl, nn = blockIdx.x * BN + nl;
          const bool in = kk < K && nn < N;
          const long long widx = (static_cast<long long>(ex) * K + kk) * N + nn;
          sw[0][kl][nl] = in ? __ldg(w0 + widx) : 0.0f;
          if (MODE == 0) sw[kW1][kl][nl] = in ? __ldg(w1 + widx) : 0.0f;
        }
        __syncthreads();
        if (n < N) {
#pragma unroll 8
          for (int kl = 0; kl < kend; ++kl) {
            const float w0v = sw[0][kl][tx];
            const float w1v = MODE == 0 ? sw[kW1][kl][tx] : 0.0f;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              if (gg[q] != grp) continue;
              const float av = sa[ty + 8 * q][kl];
              g[q] = fmaf(av, w0v, g[q]);
              if (MODE == 0) u[q] = fmaf(av, w1v, u[q]);
            }
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
