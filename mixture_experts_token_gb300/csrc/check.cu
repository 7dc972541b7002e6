// Per-expert and per-shard counts and the ragged receive-buffer overflow
// check.
//
// "Support moe_dropless_fallback=layer on the ragged all-to-all MoE path"
// (MaxText pull request 5920): section Why fixes the cap (factor x balanced
// per shard; -1 = no cap), section How the check (does any expert-parallel
// shard receive more than its buffer, computed from the router's top-k).
// "Moe dynamic redundancy" (MaxText pull request 4760), review comments:
// per-expert group_sizes, experts_per_rank consecutive experts per shard.
//
// The capacity is an integer computed on the host (capacity_rows()); the
// kernel counts with shared-memory atomics (order-free for integers), scans
// the E counts with one block-wide scan, and takes shard sums as differences
// of the scan.  A single CTA covers T*k indices: the check reads 4 bytes per
// routed row, a negligible cost next to the permute and the GEMM.
#include "internal.h"

namespace moe {
namespace {

constexpr int kCheckThreads = 1024;

// Exclusive block scan of one int per thread (blockDim.x == 1024).
__device__ int block_exclusive_scan(int v, int* warp_tot, int* total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int n = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += n;
  }
  if (lane == 31) warp_tot[w] = inc;
  __syncthreads();
  if (w == 0) {
    int x = warp_tot[lane];
    int xi = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int n = __shfl_up_sync(0xffffffffu, xi, o);
      if (lane >= o) xi += n;
    }
    warp_tot[lane] = xi - x;
    if (lane == 31) *total = xi;
  }
  __syncthreads();
  return warp_tot[w] + inc - v;
}

__global__ void __launch_bounds__(kCheckThreads) check_kernel(
    const int32_t* __restrict__ idx, long long n, int E, int S, long long cap,
    int T, int k, int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
    int32_t* __restrict__ shard, int32_t* __restrict__ flag,
    float* __restrict__ req, int32_t* __restrict__ cap_out) {
  __shared__ int hist[kMaxExperts];
  __shared__ int scan[kMaxExperts + 1];
  __shared__ int warp_tot[32];
  __shared__ int total;
  __shared__ int s_flag, s_max;
  const int tid = threadIdx.x;
  for (int e = tid; e < E; e += blockDim.x) hist[e] = 0;
  if (tid == 0) {
    s_flag = 0;
    s_max = 0;
  }
  __syncthreads();

  // 16-byte loads when the base is 16-byte aligned, else 4-byte loads.
  const bool vec = (reinterpret_cast<uintptr_t>(idx) & 15u) == 0;
  const long long n4 = vec ? n / 4 : 0;
  const int4* idx4 = reinterpret_cast<const int4*>(idx);
  for (long long i = tid; i < n4; i += blockDim.x) {
    int4 q = __ldg(idx4 + i);
    int vals[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (vals[u] >= 0 && vals[u] < E) atomicAdd(&hist[vals[u]], 1);
  }
  for (long long i = n4 * 4 + tid; i < n; i += blockDim.x) {
    int e = __ldg(idx + i);
    if (e >= 0 && e < E) atomicAdd(&hist[e], 1);
  }
  __syncthreads();

  const int c = tid < E ? hist[tid] : 0;
  const int ex = block_exclusive_scan(c, warp_tot, &total);
  if (tid < E) {
    counts[tid] = c;
    offsets[tid] = ex;
    scan[tid] = ex;
  }
  if (tid == 0) {
    offsets[E] = total;
    scan[E] = total;
  }
  __syncthreads();

  const int Es = E / S;
  if (tid < S) {
    const int r = scan[(tid + 1) * Es] - scan[tid * Es];
    shard[tid] = r;
    if (cap >= 0 && r > cap) atomicOr(&s_flag, 1);
    atomicMax(&s_max, r);
  }
  __syncthreads();
  if (tid == 0) {
    *flag = s_flag;
    const double rows = static_cast<double>(T) * static_cast<double>(k);
    *req = rows > 0.0
               ? static_cast<float>(static_cast<double>(s_max) *
                                    static_cast<double>(S) / rows)
               : 0.0f;
    *cap_out = static_cast<int32_t>(cap);
  }
}

}  // namespace

cudaError_t launch_check(const moe_config_t& c, const int32_t* topk_idx,
                         int32_t* counts, int32_t* offsets, int32_t* shard,
                         int32_t* flag, float* req, int32_t* cap,
                         cudaStream_t s) {
  const long long n = static_cast<long long>(c.T) * c.k;
  check_kernel<<<1, kCheckThreads, 0, s>>>(topk_idx, n, c.E, c.S,
                                           capacity_rows(c), c.T, c.k, counts,
                                           offsets, shard, flag, req, cap);
  return cudaGetLastError();
}

}  // namespace moe
