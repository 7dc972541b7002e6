// Stable expert-sorted permute with the capped drop rule and per-shard token
// dedup.
//
// Pages: "Support moe_dropless_fallback=layer on the ragged all-to-all MoE
// path" (MaxText pull request 5920), section Why: rows past a shard's
// factor x balanced buffer are dropped.  "Moe dynamic redundancy" (MaxText
// pull request 4760), review of ra2a_dedup_and_route: a token goes to a
// shard once and is expanded to its expert rows by expand_indices, and the
// expansion must never be truncated.  "MoE ring-of-experts ... x_sorted
// remat save" (MaxText pull request 4969), section What: the expert-sorted
// input x_sorted and its routing metadata.
//
// Order: rows (t, j) sorted by (expert, token).  A token never picks an
// expert twice, so the rank of (t, j) inside expert e is the number of
// tokens before t that picked e.  The kernels, all without inter-CTA waits:
//   1 block_count : per 128-token block, rows per expert        [nb, E]
//   2 scan_experts: per expert, exclusive scan over blocks; expert totals,
//                   dropless offsets, kept rows per expert under the cap
//                   (a shard keeps its first C rows), kept offsets
//   3 assign      : rank of every (t, j) = block base + rank among earlier
//                   warps + rank among earlier lanes (bit masks of lanes per
//                   expert); row_of, sorted_token; per-shard membership of
//                   each token and its rank among the block's members
//   4 scan_uniq   : per shard, exclusive scan of block member counts; |U_s|
//   5 scatter     : one CTA per token: dedup indices, then x[t] read once
//                   with 16-byte loads and written to each kept row
// With a duplication plan ("Moe dynamic redundancy" (MaxText pull request
// 4760), review of plan_expert_duplication) the groups are virtual: shard s
// owns its E/S experts and then its B duplicate slots, and the last
// divert[e] rows of expert e (token order) go to e's slot.  Kernel 2 splits
// each expert's rows between its two groups before the capacity rule, and
// kernel 3 places a row in the group its rank falls in.
// Algorithmic traffic: T*H*b read + R_kept*H*b written (+ small index
// arrays).
#include "internal.h"

namespace moe {
namespace {

constexpr int TB = kPermuteTokensPerBlock;  // tokens per block, 4 warps
constexpr int kWarps = TB / 32;

__global__ void __launch_bounds__(TB) block_count_kernel(
    const int32_t* __restrict__ idx, int T, int E, int k,
    int32_t* __restrict__ block_base, int32_t* __restrict__ status) {
  extern __shared__ int cnt[];
  const int b = blockIdx.x, tid = threadIdx.x;
  for (int e = tid; e < E; e += TB) cnt[e] = 0;
  __syncthreads();
  const int t = b * TB + tid;
  bool bad = false;
  if (t < T) {
    for (int j = 0; j < k; ++j) {
      const int e = __ldg(idx + static_cast<long long>(t) * k + j);
      if (e >= 0 && e < E)
        atomicAdd(&cnt[e], 1);
      else
        bad = true;
    }
  }
  if (bad && status) atomicOr(status, MOE_DEV_BAD_INDEX);
  __syncthreads();
  for (int e = tid; e < E; e += TB)
    block_base[static_cast<long long>(b) * E + e] = cnt[e];
}

__device__ int block_exclusive_scan_1024(int v, int* warp_tot, int* total) {
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
  const int r = warp_tot[w] + inc - v;
  __syncthreads();  // warp_tot may be reused by the caller's next scan
  return r;
}

// One CTA of 1024 threads.  Thread e owns expert e (its block scan and the
// split of its rows), thread g owns virtual group g (the scans over groups
// and the capacity rule).  G <= 1024.
__global__ void __launch_bounds__(1024) scan_experts_kernel(
    int32_t* __restrict__ block_base, int nb, int E, int S, int B, int cap,
    const int32_t* __restrict__ divert, const int32_t* __restrict__ slot_of,
    int32_t* __restrict__ etab, int32_t* __restrict__ group_offsets,
    int32_t* __restrict__ n_dropped) {
  __shared__ int cv[kMaxExperts];       // rows per virtual group
  __shared__ int scan[kMaxExperts + 1];
  __shared__ int keptv[kMaxExperts];
  __shared__ int goffv[kMaxExperts];
  __shared__ int warp_tot[32];
  __shared__ int total, ktotal;
  const int tid = threadIdx.x;
  const int Es = E / S, Gs = Es + B, G = S * Gs;
  if (tid < G) cv[tid] = 0;
  __syncthreads();
  int c = 0, d = 0, slot = -1;
  if (tid < E) {
    int run = 0;
    for (int b = 0; b < nb; ++b) {
      int32_t* p = block_base + static_cast<long long>(b) * E + tid;
      const int v = *p;
      *p = run;
      run += v;
    }
    c = run;
    if (divert != nullptr && slot_of != nullptr) {
      slot = slot_of[tid];
      // a duplicate must sit in a slot position of some shard
      if (slot < 0 || slot >= G || slot % Gs < Es) slot = -1;
      d = slot >= 0 ? min(max(divert[tid], 0), c) : 0;
      if (d == 0) slot = -1;
    }
    cv[(tid / Es) * Gs + tid % Es] = c - d;
    if (slot >= 0) cv[slot] = d;
  }
  __syncthreads();
  const int cg = tid < G ? cv[tid] : 0;
  const int ex = block_exclusive_scan_1024(cg, warp_tot, &total);
  if (tid < G) scan[tid] = ex;
  if (tid == 0) scan[G] = total;
  __syncthreads();
  int kept = cg;
  if (tid < G && cap >= 0) {
    const int local = ex - scan[(tid / Gs) * Gs];  // rows of the shard before g
    kept = min(max(cap - local, 0), cg);
  }
  const int kex = block_exclusive_scan_1024(tid < G ? kept : 0, warp_tot,
                                            &ktotal);
  if (tid < G) {
    keptv[tid] = kept;
    goffv[tid] = kex;
    group_offsets[tid] = kex;
  }
  if (tid == 0) {
    group_offsets[G] = ktotal;
    *n_dropped = total - ktotal;
  }
  __syncthreads();
  if (tid < E) {
    const int home = (tid / Es) * Gs + tid % Es;
    etab[0 * E + tid] = keptv[home];
    etab[1 * E + tid] = goffv[home];
    etab[2 * E + tid] = c - d;
    etab[3 * E + tid] = slot >= 0 ? keptv[slot] : 0;
    etab[4 * E + tid] = slot >= 0 ? goffv[slot] : 0;
    etab[5 * E + tid] = slot >= 0 ? slot / Gs : tid / Es;
  }
}

__global__ void __launch_bounds__(TB) assign_kernel(
    const int32_t* __restrict__ idx, int T, int E, int k, int S,
    const int32_t* __restrict__ block_base, const int32_t* __restrict__ etab_g,
    int32_t* __restrict__ row_of, int32_t* __restrict__ sorted_token,
    int32_t* __restrict__ block_ucnt, int32_t* __restrict__ urank) {
  extern __shared__ int sm[];
  uint32_t* mask = reinterpret_cast<uint32_t*>(sm);  // [kWarps][E]
  int* wpre = sm + kWarps * E;                       // [kWarps][E]
  int* base = wpre + kWarps * E;                     // [E]
  int* etab = base + E;                              // [6][E]
  uint32_t* ballot = reinterpret_cast<uint32_t*>(etab + 6 * E);  // [kWarps][S]
  int* upre = reinterpret_cast<int*>(ballot + kWarps * S);       // [kWarps][S]

  const int b = blockIdx.x, tid = threadIdx.x;
  const int w = tid >> 5, lane = tid & 31;
  const uint32_t lt = (1u << lane) - 1u;
  for (int e = tid; e < E; e += TB) {
    base[e] = block_base[static_cast<long long>(b) * E + e];
#pragma unroll
    for (int q = 0; q < 6; ++q) etab[q * E + e] = etab_g[q * E + e];
#pragma unroll
    for (int q = 0; q < kWarps; ++q) mask[q * E + e] = 0u;
  }
  __syncthreads();
  const int t = b * TB + tid;
  const bool valid = t < T;
  const long long tk = static_cast<long long>(t) * k;
  if (valid) {
    for (int j = 0; j < k; ++j) {
      const int e = __ldg(idx + tk + j);
      if (e >= 0 && e < E) atomicOr(&mask[w * E + e], 1u << lane);
    }
  }
  __syncthreads();
  for (int e = tid; e < E; e += TB) {
    int run = 0;
#pragma unroll
    for (int q = 0; q < kWarps; ++q) {
      wpre[q * E + e] = run;
      run += __popc(mask[q * E + e]);
    }
  }
  __syncthreads();
  const int Es = E / S;
  uint64_t smask = 0;
  if (valid) {
    for (int j = 0; j < k; ++j) {
      const int e = __ldg(idx + tk + j);
      int row = -1;
      if (e >= 0 && e < E) {
        const int rank =
            base[e] + wpre[w * E + e] + __popc(mask[w * E + e] & lt);
        const int own = etab[2 * E + e];
        if (rank < own) {            // the expert's own group
          if (rank < etab[0 * E + e]) {
            row = etab[1 * E + e] + rank;
            smask |= 1ull << (e / Es);
          }
        } else if (rank - own < etab[3 * E + e]) {  // its duplicate slot
          row = etab[4 * E + e] + (rank - own);
          smask |= 1ull << etab[5 * E + e];
        }
        if (row >= 0) sorted_token[row] = t;
      }
      row_of[tk + j] = row;
    }
  }
  for (int s = 0; s < S; ++s) {
    const uint32_t bal = __ballot_sync(0xffffffffu, (smask >> s) & 1ull);
    if (lane == 0) ballot[w * S + s] = bal;
  }
  __syncthreads();
  for (int s = tid; s < S; s += TB) {
    int run = 0;
#pragma unroll
    for (int q = 0; q < kWarps; ++q) {
      upre[q * S + s] = run;
      run += __popc(ballot[q * S + s]);
    }
    block_ucnt[static_cast<long long>(b) * S + s] = run;
  }
  __syncthreads();
  if (valid) {
    for (int j = 0; j < k; ++j) {
      int ur = -1;
      if (row_of[tk + j] >= 0) {
        const int e = __ldg(idx + tk + j);
        const int rank =
            base[e] + wpre[w * E + e] + __popc(mask[w * E + e] & lt);
        const int s = rank < etab[2 * E + e] ? e / Es : etab[5 * E + e];
        ur = ((upre[w * S + s] + __popc(ballot[w * S + s] & lt)) << 6) | s;
      }
      urank[tk + j] = ur;
    }
  }
}

// One block of 64 threads; thread s owns shard s.
__global__ void __launch_bounds__(64) scan_uniq_kernel(
    int32_t* __restrict__ block_ucnt, int nb, int S,
    int32_t* __restrict__ uniq_offsets) {
  __shared__ int tot[kMaxShards];
  const int s = threadIdx.x;
  if (s < S) {
    int run = 0;
    for (int b = 0; b < nb; ++b) {
      int32_t* p = block_ucnt + static_cast<long long>(b) * S + s;
      const int v = *p;
      *p = run;
      run += v;
    }
    tot[s] = run;
  }
  __syncthreads();
  if (s == 0) {
    int run = 0;
    for (int q = 0; q < S; ++q) {
      uniq_offsets[q] = run;
      run += tot[q];
    }
    uniq_offsets[S] = run;
  }
}

constexpr int kScatterThreads = 128;
constexpr int kScatterUnroll = 8;

// One CTA per token.
__global__ void __launch_bounds__(kScatterThreads) scatter_kernel(
    const int4* __restrict__ x, int n16, const int32_t* __restrict__ idx,
    int E, int k, int S, const int32_t* __restrict__ row_of,
    const int32_t* __restrict__ block_ucnt, const int32_t* __restrict__ urank,
    const int32_t* __restrict__ uniq_offsets, int4* __restrict__ x_sorted,
    int32_t* __restrict__ expand_idx, int32_t* __restrict__ uniq_tokens) {
  __shared__ int rows[kMaxTopK];
  const int t = blockIdx.x, tid = threadIdx.x;
  const long long tk = static_cast<long long>(t) * k;
  if (tid < k) {
    const int row = row_of[tk + tid];
    rows[tid] = row;
    if (row >= 0) {
      const int code = urank[tk + tid];
      const int s = code & 63;
      const int upos = uniq_offsets[s] +
                       block_ucnt[static_cast<long long>(t / TB) * S + s] +
                       (code >> 6);
      expand_idx[row] = upos;
      bool first = true;
      for (int q = 0; q < tid; ++q)
        if (row_of[tk + q] >= 0 && (urank[tk + q] & 63) == s) first = false;
      if (first) uniq_tokens[upos] = t;
    }
  }
  __syncthreads();
  const int4* src = x + static_cast<long long>(t) * n16;
  for (int c0 = tid; c0 < n16; c0 += kScatterThreads * kScatterUnroll) {
    int4 v[kScatterUnroll];
#pragma unroll
    for (int u = 0; u < kScatterUnroll; ++u) {
      const int c = c0 + u * kScatterThreads;
      if (c < n16) v[u] = __ldg(src + c);
    }
    for (int j = 0; j < k; ++j) {
      const int r = rows[j];
      if (r < 0) continue;
      int4* dst = x_sorted + static_cast<long long>(r) * n16;
#pragma unroll
      for (int u = 0; u < kScatterUnroll; ++u) {
        const int c = c0 + u * kScatterThreads;
        if (c < n16) dst[c] = v[u];
      }
    }
  }
}

size_t assign_smem_bytes(int E, int S) {
  return sizeof(int) * (2 * kWarps * E + 7 * E + 2 * kWarps * S);
}

}  // namespace

size_t permute_scratch_bytes(int T, int E, int k, int S) {
  Carve c(nullptr);
  carve_permute_scratch(c, T, E, k, S);
  return align_up(c.off, 256);
}

PermuteScratch carve_permute_scratch(Carve& c, int T, int E, int k, int S) {
  const size_t nb = static_cast<size_t>((T + TB - 1) / TB);
  PermuteScratch p;
  p.block_base = c.take<int32_t>(nb * E);
  p.etab = c.take<int32_t>(6 * static_cast<size_t>(E));
  p.block_ucnt = c.take<int32_t>(nb * S);
  p.urank = c.take<int32_t>(static_cast<size_t>(T) * k);
  p.scal = c.take<int32_t>(4);
  return p;
}

cudaError_t launch_permute(const moe_config_t& c, const void* x,
                           const int32_t* topk_idx, int64_t cap,
                           void* x_sorted, int32_t* row_of,
                           int32_t* sorted_token, int32_t* group_offsets,
                           int32_t* uniq_offsets, int32_t* uniq_tokens,
                           int32_t* expand_idx, int32_t* n_dropped,
                           const PermuteScratch& ws, int32_t* status,
                           cudaStream_t s, const PermutePlan& plan) {
  const int nb = (c.T + TB - 1) / TB;
  if (nb > 0) {
    block_count_kernel<<<nb, TB, c.E * sizeof(int), s>>>(
        topk_idx, c.T, c.E, c.k, ws.block_base, status);
  }
  scan_experts_kernel<<<1, 1024, 0, s>>>(
      ws.block_base, nb, c.E, c.S, plan.B, static_cast<int>(cap),
      plan.divert, plan.slot_of, ws.etab, group_offsets, n_dropped);
  if (nb > 0) {
    const size_t smem = assign_smem_bytes(c.E, c.S);
    if (smem > 48 * 1024) {
      const cudaError_t e = cudaFuncSetAttribute(
          assign_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
          static_cast<int>(smem));
      if (e != cudaSuccess) return e;
    }
    assign_kernel<<<nb, TB, smem, s>>>(topk_idx, c.T, c.E, c.k, c.S,
                                       ws.block_base, ws.etab, row_of,
                                       sorted_token, ws.block_ucnt, ws.urank);
  }
  scan_uniq_kernel<<<1, 64, 0, s>>>(ws.block_ucnt, nb, c.S, uniq_offsets);
  if (c.T > 0) {
    const int n16 = c.H * elem_bytes(c.dtype) / 16;
    scatter_kernel<<<c.T, kScatterThreads, 0, s>>>(
        static_cast<const int4*>(x), n16, topk_idx, c.E, c.k, c.S, row_of,
        ws.block_ucnt, ws.urank, uniq_offsets, static_cast<int4*>(x_sorted),
        expand_idx, uniq_tokens);
  }
  return cudaGetLastError();
}

}  // namespace moe
