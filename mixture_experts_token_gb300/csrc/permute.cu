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
//                   (only for tables of more than 1024 block-shard counts:
//                   below that, every scatter CTA sums the table itself)
//   5 scatter     : one CTA per token: dedup indices, then x[t] read once
//                   with 16-byte loads and written to each kept row
// Kernels 2 to 5 are programmatic dependent launches: each may start once
// its predecessor has started, does the work that needs none of its
// predecessor's output (assign: the lane masks from the routing indices;
// scatter: the read of x[t]), and then waits for its predecessor to finish.
// launch_permute_tables runs kernels 1 to 4, launch_permute_scatter kernel 5
// (a caller may run the two on different streams, ordered by an event, so
// that one chunk's tables overlap the previous chunk's expert FFN);
// launch_permute runs both on one stream.
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
constexpr int kBatch = 16;  // independent loads a thread issues together

// Programmatic dependent launch: a kernel launched with programmatic stream
// serialisation may start once every CTA of its producer has called
// allow_dependents() (or exited); wait_for_producer() returns when the
// producer grid has finished and its writes are visible.  Without that
// launch attribute the wait returns at once.
__device__ __forceinline__ void allow_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void wait_for_producer() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

__global__ void __launch_bounds__(TB) block_count_kernel(
    const int32_t* __restrict__ idx, int T, int E, int k,
    int32_t* __restrict__ block_base, int32_t* __restrict__ status) {
  extern __shared__ int cnt[];
  allow_dependents();
  const int b = blockIdx.x, tid = threadIdx.x;
  for (int e = tid; e < E; e += TB) cnt[e] = 0;
  __syncthreads();
  // the block's entries (t, j) in memory order, kBatch loads in flight
  const int32_t* src = idx + static_cast<long long>(b) * TB * k;
  const int m = min(TB, T - b * TB) * k;
  bool bad = false;
  for (int i0 = tid; i0 < m; i0 += kBatch * TB) {
    int v[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int i = i0 + u * TB;
      v[u] = i < m ? __ldg(src + i) : 0;
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      if (i0 + u * TB >= m) break;
      if (v[u] >= 0 && v[u] < E)
        atomicAdd(&cnt[v[u]], 1);
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

// In place, over one column of a row-major [n, stride] table: v[b] becomes
// the sum of v[0..b); returns the total.  The loads of a batch are issued
// before its stores, so the column costs about n/kBatch memory latencies
// rather than n.
__device__ __forceinline__ int exclusive_scan_column(int32_t* col, int n,
                                                     int stride) {
  int run = 0;
  for (int b0 = 0; b0 < n; b0 += kBatch) {
    int v[kBatch];
#pragma unroll
    for (int i = 0; i < kBatch; ++i)
      v[i] = b0 + i < n ? __ldcg(col + static_cast<long long>(b0 + i) * stride)
                        : 0;
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      if (b0 + i < n) col[static_cast<long long>(b0 + i) * stride] = run;
      run += v[i];
    }
  }
  return run;
}

// One CTA of 1024 threads.  Thread e owns expert e (its block scan and the
// split of its rows), thread g owns virtual group g (the scans over groups
// and the capacity rule).  G <= 1024.
__global__ void __launch_bounds__(1024) scan_experts_kernel(
    int32_t* __restrict__ block_base, int nb, int E, int S, int B, int cap,
    const int32_t* __restrict__ divert, const int32_t* __restrict__ slot_of,
    int32_t* __restrict__ etab, int32_t* __restrict__ group_offsets,
    int32_t* __restrict__ n_dropped, int32_t* __restrict__ uniq_offsets) {
  __shared__ int cv[kMaxExperts];       // rows per virtual group
  __shared__ int scan[kMaxExperts + 1];
  __shared__ int keptv[kMaxExperts];
  __shared__ int goffv[kMaxExperts];
  __shared__ int warp_tot[32];
  __shared__ int total, ktotal;
  allow_dependents();
  const int tid = threadIdx.x;
  const int Es = E / S, Gs = Es + B, G = S * Gs;
  if (tid < G) cv[tid] = 0;
  __syncthreads();
  wait_for_producer();
  int c = 0, d = 0, slot = -1;
  if (tid < E) {
    c = exclusive_scan_column(block_base + tid, nb, E);
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
  if (nb == 0 && tid <= S) uniq_offsets[tid] = 0;  // no tokens: no assign
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

  allow_dependents();
  const int b = blockIdx.x, tid = threadIdx.x;
  const int w = tid >> 5, lane = tid & 31;
  const uint32_t lt = (1u << lane) - 1u;
  for (int e = tid; e < E; e += TB) {
#pragma unroll
    for (int q = 0; q < kWarps; ++q) mask[q * E + e] = 0u;
  }
  __syncthreads();
  const int t = b * TB + tid;
  const bool valid = t < T;
  const long long tk = static_cast<long long>(t) * k;
  {
    // entry i of the block is (token i / k, pick i % k)
    const int32_t* src = idx + static_cast<long long>(b) * TB * k;
    const int m = min(TB, T - b * TB) * k;
    for (int i0 = tid; i0 < m; i0 += kBatch * TB) {
      int v[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int i = i0 + u * TB;
        v[u] = i < m ? __ldg(src + i) : -1;
      }
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int tl = (i0 + u * TB) / k;  // token within the block
        if (v[u] >= 0 && v[u] < E)
          atomicOr(&mask[(tl >> 5) * E + v[u]], 1u << (tl & 31));
      }
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
  // Everything above reads only the routing indices; the block bases and
  // the expert tables come from the scan.
  wait_for_producer();
  for (int e = tid; e < E; e += TB) {
    base[e] = block_base[static_cast<long long>(b) * E + e];
#pragma unroll
    for (int q = 0; q < 6; ++q) etab[q * E + e] = etab_g[q * E + e];
  }
  __syncthreads();
  const int Es = E / S;
  uint64_t smask = 0;
  uint32_t kept = 0;  // bit j: (t, j) has a row
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
        if (row >= 0) {
          sorted_token[row] = t;
          kept |= 1u << j;
        }
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
      if ((kept >> j) & 1u) {
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
  allow_dependents();
  wait_for_producer();
  const int s = threadIdx.x;
  if (s < S) tot[s] = exclusive_scan_column(block_ucnt + s, nb, S);
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
constexpr int kScatterCtasPerSm = 4;

// Block-shard tables up to this many counts are summed by every scatter CTA
// (no scan kernel between assign and the scatter).
constexpr int kInlineUniqCounts = 1024;
static_assert(kInlineUniqCounts % kScatterThreads == 0, "whole loads");
inline bool inline_uniq(int nb, int S) {
  return static_cast<long long>(nb) * S <= kInlineUniqCounts;
}

// One CTA per token, or per (token, column slice) when there are too few
// tokens to keep every SM busy: the row's 16-byte chunks are split into
// contiguous slices, one CTA each, and only the slice-0 CTA of a token
// writes its index outputs.  The first part of the CTA's slice (all of it
// up to 16 KB) is read before the wait for the tables.  Dedup position of
// (t, j) in shard s: the members of shards before s, plus those of s in
// the token blocks before t's, plus t's rank among its block's members.
// With inline_uniq the first two come from the block_ucnt counts as assign
// left them, and CTA 0 writes uniq_offsets; otherwise scan_uniq has
// scanned them.
__global__ void __launch_bounds__(kScatterThreads) scatter_kernel(
    const int4* __restrict__ x, int n16, int k, int S, int nb,
    int inline_uniq, const int32_t* __restrict__ row_of,
    const int32_t* __restrict__ block_ucnt, const int32_t* __restrict__ urank,
    int32_t* __restrict__ uniq_offsets, int4* __restrict__ x_sorted,
    int32_t* __restrict__ expand_idx, int32_t* __restrict__ uniq_tokens,
    int per_split) {
  __shared__ int rows[kMaxTopK];
  __shared__ int codes[kMaxTopK];
  __shared__ int tot[kMaxShards];     // members of shard s, all blocks
  __shared__ int before[kMaxShards];  // members of shard s, blocks before t's
  const int t = blockIdx.x, tid = threadIdx.x;
  const int bt = t / TB;
  const long long tk = static_cast<long long>(t) * k;
  // x_sorted == null: the index outputs only (no row is read or written)
  const int n16r = x_sorted != nullptr ? n16 : 0;
  const bool index_cta = blockIdx.y == 0;  // writes the index outputs
  const int begin = blockIdx.y * per_split;
  const int end = min(n16r, begin + per_split);
  const int4* src = x + static_cast<long long>(t) * n16r;
  int4 v[kScatterUnroll];
#pragma unroll
  for (int u = 0; u < kScatterUnroll; ++u) {
    const int c = begin + tid + u * kScatterThreads;
    if (c < end) v[u] = __ldg(src + c);
  }
  for (int q = tid; q < S; q += kScatterThreads) {
    tot[q] = 0;
    before[q] = 0;
  }
  wait_for_producer();
  if (tid < k) {
    rows[tid] = row_of[tk + tid];
    codes[tid] = urank[tk + tid];
  }
  if (inline_uniq && index_cta) {
    constexpr int kPer = kInlineUniqCounts / kScatterThreads;
    int c[kPer];
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int i = tid + u * kScatterThreads;
      c[u] = i < nb * S ? __ldcg(block_ucnt + i) : 0;
    }
    __syncthreads();  // the zeroed sums
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int i = tid + u * kScatterThreads;
      if (c[u] == 0) continue;
      const int q = i % S;
      atomicAdd(&tot[q], c[u]);
      if (i / S < bt) atomicAdd(&before[q], c[u]);
    }
  }
  __syncthreads();
  if (index_cta && tid < k && rows[tid] >= 0) {
    const int code = codes[tid];
    const int q = code & 63;
    int base;
    if (inline_uniq) {
      base = before[q];
      for (int p = 0; p < q; ++p) base += tot[p];
    } else {
      base = uniq_offsets[q] + block_ucnt[static_cast<long long>(bt) * S + q];
    }
    const int upos = base + (code >> 6);
    expand_idx[rows[tid]] = upos;
    bool first = true;  // the token's first row bound for shard q
    for (int p = 0; p < tid; ++p)
      if (rows[p] >= 0 && (codes[p] & 63) == q) first = false;
    if (first) uniq_tokens[upos] = t;
  }
  if (inline_uniq && index_cta && t == 0 && tid <= S) {
    int o = 0;
    for (int p = 0; p < tid; ++p) o += tot[p];
    uniq_offsets[tid] = o;
  }
  __syncthreads();
  for (int c0 = begin + tid; c0 < end;
       c0 += kScatterThreads * kScatterUnroll) {
    if (c0 != begin + tid) {
#pragma unroll
      for (int u = 0; u < kScatterUnroll; ++u) {
        const int c = c0 + u * kScatterThreads;
        if (c < end) v[u] = __ldg(src + c);
      }
    }
    for (int j = 0; j < k; ++j) {
      const int r = rows[j];
      if (r < 0) continue;
      int4* dst = x_sorted + static_cast<long long>(r) * n16;
#pragma unroll
      for (int u = 0; u < kScatterUnroll; ++u) {
        const int c = c0 + u * kScatterThreads;
        if (c < end) dst[c] = v[u];
      }
    }
  }
}

size_t assign_smem_bytes(int E, int S) {
  return sizeof(int) * (2 * kWarps * E + 7 * E + 2 * kWarps * S);
}

// A launch on stream s that may start before the previous kernel on s has
// finished (that kernel calls allow_dependents(), this one
// wait_for_producer() before reading its output).
template <typename... Params, typename... Args>
cudaError_t launch_dependent(void (*kernel)(Params...), dim3 grid,
                             unsigned block, size_t smem, cudaStream_t s,
                             Args... args) {
  cudaLaunchConfig_t lc = {};
  lc.gridDim = grid;
  lc.blockDim = dim3(block);
  lc.dynamicSmemBytes = smem;
  lc.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = at;
  lc.numAttrs = 1;
  return cudaLaunchKernelEx(&lc, kernel, static_cast<Params>(args)...);
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

cudaError_t launch_permute_tables(const moe_config_t& c,
                                  const int32_t* topk_idx, int64_t cap,
                                  int32_t* row_of, int32_t* sorted_token,
                                  int32_t* group_offsets,
                                  int32_t* uniq_offsets, int32_t* n_dropped,
                                  const PermuteScratch& ws, int32_t* status,
                                  cudaStream_t s, const PermutePlan& plan) {
  const int nb = (c.T + TB - 1) / TB;
  cudaError_t e = cudaSuccess;
  if (nb > 0) {
    block_count_kernel<<<nb, TB, c.E * sizeof(int), s>>>(
        topk_idx, c.T, c.E, c.k, ws.block_base, status);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if ((e = launch_dependent(scan_experts_kernel, 1, 1024, 0, s, ws.block_base,
                            nb, c.E, c.S, plan.B, static_cast<int>(cap),
                            plan.divert, plan.slot_of, ws.etab, group_offsets,
                            n_dropped, uniq_offsets)) != cudaSuccess)
    return e;
  if (nb > 0) {
    const size_t smem = assign_smem_bytes(c.E, c.S);
    if (smem > 48 * 1024 &&
        (e = cudaFuncSetAttribute(assign_kernel,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  static_cast<int>(smem))) != cudaSuccess)
      return e;
    if ((e = launch_dependent(assign_kernel, nb, TB, smem, s, topk_idx, c.T,
                              c.E, c.k, c.S, ws.block_base, ws.etab, row_of,
                              sorted_token, ws.block_ucnt, ws.urank)) !=
        cudaSuccess)
      return e;
  }
  if (nb > 0 && !inline_uniq(nb, c.S) &&
      (e = launch_dependent(scan_uniq_kernel, 1, 64, 0, s, ws.block_ucnt, nb,
                            c.S, uniq_offsets)) != cudaSuccess)
    return e;
  return cudaGetLastError();
}

cudaError_t launch_permute_scatter(const moe_config_t& c, const void* x,
                                   const int32_t* row_of,
                                   int32_t* uniq_offsets, void* x_sorted,
                                   int32_t* uniq_tokens, int32_t* expand_idx,
                                   const PermuteScratch& ws, cudaStream_t s) {
  if (c.T == 0) return cudaSuccess;
  const int nb = (c.T + TB - 1) / TB;
  const int n16 = c.H * elem_bytes(c.dtype) / 16;
  // CTAs per token: about kScatterCtasPerSm CTAs per SM over the grid, but
  // no slice narrower than one pass of the CTA's threads
  int splits = 1;
  int dev = 0, sms = 0;
  if (x_sorted != nullptr && cudaGetDevice(&dev) == cudaSuccess &&
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) ==
          cudaSuccess) {
    const int want = (kScatterCtasPerSm * sms + c.T - 1) / c.T;
    splits = std::max(1, std::min(want, n16 / kScatterThreads));
  }
  const int per = (n16 + splits - 1) / splits;
  return launch_dependent(scatter_kernel,
                          dim3(static_cast<unsigned>(c.T),
                               static_cast<unsigned>(splits)),
                          kScatterThreads, 0, s,
                          static_cast<const int4*>(x), n16, c.k, c.S, nb,
                          inline_uniq(nb, c.S) ? 1 : 0, row_of,
                          ws.block_ucnt, ws.urank, uniq_offsets,
                          static_cast<int4*>(x_sorted), expand_idx,
                          uniq_tokens, per);
}

cudaError_t launch_permute(const moe_config_t& c, const void* x,
                           const int32_t* topk_idx, int64_t cap,
                           void* x_sorted, int32_t* row_of,
                           int32_t* sorted_token, int32_t* group_offsets,
                           int32_t* uniq_offsets, int32_t* uniq_tokens,
                           int32_t* expand_idx, int32_t* n_dropped,
                           const PermuteScratch& ws, int32_t* status,
                           cudaStream_t s, const PermutePlan& plan) {
  const cudaError_t e =
      launch_permute_tables(c, topk_idx, cap, row_of, sorted_token,
                            group_offsets, uniq_offsets, n_dropped, ws,
                            status, s, plan);
  if (e != cudaSuccess) return e;
  return launch_permute_scatter(c, x, row_of, uniq_offsets, x_sorted,
                                uniq_tokens, expand_idx, ws, s);
}

}  // namespace moe
