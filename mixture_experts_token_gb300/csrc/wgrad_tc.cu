// Weight gradients of the grouped SwiGLU FFN on the tensor cores (tcgen05,
// accumulators in tensor memory, operands staged by TMA).
//
// "Support moe_dropless_fallback=layer on the ragged all-to-all MoE path"
// (MaxText pull request 5920), section How: the fallback's backward
// accumulates the expert-weight gradients over the chunks; "Moe dynamic
// redundancy" (MaxText pull request 4760), review comments: the expert FFN
// is a grouped matmul over experts with ragged group sizes.
#include <atomic>

#include "tc_common.cuh"

namespace moe {
namespace tc {

// ------------------------------------------------- weight gradients ------
// dW[e] (+)= P_e^T Q_e over the rows of expert e: P = x_sorted, Q = [dg | du]
// (WMODE 0: dWg and dWu, tile = 128 rows of H x (128 gate + 128 up) cols
// of F) or P = h, Q = dy_sorted (WMODE 1: dWd, 128 rows of F x BN of H).
// The reduction runs over routed rows, so both operands are read
// "MN-major" straight from the row-major activations: TMA box {64 cols,
// 64 rows}, one 8 KB box per 64 columns, descriptors LBO = 8192, SBO =
// 1024, start advanced 2048 B per K=16 step, and both major bits set.
// K is ragged: a group's last k-block holds rows of the next group (or TMA
// zero fill, or unwritten rows past the end).  The MMA warp issues only the
// K=16 steps that reach valid rows and clears the invalid rows of those
// steps in both operands (shared memory) before it issues them.
// Tiles of one expert run with the column tile fastest, so the CTAs at work
// at one time write whole rows of dW; dW goes out with an L2 evict-first
// policy and the activation rows come in with evict-last, so the 100+ MB
// gradient stream of an expert does not push its few MB of rows (read by
// every tile) out of L2.
// Segments: rows of one expert may sit in several independent row ranges
// (one per chunk of the chunked fallback); a tile accumulates all of them
// in tensor memory before its single write.  The epilogue moves each
// 32 x 32 fp32 sub-tile through a 128-byte-swizzled staging buffer to a
// TMA store (overwrite) or a TMA reduce-add (accumulate in L2).
#ifndef MOE_WGRAD_STAGES
#define MOE_WGRAD_STAGES 3
#endif
#ifndef MOE_WGRAD_STAGE_BUFS
#define MOE_WGRAD_STAGE_BUFS 4
#endif
constexpr int WSTAGES = MOE_WGRAD_STAGES;
constexpr int kWStage = BM * BK * 2 + BK * 256 * 2;  // 48 KB
constexpr int kStageBuf = 32 * 32 * 4;               // 4 KB
constexpr int kStageBufs = MOE_WGRAD_STAGE_BUFS;  // staging buffers per epilogue warp
constexpr int kMaxSeg = 16;

struct WParams {
  const int32_t* seg_off[kMaxSeg];  // [G+1] group row offsets per segment
  int seg_base[kMaxSeg];            // row of the segment's first row
  int n_seg;
  const int32_t* group_expert;      // [G] or null (identity)
  int G;
  int m_tiles;   // 128-row tiles of one expert's dW
  int n_tiles;   // column tiles
  int reduce;    // 1: TMA reduce-add everywhere; 0: TMA store, except
                 // for experts with several groups (duplicates), whose
                 // tiles add onto a slice zeroed beforehand
  int E;         // experts (dW slices)
  int32_t* status;
  // Tests of the timeout path only (the two-SM kernel): both CTAs' producers
  // stop after this many stage fills (-1: never), so the MMA's wait runs out.
  long long stall_after_fills = -1;
};

// The GEMMs' test hook (gmm_tc.cu), shared by the two-SM weight gradient.
extern std::atomic<long long> g_stall_after_fills;

// L2 policies: the weight gradients stream through L2 once (evict first);
// the activation rows feed every tile of their expert (evict last).
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;"
               : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;"
               : "=l"(p));
  return p;
}

__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst,
                                                 const CUtensorMap* m,
                                                 uint32_t bar, int c0, int c1,
                                                 uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::"
      "complete_tx::bytes.L2::cache_hint [%0], [%1, {%3, %4}], [%2], %5;" ::
          "r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(c0), "r"(c1),
      "l"(policy)
      : "memory");
}

__device__ __forceinline__ void tma_store_2d(const CUtensorMap* m,
                                             uint32_t src, int c0, int c1,
                                             uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group"
      ".L2::cache_hint [%0, {%2, %3}], [%1], %4;" ::"l"(
          reinterpret_cast<uint64_t>(m)),
      "r"(src), "r"(c0), "r"(c1), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void tma_reduce_add_2d(const CUtensorMap* m,
                                                  uint32_t src, int c0,
                                                  int c1, uint64_t policy) {
  asm volatile(
      "cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.tile."
      "bulk_group.L2::cache_hint [%0, {%2, %3}], [%1], %4;" ::"l"(
          reinterpret_cast<uint64_t>(m)),
      "r"(src), "r"(c0), "r"(c1), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// At most kStageBufs - 1 bulk groups of this thread still reading shared
// memory: the oldest staging buffer is free again.
__device__ __forceinline__ void bulk_wait_read_free() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(kStageBufs - 1)
               : "memory");
}

__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

__device__ __forceinline__ int wgrad_rows(const WParams& p, int g) {
  int n = 0;
  for (int sg = 0; sg < p.n_seg; ++sg)
    n += __ldg(p.seg_off[sg] + g + 1) - __ldg(p.seg_off[sg] + g);
  return n;
}

// tpre[g] = tiles of groups before g (a group with rows has m*n tiles).
__device__ void build_wgrad_table(const WParams& p, int* tpre, int* wsum) {
  const int G = p.G, tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int per = (G + kThreads - 1) / kThreads;
  const int g0 = min(G, tid * per), g1 = min(G, g0 + per);
  const int tiles = p.m_tiles * p.n_tiles;
  int loc = 0;
  for (int g = g0; g < g1; ++g) {
    tpre[g] = wgrad_rows(p, g) > 0 ? tiles : 0;
    loc += tpre[g];
  }
  int inc = loc;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += v;
  }
  if (lane == 31) wsum[w] = inc;
  __syncthreads();
  if (tid == 0) {
    int run = 0;
    for (int i = 0; i < kThreads / 32; ++i) {
      const int v = wsum[i];
      wsum[i] = run;
      run += v;
    }
    wsum[kThreads / 32] = run;
  }
  __syncthreads();
  int run = wsum[w] + inc - loc;
  for (int g = g0; g < g1; ++g) {
    const int v = tpre[g];
    tpre[g] = run;
    run += v;
  }
  if (tid == 0) tpre[G] = wsum[kThreads / 32];
  __syncthreads();
}

template <int WMODE, int BN>
__global__ void __launch_bounds__(kThreads, 1)
    wgrad_tc_kernel(const __grid_constant__ CUtensorMap tmP,
                    const __grid_constant__ CUtensorMap tmQ0,
                    const __grid_constant__ CUtensorMap tmQ1,
                    const __grid_constant__ CUtensorMap tmO0,
                    const __grid_constant__ CUtensorMap tmO1, WParams p) {
  static_assert(WMODE == 1 || BN == 256, "gate + up tiles are 128 + 128");
  constexpr int kAChunks = BM / 64;       // 2
  constexpr int kBChunks = BN / 64;       // 2 or 4
  constexpr uint32_t kTx = (kAChunks + kBChunks) * 8192;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stagebuf = smem + WSTAGES * kWStage;  // [4 warps][kStageBufs][4 KB]
  uint64_t* bars =
      reinterpret_cast<uint64_t*>(stagebuf + 4 * kStageBufs * kStageBuf);
  uint64_t* full = bars;
  uint64_t* empty = bars + WSTAGES;
  uint64_t* tfull = bars + 2 * WSTAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* done = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* wsum = reinterpret_cast<int*>(tmem_slot + 4);  // [16]
  int* tpre = wsum + 16;                               // [G+1]
  int* ecnt = tpre + (p.G + 1);                        // [E] groups w/ rows

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t smem_base = smem_u32(smem);

  if (threadIdx.x == 0) {
    for (int s = 0; s < WSTAGES; ++s) {
      mbar_init(smem_u32(full + s), 1);
      mbar_init(smem_u32(empty + s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(smem_u32(tfull + a), 1);
      mbar_init(smem_u32(tempty + a), kEpilogueThreads);
    }
    mbar_init(smem_u32(done), 1);
    *abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmP);
    prefetch_tmap(&tmQ0);
    if (WMODE == 0) prefetch_tmap(&tmQ1);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  build_wgrad_table(p, tpre, wsum);
  // groups with rows per expert: an expert with one writes its dW with
  // plain stores, one with several (a duplicated expert) adds each group's
  // tile onto its zeroed slice
  for (int e = threadIdx.x; e < p.E; e += blockDim.x) ecnt[e] = 0;
  __syncthreads();
  if (p.group_expert != nullptr)
    for (int g = threadIdx.x; g < p.G; g += blockDim.x)
      if (tpre[g + 1] > tpre[g]) atomicAdd(&ecnt[__ldg(p.group_expert + g)], 1);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int total_tiles = tpre[p.G];

  if (warp == 0) {
    // ------------------------------------------------ TMA producer -----
    if (lane == 0) {
      const uint64_t keep = policy_evict_last();
      int stage = 0;
      uint32_t phase = 0;
      long long fills = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total_tiles;
           tile += gridDim.x) {
        const int g = group_of(tpre, p.G, tile);
        const int local = tile - tpre[g];
        const int n = local % p.n_tiles, m = local / p.n_tiles;
        for (int sg = 0; ok && sg < p.n_seg; ++sg) {
          const int r1 = p.seg_base[sg] + __ldg(p.seg_off[sg] + g + 1);
          for (int r = p.seg_base[sg] + __ldg(p.seg_off[sg] + g); r < r1;
               r += BK) {
            if (!mbar_wait(smem_u32(empty + stage), phase ^ 1u, abort_flag,
                           p.status)) {
              ok = false;
              break;
            }
            const uint32_t fb = smem_u32(full + stage);
            mbar_expect_tx(fb, kTx);
            const uint32_t sa = smem_base + stage * kWStage;
            const uint32_t sb = sa + kAChunks * 8192;
#pragma unroll
            for (int j = 0; j < kAChunks; ++j)
              tma_load_2d_hint(sa + j * 8192, &tmP, fb, m * BM + j * 64, r,
                               keep);
            if (WMODE == 0) {
              tma_load_2d_hint(sb, &tmQ0, fb, n * 128, r, keep);
              tma_load_2d_hint(sb + 8192, &tmQ0, fb, n * 128 + 64, r, keep);
              tma_load_2d_hint(sb + 16384, &tmQ1, fb, n * 128, r, keep);
              tma_load_2d_hint(sb + 24576, &tmQ1, fb, n * 128 + 64, r, keep);
            } else {
#pragma unroll
              for (int j = 0; j < kBChunks; ++j)
                tma_load_2d_hint(sb + j * 8192, &tmQ0, fb, n * BN + j * 64, r,
                                 keep);
            }
            ++fills;
            if (++stage == WSTAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
      }
      const long long first = fills > WSTAGES ? fills - WSTAGES : 0;
      for (long long f = first; f < fills; ++f)
        mbar_wait(smem_u32(full + (f % WSTAGES)),
                  static_cast<uint32_t>((f / WSTAGES) & 1), nullptr,
                  p.status);
    }
  } else if (warp == 1) {
    // ------------------------------------ tail clearing + MMA issuer ---
    constexpr uint32_t idesc = make_idesc(BM, BN, true, true);
    int stage = 0, acc = 0;
    uint32_t phase = 0, acc_phase = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < total_tiles;
         tile += gridDim.x) {
      const int g = group_of(tpre, p.G, tile);
      bool w_ok = true;
      if (lane == 0)
        w_ok = mbar_wait(smem_u32(tempty + acc), acc_phase ^ 1u, abort_flag,
                         p.status);
      if (!__shfl_sync(0xffffffffu, w_ok, 0)) break;
      tc_fence_after();
      const uint32_t d = tmem_base + acc * kAccCols;
      bool first = true;
      for (int sg = 0; ok && sg < p.n_seg; ++sg) {
        const int r1 = p.seg_base[sg] + __ldg(p.seg_off[sg] + g + 1);
        for (int r = p.seg_base[sg] + __ldg(p.seg_off[sg] + g); r < r1;
             r += BK) {
          const bool got = mbar_wait(smem_u32(full + stage), phase,
                                     abort_flag, p.status);
          if (!__all_sync(0xffffffffu, got)) {
            ok = false;
            break;
          }
          const uint32_t sa = smem_base + stage * kWStage;
          const int valid = min(BK, r1 - r);
          // a short block issues only the K=16 steps that hold valid rows;
          // rows valid .. steps*16 of every 64-column box are cleared (a box
          // is 64 rows of 128 B, so they are contiguous, and the 128-byte
          // swizzle only permutes 16-byte units inside a row)
          const int steps = (valid + 15) >> 4;
          const int nz = (steps * 16 - valid) * 8;  // 16-byte units per box
          if (nz > 0) {
            uint4* base = reinterpret_cast<uint4*>(smem + stage * kWStage) +
                          valid * 8;
#pragma unroll
            for (int box = 0; box < kAChunks + kBChunks; ++box)
              for (int u = lane; u < nz; u += 32)
                base[box * 512 + u] = make_uint4(0, 0, 0, 0);
            fence_proxy_async_smem();
          }
          __syncwarp();
          if (lane == 0) {
            tc_fence_after();
            const uint32_t sb = sa + kAChunks * 8192;
            for (int kk = 0; kk < steps; ++kk) {
              const uint64_t ad = smem_desc(sa + kk * 2048, 8192, 1024);
              const uint64_t bd = smem_desc(sb + kk * 2048, 8192, 1024);
              umma_bf16(d, ad, bd, idesc, (!first || kk != 0) ? 1u : 0u);
            }
            umma_commit(smem_u32(empty + stage));
          }
          __syncwarp();
          first = false;
          if (++stage == WSTAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) break;
      if (lane == 0) umma_commit(smem_u32(tfull + acc));
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
    if (lane == 0) {
      umma_commit(smem_u32(done));
      mbar_wait(smem_u32(done), 0, nullptr, p.status);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------ epilogue ---------
    const int q = warp & 3;
    uint8_t* mybuf = stagebuf + q * kStageBufs * kStageBuf;
    const uint64_t stream = policy_evict_first();
    int acc = 0, nsub = 0;
    uint32_t acc_phase = 0;
    for (int tile = blockIdx.x; tile < total_tiles; tile += gridDim.x) {
      const int g = group_of(tpre, p.G, tile);
      const int local = tile - tpre[g];
      const int n = local % p.n_tiles, m = local / p.n_tiles;
      const int we = p.group_expert ? __ldg(p.group_expert + g) : g;
      bool ok = mbar_wait(smem_u32(tfull + acc), acc_phase, abort_flag,
                          p.status);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      const uint32_t taddr =
          tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * kAccCols;
      const int orow = we * p.m_tiles * BM + m * BM + q * 32;
      const bool add = p.reduce || (p.group_expert != nullptr && ecnt[we] > 1);
#pragma unroll 1
      for (int sub = 0; sub < BN / 32; ++sub, ++nsub) {
        uint32_t r[32];
        tmem_ld32(taddr + sub * 32, r);
        uint8_t* buf = mybuf + (nsub % kStageBufs) * kStageBuf;
        if (lane == 0) bulk_wait_read_free();
        __syncwarp();
        uint4* row = reinterpret_cast<uint4*>(buf + lane * 128);
#pragma unroll
        for (int j = 0; j < 8; ++j)
          row[j ^ (lane & 7)] = make_uint4(r[4 * j], r[4 * j + 1],
                                           r[4 * j + 2], r[4 * j + 3]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          const CUtensorMap* om = &tmO0;
          int col = n * BN + sub * 32;
          if (WMODE == 0) {
            om = sub < 4 ? &tmO0 : &tmO1;
            col = n * 128 + (sub & 3) * 32;
          }
          if (add)
            tma_reduce_add_2d(om, smem_u32(buf), col, orow, stream);
          else
            tma_store_2d(om, smem_u32(buf), col, orow, stream);
          bulk_commit();
        }
      }
      tc_fence_before();
      mbar_arrive(smem_u32(tempty + acc));
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

// ------------------------------------------- two-SM weight gradients ----
// A cluster of two CTAs (tcgen05.mma.cta_group::2) computes a 256 x 256
// tile of dW[e]: each CTA stages its own 128 columns of P (its 128 rows of
// the tile) and one half of the tile's 256 columns of Q (WMODE 0: the
// leader dg, the peer du, over the same 128 columns of F; WMODE 1: the
// leader the first 128, the peer the last 128 columns of H).  A CTA then
// loads 256 operand columns per routed row for its 128 x 256 outputs
// instead of 384, and a stage is 32 KB instead of 48, so more of them fit.
// The TMEM of either CTA holds its 128 rows x 256 columns laid out as in
// the one-CTA kernel (WMODE 0: gate in columns 0-127, up in 128-255), and
// both CTAs run the same epilogue.  The leader issues the MMAs and
// multicasts its commits to both CTAs; the peer's loads complete on the
// leader's barrier.  There is no ragged K=16 step: every group holds a
// multiple of 16 rows in every segment (the regrouped layout, zero pad
// rows included), which the kernel checks before it starts; otherwise it
// raises MOE_DEV_UNALIGNED and writes nothing.
#ifndef MOE_WGRAD2_STAGES
#define MOE_WGRAD2_STAGES 4
#endif
constexpr int W2STAGES = MOE_WGRAD2_STAGES;
constexpr int kW2Stage = 4 * 8192;  // 2 boxes of P + 2 of Q, 64 rows each
constexpr uint32_t kW2Tx = 2 * kW2Stage;  // both CTAs' bytes

__device__ __forceinline__ void tma_load_2d_pair_hint(uint32_t dst,
                                                      const CUtensorMap* m,
                                                      uint32_t bar_cluster,
                                                      int c0, int c1,
                                                      uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile."
      "mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%3, %4}], "
      "[%2], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(bar_cluster), "r"(c0), "r"(c1),
      "l"(policy)
      : "memory");
}

template <int WMODE>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    wgrad_tc2_kernel(const __grid_constant__ CUtensorMap tmP,
                     const __grid_constant__ CUtensorMap tmQ0,
                     const __grid_constant__ CUtensorMap tmQ1,
                     const __grid_constant__ CUtensorMap tmO0,
                     const __grid_constant__ CUtensorMap tmO1, WParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stagebuf = smem + W2STAGES * kW2Stage;  // [4][kStageBufs][4 KB]
  uint64_t* bars =
      reinterpret_cast<uint64_t*>(stagebuf + 4 * kStageBufs * kStageBuf);
  uint64_t* full = bars;
  uint64_t* empty = bars + W2STAGES;
  uint64_t* tfull = bars + 2 * W2STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* done = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* unaligned = reinterpret_cast<int*>(tmem_slot + 2);
  int* wsum = reinterpret_cast<int*>(tmem_slot + 4);  // [16]
  int* tpre = wsum + 16;                               // [G+1]
  int* ecnt = tpre + (p.G + 1);                        // [E]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();  // 0: leader, 1: peer
  const uint32_t smem_base = smem_u32(smem);

  if (threadIdx.x == 0) {
    for (int s = 0; s < W2STAGES; ++s) {
      mbar_init(smem_u32(full + s), 1);
      mbar_init(smem_u32(empty + s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(smem_u32(tfull + a), 1);
      // the leader's four epilogue warps and the peer's relay
      mbar_init(smem_u32(tempty + a), rank == 0 ? kEpilogueThreads / 32 + 1
                                                : kEpilogueThreads / 32);
    }
    mbar_init(smem_u32(done), 1);
    *abort_flag = 0;
    *unaligned = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmP);
    prefetch_tmap(&tmQ0);
    if (WMODE == 0) prefetch_tmap(&tmQ1);
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish_pair();
  }
  build_wgrad_table(p, tpre, wsum);
  for (int e = threadIdx.x; e < p.E; e += blockDim.x) ecnt[e] = 0;
  // every group's rows in every segment: a multiple of 16
  for (int g = threadIdx.x; g < p.G; g += blockDim.x)
    for (int sg = 0; sg < p.n_seg; ++sg)
      if (((__ldg(p.seg_off[sg] + g + 1) - __ldg(p.seg_off[sg] + g)) & 15) !=
          0)
        *unaligned = 1;
  __syncthreads();
  if (p.group_expert != nullptr)
    for (int g = threadIdx.x; g < p.G; g += blockDim.x)
      if (tpre[g + 1] > tpre[g]) atomicAdd(&ecnt[__ldg(p.group_expert + g)], 1);
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers exist before either signals them
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const bool bad = *unaligned != 0;
  if (bad && rank == 0 && threadIdx.x == 0 && p.status)
    atomicOr(p.status, MOE_DEV_UNALIGNED);
  const int total_tiles = bad ? 0 : tpre[p.G];
  const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;

  if (warp == 0) {
    // ---------------------------------------- TMA producer (both CTAs) ---
    if (lane == 0) {
      const uint64_t keep = policy_evict_last();
      const CUtensorMap* mq = (WMODE == 0 && rank == 1) ? &tmQ1 : &tmQ0;
      int stage = 0;
      uint32_t phase = 0;
      long long fills = 0;
      bool ok = true;
      for (int tile = pair; ok && tile < total_tiles; tile += npairs) {
        const int g = group_of(tpre, p.G, tile);
        const int local = tile - tpre[g];
        const int n = local % p.n_tiles, m = local / p.n_tiles;
        const int pcol = m * 2 * BM + static_cast<int>(rank) * BM;
        const int qcol = WMODE == 0 ? n * 128 : n * 256 + rank * 128;
        for (int sg = 0; ok && sg < p.n_seg; ++sg) {
          const int r1 = p.seg_base[sg] + __ldg(p.seg_off[sg] + g + 1);
          for (int r = p.seg_base[sg] + __ldg(p.seg_off[sg] + g); r < r1;
               r += BK) {
            if (p.stall_after_fills >= 0 && fills >= p.stall_after_fills) {
              ok = false;  // test hook: leave the MMA waiting
              break;
            }
            if (!mbar_wait(smem_u32(empty + stage), phase ^ 1u, abort_flag,
                           p.status)) {
              ok = false;
              break;
            }
            const uint32_t fb = map_to_rank(smem_u32(full + stage), 0);
            if (rank == 0) mbar_expect_tx(smem_u32(full + stage), kW2Tx);
            const uint32_t sa = smem_base + stage * kW2Stage;
            tma_load_2d_pair_hint(sa, &tmP, fb, pcol, r, keep);
            tma_load_2d_pair_hint(sa + 8192, &tmP, fb, pcol + 64, r, keep);
            tma_load_2d_pair_hint(sa + 16384, mq, fb, qcol, r, keep);
            tma_load_2d_pair_hint(sa + 24576, mq, fb, qcol + 64, r, keep);
            ++fills;
            if (++stage == W2STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
      }
      // Drain: the leader's full barriers count both CTAs' bytes.
      if (rank == 0) {
        const long long first = fills > W2STAGES ? fills - W2STAGES : 0;
        for (long long f = first; f < fills; ++f)
          mbar_wait(smem_u32(full + (f % W2STAGES)),
                    static_cast<uint32_t>((f / W2STAGES) & 1), nullptr,
                    p.status);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------- MMA issuer (leader) ------
    if (lane == 0 && rank == 0) {
      constexpr uint32_t idesc = make_idesc(2 * BM, 256, true, true);
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      for (int tile = pair; ok && tile < total_tiles; tile += npairs) {
        const int g = group_of(tpre, p.G, tile);
        if (!mbar_wait(smem_u32(tempty + acc), acc_phase ^ 1u, abort_flag,
                       p.status))
          break;
        tc_fence_after();
        const uint32_t d = tmem_base + acc * kAccCols;
        bool first = true;
        for (int sg = 0; ok && sg < p.n_seg; ++sg) {
          const int r1 = p.seg_base[sg] + __ldg(p.seg_off[sg] + g + 1);
          for (int r = p.seg_base[sg] + __ldg(p.seg_off[sg] + g); r < r1;
               r += BK) {
            if (!mbar_wait(smem_u32(full + stage), phase, abort_flag,
                           p.status)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t sa = smem_base + stage * kW2Stage;
            const uint32_t sb = sa + 16384;
            const int steps = min(BK, r1 - r) >> 4;  // whole K=16 steps
            for (int kk = 0; kk < steps; ++kk) {
              const uint64_t ad = smem_desc(sa + kk * 2048, 8192, 1024);
              const uint64_t bd = smem_desc(sb + kk * 2048, 8192, 1024);
              umma_bf16_pair(d, ad, bd, idesc, (!first || kk != 0) ? 1u : 0u);
            }
            umma_commit_pair_mc(smem_u32(empty + stage));
            first = false;
            if (++stage == W2STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
        if (!ok) break;
        umma_commit_pair_mc(smem_u32(tfull + acc));
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      umma_commit_pair(smem_u32(done));
      mbar_wait(smem_u32(done), 0, nullptr, p.status);
    } else if (lane == 0) {
      // ------------------------------ TMEM-empty relay (peer) -----------
      // the peer's epilogue warps arrive on its own barrier; this thread
      // forwards each completed phase to the leader with one cluster-scope
      // arrival, so that no epilogue warp waits on a cluster-wide fence
      int acc = 0;
      uint32_t acc_phase = 0;
      for (int tile = pair; tile < total_tiles; tile += npairs) {
        if (!mbar_wait(smem_u32(tempty + acc), acc_phase, abort_flag,
                       p.status))
          break;
        mbar_arrive_cluster(map_to_rank(smem_u32(tempty + acc), 0));
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
    }
  } else {
    // ---------------------------------------- epilogue (both CTAs) -----
    const int q = warp & 3;
    uint8_t* mybuf = stagebuf + q * kStageBufs * kStageBuf;
    const uint64_t stream = policy_evict_first();
    int acc = 0, nsub = 0;
    uint32_t acc_phase = 0;
    for (int tile = pair; tile < total_tiles; tile += npairs) {
      const int g = group_of(tpre, p.G, tile);
      const int local = tile - tpre[g];
      const int n = local % p.n_tiles, m = local / p.n_tiles;
      const int we = p.group_expert ? __ldg(p.group_expert + g) : g;
      bool ok = mbar_wait(smem_u32(tfull + acc), acc_phase, abort_flag,
                          p.status);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      const uint32_t taddr =
          tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * kAccCols;
      const int orow = (we * p.m_tiles + m) * 2 * BM +
                       static_cast<int>(rank) * BM + q * 32;
      const bool add = p.reduce || (p.group_expert != nullptr && ecnt[we] > 1);
#pragma unroll 1
      for (int sub = 0; sub < 8; ++sub, ++nsub) {
        uint32_t r[32];
        tmem_ld32(taddr + sub * 32, r);
        uint8_t* buf = mybuf + (nsub % kStageBufs) * kStageBuf;
        if (lane == 0) bulk_wait_read_free();
        __syncwarp();
        uint4* row = reinterpret_cast<uint4*>(buf + lane * 128);
#pragma unroll
        for (int j = 0; j < 8; ++j)
          row[j ^ (lane & 7)] = make_uint4(r[4 * j], r[4 * j + 1],
                                           r[4 * j + 2], r[4 * j + 3]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          const CUtensorMap* om = &tmO0;
          int col = n * 256 + sub * 32;
          if (WMODE == 0) {
            om = sub < 4 ? &tmO0 : &tmO1;
            col = n * 128 + (sub & 3) * 32;
          }
          if (add)
            tma_reduce_add_2d(om, smem_u32(buf), col, orow, stream);
          else
            tma_store_2d(om, smem_u32(buf), col, orow, stream);
          bulk_commit();
        }
      }
      // one arrival per warp, on its own CTA's barrier, once its lanes'
      // TMEM loads are done (the peer's relay forwards it to the leader)
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(tempty + acc));
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // neither CTA leaves while its peer may still use it
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

// Store mode: zeroes dW[e] of every expert that does not have exactly one
// group with rows -- none (no tile writes it) or several (its tiles add onto
// it).  Grid (E, blocks), 16-byte stores.
__global__ void zero_experts_kernel(WParams p, float* a, float* b,
                                    long long per_expert) {
  const int e = blockIdx.x;
  int n = 0;
  if (p.group_expert == nullptr) {
    n = wgrad_rows(p, e) > 0 ? 1 : 0;
  } else {
    for (int g = 0; g < p.G; ++g)
      if (__ldg(p.group_expert + g) == e && wgrad_rows(p, g) > 0) ++n;
  }
  if (n == 1) return;
  const long long n4 = per_expert / 4;
  float4* pa = reinterpret_cast<float4*>(a + e * per_expert);
  float4* pb = b ? reinterpret_cast<float4*>(b + e * per_expert) : nullptr;
  const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
  for (long long i = blockIdx.y * blockDim.x + threadIdx.x; i < n4;
       i += static_cast<long long>(gridDim.y) * blockDim.x) {
    pa[i] = z;
    if (pb) pb[i] = z;
  }
}

size_t smem_bytes_wgrad(int G, int E) {
  return 1024 + WSTAGES * kWStage + 4 * kStageBufs * kStageBuf +
         8 * (2 * WSTAGES + 5) +
         16 + 4 * (16 + G + 1 + E) + 64;
}

size_t smem_bytes_wgrad2(int G, int E) {
  return 1024 + W2STAGES * kW2Stage + 4 * kStageBufs * kStageBuf +
         8 * (2 * W2STAGES + 5) + 16 + 4 * (16 + G + 1 + E) + 64;
}

template <int WMODE>
cudaError_t launch_wgrad2(const CUtensorMap& pm, const CUtensorMap& q0,
                          const CUtensorMap& q1, const CUtensorMap& o0,
                          const CUtensorMap& o1, WParams p,
                          cudaStream_t s) {
  p.stall_after_fills = g_stall_after_fills.load();
  const size_t smem = smem_bytes_wgrad2(p.G, p.E);
  int dev = 0, sms = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (err != cudaSuccess) return err;
  err = cudaFuncSetAttribute(wgrad_tc2_kernel<WMODE>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  const int grid = sms & ~1;  // whole CTA pairs
  wgrad_tc2_kernel<WMODE><<<grid, kThreads, smem, s>>>(pm, q0, q1, o0, o1, p);
  return cudaGetLastError();
}

template <int WMODE, int BN>
cudaError_t launch_wgrad(const CUtensorMap& pm, const CUtensorMap& q0,
                         const CUtensorMap& q1, const CUtensorMap& o0,
                         const CUtensorMap& o1, const WParams& p,
                         cudaStream_t s) {
  const size_t smem = smem_bytes_wgrad(p.G, p.E);
  int dev = 0, sms = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (err != cudaSuccess) return err;
  err = cudaFuncSetAttribute(wgrad_tc_kernel<WMODE, BN>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  wgrad_tc_kernel<WMODE, BN><<<sms, kThreads, smem, s>>>(pm, q0, q1, o0, o1,
                                                          p);
  return cudaGetLastError();
}

}  // namespace tc

// Weight gradients over row segments (each {group offsets, first row}),
// all inside buffers of `rows_total` rows.  flags: kWgradAccumulate adds
// into dW, otherwise every expert's dW is overwritten (experts without rows
// get zeros); kWgradRows16 (every group holds a multiple of 16 rows in
// every segment) takes the two-SM kernel where the gradient's row count is
// a multiple of 256.
cudaError_t launch_wgrad_bf16(const moe_config_t& c, const Groups& g,
                              const WgradSegment* seg, int n_seg,
                              int64_t rows_total, const void* x_sorted,
                              const void* dg, const void* du, const void* h,
                              const void* dy_sorted, float* dw_gate,
                              float* dw_up, float* dw_down, int flags,
                              int parts, int32_t* status, cudaStream_t s) {
  const bool accumulate = (flags & kWgradAccumulate) != 0;
  const bool rows16 = (flags & kWgradRows16) != 0;
  const bool gu = (parts & kWgradGateUp) != 0;
  const bool dn = (parts & kWgradDown) != 0;
  const uint64_t E = static_cast<uint64_t>(c.E);
  const uint64_t rows = static_cast<uint64_t>(std::max<int64_t>(rows_total, 1));
  const long long per_expert = static_cast<long long>(c.H) * c.F;
  cudaError_t e = cudaSuccess;
  const int bnd = c.H % 256 == 0 ? 256 : 128;
  CUtensorMap px, qg, qu, og, ou, ph, qd, od;
  if (gu && (!tc::make_map(&px, x_sorted, c.H, rows, 64, 64) ||
             !tc::make_map(&qg, dg, c.F, rows, 64, 64) ||
             !tc::make_map(&qu, du, c.F, rows, 64, 64) ||
             !tc::make_map(&og, dw_gate, c.F, E * c.H, 32, 32, true) ||
             !tc::make_map(&ou, dw_up, c.F, E * c.H, 32, 32, true)))
    return cudaErrorInvalidValue;
  if (dn && (!tc::make_map(&ph, h, c.F, rows, 64, 64) ||
             !tc::make_map(&qd, dy_sorted, c.H, rows, 64, 64) ||
             !tc::make_map(&od, dw_down, c.H, E * c.F, 32, 32, true)))
    return cudaErrorInvalidValue;
  for (int s0 = 0; s0 < std::max(n_seg, 1); s0 += tc::kMaxSeg) {
    tc::WParams p{};
    p.n_seg = std::min(tc::kMaxSeg, n_seg - s0);
    for (int i = 0; i < p.n_seg; ++i) {
      p.seg_off[i] = seg[s0 + i].group_offsets;
      p.seg_base[i] = seg[s0 + i].first_row;
    }
    p.group_expert = g.map;
    p.G = g.n;
    p.E = c.E;
    p.reduce = (accumulate || s0 > 0) ? 1 : 0;
    p.status = status;
    if (!p.reduce) {
      // experts without rows (no tile writes their dW) and duplicated
      // experts (their groups' tiles add onto it) start from zeros
      const dim3 grid(static_cast<unsigned>(c.E), 16);
      if (gu)
        tc::zero_experts_kernel<<<grid, 256, 0, s>>>(p, dw_gate, dw_up,
                                                     per_expert);
      if (dn)
        tc::zero_experts_kernel<<<grid, 256, 0, s>>>(p, dw_down, nullptr,
                                                     per_expert);
      if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    if (p.n_seg == 0) break;
    if (gu) {
      p.n_tiles = c.F / 128;
      if (rows16 && c.H % 256 == 0) {
        p.m_tiles = c.H / 256;
        e = tc::launch_wgrad2<0>(px, qg, qu, og, ou, p, s);
      } else {
        p.m_tiles = c.H / tc::BM;
        e = tc::launch_wgrad<0, 256>(px, qg, qu, og, ou, p, s);
      }
      if (e != cudaSuccess) return e;
    }
    if (dn) {
      p.n_tiles = c.H / bnd;
      if (rows16 && c.F % 256 == 0 && bnd == 256) {
        p.m_tiles = c.F / 256;
        e = tc::launch_wgrad2<1>(ph, qd, qd, od, od, p, s);
      } else {
        p.m_tiles = c.F / tc::BM;
        e = bnd == 256 ? tc::launch_wgrad<1, 256>(ph, qd, qd, od, od, p, s)
                       : tc::launch_wgrad<1, 128>(ph, qd, qd, od, od, p, s);
      }
      if (e != cudaSuccess) return e;
    }
  }
  return cudaSuccess;
}

}  // namespace moe
