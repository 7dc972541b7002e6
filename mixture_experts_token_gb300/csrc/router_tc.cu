// Router logits for batches too small to fill the GPU: K split over a
// thread-block cluster.
//
// "Support moe_dropless_fallback=layer on the ragged all-to-all MoE path"
// (MaxText pull request 5920), section How: the overflow check is computed
// from the router's top-k, downstream of the router's dense projection of
// the tokens onto the experts, logits[t, e] = sum_h x[t, h] Wr[h, e]
// (+ offset[t, e]), accumulated in float32.
//
// The tile of the one-group GEMM (gmm_tc.cu, mode 5) is 128 tokens x 128
// experts over the whole reduction (H / 64 k-blocks, 112 at H = 7168); a
// batch of T tokens makes ceil(T / 128) * E / 128 tiles, 16 at T = 1024,
// and leaves most SMs idle while each tile walks its long k-loop.  Here a
// cluster of S CTAs shares one tile: CTA r accumulates k-blocks
// [r * ceil(kb / S), ...) in its own tensor memory (TMA-staged operands,
// tcgen05.mma M = 128, N = 128, as mode 5), writes its float32 partial
// tile to its shared memory, and after a cluster barrier each CTA reduces
// 128 / S of the tile's rows, reading the S partials through distributed
// shared memory in rank order (so each logit is ((p_0 + p_1) + ...) +
// offset whatever CTA computes it), and stores them.  A second cluster
// barrier keeps every CTA's partial alive until its peers have read it.
// The launch picks the form and the cluster size from the clusters the GPU
// can hold at once (larger clusters fit fewer times in its SM groups: at
// 1024 tokens, clusters of 4 measured 18.8 us against 24.8 us for 8 and
// 49.9 us unsplit; at one token, 8 measured 10.8 us against 14.7 us for 4).
//
// Every mbarrier wait is bounded (2 s); on expiry the kernel raises
// MOE_DEV_TIMEOUT, the other roles stop, the producer drains its loads, and
// every thread still passes both cluster barriers, so no CTA of the
// cluster waits for one that left.
#include <atomic>

#include "tc_common.cuh"

namespace moe {
namespace tc {

// The GEMMs' test hook (gmm_tc.cu): stop the producer after this many stage
// fills (-1: never), so that the next wait runs out.
extern std::atomic<long long> g_stall_after_fills;

namespace {

constexpr int kRBN = 128;                              // experts per tile
constexpr int kRStages = 4;
constexpr int kRStage = BM * BK * 2 + BK * kRBN * 2;   // 32 KB
constexpr int kPartLd = kRBN + 4;   // partial row stride in floats
constexpr int kMaxSplits = 8;       // portable cluster size

struct RouterParams {
  int T, E, kblocks, S, n_tiles;
  const float* offset;  // [T, E] or null
  float* logits;        // [T, E]
  int32_t* status;
  long long stall_after_fills;  // tests of the timeout path only (-1: off)
};

__device__ __forceinline__ float4 ld_cluster_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

__global__ void __launch_bounds__(kThreads, 1)
    router_splitk_kernel(const __grid_constant__ CUtensorMap tmA,
                         const __grid_constant__ CUtensorMap tmB,
                         RouterParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kRStages * kRStage);
  uint64_t* full = bars;
  uint64_t* empty = bars + kRStages;
  uint64_t* done = bars + 2 * kRStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  // after the k-loop the ring holds this CTA's partial tile [128][kPartLd]
  float* part = reinterpret_cast<float*>(smem);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t smem_base = smem_u32(smem);
  const int S = p.S;
  const int rank = static_cast<int>(cluster_rank());
  const int tile = blockIdx.x / S;
  const int m = tile / p.n_tiles, n = tile - (tile / p.n_tiles) * p.n_tiles;
  const int per = (p.kblocks + S - 1) / S;
  const int kb0 = min(p.kblocks, rank * per);
  const int kb1 = min(p.kblocks, kb0 + per);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kRStages; ++s) {
      mbar_init(smem_u32(full + s), 1);
      mbar_init(smem_u32(empty + s), 1);
    }
    mbar_init(smem_u32(done), 1);
    *abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kRBN);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------ TMA producer -----
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      long long fills = 0;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (p.stall_after_fills >= 0 && fills >= p.stall_after_fills)
          break;  // test hook: leave the MMA warp waiting
        if (!mbar_wait(smem_u32(empty + stage), phase ^ 1u, abort_flag,
                       p.status))
          break;
        const uint32_t fb = smem_u32(full + stage);
        mbar_expect_tx(fb, kRStage);
        const uint32_t sa = smem_base + stage * kRStage;
        const uint32_t sb = sa + BM * BK * 2;
        tma_load_2d(sa, &tmA, fb, kb * BK, m * BM);
        tma_load_2d(sb, &tmB, fb, n * kRBN, kb * BK);
        tma_load_2d(sb + 8192, &tmB, fb, n * kRBN + 64, kb * BK);
        ++fills;
        if (++stage == kRStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      // Drain: every load issued has landed before the ring is reused.
      const long long first = fills > kRStages ? fills - kRStages : 0;
      for (long long f = first; f < fills; ++f)
        mbar_wait(smem_u32(full + (f % kRStages)),
                  static_cast<uint32_t>((f / kRStages) & 1), nullptr,
                  p.status);
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer -------
    if (lane == 0) {
      constexpr uint32_t idesc = make_idesc(BM, kRBN, true);
      int stage = 0;
      uint32_t phase = 0;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!mbar_wait(smem_u32(full + stage), phase, abort_flag, p.status))
          break;
        tc_fence_after();
        const uint32_t sa = smem_base + stage * kRStage;
        const uint32_t sb = sa + BM * BK * 2;
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk)
          umma_bf16(tmem_base, smem_desc(sa + kk * 32, 16, 1024),
                    smem_desc(sb + kk * 2048, 8192, 1024), idesc,
                    (kb > kb0 || kk > 0) ? 1u : 0u);
        umma_commit(smem_u32(empty + stage));
        if (++stage == kRStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      // all MMAs issued by this thread are complete (a CTA with an empty
      // k-slice issues none and the epilogue does not wait for them); the
      // drain waits for them itself, bounded by time alone, so that the
      // tensor memory is not freed under an MMA after a timeout
      if (kb1 > kb0) {
        umma_commit(smem_u32(done));
        mbar_wait(smem_u32(done), 0, nullptr, p.status);
      }
    }
  } else {
    // ------------------- epilogue: the partial tile to shared memory ---
    const int q = warp & 3;
    const int row = q * 32 + lane;
    const bool ok =
        kb1 > kb0 && mbar_wait(smem_u32(done), 0, abort_flag, p.status);
    tc_fence_after();
    float4* dst = reinterpret_cast<float4*>(part + row * kPartLd);
    if (__all_sync(0xffffffffu, ok)) {
#pragma unroll 1
      for (int c = 0; c < kRBN; c += 32) {
        uint32_t r[32];
        tmem_ld32(tmem_base + (static_cast<uint32_t>(q * 32) << 16) + c, r);
#pragma unroll
        for (int v = 0; v < 8; ++v)
          dst[c / 4 + v] = make_float4(
              __uint_as_float(r[4 * v]), __uint_as_float(r[4 * v + 1]),
              __uint_as_float(r[4 * v + 2]), __uint_as_float(r[4 * v + 3]));
      }
    } else {
      // an empty k-slice contributes zeros (no accumulator was written);
      // after a timeout the logits are not used (MOE_DEV_TIMEOUT is set)
      for (int v = 0; v < kRBN / 4; ++v)
        dst[v] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // every CTA's partial tile is written

  // ------------------------- reduce this CTA's share of the tile's rows --
  const int rows_per = (BM + S - 1) / S;
  const int r0 = min(BM, rank * rows_per), r1 = min(BM, r0 + rows_per);
  const int units = (r1 - r0) * (kRBN / 4);
  for (int i = threadIdx.x; i < units; i += blockDim.x) {
    const int row = r0 + i / (kRBN / 4), c4 = i % (kRBN / 4);
    const int t = m * BM + row;
    if (t >= p.T) continue;
    const uint32_t local = smem_u32(part + row * kPartLd + c4 * 4);
    float4 acc = ld_cluster_f4(map_to_rank(local, 0));
    for (int r = 1; r < S; ++r) {
      const float4 v = ld_cluster_f4(map_to_rank(local, r));
      acc.x += v.x;
      acc.y += v.y;
      acc.z += v.z;
      acc.w += v.w;
    }
    const long long o = static_cast<long long>(t) * p.E + n * kRBN + c4 * 4;
    if (p.offset) {
      const float4 b = __ldg(reinterpret_cast<const float4*>(p.offset + o));
      acc.x += b.x;
      acc.y += b.y;
      acc.z += b.z;
      acc.w += b.w;
    }
    *reinterpret_cast<float4*>(p.logits + o) = acc;
  }
  __syncwarp();
  cluster_sync();  // the peers have read this CTA's partial tile

  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kRBN);
  }
}

size_t router_splitk_smem() {
  return 1024 + kRStages * kRStage + 8 * (2 * kRStages + 1) + 16;
}

// Per device, per cluster size s in {2, 4, 8}: the clusters that can be
// resident at once (+1; 0: not yet queried), and whether the kernel's
// shared-memory attribute is set, so that a launch repeats no host query.
constexpr int kMaxDevices = 64;
std::atomic<int> g_clusters[kMaxDevices][kMaxSplits + 1];
std::atomic<int> g_attr_set[kMaxDevices];

cudaLaunchConfig_t launch_config(int tiles, int splits, size_t smem,
                                 cudaStream_t s, cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(tiles * splits));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(splits);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

// The kernel's dynamic shared memory allowance (once per device): needed
// before the occupancy query as well as before a launch.
cudaError_t set_smem_attribute(int dev) {
  std::atomic<int>* set =
      dev >= 0 && dev < kMaxDevices ? &g_attr_set[dev] : nullptr;
  if (set && set->load() != 0) return cudaSuccess;
  const cudaError_t err = cudaFuncSetAttribute(
      router_splitk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
      static_cast<int>(router_splitk_smem()));
  if (err == cudaSuccess && set) set->store(1);
  return err;
}

// Resident clusters of `splits` CTAs (0 if none can be placed).
cudaError_t resident_clusters(int dev, int splits, int* n) {
  std::atomic<int>* slot =
      dev >= 0 && dev < kMaxDevices ? &g_clusters[dev][splits] : nullptr;
  if (slot && slot->load() > 0) {
    *n = slot->load() - 1;
    return cudaSuccess;
  }
  cudaError_t err = set_smem_attribute(dev);
  if (err != cudaSuccess) return err;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg =
      launch_config(1, splits, router_splitk_smem(), nullptr, attr);
  err = cudaOccupancyMaxActiveClusters(n, router_splitk_kernel, &cfg);
  if (err != cudaSuccess) return err;
  if (slot) slot->store(*n + 1);
  return cudaSuccess;
}

}  // namespace
}  // namespace tc

// The router's tensor-core launch: the one-group GEMM (gmm_tc.cu), or the
// reduction split over clusters of 2, 4 or 8 CTAs when that takes fewer
// k-block steps per SM.  Cost of a form: the waves of its resident CTAs or
// clusters times the k-blocks each walks, plus a fixed 6 for its prologue,
// epilogue and (split) reduction; ties keep the fewer splits.
cudaError_t launch_router_tc(const moe_config_t& c, const void* x,
                             const void* w_router, const float* offset,
                             float* logits, int32_t* status,
                             cudaStream_t s) {
  using namespace tc;
  if (c.T == 0) return cudaSuccess;
  int dev = 0, sms = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err == cudaSuccess)
    err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (err != cudaSuccess) return err;
  const int tiles = (c.T + BM - 1) / BM * (c.E / kRBN);
  const int kblocks = c.H / BK;
  constexpr int kOverhead = 6;
  long long best = static_cast<long long>((tiles + sms - 1) / sms) *
                   (kblocks + kOverhead);
  int splits = 1;
  if (c.E % kRBN == 0 && c.H % BK == 0) {
    for (int sp = 2; sp <= kMaxSplits && sp <= kblocks; sp *= 2) {
      int n = 0;
      if ((err = resident_clusters(dev, sp, &n)) != cudaSuccess) return err;
      if (n < 1) continue;
      const long long cost = static_cast<long long>((tiles + n - 1) / n) *
                             ((kblocks + sp - 1) / sp + kOverhead);
      if (cost < best) {
        best = cost;
        splits = sp;
      }
    }
  }
  if (splits == 1)
    return launch_router_bf16(c, x, w_router, offset, logits, status, s);
  CUtensorMap a, b;
  if (!make_map(&a, x, c.H, static_cast<uint64_t>(c.T), 64, BM) ||
      !make_map(&b, w_router, c.E, c.H, 64, 64))
    return cudaErrorInvalidValue;
  RouterParams p{c.T, c.E, kblocks, splits, c.E / kRBN, offset, logits,
                 status, g_stall_after_fills.load()};
  const size_t smem = router_splitk_smem();
  if ((err = set_smem_attribute(dev)) != cudaSuccess) return err;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = launch_config(tiles, splits, smem, s, attr);
  return cudaLaunchKernelEx(&cfg, router_splitk_kernel, a, b, p);
}

}  // namespace moe
