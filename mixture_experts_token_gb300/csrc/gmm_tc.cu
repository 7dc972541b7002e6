// Grouped GEMM SwiGLU expert FFN on the 5th-generation tensor cores
// (tcgen05, accumulators in tensor memory, operands staged by TMA).
//
// "Moe dynamic redundancy" (MaxText pull request 4760), review comments:
// the expert FFN is a grouped matmul over experts with ragged group_sizes
// (megablox / gmm), expert weights w0 of shape [E, H, H_ffn].  The SwiGLU
// form is h = silu(x Wg) * (x Wu), y = h Wd.
//
// One persistent CTA per SM, 6 warps:
//   warp 0  TMA producer (one thread): A tile [128 rows x 64 k] of the
//           expert-sorted rows, B tile [64 k x BN] of the expert's weights,
//           into a STAGES-deep ring of 128-byte-swizzled shared buffers.
//   warp 1  TMEM owner and MMA issuer (one thread): tcgen05.mma kind::f16,
//           M=128 x N=BN x K=16, fp32 accumulators in tensor memory, two
//           accumulators of 256 columns so the epilogue of one tile
//           overlaps the main loop of the next.
//   warps 2-5  epilogue: tcgen05.ld of the accumulator (one TMEM lane = one
//           row per thread), SwiGLU (GEMM1) or plain (GEMM2), bf16 stores.
// Tiles are (expert e, n-tile, m-tile) with m innermost: the CTAs running at
// one time work on the same weight tile of a hot expert, so it comes from
// HBM once and from L2 after.  Rows past an expert's group end are computed
// (on the next expert's rows or TMA zero fill) and masked at the store; each
// output row depends only on its own input row, so that garbage never mixes
// into a valid row and a row's value does not depend on its tile position.
//
// Operand layouts (no repacking of the [E, H, F] / [E, F, H] weights):
//   A (rows, K-major): TMA box {64 k, 128 rows}, SWIZZLE_128B -> 8-row atoms
//     of 1024 B; descriptor SBO = 1024, start advanced 32 B per K=16 step.
//   B (weights, N-major = "MN-major"): TMA box {64 n, 64 k}, SWIZZLE_128B,
//     one box per 64-column chunk; descriptor LBO = 8192 (next 64-column
//     chunk), SBO = 1024 (next 8 k-rows), start advanced 2048 B per K=16.
//   GEMM1 issues one N=256 MMA whose columns 0-127 are the gate projection
//     and 128-255 the up projection of the same 128 output columns.
//
// Two-SM form (gmm_tc2_kernel, used when the output tile is 256 wide): a
// cluster of two CTAs on one TPC shares each M=256 x N=256 tile through
// tcgen05.mma.cta_group::2.  Each CTA stages its own 128 rows of A and half
// of B (for GEMM1: the leader the gate columns, the peer the up columns) in
// 6 stages of 32 KB, so a stage of compute needs a third less shared memory
// and more loads are in flight.  The leader issues the MMAs and multicasts
// its commits to both CTAs; the peer's TMA loads complete on the leader's
// barrier; both CTAs run an epilogue on their own 128 rows of TMEM.
//
// Every wait is bounded (2 s of %globaltimer); on expiry the kernel raises
// MOE_DEV_TIMEOUT in the status word, tells the other roles to stop, drains
// its own TMA loads and MMAs, frees its tensor memory and returns.
#include <cuda.h>
#include <cuda_bf16.h>

#include <atomic>
#include <mutex>

#include "internal.h"

namespace moe {
namespace tc {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int STAGES = 4;
constexpr int kThreads = 192;
constexpr int kEpilogueThreads = 128;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCols = 256;
constexpr uint64_t kWaitLimitNs = 2000000000ull;

template <int BN>
struct Tile {
  static constexpr int kABytes = BM * BK * 2;
  static constexpr int kBBytes = BK * BN * 2;
  static constexpr int kStage = kABytes + kBBytes;
  static constexpr int kChunks = BN / 64;
};

struct Params {
  const int32_t* group_offsets;  // [E+1]
  const int32_t* group_expert;   // [E] weights of each group; null: identity
  int E;                         // row groups
  int K;        // reduction length: H (GEMM1) or F (GEMM2)
  int n_tiles;  // output column tiles per expert
  __nv_bfloat16* out;
  int out_ld;   // F (GEMM1) or H (GEMM2)
  int32_t* status;
  // Backward and saving modes: second/third outputs and epilogue inputs.
  __nv_bfloat16* out2 = nullptr;        // MODE 4: u;  MODE 2: du
  __nv_bfloat16* out3 = nullptr;        // MODE 4: g
  const __nv_bfloat16* aux_g = nullptr; // MODE 2: g
  const __nv_bfloat16* aux_u = nullptr; // MODE 2: u
  int k_split = 0;                      // MODE 3: k-blocks from the 1st pair
  // Tests of the timeout path only: the producer stops after this many
  // stage fills (-1: never), so the MMA warp's next wait runs out.
  long long stall_after_fills = -1;
};

std::atomic<long long> g_stall_after_fills{-1};

// ---------------------------------------------------------------- PTX ----
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar),
               "r"(count)
               : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(
                   bar),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait; false when it gave up (or another role already did).
// A drain passes abort_flag = nullptr: it waits for its own copies or MMAs
// even after another role gave up, bounded by the time limit alone.
__device__ __noinline__ bool mbar_wait(uint32_t bar, uint32_t parity,
                                       volatile int* abort_flag,
                                       int32_t* status) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  uint32_t spins = 0;
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((++spins & 63u) == 0) {
      if (abort_flag && *abort_flag) return false;
      if (globaltimer() - t0 > kWaitLimitNs) {
        if (abort_flag) *abort_flag = 1;
        if (status) atomicOr(status, MOE_DEV_TIMEOUT);
        return false;
      }
    }
  }
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m))
               : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* m,
                                            uint32_t bar, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::"
      "complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(c0), "r"(c1)
      : "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t cols) {
  asm volatile(
      "tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
          dst_smem),
      "r"(cols)
      : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::
                   : "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t cols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(
                   taddr),
               "r"(cols)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem], bf16 x bf16 -> fp32, one thread issues.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc,
                                          uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(
          d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on an mbarrier once every tcgen05 op this thread issued completed.
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 "
      "[%0];" ::"r"(bar)
      : "memory");
}

// TMEM -> registers: 32 columns of one lane per thread, with the wait for
// completion in the same statement so no use of the registers can be
// scheduled before it.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n"
      "tcgen05.wait::ld.sync.aligned;\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void tmem_ld32x2(uint32_t ta, uint32_t tb, uint32_t (&a)[32],
                                            uint32_t (&b)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%64];\n"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%65];\n"
      "tcgen05.wait::ld.sync.aligned;\n"
      : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3]), "=r"(a[4]), "=r"(a[5]), "=r"(a[6]), "=r"(a[7]), "=r"(a[8]), "=r"(a[9]), "=r"(a[10]), "=r"(a[11]), "=r"(a[12]), "=r"(a[13]), "=r"(a[14]), "=r"(a[15]), "=r"(a[16]), "=r"(a[17]), "=r"(a[18]), "=r"(a[19]), "=r"(a[20]), "=r"(a[21]), "=r"(a[22]), "=r"(a[23]), "=r"(a[24]), "=r"(a[25]), "=r"(a[26]), "=r"(a[27]), "=r"(a[28]), "=r"(a[29]), "=r"(a[30]), "=r"(a[31]), "=r"(b[0]), "=r"(b[1]), "=r"(b[2]), "=r"(b[3]), "=r"(b[4]), "=r"(b[5]), "=r"(b[6]), "=r"(b[7]), "=r"(b[8]), "=r"(b[9]), "=r"(b[10]), "=r"(b[11]), "=r"(b[12]), "=r"(b[13]), "=r"(b[14]), "=r"(b[15]), "=r"(b[16]), "=r"(b[17]), "=r"(b[18]), "=r"(b[19]), "=r"(b[20]), "=r"(b[21]), "=r"(b[22]), "=r"(b[23]), "=r"(b[24]), "=r"(b[25]), "=r"(b[26]), "=r"(b[27]), "=r"(b[28]), "=r"(b[29]), "=r"(b[30]), "=r"(b[31])
      : "r"(ta), "r"(tb)
      : "memory");
}

// ------------------------------------------------------- CTA pair ------
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// The same shared-memory variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
               : "=r"(r)
               : "r"(addr), "r"(rank));
  return r;
}

__device__ __forceinline__ void cluster_sync() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::
          : "memory");
}

// TMA load into this CTA's shared memory, completing on an mbarrier that
// may sit in either CTA of the pair (a shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst,
                                                 const CUtensorMap* m,
                                                 uint32_t bar_cluster, int c0,
                                                 int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile."
      "mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(bar_cluster), "r"(c0), "r"(c1)
      : "memory");
}

__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar_cluster) {
  asm volatile(
      "mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(
          bar_cluster)
      : "memory");
}

__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem,
                                                uint32_t cols) {
  asm volatile(
      "tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
          dst_smem),
      "r"(cols)
      : "memory");
}

__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::
                   : "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr,
                                                  uint32_t cols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(
                   taddr),
               "r"(cols)
               : "memory");
}

// D (both CTAs' TMEM, 128 rows each) (+)= A (both CTAs' smem, 128 rows
// each) * B (both CTAs' smem, N/2 columns each); one thread of the leader.
__device__ __forceinline__ void umma_bf16_pair(uint32_t d_tmem, uint64_t adesc,
                                               uint64_t bdesc, uint32_t idesc,
                                               uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(
          d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on the barrier at this shared-memory offset in both CTAs once the
// leader's tcgen05 ops are complete.
__device__ __forceinline__ void umma_commit_pair_mc(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster."
      "multicast::cluster.b64 [%0], %1;" ::"r"(bar),
      "h"(static_cast<uint16_t>(3))
      : "memory");
}

__device__ __forceinline__ void umma_commit_pair(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 "
      "[%0];" ::"r"(bar)
      : "memory");
}

// Shared-memory matrix descriptor (tcgen05 format): start address, leading
// and stride byte offsets (all >> 4), descriptor version 1 at bit 46, and
// the 128-byte swizzle mode (2) in bits 61-63.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo,
                                              uint32_t sbo) {
  return static_cast<uint64_t>((addr & 0x3FFFFu) >> 4) |
         (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) |
         (1ull << 46) | (2ull << 61);
}

// Instruction descriptor, kind::f16: D fp32 (bit 4), A bf16 (bits 7-9),
// B bf16 (bits 10-12), A K-major (bit 15 = 0), B MN-major (bit 16 = 1),
// N >> 3 in bits 17-22, M >> 4 in bits 24-28.
__host__ __device__ constexpr uint32_t make_idesc(int M, int N,
                                                  bool b_mn_major = true,
                                                  bool a_mn_major = false) {
  return (1u << 4) | (1u << 7) | (1u << 10) |
         (a_mn_major ? (1u << 15) : 0u) | (b_mn_major ? (1u << 16) : 0u) |
         (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&p);
}

// ------------------------------------------------------------ tiles ------
// A tile is (group g, n-tile, m-tile of 128 rows).  Groups with at least two
// m-tiles ("heavy": their weight tile feeds several m-tiles, so they lean on
// the tensor cores) and groups with one ("light": pure weight streaming)
// form two streams, each in (group, n-tile, m-tile) order with m fastest so
// the m-tiles of a weight tile run together and share it through L2.  The
// two streams are interleaved evenly (position i of the launch is heavy iff
// floor((i+1)*Nh/N) > floor(i*Nh/N)), so every wave of CTAs mixes
// compute-bound and HBM-bound tiles instead of running the hot experts
// first and the cold ones last.
struct TileTable {
  const int* goff;   // [G+1] row offsets of the groups
  const int* hpre;   // [G+1] m-tiles of heavy groups before g
  const int* lpre;   // [G+1] m-tiles of light groups before g
  int G, n_tiles;
  long long heavy, total;  // tiles
};

// Largest g with pre[g] <= q (the group holding stream m-tile q).
__device__ __forceinline__ int group_of(const int* pre, int G, int q) {
  int lo = 0, hi = G - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (pre[mid] <= q)
      lo = mid;
    else
      hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ void decode_tile(const TileTable& tt, int tile,
                                            int& e, int& m, int& n) {
  const long long i = tile;
  const long long hb = i * tt.heavy / tt.total;           // heavy before i
  const bool heavy = (i + 1) * tt.heavy / tt.total > hb;
  const int* pre = heavy ? tt.hpre : tt.lpre;
  const int q = static_cast<int>(heavy ? hb : i - hb);     // rank in stream
  e = group_of(pre, tt.G, q / tt.n_tiles);
  const int mt = pre[e + 1] - pre[e];
  const int local = q - pre[e] * tt.n_tiles;
  n = local / mt;
  m = local - n * mt;
}

// All threads: goff[0..G], hpre[0..G], lpre[0..G] for tiles of
// rows_per_tile rows.
__device__ void build_tile_table(const int32_t* __restrict__ off, int G,
                                 int* goff, int* hpre, int* lpre, int* wsum,
                                 int rows_per_tile) {
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int per = (G + kThreads - 1) / kThreads;
  const int g0 = min(G, tid * per), g1 = min(G, g0 + per);
  int lh = 0, ll = 0;
  for (int g = g0; g < g1; ++g) {
    const int a = __ldg(off + g), b = __ldg(off + g + 1);
    const int mt = b > a ? (b - a + rows_per_tile - 1) / rows_per_tile : 0;
    goff[g] = a;
    hpre[g] = mt >= 2 ? mt : 0;
    lpre[g] = mt == 1 ? 1 : 0;
    lh += hpre[g];
    ll += lpre[g];
  }
  if (tid == 0) goff[G] = __ldg(off + G);
  int ih = lh, il = ll;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int nh = __shfl_up_sync(0xffffffffu, ih, o);
    const int nl = __shfl_up_sync(0xffffffffu, il, o);
    if (lane >= o) {
      ih += nh;
      il += nl;
    }
  }
  if (lane == 31) {
    wsum[w] = ih;
    wsum[8 + w] = il;
  }
  __syncthreads();
  if (tid == 0) {
    int rh = 0, rl = 0;
    for (int i = 0; i < kThreads / 32; ++i) {
      const int vh = wsum[i], vl = wsum[8 + i];
      wsum[i] = rh;
      wsum[8 + i] = rl;
      rh += vh;
      rl += vl;
    }
    wsum[kThreads / 32] = rh;
    wsum[8 + kThreads / 32] = rl;
  }
  __syncthreads();
  int rh = wsum[w] + ih - lh, rl = wsum[8 + w] + il - ll;
  for (int g = g0; g < g1; ++g) {
    const int vh = hpre[g], vl = lpre[g];
    hpre[g] = rh;
    lpre[g] = rl;
    rh += vh;
    rl += vl;
  }
  if (tid == 0) {
    hpre[G] = wsum[kThreads / 32];
    lpre[G] = wsum[8 + kThreads / 32];
  }
  __syncthreads();
}

// ----------------------------------------------------------- kernel ------
// MODE 0: out = h = silu(A Wg) * (A Wu), BN = 256 (128 gate + 128 up cols)
// MODE 1: out = y_sorted = A Wd, BN = 256 or 128
// MODE 4: MODE 0 that also stores g (out3) and u (out2) for the backward
// MODE 2: dh = dy_sorted Wd^T with Wd read K-major (one 64 x 256 box); the
//         epilogue turns dh into dg (out) and du (out2) with g, u (aux_*)
// MODE 3: dx_sorted = [dg | du] [Wg^T ; Wu^T]: K = 2F, the first k_split
//         k-blocks from (tmA, tmB0), the rest from (tmA1, tmB1), K-major B
template <int MODE, int BN>
__global__ void __launch_bounds__(kThreads, 1)
    gmm_tc_kernel(const __grid_constant__ CUtensorMap tmA,
                  const __grid_constant__ CUtensorMap tmB0,
                  const __grid_constant__ CUtensorMap tmB1,
                  const __grid_constant__ CUtensorMap tmA1, Params p) {
  using L = Tile<BN>;
  static_assert(MODE == 1 || MODE == 2 || MODE == 3 || BN == 256,
                "gate + up tiles are 128 + 128 columns");
  constexpr bool kGateUp = MODE == 0 || MODE == 4;   // MN-major gate/up B
  constexpr bool kBKMajor = MODE == 2 || MODE == 3;  // K-major B
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * L::kStage);
  uint64_t* full = bars;
  uint64_t* empty = bars + STAGES;
  uint64_t* tfull = bars + 2 * STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* done = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* wsum = reinterpret_cast<int*>(tmem_slot + 4);  // [16]
  int* goff = wsum + 16;                               // [E+1]
  int* hpre = goff + (p.E + 1);                        // [E+1]
  int* lpre = hpre + (p.E + 1);                        // [E+1]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t smem_base = smem_u32(smem);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
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
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB0);
    if (kGateUp || MODE == 3) prefetch_tmap(&tmB1);
    if (MODE == 3) prefetch_tmap(&tmA1);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  build_tile_table(p.group_offsets, p.E, goff, hpre, lpre, wsum, BM);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  TileTable tt;
  tt.goff = goff;
  tt.hpre = hpre;
  tt.lpre = lpre;
  tt.G = p.E;
  tt.n_tiles = p.n_tiles;
  tt.heavy = static_cast<long long>(hpre[p.E]) * p.n_tiles;
  tt.total = tt.heavy + static_cast<long long>(lpre[p.E]) * p.n_tiles;
  const int total_tiles = static_cast<int>(tt.total);
  const int kblocks = p.K / BK;

  if (warp == 0) {
    // ------------------------------------------------ TMA producer -----
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      long long fills = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total_tiles;
           tile += gridDim.x) {
        int e, m, n;
        decode_tile(tt, tile, e, m, n);
        const int a_row = goff[e] + m * BM;
        const int we = p.group_expert ? __ldg(p.group_expert + e) : e;
        const int b_row = we * p.K;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (p.stall_after_fills >= 0 && fills >= p.stall_after_fills) {
            ok = false;  // test hook: leave the MMA warp waiting
            break;
          }
          if (!mbar_wait(smem_u32(empty + stage), phase ^ 1u, abort_flag,
                         p.status)) {
            ok = false;
            break;
          }
          const uint32_t fb = smem_u32(full + stage);
          mbar_expect_tx(fb, L::kStage);
          const uint32_t sa = smem_base + stage * L::kStage;
          const uint32_t sb = sa + L::kABytes;
          if (kGateUp) {
            tma_load_2d(sa, &tmA, fb, kb * BK, a_row);
            tma_load_2d(sb, &tmB0, fb, n * 128, b_row + kb * BK);
            tma_load_2d(sb + 8192, &tmB0, fb, n * 128 + 64, b_row + kb * BK);
            tma_load_2d(sb + 16384, &tmB1, fb, n * 128, b_row + kb * BK);
            tma_load_2d(sb + 24576, &tmB1, fb, n * 128 + 64, b_row + kb * BK);
          } else if (MODE == 1) {
            tma_load_2d(sa, &tmA, fb, kb * BK, a_row);
#pragma unroll
            for (int c = 0; c < L::kChunks; ++c)
              tma_load_2d(sb + c * 8192, &tmB0, fb, n * BN + c * 64,
                          b_row + kb * BK);
          } else if (MODE == 2) {
            // B rows = the BN output columns (f) of expert we, K-major:
            // Wd[we] is [F, H] with H (the reduction) contiguous
            tma_load_2d(sa, &tmA, fb, kb * BK, a_row);
            tma_load_2d(sb, &tmB0, fb, kb * BK, we * p.out_ld + n * BN);
          } else {  // MODE 3: Wg[we], Wu[we] are [H, F], F contiguous
            const bool second = kb >= p.k_split;
            const int kk = (second ? kb - p.k_split : kb) * BK;
            tma_load_2d(sa, second ? &tmA1 : &tmA, fb, kk, a_row);
            tma_load_2d(sb, second ? &tmB1 : &tmB0, fb, kk,
                        we * p.out_ld + n * BN);
          }
          ++fills;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Drain: every load this thread issued has landed before exit.
      const long long first = fills > STAGES ? fills - STAGES : 0;
      for (long long f = first; f < fills; ++f)
        mbar_wait(smem_u32(full + (f % STAGES)),
                  static_cast<uint32_t>((f / STAGES) & 1), nullptr,
                  p.status);
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer -------
    if (lane == 0) {
      constexpr uint32_t idesc = make_idesc(BM, BN, !kBKMajor);
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total_tiles;
           tile += gridDim.x) {
        if (!mbar_wait(smem_u32(tempty + acc), acc_phase ^ 1u, abort_flag,
                       p.status))
          break;
        tc_fence_after();
        const uint32_t d = tmem_base + acc * kAccCols;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait(smem_u32(full + stage), phase, abort_flag,
                         p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_base + stage * L::kStage;
          const uint32_t sb = sa + L::kABytes;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint64_t ad = smem_desc(sa + kk * 32, 16, 1024);
            // K-major B: 256 rows of 128 B, advanced 32 B per K=16 step;
            // N-major B: 64-column chunks 8 KB apart, 16 k-rows per step
            const uint64_t bd = kBKMajor
                                    ? smem_desc(sb + kk * 32, 16, 1024)
                                    : smem_desc(sb + kk * 2048, 8192, 1024);
            umma_bf16(d, ad, bd, idesc, (kb | kk) != 0 ? 1u : 0u);
          }
          umma_commit(smem_u32(empty + stage));
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(smem_u32(tfull + acc));
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      // Drain: all MMAs issued by this thread are complete.
      umma_commit(smem_u32(done));
      mbar_wait(smem_u32(done), 0, nullptr, p.status);
    }
  } else {
    // ------------------------------------------------ epilogue ---------
    const int q = warp & 3;  // TMEM lane quadrant this warp may access
    const int row = q * 32 + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tile = blockIdx.x; tile < total_tiles; tile += gridDim.x) {
      int e, m, n;
      decode_tile(tt, tile, e, m, n);
      bool ok = mbar_wait(smem_u32(tfull + acc), acc_phase, abort_flag,
                          p.status);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      const int grow = goff[e] + m * BM + row;
      const bool valid = grow < goff[e + 1];
      const uint32_t taddr =
          tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * kAccCols;
      if (kGateUp) {
        const long long base = static_cast<long long>(grow) * p.out_ld + n * 128;
        uint4* dst = reinterpret_cast<uint4*>(p.out + base);
#pragma unroll 1
        for (int c = 0; c < 128; c += 32) {
          uint32_t g[32], u[32];
          tmem_ld32x2(taddr + c, taddr + 128 + c, g, u);
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float g0 = __uint_as_float(g[2 * i]);
            const float g1 = __uint_as_float(g[2 * i + 1]);
            const float h0 = g0 / (1.0f + __expf(-g0)) *
                             __uint_as_float(u[2 * i]);
            const float h1 = g1 / (1.0f + __expf(-g1)) *
                             __uint_as_float(u[2 * i + 1]);
            pk[i] = pack_bf16x2(h0, h1);
          }
          if (valid) {
#pragma unroll
            for (int v = 0; v < 4; ++v)
              dst[c / 8 + v] = make_uint4(pk[4 * v], pk[4 * v + 1],
                                          pk[4 * v + 2], pk[4 * v + 3]);
          }
          if (MODE == 4 && valid) {  // keep g and u for the backward
            uint4* dg_ = reinterpret_cast<uint4*>(p.out3 + base);
            uint4* du_ = reinterpret_cast<uint4*>(p.out2 + base);
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              uint32_t a[4], b[4];
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                const int i = 4 * v + q;
                a[q] = pack_bf16x2(__uint_as_float(g[2 * i]),
                                   __uint_as_float(g[2 * i + 1]));
                b[q] = pack_bf16x2(__uint_as_float(u[2 * i]),
                                   __uint_as_float(u[2 * i + 1]));
              }
              dg_[c / 8 + v] = make_uint4(a[0], a[1], a[2], a[3]);
              du_[c / 8 + v] = make_uint4(b[0], b[1], b[2], b[3]);
            }
          }
        }
      } else if (MODE == 2) {
        // dh (TMEM) -> dg = dh * u * silu'(g), du = dh * silu(g)
        const long long base = static_cast<long long>(grow) * p.out_ld + n * BN;
#pragma unroll 1
        for (int c = 0; c < BN; c += 32) {
          uint32_t r[32];
          tmem_ld32(taddr + c, r);
          if (!valid) continue;
          uint32_t gk[16], uk[16];
          const uint4* gs = reinterpret_cast<const uint4*>(p.aux_g + base + c);
          const uint4* us = reinterpret_cast<const uint4*>(p.aux_u + base + c);
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            const uint4 a = gs[v], b = us[v];
            gk[4 * v] = a.x; gk[4 * v + 1] = a.y;
            gk[4 * v + 2] = a.z; gk[4 * v + 3] = a.w;
            uk[4 * v] = b.x; uk[4 * v + 1] = b.y;
            uk[4 * v + 2] = b.z; uk[4 * v + 3] = b.w;
          }
          uint32_t pg[16], pu[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            float dgv[2], duv[2];
#pragma unroll
            for (int hlf = 0; hlf < 2; ++hlf) {
              const float gv = __uint_as_float(
                  hlf ? (gk[i] & 0xffff0000u) : (gk[i] << 16));
              const float uv = __uint_as_float(
                  hlf ? (uk[i] & 0xffff0000u) : (uk[i] << 16));
              const float dh = __uint_as_float(r[2 * i + hlf]);
              const float sg = 1.0f / (1.0f + __expf(-gv));
              dgv[hlf] = dh * uv * sg * (1.0f + gv * (1.0f - sg));
              duv[hlf] = dh * gv * sg;
            }
            pg[i] = pack_bf16x2(dgv[0], dgv[1]);
            pu[i] = pack_bf16x2(duv[0], duv[1]);
          }
          uint4* dgo = reinterpret_cast<uint4*>(p.out + base + c);
          uint4* duo = reinterpret_cast<uint4*>(p.out2 + base + c);
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            dgo[v] = make_uint4(pg[4 * v], pg[4 * v + 1], pg[4 * v + 2],
                                pg[4 * v + 3]);
            duo[v] = make_uint4(pu[4 * v], pu[4 * v + 1], pu[4 * v + 2],
                                pu[4 * v + 3]);
          }
        }
      } else {
        uint4* dst = reinterpret_cast<uint4*>(
            p.out + static_cast<long long>(grow) * p.out_ld + n * BN);
#pragma unroll 1
        for (int c = 0; c < BN; c += 32) {
          uint32_t r[32];
          tmem_ld32(taddr + c, r);
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            pk[i] = pack_bf16x2(__uint_as_float(r[2 * i]),
                                __uint_as_float(r[2 * i + 1]));
          if (valid) {
#pragma unroll
            for (int v = 0; v < 4; ++v)
              dst[c / 8 + v] = make_uint4(pk[4 * v], pk[4 * v + 1],
                                          pk[4 * v + 2], pk[4 * v + 3]);
          }
        }
      }
      tc_fence_before();
      mbar_arrive(smem_u32(tempty + acc));
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

// ------------------------------------------------------ pair kernel ------
constexpr int STAGES2 = 6;
constexpr int BMP = 2 * BM;                     // rows of a pair tile
constexpr int kA2Bytes = BM * BK * 2;           // this CTA's 128 rows
constexpr int kB2Bytes = BK * 128 * 2;          // this CTA's half of N=256
constexpr int kStage2 = kA2Bytes + kB2Bytes;    // 32 KB
constexpr uint32_t kTxPair = 2 * kStage2;       // bytes per stage, both CTAs
constexpr int kPairArrivals = 2 * kEpilogueThreads;

// MODE 0: h = silu(A Wg) * (A Wu): the leader stages the gate columns, the
// peer the up columns of the same 128 outputs; TMEM columns 0-127 of either
// CTA hold gate, 128-255 up, for its own 128 rows.
// MODE 1: y_sorted = A Wd, 256 output columns: the leader stages the first
// 128, the peer the last 128.
template <int MODE>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    gmm_tc2_kernel(const __grid_constant__ CUtensorMap tmA,
                   const __grid_constant__ CUtensorMap tmB0,
                   const __grid_constant__ CUtensorMap tmB1, Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES2 * kStage2);
  uint64_t* full = bars;
  uint64_t* empty = bars + STAGES2;
  uint64_t* tfull = bars + 2 * STAGES2;
  uint64_t* tempty = tfull + 2;
  uint64_t* done = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* wsum = reinterpret_cast<int*>(tmem_slot + 4);  // [16]
  int* goff = wsum + 16;                               // [E+1]
  int* hpre = goff + (p.E + 1);                        // [E+1]
  int* lpre = hpre + (p.E + 1);                        // [E+1]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();  // 0: leader, 1: peer
  const uint32_t smem_base = smem_u32(smem);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES2; ++s) {
      mbar_init(smem_u32(full + s), 1);
      mbar_init(smem_u32(empty + s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(smem_u32(tfull + a), 1);
      mbar_init(smem_u32(tempty + a), kPairArrivals);
    }
    mbar_init(smem_u32(done), 1);
    *abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB0);
    if (MODE == 0) prefetch_tmap(&tmB1);
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish_pair();
  }
  build_tile_table(p.group_offsets, p.E, goff, hpre, lpre, wsum, BMP);
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers exist before either signals them
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  TileTable tt;
  tt.goff = goff;
  tt.hpre = hpre;
  tt.lpre = lpre;
  tt.G = p.E;
  tt.n_tiles = p.n_tiles;
  tt.heavy = static_cast<long long>(hpre[p.E]) * p.n_tiles;
  tt.total = tt.heavy + static_cast<long long>(lpre[p.E]) * p.n_tiles;
  const int total_tiles = static_cast<int>(tt.total);
  const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
  const int kblocks = p.K / BK;

  if (warp == 0) {
    // ---------------------------------------- TMA producer (both CTAs) ---
    if (lane == 0) {
      const CUtensorMap* mb = (MODE == 0 && rank == 1) ? &tmB1 : &tmB0;
      int stage = 0;
      uint32_t phase = 0;
      long long fills = 0;
      bool ok = true;
      for (int tile = pair; ok && tile < total_tiles; tile += npairs) {
        int e, m, n;
        decode_tile(tt, tile, e, m, n);
        const int a_row = goff[e] + m * BMP + static_cast<int>(rank) * BM;
        const int we = p.group_expert ? __ldg(p.group_expert + e) : e;
        const int b_row = we * p.K;
        const int b_col = MODE == 0 ? n * 128 : n * 256 + rank * 128;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait(smem_u32(empty + stage), phase ^ 1u, abort_flag,
                         p.status)) {
            ok = false;
            break;
          }
          const uint32_t fb = map_to_rank(smem_u32(full + stage), 0);
          if (rank == 0) mbar_expect_tx(smem_u32(full + stage), kTxPair);
          const uint32_t sa = smem_base + stage * kStage2;
          const uint32_t sb = sa + kA2Bytes;
          tma_load_2d_pair(sa, &tmA, fb, kb * BK, a_row);
          tma_load_2d_pair(sb, mb, fb, b_col, b_row + kb * BK);
          tma_load_2d_pair(sb + 8192, mb, fb, b_col + 64, b_row + kb * BK);
          ++fills;
          if (++stage == STAGES2) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Drain: the leader's full barriers count both CTAs' bytes.
      if (rank == 0) {
        const long long first = fills > STAGES2 ? fills - STAGES2 : 0;
        for (long long f = first; f < fills; ++f)
          mbar_wait(smem_u32(full + (f % STAGES2)),
                    static_cast<uint32_t>((f / STAGES2) & 1), nullptr,
                    p.status);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------- MMA issuer (leader) ------
    if (lane == 0 && rank == 0) {
      constexpr uint32_t idesc = make_idesc(BMP, 256);
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      for (int tile = pair; ok && tile < total_tiles; tile += npairs) {
        if (!mbar_wait(smem_u32(tempty + acc), acc_phase ^ 1u, abort_flag,
                       p.status))
          break;
        tc_fence_after();
        const uint32_t d = tmem_base + acc * kAccCols;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait(smem_u32(full + stage), phase, abort_flag,
                         p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_base + stage * kStage2;
          const uint32_t sb = sa + kA2Bytes;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint64_t ad = smem_desc(sa + kk * 32, 16, 1024);
            const uint64_t bd = smem_desc(sb + kk * 2048, 8192, 1024);
            umma_bf16_pair(d, ad, bd, idesc, (kb | kk) != 0 ? 1u : 0u);
          }
          umma_commit_pair_mc(smem_u32(empty + stage));
          if (++stage == STAGES2) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit_pair_mc(smem_u32(tfull + acc));
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      umma_commit_pair(smem_u32(done));
      mbar_wait(smem_u32(done), 0, nullptr, p.status);
    }
  } else {
    // ---------------------------------------- epilogue (both CTAs) -----
    const int q = warp & 3;
    const int row = static_cast<int>(rank) * BM + q * 32 + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tile = pair; tile < total_tiles; tile += npairs) {
      int e, m, n;
      decode_tile(tt, tile, e, m, n);
      bool ok = mbar_wait(smem_u32(tfull + acc), acc_phase, abort_flag,
                          p.status);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      const int grow = goff[e] + m * BMP + row;
      const bool valid = grow < goff[e + 1];
      const uint32_t taddr =
          tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * kAccCols;
      if (MODE == 0) {
        uint4* dst = reinterpret_cast<uint4*>(
            p.out + static_cast<long long>(grow) * p.out_ld + n * 128);
#pragma unroll 1
        for (int c = 0; c < 128; c += 32) {
          uint32_t g[32], u[32];
          tmem_ld32x2(taddr + c, taddr + 128 + c, g, u);
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float g0 = __uint_as_float(g[2 * i]);
            const float g1 = __uint_as_float(g[2 * i + 1]);
            const float h0 = g0 / (1.0f + __expf(-g0)) *
                             __uint_as_float(u[2 * i]);
            const float h1 = g1 / (1.0f + __expf(-g1)) *
                             __uint_as_float(u[2 * i + 1]);
            pk[i] = pack_bf16x2(h0, h1);
          }
          if (valid) {
#pragma unroll
            for (int v = 0; v < 4; ++v)
              dst[c / 8 + v] = make_uint4(pk[4 * v], pk[4 * v + 1],
                                          pk[4 * v + 2], pk[4 * v + 3]);
          }
        }
      } else {
        uint4* dst = reinterpret_cast<uint4*>(
            p.out + static_cast<long long>(grow) * p.out_ld + n * 256);
#pragma unroll 1
        for (int c = 0; c < 256; c += 32) {
          uint32_t r[32];
          tmem_ld32(taddr + c, r);
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            pk[i] = pack_bf16x2(__uint_as_float(r[2 * i]),
                                __uint_as_float(r[2 * i + 1]));
          if (valid) {
#pragma unroll
            for (int v = 0; v < 4; ++v)
              dst[c / 8 + v] = make_uint4(pk[4 * v], pk[4 * v + 1],
                                          pk[4 * v + 2], pk[4 * v + 3]);
          }
        }
      }
      tc_fence_before();
      mbar_arrive_cluster(map_to_rank(smem_u32(tempty + acc), 0));
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // neither CTA leaves while its peer may still use it
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

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
constexpr int WSTAGES = 3;
constexpr int kWStage = BM * BK * 2 + BK * 256 * 2;  // 48 KB
constexpr int kStageBuf = 32 * 32 * 4;               // 4 KB
constexpr int kMaxSeg = 16;

struct WParams {
  const int32_t* seg_off[kMaxSeg];  // [G+1] group row offsets per segment
  int seg_base[kMaxSeg];            // row of the segment's first row
  int n_seg;
  const int32_t* group_expert;      // [G] or null (identity)
  int G;
  int m_tiles;   // 128-row tiles of one expert's dW
  int n_tiles;   // column tiles
  int reduce;    // 1: TMA reduce-add, 0: TMA store
  int32_t* status;
};

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

// At most one bulk group of this thread still reading shared memory.
__device__ __forceinline__ void bulk_wait_read_1() {
  asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
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
  uint8_t* stagebuf = smem + WSTAGES * kWStage;  // [4 warps][2][4 KB]
  uint64_t* bars = reinterpret_cast<uint64_t*>(stagebuf + 8 * kStageBuf);
  uint64_t* full = bars;
  uint64_t* empty = bars + WSTAGES;
  uint64_t* tfull = bars + 2 * WSTAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* done = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* wsum = reinterpret_cast<int*>(tmem_slot + 4);  // [16]
  int* tpre = wsum + 16;                               // [G+1]

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
    uint8_t* mybuf = stagebuf + q * 2 * kStageBuf;
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
#pragma unroll 1
      for (int sub = 0; sub < BN / 32; ++sub, ++nsub) {
        uint32_t r[32];
        tmem_ld32(taddr + sub * 32, r);
        uint8_t* buf = mybuf + (nsub & 1) * kStageBuf;
        if (lane == 0) bulk_wait_read_1();
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
          if (p.reduce)
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

// Zeroes dW[e] of every expert without rows in any segment (store mode:
// no tile writes it).  Grid (G, blocks), 16-byte stores.
__global__ void zero_empty_kernel(WParams p, float* a, float* b,
                                  long long per_expert) {
  const int g = blockIdx.x;
  if (wgrad_rows(p, g) > 0) return;
  const long long n4 = per_expert / 4;
  float4* pa = reinterpret_cast<float4*>(a + g * per_expert);
  float4* pb = b ? reinterpret_cast<float4*>(b + g * per_expert) : nullptr;
  const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
  for (long long i = blockIdx.y * blockDim.x + threadIdx.x; i < n4;
       i += static_cast<long long>(gridDim.y) * blockDim.x) {
    pa[i] = z;
    if (pb) pb[i] = z;
  }
}

// ------------------------------------------------------------- host ------
using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t,
                                 void*, const cuuint64_t*, const cuuint64_t*,
                                 const cuuint32_t*, const cuuint32_t*,
                                 CUtensorMapInterleave, CUtensorMapSwizzle,
                                 CUtensorMapL2promotion,
                                 CUtensorMapFloatOOBfill);

EncodeTiled encode_fn() {
  static EncodeTiled fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiled>(ptr);
  });
  return fn;
}

// 2-D map over a row-major [outer, inner] matrix, 128-byte swizzle (bf16
// operands, or fp32 for the weight-gradient output).
bool make_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer,
              uint32_t box_inner, uint32_t box_outer, bool f32 = false) {
  EncodeTiled fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {inner * (f32 ? 4 : 2)};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m,
            f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
            2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int BN>
size_t smem_bytes(int E) {
  return 1024 + STAGES * Tile<BN>::kStage + 8 * (2 * STAGES + 5) + 16 +
         4 * (16 + 3 * (E + 1)) + 64;
}

// The pair form pays off only when groups are large: a pair tile covers 256
// rows, and for smaller groups the peer SM stages rows it then masks (more
// L2 traffic and tensor work per weight tile, measured 15-25% slower on
// weight-streaming layers).  With >= 1024 routed rows per group on average
// it was measured 2% (GEMM1) and 9% (GEMM2) faster.
constexpr long long kPairMinRowsPerGroup = 1024;

bool use_pair(const moe_config_t& c, const Groups& g) {
  return g_stall_after_fills.load() < 0 &&
         static_cast<long long>(c.T) * c.k >= kPairMinRowsPerGroup * g.n;
}

size_t smem_bytes_pair(int E) {
  return 1024 + STAGES2 * kStage2 + 8 * (2 * STAGES2 + 5) + 16 +
         4 * (16 + 3 * (E + 1)) + 64;
}

template <int MODE>
cudaError_t launch_pair(const CUtensorMap& a, const CUtensorMap& b0,
                        const CUtensorMap& b1, const Params& p,
                        cudaStream_t s) {
  const size_t smem = smem_bytes_pair(p.E);
  int dev = 0, sms = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (err != cudaSuccess) return err;
  err = cudaFuncSetAttribute(gmm_tc2_kernel<MODE>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  const int grid = sms & ~1;  // whole CTA pairs
  gmm_tc2_kernel<MODE><<<grid, kThreads, smem, s>>>(a, b0, b1, p);
  return cudaGetLastError();
}

template <int MODE, int BN>
cudaError_t launch_one(const CUtensorMap& a, const CUtensorMap& b0,
                       const CUtensorMap& b1, const CUtensorMap& a1, Params p,
                       cudaStream_t s) {
  p.stall_after_fills = g_stall_after_fills.load();
  const size_t smem = smem_bytes<BN>(p.E);
  int dev = 0, sms = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (err != cudaSuccess) return err;
  err = cudaFuncSetAttribute(gmm_tc_kernel<MODE, BN>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  gmm_tc_kernel<MODE, BN><<<sms, kThreads, smem, s>>>(a, b0, b1, a1, p);
  return cudaGetLastError();
}

size_t smem_bytes_wgrad(int G) {
  return 1024 + WSTAGES * kWStage + 8 * kStageBuf + 8 * (2 * WSTAGES + 5) +
         16 + 4 * (16 + G + 1) + 64;
}

template <int WMODE, int BN>
cudaError_t launch_wgrad(const CUtensorMap& pm, const CUtensorMap& q0,
                         const CUtensorMap& q1, const CUtensorMap& o0,
                         const CUtensorMap& o1, const WParams& p,
                         cudaStream_t s) {
  const size_t smem = smem_bytes_wgrad(p.G);
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

void set_gemm_stall_for_tests(long long fills) {
  tc::g_stall_after_fills.store(fills);
}

bool gmm_tc_supported(const moe_config_t& c) {
  return c.dtype == MOE_BF16 && c.H % 128 == 0 && c.F % 128 == 0 &&
         c.H >= 128 && c.F >= 128;
}

cudaError_t launch_gmm1_bf16(const moe_config_t& c, const Groups& g,
                             const void* x_sorted,
                             const int32_t* group_offsets, const void* w_gate,
                             const void* w_up, void* h, int32_t* status,
                             cudaStream_t s) {
  const uint64_t rows = static_cast<uint64_t>(c.T) * c.k;
  if (rows == 0) return cudaSuccess;
  CUtensorMap a1, bg, bu;
  const uint64_t E = static_cast<uint64_t>(c.E);
  if (!tc::make_map(&a1, x_sorted, c.H, rows, 64, tc::BM) ||
      !tc::make_map(&bg, w_gate, c.F, E * c.H, 64, 64) ||
      !tc::make_map(&bu, w_up, c.F, E * c.H, 64, 64))
    return cudaErrorInvalidValue;
  tc::Params p1{group_offsets, g.map, g.n, c.H, c.F / 128,
                static_cast<__nv_bfloat16*>(h), c.F, status};
  if (tc::use_pair(c, g)) return tc::launch_pair<0>(a1, bg, bu, p1, s);
  return tc::launch_one<0, 256>(a1, bg, bu, a1, p1, s);
}

cudaError_t launch_gmm2_bf16(const moe_config_t& c, const Groups& g,
                             const void* h, const int32_t* group_offsets,
                             const void* w_down, void* y_sorted,
                             int32_t* status, cudaStream_t s) {
  const uint64_t rows = static_cast<uint64_t>(c.T) * c.k;
  if (rows == 0) return cudaSuccess;
  CUtensorMap a2, bd;
  const uint64_t E = static_cast<uint64_t>(c.E);
  if (!tc::make_map(&a2, h, c.F, rows, 64, tc::BM) ||
      !tc::make_map(&bd, w_down, c.H, E * c.F, 64, 64))
    return cudaErrorInvalidValue;
  if (c.H % 256 == 0) {
    tc::Params p2{group_offsets, g.map, g.n, c.F, c.H / 256,
                  static_cast<__nv_bfloat16*>(y_sorted), c.H, status};
    if (tc::use_pair(c, g)) return tc::launch_pair<1>(a2, bd, bd, p2, s);
    return tc::launch_one<1, 256>(a2, bd, bd, a2, p2, s);
  }
  tc::Params p2{group_offsets, g.map, g.n, c.F, c.H / 128,
                static_cast<__nv_bfloat16*>(y_sorted), c.H, status};
  return tc::launch_one<1, 128>(a2, bd, bd, a2, p2, s);
}

// Forward GEMM1 + SwiGLU that also keeps g = x Wg and u = x Wu.
cudaError_t launch_gate_up_saved_bf16(const moe_config_t& c, const Groups& g,
                                      const void* x_sorted,
                                      const int32_t* group_offsets,
                                      const void* w_gate, const void* w_up,
                                      void* gbuf, void* ubuf, void* h,
                                      int32_t* status, cudaStream_t s) {
  const uint64_t rows = static_cast<uint64_t>(c.T) * c.k;
  if (rows == 0) return cudaSuccess;
  CUtensorMap a1, bg, bu;
  const uint64_t E = static_cast<uint64_t>(c.E);
  if (!tc::make_map(&a1, x_sorted, c.H, rows, 64, tc::BM) ||
      !tc::make_map(&bg, w_gate, c.F, E * c.H, 64, 64) ||
      !tc::make_map(&bu, w_up, c.F, E * c.H, 64, 64))
    return cudaErrorInvalidValue;
  tc::Params p1{group_offsets, g.map, g.n, c.H, c.F / 128,
                static_cast<__nv_bfloat16*>(h), c.F, status};
  p1.out2 = static_cast<__nv_bfloat16*>(ubuf);
  p1.out3 = static_cast<__nv_bfloat16*>(gbuf);
  return tc::launch_one<4, 256>(a1, bg, bu, a1, p1, s);
}

// dh = dy_sorted Wd^T with the SwiGLU backward in the epilogue: dg, du.
cudaError_t launch_down_dgrad_bf16(const moe_config_t& c, const Groups& g,
                                   const int32_t* group_offsets,
                                   const void* w_down, const void* gbuf,
                                   const void* ubuf, const void* dy_sorted,
                                   void* dg, void* du, int32_t* status,
                                   cudaStream_t s) {
  const uint64_t rows = static_cast<uint64_t>(c.T) * c.k;
  if (rows == 0) return cudaSuccess;
  const uint64_t E = static_cast<uint64_t>(c.E);
  const int bn = c.F % 256 == 0 ? 256 : 128;
  CUtensorMap ad, bd;
  if (!tc::make_map(&ad, dy_sorted, c.H, rows, 64, tc::BM) ||
      !tc::make_map(&bd, w_down, c.H, E * c.F, 64, bn))
    return cudaErrorInvalidValue;
  tc::Params p{group_offsets, g.map, g.n, c.H, c.F / bn,
               static_cast<__nv_bfloat16*>(dg), c.F, status};
  p.out2 = static_cast<__nv_bfloat16*>(du);
  p.aux_g = static_cast<const __nv_bfloat16*>(gbuf);
  p.aux_u = static_cast<const __nv_bfloat16*>(ubuf);
  return bn == 256 ? tc::launch_one<2, 256>(ad, bd, bd, ad, p, s)
                   : tc::launch_one<2, 128>(ad, bd, bd, ad, p, s);
}

// dx_sorted = dg Wg^T + du Wu^T as one GEMM with K = 2F.
cudaError_t launch_gate_up_dgrad_bf16(const moe_config_t& c, const Groups& g,
                                      const int32_t* group_offsets,
                                      const void* w_gate, const void* w_up,
                                      const void* dg, const void* du,
                                      void* dx_sorted, int32_t* status,
                                      cudaStream_t s) {
  const uint64_t rows = static_cast<uint64_t>(c.T) * c.k;
  if (rows == 0) return cudaSuccess;
  const uint64_t E = static_cast<uint64_t>(c.E);
  const int bn = c.H % 256 == 0 ? 256 : 128;
  CUtensorMap ag, au, bg, bu;
  if (!tc::make_map(&ag, dg, c.F, rows, 64, tc::BM) ||
      !tc::make_map(&au, du, c.F, rows, 64, tc::BM) ||
      !tc::make_map(&bg, w_gate, c.F, E * c.H, 64, bn) ||
      !tc::make_map(&bu, w_up, c.F, E * c.H, 64, bn))
    return cudaErrorInvalidValue;
  tc::Params p{group_offsets, g.map, g.n, 2 * c.F, c.H / bn,
               static_cast<__nv_bfloat16*>(dx_sorted), c.H, status};
  p.k_split = c.F / 64;
  return bn == 256 ? tc::launch_one<3, 256>(ag, bg, bu, au, p, s)
                   : tc::launch_one<3, 128>(ag, bg, bu, au, p, s);
}

// Weight gradients over row segments (each {group offsets, first row}),
// all inside buffers of `rows_total` rows.  accumulate = 0 overwrites every
// expert's dW (experts without rows get zeros); 1 adds into dW.
cudaError_t launch_wgrad_bf16(const moe_config_t& c, const Groups& g,
                              const WgradSegment* seg, int n_seg,
                              int64_t rows_total, const void* x_sorted,
                              const void* dg, const void* du, const void* h,
                              const void* dy_sorted, float* dw_gate,
                              float* dw_up, float* dw_down, int accumulate,
                              int parts, int32_t* status, cudaStream_t s) {
  const bool gu = (parts & kWgradGateUp) != 0;
  const bool dn = (parts & kWgradDown) != 0;
  const uint64_t E = static_cast<uint64_t>(c.E);
  const uint64_t rows = static_cast<uint64_t>(std::max<int64_t>(rows_total, 1));
  const long long per_expert = static_cast<long long>(c.H) * c.F;
  const bool mapped = g.map != nullptr;
  cudaError_t e = cudaSuccess;
  if (!accumulate && mapped) {  // duplicates reduce into one expert
    const size_t bytes = static_cast<size_t>(E) * per_expert * sizeof(float);
    if ((gu && (e = cudaMemsetAsync(dw_gate, 0, bytes, s)) != cudaSuccess) ||
        (gu && (e = cudaMemsetAsync(dw_up, 0, bytes, s)) != cudaSuccess) ||
        (dn && (e = cudaMemsetAsync(dw_down, 0, bytes, s)) != cudaSuccess))
      return e;
  }
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
    p.reduce = (accumulate || mapped || s0 > 0) ? 1 : 0;
    p.status = status;
    if (!p.reduce) {
      // experts without rows: no tile writes their dW
      const dim3 grid(static_cast<unsigned>(g.n), 16);
      if (gu)
        tc::zero_empty_kernel<<<grid, 256, 0, s>>>(p, dw_gate, dw_up,
                                                   per_expert);
      if (dn)
        tc::zero_empty_kernel<<<grid, 256, 0, s>>>(p, dw_down, nullptr,
                                                   per_expert);
      if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    if (p.n_seg == 0) break;
    if (gu) {
      p.m_tiles = c.H / tc::BM;
      p.n_tiles = c.F / 128;
      e = tc::launch_wgrad<0, 256>(px, qg, qu, og, ou, p, s);
      if (e != cudaSuccess) return e;
    }
    if (dn) {
      p.m_tiles = c.F / tc::BM;
      p.n_tiles = c.H / bnd;
      e = bnd == 256 ? tc::launch_wgrad<1, 256>(ph, qd, qd, od, od, p, s)
                     : tc::launch_wgrad<1, 128>(ph, qd, qd, od, od, p, s);
      if (e != cudaSuccess) return e;
    }
  }
  return cudaSuccess;
}

}  // namespace moe
