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
// Two-SM form of GEMM2 (gmm_tc2_kernel, used when its output tile is 256
// wide and groups are large): a cluster of two CTAs on one TPC shares each
// M=256 x N=256 tile through tcgen05.mma.cta_group::2.  Each CTA stages its
// own 128 rows of A and half of B in 6 stages of 32 KB, so a stage of
// compute needs a third less shared memory and more loads are in flight.
// The leader issues the MMAs and multicasts its commits to both CTAs; the
// peer's TMA loads complete on the leader's barrier; both CTAs run an
// epilogue on their own 128 rows of TMEM, and the peer's idle MMA lane
// relays its warps' release of the accumulator to the leader.
//
// Every wait is bounded (2 s of %globaltimer); on expiry the kernel raises
// MOE_DEV_TIMEOUT in the status word, tells the other roles to stop, drains
// its own TMA loads and MMAs, frees its tensor memory and returns.
#include <atomic>

#include "tc_common.cuh"

namespace moe {
namespace tc {

constexpr int STAGES = 4;

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
  // MODE 2 with unscaled dy rows: dh = row_w[r] * acc, and row_dot[r *
  // n_tiles + n] = acc . h over the tile's columns (h = aux_h)
  const float* row_w = nullptr;
  const __nv_bfloat16* aux_h = nullptr;
  float* row_dot = nullptr;
  int k_split = 0;                      // MODE 3: k-blocks from the 1st pair
  // MODE 5 (router logits): float32 output [rows, out_ld], an optional
  // float32 offset of the same shape added to it, and the row count of the
  // single group (group_offsets is then null).
  float* out_f32 = nullptr;
  const float* offset = nullptr;
  int rows1 = 0;
  // Tests of the timeout path only: the producer stops after this many
  // stage fills (-1: never), so the MMA warp's next wait runs out.
  long long stall_after_fills = -1;
};

std::atomic<long long> g_stall_after_fills{-1};

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
// rows_per_tile rows.  off == null: one group of rows1 rows (G = 1).
__device__ __forceinline__ int group_start(const int32_t* __restrict__ off,
                                           int g, int rows1) {
  return off ? __ldg(off + g) : (g == 0 ? 0 : rows1);
}

__device__ void build_tile_table(const int32_t* __restrict__ off, int G,
                                 int* goff, int* hpre, int* lpre, int* wsum,
                                 int rows_per_tile, int rows1 = 0) {
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int nthr = blockDim.x, nw = nthr >> 5;  // wsum: [2][32]
  const int per = (G + nthr - 1) / nthr;
  const int g0 = min(G, tid * per), g1 = min(G, g0 + per);
  int lh = 0, ll = 0;
  for (int g = g0; g < g1; ++g) {
    const int a = group_start(off, g, rows1);
    const int b = group_start(off, g + 1, rows1);
    const int mt = b > a ? (b - a + rows_per_tile - 1) / rows_per_tile : 0;
    goff[g] = a;
    hpre[g] = mt >= 2 ? mt : 0;
    lpre[g] = mt == 1 ? 1 : 0;
    lh += hpre[g];
    ll += lpre[g];
  }
  if (tid == 0) goff[G] = group_start(off, G, rows1);
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
    wsum[32 + w] = il;
  }
  __syncthreads();
  if (tid == 0) {
    int rh = 0, rl = 0;
    for (int i = 0; i < nw; ++i) {
      const int vh = wsum[i], vl = wsum[32 + i];
      wsum[i] = rh;
      wsum[32 + i] = rl;
      rh += vh;
      rl += vl;
    }
    wsum[nw] = rh;
    wsum[32 + nw] = rl;
  }
  __syncthreads();
  int rh = wsum[w] + ih - lh, rl = wsum[32 + w] + il - ll;
  for (int g = g0; g < g1; ++g) {
    const int vh = hpre[g], vl = lpre[g];
    hpre[g] = rh;
    lpre[g] = rl;
    rh += vh;
    rl += vl;
  }
  if (tid == 0) {
    hpre[G] = wsum[nw];
    lpre[G] = wsum[32 + nw];
  }
  __syncthreads();
}

// ----------------------------------------------------------- kernel ------
// MODE 0: out = h = silu(A Wg) * (A Wu), BN = 256 (128 gate + 128 up cols)
// MODE 1: out = y_sorted = A Wd, BN = 256 or 128
// MODE 4: MODE 0 that also stores g (out3) and u (out2) for the backward
// MODE 2: dh = dy_sorted Wd^T with Wd read K-major (one 64 x 256 box); the
//         epilogue turns dh into dg (out) and du (out2) with g, u (aux_*);
//         on unscaled dy rows (row_w set) dh = row_w[r] * acc and the row's
//         dot acc . h (aux_h) over the tile goes to row_dot
// MODE 3: dx_sorted = [dg | du] [Wg^T ; Wu^T]: K = 2F, the first k_split
//         k-blocks from (tmA, tmB0), the rest from (tmA1, tmB1), K-major B
// MODE 5: router logits = x Wr (+ offset) in float32: one group of rows1
//         token rows, Wr [H, E] read MN-major like Wd, BN = 128
template <int MODE, int BN>
__global__ void __launch_bounds__(kThreads, 1)
    gmm_tc_kernel(const __grid_constant__ CUtensorMap tmA,
                  const __grid_constant__ CUtensorMap tmB0,
                  const __grid_constant__ CUtensorMap tmB1,
                  const __grid_constant__ CUtensorMap tmA1, Params p) {
  using L = Tile<BN>;
  static_assert(MODE == 1 || MODE == 2 || MODE == 3 || MODE == 5 ||
                    BN == 256,
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
  int* wsum = reinterpret_cast<int*>(tmem_slot + 4);  // [64]
  int* goff = wsum + 64;                               // [E+1]
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
  build_tile_table(p.group_offsets, p.E, goff, hpre, lpre, wsum, BM, p.rows1);
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
          } else if (MODE == 1 || MODE == 5) {
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
        // dh (TMEM) -> dg = dh * u * silu'(g), du = dh * silu(g); with
        // unscaled dy rows dh = w_r * acc and the row's dot acc . h is kept
        const long long base = static_cast<long long>(grow) * p.out_ld + n * BN;
        const bool unscaled = p.row_w != nullptr;
        const float wr = unscaled && valid ? __ldg(p.row_w + grow) : 1.0f;
        float rdot = 0.0f;
#pragma unroll 1
        for (int c = 0; c < BN; c += 32) {
          uint32_t r[32];
          tmem_ld32(taddr + c, r);
          if (!valid) continue;
          if (unscaled) {
            const uint4* hs =
                reinterpret_cast<const uint4*>(p.aux_h + base + c);
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              const uint4 hq = hs[v];
              const uint32_t hw[4] = {hq.x, hq.y, hq.z, hq.w};
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const int e0 = 8 * v + 2 * i;
                const float a0 = __uint_as_float(r[e0]);
                const float a1 = __uint_as_float(r[e0 + 1]);
                rdot = fmaf(a0, __uint_as_float(hw[i] << 16), rdot);
                rdot = fmaf(a1, __uint_as_float(hw[i] & 0xffff0000u), rdot);
                r[e0] = __float_as_uint(wr * a0);
                r[e0 + 1] = __float_as_uint(wr * a1);
              }
            }
          }
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
        if (unscaled && valid)
          p.row_dot[static_cast<long long>(grow) * p.n_tiles + n] = rdot;
      } else if (MODE == 5) {
        // float32 logits (+ the offset), one row per thread
        const long long base =
            static_cast<long long>(grow) * p.out_ld + n * BN;
#pragma unroll 1
        for (int c = 0; c < BN; c += 32) {
          uint32_t r[32];
          tmem_ld32(taddr + c, r);
          if (!valid) continue;
          float4* dst = reinterpret_cast<float4*>(p.out_f32 + base + c);
          const float4* add =
              p.offset ? reinterpret_cast<const float4*>(p.offset + base + c)
                       : nullptr;
#pragma unroll
          for (int v = 0; v < 8; ++v) {
            float4 o = make_float4(__uint_as_float(r[4 * v]),
                                   __uint_as_float(r[4 * v + 1]),
                                   __uint_as_float(r[4 * v + 2]),
                                   __uint_as_float(r[4 * v + 3]));
            if (add) {
              const float4 b = __ldg(add + v);
              o.x += b.x;
              o.y += b.y;
              o.z += b.z;
              o.w += b.w;
            }
            dst[v] = o;
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

// y_sorted = A Wd, 256 output columns: the leader stages the first 128, the
// peer the last 128 of Wd's tile.  (GEMM1 + SwiGLU stays on the one-CTA
// kernel: at H = 7168, F = 2048 it measured 3-12 % faster than a pair form
// at 256 to 2048 rows per group.)
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    gmm_tc2_kernel(const __grid_constant__ CUtensorMap tmA,
                   const __grid_constant__ CUtensorMap tmB, Params p) {
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
  int* wsum = reinterpret_cast<int*>(tmem_slot + 4);  // [64]
  int* goff = wsum + 64;                               // [E+1]
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
      // one arrival per epilogue warp of this CTA; the leader's also
      // counts the peer's relay
      mbar_init(smem_u32(tempty + a), rank == 0 ? kEpilogueThreads / 32 + 1
                                                : kEpilogueThreads / 32);
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
        const int b_col = n * 256 + rank * 128;
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
          tma_load_2d_pair(sb, &tmB, fb, b_col, b_row + kb * BK);
          tma_load_2d_pair(sb + 8192, &tmB, fb, b_col + 64, b_row + kb * BK);
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
    } else if (lane == 0) {
      // ---------------------------------- TMEM-empty relay (peer) -------
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
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(tempty + acc));
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

// ------------------------------------------------------------- host ------
template <int BN>
size_t smem_bytes(int E) {
  return 1024 + STAGES * Tile<BN>::kStage + 8 * (2 * STAGES + 5) + 16 +
         4 * (64 + 3 * (E + 1)) + 64;
}

// The pair form of GEMM2 pays off only when groups are large: a pair tile
// covers 256 rows, and for smaller groups the peer SM stages rows it then
// masks.  At H = 7168, F = 2048, E = 256 it measured 1-11 % slower with 256
// routed rows per group and 7-10 % faster with 512 to 2048.  The row count
// is the host's bound on the rows the groups hold: T*k, or fewer when the
// caller knows them to be capped (a capped pass keeps at most S*C rows), so
// that a capped pass with many dropped rows does not take the pair kernel
// for groups that are small in fact.
#ifndef MOE_PAIR_MIN_ROWS
#define MOE_PAIR_MIN_ROWS 512
#endif
constexpr long long kPairMinRowsPerGroup = MOE_PAIR_MIN_ROWS;

long long group_rows_bound(const moe_config_t& c, const Groups& g) {
  const long long all = static_cast<long long>(c.T) * c.k;
  return g.max_rows >= 0 ? std::min<long long>(g.max_rows, all) : all;
}

bool use_pair(const moe_config_t& c, const Groups& g) {
  return g_stall_after_fills.load() < 0 &&
         group_rows_bound(c, g) >= kPairMinRowsPerGroup * g.n;
}

size_t smem_bytes_pair(int E) {
  return 1024 + STAGES2 * kStage2 + 8 * (2 * STAGES2 + 5) + 16 +
         4 * (64 + 3 * (E + 1)) + 64;
}

cudaError_t launch_pair(const CUtensorMap& a, const CUtensorMap& b,
                        const Params& p, cudaStream_t s) {
  const size_t smem = smem_bytes_pair(p.E);
  int dev = 0, sms = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (err != cudaSuccess) return err;
  err = cudaFuncSetAttribute(gmm_tc2_kernel,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  const int grid = sms & ~1;  // whole CTA pairs
  gmm_tc2_kernel<<<grid, kThreads, smem, s>>>(a, b, p);
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

}  // namespace tc

int gmm_pair_kinds(const moe_config_t& c, const Groups& g) {
  if (!gmm_tc_supported(c) || !tc::use_pair(c, g)) return 0;
  return c.H % 256 == 0 ? 2 : 0;   // GEMM2's 256-column tiles
}

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
    if (tc::use_pair(c, g)) return tc::launch_pair(a2, bd, p2, s);
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
                                   cudaStream_t s, const float* w_row,
                                   const void* h, float* row_dot) {
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
  if (w_row != nullptr) {
    if (h == nullptr || row_dot == nullptr) return cudaErrorInvalidValue;
    p.row_w = w_row;
    p.aux_h = static_cast<const __nv_bfloat16*>(h);
    p.row_dot = row_dot;
  }
  return bn == 256 ? tc::launch_one<2, 256>(ad, bd, bd, ad, p, s)
                   : tc::launch_one<2, 128>(ad, bd, bd, ad, p, s);
}

// Router logits [T, E] float32 = x [T, H] Wr [H, E] (+ offset [T, E]), on
// the tensor cores: needs bf16, H % 64 == 0 and E % 128 == 0
// (router_tc_supported).
bool router_tc_supported(const moe_config_t& c) {
  return c.dtype == MOE_BF16 && c.H % 64 == 0 && c.E % 128 == 0;
}

cudaError_t launch_router_bf16(const moe_config_t& c, const void* x,
                               const void* w_router, const float* offset,
                               float* logits, int32_t* status,
                               cudaStream_t s) {
  if (c.T == 0) return cudaSuccess;
  CUtensorMap a, b;
  if (!tc::make_map(&a, x, c.H, static_cast<uint64_t>(c.T), 64, tc::BM) ||
      !tc::make_map(&b, w_router, c.E, c.H, 64, 64))
    return cudaErrorInvalidValue;
  tc::Params p{nullptr, nullptr, 1, c.H, c.E / 128, nullptr, c.E, status};
  p.out_f32 = logits;
  p.offset = offset;
  p.rows1 = c.T;
  return tc::launch_one<5, 128>(a, b, b, a, p, s);
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

}  // namespace moe
