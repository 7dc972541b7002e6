// Expert parallelism across ranks: the rank-local kernels around the two
// exchanges (the transport itself is the caller's: NCCL all-to-all-v,
// torch.distributed, or copies between logical ranks on one GPU).
//
// "Support moe_dropless_fallback=layer on the ragged all-to-all MoE path"
// (MaxText pull request 5920), sections Why and How: each device sends its
// tokens' rows to the devices owning their experts; the overflow check is
// global (section Tests: every rank takes the same branch).  "Moe dynamic
// redundancy" (MaxText pull request 4760), review of ra2a_dedup_and_route:
// a token goes to a destination once and is expanded there to its expert
// rows.  "MoE ring-of-experts ..." (MaxText pull request 4969), section
// What: the ring variant all-gathers the tokens, every rank computes its
// local experts, and the combine is reduce-scattered.
//
// Ranks are the EP shards: rank d owns experts [d*E/S, (d+1)*E/S).  Per pass
// a source rank runs moe_permute_tables and moe_permute_scatter (index
// outputs only) with cfg.S = ranks, which give the dest-major dedup sets
// (uniq_offsets, uniq_tokens); then
//   ep_pack        one CTA per send row i: x_send[i] = x[uniq_tokens[i]]
//                  (16-byte copies) and the row's min(k, E/S) slots: the
//                  local expert and combine weight of each pick that its
//                  destination owns, in pick order, then -1 (weight 0);
//   ep_return_map  row_of_ret[t, d] = the send row of (t, d), else -1, so
//                  that the combine kernel with unit weights adds the rows
//                  the destinations return (moe_permute_backward);
//   ep_check       the global flag, required factor and capacity from the
//                  per-shard receive counts summed over the ranks;
//   ep_localize    (ring) the picks a rank owns, as local expert indices,
//                  in min(k, experts of the rank) slots;
//   ep_sum_parts   (ring) y[t] = sum over ranks of their partial outputs,
//                  accumulated in fp32 in rank order;
//   ep_delocalize  (ring backward) the transpose of ep_localize: a rank's
//                  per-slot values written back at the picks it owns.
// A receiving rank runs the ordinary permute / GEMMs / combine on the rows
// it received, with cfg.E = its local experts and cfg.k = min(k, E/S) slots
// per row in which -1 marks an empty slot.
#include <cuda_bf16.h>

#include "internal.h"

namespace moe {
namespace {

constexpr int kPackThreads = 128;

__global__ void __launch_bounds__(kPackThreads) ep_pack_kernel(
    const int4* __restrict__ x, int n16, const int32_t* __restrict__ topk_idx,
    const float* __restrict__ topk_w, int k, int kk, int S, int Ed,
    const int32_t* __restrict__ uniq_offsets,
    const int32_t* __restrict__ uniq_tokens, int4* __restrict__ x_send,
    int32_t* __restrict__ send_idx, float* __restrict__ send_w) {
  const int i = blockIdx.x, tid = threadIdx.x;
  if (i >= __ldg(uniq_offsets + S)) return;
  int d = 0;  // the destination: uniq_offsets[d] <= i < uniq_offsets[d+1]
  while (d + 1 < S && __ldg(uniq_offsets + d + 1) <= i) ++d;
  const int t = __ldg(uniq_tokens + i);
  const int4* src = x + static_cast<long long>(t) * n16;
  int4* dst = x_send + static_cast<long long>(i) * n16;
  for (int c = tid; c < n16; c += kPackThreads) dst[c] = __ldg(src + c);
  if (tid == 0) {  // the picks d owns, in pick order, then -1 padding
    const long long o = static_cast<long long>(t) * k;
    int32_t* si = send_idx + static_cast<long long>(i) * kk;
    float* sw = send_w + static_cast<long long>(i) * kk;
    int q = 0;
    for (int j = 0; j < k && q < kk; ++j) {
      const int e = __ldg(topk_idx + o + j);
      if (e >= 0 && e / Ed == d) {
        si[q] = e - d * Ed;
        sw[q] = __ldg(topk_w + o + j);
        ++q;
      }
    }
    for (; q < kk; ++q) {
      si[q] = -1;
      sw[q] = 0.0f;
    }
  }
}

__global__ void ep_return_map_kernel(int n_max, int S,
                                     const int32_t* __restrict__ uniq_offsets,
                                     const int32_t* __restrict__ uniq_tokens,
                                     int32_t* __restrict__ row_of_ret) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n_max || i >= __ldg(uniq_offsets + S)) return;
  int d = 0;
  while (d + 1 < S && __ldg(uniq_offsets + d + 1) <= i) ++d;
  const int t = __ldg(uniq_tokens + i);
  row_of_ret[static_cast<long long>(t) * S + d] = i;
}

__global__ void ep_check_kernel(const int32_t* __restrict__ shard, int S,
                                long long cap, double rows,
                                int32_t* __restrict__ flag,
                                float* __restrict__ req,
                                int32_t* __restrict__ cap_out) {
  if (threadIdx.x != 0) return;
  int f = 0, mx = 0;
  for (int s = 0; s < S; ++s) {
    const int r = shard[s];
    if (cap >= 0 && r > cap) f = 1;
    mx = max(mx, r);
  }
  *flag = f;
  *req = rows > 0.0 ? static_cast<float>(static_cast<double>(mx) *
                                         static_cast<double>(S) / rows)
                    : 0.0f;
  *cap_out = static_cast<int32_t>(cap);
}

// One thread per token: its picks in [e0, e0 + n_local) as local indices,
// in pick order, then -1 padding to kk slots.
__global__ void ep_localize_kernel(const int32_t* __restrict__ topk_idx,
                                   const float* __restrict__ topk_w, int T,
                                   int k, int kk, int e0, int n_local,
                                   int32_t* __restrict__ local_idx,
                                   float* __restrict__ local_w) {
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= T) return;
  const long long o = static_cast<long long>(t) * k;
  int32_t* li = local_idx + static_cast<long long>(t) * kk;
  float* lw = local_w + static_cast<long long>(t) * kk;
  int q = 0;
  for (int j = 0; j < k && q < kk; ++j) {
    const int e = __ldg(topk_idx + o + j);
    if (e >= e0 && e < e0 + n_local) {
      li[q] = e - e0;
      lw[q] = __ldg(topk_w + o + j);
      ++q;
    }
  }
  for (; q < kk; ++q) {
    li[q] = -1;
    lw[q] = 0.0f;
  }
}

// One thread per token: the q-th pick of t in [e0, e0 + n_local) (pick
// order) receives slot q of row r of local_v (r = row_of[t * row_stride],
// or t without a map; a negative r skips the token); the other picks are
// left as they are.
__global__ void ep_delocalize_kernel(const int32_t* __restrict__ topk_idx,
                                     const int32_t* __restrict__ row_of,
                                     int row_stride,
                                     const float* __restrict__ local_v, int T,
                                     int k, int kk, int e0, int n_local,
                                     float* __restrict__ v) {
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= T) return;
  const long long r =
      row_of ? __ldg(row_of + static_cast<long long>(t) * row_stride) : t;
  if (r < 0) return;
  const long long o = static_cast<long long>(t) * k;
  const float* lv = local_v + r * kk;
  int q = 0;
  for (int j = 0; j < k && q < kk; ++j) {
    const int e = __ldg(topk_idx + o + j);
    if (e >= e0 && e < e0 + n_local) v[o + j] = __ldg(lv + q++);
  }
}

// One CTA per token, 128 threads over its 16-byte column chunks.
template <typename TE>
__global__ void __launch_bounds__(128) ep_sum_parts_kernel(
    const int4* __restrict__ parts, int n_parts, long long T, int n16,
    int4* __restrict__ y) {
  constexpr int V = sizeof(TE) == 4 ? 4 : 8;
  const long long t = blockIdx.x;
  for (int c = threadIdx.x; c < n16; c += blockDim.x) {
    float acc[V];
#pragma unroll
    for (int v = 0; v < V; ++v) acc[v] = 0.0f;
    for (int q = 0; q < n_parts; ++q) {
      const int4 w = __ldg(parts + (q * T + t) * n16 + c);
      const uint32_t u[4] = {static_cast<uint32_t>(w.x),
                             static_cast<uint32_t>(w.y),
                             static_cast<uint32_t>(w.z),
                             static_cast<uint32_t>(w.w)};
      if (V == 4) {
#pragma unroll
        for (int v = 0; v < 4; ++v) acc[v] += __uint_as_float(u[v]);
      } else {
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          acc[2 * v] += __uint_as_float(u[v] << 16);
          acc[2 * v + 1] += __uint_as_float(u[v] & 0xffff0000u);
        }
      }
    }
    int4 o;
    if (V == 4) {
      o = make_int4(__float_as_int(acc[0]), __float_as_int(acc[1]),
                    __float_as_int(acc[2]), __float_as_int(acc[3]));
    } else {
      uint32_t p[4];
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        __nv_bfloat162 b = __floats2bfloat162_rn(acc[2 * v], acc[2 * v + 1]);
        p[v] = *reinterpret_cast<uint32_t*>(&b);
      }
      o = make_int4(static_cast<int>(p[0]), static_cast<int>(p[1]),
                    static_cast<int>(p[2]), static_cast<int>(p[3]));
    }
    y[t * n16 + c] = o;
  }
}

inline bool al4(const void* p) {
  return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 3u) == 0;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

moe_status_t moe_ep_check(const moe_config_t* cfg,
                          const int32_t* shard_counts, int32_t* overflow_flag,
                          float* required_factor, int32_t* capacity,
                          moe_stream_t stream) {
  moe_status_t st = validate(cfg);
  if (st != MOE_OK) return st;
  if (!al4(shard_counts) || !al4(overflow_flag) || !al4(required_factor) ||
      !al4(capacity))
    return MOE_ERR_INVALID_ARG;
  ep_check_kernel<<<1, 32, 0, stream>>>(
      shard_counts, cfg->S, capacity_rows(*cfg),
      static_cast<double>(cfg->T) * static_cast<double>(cfg->k),
      overflow_flag, required_factor, capacity);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status_t moe_ep_dispatch_pack(const moe_config_t* cfg, const void* x,
                                  const int32_t* topk_idx,
                                  const float* topk_w,
                                  const int32_t* uniq_offsets,
                                  const int32_t* uniq_tokens, void* x_send,
                                  int32_t* send_idx, float* send_w,
                                  moe_stream_t stream) {
  moe_status_t st = validate(cfg);
  if (st != MOE_OK) return st;
  if (!al4(uniq_offsets)) return MOE_ERR_INVALID_ARG;
  if (cfg->T == 0) return MOE_OK;
  if (!aligned16(x) || x == nullptr || !al4(topk_idx) || !al4(topk_w) ||
      !al4(uniq_tokens) || x_send == nullptr || !aligned16(x_send) ||
      !al4(send_idx) || !al4(send_w))
    return MOE_ERR_INVALID_ARG;
  const int n_max = cfg->T * std::min(cfg->k, cfg->S);
  const int n16 = cfg->H * elem_bytes(cfg->dtype) / 16;
  ep_pack_kernel<<<n_max, kPackThreads, 0, stream>>>(
      static_cast<const int4*>(x), n16, topk_idx, topk_w, cfg->k,
      std::min(cfg->k, cfg->E / cfg->S), cfg->S, cfg->E / cfg->S,
      uniq_offsets, uniq_tokens, static_cast<int4*>(x_send),
      send_idx, send_w);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status_t moe_ep_return_map(const moe_config_t* cfg,
                               const int32_t* uniq_offsets,
                               const int32_t* uniq_tokens,
                               int32_t* row_of_ret, moe_stream_t stream) {
  moe_status_t st = validate(cfg);
  if (st != MOE_OK) return st;
  if (cfg->T == 0) return MOE_OK;
  if (!al4(uniq_offsets) || !al4(uniq_tokens) || !al4(row_of_ret))
    return MOE_ERR_INVALID_ARG;
  const size_t n = static_cast<size_t>(cfg->T) * cfg->S;
  if (cudaMemsetAsync(row_of_ret, 0xff, n * sizeof(int32_t), stream) !=
      cudaSuccess)
    return MOE_ERR_CUDA;
  const int n_max = cfg->T * std::min(cfg->k, cfg->S);
  ep_return_map_kernel<<<(n_max + 255) / 256, 256, 0, stream>>>(
      n_max, cfg->S, uniq_offsets, uniq_tokens, row_of_ret);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status_t moe_ep_localize(const moe_config_t* cfg,
                             const int32_t* topk_idx, const float* topk_w,
                             int32_t first_expert, int32_t n_local,
                             int32_t* local_idx, float* local_w,
                             moe_stream_t stream) {
  moe_status_t st = validate(cfg);
  if (st != MOE_OK) return st;
  if (first_expert < 0 || n_local < 1 || first_expert + n_local > cfg->E)
    return MOE_ERR_INVALID_ARG;
  if (cfg->T == 0) return MOE_OK;
  if (!al4(topk_idx) || !al4(topk_w) || !al4(local_idx) || !al4(local_w))
    return MOE_ERR_INVALID_ARG;
  ep_localize_kernel<<<(cfg->T + 255) / 256, 256, 0, stream>>>(
      topk_idx, topk_w, cfg->T, cfg->k, std::min(cfg->k, n_local),
      first_expert, n_local, local_idx, local_w);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status_t moe_ep_delocalize(const moe_config_t* cfg,
                               const int32_t* topk_idx, int32_t first_expert,
                               int32_t n_local, const int32_t* row_of,
                               int32_t row_stride, const float* local_v,
                               float* v, moe_stream_t stream) {
  moe_status_t st = validate(cfg);
  if (st != MOE_OK) return st;
  if (first_expert < 0 || n_local < 1 || first_expert + n_local > cfg->E)
    return MOE_ERR_INVALID_ARG;
  if (row_of != nullptr && row_stride < 1) return MOE_ERR_INVALID_ARG;
  if (cfg->T == 0) return MOE_OK;
  if (!al4(topk_idx) || !al4(local_v) || !al4(v) ||
      (row_of != nullptr && !al4(row_of)))
    return MOE_ERR_INVALID_ARG;
  ep_delocalize_kernel<<<(cfg->T + 255) / 256, 256, 0, stream>>>(
      topk_idx, row_of, row_stride, local_v, cfg->T, cfg->k,
      std::min(cfg->k, n_local), first_expert, n_local, v);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status_t moe_ep_sum_partials(const moe_config_t* cfg, int32_t n_parts,
                                 const void* parts, void* y,
                                 moe_stream_t stream) {
  moe_status_t st = validate(cfg);
  if (st != MOE_OK) return st;
  if (n_parts < 1) return MOE_ERR_INVALID_ARG;
  if (cfg->T == 0) return MOE_OK;
  if (parts == nullptr || y == nullptr || !aligned16(parts) || !aligned16(y))
    return MOE_ERR_INVALID_ARG;
  const int n16 = cfg->H * elem_bytes(cfg->dtype) / 16;
  if (cfg->dtype == MOE_F32)
    ep_sum_parts_kernel<float><<<cfg->T, 128, 0, stream>>>(
        static_cast<const int4*>(parts), n_parts, cfg->T, n16,
        static_cast<int4*>(y));
  else
    ep_sum_parts_kernel<__nv_bfloat16><<<cfg->T, 128, 0, stream>>>(
        static_cast<const int4*>(parts), n_parts, cfg->T, n16,
        static_cast<int4*>(y));
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // extern "C"
