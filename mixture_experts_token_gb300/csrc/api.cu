// C ABI entry points (include/moe.h): argument validation, workspace layout,
// and the layer drivers that chain the kernels on one stream.
//
// "Support moe_dropless_fallback=layer on the ragged all-to-all MoE path"
// (MaxText pull request 5920), section How: the layer checks for overflow
// from the router's top-k, takes the capped path when no shard overflows
// and otherwise runs the layer over sequence chunks, each with the
// worst-case (force_dropless) buffer, chosen so that this buffer is no
// larger than the capped one.  Section Shortcomings: an overflowing layer
// costs about n_chunks passes.
#include <cmath>
#include <cstdint>
#include <limits>

#include "internal.h"

namespace moe {

cudaError_t launch_gmm1_f32(const moe_config_t& c, const Groups& g,
                            const void* x_sorted,
                            const int32_t* group_offsets, const void* w_gate,
                            const void* w_up, void* h, cudaStream_t s);
cudaError_t launch_gmm2_f32(const moe_config_t& c, const Groups& g,
                            const void* h, const int32_t* group_offsets,
                            const void* w_down, void* y_sorted,
                            cudaStream_t s);
cudaError_t launch_gmm1_bf16(const moe_config_t& c, const Groups& g,
                             const void* x_sorted,
                             const int32_t* group_offsets, const void* w_gate,
                             const void* w_up, void* h, int32_t* status,
                             cudaStream_t s);
cudaError_t launch_gmm2_bf16(const moe_config_t& c, const Groups& g,
                             const void* h, const int32_t* group_offsets,
                             const void* w_down, void* y_sorted,
                             int32_t* status, cudaStream_t s);

int64_t capacity_rows(const moe_config_t& c) {
  const double f = static_cast<double>(c.ragged_buffer_factor);
  if (!(f > 0.0)) return -1;  // <= 0 or NaN: uncapped
  const double v = std::floor(f * static_cast<double>(c.T) *
                              static_cast<double>(c.k) /
                              static_cast<double>(c.S));
  const int64_t rows = static_cast<int64_t>(c.T) * c.k;
  if (v >= static_cast<double>(rows)) return rows;
  return static_cast<int64_t>(v);
}

int32_t chunk_tokens(const moe_config_t& c) {
  if (c.T <= 0) return 0;
  int64_t tok;
  if (c.n_chunks > 0) {
    tok = (static_cast<int64_t>(c.T) + c.n_chunks - 1) / c.n_chunks;
  } else {
    const int64_t cap = capacity_rows(c);
    if (cap < 0) {
      tok = c.T;
    } else {
      const int64_t worst_per_token = std::min(c.k, c.E / c.S);
      tok = std::max<int64_t>(1, cap / worst_per_token);
    }
  }
  return static_cast<int32_t>(std::min<int64_t>(tok, c.T));
}

cudaError_t launch_gmm1(const moe_config_t& c, const Groups& g,
                        const void* x_sorted, const int32_t* group_offsets,
                        const void* w_gate, const void* w_up, void* h,
                        int32_t* status, cudaStream_t s) {
  if (c.dtype == MOE_F32)
    return launch_gmm1_f32(c, g, x_sorted, group_offsets, w_gate, w_up, h, s);
  return launch_gmm1_bf16(c, g, x_sorted, group_offsets, w_gate, w_up, h,
                          status, s);
}

cudaError_t launch_gmm2(const moe_config_t& c, const Groups& g, const void* h,
                        const int32_t* group_offsets, const void* w_down,
                        void* y_sorted, int32_t* status, cudaStream_t s) {
  if (c.dtype == MOE_F32)
    return launch_gmm2_f32(c, g, h, group_offsets, w_down, y_sorted, s);
  return launch_gmm2_bf16(c, g, h, group_offsets, w_down, y_sorted, status,
                          s);
}

cudaError_t launch_gmm(const moe_config_t& c, const Groups& g,
                       const void* x_sorted, const int32_t* group_offsets,
                       const void* w_gate, const void* w_up,
                       const void* w_down, void* h, void* y_sorted,
                       int32_t* status, cudaStream_t s) {
  cudaError_t e =
      launch_gmm1(c, g, x_sorted, group_offsets, w_gate, w_up, h, status, s);
  if (e != cudaSuccess) return e;
  return launch_gmm2(c, g, h, group_offsets, w_down, y_sorted, status, s);
}

moe_status_t validate(const moe_config_t* c) {
  if (c == nullptr) return MOE_ERR_INVALID_ARG;
  if (c->T < 0 || c->H < 1 || c->F < 0) return MOE_ERR_INVALID_ARG;
  if (c->E < 1 || c->E > kMaxExperts) return MOE_ERR_INVALID_ARG;
  if (c->k < 1 || c->k > c->E || c->k > kMaxTopK) return MOE_ERR_INVALID_ARG;
  if (c->S < 1 || c->S > kMaxShards || c->E % c->S != 0)
    return MOE_ERR_INVALID_ARG;
  if (c->dtype != MOE_F32 && c->dtype != MOE_BF16) return MOE_ERR_INVALID_ARG;
  if (c->renorm != 0 && c->renorm != 1) return MOE_ERR_INVALID_ARG;
  if (c->n_chunks < 0) return MOE_ERR_INVALID_ARG;
  if (std::isnan(c->ragged_buffer_factor)) return MOE_ERR_INVALID_ARG;
  if (c->redundant_slots < 0 ||
      static_cast<int64_t>(c->E) +
              static_cast<int64_t>(c->S) * c->redundant_slots >
          kMaxExperts)
    return MOE_ERR_INVALID_ARG;
  const int eb = elem_bytes(c->dtype);
  if ((static_cast<int64_t>(c->H) * eb) % 16 != 0) return MOE_ERR_INVALID_ARG;
  if ((static_cast<int64_t>(c->F) * eb) % 16 != 0) return MOE_ERR_INVALID_ARG;
  const int64_t rows = static_cast<int64_t>(c->T) * c->k;
  if (rows > std::numeric_limits<int32_t>::max()) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

bool ok_ptr(const void* p, bool need16) {
  if (p == nullptr) return false;
  const uintptr_t u = reinterpret_cast<uintptr_t>(p);
  return need16 ? (u & 15u) == 0 : (u & 3u) == 0;
}

moe_status_t cuda_status(cudaError_t e) {
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

LayerBufs carve_layer(void* base, const moe_config_t& c, int T,
                      size_t* bytes) {
  Carve cv(base);
  LayerBufs b;
  const size_t tk = static_cast<size_t>(T) * c.k;
  const size_t eb = elem_bytes(c.dtype);
  b.topk_idx = cv.take<int32_t>(tk);
  b.topk_w = cv.take<float>(tk);
  b.counts = cv.take<int32_t>(c.E);
  b.offsets = cv.take<int32_t>(c.E + 1);
  b.shard = cv.take<int32_t>(c.S);
  b.flag = cv.take<int32_t>(1);
  b.req = cv.take<float>(1);
  b.cap = cv.take<int32_t>(1);
  b.row_of = cv.take<int32_t>(tk);
  b.sorted_token = cv.take<int32_t>(tk);
  b.group_offsets = cv.take<int32_t>(num_groups(c) + 1);
  b.uniq_offsets = cv.take<int32_t>(c.S + 1);
  b.uniq_tokens =
      cv.take<int32_t>(static_cast<size_t>(T) * std::min(c.k, c.S));
  b.expand_idx = cv.take<int32_t>(tk);
  b.n_dropped = cv.take<int32_t>(1);
  b.divert = cv.take<int32_t>(c.E);
  b.slot_of = cv.take<int32_t>(c.E);
  b.group_expert = cv.take<int32_t>(num_groups(c));
  b.shard_after = cv.take<int32_t>(c.S);
  b.flag_after = cv.take<int32_t>(1);
  b.pws = carve_permute_scratch(cv, T, c.E, c.k, c.S);
  b.x_sorted = cv.take<char>(tk * c.H * eb);
  b.h = cv.take<char>(tk * static_cast<size_t>(c.F) * eb);
  b.y_sorted = cv.take<char>(tk * c.H * eb);
  b.alt.sorted_token = cv.take<int32_t>(tk);
  b.alt.group_offsets = cv.take<int32_t>(num_groups(c) + 1);
  b.alt.uniq_offsets = cv.take<int32_t>(c.S + 1);
  b.alt.uniq_tokens =
      cv.take<int32_t>(static_cast<size_t>(T) * std::min(c.k, c.S));
  b.alt.expand_idx = cv.take<int32_t>(tk);
  b.alt.n_dropped = cv.take<int32_t>(1);
  b.alt.pws = carve_permute_scratch(cv, T, c.E, c.k, c.S);
  b.row_of_alt = cv.take<int32_t>(tk);
  if (bytes) *bytes = align_up(cv.off, 256);
  return b;
}

size_t layer_bytes(const moe_config_t& c, int T) {
  size_t n = 0;
  carve_layer(nullptr, c, T, &n);
  return n;
}

moe_config_t sub_config(const moe_config_t& c, int T) {
  moe_config_t s = c;
  s.T = T;
  s.ragged_buffer_factor = -1.0f;
  s.n_chunks = 0;
  s.redundant_slots = 0;
  return s;
}

// One pass on tokens whose routing is already in `topk_idx/topk_w`:
// permute (cap or uncapped) -> grouped FFN -> combine into y.
namespace {
__global__ void stamp_kernel(int64_t* slot) {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  *slot = static_cast<int64_t>(t);
}
}  // namespace

cudaError_t stamp(int64_t* trace, int slot, cudaStream_t s) {
  if (trace == nullptr) return cudaSuccess;
  stamp_kernel<<<1, 1, 0, s>>>(trace + slot);
  return cudaGetLastError();
}

cudaError_t pass(const moe_config_t& c, const void* x, const int32_t* topk_idx,
                 const float* topk_w, int64_t cap, const void* wg,
                 const void* wu, const void* wd, void* y, const LayerBufs& b,
                 int32_t* status, cudaStream_t s, bool planned,
                 int pass_index) {
  PermutePlan plan;
  Groups groups = identity_groups(c);
  if (planned && c.redundant_slots > 0) {
    plan.divert = b.divert;
    plan.slot_of = b.slot_of;
    plan.B = c.redundant_slots;
    groups = {num_groups(c), b.group_expert};
  }
  if (cap >= 0)  // a capped pass keeps at most S*C rows
    groups.max_rows = std::min<int64_t>(static_cast<int64_t>(c.T) * c.k,
                                        static_cast<int64_t>(c.S) * cap);
  int64_t* tr = b.trace;
  cudaError_t e = stamp(tr, trace_slot(pass_index, 0), s);
  if (e != cudaSuccess) return e;
  e = launch_permute(c, x, topk_idx, cap, b.x_sorted, b.row_of,
                     b.sorted_token, b.group_offsets, b.uniq_offsets,
                     b.uniq_tokens, b.expand_idx, b.n_dropped, b.pws, status,
                     s, plan);
  if (e != cudaSuccess) return e;
  const bool ffn = c.F > 0;  // F = 0: dispatch only, combine of x_sorted
  if (tr == nullptr) {
    if (ffn)
      e = launch_gmm(c, groups, b.x_sorted, b.group_offsets, wg, wu, wd, b.h,
                     b.y_sorted, status, s);
  } else if ((e = stamp(tr, trace_slot(pass_index, 1), s)) == cudaSuccess &&
             (!ffn || (e = launch_gmm1(c, groups, b.x_sorted,
                                       b.group_offsets, wg, wu, b.h, status,
                                       s)) == cudaSuccess) &&
             (e = stamp(tr, trace_slot(pass_index, 2), s)) == cudaSuccess) {
    if (ffn)
      e = launch_gmm2(c, groups, b.h, b.group_offsets, wd, b.y_sorted,
                      status, s);
  }
  if (e != cudaSuccess) return e;
  if ((e = stamp(tr, trace_slot(pass_index, 3), s)) != cudaSuccess) return e;
  e = launch_combine(c, ffn ? b.y_sorted : b.x_sorted, b.row_of, topk_w, y,
                     s);
  if (e != cudaSuccess) return e;
  return stamp(tr, trace_slot(pass_index, 4), s);
}

// The chunked fallback with each chunk's permute tables computed one chunk
// ahead on pp.side, so that they overlap the previous chunk's expert FFN.
// Chunk i uses table set i % 2 and its own rows of row_of; the tables of
// chunk i+2 wait for chunk i's combine.  Chunk 0's tables run on s.
cudaError_t pipelined_passes(const moe_config_t& c, const void* x,
                             const int32_t* topk_idx, const float* topk_w,
                             const void* wg, const void* wu, const void* wd,
                             void* y, const LayerBufs& b, int32_t* status,
                             cudaStream_t s, int n, const PassPipeline& pp) {
  const int ct = chunk_tokens(c);
  const size_t row_bytes = static_cast<size_t>(c.H) * elem_bytes(c.dtype);
  cudaError_t e;
  if ((e = cudaEventRecord(pp.fork, s)) != cudaSuccess ||
      (e = cudaStreamWaitEvent(pp.side, pp.fork, 0)) != cudaSuccess)
    return e;
  auto tables = [&](int i, cudaStream_t st) -> cudaError_t {
    const int t0 = i * ct, tc = std::min(ct, c.T - t0);
    const PassTables tb = b.tables(i);
    const size_t o = static_cast<size_t>(t0) * c.k;
    cudaError_t r;
    if (st == pp.side && i >= 2 &&
        (r = cudaStreamWaitEvent(st, pp.done[i & 1], 0)) != cudaSuccess)
      return r;
    if ((r = launch_permute_tables(sub_config(c, tc), topk_idx + o, -1,
                                   b.row_of + o, tb.sorted_token,
                                   tb.group_offsets, tb.uniq_offsets,
                                   tb.n_dropped, tb.pws, status, st)) !=
        cudaSuccess)
      return r;
    return st == pp.side ? cudaEventRecord(pp.ready[i & 1], st) : cudaSuccess;
  };
  for (int i = 0; i < n; ++i) {
    const int t0 = i * ct, tc = std::min(ct, c.T - t0);
    const moe_config_t sc = sub_config(c, tc);
    const PassTables tb = b.tables(i);
    const size_t o = static_cast<size_t>(t0);
    int64_t* tr = b.trace;
    if ((e = stamp(tr, trace_slot(i, 0), s)) != cudaSuccess) return e;
    e = i == 0 ? (pp.first_ready ? cudaSuccess : tables(0, s))
               : cudaStreamWaitEvent(s, pp.ready[i & 1], 0);
    if (e != cudaSuccess) return e;
    if ((e = launch_permute_scatter(
             sc, static_cast<const char*>(x) + o * row_bytes,
             b.row_of + o * c.k, tb.uniq_offsets, b.x_sorted, tb.uniq_tokens,
             tb.expand_idx, tb.pws, s)) != cudaSuccess ||
        (e = stamp(tr, trace_slot(i, 1), s)) != cudaSuccess ||
        (c.F > 0 &&
         (e = launch_gmm1(sc, identity_groups(sc), b.x_sorted,
                          tb.group_offsets, wg, wu, b.h, status, s)) !=
             cudaSuccess) ||
        (e = stamp(tr, trace_slot(i, 2), s)) != cudaSuccess ||
        (c.F > 0 &&
         (e = launch_gmm2(sc, identity_groups(sc), b.h, tb.group_offsets, wd,
                          b.y_sorted, status, s)) != cudaSuccess) ||
        (e = stamp(tr, trace_slot(i, 3), s)) != cudaSuccess ||
        (e = launch_combine(sc, c.F > 0 ? b.y_sorted : b.x_sorted,
                            b.row_of + o * c.k,
                            topk_w + o * c.k,
                            static_cast<char*>(y) + o * row_bytes, s)) !=
            cudaSuccess ||
        (e = stamp(tr, trace_slot(i, 4), s)) != cudaSuccess ||
        (e = cudaEventRecord(pp.done[i & 1], s)) != cudaSuccess)
      return e;
    if (i + 1 < n && (e = tables(i + 1, pp.side)) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t capped_pass_tabled(const moe_config_t& c, const void* x,
                               const float* topk_w, const void* wg,
                               const void* wu, const void* wd, void* y,
                               const LayerBufs& b, const int32_t* row_of,
                               const PassTables& tb, int32_t* status,
                               cudaStream_t s) {
  int64_t* tr = b.trace;
  Groups groups = identity_groups(c);
  groups.max_rows = std::min<int64_t>(static_cast<int64_t>(c.T) * c.k,
                                      static_cast<int64_t>(c.S) *
                                          std::max<int64_t>(capacity_rows(c),
                                                            0));
  cudaError_t e;
  if ((e = stamp(tr, trace_slot(0, 0), s)) != cudaSuccess ||
      (e = launch_permute_scatter(c, x, row_of, tb.uniq_offsets, b.x_sorted,
                                  tb.uniq_tokens, tb.expand_idx, tb.pws, s)) !=
          cudaSuccess ||
      (e = stamp(tr, trace_slot(0, 1), s)) != cudaSuccess ||
      (c.F > 0 &&
       (e = launch_gmm1(c, groups, b.x_sorted, tb.group_offsets, wg, wu, b.h,
                        status, s)) != cudaSuccess) ||
      (e = stamp(tr, trace_slot(0, 2), s)) != cudaSuccess ||
      (c.F > 0 &&
       (e = launch_gmm2(c, groups, b.h, tb.group_offsets, wd, b.y_sorted,
                        status, s)) != cudaSuccess) ||
      (e = stamp(tr, trace_slot(0, 3), s)) != cudaSuccess ||
      (e = launch_combine(c, c.F > 0 ? b.y_sorted : b.x_sorted, row_of,
                          topk_w, y, s)) != cudaSuccess)
    return e;
  return stamp(tr, trace_slot(0, 4), s);
}

// The chunked dropless fallback over precomputed routing.
cudaError_t chunked_passes(const moe_config_t& c, const void* x,
                           const int32_t* topk_idx, const float* topk_w,
                           const void* wg, const void* wu, const void* wd,
                           void* y, const LayerBufs& b, int32_t* status,
                           cudaStream_t s, int32_t* n_run,
                           const PassPipeline* pp) {
  const int ct = chunk_tokens(c);
  const size_t row_bytes = static_cast<size_t>(c.H) * elem_bytes(c.dtype);
  const int n_all = ct > 0 ? (c.T + ct - 1) / ct : 0;
  if (pp != nullptr && n_all >= 2) {
    if (n_run) *n_run = n_all;
    return pipelined_passes(c, x, topk_idx, topk_w, wg, wu, wd, y, b, status,
                            s, n_all, *pp);
  }
  int n = 0;
  for (int t0 = 0; t0 < c.T; t0 += ct, ++n) {
    const int tc = std::min(ct, c.T - t0);
    const moe_config_t sc = sub_config(c, tc);
    const size_t o = static_cast<size_t>(t0);
    cudaError_t e = pass(sc, static_cast<const char*>(x) + o * row_bytes,
                         topk_idx + o * c.k, topk_w + o * c.k, -1, wg, wu, wd,
                         static_cast<char*>(y) + o * row_bytes, b, status, s,
                         false, n);
    if (e != cudaSuccess) return e;
  }
  if (n_run) *n_run = n;
  return cudaSuccess;
}

bool gmm_shape_ok(const moe_config_t& c) {
  if (c.F < 1) return false;
  return c.dtype == MOE_F32 || gmm_tc_supported(c);
}

bool weights_ok(const void* wg, const void* wu, const void* wd) {
  return ok_ptr(wg, true) && ok_ptr(wu, true) && ok_ptr(wd, true);
}

}  // namespace moe

using namespace moe;

extern "C" {

moe_status_t moe_validate_config(const moe_config_t* cfg) {
  return validate(cfg);
}

int64_t moe_capacity_rows(const moe_config_t* cfg) {
  if (validate(cfg) != MOE_OK) return -1;
  return capacity_rows(*cfg);
}

int32_t moe_chunk_tokens(const moe_config_t* cfg) {
  if (validate(cfg) != MOE_OK) return 0;
  return chunk_tokens(*cfg);
}

int32_t moe_num_chunks(const moe_config_t* cfg) {
  if (validate(cfg) != MOE_OK) return 0;
  const int ct = chunk_tokens(*cfg);
  return ct > 0 ? (cfg->T + ct - 1) / ct : 0;
}

int32_t moe_gmm_kernel_choice(const moe_config_t* cfg, int32_t n_groups,
                              int64_t rows_bound) {
  if (validate(cfg) != MOE_OK || n_groups < 0 || n_groups > kMaxExperts)
    return -1;
  Groups g = identity_groups(*cfg);
  if (n_groups > 0) g.n = n_groups;
  if (rows_bound > 0) g.max_rows = rows_bound;
  return gmm_pair_kinds(*cfg, g);
}

size_t moe_workspace_bytes(const moe_config_t* cfg, moe_ws_kind_t which) {
  if (validate(cfg) != MOE_OK) return 0;
  switch (which) {
    case MOE_WS_PERMUTE:
      return permute_scratch_bytes(cfg->T, cfg->E, cfg->k, cfg->S);
    case MOE_WS_CHUNKED:
      return layer_bytes(*cfg, chunk_tokens(*cfg));
    case MOE_WS_LAYER:
      return layer_bytes(*cfg, cfg->T);
    case MOE_WS_GMM_BACKWARD:
      return gmm_backward_bytes(*cfg);
    case MOE_WS_LAYER_BACKWARD:
      return layer_backward_bytes(*cfg);
  }
  return 0;
}

void moe_test_stall_gemm_producer(int64_t fills) {
  set_gemm_stall_for_tests(fills);
}

const char* moe_status_string(moe_status_t st) {
  switch (st) {
    case MOE_OK:
      return "ok";
    case MOE_ERR_INVALID_ARG:
      return "invalid argument";
    case MOE_ERR_UNSUPPORTED:
      return "shape not supported by the kernels";
    case MOE_ERR_WORKSPACE:
      return "workspace missing or too small";
    case MOE_ERR_CUDA:
      return "CUDA error";
  }
  return "unknown status";
}

moe_status_t moe_route(const moe_config_t* cfg, const float* logits,
                       int32_t* topk_idx, float* topk_w, int32_t* status_word,
                       moe_stream_t stream) {
  moe_status_t st = validate(cfg);
  if (st != MOE_OK) return st;
  if (cfg->T == 0) return MOE_OK;
  if (!ok_ptr(logits, false) || !ok_ptr(topk_idx, false) ||
      !ok_ptr(topk_w, false))
    return MOE_ERR_INVALID_ARG;
  return cuda_status(
      launch_route(*cfg, logits, topk_idx, topk_w, status_word, stream));
}

moe_status_t moe_check_overflow(const moe_config_t* cfg,
                                const int32_t* topk_idx,
                                int32_t* expert_counts,
                                int32_t* expert_offsets,
                                int32_t* shard_counts, int32_t* overflow_flag,
                                float* required_factor, int32_t* capacity,
                                moe_stream_t stream) {
  moe_status_t st = validate(cfg);
  if (st != MOE_OK) return st;
  if ((cfg->T > 0 && !ok_ptr(topk_idx, false)) ||
      !ok_ptr(expert_counts, false) || !ok_ptr(expert_offsets, false) ||
      !ok_ptr(shard_counts, false) || !ok_ptr(overflow_flag, false) ||
      !ok_ptr(required_factor, false) || !ok_ptr(capacity, false))
    return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_check(*cfg, topk_idx, expert_counts,
                                  expert_offsets, shard_counts, overflow_flag,
                                  required_factor, capacity, stream));
}

moe_status_t moe_permute(const moe_config_t* cfg, const void* x,
                         const int32_t* topk_idx, int32_t capped,
                         void* x_sorted, int32_t* row_of,
                         int32_t* sorted_token, int32_t* group_offsets,
                         int32_t* uniq_offsets, int32_t* uniq_tokens,
                         int32_t* expand_idx, int32_t* n_dropped,
                         void* workspace, size_t workspace_bytes,
                         moe_stream_t stream) {
  moe_status_t st = validate(cfg);
  if (st != MOE_OK) return st;
  if (!ok_ptr(group_offsets, false) || !ok_ptr(uniq_offsets, false) ||
      !ok_ptr(n_dropped, false))
    return MOE_ERR_INVALID_ARG;
  if (cfg->T > 0 &&
      (!ok_ptr(x, true) || !ok_ptr(topk_idx, false) ||
       !ok_ptr(x_sorted, true) || !ok_ptr(row_of, false) ||
       !ok_ptr(sorted_token, false) || !ok_ptr(uniq_tokens, false) ||
       !ok_ptr(expand_idx, false)))
    return MOE_ERR_INVALID_ARG;
  const size_t need =
      permute_scratch_bytes(cfg->T, cfg->E, cfg->k, cfg->S);
  if (workspace == nullptr || workspace_bytes < need ||
      !ok_ptr(workspace, true))
    return MOE_ERR_WORKSPACE;
  Carve cv(workspace);
  const PermuteScratch ws =
      carve_permute_scratch(cv, cfg->T, cfg->E, cfg->k, cfg->S);
  const int64_t cap = capped ? capacity_rows(*cfg) : -1;
  return cuda_status(launch_permute(*cfg, x, topk_idx, cap, x_sorted, row_of,
                                    sorted_token, group_offsets, uniq_offsets,
                                    uniq_tokens, expand_idx, n_dropped, ws,
                                    nullptr, stream));
}

moe_status_t moe_gmm_swiglu(const moe_config_t* cfg, const void* x_sorted,
                            const int32_t* group_offsets, const void* w_gate,
                            const void* w_up, const void* w_down, void* h,
                            void* y_sorted, int32_t* status_word,
                            moe_stream_t stream) {
  moe_status_t st = validate(cfg);
  if (st != MOE_OK) return st;
  if (cfg->F < 1) return MOE_ERR_INVALID_ARG;
  if (!gmm_shape_ok(*cfg)) return MOE_ERR_UNSUPPORTED;
  if (cfg->T == 0) return MOE_OK;
  if (!ok_ptr(x_sorted, true) || !ok_ptr(group_offsets, false) ||
      !weights_ok(w_gate, w_up, w_down) || !ok_ptr(h, true) ||
      !ok_ptr(y_sorted, true))
    return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_gmm(*cfg, identity_groups(*cfg), x_sorted,
                                group_offsets, w_gate, w_up, w_down, h,
                                y_sorted, status_word, stream));
}

namespace {
// n_groups = 0 with a null map: the experts' own groups.
bool groups_of(const moe_config_t& c, int32_t n, const int32_t* map,
               Groups* g) {
  if (n == 0 && map == nullptr) {
    *g = identity_groups(c);
    return true;
  }
  if (n < 1 || n > kMaxExperts || !ok_ptr(map, false)) return false;
  *g = {n, map};
  return true;
}
}  // namespace

moe_status_t moe_gmm_gate_up(const moe_config_t* cfg, int32_t n_groups,
                             const int32_t* group_expert,
                             const void* x_sorted,
                             const int32_t* group_offsets, const void* w_gate,
                             const void* w_up, void* h, int32_t* status_word,
                             moe_stream_t stream) {
  moe_status_t st = validate(cfg);
  if (st != MOE_OK) return st;
  Groups g;
  if (cfg->F < 1 || !groups_of(*cfg, n_groups, group_expert, &g))
    return MOE_ERR_INVALID_ARG;
  if (!gmm_shape_ok(*cfg)) return MOE_ERR_UNSUPPORTED;
  if (cfg->T == 0) return MOE_OK;
  if (!ok_ptr(x_sorted, true) || !ok_ptr(group_offsets, false) ||
      !ok_ptr(w_gate, true) || !ok_ptr(w_up, true) || !ok_ptr(h, true))
    return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_gmm1(*cfg, g, x_sorted, group_offsets, w_gate,
                                 w_up, h, status_word, stream));
}

moe_status_t moe_gmm_down(const moe_config_t* cfg, int32_t n_groups,
                          const int32_t* group_expert, const void* h,
                          const int32_t* group_offsets, const void* w_down,
                          void* y_sorted, int32_t* status_word,
                          moe_stream_t stream) {
  moe_status_t st = validate(cfg);
  if (st != MOE_OK) return st;
  Groups g;
  if (cfg->F < 1 || !groups_of(*cfg, n_groups, group_expert, &g))
    return MOE_ERR_INVALID_ARG;
  if (!gmm_shape_ok(*cfg)) return MOE_ERR_UNSUPPORTED;
  if (cfg->T == 0) return MOE_OK;
  if (!ok_ptr(h, true) || !ok_ptr(group_offsets, false) ||
      !ok_ptr(w_down, true) || !ok_ptr(y_sorted, true))
    return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_gmm2(*cfg, g, h, group_offsets, w_down, y_sorted,
                                 status_word, stream));
}

moe_status_t moe_plan_duplication(const moe_config_t* cfg,
                                  const int32_t* expert_counts,
                                  int32_t* divert, int32_t* slot_of,
                                  int32_t* group_expert,
                                  int32_t* shard_counts_after,
                                  int32_t* overflow_flag_after,
                                  moe_stream_t stream) {
  moe_status_t st = validate(cfg);
  if (st != MOE_OK) return st;
  if (!ok_ptr(expert_counts, false) || !ok_ptr(divert, false) ||
      !ok_ptr(slot_of, false) || !ok_ptr(group_expert, false) ||
      !ok_ptr(shard_counts_after, false) || !ok_ptr(overflow_flag_after, false))
    return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_plan(*cfg, expert_counts, divert, slot_of,
                                 group_expert, shard_counts_after,
                                 overflow_flag_after, stream));
}

moe_status_t moe_permute_planned(const moe_config_t* cfg, const void* x,
                                 const int32_t* topk_idx, int32_t capped,
                                 const int32_t* divert,
                                 const int32_t* slot_of, void* x_sorted,
                                 int32_t* row_of, int32_t* sorted_token,
                                 int32_t* group_offsets,
                                 int32_t* uniq_offsets, int32_t* uniq_tokens,
                                 int32_t* expand_idx, int32_t* n_dropped,
                                 void* workspace, size_t workspace_bytes,
                                 moe_stream_t stream) {
  moe_status_t st = validate(cfg);
  if (st != MOE_OK) return st;
  if (!ok_ptr(group_offsets, false) || !ok_ptr(uniq_offsets, false) ||
      !ok_ptr(n_dropped, false) || !ok_ptr(divert, false) ||
      !ok_ptr(slot_of, false))
    return MOE_ERR_INVALID_ARG;
  if (cfg->T > 0 &&
      (!ok_ptr(x, true) || !ok_ptr(topk_idx, false) ||
       !ok_ptr(x_sorted, true) || !ok_ptr(row_of, false) ||
       !ok_ptr(sorted_token, false) || !ok_ptr(uniq_tokens, false) ||
       !ok_ptr(expand_idx, false)))
    return MOE_ERR_INVALID_ARG;
  const size_t need = permute_scratch_bytes(cfg->T, cfg->E, cfg->k, cfg->S);
  if (workspace == nullptr || workspace_bytes < need ||
      !ok_ptr(workspace, true))
    return MOE_ERR_WORKSPACE;
  Carve cv(workspace);
  const PermuteScratch ws =
      carve_permute_scratch(cv, cfg->T, cfg->E, cfg->k, cfg->S);
  PermutePlan plan;
  plan.divert = divert;
  plan.slot_of = slot_of;
  plan.B = cfg->redundant_slots;
  const int64_t cap = capped ? capacity_rows(*cfg) : -1;
  return cuda_status(launch_permute(*cfg, x, topk_idx, cap, x_sorted, row_of,
                                    sorted_token, group_offsets, uniq_offsets,
                                    uniq_tokens, expand_idx, n_dropped, ws,
                                    nullptr, stream, plan));
}

moe_status_t moe_permute_tables(const moe_config_t* cfg,
                                const int32_t* topk_idx, int32_t capped,
                                const int32_t* divert,
                                const int32_t* slot_of, int32_t* row_of,
                                int32_t* sorted_token,
                                int32_t* group_offsets,
                                int32_t* uniq_offsets, int32_t* n_dropped,
                                void* workspace, size_t workspace_bytes,
                                moe_stream_t stream) {
  moe_status_t st = validate(cfg);
  if (st != MOE_OK) return st;
  if ((divert == nullptr) != (slot_of == nullptr)) return MOE_ERR_INVALID_ARG;
  const bool planned = divert != nullptr;
  if (!ok_ptr(group_offsets, false) || !ok_ptr(uniq_offsets, false) ||
      !ok_ptr(n_dropped, false) ||
      (planned && (!ok_ptr(divert, false) || !ok_ptr(slot_of, false))))
    return MOE_ERR_INVALID_ARG;
  if (cfg->T > 0 && (!ok_ptr(topk_idx, false) || !ok_ptr(row_of, false) ||
                     !ok_ptr(sorted_token, false)))
    return MOE_ERR_INVALID_ARG;
  const size_t need = permute_scratch_bytes(cfg->T, cfg->E, cfg->k, cfg->S);
  if (workspace == nullptr || workspace_bytes < need ||
      !ok_ptr(workspace, true))
    return MOE_ERR_WORKSPACE;
  Carve cv(workspace);
  const PermuteScratch ws =
      carve_permute_scratch(cv, cfg->T, cfg->E, cfg->k, cfg->S);
  PermutePlan plan;
  if (planned) {
    plan.divert = divert;
    plan.slot_of = slot_of;
    plan.B = cfg->redundant_slots;
  }
  const int64_t cap = capped ? capacity_rows(*cfg) : -1;
  return cuda_status(launch_permute_tables(*cfg, topk_idx, cap, row_of,
                                           sorted_token, group_offsets,
                                           uniq_offsets, n_dropped, ws,
                                           nullptr, stream, plan));
}

moe_status_t moe_permute_scatter(const moe_config_t* cfg, const void* x,
                                 const int32_t* row_of,
                                 int32_t* uniq_offsets, void* x_sorted,
                                 int32_t* uniq_tokens, int32_t* expand_idx,
                                 const void* workspace,
                                 size_t workspace_bytes,
                                 moe_stream_t stream) {
  moe_status_t st = validate(cfg);
  if (st != MOE_OK) return st;
  if (!ok_ptr(uniq_offsets, false)) return MOE_ERR_INVALID_ARG;
  // x_sorted == NULL: the index outputs only (x is then not read)
  if (cfg->T > 0 &&
      ((x_sorted != nullptr && (!ok_ptr(x, true) || !ok_ptr(x_sorted, true))) ||
       !ok_ptr(row_of, false) || !ok_ptr(uniq_tokens, false) ||
       !ok_ptr(expand_idx, false)))
    return MOE_ERR_INVALID_ARG;
  const size_t need = permute_scratch_bytes(cfg->T, cfg->E, cfg->k, cfg->S);
  if (workspace == nullptr || workspace_bytes < need ||
      !ok_ptr(workspace, true))
    return MOE_ERR_WORKSPACE;
  Carve cv(const_cast<void*>(workspace));
  const PermuteScratch ws =
      carve_permute_scratch(cv, cfg->T, cfg->E, cfg->k, cfg->S);
  return cuda_status(launch_permute_scatter(*cfg, x, row_of, uniq_offsets,
                                            x_sorted, uniq_tokens, expand_idx,
                                            ws, stream));
}

moe_status_t moe_gmm_swiglu_mapped(const moe_config_t* cfg, int32_t n_groups,
                                   const int32_t* group_expert,
                                   const void* x_sorted,
                                   const int32_t* group_offsets,
                                   const void* w_gate, const void* w_up,
                                   const void* w_down, void* h,
                                   void* y_sorted, int32_t* status_word,
                                   moe_stream_t stream) {
  moe_status_t st = validate(cfg);
  if (st != MOE_OK) return st;
  if (cfg->F < 1 || n_groups < 1 || n_groups > kMaxExperts)
    return MOE_ERR_INVALID_ARG;
  if (!gmm_shape_ok(*cfg)) return MOE_ERR_UNSUPPORTED;
  if (cfg->T == 0) return MOE_OK;
  if (!ok_ptr(x_sorted, true) || !ok_ptr(group_offsets, false) ||
      !ok_ptr(group_expert, false) || !weights_ok(w_gate, w_up, w_down) ||
      !ok_ptr(h, true) || !ok_ptr(y_sorted, true))
    return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_gmm(*cfg, {n_groups, group_expert}, x_sorted,
                                group_offsets, w_gate, w_up, w_down, h,
                                y_sorted, status_word, stream));
}

moe_status_t moe_combine(const moe_config_t* cfg, const void* y_sorted,
                         const int32_t* row_of, const float* topk_w, void* y,
                         moe_stream_t stream) {
  moe_status_t st = validate(cfg);
  if (st != MOE_OK) return st;
  if (cfg->T == 0) return MOE_OK;
  if (!ok_ptr(y_sorted, true) || !ok_ptr(row_of, false) ||
      !ok_ptr(topk_w, false) || !ok_ptr(y, true))
    return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_combine(*cfg, y_sorted, row_of, topk_w, y, stream));
}

moe_status_t moe_layer_dropless_chunked(const moe_config_t* cfg,
                                        const void* x, const float* logits,
                                        const void* w_gate, const void* w_up,
                                        const void* w_down, void* y,
                                        int32_t* status_word, void* workspace,
                                        size_t workspace_bytes,
                                        moe_stream_t stream) {
  moe_status_t st = validate(cfg);
  if (st != MOE_OK) return st;
  if (cfg->F < 1) return MOE_ERR_INVALID_ARG;
  if (!gmm_shape_ok(*cfg)) return MOE_ERR_UNSUPPORTED;
  if (cfg->T == 0) return MOE_OK;
  if (!ok_ptr(x, true) || !ok_ptr(logits, false) ||
      !weights_ok(w_gate, w_up, w_down) || !ok_ptr(y, true))
    return MOE_ERR_INVALID_ARG;
  const int ct = chunk_tokens(*cfg);
  if (workspace == nullptr || !ok_ptr(workspace, true) ||
      workspace_bytes < layer_bytes(*cfg, ct))
    return MOE_ERR_WORKSPACE;
  const LayerBufs b = carve_layer(workspace, *cfg, ct, nullptr);
  const size_t row_bytes = static_cast<size_t>(cfg->H) * elem_bytes(cfg->dtype);
  for (int t0 = 0; t0 < cfg->T; t0 += ct) {
    const int tc = std::min(ct, cfg->T - t0);
    const moe_config_t sc = sub_config(*cfg, tc);
    const size_t o = static_cast<size_t>(t0);
    cudaError_t e = launch_route(sc, logits + o * cfg->E, b.topk_idx,
                                 b.topk_w, status_word, stream);
    if (e == cudaSuccess)
      e = pass(sc, static_cast<const char*>(x) + o * row_bytes, b.topk_idx,
               b.topk_w, -1, w_gate, w_up, w_down,
               static_cast<char*>(y) + o * row_bytes, b, status_word, stream);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

moe_status_t moe_layer(const moe_config_t* cfg, const void* x,
                       const float* logits, const void* w_gate,
                       const void* w_up, const void* w_down, void* y,
                       moe_mode_t mode, moe_layer_info_t* info,
                       int32_t* status_word, void* workspace,
                       size_t workspace_bytes, moe_stream_t stream) {
  moe_status_t st = validate(cfg);
  if (st != MOE_OK) return st;
  if (mode != MOE_MODE_FALLBACK_LAYER && mode != MOE_MODE_CAPPED &&
      mode != MOE_MODE_DROPLESS)
    return MOE_ERR_INVALID_ARG;
  // F = 0: the dispatch-only layer (no expert FFN; the combine reads the
  // permuted rows back), the routing/permute/dedup round trip
  if (cfg->F > 0 && !gmm_shape_ok(*cfg)) return MOE_ERR_UNSUPPORTED;
  const int64_t cap = capacity_rows(*cfg);
  if (info) {
    info->overflow = -1;
    info->n_chunks = cfg->T > 0 ? 1 : 0;
    info->capacity = mode == MOE_MODE_DROPLESS ? -1 : cap;
  }
  if (cfg->T == 0) return MOE_OK;
  if (!ok_ptr(x, true) || !ok_ptr(logits, false) ||
      (cfg->F > 0 && !weights_ok(w_gate, w_up, w_down)) || !ok_ptr(y, true))
    return MOE_ERR_INVALID_ARG;
  if (workspace == nullptr || !ok_ptr(workspace, true) ||
      workspace_bytes < layer_bytes(*cfg, cfg->T))
    return MOE_ERR_WORKSPACE;
  const LayerBufs b = carve_layer(workspace, *cfg, cfg->T, nullptr);
  const bool planned = cfg->redundant_slots > 0 && mode != MOE_MODE_DROPLESS;
  cudaError_t e = launch_route(*cfg, logits, b.topk_idx, b.topk_w,
                               status_word, stream);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  if (mode == MOE_MODE_DROPLESS)
    return cuda_status(pass(*cfg, x, b.topk_idx, b.topk_w, -1, w_gate, w_up,
                            w_down, y, b, status_word, stream));
  if (planned || mode == MOE_MODE_FALLBACK_LAYER) {
    e = launch_check(*cfg, b.topk_idx, b.counts, b.offsets, b.shard, b.flag,
                     b.req, b.cap, stream);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
  }
  if (planned) {
    e = launch_plan(*cfg, b.counts, b.divert, b.slot_of, b.group_expert,
                    b.shard_after, b.flag_after, stream);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
  }
  if (mode == MOE_MODE_CAPPED)
    return cuda_status(pass(*cfg, x, b.topk_idx, b.topk_w, cap, w_gate, w_up,
                            w_down, y, b, status_word, stream, planned));
  // moe_dropless_fallback=layer: check (after the plan), read the flag,
  // branch.
  int32_t flag = 0;
  e = cudaMemcpyAsync(&flag, planned ? b.flag_after : b.flag, sizeof(flag),
                      cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  if (info) info->overflow = flag;
  if (!flag)
    return cuda_status(pass(*cfg, x, b.topk_idx, b.topk_w, cap, w_gate, w_up,
                            w_down, y, b, status_word, stream, planned));
  int32_t n = 0;
  e = chunked_passes(*cfg, x, b.topk_idx, b.topk_w, w_gate, w_up, w_down, y,
                     b, status_word, stream, &n);
  if (info) info->n_chunks = n;
  return cuda_status(e);
}

}  // extern "C"
