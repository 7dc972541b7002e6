// Internal declarations shared by the CUDA translation units of
// libmoe_gb300.so.  Nothing here is part of the C ABI (include/moe.h).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>

#include <algorithm>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

// Token block of the counting-sort permute: one thread per token.
constexpr int kPermuteTokensPerBlock = 128;
constexpr int kMaxExperts = 1024;
constexpr int kMaxTopK = 32;
constexpr int kMaxShards = 64;

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

inline int elem_bytes(moe_dtype_t d) { return d == MOE_F32 ? 4 : 2; }

inline bool aligned16(const void* p) {
  return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

// Bump allocator over a caller-provided workspace (no device allocation).
struct Carve {
  char* base;
  size_t off = 0;
  explicit Carve(void* b) : base(static_cast<char*>(b)) {}
  template <typename T>
  T* take(size_t count) {
    off = align_up(off, 256);
    T* p = base ? reinterpret_cast<T*>(base + off) : nullptr;
    off += count * sizeof(T);
    return p;
  }
};

// Permute scratch for `T` tokens (counting-sort block tables).
struct PermuteScratch {
  int32_t* block_base;  // [nb, E] per-block expert counts, then bases
  int32_t* etab;        // [6, E] per expert: rows kept in its own group,
                        // that group's kept offset, rows routed to its own
                        // group, rows kept in its duplicate slot, the
                        // slot's kept offset, the slot's shard
  int32_t* block_ucnt;  // [nb, S] per-block unique counts, then bases
  int32_t* urank;       // [T*k] (rank of (t,j)'s token among the members of
                        // its shard in its block) * 64 + shard, -1 dropped
  int32_t* scal;        // [4] scalars
};
// Redundancy plan of a permute (all null / 0: none).
struct PermutePlan {
  const int32_t* divert = nullptr;   // [E]
  const int32_t* slot_of = nullptr;  // [E]
  int B = 0;                         // slots per shard
};
inline int num_groups(const moe_config_t& c) {
  return c.S * (c.E / c.S + c.redundant_slots);
}
size_t permute_scratch_bytes(int T, int E, int k, int S);
PermuteScratch carve_permute_scratch(Carve& c, int T, int E, int k, int S);

// Device work of each entry point, already validated.
cudaError_t launch_route(const moe_config_t& c, const float* logits,
                         int32_t* topk_idx, float* topk_w, int32_t* status,
                         cudaStream_t s);
cudaError_t launch_check(const moe_config_t& c, const int32_t* topk_idx,
                         int32_t* counts, int32_t* offsets, int32_t* shard,
                         int32_t* flag, float* req, int32_t* cap,
                         cudaStream_t s);
cudaError_t launch_permute(const moe_config_t& c, const void* x,
                           const int32_t* topk_idx, int64_t cap,
                           void* x_sorted, int32_t* row_of,
                           int32_t* sorted_token, int32_t* group_offsets,
                           int32_t* uniq_offsets, int32_t* uniq_tokens,
                           int32_t* expand_idx, int32_t* n_dropped,
                           const PermuteScratch& ws, int32_t* status,
                           cudaStream_t s, const PermutePlan& plan = {});
// The two halves of launch_permute: the counting-sort tables (row_of,
// sorted_token, group_offsets, n_dropped, and the scatter's tables in ws),
// then the row copy with the dedup indices.  uniq_offsets is complete after
// the scatter.  Between the two, ws must not be reused.
cudaError_t launch_permute_tables(const moe_config_t& c,
                                  const int32_t* topk_idx, int64_t cap,
                                  int32_t* row_of, int32_t* sorted_token,
                                  int32_t* group_offsets,
                                  int32_t* uniq_offsets, int32_t* n_dropped,
                                  const PermuteScratch& ws, int32_t* status,
                                  cudaStream_t s, const PermutePlan& plan = {});
cudaError_t launch_permute_scatter(const moe_config_t& c, const void* x,
                                   const int32_t* row_of,
                                   int32_t* uniq_offsets, void* x_sorted,
                                   int32_t* uniq_tokens, int32_t* expand_idx,
                                   const PermuteScratch& ws, cudaStream_t s);
cudaError_t launch_plan(const moe_config_t& c, const int32_t* counts,
                        int32_t* divert, int32_t* slot_of,
                        int32_t* group_expert, int32_t* shard_after,
                        int32_t* flag_after, cudaStream_t s);
// Row groups of a grouped GEMM: n groups; group g uses the weights of
// expert map[g] (identity when map is null).
struct Groups {
  int n;
  const int32_t* map;
  // Upper bound on the rows the groups hold, known on the host (a capped
  // pass keeps at most S*C rows); -1: the allocation, T*k rows.
  int64_t max_rows = -1;
};
inline Groups identity_groups(const moe_config_t& c) { return {c.E, nullptr}; }

// Which bf16 GEMMs take the two-SM (CTA pair) kernel for these groups:
// bit 0 GEMM1 + SwiGLU, bit 1 GEMM2.
int gmm_pair_kinds(const moe_config_t& c, const Groups& g);

// GEMM1 + SwiGLU (h) and GEMM2 (y_sorted), each one kernel launch.
cudaError_t launch_gmm1(const moe_config_t& c, const Groups& g,
                        const void* x_sorted, const int32_t* group_offsets,
                        const void* w_gate, const void* w_up, void* h,
                        int32_t* status, cudaStream_t s);
cudaError_t launch_gmm2(const moe_config_t& c, const Groups& g, const void* h,
                        const int32_t* group_offsets, const void* w_down,
                        void* y_sorted, int32_t* status, cudaStream_t s);
cudaError_t launch_gmm(const moe_config_t& c, const Groups& g,
                       const void* x_sorted, const int32_t* group_offsets,
                       const void* w_gate, const void* w_up,
                       const void* w_down, void* h, void* y_sorted,
                       int32_t* status, cudaStream_t s);
cudaError_t launch_combine(const moe_config_t& c, const void* y_sorted,
                           const int32_t* row_of, const float* topk_w,
                           void* y, cudaStream_t s);

// A pass's permute tables (one set per pass in flight).
struct PassTables {
  int32_t *sorted_token, *group_offsets, *uniq_offsets, *uniq_tokens,
      *expand_idx, *n_dropped;
  PermuteScratch pws;
};
// Buffers of one layer pass over up to `T` tokens, carved from a workspace.
struct LayerBufs {
  int32_t *topk_idx, *counts, *offsets, *shard, *flag, *cap;
  float *topk_w, *req;
  int32_t *row_of, *sorted_token, *group_offsets, *uniq_offsets,
      *uniq_tokens, *expand_idx, *n_dropped;
  // redundancy plan (sized for cfg.redundant_slots; unused when 0)
  int32_t *divert, *slot_of, *group_expert, *shard_after, *flag_after;
  PermuteScratch pws;
  void *x_sorted, *h, *y_sorted;
  PassTables alt;  // a second table set, for pipelined chunked passes
  int32_t* row_of_alt;  // [T*k] row_of of the capped pass whose tables a
                        // layer graph computes before its branch
  // Stage timestamps of a traced layer graph (device int64, slots of
  // trace_slot below), or null: no stamps.
  int64_t* trace = nullptr;
  PassTables tables(int i) const {  // set i % 2
    if (i & 1) return alt;
    return {sorted_token, group_offsets, uniq_offsets, uniq_tokens,
            expand_idx, n_dropped, pws};
  }
};
// Streams and events for chunked passes whose permute tables run one pass
// ahead on a side stream (see chunked_passes).
struct PassPipeline {
  cudaStream_t side;
  cudaEvent_t fork, ready[2], done[2];
  bool first_ready = false;  // chunk 0's tables (set 0) already computed
};
LayerBufs carve_layer(void* base, const moe_config_t& c, int T,
                      size_t* bytes);
size_t layer_bytes(const moe_config_t& c, int T);
moe_config_t sub_config(const moe_config_t& c, int T);
// Trace slots of a layer graph (moe.h, moe_layer_graph_create_traced):
// 0 layer start, 1 routing done, 2 check (and plan) done; pass p's stage
// boundaries at 3 + 5p + {0 start, 1 GEMM1, 2 GEMM2, 3 combine, 4 end}.
constexpr int kTraceHead = 3;
constexpr int kTracePerPass = 5;
inline int trace_slot(int pass, int stage) {
  return kTraceHead + kTracePerPass * pass + stage;
}
// One %globaltimer stamp (ns) into trace[slot] on s; nothing if trace is
// null.
cudaError_t stamp(int64_t* trace, int slot, cudaStream_t s);

// permute (cap, or uncapped when cap < 0) -> GEMM1 -> GEMM2 -> combine;
// with planned = true, over the virtual groups of the plan in b.
// pass_index: the trace slots of the pass (b.trace).
cudaError_t pass(const moe_config_t& c, const void* x, const int32_t* topk_idx,
                 const float* topk_w, int64_t cap, const void* wg,
                 const void* wu, const void* wd, void* y, const LayerBufs& b,
                 int32_t* status, cudaStream_t s, bool planned = false,
                 int pass_index = 0);
// The capped pass over tables already computed (moe_permute_tables with cap
// into row_of and table set `tb`): row scatter, GEMM1, GEMM2, combine.
cudaError_t capped_pass_tabled(const moe_config_t& c, const void* x,
                               const float* topk_w, const void* wg,
                               const void* wu, const void* wd, void* y,
                               const LayerBufs& b, const int32_t* row_of,
                               const PassTables& tb, int32_t* status,
                               cudaStream_t s);
// the chunked dropless fallback over routing already in topk_idx/topk_w.
// With pp (b carved for all T tokens), the permute tables of chunk i+1 run
// on pp->side during chunk i's expert FFN, in two table sets.
cudaError_t chunked_passes(const moe_config_t& c, const void* x,
                           const int32_t* topk_idx, const float* topk_w,
                           const void* wg, const void* wu, const void* wd,
                           void* y, const LayerBufs& b, int32_t* status,
                           cudaStream_t s, int32_t* n_run,
                           const PassPipeline* pp = nullptr);
moe_status_t validate(const moe_config_t* c);
bool ok_ptr(const void* p, bool need16);
bool gmm_shape_ok(const moe_config_t& c);
bool weights_ok(const void* wg, const void* wu, const void* wd);

// ---------------------------------------------------------- backward ---
// Rows of one weight-gradient segment: groups at group_offsets (relative),
// shifted by first_row inside the activation buffers.
using WgradSegment = moe_row_segment_t;
constexpr int kWgradGateUp = 1;  // dWg and dWu
constexpr int kWgradDown = 2;    // dWd
// flags of launch_wgrad (the values of MOE_WGRAD_ACCUMULATE and
// MOE_WGRAD_ROWS16)
constexpr int kWgradAccumulate = 1;  // add into dW instead of overwriting
constexpr int kWgradRows16 = 2;      // groups hold multiples of 16 rows
cudaError_t launch_combine_backward(const moe_config_t& c, const void* dy,
                                    const void* y_sorted,
                                    const int32_t* row_of,
                                    const float* topk_w, void* dy_sorted,
                                    float* dtopk_w, cudaStream_t s);
// The layer backward's split form of the combine backward (bf16): unscaled
// dy rows and per-row weights now, the weights' gradient from the
// down-projection dgrad's per-tile row dots afterwards.
cudaError_t launch_gather_dy_rows(const moe_config_t& c, const void* dy,
                                  const int32_t* row_of, const float* topk_w,
                                  void* dy_rows, float* w_row,
                                  cudaStream_t s);
cudaError_t launch_dtopk_from_row_dots(const moe_config_t& c,
                                       const int32_t* row_of,
                                       const float* row_dot, int n_parts,
                                       float* dtopk_w, cudaStream_t s);
cudaError_t launch_route_backward(const moe_config_t& c, const float* logits,
                                  const int32_t* topk_idx,
                                  const float* dtopk_w, float* dlogits,
                                  cudaStream_t s);
// fp32 (CUDA cores)
cudaError_t launch_gmm_saved_f32(const moe_config_t& c, const Groups& g,
                                 const void* xs, const int32_t* off,
                                 const void* wg, const void* wu, void* gbuf,
                                 void* ubuf, void* h, cudaStream_t s);
cudaError_t launch_down_dgrad_f32(const moe_config_t& c, const Groups& g,
                                  const int32_t* off, const void* wd,
                                  const void* gbuf, const void* ubuf,
                                  const void* dys, void* dg, void* du,
                                  cudaStream_t s);
cudaError_t launch_gate_up_dgrad_f32(const moe_config_t& c, const Groups& g,
                                     const int32_t* off, const void* wg,
                                     const void* wu, const void* dg,
                                     const void* du, void* dxs,
                                     cudaStream_t s);
cudaError_t launch_wgrad_f32(const moe_config_t& c, const Groups& g,
                             const WgradSegment* seg, int n_seg,
                             const void* xs, const void* dg, const void* du,
                             const void* h, const void* dys, float* dwg,
                             float* dwu, float* dwd, int flags,
                             int parts, cudaStream_t s);
// bf16 (tensor cores)
cudaError_t launch_gate_up_saved_bf16(const moe_config_t& c, const Groups& g,
                                      const void* x_sorted,
                                      const int32_t* group_offsets,
                                      const void* w_gate, const void* w_up,
                                      void* gbuf, void* ubuf, void* h,
                                      int32_t* status, cudaStream_t s);
// With w_row: dy_sorted holds unscaled rows; the epilogue scales dh by
// w_row[r], and writes row_dot[r * (F / bn) + q] = dh_u . h over the
// column tile q (bn = 256 if F % 256 == 0, else 128), h [rows, F] bf16.
cudaError_t launch_down_dgrad_bf16(const moe_config_t& c, const Groups& g,
                                   const int32_t* group_offsets,
                                   const void* w_down, const void* gbuf,
                                   const void* ubuf, const void* dy_sorted,
                                   void* dg, void* du, int32_t* status,
                                   cudaStream_t s,
                                   const float* w_row = nullptr,
                                   const void* h = nullptr,
                                   float* row_dot = nullptr);
inline int down_dgrad_col_tiles(const moe_config_t& c) {
  return c.F % 256 == 0 ? c.F / 256 : c.F / 128;
}
cudaError_t launch_gate_up_dgrad_bf16(const moe_config_t& c, const Groups& g,
                                      const int32_t* group_offsets,
                                      const void* w_gate, const void* w_up,
                                      const void* dg, const void* du,
                                      void* dx_sorted, int32_t* status,
                                      cudaStream_t s);
cudaError_t launch_wgrad_bf16(const moe_config_t& c, const Groups& g,
                              const WgradSegment* seg, int n_seg,
                              int64_t rows_total, const void* x_sorted,
                              const void* dg, const void* du, const void* h,
                              const void* dy_sorted, float* dw_gate,
                              float* dw_up, float* dw_down, int flags,
                              int parts, int32_t* status, cudaStream_t s);
// Dispatch on the layer dtype (bf16: tensor cores, fp32: CUDA cores).
cudaError_t launch_gate_up_saved(const moe_config_t& c, const Groups& g,
                                 const void* xs, const int32_t* off,
                                 const void* wg, const void* wu, void* gbuf,
                                 void* ubuf, void* h, int32_t* status,
                                 cudaStream_t s);
cudaError_t launch_down_dgrad(const moe_config_t& c, const Groups& g,
                              const int32_t* off, const void* wd,
                              const void* gbuf, const void* ubuf,
                              const void* dys, void* dg, void* du,
                              int32_t* status, cudaStream_t s);
cudaError_t launch_gate_up_dgrad(const moe_config_t& c, const Groups& g,
                                 const int32_t* off, const void* wg,
                                 const void* wu, const void* dg,
                                 const void* du, void* dxs, int32_t* status,
                                 cudaStream_t s);
// flags: kWgradAccumulate | kWgradRows16 (see wgrad_tc.cu)
cudaError_t launch_wgrad(const moe_config_t& c, const Groups& g,
                         const WgradSegment* seg, int n_seg,
                         int64_t rows_total, const void* xs, const void* dg,
                         const void* du, const void* h, const void* dys,
                         float* dwg, float* dwu, float* dwd, int flags,
                         int parts, int32_t* status, cudaStream_t s);
// Rows of up to kMaxRegroupSegments ranges copied into one expert-major
// layout with 16-row-aligned groups and zero pad rows (see regroup.cu);
// destination buffers of regroup_rows(c) rows.
constexpr int kMaxRegroupSegments = 64;
inline int64_t regroup_rows(const moe_config_t& c) {
  return static_cast<int64_t>(c.T) * c.k +
         16 * static_cast<int64_t>(num_groups(c));
}
// w_row (optional): dys holds unscaled rows; dys2 gets them times w_row
// of their source row, rounded to bf16.
cudaError_t launch_regroup(const moe_config_t& c, int G,
                           const WgradSegment* seg,
                           int n_seg, int64_t rows_out, const void* xs,
                           const void* dg, const void* du, const void* h,
                           const void* dys, void* xs2, void* dg2, void* du2,
                           void* h2, void* dys2, int32_t* out_off,
                           cudaStream_t s, const float* w_row = nullptr);
size_t gmm_backward_bytes(const moe_config_t& c);
size_t layer_backward_bytes(const moe_config_t& c);

// Tests of the GEMM's bounded waits: stop the TMA producer after `fills`
// stage fills (-1: normal operation).
void set_gemm_stall_for_tests(long long fills);

// Shape support of the bf16 tensor-core GEMM.
bool gmm_tc_supported(const moe_config_t& c);

// Router logits [T, E] float32 = x Wr (+ offset): the tensor-core form
// (bf16, H % 64 == 0, E % 128 == 0) and the CUDA-core form (any shape).
bool router_tc_supported(const moe_config_t& c);
cudaError_t launch_router_bf16(const moe_config_t& c, const void* x,
                               const void* w_router, const float* offset,
                               float* logits, int32_t* status,
                               cudaStream_t s);
// The router's tensor-core launch (router_tc.cu): the one-group GEMM
// above, or for batches whose tiles leave SMs idle the reduction split over
// clusters of 2, 4 or 8 CTAs, whichever takes fewer k-block steps per SM.
cudaError_t launch_router_tc(const moe_config_t& c, const void* x,
                             const void* w_router, const float* offset,
                             float* logits, int32_t* status, cudaStream_t s);

// Host-side formulas shared by validation and drivers.
int64_t capacity_rows(const moe_config_t& c);
int32_t chunk_tokens(const moe_config_t& c);

}  // namespace moe
