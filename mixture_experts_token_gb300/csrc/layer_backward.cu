// C ABI entry points of the backward pass and the layer-level driver.
//
// "Support moe_dropless_fallback=layer on the ragged all-to-all MoE path"
// (MaxText pull request 5920): section Tests asks that with the layer
// fallback both the outputs and the gradients match the dropless model;
// section How says the fallback's backward recomputes each chunk's forward
// (the chunk loop is rematerialised) and accumulates the expert-weight
// gradients across chunks.
//
// moe_layer_backward follows that plan pass by pass: route once, then for
// each pass (one capped or uncapped pass, or the fallback's chunks)
// permute -> forward GEMMs keeping g, u, h -> combine backward -> data
// gradients -> permute backward.  The weight gradients of all passes are
// summed in one launch at the end: each pass leaves its rows in a disjoint
// row range of the activation buffers, and one tile of the weight-gradient
// kernel accumulates an expert's rows from every range in tensor memory, so
// dW is written once instead of read and rewritten per chunk.  Before that
// launch (bf16, up to 64 passes) the passes' rows are regrouped into one
// 16-row-aligned range per expert (regroup.cu).
#include <algorithm>
#include <limits>
#include <vector>

#include "internal.h"

namespace moe {

namespace {

struct BwdBufs {
  LayerBufs f;           // routing, permute and forward buffers for T
  void *g, *u, *dg, *du;  // [T*k, F]
  void *dys, *dxs;        // [T*k, H]
  float* dtw;             // [T, k]
  // bf16 with regrouped weight gradients: dys holds unscaled dy rows, wrow
  // their combine weights, rdot the down dgrad's per-column-tile row dots
  float* wrow;            // [T*k]
  float* rdot;            // [T*k, F / 128]
  int32_t* seg_off;       // [n_seg, G + 1] group offsets of every pass
  // the passes' rows regrouped for the weight gradients (regroup.cu)
  void *xs2, *dg2, *du2, *h2, *dys2;  // [T*k + 16*E, H or F]
  int32_t* off2;                      // [G + 1]
};

int max_passes(const moe_config_t& c, moe_mode_t mode) {
  if (mode != MOE_MODE_FALLBACK_LAYER || c.T == 0) return 1;
  const int ct = chunk_tokens(c);
  return std::max(1, (c.T + ct - 1) / ct);
}

BwdBufs carve_bwd(void* base, const moe_config_t& c, int n_seg,
                  size_t* bytes) {
  BwdBufs b;
  size_t fb = 0;
  b.f = carve_layer(base, c, c.T, &fb);
  Carve cv(base ? static_cast<char*>(base) + fb : nullptr);
  const size_t rows = static_cast<size_t>(c.T) * c.k;
  const size_t eb = elem_bytes(c.dtype);
  b.g = cv.take<char>(rows * c.F * eb);
  b.u = cv.take<char>(rows * c.F * eb);
  b.dg = cv.take<char>(rows * c.F * eb);
  b.du = cv.take<char>(rows * c.F * eb);
  b.dys = cv.take<char>(rows * c.H * eb);
  b.dxs = cv.take<char>(rows * c.H * eb);
  b.dtw = cv.take<float>(rows);
  b.wrow = cv.take<float>(rows);
  b.rdot = cv.take<float>(rows * static_cast<size_t>(c.F / 128));
  b.seg_off =
      cv.take<int32_t>(static_cast<size_t>(n_seg) * (num_groups(c) + 1));
  const size_t rr = static_cast<size_t>(regroup_rows(c));
  b.xs2 = cv.take<char>(rr * c.H * eb);
  b.dys2 = cv.take<char>(rr * c.H * eb);
  b.dg2 = cv.take<char>(rr * c.F * eb);
  b.du2 = cv.take<char>(rr * c.F * eb);
  b.h2 = cv.take<char>(rr * c.F * eb);
  b.off2 = cv.take<int32_t>(num_groups(c) + 1);
  if (bytes) *bytes = fb + align_up(cv.off, 256);
  return b;
}

void* rows_at(const void* p, size_t row, size_t row_bytes) {
  return const_cast<char*>(static_cast<const char*>(p)) + row * row_bytes;
}

// Backward of one pass over tokens [t0, t0 + tc) with capacity cap (-1:
// uncapped), all but the weight gradients.  Its rows occupy
// [t0*k, (t0+tc)*k) of the row buffers and its group offsets row `seg` of
// the segment table.  planned: over the virtual groups of the duplication
// plan in b (each computing with its expert's weights).
// unscaled (bf16, regrouped weight gradients): the combine weights' gradient
// comes from the down dgrad -- dy[t] . (h Wd) = (dy[t] Wd^T) . h -- so the
// pass does not recompute y_sorted = h Wd; dys keeps the unscaled dy rows
// and the regroup applies the weights for dWd.
cudaError_t bwd_pass(const moe_config_t& c, int t0, int tc, int64_t cap,
                     bool planned, int seg, const void* x, const void* wg,
                     const void* wu, const void* wd, const void* dy, void* dx,
                     const BwdBufs& b, bool unscaled, int32_t* status,
                     cudaStream_t s) {
  moe_config_t sc = c;
  sc.T = tc;
  const size_t eb = elem_bytes(c.dtype);
  const size_t hb = c.H * eb, fb = c.F * eb;
  const size_t base = static_cast<size_t>(t0) * c.k;
  PermutePlan plan;
  Groups ids = identity_groups(sc);
  if (planned) {
    plan.divert = b.f.divert;
    plan.slot_of = b.f.slot_of;
    plan.B = c.redundant_slots;
    ids = {num_groups(c), b.f.group_expert};
  }
  const void* xc = rows_at(x, t0, hb);
  const int32_t* idx = b.f.topk_idx + base;
  const float* w = b.f.topk_w + base;
  int32_t* row_of = b.f.row_of + base;
  int32_t* goff = b.seg_off + static_cast<size_t>(seg) * (num_groups(c) + 1);
  void* xs = rows_at(b.f.x_sorted, base, hb);
  void* h = rows_at(b.f.h, base, fb);
  void* ys = rows_at(b.f.y_sorted, base, hb);
  void* gg = rows_at(b.g, base, fb);
  void* uu = rows_at(b.u, base, fb);
  void* dg = rows_at(b.dg, base, fb);
  void* du = rows_at(b.du, base, fb);
  void* dys = rows_at(b.dys, base, hb);
  void* dxs = rows_at(b.dxs, base, hb);
  cudaError_t e = launch_permute(
      sc, xc, idx, cap, xs, row_of, b.f.sorted_token + base, goff,
      b.f.uniq_offsets, b.f.uniq_tokens, b.f.expand_idx + base, b.f.n_dropped,
      b.f.pws, status, s, plan);
  if (e != cudaSuccess) return e;
  if (unscaled) {
    const int nt = down_dgrad_col_tiles(c);
    float* rd = b.rdot + base * nt;
    if ((e = launch_gate_up_saved(sc, ids, xs, goff, wg, wu, gg, uu, h,
                                  status, s)) != cudaSuccess ||
        (e = launch_gather_dy_rows(sc, rows_at(dy, t0, hb), row_of, w, dys,
                                   b.wrow + base, s)) != cudaSuccess ||
        (e = launch_down_dgrad_bf16(sc, ids, goff, wd, gg, uu, dys, dg, du,
                                    status, s, b.wrow + base, h, rd)) !=
            cudaSuccess ||
        (e = launch_dtopk_from_row_dots(sc, row_of, rd, nt, b.dtw + base,
                                        s)) != cudaSuccess ||
        (e = launch_gate_up_dgrad(sc, ids, goff, wg, wu, dg, du, dxs, status,
                                  s)) != cudaSuccess)
      return e;
    return launch_combine(sc, dxs, row_of, nullptr, rows_at(dx, t0, hb), s);
  }
  if ((e = launch_gate_up_saved(sc, ids, xs, goff, wg, wu, gg, uu, h, status,
                                s)) != cudaSuccess ||
      (e = launch_gmm2(sc, ids, h, goff, wd, ys, status, s)) != cudaSuccess ||
      (e = launch_combine_backward(sc, rows_at(dy, t0, hb), ys, row_of, w,
                                   dys, b.dtw + base, s)) != cudaSuccess ||
      (e = launch_down_dgrad(sc, ids, goff, wd, gg, uu, dys, dg, du, status,
                             s)) != cudaSuccess ||
      (e = launch_gate_up_dgrad(sc, ids, goff, wg, wu, dg, du, dxs, status,
                                s)) != cudaSuccess)
    return e;
  return launch_combine(sc, dxs, row_of, nullptr, rows_at(dx, t0, hb), s);
}

}  // namespace

cudaError_t launch_gate_up_saved(const moe_config_t& c, const Groups& g,
                                 const void* xs, const int32_t* off,
                                 const void* wg, const void* wu, void* gbuf,
                                 void* ubuf, void* h, int32_t* status,
                                 cudaStream_t s) {
  if (c.dtype == MOE_BF16)
    return launch_gate_up_saved_bf16(c, g, xs, off, wg, wu, gbuf, ubuf, h,
                                     status, s);
  return launch_gmm_saved_f32(c, g, xs, off, wg, wu, gbuf, ubuf, h, s);
}

cudaError_t launch_down_dgrad(const moe_config_t& c, const Groups& g,
                              const int32_t* off, const void* wd,
                              const void* gbuf, const void* ubuf,
                              const void* dys, void* dg, void* du,
                              int32_t* status, cudaStream_t s) {
  if (c.dtype == MOE_BF16)
    return launch_down_dgrad_bf16(c, g, off, wd, gbuf, ubuf, dys, dg, du,
                                  status, s);
  return launch_down_dgrad_f32(c, g, off, wd, gbuf, ubuf, dys, dg, du, s);
}

cudaError_t launch_gate_up_dgrad(const moe_config_t& c, const Groups& g,
                                 const int32_t* off, const void* wg,
                                 const void* wu, const void* dg,
                                 const void* du, void* dxs, int32_t* status,
                                 cudaStream_t s) {
  if (c.dtype == MOE_BF16)
    return launch_gate_up_dgrad_bf16(c, g, off, wg, wu, dg, du, dxs, status,
                                     s);
  return launch_gate_up_dgrad_f32(c, g, off, wg, wu, dg, du, dxs, s);
}

cudaError_t launch_wgrad(const moe_config_t& c, const Groups& g,
                         const WgradSegment* seg, int n_seg,
                         int64_t rows_total, const void* xs, const void* dg,
                         const void* du, const void* h, const void* dys,
                         float* dwg, float* dwu, float* dwd, int flags,
                         int parts, int32_t* status, cudaStream_t s) {
  if (c.dtype == MOE_BF16)
    return launch_wgrad_bf16(c, g, seg, n_seg, rows_total, xs, dg, du, h, dys,
                             dwg, dwu, dwd, flags, parts, status, s);
  return launch_wgrad_f32(c, g, seg, n_seg, xs, dg, du, h, dys, dwg, dwu, dwd,
                          flags, parts, s);
}

size_t gmm_backward_bytes(const moe_config_t& c) {
  Carve cv(nullptr);
  const size_t rows = static_cast<size_t>(c.T) * c.k;
  cv.take<char>(rows * c.F * elem_bytes(c.dtype));
  cv.take<char>(rows * c.F * elem_bytes(c.dtype));
  return align_up(cv.off, 256);
}

size_t layer_backward_bytes(const moe_config_t& c) {
  size_t n = 0;
  carve_bwd(nullptr, c, max_passes(c, MOE_MODE_FALLBACK_LAYER), &n);
  return n;
}

}  // namespace moe

using namespace moe;

namespace {
moe_status_t cuda_st(cudaError_t e) {
  if (e == cudaSuccess) return MOE_OK;
  cudaGetLastError();
  return MOE_ERR_CUDA;
}
}  // namespace

extern "C" {

moe_status_t moe_combine_backward(const moe_config_t* cfg, const void* dy,
                                  const void* y_sorted, const int32_t* row_of,
                                  const float* topk_w, void* dy_sorted,
                                  float* dtopk_w, moe_stream_t stream) {
  moe_status_t st = validate(cfg);
  if (st != MOE_OK) return st;
  if (cfg->T == 0) return MOE_OK;
  if (!ok_ptr(dy, true) || !ok_ptr(y_sorted, true) || !ok_ptr(row_of, false) ||
      !ok_ptr(topk_w, false) || !ok_ptr(dy_sorted, true) ||
      !ok_ptr(dtopk_w, false))
    return MOE_ERR_INVALID_ARG;
  return cuda_st(launch_combine_backward(*cfg, dy, y_sorted, row_of, topk_w,
                                         dy_sorted, dtopk_w, stream));
}

moe_status_t moe_route_backward(const moe_config_t* cfg, const float* logits,
                                const int32_t* topk_idx, const float* dtopk_w,
                                float* dlogits, moe_stream_t stream) {
  moe_status_t st = validate(cfg);
  if (st != MOE_OK) return st;
  if (cfg->T == 0) return MOE_OK;
  if (!ok_ptr(logits, false) || !ok_ptr(topk_idx, false) ||
      !ok_ptr(dtopk_w, false) || !ok_ptr(dlogits, false))
    return MOE_ERR_INVALID_ARG;
  return cuda_st(launch_route_backward(*cfg, logits, topk_idx, dtopk_w,
                                       dlogits, stream));
}

moe_status_t moe_permute_backward(const moe_config_t* cfg,
                                  const void* dx_sorted,
                                  const int32_t* row_of, void* dx,
                                  moe_stream_t stream) {
  moe_status_t st = validate(cfg);
  if (st != MOE_OK) return st;
  if (cfg->T == 0) return MOE_OK;
  if (!ok_ptr(dx_sorted, true) || !ok_ptr(row_of, false) || !ok_ptr(dx, true))
    return MOE_ERR_INVALID_ARG;
  return cuda_st(launch_combine(*cfg, dx_sorted, row_of, nullptr, dx, stream));
}

moe_status_t moe_gmm_swiglu_saved(const moe_config_t* cfg,
                                  const void* x_sorted,
                                  const int32_t* group_offsets,
                                  const void* w_gate, const void* w_up,
                                  const void* w_down, void* g, void* u,
                                  void* h, void* y_sorted,
                                  int32_t* status_word, moe_stream_t stream) {
  moe_status_t st = validate(cfg);
  if (st != MOE_OK) return st;
  if (cfg->F < 1) return MOE_ERR_INVALID_ARG;
  if (!gmm_shape_ok(*cfg)) return MOE_ERR_UNSUPPORTED;
  if (cfg->T == 0) return MOE_OK;
  if (!ok_ptr(x_sorted, true) || !ok_ptr(group_offsets, false) ||
      !weights_ok(w_gate, w_up, w_down) || !ok_ptr(g, true) ||
      !ok_ptr(u, true) || !ok_ptr(h, true) || !ok_ptr(y_sorted, true))
    return MOE_ERR_INVALID_ARG;
  const Groups ids = identity_groups(*cfg);
  cudaError_t e = launch_gate_up_saved(*cfg, ids, x_sorted, group_offsets,
                                       w_gate, w_up, g, u, h, status_word,
                                       stream);
  if (e == cudaSuccess)
    e = launch_gmm2(*cfg, ids, h, group_offsets, w_down, y_sorted,
                    status_word, stream);
  return cuda_st(e);
}

moe_status_t moe_gmm_swiglu_backward(
    const moe_config_t* cfg, const void* x_sorted,
    const int32_t* group_offsets, const void* w_gate, const void* w_up,
    const void* w_down, const void* g, const void* u, const void* h,
    const void* dy_sorted, void* dx_sorted, float* dw_gate, float* dw_up,
    float* dw_down, int32_t accumulate, int32_t* status_word, void* workspace,
    size_t workspace_bytes, moe_stream_t stream) {
  moe_status_t st = validate(cfg);
  if (st != MOE_OK) return st;
  if (cfg->F < 1 || (accumulate != 0 && accumulate != 1))
    return MOE_ERR_INVALID_ARG;
  if (!gmm_shape_ok(*cfg)) return MOE_ERR_UNSUPPORTED;
  if (!ok_ptr(group_offsets, false) || !ok_ptr(dw_gate, true) ||
      !ok_ptr(dw_up, true) || !ok_ptr(dw_down, true))
    return MOE_ERR_INVALID_ARG;
  if (cfg->T > 0 &&
      (!ok_ptr(x_sorted, true) || !weights_ok(w_gate, w_up, w_down) ||
       !ok_ptr(g, true) || !ok_ptr(u, true) || !ok_ptr(h, true) ||
       !ok_ptr(dy_sorted, true) || !ok_ptr(dx_sorted, true)))
    return MOE_ERR_INVALID_ARG;
  if (workspace == nullptr || !ok_ptr(workspace, true) ||
      workspace_bytes < gmm_backward_bytes(*cfg))
    return MOE_ERR_WORKSPACE;
  Carve cv(workspace);
  const size_t rows = static_cast<size_t>(cfg->T) * cfg->k;
  void* dg = cv.take<char>(rows * cfg->F * elem_bytes(cfg->dtype));
  void* du = cv.take<char>(rows * cfg->F * elem_bytes(cfg->dtype));
  const Groups ids = identity_groups(*cfg);
  cudaError_t e = launch_down_dgrad(*cfg, ids, group_offsets, w_down, g, u,
                                    dy_sorted, dg, du, status_word, stream);
  if (e == cudaSuccess)
    e = launch_gate_up_dgrad(*cfg, ids, group_offsets, w_gate, w_up, dg, du,
                             dx_sorted, status_word, stream);
  if (e != cudaSuccess) return cuda_st(e);
  const WgradSegment seg{group_offsets, 0};
  return cuda_st(launch_wgrad(*cfg, ids, &seg, cfg->T > 0 ? 1 : 0,
                              static_cast<int64_t>(rows), x_sorted, dg, du, h,
                              dy_sorted, dw_gate, dw_up, dw_down,
                              accumulate != 0 ? kWgradAccumulate : 0,
                              kWgradGateUp | kWgradDown, status_word,
                              stream));
}

namespace {
// n_groups = 0 with a null map: the experts' own groups.
bool bwd_groups(const moe_config_t& c, int32_t n, const int32_t* map,
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

moe_status_t moe_gmm_gate_up_saved(const moe_config_t* cfg, int32_t n_groups,
                                   const int32_t* group_expert,
                                   const void* x_sorted,
                                   const int32_t* group_offsets,
                                   const void* w_gate, const void* w_up,
                                   void* g, void* u, void* h,
                                   int32_t* status_word, moe_stream_t stream) {
  moe_status_t st = validate(cfg);
  if (st != MOE_OK) return st;
  if (cfg->F < 1) return MOE_ERR_INVALID_ARG;
  if (!gmm_shape_ok(*cfg)) return MOE_ERR_UNSUPPORTED;
  if (cfg->T == 0) return MOE_OK;
  Groups grp;
  if (!bwd_groups(*cfg, n_groups, group_expert, &grp) ||
      !ok_ptr(x_sorted, true) || !ok_ptr(group_offsets, false) ||
      !ok_ptr(w_gate, true) || !ok_ptr(w_up, true) || !ok_ptr(g, true) ||
      !ok_ptr(u, true) || !ok_ptr(h, true))
    return MOE_ERR_INVALID_ARG;
  return cuda_st(launch_gate_up_saved(*cfg, grp, x_sorted,
                                      group_offsets, w_gate, w_up, g, u, h,
                                      status_word, stream));
}

moe_status_t moe_gmm_down_dgrad(const moe_config_t* cfg, int32_t n_groups,
                                const int32_t* group_expert,
                                const int32_t* group_offsets,
                                const void* w_down, const void* g,
                                const void* u, const void* dy_sorted,
                                void* dg, void* du, int32_t* status_word,
                                moe_stream_t stream) {
  moe_status_t st = validate(cfg);
  if (st != MOE_OK) return st;
  if (cfg->F < 1) return MOE_ERR_INVALID_ARG;
  if (!gmm_shape_ok(*cfg)) return MOE_ERR_UNSUPPORTED;
  if (cfg->T == 0) return MOE_OK;
  Groups grp;
  if (!bwd_groups(*cfg, n_groups, group_expert, &grp) ||
      !ok_ptr(group_offsets, false) || !ok_ptr(w_down, true) ||
      !ok_ptr(g, true) || !ok_ptr(u, true) || !ok_ptr(dy_sorted, true) ||
      !ok_ptr(dg, true) || !ok_ptr(du, true))
    return MOE_ERR_INVALID_ARG;
  return cuda_st(launch_down_dgrad(*cfg, grp, group_offsets,
                                   w_down, g, u, dy_sorted, dg, du,
                                   status_word, stream));
}

moe_status_t moe_gmm_gate_up_dgrad(const moe_config_t* cfg, int32_t n_groups,
                                   const int32_t* group_expert,
                                   const int32_t* group_offsets,
                                   const void* w_gate, const void* w_up,
                                   const void* dg, const void* du,
                                   void* dx_sorted, int32_t* status_word,
                                   moe_stream_t stream) {
  moe_status_t st = validate(cfg);
  if (st != MOE_OK) return st;
  if (cfg->F < 1) return MOE_ERR_INVALID_ARG;
  if (!gmm_shape_ok(*cfg)) return MOE_ERR_UNSUPPORTED;
  if (cfg->T == 0) return MOE_OK;
  Groups grp;
  if (!bwd_groups(*cfg, n_groups, group_expert, &grp) ||
      !ok_ptr(group_offsets, false) || !ok_ptr(w_gate, true) ||
      !ok_ptr(w_up, true) || !ok_ptr(dg, true) || !ok_ptr(du, true) ||
      !ok_ptr(dx_sorted, true))
    return MOE_ERR_INVALID_ARG;
  return cuda_st(launch_gate_up_dgrad(*cfg, grp,
                                      group_offsets, w_gate, w_up, dg, du,
                                      dx_sorted, status_word, stream));
}

namespace {
moe_status_t check_segments(const moe_config_t* cfg,
                            const moe_row_segment_t* segments,
                            int32_t n_segments, int64_t rows_total,
                            int32_t accumulate) {
  moe_status_t st = validate(cfg);
  if (st != MOE_OK) return st;
  if (cfg->F < 1 || n_segments < 0 || rows_total < 0 ||
      rows_total > std::numeric_limits<int32_t>::max() ||
      (accumulate & ~(kWgradAccumulate | kWgradRows16)) != 0 ||
      (n_segments > 0 && segments == nullptr))
    return MOE_ERR_INVALID_ARG;
  if (!gmm_shape_ok(*cfg)) return MOE_ERR_UNSUPPORTED;
  for (int32_t i = 0; i < n_segments; ++i)
    if (!ok_ptr(segments[i].group_offsets, false) ||
        segments[i].first_row < 0 || segments[i].first_row > rows_total)
      return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}
}  // namespace

moe_status_t moe_gmm_gate_up_wgrad(const moe_config_t* cfg, int32_t n_groups,
                                   const int32_t* group_expert,
                                   const moe_row_segment_t* segments,
                                   int32_t n_segments, int64_t rows_total,
                                   const void* x_sorted, const void* dg,
                                   const void* du, float* dw_gate,
                                   float* dw_up, int32_t accumulate,
                                   int32_t* status_word, moe_stream_t stream) {
  moe_status_t st =
      check_segments(cfg, segments, n_segments, rows_total, accumulate);
  if (st != MOE_OK) return st;
  Groups grp;
  if (!bwd_groups(*cfg, n_groups, group_expert, &grp) ||
      !ok_ptr(dw_gate, true) || !ok_ptr(dw_up, true) ||
      (n_segments > 0 &&
       (!ok_ptr(x_sorted, true) || !ok_ptr(dg, true) || !ok_ptr(du, true))))
    return MOE_ERR_INVALID_ARG;
  return cuda_st(launch_wgrad(*cfg, grp, segments,
                              n_segments, rows_total, x_sorted, dg, du,
                              nullptr, nullptr, dw_gate, dw_up, nullptr,
                              accumulate, kWgradGateUp, status_word, stream));
}

moe_status_t moe_gmm_down_wgrad(const moe_config_t* cfg, int32_t n_groups,
                                const int32_t* group_expert,
                                const moe_row_segment_t* segments,
                                int32_t n_segments, int64_t rows_total,
                                const void* h, const void* dy_sorted,
                                float* dw_down, int32_t accumulate,
                                int32_t* status_word, moe_stream_t stream) {
  moe_status_t st =
      check_segments(cfg, segments, n_segments, rows_total, accumulate);
  if (st != MOE_OK) return st;
  Groups grp;
  if (!bwd_groups(*cfg, n_groups, group_expert, &grp) ||
      !ok_ptr(dw_down, true) ||
      (n_segments > 0 && (!ok_ptr(h, true) || !ok_ptr(dy_sorted, true))))
    return MOE_ERR_INVALID_ARG;
  return cuda_st(launch_wgrad(*cfg, grp, segments,
                              n_segments, rows_total, nullptr, nullptr,
                              nullptr, h, dy_sorted, nullptr, nullptr,
                              dw_down, accumulate, kWgradDown, status_word,
                              stream));
}

moe_status_t moe_regroup_rows(const moe_config_t* cfg, int32_t n_groups,
                              const moe_row_segment_t* segments,
                              int32_t n_segments, int64_t rows_out,
                              const void* x_sorted, const void* dg,
                              const void* du, const void* h,
                              const void* dy_sorted, void* x_out,
                              void* dg_out, void* du_out, void* h_out,
                              void* dy_out, int32_t* out_offsets,
                              const float* w_row, moe_stream_t stream) {
  moe_status_t st = validate(cfg);
  if (st != MOE_OK) return st;
  const int G = n_groups == 0 ? cfg->E : n_groups;
  if (cfg->F < 1 || n_segments < 1 || n_segments > kMaxRegroupSegments ||
      n_groups < 0 || G > num_groups(*cfg) || segments == nullptr ||
      rows_out < regroup_rows(*cfg) ||
      rows_out > std::numeric_limits<int32_t>::max())
    return MOE_ERR_INVALID_ARG;
  for (int32_t i = 0; i < n_segments; ++i)
    if (!ok_ptr(segments[i].group_offsets, false) ||
        segments[i].first_row < 0)
      return MOE_ERR_INVALID_ARG;
  if (!ok_ptr(x_sorted, true) || !ok_ptr(dg, true) || !ok_ptr(du, true) ||
      !ok_ptr(h, true) || !ok_ptr(dy_sorted, true) || !ok_ptr(x_out, true) ||
      !ok_ptr(dg_out, true) || !ok_ptr(du_out, true) || !ok_ptr(h_out, true) ||
      !ok_ptr(dy_out, true) || !ok_ptr(out_offsets, false) ||
      (w_row != nullptr && !ok_ptr(w_row, false)))
    return MOE_ERR_INVALID_ARG;
  if (w_row != nullptr && cfg->dtype != MOE_BF16) return MOE_ERR_UNSUPPORTED;
  return cuda_st(launch_regroup(*cfg, G, segments, n_segments, rows_out,
                                x_sorted, dg, du, h, dy_sorted, x_out, dg_out,
                                du_out, h_out, dy_out, out_offsets, stream,
                                w_row));
}

int32_t moe_row_dot_parts(const moe_config_t* cfg) {
  if (cfg == nullptr || validate(cfg) != MOE_OK || cfg->F < 1) return -1;
  return down_dgrad_col_tiles(*cfg);
}

moe_status_t moe_combine_backward_rows(const moe_config_t* cfg,
                                       const void* dy, const int32_t* row_of,
                                       const float* topk_w, void* dy_rows,
                                       float* w_row, moe_stream_t stream) {
  moe_status_t st = validate(cfg);
  if (st != MOE_OK) return st;
  if (cfg->T == 0) return MOE_OK;
  if (!ok_ptr(dy, true) || !ok_ptr(row_of, false) ||
      !ok_ptr(topk_w, false) || !ok_ptr(dy_rows, true) ||
      !ok_ptr(w_row, false))
    return MOE_ERR_INVALID_ARG;
  return cuda_st(launch_gather_dy_rows(*cfg, dy, row_of, topk_w, dy_rows,
                                       w_row, stream));
}

moe_status_t moe_gmm_down_dgrad_rows(const moe_config_t* cfg,
                                     int32_t n_groups,
                                     const int32_t* group_expert,
                                     const int32_t* group_offsets,
                                     const void* w_down, const void* g,
                                     const void* u, const void* h,
                                     const void* dy_rows, const float* w_row,
                                     void* dg, void* du, float* row_dot,
                                     int32_t* status_word,
                                     moe_stream_t stream) {
  moe_status_t st = validate(cfg);
  if (st != MOE_OK) return st;
  if (cfg->F < 1) return MOE_ERR_INVALID_ARG;
  if (cfg->dtype != MOE_BF16 || !gmm_shape_ok(*cfg))
    return MOE_ERR_UNSUPPORTED;
  if (cfg->T == 0) return MOE_OK;
  Groups grp;
  if (!bwd_groups(*cfg, n_groups, group_expert, &grp) ||
      !ok_ptr(group_offsets, false) || !ok_ptr(w_down, true) ||
      !ok_ptr(g, true) || !ok_ptr(u, true) || !ok_ptr(h, true) ||
      !ok_ptr(dy_rows, true) || !ok_ptr(w_row, false) || !ok_ptr(dg, true) ||
      !ok_ptr(du, true) || !ok_ptr(row_dot, false))
    return MOE_ERR_INVALID_ARG;
  return cuda_st(launch_down_dgrad_bf16(*cfg, grp, group_offsets, w_down, g,
                                        u, dy_rows, dg, du, status_word,
                                        stream, w_row, h, row_dot));
}

moe_status_t moe_combine_weight_grad(const moe_config_t* cfg,
                                     const int32_t* row_of,
                                     const float* row_dot, float* dtopk_w,
                                     moe_stream_t stream) {
  moe_status_t st = validate(cfg);
  if (st != MOE_OK) return st;
  if (cfg->F < 1) return MOE_ERR_INVALID_ARG;
  if (cfg->T == 0) return MOE_OK;
  if (!ok_ptr(row_of, false) || !ok_ptr(row_dot, false) ||
      !ok_ptr(dtopk_w, false))
    return MOE_ERR_INVALID_ARG;
  return cuda_st(launch_dtopk_from_row_dots(*cfg, row_of, row_dot,
                                            down_dgrad_col_tiles(*cfg),
                                            dtopk_w, stream));
}

moe_status_t moe_layer_backward(const moe_config_t* cfg, const void* x,
                                const float* logits, const void* w_gate,
                                const void* w_up, const void* w_down,
                                const void* dy, void* dx, float* dlogits,
                                float* dw_gate, float* dw_up, float* dw_down,
                                moe_mode_t mode, moe_layer_info_t* info,
                                int32_t* status_word, void* workspace,
                                size_t workspace_bytes, moe_stream_t stream) {
  moe_status_t st = validate(cfg);
  if (st != MOE_OK) return st;
  if (mode != MOE_MODE_FALLBACK_LAYER && mode != MOE_MODE_CAPPED &&
      mode != MOE_MODE_DROPLESS)
    return MOE_ERR_INVALID_ARG;
  if (cfg->F < 1) return MOE_ERR_INVALID_ARG;
  if (!gmm_shape_ok(*cfg)) return MOE_ERR_UNSUPPORTED;
  if (!weights_ok(w_gate, w_up, w_down) || !ok_ptr(dw_gate, true) ||
      !ok_ptr(dw_up, true) || !ok_ptr(dw_down, true))
    return MOE_ERR_INVALID_ARG;
  if (cfg->T > 0 && (!ok_ptr(x, true) || !ok_ptr(logits, false) ||
                     !ok_ptr(dy, true) || !ok_ptr(dx, true) ||
                     !ok_ptr(dlogits, false)))
    return MOE_ERR_INVALID_ARG;
  if (workspace == nullptr || !ok_ptr(workspace, true) ||
      workspace_bytes < layer_backward_bytes(*cfg))
    return MOE_ERR_WORKSPACE;
  const int64_t cap = capacity_rows(*cfg);
  if (info) {
    info->overflow = -1;
    info->n_chunks = cfg->T > 0 ? 1 : 0;
    info->capacity = mode == MOE_MODE_DROPLESS ? -1 : cap;
  }
  const size_t wbytes =
      static_cast<size_t>(cfg->E) * cfg->H * cfg->F * sizeof(float);
  if (cfg->T == 0) {  // no rows: every weight gradient is zero
    cudaError_t e = cudaMemsetAsync(dw_gate, 0, wbytes, stream);
    if (e == cudaSuccess) e = cudaMemsetAsync(dw_up, 0, wbytes, stream);
    if (e == cudaSuccess) e = cudaMemsetAsync(dw_down, 0, wbytes, stream);
    return cuda_st(e);
  }
  const BwdBufs b = carve_bwd(workspace, *cfg,
                              max_passes(*cfg, MOE_MODE_FALLBACK_LAYER),
                              nullptr);
  cudaError_t e = launch_route(*cfg, logits, b.f.topk_idx, b.f.topk_w,
                               status_word, stream);
  if (e != cudaSuccess) return cuda_st(e);
  // the passes: (t0, tokens, capacity, over the plan's virtual groups)
  struct Pass {
    int t0, tc;
    int64_t cap;
    bool planned;
  };
  // duplicate-expert slots: as moe_layer, the plan is made after the check
  // and the capped pass runs over its virtual groups; the chunked fallback
  // runs plain
  const bool planned = cfg->redundant_slots > 0 && mode != MOE_MODE_DROPLESS;
  if (planned) {
    e = launch_check(*cfg, b.f.topk_idx, b.f.counts, b.f.offsets, b.f.shard,
                     b.f.flag, b.f.req, b.f.cap, stream);
    if (e == cudaSuccess)
      e = launch_plan(*cfg, b.f.counts, b.f.divert, b.f.slot_of,
                      b.f.group_expert, b.f.shard_after, b.f.flag_after,
                      stream);
    if (e != cudaSuccess) return cuda_st(e);
  }
  std::vector<Pass> passes;
  if (mode == MOE_MODE_DROPLESS) {
    passes.push_back({0, cfg->T, -1, false});
  } else if (mode == MOE_MODE_CAPPED) {
    passes.push_back({0, cfg->T, cap, planned});
  } else {
    if (!planned) {
      e = launch_check(*cfg, b.f.topk_idx, b.f.counts, b.f.offsets,
                       b.f.shard, b.f.flag, b.f.req, b.f.cap, stream);
      if (e != cudaSuccess) return cuda_st(e);
    }
    int32_t flag = 0;
    e = cudaMemcpyAsync(&flag, planned ? b.f.flag_after : b.f.flag,
                        sizeof(flag), cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return cuda_st(e);
    if (info) info->overflow = flag;
    if (!flag) {
      passes.push_back({0, cfg->T, cap, planned});
    } else {
      const int ct = chunk_tokens(*cfg);
      for (int t0 = 0; t0 < cfg->T; t0 += ct)
        passes.push_back({t0, std::min(ct, cfg->T - t0), -1, false});
      if (info) info->n_chunks = static_cast<int32_t>(passes.size());
    }
  }
  std::vector<WgradSegment> segs;
  const size_t G1 = static_cast<size_t>(num_groups(*cfg)) + 1;
  // the tensor-core path with regrouped rows takes the weights' gradient
  // from the down dgrad (bwd_pass) and scales dWd's rows in the regroup
  const bool regrouped =
      cfg->dtype == MOE_BF16 &&
      passes.size() <= static_cast<size_t>(kMaxRegroupSegments);
  for (size_t i = 0; i < passes.size(); ++i) {
    const Pass& p = passes[i];
    e = bwd_pass(*cfg, p.t0, p.tc, p.cap, p.planned, static_cast<int>(i), x,
                 w_gate, w_up, w_down, dy, dx, b, regrouped, status_word,
                 stream);
    if (e != cudaSuccess) return cuda_st(e);
    segs.push_back({b.seg_off + i * G1, p.t0 * cfg->k});
  }
  // the weight gradients' groups: the plan's virtual groups (a duplicate's
  // rows add into its expert's gradient) or the experts themselves
  const Groups wgroups = passes[0].planned
                             ? Groups{num_groups(*cfg), b.f.group_expert}
                             : identity_groups(*cfg);
  e = launch_route_backward(*cfg, logits, b.f.topk_idx, b.dtw, dlogits,
                            stream);
  if (e != cudaSuccess) return cuda_st(e);
  if (regrouped) {
    // one 16-row-aligned row range per expert for the tensor-core GEMMs;
    // the dy rows get their combine weights on the way
    const int64_t rr = regroup_rows(*cfg);
    e = launch_regroup(*cfg, wgroups.n, segs.data(),
                       static_cast<int>(segs.size()), rr, b.f.x_sorted, b.dg,
                       b.du, b.f.h, b.dys, b.xs2, b.dg2, b.du2, b.h2, b.dys2,
                       b.off2, stream, b.wrow);
    if (e != cudaSuccess) return cuda_st(e);
    const WgradSegment one{b.off2, 0};
    return cuda_st(launch_wgrad(*cfg, wgroups, &one, 1, rr,
                                b.xs2, b.dg2, b.du2, b.h2, b.dys2, dw_gate,
                                dw_up, dw_down, kWgradRows16,
                                kWgradGateUp | kWgradDown,
                                status_word, stream));
  }
  return cuda_st(launch_wgrad(
      *cfg, wgroups, segs.data(), static_cast<int>(segs.size()),
      static_cast<int64_t>(cfg->T) * cfg->k, b.f.x_sorted, b.dg, b.du, b.f.h,
      b.dys, dw_gate, dw_up, dw_down, 0, kWgradGateUp | kWgradDown,
      status_word, stream));
}

}  // extern "C"
