// The whole layer with moe_dropless_fallback=layer as one CUDA graph.
// (While the check runs, two side branches already compute the first
// permute tables of either outcome; see build().)
//
// "Support moe_dropless_fallback=layer on the ragged all-to-all MoE path"
// (MaxText pull request 5920), section How: a lax.cond picks the capped path
// when no shard overflows and the chunked dropless fallback otherwise.  On
// the GPU the same choice is a conditional IF node: the check kernel writes
// the flag, a one-thread kernel hands it to cudaGraphSetConditional, and the
// graph runs body 0 (overflow: the chunked passes) or body 1 (the capped
// pass) without the flag ever reaching the host.  One cudaGraphLaunch per
// layer replaces the host round trip and the per-kernel launches.
//
// The graph is bound to the buffers given at creation (inputs, weights,
// output, workspace); callers refresh x and the logits in place and launch
// again.  The traced form adds one-thread kernels that write %globaltimer
// at every stage boundary into a caller buffer, so that a caller can time
// the stages of the graph it runs (conditional bodies cannot hold event
// nodes).
#include "internal.h"

struct moe_layer_graph {
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
  int32_t* flag = nullptr;   // device: 1 when the last launch overflowed
  int32_t n_chunks = 0;      // passes of the overflow branch
};

namespace moe {
namespace {

__global__ void set_branch_kernel(cudaGraphConditionalHandle handle,
                                  const int32_t* __restrict__ flag) {
  cudaGraphSetConditional(handle, *flag != 0 ? 1u : 0u);
}

struct CaptureGuard {  // ends a capture left open by an early return
  cudaStream_t s = nullptr;
  ~CaptureGuard() {
    if (!s) return;
    cudaStreamCaptureStatus st;
    if (cudaStreamIsCapturing(s, &st) == cudaSuccess &&
        st != cudaStreamCaptureStatusNone) {
      cudaGraph_t g = nullptr;
      cudaStreamEndCapture(s, &g);
    }
    cudaStreamDestroy(s);
  }
};

// Events of one capture, destroyed with it (the graph keeps the edges).
struct PipelineEvents {
  cudaEvent_t ev[8] = {};
  cudaError_t create() {
    for (auto& e : ev) {
      const cudaError_t r =
          cudaEventCreateWithFlags(&e, cudaEventDisableTiming);
      if (r != cudaSuccess) return r;
    }
    return cudaSuccess;
  }
  ~PipelineEvents() {
    for (auto e : ev)
      if (e) cudaEventDestroy(e);
  }
};

cudaError_t build(const moe_config_t& c, const void* x, const float* logits,
                  const void* wg, const void* wu, const void* wd, void* y,
                  int32_t* status, const LayerBufs& b, moe_layer_graph* out) {
  cudaError_t e = cudaGraphCreate(&out->graph, 0);
  if (e != cudaSuccess) return e;
  cudaGraphConditionalHandle handle;
  e = cudaGraphConditionalHandleCreate(&handle, out->graph, 0,
                                       cudaGraphCondAssignDefault);
  if (e != cudaSuccess) return e;
  CaptureGuard main_s, body_s;
  if ((e = cudaStreamCreateWithFlags(&main_s.s, cudaStreamNonBlocking)) !=
          cudaSuccess ||
      (e = cudaStreamCreateWithFlags(&body_s.s, cudaStreamNonBlocking)) !=
          cudaSuccess)
    return e;

  // route -> check -> branch select
  e = cudaStreamBeginCaptureToGraph(main_s.s, out->graph, nullptr, nullptr, 0,
                                    cudaStreamCaptureModeRelaxed);
  if (e != cudaSuccess) return e;
  const bool planned = c.redundant_slots > 0;
  if ((e = stamp(b.trace, 0, main_s.s)) != cudaSuccess ||
      (e = launch_route(c, logits, b.topk_idx, b.topk_w, status,
                        main_s.s)) != cudaSuccess ||
      (e = stamp(b.trace, 1, main_s.s)) != cudaSuccess)
    return e;

  // While the check runs, two side branches compute the permute tables each
  // branch needs first: the capped pass's (into row_of_alt and table set
  // 1; not with a duplication plan, whose tables need the plan) and the
  // first fallback chunk's (into row_of and set 0).  Both depend only on the
  // routing; the branch not taken leaves its tables unused.
  CaptureGuard spec_a, spec_b;
  PipelineEvents se;
  const int ct = chunk_tokens(c);
  const int n_all = ct > 0 ? (c.T + ct - 1) / ct : 0;
  const bool spec_capped = !planned;
  const bool spec_chunk = n_all >= 2;
  if ((e = se.create()) != cudaSuccess ||
      (e = cudaStreamCreateWithFlags(&spec_a.s, cudaStreamNonBlocking)) !=
          cudaSuccess ||
      (e = cudaStreamCreateWithFlags(&spec_b.s, cudaStreamNonBlocking)) !=
          cudaSuccess ||
      (e = cudaEventRecord(se.ev[0], main_s.s)) != cudaSuccess)
    return e;
  if (spec_capped &&
      ((e = cudaStreamWaitEvent(spec_a.s, se.ev[0], 0)) != cudaSuccess ||
       (e = launch_permute_tables(c, b.topk_idx, capacity_rows(c),
                                  b.row_of_alt, b.alt.sorted_token,
                                  b.alt.group_offsets, b.alt.uniq_offsets,
                                  b.alt.n_dropped, b.alt.pws, status,
                                  spec_a.s)) != cudaSuccess ||
       (e = cudaEventRecord(se.ev[1], spec_a.s)) != cudaSuccess))
    return e;
  if (spec_chunk &&
      ((e = cudaStreamWaitEvent(spec_b.s, se.ev[0], 0)) != cudaSuccess ||
       (e = launch_permute_tables(sub_config(c, ct), b.topk_idx, -1,
                                  b.row_of, b.sorted_token, b.group_offsets,
                                  b.uniq_offsets, b.n_dropped, b.pws, status,
                                  spec_b.s)) != cudaSuccess ||
       (e = cudaEventRecord(se.ev[2], spec_b.s)) != cudaSuccess))
    return e;
  if ((e = launch_check(c, b.topk_idx, b.counts, b.offsets, b.shard, b.flag,
                        b.req, b.cap, main_s.s)) != cudaSuccess)
    return e;
  if (planned &&
      (e = launch_plan(c, b.counts, b.divert, b.slot_of, b.group_expert,
                       b.shard_after, b.flag_after, main_s.s)) != cudaSuccess)
    return e;
  set_branch_kernel<<<1, 1, 0, main_s.s>>>(handle,
                                           planned ? b.flag_after : b.flag);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if ((spec_capped &&
       (e = cudaStreamWaitEvent(main_s.s, se.ev[1], 0)) != cudaSuccess) ||
      (spec_chunk &&
       (e = cudaStreamWaitEvent(main_s.s, se.ev[2], 0)) != cudaSuccess))
    return e;
  if ((e = stamp(b.trace, 2, main_s.s)) != cudaSuccess) return e;

  cudaStreamCaptureStatus cst;
  const cudaGraphNode_t* deps = nullptr;
  size_t ndeps = 0;
  e = cudaStreamGetCaptureInfo(main_s.s, &cst, nullptr, nullptr, &deps,
                               nullptr, &ndeps);
  if (e != cudaSuccess) return e;
  cudaGraphNodeParams cp = {};
  cp.type = cudaGraphNodeTypeConditional;
  cp.conditional.handle = handle;
  cp.conditional.type = cudaGraphCondTypeIf;
  cp.conditional.size = 2;
  cudaGraphNode_t cond;
  e = cudaGraphAddNode(&cond, out->graph, deps, nullptr, ndeps, &cp);
  if (e != cudaSuccess) return e;
  cudaGraph_t body_overflow = cp.conditional.phGraph_out[0];
  cudaGraph_t body_capped = cp.conditional.phGraph_out[1];

  // body 0: the chunked dropless fallback on the routing already computed,
  // each chunk's permute tables a chunk ahead on a second captured stream
  cudaGraph_t tmp = nullptr;
  CaptureGuard side_s;
  PipelineEvents pe;
  if ((e = cudaStreamCreateWithFlags(&side_s.s, cudaStreamNonBlocking)) !=
          cudaSuccess ||
      (e = pe.create()) != cudaSuccess)
    return e;
  PassPipeline pp{side_s.s, pe.ev[0], {pe.ev[1], pe.ev[2]},
                  {pe.ev[3], pe.ev[4]}};
  pp.first_ready = spec_chunk;
  e = cudaStreamBeginCaptureToGraph(body_s.s, body_overflow, nullptr, nullptr,
                                    0, cudaStreamCaptureModeRelaxed);
  if (e != cudaSuccess) return e;
  e = chunked_passes(c, x, b.topk_idx, b.topk_w, wg, wu, wd, y, b, status,
                     body_s.s, &out->n_chunks, &pp);
  if (e != cudaSuccess) return e;
  if ((e = cudaStreamEndCapture(body_s.s, &tmp)) != cudaSuccess) return e;

  // body 1: the capped pass
  e = cudaStreamBeginCaptureToGraph(body_s.s, body_capped, nullptr, nullptr,
                                    0, cudaStreamCaptureModeRelaxed);
  if (e != cudaSuccess) return e;
  e = spec_capped
          ? capped_pass_tabled(c, x, b.topk_w, wg, wu, wd, y, b,
                               b.row_of_alt, b.alt, status, body_s.s)
          : pass(c, x, b.topk_idx, b.topk_w, capacity_rows(c), wg, wu, wd, y,
                 b, status, body_s.s, planned);
  if (e != cudaSuccess) return e;
  if ((e = cudaStreamEndCapture(body_s.s, &tmp)) != cudaSuccess) return e;

  e = cudaStreamUpdateCaptureDependencies(main_s.s, &cond, nullptr, 1,
                                          cudaStreamSetCaptureDependencies);
  if (e != cudaSuccess) return e;
  if ((e = cudaStreamEndCapture(main_s.s, &tmp)) != cudaSuccess) return e;
  out->flag = planned ? b.flag_after : b.flag;
  return cudaGraphInstantiate(&out->exec, out->graph, 0);
}

void release(moe_layer_graph* g) {
  if (!g) return;
  if (g->exec) cudaGraphExecDestroy(g->exec);
  if (g->graph) cudaGraphDestroy(g->graph);
  delete g;
}

moe_status_t create_graph(const moe_config_t* cfg, const void* x,
                          const float* logits, const void* w_gate,
                          const void* w_up, const void* w_down, void* y,
                          int32_t* status_word, void* workspace,
                          size_t workspace_bytes, int64_t* trace,
                          moe_layer_graph_t** graph_out) {
  if (graph_out == nullptr) return MOE_ERR_INVALID_ARG;
  *graph_out = nullptr;
  moe_status_t st = validate(cfg);
  if (st != MOE_OK) return st;
  if (cfg->T < 1) return MOE_ERR_INVALID_ARG;
  if (cfg->F > 0 && !gmm_shape_ok(*cfg)) return MOE_ERR_UNSUPPORTED;
  if (!ok_ptr(x, true) || !ok_ptr(logits, false) ||
      (cfg->F > 0 && !weights_ok(w_gate, w_up, w_down)) || !ok_ptr(y, true))
    return MOE_ERR_INVALID_ARG;
  if (workspace == nullptr || !ok_ptr(workspace, true) ||
      workspace_bytes < layer_bytes(*cfg, cfg->T))
    return MOE_ERR_WORKSPACE;
  LayerBufs b = carve_layer(workspace, *cfg, cfg->T, nullptr);
  b.trace = trace;
  moe_layer_graph* g = new moe_layer_graph();
  const cudaError_t e = build(*cfg, x, logits, w_gate, w_up, w_down, y,
                              status_word, b, g);
  if (e != cudaSuccess) {
    release(g);
    cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  *graph_out = g;
  return MOE_OK;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

int32_t moe_layer_graph_trace_slots(const moe_config_t* cfg) {
  if (validate(cfg) != MOE_OK) return 0;
  const int ct = chunk_tokens(*cfg);
  const int n = ct > 0 ? (cfg->T + ct - 1) / ct : 0;
  return trace_slot(std::max(n, 1), 0);
}

moe_status_t moe_layer_graph_create_traced(
    const moe_config_t* cfg, const void* x, const float* logits,
    const void* w_gate, const void* w_up, const void* w_down, void* y,
    int32_t* status_word, void* workspace, size_t workspace_bytes,
    int64_t* trace, moe_layer_graph_t** graph_out) {
  if (graph_out == nullptr) return MOE_ERR_INVALID_ARG;
  *graph_out = nullptr;
  if (trace == nullptr || (reinterpret_cast<uintptr_t>(trace) & 7u) != 0)
    return MOE_ERR_INVALID_ARG;
  return create_graph(cfg, x, logits, w_gate, w_up, w_down, y, status_word,
                      workspace, workspace_bytes, trace, graph_out);
}

moe_status_t moe_layer_graph_create(const moe_config_t* cfg, const void* x,
                                    const float* logits, const void* w_gate,
                                    const void* w_up, const void* w_down,
                                    void* y, int32_t* status_word,
                                    void* workspace, size_t workspace_bytes,
                                    moe_layer_graph_t** graph_out) {
  return create_graph(cfg, x, logits, w_gate, w_up, w_down, y, status_word,
                      workspace, workspace_bytes, nullptr, graph_out);
}

moe_status_t moe_layer_graph_launch(moe_layer_graph_t* graph,
                                    moe_stream_t stream) {
  if (graph == nullptr || graph->exec == nullptr) return MOE_ERR_INVALID_ARG;
  return cudaGraphLaunch(graph->exec, stream) == cudaSuccess ? MOE_OK
                                                             : MOE_ERR_CUDA;
}

const int32_t* moe_layer_graph_overflow_flag(const moe_layer_graph_t* graph) {
  return graph ? graph->flag : nullptr;
}

int32_t moe_layer_graph_fallback_chunks(const moe_layer_graph_t* graph) {
  return graph ? graph->n_chunks : 0;
}

void moe_layer_graph_destroy(moe_layer_graph_t* graph) { release(graph); }

}  // extern "C"
