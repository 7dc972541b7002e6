/*
 * moe.h -- C ABI of the GB300 (sm_103a) MoE token-dispatch + expert-compute
 * library (libmoe_gb300.so).
 *
 * The layer this library computes is the expert-parallel MoE layer of the
 * MaxText pages:
 *   router top-k -> per-expert / per-shard counts and the ragged
 *   receive-buffer overflow check -> expert-sorted permute with per-shard
 *   token dedup -> grouped-GEMM SwiGLU expert FFN -> weighted combine,
 *   with the chunked dropless fallback when a shard would overflow.
 * Sources:
 *   [PR5920] "Support moe_dropless_fallback=layer on the ragged all-to-all
 *            MoE path" (MaxText pull request 5920), sections Why, How,
 *            Shortcomings, Tests.
 *   [PR4760] "Moe dynamic redundancy" (MaxText pull request 4760), review
 *            comments on ra2a_dedup_and_route and get_gmm_for_local_experts.
 *   [PR4969] "MoE ring-of-experts: TC Pallas ring all-gather for the combine
 *            backward + x_sorted remat save" (MaxText pull request 4969),
 *            section What.
 * On one GPU the expert-parallel shards are logical ranges of E/S
 * consecutive experts; nothing is exchanged between GPUs.
 *
 * Conventions for every entry point
 * ---------------------------------
 * Ownership: the caller owns every buffer.  The library never allocates
 *   device memory; scratch space is passed in as `workspace`, sized by
 *   moe_workspace_bytes().  Device pointers are plain CUDA device pointers.
 * Execution: every call only enqueues work on `stream` (a cudaStream_t; NULL
 *   is the legacy default stream) and returns before it runs, except
 *   moe_layer() in MOE_MODE_FALLBACK_LAYER, which reads the 4-byte overflow
 *   flag back to the host (one stream synchronisation) to choose its branch.
 * Errors: arguments are validated on the host before anything is launched;
 *   a bad argument returns MOE_ERR_INVALID_ARG (or MOE_ERR_UNSUPPORTED for a
 *   valid shape the kernels do not cover) and nothing is enqueued.  A failed
 *   launch returns MOE_ERR_CUDA.  Conditions found while the kernels run are
 *   OR-ed into an optional device status word (int32, see MOE_DEV_*), which
 *   the caller zeroes and reads when it wants; a NULL status word is allowed.
 * Layouts (row-major, C order):
 *   x        [T, H]    dtype         token activations
 *   logits   [T, E]    float32       router logits
 *   topk_idx [T, k]    int32         chosen experts, best first
 *   topk_w   [T, k]    float32       combine weights
 *   w_gate   [E, H, F] dtype         gate projection of each expert
 *   w_up     [E, H, F] dtype         up projection of each expert
 *   w_down   [E, F, H] dtype         down projection of each expert
 *   x_sorted [T*k, H]  dtype         routed rows, grouped by expert
 *   h        [T*k, F]  dtype         SwiGLU activations of the routed rows
 *   y_sorted [T*k, H]  dtype         expert outputs of the routed rows
 *   y        [T, H]    dtype         layer output
 * The dtype matrices (x, w_*, x_sorted, h, y_sorted, y) must be 16-byte
 * aligned and H and F must make their rows a multiple of 16 bytes; the
 * int32/float arrays need only their natural 4-byte alignment.  A pointer
 * that breaks this is rejected.  Buffers indexed by routed row are sized for the
 * worst case of T*k rows; a capped pass fills only the first
 * group_offsets[E] of them.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *moe_stream_t; /* same type as cudaStream_t */

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1, /* bad shape, pointer, alignment or option      */
  MOE_ERR_UNSUPPORTED = 2, /* valid, but outside what the kernels cover    */
  MOE_ERR_WORKSPACE = 3,   /* workspace missing or smaller than required   */
  MOE_ERR_CUDA = 4         /* a CUDA runtime call or launch failed         */
} moe_status_t;

/* Bits OR-ed into the device status word by the kernels. */
#define MOE_DEV_NONFINITE 1 /* a NaN/inf logit was seen; it ranked as -inf */
#define MOE_DEV_TIMEOUT 2   /* a bounded wait in the GEMM gave up          */
#define MOE_DEV_BAD_INDEX 4 /* an expert index outside [0, E) was skipped  */
#define MOE_DEV_UNALIGNED 8 /* MOE_WGRAD_ROWS16 given, a group's rows are
                               not a multiple of 16: nothing was written  */

typedef enum { MOE_F32 = 0, MOE_BF16 = 1 } moe_dtype_t;

typedef struct {
  int32_t T; /* tokens (>= 0)                                             */
  int32_t H; /* hidden size                                               */
  int32_t E; /* experts, 1..1024                                          */
  int32_t k; /* experts per token, 1..min(E, 32)                          */
  int32_t F; /* expert FFN width                                          */
  int32_t S; /* logical EP shards, divides E, 1..64                       */
  /* Receive-buffer cap per shard [PR5920 Why]: > 0 gives the capacity
   * C = floor(factor * T * k / S) rows (computed in double from this float,
   * at most T*k); <= 0 means uncapped (the pages' -1).                    */
  float ragged_buffer_factor;
  /* Chunks of the dropless fallback [PR5920 How]; 0 derives the count:
   * chunks of floor(C / min(k, E/S)) tokens (at least 1), so that a
   * chunk's worst-case receive fits C.  n > 0 gives chunks of ceil(T/n). */
  int32_t n_chunks;
  moe_dtype_t dtype; /* type of x, the expert weights, h, y_sorted and y   */
  /* Combine weights: 0 = softmax over all E logits read at the chosen
   * experts; 1 = softmax over the k chosen logits.                        */
  int32_t renorm;
  /* Dynamic redundant experts [PR4760]: spare duplicate slots per shard
   * (num_slots_B); 0 = off.  With B > 0 the layer plans duplicates of the
   * hottest experts (moe_plan_duplication) before its overflow check.
   * Needs E + S*B <= 1024.                                                */
  int32_t redundant_slots;
} moe_config_t;

/* ----------------------------------------------------------------------
 * moe_router_logits -- the router's scores of every token for every expert
 * [PR5920 How: the overflow check is computed from the router's top-k,
 * i.e. from these scores]:
 *     logits[t, e] = sum_h x[t, h] w_router[h, e]  (+ logit_offset[t, e])
 * accumulated in float32.  bf16 layers with H % 64 == 0 and E % 128 == 0
 * (and 16-byte aligned logits and offset) run on the tensor cores (tcgen05,
 * 128-column float32 tiles of one token group); other shapes and fp32
 * layers on CUDA cores.
 *   x            in  [T, H] dtype, 16-byte aligned
 *   w_router     in  [H, E] dtype (E contiguous), 16-byte aligned
 *   logit_offset in  [T, E] float32 or NULL: added after the product (an
 *                    expert bias broadcast over tokens, routing noise, ...)
 *   logits       out [T, E] float32 (the input of moe_route)
 *   status_word  in/out, device int32 or NULL: MOE_DEV_TIMEOUT if a
 *                pipeline wait of the tensor-core form gave up.
 * ---------------------------------------------------------------------- */
moe_status_t moe_router_logits(const moe_config_t *cfg, const void *x,
                               const void *w_router,
                               const float *logit_offset, float *logits,
                               int32_t *status_word, moe_stream_t stream);

/* ----------------------------------------------------------------------
 * moe_route -- router top-k and combine weights [PR5920 How: the check is
 * computed from the router's top-k].  One warp per token.
 *   logits   in  [T, E] float32 (device)
 *   topk_idx out [T, k] int32: experts by descending logit; equal logits
 *            go to the lower index.  NaN/inf logits rank as -inf and set
 *            MOE_DEV_NONFINITE.
 *   topk_w   out [T, k] float32: see moe_config_t.renorm; a token with no
 *            finite logit gets zero weights.
 *   status_word  in/out, device int32 or NULL.
 * ---------------------------------------------------------------------- */
moe_status_t moe_route(const moe_config_t *cfg, const float *logits,
                       int32_t *topk_idx, float *topk_w,
                       int32_t *status_word, moe_stream_t stream);

/* ----------------------------------------------------------------------
 * moe_check_overflow -- counts and the ragged overflow check [PR5920 Why,
 * How; PR4760 review: group_sizes per expert, experts_per_rank].
 *   topk_idx        in  [T, k] int32 (device)
 *   expert_counts   out [E]   rows routed to each expert
 *   expert_offsets  out [E+1] exclusive scan of expert_counts
 *   shard_counts    out [S]   rows routed to each shard (r_s)
 *   overflow_flag   out [1]   1 iff some r_s > C (strict); 0 when uncapped
 *   required_factor out [1]   float max_s r_s * S / (T*k) (0 when T = 0)
 *   capacity        out [1]   C, or -1 when uncapped
 * All outputs are device pointers.  Indices outside [0, E) are skipped.
 * ---------------------------------------------------------------------- */
moe_status_t moe_check_overflow(const moe_config_t *cfg,
                                const int32_t *topk_idx,
                                int32_t *expert_counts,
                                int32_t *expert_offsets,
                                int32_t *shard_counts,
                                int32_t *overflow_flag,
                                float *required_factor, int32_t *capacity,
                                moe_stream_t stream);

/* ----------------------------------------------------------------------
 * moe_permute -- stable expert-sorted permute with the capped drop rule and
 * per-shard token dedup [PR5920 Why: rows past the cap are dropped; PR4760
 * review: ra2a_dedup_and_route / expand_indices must never truncate;
 * PR4969 What: x_sorted].
 *   Routed rows (t, j) are ordered by (expert, token).  With capped != 0 a
 *   row whose rank inside its shard is >= C is dropped; kept rows are
 *   compacted.  U_s is the ascending set of tokens with a kept row in shard
 *   s; uniq_tokens = U_0 ++ U_1 ++ ...
 *   x            in  [T, H] dtype
 *   topk_idx     in  [T, k] int32
 *   capped       in  nonzero: apply C from cfg; 0: uncapped
 *   x_sorted     out [T*k, H]: row r = x[sorted_token[r]]
 *   row_of       out [T, k] int32: sorted row of (t, j), -1 if dropped
 *   sorted_token out [T*k] int32: token of each kept row
 *   group_offsets out [E+1] int32: kept rows per expert, scanned
 *   uniq_offsets out [S+1] int32: scanned |U_s|
 *   uniq_tokens  out [T*min(k,S)] int32 (first uniq_offsets[S] written)
 *   expand_idx   out [T*k] int32: row r -> its token's slot in uniq_tokens
 *   n_dropped    out [1] int32
 *   workspace    scratch of moe_workspace_bytes(cfg, MOE_WS_PERMUTE) bytes
 * Entries past the valid prefix of sorted_token, expand_idx, x_sorted and
 * uniq_tokens are left unwritten.
 * ---------------------------------------------------------------------- */
moe_status_t moe_permute(const moe_config_t *cfg, const void *x,
                         const int32_t *topk_idx, int32_t capped,
                         void *x_sorted, int32_t *row_of,
                         int32_t *sorted_token, int32_t *group_offsets,
                         int32_t *uniq_offsets, int32_t *uniq_tokens,
                         int32_t *expand_idx, int32_t *n_dropped,
                         void *workspace, size_t workspace_bytes,
                         moe_stream_t stream);

/* ----------------------------------------------------------------------
 * moe_permute_noalloc -- moe_permute with no workspace argument.  The pages
 * have no counterpart to this call; it exists for callers of this library
 * that cannot allocate device memory themselves: code inside a host
 * framework whose pool allocator owns all device memory and forbids other
 * cudaMalloc calls, or latency-critical paths where cudaMalloc's implicit
 * device-wide synchronisation is unacceptable.  Arguments and outputs are
 * those of moe_permute; the caller still owns every input and output.
 *   - The counting-sort tables live in one 8 MiB device array inside the
 *     library, held by every GPU that loads it until the process exits.  A
 *     call whose tables (moe_workspace_bytes(cfg, MOE_WS_PERMUTE)) exceed
 *     8 MiB returns MOE_ERR_WORKSPACE and launches nothing.
 *   - The first call on a device looks up the array's device address with
 *     that device current and caches it; make that first call before any
 *     stream capture.  The cached address belongs to the device's context
 *     at that time: after cudaDeviceReset (or any reset of the primary
 *     context) it is stale, so a process that resets a device must not
 *     call moe_permute_noalloc on it again.
 *   - Every call on a device uses the same array, which keeps the previous
 *     call's contents (nothing in it needs to start at zero: each call
 *     writes every entry before reading it).  Calls whose work overlaps on
 *     the GPU race on it; order them on one stream or with events.
 *   - It calls no cudaMalloc, cudaFree or other allocating routine.
 * ---------------------------------------------------------------------- */
moe_status_t moe_permute_noalloc(const moe_config_t *cfg, const void *x,
                                 const int32_t *topk_idx, int32_t capped,
                                 void *x_sorted, int32_t *row_of,
                                 int32_t *sorted_token,
                                 int32_t *group_offsets,
                                 int32_t *uniq_offsets, int32_t *uniq_tokens,
                                 int32_t *expand_idx, int32_t *n_dropped,
                                 moe_stream_t stream);

/* ----------------------------------------------------------------------
 * moe_gmm_swiglu -- grouped GEMM SwiGLU expert FFN over ragged expert groups
 * [PR4760 review: grouped matmul with group_sizes per expert; expert weights
 * w0 of shape [E, H, H_ffn]].  For the rows r of group e
 * ([group_offsets[e], group_offsets[e+1])):
 *     h[r] = silu(x_sorted[r] w_gate[e]) * (x_sorted[r] w_up[e])
 *     y_sorted[r] = h[r] w_down[e],   silu(z) = z / (1 + exp(-z)).
 *   bf16: tcgen05 tensor cores, fp32 accumulate, h and y_sorted rounded to
 *   bf16 (needs H % 128 == 0 and F % 128 == 0, else MOE_ERR_UNSUPPORTED).
 *   f32: CUDA-core FMA in fp32.
 *   x_sorted, h, y_sorted have T*k rows allocated; group_offsets [E+1] is on
 *   the device (nondecreasing, group_offsets[E] <= T*k).  Rows past
 *   group_offsets[E] are not written.  status_word: MOE_DEV_TIMEOUT if a
 *   pipeline wait gave up (the output is then incomplete).
 * ---------------------------------------------------------------------- */
moe_status_t moe_gmm_swiglu(const moe_config_t *cfg, const void *x_sorted,
                            const int32_t *group_offsets,
                            const void *w_gate, const void *w_up,
                            const void *w_down, void *h, void *y_sorted,
                            int32_t *status_word, moe_stream_t stream);

/* The two halves of moe_gmm_swiglu, one kernel launch each (same rules):
 * moe_gmm_gate_up writes h = silu(x_sorted w_gate[e]) * (x_sorted w_up[e]);
 * moe_gmm_down writes y_sorted = h w_down[e].  n_groups = 0 and
 * group_expert = NULL mean the E experts' own groups; otherwise the row
 * groups and weight map of moe_gmm_swiglu_mapped.                         */
moe_status_t moe_gmm_gate_up(const moe_config_t *cfg, int32_t n_groups,
                             const int32_t *group_expert,
                             const void *x_sorted,
                             const int32_t *group_offsets,
                             const void *w_gate, const void *w_up, void *h,
                             int32_t *status_word, moe_stream_t stream);
moe_status_t moe_gmm_down(const moe_config_t *cfg, int32_t n_groups,
                          const int32_t *group_expert, const void *h,
                          const int32_t *group_offsets, const void *w_down,
                          void *y_sorted, int32_t *status_word,
                          moe_stream_t stream);

/* ----------------------------------------------------------------------
 * moe_combine -- weighted unpermute [PR4969 What: the combine reduces the
 * expert outputs back to tokens].  y[t] = sum_{j<k, row_of[t,j] >= 0}
 * topk_w[t,j] * y_sorted[row_of[t,j]], accumulated in fp32 in slot order.
 * A token whose rows were all dropped gets zeros.
 * ---------------------------------------------------------------------- */
moe_status_t moe_combine(const moe_config_t *cfg, const void *y_sorted,
                         const int32_t *row_of, const float *topk_w, void *y,
                         moe_stream_t stream);

/* ----------------------------------------------------------------------
 * moe_layer_dropless_chunked -- the chunked dropless fallback [PR5920 How,
 * Shortcomings]: the layer runs over contiguous token chunks (see
 * moe_config_t.n_chunks), each uncapped (force_dropless), one after another
 * on `stream`, each writing its own rows of y.  The result equals the
 * uncapped layer.  workspace: moe_workspace_bytes(cfg, MOE_WS_CHUNKED).
 * ---------------------------------------------------------------------- */
moe_status_t moe_layer_dropless_chunked(const moe_config_t *cfg,
                                        const void *x, const float *logits,
                                        const void *w_gate, const void *w_up,
                                        const void *w_down, void *y,
                                        int32_t *status_word, void *workspace,
                                        size_t workspace_bytes,
                                        moe_stream_t stream);

/* ----------------------------------------------------------------------
 * Dynamic redundant experts ("Moe dynamic redundancy", MaxText pull request
 * 4760, review of plan_expert_duplication).  B = cfg->redundant_slots spare
 * slots per shard; a slot holds a duplicate of one expert and computes with
 * that expert's weights (on one GPU nothing is copied).
 * Virtual groups: shard s owns groups [s*(E/S+B), (s+1)*(E/S+B)): its E/S
 * experts, then its B slots; G = S*(E/S+B) groups in all.
 *
 * moe_plan_duplication -- one warp, at most S*B rounds.  Each round takes
 * the most loaded shard (ties: lower index), its hottest expert that has
 * rows and is not yet duplicated (has_candidate; ties: lower index), and
 * the least loaded other shard with a free slot; it stops when either is
 * missing or the gap is zero, else moves n = min(rows of e,
 * (load_max - load_min) / 2) rows of e to the next free slot of that shard.
 *   expert_counts       in  [E] rows per expert (moe_check_overflow)
 *   divert              out [E] rows of e moved to its duplicate
 *   slot_of             out [E] virtual group of e's duplicate, -1 if none
 *   group_expert        out [G] expert behind each virtual group, -1 for an
 *                           unused slot
 *   shard_counts_after  out [S] shard loads after the diversion
 *   overflow_flag_after out [1] 1 iff some load after > C (0 if uncapped)
 * ---------------------------------------------------------------------- */
moe_status_t moe_plan_duplication(const moe_config_t *cfg,
                                  const int32_t *expert_counts,
                                  int32_t *divert, int32_t *slot_of,
                                  int32_t *group_expert,
                                  int32_t *shard_counts_after,
                                  int32_t *overflow_flag_after,
                                  moe_stream_t stream);

/* moe_permute_planned -- moe_permute over the virtual groups of a plan: the
 * last divert[e] rows of expert e (token order) go to group slot_of[e], the
 * rest to e's own group; capacity and dedup apply per shard of the virtual
 * layout.  group_offsets has G+1 entries; the other outputs and the
 * workspace (moe_workspace_bytes(cfg, MOE_WS_PERMUTE)) are those of
 * moe_permute. */
moe_status_t moe_permute_planned(const moe_config_t *cfg, const void *x,
                                 const int32_t *topk_idx, int32_t capped,
                                 const int32_t *divert,
                                 const int32_t *slot_of, void *x_sorted,
                                 int32_t *row_of, int32_t *sorted_token,
                                 int32_t *group_offsets,
                                 int32_t *uniq_offsets, int32_t *uniq_tokens,
                                 int32_t *expand_idx, int32_t *n_dropped,
                                 void *workspace, size_t workspace_bytes,
                                 moe_stream_t stream);

/* ----------------------------------------------------------------------
 * moe_permute_tables / moe_permute_scatter -- moe_permute (or, with divert
 * and slot_of, moe_permute_planned) in two calls, same bits.  The pages
 * have no such split; it lets a caller of the chunked fallback [PR5920
 * How: the fallback runs the layer chunk by chunk] compute the next
 * chunk's counting-sort tables on a second stream while the current
 * chunk's expert FFN runs, so that only the row copy stays between two
 * chunks' FFNs.
 * moe_permute_tables: the counting sort.
 *   topk_idx, capped         as moe_permute
 *   divert, slot_of          both NULL (no plan) or both a plan's arrays
 *                            (as moe_permute_planned)
 *   row_of, sorted_token, group_offsets, n_dropped   out, as moe_permute
 *   uniq_offsets             out [S+1]; complete only after the scatter
 *   workspace                moe_workspace_bytes(cfg, MOE_WS_PERMUTE)
 *                            bytes; holds the scatter's tables: pass the
 *                            same workspace, unchanged, to the scatter
 * moe_permute_scatter: x_sorted, uniq_tokens, expand_idx and the rest of
 *   uniq_offsets, from row_of, uniq_offsets and the workspace that
 *   moe_permute_tables wrote (same cfg).  Order the two on the device
 *   (same stream, or an event) before the scatter runs.
 * ---------------------------------------------------------------------- */
moe_status_t moe_permute_tables(const moe_config_t *cfg,
                                const int32_t *topk_idx, int32_t capped,
                                const int32_t *divert,
                                const int32_t *slot_of, int32_t *row_of,
                                int32_t *sorted_token,
                                int32_t *group_offsets,
                                int32_t *uniq_offsets, int32_t *n_dropped,
                                void *workspace, size_t workspace_bytes,
                                moe_stream_t stream);
/* (moe_permute_scatter with x_sorted = NULL writes the index outputs --
 * uniq_tokens, expand_idx, the rest of uniq_offsets -- and copies no row;
 * x is then not read and may be NULL.) */
moe_status_t moe_permute_scatter(const moe_config_t *cfg, const void *x,
                                 const int32_t *row_of,
                                 int32_t *uniq_offsets, void *x_sorted,
                                 int32_t *uniq_tokens, int32_t *expand_idx,
                                 const void *workspace,
                                 size_t workspace_bytes, moe_stream_t stream);

/* moe_gmm_swiglu_mapped -- moe_gmm_swiglu over n_groups row groups where
 * group g computes with the weights of expert group_expert[g] (device,
 * [n_groups]; a group of an expert < 0 must be empty).  group_offsets has
 * n_groups+1 entries, n_groups <= 1024. */
moe_status_t moe_gmm_swiglu_mapped(const moe_config_t *cfg, int32_t n_groups,
                                   const int32_t *group_expert,
                                   const void *x_sorted,
                                   const int32_t *group_offsets,
                                   const void *w_gate, const void *w_up,
                                   const void *w_down, void *h,
                                   void *y_sorted, int32_t *status_word,
                                   moe_stream_t stream);

/* ----------------------------------------------------------------------
 * moe_layer -- the whole layer (an extension composing the calls above).
 *   cfg->F = 0 gives the dispatch-only layer of the routing/permute/dedup
 *   sweep: no expert FFN, the combine reads the permuted rows back
 *   (y[t] = sum_j w[t,j] x[t] over its kept rows); the weights may be NULL.
 *   MOE_MODE_FALLBACK_LAYER: route, check, read the flag; no overflow -> the
 *     capped path; overflow -> the chunked dropless fallback, reusing the
 *     routing [PR5920 How, moe_dropless_fallback=layer].  With
 *     cfg->redundant_slots > 0 the check is taken after
 *     moe_plan_duplication, on the shard loads of the virtual groups, and
 *     the capped path runs over those groups.
 *   MOE_MODE_CAPPED: the capped path only; rows past C are dropped (over
 *     the virtual groups of a plan when cfg->redundant_slots > 0).
 *   MOE_MODE_DROPLESS: one uncapped pass (force_dropless).
 * info (host, may be NULL) receives what the call learned; workspace:
 * moe_workspace_bytes(cfg, MOE_WS_LAYER).
 * ---------------------------------------------------------------------- */
typedef enum {
  MOE_MODE_FALLBACK_LAYER = 0,
  MOE_MODE_CAPPED = 1,
  MOE_MODE_DROPLESS = 2
} moe_mode_t;

typedef struct {
  int32_t overflow; /* flag read back (FALLBACK_LAYER); -1 if not read   */
  int32_t n_chunks; /* passes run: 1, or the fallback's chunk count       */
  int64_t capacity; /* C, or -1 when uncapped                             */
} moe_layer_info_t;

moe_status_t moe_layer(const moe_config_t *cfg, const void *x,
                       const float *logits, const void *w_gate,
                       const void *w_up, const void *w_down, void *y,
                       moe_mode_t mode, moe_layer_info_t *info,
                       int32_t *status_word, void *workspace,
                       size_t workspace_bytes, moe_stream_t stream);

/* ----------------------------------------------------------------------
 * moe_layer_graph_* -- the MOE_MODE_FALLBACK_LAYER layer as one CUDA graph
 * (an extension; cfg->F = 0: the dispatch-only layer, as moe_layer).  The branch of [PR5920 How] is a conditional IF node:
 * the check kernel's flag selects, on the device, either the chunked
 * dropless passes or the capped pass, so a launch never waits on the host.
 * In the chunked branch each chunk's permute tables (moe_permute_tables)
 * run on a second branch of the graph during the previous chunk's expert
 * FFN; the results are those of moe_layer, bit for bit.
 *   create: validates like moe_layer (T >= 1), captures the graph on the
 *     current device and instantiates it; the graph stays bound to x,
 *     logits, the weights, y, status_word and workspace (refresh x and the
 *     logits in place between launches).  Allocates no device memory; the
 *     graph objects live on the host until moe_layer_graph_destroy.
 *   launch: enqueues one layer on `stream` (not the legacy NULL stream
 *     while another capture is open).
 *   overflow_flag: device int32 written by each launch (1 = overflowed).
 *   fallback_chunks: passes the overflow branch runs.
 * ---------------------------------------------------------------------- */
typedef struct moe_layer_graph moe_layer_graph_t;

moe_status_t moe_layer_graph_create(const moe_config_t *cfg, const void *x,
                                    const float *logits, const void *w_gate,
                                    const void *w_up, const void *w_down,
                                    void *y, int32_t *status_word,
                                    void *workspace, size_t workspace_bytes,
                                    moe_layer_graph_t **graph_out);
/* moe_layer_graph_create_traced -- the same graph with a device timestamp
 * (int64 nanoseconds of %globaltimer, written by a one-thread kernel) at
 * every stage boundary, for timing the stages of the graph a caller runs
 * (a conditional node's bodies cannot hold CUDA event nodes).  trace: device
 * int64 [moe_layer_graph_trace_slots(cfg)], 8-byte aligned; each launch
 * writes, in order on the device:
 *   0 layer start, 1 routing done, 2 check (and plan) and branch select
 *   done; then for pass p (the capped pass is p = 0; the fallback's chunks
 *   p = 0 .. n-1): 3 + 5p start (permute tables and row scatter),
 *   4 + 5p GEMM1 start, 5 + 5p GEMM2 start, 6 + 5p combine start,
 *   7 + 5p pass end.
 * Slots of passes the launch did not run keep their old values.  The
 * stamps add one small kernel per boundary (about 1 us each); the layer's
 * results are those of the untraced graph, bit for bit. */
moe_status_t moe_layer_graph_create_traced(
    const moe_config_t *cfg, const void *x, const float *logits,
    const void *w_gate, const void *w_up, const void *w_down, void *y,
    int32_t *status_word, void *workspace, size_t workspace_bytes,
    int64_t *trace, moe_layer_graph_t **graph_out);
/* Trace slots of the traced graph: 3 + 5 * max(1, fallback chunks); 0 for
 * an invalid cfg. */
int32_t moe_layer_graph_trace_slots(const moe_config_t *cfg);
moe_status_t moe_layer_graph_launch(moe_layer_graph_t *graph,
                                    moe_stream_t stream);
const int32_t *moe_layer_graph_overflow_flag(const moe_layer_graph_t *graph);
int32_t moe_layer_graph_fallback_chunks(const moe_layer_graph_t *graph);
void moe_layer_graph_destroy(moe_layer_graph_t *graph);

/* ----------------------------------------------------------------------
 * Backward pass.  "Support moe_dropless_fallback=layer on the ragged
 * all-to-all MoE path" [PR5920 Tests]: with the layer fallback, outputs
 * AND gradients match the dropless model; [PR5920 How]: the fallback's
 * backward recomputes one chunk at a time and accumulates the expert-weight
 * gradients across chunks.  Per routed row r = (t, j) of expert e:
 *   dw[t,j] = <dy[t], y_sorted[r]>,  dy_sorted[r] = w[t,j] dy[t]
 *   dWd[e] += h^T dy_sorted,  dh = dy_sorted Wd[e]^T
 *   dg = dh * u * silu'(g),  du = dh * silu(g)
 *   dWg[e] += x^T dg,  dWu[e] += x^T du,  dx_sorted = dg Wg^T + du Wu^T
 *   dx[t] = sum_j dx_sorted[r];  dlogits through the softmax weights.
 * Weight gradients are float32 [E,H,F], [E,H,F], [E,F,H]; the rest uses the
 * layer dtype (dy, dx, dy_sorted, dx_sorted, g, u) or float32 (dtopk_w,
 * dlogits).  Dropped rows (row_of < 0) get no gradient.
 * ---------------------------------------------------------------------- */

/* dy_sorted [T*k,H] and dtopk_w [T,k] (float32) from dy [T,H]. */
moe_status_t moe_combine_backward(const moe_config_t *cfg, const void *dy,
                                  const void *y_sorted, const int32_t *row_of,
                                  const float *topk_w, void *dy_sorted,
                                  float *dtopk_w, moe_stream_t stream);

/* dlogits [T,E] (float32) from dtopk_w through the combine weights. */
moe_status_t moe_route_backward(const moe_config_t *cfg, const float *logits,
                                const int32_t *topk_idx, const float *dtopk_w,
                                float *dlogits, moe_stream_t stream);

/* dx [T,H] = sum over a token's kept rows of dx_sorted. */
moe_status_t moe_permute_backward(const moe_config_t *cfg,
                                  const void *dx_sorted, const int32_t *row_of,
                                  void *dx, moe_stream_t stream);

/* Forward GEMMs that also keep g = x Wg and u = x Wu ([T*k, F] each) for
 * the backward: h and y_sorted as moe_gmm_swiglu. */
moe_status_t moe_gmm_swiglu_saved(const moe_config_t *cfg,
                                  const void *x_sorted,
                                  const int32_t *group_offsets,
                                  const void *w_gate, const void *w_up,
                                  const void *w_down, void *g, void *u,
                                  void *h, void *y_sorted,
                                  int32_t *status_word, moe_stream_t stream);

/* The steps of the FFN backward one kernel each (the compositions above
 * and below chain them).  Rows of group e use the weights of expert e;
 * only the group_offsets[E] rows are read and written.  n_groups = 0 and
 * group_expert = NULL mean the E experts' own groups; otherwise n_groups
 * row groups (group_offsets [n_groups+1]) whose group g computes with the
 * weights of expert group_expert[g] (device, [n_groups]): the virtual groups
 * of moe_plan_duplication, a duplicate's weight gradient adding into its
 * expert's.
 *
 * GEMM1 + SwiGLU of the forward that also keeps g = x Wg and u = x Wu
 * ([T*k, F] each, layer dtype); h as moe_gmm_gate_up. */
moe_status_t moe_gmm_gate_up_saved(const moe_config_t *cfg,
                                   int32_t n_groups,
                                   const int32_t *group_expert,
                                   const void *x_sorted,
                                   const int32_t *group_offsets,
                                   const void *w_gate, const void *w_up,
                                   void *g, void *u, void *h,
                                   int32_t *status_word, moe_stream_t stream);

/* dh = dy_sorted Wd^T, then dg = dh * u * silu'(g) and du = dh * silu(g)
 * ([T*k, F] each), silu'(z) = s(z) (1 + z (1 - s(z))), s the logistic. */
moe_status_t moe_gmm_down_dgrad(const moe_config_t *cfg, int32_t n_groups,
                                const int32_t *group_expert,
                                const int32_t *group_offsets,
                                const void *w_down, const void *g,
                                const void *u, const void *dy_sorted,
                                void *dg, void *du, int32_t *status_word,
                                moe_stream_t stream);

/* dx_sorted = dg Wg^T + du Wu^T ([T*k, H]). */
moe_status_t moe_gmm_gate_up_dgrad(const moe_config_t *cfg,
                                   int32_t n_groups,
                                   const int32_t *group_expert,
                                   const int32_t *group_offsets,
                                   const void *w_gate, const void *w_up,
                                   const void *dg, const void *du,
                                   void *dx_sorted, int32_t *status_word,
                                   moe_stream_t stream);

/* One row range of the weight-gradient reduction: its groups' rows are
 * first_row + group_offsets[e] .. first_row + group_offsets[e+1] of the
 * row buffers (group_offsets: device, [E+1]). */
typedef struct {
  const int32_t *group_offsets;
  int32_t first_row;
} moe_row_segment_t;

/* Weight gradients summed over n_segments row ranges (a host array; e.g.
 * one per chunk of the fallback, so that an expert's gradient over all
 * chunks is accumulated on chip and written once), over the rows of
 * expert e:
 *   gate_up: dWg[e] (+)= x^T dg,  dWu[e] (+)= x^T du   ([E,H,F] float32)
 *   down:    dWd[e] (+)= h^T dy_sorted                 ([E,F,H] float32)
 * The row buffers have rows_total rows.  accumulate: a set of flags.
 * Without MOE_WGRAD_ACCUMULATE every expert's gradient is overwritten
 * (zeros for experts without rows); with it the gradients are added into.
 * MOE_WGRAD_ROWS16 states that every group holds a multiple of 16 rows in
 * every segment (as in the layout moe_regroup_rows writes, whose pad rows
 * are zero): bf16 layers whose gradient has a multiple of 256 rows (H for
 * gate_up, F for down, with H % 256 == 0) then take a two-SM tensor-core
 * kernel.  If the statement is false, that kernel raises MOE_DEV_UNALIGNED
 * in status_word and leaves the gradients it would have written as they
 * were (those of experts without rows still zeroed). */
#define MOE_WGRAD_ACCUMULATE 1
#define MOE_WGRAD_ROWS16 2
moe_status_t moe_gmm_gate_up_wgrad(const moe_config_t *cfg,
                                   int32_t n_groups,
                                   const int32_t *group_expert,
                                   const moe_row_segment_t *segments,
                                   int32_t n_segments, int64_t rows_total,
                                   const void *x_sorted, const void *dg,
                                   const void *du, float *dw_gate,
                                   float *dw_up, int32_t accumulate,
                                   int32_t *status_word, moe_stream_t stream);
moe_status_t moe_gmm_down_wgrad(const moe_config_t *cfg, int32_t n_groups,
                                const int32_t *group_expert,
                                const moe_row_segment_t *segments,
                                int32_t n_segments, int64_t rows_total,
                                const void *h, const void *dy_sorted,
                                float *dw_down, int32_t accumulate,
                                int32_t *status_word, moe_stream_t stream);

/* Regroups the rows of several row ranges (the passes of a layer backward)
 * for the weight-gradient GEMMs: group e of the output holds, in range
 * order, e's rows from every range, starts on a 16-row boundary, and its pad
 * rows up to the next boundary are zero, so the GEMMs see one row range per
 * expert and whole K=16 steps.  Copies x_sorted [.,H], dg, du, h [.,F] and
 * dy_sorted [.,H] (layer dtype) into the *_out buffers of rows_out rows;
 * out_offsets (device, [E+1]) receives the new group offsets.  rows_out
 * must be at least T*k + 16*(E + S*redundant_slots) (cfg->T: the tokens
 * of all ranges together);
 * 1 <= n_segments <= 64.  The source ranges must lie inside the source
 * buffers; a row of the output that no range fills is zero.  n_groups: the
 * groups of the ranges' offsets (0: E; else the virtual groups of
 * moe_plan_duplication, E + S*redundant_slots).  w_row (optional, device
 * float32, indexed by source row; bf16 only): dy_sorted holds unscaled rows
 * (moe_combine_backward_rows) and each is written times its row's weight,
 * rounded to bf16 -- the rows moe_combine_backward would have produced. */
moe_status_t moe_regroup_rows(const moe_config_t *cfg, int32_t n_groups,
                              const moe_row_segment_t *segments,
                              int32_t n_segments, int64_t rows_out,
                              const void *x_sorted, const void *dg,
                              const void *du, const void *h,
                              const void *dy_sorted, void *x_out,
                              void *dg_out, void *du_out, void *h_out,
                              void *dy_out, int32_t *out_offsets,
                              const float *w_row, moe_stream_t stream);

/* The split form of the combine backward that moe_layer_backward uses (bf16;
 * "Support moe_dropless_fallback=layer on the ragged all-to-all MoE path",
 * pull request 5920, section How: the backward recomputes each pass's
 * forward).  A combine weight's gradient is dy[t] . y_e(x_t) = dy[t] .
 * (h Wd) = (dy[t] Wd^T) . h, and dy[t] Wd^T is what the down-projection
 * dgrad computes, so the pass needs no recomputed y_sorted:
 *   moe_combine_backward_rows: dy_rows [T*k, H] (layer dtype) row r = dy[t]
 *     unscaled, w_row [T*k] float32 row r = topk_w[t, j], for every kept
 *     row r = row_of[t, j] (other rows untouched);
 *   moe_gmm_down_dgrad_rows: as moe_gmm_down_dgrad on the unscaled rows,
 *     with dh = w_row[r] * (dy_rows Wd^T)[r] in the SwiGLU backward, and
 *     row_dot [T*k, moe_row_dot_parts(cfg)] float32: entry (r, q) = the
 *     dot of (dy_rows Wd^T)[r] with h[r] over the q-th column tile of F
 *     (h [T*k, F] from the forward);
 *   moe_combine_weight_grad: dtopk_w [T, k] float32 = the sum over q, in
 *     order, of row_dot[row_of[t, j], q] (0 for a dropped pick);
 *   moe_regroup_rows with w_row scales the rows for dWd.
 * Errors as moe_combine_backward and moe_gmm_down_dgrad; float32 layers:
 * MOE_ERR_UNSUPPORTED for moe_gmm_down_dgrad_rows. */
int32_t moe_row_dot_parts(const moe_config_t *cfg);
moe_status_t moe_combine_backward_rows(const moe_config_t *cfg,
                                       const void *dy, const int32_t *row_of,
                                       const float *topk_w, void *dy_rows,
                                       float *w_row, moe_stream_t stream);
moe_status_t moe_gmm_down_dgrad_rows(const moe_config_t *cfg,
                                     int32_t n_groups,
                                     const int32_t *group_expert,
                                     const int32_t *group_offsets,
                                     const void *w_down, const void *g,
                                     const void *u, const void *h,
                                     const void *dy_rows, const float *w_row,
                                     void *dg, void *du, float *row_dot,
                                     int32_t *status_word,
                                     moe_stream_t stream);
moe_status_t moe_combine_weight_grad(const moe_config_t *cfg,
                                     const int32_t *row_of,
                                     const float *row_dot, float *dtopk_w,
                                     moe_stream_t stream);

/* Backward of the grouped SwiGLU FFN (down dgrad, gate/up dgrad, then
 * both weight gradients over one row range).  accumulate != 0 adds the
 * weight
 * gradients into dw_* (float32), 0 overwrites them (every expert, also
 * those without rows).  workspace: moe_workspace_bytes(cfg,
 * MOE_WS_GMM_BACKWARD) (dg and du). */
moe_status_t moe_gmm_swiglu_backward(const moe_config_t *cfg,
                                     const void *x_sorted,
                                     const int32_t *group_offsets,
                                     const void *w_gate, const void *w_up,
                                     const void *w_down, const void *g,
                                     const void *u, const void *h,
                                     const void *dy_sorted, void *dx_sorted,
                                     float *dw_gate, float *dw_up,
                                     float *dw_down, int32_t accumulate,
                                     int32_t *status_word, void *workspace,
                                     size_t workspace_bytes,
                                     moe_stream_t stream);

/* The whole layer's backward (recomputing its forward, as the chunked
 * fallback does), for the mode given (as moe_layer): dx [T,H], dlogits
 * [T,E] float32, dw_* float32 (overwritten).  info as moe_layer.
 * workspace: moe_workspace_bytes(cfg, MOE_WS_LAYER_BACKWARD). */
moe_status_t moe_layer_backward(const moe_config_t *cfg, const void *x,
                                const float *logits, const void *w_gate,
                                const void *w_up, const void *w_down,
                                const void *dy, void *dx, float *dlogits,
                                float *dw_gate, float *dw_up, float *dw_down,
                                moe_mode_t mode, moe_layer_info_t *info,
                                int32_t *status_word, void *workspace,
                                size_t workspace_bytes, moe_stream_t stream);

/* ----------------------------------------------------------------------
 * Expert parallelism across ranks: the rank-local steps around the two
 * exchanges of the ragged all-to-all path ("Support
 * moe_dropless_fallback=layer on the ragged all-to-all MoE path", MaxText
 * pull request 5920, sections Why, How, Tests; "Moe dynamic redundancy",
 * pull request 4760, review of ra2a_dedup_and_route: each token is sent to
 * a destination once and expanded there; "MoE ring-of-experts ...", pull
 * request 4969, section What: the ring variant).  The exchanges themselves
 * are the caller's (NCCL, torch.distributed, or copies between logical
 * ranks of one GPU).  Ranks are the shards: with cfg->S = ranks, rank d
 * owns experts [d*E/S, (d+1)*E/S).  A pass on a source rank:
 *   moe_permute_tables + moe_permute_scatter (x_sorted NULL), cfg->S =
 *   ranks: the dest-major dedup sets uniq_offsets [S+1], uniq_tokens;
 *   moe_ep_dispatch_pack: the send rows and their slots;
 *   exchange 1 (rows uniq_offsets[d+1]-uniq_offsets[d] to rank d);
 * on the receiving rank, with cfg->E = E/S (its experts), cfg->k =
 * min(k, E/S) and T = rows received:
 *   moe_permute (uncapped) on recv_idx, moe_gmm_*, moe_combine with
 *   recv_w: one partial output row per received row;
 *   exchange 2 (the partial rows back to their sources);
 * and on the source: moe_ep_return_map + moe_permute_backward (cfg->k = S
 * ranks) add the returned rows into y.
 *
 * moe_ep_check -- the global overflow check from shard_counts [S] (device),
 * each shard's receive count summed over the source ranks (an all-reduce of
 * moe_check_overflow's shard_counts); cfg->T = the tokens of all ranks, so
 * C is the single-device capacity of the ranks' batches together.  Outputs
 * as moe_check_overflow. */
moe_status_t moe_ep_check(const moe_config_t *cfg, const int32_t *shard_counts,
                          int32_t *overflow_flag, float *required_factor,
                          int32_t *capacity, moe_stream_t stream);

/* moe_ep_dispatch_pack -- a source rank's send (cfg->T = its tokens of the
 * pass, cfg->S = ranks).  For every dedup row i < uniq_offsets[S] (row i of
 * destination d, token t = uniq_tokens[i]):
 *   x_send   out [T*min(k,S), H] dtype: row i = x[t]
 *   send_idx out [T*min(k,S), kk] int32, kk = min(k, E/S): the picks of t
 *            that rank d owns, in pick order, as topk_idx[t,j] - d*E/S,
 *            then -1 in the remaining slots
 *   send_w   out [T*min(k,S), kk] float32: their combine weights, then 0
 * Rows past uniq_offsets[S] are not written.  The receiver runs its pass
 * with cfg->k = kk and cfg->E = E/S. */
moe_status_t moe_ep_dispatch_pack(const moe_config_t *cfg, const void *x,
                                  const int32_t *topk_idx,
                                  const float *topk_w,
                                  const int32_t *uniq_offsets,
                                  const int32_t *uniq_tokens, void *x_send,
                                  int32_t *send_idx, float *send_w,
                                  moe_stream_t stream);

/* moe_ep_return_map -- row_of_ret [T, S] int32: the send row of token t
 * bound for rank d, or -1; with it moe_permute_backward (cfg->k = S, unit
 * weights) adds the rows the destinations return into y [T, H]. */
moe_status_t moe_ep_return_map(const moe_config_t *cfg,
                               const int32_t *uniq_offsets,
                               const int32_t *uniq_tokens,
                               int32_t *row_of_ret, moe_stream_t stream);

/* moe_ep_localize -- the ring variant: local_idx [T, kk] (kk = min(k,
 * n_local)) = the picks of token t in [first_expert, first_expert +
 * n_local), in pick order, as topk_idx - first_expert, then -1; local_w
 * [T, kk] their weights, then 0. */
moe_status_t moe_ep_localize(const moe_config_t *cfg, const int32_t *topk_idx,
                             const float *topk_w, int32_t first_expert,
                             int32_t n_local, int32_t *local_idx,
                             float *local_w, moe_stream_t stream);

/* moe_ep_delocalize -- the backward of the ring variant ("MoE
 * ring-of-experts ...", pull request 4969, section What: the backward of
 * the combine's reduce-scatter and of the tokens' all-gather) and of the EP
 * layer ("Support moe_dropless_fallback=layer on the ragged all-to-all MoE
 * path", pull request 5920, section Tests: gradients as the dropless
 * model's): the transpose of moe_ep_localize and of the slots of
 * moe_ep_dispatch_pack.  For each token t with local row r (r =
 * row_of[t * row_stride] when row_of is given, device int32, e.g. one
 * destination's column of moe_ep_return_map's [T, S] map with row_stride =
 * S; else r = t; r < 0 skips t), the q-th pick of t in [first_expert,
 * first_expert + n_local) (pick order) gets v[t, j] = local_v[r, q]
 * (local_v [rows, kk] float32, kk = min(k, n_local)); v [T, k] float32
 * keeps its value at every other pick, so the calls for all ranks together
 * fill every pick once.  Used for the gradient of the combine weights,
 * which each pick receives from the rank that owns its expert.  Errors:
 * expert range outside [0, E), row_stride < 1 with a map, pointers not
 * 4-byte aligned. */
moe_status_t moe_ep_delocalize(const moe_config_t *cfg,
                               const int32_t *topk_idx, int32_t first_expert,
                               int32_t n_local, const int32_t *row_of,
                               int32_t row_stride, const float *local_v,
                               float *v, moe_stream_t stream);

/* moe_ep_sum_partials -- the ring variant's reduce: y [T, H] = sum over
 * q < n_parts of parts[q] ([n_parts, T, H], layer dtype), accumulated in
 * float32 in part order and rounded once. */
moe_status_t moe_ep_sum_partials(const moe_config_t *cfg, int32_t n_parts,
                                 const void *parts, void *y,
                                 moe_stream_t stream);

/* ----------------------------------------------------------------------
 * Host-side queries (no GPU work).
 * ---------------------------------------------------------------------- */
typedef enum {
  MOE_WS_PERMUTE = 0,       /* moe_permute                              */
  MOE_WS_CHUNKED = 1,       /* moe_layer_dropless_chunked               */
  MOE_WS_LAYER = 2,         /* moe_layer                                */
  MOE_WS_GMM_BACKWARD = 3,  /* moe_gmm_swiglu_backward                  */
  MOE_WS_LAYER_BACKWARD = 4 /* moe_layer_backward                       */
} moe_ws_kind_t;

/* Workspace bytes an entry point needs for cfg (0 for an invalid cfg). */
size_t moe_workspace_bytes(const moe_config_t *cfg, moe_ws_kind_t which);

/* Validates cfg alone: MOE_OK or the reason it is rejected. */
moe_status_t moe_validate_config(const moe_config_t *cfg);

/* C = floor(factor*T*k/S) capped at T*k, or -1 when uncapped [PR5920 Why]. */
int64_t moe_capacity_rows(const moe_config_t *cfg);

/* Token count of each fallback chunk and the number of chunks. */
int32_t moe_chunk_tokens(const moe_config_t *cfg);
int32_t moe_num_chunks(const moe_config_t *cfg);

/* Which bf16 grouped-GEMM kernel a launch takes for n_groups row groups (0:
 * the E experts' own) holding at most rows_bound rows (<= 0: T*k): the
 * one-CTA kernel (128-row tiles, two accumulators so that a tile's epilogue
 * overlaps the next tile's MMAs) or, for GEMM2 when H % 256 == 0 and the
 * groups average at least 512 rows, the two-SM CTA-pair kernel
 * (tcgen05.mma.cta_group::2, 256-row tiles).  Both give the same bits for a
 * row.  moe_gmm_* calls use rows_bound = T*k; moe_layer's capped pass uses
 * min(T*k, S*C).  Returns bit 1 (GEMM2 on the pair kernel); bit 0 (once
 * GEMM1 on a pair kernel) is never set: GEMM1 + SwiGLU always runs on the
 * one-CTA kernel.  0 for the one-CTA kernels or an fp32 layer, -1 for an
 * invalid cfg or n_groups. */
int32_t moe_gmm_kernel_choice(const moe_config_t *cfg, int32_t n_groups,
                              int64_t rows_bound);

/* Static text for a status code. */
const char *moe_status_string(moe_status_t status);

/* For tests of failure detection only: with fills >= 0 the TMA producers of
 * the bf16 GEMM, of the router's cluster form and of the two-SM weight
 * gradient stop after that many pipeline-stage fills, so the MMA warp's
 * bounded wait runs out (about 2 s): the kernel then sets MOE_DEV_TIMEOUT in
 * the status word, stops its other roles, drains its copies and MMAs, frees
 * its tensor memory and returns, and the CUDA context stays usable.  -1
 * restores normal operation.  Process-wide; not for production use. */
void moe_test_stall_gemm_producer(int64_t fills);

#ifdef __cplusplus
}
#endif
#endif /* MOE_GB300_H */
