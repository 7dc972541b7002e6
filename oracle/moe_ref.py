"""Float64 CPU oracle for the MoE layer's token dispatch and expert compute.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the tests, the smoke check in
``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may import or run
anything in this package.  It shares no code with the CUDA library and never
imports it; the GPU path never imports this.

Sources.  Three MaxText pull-request pages describe the method:

* "Support moe_dropless_fallback=layer on the ragged all-to-all MoE path"
  (MaxText pull request 5920), sections "Why", "How", "Shortcomings", "Tests".
  Cited below as [PR5920 <section>].
* "Moe dynamic redundancy" (MaxText pull request 4760), review comments on
  ``ra2a_dedup_and_route`` and the Zipf data generator.  Cited as
  [PR4760 review <topic>].
* "MoE ring-of-experts: TC Pallas ring all-gather for the combine backward +
  x_sorted remat save" (MaxText pull request 4969), section "What".  Cited
  as [PR4969 What].

Where the pages leave a step open, the reading taken is stated at the step
(marked READING).  Every function is plain: Python
loops where the order of things is the semantics, ``numpy.matmul`` for the
dense products of the expert FFN, float64 throughout.

Notation: T tokens, H hidden, E experts, k experts per token, F expert FFN
width, S logical expert-parallel shards of E/S consecutive experts each.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Callable, Optional

import numpy as np

INT = np.int64


# ---------------------------------------------------------------------------
# Step 0: router logits.  [PR5920 How]: the check works "from the router's
# top-k", i.e. on the router's scores of each token for each expert.  The
# pages do not spell the router out; READING: the scores are a dense
# projection of the token onto the experts, logits = x Wr with Wr [H, E],
# plus an optional per-(token, expert) offset (an expert bias and/or
# routing noise; the synthetic workloads put their popularity law there).
# ---------------------------------------------------------------------------
def router_logits(x: np.ndarray, w_router: np.ndarray,
                  offset: Optional[np.ndarray] = None) -> np.ndarray:
    """logits [T, E] = x [T, H] @ w_router [H, E] (+ offset [T, E]), in
    float64."""
    x = np.asarray(x, dtype=np.float64)
    w = np.asarray(w_router, dtype=np.float64)
    out = np.matmul(x, w)
    if offset is not None:
        out = out + np.asarray(offset, dtype=np.float64)
    return out


# ---------------------------------------------------------------------------
# Step 1: router top-k and combine weights.
# [PR5920 How]: the overflow check is computed "from the router's top-k";
# route() is the function that produces it.  The pages never say how the
# combine weights are formed from the router scores.
# READING: weights are the softmax over all E logits, read at the chosen
# experts (not renormalised); with renorm=True they are the softmax over the
# k chosen logits.  Ties in the top-k go to the lower expert index.  A logit
# that is NaN or +-inf ranks as -inf and contributes exp(-inf) = 0.
# ---------------------------------------------------------------------------
def clean_logit(v: float) -> float:
    """Non-finite logits rank as -inf (READING)."""
    return v if math.isfinite(v) else -math.inf


def topk_one_token(row, k: int):
    """Top-k of one token's logits.

    Descending logit; equal logits are ordered by ascending expert index, so
    the order is total and the selected set is unique.
    """
    E = len(row)
    keyed = [(-clean_logit(float(row[e])), e) for e in range(E)]
    keyed.sort()
    return [e for _, e in keyed[:k]]


def softmax_f64(values):
    """exp(v - max) / sum, float64, over finite entries; all -inf -> zeros."""
    vals = [clean_logit(float(v)) for v in values]
    finite = [v for v in vals if v != -math.inf]
    if not finite:
        return [0.0] * len(vals)
    m = max(finite)
    ex = [math.exp(v - m) if v != -math.inf else 0.0 for v in vals]
    s = sum(ex)
    return [v / s for v in ex]


def route(logits: np.ndarray, k: int, renorm: bool = False):
    """Router top-k: returns (topk_idx [T,k] int, topk_w [T,k] f64, nonfinite).

    ``nonfinite`` is True when any logit was NaN or infinite (the GPU path
    reports that as a status code; the ranking rule is the same).
    """
    logits = np.asarray(logits)
    T, E = logits.shape
    if not (1 <= k <= E):
        raise ValueError("need 1 <= k <= E")
    idx = np.zeros((T, k), dtype=INT)
    w = np.zeros((T, k), dtype=np.float64)
    nonfinite = bool(not np.all(np.isfinite(logits)))
    for t in range(T):
        row = logits[t]
        chosen = topk_one_token(row, k)
        idx[t] = chosen
        if renorm:
            p = softmax_f64([row[e] for e in chosen])
            w[t] = p
        else:
            p = softmax_f64(row)
            w[t] = [p[e] for e in chosen]
    return idx, w, nonfinite


# ---------------------------------------------------------------------------
# Step 2: counts.  Per-expert row counts are the grouped-GEMM group sizes
# ([PR4760 review on get_gmm_for_local_experts]: group_sizes per expert);
# per-shard receive counts sum them over each shard's expert range
# (experts_per_rank consecutive experts per shard, [PR4760 review on
# plan_expert_duplication]).
# ---------------------------------------------------------------------------
def expert_counts(topk_idx: np.ndarray, E: int) -> np.ndarray:
    c = np.zeros(E, dtype=INT)
    for e in np.asarray(topk_idx).reshape(-1):
        c[int(e)] += 1
    return c


def exclusive_scan(v) -> np.ndarray:
    out = np.zeros(len(v) + 1, dtype=INT)
    run = 0
    for i, x in enumerate(v):
        out[i] = run
        run += int(x)
    out[len(v)] = run
    return out


def shard_counts(counts: np.ndarray, S: int) -> np.ndarray:
    E = len(counts)
    if E % S:
        raise ValueError("E must be a multiple of S")
    Es = E // S
    r = np.zeros(S, dtype=INT)
    for s in range(S):
        for e in range(s * Es, (s + 1) * Es):
            r[s] += int(counts[e])
    return r


# ---------------------------------------------------------------------------
# Step 3: capacity and the overflow check.
# [PR5920 Why]: with ragged_buffer_factor > 0 each shard's receive buffer is
# capped at factor x balanced and rows past it are dropped; with -1 there is
# no cap.  [PR5920 How]: the check asks whether any shard would receive more
# than its buffer.  READING: the unit is routed rows (token, slot) because the
# check works from the top-k; balanced B = T*k/S; C = floor(factor*T*k/S)
# computed in double from the float32 factor, capped at T*k (no shard can
# hold more rows than exist); factor <= 0 means uncapped.  The comparison is
# strict: a shard overflows when r_s > C.
# ---------------------------------------------------------------------------
def capacity(T: int, k: int, S: int, factor: float) -> Optional[int]:
    f = float(np.float32(factor))
    if f <= 0.0:
        return None
    c = math.floor(f * T * k / S)
    return min(c, T * k)


def overflow_flag(r: np.ndarray, C: Optional[int]) -> bool:
    if C is None:
        return False
    return any(int(x) > C for x in r)


def required_factor(r: np.ndarray, T: int, k: int) -> float:
    """max_s r_s / balanced: the factor that would have avoided overflow
    (the quantity log_required_ragged_buffer_factor reports, [PR5920
    Shortcomings])."""
    S = len(r)
    if T * k == 0:
        return 0.0
    return max(int(x) for x in r) * S / (T * k)


# ---------------------------------------------------------------------------
# Step 4: expert-sorted permute with capped drop and per-shard dedup.
# The routed rows are sorted by expert for the grouped GEMM ([PR4969 What]:
# x_sorted is the expert-sorted MoE input).  READING: the order is stable by
# (expert, token).  Capped drop [PR5920 Why] "silently dropped": READING: the
# rows of one shard keep their (expert, token) order and a row is dropped iff
# its rank inside its shard is >= C.  Dedup [PR4760 review on
# ra2a_dedup_and_route]: each token is sent once per shard and expanded to its
# per-expert rows by expand_indices; the review requires that nothing be
# truncated.  READING: U_s is the ascending set of tokens with at least one
# KEPT row in shard s.
# ---------------------------------------------------------------------------
@dataclass
class Permutation:
    sorted_token: np.ndarray      # [R_kept] token of each kept sorted row
    sorted_slot: np.ndarray       # [R_kept] slot j of each kept sorted row
    row_of: np.ndarray            # [T,k] sorted row of (t, j), -1 if dropped
    group_offsets: np.ndarray     # [E+1] kept rows per expert, scanned
    uniq_offsets: np.ndarray      # [S+1] scanned |U_s|
    uniq_tokens: np.ndarray       # [sum |U_s|] U_0 ++ U_1 ++ ...
    expand_idx: np.ndarray        # [R_kept] row -> position in uniq_tokens
    n_dropped: int
    dropless_offsets: np.ndarray  # [E+1] scan of all counts (before drops)


def permute_indices(topk_idx: np.ndarray, E: int, S: int,
                    C: Optional[int]) -> Permutation:
    topk_idx = np.asarray(topk_idx)
    T, k = topk_idx.shape
    Es = E // S
    # every routed row with its sort key (expert, token); a token never picks
    # one expert twice, so the key is unique
    rows = []
    for t in range(T):
        for j in range(k):
            rows.append((int(topk_idx[t, j]), t, j))
    rows.sort()
    counts = expert_counts(topk_idx, E)
    dropless_offsets = exclusive_scan(counts)

    kept = []
    rank_in_shard = [0] * S
    for (e, t, j) in rows:
        s = e // Es
        if C is None or rank_in_shard[s] < C:
            kept.append((e, t, j))
        rank_in_shard[s] += 1
    n_dropped = len(rows) - len(kept)

    kept_counts = np.zeros(E, dtype=INT)
    row_of = -np.ones((T, k), dtype=INT)
    sorted_token = np.zeros(len(kept), dtype=INT)
    sorted_slot = np.zeros(len(kept), dtype=INT)
    for r, (e, t, j) in enumerate(kept):
        kept_counts[e] += 1
        row_of[t, j] = r
        sorted_token[r] = t
        sorted_slot[r] = j
    group_offsets = exclusive_scan(kept_counts)

    uniq_sets = [set() for _ in range(S)]
    for (e, t, j) in kept:
        uniq_sets[e // Es].add(t)
    uniq_lists = [sorted(u) for u in uniq_sets]
    uniq_offsets = exclusive_scan([len(u) for u in uniq_lists])
    uniq_tokens = np.array([t for u in uniq_lists for t in u], dtype=INT)
    pos_in_shard = [{t: i for i, t in enumerate(u)} for u in uniq_lists]
    expand_idx = np.zeros(len(kept), dtype=INT)
    for r, (e, t, j) in enumerate(kept):
        s = e // Es
        expand_idx[r] = uniq_offsets[s] + pos_in_shard[s][t]
    return Permutation(sorted_token, sorted_slot, row_of, group_offsets,
                       uniq_offsets, uniq_tokens, expand_idx, n_dropped,
                       dropless_offsets)


def gather_rows(x: np.ndarray, sorted_token: np.ndarray) -> np.ndarray:
    """x_sorted[r] = x[sorted_token[r]]."""
    out = np.zeros((len(sorted_token), x.shape[1]), dtype=np.float64)
    for r, t in enumerate(sorted_token):
        out[r] = x[int(t)]
    return out


# ---------------------------------------------------------------------------
# Step 5: expert FFN.  The pages name the expert weights (w0 of shape
# [E, H, H_ffn], [PR4760 review on the dynamic weight manager]) and a grouped
# matmul over experts with ragged group sizes (megablox / gmm); the SwiGLU
# form is the one the workloads fix: h = silu(x Wg) * (x Wu), y = h Wd with
# silu(z) = z / (1 + exp(-z)).  Layout READING: Wg, Wu are [E, H, F]; Wd is
# [E, F, H].  Float64, no intermediate rounding.
# ---------------------------------------------------------------------------
def silu(z: np.ndarray) -> np.ndarray:
    z = np.asarray(z, dtype=np.float64)
    return z / (1.0 + np.exp(-z))


ExpertWeights = Callable[[int], tuple]


def dense_weights(w_gate, w_up, w_down) -> ExpertWeights:
    """Accessor over in-memory [E,H,F]/[E,H,F]/[E,F,H] arrays."""
    def get(e):
        return (np.asarray(w_gate[e], dtype=np.float64),
                np.asarray(w_up[e], dtype=np.float64),
                np.asarray(w_down[e], dtype=np.float64))
    return get


def expert_ffn(x_rows: np.ndarray, wg, wu, wd):
    """SwiGLU FFN of one expert over a block of rows.
    Returns (h [rows,F], y [rows,H])."""
    x_rows = np.asarray(x_rows, dtype=np.float64)
    g = np.matmul(x_rows, wg)
    u = np.matmul(x_rows, wu)
    h = silu(g) * u
    return h, np.matmul(h, wd)


def grouped_ffn(x_sorted: np.ndarray, group_offsets: np.ndarray,
                weights: ExpertWeights):
    """Grouped GEMM over experts: rows [off[e], off[e+1]) use expert e.
    Returns (h [R,F], y_sorted [R,H])."""
    E = len(group_offsets) - 1
    R = int(group_offsets[E])
    h_all = None
    y_all = np.zeros((R, x_sorted.shape[1]), dtype=np.float64)
    for e in range(E):
        a, b = int(group_offsets[e]), int(group_offsets[e + 1])
        if a == b:
            continue
        wg, wu, wd = weights(e)
        h, y = expert_ffn(x_sorted[a:b], wg, wu, wd)
        if h_all is None:
            h_all = np.zeros((R, h.shape[1]), dtype=np.float64)
        h_all[a:b] = h
        y_all[a:b] = y
    return h_all, y_all


# ---------------------------------------------------------------------------
# Step 6: weighted combine (unpermute).  Each token's output is the sum over
# its k slots of weight x expert output ([PR4969 What]: the combine is a
# reduce over expert outputs, a psum_scatter in the ring variant).  A dropped
# row contributes nothing.  Summed in slot order j = 0..k-1.
# ---------------------------------------------------------------------------
def combine(y_sorted: np.ndarray, row_of: np.ndarray, topk_w: np.ndarray,
            H: int) -> np.ndarray:
    T, k = row_of.shape
    y = np.zeros((T, H), dtype=np.float64)
    for t in range(T):
        for j in range(k):
            r = int(row_of[t, j])
            if r >= 0:
                y[t] += float(topk_w[t, j]) * y_sorted[r]
    return y


# ---------------------------------------------------------------------------
# Step 7: the chunked dropless fallback.
# [PR5920 How]: on overflow, the layer runs over n sequence chunks, each with
# the worst-case (force_dropless) buffer, and n is chosen so that this buffer
# is no larger than the capped one.  [PR5920 Shortcomings]: about n x slower,
# 8x for EP16 at factor 2.  READING: one source on one GPU can put at most
# min(k, E/S) rows per token into one shard, so a chunk of c tokens has a
# worst case of c*min(k, E/S) rows; the chunk is the largest c with
# c*min(k, E/S) <= C (at least 1 token) and n = ceil(T / c).  An explicit
# n_chunks gives chunks of ceil(T/n) tokens.  Chunks are contiguous token
# ranges; the last may be shorter.
# ---------------------------------------------------------------------------
def chunk_plan(T: int, k: int, E: int, S: int, C: Optional[int],
               n_chunks: int = 0):
    """Returns the list of (t0, t1) token ranges of the chunked fallback."""
    if T == 0:
        return []
    if n_chunks > 0:
        c = -(-T // n_chunks)
    elif C is None:
        c = T
    else:
        worst_per_token = min(k, E // S)
        c = max(1, C // worst_per_token)
    return [(t0, min(T, t0 + c)) for t0 in range(0, T, c)]


# ---------------------------------------------------------------------------
# The layer.
# ---------------------------------------------------------------------------
@dataclass
class MoEConfig:
    T: int
    H: int
    E: int
    k: int
    F: int
    S: int
    ragged_buffer_factor: float = 2.0
    n_chunks: int = 0
    renorm: bool = False


@dataclass
class LayerResult:
    y: np.ndarray
    topk_idx: np.ndarray
    topk_w: np.ndarray
    counts: np.ndarray
    shard: np.ndarray
    C: Optional[int]
    overflow: bool
    required_factor: float
    perm: Optional[Permutation] = None
    x_sorted: Optional[np.ndarray] = None
    h: Optional[np.ndarray] = None
    y_sorted: Optional[np.ndarray] = None
    chunks: list = field(default_factory=list)


def layer_pass(cfg: MoEConfig, x, logits, weights: ExpertWeights,
               C: Optional[int], topk=None) -> LayerResult:
    """One pass: route -> counts -> permute (cap C) -> FFN -> combine."""
    x = np.asarray(x, dtype=np.float64)
    if topk is None:
        idx, w, _ = route(logits, cfg.k, cfg.renorm)
    else:
        idx, w = topk
    counts = expert_counts(idx, cfg.E)
    shard = shard_counts(counts, cfg.S)
    T = x.shape[0]
    perm = permute_indices(idx, cfg.E, cfg.S, C)
    xs = gather_rows(x, perm.sorted_token)
    h, ys = grouped_ffn(xs, perm.group_offsets, weights)
    y = combine(ys, perm.row_of, w, cfg.H)
    return LayerResult(y, idx, w, counts, shard, C, overflow_flag(shard, C),
                       required_factor(shard, T, cfg.k), perm, xs, h, ys)


def layer_capped(cfg, x, logits, weights) -> LayerResult:
    """The capped ragged path alone (no fallback): rows past C are dropped."""
    C = capacity(cfg.T, cfg.k, cfg.S, cfg.ragged_buffer_factor)
    return layer_pass(cfg, x, logits, weights, C)


def layer_dropless(cfg, x, logits, weights) -> LayerResult:
    """The uncapped (force_dropless) path."""
    return layer_pass(cfg, x, logits, weights, None)


def layer_dropless_chunked(cfg, x, logits, weights,
                           n_chunks: Optional[int] = None) -> LayerResult:
    """The chunked dropless fallback: every chunk runs uncapped."""
    x = np.asarray(x, dtype=np.float64)
    logits = np.asarray(logits)
    C = capacity(cfg.T, cfg.k, cfg.S, cfg.ragged_buffer_factor)
    plan = chunk_plan(cfg.T, cfg.k, cfg.E, cfg.S, C,
                      cfg.n_chunks if n_chunks is None else n_chunks)
    y = np.zeros((cfg.T, cfg.H), dtype=np.float64)
    idx = np.zeros((cfg.T, cfg.k), dtype=INT)
    w = np.zeros((cfg.T, cfg.k), dtype=np.float64)
    parts = []
    for (t0, t1) in plan:
        sub = MoEConfig(t1 - t0, cfg.H, cfg.E, cfg.k, cfg.F, cfg.S,
                        -1.0, 0, cfg.renorm)
        res = layer_pass(sub, x[t0:t1], logits[t0:t1], weights, None)
        y[t0:t1] = res.y
        idx[t0:t1] = res.topk_idx
        w[t0:t1] = res.topk_w
        parts.append(res)
    counts = expert_counts(idx, cfg.E)
    shard = shard_counts(counts, cfg.S)
    return LayerResult(y, idx, w, counts, shard, C, overflow_flag(shard, C),
                       required_factor(shard, cfg.T, cfg.k), chunks=parts)


def layer(cfg, x, logits, weights) -> LayerResult:
    """moe_dropless_fallback=layer [PR5920 How]: check, then the capped path
    when no shard overflows, else the chunked dropless fallback.  The flag is
    global: one overflowing shard sends the whole layer to the fallback
    [PR5920 Tests]."""
    idx, w, _ = route(logits, cfg.k, cfg.renorm)
    counts = expert_counts(idx, cfg.E)
    shard = shard_counts(counts, cfg.S)
    C = capacity(cfg.T, cfg.k, cfg.S, cfg.ragged_buffer_factor)
    if overflow_flag(shard, C):
        res = layer_dropless_chunked(cfg, x, logits, weights)
        res.overflow = True
        return res
    return layer_pass(cfg, x, logits, weights, C, topk=(idx, w))


# ---------------------------------------------------------------------------
# Per-token output for large layers: one token's output depends only on its
# own row, its routing and the weights of its k experts, so sampled tokens of
# a full-size layer can be checked one by one (dropless semantics).
# ---------------------------------------------------------------------------
def token_outputs(x_rows: np.ndarray, idx_rows: np.ndarray,
                  w_rows: np.ndarray, weights: ExpertWeights,
                  keep: Optional[np.ndarray] = None) -> np.ndarray:
    """y for a few tokens: sum_j w_j FFN_{e_j}(x).  ``keep[t, j]`` False
    skips a dropped slot.  Experts are visited in ascending order so each
    expert's weights are fetched once."""
    x_rows = np.asarray(x_rows, dtype=np.float64)
    n, k = idx_rows.shape
    out = np.zeros_like(x_rows)
    by_expert = {}
    for i in range(n):
        for j in range(k):
            if keep is None or keep[i, j]:
                by_expert.setdefault(int(idx_rows[i, j]), []).append((i, j))
    for e in sorted(by_expert):
        wg, wu, wd = weights(e)
        for (i, j) in by_expert[e]:
            _, y = expert_ffn(x_rows[i:i + 1], wg, wu, wd)
            out[i] += float(w_rows[i, j]) * y[0]
    return out


def normwise_error(got: np.ndarray, ref: np.ndarray) -> float:
    """max_i |g_i - r_i| / max_i |r_i| (the tolerance measure used by the
    parity tests; 0 when both are all zero)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = float(np.max(np.abs(ref))) if ref.size else 0.0
    num = float(np.max(np.abs(got - ref))) if ref.size else 0.0
    if den == 0.0:
        return num
    return num / den


def elementwise_error(got: np.ndarray, ref: np.ndarray,
                      floor: float = 1e-3) -> float:
    """max_i |g_i - r_i| / max(|r_i|, floor * max_j |r_j|): the largest
    relative error of any single element, with a small absolute floor so
    that elements near zero (whose relative error is meaningless) are
    measured against floor * the tensor's largest magnitude.  Reported
    beside the normwise measure; 0 when both are all zero."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if ref.size == 0:
        return 0.0
    peak = float(np.max(np.abs(ref)))
    diff = np.abs(got - ref)
    if peak == 0.0:
        return float(np.max(diff))
    den = np.maximum(np.abs(ref), floor * peak)
    return float(np.max(diff / den))


# ---------------------------------------------------------------------------
# Dynamic redundant experts.  "Moe dynamic redundancy" (MaxText pull request
# 4760), review comments: plan_expert_duplication duplicates the hottest
# not-yet-duplicated expert of the most loaded rank (r_max) into a spare slot
# (num_slots_B per rank) on an underloaded rank and diverts a fraction of its
# tokens there (reroute_fractions); the review requires that (1) tokens are
# really diverted, so the slots get non-zero group sizes, and (2) the plan
# stops when r_max has no un-duplicated expert left (has_candidate), so no
# expert is duplicated twice.  On one GPU a slot uses the same weights as
# its expert (nothing is gathered).
# READINGS: each round takes r_max = the most loaded shard (ties: lower
# index), its hottest un-duplicated expert with rows (ties: lower index),
# and r_min = the least loaded other shard with a free slot (ties: lower
# index); it stops when there is no candidate, no such shard, or no gap; it
# moves n = min(c_e, (load[r_max] - load[r_min]) // 2) rows (integer halving
# of the gap, so the fraction is n / c_e).  The duplicate takes the expert's
# LAST n rows in token order.  At most S*B rounds.
# Virtual layout: shard s owns virtual groups [s*(E_s+B), (s+1)*(E_s+B)):
# its E_s experts, then its B slots.
# ---------------------------------------------------------------------------
@dataclass
class DuplicationPlan:
    divert: np.ndarray        # [E] rows of e moved to its duplicate
    slot_of: np.ndarray       # [E] virtual group of e's duplicate, -1 if none
    group_expert: np.ndarray  # [E'] expert behind each virtual group (-1 unused)
    loads_after: np.ndarray   # [S] shard loads after the diversion
    B: int


def virtual_group_of_expert(e: int, E: int, S: int, B: int) -> int:
    Es = E // S
    return (e // Es) * (Es + B) + e % Es


def virtual_group_of_slot(s: int, b: int, E: int, S: int, B: int) -> int:
    Es = E // S
    return s * (Es + B) + Es + b


def plan_duplication(counts: np.ndarray, S: int, B: int) -> DuplicationPlan:
    counts = [int(c) for c in counts]
    E = len(counts)
    Es = E // S
    load = [sum(counts[s * Es:(s + 1) * Es]) for s in range(S)]
    dup = [False] * E
    free = [B] * S
    divert = [0] * E
    slot_of = [-1] * E
    group_expert = [-1] * (S * (Es + B))
    for e in range(E):
        group_expert[virtual_group_of_expert(e, E, S, B)] = e
    for _ in range(S * B):
        r_max = 0
        for s in range(1, S):
            if load[s] > load[r_max]:
                r_max = s
        cands = [e for e in range(r_max * Es, (r_max + 1) * Es)
                 if not dup[e] and counts[e] > 0]
        has_candidate = len(cands) > 0
        r_min = -1
        for s in range(S):
            if s != r_max and free[s] > 0:
                if r_min < 0 or load[s] < load[r_min]:
                    r_min = s
        if not has_candidate or r_min < 0 or load[r_max] <= load[r_min]:
            break
        e_star = cands[0]
        for e in cands[1:]:
            if counts[e] > counts[e_star]:
                e_star = e
        n = min(counts[e_star], (load[r_max] - load[r_min]) // 2)
        if n <= 0:
            break
        b = B - free[r_min]
        free[r_min] -= 1
        g = virtual_group_of_slot(r_min, b, E, S, B)
        dup[e_star] = True
        divert[e_star] = n
        slot_of[e_star] = g
        group_expert[g] = e_star
        load[r_max] -= n
        load[r_min] += n
    return DuplicationPlan(np.array(divert, dtype=INT),
                           np.array(slot_of, dtype=INT),
                           np.array(group_expert, dtype=INT),
                           np.array(load, dtype=INT), B)


def reroute(topk_idx: np.ndarray, plan: DuplicationPlan, E: int,
            S: int) -> np.ndarray:
    """Virtual group of every routed row (t, j): its expert's group, or the
    duplicate's slot for the expert's last divert[e] rows in token order."""
    topk_idx = np.asarray(topk_idx)
    T, k = topk_idx.shape
    counts = expert_counts(topk_idx, E)
    seen = [0] * E
    out = np.zeros_like(topk_idx, dtype=INT)
    for t in range(T):
        for j in range(k):
            e = int(topk_idx[t, j])
            keep = int(counts[e]) - int(plan.divert[e])
            if seen[e] >= keep and plan.slot_of[e] >= 0:
                out[t, j] = plan.slot_of[e]
            else:
                out[t, j] = virtual_group_of_expert(e, E, S, plan.B)
            seen[e] += 1
    return out


def mapped_weights(weights: ExpertWeights,
                   group_expert: np.ndarray) -> ExpertWeights:
    """Weights of virtual group g = weights of expert group_expert[g]."""
    return lambda g: weights(int(group_expert[g]))


def layer_redundant(cfg: MoEConfig, x, logits, weights: ExpertWeights,
                    B: int) -> LayerResult:
    """fallback=layer with dynamic redundant experts: route, plan, divert,
    then the overflow check on the virtual shard loads; capped pass over the
    virtual groups, or the chunked dropless fallback when still over."""
    idx, w, _ = route(logits, cfg.k, cfg.renorm)
    counts = expert_counts(idx, cfg.E)
    plan = plan_duplication(counts, cfg.S, B)
    vidx = reroute(idx, plan, cfg.E, cfg.S)
    G = cfg.S * (cfg.E // cfg.S + B)
    vshard = shard_counts(expert_counts(vidx, G), cfg.S)
    C = capacity(cfg.T, cfg.k, cfg.S, cfg.ragged_buffer_factor)
    if overflow_flag(vshard, C):
        res = layer_dropless_chunked(cfg, x, logits, weights)
        res.overflow = True
        return res
    x = np.asarray(x, dtype=np.float64)
    perm = permute_indices(vidx, G, cfg.S, C)
    xs = gather_rows(x, perm.sorted_token)
    h, ys = grouped_ffn(xs, perm.group_offsets,
                        mapped_weights(weights, plan.group_expert))
    y = combine(ys, perm.row_of, w, cfg.H)
    return LayerResult(y, idx, w, counts, vshard, C, False,
                       required_factor(vshard, cfg.T, cfg.k), perm, xs, h, ys)


# ---------------------------------------------------------------------------
# Backward pass.  "Support moe_dropless_fallback=layer on the ragged
# all-to-all MoE path" (MaxText pull request 5920): section Tests requires
# the fallback's outputs AND gradients to match the dropless model; section
# How: the chunked fallback recomputes one chunk at a time in the backward
# and accumulates the expert-weight gradients across chunks.  "MoE
# ring-of-experts ... x_sorted remat save" (MaxText pull request 4969),
# section What: the backward reuses the expert-sorted input and its routing
# metadata instead of re-running the dispatch.
# Gradients of the layer output y w.r.t. x, the router logits (through the
# combine weights; the top-k choice itself is piecewise constant) and the
# expert weights, given dy = dL/dy.  The chain, per routed row r = (t, j)
# of expert e (dropped rows carry no gradient):
#   dw[t,j] = <dy[t], y_sorted[r]>,   dy_sorted[r] = w[t,j] dy[t]
#   dWd[e] += h_r^T dy_sorted[r],     dh_r = dy_sorted[r] Wd[e]^T
#   dg_r = dh_r * u_r * silu'(g_r),   du_r = dh_r * silu(g_r)
#   dWg[e] += x_r^T dg_r,  dWu[e] += x_r^T du_r
#   dx_sorted[r] = dg_r Wg[e]^T + du_r Wu[e]^T,   dx[t] = sum_j dx_sorted[r]
# with silu'(z) = s(z) (1 + z (1 - s(z))), s = logistic; and for the logits
#   w = softmax(all logits) read at the chosen experts:
#     dp[e] = sum_j [idx_j = e] dw_j,  dlogits = p * (dp - <p, dp>)
#   renorm (softmax over the k chosen): dlogits[idx_j] = w_j (dw_j - sum w dw)
# ---------------------------------------------------------------------------
def silu_grad(z: np.ndarray) -> np.ndarray:
    z = np.asarray(z, dtype=np.float64)
    s = 1.0 / (1.0 + np.exp(-z))
    return s * (1.0 + z * (1.0 - s))


@dataclass
class Gradients:
    dx: np.ndarray
    dlogits: np.ndarray
    dwg: np.ndarray
    dwu: np.ndarray
    dwd: np.ndarray
    dtopk_w: np.ndarray


def route_backward(logits: np.ndarray, idx: np.ndarray, dw: np.ndarray,
                   renorm: bool) -> np.ndarray:
    logits = np.asarray(logits)
    T, E = logits.shape
    k = idx.shape[1]
    dl = np.zeros((T, E), dtype=np.float64)
    for t in range(T):
        if renorm:
            w = softmax_f64([logits[t, e] for e in idx[t]])
            dot = sum(w[j] * dw[t, j] for j in range(k))
            for j in range(k):
                dl[t, idx[t, j]] += w[j] * (dw[t, j] - dot)
        else:
            p = softmax_f64(logits[t])
            dp = [0.0] * E
            for j in range(k):
                dp[int(idx[t, j])] += float(dw[t, j])
            dot = sum(p[e] * dp[e] for e in range(E))
            for e in range(E):
                dl[t, e] = p[e] * (dp[e] - dot)
    return dl


def expert_ffn_backward(x_rows, dy_rows, wg, wu, wd):
    """Backward of one expert's SwiGLU FFN over a block of rows, given the
    gradient dy_rows of its outputs y = (silu(x Wg) * (x Wu)) Wd.
    Returns (dx_rows, (dWg, dWu, dWd))."""
    x = np.asarray(x_rows, dtype=np.float64)
    dy = np.asarray(dy_rows, dtype=np.float64)
    g = x @ wg
    u = x @ wu
    h = silu(g) * u
    dh = dy @ wd.T
    dg = dh * u * silu_grad(g)
    du = dh * silu(g)
    return dg @ wg.T + du @ wu.T, (x.T @ dg, x.T @ du, h.T @ dy)


def pass_backward_touched(cfg: MoEConfig, x, logits, weights: ExpertWeights,
                          dy, C: Optional[int], groups=None):
    """Backward of one pass (capacity C, None = uncapped) with the weights
    read one expert at a time through an accessor.  Returns (Gradients with
    dwg = dwu = dwd = None, {e: (dWg[e], dWu[e], dWd[e])} for the experts
    that received rows); every other expert's gradient is zero.

    groups = (vidx, G, group_expert): the rows are permuted over G virtual
    groups by vidx instead of over the experts (dynamic redundancy); group g
    computes with the weights of expert group_expert[g], and an expert's
    weight gradient is the sum over its groups (in group order)."""
    x = np.asarray(x, dtype=np.float64)
    dy = np.asarray(dy, dtype=np.float64)
    T, H = x.shape
    idx, w, _ = route(logits, cfg.k, cfg.renorm)
    if groups is None:
        pidx, G, gexp = idx, cfg.E, None
    else:
        pidx, G, gexp = groups
    perm = permute_indices(pidx, G, cfg.S, C)
    xs = gather_rows(x, perm.sorted_token)
    R = len(perm.sorted_token)
    F = cfg.F
    dW = {}
    ys = np.zeros((R, H))
    hs = np.zeros((R, F))
    gs = np.zeros((R, F))
    us = np.zeros((R, F))
    for grp in range(G):
        a, b = int(perm.group_offsets[grp]), int(perm.group_offsets[grp + 1])
        if a == b:
            continue
        wg, wu, wd = weights(grp if gexp is None else int(gexp[grp]))
        gs[a:b] = xs[a:b] @ wg
        us[a:b] = xs[a:b] @ wu
        hs[a:b] = silu(gs[a:b]) * us[a:b]
        ys[a:b] = hs[a:b] @ wd
    dtw = np.zeros((T, cfg.k))
    dys = np.zeros((R, H))
    for t in range(T):
        for j in range(cfg.k):
            r = int(perm.row_of[t, j])
            if r >= 0:
                dtw[t, j] = float(dy[t] @ ys[r])
                dys[r] = w[t, j] * dy[t]
    dxs = np.zeros((R, H))
    for grp in range(G):
        a, b = int(perm.group_offsets[grp]), int(perm.group_offsets[grp + 1])
        if a == b:
            continue
        e = grp if gexp is None else int(gexp[grp])
        dxs[a:b], dWe = expert_ffn_backward(xs[a:b], dys[a:b], *weights(e))
        dW[e] = dWe if e not in dW else tuple(
            acc + v for acc, v in zip(dW[e], dWe))
    dx = np.zeros((T, H))
    for t in range(T):
        for j in range(cfg.k):
            r = int(perm.row_of[t, j])
            if r >= 0:
                dx[t] += dxs[r]
    dl = route_backward(logits, idx, dtw, cfg.renorm)
    return Gradients(dx, dl, None, None, None, dtw), dW


def layer_pass_backward(cfg: MoEConfig, x, logits, w_gate, w_up, w_down,
                        dy, C: Optional[int], groups=None) -> Gradients:
    """Backward of one pass (capacity C, None = uncapped) over in-memory
    float64 weights [E,H,F], [E,H,F], [E,F,H]; dense weight gradients.
    groups: as pass_backward_touched."""
    g, dW = pass_backward_touched(cfg, x, logits,
                                  dense_weights(w_gate, w_up, w_down), dy, C,
                                  groups)
    g.dwg = np.zeros(np.shape(w_gate), dtype=np.float64)
    g.dwu = np.zeros(np.shape(w_up), dtype=np.float64)
    g.dwd = np.zeros(np.shape(w_down), dtype=np.float64)
    for e, (a, b, c) in dW.items():
        g.dwg[e], g.dwu[e], g.dwd[e] = a, b, c
    return g


def segmented_weight_grads(P, Q, segments, n_groups: int, E: int,
                           group_expert=None) -> np.ndarray:
    """Weight gradient of one expert projection row -> P row -> Q row, summed
    over row ranges: dW[e] = sum over the segments s and the groups g of
    expert e of P[rows of g in s]^T Q[rows of g in s], shape [E, cols of P,
    cols of Q].  (x, dg) gives dWg, (x, du) dWu and (h, dy_sorted) dWd.

    [PR5920 How]: the fallback's backward takes one chunk at a time and
    accumulates the expert-weight gradients over the chunks: one segment
    per chunk, given as (group_offsets [n_groups + 1], first_row), the rows
    of group g being first_row + group_offsets[g] .. first_row +
    group_offsets[g + 1].  group_expert (None: group g is expert g) maps
    the groups of a duplication plan to their experts: a duplicate's rows
    add into its expert's gradient ([PR4760 review on the dynamic weight
    manager]: the copies' gradients are summed)."""
    P = np.asarray(P, dtype=np.float64)
    Q = np.asarray(Q, dtype=np.float64)
    dW = np.zeros((E, P.shape[1], Q.shape[1]))
    for off, base in segments:
        off = np.asarray(off, dtype=INT)
        for g in range(n_groups):
            e = g if group_expert is None else int(group_expert[g])
            r0, r1 = base + int(off[g]), base + int(off[g + 1])
            dW[e] += P[r0:r1].T @ Q[r0:r1]
    return dW


def layer_backward_dropless(cfg, x, logits, w_gate, w_up, w_down, dy):
    return layer_pass_backward(cfg, x, logits, w_gate, w_up, w_down, dy, None)


def layer_backward_capped(cfg, x, logits, w_gate, w_up, w_down, dy):
    C = capacity(cfg.T, cfg.k, cfg.S, cfg.ragged_buffer_factor)
    return layer_pass_backward(cfg, x, logits, w_gate, w_up, w_down, dy, C)


def layer_backward_chunked(cfg, x, logits, w_gate, w_up, w_down, dy):
    """The chunked fallback's backward: each chunk's pass is differentiated
    on its own and the weight gradients are summed over chunks."""
    x = np.asarray(x, dtype=np.float64)
    C = capacity(cfg.T, cfg.k, cfg.S, cfg.ragged_buffer_factor)
    plan = chunk_plan(cfg.T, cfg.k, cfg.E, cfg.S, C, cfg.n_chunks)
    out = Gradients(np.zeros_like(x), np.zeros((cfg.T, cfg.E)),
                    np.zeros_like(w_gate, dtype=np.float64),
                    np.zeros_like(w_up, dtype=np.float64),
                    np.zeros_like(w_down, dtype=np.float64),
                    np.zeros((cfg.T, cfg.k)))
    for (t0, t1) in plan:
        sub = MoEConfig(t1 - t0, cfg.H, cfg.E, cfg.k, cfg.F, cfg.S, -1.0, 0,
                        cfg.renorm)
        g = layer_pass_backward(sub, x[t0:t1], np.asarray(logits)[t0:t1],
                                w_gate, w_up, w_down, np.asarray(dy)[t0:t1],
                                None)
        out.dx[t0:t1] = g.dx
        out.dlogits[t0:t1] = g.dlogits
        out.dtopk_w[t0:t1] = g.dtopk_w
        out.dwg += g.dwg
        out.dwu += g.dwu
        out.dwd += g.dwd
    return out


def layer_redundant_backward(cfg: MoEConfig, x, logits, w_gate, w_up, w_down,
                             dy, B: int) -> Gradients:
    """Backward of layer_redundant ("Moe dynamic redundancy" (MaxText pull
    request 4760), review comments: a duplicated expert's weight gradient is
    the sum of its copies' gradients, a psum across devices there and a sum
    over its virtual groups on one device).  Same plan, reroute and check as
    the forward; the capped pass over the virtual groups, or the plain
    chunked fallback when the diverted loads still overflow."""
    idx, _, _ = route(logits, cfg.k, cfg.renorm)
    counts = expert_counts(idx, cfg.E)
    plan = plan_duplication(counts, cfg.S, B)
    vidx = reroute(idx, plan, cfg.E, cfg.S)
    G = cfg.S * (cfg.E // cfg.S + B)
    vshard = shard_counts(expert_counts(vidx, G), cfg.S)
    C = capacity(cfg.T, cfg.k, cfg.S, cfg.ragged_buffer_factor)
    if overflow_flag(vshard, C):
        return layer_backward_chunked(cfg, x, logits, w_gate, w_up, w_down,
                                      dy)
    return layer_pass_backward(cfg, x, logits, w_gate, w_up, w_down, dy, C,
                               groups=(vidx, G, plan.group_expert))


# ---------------------------------------------------------------------------
# Expert parallelism across ranks.  [PR5920 Why, How]: on the ragged
# all-to-all path every device sends its tokens' rows to the devices that own
# their experts, each token once per destination, and the receiver expands a
# token to its expert rows ([PR4760 review of ra2a_dedup_and_route]:
# expand_indices, never truncated).  [PR5920 Tests]: the overflow flag is
# global, so every rank takes the same branch.  READINGS:
#  * N ranks = N shards; rank d owns experts [d*E/N, (d+1)*E/N);
#  * the check sums each shard's receive count over the source ranks and
#    takes C from the global token count (the single-device formula on the
#    ranks' batches together);
#  * the fallback's chunk count comes from that global configuration; each
#    rank splits its own tokens into n contiguous chunks of ceil(T_r/n) and
#    pass i is every rank's chunk i;
#  * with fallback=layer the capped pass runs only when no shard overflows,
#    so it drops nothing (the EP layer has no capped-only mode);
#  * the receiver groups the received rows by its local expert in
#    (expert, source rank, token) order, runs the expert FFN, and returns for
#    each received token the weighted sum of its rows' outputs (the combine,
#    split across ranks); the source adds the returns of all destinations.
# ---------------------------------------------------------------------------
@dataclass
class EPDispatch:
    """One source rank's send for one pass (dest-major)."""
    uniq_offsets: np.ndarray  # [N+1]: rows bound for each destination
    uniq_tokens: np.ndarray   # [U]: local token of each row, ascending per dest
    send_idx: np.ndarray      # [U, kk]: local experts of the row's picks
                              #          its destination owns, in pick
                              #          order, then -1; kk = min(k, E/N)
    send_w: np.ndarray        # [U, kk]: their combine weights, then 0


def ep_dispatch(topk_idx: np.ndarray, topk_w: np.ndarray, E: int,
                N: int) -> EPDispatch:
    """The dedup'd send of one rank: for each destination d, the tokens
    with at least one pick among d's experts, each once, with the local
    expert index and weight of each of its picks that d owns (a token has
    at most min(k, E/N) of them)."""
    topk_idx = np.asarray(topk_idx)
    T, k = topk_idx.shape if topk_idx.size else (0, topk_idx.shape[-1])
    Ed = E // N
    kk = min(k, Ed)
    toks, idx, w, offs = [], [], [], [0]
    for d in range(N):
        for t in range(T):
            picks = [int(e) for e in topk_idx[t]]
            if any(e // Ed == d for e in picks):
                toks.append(t)
                own = [j for j in range(k) if picks[j] // Ed == d]
                idx.append([picks[j] - d * Ed for j in own]
                           + [-1] * (kk - len(own)))
                w.append([float(topk_w[t, j]) for j in own]
                         + [0.0] * (kk - len(own)))
        offs.append(len(toks))
    return EPDispatch(np.array(offs, dtype=INT), np.array(toks, dtype=INT),
                      np.array(idx, dtype=INT).reshape(-1, kk),
                      np.array(w, dtype=np.float64).reshape(-1, kk))


def ep_expert_pass(recv_x: np.ndarray, recv_idx: np.ndarray,
                   recv_w: np.ndarray, local_weights: ExpertWeights):
    """A receiving rank: every (row, pick) with a local expert goes through
    that expert's FFN; each received row gets the weighted sum of its
    picks' outputs."""
    recv_x = np.asarray(recv_x, dtype=np.float64)
    n = recv_x.shape[0]
    out = np.zeros_like(recv_x)
    by_expert = {}
    for i in range(n):
        for j in range(recv_idx.shape[1]):
            e = int(recv_idx[i, j])
            if e >= 0:
                by_expert.setdefault(e, []).append((i, j))
    for e in sorted(by_expert):
        rows = by_expert[e]
        _, y = expert_ffn(recv_x[[i for i, _ in rows]], *local_weights(e))
        for q, (i, j) in enumerate(rows):
            out[i] += float(recv_w[i, j]) * y[q]
    return out


def ep_chunk_bounds(T_r: int, n: int, c: int):
    """Tokens [t0, t1) of rank-local chunk c of n."""
    size = -(-T_r // n) if n > 0 else 0
    t0 = min(T_r, c * size)
    return t0, min(T_r, t0 + size)


def ep_global_check(cfg: MoEConfig, N: int, routes: list):
    """The check over all ranks: each shard's receive count summed over the
    ranks' routings, against the capacity of the ranks' tokens together.
    Returns (overflow, passes)."""
    E, k = cfg.E, cfg.k
    shard = np.zeros(N, dtype=INT)
    for idx, _ in routes:
        shard += shard_counts(expert_counts(idx, E), N)
    C = capacity(cfg.T, k, N, cfg.ragged_buffer_factor)
    over = overflow_flag(shard, C)
    n = len(chunk_plan(cfg.T, k, E, N, C, cfg.n_chunks)) if over else 1
    return over, n


def ep_layer(cfg: MoEConfig, N: int, xs: list, logits: list,
             weights: ExpertWeights):
    """The layer with fallback=layer over N ranks (cfg.T = all ranks'
    tokens, cfg.S = N).  Returns (per-rank outputs, overflow, passes)."""
    E, k, H = cfg.E, cfg.k, cfg.H
    Ed = E // N
    Ts = [np.asarray(x).shape[0] for x in xs]
    if sum(Ts) != cfg.T or cfg.S != N:
        raise ValueError("cfg.T must be the ranks' tokens and cfg.S = N")
    routes = [route(L, k, cfg.renorm)[:2] for L in logits]
    over, n = ep_global_check(cfg, N, routes)
    ys = [np.zeros((T_r, H)) for T_r in Ts]
    xs = [np.asarray(x, dtype=np.float64) for x in xs]
    for c in range(n):
        bounds = [ep_chunk_bounds(Ts[r], n, c) for r in range(N)]
        sends = [ep_dispatch(routes[r][0][t0:t1], routes[r][1][t0:t1], E, N)
                 for r, (t0, t1) in enumerate(bounds)]
        for d in range(N):
            parts = []
            for q in range(N):
                a, z = int(sends[q].uniq_offsets[d]), \
                    int(sends[q].uniq_offsets[d + 1])
                parts.append((q, sends[q].uniq_tokens[a:z],
                              sends[q].send_idx[a:z], sends[q].send_w[a:z]))
            recv_x = np.concatenate(
                [xs[q][bounds[q][0] + tok] for q, tok, _, _ in parts]
                + [np.zeros((0, H))])
            kk = min(k, Ed)
            recv_idx = np.concatenate([i for _, _, i, _ in parts]
                                      + [np.zeros((0, kk), dtype=INT)])
            recv_w = np.concatenate([w for _, _, _, w in parts]
                                    + [np.zeros((0, kk))])
            back = ep_expert_pass(recv_x, recv_idx, recv_w,
                                  lambda e, d=d: weights(d * Ed + e))
            pos = 0
            for q, tok, _, _ in parts:
                for u, t in enumerate(tok):
                    ys[q][bounds[q][0] + int(t)] += back[pos + u]
                pos += len(tok)
    return ys, over, n


# ---------------------------------------------------------------------------
# Ring of experts.  [PR4969 What]: tokens are all-gathered around the EP
# ring, every rank computes its local experts for all tokens, and the
# combine is reduce-scattered back to the tokens' owners.  No rank has a
# receive buffer to overflow, so the pass is dropless.  READING: the
# reduce-scatter sums each rank's weighted partial outputs; rank d owns
# experts [d*E/N, (d+1)*E/N) as above.
# ---------------------------------------------------------------------------
def ring_layer(cfg: MoEConfig, N: int, xs: list, logits: list,
               weights: ExpertWeights):
    """Returns the per-rank outputs of the ring-of-experts layer."""
    E, k, H = cfg.E, cfg.k, cfg.H
    Ed = E // N
    Ts = [np.asarray(x).shape[0] for x in xs]
    x_all = np.concatenate([np.asarray(x, dtype=np.float64) for x in xs]
                           + [np.zeros((0, H))])
    routes = [route(L, k, cfg.renorm)[:2] for L in logits]
    idx_all = np.concatenate([r[0] for r in routes]
                             + [np.zeros((0, k), dtype=INT)])
    w_all = np.concatenate([r[1] for r in routes] + [np.zeros((0, k))])
    total = np.zeros_like(x_all)
    for d in range(N):
        local = np.where(idx_all // Ed == d, idx_all - d * Ed, -1)
        total += ep_expert_pass(x_all, local, np.where(local >= 0, w_all, 0.0),
                                lambda e, d=d: weights(d * Ed + e))
    out, t0 = [], 0
    for T_r in Ts:
        out.append(total[t0:t0 + T_r])
        t0 += T_r
    return out


# ---------------------------------------------------------------------------
# Ring of experts, backward.  [PR4969 What]: the combine's reduce-scatter has
# the all-gather of the output cotangent as its transpose (the pages run it
# as a ring all-gather kernel, numerically a plain all-gather), and the
# forward's all-gather of the tokens has a reduce-scatter of the token
# gradients as its transpose.  READING: rank d differentiates its own
# experts' pass over all tokens with the gathered cotangent; each token's
# owner adds the ranks' partial dx, takes the gradient of each pick's
# combine weight from the rank that owns the pick, and runs the router's
# backward on its own logits.  Weight gradients stay with the experts'
# rank.
# ---------------------------------------------------------------------------
def ring_rank_backward(cfg: MoEConfig, N: int, d: int, x_all, idx_all,
                       w_all, dy_all, weights: ExpertWeights):
    """Rank d's share of the ring backward, over the gathered tokens x_all,
    their routing (idx_all, w_all) and the gathered cotangent dy_all.
    Returns (dx_part [T_all, H]: its experts' contribution to every token's
    dx; dtw_part [T_all, k]: the combine-weight gradient of the picks it
    owns, zero elsewhere; {e: (dWg, dWu, dWd)} of its experts with rows)."""
    k, H = cfg.k, cfg.H
    Ed = cfg.E // N
    T_all = x_all.shape[0]
    part = np.zeros((T_all, H))
    dtw = np.zeros((T_all, k))
    dW = {}
    for el in range(Ed):
        e = d * Ed + el
        picks = [(t, j) for t in range(T_all) for j in range(k)
                 if int(idx_all[t, j]) == e]
        if not picks:
            continue
        rows = [t for t, _ in picks]
        _, y = expert_ffn(x_all[rows], *weights(e))
        dy_rows = np.zeros((len(picks), H))
        for q, (t, j) in enumerate(picks):
            dtw[t, j] = float(dy_all[t] @ y[q])
            dy_rows[q] = w_all[t, j] * dy_all[t]
        dx_rows, dW[e] = expert_ffn_backward(x_all[rows], dy_rows,
                                             *weights(e))
        for q, t in enumerate(rows):
            part[t] += dx_rows[q]
    return part, dtw, dW


def ring_layer_backward(cfg: MoEConfig, N: int, xs: list, logits: list,
                        weights: ExpertWeights, dys: list):
    """Returns (dxs, dlogits) per rank and (dWg, dWu, dWd) [E, ...] (zero
    for experts without rows)."""
    E, k, H = cfg.E, cfg.k, cfg.H
    Ts = [np.asarray(x).shape[0] for x in xs]
    x_all = np.concatenate([np.asarray(x, dtype=np.float64) for x in xs]
                           + [np.zeros((0, H))])
    dy_all = np.concatenate([np.asarray(d, dtype=np.float64) for d in dys]
                            + [np.zeros((0, H))])   # cotangent all-gather
    routes = [route(L, k, cfg.renorm)[:2] for L in logits]
    idx_all = np.concatenate([r[0] for r in routes]
                             + [np.zeros((0, k), dtype=INT)])
    w_all = np.concatenate([r[1] for r in routes] + [np.zeros((0, k))])
    T_all = x_all.shape[0]
    wg0 = weights(0)[0]
    F = np.shape(wg0)[1]
    dwg, dwu, dwd = np.zeros((E, H, F)), np.zeros((E, H, F)), \
        np.zeros((E, F, H))
    dx_all = np.zeros((T_all, H))
    dtw_all = np.zeros((T_all, k))
    for d in range(N):
        part, dtw, dW = ring_rank_backward(cfg, N, d, x_all, idx_all, w_all,
                                           dy_all, weights)
        dx_all += part                    # reduce-scatter: summed over d
        dtw_all += dtw                    # each pick has one owner rank
        for e, (a, b, c) in dW.items():
            dwg[e], dwu[e], dwd[e] = a, b, c
    dxs, dls, t0 = [], [], 0
    for r, T_r in enumerate(Ts):
        dxs.append(dx_all[t0:t0 + T_r])
        dls.append(route_backward(logits[r], routes[r][0],
                                  dtw_all[t0:t0 + T_r], cfg.renorm)
                   if T_r else np.zeros((0, E)))
        t0 += T_r
    return dxs, dls, (dwg, dwu, dwd)


# ---------------------------------------------------------------------------
# Expert parallelism, backward.  [PR5920 Tests]: the fallback's gradients
# equal the dropless model's; [PR5920 How]: the backward differentiates
# each pass (each chunk of the fallback) and sums the weight gradients.
# READING: each exchange of the forward has its transpose: the rows the
# destinations returned become the output cotangent sent again to the same
# destinations (one row per dedup'd token), and the rows the source sent
# become token gradients the destinations return and the source adds.  Each
# pick's combine-weight gradient comes back in the slot that carried its
# weight.  Weight gradients stay on the experts' rank, summed over passes.
# ---------------------------------------------------------------------------
def ep_expert_pass_backward(recv_x, recv_idx, recv_w, recv_dy,
                            local_weights: ExpertWeights):
    """The receiving rank's backward of ep_expert_pass, given the cotangent
    recv_dy of its returned rows.  Returns (dx_recv [n, H], dw_recv [n, kk]
    the gradient of each slot's weight, {e: (dWg, dWu, dWd)} of its local
    experts with rows)."""
    recv_x = np.asarray(recv_x, dtype=np.float64)
    recv_dy = np.asarray(recv_dy, dtype=np.float64)
    n = recv_x.shape[0]
    kk = recv_idx.shape[1] if recv_idx.ndim == 2 else 0
    dx = np.zeros_like(recv_x)
    dw = np.zeros((n, kk))
    dW = {}
    by_expert = {}
    for i in range(n):
        for j in range(kk):
            e = int(recv_idx[i, j])
            if e >= 0:
                by_expert.setdefault(e, []).append((i, j))
    for e in sorted(by_expert):
        picks = by_expert[e]
        rows = [i for i, _ in picks]
        _, y = expert_ffn(recv_x[rows], *local_weights(e))
        dy_rows = np.zeros((len(picks), recv_x.shape[1]))
        for q, (i, j) in enumerate(picks):
            dw[i, j] = float(recv_dy[i] @ y[q])
            dy_rows[q] = float(recv_w[i, j]) * recv_dy[i]
        dx_rows, dW[e] = expert_ffn_backward(recv_x[rows], dy_rows,
                                             *local_weights(e))
        for q, i in enumerate(rows):
            dx[i] += dx_rows[q]
    return dx, dw, dW


def ep_layer_backward(cfg: MoEConfig, N: int, xs: list, logits: list,
                      weights: ExpertWeights, dys: list):
    """Backward of ep_layer: per rank (dx, dlogits), and (dWg, dWu, dWd)
    [E, ...] summed over the passes (zero for experts without rows)."""
    E, k, H = cfg.E, cfg.k, cfg.H
    Ed = E // N
    Ts = [np.asarray(x).shape[0] for x in xs]
    if sum(Ts) != cfg.T or cfg.S != N:
        raise ValueError("cfg.T must be the ranks' tokens and cfg.S = N")
    routes = [route(L, k, cfg.renorm)[:2] for L in logits]
    over, n = ep_global_check(cfg, N, routes)
    xs = [np.asarray(x, dtype=np.float64) for x in xs]
    dys = [np.asarray(d, dtype=np.float64) for d in dys]
    wg0 = weights(0)[0]
    F = np.shape(wg0)[1]
    dwg, dwu, dwd = np.zeros((E, H, F)), np.zeros((E, H, F)), \
        np.zeros((E, F, H))
    dxs = [np.zeros((T_r, H)) for T_r in Ts]
    dtws = [np.zeros((T_r, k)) for T_r in Ts]
    kk = min(k, Ed)
    for c in range(n):
        bounds = [ep_chunk_bounds(Ts[r], n, c) for r in range(N)]
        sends = [ep_dispatch(routes[r][0][t0:t1], routes[r][1][t0:t1], E, N)
                 for r, (t0, t1) in enumerate(bounds)]
        for d in range(N):
            parts = []
            for q in range(N):
                a, z = int(sends[q].uniq_offsets[d]), \
                    int(sends[q].uniq_offsets[d + 1])
                parts.append((q, sends[q].uniq_tokens[a:z],
                              sends[q].send_idx[a:z], sends[q].send_w[a:z]))
            t0s = [bounds[q][0] for q, _, _, _ in parts]
            recv_x = np.concatenate(
                [xs[q][t0 + tok] for (q, tok, _, _), t0 in zip(parts, t0s)]
                + [np.zeros((0, H))])
            recv_dy = np.concatenate(
                [dys[q][t0 + tok] for (q, tok, _, _), t0 in zip(parts, t0s)]
                + [np.zeros((0, H))])
            recv_idx = np.concatenate([i for _, _, i, _ in parts]
                                      + [np.zeros((0, kk), dtype=INT)])
            recv_w = np.concatenate([w for _, _, _, w in parts]
                                    + [np.zeros((0, kk))])
            dx_r, dw_r, dW = ep_expert_pass_backward(
                recv_x, recv_idx, recv_w, recv_dy,
                lambda e, d=d: weights(d * Ed + e))
            for el, (a, b, cc) in dW.items():
                e = d * Ed + el
                dwg[e] += a
                dwu[e] += b
                dwd[e] += cc
            pos = 0
            for (q, tok, _, _), t0 in zip(parts, t0s):
                for u, t in enumerate(tok):
                    t = t0 + int(t)
                    dxs[q][t] += dx_r[pos + u]
                    # slot s of this row = the s-th pick of t that d owns
                    own = [j for j in range(k)
                           if int(routes[q][0][t, j]) // Ed == d]
                    for s, j in enumerate(own):
                        dtws[q][t, j] = dw_r[pos + u, s]
                pos += len(tok)
    dls = [route_backward(logits[r], routes[r][0], dtws[r], cfg.renorm)
           if Ts[r] else np.zeros((0, E)) for r in range(N)]
    return dxs, dls, (dwg, dwu, dwd)
