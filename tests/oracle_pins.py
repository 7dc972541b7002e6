"""Pins for the float64 oracle: checks against what the MaxText pages and the
mathematics fix, never against a retyped copy of the oracle's own formulas.

Each ``pin_*`` function raises AssertionError on a mismatch.  They are run
directly by test_oracle_pins.py, and again by test_oracle_mutations.py against
oracles with a planted mistake, to show that each plausible mistake is caught.
"""
from __future__ import annotations

import itertools
import json
import math
import os

import numpy as np
import scipy.special
import torch

from oracle import moe_ref as ref

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


def _tie_heavy_logits(rng, T, E, levels=3):
    """Logits drawn from a handful of values so that ties are common."""
    return rng.integers(0, levels, size=(T, E)).astype(np.float32)


# --------------------------------------------------------------------------
# top-k: the selected set is the unique k-subset that dominates its
# complement under (larger logit, then lower index); found by enumeration.
# --------------------------------------------------------------------------
def _dominates(l, i, j):
    return l[i] > l[j] or (l[i] == l[j] and i < j)


def pin_topk_bruteforce():
    rng = _rng(1)
    for E in (3, 5, 6):
        L = _tie_heavy_logits(rng, 12, E)
        for k in range(1, E + 1):
            idx, _, _ = ref.route(L, k)
            for t in range(L.shape[0]):
                l = [float(v) for v in L[t]]
                valid = []
                for sub in itertools.combinations(range(E), k):
                    rest = [j for j in range(E) if j not in sub]
                    if all(_dominates(l, i, j) for i in sub for j in rest):
                        valid.append(set(sub))
                assert len(valid) == 1
                assert set(int(v) for v in idx[t]) == valid[0]
                # rank order: each pick dominates the next
                for a, b in zip(idx[t][:-1], idx[t][1:]):
                    assert _dominates(l, int(a), int(b))


def pin_topk_hand_ties():
    # all equal -> the k lowest indices, in order
    idx, _, _ = ref.route(np.zeros((1, 6), np.float32), 3)
    assert idx[0].tolist() == [0, 1, 2]
    # equal maxima at 4 and 1 -> 1 before 4, then the 0.5 at index 5
    L = np.array([[0.0, 2.0, -1.0, 0.0, 2.0, 0.5]], np.float32)
    idx, _, _ = ref.route(L, 3)
    assert idx[0].tolist() == [1, 4, 5]
    # NaN and +inf rank as -inf, after every finite logit
    L = np.array([[np.nan, 1.0, np.inf, -5.0]], np.float32)
    idx, w, nf = ref.route(L, 3)
    assert nf
    assert idx[0].tolist() == [1, 3, 0]
    # the softmax ignores the non-finite entries: two finite logits 1, -5
    p1 = 1.0 / (1.0 + math.exp(-6.0))
    assert abs(w[0, 0] - p1) < 1e-15 and abs(w[0, 1] - (1 - p1)) < 1e-15
    assert w[0, 2] == 0.0
    # no finite logit at all -> lowest indices, zero weights
    idx, w, _ = ref.route(np.full((1, 4), np.nan, np.float32), 2)
    assert idx[0].tolist() == [0, 1] and np.all(w == 0)


def pin_softmax_weights():
    rng = _rng(2)
    # equal logits -> 1/E; with renorm -> 1/k
    _, w, _ = ref.route(np.full((2, 8), 0.7, np.float32), 3)
    assert np.allclose(w, 1.0 / 8, rtol=0, atol=1e-15)
    _, w, _ = ref.route(np.full((2, 8), 0.7, np.float32), 3, renorm=True)
    assert np.allclose(w, 1.0 / 3, rtol=0, atol=1e-15)
    # two experts: the larger gets the logistic of the gap
    for d in (0.0, 0.3, 2.0, 9.0):
        L = np.array([[0.25, 0.25 + d]], np.float32)
        _, w, _ = ref.route(L, 1)
        gap = float(np.float32(0.25 + d)) - 0.25
        assert abs(w[0, 0] - 1.0 / (1.0 + math.exp(-gap))) < 1e-14
    # against scipy's softmax on random rows
    L = rng.standard_normal((20, 16)).astype(np.float32) * 3
    idx, w, _ = ref.route(L, 4)
    p = scipy.special.softmax(L.astype(np.float64), axis=1)
    assert np.allclose(w, np.take_along_axis(p, idx, 1), rtol=1e-13, atol=0)
    idx, w, _ = ref.route(L, 4, renorm=True)
    sel = np.take_along_axis(L.astype(np.float64), idx, 1)
    assert np.allclose(w, scipy.special.softmax(sel, axis=1), rtol=1e-13)
    assert np.allclose(w.sum(1), 1.0, atol=1e-14)


# --------------------------------------------------------------------------
# counts
# --------------------------------------------------------------------------
def pin_counts():
    rng = _rng(3)
    for (T, E, k, S) in ((64, 8, 2, 2), (100, 16, 3, 4), (7, 4, 4, 4)):
        L = rng.standard_normal((T, E)).astype(np.float32)
        idx, _, _ = ref.route(L, k)
        c = ref.expert_counts(idx, E)
        assert int(c.sum()) == T * k
        assert np.array_equal(c, np.bincount(idx.ravel(), minlength=E))
        r = ref.shard_counts(c, S)
        assert int(r.sum()) == T * k
        assert np.array_equal(r, c.reshape(S, E // S).sum(1))
        off = ref.exclusive_scan(c)
        assert np.array_equal(off, np.concatenate([[0], np.cumsum(c)]))


# --------------------------------------------------------------------------
# capacity and the overflow flag
# --------------------------------------------------------------------------
def pin_capacity_closed_forms():
    # factor x balanced, balanced = T*k/S rows
    assert ref.capacity(4096, 2, 4, 2.0) == 4096
    assert ref.capacity(8192, 8, 8, 2.0) == 16384
    assert ref.capacity(8192, 1, 16, 2.0) == 1024
    # capped at T*k: a shard cannot receive more rows than exist
    assert ref.capacity(256, 2, 2, 2.0) == 512
    # float32 factor 0.1 is slightly above 0.1: 25.6000003 -> 25
    assert ref.capacity(256, 2, 2, 0.1) == 25
    assert ref.capacity(10, 3, 4, 1.0) == 7          # floor(7.5)
    assert ref.capacity(8, 1, 8, 1.0) == 1
    # no cap for factor <= 0 ("-1" in the pages)
    assert ref.capacity(256, 2, 2, -1.0) is None
    assert ref.capacity(256, 2, 2, 0.0) is None


def _idx_with_shard_loads(loads, k, E, S):
    """A routing whose shard receive counts are exactly ``loads``: tokens
    take k distinct experts inside one shard (needs k <= E/S)."""
    Es = E // S
    rows = []
    for s, n in enumerate(loads):
        assert n % k == 0
        for _ in range(n // k):
            rows.append([s * Es + j for j in range(k)])
    return np.array(rows, dtype=np.int64)


def pin_overflow_flag():
    E, S, k = 8, 4, 2
    # shard loads (rows) chosen by hand; T = sum/k
    for loads in ([4, 4, 4, 4], [10, 2, 2, 2], [2, 2, 2, 10], [0, 0, 0, 16],
                  [6, 6, 2, 2]):
        idx = _idx_with_shard_loads(loads, k, E, S)
        T = idx.shape[0]
        r = ref.shard_counts(ref.expert_counts(idx, E), S)
        assert r.tolist() == loads
        for factor in (0.1, 0.5, 1.0, 1.5, 2.0, 4.0, -1.0):
            C = ref.capacity(T, k, S, factor)
            expect = C is not None and max(loads) > C
            assert ref.overflow_flag(r, C) == expect
    # strictness: a shard holding exactly C rows does not overflow
    idx = _idx_with_shard_loads([8, 4, 2, 2], k, E, S)       # T=8, B=4
    r = ref.shard_counts(ref.expert_counts(idx, E), S)
    assert ref.capacity(8, k, S, 2.0) == 8
    assert not ref.overflow_flag(r, 8)
    assert ref.overflow_flag(r, 7)
    # one asymmetric hot shard (the last) sets the global flag
    idx = _idx_with_shard_loads([2, 2, 2, 10], k, E, S)
    r = ref.shard_counts(ref.expert_counts(idx, E), S)
    assert ref.overflow_flag(r, ref.capacity(8, k, S, 2.0))
    # required factor: balanced -> 1, all in one shard -> S
    idx = _idx_with_shard_loads([4, 4, 4, 4], k, E, S)
    r = ref.shard_counts(ref.expert_counts(idx, E), S)
    assert ref.required_factor(r, 8, k) == 1.0
    idx = _idx_with_shard_loads([0, 16, 0, 0], k, E, S)
    r = ref.shard_counts(ref.expert_counts(idx, E), S)
    assert ref.required_factor(r, 8, k) == 4.0


def pin_worst_case_buffer():
    with open(os.path.join(GOLDEN, "worst_case_buffer.json")) as f:
        g = json.load(f)
    for c in g["cases"]:
        T, k, E, S = c["T"], c["k"], c["E"], c["S"]
        Es = E // S
        # adversarial routing: every token's picks inside shard 0
        idx = np.array([[j for j in range(min(k, Es))]] * T, dtype=np.int64)
        if k > Es:
            return
        r = ref.shard_counts(ref.expert_counts(idx, E), S)
        assert int(r[0]) == c["worst_rows"]
        assert T * k // S == c["balanced_rows"]
        assert ref.required_factor(r, T, k) == c["ratio"]


# --------------------------------------------------------------------------
# the permutation
# --------------------------------------------------------------------------
def pin_permutation_dropless():
    rng = _rng(4)
    for (T, E, k, S) in ((50, 8, 2, 2), (33, 16, 4, 4), (5, 4, 4, 2)):
        L = _tie_heavy_logits(rng, T, E, levels=5)
        idx, _, _ = ref.route(L, k)
        p = ref.permute_indices(idx, E, S, None)
        R = T * k
        assert p.n_dropped == 0 and len(p.sorted_token) == R
        # bijection onto all (t, j)
        pairs = sorted(zip(p.sorted_token.tolist(), p.sorted_slot.tolist()))
        assert pairs == [(t, j) for t in range(T) for j in range(k)]
        # row_of is the inverse
        for r in range(R):
            assert p.row_of[p.sorted_token[r], p.sorted_slot[r]] == r
        # order: numpy's stable lexsort by (expert, token)
        flat_e = idx.ravel()
        flat_t = np.repeat(np.arange(T), k)
        order = np.lexsort((flat_t, flat_e))
        assert np.array_equal(p.sorted_token, flat_t[order])
        assert np.array_equal(idx[p.sorted_token, p.sorted_slot],
                              flat_e[order])
        assert np.array_equal(p.group_offsets, p.dropless_offsets)
        assert np.array_equal(
            np.diff(p.group_offsets), np.bincount(flat_e, minlength=E))


def pin_permutation_capped():
    rng = _rng(5)
    for (T, E, k, S, factor) in ((64, 8, 2, 2, 0.6), (40, 16, 3, 4, 0.5),
                                 (64, 8, 2, 4, 1.0), (30, 8, 1, 2, 0.1)):
        L = rng.standard_normal((T, E)).astype(np.float32)
        L[:, : E // S] += 1.5            # make shard 0 hot
        idx, _, _ = ref.route(L, k)
        C = ref.capacity(T, k, S, factor)
        p = ref.permute_indices(idx, E, S, C)
        full = ref.permute_indices(idx, E, S, None)
        r = ref.shard_counts(ref.expert_counts(idx, E), S)
        assert p.n_dropped == int(sum(max(0, int(x) - C) for x in r))
        Es = E // S
        kept_rows = set(zip(p.sorted_token.tolist(), p.sorted_slot.tolist()))
        for s in range(S):
            # dropless rows of shard s, in order; the kept ones are its
            # first C, and they keep their relative order
            seg = [(int(full.sorted_token[q]), int(full.sorted_slot[q]))
                   for q in range(full.group_offsets[s * Es],
                                  full.group_offsets[(s + 1) * Es])]
            want = seg[:C]
            got = [(int(p.sorted_token[q]), int(p.sorted_slot[q]))
                   for q in range(p.group_offsets[s * Es],
                                  p.group_offsets[(s + 1) * Es])]
            assert got == want
            for pair in seg[C:]:
                assert pair not in kept_rows
                assert p.row_of[pair] == -1
        assert int((p.row_of >= 0).sum()) == T * k - p.n_dropped


def pin_dedup():
    rng = _rng(6)
    for (T, E, k, S, factor) in ((60, 8, 3, 2, -1.0), (48, 16, 4, 4, 0.5),
                                 (20, 8, 1, 4, -1.0)):
        L = rng.standard_normal((T, E)).astype(np.float32)
        L[:, :2] += 1.0
        idx, _, _ = ref.route(L, k)
        C = ref.capacity(T, k, S, factor)
        p = ref.permute_indices(idx, E, S, C)
        Es = E // S
        for s in range(S):
            want = set()
            for q in range(p.group_offsets[s * Es],
                           p.group_offsets[(s + 1) * Es]):
                want.add(int(p.sorted_token[q]))
            seg = p.uniq_tokens[p.uniq_offsets[s]:p.uniq_offsets[s + 1]]
            assert sorted(want) == seg.tolist()   # ascending, no truncation
        x = rng.standard_normal((T, 5))
        xs = ref.gather_rows(x, p.sorted_token)
        assert np.array_equal(xs, x[p.uniq_tokens[p.expand_idx]])
        if k == 1:
            assert len(p.uniq_tokens) == len(p.sorted_token)
    # adversarial: every pick in shard 0 -> each token sent exactly once
    T, E, k, S = 16, 8, 3, 2
    idx = np.array([[0, 1, 2]] * T)
    p = ref.permute_indices(idx, E, S, None)
    assert len(p.uniq_tokens) == T
    assert p.uniq_offsets.tolist() == [0, T, T]


# --------------------------------------------------------------------------
# the FFN and the combine
# --------------------------------------------------------------------------
def _silu(z):
    return z / (1.0 + math.exp(-z))


def pin_ffn_closed_form():
    # H=4, F=2 by hand: x.Wg = (1, 2), x.Wu = (2, 1),
    # h = (2 silu(1), silu(2)); Wd puts h0 on output 0 and h1 on output 3
    x = np.array([[1.0, 2.0, 0.0, -1.0]])
    wg = np.array([[1, 0], [0, 1], [0, 0], [0, 0]], np.float64)
    wu = np.array([[0, 1], [1, 0], [7, 7], [0, 0]], np.float64)
    wd = np.array([[1, 0, 0, 0], [0, 0, 0, 1]], np.float64)
    h, y = ref.expert_ffn(x, wg, wu, wd)
    s1 = 1.0 / (1.0 + math.exp(-1.0))
    s2 = 2.0 / (1.0 + math.exp(-2.0))
    assert abs(h[0, 0] - 2 * s1) < 1e-15 and abs(h[0, 1] - s2) < 1e-15
    assert abs(y[0, 0] - 2 * s1) < 1e-15 and abs(y[0, 3] - s2) < 1e-15
    assert y[0, 1] == 0 and y[0, 2] == 0
    # silu at a few points: 0, odd part, large |z|
    for z in (0.0, -3.0, 3.0, 30.0, -30.0):
        assert abs(ref.silu(np.array([z]))[0] - _silu(z)) < 1e-15
    assert abs(ref.silu(np.array([3.0]))[0] - ref.silu(np.array([-3.0]))[0]
               - 3.0) < 1e-14


def pin_dense_mlp_reduction():
    # E=1, k=1, renorm: the layer is a dense SwiGLU MLP (torch, float64)
    rng = _rng(7)
    T, H, F = 9, 6, 10
    x = rng.standard_normal((T, H))
    wg, wu = rng.standard_normal((1, H, F)), rng.standard_normal((1, H, F))
    wd = rng.standard_normal((1, F, H))
    cfg = ref.MoEConfig(T, H, 1, 1, F, 1, -1.0, 0, True)
    res = ref.layer_dropless(cfg, x, np.zeros((T, 1), np.float32),
                             ref.dense_weights(wg, wu, wd))
    xt = torch.from_numpy(x)
    want = (torch.nn.functional.silu(xt @ torch.from_numpy(wg[0]))
            * (xt @ torch.from_numpy(wu[0]))) @ torch.from_numpy(wd[0])
    assert np.allclose(res.y, want.numpy(), rtol=1e-12, atol=1e-12)


def pin_combine():
    rng = _rng(8)
    T, H, E, k, F, S = 24, 5, 8, 3, 7, 2
    x = rng.standard_normal((T, H))
    one = (rng.standard_normal((H, F)), rng.standard_normal((H, F)),
           rng.standard_normal((F, H)))
    same = ref.dense_weights(*[np.stack([w] * E) for w in one])
    L = rng.standard_normal((T, E)).astype(np.float32)
    _, ffn = ref.expert_ffn(x, *one)
    # identical experts + renorm: y = FFN(x)
    cfg = ref.MoEConfig(T, H, E, k, F, S, -1.0, 0, True)
    res = ref.layer_dropless(cfg, x, L, same)
    assert np.allclose(res.y, ffn, rtol=1e-12, atol=1e-12)
    # without renorm: y = (sum of the chosen softmax probabilities) FFN(x)
    cfg = ref.MoEConfig(T, H, E, k, F, S, -1.0, 0, False)
    res = ref.layer_dropless(cfg, x, L, same)
    p = scipy.special.softmax(L.astype(np.float64), axis=1)
    mass = np.sort(p, axis=1)[:, -k:].sum(1)
    assert np.allclose(res.y, mass[:, None] * ffn, rtol=1e-12, atol=1e-12)
    # all rows of a token dropped -> its output is exactly zero
    L = np.zeros((T, E), np.float32)
    L[:, 0] = 5.0                      # every token's top-1 is expert 0
    cfg = ref.MoEConfig(T, H, E, 1, F, S, 0.25, 0, True)   # C = 3
    res = ref.layer_capped(cfg, x, L, same)
    C = ref.capacity(T, 1, S, 0.25)
    assert C == 3
    assert np.allclose(res.y[:C], ffn[:C], rtol=1e-12, atol=1e-12)
    assert np.all(res.y[C:] == 0)


# --------------------------------------------------------------------------
# the chunked dropless fallback
# --------------------------------------------------------------------------
def pin_chunk_count_golden():
    with open(os.path.join(GOLDEN, "fallback_chunks.json")) as f:
        g = json.load(f)
    for c in g["cases"]:
        C = ref.capacity(c["T"], c["k"], c["S"], c["factor"])
        plan = ref.chunk_plan(c["T"], c["k"], c["E"], c["S"], C)
        assert len(plan) == c["n_chunks"]
    # DeepSeek-V3 shape: 2048-token chunks of 8 picks fill C = 16384 exactly
    assert len(ref.chunk_plan(8192, 8, 256, 8, 16384)) == 4


def pin_chunk_plan_bounds():
    rng = _rng(9)
    for _ in range(300):
        S = int(rng.choice([1, 2, 4, 8]))
        E = S * int(rng.integers(1, 6))
        k = int(rng.integers(1, E + 1))
        T = int(rng.integers(1, 200))
        factor = float(rng.choice([0.1, 0.5, 1.0, 2.0, 3.0]))
        C = ref.capacity(T, k, S, factor)
        plan = ref.chunk_plan(T, k, E, S, C)
        m = min(k, E // S)
        # contiguous cover of [0, T)
        assert plan[0][0] == 0 and plan[-1][1] == T
        assert all(a[1] == b[0] for a, b in zip(plan[:-1], plan[1:]))
        sizes = [b - a for a, b in plan]
        c = sizes[0]
        assert all(sz == c for sz in sizes[:-1]) and 0 < sizes[-1] <= c
        # the chunk's worst case fits C, one more token would not
        if C >= m:
            assert c * m <= C < (c + 1) * m or c == T
        else:
            assert c == 1
    # explicit count
    assert [b - a for a, b in ref.chunk_plan(10, 2, 4, 2, 4, n_chunks=3)] \
        == [4, 4, 2]


def pin_fallback_equivalences():
    rng = _rng(10)
    T, H, E, k, F, S = 48, 6, 8, 2, 5, 2
    x = rng.standard_normal((T, H))
    ws = ref.dense_weights(rng.standard_normal((E, H, F)),
                           rng.standard_normal((E, H, F)),
                           rng.standard_normal((E, F, H)))
    L = rng.standard_normal((T, E)).astype(np.float32)
    L[:, :3] += 1.0                                  # hot shard 0
    cfg = ref.MoEConfig(T, H, E, k, F, S, 0.1)
    drop = ref.layer_dropless(cfg, x, L, ws)
    chunked = ref.layer_dropless_chunked(cfg, x, L, ws)
    assert len(chunked.chunks) > 1
    assert np.array_equal(chunked.y, drop.y) or \
        np.allclose(chunked.y, drop.y, rtol=1e-13, atol=1e-13)
    # factor 0.1 forces overflow; the capped path diverges from dropless
    capped = ref.layer_capped(cfg, x, L, ws)
    assert capped.overflow and capped.perm.n_dropped > 0
    assert not np.allclose(capped.y, drop.y)
    # the layer with fallback=layer matches dropless in both branches
    for factor in (0.1, 2.0, 8.0):
        c2 = ref.MoEConfig(T, H, E, k, F, S, factor)
        out = ref.layer(c2, x, L, ws)
        assert np.allclose(out.y, drop.y, rtol=1e-13, atol=1e-13)
    # uncapped (factor <= 0) is dropless
    for factor in (-1.0, 0.0):
        c3 = ref.MoEConfig(T, H, E, k, F, S, factor)
        assert np.array_equal(ref.layer_capped(c3, x, L, ws).y, drop.y)


def pin_asymmetric_single_shard():
    # only the last shard is hot; the layer still takes the fallback
    rng = _rng(11)
    T, H, E, k, F, S = 40, 4, 8, 2, 3, 4
    L = rng.standard_normal((T, E)).astype(np.float32)
    L[:, 6:8] += 4.0
    idx, _, _ = ref.route(L, k)
    r = ref.shard_counts(ref.expert_counts(idx, E), S)
    C = ref.capacity(T, k, S, 2.0)
    assert int(np.argmax(r)) == 3 and r[3] > C
    assert sum(int(v) > C for v in r) == 1
    x = rng.standard_normal((T, H))
    ws = ref.dense_weights(rng.standard_normal((E, H, F)),
                           rng.standard_normal((E, H, F)),
                           rng.standard_normal((E, F, H)))
    out = ref.layer(ref.MoEConfig(T, H, E, k, F, S, 2.0), x, L, ws)
    assert out.overflow and len(out.chunks) > 1


# --------------------------------------------------------------------------
# dynamic redundant experts
# --------------------------------------------------------------------------
def pin_duplication_hand_cases():
    # one hot expert, two shards of 4 experts, one slot per shard: half the
    # gap (8 - 0) // 2 = 4 rows go to the slot of shard 1 (virtual group 9)
    p = ref.plan_duplication(np.array([8, 0, 0, 0, 0, 0, 0, 0]), 2, 1)
    assert p.divert.tolist() == [4, 0, 0, 0, 0, 0, 0, 0]
    assert p.slot_of.tolist() == [9, -1, -1, -1, -1, -1, -1, -1]
    assert p.group_expert.tolist() == [0, 1, 2, 3, -1, 4, 5, 6, 7, 0]
    assert p.loads_after.tolist() == [4, 4]
    # the review's case: once r_max's only expert is duplicated there is no
    # candidate left, so the plan stops instead of duplicating it again
    p = ref.plan_duplication(np.array([100, 0]), 2, 4)
    assert p.divert.tolist() == [50, 0]
    assert int((p.group_expert == 0).sum()) == 2      # home group + 1 slot
    assert p.loads_after.tolist() == [50, 50]
    # three shards: the hottest expert of the hottest shard goes first, to
    # the least loaded shard; ties go to the lower index
    p = ref.plan_duplication(np.array([6, 9, 2, 0, 0, 0]), 3, 1)
    # loads [15, 2, 0]: e=1 (9 rows) to shard 2, n = min(9, 15 // 2) = 7;
    # loads [8, 2, 7]: e=0 (6 rows) to shard 1, n = min(6, (8-2)//2) = 3;
    # loads [5, 5, 7]: r_max = 2 has no rows of its own -> stop
    assert p.divert.tolist() == [3, 7, 0, 0, 0, 0]
    assert p.loads_after.tolist() == [5, 5, 7]
    assert p.slot_of.tolist() == [
        ref.virtual_group_of_slot(1, 0, 6, 3, 1),
        ref.virtual_group_of_slot(2, 0, 6, 3, 1), -1, -1, -1, -1]


def pin_duplication_invariants():
    rng = _rng(12)
    for _ in range(200):
        S = int(rng.choice([2, 4, 8]))
        Es = int(rng.integers(1, 6))
        E = S * Es
        B = int(rng.integers(1, 4))
        counts = rng.integers(0, 50, size=E) * (rng.random(E) < 0.7)
        counts[: Es] *= int(rng.integers(1, 6))        # a hot shard
        p = ref.plan_duplication(counts, S, B)
        before = ref.shard_counts(counts, S)
        assert int(p.loads_after.sum()) == int(counts.sum())
        assert int(p.loads_after.max()) <= int(before.max())
        assert np.all(p.divert >= 0) and np.all(p.divert <= counts)
        G = S * (Es + B)
        assert len(p.group_expert) == G
        for e in range(E):
            home = ref.virtual_group_of_expert(e, E, S, B)
            assert p.group_expert[home] == e
            if p.slot_of[e] >= 0:
                assert p.divert[e] > 0
                g = int(p.slot_of[e])
                assert p.group_expert[g] == e
                assert g // (Es + B) != e // Es      # never on its home shard
                assert g % (Es + B) >= Es            # a slot, not an expert
            else:
                assert p.divert[e] == 0
            # an expert is duplicated at most once
            assert int((p.group_expert == e).sum()) <= 2
        for s in range(S):
            used = sum(1 for b in range(B)
                       if p.group_expert[s * (Es + B) + Es + b] >= 0)
            assert used <= B
        # loads after = virtual shard loads of the rerouted rows
        L = rng.standard_normal((40, E)).astype(np.float32)
        idx, _, _ = ref.route(L, min(2, E))
        c = ref.expert_counts(idx, E)
        p = ref.plan_duplication(c, S, B)
        v = ref.reroute(idx, p, E, S)
        vc = ref.expert_counts(v, G)
        assert np.array_equal(ref.shard_counts(vc, S), p.loads_after)
        for e in range(E):
            assert vc[ref.virtual_group_of_expert(e, E, S, B)] == \
                c[e] - p.divert[e]
            if p.slot_of[e] >= 0:
                assert vc[p.slot_of[e]] == p.divert[e]


def pin_reroute_takes_last_rows():
    # expert 0 picked by tokens 0..5; shard loads 12 and 4, so half the gap
    # (4 rows) moves and the duplicate gets the LAST 4 of expert 0's rows
    idx = np.array([[0, 1]] * 6 + [[4, 5]] * 2)
    p = ref.plan_duplication(ref.expert_counts(idx, 8), 2, 1)
    v = ref.reroute(idx, p, 8, 2)
    d = int(p.divert[0])
    assert d == 4
    home = ref.virtual_group_of_expert(0, 8, 2, 1)
    assert [int(g) for g in v[:, 0][:6]] == [home] * (6 - d) + \
        [int(p.slot_of[0])] * d


def pin_redundancy_preserves_the_layer():
    rng = _rng(13)
    T, H, E, k, F, S = 64, 5, 8, 2, 6, 4
    x = rng.standard_normal((T, H))
    ws = ref.dense_weights(rng.standard_normal((E, H, F)),
                           rng.standard_normal((E, H, F)),
                           rng.standard_normal((E, F, H)))
    L = rng.standard_normal((T, E)).astype(np.float32)
    L[:, :2] += 2.5                               # shard 0 hot
    cfg = ref.MoEConfig(T, H, E, k, F, S, 2.0)
    plain = ref.layer(cfg, x, L, ws)
    assert plain.overflow                          # without slots: fallback
    red = ref.layer_redundant(cfg, x, L, ws, B=2)
    assert not red.overflow                        # with slots: capped path
    assert red.perm.n_dropped == 0
    assert np.allclose(red.y, plain.y, rtol=1e-12, atol=1e-12)
    # every duplicate slot that got rows runs its expert's weights
    G = S * (E // S + 2)
    sizes = np.diff(red.perm.group_offsets)
    assert sizes[[g for g in range(G) if g % (E // S + 2) >= E // S]].sum() > 0


# --------------------------------------------------------------------------
# backward pass: central finite differences of L = sum(y * dy) in float64
# (independent of the analytic chain rule), chunked == dropless, and a
# dense-MLP reduction through torch.autograd
# --------------------------------------------------------------------------
def _tiny_backward_case(seed, T=6, H=4, E=4, k=2, F=3, S=2):
    rng = _rng(seed)
    x = rng.standard_normal((T, H))
    # distinct, well separated logits: the top-k choice is stable under eps
    L = rng.permutation(T * E).reshape(T, E) * 0.37 - 3.0
    w = (rng.standard_normal((E, H, F)), rng.standard_normal((E, H, F)),
         rng.standard_normal((E, F, H)))
    dy = rng.standard_normal((T, H))
    return x, L.astype(np.float64), w, dy


def _fd_check(loss, arr, grad, eps=1e-6, tol=1e-6):
    it = np.nditer(arr, flags=["multi_index"])
    for _ in it:
        i = it.multi_index
        old = arr[i]
        arr[i] = old + eps
        lp = loss()
        arr[i] = old - eps
        lm = loss()
        arr[i] = old
        fd = (lp - lm) / (2 * eps)
        assert abs(fd - grad[i]) <= tol * max(1.0, abs(fd)), (i, fd, grad[i])


def pin_backward_finite_differences():
    for renorm in (False, True):
        for factor in (-1.0, 0.6):          # dropless, and capped with drops
            x, L, (wg, wu, wd), dy = _tiny_backward_case(14)
            cfg = ref.MoEConfig(6, 4, 4, 2, 3, 2, factor, 0, renorm)
            back = ref.layer_backward_capped if factor > 0 else \
                ref.layer_backward_dropless
            run = ref.layer_capped if factor > 0 else ref.layer_dropless
            g = back(cfg, x, L, wg, wu, wd, dy)

            def loss():
                y = run(cfg, x, L, ref.dense_weights(wg, wu, wd)).y
                return float((y * dy).sum())
            _fd_check(loss, x, g.dx)
            _fd_check(loss, L, g.dlogits)
            _fd_check(loss, wg, g.dwg)
            _fd_check(loss, wu, g.dwu)
            _fd_check(loss, wd, g.dwd)
            if factor > 0:   # the capped pass dropped rows: no gradient there
                C = ref.capacity(6, 2, 2, factor)
                idx, _, _ = ref.route(L, 2, renorm)
                p = ref.permute_indices(idx, 4, 2, C)
                assert p.n_dropped > 0
                assert np.all(g.dtopk_w[p.row_of < 0] == 0)


def pin_backward_chunked_equals_dropless():
    rng = _rng(15)
    T, H, E, k, F, S = 40, 5, 8, 2, 4, 2
    x = rng.standard_normal((T, H))
    L = rng.standard_normal((T, E))
    L[:, :3] += 1.5
    w = (rng.standard_normal((E, H, F)), rng.standard_normal((E, H, F)),
         rng.standard_normal((E, F, H)))
    dy = rng.standard_normal((T, H))
    cfg = ref.MoEConfig(T, H, E, k, F, S, 0.2)
    drop = ref.layer_backward_dropless(cfg, x, L, *w, dy)
    chunk = ref.layer_backward_chunked(cfg, x, L, *w, dy)
    C = ref.capacity(T, k, S, 0.2)
    assert len(ref.chunk_plan(T, k, E, S, C)) > 1
    for a, b in ((drop.dx, chunk.dx), (drop.dlogits, chunk.dlogits),
                 (drop.dwg, chunk.dwg), (drop.dwu, chunk.dwu),
                 (drop.dwd, chunk.dwd)):
        assert np.allclose(a, b, rtol=1e-12, atol=1e-12)


def pin_segmented_weight_grads():
    """dW from segmented_weight_grads against finite differences (and torch
    autograd) of the loss sum_r Q[r] . (P[r] W[expert of r]) over the rows
    the segments name: two segments with foreign rows around and between
    them, a group with no rows in one segment, and a duplicate group whose
    rows add into its expert."""
    rng = _rng(21)
    rows, cp, cq, E = 40, 3, 2, 3
    P = rng.standard_normal((rows, cp))
    Q = rng.standard_normal((rows, cq))
    gexp = [0, 1, 2, 1]                       # group 3 duplicates expert 1
    segs = [(np.array([0, 3, 3, 7, 9]), 2),   # group 1 empty here
            (np.array([0, 4, 6, 11, 12]), 20)]
    W = rng.standard_normal((E, cp, cq))
    got = ref.segmented_weight_grads(P, Q, segs, 4, E, gexp)
    assert got.shape == (E, cp, cq)

    def loss():
        tot = 0.0
        for off, base in segs:
            for g in range(4):
                for r in range(base + off[g], base + off[g + 1]):
                    tot += float(Q[r] @ (P[r] @ W[gexp[g]]))
        return tot
    _fd_check(loss, W, got)
    # identity group map, one segment: torch autograd of the same loss
    off = np.array([0, 5, 5, 17])
    Wt = torch.tensor(W, requires_grad=True)
    Pt, Qt = torch.from_numpy(P), torch.from_numpy(Q)
    lt = sum((Qt[off[e]:off[e + 1]] * (Pt[off[e]:off[e + 1]] @ Wt[e])).sum()
             for e in range(E))
    lt.backward()
    g1 = ref.segmented_weight_grads(P, Q, [(off, 0)], 3, E)
    assert np.allclose(g1, Wt.grad.numpy(), rtol=1e-12, atol=1e-12)
    assert np.all(g1[1] == 0)                 # expert 1 has no rows


def pin_backward_dense_reduction():
    rng = _rng(16)
    T, H, F = 7, 5, 6
    x = rng.standard_normal((T, H))
    w = (rng.standard_normal((1, H, F)), rng.standard_normal((1, H, F)),
         rng.standard_normal((1, F, H)))
    dy = rng.standard_normal((T, H))
    cfg = ref.MoEConfig(T, H, 1, 1, F, 1, -1.0, 0, True)
    g = ref.layer_backward_dropless(cfg, x, np.zeros((T, 1)), *w, dy)
    xt = torch.tensor(x, requires_grad=True)
    wt = [torch.tensor(a[0], requires_grad=True) for a in w]
    y = (torch.nn.functional.silu(xt @ wt[0]) * (xt @ wt[1])) @ wt[2]
    (y * torch.from_numpy(dy)).sum().backward()
    assert np.allclose(g.dx, xt.grad.numpy(), rtol=1e-12, atol=1e-12)
    assert np.allclose(g.dwg[0], wt[0].grad.numpy(), rtol=1e-12, atol=1e-12)
    assert np.allclose(g.dwu[0], wt[1].grad.numpy(), rtol=1e-12, atol=1e-12)
    assert np.allclose(g.dwd[0], wt[2].grad.numpy(), rtol=1e-12, atol=1e-12)
    assert np.all(g.dlogits == 0)       # one expert, renorm: weight is 1


def pin_redundant_backward_equals_dropless():
    """fallback=layer with duplicate slots never drops a row (a shard over
    capacity takes the dropless fallback), so its gradients equal the
    dropless ones; the cases include plans that divert rows into slots (the
    virtual-group path: slot groups with their expert's weights, an expert's
    weight gradient summed over its groups)."""
    rng = _rng(17)
    diverted = 0
    for _ in range(24):
        S = int(rng.choice([2, 4]))
        E = S * int(rng.choice([2, 3]))
        k = int(rng.choice([1, 2]))
        B = int(rng.choice([1, 2]))
        T, H, F = int(rng.integers(12, 30)), 3, 4
        factor = float(rng.choice([1.0, 1.5, 2.0]))
        x = rng.standard_normal((T, H))
        L = rng.standard_normal((T, E)) - 1.5 * np.log(np.arange(E) + 1.0)
        w = (rng.standard_normal((E, H, F)), rng.standard_normal((E, H, F)),
             rng.standard_normal((E, F, H)))
        dy = rng.standard_normal((T, H))
        cfg = ref.MoEConfig(T, H, E, k, F, S, factor)
        red = ref.layer_redundant_backward(cfg, x, L, *w, dy, B)
        drop = ref.layer_backward_dropless(cfg, x, L, *w, dy)
        for a, b in ((red.dx, drop.dx), (red.dlogits, drop.dlogits),
                     (red.dwg, drop.dwg), (red.dwu, drop.dwu),
                     (red.dwd, drop.dwd), (red.dtopk_w, drop.dtopk_w)):
            assert np.allclose(a, b, rtol=1e-10, atol=1e-10)
        idx, _, _ = ref.route(L, k)
        plan = ref.plan_duplication(ref.expert_counts(idx, E), S, B)
        vidx = ref.reroute(idx, plan, E, S)
        G = S * (E // S + B)
        C = ref.capacity(T, k, S, factor)
        if plan.divert.sum() > 0 and not ref.overflow_flag(
                ref.shard_counts(ref.expert_counts(vidx, G), S), C):
            diverted += 1
    assert diverted >= 4   # the virtual-group pass really ran


def pin_error_measures():
    """The two tolerance measures on hand-computed arrays: normwise is the
    largest absolute error over the largest reference magnitude; the
    elementwise figure divides each error by its own reference magnitude,
    floored at 1e-3 of the largest."""
    r = np.array([4.0, -2.0, 1.0, 0.0])
    g = np.array([4.1, -2.0, 0.9, 0.002])
    # errors 0.1, 0, 0.1, 0.002; max |r| = 4
    assert math.isclose(ref.normwise_error(g, r), 0.1 / 4.0)
    # relative: 0.1/4, 0, 0.1/1, 0.002/max(0, 0.004) = 0.5
    assert math.isclose(ref.elementwise_error(g, r), 0.5)
    assert math.isclose(ref.elementwise_error(g[:3], r[:3]), 0.1)
    assert ref.elementwise_error(r, r) == 0.0
    assert ref.normwise_error(np.zeros(3), np.zeros(3)) == 0.0
    assert ref.elementwise_error(np.zeros(0), np.zeros(0)) == 0.0
    # the elementwise figure is never below the normwise one
    rng = _rng(3)
    for _ in range(20):
        a = rng.standard_normal(50)
        b = a + 1e-3 * rng.standard_normal(50)
        assert ref.elementwise_error(b, a) >= ref.normwise_error(b, a)


def pin_router_logits():
    """x Wr (+ offset): a one-hot token row reads out one row of Wr (so a
    transposed Wr or swapped operands fail); brute-force triple loop on a
    small case; the offset adds elementwise; no offset equals a zero one."""
    rng = _rng(21)
    H, E = 5, 3
    w = rng.standard_normal((H, E))
    x = np.eye(H)
    assert np.array_equal(ref.router_logits(x, w), w)
    x = rng.standard_normal((4, H))
    want = np.zeros((4, E))
    for t in range(4):
        for e in range(E):
            for h in range(H):
                want[t, e] += x[t, h] * w[h, e]
    assert np.allclose(ref.router_logits(x, w), want, rtol=1e-13, atol=1e-13)
    off = rng.standard_normal((4, E))
    assert np.allclose(ref.router_logits(x, w, off), want + off,
                       rtol=1e-13, atol=1e-13)
    assert np.array_equal(ref.router_logits(x, w, np.zeros((4, E))),
                          ref.router_logits(x, w))


def _ep_case(rng, N, Ts, E, k, H=3, F=4, shift=1.5):
    xs = [rng.standard_normal((T_r, H)) for T_r in Ts]
    Ls = [rng.standard_normal((T_r, E)) - shift * np.log(np.arange(E) + 1.0)
          for T_r in Ts]
    w = (rng.standard_normal((E, H, F)), rng.standard_normal((E, H, F)),
         rng.standard_normal((E, F, H)))
    return xs, Ls, w


def pin_ep_dispatch_plan():
    """Each source's send: every pick (t, j) appears once, in the row of
    token t bound for the rank that owns its expert, with that expert's
    local index and weight; the rows bound for a rank are the set of tokens
    with a pick there (brute force), ascending, each once."""
    rng = _rng(31)
    for _ in range(40):
        N = int(rng.choice([1, 2, 4]))
        E = N * int(rng.integers(1, 4))
        k = int(rng.integers(1, E + 1))
        T = int(rng.integers(0, 20))
        L = rng.standard_normal((T, E))
        idx, w, _ = ref.route(L, k) if T else (np.zeros((0, k), int),
                                              np.zeros((0, k)), False)
        p = ref.ep_dispatch(idx, w, E, N)
        Ed = E // N
        kk = min(k, Ed)
        assert p.send_idx.shape == (int(p.uniq_offsets[N]), kk)
        seen = set()
        for d in range(N):
            a, z = int(p.uniq_offsets[d]), int(p.uniq_offsets[d + 1])
            toks = [int(t) for t in p.uniq_tokens[a:z]]
            want = sorted({t for t in range(T)
                           for e in idx[t] if int(e) // Ed == d})
            assert toks == want
            for u, t in enumerate(toks):
                q = 0
                for j in range(k):      # the owned picks, in pick order
                    e = int(idx[t, j])
                    if e // Ed == d:
                        assert p.send_idx[a + u, q] == e - d * Ed
                        assert p.send_w[a + u, q] == w[t, j]
                        seen.add((t, j))
                        q += 1
                assert np.all(p.send_idx[a + u, q:] == -1)
                assert np.all(p.send_w[a + u, q:] == 0.0)
        assert seen == {(t, j) for t in range(T) for j in range(k)}
        assert p.uniq_offsets[N] == sum(
            len({int(e) // Ed for e in idx[t]}) for t in range(T))


def pin_ep_layer_equals_single_device():
    """fallback=layer over N ranks gives the single-device layer on the
    ranks' batches together ([PR5920 Tests]: outputs match the dropless
    model), with the same global overflow flag and the same pass count;
    cases that overflow and cases that do not, ranks with no tokens."""
    rng = _rng(32)
    over_seen = set()
    for _ in range(30):
        N = int(rng.choice([2, 4]))
        E = N * int(rng.choice([1, 2, 3]))
        k = int(rng.integers(1, min(E, 3) + 1))
        Ts = [int(rng.integers(0, 14)) for _ in range(N)]
        if sum(Ts) == 0:
            Ts[0] = 3
        factor = float(rng.choice([0.5, 1.0, 2.0, 4.0]))
        xs, Ls, w = _ep_case(rng, N, Ts, E, k)
        cfg = ref.MoEConfig(sum(Ts), 3, E, k, 4, N, factor)
        ys, over, n = ref.ep_layer(cfg, N, xs, Ls, ref.dense_weights(*w))
        single = ref.layer(cfg, np.concatenate(xs), np.concatenate(Ls),
                           ref.dense_weights(*w))
        assert over == single.overflow
        if over:
            C = ref.capacity(cfg.T, k, N, factor)
            assert n == len(ref.chunk_plan(cfg.T, k, E, N, C))
        assert np.allclose(np.concatenate(ys), single.y, rtol=1e-10,
                           atol=1e-10)
        over_seen.add(over)
    assert over_seen == {True, False}


def pin_ep_backward_equals_dropless_backward():
    """The EP layer's backward (fallback=layer over N ranks; the cotangent
    sent along the dispatch's dedup'd rows, token gradients returned and
    added, slot weight gradients returned, weight gradients summed over the
    fallback's passes) equals the dropless layer's backward on the ranks'
    batches together ([PR5920 Tests]), whether or not a shard overflows."""
    rng = _rng(36)
    over_seen = set()
    for i in range(24):
        N = int(rng.choice([2, 4]))
        E = N * int(rng.choice([1, 2, 3]))
        k = int(rng.integers(1, min(E, 3) + 1))
        Ts = [int(rng.integers(0, 10)) for _ in range(N)]
        if sum(Ts) == 0:
            Ts[0] = 3
        factor = float(rng.choice([0.5, 1.0, 2.0]))
        xs, Ls, w = _ep_case(rng, N, Ts, E, k)
        dys = [rng.standard_normal((T_r, 3)) for T_r in Ts]
        cfg = ref.MoEConfig(sum(Ts), 3, E, k, 4, N, factor,
                            renorm=bool(i % 3 == 0))
        _, over, n = ref.ep_layer(cfg, N, xs, Ls, ref.dense_weights(*w))
        over_seen.add(over)
        dxs, dls, dW = ref.ep_layer_backward(cfg, N, xs, Ls,
                                             ref.dense_weights(*w), dys)
        g = ref.layer_backward_dropless(cfg, np.concatenate(xs),
                                        np.concatenate(Ls), *w,
                                        np.concatenate(dys))
        for got, want in ((np.concatenate(dxs), g.dx),
                          (np.concatenate(dls), g.dlogits),
                          (dW[0], g.dwg), (dW[1], g.dwu), (dW[2], g.dwd)):
            assert np.allclose(got, want, rtol=1e-10, atol=1e-10)
    assert over_seen == {True, False}


def pin_ring_layer_equals_dropless():
    """The ring of experts (all-gather, local experts, reduce-scatter of the
    combine) gives the dropless layer on the ranks' batches together."""
    rng = _rng(33)
    for _ in range(20):
        N = int(rng.choice([2, 4]))
        E = N * int(rng.choice([1, 2]))
        k = int(rng.integers(1, min(E, 3) + 1))
        Ts = [int(rng.integers(0, 10)) for _ in range(N)]
        xs, Ls, w = _ep_case(rng, N, Ts, E, k)
        cfg = ref.MoEConfig(sum(Ts), 3, E, k, 4, N, 2.0)
        ys = ref.ring_layer(cfg, N, xs, Ls, ref.dense_weights(*w))
        for r in range(N):
            assert ys[r].shape == (Ts[r], 3)
        if sum(Ts):
            drop = ref.layer_dropless(cfg, np.concatenate(xs),
                                      np.concatenate(Ls),
                                      ref.dense_weights(*w))
            assert np.allclose(np.concatenate(ys), drop.y, rtol=1e-10,
                               atol=1e-10)


def pin_ring_backward_equals_dropless_backward():
    """The ring's backward (cotangent all-gather, each rank's experts
    differentiated over all tokens, partial dx summed at the owners, pick
    gradients taken from the experts' ranks) gives the dropless layer's
    gradients on the ranks' batches together -- whose backward is pinned by
    finite differences -- with both routings (softmax over all experts or
    renormalised over the k picks)."""
    rng = _rng(35)
    for i in range(16):
        N = int(rng.choice([2, 4]))
        E = N * int(rng.choice([1, 2]))
        k = int(rng.integers(1, min(E, 3) + 1))
        Ts = [int(rng.integers(0, 8)) for _ in range(N)]
        xs, Ls, w = _ep_case(rng, N, Ts, E, k)
        dys = [rng.standard_normal((T_r, 3)) for T_r in Ts]
        cfg = ref.MoEConfig(sum(Ts), 3, E, k, 4, N, 2.0, renorm=bool(i % 2))
        dxs, dls, dW = ref.ring_layer_backward(cfg, N, xs, Ls,
                                               ref.dense_weights(*w), dys)
        for r in range(N):
            assert dxs[r].shape == (Ts[r], 3) and dls[r].shape == (Ts[r], E)
        if not sum(Ts):
            assert all(not np.any(a) for a in dW)
            continue
        g = ref.layer_backward_dropless(cfg, np.concatenate(xs),
                                        np.concatenate(Ls), *w,
                                        np.concatenate(dys))
        for got, want in ((np.concatenate(dxs), g.dx),
                          (np.concatenate(dls), g.dlogits),
                          (dW[0], g.dwg), (dW[1], g.dwu), (dW[2], g.dwd)):
            assert np.allclose(got, want, rtol=1e-10, atol=1e-10)


ALL_PINS = [v for n, v in sorted(globals().items()) if n.startswith("pin_")]
