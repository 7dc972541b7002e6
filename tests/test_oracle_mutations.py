"""Planted mistakes in the oracle must fail at least one pin (CPU only).

Each mutant is the oracle's source with one plausible slip (a wrong tie
break, a floor turned ceil, a swapped operand, a dropped weight ...).  The
mutant is loaded as a separate module and the pins are run against it; the
test passes only if some pin rejects it.  The real oracle is not modified.
"""
import importlib.util
import os
import sys
import types

import pytest

from tests import oracle_pins

ORACLE_SRC = os.path.join(os.path.dirname(os.path.dirname(
    os.path.abspath(__file__))), "oracle", "moe_ref.py")

MUTANTS = {
    "ep_dest_by_modulo": (
        "            if any(e // Ed == d for e in picks):",
        "            if any(e % N == d for e in picks):"),
    "ep_return_unweighted": (
        "            out[i] += float(recv_w[i, j]) * y[q]",
        "            out[i] += y[q]"),
    "ep_flag_from_rank0_only": (
        "    for idx, _ in routes:\n        shard += shard_counts(",
        "    for idx, _ in routes[:1]:\n        shard += shard_counts("),
    "ring_partials_not_summed": (
        "        total += ep_expert_pass(", "        total = ep_expert_pass("),
    "router_offset_dropped": (
        "        out = out + np.asarray(offset, dtype=np.float64)",
        "        out = out + 0.0"),
    "router_weight_layout_misread": (
        "    out = np.matmul(x, w)\n",
        "    out = np.matmul(x, w.reshape(w.shape[1], w.shape[0]).T)\n"),
    "tie_to_higher_index": (
        "keyed = [(-clean_logit(float(row[e])), e) for e in range(E)]",
        "keyed = [(-clean_logit(float(row[e])), -e) for e in range(E)]"),
    "nan_not_cleaned": (
        "return v if math.isfinite(v) else -math.inf",
        "return v"),
    "always_renormalise": (
        "            p = softmax_f64(row)\n            w[t] = [p[e] for e in chosen]",
        "            w[t] = softmax_f64([row[e] for e in chosen])"),
    "capacity_ceil": (
        "c = math.floor(f * T * k / S)", "c = math.ceil(f * T * k / S)"),
    "flag_not_strict": (
        "return any(int(x) > C for x in r)",
        "return any(int(x) >= C for x in r)"),
    "strided_shards": (
        "for e in range(s * Es, (s + 1) * Es):",
        "for e in range(s, E, S):"),
    "inclusive_scan": (
        "        out[i] = run\n        run += int(x)\n",
        "        run += int(x)\n        out[i] = run\n"),
    "token_major_order": (
        "    rows.sort()\n", "    rows.sort(key=lambda q: (q[1], q[0]))\n"),
    "keep_one_extra_row": (
        "if C is None or rank_in_shard[s] < C:",
        "if C is None or rank_in_shard[s] <= C:"),
    "dedup_over_all_rows": (
        "    for (e, t, j) in kept:\n        uniq_sets[e // Es].add(t)",
        "    for (e, t, j) in rows:\n        uniq_sets[e // Es].add(t)"),
    "silu_sign": (
        "return z / (1.0 + np.exp(-z))", "return z / (1.0 + np.exp(z))"),
    "gate_up_swapped": ("    h = silu(g) * u\n    return h, np.matmul(h, wd)",
                        "    h = silu(u) * g\n    return h, np.matmul(h, wd)"),
    "backward_gate_up_swapped": (
        "    h = silu(g) * u\n    dh = dy @ wd.T",
        "    h = silu(u) * g\n    dh = dy @ wd.T"),
    "combine_ignores_weight": (
        "y[t] += float(topk_w[t, j]) * y_sorted[r]", "y[t] += y_sorted[r]"),
    "combine_skips_row_zero": (
        "            if r >= 0:\n"
        "                y[t] += float(topk_w[t, j]) * y_sorted[r]",
        "            if r > 0:\n"
        "                y[t] += float(topk_w[t, j]) * y_sorted[r]"),
    "chunk_ignores_shard_bound": (
        "c = max(1, C // worst_per_token)", "c = max(1, C // k)"),
    "dup_without_has_candidate": (
        "        cands = [e for e in range(r_max * Es, (r_max + 1) * Es)\n"
        "                 if not dup[e] and counts[e] > 0]\n",
        "        cands = [e for e in range(r_max * Es, (r_max + 1) * Es)\n"
        "                 if counts[e] > 0]\n"),
    "dup_moves_whole_gap": (
        "n = min(counts[e_star], (load[r_max] - load[r_min]) // 2)",
        "n = min(counts[e_star], load[r_max] - load[r_min])"),
    "reroute_never_diverts": (
        "            if seen[e] >= keep and plan.slot_of[e] >= 0:",
        "            if False:"),
    "reroute_first_rows": (
        "            if seen[e] >= keep and plan.slot_of[e] >= 0:",
        "            if seen[e] < int(plan.divert[e]) and plan.slot_of[e] >= 0:"),
    "silu_grad_wrong": (
        "    return s * (1.0 + z * (1.0 - s))",
        "    return s * (1.0 + z * s)"),
    "swiglu_backward_drops_u": (
        "    dg = dh * u * silu_grad(g)",
        "    dg = dh * silu_grad(g)"),
    "dy_sorted_unweighted": (
        "                dys[r] = w[t, j] * dy[t]",
        "                dys[r] = dy[t]"),
    "softmax_jacobian_sign": (
        "                dl[t, e] = p[e] * (dp[e] - dot)",
        "                dl[t, e] = p[e] * (dp[e] + dot)"),
    "dx_gate_only": (
        "    return dg @ wg.T + du @ wu.T, (x.T @ dg, x.T @ du, h.T @ dy)",
        "    return dg @ wg.T, (x.T @ dg, x.T @ du, h.T @ dy)"),
    "dwd_uses_x": (
        "    return dg @ wg.T + du @ wu.T, (x.T @ dg, x.T @ du, h.T @ dy)",
        "    return dg @ wg.T + du @ wu.T, (x.T @ dg, x.T @ du, "
        "x[:, :h.shape[1]].T @ dy)"),
    "dwu_uses_dg": (
        "    return dg @ wg.T + du @ wu.T, (x.T @ dg, x.T @ du, h.T @ dy)",
        "    return dg @ wg.T + du @ wu.T, (x.T @ dg, x.T @ dg, h.T @ dy)"),
    "duplicate_dw_not_summed": (
        "        dW[e] = dWe if e not in dW else tuple(",
        "        dW[e] = dWe if True else tuple("),
    "ep_bwd_dw_not_summed_over_passes": (
        "                dwg[e] += a\n",
        "                dwg[e] = a\n"),
    "ep_bwd_slot_gradient_to_first_pick": (
        "                        dtws[q][t, j] = dw_r[pos + u, s]",
        "                        dtws[q][t, own[0]] += dw_r[pos + u, s]"),
    "ring_bwd_partials_not_summed": (
        "        dx_all += part ",
        "        dx_all = part "),
    "ring_bwd_cotangent_unweighted": (
        "            dy_rows[q] = w_all[t, j] * dy_all[t]",
        "            dy_rows[q] = dy_all[t]"),
    "slot_uses_group_weights": (
        "        wg, wu, wd = weights(grp if gexp is None else int(gexp[grp]))",
        "        wg, wu, wd = weights(grp % cfg.E)"),
    "chunked_dw_not_summed": (
        "        out.dwg += g.dwg",
        "        out.dwg = g.dwg"),
    "wgrad_segment_base_dropped": (
        "            r0, r1 = base + int(off[g]), base + int(off[g + 1])",
        "            r0, r1 = int(off[g]), int(off[g + 1])"),
    "wgrad_duplicate_to_own_slot": (
        "            e = g if group_expert is None else int(group_expert[g])",
        "            e = g if group_expert is None else min(g, E - 1)"),
    "wgrad_operands_swapped": (
        "            dW[e] += P[r0:r1].T @ Q[r0:r1]",
        "            dW[e] += (Q[r0:r1].T @ P[r0:r1]).T[::-1, ::-1]"),
    "chunk_one_too_big": (
        "c = max(1, C // worst_per_token)",
        "c = max(1, C // worst_per_token + 1)"),
}


def _load_mutant(name, old, new):
    with open(ORACLE_SRC) as f:
        src = f.read()
    assert src.count(old) == 1, f"mutation site for {name} not unique"
    src = src.replace(old, new)
    modname = f"_oracle_mutant_{name}"
    mod = types.ModuleType(modname)
    mod.__file__ = ORACLE_SRC
    sys.modules[modname] = mod
    try:
        exec(compile(src, f"<mutant {name}>", "exec"), mod.__dict__)
    except Exception:
        del sys.modules[modname]
        raise
    return mod


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, monkeypatch):
    old, new = MUTANTS[name]
    mod = _load_mutant(name, old, new)
    try:
        monkeypatch.setattr(oracle_pins, "ref", mod)
        caught = None
        for pin in oracle_pins.ALL_PINS:
            try:
                pin()
            except Exception as exc:      # AssertionError or a crash
                caught = (pin.__name__, type(exc).__name__)
                break
        assert caught is not None, f"no pin catches mutant {name}"
    finally:
        sys.modules.pop(mod.__name__, None)


def test_real_oracle_passes_all_pins():
    for pin in oracle_pins.ALL_PINS:
        pin()
