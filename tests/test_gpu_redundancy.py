"""GPU parity: dynamic redundant experts (moe_plan_duplication,
moe_permute_planned, moe_gmm_swiglu_mapped, moe_layer with slots).

The plan and the planned permute are integer work and must equal the
oracle bit for bit; the mapped GEMM is within the bf16/fp32 tolerance; and
the layer with slots must equal the dropless layer bit for bit whenever it
takes the capped path (a duplicate computes its rows with its expert's
weights, and a row's result does not depend on its group or tile).
"""
import numpy as np
import pytest
import torch

import mixture_experts_token_gb300 as moe
from oracle import moe_ref as ref
from synth import WORKLOADS, make_weights, make_x, sweep_workload
from tests.gpu_util import (TOL, cfg_from, compare_permutation, f64,
                            expert_accessor, gpu_route, host_logits, np_)
from tests.parity_log import assert_close

pytestmark = pytest.mark.gpu


def gpu_plan(cfg, counts):
    E, S = cfg.E, cfg.S
    G = E + S * cfg.redundant_slots
    d = {n: torch.full((m,), -7, dtype=torch.int32, device="cuda")
         for n, m in (("divert", E), ("slot_of", E), ("group_expert", G),
                      ("after", S), ("flag", 1))}
    c = torch.from_numpy(np.asarray(counts, dtype=np.int32)).cuda()
    moe.moe_plan_duplication(cfg, c, d["divert"], d["slot_of"],
                             d["group_expert"], d["after"], d["flag"])
    torch.cuda.synchronize()
    return d


def check_plan(cfg, counts):
    d = gpu_plan(cfg, counts)
    p = ref.plan_duplication(np.asarray(counts), cfg.S, cfg.redundant_slots)
    assert np.array_equal(np_(d["divert"]), p.divert)
    assert np.array_equal(np_(d["slot_of"]), p.slot_of)
    assert np.array_equal(np_(d["group_expert"]), p.group_expert)
    assert np.array_equal(np_(d["after"]), p.loads_after)
    C = ref.capacity(cfg.T, cfg.k, cfg.S, cfg.ragged_buffer_factor)
    assert int(np_(d["flag"])[0]) == int(ref.overflow_flag(p.loads_after, C))
    return d, p


def test_plan_hand_cases():
    for counts, S, B in (([8, 0, 0, 0, 0, 0, 0, 0], 2, 1),
                         ([100, 0], 2, 4),          # has_candidate stop
                         ([6, 9, 2, 0, 0, 0], 3, 1),
                         ([0, 0, 0, 0], 2, 3),      # nothing to move
                         ([5, 5, 5, 5], 4, 2)):     # already balanced
        E = len(counts)
        cfg = moe.make_config(max(1, sum(counts)), 64, E, 1, 128, S, 2.0,
                              redundant_slots=B)
        check_plan(cfg, counts)


@pytest.mark.parametrize("B", [1, 2, 4])
@pytest.mark.parametrize("wl", [WORKLOADS["small"], WORKLOADS["dsv3"],
                                sweep_workload(4096, "adversarial"),
                                sweep_workload(16384, "zipf")],
                         ids=lambda w: w.name)
def test_plan_and_permute_parity(wl, B):
    wl = wl.with_(redundant_slots=B)
    cfg = cfg_from(wl)
    x = make_x(wl, "cuda")
    L = host_logits(wl, x)
    idx, _ = gpu_route(cfg, L)
    oi, _, _ = ref.route(L, wl.k)
    assert np.array_equal(np_(idx), oi)
    counts = ref.expert_counts(oi, wl.E)
    d, p = check_plan(cfg, counts)
    G = wl.E + wl.S * B
    vidx = ref.reroute(oi, p, wl.E, wl.S)
    C = ref.capacity(wl.T, wl.k, wl.S, wl.factor)
    for capped in (True, False):
        bufs = moe.alloc_step_buffers(cfg)
        moe.moe_permute_planned(cfg, x, idx, capped, d["divert"],
                                d["slot_of"], bufs["x_sorted"],
                                bufs["row_of"], bufs["sorted_token"],
                                bufs["group_offsets"], bufs["uniq_offsets"],
                                bufs["uniq_tokens"], bufs["expand_idx"],
                                bufs["n_dropped"], bufs["permute_ws"])
        torch.cuda.synchronize()
        want = ref.permute_indices(vidx, G, wl.S, C if capped else None)
        compare_permutation(bufs, want, x.cpu() if wl.T <= 8192 else None)
        # the same plan through the two halves of the permute
        b2 = moe.alloc_step_buffers(cfg)
        moe.moe_permute_tables(cfg, idx, capped, b2["row_of"],
                               b2["sorted_token"], b2["group_offsets"],
                               b2["uniq_offsets"], b2["n_dropped"],
                               b2["permute_ws"], divert=d["divert"],
                               slot_of=d["slot_of"])
        moe.moe_permute_scatter(cfg, x, b2["row_of"], b2["uniq_offsets"],
                                b2["x_sorted"], b2["uniq_tokens"],
                                b2["expand_idx"], b2["permute_ws"])
        torch.cuda.synchronize()
        compare_permutation(b2, want, x.cpu() if wl.T <= 8192 else None)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_gmm_mapped_parity(dtype):
    rng = np.random.default_rng(0)
    E, H, F = 6, 256, 256
    sizes = [40, 0, 130, 7, 200, 1, 90, 0, 64, 3]     # 10 groups
    gexp = [0, 1, 2, 3, 4, 5, 2, -1, 4, 0]           # groups 2/6, 4/8 share
    G = len(sizes)
    R = sum(sizes)
    dt = torch.float32 if dtype == "f32" else torch.bfloat16
    xs = torch.randn(R, H, device="cuda").to(dt)
    W = [(torch.randn(E, *shp, device="cuda") * 0.05).to(dt)
         for shp in ((H, F), (H, F), (F, H))]
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    cfg = moe.make_config(R, H, E, 1, F, 1, 2.0, 0, dtype)
    h = torch.zeros(R, F, dtype=dt, device="cuda")
    ys = torch.zeros(R, H, dtype=dt, device="cuda")
    moe.moe_gmm_swiglu_mapped(cfg, G, torch.tensor(gexp, dtype=torch.int32,
                                                    device="cuda"),
                              xs, torch.from_numpy(off).cuda(), *W, h, ys)
    torch.cuda.synchronize()
    weights = ref.mapped_weights(ref.dense_weights(*(f64(w) for w in W)),
                                 np.array(gexp))
    want_h, want_y = ref.grouped_ffn(f64(xs), off, weights)
    assert_close(f64(h), want_h, TOL[dtype], 'h')
    assert_close(f64(ys), want_y, TOL[dtype], 'ys')


def run_layer(cfg, wl, x, Ld, W, mode):
    y = torch.empty((wl.T, wl.H), dtype=x.dtype, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    info = moe.moe_layer(cfg, x, Ld, *W, y, mode, moe.layer_workspace(cfg),
                         status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return y, info


@pytest.mark.parametrize("wl,B", [(WORKLOADS["small"], 1),
                                  (WORKLOADS["small"], 2),
                                  (WORKLOADS["dsv3"], 1),
                                  (WORKLOADS["dsv3"], 2),
                                  (WORKLOADS["dsv3"], 4)],
                         ids=["small-B1", "small-B2", "dsv3-B1", "dsv3-B2",
                              "dsv3-B4"])
def test_layer_with_slots(wl, B):
    wl = wl.with_(redundant_slots=B)
    cfg = cfg_from(wl)
    x = make_x(wl, "cuda")
    L = host_logits(wl, x)
    Ld = torch.from_numpy(L).cuda()
    W = make_weights(wl, "cuda")
    oi, ow, _ = ref.route(L, wl.k)
    p = ref.plan_duplication(ref.expert_counts(oi, wl.E), wl.S, B)
    C = ref.capacity(wl.T, wl.k, wl.S, wl.factor)
    over = ref.overflow_flag(p.loads_after, C)
    y, info = run_layer(cfg, wl, x, Ld, W, moe.MOE_MODE_FALLBACK_LAYER)
    assert info["overflow"] == int(over)
    y_drop, _ = run_layer(cfg, wl, x, Ld, W, moe.MOE_MODE_DROPLESS)
    if not over:
        # capped pass over the virtual groups dropped nothing: same bits
        assert torch.equal(y, y_drop)
    # against the oracle on sampled tokens
    toks = np.sort(np.random.default_rng(2).choice(wl.T, 10, replace=False))
    tt = torch.from_numpy(toks).cuda()
    want = ref.token_outputs(f64(x[tt]), oi[toks], ow[toks],
                             expert_accessor(*W))
    assert_close(f64(y[tt]), want, 2e-2, 'y[tt]')
    # the graph gives the same bits
    yg = torch.zeros_like(y)
    ws = moe.layer_workspace(cfg)
    g = moe.MoeLayerGraph(cfg, x, Ld, *W, yg, ws)
    g.launch()
    torch.cuda.synchronize()
    assert torch.equal(yg, y)
    g.close()


def test_small_layer_with_slots_full_compare():
    wl = WORKLOADS["small"].with_(redundant_slots=2)
    cfg = cfg_from(wl)
    x = make_x(wl, "cuda")
    L = host_logits(wl, x)
    W = make_weights(wl, "cuda")
    y, info = run_layer(cfg, wl, x, torch.from_numpy(L).cuda(), W,
                        moe.MOE_MODE_FALLBACK_LAYER)
    mc = ref.MoEConfig(wl.T, wl.H, wl.E, wl.k, wl.F, wl.S, wl.factor)
    want = ref.layer_redundant(mc, f64(x), L,
                               ref.dense_weights(*(f64(w) for w in W)), 2)
    assert info["overflow"] == int(want.overflow)
    assert_close(f64(y), want.y, 2e-2, 'y')
