"""GPU parity of the backward pass against the float64 oracle.

The layer backward (moe_layer_backward) in every mode, and the backward
entry points one by one (combine, route and permute transposes, the saved
forward GEMMs and the FFN backward).  Gradient buffers are pre-filled with
NaN so that a gradient the library forgot to write shows up.
"""
import numpy as np
import pytest
import torch

import mixture_experts_token_gb300 as moe
from oracle import moe_ref as ref
from synth import WORKLOADS, make_weights, make_x
from synth.workloads import make_dy
from tests.gpu_util import TOL, cfg_from, f64, host_logits, np_
from tests.parity_log import assert_close

pytestmark = pytest.mark.gpu

BWD = [
    WORKLOADS["tiny"],
    # ragged T, F % 256 != 0 (128-wide dgrad tiles), Zipf routing
    WORKLOADS["small"].with_(name="bwd_a", T=1000, H=512, E=8, k=2, F=384,
                             S=2, zipf_s=1.0),
    # H % 256 != 0 (128-wide tiles of dx_sorted and dWd), k=4, renorm
    WORKLOADS["small"].with_(name="bwd_b", T=777, H=384, E=16, k=4, F=256,
                             S=4, renorm=True, routing="uniform"),
]


def oracle_cfg(wl, **over):
    d = dict(T=wl.T, H=wl.H, E=wl.E, k=wl.k, F=wl.F, S=wl.S,
             ragged_buffer_factor=wl.factor, n_chunks=wl.n_chunks,
             renorm=wl.renorm)
    d.update(over)
    return ref.MoEConfig(**d)


def oracle_backward(mc, mode, x, L, W, dy):
    """The oracle's gradients of the mode moe_layer_backward runs."""
    if mode == moe.MOE_MODE_DROPLESS:
        return ref.layer_backward_dropless(mc, x, L, *W, dy), None
    if mode == moe.MOE_MODE_CAPPED:
        return ref.layer_backward_capped(mc, x, L, *W, dy), None
    idx, _, _ = ref.route(L, mc.k, mc.renorm)
    shard = ref.shard_counts(ref.expert_counts(idx, mc.E), mc.S)
    C = ref.capacity(mc.T, mc.k, mc.S, mc.ragged_buffer_factor)
    over = ref.overflow_flag(shard, C)
    if over:
        return ref.layer_backward_chunked(mc, x, L, *W, dy), True
    return ref.layer_backward_capped(mc, x, L, *W, dy), False


def setup(wl):
    x = make_x(wl, "cuda")
    L = host_logits(wl, x)
    W = make_weights(wl, "cuda")
    dy = make_dy(wl, "cuda")
    return x, L, W, dy


def gpu_layer_backward(cfg, x, L, W, dy, mode):
    T, H, E, F = cfg.T, cfg.H, cfg.E, cfg.F
    dev = "cuda"
    nan = float("nan")
    out = {
        "dx": torch.full((T, H), nan, dtype=x.dtype, device=dev),
        "dlogits": torch.full((T, E), nan, dtype=torch.float32, device=dev),
        "dwg": torch.full((E, H, F), nan, dtype=torch.float32, device=dev),
        "dwu": torch.full((E, H, F), nan, dtype=torch.float32, device=dev),
        "dwd": torch.full((E, F, H), nan, dtype=torch.float32, device=dev),
    }
    ws = moe.layer_workspace(cfg, moe.MOE_WS_LAYER_BACKWARD)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    Ld = torch.from_numpy(np.ascontiguousarray(L)).to(dev)
    info = moe.moe_layer_backward(cfg, x, Ld, *W, dy, out["dx"],
                                  out["dlogits"], out["dwg"], out["dwu"],
                                  out["dwd"], mode, ws, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return out, info


def compare(out, g, tol):
    pairs = [("dx", g.dx), ("dlogits", g.dlogits), ("dwg", g.dwg),
             ("dwu", g.dwu), ("dwd", g.dwd)]
    for name, want in pairs:
        got = f64(out[name])
        assert np.isfinite(got).all(), f"{name}: unwritten or non-finite"
        assert_close(got, want, tol, name)


MODES = [(moe.MOE_MODE_DROPLESS, 2.0), (moe.MOE_MODE_CAPPED, 1.0),
         (moe.MOE_MODE_FALLBACK_LAYER, 1.0),
         (moe.MOE_MODE_FALLBACK_LAYER, 50.0)]


@pytest.mark.parametrize("mode,factor", MODES,
                         ids=["dropless", "capped_f1", "fallback_f1",
                              "fallback_f50"])
@pytest.mark.parametrize("wl", BWD, ids=lambda w: w.name)
def test_layer_backward_matches_oracle(wl, mode, factor):
    x, L, W, dy = setup(wl)
    cfg = cfg_from(wl, factor=factor)
    out, info = gpu_layer_backward(cfg, x, L, W, dy, mode)
    mc = oracle_cfg(wl, ragged_buffer_factor=factor)
    g, over = oracle_backward(mc, mode, f64(x), L, [f64(w) for w in W],
                              f64(dy))
    if over is not None:
        assert info["overflow"] == int(over)
        if over:
            assert info["n_chunks"] == moe.moe_num_chunks(cfg)
    compare(out, g, TOL[wl.dtype])


@pytest.mark.parametrize("n_chunks", [20, 70], ids=["regrouped", "segments"])
def test_fallback_backward_many_chunks(n_chunks):
    """Many fallback chunks: 20 are regrouped into one row range per expert
    (the combine weights' gradient from the down dgrad); 70 are more than
    the regroup takes, so the combine backward reads a recomputed y_sorted
    and the weight gradients sum the row segments 16 at a time, the later
    batches adding into dW."""
    wl = BWD[1].with_(name="bwd_chunks", T=700, n_chunks=n_chunks)
    x, L, W, dy = setup(wl)
    cfg = cfg_from(wl, factor=1.0)
    out, info = gpu_layer_backward(cfg, x, L, W, dy,
                                   moe.MOE_MODE_FALLBACK_LAYER)
    assert info["overflow"] == 1 and info["n_chunks"] == n_chunks
    mc = oracle_cfg(wl, ragged_buffer_factor=1.0)
    g = ref.layer_backward_dropless(mc, f64(x), L, *[f64(w) for w in W],
                                    f64(dy))
    compare(out, g, TOL["bf16"])


def test_unused_expert_gets_zero_weight_gradient():
    """An expert no token picks: its dW is exactly zero (written, not left
    as it was)."""
    wl = BWD[1].with_(name="bwd_unused", T=300)
    x, L, W, dy = setup(wl)
    L = L.copy()
    L[:, 5] = -1.0e30
    cfg = cfg_from(wl)
    out, _ = gpu_layer_backward(cfg, x, L, W, dy, moe.MOE_MODE_DROPLESS)
    for name in ("dwg", "dwu", "dwd"):
        assert torch.count_nonzero(out[name][5]).item() == 0
    g = ref.layer_backward_dropless(oracle_cfg(wl), f64(x), L,
                                    *[f64(w) for w in W], f64(dy))
    compare(out, g, TOL["bf16"])


def test_zero_tokens_zero_weight_gradients():
    wl = BWD[1].with_(name="bwd_t0", T=0)
    cfg = cfg_from(wl)
    E, H, F = wl.E, wl.H, wl.F
    dw = [torch.full(s, float("nan"), device="cuda")
          for s in ((E, H, F), (E, H, F), (E, F, H))]
    W = make_weights(wl, "cuda")
    ws = moe.layer_workspace(cfg, moe.MOE_WS_LAYER_BACKWARD)
    moe.moe_layer_backward(cfg, None, None, *W, None, None, None, *dw,
                           moe.MOE_MODE_FALLBACK_LAYER, ws)
    torch.cuda.synchronize()
    for t in dw:
        assert torch.count_nonzero(t).item() == 0


@pytest.mark.parametrize("wl", BWD, ids=lambda w: w.name)
def test_backward_entry_points_stepwise(wl):
    """route -> permute -> saved GEMMs -> combine backward -> FFN backward
    -> permute backward -> route backward, each through its own entry
    point; then the FFN backward again with accumulate = 1 doubles dW."""
    x, L, W, dy = setup(wl)
    cfg = cfg_from(wl)
    T, H, E, k, F = wl.T, wl.H, wl.E, wl.k, wl.F
    R = T * k
    dt = x.dtype
    b = moe.alloc_step_buffers(cfg)
    Ld = torch.from_numpy(L).cuda()
    moe.moe_route(cfg, Ld, b["topk_idx"], b["topk_w"], b["status"])
    moe.moe_permute(cfg, x, b["topk_idx"], 0, b["x_sorted"], b["row_of"],
                    b["sorted_token"], b["group_offsets"], b["uniq_offsets"],
                    b["uniq_tokens"], b["expand_idx"], b["n_dropped"],
                    b["permute_ws"])
    g = torch.empty((R, F), dtype=dt, device="cuda")
    u = torch.empty_like(g)
    moe.moe_gmm_swiglu_saved(cfg, b["x_sorted"], b["group_offsets"], *W, g,
                             u, b["h"], b["y_sorted"], b["status"])
    dys = torch.empty((R, H), dtype=dt, device="cuda")
    dtw = torch.empty((T, k), dtype=torch.float32, device="cuda")
    moe.moe_combine_backward(cfg, dy, b["y_sorted"], b["row_of"],
                             b["topk_w"], dys, dtw)
    dxs = torch.empty((R, H), dtype=dt, device="cuda")
    dw = [torch.full(s, float("nan"), device="cuda")
          for s in ((E, H, F), (E, H, F), (E, F, H))]
    ws = moe.layer_workspace(cfg, moe.MOE_WS_GMM_BACKWARD)
    moe.moe_gmm_swiglu_backward(cfg, b["x_sorted"], b["group_offsets"], *W,
                                g, u, b["h"], dys, dxs, *dw, 0, ws,
                                b["status"])
    dx = torch.empty((T, H), dtype=dt, device="cuda")
    moe.moe_permute_backward(cfg, dxs, b["row_of"], dx)
    dl = torch.empty((T, E), dtype=torch.float32, device="cuda")
    moe.moe_route_backward(cfg, Ld, b["topk_idx"], dtw, dl)
    torch.cuda.synchronize()
    assert int(b["status"].item()) == 0
    want = ref.layer_backward_dropless(oracle_cfg(wl), f64(x), L,
                                       *[f64(w) for w in W], f64(dy))
    tol = TOL[wl.dtype]
    assert_close(f64(dtw), want.dtopk_w, tol, 'dtw')
    compare({"dx": dx, "dlogits": dl, "dwg": dw[0], "dwu": dw[1],
             "dwd": dw[2]}, want, tol)
    # saved g, u against the oracle's x_sorted W products (g = x Wg)
    xs = f64(b["x_sorted"])
    off = np_(b["group_offsets"]).astype(np.int64)
    wg = f64(W[0])
    gs = np.zeros((R, F))
    for e in range(E):
        gs[off[e]:off[e + 1]] = xs[off[e]:off[e + 1]] @ wg[e]
    assert_close(f64(g), gs, tol, 'g')
    # accumulate: a second backward adds the same gradient again.  bf16
    # adds the finished tile to dW (a + a: exact); fp32 continues its
    # accumulation from the old value (rounding differs in the last bits).
    first = [t.clone() for t in dw]
    moe.moe_gmm_swiglu_backward(cfg, b["x_sorted"], b["group_offsets"], *W,
                                g, u, b["h"], dys, dxs, *dw, 1, ws,
                                b["status"])
    torch.cuda.synchronize()
    for a, b2 in zip(first, dw):
        if wl.dtype == "bf16":
            assert torch.equal(b2, a * 2)
        else:
            scale = a.abs().max().item()
            assert torch.allclose(b2, a * 2, rtol=1e-5, atol=1e-6 * scale)


def test_combine_backward_exact_small():
    """dy_sorted rows are w * dy exactly rounded; dtopk_w is the fp32 dot
    product within fp32 rounding; dropped rows get a zero weight gradient."""
    wl = BWD[1].with_(name="cb", T=64)
    x, L, W, dy = setup(wl)
    cfg = cfg_from(wl, factor=0.5)
    b = moe.alloc_step_buffers(cfg)
    Ld = torch.from_numpy(L).cuda()
    moe.moe_route(cfg, Ld, b["topk_idx"], b["topk_w"], b["status"])
    moe.moe_permute(cfg, x, b["topk_idx"], 1, b["x_sorted"], b["row_of"],
                    b["sorted_token"], b["group_offsets"], b["uniq_offsets"],
                    b["uniq_tokens"], b["expand_idx"], b["n_dropped"],
                    b["permute_ws"])
    R = wl.T * wl.k
    ys = torch.randn((R, wl.H), device="cuda").to(x.dtype)
    dys = torch.zeros((R, wl.H), dtype=x.dtype, device="cuda")
    dtw = torch.full((wl.T, wl.k), float("nan"), device="cuda")
    moe.moe_combine_backward(cfg, dy, ys, b["row_of"], b["topk_w"], dys, dtw)
    torch.cuda.synchronize()
    row_of = np_(b["row_of"]).astype(np.int64)
    w = np_(b["topk_w"]).astype(np.float64)
    dyh, ysh, dysh, dtwh = f64(dy), f64(ys), f64(dys), f64(dtw)
    assert (row_of < 0).any()
    for t in range(wl.T):
        for j in range(wl.k):
            r = row_of[t, j]
            if r < 0:
                assert dtwh[t, j] == 0.0
                continue
            want = (w[t, j] * dyh[t]).astype(np.float32)
            want = torch.from_numpy(want).to(torch.bfloat16).double().numpy()
            assert np.array_equal(dysh[r], want)
            dot = float(dyh[t] @ ysh[r])
            assert abs(dtwh[t, j] - dot) <= 1e-5 * (np.abs(dyh[t]) @
                                                     np.abs(ysh[r]) + 1e-30)


@pytest.mark.parametrize("F", [512, 384], ids=["F512_256wide", "F384_128wide"])
def test_split_combine_backward(F):
    """The split combine backward moe_layer_backward uses: dy rows unscaled
    and each row's weight (exact copies); the down dgrad on them scales dh
    by the row's weight and writes per-column-tile dots of dy Wd^T with h;
    their ordered sum is each pick's weight gradient dy[t] . (h Wd), within
    the bf16-product bound of the float64 value; dg and du match the float64
    SwiGLU backward; and the regroup with the row weights writes exactly the
    weighted rows moe_combine_backward produces (dropped rows included)."""
    wl = BWD[1].with_(name="split", T=96, F=F)
    x, L, W, dy = setup(wl)
    cfg = cfg_from(wl, factor=0.5)
    b = moe.alloc_step_buffers(cfg)
    Ld = torch.from_numpy(L).cuda()
    moe.moe_route(cfg, Ld, b["topk_idx"], b["topk_w"], b["status"])
    moe.moe_permute(cfg, x, b["topk_idx"], 1, b["x_sorted"], b["row_of"],
                    b["sorted_token"], b["group_offsets"], b["uniq_offsets"],
                    b["uniq_tokens"], b["expand_idx"], b["n_dropped"],
                    b["permute_ws"])
    R, H = wl.T * wl.k, wl.H
    g = torch.empty((R, F), dtype=x.dtype, device="cuda")
    u, h = torch.empty_like(g), torch.empty_like(g)
    ys = torch.empty((R, H), dtype=x.dtype, device="cuda")
    moe.moe_gmm_swiglu_saved(cfg, b["x_sorted"], b["group_offsets"], *W, g,
                             u, h, ys, b["status"])
    parts = moe.moe_row_dot_parts(cfg)
    assert parts == (F // 256 if F % 256 == 0 else F // 128)
    dyr = torch.zeros((R, H), dtype=x.dtype, device="cuda")
    wrow = torch.full((R,), float("nan"), device="cuda")
    moe.moe_combine_backward_rows(cfg, dy, b["row_of"], b["topk_w"], dyr,
                                  wrow)
    dg = torch.empty_like(g)
    du = torch.empty_like(g)
    rdot = torch.full((R * parts,), float("nan"), device="cuda")
    moe.moe_gmm_down_dgrad_rows(cfg, b["group_offsets"], W[2], g, u, h, dyr,
                                wrow, dg, du, rdot, b["status"])
    dtw = torch.full((wl.T, wl.k), float("nan"), device="cuda")
    moe.moe_combine_weight_grad(cfg, b["row_of"], rdot, dtw)
    # the weighted rows the other form writes, and the regroup's scaling
    dys_w = torch.zeros_like(dyr)
    dtw_w = torch.empty_like(dtw)
    moe.moe_combine_backward(cfg, dy, ys, b["row_of"], b["topk_w"], dys_w,
                             dtw_w)
    off = b["group_offsets"]
    rr = R + 16 * wl.E
    bufs = [torch.zeros((rr, n), dtype=x.dtype, device="cuda")
            for n in (H, F, F, F, H)]
    off2 = torch.empty(wl.E + 1, dtype=torch.int32, device="cuda")
    moe.moe_regroup_rows(cfg, [(off, 0)], rr, b["x_sorted"], dg, du, h, dyr,
                         *bufs, off2, w_row=wrow)
    bufs_w = [torch.zeros_like(t) for t in bufs]
    moe.moe_regroup_rows(cfg, [(off, 0)], rr, b["x_sorted"], dg, du, h,
                         dys_w, *bufs_w, off2)
    torch.cuda.synchronize()
    assert int(b["status"].item()) == 0
    assert torch.equal(bufs[4], bufs_w[4])
    row_of = np_(b["row_of"]).astype(np.int64)
    w = np_(b["topk_w"]).astype(np.float64)
    assert (row_of < 0).any()
    dyh, dyrh, hh = f64(dy), f64(dyr), f64(h)
    wd = f64(W[2])
    goff = np_(off)
    expert = np.searchsorted(goff, np.arange(R), side="right") - 1
    dtwh = f64(dtw)
    for t in range(wl.T):
        for j in range(wl.k):
            r = row_of[t, j]
            if r < 0:
                assert dtwh[t, j] == 0.0
                continue
            assert np.array_equal(dyrh[r], dyh[t])
            assert float(np_(wrow)[r]) == np.float32(w[t, j])
            e = expert[r]
            dh_u = wd[e] @ dyh[t]                    # dy Wd^T, float64
            want = float(dh_u @ hh[r])
            bound = 2.0 ** -8 * float(np.abs(wd[e]) @ np.abs(dyh[t]) @
                                      np.abs(hh[r])) + 1e-30
            assert abs(dtwh[t, j] - want) <= bound, (t, j)
    kept = [r for r in range(R) if r < goff[-1]]
    gh, uh = f64(g)[kept], f64(u)[kept]
    dh = np.stack([float(np_(wrow)[r]) * (wd[expert[r]] @ dyrh[r])
                   for r in kept])
    s_ = 1.0 / (1.0 + np.exp(-gh))
    assert_close(f64(dg)[kept], dh * uh * s_ * (1.0 + gh * (1.0 - s_)),
                 2e-2, "split dg")
    assert_close(f64(du)[kept], dh * gh * s_, 2e-2, "split du")
    assert_close(f64(dtw), f64(dtw_w), 2e-2, "split dtopk_w vs dy . y_sorted")


def test_regroup_rows_layout():
    """moe_regroup_rows: group e of the output holds e's rows of every range
    in range order (byte copies), starts at the exclusive scan of the
    16-rounded group sizes, and its pad rows are zero."""
    E, H, F, k, T = 6, 256, 128, 2, 300
    cfg = cfg_from(BWD[1], T=T, H=H, E=E, k=k, F=F, S=2)
    rng = np.random.default_rng(3)
    R = T * k
    # three ranges: rows [base, base + sum(counts)) grouped by expert
    counts = [rng.integers(0, 60, size=E) for _ in range(3)]
    counts[1][2] = 0
    counts[2][:] = 0
    counts[2][E - 1] = 17
    bases, offs, b0 = [], [], 0
    for cnt in counts:
        off = np.concatenate([[0], np.cumsum(cnt)]).astype(np.int32)
        bases.append(b0)
        offs.append(torch.from_numpy(off).cuda())
        b0 += int(off[-1]) + 5          # a gap of foreign rows between ranges
    assert b0 <= R
    src = {n: torch.randn((R, w), device="cuda").to(torch.bfloat16)
           for n, w in (("xs", H), ("dg", F), ("du", F), ("h", F),
                        ("dys", H))}
    rr = R + 16 * E
    out = {n: torch.full((rr, t.shape[1]), float("nan"), device="cuda",
                         dtype=torch.bfloat16) for n, t in src.items()}
    off2 = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    segs = list(zip(offs, bases))
    moe.moe_regroup_rows(cfg, segs, rr, src["xs"], src["dg"], src["du"],
                         src["h"], src["dys"], out["xs"], out["dg"],
                         out["du"], out["h"], out["dys"], off2)
    torch.cuda.synchronize()
    tot = sum(counts)
    want_off = np.concatenate([[0], np.cumsum((tot + 15) // 16 * 16)])
    assert np.array_equal(np_(off2), want_off)
    for name in src:
        s_, o_ = src[name].cpu(), out[name].cpu()
        for e in range(E):
            rows = []
            for cnt, base, off in zip(counts, bases, offs):
                a = base + int(np_(off)[e])
                rows += list(range(a, a + int(cnt[e])))
            g0 = int(want_off[e])
            if rows:
                assert torch.equal(o_[g0:g0 + len(rows)], s_[rows]), (name, e)
            pad = o_[g0 + len(rows):int(want_off[e + 1])]
            assert torch.count_nonzero(pad.float()).item() == 0, (name, e)


RED = [
    # bf16, skewed toward shard 0 so the plan diverts rows into slots
    WORKLOADS["small"].with_(name="red_a", T=1200, H=256, E=16, k=2, F=256,
                             S=4, zipf_s=1.2),
    # fp32 tiny layer (CUDA-core path), routed by x Wr
    WORKLOADS["tiny"].with_(name="red_tiny"),
]


@pytest.mark.parametrize("B,factor", [(1, 2.0), (2, 2.0), (2, 0.6)],
                         ids=["B1_f2", "B2_f2", "B2_f06"])
@pytest.mark.parametrize("wl", RED, ids=lambda w: w.name)
def test_layer_backward_redundant_fallback(wl, B, factor):
    """fallback=layer with duplicate-expert slots: plan, reroute, check on
    the diverted loads; the capped pass over the virtual groups (a slot's
    rows add into its expert's weight gradient) or the plain chunks."""
    x, L, W, dy = setup(wl)
    cfg = cfg_from(wl, factor=factor, redundant_slots=B)
    out, info = gpu_layer_backward(cfg, x, L, W, dy,
                                   moe.MOE_MODE_FALLBACK_LAYER)
    mc = oracle_cfg(wl, ragged_buffer_factor=factor)
    idx, _, _ = ref.route(L, wl.k, wl.renorm)
    plan = ref.plan_duplication(ref.expert_counts(idx, wl.E), wl.S, B)
    vidx = ref.reroute(idx, plan, wl.E, wl.S)
    G = wl.S * (wl.E // wl.S + B)
    C = ref.capacity(wl.T, wl.k, wl.S, factor)
    over = ref.overflow_flag(
        ref.shard_counts(ref.expert_counts(vidx, G), wl.S), C)
    assert info["overflow"] == int(over)
    g = ref.layer_redundant_backward(mc, f64(x), L, *[f64(w) for w in W],
                                     f64(dy), B)
    compare(out, g, TOL[wl.dtype])


@pytest.mark.parametrize("wl", RED, ids=lambda w: w.name)
def test_layer_backward_redundant_capped(wl):
    """Capped mode with slots: the capped pass over the plan's virtual
    groups, drops included, against the oracle's pass over the same
    groups."""
    B, factor = 1, 0.7
    x, L, W, dy = setup(wl)
    cfg = cfg_from(wl, factor=factor, redundant_slots=B)
    out, _ = gpu_layer_backward(cfg, x, L, W, dy, moe.MOE_MODE_CAPPED)
    mc = oracle_cfg(wl, ragged_buffer_factor=factor)
    idx, _, _ = ref.route(L, wl.k, wl.renorm)
    plan = ref.plan_duplication(ref.expert_counts(idx, wl.E), wl.S, B)
    vidx = ref.reroute(idx, plan, wl.E, wl.S)
    G = wl.S * (wl.E // wl.S + B)
    C = ref.capacity(wl.T, wl.k, wl.S, factor)
    assert ref.permute_indices(vidx, G, wl.S, C).n_dropped > 0
    g = ref.layer_pass_backward(mc, f64(x), L, *[f64(w) for w in W], f64(dy),
                                C, groups=(vidx, G, plan.group_expert))
    compare(out, g, TOL[wl.dtype])
