"""GPU parity of expert parallelism across ranks, with the ranks as logical
ranks of one GPU (LoopbackTransport: the exchanges are device copies, no
kernel waits on another rank's).

* The dispatch of every source rank -- the dedup sets per destination
  (uniq_offsets, uniq_tokens), the send rows and their expert slots -- must
  equal the oracle's ep_dispatch bit for bit (weights within 1e-4), and
  every send row must be a byte copy of its token's row.
* The EP layer (fallback=layer) must match the oracle's ep_layer per rank
  within the layer tolerance, with the same global flag and pass count, in
  both branches; the ring of experts must match ring_layer.
"""
import numpy as np
import pytest
import torch

import mixture_experts_token_gb300 as moe
from mixture_experts_token_gb300 import ep
from oracle import moe_ref as ref
from synth import WORKLOADS, make_weights, make_x
from tests.gpu_util import TOL, f64, host_logits, np_
from tests.parity_log import assert_close, assert_close_device

pytestmark = pytest.mark.gpu


def rank_inputs(wl, Ts, seed=0):
    xs, Ls = [], []
    for r, T_r in enumerate(Ts):
        w = wl.with_(T=T_r, seed=seed + 101 * r)
        x = make_x(w, "cuda")
        xs.append(x)
        Ls.append(host_logits(w, x) if T_r else
                  np.zeros((0, wl.E), dtype=np.float32))
    return xs, Ls


def gcfg(wl, Ts, N, factor):
    return moe.make_config(sum(Ts), wl.H, wl.E, wl.k, wl.F, N, factor, 0,
                           wl.dtype, wl.renorm)


CASES = [
    # (workload, ranks, tokens per rank, factor)
    (WORKLOADS["small"].with_(name="n4", H=256, F=256, E=16, k=4, S=4), 4,
     [300, 0, 517, 128], 2.0),
    (WORKLOADS["small"].with_(name="n4_ovf", H=256, F=256, E=16, k=4, S=4,
                              zipf_s=1.5), 4, [400, 250, 333, 90], 1.0),
    (WORKLOADS["small"].with_(name="n2_k1", H=384, F=128, E=8, k=1, S=2),
     2, [700, 1], 2.0),
    (WORKLOADS["tiny"].with_(name="tiny_n2", S=2), 2, [128, 128], 2.0),
    # fewer experts per rank than picks (E/S = 2 < k = 4): two slots per
    # send row, a token's picks split over several ranks or two on one
    (WORKLOADS["small"].with_(name="n4_k4_e2", H=256, F=256, E=8, k=4, S=4,
                              zipf_s=1.2), 4, [200, 150, 0, 333], 1.5),
    (WORKLOADS["small"].with_(name="n8_e256", H=512, F=256, E=256, k=8,
                              S=8, zipf_s=1.2), 8,
     [256, 200, 300, 100, 64, 256, 1, 180], 2.0),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: c[0].name)
def test_ep_dispatch_matches_oracle(case):
    wl, N, Ts, factor = case
    xs, Ls = rank_inputs(wl, Ts)
    cfg = gcfg(wl, Ts, N, factor)
    kk = min(wl.k, wl.E // N)
    for r in range(N):
        T_r = Ts[r]
        if T_r == 0:
            continue
        sc = cfg.with_(T=T_r, ragged_buffer_factor=-1.0)
        b = moe.alloc_step_buffers(sc)
        moe.moe_route(sc, torch.from_numpy(Ls[r]).cuda(), b["topk_idx"],
                      b["topk_w"])
        moe.moe_permute_tables(sc, b["topk_idx"], False, b["row_of"],
                               b["sorted_token"], b["group_offsets"],
                               b["uniq_offsets"], b["n_dropped"],
                               b["permute_ws"])
        moe.moe_permute_scatter(sc, None, b["row_of"], b["uniq_offsets"],
                                None, b["uniq_tokens"], b["expand_idx"],
                                b["permute_ws"])
        rows = T_r * min(wl.k, N)
        xsend = torch.zeros((rows, wl.H), dtype=xs[r].dtype, device="cuda")
        sidx = torch.full((rows, kk), -7, dtype=torch.int32, device="cuda")
        sw = torch.full((rows, kk), -7.0, dtype=torch.float32, device="cuda")
        moe.moe_ep_dispatch_pack(sc, xs[r], b["topk_idx"], b["topk_w"],
                                 b["uniq_offsets"], b["uniq_tokens"], xsend,
                                 sidx, sw)
        torch.cuda.synchronize()
        oi, ow, _ = ref.route(Ls[r], wl.k)
        assert np.array_equal(np_(b["topk_idx"]), oi)
        p = ref.ep_dispatch(oi, ow, wl.E, N)
        U = int(p.uniq_offsets[N])
        assert np.array_equal(np_(b["uniq_offsets"]), p.uniq_offsets)
        assert np.array_equal(np_(b["uniq_tokens"])[:U], p.uniq_tokens)
        assert np.array_equal(np_(sidx)[:U], p.send_idx)
        assert_close(np_(sw)[:U], p.send_w, 1e-4, f"send_w rank {r}")
        tok = torch.from_numpy(p.uniq_tokens.astype(np.int64)).cuda()
        assert torch.equal(xsend[:U], xs[r][tok])
        assert torch.all(sidx[U:] == -7)       # rows past U untouched
        # the return map: row_of_ret[t, d] = the send row of (t, d)
        rr = torch.empty((T_r, N), dtype=torch.int32, device="cuda")
        moe.moe_ep_return_map(sc, b["uniq_offsets"], b["uniq_tokens"], rr)
        want = -np.ones((T_r, N), dtype=np.int64)
        for d in range(N):
            for i in range(int(p.uniq_offsets[d]), int(p.uniq_offsets[d + 1])):
                want[int(p.uniq_tokens[i]), d] = i
        assert np.array_equal(np_(rr), want)


def weights_of(wl, N):
    W = make_weights(wl, "cuda")
    return W, ep.local_weights(*W, N)


@pytest.mark.parametrize("case", CASES, ids=lambda c: c[0].name)
def test_ep_layer_matches_oracle(case):
    wl, N, Ts, factor = case
    xs, Ls = rank_inputs(wl, Ts)
    cfg = gcfg(wl, Ts, N, factor)
    W, per_rank = weights_of(wl, N)
    layer = ep.EPLayer(cfg, ep.LoopbackTransport(N), per_rank)
    ys = layer.forward(xs, [torch.from_numpy(L).cuda() for L in Ls])
    torch.cuda.synchronize()
    mc = ref.MoEConfig(sum(Ts), wl.H, wl.E, wl.k, wl.F, N, factor, 0,
                       wl.renorm)
    want, over, n = ref.ep_layer(mc, N, [f64(x) for x in xs], Ls,
                                 ref.dense_weights(*(f64(w) for w in W)))
    assert layer.info["overflow"] == int(over)
    assert layer.info["n_chunks"] == n
    tol = TOL[wl.dtype]
    got = np.concatenate([f64(y) for y in ys])
    assert_close(got, np.concatenate(want), tol,
                 f"EP y (N={N}, overflow={int(over)}, passes={n})")
    for r in range(N):
        if Ts[r]:
            assert_close(f64(ys[r]), want[r], tol, f"EP y rank {r}")


@pytest.mark.parametrize("case", CASES[:3] + CASES[4:],
                         ids=lambda c: c[0].name)
def test_ep_layer_matches_single_gpu_layer(case):
    """The EP layer over N logical ranks and moe_layer on the ranks'
    batches together agree within the tolerance (the EP combine rounds each
    destination's partial row to the layer dtype before the source adds
    them, so the bits may differ)."""
    wl, N, Ts, factor = case
    xs, Ls = rank_inputs(wl, Ts)
    cfg = gcfg(wl, Ts, N, factor)
    W, per_rank = weights_of(wl, N)
    ys = ep.EPLayer(cfg, ep.LoopbackTransport(N), per_rank).forward(
        xs, [torch.from_numpy(L).cuda() for L in Ls])
    x_all = torch.cat(xs)
    L_all = torch.from_numpy(np.concatenate(Ls)).cuda()
    y1 = torch.empty_like(x_all)
    moe.moe_layer(cfg, x_all, L_all, *W, y1, moe.MOE_MODE_FALLBACK_LAYER,
                  moe.layer_workspace(cfg))
    torch.cuda.synchronize()
    assert_close(f64(torch.cat(ys)), f64(y1), TOL[wl.dtype],
                 "EP y vs single-GPU moe_layer")


@pytest.mark.parametrize("case", CASES, ids=lambda c: c[0].name)
def test_ring_layer_matches_oracle(case):
    wl, N, Ts, factor = case
    xs, Ls = rank_inputs(wl, Ts)
    cfg = gcfg(wl, Ts, N, factor)
    W, per_rank = weights_of(wl, N)
    ys = ep.RingLayer(cfg, ep.LoopbackTransport(N), per_rank).forward(
        xs, [torch.from_numpy(L).cuda() for L in Ls])
    torch.cuda.synchronize()
    mc = ref.MoEConfig(sum(Ts), wl.H, wl.E, wl.k, wl.F, N, factor, 0,
                       wl.renorm)
    want = ref.ring_layer(mc, N, [f64(x) for x in xs], Ls,
                          ref.dense_weights(*(f64(w) for w in W)))
    assert_close(np.concatenate([f64(y) for y in ys]),
                 np.concatenate(want), TOL[wl.dtype], f"ring y (N={N})")


@pytest.mark.parametrize("case", CASES[:5], ids=lambda c: c[0].name)
def test_ep_backward_matches_oracle(case):
    """The EP layer's backward over logical ranks (the forward recomputed
    pass by pass; the cotangent sent along the dispatch's dedup'd rows,
    token gradients returned and added, each slot's weight gradient back at
    its pick, weight gradients summed over the passes, the router backward
    on each rank) against the oracle's EP backward -- in the fallback too
    (n4_ovf overflows) -- and, for the token and router gradients, against
    moe_layer_backward on the ranks' batches together."""
    wl, N, Ts, factor = case
    xs, Ls = rank_inputs(wl, Ts)
    cfg = gcfg(wl, Ts, N, factor)
    W, per_rank = weights_of(wl, N)
    g = torch.Generator(device="cuda").manual_seed(78)
    dys = [torch.randn((T_r, wl.H), generator=g, device="cuda").to(x.dtype)
           for T_r, x in zip(Ts, xs)]
    Lt = [torch.from_numpy(L).cuda() for L in Ls]
    layer = ep.EPLayer(cfg, ep.LoopbackTransport(N), per_rank)
    dxs, dls, dWs = layer.backward(xs, Lt, dys)
    torch.cuda.synchronize()
    mc = ref.MoEConfig(sum(Ts), wl.H, wl.E, wl.k, wl.F, N, factor, 0,
                       wl.renorm)
    _, over, n = ref.ep_layer(mc, N, [f64(x) for x in xs], Ls,
                              ref.dense_weights(*(f64(w) for w in W)))
    assert layer.info["overflow"] == int(over)
    assert layer.info["n_chunks"] == n
    wdx, wdl, wdW = ref.ep_layer_backward(
        mc, N, [f64(x) for x in xs], Ls,
        ref.dense_weights(*(f64(w) for w in W)), [f64(d) for d in dys])
    tol = TOL[wl.dtype]
    assert_close(np.concatenate([f64(d) for d in dxs]), np.concatenate(wdx),
                 tol, f"EP dx (N={N}, passes={n})")
    assert_close(np.concatenate([f64(d) for d in dls]), np.concatenate(wdl),
                 tol, f"EP dlogits (N={N}, passes={n})")
    for i, name in enumerate(("dwg", "dwu", "dwd")):
        got = np.concatenate([f64(t[i]) for t in dWs])
        assert np.isfinite(got).all()
        assert_close(got, wdW[i], tol, f"EP {name} (N={N}, passes={n})")
    # the single-device layer's backward on all tokens at once
    T = sum(Ts)
    dev = "cuda"
    xa, dya = torch.cat(xs), torch.cat(dys)
    La = torch.cat(Lt)
    dx1 = torch.empty_like(xa)
    dl1 = torch.empty((T, wl.E), dtype=torch.float32, device=dev)
    dw1 = [torch.empty(tuple(w.shape), dtype=torch.float32, device=dev)
           for w in W]
    ws = moe.layer_workspace(cfg, moe.MOE_WS_LAYER_BACKWARD)
    moe.moe_layer_backward(cfg, xa, La, *W, dya, dx1, dl1, *dw1,
                           moe.MOE_MODE_FALLBACK_LAYER, ws)
    torch.cuda.synchronize()
    assert_close(np.concatenate([f64(d) for d in dxs]), f64(dx1), tol,
                 f"EP dx vs moe_layer_backward (N={N})")
    assert_close(np.concatenate([f64(d) for d in dls]), f64(dl1), tol,
                 f"EP dlogits vs moe_layer_backward (N={N})")
    for i, name in enumerate(("dwg", "dwu", "dwd")):
        assert_close(np.concatenate([f64(t[i]) for t in dWs]), f64(dw1[i]),
                     tol, f"EP {name} vs moe_layer_backward (N={N})")


@pytest.mark.parametrize("case", CASES[:5], ids=lambda c: c[0].name)
def test_ring_backward_matches_oracle(case):
    """The ring's backward over logical ranks (cotangent all-gather, each
    rank's expert pass differentiated over all tokens, partial dx summed at
    the owners, pick gradients from the experts' ranks, the router backward
    on the owners) against the oracle's ring backward: dx and dlogits per
    rank, each rank's weight gradients.  Saving the sorted rows in the
    forward (moe_x_sorted=device) gives the same bits as gathering and
    sorting again in the backward."""
    wl, N, Ts, factor = case
    xs, Ls = rank_inputs(wl, Ts)
    cfg = gcfg(wl, Ts, N, factor)
    W, per_rank = weights_of(wl, N)
    g = torch.Generator(device="cuda").manual_seed(77)
    dys = [torch.randn((T_r, wl.H), generator=g, device="cuda").to(x.dtype)
           for T_r, x in zip(Ts, xs)]
    Lt = [torch.from_numpy(L).cuda() for L in Ls]
    remat = ep.RingLayer(cfg, ep.LoopbackTransport(N), per_rank)
    dxs, dls, dWs = remat.backward(xs, Lt, dys)
    saved = ep.RingLayer(cfg, ep.LoopbackTransport(N), per_rank,
                         save_x_sorted=True)
    saved.forward(xs, Lt)
    dxs2, dls2, dWs2 = saved.backward(xs, Lt, dys)
    torch.cuda.synchronize()
    for a, b in zip(dxs + dls + [w for t in dWs for w in t],
                    dxs2 + dls2 + [w for t in dWs2 for w in t]):
        assert torch.equal(a, b)
    mc = ref.MoEConfig(sum(Ts), wl.H, wl.E, wl.k, wl.F, N, factor, 0,
                       wl.renorm)
    wdx, wdl, wdW = ref.ring_layer_backward(
        mc, N, [f64(x) for x in xs], Ls,
        ref.dense_weights(*(f64(w) for w in W)), [f64(d) for d in dys])
    tol = TOL[wl.dtype]
    assert_close(np.concatenate([f64(d) for d in dxs]), np.concatenate(wdx),
                 tol, f"ring dx (N={N})")
    assert_close(np.concatenate([f64(d) for d in dls]), np.concatenate(wdl),
                 tol, f"ring dlogits (N={N})")
    for i, name in enumerate(("dwg", "dwu", "dwd")):
        got = np.concatenate([f64(t[i]) for t in dWs])
        assert np.isfinite(got).all()
        assert_close(got, wdW[i], tol, f"ring {name} (N={N})")


def test_ep_delocalize_is_localize_transposed():
    """moe_ep_delocalize writes slot q of a rank's values at the q-th pick
    it owns and leaves every other pick alone, so the ranks' calls together
    rebuild a [T, k] array from its localized pieces exactly."""
    T, E, k, N = 300, 12, 3, 4
    El = E // N
    gen = np.random.default_rng(5)
    idx = np.stack([gen.permutation(E)[:k] for _ in range(T)]).astype(
        np.int32)
    v = gen.standard_normal((T, k)).astype(np.float32)
    cfg = moe.make_config(T, 128, E, k, 128, N, 2.0, 0, "bf16")
    it = torch.from_numpy(idx).cuda()
    vt = torch.from_numpy(v).cuda()
    out = torch.full((T, k), 7.0, dtype=torch.float32, device="cuda")
    kk = min(k, El)
    for d in range(N):
        li = torch.empty((T, kk), dtype=torch.int32, device="cuda")
        lv = torch.empty((T, kk), dtype=torch.float32, device="cuda")
        moe.moe_ep_localize(cfg, it, vt, d * El, El, li, lv)
        before = out.clone()
        moe.moe_ep_delocalize(cfg, it, d * El, El, lv, out)
        torch.cuda.synchronize()
        mine = (idx // El) == d
        assert np.array_equal(np_(out)[mine], v[mine])
        assert np.array_equal(np_(out)[~mine], np_(before)[~mine])
    assert np.array_equal(np_(out), v)


def test_ep_check_global_flag():
    """moe_ep_check on summed shard counts: strict > C with C from the
    global token count; required factor max_s r_s * S / (T k)."""
    cfg = moe.make_config(1000, 128, 8, 2, 128, 4, 1.5, 0, "bf16")
    C = moe.moe_capacity_rows(cfg)           # floor(1.5 * 2000 / 4) = 750
    assert C == 750
    for loads, flag in (([750, 500, 500, 250], 0), ([751, 500, 500, 249], 1),
                        ([0, 0, 0, 0], 0)):
        s = torch.tensor(loads, dtype=torch.int32, device="cuda")
        f = torch.full((1,), 9, dtype=torch.int32, device="cuda")
        q = torch.zeros(1, dtype=torch.float32, device="cuda")
        c = torch.zeros(1, dtype=torch.int32, device="cuda")
        moe.moe_ep_check(cfg, s, f, q, c)
        torch.cuda.synchronize()
        assert int(f.item()) == flag and int(c.item()) == C
        assert abs(float(q.item()) - max(loads) * 4 / 2000) < 1e-6


def test_ep_sum_partials():
    for dt in (torch.bfloat16, torch.float32):
        g = torch.Generator(device="cuda").manual_seed(3)
        parts = torch.randn(3, 77, 256, generator=g, device="cuda").to(dt)
        cfg = moe.make_config(77, 256, 4, 2, 128, 2, 2.0, 0,
                              "bf16" if dt == torch.bfloat16 else "f32")
        y = torch.empty((77, 256), dtype=dt, device="cuda")
        moe.moe_ep_sum_partials(cfg, 3, parts, y)
        torch.cuda.synchronize()
        want = f64(parts).sum(0)
        assert_close(f64(y), want, TOL["bf16" if dt == torch.bfloat16
                                        else "f32"], f"sum of parts {dt}")


def test_ep_dsv3_full_size_8_ranks():
    """The DeepSeek-V3-shaped layer's 8192-token batch split over 8 logical
    EP ranks of 1024 tokens (32 experts each): the global check overflows
    (4 chunks per rank), and the outputs match moe_layer on the whole batch
    within the tolerance, and the oracle on sampled tokens."""
    wl = WORKLOADS["dsv3"]
    N, T_r = 8, 1024
    x_all = make_x(wl, "cuda")
    L_all = host_logits(wl, x_all)
    xs = [x_all[r * T_r:(r + 1) * T_r] for r in range(N)]
    Ls = [np.ascontiguousarray(L_all[r * T_r:(r + 1) * T_r])
          for r in range(N)]
    W = make_weights(wl, "cuda")
    cfg = moe.make_config(wl.T, wl.H, wl.E, wl.k, wl.F, N, wl.factor, 0,
                          wl.dtype)
    layer = ep.EPLayer(cfg, ep.LoopbackTransport(N), ep.local_weights(*W, N))
    ys = layer.forward(xs, [torch.from_numpy(L).cuda() for L in Ls])
    y1 = torch.empty_like(x_all)
    info = moe.moe_layer(cfg, x_all, torch.from_numpy(L_all).cuda(), *W, y1,
                         moe.MOE_MODE_FALLBACK_LAYER, moe.layer_workspace(cfg))
    torch.cuda.synchronize()
    assert layer.info["overflow"] == info["overflow"] == 1
    assert layer.info["n_chunks"] == info["n_chunks"] == 4
    y_ep = torch.cat(ys)
    assert_close(f64(y_ep), f64(y1), 2e-2, "EP (8 ranks) vs moe_layer, dsv3")
    toks = np.sort(np.random.default_rng(4).choice(wl.T, 8, replace=False))
    oi, ow, _ = ref.route(L_all[toks], wl.k)
    ti = torch.from_numpy(toks).cuda()
    from tests.gpu_util import expert_accessor
    want = ref.token_outputs(f64(x_all[ti]), oi, ow, expert_accessor(*W))
    assert_close(f64(y_ep[ti]), want, 2e-2, "EP dsv3 sampled tokens")
    del W, x_all
    torch.cuda.empty_cache()


@pytest.mark.parametrize("variant", ["ep", "ring"])
def test_backward_dsv3_full_size_8_ranks(variant):
    """The DeepSeek-V3-shaped layer's backward over 8 logical ranks of 1024
    tokens: the EP layer (its global check overflows: 4 passes per rank) and
    the ring of experts (dropless).  dx, dlogits and the weight gradients
    match moe_layer_backward on the whole batch (fallback=layer, which
    equals the dropless gradients) within the tolerance."""
    wl = WORKLOADS["dsv3"]
    N, T_r = 8, 1024
    x_all = make_x(wl, "cuda")
    L_all = host_logits(wl, x_all)
    Lt_all = torch.from_numpy(L_all).cuda()
    xs = [x_all[r * T_r:(r + 1) * T_r] for r in range(N)]
    Lt = [Lt_all[r * T_r:(r + 1) * T_r] for r in range(N)]
    g = torch.Generator(device="cuda").manual_seed(79)
    dy_all = torch.randn(x_all.shape, generator=g, device="cuda").to(
        x_all.dtype)
    dys = [dy_all[r * T_r:(r + 1) * T_r] for r in range(N)]
    W = make_weights(wl, "cuda")
    cfg = moe.make_config(wl.T, wl.H, wl.E, wl.k, wl.F, N, wl.factor, 0,
                          wl.dtype)
    per_rank = ep.local_weights(*W, N)
    if variant == "ep":
        layer = ep.EPLayer(cfg, ep.LoopbackTransport(N), per_rank)
    else:
        layer = ep.RingLayer(cfg, ep.LoopbackTransport(N), per_rank,
                             save_x_sorted=True)
        layer.forward(xs, Lt)
    dxs, dls, dWs = layer.backward(xs, Lt, dys)
    torch.cuda.synchronize()
    if variant == "ep":
        assert layer.info["overflow"] == 1 and layer.info["n_chunks"] == 4
    del layer
    torch.cuda.empty_cache()
    dx1 = torch.empty_like(x_all)
    dl1 = torch.empty((wl.T, wl.E), dtype=torch.float32, device="cuda")
    dw1 = [torch.empty(tuple(w.shape), dtype=torch.float32, device="cuda")
           for w in W]
    info = moe.moe_layer_backward(cfg, x_all, Lt_all, *W, dy_all, dx1, dl1,
                                  *dw1, moe.MOE_MODE_FALLBACK_LAYER,
                                  moe.layer_workspace(
                                      cfg, moe.MOE_WS_LAYER_BACKWARD))
    torch.cuda.synchronize()
    assert info["overflow"] == 1
    what = f"{variant} (8 ranks) vs moe_layer_backward, dsv3"
    El = wl.E // N
    assert_close_device([(dxs[r], dx1[r * T_r:(r + 1) * T_r])
                         for r in range(N)], 2e-2, f"{what}: dx")
    assert_close_device([(dls[r], dl1[r * T_r:(r + 1) * T_r])
                         for r in range(N)], 2e-2, f"{what}: dlogits")
    for i, name in enumerate(("dwg", "dwu", "dwd")):
        assert_close_device([(dWs[r][i], dw1[i][r * El:(r + 1) * El])
                             for r in range(N)], 2e-2, f"{what}: {name}")
    del W, x_all, dw1, dWs
    torch.cuda.empty_cache()


def draw_ep(i):
    """A seeded random expert-parallel layer: ranks, experts per rank, k,
    dims, per-rank token counts (some ranks empty), factor, dtype."""
    rng = np.random.default_rng(7000 + i)
    N = int(rng.choice([2, 4, 8]))
    E = N * int(rng.choice([1, 2, 4]))
    k = int(rng.integers(1, min(E, 6) + 1))
    bf = i % 3 != 2
    H = int(rng.choice([128, 256, 384])) if bf else int(rng.choice([32, 64]))
    F = int(rng.choice([128, 256])) if bf else 64
    Ts = [int(rng.integers(0, 300)) if rng.random() > 0.15 else 0
          for _ in range(N)]
    if sum(Ts) == 0:
        Ts[0] = 17
    wl = WORKLOADS["small"].with_(
        name=f"ep_rand{i}", T=sum(Ts), H=H, E=E, k=k, F=F, S=N,
        dtype="bf16" if bf else "f32",
        routing=str(rng.choice(["uniform", "zipf"])), zipf_s=1.2, seed=i,
        renorm=bool(rng.integers(0, 2)), x_scale=1.0 if bf else 0.25)
    return wl, N, Ts, float(rng.choice([0.5, 1.0, 2.0]))


EP_RANDOM = [draw_ep(i) for i in range(12)]


@pytest.mark.parametrize("case", EP_RANDOM, ids=lambda c: (
    f"{c[0].name}-{c[0].dtype}-N{c[1]}-E{c[0].E}-k{c[0].k}-f{c[3]}"))
def test_random_ep_and_ring_layers(case):
    """Seeded random EP layers over logical ranks: the EP layer (fallback=
    layer, global check) and the ring of experts, forward and backward,
    against the oracle's ep_layer, ring_layer and their backward."""
    wl, N, Ts, factor = case
    xs, Ls = rank_inputs(wl, Ts)
    cfg = gcfg(wl, Ts, N, factor)
    W, per_rank = weights_of(wl, N)
    g = torch.Generator(device="cuda").manual_seed(80 + N)
    dys = [torch.randn((T_r, wl.H), generator=g, device="cuda").to(x.dtype)
           for T_r, x in zip(Ts, xs)]
    Lt = [torch.from_numpy(L).cuda() for L in Ls]
    tol = TOL[wl.dtype]
    mc = ref.MoEConfig(sum(Ts), wl.H, wl.E, wl.k, wl.F, N, factor, 0,
                       wl.renorm)
    xh = [f64(x) for x in xs]
    dense = ref.dense_weights(*(f64(w) for w in W))
    layer = ep.EPLayer(cfg, ep.LoopbackTransport(N), per_rank)
    ys = layer.forward(xs, Lt)
    want, over, n = ref.ep_layer(mc, N, xh, Ls, dense)
    torch.cuda.synchronize()
    assert layer.info["overflow"] == int(over) and layer.info["n_chunks"] == n
    assert_close(np.concatenate([f64(y) for y in ys]), np.concatenate(want),
                 tol, "EP y")
    ring = ep.RingLayer(cfg, ep.LoopbackTransport(N), per_rank)
    yr = ring.forward(xs, Lt)
    torch.cuda.synchronize()
    assert_close(np.concatenate([f64(y) for y in yr]),
                 np.concatenate(ref.ring_layer(mc, N, xh, Ls, dense)), tol,
                 "ring y")
    dyh = [f64(d) for d in dys]
    for name, lay, oracle in (("EP", layer, ref.ep_layer_backward),
                              ("ring", ring, ref.ring_layer_backward)):
        dxs, dls, dWs = lay.backward(xs, Lt, dys)
        torch.cuda.synchronize()
        wdx, wdl, wdW = oracle(mc, N, xh, Ls, dense, dyh)
        assert_close(np.concatenate([f64(d) for d in dxs]),
                     np.concatenate(wdx), tol, f"{name} dx")
        assert_close(np.concatenate([f64(d) for d in dls]),
                     np.concatenate(wdl), tol, f"{name} dlogits")
        for i, wname in enumerate(("dwg", "dwu", "dwd")):
            assert_close(np.concatenate([f64(t[i]) for t in dWs]), wdW[i],
                         tol, f"{name} {wname}")
