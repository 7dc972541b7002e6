"""GPU parity: the whole layer through moe_layer / moe_layer_dropless_chunked.

Small layers are compared with the oracle on every output; the
DeepSeek-V3- and Llama4-Maverick-shaped layers (full size, the launch
configuration the benchmark times) on sampled tokens, whose outputs the
oracle computes one by one.
"""
import numpy as np
import pytest
import torch

import mixture_experts_token_gb300 as moe
from oracle import moe_ref as ref
from synth import WORKLOADS, make_weights, make_x
from tests.gpu_util import TOL, cfg_from, expert_accessor, f64, host_logits, np_
from tests.parity_log import assert_close

pytestmark = pytest.mark.gpu


def setup(wl):
    x = make_x(wl, "cuda")
    L = host_logits(wl, x)
    wg, wu, wd = make_weights(wl, "cuda")
    return x, L, torch.from_numpy(L).cuda(), (wg, wu, wd)


def run_layer(wl, mode, x, Ld, W, **over):
    cfg = cfg_from(wl, **over)
    y = torch.empty((wl.T, wl.H), dtype=x.dtype, device="cuda")
    ws = moe.layer_workspace(cfg)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    info = moe.moe_layer(cfg, x, Ld, *W, y, mode, ws, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return y, info


def oracle_cfg(wl, **over):
    d = dict(T=wl.T, H=wl.H, E=wl.E, k=wl.k, F=wl.F, S=wl.S,
             ragged_buffer_factor=wl.factor, n_chunks=wl.n_chunks,
             renorm=wl.renorm)
    d.update(over)
    return ref.MoEConfig(**d)


SMALL = [WORKLOADS["tiny"], WORKLOADS["small"],
         WORKLOADS["small"].with_(name="small_k4_renorm", T=1500, H=512,
                                  F=256, k=4, renorm=True)]


@pytest.mark.parametrize("wl", SMALL, ids=lambda w: w.name)
def test_layer_modes_full_compare(wl):
    x, L, Ld, W = setup(wl)
    weights = ref.dense_weights(*(f64(w) for w in W))
    xh = f64(x)
    tol = TOL[wl.dtype]
    mc = oracle_cfg(wl)
    drop = ref.layer_dropless(mc, xh, L, weights)
    # fallback=layer: equals dropless in both branches
    for factor in (wl.factor, 0.1, 50.0):
        y, info = run_layer(wl, moe.MOE_MODE_FALLBACK_LAYER, x, Ld, W,
                            factor=factor)
        want = ref.layer(oracle_cfg(wl, ragged_buffer_factor=factor), xh, L,
                         weights)
        assert info["overflow"] == int(want.overflow)
        C = ref.capacity(wl.T, wl.k, wl.S, factor)
        if want.overflow:
            assert info["n_chunks"] == len(ref.chunk_plan(wl.T, wl.k, wl.E,
                                                          wl.S, C))
        assert_close(f64(y), want.y, tol, 'y')
        assert_close(f64(y), drop.y, tol, 'y vs dropless')
    # capped-only at factor 0.1 drops rows and diverges from dropless
    y_cap, _ = run_layer(wl, moe.MOE_MODE_CAPPED, x, Ld, W, factor=0.1)
    want_cap = ref.layer_capped(oracle_cfg(wl, ragged_buffer_factor=0.1), xh,
                                L, weights)
    assert want_cap.perm.n_dropped > 0
    assert_close(f64(y_cap), want_cap.y, tol, 'y_cap')
    assert ref.normwise_error(f64(y_cap), drop.y) > 10 * tol
    # one uncapped pass
    y_drop, _ = run_layer(wl, moe.MOE_MODE_DROPLESS, x, Ld, W)
    assert_close(f64(y_drop), drop.y, tol, 'y_drop')


@pytest.mark.parametrize("wl", SMALL[:2], ids=lambda w: w.name)
def test_chunked_entry_is_bit_identical_to_dropless(wl):
    x, L, Ld, W = setup(wl)
    y_drop, _ = run_layer(wl, moe.MOE_MODE_DROPLESS, x, Ld, W)
    for n in (0, 3, 8):
        cfg = cfg_from(wl, factor=0.5, n_chunks=n)
        y = torch.empty_like(y_drop)
        ws = moe.layer_workspace(cfg, moe.MOE_WS_CHUNKED)
        moe.moe_layer_dropless_chunked(cfg, x, Ld, *W, y, ws)
        torch.cuda.synchronize()
        assert torch.equal(y, y_drop), n


def sampled_tokens(T, n, seed=1):
    return np.sort(np.random.default_rng(seed).choice(T, n, replace=False))


@pytest.mark.parametrize("name", ["dsv3", "l4mav"])
def test_full_size_layer_sampled(name):
    wl = WORKLOADS[name]
    x, L, Ld, W = setup(wl)
    mc = oracle_cfg(wl)
    # global routing facts from the oracle (cheap: no FFN)
    oi, ow, _ = ref.route(L, wl.k)
    shard = ref.shard_counts(ref.expert_counts(oi, wl.E), wl.S)
    C = ref.capacity(wl.T, wl.k, wl.S, wl.factor)
    over = ref.overflow_flag(shard, C)
    y, info = run_layer(wl, moe.MOE_MODE_FALLBACK_LAYER, x, Ld, W)
    assert info["overflow"] == int(over)
    if over:
        assert info["n_chunks"] == len(ref.chunk_plan(wl.T, wl.k, wl.E, wl.S,
                                                      C))
    toks = sampled_tokens(wl.T, 12)
    want = ref.token_outputs(f64(x[torch.from_numpy(toks).cuda()]), oi[toks],
                             ow[toks], expert_accessor(*W))
    got = f64(y[torch.from_numpy(toks).cuda()])
    assert_close(got, want, 2e-2, 'got')
    # capped-only pass: dropped slots are skipped
    y_cap, _ = run_layer(wl, moe.MOE_MODE_CAPPED, x, Ld, W)
    p = ref.permute_indices(oi, wl.E, wl.S, C)
    keep = p.row_of[toks] >= 0
    want_cap = ref.token_outputs(f64(x[torch.from_numpy(toks).cuda()]),
                                 oi[toks], ow[toks], expert_accessor(*W),
                                 keep=keep)
    got_cap = f64(y_cap[torch.from_numpy(toks).cuda()])
    assert_close(got_cap, want_cap, 2e-2, 'got_cap')
    if over:
        # tokens whose every slot was dropped are exactly zero
        gone = np.where(np.all(p.row_of < 0, axis=1))[0]
        if len(gone):
            assert torch.all(y_cap[torch.from_numpy(gone).cuda()] == 0)


def test_layer_edge_cases():
    base = WORKLOADS["small"].with_(T=300, H=128, F=128, E=8, k=2, S=2)
    # T = 0: nothing to do
    wl0 = base.with_(T=0)
    cfg = cfg_from(wl0)
    x = torch.empty((0, 128), dtype=torch.bfloat16, device="cuda")
    info = moe.moe_layer(cfg, x, torch.empty((0, 8), device="cuda"),
                         *make_weights(base, "cuda"),
                         torch.empty_like(x), moe.MOE_MODE_FALLBACK_LAYER,
                         moe.layer_workspace(cfg))
    assert info["n_chunks"] == 0
    # a single token; a single expert; every token on one expert
    for wl, L in (
        (base.with_(T=1), None),
        (base.with_(E=1, k=1, S=1), None),
        (base.with_(T=1000, k=1), "hot3"),
    ):
        x, Lg, Ld, W = setup(wl)
        if L == "hot3":
            Lg = Lg.copy()
            Lg[:, 3] += 100.0
            Ld = torch.from_numpy(Lg).cuda()
        y, info = run_layer(wl, moe.MOE_MODE_DROPLESS, x, Ld, W)
        want = ref.layer_dropless(oracle_cfg(wl), f64(x), Lg,
                                  ref.dense_weights(*(f64(w) for w in W)))
        assert_close(f64(y), want.y, 2e-2, 'y')


@pytest.mark.parametrize("n_chunks,slots", [(5, 0), (2, 0), (0, 2)])
def test_pipelined_stepwise_passes_equal_moe_layer(n_chunks, slots):
    """bench.py's stepwise step -- each pass's permute tables on a side
    stream during the previous pass's FFN, two table sets in turn -- gives
    the bits of moe_layer (5 chunks reuse each table set twice)."""
    import bench
    from synth import WORKLOADS
    wl = WORKLOADS["small"].with_(T=3000, n_chunks=n_chunks,
                                  redundant_slots=slots)
    layer = bench.Layer(wl, "cuda")
    passes = layer.step()
    torch.cuda.synchronize()
    y_api = torch.empty_like(layer.b["y"])
    info = layer.api_layer(layer.x, layer.logits, y_api)
    torch.cuda.synchronize()
    assert int(layer.b["status"].item()) == 0
    if n_chunks:
        assert info["overflow"] and len(passes) == n_chunks
    assert torch.equal(y_api, layer.b["y"])
