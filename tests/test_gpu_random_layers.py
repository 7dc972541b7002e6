"""GPU parity over seeded random layer configurations: moe_layer
(fallback=layer, with and without duplicate-expert slots) and
moe_layer_backward against the float64 oracle.

Each case draws T, H, E, k, F, S, the ragged buffer factor, the dtype, the
routing law, renormalisation and the slots from its own seed, so that
shapes no hand-written case names (odd token counts, one expert per shard,
k = E, factors on both sides of the overflow, tiles with a ragged tail) meet
the same checks: the overflow flag and the pass count equal the oracle's,
and the outputs and gradients are within the layer dtype's tolerance of the
oracle's (which, with fallback=layer, drops nothing and equals the dropless
layer).
"""
import numpy as np
import pytest
import torch

import mixture_experts_token_gb300 as moe
from oracle import moe_ref as ref
from synth import WORKLOADS, make_weights, make_x
from synth.workloads import make_dy
from tests.gpu_util import TOL, cfg_from, f64, host_logits
from tests.parity_log import assert_close

pytestmark = pytest.mark.gpu

N_CASES = 24


def draw(i):
    rng = np.random.default_rng(9000 + i)
    dtype = "f32" if i % 4 == 3 else "bf16"
    S = int(rng.choice([1, 2, 4, 8]))
    E = S * int(rng.choice([1, 2, 3, 4, 8]))
    k = int(rng.integers(1, min(E, 8) + 1))
    H = int(rng.choice([128, 256, 384, 512])) if dtype == "bf16" else \
        int(rng.choice([32, 64, 96]))
    F = int(rng.choice([128, 256, 384])) if dtype == "bf16" else \
        int(rng.choice([32, 64]))
    T = int(rng.integers(1, 700))
    factor = float(rng.choice([0.3, 0.7, 1.0, 2.0]))
    routing = str(rng.choice(["uniform", "zipf"]))
    slots = int(rng.choice([0, 0, 1, 2])) if S > 1 else 0
    return WORKLOADS["small"].with_(
        name=f"rand{i}", T=T, H=H, E=E, k=k, F=F, S=S, factor=factor,
        dtype=dtype, routing=routing, zipf_s=1.2 if routing == "zipf" else 0,
        renorm=bool(rng.integers(0, 2)), seed=i, redundant_slots=slots,
        x_scale=1.0 if dtype == "bf16" else 0.25)


CASES = [draw(i) for i in range(N_CASES)]


def ids(wl):
    return (f"{wl.name}-{wl.dtype}-T{wl.T}-H{wl.H}-E{wl.E}-k{wl.k}-F{wl.F}"
            f"-S{wl.S}-f{wl.factor}-B{wl.redundant_slots}")


def oracle_cfg(wl):
    return ref.MoEConfig(wl.T, wl.H, wl.E, wl.k, wl.F, wl.S, wl.factor, 0,
                         wl.renorm)


@pytest.mark.parametrize("wl", CASES, ids=ids)
def test_random_layer_forward(wl):
    x = make_x(wl, "cuda")
    L = host_logits(wl, x)
    W = make_weights(wl, "cuda")
    cfg = cfg_from(wl)
    y = torch.empty((wl.T, wl.H), dtype=x.dtype, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    info = moe.moe_layer(cfg, x, torch.from_numpy(L).cuda(), *W, y,
                         moe.MOE_MODE_FALLBACK_LAYER, moe.layer_workspace(cfg),
                         status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    weights = ref.dense_weights(*(f64(w) for w in W))
    mc = oracle_cfg(wl)
    if wl.redundant_slots:
        want = ref.layer_redundant(mc, f64(x), L, weights, wl.redundant_slots)
    else:
        want = ref.layer(mc, f64(x), L, weights)
    assert info["overflow"] == int(want.overflow)
    if want.overflow:
        C = ref.capacity(wl.T, wl.k, wl.S, wl.factor)
        assert info["n_chunks"] == len(ref.chunk_plan(wl.T, wl.k, wl.E, wl.S,
                                                      C))
    assert_close(f64(y), want.y, TOL[wl.dtype], "y")
    drop = ref.layer_dropless(mc, f64(x), L, weights)
    assert_close(f64(y), drop.y, TOL[wl.dtype], "y vs dropless")


@pytest.mark.parametrize("wl", CASES[::2], ids=ids)
def test_random_layer_backward(wl):
    x = make_x(wl, "cuda")
    L = host_logits(wl, x)
    W = make_weights(wl, "cuda")
    dy = make_dy(wl, "cuda")
    cfg = cfg_from(wl)
    dev = "cuda"
    dx = torch.empty_like(x)
    dl = torch.empty((wl.T, wl.E), dtype=torch.float32, device=dev)
    dw = [torch.full(tuple(w.shape), float("nan"), dtype=torch.float32,
                     device=dev) for w in W]
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    moe.moe_layer_backward(cfg, x, torch.from_numpy(L).cuda(), *W, dy, dx,
                           dl, *dw, moe.MOE_MODE_FALLBACK_LAYER,
                           moe.layer_workspace(cfg, moe.MOE_WS_LAYER_BACKWARD),
                           status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    g = ref.layer_backward_dropless(oracle_cfg(wl), f64(x), L,
                                    *[f64(w) for w in W], f64(dy))
    tol = TOL[wl.dtype]
    for name, got, want in (("dx", dx, g.dx), ("dlogits", dl, g.dlogits),
                            ("dwg", dw[0], g.dwg), ("dwu", dw[1], g.dwu),
                            ("dwd", dw[2], g.dwd)):
        got = f64(got)
        assert np.isfinite(got).all(), name
        assert_close(got, want, tol, name)
