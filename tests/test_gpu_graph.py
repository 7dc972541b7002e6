"""GPU: the layer as one CUDA graph with a conditional node (moe_layer_graph_*)
gives the same bits as moe_layer in both branches, launch after launch with
inputs refreshed in place, and reports the same overflow flag."""
import pytest
import torch

import mixture_experts_token_gb300 as moe
from synth import WORKLOADS, make_weights, make_x
from tests.gpu_util import cfg_from, host_logits

pytestmark = pytest.mark.gpu


def batch(wl, seed):
    w = wl.with_(seed=seed)
    x = make_x(w, "cuda")
    L = torch.from_numpy(host_logits(w, x))
    return x, L.cuda()


def device_flag(graph, ws):
    """The graph's overflow flag lives in the workspace: read it there."""
    off = graph.overflow_flag_ptr() - ws.data_ptr()
    assert 0 <= off < ws.numel() and off % 4 == 0
    return int(ws[off:off + 4].view(torch.int32).item())


@pytest.mark.parametrize("wl,factor", [
    (WORKLOADS["tiny"], 0.1),
    (WORKLOADS["tiny"], 2.0),
    (WORKLOADS["small"], 2.0),
    (WORKLOADS["small"], 50.0),
    (WORKLOADS["l4mav"], 2.0),
    (WORKLOADS["dsv3"], 2.0),
], ids=["tiny-ovf", "tiny", "small-ovf", "small", "l4mav", "dsv3"])
def test_graph_matches_moe_layer(wl, factor):
    cfg = cfg_from(wl, factor=factor)
    W = make_weights(wl, "cuda")
    x, L = batch(wl, 0)
    y = torch.zeros((wl.T, wl.H), dtype=x.dtype, device="cuda")
    ws = moe.layer_workspace(cfg)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    g = moe.MoeLayerGraph(cfg, x, L, *W, y, ws, status)
    ref_ws = moe.layer_workspace(cfg)
    for seed in (0, 1, 2):
        xs, Ls = batch(wl, seed)
        x.copy_(xs)
        L.copy_(Ls)
        g.launch()
        torch.cuda.synchronize()
        y_ref = torch.empty_like(y)
        info = moe.moe_layer(cfg, xs, Ls, *W, y_ref,
                             moe.MOE_MODE_FALLBACK_LAYER, ref_ws)
        torch.cuda.synchronize()
        assert torch.equal(y, y_ref), seed
        assert device_flag(g, ws) == info["overflow"]
        if info["overflow"]:
            assert g.fallback_chunks() == info["n_chunks"]
    assert int(status.item()) == 0
    g.close()


def test_graph_both_branches_on_one_graph():
    """One graph, two batches: one that overflows and one that does not."""
    wl = WORKLOADS["small"].with_(T=1024, H=256, F=256, E=8, S=4, k=2)
    cfg = cfg_from(wl, factor=2.0)
    W = make_weights(wl, "cuda")
    x, L = batch(wl, 0)
    y = torch.zeros((wl.T, wl.H), dtype=x.dtype, device="cuda")
    ws = moe.layer_workspace(cfg)
    g = moe.MoeLayerGraph(cfg, x, L, *W, y, ws)
    hot = L.clone()
    hot[:, :2] += 50.0            # every pick in shard 0 -> overflow
    flat = torch.randn_like(L) * 0.01   # near-uniform -> no overflow
    flags = []
    for logits in (hot, flat, hot):
        L.copy_(logits)
        g.launch()
        y_ref = torch.empty_like(y)
        info = moe.moe_layer(cfg, x, logits, *W, y_ref,
                             moe.MOE_MODE_FALLBACK_LAYER,
                             moe.layer_workspace(cfg))
        torch.cuda.synchronize()
        assert torch.equal(y, y_ref)
        flags.append(device_flag(g, ws))
        assert flags[-1] == info["overflow"]
    assert flags == [1, 0, 1]
    g.close()


@pytest.mark.parametrize("wl", [WORKLOADS["small"], WORKLOADS["tiny"]],
                         ids=["small", "tiny"])
def test_traced_graph_bits_and_stamps(wl):
    """The traced graph writes the bits of the untraced one, and its stamps
    of the branch it took increase along the stages: layer start, routing,
    check, then each pass's start, GEMM1, GEMM2, combine and end."""
    for factor in (0.3, 50.0):          # the fallback, then the capped pass
        cfg = cfg_from(wl, factor=factor)
        W = make_weights(wl, "cuda")
        x, L = batch(wl, 0)
        slots = moe.moe_layer_graph_trace_slots(cfg)
        n_chunks = moe.moe_num_chunks(cfg)
        assert slots == 3 + 5 * max(1, n_chunks)
        trace = torch.zeros(slots, dtype=torch.int64, device="cuda")
        y = torch.zeros((wl.T, wl.H), dtype=x.dtype, device="cuda")
        y0 = torch.zeros_like(y)
        ws, ws0 = moe.layer_workspace(cfg), moe.layer_workspace(cfg)
        g = moe.MoeLayerGraph(cfg, x, L, *W, y, ws, trace=trace)
        g0 = moe.MoeLayerGraph(cfg, x, L, *W, y0, ws0)
        g.launch()
        g0.launch()
        torch.cuda.synchronize()
        assert torch.equal(y, y0)
        flag = device_flag(g, ws)
        passes = g.fallback_chunks() if flag else 1
        st = trace.cpu().tolist()
        used = st[:3 + 5 * passes]
        assert all(a <= b for a, b in zip(used, used[1:])), used
        assert used[0] > 0 and used[-1] - used[0] > 0
        assert bool(flag) == (factor < 1.0)
        g.close()
        g0.close()


@pytest.mark.parametrize("T,routing,factor", [(4096, "uniform", 2.0),
                                              (4096, "zipf", 2.0),
                                              (1024, "adversarial", 2.0)])
def test_dispatch_only_layer(T, routing, factor):
    """F = 0, the routing/permute/dedup sweep's layer: moe_layer and the
    graph give y[t] = sum_j w[t,j] x[t] over the token's kept rows (the
    combine of the permuted rows), bit for bit between the two, and within
    the bf16 tolerance of that sum from the oracle's routing (no pass
    drops a row, so it is (sum_j w[t,j]) x[t])."""
    from oracle import moe_ref as ref
    from synth import sweep_workload
    from tests.gpu_util import f64
    from tests.parity_log import assert_close
    wl = sweep_workload(T, routing)
    cfg = cfg_from(wl, factor=factor)
    x, L = batch(wl, 0)
    y = torch.zeros((wl.T, wl.H), dtype=x.dtype, device="cuda")
    ws = moe.layer_workspace(cfg)
    info = moe.moe_layer(cfg, x, L, None, None, None, y,
                         moe.MOE_MODE_FALLBACK_LAYER, ws)
    y_g = torch.zeros_like(y)
    ws_g = moe.layer_workspace(cfg)
    g = moe.MoeLayerGraph(cfg, x, L, None, None, None, y_g, ws_g)
    g.launch()
    torch.cuda.synchronize()
    assert torch.equal(y, y_g)
    assert device_flag(g, ws_g) == info["overflow"]
    Ln = L.cpu().numpy()
    idx, w, _ = ref.route(Ln, wl.k)
    C = ref.capacity(wl.T, wl.k, wl.S, factor)
    over = ref.overflow_flag(ref.shard_counts(ref.expert_counts(idx, wl.E),
                                              wl.S), C)
    assert info["overflow"] == int(over)
    # dispatch-only: every pass keeps its rows (the capped pass runs only
    # when nothing overflows), so y[t] = (sum_j w[t,j]) x[t]
    want = w.sum(axis=1, keepdims=True) * f64(x)
    assert_close(f64(y), want, 2e-2, f"dispatch-only y ({routing})")
    g.close()
