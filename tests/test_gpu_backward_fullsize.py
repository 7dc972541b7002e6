"""GPU parity of the backward at full size, in the configuration the
benchmark times (moe_layer_backward, moe_dropless_fallback=layer).

The oracle cannot differentiate a whole DeepSeek-V3-sized layer, so it
checks samples it can compute one by one:
* a token's dx and dlogits: with the chunked fallback (or a capped pass
  that drops nothing) every pass is dropless, and a token's gradients
  depend only on its own row, routing and experts, so the oracle runs the
  backward of that token as a layer of its own.  dlogits come from
  dtopk_w[t,j] = <dy[t], y_sorted[r]>, a length-H dot product with
  cancellation: y_sorted is bf16, and H independent rounding errors of
  relative size eps add up to about eps * A_j with
  A_j = sqrt(sum_i (dy_ti y_ri)^2), however small the sum itself.  So each
  dlogit is held to tol * sum_j A_j |d w_j / d logit_e| (the error pushed
  through the softmax Jacobian) rather than to a relative error;
* an expert's weight gradients: the sum over the rows routed to it, from
  the oracle's per-expert FFN backward over exactly those rows (gathered
  in token order, scaled by the oracle's combine weights).
"""
import numpy as np
import pytest
import torch

import mixture_experts_token_gb300 as moe
from oracle import moe_ref as ref
from synth import WORKLOADS, make_weights, make_x
from synth.workloads import make_dy
from tests.gpu_util import TOL, cfg_from, expert_accessor, f64, host_logits
from tests.parity_log import assert_close

pytestmark = pytest.mark.gpu


def dlogit_bound(logits_t, idx_t, A, renorm, tol):
    """Per-expert bound on the dlogits error of one token from errors
    |delta dtopk_w_j| <= tol * A_j: sum_j tol A_j |dw_j/dlogit_e|, with
    dw_j/dl_e = w_j (delta - p_e) over all E (renorm: over the k chosen)."""
    E = len(logits_t)
    k = len(idx_t)
    bound = np.zeros(E)
    if renorm:
        wk = np.array(ref.softmax_f64([logits_t[e] for e in idx_t]))
        for i in range(k):
            for j in range(k):
                bound[idx_t[i]] += tol * A[j] * wk[j] * ((i == j) + wk[i])
        return bound
    p = np.array(ref.softmax_f64(list(logits_t)))
    for j in range(k):
        ej = int(idx_t[j])
        bound += tol * A[j] * p[ej] * p
        bound[ej] += tol * A[j] * p[ej]
    return bound


@pytest.mark.parametrize("name", ["dsv3", "l4mav"])
def test_fullsize_backward_sampled(name):
    wl = WORKLOADS[name]
    x = make_x(wl, "cuda")
    L = host_logits(wl, x)
    W = make_weights(wl, "cuda")
    dy = make_dy(wl, "cuda")
    cfg = cfg_from(wl)
    T, H, E, k, F = wl.T, wl.H, wl.E, wl.k, wl.F
    dev = "cuda"
    dx = torch.empty((T, H), dtype=x.dtype, device=dev)
    dl = torch.empty((T, E), dtype=torch.float32, device=dev)
    dw = [torch.empty((E, H, F), dtype=torch.float32, device=dev),
          torch.empty((E, H, F), dtype=torch.float32, device=dev),
          torch.empty((E, F, H), dtype=torch.float32, device=dev)]
    ws = moe.layer_workspace(cfg, moe.MOE_WS_LAYER_BACKWARD)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    info = moe.moe_layer_backward(cfg, x, torch.from_numpy(L).to(dev), *W,
                                  dy, dx, dl, *dw,
                                  moe.MOE_MODE_FALLBACK_LAYER, ws, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0

    # the oracle's routing of the whole batch (the flag and the rows of the
    # sampled experts)
    idx, w, _ = ref.route(L, k, wl.renorm)
    counts = ref.expert_counts(idx, E)
    C = ref.capacity(T, k, wl.S, wl.factor)
    over = ref.overflow_flag(ref.shard_counts(counts, wl.S), C)
    assert info["overflow"] == int(over)
    if not over:   # the capped pass then drops nothing: dropless per token
        assert ref.permute_indices(idx, E, wl.S, C).n_dropped == 0

    tol = TOL[wl.dtype]
    get = expert_accessor(*W)
    rng = np.random.default_rng(7)
    tokens = sorted(rng.choice(T, size=6, replace=False).tolist())
    one = ref.MoEConfig(1, H, E, k, F, wl.S, -1.0, 0, wl.renorm)
    for t in tokens:
        xt = f64(x[t:t + 1])
        g, _ = ref.pass_backward_touched(one, xt, L[t:t + 1], get,
                                         f64(dy[t:t + 1]), None)
        got_dx = f64(dx[t:t + 1])
        assert_close(got_dx, g.dx, tol, f"dx of token {t}")
        dyt = f64(dy[t])
        A = np.array([np.linalg.norm(dyt * ref.expert_ffn(xt, *get(int(e)))[1][0])
                      for e in idx[t]])
        bound = dlogit_bound(L[t], idx[t], A, wl.renorm, tol)
        got_dl = f64(dl[t])
        slack = 1e-6 * np.abs(g.dlogits[0]).max()
        bad = np.abs(got_dl - g.dlogits[0]) > bound + slack
        assert not bad.any(), f"dlogits of token {t}: experts {np.where(bad)}"

    # weight gradients of experts with a modest number of rows
    order = np.argsort(counts)
    picks = [int(e) for e in order if 1 <= counts[e] <= 160][:2]
    picks.append(int(order[0]))          # the least used expert (maybe 0)
    dyh_all = None
    for e in picks:
        rows = [(t, j) for t in range(T) for j in range(k) if idx[t, j] == e]
        if dyh_all is None:
            dyh_all = f64(dy)
        if rows:
            ts = [t for t, _ in rows]
            x_rows = f64(x[ts])
            dy_rows = np.stack([w[t, j] * dyh_all[t] for t, j in rows])
            _, want = ref.expert_ffn_backward(x_rows, dy_rows, *get(e))
        else:
            want = (np.zeros((H, F)), np.zeros((H, F)), np.zeros((F, H)))
        for i, name_ in enumerate(("dWg", "dWu", "dWd")):
            got = f64(dw[i][e])
            if not rows:
                assert not got.any(), f"{name_}[{e}] not zero"
                continue
            assert_close(got, want[i], tol, f"{name_}[{e}] ({len(rows)} rows)")
