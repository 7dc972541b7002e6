"""Failure detection on the GPU without a fault: the bounded waits of the
GEMM, of the router's cluster kernel and of the two-SM weight gradient.

A test hook stops the GEMM's TMA producer after a few stage fills, so the
MMA warp waits on a barrier nothing will complete.  The wait gives up after
its limit (about 2 s); the kernel must report MOE_DEV_TIMEOUT in the status
word, return on its own (no trap, no hang), and leave the CUDA context
usable: the next, normal launch gives correct results.  Nothing here faults
or hangs the GPU.
"""
import time

import numpy as np
import pytest
import torch

import mixture_experts_token_gb300 as moe
from oracle import moe_ref as ref
from tests.gpu_util import f64
from tests.parity_log import assert_close

pytestmark = pytest.mark.gpu


def _case():
    E, H, F = 3, 256, 256
    sizes = [300, 0, 200]
    R = sum(sizes)
    g = torch.Generator(device="cuda").manual_seed(3)
    xs = torch.randn(R, H, generator=g, device="cuda").to(torch.bfloat16)
    W = [(torch.randn(E, *shp, generator=g, device="cuda") * 0.05)
         .to(torch.bfloat16) for shp in ((H, F), (H, F), (F, H))]
    off = torch.tensor(np.concatenate([[0], np.cumsum(sizes)]),
                       dtype=torch.int32, device="cuda")
    cfg = moe.make_config(R, H, E, 1, F, 1, 2.0, 0, "bf16")
    return cfg, xs, off, W, R


def _run(cfg, xs, off, W, R, status):
    h = torch.zeros(R, cfg.F, dtype=torch.bfloat16, device="cuda")
    ys = torch.zeros(R, cfg.H, dtype=torch.bfloat16, device="cuda")
    moe.moe_gmm_swiglu(cfg, xs, off, *W, h, ys, status)
    torch.cuda.synchronize()
    return h, ys


def test_gemm_wait_times_out_and_context_survives():
    cfg, xs, off, W, R = _case()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    try:
        moe.moe_test_stall_gemm_producer(3)
        t0 = time.time()
        _run(cfg, xs, off, W, R, status)
        took = time.time() - t0
    finally:
        moe.moe_test_stall_gemm_producer(-1)
    assert int(status.item()) & moe.MOE_DEV_TIMEOUT
    assert took < 30.0
    # the context is intact: a normal launch is correct
    status.zero_()
    h, ys = _run(cfg, xs, off, W, R, status)
    assert int(status.item()) == 0
    want_h, want_y = ref.grouped_ffn(
        f64(xs), off.cpu().numpy(),
        ref.dense_weights(*(f64(w) for w in W)))
    assert_close(f64(ys), want_y, 2e-2, 'ys')


def test_split_router_wait_times_out_and_context_survives():
    """The router's split form (a cluster of CTAs per tile, two cluster
    barriers): with the producers stopped, every CTA's MMA wait runs out,
    the status word reports MOE_DEV_TIMEOUT, every CTA still passes both
    cluster barriers and the launch returns; the next launch is correct."""
    from synth import WORKLOADS, make_logit_offset, make_router_weight, \
        make_x
    wl = WORKLOADS["dsv3"].with_(T=1024)
    cfg = moe.make_config(wl.T, wl.H, wl.E, wl.k, wl.F, wl.S, 2.0, 0, "bf16")
    x = make_x(wl, "cuda")
    wr = make_router_weight(wl, "cuda")
    off = make_logit_offset(wl)
    L = torch.empty((wl.T, wl.E), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    offd = torch.from_numpy(off).cuda()
    try:
        moe.moe_test_stall_gemm_producer(3)
        t0 = time.time()
        moe.moe_router_logits(cfg, x, wr, offd, L, status)
        torch.cuda.synchronize()
        took = time.time() - t0
    finally:
        moe.moe_test_stall_gemm_producer(-1)
    assert int(status.item()) & moe.MOE_DEV_TIMEOUT
    assert took < 30.0
    status.zero_()
    moe.moe_router_logits(cfg, x, wr, offd, L, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    want = ref.router_logits(f64(x), f64(wr), off)
    assert_close(f64(L), want, 1e-4, "logits after the timeout")


def test_pair_wgrad_wait_times_out_and_context_survives():
    """The two-SM weight gradient (a CTA pair per tile of dW): with both
    CTAs' producers stopped after 3 stage fills, the leader's MMA wait runs
    out, the status word reports MOE_DEV_TIMEOUT, both CTAs' epilogues and
    the peer's TMEM relay give up on their own bounded waits, both CTAs pass
    the final cluster barrier and the launch returns; the next launch is
    correct."""
    from tests.test_gpu_wgrad_pair import case_cfg, run
    H, F, G = 512, 256, 4
    off = np.array([0, 400, 416, 416, 688], dtype=np.int32)  # 7 and 5 blocks
    segs = [(off, 3)]
    rows = 3 + int(off[-1]) + 5
    gen = torch.Generator().manual_seed(11)
    t = {n: (torch.randn((rows, w), generator=gen) * 0.5).to(torch.bfloat16)
         for n, w in (("x", H), ("dg", F), ("du", F), ("h", F), ("dy", H))}
    cfg = case_cfg(H, F, G)
    try:
        moe.moe_test_stall_gemm_producer(3)
        t0 = time.time()
        _, st = run(cfg, segs, rows, t, moe.MOE_WGRAD_ROWS16, G, None)
        took = time.time() - t0
    finally:
        moe.moe_test_stall_gemm_producer(-1)
    assert st & moe.MOE_DEV_TIMEOUT
    assert took < 60.0
    dw, st = run(cfg, segs, rows, t, moe.MOE_WGRAD_ROWS16, G, None)
    assert st == 0
    ops = {n: f64(v) for n, v in t.items()}
    for got, p_, q_ in ((dw[0], "x", "dg"), (dw[1], "x", "du"),
                        (dw[2], "h", "dy")):
        want = ref.segmented_weight_grads(ops[p_], ops[q_], segs, G, G)
        assert_close(f64(got), want, 1e-3, f"d{q_} after the timeout")
