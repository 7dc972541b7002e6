"""GPU parity: router logits = x @ Wr (+ offset), through the C ABI.

The float64 oracle's router_logits on the same x, Wr and offset is the
reference.  Tolerance: float32 outputs, normwise 1e-4, and every element
within 2^-10 of its dot-product scale (|x| |Wr|)_i + |r_i| (float32
accumulation over H terms, whatever the cancellation in the sum).  Shapes
cover the tensor-core form (bf16, H % 64 == 0, E % 128 == 0: the
DeepSeek-V3 and Llama4-Maverick layers at full size, several column tiles,
ragged row tiles, one token; small batches with the reduction split over a
cluster, including CTAs with an empty k-slice) and the CUDA-core forms (the fp32 tiny layer,
E = 16 of the small layer, odd H and E, E = 1 and 64 with Wr staged in several
chunks; E = 96, above 64 and no multiple of 128, on the thread-per-expert kernel).
"""
import numpy as np
import pytest
import torch

import mixture_experts_token_gb300 as moe
from oracle import moe_ref as ref
from synth import (WORKLOADS, make_logit_offset, make_router_weight, make_x,
                   sweep_workload)
from tests.gpu_util import cfg_from, f64, host_logits
from tests.parity_log import assert_close

pytestmark = pytest.mark.gpu

CASES = [
    WORKLOADS["tiny"], WORKLOADS["small"], WORKLOADS["dsv3"],
    WORKLOADS["l4mav"],
    WORKLOADS["small"].with_(name="t1000_e384", T=1000, H=256, E=384, S=4,
                             routing="uniform"),
    WORKLOADS["small"].with_(name="one_token", T=1, H=64, E=128, S=2),
    WORKLOADS["small"].with_(name="h104_e24", T=333, H=104, E=24, S=4),
    WORKLOADS["tiny"].with_(name="f32_e40", T=77, H=48, E=40, S=4,
                            routing="zipf", zipf_s=1.0),
    # the warp kernel (E <= 64): Wr staged in three chunks of rows (256
    # rows a chunk at E = 64, the last one 8 rows), a last CTA with fewer
    # tokens than its warps take; one expert
    WORKLOADS["small"].with_(name="e64_h520", T=777, H=520, E=64, S=4),
    WORKLOADS["small"].with_(name="e1", T=50, H=64, E=1, k=1, S=1),
    WORKLOADS["small"].with_(name="e96", T=300, H=128, E=96, S=4),
    # batches whose tiles leave most SMs idle: the reduction split over a
    # cluster (8 CTAs at up to 1024 tokens of H = 7168, 2 at 4096 tokens)
    WORKLOADS["dsv3"].with_(name="split8_t1", T=1),
    WORKLOADS["dsv3"].with_(name="split8_t1024", T=1024),
    WORKLOADS["dsv3"].with_(name="split2_t4096", T=4096),
    # 10 k-blocks over 8 CTAs: three CTAs get no k-block and add zeros
    WORKLOADS["dsv3"].with_(name="split_empty_slices", T=200, H=640),
]


def gpu_logits(wl, x, wr, off, T=None):
    cfg = cfg_from(wl, T=x.shape[0])
    out = torch.full((x.shape[0], wl.E), float("nan"), dtype=torch.float32,
                     device="cuda")
    offd = None if off is None else torch.from_numpy(off).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    moe.moe_router_logits(cfg, x, wr, offd, out, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return out


@pytest.mark.parametrize("wl", CASES, ids=lambda w: w.name)
@pytest.mark.parametrize("with_offset", [True, False])
def test_router_logits_parity(wl, with_offset):
    x = make_x(wl, "cuda")
    wr = make_router_weight(wl, "cuda")
    off = make_logit_offset(wl) if with_offset else None
    got = f64(gpu_logits(wl, x, wr, off))
    xh, wh = f64(x), f64(wr)
    want = ref.router_logits(xh, wh, off)
    scale = np.abs(xh) @ np.abs(wh) + np.abs(want)
    assert_close(got, want, 1e-4, f"logits ({'offset' if with_offset else 'x Wr'})",
                 scale=scale, cw_bound=2.0 ** -10)


def test_split_router_is_deterministic():
    """The split form sums the cluster's partial tiles in rank order, so two
    launches give the same bits."""
    wl = WORKLOADS["dsv3"].with_(T=700)
    x = make_x(wl, "cuda")
    wr = make_router_weight(wl, "cuda")
    off = make_logit_offset(wl)
    a = gpu_logits(wl, x, wr, off)
    b = gpu_logits(wl, x, wr, off)
    assert torch.equal(a, b)


def test_router_logits_feed_the_same_routing():
    """On the DeepSeek-V3 layer, routing the GPU's logits and routing the
    oracle's float32 logits pick the same experts for all but a handful of
    near-tied tokens (the logits differ only by float32 rounding)."""
    wl = WORKLOADS["dsv3"]
    x = make_x(wl, "cuda")
    wr = make_router_weight(wl, "cuda")
    off = make_logit_offset(wl)
    g = gpu_logits(wl, x, wr, off).cpu().numpy()
    h = host_logits(wl, x)
    gi = np.argsort(-g, axis=1, kind="stable")[:, :wl.k]
    hi = np.argsort(-h, axis=1, kind="stable")[:, :wl.k]
    differ = np.any(np.sort(gi, 1) != np.sort(hi, 1), axis=1).sum()
    assert differ <= 8, differ


def test_router_sweep_64k_sampled():
    """The sweep's 65,536-token batch (the 512 m-tiles x 2 column tiles of
    one launch): sampled token rows against the oracle."""
    wl = sweep_workload(65536, "zipf")
    x = make_x(wl, "cuda")
    wr = make_router_weight(wl, "cuda")
    off = make_logit_offset(wl)
    got = gpu_logits(wl, x, wr, off)
    rows = np.sort(np.random.default_rng(5).choice(wl.T, 2048, replace=False))
    ri = torch.from_numpy(rows).cuda()
    xh, wh = f64(x[ri]), f64(wr)
    want = ref.router_logits(xh, wh, off[rows])
    scale = np.abs(xh) @ np.abs(wh) + np.abs(want)
    assert_close(f64(got[ri]), want, 1e-4, "logits (sampled rows)",
                 scale=scale, cw_bound=2.0 ** -10)
    assert torch.isfinite(got).all()


def test_router_rejects_bad_arguments():
    wl = WORKLOADS["small"]
    cfg = cfg_from(wl, T=16)
    x = make_x(wl, "cuda", T=16)
    wr = make_router_weight(wl, "cuda")
    out = torch.empty((16, wl.E), dtype=torch.float32, device="cuda")
    with pytest.raises(moe.MoeError) as err:
        moe.moe_router_logits(cfg, x, None, None, out)
    assert err.value.status == moe.MOE_ERR_INVALID_ARG
    with pytest.raises(moe.MoeError):
        moe.moe_router_logits(cfg, x.view(torch.uint8)[:, 2:], wr, None, out)
    # T = 0 does nothing
    moe.moe_router_logits(cfg_from(wl, T=0), x, wr, None, out)


def draw_small_e(i):
    """Seeded random router case for the CUDA-core kernels: E in 1..64
    (the warp kernel) or 65..200 not a multiple of 128 (thread-per-expert),
    H a whole number of 16-byte words, ragged T, bf16 or fp32."""
    rng = np.random.default_rng(6000 + i)
    dtype = "f32" if i % 3 == 2 else "bf16"
    E = int(rng.integers(1, 65)) if i % 4 else int(rng.integers(65, 200))
    if E % 128 == 0:
        E += 1
    step = 4 if dtype == "f32" else 8
    H = step * int(rng.integers(1, 400))
    T = int(rng.integers(1, 3000))
    base = WORKLOADS["tiny"] if dtype == "f32" else WORKLOADS["small"]
    return base.with_(name=f"rnd{i}", T=T, H=H, E=E, k=1, S=1,
                      routing="uniform", seed=100 + i)


@pytest.mark.parametrize("i", range(12))
def test_router_logits_random_small_e(i):
    wl = draw_small_e(i)
    x = make_x(wl, "cuda")
    wr = make_router_weight(wl, "cuda")
    off = make_logit_offset(wl) if i % 2 else None
    got = f64(gpu_logits(wl, x, wr, off))
    xh, wh = f64(x), f64(wr)
    want = ref.router_logits(xh, wh, off)
    scale = np.abs(xh) @ np.abs(wh) + np.abs(want)
    assert_close(got, want, 1e-4, f"logits {wl.name} T{wl.T} H{wl.H} E{wl.E}",
                 scale=scale, cw_bound=2.0 ** -10)
