"""GPU parity: router top-k + weights, counts and the overflow check.

Routing indices, counts, offsets, shard loads, the flag and the capacity
must equal the oracle bit for bit; the float32 combine weights must be
within the fp32 tolerance (1e-4, normwise) of the float64 oracle.
"""
import numpy as np
import pytest
import torch

import mixture_experts_token_gb300 as moe
from oracle import moe_ref as ref
from synth import WORKLOADS, make_x, sweep_workload
from tests.gpu_util import cfg_from, gpu_check, gpu_route, host_logits, np_
from tests.parity_log import assert_close

pytestmark = pytest.mark.gpu

ROUTE_CASES = [
    WORKLOADS["tiny"], WORKLOADS["small"], WORKLOADS["dsv3"],
    WORKLOADS["l4mav"], sweep_workload(1024, "adversarial"),
    sweep_workload(16384, "zipf"), sweep_workload(65536, "uniform"),
]


def logits_for(wl):
    return host_logits(wl, make_x(wl, "cuda"))


def oracle_sample(T, n=3000, seed=0):
    if T <= n:
        return np.arange(T)
    return np.sort(np.random.default_rng(seed).choice(T, n, replace=False))


@pytest.mark.parametrize("wl", ROUTE_CASES, ids=lambda w: w.name)
@pytest.mark.parametrize("renorm", [False, True])
def test_route_parity(wl, renorm):
    wl = wl.with_(renorm=renorm)
    cfg = cfg_from(wl)
    L = logits_for(wl)
    idx, w = gpu_route(cfg, L)
    idx, w = np_(idx), np_(w)
    rows = oracle_sample(wl.T)
    oi, ow, nf = ref.route(L[rows], wl.k, renorm)
    assert not nf
    assert np.array_equal(idx[rows], oi)
    assert_close(w[rows], ow, 1e-4, "topk_w (sampled tokens)")


def test_route_ties_and_odd_shapes():
    rng = np.random.default_rng(3)
    for (T, E, k) in ((3000, 64, 8), (777, 40, 5), (64, 1, 1), (512, 8, 8),
                      (300, 1024, 32), (2000, 256, 8), (50, 33, 32)):
        L = rng.integers(0, 4, size=(T, E)).astype(np.float32)  # many ties
        L[::7] = -L[::7]            # -0.0 and +0.0 must compare equal
        for renorm in (False, True):
            cfg = moe.make_config(T, 64, E, k, 128, 1, 2.0, 0, "bf16", renorm)
            idx, w = gpu_route(cfg, L)
            oi, ow, _ = ref.route(L, k, renorm)
            assert np.array_equal(np_(idx), oi), (T, E, k)
            assert_close(np_(w), ow, 1e-4, 'topk_w')


def test_route_nonfinite_logits():
    rng = np.random.default_rng(4)
    T, E, k = 500, 64, 4
    L = rng.standard_normal((T, E)).astype(np.float32)
    L[3, 5] = np.nan
    L[10, :] = np.nan                       # no finite logit at all
    L[11, 7] = np.inf
    L[12, 9] = -np.inf
    L[13, :60] = np.inf                     # fewer than k finite logits
    cfg = moe.make_config(T, 64, E, k, 128, 4, 2.0)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    idx, w = gpu_route(cfg, L, status)
    oi, ow, nf = ref.route(L, k)
    assert nf and int(status.item()) & moe.MOE_DEV_NONFINITE
    assert np.array_equal(np_(idx), oi)
    assert np.all(np_(w)[10] == 0)
    assert_close(np_(w), ow, 1e-4, 'topk_w')
    # clean logits leave the status word alone
    status.zero_()
    gpu_route(cfg, np.nan_to_num(L, nan=0.0, posinf=1.0, neginf=-1.0), status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0


def check_against_oracle(cfg, idx_gpu, oi, T, k, E, S, factor):
    got = gpu_check(cfg, idx_gpu)
    counts = ref.expert_counts(oi, E)
    shard = ref.shard_counts(counts, S)
    C = ref.capacity(T, k, S, factor)
    assert np.array_equal(got["counts"], counts)
    assert np.array_equal(got["offsets"], ref.exclusive_scan(counts))
    assert np.array_equal(got["shard"], shard)
    assert int(got["flag"][0]) == int(ref.overflow_flag(shard, C))
    assert int(got["cap"][0]) == (-1 if C is None else C)
    assert got["req"][0] == np.float32(ref.required_factor(shard, T, k))
    return got


CHECK_CASES = [WORKLOADS["tiny"], WORKLOADS["small"], WORKLOADS["dsv3"],
               WORKLOADS["l4mav"], sweep_workload(4096, "adversarial"),
               sweep_workload(65536, "zipf")]


@pytest.mark.parametrize("wl", CHECK_CASES, ids=lambda w: w.name)
def test_check_parity(wl):
    L = logits_for(wl)
    oi, _, _ = ref.route(L, wl.k)   # full routing: counts are global
    flags = {}
    for factor in (0.1, 0.5, 1.0, 2.0, 3.0, -1.0):
        cfg = cfg_from(wl, factor=factor)
        idx, _ = gpu_route(cfg, L)
        got = check_against_oracle(cfg, idx, oi, wl.T, wl.k, wl.E, wl.S,
                                   factor)
        flags[factor] = int(got["flag"][0])
    # the pages' forcing case: factor 0.1 always overflows
    assert flags[0.1] == 1 and flags[-1.0] == 0


def test_check_hand_built_loads():
    """Hand-built routings with known shard loads, including a single hot
    shard that is the last one (the asymmetric overflow case)."""
    E, S, k = 16, 4, 2
    for loads in ([8, 8, 8, 8], [2, 2, 2, 26], [26, 2, 2, 2], [0, 32, 0, 0]):
        rows = []
        for s, n in enumerate(loads):
            rows += [[s * 4, s * 4 + 1]] * (n // k)
        oi = np.array(rows, dtype=np.int64)
        T = len(rows)
        idx = torch.from_numpy(oi.astype(np.int32)).cuda()
        for factor in (1.0, 2.0, 3.25):
            cfg = moe.make_config(T, 64, E, k, 128, S, factor)
            got = check_against_oracle(cfg, idx, oi, T, k, E, S, factor)
            assert np.array_equal(got["shard"], loads)
