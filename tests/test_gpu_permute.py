"""GPU parity: expert-sorted permute, capped drop and per-shard dedup.

row_of, sorted_token, group offsets, the dedup sets and expand indices and
the dropped-row count must equal the oracle bit for bit, and every kept
x_sorted row must be a byte copy of its token's row.
"""
import numpy as np
import pytest
import torch

from oracle import moe_ref as ref
from synth import WORKLOADS, make_x, sweep_workload
from tests.gpu_util import (cfg_from, compare_permutation, gpu_permute,
                            gpu_route, host_logits, np_)

pytestmark = pytest.mark.gpu

CASES = [
    WORKLOADS["tiny"], WORKLOADS["small"], WORKLOADS["dsv3"],
    WORKLOADS["l4mav"], sweep_workload(1024, "adversarial"),
    sweep_workload(16384, "zipf"), sweep_workload(4096, "uniform"),
    # ragged token counts and odd shapes
    WORKLOADS["small"].with_(name="ragged1000", T=1000, H=256, E=16, k=4,
                             S=4),
    WORKLOADS["small"].with_(name="one_token", T=1, H=128, E=8, k=3, S=2),
    WORKLOADS["small"].with_(name="e40_s8", T=777, H=64, E=40, k=6, S=8,
                             routing="uniform"),
    WORKLOADS["small"].with_(name="k_eq_e", T=300, H=64, E=8, k=8, S=4),
    # large tables: many token blocks, E above 256
    WORKLOADS["small"].with_(name="rows_32768", T=4096, H=64, E=256, k=8,
                             S=8, zipf_s=1.2),
    WORKLOADS["small"].with_(name="rows_32776", T=4097, H=64, E=256, k=8,
                             S=8, zipf_s=1.2),
    WORKLOADS["small"].with_(name="e300", T=900, H=64, E=300, k=3, S=4,
                             routing="uniform"),
    WORKLOADS["small"].with_(name="e640", T=1500, H=64, E=640, k=4, S=8,
                             zipf_s=1.2),
    # the most shards: 64 lanes of per-shard dedup; a block-shard table
    # above 1024 counts (the dedup scan kernel runs)
    WORKLOADS["small"].with_(name="s64", T=3000, H=64, E=512, k=8, S=64,
                             routing="uniform"),
    # 157 token blocks x 8 shards: the dedup scan kernel with 8 shards
    WORKLOADS["small"].with_(name="t20000", T=20000, H=64, E=256, k=8, S=8,
                             zipf_s=1.2),
    # few tokens with wide rows: each row's copy split over several CTAs
    # (7 slices of 128 chunks at H = 7168; 5 at H = 5120; 2 at H = 2048)
    WORKLOADS["dsv3"].with_(name="split_t100_h7168", T=100),
    WORKLOADS["l4mav"].with_(name="split_t50_h5120", T=50),
    WORKLOADS["small"].with_(name="split_t333_h2048", T=333, H=2048),
]


def inputs(wl):
    x = make_x(wl, "cuda")
    L = host_logits(wl, x)
    return x, L


@pytest.mark.parametrize("wl", CASES, ids=lambda w: w.name)
@pytest.mark.parametrize("factor", [None, 0.5, -1.0])
def test_permute_parity(wl, factor):
    factor = wl.factor if factor is None else factor
    cfg = cfg_from(wl, factor=factor)
    x, L = inputs(wl)
    idx, _ = gpu_route(cfg, L)
    oi, _, _ = ref.route(L, wl.k)
    assert np.array_equal(np_(idx), oi)
    C = ref.capacity(wl.T, wl.k, wl.S, factor)
    for capped in (True, False):
        bufs = gpu_permute(cfg, x, idx, capped)
        p = ref.permute_indices(oi, wl.E, wl.S, C if capped else None)
        compare_permutation(bufs, p, x.cpu())


def test_permute_t0():
    wl = WORKLOADS["small"].with_(T=0, H=128, E=8, k=2, S=2)
    cfg = cfg_from(wl)
    x = torch.empty((0, wl.H), dtype=torch.bfloat16, device="cuda")
    idx = torch.empty((0, wl.k), dtype=torch.int32, device="cuda")
    bufs = gpu_permute(cfg, x, idx, True)
    assert np.all(np_(bufs["group_offsets"]) == 0)
    assert np.all(np_(bufs["uniq_offsets"]) == 0)
    assert int(np_(bufs["n_dropped"])[0]) == 0
    # the two halves with no tokens: the same zeros, nothing else written
    import mixture_experts_token_gb300 as moe
    b = moe.alloc_step_buffers(cfg)
    for k in ("group_offsets", "uniq_offsets", "n_dropped"):
        b[k].fill_(7)
    moe.moe_permute_tables(cfg, idx, True, b["row_of"], b["sorted_token"],
                           b["group_offsets"], b["uniq_offsets"],
                           b["n_dropped"], b["permute_ws"])
    moe.moe_permute_scatter(cfg, x, b["row_of"], b["uniq_offsets"],
                            b["x_sorted"], b["uniq_tokens"], b["expand_idx"],
                            b["permute_ws"])
    torch.cuda.synchronize()
    for k in ("group_offsets", "uniq_offsets", "n_dropped"):
        assert np.all(np_(b[k]) == 0), k


def test_dedup_counts_adversarial():
    """All picks in shard 0: every token is sent once, to shard 0 only."""
    wl = sweep_workload(4096, "adversarial")
    cfg = cfg_from(wl, factor=-1.0)
    x, L = inputs(wl)
    idx, _ = gpu_route(cfg, L)
    bufs = gpu_permute(cfg, x, idx, False)
    uo = np_(bufs["uniq_offsets"])
    assert uo[1] == wl.T and uo[-1] == wl.T
    assert np.array_equal(np_(bufs["uniq_tokens"])[:wl.T], np.arange(wl.T))


SPLIT_CASES = [WORKLOADS["small"], WORKLOADS["dsv3"],
               [c for c in CASES if c.name == "s64"][0],
               [c for c in CASES if c.name == "t20000"][0]]


@pytest.mark.parametrize("wl", SPLIT_CASES, ids=lambda w: w.name)
def test_permute_split_equals_whole(wl):
    """moe_permute_tables then moe_permute_scatter (on another stream, after
    an event) write exactly the bits of moe_permute."""
    import mixture_experts_token_gb300 as moe
    cfg = cfg_from(wl)
    x, L = inputs(wl)
    idx, _ = gpu_route(cfg, L)
    side = torch.cuda.Stream()
    for capped in (True, False):
        whole = gpu_permute(cfg, x, idx, capped)
        b = moe.alloc_step_buffers(cfg)
        b["x_sorted"].zero_()
        for k in ("sorted_token", "uniq_tokens", "expand_idx"):
            b[k].fill_(-1)
        moe.moe_permute_tables(cfg, idx, capped, b["row_of"],
                               b["sorted_token"], b["group_offsets"],
                               b["uniq_offsets"], b["n_dropped"],
                               b["permute_ws"])
        ev = torch.cuda.Event()
        ev.record()
        side.wait_event(ev)
        moe.moe_permute_scatter(cfg, x, b["row_of"], b["uniq_offsets"],
                                b["x_sorted"], b["uniq_tokens"],
                                b["expand_idx"], b["permute_ws"], stream=side)
        torch.cuda.synchronize()
        R = int(np_(whole["group_offsets"])[-1])
        U = int(np_(whole["uniq_offsets"])[-1])
        for k in ("row_of", "group_offsets", "uniq_offsets", "n_dropped"):
            assert torch.equal(b[k], whole[k]), k
        for k, n in (("sorted_token", R), ("expand_idx", R),
                     ("uniq_tokens", U)):
            assert torch.equal(b[k][:n], whole[k][:n]), k
        assert torch.equal(b["x_sorted"][:R], whole["x_sorted"][:R])


def compare_x_sorted_on_device(x, x_sorted, sorted_token, rows_per_step=32768):
    """Every kept row of x_sorted equals x[sorted_token[r]] (the oracle's
    sorted_token), compared on the device in slices so no 7.5 GB host copy
    is needed."""
    st = torch.from_numpy(sorted_token.astype(np.int64)).cuda()
    for a in range(0, len(sorted_token), rows_per_step):
        z = min(len(sorted_token), a + rows_per_step)
        assert torch.equal(x_sorted[a:z], x.index_select(0, st[a:z])), \
            f"x_sorted rows {a}..{z}"


@pytest.mark.parametrize("routing", ["zipf", "adversarial", "uniform"])
def test_permute_parity_sweep_64k(routing):
    """The sweep's largest size: 65,536 tokens at H=7168 (524,288 routed
    rows, x_sorted 7.5 GB), bit-exact on every index output, every kept
    x_sorted row checked: the whole batch capped (factor 2) and uncapped,
    and one of the 8 fallback chunks as the fallback runs it."""
    import mixture_experts_token_gb300 as moe
    wl = sweep_workload(65536, routing)
    cfg = cfg_from(wl)
    x, L = inputs(wl)
    idx, _ = gpu_route(cfg, L)
    oi, _, _ = ref.route(L, wl.k)
    assert np.array_equal(np_(idx), oi)
    C = ref.capacity(wl.T, wl.k, wl.S, wl.factor)
    for capped in (True, False):
        bufs = gpu_permute(cfg, x, idx, capped)
        p = ref.permute_indices(oi, wl.E, wl.S, C if capped else None)
        compare_permutation(bufs, p)
        compare_x_sorted_on_device(x, bufs["x_sorted"], p.sorted_token)
        del bufs
    # chunk 3 of the 8-chunk fallback (uncapped, its own tokens)
    ct = moe.moe_chunk_tokens(cfg)
    assert ct == 8192 and moe.moe_num_chunks(cfg) == 8
    t0 = 3 * ct
    sc = cfg_from(wl, T=ct, factor=-1.0, n_chunks=0)
    bufs = gpu_permute(sc, x[t0:t0 + ct], idx[t0:t0 + ct].contiguous(), False)
    p = ref.permute_indices(oi[t0:t0 + ct], wl.E, wl.S, None)
    compare_permutation(bufs, p)
    compare_x_sorted_on_device(x[t0:t0 + ct], bufs["x_sorted"],
                               p.sorted_token)
    del bufs, x
    torch.cuda.empty_cache()


def draw_split(i):
    """Seeded random pass with few tokens and wide rows (the scatter splits
    each row over several CTAs): T 1..600, H a multiple of 64 up to 8192,
    E, k and S drawn, bf16 or fp32, Zipf or uniform routing."""
    rng = np.random.default_rng(5000 + i)
    S = int(rng.choice([1, 2, 4, 8]))
    E = S * int(rng.integers(1, 33))
    k = int(rng.integers(1, min(E, 8) + 1))
    dtype = "f32" if i % 4 == 3 else "bf16"
    H = 64 * int(rng.integers(8, 129))
    if dtype == "f32":
        H = min(H, 4096)
    T = int(rng.integers(1, 601))
    routing = str(rng.choice(["uniform", "zipf"]))
    return WORKLOADS["small"].with_(
        name=f"split_rnd{i}", T=T, H=H, E=E, k=k, S=S, dtype=dtype,
        routing=routing, zipf_s=1.2 if routing == "zipf" else 0.0,
        seed=200 + i)


@pytest.mark.parametrize("i", range(8))
def test_permute_split_random(i):
    """Bit-exact against the oracle, capped (factor 0.5) and dropless."""
    wl = draw_split(i)
    cfg = cfg_from(wl, factor=0.5)
    x, L = inputs(wl)
    idx, _ = gpu_route(cfg, L)
    oi, _, _ = ref.route(L, wl.k)
    assert np.array_equal(np_(idx), oi)
    C = ref.capacity(wl.T, wl.k, wl.S, 0.5)
    for capped in (True, False):
        bufs = gpu_permute(cfg, x, idx, capped)
        p = ref.permute_indices(oi, wl.E, wl.S, C if capped else None)
        compare_permutation(bufs, p, x.cpu())
