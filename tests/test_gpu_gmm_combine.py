"""GPU parity: the grouped SwiGLU GEMM and the weighted combine.

Inputs are synthetic (rows, ragged group sizes, weights); the oracle's
float64 grouped FFN and combine are the reference.  Tolerance: normwise
2e-2 for bf16, 1e-4 for fp32, per output tensor.
"""
import numpy as np
import pytest
import torch

import mixture_experts_token_gb300 as moe
from oracle import moe_ref as ref
from tests.gpu_util import TOL, expert_accessor, f64, np_
from tests.parity_log import assert_close

pytestmark = pytest.mark.gpu


def make_gmm_case(sizes, H, F, k_rows, dtype, seed=0, std=0.05):
    """x_sorted with len(sizes) ragged groups; rows beyond the groups (up to
    the allocation of T*k rows) are filled with NaN to prove they never leak
    into a valid row."""
    E = len(sizes)
    R = int(sum(sizes))
    alloc = max(k_rows, R)
    g = torch.Generator(device="cuda").manual_seed(seed)
    dt = torch.float32 if dtype == "f32" else torch.bfloat16
    xs = torch.full((alloc, H), float("nan"), device="cuda", dtype=dt)
    xs[:R] = torch.randn(R, H, generator=g, device="cuda").to(dt)
    wg = (torch.randn(E, H, F, generator=g, device="cuda") * std).to(dt)
    wu = (torch.randn(E, H, F, generator=g, device="cuda") * std).to(dt)
    wd = (torch.randn(E, F, H, generator=g, device="cuda") * std).to(dt)
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    return xs, torch.from_numpy(off).cuda(), wg, wu, wd, off, alloc


def run_gmm(sizes, H, F, dtype, T=None, k=1, seed=0):
    E = len(sizes)
    R = int(sum(sizes))
    T = T if T is not None else R
    xs, goff, wg, wu, wd, off, alloc = make_gmm_case(sizes, H, F, T * k,
                                                     dtype, seed)
    cfg = moe.make_config(T, H, E, k, F, 1, 2.0, 0, dtype)
    dt = xs.dtype
    h = torch.zeros((alloc, F), dtype=dt, device="cuda")
    ys = torch.zeros((alloc, H), dtype=dt, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    moe.moe_gmm_swiglu(cfg, xs, goff, wg, wu, wd, h, ys, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return xs, off, (wg, wu, wd), h, ys, R


GMM_CASES = [
    # (group sizes, H, F, kernel kinds): empty groups, single rows, tile
    # edges, many tiles.  Kernel kinds is moe_gmm_kernel_choice's answer for
    # bf16: bit 1 GEMM2 on the two-SM (CTA pair) kernel (H % 256 == 0 and
    # groups averaging >= 512 rows); 0: the one-CTA kernels.
    ([0, 1, 127, 128, 129, 300], 256, 256, 0),
    ([5, 0, 0, 700, 3], 384, 128, 0),       # H % 256 != 0: 128-wide GEMM2
    ([128] * 4, 128, 128, 0),
    ([1000], 512, 384, 2),                  # one group of 1000 rows
    ([37, 250, 1, 0, 90, 64, 513, 2], 1024, 512, 0),
    # 5201 rows in 5 groups (>= 512 each on average): the pair GEMM2, with a
    # small and a one-row group among the large ones
    ([2100, 1500, 1300, 300, 1], 512, 256, 2),
    ([4096, 3000], 256, 384, 2),
    ([600, 520, 0, 1000], 512, 128, 2),     # 530 rows per group
    # H % 256 != 0: GEMM2 on the 128-wide one-CTA kernel
    ([1200, 1100], 384, 256, 0),
]


def test_gmm_kernel_choice_query():
    """moe_gmm_kernel_choice follows the average rows per group, the row
    bound given, the layer dtype and H % 256 for GEMM2."""
    c = moe.make_config(2048, 512, 2, 1, 256, 1, 2.0, 0, "bf16")
    assert moe.moe_gmm_kernel_choice(c) == 2
    assert moe.moe_gmm_kernel_choice(c, rows_bound=1024) == 2
    assert moe.moe_gmm_kernel_choice(c, rows_bound=1023) == 0
    assert moe.moe_gmm_kernel_choice(c, n_groups=4) == 2
    assert moe.moe_gmm_kernel_choice(c, n_groups=5) == 0
    assert moe.moe_gmm_kernel_choice(c.with_(H=384)) == 0
    assert moe.moe_gmm_kernel_choice(c.with_(dtype=moe.MOE_F32)) == 0
    assert moe.moe_gmm_kernel_choice(c, n_groups=-1) == -1
    # the DeepSeek-V3-shaped layer: a 2048-token fallback chunk and the
    # 8192-token uncapped pass stay on the one-CTA kernel (256 rows per
    # group at most); the 16384-token uncapped pass takes the pair GEMM2
    d = moe.make_config(8192, 7168, 256, 8, 2048, 8, 2.0, 0, "bf16")
    assert moe.moe_gmm_kernel_choice(d) == 0
    assert moe.moe_gmm_kernel_choice(d.with_(T=2048)) == 0
    assert moe.moe_gmm_kernel_choice(d.with_(T=16384)) == 2


@pytest.mark.parametrize("case", GMM_CASES, ids=lambda c: f"{len(c[0])}x{c[1]}x{c[2]}")
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_gmm_parity(case, dtype):
    sizes, H, F, kinds = case
    if dtype == "bf16":
        R0 = int(sum(sizes))
        cq = moe.make_config(R0, H, len(sizes), 1, F, 1, 2.0, 0, dtype)
        assert moe.moe_gmm_kernel_choice(cq) == kinds
    xs, off, (wg, wu, wd), h, ys, R = run_gmm(sizes, H, F, dtype)
    want_h, want_y = ref.grouped_ffn(f64(xs[:R]), off,
                                     ref.dense_weights(f64(wg), f64(wu),
                                                       f64(wd)))
    tol = TOL[dtype]
    assert_close(f64(h[:R]), want_h, tol, 'h')
    assert_close(f64(ys[:R]), want_y, tol, 'y_sorted')
    # no row outside the groups was written
    assert torch.all(h[R:] == 0) and torch.all(ys[R:] == 0)
    # each group on its own scale; for bf16 also elementwise against the
    # dot-product scale (|h| |Wd|)_i + |y_i|
    wdh = f64(wd)
    for e in range(len(sizes)):
        a, b = int(off[e]), int(off[e + 1])
        if b > a:
            scale = None
            if dtype == "bf16":
                scale = np.abs(want_h[a:b]) @ np.abs(wdh[e]) + \
                    np.abs(want_y[a:b])
            assert_close(f64(ys[a:b]), want_y[a:b], tol,
                         f"y_sorted group {e} ({b - a} rows)", scale=scale)


def test_gmm_pair_kernel_full_dims():
    """The two-SM GEMM2 at the DeepSeek-V3 layer's dims (H=7168, F=2048):
    4157 rows in 4 ragged groups, one of them a 256-row tile plus one row.
    Every row of every group against the oracle."""
    sizes = [1500, 1100, 1300, 257]
    H, F = 7168, 2048
    R0 = int(sum(sizes))
    assert moe.moe_gmm_kernel_choice(
        moe.make_config(R0, H, 4, 1, F, 1, 2.0, 0, "bf16")) == 2
    xs, off, (wg, wu, wd), h, ys, R = run_gmm(sizes, H, F, "bf16", seed=11)
    W = expert_accessor(wg, wu, wd)
    xh = f64(xs[:R])
    hh, yh = f64(h[:R]), f64(ys[:R])
    for e in range(len(sizes)):
        a, b = int(off[e]), int(off[e + 1])
        want_h, want_y = ref.expert_ffn(xh[a:b], *W(e))
        assert_close(hh[a:b], want_h, 2e-2, f"h group {e} ({b - a} rows)")
        scale = np.abs(want_h) @ np.abs(W(e)[2]) + np.abs(want_y)
        assert_close(yh[a:b], want_y, 2e-2,
                     f"y_sorted group {e} ({b - a} rows)", scale=scale)
    assert torch.all(h[R:] == 0) and torch.all(ys[R:] == 0)


def test_gmm_small_layer_shape():
    """Zipf-like group sizes at the small layer's dims (H=1024, F=2048)."""
    sizes = [2900, 1600, 1100, 800, 560, 420, 300, 190, 120, 80, 50, 30, 20,
             12, 5, 1]
    xs, off, (wg, wu, wd), h, ys, R = run_gmm(sizes, 1024, 2048, "bf16",
                                              T=4096, k=2)
    want_h, want_y = ref.grouped_ffn(f64(xs[:R]), off,
                                     ref.dense_weights(f64(wg), f64(wu),
                                                       f64(wd)))
    assert_close(f64(h[:R]), want_h, 2e-2, 'h[:R]')
    assert_close(f64(ys[:R]), want_y, 2e-2, 'ys[:R]')


def test_gmm_pair_kernel_row_independence():
    """Large groups take the CTA-pair GEMM2 (256-row tiles): a row computed
    at another offset inside its pair tile gives the same bits."""
    H, F = 256, 256
    sizes = [1500, 700]                      # 1100 rows per group: pair
    xs, off, (wg, wu, wd), h, ys, R = run_gmm(sizes, H, F, "bf16", seed=7)
    # the same rows split into many small groups of the same experts would
    # change the weights; instead shift every row by 77 positions
    shift = 77
    xs2 = torch.cat([torch.randn(shift, H, device="cuda").to(xs.dtype),
                     xs[:R]])
    off2 = torch.tensor([0, sizes[0] + shift, R + shift], dtype=torch.int32,
                        device="cuda")
    cfg = moe.make_config(R + shift, H, 2, 1, F, 1, 2.0, 0, "bf16")
    h2 = torch.empty((R + shift, F), dtype=xs.dtype, device="cuda")
    ys2 = torch.empty((R + shift, H), dtype=xs.dtype, device="cuda")
    moe.moe_gmm_swiglu(cfg, xs2, off2, wg, wu, wd, h2, ys2)
    torch.cuda.synchronize()
    assert torch.equal(h2[shift:], h[:R])
    assert torch.equal(ys2[shift:], ys[:R])


def test_gmm_pair_and_single_cta_kernels_agree_bitwise():
    """The same rows and weights through the CTA-pair GEMM2 (2 groups of
    ~1100 rows) and the one-CTA kernel (the same groups padded with empty
    ones, so fewer rows per group): identical bits.  This keeps chunked and
    dropless passes bit-identical when they pick different kernels."""
    H, F = 512, 256
    sizes = [1500, 700]
    xs, off, (wg, wu, wd), h, ys, R = run_gmm(sizes, H, F, "bf16", seed=9)
    n_groups = 16                                 # 137 rows per group
    gexp = torch.tensor([0, 1] + [0] * (n_groups - 2), dtype=torch.int32,
                        device="cuda")
    off8 = torch.tensor([0, 1500] + [R] * (n_groups - 1), dtype=torch.int32,
                        device="cuda")
    cfg = moe.make_config(R, H, 2, 1, F, 1, 2.0, 0, "bf16")
    assert moe.moe_gmm_kernel_choice(cfg) == 2
    assert moe.moe_gmm_kernel_choice(cfg, n_groups=n_groups) == 0
    h2 = torch.empty_like(h)
    ys2 = torch.empty_like(ys)
    moe.moe_gmm_swiglu_mapped(cfg, n_groups, gexp, xs, off8, wg, wu, wd, h2,
                              ys2)
    torch.cuda.synchronize()
    assert torch.equal(h2[:R], h[:R])
    assert torch.equal(ys2[:R], ys[:R])


@pytest.mark.parametrize("dtype,H,F,sizes", [
    ("bf16", 256, 256, [200, 77, 300]),
    # fp32 (CUDA cores, 32-row tiles): groups that straddle tiles in both
    # runs, a group inside one tile, one-row groups
    ("f32", 96, 64, [45, 7, 1, 70, 33, 1, 64]),
])
def test_gmm_row_result_independent_of_tile_position(dtype, H, F, sizes):
    """The same row computed at a different offset inside its tile gives
    the same bits (this makes chunked and dropless passes agree exactly)."""
    xs, off, (wg, wu, wd), h, ys, R = run_gmm(sizes, H, F, dtype, seed=5)
    shift = 37
    xs2 = torch.cat([torch.randn(shift, H, device="cuda").to(xs.dtype),
                     xs[:R]])
    off2 = torch.from_numpy(np.concatenate(
        [[0], np.cumsum([sizes[0] + shift] + sizes[1:])]).astype(np.int32)
    ).cuda()
    cfg = moe.make_config(R + shift, H, len(sizes), 1, F, 1, 2.0, 0, dtype)
    h2 = torch.empty((R + shift, F), dtype=xs.dtype, device="cuda")
    ys2 = torch.empty((R + shift, H), dtype=xs.dtype, device="cuda")
    moe.moe_gmm_swiglu(cfg, xs2, off2, wg, wu, wd, h2, ys2)
    torch.cuda.synchronize()
    assert torch.equal(h2[shift:], h[:R])
    assert torch.equal(ys2[shift:], ys[:R])


def _draw_combine(i):
    rng = np.random.default_rng(4000 + i)
    dtype = "f32" if i % 3 == 2 else "bf16"
    H = 64 * int(rng.integers(16, 113 if dtype == "bf16" else 65))
    return int(rng.integers(1, 600)), H, dtype


@pytest.mark.parametrize("T,H,dtype", [(37, 7168, "bf16"), (300, 7168, "bf16"),
                                         (90, 3072, "f32")] +
                         [_draw_combine(i) for i in range(6)])
def test_combine_split_rows(T, H, dtype):
    """Few tokens with wide rows: each token's combine is split over several
    CTAs (column slices of 128-chunk passes, the last slice ragged at
    T = 300), against the oracle and with no column left unwritten."""
    rng = np.random.default_rng(T)
    E, S, k = 64, 8, 8
    L = rng.standard_normal((T, E)).astype(np.float32)
    oi, ow, _ = ref.route(L, k)
    p = ref.permute_indices(oi, E, S, None)
    R = int(p.group_offsets[-1])
    dt = torch.float32 if dtype == "f32" else torch.bfloat16
    ys = torch.randn(T * k, H, device="cuda").to(dt)
    cfg = moe.make_config(T, H, E, k, 128, S, 2.0, 0, dtype)
    row_of = torch.from_numpy(p.row_of.astype(np.int32)).cuda()
    w = torch.from_numpy(ow.astype(np.float32)).cuda()
    y = torch.full((T, H), float("nan"), dtype=dt, device="cuda")
    moe.moe_combine(cfg, ys, row_of, w, y)
    torch.cuda.synchronize()
    want = ref.combine(f64(ys[:R]), p.row_of, ow.astype(np.float32), H)
    got = f64(y)
    assert np.isfinite(got).all()
    assert_close(got, want, TOL[dtype], 'y')


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("k", [1, 2, 8, 13])
def test_combine_parity(dtype, k):
    rng = np.random.default_rng(k)
    T, E, S, H = 1500, 16, 4, 256 if dtype == "bf16" else 64
    L = rng.standard_normal((T, E)).astype(np.float32)
    L[:, :3] += 1.0
    oi, ow, _ = ref.route(L, k)
    # cap at half the balanced load so rows are dropped (some tokens lose all)
    C = ref.capacity(T, k, S, 0.5)
    p = ref.permute_indices(oi, E, S, C)
    R = int(p.group_offsets[-1])
    dt = torch.float32 if dtype == "f32" else torch.bfloat16
    ys = torch.randn(T * k, H, device="cuda").to(dt)
    cfg = moe.make_config(T, H, E, k, 128, S, 0.5, 0, dtype)
    row_of = torch.from_numpy(p.row_of.astype(np.int32)).cuda()
    w = torch.from_numpy(ow.astype(np.float32)).cuda()
    y = torch.empty((T, H), dtype=dt, device="cuda")
    moe.moe_combine(cfg, ys, row_of, w, y)
    torch.cuda.synchronize()
    want = ref.combine(f64(ys[:R]), p.row_of, ow.astype(np.float32), H)
    assert_close(f64(y), want, TOL[dtype], 'y')
    gone = np.all(p.row_of < 0, axis=1)
    if k <= 2:   # with few slots some tokens lose every row
        assert gone.any()
    assert torch.all(y[torch.from_numpy(gone).cuda()] == 0)
