"""The two-SM weight-gradient kernel, taken by moe_gmm_gate_up_wgrad and
moe_gmm_down_wgrad under MOE_WGRAD_ROWS16, against the oracle's segmented
weight gradient, against the one-CTA kernel on the same rows, and its
check of the 16-row statement.

Rows are laid out as the regrouped backward leaves them and beyond: several
segments with foreign rows between them, groups of 0, 16, 48, 64 + 16 and
a few hundred rows (a last k-block of 16, 32 or 48 rows), and a duplicate
group whose tiles add onto its expert.  Operands are bf16, so every product
is exact in float32; the tolerance is that of a float32 sum of a few
hundred terms.
"""
import numpy as np
import pytest
import torch

import mixture_experts_token_gb300 as moe
from oracle import moe_ref as ref
from tests.gpu_util import cfg_from, f64
from tests.parity_log import assert_close
from synth import WORKLOADS

pytestmark = pytest.mark.gpu

# (name, seed, H, F, groups, experts, segments, duplicate)
CASES = [
    ("both_pair", 1, 512, 256, 6, 6, 2, False),
    ("gate_up_pair_down_one_cta", 2, 768, 384, 5, 5, 3, False),
    ("dup_groups", 3, 256, 512, 7, 6, 2, True),
    ("one_segment", 4, 256, 256, 4, 4, 1, False),
]
SIZES16 = [0, 16, 48, 64, 80, 112, 256, 272, 400]


def layout(seed, G, n_seg, H, F):
    """Segments of 16-multiple group sizes inside one row buffer, foreign
    rows before, between and after them; bf16 operands x, dg, du, h, dy."""
    rng = np.random.default_rng(seed)
    segs, base = [], 7
    for _ in range(n_seg):
        cnt = rng.choice(SIZES16, size=G)
        cnt[rng.integers(0, G)] = 0
        off = np.concatenate([[0], np.cumsum(cnt)]).astype(np.int32)
        segs.append((off, base))
        base += int(off[-1]) + int(rng.integers(1, 40))
    rows = base + 9
    gen = torch.Generator().manual_seed(seed)
    t = {n: (torch.randn((rows, w), generator=gen) * 0.5).to(torch.bfloat16)
         for n, w in (("x", H), ("dg", F), ("du", F), ("h", F), ("dy", H))}
    return segs, rows, t


def run(cfg, segs, rows, t, flags, G, gexp, dw=None):
    dev = {n: v.cuda() for n, v in t.items()}
    segs_d = [(torch.from_numpy(o).cuda(), b) for o, b in segs]
    E, H, F = cfg.E, cfg.H, cfg.F
    if dw is None:
        dw = [torch.full(s, float("nan"), device="cuda")
              for s in ((E, H, F), (E, H, F), (E, F, H))]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ge = None if gexp is None else torch.tensor(gexp, dtype=torch.int32,
                                               device="cuda")
    ng = 0 if gexp is None else G
    moe.moe_gmm_gate_up_wgrad(cfg, segs_d, rows, dev["x"], dev["dg"],
                              dev["du"], dw[0], dw[1], flags, status,
                              n_groups=ng, group_expert=ge)
    moe.moe_gmm_down_wgrad(cfg, segs_d, rows, dev["h"], dev["dy"], dw[2],
                           flags, status, n_groups=ng, group_expert=ge)
    torch.cuda.synchronize()
    return dw, int(status.item())


def case_cfg(H, F, E):
    return cfg_from(WORKLOADS["small"], T=64, H=H, E=E, k=1, F=F, S=1)


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_rows16_weight_grads_match_oracle(case):
    name, seed, H, F, G, E, n_seg, dup = case
    segs, rows, t = layout(seed, G, n_seg, H, F)
    gexp = [g if g < E else 1 for g in range(G)] if dup else None
    cfg = case_cfg(H, F, E)
    dw, st = run(cfg, segs, rows, t, moe.MOE_WGRAD_ROWS16, G, gexp)
    assert st == 0
    ops = {n: f64(v) for n, v in t.items()}
    want = {
        "dwg": ref.segmented_weight_grads(ops["x"], ops["dg"], segs, G, E,
                                          gexp),
        "dwu": ref.segmented_weight_grads(ops["x"], ops["du"], segs, G, E,
                                          gexp),
        "dwd": ref.segmented_weight_grads(ops["h"], ops["dy"], segs, G, E,
                                          gexp),
    }
    absops = {n: np.abs(v) for n, v in ops.items()}
    scale = {
        "dwg": ref.segmented_weight_grads(absops["x"], absops["dg"], segs, G,
                                          E, gexp),
        "dwu": ref.segmented_weight_grads(absops["x"], absops["du"], segs, G,
                                          E, gexp),
        "dwd": ref.segmented_weight_grads(absops["h"], absops["dy"], segs, G,
                                          E, gexp),
    }
    kmax = max(int(o[-1]) for o, _ in segs) * n_seg
    for i, n in enumerate(("dwg", "dwu", "dwd")):
        got = f64(dw[i])
        assert np.isfinite(got).all(), n
        assert_close(got, want[n], 1e-3, n, scale=scale[n],
                     cw_bound=max(2.0 ** -14, kmax * 2.0 ** -23))
    # the one-CTA kernel on the same rows: the same sums
    one, st1 = run(cfg, segs, rows, t, 0, G, gexp)
    assert st1 == 0
    for a, b, n in zip(dw, one, ("dwg", "dwu", "dwd")):
        assert_close(f64(a), f64(b), 1e-5, n + " two-SM vs one-CTA")


def test_rows16_accumulate_doubles():
    """ROWS16 | ACCUMULATE adds the finished tile onto dW: a + a, exact."""
    H, F, G, E = 512, 256, 4, 4
    segs, rows, t = layout(5, G, 2, H, F)
    cfg = case_cfg(H, F, E)
    dw, st = run(cfg, segs, rows, t, moe.MOE_WGRAD_ROWS16, G, None)
    first = [a.clone() for a in dw]
    dw, st2 = run(cfg, segs, rows, t,
                  moe.MOE_WGRAD_ROWS16 | moe.MOE_WGRAD_ACCUMULATE, G, None,
                  dw)
    assert st == 0 and st2 == 0
    for a, b in zip(first, dw):
        assert torch.equal(b, a * 2)


def test_rows16_statement_checked():
    """A group of 24 rows under ROWS16: the two-SM kernel raises
    MOE_DEV_UNALIGNED before any copy and leaves dW as it was (accumulate,
    so no zeroing runs either)."""
    H, F, G, E = 256, 256, 4, 4
    segs, rows, t = layout(9, G, 1, H, F)
    off = segs[0][0].copy()
    off[2:] += 8                     # group 1 gets 8 more rows (not 16k)
    segs = [(off, segs[0][1])]
    rows = max(rows, segs[0][1] + int(off[-1]) + 1)
    t = {n: torch.cat([v, torch.zeros((rows - v.shape[0], v.shape[1]),
                                      dtype=v.dtype)]) if v.shape[0] < rows
         else v for n, v in t.items()}
    cfg = case_cfg(H, F, E)
    dw0 = [torch.full(s, 7.0, device="cuda")
           for s in ((E, H, F), (E, H, F), (E, F, H))]
    dw, st = run(cfg, segs, rows, t,
                 moe.MOE_WGRAD_ROWS16 | moe.MOE_WGRAD_ACCUMULATE, G, None,
                 dw0)
    assert st & moe.MOE_DEV_UNALIGNED
    assert not st & moe.MOE_DEV_TIMEOUT
    for a in dw:
        assert bool((a == 7.0).all())
    # without the statement the one-CTA kernel takes the same rows
    one, st1 = run(cfg, segs, rows, t, 0, G, None)
    assert st1 == 0
    ops = {n: f64(v) for n, v in t.items()}
    want = ref.segmented_weight_grads(ops["x"], ops["dg"], segs, G, E)
    assert_close(f64(one[0]), want, 1e-3, "dwg one-CTA")


def draw_case(i):
    """Seeded random case: H, F multiples of 128 (some of 256, some not),
    1-4 segments, 16-row groups of 0-520 rows, sometimes a duplicate map."""
    rng = np.random.default_rng(7000 + i)
    H = int(rng.choice([256, 384, 512, 768]))
    F = int(rng.choice([128, 256, 384, 512]))
    E = int(rng.integers(1, 7))
    dup = bool(rng.integers(0, 2)) and E > 1
    G = E + (int(rng.integers(1, 3)) if dup else 0)
    gexp = None
    if dup:
        gexp = list(range(E)) + [int(rng.integers(0, E)) for _ in range(G - E)]
    n_seg = int(rng.integers(1, 5))
    segs, base = [], int(rng.integers(0, 20))
    for _ in range(n_seg):
        cnt = rng.integers(0, 33, size=G) * 16
        off = np.concatenate([[0], np.cumsum(cnt)]).astype(np.int32)
        segs.append((off, base))
        base += int(off[-1]) + int(rng.integers(0, 30))
    rows = base + 3
    gen = torch.Generator().manual_seed(8000 + i)
    t = {n: (torch.randn((rows, w), generator=gen) * 0.5).to(torch.bfloat16)
         for n, w in (("x", H), ("dg", F), ("du", F), ("h", F), ("dy", H))}
    acc = bool(rng.integers(0, 2))
    return H, F, E, G, gexp, segs, rows, t, acc


@pytest.mark.parametrize("i", range(10))
def test_rows16_random_cases(i):
    """Ten seeded random layouts through the ROWS16 entries (the two-SM
    kernel where the gradient's rows are a multiple of 256, else the
    one-CTA kernel), with and without ACCUMULATE onto a known dW, against
    the oracle's segmented weight gradient."""
    H, F, E, G, gexp, segs, rows, t, acc = draw_case(i)
    cfg = case_cfg(H, F, E)
    flags = moe.MOE_WGRAD_ROWS16 | (moe.MOE_WGRAD_ACCUMULATE if acc else 0)
    init = [torch.full(s, 0.25, device="cuda")
            for s in ((E, H, F), (E, H, F), (E, F, H))]
    dw, st = run(cfg, segs, rows, t, flags, G, gexp,
                 [x.clone() for x in init])
    assert st == 0
    ops = {n: f64(v) for n, v in t.items()}
    for k, (got, p_, q_) in enumerate(((dw[0], "x", "dg"), (dw[1], "x", "du"),
                                       (dw[2], "h", "dy"))):
        want = ref.segmented_weight_grads(ops[p_], ops[q_], segs, G, E, gexp)
        if acc:
            want = want + 0.25
        got = f64(got)
        assert np.isfinite(got).all()
        assert_close(got, want, 1e-3, f"d{q_} case {i}")
