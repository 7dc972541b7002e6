"""Record of every float parity comparison made in a test session.

Each comparison of a GPU output with the float64 oracle asserts the
normwise measure (max |g - r| / max |r|) against its tolerance and also
records the largest elementwise relative error (each |g_i - r_i| over
max(|r_i|, 1e-3 max |r|)), so that both figures appear in the session's
summary (see conftest.py) and, with MOE_PARITY_LOG set, in a CSV file.

Where an output is a dot product whose terms the test can bound (GEMM2's
y_sorted = h Wd), an elementwise bound is also asserted: |g_i - r_i| <=
bound * s_i with s_i = (|h| |Wd|)_i + |r_i|, the error a bf16 rounding of
each h element and of the result can cause in that element whatever the
cancellation in the sum (the plain elementwise relative error of such an
element is unbounded when the terms cancel).
"""
from __future__ import annotations

import os

import numpy as np

from oracle import moe_ref as ref

RECORDS = []   # dicts: test, what, normwise, elementwise, tol, cw, cw_bound


def _test_id() -> str:
    cur = os.environ.get("PYTEST_CURRENT_TEST", "")
    return cur.rsplit(" ", 1)[0] if cur else "(outside a test)"


def assert_close(got, want, tol: float, what: str = "", scale=None,
                 cw_bound: float = 2.0 ** -8) -> tuple:
    """Asserts normwise error <= tol (and, given the per-element scale s of
    a dot-product output, |g - r| <= cw_bound * s elementwise); records the
    figures.  Returns (normwise, elementwise)."""
    nw = ref.normwise_error(got, want)
    ew = ref.elementwise_error(got, want)
    cw = None
    if scale is not None:
        g = np.asarray(got, dtype=np.float64)
        r = np.asarray(want, dtype=np.float64)
        s = np.asarray(scale, dtype=np.float64)
        d = np.abs(g - r)
        cw = float(np.max(d / np.maximum(s, 1e-300))) if d.size else 0.0
    RECORDS.append(dict(test=_test_id(), what=what, nw=nw, ew=ew, tol=tol,
                        cw=cw, cw_bound=cw_bound if cw is not None else None))
    assert nw <= tol, (f"{what}: normwise error {nw:.3g} > {tol} "
                       f"(max elementwise relative error {ew:.3g})")
    if cw is not None:
        assert cw <= cw_bound, (f"{what}: elementwise error {cw:.3g} of the "
                                f"dot-product scale > {cw_bound:.3g}")
    return nw, ew


def assert_close_device(pairs, tol: float, what: str = "") -> tuple:
    """assert_close for device tensors too large to copy to the host: the
    same two measures over the (got, want) tensor pairs taken together
    (pieces of one output), computed on the device in float64, a slice of
    rows at a time."""
    import torch
    pairs = [(g, w) for g, w in pairs if g.numel()]
    dmax, rmax = 0.0, 0.0
    for got, want in pairs:
        g2, r2 = got.reshape(got.shape[0], -1), want.reshape(want.shape[0], -1)
        step = max(1, (1 << 26) // max(1, g2.shape[1]))
        for a in range(0, g2.shape[0], step):
            g = g2[a:a + step].to(torch.float64)
            r = r2[a:a + step].to(torch.float64)
            if g.numel():
                dmax = max(dmax, float((g - r).abs().max()))
                rmax = max(rmax, float(r.abs().max()))
    nw = dmax / rmax if rmax > 0 else dmax
    floor = 1e-3 * rmax
    ew = dmax if floor == 0 else 0.0
    for got, want in (pairs if floor > 0 else []):
        g2, r2 = got.reshape(got.shape[0], -1), want.reshape(want.shape[0], -1)
        step = max(1, (1 << 26) // max(1, g2.shape[1]))
        for a in range(0, g2.shape[0], step):
            g = g2[a:a + step].to(torch.float64)
            r = r2[a:a + step].to(torch.float64)
            if g.numel():
                den = torch.clamp(r.abs(), min=floor)
                ew = max(ew, float(((g - r).abs() / den).max()))
    RECORDS.append(dict(test=_test_id(), what=what, nw=nw, ew=ew, tol=tol,
                        cw=None, cw_bound=None))
    assert nw <= tol, (f"{what}: normwise error {nw:.3g} > {tol} "
                       f"(max elementwise relative error {ew:.3g})")
    return nw, ew


def summary_lines():
    if not RECORDS:
        return []
    out = [f"float parity: {len(RECORDS)} comparisons (normwise asserted; "
           "elementwise = max_i |g-r| / max(|r_i|, 1e-3 max|r|); "
           "dot-product elementwise = max_i |g-r| / ((|h||Wd|)_i + |r_i|), "
           "asserted where shown)",
           f"{'normwise':>10} {'elementwise':>12} {'tol':>7} "
           f"{'dot-elem':>10}  test / output"]
    for r in RECORDS:
        cw = f"{r['cw']:10.3e}" if r["cw"] is not None else f"{'-':>10}"
        out.append(f"{r['nw']:10.3e} {r['ew']:12.3e} {r['tol']:7.0e} {cw}  "
                   f"{r['test']} {r['what']}")
    worst = max(RECORDS, key=lambda r: r["nw"] / r["tol"])
    out.append(f"largest normwise / tolerance: {worst['nw'] / worst['tol']:.3f} "
               f"({worst['test']} {worst['what']})")
    cws = [r for r in RECORDS if r["cw"] is not None]
    if cws:
        w = max(cws, key=lambda r: r["cw"] / r["cw_bound"])
        out.append(f"largest dot-product elementwise / bound: "
                   f"{w['cw'] / w['cw_bound']:.3f} ({w['test']} {w['what']})")
    return out


def write_csv(path: str):
    with open(path, "w") as f:
        f.write("test,output,normwise,elementwise,tol,dot_elementwise\n")
        for r in RECORDS:
            cw = "" if r["cw"] is None else f"{r['cw']:.6e}"
            f.write(f"{r['test']},{r['what']},{r['nw']:.6e},{r['ew']:.6e},"
                    f"{r['tol']:g},{cw}\n")
