"""Record of every float parity comparison made in a test session.

Each comparison of a GPU output with the float64 oracle asserts the
normwise measure (max |g - r| / max |r|) against its tolerance and also
records the largest elementwise relative error (each |g_i - r_i| over
max(|r_i|, 1e-3 max |r|)), so that both figures appear in the session's
summary (see conftest.py) and, with MOE_PARITY_LOG set, in a CSV file.
"""
from __future__ import annotations

import os

from oracle import moe_ref as ref

RECORDS = []   # (test id, what, normwise, elementwise, tolerance)


def _test_id() -> str:
    cur = os.environ.get("PYTEST_CURRENT_TEST", "")
    return cur.rsplit(" ", 1)[0] if cur else "(outside a test)"


def assert_close(got, want, tol: float, what: str = "") -> tuple:
    """Asserts normwise error <= tol; records it with the elementwise
    error.  Returns (normwise, elementwise)."""
    nw = ref.normwise_error(got, want)
    ew = ref.elementwise_error(got, want)
    RECORDS.append((_test_id(), what, nw, ew, tol))
    assert nw <= tol, (f"{what}: normwise error {nw:.3g} > {tol} "
                       f"(max elementwise relative error {ew:.3g})")
    return nw, ew


def summary_lines():
    if not RECORDS:
        return []
    out = [f"float parity: {len(RECORDS)} comparisons "
           "(normwise asserted; elementwise = max_i |g-r| / "
           "max(|r_i|, 1e-3 max|r|))",
           f"{'normwise':>10} {'elementwise':>12} {'tol':>7}  test / output"]
    for tid, what, nw, ew, tol in RECORDS:
        out.append(f"{nw:10.3e} {ew:12.3e} {tol:7.0e}  {tid} {what}")
    worst = max(RECORDS, key=lambda r: r[2] / r[4])
    out.append(f"largest normwise / tolerance: {worst[2] / worst[4]:.3f} "
               f"({worst[0]} {worst[1]})")
    return out


def write_csv(path: str):
    with open(path, "w") as f:
        f.write("test,output,normwise,elementwise,tol\n")
        for tid, what, nw, ew, tol in RECORDS:
            f.write(f"{tid},{what},{nw:.6e},{ew:.6e},{tol:g}\n")
