"""C ABI checks that need no GPU: the library loads, exports every function
include/moe.h declares, validates arguments on the host, and its host-side
formulas (capacity, chunk plan) agree with the oracle's."""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe.h")


@pytest.fixture(scope="module")
def m():
    import mixture_experts_token_gb300 as m
    if not os.path.exists(m.LIB_PATH):
        from mixture_experts_token_gb300 import build
        build.build()
    m.lib()
    return m


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^[A-Za-z_][\w\s\*]*?\b(moe_\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("moe_route", "moe_check_overflow", "moe_permute",
              "moe_gmm_swiglu", "moe_combine", "moe_layer_dropless_chunked",
              "moe_workspace_bytes", "moe_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(m):
    h = ctypes.CDLL(m.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(h, n)]
    assert not missing, missing
    out = subprocess.run(["nm", "-D", "--defined-only", m.LIB_PATH],
                         capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (moe_\w+)", out))
    assert set(declared_functions()) <= exported


def cfg_of(m, T=64, H=64, E=8, k=2, F=128, S=2, factor=2.0, n_chunks=0,
           dtype="bf16", renorm=False):
    return m.make_config(T, H, E, k, F, S, factor, n_chunks, dtype, renorm)


def test_config_validation(m):
    ok = cfg_of(m)
    assert m.moe_validate_config(ok) == m.MOE_OK
    bad = [dict(k=0), dict(k=9), dict(E=0), dict(E=2048, k=2), dict(S=3),
           dict(S=0), dict(T=-1), dict(H=4), dict(F=4), dict(k=33, E=64),
           dict(S=128, E=256), dict(n_chunks=-2), dict(factor=float("nan"))]
    for kw in bad:
        assert m.moe_validate_config(cfg_of(m, **kw)) == \
            m.MOE_ERR_INVALID_ARG, kw
    c = cfg_of(m)
    c.dtype = 7
    assert m.moe_validate_config(c) == m.MOE_ERR_INVALID_ARG
    c = cfg_of(m)
    c.renorm = 2
    assert m.moe_validate_config(c) == m.MOE_ERR_INVALID_ARG
    # fp32 rows need H % 4 == 0, bf16 rows H % 8 == 0
    assert m.moe_validate_config(cfg_of(m, H=12, dtype="f32")) == m.MOE_OK
    assert m.moe_validate_config(cfg_of(m, H=12)) == m.MOE_ERR_INVALID_ARG


def test_bad_arguments_are_rejected_before_any_launch(m):
    c = cfg_of(m)
    st = m.lib().moe_route(ctypes.byref(c), None, None, None, None, None)
    assert st == m.MOE_ERR_INVALID_ARG
    st = m.lib().moe_permute(ctypes.byref(c), None, None, 1, None, None, None,
                             None, None, None, None, None, None, 0, None)
    assert st == m.MOE_ERR_INVALID_ARG
    # a misaligned activation pointer
    fake = 0x1000
    st = m.lib().moe_combine(ctypes.byref(c), ctypes.c_void_p(fake + 8),
                             ctypes.c_void_p(fake), ctypes.c_void_p(fake),
                             ctypes.c_void_p(fake), None)
    assert st == m.MOE_ERR_INVALID_ARG
    # workspace too small
    p = ctypes.c_void_p(fake)
    st = m.lib().moe_permute(ctypes.byref(c), p, p, 1, p, p, p, p, p, p, p, p,
                             p, 16, None)
    assert st == m.MOE_ERR_WORKSPACE
    # the two halves of the permute: a plan needs both of its arrays, and
    # each half needs the permute workspace
    st = m.lib().moe_permute_tables(ctypes.byref(c), p, 1, p, None, p, p, p,
                                    p, p, p, 1 << 20, None)
    assert st == m.MOE_ERR_INVALID_ARG
    st = m.lib().moe_permute_tables(ctypes.byref(c), p, 1, None, None, p, p,
                                    p, p, p, p, 16, None)
    assert st == m.MOE_ERR_WORKSPACE
    st = m.lib().moe_permute_scatter(ctypes.byref(c), p, p, p, p, p, p, None,
                                     0, None)
    assert st == m.MOE_ERR_WORKSPACE
    st = m.lib().moe_permute_scatter(ctypes.byref(c), ctypes.c_void_p(fake + 8),
                                     p, p, p, p, p, p, 1 << 20, None)
    assert st == m.MOE_ERR_INVALID_ARG
    # bf16 GEMM shape outside the tensor-core kernels
    c2 = cfg_of(m, H=72, F=128)
    st = m.lib().moe_gmm_swiglu(ctypes.byref(c2), p, p, p, p, p, p, p, None,
                                None)
    assert st == m.MOE_ERR_UNSUPPORTED
    assert m.moe_status_string(m.MOE_ERR_WORKSPACE) == \
        "workspace missing or too small"


def test_capacity_matches_oracle(m):
    from oracle import moe_ref as ref
    rng = np.random.default_rng(0)
    for _ in range(500):
        S = int(rng.choice([1, 2, 4, 8, 16]))
        E = S * int(rng.integers(1, 9))
        k = int(rng.integers(1, min(E, 32) + 1))
        T = int(rng.integers(0, 5000))
        factor = float(rng.choice([-1.0, 0.0, 0.1, 0.3, 0.5, 1.0, 1.25,
                                   2.0, 3.7, 100.0]))
        c = cfg_of(m, T=T, E=E, k=k, S=S, factor=factor)
        C = ref.capacity(T, k, S, factor)
        assert m.moe_capacity_rows(c) == (-1 if C is None else C)
        plan = ref.chunk_plan(T, k, E, S, C)
        assert m.moe_num_chunks(c) == len(plan)
        if plan:
            assert m.moe_chunk_tokens(c) == plan[0][1] - plan[0][0]
        for n in (1, 3, 8):
            c.n_chunks = n
            plan = ref.chunk_plan(T, k, E, S, C, n_chunks=n)
            assert m.moe_num_chunks(c) == len(plan)


def test_workspace_sizes(m):
    for name in ("small", "dsv3", "l4mav"):
        from synth import WORKLOADS
        w = WORKLOADS[name]
        c = cfg_of(m, T=w.T, H=w.H, E=w.E, k=w.k, F=w.F, S=w.S,
                   factor=w.factor)
        perm = m.moe_workspace_bytes(c, m.MOE_WS_PERMUTE)
        layer = m.moe_workspace_bytes(c, m.MOE_WS_LAYER)
        chunked = m.moe_workspace_bytes(c, m.MOE_WS_CHUNKED)
        assert 0 < perm < layer
        assert 0 < chunked <= layer
        # the layer workspace holds x_sorted, h and y_sorted for T*k rows
        R = w.T * w.k
        assert layer >= R * (2 * w.H + w.F) * 2
    assert m.moe_workspace_bytes(cfg_of(m, k=0), m.MOE_WS_LAYER) == 0


def test_backward_workspace_sizes(m):
    from synth import WORKLOADS
    for name in ("small", "dsv3", "l4mav"):
        w = WORKLOADS[name]
        c = cfg_of(m, T=w.T, H=w.H, E=w.E, k=w.k, F=w.F, S=w.S,
                   factor=w.factor)
        R = w.T * w.k
        gb = m.moe_workspace_bytes(c, m.MOE_WS_GMM_BACKWARD)
        lb = m.moe_workspace_bytes(c, m.MOE_WS_LAYER_BACKWARD)
        layer = m.moe_workspace_bytes(c, m.MOE_WS_LAYER)
        # dg and du [T*k, F]
        assert gb >= 2 * R * w.F * 2
        # the forward layer buffers + g, u, dg, du, dy_sorted, dx_sorted,
        # and the regrouped copies of five row buffers (T*k + 16*E rows)
        assert lb >= layer + R * (4 * w.F + 2 * w.H) * 2 + \
            (R + 16 * w.E) * (2 * w.H + 3 * w.F) * 2
        # one group-offset row per possible pass
        small = cfg_of(m, T=w.T, H=w.H, E=w.E, k=w.k, F=w.F, S=w.S,
                       factor=w.factor, n_chunks=1)
        assert m.moe_workspace_bytes(small, m.MOE_WS_LAYER_BACKWARD) <= lb


def test_backward_arguments_are_rejected_before_any_launch(m):
    c = cfg_of(m, H=128)   # a shape the tensor-core kernels cover
    p = ctypes.c_void_p(0x1000)
    seg = (m.MoeRowSegment * 1)()
    seg[0].group_offsets = 0x1000
    seg[0].first_row = 0
    lib = m.lib()
    # regrouping: no ranges, too many ranges, an output too small
    args = (p, p, p, p, p, p, p, p, p, p, p)
    rows = c.T * c.k + 16 * c.E
    assert lib.moe_regroup_rows(ctypes.byref(c), 0, seg, 0, rows, *args,
                                None, None) == m.MOE_ERR_INVALID_ARG
    assert lib.moe_regroup_rows(ctypes.byref(c), 0, seg, 65, rows, *args,
                                None, None) == m.MOE_ERR_INVALID_ARG
    assert lib.moe_regroup_rows(ctypes.byref(c), 0, seg, 1, rows - 1, *args,
                                None, None) == m.MOE_ERR_INVALID_ARG
    # a group count beyond the configuration's groups
    assert lib.moe_regroup_rows(ctypes.byref(c), c.E + 1, seg, 1, rows,
                                *args, None, None) == m.MOE_ERR_INVALID_ARG
    # per-row weights are a bf16 path
    c32 = cfg_of(m, H=128, dtype="f32")
    assert lib.moe_regroup_rows(ctypes.byref(c32), 0, seg, 1, rows, *args,
                                p, None) == m.MOE_ERR_UNSUPPORTED
    # the split combine backward: parts per row, f32 rejected, bad pointers
    assert m.moe_row_dot_parts(c) == c.F // 128           # F = 128
    assert m.moe_row_dot_parts(cfg_of(m, F=512)) == 2      # 256-wide tiles
    assert m.moe_row_dot_parts(cfg_of(m, F=384)) == 3
    assert lib.moe_gmm_down_dgrad_rows(
        ctypes.byref(c32), 0, None, p, p, p, p, p, p, p, p, p, p, None,
        None) == m.MOE_ERR_UNSUPPORTED
    assert lib.moe_gmm_down_dgrad_rows(
        ctypes.byref(c), 0, None, p, p, p, p, None, p, p, p, p, p, None,
        None) == m.MOE_ERR_INVALID_ARG                      # h missing
    assert lib.moe_combine_backward_rows(ctypes.byref(c), p, p, p, p, None,
                                         None) == m.MOE_ERR_INVALID_ARG
    assert lib.moe_combine_weight_grad(ctypes.byref(c), p, None, p,
                                       None) == m.MOE_ERR_INVALID_ARG
    # a group map without its group count
    assert lib.moe_gmm_down_wgrad(ctypes.byref(c), 0, p, seg, 1, rows, p, p,
                                  p, 0, None, None) == m.MOE_ERR_INVALID_ARG
    # weight gradients: a negative range start, an unknown flag bit
    seg[0].first_row = -1
    assert lib.moe_gmm_down_wgrad(ctypes.byref(c), 0, None, seg, 1, rows, p, p, p, 0,
                                  None, None) == m.MOE_ERR_INVALID_ARG
    seg[0].first_row = 0
    assert lib.moe_gmm_down_wgrad(ctypes.byref(c), 0, None, seg, 1, rows, p, p, p, 4,
                                  None, None) == m.MOE_ERR_INVALID_ARG
    # layer backward: no workspace
    info = m.MoeLayerInfo()
    assert lib.moe_layer_backward(ctypes.byref(c), p, p, p, p, p, p, p, p, p,
                                  p, p, 0, ctypes.byref(info), None, None, 0,
                                  None) == m.MOE_ERR_WORKSPACE
