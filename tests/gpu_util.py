"""Helpers for the GPU parity tests: run the library stage by stage through
the C ABI binding and bring results back as numpy; compare with the oracle.

Inputs always come from ``synth`` (or are hand-built here); the oracle only
ever receives those inputs, never an output of the CUDA path.
"""
from __future__ import annotations

import numpy as np
import torch

import mixture_experts_token_gb300 as moe
from oracle import moe_ref as ref

TOL = {"f32": 1e-4, "bf16": 2e-2}


def cfg_from(wl, **over):
    kw = dict(T=wl.T, H=wl.H, E=wl.E, k=wl.k, F=wl.F, S=wl.S,
              factor=wl.factor, n_chunks=wl.n_chunks, dtype=wl.dtype,
              renorm=wl.renorm, redundant_slots=wl.redundant_slots)
    kw.update(over)
    return moe.make_config(kw["T"], kw["H"], kw["E"], kw["k"], kw["F"],
                           kw["S"], kw["factor"], kw["n_chunks"], kw["dtype"],
                           kw["renorm"], kw["redundant_slots"])


def np_(t):
    t = t.detach()
    if t.dtype == torch.bfloat16:
        t = t.float()
    return t.cpu().numpy()


def f64(t):
    """Exact float64 copy of a device tensor (bf16/f32 values are exact)."""
    return t.detach().to("cpu", torch.float64).numpy()


def host_logits(wl, x, T=None):
    """The workload's router logits [T, E] as float32, computed by the
    oracle in float64 from x (device or host), the router weight and the
    logit offset that synth draws (x @ Wr + offset), a few thousand rows at
    a time.  Both sides of a routing parity test take these as input."""
    from synth import make_logit_offset, make_router_weight
    T = x.shape[0] if T is None else T
    wr = f64(make_router_weight(wl))
    off = make_logit_offset(wl, T=T)
    out = np.empty((T, wl.E), dtype=np.float32)
    for a in range(0, T, 4096):
        z = min(T, a + 4096)
        out[a:z] = ref.router_logits(
            f64(x[a:z]), wr, None if off is None else off[a:z]).astype(
                np.float32)
    return out


def gpu_route(cfg, logits_np, status=None):
    T, E = logits_np.shape
    d = torch.from_numpy(np.ascontiguousarray(logits_np)).cuda()
    idx = torch.empty((T, cfg.k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, cfg.k), dtype=torch.float32, device="cuda")
    moe.moe_route(cfg, d, idx, w, status)
    return idx, w


def gpu_check(cfg, idx):
    b = {n: torch.empty(s, dtype=dt, device="cuda") for n, s, dt in (
        ("counts", cfg.E, torch.int32), ("offsets", cfg.E + 1, torch.int32),
        ("shard", cfg.S, torch.int32), ("flag", 1, torch.int32),
        ("req", 1, torch.float32), ("cap", 1, torch.int32))}
    moe.moe_check_overflow(cfg, idx, b["counts"], b["offsets"], b["shard"],
                           b["flag"], b["req"], b["cap"])
    torch.cuda.synchronize()
    return {n: np_(v) for n, v in b.items()}


def gpu_permute(cfg, x, idx, capped):
    bufs = moe.alloc_step_buffers(cfg)
    moe.moe_permute(cfg, x, idx, capped, bufs["x_sorted"], bufs["row_of"],
                    bufs["sorted_token"], bufs["group_offsets"],
                    bufs["uniq_offsets"], bufs["uniq_tokens"],
                    bufs["expand_idx"], bufs["n_dropped"], bufs["permute_ws"])
    torch.cuda.synchronize()
    return bufs


def compare_permutation(bufs, p, x_host=None):
    """GPU permute buffers against an oracle Permutation, bit for bit."""
    R = int(p.group_offsets[-1])
    U = int(p.uniq_offsets[-1])
    assert np.array_equal(np_(bufs["group_offsets"]), p.group_offsets)
    assert np.array_equal(np_(bufs["row_of"]), p.row_of)
    assert np.array_equal(np_(bufs["sorted_token"])[:R], p.sorted_token)
    assert np.array_equal(np_(bufs["uniq_offsets"]), p.uniq_offsets)
    assert np.array_equal(np_(bufs["uniq_tokens"])[:U], p.uniq_tokens)
    assert np.array_equal(np_(bufs["expand_idx"])[:R], p.expand_idx)
    assert int(np_(bufs["n_dropped"])[0]) == p.n_dropped
    if x_host is not None and R > 0:
        xs = bufs["x_sorted"][:R]
        want = x_host[torch.from_numpy(p.sorted_token).long()]
        assert torch.equal(xs.cpu(), want), "x_sorted rows differ"


def normwise(got, ref_):
    return ref.normwise_error(got, ref_)


def expert_accessor(wg, wu, wd):
    """Oracle weight accessor over device tensors: one expert at a time is
    copied to the host as float64 (exact for bf16/f32)."""
    cache = {}

    def get(e):
        if e not in cache:
            cache.clear()
            cache[e] = (f64(wg[e]), f64(wu[e]), f64(wd[e]))
        return cache[e]
    return get
