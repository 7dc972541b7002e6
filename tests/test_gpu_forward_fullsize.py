"""GPU parity of the forward expert FFN at full size, whole groups at a time.

The layer tests sample tokens; this file compares every row of a few
expert groups of h and y_sorted with the float64 oracle's expert FFN over
exactly those rows, at the DeepSeek-V3- and Llama4-Maverick-shaped layers'
dims and in the launch configurations the benchmark times:

* DeepSeek-V3 layer, Zipf s=1.2: the first fallback chunk (2048 tokens,
  uncapped; "Support moe_dropless_fallback=layer on the ragged all-to-all
  MoE path", section How: the fallback runs the layer chunk by chunk with
  the worst-case buffer) and the whole 8192-token batch as one uncapped
  pass, under Zipf and under uniform routing;
* Llama4-Maverick layer, uniform routing: the capped pass the layer takes
  (no shard overflows, section End-to-end's EP16 configuration).

Per pass the experts are: the hottest (for DeepSeek-V3 a group of many
128-row m-tiles, where the heavy/light tile interleave and the long
K = 7168 loop run), the one nearest the median count, and the smallest
non-empty group (1-5 rows where one exists).  Group offsets must equal the
oracle's bit for bit; h and y_sorted are held to the bf16 tolerance per
group, with the elementwise error recorded beside it, and every y_sorted
element to 2^-8 of its dot-product scale (|h| |Wd|)_i + |y_i|.
"""
import numpy as np
import pytest
import torch

import mixture_experts_token_gb300 as moe
from oracle import moe_ref as ref
from synth import WORKLOADS, make_weights, make_x
from tests.gpu_util import cfg_from, expert_accessor, f64, gpu_permute, \
    gpu_route, host_logits, np_
from tests.parity_log import assert_close

pytestmark = pytest.mark.gpu


def pick_experts(counts):
    nz = np.nonzero(counts)[0]
    hot = int(np.argmax(counts))
    med = float(np.median(counts[nz]))
    mid = int(nz[np.argmin(np.abs(counts[nz] - med))])
    tiny = [int(e) for e in nz if 1 <= counts[e] <= 5]
    small = tiny[0] if tiny else int(nz[np.argmin(counts[nz])])
    return sorted({hot, mid, small})


def check_pass(wl, cfg, x, L, W, capped, label):
    """Route, permute, GEMM1 + SwiGLU and GEMM2 through the C ABI; then the
    chosen groups against the oracle."""
    idx, _ = gpu_route(cfg, L)
    b = gpu_permute(cfg, x, idx, capped)
    moe.moe_gmm_gate_up(cfg, b["x_sorted"], b["group_offsets"], W[0], W[1],
                        b["h"], b["status"])
    moe.moe_gmm_down(cfg, b["h"], b["group_offsets"], W[2], b["y_sorted"],
                     b["status"])
    torch.cuda.synchronize()
    assert int(b["status"].item()) == 0

    oi, _, _ = ref.route(L, cfg.k)
    assert np.array_equal(np_(idx), oi)
    C = ref.capacity(cfg.T, cfg.k, cfg.S, cfg.ragged_buffer_factor)
    p = ref.permute_indices(oi, cfg.E, cfg.S, C if capped else None)
    assert np.array_equal(np_(b["group_offsets"]), p.group_offsets)
    counts = np.diff(p.group_offsets)
    get = expert_accessor(*W)
    chosen = pick_experts(counts)
    for e in chosen:
        a, z = int(p.group_offsets[e]), int(p.group_offsets[e + 1])
        tok = torch.from_numpy(p.sorted_token[a:z].astype(np.int64)).cuda()
        wts = get(e)
        want_h, want_y = ref.expert_ffn(f64(x[tok]), *wts)
        assert_close(f64(b["h"][a:z]), want_h, 2e-2,
                     f"{label} h expert {e} ({z - a} rows)")
        scale = np.abs(want_h) @ np.abs(wts[2]) + np.abs(want_y)
        assert_close(f64(b["y_sorted"][a:z]), want_y, 2e-2,
                     f"{label} y_sorted expert {e} ({z - a} rows)",
                     scale=scale)
    return counts, chosen


def test_fullsize_dsv3_groups():
    wl = WORKLOADS["dsv3"]
    x = make_x(wl, "cuda")
    W = make_weights(wl, "cuda")
    L = host_logits(wl, x)
    full = cfg_from(wl)
    ct = moe.moe_chunk_tokens(full)
    assert ct == 2048 and moe.moe_num_chunks(full) == 4
    # the first fallback chunk: 2048 tokens, uncapped, as the layer runs it
    chunk = cfg_from(wl, T=ct, factor=-1.0, n_chunks=0)
    counts, chosen = check_pass(wl, chunk, x[:ct], np.ascontiguousarray(L[:ct]),
                                W, False, "dsv3 chunk 0")
    assert counts[chosen[0]] > 0
    assert max(counts) > 4 * 128     # the hot group spans many m-tiles
    # the whole batch as one uncapped pass, Zipf and uniform routing
    unc = cfg_from(wl, factor=-1.0)
    counts, _ = check_pass(wl, unc, x, L, W, False, "dsv3 uncapped zipf")
    assert max(counts) > 16 * 128
    Lu = host_logits(wl.with_(routing="uniform", zipf_s=0.0), x)
    check_pass(wl, unc, x, Lu, W, False, "dsv3 uncapped uniform")
    del x, W
    torch.cuda.empty_cache()


def test_fullsize_l4mav_groups():
    wl = WORKLOADS["l4mav"]
    x = make_x(wl, "cuda")
    W = make_weights(wl, "cuda")
    L = host_logits(wl, x)
    cfg = cfg_from(wl)
    oi, _, _ = ref.route(L, wl.k)
    C = ref.capacity(wl.T, wl.k, wl.S, wl.factor)
    assert not ref.overflow_flag(
        ref.shard_counts(ref.expert_counts(oi, wl.E), wl.S), C)
    check_pass(wl, cfg, x, L, W, True, "l4mav capped")
    del x, W
    torch.cuda.empty_cache()
