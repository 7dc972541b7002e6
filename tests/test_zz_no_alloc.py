"""moe_permute_noalloc against moe_permute, through the C ABI (GPU).

Callers that cannot allocate device memory (a framework pool owns it all, or
cudaMalloc's implicit synchronisation is off limits) use moe_permute_noalloc,
which keeps the permute's scratch in a fixed 8 MiB device array inside the
library.  Its outputs must equal those of the workspace version exactly
(they are integers and byte copies), on two calls in a row: the array keeps
the previous call's contents, so the second call, on a different batch,
would show any stale state.  Sizes whose scratch exceeds the array are
refused.
"""
import pytest
import torch

import mixture_experts_token_gb300 as moe
from synth import WORKLOADS, make_x, sweep_workload
from tests.gpu_util import cfg_from, gpu_route, host_logits

pytestmark = pytest.mark.gpu

OUTS = ("x_sorted", "row_of", "sorted_token", "group_offsets",
        "uniq_offsets", "uniq_tokens", "expand_idx", "n_dropped")


def _permute(cfg, x, idx, capped, noalloc):
    b = moe.alloc_step_buffers(cfg)
    for n in OUTS:
        b[n].fill_(-7) if b[n].dtype == torch.int32 else b[n].zero_()
    args = [cfg, x, idx, capped] + [b[n] for n in OUTS]
    if noalloc:
        moe.moe_permute_noalloc(*args)
    else:
        moe.moe_permute(*(args + [b["permute_ws"]]))
    torch.cuda.synchronize()
    return b


def _case(wl, factor):
    cfg = cfg_from(wl, factor=factor)
    x = make_x(wl, "cuda")
    idx, _ = gpu_route(cfg, host_logits(wl, x))
    return cfg, x, idx


def test_noalloc_matches_workspace_version_twice():
    cases = [_case(sweep_workload(4096, "zipf"), 2.0),
             _case(WORKLOADS["small"].with_(T=1000, H=256, k=4), 0.5)]
    for capped in (True, False):
        for cfg, x, idx in cases:          # two calls in a row, new batch
            want = _permute(cfg, x, idx, capped, noalloc=False)
            got = _permute(cfg, x, idx, capped, noalloc=True)
            for n in OUTS:
                assert torch.equal(got[n], want[n]), n


def test_noalloc_refuses_oversize():
    # T=1M tokens at E=1024 needs far more than 8 MiB of tables
    cfg = moe.make_config(1 << 20, 128, 1024, 8, 128, 8)
    assert moe.moe_workspace_bytes(cfg, moe.MOE_WS_PERMUTE) > (8 << 20)
    with pytest.raises(moe.MoeError) as err:
        moe.moe_permute_noalloc(cfg, *([None] * 11))
    assert err.value.status == moe.MOE_ERR_WORKSPACE


def test_noalloc_allocates_nothing_and_runs_on_a_side_stream():
    """After a first call (which looks up the array's address), a call
    changes neither the device's free memory nor torch's allocation; the
    same call enqueued on another stream gives the same outputs."""
    cfg, x, idx = _case(sweep_workload(4096, "zipf"), 2.0)
    want = _permute(cfg, x, idx, True, noalloc=False)
    b = moe.alloc_step_buffers(cfg)
    args = [cfg, x, idx, True] + [b[n] for n in OUTS]
    moe.moe_permute_noalloc(*args)
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    used0 = torch.cuda.memory_allocated()
    moe.moe_permute_noalloc(*args)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0
    assert torch.cuda.memory_allocated() == used0
    for n in OUTS:
        b[n].fill_(-7) if b[n].dtype == torch.int32 else b[n].zero_()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    moe.moe_permute_noalloc(*args, stream=side)
    side.synchronize()
    for n in OUTS:
        assert torch.equal(b[n], want[n]), n


def test_noalloc_no_tokens():
    """T = 0: the offsets come back zero and nothing is dropped."""
    cfg = moe.make_config(0, 128, 8, 2, 128, 2)
    x = torch.empty((0, 128), dtype=torch.bfloat16, device="cuda")
    idx = torch.empty((0, 2), dtype=torch.int32, device="cuda")
    b = moe.alloc_step_buffers(cfg)
    for n in ("group_offsets", "uniq_offsets", "n_dropped"):
        b[n].fill_(7)
    moe.moe_permute_noalloc(cfg, x, idx, True, *[b[n] for n in OUTS])
    torch.cuda.synchronize()
    for n in ("group_offsets", "uniq_offsets", "n_dropped"):
        assert torch.all(b[n] == 0), n
