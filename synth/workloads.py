"""Workload shapes and seeded generators.

Shapes follow the layers the MaxText pages train or benchmark: a
DeepSeek-V3-shaped layer (the recipe in "MoE ring-of-experts: TC Pallas ring
all-gather ..." (MaxText pull request 4969), section "Repro") and a
Llama4-Maverick-shaped layer at EP16 with ragged_buffer_factor 2.0 ("Support
moe_dropless_fallback=layer on the ragged all-to-all MoE path" (MaxText pull
request 5920), section "End-to-end").  Both pages run on synthetic data;
these generators stand in for it.

Routing recipes.  The router logits are x @ Wr + offset (the router's
product is the first step of the layer; the oracle and the library compute
it, this module only draws x, Wr and the offset):

* ``router``: x, Wr ~ N(0, 1)/sqrt(H) and no offset (the tiny layer).
* ``zipf``: Wr ~ N(0, 0.02) and offset_te = -s*ln(e+1) + G_te with G iid
  Gumbel(0, 1).  Without the x @ Wr term the Gumbel-max property would make
  the top-1 expert exactly Zipf(s)-distributed and the top-k Zipf-weighted
  sampling without replacement; the x @ Wr term (an independent Gaussian
  per token and expert, std 0.02*sqrt(H)) adds noise that flattens the law
  somewhat.  (The page on dynamic redundancy adds Zipf-distributed
  synthetic data; here the Zipf law is put on expert popularity, the
  quantity the overflow check sees.)  Hot experts have low indices, so they
  share shard 0.
* ``uniform``: Wr ~ N(0, 0.02), offset = G (uniform random routing, like
  use_random_routing).
* ``adversarial``: Wr ~ N(0, 0.02), offset = 30*[e < E/S] + G: every top-k
  pick lands in shard 0's experts.

Seeds: one child seed per tensor from ``numpy.random.SeedSequence(seed)``,
local generators only (no global random state).
"""
from __future__ import annotations

from dataclasses import dataclass, replace
from typing import Optional

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    H: int
    E: int
    k: int
    F: int
    S: int
    factor: float
    dtype: str            # "f32" or "bf16"
    routing: str          # router | zipf | uniform | adversarial
    zipf_s: float = 0.0
    n_chunks: int = 0     # 0: derived from the capacity
    renorm: bool = False
    seed: int = 0
    x_scale: float = 1.0  # std of x
    w_std: float = 0.02   # std of the expert weights
    redundant_slots: int = 0  # duplicate-expert slots per shard (0: off)

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS = {
    # fp32 tiny layer; x and Wr are N(0,1)/sqrt(H); experts N(0, 0.02)
    "tiny": Workload("tiny", T=256, H=64, E=8, k=2, F=128, S=2, factor=2.0,
                     dtype="f32", routing="router", x_scale=1.0 / 8.0),
    # small bf16 layer, Zipf s=1.0 expert popularity (factor unstated: 2.0)
    "small": Workload("small", T=4096, H=1024, E=16, k=2, F=2048, S=4,
                      factor=2.0, dtype="bf16", routing="zipf", zipf_s=1.0),
    # DeepSeek-V3-shaped layer, Zipf s=1.2 (overflows -> chunked fallback)
    "dsv3": Workload("dsv3", T=8192, H=7168, E=256, k=8, F=2048, S=8,
                     factor=2.0, dtype="bf16", routing="zipf", zipf_s=1.2),
    # Llama4-Maverick-shaped layer, uniform routing (no overflow)
    "l4mav": Workload("l4mav", T=8192, H=5120, E=128, k=1, F=8192, S=16,
                      factor=2.0, dtype="bf16", routing="uniform"),
}

SWEEP_TOKENS = (1024, 4096, 16384, 65536)
SWEEP_ROUTINGS = ("uniform", "zipf", "adversarial")


def sweep_workload(T: int, routing: str) -> Workload:
    """Routing/permute/dedup bandwidth sweep: H=7168 bf16, E=256, k=8, 8
    shards, fallback with 8 chunks.  No expert FFN (F=0)."""
    return Workload(f"sweep_T{T}_{routing}", T=T, H=7168, E=256, k=8, F=0,
                    S=8, factor=2.0, dtype="bf16", routing=routing,
                    zipf_s=1.2 if routing == "zipf" else 0.0, n_chunks=8)


def seeds_for(seed: int, n: int = 8):
    """Independent child seeds (ints) for the tensors of one workload:
    0 x, 1 router weight, 2 logit noise, 3 w_gate, 4 w_up, 5 w_down,
    6 the output gradient dy of the backward pass."""
    ss = np.random.SeedSequence(seed).spawn(n)
    return [int(s.generate_state(1, dtype=np.uint64)[0] & 0x7FFFFFFFFFFFFFFF)
            for s in ss]


def _torch_gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def make_x(wl: Workload, device="cpu", T: Optional[int] = None) -> torch.Tensor:
    """Token activations x [T, H] in the workload dtype."""
    T = wl.T if T is None else T
    sd = seeds_for(wl.seed)[0]
    g = _torch_gen(device, sd)
    x = torch.randn(T, wl.H, generator=g, device=device, dtype=torch.float32)
    if wl.x_scale != 1.0:
        x = x * wl.x_scale
    return x.to(wl.torch_dtype)


def make_router_weight(wl: Workload, device="cpu") -> torch.Tensor:
    """Router weight Wr [H, E] in the workload dtype, drawn on the host
    (numpy PCG64) so that routing is the same on every machine."""
    rng = np.random.default_rng(seeds_for(wl.seed)[1])
    w = rng.standard_normal((wl.H, wl.E))
    w *= (1.0 / np.sqrt(wl.H)) if wl.routing == "router" else wl.w_std
    return torch.from_numpy(w.astype(np.float32)).to(wl.torch_dtype).to(device)


def make_logit_offset(wl: Workload, T: Optional[int] = None):
    """Per-(token, expert) offset [T, E] float32 added to x @ Wr, or None
    (``router`` routing)."""
    T = wl.T if T is None else T
    E = wl.E
    if wl.routing == "router":
        return None
    rng = np.random.default_rng(seeds_for(wl.seed)[2])
    g = rng.gumbel(size=(T, E))
    if wl.routing == "zipf":
        bias = -wl.zipf_s * np.log(np.arange(E, dtype=np.float64) + 1.0)
        return (g + bias[None, :]).astype(np.float32)
    if wl.routing == "uniform":
        return g.astype(np.float32)
    if wl.routing == "adversarial":
        bias = np.zeros(E)
        bias[: E // wl.S] = 30.0
        return (g + bias[None, :]).astype(np.float32)
    raise ValueError(f"unknown routing {wl.routing}")


def make_weights(wl: Workload, device="cpu"):
    """Expert weights (w_gate [E,H,F], w_up [E,H,F], w_down [E,F,H]),
    N(0, w_std), drawn one expert at a time so no large fp32 temporary is
    needed."""
    seeds = seeds_for(wl.seed)
    out = []
    for which, shape in ((3, (wl.H, wl.F)), (4, (wl.H, wl.F)),
                         (5, (wl.F, wl.H))):
        g = _torch_gen(device, seeds[which])
        w = torch.empty((wl.E,) + shape, device=device, dtype=wl.torch_dtype)
        for e in range(wl.E):
            blk = torch.randn(shape, generator=g, device=device,
                              dtype=torch.float32)
            w[e].copy_(blk.mul_(wl.w_std))
        out.append(w)
    return tuple(out)


def make_dy(wl: Workload, device="cpu", T: Optional[int] = None) -> torch.Tensor:
    """Gradient of the loss with respect to the layer output, dy [T, H]
    ~ N(0, 1) in the workload dtype (the backward pass's input)."""
    T = wl.T if T is None else T
    g = _torch_gen(device, seeds_for(wl.seed)[6])
    dy = torch.randn(T, wl.H, generator=g, device=device, dtype=torch.float32)
    return dy.to(wl.torch_dtype)
