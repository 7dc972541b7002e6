"""Expert parallelism's host side across processes on CPU (gloo, world size
2 and 3): the transport the EP layer uses (DistTransport: all-reduce of the
shard counts, all-to-all-v of row blocks) carries each rank's dispatch --
made by the oracle, since the kernels need a GPU -- to the right ranks, and
the returned partial rows add up to the oracle's EP layer output.

Every rank can compute every rank's inputs (seeded), so each checks what it
received against the sender's plan, block by block."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

E, K, H, F = 12, 3, 4, 5


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _inputs(rank, T_r):
    rng = np.random.default_rng(1000 + rank)
    x = rng.standard_normal((T_r, H))
    L = rng.standard_normal((T_r, E)) - 1.2 * np.log(np.arange(E) + 1.0)
    return x, L


def _weights():
    rng = np.random.default_rng(7)
    return (rng.standard_normal((E, H, F)), rng.standard_normal((E, H, F)),
            rng.standard_normal((E, F, H)))


def _worker(rank, world, port, Ts, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from mixture_experts_token_gb300.ep import DistTransport
        from oracle import moe_ref as ref
        tr = DistTransport()
        assert tr.n == world and tr.ranks == [rank]
        N, Ed = world, E // world
        W = _weights()
        weights = ref.dense_weights(*W)
        ins = [_inputs(r, Ts[r]) for r in range(N)]
        routes = [ref.route(L, K)[:2] for _, L in ins]
        plans = [ref.ep_dispatch(i, w, E, N) for i, w in routes]
        # the global check: this rank's shard counts, summed over ranks
        local = ref.shard_counts(ref.expert_counts(routes[rank][0], E), N)
        (tot,) = tr.all_reduce_sum([torch.tensor(local, dtype=torch.int32)])
        want = sum(ref.shard_counts(ref.expert_counts(i, E), N)
                   for i, _ in routes)
        assert np.array_equal(tot.numpy(), want)
        # exchange 1: the dedup'd rows and their slots, per destination
        p = plans[rank]
        x = ins[rank][0]
        uo = [int(v) for v in p.uniq_offsets]
        xs = [torch.tensor(x[p.uniq_tokens[uo[d]:uo[d + 1]]],
                           dtype=torch.float32) for d in range(N)]
        si = [torch.tensor(p.send_idx[uo[d]:uo[d + 1]], dtype=torch.int32)
              for d in range(N)]
        sw = [torch.tensor(p.send_w[uo[d]:uo[d + 1]], dtype=torch.float32)
              for d in range(N)]
        (rx,) = tr.all_to_all([xs])
        (ri,) = tr.all_to_all([si])
        (rw,) = tr.all_to_all([sw])
        for q in range(N):   # what source q meant for this rank
            pq = plans[q]
            a, z = int(pq.uniq_offsets[rank]), int(pq.uniq_offsets[rank + 1])
            assert rx[q].shape == (z - a, H)
            assert np.allclose(rx[q].numpy(),
                               ins[q][0][pq.uniq_tokens[a:z]], atol=1e-6)
            assert np.array_equal(ri[q].numpy(), pq.send_idx[a:z])
            assert np.allclose(rw[q].numpy(), pq.send_w[a:z], atol=1e-7)
        # the local experts over the received rows; exchange 2 returns the
        # partial rows to their sources, which add them
        recv_x = torch.cat(rx).double().numpy()
        recv_i = torch.cat(ri).numpy()
        recv_w = torch.cat(rw).double().numpy()
        back = ref.ep_expert_pass(recv_x, recv_i, recv_w,
                                  lambda e: weights(rank * Ed + e))
        sizes = [t.shape[0] for t in rx]
        blocks = list(torch.split(torch.tensor(back, dtype=torch.float64),
                                  sizes))
        (ret,) = tr.all_to_all([blocks])
        y = np.zeros((Ts[rank], H))
        for d in range(N):
            for u, t in enumerate(p.uniq_tokens[uo[d]:uo[d + 1]]):
                y[int(t)] += ret[d][u].numpy()
        cfg = ref.MoEConfig(sum(Ts), H, E, K, F, N, -1.0)
        ys, over, n = ref.ep_layer(cfg, N, [a for a, _ in ins],
                                   [b for _, b in ins], weights)
        assert not over and n == 1
        out[rank] = float(np.max(np.abs(y - ys[rank]))) if Ts[rank] else 0.0
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("Ts", [[37, 21], [16, 0, 25]],
                         ids=["world2", "world3_empty_rank"])
def test_ep_exchange_over_gloo(Ts):
    world = len(Ts)
    port = _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(world, port, Ts, out), nprocs=world, join=True)
    for r in range(world):
        assert out[r] < 1e-5, (r, out[r])
