"""Expert parallelism's host side across processes on CPU (gloo, world size
2 and 3): the transport the EP layer uses (DistTransport: all-reduce of the
shard counts, all-to-all-v of row blocks) carries each rank's dispatch --
made by the oracle, since the kernels need a GPU -- to the right ranks, and
the returned partial rows add up to the oracle's EP layer output.

Every rank can compute every rank's inputs (seeded), so each checks what it
received against the sender's plan, block by block.  The ring of experts
runs its all-gathers and reduce-scatters (forward and backward) through the
same transport, each rank's share of the work from the oracle, against the
oracle's ring layer and its backward."""
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


def _ring_worker(rank, world, port, Ts, out):
    """The ring of experts over gloo: the all-gathers (tokens, routing, and
    in the backward the output cotangent) and the reduce-scatters (partial
    outputs, partial dx, the picks' weight gradients) through
    DistTransport, each rank's local share from the oracle."""
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from mixture_experts_token_gb300.ep import DistTransport
        from oracle import moe_ref as ref
        tr = DistTransport()
        N, Ed = world, E // world
        weights = ref.dense_weights(*_weights())
        ins = [_inputs(r, Ts[r]) for r in range(N)]
        dys = [np.random.default_rng(500 + r).standard_normal((Ts[r], H))
               for r in range(N)]
        x, L = ins[rank]
        idx, w = ref.route(L, K)[:2]
        f64 = torch.float64

        def gather(a, dtype):
            (got,) = tr.all_to_all([[torch.tensor(a, dtype=dtype)] * N])
            return torch.cat(got).numpy()

        x_all = gather(x, f64)
        idx_all = gather(idx, torch.int32)
        w_all = gather(w, f64)
        assert np.array_equal(x_all, np.concatenate([a for a, _ in ins]))
        sizes = list(Ts)
        local = np.where(idx_all // Ed == rank, idx_all - rank * Ed, -1)
        part = ref.ep_expert_pass(x_all, local,
                                  np.where(local >= 0, w_all, 0.0),
                                  lambda e: weights(rank * Ed + e))
        (ret,) = tr.all_to_all([list(torch.split(torch.tensor(part),
                                                 sizes))])
        y = sum(b.numpy() for b in ret) if Ts[rank] else np.zeros((0, H))
        cfg = ref.MoEConfig(sum(Ts), H, E, K, F, N, -1.0)
        ys = ref.ring_layer(cfg, N, [a for a, _ in ins],
                            [b for _, b in ins], weights)
        err = float(np.max(np.abs(y - ys[rank]))) if Ts[rank] else 0.0
        # backward: cotangent all-gather, this rank's share, reduce-scatters
        dy_all = gather(dys[rank], f64)
        dpart, dtw, dW = ref.ring_rank_backward(cfg, N, rank, x_all, idx_all,
                                                w_all, dy_all, weights)
        (rdx,) = tr.all_to_all([list(torch.split(torch.tensor(dpart),
                                                 sizes))])
        (rdw,) = tr.all_to_all([list(torch.split(torch.tensor(dtw),
                                                 sizes))])
        wdx, wdl, wdW = ref.ring_layer_backward(
            cfg, N, [a for a, _ in ins], [b for _, b in ins], weights, dys)
        if Ts[rank]:
            dx = sum(b.numpy() for b in rdx)
            dl = ref.route_backward(L, idx, sum(b.numpy() for b in rdw),
                                    False)
            err = max(err, float(np.max(np.abs(dx - wdx[rank]))),
                      float(np.max(np.abs(dl - wdl[rank]))))
        for e in range(rank * Ed, (rank + 1) * Ed):
            got = dW.get(e, (np.zeros((H, F)), np.zeros((H, F)),
                             np.zeros((F, H))))
            err = max([err] + [float(np.max(np.abs(g - wdW[i][e])))
                               for i, g in enumerate(got)])
        out[rank] = err
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("Ts", [[29, 17], [11, 0, 20]],
                         ids=["world2", "world3_empty_rank"])
def test_ring_exchange_over_gloo(Ts):
    world = len(Ts)
    port = _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_ring_worker, args=(world, port, Ts, out), nprocs=world,
             join=True)
    for r in range(world):
        assert out[r] < 1e-6, (r, out[r])


def _ep_bwd_worker(rank, world, port, Ts, factor, out):
    """The EP layer's backward over gloo: the global check, then per pass
    the dispatch's rows out with the cotangent along them, the token
    gradients and slot weight gradients back; each rank's receiving share
    from the oracle; against the oracle's EP backward."""
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from mixture_experts_token_gb300.ep import DistTransport
        from oracle import moe_ref as ref
        tr = DistTransport()
        N, Ed = world, E // world
        kk = min(K, Ed)
        weights = ref.dense_weights(*_weights())
        ins = [_inputs(r, Ts[r]) for r in range(N)]
        dys = [np.random.default_rng(600 + r).standard_normal((Ts[r], H))
               for r in range(N)]
        x, L = ins[rank]
        idx, w = ref.route(L, K)[:2]
        cfg = ref.MoEConfig(sum(Ts), H, E, K, F, N, factor)
        local = ref.shard_counts(ref.expert_counts(idx, E), N)
        (tot,) = tr.all_reduce_sum([torch.tensor(local, dtype=torch.int32)])
        C = ref.capacity(cfg.T, K, N, factor)
        over = ref.overflow_flag(tot.numpy(), C)
        n = len(ref.chunk_plan(cfg.T, K, E, N, C)) if over else 1
        dx = np.zeros((Ts[rank], H))
        dtw = np.zeros((Ts[rank], K))
        dW = {}
        for c in range(n):
            t0, t1 = ref.ep_chunk_bounds(Ts[rank], n, c)
            p = ref.ep_dispatch(idx[t0:t1], w[t0:t1], E, N)
            uo = [int(v) for v in p.uniq_offsets]

            def blocks(a, dtype):
                return [torch.tensor(a[uo[d]:uo[d + 1]], dtype=dtype)
                        for d in range(N)]
            tok = t0 + p.uniq_tokens
            (rx,) = tr.all_to_all([blocks(x[tok], torch.float64)])
            (rdy,) = tr.all_to_all([blocks(dys[rank][tok], torch.float64)])
            (ri,) = tr.all_to_all([blocks(p.send_idx, torch.int32)])
            (rw,) = tr.all_to_all([blocks(p.send_w, torch.float64)])
            cat = lambda bl, shp: (torch.cat(bl).numpy() if bl else
                                   np.zeros(shp))
            dx_r, dw_r, dWl = ref.ep_expert_pass_backward(
                cat(rx, (0, H)), cat(ri, (0, kk)).reshape(-1, kk),
                cat(rw, (0, kk)).reshape(-1, kk), cat(rdy, (0, H)),
                lambda e: weights(rank * Ed + e))
            for e, gs in dWl.items():
                dW[e] = gs if e not in dW else tuple(
                    a + b for a, b in zip(dW[e], gs))
            sizes = [t.shape[0] for t in rx]
            (bdx,) = tr.all_to_all([list(torch.split(torch.tensor(dx_r),
                                                     sizes))])
            (bdw,) = tr.all_to_all([list(torch.split(torch.tensor(dw_r),
                                                     sizes))])
            for d in range(N):
                for u, t in enumerate(p.uniq_tokens[uo[d]:uo[d + 1]]):
                    t = t0 + int(t)
                    dx[t] += bdx[d][u].numpy()
                    own = [j for j in range(K) if int(idx[t, j]) // Ed == d]
                    for s, j in enumerate(own):
                        dtw[t, j] = float(bdw[d][u, s])
        wdx, wdl, wdW = ref.ep_layer_backward(
            cfg, N, [a for a, _ in ins], [b for _, b in ins], weights, dys)
        err = 0.0
        if Ts[rank]:
            dl = ref.route_backward(L, idx, dtw, False)
            err = max(float(np.max(np.abs(dx - wdx[rank]))),
                      float(np.max(np.abs(dl - wdl[rank]))))
        for e in range(Ed):
            got = dW.get(e, (np.zeros((H, F)), np.zeros((H, F)),
                             np.zeros((F, H))))
            err = max([err] + [float(np.max(np.abs(g - wdW[i][rank * Ed + e])))
                               for i, g in enumerate(got)])
        out[rank] = (err, int(over), n)
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("Ts,factor", [([37, 21], 2.0), ([16, 0, 25], 2.0),
                                       ([40, 33], 0.6)],
                         ids=["world2", "world3_empty_rank",
                              "world2_fallback"])
def test_ep_backward_exchange_over_gloo(Ts, factor):
    world = len(Ts)
    port = _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_ep_bwd_worker, args=(world, port, Ts, factor, out),
             nprocs=world, join=True)
    for r in range(world):
        assert out[r][0] < 1e-6, (r, out[r])
    if factor < 1.0:
        assert out[0][1] == 1 and out[0][2] > 1   # the fallback ran
