"""Expert parallelism across ranks: the layer's passes with the two
exchanges of the ragged all-to-all path, and the ring-of-experts variant.

"Support moe_dropless_fallback=layer on the ragged all-to-all MoE path"
(MaxText pull request 5920), sections Why, How and Tests: every rank sends
its tokens' rows to the ranks that own their experts; the overflow check is
global, so every rank takes the same branch (the capped pass, or the
chunked dropless fallback).  "Moe dynamic redundancy" (pull request 4760),
review of ra2a_dedup_and_route: a token is sent to a destination once and
expanded there.  "MoE ring-of-experts ..." (pull request 4969), section
What: all-gather the tokens, compute the local experts, reduce-scatter the
combine.

Every step on the data runs in the library's kernels (include/moe.h); this
module sequences them and moves buffers between ranks through a transport:

* ``DistTransport``: one rank of a torch.distributed process group (NCCL on
  GPUs, gloo on CPU): an all-reduce of the shard counts and all-to-all-v
  exchanges of rows.
* ``LoopbackTransport``: N logical ranks held by one process on one device;
  an exchange hands each receiver the senders' buffers (device copies).  No
  kernel of one rank waits on another's: the ranks run phase by phase.

Ranks are the shards (cfg.S = ranks): rank d owns experts [d*E/S,
(d+1)*E/S) and holds their weights.  ``EPLayer`` follows the pages'
fallback=layer; since the capped pass runs only when no shard overflows, no
pass drops a row, and the result equals the single-device layer on the
ranks' batches together.  ``RingLayer`` is dropless.
"""
from __future__ import annotations

import torch

from . import (alloc_step_buffers, make_config, moe_check_overflow,
               moe_combine, moe_combine_backward, moe_ep_check,
               moe_ep_delocalize, moe_ep_dispatch_pack, moe_ep_localize,
               moe_ep_return_map, moe_ep_sum_partials, moe_gmm_down,
               moe_gmm_gate_up, moe_gmm_swiglu_backward, moe_gmm_swiglu_saved,
               moe_num_chunks, moe_permute, moe_permute_backward,
               moe_permute_scatter, moe_permute_tables, moe_route,
               moe_route_backward, moe_workspace_bytes, MOE_WS_GMM_BACKWARD,
               MOE_WS_PERMUTE)


# ------------------------------------------------------------ transports --
class LoopbackTransport:
    """All ranks in this process: the lists below hold one entry per rank,
    in rank order."""

    def __init__(self, n_ranks: int):
        self.n = n_ranks
        self.ranks = list(range(n_ranks))

    def all_reduce_sum(self, tensors):
        total = tensors[0].clone()
        for t in tensors[1:]:
            total += t
        return [total.clone() for _ in tensors]

    def all_to_all(self, sends):
        """sends[r][d]: rank r's rows for rank d -> recv[d][r]."""
        return [[sends[r][d] for r in range(self.n)] for d in range(self.n)]


class DistTransport:
    """This process is one rank of the default torch.distributed group."""

    def __init__(self, group=None):
        import torch.distributed as dist
        self.dist = dist
        self.group = group
        self.n = dist.get_world_size(group)
        self.ranks = [dist.get_rank(group)]

    def all_reduce_sum(self, tensors):
        (t,) = tensors
        out = t.clone()
        self.dist.all_reduce(out, group=self.group)
        return [out]

    def all_to_all(self, sends):
        """all-to-all-v of row blocks: first the row counts, then the rows
        (one all_to_all_single over the concatenated blocks)."""
        (blocks,) = sends
        dev = blocks[0].device
        rows = torch.tensor([b.shape[0] for b in blocks], dtype=torch.int64,
                            device=dev)
        got = torch.empty_like(rows)
        self.dist.all_to_all_single(got, rows, group=self.group)
        in_splits = rows.tolist()
        out_splits = got.tolist()
        tail = tuple(blocks[0].shape[1:])
        send = torch.cat([b.contiguous() for b in blocks])
        recv = torch.empty((sum(out_splits),) + tail, dtype=send.dtype,
                           device=dev)
        self.dist.all_to_all_single(recv, send, out_splits, in_splits,
                                    group=self.group)
        return [list(torch.split(recv, out_splits))]


# ------------------------------------------------------------- helpers ----
def _cfg(base, **kw):
    return base.with_(**kw)


def chunk_bounds(T_r: int, n: int, c: int):
    """Tokens [t0, t1) of rank-local chunk c of n (chunks of ceil(T_r/n))."""
    size = -(-T_r // n) if n > 0 else 0
    t0 = min(T_r, c * size)
    return t0, min(T_r, t0 + size)


class _Rank:
    """One rank's inputs, routing and output."""

    def __init__(self, rank, x, logits, cfg, dev):
        self.rank = rank
        self.x = x
        self.T = x.shape[0]
        self.cfg = _cfg(cfg, T=self.T)
        k, E, S = cfg.k, cfg.E, cfg.S
        i32 = dict(dtype=torch.int32, device=dev)
        self.idx = torch.empty((self.T, k), **i32)
        self.w = torch.empty((self.T, k), dtype=torch.float32, device=dev)
        if self.T:
            moe_route(self.cfg, logits, self.idx, self.w)
        self.counts = torch.empty(E, **i32)
        self.offsets = torch.empty(E + 1, **i32)
        self.shard = torch.zeros(S, **i32)
        self.flag = torch.zeros(1, **i32)
        self.req = torch.zeros(1, dtype=torch.float32, device=dev)
        self.cap = torch.zeros(1, **i32)
        self.y = torch.zeros((self.T, cfg.H), dtype=x.dtype, device=dev)


class EPLayer:
    """The layer with moe_dropless_fallback=layer over expert-parallel ranks.

    cfg: the layer's configuration with T = the tokens of all ranks together
    and S = the number of ranks.  weights(rank) -> (w_gate, w_up, w_down) of
    the rank's E/S experts ([E/S, H, F], [E/S, H, F], [E/S, F, H])."""

    def __init__(self, cfg, transport, weights):
        if cfg.E % cfg.S:
            raise ValueError("E must be a multiple of the ranks")
        if transport.n != cfg.S:
            raise ValueError("cfg.S must equal the number of ranks")
        self.cfg = cfg
        self.tr = transport
        self.weights = weights
        self.info = {}

    def forward(self, xs, logits):
        """xs[i], logits[i]: the inputs of the transport's i-th local rank;
        returns their outputs."""
        cfg, tr = self.cfg, self.tr
        dev = xs[0].device
        ranks = [_Rank(r, x, L, cfg, dev)
                 for r, x, L in zip(tr.ranks, xs, logits)]
        n = self._check(ranks)
        for c in range(n):
            self._pass(ranks, c, n)
        return [rk.y for rk in ranks]

    def _check(self, ranks):
        """The global check; returns the pass count."""
        cfg, tr = self.cfg, self.tr
        for rk in ranks:
            if rk.T:
                moe_check_overflow(rk.cfg, rk.idx, rk.counts, rk.offsets,
                                   rk.shard, rk.flag, rk.req, rk.cap)
        sums = tr.all_reduce_sum([rk.shard for rk in ranks])
        for rk, s in zip(ranks, sums):
            moe_ep_check(cfg, s, rk.flag, rk.req, rk.cap)
        over = int(ranks[0].flag.item())
        self.info = {"overflow": over,
                     "n_chunks": moe_num_chunks(cfg) if over else 1,
                     "required_factor": float(ranks[0].req.item())}
        return self.info["n_chunks"]

    def _send(self, ranks, c, n, dys=None):
        """Source side of pass c of n: dedup sets per destination and the
        send rows (x, and with dys the output cotangent along the same
        rows), split by destination."""
        cfg = self.cfg
        S, k, H = cfg.S, cfg.k, cfg.H
        kk = min(k, cfg.E // S)
        dev = ranks[0].x.device
        out = {"x": [], "i": [], "w": [], "dy": [], "state": []}
        for j, rk in enumerate(ranks):
            t0, t1 = chunk_bounds(rk.T, n, c)
            Tc = t1 - t0
            sc = _cfg(cfg, T=Tc, ragged_buffer_factor=-1.0, n_chunks=0,
                      redundant_slots=0)
            b = alloc_step_buffers(sc, dev)
            rows = Tc * min(k, S)
            x_send = torch.empty((rows, H), dtype=rk.x.dtype, device=dev)
            s_idx = torch.empty((rows, kk), dtype=torch.int32, device=dev)
            s_w = torch.empty((rows, kk), dtype=torch.float32, device=dev)
            dy_send = (torch.empty_like(x_send) if dys is not None
                       else None)
            if Tc:
                moe_permute_tables(sc, rk.idx[t0:t1], False, b["row_of"],
                                   b["sorted_token"], b["group_offsets"],
                                   b["uniq_offsets"], b["n_dropped"],
                                   b["permute_ws"])
                moe_permute_scatter(sc, None, b["row_of"], b["uniq_offsets"],
                                    None, b["uniq_tokens"], b["expand_idx"],
                                    b["permute_ws"])
                moe_ep_dispatch_pack(sc, rk.x[t0:t1], rk.idx[t0:t1],
                                     rk.w[t0:t1], b["uniq_offsets"],
                                     b["uniq_tokens"], x_send, s_idx, s_w)
                if dys is not None:
                    # the same rows and slots, carrying dy instead of x
                    i2 = torch.empty_like(s_idx)
                    w2 = torch.empty_like(s_w)
                    moe_ep_dispatch_pack(sc, dys[j][t0:t1], rk.idx[t0:t1],
                                         rk.w[t0:t1], b["uniq_offsets"],
                                         b["uniq_tokens"], dy_send, i2, w2)
                uo = b["uniq_offsets"].cpu().tolist()
            else:
                uo = [0] * (S + 1)
            out["x"].append([x_send[uo[d]:uo[d + 1]] for d in range(S)])
            out["i"].append([s_idx[uo[d]:uo[d + 1]] for d in range(S)])
            out["w"].append([s_w[uo[d]:uo[d + 1]] for d in range(S)])
            if dys is not None:
                out["dy"].append([dy_send[uo[d]:uo[d + 1]]
                                  for d in range(S)])
            out["state"].append((t0, t1, sc, b))
        return out

    def _recv_sorted(self, rk, rx, ri):
        """Receiving side: the received rows sorted by local expert."""
        cfg = self.cfg
        El = cfg.E // cfg.S
        n_recv = rx.shape[0]
        rc = _cfg(cfg, T=n_recv, E=El, k=min(cfg.k, El), S=1,
                  ragged_buffer_factor=-1.0, n_chunks=0, redundant_slots=0)
        rb = alloc_step_buffers(rc, rx.device)
        moe_permute(rc, rx, ri, False, rb["x_sorted"], rb["row_of"],
                    rb["sorted_token"], rb["group_offsets"],
                    rb["uniq_offsets"], rb["uniq_tokens"], rb["expand_idx"],
                    rb["n_dropped"], rb["permute_ws"])
        return rc, rb

    @staticmethod
    def _return_map(sc, b, T):
        row_of_ret = torch.empty((T, sc.S), dtype=torch.int32,
                                 device=b["uniq_offsets"].device)
        moe_ep_return_map(sc, b["uniq_offsets"], b["uniq_tokens"],
                          row_of_ret)
        return row_of_ret

    def _pass(self, ranks, c, n):
        cfg, tr = self.cfg, self.tr
        S, H = cfg.S, cfg.H
        dev = ranks[0].x.device
        snd = self._send(ranks, c, n)
        recv_x = tr.all_to_all(snd["x"])
        recv_i = tr.all_to_all(snd["i"])
        recv_w = tr.all_to_all(snd["w"])
        # receiving side: the local experts over the received rows
        backs = []
        for j, rk in enumerate(ranks):
            sizes = [blk.shape[0] for blk in recv_x[j]]
            n_recv = sum(sizes)
            part = torch.empty((n_recv, H), dtype=rk.x.dtype, device=dev)
            if n_recv:
                rc, rb = self._recv_sorted(rk, torch.cat(recv_x[j]),
                                           torch.cat(recv_i[j]))
                wg, wu, wd = self.weights(rk.rank)
                moe_gmm_gate_up(rc, rb["x_sorted"], rb["group_offsets"], wg,
                                wu, rb["h"], rb["status"])
                moe_gmm_down(rc, rb["h"], rb["group_offsets"], wd,
                             rb["y_sorted"], rb["status"])
                moe_combine(rc, rb["y_sorted"], rb["row_of"],
                            torch.cat(recv_w[j]), part)
            backs.append(list(torch.split(part, sizes)))
        ret = tr.all_to_all(backs)
        # source side: add the rows the destinations returned
        for rk, blocks, (t0, t1, sc, b) in zip(ranks, ret, snd["state"]):
            if t1 == t0:
                continue
            moe_permute_backward(_cfg(sc, k=S), torch.cat(blocks),
                                 self._return_map(sc, b, t1 - t0),
                                 rk.y[t0:t1])

    def backward(self, xs, logits, dys):
        """Gradients of sum_r <dys[r], forward(xs, logits)[r]> (the forward
        recomputed pass by pass): per rank (dx [T_r, H] layer dtype,
        dlogits [T_r, E] float32, (dWg, dWu, dWd) float32 of its own
        experts, summed over the passes).  Each exchange of the forward runs
        transposed: the cotangent goes out along the dispatch's dedup'd rows,
        the token gradients and the slots' weight gradients come back."""
        cfg, tr = self.cfg, self.tr
        S, H, E, F, k = cfg.S, cfg.H, cfg.E, cfg.F, cfg.k
        El = E // S
        kk = min(k, El)
        dev = xs[0].device
        f32 = dict(dtype=torch.float32, device=dev)
        ranks = [_Rank(r, x, L, cfg, dev)
                 for r, x, L in zip(tr.ranks, xs, logits)]
        n = self._check(ranks)
        dWs = [(torch.zeros((El, H, F), **f32), torch.zeros((El, H, F), **f32),
                torch.zeros((El, F, H), **f32)) for _ in ranks]
        dxs = [torch.zeros((rk.T, H), dtype=rk.x.dtype, device=dev)
               for rk in ranks]
        dtws = [torch.zeros((rk.T, k), **f32) for rk in ranks]
        for c in range(n):
            snd = self._send(ranks, c, n, dys)
            recv_x = tr.all_to_all(snd["x"])
            recv_i = tr.all_to_all(snd["i"])
            recv_w = tr.all_to_all(snd["w"])
            recv_dy = tr.all_to_all(snd["dy"])
            dx_back, dw_back = [], []
            for j, rk in enumerate(ranks):
                sizes = [blk.shape[0] for blk in recv_x[j]]
                n_recv = sum(sizes)
                dxr = torch.empty((n_recv, H), dtype=rk.x.dtype, device=dev)
                dwr = torch.zeros((n_recv, kk), **f32)
                if n_recv:
                    rc, rb = self._recv_sorted(rk, torch.cat(recv_x[j]),
                                               torch.cat(recv_i[j]))
                    R = rc.T * rc.k
                    wg, wu, wd = self.weights(rk.rank)
                    g = torch.empty((R, F), dtype=rk.x.dtype, device=dev)
                    u = torch.empty_like(g)
                    moe_gmm_swiglu_saved(rc, rb["x_sorted"],
                                         rb["group_offsets"], wg, wu, wd, g,
                                         u, rb["h"], rb["y_sorted"],
                                         rb["status"])
                    dy_sorted = torch.empty((R, H), dtype=rk.x.dtype,
                                            device=dev)
                    moe_combine_backward(rc, torch.cat(recv_dy[j]),
                                         rb["y_sorted"], rb["row_of"],
                                         torch.cat(recv_w[j]), dy_sorted, dwr)
                    dx_sorted = torch.empty_like(dy_sorted)
                    ws = torch.empty(max(moe_workspace_bytes(
                        rc, MOE_WS_GMM_BACKWARD), 256), dtype=torch.uint8,
                        device=dev)
                    dwg, dwu, dwd = dWs[j]
                    moe_gmm_swiglu_backward(rc, rb["x_sorted"],
                                            rb["group_offsets"], wg, wu, wd,
                                            g, u, rb["h"], dy_sorted,
                                            dx_sorted, dwg, dwu, dwd, 1, ws,
                                            rb["status"])
                    moe_permute_backward(rc, dx_sorted, rb["row_of"], dxr)
                dx_back.append(list(torch.split(dxr, sizes)))
                dw_back.append(list(torch.split(dwr, sizes)))
            rdx = tr.all_to_all(dx_back)
            rdw = tr.all_to_all(dw_back)
            # source side: the token gradients added over the destinations,
            # each slot's weight gradient back at its pick
            for j, (rk, (t0, t1, sc, b)) in enumerate(zip(ranks,
                                                          snd["state"])):
                if t1 == t0:
                    continue
                row_of_ret = self._return_map(sc, b, t1 - t0)
                moe_permute_backward(_cfg(sc, k=S), torch.cat(rdx[j]),
                                     row_of_ret, dxs[j][t0:t1])
                dw_rows = torch.cat(rdw[j])
                for d in range(S):
                    moe_ep_delocalize(sc, rk.idx[t0:t1], d * El, El, dw_rows,
                                      dtws[j][t0:t1],
                                      row_of=row_of_ret.data_ptr() + 4 * d,
                                      row_stride=S)
        dls = []
        for rk, L, dtw in zip(ranks, logits, dtws):
            dl = torch.zeros((rk.T, E), **f32)
            if rk.T:
                moe_route_backward(rk.cfg, L, rk.idx, dtw, dl)
            dls.append(dl)
        return dxs, dls, dWs


class RingLayer:
    """The ring-of-experts variant (dropless): every rank sees all tokens,
    computes its own experts' weighted outputs, and each token's owner adds
    the ranks' partial outputs.

    backward() differentiates it ("MoE ring-of-experts ...", pull request
    4969, section What): the output cotangents are all-gathered (the
    transpose of the combine's reduce-scatter), each rank runs the backward
    of its experts' pass over all tokens, and the owners add the ranks'
    partial token gradients (the transpose of the tokens' all-gather) and
    collect each pick's combine-weight gradient from the rank that owns its
    expert.  With save_x_sorted (the pages' moe_x_sorted=device) the forward
    keeps each rank's gathered, expert-sorted rows and routing, and the
    backward reuses them instead of gathering and sorting again."""

    def __init__(self, cfg, transport, weights, save_x_sorted=False):
        if cfg.E % cfg.S or transport.n != cfg.S:
            raise ValueError("cfg.S must equal the ranks and divide E")
        self.cfg = cfg
        self.tr = transport
        self.weights = weights
        self.save_x_sorted = save_x_sorted
        self.saved = None

    def _gather(self, ranks):
        """All-gather of the tokens and their routing; each rank then keeps
        its own picks and sorts the rows by its experts."""
        cfg, tr = self.cfg, self.tr
        S, El = cfg.S, cfg.E // cfg.S
        kk = min(cfg.k, El)
        gx = tr.all_to_all([[rk.x] * S for rk in ranks])
        gi = tr.all_to_all([[rk.idx] * S for rk in ranks])
        gw = tr.all_to_all([[rk.w] * S for rk in ranks])
        states = []
        for j, rk in enumerate(ranks):
            dev = rk.x.device
            sizes = [blk.shape[0] for blk in gx[j]]
            st = {"sizes": sizes, "T_all": sum(sizes)}
            states.append(st)
            if not st["T_all"]:
                continue
            T_all = st["T_all"]
            xa, ia, wa = torch.cat(gx[j]), torch.cat(gi[j]), torch.cat(gw[j])
            li = torch.empty((T_all, kk), dtype=torch.int32, device=dev)
            lw = torch.empty((T_all, kk), dtype=torch.float32, device=dev)
            moe_ep_localize(_cfg(cfg, T=T_all), ia, wa, rk.rank * El, El, li,
                            lw)
            rc = _cfg(cfg, T=T_all, E=El, k=kk, S=1,
                      ragged_buffer_factor=-1.0, n_chunks=0,
                      redundant_slots=0)
            rb = alloc_step_buffers(rc, dev)
            moe_permute(rc, xa, li, False, rb["x_sorted"], rb["row_of"],
                        rb["sorted_token"], rb["group_offsets"],
                        rb["uniq_offsets"], rb["uniq_tokens"],
                        rb["expand_idx"], rb["n_dropped"], rb["permute_ws"])
            st.update(li=li, lw=lw, rc=rc, rb=rb)
        return states

    def forward(self, xs, logits):
        cfg, tr = self.cfg, self.tr
        S, H = cfg.S, cfg.H
        dev = xs[0].device
        ranks = [_Rank(r, x, L, cfg, dev)
                 for r, x, L in zip(tr.ranks, xs, logits)]
        states = self._gather(ranks)
        backs = []
        for rk, st in zip(ranks, states):
            part = torch.empty((st["T_all"], H), dtype=rk.x.dtype, device=dev)
            if st["T_all"]:
                rc, rb = st["rc"], st["rb"]
                wg, wu, wd = self.weights(rk.rank)
                moe_gmm_gate_up(rc, rb["x_sorted"], rb["group_offsets"], wg,
                                wu, rb["h"], rb["status"])
                moe_gmm_down(rc, rb["h"], rb["group_offsets"], wd,
                             rb["y_sorted"], rb["status"])
                moe_combine(rc, rb["y_sorted"], rb["row_of"], st["lw"], part)
            backs.append(list(torch.split(part, st["sizes"])))
        # reduce-scatter: each owner receives the ranks' partial rows of its
        # tokens and adds them in rank order
        ret = tr.all_to_all(backs)
        for rk, blocks in zip(ranks, ret):
            if rk.T:
                moe_ep_sum_partials(rk.cfg, S, torch.cat(blocks), rk.y)
        self.saved = (ranks, states) if self.save_x_sorted else None
        return [rk.y for rk in ranks]

    def backward(self, xs, logits, dys):
        """Gradients of sum_r <dys[r], forward(xs, logits)[r]>: per rank
        (dx [T_r, H] layer dtype, dlogits [T_r, E] float32, (dWg, dWu, dWd)
        float32 of its own experts)."""
        cfg, tr = self.cfg, self.tr
        S, H, E, F = cfg.S, cfg.H, cfg.E, cfg.F
        El = E // S
        dev = xs[0].device
        if self.saved is not None:
            ranks, states = self.saved
            self.saved = None
        else:                       # remat: gather and sort again
            ranks = [_Rank(r, x, L, cfg, dev)
                     for r, x, L in zip(tr.ranks, xs, logits)]
            states = self._gather(ranks)
        f32 = dict(dtype=torch.float32, device=dev)
        # the cotangent all-gather
        gdy = tr.all_to_all([[dy] * S for dy in dys])
        dx_back, dw_back, dWs = [], [], []
        for j, (rk, st) in enumerate(zip(ranks, states)):
            T_all = st["T_all"]
            dwg = torch.zeros((El, H, F), **f32)
            dwu = torch.zeros((El, H, F), **f32)
            dwd = torch.zeros((El, F, H), **f32)
            dWs.append((dwg, dwu, dwd))
            part = torch.empty((T_all, H), dtype=rk.x.dtype, device=dev)
            kk = min(cfg.k, El)
            dlw = torch.zeros((T_all, kk), **f32)
            if T_all:
                rc, rb = st["rc"], st["rb"]
                R = rc.T * rc.k
                wg, wu, wd = self.weights(rk.rank)
                g = torch.empty((R, F), dtype=rk.x.dtype, device=dev)
                u = torch.empty_like(g)
                moe_gmm_swiglu_saved(rc, rb["x_sorted"], rb["group_offsets"],
                                     wg, wu, wd, g, u, rb["h"],
                                     rb["y_sorted"], rb["status"])
                dY = torch.cat(gdy[j])
                dys_ = torch.empty((R, H), dtype=rk.x.dtype, device=dev)
                moe_combine_backward(rc, dY, rb["y_sorted"], rb["row_of"],
                                     st["lw"], dys_, dlw)
                dxs_ = torch.empty((R, H), dtype=rk.x.dtype, device=dev)
                ws = torch.empty(max(moe_workspace_bytes(
                    rc, MOE_WS_GMM_BACKWARD), 256), dtype=torch.uint8,
                    device=dev)
                moe_gmm_swiglu_backward(rc, rb["x_sorted"],
                                        rb["group_offsets"], wg, wu, wd, g, u,
                                        rb["h"], dys_, dxs_, dwg, dwu, dwd, 0,
                                        ws, rb["status"])
                moe_permute_backward(rc, dxs_, rb["row_of"], part)
            dx_back.append(list(torch.split(part, st["sizes"])))
            dw_back.append(list(torch.split(dlw, st["sizes"])))
        # the owners: partial dx summed (the tokens' all-gather transposed),
        # each pick's weight gradient from its expert's rank, then the router
        rdx = tr.all_to_all(dx_back)
        rdw = tr.all_to_all(dw_back)
        dxs, dls = [], []
        for rk, blocks, wblocks, L in zip(ranks, rdx, rdw, logits):
            dx = torch.zeros((rk.T, H), dtype=rk.x.dtype, device=dev)
            dl = torch.zeros((rk.T, E), **f32)
            if rk.T:
                moe_ep_sum_partials(rk.cfg, S, torch.cat(blocks), dx)
                dtw = torch.zeros((rk.T, cfg.k), **f32)
                for d, blk in enumerate(wblocks):
                    moe_ep_delocalize(rk.cfg, rk.idx, d * El, El,
                                      blk.contiguous(), dtw)
                moe_route_backward(rk.cfg, L, rk.idx, dtw, dl)
            dxs.append(dx)
            dls.append(dl)
        return dxs, dls, dWs


def local_weights(w_gate, w_up, w_down, n_ranks):
    """weights(rank) over global [E, ...] weight tensors: the rank's
    contiguous slice of E/n_ranks experts (views, nothing copied)."""
    E = w_gate.shape[0]
    El = E // n_ranks

    def get(rank):
        a, z = rank * El, (rank + 1) * El
        return w_gate[a:z], w_up[a:z], w_down[a:z]
    return get


__all__ = ["LoopbackTransport", "DistTransport", "EPLayer", "RingLayer",
           "local_weights", "chunk_bounds", "make_config",
           "moe_workspace_bytes", "MOE_WS_PERMUTE"]
