"""Expert parallelism on CPU ranks: the exchange logic of
nvfp4_block_scaled_route_gb300.ep (global scales by MAX all-reduce, dispatch
of quantised token rows to the experts' owners, the return exchange and the
fixed-order reduce) with the oracle doing each process's arithmetic.  The
composition over G processes must reproduce the oracle's one-process forward
of the whole batch: the same quantised bytes reach every expert, and both
global scales are the whole batch's.  Ranks are gloo processes (world size
2) or threads of one process (LocalGroup).  Not measured on GPU hardware:
every box here has one GPU."""
import os
import socket
import sys
import threading

import numpy as np
import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

from oracle import moe as omoe       # noqa: E402
from oracle import nvfp4 as onv      # noqa: E402
from nvfp4_block_scaled_route_gb300 import synthetic as syn  # noqa: E402
from nvfp4_block_scaled_route_gb300 import ep                  # noqa: E402


class OracleBackend:
    """One process's share of the forward, in the oracle's arithmetic.
    ckpt: the whole checkpoint (w1q, w1sf, gs1, w2q, w2sf, gs2); this process
    uses experts [rank*E/G, (rank+1)*E/G)."""

    def __init__(self, ckpt, E, G, rank, H, I):
        self.ck, self.E, self.G, self.rank, self.H, self.I = ckpt, E, G, rank, H, I
        self.El = E // G

    def token_amax(self, x):
        return torch.tensor([np.max(np.abs(x.numpy())) if x.numel() else 0.0],
                            dtype=torch.float32)

    def quantize_tokens(self, x, amax):
        q, sf, gs = onv.quantize_rows(x.numpy(), onv.global_scale(np.float32(amax.item())))
        return q, sf, gs

    def dispatch(self, topk_ids, q, sf):
        ids = topk_ids.numpy().reshape(-1)
        k = topk_ids.shape[1]
        dest = ids // self.El
        counts = [int(np.sum(dest == d)) for d in range(self.G)]
        order = np.concatenate([np.nonzero(dest == d)[0] for d in range(self.G)]).astype(np.int64)
        pos = np.empty(len(ids), dtype=np.int64)
        pos[order] = np.arange(len(ids))
        rows = np.concatenate([q[order // k], sf[order // k]], axis=1)
        expert = (ids[order] - dest[order] * self.El).astype(np.int32)
        return counts, torch.from_numpy(pos), torch.from_numpy(rows), torch.from_numpy(expert)

    def expert_phase1(self, recv_rows, recv_expert, gs_x):
        rows = recv_rows.numpy()
        self.n = rows.shape[0]
        self.exp = recv_expert.numpy().astype(np.int64)
        H, I = self.H, self.I
        w1q, w1sf, gs1 = self.ck[0], self.ck[1], self.ck[2]
        self.h = np.zeros((self.n, I), dtype=np.float32)
        for e in range(self.El):
            sel = np.nonzero(self.exp == e)[0]
            if len(sel) == 0:
                continue
            g = self.rank * self.El + e
            l1 = omoe.expert_l1(rows[sel, :H // 2], rows[sel, H // 2:], gs_x, w1q[g], w1sf[g],
                                gs1[g])
            self.h[sel] = omoe.swiglu(l1)
        return torch.tensor([np.max(np.abs(self.h)) if self.n else 0.0], dtype=torch.float32)

    def expert_phase2(self, amax_h):
        w2q, w2sf, gs2 = self.ck[3], self.ck[4], self.ck[5]
        out = np.zeros((self.n, self.H), dtype=np.float64)
        if self.n:
            gs_h = onv.global_scale(np.float32(amax_h.item()))
            hq, hsf, _ = onv.quantize_rows(self.h, gs_h)
            for e in range(self.El):
                sel = np.nonzero(self.exp == e)[0]
                if len(sel):
                    g = self.rank * self.El + e
                    out[sel] = omoe.expert_l2(hq[sel], hsf[sel], gs_h, w2q[g], w2sf[g], gs2[g])
        return torch.from_numpy(out)

    def reduce(self, back_rows, send_pos, topk_w):
        return torch.from_numpy(omoe.unpermute_reduce(back_rows.numpy(), send_pos.numpy(),
                                                      topk_w.numpy()))


def _problem(E=4, H=256, I=128, T=24, k=2, routing="uniform", seed=3):
    cfg = syn.MoEConfig("ep", E=E, H=H, I=I, T=T, k=k, routing=routing, seed=seed)
    x = syn.draw_activations(cfg).float()
    ids, w = syn.draw_routing(cfg)
    W1 = [syn.draw_weight(cfg, 1, e).numpy() for e in range(E)]
    W2 = [syn.draw_weight(cfg, 2, e).numpy() for e in range(E)]
    w1q, w1sf, gs1 = omoe.quantize_expert_weights(W1)
    w2q, w2sf, gs2 = omoe.quantize_expert_weights(W2)
    ckpt = (w1q, w1sf, gs1, w2q, w2sf, gs2)
    ref = omoe.forward(x.numpy(), ids.numpy(), w.numpy(), *ckpt)
    return cfg, x, ids, w, ckpt, ref


def _shares(T, G):
    cuts = [T * r // G for r in range(G + 1)]
    return [(cuts[r], cuts[r + 1]) for r in range(G)]


def _check(y, ref_rows):
    scale = max(1e-30, float(np.max(np.abs(ref_rows))))
    assert y.shape == ref_rows.shape
    # the same operations on the same bytes; only BLAS blocking may differ
    assert float(np.max(np.abs(y - ref_rows))) <= 1e-12 * scale


def _run_local(G, E, ids_override=None):
    cfg, x, ids, w, ckpt, ref = _problem(E=E)
    if ids_override is not None:
        ids = ids_override
        ref = omoe.forward(x.numpy(), ids.numpy(), w.numpy(), *ckpt)
    grp = ep.LocalGroup(G)
    out = [None] * G
    errs = []

    def rank_main(r):
        try:
            t0, t1 = _shares(cfg.T, G)[r]
            be = OracleBackend(ckpt, E, G, r, cfg.H, cfg.I)
            m = ep.ExpertParallelMoE(be, grp.comm(r))
            out[r] = m.forward(x[t0:t1].contiguous(), ids[t0:t1].contiguous(),
                               w[t0:t1].contiguous()).numpy()
        except Exception as e:  # surfaced below
            errs.append(e)
            grp._barrier.abort()

    th = [threading.Thread(target=rank_main, args=(r,)) for r in range(G)]
    for t in th:
        t.start()
    for t in th:
        t.join()
    if errs:
        raise errs[0]
    for r in range(G):
        t0, t1 = _shares(cfg.T, G)[r]
        _check(out[r], ref["y64"][t0:t1])


def test_local_group_matches_one_process():
    _run_local(G=4, E=8)


def test_one_rank_is_the_plain_forward():
    _run_local(G=1, E=4)


def test_a_rank_that_receives_nothing():
    """Every slot goes to rank 0's experts: rank 1 receives no rows, runs an
    empty L1 (max |h| = 0) and still takes part in every exchange."""
    T, k = 24, 2
    ids = torch.tensor([[0, 1]] * T, dtype=torch.int32)
    _run_local(G=2, E=4, ids_override=ids)


# --------------------------------------------------------------- gloo ranks --
def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _gloo_worker(rank, world, port, q):
    import torch.distributed as dist
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        cfg, x, ids, w, ckpt, ref = _problem(E=4, T=20)
        t0, t1 = _shares(cfg.T, world)[rank]
        be = OracleBackend(ckpt, cfg.E, world, rank, cfg.H, cfg.I)
        m = ep.ExpertParallelMoE(be, ep.TorchComm("cpu"))
        y = m.forward(x[t0:t1].contiguous(), ids[t0:t1].contiguous(), w[t0:t1].contiguous())
        ref_rows = ref["y64"][t0:t1]
        err = float(np.max(np.abs(y.numpy() - ref_rows)))
        q.put((rank, err, float(np.max(np.abs(ref_rows)))))
    finally:
        dist.barrier()
        dist.destroy_process_group()


def test_two_gloo_ranks_match_one_process():
    import torch.multiprocessing as tmp
    world = 2
    q = tmp.get_context("spawn").SimpleQueue()
    tmp.start_processes(_gloo_worker, args=(world, _free_port(), q), nprocs=world,
                        start_method="spawn")
    got = sorted(q.get() for _ in range(world))
    assert [g[0] for g in got] == [0, 1]
    for _, err, scale in got:
        assert err <= 1e-12 * scale
