"""Expert parallelism: the MoE forward with the E experts split over G
processes (E/G consecutive experts each), every process holding its own
tokens.

The pages' 48-expert layer is itself one tensor-parallel rank's share of a
larger MoE ("NVFP4 MoE Debug Log (early)", Symptoms: every TP rank holds
the same weight shapes; Hypotheses section 7, the per-rank table).  Here the
experts are sharded instead, and a token's slot travels to the process that
owns its expert:

  1. amax of the local tokens, MAX over processes -> gs_x of the whole batch
     ("NVFP4 MoE Pipeline" step 2: one global scale per tensor);
  2. each token quantised once with it (E2M1 nibbles + row-major E4M3 scales,
     H/2 + H/16 bytes per row: a quarter of the bf16 row);
  3. dispatch: each slot's row to its expert's owner (all-to-all), with the
     expert's index on the owner;
  4. owner: the received rows routed over its experts and run through L1;
     max |h|, MAX over processes -> gs_h of the whole batch (step 4), then
     requantisation and L2;
  5. combine: the slot outputs back to the token's process (all-to-all) and
     the fixed-order top-k reduce there (step 7).

With the tokens split over the processes in order, each expert sees its
slots in the one-process order and both global scales are the whole batch's,
so every slot row is computed from the same bytes as on one process.

The exchanges go through a communicator (TorchComm: torch.distributed,
NCCL between GPUs or gloo on CPU; LocalGroup: G ranks emulated in one
process, exchanging through host memory, for tests and for running G expert
shards on one GPU).  The per-process work goes through a backend:
CudaExpertBackend runs it in the library's kernels.
"""
from __future__ import annotations

import threading
from typing import List, Optional

import torch

from . import binding as nb


# ------------------------------------------------------------ communicators --
class TorchComm:
    """torch.distributed collectives on `device` (cuda with NCCL, cpu with gloo)."""

    def __init__(self, device, group=None):
        import torch.distributed as dist
        self.dist = dist
        self.group = group
        self.device = torch.device(device)
        self.rank = dist.get_rank(group)
        self.world = dist.get_world_size(group)

    def all_reduce_max(self, t: torch.Tensor) -> None:
        self.dist.all_reduce(t, op=self.dist.ReduceOp.MAX, group=self.group)

    def exchange_counts(self, send_counts: List[int]) -> List[int]:
        s = torch.tensor(send_counts, dtype=torch.int64, device=self.device)
        r = torch.empty_like(s)
        self.dist.all_to_all_single(r, s, group=self.group)
        return [int(v) for v in r.tolist()]

    def all_to_all(self, send: torch.Tensor, send_counts: List[int],
                   recv_counts: List[int]) -> torch.Tensor:
        out = torch.empty((sum(recv_counts),) + tuple(send.shape[1:]), dtype=send.dtype,
                          device=send.device)
        self.dist.all_to_all_single(out, send.contiguous(), output_split_sizes=recv_counts,
                                    input_split_sizes=send_counts, group=self.group)
        return out


class LocalGroup:
    """G ranks emulated in one process (one thread per rank): each collective
    is a host barrier around copies through host-visible tensors.  A rank
    synchronises the device before publishing a tensor, so no kernel of one
    rank ever waits on another rank's kernels."""

    def __init__(self, world: int):
        self.world = world
        self._barrier = threading.Barrier(world)
        self._slots: list = [None] * world

    def comm(self, rank: int) -> "LocalComm":
        return LocalComm(self, rank)


class LocalComm:
    def __init__(self, group: LocalGroup, rank: int):
        self.g = group
        self.rank = rank
        self.world = group.world

    def _publish(self, value):
        if torch.cuda.is_available():
            torch.cuda.synchronize()
        self.g._slots[self.rank] = value
        self.g._barrier.wait()

    def _done(self):
        self.g._barrier.wait()

    def all_reduce_max(self, t: torch.Tensor) -> None:
        self._publish(t.clone())
        m = self.g._slots[0].clone()
        for v in self.g._slots[1:]:
            m = torch.maximum(m, v.to(m.device))
        self._done()
        t.copy_(m)

    def exchange_counts(self, send_counts: List[int]) -> List[int]:
        self._publish(list(send_counts))
        got = [self.g._slots[s][self.rank] for s in range(self.world)]
        self._done()
        return got

    def all_to_all(self, send: torch.Tensor, send_counts: List[int],
                   recv_counts: List[int]) -> torch.Tensor:
        offs = [0]
        for c in send_counts:
            offs.append(offs[-1] + c)
        self._publish((send, offs))
        parts = []
        for s in range(self.world):
            src, o = self.g._slots[s]
            parts.append(src[o[self.rank]:o[self.rank + 1]].clone())
        self._done()
        assert [p.shape[0] for p in parts] == list(recv_counts)
        if not parts:
            return send[:0].clone()
        return torch.cat(parts, dim=0)


# ---------------------------------------------------------------- backend --
class CudaExpertBackend:
    """One process's share of the work in the library's kernels: its experts'
    prepared weights (E_local = E/G of them, global ids rank*E_local + e)."""

    def __init__(self, weights: nb.PreparedWeights, E: int, G: int, k: int,
                 slot_dtype=torch.float16, out_dtype=torch.bfloat16, device="cuda"):
        if E % G != 0 or weights.E != E // G:
            raise ValueError("the process holds E/G experts")
        self.w = weights
        self.E, self.G, self.k = E, G, k
        self.H, self.I = weights.H, weights.I
        self.slot_dtype = slot_dtype
        self.out_dtype = out_dtype
        self.device = torch.device(device)
        self._st = None

    def token_amax(self, x: torch.Tensor) -> torch.Tensor:
        return nb.amax(x)

    def quantize_tokens(self, x: torch.Tensor, amax: torch.Tensor):
        q, sf, _, gs = nb.quantize_act_amax(x, amax)
        return q, sf, gs

    def dispatch(self, topk_ids: torch.Tensor, q: torch.Tensor, sf: torch.Tensor):
        counts, pos, rows, expert, ws = nb.ep_dispatch(topk_ids, self.E, self.G, q, sf)
        self._dispatch_ws = ws
        return [int(c) for c in counts.tolist()], pos, rows, expert

    def expert_phase1(self, recv_rows: torch.Tensor, recv_expert: torch.Tensor,
                      gs_x: torch.Tensor) -> torch.Tensor:
        n = recv_rows.shape[0]
        H, I, El = self.H, self.I, self.w.E
        ids = recv_expert.view(n, 1).to(torch.int32).contiguous()
        route = nb.route_permute(ids, El)
        rows = route.rows
        xq = torch.zeros((max(rows, 1), H // 2), dtype=torch.uint8, device=self.device)
        xsf = torch.zeros(max(nb.sf_mma_bytes(rows, H), 16), dtype=torch.uint8, device=self.device)
        nb.ep_scatter(recv_rows, H, route.slot_of, rows, xq, xsf)
        slot_out = torch.empty((max(rows, 1), H), dtype=self.slot_dtype, device=self.device)
        ws = nb._workspace(nb.forward_workspace_bytes(n, 1, El, H, I), self.device)
        amax_h = torch.empty(1, dtype=torch.float32, device=self.device)
        nb.nvfp4_forward_phase(self.w, xq, xsf, gs_x, route, 1, amax_h, slot_out, ws)
        self._st = (n, route, xq, xsf, gs_x, slot_out, ws, amax_h)
        return amax_h

    def expert_phase2(self, amax_h: torch.Tensor) -> torch.Tensor:
        n, route, xq, xsf, gs_x, slot_out, ws, _ = self._st
        nb.nvfp4_forward_phase(self.w, xq, xsf, gs_x, route, 2, amax_h, slot_out, ws)
        out = nb.ep_gather(slot_out, route.slot_of, n)
        self.status = nb.read_status(ws)
        self._st = None
        return out

    def reduce(self, back_rows: torch.Tensor, send_pos: torch.Tensor,
               topk_w: torch.Tensor) -> torch.Tensor:
        T, k = topk_w.shape
        if back_rows.shape[0] == 0:
            back_rows = torch.zeros((1, self.H), dtype=self.slot_dtype, device=self.device)
        return nb.unpermute_reduce(back_rows, send_pos, topk_w, out_dtype=self.out_dtype)


# ----------------------------------------------------------- orchestration --
class ExpertParallelMoE:
    """The expert-parallel forward of one process (see the module docstring)."""

    def __init__(self, backend, comm):
        self.be = backend
        self.comm = comm

    def forward(self, x: torch.Tensor, topk_ids: torch.Tensor, topk_w: torch.Tensor):
        be, comm = self.be, self.comm
        a = be.token_amax(x)
        comm.all_reduce_max(a)                                   # gs_x of the whole batch
        q, sf, gs_x = be.quantize_tokens(x, a)
        counts, pos, rows, expert = be.dispatch(topk_ids, q, sf)
        recv_counts = comm.exchange_counts(counts)
        recv_rows = comm.all_to_all(rows, counts, recv_counts)
        recv_expert = comm.all_to_all(expert, counts, recv_counts)
        amax_h = be.expert_phase1(recv_rows, recv_expert, gs_x)
        comm.all_reduce_max(amax_h)                              # gs_h of the whole batch
        out = be.expert_phase2(amax_h)
        back = comm.all_to_all(out, recv_counts, counts)
        return be.reduce(back, pos, topk_w)
