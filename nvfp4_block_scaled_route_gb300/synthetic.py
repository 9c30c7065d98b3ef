"""Seeded synthetic workloads for the NVFP4 MoE expert FFN.

This module draws random inputs only: bf16 activations, fp32 expert weights
(before any quantisation), per-expert weight spreads, and the top-k routing
choice with its weights.  It holds none of the method's arithmetic (no
quantisation, no GEMM, no activation, no reduction) so that both the CUDA
path and the CPU oracle can be fed from it without sharing any of the
computation they are compared on.

Every tensor comes from its own generator stream, keyed by (seed, purpose,
index), so the weights of expert e are the same in every configuration that
shares E, H and I, and drawing one expert does not require drawing the others.
Draws on ``device="cuda"`` use torch's CUDA generator (fast for the multi-GB
weight sets); draws on the CPU use torch's CPU generator.  The two give
different values for the same key; a test always draws on one device and
copies what the other side needs.

Workload shapes follow the debug log of the NVFP4 MegaMoE kernel ("NVFP4
MegaMoE Debug Log", Hypotheses §2: L1 w=(48,3584,6144), L2 w=(48,1536,7168),
i.e. E=48, H=7168, I=3072).
"""
from __future__ import annotations

import dataclasses
import hashlib
import math
from typing import Optional

import torch


@dataclasses.dataclass(frozen=True)
class MoEConfig:
    name: str
    E: int            # experts
    H: int            # hidden size (L1 K, L2 N)
    I: int            # intermediate size (L1 N = 2*I as [gate; up], L2 K)
    T: int            # tokens
    k: int            # top-k
    routing: str      # see draw_routing
    act: str = "normal"          # "normal" | "student_t"
    act_std: float = 1.5
    w_std: float = 0.02
    expert_spread: bool = True   # per-expert weight std multiplier u_e ~ U(0.5, 2)
    zipf_s: float = 1.2
    seed: int = 0

    @property
    def N1(self) -> int:
        return 2 * self.I

    @property
    def slots(self) -> int:
        return self.T * self.k


# The five workloads of the benchmark description, plus parity cases that
# still span several 128-row tiles with a ragged tail.
CONFIGS = {
    "tiny": MoEConfig("tiny", E=4, H=256, I=128, T=8, k=2,
                      routing="softmax_topk_probs", act_std=1.5,
                      expert_spread=False),
    "decode1": MoEConfig("decode1", E=48, H=7168, I=3072, T=1, k=8,
                         routing="softmax_topk_renorm"),
    "decode64": MoEConfig("decode64", E=48, H=7168, I=3072, T=64, k=8,
                          routing="uniform"),
    "prefill4k": MoEConfig("prefill4k", E=48, H=7168, I=3072, T=4096, k=8,
                           routing="zipf"),
    "prefill16k": MoEConfig("prefill16k", E=48, H=7168, I=3072, T=16384, k=8,
                            routing="hot_expert", act="student_t"),
    # parity-sized cases (not benchmark workloads)
    # the largest batch the single-kernel layer path takes at these sizes
    # (T*k = 16 slots: at most 16 m-tiles x 28 L2 n-tiles below 4 per SM)
    "decode2": MoEConfig("decode2", E=48, H=7168, I=3072, T=2, k=8,
                         routing="uniform"),
    "small": MoEConfig("small", E=6, H=512, I=256, T=97, k=3, routing="zipf"),
    "medium": MoEConfig("medium", E=8, H=1024, I=768, T=600, k=4,
                        routing="zipf"),
    # ~80 m-tiles x 8 n-tiles in each GEMM: more than four waves of whole
    # tiles on a 152-SM GPU, the last one partial, still small enough for
    # the oracle to finish in seconds
    "waves": MoEConfig("waves", E=8, H=2048, I=1024, T=2464, k=4,
                       routing="uniform"),
}


def _key(seed: int, *parts) -> int:
    """Stable 63-bit stream key for (seed, purpose, index...)."""
    h = hashlib.sha256(repr((seed,) + parts).encode()).digest()
    return int.from_bytes(h[:8], "little") & ((1 << 63) - 1)


def _gen(device, seed: int, *parts) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(_key(seed, *parts))
    return g


def expert_spread(cfg: MoEConfig) -> torch.Tensor:
    """u_e ~ U(0.5, 2) per expert (float64, CPU); ones when disabled."""
    if not cfg.expert_spread:
        return torch.ones(cfg.E, dtype=torch.float64)
    g = _gen("cpu", cfg.seed, "spread", cfg.E)
    return 0.5 + 1.5 * torch.rand(cfg.E, generator=g, dtype=torch.float64)


def draw_weight(cfg: MoEConfig, layer: int, e: int, device="cpu") -> torch.Tensor:
    """fp32 weight of expert e in math layout (K, N).

    layer 1: (H, 2I) = [gate | up] along N;  layer 2: (I, H).
    Entries ~ N(0, (w_std * u_e)^2).
    """
    K, N = (cfg.H, cfg.N1) if layer == 1 else (cfg.I, cfg.H)
    u = float(expert_spread(cfg)[e])
    g = _gen(device, cfg.seed, "w", layer, cfg.H, cfg.I, e)
    w = torch.randn((K, N), generator=g, device=device, dtype=torch.float32)
    return w.mul_(cfg.w_std * u)


def draw_router_weight(cfg: MoEConfig, device="cpu") -> torch.Tensor:
    """bf16 router weight [E, H] ~ N(0, s^2) with s = 1 / (act_std * sqrt(H)),
    so that the logits of the workload's activations are about N(0, 1), the
    distribution the routing recipes draw them from."""
    g = _gen(device, cfg.seed, "router", cfg.E, cfg.H)
    w = torch.randn((cfg.E, cfg.H), generator=g, device=device, dtype=torch.float32)
    return w.mul_(1.0 / (cfg.act_std * math.sqrt(cfg.H))).to(torch.bfloat16)


def draw_activations(cfg: MoEConfig, device="cpu", T: Optional[int] = None) -> torch.Tensor:
    """bf16 activations x[T, H] (fp32 draw, rounded to bf16 nearest-even)."""
    T = cfg.T if T is None else T
    g = _gen(device, cfg.seed, "x", cfg.name, cfg.H, T)
    if cfg.act == "normal":
        x = torch.randn((T, cfg.H), generator=g, device=device, dtype=torch.float32)
        x.mul_(cfg.act_std)
    elif cfg.act == "student_t":
        # Student-t(df=3) = Z / sqrt(chi2_3 / 3); scaled to std act_std
        # (the t(3) std is sqrt(3)).
        z = torch.randn((T, cfg.H), generator=g, device=device, dtype=torch.float32)
        c = torch.randn((3, T, cfg.H), generator=g, device=device, dtype=torch.float32)
        chi2 = (c * c).sum(0)
        x = z / torch.sqrt(chi2 / 3.0)
        x.mul_(cfg.act_std / math.sqrt(3.0))
    else:
        raise ValueError(cfg.act)
    return x.to(torch.bfloat16)


def _softmax_rows(logits: torch.Tensor) -> torch.Tensor:
    l64 = logits.to(torch.float64)
    l64 = l64 - l64.max(dim=1, keepdim=True).values
    p = torch.exp(l64)
    return p / p.sum(dim=1, keepdim=True)


def draw_routing(cfg: MoEConfig, T: Optional[int] = None):
    """Top-k routing choice (int32 [T, k]) and weights (float32 [T, k]), CPU.

    softmax_topk_probs   logits ~N(0,1) over E; the k largest softmax
                         probabilities, not renormalised; ties -> lower id.
    softmax_topk_renorm  logits ~N(0,1) over E; top-k; softmax over the k
                         selected logits.
    uniform              k distinct experts uniformly at random; weights =
                         softmax over k N(0,1) logits.
    zipf                 expert popularity p_r ~ r^-s (expert r-1 has rank r);
                         k distinct experts by Gumbel-top-k; weights as uniform.
    hot_expert           expert 0 in every token's top-k, the other k-1 picks
                         distinct and uniform over experts 1..E-7, experts
                         E-6..E-1 receive nothing; weights as uniform.
    """
    T = cfg.T if T is None else T
    E, k = cfg.E, cfg.k
    g = _gen("cpu", cfg.seed, "route", cfg.name, E, T, k)
    if T == 0:
        return torch.zeros((0, k), dtype=torch.int32), torch.zeros((0, k), dtype=torch.float32)
    if cfg.routing in ("softmax_topk_probs", "softmax_topk_renorm"):
        logits = torch.randn((T, E), generator=g, dtype=torch.float32)
        p = _softmax_rows(logits)
        # stable descending sort: equal values keep ascending expert id
        order = torch.sort(-p, dim=1, stable=True).indices[:, :k]
        ids = order
        if cfg.routing == "softmax_topk_probs":
            w = torch.gather(p, 1, order)
        else:
            w = _softmax_rows(torch.gather(logits, 1, order))
    else:
        if cfg.routing == "uniform":
            keys = torch.rand((T, E), generator=g, dtype=torch.float64)
            ids = torch.sort(keys, dim=1, stable=True).indices[:, :k]
        elif cfg.routing == "zipf":
            r = torch.arange(1, E + 1, dtype=torch.float64)
            logp = -cfg.zipf_s * torch.log(r)
            u = torch.rand((T, E), generator=g, dtype=torch.float64).clamp_(1e-300, 1.0)
            gumbel = -torch.log(-torch.log(u))
            ids = torch.sort(-(logp[None, :] + gumbel), dim=1, stable=True).indices[:, :k]
        elif cfg.routing == "hot_expert":
            pool = E - 6 - 1          # experts 1 .. E-7
            assert pool >= k - 1
            keys = torch.rand((T, pool), generator=g, dtype=torch.float64)
            others = torch.sort(keys, dim=1, stable=True).indices[:, : k - 1] + 1
            ids = torch.cat([torch.zeros((T, 1), dtype=torch.int64), others], dim=1)
            # place the hot expert at a random position of the top-k list
            perm = torch.sort(torch.rand((T, k), generator=g, dtype=torch.float64),
                              dim=1, stable=True).indices
            ids = torch.gather(ids, 1, perm)
        else:
            raise ValueError(cfg.routing)
        logits = torch.randn((T, k), generator=g, dtype=torch.float32)
        w = _softmax_rows(logits)
    return ids.to(torch.int32).contiguous(), w.to(torch.float32).contiguous()


def routing_with_counts(counts, k: int, seed: int = 0):
    """Routing whose per-expert slot counts are exactly ``counts``.

    Builds T = sum(counts) / k tokens; expert e appears counts[e] times, never
    twice in one token.  Used for edge cases (experts with 0, 1, 127, 128, 129
    slots).  Weights: softmax of k N(0,1) logits.
    """
    counts = [int(c) for c in counts]
    S = sum(counts)
    assert S % k == 0
    T = S // k
    assert max(counts) <= T
    # round-robin fill of the flat slot list, expert by expert, column-major
    # over tokens: token t gets entries t, t+T, t+2T, ... of the expert list.
    flat = []
    for e, c in enumerate(counts):
        flat += [e] * c
    ids = torch.tensor(flat, dtype=torch.int32).reshape(k, T).t().contiguous()
    g = _gen("cpu", seed, "counts", tuple(counts), k)
    perm = torch.sort(torch.rand((T, k), generator=g, dtype=torch.float64), dim=1).indices
    ids = torch.gather(ids, 1, perm).contiguous()
    w = _softmax_rows(torch.randn((T, k), generator=g, dtype=torch.float32)).to(torch.float32)
    return ids, w.contiguous()
