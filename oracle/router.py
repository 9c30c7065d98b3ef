"""Router front-end (oracle; test infrastructure only).

The step before the routing permutation: per token, logits over the
experts from the BF16 router ("gate") weight (NVFP4 MegaMoE Debug Log,
Checkpoint Layers: "Gate weight ... BF16"), the k largest logits, and their
softmax weights, as the workloads route (top-k with softmax weights; over
the selected logits, or the full softmax's probabilities).

fp64 throughout.  Slot j holds the j-th largest logit; equal logits go to
the lower expert id first.
"""
from __future__ import annotations

import numpy as np


def logits(x, w_router) -> np.ndarray:
    """[T, E] = x [T, H] @ w_router [E, H]^T in fp64 (inputs as given)."""
    return np.asarray(x, dtype=np.float64) @ np.asarray(w_router, dtype=np.float64).T


def topk(lg: np.ndarray, k: int) -> np.ndarray:
    """Ids of the k largest logits per row, largest first, ties to the
    lower id (a stable sort of the negated logits)."""
    return np.argsort(-lg, axis=1, kind="stable")[:, :k].astype(np.int32)


def weights(lg: np.ndarray, ids: np.ndarray, mode: str) -> np.ndarray:
    """mode "selected": softmax over the k selected logits;
    mode "all": the full softmax's probabilities of the selected experts."""
    sel = np.take_along_axis(lg, ids.astype(np.int64), axis=1)
    if mode == "selected":
        ex = np.exp(sel - sel.max(axis=1, keepdims=True))
        return ex / ex.sum(axis=1, keepdims=True)
    if mode == "all":
        m = lg.max(axis=1, keepdims=True)
        return np.exp(sel - m) / np.exp(lg - m).sum(axis=1, keepdims=True)
    raise ValueError(mode)


def route(x, w_router, k: int, mode: str = "selected"):
    lg = logits(x, w_router)
    ids = topk(lg, k)
    return ids, weights(lg, ids, mode), lg
