"""MoE expert FFN forward pass (oracle; test infrastructure only).

Follows the "NVFP4 MoE Pipeline" of the NVFP4 MegaMoE Debug Log
(Architecture Notes):

    stage_activation(x)            -> x_fp4, x_sf, igs
    L1 GEMM (x_fp4,x_sf)@(w1,sf1)  with alpha = igs * w1_gs[e]   -> gate_up
    SiLU(gate) * up                -> activated
    stage_activation(activated)    -> l1_fp4, l1_sf, l1_igs
    L2 GEMM (l1_fp4,l1_sf)@(w2,sf2) with alpha = l1_igs * w2_gs[e] -> out
    scatter with routing weights   -> y

plus the routing permutation that groups the (token, choice) slots by expert
(the Debug Log's "L2 slot_token" / ``slots=`` trace lines).  Alpha is a
per-expert fp32 pair of global scales applied to the accumulator, never
folded into the E4M3 block scales (Hypotheses §3).  The L1 output is a plain
[gate; up] concatenation along N (commit message on the removed 2-CTA
interleave): gate = columns [0, I), up = columns [I, 2I).

Accumulation is fp64 throughout; h is rounded to fp32 before it is
requantised (it is an fp32 tensor in the pipeline); y is rounded once to
bf16.
"""
from __future__ import annotations

import math

import numpy as np

from . import nvfp4

TILE_ROWS = 128   # expert segments of the grouped slot layout start at multiples of this


# -------------------------------------------------------------- routing ----

def route(topk_ids: np.ndarray, E: int):
    """Counting sort of the T*k (token, choice) pairs by expert.

    Slot order within an expert is ascending flat index t*k + j (stable).
    Returns dict with
      counts[E]          slots per expert
      offsets[E+1]       exclusive prefix sum of counts (dense slot ids)
      slot_token[S]      token of each dense slot
      slot_flat[S]       flat index t*k+j of each dense slot
      slot_of[T*k]       dense slot of each (t, j)
    Pinned: brute force on tiny inputs, permutation invariants.
    """
    ids = np.asarray(topk_ids, dtype=np.int64)
    T, k = ids.shape
    flat = ids.reshape(-1)
    if flat.size and (flat.min() < 0 or flat.max() >= E):
        raise ValueError("expert id out of range")
    counts = np.bincount(flat, minlength=E).astype(np.int64)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    order = np.argsort(flat, kind="stable")           # dense slot -> flat index
    slot_of = np.empty(T * k, dtype=np.int64)
    slot_of[order] = np.arange(T * k)
    return dict(counts=counts, offsets=offsets, slot_token=order // k,
                slot_flat=order, slot_of=slot_of)


def padded_layout(r: dict, tile_rows: int = TILE_ROWS):
    """Map dense slots onto the grouped row layout whose expert segments start
    at multiples of ``tile_rows`` (the library's slot layout).

    row_offsets[e] = sum over e' < e of ceil(counts[e'] / tile_rows) * tile_rows
    row of dense slot s of expert e = row_offsets[e] + (s - offsets[e]).
    Returns dict with row_offsets[E+1], row_token[rows] (-1 on padding),
    row_of[T*k].
    """
    counts = r["counts"]
    E = counts.size
    padded = ((counts + tile_rows - 1) // tile_rows) * tile_rows
    row_offsets = np.concatenate([[0], np.cumsum(padded)]).astype(np.int64)
    rows = int(row_offsets[-1])
    row_token = -np.ones(rows, dtype=np.int64)
    dense_to_row = np.empty(int(r["offsets"][-1]), dtype=np.int64)
    for e in range(E):
        s0, s1 = r["offsets"][e], r["offsets"][e + 1]
        dense_to_row[s0:s1] = row_offsets[e] + np.arange(s1 - s0)
    row_token[dense_to_row] = r["slot_token"]
    return dict(row_offsets=row_offsets, row_token=row_token,
                row_of=dense_to_row[r["slot_of"]])


# ----------------------------------------------------------------- GEMM ----

def block_scaled_matmul(a_q, a_sf, w_q, w_sf) -> np.ndarray:
    """acc[m, n] = sum_k dec(a)[m,k] dec(sfa)[m,k/16] dec(w)[k,n] dec(sfw)[k/16,n]

    a_q (M, K/2), a_sf (M, K/16) row layout; w_q (K/2, N), w_sf (K/16, N)
    checkpoint layout.  fp64; global scales are NOT applied here.
    Pinned: brute-force blockwise loops, constant-scale test, single-SF probes.
    """
    A = nvfp4.dequantize_rows(a_q, a_sf)
    W = nvfp4.dequantize_weight(w_q, w_sf)
    return A @ W


def silu(x: np.ndarray) -> np.ndarray:
    """x * sigmoid(x) = x / (1 + exp(-x)), fp64.  Pinned: closed forms."""
    x = np.asarray(x, dtype=np.float64)
    with np.errstate(over="ignore"):
        return x / (1.0 + np.exp(-x))


def expert_l1(a_q, a_sf, gs_a, w1_q, w1_sf, gs_w1):
    """Alpha-scaled L1 output [M, 2I] (fp64): acc * (gs_a * gs_w1).

    gs_w1 is one scalar, or a (gate, up) pair for checkpoints that quantise
    the two halves separately: then the gate columns [0, I) take
    gs_a * gs_gate and the up columns [I, 2I) gs_a * gs_up (the Debug Log's
    gate/up correction, code-review point 5: a per-column alpha)."""
    acc = block_scaled_matmul(a_q, a_sf, w1_q, w1_sf)
    g = np.atleast_1d(np.asarray(gs_w1, dtype=np.float32))
    if g.size == 1:
        return acc * (float(np.float32(gs_a)) * float(g[0]))
    I = acc.shape[1] // 2
    out = np.empty_like(acc)
    out[:, :I] = acc[:, :I] * (float(np.float32(gs_a)) * float(g[0]))
    out[:, I:] = acc[:, I:] * (float(np.float32(gs_a)) * float(g[1]))
    return out


def swiglu(l1: np.ndarray) -> np.ndarray:
    """h = SiLU(gate) * up on the [gate | up] halves, rounded to fp32."""
    I = l1.shape[1] // 2
    return (silu(l1[:, :I]) * l1[:, I:]).astype(np.float32)


def expert_l2(h_q, h_sf, gs_h, w2_q, w2_sf, gs_w2):
    """Alpha-scaled L2 output [M, H] (fp64)."""
    alpha = float(np.float32(gs_h)) * float(np.float32(gs_w2))
    return block_scaled_matmul(h_q, h_sf, w2_q, w2_sf) * alpha


# --------------------------------------------------------------- reduce ----

def unpermute_reduce(slot_out: np.ndarray, slot_of: np.ndarray, topk_w: np.ndarray):
    """y[t] = sum_j w[t, j] * slot_out[slot_of[t*k + j]]  (fp64, j ascending).
    Returns the fp64 sum (not rounded).  Pinned: brute force."""
    w = np.asarray(topk_w, dtype=np.float64)
    T, k = w.shape
    y = np.zeros((T, slot_out.shape[1]), dtype=np.float64)
    so = np.asarray(slot_out, dtype=np.float64)
    for j in range(k):
        y += w[:, j:j + 1] * so[slot_of.reshape(T, k)[:, j]]
    return y


# -------------------------------------------------------------- forward ----

def quantize_expert_weights(w_list, split_halves: bool = False):
    """List of fp32 (K, N) weights -> stacked checkpoint tensors
    (E, K/2, N), (E, K/16, N), gs (E,) float32.

    split_halves: the columns [0, N/2) and [N/2, N) (L1 gate and up) are
    quantised as two separate matrices with their own global scales, and gs
    is (E, 2) float32 (gate, up)."""
    qs, sfs, gss = [], [], []
    for w in w_list:
        if split_halves:
            n = w.shape[1] // 2
            qg, sfg, gg = nvfp4.quantize_weight(w[:, :n])
            qu, sfu, gu = nvfp4.quantize_weight(w[:, n:])
            q = np.concatenate([qg, qu], axis=1)
            sf = np.concatenate([sfg, sfu], axis=1)
            gs = (gg, gu)
        else:
            q, sf, gs = nvfp4.quantize_weight(w)
        qs.append(q)
        sfs.append(sf)
        gss.append(gs)
    return np.stack(qs), np.stack(sfs), np.array(gss, dtype=np.float32)


def forward(x, topk_ids, topk_w, w1_q, w1_sf, gs_w1, w2_q, w2_sf, gs_w2,
            expert_subset=None, gs_mid=None):
    """Whole forward pass.  x: [T, H] float32 holding bf16 values.

    Weights in checkpoint layout: w1_q (E, H/2, 2I), w1_sf (E, H/16, 2I),
    w2_q (E, I/2, H), w2_sf (E, I/16, H), gs_w* (E,); gs_w1 may be (E, 2)
    (separate gate and up global scales).
    gs_mid (E,): a static intermediate global scale per expert in place of
    the pipeline's dynamic one: h rows of expert e are requantised with
    gs_mid[e] and L2 takes alpha = gs_mid[e] * gs_w2[e]; gs_h is then None.  w*_q may also be a
    callable e -> (q, sf) that yields one expert at a time (to bound memory).
    Returns a dict of every intermediate (dense slot order).
    """
    x = np.asarray(x, dtype=np.float32)
    T, H = x.shape
    ids = np.asarray(topk_ids)
    k = ids.shape[1]
    E = len(gs_w1)
    r = route(ids, E)
    S = T * k

    xq, xsf, gs_x = nvfp4.quantize_rows(x)                       # step 2

    def w1(e):
        return w1_q(e) if callable(w1_q) else (w1_q[e], w1_sf[e])

    def w2(e):
        return w2_q(e) if callable(w2_q) else (w2_q[e], w2_sf[e])

    l1 = None
    for e in range(E):                                            # step 3 + 6
        s0, s1 = r["offsets"][e], r["offsets"][e + 1]
        if s1 == s0:
            continue
        toks = r["slot_token"][s0:s1]
        q, sf = w1(e)
        out = expert_l1(xq[toks], xsf[toks], gs_x, q, sf, gs_w1[e])
        if l1 is None:
            l1 = np.zeros((S, out.shape[1]), dtype=np.float64)
        l1[s0:s1] = out
    if l1 is None:
        I = (w1(0)[0].shape[-1]) // 2
        l1 = np.zeros((0, 2 * I))
    h = swiglu(l1)                                                # step 4
    if gs_mid is None:
        hq, hsf, gs_h = nvfp4.quantize_rows(h)                    # step 4
    else:
        hq = np.zeros((S, h.shape[1] // 2), dtype=np.uint8)
        hsf = np.zeros((S, h.shape[1] // 16), dtype=np.uint8)
        gs_h = None
        for e in range(E):
            s0, s1 = r["offsets"][e], r["offsets"][e + 1]
            if s1 > s0:
                hq[s0:s1], hsf[s0:s1], _ = nvfp4.quantize_rows(h[s0:s1], np.float32(gs_mid[e]))
    out2 = np.zeros((S, H), dtype=np.float64)
    for e in range(E):                                            # step 5 + 6
        s0, s1 = r["offsets"][e], r["offsets"][e + 1]
        if s1 == s0:
            continue
        q, sf = w2(e)
        g = gs_h if gs_mid is None else np.float32(gs_mid[e])
        out2[s0:s1] = expert_l2(hq[s0:s1], hsf[s0:s1], g, q, sf, gs_w2[e])
    y64 = unpermute_reduce(out2, r["slot_of"], topk_w)            # step 7
    return dict(route=r, xq=xq, xsf=xsf, gs_x=gs_x, l1=l1, h=h, hq=hq, hsf=hsf,
                gs_h=gs_h, gs_mid=gs_mid, out2=out2, y64=y64,
                y_bf16=nvfp4.round_to_bf16(y64))


def cosine(a, b) -> float:
    a = np.asarray(a, dtype=np.float64).ravel()
    b = np.asarray(b, dtype=np.float64).ravel()
    na, nb = math.sqrt(float(a @ a)), math.sqrt(float(b @ b))
    if na == 0 or nb == 0:
        return 1.0 if na == nb else 0.0
    return float(a @ b) / (na * nb)
