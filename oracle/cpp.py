"""ctypes front end of the C++ oracle (nvfp4_oracle.cpp) — test
infrastructure only.

Two namespaces with the same functions, arguments and results as the numpy
oracle (``oracle.nvfp4`` and ``oracle.moe``), so that every pin runs against
both and every parity test can take either:

    from oracle.cpp import nvfp4, moe

Only argument marshalling lives here; the arithmetic is the C++ code's.  The
routing dicts, the padded layout and the cosine helper (a test metric, not
part of the method) are assembled from the C++ results.
"""
from __future__ import annotations

import ctypes
import math
import os
import time
import types

import numpy as np

from . import build as _build

_lib = None
_P, _I, _I64, _F, _D = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_double
_SIGS = {
    "nvo_e2m1_decode": (_D, [_I]), "nvo_e2m1_encode": (_I, [_D]),
    "nvo_e4m3_decode": (_D, [_I]), "nvo_e4m3_encode_nonneg": (_I, [_D]),
    "nvo_global_scale": (_F, [_F]),
    "nvo_e2m1_decode_n": (None, [_P, _I64, _P]), "nvo_e2m1_encode_n": (None, [_P, _I64, _P]),
    "nvo_e4m3_decode_n": (None, [_P, _I64, _P]),
    "nvo_e4m3_encode_nonneg_n": (None, [_P, _I64, _P]),
    "nvo_pack_nibbles": (None, [_P, _I64, _I64, _P]),
    "nvo_unpack_nibbles": (None, [_P, _I64, _I64, _P]),
    "nvo_unpack_weight_k": (None, [_P, _I64, _I64, _P]),
    "nvo_quantize_rows": (None, [_P, _I64, _I64, _I, _F, _P, _P, _P]),
    "nvo_dequantize_rows": (None, [_P, _P, _I64, _I64, _P]),
    "nvo_quantize_weight": (None, [_P, _I64, _I64, _P, _P, _P]),
    "nvo_dequantize_weight": (None, [_P, _P, _I64, _I64, _P]),
    "nvo_matmul_f64": (None, [_P, _P, _I64, _I64, _I64, _P]),
    "nvo_block_scaled_matmul": (None, [_P, _P, _I64, _I64, _P, _P, _I64, _P]),
    "nvo_route": (_I, [_P, _I64, _I, _I, _P, _P, _P, _P]),
    "nvo_padded_layout": (_I64, [_P, _P, _P, _P, _I64, _I, _I, _I, _P, _P, _P, _I64]),
    "nvo_silu": (_D, [_D]),
    "nvo_swiglu": (None, [_P, _I64, _I64, _P]),
    "nvo_unpermute_reduce": (None, [_P, _I64, _P, _P, _I64, _I, _P]),
    "nvo_round_to_bf16": (_D, [_D]),
    "nvo_forward": (_I, [_P, _I64, _I64, _P, _P, _I, _I, _I64, _P, _P, _P, _I, _P, _P, _P, _P,
                         _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "nvo_max_threads": (_I, []), "nvo_set_threads": (None, [_I]),
}


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        l = ctypes.CDLL(path)
        for name, (res, args) in _SIGS.items():
            f = getattr(l, name)
            f.restype = res
            f.argtypes = args
        _lib = l
    return _lib


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _p(a):
    return a.ctypes.data if a is not None else None


def threads() -> int:
    return int(lib().nvo_max_threads())


# ------------------------------------------------------------ nvfp4 ----
def e2m1_decode(nib):
    n = _c(np.asarray(nib).astype(np.int64) & 15, np.uint8)
    out = np.empty(n.shape, np.float64)
    lib().nvo_e2m1_decode_n(_p(n), n.size, _p(out))
    return out


def e2m1_encode(v):
    """Nearest E2M1 code of each value (fp32 values widen exactly)."""
    a = _c(np.asarray(v).astype(np.float64), np.float64)
    out = np.empty(a.shape, np.uint8)
    lib().nvo_e2m1_encode_n(_p(a), a.size, _p(out))
    return out


def e4m3_decode(byte):
    b = _c(np.asarray(byte).astype(np.int64) & 255, np.uint8)
    out = np.empty(b.shape, np.float64)
    lib().nvo_e4m3_decode_n(_p(b), b.size, _p(out))
    return out


def e4m3_encode_nonneg(v):
    a = _c(v, np.float64)
    if np.any(a < 0) or np.any(np.isnan(a)):
        raise ValueError("scale inputs must be finite and non-negative")
    out = np.empty(a.shape, np.uint8)
    lib().nvo_e4m3_encode_nonneg_n(_p(a), a.size, _p(out))
    return out


def pack_nibbles(nib):
    n = _c(nib, np.uint8)
    K = n.shape[-1]
    assert K % 2 == 0
    R = n.size // K if K else 0
    out = np.empty(n.shape[:-1] + (K // 2,), np.uint8)
    lib().nvo_pack_nibbles(_p(n), R, K, _p(out))
    return out


def unpack_nibbles(packed):
    p = _c(packed, np.uint8)
    K = 2 * p.shape[-1]
    R = p.size // p.shape[-1] if p.shape[-1] else 0
    out = np.empty(p.shape[:-1] + (K,), np.uint8)
    lib().nvo_unpack_nibbles(_p(p), R, K, _p(out))
    return out


def unpack_weight_k(packed_kn):
    p = _c(packed_kn, np.uint8)
    K2, N = p.shape[-2], p.shape[-1]
    lead = p.shape[:-2]
    p2 = p.reshape(-1, K2, N)
    out = np.empty((p2.shape[0], 2 * K2, N), np.uint8)
    for i in range(p2.shape[0]):
        lib().nvo_unpack_weight_k(_p(p2[i]), 2 * K2, N, _p(out[i]))
    return out.reshape(lead + (2 * K2, N))


def global_scale(amax):
    return np.float32(lib().nvo_global_scale(float(np.float32(amax))))


def quantize_rows(v, gs=None):
    v = _c(v, np.float32)
    R, K = v.shape
    assert K % 16 == 0
    q = np.empty((R, K // 2), np.uint8)
    sf = np.empty((R, K // 16), np.uint8)
    g = ctypes.c_float(0.0)
    lib().nvo_quantize_rows(_p(v), R, K, 0 if gs is None else 1,
                            float(np.float32(gs)) if gs is not None else 0.0,
                            _p(q), _p(sf), ctypes.addressof(g))
    return q, sf, np.float32(g.value)


def dequantize_rows(q, sf):
    q, sf = _c(q, np.uint8), _c(sf, np.uint8)
    R, K = q.shape[0], 2 * q.shape[1]
    out = np.empty((R, K), np.float64)
    lib().nvo_dequantize_rows(_p(q), _p(sf), R, K, _p(out))
    return out


def quantize_weight(w_kn):
    w = _c(w_kn, np.float32)
    K, N = w.shape
    q = np.empty((K // 2, N), np.uint8)
    sf = np.empty((K // 16, N), np.uint8)
    g = ctypes.c_float(0.0)
    lib().nvo_quantize_weight(_p(w), K, N, _p(q), _p(sf), ctypes.addressof(g))
    return q, sf, np.float32(g.value)


def dequantize_weight(q_kn, sf_kn):
    q, sf = _c(q_kn, np.uint8), _c(sf_kn, np.uint8)
    K, N = 2 * q.shape[0], q.shape[1]
    out = np.empty((K, N), np.float64)
    lib().nvo_dequantize_weight(_p(q), _p(sf), K, N, _p(out))
    return out


def round_to_bf16(x):
    x = np.asarray(x, np.float64)
    f = np.vectorize(lambda v: lib().nvo_round_to_bf16(float(v)), otypes=[np.float64])
    return f(x) if x.size else x.copy()


nvfp4 = types.SimpleNamespace(
    e2m1_decode=e2m1_decode, e2m1_encode=e2m1_encode, e4m3_decode=e4m3_decode,
    e4m3_encode_nonneg=e4m3_encode_nonneg, pack_nibbles=pack_nibbles,
    unpack_nibbles=unpack_nibbles, unpack_weight_k=unpack_weight_k, global_scale=global_scale,
    quantize_rows=quantize_rows, dequantize_rows=dequantize_rows,
    quantize_weight=quantize_weight, dequantize_weight=dequantize_weight,
    round_to_bf16=round_to_bf16, backend="cpp")


# -------------------------------------------------------------- moe ----
TILE_ROWS = 128


def route(topk_ids, E):
    ids = _c(topk_ids, np.int32)
    T, k = ids.shape
    S = T * k
    counts = np.empty(E, np.int64)
    offsets = np.empty(E + 1, np.int64)
    slot_flat = np.empty(S, np.int64)
    slot_of = np.empty(S, np.int64)
    if lib().nvo_route(_p(ids), T, k, E, _p(counts), _p(offsets), _p(slot_flat), _p(slot_of)):
        raise ValueError("expert id out of range")
    return dict(counts=counts, offsets=offsets, slot_token=slot_flat // k, slot_flat=slot_flat,
                slot_of=slot_of)


def padded_layout(r, tile_rows=TILE_ROWS):
    counts, offsets = _c(r["counts"], np.int64), _c(r["offsets"], np.int64)
    slot_token, slot_of = _c(r["slot_token"], np.int64), _c(r["slot_of"], np.int64)
    E, S = counts.size, slot_of.size
    row_offsets = np.empty(E + 1, np.int64)
    row_of = np.empty(S, np.int64)
    rows = int(sum(-(-int(c) // tile_rows) * tile_rows for c in counts))
    row_token = np.empty(rows, np.int64)
    # the C++ call maps dense slot -> token as slot_flat // k; with the
    # tokens themselves as "flat indices" k is 1
    lib().nvo_padded_layout(_p(counts), _p(offsets), _p(slot_token), _p(slot_of), S, E, 1,
                            tile_rows, _p(row_offsets), _p(row_of), _p(row_token), rows)
    return dict(row_offsets=row_offsets, row_token=row_token, row_of=row_of)


def block_scaled_matmul(a_q, a_sf, w_q, w_sf):
    a_q, a_sf, w_q, w_sf = (_c(t, np.uint8) for t in (a_q, a_sf, w_q, w_sf))
    M, K, N = a_q.shape[0], 2 * a_q.shape[1], w_q.shape[1]
    out = np.empty((M, N), np.float64)
    lib().nvo_block_scaled_matmul(_p(a_q), _p(a_sf), M, K, _p(w_q), _p(w_sf), N, _p(out))
    return out


def silu(x):
    x = np.asarray(x, np.float64)
    f = np.vectorize(lambda v: lib().nvo_silu(float(v)), otypes=[np.float64])
    return f(x) if x.size else x.copy()


def swiglu(l1):
    l1 = _c(l1, np.float64)
    S, I2 = l1.shape
    h = np.empty((S, I2 // 2), np.float32)
    lib().nvo_swiglu(_p(l1), S, I2 // 2, _p(h))
    return h


def expert_l1(a_q, a_sf, gs_a, w1_q, w1_sf, gs_w1):
    acc = block_scaled_matmul(a_q, a_sf, w1_q, w1_sf)
    g = np.atleast_1d(np.asarray(gs_w1, dtype=np.float32))
    ga = float(np.float32(gs_a))
    if g.size == 1:
        return acc * (ga * float(g[0]))
    I = acc.shape[1] // 2
    out = np.empty_like(acc)
    out[:, :I] = acc[:, :I] * (ga * float(g[0]))
    out[:, I:] = acc[:, I:] * (ga * float(g[1]))
    return out


def expert_l2(h_q, h_sf, gs_h, w2_q, w2_sf, gs_w2):
    return block_scaled_matmul(h_q, h_sf, w2_q, w2_sf) * (float(np.float32(gs_h)) *
                                                          float(np.float32(gs_w2)))


def unpermute_reduce(slot_out, slot_of, topk_w):
    so = _c(slot_out, np.float64)
    w = _c(topk_w, np.float64)
    T, k = w.shape
    sl = _c(np.asarray(slot_of).reshape(-1), np.int64)
    y = np.empty((T, so.shape[1]), np.float64)
    lib().nvo_unpermute_reduce(_p(so), so.shape[1], _p(sl), _p(w), T, k, _p(y))
    return y


def quantize_expert_weights(w_list, split_halves=False):
    qs, sfs, gss = [], [], []
    for w in w_list:
        if split_halves:
            n = w.shape[1] // 2
            qg, sfg, gg = quantize_weight(w[:, :n])
            qu, sfu, gu = quantize_weight(w[:, n:])
            qs.append(np.concatenate([qg, qu], 1))
            sfs.append(np.concatenate([sfg, sfu], 1))
            gss.append((gg, gu))
        else:
            q, sf, g = quantize_weight(w)
            qs.append(q)
            sfs.append(sf)
            gss.append(g)
    return np.stack(qs), np.stack(sfs), np.array(gss, dtype=np.float32)


def forward(x, topk_ids, topk_w, w1_q, w1_sf, gs_w1, w2_q, w2_sf, gs_w2,
            expert_subset=None, gs_mid=None):
    """Same arguments and results as the numpy oracle's forward (plus
    "seconds": the wall time of the C++ pass itself).  w1_q / w2_q may be
    callables e -> (q, sf); the C++ pass then gets every expert that receives
    a slot (the others are never read and are given as zeros)."""
    x = _c(x, np.float32)
    T, H = x.shape
    ids = _c(topk_ids, np.int32)
    k = ids.shape[1]
    gs1 = np.asarray(gs_w1, np.float32)
    E = gs1.shape[0]
    split = gs1.ndim == 2
    used = sorted(set(ids.reshape(-1).tolist()))

    def stack(wq, wsf, shape_q, shape_sf):
        if not callable(wq):
            return _c(wq, np.uint8), _c(wsf, np.uint8)
        q0, s0 = wq(used[0])
        Q = np.zeros((E,) + q0.shape, np.uint8)
        SF = np.zeros((E,) + s0.shape, np.uint8)
        for e in used:
            Q[e], SF[e] = wq(e)
        return Q, SF

    W1q, W1sf = stack(w1_q, w1_sf, None, None)
    W2q, W2sf = stack(w2_q, w2_sf, None, None)
    I = W1q.shape[-1] // 2
    S = T * k
    l1 = np.empty((S, 2 * I), np.float64)
    h = np.empty((S, I), np.float32)
    hq = np.empty((S, I // 2), np.uint8)
    hsf = np.empty((S, I // 16), np.uint8)
    out2 = np.empty((S, H), np.float64)
    y64 = np.empty((T, H), np.float64)
    slot_of = np.empty(S, np.int64)
    gs_h = ctypes.c_float(0.0)
    gs_x = ctypes.c_float(0.0)
    mid = None if gs_mid is None else _c(gs_mid, np.float32)
    t0 = time.perf_counter()
    st = lib().nvo_forward(_p(x), T, H, _p(ids), _p(_c(topk_w, np.float32)), k, E, I,
                           _p(W1q), _p(W1sf), _p(_c(gs1, np.float32)), 1 if split else 0,
                           _p(W2q), _p(W2sf), _p(_c(gs_w2, np.float32)), _p(mid),
                           _p(l1), _p(h), _p(hq), _p(hsf), ctypes.addressof(gs_h),
                           ctypes.addressof(gs_x), _p(out2), _p(y64), _p(slot_of))
    seconds = time.perf_counter() - t0
    if st:
        raise ValueError("expert id out of range")
    r = route(ids, E)
    xq, xsf, gx = quantize_rows(x)
    return dict(route=r, xq=xq, xsf=xsf, gs_x=np.float32(gs_x.value), l1=l1, h=h, hq=hq,
                hsf=hsf, gs_h=None if gs_mid is not None else np.float32(gs_h.value),
                gs_mid=gs_mid, out2=out2, y64=y64, y_bf16=round_to_bf16(y64),
                seconds=seconds)


def cosine(a, b):
    a = np.asarray(a, dtype=np.float64).ravel()
    b = np.asarray(b, dtype=np.float64).ravel()
    na, nb = math.sqrt(float(a @ a)), math.sqrt(float(b @ b))
    if na == 0 or nb == 0:
        return 1.0 if na == nb else 0.0
    return float(a @ b) / (na * nb)


moe = types.SimpleNamespace(
    route=route, padded_layout=padded_layout, block_scaled_matmul=block_scaled_matmul,
    silu=silu, swiglu=swiglu, expert_l1=expert_l1, expert_l2=expert_l2,
    unpermute_reduce=unpermute_reduce, quantize_expert_weights=quantize_expert_weights,
    forward=forward, cosine=cosine, TILE_ROWS=TILE_ROWS, backend="cpp")
