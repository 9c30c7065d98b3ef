"""Thin ctypes binding of libnvfp4moe.so (argument marshalling only).

Every computation runs in the library's CUDA kernels; this module allocates
device buffers with PyTorch, passes raw pointers and the current CUDA stream,
and turns nonzero status codes into exceptions.  There is no fallback: if
the library is missing or was not built, ``lib()`` raises.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional

import torch

PKG = os.path.dirname(os.path.abspath(__file__))
# NVMOE_LIBRARY=debug loads the debug-bounds build (in-kernel index checks
# that record NVMOE_ERR_DEVICE_BOUNDS instead of touching memory out of range)
LIB_PATH = os.path.join(PKG, "libnvfp4moe_debug.so" if os.environ.get("NVMOE_LIBRARY") == "debug"
                        else "libnvfp4moe.so")

BF16, F32, F16 = 0, 1, 2
NVMOE_ERR_CUDA = 5
TILE_ROWS = 128

_lib = None


class NvmoeError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        msg = lib().nvmoe_status_str(status).decode() if _lib is not None else str(status)
        if status == NVMOE_ERR_CUDA and _lib is not None:
            msg += f" [{lib().nvmoe_last_cuda_error().decode()}]"
        super().__init__(f"{fn} failed: {msg} (status {status})")


class Weights(ctypes.Structure):
    _fields_ = [("E", ctypes.c_int), ("H", ctypes.c_int), ("I", ctypes.c_int),
                ("w1", ctypes.c_void_p), ("w1_sf", ctypes.c_void_p), ("gs_w1", ctypes.c_void_p),
                ("w2", ctypes.c_void_p), ("w2_sf", ctypes.c_void_p), ("gs_w2", ctypes.c_void_p),
                ("gs_w1_up", ctypes.c_void_p), ("gs_mid", ctypes.c_void_p)]


class Taps(ctypes.Structure):
    _fields_ = [("l1_out", ctypes.c_void_p), ("h", ctypes.c_void_p), ("hq", ctypes.c_void_p),
                ("hsf_mma", ctypes.c_void_p), ("gs_h", ctypes.c_void_p),
                ("stage_events", ctypes.c_void_p * 4), ("path", ctypes.c_int),
                ("slot_of", ctypes.c_void_p), ("ready_flag", ctypes.c_void_p),
                ("ready_value", ctypes.c_int), ("ready_wait_us", ctypes.c_int)]


PATH_AUTO, PATH_SEPARATE, PATH_FUSED, PATH_LAYER, PATH_SEPARATE_SINGLE = 0, 1, 2, 3, 4


# name -> (restype, argtypes)
_P, _I, _I64, _SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
SIGNATURES = {
    "nvmoe_status_str": (ctypes.c_char_p, [_I]),
    "nvmoe_last_cuda_error": (ctypes.c_char_p, []),
    "nvmoe_version": (_I, []),
    "nvmoe_set_pdl": (_I, [_I]),
    "nvmoe_kernel_launch_count": (ctypes.c_uint64, []),
    "nvmoe_read_status": (_I, [_P, _P, ctypes.POINTER(ctypes.c_int)]),
    "nvmoe_clear_status": (_I, [_P, _P]),
    "nvfp4_sf_mma_bytes": (_SZ, [_I64, _I64]),
    "nvmoe_fp4_mma_probe": (_I, [_I, _I, _I, _P, _P, _SZ, _P]),
    "moe_route_rows_bound": (_I64, [_I64, _I, _I]),
    "moe_route_workspace_size": (_SZ, [_I64, _I, _I]),
    "moe_route_permute": (_I, [_P, _I64, _I, _I, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_route_permute_noalloc": (_I, [_P, _I64, _I, _I, _P, _P, _P, _P, _P]),
    "nvfp4_quantize_workspace_size": (_SZ, [_I64, _I64]),
    "nvfp4_quantize_act": (_I, [_P, _I, _I64, _I64, _P, _I, _I64, _P, _P, _P, _P, _P, _SZ, _P]),
    "nvfp4_quantize_weights_workspace_size": (_SZ, [_I, _I, _I]),
    "nvfp4_quantize_weights": (_I, [_P, _I, _I, _I, _P, _P, _P, _P, _SZ, _P]),
    "moe_nvfp4_prepared_bytes": (_SZ, [_I, _I, _I]),
    "moe_nvfp4_prepare_weights": (_I, [_P, _P, _I, _I, _I, _P, _P, _P]),
    "moe_nvfp4_workspace_size": (_SZ, [_I64, _I, _I, _I, _I]),
    "moe_nvfp4_forward": (_I, [ctypes.POINTER(Weights), _P, _P, _P, _P, _P, _P, _I64, _I, _P,
                               _I, ctypes.POINTER(Taps), _P, _SZ, _P]),
    "moe_unpermute_reduce": (_I, [_P, _I, _P, _P, _I64, _I, _I64, _P, _I, _P]),
    "moe_router_workspace_size": (_SZ, [_I64, _I, _I]),
    "moe_router_topk": (_I, [_P, _P, _I64, _I, _I, _I, _I, _P, _P, _P, _SZ, _P]),
    "moe_nvfp4_forward_phase": (_I, [ctypes.POINTER(Weights), _P, _P, _P, _P, _P, _P, _I64, _I,
                                     _P, _I, _I, _P, ctypes.POINTER(Taps), _P, _SZ, _P]),
    "nvfp4_amax": (_I, [_P, _I, _I64, _I64, _P, _P, _SZ, _P]),
    "nvfp4_quantize_act_amax": (_I, [_P, _I, _I64, _I64, _P, _I, _I64, _P, _P, _P, _P, _P, _P]),
    "moe_ep_dispatch_workspace_size": (_SZ, [_I64, _I, _I]),
    "moe_ep_dispatch": (_I, [_P, _I64, _I, _I, _I, _P, _P, _I, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_ep_scatter": (_I, [_P, _I64, _I, _P, _I64, _P, _P, _P, _P]),
    "moe_ep_gather": (_I, [_P, _I, _I, _I64, _P, _I64, _P, _P, _P]),
    "moe_nvfp4_layer_workspace_size": (_SZ, [_I64, _I, _I, _I, _I]),
    "moe_nvfp4_layer_forward": (_I, [ctypes.POINTER(Weights), _P, _I, _P, _P, _I64, _I, _P, _I,
                                     ctypes.POINTER(Taps), _P, _SZ, _P]),
}


def lib():
    """Load libnvfp4moe.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: run __graft_entry__.build() first")
        l = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(l, name)
            f.restype = res
            f.argtypes = args
        _lib = l
    return _lib


def _check(fn: str, status: int):
    if status != 0:
        raise NvmoeError(fn, status)


def _ptr(t: Optional[torch.Tensor]):
    """Device address of a tensor's data.  The library reads and writes
    every buffer as dense row-major memory, so a tensor with other strides
    (a transposed or sliced view) is refused rather than passed as if it
    were dense."""
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor (the library reads dense row-major memory)")
    return t.data_ptr()


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def sf_mma_bytes(rows: int, cols: int) -> int:
    return int(lib().nvfp4_sf_mma_bytes(rows, cols))


def rows_bound(T: int, k: int, E: int) -> int:
    return int(lib().moe_route_rows_bound(T, k, E))


def _workspace(nbytes: int, device) -> torch.Tensor:
    ws = torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device)
    return ws


def read_status(ws: torch.Tensor, stream=None) -> int:
    out = ctypes.c_int(0)
    _check("nvmoe_read_status", lib().nvmoe_read_status(_ptr(ws), _stream(stream), ctypes.byref(out)))
    return out.value


# ------------------------------------------------------------ measurement --
PROBE_PAIR, PROBE_N128, PROBE_CP32, PROBE_CP256 = 1, 2, 4, 8


def fp4_mma_probe(variant: int, iters: int, grid: int, repeats: int = 3, device=None,
                  stream=None):
    """Dense NVFP4 tensor-core throughput (nvmoe_fp4_mma_probe).

    Runs the probe `repeats` times on `stream`, each launch timed with CUDA
    events on that stream.  Returns a dict: best-launch TFLOP/s, the median
    cycles per MMA of the issuing CTAs, the launch times (ms) and the status."""
    dev = torch.device(device if device is not None else "cuda")
    cycles = torch.zeros(grid, dtype=torch.int64, device=dev)
    ws = _workspace(256, dev)
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    N = 128 if variant & PROBE_N128 else 256
    flops = float(grid) * iters * 2.0 * 128 * N * 64
    ms = []
    with torch.cuda.stream(s):
        for _ in range(repeats):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(s)
            _check("nvmoe_fp4_mma_probe", lib().nvmoe_fp4_mma_probe(
                variant, iters, grid, _ptr(cycles), _ptr(ws), ws.numel(), s.cuda_stream))
            b.record(s)
            s.synchronize()
            ms.append(a.elapsed_time(b))
    c = cycles.cpu()
    c = c[c > 0].double()
    return {"variant": variant, "iters": iters, "grid": grid, "N": N,
            "tflops": flops / (min(ms) / 1e3) / 1e12, "ms": ms,
            "cycles_per_mma": float(c.median() / iters) if c.numel() else None,
            "status": read_status(ws)}


# ------------------------------------------------------------------ step 1 --
@dataclass
class Route:
    expert_offsets: torch.Tensor   # int32 [E+1]
    expert_counts: torch.Tensor    # int32 [E]
    row_token: torch.Tensor        # int32 [rows]
    slot_of: torch.Tensor          # int32 [T*k]
    rows: int                      # rows_bound
    T: int
    k: int
    E: int


def route_permute(topk_ids: torch.Tensor, E: int, ws: Optional[torch.Tensor] = None,
                  out: Optional[Route] = None, stream=None) -> Route:
    T, k = topk_ids.shape
    dev = topk_ids.device
    rows = rows_bound(T, k, E)
    if out is None:
        out = Route(torch.empty(E + 1, dtype=torch.int32, device=dev),
                    torch.empty(E, dtype=torch.int32, device=dev),
                    torch.empty(max(rows, 1), dtype=torch.int32, device=dev),
                    torch.empty(max(T * k, 1), dtype=torch.int32, device=dev), rows, T, k, E)
    need = int(lib().moe_route_workspace_size(T, k, E))
    if ws is None:
        ws = _workspace(need, dev)
    _check("moe_route_permute", lib().moe_route_permute(
        _ptr(topk_ids), T, k, E, _ptr(out.expert_offsets), _ptr(out.expert_counts),
        _ptr(out.row_token), _ptr(out.slot_of), _ptr(ws), ws.numel(), _stream(stream)))
    return out


# ------------------------------------------------------------------ step 2 --
def quantize_act(x: torch.Tensor, row_dst: Optional[torch.Tensor] = None, fanout: int = 1,
                 out_rows: Optional[int] = None, rowmajor_sf: bool = True, mma_sf: bool = True,
                 ws: Optional[torch.Tensor] = None, out=None, stream=None):
    """Returns (q [out_rows, cols/2] u8, sf_row [out_rows, cols/16] u8 or None,
    sf_mma (staged) u8 or None, gs [1] f32)."""
    assert x.dim() == 2 and x.is_contiguous()
    rows, cols = x.shape
    dtype = {torch.bfloat16: BF16, torch.float32: F32}[x.dtype]
    if out_rows is None:
        out_rows = rows
    dev = x.device
    if out is None:
        q = torch.empty((out_rows, cols // 2), dtype=torch.uint8, device=dev)
        sf_row = torch.empty((out_rows, cols // 16), dtype=torch.uint8, device=dev) if rowmajor_sf else None
        sf_mma = torch.zeros(sf_mma_bytes(out_rows, cols), dtype=torch.uint8, device=dev) if mma_sf else None
        gs = torch.empty(1, dtype=torch.float32, device=dev)
    else:
        q, sf_row, sf_mma, gs = out
    if ws is None:
        ws = _workspace(lib().nvfp4_quantize_workspace_size(rows, cols), dev)
    _check("nvfp4_quantize_act", lib().nvfp4_quantize_act(
        _ptr(x), dtype, rows, cols, _ptr(row_dst), fanout, out_rows, _ptr(q), _ptr(sf_row),
        _ptr(sf_mma), _ptr(gs), _ptr(ws), ws.numel(), _stream(stream)))
    return q, sf_row, sf_mma, gs


# ---------------------------------------------------------------- weights --
def quantize_weights(w: torch.Tensor, stream=None):
    """fp32 [E, K, N] -> checkpoint (q [E, K/2, N], sf [E, K/16, N], gs [E])."""
    E, K, N = w.shape
    dev = w.device
    q = torch.empty((E, K // 2, N), dtype=torch.uint8, device=dev)
    sf = torch.empty((E, K // 16, N), dtype=torch.uint8, device=dev)
    gs = torch.empty(E, dtype=torch.float32, device=dev)
    ws = _workspace(lib().nvfp4_quantize_weights_workspace_size(E, K, N), dev)
    _check("nvfp4_quantize_weights", lib().nvfp4_quantize_weights(
        _ptr(w), E, K, N, _ptr(q), _ptr(sf), _ptr(gs), _ptr(ws), ws.numel(), _stream(stream)))
    return q, sf, gs


def prepare_weights(q_ckpt: torch.Tensor, sf_ckpt: torch.Tensor, stream=None):
    """Checkpoint (E, K/2, N) + (E, K/16, N) -> (B tiles, staged sf)."""
    E, K2, N = q_ckpt.shape
    K = 2 * K2
    dev = q_ckpt.device
    q = torch.empty(int(lib().moe_nvfp4_prepared_bytes(E, K, N)), dtype=torch.uint8, device=dev)
    sf = torch.zeros(sf_mma_bytes(E * N, K), dtype=torch.uint8, device=dev)
    _check("moe_nvfp4_prepare_weights", lib().moe_nvfp4_prepare_weights(
        _ptr(q_ckpt), _ptr(sf_ckpt), E, K, N, _ptr(q), _ptr(sf), _stream(stream)))
    return q, sf


@dataclass
class PreparedWeights:
    E: int
    H: int
    I: int
    w1: torch.Tensor
    w1_sf: torch.Tensor
    gs_w1: torch.Tensor
    w2: torch.Tensor
    w2_sf: torch.Tensor
    gs_w2: torch.Tensor
    gs_w1_up: Optional[torch.Tensor] = None
    gs_mid: Optional[torch.Tensor] = None

    def struct(self) -> Weights:
        return Weights(self.E, self.H, self.I, _ptr(self.w1), _ptr(self.w1_sf), _ptr(self.gs_w1),
                       _ptr(self.w2), _ptr(self.w2_sf), _ptr(self.gs_w2), _ptr(self.gs_w1_up),
                       _ptr(self.gs_mid))

    @staticmethod
    def from_checkpoint(w1q, w1sf, gs1, w2q, w2sf, gs2, gs1_up=None,
                        gs_mid=None) -> "PreparedWeights":
        """w1q (E, H/2, 2I), w1sf (E, H/16, 2I), w2q (E, I/2, H), w2sf (E, I/16, H);
        gs1_up (E,) when the checkpoint quantised gate and up separately
        (then gs1 is the gate half's scale); gs_mid (E,) a static
        intermediate scale per expert (None: the dynamic global one)."""
        E, H2, N1 = w1q.shape
        q1, s1 = prepare_weights(w1q, w1sf)
        q2, s2 = prepare_weights(w2q, w2sf)
        return PreparedWeights(E, 2 * H2, N1 // 2, q1, s1, gs1.contiguous(), q2, s2,
                               gs2.contiguous(),
                               gs1_up.contiguous() if gs1_up is not None else None,
                               gs_mid.contiguous() if gs_mid is not None else None)

    def nbytes(self) -> int:
        ts = [self.w1, self.w1_sf, self.gs_w1, self.w2, self.w2_sf, self.gs_w2]
        for t in (self.gs_w1_up, self.gs_mid):
            if t is not None:
                ts.append(t)
        return sum(t.numel() * t.element_size() for t in ts)


# -------------------------------------------------------- router front end --
ROUTER_SELECTED, ROUTER_ALL = 0, 1


def router_topk(x: torch.Tensor, w_router: torch.Tensor, k: int, mode: int = ROUTER_SELECTED,
                ws: Optional[torch.Tensor] = None, stream=None):
    """bf16 x [T, H], bf16 w_router [E, H] -> (topk_ids int32 [T, k], topk_w float [T, k])."""
    T, H = x.shape
    E = w_router.shape[0]
    dev = x.device
    ids = torch.empty((T, k), dtype=torch.int32, device=dev)
    w = torch.empty((T, k), dtype=torch.float32, device=dev)
    if ws is None:
        ws = _workspace(lib().moe_router_workspace_size(T, H, E), dev)
    _check("moe_router_topk", lib().moe_router_topk(
        _ptr(x), _ptr(w_router), T, H, E, k, mode, _ptr(ids), _ptr(w), _ptr(ws), ws.numel(),
        _stream(stream)))
    return ids, w


# ------------------------------------------------------------- steps 3-6 --
def forward_workspace_bytes(T: int, k: int, E: int, H: int, I: int) -> int:
    return int(lib().moe_nvfp4_workspace_size(T, k, E, H, I))


def _taps(taps: Optional[dict]):
    if not taps:
        return None
    t = Taps(_ptr(taps.get("l1_out")), _ptr(taps.get("h")), _ptr(taps.get("hq")),
             _ptr(taps.get("hsf_mma")), _ptr(taps.get("gs_h")))
    evs = taps.get("stage_events")
    if evs is not None:
        # torch events are created on first record; their handles are plain
        # CUDA event handles
        for i, ev in enumerate(evs):
            if ev.cuda_event == 0:
                ev.record()
            t.stage_events[i] = ev.cuda_event
    t.path = int(taps.get("path", PATH_AUTO))
    t.slot_of = _ptr(taps.get("slot_of"))
    t.ready_flag = _ptr(taps.get("ready_flag"))
    t.ready_value = int(taps.get("ready_value", 0))
    t.ready_wait_us = int(taps.get("ready_wait_us", 0))
    return t


def nvfp4_forward(weights: PreparedWeights, xq: torch.Tensor, xsf_mma: torch.Tensor,
                  gs_x: torch.Tensor, route: Route, slot_out: Optional[torch.Tensor] = None,
                  taps: Optional[dict] = None, ws: Optional[torch.Tensor] = None, stream=None):
    dev = xq.device
    if slot_out is None:
        slot_out = torch.empty((route.rows, weights.H), dtype=torch.float32, device=dev)
    if ws is None:
        ws = _workspace(forward_workspace_bytes(route.T, route.k, weights.E, weights.H,
                                                weights.I), dev)
    t = _taps(taps)
    wst = weights.struct()
    code = {torch.bfloat16: BF16, torch.float32: F32, torch.float16: F16}[slot_out.dtype]
    _check("moe_nvfp4_forward", lib().moe_nvfp4_forward(
        ctypes.byref(wst), _ptr(xq), _ptr(xsf_mma), _ptr(gs_x), _ptr(route.expert_offsets),
        _ptr(route.expert_counts), _ptr(route.row_token), route.T, route.k, _ptr(slot_out),
        code, ctypes.byref(t) if t is not None else None, _ptr(ws), ws.numel(),
        _stream(stream)))
    return slot_out


def nvfp4_forward_phase(weights: PreparedWeights, xq: torch.Tensor, xsf_mma: torch.Tensor,
                        gs_x: torch.Tensor, route: Route, phase: int, amax_h: torch.Tensor,
                        slot_out: torch.Tensor, ws: torch.Tensor, taps: Optional[dict] = None,
                        stream=None):
    """moe_nvfp4_forward_phase: phase 1 (L1, *amax_h = max |h|) or 2
    (requantise with *amax_h, L2 into slot_out); same arguments and ws."""
    t = _taps(taps)
    wst = weights.struct()
    code = {torch.bfloat16: BF16, torch.float32: F32, torch.float16: F16}[slot_out.dtype]
    _check("moe_nvfp4_forward_phase", lib().moe_nvfp4_forward_phase(
        ctypes.byref(wst), _ptr(xq), _ptr(xsf_mma), _ptr(gs_x), _ptr(route.expert_offsets),
        _ptr(route.expert_counts), _ptr(route.row_token), route.T, route.k, _ptr(slot_out),
        code, phase, _ptr(amax_h), ctypes.byref(t) if t is not None else None, _ptr(ws),
        ws.numel(), _stream(stream)))
    return slot_out


# ------------------------------------------------------- expert parallel --
def amax(x: torch.Tensor, ws: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None,
         stream=None) -> torch.Tensor:
    """max |x| of a 2-D bf16/fp32 tensor as a float32 [1] device tensor."""
    assert x.dim() == 2 and x.is_contiguous()
    rows, cols = x.shape
    dtype = {torch.bfloat16: BF16, torch.float32: F32}[x.dtype]
    if out is None:
        out = torch.empty(1, dtype=torch.float32, device=x.device)
    if ws is None:
        ws = _workspace(lib().nvfp4_quantize_workspace_size(rows, cols), x.device)
    _check("nvfp4_amax", lib().nvfp4_amax(_ptr(x), dtype, rows, cols, _ptr(out), _ptr(ws),
                                          ws.numel(), _stream(stream)))
    return out


def quantize_act_amax(x: torch.Tensor, amax_in: torch.Tensor, row_dst=None, fanout: int = 1,
                      out_rows: Optional[int] = None, rowmajor_sf: bool = True,
                      mma_sf: bool = False, stream=None):
    """quantize_act with the amax given (float32 [1] device tensor)."""
    assert x.dim() == 2 and x.is_contiguous()
    rows, cols = x.shape
    dtype = {torch.bfloat16: BF16, torch.float32: F32}[x.dtype]
    out_rows = rows if out_rows is None else out_rows
    dev = x.device
    q = torch.empty((out_rows, cols // 2), dtype=torch.uint8, device=dev)
    sf_row = torch.empty((out_rows, cols // 16), dtype=torch.uint8, device=dev) if rowmajor_sf else None
    sf_mma = torch.zeros(sf_mma_bytes(out_rows, cols), dtype=torch.uint8, device=dev) if mma_sf else None
    gs = torch.empty(1, dtype=torch.float32, device=dev)
    _check("nvfp4_quantize_act_amax", lib().nvfp4_quantize_act_amax(
        _ptr(x), dtype, rows, cols, _ptr(row_dst), fanout, out_rows, _ptr(amax_in), _ptr(q),
        _ptr(sf_row), _ptr(sf_mma), _ptr(gs), _stream(stream)))
    return q, sf_row, sf_mma, gs


def ep_dispatch(topk_ids: torch.Tensor, E: int, G: int, q_tok: torch.Tensor,
                sf_tok: torch.Tensor, ws: Optional[torch.Tensor] = None, stream=None):
    """moe_ep_dispatch -> (send_counts int32 [G], send_pos int32 [T*k],
    send_rows uint8 [T*k, H/2 + H/16], send_expert int32 [T*k], ws)."""
    T, k = topk_ids.shape
    H = q_tok.shape[1] * 2
    dev = topk_ids.device
    S = T * k
    counts = torch.zeros(G, dtype=torch.int32, device=dev)
    pos = torch.empty(max(S, 1), dtype=torch.int32, device=dev)
    rows = torch.empty((max(S, 1), H // 2 + H // 16), dtype=torch.uint8, device=dev)
    expert = torch.empty(max(S, 1), dtype=torch.int32, device=dev)
    if ws is None:
        ws = _workspace(lib().moe_ep_dispatch_workspace_size(T, k, G), dev)
    _check("moe_ep_dispatch", lib().moe_ep_dispatch(
        _ptr(topk_ids), T, k, E, G, _ptr(q_tok), _ptr(sf_tok), H, _ptr(counts), _ptr(pos),
        _ptr(rows), _ptr(expert), _ptr(ws), ws.numel(), _stream(stream)))
    return counts, pos[:S], rows[:S], expert[:S], ws


def ep_scatter(recv_rows: torch.Tensor, H: int, slot_of: torch.Tensor, out_rows: int,
               xq: torch.Tensor, xsf_mma: torch.Tensor, status: Optional[torch.Tensor] = None,
               stream=None):
    """status: optional int32 [1] device tensor (debug-bounds records)."""
    n = recv_rows.shape[0]
    _check("moe_ep_scatter", lib().moe_ep_scatter(
        _ptr(recv_rows) if n else None, n, H, _ptr(slot_of) if n else None, out_rows, _ptr(xq),
        _ptr(xsf_mma), _ptr(status), _stream(stream)))


def ep_gather(slot_out: torch.Tensor, slot_of: torch.Tensor, n: int,
              status: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    H = slot_out.shape[1]
    code = {torch.bfloat16: BF16, torch.float32: F32, torch.float16: F16}[slot_out.dtype]
    out = torch.empty((n, H), dtype=slot_out.dtype, device=slot_out.device)
    if n:
        _check("moe_ep_gather", lib().moe_ep_gather(_ptr(slot_out), code, H, slot_out.shape[0],
                                                    _ptr(slot_of), n, _ptr(out), _ptr(status),
                                                    _stream(stream)))
    return out


# ------------------------------------------------------------------ step 7 --
def unpermute_reduce(slot_out: torch.Tensor, slot_of: torch.Tensor, topk_w: torch.Tensor,
                     out_dtype=torch.bfloat16, y: Optional[torch.Tensor] = None, stream=None):
    T, k = topk_w.shape
    H = slot_out.shape[1]
    if y is None:
        y = torch.empty((T, H), dtype=out_dtype, device=slot_out.device)
    code = {torch.bfloat16: BF16, torch.float32: F32}[y.dtype]
    scode = {torch.bfloat16: BF16, torch.float32: F32, torch.float16: F16}[slot_out.dtype]
    _check("moe_unpermute_reduce", lib().moe_unpermute_reduce(
        _ptr(slot_out), scode, _ptr(slot_of), _ptr(topk_w), T, k, H, _ptr(y), code,
        _stream(stream)))
    return y


# -------------------------------------------------------- whole forward --
class MoELayer:
    """The four calls of one forward pass on preallocated buffers.

    ``forward(x, topk_ids, topk_w)`` runs route -> quantise (straight into
    the grouped slot layout) -> L1 / SiLU*up / requantise / L2 -> reduce on
    the current stream, with every buffer reused between calls (so it can be
    captured in a CUDA graph).
    """

    def __init__(self, weights: PreparedWeights, T: int, k: int, device="cuda",
                 out_dtype=torch.bfloat16, slot_dtype=torch.float32):
        self.w = weights
        self.T, self.k = T, k
        E, H, I = weights.E, weights.H, weights.I
        dev = torch.device(device)
        self.rows = rows_bound(T, k, E)
        self.route = Route(torch.empty(E + 1, dtype=torch.int32, device=dev),
                           torch.empty(E, dtype=torch.int32, device=dev),
                           torch.empty(max(self.rows, 1), dtype=torch.int32, device=dev),
                           torch.empty(max(T * k, 1), dtype=torch.int32, device=dev),
                           self.rows, T, k, E)
        self.ws_route = _workspace(lib().moe_route_workspace_size(T, k, E), dev)
        self.ws_quant = _workspace(lib().nvfp4_quantize_workspace_size(T, H), dev)
        self.ws_fwd = _workspace(forward_workspace_bytes(T, k, E, H, I), dev)
        self.xq = torch.zeros((max(self.rows, 1), H // 2), dtype=torch.uint8, device=dev)
        self.xsf = torch.zeros(max(sf_mma_bytes(self.rows, H), 16), dtype=torch.uint8, device=dev)
        self.gs_x = torch.zeros(1, dtype=torch.float32, device=dev)
        self.slot_out = torch.zeros((max(self.rows, 1), H), dtype=slot_dtype, device=dev)
        self.y = torch.empty((T, H), dtype=out_dtype, device=dev)

    def forward(self, x: torch.Tensor, topk_ids: torch.Tensor, topk_w: torch.Tensor,
                taps: Optional[dict] = None, stream=None) -> torch.Tensor:
        route_permute(topk_ids, self.w.E, ws=self.ws_route, out=self.route, stream=stream)
        quantize_act(x, row_dst=self.route.slot_of, fanout=self.k, out_rows=self.rows,
                     ws=self.ws_quant, out=(self.xq, None, self.xsf, self.gs_x), stream=stream)
        nvfp4_forward(self.w, self.xq, self.xsf, self.gs_x, self.route, slot_out=self.slot_out,
                      taps=taps, ws=self.ws_fwd, stream=stream)
        unpermute_reduce(self.slot_out, self.route.slot_of, topk_w, y=self.y, stream=stream)
        return self.y

    def status(self) -> int:
        for ws in (self.ws_route, self.ws_quant, self.ws_fwd):
            s = read_status(ws)
            if s:
                return s
        return 0


class FusedLayer:
    """The whole layer through one call (moe_nvfp4_layer_forward) on one
    preallocated workspace.  Small batches run as a single cooperative
    kernel; larger ones as route, quantise, forward and reduce launches."""

    def __init__(self, weights: PreparedWeights, T: int, k: int, device="cuda",
                 out_dtype=torch.bfloat16):
        self.w = weights
        self.T, self.k = T, k
        dev = torch.device(device)
        self.rows = rows_bound(T, k, weights.E)
        self.ws = _workspace(lib().moe_nvfp4_layer_workspace_size(T, k, weights.E, weights.H,
                                                                   weights.I), dev)
        self.y = torch.empty((T, weights.H), dtype=out_dtype, device=dev)
        self._w = weights.struct()

    def forward(self, x: torch.Tensor, topk_ids: torch.Tensor, topk_w: torch.Tensor,
                taps: Optional[dict] = None, stream=None,
                y: Optional[torch.Tensor] = None) -> torch.Tensor:
        """y: output [T, H] (default: the layer's own self.y), bf16 or fp32."""
        y = self.y if y is None else y
        xcode = {torch.bfloat16: BF16, torch.float32: F32}[x.dtype]
        ycode = {torch.bfloat16: BF16, torch.float32: F32}[y.dtype]
        if tuple(y.shape) != (self.T, self.w.H):
            raise ValueError(f"y must be [{self.T}, {self.w.H}]")
        t = _taps(taps)
        _check("moe_nvfp4_layer_forward", lib().moe_nvfp4_layer_forward(
            ctypes.byref(self._w), _ptr(x), xcode, _ptr(topk_ids), _ptr(topk_w), self.T, self.k,
            _ptr(y), ycode, ctypes.byref(t) if t is not None else None, _ptr(self.ws),
            self.ws.numel(), _stream(stream)))
        return y

    def staging(self, x_dtype=torch.bfloat16):
        """Pinned host buffers for a step's inputs (x, topk_ids, topk_w) in one
        allocation, with a device twin of the same layout, and a pinned host
        y: a step then moves its inputs in one host-to-device copy and y in
        one device-to-host copy (forward_staged).  Returns the host views
        (x, topk_ids, topk_w, y) to fill and read, and the device views
        (x, topk_ids, topk_w) that forward_staged passes to the layer."""
        T, k, H = self.T, self.k, self.w.H
        el = torch.tensor([], dtype=x_dtype).element_size()
        parts = [T * H * el, T * k * 4, T * k * 4]
        offs, o = [], 0
        for n in parts:
            offs.append(o)
            o += (n + 255) // 256 * 256
        dev = self.y.device
        host = torch.empty(max(o, 256), dtype=torch.uint8).pin_memory()
        devb = torch.empty(max(o, 256), dtype=torch.uint8, device=dev)

        def views(buf):
            return (buf[offs[0]:offs[0] + parts[0]].view(x_dtype).view(T, H),
                    buf[offs[1]:offs[1] + parts[1]].view(torch.int32).view(T, k),
                    buf[offs[2]:offs[2] + parts[2]].view(torch.float32).view(T, k))
        y_host = torch.empty(self.y.shape, dtype=self.y.dtype).pin_memory()
        self._stage = (host, devb, views(devb), y_host)
        return views(host) + (y_host,), views(devb)

    def forward_staged(self, stream=None, taps: Optional[dict] = None) -> torch.Tensor:
        """One step from the pinned staging buffers (staging()): inputs to the
        device in one copy, the layer, y back in one copy; all on `stream`.
        Returns the pinned host y (valid once the stream has reached it)."""
        host, devb, (x, ids, w), y_host = self._stage
        s = stream if stream is not None else torch.cuda.current_stream()
        with torch.cuda.stream(s):
            devb.copy_(host, non_blocking=True)
            self.forward(x, ids, w, taps=taps, stream=s)
            y_host.copy_(self.y, non_blocking=True)
        return y_host

    def status(self) -> int:
        return read_status(self.ws)


class StagedPipeline:
    """Steps of a FusedLayer fed from pinned host memory with the copies
    overlapped: `depth` slots, each a pinned host input block (x, topk_ids,
    topk_w in one allocation), its device twin, a device y and a pinned host
    y.  submit() enqueues one step on three streams -- the host-to-device
    copy of the slot's inputs (copy-in stream), the layer (compute stream),
    the device-to-host copy of its y (copy-out stream) -- ordered by per-slot
    events, so that step i's input copy and step i-1's readback overlap the
    layer of another step.  Every step still moves all of its own inputs in
    and its own y out.

    Host buffers of a slot may be refilled once input_consumed(slot) has
    completed, and the slot's host y read once output_ready(slot) has.
    The layer's workspace is used by one step at a time (compute stream)."""

    def __init__(self, layer: "FusedLayer", depth: int = 2, x_dtype=torch.bfloat16):
        if depth < 1:
            raise ValueError("depth must be >= 1")
        self.layer = layer
        self.depth = depth
        T, k, H = layer.T, layer.k, layer.w.H
        dev = layer.y.device
        el = torch.tensor([], dtype=x_dtype).element_size()
        parts = [T * H * el, T * k * 4, T * k * 4]
        offs, o = [], 0
        for n in parts:
            offs.append(o)
            o += (n + 255) // 256 * 256

        def views(buf):
            return (buf[offs[0]:offs[0] + parts[0]].view(x_dtype).view(T, H),
                    buf[offs[1]:offs[1] + parts[1]].view(torch.int32).view(T, k),
                    buf[offs[2]:offs[2] + parts[2]].view(torch.float32).view(T, k))
        self.host_in = [torch.empty(max(o, 256), dtype=torch.uint8).pin_memory()
                        for _ in range(depth)]
        self.dev_in = [torch.empty(max(o, 256), dtype=torch.uint8, device=dev)
                       for _ in range(depth)]
        self.host_views = [views(b) for b in self.host_in]
        self.dev_views = [views(b) for b in self.dev_in]
        self.dev_y = [torch.empty_like(layer.y) for _ in range(depth)]
        self.host_y = [torch.empty(layer.y.shape, dtype=layer.y.dtype).pin_memory()
                       for _ in range(depth)]
        self.s_in = torch.cuda.Stream(device=dev)
        self.s_comp = torch.cuda.Stream(device=dev)
        self.s_out = torch.cuda.Stream(device=dev)
        self.ev_in = [torch.cuda.Event() for _ in range(depth)]     # inputs on the device
        self.ev_comp = [torch.cuda.Event() for _ in range(depth)]   # layer done
        self.ev_out = [torch.cuda.Event() for _ in range(depth)]    # y on the host
        self.h2d_bytes = self.host_in[0].numel()
        self.d2h_bytes = self.host_y[0].numel() * self.host_y[0].element_size()
        self._n = 0

    def inputs(self, slot: int):
        """Host views (x, topk_ids, topk_w) of a slot, to be filled."""
        return self.host_views[slot]

    def output(self, slot: int) -> torch.Tensor:
        return self.host_y[slot]

    def input_consumed(self, slot: int) -> torch.cuda.Event:
        return self.ev_in[slot]

    def output_ready(self, slot: int) -> torch.cuda.Event:
        return self.ev_out[slot]

    def submit(self, slot: Optional[int] = None) -> int:
        """Enqueue one step on a slot (default: round-robin); returns it."""
        if slot is None:
            slot = self._n % self.depth
        self._n += 1
        x, ids, w = self.dev_views[slot]
        with torch.cuda.stream(self.s_in):
            self.s_in.wait_event(self.ev_comp[slot])        # the slot's last layer read it
            self.dev_in[slot].copy_(self.host_in[slot], non_blocking=True)
            self.ev_in[slot].record(self.s_in)
        with torch.cuda.stream(self.s_comp):
            self.s_comp.wait_event(self.ev_in[slot])
            self.s_comp.wait_event(self.ev_out[slot])       # the slot's last y was read out
            self.layer.forward(x, ids, w, stream=self.s_comp, y=self.dev_y[slot])
            self.ev_comp[slot].record(self.s_comp)
        with torch.cuda.stream(self.s_out):
            self.s_out.wait_event(self.ev_comp[slot])
            self.host_y[slot].copy_(self.dev_y[slot], non_blocking=True)
            self.ev_out[slot].record(self.s_out)
        return slot

    def synchronize(self):
        for s in (self.s_in, self.s_comp, self.s_out):
            s.synchronize()
