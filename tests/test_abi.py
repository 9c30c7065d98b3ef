"""The C-ABI library builds, loads without a GPU, exports every entry point
declared in include/*.h, and rejects bad arguments on the host before
touching the device."""
import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    from nvfp4_block_scaled_route_gb300 import binding
    return binding.lib()


def declared_functions():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\**\s*([a-z][a-z0-9_]*)\s*\(",
                             src, flags=re.M):
            names.append(m.group(1))
    return sorted(set(names))


def test_header_declares_the_four_pipeline_calls():
    names = declared_functions()
    for fn in ("moe_route_permute", "nvfp4_quantize_act", "moe_nvfp4_forward",
               "moe_unpermute_reduce"):
        assert fn in names


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 15
    for fn in names:
        assert hasattr(lib, fn), fn


def test_debug_bounds_library_exports_the_same_symbols(lib):
    """libnvfp4moe_debug.so (NVMOE_DEBUG_BOUNDS: in-kernel index checks) is
    built beside the library and loads without a GPU."""
    path = os.path.join(ROOT, "nvfp4_block_scaled_route_gb300", "libnvfp4moe_debug.so")
    dbg = ctypes.CDLL(path)
    for fn in declared_functions():
        assert hasattr(dbg, fn), fn
    dbg.nvmoe_status_str.restype = ctypes.c_char_p
    assert dbg.nvmoe_status_str(9) == b"index outside its buffer (debug-bounds build)"


def test_binding_signatures_cover_header(lib):
    from nvfp4_block_scaled_route_gb300 import binding
    assert set(declared_functions()) == set(binding.SIGNATURES)


def test_host_side_helpers(lib):
    assert lib.nvmoe_version() >= 100
    assert lib.nvmoe_status_str(0) == b"ok"
    assert lib.nvmoe_status_str(4) == b"workspace too small"
    assert lib.nvmoe_last_cuda_error() == b""
    # rows bound: S + min(E, S) * 127 rounded up to 128
    assert lib.moe_route_rows_bound(1, 8, 48) == 1024
    assert lib.moe_route_rows_bound(0, 8, 48) == 0
    assert lib.moe_route_rows_bound(16384, 8, 48) == 131072 + 48 * 128
    # staged scale bytes: rows and K padded to 128 and 256
    assert lib.nvfp4_sf_mma_bytes(1, 64) == 128 * 16
    assert lib.nvfp4_sf_mma_bytes(129, 7168) == 256 * 448
    assert lib.moe_nvfp4_workspace_size(1, 8, 48, 7168, 3072) > 1024 * 3072 * 4


def test_bad_arguments_are_rejected_on_the_host(lib):
    P = ctypes.c_void_p
    fake = P(1 << 20)  # never dereferenced: every call below fails its checks first
    # k out of range
    assert lib.moe_route_permute(fake, 4, 0, 8, fake, fake, fake, fake, fake, 1 << 20, None) == 1
    # E out of range
    assert lib.moe_route_permute(fake, 4, 2, 300, fake, fake, fake, fake, fake, 1 << 20, None) == 1
    # workspace too small
    assert lib.moe_route_permute(fake, 4, 2, 8, fake, fake, fake, fake, fake, 8, None) == 4
    # cols not a multiple of 64
    assert lib.nvfp4_quantize_act(fake, 0, 4, 48, None, 1, 4, fake, None, None, fake, fake,
                                  1 << 20, None) == 2
    # bad dtype
    assert lib.nvfp4_quantize_act(fake, 7, 4, 64, None, 1, 4, fake, None, None, fake, fake,
                                  1 << 20, None) == 1
    # misaligned activation pointer
    assert lib.nvfp4_quantize_act(P((1 << 20) + 4), 0, 4, 64, None, 1, 4, fake, None, None,
                                  fake, fake, 1 << 20, None) == 3
    # unsupported hidden size for the forward (H % 256 != 0)
    from nvfp4_block_scaled_route_gb300 import binding
    w = binding.Weights(4, 320, 128, 1 << 20, 1 << 20, 1 << 20, 1 << 20, 1 << 20, 1 << 20)
    assert lib.moe_nvfp4_forward(ctypes.byref(w), fake, fake, fake, fake, fake, fake, 1, 2,
                                 fake, 1, None, fake, 1 << 30, None) == 2
    # slot_out dtype other than bf16 / fp32
    w.H = 256
    assert lib.moe_nvfp4_forward(ctypes.byref(w), fake, fake, fake, fake, fake, fake, 1, 2,
                                 fake, 7, None, fake, 1 << 30, None) == 1
    # reduce: bad dtype, bad H
    assert lib.moe_unpermute_reduce(fake, 1, fake, fake, 2, 2, 64, fake, 5, None) == 1
    assert lib.moe_unpermute_reduce(fake, 3, fake, fake, 2, 2, 64, fake, 0, None) == 1
    assert lib.moe_unpermute_reduce(fake, 0, fake, fake, 2, 2, 60, fake, 0, None) == 2


def test_router_and_layer_arguments_are_rejected_on_the_host(lib):
    """The router and the one-call layer entry point fail their argument
    checks before anything is enqueued (no GPU needed)."""
    from nvfp4_block_scaled_route_gb300 import binding
    P = ctypes.c_void_p
    fake = P(1 << 20)  # never dereferenced
    big = 1 << 30
    sel = binding.ROUTER_SELECTED
    # router: k > E, k > 32, E > 256, bad softmax mode
    assert lib.moe_router_topk(fake, fake, 4, 256, 6, 7, sel, fake, fake, fake, big, None) == 1
    assert lib.moe_router_topk(fake, fake, 4, 256, 64, 33, sel, fake, fake, fake, big, None) == 1
    assert lib.moe_router_topk(fake, fake, 4, 256, 257, 8, sel, fake, fake, fake, big, None) == 1
    assert lib.moe_router_topk(fake, fake, 4, 256, 48, 8, 9, fake, fake, fake, big, None) == 1
    # router: H not a multiple of 128; T = 0 is a no-op
    assert lib.moe_router_topk(fake, fake, 4, 192, 48, 8, sel, fake, fake, fake, big, None) == 2
    assert lib.moe_router_topk(None, None, 0, 256, 48, 8, sel, None, None, None, 0, None) == 0
    # router: misaligned x, workspace too small
    assert lib.moe_router_topk(P((1 << 20) + 2), fake, 4, 256, 48, 8, sel, fake, fake, fake, big,
                               None) == 3
    assert lib.moe_router_topk(fake, fake, 4096, 7168, 48, 8, sel, fake, fake, fake, 16,
                               None) == 4
    assert lib.moe_router_workspace_size(4096, 7168, 48) > 16
    # layer: bad x / y dtype, unsupported H, null workspace, misaligned y,
    # workspace too small; T = 0 is a no-op
    w = binding.Weights(48, 7168, 3072, 1 << 20, 1 << 20, 1 << 20, 1 << 20, 1 << 20, 1 << 20)
    wh = binding.Weights(48, 7000, 3072, 1 << 20, 1 << 20, 1 << 20, 1 << 20, 1 << 20, 1 << 20)
    need = lib.moe_nvfp4_layer_workspace_size(1, 8, 48, 7168, 3072)
    assert need > lib.moe_nvfp4_workspace_size(1, 8, 48, 7168, 3072)
    args = lambda wt, xd, y, yd, ws, n: (ctypes.byref(wt), fake, xd, fake, fake, 1, 8, y, yd,
                                         None, ws, n, None)
    assert lib.moe_nvfp4_layer_forward(*args(w, 5, fake, 0, fake, need)) == 1
    assert lib.moe_nvfp4_layer_forward(*args(w, 0, fake, 9, fake, need)) == 1
    assert lib.moe_nvfp4_layer_forward(*args(wh, 0, fake, 0, fake, need)) == 2
    assert lib.moe_nvfp4_layer_forward(*args(w, 0, fake, 0, None, need)) == 1
    assert lib.moe_nvfp4_layer_forward(*args(w, 0, P((1 << 20) + 8), 0, fake, need)) == 3
    assert lib.moe_nvfp4_layer_forward(*args(w, 0, fake, 0, fake, need - 16)) == 4
    assert lib.moe_nvfp4_layer_forward(ctypes.byref(w), None, 0, None, None, 0, 8, None, 0, None,
                                       fake, lib.moe_nvfp4_layer_workspace_size(0, 8, 48, 7168,
                                                                                3072), None) == 0
