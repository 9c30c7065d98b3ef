"""The allocation-free routing entry point (moe_route_permute_noalloc).

Some callers cannot give the library a device workspace: a serving engine
that has reserved all of HBM for its own pools, or a plug-in host that owns
every allocation, may not call cudaMalloc (which also synchronises the
device).  For them the routing permutation keeps its per-chunk histograms in
a fixed array inside the library.  These tests call that entry point through
the C ABI and check it against the workspace version, bit for bit, on two
calls in a row (the array keeps the previous call's contents), for a
single-chunk and a many-chunk input; and that inputs too large for the array
are refused before anything runs.  This file is collected last so that a run
stopping at the first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

from nvfp4_block_scaled_route_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module")
def nb():
    import __graft_entry__
    __graft_entry__.build()
    from nvfp4_block_scaled_route_gb300 import binding
    return binding


def noalloc_route(nb, ids, E):
    T, k = ids.shape
    rows = nb.rows_bound(T, k, E)
    out = dict(offsets=torch.full((E + 1,), -7, dtype=torch.int32, device=DEV),
               counts=torch.full((E,), -7, dtype=torch.int32, device=DEV),
               row_token=torch.full((max(rows, 1),), -7, dtype=torch.int32, device=DEV),
               slot_of=torch.full((max(T * k, 1),), -7, dtype=torch.int32, device=DEV))
    st = nb.lib().moe_route_permute_noalloc(
        ids.data_ptr(), T, k, E, out["offsets"].data_ptr(), out["counts"].data_ptr(),
        out["row_token"].data_ptr(), out["slot_of"].data_ptr(),
        torch.cuda.current_stream().cuda_stream)
    assert st == 0, nb.lib().nvmoe_status_str(st)
    torch.cuda.synchronize()
    return out, rows


@pytest.mark.parametrize("name", ["decode1", "prefill16k"])
def test_noalloc_route_matches_workspace_route(nb, name):
    cfg = syn.CONFIGS[name]
    ids, _ = syn.draw_routing(cfg)
    ids = ids.to(DEV)
    ref = nb.route_permute(ids, cfg.E)
    torch.cuda.synchronize()
    S = cfg.T * cfg.k
    for _ in range(2):                      # two calls in a row share the array
        got, rows = noalloc_route(nb, ids, cfg.E)
        assert rows == ref.rows
        assert torch.equal(got["offsets"], ref.expert_offsets)
        assert torch.equal(got["counts"], ref.expert_counts)
        assert torch.equal(got["row_token"][:rows], ref.row_token[:rows])
        assert torch.equal(got["slot_of"][:S], ref.slot_of[:S])


def test_noalloc_route_refuses_inputs_beyond_its_array(nb):
    E, k = 256, 32
    T = 65536                               # 512 chunks x 256 experts > 65536 words
    ids = torch.zeros((1, 1), dtype=torch.int32, device=DEV)   # never read: refused first
    buf = torch.zeros(16, dtype=torch.int32, device=DEV)
    st = nb.lib().moe_route_permute_noalloc(ids.data_ptr(), T, k, E, buf.data_ptr(),
                                            buf.data_ptr(), buf.data_ptr(), buf.data_ptr(),
                                            torch.cuda.current_stream().cuda_stream)
    assert st == 2                          # NVMOE_ERR_UNSUPPORTED_SHAPE
    assert torch.count_nonzero(buf) == 0
