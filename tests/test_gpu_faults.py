"""Faults detected on the device are reported, not trapped: the kernel
records a status code in the workspace's status word, returns, and the
context stays usable.  Each case makes the fault on purpose from the host
side, with no bad address, trap or endless wait:

  * an expert id outside [0, E) in topk_ids: the routing permutation drops
    that (token, choice) (slot_of = -1), reports NVMOE_ERR_DEVICE_BAD_INDEX,
    and places every other entry exactly as the oracle does for the valid
    entries alone;
  * an activation-ready flag that nothing sets: the L1 kernel's wait for it
    runs out after the caller's limit (a few ms), NVMOE_ERR_TIMEOUT is
    reported, and once the flag is set the same workspace gives the same
    bits as a call without the flag.  The wait comes before the kernel's
    first load, so no copy is in flight when the kernel unwinds.
"""
import numpy as np
import pytest
import torch

from oracle.cpp import moe as omoe
from nvfp4_block_scaled_route_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu

DEV = "cuda"
ERR_TIMEOUT, ERR_BAD_INDEX, ERR_INVALID_ARG = 6, 7, 1


@pytest.fixture(scope="module")
def nb():
    import __graft_entry__
    __graft_entry__.build()
    from nvfp4_block_scaled_route_gb300 import binding
    return binding


@pytest.mark.parametrize("name", ["decode64", "prefill4k"])   # one chunk / several chunks
def test_route_bad_expert_id_is_dropped_and_reported(nb, name):
    cfg = syn.CONFIGS[name]
    ids, _ = syn.draw_routing(cfg)
    T, k, E = cfg.T, cfg.k, cfg.E
    bad = [(3, 2, E), (T // 2, k - 1, -1), (T - 1, 0, E + 1000)]
    for t, j, v in bad:
        ids[t, j] = v
    ws = nb._workspace(nb.lib().moe_route_workspace_size(T, k, E), DEV)
    r = nb.route_permute(ids.to(DEV), E, ws=ws)
    torch.cuda.synchronize()
    assert nb.read_status(ws) == ERR_BAD_INDEX

    flat = ids.numpy().reshape(-1).astype(np.int64)
    valid = (flat >= 0) & (flat < E)
    # the oracle's permutation of the valid entries alone (their order, and so
    # every stable rank, is that of the full list with the bad ones removed)
    ref = omoe.route(flat[valid].reshape(-1, 1), E)
    lay = omoe.padded_layout(ref)
    slot_of = r.slot_of.cpu().numpy()[:T * k]
    assert np.all(slot_of[~valid] == -1)
    assert np.array_equal(slot_of[valid], lay["row_of"])
    assert np.array_equal(r.expert_counts.cpu().numpy(), ref["counts"])
    assert np.array_equal(r.expert_offsets.cpu().numpy(), lay["row_offsets"])
    row_token = r.row_token.cpu().numpy()
    want = np.full(r.rows, -1, dtype=np.int64)
    want[lay["row_of"]] = np.nonzero(valid)[0] // k
    assert np.array_equal(row_token[:r.rows], want)

    # the status word clears, and a clean input then reports nothing
    assert nb.lib().nvmoe_clear_status(nb._ptr(ws), nb._stream()) == 0
    ids_ok, _ = syn.draw_routing(cfg)
    nb.route_permute(ids_ok.to(DEV), E, ws=ws)
    torch.cuda.synchronize()
    assert nb.read_status(ws) == 0


def _layer(nb, cfg):
    W1 = torch.stack([syn.draw_weight(cfg, 1, e) for e in range(cfg.E)]).to(DEV)
    W2 = torch.stack([syn.draw_weight(cfg, 2, e) for e in range(cfg.E)]).to(DEV)
    q1, s1, g1 = nb.quantize_weights(W1)
    q2, s2, g2 = nb.quantize_weights(W2)
    return nb.PreparedWeights.from_checkpoint(q1, s1, g1, q2, s2, g2)


@pytest.mark.parametrize("path", [1, 2], ids=["separate", "fused"])
def test_ready_flag_wait_runs_out(nb, path):
    cfg = syn.CONFIGS["small"]
    pw = _layer(nb, cfg)
    x = syn.draw_activations(cfg).to(DEV)
    ids, w = syn.draw_routing(cfg)
    ids, w = ids.to(DEV), w.to(DEV)

    ref_layer = nb.MoELayer(pw, cfg.T, cfg.k, device=DEV, out_dtype=torch.float32)
    y_ref = ref_layer.forward(x, ids, w, taps={"path": path}).clone()
    torch.cuda.synchronize()
    assert ref_layer.status() == 0

    layer = nb.MoELayer(pw, cfg.T, cfg.k, device=DEV, out_dtype=torch.float32)
    flag = torch.zeros(4, dtype=torch.int32, device=DEV)
    taps = {"path": path, "ready_flag": flag, "ready_value": 1, "ready_wait_us": 5000}
    layer.forward(x, ids, w, taps=taps)
    torch.cuda.synchronize()
    assert nb.read_status(layer.ws_fwd) == ERR_TIMEOUT

    # the context and the workspace stay usable
    assert nb.lib().nvmoe_clear_status(nb._ptr(layer.ws_fwd), nb._stream()) == 0
    flag.fill_(1)
    y = layer.forward(x, ids, w, taps=taps)
    torch.cuda.synchronize()
    assert layer.status() == 0
    assert torch.equal(y, y_ref)


def test_layer_forward_rejects_ready_flag(nb):
    cfg = syn.CONFIGS["tiny"]
    pw = _layer(nb, cfg)
    x = syn.draw_activations(cfg).to(DEV)
    ids, w = syn.draw_routing(cfg)
    layer = nb.FusedLayer(pw, cfg.T, cfg.k, device=DEV)
    flag = torch.ones(4, dtype=torch.int32, device=DEV)
    with pytest.raises(nb.NvmoeError) as e:
        layer.forward(x, ids.to(DEV), w.to(DEV), taps={"ready_flag": flag, "ready_value": 1})
    assert e.value.status == ERR_INVALID_ARG


def test_layer_kernel_bad_expert_ids(nb):
    """The single-kernel layer with expert ids outside [0, E): the dropped
    choices take no part in the top-k reduce, exactly as in the four-call
    path (the same bits of y), a token none of whose choices is valid gets
    y = 0, and the status word reports NVMOE_ERR_DEVICE_BAD_INDEX."""
    cfg = syn.MoEConfig("layer_bad", E=8, H=512, I=256, T=6, k=4, routing="uniform")
    pw = _layer(nb, cfg)
    x = syn.draw_activations(cfg).to(DEV)
    ids, w = syn.draw_routing(cfg)
    ids[1, 2] = cfg.E + 1
    ids[4, :] = -1
    ids, w = ids.to(DEV), w.to(DEV)
    fl = nb.FusedLayer(pw, cfg.T, cfg.k, device=DEV, out_dtype=torch.float32)
    fl.y.fill_(7.0)
    outs = []
    for _ in range(2):               # the self-clearing counters, once more
        y = fl.forward(x, ids, w, taps={"path": nb.PATH_LAYER}).clone()
        torch.cuda.synchronize()
        outs.append(y.cpu())
    assert nb.read_status(fl.ws) == ERR_BAD_INDEX
    assert torch.equal(outs[0], outs[1])
    ref = nb.MoELayer(pw, cfg.T, cfg.k, device=DEV, out_dtype=torch.float32)
    y_ref = ref.forward(x, ids, w, taps={"path": nb.PATH_SEPARATE}).cpu()
    torch.cuda.synchronize()
    assert torch.equal(outs[1], y_ref)
    assert torch.all(outs[1][4] == 0)
    assert torch.all(outs[1][1] != 7.0)
