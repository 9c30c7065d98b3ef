"""Router front-end: the oracle against brute force and closed forms (CPU),
and the CUDA router (moe_router_topk, through the C ABI) against the oracle.

Where floating point decides an integer — which experts make the top k, and
in what order — the oracle (fp64) and the kernel (fp32 sums) can disagree
on near-ties.  A token whose oracle logits leave a margin above the fp32
error bound must match exactly; on a near-tie the kernel's choice must be a
valid top-k within that bound.  Weights: the oracle's softmax over the
kernel's selection, within the error the logit bound allows.
"""
import math

import numpy as np
import pytest
import torch

from oracle import router as orouter
from nvfp4_block_scaled_route_gb300 import synthetic as syn


# ------------------------------------------------------------- oracle pins --

def _brute(x, w, k, mode):
    T, E = len(x), len(w)
    out_ids, out_w = [], []
    for t in range(T):
        lg = [math.fsum(float(a) * float(b) for a, b in zip(x[t], w[e])) for e in range(E)]
        order = sorted(range(E), key=lambda e: (-lg[e], e))[:k]
        if mode == "selected":
            m = max(lg[e] for e in order)
            ex = [math.exp(lg[e] - m) for e in order]
            s = sum(ex)
            ws = [v / s for v in ex]
        else:
            m = max(lg)
            s = sum(math.exp(v - m) for v in lg)
            ws = [math.exp(lg[e] - m) / s for e in order]
        out_ids.append(order)
        out_w.append(ws)
    return np.array(out_ids), np.array(out_w)


@pytest.mark.parametrize("mode", ["selected", "all"])
def test_router_oracle_brute_force(mode):
    rng = np.random.default_rng(3)
    x = rng.normal(0, 1, (7, 24))
    w = rng.normal(0, 0.2, (9, 24))
    ids, ws, _ = orouter.route(x, w, 3, mode)
    bi, bw = _brute(x, w, 3, mode)
    assert np.array_equal(ids, bi)
    assert np.allclose(ws, bw, rtol=1e-12, atol=0)


def test_router_oracle_ties_go_to_lower_id():
    x = np.ones((1, 4))
    w = np.array([[1, 0, 0, 0], [2, 0, 0, 0], [1, 0, 0, 0], [2, 0, 0, 0], [0, 0, 0, 0.]])
    ids, ws, lg = orouter.route(x, w, 4, "selected")
    assert ids.tolist() == [[1, 3, 0, 2]]
    e = math.exp(-1.0)
    assert np.allclose(ws[0], [1 / (2 + 2 * e), 1 / (2 + 2 * e), e / (2 + 2 * e), e / (2 + 2 * e)])


def test_router_oracle_softmax_properties():
    rng = np.random.default_rng(4)
    x = rng.normal(0, 1, (20, 32))
    w = rng.normal(0, 0.3, (16, 32))
    _, ws, lg = orouter.route(x, w, 16, "selected")
    assert np.allclose(ws.sum(1), 1.0, rtol=0, atol=1e-15)
    ids, wa, _ = orouter.route(x, w, 16, "all")       # k = E: the full softmax
    full = np.exp(lg - lg.max(1, keepdims=True))
    full /= full.sum(1, keepdims=True)
    assert np.allclose(np.take_along_axis(full, ids.astype(np.int64), 1), wa, rtol=1e-14, atol=0)
    assert np.all(np.diff(np.take_along_axis(lg, ids.astype(np.int64), 1), axis=1) <= 0)


def test_router_weight_draw_gives_unit_logits():
    cfg = syn.CONFIGS["decode64"]
    x = syn.draw_activations(cfg).float().numpy()
    w = syn.draw_router_weight(cfg).float().numpy()
    lg = orouter.logits(x, w)
    assert 0.8 < lg.std() < 1.2


# --------------------------------------------------------------- CUDA path --

@pytest.fixture(scope="module")
def nb():
    import __graft_entry__
    __graft_entry__.build()
    from nvfp4_block_scaled_route_gb300 import binding
    return binding


def check_router(x, w, k, mode, ids_g, w_g):
    """Returns the number of near-tie tokens."""
    x64 = np.asarray(x, np.float64)
    w64 = np.asarray(w, np.float64)
    lg = x64 @ w64.T
    # bound on the fp32 sum of H products (longest sequential chain <= H)
    H = x64.shape[1]
    tol = H * 2.0 ** -24 * (np.abs(x64) @ np.abs(w64).T)          # [T, E]
    ids_o = orouter.topk(lg, k)
    ties = 0
    for t in range(lg.shape[0]):
        g = ids_g[t].astype(np.int64)
        assert len(set(g.tolist())) == k
        sel = np.zeros(lg.shape[1], bool)
        sel[g] = True
        # validity: every selected logit >= every unselected one, within the bound
        if (~sel).any():
            worst_gap = (lg[t, ~sel] - tol[t, ~sel]).max() - (lg[t, sel] + tol[t, sel]).min()
            assert worst_gap <= 0, (t, worst_gap)
        # order: non-increasing within the bound
        lt, tt = lg[t, g], tol[t, g]
        assert np.all(lt[1:] - tt[1:] <= lt[:-1] + tt[:-1]), t
        if not np.array_equal(g, ids_o[t]):
            ties += 1
        ref = orouter.weights(lg[t:t + 1], g[None], mode)[0]
        bound = 2.0 * tt.max() * ref + 1e-6
        assert np.all(np.abs(w_g[t] - ref) <= bound), (t, w_g[t], ref)
    return ties


@pytest.mark.gpu
@pytest.mark.parametrize("name", ["tiny", "small", "medium", "decode1", "decode64", "prefill4k",
                                  "prefill16k"])
def test_router_matches_oracle(nb, name):
    cfg = syn.CONFIGS[name]
    mode = "all" if cfg.routing == "softmax_topk_probs" else "selected"
    x = syn.draw_activations(cfg)
    w = syn.draw_router_weight(cfg)
    ids, wt = nb.router_topk(x.to("cuda"), w.to("cuda"), cfg.k,
                             nb.ROUTER_ALL if mode == "all" else nb.ROUTER_SELECTED)
    torch.cuda.synchronize()
    ties = check_router(x.float().numpy(), w.float().numpy(), cfg.k, mode,
                        ids.cpu().numpy(), wt.cpu().numpy())
    assert ties <= max(2, cfg.T // 20), ties
    print(f"{name}: {ties} near-tie tokens of {cfg.T}")


@pytest.mark.gpu
def test_router_ties_and_edges(nb):
    """Exactly equal logits go to the lower id; k = E; E = 256; T = 0."""
    H = 128
    x = torch.ones((3, H), dtype=torch.bfloat16)
    w = torch.zeros((6, H), dtype=torch.bfloat16)
    w[1, 0] = w[3, 0] = 2.0
    w[0, 0] = w[2, 0] = 1.0
    ids, wt = nb.router_topk(x.cuda(), w.cuda(), 6)
    assert ids.cpu().tolist() == [[1, 3, 0, 2, 4, 5]] * 3
    e1, e2 = math.exp(-1.0), math.exp(-2.0)
    s = 2 + 2 * e1 + 2 * e2
    assert np.allclose(wt.cpu().numpy()[0], [1 / s, 1 / s, e1 / s, e1 / s, e2 / s, e2 / s], atol=1e-6)
    g = torch.Generator().manual_seed(5)
    x = (torch.randn((70, 256), generator=g)).to(torch.bfloat16)
    w = (torch.randn((256, 256), generator=g) * 0.06).to(torch.bfloat16)
    ids, wt = nb.router_topk(x.cuda(), w.cuda(), 32)
    torch.cuda.synchronize()
    check_router(x.float().numpy(), w.float().numpy(), 32, "selected", ids.cpu().numpy(),
                 wt.cpu().numpy())
    # the tensor-core logits path (>= 1024 tokens): 256 experts in four
    # column tiles, a ragged last token tile
    x = (torch.randn((1100, 256), generator=g)).to(torch.bfloat16)
    ids, wt = nb.router_topk(x.cuda(), w.cuda(), 8)
    torch.cuda.synchronize()
    check_router(x.float().numpy(), w.float().numpy(), 8, "selected", ids.cpu().numpy(),
                 wt.cpu().numpy())
    # ... 200 experts (ragged last column tile), H = 128 (fewer chunks than
    # the staging ring), probabilities over all experts
    x = (torch.randn((1030, 128), generator=g)).to(torch.bfloat16)
    w2 = (torch.randn((200, 128), generator=g) * 0.09).to(torch.bfloat16)
    ids, wt = nb.router_topk(x.cuda(), w2.cuda(), 6, mode=nb.ROUTER_ALL)
    torch.cuda.synchronize()
    check_router(x.float().numpy(), w2.float().numpy(), 6, "all", ids.cpu().numpy(),
                 wt.cpu().numpy())
    # ... 12 experts (one 16-wide tile, 4 padded columns)
    w3 = (torch.randn((12, 128), generator=g) * 0.09).to(torch.bfloat16)
    ids, wt = nb.router_topk(x.cuda(), w3.cuda(), 2)
    torch.cuda.synchronize()
    check_router(x.float().numpy(), w3.float().numpy(), 2, "selected", ids.cpu().numpy(),
                 wt.cpu().numpy())
    ids, wt = nb.router_topk(torch.zeros((0, 256), dtype=torch.bfloat16, device="cuda"),
                             w.cuda(), 4)
    assert ids.shape == (0, 4)
