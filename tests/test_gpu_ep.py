"""Expert parallelism on the GPU: the dispatch / scatter / gather kernels,
the two-call forward, and the whole expert-parallel forward with G ranks
emulated in one process (LocalGroup: host barriers between the ranks, no
kernel waits on another).  Multi-GPU runs (NCCL) are not measured on
hardware here: every box has one GPU."""
import threading

import numpy as np
import pytest
import torch

from nvfp4_block_scaled_route_gb300 import ep
from nvfp4_block_scaled_route_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def nb():
    import __graft_entry__
    __graft_entry__.build()
    from nvfp4_block_scaled_route_gb300 import binding
    return binding


def _weights(nb, cfg):
    W1 = torch.stack([syn.draw_weight(cfg, 1, e, device=DEV) for e in range(cfg.E)])
    W2 = torch.stack([syn.draw_weight(cfg, 2, e, device=DEV) for e in range(cfg.E)])
    q1, s1, g1 = nb.quantize_weights(W1)
    q2, s2, g2 = nb.quantize_weights(W2)
    return q1, s1, g1, q2, s2, g2


def _local(nb, ck, e0, e1):
    q1, s1, g1, q2, s2, g2 = ck
    return nb.PreparedWeights.from_checkpoint(q1[e0:e1].contiguous(), s1[e0:e1].contiguous(),
                                              g1[e0:e1].contiguous(), q2[e0:e1].contiguous(),
                                              s2[e0:e1].contiguous(), g2[e0:e1].contiguous())


def test_dispatch_matches_host_restatement(nb):
    """Counts, stable send positions, packed rows and local expert ids, for
    G = 4 over E = 8, with one out-of-range id (recorded, sent nowhere)."""
    E, G = 8, 4
    T, k, H = 97, 3, 512
    g = torch.Generator().manual_seed(5)
    ids = torch.stack([torch.randperm(E, generator=g)[:k] for _ in range(T)]).to(torch.int32)
    ids[7, 1] = 11
    x = syn.draw_activations(syn.MoEConfig("d", E=E, H=H, I=256, T=T, k=k, routing="uniform"))
    q, sf, _, _ = nb.quantize_act(x.to(DEV), mma_sf=False)
    counts, pos, rows, expert, ws = nb.ep_dispatch(ids.to(DEV), E, G, q, sf)
    assert nb.read_status(ws) == 7           # NVMOE_ERR_DEVICE_BAD_INDEX
    flat = ids.reshape(-1).numpy()
    dest = np.where((flat >= 0) & (flat < E), flat // (E // G), -1)
    want_counts = [int(np.sum(dest == d)) for d in range(G)]
    assert counts.cpu().tolist() == want_counts
    order = np.concatenate([np.nonzero(dest == d)[0] for d in range(G)])
    want_pos = np.full(len(flat), -1)
    want_pos[order] = np.arange(len(order))
    assert pos.cpu().numpy().tolist() == want_pos.tolist()
    n = len(order)
    tok = order // k
    want_rows = np.concatenate([q.cpu().numpy()[tok], sf.cpu().numpy()[tok]], axis=1)
    assert np.array_equal(rows[:n].cpu().numpy(), want_rows)
    assert expert[:n].cpu().numpy().tolist() == (flat[order] - dest[order] * (E // G)).tolist()


def test_scatter_reproduces_the_slot_layout(nb):
    """Token rows routed with k = 1 and scattered give the bytes the
    quantiser writes straight into the slot layout."""
    E, T, H = 6, 300, 512
    cfg = syn.MoEConfig("s", E=E, H=H, I=256, T=T, k=1, routing="zipf")
    x = syn.draw_activations(cfg).to(DEV)
    ids, _ = syn.draw_routing(cfg)
    r = nb.route_permute(ids.to(DEV), E)
    want_q, _, want_sf, gs = nb.quantize_act(x, row_dst=r.slot_of, fanout=1, out_rows=r.rows)
    q, sf, _, _ = nb.quantize_act(x, mma_sf=False)
    rows = torch.cat([q, sf], dim=1).contiguous()
    xq = torch.zeros_like(want_q)
    xsf = torch.zeros_like(want_sf)
    nb.ep_scatter(rows, H, r.slot_of, r.rows, xq, xsf)
    torch.cuda.synchronize()
    valid = r.row_token.cpu() >= 0
    assert torch.equal(xq.cpu()[valid], want_q.cpu()[valid])
    # the staged scales of every valid row
    wsf, gsf = want_sf.cpu().numpy(), xsf.cpu().numpy()
    k_atoms = (H + 255) // 256 * 4
    for row in np.nonzero(valid.numpy())[0][::7]:
        for g in range(H // 16):
            off = ((row // 128) * k_atoms + g // 4) * 512 + (row % 32) * 16 + ((row % 128) // 32) * 4 + g % 4
            assert gsf[off] == wsf[off]
    # gather moves bits: raw nibble bytes viewed as 16-bit rows (some are NaN
    # patterns as fp16, so the comparison is on the integer view)
    out = nb.ep_gather(xq.view(torch.float16), r.slot_of, T)
    want_rows = xq.view(torch.int16).cpu()[r.slot_of.cpu().long()]
    assert torch.equal(out.view(torch.int16).cpu(), want_rows)


@pytest.mark.parametrize("name", ["small", "waves"])
def test_two_phase_forward_equals_forward(nb, name):
    """Phase 1 (L1, max |h|) then phase 2 on that amax = moe_nvfp4_forward."""
    cfg = syn.CONFIGS[name]
    ck = _weights(nb, cfg)
    pw = nb.PreparedWeights.from_checkpoint(*ck)
    x = syn.draw_activations(cfg).to(DEV)
    ids, w = syn.draw_routing(cfg)
    r = nb.route_permute(ids.to(DEV), cfg.E)
    xq, _, xsf, gs = nb.quantize_act(x, row_dst=r.slot_of, fanout=cfg.k, out_rows=r.rows,
                                     rowmajor_sf=False)
    ws = nb._workspace(nb.forward_workspace_bytes(cfg.T, cfg.k, cfg.E, cfg.H, cfg.I), DEV)
    want = nb.nvfp4_forward(pw, xq, xsf, gs, r, taps={"path": nb.PATH_SEPARATE}, ws=ws).clone()
    got = torch.empty_like(want)
    amax_h = torch.empty(1, dtype=torch.float32, device=DEV)
    nb.nvfp4_forward_phase(pw, xq, xsf, gs, r, 1, amax_h, got, ws)
    nb.nvfp4_forward_phase(pw, xq, xsf, gs, r, 2, amax_h, got, ws)
    torch.cuda.synchronize()
    rows = r.slot_of.cpu().long()
    assert torch.equal(got.cpu()[rows], want.cpu()[rows])


def _ep_forward(nb, cfg, ck, x, ids, w, G, slot_dtype):
    grp = ep.LocalGroup(G)
    El = cfg.E // G
    cuts = [cfg.T * r // G for r in range(G + 1)]
    out, errs, status = [None] * G, [], [None] * G

    def rank_main(r):
        try:
            be = ep.CudaExpertBackend(_local(nb, ck, r * El, (r + 1) * El), cfg.E, G, cfg.k,
                                      slot_dtype=slot_dtype)
            m = ep.ExpertParallelMoE(be, grp.comm(r))
            t0, t1 = cuts[r], cuts[r + 1]
            out[r] = m.forward(x[t0:t1].contiguous(), ids[t0:t1].contiguous(),
                               w[t0:t1].contiguous())
            torch.cuda.synchronize()
            status[r] = be.status
        except Exception as e:
            errs.append(e)
            grp._barrier.abort()

    th = [threading.Thread(target=rank_main, args=(r,)) for r in range(G)]
    for t in th:
        t.start()
    for t in th:
        t.join()
    if errs:
        raise errs[0]
    assert status == [0] * G
    return torch.cat([o.cpu() for o in out], dim=0)


@pytest.mark.parametrize("G", [1, 2])
def test_expert_parallel_equals_one_gpu(nb, G):
    """The expert-parallel forward (G ranks, each owning E/G experts and T/G
    tokens) against the one-GPU forward of the whole batch.  5120 tokens,
    top-4 over 8 experts of the waves shapes: every rank receives ~10k slots,
    so every GEMM launch, one-GPU or per rank, takes whole tiles (each tile
    accumulated in one order) and the outputs agree bit for bit."""
    cfg = syn.MoEConfig("ep", E=8, H=2048, I=1024, T=5120, k=4, routing="uniform")
    ck = _weights(nb, cfg)
    x = syn.draw_activations(cfg).to(DEV)
    ids, w = syn.draw_routing(cfg)
    ids, w = ids.to(DEV), w.to(DEV)
    layer = nb.MoELayer(nb.PreparedWeights.from_checkpoint(*ck), cfg.T, cfg.k, device=DEV,
                        slot_dtype=torch.float16)
    want = layer.forward(x, ids, w, taps={"path": nb.PATH_SEPARATE}).cpu()
    assert layer.status() == 0
    got = _ep_forward(nb, cfg, ck, x, ids, w, G, torch.float16)
    assert torch.equal(got, want)


def test_expert_parallel_small_batch(nb):
    """A decode-sized batch (stream-K GEMMs on every rank): within the GEMM
    tolerance of the one-GPU forward, and one rank with no slots at all."""
    cfg = syn.MoEConfig("ep_small", E=8, H=512, I=256, T=6, k=2, routing="uniform")
    ck = _weights(nb, cfg)
    x = syn.draw_activations(cfg).to(DEV)
    ids = torch.tensor([[0, 1], [2, 3], [1, 2], [3, 0], [0, 2], [1, 3]], dtype=torch.int32,
                       device=DEV)
    _, w = syn.draw_routing(cfg)
    w = w.to(DEV)
    layer = nb.MoELayer(nb.PreparedWeights.from_checkpoint(*ck), cfg.T, cfg.k, device=DEV,
                        slot_dtype=torch.float16)
    want = layer.forward(x, ids, w, taps={"path": nb.PATH_SEPARATE}).float().cpu()
    got = _ep_forward(nb, cfg, ck, x, ids, w, 2, torch.float16).float()
    # every slot goes to rank 0's experts (0..3): rank 1 receives nothing
    amax = want.abs().amax(dim=1, keepdim=True)
    assert float(((got - want).abs() / amax).max()) < 2e-2
