"""Full-size parity of the larger workloads — decode T=64 (uniform routing),
prefill T=4096 (Zipf routing) and prefill T=16384 (one hot expert, heavy-
tailed activations), all with E=48, H=7168, I=3072, top-8 — in the
configuration bench.py times: the one-call layer entry point
(moe_nvfp4_layer_forward, here its route -> quantise -> GEMM -> reduce
launches), bf16 output, weights quantised and prepared by the library (the
fp32 weights are drawn on the host, so that the oracle's workers can draw
the same ones).

The oracle cannot follow every token at these sizes, but the intermediate
global scale depends on every h row, so it runs the whole L1 pass, expert by
expert in a spawn pool (fp64 products, h rounded to fp32), keeping max |h|
and the h rows of a sample of tokens; it then takes the sampled tokens
through requantisation, L2 and the top-k reduce.  Checked:
  gs_h                    relative 1e-5
  weight global scales    bit-exact
  sampled h rows          max|err| <= 2e-3 * row-amax, cosine >= 0.9999
  sampled hq / hsf        bit-exact except on rounding boundaries
  sampled y (bf16)        2e-3 * row-amax plus one bf16 rounding (where a
                          requantised value sat on a rounding boundary, the
                          oracle follows the GPU's decision there)
  y with and without the intermediate taps: identical bits
"""
import numpy as np
import pytest
import torch

from oracle import moe as omoe
from oracle import nvfp4 as onv
from nvfp4_block_scaled_route_gb300 import synthetic as syn

from _layout import unstage
import _oracle_pool
from test_gpu_forward import DEV, GEMM_TOL, BOUNDARY_TOL, rows_close, check_requant

pytestmark = pytest.mark.gpu

N_SAMPLE = 16
CHUNK_ROWS = 4096          # oracle L1 task size (rows of one expert)


@pytest.fixture(scope="module")
def nb():
    import __graft_entry__
    __graft_entry__.build()
    from nvfp4_block_scaled_route_gb300 import binding
    return binding


@pytest.mark.parametrize("name", ["decode64", "prefill4k", "prefill16k"])
def test_full_size_sampled_tokens(nb, name):
    cfg = syn.CONFIGS[name]
    T, k, E, H, I = cfg.T, cfg.k, cfg.E, cfg.H, cfg.I
    x = syn.draw_activations(cfg)                     # bf16 [T, H]
    ids, w = syn.draw_routing(cfg)
    ids_np, w_np = ids.numpy(), w.numpy().astype(np.float64)
    rng = np.random.default_rng(7)
    sample = sorted(set([0, 1, T - 2, T - 1] + rng.choice(T, N_SAMPLE - 4, replace=False).tolist()))

    # ---- oracle work on the host (pool started before any CUDA call) ----
    x_bits = x.view(torch.int16).numpy().view(np.uint16)
    gs_x = onv.global_scale(np.abs(x.float().numpy()).max())
    flat_e = ids_np.reshape(-1)
    order = np.argsort(flat_e, kind="stable")            # dense slot order
    local = np.empty(T * k, dtype=np.int64)              # flat index -> row within its expert
    counts = np.bincount(flat_e, minlength=E)
    starts = np.concatenate([[0], np.cumsum(counts)])
    local[order] = np.arange(T * k) - starts[flat_e[order]]
    want = {}
    for t in sample:
        for j in range(k):
            want.setdefault(int(ids_np[t, j]), set()).add(int(local[t * k + j]))
    tasks = []
    for e in range(E):
        toks = order[starts[e]:starts[e + 1]] // k
        for c0 in range(0, len(toks), CHUNK_ROWS):
            wl = [i for i in want.get(e, ()) if c0 <= i < c0 + CHUNK_ROWS]
            tasks.append((name, e, c0, x_bits[toks[c0:c0 + CHUNK_ROWS]], gs_x, wl))
    w2_experts = sorted(want)
    pool = _oracle_pool.pool()
    l1_async = pool.map_async(_oracle_pool.expert_l1_task, tasks)
    w2_async = pool.map_async(_oracle_pool.expert_w2_task, [(name, e) for e in w2_experts])

    # ---- GPU, as bench.py runs it ----
    q1s, s1s, g1s, q2s, s2s, g2s = [], [], [], [], [], []
    # drawn on the host (the generator stream the oracle workers reproduce)
    for e in range(E):
        q, s, g = nb.quantize_weights(syn.draw_weight(cfg, 1, e).to(DEV)[None])
        q1s.append(q); s1s.append(s); g1s.append(g)
        q, s, g = nb.quantize_weights(syn.draw_weight(cfg, 2, e).to(DEV)[None])
        q2s.append(q); s2s.append(s); g2s.append(g)
    gs_w1_gpu = torch.cat(g1s).cpu().numpy()
    gs_w2_gpu = torch.cat(g2s).cpu().numpy()
    pw = nb.PreparedWeights.from_checkpoint(torch.cat(q1s), torch.cat(s1s), torch.cat(g1s),
                                            torch.cat(q2s), torch.cat(s2s), torch.cat(g2s))
    del q1s, s1s, q2s, s2s
    layer = nb.FusedLayer(pw, T, k, device=DEV, out_dtype=torch.bfloat16)
    xd, idsd, wd = x.to(DEV), ids.to(DEV), w.to(DEV)
    y_plain = layer.forward(xd, idsd, wd).clone()
    rows = layer.rows
    taps = dict(h=torch.zeros((rows, I), dtype=torch.float32, device=DEV),
                hq=torch.zeros((rows, I // 2), dtype=torch.uint8, device=DEV),
                hsf_mma=torch.zeros(nb.sf_mma_bytes(rows, I), dtype=torch.uint8, device=DEV),
                gs_h=torch.zeros(1, dtype=torch.float32, device=DEV),
                slot_of=torch.zeros(T * k, dtype=torch.int32, device=DEV))
    y_tap = layer.forward(xd, idsd, wd, taps=taps)
    torch.cuda.synchronize()
    assert layer.status() == 0
    assert torch.equal(y_plain, y_tap), "taps changed the output"
    slot_of = taps["slot_of"].cpu().numpy()
    sample_slots = [slot_of[t * k + j] for t in sample for j in range(k)]
    h_gpu = taps["h"][torch.as_tensor(sample_slots, device=DEV).long()].cpu().numpy()
    hq_gpu = taps["hq"][torch.as_tensor(sample_slots, device=DEV).long()].cpu().numpy()
    hsf_all = unstage(taps["hsf_mma"].cpu().numpy(), rows, I)
    hsf_gpu = hsf_all[np.asarray(sample_slots)]
    gs_h_gpu = float(taps["gs_h"].item())
    y_gpu = y_plain.float().cpu().numpy()[sample]
    del layer, pw, taps

    # ---- oracle results ----
    l1 = l1_async.get()
    w2 = {e: (q, s, g) for e, q, s, g in w2_async.get()}
    pool.close()
    pool.join()
    gs_w1 = {}
    amax_h = np.float32(0.0)
    h_rows = {}
    for e, g1, amax, rws in l1:
        gs_w1[e] = g1
        amax_h = max(amax_h, amax)
        for i, row in rws.items():
            h_rows[(e, i)] = row
    del tasks
    for e in gs_w1:                 # experts that received slots
        assert float(gs_w1[e]) == float(gs_w1_gpu[e]), e
    for e in w2_experts:
        assert float(w2[e][2]) == float(gs_w2_gpu[e]), e
    gs_h = onv.global_scale(amax_h)
    assert abs(gs_h_gpu - float(gs_h)) <= BOUNDARY_TOL * float(gs_h)

    h_ref = np.stack([h_rows[(int(ids_np[t, j]), int(local[t * k + j]))]
                      for t in sample for j in range(k)])
    rows_close(h_gpu, h_ref, "h")
    hq_ref, hsf_ref, _ = onv.quantize_rows(h_ref, gs_h)
    flips = check_requant(h_ref, gs_h, hq_ref, hsf_ref, hq_gpu, hsf_gpu)
    if sum(flips):
        # every difference lies on a rounding boundary, where both decisions
        # are correct: follow the decision the GPU took
        hq_ref, hsf_ref = hq_gpu, hsf_gpu
    y64 = np.zeros((len(sample), H), dtype=np.float64)
    for a, t in enumerate(sample):
        for j in range(k):
            e = int(ids_np[t, j])
            r = a * k + j
            q, s, g2 = w2[e]
            out = omoe.expert_l2(hq_ref[r:r + 1], hsf_ref[r:r + 1], gs_h, q, s, g2)[0]
            y64[a] += w_np[t, j] * out
    bound = GEMM_TOL * np.abs(y64).max(1, keepdims=True) + 2.0 ** -8 * np.abs(y64)
    assert np.all(np.abs(y_gpu - y64) <= bound), float(np.max(np.abs(y_gpu - y64) - bound))
    print(f"{name}: {len(sample)} tokens, requant flips (scale, nibble) = {flips}, "
          f"gs_h {gs_h_gpu:.6g}")
