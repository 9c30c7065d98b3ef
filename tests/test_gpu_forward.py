"""End-to-end parity of the MoE forward pass (route -> quantise -> L1 ->
SiLU*up -> requantise -> L2 -> reduce) through the C ABI against the oracle.

Element by element at sizes the oracle finishes in seconds (several tiles,
ragged tails, zero-token experts) and at the decode workload's full size.
Intermediates are compared through the optional taps:
  L1 output, h          max|err| <= 2e-3 * row-amax, cosine >= 0.9999
  gs_h                  relative 1e-5 (a max over fp32 values)
  hq / hsf              bit-exact except where the oracle's pre-quantisation
                        value lies within 1e-5 relative of a rounding boundary
                        (and every nibble of a block whose scale flipped)
  slot_out, y (fp32)    max|err| <= 2e-3 * row-amax, cosine >= 0.9999
  y (bf16)              the fp32 bound plus one bf16 rounding (2^-8 relative)
Where a requantised value sat on a rounding boundary (both decisions
correct), one 4-bit step moves an L2 output by more than the GEMM
tolerance; slot_out and y are then compared with the oracle's result under
the GPU's decision at those elements (flip_adjusted), after check_requant
has verified that every differing element is such a boundary case.
"""
import numpy as np
import pytest
import torch

from oracle.cpp import moe as omoe, nvfp4 as onv
from nvfp4_block_scaled_route_gb300 import synthetic as syn

from _layout import unstage

pytestmark = pytest.mark.gpu

DEV = "cuda"
GEMM_TOL = 2e-3
COS_TOL = 0.9999
BOUNDARY_TOL = 1e-5
E2M1_BOUNDARIES = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])


@pytest.fixture(scope="module")
def nb():
    import __graft_entry__
    __graft_entry__.build()
    from nvfp4_block_scaled_route_gb300 import binding
    return binding


def rows_close(got, want, what):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    worst = 0.0
    for r in range(want.shape[0]):
        amax = np.abs(want[r]).max()
        err = np.abs(got[r] - want[r]).max()
        assert err <= GEMM_TOL * amax + 1e-30, (what, r, err, amax)
        worst = max(worst, err / amax if amax else 0.0)
        if amax > 0:
            assert omoe.cosine(got[r], want[r]) >= COS_TOL, (what, r)
    return worst


def near_boundary(x, boundaries, tol=BOUNDARY_TOL):
    x = np.asarray(x, np.float64)
    d = np.min(np.abs(x[..., None] - boundaries) / boundaries, axis=-1)
    return d <= tol


def e4m3_boundaries():
    v = onv.e4m3_decode(np.arange(0, 127))
    return (v[:-1] + v[1:]) / 2


def check_requant(h_or, gs_or, hq_or, hsf_or, hq_gpu, hsf_gpu):
    """Flips of the requantised intermediate must sit on rounding boundaries
    of the oracle's own values.  gs_or: one scale, or one per row.  Returns
    (scale flips, nibble flips)."""
    S, I = h_or.shape
    blocks = h_or.reshape(S, I // 16, 16).astype(np.float64)
    gs_rows = np.broadcast_to(np.asarray(gs_or, np.float64).reshape(-1, 1), (S, 1))
    sf_flip = hsf_gpu != hsf_or
    if sf_flip.any():
        t = np.abs(blocks).max(-1) / (6.0 * gs_rows)
        assert near_boundary(t[sf_flip], e4m3_boundaries()).all(), "scale flip off a boundary"
    nib_g = onv.unpack_nibbles(hq_gpu).reshape(S, I // 16, 16)
    nib_o = onv.unpack_nibbles(hq_or).reshape(S, I // 16, 16)
    diff = (nib_g != nib_o) & ~sf_flip[..., None]
    # a sign-only difference on a value that rounds to magnitude 0 is the
    # same encoded value
    same_zero = ((nib_g & 7) == 0) & ((nib_o & 7) == 0)
    diff &= ~same_zero
    if diff.any():
        d = onv.e4m3_decode(hsf_or).astype(np.float64) * gs_rows
        r = np.abs(blocks) / d[..., None]
        assert near_boundary(r[diff], E2M1_BOUNDARIES).all(), "nibble flip off a boundary"
    return int(sf_flip.sum()), int(diff.sum())


def flip_adjusted(ref, hq_g, hsf_g, w2, topk_w):
    """The oracle's slot outputs and y with the GPU's requantisation decisions
    put in where the two differ.  check_requant has verified that every such
    element lies on a rounding boundary, where both decisions are correct
    results; one step of a 4-bit code moves an L2 output far more than the
    GEMM tolerance, so the comparison follows the decision actually taken.
    hq_g / hsf_g in dense slot order; w2 = (q, sf, gs) oracle checkpoint."""
    w2q, w2sf, gs_w2 = w2
    deq_or = onv.dequantize_rows(ref["hq"], ref["hsf"])
    deq_g = onv.dequantize_rows(hq_g, hsf_g)
    diff = deq_g - deq_or
    out2 = np.array(ref["out2"], dtype=np.float64, copy=True)
    offsets = np.asarray(ref["route"]["offsets"])
    for s_ in np.nonzero(np.any(diff != 0, axis=1))[0]:
        e = int(np.searchsorted(offsets, s_, side="right") - 1)
        gs_h = float(ref["gs_h"]) if ref.get("gs_mid") is None else float(ref["gs_mid"][e])
        W = onv.dequantize_weight(w2q[e], w2sf[e])
        out2[s_] += (diff[s_] @ W) * (gs_h * float(gs_w2[e]))
    y64 = omoe.unpermute_reduce(out2, ref["route"]["slot_of"], topk_w)
    return out2, y64


def run_gpu(nb, cfg, x, ids, w, W1_dev, W2_dev, out_dtype=torch.float32, path=0,
            slot_dtype=torch.float32):
    q1, s1, g1 = nb.quantize_weights(W1_dev)
    q2, s2, g2 = nb.quantize_weights(W2_dev)
    pw = nb.PreparedWeights.from_checkpoint(q1, s1, g1, q2, s2, g2)
    layer = nb.MoELayer(pw, cfg.T, cfg.k, device=DEV, out_dtype=out_dtype, slot_dtype=slot_dtype)
    rows = layer.rows
    taps = dict(l1_out=torch.zeros((rows, 2 * cfg.I), dtype=torch.float32, device=DEV),
                h=torch.zeros((rows, cfg.I), dtype=torch.float32, device=DEV),
                hq=torch.zeros((rows, cfg.I // 2), dtype=torch.uint8, device=DEV),
                hsf_mma=torch.zeros(nb.sf_mma_bytes(rows, cfg.I), dtype=torch.uint8, device=DEV),
                gs_h=torch.zeros(1, dtype=torch.float32, device=DEV), path=path)
    y = layer.forward(x.to(DEV), ids.to(DEV), w.to(DEV), taps=taps)
    torch.cuda.synchronize()
    assert layer.status() == 0
    out = {k: v.cpu().numpy() for k, v in taps.items() if isinstance(v, torch.Tensor)}
    out["y"] = y.float().cpu().numpy()
    out["slot_out"] = layer.slot_out.cpu().numpy()
    out["row_of"] = layer.route.slot_of.cpu().numpy()[:cfg.T * cfg.k]
    out["rows"] = rows
    out["gs_w1"], out["gs_w2"] = g1.cpu().numpy(), g2.cpu().numpy()
    return out


def compare(g, ref, cfg, out_dtype=torch.float32, w2=None, topk_w=None):
    """w2 / topk_w given: slot outputs and y are compared with the oracle's
    result under the GPU's boundary decisions (flip_adjusted)."""
    r = ref["route"]
    # dense slot s -> GPU row
    dense_rows = np.empty(cfg.T * cfg.k, dtype=np.int64)
    dense_rows[r["slot_of"]] = g["row_of"]
    rows_close(g["l1_out"][dense_rows], ref["l1"], "l1")
    rows_close(g["h"][dense_rows], ref["h"], "h")
    gs_g, gs_o = float(g["gs_h"][0]), float(ref["gs_h"])
    assert abs(gs_g - gs_o) <= BOUNDARY_TOL * gs_o
    hsf_g = unstage(g["hsf_mma"], g["rows"], cfg.I)[dense_rows]
    flips = check_requant(ref["h"], ref["gs_h"], ref["hq"], ref["hsf"],
                          g["hq"][dense_rows], hsf_g)
    out2, y64 = ref["out2"], ref["y64"]
    if w2 is not None and sum(flips):
        out2, y64 = flip_adjusted(ref, g["hq"][dense_rows], hsf_g, w2, topk_w)
    rows_close(g["slot_out"][dense_rows], out2, "slot_out")
    if out_dtype == torch.float32:
        rows_close(g["y"], y64, "y")
    else:
        bound = GEMM_TOL * np.abs(y64).max(1, keepdims=True) + 2.0 ** -8 * np.abs(y64)
        assert np.all(np.abs(g["y"] - y64) <= bound)
    return flips


@pytest.mark.parametrize("path", [1, 2], ids=["separate", "fused"])
@pytest.mark.parametrize("name", ["tiny", "small", "medium", "waves"])
def test_forward_matches_oracle(nb, name, path):
    """Both execution paths: three launches (L1, requantise, L2) and the
    single cooperative kernel."""
    cfg = syn.CONFIGS[name]
    x = syn.draw_activations(cfg)
    ids, w = syn.draw_routing(cfg)
    W1 = torch.stack([syn.draw_weight(cfg, 1, e) for e in range(cfg.E)])
    W2 = torch.stack([syn.draw_weight(cfg, 2, e) for e in range(cfg.E)])
    g = run_gpu(nb, cfg, x, ids, w, W1.to(DEV), W2.to(DEV), path=path)
    w2q = omoe.quantize_expert_weights(list(W2.numpy()))
    ref = omoe.forward(x.float().numpy(), ids.numpy(), w.numpy(),
                       *omoe.quantize_expert_weights(list(W1.numpy())),
                       *w2q)
    assert np.array_equal(g["gs_w1"], np.array([onv.quantize_weight(W1[e].numpy())[2]
                                                for e in range(cfg.E)]))
    flips = compare(g, ref, cfg, w2=w2q, topk_w=w.numpy())
    print(f"{name} path {path}: requant flips (scale, nibble) = {flips}")


@pytest.mark.parametrize("name", ["small", "medium", "waves"])
def test_paths_agree_bit_for_bit(nb, name):
    """The fused kernel and the three-launch path take the same arithmetic in
    the same order: every intermediate and the output are identical."""
    cfg = syn.CONFIGS[name]
    x = syn.draw_activations(cfg)
    ids, w = syn.draw_routing(cfg)
    W1 = torch.stack([syn.draw_weight(cfg, 1, e) for e in range(cfg.E)]).to(DEV)
    W2 = torch.stack([syn.draw_weight(cfg, 2, e) for e in range(cfg.E)]).to(DEV)
    a = run_gpu(nb, cfg, x, ids, w, W1, W2, path=1)
    b = run_gpu(nb, cfg, x, ids, w, W1, W2, path=2)
    rows = a["row_of"]
    for key in ("l1_out", "h", "hq", "slot_out"):
        assert np.array_equal(a[key][rows], b[key][rows]), key
    assert np.array_equal(a["gs_h"], b["gs_h"])
    assert np.array_equal(a["y"], b["y"])


@pytest.mark.parametrize("slot_dtype", [torch.float32, torch.bfloat16, torch.float16],
                         ids=["f32", "bf16", "f16"])
def test_untapped_matches_tapped(nb, slot_dtype):
    """Without taps the whole-tile GEMM hands the accumulator back before
    its global stores (h and 16-bit slot rows held in registers); with taps it
    stores first.  Same arithmetic, so the slot rows and y are identical.  The
    waves workload has enough tiles for the whole-tile kernel on both GEMMs."""
    cfg = syn.CONFIGS["waves"]
    x = syn.draw_activations(cfg).to(DEV)
    ids, w = syn.draw_routing(cfg)
    ids, w = ids.to(DEV), w.to(DEV)
    W1 = torch.stack([syn.draw_weight(cfg, 1, e) for e in range(cfg.E)]).to(DEV)
    W2 = torch.stack([syn.draw_weight(cfg, 2, e) for e in range(cfg.E)]).to(DEV)
    q1, s1, g1 = nb.quantize_weights(W1)
    q2, s2, g2 = nb.quantize_weights(W2)
    pw = nb.PreparedWeights.from_checkpoint(q1, s1, g1, q2, s2, g2)
    outs = []
    for tapped in (False, True):
        layer = nb.MoELayer(pw, cfg.T, cfg.k, device=DEV, slot_dtype=slot_dtype)
        taps = {"path": 1}
        if tapped:
            taps["l1_out"] = torch.zeros((layer.rows, 2 * cfg.I), dtype=torch.float32, device=DEV)
        y = layer.forward(x, ids, w, taps=taps)
        torch.cuda.synchronize()
        assert layer.status() == 0
        rows = layer.route.slot_of[:cfg.T * cfg.k].long()
        outs.append((y.float().cpu(), layer.slot_out[rows].float().cpu()))
    assert torch.equal(outs[0][1], outs[1][1])
    assert torch.equal(outs[0][0], outs[1][0])


@pytest.mark.parametrize("slot_dtype", [torch.float32, torch.float16], ids=["f32", "f16"])
@pytest.mark.parametrize("tapped", [False, True], ids=["untapped", "tapped"])
def test_cta_pair_gemm_matches_one_cta(nb, slot_dtype, tapped):
    """Enough tiles for the GEMMs over CTA pairs (one MMA across two SMs,
    M = 256) on the three-launch path: 2473 tokens, top-4 over 8 experts of
    the waves shapes (H=2048, I=1024), at least 77 m-tiles x 8 n-tiles per
    GEMM.  The counts give experts 9, 10 and 11 m-tiles, so the last pair of
    an odd expert has an empty odd CTA.  Forcing one-CTA tiles must give the
    same bits everywhere."""
    counts = [1300, 1100, 1290, 1250, 1100, 1300, 1250, 1302]
    cfg = syn.MoEConfig("pairs", E=8, H=2048, I=1024, T=sum(counts) // 4, k=4,
                        routing="uniform")
    x = syn.draw_activations(cfg).to(DEV)
    ids, w = syn.routing_with_counts(counts, cfg.k)
    ids, w = ids.to(DEV), w.to(DEV)
    W1 = torch.stack([syn.draw_weight(cfg, 1, e) for e in range(cfg.E)]).to(DEV)
    W2 = torch.stack([syn.draw_weight(cfg, 2, e) for e in range(cfg.E)]).to(DEV)
    q1, s1, g1 = nb.quantize_weights(W1)
    q2, s2, g2 = nb.quantize_weights(W2)
    pw = nb.PreparedWeights.from_checkpoint(q1, s1, g1, q2, s2, g2)
    counts = torch.bincount(ids.flatten().long(), minlength=cfg.E)
    assert bool(((counts + 127) // 128 % 2 == 1).any())
    outs = []
    for path in (nb.PATH_SEPARATE, nb.PATH_SEPARATE_SINGLE):
        layer = nb.MoELayer(pw, cfg.T, cfg.k, device=DEV, slot_dtype=slot_dtype)
        taps = {"path": path}
        if tapped:
            taps["l1_out"] = torch.zeros((layer.rows, 2 * cfg.I), dtype=torch.float32, device=DEV)
            taps["h"] = torch.zeros((layer.rows, cfg.I), dtype=torch.float32, device=DEV)
        y = layer.forward(x, ids, w, taps=taps)
        torch.cuda.synchronize()
        assert layer.status() == 0
        rows = layer.route.slot_of[:cfg.T * cfg.k].long()
        got = {"y": y.float().cpu(), "slot": layer.slot_out[rows].float().cpu()}
        if tapped:
            got["l1"] = taps["l1_out"][rows].cpu()
            got["h"] = taps["h"][rows].cpu()
        outs.append(got)
    for key in outs[0]:
        assert torch.equal(outs[0][key], outs[1][key]), key


def test_forward_bf16_output(nb):
    cfg = syn.CONFIGS["small"]
    x = syn.draw_activations(cfg)
    ids, w = syn.draw_routing(cfg)
    W1 = torch.stack([syn.draw_weight(cfg, 1, e) for e in range(cfg.E)])
    W2 = torch.stack([syn.draw_weight(cfg, 2, e) for e in range(cfg.E)])
    g = run_gpu(nb, cfg, x, ids, w, W1.to(DEV), W2.to(DEV), out_dtype=torch.bfloat16)
    w2q = omoe.quantize_expert_weights(list(W2.numpy()))
    ref = omoe.forward(x.float().numpy(), ids.numpy(), w.numpy(),
                       *omoe.quantize_expert_weights(list(W1.numpy())),
                       *w2q)
    compare(g, ref, cfg, out_dtype=torch.bfloat16, w2=w2q, topk_w=w.numpy())


@pytest.mark.parametrize("counts,k", [([0, 1, 127, 128, 129, 0], 1), ([130, 0, 2, 128], 2)])
def test_forward_edge_counts(nb, counts, k):
    """Experts with 0, 1, 127, 128, 129 slots: empty experts, single rows,
    exact and ragged 128-row tiles."""
    E = len(counts)
    cfg = syn.MoEConfig("edge", E=E, H=256, I=128, T=sum(counts) // k, k=k, routing="uniform")
    x = syn.draw_activations(cfg)
    ids, w = syn.routing_with_counts(counts, k)
    W1 = torch.stack([syn.draw_weight(cfg, 1, e) for e in range(E)])
    W2 = torch.stack([syn.draw_weight(cfg, 2, e) for e in range(E)])
    g = run_gpu(nb, cfg, x, ids, w, W1.to(DEV), W2.to(DEV))
    w2q = omoe.quantize_expert_weights(list(W2.numpy()))
    ref = omoe.forward(x.float().numpy(), ids.numpy(), w.numpy(),
                       *omoe.quantize_expert_weights(list(W1.numpy())),
                       *w2q)
    compare(g, ref, cfg, w2=w2q, topk_w=w.numpy())


def test_forward_decode_full_size(nb):
    """The one-token decode workload at full size (E=48, H=7168, I=3072,
    top-8): every element of every intermediate against the oracle."""
    cfg = syn.CONFIGS["decode1"]
    x = syn.draw_activations(cfg)
    ids, w = syn.draw_routing(cfg)
    used = sorted(set(ids.flatten().tolist()))
    W1 = torch.stack([syn.draw_weight(cfg, 1, e, device=DEV) for e in range(cfg.E)])
    W2 = torch.stack([syn.draw_weight(cfg, 2, e, device=DEV) for e in range(cfg.E)])
    qs = {}
    for e in used:
        q1, s1, g1 = onv.quantize_weight(W1[e].cpu().numpy())
        q2, s2, g2 = onv.quantize_weight(W2[e].cpu().numpy())
        qs[e] = (q1, s1, g1, q2, s2, g2)
    g = run_gpu(nb, cfg, x, ids, w, W1, W2)
    del W1, W2
    for e in used:
        assert float(qs[e][2]) == float(g["gs_w1"][e])
        assert float(qs[e][5]) == float(g["gs_w2"][e])
    gs1 = np.array([qs[e][2] if e in qs else 1.0 for e in range(cfg.E)], np.float32)
    gs2 = np.array([qs[e][5] if e in qs else 1.0 for e in range(cfg.E)], np.float32)
    ref = omoe.forward(x.float().numpy(), ids.numpy(), w.numpy(),
                       lambda e: (qs[e][0], qs[e][1]), None, gs1,
                       lambda e: (qs[e][3], qs[e][4]), None, gs2)
    w2 = ({e: qs[e][3] for e in used}, {e: qs[e][4] for e in used}, gs2)
    flips = compare(g, ref, cfg, w2=w2, topk_w=w.numpy())
    # the pages' stage magnitudes (Debug Log, Symptoms): same order of magnitude
    l1_amax = np.abs(ref["l1"]).max()
    assert 2.0 < l1_amax < 40.0
    print(f"decode1: flips {flips}, l1 amax {l1_amax:.3f}, h amax {np.abs(ref['h']).max():.3f}, "
          f"out2 amax {np.abs(ref['out2']).max():.3f}, y amax {np.abs(ref['y64']).max():.3f}")


def run_gpu_layer(nb, cfg, x, ids, w, W1_dev, W2_dev, out_dtype=torch.float32, path=3):
    """The whole layer through moe_nvfp4_layer_forward (one call)."""
    q1, s1, g1 = nb.quantize_weights(W1_dev)
    q2, s2, g2 = nb.quantize_weights(W2_dev)
    pw = nb.PreparedWeights.from_checkpoint(q1, s1, g1, q2, s2, g2)
    layer = nb.FusedLayer(pw, cfg.T, cfg.k, device=DEV, out_dtype=out_dtype)
    rows = layer.rows
    taps = dict(l1_out=torch.zeros((rows, 2 * cfg.I), dtype=torch.float32, device=DEV),
                h=torch.zeros((rows, cfg.I), dtype=torch.float32, device=DEV),
                hq=torch.zeros((rows, cfg.I // 2), dtype=torch.uint8, device=DEV),
                hsf_mma=torch.zeros(nb.sf_mma_bytes(rows, cfg.I), dtype=torch.uint8, device=DEV),
                gs_h=torch.zeros(1, dtype=torch.float32, device=DEV),
                slot_of=torch.zeros(cfg.T * cfg.k, dtype=torch.int32, device=DEV), path=path)
    outs = []
    for _ in range(2):               # a second call reuses the self-clearing counters
        y = layer.forward(x.to(DEV), ids.to(DEV), w.to(DEV), taps=taps)
        torch.cuda.synchronize()
        outs.append(y.float().cpu().numpy())
    assert np.array_equal(outs[0], outs[1])
    assert layer.status() == 0
    out = {k: v.cpu().numpy() for k, v in taps.items() if isinstance(v, torch.Tensor)}
    out["y"] = outs[1]
    out["row_of"] = out["slot_of"]
    out["rows"] = rows
    out["gs_w1"], out["gs_w2"] = g1.cpu().numpy(), g2.cpu().numpy()
    return out


LAYER_SMALL = syn.MoEConfig("layer16", E=8, H=512, I=256, T=16, k=4, routing="zipf")


@pytest.mark.parametrize("cfg", [syn.CONFIGS["tiny"], LAYER_SMALL], ids=["tiny", "layer16"])
def test_layer_kernel_matches_oracle(nb, cfg):
    """Routing, quantisation, both GEMMs, requantisation and the reduce in
    one cooperative kernel, against the oracle (y compared without slot_out:
    the kernel reduces on the fly)."""
    x = syn.draw_activations(cfg)
    ids, w = syn.draw_routing(cfg)
    W1 = torch.stack([syn.draw_weight(cfg, 1, e) for e in range(cfg.E)])
    W2 = torch.stack([syn.draw_weight(cfg, 2, e) for e in range(cfg.E)])
    g = run_gpu_layer(nb, cfg, x, ids, w, W1.to(DEV), W2.to(DEV))
    w2q = omoe.quantize_expert_weights(list(W2.numpy()))
    ref = omoe.forward(x.float().numpy(), ids.numpy(), w.numpy(),
                       *omoe.quantize_expert_weights(list(W1.numpy())),
                       *w2q)
    r = ref["route"]
    p = omoe.padded_layout(r)
    assert np.array_equal(g["slot_of"], p["row_of"])
    dense_rows = np.empty(cfg.T * cfg.k, dtype=np.int64)
    dense_rows[r["slot_of"]] = g["row_of"]
    rows_close(g["l1_out"][dense_rows], ref["l1"], "l1")
    rows_close(g["h"][dense_rows], ref["h"], "h")
    hsf_g = unstage(g["hsf_mma"], g["rows"], cfg.I)[dense_rows]
    flips = check_requant(ref["h"], ref["gs_h"], ref["hq"], ref["hsf"], g["hq"][dense_rows], hsf_g)
    y64 = ref["y64"]
    if sum(flips):
        _, y64 = flip_adjusted(ref, g["hq"][dense_rows], hsf_g, w2q, w.numpy())
    rows_close(g["y"], y64, "y")


LAYER_WIDE = syn.MoEConfig("layer_wide", E=4, H=512, I=256, T=64, k=2, routing="uniform")


def test_layer_kernel_many_rows_per_expert(nb):
    """The single kernel with experts of more than 32 rows (every token on
    experts 0 and 1: 64 rows each), where valid rows lie outside TMEM lane
    quarter 0 and the kernel stages the scales with tcgen05.cp copies into
    every quarter: against the oracle and bit for bit against the four
    calls.  (With at most 32 rows per expert it stages them with its one
    writer warp; the tiny and layer16 cases cover that.)"""
    cfg = LAYER_WIDE
    x = syn.draw_activations(cfg)
    _, w = syn.draw_routing(cfg)
    ids = torch.tensor([[0, 1]] * cfg.T, dtype=torch.int32)
    W1 = torch.stack([syn.draw_weight(cfg, 1, e) for e in range(cfg.E)])
    W2 = torch.stack([syn.draw_weight(cfg, 2, e) for e in range(cfg.E)])
    g = run_gpu_layer(nb, cfg, x, ids, w, W1.to(DEV), W2.to(DEV))
    b = run_gpu(nb, cfg, x, ids, w, W1.to(DEV), W2.to(DEV), path=1)
    assert np.array_equal(g["y"], b["y"])
    w2q = omoe.quantize_expert_weights(list(W2.numpy()))
    ref = omoe.forward(x.float().numpy(), ids.numpy(), w.numpy(),
                       *omoe.quantize_expert_weights(list(W1.numpy())), *w2q)
    r = ref["route"]
    dense_rows = np.empty(cfg.T * cfg.k, dtype=np.int64)
    dense_rows[r["slot_of"]] = g["row_of"]
    rows_close(g["h"][dense_rows], ref["h"], "h")
    hsf_g = unstage(g["hsf_mma"], g["rows"], cfg.I)[dense_rows]
    flips = check_requant(ref["h"], ref["gs_h"], ref["hq"], ref["hsf"], g["hq"][dense_rows], hsf_g)
    y64 = ref["y64"]
    if sum(flips):
        _, y64 = flip_adjusted(ref, g["hq"][dense_rows], hsf_g, w2q, w.numpy())
    rows_close(g["y"], y64, "y")


@pytest.mark.parametrize("cfg", [syn.CONFIGS["tiny"], LAYER_SMALL], ids=["tiny", "layer16"])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_layer_kernel_equals_four_calls(nb, cfg, out_dtype):
    """The single-kernel layer and the four separate calls give the same bits."""
    x = syn.draw_activations(cfg)
    ids, w = syn.draw_routing(cfg)
    W1 = torch.stack([syn.draw_weight(cfg, 1, e) for e in range(cfg.E)]).to(DEV)
    W2 = torch.stack([syn.draw_weight(cfg, 2, e) for e in range(cfg.E)]).to(DEV)
    a = run_gpu_layer(nb, cfg, x, ids, w, W1, W2, out_dtype=out_dtype, path=3)
    b = run_gpu(nb, cfg, x, ids, w, W1, W2, out_dtype=out_dtype, path=1)
    rows = b["row_of"]
    assert np.array_equal(a["row_of"], rows)
    for key in ("l1_out", "h", "hq"):
        assert np.array_equal(a[key][rows], b[key][rows]), key
    assert np.array_equal(a["gs_h"], b["gs_h"])
    assert np.array_equal(a["y"], b["y"])


@pytest.mark.parametrize("name", ["small", "waves"])
def test_layer_forward_large_batch_uses_four_launches(nb, name):
    """Above the single-kernel limits the one-call API runs the four steps
    (with fp16 slot rows): the same bits as the four calls made directly,
    with the L1 GEMM on the stream-K kernel (small) and on CTA pairs
    (waves)."""
    cfg = syn.CONFIGS[name]                          # T*k = 291 / 9856 > 128
    x = syn.draw_activations(cfg)
    ids, w = syn.draw_routing(cfg)
    W1 = torch.stack([syn.draw_weight(cfg, 1, e) for e in range(cfg.E)]).to(DEV)
    W2 = torch.stack([syn.draw_weight(cfg, 2, e) for e in range(cfg.E)]).to(DEV)
    with pytest.raises(nb.NvmoeError):
        run_gpu_layer(nb, cfg, x, ids, w, W1, W2, path=3)
    a = run_gpu_layer(nb, cfg, x, ids, w, W1, W2, path=0)
    b = run_gpu(nb, cfg, x, ids, w, W1, W2, path=0, slot_dtype=torch.float16)
    assert np.array_equal(a["y"], b["y"])


# --------------------------------------------- separate gate/up scales ----

def _split_weights(nb, W1_dev, W2_dev, I):
    """L1 weights quantised as two matrices (gate, up) with their own global
    scales, as checkpoints that quantise gate_proj and up_proj separately."""
    qg, sg, gg = nb.quantize_weights(W1_dev[:, :, :I].contiguous())
    qu, su, gu = nb.quantize_weights(W1_dev[:, :, I:].contiguous())
    q2, s2, g2 = nb.quantize_weights(W2_dev)
    pw = nb.PreparedWeights.from_checkpoint(torch.cat([qg, qu], 2), torch.cat([sg, su], 2), gg,
                                            q2, s2, g2, gs1_up=gu)
    return pw, gg.cpu().numpy(), gu.cpu().numpy()


@pytest.mark.parametrize("name,path", [("tiny", 1), ("tiny", 2), ("tiny", 3),
                                       ("small", 1), ("small", 2), ("medium", 2)])
def test_forward_gate_up_scales(nb, name, path):
    """Per-column alpha: gate columns gs_x*gs_gate[e], up columns
    gs_x*gs_up[e], on every execution path, against the oracle."""
    cfg = syn.CONFIGS[name]
    x = syn.draw_activations(cfg)
    ids, w = syn.draw_routing(cfg)
    W1 = torch.stack([syn.draw_weight(cfg, 1, e) for e in range(cfg.E)])
    W2 = torch.stack([syn.draw_weight(cfg, 2, e) for e in range(cfg.E)])
    # make the halves' maxima differ, so that the two scales do
    W1[:, :, cfg.I:] *= 3.0
    pw, gg, gu = _split_weights(nb, W1.to(DEV), W2.to(DEV), cfg.I)
    q1, s1, g1 = omoe.quantize_expert_weights(list(W1.numpy()), split_halves=True)
    assert np.array_equal(g1[:, 0], gg) and np.array_equal(g1[:, 1], gu)
    assert np.all(g1[:, 1] > 1.5 * g1[:, 0])
    w2q = omoe.quantize_expert_weights(list(W2.numpy()))
    ref = omoe.forward(x.float().numpy(), ids.numpy(), w.numpy(), q1, s1, g1,
                       *w2q)
    Layer = nb.FusedLayer if path == 3 else nb.MoELayer
    layer = Layer(pw, cfg.T, cfg.k, device=DEV, out_dtype=torch.float32)
    rows = layer.rows
    taps = dict(l1_out=torch.zeros((rows, 2 * cfg.I), dtype=torch.float32, device=DEV),
                h=torch.zeros((rows, cfg.I), dtype=torch.float32, device=DEV),
                hq=torch.zeros((rows, cfg.I // 2), dtype=torch.uint8, device=DEV),
                hsf_mma=torch.zeros(nb.sf_mma_bytes(rows, cfg.I), dtype=torch.uint8, device=DEV),
                slot_of=torch.zeros(cfg.T * cfg.k, dtype=torch.int32, device=DEV), path=path)
    y = layer.forward(x.to(DEV), ids.to(DEV), w.to(DEV), taps=taps)
    torch.cuda.synchronize()
    assert layer.status() == 0
    row_of = taps["slot_of"].cpu().numpy() if path == 3 else \
        layer.route.slot_of.cpu().numpy()[:cfg.T * cfg.k]
    r = ref["route"]
    dense_rows = np.empty(cfg.T * cfg.k, dtype=np.int64)
    dense_rows[r["slot_of"]] = row_of
    rows_close(taps["l1_out"].cpu().numpy()[dense_rows], ref["l1"], "l1")
    rows_close(taps["h"].cpu().numpy()[dense_rows], ref["h"], "h")
    hq_g = taps["hq"].cpu().numpy()[dense_rows]
    hsf_g = unstage(taps["hsf_mma"].cpu().numpy(), rows, cfg.I)[dense_rows]
    flips = check_requant(ref["h"], ref["gs_h"], ref["hq"], ref["hsf"], hq_g, hsf_g)
    y64 = ref["y64"]
    if sum(flips):
        _, y64 = flip_adjusted(ref, hq_g, hsf_g, w2q, w.numpy())
    rows_close(y.cpu().numpy(), y64, "y")


def test_layer_staged_host_step(nb):
    """forward_staged: inputs from the pinned staging area in one copy, y
    back in one copy; the same bits as forward() on device tensors."""
    cfg = syn.CONFIGS["decode1"]
    x = syn.draw_activations(cfg)
    ids, w = syn.draw_routing(cfg)
    W1 = torch.stack([syn.draw_weight(cfg, 1, e, device=DEV) for e in range(cfg.E)])
    W2 = torch.stack([syn.draw_weight(cfg, 2, e, device=DEV) for e in range(cfg.E)])
    q1, s1, g1 = nb.quantize_weights(W1)
    q2, s2, g2 = nb.quantize_weights(W2)
    del W1, W2
    pw = nb.PreparedWeights.from_checkpoint(q1, s1, g1, q2, s2, g2)
    layer = nb.FusedLayer(pw, cfg.T, cfg.k, device=DEV)
    y_dev = layer.forward(x.to(DEV), ids.to(DEV), w.to(DEV)).cpu()
    (hx, hids, hw, hy), _ = layer.staging()
    hx.copy_(x)
    hids.copy_(ids)
    hw.copy_(w)
    out = layer.forward_staged()
    torch.cuda.synchronize()
    assert layer.status() == 0
    assert torch.equal(out, y_dev)


def test_programmatic_dependent_launch_changes_nothing(nb):
    """The multi-launch path (route, quantise, L1, requantise, L2, reduce:
    the waves workload through the one-call layer) with programmatic
    dependent launch on and off, eager and replayed from a CUDA graph: the
    same bits (every kernel waits for the one before it before touching its
    memory)."""
    cfg = syn.CONFIGS["waves"]
    W1 = torch.stack([syn.draw_weight(cfg, 1, e, device=DEV) for e in range(cfg.E)])
    W2 = torch.stack([syn.draw_weight(cfg, 2, e, device=DEV) for e in range(cfg.E)])
    q1, s1, g1 = nb.quantize_weights(W1)
    q2, s2, g2 = nb.quantize_weights(W2)
    pw = nb.PreparedWeights.from_checkpoint(q1, s1, g1, q2, s2, g2)
    layer = nb.FusedLayer(pw, cfg.T, cfg.k, device=DEV)
    x = syn.draw_activations(cfg).to(DEV)
    ids, w = syn.draw_routing(cfg)
    ids, w = ids.to(DEV), w.to(DEV)
    outs = []
    prev = nb.lib().nvmoe_set_pdl(0)
    try:
        for pdl in (0, 1):
            nb.lib().nvmoe_set_pdl(pdl)
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                outs.append(layer.forward(x, ids, w).clone())
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=s):
                    layer.forward(x, ids, w)
                layer.y.zero_()
                for _ in range(3):
                    g.replay()
            s.synchronize()
            outs.append(layer.y.clone())
            assert layer.status() == 0
    finally:
        nb.lib().nvmoe_set_pdl(prev)
    for o in outs[1:]:
        assert torch.equal(o, outs[0])


@pytest.mark.parametrize("name", ["small", "waves"])
def test_staged_pipeline_overlapped_steps(nb, name):
    """StagedPipeline: two slots with different inputs, seven steps whose
    copies overlap other steps' layers; every step's host y equals a direct
    forward() of its own inputs (a missing or misplaced event would let a
    step read another slot's inputs or y)."""
    cfg = syn.CONFIGS[name]
    W1 = torch.stack([syn.draw_weight(cfg, 1, e, device=DEV) for e in range(cfg.E)])
    W2 = torch.stack([syn.draw_weight(cfg, 2, e, device=DEV) for e in range(cfg.E)])
    q1, s1, g1 = nb.quantize_weights(W1)
    q2, s2, g2 = nb.quantize_weights(W2)
    pw = nb.PreparedWeights.from_checkpoint(q1, s1, g1, q2, s2, g2)
    layer = nb.FusedLayer(pw, cfg.T, cfg.k, device=DEV)
    pipe = nb.StagedPipeline(layer, depth=2)
    want = []
    for slot in range(2):
        x = syn.draw_activations(cfg) * (1.0 + slot)
        ids, w = syn.draw_routing(cfg)
        if slot:
            ids = torch.flip(ids, dims=[1]).contiguous()
        want.append(layer.forward(x.to(DEV), ids.to(DEV), w.to(DEV)).cpu().clone())
        hx, hids, hw = pipe.inputs(slot)
        hx.copy_(x.to(torch.bfloat16))
        hids.copy_(ids)
        hw.copy_(w)
    torch.cuda.synchronize()
    for i in range(7):
        slot = pipe.submit()
        assert slot == i % 2
        if i >= 5:
            pipe.output_ready(slot).synchronize()
            assert torch.equal(pipe.output(slot), want[slot]), (i, slot)
    pipe.synchronize()
    assert layer.status() == 0
    for slot in range(2):
        assert torch.equal(pipe.output(slot), want[slot])



# ------------------------------------------ static intermediate scale ----

@pytest.mark.parametrize("name,path", [("tiny", 1), ("tiny", 2), ("tiny", 3),
                                       ("small", 1), ("small", 2), ("medium", 1),
                                       ("waves", 1)])
def test_forward_static_mid_scale(nb, name, path):
    """A static intermediate scale per expert: each CTA requantises its own
    L1 tiles with gs_mid[e] (no global amax, no requantisation pass); L2
    alpha gs_mid[e]*gs_w2[e].  Scales span saturating and coarse cases.
    At the waves size the L1 GEMM takes whole tiles on CTA pairs, where each
    epilogue set requantises the columns it has stored."""
    cfg = syn.CONFIGS[name]
    x = syn.draw_activations(cfg)
    ids, w = syn.draw_routing(cfg)
    W1 = torch.stack([syn.draw_weight(cfg, 1, e) for e in range(cfg.E)])
    W2 = torch.stack([syn.draw_weight(cfg, 2, e) for e in range(cfg.E)])
    w1q = omoe.quantize_expert_weights(list(W1.numpy()))
    w2q = omoe.quantize_expert_weights(list(W2.numpy()))
    dyn = omoe.forward(x.float().numpy(), ids.numpy(), w.numpy(), *w1q, *w2q)
    mid = (float(dyn["gs_h"]) * np.linspace(0.3, 2.0, cfg.E)).astype(np.float32)
    ref = omoe.forward(x.float().numpy(), ids.numpy(), w.numpy(), *w1q, *w2q, gs_mid=mid)
    q1, s1, g1 = nb.quantize_weights(W1.to(DEV))
    q2, s2, g2 = nb.quantize_weights(W2.to(DEV))
    pw = nb.PreparedWeights.from_checkpoint(q1, s1, g1, q2, s2, g2,
                                            gs_mid=torch.from_numpy(mid).to(DEV))
    Layer = nb.FusedLayer if path == 3 else nb.MoELayer
    layer = Layer(pw, cfg.T, cfg.k, device=DEV, out_dtype=torch.float32)
    rows = layer.rows
    taps = dict(h=torch.zeros((rows, cfg.I), dtype=torch.float32, device=DEV),
                hq=torch.zeros((rows, cfg.I // 2), dtype=torch.uint8, device=DEV),
                hsf_mma=torch.zeros(nb.sf_mma_bytes(rows, cfg.I), dtype=torch.uint8, device=DEV),
                slot_of=torch.zeros(cfg.T * cfg.k, dtype=torch.int32, device=DEV), path=path)
    y = layer.forward(x.to(DEV), ids.to(DEV), w.to(DEV), taps=taps)
    torch.cuda.synchronize()
    assert layer.status() == 0
    row_of = taps["slot_of"].cpu().numpy() if path == 3 else \
        layer.route.slot_of.cpu().numpy()[:cfg.T * cfg.k]
    r = ref["route"]
    dense_rows = np.empty(cfg.T * cfg.k, dtype=np.int64)
    dense_rows[r["slot_of"]] = row_of
    rows_close(taps["h"].cpu().numpy()[dense_rows], ref["h"], "h")
    hq_g = taps["hq"].cpu().numpy()[dense_rows]
    hsf_g = unstage(taps["hsf_mma"].cpu().numpy(), rows, cfg.I)[dense_rows]
    slot_expert = np.searchsorted(np.asarray(r["offsets"]), np.arange(cfg.T * cfg.k), side="right") - 1
    flips = check_requant(ref["h"], mid[slot_expert], ref["hq"], ref["hsf"], hq_g, hsf_g)
    y64 = ref["y64"]
    if sum(flips):
        _, y64 = flip_adjusted(ref, hq_g, hsf_g, w2q, w.numpy())
    rows_close(y.cpu().numpy(), y64, "y")


# ------------------------------------------------- 16-bit slot rows ----

@pytest.mark.parametrize("slot_dtype,rel", [(torch.float16, 2.0 ** -11), (torch.bfloat16, 2.0 ** -8)],
                         ids=["f16", "bf16"])
@pytest.mark.parametrize("name,path", [("small", 1), ("medium", 2), ("waves", 1)])
def test_forward_16bit_slot_rows(nb, name, path, slot_dtype, rel):
    """slot_out held in fp16 or bf16 (the fp32 alpha-scaled L2 result rounded
    to nearest even).  Each slot value is within the GEMM bound plus its own
    rounding (rel * |v|; fp16's 2^-11 stays inside 2e-3 * row-amax), and y
    (fp32) within the GEMM bound plus the rounding carried through the
    weighted sum (rel * sum_j w_j |slot_j|)."""
    cfg = syn.CONFIGS[name]
    x = syn.draw_activations(cfg)
    ids, w = syn.draw_routing(cfg)
    W1 = torch.stack([syn.draw_weight(cfg, 1, e) for e in range(cfg.E)])
    W2 = torch.stack([syn.draw_weight(cfg, 2, e) for e in range(cfg.E)])
    q1, s1, g1 = nb.quantize_weights(W1.to(DEV))
    q2, s2, g2 = nb.quantize_weights(W2.to(DEV))
    pw = nb.PreparedWeights.from_checkpoint(q1, s1, g1, q2, s2, g2)
    layer = nb.MoELayer(pw, cfg.T, cfg.k, device=DEV, out_dtype=torch.float32,
                        slot_dtype=slot_dtype)
    rows = layer.rows
    taps = dict(hq=torch.zeros((rows, cfg.I // 2), dtype=torch.uint8, device=DEV),
                hsf_mma=torch.zeros(nb.sf_mma_bytes(rows, cfg.I), dtype=torch.uint8, device=DEV),
                path=path)
    y = layer.forward(x.to(DEV), ids.to(DEV), w.to(DEV), taps=taps)
    torch.cuda.synchronize()
    assert layer.status() == 0
    w2q = omoe.quantize_expert_weights(list(W2.numpy()))
    ref = omoe.forward(x.float().numpy(), ids.numpy(), w.numpy(),
                       *omoe.quantize_expert_weights(list(W1.numpy())), *w2q)
    r = ref["route"]
    dense_rows = np.empty(cfg.T * cfg.k, dtype=np.int64)
    dense_rows[r["slot_of"]] = layer.route.slot_of.cpu().numpy()[:cfg.T * cfg.k]
    hq_g = taps["hq"].cpu().numpy()[dense_rows]
    hsf_g = unstage(taps["hsf_mma"].cpu().numpy(), rows, cfg.I)[dense_rows]
    flips = check_requant(ref["h"], ref["gs_h"], ref["hq"], ref["hsf"], hq_g, hsf_g)
    out2, y64 = ref["out2"], ref["y64"]
    if sum(flips):
        out2, y64 = flip_adjusted(ref, hq_g, hsf_g, w2q, w.numpy())
    so = layer.slot_out.double().cpu().numpy()[dense_rows]
    bound = GEMM_TOL * np.abs(out2).max(1, keepdims=True) + rel * np.abs(out2)
    assert np.all(np.abs(so - out2) <= bound)
    if slot_dtype == torch.float16:
        rows_close(so, out2, "slot_out")          # the GEMM bar itself holds
    carried = rel * omoe.unpermute_reduce(np.abs(out2), r["slot_of"], np.abs(w.numpy()))
    yb = GEMM_TOL * np.abs(y64).max(1, keepdims=True) + carried
    assert np.all(np.abs(y.double().cpu().numpy() - y64) <= yb)


def test_fp16_slot_rows_report_overflow(nb):
    """A slot value beyond the fp16 range is reported (NVMOE_ERR_RANGE = 8),
    not clamped; fp32 slot rows of the same input report nothing."""
    cfg = syn.CONFIGS["small"]
    x = (syn.draw_activations(cfg).float() * 3.0e4).to(torch.bfloat16)
    ids, w = syn.draw_routing(cfg)
    W1 = torch.stack([syn.draw_weight(cfg, 1, e) for e in range(cfg.E)])
    W2 = torch.stack([syn.draw_weight(cfg, 2, e) for e in range(cfg.E)])
    q1, s1, g1 = nb.quantize_weights(W1.to(DEV))
    q2, s2, g2 = nb.quantize_weights(W2.to(DEV))
    pw = nb.PreparedWeights.from_checkpoint(q1, s1, g1, q2, s2, g2)
    for dt, want in ((torch.float16, 8), (torch.float32, 0)):
        layer = nb.MoELayer(pw, cfg.T, cfg.k, device=DEV, out_dtype=torch.float32, slot_dtype=dt)
        layer.forward(x.to(DEV), ids.to(DEV), w.to(DEV))
        torch.cuda.synchronize()
        assert layer.status() == want
        if dt == torch.float32:
            assert float(layer.slot_out.abs().max()) > 65504.0

