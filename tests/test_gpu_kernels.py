"""Parity of the CUDA path (through the C ABI) against the CPU oracle.

Bit-exact where the result is integer or byte data (routing, packed nibbles,
scale bytes); within max|err| <= 2e-3 * row-amax and cosine >= 0.9999 per
row for floating-point GEMM outputs.  Every input is drawn from the seeded
generator module; no expected value comes from the CUDA path.
"""
import numpy as np
import pytest
import torch

from oracle.cpp import moe as omoe, nvfp4 as onv
from nvfp4_block_scaled_route_gb300 import synthetic as syn

from _layout import stage, unstage

pytestmark = pytest.mark.gpu

GEMM_TOL = 2e-3
COS_TOL = 0.9999


@pytest.fixture(scope="module")
def nb():
    import __graft_entry__
    __graft_entry__.build()
    from nvfp4_block_scaled_route_gb300 import binding
    assert torch.cuda.is_available()
    return binding


DEV = "cuda"


def assert_rows_close(got, want, what):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    for r in range(want.shape[0]):
        amax = np.abs(want[r]).max()
        err = np.abs(got[r] - want[r]).max()
        assert err <= GEMM_TOL * amax + 1e-30, (what, r, err, amax)
        if amax > 0:
            assert omoe.cosine(got[r], want[r]) >= COS_TOL, (what, r)


# ------------------------------------------------------------- quantiser --

@pytest.mark.parametrize("rows,cols,dist,dtype", [
    (1, 64, "normal", torch.bfloat16),
    (8, 256, "normal", torch.bfloat16),
    (97, 512, "student_t", torch.bfloat16),
    (300, 1024, "normal", torch.float32),
    (257, 3072, "student_t", torch.float32),
    (64, 7168, "normal", torch.bfloat16),
    (3, 192, "tiny_blocks", torch.float32),
])
def test_quantize_act_bit_exact(nb, rows, cols, dist, dtype):
    g = torch.Generator().manual_seed(rows * 7 + cols)
    x = torch.randn((rows, cols), generator=g) * 1.5
    if dist == "student_t":
        x = x / torch.sqrt((torch.randn((3, rows, cols), generator=g) ** 2).sum(0) / 3)
    elif dist == "tiny_blocks":
        scale = 10.0 ** (-7 * torch.rand((rows, cols // 16, 1), generator=g))
        x = (x.reshape(rows, cols // 16, 16) * scale).reshape(rows, cols)
    x = x.to(dtype)
    q, sf_row, sf_mma, gs = nb.quantize_act(x.to(DEV))
    torch.cuda.synchronize()
    xq, xsf, xgs = onv.quantize_rows(x.float().numpy())
    assert gs.item() == float(xgs)
    assert np.array_equal(q.cpu().numpy(), xq)
    assert np.array_equal(sf_row.cpu().numpy(), xsf)
    assert np.array_equal(unstage(sf_mma.cpu().numpy(), rows, cols), xsf)


def _bf16_bits(v: float) -> int:
    return int(torch.tensor([v], dtype=torch.float32).to(torch.bfloat16).view(torch.int16).item()) & 0xFFFF


@pytest.mark.parametrize("amax", [1344.0, 3.0, 2.6875])
def test_quantize_every_bf16_against_every_scale(nb, amax):
    """Every positive bf16 magnitude in [m/64, m], both signs, in blocks whose
    maximum m sets each of the 126 non-zero scale bytes (global amax fixed,
    so gs = amax/2688): nibbles and scales bit-exact against the oracle's
    true division (the kernels divide by a reciprocal plus a correction
    step)."""
    gs = float(onv.global_scale(np.float32(amax)))
    top = _bf16_bits(amax)
    blocks = [[top] * 16]                            # fixes the global amax
    for s in range(1, 127):
        m = float(onv.e4m3_decode(np.array([s], dtype=np.uint8))[0]) * 6.0 * gs
        hi = _bf16_bits(m)
        lo = _bf16_bits(m / 64.0)
        if hi == 0 or hi > top:
            continue
        vals = list(range(lo, hi + 1))
        for c0 in range(0, len(vals), 15):
            chunk = vals[c0:c0 + 15]
            chunk += [hi] * (15 - len(chunk))
            blocks.append([b | (0x8000 if i % 2 else 0) for i, b in enumerate([hi] + chunk)])
    cols = 1024
    while len(blocks) % (cols // 16):
        blocks.append([0] * 16)
    bits = np.asarray(blocks, dtype=np.uint16).reshape(-1, cols)
    x = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16)
    rows = x.shape[0]
    q, sf_row, sf_mma, gsg = nb.quantize_act(x.to(DEV))
    torch.cuda.synchronize()
    xq, xsf, xgs = onv.quantize_rows(x.float().numpy())
    assert float(xgs) == np.float32(gs)
    assert gsg.item() == float(xgs)
    assert len(set(xsf.reshape(-1).tolist())) > 100          # scales really spread
    assert np.array_equal(sf_row.cpu().numpy(), xsf)
    assert np.array_equal(q.cpu().numpy(), xq)
    assert np.array_equal(unstage(sf_mma.cpu().numpy(), rows, cols), xsf)


def test_quantize_fp32_large_random(nb):
    """12.6 M heavy-tailed fp32 values (the requantisation's input type):
    bit-exact against the oracle."""
    g = torch.Generator().manual_seed(11)
    rows, cols = 4096, 3072
    x = torch.randn((rows, cols), generator=g)
    x = x / torch.sqrt((torch.randn((3, rows, cols), generator=g) ** 2).sum(0) / 3)
    q, sf_row, _, gs = nb.quantize_act(x.to(DEV))
    torch.cuda.synchronize()
    xq, xsf, xgs = onv.quantize_rows(x.numpy())
    assert gs.item() == float(xgs)
    assert np.array_equal(sf_row.cpu().numpy(), xsf)
    assert np.array_equal(q.cpu().numpy(), xq)


def test_quantize_act_ties_and_signs(nb):
    """Blocks whose values sit exactly on E2M1 rounding ties, saturation and
    negative values that round to zero."""
    # block max 6 with amax 6 -> gs = 6/2688, sf = 448, d = 6/6 = 1 exactly?
    # (fp32 rounding of gs makes d within 1 ulp of 1; the ties below are
    # offset accordingly by the oracle, which takes the same fp32 decisions)
    ties = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0]
    row = []
    for s in (1, -1):
        row += [s * t for t in ties]
    row += [-0.1, -1e-8, 0.0, -0.0, 6.0, -6.0] + [0.3] * 10
    x = torch.tensor([row[:32]], dtype=torch.float32)
    x = torch.cat([x, torch.zeros((1, 32))], 1)
    q, sf_row, _, gs = nb.quantize_act(x.to(DEV))
    xq, xsf, xgs = onv.quantize_rows(x.numpy())
    assert np.array_equal(q.cpu().numpy(), xq)
    assert np.array_equal(sf_row.cpu().numpy(), xsf)


def test_quantize_act_empty_and_zero(nb):
    x = torch.zeros((5, 128), dtype=torch.bfloat16, device=DEV)
    q, sf_row, _, gs = nb.quantize_act(x)
    assert gs.item() == 1.0 and int(q.sum()) == 0 and int(sf_row.sum()) == 0
    x0 = torch.zeros((0, 128), dtype=torch.bfloat16, device=DEV)
    q, sf_row, _, gs = nb.quantize_act(x0)
    assert gs.item() == 1.0


@pytest.mark.parametrize("name,rowmajor", [("small", False), ("medium", False),
                                           ("medium", True), ("waves", True)])
def test_quantize_scatter_into_slot_layout(nb, name, rowmajor):
    """Token rows quantised into their k slot rows.  With both scale layouts
    asked for (and more than the single-CTA size), the staged scales come
    from a second pass over the row-major ones: both must match the oracle
    on every slot row, whatever the padding rows hold."""
    cfg = syn.CONFIGS[name]
    x = syn.draw_activations(cfg)
    ids, _ = syn.draw_routing(cfg)
    r = nb.route_permute(ids.to(DEV), cfg.E)
    q, sf_row, sf_mma, gs = nb.quantize_act(x.to(DEV), row_dst=r.slot_of, fanout=cfg.k,
                                            out_rows=r.rows, rowmajor_sf=rowmajor)
    xq, xsf, xgs = onv.quantize_rows(x.float().numpy())
    slot_of = r.slot_of.cpu().numpy().reshape(cfg.T, cfg.k)
    qn = q.cpu().numpy()
    sfn = unstage(sf_mma.cpu().numpy(), r.rows, cfg.H)
    rows = slot_of.reshape(-1)
    tok = np.repeat(np.arange(cfg.T), cfg.k)
    assert np.array_equal(qn[rows], xq[tok])
    assert np.array_equal(sfn[rows], xsf[tok])
    if rowmajor:
        assert np.array_equal(sf_row.cpu().numpy()[rows], xsf[tok])
    assert gs.item() == float(xgs)


# ---------------------------------------------------------------- routing --

def _check_route(nb, ids, E):
    T, k = ids.shape
    r = nb.route_permute(ids.to(DEV), E)
    torch.cuda.synchronize()
    o = omoe.route(ids.numpy(), E)
    p = omoe.padded_layout(o)
    assert np.array_equal(r.expert_counts.cpu().numpy(), o["counts"])
    assert np.array_equal(r.expert_offsets.cpu().numpy(), p["row_offsets"])
    rt = r.row_token.cpu().numpy()[:r.rows]
    want_rt = -np.ones(r.rows, dtype=np.int64)
    want_rt[:len(p["row_token"])] = p["row_token"]
    assert np.array_equal(rt, want_rt)
    if T * k:
        assert np.array_equal(r.slot_of.cpu().numpy()[:T * k], p["row_of"])
    return r


@pytest.mark.parametrize("name", ["tiny", "small", "medium", "decode1", "decode64",
                                  "prefill4k", "prefill16k"])
def test_route_bit_exact(nb, name):
    cfg = syn.CONFIGS[name]
    ids, _ = syn.draw_routing(cfg)
    _check_route(nb, ids, cfg.E)


@pytest.mark.parametrize("counts,k", [
    ([0, 1, 127, 128, 129, 0, 256, 257, 2], 2),
    ([5000, 4999, 3, 0], 2),
    ([0, 0, 0, 8], 1),
])
def test_route_edge_counts(nb, counts, k):
    ids, _ = syn.routing_with_counts(counts, k)
    _check_route(nb, ids, len(counts))


def test_route_empty(nb):
    ids = torch.zeros((0, 4), dtype=torch.int32)
    r = nb.route_permute(ids.to(DEV), 6)
    assert r.expert_offsets.cpu().tolist() == [0] * 7
    assert r.expert_counts.cpu().tolist() == [0] * 6


# ---------------------------------------------------------------- weights --

@pytest.mark.parametrize("E,K,N", [(2, 64, 128), (3, 256, 384), (1, 7168, 256)])
def test_quantize_weights_bit_exact(nb, E, K, N):
    cfg = syn.MoEConfig("wq", E=E, H=K, I=N // 2, T=1, k=1, routing="uniform")
    W = torch.stack([syn.draw_weight(cfg, 1, e) for e in range(E)])
    q, sf, gs = nb.quantize_weights(W.to(DEV))
    torch.cuda.synchronize()
    for e in range(E):
        oq, osf, ogs = onv.quantize_weight(W[e].numpy())
        assert gs[e].item() == float(ogs)
        assert np.array_equal(q[e].cpu().numpy(), oq)
        assert np.array_equal(sf[e].cpu().numpy(), osf)


@pytest.mark.parametrize("E,K,N", [(2, 512, 256), (3, 128, 384), (1, 768, 128)])
def test_prepare_weights_layout(nb, E, K, N):
    """B tiles: byte j of row n in K-stage kt at ((n/128)*KT + kt)*16384 +
    (n%128)*128 + j, zero past K/2; scales staged per the header formula."""
    rng = np.random.default_rng(4)
    q = rng.integers(0, 256, (E, K // 2, N), dtype=np.uint8)
    sf = rng.integers(0, 127, (E, K // 16, N), dtype=np.uint8)
    qo, sfo = nb.prepare_weights(torch.from_numpy(q).to(DEV), torch.from_numpy(sf).to(DEV))
    KT = -(-K // 256)
    rows = q.transpose(0, 2, 1).reshape(E * N, K // 2)          # K-major rows
    padded = np.zeros((E * N, KT * 128), np.uint8)
    padded[:, :K // 2] = rows
    want = padded.reshape(E * N // 128, 128, KT, 128).transpose(0, 2, 1, 3).reshape(-1)
    assert np.array_equal(qo.cpu().numpy(), want)
    sf_rows = sf.transpose(0, 2, 1).reshape(E * N, K // 16)
    assert np.array_equal(unstage(sfo.cpu().numpy(), E * N, K), sf_rows)


# ------------------------------------------------------------------ GEMM --

def _l1_only(nb, xq_rows, xsf_rows, w1q, w1sf, gs_x=1.0, gs_w=None):
    """Run the forward on crafted slot-layout activations for one expert
    (k = 1, rows = tokens) and return the alpha-scaled L1 tap."""
    M, H2 = xq_rows.shape
    H = 2 * H2
    E, _, N1 = w1q.shape
    I = N1 // 2
    ids = torch.zeros((M, 1), dtype=torch.int32)
    r = nb.route_permute(ids.to(DEV), E)
    rows = r.rows
    xq = np.zeros((rows, H2), np.uint8)
    xq[:M] = xq_rows
    sfr = np.zeros((rows, H // 16), np.uint8)
    sfr[:M] = xsf_rows
    gs1 = torch.full((E,), 1.0 if gs_w is None else gs_w, dtype=torch.float32)
    # L2 weights: zeros (their output is not inspected here)
    w2q = torch.zeros((E, I // 2, H), dtype=torch.uint8)
    w2sf = torch.full((E, I // 16, H), 0x38, dtype=torch.uint8)
    w1q, w1sf = np.ascontiguousarray(w1q), np.ascontiguousarray(w1sf)
    pw = nb.PreparedWeights.from_checkpoint(torch.from_numpy(w1q).to(DEV),
                                            torch.from_numpy(w1sf).to(DEV), gs1.to(DEV),
                                            w2q.to(DEV), w2sf.to(DEV), gs1.to(DEV))
    tap = torch.zeros((rows, N1), dtype=torch.float32, device=DEV)
    nb.nvfp4_forward(pw, torch.from_numpy(xq).to(DEV), torch.from_numpy(stage(sfr)).to(DEV),
                     torch.tensor([gs_x], dtype=torch.float32, device=DEV), r,
                     taps={"l1_out": tap})
    torch.cuda.synchronize()
    return tap.cpu().numpy()[:M]


def _rand_nibbles(rng, shape):
    return rng.integers(0, 16, shape, dtype=np.uint8)


@pytest.mark.parametrize("M,H,I", [(128, 256, 128), (200, 512, 256)])
def test_gemm_exact_integer_regime(nb, M, H, I):
    """All scales 1.0 and global scales 1: every product is a multiple of
    1/4 and every sum fits in 24 bits, so the fp32 result is exact."""
    rng = np.random.default_rng(M + H)
    an = _rand_nibbles(rng, (M, H))
    wn = _rand_nibbles(rng, (1, H, 2 * I))
    aq = onv.pack_nibbles(an)
    w1q = np.stack([onv.pack_nibbles(wn[0].T).T])
    asf = np.full((M, H // 16), 0x38, np.uint8)
    w1sf = np.full((1, H // 16, 2 * I), 0x38, np.uint8)
    got = _l1_only(nb, aq, asf, w1q, w1sf)
    want = omoe.block_scaled_matmul(aq, asf, w1q[0], w1sf[0])
    assert np.array_equal(got.astype(np.float64), want)


def test_gemm_scale_layout_every_row_and_group(nb):
    """Every (row, k-group) scale of A and every (column, k-group) scale of B
    set independently to 1 or 2: the exact result pins the staged scale
    layout at every position (generalised single-SF probe)."""
    rng = np.random.default_rng(21)
    M, H, I = 160, 512, 128
    an = _rand_nibbles(rng, (M, H))
    wn = _rand_nibbles(rng, (1, H, 2 * I))
    aq = onv.pack_nibbles(an)
    w1q = np.stack([onv.pack_nibbles(wn[0].T).T])
    asf = rng.choice(np.array([0x38, 0x40], np.uint8), (M, H // 16))
    w1sf = rng.choice(np.array([0x38, 0x40], np.uint8), (1, H // 16, 2 * I))
    got = _l1_only(nb, aq, asf, w1q, w1sf)
    want = omoe.block_scaled_matmul(aq, asf, w1q[0], w1sf[0])
    assert np.array_equal(got.astype(np.float64), want)


@pytest.mark.parametrize("m,g", [(0, 0), (0, 3), (37, 5), (100, 17), (127, 31)])
def test_gemm_single_scale_probe(nb, m, g):
    """SFA[m, g] = 2 changes only row m, by exactly k-group g's contribution
    (the pages' coordinate probe, for k-groups other than 0 too)."""
    rng = np.random.default_rng(m * 100 + g)
    M, H, I = 128, 512, 128
    an = _rand_nibbles(rng, (M, H))
    wn = _rand_nibbles(rng, (1, H, 2 * I))
    aq = onv.pack_nibbles(an)
    w1q = np.stack([onv.pack_nibbles(wn[0].T).T])
    asf = np.full((M, H // 16), 0x38, np.uint8)
    w1sf = np.full((1, H // 16, 2 * I), 0x38, np.uint8)
    base = _l1_only(nb, aq, asf, w1q, w1sf)
    asf2 = asf.copy()
    asf2[m, g] = 0x40
    probe = _l1_only(nb, aq, asf2, w1q, w1sf)
    delta = probe.astype(np.float64) - base
    A = onv.e2m1_decode(an)
    W = onv.e2m1_decode(wn[0])
    want = np.zeros_like(delta)
    want[m] = A[m, 16 * g:16 * g + 16] @ W[16 * g:16 * g + 16]
    assert np.array_equal(delta, want)


# ---------------------------------------------------------------- reduce --

@pytest.mark.parametrize("slot_dtype", [torch.float32, torch.float16, torch.bfloat16],
                         ids=["slot_f32", "slot_f16", "slot_bf16"])
@pytest.mark.parametrize("T,k,H,dtype", [(5, 2, 256, torch.float32), (64, 8, 7168, torch.bfloat16),
                                         (3, 3, 1024, torch.bfloat16)])
def test_unpermute_reduce(nb, T, k, H, dtype, slot_dtype):
    """Slot rows in fp32 or a 16-bit type: the 16-bit values widen exactly,
    so the oracle reduces the stored values themselves."""
    g = torch.Generator().manual_seed(T * k)
    rows = T * k + 7
    so = (torch.randn((rows, H), generator=g) * 3).to(slot_dtype)
    slot_of = torch.randperm(rows, generator=g)[:T * k].to(torch.int32)
    w = torch.rand((T, k), generator=g)
    y = nb.unpermute_reduce(so.to(DEV), slot_of.to(DEV), w.to(DEV), out_dtype=dtype)
    want = omoe.unpermute_reduce(so.double().numpy(), slot_of.numpy(), w.numpy())
    got = y.float().cpu().numpy()
    if dtype == torch.float32:
        assert_rows_close(got, want, "y")
    else:
        # one bf16 rounding of the fp32 sum: within half a bf16 ulp of the
        # exact value plus the fp32 accumulation error
        ulp_half = np.abs(want) * 2.0 ** -8
        assert np.all(np.abs(got - want) <= ulp_half + 1e-5 * np.abs(want).max(1, keepdims=True))
