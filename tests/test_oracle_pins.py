"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test runs against both oracles, the plain C++ one (oracle/
nvfp4_oracle.cpp, the oracle of record) and the numpy one, and ties one
oracle function to something other than itself: values
the pages print (tests/golden/, each file citing its passage), closed forms,
a library routine for a special case (torch's float8_e4m3fn view and cast),
or pure-Python brute force on tiny inputs with a different loop structure.
No GPU is needed.
"""
import math
import os
import random
import struct

import numpy as np
import pytest
import torch

from oracle import moe, nvfp4
from oracle import cpp as _cpp
from oracle import moe as _np_moe, nvfp4 as _np_nvfp4

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module", autouse=True, params=["cpp", "numpy"])
def backend(request):
    """Every pin runs against both oracles: the plain C++ one (the oracle of
    record) and the numpy one (its cross-check).  The pins name the two
    modules ``nvfp4`` and ``moe``; this rebinds them for each pass."""
    global nvfp4, moe
    if request.param == "cpp":
        nvfp4, moe = _cpp.nvfp4, _cpp.moe
    else:
        nvfp4, moe = _np_nvfp4, _np_moe
    yield request.param
    nvfp4, moe = _np_nvfp4, _np_moe


def golden_rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


# ------------------------------------------------------------------ E2M1 --

def test_e2m1_decode_matches_pages_table():
    rows = golden_rows("e2m1_table.txt")
    assert len(rows) == 16
    for code, val in rows:
        got = nvfp4.e2m1_decode(np.array([int(code)]))[0]
        assert got == float(val)
        assert math.copysign(1.0, got) == math.copysign(1.0, float(val))


def test_e2m1_encode_is_inverse_on_all_codes():
    codes = np.arange(16, dtype=np.uint8)
    vals = nvfp4.e2m1_decode(codes)
    assert np.array_equal(nvfp4.e2m1_encode(vals), codes)


@pytest.mark.parametrize("v,code", [
    (0.25, 0), (0.75, 2), (1.25, 2), (1.75, 4), (2.5, 4), (3.5, 6), (5.0, 6),
    (-0.25, 8), (-0.75, 10), (-1.25, 10), (-1.75, 12), (-2.5, 12), (-3.5, 14), (-5.0, 14),
    (0.2499, 0), (0.2501, 1), (4.99, 6), (5.01, 7), (6.0, 7), (6.5, 7), (1e30, 7),
    (-1e30, 15), (-1e-9, 8), (-0.0, 8), (0.0, 0),
])
def test_e2m1_ties_to_even_and_saturation(v, code):
    assert int(nvfp4.e2m1_encode(np.array([v], dtype=np.float64))[0]) == code


def test_e2m1_encode_brute_force():
    rng = random.Random(1)
    mags = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    vals = [rng.uniform(-7.0, 7.0) for _ in range(3000)]
    vals += [m + s for m in mags for s in (0.0, 1e-7, -1e-7)]
    vals += [(a + b) / 2 for a, b in zip(mags, mags[1:])]
    vals += [-x for x in vals]
    got = nvfp4.e2m1_encode(np.array(vals, dtype=np.float64))
    for v, c in zip(vals, got):
        a = min(abs(v), 6.0)
        best = None
        for i, m in enumerate(mags):
            d = abs(a - m)
            if best is None or d < best[0] or (d == best[0] and i % 2 == 0 and best[1] % 2 == 1):
                best = (d, i)
        want = best[1] | (8 if math.copysign(1.0, v) < 0 else 0)
        assert int(c) == want, (v, int(c), want)


# ------------------------------------------------------------------ E4M3 --

@pytest.mark.parametrize("byte,val", [
    (0x00, 0.0), (0x01, 2.0 ** -9), (0x07, 7 * 2.0 ** -9), (0x08, 2.0 ** -6),
    (0x38, 1.0), (0x3F, 1.875), (0x40, 2.0), (0x7E, 448.0), (0x80, -0.0),
    (0xB8, -1.0), (0xFE, -448.0),
])
def test_e4m3_decode_spot_values(byte, val):
    got = nvfp4.e4m3_decode(np.array([byte]))[0]
    assert got == val and math.copysign(1, got) == math.copysign(1, val)


def test_e4m3_decode_nan_codes():
    assert np.isnan(nvfp4.e4m3_decode(np.array([0x7F, 0xFF]))).all()


def test_e4m3_decode_matches_torch_view():
    """Reinterpreting the byte (not converting its integer value) — the
    view-vs-convert lesson of the FP8 commit message — equals torch's
    float8_e4m3fn bit-pattern view for every non-NaN byte."""
    b = np.array([x for x in range(256) if x not in (0x7F, 0xFF)], dtype=np.uint8)
    ref = torch.from_numpy(b).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = nvfp4.e4m3_decode(b)
    assert np.array_equal(got, ref)
    # value conversion of the byte's integer is a different (wrong) thing:
    # 0x3F converted as the number 63 is not the byte 0x3F
    conv = torch.tensor([63.0]).to(torch.float8_e4m3fn).view(torch.uint8).item()
    assert conv != 0x3F and nvfp4.e4m3_decode(np.array([0x3F]))[0] == 1.875


def _e4m3_sweep():
    vals = nvfp4.e4m3_decode(np.arange(0, 127))
    mids = (vals[:-1] + vals[1:]) / 2              # exact ties
    rng = np.random.default_rng(3)
    rand = rng.uniform(0, 448, 20000)
    small = rng.uniform(0, 2.0 ** -5, 20000)       # subnormal region
    near = np.concatenate([np.nextafter(mids.astype(np.float32), np.float32(0)),
                           np.nextafter(mids.astype(np.float32), np.float32(1e9))])
    x = np.concatenate([vals, mids, rand, small, near, [2.0 ** -10, 3 * 2.0 ** -11]])
    return x.astype(np.float32)


def test_e4m3_encode_matches_torch_cast():
    x = _e4m3_sweep()
    assert np.all(x.astype(np.float64) <= 448.0)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = nvfp4.e4m3_encode_nonneg(x)
    assert np.array_equal(got, ref)


def test_e4m3_encode_identity_and_saturation():
    b = np.arange(0, 127, dtype=np.uint8)
    assert np.array_equal(nvfp4.e4m3_encode_nonneg(nvfp4.e4m3_decode(b)), b)
    sat = nvfp4.e4m3_encode_nonneg(np.array([448.0, 448.5, 463.9, 464.0, 1e9]))
    assert (sat == 0x7E).all()
    with pytest.raises(ValueError):
        nvfp4.e4m3_encode_nonneg(np.array([-1.0]))


# --------------------------------------------------------------- packing --

def test_packing_matches_pages():
    for ne, no, byte in golden_rows("packing.txt"):
        got = nvfp4.pack_nibbles(np.array([int(ne), int(no)], dtype=np.uint8))
        assert got.tolist() == [int(byte)]
        back = nvfp4.unpack_nibbles(got)
        assert back.tolist() == [int(ne), int(no)]


@pytest.mark.parametrize("c", [0, 1, 2, 15, 16, 31, 62, 63])
def test_one_hot_nibble_lands_at_its_column(c):
    """A single nonzero element at column c comes back at exactly column c,
    in the low nibble of byte c/2 when c is even and the high nibble when odd."""
    K = 64
    v = np.zeros((3, K), dtype=np.float32)
    v[1, c] = -2.5
    q, sf, gs = nvfp4.quantize_rows(v)
    nz = np.argwhere(q != 0)
    assert nz.tolist() == [[1, c // 2]]
    byte = int(q[1, c // 2])
    nib = (byte >> 4) if c % 2 else (byte & 0xF)
    other = (byte & 0xF) if c % 2 else (byte >> 4)
    assert nib == 0xF and other == 0          # -6 * d, the block's max
    deq = nvfp4.dequantize_rows(q, sf) * float(gs)
    assert np.argwhere(deq != 0).tolist() == [[1, c]]
    assert deq[1, c] == pytest.approx(-2.5, rel=1e-6)


def test_weight_unpack_interleaves_along_k():
    K2, N = 3, 4
    p = np.zeros((K2, N), dtype=np.uint8)
    p[1, 2] = 0x3A                     # (2,2) <- 0xA, (3,2) <- 0x3
    nib = nvfp4.unpack_weight_k(p)
    assert nib.shape == (2 * K2, N)
    assert np.argwhere(nib != 0).tolist() == [[2, 2], [3, 2]]
    assert nib[2, 2] == 0xA and nib[3, 2] == 0x3


def test_weight_layout_shapes_match_pages():
    """Checkpoint layout (K/2, N) bytes and (K/16, N) scales for the
    48-expert layer (H=7168, I=3072): K and N axes pinned on a narrow slice."""
    shapes = {r[0]: tuple(int(x) for x in r[1:]) for r in golden_rows("weight_shapes.txt")}
    H, I = 7168, 3072
    rng = np.random.default_rng(0)
    for layer, (K, N) in (("l1", (H, 2 * I)), ("l2", (I, H))):
        w = rng.standard_normal((K, 16)).astype(np.float32)
        q, sf, gs = nvfp4.quantize_weight(w)
        assert q.shape == (shapes[layer + "_w"][1], 16)
        assert sf.shape == (shapes[layer + "_sf"][1], 16)
        assert shapes[layer + "_w"][2] == N and shapes[layer + "_sf"][2] == N
        assert shapes[layer + "_w"][0] == shapes[layer + "_sf"][0] == 48


# ------------------------------------------------------------- quantiser --

def test_constant_block_hits_the_top_codes():
    for c in (1e-3, 0.37, 1.0, 5.5, 1234.5):
        v = np.full((2, 32), c, dtype=np.float32)
        v[1] *= -1
        q, sf, gs = nvfp4.quantize_rows(v)
        assert (sf == 0x7E).all()                        # 448
        assert (q[0] == 0x77).all() and (q[1] == 0xFF).all()   # +6 / -6
        deq = nvfp4.dequantize_rows(q, sf) * float(gs)
        assert np.allclose(np.abs(deq), c, rtol=1e-6)


def test_e2m1_grid_block_is_reproduced():
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6] * 2, dtype=np.float32)
    for j in (-3, 0, 5):
        v = (grid * np.float32(2.0 ** j))[None, :].astype(np.float32)
        v[0, 1::2] *= -1
        q, sf, gs = nvfp4.quantize_rows(v)
        nib = nvfp4.unpack_nibbles(q)[0]
        assert np.array_equal(np.abs(nvfp4.e2m1_decode(nib)), np.abs(grid))
        deq = nvfp4.dequantize_rows(q, sf) * float(gs)
        assert np.allclose(deq, v, rtol=1e-6, atol=0)


def _grid_half_step(a):
    # half the distance to the neighbouring representable magnitudes
    return np.where(a < 2, 0.25, np.where(a < 4, 0.5, 1.0))


@pytest.mark.parametrize("dist", ["normal", "student_t", "tiny_blocks"])
def test_roundtrip_error_bound(dist):
    rng = np.random.default_rng(7)
    if dist == "normal":
        v = rng.normal(0, 1.5, (64, 256))
    elif dist == "student_t":
        v = rng.standard_t(3, (64, 256)) * 0.866
    else:                                # blocks far below the tensor amax
        v = rng.normal(0, 1, (64, 256)) * np.repeat(10.0 ** rng.uniform(-7, 0, (64, 16)), 16, axis=1)
    v = v.astype(np.float32)
    q, sf, gs = nvfp4.quantize_rows(v)
    d = nvfp4.e4m3_decode(sf).astype(np.float64) * float(gs)
    deq = nvfp4.dequantize_rows(q, sf) * float(gs)
    dd = np.repeat(d, 16, axis=1)
    ratio = np.abs(v.astype(np.float64)) / np.where(dd == 0, np.inf, dd)
    bound = np.where(ratio > 6, np.abs(v) - 6 * dd, _grid_half_step(ratio) * dd)
    # a block whose scale underflowed to 0 had b / (6 gs) <= 2^-10
    bound = np.where(dd == 0, 6 * float(gs) * 2.0 ** -10, bound)
    err = np.abs(deq - v.astype(np.float64))
    assert np.all(err <= bound * (1 + 1e-6) + 1e-30)
    # scale choice: b/(6 gs) rounded to the nearest E4M3 value (relative
    # error <= 2^-4 in the normal range)
    b = np.abs(v.reshape(64, 16, 16)).max(-1).astype(np.float64)
    target = b / (6 * float(gs))
    normal = target >= 2.0 ** -6
    rel = np.abs(nvfp4.e4m3_decode(sf)[normal] - target[normal]) / target[normal]
    assert rel.max() <= 2.0 ** -4 * (1 + 1e-6)


def test_global_scale_matches_pages_roundtrip_numbers():
    vals = dict((r[0], float(r[1])) for r in golden_rows("roundtrip.txt"))
    gs = nvfp4.global_scale(vals["reconstructed_amax"])
    assert float(f"{gs:.1e}") == vals["igs"]
    # gs * 2688 recovers amax to within fp32 rounding
    for amax in (vals["reconstructed_amax"], 8.625, 34.5, 1e-3, 3e4):
        g = nvfp4.global_scale(amax)
        assert abs(float(g) * 2688.0 - amax) <= 2 * np.spacing(np.float32(amax))


def test_zero_cases():
    q, sf, gs = nvfp4.quantize_rows(np.zeros((2, 32), np.float32))
    assert gs == 1.0 and (q == 0).all() and (sf == 0).all()
    # a block far below the tensor amax underflows its scale to 0 -> nibbles 0
    v = np.zeros((1, 32), np.float32)
    v[0, 0] = 1000.0
    v[0, 16:] = -1e-6
    q, sf, gs = nvfp4.quantize_rows(v)
    assert sf[0, 1] == 0 and (q[0, 8:] == 0).all()


def test_small_negative_keeps_sign_bit():
    v = np.zeros((1, 16), np.float32)
    v[0, 0] = 6.0
    v[0, 3] = -0.1                      # rounds to magnitude 0
    q, _, _ = nvfp4.quantize_rows(v)
    nib = nvfp4.unpack_nibbles(q)[0]
    assert nib[3] == 0x8 and nib[0] == 0x7


def test_quantizer_matches_scalar_restatement():
    """Scalar, per-element restatement with fp32 scalars and a brute-force
    nearest search; different loop structure from the vectorised oracle."""
    rng = np.random.default_rng(11)
    v = (rng.standard_t(3, (3, 64)) * 2).astype(np.float32)
    q, sf, gs = nvfp4.quantize_rows(v)
    f32 = np.float32
    amax = f32(0)
    for x in v.ravel():
        amax = max(amax, abs(x))
    g = f32(amax / f32(2688))
    assert g == gs
    e4 = [(float(nvfp4.e4m3_decode(np.array([b]))[0]), b) for b in range(127)]
    mags = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    for r in range(3):
        for blk in range(4):
            xs = v[r, blk * 16:(blk + 1) * 16]
            b = f32(0)
            for x in xs:
                b = max(b, abs(x))
            t = float(f32(b / f32(f32(6) * g)))
            t = min(t, 448.0)
            best = min(e4, key=lambda p: (abs(p[0] - t), p[1] % 2))
            assert sf[r, blk] == best[1]
            d = f32(f32(best[0]) * g)
            for i, x in enumerate(xs):
                a = min(abs(float(f32(x / d))), 6.0)
                idx = min(range(8), key=lambda j: (abs(mags[j] - a), j % 2))
                code = idx | (8 if x < 0 or (x == 0 and math.copysign(1, x) < 0) else 0)
                byte = int(q[r, (blk * 16 + i) // 2])
                got = (byte >> 4) if i % 2 else (byte & 0xF)
                assert got == code


# ------------------------------------------------------------------ GEMM --

def _rand_nvfp4(rng, R, K):
    v = rng.normal(0, 1, (R, K)).astype(np.float32)
    return nvfp4.quantize_rows(v)


def _brute_block_gemm(aq, asf, wq, wsf):
    """Pure-Python blockwise sum: sum_g sfa*sfw*sum_{i in g} a_i*w_i."""
    M, K = aq.shape[0], aq.shape[1] * 2
    N = wq.shape[1]
    tab = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]

    def nib_a(m, kk):
        byte = int(aq[m, kk // 2])
        n = (byte >> 4) if kk % 2 else (byte & 15)
        return -tab[n & 7] if n & 8 else tab[n & 7]

    def nib_w(kk, n):
        byte = int(wq[kk // 2, n])
        x = (byte >> 4) if kk % 2 else (byte & 15)
        return -tab[x & 7] if x & 8 else tab[x & 7]

    def e4(b):
        b = int(b)
        e, m = (b >> 3) & 15, b & 7
        return (m / 8) * 2 ** -6 if e == 0 else (1 + m / 8) * 2 ** (e - 7)

    out = np.zeros((M, N))
    for m in range(M):
        for n in range(N):
            s = 0.0
            for g in range(K // 16):
                part = 0.0
                for kk in range(16 * g, 16 * g + 16):
                    part += nib_a(m, kk) * nib_w(kk, n)
                s += e4(asf[m, g]) * e4(wsf[g, n]) * part
            out[m, n] = s
    return out


def test_gemm_matches_brute_force():
    rng = np.random.default_rng(5)
    aq, asf, _ = _rand_nvfp4(rng, 5, 64)
    wq, wsf, _ = nvfp4.quantize_weight(rng.normal(0, 1, (64, 7)).astype(np.float32))
    got = moe.block_scaled_matmul(aq, asf, wq, wsf)
    want = _brute_block_gemm(aq, asf, wq, wsf)
    assert np.allclose(got, want, rtol=1e-12, atol=1e-12)


def test_constant_scale_gemm_is_plain_matmul():
    """All block scales 1.0 (0x38): the GEMM is the plain matmul of the E2M1
    values (the pages' constant-scale test, cosine 1)."""
    rng = np.random.default_rng(6)
    M, K, N = 4, 64, 6
    an = rng.integers(0, 16, (M, K), dtype=np.uint8)
    wn = rng.integers(0, 16, (K, N), dtype=np.uint8)
    aq = nvfp4.pack_nibbles(an)
    wq = nvfp4.pack_nibbles(wn.T).T.copy()        # bytes pair along K
    asf = np.full((M, K // 16), 0x38, np.uint8)
    wsf = np.full((K // 16, N), 0x38, np.uint8)
    got = moe.block_scaled_matmul(aq, asf, wq, wsf)
    tab = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    dec = lambda c: -tab[c & 7] if c & 8 else tab[c & 7]
    for m in range(M):
        for n in range(N):
            want = sum(dec(int(an[m, kk])) * dec(int(wn[kk, n])) for kk in range(K))
            assert got[m, n] == want          # exact: multiples of 1/4
    assert moe.cosine(got, got) == 1.0


@pytest.mark.parametrize("side", ["A", "B"])
def test_single_scale_probes_every_row_and_group(side):
    """Doubling one block scale (1.0 -> 2.0) changes only its row (A) or
    column (B), by exactly that k-group's contribution — for every row/column
    and every k-group, not only k-group 0."""
    rng = np.random.default_rng(8)
    M, K, N = 3, 64, 4
    an = rng.integers(0, 16, (M, K), dtype=np.uint8)
    wn = rng.integers(0, 16, (K, N), dtype=np.uint8)
    aq = nvfp4.pack_nibbles(an)
    wq = nvfp4.pack_nibbles(wn.T).T.copy()
    asf = np.full((M, K // 16), 0x38, np.uint8)
    wsf = np.full((K // 16, N), 0x38, np.uint8)
    base = moe.block_scaled_matmul(aq, asf, wq, wsf)
    A = nvfp4.e2m1_decode(an)
    W = nvfp4.e2m1_decode(wn)
    rows = M if side == "A" else N
    for r in range(rows):
        for g in range(K // 16):
            a2, w2 = asf.copy(), wsf.copy()
            if side == "A":
                a2[r, g] = 0x40
            else:
                w2[g, r] = 0x40
            delta = moe.block_scaled_matmul(aq, a2, wq, w2) - base
            want = np.zeros_like(delta)
            sl = slice(16 * g, 16 * g + 16)
            if side == "A":
                want[r, :] = A[r, sl] @ W[sl, :]
            else:
                want[:, r] = A[:, sl] @ W[sl, r]
            assert np.array_equal(delta, want), (r, g)


def test_alpha_is_linear_per_expert():
    rng = np.random.default_rng(9)
    aq, asf, gs_a = _rand_nvfp4(rng, 3, 64)
    wq, wsf, gs_w = nvfp4.quantize_weight(rng.normal(0, 1, (64, 8)).astype(np.float32))
    base = moe.expert_l1(aq, asf, gs_a, wq, wsf, gs_w)
    assert np.array_equal(moe.expert_l1(aq, asf, gs_a, wq, wsf, np.float32(2 * gs_w)), 2 * base)
    assert np.array_equal(moe.expert_l1(aq, asf, np.float32(4 * gs_a), wq, wsf, gs_w), 4 * base)


def test_gate_up_scales_per_column_alpha():
    """Separate gate/up global scales (Debug Log, code-review point 5): the
    up half scales with gs_up alone, the gate half with gs_gate alone, and
    the per-column alpha equals the pages' correction up *= gs_up / gs_gate
    applied on top of one alpha."""
    rng = np.random.default_rng(10)
    aq, asf, gs_a = _rand_nvfp4(rng, 3, 64)
    wq, wsf, gs_w = nvfp4.quantize_weight(rng.normal(0, 1, (64, 8)).astype(np.float32))
    one = moe.expert_l1(aq, asf, gs_a, wq, wsf, gs_w)
    same = moe.expert_l1(aq, asf, gs_a, wq, wsf, (gs_w, gs_w))
    assert np.array_equal(one, same)
    pair = moe.expert_l1(aq, asf, gs_a, wq, wsf, (gs_w, np.float32(2 * gs_w)))
    assert np.array_equal(pair[:, :4], one[:, :4])
    assert np.array_equal(pair[:, 4:], 2 * one[:, 4:])
    g_gate, g_up = np.float32(gs_w), np.float32(0.37 * gs_w)
    pc = moe.expert_l1(aq, asf, gs_a, wq, wsf, (g_gate, g_up))
    corrected = moe.expert_l1(aq, asf, gs_a, wq, wsf, g_gate)
    corrected[:, 4:] *= float(g_up) / float(g_gate)
    assert np.allclose(pc, corrected, rtol=1e-13, atol=0)


def test_split_halves_quantisation():
    """Quantising [gate | up] as two matrices: each half equals quantising it
    alone; with equal half maxima it equals the joint quantisation."""
    rng = np.random.default_rng(12)
    g = rng.normal(0, 1, (64, 8)).astype(np.float32)
    u = rng.normal(0, 3, (64, 8)).astype(np.float32)
    q, sf, gs = moe.quantize_expert_weights([np.concatenate([g, u], 1)], split_halves=True)
    qg, sfg, gg = nvfp4.quantize_weight(g)
    qu, sfu, gu = nvfp4.quantize_weight(u)
    assert gs.shape == (1, 2) and gs[0, 0] == gg and gs[0, 1] == gu
    assert np.array_equal(q[0], np.concatenate([qg, qu], 1))
    assert np.array_equal(sf[0], np.concatenate([sfg, sfu], 1))
    u2 = u / np.abs(u).max() * np.abs(g).max()       # same maximum in both halves
    w = np.concatenate([g, u2.astype(np.float32)], 1)
    qs, sfs, gss = moe.quantize_expert_weights([w], split_halves=True)
    qj, sfj, gj = moe.quantize_expert_weights([w])
    assert gss[0, 0] == gss[0, 1] == gj[0]
    assert np.array_equal(qs, qj) and np.array_equal(sfs, sfj)


def test_silu_closed_forms():
    x = np.array([-30.0, -2.0, -0.5, 0.0, 0.5, 1.0, 3.0, 40.0])
    s = moe.silu(x)
    assert np.allclose(s - moe.silu(-x), x, rtol=0, atol=1e-12)   # silu(x)-silu(-x)=x
    assert s[3] == 0.0
    assert s[5] == pytest.approx(1.0 / (1.0 + math.exp(-1.0)), rel=1e-15)
    assert s[-1] == pytest.approx(40.0, rel=1e-15)
    l1 = np.array([[1.0, -2.0, 3.0, 0.5]])                # [gate | up], I = 2
    h = moe.swiglu(l1)
    assert h.dtype == np.float32
    assert h[0, 0] == np.float32(moe.silu(np.array([1.0]))[0] * 3.0)
    assert h[0, 1] == np.float32(moe.silu(np.array([-2.0]))[0] * 0.5)


# --------------------------------------------------------------- routing --

def _brute_route(ids, E):
    T = len(ids)
    k = len(ids[0]) if T else 0
    slots = []
    for e in range(E):
        for t in range(T):
            for j in range(k):
                if ids[t][j] == e:
                    slots.append((t, j))
    return slots


@pytest.mark.parametrize("T,k,E,seed", [(5, 2, 4, 0), (9, 3, 5, 1), (1, 8, 48, 2), (0, 2, 4, 3)])
def test_route_matches_brute_force(T, k, E, seed):
    rng = random.Random(seed)
    ids = [rng.sample(range(E), k) for _ in range(T)]
    arr = np.array(ids, dtype=np.int32).reshape(T, k)
    r = moe.route(arr, E)
    slots = _brute_route(ids, E)
    assert [int(x) for x in r["slot_token"]] == [t for t, _ in slots]
    assert [int(x) for x in r["slot_flat"]] == [t * k + j for t, j in slots]
    for s, (t, j) in enumerate(slots):
        assert r["slot_of"][t * k + j] == s
    assert r["counts"].sum() == T * k
    assert r["offsets"][-1] == T * k
    for e in range(E):
        assert r["counts"][e] == sum(1 for row in ids for x in row if x == e)


def test_padded_layout():
    ids = np.array([[0, 2], [2, 0], [2, 1]], dtype=np.int32)
    r = moe.route(ids, 4)
    p = moe.padded_layout(r, tile_rows=4)
    # counts 2,1,3,0 -> padded 4,4,4,0
    assert p["row_offsets"].tolist() == [0, 4, 8, 12, 12]
    assert p["row_token"].tolist() == [0, 1, -1, -1, 2, -1, -1, -1, 0, 1, 2, -1]
    assert p["row_of"].tolist() == [0, 8, 9, 1, 10, 4]
    for f, row in enumerate(p["row_of"]):
        assert p["row_token"][row] == f // 2


# ---------------------------------------------------------------- reduce --

def test_reduce_matches_brute_force():
    rng = np.random.default_rng(12)
    T, k, H = 4, 3, 5
    S = T * k
    so = rng.normal(0, 1, (S, H))
    slot_of = rng.permutation(S)
    w = rng.uniform(0, 1, (T, k))
    y = moe.unpermute_reduce(so, slot_of, w)
    for t in range(T):
        for c in range(H):
            acc = 0.0
            for j in range(k):
                acc += w[t, j] * so[slot_of[t * k + j], c]
            assert y[t, c] == acc


def test_round_to_bf16_brute_force():
    allbits = np.arange(0, 1 << 16, dtype=np.uint32)
    f = (allbits << 16).view(np.float32).astype(np.float64)
    ok = np.isfinite(f) & (f > 0) & (np.abs(f) >= 2.0 ** -126)
    pos = np.sort(f[ok])
    bits_of = {v: int(b) for v, b in zip(f[ok], allbits[ok])}
    rng = np.random.default_rng(13)
    xs = list(rng.normal(0, 10, 2000)) + list((pos[100:110] + pos[101:111]) / 2)
    got = nvfp4.round_to_bf16(np.array(xs))
    for x, g in zip(xs, got):
        a = abs(x)
        i = np.searchsorted(pos, a)
        lo, hi = pos[i - 1], pos[i]
        if a - lo < hi - a:
            want = lo
        elif hi - a < a - lo:
            want = hi
        else:
            want = lo if bits_of[lo] % 2 == 0 else hi
        assert abs(g) == want and math.copysign(1, g) == math.copysign(1, x)


# --------------------------------------------------------------- forward --

def test_forward_tiny_matches_brute_force():
    """The whole pipeline on the tiny workload against a per-slot pure-Python
    restatement (blockwise loops for both GEMMs)."""
    from nvfp4_block_scaled_route_gb300 import synthetic as syn
    cfg = syn.MoEConfig("pin", E=3, H=32, I=16, T=4, k=2, routing="softmax_topk_probs",
                        expert_spread=False)
    x = syn.draw_activations(cfg).float().numpy()
    ids, w = syn.draw_routing(cfg)
    W1 = [syn.draw_weight(cfg, 1, e).numpy() for e in range(cfg.E)]
    W2 = [syn.draw_weight(cfg, 2, e).numpy() for e in range(cfg.E)]
    w1q, w1sf, g1 = moe.quantize_expert_weights(W1)
    w2q, w2sf, g2 = moe.quantize_expert_weights(W2)
    out = moe.forward(x, ids.numpy(), w.numpy(), w1q, w1sf, g1, w2q, w2sf, g2)
    xq, xsf, gsx = nvfp4.quantize_rows(x)
    ids_l = ids.tolist()
    slots = _brute_route(ids_l, cfg.E)
    l1 = np.zeros((len(slots), 2 * cfg.I))
    for s, (t, j) in enumerate(slots):
        e = ids_l[t][j]
        l1[s] = _brute_block_gemm(xq[t:t + 1], xsf[t:t + 1], w1q[e], w1sf[e])[0] * (
            float(gsx) * float(g1[e]))
    assert np.allclose(out["l1"], l1, rtol=1e-12, atol=1e-12)
    h = np.zeros((len(slots), cfg.I), np.float32)
    for s in range(len(slots)):
        for c in range(cfg.I):
            g, u = l1[s, c], l1[s, cfg.I + c]
            h[s, c] = np.float32(g / (1 + math.exp(-g)) * u)
    assert np.array_equal(out["h"], h)
    hq, hsf, gsh = nvfp4.quantize_rows(h)
    y = np.zeros((cfg.T, cfg.H))
    for s, (t, j) in enumerate(slots):
        e = ids_l[t][j]
        o = _brute_block_gemm(hq[s:s + 1], hsf[s:s + 1], w2q[e], w2sf[e])[0] * (
            float(gsh) * float(g2[e]))
        y[t] += float(w[t, j]) * o
    assert np.allclose(out["y64"], y, rtol=1e-12, atol=1e-12)


def test_static_mid_scale_equals_dynamic_when_equal():
    """A static intermediate scale equal to the dynamic one changes nothing;
    otherwise expert e's rows are quantised with gs_mid[e] alone."""
    rng = np.random.default_rng(21)
    T, k, E, H, I = 6, 2, 3, 64, 32
    x = rng.normal(0, 1.5, (T, H)).astype(np.float32)
    ids = np.array([rng.choice(E, k, replace=False) for _ in range(T)], dtype=np.int32)
    w = rng.uniform(0.1, 1, (T, k)).astype(np.float32)
    W1 = [rng.normal(0, 0.2, (H, 2 * I)).astype(np.float32) for _ in range(E)]
    W2 = [rng.normal(0, 0.2, (I, H)).astype(np.float32) for _ in range(E)]
    q1 = moe.quantize_expert_weights(W1)
    q2 = moe.quantize_expert_weights(W2)
    dyn = moe.forward(x, ids, w, *q1, *q2)
    same = moe.forward(x, ids, w, *q1, *q2, gs_mid=np.full(E, dyn["gs_h"], np.float32))
    assert np.array_equal(dyn["hq"], same["hq"]) and np.array_equal(dyn["hsf"], same["hsf"])
    assert np.array_equal(dyn["y64"], same["y64"])
    mid = np.array([0.5, 1.0, 2.0], np.float32) * dyn["gs_h"]
    st = moe.forward(x, ids, w, *q1, *q2, gs_mid=mid)
    r = st["route"]
    for e in range(E):
        s0, s1 = r["offsets"][e], r["offsets"][e + 1]
        if s1 > s0:
            hq, hsf, _ = nvfp4.quantize_rows(st["h"][s0:s1], mid[e])
            assert np.array_equal(st["hq"][s0:s1], hq) and np.array_equal(st["hsf"][s0:s1], hsf)
            want = moe.expert_l2(hq, hsf, mid[e], q2[0][e], q2[1][e], q2[2][e])
            assert np.array_equal(st["out2"][s0:s1], want)
