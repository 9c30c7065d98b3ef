"""The two oracles agree: the plain C++ oracle (the oracle of record) and
the numpy one, written separately from the same pages (the C++ encoders walk
the rounding midpoints, the numpy ones search for the nearest value; the C++
GEMM adds its K terms in ascending order, numpy hands the dequantised
matrices to BLAS).  Where both take the same integer decision from the same
fp32 values (codes, scale bytes, routing), they must agree bit for bit;
fp64 sums may differ in their last bits only, and so may an fp32 h whose
fp64 value lies that close to an fp32 rounding boundary.
"""
import numpy as np
import pytest

from oracle import cpp
from oracle import moe as nmoe, nvfp4 as nnv
from nvfp4_block_scaled_route_gb300 import synthetic as syn


def test_quantiser_agrees_on_a_full_size_expert_weight():
    cfg = syn.CONFIGS["decode1"]
    w = syn.draw_weight(cfg, 2, 5).numpy()             # (3072, 7168)
    a = cpp.nvfp4.quantize_weight(w)
    b = nnv.quantize_weight(w)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1]) and a[2] == b[2]


@pytest.mark.parametrize("dist", ["normal", "student_t"])
def test_quantiser_agrees_on_activations(dist):
    cfg = syn.CONFIGS["prefill16k" if dist == "student_t" else "decode64"]
    x = syn.draw_activations(cfg, T=64).float().numpy()
    a = cpp.nvfp4.quantize_rows(x)
    b = nnv.quantize_rows(x)
    for u, v in zip(a, b):
        assert np.array_equal(u, v)


@pytest.mark.parametrize("name", ["tiny", "small", "medium"])
def test_forward_agrees(name):
    cfg = syn.CONFIGS[name]
    x = syn.draw_activations(cfg).float().numpy()
    ids, w = syn.draw_routing(cfg)
    W1 = [syn.draw_weight(cfg, 1, e).numpy() for e in range(cfg.E)]
    W2 = [syn.draw_weight(cfg, 2, e).numpy() for e in range(cfg.E)]
    w1c, w2c = cpp.moe.quantize_expert_weights(W1), cpp.moe.quantize_expert_weights(W2)
    w1n, w2n = nmoe.quantize_expert_weights(W1), nmoe.quantize_expert_weights(W2)
    for u, v in zip(w1c + w2c, w1n + w2n):
        assert np.array_equal(u, v)
    a = cpp.moe.forward(x, ids.numpy(), w.numpy(), *w1c, *w2c)
    b = nmoe.forward(x, ids.numpy(), w.numpy(), *w1n, *w2n)
    for key in ("counts", "offsets", "slot_token", "slot_of"):
        assert np.array_equal(a["route"][key], b["route"][key]), key
    assert np.array_equal(a["xq"], b["xq"]) and np.array_equal(a["xsf"], b["xsf"])
    assert a["gs_x"] == b["gs_x"]
    scale = np.abs(b["l1"]).max()
    assert np.abs(a["l1"] - b["l1"]).max() <= 1e-12 * scale
    # h: fp32 roundings of fp64 values that agree to ~1e-15
    ulp = np.spacing(np.abs(b["h"]).astype(np.float32))
    assert np.all(np.abs(a["h"].astype(np.float64) - b["h"]) <= ulp)
    same_h = (a["h"] == b["h"]).reshape(a["h"].shape[0], -1, 16).all(-1)
    assert a["gs_h"] == b["gs_h"] or abs(a["gs_h"] - b["gs_h"]) <= np.spacing(b["gs_h"])
    if a["gs_h"] == b["gs_h"]:
        hq_a = nnv.unpack_nibbles(a["hq"]).reshape(same_h.shape + (16,))
        hq_b = nnv.unpack_nibbles(b["hq"]).reshape(same_h.shape + (16,))
        assert np.array_equal(hq_a[same_h], hq_b[same_h])
        assert np.array_equal(a["hsf"][same_h], b["hsf"][same_h])
        if same_h.all():
            s2 = np.abs(b["out2"]).max()
            assert np.abs(a["out2"] - b["out2"]).max() <= 1e-12 * s2
            assert np.abs(a["y64"] - b["y64"]).max() <= 1e-12 * np.abs(b["y64"]).max()
