"""Process-pool helpers that run oracle work for the GPU tests in parallel.

The pool is created with the "spawn" start method (never forked from a
process that already holds a CUDA context).  Workers call only oracle/.
"""
import multiprocessing as mp
import os

import numpy as np


def quantize_pair(args):
    """(W1_e, W2_e) fp32 -> checkpoint NVFP4 tensors of both layers."""
    from oracle import nvfp4
    w1, w2 = args
    q1, s1, g1 = nvfp4.quantize_weight(w1)
    q2, s2, g2 = nvfp4.quantize_weight(w2)
    return q1, s1, np.float32(g1), q2, s2, np.float32(g2)


def dequant_pair(args):
    """Checkpoint tensors -> fp64 dequantised (K, N) matrices (no global scale)."""
    from oracle import nvfp4
    q1, s1, q2, s2 = args
    return nvfp4.dequantize_weight(q1, s1), nvfp4.dequantize_weight(q2, s2)


def expert_l1_task(args):
    """L1 of rows [c0, c0 + n) of one expert's slots: (e, gs_w1, max |h|,
    {expert-local row: h row} for the rows asked for).

    x rows arrive as bf16 bit patterns; the weight is drawn here from the
    seeded synthetic generator and quantised by the oracle."""
    from oracle import moe, nvfp4
    from nvfp4_block_scaled_route_gb300 import synthetic
    cfg_name, e, c0, x_bits, gs_x, want = args
    cfg = synthetic.CONFIGS[cfg_name]
    q1, s1, g1 = nvfp4.quantize_weight(synthetic.draw_weight(cfg, 1, e).numpy())
    x = (x_bits.astype(np.uint32) << 16).view(np.float32)
    xq, xsf, _ = nvfp4.quantize_rows(x, gs_x)
    amax = np.float32(0.0)
    rows = {}
    for b0 in range(0, x.shape[0], 1024):
        h = moe.swiglu(moe.expert_l1(xq[b0:b0 + 1024], xsf[b0:b0 + 1024], gs_x, q1, s1, g1))
        amax = max(amax, np.float32(np.abs(h).max()))
        for i in want:
            if c0 + b0 <= i < c0 + b0 + h.shape[0]:
                rows[i] = h[i - c0 - b0]
    return e, np.float32(g1), amax, rows


def expert_w2_task(args):
    """Checkpoint NVFP4 of one expert's L2 weight (drawn here)."""
    from oracle import nvfp4
    from nvfp4_block_scaled_route_gb300 import synthetic
    cfg_name, e = args
    q2, s2, g2 = nvfp4.quantize_weight(synthetic.draw_weight(synthetic.CONFIGS[cfg_name], 2, e).numpy())
    return e, q2, s2, np.float32(g2)


def pool(n=None):
    n = n or min(16, os.cpu_count() or 1)
    # one BLAS thread per worker: the pool supplies the parallelism
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[var] = "1"
    return mp.get_context("spawn").Pool(n)
