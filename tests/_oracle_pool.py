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


def pool(n=None):
    n = n or min(16, os.cpu_count() or 1)
    return mp.get_context("spawn").Pool(n)
