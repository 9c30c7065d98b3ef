"""Host-side restatement of the staged block-scale layout documented in
include/nvfp4moe.h (512-byte atoms of 128 rows x 4 scale bytes, atoms along
K within a 128-row block).  Used by the tests to build and read staged
buffers; independent of the CUDA code."""
import numpy as np


def sf_mma_size(rows, cols):
    rows_pad = -(-rows // 128) * 128
    k_pad = -(-cols // 256) * 256
    return rows_pad * (k_pad // 16)


def staged_offsets(rows, cols):
    """Offset of scale (r, g) for every r < rows, g < cols/16."""
    k_pad = -(-cols // 256) * 256
    r = np.arange(rows)[:, None]
    g = np.arange(cols // 16)[None, :]
    return ((r // 128) * (k_pad // 64) + g // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + (g % 4)


def stage(sf_row):
    rows, groups = sf_row.shape
    cols = groups * 16
    buf = np.zeros(sf_mma_size(rows, cols), dtype=np.uint8)
    buf[staged_offsets(rows, cols)] = sf_row
    return buf


def unstage(buf, rows, cols):
    return np.asarray(buf)[staged_offsets(rows, cols)]
