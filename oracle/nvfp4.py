"""NVFP4 codecs, packing and quantiser (oracle; test infrastructure only).

Sources (web pages of the NVFP4 MegaMoE kernel debug effort):

* E2M1 values and nibble layout: commit message "Three bugs fixed" on ``src``
  — sign-magnitude 4-bit nibble, bit 3 = sign, bits 2:0 index the magnitudes
  {0, 0.5, 1, 1.5, 2, 3, 4, 6}; values snap to the nearest magnitude.
* Packing: "NVFP4 MegaMoE Debug Log", Hypotheses §5 — two nibbles per byte,
  element 2j in the low nibble, element 2j+1 in the high nibble.
* Scales: Debug Log, Hypotheses §6 steps 1–5 — global scale
  ``amax / (6 * 448)``, block scale ``block_amax / (6 * global_scale)``
  stored as float8 (E4M3), then nearest-E2M1 of each element.
* E4M3 decoding: commit message on the FP8 view-vs-convert bug — a stored
  scale byte must be read by its bit pattern, not converted by value.  The
  passage's example value for 0x3F is garbled; the bit pattern of 0x3F is
  1.875 under the OCP E4M3 definition used here (bias 7, no infinities,
  0x7F/0xFF NaN, max 448).

Readings where the pages are silent:

* rounding is nearest, ties to the even mantissa (code with bit 0 clear);
* encoders saturate to the largest finite value (6 for E2M1, 448 for E4M3);
* the nibble divisor is the *stored* scale: d = dec(sf) * gs in fp32;
* a block whose stored scale decodes to 0 quantises to nibbles 0x0;
* an all-zero tensor gets gs = 1.0;
* a negative element that rounds to magnitude 0 keeps its sign bit (0x8);
* scale bytes are non-negative (block amax >= 0), i.e. unsigned E4M3.
"""
from __future__ import annotations

import numpy as np

# ---------------------------------------------------------------- E2M1 ----

E2M1_MAGNITUDES = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], dtype=np.float64)


def e2m1_decode(nib: np.ndarray) -> np.ndarray:
    """Nibble codes (0..15) -> float64 values.  Pinned: golden table."""
    nib = np.asarray(nib).astype(np.int64)
    mag = E2M1_MAGNITUDES[nib & 7]
    return np.where((nib & 8) != 0, -mag, mag)


def e2m1_encode(v: np.ndarray) -> np.ndarray:
    """float -> nibble code: nearest magnitude, ties to even code, saturate 6.

    The sign bit is the sign bit of the input (so -0.0 and small negatives
    give 0x8).  Pinned: identity on all 16 codes, listed ties, brute force.
    """
    v = np.asarray(v)
    # fp32 inputs are compared in fp32 (every magnitude and midpoint is
    # exact there); anything else in fp64.
    ft = np.float32 if v.dtype == np.float32 else np.float64
    mags = E2M1_MAGNITUDES.astype(ft)
    a = np.minimum(np.abs(v.astype(ft, copy=False)), mags[-1])
    # the two representable magnitudes around a: lo <= a <= hi
    hi = np.minimum(np.searchsorted(mags, a, side="left"), 7).astype(np.uint8)
    lo = np.maximum(hi, 1) - 1
    dlo = a - mags[lo]
    dhi = mags[hi] - a
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (hi % 2 == 0))
    code = np.where(pick_hi | (dhi == 0), hi, lo)
    sign = np.signbit(v).astype(np.uint8)
    return (code | (sign << 3)).astype(np.uint8)


# ---------------------------------------------------------------- E4M3 ----

def e4m3_decode(byte: np.ndarray) -> np.ndarray:
    """E4M3 byte -> float64 by bit pattern (OCP E4M3, bias 7).

    e == 0: (m/8) * 2^-6 (subnormal); otherwise (1 + m/8) * 2^(e-7);
    S.1111.111 is NaN.  Pinned: spot values, torch float8_e4m3fn ``.view``.
    """
    b = np.asarray(byte).astype(np.int64)
    s = (b >> 7) & 1
    e = (b >> 3) & 15
    m = b & 7
    mag = np.where(e == 0, (m / 8.0) * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return np.where(s == 1, -mag, mag)


# all non-negative finite E4M3 values, ascending with the byte value
_E4M3_POS_BYTES = np.arange(0, 127, dtype=np.int64)       # 0x00 .. 0x7E
_E4M3_POS_VALUES = e4m3_decode(_E4M3_POS_BYTES)


def e4m3_encode_nonneg(v: np.ndarray) -> np.ndarray:
    """Non-negative float -> unsigned E4M3 byte: nearest, ties to even,
    saturating at 448 (0x7E).  Pinned: torch float8_e4m3fn cast on [0, 448]."""
    a = np.asarray(v).astype(np.float64)
    if np.any(a < 0) or np.any(np.isnan(a)):
        raise ValueError("scale inputs must be finite and non-negative")
    a = np.minimum(a, _E4M3_POS_VALUES[-1])
    hi = np.searchsorted(_E4M3_POS_VALUES, a, side="left")      # first >= a
    hi = np.minimum(hi, 126)
    lo = np.maximum(hi - 1, 0)
    dlo = a - _E4M3_POS_VALUES[lo]
    dhi = _E4M3_POS_VALUES[hi] - a
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (_E4M3_POS_BYTES[hi] % 2 == 0))
    exact = _E4M3_POS_VALUES[hi] == a
    out = np.where(exact | pick_hi, _E4M3_POS_BYTES[hi], _E4M3_POS_BYTES[lo])
    return out.astype(np.uint8)


# ------------------------------------------------------------- packing ----

def pack_nibbles(nib: np.ndarray) -> np.ndarray:
    """[..., K] nibbles -> [..., K/2] bytes, element 2j low, 2j+1 high."""
    nib = np.asarray(nib).astype(np.uint8)
    assert nib.shape[-1] % 2 == 0
    lo = nib[..., 0::2]
    hi = nib[..., 1::2]
    return ((hi << 4) | lo).astype(np.uint8)


def unpack_nibbles(packed: np.ndarray) -> np.ndarray:
    """[..., K/2] bytes -> [..., K] nibbles (inverse of pack_nibbles)."""
    p = np.asarray(packed).astype(np.uint8)
    out = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = p >> 4
    return out


def unpack_weight_k(packed_kn: np.ndarray) -> np.ndarray:
    """Checkpoint weight bytes (K/2, N) -> nibbles (K, N).

    Byte (j, n) holds element (2j, n) in its low nibble and (2j+1, n) in its
    high nibble; the two elements are interleaved along K, never along N
    (the Debug Log's "weight nibble unpack reshape bug" passage).
    """
    p = np.asarray(packed_kn).astype(np.uint8)
    K2, N = p.shape[-2], p.shape[-1]
    out = np.empty(p.shape[:-2] + (2 * K2, N), dtype=np.uint8)
    out[..., 0::2, :] = p & 0xF
    out[..., 1::2, :] = p >> 4
    return out


# ----------------------------------------------------------- quantiser ----

F32 = np.float32
GLOBAL_DIVISOR = F32(6.0 * 448.0)     # 2688, the E2M1 max times the E4M3 max


def global_scale(amax) -> np.float32:
    """gs = amax / (6*448) in fp32; an all-zero tensor gets 1.0."""
    amax = F32(amax)
    if amax == 0:
        return F32(1.0)
    return F32(amax / GLOBAL_DIVISOR)


def quantize_rows(v: np.ndarray, gs: np.float32 | None = None):
    """Quantise rows of a [R, K] fp32 matrix along K in 16-element blocks.

    Steps (Debug Log, Hypotheses §6; commit "Three bugs fixed"), all fp32:
      1. amax = max |v| over the whole tensor          (unless gs is given)
      2. gs   = amax / 2688
      3. per block: b = max |v_i|;  sf = E4M3(b / (6 * gs))
      4. d = dec(sf) * gs;  nibble_i = E2M1(v_i / d)   (d == 0 -> 0x0)
      5. pack element 2j low, 2j+1 high.
    Returns (q uint8 [R, K/2], sf uint8 [R, K/16], gs float32).
    Pinned: constant blocks, E2M1-grid blocks, round-trip bound, one-hot
    packing, the Debug Log's round-trip numbers.
    """
    v = np.ascontiguousarray(v, dtype=np.float32)
    R, K = v.shape
    assert K % 16 == 0
    if gs is None:
        amax = np.max(np.abs(v)) if v.size else F32(0.0)
        gs = global_scale(amax)
    gs = F32(gs)
    q = np.empty((R, K // 2), dtype=np.uint8)
    sf = np.empty((R, K // 16), dtype=np.uint8)
    # rows are independent once gs is fixed; they are taken in groups only to
    # bound the size of the temporaries.
    step = max(1, (1 << 22) // max(K, 1))
    for r0 in range(0, R, step):
        q[r0:r0 + step], sf[r0:r0 + step] = _quantize_blocks(v[r0:r0 + step], gs)
    return q, sf, gs


def _quantize_blocks(v: np.ndarray, gs: np.float32):
    """Steps 3-5 of quantize_rows for a group of rows, given gs."""
    R, K = v.shape
    blocks = v.reshape(R, K // 16, 16)
    bmax = np.max(np.abs(blocks), axis=-1) if v.size else np.zeros((R, K // 16), F32)
    denom = F32(F32(6.0) * gs)
    with np.errstate(divide="ignore", invalid="ignore"):
        sf = e4m3_encode_nonneg((bmax / denom).astype(np.float32))
        d = (e4m3_decode(sf).astype(np.float32) * gs).astype(np.float32)
        ratio = (blocks / d[..., None]).astype(np.float32)
    zero = d[..., None] == 0
    nib = e2m1_encode(np.where(zero, F32(0.0), ratio))
    nib = np.where(zero, np.uint8(0), nib).reshape(R, K)
    return pack_nibbles(nib), sf.astype(np.uint8)


def dequantize_rows(q: np.ndarray, sf: np.ndarray) -> np.ndarray:
    """Packed rows + block scales -> float64 [R, K], WITHOUT the global scale
    (the global scales enter the GEMM as alpha)."""
    nib = unpack_nibbles(q)
    R, K = nib.shape
    vals = e2m1_decode(nib).reshape(R, K // 16, 16)
    return (vals * e4m3_decode(sf)[..., None]).reshape(R, K)


def quantize_weight(w_kn: np.ndarray):
    """One expert's fp32 weight (K, N) -> checkpoint NVFP4 (Hypotheses §2/§6).

    Blocks of 16 run along K for each output column n; the global scale is
    per expert (amax over the whole expert matrix).  Returns
    (q uint8 (K/2, N), sf uint8 (K/16, N), gs float32).
    """
    w = np.asarray(w_kn, dtype=np.float32)
    q_nk, sf_nk, gs = quantize_rows(np.ascontiguousarray(w.T))
    # (N, K/2) bytes pack (n, 2j) low and (n, 2j+1) high: transposing the
    # byte matrix gives the checkpoint's (K/2, N) bytes with the same pairs.
    return np.ascontiguousarray(q_nk.T), np.ascontiguousarray(sf_nk.T), gs


def dequantize_weight(q_kn: np.ndarray, sf_kn: np.ndarray) -> np.ndarray:
    """Checkpoint (K/2, N) bytes + (K/16, N) scales -> float64 (K, N),
    without the global scale."""
    nib = unpack_weight_k(q_kn)
    K, N = nib.shape
    vals = e2m1_decode(nib).reshape(K // 16, 16, N)
    return (vals * e4m3_decode(sf_kn)[:, None, :]).reshape(K, N)


# ---------------------------------------------------------------- bf16 ----

def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """float64 -> nearest bf16 value (ties to even), returned as float64.

    Rounds once, directly from fp64 (no intermediate fp32).  Pinned against a
    brute-force search over all bf16 values.
    """
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)                 # x = m * 2^e, 0.5 <= |m| < 1
    scaled = np.ldexp(m, 8)            # 8 significant bits
    r = np.rint(scaled)                # ties to even
    out = np.ldexp(r, e - 8)
    return np.where(x == 0, x, out)
