"""KV-pool helpers of the oracle: widening, the INT8 codec, page tables, appends.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Paged KV with 64-token pages and an INT8 cache follow the v100llm article
(sections 1-2: "Paged KV cache", INT4/INT8/FP16 storage).  The pages give no
quantisation rule; the one written here is the workload's own statement:
symmetric INT8 per (pool row, KV head) with an fp16 scale, x = q * s.
Readings (the pages are silent on each):

* ``s = fp16(min(amax / 127, 65504))`` where ``amax / 127`` is one correctly
  rounded fp32 division and the fp16 conversion rounds to nearest even;
* ``q = clamp(round_half_even(x / s), -127, 127)`` with ``x / s`` one correctly
  rounded fp32 division; ``s == 0`` gives ``q = 0``;
* dequantisation is ``float32(q) * float32(s)``, which is exact in fp32 (an
  8-bit by 11-bit significand product), so bit-exact agreement is well defined;
* scales are stored per 64-row page and KV head, 64 to a run:
  ``scale[r // 64, g, r % 64]``;
* non-finite inputs (the pages say nothing of them): a (row, head) with a NaN
  anywhere among its D values keeps the NaN -- its scale is stored as the
  fp16 quiet NaN 0x7E00 and every code is 0 (INT8, INT4) or the E4M3 NaN
  code 0x7F (FP8), so its dequantised values are all NaN, as a 16-bit pool
  would hold a NaN; a +-Inf element (with no NaN in its row) needs no extra
  rule: amax = Inf gives s = 65504 by the clamp above, the Inf quotient
  saturates to the largest code and the finite quotients round to nearly 0.
"""
from __future__ import annotations

from typing import Optional, Tuple

import numpy as np

PAGE = 64


# ---------------------------------------------------------------------------
# widening of the 16-bit storage formats


def widen_bf16(bits: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns -> float64 (exact: bf16 is the top half of fp32)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def widen_f16(bits: np.ndarray) -> np.ndarray:
    """IEEE half bit patterns -> float64 (exact)."""
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def widen(bits: np.ndarray, fmt: str) -> np.ndarray:
    if fmt == "bf16":
        return widen_bf16(bits)
    if fmt == "f16":
        return widen_f16(bits)
    raise ValueError(fmt)


# ---------------------------------------------------------------------------
# INT8 codec


def _row_scale(x32: np.ndarray, top: float):
    """The fp16 scale of each (row, head) for a codec whose largest code is
    ``top``, and which rows hold a NaN.

    s = fp16_rne(min(amax / top, 65504)) with amax / top one correctly rounded
    fp32 division (amax = +Inf gives 65504); a row with a NaN gets the fp16
    quiet NaN 0x7E00, written out explicitly rather than left to numpy's NaN
    propagation.
    """
    nan_row = np.isnan(x32).any(axis=-1)
    amax = np.max(np.abs(np.where(np.isnan(x32), np.float32(0), x32)), axis=-1)   # exact
    ratio = amax / np.float32(top)                                                # fp32, correctly rounded
    s16 = np.minimum(ratio, np.float32(65504.0)).astype(np.float16)               # nearest-even into fp16
    bits = s16.view(np.uint16).copy()
    bits[nan_row] = 0x7E00
    return bits.view(np.float16), nan_row


def quantize_int8(x: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """Symmetric INT8 per (row, head) over the last axis.

    x: values exactly representable in fp32 (widened fp16/bf16), shape [N, H, D].
    Returns (q int8 [N, H, D], s float16 [N, H]).
    """
    x32 = np.asarray(x, dtype=np.float32)
    s16, nan_row = _row_scale(x32, 127.0)
    s32 = s16.astype(np.float32)[..., None]
    with np.errstate(divide="ignore", invalid="ignore"):
        quot = x32 / s32                                      # fp32, correctly rounded
    qv = np.clip(np.rint(quot), -127, 127)                    # rint: ties to even; +-Inf -> +-127
    qv = np.where((s32 == 0) | nan_row[..., None], 0, qv)     # zero rows and NaN rows: code 0
    return qv.astype(np.int8), s16


def dequantize_int8(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    """float32(q) * float32(s), per (row, head) scale broadcast over the last axis."""
    return np.asarray(q, dtype=np.float32) * np.asarray(s, dtype=np.float16).astype(np.float32)[..., None]


def pack_scales(s: np.ndarray) -> np.ndarray:
    """Per-(row, head) scales [R, H] -> the stored layout [R/64, H, 64]."""
    R, H = s.shape
    assert R % PAGE == 0
    return np.ascontiguousarray(s.reshape(R // PAGE, PAGE, H).transpose(0, 2, 1))


def unpack_scales(sp: np.ndarray) -> np.ndarray:
    """The stored layout [R/64, H, 64] -> per-(row, head) scales [R, H]."""
    P, H, _ = sp.shape
    return np.ascontiguousarray(sp.transpose(0, 2, 1).reshape(P * PAGE, H))


# ---------------------------------------------------------------------------
# INT4 codec (paged INT4 KV, v100llm article section 2)


def quantize_int4(x: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """Symmetric INT4 per (row, head): levels -7..7, fp16 scale, two codes per byte.

    Readings (the pages name INT4 KV but give no rule): same steps as INT8 with
    127 replaced by 7; codes are stored as 4-bit two's complement, element
    ``2t`` in the low nibble and ``2t+1`` in the high nibble of byte ``t``.
    Returns (packed uint8 [N, H, D/2], s float16 [N, H]).
    """
    x32 = np.asarray(x, dtype=np.float32)
    s16, nan_row = _row_scale(x32, 7.0)
    s32 = s16.astype(np.float32)[..., None]
    with np.errstate(divide="ignore", invalid="ignore"):
        quot = x32 / s32
    qv = np.clip(np.rint(quot), -7, 7)
    qv = np.where((s32 == 0) | nan_row[..., None], 0, qv).astype(np.int64)
    nib = (qv & 0xF).astype(np.uint8)
    packed = nib[..., 0::2] | (nib[..., 1::2] << np.uint8(4))
    return packed.astype(np.uint8), s16


def dequantize_int4(packed: np.ndarray, s: np.ndarray) -> np.ndarray:
    """Unpack two's-complement nibbles and multiply by the fp16 scale (exact in fp32)."""
    p = np.asarray(packed, dtype=np.uint8).astype(np.int64)
    lo = p & 0xF
    hi = (p >> 4) & 0xF
    codes = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), dtype=np.int64)
    codes[..., 0::2] = lo
    codes[..., 1::2] = hi
    codes = np.where(codes >= 8, codes - 16, codes)
    return codes.astype(np.float32) * np.asarray(s, dtype=np.float16).astype(np.float32)[..., None]


# ---------------------------------------------------------------------------
# page tables


def page_table_to_rows(page_table: np.ndarray, seq_len: np.ndarray, list_len: int, page: int = PAGE) -> np.ndarray:
    """Expand per-sequence page tables into row lists.

    Position ``j`` of sequence ``s`` lives in page ``page_table[s, j // page]``
    at offset ``j % page``, so its pool row is ``page_id * page + j % page``;
    positions at or beyond ``seq_len[s]`` (and up to ``list_len``) are padding,
    written as -1.  Reading (the pages are silent): a negative page id marks an
    unused page-table slot, so its positions are padding (-1) as well, and
    ``seq_len`` is clamped to the table's ``max_pages * page`` positions.
    """
    S = page_table.shape[0]
    out = np.full((S, list_len), -1, dtype=np.int32)
    max_pos = page_table.shape[1] * page
    for s in range(S):
        for j in range(min(int(seq_len[s]), list_len, max_pos)):
            page_id = int(page_table[s, j // page])
            if page_id >= 0:
                out[s, j] = page_id * page + (j % page)
    return out


# ---------------------------------------------------------------------------
# appending new rows to the pool


def append_rows(pool: np.ndarray, new: np.ndarray, dst_rows: np.ndarray,
                pool_scales: Optional[np.ndarray] = None, fmt: str = "copy"):
    """Write ``new[i]`` into pool row ``dst_rows[i]`` (negative = skip).

    fmt 'copy': ``pool`` holds raw 16-bit patterns [R, H, D] and is written as is.
    fmt 'int8': ``new`` holds fp32-exact values; each row is quantised with
    ``quantize_int8`` into ``pool`` (int8 [R, H, D]) and ``pool_scales`` (the
    stored layout [R/64, H, 64], fp16).
    Returns the updated (pool, pool_scales) copies.
    """
    pool = pool.copy()
    sc = None if pool_scales is None else pool_scales.copy()
    if fmt == "int8":
        qv, s = quantize_int8(new)
    for i, r in enumerate(np.asarray(dst_rows).tolist()):
        if r < 0:
            continue
        if fmt == "copy":
            pool[r] = new[i]
        else:
            pool[r] = qv[i]
            sc[r // PAGE, :, r % PAGE] = s[i]
    return pool, sc


# ---------------------------------------------------------------------------
# FP8 E4M3 codec ("llama.cpp 0.9.0 inference boundaries", section 4: the OCP
# FP8 E4M3 type in saturating mode; the pages defer its use for the KV cache
# and its scaling, so the reading here mirrors the INT8 one)
#
# * s = fp16(min(amax / 448, 65504)) (one fp32 division, round to nearest
#   even), per (row, head); s == 0 gives code 0;
# * code = E4M3(x / s): x / s one fp32 division, then round to nearest even on
#   the E4M3 grid (1 sign, 4 exponent bits with bias 7, 3 mantissa bits,
#   subnormal step 2^-9, largest finite 448, no infinities), saturating to
#   +-448 (an Inf element of a NaN-free row therefore codes as +-448); a row
#   holding a NaN gets the NaN scale 0x7E00 and the NaN code 0x7f throughout
#   (the non-finite reading above);
# * dequantisation is float32(E4M3 value) * float32(s), exact in fp32 (a 4-bit
#   by 11-bit significand product).

E4M3_MAX = 448.0


def e4m3_value(code: np.ndarray) -> np.ndarray:
    """Value of each E4M3 byte (float64; NaN for the two NaN codes)."""
    c = np.asarray(code, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * 2.0 ** (e - 7.0))
    mag = np.where((e == 0xF) & (m == 0x7), np.nan, mag)
    return sign * mag


def e4m3_encode(y: np.ndarray) -> np.ndarray:
    """Round fp32 values to the nearest E4M3 code (ties to even), saturating."""
    y = np.asarray(y, dtype=np.float64)
    out = np.zeros(y.shape, dtype=np.uint8)
    nan = np.isnan(y)
    sign = np.signbit(y)
    a = np.minimum(np.abs(np.where(nan, 0.0, y)), E4M3_MAX)
    # step of the grid around a: 2^-9 below the smallest normal 2^-6, else 2^(e-3)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    step = np.where(a < 2.0 ** -6, 2.0 ** -9, 2.0 ** (e - 3))
    q = np.rint(a / step) * step            # exact: a / step is representable, rint ties to even
    q = np.minimum(q, E4M3_MAX)
    # encode the magnitude q
    sub = q < 2.0 ** -6
    qe = np.floor(np.log2(np.where(q > 0, q, 1.0)))
    mant = np.where(sub, q / 2.0 ** -9, (q / 2.0 ** qe - 1.0) * 8.0)
    expo = np.where(sub, 0, qe + 7)
    code = (expo.astype(np.int64) << 3) | np.rint(mant).astype(np.int64)
    code = np.where(sign, code | 0x80, code)
    out[...] = code.astype(np.uint8)
    out[nan] = 0x7F
    return out


def quantize_fp8(x: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """FP8 E4M3 per (row, head) with an fp16 scale; returns (codes uint8 [N, H, D], s float16 [N, H])."""
    x32 = np.asarray(x, dtype=np.float32)
    s16, nan_row = _row_scale(x32, E4M3_MAX)
    s32 = s16.astype(np.float32)[..., None]
    with np.errstate(divide="ignore", invalid="ignore"):
        quot = x32 / s32
    codes = e4m3_encode(np.where(nan_row[..., None], np.float32(0), quot))
    codes = np.where(s32 == 0, np.uint8(0), codes)
    codes = np.where(nan_row[..., None], np.uint8(0x7F), codes)   # NaN rows: the E4M3 NaN code
    return codes.astype(np.uint8), s16


def dequantize_fp8(codes: np.ndarray, s: np.ndarray) -> np.ndarray:
    """float32(E4M3 value) * float32(s), exact in fp32."""
    v = e4m3_value(codes).astype(np.float32)
    return v * np.asarray(s, dtype=np.float16).astype(np.float32)[..., None]
