"""Oracle: dequantisation of the canonical weight blocks, in float64.

TEST INFRASTRUCTURE.  Only tests/, __graft_entry__.smoke() and bench.py's
cpu_baseline / reference leg may import anything under oracle/.  The product
path (the CUDA library and its binding) never does.

Block definitions (all blocks hold 32 consecutive values of one weight row,
blocks run along the row, rows are stored one after another):

* Q8_0   {fp16 d; int8 q[32]}            value = d * q
* Q4_0   {fp16 d; uint8 qs[16]}          value = d * (q - 8), where q for
         element j < 16 is the low nibble of qs[j] and for j >= 16 the high
         nibble of qs[j - 16]
* I8ASYM {fp16 s; fp16 z; uint8 q[32]}   value = s * (q - z)
* F16    plain little-endian fp16 matrix

and the same Q8_0 / Q4_0 definitions over groups of 64 values (the Metal
page's "La quantizzazione opera su gruppi di 64 valori"):

* Q8_0_G64 {fp16 d; int8 q[64]}          value = d * q
* Q4_0_G64 {fp16 d; uint8 qs[32]}        value = d * (q - 8), q of element
           j < 32 the low nibble of qs[j], of j >= 32 the high nibble of
           qs[j - 32] (the 32-value rule with the half moved to 32: a reading)

Cites: "Unlimited-OCR on Apple Silicon with C and Metal", section
"Quantizzazione: Q8 prima, Q4 dove conviene" (Q8_0 / Q4_0 profiles with the
dequantisation fused into the kernels); "Falcon-OCR INT8 OpenVINO IR" model
card (INT8_ASYM weights, unsigned codes).  Group size 32 and the exact block
formulas are the decode-step statement's definitions; the Metal page's group
size of 64 is a different choice of the same format family.
"""
from __future__ import annotations

import numpy as np

F16, Q8_0, Q4_0, I8ASYM, Q8_0_G64, Q4_0_G64 = 0, 1, 2, 3, 4, 5
BLOCK = 32
_GROUP = {Q8_0: 32, Q4_0: 32, I8ASYM: 32, Q8_0_G64: 64, Q4_0_G64: 64}
_BYTES = {Q8_0: 34, Q4_0: 18, I8ASYM: 36, Q8_0_G64: 66, Q4_0_G64: 34}


def _blocks(blob, fmt, rows, cols):
    g = _GROUP[fmt]
    if cols % g:
        raise ValueError(f"cols must be a multiple of {g}")
    raw = np.frombuffer(np.asarray(blob, dtype=np.uint8).tobytes(), dtype=np.uint8)
    nb = cols // g
    if raw.size != rows * nb * _BYTES[fmt]:
        raise ValueError("blob size does not match the shape")
    return raw.reshape(rows, nb, _BYTES[fmt])


def _f16_field(raw, lo):
    """The little-endian fp16 at byte offset lo of every block, as float64."""
    return raw[:, :, lo:lo + 2].copy().view("<f2")[:, :, 0].astype(np.float64)


def dequant_q8_0(blob, rows, cols, fmt=Q8_0):
    raw = _blocks(blob, fmt, rows, cols)
    d = _f16_field(raw, 0)
    q = raw[:, :, 2:].copy().view(np.int8).astype(np.float64)
    return (d[:, :, None] * q).reshape(rows, cols)


def dequant_q4_0(blob, rows, cols, fmt=Q4_0):
    raw = _blocks(blob, fmt, rows, cols)
    d = _f16_field(raw, 0)
    qs = raw[:, :, 2:]
    q = np.concatenate([qs & 0x0F, qs >> 4], axis=-1).astype(np.float64)
    return (d[:, :, None] * (q - 8.0)).reshape(rows, cols)


def dequant_i8asym(blob, rows, cols):
    raw = _blocks(blob, I8ASYM, rows, cols)
    s = _f16_field(raw, 0)
    z = _f16_field(raw, 2)
    q = raw[:, :, 4:36].astype(np.float64)
    return (s[:, :, None] * (q - z[:, :, None])).reshape(rows, cols)


def dequant_f16(blob, rows, cols):
    a = np.frombuffer(np.asarray(blob, dtype=np.uint8).tobytes(), dtype="<f2")
    if a.size != rows * cols:
        raise ValueError("blob size does not match the shape")
    return a.reshape(rows, cols).astype(np.float64)


def dequant(blob, fmt, rows, cols):
    """Dequantise a canonical blob of the given format to float64 [rows, cols]."""
    if fmt == F16:
        return dequant_f16(blob, rows, cols)
    if fmt == Q8_0:
        return dequant_q8_0(blob, rows, cols)
    if fmt == Q4_0:
        return dequant_q4_0(blob, rows, cols)
    if fmt == I8ASYM:
        return dequant_i8asym(blob, rows, cols)
    if fmt == Q8_0_G64:
        return dequant_q8_0(blob, rows, cols, Q8_0_G64)
    if fmt == Q4_0_G64:
        return dequant_q4_0(blob, rows, cols, Q4_0_G64)
    raise ValueError(f"unknown format {fmt}")


def float32_is_exact(w64):
    """True when every value survives a round trip through float32 unchanged.

    Q8_0 / Q4_0 values are an fp16 scale (11 significant bits) times an
    integer of at most 8 bits, so they always fit float32's 24-bit
    significand; the oracle may then keep them in float32 to halve its memory
    without changing any result (they are widened back to float64 before use).
    """
    return bool(np.array_equal(w64.astype(np.float32).astype(np.float64), w64))
