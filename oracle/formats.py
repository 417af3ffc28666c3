"""Oracle: decoding of the stored KV-cache element formats, written from their public definitions.

TEST INFRASTRUCTURE ONLY. Nothing on the product path imports this package;
only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s cpu_baseline
leg may use it.

Formats
-------
* bf16: the upper 16 bits of an IEEE-754 binary32 value (exact widening).
* fp8 E4M3 (OCP 8-bit floating point specification, "E4M3"): 1 sign bit,
  4 exponent bits with bias 7, 3 mantissa bits; exponent field 0 encodes
  subnormals m/8 * 2^-6; the all-ones pattern S.1111.111 is NaN (no infinities);
  largest finite magnitude 448.
* fp4 E2M1 (OCP Microscaling Formats v1.0, element type FP4): 1 sign bit,
  2 exponent bits with bias 1, 1 mantissa bit; exponent field 0 encodes the
  subnormal m/2 (0 or 0.5); magnitudes {0, 0.5, 1, 1.5, 2, 3, 4, 6}.

The NVFP4 KV cache of the MiniMax-M3 NVFP4 backend (vLLM page
``vllm.models.minimax_m3.amd.sparse_attention_nvfp4``, ``customize_spec``)
stores each head's K and V as two slots of "packed data + block scales"; the
byte order inside a slot is backend-specific and not shown. The reading used
here: a slot is 16 rows x 64 bytes of e2m1 codes (element 2i in the low nibble
of byte i, 2i+1 in the high nibble) followed by 16 rows x 8 bytes of e4m3
scales, scale j covering elements 16j..16j+15 of its row; slot 2g holds K of
kv head g and slot 2g+1 holds V.
"""
from __future__ import annotations

import numpy as np


def bf16_bits_to_float(bits: np.ndarray) -> np.ndarray:
    """uint16 bf16 bit patterns -> float64 (exact)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def e4m3_to_float(codes: np.ndarray) -> np.ndarray:
    """uint8 E4M3 codes -> float64, from the field definition (NaN for S.1111.111)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    normal = (1.0 + m / 8.0) * np.exp2(e - 7.0)
    subnormal = (m / 8.0) * np.exp2(-6.0)
    mag = np.where(e == 0, subnormal, normal)
    mag = np.where((e == 0xF) & (m == 0x7), np.nan, mag)
    return sign * mag


def e2m1_to_float(nibbles: np.ndarray) -> np.ndarray:
    """4-bit E2M1 codes (values 0..15 in a uint8) -> float64, from the field definition."""
    c = np.asarray(nibbles, dtype=np.uint8).astype(np.int64) & 0xF
    sign = np.where(c & 0x8, -1.0, 1.0)
    e = (c >> 1) & 0x3
    m = c & 0x1
    normal = (1.0 + m / 2.0) * np.exp2(e - 1.0)
    subnormal = m / 2.0
    return sign * np.where(e == 0, subnormal, normal)


NVFP4_ROWS = 16
NVFP4_CODE_BYTES = 64       # one row of 128 e2m1 codes
NVFP4_SCALE_BYTES = 8       # one row of 8 e4m3 scales
NVFP4_SLOT_BYTES = NVFP4_ROWS * (NVFP4_CODE_BYTES + NVFP4_SCALE_BYTES)


def nvfp4_slot_rows(slot: np.ndarray, rows: np.ndarray) -> np.ndarray:
    """Dequantise rows of one (page, K-or-V) slot: e2m1 code x e4m3 block scale.

    ``slot`` is the slot's 1152 bytes; returns float64 [len(rows), 128]
    (without the per-tensor global scale).
    """
    slot = np.asarray(slot, dtype=np.uint8)
    codes = slot[:NVFP4_ROWS * NVFP4_CODE_BYTES].reshape(NVFP4_ROWS, NVFP4_CODE_BYTES)[rows]
    scales = slot[NVFP4_ROWS * NVFP4_CODE_BYTES:].reshape(NVFP4_ROWS, NVFP4_SCALE_BYTES)[rows]
    lo = e2m1_to_float(codes & 0xF)
    hi = e2m1_to_float(codes >> 4)
    elems = np.empty((codes.shape[0], 2 * NVFP4_CODE_BYTES))
    elems[:, 0::2] = lo
    elems[:, 1::2] = hi
    sc = e4m3_to_float(scales)                       # [rows, 8]
    return elems * np.repeat(sc, 16, axis=1)
