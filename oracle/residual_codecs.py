"""CPU oracle of the hidden-state storage formats compared in the quantization
ablation of "Polestar: Drift-Aware Cache Calibration and Token Commitment for
Efficient Inference of Diffusion LLMs" (Table 11; App. C.3 for NVFP4).

TEST INFRASTRUCTURE ONLY: imported by the tests; shares no code with the CUDA
library.  Plain numpy in float64, one function per format, each encode paired
with its decode.  The paper names the formats but fixes only NVFP4's layout, so
the others follow their usual definitions, with these readings:

  FP16     IEEE binary16, round to nearest even, of the hidden state itself (the
           "full precision" row: no residual).
  FP8      E4M3 elements (nearest even, saturating at 448) with one fp32 scale per
           row (token), s = fp32(amax / 448).
  INT8     symmetric integers in [-127, 127] (nearest even) with one fp32 scale per
           row, s = fp32(amax / 127).
  MXFP4    the OCP microscaling format: blocks of 32 elements share a power-of-two
           scale X = 2^(floor(log2 amax) - 2) (2 = the largest E2M1 exponent),
           the exponent held to the E8M0 scale range [-127, 127]; elements E2M1,
           nearest even, saturating at 6; an all-zero block keeps zero codes.
  INT2     symmetric ternary {-1, 0, +1} (two bits) with one fp32 scale per row,
           s = amax: an element becomes sign(r) * s when |r| > s / 2, else 0
           (nearest; a tie at s / 2 goes to the even value 0).
  NVFP4    App. C.3, from polestar_oracle.nvfp4_encode (E2M1 elements, one E4M3
           scale per 16).

"Residual" applies a format to r = h - A_label (the row's cluster anchor, App. C.3
and §4.1) and reconstructs h' = A_label + decode(encode(r)); "plain" applies it to h.

Parity status: pinned by tests/test_oracle_codecs.py (binary16 constants, grid
membership, exact scale maps, error bounds, the OCP scale rule on worked blocks, and
Table 11's ordering of the formats on clustered synthetic states).
"""
from __future__ import annotations

import numpy as np

from oracle.polestar_oracle import (E2M1_VALUES, e2m1_round, e2m1_value, e4m3_round, e4m3_value, nvfp4_decode,
                                    nvfp4_encode, to_f32)


def _f32(x):
    return np.asarray(x, dtype=np.float64).astype(np.float32)


# ---- FP16 -----------------------------------------------------------------------------
def fp16_roundtrip(h):
    """binary16 nearest-even of every element (numpy's float16 conversion)."""
    return np.asarray(h, dtype=np.float64).astype(np.float16).astype(np.float64)


# ---- FP8 E4M3, per-row scale ----------------------------------------------------------
def fp8_encode(r):
    """Returns (bytes [rows, d] u8: sign bit 7 + E4M3 magnitude, scales [rows] fp32)."""
    r32 = _f32(r)
    amax = np.max(np.abs(r32), axis=-1)
    s = (amax / np.float32(448.0)).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        q = (r32 / s[:, None]).astype(np.float64)
    q = np.where(s[:, None] == 0, 0.0, q)
    _, mag, _ = e4m3_round(np.abs(q))
    sign = np.signbit(q).astype(np.uint8) << 7
    return (mag | sign).astype(np.uint8), s


def fp8_decode(codes, s):
    return to_f32(e4m3_value(codes) * np.asarray(s, dtype=np.float64)[:, None])


# ---- INT8, per-row scale --------------------------------------------------------------
def int8_encode(r):
    """Returns (int8 codes [rows, d], scales [rows] fp32)."""
    r32 = _f32(r)
    amax = np.max(np.abs(r32), axis=-1)
    s = (amax / np.float32(127.0)).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        q = (r32 / s[:, None]).astype(np.float64)
    q = np.where(s[:, None] == 0, 0.0, q)
    return np.clip(np.rint(q), -127, 127).astype(np.int8), s


def int8_decode(codes, s):
    return to_f32(codes.astype(np.float64) * np.asarray(s, dtype=np.float64)[:, None])


# ---- MXFP4 (OCP microscaling), blocks of 32 ------------------------------------------
MX_BLOCK = 32


def mxfp4_encode(r):
    """Returns (E2M1 codes [rows, d] u8, scale exponents [rows, d/32] int: X = 2^e)."""
    r32 = _f32(r).astype(np.float64)
    rows, d = r32.shape
    g = r32.reshape(rows, d // MX_BLOCK, MX_BLOCK)
    amax = np.max(np.abs(g), axis=-1)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(amax > 0, amax, 1.0))) - 2
    e = np.clip(np.where(amax > 0, e, 0), -127, 127).astype(np.int64)  # E8M0 scale range
    q = g / np.power(2.0, e)[..., None]  # exact: a power-of-two scale
    codes, _ = e2m1_round(q)
    codes = np.where(amax[..., None] > 0, codes, 0).astype(np.uint8)
    return codes.reshape(rows, d), e


def mxfp4_decode(codes, e):
    rows, d = codes.shape
    v = e2m1_value(codes).reshape(rows, d // MX_BLOCK, MX_BLOCK) * np.power(2.0, e)[..., None]
    return to_f32(v.reshape(rows, d))


# ---- INT2 (ternary), per-row scale -----------------------------------------------------
def int2_encode(r):
    """Returns (codes in {-1, 0, 1} [rows, d] int8, scales [rows] fp32 = row amax)."""
    r32 = _f32(r).astype(np.float64)
    s = np.max(np.abs(r32), axis=-1)
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.where(s[:, None] > 0, r32 / s[:, None], 0.0)
    return np.clip(np.rint(q), -1, 1).astype(np.int8), s.astype(np.float32)


def int2_decode(codes, s):
    return to_f32(codes.astype(np.float64) * np.asarray(s, dtype=np.float64)[:, None])


# ---- NVFP4 -----------------------------------------------------------------------------
def nvfp4_roundtrip(r):
    codes, sb, _ = nvfp4_encode(r)
    return nvfp4_decode(codes, sb)


FORMATS = {
    # name: (round trip of a [rows, d] array, storage bytes per element for d channels)
    "fp8": (lambda r: fp8_decode(*fp8_encode(r)), lambda d: 1.0 + 4.0 / d),
    "int8": (lambda r: int8_decode(*int8_encode(r)), lambda d: 1.0 + 4.0 / d),
    "mxfp4": (lambda r: mxfp4_decode(*mxfp4_encode(r)), lambda d: 0.5 + 1.0 / MX_BLOCK),
    "int2": (lambda r: int2_decode(*int2_encode(r)), lambda d: 0.25 + 4.0 / d),
    "nvfp4": (nvfp4_roundtrip, lambda d: 0.5 + 1.0 / 16),
}


def reconstruct(h, anchors, labels, fmt, residual=True):
    """Stored-and-restored hidden states of the window rows h [rows, d] (fp32
    values) under one format: with residual=True the format holds h - A_label and
    the anchor is added back (App. C.3 / §4.1), else it holds h itself.  "fp16" is
    always plain.  Returns (h' [rows, d], bytes per element)."""
    h = to_f32(h)
    d = h.shape[1]
    if fmt == "fp16":
        return fp16_roundtrip(h), 2.0
    rt, nbytes = FORMATS[fmt]
    if not residual:
        return rt(h), nbytes(d)
    base = to_f32(np.asarray(anchors, dtype=np.float64)[np.asarray(labels)])
    return to_f32(base + rt(to_f32(h - base))), nbytes(d)


__all__ = ["fp16_roundtrip", "fp8_encode", "fp8_decode", "int8_encode", "int8_decode", "mxfp4_encode",
           "mxfp4_decode", "int2_encode", "int2_decode", "nvfp4_roundtrip", "reconstruct", "FORMATS",
           "E2M1_VALUES", "MX_BLOCK"]
