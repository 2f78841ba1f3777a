"""Bit-level decoders used by the oracle (test infrastructure only).

bf16: the upper 16 bits of an IEEE-754 binary32.
e4m3 (OCP FP8 "E4M3FN"): 1 sign bit, 4 exponent bits with bias 7, 3 mantissa
bits; exponent field 0 encodes subnormals m/8 * 2^-6; the single pattern
S.1111.111 is NaN; there is no infinity; the largest finite magnitude is 448.

FP8 KV row (656 bytes, data and scale adjacent per token, as asked for by
"Ascend Sparse Attention Forward 算法与优化技术简析", section
"Decoding KV Cache Layout 优化"): 512 e4m3 latent codes, 4 float32 scales (one
per 128 latent channels), 64 bf16 rope values.  Group size and rope dtype are
this library's reading; the page only fixes that data and scale sit together.

e2m1 (OCP FP4): 1 sign bit, 2 exponent bits with bias 1, 1 mantissa bit;
exponent field 0 encodes the subnormals 0 and 0.5; magnitudes 0, 0.5, 1, 1.5,
2, 3, 4, 6; no infinity or NaN.

FP4 KV row (448 bytes; the same page, section "能不能用 1C1V", names FP4 as a
decoding KV format but gives no layout): 512 e2m1 latent codes packed two per
byte (the low nibble holds the even channel) = 256 bytes, then 16 float32
scales (one per 32 latent channels, the block size of the OCP microscaling
formats) = 64 bytes, then 64 bf16 rope values = 128 bytes.  This is the FP8
row's pattern with 4-bit codes; byte layout and block size are this library's
reading.

Dequantisation: the same page, section "能不能用 1C1V", has decoding turn the
FP8 (or FP4) cache into bfloat16 before the matrix unit.  A dequantised latent channel
is therefore bf16 (round to nearest even) of the float32 product e4m3 * scale:
the rounding is part of the method's input to the attention, taken in float32
as the kernel takes it.
"""
from __future__ import annotations

import numpy as np

D_V = 512
D_ROPE = 64
FP8_GROUP = 128
FP8_ROW_BYTES = 656
FP4_GROUP = 32
FP4_ROW_BYTES = 448


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Decode raw bf16 bit patterns (uint16/int16 array) exactly to float64."""
    u32 = bits.astype(np.uint16).astype(np.uint32) << np.uint32(16)
    return u32.view(np.float32).astype(np.float64)


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 (ties to even), returned as float32."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    b = x.view(np.uint32).astype(np.uint64)
    rounded = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    return bf16_bits_to_f64(rounded.astype(np.uint16)).astype(np.float32)


def e4m3_to_f64(codes: np.ndarray) -> np.ndarray:
    """Decode e4m3 codes (uint8 array) from the format's definition."""
    c = codes.astype(np.int64)
    sign = np.where((c >> 7) & 1, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    normal = (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0)
    sub = (m / 8.0) * 2.0 ** (1 - 7)
    val = np.where(e == 0, sub, normal)
    val = np.where((e == 15) & ((c & 7) == 7), np.nan, val)
    return sign * val


def fp8_rows_to_f64(rows: np.ndarray) -> np.ndarray:
    """Dequantise 656-byte FP8 KV rows [n, 656] (uint8) to float64 [n, 576].

    latent[c] = bf16(float32(e4m3(code[c]) * scale[c // 128])) (see the module note);
    rope = the bf16 values as stored.
    """
    rows = np.ascontiguousarray(rows, dtype=np.uint8)
    n = rows.shape[0]
    lat = e4m3_to_f64(rows[:, :D_V]).astype(np.float32)  # e4m3 values are exact in float32
    scale = rows[:, D_V:D_V + 16].copy().view(np.float32)  # [n, 4]
    lat = round_to_bf16(lat * np.repeat(scale, FP8_GROUP, axis=1)).astype(np.float64)
    rope = bf16_bits_to_f64(rows[:, D_V + 16:].copy().view(np.uint16))
    out = np.empty((n, D_V + D_ROPE), dtype=np.float64)
    out[:, :D_V] = lat
    out[:, D_V:] = rope
    return out


def e2m1_to_f64(codes: np.ndarray) -> np.ndarray:
    """Decode 4-bit e2m1 codes (values 0..15 in an integer array) from the format's definition."""
    c = codes.astype(np.int64)
    sign = np.where((c >> 3) & 1, -1.0, 1.0)
    e = (c >> 1) & 0x3
    m = (c & 0x1).astype(np.float64)
    normal = (1.0 + m / 2.0) * np.exp2(e.astype(np.float64) - 1.0)
    sub = (m / 2.0) * 2.0 ** (1 - 1)
    return sign * np.where(e == 0, sub, normal)


def fp4_rows_to_f64(rows: np.ndarray) -> np.ndarray:
    """Dequantise 448-byte FP4 KV rows [n, 448] (uint8) to float64 [n, 576].

    latent[c] = bf16(float32(e2m1(code[c]) * scale[c // 32])), code[2i] in the low nibble of byte i;
    rope = the bf16 values as stored.
    """
    rows = np.ascontiguousarray(rows, dtype=np.uint8)
    n = rows.shape[0]
    packed = rows[:, :D_V // 2].astype(np.int64)
    codes = np.empty((n, D_V), dtype=np.int64)
    codes[:, 0::2] = packed & 0xF
    codes[:, 1::2] = packed >> 4
    lat = e2m1_to_f64(codes).astype(np.float32)  # e2m1 values are exact in float32
    scale = rows[:, D_V // 2:D_V // 2 + 64].copy().view(np.float32)  # [n, 16]
    lat = round_to_bf16(lat * np.repeat(scale, FP4_GROUP, axis=1)).astype(np.float64)
    rope = bf16_bits_to_f64(rows[:, D_V // 2 + 64:].copy().view(np.uint16))
    out = np.empty((n, D_V + D_ROPE), dtype=np.float64)
    out[:, :D_V] = lat
    out[:, D_V:] = rope
    return out
