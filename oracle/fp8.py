"""Storage-format decoders for the oracle (test infrastructure only).

Only tests/, the smoke check and the bench's CPU-baseline leg may import this
package; the CUDA library never does.

E4M3 follows the OCP 8-bit floating point specification (the "fn" variant):
1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits; exponent field 0
encodes subnormals m * 2^-9; S.1111.111 is NaN; there are no infinities and
the largest finite magnitude is 448. BF16 is the upper half of an IEEE-754
binary32 pattern. The pages name the formats (lmdeploy "feat: support GLM-5.2",
Changes: "BF16/FP8 sparse FlashMLA cache paths") but print no encoding.
"""
from __future__ import annotations

import numpy as np


def _e4m3_value(code: int) -> float:
    sign = -1.0 if code & 0x80 else 1.0
    exp = (code >> 3) & 0xF
    man = code & 0x7
    if exp == 0xF and man == 0x7:
        return float("nan")
    if exp == 0:
        return sign * man * 2.0 ** -9
    return sign * (1.0 + man / 8.0) * 2.0 ** (exp - 7)


E4M3_TABLE = np.array([_e4m3_value(c) for c in range(256)], dtype=np.float64)


def decode_e4m3(codes: np.ndarray) -> np.ndarray:
    """uint8 e4m3 codes -> float64 values (exact)."""
    codes = np.asarray(codes)
    if codes.dtype != np.uint8:
        raise TypeError("e4m3 codes must be uint8")
    return E4M3_TABLE[codes]


def decode_bf16(bits: np.ndarray) -> np.ndarray:
    """uint16 bf16 bit patterns -> float64 values (exact)."""
    bits = np.asarray(bits)
    if bits.dtype != np.uint16:
        raise TypeError("bf16 bits must be uint16")
    with np.errstate(invalid="ignore"):
        return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def decode_f32le(raw: np.ndarray) -> np.ndarray:
    """Little-endian fp32 stored as raw bytes (last axis a multiple of 4) -> float64."""
    raw = np.ascontiguousarray(raw, dtype=np.uint8)
    return raw.view("<f4").astype(np.float64)


def decode_int8(codes: np.ndarray) -> np.ndarray:
    """uint8 bytes holding two's-complement int8 codes -> float64 values (exact)."""
    codes = np.asarray(codes)
    if codes.dtype != np.uint8:
        raise TypeError("int8 codes must be stored as uint8 bytes")
    return codes.view(np.int8).astype(np.float64)
