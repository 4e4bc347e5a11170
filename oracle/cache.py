"""Cache append for the oracle (test infrastructure only): writing new tokens' latent
rows and index keys into the paged caches, with the e4m3 encodings written out from
their definition.

Only tests/, the smoke check and the bench's CPU-baseline leg may import this
package; the CUDA library never does.

What it computes (lmdeploy "feat: support GLM-5.2", Changes: "BF16/FP8 sparse
FlashMLA cache paths", the MLA cache dtype policy; lmdeploy "glm5.3-flash support":
"cache updates still run on every draft step"). The pages name the cache write but
print no layout or rounding, so this follows the layouts the attention reads:
  * token j of request b (flattened like the queries) sits at position
    L_b - n_b + j, physical row block_table[b][pos // 64] * 64 + pos % 64;
  * bf16 latent cache: the 576 bf16 values as given;
  * int8 latent record (mlx-lm "GLM-5.2 (glm_moe_dsa) inference": int8 MLA latent
    KV, only the compressed latent quantized): the e4m3 record's layout with
    two's-complement int8 codes, scale_c = amax_c / 127 and the quotient rounded to
    the nearest integer (ties to even), clamped to +-127;
  * e4m3 latent record (656 bytes): for each group c of 128 latent values,
    scale_c = amax_c / 448 in fp32 (1 for an all-zero group) and
    code = e4m3(x / scale_c), the quotient taken in fp32 and rounded to the nearest
    e4m3 value, ties to the even code, saturating at +-448; the 512 codes, the four
    scales (little-endian fp32) and the 64 RoPE values (bf16) go to the token's slot
    of its page's three planes (codes [64][512], scales [64][4], RoPE [64][64]);
  * index keys: e4m3 with one such scale per token over its 128 values (or bf16 as
    given); the scale goes to the [P, 64] scale tensor.
The fp32 steps are taken in fp32 on purpose: they decide integer codes, and the
kernel takes them in fp32.
"""
from __future__ import annotations

import numpy as np

from .dsa import record_planes
from .fp8 import E4M3_TABLE

E4M3_MAX = 448.0
PAGE = 64

# finite non-negative e4m3 magnitudes and their codes, ascending (codes 0x00..0x7E)
_POS_CODES = np.arange(0x7F, dtype=np.uint8)
_POS_VALUES = E4M3_TABLE[:0x7F]


def encode_e4m3(v: np.ndarray) -> np.ndarray:
    """Round values (held exactly in float64) to e4m3 codes: the nearest finite e4m3
    value, ties to the code with an even mantissa (even code), magnitudes at or beyond
    448 saturating to 448, the sign kept (so -0 and small negatives give 0x80)."""
    v = np.asarray(v, dtype=np.float64)
    if not np.all(np.isfinite(v)):
        raise ValueError("e4m3 encoding expects finite values")
    mag = np.abs(v)
    hi = np.searchsorted(_POS_VALUES, mag, side="left")          # first value >= mag
    hi = np.minimum(hi, len(_POS_VALUES) - 1)
    lo = np.maximum(hi - 1, 0)
    d_lo = mag - _POS_VALUES[lo]
    d_hi = _POS_VALUES[hi] - mag
    take_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (_POS_CODES[hi] % 2 == 0))
    code = np.where(take_hi, _POS_CODES[hi], _POS_CODES[lo]).astype(np.uint8)
    code = np.where(mag >= E4M3_MAX, np.uint8(0x7E), code)        # saturate
    code = np.where(mag == _POS_VALUES[hi], _POS_CODES[hi], code)  # exact values
    neg = np.signbit(v)
    return (code | np.where(neg, np.uint8(0x80), np.uint8(0))).astype(np.uint8)


def group_scale(x32: np.ndarray) -> np.ndarray:
    """fp32 scale per row of the last axis: amax / 448 in fp32, 1 for an all-zero row."""
    x32 = np.asarray(x32, dtype=np.float32)
    amax = np.abs(x32).max(axis=-1)
    return np.where(amax > 0, amax / np.float32(E4M3_MAX), np.float32(1.0)).astype(np.float32)


def quantize_groups(x32: np.ndarray, group: int) -> tuple[np.ndarray, np.ndarray]:
    """e4m3 codes of x / scale (fp32 quotient) per run of `group` values along the last
    axis, and the fp32 scales."""
    x32 = np.asarray(x32, dtype=np.float32)
    g = x32.reshape(*x32.shape[:-1], x32.shape[-1] // group, group)
    scale = group_scale(g)
    q = (g / scale[..., None]).astype(np.float32)                 # fp32 division
    return encode_e4m3(q.astype(np.float64)).reshape(x32.shape), scale


I8_MAX = 127.0


def encode_int8(v: np.ndarray) -> np.ndarray:
    """Round values (held exactly in float64) to the nearest integer, ties to even,
    clamp to [-127, 127], and return the two's-complement bytes."""
    v = np.asarray(v, dtype=np.float64)
    if not np.all(np.isfinite(v)):
        raise ValueError("int8 encoding expects finite values")
    fl = np.floor(v)
    frac = v - fl
    up = (frac > 0.5) | ((frac == 0.5) & (np.mod(fl, 2) == 1))
    q = np.clip(fl + up, -I8_MAX, I8_MAX).astype(np.int64)
    return q.astype(np.int8).view(np.uint8)


def quantize_groups_int8(x32: np.ndarray, group: int) -> tuple[np.ndarray, np.ndarray]:
    """int8 codes of x / scale (fp32 quotient), scale = amax / 127 in fp32 (1 for an
    all-zero group), per run of `group` values along the last axis."""
    x32 = np.asarray(x32, dtype=np.float32)
    g = x32.reshape(*x32.shape[:-1], x32.shape[-1] // group, group)
    amax = np.abs(g).max(axis=-1)
    scale = np.where(amax > 0, amax / np.float32(I8_MAX), np.float32(1.0)).astype(np.float32)
    q = (g / scale[..., None]).astype(np.float32)
    return encode_int8(q.astype(np.float64)).reshape(x32.shape), scale


def token_rows(seq_lens, n_q, block_table) -> np.ndarray:
    """Physical cache row of every new token (flattened like the queries)."""
    rows = []
    for b, (L, n) in enumerate(zip(seq_lens, n_q)):
        for j in range(int(n)):
            pos = int(L) - int(n) + j
            rows.append(int(block_table[b][pos // PAGE]) * PAGE + pos % PAGE)
    return np.asarray(rows, dtype=np.int64)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    bits = np.asarray(bits, dtype=np.uint16)
    return (bits.astype(np.uint32) << 16).view(np.float32)


def cache_append(kv_cache, kv_dtype, kv_new_bits, idx_k_cache, idx_k_scale, qk_dtype, k_new_bits,
                 seq_lens, n_q, block_table):
    """Return updated copies of the caches after appending the new tokens.

    kv_cache: [P, 64, 576] uint16 (bf16 bits) or [P, 64 * 656] uint8 (e4m3 / int8 record pages).
    kv_new_bits: [T, 576] uint16 bf16 bits.
    idx_k_cache: [P, 64, 128] uint8 (e4m3) or uint16 (bf16 bits), or None;
    idx_k_scale: [P, 64] float32 or None; k_new_bits: [T, 128] uint16 or None.
    """
    rows = token_rows(seq_lens, n_q, block_table)
    kv = np.array(kv_cache, copy=True)
    x = bf16_bits_to_f32(kv_new_bits)
    if kv_dtype == "bf16":
        flat = kv.reshape(-1, kv.shape[-1])
    else:
        code_plane, scale_plane, rope_plane = record_planes(kv)
    for t, r in enumerate(rows):
        if kv_dtype == "bf16":
            flat[r] = np.asarray(kv_new_bits[t], dtype=np.uint16)
        else:
            quant = quantize_groups if kv_dtype == "e4m3" else quantize_groups_int8
            codes, scales = quant(x[t, :512], 128)
            page, slot = r // PAGE, r % PAGE
            code_plane[page, slot] = codes
            scale_plane[page, slot] = np.ascontiguousarray(scales, dtype="<f4").view(np.uint8)
            rope_plane[page, slot] = np.ascontiguousarray(np.asarray(kv_new_bits[t, 512:], dtype=np.uint16),
                                                          dtype="<u2").view(np.uint8)
    out_k = out_s = None
    if idx_k_cache is not None:
        out_k = np.array(idx_k_cache, copy=True)
        kflat = out_k.reshape(-1, 128)
        out_s = None if idx_k_scale is None else np.array(idx_k_scale, copy=True).reshape(-1)
        xk = bf16_bits_to_f32(k_new_bits)
        for t, r in enumerate(rows):
            if qk_dtype == "bf16":
                kflat[r] = np.asarray(k_new_bits[t], dtype=np.uint16)
            else:
                codes, scale = quantize_groups(xk[t], 128)
                kflat[r] = codes
                out_s[r] = scale[0]
        if out_s is not None:
            out_s = out_s.reshape(np.shape(idx_k_scale))
    return kv, out_k, out_s
