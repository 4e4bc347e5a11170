"""Indexer query/key preparation for the oracle (test infrastructure only).

Only tests/, the smoke check and the bench's CPU-baseline leg may import this
package; the CUDA library never does.

What it computes (lmdeploy "feat: support GLM-5.2", Changes: "fused indexer
preparation" in the DSA indexing work, and Performance: fused Q/K preprocessing of
the indexer; mlx-lm "GLM-5.2 (glm_moe_dsa) inference", Changes: the indexer's RoPE is
non-interleaved, unlike the main attention's interleaved RoPE, and its LayerNorm
uses eps 1e-6). The pages name these steps without formulas; this file follows the
plainest reading of them:
  * RoPE, non-interleaved ("rotate half"): on the first rope_dim values of a
    128-value vector, element i < rope_dim/2 pairs with element i + rope_dim/2:
        y_i          = x_i * cos[p, i] - x_{i+r} * sin[p, i]
        y_{i+r}      = x_{i+r} * cos[p, i] + x_i * sin[p, i]      (r = rope_dim/2)
    at the token's position p; values past rope_dim pass through. The cos/sin
    tables are inputs (the model's RoPE base is not a reading made here).
  * the key is layer-normalized before its RoPE: (x - mean) / sqrt(var + eps) *
    gamma + beta over its 128 values, var the biased (population) variance;
  * each query head (per token and head) and each key (per token) is then
    quantized to e4m3 with scale = amax / 448 (1 for an all-zero vector), the
    quotient taken in fp32 and rounded to the nearest e4m3 value (oracle.cache);
  * the key's codes and scale go to the paged index cache at the token's row.
RoPE and LayerNorm are computed in float64 here; the fp32 rounding of their
results is the one step where a kernel computing in fp32 may differ from this
file by an ulp, which can move a quantized code across a rounding boundary.
"""
from __future__ import annotations

import numpy as np

from .cache import quantize_groups, token_rows, bf16_bits_to_f32

DIM = 128


def rope_rotate_half(x, cos, sin, rope_dim):
    """Apply non-interleaved RoPE to the first rope_dim values of the last axis.

    x: [..., 128] float64; cos, sin: [..., rope_dim/2] (broadcast against x's
    leading axes) float64."""
    x = np.asarray(x, dtype=np.float64)
    r = rope_dim // 2
    a, b = x[..., :r], x[..., r:rope_dim]
    c, s = np.asarray(cos, dtype=np.float64), np.asarray(sin, dtype=np.float64)
    y = x.copy()
    y[..., :r] = a * c - b * s
    y[..., r:rope_dim] = b * c + a * s
    return y


def layer_norm(x, gamma, beta, eps):
    """LayerNorm over the last axis with the biased variance, in float64."""
    x = np.asarray(x, dtype=np.float64)
    mu = x.mean(axis=-1, keepdims=True)
    var = ((x - mu) ** 2).mean(axis=-1, keepdims=True)
    return (x - mu) / np.sqrt(var + float(eps)) * np.asarray(gamma, np.float64) + np.asarray(beta, np.float64)


def prepared_q(q_bits, pos, cos_table, sin_table, rope_dim):
    """Indexer queries after RoPE, before quantization: [T, H, 128] float64.

    q_bits: [T, H, 128] bf16 bits; pos: [T] positions; tables [max_len, rope_dim/2]."""
    q = bf16_bits_to_f32(q_bits).astype(np.float64)
    c = np.asarray(cos_table, np.float64)[pos][:, None, :]
    s = np.asarray(sin_table, np.float64)[pos][:, None, :]
    return rope_rotate_half(q, c, s, rope_dim)


def prepared_k(k_bits, pos, cos_table, sin_table, rope_dim, gamma, beta, eps):
    """Indexer keys after LayerNorm and RoPE, before quantization: [T, 128] float64."""
    k = bf16_bits_to_f32(k_bits).astype(np.float64)
    kn = layer_norm(k, gamma, beta, eps)
    c = np.asarray(cos_table, np.float64)[pos]
    s = np.asarray(sin_table, np.float64)[pos]
    return rope_rotate_half(kn, c, s, rope_dim)


def indexer_prepare(q_bits, k_bits, seq_lens, n_q, block_table, cos_table, sin_table, rope_dim,
                    gamma, beta, eps, idx_k_cache=None, idx_k_scale=None):
    """The whole preparation: (q codes [T,H,128] u8, q scales [T,H] f32, updated key
    cache copy, updated key-scale copy). Positions and rows follow the query
    flattening (request b's token j at seq_lens[b] - n_b + j)."""
    from .dsa import query_positions
    _, pos = query_positions(seq_lens, n_q)
    qx = prepared_q(q_bits, pos, cos_table, sin_table, rope_dim)
    T, H, _ = qx.shape
    q_codes, q_scale = quantize_groups(qx.astype(np.float32).reshape(T, H * DIM), DIM)
    q_codes = q_codes.reshape(T, H, DIM)
    out_k = out_s = None
    if k_bits is not None:
        kx = prepared_k(k_bits, pos, cos_table, sin_table, rope_dim, gamma, beta, eps)
        k_codes, k_scale = quantize_groups(kx.astype(np.float32), DIM)
        rows = token_rows(seq_lens, n_q, block_table)
        out_k = np.array(idx_k_cache, copy=True)
        out_s = np.array(idx_k_scale, copy=True)
        kflat, sflat = out_k.reshape(-1, DIM), out_s.reshape(-1)
        for t, r in enumerate(rows):
            kflat[r] = k_codes[t]
            sflat[r] = k_scale[t, 0]
    return q_codes, q_scale, out_k, out_s
