"""Plain float64 CPU oracle for the DSA sparse-attention step (test infrastructure only).

Only tests/, the smoke check and the bench's CPU-baseline leg may import this
package. It shares no code with the CUDA library and imports nothing from it:
inputs arrive as the raw bytes/bit patterns the caches hold and are decoded
here with the decoders in oracle/fp8.py.

Every function computes the plain definition, one query at a time, with numpy
float64 matmuls as the only library primitive.

Method sources (page title, section):
  * lmdeploy "feat: support GLM-5.2", Changes: the DSA step is indexing with a
    radix top-k, shared top-k reuse and sparse FlashMLA over BF16/FP8 caches.
  * mlx-lm "GLM-5.2 (glm_moe_dsa) inference", commit "Add IndexShare": the
    lightning indexer runs on full layers; shared layers reuse the previous
    full layer's top-k. Commit "small-L gather path": attention over each
    position's selected keys with k = v = latent and unembed after; a position
    with fewer than K causally valid keys keeps only the valid ones.
  * mstar "GLM-5.2 with MLA, fp8 MoE and DSA", Tests: sparse equals dense
    within index_topk; absorbed MLA; per-request page tables.
  * lmdeploy "glm5.3-flash support", Operator-level gains: negative indices
    are padding in the sparse MLA index list.
The pages print no formula for the indexer score; this oracle uses the
DeepSeek-V3.2 lightning-indexer definition
    I[t, s] = sum_h w[t, h] * ReLU(q[t, h, :] . k[s, :])
with q and k dequantized (e4m3 code times its fp32 scale), and ties in the
top-k broken toward the lower key position.

Readings where the pages are silent:
  * query j (0-based) of request b sits at position L_b - n_b + j, where L_b
    counts the cached tokens including the query tokens' own keys; it sees keys
    0..pos (causal);
  * the attention value vector is the 512-wide latent part of the selected row;
    the score uses all 576 columns;
  * an empty selection gives O = 0 and LSE = -inf.
"""
from __future__ import annotations

import numpy as np

from .fp8 import decode_bf16, decode_e4m3, decode_f32le, decode_int8

PAGE = 64
D_LATENT = 512
# Latent record pages (e4m3 or int8 latent): 656 bytes per token, laid out per page
# of 64 tokens as three planes, codes [64][512] | fp32 scales [64][4] | bf16 RoPE
# [64][64], so that every token's codes, scales and RoPE values start on their own
# 512-, 16- and 128-byte boundaries.
REC_PAGE_BYTES = PAGE * 656
REC_SCALES_AT = PAGE * D_LATENT
REC_ROPE_AT = REC_SCALES_AT + PAGE * 16


# ----------------------------------------------------------------------------- geometry

def query_positions(seq_lens, n_q):
    """(request id, position) of every flattened query token."""
    req, pos = [], []
    for b, (L, n) in enumerate(zip(np.asarray(seq_lens).tolist(), np.asarray(n_q).tolist())):
        for j in range(n):
            req.append(b)
            pos.append(L - n + j)
    return np.array(req, dtype=np.int64), np.array(pos, dtype=np.int64)


def physical_rows(block_table_row, s):
    """Logical token positions of one request -> rows of the flat [P*64, .] cache."""
    s = np.asarray(s, dtype=np.int64)
    return np.asarray(block_table_row, dtype=np.int64)[s // PAGE] * PAGE + s % PAGE


# ----------------------------------------------------------------------------- decoding

def decode_index_q(q_idx, q_scale, qk_dtype):
    """Indexer queries [T, Hi, 128] -> float64 (code * per-(t,h) scale for e4m3)."""
    if qk_dtype == "bf16":
        return decode_bf16(q_idx)
    return decode_e4m3(q_idx) * np.asarray(q_scale, dtype=np.float64)[..., None]


def decode_index_keys(idx_k, idx_k_scale, qk_dtype, rows):
    """Selected rows of the paged index-key cache -> float64 [len(rows), 128]."""
    flat = idx_k.reshape(-1, idx_k.shape[-1])[rows]
    if qk_dtype == "bf16":
        return decode_bf16(flat)
    return decode_e4m3(flat) * np.asarray(idx_k_scale, dtype=np.float64).reshape(-1)[rows][:, None]


def record_planes(kv):
    """A latent record cache [P, 64*656] bytes -> its per-token fields as views:
    codes [P, 64, 512], scale bytes [P, 64, 16], RoPE bytes [P, 64, 128]."""
    pages = np.asarray(kv).reshape(-1, REC_PAGE_BYTES)
    P = pages.shape[0]
    return (pages[:, :REC_SCALES_AT].reshape(P, PAGE, D_LATENT),
            pages[:, REC_SCALES_AT:REC_ROPE_AT].reshape(P, PAGE, 16),
            pages[:, REC_ROPE_AT:].reshape(P, PAGE, 128))


def decode_kv_rows(kv, kv_dtype, rows):
    """Selected rows of the paged latent cache -> float64 [len(rows), 576].

    bf16: the 576 stored values. e4m3 or int8 (656-byte record): element 128c+e of
    the latent is code[128c+e] * scale[c] for c = 0..3, followed by the 64 bf16 RoPE
    values; each page stores its tokens' codes, scales and RoPE values as three planes
    (record_planes). The int8 latent cache is mlx-lm "GLM-5.2 (glm_moe_dsa)
    inference", int8 MLA latent KV (only the compressed latent is quantized,
    dequantized on read); its layout is the e4m3 record's with two's-complement codes.
    """
    rows = np.asarray(rows, dtype=np.int64)
    if kv_dtype == "bf16":
        return decode_bf16(kv.reshape(-1, kv.shape[-1])[rows])
    codes, scale_bytes, rope_bytes = record_planes(kv)
    page, slot = rows // PAGE, rows % PAGE
    c = codes[page, slot]                                             # [n, 512]
    lat = decode_e4m3(c) if kv_dtype == "e4m3" else decode_int8(c)
    scales = decode_f32le(scale_bytes[page, slot])                    # [n, 4]
    lat = lat * np.repeat(scales, 128, axis=1)
    rope = decode_bf16(np.ascontiguousarray(rope_bytes[page, slot]).view("<u2").astype(np.uint16))
    return np.concatenate([lat, rope], axis=1)


# ----------------------------------------------------------------------------- indexer

def indexer_scores(q_idx, q_scale, w, idx_k, idx_k_scale, qk_dtype, seq_lens, n_q,
                   block_table, ts=None):
    """Lightning-indexer scores, one float64 row per query token t in `ts`.

    Row t has pos(t)+1 entries: I[t, s] = sum_h w[t,h] * ReLU(q[t,h,:] . k[s,:]) for
    s = 0..pos(t). Returns a dict t -> row.
    """
    req, pos = query_positions(seq_lens, n_q)
    T = len(req)
    ts = range(T) if ts is None else ts
    out = {}
    cache = {}
    for t in ts:
        b, p = int(req[t]), int(pos[t])
        if b not in cache:
            L = int(np.asarray(seq_lens)[b])
            rows = physical_rows(block_table[b], np.arange(L))
            cache = {b: decode_index_keys(idx_k, idx_k_scale, qk_dtype, rows)}
        keys = cache[b][: p + 1]                                        # [n, 128]
        q = decode_index_q(q_idx[t:t + 1], None if q_scale is None else q_scale[t:t + 1],
                           qk_dtype)[0]                                 # [Hi, 128]
        logits = keys @ q.T                                             # [n, Hi]
        out[t] = np.maximum(logits, 0.0) @ np.asarray(w[t], dtype=np.float64)
    return out


# ----------------------------------------------------------------------------- top-k

def topk_row(scores, k):
    """The k largest entries of one score row (positions 0..n-1), ties to the lower
    position, returned as ascending positions padded with -1 to length k."""
    scores = np.asarray(scores, dtype=np.float64)
    if not np.all(np.isfinite(scores)):
        raise ValueError("scores must be finite")
    n = scores.shape[0]
    order = np.lexsort((np.arange(n), -scores))      # primary: score desc; then position asc
    keep = np.sort(order[: min(k, n)])
    out = np.full(k, -1, dtype=np.int32)
    out[: keep.shape[0]] = keep
    return out


def topk(score_rows, k):
    """dict t -> row  ==>  dict t -> top-k positions."""
    return {t: topk_row(r, k) for t, r in score_rows.items()}


# ----------------------------------------------------------------------------- sparse MLA

def sparse_mla(q, kv, kv_dtype, idx, seq_lens, n_q, block_table, sm_scale, ts=None,
               dv=D_LATENT):
    """Absorbed-MLA attention of each query token over its selected latent rows.

    q: [T, H, D] bf16 bits; idx: [T, k] logical positions (-1 = padding).
    z_i = sm_scale * q[t,h,:] . kv[s_i, :];  p = softmax(z);  O = sum_i p_i kv[s_i, :dv];
    LSE = log(sum_i exp(z_i)). Returns dict t -> (O [H, dv], LSE [H]).
    """
    req, _ = query_positions(seq_lens, n_q)
    T = len(req)
    ts = range(T) if ts is None else ts
    out = {}
    for t in ts:
        b = int(req[t])
        sel = np.asarray(idx[t])
        sel = sel[sel >= 0]
        qt = decode_bf16(q[t])                                           # [H, D]
        H = qt.shape[0]
        if sel.shape[0] == 0:
            out[t] = (np.zeros((H, dv)), np.full(H, -np.inf))
            continue
        rows = physical_rows(block_table[b], sel)
        kvr = decode_kv_rows(kv, kv_dtype, rows)                         # [n, D]
        z = sm_scale * (qt @ kvr.T)                                      # [H, n]
        m = z.max(axis=1, keepdims=True)
        e = np.exp(z - m)
        l = e.sum(axis=1, keepdims=True)
        o = (e / l) @ kvr[:, :dv]
        out[t] = (o, (m + np.log(l))[:, 0])
    return out


def masked_dense_mla(q, kv, kv_dtype, idx, seq_lens, n_q, block_table, sm_scale, ts=None,
                     dv=D_LATENT):
    """The mask formulation of the same attention: every causally valid key of the
    request is scored and the unselected ones get -inf before the softmax."""
    req, pos = query_positions(seq_lens, n_q)
    T = len(req)
    ts = range(T) if ts is None else ts
    out = {}
    for t in ts:
        b, p = int(req[t]), int(pos[t])
        rows = physical_rows(block_table[b], np.arange(p + 1))
        kvr = decode_kv_rows(kv, kv_dtype, rows)
        qt = decode_bf16(q[t])
        z = sm_scale * (qt @ kvr.T)                                      # [H, p+1]
        mask = np.zeros(p + 1, dtype=bool)
        sel = np.asarray(idx[t])
        mask[sel[sel >= 0]] = True
        z = np.where(mask[None, :], z, -np.inf)
        m = z.max(axis=1, keepdims=True)
        e = np.exp(z - m)
        l = e.sum(axis=1, keepdims=True)
        out[t] = ((e / l) @ kvr[:, :dv], (m + np.log(l))[:, 0])
    return out


# ----------------------------------------------------------------------------- full step

def dsa_step(wl, ts=None, reuse_idx=None):
    """One DSA step over every layer of a workload (see the input generator):
    layer 0 runs indexer -> top-k -> attention; later layers reuse layer 0's
    selection (IndexShare). With `reuse_idx` given, no layer runs the indexer.

    Returns dict with 'scores' (t -> row), 'idx' (t -> [k]), 'out' (list per layer of
    t -> (O, LSE)).
    """
    req, _ = query_positions(wl.seq_lens, wl.n_q)
    ts = list(range(len(req))) if ts is None else list(ts)
    if reuse_idx is None:
        scores = indexer_scores(wl.q_idx, wl.q_scale, wl.w, wl.idx_k, wl.idx_k_scale,
                                wl.qk_dtype, wl.seq_lens, wl.n_q, wl.block_table, ts)
        sel = topk(scores, wl.topk)
    else:
        scores = {}
        sel = {t: np.asarray(reuse_idx[t]) for t in ts}
    idx_arr = {t: sel[t] for t in ts}
    outs = []
    for layer in wl.layers:
        outs.append(sparse_mla(layer.q, layer.kv, layer.kv_dtype, idx_arr, wl.seq_lens, wl.n_q,
                               wl.block_table, wl.sm_scale, ts))
    return {"scores": scores, "idx": sel, "out": outs}
