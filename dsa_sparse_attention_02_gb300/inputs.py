"""Seeded synthetic inputs for the DSA sparse-attention step.

This module is the one piece shared by the CUDA path's tests/bench and the
CPU oracle. It draws random tensors and stores them in the formats the caches
use (e4m3 bytes, bf16 bit patterns, fp32); it computes none of the method's
arithmetic (no scores, no selection, no attention).

The workloads are the five configurations of the DSA step:

  tiny       batch 2, contexts {200, 256}, 1 query token, index_topk 64,
             4 indexer heads with bf16 q/k, 16 MLA heads, bf16 latent KV
  decode     batch 64, contexts ~U[2048, 8192], 1 query token, index_topk 2048,
             64 indexer heads with e4m3 q/k + fp32 scales, bf16 latent KV
  mtp        batch 32, contexts ~U[4096, 16384], 4 causal query tokens,
             index_topk 2048, e4m3 latent KV (per-128 scales + bf16 RoPE),
             two layers where the second reuses the first's selection
  prefill    1 request, 16384 cached tokens, 2048-token query chunk at
             positions 14336..16383, index_topk 2048, bf16 latent KV
  longctx    batch 8, contexts 131072, 1 query token, index_topk 2048,
             1% of index-key rows duplicated so that scores tie exactly

The pages describe GLM-5.2 serving (lmdeploy "feat: support GLM-5.2",
mstar "GLM-5.2 with MLA, fp8 MoE and DSA", mlx-lm "GLM-5.2 (glm_moe_dsa)
inference") on trained weights; these synthetic tensors stand in for them
with the same shapes.

Storage formats (one token per row, pages of 64 tokens):
  index key cache   [P, 64, 128] e4m3 bytes + [P, 64] fp32 per-token scale,
                    or [P, 64, 128] bf16 bits (no scale) for the tiny case
  latent KV, bf16   [P, 64, 576] bf16 bits (512 latent + 64 RoPE)
  latent KV, e4m3   [P, 64 * 656] bytes, 656 per token as three planes per page:
                    codes [64][512] e4m3, scales [64][4] fp32 (one per 128 latent
                    elements), RoPE [64][64] bf16; int8 latent the same with
                    two's-complement codes
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

PAGE = 64
D_IDX = 128
D_LATENT = 512
D_ROPE = 64
D_QK = D_LATENT + D_ROPE
FP8_RECORD = D_LATENT + 4 * 4 + 2 * D_ROPE  # 656 bytes per token
REC_PAGE_BYTES = PAGE * FP8_RECORD           # a page of latent records: codes | scales | RoPE planes
E4M3_MAX = 448.0

CONFIG_NAMES = ("tiny", "decode", "mtp", "prefill", "longctx")
CONFIG_SEEDS = {"tiny": 1, "decode": 2, "mtp": 3, "prefill": 4, "longctx": 5}


@dataclass
class Layer:
    """One attention layer's MLA inputs."""
    q: np.ndarray            # [T, H, 576] uint16 (bf16 bits)
    kv: np.ndarray           # [P, 64, 576] uint16 (bf16) or [P, 64 * 656] uint8 (record pages)
    kv_dtype: str            # "bf16", "e4m3" or "int8"


@dataclass
class Workload:
    name: str
    seq_lens: np.ndarray     # [B] int32, cached tokens including the query tokens
    n_q: np.ndarray          # [B] int32, query tokens per request
    cu_q: np.ndarray         # [B+1] int32
    block_table: np.ndarray  # [B, max_pages] int32, physical page ids
    num_pages: int
    topk: int
    qk_dtype: str            # "e4m3" or "bf16" (indexer q and keys)
    q_idx: np.ndarray        # [T, Hi, 128] uint8 (e4m3) or uint16 (bf16 bits)
    q_scale: np.ndarray | None   # [T, Hi] fp32 or None
    w: np.ndarray            # [T, Hi] fp32
    idx_k: np.ndarray        # [P, 64, 128] uint8 (e4m3) or uint16 (bf16 bits)
    idx_k_scale: np.ndarray | None  # [P, 64] fp32 or None
    layers: list = field(default_factory=list)   # list[Layer]; layer 0 is the full layer
    sm_scale: float = 1.0 / math.sqrt(192.0)
    heads: int = 16

    @property
    def B(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def T(self) -> int:
        return int(self.cu_q[-1])

    @property
    def Hi(self) -> int:
        return int(self.w.shape[1])

    @property
    def max_seq_len(self) -> int:
        return int(self.seq_lens.max()) if self.B else 0


# --------------------------------------------------------------------------- storage casts

def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (round to nearest even) and return the bit patterns."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


def to_e4m3_bytes(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to e4m3 (nearest even), saturating at +-448, and return the bytes."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).clamp(-E4M3_MAX, E4M3_MAX)
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy().copy()


def quantize_rows_e4m3(x: np.ndarray, group: int) -> tuple[np.ndarray, np.ndarray]:
    """Scale each run of `group` trailing elements by amax/448 and cast to e4m3.

    Returns (bytes with x's shape, fp32 scales with shape x.shape[:-1] + (x.shape[-1]//group,)).
    """
    shp = x.shape
    g = x.reshape(*shp[:-1], shp[-1] // group, group).astype(np.float32)
    amax = np.abs(g).max(axis=-1)
    scale = np.where(amax > 0, amax / np.float32(E4M3_MAX), np.float32(1.0)).astype(np.float32)
    codes = to_e4m3_bytes(g / scale[..., None])
    return codes.reshape(shp), scale


# --------------------------------------------------------------------------- geometry

def make_geometry(rng: np.random.Generator, seq_lens, n_q, spare_frac: float = 0.05):
    """Block tables: a random permutation of all physical pages, split across requests,
    plus `spare_frac` extra pages that no request references."""
    seq_lens = np.asarray(seq_lens, dtype=np.int64)
    n_q = np.asarray(n_q, dtype=np.int64)
    pages_per = (seq_lens + PAGE - 1) // PAGE
    used = int(pages_per.sum())
    num_pages = used + int(math.ceil(spare_frac * used))
    perm = rng.permutation(num_pages).astype(np.int32)
    max_pages = int(pages_per.max()) if len(pages_per) else 1
    bt = np.zeros((len(seq_lens), max(max_pages, 1)), dtype=np.int32)
    off = 0
    for b, npg in enumerate(pages_per):
        bt[b, :npg] = perm[off:off + npg]
        off += int(npg)
    cu_q = np.zeros(len(seq_lens) + 1, dtype=np.int32)
    cu_q[1:] = np.cumsum(n_q)
    return seq_lens.astype(np.int32), n_q.astype(np.int32), cu_q, bt, num_pages


def _normal(rng, shape, std=1.0) -> np.ndarray:
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return x


def make_kv_bf16(rng, num_pages: int) -> np.ndarray:
    """Latent KV rows ~ N(0, 0.5^2), stored as bf16 bits, [P, 64, 576]."""
    return to_bf16_bits(_normal(rng, (num_pages, PAGE, D_QK), 0.5))


def record_pages(codes: np.ndarray, scales: np.ndarray, rope_bits: np.ndarray) -> np.ndarray:
    """Latent record pages [P, 64 * 656] from codes [P, 64, 512] (bytes), scales
    [P, 64, 4] (fp32) and RoPE [P, 64, 64] (bf16 bits): per page the 64 tokens' codes,
    then their scales, then their RoPE values (a storage layout, no arithmetic)."""
    P = codes.shape[0]
    rec = np.empty((P, REC_PAGE_BYTES), dtype=np.uint8)
    rec[:, :PAGE * D_LATENT] = codes.reshape(P, -1)
    rec[:, PAGE * D_LATENT:PAGE * (D_LATENT + 16)] = np.ascontiguousarray(scales, dtype="<f4").view(np.uint8).reshape(P, -1)
    rec[:, PAGE * (D_LATENT + 16):] = np.ascontiguousarray(rope_bits, dtype="<u2").view(np.uint8).reshape(P, -1)
    return rec


def make_kv_e4m3(rng, num_pages: int) -> np.ndarray:
    """Latent KV rows ~ N(0, 0.5^2) as 656-byte records: the 512 latent values in
    e4m3 with one fp32 scale (amax/448) per 128 of them, then the 64 RoPE values in bf16."""
    x = _normal(rng, (num_pages, PAGE, D_QK), 0.5)
    codes, scales = quantize_rows_e4m3(x[..., :D_LATENT], 128)
    return record_pages(codes, scales, to_bf16_bits(x[..., D_LATENT:]))


def make_kv_int8(rng, num_pages: int) -> np.ndarray:
    """Latent KV rows ~ N(0, 0.5^2) as 656-byte records: the 512 latent values as int8
    with one fp32 scale (amax/127) per 128 of them, then the 64 RoPE values in bf16."""
    x = _normal(rng, (num_pages, PAGE, D_QK), 0.5)
    g = x[..., :D_LATENT].reshape(num_pages, PAGE, 4, 128)
    amax = np.abs(g).max(axis=-1)
    scales = np.where(amax > 0, amax / np.float32(127.0), np.float32(1.0)).astype(np.float32)
    codes = np.clip(np.rint(g / scales[..., None]), -127, 127).astype(np.int8).view(np.uint8)
    return record_pages(codes.reshape(num_pages, PAGE, D_LATENT), scales, to_bf16_bits(x[..., D_LATENT:]))


def make_workload(name: str, seq_lens, n_q, topk: int, hi: int, qk_dtype: str,
                  kv_dtypes=("bf16",), heads: int = 16, seed: int = 0,
                  dup_key_frac: float = 0.0, spare_frac: float = 0.05) -> Workload:
    """Build one synthetic workload. `kv_dtypes` has one entry per layer."""
    rng = np.random.Generator(np.random.PCG64(seed))
    seq_lens, n_q, cu_q, bt, P = make_geometry(rng, seq_lens, n_q, spare_frac)
    if np.any(n_q > seq_lens):
        raise ValueError("a request has more query tokens than cached tokens")
    T = int(cu_q[-1])
    if qk_dtype == "e4m3":
        q_idx, q_scale = quantize_rows_e4m3(_normal(rng, (T, hi, D_IDX)), D_IDX)
        q_scale = q_scale[..., 0]
        idx_k, k_scale = quantize_rows_e4m3(_normal(rng, (P, PAGE, D_IDX)), D_IDX)
        k_scale = k_scale[..., 0]
    elif qk_dtype == "bf16":
        q_idx = to_bf16_bits(_normal(rng, (T, hi, D_IDX)))
        q_scale = None
        idx_k = to_bf16_bits(_normal(rng, (P, PAGE, D_IDX)))
        k_scale = None
    else:
        raise ValueError(qk_dtype)
    w = (_normal(rng, (T, hi)) * np.float32(0.5)).astype(np.float32)

    if dup_key_frac > 0:
        # Copy whole index-key rows (bytes and scale) onto other positions of the same
        # request so that their scores tie exactly.
        flat_k = idx_k.reshape(P * PAGE, -1)
        flat_s = k_scale.reshape(-1) if k_scale is not None else None
        for b in range(len(seq_lens)):
            L = int(seq_lens[b])
            nd = int(round(dup_key_frac * L))
            if nd == 0 or L < 2:
                continue
            dst = rng.choice(L, size=nd, replace=False)
            src = rng.integers(0, L, size=nd)
            prow = lambda s: bt[b, s // PAGE].astype(np.int64) * PAGE + s % PAGE
            flat_k[prow(dst)] = flat_k[prow(src)]
            if flat_s is not None:
                flat_s[prow(dst)] = flat_s[prow(src)]

    layers = []
    for kd in kv_dtypes:
        q = to_bf16_bits(_normal(rng, (T, heads, D_QK)))
        kv = make_kv_bf16(rng, P) if kd == "bf16" else (make_kv_e4m3(rng, P) if kd == "e4m3" else make_kv_int8(rng, P))
        layers.append(Layer(q=q, kv=kv, kv_dtype=kd))

    return Workload(name=name, seq_lens=seq_lens, n_q=n_q, cu_q=cu_q, block_table=bt,
                    num_pages=P, topk=int(topk), qk_dtype=qk_dtype, q_idx=q_idx,
                    q_scale=None if q_scale is None else q_scale.astype(np.float32),
                    w=w, idx_k=idx_k,
                    idx_k_scale=None if k_scale is None else k_scale.astype(np.float32),
                    layers=layers, heads=heads)


def make_config(name: str, batch: int | None = None, seed: int | None = None,
                ctx_scale: float = 1.0, latent: str | None = None) -> Workload:
    """The five configurations, optionally with a smaller batch or shorter contexts
    (`ctx_scale` < 1 shrinks the context range; used for quick parity runs), or with
    every layer's latent cache in another format (`latent`: "bf16", "e4m3", "int8")."""
    wl = _make_config(name, batch, seed, ctx_scale, latent)
    return wl


def _make_config(name, batch, seed, ctx_scale, latent):
    s = CONFIG_SEEDS[name] if seed is None else seed
    rng = np.random.Generator(np.random.PCG64(s + 1000))

    def U(lo, hi, n):
        lo, hi = int(lo * ctx_scale), int(hi * ctx_scale)
        return rng.integers(lo, hi, size=n, endpoint=True)

    if name == "tiny":
        B = 2 if batch is None else batch
        lens = ([200, 256] * B)[:B]
        return make_workload(name, lens, [1] * B, 64, 4, "bf16", _lat(("bf16",), latent), seed=s)
    if name == "decode":
        B = 64 if batch is None else batch
        return make_workload(name, U(2048, 8192, B), [1] * B, 2048, 64, "e4m3", _lat(("bf16",), latent), seed=s)
    if name == "mtp":
        B = 32 if batch is None else batch
        return make_workload(name, U(4096, 16384, B), [4] * B, 2048, 64, "e4m3",
                             _lat(("e4m3", "e4m3"), latent), seed=s)
    if name == "prefill":
        L = int(16384 * ctx_scale)
        nq = min(2048, L) if batch is None else batch
        return make_workload(name, [L], [nq], 2048, 64, "e4m3", _lat(("bf16",), latent), seed=s)
    if name == "longctx":
        B = 8 if batch is None else batch
        L = int(131072 * ctx_scale)
        return make_workload(name, [L] * B, [1] * B, 2048, 64, "e4m3", _lat(("bf16",), latent), seed=s,
                             dup_key_frac=0.01)
    raise KeyError(name)


def _lat(kv_dtypes, latent):
    return kv_dtypes if latent is None else tuple(latent for _ in kv_dtypes)


def tied_scores(rng: np.random.Generator, rows: int, n: int, frac: float = 0.01,
                kth_copies: int = 4, k: int = 2048) -> np.ndarray:
    """fp32 score rows ~N(0,1) where `frac` of the entries are overwritten with copies of
    other entries of the same row, including several copies of the row's k-th largest
    value (the standalone top-k workload of the long-context case)."""
    s = rng.standard_normal(size=(rows, n), dtype=np.float32)
    nd = max(1, int(frac * n))
    for r in range(rows):
        dst = rng.choice(n, size=nd, replace=False)
        src = rng.integers(0, n, size=nd)
        s[r, dst] = s[r, src]
        if n > k:
            kth = np.sort(s[r])[::-1][k - 1]
            where = rng.choice(n, size=kth_copies, replace=False)
            s[r, where] = kth
    return s


@dataclass
class PrepInputs:
    """Raw indexer inputs of the new tokens, before RoPE / LayerNorm / quantization."""
    q_in: np.ndarray         # [T, Hi, 128] uint16 (bf16 bits) ~N(0, 1)
    k_in: np.ndarray         # [T, 128] uint16 (bf16 bits) ~N(0.3, 2^2)
    rope_cos: np.ndarray     # [max_seq_len, rope_dim/2] fp32
    rope_sin: np.ndarray     # [max_seq_len, rope_dim/2] fp32
    ln_gamma: np.ndarray     # [128] fp32 ~1 + N(0, 0.1^2)
    ln_beta: np.ndarray      # [128] fp32 ~N(0, 0.1^2)
    ln_eps: float
    rope_dim: int


def make_prep_inputs(wl: Workload, hi: int = 64, rope_dim: int = 64, seed: int = 0,
                     rope_base: float = 10000.0) -> PrepInputs:
    """Seeded raw indexer q/k for the workload's query tokens and the model's RoPE
    tables (angle p * base^(-2i/rope_dim) at position p, pair i), which are weights
    of the model, not a step of the preparation."""
    rng = np.random.default_rng(seed)
    T = int(wl.n_q.sum())
    q = _normal(rng, (T, hi, 128))
    k = _normal(rng, (T, 128), std=2.0) + np.float32(0.3)
    r = rope_dim // 2
    inv = rope_base ** (-np.arange(r, dtype=np.float64) * 2.0 / rope_dim)
    ang = np.arange(int(wl.max_seq_len), dtype=np.float64)[:, None] * inv[None, :]
    return PrepInputs(q_in=to_bf16_bits(q), k_in=to_bf16_bits(k),
                      rope_cos=np.cos(ang).astype(np.float32), rope_sin=np.sin(ang).astype(np.float32),
                      ln_gamma=(1.0 + 0.1 * rng.standard_normal(128)).astype(np.float32),
                      ln_beta=(0.1 * rng.standard_normal(128)).astype(np.float32),
                      ln_eps=1e-6, rope_dim=rope_dim)
