"""Shared helpers of the GPU parity tests (imported by tests/test_gpu_*.py only)."""
import numpy as np
import torch

import oracle
from dsa_sparse_attention_02_gb300 import _lib

DEV = "cuda:0"


def geometry_for_rows(lengths, device=DEV):
    """One request per row with one query at position len-1, so row t has len[t] valid keys."""
    lengths = np.asarray(lengths, dtype=np.int32)
    B = len(lengths)
    max_len = int(lengths.max())
    pages = (max_len + 63) // 64
    seq = torch.tensor(lengths, dtype=torch.int32, device=device)
    cu = torch.arange(B + 1, dtype=torch.int32, device=device)
    bt = torch.zeros(B, pages, dtype=torch.int32, device=device)
    keep = (seq, cu, bt)
    g = _lib.Geometry(seq, cu, bt, num_pages=max(pages, 1), max_seq_len=max_len, T=B)
    g._keep = keep
    return g


def index_set_parity(gpu_row, ref_scores, k, rel=1e-3):
    """Equal set sizes; every element of the symmetric difference scores within
    rel*|tau| (floor 1e-6 * max|I|) of the oracle's k-th score tau."""
    got = set(int(x) for x in gpu_row if x >= 0)
    ref_idx = oracle.topk_row(ref_scores, k)
    exp = set(int(x) for x in ref_idx if x >= 0)
    if len(got) != len(exp):
        return False, f"sizes {len(got)} vs {len(exp)}"
    diff = got ^ exp
    if not diff:
        return True, "exact"
    srt = np.sort(ref_scores)[::-1]
    tau = srt[min(k, len(srt)) - 1]
    tol = max(rel * abs(tau), 1e-6 * np.abs(ref_scores).max())
    worst = max(abs(ref_scores[s] - tau) for s in diff)
    return worst <= tol, f"{len(diff)} swapped, worst |I - tau| = {worst:.3g} (tol {tol:.3g})"


def assert_close(got, ref, atol, rtol, what):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    both_inf = np.isinf(got) & np.isinf(ref) & (np.sign(got) == np.sign(ref))
    with np.errstate(invalid="ignore"):
        err = np.where(both_inf, 0.0, np.abs(got - ref))
    bound = atol + rtol * np.where(np.isinf(ref), 0.0, np.abs(ref))
    bad = ~(err <= bound)
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {bad.size} outside tolerance; "
                           f"max err {np.nanmax(err):.3g}")
    return float(np.nanmax(err)) if err.size else 0.0


TOL = {"bf16": 2e-2, "e4m3": 5e-2, "int8": 5e-2}


def verify_step(wl, dw, ts, idx=None):
    """The step's selection (dw.idx, or `idx`) against the oracle's index sets, and every
    layer's output and LSE against the oracle's attention over that same selection."""
    idx = dw.idx.cpu().numpy() if idx is None else idx
    ref_scores = oracle.indexer_scores(wl.q_idx, wl.q_scale, wl.w, wl.idx_k, wl.idx_k_scale,
                                       wl.qk_dtype, wl.seq_lens, wl.n_q, wl.block_table, ts)
    for t in ts:
        ok, msg = index_set_parity(idx[t], ref_scores[t], wl.topk)
        assert ok, (t, msg)
    sel = {t: idx[t] for t in ts}
    for li, (lay, dl) in enumerate(zip(wl.layers, dw.layers)):
        ref = oracle.sparse_mla(lay.q, lay.kv, lay.kv_dtype, sel, wl.seq_lens, wl.n_q,
                                wl.block_table, wl.sm_scale, ts)
        out = dl.out.float().cpu().numpy()
        lse = dl.lse.cpu().numpy()
        tol = TOL[lay.kv_dtype]
        for t in ts:
            assert_close(out[t], ref[t][0], tol, tol, f"layer {li} out t={t}")
            assert_close(lse[t], ref[t][1], tol, tol, f"layer {li} lse t={t}")
    return ref_scores


def gpu_scores(wl, dw, fill=None):
    """The indexer's fp32 scores of every query through the standalone entry point."""
    stride = int(-(-wl.max_seq_len // 64) * 64)
    scores = torch.empty((wl.T, stride), dtype=torch.float32, device=DEV)
    if fill is not None:
        scores.fill_(fill)
    ws = _lib.workspace(_lib.dsa_indexer_scores_workspace_size(dw.geom), DEV)
    _lib.dsa_indexer_scores(dw.geom, dw.qk_dtype, dw.q_idx, dw.q_scale, dw.w, dw.idx_k, dw.idx_k_scale,
                            scores, ws)
    assert _lib.dsa_get_error(ws) == 0
    return scores
