"""dsa_indexer_scores on the GPU against the float64 oracle, then index-set parity of
indexer + top-k, and bit-exact top-k on the GPU's own scores."""
import numpy as np
import pytest
import torch

import oracle
from dsa_sparse_attention_02_gb300 import _lib, inputs, runner
from gpu_helpers import DEV, index_set_parity

pytestmark = pytest.mark.gpu

SENTINEL = np.float32(12345.0)

CASES = [
    ("tiny", dict()),
    ("decode", dict(batch=4)),
    ("mtp", dict(batch=3, ctx_scale=0.25)),
    ("prefill", dict(ctx_scale=1 / 8)),            # 2048 cached tokens, 2048 causal queries
    ("longctx", dict(batch=1, ctx_scale=1 / 16)),  # 8192 tokens with exact ties
]


def _scores(wl, dw):
    stride = int(-(-wl.max_seq_len // 64) * 64)
    scores = torch.full((wl.T, stride), float(SENTINEL), dtype=torch.float32, device=DEV)
    ws = _lib.workspace(_lib.dsa_indexer_scores_workspace_size(dw.geom), DEV)
    _lib.dsa_indexer_scores(dw.geom, dw.qk_dtype, dw.q_idx, dw.q_scale, dw.w, dw.idx_k, dw.idx_k_scale,
                            scores, ws)
    assert _lib.dsa_get_error(ws) == 0
    return scores


@pytest.mark.parametrize("name,kw", CASES, ids=[c[0] for c in CASES])
def test_indexer_scores_match_oracle(name, kw):
    wl = inputs.make_config(name, **kw)
    dw = runner.DeviceWorkload(wl, DEV)
    sc = _scores(wl, dw).cpu().numpy()
    _, pos = oracle.query_positions(wl.seq_lens, wl.n_q)
    req, _ = oracle.query_positions(wl.seq_lens, wl.n_q)
    ts = list(range(wl.T)) if wl.T <= 64 else list(np.linspace(0, wl.T - 1, 24).astype(int))
    ref = oracle.indexer_scores(wl.q_idx, wl.q_scale, wl.w, wl.idx_k, wl.idx_k_scale, wl.qk_dtype,
                                wl.seq_lens, wl.n_q, wl.block_table, ts)
    worst = 0.0
    for t in ts:
        p, L = int(pos[t]), int(wl.seq_lens[req[t]])
        r = ref[t]
        got = sc[t, : p + 1].astype(np.float64)
        scale = np.abs(r).max()
        err = np.abs(got - r).max() / scale
        worst = max(worst, err)
        assert err <= 1e-4, (t, err)
        assert np.all(np.isneginf(sc[t, p + 1: L])), t            # causally masked
        assert np.all(sc[t, L:] == SENTINEL), t                     # never written past the context
    print(f"{name}: max |I_gpu - I_ref| / max|I| = {worst:.3g}")


@pytest.mark.parametrize("name,kw", CASES, ids=[c[0] for c in CASES])
def test_topk_of_gpu_scores_exact_and_index_sets_match_oracle(name, kw):
    wl = inputs.make_config(name, **kw)
    dw = runner.DeviceWorkload(wl, DEV)
    scores = _scores(wl, dw)
    k = wl.topk
    idx = torch.empty(wl.T, k, dtype=torch.int32, device=DEV)
    ws = _lib.workspace(_lib.dsa_topk_workspace_size(dw.geom, k), DEV)
    _lib.dsa_topk(dw.geom, scores, k, idx, ws)
    assert _lib.dsa_get_error(ws) == 0
    got = idx.cpu().numpy()
    sc = scores.cpu().numpy()
    _, pos = oracle.query_positions(wl.seq_lens, wl.n_q)
    ts = list(range(wl.T)) if wl.T <= 64 else list(np.linspace(0, wl.T - 1, 24).astype(int))
    ref = oracle.indexer_scores(wl.q_idx, wl.q_scale, wl.w, wl.idx_k, wl.idx_k_scale, wl.qk_dtype,
                                wl.seq_lens, wl.n_q, wl.block_table, ts)
    for t in ts:
        p = int(pos[t])
        # bit-exact top-k over the same fp32 scores
        assert np.array_equal(got[t], oracle.topk_row(sc[t, : p + 1].astype(np.float64), k)), t
        ok, msg = index_set_parity(got[t], ref[t], k)
        assert ok, (t, msg)


@pytest.mark.parametrize("hi", [1, 3, 5, 16, 63, 64])
@pytest.mark.parametrize("qk", ["e4m3", "bf16"])
def test_indexer_any_head_count(hi, qk):
    """Head counts that are not a multiple of 4 (w and q_scale rows off 16-byte copies)
    and below the MMA's 16: padded with zero weights in the kernel. Hi = 16 and 64 fill
    the padded head count, so a multi-query group arrives as one copy per operand
    (requests of 1, 3 and 2 queries: groups shorter than 4, and a last group whose box
    runs past the final query row)."""
    wl = inputs.make_workload(f"hi{hi}", [700, 3000, 129], [1, 3, 2], topk=256, hi=hi, qk_dtype=qk, seed=20 + hi)
    dw = runner.DeviceWorkload(wl, DEV)
    sc = _scores(wl, dw).cpu().numpy()
    req, pos = oracle.query_positions(wl.seq_lens, wl.n_q)
    ref = oracle.indexer_scores(wl.q_idx, wl.q_scale, wl.w, wl.idx_k, wl.idx_k_scale, wl.qk_dtype,
                                wl.seq_lens, wl.n_q, wl.block_table)
    for t in range(wl.T):
        p, L = int(pos[t]), int(wl.seq_lens[req[t]])
        r = ref[t]
        err = np.abs(sc[t, : p + 1].astype(np.float64) - r).max() / max(np.abs(r).max(), 1e-30)
        assert err <= 1e-4, (hi, qk, t, err)
        assert np.all(np.isneginf(sc[t, p + 1: L]))


def test_indexer_more_requests_than_one_launch_holds():
    """1100 requests (the kernel holds 1024 per launch): scored in two launches."""
    rng = np.random.default_rng(4)
    lens = rng.integers(70, 400, size=1100)
    wl = inputs.make_workload("many", lens, [1] * 1100, topk=64, hi=16, qk_dtype="e4m3", seed=5)
    dw = runner.DeviceWorkload(wl, DEV)
    sc = _scores(wl, dw).cpu().numpy()
    _, pos = oracle.query_positions(wl.seq_lens, wl.n_q)
    ts = [0, 1, 511, 1023, 1024, 1025, 1099]
    ref = oracle.indexer_scores(wl.q_idx, wl.q_scale, wl.w, wl.idx_k, wl.idx_k_scale, wl.qk_dtype,
                                wl.seq_lens, wl.n_q, wl.block_table, ts)
    for t in ts:
        p = int(pos[t])
        err = np.abs(sc[t, : p + 1].astype(np.float64) - ref[t]).max() / np.abs(ref[t]).max()
        assert err <= 1e-4, (t, err)
