"""Contexts of 262144 tokens (bounded KPool scoring, lmdeploy "glm5.3-flash support",
Capacity improvement: 128K/256K requests complete with identical selections).

One request of 262144 cached tokens with two causal query tokens, 64 e4m3 indexer
heads, index_topk 2048, 1% of the index-key rows duplicated so that scores tie
exactly. dsa_decode_step (rows of 16 chunks merged over two levels) and
dsa_decode_step_bounded (a budget of one score row; spans of one and of three top-k
chunks, so that no query's whole row of scores ever exists) are each checked against
the oracle: index-set parity with the oracle's float64 scores, the selection bit for bit
equal to the oracle's top-k of the GPU's own fp32 scores, attention within 2e-2 over
the GPU's selection; and the bounded runs equal the unbounded one bit for bit."""
import numpy as np
import pytest
import torch

import oracle
from dsa_sparse_attention_02_gb300 import _lib, inputs, runner
from gpu_helpers import DEV, gpu_scores, verify_step

pytestmark = pytest.mark.gpu

L_CTX = 262144


@pytest.fixture(scope="module")
def long_step():
    wl = inputs.make_workload("long256k", [L_CTX], [2], topk=2048, hi=64, qk_dtype="e4m3",
                              kv_dtypes=("bf16",), seed=11, dup_key_frac=0.01)
    dw = runner.DeviceWorkload(wl, DEV)
    dw.step()
    torch.cuda.synchronize()
    assert dw.check_error() == 0
    ref = [dw.idx.clone(), dw.layers[0].out.clone(), dw.layers[0].lse.clone()]
    sc = gpu_scores(wl, dw).cpu().numpy()
    return wl, dw, ref, sc


def _check(wl, dw, sc):
    _, pos = oracle.query_positions(wl.seq_lens, wl.n_q)
    idx = dw.idx.cpu().numpy()
    for t in range(wl.T):
        p = int(pos[t])
        assert np.array_equal(idx[t], oracle.topk_row(sc[t, : p + 1].astype(np.float64), wl.topk)), t
    verify_step(wl, dw, list(range(wl.T)))


def test_decode_step_262144_tokens_matches_oracle(long_step):
    wl, dw, ref, sc = long_step
    _check(wl, dw, sc)


@pytest.mark.parametrize("budget", [L_CTX * 4, 65536, 3 * 65536 + 100],
                         ids=["one-row", "span-16384", "span-49152"])
def test_bounded_step_262144_tokens_matches_oracle(long_step, budget):
    wl, dw, ref, sc = long_step
    a = dw.args[0]
    ws = _lib.workspace(_lib.dsa_decode_step_bounded_workspace_size(a, budget), DEV)
    if budget < L_CTX * 4:
        # the scores of one span at a time: far less than one query's whole row
        assert ws.numel() < _lib.dsa_decode_step_bounded_workspace_size(a, L_CTX * 4)
    dw.idx.fill_(-7)
    dw.layers[0].out.fill_(float("nan"))
    dw.layers[0].lse.fill_(float("nan"))
    _lib.dsa_decode_step_bounded(a, budget, ws)
    assert _lib.dsa_get_error(ws) == 0
    assert torch.equal(dw.idx, ref[0])
    assert torch.equal(dw.layers[0].out.view(torch.int16), ref[1].view(torch.int16))
    assert torch.equal(dw.layers[0].lse.view(torch.int32), ref[2].view(torch.int32))
    _check(wl, dw, sc)
