"""dsa_decode_step_bounded (bounded scoring: the indexer's scores of at most a budget's
worth of queries exist at a time, each range reduced to its selection before the next)
against the oracle and against dsa_decode_step on the same inputs: index sets and
attention match the oracle, and the selection, the output and the LSE are bitwise
those of the unbounded step for every budget, from one query's score row up to all but
one; the bounded step is graph-capturable; a budget below one row is rejected before
launch. Contexts of 262144 tokens, with budgets below one row, are in
test_gpu_long_context.py."""
import numpy as np
import pytest
import torch

from dsa_sparse_attention_02_gb300 import _lib, inputs, runner
from gpu_helpers import DEV, verify_step

pytestmark = pytest.mark.gpu

CASES = [
    ("mtp", dict(batch=3, ctx_scale=0.25)),        # 4 causal queries per request
    ("prefill", dict(ctx_scale=1 / 8)),            # 2048 queries of one request
    ("longctx", dict(batch=2, ctx_scale=1 / 16)),  # 8192-token rows with exact ties
    ("decode", dict(batch=8)),
]


def _snapshot(dw):
    return [dw.idx.clone()] + [t.clone() for L in dw.layers for t in (L.out.view(torch.int16), L.lse.view(torch.int32))]


def _bounded_step(dw, rows, ws=None, stream=None):
    row_bytes = (-(-dw.wl.max_seq_len // 64) * 64) * 4
    budget = rows * row_bytes + row_bytes // 2          # not a multiple of the row: rounds down
    a0 = dw.args[0]
    if ws is None:
        ws = _lib.workspace(max([_lib.dsa_decode_step_bounded_workspace_size(a0, budget)] +
                                [_lib.dsa_decode_step_workspace_size(a) for a in dw.args[1:]]), DEV)
    _lib.dsa_decode_step_bounded(a0, budget, ws, stream)
    for a in dw.args[1:]:
        _lib.dsa_decode_step_bounded(a, budget, ws, stream)
    return ws


@pytest.mark.parametrize("name,kw", CASES, ids=[c[0] for c in CASES])
def test_bounded_step_equals_unbounded_bitwise(name, kw):
    wl = inputs.make_config(name, **kw)
    dw = runner.DeviceWorkload(wl, DEV)
    dw.step()
    assert dw.check_error() == 0
    ref = _snapshot(dw)
    T = wl.T
    for rows in sorted({1, 3, 100, max(1, T - 1)}):
        for L in dw.layers:
            L.out.fill_(float("nan"))
            L.lse.fill_(float("nan"))
        dw.idx.fill_(-7)
        ws = _bounded_step(dw, rows)
        assert _lib.dsa_get_error(ws) == 0
        got = _snapshot(dw)
        for r, g in zip(ref, got):
            assert torch.equal(r, g), (name, rows)
        if rows == 3:
            # and against the oracle directly (index sets, attention over the selection)
            ts = list(range(T)) if T <= 32 else list(np.linspace(0, T - 1, 12).astype(int))
            verify_step(wl, dw, ts)
    # the bounded workspace is smaller than the unbounded one once it holds fewer rows
    a0 = dw.args[0]
    row_bytes = (-(-wl.max_seq_len // 64) * 64) * 4
    if T > 4:
        assert _lib.dsa_decode_step_bounded_workspace_size(a0, row_bytes) < _lib.dsa_decode_step_workspace_size(a0)


def test_bounded_step_graph_capture_and_budget_floor():
    wl = inputs.make_config("mtp", batch=3, ctx_scale=0.25)
    dw = runner.DeviceWorkload(wl, DEV)
    dw.step()
    ref = _snapshot(dw)
    ws = _bounded_step(dw, 5)                                       # warm-up, sizes the workspace
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        _bounded_step(dw, 5, ws=ws, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    with torch.cuda.graph(g):
        _bounded_step(dw, 5, ws=ws)
    for L in dw.layers:
        L.out.fill_(0)
    dw.idx.fill_(0)
    g.replay()
    torch.cuda.synchronize()
    assert _lib.dsa_get_error(ws) == 0
    for r, got in zip(ref, _snapshot(dw)):
        assert torch.equal(r, got)
    row_bytes = (-(-wl.max_seq_len // 64) * 64) * 4
    with pytest.raises(_lib.DsaError) as e:
        _lib.dsa_decode_step_bounded(dw.args[0], row_bytes - 4, ws)
    assert e.value.status == _lib.DSA_ERR_INVALID_ARG
