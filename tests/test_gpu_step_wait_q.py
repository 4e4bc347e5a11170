"""dsa_decode_step_wait_q: the MLA query's copy runs on another stream while the indexer
and top-k run; the attention waits for it. Selection, output and LSE are bitwise those of
dsa_decode_step, eagerly and in a captured graph, also for an IndexShare layer after it."""
import pytest
import torch

from dsa_sparse_attention_02_gb300 import _lib, inputs, runner
from gpu_helpers import DEV

pytestmark = pytest.mark.gpu


def _snapshot(dw):
    return [dw.idx.clone()] + [t.clone() for L in dw.layers for t in (L.out.view(torch.int16), L.lse.view(torch.int32))]


@pytest.mark.parametrize("name,kw", [("decode", dict(batch=8)), ("mtp", dict(batch=3, ctx_scale=0.25))])
def test_wait_q_equals_plain_step(name, kw):
    wl = inputs.make_config(name, **kw)
    dw = runner.DeviceWorkload(wl, DEV)
    dw.step()
    ref = _snapshot(dw)
    off = dw.inputs_mla_q_offset
    host_q = dw.inputs[off:].cpu().pin_memory()
    side = torch.cuda.Stream()
    fork, q_ready = torch.cuda.Event(), torch.cuda.Event()

    def enqueue():
        dw.inputs[off:].zero_()                      # the query is really re-delivered by the side copy
        fork.record(torch.cuda.current_stream())
        side.wait_event(fork)
        with torch.cuda.stream(side):
            torch.cuda._sleep(2_000_000)             # the copy lands well after the indexer has started
            _lib.dsa_stage_copy(dw.inputs[off:], host_q, host_q.numel())
            q_ready.record(side)
        for i, a in enumerate(dw.args):
            if i == 0:
                _lib.dsa_decode_step_wait_q(a, q_ready, dw.ws)
            else:
                _lib.dsa_decode_step(a, dw.ws)

    for L in dw.layers:
        L.out.zero_()
    enqueue()
    torch.cuda.synchronize()
    assert dw.check_error() == 0
    for r, g in zip(ref, _snapshot(dw)):
        assert torch.equal(r, g)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        enqueue()
    for L in dw.layers:
        L.out.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert dw.check_error() == 0
    for r, g in zip(ref, _snapshot(dw)):
        assert torch.equal(r, g)
