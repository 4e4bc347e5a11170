"""Failure detection on the GPU without a fault: a bounded wait that nothing completes
runs out, the kernel records DSA_ERR_TIMEOUT in the workspace's error word and exits,
the host reads the status, and the context stays usable for the next step."""
import time

import pytest
import torch

from dsa_sparse_attention_02_gb300 import _lib, inputs, runner
from gpu_helpers import DEV

pytestmark = pytest.mark.gpu


def test_bounded_wait_runs_out_and_reports_timeout():
    ws = _lib.workspace(256, DEV)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    _lib.dsa_wait_probe(ws, 2000)                          # 2 ms limit
    assert _lib.dsa_get_error(ws) == _lib.DSA_ERR_TIMEOUT   # synchronizes; reads and clears
    elapsed = time.perf_counter() - t0
    assert 0.002 <= elapsed < 5.0
    assert _lib.dsa_get_error(ws) == _lib.DSA_OK           # the read cleared the word
    # the context is still usable: a full step runs clean afterwards
    wl = inputs.make_config("tiny")
    dw = runner.DeviceWorkload(wl, DEV)
    dw.step()
    torch.cuda.synchronize()
    assert dw.check_error() == 0
    assert torch.isfinite(dw.layers[0].out.float()).all()
