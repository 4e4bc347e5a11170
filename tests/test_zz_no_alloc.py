"""dsa_sparse_mla_attend_static: the attention entry point for callers that cannot
allocate device memory at call time (a runtime with memory planned up front, a
plugin host without workspace, code where an allocation would synchronize the
device). It uses the library's static per-GPU scratch buffer instead of a
workspace. This file sorts last so that a run stopping at its first failure has
already run every other test; it must also pass alone in a fresh process."""
import numpy as np
import pytest
import torch

import oracle
from dsa_sparse_attention_02_gb300 import _lib, inputs, runner
from gpu_helpers import DEV, assert_close

pytestmark = pytest.mark.gpu

TOL = 2e-2      # the bf16-KV attention tolerance of the other GPU tests


def _selection(wl, k, seed):
    rng = np.random.default_rng(seed)
    idx = np.full((wl.T, k), -1, dtype=np.int32)
    for t in range(wl.T):
        L = int(wl.seq_lens[t])
        n = min(k, L)
        idx[t, :n] = np.sort(rng.choice(L, size=n, replace=False))
    return torch.from_numpy(idx).to(DEV)


def _static(dw, idx, k, err):
    L = dw.layers[0]
    out = torch.full_like(L.out, float("nan"))
    lse = torch.full_like(L.lse, float("nan"))
    _lib.dsa_sparse_mla_attend_static(dw.geom, L.kv_dtype, L.q, L.kv, idx, k, dw.wl.sm_scale, out, lse, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return out, lse


def test_static_scratch_matches_workspace_entry_point_and_oracle_twice():
    wl = inputs.make_config("decode", batch=12)
    dw = runner.DeviceWorkload(wl, DEV)
    L = dw.layers[0]
    idx = _selection(wl, wl.topk, 1)
    ref_out, ref_lse = torch.empty_like(L.out), torch.empty_like(L.lse)
    ws = _lib.workspace(_lib.dsa_sparse_mla_attend_workspace_size(dw.geom, 16, wl.topk), DEV)
    _lib.dsa_sparse_mla_attend(dw.geom, L.kv_dtype, L.q, L.kv, idx, wl.topk, wl.sm_scale, ref_out, ref_lse, ws)
    torch.cuda.synchronize()
    assert _lib.dsa_get_error(ws) == 0
    sel = idx.cpu().numpy()
    oref = oracle.sparse_mla(wl.layers[0].q, wl.layers[0].kv, "bf16", {t: sel[t] for t in range(wl.T)},
                             wl.seq_lens, wl.n_q, wl.block_table, wl.sm_scale)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    # A call with another selection, index_topk and batch first leaves different partial
    # rows in the shared buffer: nothing of it may leak into the calls checked below.
    other = inputs.make_config("decode", batch=7, seed=77)
    dwo = runner.DeviceWorkload(other, DEV)
    _static(dwo, _selection(other, 1536, 9), 1536, err)
    for _ in range(2):                     # the buffer keeps the previous call's contents
        out, lse = _static(dw, idx, wl.topk, err)
        o, r = out.float().cpu().numpy(), ref_out.float().cpu().numpy()
        assert np.all(np.abs(o - r) <= TOL + TOL * np.abs(r))
        l, rl = lse.cpu().numpy(), ref_lse.cpu().numpy()
        assert np.all(np.abs(l - rl) <= TOL + TOL * np.abs(rl))
        for t in range(wl.T):
            assert_close(o[t], oref[t][0], TOL, TOL, f"static out t={t}")
            assert_close(l[t], oref[t][1], TOL, TOL, f"static lse t={t}")


def test_static_scratch_rejects_calls_beyond_its_size():
    wl = inputs.make_workload("big", [4096], [4000], topk=2048, hi=4, qk_dtype="bf16", seed=3)
    dw = runner.DeviceWorkload(wl, DEV)
    L = dw.layers[0]
    idx = torch.full((wl.T, wl.topk), -1, dtype=torch.int32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    with pytest.raises(_lib.DsaError) as e:
        _lib.dsa_sparse_mla_attend_static(dw.geom, L.kv_dtype, L.q, L.kv, idx, wl.topk, wl.sm_scale,
                                          L.out, L.lse, err)
    assert e.value.status == _lib.DSA_ERR_WORKSPACE
    assert "static scratch" in str(e.value)


def test_attend_entry_points_write_page_locked_host_outputs():
    """Both attention entry points with O and LSE in page-locked host memory give the
    device-output results bit for bit."""
    wl = inputs.make_config("decode", batch=6)
    dw = runner.DeviceWorkload(wl, DEV)
    L = dw.layers[0]
    idx = _selection(wl, wl.topk, 5)
    dev_out, dev_lse = torch.empty_like(L.out), torch.empty_like(L.lse)
    ws = _lib.workspace(_lib.dsa_sparse_mla_attend_workspace_size(dw.geom, 16, wl.topk), DEV)
    _lib.dsa_sparse_mla_attend(dw.geom, L.kv_dtype, L.q, L.kv, idx, wl.topk, wl.sm_scale, dev_out, dev_lse, ws)
    torch.cuda.synchronize()
    assert _lib.dsa_get_error(ws) == 0
    host_out = torch.full(L.out.shape, float("nan"), dtype=L.out.dtype).pin_memory()
    host_lse = torch.full(L.lse.shape, float("nan"), dtype=L.lse.dtype).pin_memory()
    _lib.dsa_sparse_mla_attend(dw.geom, L.kv_dtype, L.q, L.kv, idx, wl.topk, wl.sm_scale, host_out, host_lse, ws)
    torch.cuda.synchronize()
    assert _lib.dsa_get_error(ws) == 0
    assert torch.equal(host_out, dev_out.cpu()) and torch.equal(host_lse, dev_lse.cpu())
    host_out.fill_(float("nan")); host_lse.fill_(float("nan"))
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    _lib.dsa_sparse_mla_attend_static(dw.geom, L.kv_dtype, L.q, L.kv, idx, wl.topk, wl.sm_scale, host_out,
                                      host_lse, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(host_out, dev_out.cpu()) and torch.equal(host_lse, dev_lse.cpu())
