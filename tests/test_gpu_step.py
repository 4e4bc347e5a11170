"""dsa_decode_step end to end on the GPU: index sets and attention against the oracle
on every configuration (reduced and full size, sampled queries at full size),
IndexShare reuse, determinism and CUDA-graph capture."""
import numpy as np
import pytest
import torch

import oracle
from dsa_sparse_attention_02_gb300 import _lib, inputs, runner
from gpu_helpers import DEV, verify_step

pytestmark = pytest.mark.gpu

_verify = verify_step


SMALL = [
    ("tiny", dict()),
    ("decode", dict(batch=6)),
    ("decode", dict(batch=6, latent="int8")),      # the int8 latent cache (next row f4)
    ("mtp", dict(batch=3, ctx_scale=0.25)),
    ("prefill", dict(ctx_scale=1 / 8)),
    ("longctx", dict(batch=2, ctx_scale=1 / 16)),
]


@pytest.mark.parametrize("name,kw", SMALL, ids=[c[0] + ("-" + c[1]["latent"] if "latent" in c[1] else "") for c in SMALL])
def test_step_small_configs(name, kw):
    wl = inputs.make_config(name, **kw)
    dw = runner.DeviceWorkload(wl, DEV)
    dw.step()
    torch.cuda.synchronize()
    assert dw.check_error() == 0
    ts = list(range(wl.T)) if wl.T <= 64 else list(np.linspace(0, wl.T - 1, 16).astype(int))
    _verify(wl, dw, ts)


FULL = [
    ("decode", 64),   # the bench configuration: every query checked
    ("decode-int8", 16),
    ("mtp", 10),
    ("prefill", 8),
    ("longctx", 4),
]


@pytest.mark.parametrize("name,nsample", FULL, ids=[c[0] for c in FULL])
def test_step_full_size_sampled(name, nsample):
    wl = inputs.make_config("decode", latent="int8") if name == "decode-int8" else inputs.make_config(name)
    dw = runner.DeviceWorkload(wl, DEV)
    dw.step()
    torch.cuda.synchronize()
    assert dw.check_error() == 0
    ts = list(np.unique(np.linspace(0, wl.T - 1, nsample).astype(int)))
    _verify(wl, dw, ts)


SELECTION = [
    ("tiny", dict()),
    ("decode", dict()),                            # the bench configuration, 64 queries
    ("decode", dict(batch=5, ctx_scale=0.25)),     # rows no longer than index_topk
    ("longctx", dict(batch=2, ctx_scale=1 / 16)),  # 8192-entry rows with exact score ties
]


@pytest.mark.parametrize("name,kw", SELECTION, ids=["tiny", "decode", "decode-short", "longctx-ties"])
def test_step_selection_bit_exact_on_gpu_scores(name, kw):
    """The step's selection equals the oracle's top-k of the GPU's own fp32 scores bit
    for bit (the indexer is deterministic, so a standalone indexer call reproduces the
    scores the step ranked)."""
    wl = inputs.make_config(name, **kw)
    dw = runner.DeviceWorkload(wl, DEV)
    dw.step()
    torch.cuda.synchronize()
    assert dw.check_error() == 0
    stride = int(-(-wl.max_seq_len // 64) * 64)
    scores = torch.empty((wl.T, stride), dtype=torch.float32, device=DEV)
    ws = _lib.workspace(_lib.dsa_indexer_scores_workspace_size(dw.geom), DEV)
    _lib.dsa_indexer_scores(dw.geom, dw.qk_dtype, dw.q_idx, dw.q_scale, dw.w, dw.idx_k, dw.idx_k_scale,
                            scores, ws)
    assert _lib.dsa_get_error(ws) == 0
    sc = scores.cpu().numpy()
    idx = dw.idx.cpu().numpy()
    _, pos = oracle.query_positions(wl.seq_lens, wl.n_q)
    for t in range(wl.T):
        p = int(pos[t])
        assert np.array_equal(idx[t], oracle.topk_row(sc[t, : p + 1].astype(np.float64), wl.topk)), t


def test_indexshare_layer_reuses_full_layer_selection():
    wl = inputs.make_config("mtp", batch=2, ctx_scale=0.3)
    dw = runner.DeviceWorkload(wl, DEV)
    dw.step()
    torch.cuda.synchronize()
    idx = dw.idx.clone()
    out1 = dw.layers[1].out.clone()
    # layer 1 alone through the standalone entry point over layer 0's selection
    L = dw.layers[1]
    out = torch.empty_like(L.out)
    ws = _lib.workspace(_lib.dsa_sparse_mla_attend_workspace_size(dw.geom, 16, wl.topk), DEV)
    _lib.dsa_sparse_mla_attend(dw.geom, L.kv_dtype, L.q, L.kv, idx, wl.topk, wl.sm_scale, out, None, ws)
    torch.cuda.synchronize()
    assert torch.equal(out, out1)
    # a shared-layer step leaves the selection untouched and reproduces layer 1
    a = _lib.make_step_args(dw.geom, wl.topk, reuse_idx=idx, kv_dtype=L.kv_dtype, q=L.q, kv_cache=L.kv,
                            sm_scale=wl.sm_scale, out=out, lse=None)
    ws2 = _lib.workspace(_lib.dsa_decode_step_workspace_size(a), DEV)
    _lib.dsa_decode_step(a, ws2)
    torch.cuda.synchronize()
    assert torch.equal(out, out1) and torch.equal(idx, dw.idx)


def test_step_is_deterministic_and_graph_capturable():
    wl = inputs.make_config("decode", batch=8)
    dw = runner.DeviceWorkload(wl, DEV)
    dw.step()
    torch.cuda.synchronize()
    idx0, out0, lse0 = dw.idx.clone(), dw.layers[0].out.clone(), dw.layers[0].lse.clone()
    dw.step()
    torch.cuda.synchronize()
    assert torch.equal(idx0, dw.idx) and torch.equal(out0, dw.layers[0].out)
    assert torch.equal(lse0, dw.layers[0].lse)
    graph = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        dw.step()
    torch.cuda.current_stream().wait_stream(s)
    dw.layers[0].out.zero_()
    dw.idx.zero_()
    with torch.cuda.graph(graph):
        dw.step()
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(idx0, dw.idx) and torch.equal(out0, dw.layers[0].out)
    assert dw.check_error() == 0


def test_causality_on_gpu():
    # rewriting every key and latent row after the first query's position changes nothing for it
    wl = inputs.make_config("mtp", batch=1, ctx_scale=0.3)
    dw = runner.DeviceWorkload(wl, DEV)
    dw.step()
    torch.cuda.synchronize()
    idx0 = dw.idx[0].clone()
    out0 = dw.layers[0].out[0].clone()
    _, pos = oracle.query_positions(wl.seq_lens, wl.n_q)
    p0 = int(pos[0])
    rows = oracle.physical_rows(wl.block_table[0], np.arange(p0 + 1, int(wl.seq_lens[0])))
    wl2 = inputs.Workload(**{**wl.__dict__})
    wl2.idx_k = wl.idx_k.copy()
    wl2.idx_k.reshape(-1, 128)[rows] = np.uint8(0x48)
    kv = wl.layers[0].kv.copy()
    pages = kv.reshape(-1, 64 * 656)                 # e4m3 record pages: codes | scales | RoPE planes
    for r in rows:
        pg, sl = divmod(int(r), 64)
        pages[pg, 512 * sl:512 * (sl + 1)] = np.uint8(0x48)
        pages[pg, 32768 + 16 * sl:32768 + 16 * (sl + 1)] = np.uint8(0x48)
        pages[pg, 33792 + 128 * sl:33792 + 128 * (sl + 1)] = np.uint8(0x48)
    wl2.layers = [inputs.Layer(q=wl.layers[0].q, kv=kv, kv_dtype=wl.layers[0].kv_dtype), wl.layers[1]]
    dw2 = runner.DeviceWorkload(wl2, DEV)
    dw2.step()
    torch.cuda.synchronize()
    assert torch.equal(idx0, dw2.idx[0]) and torch.equal(out0, dw2.layers[0].out[0])


# ---- dsa_decode_step_hist: the indexer's first-digit histograms (the top 11 bits of
# each visible score's radix key, per query and 16384-position chunk), which the top-k
# reads instead of counting them. They sit at the end of the full layer's workspace and
# the top-k leaves them zero; whatever else they hold, the selection stays exact.

def _orderable(scores: np.ndarray) -> np.ndarray:
    u = scores.astype(np.float32).view(np.uint32).copy()
    u[u == 0x80000000] = 0
    return np.where(u & 0x80000000, ~u, u | 0x80000000).astype(np.uint32)


def _hist_view(dw, wl):
    """The histogram region of layer 0's step workspace as [T, chunks, 2048] int32."""
    nch = max(1, -(-wl.max_seq_len // 16384))
    nbytes = wl.T * nch * 2048 * 4
    end = _lib.dsa_decode_step_hist_workspace_size(dw.args[0])
    off = end - (-(-nbytes // 256) * 256)
    return dw.ws[off:off + nbytes].view(torch.int32).view(wl.T, nch, 2048), nch


def _gpu_scores(dw, wl):
    stride = int(-(-wl.max_seq_len // 64) * 64)
    scores = torch.empty((wl.T, stride), dtype=torch.float32, device=DEV)
    ws = _lib.workspace(_lib.dsa_indexer_scores_workspace_size(dw.geom), DEV)
    _lib.dsa_indexer_scores(dw.geom, dw.qk_dtype, dw.q_idx, dw.q_scale, dw.w, dw.idx_k, dw.idx_k_scale,
                            scores, ws)
    assert _lib.dsa_get_error(ws) == 0
    return scores.cpu().numpy()


HIST = [
    ("decode", dict(batch=8)),
    ("mtp", dict(batch=3, ctx_scale=0.25)),         # query groups of 4, two layers on one workspace
    ("longctx", dict(batch=2, ctx_scale=0.25)),    # rows of 32768: two chunks each
]


def _rejected(dw) -> int:
    return int(dw.ws[:8].view(torch.int32)[1])


CLEAN = HIST + [("tiny", dict())]   # bf16 index keys: no histograms, the default step's path


@pytest.mark.parametrize("name,kw", CLEAN, ids=[c[0] for c in CLEAN])
def test_step_histograms_accepted_on_clean_workspace(name, kw):
    """On a zeroed workspace every segment's selection made from the indexer's
    histogram passes the exact final-count check (none is redone), step after step
    (the top-k leaves the region zero), equals the oracle's top-k of the GPU's scores,
    and every output is bitwise that of dsa_decode_step."""
    wl = inputs.make_config(name, **kw)
    dw = runner.DeviceWorkload(wl, DEV, hist=True)
    hv, _ = _hist_view(dw, wl)
    for _ in range(3):
        dw.step()
        torch.cuda.synchronize()
        assert dw.check_error() == 0
        assert _rejected(dw) == 0
        assert int(hv.abs().sum()) == 0
    sc = _gpu_scores(dw, wl)
    _, pos = oracle.query_positions(wl.seq_lens, wl.n_q)
    idx = dw.idx.cpu().numpy()
    for t in range(wl.T):
        p = int(pos[t])
        assert np.array_equal(idx[t], oracle.topk_row(sc[t, : p + 1].astype(np.float64), wl.topk)), t
    ref = runner.DeviceWorkload(wl, DEV)
    ref.step()
    torch.cuda.synchronize()
    assert torch.equal(ref.idx, dw.idx)
    for L0, L1 in zip(ref.layers, dw.layers):
        assert torch.equal(L0.out, L1.out) and torch.equal(L0.lse, L1.lse)


@pytest.mark.parametrize("name,kw", HIST, ids=[c[0] for c in HIST])
@pytest.mark.parametrize("plant", ["exact", "random", "top-bin", "cancel"])
def test_step_first_digit_histograms(name, kw, plant):
    """A histogram region holding something else when the step starts (the true
    histogram, which the indexer then doubles; random words; the right totals in the
    top bin, above every score; the true histogram's negative, which the indexer's counts bring
    to zero) still gives the oracle's top-k of the GPU's scores bit for bit, the
    segments whose check fails are counted, and the region is left zero."""
    wl = inputs.make_config(name, **kw)
    dw = runner.DeviceWorkload(wl, DEV, hist=True)
    sc = _gpu_scores(dw, wl)
    _, pos = oracle.query_positions(wl.seq_lens, wl.n_q)
    hv, nch = _hist_view(dw, wl)
    true = np.zeros((wl.T, nch, 2048), dtype=np.int64)
    for t in range(wl.T):
        p = int(pos[t])
        keys = _orderable(sc[t, : p + 1])
        chunk = np.arange(p + 1) >> 14
        np.add.at(true[t], (chunk, keys >> 21), 1)
    rng = np.random.default_rng(7)
    if plant == "exact":
        planted = true
    elif plant == "random":
        planted = rng.integers(-2**31, 2**31, size=true.shape)
    elif plant == "top-bin":
        # above every real score's bin, so the first digit lands there and is wrong
        assert true[..., 2047].sum() == 0
        planted = np.zeros_like(true)
        planted[..., 2047] = true.sum(axis=2)
    else:  # cancel: the indexer's counts bring the region back to zero
        planted = -true
    hv.copy_(torch.from_numpy(planted.astype(np.int32)))
    dw.step()
    torch.cuda.synchronize()
    assert dw.check_error() == 0
    assert int(hv.abs().sum()) == 0
    # segments with more visible keys than index_topk are selected from a histogram
    selected = sum(int(min(16384, int(pos[t]) + 1 - 16384 * c) > wl.topk)
                   for t in range(wl.T) for c in range(nch) if int(pos[t]) + 1 > 16384 * c)
    if plant in ("top-bin", "cancel"):
        assert _rejected(dw) == selected
    else:
        assert 0 <= _rejected(dw) <= selected
    idx = dw.idx.cpu().numpy()
    for t in range(wl.T):
        p = int(pos[t])
        assert np.array_equal(idx[t], oracle.topk_row(sc[t, : p + 1].astype(np.float64), wl.topk)), t
    # with the region left zero, the next step's histograms are its own and accepted
    before, n_rej = dw.idx.clone(), _rejected(dw)
    dw.step()
    torch.cuda.synchronize()
    assert torch.equal(before, dw.idx) and _rejected(dw) == n_rej
