"""dsa_sparse_mla_attend on the GPU against the float64 oracle over the same index rows."""
import numpy as np
import pytest
import torch

import oracle
from dsa_sparse_attention_02_gb300 import _lib, inputs, runner
from gpu_helpers import DEV, assert_close

pytestmark = pytest.mark.gpu

TOL = {"bf16": 2e-2, "e4m3": 5e-2, "int8": 5e-2}   # int8 latent: the quantized-cache bound


def _random_idx(rng, wl, k, pad_frac=0.1, empty_rows=()):
    _, pos = oracle.query_positions(wl.seq_lens, wl.n_q)
    idx = np.full((wl.T, k), -1, dtype=np.int32)
    for t in range(wl.T):
        if t in empty_rows:
            continue
        n = min(k, int(pos[t]) + 1)
        sel = rng.choice(int(pos[t]) + 1, size=n, replace=False)
        if rng.random() < 0.5:
            sel = np.sort(sel)
        row = np.full(k, -1, dtype=np.int32)
        row[:n] = sel
        drop = rng.random(k) < pad_frac               # scattered -1 padding
        row[drop] = -1
        idx[t] = row
    return idx


def _attend(wl, dw, layer, idx_np, k):
    L = dw.layers[layer]
    idx = torch.from_numpy(idx_np).to(DEV)
    out = torch.full_like(L.out, float("nan"))
    lse = torch.full_like(L.lse, float("nan"))
    ws = _lib.workspace(_lib.dsa_sparse_mla_attend_workspace_size(dw.geom, L.q.shape[1], k), DEV)
    _lib.dsa_sparse_mla_attend(dw.geom, L.kv_dtype, L.q, L.kv, idx, k, wl.sm_scale, out, lse, ws)
    assert _lib.dsa_get_error(ws) == 0
    return out.float().cpu().numpy(), lse.cpu().numpy()


def _check(wl, layer, idx_np, out, lse, ts=None):
    lay = wl.layers[layer]
    ts = range(wl.T) if ts is None else ts
    ref = oracle.sparse_mla(lay.q, lay.kv, lay.kv_dtype, {t: idx_np[t] for t in ts}, wl.seq_lens,
                            wl.n_q, wl.block_table, wl.sm_scale, ts)
    tol = TOL[lay.kv_dtype]
    worst = 0.0
    for t in ts:
        o_ref, l_ref = ref[t]
        worst = max(worst, assert_close(out[t], o_ref, tol, tol, f"out t={t}"))
        assert_close(lse[t], l_ref, tol, tol, f"lse t={t}")
    return worst


@pytest.mark.parametrize("kv_dtype", ["bf16", "e4m3", "int8"])
@pytest.mark.parametrize("k", [64, 200, 2048])
def test_attend_random_selections(kv_dtype, k):
    rng = np.random.default_rng(k)
    wl = inputs.make_workload("attn", [300, 1000, 2500, 4100], [1, 2, 1, 3], topk=k, hi=4,
                              qk_dtype="bf16", kv_dtypes=(kv_dtype,), seed=31)
    dw = runner.DeviceWorkload(wl, DEV)
    idx = _random_idx(rng, wl, k, empty_rows=(1,))
    out, lse = _attend(wl, dw, 0, idx, k)
    worst = _check(wl, 0, idx, out, lse)
    assert np.all(out[1] == 0) and np.all(np.isneginf(lse[1]))      # all-padding row
    print(f"{kv_dtype} k={k}: max |O err| {worst:.3g}")


@pytest.mark.parametrize("heads", [8, 32])
def test_attend_head_counts(heads):
    rng = np.random.default_rng(heads)
    wl = inputs.make_workload("attn", [700, 3000], [2, 1], topk=512, hi=4, qk_dtype="bf16",
                              kv_dtypes=("bf16",), heads=heads, seed=32)
    dw = runner.DeviceWorkload(wl, DEV)
    idx = _random_idx(rng, wl, 512)
    out, lse = _attend(wl, dw, 0, idx, 512)
    _check(wl, 0, idx, out, lse)


def test_attend_many_queries_split_over_ctas():
    # 300 queries x 16 chunks: most queries are split across CTAs and merged by the combine
    rng = np.random.default_rng(7)
    wl = inputs.make_workload("attn", [6000] * 3, [100] * 3, topk=2048, hi=4, qk_dtype="bf16",
                              kv_dtypes=("bf16",), seed=33)
    dw = runner.DeviceWorkload(wl, DEV)
    idx = _random_idx(rng, wl, 2048, pad_frac=0.02)
    out, lse = _attend(wl, dw, 0, idx, 2048)
    _check(wl, 0, idx, out, lse, ts=list(range(0, wl.T, 13)))


def test_attend_indices_outside_request_are_skipped_and_reported():
    rng = np.random.default_rng(8)
    wl = inputs.make_workload("attn", [500, 900], [1, 1], topk=128, hi=4, qk_dtype="bf16",
                              kv_dtypes=("bf16",), seed=34)
    dw = runner.DeviceWorkload(wl, DEV)
    idx = _random_idx(rng, wl, 128, pad_frac=0.0)
    bad = idx.copy()
    bad[0, 5] = 10_000                                  # beyond seq_lens[0]
    L = dw.layers[0]
    ws = _lib.workspace(_lib.dsa_sparse_mla_attend_workspace_size(dw.geom, 16, 128), DEV)
    _lib.dsa_sparse_mla_attend(dw.geom, L.kv_dtype, L.q, L.kv, torch.from_numpy(bad).to(DEV), 128,
                               wl.sm_scale, L.out, L.lse, ws)
    assert _lib.dsa_get_error(ws) == _lib.DSA_ERR_BAD_INDEX
    assert _lib.dsa_get_error(ws) == 0                  # reading clears it
    skipped = bad.copy()
    skipped[0, 5] = -1
    _check(wl, 0, skipped, L.out.float().cpu().numpy(), L.lse.cpu().numpy())


def test_attend_split_merge_is_deterministic_and_needs_no_initial_workspace():
    # 120 queries x 16 chunks over the persistent grid: nearly every query is split
    # over two clusters and merged by the combine in a fixed order, so repeated
    # calls are bit-identical; a workspace whose body holds another workspace's
    # partials, or random bytes, gives the same result (only the header must start
    # at zero).
    rng = np.random.default_rng(9)
    wl = inputs.make_workload("attn", [6000] * 3, [40] * 3, topk=2048, hi=4, qk_dtype="bf16",
                              kv_dtypes=("bf16",), seed=35)
    dw = runner.DeviceWorkload(wl, DEV)
    idx = torch.from_numpy(_random_idx(rng, wl, 2048, pad_frac=0.02)).to(DEV)
    L = dw.layers[0]
    size = _lib.dsa_sparse_mla_attend_workspace_size(dw.geom, 16, 2048)

    def run(ws):
        out = torch.full_like(L.out, float("nan"))
        lse = torch.full_like(L.lse, float("nan"))
        _lib.dsa_sparse_mla_attend(dw.geom, L.kv_dtype, L.q, L.kv, idx, 2048, wl.sm_scale, out, lse, ws)
        assert _lib.dsa_get_error(ws) == 0
        return out.view(torch.int16).clone(), lse.view(torch.int32).clone()

    ws1 = _lib.workspace(size, DEV)
    ref = run(ws1)
    for _ in range(3):
        got = run(ws1)
        assert torch.equal(got[0], ref[0]) and torch.equal(got[1], ref[1])
    ws2 = _lib.workspace(size, DEV)
    ws2[256:] = ws1[256:]                                # another workspace's partials, fresh header
    got = run(ws2)
    assert torch.equal(got[0], ref[0]) and torch.equal(got[1], ref[1])
    ws3 = _lib.workspace(size, DEV)
    ws3[256:] = torch.randint(0, 256, (size - 256,), dtype=torch.uint8, device=DEV)
    got = run(ws3)
    assert torch.equal(got[0], ref[0]) and torch.equal(got[1], ref[1])
    out = ref[0].view(torch.bfloat16).float().cpu().numpy()
    lse = ref[1].view(torch.float32).cpu().numpy()
    _check(wl, 0, idx.cpu().numpy(), out, lse, ts=list(range(0, wl.T, 11)))


@pytest.mark.parametrize("heads,k,ctx", [(128, 512, [900, 3000]), (16, 16384, [20000])],
                         ids=["128-heads", "k-16384"])
def test_attend_maximum_sizes(heads, k, ctx):
    # the API's limits: H = 128 (eight head groups of 16 on the grid's y axis) and
    # k = 16384 (128 key chunks per query, spread over the clusters and merged)
    rng = np.random.default_rng(heads + k)
    wl = inputs.make_workload("attn", ctx, [1] * len(ctx), topk=k, hi=4, qk_dtype="bf16",
                              kv_dtypes=("bf16",), heads=heads, seed=36)
    dw = runner.DeviceWorkload(wl, DEV)
    idx = _random_idx(rng, wl, k, pad_frac=0.01)
    out, lse = _attend(wl, dw, 0, idx, k)
    worst = _check(wl, 0, idx, out, lse)
    print(f"H={heads} k={k}: max |O err| {worst:.3g}")


@pytest.mark.parametrize("kv_dtype", ["e4m3", "int8"])
def test_record_dequantization_bit_exact(kv_dtype):
    """Every code value times scales from 2^-110 to 1000, read back through the
    attention with one selected row per query (softmax weight exactly 1, so the output
    is the dequantized latent row itself): bit for bit bf16(fp32(code * scale)), the
    rounding the kernel documents, and within bf16 rounding of the oracle's exact
    value. A row holding a NaN code scores NaN, so its whole output row is NaN (as the
    oracle's)."""
    rng = np.random.default_rng(40)
    P, T, H, k = 4, 64, 16, 8
    n_rows = P * 64
    codes = np.empty((n_rows, 512), dtype=np.uint8)
    for r in range(n_rows):
        codes[r] = (np.arange(512) + 37 * r) % 256          # every byte value in every row
    if kv_dtype == "e4m3":   # every 7th row without NaN codes; the others hold both NaN codes
        codes[5:n_rows:7] = np.where(codes[5:n_rows:7] % 128 == 127, 0x7E, codes[5:n_rows:7])
    # scales below 2^7 take the kernel's integer path, larger ones the conversion path;
    # 2^-110 makes the subnormal codes' intermediate fp32 values subnormal too
    scale_set = np.array([1.0, 0.125, 3.7, 200.0, 1e-3, 2.0 ** -110, 0.0078125, 1000.0], dtype=np.float32)
    scales = scale_set[rng.integers(0, len(scale_set), size=(n_rows, 4))].astype(np.float32)
    rope = inputs.to_bf16_bits(rng.standard_normal((n_rows, 64)).astype(np.float32))
    kv = inputs.record_pages(codes.reshape(P, 64, 512), scales.reshape(P, 64, 4), rope.reshape(P, 64, 64))
    # T one-query requests over the same pages (identity block table: position = row)
    bt = np.arange(P, dtype=np.int32)[None].repeat(T, axis=0)
    sel_rows = rng.permutation(n_rows)[:T]
    sel_rows[:2] = [5, 6]                                    # a row without NaN codes and one with them
    q = inputs.to_bf16_bits(rng.standard_normal((T, H, 576)).astype(np.float32))
    seq_t = torch.full((T,), n_rows, dtype=torch.int32, device=DEV)
    cu_t = torch.arange(T + 1, dtype=torch.int32, device=DEV)
    bt_t = torch.from_numpy(bt).to(DEV)
    g = _lib.Geometry(seq_t, cu_t, bt_t, num_pages=P, max_seq_len=n_rows, T=T)
    idx = np.full((T, k), -1, dtype=np.int32)
    idx[:, 3] = sel_rows
    kv_t = torch.from_numpy(kv).to(DEV)
    q_t = torch.from_numpy(q.view(np.int16)).to(DEV).view(torch.bfloat16)
    out = torch.empty(T, H, 512, dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(T, H, dtype=torch.float32, device=DEV)
    ws = _lib.workspace(_lib.dsa_sparse_mla_attend_workspace_size(g, H, k), DEV)
    kvd = _lib.DSA_E4M3 if kv_dtype == "e4m3" else _lib.DSA_I8
    _lib.dsa_sparse_mla_attend(g, kvd, q_t, kv_t, torch.from_numpy(idx).to(DEV), k, 0.1, out, lse, ws)
    assert _lib.dsa_get_error(ws) == 0
    got = out.float().cpu().numpy()
    table = oracle.fp8.E4M3_TABLE if kv_dtype == "e4m3" else np.arange(256, dtype=np.uint8).view(np.int8).astype(np.float64)
    for t in range(T):
        r = int(sel_rows[t])
        vals = table[codes[r]].astype(np.float32) * np.repeat(scales[r], 128)    # fp32 product, one rounding
        exp = torch.from_numpy(vals).to(torch.bfloat16).float().numpy()
        exact = oracle.decode_kv_rows(kv, kv_dtype, np.array([r]))[0, :512]
        ref = oracle.sparse_mla(q, kv, kv_dtype, {t: idx[t]}, seq_t.cpu().numpy(), np.ones(T, dtype=np.int32),
                                bt, 0.1, ts=[t])[t][0]
        if np.isnan(exp).any():
            assert np.isnan(got[t]).all() and np.isnan(ref).all(), (t, r)
            continue
        for h in range(H):
            assert np.array_equal(got[t, h], exp), (t, h, r)
            assert np.all(np.abs(got[t, h] - exact) <= 2.0 ** -8 * np.abs(exact)), (t, h)
            assert np.all(np.abs(got[t, h] - ref[h]) <= 2.0 ** -8 * np.abs(ref[h]) + 1e-12), (t, h)


def _scale_rows(lay, rows, e):
    """Multiply the latent rows `rows` (physical) by 2**e exactly, in place: bf16 values
    by their exponent; records by their four scales and their bf16 RoPE values."""
    def bf16_times(bits, e):
        f = (bits.astype(np.uint32) << 16).view(np.float32) * np.float32(2.0 ** e)
        return (f.view(np.uint32) >> 16).astype(np.uint16)
    P = lay.kv.shape[0]
    if lay.kv_dtype == "bf16":
        kv = lay.kv.reshape(P * inputs.PAGE, -1)
        kv[rows] = bf16_times(kv[rows].view(np.uint16), e).view(kv.dtype)
        return
    pages = lay.kv.reshape(P, -1)
    for r in rows:
        p, s = divmod(int(r), inputs.PAGE)
        sa = inputs.PAGE * inputs.D_LATENT + 16 * s
        sc = pages[p, sa:sa + 16].view(np.float32) * np.float32(2.0 ** e)
        pages[p, sa:sa + 16] = sc.view(np.uint8)
        ra = inputs.PAGE * inputs.D_LATENT + inputs.PAGE * 16 + 128 * s
        pages[p, ra:ra + 128] = bf16_times(pages[p, ra:ra + 128].view(np.uint16), e).view(np.uint8)


@pytest.mark.parametrize("kv_dtype", ["bf16", "e4m3"])
def test_attend_reference_max_rises_over_chunks(kv_dtype):
    """Scores that grow chunk after chunk (the rows of a query's 128-key chunk c scaled by
    2**(c // 2)), so the online softmax's reference max moves by more than 2**8 several
    times within a segment and O is rescaled in TMEM between PVs (both the bf16 and the
    record producers feed it)."""
    rng = np.random.default_rng(77)
    k = 2048
    wl = inputs.make_workload("rise", [3000, 5000, 2600, 8000], [1, 1, 1, 1], topk=k, hi=4,
                              qk_dtype="bf16", kv_dtypes=(kv_dtype,), seed=41)
    lay = wl.layers[0]
    if kv_dtype != "bf16":
        # every record scale a power of two, so that code x scale is exact in bf16 and the
        # kernel's bf16 operands equal the oracle's values: at scores of a few hundred a
        # 2**-9 rounding of the operands would move the softmax weights by itself
        P = lay.kv.shape[0]
        pages = lay.kv.reshape(P, -1)
        sa = inputs.PAGE * inputs.D_LATENT
        pages[:, sa:sa + inputs.PAGE * 16] = np.full(P * inputs.PAGE * 4, 2.0 ** -8, np.float32).view(
            np.uint8).reshape(P, -1)
    _, pos = oracle.query_positions(wl.seq_lens, wl.n_q)
    idx = np.full((wl.T, k), -1, dtype=np.int32)
    for t in range(wl.T):
        sel = np.sort(rng.choice(int(pos[t]) + 1, size=k, replace=False)).astype(np.int32)
        idx[t] = sel
        bt = wl.block_table[t]
        phys = bt[sel // inputs.PAGE].astype(np.int64) * inputs.PAGE + sel % inputs.PAGE
        for c in range(k // 128):
            _scale_rows(lay, phys[128 * c: 128 * (c + 1)], c // 2)
    dw = runner.DeviceWorkload(wl, DEV)
    out, lse = _attend(wl, dw, 0, idx, k)
    # The values are up to 2**7 times the usual latent scale, so the absolute part of the
    # tolerance scales with them: TOL of max|O_ref| (the same relative bound as at unit
    # scale; bf16 output rounding alone is 2**-9 of it). A lost rescale or a PV read
    # before it completed is off by a large fraction of max|O_ref|.
    ref = oracle.sparse_mla(lay.q, lay.kv, lay.kv_dtype, {t: idx[t] for t in range(wl.T)}, wl.seq_lens,
                            wl.n_q, wl.block_table, wl.sm_scale, range(wl.T))
    tol = TOL[kv_dtype]
    worst = 0.0
    for t in range(wl.T):
        o_ref, l_ref = ref[t]
        scale = max(1.0, float(np.abs(o_ref).max()))
        worst = max(worst, assert_close(out[t], o_ref, tol * scale, tol, f"out t={t}") / scale)
        assert_close(lse[t], l_ref, tol, tol, f"lse t={t}")
        assert l_ref.min() > 20.0 and scale > 100.0   # the last chunks dominate
    print(f"{kv_dtype}: max |O err| / max|O| {worst:.3g}")
