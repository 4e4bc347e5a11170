"""dsa_indexer_prepare on the GPU against the oracle's preparation (oracle/prep.py).

The GPU computes RoPE and LayerNorm in fp32, the oracle in float64. The fp32
results carry an error of a few ulps of their operands, not of themselves (the two
RoPE products can nearly cancel); RoPE keeps each pair's norm, so the operands are at
most 2x the vector's amax, and the error stays below 2^-18 of the amax (with a 4x
margin for RoPE; LayerNorm's sums over 128 values are of the same order here). In
quotient units (amax -> 448) that is 448 * 2^-18. Codes are therefore equal except
where the exact quotient lies within that distance of the midpoint between two
neighbouring e4m3 values, and there the GPU's code is one of those two; scales
agree to 1e-5 (relative). Rows of the key cache other than the new tokens' are
bit-exact. Then the prepared outputs feed dsa_indexer_scores, checked against the
oracle's scores from the oracle's own preparation."""
import numpy as np
import pytest
import torch

import oracle
from oracle import prep
from oracle import cache as oc
from oracle.fp8 import decode_e4m3
from dsa_sparse_attention_02_gb300 import _lib, inputs, runner
from gpu_helpers import DEV

pytestmark = pytest.mark.gpu

REL = 1e-5
MID_TOL = 448.0 * 2.0 ** -18      # quotient units


def _dev(a):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(DEV)
    return torch.from_numpy(a).to(DEV)


def _check_codes(got, x64, scale_ref, what):
    """got: GPU codes [N, 128]; x64: the oracle's prepared values [N, 128]; scale_ref: [N]."""
    ref, _ = oc.quantize_groups(x64.astype(np.float32), 128)
    bad = got != ref
    if bad.any():
        u = (x64 / scale_ref[:, None].astype(np.float64))[bad]
        vg, vr = decode_e4m3(got[bad]), decode_e4m3(ref[bad])
        mid = (vg + vr) / 2
        near = np.abs(u - mid) <= MID_TOL
        zero = (vg == 0) & (vr == 0)                          # +0 / -0 of a tiny value
        ok = (near | zero) & (np.sign(vg) * np.sign(vr) >= 0)
        assert ok.all(), (what, int((~ok).sum()), u[~ok][:5], vg[~ok][:5], vr[~ok][:5])
        assert bad.mean() < 1e-3, (what, bad.mean())
    return int(bad.sum())


def _run(wl, pi, hi, with_k=True, ln=True, bt=None):
    T = int(wl.n_q.sum())
    dw_geom_bt = wl.block_table if bt is None else bt
    cu = np.concatenate([[0], np.cumsum(wl.n_q)]).astype(np.int32)
    tens = [torch.from_numpy(np.ascontiguousarray(a).astype(np.int32)).to(DEV)
            for a in (wl.seq_lens, cu, dw_geom_bt)]
    g = _lib.Geometry(tens[0], tens[1], tens[2], num_pages=wl.num_pages, max_seq_len=int(wl.max_seq_len), T=T)
    g._keep = tens
    q_out = torch.zeros(T, hi, 128, dtype=torch.uint8, device=DEV)
    q_scale = torch.full((T, hi), float("nan"), dtype=torch.float32, device=DEV)
    kc = _dev(wl.idx_k.copy())
    ks = _dev(wl.idx_k_scale.copy())
    ws = _lib.workspace(_lib.dsa_indexer_prepare_workspace_size(g), DEV)
    _lib.dsa_indexer_prepare(g, hi, pi.rope_dim, _dev(pi.q_in), _dev(pi.k_in) if with_k else None,
                             _dev(pi.rope_cos), _dev(pi.rope_sin),
                             _dev(pi.ln_gamma) if ln else None, _dev(pi.ln_beta) if ln else None, pi.ln_eps,
                             q_out, q_scale, kc, ks, ws)
    err = _lib.dsa_get_error(ws)
    return (g, q_out.cpu().numpy(), q_scale.cpu().numpy(), kc.cpu().numpy(), ks.cpu().numpy(), err)


def _reference(wl, pi, hi, ln=True, with_k=True):
    gamma = pi.ln_gamma if ln else np.ones(128, np.float32)
    beta = pi.ln_beta if ln else np.zeros(128, np.float32)
    _, pos = oracle.query_positions(wl.seq_lens, wl.n_q)
    qx = prep.prepared_q(pi.q_in, pos, pi.rope_cos, pi.rope_sin, pi.rope_dim)
    kx = prep.prepared_k(pi.k_in, pos, pi.rope_cos, pi.rope_sin, pi.rope_dim, gamma, beta, pi.ln_eps)
    qc, qs, kc, ks = prep.indexer_prepare(pi.q_in, pi.k_in if with_k else None, wl.seq_lens, wl.n_q,
                                          wl.block_table, pi.rope_cos, pi.rope_sin, pi.rope_dim, gamma, beta,
                                          pi.ln_eps, wl.idx_k, wl.idx_k_scale)
    return qx, kx, qc, qs, kc, ks


def _compare(wl, pi, hi, got, ref, with_k=True):
    _, q_out, q_scale, kc, ks, err = got
    qx, kx, _, qs, kc_ref, ks_ref = ref
    assert err == 0
    T = int(wl.n_q.sum())
    assert np.allclose(q_scale, qs, rtol=REL, atol=0)
    nq = _check_codes(q_out.reshape(T * hi, 128), qx.reshape(T * hi, 128), qs.reshape(-1), "q")
    rows = oc.token_rows(wl.seq_lens, wl.n_q, wl.block_table)
    kflat, sflat = kc.reshape(-1, 128), ks.reshape(-1)
    untouched = np.ones(kflat.shape[0], dtype=bool)
    if with_k:
        untouched[rows] = False
        assert np.allclose(sflat[rows], ks_ref.reshape(-1)[rows], rtol=REL, atol=0)
        _check_codes(kflat[rows], kx, sflat[rows], "k")
    assert np.array_equal(kflat[untouched], wl.idx_k.reshape(-1, 128)[untouched])
    assert np.array_equal(sflat[untouched].view(np.uint32), wl.idx_k_scale.reshape(-1)[untouched].view(np.uint32))
    return nq


def test_prepare_decode_size_matches_oracle():
    wl = inputs.make_config("decode")
    pi = inputs.make_prep_inputs(wl, hi=64, rope_dim=64, seed=41)
    got = _run(wl, pi, 64)
    n = _compare(wl, pi, 64, got, _reference(wl, pi, 64))
    print(f"decode: {n} of {wl.T * 64 * 128} query codes on a rounding midpoint")


@pytest.mark.parametrize("rope_dim", [8, 128])
def test_prepare_rope_widths_position_zero_and_no_affine(rope_dim):
    # request 0 has one token at position 0 (no rotation), request 1 two tokens, request 2 one
    wl = inputs.make_workload("prep", [1, 200, 70], [1, 2, 1], topk=64, hi=4, qk_dtype="e4m3", seed=42)
    pi = inputs.make_prep_inputs(wl, hi=4, rope_dim=rope_dim, seed=43)
    pi.q_in[2, 1] = 0                                   # an all-zero query head: scale 1, codes 0
    got = _run(wl, pi, 4, ln=False)
    _compare(wl, pi, 4, got, _reference(wl, pi, 4, ln=False))
    assert got[2][2, 1] == 1.0 and not (got[1][2, 1] & 0x7F).any()   # +-0 codes (RoPE may flip the sign of 0)


def test_prepare_queries_only_leaves_the_key_cache():
    wl = inputs.make_workload("prep", [300, 90], [3, 1], topk=64, hi=16, qk_dtype="e4m3", seed=44)
    pi = inputs.make_prep_inputs(wl, hi=16, rope_dim=64, seed=45)
    got = _run(wl, pi, 16, with_k=False)
    _compare(wl, pi, 16, got, _reference(wl, pi, 16, with_k=False), with_k=False)


def test_prepare_skips_and_reports_out_of_range_pages():
    wl = inputs.make_workload("prep", [130, 64, 500], [2, 1, 1], topk=64, hi=8, qk_dtype="e4m3", seed=46)
    pi = inputs.make_prep_inputs(wl, hi=8, rope_dim=64, seed=47)
    bad = wl.block_table.copy()
    bad[0, 2] = 10_000                                  # request 0's tokens (positions 128, 129)
    got = _run(wl, pi, 8, bt=bad)
    assert got[5] == _lib.DSA_ERR_BAD_INDEX
    _, q_out, q_scale, kc, ks, _ = got
    qx, kx, qc, qs, _, _ = _reference(wl, pi, 8)
    assert np.allclose(q_scale, qs, rtol=REL, atol=0)   # the queries are prepared regardless
    rows = oc.token_rows(wl.seq_lens, wl.n_q, wl.block_table)
    kflat, sflat = kc.reshape(-1, 128), ks.reshape(-1)
    _check_codes(kflat[rows[2:]], kx[2:], sflat[rows[2:]], "k")   # the other requests' keys are written
    keep = np.ones(kflat.shape[0], dtype=bool)
    keep[rows[2:]] = False
    assert np.array_equal(kflat[keep], wl.idx_k.reshape(-1, 128)[keep])


def test_prepare_prefill_chunk():
    wl = inputs.make_config("prefill", ctx_scale=1 / 8)     # 2048 tokens at positions 0..2047 of 2048
    pi = inputs.make_prep_inputs(wl, hi=64, rope_dim=64, seed=48)
    got = _run(wl, pi, 64)
    _compare(wl, pi, 64, got, _reference(wl, pi, 64))


def test_prepared_outputs_feed_the_indexer():
    wl = inputs.make_config("decode", batch=4)
    pi = inputs.make_prep_inputs(wl, hi=64, rope_dim=64, seed=49)
    g, q_out, q_scale, kc, ks, err = _run(wl, pi, 64)
    assert err == 0
    _, _, qc_ref, qs_ref, kc_ref, ks_ref = _reference(wl, pi, 64)
    T = wl.T
    stride = int(-(-wl.max_seq_len // 64) * 64)
    scores = torch.zeros(T, stride, dtype=torch.float32, device=DEV)
    ws = _lib.workspace(_lib.dsa_indexer_scores_workspace_size(g), DEV)
    _lib.dsa_indexer_scores(g, _lib.DSA_E4M3, _dev(q_out).view(torch.float8_e4m3fn), _dev(q_scale), _dev(wl.w),
                            _dev(kc).view(torch.float8_e4m3fn), _dev(ks), scores, ws)
    assert _lib.dsa_get_error(ws) == 0
    sc = scores.cpu().numpy()
    ts = list(range(T))
    ref = oracle.indexer_scores(qc_ref, qs_ref, wl.w, kc_ref, ks_ref, "e4m3", wl.seq_lens, wl.n_q, wl.block_table, ts)
    _, pos = oracle.query_positions(wl.seq_lens, wl.n_q)
    for t in ts:
        p = int(pos[t])
        r = ref[t]
        err_t = np.abs(sc[t, : p + 1].astype(np.float64) - r).max() / np.abs(r).max()
        assert err_t <= 1e-3, (t, err_t)
