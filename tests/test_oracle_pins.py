"""Pins of the CPU oracle to facts outside itself (no GPU needed).

Each test ties one oracle function to a hand-worked example (tests/golden/),
a library routine it does not itself call for that step, a closed form, or an
invariant the method must satisfy, so that a dropped term, a wrong sign or
index, or a transposed operand fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle.fp8 import decode_bf16
from dsa_sparse_attention_02_gb300 import inputs as synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ----------------------------------------------------------------------------- decoders

def test_e4m3_table_matches_torch_all_codes():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = oracle.E4M3_TABLE
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(ours))
    assert nan.sum() == 2                       # 0x7F and 0xFF
    assert np.array_equal(ref[~nan], ours[~nan])
    assert np.nanmax(ours) == 448.0 and ours[1] == 2.0 ** -9


def test_bf16_decode_matches_torch():
    rng = np.random.default_rng(0)
    bits = rng.integers(0, 65536, size=4096, dtype=np.int64).astype(np.uint16)
    t = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    ours = oracle.decode_bf16(bits)
    ok = ~np.isnan(t)
    assert np.array_equal(np.isnan(ours), np.isnan(t))
    assert np.array_equal(ours[ok], t[ok])


def test_fp8_record_decode_by_hand():
    g = _golden("fp8_record.json")
    # two pages of records; the record sits at page 1, slot 5 (physical row 69), at the
    # byte offsets the golden gives: codes, scales and RoPE each in their own plane
    rec = np.zeros((2, 64 * 656), dtype=np.uint8)
    off = g["offsets_in_page_for_slot_5"]
    rec[1, off["codes"]:off["codes"] + 512] = g["latent_code"]
    rec[1, off["scales"]:off["scales"] + 16] = np.array(g["scales"], dtype="<f4").view(np.uint8)
    rec[1, off["rope"]:off["rope"] + 128] = np.full(64, g["rope_bf16_bits"], dtype="<u2").view(np.uint8)
    row = oracle.decode_kv_rows(rec, "e4m3", np.array([69]))[0]
    exp = np.concatenate([np.full(128, s) for s in g["scales"]] + [np.full(64, g["rope_value"])])
    assert np.array_equal(row, exp)
    # every other row of the two pages decodes to zeros (nothing of it was written)
    others = oracle.decode_kv_rows(rec, "e4m3", np.array([r for r in range(128) if r != 69]))
    assert not others.any()


# ----------------------------------------------------------------------------- geometry

def test_query_positions_hand():
    req, pos = oracle.query_positions([5, 3, 7], [2, 1, 3])
    assert req.tolist() == [0, 0, 1, 2, 2, 2]
    assert pos.tolist() == [3, 4, 2, 4, 5, 6]


def test_physical_rows_hand():
    bt = np.array([7, 2, 5])
    assert oracle.physical_rows(bt, [0, 63, 64, 130]).tolist() == [448, 511, 128, 322]


# ----------------------------------------------------------------------------- indexer

def _hand_indexer_inputs():
    g = _golden("indexer_hand.json")
    q = np.array(g["q_idx_codes"], dtype=np.uint8)
    qs = np.array(g["q_scale"], dtype=np.float32)
    w = np.array(g["w"], dtype=np.float32)
    keys = np.zeros((1, 64, 4), dtype=np.uint8)
    keys[0, :3] = np.array(g["key_codes_rows_0_to_2"], dtype=np.uint8)
    ks = np.ones((1, 64), dtype=np.float32)
    ks[0, :3] = g["k_scale_rows_0_to_2"]
    return g, q, qs, w, keys, ks


def test_indexer_hand_example():
    g, q, qs, w, keys, ks = _hand_indexer_inputs()
    sc = oracle.indexer_scores(q, qs, w, keys, ks, "e4m3", g["seq_lens"], g["n_q"],
                               np.array(g["block_table"]))
    for t, exp in g["expected_scores"].items():
        assert sc[int(t)].tolist() == exp
    for kk, table in g["expected_topk"].items():
        k = int(kk.split("=")[1])
        for t, exp in table.items():
            assert oracle.topk_row(sc[int(t)], k).tolist() == exp


def _rand_indexer(seed, Hi=3, D=16, L=40, n_q=3):
    rng = np.random.default_rng(seed)
    q = rng.integers(0, 256, size=(n_q, Hi, D)).astype(np.uint8)
    q[(q & 0x7F) == 0x7F] = 0x38                                # no NaN codes
    keys = rng.integers(0, 256, size=(1, 64, D)).astype(np.uint8)
    keys[(keys & 0x7F) == 0x7F] = 0x30
    qs = rng.uniform(0.1, 2.0, size=(n_q, Hi)).astype(np.float32)
    ks = rng.uniform(0.1, 2.0, size=(1, 64)).astype(np.float32)
    w = rng.standard_normal((n_q, Hi)).astype(np.float32)
    return dict(q_idx=q, q_scale=qs, w=w, idx_k=keys, idx_k_scale=ks, qk_dtype="e4m3",
                seq_lens=[L], n_q=[n_q], block_table=np.array([[0]]))


def test_indexer_linear_in_w_and_positively_homogeneous_in_scales():
    a = _rand_indexer(1)
    base = oracle.indexer_scores(**a)
    # linear in w
    w2 = np.random.default_rng(9).standard_normal(a["w"].shape).astype(np.float32)
    s2 = oracle.indexer_scores(**{**a, "w": w2})
    s12 = oracle.indexer_scores(**{**a, "w": a["w"].astype(np.float64) + w2})
    for t in base:
        np.testing.assert_allclose(s12[t], base[t] + s2[t], rtol=1e-12, atol=1e-9)
    # ReLU(c x) = c ReLU(x) for c > 0: scaling q_scale by 3 scales the scores by 3
    s3 = oracle.indexer_scores(**{**a, "q_scale": a["q_scale"] * 3})
    for t in base:
        np.testing.assert_allclose(s3[t], 3 * base[t], rtol=1e-6)
    # negating q flips the sign of every logit: the ReLU keeps the other half
    neg = a["q_idx"] ^ np.uint8(0x80)
    sn = oracle.indexer_scores(**{**a, "q_idx": neg, "w": np.ones_like(a["w"])})
    sp = oracle.indexer_scores(**{**a, "w": np.ones_like(a["w"])})
    for t in base:
        assert np.all(sn[t] >= 0) and np.all(sp[t] >= 0)


def test_indexer_single_head_is_relu_of_dot():
    a = _rand_indexer(2, Hi=1)
    a["w"] = np.ones_like(a["w"])
    sc = oracle.indexer_scores(**a)
    qd = oracle.decode_e4m3(a["q_idx"]) * a["q_scale"][..., None]
    kd = oracle.decode_e4m3(a["idx_k"][0]) * a["idx_k_scale"][0][:, None]
    _, pos = oracle.query_positions(a["seq_lens"], a["n_q"])
    for t in sc:
        # dot products via einsum over explicit loops of the keys (a different route)
        dots = np.array([float(np.einsum("d,d->", kd[s], qd[t, 0])) for s in range(pos[t] + 1)])
        np.testing.assert_allclose(sc[t], np.maximum(dots, 0.0), rtol=1e-12, atol=1e-12)


def test_indexer_causal():
    a = _rand_indexer(3)
    base = oracle.indexer_scores(**a)
    _, pos = oracle.query_positions(a["seq_lens"], a["n_q"])
    k2 = a["idx_k"].copy()
    k2[0, pos.min() + 1:] = np.uint8(0x48)     # rewrite every key a query may not see
    alt = oracle.indexer_scores(**{**a, "idx_k": k2})
    for t in base:
        assert len(base[t]) == pos[t] + 1
        n_vis = pos.min() + 1
        np.testing.assert_array_equal(base[t][:n_vis], alt[t][:n_vis])


# ----------------------------------------------------------------------------- top-k

def test_topk_hand_cases():
    for c in _golden("topk_ties.json")["cases"]:
        assert oracle.topk_row(np.array(c["row"], dtype=np.float64), c["k"]).tolist() == c["expected"], c


def test_topk_matches_brute_force_sort_with_ties():
    rng = np.random.default_rng(5)
    for _ in range(200):
        n = int(rng.integers(1, 60))
        k = int(rng.integers(1, 70))
        row = rng.integers(-5, 6, size=n).astype(np.float64)   # many exact ties
        ranked = sorted(range(n), key=lambda s: (-row[s], s))
        exp = sorted(ranked[:k]) + [-1] * max(0, k - n)
        assert oracle.topk_row(row, k).tolist() == exp


def test_topk_set_matches_torch_topk_on_distinct_values():
    rng = np.random.default_rng(6)
    for n, k in [(100, 10), (5000, 2048), (2048, 2048), (3000, 1)]:
        row = rng.permutation(n).astype(np.float64) + rng.uniform(0, 0.5, n)
        ref = torch.topk(torch.from_numpy(row), min(k, n)).indices.numpy()
        got = oracle.topk_row(row, k)
        assert set(got[got >= 0].tolist()) == set(ref.tolist())
        assert np.all(np.diff(got[got >= 0]) > 0)


def test_topk_invariant_to_positive_rescale_of_w():
    a = _rand_indexer(7, L=60)
    s1 = oracle.indexer_scores(**a)
    s2 = oracle.indexer_scores(**{**a, "w": a["w"] * np.float32(4.0)})
    for t in s1:
        assert np.array_equal(oracle.topk_row(s1[t], 8), oracle.topk_row(s2[t], 8))


# ----------------------------------------------------------------------------- attention

def _bf16(x):
    return synth.to_bf16_bits(np.asarray(x, dtype=np.float32))


def test_attention_hand_example():
    # one head, D = 3 with a 2-wide value part; q only touches the last ("RoPE") column
    q = _bf16([[[0.0, 0.0, 1.0]]])                                   # [T=1, H=1, 3]
    kv = np.zeros((1, 64, 3), dtype=np.float32)
    kv[0, 0] = [1, 2, 0]
    kv[0, 1] = [3, -1, 1]
    kv[0, 2] = [0.5, 0.5, 1]
    idx = np.array([[0, 1, -1]])                                      # row 2 is padding
    out = oracle.sparse_mla(q, _bf16(kv), "bf16", idx, [3], [1], np.array([[0]]), 1.0, dv=2)
    o, lse = out[0]
    e = math.e
    np.testing.assert_allclose(o[0], [(1 + 3 * e) / (1 + e), (2 - e) / (1 + e)], rtol=1e-14)
    np.testing.assert_allclose(lse[0], math.log(1 + e), rtol=1e-14)


def test_attention_identical_rows_closed_form():
    rng = np.random.default_rng(11)
    v = rng.standard_normal(576).astype(np.float32)
    kv = np.tile(v, (1, 64, 1))
    q = rng.standard_normal((1, 4, 576)).astype(np.float32)
    qb, kvb = _bf16(q), _bf16(kv)
    idx = np.array([[3, 9, 17, 40, 41, -1, -1]])
    o, lse = oracle.sparse_mla(qb, kvb, "bf16", idx, [64], [1], np.array([[0]]), 0.1)[0]
    vd = oracle.decode_bf16(kvb[0, 0])
    z = 0.1 * (oracle.decode_bf16(qb[0]) @ vd)
    np.testing.assert_allclose(o, np.tile(vd[:512], (4, 1)), rtol=1e-12)
    np.testing.assert_allclose(lse, z + math.log(5), rtol=1e-12)


def test_sparse_equals_dense_sdpa_when_context_within_topk():
    wl = synth.make_workload("pin", [50, 64, 37], [1, 2, 3], topk=64, hi=4, qk_dtype="bf16",
                             seed=21)
    res = oracle.dsa_step(wl)
    req, pos = oracle.query_positions(wl.seq_lens, wl.n_q)
    layer = wl.layers[0]
    for t in range(wl.T):
        b, p = int(req[t]), int(pos[t])
        assert res["idx"][t][: p + 1].tolist() == list(range(p + 1))
        rows = oracle.physical_rows(wl.block_table[b], np.arange(p + 1))
        kv = torch.from_numpy(oracle.decode_kv_rows(layer.kv, "bf16", rows))       # [n, 576]
        qt = torch.from_numpy(oracle.decode_bf16(layer.q[t]))                      # [H, 576]
        ref = torch.nn.functional.scaled_dot_product_attention(
            qt[:, None, :], kv[None].expand(qt.shape[0], -1, -1),
            kv[None, :, :512].expand(qt.shape[0], -1, -1), scale=wl.sm_scale)[:, 0]
        np.testing.assert_allclose(res["out"][0][t][0], ref.numpy(), rtol=1e-10, atol=1e-12)


def test_gather_equals_mask_formulation():
    wl = synth.make_workload("pin", [300, 190], [2, 1], topk=32, hi=4, qk_dtype="bf16", seed=22)
    res = oracle.dsa_step(wl)
    layer = wl.layers[0]
    dense = oracle.masked_dense_mla(layer.q, layer.kv, "bf16", res["idx"], wl.seq_lens, wl.n_q,
                                    wl.block_table, wl.sm_scale)
    for t in range(wl.T):
        np.testing.assert_allclose(res["out"][0][t][0], dense[t][0], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(res["out"][0][t][1], dense[t][1], rtol=1e-12)


def test_block_table_permutation_invariance():
    wl = synth.make_workload("pin", [130, 200], [1, 2], topk=48, hi=4, qk_dtype="e4m3",
                             kv_dtypes=("e4m3",), seed=23)
    base = oracle.dsa_step(wl)
    rng = np.random.default_rng(3)
    perm = rng.permutation(wl.num_pages)            # new physical slot of each old page
    inv = np.argsort(perm)
    wl2 = synth.Workload(**{**wl.__dict__})
    wl2.block_table = perm[wl.block_table].astype(np.int32)
    wl2.idx_k = wl.idx_k[inv]
    wl2.idx_k_scale = wl.idx_k_scale[inv]
    wl2.layers = [synth.Layer(q=l.q, kv=l.kv[inv], kv_dtype=l.kv_dtype) for l in wl.layers]
    alt = oracle.dsa_step(wl2)
    for t in range(wl.T):
        assert np.array_equal(base["idx"][t], alt["idx"][t])
        np.testing.assert_array_equal(base["out"][0][t][0], alt["out"][0][t][0])


def test_causality_of_the_whole_step():
    wl = synth.make_workload("pin", [260], [4], topk=40, hi=4, qk_dtype="e4m3", seed=24)
    base = oracle.dsa_step(wl)
    # rewrite every key and latent row at positions > the first query's position
    _, pos = oracle.query_positions(wl.seq_lens, wl.n_q)
    p0 = int(pos[0])
    wl2 = synth.Workload(**{**wl.__dict__})
    wl2.idx_k = wl.idx_k.copy()
    kv2 = wl.layers[0].kv.copy()
    rows = oracle.physical_rows(wl.block_table[0], np.arange(p0 + 1, 260))
    wl2.idx_k.reshape(-1, 128)[rows] = np.uint8(0x48)
    kv2.reshape(-1, 576)[rows] = _bf16(np.full(576, 3.0))
    wl2.layers = [synth.Layer(q=wl.layers[0].q, kv=kv2, kv_dtype="bf16")]
    alt = oracle.dsa_step(wl2, ts=[0])
    assert np.array_equal(base["idx"][0], alt["idx"][0])
    np.testing.assert_array_equal(base["out"][0][0][0], alt["out"][0][0][0])


def test_fewer_valid_keys_than_topk_are_padded():
    wl = synth.make_workload("pin", [20, 70], [1, 1], topk=64, hi=4, qk_dtype="bf16", seed=25)
    res = oracle.dsa_step(wl)
    assert res["idx"][0].tolist() == list(range(20)) + [-1] * 44
    assert (res["idx"][1] >= 0).sum() == 64


def test_indexshare_layer_reuses_full_layer_selection():
    wl = synth.make_workload("pin", [300, 150], [4, 2], topk=32, hi=4, qk_dtype="e4m3",
                             kv_dtypes=("e4m3", "bf16"), seed=26)
    res = oracle.dsa_step(wl)
    l1 = wl.layers[1]
    alone = oracle.sparse_mla(l1.q, l1.kv, l1.kv_dtype, res["idx"], wl.seq_lens, wl.n_q,
                              wl.block_table, wl.sm_scale)
    reused = oracle.dsa_step(wl, reuse_idx=res["idx"])
    for t in range(wl.T):
        np.testing.assert_array_equal(res["out"][1][t][0], alone[t][0])
        assert np.array_equal(reused["idx"][t], res["idx"][t])
        np.testing.assert_array_equal(reused["out"][0][t][0], res["out"][0][t][0])
    # a given selection that is not the indexer's: every layer attends over exactly it,
    # and no score is computed (the shared layer skips the indexer)
    _, pos = oracle.query_positions(wl.seq_lens, wl.n_q)
    other = {t: np.array([s if s <= pos[t] else -1 for s in range(0, 2 * 32, 2)], dtype=np.int32)
             for t in range(wl.T)}
    assert any(set(other[t]) != set(res["idx"][t]) for t in range(wl.T))
    given = oracle.dsa_step(wl, reuse_idx=other)
    assert given["scores"] == {}
    for li, layer in enumerate(wl.layers):
        ref = oracle.sparse_mla(layer.q, layer.kv, layer.kv_dtype, other, wl.seq_lens, wl.n_q,
                                wl.block_table, wl.sm_scale)
        for t in range(wl.T):
            assert np.array_equal(given["idx"][t], other[t])
            np.testing.assert_array_equal(given["out"][li][t][0], ref[t][0])


def test_split_merge_identity_and_empty_selection():
    """Attention over a set S equals the log-sum-exp merge of attention over any two
    disjoint parts of S: LSE = log(e^LSE1 + e^LSE2), O = e^(LSE1-LSE) O1 + e^(LSE2-LSE) O2
    (the split-KV combine's identity). An all-padding selection is the empty sum:
    LSE = log 0 = -inf and, as the merge requires, contributes nothing (O = 0)."""
    wl = synth.make_workload("pin", [400, 230], [2, 1], topk=64, hi=4, qk_dtype="bf16",
                             kv_dtypes=("bf16", "e4m3"), seed=28)
    res = oracle.dsa_step(wl)
    rng = np.random.default_rng(8)
    for layer in wl.layers:
        full = oracle.sparse_mla(layer.q, layer.kv, layer.kv_dtype, res["idx"], wl.seq_lens, wl.n_q,
                                 wl.block_table, wl.sm_scale)
        for t in range(wl.T):
            sel = res["idx"][t]
            part = rng.random(sel.shape[0]) < 0.3
            a = {t: np.where(part, sel, -1)}
            b = {t: np.where(part, -1, sel)}
            empty = {t: np.full(sel.shape[0], -1, dtype=np.int32)}
            (o1, l1), (o2, l2), (o0, l0) = (
                oracle.sparse_mla(layer.q, layer.kv, layer.kv_dtype, x, wl.seq_lens, wl.n_q,
                                  wl.block_table, wl.sm_scale, ts=[t])[t] for x in (a, b, empty))
            lse = np.logaddexp(l1, l2)
            o = np.exp(l1 - lse)[:, None] * o1 + np.exp(l2 - lse)[:, None] * o2
            np.testing.assert_allclose(lse, full[t][1], rtol=1e-13)
            np.testing.assert_allclose(o, full[t][0], rtol=1e-11, atol=1e-13)
            assert np.all(l0 == -np.inf) and np.all(o0 == 0.0)
            lse0 = np.logaddexp(full[t][1], l0)
            np.testing.assert_array_equal(lse0, full[t][1])
            np.testing.assert_array_equal(np.exp(full[t][1] - lse0)[:, None] * full[t][0]
                                          + np.exp(l0 - lse0)[:, None] * o0, full[t][0])


def test_fp8_latent_dequant_is_exact_product():
    wl = synth.make_workload("pin", [64], [1], topk=8, hi=4, qk_dtype="bf16",
                             kv_dtypes=("e4m3",), seed=27)
    rec = wl.layers[0].kv
    rows = np.arange(64)
    dec = oracle.decode_kv_rows(rec, "e4m3", rows)
    page = rec.reshape(-1, 64 * 656)[0]                       # rows 0..63 are page 0's slots
    scales = page[32768:33792].reshape(64, 16).copy().view("<f4").astype(np.float64)
    codes = torch.from_numpy(page[:32768].reshape(64, 512).copy()).view(torch.float8_e4m3fn)
    ref = codes.to(torch.float64).numpy() * np.repeat(scales, 128, axis=1)
    np.testing.assert_array_equal(dec[:, :512], ref)
    # the quantized latent stays within half an e4m3 step (2^-4 relative) of amax-scaled data
    assert np.all(np.abs(dec[:, :512]).max(axis=1) <= 448 * scales.max(axis=1) + 1e-12)


def test_int8_latent_record_decodes_like_the_bf16_rows_it_stands_for():
    """An int8 record whose codes times scales are exact bf16 values gives the same
    attention as the bf16 cache holding those values (mlx-lm int8 MLA latent KV:
    dequantized on read)."""
    rng = np.random.default_rng(31)
    P, T, H = 3, 2, 4
    scales = np.float32(2.0) ** rng.integers(-6, -2, size=(P, 64, 4)).astype(np.float32)
    codes = rng.integers(-127, 128, size=(P, 64, 512)).astype(np.int8)
    rope = rng.standard_normal((P, 64, 64)).astype(np.float32)
    rope_bits = (rope.view(np.uint32) >> 16).astype(np.uint16)
    rec = np.empty((P, 64 * 656), dtype=np.uint8)              # per page: codes | scales | RoPE planes
    rec[:, :32768] = codes.view(np.uint8).reshape(P, -1)
    rec[:, 32768:33792] = np.ascontiguousarray(scales, dtype="<f4").view(np.uint8).reshape(P, -1)
    rec[:, 33792:] = np.ascontiguousarray(rope_bits, dtype="<u2").view(np.uint8).reshape(P, -1)
    lat = codes.astype(np.float32) * np.repeat(scales, 128, axis=-1)          # exact in bf16 (8-bit codes x 2^k)
    full = np.concatenate([lat, decode_bf16(rope_bits).astype(np.float32)], axis=-1)
    kv_bf16 = (full.view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal(decode_bf16(kv_bf16), full.astype(np.float64))
    seq = np.array([150, 40], dtype=np.int32)
    nq = np.array([1, 1], dtype=np.int32)
    bt = np.array([[2, 0, 1], [1, 0, 0]], dtype=np.int32)
    q = (rng.standard_normal((T, H, 576)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    idx = {0: np.array([0, 5, 64, 149, -1], dtype=np.int32), 1: np.array([3, 39, -1, -1, -1], dtype=np.int32)}
    a = oracle.sparse_mla(q, rec, "int8", idx, seq, nq, bt, 0.07, [0, 1])
    b = oracle.sparse_mla(q, kv_bf16, "bf16", idx, seq, nq, bt, 0.07, [0, 1])
    for t in (0, 1):
        assert np.allclose(a[t][0], b[t][0], rtol=0, atol=1e-12)
        assert np.allclose(a[t][1], b[t][1], rtol=0, atol=1e-12)
