"""Pins of the oracle's indexer preparation (oracle/prep.py) against things fixed
outside it: hand-worked non-interleaved RoPE cases (tests/golden/rope_hand.json),
RoPE's rotation invariants (norm, identity, composition, relative position), torch's
float64 layer_norm (with inputs small enough that eps matters), and the quantized
outputs' amax code and error bound, plus the rows the key is written to."""
import json
import os

import numpy as np
import pytest
import torch

from oracle import prep
from oracle import cache as oc
from oracle.fp8 import decode_e4m3

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _tables(max_len, rope_dim, base=10000.0):
    r = rope_dim // 2
    inv = base ** (-np.arange(r, dtype=np.float64) * 2.0 / rope_dim)
    ang = np.arange(max_len, dtype=np.float64)[:, None] * inv[None, :]
    return np.cos(ang), np.sin(ang)


def test_rope_hand_cases():
    with open(os.path.join(GOLDEN, "rope_hand.json")) as f:
        g = json.load(f)
    rd = g["rope_dim"]
    for c in g["cases"]:
        x = np.zeros(128)
        for k, v in c["set"].items():
            x[int(k)] = v
        cos = np.ones(rd // 2)
        sin = np.zeros(rd // 2)
        for k, v in c["cos"].items():
            cos[int(k)] = v
        for k, v in c["sin"].items():
            sin[int(k)] = v
        y = prep.rope_rotate_half(x, cos, sin, rd)
        expect = np.zeros(128)
        expect[:] = x
        for k in c["set"]:
            if int(k) < rd:
                expect[int(k)] = 0.0
        for k, v in c["expect"].items():
            expect[int(k)] = v
        assert np.allclose(y, expect, rtol=0, atol=1e-12), c["note"]


def test_rope_keeps_pair_norms_and_is_identity_at_position_zero():
    rng = np.random.default_rng(1)
    cos, sin = _tables(4096, 64)
    x = rng.standard_normal((50, 128))
    p = rng.integers(0, 4096, 50)
    y = prep.rope_rotate_half(x, cos[p], sin[p], 64)
    n_x = x[:, :32] ** 2 + x[:, 32:64] ** 2
    n_y = y[:, :32] ** 2 + y[:, 32:64] ** 2
    assert np.allclose(n_x, n_y, rtol=1e-12)
    assert np.array_equal(y[:, 64:], x[:, 64:])
    y0 = prep.rope_rotate_half(x, cos[0], sin[0], 64)
    assert np.allclose(y0, x, rtol=0, atol=0)


def test_rope_composes_and_depends_only_on_relative_position():
    rng = np.random.default_rng(2)
    cos, sin = _tables(8192, 64)
    q = rng.standard_normal(128)
    k = rng.standard_normal(128)
    a, b = 1234, 777
    twice = prep.rope_rotate_half(prep.rope_rotate_half(q, cos[a], sin[a], 64), cos[b], sin[b], 64)
    once = prep.rope_rotate_half(q, cos[a + b], sin[a + b], 64)
    assert np.allclose(twice, once, rtol=1e-9, atol=1e-9)
    d0 = prep.rope_rotate_half(q, cos[3000], sin[3000], 64) @ prep.rope_rotate_half(k, cos[2000], sin[2000], 64)
    d1 = prep.rope_rotate_half(q, cos[5500], sin[5500], 64) @ prep.rope_rotate_half(k, cos[4500], sin[4500], 64)
    assert np.isclose(d0, d1, rtol=1e-9, atol=1e-9)


@pytest.mark.parametrize("scale", [1.0, 1e-3])
def test_layer_norm_equals_torch(scale):
    rng = np.random.default_rng(3)
    x = rng.standard_normal((40, 128)) * scale + rng.standard_normal((40, 1))
    gamma = rng.standard_normal(128)
    beta = rng.standard_normal(128)
    eps = 1e-6
    ref = torch.nn.functional.layer_norm(torch.tensor(x), (128,), torch.tensor(gamma), torch.tensor(beta), eps).numpy()
    assert np.allclose(prep.layer_norm(x, gamma, beta, eps), ref, rtol=1e-12, atol=1e-12)
    # eps matters at this size: dropping it moves the result
    if scale < 1:
        assert not np.allclose(prep.layer_norm(x, gamma, beta, 0.0), ref, rtol=1e-6, atol=1e-6)


def test_layer_norm_special_cases():
    beta = np.linspace(-1, 1, 128)
    assert np.allclose(prep.layer_norm(np.full(128, 3.5), np.ones(128), beta, 1e-6), beta)
    rng = np.random.default_rng(4)
    x = rng.standard_normal(128) * 2 + 5
    y = prep.layer_norm(x, np.ones(128), np.zeros(128), 1e-6)
    assert abs(y.mean()) < 1e-12
    var = x.var()
    assert np.isclose(y.var(), var / (var + 1e-6), rtol=1e-12)


def test_prepared_key_closed_form_layernorm_then_rope():
    """Key = +a on its first 64 values and -a on the rest: mean 0, biased variance a^2,
    so LayerNorm gives x_hat = +-a / sqrt(a^2 + eps), then gamma * x_hat + beta; RoPE
    (rope_dim 64) then turns pair i (elements i and i + 32, both from the +a half) by
    the angle of position p, and the other 64 values pass through."""
    a, eps, p = 1.5, 1e-6, 5
    k = np.concatenate([np.full(64, a), np.full(64, -a)]).astype(np.float32)
    k_bits = (k.view(np.uint32) >> 16).astype(np.uint16)[None, :]       # exact in bf16
    gamma = 1.0 + np.arange(128) / 128.0
    beta = np.arange(128) / 256.0
    cos, sin = _tables(16, 64)
    got = prep.prepared_k(k_bits, np.array([p]), cos, sin, 64, gamma, beta, eps)[0]
    xh = np.concatenate([np.full(64, a), np.full(64, -a)]) / np.sqrt(a * a + eps)
    n = xh * gamma + beta
    exp = n.copy()
    for i in range(32):
        c, s = cos[p, i], sin[p, i]
        exp[i] = n[i] * c - n[i + 32] * s
        exp[i + 32] = n[i + 32] * c + n[i] * s
    np.testing.assert_allclose(got, exp, rtol=1e-13, atol=1e-15)


def test_rope_uses_the_table_row_of_each_tokens_position():
    """Tables that hold a quarter turn at one position and the identity elsewhere: only
    the token at that position is turned (y_i = -x_(i+r), y_(i+r) = x_i), for queries
    and keys alike."""
    rng = np.random.default_rng(12)
    r, L, p_turn = 32, 12, 7
    cos, sin = np.ones((L, r)), np.zeros((L, r))
    cos[p_turn], sin[p_turn] = 0.0, 1.0
    pos = np.array([p_turn - 1, p_turn, p_turn + 1])
    q = rng.standard_normal((3, 2, 128)).astype(np.float32)
    q_bits = (q.view(np.uint32) >> 16).astype(np.uint16)
    qd = (q_bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    got = prep.prepared_q(q_bits, pos, cos, sin, 2 * r)
    turned = qd.copy()
    turned[..., :r], turned[..., r:2 * r] = -qd[..., r:2 * r], qd[..., :r]
    np.testing.assert_array_equal(got[0], qd[0])
    np.testing.assert_array_equal(got[1], turned[1])
    np.testing.assert_array_equal(got[2], qd[2])
    # keys: the same rows, applied after the LayerNorm (pinned to torch above)
    kv = rng.standard_normal((3, 128)).astype(np.float32)
    k_bits = (kv.view(np.uint32) >> 16).astype(np.uint16)
    kd = (k_bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    kn = prep.layer_norm(kd, np.ones(128), np.zeros(128), 1e-6)
    gk = prep.prepared_k(k_bits, pos, cos, sin, 2 * r, np.ones(128), np.zeros(128), 1e-6)
    kt = kn.copy()
    kt[:, :r], kt[:, r:2 * r] = -kn[:, r:2 * r], kn[:, :r]
    np.testing.assert_array_equal(gk[0], kn[0])
    np.testing.assert_array_equal(gk[1], kt[1])
    np.testing.assert_array_equal(gk[2], kn[2])


def _geometry():
    seq = np.array([70, 200, 129], dtype=np.int32)
    nq = np.array([2, 1, 3], dtype=np.int32)
    bt = np.array([[3, 1, 0, 0], [5, 2, 4, 6], [7, 8, 9, 0]], dtype=np.int32)
    return seq, nq, bt


def test_prepare_quantizes_to_amax_code_within_bound_and_writes_key_rows():
    rng = np.random.default_rng(5)
    seq, nq, bt = _geometry()
    T, H, P = int(nq.sum()), 4, 10
    cos, sin = _tables(256, 64)
    q_bits = (torch.tensor(rng.standard_normal((T, H, 128)), dtype=torch.float32).to(torch.bfloat16)
              .view(torch.int16).numpy().view(np.uint16))
    k_bits = (torch.tensor(rng.standard_normal((T, 128)) * 2, dtype=torch.float32).to(torch.bfloat16)
              .view(torch.int16).numpy().view(np.uint16))
    gamma = rng.standard_normal(128)
    beta = rng.standard_normal(128) * 0.1
    cache = rng.integers(0, 256, (P, 64, 128), dtype=np.uint8)
    kscale = rng.standard_normal((P, 64)).astype(np.float32)
    qc, qs, kc, ks = prep.indexer_prepare(q_bits, k_bits, seq, nq, bt, cos, sin, 64, gamma, beta, 1e-6, cache, kscale)
    from oracle.dsa import query_positions
    _, pos = query_positions(seq, nq)
    qx = prep.prepared_q(q_bits, pos, cos, sin, 64)
    kx = prep.prepared_k(k_bits, pos, cos, sin, 64, gamma, beta, 1e-6)
    # the largest magnitude of every vector encodes to +-448 (code 0x7E / 0xFE)
    amax_i = np.abs(qx).argmax(axis=-1)
    top = np.take_along_axis(qc, amax_i[..., None], axis=-1)[..., 0]
    assert np.all((top & 0x7F) == 0x7E)
    # dequantized values are within e4m3's half-step of the prepared values
    deq = decode_e4m3(qc) * qs[..., None]
    bound = np.maximum(np.abs(qx) * 2.0 ** -4, qs[..., None] * 2.0 ** -10) * (1 + 1e-6)
    assert np.all(np.abs(deq - qx) <= bound)
    rows = oc.token_rows(seq, nq, bt)
    kflat, sflat = kc.reshape(-1, 128), ks.reshape(-1)
    kdeq = decode_e4m3(kflat[rows]) * sflat[rows][:, None]
    kbound = np.maximum(np.abs(kx) * 2.0 ** -4, sflat[rows][:, None] * 2.0 ** -10) * (1 + 1e-6)
    assert np.all(np.abs(kdeq - kx) <= kbound)
    assert np.allclose(sflat[rows], np.abs(kx).max(axis=-1) / 448.0, rtol=1e-6)
    untouched = np.ones(P * 64, dtype=bool)
    untouched[rows] = False
    assert np.array_equal(kflat[untouched], cache.reshape(-1, 128)[untouched])
    assert np.array_equal(sflat[untouched], kscale.reshape(-1)[untouched])
    # a row the queries' positions map to: request 1's token sits at 199 -> page 2 of its table
    assert rows[2] == bt[1][199 // 64] * 64 + 199 % 64
