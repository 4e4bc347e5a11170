"""Pins of the oracle's cache append (oracle/cache.py) against things fixed outside it:
torch's e4m3 cast over a dense sweep, hand-worked encodings and a hand-worked record
(tests/golden/), round-trip error bounds, the row mapping the attention reads, and
that no other row changes."""
import json
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from oracle import cache as oc
from oracle.fp8 import E4M3_TABLE, decode_bf16, decode_e4m3, decode_f32le

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _record(kv, r):
    """Bytes of physical row r in a latent record cache, read at the layout's offsets:
    per 64-token page, codes [64][512] at 0, scales [64][4] fp32 at 32768, RoPE
    [64][64] bf16 at 33792."""
    page, s = divmod(int(r), 64)
    pg = kv.reshape(-1, 64 * 656)[page]
    return pg[s * 512:(s + 1) * 512], pg[32768 + s * 16:32768 + (s + 1) * 16], pg[33792 + s * 128:33792 + (s + 1) * 128]


def torch_e4m3(v):
    t = torch.tensor(np.asarray(v, dtype=np.float32)).clamp(-448.0, 448.0)
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_encoder_equals_torch_cast_on_values_midpoints_and_neighbours():
    vals = E4M3_TABLE[:0x7F]
    mids = (vals[:-1] + vals[1:]) / 2
    base = np.concatenate([vals, mids, -vals, -mids, [0.0, -0.0, 449.0, 470.0, -1e30, 1e-30, -1e-30]])
    f32 = base.astype(np.float32)
    rng = np.random.default_rng(7)
    wide = (rng.standard_normal(20000) * np.exp2(rng.uniform(-14, 9, 20000))).astype(np.float32)
    allv = np.concatenate([f32, np.nextafter(f32, np.float32(np.inf)), np.nextafter(f32, np.float32(-np.inf)), wide])
    assert np.array_equal(oc.encode_e4m3(allv.astype(np.float64)), torch_e4m3(allv))


def test_encoder_hand_cases():
    with open(os.path.join(GOLDEN, "e4m3_encode.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        assert oc.encode_e4m3(np.array([c["value"]]))[0] == int(c["code"], 16), c


def test_group_quotient_is_rounded_to_fp32_before_the_code():
    """A hand-worked group where the fp32 quotient sits exactly on an e4m3 midpoint
    (ties to the even code) while the exact quotient lies just above it
    (tests/golden/e4m3_fp32_quotient.json holds the derivation)."""
    with open(os.path.join(GOLDEN, "e4m3_fp32_quotient.json")) as f:
        g = json.load(f)
    vals = np.array([int(b, 16) for b in g["values_f32_bits"]], dtype=np.uint32).view(np.float32)
    x = np.zeros(g["group"], dtype=np.float32)
    x[: vals.shape[0]] = vals
    codes, scale = oc.quantize_groups(x, g["group"])
    assert int(np.asarray(scale, dtype=np.float32).reshape(-1).view(np.uint32)[0]) == int(g["expected_scale_f32_bits"], 16)
    assert codes[: vals.shape[0]].tolist() == [int(c, 16) for c in g["expected_codes"]]
    assert np.all(codes[vals.shape[0]:] == 0)
    # the premise: rounding the exact quotient would pick the other code
    exact = Fraction(float(vals[1])) / Fraction(float(np.float32(vals[0]) / np.float32(448.0)))
    lo, hi = Fraction(1), Fraction(9, 8)
    assert (lo + hi) / 2 < exact < hi and int(g["code_if_rounded_exactly"], 16) == 0x39


def test_encoder_round_trip_is_nearest():
    rng = np.random.default_rng(3)
    v = rng.uniform(-448, 448, 5000)
    codes = oc.encode_e4m3(v)
    back = decode_e4m3(codes)
    finite = E4M3_TABLE[np.isfinite(E4M3_TABLE)]
    best = np.abs(v[:, None] - finite[None, :]).min(axis=1)
    assert np.allclose(np.abs(back - v), best, rtol=0, atol=1e-12)


def _one_token_geometry(pos):
    """One request whose last (new) token sits at `pos`; block table [2, 0, 1]."""
    bt = np.array([[2, 0, 1]], dtype=np.int32)
    return np.array([pos + 1], dtype=np.int32), np.array([1], dtype=np.int32), bt


def test_hand_worked_e4m3_record():
    with open(os.path.join(GOLDEN, "cache_record_hand.json")) as f:
        g = json.load(f)
    x = np.zeros(576, dtype=np.float32)
    for k, v in g["latent_nonzero"].items():
        x[int(k)] = v
    x[512:] = np.where(np.arange(64) % 2 == 0, 1.0, -2.0)
    bits = (x.view(np.uint32) >> 16).astype(np.uint16)          # exact in bf16
    assert np.array_equal(decode_bf16(bits), x.astype(np.float64))
    seq, nq, bt = _one_token_geometry(pos=70)   # logical page 1 -> physical page bt[0][1] = 0, slot 6
    kv = np.zeros((3, 64 * 656), dtype=np.uint8)
    out, _, _ = oc.cache_append(kv, "e4m3", bits[None], None, None, "e4m3", None, seq, nq, bt)
    codes, sc_bytes, rope_bytes = _record(out, 0 * 64 + 70 % 64)
    for k, code in g["expected_codes"].items():
        assert codes[int(k)] == int(code, 16), (k, hex(codes[int(k)]))
    scales = decode_f32le(sc_bytes)
    for c, s in enumerate(g["expected_scales_exact"]):
        if s is None:
            assert scales[c] == float(np.float32(3.0) / np.float32(448.0))
        else:
            assert scales[c] == s
    assert np.array_equal(decode_bf16(rope_bytes.view(np.uint16)), x[512:].astype(np.float64))
    # every other byte is untouched
    rest = out.copy()
    page = rest.reshape(-1, 64 * 656)[0]
    page[6 * 512:7 * 512] = 0
    page[32768 + 6 * 16:32768 + 7 * 16] = 0
    page[33792 + 6 * 128:33792 + 7 * 128] = 0
    assert not rest.any()


def _random_append_case(rng, kv_dtype, qk_dtype):
    seq = np.array([130, 64, 200], dtype=np.int32)
    nq = np.array([2, 1, 4], dtype=np.int32)
    P = 12
    bt = rng.permutation(P)[:12].reshape(3, 4).astype(np.int32)
    T = int(nq.sum())
    x = (rng.standard_normal((T, 576)) * 0.5).astype(np.float32)
    x[0, 128:256] = 0.0                                           # an all-zero group
    x[1, :128] *= np.float32(2.0 ** -20)                          # tiny values
    bits = (x.view(np.uint32) >> 16).astype(np.uint16)
    k = rng.standard_normal((T, 128)).astype(np.float32)
    kbits = (k.view(np.uint32) >> 16).astype(np.uint16)
    if kv_dtype == "bf16":
        kv = rng.integers(0, 2 ** 16, size=(P, 64, 576), dtype=np.uint16)
    else:
        kv = rng.integers(0, 256, size=(P, 64 * 656), dtype=np.uint8)
    if qk_dtype == "bf16":
        ik = rng.integers(0, 2 ** 16, size=(P, 64, 128), dtype=np.uint16)
        isc = None
    else:
        ik = rng.integers(0, 256, size=(P, 64, 128), dtype=np.uint8)
        isc = rng.standard_normal((P, 64)).astype(np.float32)
    return seq, nq, bt, bits, kbits, kv, ik, isc


@pytest.mark.parametrize("kv_dtype,qk_dtype", [("bf16", "e4m3"), ("e4m3", "e4m3"), ("bf16", "bf16")])
def test_append_rows_round_trip_and_untouched_rows(kv_dtype, qk_dtype):
    rng = np.random.default_rng(11)
    seq, nq, bt, bits, kbits, kv, ik, isc = _random_append_case(rng, kv_dtype, qk_dtype)
    out, ok_, os_ = oc.cache_append(kv, kv_dtype, bits, ik, isc, qk_dtype, kbits, seq, nq, bt)
    # rows follow the attention's position rule: query j of request b is at L_b - n_b + j
    req, pos = oracle.query_positions(seq, nq)
    rows = np.array([bt[b][p // 64] * 64 + p % 64 for b, p in zip(req, pos)])
    assert np.array_equal(rows, oc.token_rows(seq, nq, bt))
    touched = np.zeros(out.shape[0] * 64, dtype=bool)
    touched[rows] = True
    if kv_dtype == "bf16":
        assert np.array_equal(out.reshape(-1, 576)[~touched], kv.reshape(-1, 576)[~touched])
    else:
        # every byte outside the new tokens' codes, scales and RoPE values is unchanged
        mask = np.ones(out.size, dtype=bool)
        for r in rows:
            for field in _record(np.arange(out.size).reshape(out.shape), r):
                mask[field] = False
        assert np.array_equal(out.reshape(-1)[mask], kv.reshape(-1)[mask])
    assert np.array_equal(ok_.reshape(-1, 128)[~touched], ik.reshape(-1, 128)[~touched])
    x = decode_bf16(bits)
    for t, r in enumerate(rows):
        if kv_dtype == "bf16":
            assert np.array_equal(out.reshape(-1, 576)[r], bits[t])
        else:
            codes, sc_bytes, rope_bytes = _record(out, r)
            scales = decode_f32le(sc_bytes)
            deq = decode_e4m3(codes) * np.repeat(scales, 128)
            amax = np.abs(x[t, :512]).reshape(4, 128).max(axis=1)
            # scale = amax/448 in fp32; round trip within half an e4m3 step (2^-4 relative,
            # 2^-10 * scale absolute in the subnormal range)
            assert np.all(scales[amax > 0] == (amax[amax > 0].astype(np.float32) / np.float32(448)))
            assert np.all(scales[amax == 0] == 1.0)
            bound = np.abs(x[t, :512]) * 2.0 ** -4 + np.repeat(scales, 128) * 2.0 ** -10
            assert np.all(np.abs(deq - x[t, :512]) <= bound * (1 + 1e-6))
            assert np.array_equal(rope_bytes.view(np.uint16), bits[t, 512:])
        krow = ok_.reshape(-1, 128)[r]
        if qk_dtype == "bf16":
            assert np.array_equal(krow, kbits[t])
        else:
            kx = decode_bf16(kbits[t])
            s = os_.reshape(-1)[r]
            assert s == np.float32(np.abs(kx).max()) / np.float32(448)
            assert np.all(np.abs(decode_e4m3(krow) * s - kx) <= np.abs(kx) * 2.0 ** -4 + s * 2.0 ** -10 + 1e-12)


def test_append_is_idempotent_and_bf16_rope_passes_through():
    rng = np.random.default_rng(5)
    seq, nq, bt, bits, kbits, kv, ik, isc = _random_append_case(rng, "e4m3", "e4m3")
    a = oc.cache_append(kv, "e4m3", bits, ik, isc, "e4m3", kbits, seq, nq, bt)
    b = oc.cache_append(a[0], "e4m3", bits, a[1], a[2], "e4m3", kbits, seq, nq, bt)
    for u, v in zip(a, b):
        assert np.array_equal(u, v)


def test_int8_encoder_hand_cases_and_rint():
    with open(os.path.join(GOLDEN, "int8_encode.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        assert oc.encode_int8(np.array([c["value"]]))[0] == int(c["byte"], 16), c
    rng = np.random.default_rng(9)
    v = np.concatenate([rng.uniform(-140, 140, 20000), np.arange(-130, 130) + 0.5])
    ref = np.clip(np.rint(v), -127, 127).astype(np.int8).view(np.uint8)   # library round-half-even
    assert np.array_equal(oc.encode_int8(v), ref)


def test_int8_append_round_trip_within_half_a_step():
    rng = np.random.default_rng(12)
    seq, nq, bt, bits, kbits, kv, ik, isc = _random_append_case(rng, "e4m3", "e4m3")
    out, _, _ = oc.cache_append(kv, "int8", bits, None, None, "e4m3", None, seq, nq, bt)
    rows = oc.token_rows(seq, nq, bt)
    x = decode_bf16(bits)
    for t, r in enumerate(rows):
        codes, sc_bytes, rope_bytes = _record(out, r)
        scales = decode_f32le(sc_bytes)
        amax = np.abs(x[t, :512]).reshape(4, 128).max(axis=1)
        assert np.all(scales[amax > 0] == amax[amax > 0].astype(np.float32) / np.float32(127))
        deq = codes.view(np.int8).astype(np.float64) * np.repeat(scales, 128)
        assert np.all(np.abs(deq - x[t, :512]) <= np.repeat(scales, 128) * (0.5 + 1e-6))
        assert np.array_equal(rope_bytes.view(np.uint16), bits[t, 512:])
