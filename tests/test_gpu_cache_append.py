"""dsa_cache_append on the GPU against the oracle's cache append: bit-exact cache bytes
(codes, scales, copied bf16 rows) for every latent/index dtype pair, with exact ties,
subnormal codes, all-zero groups, negative zeros and saturating quotients; untouched
rows at full decode size; a prefill-sized append; out-of-range page ids skipped and
reported."""
import numpy as np
import pytest
import torch

from oracle import cache as oc
from oracle.fp8 import E4M3_TABLE
from dsa_sparse_attention_02_gb300 import _lib, inputs
from gpu_helpers import DEV

pytestmark = pytest.mark.gpu

DT = {"bf16": _lib.DSA_BF16, "e4m3": _lib.DSA_E4M3, "int8": _lib.DSA_I8}


def _bits(x32):
    return (np.ascontiguousarray(x32, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)


def _special_rows(rng, T):
    """New-token latent rows (fp32, exact in bf16) that exercise the encoder's edges."""
    x = (rng.standard_normal((T, 576)) * 0.5).astype(np.float32)
    vals = E4M3_TABLE[:0x7F]
    mids = ((vals[:-1] + vals[1:]) / 2).astype(np.float32)
    # group 0 of token 0: amax 448 -> scale 1, then exact midpoints (ties) and values
    x[0, :128] = 0.0
    x[0, 0] = 448.0
    x[0, 1:1 + 100] = (mids[-100:] * np.where(np.arange(100) % 2, 1, -1)).astype(np.float32) / 4
    # group 1 of token 0: all zero; group 2: negative zeros and tiny values
    x[0, 128:256] = 0.0
    x[0, 256:384] = -0.0
    x[0, 256:260] = np.array([1e-3, -2e-3, 3e-6, 0.0], dtype=np.float32)
    # token 1: a group whose amax is not a power-of-two multiple of 448 (quotients near 448)
    x[1, :128] = np.linspace(-3.0, 3.0, 128, dtype=np.float32)
    # token 2: a tiny group (amax ~1e-20) -> scales in the fp32 subnormal-free range
    if T > 2:
        x[2, 128:256] *= np.float32(1e-20)
    return _bits(x)


def _case(rng, kv_dtype, qk_dtype):
    seq = np.array([130, 64, 200, 1], dtype=np.int32)
    nq = np.array([2, 1, 4, 1], dtype=np.int32)
    P = 16
    bt = rng.permutation(P)[:16].reshape(4, 4).astype(np.int32)
    T = int(nq.sum())
    bits = _special_rows(rng, T)
    kx = rng.standard_normal((T, 128)).astype(np.float32)
    kx[0] = 0.0
    kx[1, :4] = [448.0, 1.0625 * 4, -1.1875 * 4, -0.0]
    kbits = _bits(kx)
    kv = (rng.integers(0, 2 ** 16, size=(P, 64, 576), dtype=np.uint16) if kv_dtype == "bf16"
          else rng.integers(0, 256, size=(P, 64 * 656), dtype=np.uint8))
    if qk_dtype == "bf16":
        ik = rng.integers(0, 2 ** 16, size=(P, 64, 128), dtype=np.uint16)
        isc = None
    else:
        ik = rng.integers(0, 256, size=(P, 64, 128), dtype=np.uint8)
        isc = rng.standard_normal((P, 64)).astype(np.float32)
    return seq, nq, bt, bits, kbits, kv, ik, isc


def _geometry(seq, nq, bt, P):
    cu = np.zeros(len(seq) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(nq)
    tens = [torch.from_numpy(a).to(DEV) for a in (seq, cu, np.ascontiguousarray(bt))]
    g = _lib.Geometry(tens[0], tens[1], tens[2], num_pages=P, max_seq_len=int(seq.max()), T=int(nq.sum()))
    g._keep = tens
    return g


def _dev(a):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(DEV)
    return torch.from_numpy(a).to(DEV)


def _host(t, dtype):
    a = t.cpu().numpy()
    return a.view(dtype) if a.dtype != dtype else a


@pytest.mark.parametrize("kv_dtype,qk_dtype", [("bf16", "e4m3"), ("e4m3", "e4m3"), ("e4m3", "bf16"), ("bf16", "bf16"),
                                               ("int8", "e4m3"), ("int8", "bf16")])
def test_append_bit_exact_against_oracle(kv_dtype, qk_dtype):
    rng = np.random.default_rng(21)
    seq, nq, bt, bits, kbits, kv, ik, isc = _case(rng, kv_dtype, qk_dtype)
    g = _geometry(seq, nq, bt, kv.shape[0])
    d_kv, d_ik = _dev(kv), _dev(ik)
    d_isc = None if isc is None else _dev(isc)
    ws = _lib.workspace(_lib.dsa_cache_append_workspace_size(g), DEV)
    _lib.dsa_cache_append(g, DT[kv_dtype], _dev(bits), d_kv, DT[qk_dtype], _dev(kbits), d_ik, d_isc, ws)
    assert _lib.dsa_get_error(ws) == 0
    ref_kv, ref_ik, ref_isc = oc.cache_append(kv, kv_dtype, bits, ik, isc, qk_dtype, kbits, seq, nq, bt)
    assert np.array_equal(_host(d_kv, kv.dtype), ref_kv)
    assert np.array_equal(_host(d_ik, ik.dtype), ref_ik)
    if isc is not None:
        assert np.array_equal(_host(d_isc, np.float32).view(np.uint32), ref_isc.view(np.uint32))


def test_append_at_decode_size_touches_only_the_new_rows():
    wl = inputs.make_config("decode")
    rng = np.random.default_rng(22)
    bits = _bits((rng.standard_normal((wl.T, 576)) * 0.5).astype(np.float32))
    kbits = _bits(rng.standard_normal((wl.T, 128)).astype(np.float32))
    g = _geometry(wl.seq_lens.astype(np.int32), wl.n_q.astype(np.int32), wl.block_table, wl.num_pages)
    kv = _dev(wl.layers[0].kv)
    ik, isc = _dev(wl.idx_k), _dev(wl.idx_k_scale)
    kv0, ik0, isc0 = kv.clone(), ik.clone(), isc.clone()
    ws = _lib.workspace(256, DEV)
    _lib.dsa_cache_append(g, _lib.DSA_BF16, _dev(bits), kv, _lib.DSA_E4M3, _dev(kbits), ik, isc, ws)
    assert _lib.dsa_get_error(ws) == 0
    rows = torch.from_numpy(oc.token_rows(wl.seq_lens, wl.n_q, wl.block_table)).to(DEV)
    touched = torch.zeros(kv.shape[0] * 64, dtype=torch.bool, device=DEV)
    touched[rows] = True
    assert torch.equal(kv.view(-1, 576)[~touched], kv0.view(-1, 576)[~touched])
    assert torch.equal(ik.view(-1, 128)[~touched], ik0.view(-1, 128)[~touched])
    assert torch.equal(isc.view(-1)[~touched], isc0.view(-1)[~touched])
    # the new rows equal the oracle's encoding of the same tokens
    r = rows.cpu().numpy()
    assert np.array_equal(_host(kv.view(-1, 576)[rows], np.uint16), bits)
    codes, scales = oc.quantize_groups(oc.bf16_bits_to_f32(kbits), 128)
    assert np.array_equal(ik.view(-1, 128)[rows].cpu().numpy(), codes)
    assert np.array_equal(isc.view(-1)[rows].cpu().numpy(), scales[:, 0])
    assert len(np.unique(r)) == wl.T


def test_append_prefill_chunk_e4m3():
    rng = np.random.default_rng(23)
    L, n = 4096, 2048
    seq, nq = np.array([L], dtype=np.int32), np.array([n], dtype=np.int32)
    P = L // 64 + 3
    bt = rng.permutation(P)[: L // 64].reshape(1, -1).astype(np.int32)
    bits = _bits((rng.standard_normal((n, 576)) * 0.5).astype(np.float32))
    kbits = _bits(rng.standard_normal((n, 128)).astype(np.float32))
    kv = np.zeros((P, 64 * 656), dtype=np.uint8)
    ik = np.zeros((P, 64, 128), dtype=np.uint8)
    isc = np.zeros((P, 64), dtype=np.float32)
    g = _geometry(seq, nq, bt, P)
    d_kv, d_ik, d_isc = _dev(kv), _dev(ik), _dev(isc)
    ws = _lib.workspace(256, DEV)
    _lib.dsa_cache_append(g, _lib.DSA_E4M3, _dev(bits), d_kv, _lib.DSA_E4M3, _dev(kbits), d_ik, d_isc, ws)
    assert _lib.dsa_get_error(ws) == 0
    ref_kv, ref_ik, ref_isc = oc.cache_append(kv, "e4m3", bits, ik, isc, "e4m3", kbits, seq, nq, bt)
    assert np.array_equal(d_kv.cpu().numpy(), ref_kv)
    assert np.array_equal(d_ik.cpu().numpy(), ref_ik)
    assert np.array_equal(d_isc.cpu().numpy().view(np.uint32), ref_isc.view(np.uint32))


def test_append_skips_and_reports_out_of_range_pages():
    rng = np.random.default_rng(24)
    seq, nq, bt, bits, kbits, kv, ik, isc = _case(rng, "bf16", "e4m3")
    bad = bt.copy()
    bad[0, 2] = 10_000                       # request 0's new tokens (positions 128, 129) land here
    g = _geometry(seq, nq, bad, kv.shape[0])
    d_kv, d_ik, d_isc = _dev(kv), _dev(ik), _dev(isc)
    ws = _lib.workspace(256, DEV)
    _lib.dsa_cache_append(g, _lib.DSA_BF16, _dev(bits), d_kv, _lib.DSA_E4M3, _dev(kbits), d_ik, d_isc, ws)
    assert _lib.dsa_get_error(ws) == _lib.DSA_ERR_BAD_INDEX
    # the other requests' tokens are written as the oracle writes them
    keep_seq, keep_nq = seq[1:], nq[1:]
    ref_kv, _, _ = oc.cache_append(kv, "bf16", bits[2:], ik, isc, "e4m3", kbits[2:], keep_seq, keep_nq, bt[1:])
    assert np.array_equal(_host(d_kv, np.uint16), ref_kv)
