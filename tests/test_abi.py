"""The C-ABI library loads and exports every function include/dsa.h declares; host-side
argument validation answers before anything reaches a GPU (no compute calls here)."""
import ctypes as C
import os
import re

import pytest

import dsa_sparse_attention_02_gb300 as dsa
from dsa_sparse_attention_02_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dsa.h")


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dsa_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(_lib.LIB_PATH):
        from dsa_sparse_attention_02_gb300 import build
        build.build()
    return _lib.load()


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert len(names) >= 12
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(_lib.EXPORTED) == names


def test_abi_version_and_status_strings(lib):
    assert dsa.dsa_abi_version() == 1
    assert _lib.status_string(0) == "ok"
    assert "invalid" in _lib.status_string(1)


def _geom(**kw):
    g = dict(B=1, T=1, max_seq_len=128, num_pages=4, page_size=64, bt_stride=2,
             seq_lens=1, cu_q=1, block_table=1)       # dummy non-null pointers: never dereferenced
    g.update(kw)
    return _lib.dsa_geom_t(g["B"], g["T"], g["max_seq_len"], g["num_pages"], g["page_size"],
                           g["bt_stride"], g["seq_lens"], g["cu_q"], g["block_table"])


def _topk(lib, g, k=8, scores=16, idx=16, ws=256, ws_bytes=1 << 20):
    return lib.dsa_topk(C.byref(g), scores, g.max_seq_len, k, idx, ws, ws_bytes, None)


def test_host_validation(lib):
    assert lib.dsa_topk(None, 16, 128, 8, 16, 256, 1 << 20, None) == _lib.DSA_ERR_INVALID_ARG
    assert _topk(lib, _geom(page_size=32)) == _lib.DSA_ERR_UNSUPPORTED
    assert _topk(lib, _geom(), k=0) == _lib.DSA_ERR_INVALID_ARG
    assert _topk(lib, _geom(), k=20000) == _lib.DSA_ERR_INVALID_ARG
    assert _topk(lib, _geom(bt_stride=1)) == _lib.DSA_ERR_INVALID_ARG
    assert _topk(lib, _geom(), scores=None) == _lib.DSA_ERR_INVALID_ARG
    assert _topk(lib, _geom(), ws=None) == _lib.DSA_ERR_WORKSPACE
    assert _topk(lib, _geom(), ws=260) == _lib.DSA_ERR_WORKSPACE          # misaligned
    # rows longer than one top-k pass need k <= 8192 (merges of at least two lists);
    # any length works below that (checked with zero queries: nothing is launched)
    assert _topk(lib, _geom(max_seq_len=200000, bt_stride=4000), k=8193) == _lib.DSA_ERR_UNSUPPORTED
    for L in (16385, 200000, 1 << 20, 1 << 28):
        assert _topk(lib, _geom(T=0, max_seq_len=L, bt_stride=(L + 63) // 64), k=8192) == _lib.DSA_OK
    # zero work: OK without touching the device
    assert _topk(lib, _geom(T=0)) == _lib.DSA_OK
    g = _geom()
    # indexer: Hi out of range, bf16 with a scale pointer, misaligned cache
    for hi in (0, -1, 65, 128):
        assert lib.dsa_indexer_scores(C.byref(g), _lib.DSA_E4M3, hi, 16, 16, 16, 16, 16, 16, 128, 256,
                                      4096, None) == _lib.DSA_ERR_INVALID_ARG, hi
    assert lib.dsa_indexer_scores(C.byref(g), _lib.DSA_BF16, 4, 16, 16, 16, 16, None, 16, 128, 256,
                                  4096, None) == _lib.DSA_ERR_INVALID_ARG
    assert lib.dsa_indexer_scores(C.byref(g), _lib.DSA_E4M3, 4, 16, 16, 16, 24, 16, 16, 128, 256,
                                  4096, None) == _lib.DSA_ERR_INVALID_ARG
    assert lib.dsa_indexer_scores(C.byref(g), _lib.DSA_E4M3, 4, 16, 16, 16, 16, 16, 16, 64, 256,
                                  4096, None) == _lib.DSA_ERR_INVALID_ARG   # stride < max_seq_len
    # attention: unsupported head count, bad dtype, non-finite scale
    assert lib.dsa_sparse_mla_attend(C.byref(g), _lib.DSA_BF16, 24, 16, 16, 16, 64, 0.1, 16, None,
                                     256, 1 << 24, None) == _lib.DSA_ERR_INVALID_ARG
    assert lib.dsa_sparse_mla_attend(C.byref(g), 7, 16, 16, 16, 16, 64, 0.1, 16, None,
                                     256, 1 << 24, None) == _lib.DSA_ERR_INVALID_ARG
    assert lib.dsa_sparse_mla_attend(C.byref(g), _lib.DSA_BF16, 16, 16, 16, 16, 64, float("inf"),
                                     16, None, 256, 1 << 24, None) == _lib.DSA_ERR_INVALID_ARG
    # cache append: bad dtypes, e4m3 keys without scales, bf16 keys with scales,
    # misaligned buffers, no workspace; zero tokens is a no-op
    ca = lib.dsa_cache_append
    assert ca(C.byref(g), 9, 16, 16, _lib.DSA_E4M3, None, None, None, 256, 256, None) == _lib.DSA_ERR_INVALID_ARG
    assert ca(C.byref(g), _lib.DSA_BF16, 16, 16, 9, 16, 16, 16, 256, 256, None) == _lib.DSA_ERR_INVALID_ARG
    assert ca(C.byref(g), _lib.DSA_BF16, 16, 16, _lib.DSA_E4M3, 16, 16, None, 256, 256, None) == _lib.DSA_ERR_INVALID_ARG
    assert ca(C.byref(g), _lib.DSA_BF16, 16, 16, _lib.DSA_BF16, 16, 16, 16, 256, 256, None) == _lib.DSA_ERR_INVALID_ARG
    assert ca(C.byref(g), _lib.DSA_BF16, 24, 16, _lib.DSA_E4M3, None, None, None, 256, 256, None) == _lib.DSA_ERR_INVALID_ARG
    assert ca(C.byref(g), _lib.DSA_BF16, 16, 16, _lib.DSA_E4M3, None, None, None, None, 0, None) == _lib.DSA_ERR_WORKSPACE
    g0 = _geom(T=0)
    assert ca(C.byref(g0), _lib.DSA_BF16, None, None, _lib.DSA_E4M3, None, None, None, 256, 256, None) == _lib.DSA_OK
    assert lib.dsa_cache_append_workspace_size(C.byref(g)) == 256
    assert lib.dsa_get_error(None, None) == _lib.DSA_ERR_INVALID_ARG


def test_indexer_prepare_rejects_bad_arguments_before_launch(lib):
    g = _geom(T=4)
    pr = lib.dsa_indexer_prepare
    ok = dict(Hi=64, rd=64, q=16, k=16, cs=16, sn=16, gm=None, bt=None, eps=1e-6, qo=16, qs=16, kc=16, ks=16,
              ws=256, wb=256)

    def call(geom=g, **kw):
        a = dict(ok, **kw)
        return pr(C.byref(geom), a["Hi"], a["rd"], a["q"], a["k"], a["cs"], a["sn"], a["gm"], a["bt"], a["eps"],
                  a["qo"], a["qs"], a["kc"], a["ks"], a["ws"], a["wb"], None)

    for bad in (dict(Hi=0), dict(Hi=129), dict(rd=0), dict(rd=12), dict(rd=136), dict(eps=-1.0),
                dict(eps=float("nan")), dict(kc=None), dict(ks=None), dict(k=24), dict(gm=8),
                dict(q=None), dict(cs=None), dict(qs=None), dict(q=24), dict(sn=20)):
        assert call(**bad) == _lib.DSA_ERR_INVALID_ARG, bad
    assert call(ws=None, wb=0) == _lib.DSA_ERR_WORKSPACE
    assert call(ws=264) == _lib.DSA_ERR_WORKSPACE                   # not 256-byte aligned
    assert call(geom=_geom(T=0), q=None, qo=None, qs=None, cs=None, sn=None) == _lib.DSA_OK
    assert lib.dsa_indexer_prepare_workspace_size(C.byref(g)) == 256


def test_workspace_sizes_are_consistent(lib):
    g = _geom(T=64, B=64, max_seq_len=131072, bt_stride=2048)
    assert lib.dsa_topk_workspace_size(C.byref(g), 2048) >= 256 + 64 * 8 * 2048 * 8
    g2 = _geom(T=64, B=64, max_seq_len=8192, bt_stride=128)
    assert lib.dsa_topk_workspace_size(C.byref(g2), 2048) == 256
    a = _lib.dsa_step_args_t()
    a.geom = g2
    a.topk = 2048
    a.H = 16
    base = lib.dsa_decode_step_workspace_size(C.byref(a))
    assert base >= 256 + 64 * 8192 * 4 + 64 * 2048 * 4
    a.reuse_idx = 16
    assert lib.dsa_decode_step_workspace_size(C.byref(a)) < base


def test_histogram_step_workspace_adds_the_histograms(lib):
    """dsa_decode_step_hist asks for the default step's workspace plus 8 KB of first-digit
    histogram per query and 16384-position chunk of max_seq_len (the region at its end);
    a shared layer's call (reuse_idx) counts nothing and asks for the default size."""
    a = _lib.dsa_step_args_t()
    a.topk = 2048
    a.H = 16
    a.Hi = 64
    for T, L, chunks in ((64, 8192, 1), (8, 131072, 8), (2, 16384, 1), (2, 16385, 2)):
        a.geom = _geom(T=T, B=T, max_seq_len=L, bt_stride=-(-L // 64))
        a.reuse_idx = None
        base = lib.dsa_decode_step_workspace_size(C.byref(a))
        assert lib.dsa_decode_step_hist_workspace_size(C.byref(a)) == base + T * chunks * 8192
        a.reuse_idx = 16
        assert lib.dsa_decode_step_hist_workspace_size(C.byref(a)) == lib.dsa_decode_step_workspace_size(C.byref(a))
    # the same argument checks as the default step, before anything is enqueued
    a.reuse_idx = None
    a.topk = 0
    assert lib.dsa_decode_step_hist(C.byref(a), 256, 1 << 30, None) == _lib.DSA_ERR_INVALID_ARG


def test_bounded_step_budget_floor_and_workspace_sizes(lib):
    a = _lib.dsa_step_args_t()
    a.geom = _geom(T=64, B=64, max_seq_len=8192, bt_stride=128)
    a.topk = 2048
    a.H = 16
    a.Hi = 64
    row = 8192 * 4
    # below one query's score row: rejected before anything is enqueued
    assert lib.dsa_decode_step_bounded(C.byref(a), row - 1, 256, 1 << 30, None) == _lib.DSA_ERR_INVALID_ARG
    full = lib.dsa_decode_step_workspace_size(C.byref(a))
    assert lib.dsa_decode_step_bounded_workspace_size(C.byref(a), 64 * row) == full   # all rows fit: no ranges
    one = lib.dsa_decode_step_bounded_workspace_size(C.byref(a), row)
    assert one < full - 62 * row                               # 63 fewer score rows, plus the range geometry
    assert lib.dsa_decode_step_bounded_workspace_size(C.byref(a), 8 * row) > one


# ----------------------------------------------------------------------------- header vs binding

_SCALAR = {"int32_t": C.c_int32, "uint32_t": C.c_uint32, "int64_t": C.c_int64, "size_t": C.c_size_t, "float": C.c_float,
           "dsa_dtype_t": C.c_int, "dsa_status_t": C.c_int, "int": C.c_int}


def _header_text():
    return re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)


def _ctype_of(decl):
    """ctypes type of one C declaration's type part ('const float*', 'int32_t', ...)."""
    decl = decl.replace("const", "").strip()
    if "*" in decl:
        return "pointer"
    return _SCALAR[decl.split()[0]]


def _prototypes():
    protos = {}
    for ret, name, params in re.findall(r"([A-Za-z_][\w\s\*]*?)\b(dsa_\w+)\s*\(([^)]*)\)\s*;", _header_text()):
        params = params.strip()
        plist = [] if params in ("", "void") else [p.strip() for p in params.split(",")]
        types = []
        for p in plist:
            m = re.match(r"(.*?)(\w+)$", p)                 # drop the parameter name
            types.append(_ctype_of(m.group(1) if m and m.group(1).strip() else p))
        protos[name] = (ret.strip(), types)
    return protos


def _is_pointer_type(t):
    return t in (C.c_void_p, C.c_char_p) or (isinstance(t, type) and issubclass(t, C._Pointer))


def test_binding_signatures_match_the_header(lib):
    protos = _prototypes()
    assert sorted(protos) == sorted(_lib.EXPORTED)
    for name, (ret, params) in protos.items():
        fn = getattr(lib, name)
        assert fn.argtypes is not None and len(fn.argtypes) == len(params), (name, params, fn.argtypes)
        for i, (want, got) in enumerate(zip(params, fn.argtypes)):
            if want == "pointer":
                assert _is_pointer_type(got), (name, i, got)
            else:
                assert got is want, (name, i, want, got)
        want_ret = "pointer" if "*" in ret else _SCALAR[ret.replace("const", "").strip()]
        if want_ret == "pointer":
            assert fn.restype is C.c_char_p, name
        else:
            assert fn.restype is want_ret, (name, ret, fn.restype)


def _header_struct(name):
    m = re.search(r"typedef struct\s*\{([^{}]*)\}\s*" + name + r"\s*;", _header_text())
    fields = []
    for decl in m.group(1).split(";"):
        decl = " ".join(decl.split())
        if not decl:
            continue
        fm = re.match(r"(.*?)(\w+)$", decl)
        fields.append((fm.group(2), fm.group(1).strip()))
    return fields


@pytest.mark.parametrize("name", ["dsa_geom_t", "dsa_step_args_t"])
def test_binding_structs_match_the_header(name):
    fields = _header_struct(name)
    ct = getattr(_lib, name)
    assert [f for f, _ in fields] == [f for f, _ in ct._fields_]
    for (fname, ctype), (_, got) in zip(fields, ct._fields_):
        if ctype in ("dsa_geom_t",):
            assert got is _lib.dsa_geom_t, fname
        elif "*" in ctype:
            assert got is C.c_void_p, fname
        else:
            assert got is _SCALAR[ctype.replace("const", "").strip()], (fname, ctype, got)


def test_binding_refuses_host_tensors_for_device_arguments(lib):
    """Host tensors are refused by the binding before any call reaches the library,
    so a host address never reaches a kernel (dsa_stage_copy takes host memory, and the
    attention's outputs may be page-locked host memory; the C side checks both). A
    pageable host tensor is refused for an output too."""
    import torch
    seq = torch.tensor([64], dtype=torch.int32)
    cu = torch.tensor([0, 1], dtype=torch.int32)
    bt = torch.zeros(1, 1, dtype=torch.int32)
    with pytest.raises(TypeError, match="CUDA tensor"):
        _lib.Geometry(seq, cu, bt, num_pages=1, max_seq_len=64, T=1)
    with pytest.raises(TypeError, match="CUDA tensor"):
        _lib.dsa_decode_step(_lib.dsa_step_args_t(), torch.zeros(256, dtype=torch.uint8))
    with pytest.raises(TypeError, match="CUDA tensor"):
        _lib.dsa_get_error(torch.zeros(256, dtype=torch.uint8))
    with pytest.raises(TypeError, match="CUDA tensor"):
        _lib._dptr(bytearray(16))
    assert _lib._dptr(None) is None
    with pytest.raises(TypeError, match="CUDA tensor"):
        _lib._optr(torch.zeros(16))                      # pageable
    assert _lib._optr(None) is None


def test_wait_probe_validates_before_launch(lib):
    assert lib.dsa_wait_probe(256, 256, 0, None) == _lib.DSA_ERR_INVALID_ARG
    assert lib.dsa_wait_probe(256, 256, 1000001, None) == _lib.DSA_ERR_INVALID_ARG
    assert lib.dsa_wait_probe(None, 256, 1000, None) == _lib.DSA_ERR_WORKSPACE
    assert lib.dsa_wait_probe(260, 256, 1000, None) == _lib.DSA_ERR_WORKSPACE      # misaligned
    assert lib.dsa_wait_probe(256, 128, 1000, None) == _lib.DSA_ERR_WORKSPACE      # too small


def test_indexer_accepts_any_head_count_up_to_64(lib):
    # zero queries: the arguments are checked, nothing is launched
    g = _geom(T=0)
    for hi in (1, 2, 3, 5, 17, 63, 64):
        assert lib.dsa_indexer_scores(C.byref(g), _lib.DSA_E4M3, hi, 16, 16, 16, 16, 16, 16, 128, 256,
                                      4096, None) == _lib.DSA_OK, hi
        assert lib.dsa_indexer_scores(C.byref(g), _lib.DSA_BF16, hi, 16, None, 16, 16, None, 16, 128, 256,
                                      4096, None) == _lib.DSA_OK, hi
    # more requests than one launch holds are accepted too
    gb = _geom(T=0, B=5000)
    assert lib.dsa_indexer_scores(C.byref(gb), _lib.DSA_E4M3, 64, 16, 16, 16, 16, 16, 16, 128, 256,
                                  4096, None) == _lib.DSA_OK


_ATTEND_BAD = [
    dict(H=24), dict(H=0), dict(H=129), dict(kv=7), dict(k=0), dict(k=16385), dict(scale=float("inf")),
    dict(scale=float("nan")), dict(q=None), dict(kvp=None), dict(idx=None), dict(out=None), dict(q=24),
    dict(kvp=40), dict(geom=dict(page_size=32)), dict(geom=dict(bt_stride=1)),
    dict(geom=dict(num_pages=(1 << 25) + 1)), dict(geom=dict(max_seq_len=0)), dict(geom=dict(B=0)),
]


@pytest.mark.parametrize("bad", _ATTEND_BAD, ids=[str(b) for b in _ATTEND_BAD])
def test_static_entry_point_refuses_what_the_workspace_entry_point_refuses(lib, bad):
    a = dict(H=16, kv=_lib.DSA_BF16, k=64, scale=0.1, q=16, kvp=16, idx=16, out=16, geom={})
    a.update(bad)
    g = _geom(**a["geom"])
    ws = lib.dsa_sparse_mla_attend(C.byref(g), a["kv"], a["H"], a["q"], a["kvp"], a["idx"], a["k"], a["scale"],
                                   a["out"], None, 256, 1 << 30, None)
    st = lib.dsa_sparse_mla_attend_static(C.byref(g), a["kv"], a["H"], a["q"], a["kvp"], a["idx"], a["k"],
                                          a["scale"], a["out"], None, 64, None)
    assert ws in (_lib.DSA_ERR_INVALID_ARG, _lib.DSA_ERR_UNSUPPORTED), ws
    assert st == ws


def test_static_entry_point_requires_an_error_word(lib):
    g = _geom()
    for err in (None, 66):        # missing, or not 4-byte aligned
        assert lib.dsa_sparse_mla_attend_static(C.byref(g), _lib.DSA_BF16, 16, 16, 16, 16, 64, 0.1, 16, None,
                                                err, None) == _lib.DSA_ERR_INVALID_ARG
    g0 = _geom(T=0)
    assert lib.dsa_sparse_mla_attend_static(C.byref(g0), _lib.DSA_BF16, 16, None, None, None, 64, 0.1, None,
                                            None, 64, None) == _lib.DSA_OK


def test_bounded_step_key_spans_below_one_row(lib):
    L = 262144
    a = _lib.dsa_step_args_t()
    a.geom = _geom(T=2, B=1, max_seq_len=L, bt_stride=L // 64)
    a.topk = 2048
    a.H = 16
    a.Hi = 64
    row = L * 4
    full = lib.dsa_decode_step_workspace_size(C.byref(a))
    one_row = lib.dsa_decode_step_bounded_workspace_size(C.byref(a), row)
    span = lib.dsa_decode_step_bounded_workspace_size(C.byref(a), 65536)       # one 16384-key span
    assert span < one_row < full
    assert one_row - span >= row - 65536
    # a budget that holds neither a row nor one top-k chunk is refused before launch
    assert lib.dsa_decode_step_bounded(C.byref(a), 65535, 256, 1 << 30, None) == _lib.DSA_ERR_INVALID_ARG
    assert b"top-k chunk" in lib.dsa_last_error()
