"""ctypes binding of libdsa.so (include/dsa.h): argument marshalling only.

Every function here forwards torch tensors' device pointers, the host sizes and
the current CUDA stream to the C ABI and raises DsaError on a non-OK status. No
step of the DSA computation runs in Python; if libdsa.so is missing the first
call raises instead of falling back to anything else.
"""
from __future__ import annotations

import ctypes as C
import os

import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libdsa.so")

DSA_OK, DSA_ERR_INVALID_ARG, DSA_ERR_UNSUPPORTED, DSA_ERR_CUDA = 0, 1, 2, 3
DSA_ERR_TIMEOUT, DSA_ERR_WORKSPACE, DSA_ERR_BAD_INDEX = 4, 5, 6
DSA_BF16, DSA_E4M3, DSA_I8 = 0, 1, 2

EXPORTED = (
    "dsa_indexer_scores", "dsa_indexer_scores_workspace_size",
    "dsa_topk", "dsa_topk_workspace_size",
    "dsa_sparse_mla_attend", "dsa_sparse_mla_attend_workspace_size", "dsa_sparse_mla_attend_static",
    "dsa_decode_step", "dsa_decode_step_workspace_size",
    "dsa_decode_step_bounded", "dsa_decode_step_bounded_workspace_size", "dsa_decode_step_wait_q",
    "dsa_decode_step_hist", "dsa_decode_step_hist_workspace_size",
    "dsa_cache_append", "dsa_cache_append_workspace_size",
    "dsa_indexer_prepare", "dsa_indexer_prepare_workspace_size", "dsa_stage_copy",
    "dsa_get_error", "dsa_clear_error", "dsa_wait_probe", "dsa_status_string", "dsa_last_error", "dsa_abi_version",
)


class DsaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        detail = ""
        if status in (DSA_ERR_CUDA, DSA_ERR_WORKSPACE):
            try:
                detail = " [" + load().dsa_last_error().decode() + "]"
            except ImportError:
                pass
        super().__init__(f"{where}: {status_string(status)} (status {status}){detail}")


class dsa_geom_t(C.Structure):
    _fields_ = [("B", C.c_int32), ("T", C.c_int32), ("max_seq_len", C.c_int32),
                ("num_pages", C.c_int32), ("page_size", C.c_int32), ("bt_stride", C.c_int32),
                ("seq_lens", C.c_void_p), ("cu_q", C.c_void_p), ("block_table", C.c_void_p)]


class dsa_step_args_t(C.Structure):
    _fields_ = [("geom", dsa_geom_t), ("topk", C.c_int32),
                ("qk_dtype", C.c_int), ("Hi", C.c_int32),
                ("q_idx", C.c_void_p), ("q_scale", C.c_void_p), ("w", C.c_void_p),
                ("idx_k_cache", C.c_void_p), ("idx_k_scale", C.c_void_p),
                ("reuse_idx", C.c_void_p), ("idx_out", C.c_void_p),
                ("kv_dtype", C.c_int), ("H", C.c_int32),
                ("q", C.c_void_p), ("kv_cache", C.c_void_p), ("sm_scale", C.c_float),
                ("out", C.c_void_p), ("lse", C.c_void_p)]


_lib = None


def load(path: str = LIB_PATH):
    """Loads libdsa.so once and declares every entry point's signature."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build it with `python -m dsa_sparse_attention_02_gb300.build`")
    lib = C.CDLL(path)
    P, I32, I64, SZ, F = C.c_void_p, C.c_int32, C.c_int64, C.c_size_t, C.c_float
    G = C.POINTER(dsa_geom_t)
    S = C.POINTER(dsa_step_args_t)
    sig = {
        "dsa_indexer_scores": (C.c_int, [G, C.c_int, I32, P, P, P, P, P, P, I64, P, SZ, P]),
        "dsa_indexer_scores_workspace_size": (SZ, [G]),
        "dsa_topk": (C.c_int, [G, P, I64, I32, P, P, SZ, P]),
        "dsa_topk_workspace_size": (SZ, [G, I32]),
        "dsa_sparse_mla_attend": (C.c_int, [G, C.c_int, I32, P, P, P, I32, F, P, P, P, SZ, P]),
        "dsa_sparse_mla_attend_workspace_size": (SZ, [G, I32, I32]),
        "dsa_sparse_mla_attend_static": (C.c_int, [G, C.c_int, I32, P, P, P, I32, F, P, P, P, P]),
        "dsa_decode_step": (C.c_int, [S, P, SZ, P]),
        "dsa_decode_step_workspace_size": (SZ, [S]),
        "dsa_decode_step_bounded": (C.c_int, [S, SZ, P, SZ, P]),
        "dsa_decode_step_wait_q": (C.c_int, [S, P, P, SZ, P]),
        "dsa_decode_step_hist": (C.c_int, [S, P, SZ, P]),
        "dsa_decode_step_hist_workspace_size": (SZ, [S]),
        "dsa_decode_step_bounded_workspace_size": (SZ, [S, SZ]),
        "dsa_cache_append": (C.c_int, [G, C.c_int, P, P, C.c_int, P, P, P, P, SZ, P]),
        "dsa_cache_append_workspace_size": (SZ, [G]),
        "dsa_indexer_prepare": (C.c_int, [G, I32, I32, P, P, P, P, P, P, F, P, P, P, P, P, SZ, P]),
        "dsa_indexer_prepare_workspace_size": (SZ, [G]),
        "dsa_stage_copy": (C.c_int, [P, P, SZ, P]),
        "dsa_get_error": (C.c_int, [P, P]),
        "dsa_clear_error": (C.c_int, [P, P]),
        "dsa_wait_probe": (C.c_int, [P, SZ, C.c_uint32, P]),
        "dsa_status_string": (C.c_char_p, [C.c_int]),
        "dsa_last_error": (C.c_char_p, []),
        "dsa_abi_version": (I32, []),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def status_string(status: int) -> str:
    try:
        return load().dsa_status_string(int(status)).decode()
    except ImportError:
        return f"status {status}"


def _ptr(t):
    """Address of a tensor of any device (None -> NULL): only for dsa_stage_copy, whose
    C side resolves and checks both ends itself."""
    return None if t is None else t.data_ptr()


def _dptr(t):
    """Address of a CUDA tensor (None -> NULL). Anything else is refused here, so that a
    host address never reaches a kernel."""
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"expected a CUDA tensor, got {type(t).__name__}"
                        + (f" on {t.device}" if isinstance(t, torch.Tensor) else ""))
    return t.data_ptr()


def _optr(t):
    """Address of an attention output (None -> NULL): a CUDA tensor, or a page-locked
    host tensor, which the C side resolves to its device mapping (and refuses if it has
    none). Anything else is refused here."""
    if t is None:
        return None
    if isinstance(t, torch.Tensor) and not t.is_cuda and t.is_pinned():
        return t.data_ptr()
    return _dptr(t)


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return C.c_void_p(s.cuda_stream)


def _check(status: int, where: str):
    if status != DSA_OK:
        raise DsaError(status, where)


class Geometry:
    """Request geometry: device tensors plus the host sizes the C ABI needs."""

    def __init__(self, seq_lens: torch.Tensor, cu_q: torch.Tensor, block_table: torch.Tensor,
                 num_pages: int, max_seq_len: int, T: int):
        for name, t in (("seq_lens", seq_lens), ("cu_q", cu_q), ("block_table", block_table)):
            if t.dtype != torch.int32 or not t.is_contiguous():
                raise TypeError(f"{name} must be a contiguous int32 tensor")
        self.seq_lens, self.cu_q, self.block_table = seq_lens, cu_q, block_table
        self.B = int(seq_lens.shape[0])
        self.T = int(T)
        self.num_pages = int(num_pages)
        self.max_seq_len = int(max_seq_len)
        self.c = dsa_geom_t(self.B, self.T, self.max_seq_len, self.num_pages, 64,
                            int(block_table.shape[1]) if block_table.dim() == 2 else 0,
                            _dptr(seq_lens), _dptr(cu_q), _dptr(block_table))

    @property
    def ref(self):
        return C.byref(self.c)


def workspace(nbytes: int, device) -> torch.Tensor:
    """A zeroed device workspace of at least `nbytes` (256-byte aligned by the allocator)."""
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def dsa_indexer_scores_workspace_size(geom: Geometry) -> int:
    return int(load().dsa_indexer_scores_workspace_size(geom.ref))


def dsa_indexer_scores(geom: Geometry, qk_dtype: int, q_idx, q_scale, w, idx_k_cache, idx_k_scale,
                       scores: torch.Tensor, ws: torch.Tensor, stream=None):
    Hi = int(w.shape[1])
    st = load().dsa_indexer_scores(geom.ref, qk_dtype, Hi, _dptr(q_idx), _dptr(q_scale), _dptr(w),
                                   _dptr(idx_k_cache), _dptr(idx_k_scale), _dptr(scores),
                                   int(scores.stride(0)), _dptr(ws), ws.numel(), _stream(stream))
    _check(st, "dsa_indexer_scores")


def dsa_topk_workspace_size(geom: Geometry, k: int) -> int:
    return int(load().dsa_topk_workspace_size(geom.ref, int(k)))


def dsa_topk(geom: Geometry, scores: torch.Tensor, k: int, idx: torch.Tensor, ws: torch.Tensor,
             stream=None):
    st = load().dsa_topk(geom.ref, _dptr(scores), int(scores.stride(0)), int(k), _dptr(idx),
                         _dptr(ws), ws.numel(), _stream(stream))
    _check(st, "dsa_topk")


def dsa_sparse_mla_attend_workspace_size(geom: Geometry, H: int, k: int) -> int:
    return int(load().dsa_sparse_mla_attend_workspace_size(geom.ref, int(H), int(k)))


def dsa_sparse_mla_attend(geom: Geometry, kv_dtype: int, q, kv_cache, idx, k: int, sm_scale: float,
                          out, lse, ws, stream=None):
    H = int(q.shape[1])
    st = load().dsa_sparse_mla_attend(geom.ref, kv_dtype, H, _dptr(q), _dptr(kv_cache), _dptr(idx),
                                      int(k), float(sm_scale), _optr(out), _optr(lse),
                                      _dptr(ws), ws.numel(), _stream(stream))
    _check(st, "dsa_sparse_mla_attend")


def dsa_sparse_mla_attend_static(geom: Geometry, kv_dtype: int, q, kv_cache, idx, k: int,
                                 sm_scale: float, out, lse, err_word, stream=None):
    """dsa_sparse_mla_attend without a workspace, for callers that cannot allocate device
    memory at call time; its partials use the library's static per-GPU buffer. err_word
    is a device int32 (zeroed by the caller) that receives device-side errors."""
    H = int(q.shape[1])
    st = load().dsa_sparse_mla_attend_static(geom.ref, kv_dtype, H, _dptr(q), _dptr(kv_cache), _dptr(idx),
                                             int(k), float(sm_scale), _optr(out), _optr(lse),
                                             _dptr(err_word), _stream(stream))
    _check(st, "dsa_sparse_mla_attend_static")


def dsa_cache_append_workspace_size(geom: Geometry) -> int:
    return int(load().dsa_cache_append_workspace_size(geom.ref))


def dsa_cache_append(geom: Geometry, kv_dtype: int, kv_new, kv_cache, qk_dtype: int = DSA_E4M3, k_new=None,
                     idx_k_cache=None, idx_k_scale=None, ws=None, stream=None):
    """Writes the geom.T new tokens (flattened like queries) into the paged caches."""
    st = load().dsa_cache_append(geom.ref, kv_dtype, _dptr(kv_new), _dptr(kv_cache), qk_dtype, _dptr(k_new),
                                 _dptr(idx_k_cache), _dptr(idx_k_scale), _dptr(ws), ws.numel() if ws is not None else 0,
                                 _stream(stream))
    _check(st, "dsa_cache_append")


def dsa_indexer_prepare_workspace_size(geom: Geometry) -> int:
    return int(load().dsa_indexer_prepare_workspace_size(geom.ref))


def dsa_indexer_prepare(geom: Geometry, Hi: int, rope_dim: int, q_in, k_in, rope_cos, rope_sin, ln_gamma,
                        ln_beta, ln_eps: float, q_out, q_scale, idx_k_cache=None, idx_k_scale=None, ws=None,
                        stream=None):
    """RoPE + e4m3 of the indexer queries into q_out / q_scale; LayerNorm + RoPE + e4m3
    of the new tokens' keys (k_in, or None) into the paged index cache."""
    st = load().dsa_indexer_prepare(geom.ref, int(Hi), int(rope_dim), _dptr(q_in), _dptr(k_in), _dptr(rope_cos),
                                    _dptr(rope_sin), _dptr(ln_gamma), _dptr(ln_beta), float(ln_eps), _dptr(q_out),
                                    _dptr(q_scale), _dptr(idx_k_cache), _dptr(idx_k_scale), _dptr(ws),
                                    ws.numel() if ws is not None else 0, _stream(stream))
    _check(st, "dsa_indexer_prepare")


def make_step_args(geom: Geometry, topk: int, *, qk_dtype=DSA_E4M3, q_idx=None, q_scale=None,
                   w=None, idx_k_cache=None, idx_k_scale=None, reuse_idx=None, idx_out=None,
                   kv_dtype=DSA_BF16, q=None, kv_cache=None, sm_scale=1.0, out=None,
                   lse=None) -> dsa_step_args_t:
    Hi = int(w.shape[1]) if w is not None else 0
    H = int(q.shape[1]) if q is not None else 0
    return dsa_step_args_t(geom.c, int(topk), int(qk_dtype), Hi, _dptr(q_idx), _dptr(q_scale),
                           _dptr(w), _dptr(idx_k_cache), _dptr(idx_k_scale), _dptr(reuse_idx),
                           _dptr(idx_out), int(kv_dtype), H, _dptr(q), _dptr(kv_cache),
                           float(sm_scale), _optr(out), _optr(lse))


def dsa_decode_step_workspace_size(args: dsa_step_args_t) -> int:
    return int(load().dsa_decode_step_workspace_size(C.byref(args)))


def dsa_decode_step(args: dsa_step_args_t, ws: torch.Tensor, stream=None):
    st = load().dsa_decode_step(C.byref(args), _dptr(ws), ws.numel(), _stream(stream))
    _check(st, "dsa_decode_step")


def dsa_decode_step_hist_workspace_size(args: dsa_step_args_t) -> int:
    return int(load().dsa_decode_step_hist_workspace_size(C.byref(args)))


def dsa_decode_step_hist(args: dsa_step_args_t, ws: torch.Tensor, stream=None):
    """dsa_decode_step with the top-k's first radix digit counted by the indexer."""
    st = load().dsa_decode_step_hist(C.byref(args), _dptr(ws), ws.numel(), _stream(stream))
    _check(st, "dsa_decode_step_hist")


def dsa_stage_copy(dst, src, nbytes: int, stream=None):
    """Copies nbytes from src to dst (device tensors or pinned host tensors) with the SMs."""
    st = load().dsa_stage_copy(_ptr(dst), _ptr(src), int(nbytes), _stream(stream))
    _check(st, "dsa_stage_copy")


def dsa_decode_step_wait_q(args: dsa_step_args_t, q_ready: torch.cuda.Event, ws: torch.Tensor, stream=None):
    """dsa_decode_step whose attention waits on q_ready (the MLA query's copy)."""
    ev = None if q_ready is None else C.c_void_p(q_ready.cuda_event)
    st = load().dsa_decode_step_wait_q(C.byref(args), ev, _dptr(ws), ws.numel(), _stream(stream))
    _check(st, "dsa_decode_step_wait_q")


def dsa_decode_step_bounded_workspace_size(args: dsa_step_args_t, score_budget_bytes: int) -> int:
    return int(load().dsa_decode_step_bounded_workspace_size(C.byref(args), int(score_budget_bytes)))


def dsa_decode_step_bounded(args: dsa_step_args_t, score_budget_bytes: int, ws: torch.Tensor, stream=None):
    """dsa_decode_step holding the scores of at most score_budget_bytes // (stride * 4)
    queries at a time; bitwise the same results."""
    st = load().dsa_decode_step_bounded(C.byref(args), int(score_budget_bytes), _dptr(ws), ws.numel(), _stream(stream))
    _check(st, "dsa_decode_step_bounded")


def dsa_get_error(ws: torch.Tensor, stream=None) -> int:
    return int(load().dsa_get_error(_dptr(ws), _stream(stream)))


def dsa_clear_error(ws: torch.Tensor, stream=None):
    _check(load().dsa_clear_error(_dptr(ws), _stream(stream)), "dsa_clear_error")


def dsa_wait_probe(ws: torch.Tensor, limit_us: int, stream=None):
    """Enqueues a wait that nothing completes, bounded by limit_us; the kernel records
    DSA_ERR_TIMEOUT in ws's error word (read it with dsa_get_error)."""
    _check(load().dsa_wait_probe(_dptr(ws), ws.numel(), int(limit_us), _stream(stream)), "dsa_wait_probe")


def dsa_abi_version() -> int:
    return int(load().dsa_abi_version())
