"""Device residency for a synthetic workload and the per-layer calls of one DSA step.

Uploads the numpy tensors of an inputs.Workload to the GPU (bytes and bit patterns
reinterpreted as e4m3/bf16 torch tensors) and issues the fused step through the
C ABI: the full layer runs indexer -> top-k -> sparse MLA and writes its
selection; every later (IndexShare) layer reuses that selection.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

from . import _lib
from .inputs import Workload


def _dev(a: np.ndarray, device, view=None) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(a)).to(device)
    return t.view(view) if view is not None else t


class _Arena:
    """Several tensors back to back in one device buffer (each 256-byte aligned), so that
    a step's per-call inputs, or its outputs, move between host and device in one copy."""

    def __init__(self):
        self.parts = []
        self.nbytes = 0

    def add(self, nbytes: int, dtype, shape):
        self.parts.append((self.nbytes, int(nbytes), dtype, tuple(shape)))
        self.nbytes = (self.nbytes + int(nbytes) + 255) // 256 * 256
        return len(self.parts) - 1

    def build(self, device):
        self.buf = torch.empty(max(self.nbytes, 256), dtype=torch.uint8, device=device)
        return [self.buf[o:o + n].view(dt).view(sh) for o, n, dt, sh in self.parts]


def _bytes_of(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).reshape(-1).view(np.uint8))


@dataclass
class DeviceLayer:
    q: torch.Tensor          # [T, H, 576] bf16
    kv: torch.Tensor         # [P, 64, 576] bf16 or [P, 64 * 656] uint8 record pages
    kv_dtype: int
    out: torch.Tensor        # [T, H, 512] bf16
    lse: torch.Tensor        # [T, H] fp32


class DeviceWorkload:
    """The workload on the device. The per-call inputs (geometry, indexer q / scales /
    weights, each layer's MLA q) are views into one buffer, `inputs`, and the layers'
    outputs into another, `outputs`; the caches are resident tensors of their own."""

    def __init__(self, wl: Workload, device="cuda", hist: bool = False):
        self.wl = wl
        self.device = torch.device(device)
        self.hist = hist   # the full layer through dsa_decode_step_hist
        d = self.device
        fp8 = wl.qk_dtype == "e4m3"
        self.qk_dtype = _lib.DSA_E4M3 if fp8 else _lib.DSA_BF16
        T = wl.T
        ins = _Arena()
        src = []

        def put(a, dtype, shape):
            src.append(_bytes_of(a))
            return ins.add(src[-1].numel(), dtype, shape)

        i_seq = put(wl.seq_lens.astype(np.int32), torch.int32, wl.seq_lens.shape)
        i_cu = put(wl.cu_q.astype(np.int32), torch.int32, wl.cu_q.shape)
        i_bt = put(wl.block_table.astype(np.int32), torch.int32, wl.block_table.shape)
        i_qi = put(wl.q_idx, torch.float8_e4m3fn if fp8 else torch.bfloat16, wl.q_idx.shape)
        i_qs = put(wl.q_scale, torch.float32, wl.q_scale.shape) if fp8 else None
        i_w = put(wl.w, torch.float32, wl.w.shape)
        i_q = [put(L.q, torch.bfloat16, L.q.shape) for L in wl.layers]
        views = ins.build(d)
        for v, b in zip(views, src):
            v.view(-1).view(torch.uint8).copy_(b)
        self.inputs = ins.buf
        # byte offset of the first MLA query: what the indexer and top-k read lies before it
        self.inputs_mla_q_offset = ins.parts[i_q[0]][0]
        self.seq_lens, self.cu_q, self.block_table = views[i_seq], views[i_cu], views[i_bt]
        self.geom = _lib.Geometry(self.seq_lens, self.cu_q, self.block_table, wl.num_pages,
                                  wl.max_seq_len, wl.T)
        self.q_idx = views[i_qi]
        self.q_scale = views[i_qs] if fp8 else None
        self.w = views[i_w]
        if fp8:
            self.idx_k = _dev(wl.idx_k, d, torch.float8_e4m3fn)
            self.idx_k_scale = _dev(wl.idx_k_scale, d)
        else:
            self.idx_k = _dev(wl.idx_k.view(np.int16), d, torch.bfloat16)
            self.idx_k_scale = None
        outs = _Arena()
        o_idx = []
        for L in wl.layers:
            H = L.q.shape[1]
            o_idx.append((outs.add(T * H * 512 * 2, torch.bfloat16, (T, H, 512)),
                          outs.add(T * H * 4, torch.float32, (T, H))))
        oviews = outs.build(d)
        self.outputs = outs.buf
        self.layers = []
        for li, L in enumerate(wl.layers):
            q = views[i_q[li]]
            if L.kv_dtype == "bf16":
                kv, kd = _dev(L.kv.view(np.int16), d, torch.bfloat16), _lib.DSA_BF16
            else:
                kv, kd = _dev(L.kv, d), (_lib.DSA_E4M3 if L.kv_dtype == "e4m3" else _lib.DSA_I8)
            self.layers.append(DeviceLayer(q, kv, kd, oviews[o_idx[li][0]], oviews[o_idx[li][1]]))
        self.idx = torch.empty(wl.T, wl.topk, dtype=torch.int32, device=d)
        self.args = [self._args(i) for i in range(len(self.layers))]
        need = max(self.workspace_size(i) for i in range(len(self.args)))
        self.ws = _lib.workspace(need, d)

    def _args(self, i: int):
        L = self.layers[i]
        common = dict(kv_dtype=L.kv_dtype, q=L.q, kv_cache=L.kv, sm_scale=self.wl.sm_scale,
                      out=L.out, lse=L.lse)
        if i == 0:
            return _lib.make_step_args(self.geom, self.wl.topk, qk_dtype=self.qk_dtype,
                                       q_idx=self.q_idx, q_scale=self.q_scale, w=self.w,
                                       idx_k_cache=self.idx_k, idx_k_scale=self.idx_k_scale,
                                       idx_out=self.idx, **common)
        return _lib.make_step_args(self.geom, self.wl.topk, reuse_idx=self.idx, **common)

    def workspace_size(self, i: int) -> int:
        if self.hist and i == 0:
            return _lib.dsa_decode_step_hist_workspace_size(self.args[0])
        return _lib.dsa_decode_step_workspace_size(self.args[i])

    def step(self, stream=None):
        """One DSA step over every layer, enqueued on `stream` (default: current)."""
        for i, a in enumerate(self.args):
            if self.hist and i == 0:
                _lib.dsa_decode_step_hist(a, self.ws, stream)
            else:
                _lib.dsa_decode_step(a, self.ws, stream)

    def check_error(self) -> int:
        return _lib.dsa_get_error(self.ws)
