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


@dataclass
class DeviceLayer:
    q: torch.Tensor          # [T, H, 576] bf16
    kv: torch.Tensor         # [P, 64, 576] bf16 or [P, 64, 656] uint8
    kv_dtype: int
    out: torch.Tensor        # [T, H, 512] bf16
    lse: torch.Tensor        # [T, H] fp32


class DeviceWorkload:
    def __init__(self, wl: Workload, device="cuda"):
        self.wl = wl
        self.device = torch.device(device)
        d = self.device
        self.seq_lens = _dev(wl.seq_lens.astype(np.int32), d)
        self.cu_q = _dev(wl.cu_q.astype(np.int32), d)
        self.block_table = _dev(wl.block_table.astype(np.int32), d)
        self.geom = _lib.Geometry(self.seq_lens, self.cu_q, self.block_table, wl.num_pages,
                                  wl.max_seq_len, wl.T)
        if wl.qk_dtype == "e4m3":
            self.qk_dtype = _lib.DSA_E4M3
            self.q_idx = _dev(wl.q_idx, d, torch.float8_e4m3fn)
            self.q_scale = _dev(wl.q_scale, d)
            self.idx_k = _dev(wl.idx_k, d, torch.float8_e4m3fn)
            self.idx_k_scale = _dev(wl.idx_k_scale, d)
        else:
            self.qk_dtype = _lib.DSA_BF16
            self.q_idx = _dev(wl.q_idx.view(np.int16), d, torch.bfloat16)
            self.q_scale = None
            self.idx_k = _dev(wl.idx_k.view(np.int16), d, torch.bfloat16)
            self.idx_k_scale = None
        self.w = _dev(wl.w, d)
        self.layers = []
        for L in wl.layers:
            q = _dev(L.q.view(np.int16), d, torch.bfloat16)
            if L.kv_dtype == "bf16":
                kv, kd = _dev(L.kv.view(np.int16), d, torch.bfloat16), _lib.DSA_BF16
            else:
                kv, kd = _dev(L.kv, d), (_lib.DSA_E4M3 if L.kv_dtype == "e4m3" else _lib.DSA_I8)
            T, H = q.shape[0], q.shape[1]
            self.layers.append(DeviceLayer(q, kv, kd,
                                           torch.empty(T, H, 512, dtype=torch.bfloat16, device=d),
                                           torch.empty(T, H, dtype=torch.float32, device=d)))
        self.idx = torch.empty(wl.T, wl.topk, dtype=torch.int32, device=d)
        self.args = [self._args(i) for i in range(len(self.layers))]
        need = max(_lib.dsa_decode_step_workspace_size(a) for a in self.args)
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

    def step(self, stream=None):
        """One DSA step over every layer, enqueued on `stream` (default: current)."""
        for a in self.args:
            _lib.dsa_decode_step(a, self.ws, stream)

    def check_error(self) -> int:
        return _lib.dsa_get_error(self.ws)
