"""Device buffers for one workload and the calls that drive them through the C ABI.

torch is used only to hold device memory and streams; every step of the method runs in
libxattn.so's kernels (xattn_beam_update builds the Non-Shared pool and ancestry table,
xattn_decode runs the Shared stage, the Non-Shared stage and the Merge).
"""

from __future__ import annotations

import numpy as np
import torch

from . import workloads as wl
from . import xattn


def to_bf16_tensor(x: np.ndarray, device) -> torch.Tensor:
    """float32 array of exact bf16 values -> bf16 tensor with the same bits."""
    bits = wl.bf16_bits(x)
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(device)


def bf16_tensor_to_f32(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy()


class DeviceBatch:
    """All device tensors of one decode batch (inputs resident in HBM)."""

    def __init__(self, inp: wl.Inputs, device="cuda", shared_kernel=0, split_tokens=0, stream=None,
                 extra_steps=0, out_fp32=False, input_f32=False):
        """input_f32: hold the inputs as fp32, unrounded (XATTN_DTYPE_F32: the CUDA-core
        kernels); otherwise they are rounded to bf16 (a no-op for bf16 workloads)."""
        w = inp.w
        self.input_f32 = bool(input_f32)
        if not self.input_f32:
            inp = inp.as_bf16()
        self.inputs = inp  # the values the device holds
        self.w = w
        self.device = device
        self.stream = stream
        R, BW, Hq, Hkv, d = w.num_requests, w.beam_width, w.num_q_heads, w.num_kv_heads, w.head_dim
        self.Tmax = w.max_steps + extra_steps
        self.S = BW * self.Tmax
        self.desc = xattn.make_desc(R, BW, Hq, Hkv, d, w.max_shared_len, self.S, self.Tmax, w.softmax_scale,
                                    shared_kernel, split_tokens,
                                    xattn.XATTN_DTYPE_F32 if out_fp32 else xattn.XATTN_DTYPE_BF16,
                                    xattn.XATTN_DTYPE_F32 if self.input_f32 else xattn.XATTN_DTYPE_BF16)
        if self.input_f32:
            def dev(x):
                return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(device)
        else:
            def dev(x):
                return to_bf16_tensor(x, device)
        self.q = dev(inp.q)
        if w.max_shared_len > 0:
            self.shared_k = dev(inp.shared_k)
            self.shared_v = dev(inp.shared_v)
        else:
            self.shared_k = self.shared_v = None
        self.shared_len = torch.from_numpy(inp.shared_len.astype(np.int32)).to(device)
        self.new_k = dev(inp.new_k) if w.steps > 0 else None
        self.new_v = dev(inp.new_v) if w.steps > 0 else None
        self.parents = torch.from_numpy(inp.parents.astype(np.int32)).to(device)
        self.pool_k = torch.zeros((R, self.S, Hkv, d), dtype=torch.float32 if self.input_f32 else torch.bfloat16,
                                  device=device)
        self.pool_v = torch.zeros_like(self.pool_k)
        self.idx = torch.zeros((R, BW, max(self.Tmax, 1)), dtype=torch.int32, device=device)
        self.out = torch.empty((R, BW, Hq, d), dtype=torch.float32 if out_fp32 else torch.bfloat16, device=device)
        self.lse = torch.empty((R, BW, Hq), dtype=torch.float32, device=device)
        self.ws_bytes = xattn.xattn_decode_workspace_size(self.desc)
        if self.ws_bytes == 0:
            raise xattn.XAttnError("descriptor rejected")
        self.workspace = torch.zeros((self.ws_bytes + 255) // 256 * 64, dtype=torch.int32, device=device)
        self.status = torch.zeros((1,), dtype=torch.int32, device=device)

    def clone(self) -> "DeviceBatch":
        """Another batch with the same values in buffers of its own (a device-to-device copy
        of every tensor): distinct addresses, so that rotating through clones defeats the L2."""
        c = object.__new__(DeviceBatch)
        c.__dict__.update(self.__dict__)
        for k, v in self.__dict__.items():
            if isinstance(v, torch.Tensor):
                setattr(c, k, v.clone())
        return c

    # -- the method's calls --------------------------------------------------------------
    def beam_update(self, s: int) -> int:
        return xattn.xattn_beam_update(self.desc, self.parents[s] if s > 0 else None, self.new_k[s], self.new_v[s],
                                       self.pool_k, self.pool_v, self.idx, s, self.status, self.stream)

    def build_cache(self, steps=None) -> None:
        for s in range(self.w.steps if steps is None else steps):
            xattn.check(self.beam_update(s))

    def decode(self, step=None, out=None, lse=None) -> int:
        step = self.w.steps if step is None else step
        return xattn.xattn_decode(self.desc, self.q, self.shared_k, self.shared_v, self.shared_len, self.pool_k,
                                  self.pool_v, self.idx if step > 0 else None, step,
                                  self.out if out is None else out, self.lse if lse is None else lse,
                                  self.workspace, self.ws_bytes, self.stream)

    def decode_step(self, s: int, out=None, lse=None) -> int:
        """Token s's bookkeeping and the decode over tokens 0..s in one call
        (xattn_decode_step with step = s + 1)."""
        return xattn.xattn_decode_step(self.desc, self.parents[s] if s > 0 else None, self.new_k[s], self.new_v[s],
                                       self.q, self.shared_k, self.shared_v, self.shared_len, self.pool_k,
                                       self.pool_v, self.idx, s + 1, self.out if out is None else out,
                                       self.lse if lse is None else lse, self.workspace, self.ws_bytes, self.stream)

    def decode_shared(self) -> int:
        return xattn.xattn_decode_shared(self.desc, self.q, self.shared_k, self.shared_v, self.shared_len,
                                         self.workspace, self.ws_bytes, self.stream)

    def decode_merge(self, step=None) -> int:
        step = self.w.steps if step is None else step
        return xattn.xattn_decode_merge(self.desc, self.q, self.shared_len, self.pool_k, self.pool_v,
                                        self.idx if step > 0 else None, step, self.out, self.lse, self.workspace,
                                        self.ws_bytes, self.stream)

    def partials(self):
        """(part_o [R, Hkv, pieces, M, d], part_lse [R, Hkv, pieces, M]) views of the workspace;
        pieces 0 .. num_splits-1 are the prefix pieces."""
        p = self.plan()
        w = self.w
        rows = w.num_requests * w.num_kv_heads * p.piece_stride * p.rows_per_unit
        f = self.workspace.view(torch.float32)
        po = f[64:64 + rows * w.head_dim].view(w.num_requests, w.num_kv_heads, p.piece_stride, p.rows_per_unit,
                                                w.head_dim)
        pl = f[64 + rows * w.head_dim:64 + rows * w.head_dim + rows].view(w.num_requests, w.num_kv_heads,
                                                                             p.piece_stride, p.rows_per_unit)
        return po, pl

    def read_status(self, clear=True) -> int:
        rc, st = xattn.xattn_read_status(self.workspace, clear, self.stream)
        xattn.check(rc)
        return st

    def plan(self, step=None):
        rc, p = xattn.xattn_query_plan(self.desc, self.w.steps if step is None else step)
        xattn.check(rc)
        return p
