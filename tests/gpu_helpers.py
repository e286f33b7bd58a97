"""Shared pieces of the GPU parity tests: run a workload through the C ABI and through the
oracle on the same seeded inputs, and compare."""

from __future__ import annotations

import numpy as np
import torch

import oracle
from decode_attention_xattention_gb300 import workloads as wl
from decode_attention_xattention_gb300.runner import DeviceBatch, bf16_tensor_to_f32
from decode_attention_xattention_gb300 import xattn

# Tolerances against the fp64 oracle (bf16 inputs, fp32 accumulation, bf16 output).
TOL_MAX = 1e-2
TOL_MEAN = 1e-3
TOL_LSE = 1e-3


def compare(got_o, got_l, ref_o, ref_l, what="", tol=None):
    """tol: (max |dout|, mean |dout|, max |dlse|); default the bf16 bounds above."""
    tmax, tmean, tlse = tol if tol is not None else (TOL_MAX, TOL_MEAN, TOL_LSE)
    got_o = np.asarray(got_o, np.float64)
    ref_o = np.asarray(ref_o, np.float64)
    assert np.isfinite(got_o).all(), f"{what}: non-finite output"
    err = np.abs(got_o - ref_o)
    lerr = np.abs(np.asarray(got_l, np.float64) - np.asarray(ref_l, np.float64))
    stats = dict(max=float(err.max()), mean=float(err.mean()), lse=float(lerr.max()))
    assert stats["max"] <= tmax, f"{what}: max |dout| {stats}"
    assert stats["mean"] <= tmean, f"{what}: mean |dout| {stats}"
    assert stats["lse"] <= tlse, f"{what}: max |dlse| {stats}"
    return stats


def run_and_check(w, rows=None, shared_kernel=0, split_tokens=0, check_cache=True, inp=None, step=None,
                  out_fp32=True, input_f32=False, tol=None):
    """GPU: beam updates for steps 0..T-1 then one decode. Oracle: its own beam updates
    then the plain definition. The kernels compute in fp32; by default they also write fp32
    output so the comparison measures the computation, not the final bf16 rounding (which
    test_bf16_output_is_rounded_fp32_output checks exactly). Returns (stats, DeviceBatch,
    inputs)."""
    orc = oracle.load()
    inp = wl.make_inputs(w) if inp is None else inp
    db = DeviceBatch(inp, shared_kernel=shared_kernel, split_tokens=split_tokens, out_fp32=out_fp32,
                     input_f32=input_f32)
    inp = db.inputs  # the values on the device: bf16-rounded, or fp32 kept unrounded
    db.build_cache()
    step = w.steps if step is None else step
    xattn.check(db.decode(step))
    torch.cuda.synchronize()
    assert db.read_status() == 0
    pk, pv, idx = oracle.build_cache(orc, inp)
    if check_cache:
        np.testing.assert_array_equal(db.idx.cpu().numpy(), idx)
        np.testing.assert_array_equal(bf16_tensor_to_f32(db.pool_k), pk)
        np.testing.assert_array_equal(bf16_tensor_to_f32(db.pool_v), pv)
    D = oracle.dims_of(w)
    ref_o, ref_l = orc.decode(D, inp.q, inp.shared_k, inp.shared_v, inp.shared_len, pk, pv, idx, step, rows=rows)
    got_o = db.out.float().cpu().numpy().reshape(-1, w.head_dim)
    got_l = db.lse.cpu().numpy().reshape(-1)
    if rows is not None:
        got_o, got_l = got_o[rows], got_l[rows]
    return compare(got_o, got_l, ref_o, ref_l, w.name, tol), db, inp
