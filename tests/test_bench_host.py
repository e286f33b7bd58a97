"""Host-side pieces of the benchmark, checked without a GPU: the count of this library's
kernel launches per timed step (the bench's `gpu_launches` claim) follows the decode form
each workload's plan selects."""

from __future__ import annotations

import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from decode_attention_xattention_gb300 import workloads as wl, xattn  # noqa: E402


def _plan(w, f32=False):
    d = xattn.make_desc(w.num_requests, w.beam_width, w.num_q_heads, w.num_kv_heads, w.head_dim,
                        w.max_shared_len, w.ns_slots, w.max_steps,
                        dtype=xattn.XATTN_DTYPE_F32 if f32 else xattn.XATTN_DTYPE_BF16)
    rc, p = xattn.xattn_query_plan(d, w.steps)
    assert rc == 0
    return p


@pytest.mark.parametrize("w, f32, launches", [
    (wl.GR, False, 2),         # beam update, then the decode in one kernel (Non-Shared part in the tile)
    (wl.WIDE, False, 2),
    (wl.LONG, False, 4),       # update, Shared stage, warp-per-beam Non-Shared piece, row merge
    (wl.FEATHER_1, False, 4),  # update, Shared stage, Non-Shared piece kernel, row merge
    (wl.FEATHER_8, False, 4),
    (wl.FEATHER_64, False, 4),
    (wl.TINY, True, 3),        # fp32 storage: update, CUDA-core Shared stage, walk-and-merge kernel
], ids=lambda x: getattr(x, "name", str(x)))
def test_launches_per_step_follow_the_plan(w, f32, launches):
    assert bench.launches_per_step(_plan(w, f32), w.steps, f32) == launches
