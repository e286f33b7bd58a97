"""xattn_decode_noalloc: the decode entry point for callers that cannot allocate device
memory (a runtime that owns every allocation, a latency-critical thread that must not call
cudaMalloc, a fixed memory budget). Call after call, using only the library's static
scratch array, it must match the fp64 oracle and give bit for bit what xattn_decode gives
with a workspace of the caller's. This file is collected last on purpose."""

import numpy as np
import pytest
import torch

from decode_attention_xattention_gb300 import build, workloads as wl, xattn
from decode_attention_xattention_gb300.runner import DeviceBatch
import oracle
from gpu_helpers import compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    xattn.load()


def _noalloc(db, status):
    return xattn.xattn_decode_noalloc(db.desc, db.q, db.shared_k, db.shared_v, db.shared_len, db.pool_k, db.pool_v,
                                      db.idx, db.w.steps, db.out, db.lse, status, db.stream)


# one shape on the single-kernel path, one on the split path (scratch holds the pieces)
CASES = [
    (wl.custom(R=2, BW=32, Hq=8, Hkv=2, d=128, lens=(1500, 700), T=3, seed=31), 1536),
    (wl.custom(R=2, BW=16, Hq=8, Hkv=2, d=64, lens=(2000, 900), T=4, seed=32), 256),
]


@pytest.mark.parametrize("case", CASES, ids=["fused", "split"])
def test_noalloc_matches_oracle_and_workspace_entry_point(case):
    """Two calls in a row on the shared scratch array: each matches the fp64 oracle within
    the bf16 tolerances, and each is bit for bit what xattn_decode gives with a workspace of
    the caller's (same plan, same kernels), so no stale scratch contents leak in."""
    w, split = case
    db = DeviceBatch(wl.make_inputs(w), split_tokens=split)
    db.build_cache()
    assert db.plan().fused == (1 if split >= w.max_shared_len else 0)
    xattn.check(db.decode())
    torch.cuda.synchronize()
    ws_out, ws_lse = db.out.clone(), db.lse.clone()
    orc = oracle.load()
    inp = db.inputs
    pk, pv, idx = oracle.build_cache(orc, inp)
    ref_o, ref_l = orc.decode(oracle.dims_of(w), inp.q, inp.shared_k, inp.shared_v, inp.shared_len, pk, pv, idx,
                              w.steps)
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    for call in range(2):  # two calls in a row share the scratch array
        db.out.fill_(float("nan"))
        db.lse.fill_(float("nan"))
        xattn.check(_noalloc(db, status))
        torch.cuda.synchronize()
        assert int(status.item()) == 0, f"call {call}: status {int(status.item())}"
        assert torch.equal(db.out, ws_out) and torch.equal(db.lse, ws_lse), f"call {call}: differs from xattn_decode"
        got_o = db.out.float().cpu().numpy().reshape(-1, w.head_dim)
        got_l = db.lse.cpu().numpy().reshape(-1)
        compare(got_o, got_l, ref_o, ref_l, f"noalloc call {call}")


def test_noalloc_rejected_call_launches_nothing():
    """A call that fails a host-side check (here a step past max_steps) returns its error and
    enqueues nothing: the outputs keep their contents."""
    w = wl.custom(R=1, BW=4, Hq=4, Hkv=2, d=128, lens=(200,), T=2, seed=34)
    db = DeviceBatch(wl.make_inputs(w))
    db.build_cache()
    db.out.fill_(7.0)
    rc = xattn.xattn_decode_noalloc(db.desc, db.q, db.shared_k, db.shared_v, db.shared_len, db.pool_k, db.pool_v,
                                    db.idx, w.steps + 1, db.out, db.lse, None, db.stream)
    assert rc == xattn.XATTN_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert bool((db.out.float() == 7.0).all())


def test_noalloc_reports_device_status_per_call():
    w = wl.custom(R=1, BW=8, Hq=4, Hkv=2, d=128, lens=(300,), T=2, seed=33)
    db = DeviceBatch(wl.make_inputs(w))
    db.build_cache()
    status = torch.zeros((1,), dtype=torch.int32, device="cuda")
    good = db.idx.clone()
    db.idx[0, 3, 1] = 1 << 20  # an ancestry slot outside the pool
    xattn.check(_noalloc(db, status))
    torch.cuda.synchronize()
    assert int(status.item()) & xattn.XATTN_STATUS_BAD_SLOT
    assert torch.isnan(db.out[0, 3].float()).all()
    db.idx.copy_(good)
    xattn.check(_noalloc(db, status))  # the status starts from zero again
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.isfinite(db.out.float()).all()


def test_noalloc_rejects_shapes_beyond_its_scratch():
    # Shared-stage pieces of 64 x 4096 stacked rows x 128 fp32 need far more than 32 MiB.
    d = xattn.make_desc(64, 1024, 32, 8, 128, 8192, 1024, 1, 0.0, 0, 128)
    need = xattn.xattn_decode_workspace_size(d)
    assert need > xattn.XATTN_NOALLOC_SCRATCH_BYTES
    A = 0x10000  # never dereferenced: the call is rejected before any launch
    rc = xattn.xattn_decode_noalloc(d, A, A, A, A, A, A, A, 1, A, A, None)
    assert rc == xattn.XATTN_ERR_WORKSPACE_TOO_SMALL
