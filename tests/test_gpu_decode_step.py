"""xattn_decode_step: a step's bookkeeping and its decode in one call. It must give, bit for
bit, what xattn_beam_update followed by xattn_decode gives (output, LSE, pool, ancestry
table, status bits), step after step, both when the decode is launched as the update's
programmatic dependent (the Shared-stage kernel takes the Non-Shared part in its tile) and
otherwise, and match the oracle."""

import numpy as np
import pytest
import torch

import oracle
from decode_attention_xattention_gb300 import build, workloads as wl, xattn
from decode_attention_xattention_gb300.runner import DeviceBatch
from gpu_helpers import compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    xattn.load()


def bits(t):
    return t.contiguous().view(torch.int32) if t.element_size() == 4 else t.contiguous().view(torch.int16)


STEP_SHAPES = [
    # (R, BW, Hq, Hkv, d, lens, T, split_tokens, in-tile Non-Shared part: dependent launch)
    (2, 40, 16, 4, 128, (1000, 129), 4, 4096, True),    # G 4: 32 beams x 4 keys fill the tile
    (3, 24, 16, 2, 64, (517, 256, 1), 5, 4096, True),   # G 8, d 64, ragged prefixes
    (2, 8, 8, 2, 128, (300, 0), 3, 4096, True),         # request 1 has no prefix
    (1, 130, 2, 2, 128, (700,), 1, 4096, True),         # G 1, one token: no parents yet
    (2, 6, 8, 4, 128, (300, 200), 5, 4096, False),      # G 2: 64 beams x 5 keys do not fit
    (2, 5, 8, 2, 128, (700, 300), 3, 256, False),       # prefix split in pieces
    (2, 5, 8, 2, 128, (700, 300), 20, 256, False),      # ... 20 Non-Shared tokens: one piece by the piece kernel
    (1, 6, 8, 1, 64, (600,), 12, 256, False),           # ... G 8, d 64
    (1, 4, 8, 2, 128, (300,), 40, 4096, False),         # 40 Non-Shared tokens: the piece kernels
]


@pytest.mark.parametrize("shape", STEP_SHAPES, ids=lambda s: f"R{s[0]}_BW{s[1]}_H{s[2]}x{s[3]}_d{s[4]}_t{s[6]}_"
                                                         f"{'pdl' if s[8] else 'plain'}")
def test_decode_step_equals_update_then_decode(shape):
    R, BW, Hq, Hkv, d, lens, T, split, one = shape
    w = wl.custom(R=R, BW=BW, Hq=Hq, Hkv=Hkv, d=d, lens=lens, T=T, seed=110 + T)
    inp = wl.make_inputs(w)
    a = DeviceBatch(inp, split_tokens=split, out_fp32=True)
    b = DeviceBatch(inp, split_tokens=split, out_fp32=True)
    assert bool(b.plan(T).ns_tile) == one
    for s in range(T):
        xattn.check(a.beam_update(s))
        xattn.check(a.decode(s + 1))
        xattn.check(b.decode_step(s))
        torch.cuda.synchronize()
        for x, y, what in ((a.out, b.out, "out"), (a.lse, b.lse, "lse"), (a.idx, b.idx, "table"),
                           (a.pool_k, b.pool_k, "pool_k"), (a.pool_v, b.pool_v, "pool_v")):
            assert torch.equal(bits(x), bits(y)), f"step {s}: {what} differs"
    assert a.read_status() == 0 and b.read_status() == 0 and int(a.status.item()) == 0
    orc = oracle.load()
    dev_in = b.inputs
    pk, pv, idx = oracle.build_cache(orc, dev_in)
    np.testing.assert_array_equal(b.idx.cpu().numpy(), idx)
    ref_o, ref_l = orc.decode(oracle.dims_of(w), dev_in.q, dev_in.shared_k, dev_in.shared_v, dev_in.shared_len, pk,
                              pv, idx, T)
    compare(b.out.cpu().numpy().reshape(-1, d), b.lse.cpu().numpy().reshape(-1), ref_o, ref_l, w.name)


def test_decode_step_bad_parent():
    """A parent outside [0, BW) at the last step: BAD_PARENT and BAD_SLOT, -1 in that beam's
    table row and NaN in its output, exactly as the two calls give them."""
    w = wl.custom(R=2, BW=16, Hq=8, Hkv=2, d=128, lens=(300, 500), T=3, seed=21)
    inp = wl.make_inputs(w)
    inp.parents[2, 1, 4] = 99
    a = DeviceBatch(inp, split_tokens=512, out_fp32=True)
    b = DeviceBatch(inp, split_tokens=512, out_fp32=True)
    assert b.plan(3).ns_tile == 1
    for s in range(3):
        xattn.check(a.beam_update(s))
        xattn.check(a.decode(s + 1))
        xattn.check(b.decode_step(s))
    torch.cuda.synchronize()
    st_a = int(a.status.item()) | a.read_status()
    st_b = b.read_status()
    assert st_a == st_b == (xattn.XATTN_STATUS_BAD_PARENT | xattn.XATTN_STATUS_BAD_SLOT), (st_a, st_b)
    for x, y in ((a.out, b.out), (a.lse, b.lse), (a.idx, b.idx), (a.pool_k, b.pool_k), (a.pool_v, b.pool_v)):
        assert torch.equal(bits(x), bits(y))
    assert (b.idx[1, 4, :2] == -1).all()
    assert torch.isnan(b.out[1, 4]).all() and torch.isfinite(b.out[0]).all()


def test_decode_step_rejects_bad_arguments():
    w = wl.custom(R=1, BW=4, Hq=4, Hkv=2, d=128, lens=(200,), T=2, seed=3)
    db = DeviceBatch(wl.make_inputs(w))
    args = lambda step, parent: (db.desc, parent, db.new_k[0], db.new_v[0], db.q, db.shared_k, db.shared_v,
                                 db.shared_len, db.pool_k, db.pool_v, db.idx, step, db.out, db.lse, db.workspace,
                                 db.ws_bytes, db.stream)
    assert xattn.xattn_decode_step(*args(0, None)) == xattn.XATTN_ERR_INVALID_ARG   # no token to add
    assert xattn.xattn_decode_step(*args(3, db.parents[1])) == xattn.XATTN_ERR_INVALID_ARG  # past max_steps
    assert xattn.xattn_decode_step(*args(2, None)) == xattn.XATTN_ERR_INVALID_ARG  # parents needed


@pytest.mark.parametrize("kernel", [2, 1], ids=["cuda_core", "tf32"])
def test_decode_step_fp32_storage(kernel):
    """fp32 storage: the Shared stage (fp32 on the CUDA cores, or tf32 on the tensor cores)
    launched beside the beam update gives, step after step, the same bits as the two calls."""
    w = wl.custom(R=2, BW=6, Hq=8, Hkv=2, d=64, lens=(300, 129), T=4, seed=17, input_dtype="fp32")
    inp = wl.make_inputs(w)
    a = DeviceBatch(inp, shared_kernel=kernel, out_fp32=True, input_f32=True)
    b = DeviceBatch(inp, shared_kernel=kernel, out_fp32=True, input_f32=True)
    assert b.plan(w.steps).shared_kernel == (2 if kernel == 2 else 3) and b.plan(w.steps).fused == 0
    for s in range(w.steps):
        xattn.check(a.beam_update(s))
        xattn.check(a.decode(s + 1))
        xattn.check(b.decode_step(s))
        torch.cuda.synchronize()
        for x, y, what in ((a.out, b.out, "out"), (a.lse, b.lse, "lse"), (a.idx, b.idx, "table"),
                           (a.pool_k, b.pool_k, "pool_k"), (a.pool_v, b.pool_v, "pool_v")):
            assert torch.equal(bits(x), bits(y)), f"step {s}: {what} differs"
    assert a.read_status() == 0 and b.read_status() == 0
