"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on the same seeded
inputs. Small shapes compare every output; the full-size workloads compare sampled rows."""

import numpy as np
import pytest
import torch

import oracle
from decode_attention_xattention_gb300 import build, workloads as wl, xattn
from decode_attention_xattention_gb300.runner import DeviceBatch, bf16_tensor_to_f32
from gpu_helpers import compare, run_and_check

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    xattn.load()


# -- small shapes: every output row, both Shared-stage kernels ---------------------------
SMALL = [
    # (R, BW, Hq, Hkv, d, lens, T): several tiles with ragged tails, ragged requests
    (1, 4, 2, 1, 64, (256,), 3),
    (2, 5, 8, 2, 128, (300, 129), 3),
    (3, 40, 16, 4, 128, (1000, 1, 517), 2),     # M = 160 rows: two row tiles, ragged
    (2, 16, 8, 8, 64, (640, 383), 4),           # G = 1
    (1, 3, 16, 2, 128, (2049,), 5),             # G = 8
    (2, 2, 16, 1, 64, (130, 255), 1),           # G = 16
    (1, 64, 8, 2, 128, (4096,), 6),             # M = 256
]


@pytest.mark.parametrize("shape", SMALL, ids=lambda s: f"R{s[0]}_BW{s[1]}_H{s[2]}x{s[3]}_d{s[4]}_L{'-'.join(map(str, s[5]))}_t{s[6]}")
@pytest.mark.parametrize("kernel", [1, 2], ids=["tensor_core", "cuda_core"])
def test_small_all_rows(shape, kernel):
    R, BW, Hq, Hkv, d, lens, T = shape
    w = wl.custom(R=R, BW=BW, Hq=Hq, Hkv=Hkv, d=d, lens=lens, T=T, seed=7)
    run_and_check(w, shared_kernel=kernel)


@pytest.mark.parametrize("split", [128, 256, 384, 1024, 2048])
def test_forced_splits_merge(split):
    w = wl.custom(R=2, BW=8, Hq=8, Hkv=2, d=128, lens=(1100, 700), T=3, seed=3)
    _, db, _ = run_and_check(w, split_tokens=split)
    assert db.plan().fused == (1 if split >= 1100 else 0)


def test_fused_and_split_paths_agree():
    """The single-kernel path (Shared stage + fused Non-Shared + Merge) and the split path
    (pieces + Non-Shared/Merge kernel) on the same inputs."""
    w = wl.custom(R=2, BW=24, Hq=8, Hkv=2, d=128, lens=(1500, 640), T=4, seed=19)
    _, a, _ = run_and_check(w, split_tokens=2048)
    _, b, _ = run_and_check(w, split_tokens=256)
    assert a.plan().fused == 1 and b.plan().fused == 0
    d = (a.out - b.out).abs().max().item()
    assert d <= 2e-3, d


@pytest.mark.parametrize("w", [wl.GR, wl.LONG, wl.custom(R=2, BW=8, Hq=8, Hkv=2, d=64, lens=(700, 300), T=3, seed=2)],
                         ids=lambda w: w.name)
def test_bf16_output_is_rounded_fp32_output(w):
    """The bf16 output is exactly the round-to-nearest-even of the fp32 output computed by
    the same kernels on the same inputs (so the precision checks made on the fp32 output
    carry over, plus at most half a bf16 ulp)."""
    inp = wl.make_inputs(w)
    outs = []
    for fp32 in (True, False):
        db = DeviceBatch(inp, out_fp32=fp32)
        db.build_cache()
        xattn.check(db.decode())
        torch.cuda.synchronize()
        outs.append((db.out.clone(), db.lse.clone()))
    (o32, l32), (o16, l16) = outs
    assert torch.equal(o32.to(torch.bfloat16), o16)
    assert torch.equal(l32, l16)


@pytest.mark.parametrize("T,d", [(33, 128), (64, 128), (70, 64), (130, 128)])
def test_long_non_shared_parts(T, d):
    """More than 32 ancestry tokens per beam: the Non-Shared part is cut into pieces of 64
    positions computed in parallel (last piece ragged), then merged with the prefix pieces.
    Request 1 has an empty prefix (Non-Shared only)."""
    w = wl.custom(R=2, BW=6, Hq=8, Hkv=2, d=d, lens=(300, 0), T=T, seed=T)
    _, db, _ = run_and_check(w)
    assert db.plan().fused == 0


@pytest.mark.parametrize("Hq,Hkv,d,T", [(16, 1, 128, 77), (32, 2, 64, 50), (2, 1, 64, 45), (8, 1, 128, 100),
                                         (4, 4, 64, 40)],
                         ids=["G16_d128", "G16_d64", "G2_d64", "G8_d128", "G1_d64"])
def test_long_non_shared_parts_group_sizes(Hq, Hkv, d, T):
    """The piece kernel holds the G query heads of a KV head as rows of one 16-row MMA tile:
    every group size (rows 8..15 in use only for G = 16), both head dims, ragged blocks."""
    w = wl.custom(R=2, BW=5, Hq=Hq, Hkv=Hkv, d=d, lens=(260, 0), T=T, seed=60 + T)
    _, db, _ = run_and_check(w)
    assert db.plan().fused == 0


@pytest.mark.parametrize("lens,T,d", [((5000, 300), 130, 128), ((9000, 0), 70, 64)], ids=["43_pieces", "73_pieces"])
def test_row_merge_many_pieces(lens, T, d):
    """The row merge keeps the LSEs of 64 pieces in registers and reloads the rest: 128-token
    prefix pieces plus a long Non-Shared part give 43 and 73 pieces per row, with empty prefix
    pieces (request 1's shorter or absent prefix) among them."""
    w = wl.custom(R=2, BW=3, Hq=8, Hkv=2, d=d, lens=lens, T=T, seed=70 + T)
    _, db, _ = run_and_check(w, split_tokens=128)
    assert db.plan().fused == 0


def test_bad_slot_in_long_part():
    """An out-of-range ancestry slot in the second piece of a long Non-Shared part: status
    BAD_SLOT and a NaN row for that beam only."""
    w = wl.custom(R=1, BW=4, Hq=8, Hkv=2, d=128, lens=(200,), T=100, seed=3)
    db = DeviceBatch(wl.make_inputs(w))
    db.build_cache()
    db.idx[0, 2, 70] = -5
    xattn.check(db.decode())
    assert db.read_status() & xattn.XATTN_STATUS_BAD_SLOT
    o = db.out.float().cpu()
    assert torch.isnan(o[0, 2]).all()
    assert torch.isfinite(o[0, [0, 1, 3]]).all()


@pytest.mark.parametrize("T,d,Hq,Hkv", [(9, 128, 8, 2), (16, 64, 8, 2), (32, 128, 16, 2), (20, 128, 4, 4)])
def test_medium_non_shared_parts_fused(T, d, Hq, Hkv):
    """9..32 ancestry tokens per beam with a one-piece prefix: the fused decode computes the
    Non-Shared part with the per-head piece kernel (one piece) ahead of the Shared stage."""
    w = wl.custom(R=2, BW=6, Hq=Hq, Hkv=Hkv, d=d, lens=(700, 129), T=T, seed=40 + T)
    _, db, _ = run_and_check(w, split_tokens=4096)
    assert db.plan().fused == 1


@pytest.mark.parametrize("shape", [(3, 8, 8, 4, 64, 5), (2, 5, 8, 2, 128, 7), (1, 4, 16, 16, 128, 8)],
                         ids=["G2_d64_t5", "G4_d128_t7", "G1_Hkv16_t8_wide_rows"])
def test_short_non_shared_beam_kernel_shapes(shape):
    """Short Non-Shared parts (step <= 8) whose keys do not fit one tile of the Shared-stage
    kernel ((128 / G) * step > 128) go through the warp-per-beam kernel when the beam's rows
    fit its shared memory, else through the per-head piece kernel (the last shape: 16 KV
    heads x 8 tokens x K and V rows exceed it); the Shared stage merges the piece."""
    R, BW, Hq, Hkv, d, T = shape
    w = wl.custom(R=R, BW=BW, Hq=Hq, Hkv=Hkv, d=d, lens=(300,) * R, T=T, seed=50 + T)
    _, db, _ = run_and_check(w, split_tokens=4096)
    p = db.plan()
    assert p.fused == 1 and p.ns_tile == 0


NS_TILE = [
    # (R, BW, Hq, Hkv, d, lens, T): (128 / G) * T <= 128 Non-Shared keys per row tile
    (2, 40, 16, 4, 128, (1000, 129), 4),     # G 4: a full 128-key tile; M = 160 (ragged row tile)
    (2, 5, 32, 2, 128, (300, 0), 16),        # G 16: 8 beams x 16 keys; request 1 Non-Shared only
    (3, 24, 16, 2, 64, (517, 256, 1), 8),    # G 8, d 64: 16 beams x 8 keys
    (1, 130, 2, 2, 128, (700,), 1),          # G 1: 128 beams x 1 key, two row tiles
    (2, 64, 4, 2, 64, (384, 200), 2),        # G 2, d 64
    (1, 3, 16, 2, 128, (2049,), 5),          # G 8: 3 of the tile's 16 beams exist
    (2, 8, 8, 2, 128, (128, 255), 3),        # a prefix of exactly one tile; a ragged one
]


@pytest.mark.parametrize("shape", NS_TILE, ids=lambda s: f"R{s[0]}_BW{s[1]}_H{s[2]}x{s[3]}_d{s[4]}_t{s[6]}")
def test_ns_tile_all_rows(shape):
    """One launch: the Shared-stage kernel gathers every beam's Non-Shared rows through the
    ancestry table into one more 128-key tile per row tile and attends to it (keys of other
    beams masked) before the prefix tiles. Every row against the oracle."""
    R, BW, Hq, Hkv, d, lens, T = shape
    w = wl.custom(R=R, BW=BW, Hq=Hq, Hkv=Hkv, d=d, lens=lens, T=T, seed=90 + T)
    _, db, _ = run_and_check(w, split_tokens=max(4096, w.max_shared_len))
    p = db.plan()
    assert p.fused == 1 and p.ns_tile == 1, (p.fused, p.ns_tile)


def test_ns_tile_bad_slot_in_one_beam():
    """A slot outside the pool in one beam's ancestry row on the one-launch path: status
    BAD_SLOT, NaN output and LSE for that beam's rows only, the other beams exact."""
    w = wl.custom(R=2, BW=16, Hq=8, Hkv=2, d=128, lens=(500, 300), T=3, seed=12)
    db = DeviceBatch(wl.make_inputs(w), out_fp32=True, split_tokens=512)
    db.build_cache()
    assert db.plan().ns_tile == 1
    db.idx[1, 9, 2] = 1 << 22
    xattn.check(db.decode())
    assert db.read_status() & xattn.XATTN_STATUS_BAD_SLOT
    o = db.out.cpu()
    l = db.lse.cpu()
    assert torch.isnan(o[1, 9]).all() and torch.isnan(l[1, 9]).all()
    good = torch.ones(w.num_requests, w.beam_width, dtype=torch.bool)
    good[1, 9] = False
    assert torch.isfinite(o[good]).all() and torch.isfinite(l[good]).all()


def test_tiny_config_both_kernels():
    for k in (0, 1, 2):
        stats, _, _ = run_and_check(wl.TINY, shared_kernel=k)


# fp32 inputs kept unrounded (CUDA-core kernels, fp32 arithmetic): against the fp64 oracle
# on the same unrounded values the error is that of fp32 accumulation and the approximate
# exp2, far below the bf16 bounds.
TOL_F32 = (2e-5, 2e-6, 2e-5)


def check_tf32(w, split_tokens=0):
    """fp32 storage with the Shared stage on the tensor cores (tcgen05 kind::tf32), against
    the fp64 oracle within a bound derived from the tf32 operands, per row:
      each prefix logit z = scale * q.k is off by at most eps = scale * 2^-9 * max_k sum|q_i k_i|
      (both operands carry at most 2^-10 relative error; fp32 accumulation adds far less), so
      every softmax weight moves by a factor within [e^-2eps, e^2eps] and their total
      variation is at most e^2eps - 1; P and V enter the P.V product with 2^-10 relative
      error each. Hence |dout| <= max|v| * ((e^2eps - 1) + 2^-9 e^2eps) and |dlse| <= eps,
      plus a 1e-5 allowance for the fp32 arithmetic of the rest of the path (the Non-Shared
      part and the merge are fp32)."""
    orc = oracle.load()
    db = DeviceBatch(wl.make_inputs(w), shared_kernel=1, split_tokens=split_tokens, out_fp32=True, input_f32=True)
    assert db.plan().shared_kernel == 3 and db.input_f32 and db.pool_k.dtype == torch.float32
    inp = db.inputs
    db.build_cache()
    xattn.check(db.decode())
    torch.cuda.synchronize()
    assert db.read_status() == 0
    pk, pv, idx = oracle.build_cache(orc, inp)
    ref_o, ref_l = orc.decode(oracle.dims_of(w), inp.q, inp.shared_k, inp.shared_v, inp.shared_len, pk, pv, idx,
                              w.steps)
    got_o = db.out.float().cpu().numpy().reshape(-1, w.head_dim).astype(np.float64)
    got_l = db.lse.cpu().numpy().reshape(-1).astype(np.float64)
    R, BW, Hq, Hkv, d = w.num_requests, w.beam_width, w.num_q_heads, w.num_kv_heads, w.head_dim
    G = Hq // Hkv
    scale = w.softmax_scale if w.softmax_scale > 0 else 1.0 / np.sqrt(d)
    q = np.abs(np.asarray(inp.q, np.float64)).reshape(R, BW, Hkv, G, d)
    eps = np.zeros((R, BW, Hkv, G))
    vmax = np.zeros((R, Hkv))
    for r in range(R):
        L = int(inp.shared_len[r])
        for h in range(Hkv):
            vmax[r, h] = max(np.abs(np.asarray(pv[r, :, h], np.float64)).max(),
                             np.abs(np.asarray(inp.shared_v[r, :L, h], np.float64)).max() if L else 0.0)
            if L:
                kabs = np.abs(np.asarray(inp.shared_k[r, :L, h], np.float64))
                eps[r, :, h] = scale * 2.0 ** -9 * np.einsum("bgd,ld->bgl", q[r, :, h], kabs).max(axis=-1)
    grow = np.exp(2 * eps)
    bound_o = (vmax[:, None, :, None] * ((grow - 1) + 2.0 ** -9 * grow) + 1e-5).reshape(-1, 1)
    bound_l = (eps + 1e-5).reshape(-1)
    assert bound_o.max() < 0.5, bound_o.max()  # not vacuous for these inputs (|v| up to ~4)
    err_o = np.abs(got_o - ref_o)
    err_l = np.abs(got_l - ref_l)
    assert np.isfinite(got_o).all() and np.isfinite(got_l).all()
    assert (err_o <= bound_o).all(), (err_o.max(), float(bound_o.min()))
    assert (err_l <= bound_l).all(), (err_l.max(), float(bound_l.min()))
    # The bound is a worst case over operand errors of one sign; on these random inputs the
    # errors average about 1e-4, while a key dropped or counted twice moves outputs by about
    # 1/L: a regression guard on the mean.
    assert err_o.mean() <= 1e-3, err_o.mean()
    stats = dict(max=float(err_o.max()), mean=float(err_o.mean()), lse=float(err_l.max()),
                 bound_min=float(bound_o.min()), bound_mean=float(bound_o.mean()),
                 worst_ratio=float((err_o / bound_o).max()))
    print(w.name, stats)
    return stats


@pytest.mark.parametrize("kernel", [0, 1, 2])
def test_tiny_config_native_fp32(kernel):
    """The Tiny configuration as specified: fp32 Q/K/V used unrounded (no bf16 step): fp32
    arithmetic on the CUDA cores (kernels 0 and 2), or the tensor cores in tf32 (kernel 1,
    within the bound check_tf32 derives)."""
    if kernel == 1:
        check_tf32(wl.TINY)
        return
    stats, db, _ = run_and_check(wl.TINY, shared_kernel=kernel, input_f32=True, tol=TOL_F32)
    assert db.input_f32 and db.plan().shared_kernel == 2 and db.pool_k.dtype == torch.float32


@pytest.mark.parametrize("shape,split", [((2, 48, 8, 2, 128, (700, 0), 3), 256),
                                         ((1, 64, 16, 1, 64, (300,), 5), 0),
                                         ((2, 8, 4, 4, 128, (130, 129), 2), 128)],
                         ids=["d128_2rowtiles_split_emptyprefix", "d64_G16_8rowtiles", "d128_G1_ragged"])
def test_tf32_shapes(shape, split):
    """The tf32 Shared stage on several row tiles, split and ragged prefixes (64-key tiles with
    a ragged last tile), an empty prefix next to a full one, d = 64 and 128, G = 1 and 16."""
    R, BW, Hq, Hkv, d, lens, T = shape
    w = wl.custom(R=R, BW=BW, Hq=Hq, Hkv=Hkv, d=d, lens=lens, T=T, seed=60 + T, input_dtype="fp32")
    check_tf32(w, split_tokens=split)


@pytest.mark.parametrize("shape", [(2, 6, 8, 2, 128, (300, 129), 5), (1, 3, 16, 1, 64, (0,), 32),
                                   (2, 4, 4, 4, 128, (513, 7), 0)],
                         ids=["G4_d128_split", "G16_d64_ns_only_32tok", "G1_d128_shared_only"])
def test_fp32_inputs_shapes(shape):
    """fp32 storage through every part the fp32 path has: split prefixes, a Non-Shared-only
    request (empty prefix), 32 ancestry tokens (the most the direct walk takes), step 0."""
    R, BW, Hq, Hkv, d, lens, T = shape
    w = wl.custom(R=R, BW=BW, Hq=Hq, Hkv=Hkv, d=d, lens=lens, T=max(T, 1), seed=80 + T, input_dtype="fp32",
                  lmax=256 if max(lens) == 0 else 0)
    run_and_check(w, input_f32=True, tol=TOL_F32, split_tokens=128, step=T)


def test_fp32_bf16_out():
    """fp32 inputs with bf16 output: the fp32 result rounded once at the store."""
    w = wl.custom(R=1, BW=4, Hq=8, Hkv=2, d=128, lens=(200,), T=3, seed=9, input_dtype="fp32")
    outs = []
    for fp32_out in (True, False):
        db = DeviceBatch(wl.make_inputs(w), out_fp32=fp32_out, input_f32=True)
        db.build_cache()
        xattn.check(db.decode())
        torch.cuda.synchronize()
        outs.append(db.out.clone())
    assert torch.equal(outs[0].to(torch.bfloat16), outs[1])


def test_shared_only_and_ns_only():
    w = wl.custom(R=2, BW=6, Hq=8, Hkv=2, d=128, lens=(777, 300), T=3, seed=5)
    run_and_check(w, step=0)  # Shared stage alone
    w0 = wl.custom(R=2, BW=6, Hq=8, Hkv=2, d=128, lens=(0, 0), T=3, seed=5, lmax=256)
    run_and_check(w0)  # Non-Shared stage alone (prefix length 0, storage present)
    wn = wl.custom(R=2, BW=6, Hq=8, Hkv=2, d=64, lens=(0, 0), T=3, seed=5)
    assert wn.max_shared_len == 0
    run_and_check(wn)  # no prefix storage at all (max_shared_len 0)


@pytest.mark.parametrize("kernel", [1, 2], ids=["tensor_core", "cuda_core"])
@pytest.mark.parametrize("split", [0, 256])
def test_cache_past_prefix_is_never_read(kernel, split):
    """Prefix-cache positions at or past a request's shared length may hold anything (here
    NaN and inf, in the ragged last tile and beyond): they take no part in the result."""
    w = wl.custom(R=3, BW=6, Hq=8, Hkv=2, d=128, lens=(1000, 300, 129), T=2, seed=23, lmax=1024)
    inp = wl.make_inputs(w).as_bf16()
    orc = oracle.load()
    db = DeviceBatch(inp, shared_kernel=kernel, split_tokens=split, out_fp32=True)
    for r, L in enumerate(inp.shared_len):
        db.shared_k[r, int(L):] = float("nan")
        db.shared_v[r, int(L):] = float("nan")
        db.shared_v[r, int(L) + 1::2] = float("inf")
    db.build_cache()
    xattn.check(db.decode())
    torch.cuda.synchronize()
    assert db.read_status() == 0
    pk, pv, idx = oracle.build_cache(orc, inp)
    ref_o, ref_l = orc.decode(oracle.dims_of(w), inp.q, inp.shared_k, inp.shared_v, inp.shared_len, pk, pv, idx,
                              w.steps)
    compare(db.out.float().cpu().numpy().reshape(-1, w.head_dim), db.lse.cpu().numpy().reshape(-1), ref_o, ref_l,
            "poisoned cache tail")


@pytest.mark.parametrize("kernel", [1, 2], ids=["tensor_core", "cuda_core"])
def test_shared_stage_pieces_match_oracle_partials(kernel):
    """xattn_decode_shared alone: every prefix piece's (normalised output, lse) against the
    oracle's attention restricted to that piece's tokens."""
    w = wl.custom(R=2, BW=8, Hq=8, Hkv=2, d=128, lens=(1100, 300), T=3, seed=3)
    inp = wl.make_inputs(w)
    db = DeviceBatch(inp, shared_kernel=kernel, split_tokens=256)
    xattn.check(db.decode_shared())
    torch.cuda.synchronize()
    p = db.plan()
    assert p.num_splits == 5 and p.split_tokens == 256
    po, pl = (t.cpu().numpy() for t in db.partials())
    orc = oracle.load()
    D = oracle.dims_of(w)
    R, BW, Hkv, G, d = w.num_requests, w.beam_width, w.num_kv_heads, w.group_size, w.head_dim
    for c in range(p.num_splits):
        ro, rl = orc.partial(D, inp.q, inp.shared_k, inp.shared_v, inp.shared_len, inp.shared_k[:, :1] * 0,
                             inp.shared_v[:, :1] * 0, np.zeros((R, BW, w.max_steps), np.int32), c * 256,
                             (c + 1) * 256, 0, 0)
        ro = ro.reshape(R, BW, Hkv, G, d).transpose(0, 2, 1, 3, 4).reshape(R, Hkv, BW * G, d)
        rl = rl.reshape(R, BW, Hkv, G).transpose(0, 2, 1, 3).reshape(R, Hkv, BW * G)
        for r in range(R):
            if np.isneginf(rl[r]).all():  # piece past this request's prefix
                assert np.isneginf(pl[r, :, c]).all() and not po[r, :, c].any()
                continue
            compare(po[r, :, c], pl[r, :, c], ro[r], rl[r], f"piece {c} of request {r}")


@pytest.mark.parametrize("Hkv,ns_tile", [(4, 0), (2, 1)], ids=["staged", "ns_tile"])
def test_equal_ancestry_equal_output(Hkv, ns_tile):
    """Beams with the same ancestry row and the same q rows get the same output. Bitwise
    when the Non-Shared part is computed per beam (staged piece). With the Non-Shared part in
    the Shared-stage tile, the two beams' keys sit in different columns of the tile, so the
    tensor core may group their P.V terms differently: equal to fp32 rounding."""
    w = wl.custom(R=1, BW=8, Hq=8, Hkv=Hkv, d=128, lens=(900,), T=3, seed=11)
    inp = wl.make_inputs(w)
    par = inp.parents.copy()
    par[1:, 0, :] = 3
    q = inp.q.copy()
    q[0, 5] = q[0, 2]
    inp = wl.Inputs(w, q, inp.shared_k, inp.shared_v, inp.shared_len, inp.new_k, inp.new_v, par)
    db = DeviceBatch(inp, out_fp32=True, split_tokens=1024)
    db.build_cache()
    assert db.plan().ns_tile == ns_tile
    idx = db.idx.clone()
    idx[0, 5] = idx[0, 2]
    db.idx.copy_(idx)
    xattn.check(db.decode())
    torch.cuda.synchronize()
    o = db.out.cpu().numpy()
    l = db.lse.cpu().numpy()
    if ns_tile:
        np.testing.assert_allclose(o[0, 5], o[0, 2], rtol=0, atol=2e-6)
        np.testing.assert_allclose(l[0, 5], l[0, 2], rtol=0, atol=2e-6)
    else:
        np.testing.assert_array_equal(o[0, 5], o[0, 2])
        np.testing.assert_array_equal(l[0, 5], l[0, 2])


def test_repeated_calls_deterministic():
    w = wl.custom(R=2, BW=16, Hq=8, Hkv=2, d=128, lens=(1500, 900), T=3, seed=13)
    db = DeviceBatch(wl.make_inputs(w))
    db.build_cache()
    xattn.check(db.decode())
    a = db.out.clone()
    for _ in range(3):
        xattn.check(db.decode())
    torch.cuda.synchronize()
    assert torch.equal(a, db.out)


def test_cuda_graph_capture_replay():
    w = wl.custom(R=2, BW=16, Hq=8, Hkv=2, d=128, lens=(1500, 900), T=3, seed=17)
    inp = wl.make_inputs(w)
    s = torch.cuda.Stream()
    db = DeviceBatch(inp, stream=s)
    with torch.cuda.stream(s):
        db.build_cache()
        xattn.check(db.decode())
    s.synchronize()
    ref = db.out.clone()
    db.out.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        xattn.check(db.decode())
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(ref, db.out)


# -- device-detected data errors: status word + NaN rows, no trap --------------------------
def test_bounded_wait_gives_up_and_context_stays_usable():
    """The timeout path of the bounded on-chip waits, without a fault: a wait on a phase that
    nothing completes gives up after its limit and records XATTN_STATUS_TIMEOUT; afterwards
    an ordinary decode still runs and matches the oracle."""
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    waited = torch.zeros(1, dtype=torch.int64, device="cuda")
    limit = 2_000_000  # SM cycles, about a millisecond
    xattn.check(xattn.xattn_check_bounded_wait(limit, st, waited))
    torch.cuda.synchronize()
    assert int(st.item()) & xattn.XATTN_STATUS_TIMEOUT
    assert int(waited.item()) >= limit
    run_and_check(wl.custom(R=1, BW=4, Hq=4, Hkv=2, d=128, lens=(300,), T=3, seed=2))


# split 2048: one prefix piece (the decode in one kernel, the Non-Shared part in its tile);
# 128: the prefix in two pieces, the short Non-Shared part written as one more piece beside
# the Shared stage and the row merge after both
@pytest.mark.parametrize("split", [2048, 128])
def test_bad_slot_sets_status_and_nan_row(split):
    w = wl.custom(R=1, BW=4, Hq=4, Hkv=2, d=128, lens=(200,), T=2, seed=1)
    db = DeviceBatch(wl.make_inputs(w), split_tokens=split)
    assert (db.plan().num_splits > 1) == (split < 200)
    db.build_cache()
    db.idx[0, 1, 0] = 10_000
    xattn.check(db.decode())
    st = db.read_status()
    assert st & xattn.XATTN_STATUS_BAD_SLOT
    o = db.out.float().cpu()
    assert torch.isnan(o[0, 1]).all() and torch.isfinite(o[0, 0]).all()
    assert db.read_status() == 0  # cleared by the previous read


@pytest.mark.parametrize("split", [2048, 128])
def test_bad_shared_len_sets_status(split):
    w = wl.custom(R=2, BW=4, Hq=4, Hkv=2, d=128, lens=(200, 100), T=2, seed=1)
    db = DeviceBatch(wl.make_inputs(w), split_tokens=split)
    assert (db.plan().num_splits > 1) == (split < 200)
    db.build_cache()
    db.shared_len[1] = 5000
    xattn.check(db.decode())
    st = db.read_status()
    assert st & xattn.XATTN_STATUS_BAD_SHARED_LEN
    o = db.out.float().cpu()
    assert torch.isnan(o[1]).all() and torch.isfinite(o[0]).all()


def test_bad_parent_sets_status():
    w = wl.custom(R=1, BW=4, Hq=4, Hkv=2, d=128, lens=(64,), T=3, seed=1)
    db = DeviceBatch(wl.make_inputs(w))
    xattn.check(db.beam_update(0))
    db.parents[1, 0, 2] = 9
    xattn.check(db.beam_update(1))
    torch.cuda.synchronize()
    assert int(db.status.item()) & xattn.XATTN_STATUS_BAD_PARENT
    assert int(db.idx[0, 2, 0].item()) == -1


def test_empty_row_status():
    w = wl.custom(R=1, BW=2, Hq=2, Hkv=1, d=64, lens=(0,), T=1, seed=1, lmax=64)
    db = DeviceBatch(wl.make_inputs(w))
    xattn.check(db.decode(0))
    assert db.read_status() & xattn.XATTN_STATUS_EMPTY_ROW


# -- the full-size workloads: sampled rows vs the oracle ---------------------------------
FULL = [wl.GR, wl.WIDE, wl.LONG, wl.FEATHER_1, wl.FEATHER_8, wl.FEATHER_64]


@pytest.mark.parametrize("w", FULL, ids=lambda w: w.name)
def test_full_size_sampled_rows(w):
    """Every beam's first and last query head plus 384 random rows against the oracle
    (fp32 output: the computation itself); every output row and lse finite."""
    rows = wl.sample_rows_every_beam(w, 384, seed=2)
    stats, db, _ = run_and_check(w, rows=rows)
    assert torch.isfinite(db.out.float()).all()
    assert torch.isfinite(db.lse).all()


@pytest.mark.parametrize("w", [wl.GR, wl.LONG, wl.FEATHER_1, wl.FEATHER_8], ids=lambda w: w.name)
def test_full_size_decode_step_sampled_rows(w):
    """The bench's timed call, xattn_decode_step for the last token (beam update + decode in
    one call: the in-tile decode as the update's dependent at GR; the Shared stage on the side
    stream beside the update and the Non-Shared kernels for Long and Feather), at full size:
    the pool and table bit-equal to the oracle's, and every beam's first and last query head
    plus 384 random rows against the oracle."""
    orc = oracle.load()
    inp = wl.make_inputs(w)
    db = DeviceBatch(inp, out_fp32=True)
    db.build_cache(steps=w.steps - 1)
    xattn.check(db.decode_step(w.steps - 1))
    torch.cuda.synchronize()
    assert db.read_status() == 0
    dev_in = db.inputs
    pk, pv, idx = oracle.build_cache(orc, dev_in)
    np.testing.assert_array_equal(db.idx.cpu().numpy(), idx)
    np.testing.assert_array_equal(bf16_tensor_to_f32(db.pool_k), pk)
    np.testing.assert_array_equal(bf16_tensor_to_f32(db.pool_v), pv)
    rows = wl.sample_rows_every_beam(w, 384, seed=4)
    ref_o, ref_l = orc.decode(oracle.dims_of(w), dev_in.q, dev_in.shared_k, dev_in.shared_v, dev_in.shared_len, pk,
                              pv, idx, w.steps, rows=rows)
    got_o = db.out.float().cpu().numpy().reshape(-1, w.head_dim)[rows]
    got_l = db.lse.cpu().numpy().reshape(-1)[rows]
    compare(got_o, got_l, ref_o, ref_l, w.name)
    assert torch.isfinite(db.out.float()).all() and torch.isfinite(db.lse).all()


@pytest.mark.parametrize("w", [wl.WIDE, wl.FEATHER_1], ids=lambda w: w.name)
def test_full_size_bf16_output(w):
    """The output the library returns by default (bf16) against the oracle at the stated
    tolerances, at full size: every beam's first and last query head plus 384 random rows."""
    rows = wl.sample_rows_every_beam(w, 384, seed=3)
    stats, db, _ = run_and_check(w, rows=rows, out_fp32=False)
    assert db.out.dtype == torch.bfloat16
    assert torch.isfinite(db.out.float()).all()
