"""Valid-path constraint (xGR section 2.2, xBeam): the host trie (CPU) and the dense / sparse
device masks (GPU) through the C ABI, against the brute-force oracle over the catalogue."""

import itertools

import numpy as np
import pytest

import oracle
from oracle.valid_path import mask_dense, sparse_best, valid_next
from decode_attention_xattention_gb300 import build, xattn


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()


def catalogue(rng, N, L, V, shared=True):
    """Items as token paths: a few popular first tokens (many items under them) when shared,
    duplicates included; tokens < V."""
    first = rng.integers(0, V, size=max(2, V // 8)) if shared else None
    items = rng.integers(0, V, size=(N, L)).astype(np.int32)
    if shared:
        items[:, 0] = first[rng.integers(0, len(first), size=N)]
        if L > 1:
            items[: N // 4, 1] = items[0, 1]
    items[N - 3:] = items[:3]  # duplicates
    return items


def prefixes(rng, items, rows, step, V):
    """Rows' prefixes: most follow an item's path, some leave the catalogue."""
    L = items.shape[1]
    pre = items[rng.integers(0, len(items), size=rows)].copy()
    off = rng.random(rows) < 0.25
    if step > 0:
        pre[off, step - 1] = rng.integers(0, V, size=off.sum())
    return np.ascontiguousarray(pre[:, :L], dtype=np.int32)


def trie_valid(off, tok, prefix_row, step):
    node = 0
    for l in range(step):
        kids = tok[off[node]:off[node + 1]]
        j = int(np.searchsorted(kids, prefix_row[l]))
        if j >= len(kids) or kids[j] != prefix_row[l]:
            return set()
        node = off[node] + j + 1
    return set(int(x) for x in tok[off[node]:off[node + 1]])


# -- host trie (CPU) ------------------------------------------------------------------------
@pytest.mark.parametrize("N,L,V,seed", [(1, 1, 4, 0), (40, 3, 6, 1), (300, 4, 20, 2), (200, 2, 500, 3)])
def test_trie_matches_oracle(N, L, V, seed):
    rng = np.random.default_rng(seed)
    items = catalogue(rng, N, L, V)
    off, tok = xattn.trie_build(items)
    uniq = {tuple(it[:l]) for it in items.tolist() for l in range(1, L + 1)}
    assert len(off) - 1 == 1 + len(uniq)  # root + distinct non-empty prefixes
    assert off[0] == 0 and np.all(np.diff(off) >= 0) and off[-1] == len(tok)
    for step in range(L):
        for row in prefixes(rng, items, 50, step, V):
            assert trie_valid(off, tok, row, step) == valid_next(items, row, step)
        for n in range(len(off) - 1):  # children in increasing order
            assert np.all(np.diff(tok[off[n]:off[n + 1]]) > 0)


def test_trie_full_product_and_errors():
    items = np.array(list(itertools.product(range(3), repeat=3)), np.int32)
    off, tok = xattn.trie_build(items)
    assert len(off) - 1 == 1 + 3 + 9 + 27
    lib = xattn.load()
    import ctypes
    n = ctypes.c_int64(0)
    bad = np.array([[0, -1]], np.int32)
    assert lib.xattn_trie_size(bad.ctypes.data_as(ctypes.c_void_p), 1, 2, ctypes.byref(n)) == xattn.XATTN_ERR_INVALID_ARG
    o = np.zeros(3, np.int32)
    t = np.zeros(2, np.int32)
    good = np.array([[1, 2]], np.int32)
    assert lib.xattn_trie_build(good.ctypes.data_as(ctypes.c_void_p), 1, 2, 5, o.ctypes.data_as(ctypes.c_void_p),
                                t.ctypes.data_as(ctypes.c_void_p)) == xattn.XATTN_ERR_INVALID_ARG  # wrong size


def test_device_calls_rejected_on_host():
    P = 0x1000
    f, g = xattn.xattn_valid_path_mask, xattn.xattn_valid_path_topk
    assert f(P, P, 5, 3, P, 3, 3, 4, 8, P) == xattn.XATTN_ERR_INVALID_ARG  # step == path_len
    assert f(P, P, 5, 3, P, 1, 2, 4, 8, P) == xattn.XATTN_ERR_INVALID_ARG  # stride < step
    assert f(P, P, 5, 3, None, 3, 1, 4, 8, P) == xattn.XATTN_ERR_INVALID_ARG  # prefix needed
    assert f(P, P, 5, 3, P, 3, 1, 4, 262145, P) == xattn.XATTN_ERR_UNSUPPORTED
    assert f(P + 2, P, 5, 3, P, 3, 1, 4, 8, P) == xattn.XATTN_ERR_MISALIGNED
    assert g(P, P, 5, 3, P, 3, 1, 4, 8, P, 1025, P, P) == xattn.XATTN_ERR_UNSUPPORTED
    assert g(P, P, 5, 3, P, 3, 1, 4, 8, P, 0, P, P) == xattn.XATTN_ERR_INVALID_ARG


# -- device masks (GPU) ---------------------------------------------------------------------
def _device(items, pre, logp):
    import torch
    off, tok = xattn.trie_build(items)
    d = {k: torch.from_numpy(np.ascontiguousarray(v)).cuda() for k, v in
         (("off", off), ("tok", tok if len(tok) else np.zeros(1, np.int32)), ("pre", pre), ("logp", logp))}
    d["nodes"] = len(off) - 1
    return d


@pytest.mark.gpu
@pytest.mark.parametrize("N,L,V,rows,seed", [(40, 3, 6, 16, 1), (3000, 3, 300, 256, 2), (500, 4, 4100, 64, 3),
                                             (2000, 2, 33, 100, 4)])
def test_dense_mask_matches_oracle(N, L, V, rows, seed):
    import torch
    rng = np.random.default_rng(seed)
    items = catalogue(rng, N, L, V)
    for step in range(L):
        pre = prefixes(rng, items, rows, step, V)
        logp = rng.standard_normal((rows, V)).astype(np.float32)
        d = _device(items, pre, logp)
        cnt = torch.full((rows,), -1, dtype=torch.int32, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        xattn.check(xattn.xattn_valid_path_mask(d["off"], d["tok"], d["nodes"], L, d["pre"], L, step, rows, V,
                                                d["logp"], cnt, st))
        want, wcnt = mask_dense(items, pre, step, logp)
        np.testing.assert_array_equal(d["logp"].cpu().numpy(), want)
        np.testing.assert_array_equal(cnt.cpu().numpy(), wcnt)
        assert int(st.item()) == 0


@pytest.mark.gpu
@pytest.mark.parametrize("N,L,V,rows,C,seed", [(40, 3, 6, 16, 4, 1), (3000, 3, 300, 256, 64, 2),
                                               (500, 4, 4100, 64, 1024, 3), (2000, 2, 33, 100, 7, 4)])
def test_sparse_list_matches_oracle(N, L, V, rows, C, seed):
    import torch
    rng = np.random.default_rng(seed)
    items = catalogue(rng, N, L, V)
    for step in range(L):
        pre = prefixes(rng, items, rows, step, V)
        logp = (np.round(rng.standard_normal((rows, V)) * 4) / 4).astype(np.float32)  # many equal values
        d = _device(items, pre, logp)
        ct = torch.zeros((rows, C), dtype=torch.int32, device="cuda")
        cl = torch.zeros((rows, C), dtype=torch.float32, device="cuda")
        cnt = torch.full((rows,), -1, dtype=torch.int32, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        xattn.check(xattn.xattn_valid_path_topk(d["off"], d["tok"], d["nodes"], L, d["pre"], L, step, rows, V,
                                                d["logp"], C, ct, cl, cnt, st))
        wt, wl, wc = sparse_best(items, pre, step, logp, C)
        np.testing.assert_array_equal(ct.cpu().numpy(), wt)
        np.testing.assert_array_equal(cl.cpu().numpy(), wl)
        np.testing.assert_array_equal(cnt.cpu().numpy(), wc)
        assert int(st.item()) == 0


@pytest.mark.gpu
def test_sparse_list_too_many_valid_and_pipeline_to_beam_select():
    """A row with more than 4096 valid tokens gets an empty list and a status bit; the
    sparse lists of a late step feed the beam selection (masked-out tails are -inf), whose
    result must equal the oracle's selection over the oracle's lists."""
    import torch
    V = 5000
    items = np.stack([np.arange(V), np.zeros(V)], 1).astype(np.int32)  # 5000 first tokens
    pre = np.zeros((2, 2), np.int32)
    logp = np.zeros((2, V), np.float32)
    d = _device(items, pre, logp)
    ct = torch.zeros((2, 8), dtype=torch.int32, device="cuda")
    cl = torch.zeros((2, 8), dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    xattn.check(xattn.xattn_valid_path_topk(d["off"], d["tok"], d["nodes"], 2, d["pre"], 2, 0, 2, V, d["logp"], 8,
                                            ct, cl, None, st))
    assert int(st.item()) & xattn.XATTN_STATUS_TOO_MANY_VALID
    assert (ct.cpu().numpy() == -1).all() and np.isneginf(cl.cpu().numpy()).all()

    rng = np.random.default_rng(9)
    R, BW, L, Vc, K = 2, 32, 3, 64, 16
    items = catalogue(rng, 4000, L, Vc)
    pre = prefixes(rng, items, R * BW, 2, Vc)
    logp = (-np.abs(rng.standard_normal((R * BW, Vc)))).astype(np.float32)
    d = _device(items, pre, logp)
    ct = torch.zeros((R * BW, K), dtype=torch.int32, device="cuda")
    cl = torch.zeros((R * BW, K), dtype=torch.float32, device="cuda")
    xattn.check(xattn.xattn_valid_path_topk(d["off"], d["tok"], d["nodes"], L, d["pre"], L, 2, R * BW, Vc, d["logp"],
                                            K, ct, cl))
    bs = (-rng.exponential(2.0, size=(R, BW))).astype(np.float32)
    d_bs = torch.from_numpy(bs).cuda()
    par = torch.zeros((R, BW), dtype=torch.int32, device="cuda")
    tk = torch.zeros_like(par)
    sc = torch.zeros((R, BW), dtype=torch.float32, device="cuda")
    xattn.check(xattn.xattn_beam_select(R, BW, K, BW, d_bs, cl, ct, par, tk, sc))
    wt, wl, _ = sparse_best(items, pre, 2, logp, K)
    want = oracle.load().beam_select(bs, wl.reshape(R, BW, K), wt.reshape(R, BW, K), BW)
    for g, w in zip((par, tk, sc), want):
        np.testing.assert_array_equal(g.cpu().numpy(), w)
