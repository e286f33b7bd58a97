"""Pins of the fp64 oracle to facts outside itself.

Each check takes an oracle handle (the real one, or a variant with a planted mistake) and
raises AssertionError when the oracle disagrees with:
  * hand-derived worked examples (tests/golden/*.json),
  * closed forms of softmax attention,
  * torch's own scaled_dot_product_attention / logsumexp in fp64 (a library routine the
    oracle does not use),
  * invariants the split-cache method rests on (split-and-merge equals unsplit; keys are a
    set; a prefix token may equally live in the pool; equal ancestry and query give equal
    output),
  * the bookkeeping rule worked by hand, and "nothing copied on fork".
"""

from __future__ import annotations

import json
import math
import os

import numpy as np

from decode_attention_xattention_gb300 import workloads as wl
import oracle as oracle_mod

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _arr(x, dt=np.float32):
    return np.asarray(x, dtype=dt)


# ---------------------------------------------------------------------------------------
def check_golden_decode(orc):
    g = json.load(open(os.path.join(GOLDEN, "decode_hand.json")))
    dm = g["dims"]
    D = orc.dims(dm["R"], dm["BW"], dm["Hq"], dm["Hkv"], dm["d"], dm["Lmax"], dm["S"], dm["Tmax"], dm["scale"])
    out, lse = orc.decode(D, _arr(g["q"]), _arr(g["shared_k"]), _arr(g["shared_v"]),
                          _arr(g["shared_len"], np.int32), _arr(g["pool_k"]), _arr(g["pool_v"]),
                          _arr(g["beam_tok_idx"], np.int32), g["step"])
    np.testing.assert_allclose(out, np.asarray(g["expect_out"]), rtol=0, atol=1e-6)
    np.testing.assert_allclose(lse, np.asarray(g["expect_lse"]), rtol=0, atol=1e-6)


def check_golden_beam_update(orc):
    g = json.load(open(os.path.join(GOLDEN, "beam_update_hand.json")))
    BW, T = g["BW"], g["Tmax"]
    Hkv, d = 1, 2
    D = orc.dims(1, BW, 1, Hkv, d, 0, T * BW, T, 1.0)
    pool_k = np.full((1, T * BW, Hkv, d), -7.0, np.float32)
    pool_v = np.full_like(pool_k, -9.0)
    idx = np.full((1, BW, T), -1, np.int32)
    for s in range(T):
        par = np.asarray(g["parents"][s] if g["parents"][s] is not None else list(range(BW)), np.int32)[None]
        nk = np.arange(BW * Hkv * d, dtype=np.float32).reshape(1, BW, Hkv, d) + 100 * s
        nv = -nk
        before_k = pool_k.copy()
        orc.beam_update(D, par, nk, nk * 0 + nv, pool_k, pool_v, idx, s)
        np.testing.assert_array_equal(idx[0], np.asarray(g["expect_after_step"][s], np.int32))
        # new tokens land in slots s*BW .. s*BW+BW-1, one per beam, in beam order
        np.testing.assert_array_equal(pool_k[0, s * BW:(s + 1) * BW], nk[0])
        np.testing.assert_array_equal(pool_v[0, s * BW:(s + 1) * BW], nv[0])
        # nothing else in the pool moves (no copy on fork)
        keep = np.ones(T * BW, bool)
        keep[s * BW:(s + 1) * BW] = False
        np.testing.assert_array_equal(pool_k[0, keep], before_k[0, keep])


# ---------------------------------------------------------------------------------------
def _single_case(orc, Lp, step, d=8, Hq=2, Hkv=1, BW=2, seed=0):
    rng = np.random.default_rng(seed)
    R, T = 1, max(step, 1)
    S = T * BW
    q = rng.standard_normal((R, BW, Hq, d)).astype(np.float32)
    sk = rng.standard_normal((R, max(Lp, 1), Hkv, d)).astype(np.float32)
    sv = rng.standard_normal((R, max(Lp, 1), Hkv, d)).astype(np.float32)
    pk = rng.standard_normal((R, S, Hkv, d)).astype(np.float32)
    pv = rng.standard_normal((R, S, Hkv, d)).astype(np.float32)
    idx = np.zeros((R, BW, T), np.int32)
    for b in range(BW):
        for i in range(T):
            idx[0, b, i] = i * BW + b
    return q, sk, sv, pk, pv, idx, (R, BW, Hq, Hkv, d, max(Lp, 1), S, T)


def check_closed_form_single_key(orc):
    """One key: out = v exactly and lse = the single score."""
    scale = 0.37
    for where in ("prefix", "pool"):
        q, sk, sv, pk, pv, idx, dims = _single_case(orc, 1, 1, seed=3)
        D = orc.dims(*dims, scale)
        if where == "prefix":
            slen, step = np.array([1], np.int32), 0
            k, v = sk[0, 0, 0], sv[0, 0, 0]
        else:
            slen, step = np.array([0], np.int32), 1
        out, lse = orc.decode(D, q, sk, sv, slen, pk, pv, idx, step)
        R, BW, Hq = dims[0], dims[1], dims[2]
        for b in range(BW):
            if where == "pool":
                k, v = pk[0, idx[0, b, 0], 0], pv[0, idx[0, b, 0], 0]
            for h in range(Hq):
                row = b * Hq + h
                s = scale * float(np.dot(q[0, b, h].astype(np.float64), k.astype(np.float64)))
                np.testing.assert_allclose(out[row], v.astype(np.float64), rtol=0, atol=1e-12)
                assert abs(lse[row] - s) < 1e-9, (lse[row], s)


def check_closed_form_equal_keys(orc):
    """All keys equal: uniform weights, out = mean(V), lse = s + ln N."""
    d, N, scale = 16, 37, 0.25
    rng = np.random.default_rng(5)
    kvec = rng.standard_normal(d).astype(np.float32)
    q = rng.standard_normal((1, 1, 1, d)).astype(np.float32)
    sk = np.tile(kvec, (1, N, 1, 1)).reshape(1, N, 1, d).astype(np.float32)
    sv = rng.standard_normal((1, N, 1, d)).astype(np.float32)
    pk = np.zeros((1, 1, 1, d), np.float32)
    idx = np.zeros((1, 1, 1), np.int32)
    D = orc.dims(1, 1, 1, 1, d, N, 1, 1, scale)
    out, lse = orc.decode(D, q, sk, sv, np.array([N], np.int32), pk, pk, idx, 0)
    s = scale * float(np.dot(q[0, 0, 0].astype(np.float64), kvec.astype(np.float64)))
    np.testing.assert_allclose(out[0], sv[0, :, 0].astype(np.float64).mean(0), rtol=0, atol=1e-12)
    assert abs(lse[0] - (s + math.log(N))) < 1e-9


def check_closed_form_constant_v(orc):
    """V rows all equal to c: out = c whatever the scores."""
    w = wl.custom(R=2, BW=3, Hq=4, Hkv=2, d=16, lens=(20, 9), T=2, seed=11)
    inp = wl.make_inputs(w)
    c = np.linspace(-2, 2, w.head_dim).astype(np.float32)
    sv = np.broadcast_to(c, inp.shared_v.shape).copy()
    nv = np.broadcast_to(c, inp.new_v.shape).copy()
    inp2 = wl.Inputs(w, inp.q, inp.shared_k, sv, inp.shared_len, inp.new_k, nv, inp.parents)
    pk, pv, idx = oracle_mod.build_cache(orc, inp2)
    D = oracle_mod.dims_of(w)
    out, _ = orc.decode(D, inp.q, inp.shared_k, sv, inp.shared_len, pk, pv, idx, w.steps)
    np.testing.assert_allclose(out, np.broadcast_to(c.astype(np.float64), out.shape), rtol=0, atol=1e-12)


def check_closed_form_dominant_logit(orc):
    """One logit above all others by > 60: out equals that key's value to fp64 precision."""
    d = 8
    q = np.zeros((1, 1, 1, d), np.float32)
    q[0, 0, 0, 0] = 1.0
    N = 5
    sk = np.zeros((1, N, 1, d), np.float32)
    sk[0, 3, 0, 0] = 64.0
    sv = np.random.default_rng(2).standard_normal((1, N, 1, d)).astype(np.float32)
    pk = np.zeros((1, 1, 1, d), np.float32)
    idx = np.zeros((1, 1, 1), np.int32)
    D = orc.dims(1, 1, 1, 1, d, N, 1, 1, 1.0)
    out, lse = orc.decode(D, q, sk, sv, np.array([N], np.int32), pk, pk, idx, 0)
    np.testing.assert_allclose(out[0], sv[0, 3, 0].astype(np.float64), rtol=0, atol=1e-20 + 1e-12)
    assert abs(lse[0] - 64.0) < 1e-12


# ---------------------------------------------------------------------------------------
def _torch_reference(inp, pk, pv, idx, step):
    """Per beam: concatenate prefix and ancestry tokens, then torch SDPA (fp64, CPU) with
    torch's own GQA grouping; lse from torch.logsumexp of torch-computed scores."""
    import torch

    w = inp.w
    R, BW, Hq, Hkv, d = w.num_requests, w.beam_width, w.num_q_heads, w.num_kv_heads, w.head_dim
    out = np.zeros((R, BW, Hq, d))
    lse = np.zeros((R, BW, Hq))
    for r in range(R):
        L = int(inp.shared_len[r])
        for b in range(BW):
            k = np.concatenate([inp.shared_k[r, :L], pk[r, idx[r, b, :step]]], 0)  # [n, Hkv, d]
            v = np.concatenate([inp.shared_v[r, :L], pv[r, idx[r, b, :step]]], 0)
            qt = torch.from_numpy(inp.q[r, b].astype(np.float64))[:, None, :]  # [Hq, 1, d]
            kt = torch.from_numpy(k.astype(np.float64)).transpose(0, 1)  # [Hkv, n, d]
            vt = torch.from_numpy(v.astype(np.float64)).transpose(0, 1)
            o = torch.nn.functional.scaled_dot_product_attention(
                qt[None], kt[None], vt[None], scale=w.softmax_scale, enable_gqa=True)[0]
            out[r, b] = o[:, 0].numpy()
            kg = kt.repeat_interleave(Hq // Hkv, dim=0)
            sc = torch.matmul(qt, kg.transpose(1, 2))[:, 0] * w.softmax_scale
            lse[r, b] = torch.logsumexp(sc, dim=-1).numpy()
    return out.reshape(-1, d), lse.reshape(-1)


def check_against_torch_sdpa(orc):
    """Random ancestry, GQA, ragged prefixes: the oracle equals torch's own attention."""
    for w in (wl.custom(R=2, BW=5, Hq=6, Hkv=2, d=16, lens=(13, 7), T=3, seed=1),
              wl.custom(R=1, BW=3, Hq=4, Hkv=4, d=8, lens=(5,), T=4, seed=2),
              wl.custom(R=3, BW=2, Hq=8, Hkv=2, d=32, lens=(0, 3, 40), T=2, seed=3)):
        inp = wl.make_inputs(w)
        pk, pv, idx = oracle_mod.build_cache(orc, inp)
        D = oracle_mod.dims_of(w)
        out, lse = orc.decode(D, inp.q, inp.shared_k, inp.shared_v, inp.shared_len, pk, pv, idx, w.steps)
        # the reference takes the ancestry from the rule worked by hand: check the table first
        ro, rl = _torch_reference(inp, pk, pv, idx, w.steps)
        np.testing.assert_allclose(out, ro, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse, rl, rtol=0, atol=1e-12)


def check_plain_decode_special_case(orc):
    """BW = 1 and an empty Non-Shared part: plain decode attention (torch SDPA, fp64)."""
    import torch

    w = wl.custom(R=2, BW=1, Hq=8, Hkv=2, d=32, lens=(50, 17), T=1, seed=9)
    inp = wl.make_inputs(w)
    D = oracle_mod.dims_of(w)
    pk = np.zeros((w.num_requests, w.ns_slots, w.num_kv_heads, w.head_dim), np.float32)
    idx = np.zeros((w.num_requests, 1, 1), np.int32)
    out, _ = orc.decode(D, inp.q, inp.shared_k, inp.shared_v, inp.shared_len, pk, pk, idx, 0)
    out = out.reshape(w.num_requests, w.num_q_heads, w.head_dim)
    for r in range(w.num_requests):
        L = int(inp.shared_len[r])
        qt = torch.from_numpy(inp.q[r, 0].astype(np.float64))[None, :, None, :]
        kt = torch.from_numpy(inp.shared_k[r, :L].astype(np.float64)).transpose(0, 1)[None]
        vt = torch.from_numpy(inp.shared_v[r, :L].astype(np.float64)).transpose(0, 1)[None]
        ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=w.softmax_scale,
                                                               enable_gqa=True)[0, :, 0].numpy()
        np.testing.assert_allclose(out[r], ref, rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------------------
def check_split_merge_equals_unsplit(orc):
    """Shared pieces (any split points, empty ones included) + the Non-Shared part,
    merged by log-sum-exp, equal the unsplit result."""
    w = wl.custom(R=2, BW=4, Hq=4, Hkv=2, d=16, lens=(33, 12), T=3, seed=21)
    inp = wl.make_inputs(w)
    pk, pv, idx = oracle_mod.build_cache(orc, inp)
    D = oracle_mod.dims_of(w)
    args = (D, inp.q, inp.shared_k, inp.shared_v, inp.shared_len, pk, pv, idx)
    full_o, full_l = orc.decode(*args, w.steps)
    for cuts in ([0, 33], [0, 5, 5, 20, 33], [0, 1, 2, 3, 40], [0, 16, 32, 48]):
        parts = [orc.partial(*args, lo, hi, 0, 0) for lo, hi in zip(cuts[:-1], cuts[1:])]
        parts.append(orc.partial(*args, 0, 0, 0, w.steps))
        po = np.stack([p[0] for p in parts])
        pl = np.stack([p[1] for p in parts])
        mo, ml = orc.merge(po, pl)
        np.testing.assert_allclose(mo, full_o, rtol=0, atol=1e-12)
        np.testing.assert_allclose(ml, full_l, rtol=0, atol=1e-12)
    # Non-Shared positions may be split too
    parts = [orc.partial(*args, 0, 64, 0, 0), orc.partial(*args, 0, 0, 0, 1), orc.partial(*args, 0, 0, 1, 3)]
    mo, ml = orc.merge(np.stack([p[0] for p in parts]), np.stack([p[1] for p in parts]))
    np.testing.assert_allclose(mo, full_o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(ml, full_l, rtol=0, atol=1e-12)


def check_prefix_permutation_invariance(orc):
    w = wl.custom(R=1, BW=3, Hq=4, Hkv=2, d=16, lens=(25,), T=2, seed=31)
    inp = wl.make_inputs(w)
    pk, pv, idx = oracle_mod.build_cache(orc, inp)
    D = oracle_mod.dims_of(w)
    o1, l1 = orc.decode(D, inp.q, inp.shared_k, inp.shared_v, inp.shared_len, pk, pv, idx, w.steps)
    perm = np.random.default_rng(0).permutation(25)
    o2, l2 = orc.decode(D, inp.q, inp.shared_k[:, perm], inp.shared_v[:, perm], inp.shared_len, pk, pv, idx, w.steps)
    np.testing.assert_allclose(o2, o1, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l2, l1, rtol=0, atol=1e-12)


def check_prefix_token_moved_to_pool(orc):
    """Moving the last prefix token into the pool, as a slot every beam references, gives
    the same result: the Shared and Non-Shared parts are one key set."""
    w = wl.custom(R=2, BW=3, Hq=4, Hkv=2, d=16, lens=(10, 6), T=2, seed=41)
    inp = wl.make_inputs(w)
    pk, pv, idx = oracle_mod.build_cache(orc, inp)
    D = oracle_mod.dims_of(w)
    o1, l1 = orc.decode(D, inp.q, inp.shared_k, inp.shared_v, inp.shared_len, pk, pv, idx, w.steps)
    R, BW, T, S = w.num_requests, w.beam_width, w.steps, w.ns_slots
    pk2 = np.concatenate([pk, np.zeros_like(pk[:, :1])], 1)
    pv2 = np.concatenate([pv, np.zeros_like(pv[:, :1])], 1)
    idx2 = np.concatenate([idx, np.full((R, BW, 1), S, np.int32)], 2)
    for r in range(R):
        L = int(inp.shared_len[r])
        pk2[r, S] = inp.shared_k[r, L - 1]
        pv2[r, S] = inp.shared_v[r, L - 1]
    D2 = orc.dims(R, BW, w.num_q_heads, w.num_kv_heads, w.head_dim, w.max_shared_len, S + 1, T + 1, w.softmax_scale)
    o2, l2 = orc.decode(D2, inp.q, inp.shared_k, inp.shared_v, inp.shared_len - 1, pk2, pv2, idx2, T + 1)
    np.testing.assert_allclose(o2, o1, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l2, l1, rtol=0, atol=1e-12)


def check_equal_ancestry_equal_output(orc):
    w = wl.custom(R=1, BW=4, Hq=2, Hkv=1, d=16, lens=(12,), T=3, seed=51)
    inp = wl.make_inputs(w)
    par = inp.parents.copy()
    par[1:, 0, :] = 2  # every beam descends from beam 2 -> rows 0..3 share positions 0..T-2
    inp = wl.Inputs(w, inp.q, inp.shared_k, inp.shared_v, inp.shared_len, inp.new_k, inp.new_v, par)
    pk, pv, idx = oracle_mod.build_cache(orc, inp)
    # beams 1 and 3 get the same ancestry (row of beam 1) and the same q
    idx[0, 3] = idx[0, 1]
    q = inp.q.copy()
    q[0, 3] = q[0, 1]
    D = oracle_mod.dims_of(w)
    o, l = orc.decode(D, q, inp.shared_k, inp.shared_v, inp.shared_len, pk, pv, idx, w.steps)
    o = o.reshape(4, 2, -1)
    l = l.reshape(4, 2)
    np.testing.assert_array_equal(o[3], o[1])
    np.testing.assert_array_equal(l[3], l[1])
    assert not np.array_equal(o[2], o[1])


def check_ancestry_table_structure(orc):
    """After steps 0..T-1 with random parents: position i of every row is a slot written at
    step i, and row b's prefix is its parent's previous row."""
    w = wl.custom(R=2, BW=6, Hq=2, Hkv=1, d=8, lens=4, T=5, seed=61)
    inp = wl.make_inputs(w)
    D = oracle_mod.dims_of(w)
    pk = np.zeros((w.num_requests, w.ns_slots, 1, 8), np.float32)
    pv = np.zeros_like(pk)
    idx = np.zeros((w.num_requests, w.beam_width, w.steps), np.int32)
    for s in range(w.steps):
        prev = idx.copy()
        orc.beam_update(D, inp.parents[s], inp.new_k[s], inp.new_v[s], pk, pv, idx, s)
        for r in range(w.num_requests):
            for b in range(w.beam_width):
                p = inp.parents[s, r, b] if s > 0 else b
                assert list(idx[r, b, :s]) == list(prev[r, p, :s])
                assert idx[r, b, s] == s * w.beam_width + b
    for i in range(w.steps):
        assert np.all(idx[:, :, i] // w.beam_width == i)


# -- beam selection (xBeam) ----------------------------------------------------------------
def check_golden_beam_select(orc):
    g = json.load(open(os.path.join(GOLDEN, "beam_select_hand.json")))
    par, tok, sc = orc.beam_select(_arr(g["beam_score"]), _arr(g["cand_logp"]), _arr(g["cand_token"], np.int32),
                                   g["out_width"])
    np.testing.assert_array_equal(par, np.asarray(g["expect_parent"], np.int32))
    np.testing.assert_array_equal(tok, np.asarray(g["expect_token"], np.int32))
    np.testing.assert_array_equal(sc, np.asarray(g["expect_score"], np.float32))


def _select_case(rng, R, BW, K, levels):
    """Per-beam lists in non-increasing order drawn from a few multiples of 1/8 (many
    equal scores, every float32 sum exact), beam scores likewise, distinct tokens."""
    lp = -np.sort(rng.integers(0, levels, size=(R, BW, K)), axis=2).astype(np.float32) / 8
    bs = -rng.integers(0, levels, size=(R, BW)).astype(np.float32) / 8
    tok = rng.permutation(R * BW * K).astype(np.int32).reshape(R, BW, K)
    return bs, lp, tok


def _select_by_repeated_max(bs, lp, tok, W):
    """Independent restatement: W times, take the best remaining candidate (largest
    score, then smallest flat index) by a plain scan."""
    R, BW, K = lp.shape
    par = np.zeros((R, W), np.int32)
    tk = np.zeros((R, W), np.int32)
    sc = np.zeros((R, W), np.float32)
    for r in range(R):
        taken = set()
        for j in range(W):
            best = None
            for b in range(BW):
                for k in range(K):
                    if (b, k) in taken:
                        continue
                    s = np.float32(bs[r, b]) + np.float32(lp[r, b, k])
                    if best is None or s > best[0] or (s == best[0] and b * K + k < best[1] * K + best[2]):
                        best = (s, b, k)
            taken.add((best[1], best[2]))
            par[r, j], tk[r, j], sc[r, j] = best[1], tok[r, best[1], best[2]], best[0]
    return par, tk, sc


def check_beam_select_brute_force(orc):
    rng = np.random.default_rng(11)
    for R, BW, K, W, levels in ((1, 3, 4, 5, 4), (2, 4, 3, 12, 3), (1, 5, 6, 7, 20), (2, 2, 5, 1, 2)):
        bs, lp, tok = _select_case(rng, R, BW, K, levels)
        got = orc.beam_select(bs, lp, tok, W)
        want = _select_by_repeated_max(bs, lp, tok, W)
        for a, b in zip(got, want):
            np.testing.assert_array_equal(a, b)


def check_beam_select_shift_invariance(orc):
    """Adding one constant to every beam score (exactly, multiples of 1/8) shifts every
    chosen score by it and changes no choice."""
    rng = np.random.default_rng(12)
    bs, lp, tok = _select_case(rng, 2, 6, 5, 6)
    p0, t0, s0 = orc.beam_select(bs, lp, tok, 9)
    p1, t1, s1 = orc.beam_select(bs + np.float32(8.0), lp, tok, 9)
    np.testing.assert_array_equal(p0, p1)
    np.testing.assert_array_equal(t0, t1)
    np.testing.assert_array_equal(s1, s0 + np.float32(8.0))


def check_beam_select_prefix_structure(orc):
    """What early termination rests on: with every beam's list in order, the chosen
    candidates of each beam are a prefix of its list, and the scores come out in order."""
    rng = np.random.default_rng(13)
    bs, lp, tok = _select_case(rng, 3, 8, 6, 12)
    par, tk, sc = orc.beam_select(bs, lp, tok, 10)
    assert np.all(np.diff(sc, axis=1) <= 0)
    for r in range(3):
        for b in range(8):
            toks = [int(t) for t, p in zip(tk[r], par[r]) if p == b]
            assert toks == [int(t) for t in tok[r, b, :len(toks)]], (r, b)


ALL_CHECKS = [
    check_golden_decode, check_golden_beam_update, check_closed_form_single_key,
    check_closed_form_equal_keys, check_closed_form_constant_v, check_closed_form_dominant_logit,
    check_against_torch_sdpa, check_plain_decode_special_case, check_split_merge_equals_unsplit,
    check_prefix_permutation_invariance, check_prefix_token_moved_to_pool,
    check_equal_ancestry_equal_output, check_ancestry_table_structure,
    check_golden_beam_select, check_beam_select_brute_force, check_beam_select_shift_invariance,
    check_beam_select_prefix_structure,
]
