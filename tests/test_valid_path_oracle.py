"""Pins of the valid-path oracle (xGR section 2.2, xBeam valid path constraint) to facts
outside itself: a hand-worked catalogue and closed forms (CPU only)."""

import itertools
import json
import os

import numpy as np

from oracle.valid_path import mask_dense, sparse_best, valid_next

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "valid_path_hand.json")


def test_hand_example():
    g = json.load(open(GOLDEN))
    items, logp = np.array(g["items"]), np.array(g["logp"], np.float32)
    for c in g["cases"]:
        pre = np.array(c["prefix"])
        masked, counts = mask_dense(items, pre, c["step"], logp)
        valid = [sorted(np.nonzero(np.isfinite(masked[r]))[0].tolist()) for r in range(len(pre))]
        assert valid == c["expect_valid"], c["why"]
        assert counts.tolist() == [len(v) for v in c["expect_valid"]]
        tok, val, counts2 = sparse_best(items, pre, c["step"], logp, c["C"])
        assert tok.tolist() == c["expect_sparse_tokens"], c["why"]
        assert np.array_equal(counts, counts2)
        for r in range(len(pre)):
            for j, v in enumerate(tok[r]):
                assert (v < 0 and val[r, j] == -np.inf) or val[r, j] == logp[r, v]


def test_closed_forms():
    """A catalogue of every path over V tokens leaves everything valid at every step; a
    prefix that starts no item leaves nothing valid; unmasked entries keep their value."""
    V, L = 3, 3
    full = np.array(list(itertools.product(range(V), repeat=L)))
    logp = -np.arange(2 * V, dtype=np.float32).reshape(2, V)
    for step in range(L):
        m, counts = mask_dense(full, np.array([[1, 2, 0], [0, 0, 2]]), step, logp)
        assert np.array_equal(m, logp) and counts.tolist() == [V, V]
    part = full[full[:, 0] != 2]
    m, counts = mask_dense(part, np.array([[2, 0, 0], [1, 0, 0]]), 1, logp)
    assert counts.tolist() == [0, V] and np.isneginf(m[0]).all() and np.array_equal(m[1], logp[1])
    assert valid_next(part, [9, 9], 0) == {0, 1}
