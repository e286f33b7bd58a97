"""Plain restatement of the valid-path constraint, by brute force over the item catalogue.

TEST INFRASTRUCTURE ONLY: the tests and the bench's CPU leg are the only callers; nothing
here is shared with the native trie builder or the CUDA kernels.

What it computes (xGR: Efficient Generative Recommendation Serving at Scale, section 2.2,
xBeam "valid path constraint": only token sequences that map to real items may be
generated, enforced by masks made from a pre-built vocabulary of valid items):
    items [N, L]   the token path of every valid item
    prefix[row]    the tokens row (a beam) emitted so far; positions 0 .. step-1 count
    valid(row)     = { items[i, step] : items[i, 0:step] == prefix[row, 0:step] }
    dense mask     logp[row, v] unchanged for v in valid(row), -inf otherwise
    sparse list    the C valid tokens of largest logp[row, v] (ties to the smaller token),
                   best first, padded with token -1 and -inf; count = |valid(row)|
Plain Python loops over the catalogue: meant for the small cases the tests use.
"""

from __future__ import annotations

import numpy as np


def valid_next(items, prefix_row, step):
    out = set()
    p = [int(x) for x in prefix_row[:step]]
    for it in items:
        if [int(x) for x in it[:step]] == p:
            out.add(int(it[step]))
    return out


def mask_dense(items, prefix, step, logp):
    """(masked copy of logp [rows, V] float32, valid counts [rows])."""
    out = np.array(logp, dtype=np.float32, copy=True)
    counts = np.zeros(len(out), np.int32)
    for r in range(len(out)):
        ok = valid_next(items, prefix[r], step)
        counts[r] = len(ok)
        for v in range(out.shape[1]):
            if v not in ok:
                out[r, v] = -np.inf
    return out, counts


def sparse_best(items, prefix, step, logp, C):
    """(tokens [rows, C] int32, logp [rows, C] float32, counts [rows])."""
    rows = len(logp)
    tok = np.full((rows, C), -1, np.int32)
    val = np.full((rows, C), -np.inf, np.float32)
    counts = np.zeros(rows, np.int32)
    for r in range(rows):
        ok = sorted(valid_next(items, prefix[r], step), key=lambda v: (-float(logp[r][v]), v))
        counts[r] = len(ok)
        for j, v in enumerate(ok[:C]):
            tok[r, j] = v
            val[r, j] = logp[r][v]
    return tok, val, counts
