"""Chunked hash tree ("Requests of a Feather Must Flock Together", methodology, component 1)
through the C ABI, against the brute-force oracle that compares tokens directly (CPU only:
the structure is host code)."""

import json
import os

import numpy as np
import pytest

from oracle.cht import BruteForceScheduler, blocks, shared_blocks
from decode_attention_xattention_gb300 import build, xattn
from decode_attention_xattention_gb300.cht import ChunkedHashTree

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "cht_hand.json")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()


def _replay(sched_factory, g, check):
    s = sched_factory(g["block_tokens"])
    for st in g["steps"]:
        if st["op"] == "insert":
            for rid in st["ids"]:
                s.insert(rid, g["requests"][str(rid)])
        else:
            getattr(s, st["op"])(st["id"])
        check(s, st)


# -- the oracle against facts outside itself ----------------------------------------------
def test_oracle_hand_example():
    g = json.load(open(GOLDEN))

    def check(s, st):
        assert {str(k): s.missing(k) for k in s.waiting} == st["expect_missing"], st["why"]
        assert list(s.best()) == st["expect_best"], st["why"]

    _replay(BruteForceScheduler, g, check)


def test_oracle_closed_forms():
    """Empty batch: missing = whole blocks; a waiting copy of an active prompt misses 0;
    shared blocks never exceed either prompt's whole blocks."""
    s = BruteForceScheduler(4)
    s.insert(1, range(10))
    s.insert(2, range(10))
    s.insert(3, list(range(8)) + [99, 99, 99])
    assert s.missing(1) == 2 and s.missing(3) == 2
    s.admit(1)
    assert s.missing(2) == 0 and s.missing(3) == 0  # its two whole blocks equal r1's
    assert shared_blocks(list(range(9)), list(range(20)), 4) == blocks(list(range(9)), 4) == 2


# -- the native structure against the oracle ---------------------------------------------
class _Native:
    def __init__(self, B):
        self.t = ChunkedHashTree(B)

    def insert(self, rid, tok):
        assert self.t.insert(rid, tok) == 0

    def admit(self, rid):
        assert self.t.admit(rid) == 0

    def finish(self, rid):
        assert self.t.finish(rid) == 0

    def cancel(self, rid):
        assert self.t.cancel(rid) == 0


def test_native_hand_example():
    g = json.load(open(GOLDEN))
    waiting = set()

    def check(s, st):
        if st["op"] == "insert":
            waiting.update(st["ids"])
        elif st["op"] in ("admit", "cancel"):
            waiting.discard(st["id"])
        got = {str(k): s.t.missing(k)[1] for k in sorted(waiting)}
        assert got == st["expect_missing"], st["why"]
        rc, rid, miss = s.t.best()
        assert rc == 1 and [rid, miss] == st["expect_best"], st["why"]

    _replay(_Native, g, check)


def _streams(rng, n, groups, B):
    """Prompts in a few prefix groups: a group prefix cut at a random point (not on block
    boundaries), then a private suffix; some prompts shorter than a block."""
    bases = [rng.integers(0, 50, size=rng.integers(0, 12 * B + 1)).tolist() for _ in range(groups)]
    out = []
    for _ in range(n):
        base = bases[rng.integers(0, groups)]
        cut = int(rng.integers(0, len(base) + 1))
        out.append(base[:cut] + rng.integers(0, 50, size=rng.integers(0, 3 * B + 1)).tolist())
    return out


@pytest.mark.parametrize("B,groups,seed", [(1, 3, 0), (2, 4, 1), (3, 2, 2), (4, 5, 3), (8, 3, 4), (16, 2, 5)])
def test_native_matches_oracle_random_operations(B, groups, seed):
    rng = np.random.default_rng(seed)
    prompts = _streams(rng, 120, groups, B)
    nat, ora = ChunkedHashTree(B), BruteForceScheduler(B)
    next_id = 0
    done = []
    for step in range(400):
        op = rng.integers(0, 10)
        if op <= 3 or not ora.waiting:
            if done and rng.integers(0, 4) == 0:
                rid = done.pop(int(rng.integers(0, len(done))))  # an id used before, new prompt
            else:
                rid, next_id = next_id, next_id + 1
            tok = prompts[int(rng.integers(0, len(prompts)))]
            assert nat.insert(rid, tok) == 0
            ora.insert(rid, tok)
        elif op <= 6:
            rid = ora.best()[0]  # admit the best, as the scheduler does
            assert nat.admit(rid) == 0
            ora.admit(rid)
        elif op <= 8 and ora.active:
            rid = list(ora.active)[int(rng.integers(0, len(ora.active)))]
            assert nat.finish(rid) == 0
            ora.finish(rid)
            done.append(rid)
        else:
            rid = list(ora.waiting)[int(rng.integers(0, len(ora.waiting)))]
            assert nat.cancel(rid) == 0
            ora.cancel(rid)
            done.append(rid)
        want = ora.best()
        rc, rid, miss = nat.best()
        if want is None:
            assert rc == 0
        else:
            assert rc == 1 and (rid, miss) == want, (step, (rid, miss), want)
        for k in ora.waiting:
            assert nat.missing(k) == (0, ora.missing(k)), (step, k)
        assert nat.counts()[:2] == (len(ora.waiting), len(ora.active))


def test_native_rejects_bad_calls():
    t = ChunkedHashTree(4)
    assert t.insert(1, [1, 2, 3, 4]) == 0
    assert t.insert(1, [5]) == xattn.XATTN_ERR_INVALID_ARG  # id in use
    assert t.finish(1) == xattn.XATTN_ERR_INVALID_ARG  # waiting, not active
    assert t.admit(7) == xattn.XATTN_ERR_INVALID_ARG
    assert t.admit(1) == 0
    assert t.admit(1) == xattn.XATTN_ERR_INVALID_ARG  # already active
    assert t.cancel(1) == xattn.XATTN_ERR_INVALID_ARG
    assert t.missing(1)[0] == xattn.XATTN_ERR_INVALID_ARG
    assert t.best()[0] == 0  # nothing waits
    assert t.insert(2, []) == 0 and t.best() == (1, 2, 0)  # an empty prompt has no blocks
    assert t.finish(1) == 0 and t.counts() == (1, 0, 0)
    lib = xattn.load()
    assert lib.xattn_cht_create(0) is None
