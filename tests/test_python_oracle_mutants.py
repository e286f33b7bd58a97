"""Each deliberate mistake planted (on the CPU, by patching) in the Python oracles of the
chunked hash tree and of the valid-path constraint must make at least one of their pins
fail: the pins catch a partial block counted, coverage added up instead of maxed, the
wrong tie rule, an off-by-one position and a short prefix comparison."""

import numpy as np
import pytest

import oracle.cht as cht_mod
import oracle.valid_path as vp_mod
import test_cht
import test_valid_path_oracle


def _fails(check) -> bool:
    """True when the pin rejects the planted mistake (an assertion, not a crash)."""
    try:
        check()
    except AssertionError:
        return True
    return False


def _cht_pins():
    return [test_cht.test_oracle_hand_example, test_cht.test_oracle_closed_forms]


def _vp_pins():
    return [test_valid_path_oracle.test_hand_example, test_valid_path_oracle.test_closed_forms]


CHT_MUTANTS = {
    "partial block counted": lambda mp: mp.setattr(cht_mod, "blocks", lambda tokens, B: -(-len(tokens) // B)),
    "coverage added over active requests": lambda mp: mp.setattr(
        cht_mod.BruteForceScheduler, "missing",
        lambda self, rid: cht_mod.blocks(self.waiting[rid][1], self.B) - sum(
            cht_mod.shared_blocks(self.waiting[rid][1], a, self.B) for a in self.active.values())),
    "ties to the latest inserted": lambda mp: mp.setattr(
        cht_mod.BruteForceScheduler, "best",
        lambda self: None if not self.waiting else (lambda rid: (rid, self.missing(rid)))(
            min(self.waiting, key=lambda k: (self.missing(k), -self.waiting[k][0])))),
    "blocks compared one by one, not as a prefix": lambda mp: mp.setattr(cht_mod, "shared_blocks",
                                                                         _shared_blocks_unchained),
}


def _shared_blocks_unchained(r, a, B):
    """Counts every equal block, whether or not the blocks before it are equal."""
    n = min(len(r), len(a)) // B
    return sum(1 for i in range(n) if list(r[i * B:(i + 1) * B]) == list(a[i * B:(i + 1) * B]))


def _vp_valid_next_off_by_one(items, prefix_row, step):
    out = set()
    p = [int(x) for x in prefix_row[:step]]
    for it in items:
        if [int(x) for x in it[:step]] == p and step + 1 < len(it):
            out.add(int(it[step + 1]))
    return out


def _vp_valid_next_short_prefix(items, prefix_row, step):
    out = set()
    p = [int(x) for x in prefix_row[:max(step - 1, 0)]]
    for it in items:
        if [int(x) for x in it[:max(step - 1, 0)]] == p:
            out.add(int(it[step]))
    return out


VP_MUTANTS = {
    "next token read one position late": lambda mp: mp.setattr(vp_mod, "valid_next", _vp_valid_next_off_by_one),
    "prefix compared one token short": lambda mp: mp.setattr(vp_mod, "valid_next", _vp_valid_next_short_prefix),
    "sparse ties to the larger token": lambda mp: mp.setattr(
        vp_mod, "sparse_best",
        lambda items, prefix, step, logp, C: _sparse_ties_reversed(items, prefix, step, logp, C)),
}


def _sparse_ties_reversed(items, prefix, step, logp, C):
    rows = len(logp)
    tok = np.full((rows, C), -1, np.int32)
    val = np.full((rows, C), -np.inf, np.float32)
    counts = np.zeros(rows, np.int32)
    for r in range(rows):
        ok = sorted(vp_mod.valid_next(items, prefix[r], step), key=lambda v: (-float(logp[r][v]), -v))
        counts[r] = len(ok)
        for j, v in enumerate(ok[:C]):
            tok[r, j], val[r, j] = v, logp[r][v]
    return tok, val, counts


@pytest.mark.parametrize("name", sorted(CHT_MUTANTS))
def test_cht_pins_catch(name, monkeypatch):
    CHT_MUTANTS[name](monkeypatch)
    for mod in (test_cht,):  # the pins imported the names; patch their view too
        for attr in ("blocks", "shared_blocks"):
            monkeypatch.setattr(mod, attr, getattr(cht_mod, attr), raising=False)
    assert any(_fails(p) for p in _cht_pins()), name


@pytest.mark.parametrize("name", sorted(VP_MUTANTS))
def test_valid_path_pins_catch(name, monkeypatch):
    VP_MUTANTS[name](monkeypatch)
    for attr in ("valid_next", "sparse_best", "mask_dense"):
        monkeypatch.setattr(test_valid_path_oracle, attr, getattr(vp_mod, attr))
    assert any(_fails(p) for p in _vp_pins()), name
