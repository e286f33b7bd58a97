"""Plain restatement of the chunked hash tree's queries, by direct token comparison.

TEST INFRASTRUCTURE ONLY: the tests and the bench's CPU leg are the only callers; the
product path never imports this module, and it shares no code with the native structure
(which works on block hashes; this module never hashes).

What it computes ("Requests of a Feather Must Flock Together", methodology, component 1,
Chunked Hash Tree: requests are represented over fixed-size token blocks; the scheduler
wants the waiting request with the fewest blocks not covered by the active batch):
    blocks(r)            = floor(len(tokens_r) / B)            (only whole blocks count)
    shared(r, a)         = the number of leading whole blocks i of r with
                           tokens_r[:(i+1)B] == tokens_a[:(i+1)B]
    covered(r)           = max over active requests a of shared(r, a)   (0 if none active)
    missing(r)           = blocks(r) - covered(r)
    best                 = the waiting request with the smallest missing(r), ties to the
                           earliest inserted.
Plain Python loops: meant for the small cases the tests use.
"""

from __future__ import annotations


def blocks(tokens, B: int) -> int:
    return len(tokens) // B


def shared_blocks(r, a, B: int) -> int:
    n = min(blocks(r, B), blocks(a, B))
    i = 0
    while i < n and list(r[: (i + 1) * B]) == list(a[: (i + 1) * B]):
        i += 1
    return i


class BruteForceScheduler:
    """Waiting and active requests kept as token lists; every query recomputes from them."""

    def __init__(self, block_tokens: int):
        if block_tokens < 1:
            raise ValueError("block_tokens must be >= 1")
        self.B = block_tokens
        self.seq = 0
        self.waiting = {}  # id -> (seq, tokens)
        self.active = {}  # id -> tokens

    def insert(self, rid, tokens):
        if rid in self.waiting or rid in self.active:
            raise ValueError("request id in use")
        self.waiting[rid] = (self.seq, list(tokens))
        self.seq += 1

    def missing(self, rid) -> int:
        tok = self.waiting[rid][1]
        cov = max((shared_blocks(tok, a, self.B) for a in self.active.values()), default=0)
        return blocks(tok, self.B) - cov

    def best(self):
        """(id, missing) of the best waiting request, or None."""
        if not self.waiting:
            return None
        rid = min(self.waiting, key=lambda k: (self.missing(k), self.waiting[k][0]))
        return rid, self.missing(rid)

    def admit(self, rid):
        self.active[rid] = self.waiting.pop(rid)[1]

    def finish(self, rid):
        del self.active[rid]

    def cancel(self, rid):
        del self.waiting[rid]
