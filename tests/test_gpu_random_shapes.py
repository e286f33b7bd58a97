"""Seeded random shapes through every decode form against the fp64 oracle: ragged and empty
prefixes, one to 16 query heads per KV head, d 64 and 128, Non-Shared parts of 1 to 90
tokens (in the tile, staged, beside a split prefix, long enough for the piece kernel), the
automatic split plan and forced splits. Each case also runs xattn_decode_step for its last
token and must match update-then-decode bit for bit."""

from __future__ import annotations

import numpy as np
import pytest
import torch

from decode_attention_xattention_gb300 import workloads as wl
from decode_attention_xattention_gb300 import xattn
from decode_attention_xattention_gb300.runner import DeviceBatch
from gpu_helpers import run_and_check

pytestmark = pytest.mark.gpu


def _cases(n=24, seed=20261203):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        R = int(rng.integers(1, 4))
        Hkv = int(rng.choice([1, 2, 4]))
        G = int(rng.choice([1, 2, 4, 8, 16]))
        BW = int(rng.integers(1, 41))
        d = int(rng.choice([64, 128]))
        lens = tuple(int(x) for x in rng.choice([0, 1, 37, 128, 300, 700, 1500], size=R))
        if max(lens) == 0:
            lens = (lens[0] + 200,) + lens[1:]
        T = int(rng.choice([1, 3, 8, 20, 33, 70, 90]))
        split = int(rng.choice([0, 0, 128, 256]))
        out.append((R, BW, Hkv * G, Hkv, d, lens, T, split, 500 + i))
    return out


CASES = _cases()


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"R{c[0]}_BW{c[1]}_H{c[2]}x{c[3]}_d{c[4]}_t{c[6]}_s{c[7]}")
def test_random_shape_decode_and_step(case):
    R, BW, Hq, Hkv, d, lens, T, split, seed = case
    w = wl.custom(R=R, BW=BW, Hq=Hq, Hkv=Hkv, d=d, lens=lens, T=T, seed=seed)
    run_and_check(w, split_tokens=split)
    # the step form: xattn_decode_step(T) == xattn_beam_update(T-1) + xattn_decode(T)
    inp = wl.make_inputs(w)
    a = DeviceBatch(inp, split_tokens=split, out_fp32=True)
    b = DeviceBatch(inp, split_tokens=split, out_fp32=True)
    for db in (a, b):
        for s in range(T - 1):
            xattn.check(db.beam_update(s))
    xattn.check(a.decode_step(T - 1))
    xattn.check(b.beam_update(T - 1))
    xattn.check(b.decode(T))
    torch.cuda.synchronize()
    assert a.read_status() == 0 and b.read_status() == 0
    assert torch.equal(a.idx, b.idx)
    assert torch.equal(a.pool_k, b.pool_k) and torch.equal(a.pool_v, b.pool_v)
    assert torch.equal(a.out, b.out) and torch.equal(a.lse, b.lse)
