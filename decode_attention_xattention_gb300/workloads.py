"""Seeded synthetic workloads for split Shared / Non-Shared beam-search decode attention.

This module only draws random inputs and describes their shapes. It holds none of the
method's arithmetic: no scores, no softmax, no ancestry rewrite. Both the CUDA path and
the CPU oracle consume what it returns, each applying the method on its own.

The workloads follow the shapes of the xGR / Feather pages ("xGR: Efficient Generative
Recommendation Serving at Scale", section 4: beam widths 128 to 512 over long user-history
prompts; "Requests of a Feather Must Flock Together", results: shared prefixes of 1K-10K
tokens in a few prefix groups). The pages' datasets (Amazon Review, JD Trace, L-Eval,
LongBench) are not available; seeded N(0, 1) tensors of the same shapes stand in for them.

Layouts (row-major, innermost last):
    q            [R, BW, Hq, d]
    shared_k/v   [R, Lmax, Hkv, d]     prefix tokens j < shared_len[r] are valid
    new_k/v      [T, R, BW, Hkv, d]    the token each beam emits at decode step s < T
    parents      [T, R, BW] int32      beam chosen as parent at step s (row 0 unused)
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np


@dataclass(frozen=True)
class Workload:
    name: str
    num_requests: int
    beam_width: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    shared_lens: tuple
    steps: int  # Non-Shared tokens per beam seen by the decode step being measured
    # Parents at steps >= 1 are drawn from U{0 .. parent_range-1}; 0 means identity
    # ancestry (each sequence is its own parent: no sharing in the Non-Shared part).
    parent_range: int
    input_dtype: str = "bf16"  # "fp32" keeps full fp32 inputs (the CUDA path rounds to bf16)
    outlier_frac: float = 0.0  # fraction of prefix key rows scaled by outlier_scale
    outlier_scale: float = 8.0
    seed: int = 0
    description: str = field(default="", compare=False)
    lmax: int = 0  # prefix storage per request; 0 = the longest prefix

    @property
    def max_shared_len(self) -> int:
        return max(self.lmax, max(self.shared_lens) if self.shared_lens else 0)

    @property
    def ns_slots(self) -> int:
        return self.steps * self.beam_width

    @property
    def max_steps(self) -> int:
        return self.steps

    @property
    def group_size(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def softmax_scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    @property
    def num_beams(self) -> int:
        return self.num_requests * self.beam_width


def _w(name, R, BW, Hq, Hkv, d, lens, T, pr, **kw) -> Workload:
    if isinstance(lens, int):
        lens = (lens,) * R
    return Workload(name, R, BW, Hq, Hkv, d, tuple(lens), T, pr, **kw)


# The five workloads of the measured configuration list, by what they are.
TINY = _w("tiny_r1_bw4_h2x1_d64_L256_t3", 1, 4, 2, 1, 64, 256, 3, 4, input_dtype="fp32",
          description="1 request, beam width 4, 2 query / 1 KV head, d 64, prefix 256, "
                      "3 Non-Shared tokens, fp32 N(0,1)")
GR = _w("gr_r8_bw128_h32x8_d128_L2048_t3", 8, 128, 32, 8, 128, 2048, 3, 128,
        description="8 requests, beam width 128, GQA 32/8, d 128, prefix 2048, "
                    "3 Non-Shared tokens with random ancestry, bf16 N(0,1)")
WIDE = _w("wide_r4_bw512_h16x4_d128_L4096_t4", 4, 512, 16, 4, 128, 4096, 4, 256,
          description="4 requests, beam width 512, GQA 16/4, d 128, prefix 4096, "
                      "4 Non-Shared tokens, parents from the top half of the beams, bf16")
LONG = _w("long_r2_bw256_h32x8_d128_L32768+20000_t8", 2, 256, 32, 8, 128, (32768, 20000), 8, 256,
          outlier_frac=0.01,
          description="2 requests with prefixes 32768 and 20000, beam width 256, GQA 32/8, "
                      "d 128, 8 Non-Shared tokens, 1% of prefix keys scaled x8")


def feather(groups: int) -> Workload:
    """64 sequences over `groups` equal prefix groups (8192 shared tokens each) plus a
    512-token unshared suffix per sequence. A prefix group is one request and a sequence
    is one beam with identity ancestry."""
    assert 64 % groups == 0
    return _w(f"feather_g{groups}_seq64_h32x8_d128_L8192_s512", groups, 64 // groups, 32, 8,
              128, 8192, 512, 0,
              description=f"64 sequences in {groups} prefix group(s), GQA 32/8, d 128, "
                          f"shared prefix 8192, unshared suffix 512, bf16")


FEATHER_1, FEATHER_8, FEATHER_64 = feather(1), feather(8), feather(64)
ALL = {w.name: w for w in (TINY, GR, WIDE, LONG, FEATHER_1, FEATHER_8, FEATHER_64)}


def custom(R=1, BW=4, Hq=2, Hkv=1, d=64, lens=64, T=2, parent_range=None, seed=0,
           input_dtype="bf16", outlier_frac=0.0, lmax=0) -> Workload:
    """A small workload of arbitrary shape (tests)."""
    if parent_range is None:
        parent_range = BW
    return _w(f"custom_r{R}_bw{BW}_h{Hq}x{Hkv}_d{d}_t{T}_s{seed}", R, BW, Hq, Hkv, d, lens, T,
              parent_range, seed=seed, input_dtype=input_dtype, outlier_frac=outlier_frac, lmax=lmax)


# --------------------------------------------------------------------------------------
# bf16 handling of inputs (storage format only).

def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 (ties to even); returns float32 holding
    exactly representable bf16 values. NaN/Inf are not produced by the generators."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    r = (u + np.uint32(0x7FFF) + lsb) & np.uint32(0xFFFF0000)
    return r.view(np.float32)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Upper 16 bits of float32 values that are already exact bf16 values."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    return (x.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


# --------------------------------------------------------------------------------------

@dataclass
class Inputs:
    """Host arrays of one workload. Float arrays are float32; when the workload is bf16
    they hold exact bf16 values (so bf16_bits() recovers the device bits losslessly)."""
    w: Workload
    q: np.ndarray
    shared_k: np.ndarray
    shared_v: np.ndarray
    shared_len: np.ndarray
    new_k: np.ndarray
    new_v: np.ndarray
    parents: np.ndarray

    def as_bf16(self) -> "Inputs":
        """The same inputs rounded to bf16 (a no-op for bf16 workloads)."""
        if self.w.input_dtype == "bf16":
            return self
        return Inputs(self.w, round_to_bf16(self.q), round_to_bf16(self.shared_k),
                      round_to_bf16(self.shared_v), self.shared_len.copy(),
                      round_to_bf16(self.new_k), round_to_bf16(self.new_v), self.parents.copy())


def _normal(rng: np.random.Generator, shape, bf16: bool) -> np.ndarray:
    x = rng.standard_normal(size=shape, dtype=np.float32)
    return round_to_bf16(x) if bf16 else x


def make_inputs(w: Workload, seed: int | None = None) -> Inputs:
    """Draw one workload's inputs in a fixed order: q, shared_k, shared_v, new_k, new_v,
    parents, outlier mask. Prefix rows past shared_len[r] are zero."""
    rng = np.random.default_rng(w.seed if seed is None else seed)
    bf = w.input_dtype == "bf16"
    R, BW, Hq, Hkv, d, T = w.num_requests, w.beam_width, w.num_q_heads, w.num_kv_heads, w.head_dim, w.steps
    Lmax = w.max_shared_len
    q = _normal(rng, (R, BW, Hq, d), bf)
    sk = _normal(rng, (R, Lmax, Hkv, d), False)
    sv = _normal(rng, (R, Lmax, Hkv, d), False)
    new_k = _normal(rng, (T, R, BW, Hkv, d), bf)
    new_v = _normal(rng, (T, R, BW, Hkv, d), bf)
    parents = np.zeros((T, R, BW), dtype=np.int32)
    for s in range(1, T):
        if w.parent_range > 0:
            parents[s] = rng.integers(0, w.parent_range, size=(R, BW), dtype=np.int32)
        else:
            parents[s] = np.arange(BW, dtype=np.int32)[None, :]
    if T > 0:
        parents[0] = np.arange(BW, dtype=np.int32)[None, :]
    lens = np.asarray(w.shared_lens, dtype=np.int32)
    if w.outlier_frac > 0.0 and Lmax > 0:
        mask = rng.random(size=(R, Lmax)) < w.outlier_frac
        sk[mask] *= np.float32(w.outlier_scale)
    for r in range(R):
        sk[r, lens[r]:] = 0.0
        sv[r, lens[r]:] = 0.0
    if bf:
        sk = round_to_bf16(sk)
        sv = round_to_bf16(sv)
    return Inputs(w, q, sk, sv, lens, new_k, new_v, parents)


def sample_rows(w: Workload, n: int, seed: int = 1) -> np.ndarray:
    """n distinct flat row ids (r*BW + b)*Hq + h, always including the first and last row
    and, for every request, its first and last beam."""
    total = w.num_requests * w.beam_width * w.num_q_heads
    rng = np.random.default_rng(seed)
    forced = {0, total - 1}
    for r in range(w.num_requests):
        forced.add(r * w.beam_width * w.num_q_heads)
        forced.add(((r + 1) * w.beam_width - 1) * w.num_q_heads + w.num_q_heads - 1)
    n = min(n, total)
    extra = rng.choice(total, size=min(total, n + len(forced)), replace=False)
    rows = list(sorted(forced))
    for e in extra:
        if len(rows) >= max(n, len(forced)):
            break
        if int(e) not in forced:
            rows.append(int(e))
    return np.asarray(sorted(rows), dtype=np.int64)


def sample_rows_every_beam(w: Workload, extra: int, seed: int = 1) -> np.ndarray:
    """Flat row ids (r*BW + b)*Hq + h: every beam's first and last query head, plus `extra`
    more rows drawn at random (distinct, sorted)."""
    beams = np.arange(w.num_requests * w.beam_width, dtype=np.int64)
    forced = np.concatenate([beams * w.num_q_heads, beams * w.num_q_heads + w.num_q_heads - 1])
    total = w.num_requests * w.beam_width * w.num_q_heads
    rng = np.random.default_rng(seed)
    pick = rng.choice(total, size=min(total, extra + len(forced)), replace=False)
    rows = np.unique(forced)
    rest = np.setdiff1d(pick, rows)[:extra]
    return np.unique(np.concatenate([rows, rest]))


# --------------------------------------------------------------------------------------
# Beam-selection inputs (xGR section 2.2, xBeam): every beam's candidate list as a per-beam
# top-K returns it, best first.

def make_candidates(R: int, BW: int, K: int, seed: int = 0, vocab: int = 0, tie_levels: int = 0,
                    masked_frac: float = 0.0):
    """Seeded (beam_score [R, BW], cand_logp [R, BW, K], cand_token [R, BW, K]).

    cand_logp[r, b] is non-increasing: minus a running sum of positive exponential steps
    (or, with tie_levels > 0, sorted multiples of 1/8 from that many levels, which gives many
    equal scores and exact float32 sums); beam_score holds the beams' running scores (minus
    exponential, or multiples of 1/8). masked_frac of each list's tail is set to -inf (masked
    candidates, still in order). Tokens are drawn from a vocabulary of `vocab` (default 4K)."""
    rng = np.random.default_rng(seed)
    if tie_levels > 0:
        lp = -np.sort(rng.integers(0, tie_levels, size=(R, BW, K)), axis=2).astype(np.float32) / 8
        bs = -rng.integers(0, tie_levels, size=(R, BW)).astype(np.float32) / 8
    else:
        steps = rng.exponential(0.5, size=(R, BW, K)).astype(np.float32)
        lp = -np.cumsum(steps, axis=2, dtype=np.float32)
        bs = -rng.exponential(3.0, size=(R, BW)).astype(np.float32)
    if masked_frac > 0:
        keep = max(1, int(round(K * (1 - masked_frac))))
        lp[:, :, keep:] = -np.inf
    tok = rng.integers(0, vocab if vocab > 0 else 4 * K, size=(R, BW, K)).astype(np.int32)
    return np.ascontiguousarray(bs), np.ascontiguousarray(lp), np.ascontiguousarray(tok)
