"""fp64 CPU oracle for split Shared / Non-Shared beam-search decode attention.

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the bench's CPU-baseline leg are
the only callers. The product path never imports this package.

`load()` compiles `xattn_oracle.c` with gcc (once per variant) and wraps it with ctypes.
The arithmetic lives in the C file; this module only marshals numpy arrays.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "xattn_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_lock = threading.Lock()
_cache: dict = {}

# Deliberate mistakes that `-DORACLE_MUTANT=n` plants (tests show the pins catch each).
MUTANTS = {
    1: "Non-Shared part dropped",
    2: "GQA heads interleaved instead of grouped",
    3: "softmax scale dropped",
    4: "ancestry table read transposed",
    5: "max term dropped from the log-sum-exp",
    6: "last prefix token dropped",
    7: "new token recorded under the parent's slot",
    8: "ancestry not inherited from the parent",
    9: "merge weights not normalised",
    10: "beam selection: equal scores ordered by the larger index",
    11: "beam selection: the beam's own score not added",
}


def lib_path(mutant: int = 0) -> str:
    return os.path.join(_BUILD, "liboracle.so" if mutant == 0 else f"liboracle_m{mutant}.so")


def build(mutant: int = 0, force: bool = False) -> str:
    """Compile the oracle (plain C, OpenMP, no fast-math, no FMA contraction)."""
    out = lib_path(mutant)
    with _lock:
        if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(_SRC):
            return out
        os.makedirs(_BUILD, exist_ok=True)
        tmp = out + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
               f"-DORACLE_MUTANT={mutant}", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True, capture_output=True, text=True)
        os.replace(tmp, out)
    return out


class _Dims(ctypes.Structure):
    _fields_ = [("R", ctypes.c_int32), ("BW", ctypes.c_int32), ("Hq", ctypes.c_int32),
                ("Hkv", ctypes.c_int32), ("d", ctypes.c_int32), ("Lmax", ctypes.c_int32),
                ("S", ctypes.c_int32), ("Tmax", ctypes.c_int32), ("scale", ctypes.c_double)]


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def _i32(a):
    return np.ascontiguousarray(a, dtype=np.int32)


class Oracle:
    def __init__(self, mutant: int = 0):
        self.mutant = mutant
        self.lib = ctypes.CDLL(build(mutant))
        vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
        self.lib.oracle_partial_rows.argtypes = [ctypes.POINTER(_Dims)] + [vp] * 7 + [i32] * 4 + [vp, i64, vp, vp, i32]
        self.lib.oracle_decode_rows.argtypes = [ctypes.POINTER(_Dims)] + [vp] * 7 + [i32, vp, i64, vp, vp, i32]
        self.lib.oracle_merge.argtypes = [i32, i64, i32, vp, vp, vp, vp]
        self.lib.oracle_beam_update.argtypes = [ctypes.POINTER(_Dims), vp, vp, vp, vp, vp, vp, i32]
        self.lib.oracle_beam_select.argtypes = [i32, i32, i32, i32, vp, vp, vp, vp, vp, vp]
        for f in ("oracle_partial_rows", "oracle_decode_rows", "oracle_merge", "oracle_beam_update",
                  "oracle_beam_select", "oracle_mutant_id", "oracle_max_threads"):
            getattr(self.lib, f).restype = ctypes.c_int

    @staticmethod
    def dims(R, BW, Hq, Hkv, d, Lmax, S, Tmax, scale) -> _Dims:
        return _Dims(R, BW, Hq, Hkv, d, Lmax, S, Tmax, float(scale))

    def max_threads(self) -> int:
        return int(self.lib.oracle_max_threads())

    # -- attention ------------------------------------------------------------------
    def partial(self, D, q, sk, sv, slen, pk, pv, idx, p_lo, p_hi, t_lo, t_hi, rows=None,
                nthreads=0):
        """Attention over prefix tokens [p_lo, p_hi) and ancestry positions [t_lo, t_hi).
        Returns (out [n, d] fp64, lse [n] fp64)."""
        q, sk, sv, pk, pv = map(_f32, (q, sk, sv, pk, pv))
        slen, idx = _i32(slen), _i32(idx)
        if rows is not None:
            rows = np.ascontiguousarray(rows, dtype=np.int64)
        n = D.R * D.BW * D.Hq if rows is None else len(rows)
        out = np.zeros((n, D.d), np.float64)
        lse = np.zeros((n,), np.float64)
        rc = self.lib.oracle_partial_rows(ctypes.byref(D), _p(q), _p(sk), _p(sv), _p(slen), _p(pk),
                                          _p(pv), _p(idx), p_lo, p_hi, t_lo, t_hi, _p(rows),
                                          0 if rows is None else len(rows), _p(out), _p(lse), nthreads)
        if rc != 0:
            raise ValueError("oracle_partial_rows rejected its arguments")
        return out, lse

    def decode(self, D, q, sk, sv, slen, pk, pv, idx, step, rows=None, nthreads=0):
        """Full decode attention (whole valid prefix + first `step` ancestry tokens)."""
        q, sk, sv, pk, pv = map(_f32, (q, sk, sv, pk, pv))
        slen, idx = _i32(slen), _i32(idx)
        if rows is not None:
            rows = np.ascontiguousarray(rows, dtype=np.int64)
        n = D.R * D.BW * D.Hq if rows is None else len(rows)
        out = np.zeros((n, D.d), np.float64)
        lse = np.zeros((n,), np.float64)
        rc = self.lib.oracle_decode_rows(ctypes.byref(D), _p(q), _p(sk), _p(sv), _p(slen), _p(pk),
                                         _p(pv), _p(idx), step, _p(rows),
                                         0 if rows is None else len(rows), _p(out), _p(lse), nthreads)
        if rc != 0:
            raise ValueError("oracle_decode_rows rejected its arguments")
        return out, lse

    def merge(self, part_out, part_lse):
        part_out = np.ascontiguousarray(part_out, np.float64)
        part_lse = np.ascontiguousarray(part_lse, np.float64)
        P, n, d = part_out.shape
        out = np.zeros((n, d), np.float64)
        lse = np.zeros((n,), np.float64)
        rc = self.lib.oracle_merge(P, n, d, _p(part_out), _p(part_lse), _p(out), _p(lse))
        if rc != 0:
            raise ValueError("oracle_merge rejected its arguments")
        return out, lse

    # -- bookkeeping ----------------------------------------------------------------
    def beam_update(self, D, parent, new_k, new_v, pool_k, pool_v, idx, step):
        """In place on pool_k, pool_v (float32) and idx (int32), all C-contiguous."""
        for a, dt in ((pool_k, np.float32), (pool_v, np.float32), (idx, np.int32)):
            if a.dtype != dt or not a.flags.c_contiguous:
                raise TypeError("beam_update works in place on contiguous arrays")
        parent, new_k, new_v = _i32(parent), _f32(new_k), _f32(new_v)
        rc = self.lib.oracle_beam_update(ctypes.byref(D), _p(parent), _p(new_k), _p(new_v),
                                         _p(pool_k), _p(pool_v), _p(idx), step)
        if rc != 0:
            raise ValueError("oracle_beam_update rejected its arguments")


    # -- beam selection -------------------------------------------------------------
    def beam_select(self, beam_score, cand_logp, cand_token, out_width):
        """beam_score [R, BW], cand_logp / cand_token [R, BW, K] -> (parent, token, score),
        each [R, out_width], best first (full sort; ties to the smaller flat index)."""
        cand_logp = _f32(cand_logp)
        R, BW, K = cand_logp.shape
        beam_score, cand_token = _f32(beam_score), _i32(cand_token)
        if beam_score.shape != (R, BW) or cand_token.shape != (R, BW, K):
            raise ValueError("beam_select: shapes do not match")
        parent = np.zeros((R, out_width), np.int32)
        token = np.zeros((R, out_width), np.int32)
        score = np.zeros((R, out_width), np.float32)
        rc = self.lib.oracle_beam_select(R, BW, K, out_width, _p(beam_score), _p(cand_logp), _p(cand_token),
                                         _p(parent), _p(token), _p(score))
        if rc != 0:
            raise ValueError("oracle_beam_select rejected its arguments")
        return parent, token, score


def load(mutant: int = 0) -> Oracle:
    if mutant not in _cache:
        _cache[mutant] = Oracle(mutant)
    return _cache[mutant]


# -- convenience over a workload's inputs -----------------------------------------------

def dims_of(w, Lmax=None, S=None, Tmax=None) -> _Dims:
    return Oracle.dims(w.num_requests, w.beam_width, w.num_q_heads, w.num_kv_heads, w.head_dim,
                       w.max_shared_len if Lmax is None else Lmax,
                       w.ns_slots if S is None else S, w.max_steps if Tmax is None else Tmax,
                       w.softmax_scale)


def build_cache(orc: Oracle, inp, steps=None):
    """Run the oracle's beam update for steps 0 .. steps-1 over a workload's inputs and
    return (pool_k, pool_v, idx) in float32 / int32."""
    w = inp.w
    T = w.steps if steps is None else steps
    D = dims_of(w)
    pool_k = np.zeros((w.num_requests, w.ns_slots, w.num_kv_heads, w.head_dim), np.float32)
    pool_v = np.zeros_like(pool_k)
    idx = np.zeros((w.num_requests, w.beam_width, w.max_steps), np.int32)
    for s in range(T):
        orc.beam_update(D, inp.parents[s], inp.new_k[s], inp.new_v[s], pool_k, pool_v, idx, s)
    return pool_k, pool_v, idx
