#!/usr/bin/env python3
"""Benchmark of split Shared / Non-Shared beam-search decode attention on one GB300.

One step = one pass of the whole hot path over one batch:
  xattn_beam_update (the beams' newest token into the Non-Shared pool, ancestry rewrite)
  + xattn_decode (Shared stage on tensor cores, Non-Shared stage, log-sum-exp Merge).
Default workload: 8 requests x beam width 128, GQA 32/8, head_dim 128, shared prefix 2048,
3 Non-Shared tokens per beam with random ancestry, bf16 N(0,1) (synthetic, seeded).

Timing: CUDA graphs of one step per input set, replayed back to back between CUDA events;
the input sets rotate and together exceed twice the L2 size, so no step finds its inputs
in L2. Clocks are sampled with nvidia-smi during the timed region. One JSON line is printed
by rank 0.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference] [--workload NAME]

--impl reference times the fp64 CPU oracle (the plain definition) on the host cores, on a
bounded sample of the same workload per step.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode-attn beams/s and µs/step; achieved HBM GB/s as % of GB300 roofline"
NOMINAL_HBM_GBS = 8000.0
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="gr_r8_bw128_h32x8_d128_L2048_t3")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="wall budget of the CPU-baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true", help="time the default workload only")
    ap.add_argument("--configs", default="", help="comma-separated name prefixes of the other workloads to time")
    ap.add_argument("--config-cpu-seconds", type=float, default=2.5,
                    help="wall budget of each other workload's CPU-baseline sample")
    return ap.parse_args()


# ----------------------------------------------------------------------------------------
def dist_info():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(x: float, device="cpu") -> float:
    """The maximum of x over all ranks (x itself when not distributed)."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def input_seed(rank: int, set_index: int) -> int:
    """Seed of one rank's input set: every rank decodes its own batch (weak scaling)."""
    return 1000 * rank + set_index


def whole_job_beams_per_s(beams_per_rank: int, world: int, ms_per_step: float) -> float:
    """Beams decoded per second by all ranks together; ms_per_step is the max over ranks."""
    return beams_per_rank * world / (ms_per_step * 1e-3)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            d = json.load(open(path))
            out = {}
            for k in FALLBACK:
                v = d.get(k)
                if isinstance(v, dict):
                    v = v.get("value")
                if v is not None:
                    out[k] = float(v)
            if "hbm_gbs" in out and "bf16_tflops" in out:
                out.setdefault("bf16_tflops_sustained", out["bf16_tflops"])
                return out, "measured"
        except Exception:
            pass
    return dict(FALLBACK), "fallback"


class ClockSampler:
    """nvidia-smi samples (SM clock, max clock, throttle reasons) while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 6:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[2:6]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------------------
def unique_bytes(w, idx_np, shared_lens, elem=2):
    """Bytes the step must move at least once: prefix K/V over valid tokens (once per
    request), the distinct Non-Shared pool rows the ancestry references, q, out, lse and the
    ancestry entries read. elem: bytes per stored q/K/V element (2 bf16, 4 fp32)."""
    import numpy as np

    d, Hkv = w.head_dim, w.num_kv_heads
    prefix = int(sum(shared_lens)) * Hkv * d * 2 * elem
    T = w.steps
    distinct = sum(len(np.unique(idx_np[r, :, :T])) for r in range(w.num_requests)) if T > 0 else 0
    ns = distinct * Hkv * d * 2 * elem
    rows = w.num_requests * w.beam_width * w.num_q_heads
    q = rows * d * elem
    out = rows * d * 2 + rows * 4
    idx = w.num_requests * w.beam_width * T * 4
    return prefix + ns + q + out + idx, {"prefix_kv": prefix, "ns_kv": ns, "q": q, "out_lse": out, "idx": idx}


def shared_stage_flops(w):
    """Algorithmic FLOPs of the Shared stage: two matmuls of M x L x d per (request, KV head)."""
    M = w.beam_width * w.group_size
    return sum(4.0 * M * L * w.head_dim * w.num_kv_heads for L in w.shared_lens)


def shared_stage_bytes(w, plan):
    M = w.beam_width * w.group_size
    kv = sum(w.shared_lens) * w.num_kv_heads * w.head_dim * 2 * 2
    q = w.num_requests * w.beam_width * w.num_q_heads * w.head_dim * 2
    parts = w.num_requests * w.num_kv_heads * plan.num_splits * M * (w.head_dim + 1) * 4
    return kv + q + parts


def profile_traffic(kernel_file: str, workload: str):
    """dram bytes per launch from the committed ncu summary, if it was taken on the
    current source of the kernel; else None."""
    path = os.path.join(ROOT, "profiles", f"{os.path.splitext(os.path.basename(kernel_file))[0]}__{workload}.md")
    if not os.path.exists(path):
        return None
    src = os.path.join(ROOT, "decode_attention_xattention_gb300", "csrc", kernel_file)
    sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    traffic, src_sha = None, None
    for line in open(path):
        if line.startswith("traffic_bytes_per_launch:"):
            traffic = float(line.split(":", 1)[1].strip())
        if line.startswith("kernel_source_sha256_16:"):
            src_sha = line.split(":", 1)[1].strip()
    return traffic if (traffic is not None and src_sha == sha) else None


def launches_per_step(plan, step, f32=False):
    """Kernels of this library launched by one timed step (xattn_decode_step): the beam update,
    then the decode (the Shared-stage kernel alone when it takes the Non-Shared part in its own
    tile; the Non-Shared kernel + Shared stage with merging epilogue when fused; else
    the Shared stage, if the prefix has storage, and the Non-Shared/Merge kernel, or two
    kernels, the Non-Shared part as pieces and the row merge, when the Non-Shared part is long
    or, with bf16 storage, sits next to a prefix cut in pieces)."""
    if plan.ns_tile:  # the beam update, then the decode as its programmatic dependent
        return 2
    n = 1
    if plan.fused:
        n += (1 if step > 0 else 0) + 1
    else:
        split_short = (not f32 and plan.shared_kernel != 0 and plan.num_splits > 1 and 0 < step <= 32)
        n += (1 if plan.shared_kernel != 0 else 0) + (2 if (step > 32 or split_short) else 1)
    return n


# ----------------------------------------------------------------------------------------
def cpu_oracle_sample(w, inp, budget_s, nthreads=0):
    """Times the fp64 oracle (as it stands; all host cores, or `nthreads`) on whole beams
    until about budget_s of wall time. Returns (beams/s, cores, description)."""
    import numpy as np

    import oracle

    orc = oracle.load()
    pk, pv, idx = oracle.build_cache(orc, inp)
    D = oracle.dims_of(w)
    Hq = w.num_q_heads
    cores = nthreads if nthreads > 0 else orc.max_threads()

    def run(nbeams, offset=0):
        b0 = offset % w.num_beams
        beams = [(b0 + i) % w.num_beams for i in range(nbeams)]
        rows = np.asarray([b * Hq + h for b in beams for h in range(Hq)], np.int64)
        t0 = time.perf_counter()
        orc.decode(D, inp.q, inp.shared_k, inp.shared_v, inp.shared_len, pk, pv, idx, w.steps, rows=rows,
                   nthreads=nthreads)
        return time.perf_counter() - t0

    t = run(1)
    n = 1
    while t < 0.2 and n < w.num_beams:
        n = min(w.num_beams, n * 4)
        t = run(n)
    rate = n / t
    nb = max(1, min(w.num_beams, int(rate * budget_s)))
    t = run(nb)
    return nb / t, cores, f"{nb} of {w.num_beams} beams (all {Hq} query heads each), one decode step, " \
                          f"{cores} OpenMP threads"


def run_reference(args, w):
    """The oracle as the reference arm: each step decodes a bounded sample of beams."""
    import numpy as np

    import oracle
    from decode_attention_xattention_gb300 import workloads as wl

    rank, world, _ = dist_info()
    if rank != 0:
        return
    inp = wl.make_inputs(w).as_bf16()
    orc = oracle.load()
    pk, pv, idx = oracle.build_cache(orc, inp)
    D = oracle.dims_of(w)
    Hq = w.num_q_heads
    cores = orc.max_threads()

    def step(nb, k):
        b0 = (k * nb) % w.num_beams
        rows = np.asarray([((b0 + i) % w.num_beams) * Hq + h for i in range(nb) for h in range(Hq)], np.int64)
        orc.decode(D, inp.q, inp.shared_k, inp.shared_v, inp.shared_len, pk, pv, idx, w.steps, rows=rows)

    t0 = time.perf_counter()
    step(1, 0)
    per_beam = max(time.perf_counter() - t0, 1e-6)
    total_budget = 120.0
    nb = int(max(1, min(w.num_beams, total_budget / max(1, args.steps + args.warmup) / per_beam)))
    for k in range(args.warmup):
        step(nb, k)
    t0 = time.perf_counter()
    for k in range(args.steps):
        step(nb, k)
    el = time.perf_counter() - t0
    value = nb * args.steps / el
    ms = el / args.steps * 1e3
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "beams/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(w),
        "cpu_baseline": {"value": value, "unit": "beams/s", "cores": cores, "kind": "oracle",
                         "sample": f"{nb} of {w.num_beams} beams per step (all {Hq} query heads each), "
                                   f"fp64 C oracle, {cores} OpenMP threads"},
        "e2e": {"value": value, "unit": "beams/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def config_of(w, extra=None):
    c = {"workload": w.name, "requests": w.num_requests, "beam_width": w.beam_width, "q_heads": w.num_q_heads,
         "kv_heads": w.num_kv_heads, "head_dim": w.head_dim, "shared_prefix": list(w.shared_lens),
         "ns_tokens_per_beam": w.steps}
    if extra:
        c.update(extra)
    return c


# ----------------------------------------------------------------------------------------
def time_beam_select(device, stream, with_oracle: bool) -> dict:
    """The beam selection (xGR section 2.2, xBeam) timed alone through the C ABI on the
    pages' two candidate-pool sizes (128 x 128 and 512 x 512 per request), CUDA events over
    200 calls on the launching stream; inputs (0.5 / 4 MB) stay in L2. With `with_oracle`,
    the oracle's full sort of the same call is timed on the host beside it."""
    import torch

    import oracle
    from decode_attention_xattention_gb300 import workloads as wl, xattn

    out = {"note": "not part of the decode step; per-beam sorted synthetic candidate lists, L2-resident"}
    for name, (R, BW, K, Wd) in (("pool_128x128", (8, 128, 128, 128)), ("pool_512x512", (4, 512, 512, 512))):
        bs, lp, tok = wl.make_candidates(R, BW, K, seed=7)
        d_bs, d_lp, d_tok = (torch.from_numpy(a).to(device) for a in (bs, lp, tok))
        par = torch.empty((R, Wd), dtype=torch.int32, device=device)
        tk = torch.empty_like(par)
        sc = torch.empty((R, Wd), dtype=torch.float32, device=device)

        def call():
            xattn.check(xattn.xattn_beam_select(R, BW, K, Wd, d_bs, d_lp, d_tok, par, tk, sc, stream))

        n = 200
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            for _ in range(5):
                call()
            e0.record(stream)
            for _ in range(n):
                call()
            e1.record(stream)
        e1.synchronize()
        us = e0.elapsed_time(e1) / n * 1e3
        entry = {"requests": R, "beam_width": BW, "cand_per_beam": K, "out_width": Wd, "us_per_call": us,
                 "beams_selected_per_s": R * Wd / (us * 1e-6), "gpu_launches_per_call": 1}
        if with_oracle:
            orc = oracle.load()
            t0 = time.perf_counter()
            orc.beam_select(bs, lp, tok, Wd)
            entry["oracle_us_per_call"] = (time.perf_counter() - t0) * 1e6
            entry["oracle_cores"] = 1
        out[name] = entry
    return out


def time_cht(with_oracle: bool) -> dict:
    """The chunked hash tree (Feather's prefix-aware batching structure, host code) timed on
    the host through its binding: 4096 waiting prompts of 1280-2304 tokens in 8 prefix
    groups (blocks of 16 tokens), then batches of 64 formed by best + admit and released by
    finish until the queue is empty. With `with_oracle`, one brute-force `best` over 256
    waiting and 8 active prompts of the same kind is timed beside it."""
    import numpy as np

    from decode_attention_xattention_gb300.cht import ChunkedHashTree

    rng = np.random.default_rng(3)
    B, n, groups, batch = 16, 4096, 8, 64
    bases = [rng.integers(0, 32000, size=2048).astype(np.int32) for _ in range(groups)]
    prompts = [np.concatenate([bases[i % groups][: int(rng.integers(1024, 2049))],
                               rng.integers(0, 32000, size=256).astype(np.int32)]) for i in range(n)]
    t = ChunkedHashTree(B)
    t0 = time.perf_counter()
    for i, p in enumerate(prompts):
        t.insert(i, p)
    t_insert = time.perf_counter() - t0
    t_pick = t_finish = 0.0
    picks = 0
    while True:
        chosen = []
        t0 = time.perf_counter()
        for _ in range(batch):
            rc, rid, _ = t.best()
            if rc != 1:
                break
            t.admit(rid)
            chosen.append(rid)
        t_pick += time.perf_counter() - t0
        picks += len(chosen)
        if not chosen:
            break
        t0 = time.perf_counter()
        for rid in chosen:
            t.finish(rid)
        t_finish += time.perf_counter() - t0
    out = {"note": "host code through the ctypes binding (a call costs about 1 us of Python itself)",
           "waiting": n, "block_tokens": B, "batch": batch,
           "insert_us_per_request": t_insert / n * 1e6, "best_admit_us_per_request": t_pick / picks * 1e6,
           "finish_us_per_request": t_finish / picks * 1e6}
    if with_oracle:
        from oracle.cht import BruteForceScheduler

        bf = BruteForceScheduler(B)
        for i in range(256):
            bf.insert(i, prompts[i].tolist())
        for i in range(8):
            bf.admit(i)
        t0 = time.perf_counter()
        bf.best()
        out["oracle_best_us_at_256_waiting_8_active"] = (time.perf_counter() - t0) * 1e6
    return out


def time_valid_path(device, stream, with_oracle: bool) -> dict:
    """The valid-path masks timed through the C ABI on a synthetic catalogue: 262144 items as
    3-token paths over V = 8192 tokens, 1024 rows (8 requests x 128 beams) following item
    paths; the dense mask at step 0 (about every token valid) and the sparse best-128 list at
    step 1 (about 32 valid tokens per row), CUDA events over 100 calls each."""
    import numpy as np
    import torch

    from decode_attention_xattention_gb300 import xattn

    rng = np.random.default_rng(4)
    N, L, V, rows, C = 262144, 3, 8192, 1024, 128
    items = rng.integers(0, V, size=(N, L)).astype(np.int32)
    t0 = time.perf_counter()
    off, tok = xattn.trie_build(items)
    t_build = time.perf_counter() - t0
    pre = items[rng.integers(0, N, size=rows)].copy()
    logp = rng.standard_normal((rows, V)).astype(np.float32)
    d_off, d_tok, d_pre, d_logp = (torch.from_numpy(np.ascontiguousarray(a)).to(device) for a in (off, tok, pre, logp))
    nodes = len(off) - 1
    ct = torch.empty((rows, C), dtype=torch.int32, device=device)
    cl = torch.empty((rows, C), dtype=torch.float32, device=device)
    cnt = torch.empty((rows,), dtype=torch.int32, device=device)
    st = torch.zeros((1,), dtype=torch.int32, device=device)

    def timed(fn, n=100):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            for _ in range(3):
                fn()
            e0.record(stream)
            for _ in range(n):
                fn()
            e1.record(stream)
        e1.synchronize()
        return e0.elapsed_time(e1) / n * 1e3

    us_dense = timed(lambda: xattn.check(xattn.xattn_valid_path_mask(d_off, d_tok, nodes, L, d_pre, L, 0, rows, V,
                                                                     d_logp, cnt, st, stream)))
    dense_valid = float(cnt.float().mean().item())
    us_sparse = timed(lambda: xattn.check(xattn.xattn_valid_path_topk(d_off, d_tok, nodes, L, d_pre, L, 1, rows, V,
                                                                      d_logp, C, ct, cl, cnt, st, stream)))
    out = {"note": "not part of the decode step; synthetic catalogue",
           "items": N, "path_len": L, "V": V, "rows": rows, "trie_nodes": nodes, "trie_build_ms_host": t_build * 1e3,
           "dense_step0": {"us_per_call": us_dense, "mean_valid": dense_valid,
                           "masked_per_row": V - dense_valid},
           "sparse_step1": {"us_per_call": us_sparse, "C": C, "mean_valid": float(cnt.float().mean().item())},
           "status": int(st.item())}
    if with_oracle:
        from oracle.valid_path import valid_next

        t0 = time.perf_counter()
        valid_next(items, pre[0], 1)
        out["oracle_us_per_row_step1"] = (time.perf_counter() - t0) * 1e6
    return out


# The measured configuration list, in order: the default (headline) workload first.
CONFIG_ORDER = ["gr_r8_bw128_h32x8_d128_L2048_t3", "tiny_r1_bw4_h2x1_d64_L256_t3", "wide_r4_bw512_h16x4_d128_L4096_t4",
                "long_r2_bw256_h32x8_d128_L32768+20000_t8", "feather_g1_seq64_h32x8_d128_L8192_s512",
                "feather_g8_seq64_h32x8_d128_L8192_s512", "feather_g64_seq64_h32x8_d128_L8192_s512"]
FP32_ALU_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12  # 152 SMs x 128 fp32 FMA lanes x 2 flop x 2.07 GHz
TF32_OVER_BF16 = 1.1 / 2.25  # nominal dense tf32 / bf16 tensor rates (the measured peak is bf16)


def ns_merge_bytes(w, plan, idx_np, elem):
    """Algorithmic bytes of the Non-Shared + Merge kernels (xattn_decode_merge): the distinct
    pool rows the ancestry references (K and V), q, the prefix pieces' partials read back,
    out and lse written, the ancestry entries read."""
    import numpy as np

    T, d, Hkv = w.steps, w.head_dim, w.num_kv_heads
    rows = w.num_requests * w.beam_width * w.num_q_heads
    distinct = sum(len(np.unique(idx_np[r, :, :T])) for r in range(w.num_requests)) if T > 0 else 0
    M = w.beam_width * w.group_size
    parts = w.num_requests * Hkv * plan.num_splits * M * (d + 1) * 4
    return distinct * Hkv * d * 2 * elem + rows * d * elem + parts + rows * (d * 2 + 4) + \
        w.num_requests * w.beam_width * T * 4


def beam_update_bytes(w, elem):
    """Algorithmic bytes of one beam update: the BW new tokens' K/V read and written into the
    pool, the ancestry table read and rewritten, the parents read."""
    R, BW, T = w.num_requests, w.beam_width, w.steps
    return 2 * R * BW * w.num_kv_heads * w.head_dim * 2 * elem + 2 * R * BW * T * 4 + R * BW * 4


def measure_config(w, local, stream, peaks, peak_src, l2, cpu_budget_s, target_s=0.3, shared_kernel=0):
    """One workload measured the way the headline line is: CUDA-graph replays of one step
    (beam update + decode) on inputs resident in HBM, with either rotating copies of the
    inputs that together exceed twice the L2, or (small workloads) the L2 flushed before
    every timed step; each stage timed alone the same way; the roofline of the dominant
    kernel; the oracle timed on a bounded sample of beams (all host cores)."""
    import numpy as np
    import torch

    from decode_attention_xattention_gb300 import workloads as wl, xattn
    from decode_attention_xattention_gb300.runner import DeviceBatch

    T = w.steps
    f32 = w.input_dtype == "fp32"
    elem = 4 if f32 else 2
    inp = wl.make_inputs(w)
    if not f32:
        inp = inp.as_bf16()
    base = DeviceBatch(inp, device=f"cuda:{local}", stream=stream, input_f32=f32, shared_kernel=shared_kernel)
    with torch.cuda.stream(stream):
        base.build_cache(steps=T - 1)
    set_bytes = sum(t.numel() * t.element_size() for t in
                    (base.q, base.shared_k, base.shared_v, base.pool_k, base.pool_v, base.out, base.lse,
                     base.workspace) if t is not None)
    flush = set_bytes * 8 < l2  # too small to rotate past the L2: flush it before each step
    sets = [base]
    while not flush and (len(sets) < 2 or len(sets) * set_bytes < 2 * l2):
        sets.append(base.clone())
    nsets = len(sets)
    plan = base.plan()
    flush_buf = torch.empty(int(2 * l2) // 4 + 1, dtype=torch.int32, device=f"cuda:{local}") if flush else None

    def step(db):  # token T-1's bookkeeping + the decode over tokens 0..T-1
        xattn.check(db.decode_step(T - 1))

    with torch.cuda.stream(stream):
        for db in sets:
            step(db)
            if w.max_shared_len > 0:
                xattn.check(db.decode_shared())
            if not plan.fused:
                xattn.check(db.decode_merge())
            xattn.check(db.beam_update(T - 1))
    stream.synchronize()
    for db in sets:
        assert db.read_status() == 0, f"{w.name}: device status set"

    def capture(fn):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            fn()
        return g

    graphs = {"step": [capture(lambda db=db: step(db)) for db in sets],
              "decode": [capture(lambda db=db: xattn.check(db.decode())) for db in sets],
              "beam_update": [capture(lambda db=db: xattn.check(db.beam_update(T - 1))) for db in sets]}
    if w.max_shared_len > 0:
        graphs["shared_stage_alone"] = [capture(lambda db=db: xattn.check(db.decode_shared())) for db in sets]
    if not plan.fused:
        graphs["merge_alone"] = [capture(lambda db=db: xattn.check(db.decode_merge())) for db in sets]

    def timed(gs, K, W=3):
        with torch.cuda.stream(stream):
            for k in range(W):
                if flush:
                    flush_buf.zero_()
                gs[k % nsets].replay()
        stream.synchronize()
        if not flush:
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                e0.record(stream)
                for k in range(K):
                    gs[k % nsets].replay()
                e1.record(stream)
            e1.synchronize()
            return e0.elapsed_time(e1) / K
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
        with torch.cuda.stream(stream):
            for k in range(K):
                flush_buf.zero_()
                ev[k][0].record(stream)
                gs[k % nsets].replay()
                ev[k][1].record(stream)
        stream.synchronize()
        return sum(a.elapsed_time(b) for a, b in ev) / K

    est = timed(graphs["step"], 20)
    K = int(max(200, min(20000, target_s / max(est * 1e-3, 1e-6))))
    if flush:
        K = min(K, 2000)
    ms = {name: timed(gs, K if name == "step" else max(200, K // 2)) for name, gs in graphs.items()}
    for db in sets:
        assert db.read_status() == 0, f"{w.name}: device status set during timing"

    idx_np = base.idx.cpu().numpy()
    ub, ub_parts = unique_bytes(w, idx_np, inp.shared_len, elem)
    flops = shared_stage_flops(w)
    kernels = {}
    if "shared_stage_alone" in ms:
        M = w.beam_width * w.group_size
        sbytes = sum(w.shared_lens) * w.num_kv_heads * w.head_dim * 2 * elem + \
            w.num_requests * w.beam_width * w.num_q_heads * w.head_dim * elem + \
            w.num_requests * w.num_kv_heads * plan.num_splits * M * (w.head_dim + 1) * 4
        kernels["shared_stage_alone"] = (
            {1: "shared_stage_tc", 2: "shared_stage_simt", 3: "shared_stage_tf32"}[plan.shared_kernel], flops, sbytes,
            "tensor" if plan.shared_kernel in (1, 3) else "alu")
    if "merge_alone" in ms:
        kernels["merge_alone"] = ("ns_merge", 0.0, ns_merge_bytes(w, plan, idx_np, elem), None)
    kernels["beam_update"] = ("beam_update", 0.0, beam_update_bytes(w, elem), None)
    dom = max(kernels, key=lambda k: ms[k])
    kname, kflops, kbytes, compute_kind = kernels[dom]
    t_hbm = kbytes / (peaks["hbm_gbs"] * 1e9)
    tf32 = plan.shared_kernel == 3
    cpeak = (peaks["bf16_tflops"] * (TF32_OVER_BF16 if tf32 else 1.0)) if compute_kind == "tensor" else FP32_ALU_TFLOPS
    t_c = kflops / (cpeak * 1e12) if kflops > 0 else 0.0
    s_k = ms[dom] * 1e-3
    if t_c > t_hbm:
        roof = {"kernel": kname, "stage": dom, "bound": compute_kind, "achieved": kflops / s_k / 1e12,
                "peak": cpeak, "unit": "TFLOP/s", "frac": kflops / s_k / 1e12 / cpeak,
                "algorithmic_per_launch": kflops,
                "peak_source": (f"{peak_src} bf16 burst x 1.1/2.25 (nominal tf32/bf16)" if tf32 else
                                f"{peak_src} (burst; kernel timed alone)") if compute_kind == "tensor" else
                "fp32 FMA issue rate: 152 SMs x 128 lanes x 2 flop x 2.07 GHz"}
    else:
        roof = {"kernel": kname, "stage": dom, "bound": "hbm", "achieved": kbytes / s_k / 1e9,
                "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": kbytes / s_k / 1e9 / peaks["hbm_gbs"],
                "algorithmic_per_launch": kbytes, "peak_source": f"{peak_src} (copy bandwidth)"}
    src = {"shared_stage_tc": "shared_stage_tc.cu", "shared_stage_simt": "shared_stage_simt.cu",
           "shared_stage_tf32": "shared_stage_tf32.cu", "ns_merge": "ns_merge.cu", "beam_update": "beam_update.cu"}[kname]
    roof["traffic"] = profile_traffic(src, w.name)
    step_s = ms["step"] * 1e-3
    t_bind = max(ub / (peaks["hbm_gbs"] * 1e9), flops / (peaks["bf16_tflops"] * 1e12))
    entry = {
        "config": config_of(w, {"shared_splits": plan.num_splits, "split_tokens": plan.split_tokens,
                                "shared_kernel": {0: "none", 1: "tcgen05", 2: "cuda-core",
                                                  3: "tcgen05-tf32"}[plan.shared_kernel],
                                "fused_ns_merge": bool(plan.fused), "dtype": "f32" if f32 else "bf16"}),
        "l2": (f"L2 flushed (a {flush_buf.numel() * 4 / 1e6:.0f} MB write) before every timed step; per-step CUDA "
               f"events" if flush else f"{nsets} rotating copies of the {set_bytes / 1e6:.0f} MB input set "
                                       f"(> 2x the {l2 / 1e6:.0f} MB L2); CUDA graph replays between CUDA events"),
        "steps_timed": K,
        "us_per_step": ms["step"] * 1e3,
        "beams_per_s": w.num_beams / step_s,
        "attention_us_per_step": ms["decode"] * 1e3,
        "stage_us": {k: v * 1e3 for k, v in ms.items() if k != "step"},
        "hbm": {"unique_bytes_per_step": ub, "parts": ub_parts, "achieved_gbs": ub / step_s / 1e9,
                "frac_of_8tbs": ub / step_s / 1e9 / NOMINAL_HBM_GBS,
                "frac_of_peak": ub / step_s / 1e9 / peaks["hbm_gbs"]},
        "tensor": {"shared_stage_flops": flops,
                   "frac_of_peak": (flops / (ms["shared_stage_alone"] * 1e-3) / 1e12 / peaks["bf16_tflops"]
                                    if "shared_stage_alone" in ms and plan.shared_kernel == 1 else None)},
        "binding_roofline_frac": t_bind / step_s,
        "roofline": roof,
        "gpu_launches_per_step": launches_per_step(plan, T, f32),
    }
    if cpu_budget_s > 0:
        v, cores, sample = cpu_oracle_sample(w, inp, cpu_budget_s)
        entry["cpu_baseline"] = {"value": v, "unit": "beams/s", "cores": cores, "kind": "oracle", "sample": sample}
    del sets, graphs, base
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return entry


def main():
    args = parse_args()
    from decode_attention_xattention_gb300 import workloads as wl

    if args.workload not in wl.ALL:
        sys.exit(f"unknown workload {args.workload}; choose from {sorted(wl.ALL)}")
    w = wl.ALL[args.workload]
    if args.impl == "reference":
        run_reference(args, w)
        return

    import numpy as np
    import torch
    import torch.distributed as dist

    from decode_attention_xattention_gb300 import build as xbuild, xattn
    from decode_attention_xattention_gb300.runner import DeviceBatch

    rank, world, local = dist_info()
    if world > 1:
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    xbuild.build()
    xattn.load()
    T = w.steps
    peaks, peak_src = load_peaks()

    # -- input sets: enough copies that rotating through them defeats the L2 ------------
    l2 = torch.cuda.get_device_properties(local).L2_cache_size if hasattr(
        torch.cuda.get_device_properties(local), "L2_cache_size") else 128 << 20
    stream = torch.cuda.Stream()
    sets, inputs = [], []
    set_bytes = None
    while True:
        seed = input_seed(rank, len(sets))
        inp = wl.make_inputs(w, seed=seed).as_bf16()
        db = DeviceBatch(inp, device=f"cuda:{local}", stream=stream)
        with torch.cuda.stream(stream):
            db.build_cache(steps=T - 1)  # the timed step writes token T-1 itself
        sets.append(db)
        inputs.append(inp)
        if set_bytes is None:
            set_bytes = sum(t.numel() * t.element_size() for t in
                            (db.q, db.shared_k, db.shared_v, db.pool_k, db.pool_v, db.out, db.lse, db.workspace)
                            if t is not None)
        if len(sets) >= 2 and len(sets) * set_bytes >= 2 * l2:
            break
    nsets = len(sets)
    plan = sets[0].plan()

    def step(db):  # token T-1's bookkeeping + the decode over tokens 0..T-1
        xattn.check(db.decode_step(T - 1))

    # eager warm-up of every call (also sets kernel attributes before capture)
    with torch.cuda.stream(stream):
        for db in sets:
            step(db)
            xattn.check(db.decode_shared())
            xattn.check(db.decode_merge())
            xattn.check(db.beam_update(T - 1))
    stream.synchronize()
    for db in sets:
        assert db.read_status() == 0

    def capture(fn):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            fn()
        return g

    g_step = [capture(lambda db=db: step(db)) for db in sets]
    g_bu = [capture(lambda db=db: xattn.check(db.beam_update(T - 1))) for db in sets]
    g_decode = [capture(lambda db=db: xattn.check(db.decode())) for db in sets]
    # The dominant kernel is the Shared stage's tensor-core kernel; xattn_decode_shared runs
    # it alone (same main loop; its epilogue writes the prefix piece instead of merging).
    g_dominant = [capture(lambda db=db: xattn.check(db.decode_shared())) for db in sets]
    g_merge = None if plan.fused else [capture(lambda db=db: xattn.check(db.decode_merge())) for db in sets]

    def timed(graphs, K, W):
        with torch.cuda.stream(stream):
            for k in range(W):
                graphs[k % nsets].replay()
        stream.synchronize()
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for k in range(K):
                graphs[k % nsets].replay()
            e1.record(stream)
        e1.synchronize()
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        return max_over_ranks(e0.elapsed_time(e1), f"cuda:{local}")

    K, W = args.steps, max(3, args.warmup)
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    total_ms = timed(g_step, K, W)
    clocks = sampler.stop()
    ms_step = total_ms / K

    # per-kernel average launch durations (each alone, same rotation of input sets)
    Kk = max(200, min(K, 5000))
    ms_dom = timed(g_dominant, Kk, W) / Kk
    ms_merge = timed(g_merge, Kk, W) / Kk if g_merge else 0.0
    ms_bu = timed(g_bu, Kk, W) / Kk
    ms_decode = timed(g_decode, Kk, W) / Kk
    for db in sets:
        assert db.read_status() == 0, "device status set during the bench"

    # -- end to end through the C ABI with host buffers ----------------------------------
    db = sets[0]
    inp = inputs[0]
    from decode_attention_xattention_gb300.runner import to_bf16_tensor

    h_q = to_bf16_tensor(inp.q, "cpu").pin_memory()
    h_nk = to_bf16_tensor(inp.new_k[T - 1], "cpu").pin_memory()
    h_nv = to_bf16_tensor(inp.new_v[T - 1], "cpu").pin_memory()
    h_par = torch.from_numpy(inp.parents[T - 1].astype(np.int32)).pin_memory()
    h_out = torch.empty(db.out.shape, dtype=db.out.dtype).pin_memory()
    h_lse = torch.empty(db.lse.shape, dtype=db.lse.dtype).pin_memory()
    d_nk, d_nv, d_par = db.new_k[T - 1], db.new_v[T - 1], db.parents[T - 1]
    h2d = sum(t.numel() * t.element_size() for t in (h_q, h_nk, h_nv, h_par))
    d2h = h_out.numel() * h_out.element_size() + h_lse.numel() * h_lse.element_size()

    def e2e_step():
        db.q.copy_(h_q, non_blocking=True)
        d_nk.copy_(h_nk, non_blocking=True)
        d_nv.copy_(h_nv, non_blocking=True)
        d_par.copy_(h_par, non_blocking=True)
        xattn.check(db.decode_step(T - 1))
        h_out.copy_(db.out, non_blocking=True)
        h_lse.copy_(db.lse, non_blocking=True)

    Ke = max(50, min(K, 2000))
    with torch.cuda.stream(stream):
        for _ in range(W):
            e2e_step()
    stream.synchronize()
    if world > 1:
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(Ke):
            e2e_step()
        e1.record(stream)
    e1.synchronize()
    ms_e2e = max_over_ranks(e0.elapsed_time(e1) / Ke, f"cuda:{local}")

    # -- the same end-to-end step, pipelined across steps: while step k computes, step k+1's
    #    inputs go up and step k-1's results come down (two slots of device inputs and
    #    outputs, one upload and one readback stream). Every step still copies its own
    #    inputs from pinned host memory and reads its own out / lse back.
    # Two pipelined schedules. Both alternate two slots of device inputs and outputs, so
    # that the upload of step k+1 and the readback of step k-1 overlap step k, and every step
    # still copies its own inputs from pinned host memory and reads its own out / lse back.
    #  eager: each step's calls issued from the host; one upload and one readback stream,
    #         one copy per tensor.
    #  graph: GRAPH_STEPS steps captured once as a CUDA graph (the library's calls are
    #         capturable) and replayed; the upload is cut into ~1 MB pieces over NU streams
    #         and the readback over ND, so several copy engines move them at once.
    NU, ND, GRAPH_STEPS = 4, 2, 16
    dev = f"cuda:{local}"
    ups = [torch.cuda.Stream(device=dev) for _ in range(NU)]
    downs = [torch.cuda.Stream(device=dev) for _ in range(ND)]
    slots = [{"q": torch.empty_like(db.q), "nk": torch.empty_like(d_nk), "nv": torch.empty_like(d_nv),
              "par": torch.empty_like(d_par), "out": torch.empty_like(db.out), "lse": torch.empty_like(db.lse)}
             for _ in range(2)]
    h_outs = [h_out, torch.empty_like(h_out).pin_memory()]
    h_lses = [h_lse, torch.empty_like(h_lse).pin_memory()]

    def chunks(t, n):
        return list(torch.chunk(t, n, dim=0)) if (n > 1 and t.shape[0] >= n) else [t]

    def upload_plan(sl, nu, fine):
        pieces = list(zip(chunks(sl["q"], w.num_requests if fine else 1), chunks(h_q, w.num_requests if fine else 1)))
        pieces += list(zip(chunks(sl["nk"], 2 if fine else 1), chunks(h_nk, 2 if fine else 1)))
        pieces += list(zip(chunks(sl["nv"], 2 if fine else 1), chunks(h_nv, 2 if fine else 1)))
        pieces.append((sl["par"], h_par))
        return [pieces[i::nu] for i in range(nu)]

    def readback_plan(sl, ho, hl, nd, fine):
        pieces = list(zip(chunks(ho, 2 * nd if fine else 1), chunks(sl["out"], 2 * nd if fine else 1)))
        pieces.append((hl, sl["lse"]))
        return [pieces[i::nd] for i in range(nd)]

    def e2e_pipelined(n, collect=None, graph=False):
        """Enqueue n pipelined steps (graph: NU / ND streams and fine pieces, for capture)."""
        nu, nd = (NU, ND) if graph else (1, 1)
        us_, ds_ = ups[:nu], downs[:nd]
        up_done = [[torch.cuda.Event() for _ in range(nu)] for _ in range(2)]
        comp_done = [torch.cuda.Event() for _ in range(2)]
        down_done = [[torch.cuda.Event() for _ in range(nd)] for _ in range(2)]
        start = torch.cuda.Event()
        start.record(stream)
        for k in range(n):
            s = k % 2
            sl = slots[s]
            plan_up = upload_plan(sl, nu, graph)
            for i, us in enumerate(us_):
                us.wait_event(start if k < 2 else comp_done[s])  # the slot's inputs were read by step k-2
                with torch.cuda.stream(us):
                    for dst, src in plan_up[i]:
                        dst.copy_(src, non_blocking=True)
                    up_done[s][i].record(us)
            for i in range(nu):
                stream.wait_event(up_done[s][i])
            if k >= 2:
                for j in range(nd):
                    stream.wait_event(down_done[s][j])  # the slot's outputs were read back by step k-2
            with torch.cuda.stream(stream):
                xattn.check(xattn.xattn_decode_step(db.desc, sl["par"] if T > 1 else None, sl["nk"], sl["nv"],
                                                    sl["q"], db.shared_k, db.shared_v, db.shared_len, db.pool_k,
                                                    db.pool_v, db.idx, T, sl["out"], sl["lse"], db.workspace,
                                                    db.ws_bytes, stream))
                comp_done[s].record(stream)
            ho, hl = collect[k] if collect is not None else (h_outs[s], h_lses[s])
            plan_dn = readback_plan(sl, ho, hl, nd, graph)
            for j, ds in enumerate(ds_):
                ds.wait_event(comp_done[s])
                with torch.cuda.stream(ds):
                    for dst, src in plan_dn[j]:
                        dst.copy_(src, non_blocking=True)
                    down_done[s][j].record(ds)
        for x in us_ + ds_:  # join every side stream back into `stream`
            ev = torch.cuda.Event()
            ev.record(x)
            stream.wait_event(ev)

    def capture_pipeline(n, collect=None):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            e2e_pipelined(n, collect, graph=True)
        return g

    def pipelined_e2e_checked_and_timed():
        """Bitwise check of both pipelined schedules against the serial one, then their
        timings; returns (checks passed, eager ms per step, graph ms per step)."""
        torch.cuda.synchronize()
        state = [t.clone() for t in (db.pool_k, db.pool_v, db.idx)]
        n_chk = 6
        serial = []
        with torch.cuda.stream(stream):
            for _ in range(n_chk):
                e2e_step()
                stream.synchronize()
                serial.append((h_out.clone(), h_lse.clone()))

        def restore():
            torch.cuda.synchronize()
            for t, s0 in zip((db.pool_k, db.pool_v, db.idx), state):
                t.copy_(s0)
            torch.cuda.synchronize()

        def same(piped):
            return all(torch.equal(a[0], b_[0]) and torch.equal(a[1], b_[1]) for a, b_ in zip(serial, piped))

        restore()
        piped = [(torch.empty_like(h_out).pin_memory(), torch.empty_like(h_lse).pin_memory()) for _ in range(n_chk)]
        e2e_pipelined(n_chk, piped)
        torch.cuda.synchronize()
        ok_eager = same(piped) and db.read_status() == 0
        restore()
        piped_g = [(torch.empty_like(h_out).pin_memory(), torch.empty_like(h_lse).pin_memory()) for _ in range(n_chk)]
        gchk = capture_pipeline(n_chk, piped_g)
        gchk.replay()
        torch.cuda.synchronize()
        ok_graph = same(piped_g) and db.read_status() == 0
        ms_eager = ms_graph = None
        if ok_eager:
            e2e_pipelined(W)
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            e2e_pipelined(Ke)  # every side stream joins `stream` at the end
            e1.record(stream)
            e1.synchronize()
            ms_eager = max_over_ranks(e0.elapsed_time(e1) / Ke, f"cuda:{local}")
        if ok_graph:
            gt = capture_pipeline(GRAPH_STEPS)
            for _ in range(2):
                gt.replay()
            torch.cuda.synchronize()
            reps = max(4, Ke // GRAPH_STEPS)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(reps):
                gt.replay()
            e1.record(stream)
            e1.synchronize()
            ms_graph = max_over_ranks(e0.elapsed_time(e1) / (reps * GRAPH_STEPS), f"cuda:{local}")
        return (ok_eager, ok_graph), ms_eager, ms_graph

    # self-check before timing: the pipelined steps give, bit for bit, the serial steps'
    # results from the same starting state (the kernels are deterministic)
    oks, ms_pipe, ms_graph, pipe_err = (False, False), None, None, None
    try:
        oks, ms_pipe, ms_graph = pipelined_e2e_checked_and_timed()
    except Exception as ex:  # reported in the JSON line; the serial figure stands
        torch.cuda.synchronize()
        pipe_err = repr(ex)[:300]
    e2e_candidates = [("serial", ms_e2e)] + ([("eager_pipelined", ms_pipe)] if ms_pipe else []) + \
        ([("graph_pipelined", ms_graph)] if ms_graph else [])
    e2e_kind, e2e_ms = min(e2e_candidates, key=lambda kv: kv[1])

    # -- derived figures ------------------------------------------------------------------
    beams = w.num_beams * world
    ub, ub_parts = unique_bytes(w, db.idx.cpu().numpy(), inp.shared_len)
    flops = shared_stage_flops(w)
    sbytes = ub if plan.fused else shared_stage_bytes(w, plan)  # fused: the kernel moves the step's unique bytes
    t_tc = flops / (peaks["bf16_tflops"] * 1e12)
    t_hbm = sbytes / (peaks["hbm_gbs"] * 1e9)
    bound = "tensor" if t_tc >= t_hbm else "hbm"
    s_shared = ms_dom * 1e-3
    if bound == "tensor":
        achieved, peak, unit = flops / s_shared / 1e12, peaks["bf16_tflops"], "TFLOP/s"
    else:
        achieved, peak, unit = sbytes / s_shared / 1e9, peaks["hbm_gbs"], "GB/s"
    kernel_file = "shared_stage_tc.cu" if plan.shared_kernel == 1 else "shared_stage_simt.cu"
    traffic = profile_traffic(kernel_file, w.name)
    step_s = ms_step * 1e-3
    hbm_gbs = ub / step_s / 1e9
    line = {
        "metric": METRIC,
        "value": whole_job_beams_per_s(w.num_beams, world, ms_step),
        "unit": "beams/s",
        "n_gpus": world,
        "steps": K,
        "warmup": W,
        "ms_per_step": ms_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": config_of(w, {"l2": f"{nsets} rotating input sets of {set_bytes / 1e6:.0f} MB "
                                      f"(> 2x the {l2 / 1e6:.0f} MB L2)", "timing": "CUDA graph replays, CUDA events",
                                "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                                "shared_splits": plan.num_splits, "split_tokens": plan.split_tokens,
                                "shared_kernel": "tcgen05" if plan.shared_kernel == 1 else "cuda-core",
                                "fused_ns_merge": bool(plan.fused)}),
        "us_per_step": ms_step * 1e3,
        "attention_us_per_step": ms_decode * 1e3,
        "stage_us": {"beam_update": ms_bu * 1e3, "decode": ms_decode * 1e3, "shared_stage_alone": ms_dom * 1e3,
                     "merge_alone": ms_merge * 1e3,
                     "note": ("decode = one Shared-stage kernel that also gathers and attends to the "
                              "Non-Shared part" if plan.ns_tile else
                              "decode = Non-Shared piece kernel + Shared-stage kernel with merging epilogue"
                              if plan.fused else "decode = Shared-stage kernel + Non-Shared/Merge kernel")},
        "hbm": {"unique_bytes_per_step": ub, "parts": ub_parts, "achieved_gbs": hbm_gbs,
                "frac_of_8tbs": hbm_gbs / NOMINAL_HBM_GBS, "frac_of_peak": hbm_gbs / peaks["hbm_gbs"],
                "peak_gbs": peaks["hbm_gbs"], "peak_source": peak_src},
        "tensor": {"shared_stage_flops": flops, "achieved_tflops": flops / s_shared / 1e12,
                   "frac_of_peak": flops / s_shared / 1e12 / peaks["bf16_tflops"],
                   "peak_tflops": peaks["bf16_tflops"], "peak_source": peak_src},
        "binding_roofline_frac": max(ub / (peaks["hbm_gbs"] * 1e9), flops / (peaks["bf16_tflops"] * 1e12)) / step_s,
        "roofline": {"kernel": kernel_file.replace(".cu", ""), "bound": bound, "achieved": achieved, "peak": peak,
                     "unit": unit, "frac": achieved / peak, "traffic": traffic,
                     "peak_source": f"{peak_src} (burst; kernel timed alone)",
                     "algorithmic_per_launch": flops if bound == "tensor" else sbytes},
        "e2e": {"value": whole_job_beams_per_s(w.num_beams, world, e2e_ms),
                "unit": "beams/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_ms, "schedule": {
                    "serial": "each step: upload, beam update + decode, readback, one stream, calls from the host",
                    "eager_pipelined": "upload of step k+1 and readback of step k-1 overlap step k (two slots, one "
                                       "upload and one readback stream), calls from the host",
                    "graph_pipelined": f"the same pipeline, {GRAPH_STEPS} steps captured once as a CUDA graph and "
                                       f"replayed; uploads in ~1 MB pieces over {NU} streams, readback over {ND}"}[e2e_kind],
                "serial_ms_per_step": ms_e2e, "eager_pipelined_ms_per_step": ms_pipe,
                "graph_pipelined_ms_per_step": ms_graph,
                "pipeline_check": (f"bitwise equal to the serial schedule over 6 steps: eager {oks[0]}, graph {oks[1]}"
                                   if pipe_err is None else "error: " + pipe_err)},
        "gpu_launches": launches_per_step(plan, T, w.input_dtype == "fp32") * K,
        "clocks": clocks,
    }
    line["beam_select"] = time_beam_select(f"cuda:{local}", stream, rank == 0 and not args.no_cpu_baseline)
    if rank == 0:
        line["cht"] = time_cht(not args.no_cpu_baseline)
    line["valid_path"] = time_valid_path(f"cuda:{local}", stream, rank == 0 and not args.no_cpu_baseline)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, cores, sample = cpu_oracle_sample(w, inputs[0], args.cpu_seconds)
        line["cpu_baseline"] = {"value": v, "unit": "beams/s", "cores": cores, "kind": "oracle", "sample": sample}
        v1, _, sample1 = cpu_oracle_sample(w, inputs[0], args.cpu_seconds / 2, nthreads=1)
        line["cpu_baseline_1core"] = {"value": v1, "unit": "beams/s", "cores": 1, "kind": "oracle",
                                      "sample": sample1}

    # -- every other workload of the measured configuration list, each on its own ----------
    if world == 1 and not args.no_configs:
        del g_step, g_bu, g_decode, g_dominant, g_merge, sets, slots
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        names = [n for n in CONFIG_ORDER if n != w.name]
        if args.configs:
            names = [n for n in names if any(n.startswith(p) for p in args.configs.split(","))]
        sampler = ClockSampler(local)
        sampler.start()
        line["configs"] = {}
        for name in names:
            line["configs"][name] = measure_config(
                wl.ALL[name], local, stream, peaks, peak_src, l2,
                0.0 if (args.no_cpu_baseline or rank != 0) else args.config_cpu_seconds)
            if wl.ALL[name].input_dtype == "fp32":
                # fp32 storage runs on the CUDA cores by default; its tensor-core (tf32) Shared
                # stage measured the same way beside it
                e = measure_config(wl.ALL[name], local, stream, peaks, peak_src, l2, 0.0, shared_kernel=1)
                line["configs"][name]["tensor_core_tf32"] = {
                    k: e[k] for k in ("us_per_step", "beams_per_s", "stage_us", "roofline", "config")}
        line["configs_clocks"] = sampler.stop()
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
