"""The C-ABI library builds, loads without a GPU, exports every declared symbol, and rejects
bad arguments on the host before anything reaches the device (CPU only)."""

import ctypes
import os
import re

import pytest

from decode_attention_xattention_gb300 import build, xattn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = sorted(os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include"))
                 if f.endswith(".h"))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return xattn.load()


def declared_functions():
    text = "\n".join(open(h).read() for h in HEADERS)
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(xattn_\w+)\s*\(", text)))


def test_header_declares_binding_exports():
    assert declared_functions() == sorted(xattn.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_desc_layout_matches_header():
    # 13 four-byte fields
    assert ctypes.sizeof(xattn.xattn_desc) == 52
    assert ctypes.sizeof(xattn.xattn_plan) == 44


def test_status_strings(lib):
    for code in (0, -1, -2, -3, -4, -5, -6):
        assert xattn.xattn_status_string(code)
    assert xattn.xattn_status_string(-99) == "unknown status"


def _desc(**kw):
    base = dict(R=2, BW=4, Hq=8, Hkv=2, d=128, Lmax=256, S=16, Tmax=4)
    base.update(kw)
    return xattn.make_desc(base["R"], base["BW"], base["Hq"], base["Hkv"], base["d"], base["Lmax"], base["S"],
                           base["Tmax"])


@pytest.mark.parametrize("kw,code", [
    (dict(R=0), xattn.XATTN_ERR_INVALID_ARG),
    (dict(BW=0), xattn.XATTN_ERR_INVALID_ARG),
    (dict(Hq=6, Hkv=4), xattn.XATTN_ERR_INVALID_ARG),
    (dict(Lmax=-1), xattn.XATTN_ERR_INVALID_ARG),
    (dict(d=96), xattn.XATTN_ERR_UNSUPPORTED),
    (dict(Hq=6, Hkv=2), xattn.XATTN_ERR_UNSUPPORTED),
])
def test_bad_descriptor_rejected_on_host(lib, kw, code):
    d = _desc(**kw)
    assert xattn.xattn_decode_workspace_size(d) == 0
    rc = xattn.xattn_decode(d, 0x1000, 0x1000, 0x1000, 0x1000, 0x1000, 0x1000, 0x1000, 1, 0x1000, 0x1000, 0x1000,
                            1 << 20)
    assert rc == code
    rc, _ = xattn.xattn_query_plan(d, 1)
    assert rc == code


def test_bad_calls_rejected_on_host(lib):
    d = _desc()
    ws = xattn.xattn_decode_workspace_size(d)
    assert ws >= 256
    A = 0x10000  # aligned dummy address; never dereferenced: every case fails validation first
    args = [A, A, A, A, A, A, A]
    # step out of range
    assert xattn.xattn_decode(d, *args, 5, A, A, A, ws) == xattn.XATTN_ERR_INVALID_ARG
    assert xattn.xattn_decode(d, *args, -1, A, A, A, ws) == xattn.XATTN_ERR_INVALID_ARG
    # no keys at all
    d0 = _desc(Lmax=0)
    assert xattn.xattn_decode(d0, A, None, None, None, A, A, A, 0, A, A, A, ws) == xattn.XATTN_ERR_INVALID_ARG
    # missing pointers
    assert xattn.xattn_decode(d, A, None, A, A, A, A, A, 1, A, A, A, ws) == xattn.XATTN_ERR_INVALID_ARG
    assert xattn.xattn_decode(d, A, A, A, A, None, A, A, 1, A, A, A, ws) == xattn.XATTN_ERR_INVALID_ARG
    # misaligned tensors / workspace
    assert xattn.xattn_decode(d, A + 2, A, A, A, A, A, A, 1, A, A, A, ws) == xattn.XATTN_ERR_MISALIGNED
    assert xattn.xattn_decode(d, A, A, A, A, A, A, A, 1, A, A, A + 16, ws) == xattn.XATTN_ERR_MISALIGNED
    # workspace too small
    assert xattn.xattn_decode(d, *args, 1, A, A, A, ws - 1) == xattn.XATTN_ERR_WORKSPACE_TOO_SMALL
    # beam update: step range, slots, pointers
    assert xattn.xattn_beam_update(d, A, A, A, A, A, A, 4) == xattn.XATTN_ERR_INVALID_ARG
    assert xattn.xattn_beam_update(_desc(S=8), A, A, A, A, A, A, 2) == xattn.XATTN_ERR_INVALID_ARG
    assert xattn.xattn_beam_update(d, None, A, A, A, A, A, 1) == xattn.XATTN_ERR_INVALID_ARG
    assert xattn.xattn_beam_update(d, A, A + 8, A, A, A, A, 1) == xattn.XATTN_ERR_MISALIGNED


def test_split_plan_covers_prefix(lib):
    for Lmax in (128, 300, 2048, 32768):
        for split in (0, 128, 1024):
            d = xattn.make_desc(8, 128, 32, 8, 128, Lmax, 384, 3, 0.0, 0, split)
            rc, p = xattn.xattn_query_plan(d, 3)
            assert rc == 0
            assert p.split_tokens % 128 == 0 and p.split_tokens > 0
            assert (p.num_splits - 1) * p.split_tokens < Lmax <= p.num_splits * p.split_tokens
            assert p.rows_per_unit == 512 and p.row_tiles == 4
            assert p.shared_kernel == 1


def test_plan_properties_over_shapes(lib):
    """The host plan over a grid of shapes: the prefix pieces cover the prefix in whole
    128-token tiles, the decode is fused exactly when the tensor-core Shared stage has one
    piece and at most 32 Non-Shared tokens, the workspace holds every piece row the kernels
    address, and merge launches exist only when the decode is not fused."""
    import itertools
    import math
    for (R, BW, Hq, Hkv, d), Lmax, Tmax, split, kernel in itertools.product(
            [(1, 4, 2, 1, 64), (8, 128, 32, 8, 128), (2, 5, 16, 1, 128), (3, 33, 8, 8, 64)],
            [0, 1, 127, 129, 2048, 40000], [0, 1, 3, 32, 33, 64, 200], [0, 128, 640], [0, 1, 2]):
        if Lmax == 0 and Tmax == 0:
            continue
        G = Hq // Hkv
        M = BW * G
        S = BW * max(Tmax, 1)
        desc = xattn.make_desc(R, BW, Hq, Hkv, d, Lmax, S, Tmax, 0.0, kernel, split)
        for step in sorted({0, min(1, Tmax), Tmax // 2, Tmax}):
            if Lmax == 0 and step == 0:
                continue
            rc, p = xattn.xattn_query_plan(desc, step)
            assert rc == 0, (R, BW, Hq, Hkv, d, Lmax, Tmax, split, kernel, step)
            assert p.rows_per_unit == M and p.row_tiles == math.ceil(M / 128)
            if Lmax > 0:
                assert p.shared_kernel == (kernel or 1)
                assert p.split_tokens > 0 and p.split_tokens % 128 == 0
                assert (p.num_splits - 1) * p.split_tokens < Lmax <= p.num_splits * p.split_tokens
                if split:
                    assert p.split_tokens == split
            else:
                assert p.shared_kernel == 0 and p.num_splits == 0
            ns_pieces = math.ceil(Tmax / 64) if Tmax > 32 else (1 if Tmax > 0 else 0)
            assert p.piece_stride == p.num_splits + ns_pieces
            fused = p.shared_kernel == 1 and p.num_splits == 1 and step <= 32
            assert p.fused == int(fused)
            assert (p.merge_ctas == 0) == bool(p.fused)
            ws = xattn.xattn_decode_workspace_size(desc)
            rows = R * Hkv * p.piece_stride * M
            assert ws >= 256 + rows * d * 4 + rows * 4


def test_plan_with_long_non_shared_part(lib):
    """A decode whose long Non-Shared part runs beside the tensor-core Shared stage is planned
    with fewer, longer prefix pieces where that leaves the Non-Shared kernel SMs (one prefix
    group of 64 sequences, 8192-token prefix, 512-token suffixes: 16 pieces at step 0, 4 at
    step 512), never with more pieces than at step 0 (the workspace is sized by that plan),
    and only for bf16 storage on the tensor cores with more than 32 Non-Shared tokens."""
    import itertools
    d = xattn.make_desc(1, 64, 32, 8, 128, 8192, 512 * 64, 512)
    _, p0 = xattn.xattn_query_plan(d, 0)
    _, p32 = xattn.xattn_query_plan(d, 32)
    _, p512 = xattn.xattn_query_plan(d, 512)
    assert (p0.num_splits, p32.num_splits, p512.num_splits) == (16, 16, 4)
    assert p512.shared_ctas == 32 and p512.fused == 0
    ws = xattn.xattn_decode_workspace_size(d)
    for step in (0, 33, 100, 512):
        _, p = xattn.xattn_query_plan(d, step)
        rows = 1 * 8 * p.piece_stride * 64 * 4
        assert ws >= 256 + rows * 128 * 4 + rows * 4
    # the CUDA-core kernel and fp32 storage keep the step's split
    for kernel, dtype in ((2, xattn.XATTN_DTYPE_BF16), (2, xattn.XATTN_DTYPE_F32)):
        dk = xattn.make_desc(1, 64, 32, 8, 128, 8192, 512 * 64, 512, shared_kernel=kernel, dtype=dtype)
        assert xattn.xattn_query_plan(dk, 512)[1].num_splits == xattn.xattn_query_plan(dk, 0)[1].num_splits
    # never more pieces than at step 0, over a grid of shapes
    for (R, BW, Hq, Hkv), Lmax, T in itertools.product(
            [(1, 64, 32, 8), (8, 8, 32, 8), (64, 1, 32, 8), (4, 128, 16, 4), (2, 256, 32, 8)],
            [1024, 8192, 32768], [33, 100, 512]):
        dg = xattn.make_desc(R, BW, Hq, Hkv, 128, Lmax, BW * T, T)
        n0 = xattn.xattn_query_plan(dg, 0)[1].num_splits
        nT = xattn.xattn_query_plan(dg, T)[1].num_splits
        assert 1 <= nT <= n0, (R, BW, Hq, Hkv, Lmax, T, n0, nT)


def test_fp32_inputs_plan_and_limits(lib):
    """fp32 storage: by default the planner picks the CUDA-core Shared stage (fp32 throughout)
    and the unfused path; asking for tensor cores picks the tf32 kernel (3), one CTA per
    (request, KV head, piece, 128-row tile), still unfused. Non-Shared parts longer than the
    direct walk (32 tokens) are rejected before any launch, as is an unknown dtype."""
    f32 = xattn.XATTN_DTYPE_F32
    d = xattn.make_desc(1, 4, 2, 1, 64, 256, 12, 3, 0.0, 0, 0, f32, f32)
    rc, p = xattn.xattn_query_plan(d, 3)
    assert rc == 0 and p.shared_kernel == 2 and p.fused == 0
    assert xattn.xattn_decode_workspace_size(d) > 0
    d = xattn.make_desc(2, 96, 16, 4, 128, 1000, 96 * 3, 3, 0.0, 1, 256, f32, f32)
    rc, p = xattn.xattn_query_plan(d, 3)
    assert rc == 0 and p.shared_kernel == 3 and p.fused == 0 and p.ns_tile == 0
    assert p.row_tiles == 3 and p.num_splits == 4 and p.shared_ctas == 2 * 4 * 3 * 4
    assert xattn.xattn_decode_workspace_size(d) > 0
    for bad in (xattn.make_desc(1, 4, 2, 1, 64, 256, 4 * 33, 33, 0.0, 1, 0, f32, f32),
                xattn.make_desc(1, 4, 2, 1, 64, 256, 4 * 33, 33, 0.0, 0, 0, f32, f32),
                xattn.make_desc(1, 4, 2, 1, 64, 256, 12, 3, 0.0, 0, 0, f32, 7)):
        assert xattn.xattn_decode_workspace_size(bad) == 0
        rc, _ = xattn.xattn_query_plan(bad, 3)
        assert rc == xattn.XATTN_ERR_UNSUPPORTED
        assert xattn.xattn_beam_update(bad, None, 0x1000, 0x1000, 0x1000, 0x1000, 0x1000, 0) == \
            xattn.XATTN_ERR_UNSUPPORTED


def test_kernel_choice(lib):
    # tensor cores by default, also for plain per-sequence decode (4 stacked rows)
    d = xattn.make_desc(64, 1, 32, 8, 128, 8192, 512, 512)
    rc, p = xattn.xattn_query_plan(d, 512)
    assert rc == 0 and p.shared_kernel == 1 and p.rows_per_unit == 4 and p.fused == 0
    d = xattn.make_desc(64, 1, 32, 8, 128, 8192, 512, 512, 0.0, 2)
    rc, p = xattn.xattn_query_plan(d, 512)
    assert rc == 0 and p.shared_kernel == 2
    # one prefix piece and few Non-Shared tokens: one fused kernel, no merge launch
    d = xattn.make_desc(8, 128, 32, 8, 128, 2048, 384, 3)
    rc, p = xattn.xattn_query_plan(d, 3)
    assert rc == 0 and p.fused == 1 and p.merge_ctas == 0 and p.num_splits == 1


def test_beam_select_rejected_on_host(lib):
    """Sizes, pointers and alignment of the beam selection are checked before any launch."""
    f = xattn.xattn_beam_select
    P = 0x1000
    assert f(0, 4, 4, 4, P, P, P, P, P, P) == xattn.XATTN_ERR_INVALID_ARG
    assert f(1, 4, 0, 4, P, P, P, P, P, P) == xattn.XATTN_ERR_INVALID_ARG
    assert f(1, 4, 2, 9, P, P, P, P, P, P) == xattn.XATTN_ERR_INVALID_ARG      # W > BW*K
    assert f(1, 1025, 4, 4, P, P, P, P, P, P) == xattn.XATTN_ERR_UNSUPPORTED   # BW > 1024
    assert f(1, 64, 64, 1025, P, P, P, P, P, P) == xattn.XATTN_ERR_UNSUPPORTED  # W > 1024
    assert f(1, 1024, 1 << 21, 4, P, P, P, P, P, P) == xattn.XATTN_ERR_UNSUPPORTED  # BW*K > 2^30
    assert f(1, 4, 4, 4, P, None, P, P, P, P) == xattn.XATTN_ERR_INVALID_ARG
    assert f(1, 4, 4, 4, P, P + 2, P, P, P, P) == xattn.XATTN_ERR_MISALIGNED


def test_bounded_wait_check_rejected_on_host(lib):
    P = 0x1000
    assert xattn.xattn_check_bounded_wait(1000, None) == xattn.XATTN_ERR_INVALID_ARG
    assert xattn.xattn_check_bounded_wait(-1, P) == xattn.XATTN_ERR_INVALID_ARG
    assert xattn.xattn_check_bounded_wait(1 << 33, P) == xattn.XATTN_ERR_INVALID_ARG
    assert xattn.xattn_check_bounded_wait(1000, P + 2) == xattn.XATTN_ERR_MISALIGNED
    assert xattn.xattn_check_bounded_wait(1000, P, P + 4) == xattn.XATTN_ERR_MISALIGNED
