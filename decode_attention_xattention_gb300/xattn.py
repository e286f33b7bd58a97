"""ctypes binding of libxattn.so (argument marshalling only).

Every function here has the name and argument order of its C entry point in
include/xattn.h and returns the C return code. Tensor arguments may be torch tensors (their
data_ptr() is passed), plain integer addresses, or None (NULL). All compute runs in the
library's CUDA kernels; if the library is missing this module raises instead of falling
back to anything else.
"""

from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libxattn.so")

XATTN_OK = 0
XATTN_ERR_INVALID_ARG = -1
XATTN_ERR_UNSUPPORTED = -2
XATTN_ERR_WORKSPACE_TOO_SMALL = -3
XATTN_ERR_MISALIGNED = -4
XATTN_ERR_CUDA = -5
XATTN_ERR_HOST_MEMORY = -6

XATTN_STATUS_BAD_SHARED_LEN = 1
XATTN_STATUS_BAD_SLOT = 2
XATTN_STATUS_BAD_PARENT = 4
XATTN_STATUS_EMPTY_ROW = 8
XATTN_STATUS_TIMEOUT = 16
XATTN_STATUS_BAD_TRIE = 32
XATTN_STATUS_TOO_MANY_VALID = 64

XATTN_DTYPE_BF16 = 0
XATTN_DTYPE_F32 = 1

# Every symbol include/xattn.h declares.
EXPORTS = ("xattn_decode_workspace_size", "xattn_decode", "xattn_decode_shared", "xattn_decode_merge",
           "xattn_beam_update", "xattn_decode_step", "xattn_read_status", "xattn_query_plan", "xattn_status_string",
           "xattn_decode_noalloc", "xattn_beam_select",
           "xattn_cht_create", "xattn_cht_destroy", "xattn_cht_insert", "xattn_cht_best", "xattn_cht_admit",
           "xattn_cht_finish", "xattn_cht_cancel", "xattn_cht_missing", "xattn_cht_counts",
           "xattn_trie_size", "xattn_trie_build", "xattn_valid_path_mask", "xattn_valid_path_topk",
           "xattn_check_bounded_wait")

XATTN_NOALLOC_SCRATCH_BYTES = 32 << 20


class XAttnError(RuntimeError):
    pass


class xattn_desc(ctypes.Structure):
    _fields_ = [("num_requests", ctypes.c_int32), ("beam_width", ctypes.c_int32),
                ("num_q_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("max_shared_len", ctypes.c_int32),
                ("ns_slots", ctypes.c_int32), ("max_steps", ctypes.c_int32),
                ("softmax_scale", ctypes.c_float), ("dtype", ctypes.c_int32),
                ("shared_kernel", ctypes.c_int32), ("split_tokens", ctypes.c_int32),
                ("out_dtype", ctypes.c_int32)]


class xattn_plan(ctypes.Structure):
    _fields_ = [("shared_kernel", ctypes.c_int32), ("num_splits", ctypes.c_int32),
                ("split_tokens", ctypes.c_int32), ("rows_per_unit", ctypes.c_int32),
                ("row_tiles", ctypes.c_int32), ("shared_ctas", ctypes.c_int32),
                ("merge_ctas", ctypes.c_int32), ("fused", ctypes.c_int32), ("piece_stride", ctypes.c_int32),
                ("ns_tile", ctypes.c_int32), ("reserved", ctypes.c_int32 * 1)]


_lib = None


def load(path: str = LIB_PATH):
    """Load libxattn.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise XAttnError(f"libxattn.so not built at {path}: run decode_attention_xattention_gb300.build.build()")
    lib = ctypes.CDLL(path)
    vp, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
    pdesc = ctypes.POINTER(xattn_desc)
    lib.xattn_decode_workspace_size.argtypes = [pdesc]
    lib.xattn_decode_workspace_size.restype = sz
    lib.xattn_decode.argtypes = [pdesc, vp, vp, vp, vp, vp, vp, vp, i32, vp, vp, vp, sz, vp]
    lib.xattn_decode.restype = ctypes.c_int
    lib.xattn_decode_shared.argtypes = [pdesc, vp, vp, vp, vp, vp, sz, vp]
    lib.xattn_decode_shared.restype = ctypes.c_int
    lib.xattn_decode_merge.argtypes = [pdesc, vp, vp, vp, vp, vp, i32, vp, vp, vp, sz, vp]
    lib.xattn_decode_merge.restype = ctypes.c_int
    lib.xattn_decode_noalloc.argtypes = [pdesc, vp, vp, vp, vp, vp, vp, vp, i32, vp, vp, vp, vp]
    lib.xattn_decode_noalloc.restype = ctypes.c_int
    lib.xattn_beam_update.argtypes = [pdesc, vp, vp, vp, vp, vp, vp, i32, vp, vp]
    lib.xattn_beam_update.restype = ctypes.c_int
    lib.xattn_decode_step.argtypes = [pdesc, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, vp, vp, vp, sz, vp]
    lib.xattn_decode_step.restype = ctypes.c_int
    lib.xattn_beam_select.argtypes = [i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp]
    lib.xattn_beam_select.restype = ctypes.c_int
    i64 = ctypes.c_int64
    lib.xattn_trie_size.argtypes = [vp, i64, i32, ctypes.POINTER(i64)]
    lib.xattn_trie_build.argtypes = [vp, i64, i32, i64, vp, vp]
    lib.xattn_valid_path_mask.argtypes = [vp, vp, i64, i32, vp, i32, i32, i32, i32, vp, vp, vp, vp]
    lib.xattn_valid_path_topk.argtypes = [vp, vp, i64, i32, vp, i32, i32, i32, i32, vp, i32, vp, vp, vp, vp, vp]
    for f in ("xattn_trie_size", "xattn_trie_build", "xattn_valid_path_mask", "xattn_valid_path_topk"):
        getattr(lib, f).restype = ctypes.c_int
    lib.xattn_check_bounded_wait.argtypes = [i64, vp, vp, vp]
    lib.xattn_check_bounded_wait.restype = ctypes.c_int
    lib.xattn_read_status.argtypes = [vp, ctypes.POINTER(i32), i32, vp]
    lib.xattn_read_status.restype = ctypes.c_int
    lib.xattn_query_plan.argtypes = [pdesc, i32, ctypes.POINTER(xattn_plan)]
    lib.xattn_query_plan.restype = ctypes.c_int
    lib.xattn_status_string.argtypes = [ctypes.c_int]
    lib.xattn_status_string.restype = ctypes.c_char_p
    _lib = lib
    return lib


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(s):
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return s.cuda_stream  # torch.cuda.Stream


def make_desc(R, BW, Hq, Hkv, d, Lmax, S, Tmax, scale=0.0, shared_kernel=0, split_tokens=0,
              out_dtype=XATTN_DTYPE_BF16, dtype=XATTN_DTYPE_BF16) -> xattn_desc:
    return xattn_desc(R, BW, Hq, Hkv, d, Lmax, S, Tmax, float(scale), dtype,
                      shared_kernel, split_tokens, out_dtype)


def xattn_decode_workspace_size(desc: xattn_desc) -> int:
    return int(load().xattn_decode_workspace_size(ctypes.byref(desc)))


def xattn_decode(desc, q, shared_k, shared_v, shared_len, ns_k_pool, ns_v_pool, beam_tok_idx, step,
                 out, lse, workspace, workspace_bytes, stream=None) -> int:
    return int(load().xattn_decode(ctypes.byref(desc), _ptr(q), _ptr(shared_k), _ptr(shared_v),
                                   _ptr(shared_len), _ptr(ns_k_pool), _ptr(ns_v_pool), _ptr(beam_tok_idx),
                                   int(step), _ptr(out), _ptr(lse), _ptr(workspace), int(workspace_bytes),
                                   _stream(stream)))


def xattn_decode_noalloc(desc, q, shared_k, shared_v, shared_len, ns_k_pool, ns_v_pool, beam_tok_idx, step,
                         out, lse, status_out=None, stream=None) -> int:
    """xattn_decode with the library's own static scratch instead of a caller workspace."""
    return int(load().xattn_decode_noalloc(ctypes.byref(desc), _ptr(q), _ptr(shared_k), _ptr(shared_v),
                                           _ptr(shared_len), _ptr(ns_k_pool), _ptr(ns_v_pool),
                                           _ptr(beam_tok_idx), int(step), _ptr(out), _ptr(lse), _ptr(status_out),
                                           _stream(stream)))


def xattn_decode_shared(desc, q, shared_k, shared_v, shared_len, workspace, workspace_bytes, stream=None) -> int:
    return int(load().xattn_decode_shared(ctypes.byref(desc), _ptr(q), _ptr(shared_k), _ptr(shared_v),
                                          _ptr(shared_len), _ptr(workspace), int(workspace_bytes), _stream(stream)))


def xattn_decode_merge(desc, q, shared_len, ns_k_pool, ns_v_pool, beam_tok_idx, step, out, lse, workspace,
                       workspace_bytes, stream=None) -> int:
    return int(load().xattn_decode_merge(ctypes.byref(desc), _ptr(q), _ptr(shared_len), _ptr(ns_k_pool),
                                         _ptr(ns_v_pool), _ptr(beam_tok_idx), int(step), _ptr(out), _ptr(lse),
                                         _ptr(workspace), int(workspace_bytes), _stream(stream)))


def xattn_decode_step(desc, parent, new_k, new_v, q, shared_k, shared_v, shared_len, ns_k_pool, ns_v_pool,
                      beam_tok_idx, step, out, lse, workspace, workspace_bytes, stream=None) -> int:
    return int(load().xattn_decode_step(ctypes.byref(desc), _ptr(parent), _ptr(new_k), _ptr(new_v), _ptr(q),
                                        _ptr(shared_k), _ptr(shared_v), _ptr(shared_len), _ptr(ns_k_pool),
                                        _ptr(ns_v_pool), _ptr(beam_tok_idx), int(step), _ptr(out), _ptr(lse),
                                        _ptr(workspace), int(workspace_bytes), _stream(stream)))


def xattn_beam_update(desc, parent, new_k, new_v, ns_k_pool, ns_v_pool, beam_tok_idx, step, status=None,
                      stream=None) -> int:
    return int(load().xattn_beam_update(ctypes.byref(desc), _ptr(parent), _ptr(new_k), _ptr(new_v),
                                        _ptr(ns_k_pool), _ptr(ns_v_pool), _ptr(beam_tok_idx), int(step),
                                        _ptr(status), _stream(stream)))


def xattn_beam_select(num_requests, beam_width, cand_per_beam, out_width, beam_score, cand_logp, cand_token,
                      parent, token, score, stream=None) -> int:
    return int(load().xattn_beam_select(int(num_requests), int(beam_width), int(cand_per_beam), int(out_width),
                                        _ptr(beam_score), _ptr(cand_logp), _ptr(cand_token), _ptr(parent),
                                        _ptr(token), _ptr(score), _stream(stream)))


def trie_build(items):
    """Host trie of the item catalogue `items` [N, L] (int32 array): (child_off, child_tok)
    numpy arrays, laid out as xattn_valid_path.h describes."""
    import numpy as np

    items = np.ascontiguousarray(items, dtype=np.int32)
    N, L = items.shape
    lib = load()
    n = ctypes.c_int64(0)
    check(int(lib.xattn_trie_size(items.ctypes.data_as(ctypes.c_void_p), N, L, ctypes.byref(n))))
    off = np.zeros(n.value + 1, np.int32)
    tok = np.zeros(max(n.value - 1, 1), np.int32)
    check(int(lib.xattn_trie_build(items.ctypes.data_as(ctypes.c_void_p), N, L, n.value,
                                   off.ctypes.data_as(ctypes.c_void_p), tok.ctypes.data_as(ctypes.c_void_p))))
    return off, tok[: n.value - 1]


def xattn_valid_path_mask(child_off, child_tok, num_nodes, path_len, prefix, prefix_stride, step, rows, V, logp,
                          valid_count=None, status=None, stream=None) -> int:
    return int(load().xattn_valid_path_mask(_ptr(child_off), _ptr(child_tok), int(num_nodes), int(path_len),
                                            _ptr(prefix), int(prefix_stride), int(step), int(rows), int(V), _ptr(logp),
                                            _ptr(valid_count), _ptr(status), _stream(stream)))


def xattn_valid_path_topk(child_off, child_tok, num_nodes, path_len, prefix, prefix_stride, step, rows, V, logp, C,
                          cand_token, cand_logp, valid_count=None, status=None, stream=None) -> int:
    return int(load().xattn_valid_path_topk(_ptr(child_off), _ptr(child_tok), int(num_nodes), int(path_len),
                                            _ptr(prefix), int(prefix_stride), int(step), int(rows), int(V), _ptr(logp),
                                            int(C), _ptr(cand_token), _ptr(cand_logp), _ptr(valid_count),
                                            _ptr(status), _stream(stream)))


def xattn_check_bounded_wait(limit_cycles, status, waited_cycles=None, stream=None) -> int:
    return int(load().xattn_check_bounded_wait(int(limit_cycles), _ptr(status), _ptr(waited_cycles),
                                               _stream(stream)))


def xattn_read_status(workspace, clear: bool = True, stream=None) -> tuple[int, int]:
    """Returns (return code, status word)."""
    st = ctypes.c_int32(0)
    rc = load().xattn_read_status(_ptr(workspace), ctypes.byref(st), 1 if clear else 0, _stream(stream))
    return int(rc), int(st.value)


def xattn_query_plan(desc, step) -> tuple[int, xattn_plan]:
    p = xattn_plan()
    rc = load().xattn_query_plan(ctypes.byref(desc), int(step), ctypes.byref(p))
    return int(rc), p


def xattn_status_string(code: int) -> str:
    return load().xattn_status_string(int(code)).decode()


def check(rc: int) -> None:
    if rc != XATTN_OK:
        raise XAttnError(f"xattn call failed: {rc} ({xattn_status_string(rc)})")
