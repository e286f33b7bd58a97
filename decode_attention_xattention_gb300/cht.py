"""ctypes binding of the chunked hash tree (xattn_cht.h): argument marshalling only; the
structure lives in libxattn.so (csrc/cht.cpp)."""

from __future__ import annotations

import ctypes

import numpy as np

from . import xattn

_bound = False


def _lib():
    global _bound
    lib = xattn.load()
    if not _bound:
        vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
        lib.xattn_cht_create.argtypes = [i32]
        lib.xattn_cht_create.restype = vp
        lib.xattn_cht_destroy.argtypes = [vp]
        lib.xattn_cht_destroy.restype = None
        lib.xattn_cht_insert.argtypes = [vp, i64, vp, i64]
        lib.xattn_cht_best.argtypes = [vp, ctypes.POINTER(i64), ctypes.POINTER(i32)]
        lib.xattn_cht_admit.argtypes = [vp, i64]
        lib.xattn_cht_finish.argtypes = [vp, i64]
        lib.xattn_cht_cancel.argtypes = [vp, i64]
        lib.xattn_cht_missing.argtypes = [vp, i64, ctypes.POINTER(i32)]
        lib.xattn_cht_counts.argtypes = [vp, ctypes.POINTER(i64), ctypes.POINTER(i64), ctypes.POINTER(i64)]
        for f in ("insert", "best", "admit", "finish", "cancel", "missing", "counts"):
            getattr(lib, f"xattn_cht_{f}").restype = ctypes.c_int
        _bound = True
    return lib


class ChunkedHashTree:
    """Owner of one native structure (released on close() or garbage collection)."""

    def __init__(self, block_tokens: int):
        self._lib = _lib()
        self._h = self._lib.xattn_cht_create(int(block_tokens))
        if not self._h:
            raise xattn.XAttnError("xattn_cht_create failed")

    def close(self) -> None:
        if self._h:
            self._lib.xattn_cht_destroy(self._h)
            self._h = None

    def __del__(self):
        self.close()

    def insert(self, request_id: int, tokens) -> int:
        t = np.ascontiguousarray(tokens, dtype=np.int32)
        return int(self._lib.xattn_cht_insert(self._h, int(request_id),
                                              t.ctypes.data_as(ctypes.c_void_p) if t.size else None, int(t.size)))

    def best(self):
        """(rc, request_id, missing): rc 1 found, 0 nothing waits, < 0 error."""
        rid, miss = ctypes.c_int64(0), ctypes.c_int32(0)
        rc = int(self._lib.xattn_cht_best(self._h, ctypes.byref(rid), ctypes.byref(miss)))
        return rc, int(rid.value), int(miss.value)

    def admit(self, request_id: int) -> int:
        return int(self._lib.xattn_cht_admit(self._h, int(request_id)))

    def finish(self, request_id: int) -> int:
        return int(self._lib.xattn_cht_finish(self._h, int(request_id)))

    def cancel(self, request_id: int) -> int:
        return int(self._lib.xattn_cht_cancel(self._h, int(request_id)))

    def missing(self, request_id: int):
        """(rc, missing)."""
        m = ctypes.c_int32(0)
        rc = int(self._lib.xattn_cht_missing(self._h, int(request_id), ctypes.byref(m)))
        return rc, int(m.value)

    def counts(self):
        """(waiting, active, working-set hashes)."""
        w, a, h = ctypes.c_int64(0), ctypes.c_int64(0), ctypes.c_int64(0)
        xattn.check(int(self._lib.xattn_cht_counts(self._h, ctypes.byref(w), ctypes.byref(a), ctypes.byref(h))))
        return int(w.value), int(a.value), int(h.value)
