"""CPU oracle for the sparse KV assembly path -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path never imports it and
shares no code with it.

``Oracle`` wraps ``skv_oracle.cpp`` (plain C++: a ``std::unordered_map`` per
(request, layer), an explicit ``std::list`` LRU, ``memcpy`` gathers).  See the
header of that file for what each step computes and which passage of the pages
it follows.

Parity status: every function is pinned by tests that do not re-run the oracle's
own formula -- hand-derived worked examples (tests/golden), closed forms for
special Top-k sequences, per-step invariants, brute-force agreement with an
independent definition on exhaustively enumerated tiny inputs, and planted
mistakes that each of those pins must catch.  The LRU tie-break (lowest slot
index) and the miss placement order (ascending token) are not fixed by the
pages; they are pinned to the stated reading, not to the pages.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(_HERE, "skv_oracle.cpp")
_LIB = os.path.join(_HERE, "libskv_oracle.so")

E_BAD_REQUEST, E_BAD_INDEX, E_DUPLICATE, E_CONTEXT_FULL = 1, 2, 4, 8


def compile_oracle(src: str, out: str) -> str:
    cmd = ["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-fopenmp", "-Wall", "-Wextra", "-o", out + ".tmp", src]
    subprocess.run(cmd, check=True)
    os.replace(out + ".tmp", out)
    return out


def build(force: bool = False) -> str:
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(SRC):
        compile_oracle(SRC, _LIB)
    return _LIB


def load(path: str | None = None):
    """Load an oracle shared library (the default one, or a variant)."""
    if path is None:
        path = build()
    L = ctypes.CDLL(path)
    vp, i32, i64, u32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_uint32
    L.orc_create.restype = vp
    L.orc_create.argtypes = [i32, i32, i64, i32, i32, i32, vp]
    L.orc_destroy.restype = None
    L.orc_destroy.argtypes = [vp]
    L.orc_publish.restype = i32
    L.orc_publish.argtypes = [vp, i64]
    L.orc_release.restype = i32
    L.orc_release.argtypes = [vp, i32]
    L.orc_write_back.restype = i32
    L.orc_write_back.argtypes = [vp, vp, i32, vp]
    L.orc_extend.restype = i32
    L.orc_extend.argtypes = [vp, i32, vp, i64]
    L.orc_assemble.restype = i32
    L.orc_assemble.argtypes = [vp, vp, i32, vp, vp, vp, vp, i32]
    L.orc_assemble_layer.restype = i32
    L.orc_assemble_layer.argtypes = [vp, vp, i32, i32, vp, vp, vp, vp, i32]
    L.orc_get_error.restype = i32
    L.orc_get_error.argtypes = [vp]
    L.orc_now.restype = u32
    L.orc_now.argtypes = [vp]
    L.orc_export.restype = None
    L.orc_export.argtypes = [vp, i32, vp, vp, vp, vp, vp, vp]
    L.orc_export_hot.restype = None
    L.orc_export_hot.argtypes = [vp, i32, vp]
    L.orc_pool_row.restype = i32
    L.orc_pool_row.argtypes = [vp, i32, i32, i64, vp]
    return L


_default = None


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


class Oracle:
    """The oracle over a pool view.

    ``pool`` is either a numpy uint8 array shaped [R][L][T_max][row_bytes] or an
    integer host address of memory with that layout (e.g. the library's pinned
    pool, filled by the workload generator).  The view must stay alive and
    unchanged (except for rows the caller publishes) while the oracle is used.
    """

    def __init__(self, R, L, T_max, row_bytes, k, S, pool, lib_path: str | None = None):
        global _default
        if lib_path is None:
            if _default is None:
                _default = load()
            self.lib = _default
        else:
            self.lib = load(lib_path)
        self.R, self.L, self.T_max, self.row_bytes, self.k, self.S = R, L, T_max, row_bytes, k, S
        if isinstance(pool, np.ndarray):
            assert pool.dtype == np.uint8 and pool.flags.c_contiguous
            assert pool.size == R * L * T_max * row_bytes
            self._pool_ref = pool
            addr = _ptr(pool)
        else:
            self._pool_ref = None
            addr = int(pool)
        self.h = self.lib.orc_create(R, L, T_max, row_bytes, k, S, addr)
        if not self.h:
            raise ValueError("bad oracle configuration")

    def close(self):
        if self.h:
            self.lib.orc_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def publish(self, T: int) -> int:
        return int(self.lib.orc_publish(self.h, T))

    def release(self, r: int) -> int:
        return int(self.lib.orc_release(self.h, r))

    def write_back(self, req_ids, rows: np.ndarray) -> int:
        req = np.ascontiguousarray(np.asarray(req_ids, dtype=np.int32))
        rows = np.ascontiguousarray(rows, dtype=np.uint8)
        assert rows.size == req.size * self.L * self.row_bytes
        return int(self.lib.orc_write_back(self.h, _ptr(req), req.size, _ptr(rows)))

    def extend(self, r: int, rows: np.ndarray) -> int:
        """Append rows [L][n][row_bytes] to request r."""
        rows = np.ascontiguousarray(rows, dtype=np.uint8)
        n = rows.size // (self.L * self.row_bytes)
        assert rows.size == n * self.L * self.row_bytes
        return int(self.lib.orc_extend(self.h, r, _ptr(rows), n))

    def assemble(self, req_ids, topk: np.ndarray, nthreads: int = 1):
        """Returns (err, slots[B][L][k], hits[B][L], misses[B][L])."""
        req = np.ascontiguousarray(np.asarray(req_ids, dtype=np.int32))
        B = req.size
        topk = np.ascontiguousarray(topk, dtype=np.int32).reshape(B, self.L, self.k)
        slots = np.empty_like(topk)
        hits = np.empty((B, self.L), dtype=np.int32)
        misses = np.empty((B, self.L), dtype=np.int32)
        err = self.lib.orc_assemble(self.h, _ptr(req), B, _ptr(topk), _ptr(slots), _ptr(hits), _ptr(misses),
                                    nthreads)
        return int(err), slots, hits, misses

    def assemble_layer(self, layer: int, req_ids, topk: np.ndarray, nthreads: int = 1):
        """One layer: topk [B][k] -> (err, slots[B][k], hits[B], misses[B])."""
        req = np.ascontiguousarray(np.asarray(req_ids, dtype=np.int32))
        B = req.size
        topk = np.ascontiguousarray(topk, dtype=np.int32).reshape(B, self.k)
        slots = np.empty_like(topk)
        hits = np.empty(B, dtype=np.int32)
        misses = np.empty(B, dtype=np.int32)
        err = self.lib.orc_assemble_layer(self.h, _ptr(req), B, layer, _ptr(topk), _ptr(slots), _ptr(hits),
                                          _ptr(misses), nthreads)
        return int(err), slots, hits, misses

    def prefetch(self, req_ids, cand: np.ndarray, layer: int = -1, nthreads: int = 1):
        """Prefetch of candidate tokens -- HiSparse's prefetching, kept by XM-Sparse
        ("XM-Sparse: Netpreme X-Mem ...", section on the SGLang HiSparse
        integration).  The pages say no more than that it exists; read plainly, a
        prefetch makes tokens resident before the step that selects them, which in
        this model is exactly an assemble of those tokens (same checks, LRU rule,
        gather and clock tick) whose slots are not handed out.  cand is [B][L][k]
        (layer -1) or [B][k].  Returns (err, hits, misses)."""
        if layer < 0:
            err, _, hits, misses = self.assemble(req_ids, cand, nthreads)
        else:
            err, _, hits, misses = self.assemble_layer(layer, req_ids, cand, nthreads)
        return err, hits, misses

    def recent_candidates(self, req_ids, n: int, layer: int = -1) -> np.ndarray:
        """The recency-window candidates: for each batch entry, its request's n newest
        tokens [len - n, len) ascending (all of [0, len) when len < n), -1 padded to
        k, for every layer ([B][L][k]) or one ([B][k]).  An id that is not an active
        request gets an all -1 row (the call is rejected for it anyway)."""
        req = [int(r) for r in req_ids]
        rows = self.L if layer < 0 else 1
        out = np.full((len(req), rows, self.k), -1, dtype=np.int32)
        for b, r in enumerate(req):
            if not 0 <= r < self.R:
                continue
            st = self.export(r, tok2slot=False)
            if not st["active"]:
                continue
            toks = np.arange(max(0, st["len"] - n), st["len"], dtype=np.int32)
            out[b, :, :toks.size] = toks
        return out if layer < 0 else out[:, 0, :]

    def prefetch_recent(self, req_ids, n: int, layer: int = -1, nthreads: int = 1):
        """Prefetch of each request's n newest tokens; returns (err, hits, misses)."""
        return self.prefetch(req_ids, self.recent_candidates(req_ids, n, layer), layer, nthreads)

    def get_error(self) -> int:
        return int(self.lib.orc_get_error(self.h))

    @property
    def now(self) -> int:
        return int(self.lib.orc_now(self.h))

    def export(self, r: int, tok2slot: bool = True):
        """dict with slot2tok, ts, lru ([L][S]), tok2slot ([L][T_max]), len, active."""
        s2t = np.empty((self.L, self.S), dtype=np.int32)
        ts = np.empty((self.L, self.S), dtype=np.uint32)
        lru = np.empty((self.L, self.S), dtype=np.int32)
        t2s = np.empty((self.L, self.T_max), dtype=np.int32) if tok2slot else None
        ln = np.zeros(1, dtype=np.int64)
        act = np.zeros(1, dtype=np.int32)
        self.lib.orc_export(self.h, r, _ptr(s2t), _ptr(ts), _ptr(t2s) if tok2slot else None, _ptr(lru),
                            _ptr(ln), _ptr(act))
        return {"slot2tok": s2t, "ts": ts, "lru": lru, "tok2slot": t2s, "len": int(ln[0]), "active": int(act[0])}

    def export_hot(self, r: int) -> np.ndarray:
        out = np.empty((self.L, self.S, self.row_bytes), dtype=np.uint8)
        self.lib.orc_export_hot(self.h, r, _ptr(out))
        return out

    def pool_row(self, r: int, l: int, t: int) -> np.ndarray:
        out = np.empty(self.row_bytes, dtype=np.uint8)
        if self.lib.orc_pool_row(self.h, r, l, t, _ptr(out)) != 0:
            raise IndexError((r, l, t))
        return out
