"""Python binding of libskv.so (include/skv.h): argument marshalling only.

Every function has the name of the C entry point it calls and passes plain
integers (device or host addresses, sizes, CUDA stream handles) through
ctypes.  No step of the path runs in Python, and there is no fallback: if the
library is missing, importing this module raises.

``Context`` is a convenience wrapper that takes torch tensors (it reads their
``data_ptr()`` and torch's current CUDA stream) and raises ``SkvError`` for
non-OK statuses.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libskv.so")

SKV_OK = 0
SKV_ERR_INVALID_ARG = 1
SKV_ERR_OOM = 2
SKV_ERR_BAD_REQUEST = 3
SKV_ERR_NO_FREE_REQUEST = 4
SKV_ERR_CONTEXT_FULL = 5
SKV_ERR_CUDA = 6

SKV_DEVERR_BAD_REQUEST = 1
SKV_DEVERR_BAD_INDEX = 2
SKV_DEVERR_DUPLICATE = 4
SKV_DEVERR_CONTEXT_FULL = 8
SKV_DEVERR_TIMEOUT = 16


class skv_config(ctypes.Structure):
    _fields_ = [
        ("max_requests", ctypes.c_int32),
        ("num_layers", ctypes.c_int32),
        ("max_context", ctypes.c_int64),
        ("row_bytes", ctypes.c_int32),
        ("topk", ctypes.c_int32),
        ("hot_slots", ctypes.c_int32),
        ("max_batch", ctypes.c_int32),
        ("device", ctypes.c_int32),
    ]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with `python -m sparse_attention_kv_skv_gb300.build` "
                          "(the CUDA library is required; there is no fallback)")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i32, i64, st = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_int
    P = ctypes.POINTER
    sigs = {
        "skv_create": [P(skv_config), P(vp)],
        "skv_destroy": [vp],
        "skv_publish": [vp, vp, i64, P(i32), vp],
        "skv_write_back": [vp, vp, i32, vp, vp],
        "skv_extend": [vp, i32, vp, i64, vp],
        "skv_assemble": [vp, vp, i32, vp, vp, vp, vp, vp],
        "skv_assemble_host": [vp, vp, i32, vp, vp, vp, vp, vp],
        "skv_assemble_noalloc": [vp, vp, i32, vp, vp, vp, vp, vp],
        "skv_assemble_layer": [vp, vp, i32, i32, vp, vp, vp, vp, vp],
        "skv_prefetch": [vp, vp, i32, i32, vp, vp, vp, vp],
        "skv_prefetch_recent": [vp, vp, i32, i32, i32, vp, vp, vp],
        "skv_release": [vp, i32, vp],
        "skv_get_device_error": [vp, P(i32), vp],
        "skv_hot_buffer": [vp, P(vp), P(i64)],
        "skv_pool_rows": [vp, P(vp)],
        "skv_export_state": [vp, i32, vp, vp, vp, vp, vp, vp, vp],
        "skv_export_hot": [vp, i32, vp, vp],
        "skv_get_clock": [vp, P(ctypes.c_uint32), vp],
        "skv_get_stats": [vp, P(ctypes.c_uint64), P(ctypes.c_uint64), P(ctypes.c_uint64), vp],
        "skv_set_gather_events": [vp, vp, vp],
        "skv_set_attend_sms": [vp, i32],
        "skv_selftest_mma": [vp, vp, vp, i32, i32, i32, vp],
        "skv_attend": [vp, vp, i32, i32, vp, vp, vp, vp, ctypes.c_float, vp],
        "skv_selftest_attend_timeout": [vp, vp, i32, vp, vp, vp, vp],
        "skv_pool_placement": [vp, P(i32), P(i32), P(ctypes.c_float)],
        "skv_host_node_for_pci": [ctypes.c_char_p, ctypes.c_char_p, P(i32)],
    }
    for name, args in sigs.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = st
    lib.skv_last_cuda_error.argtypes = []
    lib.skv_last_cuda_error.restype = ctypes.c_char_p
    lib.skv_status_string.argtypes = [st]
    lib.skv_status_string.restype = ctypes.c_char_p
    return lib


lib = _load()

# The C entry points under their own names (raw: they return the status).
skv_create = lib.skv_create
skv_destroy = lib.skv_destroy
skv_publish = lib.skv_publish
skv_write_back = lib.skv_write_back
skv_extend = lib.skv_extend
skv_assemble = lib.skv_assemble
skv_assemble_host = lib.skv_assemble_host
skv_assemble_noalloc = lib.skv_assemble_noalloc
skv_assemble_layer = lib.skv_assemble_layer
skv_prefetch = lib.skv_prefetch
skv_prefetch_recent = lib.skv_prefetch_recent
skv_release = lib.skv_release
skv_get_device_error = lib.skv_get_device_error
skv_hot_buffer = lib.skv_hot_buffer
skv_pool_rows = lib.skv_pool_rows
skv_export_state = lib.skv_export_state
skv_export_hot = lib.skv_export_hot
skv_get_clock = lib.skv_get_clock
skv_get_stats = lib.skv_get_stats
skv_set_gather_events = lib.skv_set_gather_events
skv_set_attend_sms = lib.skv_set_attend_sms
skv_selftest_mma = lib.skv_selftest_mma
skv_attend = lib.skv_attend
skv_selftest_attend_timeout = lib.skv_selftest_attend_timeout
skv_pool_placement = lib.skv_pool_placement
skv_host_node_for_pci = lib.skv_host_node_for_pci
skv_last_cuda_error = lib.skv_last_cuda_error
skv_status_string = lib.skv_status_string


def host_node_for_pci(pci_bus_id: str, sysfs_root: str | None = None) -> int:
    """The host NUMA node nearest a PCI device (see skv_host_node_for_pci)."""
    n = ctypes.c_int32()
    check(skv_host_node_for_pci(sysfs_root.encode() if sysfs_root else None, pci_bus_id.encode(), ctypes.byref(n)),
          "skv_host_node_for_pci")
    return n.value


class SkvError(RuntimeError):
    def __init__(self, status: int, what: str):
        msg = f"{what}: {skv_status_string(status).decode()}"
        if status == SKV_ERR_CUDA:
            msg += f" ({skv_last_cuda_error().decode()})"
        super().__init__(msg)
        self.status = status


def check(status: int, what: str) -> None:
    if status != SKV_OK:
        raise SkvError(status, what)


def _stream_handle(stream) -> int:
    """A stream argument: None -> torch's current stream; an int -> as is;
    a torch.cuda.Stream -> its handle."""
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _ptr(t) -> int:
    if t is None:
        return 0
    if isinstance(t, int):
        return t
    if hasattr(t, "data_ptr"):
        return t.data_ptr()
    return t.ctypes.data  # numpy


@dataclasses.dataclass
class Config:
    max_requests: int
    num_layers: int
    max_context: int
    topk: int
    hot_slots: int
    max_batch: int
    row_bytes: int = 1152
    device: int = 0

    def c(self) -> skv_config:
        return skv_config(self.max_requests, self.num_layers, self.max_context, self.row_bytes, self.topk,
                          self.hot_slots, self.max_batch, self.device)


class Context:
    """One library context (pool, hot buffer, maps) on one GPU."""

    def __init__(self, cfg: Config):
        self.cfg = cfg
        h = ctypes.c_void_p()
        c = cfg.c()
        check(skv_create(ctypes.byref(c), ctypes.byref(h)), "skv_create")
        self.h = h.value

    def close(self):
        if getattr(self, "h", None):
            check(skv_destroy(self.h), "skv_destroy")
            self.h = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # lifecycle -------------------------------------------------------------
    def publish(self, T: int, rows=None, stream=None) -> int:
        r = ctypes.c_int32()
        check(skv_publish(self.h, _ptr(rows), T, ctypes.byref(r), _stream_handle(stream)), "skv_publish")
        return r.value

    def release(self, req: int, stream=None) -> None:
        check(skv_release(self.h, req, _stream_handle(stream)), "skv_release")

    def write_back(self, req_ids, rows, n: int | None = None, stream=None) -> None:
        n = req_ids.numel() if n is None else n
        check(skv_write_back(self.h, _ptr(req_ids), n, _ptr(rows), _stream_handle(stream)), "skv_write_back")

    def extend(self, req: int, rows, n: int, stream=None) -> None:
        """Append n tokens' rows [L][n][row_bytes] to request req."""
        check(skv_extend(self.h, req, _ptr(rows), n, _stream_handle(stream)), "skv_extend")

    def assemble(self, req_ids, topk, slots, hits, misses, B: int | None = None, stream=None) -> None:
        B = req_ids.numel() if B is None else B
        check(skv_assemble(self.h, _ptr(req_ids), B, _ptr(topk), _ptr(slots), _ptr(hits), _ptr(misses),
                           _stream_handle(stream)), "skv_assemble")

    def assemble_layer(self, layer: int, req_ids, topk, slots, hits, misses, B: int | None = None,
                       stream=None) -> None:
        """One layer's assemble: topk / slots are [B][k], hits / misses [B]."""
        B = req_ids.numel() if B is None else B
        check(skv_assemble_layer(self.h, _ptr(req_ids), B, layer, _ptr(topk), _ptr(slots), _ptr(hits),
                                 _ptr(misses), _stream_handle(stream)), "skv_assemble_layer")

    def prefetch(self, req_ids, cand, layer: int = -1, hits=None, misses=None, B: int | None = None,
                 stream=None) -> None:
        """Assemble of the candidate tokens without a slot tensor: cand is [B][L][k]
        (layer -1) or [B][k]; hits / misses ([B][L] or [B]) are optional."""
        B = req_ids.numel() if B is None else B
        check(skv_prefetch(self.h, _ptr(req_ids), B, layer, _ptr(cand), _ptr(hits), _ptr(misses),
                           _stream_handle(stream)), "skv_prefetch")

    def prefetch_recent(self, req_ids, n: int, layer: int = -1, hits=None, misses=None, B: int | None = None,
                        stream=None) -> None:
        """Prefetch of each request's n newest tokens (every layer, or one)."""
        B = req_ids.numel() if B is None else B
        check(skv_prefetch_recent(self.h, _ptr(req_ids), B, layer, n, _ptr(hits), _ptr(misses),
                                  _stream_handle(stream)), "skv_prefetch_recent")

    def assemble_noalloc(self, req_ids, topk, slots, hits, misses, B: int | None = None, stream=None) -> None:
        """skv_assemble with the gather work list in the library's static
        device array (allocates nothing; see include/skv.h)."""
        B = req_ids.numel() if B is None else B
        check(skv_assemble_noalloc(self.h, _ptr(req_ids), B, _ptr(topk), _ptr(slots), _ptr(hits), _ptr(misses),
                                   _stream_handle(stream)), "skv_assemble_noalloc")

    def assemble_host(self, req_ids, topk, slots, hits, misses, B: int | None = None, stream=None) -> None:
        B = len(req_ids) if B is None else B
        check(skv_assemble_host(self.h, _ptr(req_ids), B, _ptr(topk), _ptr(slots), _ptr(hits), _ptr(misses),
                                _stream_handle(stream)), "skv_assemble_host")

    def attend(self, req_ids, q, slots, out, lse=None, layer: int = -1, sm_scale: float | None = None,
               B: int | None = None, stream=None) -> None:
        """Sparse MLA attention over assembled slots (see skv_attend):
        q [units][128][576] bf16 -> out [units][128][512] bf16, lse [units][128]."""
        B = req_ids.numel() if B is None else B
        scale = (1.0 / 576 ** 0.5) if sm_scale is None else sm_scale
        check(skv_attend(self.h, _ptr(req_ids), B, layer, _ptr(q), _ptr(slots), _ptr(out), _ptr(lse), scale,
                         _stream_handle(stream)), "skv_attend")

    def selftest_attend_timeout(self, req_ids, q, slots, out, B: int | None = None, stream=None) -> None:
        """The attention kernel with its key loads withheld: its waits run out
        and it reports SKV_DEVERR_TIMEOUT (see skv_selftest_attend_timeout)."""
        B = req_ids.numel() if B is None else B
        check(skv_selftest_attend_timeout(self.h, _ptr(req_ids), B, _ptr(q), _ptr(slots), _ptr(out),
                                          _stream_handle(stream)), "skv_selftest_attend_timeout")

    # inspection ------------------------------------------------------------
    def get_device_error(self, stream=None) -> int:
        bits = ctypes.c_int32()
        check(skv_get_device_error(self.h, ctypes.byref(bits), _stream_handle(stream)), "skv_get_device_error")
        return bits.value

    def hot_buffer(self):
        base, stride = ctypes.c_void_p(), ctypes.c_int64()
        check(skv_hot_buffer(self.h, ctypes.byref(base), ctypes.byref(stride)), "skv_hot_buffer")
        return base.value, stride.value

    def pool_rows(self) -> int:
        base = ctypes.c_void_p()
        check(skv_pool_rows(self.h, ctypes.byref(base)), "skv_pool_rows")
        return base.value

    def export_state(self, req: int, tok2slot: bool = True, stream=None):
        import numpy as np
        L, S, T = self.cfg.num_layers, self.cfg.hot_slots, self.cfg.max_context
        s2t = np.empty((L, S), np.int32)
        ts = np.empty((L, S), np.uint32)
        lru = np.empty((L, S), np.int32)
        t2s = np.empty((L, T), np.int32) if tok2slot else None
        ln = np.zeros(1, np.int64)
        act = np.zeros(1, np.int32)
        check(skv_export_state(self.h, req, _ptr(s2t), _ptr(ts), _ptr(t2s), _ptr(lru), _ptr(ln), _ptr(act),
                               _stream_handle(stream)), "skv_export_state")
        return {"slot2tok": s2t, "ts": ts, "lru": lru, "tok2slot": t2s, "len": int(ln[0]), "active": int(act[0])}

    def export_hot(self, req: int, stream=None):
        import numpy as np
        out = np.empty((self.cfg.num_layers, self.cfg.hot_slots, self.cfg.row_bytes), np.uint8)
        check(skv_export_hot(self.h, req, _ptr(out), _stream_handle(stream)), "skv_export_hot")
        return out

    def clock(self, stream=None) -> int:
        c = ctypes.c_uint32()
        check(skv_get_clock(self.h, ctypes.byref(c), _stream_handle(stream)), "skv_get_clock")
        return c.value

    def stats(self, stream=None):
        a, b, c = ctypes.c_uint64(), ctypes.c_uint64(), ctypes.c_uint64()
        check(skv_get_stats(self.h, ctypes.byref(a), ctypes.byref(b), ctypes.byref(c), _stream_handle(stream)),
              "skv_get_stats")
        return {"calls": a.value, "hits": b.value, "misses": c.value}

    def pool_placement(self):
        """(wanted node, node holding most sampled pool pages, share there); -1 = none / not reported."""
        a, b, f = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_float()
        check(skv_pool_placement(self.h, ctypes.byref(a), ctypes.byref(b), ctypes.byref(f)), "skv_pool_placement")
        return a.value, b.value, f.value

    def set_attend_sms(self, sms: int = 0) -> None:
        """At most `sms` SMs for later attend() calls (0: all; see skv_set_attend_sms)."""
        check(skv_set_attend_sms(self.h, sms), "skv_set_attend_sms")

    def set_gather_events(self, before=None, after=None) -> None:
        check(skv_set_gather_events(self.h, before.cuda_event if before is not None else None,
                                    after.cuda_event if after is not None else None), "skv_set_gather_events")
