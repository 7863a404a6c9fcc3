"""Python binding of the cache manager and policy simulator (``include/lazy_cache.h``).

Argument marshalling only: the allocator, the entry map, eviction and the replay
all run in ``liblazyattn.so``'s host C++ code. Three policies decide which
segments of a request may reuse a cached run of blocks:

- ``AGNOSTIC``: any earlier copy of the document, at any offset (stored keys carry
  no position, so one copy serves every placement);
- ``AWARE``: only a copy stored at the same offset (keys stored with their
  absolute positions);
- ``PREFIX``: only a copy stored after the same preceding segments (prefix caching).
"""
from __future__ import annotations

import ctypes
from typing import List, Optional, Sequence, Tuple

import numpy as np

from .lazy_attn import LAZY_ERR_LAYOUT, LAZY_OK, BLOCK, LazyAttnError, _lib

AGNOSTIC, AWARE, PREFIX = 0, 1, 2
POLICIES = {"agnostic": AGNOSTIC, "aware": AWARE, "prefix": PREFIX}
EXPORTED = ("lazy_cache_create", "lazy_cache_destroy", "lazy_cache_admit", "lazy_cache_release",
            "lazy_cache_get_stats", "lazy_cache_simulate")


class CacheStats(ctypes.Structure):
    """Mirror of ``lazy_cache_stats``."""
    _fields_ = [("hit_blocks", ctypes.c_int64), ("miss_blocks", ctypes.c_int64), ("evicted_blocks", ctypes.c_int64),
                ("rejected", ctypes.c_int64), ("resident_blocks", ctypes.c_int64),
                ("peak_resident_blocks", ctypes.c_int64)]

    def as_dict(self) -> dict:
        d = {k: int(getattr(self, k)) for k, _ in self._fields_}
        total = d["hit_blocks"] + d["miss_blocks"]
        d["hit_rate"] = d["hit_blocks"] / total if total else 0.0
        return d


_vp, _i32, _i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
_sig = {
    "lazy_cache_create": (_vp, [_i32, _i32]),
    "lazy_cache_destroy": (None, [_vp]),
    "lazy_cache_admit": (ctypes.c_int, [_vp, _i32, _vp, _vp, _i32, _vp, _vp, _i32, _vp, ctypes.POINTER(_i64)]),
    "lazy_cache_release": (ctypes.c_int, [_vp, _i64]),
    "lazy_cache_get_stats": (ctypes.c_int, [_vp, ctypes.POINTER(CacheStats)]),
    "lazy_cache_simulate": (ctypes.c_int, [_i32, _i32, _i32, _vp, _vp, _vp, _vp, _i32, ctypes.POINTER(CacheStats)]),
}
for _name, (_res, _args) in _sig.items():
    _f = getattr(_lib, _name)
    _f.restype, _f.argtypes = _res, _args


def _i32_array(x) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(x, dtype=np.int64).astype(np.int32))


def _policy(policy) -> int:
    return POLICIES[policy] if isinstance(policy, str) else int(policy)


class Admission:
    """One admitted request: per-segment block ids and hit flags, and its ticket."""

    def __init__(self, ticket: int, indptr: np.ndarray, blocks: np.ndarray, hit: np.ndarray):
        self.ticket, self.indptr, self.blocks, self.hit = ticket, indptr, blocks, hit

    def segment_blocks(self, i: int) -> np.ndarray:
        return self.blocks[self.indptr[i]:self.indptr[i + 1]]


class PagedCache:
    """A cache over block ids 0 .. num_blocks-1 under one policy."""

    def __init__(self, num_blocks: int, policy="agnostic"):
        self._c = _lib.lazy_cache_create(int(num_blocks), _policy(policy))
        if not self._c:
            raise ValueError(f"lazy_cache_create({num_blocks}, {policy!r}) failed")
        self.num_blocks = int(num_blocks)

    def close(self) -> None:
        if self._c:
            _lib.lazy_cache_destroy(self._c)
            self._c = None

    def __del__(self):
        self.close()

    def admit(self, segments: Sequence[Tuple[int, int]], pos0: int = 0) -> Optional[Admission]:
        """Admits segments [(doc, len), ...] from position pos0. Returns None when the
        pool cannot hold the request (counted as rejected); raises on bad arguments."""
        doc = _i32_array([s[0] for s in segments])
        ln = _i32_array([s[1] for s in segments])
        n = len(segments)
        cap = int(sum((int(x) + BLOCK - 1) // BLOCK for x in ln)) if n else 0
        indptr = np.zeros(n + 1, np.int32)
        blocks = np.zeros(max(cap, 1), np.int32)
        hit = np.zeros(max(n, 1), np.int32)
        t = ctypes.c_int64(0)
        rc = _lib.lazy_cache_admit(self._c, n, doc.ctypes.data if n else None, ln.ctypes.data if n else None,
                                   int(pos0), indptr.ctypes.data, blocks.ctypes.data, cap, hit.ctypes.data,
                                   ctypes.byref(t))
        if rc == LAZY_ERR_LAYOUT:
            return None
        if rc != LAZY_OK:
            raise LazyAttnError(rc, "lazy_cache_admit")
        return Admission(int(t.value), indptr, blocks[:cap], hit[:n])

    def release(self, ticket) -> None:
        t = ticket.ticket if isinstance(ticket, Admission) else int(ticket)
        rc = _lib.lazy_cache_release(self._c, t)
        if rc != LAZY_OK:
            raise LazyAttnError(rc, "lazy_cache_release")

    def stats(self) -> dict:
        s = CacheStats()
        rc = _lib.lazy_cache_get_stats(self._c, ctypes.byref(s))
        if rc != LAZY_OK:
            raise LazyAttnError(rc, "lazy_cache_get_stats")
        return s.as_dict()


def simulate(policy, num_blocks: int, requests: Sequence[Sequence[Tuple[int, int]]],
             pos0: Optional[Sequence[int]] = None, concurrency: int = 1) -> dict:
    """Replays requests (each a list of (doc, len) segments) through a fresh cache
    and returns its final counters, with ``hit_rate`` = hit / (hit + miss) blocks."""
    lens = [len(r) for r in requests]
    indptr = _i32_array(np.concatenate([[0], np.cumsum(lens)]) if lens else [0])
    flat = [s for r in requests for s in r]
    doc = _i32_array([s[0] for s in flat] or [0])
    ln = _i32_array([s[1] for s in flat] or [1])
    p0 = _i32_array(pos0) if pos0 is not None else None
    if p0 is not None and len(p0) != len(requests):
        raise ValueError("pos0 needs one entry per request")
    s = CacheStats()
    rc = _lib.lazy_cache_simulate(_policy(policy), int(num_blocks), len(requests), indptr.ctypes.data,
                                  doc.ctypes.data, ln.ctypes.data, p0.ctypes.data if p0 is not None else None,
                                  int(concurrency), ctypes.byref(s))
    if rc != LAZY_OK:
        raise LazyAttnError(rc, "lazy_cache_simulate")
    return s.as_dict()
