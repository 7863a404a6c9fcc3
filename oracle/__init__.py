"""CPU fp64 oracle for LazyAttention (test infrastructure only).

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package. The product (``paged_kv_cache_57_gb300``) never
imports it, and it imports nothing from the product.

The arithmetic lives in ``lazy_oracle.c`` (plain C, fp64, OpenMP); this module
compiles it with gcc and marshals arrays. Definitions and citations are in the
C file's header. Parity status: the attention output is pinned only through the
checks in ``tests/test_oracle_pins.py`` (brute force from raw keys, the
relative-offset identity, textbook reductions and closed forms); the pages
print no numeric worked example of LazyAttention itself.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "lazy_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "liblazyoracle.so")
_lock = threading.Lock()
_lib = None

_i32p = np.ctypeslib.ndpointer(dtype=np.int32, flags="C_CONTIGUOUS")
_f64p = np.ctypeslib.ndpointer(dtype=np.float64, flags="C_CONTIGUOUS")


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/liblazyoracle.so`` (gcc, -O2, OpenMP)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c99", _SRC,
                               "-o", tmp, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_SO)
            L.lo_rope_rotate.argtypes = [ctypes.c_int, ctypes.c_double, ctypes.c_double, _f64p, _f64p]
            L.lo_rope_rotate_ex.argtypes = [ctypes.c_int, ctypes.c_double, ctypes.c_void_p, ctypes.c_int,
                                            ctypes.c_double, _f64p, _f64p]
            L.lo_rope_rotate_partial.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_void_p,
                                                 ctypes.c_int, ctypes.c_double, _f64p, _f64p]
            L.lo_llama3_freqs.argtypes = [ctypes.c_int] + [ctypes.c_double] * 5 + [_f64p]
            L.lo_softmax_dot.argtypes = [ctypes.c_int, ctypes.c_int, _f64p, _f64p, _f64p, _f64p]
            L.lo_tiled_softmax_dot.argtypes = [ctypes.c_int, ctypes.c_int, _f64p, _f64p, _f64p,
                                               ctypes.c_int, _f64p]
            L.lo_kv_cache_bytes.restype = ctypes.c_double
            L.lo_kv_cache_bytes.argtypes = [ctypes.c_double] * 6
            L.lo_num_threads.restype = ctypes.c_int
            L.lo_set_num_threads.argtypes = [ctypes.c_int]
            L.lo_attention.restype = ctypes.c_int
            L.lo_attention.argtypes = [
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_double,
                ctypes.c_int, ctypes.c_int, ctypes.c_void_p, _i32p, _i32p, ctypes.c_void_p,
                ctypes.c_void_p, ctypes.c_int64, _i32p, _i32p, _i32p, _i32p, _i32p, _i32p, _f64p]
            L.lo_attention_ex.restype = ctypes.c_int
            L.lo_attention_ex.argtypes = [
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_void_p,
                ctypes.c_int, ctypes.c_double, ctypes.c_int, ctypes.c_int, ctypes.c_void_p, _i32p, _i32p,
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, _i32p, _i32p, _i32p, _i32p, _i32p, _i32p, _f64p]
            L.lo_attention_partial.restype = ctypes.c_int
            L.lo_attention_partial.argtypes = [
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double,
                ctypes.c_void_p, ctypes.c_int, ctypes.c_double, ctypes.c_int, ctypes.c_int, ctypes.c_void_p, _i32p,
                _i32p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, _i32p, _i32p, _i32p, _i32p, _i32p, _i32p,
                ctypes.c_void_p, _f64p]
            _lib = L
    return _lib


def num_threads() -> int:
    return int(lib().lo_num_threads())


def set_num_threads(n: int) -> None:
    lib().lo_set_num_threads(int(n))


def rope_rotate(x: np.ndarray, n: float, theta: float) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float64)
    y = np.empty_like(x)
    lib().lo_rope_rotate(x.shape[-1], float(theta), float(n), x, y)
    return y


def rope_rotate_ex(x: np.ndarray, n: float, theta: float, freqs: Optional[np.ndarray] = None,
                   interleaved: bool = False, rot_dims: Optional[int] = None) -> np.ndarray:
    """R_n x with explicit frequencies (None: theta^(-2i/r)) and rotate-half or
    interleaved (2i, 2i+1) pairing, on the first ``rot_dims`` dims (None: all)."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    y = np.empty_like(x)
    f = None if freqs is None else np.ascontiguousarray(freqs, dtype=np.float64)
    d = x.shape[-1]
    lib().lo_rope_rotate_partial(d, int(rot_dims or d), float(theta), None if f is None else f.ctypes.data,
                                 int(interleaved), float(n), x, y)
    return y


def llama3_freqs(d: int, theta: float, factor: float, low_freq_factor: float, high_freq_factor: float,
                 original_max_position: int) -> np.ndarray:
    """The d/2 rotation frequencies under Llama-3.1 scaling (see lo_llama3_freqs)."""
    out = np.empty(d // 2, np.float64)
    lib().lo_llama3_freqs(int(d), float(theta), float(factor), float(low_freq_factor), float(high_freq_factor),
                          float(original_max_position), out)
    return out


def softmax_dot(q, K, V) -> np.ndarray:
    q, K, V = (np.ascontiguousarray(a, dtype=np.float64) for a in (q, K, V))
    out = np.empty(V.shape[1], np.float64)
    lib().lo_softmax_dot(K.shape[0], q.shape[0], q, K, V, out)
    return out


def tiled_softmax_dot(q, K, V, tile: int) -> np.ndarray:
    q, K, V = (np.ascontiguousarray(a, dtype=np.float64) for a in (q, K, V))
    out = np.empty(V.shape[1], np.float64)
    lib().lo_tiled_softmax_dot(K.shape[0], q.shape[0], q, K, V, int(tile), out)
    return out


def kv_cache_bytes(layers, heads, head_dim, seq, batch, elt_bytes) -> float:
    return float(lib().lo_kv_cache_bytes(layers, heads, head_dim, seq, batch, elt_bytes))


def _bits(t) -> tuple:
    """(numpy view of the stored bits, dtype code) of a CPU torch tensor."""
    import torch
    t = t.contiguous()
    if t.dtype == torch.float32:
        return t.numpy(), 0
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy(), 1
    raise TypeError(f"oracle reads fp32 or bf16 stored tensors, not {t.dtype}")


def e4m3_decode(codes) -> np.ndarray:
    """Values of OCP FP8 E4M3 codes (uint8 array), fp64, from the format's definition:
    sign bit 7, exponent bits 6..3 with bias 7, mantissa bits 2..0; exponent 0 encodes
    subnormals (-1)^s 2^-6 (m / 8); S.1111.111 is NaN; there are no infinities."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    s = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    val = np.where(e == 0, np.ldexp(m / 8.0, -6), np.ldexp(1.0 + m / 8.0, (e - 7).astype(np.int64)))
    val = s * val
    return np.where((c & 0x7F) == 0x7F, np.nan, val)


def fp8_pool_as_bf16(pool):
    """An e4m3 pool (torch.float8_e4m3fn, CPU) as a bf16 tensor of the same values.
    Every e4m3 value has at most 4 significant bits and an exponent in [-9, 8], so it
    is exact in bf16; the conversion is checked."""
    import torch
    vals = e4m3_decode(pool.contiguous().view(torch.uint8).numpy())
    out = torch.from_numpy(vals).to(torch.bfloat16)
    assert np.array_equal(out.double().numpy(), vals, equal_nan=True)
    return out


def query_rows(w):
    """(q_seq, q_m) for every query row of a workload."""
    if w.kind == "decode":
        return np.arange(w.num_seqs, dtype=np.int32), np.asarray(w.q_pos, np.int32)
    cu = np.asarray(w.cu_seqlens_q)
    q_seq = np.repeat(np.arange(w.num_seqs, dtype=np.int32), np.diff(cu)).astype(np.int32)
    q_m = np.concatenate([w.q_start[s] + np.arange(cu[s + 1] - cu[s]) for s in range(w.num_seqs)] or
                         [np.zeros(0)]).astype(np.int32)
    return q_seq, q_m


def attention(w, rows: Optional[Sequence[int]] = None, sm_scale: float = 0.0,
              k_pool=None, v_pool=None, freqs: Optional[np.ndarray] = None, interleaved: bool = False,
              rot_dims: Optional[int] = None, alibi: Optional[np.ndarray] = None, k_scale: float = 1.0,
              v_scale: float = 1.0) -> np.ndarray:
    """fp64 reference output of workload ``w`` for the query rows ``rows`` (all by
    default): decode rows are sequences, prefill rows are chunk tokens. ``freqs``
    replaces theta^(-2i/r); ``interleaved`` pairs dimensions (2i, 2i+1);
    ``rot_dims`` rotates only the first r dims (partial rotary; None: all);
    ``alibi`` [Hq] adds the bias -alibi[h] (m - n) to every score (ALiBi).
    Pools of e4m3 codes (torch.float8_e4m3fn) hold keys code * k_scale and values
    code * v_scale: the scores scale by k_scale (folded into the softmax scale) and
    the output, linear in V, by v_scale.
    Returns [len(rows), Hq, d]."""
    import torch
    kp = w.k_pool if k_pool is None else k_pool
    vp = w.v_pool if v_pool is None else v_pool
    if kp.dtype == torch.float8_e4m3fn or vp.dtype == torch.float8_e4m3fn:
        base = sm_scale if sm_scale > 0 else 1.0 / np.sqrt(w.head_dim)
        return v_scale * attention(w, rows, base * k_scale, fp8_pool_as_bf16(kp), fp8_pool_as_bf16(vp), freqs,
                                   interleaved, rot_dims, alibi)
    q_seq, q_m = query_rows(w)
    q = w.q
    if rows is not None:
        rows = np.asarray(rows, dtype=np.int64)
        q_seq, q_m, q = q_seq[rows], q_m[rows], w.q[rows]
    qb, dt = _bits(q)
    kb, dk = _bits(w.k_pool if k_pool is None else k_pool)
    vb, dv = _bits(w.v_pool if v_pool is None else v_pool)
    assert dt == dk == dv
    nq = qb.shape[0]
    out = np.zeros((nq, w.num_q_heads, w.head_dim), np.float64)
    f = None if freqs is None else np.ascontiguousarray(freqs, dtype=np.float64)
    al = None if alibi is None else np.ascontiguousarray(alibi, dtype=np.float64)
    if al is not None and al.shape != (w.num_q_heads,):
        raise ValueError("alibi needs one slope per query head")
    rc = lib().lo_attention_partial(w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim,
                            int(rot_dims or w.head_dim), float(w.rope_theta),
                            None if f is None else f.ctypes.data, int(interleaved),
                            float(sm_scale), dt, nq, qb.ctypes.data, np.ascontiguousarray(q_seq, np.int32),
                            np.ascontiguousarray(q_m, np.int32), kb.ctypes.data, vb.ctypes.data,
                            int(kb.shape[0]), np.ascontiguousarray(w.seg_indptr, np.int32),
                            np.ascontiguousarray(w.seg_doc, np.int32), np.ascontiguousarray(w.seg_len, np.int32),
                            np.ascontiguousarray(w.seq_pos0, np.int32),
                            np.ascontiguousarray(w.doc_block_indptr, np.int32),
                            np.ascontiguousarray(w.doc_blocks, np.int32),
                            None if al is None else al.ctypes.data, out)
    if rc != 0:
        raise ValueError("oracle: malformed layout")
    return out
