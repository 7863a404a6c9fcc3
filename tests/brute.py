"""Brute-force LazyAttention from raw (unrotated) keys, numpy fp64, tiny inputs only.

Written independently of the C oracle, in complex form: the rotate-half pair
(x_i, x_{i+d/2}) is the complex number z_i = x_i + 1j*x_{i+d/2}, and RoPE at
position n multiplies it by exp(1j * n * omega_i), omega_i = theta**(-2i/d).

The raw key of document token j is recovered from the stored row as
R_{-j} K_stored[j]; the score of a query at absolute position m against that
token placed at absolute position p+j is then <R_m q, R_{p+j} k_raw> / sqrt(d):
full absolute RoPE, no relative-offset shortcut (LazyAttention technical summary,
"Mathematical Equivalence", states the two agree).
"""
from __future__ import annotations

import numpy as np


def _omega(d: int, theta: float) -> np.ndarray:
    return theta ** (-2.0 * np.arange(d // 2) / d)


def to_complex(x: np.ndarray) -> np.ndarray:
    h = x.shape[-1] // 2
    return x[..., :h] + 1j * x[..., h:]


def from_complex(z: np.ndarray) -> np.ndarray:
    return np.concatenate([z.real, z.imag], axis=-1)


def rope(x: np.ndarray, n, theta: float, freqs=None) -> np.ndarray:
    """R_n x for x [..., d]; n broadcasts against x's leading dims. ``freqs`` replaces
    theta^(-2i/d)."""
    d = x.shape[-1]
    ang = np.asarray(n, dtype=np.float64)[..., None] * (_omega(d, theta) if freqs is None else np.asarray(freqs))
    return from_complex(to_complex(x) * np.exp(1j * ang))


def brute_attention(w, rows=None, k_pool=None, v_pool=None) -> np.ndarray:
    import torch

    kp = (w.k_pool if k_pool is None else k_pool).to(torch.float64).numpy()
    vp = (w.v_pool if v_pool is None else v_pool).to(torch.float64).numpy()
    q = w.q.to(torch.float64).numpy()
    if w.kind == "decode":
        q_seq = np.arange(w.num_seqs)
        q_m = np.asarray(w.q_pos, np.int64)
    else:
        cu = np.asarray(w.cu_seqlens_q)
        q_seq = np.repeat(np.arange(w.num_seqs), np.diff(cu))
        q_m = np.concatenate([w.q_start[s] + np.arange(cu[s + 1] - cu[s]) for s in range(w.num_seqs)])
    if rows is None:
        rows = np.arange(q.shape[0])
    g = w.num_q_heads // w.num_kv_heads
    d, theta = w.head_dim, w.rope_theta
    out = np.zeros((len(rows), w.num_q_heads, d))
    for oi, r in enumerate(rows):
        s, m = int(q_seq[r]), int(q_m[r])
        kraw, vals, kpos = [], [], []
        p = int(w.seq_pos0[s])
        for doc, L in w.seq_segments(s):
            base = int(w.doc_block_indptr[doc])
            for j in range(L):
                phys = int(w.doc_blocks[base + j // 16])
                kraw.append(rope(kp[phys, :, j % 16, :], -j, theta))  # [Hkv, d]
                vals.append(vp[phys, :, j % 16, :])
                kpos.append(p + j)
            p += L
        if not kraw:
            continue
        kraw, vals, kpos = np.stack(kraw), np.stack(vals), np.asarray(kpos)
        vis = kpos <= m
        if not vis.any():
            continue
        kabs = rope(kraw, kpos[:, None], theta)  # [n, Hkv, d] at absolute positions
        for h in range(w.num_q_heads):
            qa = rope(q[r, h], m, theta)
            sc = kabs[vis, h // g, :] @ qa / np.sqrt(d)
            e = np.exp(sc - sc.max())
            out[oi, h] = (e[:, None] * vals[vis, h // g, :]).sum(0) / e.sum()
    return out
