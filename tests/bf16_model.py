"""Emulation of the bf16 tensor-core path's operand roundings (numpy fp64).

The CUDA kernels multiply bf16 operands on the tensor cores: the rotated query
q' (scaled by sm_scale * log2(e)), in prefill the rotated key block R_p K, and
the softmax weights P are rounded to bf16 before their products; everything
else is fp32 or exact. On a
row whose output element is near zero (values that cancel), those two or three
roundings alone can move the result by more than 2e-3 + 2e-2 |ref|.

This module restates the attention with exactly those rounding points and
nothing else, so that a GPU element outside the oracle tolerance can be
checked against it: if the GPU agrees with this emulation (to the same
tolerance), the deviation is the arithmetic of bf16 operands, not an error in
keys, masks, positions or rotations -- those would miss both references.
It is test support, written from the method's definition like the brute force
(complex-form RoPE from tests/brute.py), and shares nothing with the kernels.
"""
from __future__ import annotations

import numpy as np
import torch

from brute import rope


def _bf16(x):
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16).double().numpy()


# Unit roundoff of bf16 (8 significand bits): round-to-nearest moves a value by at
# most this fraction of itself.
BF16_U = 2.0 ** -8


def emulate(w, rows, lazy: bool = True, k_pool=None, freqs=None, alibi=None, weight_bound: bool = False,
            sm_scale: float = 0.0):
    """[len(rows), Hq, d] for query rows ``rows`` of workload ``w`` (``freqs``: rotation
    frequencies other than theta^(-2i/d); ``alibi``: per-head slopes of the bias
    -slope (m - n), added in fp32 to the scores before the exponentials; ``sm_scale``:
    softmax scale, 0 for 1/sqrt(d)).

    The weights here are rounded to bf16 relative to the row's global maximum; a
    split-K kernel rounds each one relative to the running maximum of its own split,
    a different but equally valid bf16 value within BF16_U of the exact weight. With
    ``weight_bound`` the call also returns, per element, the first-order bound on what
    two such roundings can change in the output, 2 BF16_U sum_j p_j |v_j - o| (exact
    weights p, output o), as a second array of the same shape."""
    kp = (w.k_pool if k_pool is None else k_pool).double().numpy()
    vp = w.v_pool.double().numpy()
    q = w.q.double().numpy()
    if w.kind == "decode":
        q_seq = np.arange(w.num_seqs)
        q_m = np.asarray(w.q_pos, np.int64)
    else:
        cu = np.asarray(w.cu_seqlens_q)
        q_seq = np.repeat(np.arange(w.num_seqs), np.diff(cu))
        q_m = np.concatenate([w.q_start[s] + np.arange(cu[s + 1] - cu[s]) for s in range(w.num_seqs)])
    g = w.num_q_heads // w.num_kv_heads
    d, theta = w.head_dim, w.rope_theta
    scale = np.log2(np.e) * (sm_scale if sm_scale > 0 else 1.0 / np.sqrt(d))
    out = np.zeros((len(rows), w.num_q_heads, d))
    bound = np.zeros_like(out)
    for oi, r in enumerate(np.asarray(rows)):
        s, m = int(q_seq[r]), int(q_m[r])
        Ks, Vs, Ps, pos = [], [], [], []
        p = int(w.seq_pos0[s])
        for doc, L in w.seq_segments(s):
            base = int(w.doc_block_indptr[doc])
            ids = [int(w.doc_blocks[base + j // 16]) for j in range(L)]
            Ks.append(np.stack([kp[ids[j], :, j % 16] for j in range(L)]))
            Vs.append(np.stack([vp[ids[j], :, j % 16] for j in range(L)]))
            Ps.append(np.full(L, p))
            pos.append(p + np.arange(L))
            p += L
        if not Ks:
            continue
        K, V, P, pos = np.concatenate(Ks), np.concatenate(Vs), np.concatenate(Ps), np.concatenate(pos)
        vis = pos <= m
        K, V, P = K[vis], V[vis], P[vis]
        if w.kind == "prefill" and lazy:
            K = _bf16(rope(K.transpose(1, 0, 2), P, theta, freqs).transpose(1, 0, 2))  # one rotation by R_p, bf16
        for h in range(w.num_q_heads):
            kh = K[:, h // g]
            # every kernel folds scale * log2(e) into q' before the bf16 rounding
            if w.kind == "decode" and lazy:
                # q re-rotated by R_{m-p} per document
                qd = {pp: _bf16(rope(q[r, h], m - pp, theta, freqs) * scale) for pp in np.unique(P)}
                sc = np.array([qd[P[j]] @ kh[j] for j in range(len(P))])
            else:
                sc = kh @ _bf16(rope(q[r, h], m, theta, freqs) * scale)
            if alibi is not None:
                sc = sc - float(alibi[h]) * np.log2(np.e) * (m - pos[vis])
            e = _bf16(np.exp2(sc - sc.max()))
            out[oi, h] = (e[:, None] * V[:, h // g]).sum(0) / e.sum()
            if weight_bound:
                pw = np.exp2(sc - sc.max())
                pw /= pw.sum()
                o = pw @ V[:, h // g]
                bound[oi, h] = 2 * BF16_U * (pw[:, None] * np.abs(V[:, h // g] - o)).sum(0)
    return (_bf16(out), bound) if weight_bound else _bf16(out)
