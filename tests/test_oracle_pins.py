"""Pins of the CPU oracle against things other than itself (CPU only).

Each test fixes a part of the oracle by something the pages or the mathematics
determine: closed forms of the rotation, the relative-offset identity, brute
force from raw keys, textbook attention via torch's CPU SDPA, one-key and
zero-query closed forms, the GQA-as-repeated-heads reduction, the running
softmax of the FlashAttention lesson, and the cache byte counts printed on the
pages.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from brute import brute_attention, rope
from paged_kv_cache_57_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rel_err(a, b):
    return float(np.max(np.abs(a - b)) / max(1e-300, np.max(np.abs(b))))


# ---------------------------------------------------------------- rotation closed forms

def test_rotation_d2_closed_form():
    # d = 2: one pair, omega_0 = theta^0 = 1, so R_n is the plane rotation by n radians.
    for n in (1.0, 2.0, -3.0, 100.0):
        y = oracle.rope_rotate(np.array([1.0, 0.0]), n, 1e4)
        assert np.allclose(y, [math.cos(n), math.sin(n)], atol=1e-15)
        y = oracle.rope_rotate(np.array([0.0, 1.0]), n, 1e4)
        assert np.allclose(y, [-math.sin(n), math.cos(n)], atol=1e-15)


def test_rotation_pairing_and_frequencies():
    # d = 4, theta = 1e4: pairs (0, 2) and (1, 3), omegas 1 and 1e4^(-1/2) = 0.01.
    x = np.array([0.0, 1.0, 0.0, 0.0])
    y = oracle.rope_rotate(x, 3.0, 1e4)
    assert np.allclose(y, [0.0, math.cos(0.03), 0.0, math.sin(0.03)], atol=1e-15)
    x = np.array([0.0, 0.0, 2.0, 0.0])
    y = oracle.rope_rotate(x, 5.0, 1e4)
    assert np.allclose(y, [-2 * math.sin(5.0), 0.0, 2 * math.cos(5.0), 0.0], atol=1e-14)


def test_rotation_group_law_and_orthogonality():
    rng = np.random.default_rng(1)
    for d, theta in ((64, 1e4), (128, 5e5)):
        x = rng.standard_normal(d)
        for a, b in ((3, 5), (1000, -7), (65536, 4096)):
            ab = oracle.rope_rotate(oracle.rope_rotate(x, b, theta), a, theta)
            assert rel_err(ab, oracle.rope_rotate(x, a + b, theta)) < 1e-11
            assert abs(np.linalg.norm(oracle.rope_rotate(x, a, theta)) - np.linalg.norm(x)) < 1e-12
        assert np.array_equal(oracle.rope_rotate(x, 0.0, theta), x)


def test_rotation_matches_complex_brute_force():
    rng = np.random.default_rng(2)
    x = rng.standard_normal(128)
    for n in (0, 1, 17, 4160, 131071):
        assert np.allclose(oracle.rope_rotate(x, n, 5e5), rope(x, n, 5e5), atol=1e-12)


def test_relative_offset_identity():
    # <R_m q, R_n k> = <R_{m-n} q, k>  (summary, "Mathematical Equivalence")
    rng = np.random.default_rng(3)
    q, k = rng.standard_normal(128), rng.standard_normal(128)
    for m, n in ((4160, 512), (16384, 0), (100, 99), (131072, 65536)):
        lhs = oracle.rope_rotate(q, m, 5e5) @ oracle.rope_rotate(k, n, 5e5)
        rhs = oracle.rope_rotate(q, m - n, 5e5) @ k
        assert abs(lhs - rhs) < 1e-10 * max(1.0, abs(lhs))


# ---------------------------------------------------------------- online softmax (P1)

@pytest.mark.parametrize("tile", [1, 3, 16, 100])
def test_tiled_softmax_equals_one_shot(tile):
    rng = np.random.default_rng(4)
    n, d = 37, 8
    q, K, V = rng.standard_normal(d) * 3, rng.standard_normal((n, d)), rng.standard_normal((n, d))
    ref = oracle.softmax_dot(q, K, V)
    # textbook definition written out
    s = K @ q
    e = np.exp(s - s.max())
    assert np.allclose(ref, (e[:, None] * V).sum(0) / e.sum(), atol=1e-14)
    assert np.allclose(oracle.tiled_softmax_dot(q, K, V, tile), ref, atol=1e-13)


# ---------------------------------------------------------------- attention vs brute force

def _small_workloads():
    yield W.tiny_fp32()
    yield W.decode_zipf("gqa_small", batch=3, hq=8, hkv=2, d=64, theta=5e5, docs_per_seq=3, doc_tokens=32,
                        pool_docs=6, zipf_s=1.0, suffix_tokens=5, seed=11)
    yield W.prefill_zipf("prefill_small", batch=2, hq=4, hkv=2, d=64, theta=1e4, docs_per_seq=2,
                         doc_tokens=40, pool_docs=4, zipf_s=1.2, chunk_tokens=[19, 33], seed=12)
    d, p = W.mixed_mqa(n_decode=2, n_prefill=1, chunk=20, hq=4, hkv=1, d=64, pool_docs=8, ctx_lo=20,
                       ctx_hi=150, doc_lo=5, doc_hi=40, seed=13)
    yield d
    yield p


@pytest.mark.parametrize("w", list(_small_workloads()), ids=lambda w: w.name)
def test_oracle_matches_brute_force(w):
    ref = brute_attention(w)
    got = oracle.attention(w)
    assert got.shape == ref.shape
    assert rel_err(got, ref) < 1e-12


def test_shift_invariance():
    base = oracle.attention(W.tiny_fp32())
    for c in (1, 16, 1000, 70000):
        assert rel_err(oracle.attention(W.tiny_fp32(shift=c)), base) < 1e-12
    pw = dict(batch=2, hq=4, hkv=2, d=64, theta=1e4, docs_per_seq=2, doc_tokens=24, pool_docs=3,
              zipf_s=1.0, chunk_tokens=17, seed=21)
    pbase = oracle.attention(W.prefill_zipf("p", **pw))
    assert rel_err(oracle.attention(W.prefill_zipf("p", shift=777, **pw)), pbase) < 1e-12


# ---------------------------------------------------------------- textbook reductions

def _sdpa(q, k, v, causal):
    return torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q), torch.from_numpy(k), torch.from_numpy(v), is_causal=causal).numpy()


def test_single_document_at_zero_is_plain_rope_attention():
    # One document at p = 0: K_adj = K_stored, so decode is softmax(R_m q K^T / sqrt d) V.
    w = W.decode_zipf("one_doc", batch=1, hq=4, hkv=4, d=64, theta=1e4, docs_per_seq=1, doc_tokens=45,
                      pool_docs=1, zipf_s=1.0, seed=31)
    got = oracle.attention(w)[0]
    kp, vp = w.k_pool.double().numpy(), w.v_pool.double().numpy()
    ids = w.doc_blocks
    K = np.concatenate([kp[i] for i in ids], axis=1)[:, :45]  # [H, 45, d]
    V = np.concatenate([vp[i] for i in ids], axis=1)[:, :45]
    q = rope(w.q.double().numpy()[0], int(w.q_pos[0]), 1e4)[:, None, :]  # [H, 1, d]
    assert rel_err(got, _sdpa(q, K, V, False)[:, 0]) < 1e-12


def test_single_chunk_prefill_is_causal_rope_attention():
    # Prefill with no cached documents: the chunk alone at p = q_start = 0 must be
    # standard causal RoPE self-attention (GQA mapping h -> h // g).
    w = W.prefill_zipf("chunk_only", batch=1, hq=4, hkv=2, d=64, theta=1e4, docs_per_seq=0,
                       doc_tokens=16, pool_docs=1, zipf_s=1.0, chunk_tokens=37, seed=32)
    got = oracle.attention(w)  # [37, 4, d]
    kp, vp = w.k_pool.double().numpy(), w.v_pool.double().numpy()
    K = np.concatenate([kp[i] for i in w.doc_blocks], axis=1)[:, :37]  # [Hkv, 37, d]
    V = np.concatenate([vp[i] for i in w.doc_blocks], axis=1)[:, :37]
    q = rope(w.q.double().numpy().transpose(1, 0, 2), np.arange(37), 1e4)  # [Hq, 37, d]
    ref = _sdpa(q, np.repeat(K, 2, axis=0), np.repeat(V, 2, axis=0), True)
    assert rel_err(got.transpose(1, 0, 2), ref) < 1e-12


def test_one_key_context_returns_v():
    w = W.decode_zipf("one_key", batch=2, hq=4, hkv=2, d=64, theta=5e5, docs_per_seq=1, doc_tokens=1,
                      pool_docs=2, zipf_s=1.0, seed=33)
    got = oracle.attention(w)
    vp = w.v_pool.double().numpy()
    for s in range(2):
        doc = w.seg_doc[w.seg_indptr[s]]
        phys = w.doc_blocks[w.doc_block_indptr[doc]]
        for h in range(4):
            assert np.array_equal(got[s, h], vp[phys, h // 2, 0])


def test_zero_query_averages_values():
    w = W.decode_zipf("zero_q", batch=2, hq=2, hkv=1, d=64, theta=5e5, docs_per_seq=3, doc_tokens=21,
                      pool_docs=5, zipf_s=1.0, seed=34)
    w.q.zero_()
    got = oracle.attention(w)
    vp = w.v_pool.double().numpy()
    for s in range(2):
        rows = []
        for doc, L in w.seq_segments(s):
            for j in range(L):
                rows.append(vp[w.doc_blocks[w.doc_block_indptr[doc] + j // 16], 0, j % 16])
        assert rel_err(got[s, 0], np.mean(rows, axis=0)) < 1e-13


def test_gqa_equals_repeated_kv_heads():
    w = W.decode_zipf("gqa", batch=2, hq=8, hkv=2, d=64, theta=5e5, docs_per_seq=2, doc_tokens=20,
                      pool_docs=3, zipf_s=1.0, seed=35)
    got = oracle.attention(w)
    w_mha = W.Workload(**{**w.__dict__, "num_kv_heads": 8})
    ref = oracle.attention(w_mha, k_pool=w.k_pool.repeat_interleave(4, dim=1),
                           v_pool=w.v_pool.repeat_interleave(4, dim=1))
    assert np.array_equal(got, ref)


def test_empty_sequence_gives_zero():
    w = W.tiny_fp32()
    w0 = W.Workload(**{**w.__dict__, "seg_indptr": np.array([0, 0], np.int32),
                       "seg_doc": np.zeros(0, np.int32), "seg_len": np.zeros(0, np.int32)})
    assert np.array_equal(oracle.attention(w0), np.zeros((1, 4, 64)))


def test_hole_slots_are_not_read():
    # Partial tail blocks hold NaN past each document's end; the oracle must not touch them.
    d, p = W.mixed_mqa(n_decode=3, n_prefill=1, chunk=21, hq=2, hkv=1, d=64, pool_docs=8, ctx_lo=30,
                       ctx_hi=200, doc_lo=5, doc_hi=40, seed=36)
    assert np.isfinite(oracle.attention(d)).all()
    assert np.isfinite(oracle.attention(p)).all()


# ---------------------------------------------------------------- cache byte counts (pages)

def test_kv_cache_bytes_match_pages():
    rows = [ln.split() for ln in open(os.path.join(GOLDEN, "kv_cache_bytes.txt"))
            if ln.strip() and not ln.startswith("#")]
    assert len(rows) == 5
    for r in rows:
        *args, expected = map(float, r)
        assert oracle.kv_cache_bytes(*args) == expected


def test_workload_byte_accounting_follows_page_formula():
    for w in (W.tiny_fp32(), next(iter(_small_workloads()))):
        elt = 4 if w.dtype == "f32" else 2
        assert W.kv_bytes_logical(w) == oracle.kv_cache_bytes(1, w.num_kv_heads, w.head_dim,
                                                              int(w.tokens_per_seq().sum()), 1, elt)
