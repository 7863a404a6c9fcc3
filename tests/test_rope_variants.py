"""Positional variants: the oracle's explicit-frequency and interleaved rotations and
its Llama-3.1 frequency rule, pinned against closed forms and invariants; and the
host-side checks of the scaled rotation-table entry point (no GPU needed).

The pages state the method for RoPE in general ("Implementação Técnica": only the
relative offset enters a score). Two variants change no kernel: frequency scaling
(only the frequencies move) and the interleaved (GPT-J) pairing (a permutation of
the head dimension applied to q and to the stored K)."""
import ctypes
import dataclasses
import math

import numpy as np
import pytest

import oracle
from paged_kv_cache_57_gb300 import workloads as W


def _omega(d, theta):
    return theta ** (-2.0 * np.arange(d // 2) / d)


def test_rotate_ex_with_default_frequencies_is_rotate():
    x = np.random.default_rng(1).standard_normal(64)
    for n in (0.0, 3.0, -17.0, 12345.0):
        a = oracle.rope_rotate(x, n, 1e4)
        assert np.array_equal(oracle.rope_rotate_ex(x, n, 1e4), a)
        # numpy's power may differ from C's pow in the last bit of a frequency
        assert np.allclose(oracle.rope_rotate_ex(x, n, 1e4, freqs=_omega(64, 1e4)), a, rtol=0, atol=1e-14 * (1 + abs(n)))


def test_d2_both_pairings_are_the_plane_rotation():
    # d = 2: one pair, omega_0 = 1; both pairings are [[c, -s], [s, c]].
    x = np.array([0.3, -1.7])
    for n in (0.5, 2.0, -4.25):
        c, s = math.cos(n), math.sin(n)
        want = np.array([c * x[0] - s * x[1], s * x[0] + c * x[1]])
        assert np.allclose(oracle.rope_rotate_ex(x, n, 1e4), want, atol=1e-15)
        assert np.allclose(oracle.rope_rotate_ex(x, n, 1e4, interleaved=True), want, atol=1e-15)


def test_interleaved_is_rotate_half_on_the_deinterleaved_dimension():
    d = 64
    perm = np.concatenate([np.arange(0, d, 2), np.arange(1, d, 2)])  # pair (2f, 2f+1) -> (f, f + d/2)
    x = np.random.default_rng(2).standard_normal(d)
    for n in (1.0, 77.0, -300.0):
        y_int = oracle.rope_rotate_ex(x, n, 1e4, interleaved=True)
        y_half = oracle.rope_rotate(x[perm], n, 1e4)
        assert np.allclose(y_int[perm], y_half, atol=1e-13)


@pytest.mark.parametrize("interleaved", [False, True])
def test_relative_offset_property_for_both_pairings(interleaved):
    rng = np.random.default_rng(3)
    q, k = rng.standard_normal(64), rng.standard_normal(64)
    f = oracle.llama3_freqs(64, 5e5, 8.0, 1.0, 4.0, 8192)
    for m, p in ((100, 40), (5000, 4990), (20000, 3)):
        lhs = oracle.rope_rotate_ex(q, m, 5e5, f, interleaved) @ oracle.rope_rotate_ex(k, p, 5e5, f, interleaved)
        rhs = oracle.rope_rotate_ex(q, m - p, 5e5, f, interleaved) @ k
        assert abs(lhs - rhs) < 1e-10


def test_llama3_factor_one_is_identity():
    for d, theta in ((64, 1e4), (128, 5e5)):
        assert np.allclose(oracle.llama3_freqs(d, theta, 1.0, 1.0, 4.0, 8192), _omega(d, theta), rtol=1e-15)


def test_llama3_wavelength_bands():
    d, theta, factor, lo, hi, L = 128, 5e5, 8.0, 1.0, 4.0, 8192
    w = oracle.llama3_freqs(d, theta, 1.0, lo, hi, L)  # unscaled, with the oracle's own pow
    assert np.allclose(w, _omega(d, theta), rtol=1e-14)
    f = oracle.llama3_freqs(d, theta, factor, lo, hi, L)
    lam = 2 * math.pi / w
    short, long_ = lam < L / hi, lam > L / lo
    assert short.any() and long_.any() and (~short & ~long_).any()  # all three bands occur at these sizes
    assert np.array_equal(f[short], w[short])                       # short wavelengths are kept
    assert np.array_equal(f[long_], w[long_] / factor)              # long ones slowed by the factor
    mid = ~short & ~long_
    r = f[mid] / w[mid]                                              # in between: 1/factor < ratio < 1
    assert ((r > 1 / factor) & (r < 1)).all()
    assert (np.diff(r) <= 0).all()                                   # and falls as the wavelength grows
    # The blend is continuous at both band edges: s = 1 at lambda = L / hi, s = 0 at L / lo.
    s = lambda lam_: (L / lam_ - lo) / (hi - lo)
    assert s(L / hi) == 1.0 and s(L / lo) == 0.0
    # Llama-3.1-8B values: the fastest frequency (1 rad/token) is kept, the slowest divided by 8.
    assert f[0] == 1.0 and f[-1] == w[-1] / 8


def test_oracle_attention_interleaved_equals_rotate_half_on_permuted_inputs():
    w = W.decode_zipf("rint", batch=3, hq=4, hkv=2, d=64, docs_per_seq=3, doc_tokens=40, pool_docs=5,
                      zipf_s=1.0, suffix_tokens=5, dtype="f32", theta=1e4, seed=211)
    d = w.head_dim
    perm = np.concatenate([np.arange(0, d, 2), np.arange(1, d, 2)])
    wp = dataclasses.replace(w, q=w.q[..., perm].contiguous(), k_pool=w.k_pool[..., perm].contiguous())
    a = oracle.attention(w, interleaved=True)
    b = oracle.attention(wp)
    assert np.allclose(a, b, atol=1e-12)
    # and the pairing matters: the rotate-half result on the unpermuted inputs differs
    assert np.abs(oracle.attention(w) - a).max() > 1e-3


def test_oracle_attention_scaled_frequencies_shift_invariant():
    # Shifting every position by the same constant leaves the outputs unchanged for any frequencies.
    w0 = W.tiny_fp32()
    w1 = W.tiny_fp32(shift=1000)
    f = oracle.llama3_freqs(w0.head_dim, w0.rope_theta, 8.0, 1.0, 4.0, 64)
    assert np.allclose(oracle.attention(w0, freqs=f), oracle.attention(w1, freqs=f), atol=1e-12)
    assert np.abs(oracle.attention(w0, freqs=f) - oracle.attention(w0)).max() > 1e-6


def test_scaled_table_rejects_bad_scaling_without_cuda():
    from paged_kv_cache_57_gb300 import lazy_attn as L
    w = W.tiny_fp32()
    p = L.make_params(num_seqs=w.num_seqs, num_q_heads=w.num_q_heads, num_kv_heads=w.num_kv_heads,
                      head_dim=w.head_dim, num_pool_blocks=w.num_pool_blocks, max_blocks_per_seq=w.max_blocks_per_seq,
                      dtype=w.dtype, rope_theta=w.rope_theta)
    fake = ctypes.c_void_p(4096)  # never dereferenced: the arguments are rejected first
    for bad in ((0.0, 1.0, 4.0, 8192), (8.0, 4.0, 1.0, 8192), (8.0, 1.0, 4.0, 0), (-2.0, 1.0, 4.0, 8192)):
        sc = L.RopeScaling(*bad)
        rc = L._lib.lazy_attn_rope_table_init_scaled(ctypes.byref(p), ctypes.addressof(sc), fake, 1 << 20, None)
        assert rc == L.LAZY_ERR_INVALID_ARG, bad
    perm = L.interleave_perm(8)
    assert list(perm) == [0, 2, 4, 6, 1, 3, 5, 7]


# ---------------------------------------------------------------- partial rotary

def test_partial_rotary_full_width_is_the_full_rotation():
    x = np.random.default_rng(4).standard_normal(64)
    for n in (0.0, 5.0, -123.0):
        assert np.array_equal(oracle.rope_rotate_ex(x, n, 1e4, rot_dims=64), oracle.rope_rotate(x, n, 1e4))


def test_partial_rotary_two_dims_is_one_plane_rotation():
    # r = 2: one pair (0, 1) at rate theta^0 = 1; every other dim passes through.
    x = np.random.default_rng(5).standard_normal(16)
    for interleaved in (False, True):
        for n in (0.75, -3.0, 40.0):
            y = oracle.rope_rotate_ex(x, n, 1e4, interleaved=interleaved, rot_dims=2)
            c, s = math.cos(n), math.sin(n)
            assert np.allclose(y[:2], [c * x[0] - s * x[1], s * x[0] + c * x[1]], atol=1e-14)
            assert np.array_equal(y[2:], x[2:])


def test_partial_rotary_head_is_an_r_dim_rotation_and_tail_passes():
    x = np.random.default_rng(6).standard_normal(128)
    for r in (32, 64):
        for n in (7.0, -1000.0):
            y = oracle.rope_rotate_ex(x, n, 1e4, rot_dims=r)
            assert np.array_equal(y[r:], x[r:])
            # rates theta^(-2i/r): the r-dim vector rotated on its own (rates given
            # explicitly from numpy, so the check does not share the oracle's rate code)
            w = 1e4 ** (-2.0 * np.arange(r // 2) / r)
            half = r // 2
            a, b = x[:half], x[half:r]
            want = np.concatenate([a * np.cos(n * w) - b * np.sin(n * w), b * np.cos(n * w) + a * np.sin(n * w)])
            assert np.allclose(y[:r], want, atol=1e-12)
            assert np.isclose(np.linalg.norm(y), np.linalg.norm(x), rtol=1e-14)


@pytest.mark.parametrize("interleaved", [False, True])
def test_partial_rotary_relative_offset_property(interleaved):
    rng = np.random.default_rng(7)
    q, k = rng.standard_normal(128), rng.standard_normal(128)
    for m, p in ((50, 10), (9000, 8999), (3, 300)):
        lhs = oracle.rope_rotate_ex(q, m, 1e4, None, interleaved, 32) @ oracle.rope_rotate_ex(k, p, 1e4, None,
                                                                                              interleaved, 32)
        rhs = oracle.rope_rotate_ex(q, m - p, 1e4, None, interleaved, 32) @ k
        assert abs(lhs - rhs) < 1e-10


@pytest.mark.parametrize("interleaved", [False, True])
def test_library_layout_reproduces_partial_rotary_in_the_oracle(interleaved):
    """The library's layout (permutation + rates, zero for the unrotated pairs) turned
    into a full-width rotate-half attention on permuted inputs equals the oracle's
    partial rotary on the original inputs: two independent code paths of the oracle."""
    from paged_kv_cache_57_gb300 import lazy_attn as L
    w = W.decode_zipf("rpart", batch=3, hq=4, hkv=2, d=64, docs_per_seq=3, doc_tokens=40, pool_docs=5,
                      zipf_s=1.0, suffix_tokens=5, dtype="f32", theta=1e4, seed=212)
    perm, freqs = L.rotary_layout(64, 16, 1e4, interleaved)
    assert sorted(perm) == list(range(64)) and (freqs[8:] == 0).all()
    wp = dataclasses.replace(w, q=w.q[..., perm].contiguous(), k_pool=w.k_pool[..., perm].contiguous())
    a = oracle.attention(w, rot_dims=16, interleaved=interleaved)
    b = oracle.attention(wp, freqs=freqs)
    assert np.allclose(a, b, atol=1e-12)
    assert np.abs(oracle.attention(w) - a).max() > 1e-3  # rotating only 16 of 64 dims changes the result


def test_rotary_layout_and_explicit_rates_argument_checks():
    from paged_kv_cache_57_gb300 import lazy_attn as L
    for bad in ((64, 0), (64, 3), (64, 66), (63, 32)):
        with pytest.raises(L.LazyAttnError):
            L.rotary_layout(bad[0], bad[1], 1e4)
    w = W.tiny_fp32()
    p = L.make_params(num_seqs=w.num_seqs, num_q_heads=w.num_q_heads, num_kv_heads=w.num_kv_heads,
                      head_dim=w.head_dim, num_pool_blocks=w.num_pool_blocks, max_blocks_per_seq=w.max_blocks_per_seq,
                      dtype=w.dtype, rope_theta=w.rope_theta)
    fake = ctypes.c_void_p(4096)  # never dereferenced: the rates are rejected first
    for bad in (-1e-3, 4.5, float("nan"), float("inf")):
        f = np.full(w.head_dim // 2, 0.5)
        f[3] = bad
        rc = L._lib.lazy_attn_rope_table_init_freqs(ctypes.byref(p), f.ctypes.data, fake, 1 << 20, None)
        assert rc == L.LAZY_ERR_INVALID_ARG, bad


# ---------------------------------------------------------------- ALiBi

def _alibi_w(shift=0, hq=4, hkv=2):
    return W.decode_zipf("ralibi", batch=3, hq=hq, hkv=hkv, d=64, docs_per_seq=3, doc_tokens=40, pool_docs=4,
                         zipf_s=1.0, suffix_tokens=5, dtype="f32", theta=1e4, seed=213, shift=shift)


def test_alibi_zero_slopes_is_no_bias():
    w = _alibi_w()
    zero = np.zeros(w.head_dim // 2)
    assert np.array_equal(oracle.attention(w, freqs=zero, alibi=np.zeros(w.num_q_heads)),
                          oracle.attention(w, freqs=zero))


def test_alibi_depends_only_on_relative_positions():
    slopes = np.array([0.5, 0.25, 0.125, 0.0625])
    zero = np.zeros(32)
    a = oracle.attention(_alibi_w(), freqs=zero, alibi=slopes)
    b = oracle.attention(_alibi_w(shift=777), freqs=zero, alibi=slopes)
    assert np.allclose(a, b, atol=1e-12)
    assert np.abs(a - oracle.attention(_alibi_w(), freqs=zero)).max() > 1e-3


def test_alibi_steep_slope_selects_the_most_recent_key():
    # slope -> infinity: all weight on the key nearest the query (position m - 1 in decode)
    w = _alibi_w()
    out = oracle.attention(w, freqs=np.zeros(32), alibi=np.full(w.num_q_heads, 1e4))
    for s in range(w.num_seqs):
        doc, ln = w.seq_segments(s)[-1]
        phys = int(w.doc_blocks[w.doc_block_indptr[doc] + (ln - 1) // 16])
        for h in range(w.num_q_heads):
            v_last = w.v_pool[phys, h // (w.num_q_heads // w.num_kv_heads), (ln - 1) % 16].double().numpy()
            assert np.allclose(out[s, h], v_last, atol=1e-12)


def test_alibi_slopes_closed_form():
    from paged_kv_cache_57_gb300 import lazy_attn as L
    assert np.array_equal(L.alibi_slopes(8), np.float32(2.0) ** -np.arange(1, 9, dtype=np.float32))
    s12 = L.alibi_slopes(12)  # 8 of the 8-head sequence, then the odd-indexed slopes of 16 heads
    assert np.array_equal(s12[:8], L.alibi_slopes(8))
    assert np.allclose(s12[8:], 2.0 ** -(np.arange(4) + 0.5), rtol=1e-7)
    with pytest.raises(L.LazyAttnError):
        L.alibi_slopes(0)


def test_alibi_calls_and_key_position_words_go_together_without_cuda():
    # The ALiBi calls read key positions from words packed with key_positions = 1;
    # every other call reads document starts and must refuse such words.
    from paged_kv_cache_57_gb300 import lazy_attn as L
    w = _alibi_w()
    fake = ctypes.c_void_p(4096)  # never dereferenced: the arguments are rejected first

    def params(key_positions, dtype="bf16"):
        return L.make_params(num_seqs=w.num_seqs, num_q_heads=w.num_q_heads, num_kv_heads=w.num_kv_heads,
                             head_dim=w.head_dim, num_pool_blocks=w.num_pool_blocks,
                             max_blocks_per_seq=w.max_blocks_per_seq, dtype=dtype, rope_theta=w.rope_theta,
                             key_positions=key_positions)

    def shared_alibi(p, slopes):
        return L._lib.lazy_attn_decode_shared_alibi(ctypes.byref(p), *([fake] * 6), 1, fake, 1, fake, slopes,
                                                    fake, fake, 1 << 20, None)

    def decode_alibi(p, slopes):
        return L._lib.lazy_attn_decode_alibi(ctypes.byref(p), *([fake] * 7), slopes, fake, fake, 1 << 20, None)

    doc_words, key_words = params(False), params(True)
    bad = L.LAZY_ERR_INVALID_ARG
    assert shared_alibi(doc_words, fake) == bad and decode_alibi(doc_words, fake) == bad
    assert shared_alibi(key_words, None) == bad and decode_alibi(key_words, None) == bad
    assert shared_alibi(key_words, ctypes.c_void_p(4098)) == bad  # slopes not 4-byte aligned
    assert decode_alibi(params(True, "f32"), fake) == L.LAZY_ERR_UNSUPPORTED
    assert L._lib.lazy_attn_decode(ctypes.byref(key_words), *([fake] * 8), fake, 1 << 20, None) == bad
    assert L._lib.lazy_attn_decode_shared(ctypes.byref(key_words), *([fake] * 6), 1, fake, 1, fake, fake, fake,
                                          1 << 20, None) == bad
    p = params(True)
    p.head_dim = 128  # the prefill's only head size
    assert L._lib.lazy_attn_prefill(ctypes.byref(p), fake, fake, fake, 1, 1, *([fake] * 7), 1 << 20, None) == bad
    p = params(True)
    p.key_positions = 2
    assert decode_alibi(p, fake) == bad
