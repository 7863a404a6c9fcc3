"""GPU parity for the positional variants that need no kernel of their own:
Llama-3.1 frequency scaling (a rotation table built from the scaled frequencies)
and the interleaved (GPT-J) pairing (q and stored K permuted along the head
dimension), on the per-sequence decode, the shared-run decode and the prefill,
against the oracle's explicit-frequency / interleaved rotation."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from bf16_model import emulate
from gpu_util import FEW_KEY_FALLBACK_FRAC, assert_close, decode, decode_shared, la, prefill, shared_plan, to_device
from paged_kv_cache_57_gb300 import workloads as W

pytestmark = pytest.mark.gpu

# A short original context so that all three wavelength bands fall inside these workloads' positions.
SCALING = dict(factor=8.0, low_freq_factor=1.0, high_freq_factor=4.0, original_max_position=256)


@pytest.fixture(autouse=True)
def _clean_status():
    la().device_status(clear=True)
    yield
    assert la().device_status(clear=True) == 0, "device status word set"


def _freqs(w):
    return oracle.llama3_freqs(w.head_dim, w.rope_theta, SCALING["factor"], SCALING["low_freq_factor"],
                               SCALING["high_freq_factor"], SCALING["original_max_position"])


def _scaled_device(w):
    L = la()
    dv = to_device(w)
    dv.rope = L.rope_table_init(dv.p, scaling=L.RopeScaling(**SCALING))
    return dv


def _interleaved_device(w):
    perm = la().interleave_perm(w.head_dim)
    wp = dataclasses.replace(w, q=w.q[..., perm].contiguous(), k_pool=w.k_pool[..., perm].contiguous())
    return wp, to_device(wp)


def test_decode_f32_scaled_frequencies():
    w = W.decode_zipf("vs32", batch=4, hq=8, hkv=2, d=64, docs_per_seq=4, doc_tokens=300, pool_docs=6, zipf_s=1.0,
                      suffix_tokens=9, dtype="f32", theta=1e4, seed=301)
    f = _freqs(w)
    ref = oracle.attention(w, freqs=f)
    assert np.abs(ref - oracle.attention(w)).max() > 1e-3  # the scaling changes the result at these positions
    assert_close(decode(_scaled_device(w)), ref, "f32", "f32 decode, scaled frequencies")


def test_shared_decode_bf16_scaled_frequencies():
    w = W.decode_zipf("vsb", batch=8, hq=32, hkv=8, d=128, docs_per_seq=3, doc_tokens=260, pool_docs=4, zipf_s=1.0,
                      suffix_tokens=20, seed=302)
    f = _freqs(w)
    dv = _scaled_device(w)
    ref = oracle.attention(w, freqs=f)
    emu = lambda r: emulate(w, r, freqs=f)
    assert_close(decode_shared(dv, shared_plan(dv)), ref, "bf16", "shared decode, scaled", emulate=emu)
    assert_close(decode(dv), ref, "bf16", "per-sequence decode, scaled", emulate=emu)


@pytest.mark.parametrize("hq,hkv", [(8, 2), (6, 2)])  # even GQA ratio: stream-K kernel; odd: one-tile kernel
def test_prefill_scaled_frequencies(hq, hkv):
    w = W.prefill_zipf("psc", batch=2, hq=hq, hkv=hkv, docs_per_seq=3, doc_tokens=300, pool_docs=4, zipf_s=1.2,
                       chunk_tokens=[150, 70], seed=303)
    f = _freqs(w)
    ref = oracle.attention(w, freqs=f)
    assert_close(prefill(_scaled_device(w)), ref, "bf16", "prefill, scaled",
                 emulate=lambda r: emulate(w, r, freqs=f))


def test_decode_interleaved_pairing():
    w = W.decode_zipf("vi32", batch=4, hq=8, hkv=2, d=64, docs_per_seq=3, doc_tokens=200, pool_docs=5, zipf_s=1.0,
                      suffix_tokens=7, dtype="f32", theta=1e4, seed=304)
    ref = oracle.attention(w, interleaved=True)
    _, dv = _interleaved_device(w)
    assert_close(decode(dv), ref, "f32", "f32 decode, interleaved pairing")


def test_shared_decode_and_prefill_interleaved_pairing():
    w = W.decode_zipf("vib", batch=6, hq=16, hkv=4, d=128, docs_per_seq=3, doc_tokens=180, pool_docs=3, zipf_s=1.0,
                      suffix_tokens=12, seed=305)
    ref = oracle.attention(w, interleaved=True)
    wp, dv = _interleaved_device(w)
    assert_close(decode_shared(dv, shared_plan(dv)), ref, "bf16", "shared decode, interleaved",
                 emulate=lambda r: emulate(wp, r))
    wpf = W.prefill_zipf("pint", batch=2, hq=8, hkv=2, docs_per_seq=2, doc_tokens=200, pool_docs=3, zipf_s=1.0,
                         chunk_tokens=[130, 40], seed=306)
    ref = oracle.attention(wpf, interleaved=True)
    wpp, dvp = _interleaved_device(wpf)
    assert_close(prefill(dvp), ref, "bf16", "prefill, interleaved", emulate=lambda r: emulate(wpp, r))


# ---------------------------------------------------------------- partial rotary
# Only the first r dims rotate: q and stored K permuted by the library's layout, the
# table built from its rates (0 for the unrotated pairs); the oracle rotates the first
# r dims of the unpermuted inputs directly.

def _partial_device(w, r, interleaved=False):
    L = la()
    perm, freqs = L.rotary_layout(w.head_dim, r, w.rope_theta, interleaved)
    wp = dataclasses.replace(w, q=w.q[..., perm].contiguous(), k_pool=w.k_pool[..., perm].contiguous())
    dv = to_device(wp)
    dv.rope = L.rope_table_init(dv.p, freqs=freqs)
    return wp, dv, freqs


def test_decode_f32_partial_rotary():
    w = W.decode_zipf("vp32", batch=4, hq=8, hkv=2, d=64, docs_per_seq=3, doc_tokens=150, pool_docs=5, zipf_s=1.0,
                      suffix_tokens=11, dtype="f32", theta=1e4, seed=307)
    ref = oracle.attention(w, rot_dims=16)
    _, dv, _ = _partial_device(w, 16)
    assert_close(decode(dv), ref, "f32", "f32 decode, partial rotary")


@pytest.mark.parametrize("hq,hkv,interleaved", [(16, 4, False), (32, 1, False), (32, 1, True)])
def test_shared_and_per_sequence_decode_partial_rotary(hq, hkv, interleaved):
    # 4 query heads per KV head: mma.sync shared-run kernel; 32: the tensor-core one
    w = W.decode_zipf(f"vpb{hq}", batch=8, hq=hq, hkv=hkv, d=128, docs_per_seq=3, doc_tokens=230, pool_docs=3,
                      zipf_s=1.0, suffix_tokens=17, seed=308 + hq)
    ref = oracle.attention(w, rot_dims=32, interleaved=interleaved)
    wp, dv, freqs = _partial_device(w, 32, interleaved)
    emu = lambda r: emulate(wp, r, freqs=freqs)
    assert_close(decode_shared(dv, shared_plan(dv)), ref, "bf16", "shared decode, partial rotary", emulate=emu)
    assert_close(decode(dv), ref, "bf16", "per-sequence decode, partial rotary", emulate=emu)


@pytest.mark.parametrize("hq,hkv", [(8, 2), (6, 2)])  # stream-K and one-tile prefill kernels
def test_prefill_partial_rotary(hq, hkv):
    w = W.prefill_zipf("ppart", batch=2, hq=hq, hkv=hkv, docs_per_seq=3, doc_tokens=260, pool_docs=4, zipf_s=1.2,
                       chunk_tokens=[140, 60], seed=310)
    ref = oracle.attention(w, rot_dims=64)
    wp, dv, freqs = _partial_device(w, 64)
    assert_close(prefill(dv), ref, "bf16", "prefill, partial rotary", emulate=lambda r: emulate(wp, r, freqs=freqs))


# ---------------------------------------------------------------- ALiBi
# No rotation (a zero-rate table) and the bias -slope_h (m - n), formed in the
# kernels from key-position words (each word gives its block's first key).
# The steepest slopes put most of a row's weight on two or three keys, where the
# bf16 rounding of those weights alone (relative to each split's running maximum
# in the kernels, to the row maximum in the emulation) can exceed 2e-3; the
# emulation check then allows that rounding's first-order bound. A wrong key
# position moves such a row by about a tenth of |v|, far outside it.

def _alibi_device(w, pack_on_device=True):
    L = la()
    dv = to_device(w, key_positions=True, pack_on_device=pack_on_device)
    dv.rope = L.rope_table_init(dv.p, freqs=np.zeros(w.head_dim // 2))
    return dv


@pytest.mark.parametrize("hq,hkv,chunk", [(8, 8, 0), (8, 2, 3), (16, 2, 0), (32, 1, 5)])
def test_shared_decode_alibi(hq, hkv, chunk):
    # 1 and 4 query heads per KV head: the mma.sync kernel; 8 and 32: the tcgen05 one.
    # Chunks of 3 or 5 blocks start items inside documents.
    L = la()
    w = W.decode_zipf(f"valibi{hq}", batch=8, hq=hq, hkv=hkv, d=128, docs_per_seq=3, doc_tokens=170, pool_docs=3,
                      zipf_s=1.0, suffix_tokens=13, seed=320 + hq)
    slopes = L.alibi_slopes(hq)
    ref = oracle.attention(w, freqs=np.zeros(64), alibi=slopes.astype(np.float64))
    dv = _alibi_device(w)
    plan = shared_plan(dv, chunk)
    out = L.decode_shared(dv.p, dv.q, dv.k_pool, dv.v_pool, dv.words, dv.q_pos, dv.rope, plan,
                          alibi_slopes=torch.from_numpy(slopes).cuda())
    assert_close(out, ref, "bf16", f"shared decode, ALiBi, {hq}/{hkv}",
                 emulate=lambda r: emulate(w, r, freqs=np.zeros(64), alibi=slopes, weight_bound=True),
                 fallback_frac=FEW_KEY_FALLBACK_FRAC)
    # the bias matters at these positions
    assert np.abs(ref - oracle.attention(w, freqs=np.zeros(64))).max() > 1e-2


@pytest.mark.parametrize("hq,hkv,d,splits,host_pack", [(8, 8, 128, 0, False), (8, 2, 128, 3, True),
                                                       (32, 1, 128, 0, False), (4, 2, 64, 1, False)])
def test_per_sequence_decode_alibi(hq, hkv, d, splits, host_pack):
    # the split-K per-sequence kernel: 1, 4 and 32 query heads per KV head, d 64 and 128,
    # one split, three and the automatic count; words from the device and the host packer
    L = la()
    w = W.decode_zipf(f"vpsalibi{hq}", batch=6, hq=hq, hkv=hkv, d=d, docs_per_seq=4, doc_tokens=150, pool_docs=5,
                      zipf_s=1.0, suffix_tokens=21, seed=340 + hq + d)
    slopes = L.alibi_slopes(hq)
    ref = oracle.attention(w, freqs=np.zeros(d // 2), alibi=slopes.astype(np.float64))
    dv = _alibi_device(w, pack_on_device=not host_pack)
    dv.p.num_splits = splits
    out = L.decode(dv.p, dv.q, dv.k_pool, dv.v_pool, dv.words, dv.seq_lens, dv.q_pos, dv.rope,
                   alibi_slopes=torch.from_numpy(slopes).cuda())
    assert_close(out, ref, "bf16", f"per-sequence decode, ALiBi, {hq}/{hkv} d{d}",
                 emulate=lambda r: emulate(w, r, freqs=np.zeros(d // 2), alibi=slopes, weight_bound=True),
                 fallback_frac=FEW_KEY_FALLBACK_FRAC)
    assert np.abs(ref - oracle.attention(w, freqs=np.zeros(d // 2))).max() > 1e-2


@pytest.mark.parametrize("hq,hkv", [(8, 2), (32, 1), (8, 8), (6, 2)])
def test_prefill_alibi(hq, hkv):
    # even GQA ratios (4, 32 per KV head): the stream-K kernel; odd (MHA, 3): the
    # TMEM-Q kernel. Chunks of 140 and 33 rows over two 150-token documents: the
    # bias reaches the cached keys and the chunk's own causal keys.
    L = la()
    w = W.prefill_zipf(f"palibi{hq}", batch=2, hq=hq, hkv=hkv, docs_per_seq=2, doc_tokens=150, pool_docs=3,
                       zipf_s=1.0, chunk_tokens=[140, 33], seed=360 + hq + hkv)
    slopes = L.alibi_slopes(hq)
    ref = oracle.attention(w, freqs=np.zeros(64), alibi=slopes.astype(np.float64))
    dv = _alibi_device(w)
    out = L.prefill(dv.p, dv.q, dv.cu_seqlens_q, dv.q_start, dv.max_q_len, dv.k_pool, dv.v_pool, dv.words,
                    dv.seq_lens, dv.rope, alibi_slopes=torch.from_numpy(slopes).cuda())
    assert_close(out, ref, "bf16", f"prefill, ALiBi, {hq}/{hkv}",
                 emulate=lambda r: emulate(w, r, freqs=np.zeros(64), alibi=slopes, weight_bound=True),
                 fallback_frac=FEW_KEY_FALLBACK_FRAC)
    assert np.abs(ref - oracle.attention(w, freqs=np.zeros(64))).max() > 1e-2
    # the rotating call refuses key-position words
    with pytest.raises(L.LazyAttnError):
        L.prefill(dv.p, dv.q, dv.cu_seqlens_q, dv.q_start, dv.max_q_len, dv.k_pool, dv.v_pool, dv.words,
                  dv.seq_lens, dv.rope)
