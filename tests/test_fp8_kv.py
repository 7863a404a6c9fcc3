"""FP8 (OCP E4M3) KV cache: the oracle's code decoding and scale folding, pinned
on the CPU, and the ABI's argument rules for pools of e4m3 codes."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_57_gb300 import workloads as W


def test_e4m3_decode_matches_torch_for_every_code():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_decode(codes)
    lib = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(ours, lib, equal_nan=True)


def test_e4m3_decode_format_values():
    d = oracle.e4m3_decode(np.array([0x7E, 0x01, 0x07, 0x08, 0x38, 0x39, 0xB8, 0x00, 0x80, 0x7F, 0xFF],
                                    dtype=np.uint8))
    assert d[0] == 448.0                      # largest finite: 2^8 * 1.75
    assert d[1] == 2.0 ** -9                  # smallest subnormal
    assert d[2] == 7 * 2.0 ** -9              # largest subnormal
    assert d[3] == 2.0 ** -6                  # smallest normal
    assert d[4] == 1.0 and d[5] == 1.125 and d[6] == -1.0
    assert d[7] == 0.0 and d[8] == 0.0 and np.signbit(d[8])
    assert np.isnan(d[9]) and np.isnan(d[10])


def test_fp8_scales_fold_into_softmax_scale_and_output():
    # With power-of-two scales every dequantised value is exact in bf16, so the
    # oracle on the codes with scales must equal the oracle on explicit values.
    w = W.decode_zipf("fp8pin", batch=3, hq=8, hkv=2, d=64, docs_per_seq=3, doc_tokens=40, pool_docs=4,
                      zipf_s=1.0, suffix_tokens=7, seed=501)
    k8, v8, _, _ = W.fp8_pools(w)
    ks, vs = 2.0 ** -3, 4.0
    kv = torch.from_numpy(oracle.e4m3_decode(k8.view(torch.uint8).numpy()) * ks).to(torch.bfloat16)
    vv = torch.from_numpy(oracle.e4m3_decode(v8.view(torch.uint8).numpy()) * vs).to(torch.bfloat16)
    a = oracle.attention(w, k_pool=k8, v_pool=v8, k_scale=ks, v_scale=vs)
    b = oracle.attention(w, k_pool=kv, v_pool=vv)
    assert np.allclose(a, b, rtol=1e-12, atol=1e-14)
    assert np.abs(a - oracle.attention(w, k_pool=k8, v_pool=v8)).max() > 1e-2  # the scales matter


def test_fp8_pools_quantise_within_half_an_ulp():
    w = W.decode_zipf("fp8q", batch=2, hq=4, hkv=2, d=64, docs_per_seq=2, doc_tokens=20, pool_docs=3,
                      zipf_s=1.0, seed=502)
    k8, _, ks, _ = W.fp8_pools(w)
    x = w.k_pool.double().numpy() / ks
    q = oracle.e4m3_decode(k8.view(torch.uint8).numpy())
    fin = np.isfinite(x)  # hole slots hold non-finite filler, kept as NaN codes
    assert np.isnan(q[~fin]).all()
    x, q = x[fin], q[fin]
    assert np.abs(q).max() <= 448.0
    # relative error of round-to-nearest with 4 significant bits, or half the subnormal step
    assert (np.abs(q - x) <= np.maximum(np.abs(x) * 2.0 ** -4, 2.0 ** -10) + 1e-12).all()


def test_fp8_argument_rules_without_cuda():
    from paged_kv_cache_57_gb300 import lazy_attn as L
    w = W.tiny_fp32()
    fake = ctypes.c_void_p(4096)  # never dereferenced: the arguments are rejected first

    def params(**kw):
        base = dict(num_seqs=w.num_seqs, num_q_heads=w.num_q_heads, num_kv_heads=w.num_kv_heads, head_dim=128,
                    num_pool_blocks=w.num_pool_blocks, max_blocks_per_seq=w.max_blocks_per_seq, dtype="bf16",
                    rope_theta=w.rope_theta, kv_dtype="fp8_e4m3", k_scale=0.5, v_scale=0.25)
        base.update(kw)
        return L.make_params(**base)

    def decode(p):
        return L._lib.lazy_attn_decode(ctypes.byref(p), *([fake] * 8), fake, 1 << 20, None)

    un, bad = L.LAZY_ERR_UNSUPPORTED, L.LAZY_ERR_INVALID_ARG
    assert decode(params(dtype="f32")) == un
    assert decode(params(head_dim=64)) == un
    assert decode(params(k_scale=float("nan"))) == bad
    assert decode(params(v_scale=-1.0)) == bad
    p = params()
    p.kv_dtype = 7
    assert decode(p) == un
    # the shared-run decode takes e4m3 pools at d = 128 only, and not with ALiBi
    p = params(head_dim=64)
    assert L._lib.lazy_attn_decode_shared(ctypes.byref(p), *([fake] * 6), 1, fake, 1, fake, fake, fake, 1 << 20,
                                          None) == un
    p = params(key_positions=True)
    assert L._lib.lazy_attn_decode_shared_alibi(ctypes.byref(p), *([fake] * 6), 1, fake, 1, fake, fake, fake, fake,
                                                1 << 20, None) == un
    p = params()
    assert L._lib.lazy_attn_prefill(ctypes.byref(p), fake, fake, fake, 1, 1, *([fake] * 7), 1 << 20, None) == un
    assert L._lib.lazy_attn_materialize(ctypes.byref(p), *([fake] * 8), None) == un
    assert L._lib.lazy_attn_decode_alibi(ctypes.byref(params(key_positions=True)), *([fake] * 7), fake, fake, fake,
                                         1 << 20, None) == un


def test_fp8_plan_keeps_longest_first_and_bf16_plan_spreads_small_items():
    """The planner's item order for the same batch: with e4m3 params the items run
    longest first; with bf16 params (mma.sync kernel) the items of at most 8 blocks
    (the 64-token private tails here) are spread through the order instead of ending it."""
    from paged_kv_cache_57_gb300 import lazy_attn as L
    w = W.decode_zipf("planord", batch=16, hq=32, hkv=8, d=128, docs_per_seq=4, doc_tokens=512, pool_docs=24,
                      zipf_s=1.0, suffix_tokens=64, seed=77)

    def plan(**kw):
        p = L.make_params(num_seqs=w.num_seqs, num_q_heads=w.num_q_heads, num_kv_heads=w.num_kv_heads,
                          head_dim=w.head_dim, num_pool_blocks=w.num_pool_blocks,
                          max_blocks_per_seq=w.max_blocks_per_seq, dtype="bf16", rope_theta=w.rope_theta, **kw)
        items, _ = L.plan_shared_host(p, len(w.doc_len), w.seg_indptr, w.seg_doc, w.seg_len, w.doc_block_indptr,
                                      w.doc_blocks)
        return items[:, 2]

    nb8 = plan(kv_dtype="fp8_e4m3", k_scale=1.0, v_scale=1.0)
    assert (np.diff(nb8) <= 0).all()
    nb16 = plan()
    small = np.flatnonzero(nb16 <= 8)
    assert 0 < len(small) < len(nb16)
    assert sorted(nb16.tolist()) == sorted(nb8.tolist())  # the same items, another order
    assert small[0] < len(nb16) // 2 and (np.diff(nb16[nb16 > 8]) <= 0).all()
