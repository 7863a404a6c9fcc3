"""GPU parity of the FP8-KV decodes, per-sequence and shared-run (pools of OCP E4M3
codes with per-tensor scales), against the oracle on the same codes and scales."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_close, la, shared_plan, to_device
from paged_kv_cache_57_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _clean_status():
    la().device_status(clear=True)
    yield
    assert la().device_status(clear=True) == 0, "device status word set"


# 1, 4, 32 and 64 query heads per KV head (one-, two- and four-warp tiles), the
# automatic split count and fixed ones; documents of 150 tokens and a 21-token
# suffix leave partial blocks whose hole slots hold NaN codes.
@pytest.mark.parametrize("hq,hkv,splits", [(8, 8, 0), (32, 8, 3), (32, 1, 0), (64, 1, 2)])
def test_fp8_decode_matches_oracle(hq, hkv, splits):
    L = la()
    w = W.decode_zipf(f"fp8{hq}", batch=6, hq=hq, hkv=hkv, d=128, docs_per_seq=4, doc_tokens=150, pool_docs=5,
                      zipf_s=1.0, suffix_tokens=21, seed=520 + hq + splits)
    k8, v8, ks, vs = W.fp8_pools(w)
    ref = oracle.attention(w, k_pool=k8, v_pool=v8, k_scale=ks, v_scale=vs)
    dv = to_device(w)
    p = dv.p
    p.kv_dtype, p.k_scale, p.v_scale, p.num_splits = L.LAZY_FP8_E4M3, ks, vs, splits
    out = L.decode(p, dv.q, k8.cuda(), v8.cuda(), dv.words, dv.seq_lens, dv.q_pos, dv.rope)
    assert_close(out, ref, "bf16", f"fp8 decode {hq}/{hkv} splits {splits}")
    # the codes, not the bf16 pool, were read: the two references differ here
    assert np.abs(ref - oracle.attention(w)).max() > 2e-3


def test_fp8_decode_noalloc_and_empty_sequences():
    L = la()
    w = W.decode_zipf("fp8e", batch=4, hq=16, hkv=4, d=128, docs_per_seq=2, doc_tokens=70, pool_docs=3,
                      zipf_s=1.0, suffix_tokens=5, seed=530)
    k8, v8, ks, vs = W.fp8_pools(w)
    ref = oracle.attention(w, k_pool=k8, v_pool=v8, k_scale=ks, v_scale=vs)
    dv = to_device(w)
    p = dv.p
    p.kv_dtype, p.k_scale, p.v_scale = L.LAZY_FP8_E4M3, ks, vs
    out = L.decode_noalloc(p, dv.q, k8.cuda(), v8.cuda(), dv.words, dv.seq_lens, dv.q_pos, dv.rope,
                           torch.empty_like(dv.q))
    assert_close(out, ref, "bf16", "fp8 decode, no-workspace entry point")
    lens = dv.seq_lens.clone()
    lens[1] = 0  # an empty sequence gives zeros
    out = L.decode(p, dv.q, k8.cuda(), v8.cuda(), dv.words, lens, dv.q_pos, dv.rope)
    assert torch.count_nonzero(out[1]) == 0
    keep = [0, 2, 3]
    assert_close(out[keep], ref[keep], "bf16", "fp8 decode beside an empty sequence")


def test_fp8_decode_control_path_with_identity_rotation():
    # lazy = 0 (the pool holds absolute-position keys; q rotated once by R_m) with a
    # zero-rate table, where every rotation is the identity: the control kernel's
    # permuted q fragments and its single-pass loop against the oracle on the codes.
    L = la()
    w = W.decode_zipf("fp8ctl", batch=5, hq=32, hkv=8, d=128, docs_per_seq=3, doc_tokens=90, pool_docs=4,
                      zipf_s=1.0, suffix_tokens=11, share=False, seed=540)
    k8, v8, ks, vs = W.fp8_pools(w)
    zero = np.zeros(64)
    ref = oracle.attention(w, freqs=zero, k_pool=k8, v_pool=v8, k_scale=ks, v_scale=vs)
    dv = to_device(w, lazy=False)
    p = dv.p
    p.kv_dtype, p.k_scale, p.v_scale = L.LAZY_FP8_E4M3, ks, vs
    rope = L.rope_table_init(p, freqs=zero)
    out = L.decode(p, dv.q, k8.cuda(), v8.cuda(), dv.words, dv.seq_lens, dv.q_pos, rope)
    assert_close(out, ref, "bf16", "fp8 decode, lazy=0 control")


# ---------------------------------------------------------------- shared-run decode on e4m3 pools

def _fp8_device(w, lazy=True):
    L = la()
    k8, v8, ks, vs = W.fp8_pools(w)
    dv = to_device(w, lazy=lazy)
    dv.p.kv_dtype, dv.p.k_scale, dv.p.v_scale = L.LAZY_FP8_E4M3, ks, vs
    return dv, k8, v8, ks, vs


# 1, 4, 8, 32 and 64 query heads per KV head (items of up to 64 rows on the mma.sync
# kernel, which runs e4m3 pools at every ratio), whole-document items and chunks of 3
# or 5 blocks that start items inside documents; 150-token documents and a 21-token
# suffix leave partial blocks whose hole slots hold NaN codes.
@pytest.mark.parametrize("hq,hkv,chunk", [(8, 8, 0), (32, 8, 3), (16, 2, 0), (32, 1, 0), (64, 1, 5)])
def test_fp8_shared_decode_matches_oracle(hq, hkv, chunk):
    L = la()
    w = W.decode_zipf(f"fp8s{hq}", batch=10, hq=hq, hkv=hkv, d=128, docs_per_seq=4, doc_tokens=150, pool_docs=4,
                      zipf_s=1.0, suffix_tokens=21, seed=560 + hq + chunk)
    dv, k8, v8, ks, vs = _fp8_device(w)
    ref = oracle.attention(w, k_pool=k8, v_pool=v8, k_scale=ks, v_scale=vs)
    plan = shared_plan(dv, chunk)  # planned for e4m3 pools: items of at most 64 rows
    assert (plan.items_host[:, 4] * (hq // hkv) <= 64).all()
    out = L.decode_shared(dv.p, dv.q, k8.cuda(), v8.cuda(), dv.words, dv.q_pos, dv.rope, plan)
    assert_close(out, ref, "bf16", f"fp8 shared-run decode {hq}/{hkv} chunk {chunk}")
    assert np.abs(ref - oracle.attention(w)).max() > 2e-3


def test_fp8_shared_decode_holes_and_partial_blocks():
    L = la()
    d, _ = W.mixed_mqa(n_decode=8, n_prefill=1, chunk=16, hq=32, hkv=1, d=128, pool_docs=40, ctx_lo=100,
                       ctx_hi=3000, doc_lo=5, doc_hi=400, seed=565)
    dv, k8, v8, ks, vs = _fp8_device(d)
    ref = oracle.attention(d, k_pool=k8, v_pool=v8, k_scale=ks, v_scale=vs)
    for chunk in (0, 4):
        out = L.decode_shared(dv.p, dv.q, k8.cuda(), v8.cuda(), dv.words, dv.q_pos, dv.rope, shared_plan(dv, chunk))
        assert_close(out, ref, "bf16", f"fp8 shared-run decode, holes, chunk {chunk}")


def test_fp8_shared_decode_control_path_with_identity_rotation():
    L = la()
    w = W.decode_zipf("fp8sctl", batch=5, hq=32, hkv=8, d=128, docs_per_seq=3, doc_tokens=90, pool_docs=4,
                      zipf_s=1.0, suffix_tokens=11, share=False, seed=570)
    dv, k8, v8, ks, vs = _fp8_device(w, lazy=False)
    zero = np.zeros(64)
    ref = oracle.attention(w, freqs=zero, k_pool=k8, v_pool=v8, k_scale=ks, v_scale=vs)
    rope = L.rope_table_init(dv.p, freqs=zero)
    out = L.decode_shared(dv.p, dv.q, k8.cuda(), v8.cuda(), dv.words, dv.q_pos, rope, shared_plan(dv))
    assert_close(out, ref, "bf16", "fp8 shared-run decode, lazy=0 control")


def test_fp8_shared_decode_llama8b_full():
    L = la()
    w = W.FULL["llama8b_decode"]()
    dv, k8, v8, ks, vs = _fp8_device(w)
    ref = oracle.attention(w, k_pool=k8, v_pool=v8, k_scale=ks, v_scale=vs)
    out = L.decode_shared(dv.p, dv.q, k8.cuda(), v8.cuda(), dv.words, dv.q_pos, dv.rope, shared_plan(dv))
    assert_close(out, ref, "bf16", "fp8 shared-run decode, llama8b_decode")
