"""GPU parity of the FP8-KV per-sequence decode (pools of OCP E4M3 codes with
per-tensor scales) against the oracle on the same codes and scales."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_close, la, to_device
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
