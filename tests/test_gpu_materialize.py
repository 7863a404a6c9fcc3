"""GPU checks of the eager materialisation baseline (lazy_attn_materialize): per-
sequence copies with K rotated to absolute positions and V copied, read by the
control path of the decode kernel. The copies are compared with an fp64 rotation
(complex-form RoPE from tests/brute.py), and the decode on them with the oracle."""
import numpy as np
import pytest
import torch

import oracle
from brute import rope
from gpu_util import assert_close, decode, la, to_device
from paged_kv_cache_57_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _clean_status():
    la().device_status(clear=True)
    yield
    assert la().device_status(clear=True) == 0, "device status word set"


def _workloads():
    yield W.decode_zipf("mz", batch=6, hq=16, hkv=4, d=128, docs_per_seq=4, doc_tokens=70, pool_docs=3,
                        zipf_s=1.0, suffix_tokens=9, seed=171)
    yield W.decode_zipf("mz64", batch=3, hq=8, hkv=2, d=64, docs_per_seq=3, doc_tokens=40, pool_docs=2,
                        zipf_s=1.0, suffix_tokens=5, seed=172)
    d, _ = W.mixed_mqa(n_decode=5, n_prefill=1, chunk=16, hq=8, hkv=1, d=128, pool_docs=30, ctx_lo=100,
                       ctx_hi=3000, doc_lo=5, doc_hi=300, seed=173)
    yield d


@pytest.mark.parametrize("w", list(_workloads()), ids=lambda w: w.name)
def test_materialized_copies(w):
    L = la()
    dv = to_device(w)
    k_out, v_out, words_out = L.materialize(dv.p, dv.k_pool, dv.v_pool, dv.words, dv.seq_lens, dv.rope)
    k_out, v_out, wo = k_out.cpu(), v_out.cpu(), words_out.cpu().numpy().view(np.uint32)
    words = dv.words.cpu().numpy().view(np.uint32)
    mb, id_mask = dv.p.max_blocks_per_seq, (1 << 18) - 1
    ulp_errs = []
    for s in range(w.num_seqs):
        b, p = 0, int(w.seq_pos0[s])
        for doc, Ln in w.seq_segments(s):
            base = int(w.doc_block_indptr[doc])
            for q in range((Ln + 15) // 16):
                phys, dst = int(w.doc_blocks[base + q]), s * mb + b
                nv = min(16, Ln - 16 * q)
                assert wo[s, b] & id_mask == dst and wo[s, b] >> 18 == words[s, b] >> 18
                assert torch.equal(v_out[dst, :, :nv].view(torch.int16), w.v_pool[phys, :, :nv].view(torch.int16))
                kin = w.k_pool[phys, :, :nv].double()
                ref = torch.from_numpy(rope(kin.numpy(), p, w.rope_theta))
                got = k_out[dst, :, :nv].double()
                # one bf16 rounding of an fp32 rotation: one ulp of the exact value, plus the
                # rotation's absolute error (angle < 5e-7 rad, fp32 products) on the input row
                ulp = ref.abs().clamp_min(1e-30).log2().floor().exp2() * 2.0 ** -7
                slack = 2e-6 * kin.abs().amax(dim=-1, keepdim=True)
                ulp_errs.append((((got - ref).abs() - slack).clamp_min(0) / ulp).max().item())
                b += 1
            p += Ln
        assert (wo[s, b:] == 0).all()
    assert max(ulp_errs) <= 1.0, max(ulp_errs)


@pytest.mark.parametrize("w", list(_workloads()), ids=lambda w: w.name)
def test_decode_on_materialized_copies_matches_oracle(w):
    L = la()
    dv = to_device(w)
    k_out, v_out, words_out = L.materialize(dv.p, dv.k_pool, dv.v_pool, dv.words, dv.seq_lens, dv.rope)
    dv.p.lazy = 0
    dv.p.num_pool_blocks = k_out.shape[0]
    dv.k_pool, dv.v_pool, dv.words = k_out, v_out, words_out
    assert_close(decode(dv), oracle.attention(w), "bf16", f"{w.name} eager")
