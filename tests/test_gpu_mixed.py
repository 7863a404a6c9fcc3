"""GPU parity of the one-launch mixed batch (lazy_attn_mixed): the shared-run decode
of one batch and the prefill of other sequences' chunks in a single cooperative
launch of the prefill pipeline, over one pool. Both halves are checked against the
oracle; the prefill half must also equal lazy_attn_prefill bit for bit (the same
units and split pieces, only preceded by the decode units)."""
import numpy as np
import pytest
import torch

import oracle
from bf16_model import emulate
from gpu_util import assert_close, decode_shared, la, prefill, shared_plan, to_device
from paged_kv_cache_57_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _clean_status():
    la().device_status(clear=True)
    yield
    assert la().device_status(clear=True) == 0, "device status word set"


def _mixed(wd, wp, rows_dec=None, rows_pf=None):
    L = la()
    dd = to_device(wd)
    dp = to_device(wp)
    plan = shared_plan(dd)
    # one pool for both halves (the generator places both batches' documents in it)
    assert torch.equal(dd.k_pool.view(torch.int16), dp.k_pool.view(torch.int16))
    out_dec, out_pf = L.mixed(dd.p, dd.q, dd.words, dd.q_pos, plan, dp.p, dp.q, dp.cu_seqlens_q, dp.q_start,
                              dp.max_q_len, dp.words, dp.seq_lens, dd.k_pool, dd.v_pool, dd.rope)
    torch.cuda.synchronize()
    return dd, dp, plan, out_dec, out_pf


@pytest.mark.parametrize("hq,hkv", [(32, 1), (32, 2)])
def test_mixed_launch_matches_oracle_and_separate_calls(hq, hkv):
    wd, wp = W.mixed_mqa(n_decode=10, n_prefill=3, chunk=150, hq=hq, hkv=hkv, d=128, pool_docs=60, ctx_lo=100,
                         ctx_hi=4000, doc_lo=5, doc_hi=400, seed=600 + hq)
    dd, dp, plan, out_dec, out_pf = _mixed(wd, wp)
    assert_close(out_dec, oracle.attention(wd), "bf16", f"mixed launch, decode half {hq}/{hkv}",
                 emulate=lambda r: emulate(wd, r))
    assert_close(out_pf, oracle.attention(wp), "bf16", f"mixed launch, prefill half {hq}/{hkv}",
                 emulate=lambda r: emulate(wp, r))
    sep_pf = prefill(dp)
    assert torch.equal(out_pf.view(torch.int16), sep_pf.view(torch.int16))
    sep_dec = decode_shared(dd, plan)
    assert_close(out_dec, sep_dec.float().cpu().double().numpy(), "bf16", "mixed decode half vs lazy_attn_decode_shared")


def test_mixed_launch_two_calls_in_a_row():
    # the per-sequence counters are zeroed by every call: a second call gives the same bits
    wd, wp = W.mixed_mqa(n_decode=6, n_prefill=2, chunk=64, hq=32, hkv=1, d=128, pool_docs=40, ctx_lo=100,
                         ctx_hi=2000, doc_lo=5, doc_hi=300, seed=610)
    L = la()
    dd, dp, plan, a_dec, a_pf = _mixed(wd, wp)
    b_dec, b_pf = L.mixed(dd.p, dd.q, dd.words, dd.q_pos, plan, dp.p, dp.q, dp.cu_seqlens_q, dp.q_start,
                          dp.max_q_len, dp.words, dp.seq_lens, dd.k_pool, dd.v_pool, dd.rope)
    assert torch.equal(a_dec.view(torch.int16), b_dec.view(torch.int16))
    assert torch.equal(a_pf.view(torch.int16), b_pf.view(torch.int16))


def test_mixed_launch_full_size_sampled():
    # the mixed continuous batch: 48 decode sequences (contexts up to 131072) and 4
    # prefill chunks of 512, one launch; sampled rows of both halves against the oracle
    wd, wp = W.mixed_mqa()
    dd, dp, plan, out_dec, out_pf = _mixed(wd, wp)
    rng = np.random.default_rng(7)
    rows_d = sorted(rng.choice(wd.num_seqs, 4, replace=False).tolist())
    assert_close(out_dec[torch.tensor(rows_d, device=out_dec.device)], oracle.attention(wd, rows=rows_d), "bf16",
                 "mixed launch full size, decode rows")
    cu = np.asarray(wp.cu_seqlens_q)
    rows_p = sorted(set(int(cu[s] + r) for s in range(wp.num_seqs) for r in (0, 1, 200, 511)))
    assert_close(out_pf[torch.tensor(rows_p, device=out_pf.device)], oracle.attention(wp, rows=rows_p), "bf16",
                 "mixed launch full size, prefill rows")
    assert torch.equal(out_pf.view(torch.int16), prefill(dp).view(torch.int16))


def test_mixed_launch_refuses_small_query_groups():
    # 8 query heads per KV head: a 16-row group would straddle two members
    L = la()
    wd, wp = W.mixed_mqa(n_decode=3, n_prefill=1, chunk=32, hq=16, hkv=2, d=128, pool_docs=20, ctx_lo=100,
                         ctx_hi=500, doc_lo=5, doc_hi=100, seed=620)
    dd, dp = to_device(wd), to_device(wp)
    with pytest.raises(L.LazyAttnError) as e:
        L.mixed(dd.p, dd.q, dd.words, dd.q_pos, shared_plan(dd), dp.p, dp.q, dp.cu_seqlens_q, dp.q_start,
                dp.max_q_len, dp.words, dp.seq_lens, dd.k_pool, dd.v_pool, dd.rope)
    assert e.value.status == L.LAZY_ERR_UNSUPPORTED
