"""The allocation-free decode entry point, through the C ABI.

Some callers cannot allocate a device workspace (an engine whose KV-cache pool
already holds nearly all of HBM, a plugin limited to its host framework's
buffers, a step that must not call cudaMalloc). lazy_attn_decode_noalloc keeps
the split-K partials in the library's static device array instead; it must give
the same outputs as lazy_attn_decode with a caller-provided workspace. This file
is collected last so that a failure here never hides the other tests.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_close, decode, la, to_device
from paged_kv_cache_57_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _workload(seed):
    # 64 sequences x 32/8 heads x ~1.7k tokens: the split plan needs a few MiB of partials
    return W.decode_zipf("noalloc", batch=64, hq=32, hkv=8, d=128, docs_per_seq=6, doc_tokens=272, pool_docs=40,
                         zipf_s=1.0, suffix_tokens=33, seed=seed)


def test_decode_noalloc_matches_decode_on_two_calls():
    L = la()
    L.device_status(clear=True)
    for seed in (91, 92):  # two calls in a row, different inputs: the shared array is reused
        dv = to_device(_workload(seed))
        need = L.decode_workspace_bytes(dv.p)
        assert 0 < need <= L.NOALLOC_SCRATCH_BYTES  # the scratch array is really used
        ref = decode(dv)  # existing entry point, caller-provided workspace
        out = torch.full_like(dv.q, float("nan"))
        L.decode_noalloc(dv.p, dv.q, dv.k_pool, dv.v_pool, dv.words, dv.seq_lens, dv.q_pos, dv.rope, out)
        torch.cuda.synchronize()
        assert torch.isfinite(out.float()).all()
        # the same kernels on the same inputs and split plan: only where the partials
        # live differs, so the outputs must agree bit for bit (a partial overwrite of
        # the shared array would show here), and both must match the oracle
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
        assert_close(out, oracle.attention(dv.w), "bf16", f"decode_noalloc, call {seed - 90}")
    assert L.device_status(clear=True) == 0


def test_decode_noalloc_rejects_plans_larger_than_the_scratch():
    L = la()
    dv = to_device(_workload(93))
    dv.p.num_splits = 64  # 64 x 32 x 64 x 130 x 4 bytes of partials > 8 MiB
    assert L.decode_workspace_bytes(dv.p) > L.NOALLOC_SCRATCH_BYTES
    out = torch.zeros_like(dv.q)
    with pytest.raises(L.LazyAttnError) as e:
        L.decode_noalloc(dv.p, dv.q, dv.k_pool, dv.v_pool, dv.words, dv.seq_lens, dv.q_pos, dv.rope, out)
    assert e.value.status == L.LAZY_ERR_WORKSPACE
    assert (out == 0).all()  # nothing was launched
