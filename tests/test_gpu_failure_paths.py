"""Device-side failure handling, through the C ABI: every status bit of the device
status word is raised by the condition it names, the kernel returns instead of
trapping, and the device stays usable for the next call.

The bounded-wait test withholds one block's copies in the test-only gather
(lazy_attn_debug_gather_withheld) so that a pipeline wait runs out after a short
limit; nothing here faults or hangs the GPU."""
import time

import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_close, decode, decode_shared, la, prefill, shared_plan, to_device
from paged_kv_cache_57_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _clean_status():
    la().device_status(clear=True)
    yield
    la().device_status(clear=True)


def _small_decode(seed=401, batch=3):
    return W.decode_zipf("fail", batch=batch, hq=8, hkv=2, d=128, docs_per_seq=3, doc_tokens=70, pool_docs=4,
                         zipf_s=1.0, suffix_tokens=9, seed=seed)


def test_withheld_copy_times_out_and_the_device_recovers():
    L = la()
    w = _small_decode()
    dv = to_device(w)
    ko, vo, po = L.debug_gather(dv.p, dv.k_pool, dv.v_pool, dv.words, dv.seq_lens)
    torch.cuda.synchronize()
    assert L.device_status(clear=True) == 0
    limit_us = 2000
    t0 = time.perf_counter()
    kb, vb, pb = L.debug_gather(dv.p, dv.k_pool, dv.v_pool, dv.words, dv.seq_lens, withhold_block=1,
                                wait_limit_us=limit_us)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert L.device_status(clear=True) & L.LAZY_DEV_TIMEOUT
    # the waits gave up after their short limit (three waits in sequence at most), far
    # below the 2 s default
    assert elapsed < 0.5, elapsed
    # every other (sequence, KV head) pair was gathered as usual
    for s in range(w.num_seqs):
        for h in range(w.num_kv_heads):
            if s == 0 and h == 0:
                continue
            assert torch.equal(kb[s, h].view(torch.int16), ko[s, h].view(torch.int16))
            assert torch.equal(vb[s, h].view(torch.int16), vo[s, h].view(torch.int16))
    # block 0 of the stalled pair was copied before the withheld one
    assert torch.equal(kb[0, 0, :16].view(torch.int16), ko[0, 0, :16].view(torch.int16))
    # the context is intact: a normal decode right after matches the oracle
    assert_close(decode(dv), oracle.attention(w), "bf16", "decode after a timed-out launch")
    assert L.device_status(clear=True) == 0


def test_withheld_gather_rejects_bad_arguments():
    L = la()
    dv = to_device(_small_decode())
    with pytest.raises(L.LazyAttnError) as e:
        L.debug_gather(dv.p, dv.k_pool, dv.v_pool, dv.words, dv.seq_lens, withhold_block=0, wait_limit_us=0)
    assert e.value.status == L.LAZY_ERR_INVALID_ARG
    with pytest.raises(L.LazyAttnError) as e:
        L.debug_gather(dv.p, dv.k_pool, dv.v_pool, dv.words, dv.seq_lens, withhold_block=0,
                       wait_limit_us=3_000_000)
    assert e.value.status == L.LAZY_ERR_INVALID_ARG


@pytest.mark.parametrize("path", ["per-sequence", "shared-run"])
def test_rotation_offset_out_of_range_sets_status(path):
    # q_pos past 2^24: the offset m - p leaves the rotation's range; it is clamped and
    # flagged, the output stays finite, and the other sequences are unaffected.
    L = la()
    w = _small_decode(seed=402)
    dv = to_device(w)
    ref = decode(dv).float().cpu()
    q_pos = dv.q_pos.clone()
    q_pos[0] += 1 << 24
    dv.q_pos = q_pos
    out = decode(dv) if path == "per-sequence" else decode_shared(dv, shared_plan(dv))
    torch.cuda.synchronize()
    assert L.device_status(clear=True) & L.LAZY_DEV_POS_RANGE
    out = out.float().cpu()
    assert torch.isfinite(out).all()
    assert_close(out[1:], oracle.attention(w)[1:], "bf16", f"{path}: other sequences")
    assert not torch.equal(out[0], ref[0])


@pytest.mark.parametrize("bad", [-5, "past"])
def test_bad_sequence_length_sets_status(bad):
    L = la()
    w = _small_decode(seed=403)
    dv = to_device(w)
    sl = dv.seq_lens.clone()
    sl[1] = -5 if bad == -5 else 16 * dv.p.max_blocks_per_seq + 3
    dv.seq_lens = sl
    out = decode(dv)
    torch.cuda.synchronize()
    assert L.device_status(clear=True) & L.LAZY_DEV_BAD_LEN
    ref = oracle.attention(w)
    keep = [0, 2]
    assert_close(out[torch.tensor(keep, device=out.device)], ref[keep], "bf16", "decode beside a bad length")
    if bad == -5:  # clamped to an empty sequence
        assert (out[1] == 0).all()


def test_prefill_bad_sequence_length_sets_status():
    L = la()
    w = W.prefill_zipf("pfbadlen", batch=2, hq=8, hkv=2, docs_per_seq=2, doc_tokens=100, pool_docs=3, zipf_s=1.0,
                       chunk_tokens=[40, 21], seed=404)
    dv = to_device(w)
    sl = dv.seq_lens.clone()
    sl[0] = 16 * dv.p.max_blocks_per_seq + 7
    dv.seq_lens = sl
    prefill(dv)
    torch.cuda.synchronize()
    assert L.device_status(clear=True) & L.LAZY_DEV_BAD_LEN


def _bad_word(words: torch.Tensor, s: int, b: int, bad_id: int) -> torch.Tensor:
    wh = words.cpu().numpy().view(np.uint32).copy()
    wh[s, b] = (wh[s, b] & ~np.uint32((1 << 18) - 1)) | np.uint32(bad_id)
    return torch.from_numpy(wh.view(np.int32)).cuda()


def test_prefill_bad_block_id_sets_status_and_does_not_fault():
    L = la()
    w = W.prefill_zipf("pfbadid", batch=2, hq=8, hkv=2, docs_per_seq=2, doc_tokens=100, pool_docs=3, zipf_s=1.0,
                       chunk_tokens=[40, 21], seed=405)
    dv = to_device(w)
    dv.words = _bad_word(dv.words, 0, 2, (1 << 18) - 1)  # an id past the pool (and past the tensor map)
    out = prefill(dv)
    torch.cuda.synchronize()
    assert L.device_status(clear=True) & L.LAZY_DEV_BAD_BLOCK_ID
    assert torch.isfinite(out.float()).all()
    # sequence 1 is untouched
    cu = np.asarray(w.cu_seqlens_q)
    rows = list(range(int(cu[1]), int(cu[2])))
    assert_close(out[torch.tensor(rows, device=out.device)], oracle.attention(w, rows=rows), "bf16",
                 "prefill beside a bad block id")


@pytest.mark.parametrize("hq,hkv", [(8, 2), (32, 1)])
def test_shared_decode_bad_block_id_sets_status_and_does_not_fault(hq, hkv):
    # The block word and the item record agree on an id past the pool: the block is
    # skipped (never loaded) and flagged, on both shared-run kernels.
    L = la()
    w = W.decode_zipf("sbadpool", batch=4, hq=hq, hkv=hkv, d=128, docs_per_seq=2, doc_tokens=40, pool_docs=3,
                      zipf_s=1.0, seed=406)
    dv = to_device(w)
    plan = shared_plan(dv)
    items = plan.items_host.copy()
    src, b0 = int(items[0, 0]), int(items[0, 1])
    assert int(items[0, 2]) >= 2  # the item has a second block
    bad_id = (1 << 18) - 1
    items[0, 8 + 4 * L.PLAN_MAX_MEMBERS + 1] = bad_id
    dv.words = _bad_word(dv.words, src, b0 + 1, bad_id)
    out = decode_shared(dv, L.SharedPlan(items, plan.slot_indptr_host))
    torch.cuda.synchronize()
    assert L.device_status(clear=True) & L.LAZY_DEV_BAD_BLOCK_ID
    assert torch.isfinite(out.float()).all()
