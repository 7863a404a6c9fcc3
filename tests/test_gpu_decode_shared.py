"""GPU parity of the shared-run decode (lazy_attn_decode_shared) against the CPU
oracle, through the C ABI. The shared-run kernel reads each cited document chunk
once per KV head for every sequence citing it; its results must match the oracle
exactly as the per-sequence decode's do."""
import numpy as np
import pytest
import torch

import oracle
from bf16_model import emulate
from brute import rope
from gpu_util import FEW_KEY_FALLBACK_FRAC, assert_close, decode, decode_shared, la, shared_plan, to_device
from paged_kv_cache_57_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _clean_status():
    la().device_status(clear=True)
    yield
    assert la().device_status(clear=True) == 0, "device status word set"


def _check(w, rows=None, chunk=0, lazy=True, k_pool=None, fallback_frac=0.0):
    dv = to_device(w, lazy=lazy, k_pool=k_pool)
    out = decode_shared(dv, shared_plan(dv, chunk))
    ref = oracle.attention(w, rows=rows)
    got = out if rows is None else out[torch.as_tensor(rows, device=out.device)]
    sel = np.arange(ref.shape[0]) if rows is None else np.asarray(rows)
    emu = (lambda r: emulate(w, sel[r], lazy=lazy, k_pool=k_pool)) if w.dtype == "bf16" else None
    return assert_close(got, ref, w.dtype, w.name, emulate=emu, fallback_frac=fallback_frac)


@pytest.mark.parametrize("hq,hkv", [(4, 4), (8, 2), (16, 2), (32, 1), (64, 8), (64, 1), (24, 8)])
@pytest.mark.parametrize("d", [64, 128])
def test_shared_decode_gqa_shapes(hq, hkv, d):
    # 12 sequences citing 4 documents: groups of several members at different offsets
    w = W.decode_zipf(f"sgqa{hq}x{hkv}d{d}", batch=12, hq=hq, hkv=hkv, d=d, docs_per_seq=4, doc_tokens=80,
                      pool_docs=4, zipf_s=1.0, suffix_tokens=16, seed=150 + hq + d)
    _check(w)


@pytest.mark.parametrize("chunk", [1, 3, 32])
def test_shared_decode_chunk_sweep(chunk):
    w = W.decode_zipf("schunk", batch=6, hq=32, hkv=8, d=128, docs_per_seq=5, doc_tokens=300, pool_docs=3,
                      zipf_s=1.0, suffix_tokens=21, seed=161)
    _check(w, chunk=chunk)


# (query heads, KV heads): the mma.sync kernel (4 per KV head) and the tensor-core one (32)
EDGE_SHAPES = [(8, 2), (32, 1)]


@pytest.mark.parametrize("chunk", [1, 5, 40])
@pytest.mark.parametrize("hq", [8, 16, 32, 64])
def test_shared_decode_tensor_core_path(hq, chunk):
    # hq query heads on one KV head, d = 128: the tcgen05 kernel, items of up to 128 rows
    # (16 members at 8 heads). 700-token documents end in a partial block; at chunk 40 an
    # item runs past the 32 block ids its record names.
    w = W.decode_zipf(f"stc{hq}c{chunk}", batch=max(10, 128 // hq + 4), hq=hq, hkv=1, d=128, docs_per_seq=3,
                      doc_tokens=700, pool_docs=3, zipf_s=0.8, suffix_tokens=23, seed=190 + hq + chunk)
    dv = to_device(w)
    plan = shared_plan(dv, chunk)
    assert plan.items_host[:, 4].max() * hq == 128  # full tensor-core tiles occur
    _check(w, chunk=chunk)



@pytest.mark.parametrize("hq,hkv,cap", [(8, 2, 16), (16, 2, 16), (32, 1, 4)])
def test_shared_decode_many_members_per_document(hq, hkv, cap):
    # 40 sequences all citing one document (repeatedly): groups are split into items of at
    # most 16 members and at most 64 (mma.sync) or 128 (tcgen05) rows
    w = W.decode_zipf("smany", batch=40, hq=hq, hkv=hkv, d=128, docs_per_seq=3, doc_tokens=50, pool_docs=1,
                      zipf_s=1.0, suffix_tokens=5, seed=162)
    dv = to_device(w)
    plan = shared_plan(dv)
    assert plan.items_host[:, 4].max() == cap and plan.num_items < int(plan.items_host[:, 4].sum())
    _check(w)


def test_shared_decode_holes_and_partial_blocks():
    d, _ = W.mixed_mqa(n_decode=10, n_prefill=1, chunk=16, hq=32, hkv=1, d=128, pool_docs=40, ctx_lo=100,
                       ctx_hi=6000, doc_lo=5, doc_hi=500, seed=163)
    _check(d)
    _check(d, chunk=4)


@pytest.mark.parametrize("hq,hkv", EDGE_SHAPES)
def test_shared_decode_few_keys(hq, hkv):
    w = W.decode_zipf("sfew", batch=6, hq=hq, hkv=hkv, d=128, docs_per_seq=1, doc_tokens=3, pool_docs=2,
                      zipf_s=1.0, seed=164)
    w.seg_len[:] = np.array([2, 3, 2, 3, 1, 2], np.int32)
    _check(w, fallback_frac=FEW_KEY_FALLBACK_FRAC)  # few-key edge case (capped)


@pytest.mark.parametrize("hq,hkv", EDGE_SHAPES)
def test_shared_decode_empty_and_one_key_sequences(hq, hkv):
    w = W.decode_zipf("sone", batch=3, hq=hq, hkv=hkv, d=128, docs_per_seq=1, doc_tokens=1, pool_docs=3,
                      zipf_s=1.0, seed=64)
    w.seg_indptr = np.array([0, 1, 1, 2], np.int32)  # sequence 1 is empty
    w.seg_doc, w.seg_len = w.seg_doc[:2].copy(), w.seg_len[:2].copy()
    dv = to_device(w)
    out = torch.full_like(dv.q, float("nan"))
    decode_shared(dv, shared_plan(dv), out=out)
    out = out.cpu()
    assert (out[1] == 0).all()
    for s, k in ((0, 0), (2, 1)):
        phys = int(w.doc_blocks[w.doc_block_indptr[w.seg_doc[k]]])
        for h in range(hq):
            assert torch.equal(out[s, h], w.v_pool[phys, h // (hq // hkv), 0])  # one key: output is v, exactly


def test_shared_decode_agrees_with_per_sequence_decode():
    w = W.decode_zipf("sagree", batch=16, hq=32, hkv=8, d=128, docs_per_seq=6, doc_tokens=200, pool_docs=5,
                      zipf_s=1.0, suffix_tokens=30, seed=165)
    dv = to_device(w)
    a = decode(dv).float().cpu().numpy()
    b = decode_shared(dv, shared_plan(dv)).float().cpu().numpy()
    assert np.abs(a - b).max() <= 2e-3 + 2e-2 * np.abs(a).max()
    assert np.mean(np.abs(a - b) <= 1e-2 * np.abs(a) + 1e-3) > 0.99


@pytest.mark.parametrize("hkv", [8, 1])
def test_shared_decode_shift_invariance_is_bitwise(hkv):
    kw = dict(batch=6, hq=32, hkv=hkv, d=128, docs_per_seq=3, doc_tokens=64, pool_docs=3, zipf_s=1.0,
              suffix_tokens=7, seed=166)
    da = to_device(W.decode_zipf("ss0", **kw))
    a = decode_shared(da, shared_plan(da)).cpu()
    for c in (1, 16, 4000):
        db = to_device(W.decode_zipf("ssc", shift=c, **kw))
        b = decode_shared(db, shared_plan(db)).cpu()
        assert torch.equal(a.view(torch.int16), b.view(torch.int16)), c


@pytest.mark.parametrize("hq,hkv", [(16, 4), (32, 1)])
def test_shared_decode_lazy0_control_on_materialised_pool(hq, hkv):
    w = W.decode_zipf("sctl", batch=4, hq=hq, hkv=hkv, d=128, docs_per_seq=3, doc_tokens=48, pool_docs=4,
                      zipf_s=1.0, suffix_tokens=8, share=False, seed=66)
    kabs = w.k_pool.double().clone()
    for s in range(w.num_seqs):
        p = 0
        for doc, Ln in w.seq_segments(s):
            for phys in w.doc_blocks[w.doc_block_indptr[doc]:w.doc_block_indptr[doc + 1]]:
                kabs[phys] = torch.from_numpy(rope(kabs[phys].numpy(), p, w.rope_theta))
            p += Ln
    dv = to_device(w, lazy=False, k_pool=kabs.to(torch.bfloat16))
    assert_close(decode_shared(dv, shared_plan(dv)), oracle.attention(w), "bf16", "shared lazy=0 control")


@pytest.mark.parametrize("hq,hkv", EDGE_SHAPES)
def test_shared_decode_flags_inconsistent_plan(hq, hkv):
    L = la()
    w = W.decode_zipf("sbadplan", batch=4, hq=hq, hkv=hkv, d=128, docs_per_seq=2, doc_tokens=40, pool_docs=3,
                      zipf_s=1.0, seed=167)
    dv = to_device(w)
    plan = shared_plan(dv)
    items = plan.items_host.copy()
    items[0, 8 + 1] += 1  # member 0's first block no longer holds the item's physical block
    bad = L.SharedPlan(items, plan.slot_indptr_host)
    out = decode_shared(dv, bad)
    torch.cuda.synchronize()
    assert L.device_status(clear=True) & L.LAZY_DEV_LAYOUT
    assert torch.isfinite(out.float()).all()


@pytest.mark.parametrize("hq,hkv", EDGE_SHAPES)
def test_shared_decode_flags_record_block_id_mismatch(hq, hkv):
    """A record whose block id disagrees with the block word (inside the pool, or past
    its end) is flagged; the kernel loads nothing outside the pool."""
    L = la()
    w = W.decode_zipf("sbadid", batch=4, hq=hq, hkv=hkv, d=128, docs_per_seq=2, doc_tokens=40, pool_docs=3,
                      zipf_s=1.0, seed=168)
    dv = to_device(w)
    plan = shared_plan(dv)
    ids0 = 8 + 4 * L.PLAN_MAX_MEMBERS
    for bad_id in (int(plan.items_host[0, ids0]) ^ 1, w.num_pool_blocks + 5):
        items = plan.items_host.copy()
        items[0, ids0] = bad_id
        out = decode_shared(dv, L.SharedPlan(items, plan.slot_indptr_host))
        torch.cuda.synchronize()
        assert L.device_status(clear=True) & L.LAZY_DEV_LAYOUT
        assert torch.isfinite(out.float()).all()


# ---------------------------------------------------------------- full sizes

def test_llama8b_shared_decode_full():
    _check(W.FULL["llama8b_decode"]())


def test_llama70b_shared_decode_full_sampled():
    _check(W.FULL["llama70b_decode"](), rows=[0, 7, 13, 31])


def test_mixed_shared_decode_full_sampled():
    d, _ = W.mixed_mqa()
    rng = np.random.default_rng(5)
    _check(d, rows=sorted(rng.choice(d.num_seqs, 6, replace=False).tolist()))


@pytest.mark.parametrize("hq,hkv", EDGE_SHAPES)
def test_split_phase_calls_equal_the_fused_call(hq, hkv):
    # lazy_attn_decode_shared_partials then lazy_attn_decode_shared_combine run the same
    # two kernels as lazy_attn_decode_shared: bit-identical outputs, and the partials
    # left in the workspace merge (here in fp64 on the host) to the oracle's result.
    L = la()
    w = W.decode_zipf("ssplit", batch=6, hq=hq, hkv=hkv, d=128, docs_per_seq=4, doc_tokens=120, pool_docs=3,
                      zipf_s=1.0, suffix_tokens=13, seed=175)
    dv = to_device(w)
    plan = shared_plan(dv)
    fused = decode_shared(dv, plan)
    ws = torch.empty(L.decode_shared_workspace_bytes(dv.p, plan.num_slots), dtype=torch.uint8, device="cuda")
    L.decode_shared_partials(dv.p, dv.q, dv.k_pool, dv.v_pool, dv.words, dv.q_pos, dv.rope, plan, ws)
    out = L.decode_shared_combine(dv.p, plan, ws, torch.empty_like(dv.q))
    assert torch.equal(out.view(torch.int16), fused.view(torch.int16))
    S, Hq, D = plan.num_slots, w.num_q_heads, w.head_dim
    f = ws.view(torch.float32).cpu().double().numpy()
    o, ml = f[: S * Hq * D].reshape(S, Hq, D), f[S * Hq * D: S * Hq * (D + 2)].reshape(S, Hq, 2)
    si = plan.slot_indptr_host
    merged = np.zeros((w.num_seqs, Hq, D))
    for s in range(w.num_seqs):
        m = ml[si[s]:si[s + 1], :, 0]
        M = m.max(0)
        wgt = np.exp2(m - M)
        merged[s] = (wgt[..., None] * o[si[s]:si[s + 1]]).sum(0) / (wgt * ml[si[s]:si[s + 1], :, 1]).sum(0)[:, None]
    assert_close(torch.from_numpy(merged), oracle.attention(w), "bf16", "partials merged on the host",
                 emulate=lambda r: emulate(w, r))
