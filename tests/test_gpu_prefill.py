"""GPU parity of the tcgen05 prefill kernel against the CPU oracle (through the C ABI)."""
import numpy as np
import pytest
import torch

import oracle
from brute import rope
from bf16_model import emulate
from gpu_util import FEW_KEY_FALLBACK_FRAC, assert_close, la, prefill, to_device
from paged_kv_cache_57_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _clean_status():
    la().device_status(clear=True)
    yield
    assert la().device_status(clear=True) == 0, "device status word set"


def _check(w, rows=None, lazy=True, k_pool=None, fallback_frac=0.0):
    dv = to_device(w, lazy=lazy, k_pool=k_pool)
    out = prefill(dv)
    ref = oracle.attention(w, rows=rows)
    got = out if rows is None else out[torch.as_tensor(rows, device=out.device)]
    sel = np.arange(ref.shape[0]) if rows is None else np.asarray(rows)
    return assert_close(got, ref, w.dtype, w.name,
                        emulate=lambda r: emulate(w, sel[r], lazy=lazy, k_pool=k_pool), fallback_frac=fallback_frac)


def test_prefill_single_tile():
    w = W.prefill_zipf("p1", batch=1, hq=4, hkv=2, docs_per_seq=2, doc_tokens=64, pool_docs=3, zipf_s=1.0,
                       chunk_tokens=128, seed=71)
    _check(w)


@pytest.mark.parametrize("chunks", [[1], [17, 130], [128, 256], [255, 3, 64], [64, 0, 17], [0, 1]])
def test_prefill_varlen_chunks(chunks):
    w = W.prefill_zipf("pv", batch=len(chunks), hq=8, hkv=2, docs_per_seq=3, doc_tokens=200, pool_docs=5,
                       zipf_s=1.2, chunk_tokens=chunks, seed=72 + len(chunks))
    _check(w)


def test_prefill_chunk_only_is_causal():
    w = W.prefill_zipf("pc", batch=2, hq=4, hkv=4, docs_per_seq=0, doc_tokens=16, pool_docs=1, zipf_s=1.0,
                       chunk_tokens=[300, 45], seed=74)
    # the first rows of a chunk with no cached context see 1, 2, 3 ... keys: few-key edge case (capped)
    _check(w, fallback_frac=FEW_KEY_FALLBACK_FRAC)


@pytest.mark.parametrize("hq,hkv", [(32, 8), (32, 1), (8, 8)])
def test_prefill_gqa(hq, hkv):
    w = W.prefill_zipf("pg", batch=2, hq=hq, hkv=hkv, docs_per_seq=2, doc_tokens=300, pool_docs=4, zipf_s=1.2,
                       chunk_tokens=[200, 129], seed=75 + hq + hkv)
    _check(w)


def test_prefill_holes_and_partial_blocks():
    _, p = W.mixed_mqa(n_decode=1, n_prefill=3, chunk=150, hq=8, hkv=1, pool_docs=60, ctx_lo=100, ctx_hi=3000,
                       doc_lo=5, doc_hi=300, seed=76)
    _check(p)


def test_prefill_shift_invariance():
    kw = dict(batch=2, hq=8, hkv=2, docs_per_seq=2, doc_tokens=96, pool_docs=3, zipf_s=1.0, chunk_tokens=[100, 37],
              seed=77)
    a = prefill(to_device(W.prefill_zipf("s0", **kw))).float().cpu().numpy()
    w0 = W.prefill_zipf("s0", **kw)
    ref = oracle.attention(w0)
    for c in (16, 5000, 100000):
        # a shift of 100000 needs a wider offset field: 12 id bits leave 20 signed bits
        b = prefill(to_device(W.prefill_zipf("sc", shift=c, **kw), id_bits=12 if c > 8000 else 0))
        assert_close(b, ref, "bf16", f"shift {c}", emulate=lambda r: emulate(w0, r))
    assert np.isfinite(a).all()


def test_prefill_lazy0_control_on_materialised_pool():
    w = W.prefill_zipf("pctl", batch=2, hq=8, hkv=2, docs_per_seq=2, doc_tokens=80, pool_docs=500, zipf_s=0.0,
                       chunk_tokens=[70, 33], seed=78)
    # distinct documents per sequence so that each pool block has one absolute position
    assert len(set(w.seg_doc.tolist())) == len(w.seg_doc)
    kabs = w.k_pool.double().clone()
    for s in range(w.num_seqs):
        p = 0
        for doc, Ln in w.seq_segments(s):
            for phys in w.doc_blocks[w.doc_block_indptr[doc]:w.doc_block_indptr[doc + 1]]:
                kabs[phys] = torch.from_numpy(rope(kabs[phys].numpy(), p, w.rope_theta))
            p += Ln
    _check(w, lazy=False, k_pool=kabs.to(torch.bfloat16))


def test_llama8b_prefill_full_sampled():
    w = W.FULL["llama8b_prefill"]()
    rng = np.random.default_rng(3)
    cu = w.cu_seqlens_q
    rows = sorted(set(int(cu[s]) + int(x) for s in range(w.num_seqs)
                      for x in rng.choice(int(cu[s + 1] - cu[s]), 16, replace=False)))
    _check(w, rows=rows)


def test_mixed_prefill_full_sampled():
    _, p = W.mixed_mqa()
    rng = np.random.default_rng(4)
    rows = sorted(int(x) for x in rng.choice(p.q.shape[0], 24, replace=False))
    _check(p, rows=rows)


# ---------------------------------------------------------------- stream-K splits

def _split_units(w, sms):
    """Host replica of the two-tile kernel's schedule: when all (sequence, tile, head pair)
    units are about equally long, the first floor(units / sms) * sms run whole, one per
    CTA; the rest are laid end to end by K tiles and cut into sms ranges of W tiles. Returns the units cut by a range
    boundary, as (s, tile, hp, n, U0), and W."""
    P = w.num_q_heads // 2
    cu = np.asarray(w.cu_seqlens_q)
    C = np.diff(cu)
    T = int((C.max() + 127) // 128)
    nb = w.blocks_per_seq()
    units = []
    for s in range(w.num_seqs):
        for tile in range(T):
            row0 = 128 * tile
            if row0 >= C[s]:
                continue
            b_chunk = max(0, int(nb[s]) - (int(C[s]) + 15) // 16)
            last_block = min(int(nb[s]) - 1, b_chunk + (min(int(C[s]), row0 + 128) - 1) // 16)
            n = last_block // 8 + 1 if last_block >= 0 else 0
            if n:
                units += [(s, tile, hp, n) for hp in range(P)]
    ns = [u[3] for u in units]
    uniform = bool(units) and max(ns) * 4 <= min(ns) * 5
    D = len(units) // sms * sms if uniform else 0
    tot, out = 0, []
    for s, tile, hp, n in units[D:]:
        out.append((s, tile, hp, n, tot))
        tot += n
    W = -(-tot // sms) if tot else 0
    return [u for u in out if u[4] // W != (u[4] + u[3] - 1) // W], W


def test_prefill_one_unit_across_many_ctas():
    # one sequence, one 128-row tile, one head pair: ~50 K tiles cut into ~50 one-tile pieces
    w = W.prefill_zipf("psplit", batch=1, hq=2, hkv=1, docs_per_seq=6, doc_tokens=1000, pool_docs=6, zipf_s=0.0,
                       chunk_tokens=[128], seed=79)
    split, Wr = _split_units(w, torch.cuda.get_device_properties(0).multi_processor_count)
    assert split and Wr <= 2
    _check(w)


def test_llama8b_prefill_split_units_sampled():
    w = W.FULL["llama8b_prefill"]()
    split, _ = _split_units(w, torch.cuda.get_device_properties(0).multi_processor_count)
    assert len(split) > 50
    cu = np.asarray(w.cu_seqlens_q)
    rng = np.random.default_rng(6)
    rows = set()
    for s, tile, hp, n, U0 in split[:: max(1, len(split) // 12)]:
        lo, hi = int(cu[s]) + 128 * tile, min(int(cu[s + 1]), int(cu[s]) + 128 * tile + 128)
        rows.update(int(x) for x in rng.choice(np.arange(lo, hi), 4, replace=False))
    _check(w, rows=sorted(rows))


@pytest.mark.parametrize("hq,hkv", [(8, 2), (6, 2)])
def test_prefill_non_default_sm_scale(hq, hkv):
    # even GQA ratio: the stream-K kernel; odd (3 per KV head): the TMEM-Q kernel
    w = W.prefill_zipf("pscale", batch=2, hq=hq, hkv=hkv, docs_per_seq=2, doc_tokens=150, pool_docs=3,
                       zipf_s=1.0, chunk_tokens=[140, 33], seed=79 + hq)
    dv = to_device(w)
    dv.p.sm_scale = 0.05
    ref = oracle.attention(w, sm_scale=0.05)
    assert_close(prefill(dv), ref, "bf16", f"prefill {hq}/{hkv}, sm_scale 0.05")
    assert np.abs(ref - oracle.attention(w)).max() > 1e-2
