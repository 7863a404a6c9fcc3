"""CPU tests of the C ABI: symbols, argument checks and the host packer.

Nothing here launches a kernel; every call either returns before touching CUDA
(argument and layout checks, size queries) or is pure host code (the packer).
The expected words are rebuilt from the generator's document lists by plain
Python, independently of the library.
"""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

from paged_kv_cache_57_gb300 import build as B
from paged_kv_cache_57_gb300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def la():
    B.build()
    from paged_kv_cache_57_gb300 import lazy_attn
    return lazy_attn


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "lazy_attn.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(lazy_attn_\w+)\s*\(", src)))


def test_library_exports_every_declared_symbol(la):
    names = declared_symbols()
    assert len(names) >= 12
    lib = ctypes.CDLL(la.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(la.EXPORTED)
    out = subprocess.run(["nm", "-D", "--defined-only", la.LIB_PATH], capture_output=True, text=True).stdout
    for n in names:
        assert re.search(rf"\bT {n}\b", out), n


def test_status_strings(la):
    for s in range(7):
        assert la.status_string(s).startswith("LAZY_")
    assert "unknown" in la.status_string(99)


def _params(la, w, **kw):
    return la.make_params(num_seqs=w.num_seqs, num_q_heads=w.num_q_heads, num_kv_heads=w.num_kv_heads,
                          head_dim=w.head_dim, num_pool_blocks=w.num_pool_blocks,
                          max_blocks_per_seq=kw.pop("max_blocks", w.max_blocks_per_seq), dtype=w.dtype,
                          rope_theta=w.rope_theta, **kw)


def expected_blocks(w, s):
    """(phys, p, valid) per logical block, from the document lists."""
    out = []
    p = int(w.seq_pos0[s])
    for doc, L in w.seq_segments(s):
        base = int(w.doc_block_indptr[doc])
        for j in range((L + 15) // 16):
            out.append((int(w.doc_blocks[base + j]), p, min(16, L - 16 * j)))
        p += L
    return out


def unpack(word, b, id_bits):
    phys = int(word) & ((1 << id_bits) - 1)
    off = int(np.int32(np.uint32(word))) >> id_bits
    return phys, 16 * b - off


def valid_by_rule(ps, b, nb, seq_len):
    if b == nb - 1:
        return seq_len - 16 * (nb - 1)
    if ps[b + 1] != ps[b]:
        return ((ps[b + 1] - ps[b] - 1) & 15) + 1
    return 16


def _workloads():
    yield W.tiny_fp32()
    yield W.tiny_fp32(shift=3000)
    yield W.decode_zipf("d", batch=5, hq=8, hkv=2, d=64, docs_per_seq=4, doc_tokens=48, pool_docs=7,
                        zipf_s=1.0, suffix_tokens=9, seed=5)
    yield W.prefill_zipf("p", batch=3, hq=4, hkv=2, d=64, docs_per_seq=2, doc_tokens=40, pool_docs=4,
                         zipf_s=1.2, chunk_tokens=[1, 17, 130], seed=6)
    d, p = W.mixed_mqa(n_decode=6, n_prefill=2, chunk=40, hq=4, hkv=1, d=64, pool_docs=30, ctx_lo=50,
                       ctx_hi=3000, doc_lo=5, doc_hi=300, seed=7)
    yield d
    yield p


@pytest.mark.parametrize("w", list(_workloads()), ids=lambda w: f"{w.name}-{w.num_seqs}")
def test_host_packer_round_trip(la, w):
    p = _params(la, w)
    words, seq_lens = la.pack_block_words_host(p, len(w.doc_len), w.seg_indptr, w.seg_doc, w.seg_len, w.seq_pos0,
                                               w.doc_block_indptr, w.doc_blocks)
    id_bits = 18
    for s in range(w.num_seqs):
        exp = expected_blocks(w, s)
        nb = len(exp)
        assert seq_lens[s] == (16 * (nb - 1) + exp[-1][2] if nb else 0)
        got = [unpack(words[s, b], b, id_bits) for b in range(nb)]
        assert [g[0] for g in got] == [e[0] for e in exp]
        assert [g[1] for g in got] == [e[1] for e in exp]
        ps = [g[1] for g in got]
        assert [valid_by_rule(ps, b, nb, int(seq_lens[s])) for b in range(nb)] == [e[2] for e in exp]
        assert (words[s, nb:] == 0).all()


@pytest.mark.parametrize("w", list(_workloads())[2:], ids=lambda w: f"{w.name}-{w.num_seqs}")
def test_host_packer_key_position_words(la, w):
    # key_positions = 1: a word's position is that of its block's first key (the
    # document start plus 16 per earlier block of the document); ids, sequence
    # lengths and the valid-count rule are those of the document-start form.
    words0, lens0 = la.pack_block_words_host(_params(la, w), len(w.doc_len), w.seg_indptr, w.seg_doc, w.seg_len,
                                             w.seq_pos0, w.doc_block_indptr, w.doc_blocks)
    words, seq_lens = la.pack_block_words_host(_params(la, w, key_positions=True), len(w.doc_len), w.seg_indptr,
                                               w.seg_doc, w.seg_len, w.seq_pos0, w.doc_block_indptr, w.doc_blocks)
    assert np.array_equal(seq_lens, lens0)
    id_bits = 18
    for s in range(w.num_seqs):
        first_keys, p = [], int(w.seq_pos0[s])
        for doc, L in w.seq_segments(s):
            first_keys += [p + 16 * j for j in range((L + 15) // 16)]
            p += L
        nb = len(first_keys)
        got = [unpack(words[s, b], b, id_bits) for b in range(nb)]
        assert [g[1] for g in got] == first_keys
        assert [g[0] for g in got] == [unpack(words0[s, b], b, id_bits)[0] for b in range(nb)]
        assert [valid_by_rule(first_keys, b, nb, int(seq_lens[s])) for b in range(nb)] == \
            [e[2] for e in expected_blocks(w, s)]
        assert (words[s, nb:] == 0).all()


def test_host_packer_rejects_bad_layouts(la):
    w = W.decode_zipf("bad", batch=2, hq=4, hkv=2, d=64, docs_per_seq=2, doc_tokens=20, pool_docs=3, zipf_s=1.0,
                      seed=8)
    p = _params(la, w)
    args = [w.seg_indptr, w.seg_doc, w.seg_len, w.seq_pos0, w.doc_block_indptr, w.doc_blocks]

    def run(params=p, **repl):
        a = dict(zip(["seg_indptr", "seg_doc", "seg_len", "seq_pos0", "doc_block_indptr", "doc_blocks"],
                     [x.copy() for x in args]))
        for k, fn in repl.items():
            a[k] = fn(a[k])
        with pytest.raises(la.LazyAttnError) as e:
            la.pack_block_words_host(params, len(w.doc_len), *a.values())
        return e.value.status

    def set_at(i, v):
        def f(x):
            x[i] = v
            return x
        return f

    assert run(seg_len=set_at(0, 33)) == la.LAZY_ERR_LAYOUT      # longer than its document
    assert run(seg_len=set_at(0, 0)) == la.LAZY_ERR_LAYOUT       # empty segment
    assert run(seg_doc=set_at(0, 99)) == la.LAZY_ERR_LAYOUT      # unknown document
    assert run(doc_blocks=set_at(0, w.num_pool_blocks)) == la.LAZY_ERR_LAYOUT  # outside the pool
    assert run(seq_pos0=set_at(0, 9000)) == la.LAZY_ERR_LAYOUT   # off = -9000 does not fit 14 bits
    small = _params(la, w, max_blocks=1)
    assert run(params=small) == la.LAZY_ERR_LAYOUT               # too many blocks for the table


def test_argument_checks_return_before_cuda(la):
    w = W.tiny_fp32()
    bad = [dict(head_dim=96), dict(num_kv_heads=3), dict(id_bits=30), dict(num_splits=-1)]
    for kw in bad:
        p = _params(la, w)
        for k, v in kw.items():
            setattr(p, k, v)
        st = la._lib.lazy_attn_decode(ctypes.byref(p), *([None] * 9), 0, None)
        assert st in (la.LAZY_ERR_UNSUPPORTED, la.LAZY_ERR_INVALID_ARG), kw
    p = _params(la, w)
    p.block_size = 32
    assert la._lib.lazy_attn_decode(ctypes.byref(p), *([None] * 9), 0, None) == la.LAZY_ERR_UNSUPPORTED
    p = _params(la, w)
    assert la._lib.lazy_attn_decode(ctypes.byref(p), *([None] * 9), 0, None) == la.LAZY_ERR_INVALID_ARG
    p.dtype = la.LAZY_F32
    assert la._lib.lazy_attn_prefill(ctypes.byref(p), None, None, None, 1, 1, *([None] * 7), 0, None) \
        == la.LAZY_ERR_UNSUPPORTED


def test_size_queries(la):
    w = W.FULL["tiny_fp32"]()
    p = _params(la, w)
    assert la.rope_table_bytes(p) == 32 * 8 * 129
    p.head_dim = 128
    assert la.rope_table_bytes(p) == 64 * 8 * 129
    p.num_splits = 1
    assert la.decode_workspace_bytes(p) == 0
    p.num_splits, p.max_blocks_per_seq = 4, 64
    assert la.decode_workspace_bytes(p) == 1 * 4 * 4 * (128 + 2) * 4


# ---------------------------------------------------------------- shared-run planner

def _shared_workloads():
    yield W.decode_zipf("sd", batch=9, hq=8, hkv=2, d=64, docs_per_seq=5, doc_tokens=600, pool_docs=4,
                        zipf_s=1.0, suffix_tokens=9, seed=15)
    yield W.decode_zipf("sd1", batch=40, hq=4, hkv=4, d=128, docs_per_seq=3, doc_tokens=40, pool_docs=2,
                        zipf_s=1.0, seed=16)  # G = 1: items of up to 16 members, 16 rows
    d, _ = W.mixed_mqa(n_decode=6, n_prefill=1, chunk=40, hq=8, hkv=1, d=64, pool_docs=30, ctx_lo=50,
                       ctx_hi=3000, doc_lo=5, doc_hi=300, seed=17)
    yield d
    # G = 32, d = 128: the tensor-core kernel's items, up to 4 members (128 rows)
    yield W.decode_zipf("sdw", batch=12, hq=32, hkv=1, d=128, docs_per_seq=3, doc_tokens=100, pool_docs=2,
                        zipf_s=1.0, seed=19)


@pytest.mark.parametrize("chunk", [0, 1, 3, 32])
@pytest.mark.parametrize("w", list(_shared_workloads()), ids=lambda w: w.name)
def test_shared_plan_covers_every_block_once(la, w, chunk):
    """Every logical block of every sequence is computed exactly once, in a slot of
    its own sequence, by an item whose source blocks are the same physical blocks."""
    p = _params(la, w)
    items, slot_indptr = la.plan_shared_host(p, len(w.doc_len), w.seg_indptr, w.seg_doc, w.seg_len,
                                             w.doc_block_indptr, w.doc_blocks, chunk_blocks=chunk)
    G = w.num_q_heads // w.num_kv_heads
    rows_cap = 128 if G >= 8 and w.head_dim == 128 else 64  # one tcgen05 tile, or 4 mma.sync row tiles
    exp = {s: expected_blocks(w, s) for s in range(w.num_seqs)}
    cover = {s: np.zeros(len(exp[s]), np.int64) for s in range(w.num_seqs)}
    slots_seen = set()
    cost = []
    for it in items:
        src, b0, nb, last, nm = (int(x) for x in it[:5])
        ids = it[8 + 4 * la.PLAN_MAX_MEMBERS:]
        assert (it[6:8] == 0).all() and (it[8 + 4 * nm: 8 + 4 * la.PLAN_MAX_MEMBERS] == 0).all()
        # [5]: the item's first block within its document, whose start is the member's segment start
        seg_first = {}
        bpos = 0
        for doc, ln in w.seq_segments(src):
            nbk = -(-ln // 16)
            for q in range(nbk):
                seg_first[bpos + q] = bpos
            bpos += nbk
        assert int(it[5]) == b0 - seg_first[b0]
        assert 1 <= nm <= la.PLAN_MAX_MEMBERS and nm * G <= rows_cap
        cost.append(nb)
        assert nb <= (chunk or (256 if rows_cap == 128 else 32))
        src_phys = [exp[src][b][0] for b in range(b0, b0 + nb)]
        nid = min(nb, la.PLAN_ITEM_BLOCK_IDS)  # the record names the item's first blocks
        assert list(ids[:nid]) == src_phys[:nid] and (ids[nid:] == 0).all()
        assert [exp[src][b][2] for b in range(b0, b0 + nb)] == [16] * (nb - 1) + [last]
        for seq, bm, slot, zero in it[8: 8 + 4 * nm].reshape(nm, 4):
            assert zero == 0
            assert [exp[seq][b][0] for b in range(bm, bm + nb)] == src_phys
            assert [exp[seq][b][2] for b in range(bm, bm + nb)] == [16] * (nb - 1) + [last]
            assert len({exp[seq][b][1] for b in range(bm, bm + nb)}) == 1  # one document run
            assert slot_indptr[seq] <= slot < slot_indptr[seq + 1]
            assert slot not in slots_seen
            slots_seen.add(slot)
            cover[seq][bm:bm + nb] += 1
    # longest items first; for the bf16 mma.sync kernel (64-row items), items of at most
    # 8 blocks are spread evenly through the order instead (each small item k at
    # position floor((k + 1/2) n / n_small) or just after, never clustered at the end)
    cost = np.asarray(cost)
    small = (cost <= 8) if rows_cap == 64 else np.zeros(len(cost), bool)
    big_costs = cost[~small]
    assert (np.diff(big_costs) <= 0).all()
    if small.any() and (~small).any():
        pos = np.flatnonzero(small)
        n, ns = len(cost), len(pos)
        assert all(pos[k] >= int((k + 0.5) * n / ns) for k in range(ns))
        assert np.diff(np.concatenate([[-1], pos, [n]])).max() <= -(-n // ns) + 1
    else:
        assert (np.diff(cost) <= 0).all()
    if w.name == "sdw":  # a document shared by more than two sequences fills a 128-row tile
        assert items[:, 4].max() * G == 128
    assert len(slots_seen) == slot_indptr[-1]
    for s in range(w.num_seqs):
        assert (cover[s] == 1).all(), s
    # Loads are shared: no more source blocks than logical ones.
    assert items[:, 2].sum() <= sum(len(e) for e in exp.values())


def test_shared_plan_automatic_chunk_for_the_tensor_core_kernel(la):
    # 0 selects 32 blocks for the mma.sync kernel; for the tensor-core kernel (G >= 8,
    # d = 128) about one item per resident CTA (2 x 152 over the KV heads): the sum of
    # the member sets' blocks over that count, rounded up to 4, within 32 .. 256.
    for hkv, docs in ((1, 6), (2, 40)):
        w = W.decode_zipf("sauto", batch=24, hq=32 * hkv, hkv=hkv, d=128, docs_per_seq=docs, doc_tokens=1000,
                          pool_docs=60, zipf_s=0.5, seed=20)
        p = _params(la, w)
        items, _ = la.plan_shared_host(p, len(w.doc_len), w.seg_indptr, w.seg_doc, w.seg_len,
                                       w.doc_block_indptr, w.doc_blocks, chunk_blocks=0)
        per_set = 128 // 32
        groups = {}
        for s_ in range(w.num_seqs):
            for doc, ln in w.seq_segments(s_):
                groups[(doc, ln)] = groups.get((doc, ln), 0) + 1
        total = sum(-(-ln // 16) * -(-n // per_set) for (doc, ln), n in groups.items())
        want = min(256, max(32, -(-(-(-total // (304 // hkv))) // 4) * 4))
        assert items[:, 2].max() == min(want, 63)  # 1000-token documents have 63 blocks
        assert want > 32 or hkv == 1
    w = W.decode_zipf("sauto8", batch=8, hq=8, hkv=2, d=128, docs_per_seq=4, doc_tokens=2000, pool_docs=30,
                      zipf_s=0.5, seed=21)
    items, _ = la.plan_shared_host(_params(la, w), len(w.doc_len), w.seg_indptr, w.seg_doc, w.seg_len,
                                   w.doc_block_indptr, w.doc_blocks, chunk_blocks=0)
    assert items[:, 2].max() == 32  # mma.sync kernel: 32 blocks


def test_shared_plan_rejects_bad_layouts(la):
    w = W.decode_zipf("sbad", batch=2, hq=4, hkv=2, d=64, docs_per_seq=2, doc_tokens=20, pool_docs=3,
                      zipf_s=1.0, seed=18)
    p = _params(la, w)

    def run(params=p, **repl):
        a = dict(seg_indptr=w.seg_indptr.copy(), seg_doc=w.seg_doc.copy(), seg_len=w.seg_len.copy(),
                 doc_block_indptr=w.doc_block_indptr.copy(), doc_blocks=w.doc_blocks.copy())
        a.update(repl)
        with pytest.raises(la.LazyAttnError) as e:
            la.plan_shared_host(params, len(w.doc_len), *a.values())
        return e.value.status

    sl = w.seg_len.copy()
    sl[0] = 33
    assert run(seg_len=sl) == la.LAZY_ERR_LAYOUT
    db = w.doc_blocks.copy()
    db[0] = w.num_pool_blocks
    assert run(doc_blocks=db) == la.LAZY_ERR_LAYOUT
    assert run(params=_params(la, w, max_blocks=1)) == la.LAZY_ERR_LAYOUT
    big = _params(la, w)
    big.num_q_heads = 4 * 65
    big.num_kv_heads = 4
    assert run(params=big) == la.LAZY_ERR_UNSUPPORTED


def test_shared_decode_argument_checks(la):
    w = W.tiny_fp32()
    p = _params(la, w)
    null = [None] * 6
    # fp32 has no shared-run kernel; bf16 with null pointers is an invalid argument; no CUDA call either way
    assert la._lib.lazy_attn_decode_shared(ctypes.byref(p), *null, 1, None, 1, None, None, None, 0,
                                           None) == la.LAZY_ERR_UNSUPPORTED
    p.dtype = la.LAZY_BF16
    assert la._lib.lazy_attn_decode_shared(ctypes.byref(p), *null, 1, None, 1, None, None, None, 0,
                                           None) == la.LAZY_ERR_INVALID_ARG
    assert la.decode_shared_workspace_bytes(p, 10) == 10 * 4 * (64 + 2) * 4
