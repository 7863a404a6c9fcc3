"""CPU tests of the cache manager and policy simulator (host C++ behind the C ABI).

Pins that do not depend on the library's own bookkeeping:
- closed forms with an unbounded pool: every distinct key misses once, so the miss
  blocks are the block count summed over the distinct documents (position-agnostic),
  distinct (document, offset) pairs (position-aware) or distinct prefixes (prefix
  caching), and the hit flags follow first occurrence;
- the content invariant under eviction: a block id handed out as a hit still holds
  what its last miss wrote (checked against a shadow "device memory"), and blocks
  of different contents never alias among admitted requests;
- the release window of the replay, from a pool sized for exactly two requests;
- the ordering the pages report: under a Zipf trace and a 1 GiB KV budget the
  position-agnostic hit rate is above the position-aware one, which is above
  prefix caching ("Resumo Técnico: LazyAttention", "Principais Contribuições" 2 and
  "Eficiência de Cache").
And, step by step, the library against a plain-Python model of the same rules
(``cache_model.py``): the same block ids, hit flags and counters.
"""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

import cache_model as M
from paged_kv_cache_57_gb300 import build as B
from paged_kv_cache_57_gb300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
POLICIES = (M.AGNOSTIC, M.AWARE, M.PREFIX)

# Llama-3.1-8B keeps 2 (K, V) x 32 layers x 8 KV heads x 128 x 2 B = 128 KiB per token,
# so a 1 GiB KV budget holds 8192 tokens = 512 blocks of 16.
BLOCKS_PER_GIB_LLAMA8B = (1 << 30) // (2 * 32 * 8 * 128 * 2) // 16


@pytest.fixture(scope="module")
def C():
    B.build()
    from paged_kv_cache_57_gb300 import cache
    return cache


def test_library_exports_every_declared_cache_symbol(C):
    src = re.sub(r"/\*.*?\*/", "", open(os.path.join(ROOT, "include", "lazy_cache.h")).read(), flags=re.S)
    names = sorted(set(re.findall(r"\b(lazy_cache_\w+)\s*\(", src)))
    assert set(names) == set(C.EXPORTED)
    out = subprocess.run(["nm", "-D", "--defined-only", C._lib._name], capture_output=True, text=True).stdout
    for n in names:
        assert re.search(rf"\bT {n}\b", out), n
    assert BLOCKS_PER_GIB_LLAMA8B == 512


def test_create_and_admit_argument_checks(C):
    L = C._lib
    assert not L.lazy_cache_create(0, 0)
    assert not L.lazy_cache_create(8, 3)
    assert not L.lazy_cache_create(8, -1)
    c = C.PagedCache(8, "agnostic")
    from paged_kv_cache_57_gb300.lazy_attn import LAZY_ERR_INVALID_ARG, LAZY_ERR_WORKSPACE, LazyAttnError
    for segs, pos0 in (([(-1, 5)], 0), ([(1, 0)], 0), ([(1, 5)], -3)):
        with pytest.raises(LazyAttnError) as e:
            c.admit(segs, pos0)
        assert e.value.status == LAZY_ERR_INVALID_ARG
    doc = np.array([1, 2], np.int32)
    ln = np.array([40, 20], np.int32)  # 3 + 2 blocks
    ind, blk, hit = np.zeros(3, np.int32), np.zeros(8, np.int32), np.zeros(2, np.int32)
    t = ctypes.c_int64()
    rc = L.lazy_cache_admit(c._c, 2, doc.ctypes.data, ln.ctypes.data, 0, ind.ctypes.data, blk.ctypes.data, 4,
                            hit.ctypes.data, ctypes.byref(t))
    assert rc == LAZY_ERR_WORKSPACE
    rc = L.lazy_cache_admit(c._c, 2, doc.ctypes.data, ln.ctypes.data, 0, None, blk.ctypes.data, 8,
                            hit.ctypes.data, ctypes.byref(t))
    assert rc == LAZY_ERR_INVALID_ARG
    assert c.stats()["hit_blocks"] + c.stats()["miss_blocks"] == 0  # nothing was admitted
    a = c.admit([(1, 40), (2, 20)])
    assert list(a.indptr) == [0, 3, 5] and list(a.hit) == [0, 0]
    c.release(a)
    for bad in (a.ticket, 999):  # released twice; never issued
        with pytest.raises(LazyAttnError):
            c.release(bad)
    empty = c.admit([])
    assert list(empty.indptr) == [0] and len(empty.blocks) == 0
    c.release(empty)
    with pytest.raises(LazyAttnError):
        C.simulate("agnostic", 8, [[(1, 5)]], concurrency=0)


def test_position_agnostic_reuse_across_offsets(C):
    # The same document at two offsets: one copy under the agnostic policy, two under
    # the position-aware one; prefix caching shares only an identical prefix.
    for policy, shared in (("agnostic", True), ("aware", False), ("prefix", False)):
        c = C.PagedCache(64, policy)
        a = c.admit([(7, 100), (3, 50)], pos0=0)
        b = c.admit([(3, 50), (7, 100)], pos0=0)
        assert (list(b.segment_blocks(1)) == list(a.segment_blocks(0))) == shared, policy
        assert list(b.hit) == ([1, 1] if shared else [0, 0]), policy
        d = c.admit([(7, 100), (3, 50)], pos0=0)  # the same request again: a hit under every policy
        assert list(d.hit) == [1, 1] and list(d.blocks) == list(a.blocks), policy
        e = c.admit([(7, 100), (3, 50)], pos0=16)  # moved by one block: only the agnostic copy serves
        assert list(e.hit) == ([1, 1] if shared else [0, 0]), policy


def _distinct_key_misses(policy, reqs, pos0):
    keys = {}
    for segs, p in zip(reqs, pos0):
        off, prefix = p, (p,)
        for doc, ln in segs:
            prefix = prefix + ((doc, ln),)
            k = doc if policy == M.AGNOSTIC else ((doc, off) if policy == M.AWARE else prefix)
            keys.setdefault(k, M.nblocks(ln))
            off += ln
    return sum(keys.values())


@pytest.mark.parametrize("policy", POLICIES)
def test_unbounded_pool_closed_form(C, policy):
    reqs, pos0 = W.cache_trace(num_requests=300, pool_docs=40, docs_per_request=4, zipf_s=1.1,
                               doc_tokens=(20, 90), prompt_tokens=0, seed=11)
    # a few requests with a prompt of another length and with repeated orders
    reqs += [list(r) for r in reqs[:20]]
    pos0 = pos0 + [32] * 10 + [0] * 10
    total = sum(M.nblocks(ln) for r in reqs for _, ln in r)
    st = C.simulate(policy, total, reqs, pos0, concurrency=3)
    miss = _distinct_key_misses(policy, reqs, pos0)
    assert st["miss_blocks"] == miss
    assert st["hit_blocks"] == total - miss
    assert st["evicted_blocks"] == 0 and st["rejected"] == 0
    assert st["resident_blocks"] == miss == st["peak_resident_blocks"]
    # a pool of 2^30 ids costs nothing until used: never-used ids are a counter
    assert C.simulate(policy, 1 << 30, reqs, pos0, concurrency=3) == st


def test_unbounded_hit_rates_are_ordered(C):
    reqs, pos0 = W.cache_trace(num_requests=400, pool_docs=100, docs_per_request=5, zipf_s=1.0, seed=12)
    total = sum(M.nblocks(ln) for r in reqs for _, ln in r)
    hr = [C.simulate(p, total, reqs, pos0)["hit_rate"] for p in POLICIES]
    # a (document, offset) or prefix match implies a document match, and a prefix match an offset match
    assert hr[0] >= hr[1] >= hr[2]
    assert hr[0] > hr[1]


def _run_with_shadow(C, policy, num_blocks, reqs, pos0, rng, hold):
    """Admits reqs with a random number (< hold) of requests kept pinned; checks hits
    against a shadow memory and the no-alias rule among pinned requests."""
    c = C.PagedCache(num_blocks, policy)
    shadow = {}
    live = []
    for segs, p in zip(reqs, pos0):
        a = c.admit(segs, p)
        if a is not None:
            off, prefix = p, (p,)
            for i, (doc, ln) in enumerate(segs):
                prefix = prefix + ((doc, ln),)
                ident = doc if policy == M.AGNOSTIC else ((doc, off) if policy == M.AWARE else prefix)
                ids = a.segment_blocks(i)
                assert len(ids) == M.nblocks(ln)
                assert ((ids >= 0) & (ids < num_blocks)).all()
                for k, b in enumerate(ids):
                    if a.hit[i]:
                        assert shadow[int(b)] == (ident, k), "a hit returned blocks that were reused"
                    else:
                        shadow[int(b)] = (ident, k)
                off += ln
            live.append((a, segs, p))
        while live and (len(live) >= hold or rng.random() < 0.3):
            c.release(live.pop(int(rng.integers(len(live))))[0])
        owner = {}
        for a, segs, _ in live:  # pinned requests: one content per block id
            for i in range(len(segs)):
                for k, b in enumerate(a.segment_blocks(i)):
                    assert owner.setdefault(int(b), shadow[int(b)]) == shadow[int(b)]
    st = c.stats()
    assert st["resident_blocks"] <= num_blocks and st["peak_resident_blocks"] <= num_blocks
    return st


@pytest.mark.parametrize("policy", POLICIES)
def test_hits_never_return_reused_blocks_under_eviction(C, policy):
    rng = np.random.default_rng(13 + policy)
    reqs, pos0 = W.cache_trace(num_requests=600, pool_docs=30, docs_per_request=3, zipf_s=1.2,
                               doc_tokens=(10, 70), seed=14)
    pos0 = [int(x) for x in rng.choice([0, 16, 40], size=len(reqs))]
    st = _run_with_shadow(C, policy, 40, reqs, pos0, rng, hold=4)
    assert st["evicted_blocks"] > 0 and st["hit_blocks"] > 0


def _random_requests(rng, n, docs, max_segs, lens):
    out = []
    for _ in range(n):
        segs = []
        for _ in range(int(rng.integers(0, max_segs + 1))):
            doc = int(rng.integers(docs))
            segs.append((doc, int(rng.choice(lens))))
        out.append((segs, int(rng.choice([0, 7, 16]))))
    return out


@pytest.mark.parametrize("policy", POLICIES)
def test_library_matches_python_model_step_by_step(C, policy):
    # Small pools, repeated documents within a request, a document requested at
    # several lengths (a longer request replaces a shorter cached copy, even one still
    # pinned), releases in random order: ids, flags and counters must all agree.
    rng = np.random.default_rng(100 + policy)
    for trial in range(6):
        num_blocks = int(rng.integers(6, 30))
        lib, mod = C.PagedCache(num_blocks, policy), M.CacheModel(num_blocks, policy)
        live = []
        for segs, p in _random_requests(rng, 150, docs=8, max_segs=4, lens=[5, 16, 17, 40, 64]):
            a, b = lib.admit(segs, p), mod.admit(segs, p)
            assert (a is None) == (b is None)
            if a is not None:
                assert [list(a.segment_blocks(i)) for i in range(len(segs))] == b[1]
                assert list(a.hit) == b[2]
                live.append((a.ticket, b[0]))
            while live and rng.random() < 0.45:
                ta, tb = live.pop(int(rng.integers(len(live))))
                lib.release(ta)
                mod.release(tb)
            got = lib.stats()
            got.pop("hit_rate")
            assert got == mod.st, (trial, got, mod.st)
        for ta, tb in live:
            lib.release(ta)
            mod.release(tb)
        got = lib.stats()
        got.pop("hit_rate")
        assert got == mod.st


@pytest.mark.parametrize("concurrency", [1, 2, 5])
def test_simulate_matches_the_model_and_the_manual_replay(C, concurrency):
    rng = np.random.default_rng(21)
    reqs, pos0 = W.cache_trace(num_requests=200, pool_docs=25, docs_per_request=3, zipf_s=1.0,
                               doc_tokens=(16, 80), seed=22)
    for policy in POLICIES:
        st = C.simulate(policy, 48, reqs, pos0, concurrency=concurrency)
        ref = M.simulate(policy, 48, reqs, pos0, concurrency=concurrency)
        assert {k: v for k, v in st.items() if k != "hit_rate"} == ref, policy
    del rng


def test_release_window(C):
    # Each request needs 4 new blocks (distinct documents); the pool holds 8. With up to
    # two requests pinned every admission fits; with three pinned the third always waits.
    reqs = [[(r, 64)] for r in range(12)]
    for conc, rejected in ((1, 0), (2, 0), (3, 4)):
        st = C.simulate("agnostic", 8, reqs, concurrency=conc)
        assert st["rejected"] == rejected, conc
        assert st["miss_blocks"] == 4 * (12 - rejected)


def test_zipf_one_gib_budget_ordering(C):
    # RAG-shaped trace: 5 retrieved documents of 128..512 tokens per request from a pool
    # of 500, high skew, after a 64-token prompt; 1 GiB of Llama-3.1-8B KV.
    reqs, pos0 = W.cache_trace(num_requests=3000, pool_docs=500, docs_per_request=5, zipf_s=1.2,
                               doc_tokens=(128, 512), prompt_tokens=64, seed=23)
    hr = {p: C.simulate(p, BLOCKS_PER_GIB_LLAMA8B, reqs, pos0, concurrency=4)["hit_rate"]
          for p in ("agnostic", "aware", "prefix")}
    assert hr["agnostic"] > 1.5 * hr["aware"] > 0
    assert hr["aware"] > hr["prefix"]
