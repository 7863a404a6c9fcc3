"""Seeded synthetic workloads for LazyAttention over a paged, position-agnostic KV cache.

This module only draws random numbers and lays them out: it holds none of the
attention or rotary arithmetic. Both the CUDA path and the CPU oracle read what
it produces, so it must stay free of the method's math.

What is generated (the shapes follow the LazyAttention technical summary,
"Experimental Results": Llama-3.1-8B/70B under skewed, Zipf-like document reuse,
and the vLLM 16-token paged layout from "KV Cache, Flash Attention & Otimização
de Inferência", section "PagedAttention"):

* a pool of cached documents. Document ``doc`` has a fixed length and its own
  stored K and V rows, drawn N(0, 1) from a PCG64 stream keyed by
  ``(seed, doc)``, so every occurrence of a document is byte-identical. Stored K
  is the document's key already rotated at its local positions 0..len-1; an
  isotropic Gaussian is invariant under rotation, so drawing the stored rows
  directly has the same distribution as rotating raw N(0, 1) keys;
* per sequence, a list of segments ``(doc, used_len)`` placed at concatenated
  global offsets starting at ``seq_pos0``; documents are drawn from a finite
  Zipf law P(rank r) ~ r^-s, r = 1..N (rank -> doc id is the identity), with
  replacement;
* physical 16-token blocks: every used document gets ceil(len/16) blocks whose
  ids are a seeded random permutation of the pool (fragmented, as after
  allocator churn). Unused pool blocks and the slots past a document's end are
  filled with NaN, so that any read of a slot that is not part of the context
  poisons the output;
* queries q ~ N(0, 1), unrotated, with their absolute positions.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np
import torch

BLOCK = 16  # tokens per physical block

_TORCH_DTYPE = {"f32": torch.float32, "bf16": torch.bfloat16}


@dataclasses.dataclass
class Workload:
    """One attention call's worth of inputs (host tensors)."""

    name: str
    kind: str  # "decode" or "prefill"
    dtype: str  # "f32" or "bf16"
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    rope_theta: float
    # layout, host int32 arrays
    seg_indptr: np.ndarray  # [B+1]
    seg_doc: np.ndarray  # [nseg]
    seg_len: np.ndarray  # [nseg] tokens of the document used (a prefix)
    seq_pos0: np.ndarray  # [B] global position of the first cached token
    doc_len: np.ndarray  # [ndocs] full stored length of each document
    doc_block_indptr: np.ndarray  # [ndocs+1]
    doc_blocks: np.ndarray  # physical block ids, per document in token order
    num_pool_blocks: int
    k_pool: torch.Tensor  # [num_pool_blocks, Hkv, 16, d] stored (locally rotated) K
    v_pool: torch.Tensor  # [num_pool_blocks, Hkv, 16, d]
    q: torch.Tensor  # decode [B, Hq, d]; prefill [total_q, Hq, d]
    q_pos: Optional[np.ndarray] = None  # decode: [B]
    cu_seqlens_q: Optional[np.ndarray] = None  # prefill: [B+1]
    q_start: Optional[np.ndarray] = None  # prefill: [B]
    seed: int = 0
    notes: str = ""

    @property
    def num_seqs(self) -> int:
        return len(self.seg_indptr) - 1

    def seq_segments(self, s: int) -> List[Tuple[int, int]]:
        a, b = int(self.seg_indptr[s]), int(self.seg_indptr[s + 1])
        return [(int(self.seg_doc[k]), int(self.seg_len[k])) for k in range(a, b)]

    def blocks_per_seq(self) -> np.ndarray:
        """Logical blocks of each sequence: every segment starts a fresh block."""
        out = np.zeros(self.num_seqs, dtype=np.int64)
        for s in range(self.num_seqs):
            out[s] = sum((L + BLOCK - 1) // BLOCK for _, L in self.seq_segments(s))
        return out

    def tokens_per_seq(self) -> np.ndarray:
        out = np.zeros(self.num_seqs, dtype=np.int64)
        for s in range(self.num_seqs):
            out[s] = sum(L for _, L in self.seq_segments(s))
        return out

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.blocks_per_seq().max()) if self.num_seqs else 0

    def unique_blocks(self) -> int:
        """Distinct (physical block) rows that a full pass reads."""
        used = set()
        for s in range(self.num_seqs):
            for doc, L in self.seq_segments(s):
                a = int(self.doc_block_indptr[doc])
                used.update(int(x) for x in self.doc_blocks[a:a + (L + BLOCK - 1) // BLOCK])
        return len(used)


def finite_zipf_probs(n: int, s: float) -> np.ndarray:
    r = np.arange(1, n + 1, dtype=np.float64)
    w = r ** (-s)
    return w / w.sum()


def _doc_rows(seed: int, doc: int, length: int, hkv: int, d: int) -> Tuple[np.ndarray, np.ndarray]:
    rng = np.random.Generator(np.random.PCG64([seed, 1, doc]))
    k = rng.standard_normal((length, hkv, d), dtype=np.float32)
    v = rng.standard_normal((length, hkv, d), dtype=np.float32)
    return k, v


def _assemble(name: str, kind: str, dtype: str, hq: int, hkv: int, d: int, theta: float,
              seqs: Sequence[Sequence[Tuple[int, int]]], doc_len: Dict[int, int], seed: int,
              pool_cap_blocks: Optional[int] = None, seq_pos0: Optional[Sequence[int]] = None,
              poison: bool = True) -> Dict:
    """Allocate physical blocks for every used document and fill the pools."""
    used_docs = sorted({doc for segs in seqs for doc, _ in segs})
    ndocs = (max(doc_len) + 1) if doc_len else 0
    nblk = {doc: (doc_len[doc] + BLOCK - 1) // BLOCK for doc in used_docs}
    need = sum(nblk.values())
    num_pool_blocks = need if pool_cap_blocks is None else int(pool_cap_blocks)
    if need > num_pool_blocks:
        raise ValueError(f"{name}: {need} blocks needed but the pool holds {num_pool_blocks}")
    rng = np.random.Generator(np.random.PCG64([seed, 2]))
    perm = rng.permutation(num_pool_blocks).astype(np.int32)

    doc_block_indptr = np.zeros(ndocs + 1, dtype=np.int32)
    doc_len_arr = np.zeros(ndocs, dtype=np.int32)
    for doc in range(ndocs):
        doc_len_arr[doc] = doc_len.get(doc, 0)
        doc_block_indptr[doc + 1] = doc_block_indptr[doc] + (nblk.get(doc, 0))
    doc_blocks = perm[:need].copy()

    tdt = _TORCH_DTYPE[dtype]
    fill = float("nan") if poison else 0.0
    k_pool = torch.full((num_pool_blocks, hkv, BLOCK, d), fill, dtype=tdt)
    v_pool = torch.full((num_pool_blocks, hkv, BLOCK, d), fill, dtype=tdt)
    for doc in used_docs:
        L = doc_len[doc]
        k, v = _doc_rows(seed, doc, L, hkv, d)
        nb = nblk[doc]
        ids = torch.from_numpy(doc_blocks[doc_block_indptr[doc]:doc_block_indptr[doc + 1]].astype(np.int64))
        for src, pool in ((k, k_pool), (v, v_pool)):
            t = torch.from_numpy(src).to(tdt)  # round to nearest even
            pad = torch.full((nb * BLOCK, hkv, d), fill, dtype=tdt)
            pad[:L] = t
            pool.index_copy_(0, ids, pad.view(nb, BLOCK, hkv, d).transpose(1, 2).contiguous())

    B = len(seqs)
    seg_indptr = np.zeros(B + 1, dtype=np.int32)
    seg_doc: List[int] = []
    seg_len: List[int] = []
    for s, segs in enumerate(seqs):
        for doc, L in segs:
            if not (1 <= L <= doc_len[doc]):
                raise ValueError(f"{name}: segment uses {L} tokens of doc {doc} (len {doc_len[doc]})")
            seg_doc.append(doc)
            seg_len.append(L)
        seg_indptr[s + 1] = len(seg_doc)
    pos0 = np.zeros(B, dtype=np.int32) if seq_pos0 is None else np.asarray(seq_pos0, dtype=np.int32)
    return dict(name=name, kind=kind, dtype=dtype, num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                rope_theta=float(theta), seg_indptr=seg_indptr, seg_doc=np.asarray(seg_doc, np.int32),
                seg_len=np.asarray(seg_len, np.int32), seq_pos0=pos0, doc_len=doc_len_arr,
                doc_block_indptr=doc_block_indptr, doc_blocks=doc_blocks,
                num_pool_blocks=num_pool_blocks, k_pool=k_pool, v_pool=v_pool, seed=seed)


def _queries(seed: int, rows: int, hq: int, d: int, dtype: str) -> torch.Tensor:
    rng = np.random.Generator(np.random.PCG64([seed, 3]))
    return torch.from_numpy(rng.standard_normal((rows, hq, d), dtype=np.float32)).to(_TORCH_DTYPE[dtype])


def _ctx_len(segs: Sequence[Tuple[int, int]]) -> int:
    return sum(L for _, L in segs)


# --------------------------------------------------------------------------- configs

def tiny_fp32(seed: int = 20260001, shift: int = 0) -> Workload:
    """One sequence, fp32, 4 q heads / 2 KV heads, d=64, theta 1e4; documents of
    48, 32 and 16 tokens at global offsets 0, 48, 80; one query at position 96."""
    doc_len = {0: 48, 1: 32, 2: 16}
    a = _assemble("tiny_fp32", "decode", "f32", 4, 2, 64, 1e4, [[(0, 48), (1, 32), (2, 16)]],
                  doc_len, seed, seq_pos0=[shift])
    q = _queries(seed, 1, 4, 64, "f32")
    return Workload(q=q, q_pos=np.array([96 + shift], np.int32), **a)


def decode_zipf(name: str, *, batch: int, hq: int, hkv: int, d: int = 128, theta: float = 5e5,
                docs_per_seq: int, doc_tokens: int, pool_docs: int, zipf_s: float,
                suffix_tokens: int = 0, dtype: str = "bf16", pool_cap_blocks: Optional[int] = None,
                share: bool = True, seed: int = 20260002, shift: int = 0) -> Workload:
    """Decode batch: each context is ``docs_per_seq`` Zipf-drawn documents of
    ``doc_tokens`` tokens, then an optional private suffix, then one query at the
    end of the context. ``share=False`` gives the no-sharing control: every
    sequence owns distinct documents, so logical bytes equal unique bytes."""
    rng = np.random.Generator(np.random.PCG64([seed, 0]))
    p = finite_zipf_probs(pool_docs, zipf_s)
    doc_len: Dict[int, int] = {}
    seqs = []
    next_private = pool_docs
    for s in range(batch):
        segs = []
        if share:
            for doc in rng.choice(pool_docs, size=docs_per_seq, p=p):
                doc_len[int(doc)] = doc_tokens
                segs.append((int(doc), doc_tokens))
        else:
            for _ in range(docs_per_seq):
                doc_len[next_private] = doc_tokens
                segs.append((next_private, doc_tokens))
                next_private += 1
        if suffix_tokens:
            doc = next_private if not share else pool_docs + s
            next_private = max(next_private, doc + 1)
            doc_len[doc] = suffix_tokens
            segs.append((doc, suffix_tokens))
        seqs.append(segs)
    a = _assemble(name, "decode", dtype, hq, hkv, d, theta, seqs, doc_len, seed,
                  pool_cap_blocks=pool_cap_blocks, seq_pos0=[shift] * batch)
    q_pos = np.array([_ctx_len(sg) + shift for sg in seqs], np.int32)
    return Workload(q=_queries(seed, batch, hq, d, dtype), q_pos=q_pos, **a)


def prefill_zipf(name: str, *, batch: int, hq: int, hkv: int, d: int = 128, theta: float = 5e5,
                 docs_per_seq: int, doc_tokens: int, pool_docs: int, zipf_s: float,
                 chunk_tokens: Sequence[int] | int, dtype: str = "bf16",
                 seed: int = 20260003, shift: int = 0) -> Workload:
    """Prefill batch: Zipf-drawn cached documents at concatenated offsets, then a
    fresh query chunk whose own K/V form the last segment (a private document)."""
    rng = np.random.Generator(np.random.PCG64([seed, 0]))
    p = finite_zipf_probs(pool_docs, zipf_s)
    chunks = [chunk_tokens] * batch if isinstance(chunk_tokens, int) else list(chunk_tokens)
    doc_len: Dict[int, int] = {}
    seqs = []
    for s in range(batch):
        segs = []
        for doc in rng.choice(pool_docs, size=docs_per_seq, p=p):
            doc_len[int(doc)] = doc_tokens
            segs.append((int(doc), doc_tokens))
        if chunks[s] > 0:
            doc_len[pool_docs + s] = chunks[s]
            segs.append((pool_docs + s, chunks[s]))
        seqs.append(segs)
    a = _assemble(name, "prefill", dtype, hq, hkv, d, theta, seqs, doc_len, seed,
                  seq_pos0=[shift] * batch)
    cu = np.zeros(batch + 1, np.int32)
    cu[1:] = np.cumsum(chunks)
    q_start = np.array([_ctx_len(sg) - c + shift for sg, c in zip(seqs, chunks)], np.int32)
    return Workload(q=_queries(seed, int(cu[-1]), hq, d, dtype), cu_seqlens_q=cu, q_start=q_start, **a)


def _fill_context(rng: np.random.Generator, target: int, p: np.ndarray, doc_len: Dict[int, int],
                  lens: np.ndarray) -> List[Tuple[int, int]]:
    segs, total = [], 0
    while total < target:
        doc = int(rng.choice(len(p), p=p))
        L = int(lens[doc])
        use = min(L, target - total)
        doc_len[doc] = L
        segs.append((doc, use))
        total += use
    return segs


def mixed_mqa(*, n_decode: int = 48, n_prefill: int = 4, chunk: int = 512, hq: int = 32, hkv: int = 1,
              d: int = 128, theta: float = 5e5, pool_docs: int = 1024, zipf_s: float = 0.8,
              ctx_lo: int = 256, ctx_hi: int = 131072, doc_lo: int = 64, doc_hi: int = 4096,
              seed: int = 20260005, dtype: str = "bf16") -> Tuple[Workload, Workload]:
    """Mixed continuous batch, MQA: decode contexts ~ U[ctx_lo, ctx_hi] built from
    documents of length ~ U[doc_lo, doc_hi] (fixed per document) drawn Zipf from a
    ``pool_docs`` pool, the last document cut to a prefix; plus ``n_prefill`` chunks
    of ``chunk`` tokens over contexts drawn the same way. Both halves share one
    physical pool. Returns (decode, prefill) workloads."""
    rng = np.random.Generator(np.random.PCG64([seed, 0]))
    lens = rng.integers(doc_lo, doc_hi + 1, size=pool_docs)
    p = finite_zipf_probs(pool_docs, zipf_s)
    doc_len: Dict[int, int] = {}
    dec = [_fill_context(rng, int(rng.integers(ctx_lo, ctx_hi + 1)), p, doc_len, lens) for _ in range(n_decode)]
    pre = []
    for i in range(n_prefill):
        segs = _fill_context(rng, int(rng.integers(ctx_lo, ctx_hi - chunk + 1)), p, doc_len, lens)
        doc_len[pool_docs + i] = chunk
        segs.append((pool_docs + i, chunk))
        pre.append(segs)
    a = _assemble("mixed_mqa", "decode", dtype, hq, hkv, d, theta, dec + pre, doc_len, seed)
    pool_k, pool_v = a.pop("k_pool"), a.pop("v_pool")
    seg_indptr, seg_doc, seg_len = a.pop("seg_indptr"), a.pop("seg_doc"), a.pop("seg_len")
    a.pop("seq_pos0"), a.pop("name"), a.pop("kind")

    def sub(lo, hi):
        base = int(seg_indptr[lo])
        ind = (seg_indptr[lo:hi + 1] - base).astype(np.int32)
        return ind, seg_doc[base:int(seg_indptr[hi])].copy(), seg_len[base:int(seg_indptr[hi])].copy()

    di, dd, dl = sub(0, n_decode)
    wd = Workload(name="mixed_mqa.decode", kind="decode", seg_indptr=di, seg_doc=dd, seg_len=dl,
                  seq_pos0=np.zeros(n_decode, np.int32), k_pool=pool_k, v_pool=pool_v,
                  q=_queries(seed, n_decode, hq, d, dtype),
                  q_pos=np.array([_ctx_len(s) for s in dec], np.int32), **a)
    pi, pd, pl = sub(n_decode, n_decode + n_prefill)
    cu = np.arange(n_prefill + 1, dtype=np.int32) * chunk
    wp = Workload(name="mixed_mqa.prefill", kind="prefill", seg_indptr=pi, seg_doc=pd, seg_len=pl,
                  seq_pos0=np.zeros(n_prefill, np.int32), k_pool=pool_k, v_pool=pool_v,
                  q=_queries(seed + 100, n_prefill * chunk, hq, d, dtype), cu_seqlens_q=cu,
                  q_start=np.array([_ctx_len(s) - chunk for s in pre], np.int32), **a)
    return wd, wp


def cache_trace(*, num_requests: int, pool_docs: int, docs_per_request: int, zipf_s: float,
                doc_tokens: Tuple[int, int] = (256, 1024), prompt_tokens: int = 0,
                seed: int = 20260007) -> Tuple[List[List[Tuple[int, int]]], List[int]]:
    """Request trace for the cache-policy simulator, RAG-shaped: every request
    retrieves ``docs_per_request`` distinct documents drawn by finite Zipf(s) over
    ``pool_docs`` (placed in draw order, i.e. retrieval rank), each at its own
    fixed length drawn once uniformly in ``doc_tokens`` (inclusive), after a
    shared prompt of ``prompt_tokens`` tokens. Returns (requests as lists of
    (doc, len) segments, pos0 of each request)."""
    rng = np.random.Generator(np.random.PCG64([seed, 7]))
    p = finite_zipf_probs(pool_docs, zipf_s)
    lens = rng.integers(doc_tokens[0], doc_tokens[1] + 1, size=pool_docs)
    reqs = []
    for _ in range(num_requests):
        docs = rng.choice(pool_docs, size=docs_per_request, replace=False, p=p)
        reqs.append([(int(d), int(lens[d])) for d in docs])
    return reqs, [int(prompt_tokens)] * num_requests


# Full-size workloads, by name. Each is a zero-argument constructor.
FULL = {
    "tiny_fp32": lambda: tiny_fp32(),
    "llama8b_decode": lambda: decode_zipf("llama8b_decode", batch=64, hq=32, hkv=8, docs_per_seq=8,
                                          doc_tokens=512, pool_docs=256, zipf_s=1.0, suffix_tokens=64,
                                          seed=20260002),
    "llama8b_decode_noshare": lambda: decode_zipf("llama8b_decode_noshare", batch=64, hq=32, hkv=8,
                                                  docs_per_seq=8, doc_tokens=512, pool_docs=256,
                                                  zipf_s=1.0, suffix_tokens=64, share=False,
                                                  seed=20260002),
    "llama8b_prefill": lambda: prefill_zipf("llama8b_prefill", batch=8, hq=32, hkv=8, docs_per_seq=6,
                                            doc_tokens=1024, pool_docs=128, zipf_s=1.2, chunk_tokens=256,
                                            seed=20260003),
    "llama70b_decode": lambda: decode_zipf("llama70b_decode", batch=32, hq=64, hkv=8, docs_per_seq=16,
                                           doc_tokens=1024, pool_docs=512, zipf_s=1.0,
                                           pool_cap_blocks=16384, seed=20260004),
    "llama70b_decode_noshare": lambda: decode_zipf("llama70b_decode_noshare", batch=32, hq=64, hkv=8,
                                                   docs_per_seq=16, doc_tokens=1024, pool_docs=512,
                                                   zipf_s=1.0, share=False, seed=20260004),
    # the two halves of the mixed continuous batch (one shared pool), each on its own
    "mixed_mqa_decode": lambda: mixed_mqa()[0],
    "mixed_mqa_prefill": lambda: mixed_mqa()[1],
}


def kv_bytes_logical(w: Workload) -> int:
    """K+V bytes a full pass reads if every logical token is fetched once."""
    elt = 4 if w.dtype == "f32" else 2
    return int(w.tokens_per_seq().sum()) * w.num_kv_heads * w.head_dim * 2 * elt


def kv_bytes_blocks(w: Workload) -> int:
    """K+V bytes of every logical block (16-token granularity, what the kernels fetch)."""
    elt = 4 if w.dtype == "f32" else 2
    return int(w.blocks_per_seq().sum()) * BLOCK * w.num_kv_heads * w.head_dim * 2 * elt


def kv_bytes_unique(w: Workload) -> int:
    """K+V bytes of the distinct physical blocks touched: the lower bound on DRAM reads."""
    elt = 4 if w.dtype == "f32" else 2
    return w.unique_blocks() * BLOCK * w.num_kv_heads * w.head_dim * 2 * elt


def fp8_pools(w: Workload):
    """e4m3 copies of a workload's pools for the FP8-KV decode: per-tensor scales
    amax / 448 (the largest e4m3 value; amax over the finite entries, hole slots keep
    their non-finite filler as NaN codes), codes = round-to-nearest-even of x / scale.
    Returns (k_codes, v_codes, k_scale, v_scale); codes are torch.float8_e4m3fn."""
    out = []
    for pool in (w.k_pool, w.v_pool):
        x = pool.float()
        fin = x[torch.isfinite(x)]
        scale = (float(fin.abs().max()) / 448.0 if fin.numel() else 0.0) or 1.0
        out.append(((x / scale).to(torch.float8_e4m3fn), scale))
    return out[0][0], out[1][0], out[0][1], out[1][1]
