"""GPU parity of the packer, the block gather and the decode kernels against the
CPU oracle (all calls go through the C ABI of liblazyattn.so)."""
import numpy as np
import pytest
import torch

import oracle
from brute import rope
from bf16_model import emulate
from gpu_util import FEW_KEY_FALLBACK_FRAC, assert_close, decode, la, to_device
from paged_kv_cache_57_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _clean_status():
    la().device_status(clear=True)
    yield
    assert la().device_status(clear=True) == 0, "device status word set"


# ---------------------------------------------------------------- rotation table

@pytest.mark.parametrize("d,theta", [(64, 1e4), (128, 5e5)])
def test_rotation_matches_fp64(d, theta):
    # cos/sin of n * w_i as the kernels evaluate them, against numpy fp64.
    L = la()
    p = L.make_params(num_seqs=1, num_q_heads=1, num_kv_heads=1, head_dim=d, num_pool_blocks=1,
                      max_blocks_per_seq=1, rope_theta=theta)
    table = L.rope_table_init(p)
    full = table.view(torch.float32).view(-1, 2).cpu().double().numpy()
    t = full[: d // 2]
    w = theta ** (-2.0 * np.arange(d // 2) / d)
    assert np.abs((t[:, 0] + t[:, 1]) * 2 * np.pi / w - 1).max() < 1e-14
    # Row part: (cos, sin)(i * w_f) for the prefill row offsets i < LAZY_ROPE_ROWS, rounded once.
    rows = full[d // 2:].reshape(128, d // 2, 2)
    ang_r = np.arange(128)[:, None] * w[None, :]
    assert np.abs(rows[..., 0] - np.cos(ang_r)).max() < 6e-8
    assert np.abs(rows[..., 1] - np.sin(ang_r)).max() < 6e-8
    rng = np.random.default_rng(9)
    deltas = np.concatenate([np.arange(-5, 300), rng.integers(-(1 << 24) + 1, 1 << 24, 3000),
                             [131072, 131071, 4160, 16384, (1 << 24) - 1, -(1 << 24) + 1]]).astype(np.int32)
    cs = L.debug_rope(p, table, torch.from_numpy(deltas).cuda()).cpu().double().numpy()
    ang = deltas[:, None].astype(np.float64) * w[None, :]
    err = max(np.abs(cs[..., 0] - np.cos(ang)).max(), np.abs(cs[..., 1] - np.sin(ang)).max())
    assert err < 1e-6, err


# ---------------------------------------------------------------- packer and gather

def _layout_workloads():
    yield W.tiny_fp32()
    yield W.tiny_fp32(shift=1234)
    yield W.decode_zipf("dz", batch=7, hq=8, hkv=2, d=128, docs_per_seq=5, doc_tokens=48, pool_docs=9,
                        zipf_s=1.0, suffix_tokens=23, seed=41)
    d, p = W.mixed_mqa(n_decode=9, n_prefill=3, chunk=50, hq=8, hkv=1, d=128, pool_docs=60, ctx_lo=40,
                       ctx_hi=5000, doc_lo=5, doc_hi=400, seed=42)
    yield d
    yield p
    # 40+ segments per sequence: exercises the packer's 32-segment chunking
    d2, _ = W.mixed_mqa(n_decode=3, n_prefill=1, chunk=16, hq=2, hkv=1, d=64, pool_docs=200, ctx_lo=2000,
                        ctx_hi=3000, doc_lo=5, doc_hi=60, seed=43)
    yield d2


@pytest.mark.parametrize("w", list(_layout_workloads()), ids=lambda w: w.name)
def test_device_packer_equals_host_packer(w):
    L = la()
    dv = to_device(w, pack_on_device=True)
    wh, sh = L.pack_block_words_host(dv.p, len(w.doc_len), w.seg_indptr, w.seg_doc, w.seg_len, w.seq_pos0,
                                     w.doc_block_indptr, w.doc_blocks)
    assert np.array_equal(dv.words.cpu().numpy().view(np.uint32), wh)
    assert np.array_equal(dv.seq_lens.cpu().numpy(), sh)


def test_device_packer_flags_bad_layout():
    L = la()
    w = W.decode_zipf("bad", batch=3, hq=4, hkv=2, d=64, docs_per_seq=2, doc_tokens=20, pool_docs=3,
                      zipf_s=1.0, seed=44)
    w.seg_len[w.seg_indptr[1]] = 999  # sequence 1: segment longer than its document
    dv = to_device(w, pack_on_device=True)
    assert L.device_status(clear=True) & L.LAZY_DEV_LAYOUT
    sl = dv.seq_lens.cpu().numpy()
    assert sl[1] == 0 and sl[0] > 0 and sl[2] > 0
    assert (dv.words.cpu().numpy()[1] == 0).all()


def host_gather(w, s, h):
    rows_k, rows_v, pos = {}, {}, {}
    b0, p = 0, int(w.seq_pos0[s])
    kp, vp = w.k_pool, w.v_pool
    for doc, Ln in w.seq_segments(s):
        base = int(w.doc_block_indptr[doc])
        for j in range(Ln):
            phys = int(w.doc_blocks[base + j // 16])
            r = 16 * (b0 + j // 16) + j % 16
            rows_k[r], rows_v[r], pos[r] = kp[phys, h, j % 16], vp[phys, h, j % 16], p
        b0 += (Ln + 15) // 16
        p += Ln
    return rows_k, rows_v, pos


@pytest.mark.parametrize("w", list(_layout_workloads()), ids=lambda w: w.name)
def test_gather_is_bit_exact(w):
    L = la()
    dv = to_device(w)
    ko, vo, po = L.debug_gather(dv.p, dv.k_pool, dv.v_pool, dv.words, dv.seq_lens)
    ko, vo, po = ko.cpu(), vo.cpu(), po.cpu().numpy()
    as_bits = (lambda t: t.view(torch.int16)) if w.dtype == "bf16" else (lambda t: t.view(torch.int32))
    for s in range(w.num_seqs):
        for h in range(w.num_kv_heads):
            rk, rv, rp = host_gather(w, s, h)
            rows = np.array(sorted(rk), dtype=np.int64)
            if len(rows):
                assert torch.equal(as_bits(ko[s, h, rows]), as_bits(torch.stack([rk[r] for r in rows])))
                assert torch.equal(as_bits(vo[s, h, rows]), as_bits(torch.stack([rv[r] for r in rows])))
            holes = np.setdiff1d(np.arange(ko.shape[2]), rows)
            assert (ko[s, h, holes] == 0).all() and (vo[s, h, holes] == 0).all()
            if h == 0:
                assert all(po[s, r] == rp[r] for r in rows)
                assert (po[s, holes] == -1).all()


# ---------------------------------------------------------------- decode parity

def _check_decode(w, rows=None, num_splits=0, lazy=True, fallback_frac=0.0):
    dv = to_device(w, num_splits=num_splits, lazy=lazy)
    out = decode(dv)
    ref = oracle.attention(w, rows=rows)
    got = out if rows is None else out[torch.as_tensor(rows, device=out.device)]
    sel = np.arange(ref.shape[0]) if rows is None else np.asarray(rows)
    emu = (lambda r: emulate(w, sel[r], lazy=lazy)) if w.dtype == "bf16" else None
    return assert_close(got, ref, w.dtype, w.name, emulate=emu, fallback_frac=fallback_frac)


def test_two_and_three_key_contexts():
    w = W.decode_zipf("fewkeys", batch=6, hq=8, hkv=2, d=128, docs_per_seq=1, doc_tokens=3, pool_docs=6,
                      zipf_s=1.0, seed=69)
    w.seg_len[:] = np.array([2, 3, 2, 3, 1, 2], np.int32)
    # few-key edge case: the bf16 rounding of q' and of two or three O(1) weights can
    # exceed 2e-3 where the values cancel (capped, see gpu_util.assert_close)
    _check_decode(w, fallback_frac=FEW_KEY_FALLBACK_FRAC)


def test_tiny_fp32_decode():
    _check_decode(W.tiny_fp32())


@pytest.mark.parametrize("splits", [1, 2, 3, 6])
def test_tiny_fp32_decode_splits(splits):
    _check_decode(W.tiny_fp32(), num_splits=splits)


@pytest.mark.parametrize("hq,hkv", [(4, 4), (8, 2), (16, 2), (32, 1), (64, 8), (64, 1)])
@pytest.mark.parametrize("d", [64, 128])
def test_bf16_decode_gqa_shapes(hq, hkv, d):
    w = W.decode_zipf(f"gqa{hq}x{hkv}d{d}", batch=5, hq=hq, hkv=hkv, d=d, docs_per_seq=4, doc_tokens=80,
                      pool_docs=6, zipf_s=1.0, suffix_tokens=16, seed=50 + hq + d)
    _check_decode(w)


@pytest.mark.parametrize("splits", [1, 2, 7, 64])
def test_bf16_decode_split_sweep(splits):
    w = W.decode_zipf("splits", batch=3, hq=32, hkv=8, d=128, docs_per_seq=8, doc_tokens=96, pool_docs=10,
                      zipf_s=1.0, suffix_tokens=16, seed=61)
    _check_decode(w, num_splits=splits)


def test_fp32_decode_long_context():
    # offsets up to ~100k exercise the rotation far from the document start (fp32: 1e-5)
    w = W.decode_zipf("f32long", batch=1, hq=4, hkv=1, d=128, theta=5e5, docs_per_seq=24, doc_tokens=4096,
                      pool_docs=24, zipf_s=0.0, dtype="f32", seed=68)
    _check_decode(w)


def test_fp32_decode_gqa():
    w = W.decode_zipf("f32gqa", batch=4, hq=16, hkv=2, d=128, theta=5e5, docs_per_seq=3, doc_tokens=70,
                      pool_docs=5, zipf_s=1.0, suffix_tokens=5, dtype="f32", seed=62)
    _check_decode(w)
    _check_decode(w, num_splits=3)


def test_mixed_holes_and_partial_blocks():
    d, _ = W.mixed_mqa(n_decode=10, n_prefill=1, chunk=16, hq=32, hkv=1, d=128, pool_docs=80, ctx_lo=100,
                       ctx_hi=6000, doc_lo=5, doc_hi=500, seed=63)
    _check_decode(d)
    _check_decode(d, num_splits=5)


def test_empty_and_one_key_sequences():
    w = W.decode_zipf("onekey", batch=3, hq=8, hkv=2, d=128, docs_per_seq=1, doc_tokens=1, pool_docs=3,
                      zipf_s=1.0, seed=64)
    w.seg_indptr = np.array([0, 1, 1, 2], np.int32)  # sequence 1 is empty
    w.seg_doc, w.seg_len = w.seg_doc[:2].copy(), w.seg_len[:2].copy()
    dv = to_device(w)
    out = decode(dv).cpu()
    assert (out[1] == 0).all()
    vp = w.v_pool
    for s, k in ((0, 0), (2, 1)):
        phys = int(w.doc_blocks[w.doc_block_indptr[w.seg_doc[k]]])
        for h in range(8):
            assert torch.equal(out[s, h], vp[phys, h // 4, 0])  # one key: output is v, exactly


def test_shift_invariance_is_bitwise():
    kw = dict(batch=4, hq=32, hkv=8, d=128, docs_per_seq=3, doc_tokens=64, pool_docs=5, zipf_s=1.0,
              suffix_tokens=7, seed=65)
    a = decode(to_device(W.decode_zipf("s0", **kw))).cpu()
    for c in (1, 16, 4000):
        b = decode(to_device(W.decode_zipf("sc", shift=c, **kw))).cpu()
        assert torch.equal(a.view(torch.int16), b.view(torch.int16)), c


def test_lazy0_control_on_materialised_pool():
    # Control path: a pool holding each sequence's keys already rotated to their
    # absolute positions (no sharing), read without per-document rotation.
    w = W.decode_zipf("ctl", batch=4, hq=16, hkv=4, d=128, docs_per_seq=3, doc_tokens=48, pool_docs=4,
                      zipf_s=1.0, suffix_tokens=8, share=False, seed=66)
    kabs = w.k_pool.double().clone()
    for s in range(w.num_seqs):
        p = 0
        for doc, Ln in w.seq_segments(s):
            ids = w.doc_blocks[w.doc_block_indptr[doc]:w.doc_block_indptr[doc + 1]]
            for phys in ids:
                kabs[phys] = torch.from_numpy(rope(kabs[phys].numpy(), p, w.rope_theta))
            p += Ln
    dv = to_device(w, lazy=False, k_pool=kabs.to(torch.bfloat16))
    ref = oracle.attention(w)
    assert_close(decode(dv), ref, "bf16", "lazy=0 control")


def test_bad_block_id_sets_status_and_does_not_fault():
    L = la()
    w = W.decode_zipf("badid", batch=2, hq=8, hkv=2, d=128, docs_per_seq=2, doc_tokens=32, pool_docs=3,
                      zipf_s=1.0, seed=67)
    dv = to_device(w)
    words = dv.words.cpu().numpy().view(np.uint32).copy()
    words[0, 1] = (words[0, 1] & ~np.uint32((1 << 18) - 1)) | np.uint32((1 << 18) - 1)  # id past the pool
    dv.words = torch.from_numpy(words.view(np.int32)).cuda()
    out = decode(dv)
    torch.cuda.synchronize()
    assert L.device_status(clear=True) & L.LAZY_DEV_BAD_BLOCK_ID
    assert torch.isfinite(out.float()).all()


# ---------------------------------------------------------------- full sizes (sampled)

def test_llama8b_decode_full():
    _check_decode(W.FULL["llama8b_decode"]())


def test_llama70b_decode_full_sampled():
    w = W.FULL["llama70b_decode"]()
    _check_decode(w, rows=[0, 7, 13, 31])


def test_mixed_decode_full_sampled():
    d, _ = W.mixed_mqa()
    rng = np.random.default_rng(5)
    _check_decode(d, rows=sorted(rng.choice(d.num_seqs, 6, replace=False).tolist()))


# ---------------------------------------------------------------- softmax scale other than 1/sqrt(d)

@pytest.mark.parametrize("scale", [0.05, 0.15])
def test_non_default_sm_scale(scale):
    # 0.05 flattens the softmax; 0.15 (1.7 x 1/sqrt(d)) sharpens it, so that a few keys
    # carry most of a row's weight: the sharp-softmax edge case, where the bf16
    # rounding of q' and P can exceed 2e-3 (capped, see gpu_util.assert_close)
    from gpu_util import decode_shared, shared_plan
    w = W.decode_zipf("scale", batch=5, hq=32, hkv=8, d=128, docs_per_seq=3, doc_tokens=90, pool_docs=4,
                      zipf_s=1.0, suffix_tokens=11, seed=70)
    dv = to_device(w)
    dv.p.sm_scale = scale
    ref = oracle.attention(w, sm_scale=scale)
    emu = lambda r: emulate(w, r, sm_scale=scale)
    frac = FEW_KEY_FALLBACK_FRAC if scale > 0.1 else 0.0
    assert_close(decode(dv), ref, "bf16", f"per-sequence decode, sm_scale {scale}", emulate=emu,
                 fallback_frac=frac)
    assert_close(decode_shared(dv, shared_plan(dv)), ref, "bf16", f"shared-run decode, sm_scale {scale}",
                 emulate=emu, fallback_frac=frac)
    # the scale matters here
    assert np.abs(ref - oracle.attention(w)).max() > 1e-2


def test_non_default_sm_scale_fp32():
    w = W.tiny_fp32()
    dv = to_device(w)
    dv.p.sm_scale = 0.3
    assert_close(decode(dv), oracle.attention(w, sm_scale=0.3), "f32", "fp32 decode, sm_scale 0.3")
