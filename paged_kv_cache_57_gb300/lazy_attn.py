"""Python binding of the LazyAttention C ABI (``include/lazy_attn.h``).

Argument marshalling only: every function here checks shapes and dtypes of
torch tensors, then passes raw pointers, sizes and the current CUDA stream to
``liblazyattn.so``. All computation happens in the library's CUDA kernels (or,
for ``pack_block_words_host``, in its C++ host code). Importing this module
raises if the library has not been built: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "liblazyattn.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build it with `python -m paged_kv_cache_57_gb300.build`")
_lib = ctypes.CDLL(LIB_PATH)

LAZY_OK, LAZY_ERR_INVALID_ARG, LAZY_ERR_UNSUPPORTED, LAZY_ERR_WORKSPACE, LAZY_ERR_LAYOUT, LAZY_ERR_CUDA, \
    LAZY_ERR_DEVICE = range(7)
LAZY_F32, LAZY_BF16, LAZY_FP8_E4M3 = 0, 1, 2
LAZY_DEV_BAD_BLOCK_ID, LAZY_DEV_POS_RANGE, LAZY_DEV_TIMEOUT, LAZY_DEV_LAYOUT, LAZY_DEV_BAD_LEN = 1, 2, 4, 8, 16
BLOCK = 16

EXPORTED = (
    "lazy_attn_status_string", "lazy_attn_rope_table_bytes", "lazy_attn_rope_table_init",
    "lazy_attn_pack_block_words_host", "lazy_attn_pack_block_words", "lazy_attn_decode_workspace_bytes",
    "lazy_attn_decode", "lazy_attn_prefill_workspace_bytes", "lazy_attn_prefill", "lazy_attn_debug_gather",
    "lazy_attn_device_status", "lazy_attn_launch_count", "lazy_attn_debug_rope", "lazy_attn_decode_noalloc",
    "lazy_attn_plan_shared_host", "lazy_attn_decode_shared_workspace_bytes", "lazy_attn_decode_shared",
    "lazy_attn_materialize", "lazy_attn_rope_table_init_scaled", "lazy_attn_rope_table_init_freqs",
    "lazy_attn_rotary_layout_host", "lazy_attn_decode_shared_alibi", "lazy_attn_alibi_slopes_host",
    "lazy_attn_decode_alibi", "lazy_attn_debug_gather_withheld", "lazy_attn_prefill_alibi",
    "lazy_attn_decode_shared_partials", "lazy_attn_decode_shared_combine", "lazy_attn_mixed_workspace_bytes",
    "lazy_attn_mixed",
)
PLAN_MAX_MEMBERS = 16
PLAN_ITEM_BLOCK_IDS = 32
PLAN_ITEM_INTS = 8 + 4 * PLAN_MAX_MEMBERS + PLAN_ITEM_BLOCK_IDS
NOALLOC_SCRATCH_BYTES = 8 << 20


class Params(ctypes.Structure):
    """Mirror of ``lazy_attn_params``."""
    _fields_ = [
        ("num_seqs", ctypes.c_int32), ("num_q_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32), ("block_size", ctypes.c_int32), ("num_pool_blocks", ctypes.c_int32),
        ("max_blocks_per_seq", ctypes.c_int32), ("id_bits", ctypes.c_int32), ("dtype", ctypes.c_int32),
        ("lazy", ctypes.c_int32), ("rope_theta", ctypes.c_double), ("sm_scale", ctypes.c_float),
        ("num_splits", ctypes.c_int32), ("key_positions", ctypes.c_int32), ("kv_dtype", ctypes.c_int32),
        ("k_scale", ctypes.c_float), ("v_scale", ctypes.c_float),
    ]


class LazyAttnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)}")


_vp, _sz, _i32, _u64 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int32, ctypes.c_uint64
_P = ctypes.POINTER(Params)
_sig = {
    "lazy_attn_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "lazy_attn_rope_table_bytes": (_sz, [_P]),
    "lazy_attn_rope_table_init": (ctypes.c_int, [_P, _vp, _sz, _vp]),
    "lazy_attn_rope_table_init_scaled": (ctypes.c_int, [_P, _vp, _vp, _sz, _vp]),
    "lazy_attn_rope_table_init_freqs": (ctypes.c_int, [_P, _vp, _vp, _sz, _vp]),
    "lazy_attn_rotary_layout_host": (ctypes.c_int, [_i32, _i32, _i32, ctypes.c_double, _vp, _vp]),
    "lazy_attn_pack_block_words_host": (ctypes.c_int, [_P, _i32] + [_vp] * 8),
    "lazy_attn_pack_block_words": (ctypes.c_int, [_P, _i32] + [_vp] * 8 + [_vp]),
    "lazy_attn_decode_workspace_bytes": (_sz, [_P]),
    "lazy_attn_decode": (ctypes.c_int, [_P] + [_vp] * 9 + [_sz, _vp]),
    "lazy_attn_prefill_workspace_bytes": (_sz, [_P, _i32]),
    "lazy_attn_prefill": (ctypes.c_int, [_P, _vp, _vp, _vp, _i32, _i32] + [_vp] * 7 + [_sz, _vp]),
    "lazy_attn_prefill_alibi": (ctypes.c_int, [_P, _vp, _vp, _vp, _i32, _i32] + [_vp] * 8 + [_sz, _vp]),
    "lazy_attn_debug_gather": (ctypes.c_int, [_P] + [_vp] * 7 + [_vp]),
    "lazy_attn_debug_gather_withheld": (ctypes.c_int, [_P] + [_vp] * 7 + [_i32, ctypes.c_uint32, _vp]),
    "lazy_attn_device_status": (ctypes.c_int, [ctypes.POINTER(ctypes.c_uint32), ctypes.c_int]),
    "lazy_attn_launch_count": (_u64, []),
    "lazy_attn_debug_rope": (ctypes.c_int, [_P, _vp, _vp, _i32, _vp, _vp]),
    "lazy_attn_decode_noalloc": (ctypes.c_int, [_P] + [_vp] * 8 + [_vp]),
    "lazy_attn_plan_shared_host": (ctypes.c_int, [_P, _i32] + [_vp] * 5 + [_i32, _i32] + [_vp] * 3),
    "lazy_attn_decode_shared_workspace_bytes": (_sz, [_P, _i32]),
    "lazy_attn_materialize": (ctypes.c_int, [_P] + [_vp] * 8 + [_vp]),
    "lazy_attn_decode_shared": (ctypes.c_int, [_P] + [_vp] * 6 + [_i32, _vp, _i32, _vp, _vp, _vp, _sz, _vp]),
    "lazy_attn_decode_shared_alibi": (ctypes.c_int,
                                      [_P] + [_vp] * 6 + [_i32, _vp, _i32, _vp, _vp, _vp, _vp, _sz, _vp]),
    "lazy_attn_alibi_slopes_host": (ctypes.c_int, [_i32, _vp]),
    "lazy_attn_decode_shared_partials": (ctypes.c_int, [_P] + [_vp] * 6 + [_i32, _vp, _i32, _vp, _sz, _vp]),
    "lazy_attn_decode_shared_combine": (ctypes.c_int, [_P, _i32, _vp, _vp, _sz, _vp, _vp]),
    "lazy_attn_mixed_workspace_bytes": (_sz, [_P, _P, _i32]),
    "lazy_attn_mixed": (ctypes.c_int, [_P] + [_vp] * 3 + [_i32, _vp, _i32, _vp, _vp, _P] + [_vp] * 3 +
                        [_i32, _i32] + [_vp] * 6 + [_sz, _vp]),
    "lazy_attn_decode_alibi": (ctypes.c_int, [_P] + [_vp] * 9 + [_vp, _sz, _vp]),
}
for _name, (_res, _args) in _sig.items():
    _f = getattr(_lib, _name)
    _f.restype, _f.argtypes = _res, _args


def status_string(status: int) -> str:
    return _lib.lazy_attn_status_string(int(status)).decode()


def _check(rc: int, where: str) -> None:
    if rc != LAZY_OK:
        raise LazyAttnError(rc, where)


def make_params(*, num_seqs: int, num_q_heads: int, num_kv_heads: int, head_dim: int, num_pool_blocks: int,
                max_blocks_per_seq: int, dtype: str = "bf16", rope_theta: float = 5e5, lazy: bool = True,
                sm_scale: float = 0.0, id_bits: int = 0, num_splits: int = 0, key_positions: bool = False,
                kv_dtype: Optional[str] = None, k_scale: float = 0.0, v_scale: float = 0.0) -> Params:
    """kv_dtype "fp8_e4m3": pools of e4m3 codes (torch.float8_e4m3fn), values code * k_scale / v_scale."""
    kv = 0 if kv_dtype is None else {"fp8_e4m3": LAZY_FP8_E4M3}[kv_dtype]
    return Params(num_seqs, num_q_heads, num_kv_heads, head_dim, BLOCK, num_pool_blocks, max_blocks_per_seq,
                  id_bits, LAZY_BF16 if dtype == "bf16" else LAZY_F32, int(bool(lazy)), float(rope_theta),
                  float(sm_scale), num_splits, int(bool(key_positions)), kv, float(k_scale), float(v_scale))


def _dptr(t: Optional[torch.Tensor], name: str, dtype=None, device_required=True):
    if t is None:
        return None
    if device_required and not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _tdt(p: Params):
    return torch.bfloat16 if p.dtype == LAZY_BF16 else torch.float32


def _kvdt(p: Params):
    """torch dtype of the pools."""
    return torch.float8_e4m3fn if p.kv_dtype == LAZY_FP8_E4M3 else _tdt(p)


# ---------------------------------------------------------------- rotation table

def rope_table_bytes(p: Params) -> int:
    return int(_lib.lazy_attn_rope_table_bytes(ctypes.byref(p)))


class RopeScaling(ctypes.Structure):
    """Llama-3.1 frequency scaling (lazy_rope_scaling)."""
    _fields_ = [("factor", ctypes.c_double), ("low_freq_factor", ctypes.c_double),
                ("high_freq_factor", ctypes.c_double), ("original_max_position", ctypes.c_int32)]


def rope_table_init(p: Params, table: Optional[torch.Tensor] = None, stream=None,
                    scaling: Optional[RopeScaling] = None, freqs: Optional[np.ndarray] = None) -> torch.Tensor:
    """Rotation table from theta (default), the Llama-3.1 scaling, or explicit rates
    ``freqs`` [head_dim/2] in radians per position (see rotary_layout)."""
    n = rope_table_bytes(p)
    if n == 0:
        raise LazyAttnError(LAZY_ERR_INVALID_ARG, "rope_table_bytes")
    if table is None:
        table = torch.empty(n, dtype=torch.uint8, device="cuda")
    nbytes = table.numel() * table.element_size()
    if freqs is not None:
        f = np.ascontiguousarray(freqs, dtype=np.float64)
        if f.shape != (p.head_dim // 2,):
            raise ValueError(f"freqs must have shape ({p.head_dim // 2},)")
        rc = _lib.lazy_attn_rope_table_init_freqs(ctypes.byref(p), f.ctypes.data, _dptr(table, "table"), nbytes,
                                                  _stream(stream))
    elif scaling is None:
        rc = _lib.lazy_attn_rope_table_init(ctypes.byref(p), _dptr(table, "table"), nbytes, _stream(stream))
    else:
        rc = _lib.lazy_attn_rope_table_init_scaled(ctypes.byref(p), ctypes.addressof(scaling), _dptr(table, "table"),
                                                   nbytes, _stream(stream))
    _check(rc, "rope_table_init")
    return table


def rotary_layout(d: int, rot_dims: int, theta: float, interleaved: bool = False):
    """(perm [d], freqs [d/2]) of lazy_attn_rotary_layout_host: permute q and the stored
    K rows by ``perm`` and build the table with ``freqs`` to rotate only the first
    ``rot_dims`` dims (partial rotary), rotate-half or interleaved."""
    perm = np.empty(d, np.int32)
    freqs = np.empty(d // 2, np.float64)
    _check(_lib.lazy_attn_rotary_layout_host(int(d), int(rot_dims), int(bool(interleaved)), float(theta),
                                             perm.ctypes.data, freqs.ctypes.data), "rotary_layout")
    return perm.astype(np.int64), freqs


def interleave_perm(d: int) -> np.ndarray:
    """Head-dimension order [0, 2, ..., d-2, 1, 3, ..., d-1]: q and stored K permuted this
    way make the interleaved (GPT-J) pairing (2f, 2f+1) the library's (f, f + d/2)."""
    return np.concatenate([np.arange(0, d, 2), np.arange(1, d, 2)])


# ---------------------------------------------------------------- packer

def _i32_np(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a), dtype=np.int32)


def pack_block_words_host(p: Params, num_docs: int, seg_indptr, seg_doc, seg_len, seq_pos0, doc_block_indptr,
                          doc_blocks, out=None):
    """Host packer; arrays are numpy-compatible. Returns (words [B, max_blocks] uint32, seq_lens [B] int32),
    written into ``out`` = (words, seq_lens) when given (caller buffers, e.g. pinned host memory)."""
    B, MB = p.num_seqs, p.max_blocks_per_seq
    if out is None:
        words = np.zeros((B, MB), dtype=np.uint32)
        seq_lens = np.zeros(B, dtype=np.int32)
    else:
        words, seq_lens = out
    # None stays NULL; an empty array is passed as a valid (never read) one-element buffer.
    arrs = [None if x is None else (_i32_np(x) if np.size(x) else np.zeros(1, np.int32))
            for x in (seg_indptr, seg_doc, seg_len, seq_pos0, doc_block_indptr, doc_blocks)]
    ptrs = [None if a is None else a.ctypes.data for a in arrs]
    rc = _lib.lazy_attn_pack_block_words_host(ctypes.byref(p), int(num_docs), *ptrs, words.ctypes.data,
                                              seq_lens.ctypes.data)
    _check(rc, "pack_block_words_host")
    return words, seq_lens


def pack_block_words(p: Params, num_docs: int, seg_indptr: torch.Tensor, seg_doc: torch.Tensor,
                     seg_len: torch.Tensor, seq_pos0: Optional[torch.Tensor], doc_block_indptr: torch.Tensor,
                     doc_blocks: torch.Tensor, block_words: Optional[torch.Tensor] = None,
                     seq_lens: Optional[torch.Tensor] = None, stream=None):
    """Device packer; every tensor is int32 on the GPU. Returns (block_words, seq_lens)."""
    if block_words is None:
        block_words = torch.empty((p.num_seqs, p.max_blocks_per_seq), dtype=torch.int32, device="cuda")
    if seq_lens is None:
        seq_lens = torch.empty(p.num_seqs, dtype=torch.int32, device="cuda")
    i32 = torch.int32
    rc = _lib.lazy_attn_pack_block_words(
        ctypes.byref(p), int(num_docs), _dptr(seg_indptr, "seg_indptr", i32), _dptr(seg_doc, "seg_doc", i32),
        _dptr(seg_len, "seg_len", i32), _dptr(seq_pos0, "seq_pos0", i32),
        _dptr(doc_block_indptr, "doc_block_indptr", i32), _dptr(doc_blocks, "doc_blocks", i32),
        _dptr(block_words, "block_words"), _dptr(seq_lens, "seq_lens", i32), _stream(stream))
    _check(rc, "pack_block_words")
    return block_words, seq_lens


# ---------------------------------------------------------------- decode / prefill

def decode_workspace_bytes(p: Params) -> int:
    return int(_lib.lazy_attn_decode_workspace_bytes(ctypes.byref(p)))


def decode(p: Params, q: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor, block_words: torch.Tensor,
           seq_lens: torch.Tensor, q_pos: torch.Tensor, rope_table: torch.Tensor, out: Optional[torch.Tensor] = None,
           workspace: Optional[torch.Tensor] = None, stream=None,
           alibi_slopes: Optional[torch.Tensor] = None) -> torch.Tensor:
    """alibi_slopes (fp32 [Hq]) selects lazy_attn_decode_alibi: words packed with key_positions=True."""
    dt = _tdt(p)
    if out is None:
        out = torch.empty_like(q)
    nws = decode_workspace_bytes(p)
    if workspace is None and nws:
        workspace = torch.empty(nws, dtype=torch.uint8, device=q.device)
    wsz = 0 if workspace is None else workspace.numel() * workspace.element_size()
    head = (ctypes.byref(p), _dptr(q, "q", dt), _dptr(k_pool, "k_pool", _kvdt(p)), _dptr(v_pool, "v_pool", _kvdt(p)),
            _dptr(block_words, "block_words"), _dptr(seq_lens, "seq_lens", torch.int32),
            _dptr(q_pos, "q_pos", torch.int32), _dptr(rope_table, "rope_table"))
    tail = (_dptr(out, "out", dt), _dptr(workspace, "workspace"), wsz, _stream(stream))
    if alibi_slopes is None:
        rc = _lib.lazy_attn_decode(*head, *tail)
    else:
        if alibi_slopes.numel() != p.num_q_heads:
            raise ValueError("alibi_slopes needs one slope per query head")
        rc = _lib.lazy_attn_decode_alibi(*head, _dptr(alibi_slopes, "alibi_slopes", torch.float32), *tail)
    _check(rc, "decode")
    return out


def decode_noalloc(p: Params, q: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor,
                   block_words: torch.Tensor, seq_lens: torch.Tensor, q_pos: torch.Tensor, rope_table: torch.Tensor,
                   out: torch.Tensor, stream=None) -> torch.Tensor:
    """Decode whose split-K scratch is the library's static device array (for callers
    that cannot allocate a workspace). ``out`` is required: the call allocates nothing.
    Calls that overlap on the GPU share that array and must not run concurrently."""
    dt = _tdt(p)
    rc = _lib.lazy_attn_decode_noalloc(ctypes.byref(p), _dptr(q, "q", dt), _dptr(k_pool, "k_pool", _kvdt(p)),
                                       _dptr(v_pool, "v_pool", _kvdt(p)), _dptr(block_words, "block_words"),
                                       _dptr(seq_lens, "seq_lens", torch.int32), _dptr(q_pos, "q_pos", torch.int32),
                                       _dptr(rope_table, "rope_table"), _dptr(out, "out", dt), _stream(stream))
    _check(rc, "decode_noalloc")
    return out


class SharedPlan:
    """Work list of the shared-run decode: the planner's host arrays and their device copies.

    ``items_host`` is [num_items, PLAN_ITEM_INTS] int32: header, members {seq, first block,
    slot, 0}, then the physical ids of the item's first blocks; ``slot_indptr_host`` is [B+1]."""

    def __init__(self, items: np.ndarray, slot_indptr: np.ndarray, device="cuda"):
        self.items_host, self.slot_indptr_host = items, slot_indptr
        self.num_items = int(items.shape[0])
        self.num_slots = int(slot_indptr[-1]) if len(slot_indptr) else 0
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32).reshape(-1) if a.size else
                                       np.zeros(PLAN_ITEM_INTS, np.int32)).to(device)
        self.items, self.slot_indptr = t(items), t(slot_indptr)

    def members(self, i: int) -> np.ndarray:
        """[nmem, 4] member records of item i (host)."""
        n = int(self.items_host[i, 4])
        return self.items_host[i, 8: 8 + 4 * n].reshape(n, 4)


def plan_shared_host(p: Params, num_docs: int, seg_indptr, seg_doc, seg_len, doc_block_indptr, doc_blocks,
                     chunk_blocks: int = 0, out=None):
    """Host planner of the shared-run decode. Returns (items [n, PLAN_ITEM_INTS], slot_indptr [B+1]), int32.

    ``out`` = (items [capacity, PLAN_ITEM_INTS], slot_indptr [B+1], counts [2]) int32 arrays
    (pinned host memory, for instance) that the planner fills in place; the call then
    returns views of them and allocates nothing."""
    arrs = [_i32_np(x) if np.size(x) else np.zeros(1, np.int32)
            for x in (seg_indptr, seg_doc, seg_len, doc_block_indptr, doc_blocks)]
    if out is None:
        cap = int(np.sum((np.asarray(seg_len, dtype=np.int64) + BLOCK - 1) // BLOCK)) + 1
        items = np.zeros((cap, PLAN_ITEM_INTS), np.int32)
        slot_indptr = np.zeros(p.num_seqs + 1, np.int32)
        counts = np.zeros(2, np.int32)
    else:
        items, slot_indptr, counts = out
        cap = int(items.shape[0])
    rc = _lib.lazy_attn_plan_shared_host(ctypes.byref(p), int(num_docs), *[a.ctypes.data for a in arrs],
                                         int(chunk_blocks), cap, items.ctypes.data, slot_indptr.ctypes.data,
                                         counts.ctypes.data)
    _check(rc, "plan_shared_host")
    if out is not None:
        return items[: counts[0]], slot_indptr
    return items[: counts[0]].copy(), slot_indptr


def decode_shared_workspace_bytes(p: Params, num_slots: int) -> int:
    return int(_lib.lazy_attn_decode_shared_workspace_bytes(ctypes.byref(p), int(num_slots)))


def decode_shared(p: Params, q: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor, block_words: torch.Tensor,
                  q_pos: torch.Tensor, rope_table: torch.Tensor, plan: SharedPlan, out: Optional[torch.Tensor] = None,
                  workspace: Optional[torch.Tensor] = None, stream=None,
                  alibi_slopes: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Shared-run decode; ``alibi_slopes`` (device fp32 [Hq]) selects the ALiBi call."""
    dt = _tdt(p)
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:  # the library checks a given workspace's size itself
        nws = decode_shared_workspace_bytes(p, plan.num_slots)
        if nws:
            workspace = torch.empty(nws, dtype=torch.uint8, device=q.device)
    wsz = 0 if workspace is None else workspace.numel() * workspace.element_size()
    i32 = torch.int32
    args = (ctypes.byref(p), _dptr(q, "q", dt), _dptr(k_pool, "k_pool", _kvdt(p)), _dptr(v_pool, "v_pool", _kvdt(p)),
            _dptr(block_words, "block_words"), _dptr(q_pos, "q_pos", i32), _dptr(rope_table, "rope_table"),
            plan.num_items, _dptr(plan.items, "items", i32), plan.num_slots,
            _dptr(plan.slot_indptr, "slot_indptr", i32))
    tail = (_dptr(out, "out", dt), _dptr(workspace, "workspace"), wsz, _stream(stream))
    if alibi_slopes is None:
        rc = _lib.lazy_attn_decode_shared(*args, *tail)
    else:
        if alibi_slopes.numel() != p.num_q_heads:
            raise ValueError("alibi_slopes needs one slope per query head")
        rc = _lib.lazy_attn_decode_shared_alibi(*args, _dptr(alibi_slopes, "alibi_slopes", torch.float32), *tail)
    _check(rc, "decode_shared")
    return out


def decode_shared_partials(p: Params, q: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor,
                           block_words: torch.Tensor, q_pos: torch.Tensor, rope_table: torch.Tensor, plan: SharedPlan,
                           workspace: torch.Tensor, stream=None) -> torch.Tensor:
    """First pass of decode_shared: fp32 partials of every slot into ``workspace``."""
    wsz = workspace.numel() * workspace.element_size()
    i32 = torch.int32
    rc = _lib.lazy_attn_decode_shared_partials(
        ctypes.byref(p), _dptr(q, "q", _tdt(p)), _dptr(k_pool, "k_pool", _kvdt(p)), _dptr(v_pool, "v_pool", _kvdt(p)),
        _dptr(block_words, "block_words"), _dptr(q_pos, "q_pos", i32), _dptr(rope_table, "rope_table"),
        plan.num_items, _dptr(plan.items, "items", i32), plan.num_slots, _dptr(workspace, "workspace"), wsz,
        _stream(stream))
    _check(rc, "decode_shared_partials")
    return workspace


def decode_shared_combine(p: Params, plan: SharedPlan, workspace: torch.Tensor, out: torch.Tensor,
                          stream=None) -> torch.Tensor:
    """Second pass of decode_shared: each sequence's slots merged into ``out``."""
    wsz = workspace.numel() * workspace.element_size()
    rc = _lib.lazy_attn_decode_shared_combine(ctypes.byref(p), plan.num_slots,
                                              _dptr(plan.slot_indptr, "slot_indptr", torch.int32),
                                              _dptr(workspace, "workspace"), wsz, _dptr(out, "out", _tdt(p)),
                                              _stream(stream))
    _check(rc, "decode_shared_combine")
    return out


def mixed_workspace_bytes(p_dec: Params, p_pf: Params, num_slots: int) -> int:
    return int(_lib.lazy_attn_mixed_workspace_bytes(ctypes.byref(p_dec), ctypes.byref(p_pf), int(num_slots)))


def mixed(p_dec: Params, q_dec: torch.Tensor, words_dec: torch.Tensor, q_pos: torch.Tensor, plan: SharedPlan,
          p_pf: Params, q_pf: torch.Tensor, cu_seqlens_q: torch.Tensor, q_start: torch.Tensor, max_q_len: int,
          words_pf: torch.Tensor, seq_lens_pf: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor,
          rope_table: torch.Tensor, out_dec: Optional[torch.Tensor] = None, out_pf: Optional[torch.Tensor] = None,
          workspace: Optional[torch.Tensor] = None, stream=None):
    """One launch: shared-run decode of one batch and prefill of another. Returns (out_dec, out_pf)."""
    dt = _tdt(p_dec)
    out_dec = torch.empty_like(q_dec) if out_dec is None else out_dec
    out_pf = torch.empty_like(q_pf) if out_pf is None else out_pf
    if workspace is None:
        workspace = torch.empty(max(1, mixed_workspace_bytes(p_dec, p_pf, plan.num_slots)), dtype=torch.uint8,
                                device=q_dec.device)
    wsz = workspace.numel() * workspace.element_size()
    i32 = torch.int32
    rc = _lib.lazy_attn_mixed(
        ctypes.byref(p_dec), _dptr(q_dec, "q_dec", dt), _dptr(words_dec, "words_dec"), _dptr(q_pos, "q_pos", i32),
        plan.num_items, _dptr(plan.items, "items", i32), plan.num_slots, _dptr(plan.slot_indptr, "slot_indptr", i32),
        _dptr(out_dec, "out_dec", dt), ctypes.byref(p_pf), _dptr(q_pf, "q_pf", dt),
        _dptr(cu_seqlens_q, "cu_seqlens_q", i32), _dptr(q_start, "q_start", i32), int(q_pf.shape[0]), int(max_q_len),
        _dptr(words_pf, "words_pf"), _dptr(seq_lens_pf, "seq_lens_pf", i32), _dptr(out_pf, "out_pf", dt),
        _dptr(k_pool, "k_pool", dt), _dptr(v_pool, "v_pool", dt), _dptr(rope_table, "rope_table"),
        _dptr(workspace, "workspace"), wsz, _stream(stream))
    _check(rc, "mixed")
    return out_dec, out_pf


def alibi_slopes(num_heads: int) -> np.ndarray:
    """The usual ALiBi slopes (lazy_attn_alibi_slopes_host), fp32 [num_heads]."""
    out = np.empty(num_heads, np.float32)
    _check(_lib.lazy_attn_alibi_slopes_host(int(num_heads), out.ctypes.data), "alibi_slopes")
    return out


def materialize(p: Params, k_pool: torch.Tensor, v_pool: torch.Tensor, block_words: torch.Tensor,
                seq_lens: torch.Tensor, rope_table: torch.Tensor, stream=None):
    """Eager baseline: per-sequence copies with K at absolute positions. Returns
    (k_out, v_out, block_words_out) for lazy_attn_decode with lazy = 0."""
    dt = _tdt(p)
    nb = p.num_seqs * p.max_blocks_per_seq
    k_out = torch.empty((nb,) + tuple(k_pool.shape[1:]), dtype=dt, device=k_pool.device)
    v_out = torch.empty_like(k_out)
    words_out = torch.empty((p.num_seqs, p.max_blocks_per_seq), dtype=torch.int32, device=k_pool.device)
    rc = _lib.lazy_attn_materialize(ctypes.byref(p), _dptr(k_pool, "k_pool", dt), _dptr(v_pool, "v_pool", dt),
                                    _dptr(block_words, "block_words"), _dptr(seq_lens, "seq_lens", torch.int32),
                                    _dptr(rope_table, "rope_table"), _dptr(k_out, "k_out"), _dptr(v_out, "v_out"),
                                    _dptr(words_out, "block_words_out"), _stream(stream))
    _check(rc, "materialize")
    return k_out, v_out, words_out


def prefill_workspace_bytes(p: Params, total_q: int) -> int:
    return int(_lib.lazy_attn_prefill_workspace_bytes(ctypes.byref(p), int(total_q)))


def prefill(p: Params, q: torch.Tensor, cu_seqlens_q: torch.Tensor, q_start: torch.Tensor, max_q_len: int,
            k_pool: torch.Tensor, v_pool: torch.Tensor, block_words: torch.Tensor, seq_lens: torch.Tensor,
            rope_table: torch.Tensor, out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
            stream=None, alibi_slopes: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Prefill; ``alibi_slopes`` (device fp32 [Hq]) selects the ALiBi call."""
    dt = _tdt(p)
    if out is None:
        out = torch.empty_like(q)
    nws = prefill_workspace_bytes(p, int(q.shape[0]))
    if workspace is None and nws:
        workspace = torch.empty(nws, dtype=torch.uint8, device=q.device)
    wsz = 0 if workspace is None else workspace.numel() * workspace.element_size()
    head = (ctypes.byref(p), _dptr(q, "q", dt), _dptr(cu_seqlens_q, "cu_seqlens_q", torch.int32),
            _dptr(q_start, "q_start", torch.int32), int(q.shape[0]), int(max_q_len),
            _dptr(k_pool, "k_pool", dt), _dptr(v_pool, "v_pool", dt),
            _dptr(block_words, "block_words"), _dptr(seq_lens, "seq_lens", torch.int32), _dptr(rope_table, "rope_table"))
    tail = (_dptr(out, "out", dt), _dptr(workspace, "workspace"), wsz, _stream(stream))
    if alibi_slopes is None:
        rc = _lib.lazy_attn_prefill(*head, *tail)
    else:
        if alibi_slopes.numel() != p.num_q_heads:
            raise ValueError("alibi_slopes needs one slope per query head")
        rc = _lib.lazy_attn_prefill_alibi(*head, _dptr(alibi_slopes, "alibi_slopes", torch.float32), *tail)
    _check(rc, "prefill")
    return out


def debug_gather(p: Params, k_pool: torch.Tensor, v_pool: torch.Tensor, block_words: torch.Tensor,
                 seq_lens: torch.Tensor, with_pos: bool = True, stream=None, withhold_block: int = -1,
                 wait_limit_us: int = 0):
    """Dense copies of every logical K/V slot through the decode load path. With
    ``withhold_block >= 0`` (failure-path test) that block of sequence 0, KV head 0 is
    never loaded and every wait gives up after ``wait_limit_us``."""
    dt = _tdt(p)
    rows = BLOCK * p.max_blocks_per_seq
    k_out = torch.empty((p.num_seqs, p.num_kv_heads, rows, p.head_dim), dtype=dt, device=k_pool.device)
    v_out = torch.empty_like(k_out)
    pos = torch.empty((p.num_seqs, rows), dtype=torch.int32, device=k_pool.device) if with_pos else None
    args = (ctypes.byref(p), _dptr(k_pool, "k_pool", dt), _dptr(v_pool, "v_pool", dt),
            _dptr(block_words, "block_words"), _dptr(seq_lens, "seq_lens", torch.int32),
            _dptr(k_out, "k_out"), _dptr(v_out, "v_out"), _dptr(pos, "pos_out"))
    if withhold_block >= 0:
        rc = _lib.lazy_attn_debug_gather_withheld(*args, int(withhold_block), int(wait_limit_us), _stream(stream))
    else:
        rc = _lib.lazy_attn_debug_gather(*args, _stream(stream))
    _check(rc, "debug_gather")
    return k_out, v_out, pos


def debug_rope(p: Params, rope_table: torch.Tensor, deltas: torch.Tensor, stream=None) -> torch.Tensor:
    """(cos, sin) of deltas[k] * w_i as the kernels compute them: [n, head_dim/2, 2] fp32."""
    n = int(deltas.numel())
    out = torch.empty((n, p.head_dim // 2, 2), dtype=torch.float32, device=deltas.device)
    _check(_lib.lazy_attn_debug_rope(ctypes.byref(p), _dptr(rope_table, "rope_table"),
                                     _dptr(deltas, "deltas", torch.int32), n, _dptr(out, "cs_out"), _stream(stream)),
           "debug_rope")
    return out


def device_status(clear: bool = True) -> int:
    v = ctypes.c_uint32(0)
    _check(_lib.lazy_attn_device_status(ctypes.byref(v), int(bool(clear))), "device_status")
    return int(v.value)


def launch_count() -> int:
    return int(_lib.lazy_attn_launch_count())
