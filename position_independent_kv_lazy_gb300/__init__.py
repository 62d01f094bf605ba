"""Python binding of ``liblazyattn.so``: deferred-RoPE attention over a position-agnostic paged
KV cache for GB300 (sm_103a).

Argument marshalling only: every step of the attention path runs in the library's CUDA kernels
(``include/lazy_attn.h`` documents each call). PyTorch supplies device memory and streams. If the
library is not built the import of any call raises: there is no fallback implementation.

The functions keep the C names: ``kv_pool_insert_doc``, ``lazy_attn_prefill``,
``lazy_attn_decode`` and the pool / page-word / error helpers.
"""
from __future__ import annotations

import collections
import ctypes
import os
from typing import List, Optional, Sequence, Tuple

import itertools

import numpy as np

from ._build import build_library, library_path  # noqa: F401

LAZY_OK = 0
LAZY_ERR_INVALID_ARG = -1
LAZY_ERR_OUT_OF_BLOCKS = -2
LAZY_ERR_UNSUPPORTED = -3
LAZY_ERR_CUDA = -4
LAZY_ERR_BAD_PAGE = -5
LAZY_ERR_TIMEOUT = -6
LAZY_ERR_SCRATCH_LIMIT = -7
LAZY_NOALLOC_SCRATCH_BYTES = 8 * 1024 * 1024
LAZY_DECODE_AUTO = 0
LAZY_DECODE_SIMT = 1
LAZY_POS_ROPE = 0
LAZY_POS_ALIBI = 1
LAZY_DTYPE_BF16 = 0
LAZY_DTYPE_FP32 = 1
LAZY_DEVERR_BAD_PAGE = 1
LAZY_DEVERR_TIMEOUT = 2
LAZY_PREFILL_AUTO = 0
LAZY_PREFILL_SIMT = 1
LAZY_PREFILL_TC = 2
LAZY_PREFILL_SIMT_QSIDE = 3
LAZY_PREFILL_TC_QSIDE = 4
LAZY_PREFILL_ABSOLUTE_KEYS = 16

# Every symbol declared in include/lazy_attn.h (checked by the tests).
EXPORTS = [
    "lazy_version", "lazy_status_string", "lazy_last_error", "lazy_pool_create",
    "lazy_pool_destroy", "lazy_pool_set_wait_limit", "kv_pool_alloc", "kv_pool_retain",
    "kv_pool_release", "kv_pool_num_free", "kv_pool_refcount", "kv_pool_insert_doc",
    "kv_pool_write_tokens", "kv_pool_materialise", "kv_pool_materialise_batch",
    "lazy_pack_page", "lazy_unpack_page",
    "lazy_pack_pages",
    "lazy_pack_segment", "lazy_decode_workspace_bytes", "lazy_attn_decode",
    "lazy_decode_partition", "lazy_order_segments",
    "lazy_prefill_workspace_bytes",
    "lazy_attn_prefill", "lazy_get_device_error", "lazy_debug_gather", "lazy_debug_wait_timeout",
    "lazy_attn_decode_noalloc", "lazy_attn_prefill_append",
    "lazy_pool_set_schedule_sms", "lazy_decode_shared_plan", "lazy_decode_shared_workspace_bytes",
    "lazy_attn_decode_shared",
    "lazy_pool_set_alibi", "lazy_pool_position_mode", "lazy_pool_set_decode_kernel",
    "lazy_copy_to_device",
]


class LazyError(RuntimeError):
    def __init__(self, fn: str, status: int):
        lib = _LIB
        msg = lib.lazy_status_string(status).decode() if lib else str(status)
        extra = ""
        if status == LAZY_ERR_CUDA and lib:
            extra = ": " + lib.lazy_last_error().decode()
        super().__init__(f"{fn} failed: {msg} ({status}){extra}")
        self.status = status


_LIB = None

_vp = ctypes.c_void_p
_i32 = ctypes.c_int32
_u32 = ctypes.c_uint32
_u64 = ctypes.c_uint64
_f32 = ctypes.c_float
_pi32 = ctypes.POINTER(ctypes.c_int32)
_pu32 = ctypes.POINTER(ctypes.c_uint32)
_pu64 = ctypes.POINTER(ctypes.c_uint64)
_psz = ctypes.POINTER(ctypes.c_size_t)

_SIGS = {
    "lazy_version": ([], ctypes.c_int),
    "lazy_status_string": ([ctypes.c_int], ctypes.c_char_p),
    "lazy_last_error": ([], ctypes.c_char_p),
    "lazy_pool_create": ([ctypes.POINTER(_vp), _vp, _vp, _i32, _i32, _i32, _i32, _i32,
                          ctypes.c_double], ctypes.c_int),
    "lazy_pool_destroy": ([_vp], ctypes.c_int),
    "lazy_pool_set_wait_limit": ([_vp, _u64], ctypes.c_int),
    "lazy_pool_set_alibi": ([_vp, ctypes.POINTER(ctypes.c_float), _i32], ctypes.c_int),
    "lazy_pool_position_mode": ([_vp, _pi32, _pi32], ctypes.c_int),
    "lazy_pool_set_decode_kernel": ([_vp, _i32], ctypes.c_int),
    "lazy_pool_set_schedule_sms": ([_vp, _i32], ctypes.c_int),
    "kv_pool_alloc": ([_vp, _i32, _pi32], ctypes.c_int),
    "kv_pool_retain": ([_vp, _pi32, _i32], ctypes.c_int),
    "kv_pool_release": ([_vp, _pi32, _i32], ctypes.c_int),
    "kv_pool_num_free": ([_vp, _pi32], ctypes.c_int),
    "kv_pool_refcount": ([_vp, _i32, _pi32], ctypes.c_int),
    "kv_pool_insert_doc": ([_vp, _vp, _vp, _i32, _i32, _pi32, _pi32, _i32, _vp], ctypes.c_int),
    "kv_pool_write_tokens": ([_vp, _vp, _vp, _i32, _vp, _vp, _vp], ctypes.c_int),
    "kv_pool_materialise": ([_vp, _pi32, _pi32, _i32, _i32, _vp], ctypes.c_int),
    "kv_pool_materialise_batch": ([_vp, _i32, _pi32, _pi32, _pi32, _pi32, _pi32, _vp],
                                  ctypes.c_int),
    "lazy_pack_page": ([_u32, _u32, _u32, _pu64], ctypes.c_int),
    "lazy_unpack_page": ([_u64, _pu32, _pu32, _pu32], ctypes.c_int),
    "lazy_pack_pages": ([_i32, _pu32, _pu32, _pu32, _pu64], ctypes.c_int),
    "lazy_pack_segment": ([_pu32, _i32, ctypes.c_uint32, _i32, _i32, _i32, _pu64, _i32, _pi32],
                          ctypes.c_int),
    "lazy_decode_workspace_bytes": ([_vp, _i32, _i32, _i32, _psz], ctypes.c_int),
    "lazy_decode_partition": ([_vp, _i32, _i32, _pi32, ctypes.POINTER(ctypes.c_int64)],
                              ctypes.c_int),
    "lazy_order_segments": ([_i32, _pi32, ctypes.POINTER(ctypes.c_int64), _pi32,
                             ctypes.POINTER(ctypes.c_uint8), _i32, ctypes.c_int64, _pi32],
                            ctypes.c_int),
    "lazy_attn_decode": ([_vp, _vp, _vp, _vp, _vp, _i32, _i32, _f32, _i32, _vp, _vp, _vp,
                          ctypes.c_size_t, _vp], ctypes.c_int),
    "lazy_prefill_workspace_bytes": ([_vp, _i32, _i32, _i32, _i32, _i32, _psz], ctypes.c_int),
    "lazy_attn_prefill": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _f32,
                           _vp, _vp, _vp, ctypes.c_size_t, _i32, _vp], ctypes.c_int),
    "lazy_attn_prefill_append": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32,
                                  _i32, _f32, _vp, _vp, _vp, ctypes.c_size_t, _i32, _vp, _vp,
                                  _vp], ctypes.c_int),
    "lazy_get_device_error": ([_vp, _pi32, _vp], ctypes.c_int),
    "lazy_copy_to_device": ([_vp, _vp, ctypes.c_size_t, _vp], ctypes.c_int),
    "lazy_debug_gather": ([_vp, _vp, _i32, _vp, _vp, _vp, _vp], ctypes.c_int),
    "lazy_debug_wait_timeout": ([_vp, _u64, _vp], ctypes.c_int),
    "lazy_attn_decode_noalloc": ([_vp, _vp, _vp, _vp, _vp, _i32, _i32, _f32, _i32, _vp, _vp, _vp],
                                 ctypes.c_int),
    "lazy_decode_shared_plan": ([_vp, _vp, _i32, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _pi32,
                                 _pi32],
                                ctypes.c_int),
    "lazy_decode_shared_workspace_bytes": ([_vp, _i32, _i32, _i32, _psz], ctypes.c_int),
    "lazy_attn_decode_shared": ([_vp, _vp, _vp, _vp, _vp, _vp, _i32, _vp, _vp, _vp, _i32, _i32,
                                 _f32, _i32, _vp, _vp, _vp, ctypes.c_size_t, _vp], ctypes.c_int),
}


def load_library(path: Optional[str] = None):
    """Load the built library (raises if it has not been built)."""
    global _LIB
    if _LIB is None:
        path = path or library_path()
        if not os.path.exists(path):
            raise RuntimeError(
                f"{path} is missing: build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'` (no fallback exists)")
        lib = ctypes.CDLL(path)
        for name, (args, res) in _SIGS.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _LIB = lib
    return _LIB


def _check(fn: str, status: int):
    if status != LAZY_OK:
        raise LazyError(fn, status)


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream) -> Optional[int]:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _dtype_code(dtype) -> int:
    import torch
    if dtype == torch.bfloat16:
        return LAZY_DTYPE_BF16
    if dtype == torch.float32:
        return LAZY_DTYPE_FP32
    raise ValueError(f"unsupported pool dtype {dtype}")


# ------------------------------------------------------------------------------------------------
# Pool
# ------------------------------------------------------------------------------------------------
class LazyPool:
    """A paged KV pool: page buffers [num_blocks][Hkv][16][D] allocated with torch on `device`."""

    def __init__(self, num_blocks: int, num_kv_heads: int, head_dim: int, dtype, rope_base: float,
                 page_size: int = 16, device="cuda", alibi_slopes=None):
        """alibi_slopes (per query head) switches the pool to ALiBi mode: K cached unrotated, a
        bias slope * (n - m) at attention time, page words carrying page start positions."""
        import torch
        lib = load_library()
        self.num_blocks, self.hkv, self.d, self.page_size = num_blocks, num_kv_heads, head_dim, page_size
        self.dtype = dtype
        self.rope_base = rope_base
        shape = (num_blocks, num_kv_heads, page_size, head_dim)
        self.k_pages = torch.empty(shape, dtype=dtype, device=device)
        self.v_pages = torch.empty(shape, dtype=dtype, device=device)
        h = _vp()
        _check("lazy_pool_create", lib.lazy_pool_create(
            ctypes.byref(h), self.k_pages.data_ptr(), self.v_pages.data_ptr(), num_blocks,
            page_size, num_kv_heads, head_dim, _dtype_code(dtype), float(rope_base)))
        self.handle = h
        self.alibi_slopes = None
        if alibi_slopes is not None:
            sl = [float(x) for x in alibi_slopes]
            arr = (ctypes.c_float * len(sl))(*sl)
            _check("lazy_pool_set_alibi", lib.lazy_pool_set_alibi(h, arr, len(sl)))
            self.alibi_slopes = sl

    def close(self):
        if getattr(self, "handle", None):
            load_library().lazy_pool_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def lazy_pool_set_decode_kernel(pool: LazyPool, kind: int):
    """LAZY_DECODE_AUTO (tensor-core decode for bf16 / head_dim 128) or LAZY_DECODE_SIMT."""
    _check("lazy_pool_set_decode_kernel",
           load_library().lazy_pool_set_decode_kernel(pool.handle, int(kind)))


def lazy_pool_set_schedule_sms(pool: LazyPool, sms: int):
    """SMs the tensor-core prefill plans its last wave for (0 = the device's)."""
    _check("lazy_pool_set_schedule_sms",
           load_library().lazy_pool_set_schedule_sms(pool.handle, int(sms)))


def lazy_pool_set_wait_limit(pool: LazyPool, ns: int):
    _check("lazy_pool_set_wait_limit", load_library().lazy_pool_set_wait_limit(pool.handle, ns))


def kv_pool_alloc(pool: LazyPool, n: int) -> List[int]:
    ids = (ctypes.c_int32 * max(n, 1))()
    _check("kv_pool_alloc", load_library().kv_pool_alloc(pool.handle, n, ids))
    return list(ids[:n])


def kv_pool_retain(pool: LazyPool, ids: Sequence[int]):
    arr = (ctypes.c_int32 * max(len(ids), 1))(*ids)
    _check("kv_pool_retain", load_library().kv_pool_retain(pool.handle, arr, len(ids)))


def kv_pool_release(pool: LazyPool, ids: Sequence[int]):
    arr = (ctypes.c_int32 * max(len(ids), 1))(*ids)
    _check("kv_pool_release", load_library().kv_pool_release(pool.handle, arr, len(ids)))


def kv_pool_num_free(pool: LazyPool) -> int:
    n = ctypes.c_int32()
    _check("kv_pool_num_free", load_library().kv_pool_num_free(pool.handle, ctypes.byref(n)))
    return n.value


def kv_pool_refcount(pool: LazyPool, block: int) -> int:
    n = ctypes.c_int32()
    _check("kv_pool_refcount", load_library().kv_pool_refcount(pool.handle, block, ctypes.byref(n)))
    return n.value


def kv_pool_insert_doc(pool: LazyPool, k_raw, v, local_pos0: int = 0,
                       block_ids: Optional[Sequence[int]] = None, stream=None) -> List[int]:
    """Encode a segment's tokens (k rotated at local positions local_pos0.., v copied) into the
    pool; returns the segment's block ids (existing ones first, new ones appended)."""
    n = int(k_raw.shape[0])
    owned = np.asarray(block_ids if block_ids is not None else [], dtype=np.int32)
    cap = max(owned.shape[0], (local_pos0 + n + pool.page_size - 1) // pool.page_size, 1)
    arr = np.zeros(cap, dtype=np.int32)
    arr[: owned.shape[0]] = owned
    nb = ctypes.c_int32(owned.shape[0])
    _check("kv_pool_insert_doc", load_library().kv_pool_insert_doc(
        pool.handle, _ptr(k_raw.contiguous()), _ptr(v.contiguous()), n, local_pos0,
        arr.ctypes.data_as(_pi32), ctypes.byref(nb), cap, _stream(stream)))
    return arr[: nb.value].tolist()


def kv_pool_write_tokens(pool: LazyPool, k_raw, v, slot_mapping, local_pos, stream=None):
    _check("kv_pool_write_tokens", load_library().kv_pool_write_tokens(
        pool.handle, _ptr(k_raw), _ptr(v), int(k_raw.shape[0]), _ptr(slot_mapping),
        _ptr(local_pos), _stream(stream)))


def kv_pool_materialise(pool: LazyPool, src_block_ids: Sequence[int], n_tokens: int,
                        offset: int, dst_block_ids: Optional[Sequence[int]] = None,
                        stream=None) -> List[int]:
    """Re-encode a cached segment (n_tokens tokens in src_block_ids) for logical offset
    `offset` into blocks of its own (allocated here unless dst_block_ids is given): keys at
    absolute positions, the copy-per-offset baseline. Returns the copy's block ids."""
    n_pages = (n_tokens + pool.page_size - 1) // pool.page_size
    dst = list(dst_block_ids) if dst_block_ids is not None else kv_pool_alloc(pool, n_pages)
    src = (ctypes.c_int32 * max(n_pages, 1))(*list(src_block_ids)[:n_pages])
    dd = (ctypes.c_int32 * max(n_pages, 1))(*dst[:n_pages])
    _check("kv_pool_materialise", load_library().kv_pool_materialise(
        pool.handle, src, dd, n_tokens, offset, _stream(stream)))
    return dst[:n_pages]


def kv_pool_materialise_batch(pool: LazyPool, copies: Sequence[tuple], stream=None) -> List[List[int]]:
    """kv_pool_materialise for many copies in one launch. copies: (src_block_ids, n_tokens,
    offset) or (src_block_ids, n_tokens, offset, dst_block_ids); destination blocks are
    allocated here (in one allocation) where not given. Returns each copy's block ids."""
    nc = len(copies)
    ps = pool.page_size
    n_tok = np.fromiter((int(cp[1]) for cp in copies), dtype=np.int64, count=nc)
    offs = np.fromiter((int(cp[2]) for cp in copies), dtype=np.int64, count=nc)
    pages = (n_tok + ps - 1) // ps
    cu = np.zeros(nc + 1, dtype=np.int32)
    cu[1:] = np.cumsum(pages)
    total = int(cu[-1])
    given = np.fromiter((len(cp) > 3 and cp[3] is not None for cp in copies), dtype=bool,
                        count=nc)
    pl = pages.tolist()
    src = np.zeros(max(total, 1), dtype=np.int32)
    src[:total] = np.fromiter(itertools.chain.from_iterable(
        cp[0][:n] for cp, n in zip(copies, pl)), dtype=np.int32, count=total)
    need = int(pages[~given].sum()) if nc else 0
    fresh = np.asarray(kv_pool_alloc(pool, need) if need else [], dtype=np.int32)
    if need == total:  # every destination allocated here, in copy order
        dst = fresh if total else np.zeros(1, dtype=np.int32)
    else:
        dst = np.zeros(max(total, 1), dtype=np.int32)
        k = 0
        for c, cp in enumerate(copies):
            lo, hi = int(cu[c]), int(cu[c + 1])
            if given[c]:
                dst[lo:hi] = np.asarray(list(cp[3])[: hi - lo], dtype=np.int32)
            else:
                dst[lo:hi] = fresh[k:k + hi - lo]
                k += hi - lo
    nt32, off32 = n_tok.astype(np.int32), offs.astype(np.int32)
    if nc == 0:
        nt32 = off32 = np.zeros(1, dtype=np.int32)
    p32 = lambda a: a.ctypes.data_as(_pi32)
    _check("kv_pool_materialise_batch", load_library().kv_pool_materialise_batch(
        pool.handle, nc, p32(cu), p32(src), p32(dst), p32(nt32), p32(off32), _stream(stream)))
    flat, cl = dst.tolist(), cu.tolist()
    return [flat[cl[c]:cl[c + 1]] for c in range(nc)]


# ------------------------------------------------------------------------------------------------
# Page words
# ------------------------------------------------------------------------------------------------
def lazy_pack_page(block_id: int, offset: int, n_valid: int) -> int:
    w = ctypes.c_uint64()
    _check("lazy_pack_page", load_library().lazy_pack_page(block_id, offset, n_valid,
                                                           ctypes.byref(w)))
    return w.value


def lazy_unpack_page(word: int) -> Tuple[int, int, int]:
    a, b, c = ctypes.c_uint32(), ctypes.c_uint32(), ctypes.c_uint32()
    _check("lazy_unpack_page", load_library().lazy_unpack_page(
        word, ctypes.byref(a), ctypes.byref(b), ctypes.byref(c)))
    return a.value, b.value, c.value


def lazy_pack_pages(block_ids, offsets, n_valid) -> np.ndarray:
    b = np.ascontiguousarray(block_ids, dtype=np.uint32)
    o = np.ascontiguousarray(offsets, dtype=np.uint32)
    v = np.ascontiguousarray(n_valid, dtype=np.uint32)
    out = np.zeros(b.shape[0], dtype=np.uint64)
    _check("lazy_pack_pages", load_library().lazy_pack_pages(
        b.shape[0], b.ctypes.data_as(_pu32), o.ctypes.data_as(_pu32), v.ctypes.data_as(_pu32),
        out.ctypes.data_as(_pu64)))
    return out


def align_shared_segments(requests: Sequence[Sequence[Tuple[Sequence[int], int, int]]]
                          ) -> List[List[Tuple[Sequence[int], int, int]]]:
    """Reorder each request's segments so that a segment cached once and used by several
    requests (the same block ids) sits at the same index of every request's list.

    Attention over a request does not depend on the order of its pages (each page word carries
    its own offset), so the order is free. The decode kernels stream every request's pages
    front to back at about the same rate; with a shared document at the same index everywhere,
    its pages are read by all its requests at about the same time, and all but the first read
    hit L2. Greedy: segments in order of decreasing use count take the index that is free in
    most of their requests; a segment that finds it taken, and every segment used once, fills
    the first free index, in the request's own order."""
    keys = [[tuple(ids) for ids, _, _ in segs] for segs in requests]
    count = collections.Counter(k for ks in keys for k in set(ks))
    shared = sorted((k for k, c in count.items() if c > 1),
                    key=lambda k: (-count[k], k[:1]))
    placed = [[None] * len(segs) for segs in requests]     # index -> segment position
    used = [set() for _ in requests]                        # segment positions placed
    where = collections.defaultdict(list)                   # key -> [(request, position)]
    for b, ks in enumerate(keys):
        for i, k in enumerate(ks):
            where[k].append((b, i))
    for k in shared:
        first = {}
        for b, i in where[k]:
            first.setdefault(b, i)                          # one occurrence per request
        width = max(len(placed[b]) for b in first)
        best = max(range(width), key=lambda s: (
            sum(1 for b in first if s < len(placed[b]) and placed[b][s] is None), -s))
        for b, i in first.items():
            if best < len(placed[b]) and placed[b][best] is None:
                placed[b][best] = i
                used[b].add(i)
    out = []
    for b, segs in enumerate(requests):
        rest = iter(i for i in range(len(segs)) if i not in used[b])
        order = [i if i is not None else next(rest) for i in placed[b]]
        out.append([segs[i] for i in order])
    return out


def lazy_decode_partition(pool: LazyPool, num_q_heads: int, grid_ctas: int = 0):
    """(units per request, ranges) of the decode's work partition (see the C header)."""
    u = ctypes.c_int32()
    r = ctypes.c_int64()
    _check("lazy_decode_partition", load_library().lazy_decode_partition(
        pool.handle, num_q_heads, grid_ctas, ctypes.byref(u), ctypes.byref(r)))
    return u.value, r.value


def order_segments_by_phase(requests: Sequence[Sequence[Tuple[Sequence[int], int, int]]],
                            units_per_request: int, ranges: int, page_size: int = 16,
                            pin_last: bool = True) -> List[List[Tuple[Sequence[int], int, int]]]:
    """Reorder each request's segments (block_ids, offset, length) with lazy_order_segments:
    a segment is identified by its first block id; with ``pin_last`` each request's last
    segment (its private tail) stays last. The attention does not change; the decode reads a
    shared document's pages for all its requests at about the same time."""
    cu, keys, pages, pin = [0], [], [], []
    for segs in requests:
        for i, (ids, _, length) in enumerate(segs):
            keys.append(int(ids[0]) if len(ids) else -1 - len(keys))
            pages.append((int(length) + page_size - 1) // page_size)
            pin.append(1 if (pin_last and i == len(segs) - 1) else 0)
        cu.append(len(keys))
    n = len(keys)
    cu_a = np.asarray(cu, dtype=np.int32)
    key_a = np.asarray(keys, dtype=np.int64)
    pg_a = np.asarray(pages, dtype=np.int32)
    pin_a = np.asarray(pin, dtype=np.uint8)
    perm = np.zeros(max(n, 1), dtype=np.int32)
    _check("lazy_order_segments", load_library().lazy_order_segments(
        len(requests), cu_a.ctypes.data_as(_pi32), key_a.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
        pg_a.ctypes.data_as(_pi32), pin_a.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8)),
        units_per_request, ranges, perm.ctypes.data_as(_pi32)))
    return [[segs[int(perm[cu[b] + i])] for i in range(len(segs))]
            for b, segs in enumerate(requests)]


def build_page_table(requests: Sequence[Sequence[Tuple[Sequence[int], int, int]]],
                     page_size: int = 16, page_positions: bool = False,
                     align_shared: bool = False) -> Tuple[np.ndarray, np.ndarray]:
    """Page table of a batch: ``requests[b]`` lists segments (block_ids, logical offset, length).
    The word's offset field is the segment's offset (RoPE pools) or, with ``page_positions``
    (ALiBi pools), the logical position of each page's first token. ``align_shared`` orders
    each request's segments with align_shared_segments (same attention result, more L2 reuse).
    Returns (words uint64 [total pages], cu_pages int32 [B+1])."""
    if align_shared:
        requests = align_shared_segments(requests)
    lib = load_library()
    parts, cu = [], [0]
    for segs in requests:
        total = cu[-1]
        for ids, o, length in segs:
            b = np.ascontiguousarray(ids, dtype=np.uint32)
            w = np.zeros(max(1, b.shape[0]), dtype=np.uint64)
            n = ctypes.c_int32()
            _check("lazy_pack_segment", lib.lazy_pack_segment(
                b.ctypes.data_as(_pu32), b.shape[0], int(o), int(length), page_size,
                1 if page_positions else 0, w.ctypes.data_as(_pu64), w.shape[0],
                ctypes.byref(n)))
            parts.append(w[:n.value])
            total += n.value
        cu.append(total)
    words = np.concatenate(parts) if parts else np.zeros(0, dtype=np.uint64)
    return words, np.asarray(cu, dtype=np.int32)


# ------------------------------------------------------------------------------------------------
# Attention
# ------------------------------------------------------------------------------------------------
def lazy_decode_workspace_bytes(pool: LazyPool, batch: int, num_q_heads: int,
                                grid_ctas: int = 0) -> int:
    n = ctypes.c_size_t()
    _check("lazy_decode_workspace_bytes", load_library().lazy_decode_workspace_bytes(
        pool.handle, batch, num_q_heads, grid_ctas, ctypes.byref(n)))
    return n.value


def lazy_attn_decode(pool: LazyPool, q, q_pos, page_words, cu_pages, sm_scale=None,
                     grid_ctas: int = 0, out=None, lse=None, workspace=None, stream=None):
    """q [B,Hq,D] raw; q_pos int32 [B]; page_words uint64/int64 [P]; cu_pages int32 [B+1]
    (all device tensors). Returns (out [B,Hq,D], lse [B,Hq] float32)."""
    import torch
    B, Hq, D = q.shape
    if sm_scale is None:
        sm_scale = 1.0 / float(D) ** 0.5
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    if workspace is None:
        nbytes = lazy_decode_workspace_bytes(pool, B, Hq, grid_ctas)
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    _check("lazy_attn_decode", load_library().lazy_attn_decode(
        pool.handle, _ptr(q), _ptr(q_pos), _ptr(page_words), _ptr(cu_pages), B, Hq,
        float(sm_scale), grid_ctas, _ptr(out), _ptr(lse), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))
    return out, lse


class SharedPlan:
    """A shared-segment decode plan (host numpy arrays; `to(device)` gives torch tensors)."""

    def __init__(self, entries, cu_entries, unit_req, cu_members, members, member_entries):
        self.entries = entries                # uint64 [2 * n_entries]
        self.cu_entries = cu_entries          # int32 [n_units + 1]
        self.unit_req = unit_req              # int32 [2 * n_units]
        self.cu_members = cu_members          # int32 [batch + 1]
        self.members = members                # int32 [n_members]
        self.member_entries = member_entries  # int32 [2 * n_members]
        self.n_units = int(len(cu_entries) - 1)

    @property
    def n_entries(self) -> int:
        return int(self.cu_entries[-1])

    def to(self, device):
        import torch
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(device)
        d = SharedPlan(t(self.entries.view(np.int64)), t(self.cu_entries), t(self.unit_req),
                       t(self.cu_members), t(self.members), t(self.member_entries))
        d.n_units = self.n_units
        return d


def lazy_decode_shared_plan(page_words, cu_pages, page_positions: bool = False) -> SharedPlan:
    """Plan the shared-segment decode from host page tables (numpy uint64 [P], int32 [B+1]);
    page_positions for ALiBi pools' words (each page's first position)."""
    w = np.ascontiguousarray(np.asarray(page_words).view(np.uint64))
    cu = np.ascontiguousarray(np.asarray(cu_pages, dtype=np.int32))
    B = len(cu) - 1
    P = int(cu[-1] - cu[0]) if B > 0 else 0
    # capacities for P pages; the planner fills the leading parts (returned as views)
    entries = np.empty(max(2 * P, 2), dtype=np.uint64)
    cu_e = np.empty(P + 1, dtype=np.int32)
    unit_req = np.empty(max(2 * P, 2), dtype=np.int32)
    cu_m = np.empty(B + 1, dtype=np.int32)
    members = np.empty(max(P, 1), dtype=np.int32)
    member_entries = np.empty(max(2 * P, 2), dtype=np.int32)
    nu, ne = ctypes.c_int32(), ctypes.c_int32()
    _check("lazy_decode_shared_plan", load_library().lazy_decode_shared_plan(
        w.ctypes.data, cu.ctypes.data, B, int(bool(page_positions)), entries.ctypes.data,
        cu_e.ctypes.data,
        unit_req.ctypes.data, cu_m.ctypes.data, members.ctypes.data, member_entries.ctypes.data,
        ctypes.byref(nu), ctypes.byref(ne)))
    nu, ne = nu.value, ne.value
    nm = int(cu_m[-1])
    return SharedPlan(entries[:2 * ne], cu_e[:nu + 1], unit_req[:2 * nu], cu_m, members[:nm],
                      member_entries[:2 * nm])


def lazy_decode_shared_workspace_bytes(pool: LazyPool, n_units: int, num_q_heads: int,
                                       grid_ctas: int = 0) -> int:
    n = ctypes.c_size_t()
    _check("lazy_decode_shared_workspace_bytes", load_library().lazy_decode_shared_workspace_bytes(
        pool.handle, n_units, num_q_heads, grid_ctas, ctypes.byref(n)))
    return n.value


def lazy_attn_decode_shared(pool: LazyPool, q, q_pos, plan: SharedPlan, sm_scale=None,
                            grid_ctas: int = 0, out=None, lse=None, workspace=None, stream=None):
    """lazy_attn_decode over a shared-segment plan (`plan` on q's device: SharedPlan.to).
    Returns (out [B,Hq,D], lse [B,Hq] float32)."""
    import torch
    B, Hq, D = q.shape
    if sm_scale is None:
        sm_scale = 1.0 / float(D) ** 0.5
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    if workspace is None:
        nbytes = lazy_decode_shared_workspace_bytes(pool, plan.n_units, Hq, grid_ctas)
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    _check("lazy_attn_decode_shared", load_library().lazy_attn_decode_shared(
        pool.handle, _ptr(q), _ptr(q_pos), _ptr(plan.entries), _ptr(plan.cu_entries),
        _ptr(plan.unit_req), plan.n_units, _ptr(plan.cu_members), _ptr(plan.members),
        _ptr(plan.member_entries), B, Hq,
        float(sm_scale), grid_ctas, _ptr(out), _ptr(lse), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))
    return out, lse


def lazy_prefill_workspace_bytes(pool: LazyPool, batch: int, total_q: int, max_q_len: int,
                                 num_q_heads: int, flags: int = 0) -> int:
    """Scratch bytes a prefill of this shape can use (0 when its schedule needs none)."""
    n = ctypes.c_size_t()
    _check("lazy_prefill_workspace_bytes", load_library().lazy_prefill_workspace_bytes(
        pool.handle, batch, total_q, max_q_len, num_q_heads, flags, ctypes.byref(n)))
    return n.value


def _prefill_workspace(pool, q, B, max_q_len, flags, workspace):
    import torch
    if workspace is not None:
        return workspace, workspace.numel() * workspace.element_size()
    Tq, Hq, _ = q.shape
    n = lazy_prefill_workspace_bytes(pool, B, Tq, max_q_len, Hq, flags)
    return torch.empty(max(n, 1), dtype=torch.uint8, device=q.device), n


def lazy_attn_prefill(pool: LazyPool, q, k_new, v_new, cu_q, q_pos0, page_words, cu_pages,
                      max_q_len: int, sm_scale=None, out=None, lse=None, flags: int = 0,
                      workspace=None, stream=None):
    """q [Tq,Hq,D] raw; k_new/v_new [Tq,Hkv,D] raw or None; cu_q, q_pos0, cu_pages int32;
    page_words uint64 (device). workspace: device scratch (default: allocated at
    lazy_prefill_workspace_bytes); a smaller one only turns off the last-wave split.
    Returns (out [Tq,Hq,D], lse [Tq,Hq] float32)."""
    import torch
    Tq, Hq, D = q.shape
    B = int(cu_q.shape[0]) - 1
    if sm_scale is None:
        sm_scale = 1.0 / float(D) ** 0.5
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((Tq, Hq), dtype=torch.float32, device=q.device)
    ws, nbytes = _prefill_workspace(pool, q, B, max_q_len, flags, workspace)
    _check("lazy_attn_prefill", load_library().lazy_attn_prefill(
        pool.handle, _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(cu_q), _ptr(q_pos0),
        _ptr(page_words), _ptr(cu_pages), B, Tq, max_q_len, Hq, float(sm_scale), _ptr(out),
        _ptr(lse), _ptr(ws), nbytes, flags, _stream(stream)))
    return out, lse


def lazy_attn_prefill_append(pool: LazyPool, q, k_new, v_new, cu_q, q_pos0, page_words, cu_pages,
                             max_q_len: int, append_slots, append_local_pos, sm_scale=None,
                             out=None, lse=None, flags: int = 0, workspace=None, stream=None):
    """lazy_attn_prefill, then every question token t written into the pool at slot
    append_slots[t] (int32, block * page_size + slot, < 0 skips) as R(append_local_pos[t])
    k_new[t] and v_new[t]. Returns (out, lse)."""
    import torch
    Tq, Hq, D = q.shape
    B = int(cu_q.shape[0]) - 1
    if sm_scale is None:
        sm_scale = 1.0 / float(D) ** 0.5
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((Tq, Hq), dtype=torch.float32, device=q.device)
    ws, nbytes = _prefill_workspace(pool, q, B, max_q_len, flags, workspace)
    _check("lazy_attn_prefill_append", load_library().lazy_attn_prefill_append(
        pool.handle, _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(cu_q), _ptr(q_pos0),
        _ptr(page_words), _ptr(cu_pages), B, Tq, max_q_len, Hq, float(sm_scale), _ptr(out),
        _ptr(lse), _ptr(ws), nbytes, flags, _ptr(append_slots), _ptr(append_local_pos),
        _stream(stream)))
    return out, lse


def lazy_get_device_error(pool: LazyPool, stream=None) -> int:
    e = ctypes.c_int32()
    _check("lazy_get_device_error", load_library().lazy_get_device_error(
        pool.handle, ctypes.byref(e), _stream(stream)))
    return e.value


def lazy_copy_to_device(dst, src, stream=None) -> None:
    """Copy the pinned host tensor `src` into the device tensor `dst` (same number of bytes, a
    multiple of 16) with the SM-driven upload kernel; stream-ordered and asynchronous."""
    n = src.numel() * src.element_size()
    if dst.numel() * dst.element_size() != n:
        raise ValueError("lazy_copy_to_device: dst and src differ in size")
    _check("lazy_copy_to_device", load_library().lazy_copy_to_device(
        _ptr(dst), _ptr(src), n, _stream(stream)))


def lazy_debug_gather(pool: LazyPool, page_words, stream=None):
    import torch
    n = int(page_words.shape[0])
    shape = (n, pool.hkv, pool.page_size, pool.d)
    k = torch.empty(shape, dtype=pool.dtype, device=page_words.device)
    v = torch.empty(shape, dtype=pool.dtype, device=page_words.device)
    f = torch.empty((n, 3), dtype=torch.int32, device=page_words.device)
    _check("lazy_debug_gather", load_library().lazy_debug_gather(
        pool.handle, _ptr(page_words), n, _ptr(k), _ptr(v), _ptr(f), _stream(stream)))
    return k, v, f


def lazy_debug_wait_timeout(pool: LazyPool, limit_ns: int, stream=None):
    _check("lazy_debug_wait_timeout", load_library().lazy_debug_wait_timeout(
        pool.handle, limit_ns, _stream(stream)))


def lazy_attn_decode_noalloc(pool: LazyPool, q, q_pos, page_words, cu_pages, sm_scale=None,
                             grid_ctas: int = 0, out=None, lse=None, stream=None):
    """Decode without a workspace: the library's fixed scratch array takes the partial results.
    For callers that cannot allocate device memory. ``out`` and ``lse`` should be passed in by
    such callers; when omitted they are created here for convenience."""
    import torch
    B, Hq, D = q.shape
    if sm_scale is None:
        sm_scale = 1.0 / float(D) ** 0.5
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    _check("lazy_attn_decode_noalloc", load_library().lazy_attn_decode_noalloc(
        pool.handle, _ptr(q), _ptr(q_pos), _ptr(page_words), _ptr(cu_pages), B, Hq,
        float(sm_scale), grid_ctas, _ptr(out), _ptr(lse), _stream(stream)))
    return out, lse
