"""CPU checks of the C-ABI library: it builds, loads, exports every declared symbol, and its host
logic (page-word packing, block allocator, argument validation) behaves as documented. No kernel
is launched here."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
import position_independent_kv_lazy_gb300 as pk

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "lazy_attn.h")


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", src, flags=re.M)))


def test_header_symbols_are_exported(lazylib):
    names = _declared()
    assert len(names) >= 20
    assert sorted(pk.EXPORTS) == names
    for n in names:
        assert hasattr(lazylib, n), n


def test_status_strings(lazylib):
    assert lazylib.lazy_version() >= 100
    for code in range(-6, 1):
        assert lazylib.lazy_status_string(code).decode() != "unknown status"


def test_pack_matches_oracle_spec_boundaries(lazylib):
    for blk in (0, 1, 2**31 - 1, 2**31, 2**32 - 1):
        for off in (0, 1, 2**25, 2**26 - 1):
            for nv in (1, 2, 16, 63, 64):
                w = pk.lazy_pack_page(blk, off, nv)
                assert w == oracle.pack_page(blk, off, nv)
                assert pk.lazy_unpack_page(w) == (blk, off, nv)


def test_pack_pages_random_bit_exact(lazylib):
    rng = np.random.default_rng(7)
    n = 200000
    b = rng.integers(0, 2**32, n, dtype=np.uint64).astype(np.uint32)
    o = rng.integers(0, 2**26, n).astype(np.uint32)
    v = rng.integers(1, 65, n).astype(np.uint32)
    w = pk.lazy_pack_pages(b, o, v)
    idx = rng.integers(0, n, 2000)
    for i in idx:
        assert int(w[i]) == oracle.pack_page(int(b[i]), int(o[i]), int(v[i]))
    # vectorised unpack with the oracle's field layout
    assert np.array_equal(w & np.uint64(0xFFFFFFFF), b.astype(np.uint64))
    assert np.array_equal((w >> np.uint64(32)) & np.uint64(2**26 - 1), o.astype(np.uint64))
    assert np.array_equal((w >> np.uint64(58)) + np.uint64(1), v.astype(np.uint64))


@pytest.mark.parametrize("args", [(0, 2**26, 1), (0, 0, 0), (0, 0, 65)])
def test_pack_rejects_out_of_range(lazylib, args):
    with pytest.raises(pk.LazyError):
        pk.lazy_pack_page(*args)


def test_pack_pages_stops_at_bad_entry(lazylib):
    with pytest.raises(pk.LazyError):
        pk.lazy_pack_pages([1, 2, 3], [0, 0, 0], [16, 0, 16])


def _raw_pool(lazylib, num_blocks=10, page=16, hkv=2, d=64, dtype=0, base=1e4, k=0x10000,
              v=0x20000):
    h = ctypes.c_void_p()
    rc = lazylib.lazy_pool_create(ctypes.byref(h), k, v, num_blocks, page, hkv, d, dtype, base)
    return rc, h


def test_pool_create_validation(lazylib):
    assert _raw_pool(lazylib)[0] == 0
    assert _raw_pool(lazylib, num_blocks=0)[0] == pk.LAZY_ERR_INVALID_ARG
    assert _raw_pool(lazylib, page=32)[0] == pk.LAZY_ERR_UNSUPPORTED
    assert _raw_pool(lazylib, d=96)[0] == pk.LAZY_ERR_UNSUPPORTED
    assert _raw_pool(lazylib, dtype=7)[0] == pk.LAZY_ERR_UNSUPPORTED
    assert _raw_pool(lazylib, base=-1.0)[0] == pk.LAZY_ERR_INVALID_ARG
    assert _raw_pool(lazylib, k=0x10008)[0] == pk.LAZY_ERR_INVALID_ARG   # misaligned
    assert _raw_pool(lazylib, k=0)[0] == pk.LAZY_ERR_INVALID_ARG


def test_block_allocator(lazylib):
    rc, h = _raw_pool(lazylib, num_blocks=6)
    assert rc == 0

    def free():
        n = ctypes.c_int32()
        assert lazylib.kv_pool_num_free(h, ctypes.byref(n)) == 0
        return n.value

    def rc_of(b):
        n = ctypes.c_int32()
        assert lazylib.kv_pool_refcount(h, b, ctypes.byref(n)) == 0
        return n.value

    ids = (ctypes.c_int32 * 6)()
    assert lazylib.kv_pool_alloc(h, 4, ids) == 0
    got = list(ids[:4])
    assert len(set(got)) == 4 and free() == 2
    assert lazylib.kv_pool_alloc(h, 3, ids) == pk.LAZY_ERR_OUT_OF_BLOCKS and free() == 2
    a = (ctypes.c_int32 * 1)(got[0])
    assert lazylib.kv_pool_retain(h, a, 1) == 0 and rc_of(got[0]) == 2
    assert lazylib.kv_pool_release(h, a, 1) == 0 and rc_of(got[0]) == 1 and free() == 2
    assert lazylib.kv_pool_release(h, a, 1) == 0 and rc_of(got[0]) == 0 and free() == 3
    # releasing a free block or one twice past zero is rejected and changes nothing
    assert lazylib.kv_pool_release(h, a, 1) == pk.LAZY_ERR_INVALID_ARG and free() == 3
    two = (ctypes.c_int32 * 2)(got[1], got[1])
    assert lazylib.kv_pool_release(h, two, 2) == pk.LAZY_ERR_INVALID_ARG and rc_of(got[1]) == 1
    assert lazylib.kv_pool_retain(h, a, 1) == pk.LAZY_ERR_INVALID_ARG
    bad = (ctypes.c_int32 * 1)(99)
    assert lazylib.kv_pool_retain(h, bad, 1) == pk.LAZY_ERR_INVALID_ARG
    assert lazylib.lazy_pool_destroy(h) == 0


def test_attention_argument_checks_return_before_device_use(lazylib):
    rc, h = _raw_pool(lazylib)
    assert rc == 0
    # bad scale / null pointers / inconsistent heads are rejected without touching a GPU
    assert lazylib.lazy_attn_decode(h, None, None, None, None, 1, 4, 0.0, 0, None, None, None, 0,
                                    None) == pk.LAZY_ERR_INVALID_ARG
    assert lazylib.lazy_attn_decode(h, None, None, None, None, 1, 4, 0.1, 0, None, None, None, 0,
                                    None) == pk.LAZY_ERR_INVALID_ARG
    assert lazylib.lazy_attn_prefill(h, None, None, None, None, None, None, None, 1, 4, 4, 3,
                                     0.1, None, None, None, 0, 0, None) == pk.LAZY_ERR_INVALID_ARG
    assert lazylib.lazy_attn_prefill(h, None, None, None, None, None, None, None, 1, 4, 4, 4,
                                     0.1, None, None, None, 0, 9, None) == pk.LAZY_ERR_INVALID_ARG
    assert lazylib.lazy_attn_prefill(h, None, None, None, None, None, None, None, 1, 4, 4, 4,
                                     0.1, None, None, None, 0, 5, None) == pk.LAZY_ERR_INVALID_ARG
    # the fused prefill + append needs the question k/v and both append arrays
    dummy = ctypes.c_void_p(16)
    assert lazylib.lazy_attn_prefill_append(h, dummy, None, None, dummy, dummy, None, dummy, 1, 4,
                                            4, 4, 0.1, dummy, dummy, None, 0, 0, dummy, dummy,
                                            None) == pk.LAZY_ERR_INVALID_ARG
    assert lazylib.lazy_attn_prefill_append(h, dummy, dummy, dummy, dummy, dummy, None, dummy, 1,
                                            4, 4, 4, 0.1, dummy, dummy, None, 0, 0, None, dummy,
                                            None) == pk.LAZY_ERR_INVALID_ARG
    assert lazylib.lazy_attn_prefill_append(h, dummy, dummy, dummy, dummy, dummy, None, dummy, 1,
                                            4, 4, 3, 0.1, dummy, dummy, None, 0, 0, dummy, dummy,
                                            None) == pk.LAZY_ERR_INVALID_ARG
    # the upload call checks pointers and size before any device query
    assert lazylib.lazy_copy_to_device(None, dummy, 16, None) == pk.LAZY_ERR_INVALID_ARG
    assert lazylib.lazy_copy_to_device(dummy, ctypes.c_void_p(24), 16, None) == \
        pk.LAZY_ERR_INVALID_ARG
    assert lazylib.lazy_copy_to_device(dummy, dummy, 24, None) == pk.LAZY_ERR_INVALID_ARG
    assert lazylib.lazy_copy_to_device(None, None, 0, None) == 0
    # empty batches are a no-op
    assert lazylib.lazy_attn_decode(h, None, None, None, None, 0, 4, 0.1, 0, None, None, None, 0,
                                    None) == 0
    assert lazylib.lazy_attn_prefill_append(h, None, None, None, None, None, None, None, 1, 0, 0,
                                            4, 0.1, None, None, None, 0, 0, None, None,
                                            None) == 0
    assert lazylib.lazy_pool_destroy(h) == 0


def test_alibi_mode_switch_checks(lazylib):
    rc, h = _raw_pool(lazylib)
    assert rc == 0
    mode, nq = ctypes.c_int32(-1), ctypes.c_int32(-1)
    assert lazylib.lazy_pool_position_mode(h, ctypes.byref(mode), ctypes.byref(nq)) == 0
    assert mode.value == pk.LAZY_POS_ROPE and nq.value == 0
    bad = (ctypes.c_float * 4)(0.5, -0.25, 0.125, 0.0625)    # negative slope
    assert lazylib.lazy_pool_set_alibi(h, bad, 4) == pk.LAZY_ERR_INVALID_ARG
    nan = (ctypes.c_float * 4)(0.5, float("nan"), 0.125, 0.0625)
    assert lazylib.lazy_pool_set_alibi(h, nan, 4) == pk.LAZY_ERR_INVALID_ARG
    ok = (ctypes.c_float * 4)(0.5, 0.25, 0.125, 0.0625)
    assert lazylib.lazy_pool_set_alibi(h, ok, 3) == pk.LAZY_ERR_INVALID_ARG  # not a multiple
    assert lazylib.lazy_pool_set_alibi(h, None, 4) == pk.LAZY_ERR_INVALID_ARG
    assert lazylib.lazy_pool_position_mode(h, ctypes.byref(mode), None) == 0
    assert mode.value == pk.LAZY_POS_ROPE                                      # unchanged
    assert lazylib.lazy_pool_set_alibi(h, ok, 4) == 0
    assert lazylib.lazy_pool_position_mode(h, ctypes.byref(mode), ctypes.byref(nq)) == 0
    assert mode.value == pk.LAZY_POS_ALIBI and nq.value == 4
    # attention with another head count than the slopes is rejected before any device use
    assert lazylib.lazy_attn_prefill(h, None, None, None, None, None, None, None, 1, 4, 4, 8,
                                     0.1, None, None, None, 0, 0, None) == pk.LAZY_ERR_INVALID_ARG
    assert lazylib.lazy_pool_destroy(h) == 0


def test_page_table_page_positions():
    # ALiBi page words: each page's offset field is the position of its first token
    w, cu = pk.build_page_table([[([7, 8, 9], 100, 40)], [([3], 5, 1)]], 16, page_positions=True)
    fields = [pk.lazy_unpack_page(int(x)) for x in w]
    assert [f[1] for f in fields] == [100, 116, 132, 5]
    assert [f[2] for f in fields] == [16, 16, 8, 1]
    assert list(cu) == [0, 3, 4]


def test_pack_segment_matches_the_page_word_spec():
    # one segment's words from the C helper against the oracle's independent page-word spec
    import oracle
    ids = [11, 12, 13, 2 ** 32 - 1]
    for page_positions in (0, 1):
        w, cu = pk.build_page_table([[(ids, 1000, 61)]], 16, page_positions=bool(page_positions))
        want = [oracle.pack_page(b, 1000 + (16 * i if page_positions else 0),
                                 min(16, 61 - 16 * i)) for i, b in enumerate(ids)]
        assert [int(x) for x in w] == want and list(cu) == [0, 4]
    # an empty segment, and a request without segments
    w, cu = pk.build_page_table([[([], 0, 0)], []], 16)
    assert len(w) == 0 and list(cu) == [0, 0, 0]


def test_pack_segment_rejects_bad_arguments(lazylib):
    b = (ctypes.c_uint32 * 4)(1, 2, 3, 4)
    w = (ctypes.c_uint64 * 4)()
    n = ctypes.c_int32()
    ok = lazylib.lazy_pack_segment(b, 4, 0, 64, 16, 0, w, 4, ctypes.byref(n))
    assert ok == 0 and n.value == 4
    # fewer blocks or word slots than pages
    assert lazylib.lazy_pack_segment(b, 3, 0, 64, 16, 0, w, 4, ctypes.byref(n)) == \
        pk.LAZY_ERR_INVALID_ARG
    assert lazylib.lazy_pack_segment(b, 4, 0, 64, 16, 0, w, 3, ctypes.byref(n)) == \
        pk.LAZY_ERR_INVALID_ARG
    # a page position at 2^26 (ALiBi words) or a segment offset past the field
    assert lazylib.lazy_pack_segment(b, 4, (1 << 26) - 40, 64, 16, 1, w, 4, ctypes.byref(n)) == \
        pk.LAZY_ERR_INVALID_ARG
    assert lazylib.lazy_pack_segment(b, 4, (1 << 26) - 40, 64, 16, 0, w, 4, ctypes.byref(n)) == 0
    assert lazylib.lazy_pack_segment(b, 4, 1 << 26, 64, 16, 0, w, 4, ctypes.byref(n)) == \
        pk.LAZY_ERR_INVALID_ARG
    # page sizes outside 1..64
    assert lazylib.lazy_pack_segment(b, 4, 0, 64, 65, 0, w, 4, ctypes.byref(n)) == \
        pk.LAZY_ERR_INVALID_ARG
