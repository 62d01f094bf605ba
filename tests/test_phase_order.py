"""Host checks of lazy_order_segments (the phase-aligned order of each request's segments for the
split-KV decode): valid permutations with pinned segments last, unchanged order for requests
whose segments differ in length, shared segments brought to nearby read steps, and, under an
independent lockstep model of the decode's warps and an LRU cache, less modelled DRAM traffic
than the index-aligned order on the decode-step workload's structure."""
import collections

import numpy as np
import pytest

import position_independent_kv_lazy_gb300 as pk
import workload as W


def _order(requests, units, ranges):
    return pk.order_segments_by_phase(requests, units, ranges, 16, pin_last=True)


def test_permutations_with_private_tail_last(lazylib):
    rng = np.random.default_rng(1)
    reqs = []
    for b in range(20):
        n = int(rng.integers(1, 9))
        segs = [([int(d) * 100], int(rng.integers(0, 9999)), 64) for d in rng.integers(0, 12, n)]
        segs.append(([5000 + b], 777, int(rng.integers(1, 40))))   # private tail
        reqs.append(segs)
    out = _order(reqs, 8, 1824)
    for a, b in zip(reqs, out):
        assert sorted(map(repr, a)) == sorted(map(repr, b))
        assert b[-1] == a[-1]


def test_requests_with_mixed_lengths_keep_their_order(lazylib):
    reqs = [[([1], 0, 64), ([2], 64, 32), ([3], 96, 64), ([9], 200, 5)],
            [([2], 0, 32), ([1], 32, 64), ([8], 96, 5)]]
    out = _order(reqs, 8, 100)
    assert out == reqs


def _step(flat_index, n_total, ranges):
    # local step of flattened page x in the equal-range partition (ranges side by side)
    w = (flat_index * ranges) // n_total
    return flat_index - (w * n_total) // ranges


def test_shared_segment_lands_on_nearby_steps(lazylib):
    # 6 requests x (4 documents of 4 pages + a 1-page tail), document 7 in every request, one
    # unit per request, 3 ranges: the shared document should be read at close steps everywhere
    rng = np.random.default_rng(2)
    reqs = []
    for b in range(6):
        docs = [7] + [int(d) for d in rng.choice(np.arange(10, 40), 3, replace=False)]
        rng.shuffle(docs)
        reqs.append([([d], 0, 64) for d in docs] + [([100 + b], 0, 16)])
    units, ranges = 1, 3
    out = _order(reqs, units, ranges)
    n_total = units * sum(4 * 4 + 1 for _ in out)
    steps = []
    base = 0
    for segs in out:
        pos = 0
        for ids, _, length in segs:
            if ids[0] == 7:
                steps.append(_step(base + pos, n_total, ranges))
            pos += length // 16
        base += pos * units
    R = n_total / ranges

    def spread(st):
        return max(min(abs(a - b), R - abs(a - b)) for a in st for b in st)

    # the best spread any placement achieves (each request: document 7 in one of its 4 slots)
    import itertools
    phases = [[(17 * b + 4 * k) % R for k in range(4)] for b in range(6)]
    best = min(spread(c) for c in itertools.product(*phases))
    assert spread(steps) <= best + 1e-9, (steps, best)


def _lockstep_lru_bytes(orders, doc_pages, priv_pages, units, ranges, cache_pages):
    # an independent model: every range reads its next page at each step; LRU cache of pages
    flat = []
    for b, order in enumerate(orders):
        pages = [("d", d, p) for d in order for p in range(doc_pages)]
        pages += [("p", b, p) for p in range(priv_pages[b])]
        for h in range(units):
            flat += [(pg, h) for pg in pages]
    n = len(flat)
    bounds = [w * n // ranges for w in range(ranges + 1)]
    lru = collections.OrderedDict()
    misses = 0
    for t in range(max(bounds[w + 1] - bounds[w] for w in range(ranges))):
        for w in range(ranges):
            x = bounds[w] + t
            if x >= bounds[w + 1]:
                continue
            k = flat[x]
            if k in lru:
                lru.move_to_end(k)
            else:
                misses += 1
                lru[k] = None
                if len(lru) > cache_pages:
                    lru.popitem(last=False)
    return misses


def test_phase_order_cuts_modelled_dram_traffic_on_decode_b64(lazylib):
    wl = W.decode_workload()
    units, ranges = 8, 1824              # 32/8 heads, 152 SMs x 3 CTAs x 4 warps
    segs = [[([d], o, wl.doc_len) for d, o in zip(r.docs, r.offsets)] +
            [([10_000 + r.index], r.priv_offset, r.priv_len)] for r in wl.requests]
    aligned = pk.align_shared_segments(segs)
    phased = _order(segs, units, ranges)
    priv = [-(-r.priv_len // 16) for r in wl.requests]
    cache = int(126e6 // 8192)
    doc_order = lambda oo: [[s[0][0] for s in req[:-1]] for req in oo]  # noqa: E731
    m_al = _lockstep_lru_bytes(doc_order(aligned), wl.doc_len // 16, priv, units, ranges, cache)
    m_ph = _lockstep_lru_bytes(doc_order(phased), wl.doc_len // 16, priv, units, ranges, cache)
    unique = (len(wl.used_docs()) * (wl.doc_len // 16) + sum(priv)) * units
    assert m_ph < 0.9 * m_al and m_ph < 1.1 * unique, (m_al, m_ph, unique)


def test_order_segments_rejects_bad_arguments(lazylib):
    import ctypes
    cu = (ctypes.c_int32 * 2)(0, 1)
    key = (ctypes.c_int64 * 1)(5)
    pages = (ctypes.c_int32 * 1)(-1)
    pin = (ctypes.c_uint8 * 1)(0)
    perm = (ctypes.c_int32 * 1)()
    assert lazylib.lazy_order_segments(1, cu, key, pages, pin, 8, 10, perm) == \
        pk.LAZY_ERR_INVALID_ARG
    pages[0] = 4
    assert lazylib.lazy_order_segments(1, cu, key, pages, pin, 0, 10, perm) == \
        pk.LAZY_ERR_INVALID_ARG
    assert lazylib.lazy_order_segments(1, cu, key, pages, pin, 8, 10, perm) == 0
    assert perm[0] == 0
