"""Host checks of align_shared_segments: a per-request permutation that puts a shared segment
at the same index in every request using it, and leaves the packed page words of each request
the same multiset."""
import collections

import numpy as np

import position_independent_kv_lazy_gb300 as pk
import workload as W


def _segs(blocks, n=2):
    return (list(range(blocks, blocks + n)), 0, 16 * n)


def _perm_ok(a, b):
    return sorted(map(repr, a)) == sorted(map(repr, b))


def test_permutation_and_alignment_small():
    A, B, C = _segs(100), _segs(200), _segs(300)
    reqs = [[_segs(1), A, B, _segs(2)], [B, _segs(3), A], [_segs(4), C, A, B], [C, _segs(5)]]
    out = pk.align_shared_segments(reqs)
    for r, o in zip(reqs, out):
        assert _perm_ok(r, o)
    idx = lambda seg: {o.index(seg) for o in out if seg in o}
    assert len(idx(A)) == 1 and len(idx(B)) == 1   # A, B shared by 3 requests each
    # C (2 requests) has no index free in both once A and B are placed: it keeps one request's
    # choice and the other request's first free index
    assert idx(C) <= {0, 1, 2, 3}


def test_repeated_segment_in_one_request():
    A = _segs(100)
    reqs = [[A, _segs(1), A], [_segs(2), A]]
    out = pk.align_shared_segments(reqs)
    for r, o in zip(reqs, out):
        assert _perm_ok(r, o)
    assert out[0].index(A) == out[1].index(A)


def test_decode_workload_alignment_and_words():
    wl = W.decode_workload()
    blocks, nxt = {}, 0
    for d in sorted({d for r in wl.requests for d in r.docs}):
        blocks[d] = list(range(nxt, nxt + wl.doc_len // 16))
        nxt += wl.doc_len // 16
    reqs = [[(blocks[d], o, wl.doc_len) for d, o in zip(r.docs, r.offsets)] for r in wl.requests]
    out = pk.align_shared_segments(reqs)
    cnt = collections.Counter(tuple(s[0]) for r in reqs for s in r)
    pos = collections.defaultdict(collections.Counter)
    for o in out:
        for i, s in enumerate(o):
            pos[tuple(s[0])][i] += 1
    multi = [k for k, c in cnt.items() if c > 1]
    at_slot = sum(max(pos[k].values()) for k in multi)
    assert at_slot >= 0.9 * sum(cnt[k] for k in multi)
    w0, cu0 = pk.build_page_table(reqs, 16)
    w1, cu1 = pk.build_page_table(reqs, 16, align_shared=True)
    assert np.array_equal(cu0, cu1)
    for b in range(len(reqs)):
        assert sorted(w0[cu0[b]:cu0[b + 1]].tolist()) == sorted(w1[cu1[b]:cu1[b + 1]].tolist())


def test_degenerate_batches():
    assert pk.align_shared_segments([]) == []
    one = [[_segs(1), _segs(2), _segs(3)]]
    assert pk.align_shared_segments(one) == one              # nothing shared: order kept
    reqs = [[], [_segs(7)], []]
    assert pk.align_shared_segments(reqs) == reqs             # empty requests stay empty
    uniq = [[_segs(10 * b + i) for i in range(3)] for b in range(4)]
    assert pk.align_shared_segments(uniq) == uniq             # all unique: order kept
