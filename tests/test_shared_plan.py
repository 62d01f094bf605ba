"""Host checks of the shared-segment decode planner (lazy_decode_shared_plan): every request's
pages are covered exactly once by its units, a pair unit holds two requests' copies of the same
(block, valid count) sequence, and a group of r identical segments gives r // 2 pairs."""
import collections

import numpy as np
import pytest

import position_independent_kv_lazy_gb300 as pk
import workload as W

OFF = 0x3FFFFFF << 32


def _check_plan(words, cu, plan):
    words = np.asarray(words).view(np.uint64)
    B = len(cu) - 1
    assert len(plan.cu_members) == B + 1 and plan.cu_entries[0] == 0
    assert np.all(np.diff(plan.cu_entries) > 0)
    seen = collections.defaultdict(list)
    for u in range(plan.n_units):
        a, b = plan.unit_req[2 * u], plan.unit_req[2 * u + 1]
        e = plan.entries[2 * plan.cu_entries[u]:2 * plan.cu_entries[u + 1]].reshape(-1, 2)
        seen[a].extend(int(x) for x in e[:, 0])
        if b >= 0:
            seen[b].extend(int(x) for x in e[:, 1])
            # the same blocks and valid counts; each half may have its own offsets
            assert np.array_equal(e[:, 0] & ~np.uint64(OFF), e[:, 1] & ~np.uint64(OFF))
        else:
            assert np.all(e[:, 1] == 0)
    for r in range(B):
        mine = sorted(int(x) for x in words[cu[r]:cu[r + 1]])
        assert sorted(seen.get(r, [])) == mine, r
        # the member list names exactly the units (and halves) that hold request r
        mem = plan.members[plan.cu_members[r]:plan.cu_members[r + 1]]
        ment = plan.member_entries[2 * plan.cu_members[r]:2 * plan.cu_members[r + 1]]
        for i, m in enumerate(mem):
            assert plan.unit_req[2 * (m >> 1) + (m & 1)] == r
            u = m >> 1
            assert ment[2 * i] == plan.cu_entries[u]
            assert ment[2 * i + 1] == plan.cu_entries[u + 1] - plan.cu_entries[u]
        n_units_with_r = sum(int(plan.unit_req[2 * u] == r) + int(plan.unit_req[2 * u + 1] == r)
                             for u in range(plan.n_units))
        assert len(mem) == n_units_with_r


def test_small_batch_pairs_the_shared_document():
    A = (list(range(100, 102)), 0, 32)
    reqs = [[A, ([5], 32, 10)],
            [([7, 8], 0, 20), (list(range(100, 102)), 20, 32), ([6], 52, 3)]]
    w, cu = pk.build_page_table(reqs, 16)
    plan = pk.lazy_decode_shared_plan(w, cu)
    _check_plan(w, cu, plan)
    pairs = [u for u in range(plan.n_units) if plan.unit_req[2 * u + 1] >= 0]
    assert len(pairs) == 1
    u = pairs[0]
    assert sorted(plan.unit_req[2 * u:2 * u + 2]) == [0, 1]
    assert plan.cu_entries[u + 1] - plan.cu_entries[u] == 2
    # the two halves carry their own offsets (0 and 20)
    e = plan.entries[2 * plan.cu_entries[u]:2 * plan.cu_entries[u + 1]].reshape(-1, 2)
    assert {int(x) >> 32 & 0x3FFFFFF for x in e[:, 0]} | \
        {int(x) >> 32 & 0x3FFFFFF for x in e[:, 1]} == {0, 20}


def test_group_of_r_members_gives_r_over_2_pairs():
    D = (list(range(50, 54)), 0, 64)
    for r in range(1, 8):
        reqs = [[([1000 + b], 0, 16), (D[0], 16 + 7 * b, 64)] for b in range(r)]
        w, cu = pk.build_page_table(reqs, 16)
        plan = pk.lazy_decode_shared_plan(w, cu)
        _check_plan(w, cu, plan)
        pairs = sum(int(plan.unit_req[2 * u + 1] >= 0) for u in range(plan.n_units))
        assert pairs == r // 2
        # r private tails (each its request's merged single unit) + the document's units; a
        # document held by one request joins that request's single unit
        assert plan.n_units == r + ((r + 1) // 2 if r > 1 else 0)
        assert plan.n_entries == r + 4 * ((r + 1) // 2)


def test_same_first_page_different_segments_are_not_paired():
    # segments that share their first block and length but differ later land in one bucket of
    # the planner's index and must still be told apart word by word
    reqs = [[([100, 101, 102], 0, 48)], [([100, 101, 103], 0, 48)], [([100, 101, 102], 7, 48)],
            [([100, 101, 103], 9, 48)], [([100, 101, 102], 50, 40)]]
    w, cu = pk.build_page_table(reqs, 16)
    plan = pk.lazy_decode_shared_plan(w, cu)
    _check_plan(w, cu, plan)
    pairs = sorted(tuple(plan.unit_req[2 * u:2 * u + 2]) for u in range(plan.n_units)
                   if plan.unit_req[2 * u + 1] >= 0)
    # (0, 2) share [100, 101, 102] with 16 valid keys on every page, (1, 3) [100, 101, 103];
    # request 4's last page holds 8 keys, so its words differ: alone
    assert pairs == [(0, 2), (1, 3)]


def test_repeated_document_in_one_request_pairs_with_itself():
    D = (list(range(10, 12)), 0, 32)
    reqs = [[(D[0], 0, 32), ([3], 32, 5), (D[0], 37, 32)]]
    w, cu = pk.build_page_table(reqs, 16)
    plan = pk.lazy_decode_shared_plan(w, cu)
    _check_plan(w, cu, plan)
    u = [u for u in range(plan.n_units) if plan.unit_req[2 * u + 1] >= 0]
    assert len(u) == 1 and list(plan.unit_req[2 * u[0]:2 * u[0] + 2]) == [0, 0]
    assert list(plan.members[plan.cu_members[0]:plan.cu_members[1]]).count(2 * u[0]) == 1
    assert list(plan.members[plan.cu_members[0]:plan.cu_members[1]]).count(2 * u[0] + 1) == 1


def test_empty_batch_and_empty_requests():
    w, cu = pk.build_page_table([], 16)
    plan = pk.lazy_decode_shared_plan(w, cu)
    assert plan.n_units == 0 and list(plan.cu_members) == [0]
    reqs = [[], [([4, 5], 0, 20)], []]
    w, cu = pk.build_page_table(reqs, 16)
    plan = pk.lazy_decode_shared_plan(w, cu)
    _check_plan(w, cu, plan)
    assert list(plan.cu_members) == [0, 0, 1, 1]


def test_alibi_page_positions_cut_at_block_jumps():
    # ALiBi words carry each page's first position, which runs on through the whole context;
    # documents are cut where the block id stops advancing by one
    D = (list(range(60, 63)), 0, 40)
    reqs = [[([1], 0, 16), (D[0], 16, 40)], [(D[0], 300, 40), ([2], 340, 8)],
            [([1], 1000, 16), (D[0], 1016, 40)]]
    w, cu = pk.build_page_table(reqs, 16, page_positions=True)
    plan = pk.lazy_decode_shared_plan(w, cu, page_positions=True)
    _check_plan(w, cu, plan)
    # D is shared by all three requests (one pair, one leftover next to it); [1] by requests 0
    # and 2 (one pair); [2] only by request 1 (its merged single unit)
    pairs = [tuple(plan.unit_req[2 * u:2 * u + 2]) for u in range(plan.n_units)
             if plan.unit_req[2 * u + 1] >= 0]
    assert sorted(pairs) == [(0, 1), (0, 2)]
    assert plan.n_units == 4
    # a document whose blocks follow another's in the context joins it in one segment
    E = (list(range(63, 65)), 0, 32)
    reqs = [[(D[0], 0, 48), (E[0], 48, 32)], [(D[0], 100, 48)]]
    w, cu = pk.build_page_table(reqs, 16, page_positions=True)
    plan = pk.lazy_decode_shared_plan(w, cu, page_positions=True)
    _check_plan(w, cu, plan)
    assert all(plan.unit_req[2 * u + 1] < 0 for u in range(plan.n_units))
    # the same tables read as RoPE words (one offset per segment) cut at every page
    plan = pk.lazy_decode_shared_plan(w, cu)
    _check_plan(w, cu, plan)
    assert sum(int(plan.unit_req[2 * u + 1] >= 0) for u in range(plan.n_units)) == 3


def test_decreasing_cu_pages_is_rejected():
    w, cu = pk.build_page_table([[([4], 0, 16)], [([5], 0, 16)]], 16)
    bad = cu.copy()
    bad[1] = 2
    bad[2] = 1
    with pytest.raises(pk.LazyError):
        pk.lazy_decode_shared_plan(w, bad)


@pytest.mark.parametrize("align", [False, True])
def test_decode_workload_plan(align):
    # decode_b64's documents: 512 references to 227 documents, 356 of them to 71 shared ones
    wl = W.decode_workload()
    blocks = {d: list(range(1000 * d, 1000 * d + 32)) for r in wl.requests for d in r.docs}
    reqs = []
    for r in wl.requests:
        s = [(blocks[d], o, wl.doc_len) for d, o in zip(r.docs, r.offsets)]
        s.append((list(range(10 ** 7 + 100 * r.index, 10 ** 7 + 100 * r.index + 5)),
                  r.priv_offset, r.priv_len))
        reqs.append(s)
    w, cu = pk.build_page_table(reqs, 16, align_shared=align)
    plan = pk.lazy_decode_shared_plan(w, cu)
    _check_plan(w, cu, plan)
    refs = collections.Counter(d for r in wl.requests for d in r.docs)
    # shared documents: ceil(n / 2) units each; every request's private tail and the documents
    # only it holds: one merged single unit per request
    want_doc_units = sum((n + 1) // 2 for n in refs.values() if n > 1)
    assert plan.n_units == want_doc_units + len(wl.requests)
    lone = sum(1 for n in refs.values() if n == 1)
    assert plan.n_entries == 32 * (want_doc_units + lone) + 5 * len(wl.requests)
