"""The cache hit-rate simulator (the pages' "Main contributions" item 2 and cache-efficiency
results): hand-computed streams, LRU eviction, and the ordering that holds by construction."""
import pytest

import workload as W
from position_independent_kv_lazy_gb300 import cachesim as C

L = 10  # tokens per document


def test_hand_computed_unlimited_budget():
    # r1 [A,B]: all miss. r2 [B,A]: agnostic hits both; positional (B,0),(A,L) are new; prefix
    # [B] is new. r3 [A,B]: every design hits both. r4 [A,C]: A hits (same offset, same prefix),
    # C misses everywhere.
    A, B, Cd = 0, 1, 2
    stream = [[A, B], [B, A], [A, B], [A, Cd]]
    r = C.compare(stream, L, float("inf"))
    assert r["agnostic"].hit_tokens == 5 * L
    assert r["positional"].hit_tokens == 3 * L
    assert r["prefix"].hit_tokens == 3 * L
    assert all(x.total_tokens == 8 * L for x in r.values())


def test_prefix_breaks_after_first_mismatch():
    # [A,B,C] then [D,B,C]: B and C sit at the same offsets (positional hits 2 docs) but behind a
    # different first document (prefix hits nothing)
    stream = [[0, 1, 2], [3, 1, 2]]
    r = C.compare(stream, L, float("inf"))
    assert r["positional"].hit_tokens == 2 * L
    assert r["prefix"].hit_tokens == 0
    assert r["agnostic"].hit_tokens == 2 * L


def test_lru_eviction_order():
    c = C.LRUCache(budget_tokens=3 * L)
    for k in "abc":
        c.insert(k, L)
    assert c.hit("a")          # a becomes most recent
    c.insert("d", L)           # evicts b, the least recently used
    assert not c.hit("b") and c.hit("a") and c.hit("c") and c.hit("d")
    c.insert("big", 4 * L)     # larger than the budget: not cached, nothing evicted
    assert not c.hit("big") and len(c) == 3


def test_budget_counts_tokens_per_copy():
    # budget for 2 documents: the positional design keeps one copy per offset, so one document
    # at two offsets fills it; the agnostic design keeps one copy
    stream = [[0, 1], [1, 0], [0, 1], [1, 0]]
    r = C.compare(stream, L, 2 * L)
    assert r["agnostic"].hit_tokens == 6 * L          # both docs stay resident after r1
    assert r["positional"].hit_tokens == 0            # 4 distinct (doc, offset) keys cycle


@pytest.mark.parametrize("alpha", [0.6, 1.2])
def test_unlimited_budget_ordering(alpha):
    # with no eviction every positional hit is an agnostic hit and every prefix hit a positional
    # hit (a matching prefix fixes the offset)
    stream = W.request_stream(400, 300, 8, alpha, seed=1)
    r = C.compare(stream, L, float("inf"))
    assert r["agnostic"].hit_tokens >= r["positional"].hit_tokens >= r["prefix"].hit_tokens
    assert r["agnostic"].hit_tokens > r["positional"].hit_tokens


def test_request_stream_draws_distinct_zipf_docs():
    s = W.request_stream(200, 50, 8, 1.0, seed=3)
    assert len(s) == 200 and all(len(set(r)) == 8 and max(r) < 50 for r in s)
    assert s == W.request_stream(200, 50, 8, 1.0, seed=3)  # seeded
