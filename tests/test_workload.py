"""Host checks of the seeded workload generator (shapes of the five workloads, Zipf skew)."""
import numpy as np

import workload as W


def test_bf16_round_ties_to_even_and_exactness():
    x = np.array([1.0, 1.0 + 2**-8, 1.0 + 3 * 2**-8, 1.0 + 2**-9, -2.5, 3.1415926], np.float32)
    r = W.bf16_round(x)
    assert r[0] == 1.0
    assert r[1] == 1.0                      # tie -> even (mantissa ...0)
    assert r[2] == np.float32(1.0 + 4 * 2**-8)  # tie -> even (rounds up)
    assert r[3] == 1.0
    assert r[4] == -2.5
    assert (r.view(np.uint32) & 0xFFFF == 0).all()


def test_value_streams_are_seeded_and_independent():
    a = W.normal(0, W.KIND_DOC_K, 3, (4, 2, 8), "bf16")
    b = W.normal(0, W.KIND_DOC_K, 3, (4, 2, 8), "bf16")
    c = W.normal(0, W.KIND_DOC_K, 4, (4, 2, 8), "bf16")
    assert np.array_equal(a, b) and not np.array_equal(a, c)


def test_decode_workload_shape():
    wl = W.decode_workload()
    assert wl.batch == 64 and (wl.Hq, wl.Hkv, wl.D) == (32, 8, 128)
    for r in wl.requests:
        assert len(r.docs) == 8 and len(set(r.docs)) == 8
        assert sorted(r.offsets) == [512 * i for i in range(8)]
        assert (r.priv_offset, r.priv_len, r.m) == (4096, 65, 4160)


def test_prefill_and_long_decode_shapes():
    p = W.prefill_workload()
    assert p.batch == 8 and all(len(r.docs) == 16 and r.T == 256 and r.q_pos0 == 16384
                                for r in p.requests)
    d = W.long_decode_workload()
    assert d.batch == 16 and all(len(r.docs) == 64 and r.m == 131072 and r.priv_len == 1
                                 for r in d.requests)


def test_mixed_workload_split():
    wl = W.mixed_workload(0.9)
    assert wl.batch == 128
    assert len(wl.prefill_requests()) == 32 and len(wl.decode_requests()) == 96
    for r in wl.requests:
        assert 8 <= len(r.docs) <= 32
        if r.mode == "prefill":
            assert 128 <= r.T <= 512
        else:
            assert 129 <= r.priv_len <= 513


def test_zipf_skew():
    rng = np.random.default_rng(0)
    counts = np.zeros(50)
    for _ in range(4000):
        for d in W.zipf_distinct(rng, 50, 1.0, 1):
            counts[d] += 1
    w = 1.0 / np.arange(1, 51)
    expect = 4000 * w / w.sum()
    assert abs(counts[0] / expect[0] - 1) < 0.1 and abs(counts[1] / expect[1] - 1) < 0.15
    assert counts[:5].sum() > counts[25:].sum()


def test_kv_bytes_accounting():
    from position_independent_kv_lazy_gb300 import harness as H
    # doc 0 at offsets 0 and 100 in request 0 and at 0 in request 1; doc 1 at 7 in request 1
    wl = W.custom("decode", [[(0, 0), (0, 100)], [(0, 0), (1, 7)]], doc_len=10, n_pool=2,
                  Hq=4, Hkv=2, D=64, priv=[(200, 3), (50, 5)])
    per_tok = 2 * 2 * 64 * 2
    acct = H.kv_bytes_accounting(wl)
    assert acct["resident"] == (2 * 10 + 8) * per_tok            # docs 0, 1 once + private
    assert acct["materialised"] == (3 * 10 + 8) * per_tok        # (0,0) (0,100) (1,7)
    assert acct["per_request"] == (4 * 10 + 8) * per_tok
