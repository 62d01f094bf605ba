"""Pins of the fp64 oracle against facts fixed by the mathematics and by the pages.

Each test names what it pins. Sources: "LazyAttention: Efficient Retrieval-Augmented Generation
with Deferred Positional Encoding" (technical summaries): "Mathematical equivalence" (RoPE scores
depend only on n - m, lazy == materialised), "Core concept: deferred positional encoding",
decoding section (bit-packed block id + offset). Conventions the summaries leave open are pinned
by closed forms so that a dropped term, a wrong sign, a wrong pairing or a wrong index fails.
"""
import math

import numpy as np
import pytest

import oracle
import workload as W


def _polar(r, phi):
    return np.array([r * math.cos(phi), r * math.sin(phi)])


# ---------------------------------------------------------------- rotation itself
@pytest.mark.parametrize("pos", [0, 1, 7, -3, 131072])
def test_rope_d2_is_planar_rotation(pos):
    # D=2: theta_0 = base^0 = 1 for any base, so R(p) turns the vector by p radians.
    r, phi = 1.7, 0.4
    x = _polar(r, phi)
    y = oracle.rope(x, pos, base=500000.0)
    assert np.allclose(y, _polar(r, phi + pos), atol=1e-9)


def test_rope_d4_pairs_and_frequencies():
    # D=4, half-split: pairs are (0,2) with theta=1 and (1,3) with theta=base^(-1/2).
    base, p = 10000.0, 5
    x = np.array([1.0, 0.0, 0.0, 0.0])
    y = oracle.rope(x, p, base)
    assert np.allclose(y, [math.cos(p), 0.0, math.sin(p), 0.0], atol=1e-12)
    x = np.array([0.0, 2.0, 0.0, 0.0])
    y = oracle.rope(x, p, base)
    th = base ** -0.5
    assert np.allclose(y, [0.0, 2 * math.cos(p * th), 0.0, 2 * math.sin(p * th)], atol=1e-12)


def test_rope_norm_composition_inverse():
    rng = np.random.default_rng(1)
    x = rng.standard_normal(128)
    for a, b in [(3, 11), (-40, 1000), (123456, 7)]:
        ra = oracle.rope(x, a, 5e5)
        assert abs(np.linalg.norm(ra) - np.linalg.norm(x)) < 1e-12
        assert np.allclose(oracle.rope(ra, b, 5e5), oracle.rope(x, a + b, 5e5), atol=1e-9)
        assert np.allclose(oracle.rope(ra, -a, 5e5), x, atol=1e-9)


# ---------------------------------------------------------------- attention closed forms
def test_d2_two_keys_worked_example():
    # Hand-worked: D=2, scale 1/sqrt(2), q=(1,0) at m=0, k1=(1,0) at p=0, k2=(1,0) at p=1,
    # v1=(1,0), v2=(0,1).  s1 = 1/sqrt2, s2 = cos(1)/sqrt2 (key turned by 1 rad).
    s1, s2 = 1 / math.sqrt(2), math.cos(1.0) / math.sqrt(2)
    e1, e2 = math.exp(s1), math.exp(s2)
    want_out = [e1 / (e1 + e2), e2 / (e1 + e2)]
    want_lse = math.log(e1 + e2)
    k = np.array([[1.0, 0.0], [1.0, 0.0]])
    v = np.array([[1.0, 0.0], [0.0, 1.0]])
    out, lse = oracle.attend_materialised(k, v, [0, 1], [0, 0], np.array([[[1.0, 0.0]]]), [0],
                                          base=10000.0, scale=1 / math.sqrt(2))
    assert np.allclose(out[0, 0], want_out, atol=1e-14)
    assert abs(lse[0, 0] - want_lse) < 1e-14


def test_d2_score_depends_on_relative_position():
    # s = |q||k| cos(phi_k - phi_q + (p - m)) / sqrt(2) in D=2; single key => lse = s, out = v.
    rq, fq, rk, fk = 1.3, 0.2, 0.8, -1.1
    for p, m in [(0, 0), (5, 9), (100, 3), (70000, 131072)]:
        out, lse = oracle.attend_materialised(_polar(rk, fk)[None], np.array([[2.0, -3.0]]), [p], [0],
                                              _polar(rq, fq)[None, None], [m], base=5e5,
                                              scale=1 / math.sqrt(2))
        s = rq * rk * math.cos(fk - fq + (p - m)) / math.sqrt(2)
        assert abs(lse[0, 0] - s) < 1e-9
        assert np.allclose(out[0, 0], [2.0, -3.0], atol=1e-15)


def test_q_zero_gives_uniform_weights_over_visible_keys():
    rng = np.random.default_rng(2)
    D, n = 16, 11
    k = rng.standard_normal((n, D)); v = rng.standard_normal((n, D))
    pos = np.arange(n) + 100
    causal = np.array([0] * 5 + [1] * 6, np.uint8)      # last 6 keys causal at 105..110
    q = np.zeros((3, 2, D))
    qpos = np.array([104, 107, 110])
    out, lse = oracle.attend_materialised(k, v, pos, causal, q, qpos, base=1e4, scale=0.25)
    for i, m in enumerate(qpos):
        vis = (causal == 0) | (pos <= m)
        for g in range(2):
            assert np.allclose(out[i, g], v[vis].mean(0), atol=1e-14)
            assert abs(lse[i, g] - math.log(vis.sum())) < 1e-14


def test_constant_values_give_constant_output():
    rng = np.random.default_rng(3)
    D, n = 32, 20
    v = np.full((n, D), 0.625)
    out, _ = oracle.attend_materialised(rng.standard_normal((n, D)), v, np.arange(n), np.zeros(n),
                                        rng.standard_normal((4, 1, D)), [19, 20, 40, 1000],
                                        base=1e4, scale=1 / math.sqrt(D))
    assert np.allclose(out, 0.625, atol=1e-14)


def test_fully_masked_row():
    out, lse = oracle.attend_materialised(np.ones((2, 4)), np.ones((2, 4)), [10, 11], [1, 1],
                                          np.ones((1, 1, 4)), [5], base=1e4, scale=0.5)
    assert lse[0, 0] == -np.inf and np.all(out == 0)


def test_gqa_mapping_is_consecutive():
    # Hq=4, Hkv=2: q heads 0,1 read kv head 0, heads 2,3 read kv head 1 (h // (Hq/Hkv)).
    wl = W.custom("decode", [[(0, 0)]], doc_len=16, n_pool=1, Hq=4, Hkv=2, D=16, dtype="fp32",
                  priv=[(16, 3)])

    class Src:
        def doc_k(self, d): return wl.doc_k(d)
        def doc_v(self, d):
            v = np.empty((16, 2, 16)); v[:, 0] = 1.5; v[:, 1] = -2.0; return v
        def q(self, b): return wl.q(b)
        def new_k(self, b): return wl.new_k(b)
        def new_v(self, b):
            v = np.empty((3, 2, 16)); v[:, 0] = 1.5; v[:, 1] = -2.0; return v

    out, _ = oracle.attend_request(wl, 0, src=Src())
    assert np.allclose(out[0, :2], 1.5) and np.allclose(out[0, 2:], -2.0)


# ---------------------------------------------------------------- the pages' equivalence claim
def _small_prefill():
    return W.custom("prefill", [[(0, 0), (1, 40), (0, 90)], [(2, 7), (1, 300)]], doc_len=24,
                    n_pool=3, Hq=4, Hkv=2, D=16, dtype="fp32", base=1e4, T=[5, 9],
                    q_pos0=[130, 400])


def test_lazy_form_equals_materialised():
    wl = _small_prefill()
    for b in range(wl.batch):
        a = oracle.attend_request(wl, b, form="A")
        bb = oracle.attend_request(wl, b, form="B")
        assert np.allclose(a[0], bb[0], atol=1e-12, rtol=0)
        assert np.allclose(a[1], bb[1], atol=1e-12, rtol=0)


def test_bruteforce_agrees():
    rng = np.random.default_rng(4)
    D, base, scale = 8, 100.0, 1 / math.sqrt(8)
    keys = []
    for i in range(30):
        keys.append((int(rng.integers(0, 60)), 0, rng.standard_normal(D), rng.standard_normal(D)))
    for i in range(8):
        keys.append((60 + i, 1, rng.standard_normal(D), rng.standard_normal(D)))
    qs = [(60 + i, rng.standard_normal(D)) for i in range(8)]
    ref = oracle.attend_bruteforce(keys, qs, base=base, scale=scale)
    k = np.array([x[2] for x in keys]); v = np.array([x[3] for x in keys])
    out, lse = oracle.attend_materialised(k, v, [x[0] for x in keys], [x[1] for x in keys],
                                          np.array([x[1] for x in qs])[:, None, :],
                                          [x[0] for x in qs], base=base, scale=scale)
    for i, (o, l) in enumerate(ref):
        assert np.allclose(out[i, 0], o, atol=1e-12)
        assert abs(lse[i, 0] - l) < 1e-12


def test_offset_zero_reduces_to_textbook_rope_attention():
    # Docs laid end to end from position 0 followed by the question == ordinary RoPE causal
    # attention over the concatenated sequence.
    L, T = 20, 6
    wl = W.custom("prefill", [[(0, 0), (1, L), (2, 2 * L)]], doc_len=L, n_pool=3, Hq=2, Hkv=1,
                  D=32, dtype="fp32", base=10000.0, T=[T], q_pos0=[3 * L])
    out, lse = oracle.attend_request(wl, 0)
    k = np.concatenate([wl.doc_k(0), wl.doc_k(1), wl.doc_k(2), wl.new_k(0)])[:, 0]
    v = np.concatenate([wl.doc_v(0), wl.doc_v(1), wl.doc_v(2), wl.new_v(0)])[:, 0]
    for g in range(2):
        o, l = oracle.textbook_rope_attention(wl.q(0)[:, g], k, v, np.arange(3 * L, 3 * L + T),
                                              10000.0, wl.sm_scale)
        assert np.allclose(out[:, g], o, atol=1e-12)
        assert np.allclose(lse[:, g], l, atol=1e-12)


@pytest.mark.parametrize("c", [1, 12345, 1000000])
def test_shift_invariance(c):
    wl = _small_prefill()
    a = oracle.attend_request(wl, 1)
    for r in wl.requests:
        r.offsets = [o + c for o in r.offsets]
        r.q_pos0 += c
    b = oracle.attend_request(wl, 1)
    assert np.allclose(a[0], b[0], atol=1e-8) and np.allclose(a[1], b[1], atol=1e-8)


def test_segment_order_does_not_matter():
    wl = _small_prefill()
    a = oracle.attend_request(wl, 0)
    r = wl.requests[0]
    r.docs, r.offsets = r.docs[::-1], r.offsets[::-1]
    b = oracle.attend_request(wl, 0)
    assert np.allclose(a[0], b[0], atol=1e-12) and np.allclose(a[1], b[1], atol=1e-12)


def test_same_doc_at_two_offsets_acts_like_two_copies():
    # request 0 of _small_prefill holds doc 0 at offsets 0 and 90; replace the second occurrence
    # by a distinct doc id whose arrays are a copy of doc 0.
    wl = _small_prefill()
    a = oracle.attend_request(wl, 0)

    class Src:
        def doc_k(self, d): return wl.doc_k(0 if d == 9 else d)
        def doc_v(self, d): return wl.doc_v(0 if d == 9 else d)
        def q(self, b): return wl.q(b)
        def new_k(self, b): return wl.new_k(b)
        def new_v(self, b): return wl.new_v(b)

    wl.requests[0].docs = [0, 1, 9]
    b = oracle.attend_request(wl, 0, src=Src())
    assert np.allclose(a[0], b[0], atol=0) and np.allclose(a[1], b[1], atol=0)


def test_sampling_matches_full_computation():
    wl = _small_prefill()
    full = oracle.attend_request(wl, 1)
    part = oracle.attend_request(wl, 1, kv_heads=[1], queries=[2, 7])
    assert np.allclose(part[0][[2, 7]][:, 2:], full[0][[2, 7]][:, 2:], atol=0)
    assert np.isnan(part[0][0]).all() and np.isnan(part[0][2][:2]).all()


# ---------------------------------------------------------------- stored-key form (S)
# The cache keeps each document's keys once, rotated at their document-local positions, in its
# own element type ("Core concept: deferred positional encoding"). Form S writes that storage
# rounding out; with exact storage it is form A.
@pytest.mark.parametrize("x,want", [
    (1.0 + 2 ** -8, 1.0),                         # halfway to 1 + 2^-7: ties to even (down)
    (1.0 + 3 * 2 ** -8, 1.0 + 2 ** -6),           # halfway between 1 + 2^-7 and 1 + 2^-6 (up)
    (1.0 + 2 ** -8 + 2 ** -30, 1.0 + 2 ** -7),    # just above halfway
    (-(1.0 + 3 * 2 ** -8), -(1.0 + 2 ** -6)),     # sign symmetry
    (0.1, 205 * 2.0 ** -11),                      # 0.1 in [2^-4, 2^-3): spacing 2^-11, 204.8 -> 205
    (3 * 2.0 ** -135, 2.0 ** -133),               # below 2^-126 the spacing stays 2^-133
    ((2 - 2 ** -7) * 2.0 ** 127, (2 - 2 ** -7) * 2.0 ** 127),   # largest finite bf16
    ((2 - 2 ** -8) * 2.0 ** 127, math.inf),       # halfway to 2^128 rounds to even -> overflow
    (0.0, 0.0)])
def test_round_bf16_hand_values(x, want):
    assert oracle.round_bf16(x) == want


def test_round_bf16_matches_bit_level_rounding():
    # an independent implementation (integer rounding of the float32 bit pattern)
    rng = np.random.default_rng(7)
    x = np.concatenate([rng.standard_normal(20000).astype(np.float32),
                        (rng.standard_normal(2000) * 1e-30).astype(np.float32),
                        (rng.standard_normal(2000) * 1e30).astype(np.float32)])
    want = W.bf16_round(x).astype(np.float64)
    got = np.array([oracle.round_bf16(float(t)) for t in x])
    assert np.array_equal(got, want)


def _stored_case(rng, D=16, n_docs=4, L=5, nq=3, G=2, bf16_inputs=True):
    k = rng.standard_normal((n_docs * L, D))
    v = rng.standard_normal((n_docs * L, D))
    q = rng.standard_normal((nq, G, D))
    if bf16_inputs:
        k, v, q = (W.bf16_round(a.astype(np.float32)).astype(np.float64) for a in (k, v, q))
    off = np.repeat(rng.integers(0, 5000, n_docs), L)
    loc = np.tile(np.arange(L), n_docs)
    q_pos = np.array([6000, 6100, 7777])[:nq]
    return k, v, off, loc, q, q_pos


def test_stored_form_with_exact_storage_is_form_a():
    rng = np.random.default_rng(8)
    k, v, off, loc, q, q_pos = _stored_case(rng)
    n = len(off)
    caus = np.zeros(n, np.uint8)
    oa, la = oracle.attend_materialised(k, v, off + loc, caus, q, q_pos, base=1e4, scale=0.25)
    for stored in (np.ones(n, np.uint8), np.zeros(n, np.uint8)):
        os_, ls = oracle.attend_stored(k, v, off, loc, stored, caus, q, q_pos, base=1e4,
                                       scale=0.25, store="exact")
        assert np.abs(os_ - oa).max() < 1e-12 and np.abs(ls - la).max() < 1e-12


def test_stored_form_rounds_before_the_offset_rotation():
    # keys at local position 0 with bf16-exact raw values: R(0) k = k is already a bf16 value, so
    # the cache's copy is exact and S equals A, whatever the offsets. Rounding R(o + j) k instead
    # (storage after the offset) would not be exact and fails this.
    rng = np.random.default_rng(9)
    k, v, off, loc, q, q_pos = _stored_case(rng, L=1, n_docs=12)
    n = len(off)
    caus = np.zeros(n, np.uint8)
    oa, la = oracle.attend_materialised(k, v, off, caus, q, q_pos, base=5e5, scale=0.25)
    os_, ls = oracle.attend_stored(k, v, off, np.zeros(n), np.ones(n, np.uint8), caus, q, q_pos,
                                   base=5e5, scale=0.25, store="bf16")
    assert np.abs(os_ - oa).max() < 1e-12 and np.abs(ls - la).max() < 1e-12


def test_stored_form_d2_worked_example():
    # D=2 (theta_0 = 1): raw key (1, 0) stored at local position 1 is
    # round_bf16((cos 1, sin 1)) = (0.5390625, 0.83984375) (hand-rounded: 138/256 and 215/256);
    # attended at offset 2 by a query (1, 0) at m = 3, the score is
    # scale * (R(3) q) . (R(2) stored) = scale * (cos 1 * 0.5390625 + sin 1 * 0.83984375);
    # with a single key, lse = that score and out = v.
    scale = 1 / math.sqrt(2)
    want = scale * (math.cos(1.0) * 0.5390625 + math.sin(1.0) * 0.83984375)
    out, lse = oracle.attend_stored(np.array([[1.0, 0.0]]), np.array([[0.25, -2.0]]), [2], [1],
                                    [1], [0], np.array([[[1.0, 0.0]]]), [3], base=10.0,
                                    scale=scale, store="bf16")
    assert abs(lse[0, 0] - want) < 1e-14
    assert np.allclose(out[0, 0], [0.25, -2.0], atol=1e-15)
    # the exact form differs: cos(1)^2 + sin(1)^2 = 1
    _, la = oracle.attend_materialised(np.array([[1.0, 0.0]]), np.array([[0.25, -2.0]]), [3], [0],
                                       np.array([[[1.0, 0.0]]]), [3], base=10.0, scale=scale)
    assert abs(la[0, 0] - scale) < 1e-14 and abs(lse[0, 0] - scale) > 1e-4


def test_stored_form_differs_from_a_by_the_storage_rounding_only():
    # fp32 storage moves lse by ~1e-7, bf16 storage by ~1e-3 on a 20-key context
    rng = np.random.default_rng(10)
    k, v, off, loc, q, q_pos = _stored_case(rng, D=64)
    n = len(off)
    caus = np.zeros(n, np.uint8)
    st = np.ones(n, np.uint8)
    _, la = oracle.attend_materialised(k, v, off + loc, caus, q, q_pos, base=1e4, scale=0.125)
    _, l32 = oracle.attend_stored(k, v, off, loc, st, caus, q, q_pos, base=1e4, scale=0.125,
                                  store="fp32")
    _, l16 = oracle.attend_stored(k, v, off, loc, st, caus, q, q_pos, base=1e4, scale=0.125,
                                  store="bf16")
    assert np.abs(l32 - la).max() < 1e-5
    assert 1e-5 < np.abs(l16 - la).max() < 2e-2


def test_stored_form_leaves_question_keys_exact():
    # a prefill request without documents: its question keys are not cached, so S equals A
    wl = W.custom("prefill", [[]], doc_len=16, n_pool=1, Hq=4, Hkv=2, D=32, dtype="bf16",
                  T=[9], q_pos0=[40], seed=4)
    oa, la = oracle.attend_request(wl, 0, form="A")
    os_, ls = oracle.attend_request(wl, 0, form="S")
    assert np.abs(os_ - oa).max() < 1e-12 and np.abs(ls - la).max() < 1e-12
    # with a document, only the document's keys are rounded: S moves away from A
    wl = W.custom("prefill", [[(0, 0)]], doc_len=16, n_pool=1, Hq=4, Hkv=2, D=32, dtype="bf16",
                  T=[9], q_pos0=[16], seed=4)
    _, la = oracle.attend_request(wl, 0, form="A")
    _, ls = oracle.attend_request(wl, 0, form="S")
    assert 0 < np.abs(ls - la).max() < 2e-2


# ---------------------------------------------------------------- page word spec
def test_page_word_boundaries_exhaustive():
    for blk in (0, 1, 2**31 - 1, 2**31, 2**32 - 1):
        for off in (0, 1, 2**25, 2**26 - 1):
            for nv in (1, 2, 16, 63, 64):
                w = oracle.pack_page(blk, off, nv)
                assert 0 <= w < 2**64
                assert oracle.unpack_page(w) == (blk, off, nv)
    assert oracle.pack_page(0, 0, 1) == 0
    assert oracle.pack_page(2**32 - 1, 2**26 - 1, 64) == 2**64 - 1
    assert oracle.pack_page(5, 3, 16) == 5 | (3 << 32) | (15 << 58)


def test_page_word_random_round_trip():
    rng = np.random.default_rng(5)
    for _ in range(20000):
        blk = int(rng.integers(0, 2**32)); off = int(rng.integers(0, 2**26))
        nv = int(rng.integers(1, 65))
        assert oracle.unpack_page(oracle.pack_page(blk, off, nv)) == (blk, off, nv)


@pytest.mark.parametrize("args", [(-1, 0, 1), (2**32, 0, 1), (0, -1, 1), (0, 2**26, 1),
                                  (0, 0, 0), (0, 0, 65)])
def test_page_word_rejects_out_of_range(args):
    with pytest.raises(ValueError):
        oracle.pack_page(*args)


def test_tiny_fp32_golden_regression():
    # Stored by tests/golden/make_golden.py (oracle only): guards the oracle against silent drift.
    import json, os
    with open(os.path.join(os.path.dirname(__file__), "golden", "tiny_fp32_oracle.json")) as f:
        g = json.load(f)
    out, lse = oracle.attend_request(W.tiny_fp32(), 0)
    assert np.allclose(out, np.array(g["out"]), atol=1e-13)
    assert np.allclose(lse, np.array(g["lse"]), atol=1e-13)


# ---------------------------------------------------------------- ALiBi variant
# "Main contributions" item 4 (generalisability): the mechanism also serves ALiBi. Keys are
# cached unrotated and the position enters as slope * (n - m).
def test_alibi_slopes_standard_sequence():
    # 8 heads: 1/2, 1/4, ..., 1/256 (ratio 2^(-8/H) between consecutive heads)
    assert np.allclose(W.alibi_slopes(8), [2.0 ** -(h + 1) for h in range(8)], rtol=0, atol=0)
    s32 = W.alibi_slopes(32).astype(np.float64)
    assert np.allclose(s32[1:] / s32[:-1], 2.0 ** (-8.0 / 32), rtol=1e-6)


@pytest.mark.parametrize("slope,N", [(0.5, 5), (0.03125, 300), (2.0 ** -8, 1000)])
def test_alibi_q_zero_truncated_geometric_closed_form(slope, N):
    # q = 0: weights are exp(-slope * d) for d = m - n = 0..N-1 (causal keys at m-N+1..m).
    # lse = log((1 - e^{-sN}) / (1 - e^{-s})); with v = d the output is the truncated geometric
    # mean e^{-s}/(1-e^{-s}) - N e^{-sN}/(1-e^{-sN}).
    m = 10_000
    pos = np.arange(m - N + 1, m + 1)
    d = (m - pos).astype(np.float64)
    k = np.random.default_rng(0).standard_normal((N, 4))
    v = np.repeat(d[:, None], 4, axis=1)
    out, lse = oracle.attend_alibi(k, v, pos, np.ones(N), np.zeros((1, 1, 4)), [m], [slope],
                                   scale=0.5)
    e1, eN = math.exp(-slope), math.exp(-slope * N)
    assert lse[0, 0] == pytest.approx(math.log((1 - eN) / (1 - e1)), abs=1e-12)
    assert out[0, 0, 0] == pytest.approx(e1 / (1 - e1) - N * eN / (1 - eN), rel=1e-10)


def test_alibi_matches_library_sdpa_with_additive_bias():
    # torch's scaled_dot_product_attention with the bias as an additive float mask (fp64, CPU),
    # and scipy's logsumexp for lse; includes hidden (causal) keys and several slopes
    torch = pytest.importorskip("torch")
    sp = pytest.importorskip("scipy.special")
    rng = np.random.default_rng(3)
    n, D, G = 23, 8, 3
    k = rng.standard_normal((n, D))
    v = rng.standard_normal((n, D))
    pos = np.concatenate([np.arange(100, 110), 200 + np.arange(13)])
    caus = np.concatenate([np.zeros(10), np.ones(13)])
    q = rng.standard_normal((4, G, D))
    q_pos = np.array([200, 203, 207, 212])
    slopes = np.array([0.5, 0.0625, 0.0])
    scale = 1 / math.sqrt(D)
    out, lse = oracle.attend_alibi(k, v, pos, caus, q, q_pos, slopes, scale=scale)
    for i in range(4):
        vis = (caus == 0) | (pos <= q_pos[i])
        for g in range(G):
            bias = np.where(vis, slopes[g] * (pos - q_pos[i]), -np.inf)
            ref = torch.nn.functional.scaled_dot_product_attention(
                torch.from_numpy(q[i, g][None, None, None, :]),
                torch.from_numpy(k[None, None]), torch.from_numpy(v[None, None]),
                attn_mask=torch.from_numpy(bias[None, None, None, :]), scale=scale)
            assert np.allclose(out[i, g], ref.numpy()[0, 0, 0], atol=1e-12)
            assert lse[i, g] == pytest.approx(sp.logsumexp(scale * (k @ q[i, g]) + bias),
                                              abs=1e-12)


@pytest.mark.parametrize("c", [1, 4321, 10 ** 6])
def test_alibi_shift_invariance(c):
    # only n - m enters: shifting every key and query position by c changes nothing
    rng = np.random.default_rng(4)
    k, v = rng.standard_normal((40, 16)), rng.standard_normal((40, 16))
    pos = np.concatenate([np.arange(0, 20), 50 + np.arange(20)])
    caus = np.concatenate([np.zeros(20), np.ones(20)])
    q = rng.standard_normal((3, 2, 16))
    qp = np.array([55, 60, 69])
    a = oracle.attend_alibi(k, v, pos, caus, q, qp, [0.25, 0.01], scale=0.25)
    b = oracle.attend_alibi(k, v, pos + c, caus, q, qp + c, [0.25, 0.01], scale=0.25)
    assert np.allclose(a[0], b[0], atol=1e-12) and np.allclose(a[1], b[1], atol=1e-12)


def test_alibi_request_uses_logical_positions_of_segments():
    # the request-level oracle places document keys at offset + local index: equal to calling
    # attend_alibi on the explicitly concatenated keys
    wl = W.custom("decode", [[(0, 0), (1, 300)]], doc_len=20, n_pool=2, Hq=4, Hkv=2, D=8,
                  dtype="fp32", base=1e4, priv=[(500, 3)], seed=7)
    slopes = W.alibi_slopes(4)
    out, lse = oracle.attend_request_alibi(wl, 0, slopes)
    r = wl.requests[0]
    G = 2
    for h in range(2):
        k = np.concatenate([wl.doc_k(0)[:, h], wl.doc_k(1)[:, h], wl.new_k(0)[:, h]])
        v = np.concatenate([wl.doc_v(0)[:, h], wl.doc_v(1)[:, h], wl.new_v(0)[:, h]])
        pos = np.concatenate([np.arange(20), 300 + np.arange(20), 500 + np.arange(3)])
        o, l = oracle.attend_alibi(k, v, pos, np.zeros(43), wl.q(0)[:, h * G:(h + 1) * G],
                                   [r.m], slopes[h * G:(h + 1) * G], scale=wl.sm_scale)
        assert np.allclose(out[0, h * G:(h + 1) * G], o[0], atol=1e-13)
        assert np.allclose(lse[0, h * G:(h + 1) * G], l[0], atol=1e-13)
