"""GPU checks of the copy-per-offset baseline: kv_pool_materialise writes a document re-encoded
for one logical offset (keys at absolute positions), the decode reads such copies through page
words of offset 0, and the tensor-core prefill reads them with LAZY_PREFILL_ABSOLUTE_KEYS. The
attention over the copies is the same attention, so the oracle tolerances hold.
"""
import numpy as np
import pytest

import oracle
import workload as W

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def pk(lazylib, cuda_ok):
    import position_independent_kv_lazy_gb300 as m
    return m


def _h():
    from position_independent_kv_lazy_gb300 import harness
    return harness


@pytest.mark.parametrize("off", [123457, (1 << 26) - 100])
@pytest.mark.parametrize("dtype,D", [("bf16", 128), ("fp32", 64)])
def test_materialised_pages_hold_keys_at_absolute_positions(pk, dtype, D, off):
    # a 40-token document (the last page partial) re-encoded for offset `off` (the second just
    # below the 2^26 position limit): K rows equal R(offset + j) k up to the cache's rounding
    # (twice: the cached copy, then the re-encoded one); V rows are the raw values
    H = _h()
    wl = W.custom("decode", [[(0, off)]], doc_len=40, n_pool=1, Hq=4, Hkv=2, D=D, dtype=dtype,
                  base=500000.0, priv=[(off + 40, 1)], seed=31)
    src = H.HostSource(wl)
    res = H.build_resident(wl, src, resident_pool=False, extra_blocks=4)
    o = wl.requests[0].offsets[0]
    blocks = pk.kv_pool_materialise(res.pool, res.doc_blocks[0], wl.doc_len, o)
    torch.cuda.synchronize()
    assert pk.lazy_get_device_error(res.pool) == 0
    assert not set(blocks) & set(res.doc_blocks[0])
    kr, vr = wl.doc_k(0), wl.doc_v(0)
    tol = 2 ** -7 if dtype == "bf16" else 1e-6
    for j in range(wl.doc_len):
        gk = res.pool.k_pages[blocks[j // 16], :, j % 16].float().cpu().numpy()
        gv = res.pool.v_pages[blocks[j // 16], :, j % 16].float().cpu().numpy()
        assert np.array_equal(gv, vr[j])
        for h in range(wl.Hkv):
            exact = oracle.rope(kr[j, h], o + j, wl.rope_base)
            pair = np.hypot(exact[:D // 2], exact[D // 2:])
            err = np.abs(gk[h] - exact)
            assert (err <= tol * np.maximum(1.0, np.concatenate([pair, pair]))).all(), (j, h)


def test_materialise_rejects_in_place_and_alibi(pk):
    H = _h()
    wl = W.custom("decode", [[(0, 5)]], doc_len=32, n_pool=1, Hq=4, Hkv=2, D=128, dtype="bf16",
                  base=500000.0, priv=[(37, 1)], seed=32)
    src = H.HostSource(wl)
    res = H.build_resident(wl, src, resident_pool=False, extra_blocks=2)
    ids = res.doc_blocks[0]
    with pytest.raises(pk.LazyError):
        pk.kv_pool_materialise(res.pool, ids, 32, 7, dst_block_ids=[ids[1], ids[0]])
    ares = H.build_resident(wl, src, resident_pool=False, extra_blocks=2,
                            alibi_slopes=W.alibi_slopes(4))
    with pytest.raises(pk.LazyError):
        pk.kv_pool_materialise(ares.pool, ares.doc_blocks[0], 32, 7)


@pytest.mark.parametrize("dtype,D", [("bf16", 128), ("fp32", 64)])
def test_materialise_batch_equals_single_copies(pk, dtype, D):
    # copies of three documents for different offsets (partial last pages, one offset twice
    # for one document, one copy of 0 tokens) in one launch equal the copies written one call
    # at a time, bit for bit
    H = _h()
    wl = W.custom("decode", [[(0, 9), (1, 700), (2, 123457)]], doc_len=57, n_pool=3, Hq=4,
                  Hkv=2, D=D, dtype=dtype, base=500000.0, priv=[(123514, 1)], seed=33)
    src = H.HostSource(wl)
    res = H.build_resident(wl, src, resident_pool=False, extra_blocks=64)
    jobs = [(0, 57, 9), (1, 57, 700), (2, 40, 123457), (0, 57, 3001), (1, 0, 5), (2, 57, 0)]
    single = [pk.kv_pool_materialise(res.pool, res.doc_blocks[d], n, o) if n else []
              for d, n, o in jobs]
    batch = pk.kv_pool_materialise_batch(res.pool, [(res.doc_blocks[d], n, o)
                                                     for d, n, o in jobs])
    torch.cuda.synchronize()
    assert pk.lazy_get_device_error(res.pool) == 0
    for (d, n, o), a, b in zip(jobs, single, batch):
        assert len(a) == len(b) == (n + 15) // 16
        if n:
            ia = torch.tensor(a, device="cuda")
            ib = torch.tensor(b, device="cuda")
            full = n // 16
            for pages in (res.pool.k_pages, res.pool.v_pages):
                if full:
                    assert torch.equal(pages[ia[:full]], pages[ib[:full]]), (d, n, o)
                if n % 16:  # slots past the copy's last token are not written
                    assert torch.equal(pages[ia[full]][:, :n % 16], pages[ib[full]][:, :n % 16])


def test_materialise_batch_rejects(pk):
    H = _h()
    wl = W.custom("decode", [[(0, 5)]], doc_len=32, n_pool=1, Hq=4, Hkv=2, D=128, dtype="bf16",
                  base=500000.0, priv=[(37, 1)], seed=34)
    src = H.HostSource(wl)
    res = H.build_resident(wl, src, resident_pool=False, extra_blocks=8)
    ids = res.doc_blocks[0]
    free = pk.kv_pool_alloc(res.pool, 4)
    bad = [
        [(ids, 32, 7, [ids[1], ids[0]])],                          # a destination is a source
        [(ids, 32, 7, free[:2]), (ids, 32, 9, [free[1], free[2]])],  # a block written twice
        [(ids, 32, (1 << 26) - 16, free[:2])],                     # offset + tokens past 2^26
        [(ids, 32, 7, [free[0], res.pool.num_blocks])],            # a block outside the pool
    ]
    for copies in bad:
        with pytest.raises(pk.LazyError) as e:
            pk.kv_pool_materialise_batch(res.pool, copies)
        assert e.value.status == pk.LAZY_ERR_INVALID_ARG
    ares = H.build_resident(wl, src, resident_pool=False, extra_blocks=2,
                            alibi_slopes=W.alibi_slopes(4))
    with pytest.raises(pk.LazyError) as e:
        pk.kv_pool_materialise_batch(ares.pool, [(ares.doc_blocks[0], 32, 7)])
    assert e.value.status == pk.LAZY_ERR_UNSUPPORTED


def _copy_setup(pk, wl, src):
    H = _h()
    res = H.build_resident(wl, src, resident_pool=False, drop_raw=False,
                           extra_blocks=H.materialised_blocks_needed(wl))
    copies = H.materialise_copies(wl, res)
    torch.cuda.synchronize()
    assert pk.lazy_get_device_error(res.pool) == 0
    return res, copies


def test_decode_over_materialised_copies(pk):
    # gaps, overlaps, one document at several offsets (one copy each). A copy holds each key
    # rounded twice (the cache's R(j) k, then R(o + j) k), so contexts are kept at a thousand
    # keys or more: on a few hundred keys that double storage rounding alone reaches 1e-3 of lse
    H = _h()
    segs = [[(0, 0), (1, 1024), (2, 2048)], [(2, 5), (0, 4000), (2, 9000)], [(1, 0)],
            [(3, 1000), (0, 1000)]]
    wl = W.custom("decode", segs, doc_len=1024, n_pool=4, Hq=32, Hkv=8, D=128, dtype="bf16",
                  base=500000.0, priv=[(3072, 9), (10100, 16), (1024, 33), (2100, 1)], seed=3)
    src = H.HostSource(wl)
    res, copies = _copy_setup(pk, wl, src)
    assert len(copies) == 9  # distinct (doc, offset) pairs
    words, cu = H.copy_page_table(wl, res, copies, wl.requests, with_private=True)
    db = H.decode_batch(wl, res, src)
    out, lse = pk.lazy_attn_decode(res.pool, db.q, db.q_pos,
                                   torch.from_numpy(words.view(np.int64)).cuda(),
                                   torch.from_numpy(cu).cuda(), sm_scale=wl.sm_scale)
    torch.cuda.synchronize()
    assert pk.lazy_get_device_error(res.pool) == 0
    out, lse = out.float().cpu().numpy(), lse.cpu().numpy()
    for b in range(wl.batch):
        ro, rl = oracle.attend_request(wl, b)
        assert np.abs(out[b] - ro[0]).max() <= 2e-2
        assert np.abs(lse[b] - rl[0]).max() <= 1e-3


def _prefill_wl():
    # 16 documents of 1024 tokens per request (the prefill configuration's context), one
    # listed at two offsets (two copies). Copies hold each key rounded twice (the cache's
    # R(j) k, then R(o + j) k), an error that averages out over many keys.
    rng = __import__("numpy").random.default_rng(7)
    segs = []
    for b, shift in enumerate((0, 3, 700)):
        docs = [int(d) for d in rng.permutation(16)]
        docs[-1] = docs[0]  # one document twice in the request: two copies
        segs.append([(d, 1024 * i + shift) for i, d in enumerate(docs)])
    return W.custom("prefill", segs, doc_len=1024, n_pool=16, Hq=32, Hkv=8, D=128, dtype="bf16",
                    base=500000.0, T=[37, 100, 130], q_pos0=[16384, 16387, 17200], seed=33)


@pytest.mark.parametrize("sms", [0, 20])
def test_prefill_absolute_keys_over_copies(pk, sms):
    H = _h()
    wl = _prefill_wl()
    src = H.HostSource(wl)
    res, copies = _copy_setup(pk, wl, src)
    pb = H.prefill_batch(wl, res, src)
    words, cu = H.copy_page_table(wl, res, copies, pb.reqs, with_private=False)
    d_words = torch.from_numpy(words.view(np.int64)).cuda()
    d_cu = torch.from_numpy(cu).cuda()
    pk.lazy_pool_set_schedule_sms(res.pool, sms)
    results = {}
    for name, fl, w, c in (
            ("abs_copies", pk.LAZY_PREFILL_TC | pk.LAZY_PREFILL_ABSOLUTE_KEYS, d_words, d_cu),
            ("rel_copies", pk.LAZY_PREFILL_TC, d_words, d_cu),
            ("abs_lazy", pk.LAZY_PREFILL_TC | pk.LAZY_PREFILL_ABSOLUTE_KEYS, pb.words,
             pb.cu_pages),
            ("qside_copies", pk.LAZY_PREFILL_TC_QSIDE, d_words, d_cu)):
        out, lse = pk.lazy_attn_prefill(res.pool, pb.q, pb.k_new, pb.v_new, pb.cu_q, pb.q_pos0,
                                        w, c, pb.max_q_len, sm_scale=wl.sm_scale, flags=fl)
        torch.cuda.synchronize()
        assert pk.lazy_get_device_error(res.pool) == 0
        results[name] = (out.float().cpu().numpy(), lse.cpu().numpy())
    cuq = pb.cu_q.cpu().numpy()
    for b in range(wl.batch):
        ro, rl = oracle.attend_request(wl, b)
        rows = slice(cuq[b], cuq[b + 1])
        for name, (o, l) in results.items():
            assert np.abs(o[rows] - ro).max() <= 2e-2, (name, b)
            assert np.abs(l[rows] - rl).max() <= 1e-3, (name, b)


def test_materialise_batch_staging_grows_between_calls(pk):
    # a 3-copy batch, then 70,000 one-page copies (a 1.7 MB page list: the pool's pinned staging
    # buffer grows past its first 1 MB), then a 3-copy batch again; sampled copies equal the
    # single-copy results bit for bit
    H = _h()
    wl = W.custom("decode", [[(0, 3)]], doc_len=16, n_pool=1, Hq=2, Hkv=1, D=64, dtype="bf16",
                  base=500000.0, priv=[(19, 1)], seed=34)
    src = H.HostSource(wl)
    n_big = 70000
    res = H.build_resident(wl, src, resident_pool=False, extra_blocks=n_big + 32)
    doc = res.doc_blocks[0]
    small = pk.kv_pool_materialise_batch(res.pool, [(doc, 16, o) for o in (5, 77, 1000)])
    big_offs = [7 * k + 1 for k in range(n_big)]
    big = pk.kv_pool_materialise_batch(res.pool, [(doc, 16, o) for o in big_offs])
    small2 = pk.kv_pool_materialise_batch(res.pool, [(doc, 16, o) for o in (5, 77, 1000)])
    torch.cuda.synchronize()
    assert pk.lazy_get_device_error(res.pool) == 0
    checks = [(small[i], o) for i, o in enumerate((5, 77, 1000))]
    checks += [(small2[i], o) for i, o in enumerate((5, 77, 1000))]
    checks += [(big[k], big_offs[k]) for k in (0, 1, 4097, 65535, n_big - 1)]
    for ids, o in checks:
        ref = pk.kv_pool_materialise(res.pool, doc, 16, o)
        torch.cuda.synchronize()
        for pages in (res.pool.k_pages, res.pool.v_pages):
            assert torch.equal(pages[ids[0]], pages[ref[0]]), o
        pk.kv_pool_release(res.pool, ref)
