"""GPU parity of the shared-segment decode (lazy_attn_decode_shared) against the fp64 oracle and
against the per-request decode (lazy_attn_decode) on the same inputs.

Tolerances as for the decode: bf16 pools 2e-2 absolute on outputs, 1e-3 on log-sum-exp. Against
lazy_attn_decode the two paths differ only in how partial results are cut and merged (fp32), so
outputs agree to one bf16 rounding and lse to 1e-4.
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


def _plan(pk, db, page_positions=False):
    words = db.words.cpu().numpy().view(np.uint64)
    cu = db.cu_pages.cpu().numpy()
    plan = pk.lazy_decode_shared_plan(words, cu, page_positions=page_positions)
    return plan, plan.to(db.q.device)


def _both(pk, wl, src=None, grid_ctas=0, align=False, slopes=None):
    H = _h()
    src = src or H.HostSource(wl)
    res = H.build_resident(wl, src, resident_pool=False, alibi_slopes=slopes)
    db = H.decode_batch(wl, res, src, align_shared=align)
    host_plan, plan = _plan(pk, db, page_positions=slopes is not None)
    o_s, l_s = pk.lazy_attn_decode_shared(res.pool, db.q, db.q_pos, plan, sm_scale=wl.sm_scale,
                                          grid_ctas=grid_ctas)
    o_d, l_d = pk.lazy_attn_decode(res.pool, db.q, db.q_pos, db.words, db.cu_pages,
                                   sm_scale=wl.sm_scale, grid_ctas=grid_ctas)
    torch.cuda.synchronize()
    assert pk.lazy_get_device_error(res.pool) == 0
    return (host_plan, o_s.float().cpu().numpy(), l_s.cpu().numpy(),
            o_d.float().cpu().numpy(), l_d.cpu().numpy())


def _check(wl, out, lse, reqs=None, kv_heads=None, src=None, form="A"):
    reqs = reqs if reqs is not None else range(wl.batch)
    G = wl.Hq // wl.Hkv
    heads = list(range(wl.Hq)) if kv_heads is None else \
        [h * G + g for h in kv_heads for g in range(G)]
    for b in reqs:
        ro, rl = oracle.attend_request(wl, b, kv_heads=kv_heads, src=src, form=form)
        assert np.abs(out[b][heads] - ro[0][heads]).max() <= 2e-2, b
        assert np.abs(lse[b][heads] - rl[0][heads]).max() <= 1e-3, b


def _edge(Hq, Hkv):
    # doc 0 in three requests (one of them next to doc 3 at the same offset), doc 1 in two,
    # doc 2 twice in request 1 (a request paired with itself) and once in request 0; 200-token
    # documents end in a half page; ragged private segments
    segs = [[(0, 0), (1, 200), (2, 400)],
            [(2, 5), (0, 900), (2, 3000)],
            [(1, 0)],
            [(3, 177), (0, 177)]]
    priv = [(600, 9), (3200, 16), (200, 33), (377, 1)]
    return W.custom("decode", segs, doc_len=200, n_pool=4, Hq=Hq, Hkv=Hkv, D=128, dtype="bf16",
                    base=500000.0, priv=priv, seed=3)


@pytest.mark.parametrize("Hq,Hkv", [(32, 8), (16, 8), (8, 8), (16, 4), (4, 1)])
def test_shared_decode_edge_layouts(pk, Hq, Hkv):
    wl = _edge(Hq, Hkv)
    plan, o_s, l_s, o_d, l_d = _both(pk, wl)
    assert any(plan.unit_req[2 * u + 1] >= 0 for u in range(plan.n_units))
    _check(wl, o_s, l_s)
    assert np.abs(o_s - o_d).max() <= 1e-2 and np.abs(l_s - l_d).max() <= 1e-4


@pytest.mark.parametrize("grid_ctas", [1, 3, 7, 100, 1000])
def test_shared_decode_grids(pk, grid_ctas):
    # ranges from the whole flattened sequence in one CTA to many empty warps
    wl = W.decode_workload(batch=16, docs_per_req=4, doc_len=512, n_pool=8, question=8, seed=4)
    plan, o_s, l_s, o_d, l_d = _both(pk, wl, grid_ctas=grid_ctas)
    _check(wl, o_s, l_s, reqs=range(4))
    assert np.abs(o_s - o_d).max() <= 1e-2 and np.abs(l_s - l_d).max() <= 1e-4


@pytest.mark.parametrize("align", [False, True])
def test_shared_decode_small_pool_all_requests(pk, align):
    # 16 requests drawing 4 of 8 documents: most documents are shared by several requests
    wl = W.decode_workload(batch=16, docs_per_req=4, doc_len=512, n_pool=8, question=8, seed=4)
    plan, o_s, l_s, o_d, l_d = _both(pk, wl, align=align)
    pairs = sum(int(plan.unit_req[2 * u + 1] >= 0) for u in range(plan.n_units))
    assert pairs >= 16
    _check(wl, o_s, l_s)
    assert np.abs(o_s - o_d).max() <= 1e-2 and np.abs(l_s - l_d).max() <= 1e-4


def test_shared_decode_alibi(pk):
    wl = _edge(32, 8)
    slopes = W.alibi_slopes(wl.Hq)
    H = _h()
    src = H.HostSource(wl)
    res = H.build_resident(wl, src, resident_pool=False, alibi_slopes=slopes)
    db = H.decode_batch(wl, res, src)
    # ALiBi words hold page positions; read them as RoPE words so that pages are paired one by
    # one (each page its own segment): the attention must not change
    for page_positions in (True, False):
        _, plan = _plan(pk, db, page_positions=page_positions)
        o_s, l_s = pk.lazy_attn_decode_shared(res.pool, db.q, db.q_pos, plan,
                                              sm_scale=wl.sm_scale)
        o_d, l_d = pk.lazy_attn_decode(res.pool, db.q, db.q_pos, db.words, db.cu_pages,
                                       sm_scale=wl.sm_scale)
        torch.cuda.synchronize()
        assert pk.lazy_get_device_error(res.pool) == 0
        o_s, l_s = o_s.float().cpu().numpy(), l_s.cpu().numpy()
        o_d, l_d = o_d.float().cpu().numpy(), l_d.cpu().numpy()
        assert np.abs(o_s - o_d).max() <= 1e-2 and np.abs(l_s - l_d).max() <= 1e-4
    for b in range(wl.batch):
        ro, rl = oracle.attend_request_alibi(wl, b, slopes)
        assert np.abs(o_s[b] - ro[0]).max() <= 2e-2 and np.abs(l_s[b] - rl[0]).max() <= 1e-3


def test_shared_decode_empty_request_and_page_cut(pk):
    # request 1 has no pages (zeros, lse -inf); the RoPE tables cut at every page still decode
    H = _h()
    wl = _edge(32, 8)
    src = H.HostSource(wl)
    res = H.build_resident(wl, src, resident_pool=False)
    db = H.decode_batch(wl, res, src)
    words = db.words.cpu().numpy().view(np.uint64)
    cu = db.cu_pages.cpu().numpy().copy()
    n1 = cu[2] - cu[1]
    keep = np.r_[0:cu[1], cu[2]:cu[-1]]
    words2 = words[keep]
    cu2 = cu.copy()
    cu2[2:] -= n1
    plan = pk.lazy_decode_shared_plan(words2, cu2).to("cuda")
    o_s, l_s = pk.lazy_attn_decode_shared(res.pool, db.q, db.q_pos, plan, sm_scale=wl.sm_scale)
    d_words = torch.from_numpy(words2.view(np.int64)).cuda()
    d_cu = torch.from_numpy(cu2).cuda()
    o_d, l_d = pk.lazy_attn_decode(res.pool, db.q, db.q_pos, d_words, d_cu, sm_scale=wl.sm_scale)
    torch.cuda.synchronize()
    assert pk.lazy_get_device_error(res.pool) == 0
    o_s, l_s = o_s.float().cpu().numpy(), l_s.cpu().numpy()
    assert np.all(o_s[1] == 0) and np.all(np.isneginf(l_s[1]))
    assert np.abs(o_s - o_d.float().cpu().numpy()).max() <= 1e-2
    fin = np.isfinite(l_s)
    assert np.abs(l_s[fin] - l_d.cpu().numpy()[fin]).max() <= 1e-4


def test_shared_decode_full_size_sampled(pk):
    # decode_b64 (64 requests x 8 Zipf documents x 512 + 65 private), aligned page order
    H = _h()
    wl = W.decode_workload()
    src = H.DeviceSource(wl)
    plan, o_s, l_s, o_d, l_d = _both(pk, wl, src=src, align=True)
    refs = sum(len(r.docs) for r in wl.requests)
    pairs = sum(int(plan.unit_req[2 * u + 1] >= 0) for u in range(plan.n_units))
    assert pairs >= 150 and plan.n_entries < 0.75 * (32 * refs + 5 * len(wl.requests))
    assert np.abs(o_s - o_d).max() <= 1e-2 and np.abs(l_s - l_d).max() <= 1e-4
    _check(wl, o_s, l_s, reqs=[0, 17, 63], kv_heads=[0, 5], src=src.host_view())


@pytest.mark.parametrize("Hq,Hkv", [(32, 8), (8, 8), (4, 1)])
def test_shared_decode_small_contexts(pk, Hq, Hkv):
    # contexts of 1 to 88 keys with 24-token documents shared by several requests, checked
    # against the oracle's stored-key form (the pool's bf16 copy of R(j) k written out)
    segs = [[(0, 0), (1, 24)], [(1, 5), (0, 77)], [], [(1, 100), (0, 7), (1, 300)]]
    priv = [(48, 3), (29, 9), (0, 1), (500, 16)]
    wl = W.custom("decode", segs, doc_len=24, n_pool=2, Hq=Hq, Hkv=Hkv, D=128, dtype="bf16",
                  base=500000.0, priv=priv, seed=23)
    plan, o_s, l_s, o_d, l_d = _both(pk, wl)
    assert any(plan.unit_req[2 * u + 1] >= 0 for u in range(plan.n_units))
    _check(wl, o_s, l_s, form="S")
    assert np.abs(o_s - o_d).max() <= 1e-2 and np.abs(l_s - l_d).max() <= 1e-4


def test_long_decode_shared_full_size_sampled(pk):
    # long_decode_b16 (16 requests x 64 Zipf(1.2) documents x 2048 + the new token) through the
    # shared-segment plan of the aligned tables, as the bench times it: 3 requests x 2 kv heads
    H = _h()
    wl = W.long_decode_workload()
    src = H.DeviceSource(wl)
    res = H.build_resident(wl, src, drop_raw=False)
    db = H.decode_batch(wl, res, src, align_shared=True)
    host_plan, plan = _plan(pk, db)
    o_s, l_s = pk.lazy_attn_decode_shared(res.pool, db.q, db.q_pos, plan, sm_scale=wl.sm_scale)
    torch.cuda.synchronize()
    assert pk.lazy_get_device_error(res.pool) == 0
    assert sum(int(host_plan.unit_req[2 * u + 1] >= 0) for u in range(host_plan.n_units)) >= 16
    _check(wl, o_s.float().cpu().numpy(), l_s.cpu().numpy(), reqs=[0, 7, 15], kv_heads=[2, 6],
           src=src.host_view())


@pytest.mark.parametrize("which", ["a_out_of_range", "b_out_of_range", "b_other_block"])
def test_shared_decode_bad_entry_sets_flag_without_fault(pk, which):
    # a corrupted entry of a pair unit (request A's word, request B's word, or a B word naming
    # another block than A's) is reported as LAZY_DEVERR_BAD_PAGE; a clean call afterwards is exact
    H = _h()
    wl = _edge(32, 8)
    src = H.HostSource(wl)
    res = H.build_resident(wl, src, resident_pool=False)
    db = H.decode_batch(wl, res, src)
    host_plan, plan = _plan(pk, db)
    u = next(u for u in range(host_plan.n_units) if host_plan.unit_req[2 * u + 1] >= 0)
    e = int(host_plan.cu_entries[u])
    ent = plan.entries.clone()
    w = np.array(ent[2 * e:2 * e + 2].cpu().numpy()).view(np.uint64)
    if which == "a_out_of_range":
        ent[2 * e] = int(pk.lazy_pack_page(res.pool.num_blocks + 5, 0, 16))
    elif which == "b_out_of_range":
        ent[2 * e + 1] = int(pk.lazy_pack_page(res.pool.num_blocks + 5, 0, 16))
    else:
        other = (int(w[0]) & 0xFFFFFFFF) ^ 1
        ent[2 * e + 1] = int(pk.lazy_pack_page(other, 0, 16))
    bad = pk.SharedPlan(ent, plan.cu_entries, plan.unit_req, plan.cu_members, plan.members,
                        plan.member_entries)
    pk.lazy_attn_decode_shared(res.pool, db.q, db.q_pos, bad, sm_scale=wl.sm_scale)
    assert pk.lazy_get_device_error(res.pool) & pk.LAZY_DEVERR_BAD_PAGE
    assert pk.lazy_get_device_error(res.pool) == 0
    out, lse = pk.lazy_attn_decode_shared(res.pool, db.q, db.q_pos, plan, sm_scale=wl.sm_scale)
    torch.cuda.synchronize()
    assert pk.lazy_get_device_error(res.pool) == 0
    _check(wl, out.float().cpu().numpy(), lse.cpu().numpy())


def test_shared_decode_rejects_unsupported_groups(pk):
    # 8 query heads per kv head fill a whole fragment half pair: not served by this path
    H = _h()
    wl = _edge(32, 4)
    src = H.HostSource(wl)
    res = H.build_resident(wl, src, resident_pool=False)
    with pytest.raises(pk.LazyError):
        pk.lazy_decode_shared_workspace_bytes(res.pool, 4, wl.Hq)
