"""GPU parity: the library's kernels (through the C ABI) against the fp64 oracle.

Tolerances (fixed by the contract of this path): bf16 pools 2e-2 absolute on outputs and 1e-3
absolute on log-sum-exp; fp32 pools 1e-5 on both; page-word and page indexing bit-exact.

Reference forms. Layouts whose contexts hold at least 200 keys are checked against the oracle's
form A (keys materialised at absolute positions). The pool keeps each cached key as R(j) k in its
own element type; on a bf16 pool that storage rounding alone moves the log-sum-exp by about
2e-3 / sqrt(keys), past 1e-3 on contexts of a few dozen keys. Small-context layouts are
therefore checked against form S, the oracle with that storage step written out, at the same
tolerances.
"""
import math

import numpy as np
import pytest

import oracle
import workload as W

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def _tol(wl):
    return (2e-2, 1e-3) if wl.dtype == "bf16" else (1e-5, 1e-5)


@pytest.fixture(scope="module")
def pk(lazylib, cuda_ok):
    import position_independent_kv_lazy_gb300 as m
    return m


def _h():
    from position_independent_kv_lazy_gb300 import harness
    return harness


def _decode(pk, wl, src=None, grid_ctas=0):
    H = _h()
    src = src or H.HostSource(wl)
    res = H.build_resident(wl, src, resident_pool=False)
    db = H.decode_batch(wl, res, src)
    out, lse = pk.lazy_attn_decode(res.pool, db.q, db.q_pos, db.words, db.cu_pages,
                                   sm_scale=wl.sm_scale, grid_ctas=grid_ctas)
    torch.cuda.synchronize()
    assert pk.lazy_get_device_error(res.pool) == 0
    return res, db, out.float().cpu().numpy(), lse.cpu().numpy()


def _check_decode(wl, out, lse, reqs=None, kv_heads=None, src=None, form="A"):
    to, tl = _tol(wl)
    reqs = reqs if reqs is not None else range(wl.batch)
    G = wl.Hq // wl.Hkv
    for i, b in enumerate(reqs):
        ro, rl = oracle.attend_request(wl, b, kv_heads=kv_heads, src=src, form=form)
        heads = range(wl.Hq) if kv_heads is None else [h * G + g for h in kv_heads for g in range(G)]
        heads = list(heads)
        do = np.abs(out[i][heads] - ro[0][heads]).max()
        dl = np.abs(lse[i][heads] - rl[0][heads]).max()
        assert do <= to, (b, do)
        assert dl <= tl, (b, dl)


def _edge_decode_workload(D, Hq, Hkv, dtype, doc_len=200):
    # gaps, an overlap, the same doc at two offsets, offset 0, ragged documents (200 tokens =
    # 12.5 pages) and ragged private segments. Every request keeps >= 200 keys: with bf16 keys
    # in the cache, the log-sum-exp error from that storage rounding alone shrinks like
    # 1/sqrt(keys) and exceeds 1e-3 only for contexts of a few dozen keys.
    segs = [[(0, 0), (1, 200), (2, 400)],
            [(2, 5), (0, 900), (2, 3000)],
            [(1, 0)],
            [(3, 177), (0, 177)]]
    priv = [(600, 9), (3200, 16), (200, 33), (377, 1)]
    return W.custom("decode", segs, doc_len=doc_len, n_pool=4, Hq=Hq, Hkv=Hkv, D=D, dtype=dtype,
                    base=500000.0 if D == 128 else 10000.0, priv=priv, seed=3)


# ------------------------------------------------------------------ indexing (bit-exact)
def test_debug_gather_indexing_bit_exact(pk):
    H = _h()
    wl = _edge_decode_workload(128, 8, 2, "bf16")
    src = H.HostSource(wl)
    res = H.build_resident(wl, src, resident_pool=False)
    db = H.decode_batch(wl, res, src)
    k, v, f = pk.lazy_debug_gather(res.pool, db.words)
    torch.cuda.synchronize()
    words = db.words.cpu().numpy().view(np.uint64)
    f = f.cpu().numpy().view(np.uint32)
    for i, w in enumerate(words):
        assert tuple(f[i]) == oracle.unpack_page(int(w))
    blk = torch.from_numpy(f[:, 0].astype(np.int64)).cuda()
    assert torch.equal(k, res.pool.k_pages[blk]) and torch.equal(v, res.pool.v_pages[blk])
    # V pages are verbatim copies of the raw values; K pages hold R(j) k at local positions
    d = wl.requests[0].docs[1]
    ids = res.doc_blocks[d]
    vr = wl.doc_v(d)
    kr = wl.doc_k(d)
    for j in range(wl.doc_len):
        gv = res.pool.v_pages[ids[j // 16], :, j % 16].float().cpu().numpy()
        assert np.array_equal(gv, vr[j])
        gk = res.pool.k_pages[ids[j // 16], :, j % 16].float().cpu().numpy()
        for h in range(wl.Hkv):
            exact = oracle.rope(kr[j, h], j, wl.rope_base)
            assert np.abs(gk[h] - exact).max() <= 2 ** -8 * max(1.0, np.abs(exact).max())
    assert pk.lazy_get_device_error(res.pool) == 0


def test_long_document_insert_spans_launches(pk):
    # A 70,000-token document at local position 37 covers 4,378 pages: more than one launch's
    # block list (4,096 pages). Sampled rows (the first and last, both sides of the launch
    # boundary, every 997th) against the oracle: V verbatim, K within one bf16 rounding of R(j) k.
    n, pos0, hkv, d, base = 70000, 37, 2, 128, 500000.0
    pool = pk.LazyPool(num_blocks=(pos0 + n + 15) // 16 + 8, num_kv_heads=hkv, head_dim=d,
                       dtype=torch.bfloat16, rope_base=base)
    g = torch.Generator(device="cuda").manual_seed(5)
    k = torch.randn((n, hkv, d), generator=g, device="cuda").to(torch.bfloat16)
    v = torch.randn((n, hkv, d), generator=g, device="cuda").to(torch.bfloat16)
    ids = pk.kv_pool_insert_doc(pool, k, v, local_pos0=pos0)
    torch.cuda.synchronize()
    assert pk.lazy_get_device_error(pool) == 0
    assert len(ids) == (pos0 + n + 15) // 16
    boundary = (pos0 // 16 + 4096) * 16 - pos0  # first token of the second launch
    sample = sorted(set([0, 1, n - 1] + list(range(boundary - 20, boundary + 20)) +
                        list(range(0, n, 997))))
    pos = [pos0 + t for t in sample]
    blk = torch.tensor([ids[j // 16] for j in pos], device="cuda")
    slot = torch.tensor([j % 16 for j in pos], device="cuda")
    gk = pool.k_pages[blk, :, slot].float().cpu().numpy()
    gv = pool.v_pages[blk, :, slot].float().cpu().numpy()
    kh = k[sample].float().cpu().numpy()
    vh = v[sample].float().cpu().numpy()
    assert np.array_equal(gv, vh)
    for i, j in enumerate(pos):
        for h in range(hkv):
            exact = oracle.rope(kh[i, h], j, base)
            assert np.abs(gk[i, h] - exact).max() <= 2 ** -8 * max(1.0, np.abs(exact).max())
    pool.close()


# ------------------------------------------------------------------ decode
@pytest.mark.parametrize("D,Hq,Hkv,dtype", [
    (128, 32, 8, "bf16"), (128, 8, 8, "bf16"), (128, 16, 8, "bf16"), (64, 16, 8, "bf16"),
    (64, 16, 2, "bf16"), (128, 32, 2, "bf16"), (64, 8, 2, "fp32"), (128, 4, 1, "fp32"),
    (128, 32, 1, "bf16")])
def test_decode_parity_edge_layouts(pk, D, Hq, Hkv, dtype):
    wl = _edge_decode_workload(D, Hq, Hkv, dtype)
    _, _, out, lse = _decode(pk, wl)
    _check_decode(wl, out, lse)


def test_decode_aligned_page_order_parity(pk):
    # shared documents lined up across requests: the same attention, so the oracle tolerances
    # hold; the edge workload repeats one document at two offsets within a request
    H = _h()
    wl = _edge_decode_workload(128, 32, 8, "bf16")
    src = H.HostSource(wl)
    res = H.build_resident(wl, src, resident_pool=False)
    db = H.decode_batch(wl, res, src, align_shared=True)
    out, lse = pk.lazy_attn_decode(res.pool, db.q, db.q_pos, db.words, db.cu_pages,
                                   sm_scale=wl.sm_scale)
    torch.cuda.synchronize()
    assert pk.lazy_get_device_error(res.pool) == 0
    _check_decode(wl, out.float().cpu().numpy(), lse.cpu().numpy())


@pytest.mark.parametrize("order", ["aligned", "phase"])
def test_decode_ordered_full_size_matches_context_order(pk, order):
    # decode_b64 in the context order and in the index- or phase-aligned order: only the
    # summation order differs
    H = _h()
    wl = W.decode_workload()
    src = H.DeviceSource(wl)
    res = H.build_resident(wl, src)
    res_out = []
    for ordered in (False, True):
        db = H.decode_batch(wl, res, src, align_shared=ordered and order == "aligned",
                            phase_order=ordered and order == "phase")
        o, l = pk.lazy_attn_decode(res.pool, db.q, db.q_pos, db.words, db.cu_pages,
                                   sm_scale=wl.sm_scale)
        torch.cuda.synchronize()
        res_out.append((o.float().cpu().numpy(), l.cpu().numpy()))
    assert pk.lazy_get_device_error(res.pool) == 0
    (o0, l0), (o1, l1) = res_out
    assert np.abs(l0 - l1).max() <= 1e-4
    assert np.abs(o0 - o1).max() <= 2 ** -7 * max(1.0, np.abs(o0).max())


@pytest.mark.parametrize("kind", ["simt", "auto"])
def test_decode_output_to_pinned_host_memory(pk, kind):
    # out and lse may live in pinned host memory: the merge writes them there directly
    H = _h()
    wl = _edge_decode_workload(128, 32, 8, "bf16")
    src = H.HostSource(wl)
    res = H.build_resident(wl, src, resident_pool=False)
    pk.lazy_pool_set_decode_kernel(res.pool, pk.LAZY_DECODE_SIMT if kind == "simt"
                                   else pk.LAZY_DECODE_AUTO)
    db = H.decode_batch(wl, res, src)
    o_dev, l_dev = pk.lazy_attn_decode(res.pool, db.q, db.q_pos, db.words, db.cu_pages,
                                       sm_scale=wl.sm_scale)
    o_host = torch.empty(tuple(o_dev.shape), dtype=o_dev.dtype).pin_memory()
    l_host = torch.empty(tuple(l_dev.shape), dtype=torch.float32).pin_memory()
    pk.lazy_attn_decode(res.pool, db.q, db.q_pos, db.words, db.cu_pages, sm_scale=wl.sm_scale,
                        out=o_host, lse=l_host)
    torch.cuda.synchronize()
    assert pk.lazy_get_device_error(res.pool) == 0
    assert torch.equal(o_host, o_dev.cpu()) and torch.equal(l_host, l_dev.cpu())
    _check_decode(wl, o_host.float().numpy(), l_host.numpy())


@pytest.mark.parametrize("kind", ["simt", "auto"])
@pytest.mark.parametrize("Hq,Hkv", [(32, 8), (8, 8), (16, 8), (64, 8), (32, 1)])
def test_decode_both_kernels_edge_layouts(pk, kind, Hq, Hkv):
    # bf16 / head_dim 128 runs the tensor-core (mma.sync) kernel by default; the CUDA-core
    # kernel stays selectable and both must meet the tolerances (groups 4, 1, 8, MQA 32)
    H = _h()
    wl = _edge_decode_workload(128, Hq, Hkv, "bf16")
    src = H.HostSource(wl)
    res = H.build_resident(wl, src, resident_pool=False)
    pk.lazy_pool_set_decode_kernel(res.pool, pk.LAZY_DECODE_SIMT if kind == "simt"
                                   else pk.LAZY_DECODE_AUTO)
    db = H.decode_batch(wl, res, src)
    out, lse = pk.lazy_attn_decode(res.pool, db.q, db.q_pos, db.words, db.cu_pages,
                                   sm_scale=wl.sm_scale)
    torch.cuda.synchronize()
    assert pk.lazy_get_device_error(res.pool) == 0
    _check_decode(wl, out.float().cpu().numpy(), lse.cpu().numpy())


def test_decode_kernels_agree_full_size(pk):
    # decode_b64 (64 x 4161 keys): the tensor-core and CUDA-core kernels on the same inputs
    H = _h()
    wl = W.decode_workload()
    src = H.DeviceSource(wl)
    res = H.build_resident(wl, src)
    db = H.decode_batch(wl, res, src)
    outs = {}
    for kind in (pk.LAZY_DECODE_AUTO, pk.LAZY_DECODE_SIMT):
        pk.lazy_pool_set_decode_kernel(res.pool, kind)
        o, l = pk.lazy_attn_decode(res.pool, db.q, db.q_pos, db.words, db.cu_pages,
                                   sm_scale=wl.sm_scale)
        torch.cuda.synchronize()
        outs[kind] = (o.float().cpu().numpy(), l.cpu().numpy())
    assert pk.lazy_get_device_error(res.pool) == 0
    (oa, la), (os_, ls) = outs[pk.LAZY_DECODE_AUTO], outs[pk.LAZY_DECODE_SIMT]
    assert np.abs(oa - os_).max() <= 2e-2 and np.abs(la - ls).max() <= 1e-3


@pytest.mark.parametrize("grid", [1, 2, 5, 37, 1000])
def test_decode_any_grid_same_result(pk, grid):
    wl = W.decode_workload(batch=5, docs_per_req=3, doc_len=100, n_pool=6, question=21, seed=1)
    _, _, out, lse = _decode(pk, wl, grid_ctas=grid)
    _check_decode(wl, out, lse)


@pytest.mark.parametrize("grid", [1, 3, 7, 100, 1000])
def test_mqa_group_kernel_any_grid(pk, grid):
    # 32 query heads over 1 kv head: the group kernel (4 warps = 4 chunks of 8 heads sharing
    # one page ring per CTA) and the combine's shared-range slots; 1000 CTAs exceed the pages
    # (empty ranges)
    wl = W.decode_workload(batch=5, docs_per_req=3, doc_len=100, n_pool=6, question=21, Hkv=1,
                           seed=2, name="mqa_small")
    _, _, out, lse = _decode(pk, wl, grid_ctas=grid)
    _check_decode(wl, out, lse)


def test_mqa_decode_full_size_sampled(pk):
    # decode_b64 shapes with Hkv 1 (the bench's MQA line), pages aligned, default grid
    H = _h()
    wl = W.decode_workload(Hkv=1, name="decode_b64_mqa")
    src = H.DeviceSource(wl)
    res = H.build_resident(wl, src, drop_raw=False)
    db = H.decode_batch(wl, res, src, align_shared=True)
    out, lse = pk.lazy_attn_decode(res.pool, db.q, db.q_pos, db.words, db.cu_pages,
                                   sm_scale=wl.sm_scale)
    torch.cuda.synchronize()
    assert pk.lazy_get_device_error(res.pool) == 0
    reqs = [0, 31, 63]
    _check_decode(wl, out.float().cpu().numpy()[reqs], lse.cpu().numpy()[reqs], reqs=reqs,
                  src=src.host_view())


def test_decode_request_without_keys(pk):
    H = _h()
    wl = _edge_decode_workload(128, 8, 2, "bf16")
    src = H.HostSource(wl)
    res = H.build_resident(wl, src, resident_pool=False)
    db = H.decode_batch(wl, res, src)
    # request 1 keeps no page: its rows must be 0 with lse = -inf; the others are unaffected
    cu = db.cu_pages.cpu().numpy()
    words = db.words.cpu().numpy()
    keep = np.r_[0:cu[1], cu[2]:cu[-1]]
    cu2 = cu.copy()
    cu2[2:] -= cu[2] - cu[1]
    out, lse = pk.lazy_attn_decode(res.pool, db.q, db.q_pos,
                                   torch.from_numpy(words[keep]).cuda(),
                                   torch.from_numpy(cu2).cuda(), sm_scale=wl.sm_scale)
    torch.cuda.synchronize()
    out = out.float().cpu().numpy()
    lse = lse.cpu().numpy()
    assert np.all(out[1] == 0) and np.all(np.isneginf(lse[1]))
    _check_decode(wl, out[[0, 2, 3]], lse[[0, 2, 3]], reqs=[0, 2, 3])


def test_decode_shift_invariance(pk):
    wl = _edge_decode_workload(128, 8, 2, "bf16")
    _, _, out0, lse0 = _decode(pk, wl)
    for r in wl.requests:
        r.offsets = [o + 123457 for o in r.offsets]
        r.priv_offset += 123457
        r.m += 123457
    _, _, out1, lse1 = _decode(pk, wl)
    assert np.abs(out0 - out1).max() <= 2e-2 and np.abs(lse0 - lse1).max() <= 1e-3
    _check_decode(wl, out1, lse1)


@pytest.mark.parametrize("kind", ["simt", "auto"])
def test_decode_offsets_near_the_page_word_limit(pk, kind):
    # every position moved up to just below 2^26 (the page word's 26-bit offset field): the
    # fixed-point angles stay exact there, and the result matches the unshifted one and the oracle
    H = _h()
    wl = _edge_decode_workload(128, 32, 8, "bf16")
    top = max(max(r.offsets) + wl.doc_len for r in wl.requests)
    top = max(top, max(r.priv_offset + r.priv_len for r in wl.requests))
    c = (1 << 26) - 1 - top
    src = H.HostSource(wl)
    res = H.build_resident(wl, src, resident_pool=False)
    pk.lazy_pool_set_decode_kernel(res.pool, pk.LAZY_DECODE_SIMT if kind == "simt"
                                   else pk.LAZY_DECODE_AUTO)
    db = H.decode_batch(wl, res, src)
    o0, l0 = pk.lazy_attn_decode(res.pool, db.q, db.q_pos, db.words, db.cu_pages,
                                 sm_scale=wl.sm_scale)
    for r in wl.requests:
        r.offsets = [o + c for o in r.offsets]
        r.priv_offset += c
        r.m += c
    db1 = H.decode_batch(wl, res, src)
    o1, l1 = pk.lazy_attn_decode(res.pool, db1.q, db1.q_pos, db1.words, db1.cu_pages,
                                 sm_scale=wl.sm_scale)
    torch.cuda.synchronize()
    assert pk.lazy_get_device_error(res.pool) == 0
    words = db1.words.cpu().numpy().view(np.uint64)
    assert max(int(w) >> 32 & ((1 << 26) - 1) for w in words) > 1 << 25
    o0, o1 = o0.float().cpu().numpy(), o1.float().cpu().numpy()
    l0, l1 = l0.cpu().numpy(), l1.cpu().numpy()
    assert np.abs(o0 - o1).max() <= 2e-2 and np.abs(l0 - l1).max() <= 1e-3
    _check_decode(wl, o1, l1)


def test_decode_after_token_append(pk):
    # the bench's step: write the new token's k/v into its slot, then decode
    H = _h()
    wl = W.decode_workload(batch=6, docs_per_req=2, doc_len=160, n_pool=5, question=30, seed=2)
    src = H.HostSource(wl)
    res = H.build_resident(wl, src, resident_pool=False)
    db = H.decode_batch(wl, res, src)
    for b in range(wl.batch):   # scribble over the new-token slot first
        blk = res.priv_blocks[b][(wl.requests[b].priv_len - 1) // 16]
        res.pool.k_pages[blk, :, (wl.requests[b].priv_len - 1) % 16] = 7.0
    pk.kv_pool_write_tokens(res.pool, db.new_k, db.new_v, db.slot_mapping, db.local_pos)
    out, lse = pk.lazy_attn_decode(res.pool, db.q, db.q_pos, db.words, db.cu_pages,
                                   sm_scale=wl.sm_scale)
    torch.cuda.synchronize()
    _check_decode(wl, out.float().cpu().numpy(), lse.cpu().numpy())


def test_decode_full_size_sampled(pk):
    # 64 requests x 4161 keys, 32/8/128 bf16, in the bench's launch configuration (default grid,
    # phase-aligned page order)
    H = _h()
    wl = W.decode_workload()
    src = H.DeviceSource(wl)
    res = H.build_resident(wl, src, drop_raw=False)
    db = H.decode_batch(wl, res, src, phase_order=True)
    out, lse = pk.lazy_attn_decode(res.pool, db.q, db.q_pos, db.words, db.cu_pages,
                                   sm_scale=wl.sm_scale)
    torch.cuda.synchronize()
    assert pk.lazy_get_device_error(res.pool) == 0
    out = out.float().cpu().numpy()
    lse = lse.cpu().numpy()
    reqs = [0, 17, 63]
    _check_decode(wl, out[reqs], lse[reqs], reqs=reqs, kv_heads=[0, 5], src=src.host_view())


def test_long_decode_full_size_sampled(pk):
    # 16 requests x 131073 keys (64 docs of 2048), split-KV across the whole GPU, phase-aligned
    # page order as the bench runs it: 3 requests x 2 kv heads
    H = _h()
    wl = W.long_decode_workload()
    src = H.DeviceSource(wl)
    res = H.build_resident(wl, src, drop_raw=False)
    db = H.decode_batch(wl, res, src, phase_order=True)
    out, lse = pk.lazy_attn_decode(res.pool, db.q, db.q_pos, db.words, db.cu_pages,
                                   sm_scale=wl.sm_scale)
    torch.cuda.synchronize()
    assert pk.lazy_get_device_error(res.pool) == 0
    out = out.float().cpu().numpy()
    lse = lse.cpu().numpy()
    reqs = [2, 9, 15]
    _check_decode(wl, out[reqs], lse[reqs], reqs=reqs, kv_heads=[3, 6], src=src.host_view())


# ------------------------------------------------------------------ device-detected errors
def test_bad_page_word_sets_flag_without_fault(pk):
    H = _h()
    wl = _edge_decode_workload(128, 8, 2, "bf16")
    src = H.HostSource(wl)
    res = H.build_resident(wl, src, resident_pool=False)
    db = H.decode_batch(wl, res, src)
    words = db.words.clone()
    words[3] = int(pk.lazy_pack_page(res.pool.num_blocks + 5, 0, 16))
    pk.lazy_attn_decode(res.pool, db.q, db.q_pos, words, db.cu_pages, sm_scale=wl.sm_scale)
    assert pk.lazy_get_device_error(res.pool) & pk.LAZY_DEVERR_BAD_PAGE
    assert pk.lazy_get_device_error(res.pool) == 0          # read-and-clear
    out, lse = pk.lazy_attn_decode(res.pool, db.q, db.q_pos, db.words, db.cu_pages,
                                   sm_scale=wl.sm_scale)
    torch.cuda.synchronize()
    _check_decode(wl, out.float().cpu().numpy(), lse.cpu().numpy())


def test_expired_wait_sets_flag_and_context_survives(pk):
    # A wait on a barrier that nothing arrives at gives up after 50 ms, reports
    # LAZY_DEVERR_TIMEOUT through the error word, and leaves the context usable.
    H = _h()
    wl = W.decode_workload(batch=16, docs_per_req=4, doc_len=512, n_pool=8, question=8, seed=4)
    src = H.HostSource(wl)
    res = H.build_resident(wl, src, resident_pool=False)
    db = H.decode_batch(wl, res, src)
    pk.lazy_debug_wait_timeout(res.pool, 50_000_000)
    assert pk.lazy_get_device_error(res.pool) == pk.LAZY_DEVERR_TIMEOUT
    assert pk.lazy_get_device_error(res.pool) == 0
    out, lse = pk.lazy_attn_decode(res.pool, db.q, db.q_pos, db.words, db.cu_pages,
                                   sm_scale=wl.sm_scale)
    torch.cuda.synchronize()
    assert pk.lazy_get_device_error(res.pool) == 0
    _check_decode(wl, out.float().cpu().numpy(), lse.cpu().numpy(), reqs=range(4))


# ------------------------------------------------------------------ prefill
def _prefill(pk, wl, flags, src=None):
    H = _h()
    src = src or H.HostSource(wl)
    res = H.build_resident(wl, src, resident_pool=False, drop_raw=False)
    pb = H.prefill_batch(wl, res, src)
    out, lse = pk.lazy_attn_prefill(res.pool, pb.q, pb.k_new, pb.v_new, pb.cu_q, pb.q_pos0,
                                    pb.words, pb.cu_pages, pb.max_q_len, sm_scale=wl.sm_scale,
                                    flags=flags)
    torch.cuda.synchronize()
    assert pk.lazy_get_device_error(res.pool) == 0
    return res, pb, out.float().cpu().numpy(), lse.cpu().numpy()


def _check_prefill(wl, pb, out, lse, reqs=None, kv_heads=None, queries=None, src=None,
                   form="A"):
    to, tl = _tol(wl)
    cu = pb.cu_q.cpu().numpy()
    G = wl.Hq // wl.Hkv
    reqs = range(wl.batch) if reqs is None else reqs
    for b in reqs:
        ro, rl = oracle.attend_request(wl, b, kv_heads=kv_heads, queries=queries, src=src,
                                       form=form)
        rows = np.arange(cu[b], cu[b + 1])
        qi = np.arange(len(rows)) if queries is None else np.asarray(queries)
        heads = list(range(wl.Hq)) if kv_heads is None else \
            [h * G + g for h in kv_heads for g in range(G)]
        o = out[rows[qi]][:, heads]
        l = lse[rows[qi]][:, heads]
        do = np.abs(o - ro[qi][:, heads]).max()
        dl = np.abs(l - rl[qi][:, heads]).max()
        assert do <= to, (b, do)
        assert dl <= tl, (b, dl)


def test_prefill_tiny_fp32_matches_oracle_and_golden(pk):
    import json, os
    wl = W.tiny_fp32()
    _, pb, out, lse = _prefill(pk, wl, pk.LAZY_PREFILL_AUTO)
    _check_prefill(wl, pb, out, lse)
    with open(os.path.join(os.path.dirname(__file__), "golden", "tiny_fp32_oracle.json")) as f:
        g = json.load(f)
    assert np.abs(out - np.array(g["out"])).max() <= 1e-5
    assert np.abs(lse - np.array(g["lse"])).max() <= 1e-5


def _edge_prefill_workload(D, Hq, Hkv, dtype):
    segs = [[(0, 0), (1, 200), (0, 1000)], [(2, 3)], [(1, 5000), (2, 17), (0, 9000)]]
    return W.custom("prefill", segs, doc_len=200, n_pool=3, Hq=Hq, Hkv=Hkv, D=D, dtype=dtype,
                    base=500000.0 if D == 128 else 10000.0, T=[37, 5, 130],
                    q_pos0=[1200, 203, 9200], seed=5)


@pytest.mark.parametrize("D,Hq,Hkv,dtype", [
    (128, 32, 8, "bf16"), (64, 8, 8, "bf16"), (128, 16, 2, "bf16"), (64, 4, 1, "fp32"),
    (128, 8, 2, "fp32")])
def test_prefill_simt_parity(pk, D, Hq, Hkv, dtype):
    wl = _edge_prefill_workload(D, Hq, Hkv, dtype)
    _, pb, out, lse = _prefill(pk, wl, pk.LAZY_PREFILL_SIMT)
    _check_prefill(wl, pb, out, lse)


@pytest.mark.parametrize("D,Hq,Hkv,dtype", [
    (128, 32, 8, "bf16"), (64, 8, 8, "bf16"), (128, 16, 2, "bf16"), (64, 4, 1, "fp32"),
    (128, 8, 2, "fp32")])
def test_prefill_simt_query_side_rotation_parity(pk, D, Hq, Hkv, dtype):
    # the query-side variant: key pages as stored, the query rows rotated once per document
    # offset; against the oracle, and against the key-side kernel (fp32: to rounding)
    wl = _edge_prefill_workload(D, Hq, Hkv, dtype)
    _, pb, out, lse = _prefill(pk, wl, pk.LAZY_PREFILL_SIMT_QSIDE)
    _check_prefill(wl, pb, out, lse)
    _, _, o_k, l_k = _prefill(pk, wl, pk.LAZY_PREFILL_SIMT)
    if dtype == "fp32":
        assert np.abs(out - o_k).max() <= 2e-6 and np.abs(lse - l_k).max() <= 2e-6
    else:
        assert np.abs(out - o_k).max() <= 1e-2 and np.abs(lse - l_k).max() <= 1e-5


def test_prefill_full_size_sampled(pk):
    # 8 requests x (16 docs x 1024 + 256 causal question tokens), 32/8/128 bf16
    H = _h()
    wl = W.prefill_workload()
    src = H.DeviceSource(wl)
    _, pb, out, lse = _prefill(pk, wl, pk.LAZY_PREFILL_AUTO, src=src)
    # 2 requests x all 8 kv heads (32 query heads) x 16 question tokens spanning every CTA
    _check_prefill(wl, pb, out, lse, reqs=[0, 5], kv_heads=list(range(8)),
                   queries=[0, 1, 31, 32, 63, 64, 95, 127, 128, 160, 191, 192, 200, 223, 254, 255],
                   src=src.host_view())


@pytest.mark.parametrize("Hq,Hkv", [(32, 8), (8, 8), (16, 8), (16, 2), (32, 2), (32, 1)])
def test_prefill_tensor_core_parity(pk, Hq, Hkv):
    # group sizes 4, 1, 2, 8, 16, 32 (MQA at 32/1); ragged documents (200 tokens), question
    # lengths 37 / 5 / 130
    wl = _edge_prefill_workload(128, Hq, Hkv, "bf16")
    _, pb, out, lse = _prefill(pk, wl, pk.LAZY_PREFILL_TC)
    _check_prefill(wl, pb, out, lse)


@pytest.mark.parametrize("Hq,Hkv", [(32, 8), (8, 8), (16, 8), (16, 2), (32, 2), (32, 1)])
def test_prefill_tensor_core_query_side_parity(pk, Hq, Hkv):
    # the tensor-core kernel's query-side mode: 200-token documents put two offsets in some
    # 128-key tiles (the second document's pages rotated against the tile's reference), and
    # every document start re-rotates the query tiles; against the oracle and the key-side mode
    wl = _edge_prefill_workload(128, Hq, Hkv, "bf16")
    _, pb, out, lse = _prefill(pk, wl, pk.LAZY_PREFILL_TC_QSIDE)
    _check_prefill(wl, pb, out, lse)
    _, _, o_k, l_k = _prefill(pk, wl, pk.LAZY_PREFILL_TC)
    assert np.abs(out - o_k).max() <= 2e-2 and np.abs(lse - l_k).max() <= 1e-3


def test_prefill_query_side_full_size_sampled(pk):
    # the prefill workload (16 documents of 1024 tokens per request: 8 key tiles per reference)
    # through the query-side mode, sampled as in the key-side test
    H = _h()
    wl = W.prefill_workload()
    src = H.DeviceSource(wl)
    _, pb, out, lse = _prefill(pk, wl, pk.LAZY_PREFILL_TC_QSIDE, src=src)
    _check_prefill(wl, pb, out, lse, reqs=[1, 6], kv_heads=list(range(8)),
                   queries=[0, 1, 31, 32, 63, 64, 95, 127, 128, 160, 191, 192, 200, 223, 254, 255],
                   src=src.host_view())


@pytest.mark.parametrize("flags", ["tc", "simt", "simt_qside", "tc_qside"])
def test_prefill_offsets_near_the_page_word_limit(pk, flags):
    # documents and question moved up to just below 2^26 (the offset field's limit)
    H = _h()
    wl = _edge_prefill_workload(128, 32, 8, "bf16")
    top = max(max(max(r.offsets) + wl.doc_len, r.q_pos0 + r.T) for r in wl.requests)
    c = (1 << 26) - 1 - top
    for r in wl.requests:
        r.offsets = [o + c for o in r.offsets]
        r.q_pos0 += c
    fl = {"tc": pk.LAZY_PREFILL_TC, "simt": pk.LAZY_PREFILL_SIMT,
          "simt_qside": pk.LAZY_PREFILL_SIMT_QSIDE, "tc_qside": pk.LAZY_PREFILL_TC_QSIDE}[flags]
    _, pb, out, lse = _prefill(pk, wl, fl)
    _check_prefill(wl, pb, out, lse)


# Last-wave split of the tensor-core prefill. The edge layout has 3 requests (question lengths
# 37 / 5 / 130) and X = ceil(130 / (256 / group)) token blocks per (request, kv head), so
# X * Hkv * 3 units (72 for 32/8). Planned for `sms` SMs: 1 never splits (every wave is full);
# for 32/8, 5, 7, 20, 27, 62, 100 and 1000 cut the units past the last full wave into 5, 7, 5,
# 3, 6, 4 and 8 key-range chunks (every combine width; groups of 3 split units, a short last
# group at 5), and the device's own count (0) gives 2. The short request's chunks past its
# 3 key tiles are empty.
@pytest.mark.parametrize("Hq,Hkv", [(32, 8), (16, 2), (32, 1)])
@pytest.mark.parametrize("sms", [1, 5, 7, 20, 27, 62, 100, 1000, 0])
def test_prefill_last_wave_split(pk, Hq, Hkv, sms):
    H = _h()
    wl = _edge_prefill_workload(128, Hq, Hkv, "bf16")
    src = H.HostSource(wl)
    res = H.build_resident(wl, src, resident_pool=False, drop_raw=False)
    pb = H.prefill_batch(wl, res, src)

    def run(n, workspace=None):
        pk.lazy_pool_set_schedule_sms(res.pool, n)
        out, lse = pk.lazy_attn_prefill(res.pool, pb.q, pb.k_new, pb.v_new, pb.cu_q, pb.q_pos0,
                                        pb.words, pb.cu_pages, pb.max_q_len,
                                        sm_scale=wl.sm_scale, flags=pk.LAZY_PREFILL_TC,
                                        workspace=workspace)
        torch.cuda.synchronize()
        assert pk.lazy_get_device_error(res.pool) == 0
        return out.float().cpu().numpy(), lse.cpu().numpy()

    out, lse = run(sms)
    _check_prefill(wl, pb, out, lse)
    # against the unsplit schedule: the chunks' fp32 partials merge to the same rows up to
    # the bf16 rounding of the weights (chunk-local maxima) and of the output
    o1, l1 = run(1)
    assert np.abs(out - o1).max() <= 1e-2 and np.abs(lse - l1).max() <= 1e-4
    # a workspace smaller than the plan's falls back to whole units, with the same result
    o2, l2 = run(sms, workspace=torch.empty(16, dtype=torch.uint8, device="cuda"))
    assert np.array_equal(o2, o1) and np.array_equal(l2, l1)


@pytest.mark.parametrize("Hq,Hkv", [(32, 8), (32, 1)])
@pytest.mark.parametrize("sms", [5, 27, 1000])
def test_prefill_query_side_last_wave_split(pk, Hq, Hkv, sms):
    # key-range chunks of the query-side mode start inside a document: a chunk's first tile
    # sets its reference
    H = _h()
    wl = _edge_prefill_workload(128, Hq, Hkv, "bf16")
    src = H.HostSource(wl)
    res = H.build_resident(wl, src, resident_pool=False, drop_raw=False)
    pb = H.prefill_batch(wl, res, src)
    pk.lazy_pool_set_schedule_sms(res.pool, sms)
    out, lse = pk.lazy_attn_prefill(res.pool, pb.q, pb.k_new, pb.v_new, pb.cu_q, pb.q_pos0,
                                    pb.words, pb.cu_pages, pb.max_q_len, sm_scale=wl.sm_scale,
                                    flags=pk.LAZY_PREFILL_TC_QSIDE)
    torch.cuda.synchronize()
    assert pk.lazy_get_device_error(res.pool) == 0
    _check_prefill(wl, pb, out.float().cpu().numpy(), lse.cpu().numpy())


def test_prefill_split_workspace_sizes(pk):
    # 32/8 edge layout: X = 3, 72 units. 1 SM: no split. 5 SMs: 14 full waves, 2 split units
    # x 5 chunks. 20 SMs: 3 waves, 12 split units x 5. 100 SMs: 72 split units x 4 chunks.
    # One item holds 256 rows of 128 + 1 fp32.
    H = _h()
    wl = _edge_prefill_workload(128, 32, 8, "bf16")
    src = H.HostSource(wl)
    res = H.build_resident(wl, src, resident_pool=False)
    pb = H.prefill_batch(wl, res, src)
    item = 256 * 129 * 4
    want = {1: 0, 5: 2 * 5 * item, 20: 12 * 5 * item, 100: 72 * 4 * item}
    for sms, n in want.items():
        pk.lazy_pool_set_schedule_sms(res.pool, sms)
        assert pk.lazy_prefill_workspace_bytes(res.pool, wl.batch, pb.total_q, pb.max_q_len,
                                               wl.Hq) == n, sms
        assert pk.lazy_prefill_workspace_bytes(res.pool, wl.batch, pb.total_q, pb.max_q_len,
                                               wl.Hq, flags=pk.LAZY_PREFILL_SIMT) == 0


def test_prefill_tensor_core_matches_cuda_core_kernel(pk):
    wl = _edge_prefill_workload(128, 32, 8, "bf16")
    _, _, o_tc, l_tc = _prefill(pk, wl, pk.LAZY_PREFILL_TC)
    _, _, o_si, l_si = _prefill(pk, wl, pk.LAZY_PREFILL_SIMT)
    assert np.abs(o_tc - o_si).max() <= 2e-2 and np.abs(l_tc - l_si).max() <= 1e-3


def test_prefill_without_question_keys(pk):
    # documents only (no causal question keys): the oracle gets the document keys alone
    H = _h()
    wl = _edge_prefill_workload(128, 32, 8, "bf16")
    src = H.HostSource(wl)
    res = H.build_resident(wl, src, resident_pool=False)
    pb = H.prefill_batch(wl, res, src)
    cu = pb.cu_q.cpu().numpy()
    for flags in (pk.LAZY_PREFILL_TC, pk.LAZY_PREFILL_TC_QSIDE, pk.LAZY_PREFILL_SIMT):
        out, lse = pk.lazy_attn_prefill(res.pool, pb.q, None, None, pb.cu_q, pb.q_pos0, pb.words,
                                        pb.cu_pages, pb.max_q_len, sm_scale=wl.sm_scale,
                                        flags=flags)
        torch.cuda.synchronize()
        out = out.float().cpu().numpy()
        lse = lse.cpu().numpy()
        for b in range(wl.batch):
            k, v, off, loc, caus = oracle.request_keys(wl, b)
            r = wl.requests[b]
            n_doc = len(r.docs) * wl.doc_len
            q = wl.q(b)
            G = wl.Hq // wl.Hkv
            for h in range(wl.Hkv):
                o, l = oracle.attend_materialised(
                    k[:n_doc, h], v[:n_doc, h], (off + loc)[:n_doc], caus[:n_doc],
                    q[:, h * G:(h + 1) * G], r.q_pos0 + np.arange(r.T), base=wl.rope_base,
                    scale=wl.sm_scale)
                rows = slice(cu[b], cu[b + 1])
                assert np.abs(out[rows, h * G:(h + 1) * G] - o).max() <= 2e-2
                assert np.abs(lse[rows, h * G:(h + 1) * G] - l).max() <= 1e-3


@pytest.mark.parametrize("alpha", [0.6, 0.9, 1.2])
def test_mixed_step_full_size_sampled(pk, alpha):
    # skew-sweep mixed step: one prefill launch (32 ragged questions) and one decode step
    # (96 requests) over the same resident 4096-doc pool, as the bench runs it; sampled against
    # the oracle on both halves: 3 prefill requests x 2 kv heads x 4 question rows (first, middle,
    # last and a row of the second Q tile) and 4 decode requests x 2 kv heads
    H = _h()
    wl = W.mixed_workload(alpha)
    src = H.DeviceSource(wl)
    res = H.build_resident(wl, src, drop_raw=False)
    pb = H.prefill_batch(wl, res, src)
    db = H.decode_batch(wl, res, src, phase_order=True)
    pout, plse = pk.lazy_attn_prefill(res.pool, pb.q, pb.k_new, pb.v_new, pb.cu_q, pb.q_pos0,
                                      pb.words, pb.cu_pages, pb.max_q_len, sm_scale=wl.sm_scale)
    pk.kv_pool_write_tokens(res.pool, db.new_k, db.new_v, db.slot_mapping, db.local_pos)
    dout, dlse = pk.lazy_attn_decode(res.pool, db.q, db.q_pos, db.words, db.cu_pages,
                                     sm_scale=wl.sm_scale)
    torch.cuda.synchronize()
    assert pk.lazy_get_device_error(res.pool) == 0
    view = src.host_view()
    G = wl.Hq // wl.Hkv
    cu = pb.cu_q.cpu().numpy()
    pout = pout.float().cpu().numpy()
    plse = plse.cpu().numpy()
    for i in (0, 3, len(pb.reqs) - 1):
        pr = pb.reqs[i]
        qi = sorted({0, min(40, pr.T - 1), pr.T // 2, pr.T - 1})
        kvh = [1, 6]
        ro, rl = oracle.attend_request(wl, pr.index, kv_heads=kvh, queries=qi, src=view)
        heads = [h * G + g for h in kvh for g in range(G)]
        rows = cu[i] + np.array(qi)
        assert np.abs(pout[rows][:, heads] - ro[qi][:, heads]).max() <= 2e-2, pr.index
        assert np.abs(plse[rows][:, heads] - rl[qi][:, heads]).max() <= 1e-3, pr.index
    dout = dout.float().cpu().numpy()
    dlse = dlse.cpu().numpy()
    for i in (0, 10, 50, len(db.reqs) - 1):
        dr = db.reqs[i]
        kvh = [3, 7]
        ro, rl = oracle.attend_request(wl, dr.index, kv_heads=kvh, src=view)
        heads = [h * G + g for h in kvh for g in range(G)]
        assert np.abs(dout[i][heads] - ro[0][heads]).max() <= 2e-2, dr.index
        assert np.abs(dlse[i][heads] - rl[0][heads]).max() <= 1e-3, dr.index


# ------------------------------------------------------------------ small contexts (form S)
def _small_decode_workload(Hq, Hkv, dtype="bf16", D=128):
    # contexts of 1 to 88 keys: 24-token documents (a whole and a half page), one document at
    # two offsets, a request holding only its 1-token private segment (m = 0, one key)
    segs = [[(0, 0), (1, 24)], [(2, 5)], [], [(1, 100), (0, 7), (1, 300)]]
    priv = [(48, 3), (29, 9), (0, 1), (500, 16)]
    return W.custom("decode", segs, doc_len=24, n_pool=3, Hq=Hq, Hkv=Hkv, D=D, dtype=dtype,
                    base=500000.0 if D == 128 else 10000.0, priv=priv, seed=21)


def _small_prefill_workload(Hq, Hkv, dtype="bf16", D=128):
    # 16-token documents, a 5-token question after one document, a 100-token question with no
    # document at all (row 0 sees one key), and questions crossing Q-tile boundaries
    segs = [[(0, 0), (1, 16)], [(2, 3)], [], [(1, 5000), (0, 17)]]
    return W.custom("prefill", segs, doc_len=16, n_pool=3, Hq=Hq, Hkv=Hkv, D=D, dtype=dtype,
                    base=500000.0 if D == 128 else 10000.0, T=[37, 5, 100, 64],
                    q_pos0=[32, 19, 0, 9000], seed=22)


@pytest.mark.parametrize("kind", ["simt", "auto"])
@pytest.mark.parametrize("D,Hq,Hkv,dtype", [
    (128, 32, 8, "bf16"), (128, 8, 8, "bf16"), (128, 16, 8, "bf16"), (128, 64, 8, "bf16"),
    (128, 32, 1, "bf16"), (64, 16, 8, "bf16"), (64, 8, 2, "fp32")])
def test_decode_small_contexts(pk, kind, D, Hq, Hkv, dtype):
    H = _h()
    wl = _small_decode_workload(Hq, Hkv, dtype, D)
    src = H.HostSource(wl)
    res = H.build_resident(wl, src, resident_pool=False)
    pk.lazy_pool_set_decode_kernel(res.pool, pk.LAZY_DECODE_SIMT if kind == "simt"
                                   else pk.LAZY_DECODE_AUTO)
    db = H.decode_batch(wl, res, src)
    out, lse = pk.lazy_attn_decode(res.pool, db.q, db.q_pos, db.words, db.cu_pages,
                                   sm_scale=wl.sm_scale)
    torch.cuda.synchronize()
    assert pk.lazy_get_device_error(res.pool) == 0
    out, lse = out.float().cpu().numpy(), lse.cpu().numpy()
    _check_decode(wl, out, lse, form="S")
    # one key: the output is that key's value and lse its score
    G = wl.Hq // wl.Hkv
    v = wl.new_v(2)[0]
    assert np.abs(out[2] - np.repeat(v, G, axis=0)).max() <= (1e-2 if dtype == "bf16" else 1e-6)


@pytest.mark.parametrize("flags", ["tc", "simt", "simt_qside", "tc_qside"])
@pytest.mark.parametrize("Hq,Hkv", [(32, 8), (8, 8), (16, 2), (32, 1)])
def test_prefill_small_contexts(pk, flags, Hq, Hkv):
    wl = _small_prefill_workload(Hq, Hkv)
    fl = {"tc": pk.LAZY_PREFILL_TC, "simt": pk.LAZY_PREFILL_SIMT,
          "simt_qside": pk.LAZY_PREFILL_SIMT_QSIDE, "tc_qside": pk.LAZY_PREFILL_TC_QSIDE}[flags]
    _, pb, out, lse = _prefill(pk, wl, fl)
    _check_prefill(wl, pb, out, lse, form="S")


@pytest.mark.parametrize("flags", ["tc", "tc_qside", "simt"])
def test_prefill_request_without_question_tokens(pk, flags):
    # a request with T = 0 between two others (an empty cu_q range): the other requests' rows
    # are unaffected; the last request has a 1-token question over overlapping document offsets
    wl = W.custom("prefill", [[(0, 0), (1, 200)], [(2, 7)], [(0, 50), (2, 1)]], doc_len=200,
                  n_pool=3, Hq=32, Hkv=8, D=128, dtype="bf16", base=500000.0, T=[37, 0, 1],
                  q_pos0=[400, 207, 250], seed=41)
    fl = {"tc": pk.LAZY_PREFILL_TC, "tc_qside": pk.LAZY_PREFILL_TC_QSIDE,
          "simt": pk.LAZY_PREFILL_SIMT}[flags]
    _, pb, out, lse = _prefill(pk, wl, fl)
    cu = pb.cu_q.cpu().numpy()
    assert cu[1] == cu[2]
    _check_prefill(wl, pb, out, lse, reqs=[0, 2])


@pytest.mark.parametrize("flags", ["simt", "simt_qside"])
def test_prefill_small_contexts_fp32(pk, flags):
    wl = _small_prefill_workload(8, 2, "fp32", 64)
    fl = pk.LAZY_PREFILL_SIMT if flags == "simt" else pk.LAZY_PREFILL_SIMT_QSIDE
    _, pb, out, lse = _prefill(pk, wl, fl)
    _check_prefill(wl, pb, out, lse, form="S")


@pytest.mark.parametrize("sms", [5, 20])
def test_prefill_small_contexts_last_wave_split(pk, sms):
    # the tensor-core prefill's key-range chunks on short contexts (some chunks see no key)
    H = _h()
    wl = _small_prefill_workload(32, 8)
    src = H.HostSource(wl)
    res = H.build_resident(wl, src, resident_pool=False, drop_raw=False)
    pb = H.prefill_batch(wl, res, src)
    pk.lazy_pool_set_schedule_sms(res.pool, sms)
    out, lse = pk.lazy_attn_prefill(res.pool, pb.q, pb.k_new, pb.v_new, pb.cu_q, pb.q_pos0,
                                    pb.words, pb.cu_pages, pb.max_q_len, sm_scale=wl.sm_scale,
                                    flags=pk.LAZY_PREFILL_TC)
    torch.cuda.synchronize()
    assert pk.lazy_get_device_error(res.pool) == 0
    _check_prefill(wl, pb, out.float().cpu().numpy(), lse.cpu().numpy(), form="S")


# ------------------------------------------------------------------ page order
def _permuted_table(pk, wl, res, rng, with_private):
    # each request's segments in a random order: attention does not depend on page order
    segs = []
    for r in wl.requests:
        s = [(res.doc_blocks[d], o, wl.doc_len) for d, o in zip(r.docs, r.offsets)]
        if with_private:
            s.append((res.priv_blocks[r.index], r.priv_offset, r.priv_len))
        segs.append([s[i] for i in rng.permutation(len(s))])
    words, cu = pk.build_page_table(segs, wl.page_size)
    return (torch.from_numpy(words.view(np.int64)).cuda(), torch.from_numpy(cu).cuda())


@pytest.mark.parametrize("seed", [1, 2, 3])
@pytest.mark.parametrize("kind", ["simt", "auto"])
def test_decode_random_segment_orders(pk, seed, kind):
    H = _h()
    wl = _edge_decode_workload(128, 32, 8, "bf16")
    src = H.HostSource(wl)
    res = H.build_resident(wl, src, resident_pool=False)
    pk.lazy_pool_set_decode_kernel(res.pool, pk.LAZY_DECODE_SIMT if kind == "simt"
                                   else pk.LAZY_DECODE_AUTO)
    db = H.decode_batch(wl, res, src)
    words, cu = _permuted_table(pk, wl, res, np.random.default_rng(seed), with_private=True)
    out, lse = pk.lazy_attn_decode(res.pool, db.q, db.q_pos, words, cu, sm_scale=wl.sm_scale)
    torch.cuda.synchronize()
    assert pk.lazy_get_device_error(res.pool) == 0
    _check_decode(wl, out.float().cpu().numpy(), lse.cpu().numpy())


@pytest.mark.parametrize("seed", [1, 2])
@pytest.mark.parametrize("flags", ["tc", "simt", "tc_qside"])
def test_prefill_random_segment_orders(pk, seed, flags):
    # permuted documents change which pages share a 128-key tile (mixed offsets within a tile)
    H = _h()
    wl = _edge_prefill_workload(128, 32, 8, "bf16")
    src = H.HostSource(wl)
    res = H.build_resident(wl, src, resident_pool=False, drop_raw=False)
    pb = H.prefill_batch(wl, res, src)
    words, cu = _permuted_table(pk, wl, res, np.random.default_rng(seed), with_private=False)
    out, lse = pk.lazy_attn_prefill(res.pool, pb.q, pb.k_new, pb.v_new, pb.cu_q, pb.q_pos0,
                                    words, cu, pb.max_q_len, sm_scale=wl.sm_scale,
                                    flags={"tc": pk.LAZY_PREFILL_TC,
                                           "tc_qside": pk.LAZY_PREFILL_TC_QSIDE,
                                           "simt": pk.LAZY_PREFILL_SIMT}[flags])
    torch.cuda.synchronize()
    assert pk.lazy_get_device_error(res.pool) == 0
    _check_prefill(wl, pb, out.float().cpu().numpy(), lse.cpu().numpy())
