"""GPU parity of the ALiBi variant (the summaries' "Main contributions" item 4: the mechanism also
serves ALiBi). The pool caches K unrotated; decode and both prefill kernels add
slope * (n - m) from logical positions (page words carry page start positions) and rotate
nothing. Compared with the oracle's plain ALiBi definition (oracle.attend_request_alibi).

Tolerances as for every path: bf16 2e-2 absolute on outputs and 1e-3 on log-sum-exp (with no
rotation the tensor-core path's operands are the cached bf16 values themselves, so the contract
tolerance holds there too); fp32 1e-5 on both."""
import dataclasses

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


def _decode_wl(D, Hq, Hkv, dtype):
    # gaps, an overlap, one document at two offsets, ragged documents and private segments
    segs = [[(0, 0), (1, 200), (2, 400)],
            [(2, 5), (0, 900), (2, 3000)],
            [(1, 0)],
            [(3, 177), (0, 177)]]
    priv = [(600, 9), (3200, 16), (200, 33), (377, 1)]
    return W.custom("decode", segs, doc_len=200, n_pool=4, Hq=Hq, Hkv=Hkv, D=D, dtype=dtype,
                    base=1e4, priv=priv, seed=11)


def _prefill_wl(D, Hq, Hkv, dtype):
    segs = [[(0, 0), (1, 200), (0, 1000)], [(2, 3)], [(1, 5000), (2, 17), (0, 9000)]]
    return W.custom("prefill", segs, doc_len=200, n_pool=3, Hq=Hq, Hkv=Hkv, D=D, dtype=dtype,
                    base=1e4, T=[37, 5, 130], q_pos0=[1200, 203, 9200], seed=12)


def _check(wl, slopes, out_rows, lse_rows, b, kv_heads=None, queries=None, src=None):
    to, tl = _tol(wl)
    ro, rl = oracle.attend_request_alibi(wl, b, slopes, kv_heads=kv_heads, queries=queries,
                                         src=src)
    G = wl.Hq // wl.Hkv
    qi = np.arange(ro.shape[0]) if queries is None else np.asarray(queries)
    heads = list(range(wl.Hq)) if kv_heads is None else \
        [h * G + g for h in kv_heads for g in range(G)]
    do = np.abs(out_rows[qi][:, heads] - ro[qi][:, heads]).max()
    dl = np.abs(lse_rows[qi][:, heads] - rl[qi][:, heads]).max()
    assert do <= to, (b, do)
    assert dl <= tl, (b, dl)


def _decode(pk, wl, slopes, src=None):
    H = _h()
    src = src or H.HostSource(wl)
    res = H.build_resident(wl, src, resident_pool=False, alibi_slopes=slopes)
    db = H.decode_batch(wl, res, src)
    out, lse = pk.lazy_attn_decode(res.pool, db.q, db.q_pos, db.words, db.cu_pages,
                                   sm_scale=wl.sm_scale)
    torch.cuda.synchronize()
    assert pk.lazy_get_device_error(res.pool) == 0
    return res, db, out.float().cpu().numpy(), lse.cpu().numpy()


def _prefill(pk, wl, slopes, flags, src=None):
    H = _h()
    src = src or H.HostSource(wl)
    res = H.build_resident(wl, src, resident_pool=False, drop_raw=False, alibi_slopes=slopes)
    pb = H.prefill_batch(wl, res, src)
    out, lse = pk.lazy_attn_prefill(res.pool, pb.q, pb.k_new, pb.v_new, pb.cu_q, pb.q_pos0,
                                    pb.words, pb.cu_pages, pb.max_q_len, sm_scale=wl.sm_scale,
                                    flags=flags)
    torch.cuda.synchronize()
    assert pk.lazy_get_device_error(res.pool) == 0
    return res, pb, out.float().cpu().numpy(), lse.cpu().numpy()


def test_alibi_cache_holds_unrotated_keys(pk):
    # the encode stores K as given in ALiBi mode (bit-exact copy), and page words carry page
    # start positions
    H = _h()
    wl = _decode_wl(128, 8, 2, "bf16")
    src = H.HostSource(wl)
    res = H.build_resident(wl, src, resident_pool=False, alibi_slopes=W.alibi_slopes(8))
    d = wl.requests[1].docs[1]
    ids = res.doc_blocks[d]
    for j in (0, 15, 16, 199):
        gk = res.pool.k_pages[ids[j // 16], :, j % 16].float().cpu().numpy()
        assert np.array_equal(gk, wl.doc_k(d)[j])
    words, cu = H.page_table(wl, res, wl.requests[1:2], with_private=True)
    offs = [oracle.unpack_page(int(w))[1] for w in words]
    assert offs[:13] == [5 + 16 * i for i in range(13)]          # doc at offset 5, 13 pages
    assert offs[13:26] == [900 + 16 * i for i in range(13)]      # doc at offset 900


@pytest.mark.parametrize("D,Hq,Hkv,dtype", [
    (128, 32, 8, "bf16"), (128, 8, 8, "bf16"), (64, 8, 2, "fp32"), (128, 32, 1, "bf16")])
def test_alibi_decode_parity(pk, D, Hq, Hkv, dtype):
    wl = _decode_wl(D, Hq, Hkv, dtype)
    slopes = W.alibi_slopes(Hq)
    _, _, out, lse = _decode(pk, wl, slopes)
    for b in range(wl.batch):
        _check(wl, slopes, out[b:b + 1], lse[b:b + 1], b)


@pytest.mark.parametrize("D,Hq,Hkv,dtype", [(128, 32, 8, "bf16"), (64, 4, 1, "fp32")])
def test_alibi_prefill_cuda_core_parity(pk, D, Hq, Hkv, dtype):
    wl = _prefill_wl(D, Hq, Hkv, dtype)
    slopes = W.alibi_slopes(Hq)
    _, pb, out, lse = _prefill(pk, wl, slopes, pk.LAZY_PREFILL_SIMT)
    cu = pb.cu_q.cpu().numpy()
    for b in range(wl.batch):
        _check(wl, slopes, out[cu[b]:cu[b + 1]], lse[cu[b]:cu[b + 1]], b)


@pytest.mark.parametrize("Hq,Hkv", [(32, 8), (8, 8), (16, 2), (32, 1)])
def test_alibi_prefill_tensor_core_parity(pk, Hq, Hkv):
    wl = _prefill_wl(128, Hq, Hkv, "bf16")
    slopes = W.alibi_slopes(Hq)
    _, pb, out, lse = _prefill(pk, wl, slopes, pk.LAZY_PREFILL_TC)
    cu = pb.cu_q.cpu().numpy()
    for b in range(wl.batch):
        _check(wl, slopes, out[cu[b]:cu[b + 1]], lse[cu[b]:cu[b + 1]], b)


def test_alibi_prefill_query_side_flag_runs_the_alibi_kernel(pk):
    # an ALiBi pool rotates nothing, so the tensor-core query-side flag takes the ALiBi kernel:
    # the same result as LAZY_PREFILL_TC, bit for bit
    wl = _prefill_wl(128, 32, 8, "bf16")
    slopes = W.alibi_slopes(32)
    _, _, out_tc, lse_tc = _prefill(pk, wl, slopes, pk.LAZY_PREFILL_TC)
    _, _, out_qs, lse_qs = _prefill(pk, wl, slopes, pk.LAZY_PREFILL_TC_QSIDE)
    assert np.array_equal(out_tc, out_qs) and np.array_equal(lse_tc, lse_qs)


def test_alibi_full_size_sampled(pk):
    # the bench's shapes: decode_b64 (4161 keys per request) and prefill_b8 (16 x 1024 + 256),
    # 32/8/128 bf16, device-drawn inputs read back for the oracle
    H = _h()
    slopes = W.alibi_slopes(32)
    wl = W.decode_workload()
    src = H.DeviceSource(wl)
    _, _, out, lse = _decode(pk, wl, slopes, src=src)
    view = src.host_view()
    for b in (0, 37, 63):
        _check(wl, slopes, out[b:b + 1], lse[b:b + 1], b, src=view)
    pwl = W.prefill_workload()
    psrc = H.DeviceSource(pwl)
    _, pb, out, lse = _prefill(pk, pwl, slopes, pk.LAZY_PREFILL_AUTO, src=psrc)
    pview = psrc.host_view()
    cu = pb.cu_q.cpu().numpy()
    for b in (0, 5):
        _check(pwl, slopes, out[cu[b]:cu[b + 1]], lse[cu[b]:cu[b + 1]], b,
               kv_heads=[0, 3, 7], queries=[0, 31, 32, 63, 64, 127, 128, 200, 255], src=pview)


def test_alibi_prefill_then_decode_chain(pk):
    # the question enters the ALiBi pool as a private segment, then decode steps append tokens
    H = _h()
    wl = W.prefill_workload(batch=2, docs_per_req=2, doc_len=200, n_pool=4, T=40, Hq=8, Hkv=2)
    slopes = W.alibi_slopes(8)
    src = H.HostSource(wl)
    n_steps = 9
    res = H.build_resident(wl, src, resident_pool=False,
                           extra_blocks=H.chain_blocks_needed(wl, n_steps), alibi_slopes=slopes)
    ch = H.chain_setup(wl, res, src, n_steps)
    pb = ch.pb
    out, lse = pk.lazy_attn_prefill_append(res.pool, pb.q, pb.k_new, pb.v_new, pb.cu_q,
                                           pb.q_pos0, pb.words, pb.cu_pages, pb.max_q_len,
                                           ch.append_slots, ch.append_local_pos,
                                           sm_scale=wl.sm_scale)
    torch.cuda.synchronize()
    out, lse = out.float().cpu().numpy(), lse.cpu().numpy()
    cu = pb.cu_q.cpu().numpy()
    for b in range(wl.batch):
        _check(wl, slopes, out[cu[b]:cu[b + 1]], lse[cu[b]:cu[b + 1]], b)

    class StepSrc:
        def __init__(self, step):
            self.step = step

        def doc_k(self, d):
            return wl.doc_k(d)

        def doc_v(self, d):
            return wl.doc_v(d)

        def q(self, b):
            return wl.step_q(b, self.step)

        def new_k(self, b):
            return np.concatenate([wl.new_k(b)] + [wl.step_k(b, s) for s in range(self.step + 1)])

        def new_v(self, b):
            return np.concatenate([wl.new_v(b)] + [wl.step_v(b, s) for s in range(self.step + 1)])

    for step in range(n_steps):
        db = H.chain_step_batch(wl, res, ch, step, src)
        pk.kv_pool_write_tokens(res.pool, db.new_k, db.new_v, db.slot_mapping, db.local_pos)
        o, l = pk.lazy_attn_decode(res.pool, db.q, db.q_pos, db.words, db.cu_pages,
                                   sm_scale=wl.sm_scale)
        torch.cuda.synchronize()
        o, l = o.float().cpu().numpy(), l.cpu().numpy()
        swl = dataclasses.replace(wl, requests=[
            dataclasses.replace(r, mode="decode", priv_offset=r.q_pos0, priv_len=r.T + step + 1,
                                m=r.q_pos0 + r.T + step) for r in wl.requests])
        for b in range(wl.batch):
            _check(swl, slopes, o[b:b + 1], l[b:b + 1], b, src=StepSrc(step))
    assert pk.lazy_get_device_error(res.pool) == 0
