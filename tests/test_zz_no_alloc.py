"""The allocation-free decode entry point against the workspace one.

lazy_attn_decode_noalloc serves callers that cannot allocate device memory, for example a plugin
inside a serving process whose memory manager already owns the GPU. Instead of a caller
workspace it uses a fixed scratch array compiled into the library. These tests call it through
the C ABI and compare it with lazy_attn_decode on the same inputs, on two calls in a row with
different batches: the two run the same kernels on the same grid, so the results must be
bit-identical (only where the partial results live differs); against the fp64 oracle the decode
tolerances hold (2e-2 on outputs, 1e-3 on log-sum-exp). This file is collected last on purpose.
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


def _setup(pk, wl):
    from position_independent_kv_lazy_gb300 import harness as H
    src = H.HostSource(wl)
    res = H.build_resident(wl, src, resident_pool=False)
    return res, H.decode_batch(wl, res, src)


def test_noalloc_matches_workspace_decode_on_two_calls(pk):
    cases = [W.decode_workload(batch=12, docs_per_req=3, doc_len=256, n_pool=9, question=40,
                               seed=21, name="noalloc_a"),
             W.decode_workload(batch=5, docs_per_req=6, doc_len=200, n_pool=12, question=7,
                               Hq=16, Hkv=4, seed=22, name="noalloc_b")]
    prepared = [(wl, *_setup(pk, wl)) for wl in cases]
    refs = []
    for wl, res, db in prepared:
        o, l = pk.lazy_attn_decode(res.pool, db.q, db.q_pos, db.words, db.cu_pages,
                                   sm_scale=wl.sm_scale)
        refs.append((o.float().cpu().numpy(), l.cpu().numpy()))
    # two allocation-free calls back to back, each on its own batch
    outs = []
    for wl, res, db in prepared:
        out = torch.empty_like(db.q)
        lse = torch.empty((wl.batch, wl.Hq), dtype=torch.float32, device="cuda")
        pk.lazy_attn_decode_noalloc(res.pool, db.q, db.q_pos, db.words, db.cu_pages,
                                    sm_scale=wl.sm_scale, out=out, lse=lse)
        outs.append((out, lse))
    torch.cuda.synchronize()
    for (wl, res, _), (ro, rl), (o, l) in zip(prepared, refs, outs):
        assert pk.lazy_get_device_error(res.pool) == 0
        o, l = o.float().cpu().numpy(), l.cpu().numpy()
        assert np.array_equal(o, ro) and np.array_equal(l, rl)
        for b in (0, wl.batch - 1):
            eo, el = oracle.attend_request(wl, b)
            assert np.abs(o[b] - eo[0]).max() <= 2e-2
            assert np.abs(l[b] - el[0]).max() <= 1e-3


def test_noalloc_rejects_batches_beyond_the_scratch(pk):
    wl = W.decode_workload(batch=2, docs_per_req=1, doc_len=64, n_pool=2, question=3, seed=23)
    res, db = _setup(pk, wl)
    B = 400   # 400 requests x 8 kv heads of partials exceed the 8 MiB array
    q = torch.zeros((B, wl.Hq, wl.D), dtype=torch.bfloat16, device="cuda")
    q_pos = torch.zeros(B, dtype=torch.int32, device="cuda")
    cu = torch.zeros(B + 1, dtype=torch.int32, device="cuda")
    with pytest.raises(pk.LazyError) as e:
        pk.lazy_attn_decode_noalloc(res.pool, q, q_pos, db.words, cu, sm_scale=wl.sm_scale)
    assert e.value.status == pk.LAZY_ERR_SCRATCH_LIMIT
    # 280 requests fit (the limit stated for 32/8/128 heads at 3 CTAs per SM on 152 SMs); with
    # no pages every row is 0 with lse -inf
    B = 280
    out, lse = pk.lazy_attn_decode_noalloc(res.pool, q[:B], q_pos[:B], db.words, cu[:B + 1],
                                           sm_scale=wl.sm_scale)
    torch.cuda.synchronize()
    assert pk.lazy_get_device_error(res.pool) == 0
    assert torch.all(out == 0) and torch.all(torch.isneginf(lse))
