"""GPU parity of the prefill -> decode chain (the summaries' prefilling and decoding parts, run
back to back through the pool): lazy_attn_prefill_append leaves the question in the pool as a
private segment, then decode steps append one token each and attend everything so far.

Tolerances as for every bf16 path: 2e-2 absolute on outputs, 1e-3 absolute on log-sum-exp."""
import dataclasses

import numpy as np
import pytest

import oracle
import workload as W

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

N_STEPS = 10  # question of 40 tokens: steps 8 and 9 start the private segment's fourth page


@pytest.fixture(scope="module")
def pk(lazylib, cuda_ok):
    import position_independent_kv_lazy_gb300 as m
    return m


class _StepSource:
    """The oracle's inputs at chain step `step`: the workload's documents, the step's query, and
    the private segment = the question's raw k/v followed by the tokens of steps 0..step."""

    def __init__(self, wl, step):
        self.wl, self.step = wl, step

    def doc_k(self, d):
        return self.wl.doc_k(d)

    def doc_v(self, d):
        return self.wl.doc_v(d)

    def q(self, b):
        return self.wl.step_q(b, self.step)

    def new_k(self, b):
        return np.concatenate([self.wl.new_k(b)] +
                              [self.wl.step_k(b, s) for s in range(self.step + 1)])

    def new_v(self, b):
        return np.concatenate([self.wl.new_v(b)] +
                              [self.wl.step_v(b, s) for s in range(self.step + 1)])


def _step_workload(wl, step):
    """The same requests as decode requests at chain step `step`: private segment at the
    question's offset holding T + step + 1 tokens, query at q_pos0 + T + step."""
    reqs = [dataclasses.replace(r, mode="decode", priv_offset=r.q_pos0, priv_len=r.T + step + 1,
                                m=r.q_pos0 + r.T + step) for r in wl.requests]
    return dataclasses.replace(wl, requests=reqs)


def _chain_setup(pk, wl):
    from position_independent_kv_lazy_gb300 import harness as H
    src = H.HostSource(wl)
    extra = H.chain_blocks_needed(wl, N_STEPS) + sum(
        -(-r.T // wl.page_size) for r in wl.requests)  # room for the reference encode below
    res = H.build_resident(wl, src, resident_pool=False, extra_blocks=extra)
    ch = H.chain_setup(wl, res, src, N_STEPS)
    return H, src, res, ch


def test_prefill_append_matches_prefill_and_encode(pk):
    """The fused call's attention equals lazy_attn_prefill bit for bit, and the private pages it
    writes equal kv_pool_insert_doc of the same question k/v bit for bit."""
    wl = W.prefill_workload(batch=3, docs_per_req=2, doc_len=200, n_pool=6, T=40, Hq=8, Hkv=2)
    H, src, res, ch = _chain_setup(pk, wl)
    pb = ch.pb
    out_a, lse_a = pk.lazy_attn_prefill_append(
        res.pool, pb.q, pb.k_new, pb.v_new, pb.cu_q, pb.q_pos0, pb.words, pb.cu_pages,
        pb.max_q_len, ch.append_slots, ch.append_local_pos, sm_scale=wl.sm_scale)
    out_p, lse_p = pk.lazy_attn_prefill(res.pool, pb.q, pb.k_new, pb.v_new, pb.cu_q, pb.q_pos0,
                                        pb.words, pb.cu_pages, pb.max_q_len, sm_scale=wl.sm_scale)
    torch.cuda.synchronize()
    assert pk.lazy_get_device_error(res.pool) == 0
    assert torch.equal(out_a, out_p) and torch.equal(lse_a, lse_p)
    for r in pb.reqs:
        k, v = src.new_kv(r.index, "cuda")
        ref_blocks = pk.kv_pool_insert_doc(res.pool, k, v)
        w_priv, _ = pk.build_page_table([[(ch.priv_blocks[r.index], 0, r.T)]], wl.page_size)
        w_ref, _ = pk.build_page_table([[(ref_blocks, 0, r.T)]], wl.page_size)
        kp, vp, _ = pk.lazy_debug_gather(res.pool, torch.from_numpy(w_priv.view(np.int64)).cuda())
        kr, vr, _ = pk.lazy_debug_gather(res.pool, torch.from_numpy(w_ref.view(np.int64)).cuda())
        torch.cuda.synchronize()
        n_full = r.T // wl.page_size
        rows = r.T - n_full * wl.page_size
        assert torch.equal(kp[:n_full], kr[:n_full]) and torch.equal(vp[:n_full], vr[:n_full])
        assert torch.equal(kp[n_full, :, :rows], kr[n_full, :, :rows])
        assert torch.equal(vp[n_full, :, :rows], vr[n_full, :, :rows])


@pytest.mark.parametrize("align", [False, True])
def test_chain_decode_steps_match_oracle(pk, align):
    """Prefill with append, then N_STEPS decode steps (token append + decode); every step of
    every request and head against the oracle's decode over documents + question + tokens, with
    each step's page table in context order or with shared documents aligned (as the bench
    runs it)."""
    wl = W.prefill_workload(batch=3, docs_per_req=2, doc_len=200, n_pool=6, T=40, Hq=8, Hkv=2)
    H, src, res, ch = _chain_setup(pk, wl)
    pb = ch.pb
    pk.lazy_attn_prefill_append(res.pool, pb.q, pb.k_new, pb.v_new, pb.cu_q, pb.q_pos0, pb.words,
                                pb.cu_pages, pb.max_q_len, ch.append_slots, ch.append_local_pos,
                                sm_scale=wl.sm_scale)
    for step in range(N_STEPS):
        db = H.chain_step_batch(wl, res, ch, step, src, align_shared=align)
        pk.kv_pool_write_tokens(res.pool, db.new_k, db.new_v, db.slot_mapping, db.local_pos)
        out, lse = pk.lazy_attn_decode(res.pool, db.q, db.q_pos, db.words, db.cu_pages,
                                       sm_scale=wl.sm_scale)
        torch.cuda.synchronize()
        assert pk.lazy_get_device_error(res.pool) == 0
        out, lse = out.float().cpu().numpy(), lse.cpu().numpy()
        swl, ssrc = _step_workload(wl, step), _StepSource(wl, step)
        for b in range(wl.batch):
            ro, rl = oracle.attend_request(swl, b, src=ssrc)
            assert np.abs(out[b] - ro[0]).max() <= 2e-2, (step, b)
            assert np.abs(lse[b] - rl[0]).max() <= 1e-3, (step, b)


def test_append_slot_outside_pool_flags_without_writing(pk):
    """A question token whose slot lies beyond the pool is skipped by the encode's bounds check
    and reported as LAZY_DEVERR_BAD_PAGE; the in-range tokens are still written."""
    wl = W.prefill_workload(batch=1, docs_per_req=2, doc_len=200, n_pool=2, T=40, Hq=8, Hkv=2)
    H, src, res, ch = _chain_setup(pk, wl)
    pb = ch.pb
    slots = ch.append_slots.clone()
    slots[5] = res.pool.num_blocks * wl.page_size + 3
    pk.lazy_attn_prefill_append(res.pool, pb.q, pb.k_new, pb.v_new, pb.cu_q, pb.q_pos0, pb.words,
                                pb.cu_pages, pb.max_q_len, slots, ch.append_local_pos,
                                sm_scale=wl.sm_scale)
    torch.cuda.synchronize()
    assert pk.lazy_get_device_error(res.pool) & pk.LAZY_DEVERR_BAD_PAGE
    assert pk.lazy_get_device_error(res.pool) == 0  # read-and-clear
