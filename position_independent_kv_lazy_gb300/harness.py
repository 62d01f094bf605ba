"""Turn a seeded workload (``workload.Workload``) into device state for the library: a resident
pool holding each retrieved document once, page tables with (block, offset, n_valid) words, and
the per-request device inputs of a prefill or decode call. Used by the tests, the bench and the
smoke check; every computation on the path itself happens in the library's kernels.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Optional

import numpy as np

from . import (LazyPool, build_page_table, kv_pool_alloc, kv_pool_insert_doc,
               kv_pool_materialise_batch, lazy_decode_partition, order_segments_by_phase)


def _torch_dtype(wl):
    import torch
    return torch.bfloat16 if wl.dtype == "bf16" else torch.float32


class HostSource:
    """Host arrays of the workload (numpy float32, bf16-exact for bf16 workloads)."""

    def __init__(self, wl):
        self.wl = wl

    def doc_kv(self, d, device):
        import torch
        dt = _torch_dtype(self.wl)
        return (torch.from_numpy(self.wl.doc_k(d)).to(device=device, dtype=dt),
                torch.from_numpy(self.wl.doc_v(d)).to(device=device, dtype=dt))

    def q(self, b, device):
        import torch
        return torch.from_numpy(self.wl.q(b)).to(device=device, dtype=_torch_dtype(self.wl))

    def new_kv(self, b, device):
        import torch
        dt = _torch_dtype(self.wl)
        return (torch.from_numpy(self.wl.new_k(b)).to(device=device, dtype=dt),
                torch.from_numpy(self.wl.new_v(b)).to(device=device, dtype=dt))

    def step_q(self, b, step, device):
        import torch
        return torch.from_numpy(self.wl.step_q(b, step)).to(device=device,
                                                            dtype=_torch_dtype(self.wl))

    def step_kv(self, b, step, device):
        import torch
        dt = _torch_dtype(self.wl)
        return (torch.from_numpy(self.wl.step_k(b, step)).to(device=device, dtype=dt),
                torch.from_numpy(self.wl.step_v(b, step)).to(device=device, dtype=dt))


class DeviceSource:
    """Device-side draws (``workload.normal_torch``) for workloads too large to draw on the host.
    ``host_view()`` exposes the same tensors to the oracle (copied back) for sampled checks."""

    def __init__(self, wl):
        self.wl = wl
        self._docs: Dict[int, tuple] = {}
        self._q: Dict[int, object] = {}
        self._new: Dict[int, tuple] = {}

    def doc_kv(self, d, device):
        if d not in self._docs:
            self._docs[d] = self.wl.doc_kv_torch(d, device)
        return self._docs[d]

    def q(self, b, device):
        if b not in self._q:
            self._q[b] = self.wl.q_torch(b, device)
        return self._q[b]

    def new_kv(self, b, device):
        if b not in self._new:
            self._new[b] = self.wl.new_kv_torch(b, device)
        return self._new[b]

    def step_q(self, b, step, device):
        return self.wl.step_q_torch(b, step, device)

    def step_kv(self, b, step, device):
        return self.wl.step_kv_torch(b, step, device)

    def forget_docs(self):
        """Drop the raw document tensors once encoded (the pool holds the cache)."""
        self._docs.clear()

    def host_view(self, device="cuda"):
        src = self

        def h(t):
            return t.float().cpu().numpy()

        class View:
            def doc_k(self, d): return h(src.doc_kv(d, device)[0])
            def doc_v(self, d): return h(src.doc_kv(d, device)[1])
            def q(self, b): return h(src.q(b, device))
            def new_k(self, b): return h(src.new_kv(b, device)[0])
            def new_v(self, b): return h(src.new_kv(b, device)[1])
        return View()


@dataclasses.dataclass
class Resident:
    pool: LazyPool
    doc_blocks: Dict[int, List[int]]
    priv_blocks: Dict[int, List[int]]


def pool_blocks_needed(wl, resident_pool: bool = True) -> int:
    per_doc = -(-wl.doc_len // wl.page_size)
    n_docs = wl.n_pool_docs if resident_pool else len(wl.used_docs())
    priv = sum(-(-r.priv_len // wl.page_size) for r in wl.decode_requests())
    return n_docs * per_doc + priv


def chain_blocks_needed(wl, n_steps: int) -> int:
    """Private-segment blocks a prefill -> decode chain of n_steps needs (see chain_setup)."""
    return sum(-(-(r.T + n_steps) // wl.page_size) for r in wl.prefill_requests())


def build_resident(wl, src, device="cuda", resident_pool: bool = True, stream=None,
                   drop_raw: bool = True, extra_blocks: int = 0, alibi_slopes=None) -> Resident:
    """Create the pool (sized for the whole document pool when ``resident_pool``, plus
    ``extra_blocks`` free blocks; in ALiBi mode when ``alibi_slopes`` is given) and encode every
    document some request retrieved, once, plus each decode request's private segment."""
    import torch
    pool = LazyPool(pool_blocks_needed(wl, resident_pool) + extra_blocks, wl.Hkv, wl.D,
                    _torch_dtype(wl), wl.rope_base, wl.page_size, device,
                    alibi_slopes=alibi_slopes)
    doc_blocks: Dict[int, List[int]] = {}
    for d in wl.used_docs():
        k, v = src.doc_kv(d, device)
        doc_blocks[d] = kv_pool_insert_doc(pool, k, v, 0, None, stream)
    priv_blocks: Dict[int, List[int]] = {}
    for r in wl.decode_requests():
        k, v = src.new_kv(r.index, device)
        priv_blocks[r.index] = kv_pool_insert_doc(pool, k, v, 0, None, stream)
    torch.cuda.synchronize()
    if drop_raw and hasattr(src, "forget_docs"):
        src.forget_docs()
    return Resident(pool, doc_blocks, priv_blocks)


def page_table(wl, res: Resident, reqs, with_private: bool, align_shared: bool = False,
               phase=None):
    """Page words of the requests' documents (and private segments). ``align_shared``: shared
    documents at the same index of every request; ``phase`` = (units per request, ranges) of
    the decode's partition: the phase-aligned order of order_segments_by_phase instead."""
    segs = []
    for r in reqs:
        s = [(res.doc_blocks[d], o, wl.doc_len) for d, o in zip(r.docs, r.offsets)]
        if with_private:
            s.append((res.priv_blocks[r.index], r.priv_offset, r.priv_len))
        segs.append(s)
    if phase is not None:
        segs = order_segments_by_phase(segs, phase[0], phase[1], wl.page_size,
                                       pin_last=with_private)
        align_shared = False
    return build_page_table(segs, wl.page_size, page_positions=res.pool.alibi_slopes is not None,
                            align_shared=align_shared)


@dataclasses.dataclass
class DecodeBatch:
    reqs: list
    q: object
    q_pos: object
    words: object
    cu_pages: object
    # the new token of each request (last slot of its private segment) for the append step
    new_k: object
    new_v: object
    slot_mapping: object
    local_pos: object
    n_keys: int


def decode_batch(wl, res: Resident, src, device="cuda", reqs=None,
                 align_shared: bool = False, phase_order: bool = False,
                 grid_ctas: int = 0) -> DecodeBatch:
    """The batch's decode inputs. ``align_shared`` orders each request's segments so that
    shared documents sit at the same index in every request (see align_shared_segments);
    ``phase_order`` so that the decode (default grid, or ``grid_ctas``) reads them at about the
    same time (see order_segments_by_phase)."""
    import torch
    reqs = reqs if reqs is not None else wl.decode_requests()
    phase = lazy_decode_partition(res.pool, wl.Hq, grid_ctas) if phase_order else None
    words, cu = page_table(wl, res, reqs, with_private=True, align_shared=align_shared,
                           phase=phase)
    q = torch.cat([src.q(r.index, device) for r in reqs], dim=0).contiguous()
    q_pos = torch.tensor([r.m for r in reqs], dtype=torch.int32, device=device)
    nk, nv, slots, lpos = [], [], [], []
    for r in reqs:
        k, v = src.new_kv(r.index, device)
        j = r.priv_len - 1
        nk.append(k[j:j + 1]); nv.append(v[j:j + 1])
        blk = res.priv_blocks[r.index][j // wl.page_size]
        slots.append(blk * wl.page_size + j % wl.page_size)
        lpos.append(j)
    n_keys = sum(len(r.docs) * wl.doc_len + r.priv_len for r in reqs)
    return DecodeBatch(
        reqs, q, q_pos,
        torch.from_numpy(words.view(np.int64)).to(device),
        torch.from_numpy(cu).to(device),
        torch.cat(nk).contiguous(), torch.cat(nv).contiguous(),
        torch.tensor(slots, dtype=torch.int32, device=device),
        torch.tensor(lpos, dtype=torch.int32, device=device), n_keys)


@dataclasses.dataclass
class PrefillBatch:
    reqs: list
    q: object
    k_new: object
    v_new: object
    cu_q: object
    q_pos0: object
    words: object
    cu_pages: object
    total_q: int
    max_q_len: int
    flops: float   # causal-visible QK^T and PV FLOPs


def prefill_batch(wl, res: Resident, src, device="cuda", reqs=None) -> PrefillBatch:
    import torch
    reqs = reqs if reqs is not None else wl.prefill_requests()
    words, cu = page_table(wl, res, reqs, with_private=False)
    q = torch.cat([src.q(r.index, device) for r in reqs], dim=0).contiguous()
    kn = torch.cat([src.new_kv(r.index, device)[0] for r in reqs], dim=0).contiguous()
    vn = torch.cat([src.new_kv(r.index, device)[1] for r in reqs], dim=0).contiguous()
    cu_q = np.concatenate([[0], np.cumsum([r.T for r in reqs])]).astype(np.int32)
    flops = 0.0
    for r in reqs:
        n_doc = len(r.docs) * wl.doc_len
        flops += 4.0 * wl.D * wl.Hq * (r.T * n_doc + r.T * (r.T + 1) / 2)
    return PrefillBatch(
        reqs, q, kn, vn, torch.from_numpy(cu_q).to(device),
        torch.tensor([r.q_pos0 for r in reqs], dtype=torch.int32, device=device),
        torch.from_numpy(words.view(np.int64)).to(device), torch.from_numpy(cu).to(device),
        int(cu_q[-1]), max(r.T for r in reqs), flops)


@dataclasses.dataclass
class Chain:
    """A prefill whose question then stays in the pool as each request's private segment, at
    logical offset q_pos0 and local positions 0..T-1, followed by decode steps: step s appends
    the token generated at local position T + s and decodes the query at q_pos0 + T + s."""
    pb: PrefillBatch
    priv_blocks: Dict[int, List[int]]
    append_slots: object        # int32 [total_q]: block * page_size + slot of each question token
    append_local_pos: object    # int32 [total_q]: its local position in the private segment
    n_steps: int


def chain_setup(wl, res: Resident, src, n_steps: int, device="cuda", reqs=None) -> Chain:
    """Prefill inputs plus private-segment blocks sized for the question and n_steps tokens."""
    import torch
    pb = prefill_batch(wl, res, src, device, reqs)
    P = wl.page_size
    priv, slots, lpos = {}, [], []
    for r in pb.reqs:
        blocks = kv_pool_alloc(res.pool, -(-(r.T + n_steps) // P))
        priv[r.index] = blocks
        for t in range(r.T):
            slots.append(blocks[t // P] * P + t % P)
            lpos.append(t)
    return Chain(pb, priv, torch.tensor(slots, dtype=torch.int32, device=device),
                 torch.tensor(lpos, dtype=torch.int32, device=device), n_steps)


def chain_step_batch(wl, res: Resident, ch: Chain, step: int, src, device="cuda",
                     align_shared: bool = False) -> DecodeBatch:
    """Decode inputs of chain step `step`: page words over every document plus the private
    segment (question + tokens 0..step), the step's queries and the new token's k/v and slot."""
    import torch
    P = wl.page_size
    segs, nk, nv, slots, lpos, qs, qpos = [], [], [], [], [], [], []
    n_keys = 0
    for r in ch.pb.reqs:
        seg = [(res.doc_blocks[d], o, wl.doc_len) for d, o in zip(r.docs, r.offsets)]
        j = r.T + step
        seg.append((ch.priv_blocks[r.index], r.q_pos0, j + 1))
        segs.append(seg)
        n_keys += len(r.docs) * wl.doc_len + j + 1
        k, v = src.step_kv(r.index, step, device)
        nk.append(k)
        nv.append(v)
        qs.append(src.step_q(r.index, step, device))
        blk = ch.priv_blocks[r.index][j // P]
        slots.append(blk * P + j % P)
        lpos.append(j)
        qpos.append(r.q_pos0 + j)
    words, cu = build_page_table(segs, P, page_positions=res.pool.alibi_slopes is not None,
                                 align_shared=align_shared)
    return DecodeBatch(
        ch.pb.reqs, torch.cat(qs).contiguous(),
        torch.tensor(qpos, dtype=torch.int32, device=device),
        torch.from_numpy(words.view(np.int64)).to(device), torch.from_numpy(cu).to(device),
        torch.cat(nk).contiguous(), torch.cat(nv).contiguous(),
        torch.tensor(slots, dtype=torch.int32, device=device),
        torch.tensor(lpos, dtype=torch.int32, device=device), n_keys)


def materialised_blocks_needed(wl, reqs=None) -> int:
    """Blocks that one materialised copy per distinct (document, offset) pair takes."""
    reqs = reqs if reqs is not None else wl.requests
    pairs = {(d, o) for r in reqs for d, o in zip(r.docs, r.offsets)}
    return len(pairs) * (-(-wl.doc_len // wl.page_size))


def materialise_copies(wl, res: Resident, reqs=None, stream=None) -> Dict[tuple, List[int]]:
    """The copy-per-offset baseline: one re-encoded copy (keys at absolute positions, written by
    kv_pool_materialise_batch in one launch) of every distinct (document, offset) pair the requests use. Returns
    {(doc, offset): block ids}."""
    reqs = reqs if reqs is not None else wl.requests
    pairs = list(dict.fromkeys((d, o) for r in reqs for d, o in zip(r.docs, r.offsets)))
    # one launch for all copies
    ids = kv_pool_materialise_batch(
        res.pool, [(res.doc_blocks[d], wl.doc_len, o) for d, o in pairs], stream=stream)
    return dict(zip(pairs, ids))


def copy_page_table(wl, res: Resident, copies, reqs, with_private: bool):
    """Page words over the materialised copies: every document page at offset 0 (its keys
    already carry their absolute positions); the private segment as in page_table."""
    segs = []
    for r in reqs:
        s = [(copies[(d, o)], 0, wl.doc_len) for d, o in zip(r.docs, r.offsets)]
        if with_private:
            s.append((res.priv_blocks[r.index], r.priv_offset, r.priv_len))
        segs.append(s)
    return build_page_table(segs, wl.page_size)


def kv_bytes_accounting(wl) -> Dict[str, int]:
    """Bytes of K+V the pool keeps for a workload versus copies that bake positions in.

    resident:      every retrieved document once (position-free pages) + private segments
    materialised:  one re-encoded copy per distinct (document, logical offset) pair, the
                   position-aware alternative + private segments
    per_request:   every request's own copy of each document it holds + private segments
    """
    per_tok = wl.kv_bytes_per_token()
    priv = sum(r.priv_len for r in wl.decode_requests()) * per_tok
    pairs = set()
    for r in wl.requests:
        pairs.update(zip(r.docs, r.offsets))
    return {
        "resident": len(wl.used_docs()) * wl.doc_len * per_tok + priv,
        "materialised": len(pairs) * wl.doc_len * per_tok + priv,
        "per_request": sum(len(r.docs) for r in wl.requests) * wl.doc_len * per_tok + priv,
    }
