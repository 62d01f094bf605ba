"""Seeded synthetic inputs for deferred-RoPE attention over a position-agnostic paged KV cache.

This module holds no attention or RoPE arithmetic. It only decides *what* the inputs are:
which documents each request retrieves, at which logical offsets, how long each question or
private segment is, and the raw (unrotated) Q/K/V values. Both the CUDA path's tests and bench
and the fp64 oracle take their inputs from here; neither side imports the other.

Recipe
------
* Structure (document draws, orders, lengths, the prefill/decode split) comes from one
  ``numpy.random.Generator(PCG64(SeedSequence(seed)))`` consumed in a fixed order.
* Values are i.i.d. N(0, 1) float32. Each array has its own stream,
  ``PCG64(SeedSequence([seed, KIND, index]))``, so a document can be generated on its own without
  drawing the whole pool. For bf16 workloads every value is rounded to bfloat16
  (round-to-nearest-even) *before* anyone sees it, so the oracle and the GPU consume identical
  numbers.
* Device generation (``*_torch`` helpers) draws the same distribution with torch's CUDA Philox
  generator seeded from the same key. It is used only where the host would take too long
  (full-size bench workloads); the oracle then reads those same input tensors back.

Documents are drawn with Zipf skew as the summaries describe for RAG access patterns (LazyAttention
technical summary, "Problem statement": skewed, Zipf-like document access): P(rank k) ∝ k^-alpha,
k = 1..pool, doc id = k-1, distinct within a request.
"""
from __future__ import annotations

import dataclasses
import hashlib
from typing import Dict, List, Optional, Tuple

import numpy as np

KIND_DOC_K = 1
KIND_DOC_V = 2
KIND_Q = 3
KIND_NEW_K = 4
KIND_NEW_V = 5
KIND_PRIV_K = 6
KIND_PRIV_V = 7
# decode steps that follow a prefill (prefill -> decode chain): the step's query and the
# generated token's k/v, keyed by (request, step)
KIND_STEP_Q = 8
KIND_STEP_K = 9
KIND_STEP_V = 10


def step_index(b: int, step: int) -> int:
    """Stream index of (request b, decode step `step`) for the KIND_STEP_* draws."""
    return (b << 20) | step


# ----------------------------------------------------------------------------------------------
# bfloat16 rounding (storage format of the inputs; not part of the method)
# ----------------------------------------------------------------------------------------------
def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even); return them as float32."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) >> 16) << 16
    out = r.astype(np.uint32).view(np.float32)
    # NaN inputs never occur (values are drawn from a normal distribution).
    return out.reshape(x.shape)


def _stream(seed: int, kind: int, index: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, kind, index])))


def normal(seed: int, kind: int, index: int, shape, dtype: str) -> np.ndarray:
    """N(0,1) float32 array for (seed, kind, index), rounded to bf16 when dtype == 'bf16'."""
    a = _stream(seed, kind, index).standard_normal(size=shape, dtype=np.float32)
    return bf16_round(a) if dtype == "bf16" else a


def alibi_slopes(n_heads: int) -> np.ndarray:
    """ALiBi head slopes, an input of the ALiBi variant (a model parameter, not part of the
    method): the standard geometric sequence 2^(-8 (h + 1) / H) for h = 0 .. H-1, for H a power
    of two. Returned as float32, the precision both sides receive."""
    if n_heads < 1 or n_heads & (n_heads - 1):
        raise ValueError("ALiBi slopes here are defined for a power-of-two head count")
    h = np.arange(1, n_heads + 1, dtype=np.float64)
    return np.power(2.0, -8.0 * h / n_heads).astype(np.float32)


def _torch_seed(seed: int, kind: int, index: int) -> int:
    h = hashlib.blake2b(f"{seed}:{kind}:{index}".encode(), digest_size=8).digest()
    return int.from_bytes(h, "little") & ((1 << 63) - 1)


def normal_torch(seed: int, kind: int, index: int, shape, dtype: str, device):
    """Device-side draw of the same distribution (Philox stream keyed like ``normal``)."""
    import torch

    g = torch.Generator(device=device)
    g.manual_seed(_torch_seed(seed, kind, index))
    t = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    return t.to(torch.bfloat16) if dtype == "bf16" else t


# ----------------------------------------------------------------------------------------------
# Workload structure
# ----------------------------------------------------------------------------------------------
@dataclasses.dataclass
class Request:
    """One request: retrieved documents at logical offsets, then its own tokens.

    prefill: ``T`` question tokens at logical positions ``q_pos0 .. q_pos0+T-1``; their raw q and
             k/v (``new``) are attended causally among themselves and see every document key.
    decode:  a private segment of ``priv_len`` tokens already in the cache at logical offset
             ``priv_offset`` (the question plus the just-generated token, whose k/v is appended
             before attention) and one query at position ``m``.
    """

    index: int
    mode: str                      # "prefill" | "decode"
    docs: List[int]
    offsets: List[int]
    T: int = 0
    q_pos0: int = 0
    priv_offset: int = 0
    priv_len: int = 0
    m: int = 0


@dataclasses.dataclass
class Workload:
    name: str
    dtype: str                     # "bf16" | "fp32"
    Hq: int
    Hkv: int
    D: int
    rope_base: float
    page_size: int
    doc_len: int
    n_pool_docs: int
    requests: List[Request]
    seed: int = 0
    sm_scale: Optional[float] = None
    _cache: Dict[Tuple[int, int], np.ndarray] = dataclasses.field(default_factory=dict, repr=False)

    def __post_init__(self):
        if self.sm_scale is None:
            self.sm_scale = 1.0 / float(np.sqrt(self.D))

    # ---------------- structure helpers ----------------
    @property
    def batch(self) -> int:
        return len(self.requests)

    def used_docs(self) -> List[int]:
        s = set()
        for r in self.requests:
            s.update(r.docs)
        return sorted(s)

    def prefill_requests(self) -> List[Request]:
        return [r for r in self.requests if r.mode == "prefill"]

    def decode_requests(self) -> List[Request]:
        return [r for r in self.requests if r.mode == "decode"]

    # ---------------- host values (float32, bf16-exact when dtype == bf16) ----------------
    def _get(self, kind, index, shape):
        key = (kind, index)
        if key not in self._cache:
            self._cache[key] = normal(self.seed, kind, index, shape, self.dtype)
        return self._cache[key]

    def doc_k(self, d):
        return self._get(KIND_DOC_K, d, (self.doc_len, self.Hkv, self.D))

    def doc_v(self, d):
        return self._get(KIND_DOC_V, d, (self.doc_len, self.Hkv, self.D))

    def q(self, b):
        r = self.requests[b]
        n = r.T if r.mode == "prefill" else 1
        return self._get(KIND_Q, b, (n, self.Hq, self.D))

    def new_k(self, b):
        """prefill: raw keys of the question tokens; decode: raw keys of the private segment."""
        r = self.requests[b]
        if r.mode == "prefill":
            return self._get(KIND_NEW_K, b, (r.T, self.Hkv, self.D))
        return self._get(KIND_PRIV_K, b, (r.priv_len, self.Hkv, self.D))

    def new_v(self, b):
        r = self.requests[b]
        if r.mode == "prefill":
            return self._get(KIND_NEW_V, b, (r.T, self.Hkv, self.D))
        return self._get(KIND_PRIV_V, b, (r.priv_len, self.Hkv, self.D))

    # ---------------- device values (torch) ----------------
    # ---------------- decode steps after a prefill (chain) ----------------
    def step_q(self, b, step):
        """Query of request b at decode step `step`: [1, Hq, D]."""
        return self._get(KIND_STEP_Q, step_index(b, step), (1, self.Hq, self.D))

    def step_k(self, b, step):
        """Raw key of the token generated at that step: [1, Hkv, D]."""
        return self._get(KIND_STEP_K, step_index(b, step), (1, self.Hkv, self.D))

    def step_v(self, b, step):
        return self._get(KIND_STEP_V, step_index(b, step), (1, self.Hkv, self.D))

    def step_q_torch(self, b, step, device):
        return normal_torch(self.seed, KIND_STEP_Q, step_index(b, step), (1, self.Hq, self.D),
                            self.dtype, device)

    def step_kv_torch(self, b, step, device):
        s = (1, self.Hkv, self.D)
        return (normal_torch(self.seed, KIND_STEP_K, step_index(b, step), s, self.dtype, device),
                normal_torch(self.seed, KIND_STEP_V, step_index(b, step), s, self.dtype, device))

    def doc_kv_torch(self, d, device):
        s = (self.doc_len, self.Hkv, self.D)
        return (normal_torch(self.seed, KIND_DOC_K, d, s, self.dtype, device),
                normal_torch(self.seed, KIND_DOC_V, d, s, self.dtype, device))

    def q_torch(self, b, device):
        r = self.requests[b]
        n = r.T if r.mode == "prefill" else 1
        return normal_torch(self.seed, KIND_Q, b, (n, self.Hq, self.D), self.dtype, device)

    def new_kv_torch(self, b, device):
        r = self.requests[b]
        if r.mode == "prefill":
            s = (r.T, self.Hkv, self.D)
            return (normal_torch(self.seed, KIND_NEW_K, b, s, self.dtype, device),
                    normal_torch(self.seed, KIND_NEW_V, b, s, self.dtype, device))
        s = (r.priv_len, self.Hkv, self.D)
        return (normal_torch(self.seed, KIND_PRIV_K, b, s, self.dtype, device),
                normal_torch(self.seed, KIND_PRIV_V, b, s, self.dtype, device))

    # ---------------- byte accounting ----------------
    def kv_bytes_per_token(self) -> int:
        return 2 * self.Hkv * self.D * (2 if self.dtype == "bf16" else 4)


def zipf_distinct(rng: np.random.Generator, n_pool: int, alpha: float, k: int) -> List[int]:
    """k distinct doc ids, each draw P(id = r-1) ∝ r^-alpha; duplicates are redrawn."""
    if k > n_pool:
        raise ValueError("cannot draw more distinct docs than the pool holds")
    w = np.arange(1, n_pool + 1, dtype=np.float64) ** (-alpha)
    cdf = np.cumsum(w / w.sum())
    cdf[-1] = 1.0
    out: List[int] = []
    seen = set()
    while len(out) < k:
        u = rng.random(64)
        for d in np.searchsorted(cdf, u, side="right"):
            d = int(min(d, n_pool - 1))
            if d not in seen:
                seen.add(d)
                out.append(d)
                if len(out) == k:
                    break
    return out


def _docs_at_offsets(rng, n_pool, alpha, k, doc_len):
    docs = zipf_distinct(rng, n_pool, alpha, k)
    order = rng.permutation(k)
    docs = [docs[i] for i in order]
    offsets = [i * doc_len for i in range(k)]
    return docs, offsets


def request_stream(n_requests: int, n_pool: int, docs_per_req: int, alpha: float,
                   seed: int = 0) -> List[List[int]]:
    """A stream of retrievals for the cache-hit simulator: each request draws ``docs_per_req``
    distinct Zipf(alpha) documents and puts them in a random order, as the workloads do."""
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 99])))
    return [_docs_at_offsets(rng, n_pool, alpha, docs_per_req, 1)[0] for _ in range(n_requests)]


# ----------------------------------------------------------------------------------------------
# The five workloads (and scaled-down variants with the same structure for parity tests)
# ----------------------------------------------------------------------------------------------
def tiny_fp32(seed: int = 0) -> Workload:
    """1 request, 1 head, D=64, fp32, base 1e4; docs 0 and 1 (16 tokens) at offsets 0 and 16;
    8 question tokens at positions 32..39 (causal among themselves, full view of both docs)."""
    req = Request(index=0, mode="prefill", docs=[0, 1], offsets=[0, 16], T=8, q_pos0=32)
    return Workload("tiny_fp32", "fp32", 1, 1, 64, 10000.0, 16, 16, 2, [req], seed)


def decode_workload(batch=64, docs_per_req=8, doc_len=512, n_pool=1000, alpha=1.0, question=64,
                    Hq=32, Hkv=8, D=128, base=500000.0, seed=0, name="decode_b64",
                    no_reuse=False) -> Workload:
    """Decode step: each request holds ``docs_per_req`` distinct Zipf docs in random order at
    offsets 0, L, 2L, ..., then a private segment (question + the new token) right after them;
    the query is the new token. ``no_reuse`` gives every request its own documents (pool =
    batch x docs_per_req), the control in which no page is shared between requests."""
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence(seed)))
    if no_reuse:
        n_pool = batch * docs_per_req
    reqs = []
    for b in range(batch):
        if no_reuse:
            order = rng.permutation(docs_per_req)
            docs = [b * docs_per_req + int(i) for i in order]
            offs = [i * doc_len for i in range(docs_per_req)]
        else:
            docs, offs = _docs_at_offsets(rng, n_pool, alpha, docs_per_req, doc_len)
        o_priv = docs_per_req * doc_len
        plen = question + 1
        reqs.append(Request(index=b, mode="decode", docs=docs, offsets=offs,
                            priv_offset=o_priv, priv_len=plen, m=o_priv + plen - 1))
    return Workload(name, "bf16", Hq, Hkv, D, base, 16, doc_len, n_pool, reqs, seed)


def prefill_workload(batch=8, docs_per_req=16, doc_len=1024, n_pool=2000, alpha=1.0, T=256,
                     Hq=32, Hkv=8, D=128, base=500000.0, seed=0, name="prefill_b8") -> Workload:
    """Prefill: ``docs_per_req`` distinct Zipf docs in random order, then T question tokens."""
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence(seed)))
    reqs = []
    for b in range(batch):
        docs, offs = _docs_at_offsets(rng, n_pool, alpha, docs_per_req, doc_len)
        reqs.append(Request(index=b, mode="prefill", docs=docs, offsets=offs, T=T,
                            q_pos0=docs_per_req * doc_len))
    return Workload(name, "bf16", Hq, Hkv, D, base, 16, doc_len, n_pool, reqs, seed)


def long_decode_workload(batch=16, docs_per_req=64, doc_len=2048, n_pool=512, alpha=1.2,
                         Hq=32, Hkv=8, D=128, base=500000.0, seed=0,
                         name="long_decode_b16") -> Workload:
    """Long-context decode: 64 docs x 2048 tokens (131072 keys) + the new token at 131072."""
    return decode_workload(batch, docs_per_req, doc_len, n_pool, alpha, 0, Hq, Hkv, D, base, seed,
                           name)


def mixed_workload(alpha: float, batch=128, n_pool=4096, doc_len=1024, docs_lo=8, docs_hi=32,
                   q_lo=128, q_hi=512, prefill_frac=0.25, Hq=32, Hkv=8, D=128, base=500000.0,
                   seed=0, name=None) -> Workload:
    """Mixed serving step: U{docs_lo..docs_hi} Zipf(alpha) docs per request; the first 25% of a
    seeded shuffle prefill a U{q_lo..q_hi}-token question, the rest decode one token after a
    U{q_lo..q_hi}-token private segment."""
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence(seed)))
    n_docs = rng.integers(docs_lo, docs_hi + 1, size=batch)
    qlen = rng.integers(q_lo, q_hi + 1, size=batch)
    is_prefill = np.zeros(batch, dtype=bool)
    is_prefill[rng.permutation(batch)[: int(round(prefill_frac * batch))]] = True
    reqs = []
    for b in range(batch):
        docs, offs = _docs_at_offsets(rng, n_pool, alpha, int(n_docs[b]), doc_len)
        o = int(n_docs[b]) * doc_len
        if is_prefill[b]:
            reqs.append(Request(index=b, mode="prefill", docs=docs, offsets=offs, T=int(qlen[b]),
                                q_pos0=o))
        else:
            plen = int(qlen[b]) + 1
            reqs.append(Request(index=b, mode="decode", docs=docs, offsets=offs, priv_offset=o,
                                priv_len=plen, m=o + plen - 1))
    return Workload(name or f"mixed_a{alpha}", "bf16", Hq, Hkv, D, base, 16, doc_len, n_pool,
                    reqs, seed)


def custom(mode: str, segs: List[List[Tuple[int, int]]], doc_len: int, n_pool: int, *, Hq=4,
           Hkv=2, D=64, dtype="bf16", base=10000.0, T=None, q_pos0=None, priv=None,
           seed=0, name="custom") -> Workload:
    """Hand-laid workload for edge cases. ``segs[b]`` lists (doc, offset) pairs; gaps, overlaps
    and repeated docs are allowed. prefill: T[b] question tokens at q_pos0[b]. decode:
    priv[b] = (priv_offset, priv_len); the query sits at priv_offset + priv_len - 1."""
    reqs = []
    for b, s in enumerate(segs):
        docs = [d for d, _ in s]
        offs = [o for _, o in s]
        if mode == "prefill":
            reqs.append(Request(index=b, mode="prefill", docs=docs, offsets=offs, T=T[b],
                                q_pos0=q_pos0[b]))
        else:
            po, pl = priv[b]
            reqs.append(Request(index=b, mode="decode", docs=docs, offsets=offs, priv_offset=po,
                                priv_len=pl, m=po + pl - 1))
    return Workload(name, dtype, Hq, Hkv, D, base, 16, doc_len, n_pool, reqs, seed)
