"""Oracle for deferred-RoPE attention over a position-agnostic paged KV cache.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()`` and the bench's
CPU-baseline leg. The product (the CUDA library and its binding) never imports it, and it imports
nothing from the product. It shares no code with the CUDA path; the only common module is the
seeded input generator ``workload`` (which holds none of the method's arithmetic).

Sources followed (pages of "LazyAttention: Efficient Retrieval-Augmented Generation with Deferred
Positional Encoding", technical summaries):
  * "Mathematical equivalence": RoPE attention depends only on n - m, so the deferred form equals
    attention over keys materialised at absolute positions -> form A (``attend_materialised``).
  * "Core concept: deferred positional encoding" and the decoding section: keys are cached
    content-only (here: rotated at document-local positions) and the position is applied on the
    fly -> form B (``attend_lazy``): q rotated by m - o, key by its local index j.
  * Decoding section: (block ID, offset) metadata bit-packed into one word -> ``pack_page``.

Forms:
  A  ``attend_materialised``  C, fp64, threaded (oracle.c)
  S  ``attend_stored``        C, fp64, threaded: form A with the cache's storage step written out
                              (a cached key is round(R(j) k) in the cache's element type, attended
                              at its offset); it differs from A only by that rounding, which
                              shrinks like 1/sqrt(keys) in the log-sum-exp
  B  ``attend_lazy``          C, fp64, single-threaded, small cases
  C  ``attend_bruteforce``    pure Python loops, explicit cos/sin, exp-sum without max shift
  ``textbook_rope_attention`` standard RoPE causal attention over one sequence (positions 0..N-1)

ALiBi variant ("Main contributions" item 4, generalisability: the mechanism also serves ALiBi):
  ``attend_alibi`` / ``attend_request_alibi``  numpy fp64. Keys are cached unrotated; the
  position enters only as the bias slope_h * (n - m) from logical positions at attention time.

Conventions that the summaries leave open (half-split pairing, theta_i = base^(-2i/D),
scale 1/sqrt(D), q head h -> kv head h // (Hq/Hkv), natural-log lse of the scaled scores) are the
plainest readings; every one of them is pinned by a closed-form test in ``tests/``.

Pins: tests/test_oracle_pins.py checks every function above against closed forms, invariants,
brute force and the textbook routine; the page-word spec is pinned by exhaustive boundary and
random round trips.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading
from typing import List, Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (gcc -O2, no fast-math). Returns the path."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", _SRC,
                               "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            dp = ctypes.POINTER(ctypes.c_double)
            ip = ctypes.POINTER(ctypes.c_int64)
            up = ctypes.POINTER(ctypes.c_uint8)
            lib.oracle_attend_materialised.argtypes = [
                ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_double, ctypes.c_int,
                dp, dp, ip, up, ctypes.c_int, dp, ip, dp, dp, ctypes.c_int]
            lib.oracle_attend_materialised.restype = ctypes.c_int
            lib.oracle_attend_lazy.argtypes = [
                ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_double, ctypes.c_int,
                dp, dp, ip, ip, up, ctypes.c_int, dp, ip, dp, dp]
            lib.oracle_attend_lazy.restype = ctypes.c_int
            lib.oracle_rope.argtypes = [ctypes.c_int, ctypes.c_double, ctypes.c_double, dp, dp]
            lib.oracle_rope.restype = None
            lib.oracle_attend_stored.argtypes = [
                ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_double, ctypes.c_int,
                dp, dp, ip, ip, up, up, ctypes.c_int, dp, ip, ctypes.c_int, dp, dp, ctypes.c_int]
            lib.oracle_attend_stored.restype = ctypes.c_int
            lib.oracle_round_bf16.argtypes = [ctypes.c_double]
            lib.oracle_round_bf16.restype = ctypes.c_double
            _lib = lib
    return _lib


def _p(a, t):
    return a.ctypes.data_as(ctypes.POINTER(t))


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


# ----------------------------------------------------------------------------------------------
# Kernel-free primitives
# ----------------------------------------------------------------------------------------------
def rope(x: np.ndarray, pos: float, base: float) -> np.ndarray:
    """R(pos) x for one head vector (half-split pairs (i, i+D/2))."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty_like(x)
    _load().oracle_rope(x.shape[0], float(base), float(pos), _p(x, ctypes.c_double),
                        _p(out, ctypes.c_double))
    return out


def attend_materialised(k_raw, v, key_pos, key_causal, q, q_pos, *, base, scale, threads=None):
    """Form A for one kv head. k_raw, v: [n, D]; q: [n_q, G, D]. Returns (out [n_q,G,D], lse [n_q,G])."""
    k_raw = np.ascontiguousarray(k_raw, dtype=np.float64)
    v = np.ascontiguousarray(v, dtype=np.float64)
    q = np.ascontiguousarray(q, dtype=np.float64)
    n, D = k_raw.shape
    n_q, G, _ = q.shape
    key_pos = np.ascontiguousarray(key_pos, dtype=np.int64)
    key_causal = np.ascontiguousarray(key_causal, dtype=np.uint8)
    q_pos = np.ascontiguousarray(q_pos, dtype=np.int64)
    out = np.zeros((n_q, G, D), dtype=np.float64)
    lse = np.zeros((n_q, G), dtype=np.float64)
    rc = _load().oracle_attend_materialised(
        D, G, float(base), float(scale), n, _p(k_raw, ctypes.c_double), _p(v, ctypes.c_double),
        _p(key_pos, ctypes.c_int64), _p(key_causal, ctypes.c_uint8), n_q, _p(q, ctypes.c_double),
        _p(q_pos, ctypes.c_int64), _p(out, ctypes.c_double), _p(lse, ctypes.c_double),
        threads or default_threads())
    if rc != 0:
        raise ValueError("oracle_attend_materialised rejected its arguments")
    return out, lse


STORE = {"exact": 0, "bf16": 1, "fp32": 2}


def round_bf16(x: float) -> float:
    """x rounded to the nearest bfloat16 (ties to even), as the stored-key form rounds."""
    return float(_load().oracle_round_bf16(float(x)))


def attend_stored(k_raw, v, key_off, key_local, key_stored, key_causal, q, q_pos, *, base, scale,
                  store="bf16", threads=None):
    """Form S for one kv head: a key with key_stored = 1 is the cache's copy
    round(R(local) k) in the cache's element type (``store``: "bf16", "fp32" or "exact"),
    attended at its offset; other keys enter as R(off + local) k. Returns (out, lse)."""
    k_raw = np.ascontiguousarray(k_raw, dtype=np.float64)
    v = np.ascontiguousarray(v, dtype=np.float64)
    q = np.ascontiguousarray(q, dtype=np.float64)
    n, D = k_raw.shape
    n_q, G, _ = q.shape
    key_off = np.ascontiguousarray(key_off, dtype=np.int64)
    key_local = np.ascontiguousarray(key_local, dtype=np.int64)
    key_stored = np.ascontiguousarray(key_stored, dtype=np.uint8)
    key_causal = np.ascontiguousarray(key_causal, dtype=np.uint8)
    q_pos = np.ascontiguousarray(q_pos, dtype=np.int64)
    out = np.zeros((n_q, G, D), dtype=np.float64)
    lse = np.zeros((n_q, G), dtype=np.float64)
    rc = _load().oracle_attend_stored(
        D, G, float(base), float(scale), n, _p(k_raw, ctypes.c_double), _p(v, ctypes.c_double),
        _p(key_off, ctypes.c_int64), _p(key_local, ctypes.c_int64),
        _p(key_stored, ctypes.c_uint8), _p(key_causal, ctypes.c_uint8), n_q,
        _p(q, ctypes.c_double), _p(q_pos, ctypes.c_int64), STORE[store],
        _p(out, ctypes.c_double), _p(lse, ctypes.c_double), threads or default_threads())
    if rc != 0:
        raise ValueError("oracle_attend_stored rejected its arguments")
    return out, lse


def attend_lazy(k_raw, v, key_off, key_local, key_causal, q, q_pos, *, base, scale):
    """Form B for one kv head: s = scale * (R(m - off) q) . (R(local) k)."""
    k_raw = np.ascontiguousarray(k_raw, dtype=np.float64)
    v = np.ascontiguousarray(v, dtype=np.float64)
    q = np.ascontiguousarray(q, dtype=np.float64)
    n, D = k_raw.shape
    n_q, G, _ = q.shape
    key_off = np.ascontiguousarray(key_off, dtype=np.int64)
    key_local = np.ascontiguousarray(key_local, dtype=np.int64)
    key_causal = np.ascontiguousarray(key_causal, dtype=np.uint8)
    q_pos = np.ascontiguousarray(q_pos, dtype=np.int64)
    out = np.zeros((n_q, G, D), dtype=np.float64)
    lse = np.zeros((n_q, G), dtype=np.float64)
    rc = _load().oracle_attend_lazy(
        D, G, float(base), float(scale), n, _p(k_raw, ctypes.c_double), _p(v, ctypes.c_double),
        _p(key_off, ctypes.c_int64), _p(key_local, ctypes.c_int64), _p(key_causal, ctypes.c_uint8),
        n_q, _p(q, ctypes.c_double), _p(q_pos, ctypes.c_int64), _p(out, ctypes.c_double),
        _p(lse, ctypes.c_double))
    if rc != 0:
        raise ValueError("oracle_attend_lazy rejected its arguments")
    return out, lse


def attend_bruteforce(keys, queries, *, base, scale):
    """Form C: pure-Python triple loops, tiny inputs only.

    keys:    list of (pos, causal, k_vec, v_vec)
    queries: list of (pos, q_vec)
    Returns list of (out_vec, lse). Uses exp(s) directly (no max shift) and explicit cos/sin per
    pair, independent of the C code.
    """
    def rot(x, p):
        D = len(x)
        h = D // 2
        y = list(x)
        for i in range(h):
            th = base ** (-2.0 * i / D)
            c, s = math.cos(p * th), math.sin(p * th)
            y[i] = x[i] * c - x[i + h] * s
            y[i + h] = x[i] * s + x[i + h] * c
        return y

    res = []
    for m, qv in queries:
        qr = rot([float(t) for t in qv], m)
        num = None
        den = 0.0
        for p, causal, kv, vv in keys:
            if causal and p > m:
                continue
            kr = rot([float(t) for t in kv], p)
            s = scale * sum(a * b for a, b in zip(qr, kr))
            w = math.exp(s)
            den += w
            if num is None:
                num = [0.0] * len(vv)
            for d in range(len(vv)):
                num[d] += w * float(vv[d])
        if num is None:
            res.append(([0.0] * len(qv), -math.inf))
        else:
            res.append(([t / den for t in num], math.log(den)))
    return res


def textbook_rope_attention(q, k, v, q_positions, base, scale):
    """Standard RoPE attention over ONE sequence whose tokens sit at positions 0..N-1.

    q: [n_q, D] raw queries at ``q_positions``; k, v: [N, D] raw keys/values of the sequence.
    Rotary embedding written the usual way, x*cos + rotate_half(x)*sin with
    rotate_half(x) = cat(-x2, x1); causal mask: key j visible to query at position m iff j <= m.
    Returns (out [n_q, D], lse [n_q]).
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    N, D = k.shape
    inv_freq = 1.0 / (base ** (np.arange(0, D, 2, dtype=np.float64) / D))

    def cos_sin(pos):
        ang = np.outer(np.asarray(pos, np.float64), inv_freq)
        emb = np.concatenate([ang, ang], axis=-1)
        return np.cos(emb), np.sin(emb)

    def rotate_half(x):
        return np.concatenate([-x[:, D // 2:], x[:, : D // 2]], axis=-1)

    ck, sk = cos_sin(np.arange(N))
    cq, sq = cos_sin(q_positions)
    kr = k * ck + rotate_half(k) * sk
    qr = q * cq + rotate_half(q) * sq
    scores = scale * (qr @ kr.T)
    mask = np.arange(N)[None, :] <= np.asarray(q_positions)[:, None]
    scores = np.where(mask, scores, -np.inf)
    mx = scores.max(axis=1, keepdims=True)
    w = np.exp(scores - mx)
    den = w.sum(axis=1, keepdims=True)
    return (w @ v) / den, (mx + np.log(den))[:, 0]


# ----------------------------------------------------------------------------------------------
# Page-word format (block id, offset, valid count in one 64-bit word)
# ----------------------------------------------------------------------------------------------
BLOCK_BITS, OFFSET_BITS, NVALID_BITS = 32, 26, 6


def attend_alibi(k, v, key_pos, key_causal, q, q_pos, slopes, *, scale):
    """ALiBi attention by its plain definition, fp64 (pages' "Main contributions" item 4).

    k, v [n, D] (unrotated keys); key_pos [n] logical positions; key_causal [n] (a causal key is
    visible only to queries at position >= its own; others are always visible); q [nq, G, D];
    q_pos [nq]; slopes [G], the query heads' slopes. For query m and key n:
        score = scale * q.k + slope * (n - m)
    softmax over the visible keys. Returns out [nq, G, D] and lse [nq, G] (natural log of the sum
    of exp(score)); a query with no visible key gets out 0 and lse -inf."""
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    pos = np.asarray(key_pos, np.int64)
    caus = np.asarray(key_causal).astype(bool)
    q = np.asarray(q, np.float64)
    slopes = np.asarray(slopes, np.float64)
    nq, G, D = q.shape
    out = np.zeros((nq, G, D))
    lse = np.full((nq, G), -np.inf)
    for i in range(nq):
        m = int(q_pos[i])
        vis = ~caus | (pos <= m)
        if not vis.any():
            continue
        kv, vv, dn = k[vis], v[vis], (pos[vis] - m).astype(np.float64)
        for g in range(G):
            s = scale * (kv @ q[i, g]) + slopes[g] * dn
            mx = s.max()
            w = np.exp(s - mx)
            l = w.sum()
            out[i, g] = (w @ vv) / l
            lse[i, g] = mx + math.log(l)
    return out, lse


def attend_request_alibi(wl, b, slopes, kv_heads: Optional[Sequence[int]] = None,
                         queries: Optional[Sequence[int]] = None, src=None):
    """ALiBi oracle for request b of a workload (same key layout as ``attend_request``: documents
    at their offsets, then the question / private segment), slopes [Hq]. Returns (out, lse) with
    NaN outside the requested heads / queries."""
    src = src or wl
    r = wl.requests[b]
    Hq, Hkv, D = wl.Hq, wl.Hkv, wl.D
    G = Hq // Hkv
    k_raw, v, off, loc, caus = request_keys(wl, b, src)
    qa = np.asarray(src.q(b))
    n_q = qa.shape[0]
    q_pos = (r.q_pos0 + np.arange(n_q)) if r.mode == "prefill" else np.array([r.m])
    qi = np.arange(n_q) if queries is None else np.asarray(list(queries))
    heads = range(Hkv) if kv_heads is None else kv_heads
    out = np.full((n_q, Hq, D), np.nan)
    lse = np.full((n_q, Hq), np.nan)
    sl = np.asarray(slopes, np.float64)
    for h in heads:
        o, l = attend_alibi(k_raw[:, h, :], v[:, h, :], off + loc, caus,
                            qa[qi][:, h * G:(h + 1) * G, :], q_pos[qi], sl[h * G:(h + 1) * G],
                            scale=wl.sm_scale)
        out[qi, h * G:(h + 1) * G, :] = o
        lse[qi, h * G:(h + 1) * G] = l
    return out, lse


def pack_page(block_id: int, offset: int, n_valid: int) -> int:
    """bits 0-31 block id, bits 32-57 logical offset, bits 58-63 n_valid - 1 (1..64)."""
    if not (0 <= block_id < (1 << BLOCK_BITS)):
        raise ValueError("block id out of range")
    if not (0 <= offset < (1 << OFFSET_BITS)):
        raise ValueError("offset out of range")
    if not (1 <= n_valid <= (1 << NVALID_BITS)):
        raise ValueError("n_valid out of range")
    return block_id | (offset << BLOCK_BITS) | ((n_valid - 1) << (BLOCK_BITS + OFFSET_BITS))


def unpack_page(word: int):
    word &= (1 << 64) - 1
    return (word & 0xFFFFFFFF, (word >> 32) & ((1 << OFFSET_BITS) - 1),
            ((word >> (BLOCK_BITS + OFFSET_BITS)) & ((1 << NVALID_BITS) - 1)) + 1)


# ----------------------------------------------------------------------------------------------
# Request-level oracle over the workload's own segment representation
# ----------------------------------------------------------------------------------------------
def request_keys(wl, b, src=None):
    """Keys of request b in logical order: (k_raw [n,Hkv,D], v, offset [n], local [n], causal [n]).

    Documents first (each at its offset, local positions 0..L-1), then the request's own tokens:
    prefill question keys (causal, at q_pos0 + t) or the decode private segment (at priv_offset + j).
    """
    src = src or wl
    r = wl.requests[b]
    ks, vs, offs, locs, caus = [], [], [], [], []
    for d, o in zip(r.docs, r.offsets):
        kd, vd = np.asarray(src.doc_k(d)), np.asarray(src.doc_v(d))
        L = kd.shape[0]
        ks.append(kd); vs.append(vd)
        offs.append(np.full(L, o, np.int64)); locs.append(np.arange(L, dtype=np.int64))
        caus.append(np.zeros(L, np.uint8))
    kn, vn = np.asarray(src.new_k(b)), np.asarray(src.new_v(b))
    n = kn.shape[0]
    o = r.q_pos0 if r.mode == "prefill" else r.priv_offset
    ks.append(kn); vs.append(vn)
    offs.append(np.full(n, o, np.int64)); locs.append(np.arange(n, dtype=np.int64))
    caus.append(np.full(n, 1 if r.mode == "prefill" else 0, np.uint8))
    return (np.concatenate(ks), np.concatenate(vs), np.concatenate(offs), np.concatenate(locs),
            np.concatenate(caus))


def attend_request(wl, b, kv_heads: Optional[Sequence[int]] = None,
                   queries: Optional[Sequence[int]] = None, form: str = "A", src=None,
                   threads=None):
    """Oracle output of request b: (out [n_q, Hq, D], lse [n_q, Hq]) in float64.

    Only the kv heads in ``kv_heads`` (their G query heads) and the query rows in ``queries`` are
    computed; other entries are NaN. ``src`` supplies the input arrays (defaults to the workload's
    host arrays); it must expose doc_k, doc_v, q, new_k, new_v like ``workload.Workload``.
    ``form``: "A" (materialised), "B" (lazy) or "S" (stored keys: every key the cache holds, i.e.
    the documents and a decode request's private segment, is round(R(j) k) in the workload's
    dtype; a prefill question's own keys are not cached and enter exactly).
    """
    src = src or wl
    r = wl.requests[b]
    Hq, Hkv, D = wl.Hq, wl.Hkv, wl.D
    G = Hq // Hkv
    k_raw, v, off, loc, caus = request_keys(wl, b, src)
    qa = np.asarray(src.q(b))
    n_q = qa.shape[0]
    q_pos = (r.q_pos0 + np.arange(n_q)) if r.mode == "prefill" else np.array([r.m])
    qi = np.arange(n_q) if queries is None else np.asarray(list(queries))
    heads = range(Hkv) if kv_heads is None else kv_heads
    out = np.full((n_q, Hq, D), np.nan)
    lse = np.full((n_q, Hq), np.nan)
    for h in heads:
        qh = qa[qi][:, h * G:(h + 1) * G, :]
        if form == "A":
            o, l = attend_materialised(k_raw[:, h, :], v[:, h, :], off + loc, caus, qh, q_pos[qi],
                                       base=wl.rope_base, scale=wl.sm_scale, threads=threads)
        elif form == "B":
            o, l = attend_lazy(k_raw[:, h, :], v[:, h, :], off, loc, caus, qh, q_pos[qi],
                               base=wl.rope_base, scale=wl.sm_scale)
        elif form == "S":
            stored = np.ones(len(off), np.uint8) if r.mode == "decode" else (caus == 0)
            o, l = attend_stored(k_raw[:, h, :], v[:, h, :], off, loc, stored, caus, qh,
                                 q_pos[qi], base=wl.rope_base, scale=wl.sm_scale,
                                 store=wl.dtype, threads=threads)
        else:
            raise ValueError(form)
        out[qi, h * G:(h + 1) * G, :] = o
        lse[qi, h * G:(h + 1) * G] = l
    return out, lse
