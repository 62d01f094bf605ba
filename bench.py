"""Benchmark of the deferred-RoPE attention path on GB300.

Headline (the ``value`` of the JSON line): decode KV GB/s on the decode-step workload
(64 requests x 8 Zipf(1.0) docs of 512 tokens + 65-token private segment, 32/8/128 bf16, RoPE
base 5e5, page size 16), each request's segments in the phase-aligned order (a document shared
by several requests placed where the decode's warps reach it at about the same time). One step = append each request's new token to its private
segment (kv_pool_write_tokens) + lazy_attn_decode (split-KV kernel + log-sum-exp combine).
GB/s counts the logical K+V bytes each request attends (4096 B per key). Before every timed step
the L2 is flushed: a 512 MB write, then a 512 MB read, so that shared documents come from HBM
and the cache holds clean lines (the write-back of the flush's own dirty lines stays outside
the timed region; a control line times the write-only flush).

Extra objects on the same line:
  roofline      of the decode call against MEASURED_PEAKS.json: achieved = the step's unique
                K+V bytes (each distinct cached page once, the least any schedule must read)
                over the call's time; beside it the DRAM bytes ncu counted for the kernel, the
                logical-byte rate and the no-reuse control.
  prefill       TFLOP/s of lazy_attn_prefill on the prefill workload (8 requests x 16 docs of
                1024 + 256-token causal question), causal-visible QK^T + PV FLOPs only.
  long_decode   KV GB/s and tokens/s on the long-context decode (16 x 131073 keys).
  cpu_baseline  the fp64 oracle on the host cores over a bounded sample of the same workload.
  e2e           the decode step through the public API from pinned host buffers, transfers inside
                the timed region: the inputs uploaded by lazy_copy_to_device (SM-driven reads
                of the pinned buffer), the output written by the decode into pinned memory.

--impl reference times the oracle (the only reference arm this path has) on the host cores.
Multi-GPU: replicas only (the path needs no exchange); value = units of all ranks / max time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

L2_FLUSH_BYTES = 512 << 20


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(
            p.get("bf16_tflops_sustained", p["bf16_tflops"])), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 20 ms from before the warm-up until
    after the last timed step. summary() keeps only the samples whose timestamp falls inside a
    timed window (see _timed_steps), so the median is taken under load."""

    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def _start(self, interval_ms):
        return subprocess.Popen(
            ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
             "--format=csv,noheader,nounits", "-lms", str(interval_ms)],
            stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)

    def __enter__(self):
        try:
            self.proc = self._start(20)
            time.sleep(0.5)                      # let the first samples start before timing
            if self.proc.poll() is not None:     # interval refused: fall back to 100 ms
                self.proc = self._start(100)
                time.sleep(0.5)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    @staticmethod
    def _stamp(text):
        import datetime
        try:
            return datetime.datetime.strptime(text.strip(), "%Y/%m/%d %H:%M:%S.%f").timestamp()
        except ValueError:
            return None

    def summary(self, windows=None):
        sm, mx, reasons, total = [], None, set(), 0
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 10:
                continue
            try:
                clk, mxv = float(f[2]), float(f[3])
            except ValueError:
                continue
            total += 1
            t = self._stamp(f[0])
            if windows and t is not None and not any(a <= t <= b for a, b in windows):
                continue
            sm.append(clk)
            mx = mxv
            for n, v in zip(names, f[6:10]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm), "samples_total": total,
                "timed_windows_ms": round(sum(b - a for a, b in (windows or [])) * 1e3, 1)}


def _dist():
    import torch
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws > 1:
        import torch.distributed as dist
        local = int(os.environ.get("LOCAL_RANK", "0"))
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
        return dist.get_rank(), ws, local
    return 0, 1, 0


def _barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def _max_over_ranks(x, ws):
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _job_rate(units_per_rank, slowest_ms, ws):
    """Whole-job rate (units/s): the units all ranks processed over the slowest rank's time
    (_max_over_ranks of the per-rank times)."""
    return ws * units_per_rank / (slowest_ms * 1e-3)


# ------------------------------------------------------------------------------------------------
# Our arm
# ------------------------------------------------------------------------------------------------
def _dist_ms(times):
    """Median, p10 and p90 of per-step times (ms)."""
    t = sorted(times)

    def q(f):
        x = f * (len(t) - 1)
        lo = int(x)
        hi = min(lo + 1, len(t) - 1)
        return t[lo] + (t[hi] - t[lo]) * (x - lo)
    return {"median": round(q(0.5), 5), "p10": round(q(0.1), 5), "p90": round(q(0.9), 5),
            "n": len(t)}


def _cpu_model():
    try:
        import subprocess
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.lower().startswith("model name"):
                return ln.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for ln in f:
                k = ln.split(":")[0].strip().lower()
                if k in ("model name", "cpu model", "hardware"):
                    return ln.split(":", 1)[1].strip()
        import platform
        return platform.processor() or platform.machine()
    except OSError:
        return None


TIMED_WINDOWS = []   # host wall-clock spans of every timed region, for the clock samples


def _prefill_workspace(pk, pool, pb, hq):
    """The prefill's scratch, allocated once outside the timed region."""
    import torch
    n = pk.lazy_prefill_workspace_bytes(pool, int(pb.cu_q.shape[0]) - 1, pb.total_q, pb.max_q_len,
                                        hq)
    return torch.empty(max(n, 1), dtype=torch.uint8, device="cuda")


def _timed_steps(fn, steps, flush, stream):
    """Run `steps` calls of fn, each after an untimed L2 flush; return per-step ms (events).
    The wall-clock span of the region is appended to TIMED_WINDOWS."""
    import torch
    torch.cuda.synchronize()
    t0 = time.time()
    times = []
    for _ in range(steps):
        flush()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        times.append((a, b))
    torch.cuda.synchronize()
    TIMED_WINDOWS.append((t0, time.time()))
    return [a.elapsed_time(b) for a, b in times]


def shared_decode_bench(args, flush, stream):
    """lazy_attn_decode_shared (identical document segments of two requests paired in one
    fragment, one page load for both) against lazy_attn_decode, on decode_b64 and
    long_decode_b16, with the page tables in aligned and in context order."""
    import numpy as np
    import torch

    import position_independent_kv_lazy_gb300 as pk
    import workload as W
    from position_independent_kv_lazy_gb300 import harness as H
    out = {"note": "the plan is built on the host from the page tables, outside the timed calls"}
    for name, mk in (("decode_b64", W.decode_workload), ("long_decode_b16",
                                                         W.long_decode_workload)):
        wl = mk()
        src = H.DeviceSource(wl)
        res = H.build_resident(wl, src)
        rec = {}
        for order, align in (("aligned", True), ("context_order", False)):
            db = H.decode_batch(wl, res, src, align_shared=align)
            plan_h = pk.lazy_decode_shared_plan(db.words.cpu().numpy().view(np.uint64),
                                                db.cu_pages.cpu().numpy())
            plan = plan_h.to("cuda")
            B = len(db.reqs)
            o = torch.empty_like(db.q)
            l = torch.empty((B, wl.Hq), dtype=torch.float32, device="cuda")
            ws_d = torch.empty(pk.lazy_decode_workspace_bytes(res.pool, B, wl.Hq),
                               dtype=torch.uint8, device="cuda")
            ws_s = torch.empty(pk.lazy_decode_shared_workspace_bytes(res.pool, plan.n_units,
                                                                      wl.Hq),
                               dtype=torch.uint8, device="cuda")
            kvb = db.n_keys * wl.kv_bytes_per_token()

            def per_request():
                pk.lazy_attn_decode(res.pool, db.q, db.q_pos, db.words, db.cu_pages,
                                    sm_scale=wl.sm_scale, out=o, lse=l, workspace=ws_d)

            def shared():
                pk.lazy_attn_decode_shared(res.pool, db.q, db.q_pos, plan, sm_scale=wl.sm_scale,
                                           out=o, lse=l, workspace=ws_s)

            r = {"pages": int(db.cu_pages[-1].item()), "units": plan.n_units,
                 "entries": plan_h.n_entries}
            for tag, fn in (("per_request", per_request), ("shared", shared)):
                for _ in range(args.warmup):
                    flush(); fn()
                ms = _timed_steps(fn, max(3, args.steps // 2), flush, stream)
                med = sorted(ms)[len(ms) // 2]
                r[tag] = {"value": round(kvb / (med * 1e-3) / 1e9, 2), "unit": "GB/s",
                          "ms_per_call": round(med, 5)}
            if pk.lazy_get_device_error(res.pool) != 0:
                raise RuntimeError("device error in the shared decode bench")
            rec[order] = r
        out[name] = rec
        del res, src
        torch.cuda.empty_cache()
    return out


def rotation_side_bench(args, flush, stream, tc_peak=None):
    """The prefill on prefill_b8 with the relative rotation on the key side (every cached key
    page rotated by R(o - m0)) and on the query side (the query rows reloaded as R(m - o) q once
    per document offset): same attention, 3/(4M) against 3/(4 L_d) rotation work per key. Both
    kernels: CUDA-core (fp32) and tensor-core (fp16 Q.K; its query-side mode still converts
    every key tile to fp16)."""
    import torch

    import position_independent_kv_lazy_gb300 as pk
    import workload as W
    from position_independent_kv_lazy_gb300 import harness as H
    wl = W.prefill_workload()
    src = H.DeviceSource(wl)
    res = H.build_resident(wl, src, resident_pool=False)
    pb = H.prefill_batch(wl, res, src)
    o = torch.empty_like(pb.q)
    l = torch.empty((pb.total_q, wl.Hq), dtype=torch.float32, device="cuda")
    out = {"workload": "prefill_b8 (16 docs x 1024 + 256 question tokens per request), "
                       "CUDA-core kernel, fp32 arithmetic"}
    for tag, fl in (("key_side", pk.LAZY_PREFILL_SIMT), ("query_side", pk.LAZY_PREFILL_SIMT_QSIDE)):
        def call():
            pk.lazy_attn_prefill(res.pool, pb.q, pb.k_new, pb.v_new, pb.cu_q, pb.q_pos0,
                                 pb.words, pb.cu_pages, pb.max_q_len, sm_scale=wl.sm_scale,
                                 out=o, lse=l, flags=fl)
        flush(); call()
        ms = _timed_steps(call, 3, flush, stream)
        med = sorted(ms)[1]
        out[tag] = {"value": round(pb.flops / (med * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
                    "ms_per_call": round(med, 4)}
    ws = _prefill_workspace(pk, res.pool, pb, wl.Hq)
    tc = {}
    for tag, fl in (("key_side", pk.LAZY_PREFILL_TC), ("query_side", pk.LAZY_PREFILL_TC_QSIDE)):
        def call():
            pk.lazy_attn_prefill(res.pool, pb.q, pb.k_new, pb.v_new, pb.cu_q, pb.q_pos0,
                                 pb.words, pb.cu_pages, pb.max_q_len, sm_scale=wl.sm_scale,
                                 out=o, lse=l, workspace=ws, flags=fl)
        for _ in range(3):
            flush(); call()
        ms = _timed_steps(call, max(5, args.steps // 2), flush, stream)
        med = _dist_ms(ms)["median"]
        tf = pb.flops / (med * 1e-3) / 1e12
        tc[tag] = {"value": round(tf, 2), "unit": "TFLOP/s", "ms_per_call": round(med, 4)}
        if tc_peak:
            tc[tag]["frac"] = round(tf / tc_peak, 4)
    out["tensor_core"] = tc
    if pk.lazy_get_device_error(res.pool) != 0:
        raise RuntimeError("device error in the rotation-side bench")
    del res, src
    return out


def bench_prefill_only(args):
    """Prefill workload alone (pool sized to the documents used): for profiling runs."""
    import torch

    import position_independent_kv_lazy_gb300 as pk
    import workload as W
    from position_independent_kv_lazy_gb300 import harness as H

    pk.build_library()
    pk.load_library()
    _, tc_peak, _, peak_kind = _peaks()
    stream = torch.cuda.current_stream()
    flush, _ = _make_flush(torch)
    pwl = W.prefill_workload()
    psrc = H.DeviceSource(pwl)
    pres = H.build_resident(pwl, psrc, resident_pool=False)
    pb = H.prefill_batch(pwl, pres, psrc)
    pout = torch.empty_like(pb.q)
    plse = torch.empty((pb.total_q, pwl.Hq), dtype=torch.float32, device="cuda")
    pws = _prefill_workspace(pk, pres.pool, pb, pwl.Hq)

    def prefill_call():
        pk.lazy_attn_prefill(pres.pool, pb.q, pb.k_new, pb.v_new, pb.cu_q, pb.q_pos0, pb.words,
                             pb.cu_pages, pb.max_q_len, sm_scale=pwl.sm_scale, out=pout, lse=plse,
                             workspace=pws)

    for _ in range(args.warmup):
        prefill_call()
    torch.cuda.synchronize()
    if pk.lazy_get_device_error(pres.pool) != 0:
        raise RuntimeError("device error during warm-up")
    torch.cuda.nvtx.range_push("timed_region")
    ms = _timed_steps(prefill_call, args.steps, flush, stream)
    torch.cuda.nvtx.range_pop()
    avg = sum(ms) / len(ms)
    tflops = pb.flops / (avg * 1e-3) / 1e12
    print(json.dumps({"mode": "prefill only", "value": round(tflops, 2), "unit": "TFLOP/s",
                      "ms_per_call": round(avg, 4), "frac": round(tflops / tc_peak, 4),
                      "peak_kind": peak_kind, "steps": args.steps}), flush=True)


def _unique_kv_bytes(words_u64, per_token):
    """K+V bytes of the distinct pages a batch's page words address: each (block) once, with its
    valid tokens (the least any schedule must read from HBM)."""
    import numpy as np
    w = np.asarray(words_u64, dtype=np.uint64)
    blk = (w & np.uint64(0xFFFFFFFF)).astype(np.int64)
    nv = ((w >> np.uint64(58)) + np.uint64(1)).astype(np.int64)
    order = np.lexsort((-nv, blk))
    blk, nv = blk[order], nv[order]
    first = np.ones(len(blk), dtype=bool)
    first[1:] = blk[1:] != blk[:-1]
    return int(nv[first].sum()) * per_token


def _make_flush(torch):
    """L2 flush between timed steps: a 512 MB write, then a 512 MB read. The read evicts the
    write's dirty lines (their write-back happens here, untimed) and leaves the cache holding
    clean lines of a buffer the timed work never touches."""
    wbuf = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    rbuf = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")

    def flush():
        wbuf.zero_()
        rbuf.sum()

    def flush_write_only():
        wbuf.zero_()
    return flush, flush_write_only


def _traffic(name):
    """The recorded ncu DRAM bytes per launch for a workload (profiles/TRAFFIC_FILE), or None
    when the kernel sources have changed since the capture."""
    prof = os.path.join(ROOT, "profiles", TRAFFIC_FILE)
    try:
        with open(prof) as f:
            rec = json.load(f).get(name)
        if rec and rec.get("kernel_hash") == _kernel_hash(name):
            return rec
    except (OSError, ValueError):
        pass
    return None


def bench_materialised_only(args):
    """The copy-per-offset baseline section alone."""
    import torch

    import position_independent_kv_lazy_gb300 as pk
    pk.build_library()
    pk.load_library()
    hbm_peak, tc_peak, _, _ = _peaks()
    flush, _ = _make_flush(torch)
    print(json.dumps({"mode": "materialised only", "materialised": materialised_bench(
        args, flush, torch.cuda.current_stream(), hbm_peak, tc_peak)}), flush=True)


def bench_mqa_only(args):
    """The MQA section alone (decode and prefill with 32 query heads per kv head)."""
    import torch

    import position_independent_kv_lazy_gb300 as pk
    pk.build_library()
    pk.load_library()
    hbm_peak, tc_peak, _, _ = _peaks()
    flush, _ = _make_flush(torch)
    print(json.dumps({"mode": "mqa only", "mqa": mqa_bench(
        args, flush, torch.cuda.current_stream(), hbm_peak, tc_peak)}), flush=True)


def bench_rotation_side_only(args):
    """The key-side / query-side prefill section alone."""
    import torch

    import position_independent_kv_lazy_gb300 as pk
    pk.build_library()
    pk.load_library()
    _, tc_peak, _, _ = _peaks()
    flush, _ = _make_flush(torch)
    print(json.dumps({"mode": "rotation side only", "prefill_rotation_side": rotation_side_bench(
        args, flush, torch.cuda.current_stream(), tc_peak)}), flush=True)


def bench_long_decode_only(args):
    """Long-context decode alone (resident pool of its 512 documents): for profiling runs."""
    import numpy as np
    import torch

    import position_independent_kv_lazy_gb300 as pk
    import workload as W
    from position_independent_kv_lazy_gb300 import harness as H

    pk.build_library()
    pk.load_library()
    hbm_peak, _, _, peak_kind = _peaks()
    stream = torch.cuda.current_stream()
    flush, _ = _make_flush(torch)
    lwl = W.long_decode_workload()
    lsrc = H.DeviceSource(lwl)
    lres = H.build_resident(lwl, lsrc)
    ldb = H.decode_batch(lwl, lres, lsrc, phase_order=True)
    lws = torch.empty(pk.lazy_decode_workspace_bytes(lres.pool, lwl.batch, lwl.Hq),
                      dtype=torch.uint8, device="cuda")
    lout = torch.empty_like(ldb.q)
    llse = torch.empty((lwl.batch, lwl.Hq), dtype=torch.float32, device="cuda")
    l_bytes = ldb.n_keys * lwl.kv_bytes_per_token()
    l_uniq = _unique_kv_bytes(ldb.words.cpu().numpy().view(np.uint64), lwl.kv_bytes_per_token())

    def long_call():
        pk.lazy_attn_decode(lres.pool, ldb.q, ldb.q_pos, ldb.words, ldb.cu_pages,
                            sm_scale=lwl.sm_scale, out=lout, lse=llse, workspace=lws)

    for _ in range(args.warmup):
        flush(); long_call()
    torch.cuda.synchronize()
    if pk.lazy_get_device_error(lres.pool) != 0:
        raise RuntimeError("device error during warm-up")
    ms = _timed_steps(long_call, args.steps, flush, stream)
    avg = sum(ms) / len(ms)
    print(json.dumps({"mode": "long decode only", "value": round(l_bytes / avg / 1e6, 2),
                      "unit": "GB/s", "ms_per_call": round(avg, 4), "unique_bytes": l_uniq,
                      "frac_unique": round(l_uniq / avg / 1e6 / hbm_peak, 4),
                      "peak_kind": peak_kind, "steps": args.steps}), flush=True)


def bench_ours(args):
    import numpy as np
    import torch

    import position_independent_kv_lazy_gb300 as pk
    import workload as W
    from position_independent_kv_lazy_gb300 import harness as H

    rank, ws, local = _dist()
    torch.cuda.set_device(local)
    pk.build_library()
    pk.load_library()
    hbm_peak, tc_peak, tc_sus, peak_kind = _peaks()
    stream = torch.cuda.current_stream()
    flush, flush_write_only = _make_flush(torch)

    # ---------------- decode-step workload (headline)
    wl = W.decode_workload()
    src = H.DeviceSource(wl)
    res = H.build_resident(wl, src)
    # each request's segments in the phase-aligned order: the decode's warps read a document
    # shared by several requests at about the same time (the attention result does not depend
    # on page order); the index-aligned and the context order are timed as controls
    db = H.decode_batch(wl, res, src, phase_order=True)
    adb = H.decode_batch(wl, res, src, align_shared=True)
    cdb = H.decode_batch(wl, res, src)
    per_tok = wl.kv_bytes_per_token()
    kv_bytes = db.n_keys * per_tok  # K and V, 4096 B per key of every request's context
    words_h = db.words.cpu().numpy().view(np.uint64)
    uniq_bytes = _unique_kv_bytes(words_h, per_tok)
    B = wl.batch
    ws_bytes = pk.lazy_decode_workspace_bytes(res.pool, B, wl.Hq)
    workspace = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    out = torch.empty_like(db.q)
    lse = torch.empty((B, wl.Hq), dtype=torch.float32, device="cuda")

    def decode_call():
        pk.lazy_attn_decode(res.pool, db.q, db.q_pos, db.words, db.cu_pages,
                            sm_scale=wl.sm_scale, out=out, lse=lse, workspace=workspace)

    def context_order_call():
        pk.lazy_attn_decode(res.pool, cdb.q, cdb.q_pos, cdb.words, cdb.cu_pages,
                            sm_scale=wl.sm_scale, out=out, lse=lse, workspace=workspace)

    def aligned_order_call():
        pk.lazy_attn_decode(res.pool, adb.q, adb.q_pos, adb.words, adb.cu_pages,
                            sm_scale=wl.sm_scale, out=out, lse=lse, workspace=workspace)

    t_order = time.perf_counter()
    pk.order_segments_by_phase(
        [[(res.doc_blocks[d], o, wl.doc_len) for d, o in zip(r.docs, r.offsets)] +
         [(res.priv_blocks[r.index], r.priv_offset, r.priv_len)] for r in wl.requests],
        *pk.lazy_decode_partition(res.pool, wl.Hq))
    order_host_ms = (time.perf_counter() - t_order) * 1e3

    # the shared-segment path over the index-aligned tables (control): its plan is host data
    # rebuilt from the page tables; its build time is reported beside it
    t_plan = time.perf_counter()
    plan_h = pk.lazy_decode_shared_plan(adb.words.cpu().numpy().view(np.uint64),
                                        adb.cu_pages.cpu().numpy())
    plan_host_ms = (time.perf_counter() - t_plan) * 1e3
    plan = plan_h.to("cuda")
    sws = torch.empty(pk.lazy_decode_shared_workspace_bytes(res.pool, plan.n_units, wl.Hq),
                      dtype=torch.uint8, device="cuda")

    def shared_call():
        pk.lazy_attn_decode_shared(res.pool, adb.q, adb.q_pos, plan, sm_scale=wl.sm_scale,
                                   out=out, lse=lse, workspace=sws)

    def step():
        pk.kv_pool_write_tokens(res.pool, db.new_k, db.new_v, db.slot_mapping, db.local_pos)
        decode_call()

    launches_per_step = 3  # encode (append) + decode kernel + its combine

    # no-reuse control: same shapes, every request with its own documents (logical = DRAM bytes)
    nwl = W.decode_workload(no_reuse=True, name="decode_b64_no_reuse")
    nsrc = H.DeviceSource(nwl)
    nres = H.build_resident(nwl, nsrc)
    ndb = H.decode_batch(nwl, nres, nsrc)
    n_bytes = ndb.n_keys * nwl.kv_bytes_per_token()
    nws = torch.empty(pk.lazy_decode_workspace_bytes(nres.pool, nwl.batch, nwl.Hq),
                      dtype=torch.uint8, device="cuda")
    nout = torch.empty_like(ndb.q)
    nlse = torch.empty((nwl.batch, nwl.Hq), dtype=torch.float32, device="cuda")

    def no_reuse_call():
        pk.lazy_attn_decode(nres.pool, ndb.q, ndb.q_pos, ndb.words, ndb.cu_pages,
                            sm_scale=nwl.sm_scale, out=nout, lse=nlse, workspace=nws)

    # e2e buffers: the step's inputs packed in one pinned host buffer (one H2D copy); the result
    # reaches the host through the decode itself (see e2e_step)
    def _layout(items):
        offs, total = [], 0
        for t in items:
            offs.append(total)
            total += (t.numel() * t.element_size() + 255) // 256 * 256
        return offs, total

    in_src = [db.q, db.new_k, db.new_v, db.words, db.cu_pages, db.q_pos, db.slot_mapping,
              db.local_pos]
    in_offs, in_total = _layout(in_src)
    h_in = torch.empty(in_total, dtype=torch.uint8).pin_memory()
    d_in = torch.empty(in_total, dtype=torch.uint8, device="cuda")

    def _view(buf, off, like):
        n = like.numel() * like.element_size()
        return buf[off:off + n].view(like.dtype).view(like.shape)

    for t, o in zip(in_src, in_offs):
        _view(h_in, o, t).copy_(t.cpu())
    (d_q, d_k, d_v, d_words, d_cu, d_pos, d_slot, d_lpos) = [
        _view(d_in, o, t) for t, o in zip(in_src, in_offs)]
    # out and lse live in pinned host memory, which the GPU addresses directly, so the combine
    # writes the result there
    out_offs, out_total = _layout([out, lse])
    h_res = torch.empty(out_total, dtype=torch.uint8).pin_memory()
    e_out, e_lse = _view(h_res, out_offs[0], out), _view(h_res, out_offs[1], lse)
    h2d = sum(t.numel() * t.element_size() for t in in_src)
    d2h = out.numel() * out.element_size() + lse.numel() * lse.element_size()

    def e2e_step():
        pk.lazy_copy_to_device(d_in, h_in)  # SM-driven upload from the pinned buffer
        pk.kv_pool_write_tokens(res.pool, d_k, d_v, d_slot, d_lpos)
        pk.lazy_attn_decode(res.pool, d_q, d_pos, d_words, d_cu, sm_scale=wl.sm_scale,
                            out=e_out, lse=e_lse, workspace=workspace)

    only_decode = args.only == "decode"

    # ---------------- prefill workload (extra object)
    pwl = W.prefill_workload() if not only_decode else None
    pools = [res.pool, nres.pool]
    if not only_decode:
        psrc = H.DeviceSource(pwl)
        pres = H.build_resident(pwl, psrc)
        pb = H.prefill_batch(pwl, pres, psrc)
        pout = torch.empty_like(pb.q)
        plse = torch.empty((pb.total_q, pwl.Hq), dtype=torch.float32, device="cuda")
        pws = _prefill_workspace(pk, pres.pool, pb, pwl.Hq)
        pools.append(pres.pool)

    def prefill_call():
        pk.lazy_attn_prefill(pres.pool, pb.q, pb.k_new, pb.v_new, pb.cu_q, pb.q_pos0, pb.words,
                             pb.cu_pages, pb.max_q_len, sm_scale=pwl.sm_scale, out=pout, lse=plse,
                             workspace=pws)

    # ---------------- long-context decode (extra object)
    if not only_decode:
        lwl = W.long_decode_workload()
        lsrc = H.DeviceSource(lwl)
        lres = H.build_resident(lwl, lsrc)
        ldb = H.decode_batch(lwl, lres, lsrc, phase_order=True)
        lws = torch.empty(pk.lazy_decode_workspace_bytes(lres.pool, lwl.batch, lwl.Hq),
                          dtype=torch.uint8, device="cuda")
        lout = torch.empty_like(ldb.q)
        llse = torch.empty((lwl.batch, lwl.Hq), dtype=torch.float32, device="cuda")
        l_bytes = ldb.n_keys * lwl.kv_bytes_per_token()
        l_uniq = _unique_kv_bytes(ldb.words.cpu().numpy().view(np.uint64),
                                  lwl.kv_bytes_per_token())
        pools.append(lres.pool)

    def long_call():
        pk.lazy_attn_decode(lres.pool, ldb.q, ldb.q_pos, ldb.words, ldb.cu_pages,
                            sm_scale=lwl.sm_scale, out=lout, lse=llse, workspace=lws)

    # ---------------- mixed serving step, skew sweep (extra object; built and timed one alpha
    # at a time after the main timed region, see mixed_sweep)

    clk = ClockSampler(local).__enter__()
    torch.cuda.synchronize()
    for _ in range(args.warmup):
        flush(); step(); e2e_step(); no_reuse_call(); context_order_call(); shared_call()
        aligned_order_call()
        if not only_decode:
            prefill_call(); long_call()
    torch.cuda.synchronize()
    for pool in pools:
        if pk.lazy_get_device_error(pool) != 0:
            clk.__exit__()
            raise RuntimeError("device error during warm-up")

    torch.cuda.nvtx.range_push("timed_region")
    _barrier(ws)
    torch.cuda.synchronize()
    step_ms = _timed_steps(step, args.steps, flush, stream)
    torch.cuda.synchronize()
    _barrier(ws)
    dec_ms = _timed_steps(decode_call, args.steps, flush, stream)
    e2e_ms = _timed_steps(e2e_step, args.steps, flush, stream)
    nr_ms = _timed_steps(no_reuse_call, args.steps, flush, stream)
    co_ms = _timed_steps(context_order_call, args.steps, flush, stream)
    al_ms = _timed_steps(aligned_order_call, args.steps, flush, stream)
    sh_ms = _timed_steps(shared_call, args.steps, flush, stream)
    wo_ms = _timed_steps(decode_call, args.steps, flush_write_only, stream)
    if not only_decode:
        pre_ms = _timed_steps(prefill_call, max(3, args.steps // 2), flush, stream)
        long_ms = _timed_steps(long_call, max(3, args.steps // 2), flush, stream)
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_pop()

    total_ms = _max_over_ranks(sum(step_ms), ws)
    ms_per_step = total_ms / args.steps
    value = _job_rate(kv_bytes * args.steps, total_ms, ws) / 1e9
    dec_avg = sum(dec_ms) / len(dec_ms)
    e2e_avg = sum(e2e_ms) / len(e2e_ms)
    nr_avg = sum(nr_ms) / len(nr_ms)

    def rate(nbytes, ms):
        return nbytes / (ms * 1e-3) / 1e9

    med = lambda t: sorted(t)[len(t) // 2]  # noqa: E731
    tr = _traffic("decode_b64")
    traffic = tr["bytes_per_launch"] if tr else None
    achieved = rate(uniq_bytes, dec_avg)
    roofline = {
        "bound": "hbm", "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
        "frac": round(achieved / hbm_peak, 4), "traffic": traffic, "peak_kind": peak_kind,
        "kernel": "lazy_attn_decode (decode_mma_kernel + combine_kernel), mean call time",
        "algorithmic_bytes": uniq_bytes,
        "algorithmic": "unique K+V of the step: every distinct cached page once (4096 B per "
                       "valid key per kv-head set), the least any schedule must read",
        "logical_bytes": kv_bytes,
        "logical_frac": round(rate(kv_bytes, dec_avg) / hbm_peak, 4),
        "dram_frac": round(rate(traffic, dec_avg) / hbm_peak, 4) if traffic else None,
        "no_reuse_control": {"achieved": round(rate(n_bytes, nr_avg), 1),
                             "frac": round(rate(n_bytes, nr_avg) / hbm_peak, 4),
                             "bytes": n_bytes,
                             "note": "every request its own documents: logical = unique = "
                                     "DRAM bytes"}}
    line = {
        "metric": "decode KV GB/s (LazyAttention decode step, deferred RoPE, paged pool)",
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) values, Zipf document draws)",
        "config": {"workload": "decode_b64: 64 req x (8 Zipf(1.0) docs x 512 + 65 private) keys, "
                               "Hq32/Hkv8/D128, base 5e5, page 16",
                   "keys_per_step": db.n_keys, "kv_bytes_per_step": kv_bytes,
                   "unique_kv_bytes_per_step": uniq_bytes,
                   "l2": "flushed before every timed step: 512 MB write, then 512 MB read",
                   "decode_path": "lazy_attn_decode over the phase-aligned page tables",
                   "order_host_ms": round(order_host_ms, 3),
                   "parallelism": f"replicas x{ws}"},
        "gpu_launches": launches_per_step * args.steps,
        "roofline": roofline,
        "e2e": {"value": round(ws * rate(kv_bytes, e2e_avg), 2), "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(e2e_avg, 5),
                "transfers": "inputs: one lazy_copy_to_device launch from pinned host memory; "
                             "output: the combine writes out and lse into pinned host memory"},
        "decode_no_reuse": {
            "workload": "decode_b64_no_reuse: same shapes, every request its own 8 docs "
                        "(no page shared, logical bytes = DRAM bytes)",
            "value": round(rate(n_bytes, nr_avg), 2), "unit": "GB/s",
            "ms_per_call": round(nr_avg, 5), "frac": round(rate(n_bytes, nr_avg) / hbm_peak, 4)},
        "decode_aligned_order": {
            "workload": "decode_b64 through lazy_attn_decode with shared documents at the same "
                        "index of every request (index-aligned order)",
            "value": round(rate(kv_bytes, med(al_ms)), 2),
            "unit": "GB/s", "ms_per_call": round(med(al_ms), 5)},
        "decode_shared_plan": {
            "workload": "decode_b64, index-aligned order, through lazy_attn_decode_shared "
                        "(identical document segments of two requests paired in one fragment)",
            "value": round(rate(kv_bytes, med(sh_ms)), 2), "unit": "GB/s",
            "ms_per_call": round(med(sh_ms), 5), "plan_units": plan.n_units,
            "plan_entries": plan_h.n_entries, "plan_host_ms": round(plan_host_ms, 3),
            "note": "the plan is rebuilt on the host from the page tables (plan_host_ms, not "
                    "in ms_per_call)"},
        "decode_context_order": {
            "workload": "decode_b64 through lazy_attn_decode with each request's pages in "
                        "context order (documents not lined up across requests)",
            "value": round(rate(kv_bytes, med(co_ms)), 2),
            "unit": "GB/s", "ms_per_call": round(med(co_ms), 5)},
        "decode_write_only_flush": {
            "workload": "the headline decode call after a write-only L2 flush (512 MB of dirty "
                        "lines left in the cache, written back inside the timed call)",
            "value": round(rate(kv_bytes, med(wo_ms)), 2), "unit": "GB/s",
            "ms_per_call": round(med(wo_ms), 5)},
        "decode_tokens_per_s": round(ws * B / (ms_per_step * 1e-3), 1),
        "step_ms_dist": _dist_ms(step_ms),
        "decode_call_ms_dist": _dist_ms(dec_ms),
        "clocks": None,   # filled in after the last timed section
    }
    if not only_decode:
        pre_avg = sum(pre_ms) / len(pre_ms)
        long_avg = sum(long_ms) / len(long_ms)
        tflops = pb.flops / (pre_avg * 1e-3) / 1e12
        line["prefill"] = {
            "workload": "prefill_b8: 8 req x (16 Zipf(1.0) docs x 1024 + 256 causal question), "
                        "Hq32/Hkv8/D128 bf16",
            "value": round(tflops, 2), "unit": "TFLOP/s", "ms_per_call": round(pre_avg, 4),
            "ms_dist": _dist_ms(pre_ms), "flops_per_call": pb.flops,
            "roofline": {"bound": "tensor", "achieved": round(tflops, 2), "peak": tc_peak,
                         "unit": "TFLOP/s", "frac": round(tflops / tc_peak, 4),
                         "peak_kind": peak_kind}}
        ltr = _traffic("long_decode_b16")
        line["long_decode"] = {
            "workload": "long_decode_b16: 16 req x 131073 keys (64 Zipf(1.2) docs x 2048 + 1), "
                        "phase-aligned page tables, lazy_attn_decode",
            "value": round(rate(l_bytes, long_avg), 2), "unit": "GB/s",
            "tokens_per_s": round(lwl.batch / (long_avg * 1e-3), 1),
            "ms_per_step": round(long_avg, 4), "ms_dist": _dist_ms(long_ms),
            "logical_bytes": l_bytes, "unique_bytes": l_uniq,
            "frac": round(rate(l_uniq, long_avg) / hbm_peak, 4),
            "logical_frac": round(rate(l_bytes, long_avg) / hbm_peak, 4),
            "traffic": ltr["bytes_per_launch"] if ltr else None,
            "dram_frac": round(rate(ltr["bytes_per_launch"], long_avg) / hbm_peak, 4)
            if ltr else None}
    if not only_decode:
        # free the other workloads' pools before the chain's and the 17 GB mixed pools
        del pres, pb, pout, plse, lres, ldb, lws, lout, llse
        torch.cuda.empty_cache()
        line["chain"] = chain_bench(args, flush, stream)
        torch.cuda.empty_cache()
        line["mqa"] = mqa_bench(args, flush, stream, hbm_peak, tc_peak)
        torch.cuda.empty_cache()
        line["alibi"] = alibi_bench(args, flush, stream, hbm_peak, tc_peak)
        torch.cuda.empty_cache()
        line["mixed"] = mixed_sweep(args, flush, stream, hbm_peak)
        torch.cuda.empty_cache()
        line["encode"] = encode_bench(args, flush, stream, hbm_peak)
        torch.cuda.empty_cache()
        line["shared_decode"] = shared_decode_bench(args, flush, stream)
        torch.cuda.empty_cache()
        line["prefill_rotation_side"] = rotation_side_bench(args, flush, stream, tc_peak)
        torch.cuda.empty_cache()
        line["materialised"] = materialised_bench(args, flush, stream, hbm_peak, tc_peak)
    clk.__exit__()
    line["clocks"] = clk.summary(TIMED_WINDOWS)
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, src, kv_bytes, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def encode_bench(args, flush, stream, hbm_peak):
    """Document encode (kv_pool_insert_doc) into blocks the segment already owns, i.e. the K
    rotation at local positions, the V copy and the page scatter, for an 8192-token segment
    and a 65536-token segment (537 MB moved; each is one launch of up to 4096 pages: the large
    one shows whether the short launch is bound by its tail). Bytes moved = read raw K and V +
    write both = 8192 B per token (Hkv 8, D 128, bf16)."""
    import torch

    import position_independent_kv_lazy_gb300 as pk

    hkv, d = 8, 128
    out = {}
    for n_tok in (8192, 65536):
        pool = pk.LazyPool(num_blocks=n_tok // 16, num_kv_heads=hkv, head_dim=d,
                           dtype=torch.bfloat16, rope_base=500000.0)
        g = torch.Generator(device="cuda").manual_seed(0)
        k = torch.randn((n_tok, hkv, d), generator=g, device="cuda").to(torch.bfloat16)
        v = torch.randn((n_tok, hkv, d), generator=g, device="cuda").to(torch.bfloat16)
        ids = pk.kv_pool_insert_doc(pool, k, v)

        def insert():
            pk.kv_pool_insert_doc(pool, k, v, block_ids=ids)

        for _ in range(3):
            flush(); insert()
        torch.cuda.synchronize()
        if pk.lazy_get_device_error(pool) != 0:
            raise RuntimeError("device error in encode")
        ms = _timed_steps(insert, max(5, args.steps // 2), flush, stream)
        med = sorted(ms)[len(ms) // 2]
        moved = n_tok * hkv * d * 2 * 2 * 2
        pool.close()
        del k, v
        rec = {"workload": f"one {n_tok}-token segment, Hkv 8, D 128, bf16, into owned blocks "
                           f"({-(-n_tok // 65536)} launch(es))",
               "value": round(moved / (med * 1e-3) / 1e9, 2), "unit": "GB/s",
               "bytes_moved_per_call": moved, "ms_dist": _dist_ms(ms),
               "frac": round(moved / (med * 1e-3) / 1e9 / hbm_peak, 4)}
        if n_tok == 8192:
            out.update(rec)
        else:
            out["large"] = rec
    return out


def mixed_sweep(args, flush, stream, hbm_peak):
    """Mixed serving step on the skew-sweep workload for alpha in (0.6, 0.9, 1.2): one prefill
    launch (32 requests, 128-512-token questions) and one decode step (96 requests: append +
    split-KV decode + combine) back to back on one stream; aggregate tokens/s plus the KV bytes
    the pool keeps against position-baked copies."""
    import torch

    import position_independent_kv_lazy_gb300 as pk
    import workload as W
    from position_independent_kv_lazy_gb300 import harness as H

    out = {"workload": "mixed: pool 4096 docs x 1024, 128 req x U{8..32} Zipf(alpha) docs, "
                       "32 prefill (U{128..512} question) + 96 decode (U{128..512}+1 private)",
           "unit": "tokens/s", "alphas": {}}
    steps = max(3, args.steps // 5)
    for alpha in (0.6, 0.9, 1.2):
        wl = W.mixed_workload(alpha)
        src = H.DeviceSource(wl)
        res = H.build_resident(wl, src)
        pb = H.prefill_batch(wl, res, src)
        db = H.decode_batch(wl, res, src, phase_order=True)
        ws = torch.empty(pk.lazy_decode_workspace_bytes(res.pool, len(db.reqs), wl.Hq),
                         dtype=torch.uint8, device="cuda")
        dout = torch.empty_like(db.q)
        dlse = torch.empty((len(db.reqs), wl.Hq), dtype=torch.float32, device="cuda")
        pout = torch.empty_like(pb.q)
        plse = torch.empty((pb.total_q, wl.Hq), dtype=torch.float32, device="cuda")
        pws = _prefill_workspace(pk, res.pool, pb, wl.Hq)

        def mixed_step():
            pk.lazy_attn_prefill(res.pool, pb.q, pb.k_new, pb.v_new, pb.cu_q, pb.q_pos0,
                                 pb.words, pb.cu_pages, pb.max_q_len, sm_scale=wl.sm_scale,
                                 out=pout, lse=plse, workspace=pws)
            pk.kv_pool_write_tokens(res.pool, db.new_k, db.new_v, db.slot_mapping, db.local_pos)
            pk.lazy_attn_decode(res.pool, db.q, db.q_pos, db.words, db.cu_pages,
                                sm_scale=wl.sm_scale, out=dout, lse=dlse, workspace=ws)

        for _ in range(args.warmup):
            flush(); mixed_step()
        torch.cuda.synchronize()
        if pk.lazy_get_device_error(res.pool) != 0:
            raise RuntimeError("device error in the mixed step")
        ms = _timed_steps(mixed_step, steps, flush, stream)
        avg = sum(ms) / len(ms)
        tokens = pb.total_q + len(db.reqs)
        acct = H.kv_bytes_accounting(wl)
        out["alphas"][str(alpha)] = {
            "tokens_per_step": tokens, "ms_per_step": round(avg, 4),
            "tokens_per_s": round(tokens / (avg * 1e-3), 1),
            "prefill_tokens": pb.total_q, "decode_tokens": len(db.reqs),
            "unique_docs": len(wl.used_docs()),
            "kv_bytes_resident": acct["resident"],
            "kv_bytes_materialised": acct["materialised"],
            "kv_bytes_per_request_copies": acct["per_request"],
            "materialised_over_resident": round(acct["materialised"] / acct["resident"], 3)}
        del res, pb, db, ws, dout, dlse, pout, plse, src
        torch.cuda.empty_cache()
    return out


def _materialise_warmup(pk, res):
    """One one-token copy into a block that is released again: the stream-ordered allocator's
    first use (milliseconds, once per process) stays out of the timed copies."""
    d0 = next(iter(res.doc_blocks))
    ids = pk.kv_pool_materialise_batch(res.pool, [(res.doc_blocks[d0], 1, 0)])
    pk.kv_pool_release(res.pool, ids[0])


def _copy_device_ms(pk, wl, res, copies, stream, reps=3):
    """Device time of kv_pool_materialise_batch alone: the same copies written again into their
    blocks (same bytes), each call queued behind a sleep kernel so the host's list building and
    launch overlap it and the event pair holds only the page-list upload and the copy kernel."""
    import torch

    spec = [(res.doc_blocks[d], wl.doc_len, o, ids) for (d, o), ids in copies.items()]
    ts = []
    for _ in range(reps):
        torch.cuda.synchronize()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        torch.cuda._sleep(20_000_000)  # ~10 ms of GPU time
        ev[0].record(stream)
        pk.kv_pool_materialise_batch(res.pool, spec, stream=stream)
        ev[1].record(stream)
        torch.cuda.synchronize()
        ts.append(ev[0].elapsed_time(ev[1]))
    return sorted(ts)[len(ts) // 2]


def materialised_bench(args, flush, stream, hbm_peak, tc_peak):
    """The copy-per-offset baseline (a document re-encoded for each offset it is used at, by
    kv_pool_materialise) against the lazy path on identical inputs: the copies' cost (bytes
    resident, time to write them), decode and prefill over the copies, and the rotation
    overhead of the lazy path (the same kernels, keys stored once vs keys at absolute
    positions needing no per-document rotation)."""
    import numpy as np
    import torch

    import position_independent_kv_lazy_gb300 as pk
    import workload as W
    from position_independent_kv_lazy_gb300 import harness as H

    def med_ms(fn, n):
        for _ in range(args.warmup):
            flush(); fn()
        return sorted(_timed_steps(fn, n, flush, stream))[n // 2]

    n_t = max(5, args.steps // 2)
    out = {"note": "copies: one per distinct (document, offset) pair, written by "
                   "kv_pool_materialise (un-rotate by R(-j), re-rotate by R(o + j), applied as their "
                   "exact composition R(o)); decode over "
                   "copies uses page words of offset 0, prefill over copies "
                   "LAZY_PREFILL_ABSOLUTE_KEYS (reference position 0: offset-0 pages are only "
                   "converted to the fp16 Q.K operand type, not rotated); copy_ms is the "
                   "copy's device time (page-list upload + kernel), copy_call_ms the call with "
                   "its host-side list building"}
    # ---- decode: decode_b64 (shared documents) and the no-reuse controls of decode_b64 and
    # long_decode_b16 (every request its own documents: the same bytes both ways, so the time
    # difference is the lazy path's per-document rotation)
    for name, wl in (("decode_b64", W.decode_workload()),
                     ("decode_b64_no_reuse", W.decode_workload(no_reuse=True,
                                                               name="decode_b64_no_reuse")),
                     ("long_decode_b16_no_reuse",
                      W.decode_workload(16, 64, 2048, alpha=1.2, question=0, no_reuse=True,
                                        name="long_decode_b16_no_reuse"))):
        src = H.DeviceSource(wl)
        res = H.build_resident(wl, src, resident_pool=False,
                               extra_blocks=H.materialised_blocks_needed(wl))
        db = H.decode_batch(wl, res, src, phase_order=True)
        _materialise_warmup(pk, res)
        torch.cuda.synchronize()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        ev[0].record(stream)
        copies = H.materialise_copies(wl, res)
        ev[1].record(stream)
        torch.cuda.synchronize()
        copy_call_ms = ev[0].elapsed_time(ev[1])
        copy_ms = _copy_device_ms(pk, wl, res, copies, stream)
        words, cu = H.copy_page_table(wl, res, copies, db.reqs, with_private=True)
        cw = torch.from_numpy(words.view(np.int64)).cuda()
        ccu = torch.from_numpy(cu).cuda()
        B = wl.batch
        o = torch.empty_like(db.q)
        l = torch.empty((B, wl.Hq), dtype=torch.float32, device="cuda")
        wsd = torch.empty(pk.lazy_decode_workspace_bytes(res.pool, B, wl.Hq), dtype=torch.uint8,
                          device="cuda")
        kvb = db.n_keys * wl.kv_bytes_per_token()
        per_doc = wl.doc_len * wl.kv_bytes_per_token()

        def lazy_call():
            pk.lazy_attn_decode(res.pool, db.q, db.q_pos, db.words, db.cu_pages,
                                sm_scale=wl.sm_scale, out=o, lse=l, workspace=wsd)

        def copy_call():
            pk.lazy_attn_decode(res.pool, db.q, db.q_pos, cw, ccu, sm_scale=wl.sm_scale,
                                out=o, lse=l, workspace=wsd)

        t_lazy, t_copy = med_ms(lazy_call, n_t), med_ms(copy_call, n_t)
        if pk.lazy_get_device_error(res.pool) != 0:
            raise RuntimeError("device error in the materialised decode bench")
        out[name] = {
            "distinct_doc_offset_pairs": len(copies), "unique_docs": len(wl.used_docs()),
            "kv_bytes_documents_lazy": len(wl.used_docs()) * per_doc,
            "kv_bytes_documents_copies": len(copies) * per_doc,
            "copy_call_ms": round(copy_call_ms, 4), "copy_ms": round(copy_ms, 4),
            "copy_launches": 1,  # kv_pool_materialise_batch
            "copy_gbs": round(2 * len(copies) * per_doc / (copy_ms * 1e-3) / 1e9, 1),
            "copy_frac": round(2 * len(copies) * per_doc / (copy_ms * 1e-3) / 1e9 / hbm_peak, 4),
            "lazy": {"ms_per_call": round(t_lazy, 5),
                     "value": round(kvb / (t_lazy * 1e-3) / 1e9, 2), "unit": "GB/s"},
            "copies": {"ms_per_call": round(t_copy, 5),
                       "value": round(kvb / (t_copy * 1e-3) / 1e9, 2), "unit": "GB/s"},
            "lazy_over_copies": round(t_lazy / t_copy, 4)}
        del res, db, copies, cw, ccu, src
        torch.cuda.empty_cache()
    for name in ("decode_b64_no_reuse", "long_decode_b16_no_reuse"):
        out[name]["rotation_overhead"] = round(out[name]["lazy_over_copies"] - 1.0, 4)
    # ---- prefill: prefill_b8
    wl = W.prefill_workload()
    src = H.DeviceSource(wl)
    res = H.build_resident(wl, src, resident_pool=False,
                           extra_blocks=H.materialised_blocks_needed(wl))
    pb = H.prefill_batch(wl, res, src)
    _materialise_warmup(pk, res)
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    ev[0].record(stream)
    copies = H.materialise_copies(wl, res)
    ev[1].record(stream)
    torch.cuda.synchronize()
    copy_call_ms = ev[0].elapsed_time(ev[1])
    copy_ms = _copy_device_ms(pk, wl, res, copies, stream)
    words, cu = H.copy_page_table(wl, res, copies, pb.reqs, with_private=False)
    cw = torch.from_numpy(words.view(np.int64)).cuda()
    ccu = torch.from_numpy(cu).cuda()
    po = torch.empty_like(pb.q)
    pl = torch.empty((pb.total_q, wl.Hq), dtype=torch.float32, device="cuda")
    pws = _prefill_workspace(pk, res.pool, pb, wl.Hq)
    per_doc = wl.doc_len * wl.kv_bytes_per_token()

    def prefill(words_, cu_, flags):
        def f():
            pk.lazy_attn_prefill(res.pool, pb.q, pb.k_new, pb.v_new, pb.cu_q, pb.q_pos0, words_,
                                 cu_, pb.max_q_len, sm_scale=wl.sm_scale, out=po, lse=pl,
                                 workspace=pws, flags=flags)
        return f

    t_lazy = med_ms(prefill(pb.words, pb.cu_pages, pk.LAZY_PREFILL_AUTO), n_t)
    t_abs = med_ms(prefill(cw, ccu, pk.LAZY_PREFILL_AUTO | pk.LAZY_PREFILL_ABSOLUTE_KEYS), n_t)
    t_rel = med_ms(prefill(cw, ccu, pk.LAZY_PREFILL_AUTO), n_t)
    if pk.lazy_get_device_error(res.pool) != 0:
        raise RuntimeError("device error in the materialised prefill bench")
    tf = lambda t: round(pb.flops / (t * 1e-3) / 1e12, 2)  # noqa: E731
    out["prefill_b8"] = {
        "distinct_doc_offset_pairs": len(copies), "unique_docs": len(wl.used_docs()),
        "kv_bytes_documents_lazy": len(wl.used_docs()) * per_doc,
        "kv_bytes_documents_copies": len(copies) * per_doc,
        "copy_call_ms": round(copy_call_ms, 4), "copy_ms": round(copy_ms, 4),
        "copy_gbs": round(2 * len(copies) * per_doc / (copy_ms * 1e-3) / 1e9, 1),
        "copy_frac": round(2 * len(copies) * per_doc / (copy_ms * 1e-3) / 1e9 / hbm_peak, 4),
        "lazy": {"ms_per_call": round(t_lazy, 5), "tflops": tf(t_lazy)},
        "copies_absolute_keys": {"ms_per_call": round(t_abs, 5), "tflops": tf(t_abs)},
        "copies_relative_kernel": {"ms_per_call": round(t_rel, 5), "tflops": tf(t_rel),
                                   "note": "the lazy kernel over the copies at offset 0"},
        "rotation_overhead": round(t_lazy / t_abs - 1.0, 4),
        "rotation_overhead_analytic_flops": round(3.0 / (4 * 128), 4)}
    del res, pb, copies, cw, ccu, src
    torch.cuda.empty_cache()
    return out


def chain_bench(args, flush, stream, n_steps=32, reps=3):
    """Prefill -> decode chain on the prefill workload: one lazy_attn_prefill_append (the
    question enters the pool as each request's private segment), then n_steps decode steps
    (token append + decode) over documents + question + generated tokens. L2 is flushed before
    each chain; step inputs are on the device before timing."""
    import torch

    import position_independent_kv_lazy_gb300 as pk
    import workload as W
    from position_independent_kv_lazy_gb300 import harness as H

    wl = W.prefill_workload()
    src = H.DeviceSource(wl)
    res = H.build_resident(wl, src, extra_blocks=H.chain_blocks_needed(wl, n_steps))
    ch = H.chain_setup(wl, res, src, n_steps)
    pb = ch.pb
    steps = [H.chain_step_batch(wl, res, ch, s, src, align_shared=True) for s in range(n_steps)]
    B = len(pb.reqs)
    pout = torch.empty_like(pb.q)
    plse = torch.empty((pb.total_q, wl.Hq), dtype=torch.float32, device="cuda")
    dws = torch.empty(pk.lazy_decode_workspace_bytes(res.pool, B, wl.Hq), dtype=torch.uint8,
                      device="cuda")
    pws = _prefill_workspace(pk, res.pool, pb, wl.Hq)
    dout = torch.empty((B, wl.Hq, wl.D), dtype=torch.bfloat16, device="cuda")
    dlse = torch.empty((B, wl.Hq), dtype=torch.float32, device="cuda")

    def run_chain(events):
        flush()
        e = [torch.cuda.Event(enable_timing=True) for _ in range(n_steps + 2)]
        e[0].record(stream)
        pk.lazy_attn_prefill_append(res.pool, pb.q, pb.k_new, pb.v_new, pb.cu_q, pb.q_pos0,
                                    pb.words, pb.cu_pages, pb.max_q_len, ch.append_slots,
                                    ch.append_local_pos, sm_scale=wl.sm_scale, out=pout,
                                    lse=plse, workspace=pws)
        e[1].record(stream)
        for s, db in enumerate(steps):
            pk.kv_pool_write_tokens(res.pool, db.new_k, db.new_v, db.slot_mapping, db.local_pos)
            pk.lazy_attn_decode(res.pool, db.q, db.q_pos, db.words, db.cu_pages,
                                sm_scale=wl.sm_scale, out=dout, lse=dlse, workspace=dws)
            e[s + 2].record(stream)
        events.append(e)

    warm = []
    run_chain(warm)
    torch.cuda.synchronize()
    if pk.lazy_get_device_error(res.pool) != 0:
        raise RuntimeError("device error in the prefill -> decode chain")
    runs = []
    torch.cuda.synchronize()
    t0 = time.time()
    for _ in range(reps):
        run_chain(runs)
    torch.cuda.synchronize()
    TIMED_WINDOWS.append((t0, time.time()))
    pre = [e[0].elapsed_time(e[1]) for e in runs]
    stp = [e[s + 1].elapsed_time(e[s + 2]) for e in runs for s in range(n_steps)]
    tot = [e[0].elapsed_time(e[-1]) for e in runs]
    tokens = pb.total_q + B * n_steps
    step_bytes = sum(db.n_keys for db in steps) / n_steps * wl.kv_bytes_per_token()
    med = sorted(tot)[len(tot) // 2]
    res.pool.close()
    return {
        "workload": f"prefill_b8 question (8 x 256 tokens) kept in the pool, then {n_steps} "
                    "decode steps of 8 requests (token append + decode), 16 docs x 1024 each",
        "unit": "tokens/s",
        "tokens_per_s": round(tokens / (med * 1e-3), 1),
        "ms_per_chain": _dist_ms(tot),
        "prefill_append_ms": _dist_ms(pre),
        "prefill_append_tflops": round(pb.flops / (sorted(pre)[len(pre) // 2] * 1e-3) / 1e12, 2),
        "decode_step_ms": _dist_ms(stp),
        "decode_step_gbs": round(step_bytes / (sorted(stp)[len(stp) // 2] * 1e-3) / 1e9, 2),
        "reps": reps,
    }


def mqa_bench(args, flush, stream, hbm_peak, tc_peak):
    """Multi-query attention (32 query heads over 1 kv head) on the decode and prefill
    workloads' shapes: decode GB/s of algorithmic K+V (512 B per key) and prefill TFLOP/s."""
    import torch

    import position_independent_kv_lazy_gb300 as pk
    import workload as W
    from position_independent_kv_lazy_gb300 import harness as H

    steps = max(5, args.steps // 2)
    out = {}
    wl = W.decode_workload(Hkv=1, name="decode_b64_mqa")
    src = H.DeviceSource(wl)
    res = H.build_resident(wl, src)
    db = H.decode_batch(wl, res, src, align_shared=True)
    B = len(db.reqs)
    dws = torch.empty(pk.lazy_decode_workspace_bytes(res.pool, B, wl.Hq), dtype=torch.uint8,
                      device="cuda")
    dout = torch.empty_like(db.q)
    dlse = torch.empty((B, wl.Hq), dtype=torch.float32, device="cuda")

    def decode_call():
        pk.lazy_attn_decode(res.pool, db.q, db.q_pos, db.words, db.cu_pages,
                            sm_scale=wl.sm_scale, out=dout, lse=dlse, workspace=dws)

    for _ in range(args.warmup):
        flush(); decode_call()
    ms = _timed_steps(decode_call, steps, flush, stream)
    med = _dist_ms(ms)["median"]
    kv = db.n_keys * wl.kv_bytes_per_token()
    flops = 4.0 * wl.D * wl.Hq * db.n_keys  # QK and PV, every query head against every key
    out["decode"] = {"workload": "decode_b64 shapes with Hkv 1 (32 query heads per kv head)",
                     "value": round(kv / (med * 1e-3) / 1e9, 2), "unit": "GB/s",
                     "ms_dist": _dist_ms(ms), "frac": round(kv / (med * 1e-3) / 1e9 / hbm_peak, 4),
                     "kv_bytes_per_step": kv,
                     "tflops": round(flops / (med * 1e-3) / 1e12, 2),
                     "note": "32 FLOP per K/V byte; the 4 chunks of 8 heads share each page in "
                             "shared memory; the per-page MMA chain, not HBM, bounds it"}
    res.pool.close()
    del res, db, dws
    torch.cuda.empty_cache()

    pwl = W.prefill_workload(Hkv=1, name="prefill_b8_mqa")
    psrc = H.DeviceSource(pwl)
    pres = H.build_resident(pwl, psrc)
    pb = H.prefill_batch(pwl, pres, psrc)
    pout = torch.empty_like(pb.q)
    plse = torch.empty((pb.total_q, pwl.Hq), dtype=torch.float32, device="cuda")
    pws = _prefill_workspace(pk, pres.pool, pb, pwl.Hq)

    def prefill_call():
        pk.lazy_attn_prefill(pres.pool, pb.q, pb.k_new, pb.v_new, pb.cu_q, pb.q_pos0, pb.words,
                             pb.cu_pages, pb.max_q_len, sm_scale=pwl.sm_scale, out=pout,
                             lse=plse, workspace=pws)

    for _ in range(args.warmup):
        flush(); prefill_call()
    torch.cuda.synchronize()
    if pk.lazy_get_device_error(pres.pool) != 0:
        raise RuntimeError("device error in the MQA runs")
    ms = _timed_steps(prefill_call, steps, flush, stream)
    med = _dist_ms(ms)["median"]
    tf = pb.flops / (med * 1e-3) / 1e12
    out["prefill"] = {"workload": "prefill_b8 shapes with Hkv 1 (group 32, 4 tokens per Q tile)",
                      "value": round(tf, 2), "unit": "TFLOP/s", "ms_dist": _dist_ms(ms),
                      "frac": round(tf / tc_peak, 4)}

    # the query-side mode on the same shapes: a Q tile holds 4 tokens, so its re-rotation per
    # document evaluates few angles
    def prefill_qside_call():
        pk.lazy_attn_prefill(pres.pool, pb.q, pb.k_new, pb.v_new, pb.cu_q, pb.q_pos0, pb.words,
                             pb.cu_pages, pb.max_q_len, sm_scale=pwl.sm_scale, out=pout,
                             lse=plse, workspace=pws, flags=pk.LAZY_PREFILL_TC_QSIDE)

    for _ in range(3):
        flush(); prefill_qside_call()
    ms = _timed_steps(prefill_qside_call, steps, flush, stream)
    med = _dist_ms(ms)["median"]
    tf = pb.flops / (med * 1e-3) / 1e12
    out["prefill_query_side"] = {"value": round(tf, 2), "unit": "TFLOP/s",
                                 "ms_dist": _dist_ms(ms), "frac": round(tf / tc_peak, 4)}
    if pk.lazy_get_device_error(pres.pool) != 0:
        raise RuntimeError("device error in the MQA runs")
    pres.pool.close()
    return out


def alibi_bench(args, flush, stream, hbm_peak, tc_peak):
    """ALiBi variant on the decode and prefill workloads' shapes (32/8/128 bf16, standard
    slopes): the same kernels with no rotation and a slope * (n - m) bias."""
    import torch

    import position_independent_kv_lazy_gb300 as pk
    import workload as W
    from position_independent_kv_lazy_gb300 import harness as H

    steps = max(5, args.steps // 2)
    out = {}
    wl = W.decode_workload(name="decode_b64_alibi")
    slopes = W.alibi_slopes(wl.Hq)
    src = H.DeviceSource(wl)
    res = H.build_resident(wl, src, alibi_slopes=slopes)
    db = H.decode_batch(wl, res, src, align_shared=True)
    B = len(db.reqs)
    dws = torch.empty(pk.lazy_decode_workspace_bytes(res.pool, B, wl.Hq), dtype=torch.uint8,
                      device="cuda")
    dout = torch.empty_like(db.q)
    dlse = torch.empty((B, wl.Hq), dtype=torch.float32, device="cuda")

    def decode_call():
        pk.lazy_attn_decode(res.pool, db.q, db.q_pos, db.words, db.cu_pages,
                            sm_scale=wl.sm_scale, out=dout, lse=dlse, workspace=dws)

    for _ in range(args.warmup):
        flush(); decode_call()
    ms = _timed_steps(decode_call, steps, flush, stream)
    med = _dist_ms(ms)["median"]
    kv = db.n_keys * wl.kv_bytes_per_token()
    out["decode"] = {"workload": "decode_b64 with ALiBi (32 standard slopes)",
                     "value": round(kv / (med * 1e-3) / 1e9, 2), "unit": "GB/s",
                     "ms_dist": _dist_ms(ms), "frac": round(kv / (med * 1e-3) / 1e9 / hbm_peak, 4)}
    # the same batch through the shared-segment plan (ALiBi words: page positions)
    import numpy as np
    plan_h = pk.lazy_decode_shared_plan(db.words.cpu().numpy().view(np.uint64),
                                        db.cu_pages.cpu().numpy(), page_positions=True)
    plan = plan_h.to("cuda")
    sws = torch.empty(pk.lazy_decode_shared_workspace_bytes(res.pool, plan.n_units, wl.Hq),
                      dtype=torch.uint8, device="cuda")

    def shared_call():
        pk.lazy_attn_decode_shared(res.pool, db.q, db.q_pos, plan, sm_scale=wl.sm_scale,
                                   out=dout, lse=dlse, workspace=sws)

    for _ in range(args.warmup):
        flush(); shared_call()
    ms = _timed_steps(shared_call, steps, flush, stream)
    med = _dist_ms(ms)["median"]
    out["decode_shared"] = {"workload": "decode_b64 with ALiBi through lazy_attn_decode_shared",
                            "value": round(kv / (med * 1e-3) / 1e9, 2), "unit": "GB/s",
                            "ms_per_call": round(med, 5), "units": plan.n_units,
                            "entries": plan_h.n_entries}
    if pk.lazy_get_device_error(res.pool) != 0:
        raise RuntimeError("device error in the ALiBi decode bench")
    res.pool.close()
    del res, db, dws, plan, sws
    torch.cuda.empty_cache()

    pwl = W.prefill_workload(name="prefill_b8_alibi")
    psrc = H.DeviceSource(pwl)
    pres = H.build_resident(pwl, psrc, alibi_slopes=slopes)
    pb = H.prefill_batch(pwl, pres, psrc)
    pout = torch.empty_like(pb.q)
    plse = torch.empty((pb.total_q, pwl.Hq), dtype=torch.float32, device="cuda")
    pws = _prefill_workspace(pk, pres.pool, pb, pwl.Hq)

    def prefill_call():
        pk.lazy_attn_prefill(pres.pool, pb.q, pb.k_new, pb.v_new, pb.cu_q, pb.q_pos0, pb.words,
                             pb.cu_pages, pb.max_q_len, sm_scale=pwl.sm_scale, out=pout,
                             lse=plse, workspace=pws)

    for _ in range(args.warmup):
        flush(); prefill_call()
    torch.cuda.synchronize()
    if pk.lazy_get_device_error(pres.pool) != 0:
        raise RuntimeError("device error in the ALiBi runs")
    ms = _timed_steps(prefill_call, steps, flush, stream)
    med = _dist_ms(ms)["median"]
    tf = pb.flops / (med * 1e-3) / 1e12
    out["prefill"] = {"workload": "prefill_b8 with ALiBi (32 standard slopes)",
                      "value": round(tf, 2), "unit": "TFLOP/s", "ms_dist": _dist_ms(ms),
                      "frac": round(tf / tc_peak, 4)}
    pres.pool.close()
    return out


# DRAM traffic of the decode kernel, one captured launch per workload (ncu, --clock-control
# none), kept in profiles/TRAFFIC_FILE and reported only while the kernel's sources still hash to
# the recorded value. decode_b64's capture skips the five decode launches of the first warm-up
# iteration (headline step, e2e step, no-reuse, context-order and index-aligned controls) and
# takes the second iteration's headline step. Capture: run the workload's command below with the CSV path in place of
# {csv}, then `python bench.py --record-traffic NAME CSV`.
TRAFFIC_FILE = "decode_traffic.json"
TRAFFIC_SOURCES = ("decode.cu", "lazy_common.cuh")
TRAFFIC_RUNS = {
    "decode_b64": {
        "workload": "decode_b64 (64 req x 4161 keys, Hq32/Hkv8/D128 bf16), phase-aligned page "
                    "tables, lazy_attn_decode",
        "kernel": "decode_mma_kernel",
        "command": "ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum,"
                   "gpu__time_duration.sum --clock-control none -k regex:decode_mma_kernel -s 5 "
                   "-c 1 --csv --log-file {csv} python bench.py --only decode --steps 3 "
                   "--warmup 3 --no-cpu-baseline"},
    "long_decode_b16": {
        "workload": "long_decode_b16 (16 req x 131073 keys, Hq32/Hkv8/D128 bf16), phase-aligned "
                    "page tables, lazy_attn_decode",
        "kernel": "decode_mma_kernel",
        "command": "ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum,"
                   "gpu__time_duration.sum --clock-control none -k regex:decode_mma_kernel -s 4 "
                   "-c 1 --csv --log-file {csv} python bench.py --only long_decode --steps 3 "
                   "--warmup 3"},
}


def _kernel_hash(name):
    """Hash of the decode kernel's sources and of the workload's description."""
    import hashlib
    h = hashlib.sha256(TRAFFIC_RUNS[name]["workload"].encode())
    for src in TRAFFIC_SOURCES:
        with open(os.path.join(ROOT, "position_independent_kv_lazy_gb300", "csrc", src), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def record_traffic(name, csv_path):
    """Add the record of workload `name` to profiles/TRAFFIC_FILE from the CSV its command wrote
    (one captured launch), stamped with the current source hash."""
    import csv
    run = TRAFFIC_RUNS[name]
    vals, kernel = {}, None
    with open(csv_path) as f:
        rows = [r for r in csv.reader(l for l in f if l.startswith('"'))]
    hdr = rows[0]
    ki, mi, vi = hdr.index("Kernel Name"), hdr.index("Metric Name"), hdr.index("Metric Value")
    for r in rows[1:]:
        if run["kernel"] not in r[ki]:
            continue
        kernel = r[ki]
        vals[r[mi]] = float(r[vi].replace(",", ""))
    rd, wr = int(vals["dram__bytes_read.sum"]), int(vals["dram__bytes_write.sum"])
    rec = {"kernel": kernel, "kernel_hash": _kernel_hash(name), "workload": run["workload"],
           "bytes_per_launch": rd + wr, "dram_bytes_read": rd, "dram_bytes_write": wr,
           "gpu_time_ns_under_ncu": int(vals.get("gpu__time_duration.sum", 0)),
           "command": run["command"]}
    path = os.path.join(ROOT, "profiles", TRAFFIC_FILE)
    try:
        with open(path) as f:
            allrec = json.load(f)
    except (OSError, ValueError):
        allrec = {}
    allrec[name] = rec
    with open(path, "w") as f:
        json.dump(allrec, f, indent=1, sort_keys=True)
        f.write("\n")
    print(json.dumps(rec))


def cpu_baseline(wl, src, kv_bytes_total, budget_s):
    """The oracle as it stands, on the host cores, over a bounded sample of the workload's
    requests (all heads), scaled to GB/s of logical KV."""
    import oracle
    view = src.host_view() if hasattr(src, "host_view") else wl
    threads = oracle.default_threads()
    per_req = kv_bytes_total / wl.batch
    t0 = time.perf_counter()
    oracle.attend_request(wl, 0, src=view, threads=threads)
    t1 = time.perf_counter() - t0
    n = max(1, min(wl.batch - 1, int(budget_s / max(t1, 1e-3))))
    t0 = time.perf_counter()
    for b in range(1, 1 + n):
        oracle.attend_request(wl, b, src=view, threads=threads)
    dt = time.perf_counter() - t0
    # the same oracle on one core, one request
    t0 = time.perf_counter()
    oracle.attend_request(wl, wl.batch - 1, src=view, threads=1)
    dt1 = time.perf_counter() - t0
    return {"value": round(n * per_req / dt / 1e9, 4), "unit": "GB/s", "cores": threads,
            "kind": "oracle",
            "sample": f"{n} of {wl.batch} requests, all 32 heads ({n * per_req / 1e9:.3f} GB "
                      f"logical KV, {dt:.1f} s), fp64 C oracle form A",
            "one_core_value": round(per_req / dt1 / 1e9, 4),
            "cpu_model": _cpu_model()}


# ------------------------------------------------------------------------------------------------
# Reference arm: the oracle (fp64 CPU), the only other implementation of this path
# ------------------------------------------------------------------------------------------------
def bench_reference(args):
    import workload as W
    import oracle

    rank = int(os.environ.get("RANK", "0"))
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if rank != 0:
        return
    wl = W.decode_workload()
    kv_per_req = (len(wl.requests[0].docs) * wl.doc_len + wl.requests[0].priv_len) * \
        wl.kv_bytes_per_token()
    threads = oracle.default_threads()
    # each step: one request of the workload, all heads (a bounded sample of the decode step)
    for i in range(args.warmup):
        oracle.attend_request(wl, i % wl.batch, threads=threads)
    t0 = time.perf_counter()
    for i in range(args.steps):
        oracle.attend_request(wl, (args.warmup + i) % wl.batch, threads=threads)
    dt = time.perf_counter() - t0
    value = args.steps * kv_per_req / dt / 1e9
    line = {
        "impl": "reference",
        "metric": "decode KV GB/s (LazyAttention decode step, deferred RoPE, paged pool)",
        "value": round(value, 4), "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1) values, Zipf document draws)",
        "config": {"workload": "decode_b64: 64 req x (8 Zipf(1.0) docs x 512 + 65 private) keys, "
                               "Hq32/Hkv8/D128, base 5e5, page 16",
                   "parallelism": "host cores"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads,
                         "kind": "oracle",
                         "sample": "each step = one request of the decode workload, all heads",
                         "cpu_model": _cpu_model()},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only", choices=["all", "decode", "prefill", "long_decode", "materialised",
                                       "rotation_side", "mqa"],
                    default="all",
                    help="decode / prefill / long_decode: time only that workload (smaller "
                         "footprint, for profiling)")
    ap.add_argument("--record-traffic", nargs=2, metavar=("NAME", "CSV"),
                    help="add workload NAME's decode traffic record (profiles/TRAFFIC_FILE) from "
                         "the ncu CSV of its capture and exit (no GPU needed)")
    args = ap.parse_args()
    if args.record_traffic:
        record_traffic(*args.record_traffic)
        return
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        bench_reference(args)
    elif args.only == "prefill":
        bench_prefill_only(args)
    elif args.only == "long_decode":
        bench_long_decode_only(args)
    elif args.only == "materialised":
        bench_materialised_only(args)
    elif args.only == "rotation_side":
        bench_rotation_side_only(args)
    elif args.only == "mqa":
        bench_mqa_only(args)
    else:
        bench_ours(args)


if __name__ == "__main__":
    main()
