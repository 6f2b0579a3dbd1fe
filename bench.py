"""Benchmark: decode-attention KV bytes read (GB/s) on the gqa32k workload.

Workload (one step): batch 1, 32 query / 8 KV heads, head_dim 128, a
32768-cell context; append one cell (K and V) and decode one token, on an
FP16 cache and on an int8 cache (both formats every step).  The context
grows by one cell per step for 64 steps, as the workload states.  32 layer
caches (32 x 203 MB = 6.5 GB, far above the 129 MB L2) are visited in
turn, so no step reads a cache that is still in L2.

Printed: one JSON line.  `value` = cache bytes the two decodes read per step
(every visible cell, K + V, codes + scales) / step time, over all ranks.
The timed region replays CUDA graphs of the captured steps (the library's C
entry points, called through the binding while capturing); `e2e` repeats
the measurement through the C ABI without graphs (tests/e2e_host.c, plain C
and the CUDA runtime, in its own process), with the step's inputs copied
from pinned host memory (one packed copy) and both outputs read back (one
copy) every step; the same step through the Python binding is timed too,
and the record splits the host cost into the binding's share and the rest
(with more than one rank, or without the C leg, `e2e` is the binding's
leg).  `--impl reference` times the CPU oracle on the same workload.

Beside the step (not in `value`): the K8V4 format (int8 K, rotated 4-bit V)
on the same workload -- decode, one-cell and bulk append, compaction and
gather / scatter -- under the "decode", "append", "compact_f16" and
"persist" keys; and block streaming ("stream"): a whole layer fetched from a
pinned host copy into a device window, against the pinned host-to-device
copy rate.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = ("decode-attn KV bytes read GB/s (% of HBM peak); append Mcells/s; FP16 & int8")
# Layer caches rotated through the timed steps.  The decode's copies mark
# the cache lines they bring in evict-first, and lines of a layer read
# with that policy can outlive a rotation of a few times L2: with 4 to 8
# layers the measured decode time was up to 7 % short of its converged
# value, with 16 and 32 layers the two agree to 0.3 %.
LAYERS = 32
STEPS_PER_LAYER = 64
WORKLOAD_DESC = ("gqa32k: batch 1, n_q 32, n_kv 8, head_dim 128, 32768-cell context + 1 "
                 "appended cell per step (64 steps), K with 4 outlier channels x20; "
                 "each step = append + decode on an FP16 cache and on an int8 cache")


def _config(world: int) -> dict:
    """The workload description both arms print (same keys, same values)."""
    rot_gb = LAYERS * 32769 * 8 * (_row_bytes("f16", 128) + _row_bytes("q8", 128)) / 1e9
    return {"workload": WORKLOAD_DESC, "layers": LAYERS,
            "l2": f"inputs larger than L2: {LAYERS} layer caches rotated, {rot_gb:.1f} GB",
            "graph": f"CUDA graphs of {LAYERS * STEPS_PER_LAYER} captured steps",
            "parallelism": f"replicas x{world}"}


def _dist():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def _max_over_ranks(x: float, dist, world: int, device) -> float:
    """The largest x over all ranks (the timed region is as long as the
    slowest rank's); x itself at world size 1."""
    if world <= 1:
        return x
    import torch

    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _row_bytes(fmt, hd: int) -> int:
    """Cache bytes per (cell, KV head): K and V codes (+ fp16 scale per 64
    dims; K8V4: int8 K + scales, V nibbles + one fp16 scale per 32 dims).
    fmt: "f16", "q8", "k8v4" (or a bool, True meaning "q8")."""
    if fmt is True or fmt == "q8":
        return 2 * (hd + 2 * (hd // 64))
    if fmt == "k8v4":
        return hd + 2 * (hd // 64) + hd // 2 + 2 * (hd // 32)
    return 2 * 2 * hd


def _step_ctx(s: int, L: int) -> int:
    return L + (s // LAYERS) % STEPS_PER_LAYER + 1


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.lines = []
        self.t_on = None
        self.t_off = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append((time.time(), ln.strip()))

    def mark(self, on: bool):
        if on:
            self.t_on = time.time()
        else:
            self.t_off = time.time()

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        for t, ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            rows.append((t, parts))
        during = [p for t, p in rows if self.t_on and self.t_off and
                  self.t_on - 0.15 <= t <= self.t_off + 0.15]
        use = during if during else rows
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(p[1]) for p in use if num(p[1]) is not None]
        smax = [num(p[2]) for p in use if num(p[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in use for i in range(4)
                          if p[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(use),
                "samples_in_timed_region": len(during)}


# --------------------------------------------------------------------------
# the CUDA library arm
# --------------------------------------------------------------------------

def run_kvq(args):
    import torch
    import torch.distributed as dist

    import quantized_kv_cache_append_gb300 as kvq
    import workloads
    from quantized_kv_cache_append_gb300.pool import PagedPool, row_layout

    rank, world, local = _dist()
    kvq.build()
    # the e2e step from plain C runs first, while this process holds no CUDA
    # context on the device (a second live context slowed it 18x)
    c_leg = _e2e_c_leg(min(args.steps, 512), min(args.warmup, 32), local) if rank == 0 else None
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    kvq.load_library()

    wl = workloads.make("gqa32k")
    L, n_kv, hd, n_q, bs = int(wl.ctx_lens[0]), wl.n_kv, wl.head_dim, wl.n_q, wl.block_size
    cap = L + STEPS_PER_LAYER
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    bt = dev(wl.block_table)

    # 8 layers x (FP16 pool, int8 pool), each prefilled with the workload's cells
    k_pre, v_pre = dev(wl.k), dev(wl.v)
    seq_pre, pos_pre = dev(wl.tok_seq), dev(wl.tok_pos)
    layers = []
    for _ in range(LAYERS):
        pair = {}
        # (K8V4, timed beside the step, not in it)
        for name, fmt in (("f16", kvq.KVQ_F16), ("q8", kvq.KVQ_Q8), ("k8v4", kvq.KVQ_K8V4)):
            pool = PagedPool(fmt, n_kv, hd, bs, wl.n_blocks)
            pool.append(k_pre, v_pre, seq_pre, pos_pre, bt)
            ws_bytes = pool.workspace_bytes(1, 1, n_q, cap)
            pair[name] = (pool, torch.zeros(ws_bytes, dtype=torch.uint8, device="cuda"),
                          torch.empty((1, 1, n_q, hd), dtype=torch.float32, device="cuda"))
        layers.append(pair)
    torch.cuda.synchronize()

    # append throughput (bulk: the 32768-cell prefill), outside the timed steps
    append_mcells = {}
    for name in ("f16", "q8", "k8v4"):
        pool = layers[0][name][0]
        for _ in range(3):
            pool.append(k_pre, v_pre, seq_pre, pos_pre, bt)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = 10
        e0.record()
        for _ in range(reps):
            pool.append(k_pre, v_pre, seq_pre, pos_pre, bt)
        e1.record()
        torch.cuda.synchronize()
        append_mcells[name] = L * reps / (e0.elapsed_time(e1) * 1e-3) / 1e6

    # per-step inputs (64 distinct new cells and queries), resident in HBM
    sk = dev(np.stack([st["k"] for st in wl.steps]))          # [64][1][n_kv][hd]
    sv = dev(np.stack([st["v"] for st in wl.steps]))
    sq = dev(np.stack([st["q"] for st in wl.steps]))          # [64][1][1][n_q][hd]
    spos = dev(np.stack([st["tok_pos"] for st in wl.steps]))  # [64][1]
    sctx = dev(np.stack([st["ctx_lens"] for st in wl.steps]))  # [64][1]
    seq0 = dev(np.zeros(1, np.int32))

    def step(s, formats=("f16", "q8"), do_append=True, do_decode=True):
        j = (s // LAYERS) % STEPS_PER_LAYER
        for name in formats:
            pool, ws, out = layers[s % LAYERS][name]
            if do_append:
                pool.append(sk[j], sv[j], seq0, spos[j], bt)
            if do_decode:
                pool.decode(sq[j], sctx[j], cap, bt, wl.sm_scale, out=out, workspace=ws)

    def capture(n, **kw):
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            step(0, **kw)                      # warm the binding outside capture
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        with torch.cuda.graph(g):
            for i in range(n):
                step(i, **kw)
        return g

    chunk = LAYERS * STEPS_PER_LAYER            # every layer through its 64 steps
    g_full = capture(chunk)
    K, W = args.steps, args.warmup
    rem = K % chunk
    g_rem = capture(rem) if rem else None

    def run_steps(n):
        for _ in range(n // chunk):
            g_full.replay()
        if n % chunk:
            if n % chunk == rem and g_rem is not None:
                g_rem.replay()
            else:
                for i in range(n % chunk):
                    step(i)

    bytes_per_step = {"f16": [], "q8": [], "k8v4": []}
    for s in range(chunk):
        ctx = _step_ctx(s, L)
        for name in bytes_per_step:
            bytes_per_step[name].append(ctx * n_kv * _row_bytes(name, hd))
    total_bytes = sum(bytes_per_step["f16"][s % chunk] + bytes_per_step["q8"][s % chunk]
                      for s in range(K))

    # warm-up (untimed), then exactly K timed steps between barriers
    run_steps(W)
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.mark(True)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    run_steps(K)
    e1.record()
    torch.cuda.synchronize()
    clocks.mark(False)
    if world > 1:
        dist.barrier()
    ms = e0.elapsed_time(e1)
    clock_info = clocks.stop()
    ms = _max_over_ranks(ms, dist, world, "cuda")
    value = total_bytes * world / (ms * 1e-3) / 1e9

    # per-kernel durations: graphs of decode-only steps, one format at a time
    kernel_ms = {}
    for name in ("f16", "q8", "k8v4"):
        g = capture(chunk, formats=(name,), do_append=False)
        g.replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        g.replay()
        b.record()
        torch.cuda.synchronize()
        kernel_ms[name] = a.elapsed_time(b) / chunk
    g = capture(chunk, formats=("f16", "q8"), do_decode=False)
    g.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    g.replay()
    b.record()
    torch.cuda.synchronize()
    append_step_us = a.elapsed_time(b) / chunk / 2 * 1e3
    g = capture(chunk, formats=("k8v4",), do_decode=False)
    g.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    g.replay()
    b.record()
    torch.cuda.synchronize()
    append_step_us_k8v4 = a.elapsed_time(b) / chunk * 1e3

    # FP16 compaction of a whole layer (32768 cells, both formats), layers in turn
    compact_us = {}
    ck = torch.empty((n_kv, L, hd), dtype=torch.float16, device="cuda")
    cv = torch.empty_like(ck)
    for name in ("f16", "q8", "k8v4"):
        gc = torch.cuda.CUDAGraph()
        for i in range(LAYERS):
            layers[i][name][0].compact(bt[0], L, ck, cv)
        torch.cuda.synchronize()
        with torch.cuda.graph(gc):
            for i in range(4 * LAYERS):
                layers[i % LAYERS][name][0].compact(bt[0], L, ck, cv)
        gc.replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        gc.replay()
        b.record()
        torch.cuda.synchronize()
        compact_us[name] = a.elapsed_time(b) / (4 * LAYERS) * 1e3

    chunk = _chunk_attn_bench(torch, kvq)

    # gather / scatter of a whole layer's sequence (32768 cells), both formats
    persist_us = {}
    for name in ("f16", "q8", "k8v4"):
        pool0 = layers[0][name][0]
        kdt, kn, vdt, vn, kng, vng = row_layout(pool0.fmt, hd)
        ck = torch.empty((L, n_kv, kn), dtype=kdt, device="cuda")
        cvv = torch.empty((L, n_kv, vn), dtype=vdt, device="cuda")
        sk = sv = None
        if kng:
            sk = torch.empty((L, n_kv, kng), dtype=torch.float16, device="cuda")
            sv = torch.empty((L, n_kv, vng), dtype=torch.float16, device="cuda")
        times = {}
        for op, fn in (("gather", kvq.kvq_gather_cells), ("scatter", kvq.kvq_scatter_cells)):
            for _ in range(3):
                fn(pool0.cache, bt[0], L, ck, cvv, sk, sv)
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            for _ in range(10):
                fn(pool0.cache, bt[0], L, ck, cvv, sk, sv)
            b.record()
            torch.cuda.synchronize()
            times[op] = a.elapsed_time(b) / 10 * 1e3
        persist_us[name] = times

    stream = _stream_bench(torch, kvq, layers, n_kv, hd, bs, wl.n_blocks)

    peak, peak_kind = _peaks()
    by_workload = _decode_workloads(torch, kvq, peak)
    avg_bytes = {n: sum(v) / len(v) for n, v in bytes_per_step.items()}
    gbs = {n: avg_bytes[n] / (kernel_ms[n] * 1e-3) / 1e9 for n in kernel_ms}
    dominant = max(("f16", "q8"), key=kernel_ms.get)   # of the step's two formats
    traffic = _ncu_traffic(dominant)

    # end to end, host buffers, no graphs: through the C ABI (the C leg, run
    # above in its own process) and through the Python binding
    K_e2e = min(K, 512)
    e2e_py = _e2e(step_fn=None, torch=torch, layers=layers, wl=wl, bt=bt, cap=cap, L=L,
                  n_kv=n_kv, hd=hd, K=K_e2e, W=min(W, 32), world=world, dist=dist)
    e2e = e2e_py
    if rank == 0:
        ok = "ms_per_step" in c_leg
        breakdown = {
            "device_ms_per_step": round(ms / K, 4),
            "c_abi": c_leg,
            "binding_ms_per_step": round(e2e_py["ms_per_step"] - c_leg["ms_per_step"], 4) if ok else None,
            "note": ("device: the step's kernels in CUDA graphs; c_abi: the e2e step from plain C "
                     "(tests/e2e_host.c) through the C ABI, host buffers, no graphs, with its host "
                     "microseconds per step in the copies' enqueue, the four library calls and the "
                     "synchronize; binding: the Python binding's leg minus the C one (ctypes "
                     "marshalling and the Python around the calls)"),
        }
        if ok and world == 1:
            # the C ABI leg is the e2e figure: the same steps (context lengths,
            # layers) as the binding's leg, so the same bytes per step
            total = sum(_step_ctx(s, L) * n_kv * (_row_bytes(False, hd) + _row_bytes(True, hd))
                        for s in range(K_e2e))
            e2e = {"value": round(total / (K_e2e * c_leg["ms_per_step"] * 1e-3) / 1e9, 2),
                   "unit": "GB/s", "steps": K_e2e,
                   "h2d_bytes_per_step": int(c_leg["h2d_bytes"]),
                   "d2h_bytes_per_step": int(c_leg["d2h_bytes"]),
                   "ms_per_step": c_leg["ms_per_step"],
                   "path": "C ABI (tests/e2e_host.c), pinned host buffers, copies in the timed region",
                   "python_binding": {k: e2e_py[k] for k in ("value", "unit", "ms_per_step")}}
        else:
            e2e["path"] = "Python binding, pinned host buffers, copies in the timed region"
        e2e["breakdown"] = breakdown

    result = None
    if rank == 0:
        result = {
            "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
            "steps": K, "warmup": W, "ms_per_step": ms / K, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "storage": ["f16", "int8+fp16 scale/64"], "data": "synthetic (seeded N(0,1))",
            "config": _config(world),
            "gpu_launches": 6 * K,
            "roofline": {"kernel": f"decode partial+combine ({dominant})", "bound": "hbm",
                         "achieved": round(gbs[dominant], 1), "peak": peak,
                         "peak_kind": peak_kind, "unit": "GB/s",
                         "frac": round(gbs[dominant] / peak, 4), "traffic": traffic,
                         "algorithmic_bytes_per_launch": int(avg_bytes[dominant]),
                         "launch_us": round(kernel_ms[dominant] * 1e3, 3)},
            "decode": {**{n: {"us": round(kernel_ms[n] * 1e3, 3), "GB/s": round(gbs[n], 1),
                              "frac_of_measured_hbm": round(gbs[n] / peak, 4),
                              "frac_of_nominal_8TBs": round(gbs[n] / 8000.0, 4)}
                          for n in kernel_ms},
                       **by_workload},
            "append": {"bulk_Mcells_per_s": {n: round(v, 1) for n, v in append_mcells.items()},
                       "one_cell_step_us": round(append_step_us, 3),
                       "one_cell_step_us_k8v4": round(append_step_us_k8v4, 3)},
            "chunk_attn": chunk,
            "stream": stream,
            "persist": {n: {op: {"us": round(t, 3),
                                 "GB/s": round(2 * L * n_kv * _row_bytes(n, hd)
                                               / (t * 1e-6) / 1e9, 1)}
                            for op, t in persist_us[n].items()}
                        for n in persist_us},
            "compact_f16": {n: {"us": round(compact_us[n], 3),
                                "GB/s": round(L * n_kv * (_row_bytes(n, hd) + 4 * hd)
                                              / (compact_us[n] * 1e-6) / 1e9, 1),
                                "frac_of_measured_hbm": round(
                                    L * n_kv * (_row_bytes(n, hd) + 4 * hd)
                                    / (compact_us[n] * 1e-6) / 1e9 / peak, 4)}
                            for n in compact_us},
            "clocks": clock_info,
            "e2e": e2e,
        }
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return result


def _decode_workloads(torch, kvq, peak):
    """Decode time of every other workload and cache format, timed like the
    step's decodes: a CUDA graph of decode calls over layer caches rotated
    past L2 (at least 16 layers and 2 GB, at most 64 layers: the tiny
    workload's 64 layers still fit in L2), the partial and combine kernels
    of each call, bytes = the cache rows read (cells x KV heads x row
    bytes)."""
    import workloads
    from quantized_kv_cache_append_gb300.pool import PagedPool

    fmts = {"f16": kvq.KVQ_F16, "q8": kvq.KVQ_Q8, "k8v4": kvq.KVQ_K8V4}
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    res = {}
    for name in ("tiny", "ragged", "long256k", "chunk_verify"):
        wl = workloads.make(name)
        ctx = wl.chunk["ctx_lens"] if wl.chunk is not None else wl.ctx_lens
        bt, q, dctx = dev(wl.block_table), dev(wl.q), dev(ctx)
        k, v, seq, pos = dev(wl.k), dev(wl.v), dev(wl.tok_seq), dev(wl.tok_pos)
        res[name] = {}
        for fn in list(wl.formats) + ["k8v4"]:
            nbytes = int(ctx.sum()) * wl.n_kv * _row_bytes(fn, wl.head_dim)
            nl = max(16, min(64, -(-2_000_000_000 // nbytes)))
            pools = []
            for _ in range(nl):
                p = PagedPool(fmts[fn], wl.n_kv, wl.head_dim, wl.block_size, wl.n_blocks)
                p.append(k, v, seq, pos, bt)
                if wl.chunk is not None:
                    c = wl.chunk
                    p.append(dev(c["k"]), dev(c["v"]), dev(c["tok_seq"]), dev(c["tok_pos"]), bt)
                ws = torch.empty(max(256, p.workspace_bytes(wl.n_seq, wl.W, wl.n_q, int(ctx.max()))),
                                 dtype=torch.uint8, device="cuda")
                pools.append((p, ws, torch.empty_like(q)))

            def one(i):
                p, ws, out = pools[i % nl]
                p.decode(q, dctx, int(ctx.max()), bt, wl.sm_scale, out=out, workspace=ws)

            for i in range(2 * nl):
                one(i)
            torch.cuda.synchronize()
            n = 8 * nl
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                for i in range(n):
                    one(i)
            g.replay()
            torch.cuda.synchronize()
            ts = []
            for _ in range(5):
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record()
                g.replay()
                b.record()
                torch.cuda.synchronize()
                ts.append(a.elapsed_time(b) / n * 1e3)
            us = statistics.median(ts)
            gbs = nbytes / (us * 1e-6) / 1e9
            res[name][fn] = {"us": round(us, 3), "GB/s": round(gbs, 1),
                             "frac_of_measured_hbm": round(gbs / peak, 4),
                             "bytes": nbytes, "layers": nl}
            del pools, g
            torch.cuda.empty_cache()
    return res


def _stream_bench(torch, kvq, layers, n_kv, hd, bs, n_blocks):
    """Block streaming: a whole gqa32k layer (all its blocks) fetched from a
    pinned host copy into an empty window by kvq_stream_fetch, per format,
    against the pinned host-to-device copy of the same runs by the copy
    engine (cudaMemcpyAsync through torch), the link's measured rate."""
    from quantized_kv_cache_append_gb300.pool import PagedPool

    out = {}
    src = torch.arange(n_blocks, dtype=torch.int32, device="cuda")
    for name in ("f16", "q8", "k8v4"):
        dpool = layers[0][name][0]
        host = PagedPool(dpool.fmt, n_kv, hd, bs, n_blocks, pinned=True)
        win = PagedPool(dpool.fmt, n_kv, hd, bs, n_blocks)
        runs = [(h, d) for h, d in ((host.k, dpool.k), (host.v, dpool.v), (host.ks, dpool.ks),
                                    (host.vs, dpool.vs)) if h is not None]
        for h, d in runs:
            h.copy_(d)
        torch.cuda.synchronize()
        nbytes = sum(h.numel() * h.element_size() for h, _ in runs)

        def timed(fn, reps=10):
            for _ in range(3):
                fn()
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            for _ in range(reps):
                fn()
            b.record()
            torch.cuda.synchronize()
            return a.elapsed_time(b) / reps * 1e3

        fetch_us = timed(lambda: kvq.check(
            kvq.kvq_stream_fetch(host.cache, win.cache, src, src, n_blocks), "kvq_stream_fetch"))
        wins = [(w, h) for w, h in ((win.k, host.k), (win.v, host.v), (win.ks, host.ks),
                                    (win.vs, host.vs)) if h is not None]
        copy_us = timed(lambda: [w.copy_(h, non_blocking=True) for w, h in wins])
        ok = all(torch.equal(w, d) for (w, _), (_, d) in zip(wins, runs))
        out[name] = {"bytes": nbytes, "fetch_us": round(fetch_us, 2),
                     "fetch_GB/s": round(nbytes / (fetch_us * 1e-6) / 1e9, 1),
                     "h2d_copy_GB/s": round(nbytes / (copy_us * 1e-6) / 1e9, 1),
                     "frac_of_h2d_copy": round(copy_us / fetch_us, 4), "bits_equal": ok}
        del host, win
    return out


def _chunk_attn_bench(torch, kvq):
    """Prompt-chunk attention at the chunk_verify sizes: a 4096-token chunk
    at the end of 131072 cells, 32/8 heads, head_dim 128, over fp16 staging;
    synthetic N(0, 1) staging and queries.  Tensor-bound: algorithmic flops
    are 4 * head_dim per (query head, visible cell) -- q.k and p.v -- against
    the measured dense bf16 peak (fp16 runs at the same nominal rate).  The
    other head dims the call serves (64 and 256, on the same tcgen05
    kernel) are timed beside it on a 4096-token chunk over 32768 cells
    (16/4 and 16/2 heads), and so is a 256-token chunk over the 131072
    cells (few row tiles: its key tiles are split over clusters of CTAs)."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peak, kind = float(json.load(f)["bf16_tflops"]), "measured bf16 dense"
    except Exception:
        peak, kind = 1900.0, "fallback bf16 dense"

    def timed(n_kv, n_q, hd, P, T, seed):
        g = torch.Generator(device="cuda").manual_seed(seed)
        k16 = torch.randn(n_kv, P, hd, device="cuda", generator=g).half()
        v16 = torch.randn(n_kv, P, hd, device="cuda", generator=g).half()
        q = torch.randn(T, n_q, hd, device="cuda", generator=g)
        out = torch.empty_like(q)
        sm = float(1.0 / np.sqrt(hd))

        def run():
            st = kvq.kvq_chunk_attn(k16, v16, n_kv, P, hd, q, T, n_q, sm, out)
            if st != kvq.KVQ_OK:
                raise RuntimeError(kvq.kvq_status_string(st))

        for _ in range(3):
            run()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = 5
        a.record()
        for _ in range(reps):
            run()
        b.record()
        torch.cuda.synchronize()
        ms = a.elapsed_time(b) / reps
        flops = 4.0 * hd * n_q * (T * (P - T) + T * (T + 1) / 2)
        tflops = flops / (ms * 1e-3) / 1e12
        return ms, tflops

    ms, tflops = timed(8, 32, 128, 131072, 4096, 1005)
    # a short chunk (the tail of a long prompt): 64 (row tile, KV head)
    # CTAs, so each one's key tiles are split over a cluster
    ms_s, tf_s = timed(8, 32, 128, 131072, 256, 1777)
    others = {}
    for hd, n_kv, n_q in ((64, 4, 16), (256, 2, 16)):
        ms_o, tf_o = timed(n_kv, n_q, hd, 32768, 4096, 1005 + hd)
        others[f"hd{hd}"] = {"workload": f"4096-token chunk over 32768 cells, {n_q}/{n_kv} heads, "
                                         f"head_dim {hd} (tcgen05)",
                             "ms": round(ms_o, 3), "TFLOP/s": round(tf_o, 1),
                             "frac": round(tf_o / peak, 4)}
    return {"workload": "4096-token chunk over 131072 cells, 32/8 heads, head_dim 128",
            "ms": round(ms, 3), "TFLOP/s": round(tflops, 1), "peak_TFLOP/s": peak,
            "peak_kind": kind, "frac": round(tflops / peak, 4),
            "note": "tcgen05 MMAs (fp32 accumulators in tensor memory); q as fp16 hi+lo "
                    "(two MMAs for q.k), p as one fp16 value (one MMA for p.v)",
            "other_head_dims": others,
            "short_chunk": {"workload": "256-token chunk over 131072 cells, 32/8 heads, head_dim 128 "
                                        "(key tiles split over clusters of CTAs)",
                            "ms": round(ms_s, 3), "TFLOP/s": round(tf_s, 1), "frac": round(tf_s / peak, 4)}}


def _decode_sources_sha() -> str:
    """sha256[:16] over the decode kernel sources (the partial kernel and
    the combine, and the PTX helpers they use)."""
    h = hashlib.sha256()
    for f in ("kvq_decode_mma.cu", "kvq_ptx.cuh"):
        h.update(open(os.path.join(ROOT, "quantized_kv_cache_append_gb300", "csrc", f),
                      "rb").read())
    return h.hexdigest()[:16]


def _ncu_traffic(fmt: str):
    """DRAM bytes per launch of the decode kernels from the committed ncu
    summary, if it was taken on the current decode sources (else null)."""
    path = os.path.join(ROOT, "profiles", "decode_mma_gqa32k_traffic.txt")
    try:
        fields = {}
        for ln in open(path):
            if ":" in ln and not ln.startswith("#"):
                k, v = ln.split(":", 1)
                fields[k.strip()] = v.strip()
        if fields.get("decode_sources_sha256_16") != _decode_sources_sha():
            return None
        return int(float(fields[f"traffic_bytes_per_launch_{fmt}"]))
    except Exception:
        return None


def _e2e_c_leg(K: int, W: int, device: int) -> dict:
    """The e2e step driven from plain C (tests/e2e_host.c) through the C ABI
    and the CUDA runtime, in its own process with caches of the same
    geometry: its printed name-value pairs (ms_per_step and the host time
    split), or {"error": why} if it cannot be built or run."""
    import importlib
    kb = importlib.import_module("quantized_kv_cache_append_gb300.build")   # the module, not build()
    src = os.path.join(ROOT, "tests", "e2e_host.c")
    exe = os.path.join(kb.BUILD_DIR, "e2e_host")
    r = subprocess.run([kb._nvcc(), "-O2", "-o", exe, src, "-I", kb.INCLUDE, "-L", kb.BUILD_DIR, "-lkvq",
                        "-Xlinker", f"-rpath,{kb.BUILD_DIR}"], capture_output=True, text=True)
    if r.returncode != 0:
        return {"error": "build: " + (r.stderr or r.stdout).strip()[-200:]}
    try:
        r = subprocess.run([exe, str(K), str(W), str(LAYERS), str(device)], capture_output=True,
                           text=True, timeout=900)
    except subprocess.TimeoutExpired:
        return {"error": "timed out"}
    if r.returncode != 0:
        return {"error": (r.stderr or r.stdout).strip()[-200:]}
    f = r.stdout.split()
    return {k: round(float(v), 4) for k, v in zip(f[::2], f[1::2])}


def _e2e(step_fn, torch, layers, wl, bt, cap, L, n_kv, hd, K, W, world, dist):
    """Per step: one pinned host -> device copy of the step's inputs (the new
    cell's K and V, the query, its position and the context length, packed
    back to back in one staging buffer), append + decode on both formats
    through the public calls, one device -> host copy of both outputs,
    synchronize."""
    n_q = wl.n_q
    segs = [("k", np.float32), ("v", np.float32), ("q", np.float32),
            ("tok_pos", np.int32), ("ctx_lens", np.int32)]
    offs, words = {}, 0
    for name, _ in segs:   # each input starts on a 256-byte boundary
        n = int(np.asarray(wl.steps[0][name]).size)
        offs[name] = (words, n)
        words += -(-n // 64) * 64
    pack = np.zeros((STEPS_PER_LAYER, words), np.float32)
    for j, st in enumerate(wl.steps[:STEPS_PER_LAYER]):
        for name, dt in segs:
            o, n = offs[name]
            pack[j, o:o + n] = np.ascontiguousarray(st[name], dt).reshape(-1).view(np.float32)
    hin = torch.from_numpy(pack).pin_memory()
    din = torch.empty(words, dtype=torch.float32, device="cuda")

    def view(name, dtype, shape):
        o, n = offs[name]
        t = din[o:o + n]
        return (t.view(torch.int32) if dtype is np.int32 else t).view(shape)

    st0 = wl.steps[0]
    dk = view("k", np.float32, st0["k"].shape)
    dv = view("v", np.float32, st0["v"].shape)
    dq = view("q", np.float32, st0["q"].shape)
    dpos = view("tok_pos", np.int32, st0["tok_pos"].shape)
    dctx = view("ctx_lens", np.int32, st0["ctx_lens"].shape)
    dout = torch.empty((2,) + tuple(st0["q"].shape), dtype=torch.float32, device="cuda")
    hout = torch.empty_like(dout, device="cpu").pin_memory()
    seq0 = torch.zeros(1, dtype=torch.int32, device="cuda")
    h2d = words * 4
    d2h = hout.numel() * 4

    douts = (dout[0], dout[1])   # the two formats' output views, made once
    hins = [hin[j] for j in range(STEPS_PER_LAYER)]

    def one(s):
        j = (s // LAYERS) % STEPS_PER_LAYER
        din.copy_(hins[j], non_blocking=True)
        for i, name in enumerate(("f16", "q8")):
            pool, ws, _ = layers[s % LAYERS][name]
            pool.append(dk, dv, seq0, dpos, bt)
            pool.decode(dq, dctx, cap, bt, wl.sm_scale, out=douts[i], workspace=ws)
        hout.copy_(dout, non_blocking=True)
        torch.cuda.current_stream().synchronize()

    for s in range(W):
        one(s)
    if world > 1:
        dist.barrier()
    t0 = time.perf_counter()
    total = 0
    for s in range(K):
        one(s)
        ctx = _step_ctx(s, L)
        total += ctx * n_kv * (_row_bytes(False, hd) + _row_bytes(True, hd))
    dt = time.perf_counter() - t0
    dt = _max_over_ranks(dt, dist, world, "cuda")
    return {"value": round(total * world / dt / 1e9, 2), "unit": "GB/s", "steps": K,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": round(dt / K * 1e3, 4)}


# --------------------------------------------------------------------------
# the reference arm: the CPU oracle on the same workload
# --------------------------------------------------------------------------

def _oracle_steps(n_steps: int, budget_s: float = None, lib_path: str = None):
    """Prefill both oracle caches, then run oracle steps (append one cell +
    float64 decode, FP16 and int8).  Returns (bytes, seconds, steps).
    lib_path: another build of the oracle (its OpenMP build) to time."""
    import contextlib

    import oracle
    import workloads

    wl = workloads.make("gqa32k")
    L, n_kv, hd = int(wl.ctx_lens[0]), wl.n_kv, wl.head_dim
    imgs = {}
    for name, fmt in (("f16", oracle.FMT_F16), ("q8", oracle.FMT_Q8)):
        img = oracle.PoolImage(fmt, n_kv, hd, wl.block_size, wl.n_blocks)
        oracle.append(img, wl.k, wl.v, wl.tok_seq, wl.tok_pos, wl.block_table)
        imgs[name] = img
    ctx = oracle.use_library(lib_path) if lib_path else contextlib.nullcontext()
    with ctx:
        t0 = time.perf_counter()
        total = 0
        done = 0
        for s in range(n_steps):
            j = s % STEPS_PER_LAYER
            st = wl.steps[j]
            for name in ("f16", "q8"):
                oracle.append(imgs[name], st["k"], st["v"], st["tok_seq"], st["tok_pos"],
                              wl.block_table)
                oracle.attention(imgs[name], st["q"], st["ctx_lens"], wl.block_table,
                                 wl.sm_scale)
            total += int(st["ctx_lens"][0]) * n_kv * (_row_bytes(False, hd) + _row_bytes(True, hd))
            done += 1
            if budget_s is not None and time.perf_counter() - t0 > budget_s:
                break
        return total, time.perf_counter() - t0, done


def _host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def _parallel_oracle():
    """(path, threads) of the oracle's OpenMP build on every host core, or
    (None, 1) when it cannot be built."""
    import oracle

    cores = _host_cores()
    path = oracle.parallel_library(cores)
    return (path, cores) if path is not None else (None, 1)


def cpu_baseline(budget_s: float = 10.0):
    """The oracle on the host cores: single-threaded, and its OpenMP build
    over the (sequence, token, head) rows on every core.  The line's value is
    the multi-core leg (the single-threaded one when OpenMP is missing)."""
    legs = []
    total, dt, done = _oracle_steps(10_000, budget_s)
    legs.append({"value": round(total / dt / 1e9, 4), "unit": "GB/s", "cores": 1,
                 "steps": done})
    path, cores = _parallel_oracle()
    if path is not None:
        total, dt, done = _oracle_steps(10_000, budget_s, lib_path=path)
        legs.append({"value": round(total / dt / 1e9, 4), "unit": "GB/s", "cores": cores,
                     "steps": done})
    top = legs[-1]
    return {"value": top["value"], "unit": "GB/s", "cores": top["cores"], "kind": "oracle",
            "sample": f"{top['steps']} steps of the same workload (append 1 cell + float64 "
                      f"decode over 32769+ cells, FP16 and int8), C oracle on "
                      f"{top['cores']} host core(s)",
            "legs": legs}


def run_reference(args):
    rank, world, _ = _dist()
    if rank != 0:
        return None
    for _ in range(args.warmup):
        pass  # the oracle has no warm-up state; its prefill is untimed
    path, cores = _parallel_oracle()
    total, dt, done = _oracle_steps(args.steps, lib_path=path)
    value = total / dt / 1e9
    return {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
            "n_gpus": world, "steps": done, "warmup": args.warmup,
            "ms_per_step": dt / done * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded N(0,1))",
            "config": _config(world),
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores,
                             "kind": "oracle",
                             "sample": f"{done} steps, C oracle on {cores} host core(s)"},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def run_profile_case(args):
    """A few launches of each kernel on one layer of the workload, for ncu
    (small device footprint, no graphs, no timing)."""
    import torch

    import quantized_kv_cache_append_gb300 as kvq
    import workloads
    from quantized_kv_cache_append_gb300.pool import PagedPool

    kvq.build()
    kvq.load_library()
    chunk_cases = {"chunk": (8, 32, 128), "chunk64": (4, 16, 64), "chunk256": (2, 16, 256)}
    if args.profile_workload in chunk_cases:
        # prompt-chunk attention: a 4096-token chunk over 32768 cells of fp16
        # staging; 32/8 heads at head_dim 128 (134 MB of staging, above L2),
        # 16/4 at 64, 16/2 at 256 (the bench's other head dims)
        n_kv, n_q, hd = chunk_cases[args.profile_workload]
        P, T = 32768, 4096
        g = torch.Generator(device="cuda").manual_seed(1005)
        k16 = torch.randn(n_kv, P, hd, device="cuda", generator=g).half()
        v16 = torch.randn(n_kv, P, hd, device="cuda", generator=g).half()
        q = torch.randn(T, n_q, hd, device="cuda", generator=g)
        out = torch.empty_like(q)
        for _ in range(args.profile_reps):
            st = kvq.kvq_chunk_attn(k16, v16, n_kv, P, hd, q, T, n_q, float(1 / np.sqrt(hd)), out)
            assert st == kvq.KVQ_OK, kvq.kvq_status_string(st)
        torch.cuda.synchronize()
        print(json.dumps({"profile_case": args.profile_workload, "reps": args.profile_reps}))
        return
    if args.profile_workload == "stream":
        # block streaming: one gqa32k int8 layer (128 blocks, 70 MB) in a
        # pinned host copy, fetched whole into an empty device window
        from quantized_kv_cache_append_gb300.pool import PagedPool
        wl = workloads.make("gqa32k")
        dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
        host = PagedPool(kvq.KVQ_Q8, wl.n_kv, wl.head_dim, wl.block_size, wl.n_blocks, pinned=True)
        win = PagedPool(kvq.KVQ_Q8, wl.n_kv, wl.head_dim, wl.block_size, wl.n_blocks)
        host.append(dev(wl.k), dev(wl.v), dev(wl.tok_seq), dev(wl.tok_pos), dev(wl.block_table))
        ids = torch.arange(wl.n_blocks, dtype=torch.int32, device="cuda")
        for _ in range(args.profile_reps):
            st = kvq.kvq_stream_fetch(host.cache, win.cache, ids, ids, wl.n_blocks)
            assert st == kvq.KVQ_OK, kvq.kvq_status_string(st)
        torch.cuda.synchronize()
        print(json.dumps({"profile_case": "stream", "reps": args.profile_reps}))
        return
    wl = workloads.make(args.profile_workload)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    bt = dev(wl.block_table)
    L = int(wl.ctx_lens[0])
    k, v, seq, pos = dev(wl.k), dev(wl.v), dev(wl.tok_seq), dev(wl.tok_pos)
    q, ctx = dev(wl.q), dev(wl.ctx_lens)
    formats = args.profile_formats.split(",") if args.profile_formats else wl.formats
    for name, fmt in (("f16", kvq.KVQ_F16), ("q8", kvq.KVQ_Q8), ("k8v4", kvq.KVQ_K8V4)):
        if name not in formats:
            continue
        pool = PagedPool(fmt, wl.n_kv, wl.head_dim, wl.block_size, wl.n_blocks)
        for _ in range(args.profile_reps):
            pool.append(k, v, seq, pos, bt)
        for _ in range(args.profile_reps):
            pool.decode(q, ctx, int(wl.ctx_lens.max()), bt, wl.sm_scale)
        for _ in range(args.profile_reps):
            pool.compact(bt[0], L)
        torch.cuda.synchronize()
    print(json.dumps({"profile_case": args.profile_workload, "reps": args.profile_reps}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--profile-case", action="store_true",
                    help="run a few launches of every kernel on one layer (for ncu)")
    ap.add_argument("--profile-workload", default="gqa32k")
    ap.add_argument("--profile-reps", type=int, default=3)
    ap.add_argument("--profile-formats", default="",
                    help="comma-separated cache formats for --profile-case (f16, q8, k8v4)")
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=8192)
    ap.add_argument("--warmup", type=int, default=512)
    ap.add_argument("--impl", choices=["kvq", "reference"], default="kvq")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.profile_case:
        run_profile_case(args)
        return
    if args.impl == "reference":
        res = run_reference(args)
    else:
        res = run_kvq(args)
        rank, world, _ = _dist()
        if res is not None and world == 1 and not args.no_cpu_baseline:
            res["cpu_baseline"] = cpu_baseline()
    if res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
