"""Benchmark of the QSA decode step on one GB300.

Workload (default): 8 requests x 12 QSA layers x 262144 cached tokens; full
KV history in pinned host memory with a 4096-token HBM tail ring per request
and layer; half of the selected blocks in the ring.  One step = one decode
step of every request through all 12 layers, layer after layer (as a model
would run them): per layer one index-score + C4-max launch, one top-k launch
and one attention launch (split-K + merge) over the 8 requests.

Metric: QSA layer-steps per second (96 per step).  Printed as one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the fp64 CPU oracle on the host cores on a bounded
sample of the same workload.  Under torchrun (N > 1) every rank runs its own
replica on its own GPU (no collective on the data path); the time is the
maximum over ranks.
"""
from __future__ import annotations

import argparse
import contextlib
import gc
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "QSA decode layer-steps/sec at 256K ctx; achieved HBM & PCIe GB/s vs peak"
WORKLOAD = "c256k_x8"
N_LAYERS, N_REQ, CTX, BUDGET, RING = 12, 8, 262144, 2048, 4096
ROW = 2048
ROW_FP8 = 1040
IDX_BYTES = 66


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def measured_traffic(kind):
    """DRAM bytes per launch of a kernel from the committed ncu capture, or
    None when the kernel's source has changed since the capture."""
    import hashlib
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    rec = json.load(open(p))["kernels"].get(kind)
    if not rec:
        return None
    src = os.path.join(ROOT, rec["source"])
    if not os.path.exists(src) or hashlib.sha256(open(src, "rb").read()).hexdigest() != rec["sha256"]:
        return None
    return rec["dram_read_bytes"] + rec["dram_write_bytes"]


def config_block():
    return {"workload": WORKLOAD, "requests": N_REQ, "qsa_layers": N_LAYERS, "ctx_tokens": CTX,
            "indexer_budget": BUDGET, "ring_tokens": RING, "kv_placement": "pinned host + HBM tail ring",
            "layer_order": "sequential", "l2": "inputs larger than L2 (1.66 GB index keys per step)"}


@contextlib.contextmanager
def quiet_host():
    """No Python garbage collection inside a timed region.  On this Grace machine
    the GPU reads the registered host histories through the CPU's page
    tables (ATS): a host munmap anywhere in the process (the collector or an
    allocator returning memory) invalidates the GPU's translations of those
    pages, and the next step pays ~4 ms to take them again (measured: a 64 MiB
    allocate-and-free between replays put a 5 ms step after each).  The
    harness should not add that to the workload's steps."""
    was = gc.isenabled()
    gc.disable()
    try:
        yield
    finally:
        if was:
            gc.enable()


class Clocks:
    """Sample SM clocks and throttle reasons with nvidia-smi during a region.
    busy(), if given, keeps the GPU at work while the sampler starts (it
    replays the measured step): the samples are then taken under load, and
    the step's host-page translations are warm again when the timed region
    begins (an idle GPU lets them go stale: measured, a 1 s pause left 9-15
    of the next 40 steps 0.5-2 ms slower)."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index, busy=None, dev=None):
        self.index = index
        self.busy = busy
        self.dev = dev
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        t_end = time.monotonic() + 0.3
        if self.busy is None:
            time.sleep(0.3)
        while self.busy is not None and time.monotonic() < t_end:
            for _ in range(8):
                self.busy()
            torch.cuda.synchronize(self.dev)
        return self

    def __exit__(self, *a):
        self.summary = {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        if not self.proc:
            return
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 7:
                continue
            try:
                sm.append(float(f[0]))
                mx.append(float(f[1]))
            except ValueError:
                continue
            for nm, v in zip(names, f[3:7]):
                if v.lower() == "active":
                    reasons.add(nm)
        if sm:
            self.summary = {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                            "reasons": sorted(reasons), "samples": len(sm)}


def host_link_peak(dev):
    """Best pinned host->device copy rate (GB/s) over a 1 GiB buffer."""
    n = 1 << 30
    h = torch.empty(n, dtype=torch.uint8, pin_memory=True)
    d = torch.empty(n, dtype=torch.uint8, device=dev)
    best = 0.0
    for _ in range(5):
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        d.copy_(h, non_blocking=True)
        e.record()
        e.synchronize()
        best = max(best, n / (s.elapsed_time(e) * 1e-3) / 1e9)
    del h, d
    return best


def zero_copy_peak(dev, n_req=8, n=262144, budget=8192):
    """Host->device read rate (GB/s) of the library's gather kernel when every
    selected row is cold: 8 requests x 8192 rows of 2 KiB spread over a
    262144-token pinned history each (128 MiB per launch)."""
    import sparse_attention_decode_qsa_gb300 as Q
    from sparse_attention_decode_qsa_gb300 import workloads
    c = Q.Cache(n_layers=1, max_requests=n_req, ctx_capacity=n, hbm_pool_rows=8,
                budget_tokens=budget, staging_rows=0, device=dev)
    host = [workloads.register_pinned(torch.zeros(1, n, ROW, dtype=torch.uint8))
            for _ in range(n_req)]
    try:
        hs = [c.request_begin(n, Q.KV_HOST, host_rows=h) for h in host]
        kb = budget // 4
        sel = (torch.arange(kb, dtype=torch.int32, device=dev) * (n // 4 // kb)).repeat(n_req, 1)
        nsel = torch.full((n_req,), kb, dtype=torch.int32, device=dev)
        out = torch.empty(n_req, budget, ROW, dtype=torch.uint8, device=dev)
        best = 0.0
        for it in range(8):
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record()
            c.gather_rows(hs, 0, 1, sel.contiguous(), nsel, budget, out)
            e.record()
            e.synchronize()
            if it >= 2:
                best = max(best, n_req * budget * ROW / (s.elapsed_time(e) * 1e-3) / 1e9)
        return best
    finally:
        c.close()
        for h in host:
            workloads.unregister_pinned(h)


def max_over_ranks(times, world):
    """Each timing's maximum over the ranks (replicas on their own GPUs; the
    slowest rank sets the job's time).  Host tensors, so it runs on any
    process group backend."""
    if world <= 1:
        return list(times)
    t = torch.tensor(list(times), dtype=torch.float64)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return [float(x) for x in t]


def whole_job_rate(units_per_rank, world, step_s):
    """Layer-steps per second of the whole job: every rank's units of a step
    over the slowest rank's step time (weak scaling: each rank owns its
    requests, no data is exchanged)."""
    return units_per_rank * world / step_s


def append_timing(dev, n_req=8, n_layers=12, steps=20):
    """Per-launch time of qsa_append_token for n_req units (one layer), on a
    cache of its own (8 HBM-resident requests of 4096 tokens with room to
    grow): one position reserved per request, then the 12 layers' appends
    captured once as a CUDA graph and replayed (each replay rewrites the same
    position)."""
    import sparse_attention_decode_qsa_gb300 as Q
    from sparse_attention_decode_qsa_gb300 import synth
    n = 4096
    c = Q.Cache(n_layers=n_layers, max_requests=n_req, ctx_capacity=n + 8,
                hbm_pool_rows=n_layers * n_req * (n + 8), budget_tokens=BUDGET,
                staging_rows=0, device=dev)
    try:
        hs = [c.request_begin(n, Q.KV_HBM, max_ctx=n + 8) for _ in range(n_req)]
        for h in hs:
            c.advance(h)
        g_ = torch.Generator(device="cpu").manual_seed(5)
        k = torch.randn(n_layers, n_req, 64, generator=g_).to(dev)
        rows = synth.kv_rows(n_layers * n_req, 6).view(n_layers, n_req, ROW).to(dev)
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        for l in range(n_layers):
            c.append_token(hs, l, 1, k[l], rows[l], s)
        torch.cuda.synchronize(dev)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for l in range(n_layers):
                c.append_token(hs, l, 1, k[l], rows[l], s)
        g.replay()
        torch.cuda.synchronize(dev)
        cur = torch.cuda.current_stream(dev)          # graph replays launch on it
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(cur)
        for _ in range(steps):
            g.replay()
        e1.record(cur)
        torch.cuda.synchronize(dev)
        st, det = c.poll_error()
        if st != 0:
            raise RuntimeError(f"device error word {st} ({det}) in the append timing")
        return e0.elapsed_time(e1) * 1e3 / (steps * n_layers)
    finally:
        c.close()


def fp8_timing(dev, args):
    """The FP8 KV variant (QSA_KV_FP8, 1040-byte rows) on the benchmark
    workload: 8 requests x 12 layers x 262144 tokens, host history +
    4096-token tail ring, half of the selected rows cold.  Returns the
    captured two-micro-batch step's time (ms, mean of args.steps replays
    after args.warmup) and the attention launch's time (us, 12 launches at
    one layer captured as a CUDA graph)."""
    import sparse_attention_decode_qsa_gb300 as Q
    from sparse_attention_decode_qsa_gb300 import workloads
    wl = workloads.c256k_x8(device=dev, n_layers=args.layers, n_req=args.requests, kv_format=Q.KV_FP8)
    try:
        cur = torch.cuda.current_stream(dev)
        graph = wl.capture(args.groups)
        for _ in range(args.warmup):
            graph.replay()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(cur)
        for _ in range(args.steps):
            graph.replay()
        e1.record(cur)
        torch.cuda.synchronize(dev)
        step_ms = e0.elapsed_time(e1) / args.steps
        del graph
        c, hs, R = wl.cache, wl.handles, wl.n_req
        s = torch.cuda.Stream()
        s.wait_stream(cur)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for _ in range(N_LAYERS):
                c.sparse_decode_attn(hs, 0, 1, wl.q[:R], wl.sel[:R], wl.nsel[:R], BUDGET, None,
                                     wl.softmax_scale, wl.out[:R], wl.lse[:R], s)
        g.replay()
        torch.cuda.synchronize(dev)
        e0.record(cur)
        for _ in range(args.steps):
            g.replay()
        e1.record(cur)
        torch.cuda.synchronize(dev)
        attn_us = e0.elapsed_time(e1) * 1e3 / (args.steps * N_LAYERS)
        st, det = c.poll_error()
        return step_ms, attn_us, ({"status": st, "detail": det} if st else None)
    finally:
        wl.close()


def hbm_resident_timing(dev, args):
    """The HBM-resident configuration: 1 request x 12 layers x 131072 tokens,
    every KV row in HBM.  Times (CUDA events, captured graphs) the faithful
    layer-sequential step (12 dependent layers of one request) and the upper
    bound with the 12 layers batched into one call per kernel, each step by
    its own events after warm-up (mean, p10, median, p90), then each kernel
    over the 12 units and over one unit (the launches of the
    layer-sequential chain), averaged over repeated launches."""
    from sparse_attention_decode_qsa_gb300 import workloads
    wl = workloads.c128k(device=dev)
    try:
        c, hs, L = wl.cache, wl.handles, wl.n_layers
        cur = torch.cuda.current_stream(dev)
        wl.step(cur)
        torch.cuda.synchronize(dev)

        def gtime(fn, reps):
            s = torch.cuda.Stream()
            s.wait_stream(cur)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                for _ in range(reps):
                    fn(s)
            g.replay()
            torch.cuda.synchronize(dev)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(cur)
            for _ in range(args.steps):
                g.replay()
            e1.record(cur)
            torch.cuda.synchronize(dev)
            return e0.elapsed_time(e1) * 1e3 / (args.steps * reps)

        def seq(s):
            for l in range(L):
                wl.step_layer(l, s)

        def score(s):
            c.index_score(hs, 0, L, wl.q_idx, wl.w, wl.blk, s)

        def topk(s):
            c.select_c4_topk(hs, 0, L, wl.blk, BUDGET, wl.sel, wl.nsel, s)

        def attn(s):
            c.sparse_decode_attn(hs, 0, L, wl.q, wl.sel, wl.nsel, BUDGET, None, wl.softmax_scale,
                                 wl.out, wl.lse, s)

        def batched(s):
            score(s)
            topk(s)
            attn(s)

        # one unit (layer 0 of the request), the launches of the sequential chain
        def score1(s):
            c.index_score(hs, 0, 1, wl.q_idx[:1], wl.w[:1], wl.blk[:1], s)

        def topk1(s):
            c.select_c4_topk(hs, 0, 1, wl.blk[:1], BUDGET, wl.sel[:1], wl.nsel[:1], s)

        def attn1(s):
            c.sparse_decode_attn(hs, 0, 1, wl.q[:1], wl.sel[:1], wl.nsel[:1], BUDGET, None,
                                 wl.softmax_scale, wl.out[:1], wl.lse[:1], s)

        def capture(fn):
            s = torch.cuda.Stream()
            s.wait_stream(cur)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                fn(s)
            g.replay()
            torch.cuda.synchronize(dev)
            return g

        # the two steps: per-step CUDA events after warm-up (median, p10, p90)
        steps_ms = {k: _replay_ms(capture(f), dev, args) for k, f in [("seq", seq), ("batched", batched)]}
        t = {k: 1e3 * sum(v) / len(v) for k, v in steps_ms.items()}
        pcts = {k: [round(1e3 * _pct(v, q), 2) for q in (0.1, 0.5, 0.9)] for k, v in steps_ms.items()}
        t.update({k: gtime(f, r) for k, f, r in [("score", score, 10), ("topk", topk, 10), ("attn", attn, 10),
                                                  ("score1", score1, 10), ("topk1", topk1, 10),
                                                  ("attn1", attn1, 10)]})
        st, det = c.poll_error()
        if st != 0:
            raise RuntimeError(f"device error word {st} ({det}) in the HBM-resident timing")
        n = wl.ctxs[0]
        key_b, row_b = L * IDX_BYTES * n, L * BUDGET * ROW
        hbm_peak, _ = peaks()
        gbs = lambda b, us: round(b / (us * 1e-6) / 1e9, 1)
        return {"workload": f"c128k: 1 request x {L} layers x {n} tokens, KV in HBM",
                "algorithmic_bytes_per_step": key_b + row_b,
                "layer_sequential": {"us_per_step": round(t["seq"], 2),
                                     "step_us_p10_p50_p90": pcts["seq"],
                                     "layer_steps_per_s": round(L / (t["seq"] * 1e-6), 1),
                                     "hbm_gbs": gbs(key_b + row_b, t["seq"]),
                                     "frac": round(gbs(key_b + row_b, t["seq"]) / hbm_peak, 4)},
                "layers_batched_upper_bound": {"us_per_step": round(t["batched"], 2),
                                               "step_us_p10_p50_p90": pcts["batched"],
                                               "hbm_gbs": gbs(key_b + row_b, t["batched"]),
                                               "frac": round(gbs(key_b + row_b, t["batched"]) / hbm_peak, 4)},
                "kernels_12_units": {
                    "index_score": {"us": round(t["score"], 2), "hbm_gbs": gbs(key_b, t["score"]),
                                    "frac": round(gbs(key_b, t["score"]) / hbm_peak, 4)},
                    "select_topk": {"us": round(t["topk"], 2)},
                    "sparse_attn": {"us": round(t["attn"], 2), "hbm_gbs": gbs(row_b, t["attn"]),
                                    "frac": round(gbs(row_b, t["attn"]) / hbm_peak, 4)}},
                "kernels_1_unit": {"index_score_us": round(t["score1"], 2),
                                   "select_topk_us": round(t["topk1"], 2),
                                   "sparse_attn_us": round(t["attn1"], 2)}}
    finally:
        wl.close()


def _replay_ms(graph, dev, args, settle_s=0.3):
    """Per-replay times (ms) of a captured step: untimed replays for settle_s
    seconds (the step's host-page translations are taken again after the
    workload's set-up), args.warmup untimed replays, then args.steps replays
    with a CUDA event after each on the launching stream."""
    cur = torch.cuda.current_stream(dev)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    with quiet_host():
        t_end = time.monotonic() + settle_s
        while time.monotonic() < t_end:
            for _ in range(8):
                graph.replay()
            torch.cuda.synchronize(dev)
        for _ in range(args.warmup):
            graph.replay()
        torch.cuda.synchronize(dev)
        ev[0].record(cur)
        for i in range(args.steps):
            graph.replay()
            ev[i + 1].record(cur)
        torch.cuda.synchronize(dev)
    return [ev[i].elapsed_time(ev[i + 1]) for i in range(args.steps)]


def _attn_launch_us(wl, dev, args, r0=0, r1=None):
    """Average time (us) of one attention launch over requests r0..r1-1 at
    layer 0: 12 launches captured as one CUDA graph, replayed args.steps
    times between CUDA events."""
    cur = torch.cuda.current_stream(dev)
    c, R = wl.cache, wl.n_req
    r1 = R if r1 is None else r1
    hs = wl.handles[r0:r1]
    s = torch.cuda.Stream()
    s.wait_stream(cur)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for _ in range(N_LAYERS):
            c.sparse_decode_attn(hs, 0, 1, wl.q[r0:r1], wl.sel[r0:r1], wl.nsel[r0:r1], BUDGET, None,
                                 wl.softmax_scale, wl.out[r0:r1], wl.lse[r0:r1], s)
    g.replay()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(cur)
    for _ in range(args.steps):
        g.replay()
    e1.record(cur)
    torch.cuda.synchronize(dev)
    return e0.elapsed_time(e1) * 1e3 / (args.steps * N_LAYERS)


def _pct(xs, q):
    xs = sorted(xs)
    return xs[min(len(xs) - 1, int(round(q * (len(xs) - 1))))]


def host_only_timing(dev, args, link_peak):
    """The host-only configuration: 4 requests x 12 layers x 1048576 tokens,
    KV only in pinned host memory (every selected row crosses the host link:
    2048 rows x 2 KiB per unit, 48 MiB per step of the 12 layers of one
    request), index keys (66 B per token, 3.32 GB per step) in HBM.  Times
    the captured two-micro-batch step and one attention launch (4 units)."""
    from sparse_attention_decode_qsa_gb300 import workloads
    wl = workloads.c1m_x4(device=dev, n_layers=args.layers)
    try:
        R, L, n = wl.n_req, wl.n_layers, wl.ctxs[0]
        units = R * L
        graph = wl.capture(args.groups)
        ms = _replay_ms(graph, dev, args)
        del graph
        attn_us = _attn_launch_us(wl, dev, args)
        st, det = wl.cache.poll_error()
        step_s = statistics.mean(ms) / 1e3
        host_b, hbm_b = units * BUDGET * ROW, units * IDX_BYTES * n
        attn_host = R * BUDGET * ROW
        hbm_peak, _ = peaks()
        return {"workload": f"c1m_x4: {R} requests x {L} layers x {n} tokens, KV only in pinned host "
                            "memory (sinks 0-3 + recency Zipf(1.1)/uniform planting)",
                "ms_per_step": round(step_s * 1e3, 4),
                "step_ms_p10_p50_p90": [round(_pct(ms, q), 4) for q in (0.1, 0.5, 0.9)],
                "layer_steps_per_s": round(units / step_s, 1),
                "host_bytes_per_step": host_b, "hbm_bytes_per_step": hbm_b,
                "host_gbs": round(host_b / step_s / 1e9, 1),
                "host_frac": round(host_b / step_s / 1e9 / link_peak, 4),
                "hbm_gbs": round(hbm_b / step_s / 1e9, 1),
                "hbm_frac": round(hbm_b / step_s / 1e9 / hbm_peak, 4),
                "roofline_ms": round(max(host_b / (link_peak * 1e9), hbm_b / (hbm_peak * 1e9)) * 1e3, 4),
                "device_error": {"status": st, "detail": det} if st else None,
                "sparse_attn": {"units_per_launch": R, "host_bytes_per_launch": attn_host,
                                "avg_launch_us": round(attn_us, 2),
                                "achieved": round(attn_host / (attn_us * 1e-6) / 1e9, 1),
                                "peak": round(link_peak, 1), "unit": "GB/s",
                                "frac": round(attn_host / (attn_us * 1e-6) / 1e9 / link_peak, 4)}}
    finally:
        wl.close()


def ragged_timing(dev, args, link_peak):
    """The ragged batch: 64 requests with contexts log-uniform in [4096,
    262144] (multiples of 4) x 12 layers; KV in HBM below 32768 tokens, pinned
    host history + HBM tail ring above.  Times the captured step (one batch
    per layer, split into micro-batches); then finishes 16 requests, admits
    16 new ones in their slots under new generations, times the step again,
    ends every request and checks that the cache counters are back at their
    initial values."""
    import sparse_attention_decode_qsa_gb300 as Q
    from sparse_attention_decode_qsa_gb300 import synth, workloads
    L = args.layers
    new_ctx = synth.log_uniform_contexts(16, 4096, 262144, seed=77)
    spare = sum(L * (n if n < 32768 else 4096) for n in new_ctx)
    wl = workloads.ragged(device=dev, n_layers=L, extra_requests=0, spare_rows=spare)
    try:
        c, R = wl.cache, wl.n_req
        units = R * L
        s0 = dict(c.stats())

        def measure():
            g = wl.capture(args.groups)
            ms = _replay_ms(g, dev, args)
            del g
            st, det = c.poll_error()
            ctx = list(wl.ctxs)
            off = [r for r in range(R) if wl.placements[r] != Q.KV_HBM]
            host_rows = sum(L * BUDGET // 2 for r in off)      # half of an offloaded unit's rows are cold
            hbm_b = sum(L * (IDX_BYTES * n + (BUDGET * ROW if wl.placements[r] == Q.KV_HBM else BUDGET * ROW // 2))
                        for r, n in enumerate(ctx))
            step_s = statistics.mean(ms) / 1e3
            return {"ms_per_step": round(step_s * 1e3, 4),
                    "step_ms_p10_p50_p90": [round(_pct(ms, q), 4) for q in (0.1, 0.5, 0.9)],
                    "layer_steps_per_s": round(units / step_s, 1),
                    "device_error": {"status": st, "detail": det} if st else None,
                    "requests_hbm": R - len(off), "requests_offloaded": len(off),
                    "tokens_total": sum(ctx),
                    "host_gbs": round(host_rows * ROW / step_s / 1e9, 1),
                    "hbm_gbs": round(hbm_b / step_s / 1e9, 1)}

        before = measure()
        rng = np.random.default_rng(3)
        done = [int(x) for x in rng.choice(R, 16, replace=False)]
        gens = []
        for j, r in enumerate(done):
            n = new_ctx[j]
            h = wl.reissue(r, n, Q.KV_HBM if n < 32768 else Q.KV_HOST_RING, seed=500 + j)
            gens.append(int(h.generation))
        after = measure()
        for h in wl.handles:
            c.request_end(h)
        wl.handles = []
        s_end = dict(c.stats())
        restored = (s_end["active_requests"] == 0 and s_end["free_request_slots"] == s0["free_request_slots"] + R
                    and s_end["hbm_kv_bytes_in_use"] == 0 and s_end["free_ranges"] == 1
                    and s_end["free_hbm_rows"] == s0["hbm_pool_rows"] - s0["staging_rows_total"])
        return {"workload": f"ragged: {R} requests x {L} layers, contexts log-uniform in [4096, 262144]; "
                            "KV in HBM below 32768 tokens, pinned host + 4096-token HBM tail ring above",
                "before_recycling": before, "after_recycling": after,
                "recycled": {"finished": 16, "admitted": 16, "new_generations": sorted(set(gens))},
                "counters_restored": bool(restored), "stats_initial": s0, "stats_end": s_end}
    finally:
        wl.close()


def _cold_selected_rows(wl):
    """Selected tokens of the offloaded units that are cold (slot -1) before
    the next step: the rows that step fetches from host memory.  The
    selection of a unit is its planted set."""
    c = wl.cache
    idx = []
    for l in range(wl.n_layers):
        for r, h in enumerate(wl.handles):
            if wl.placements[r] == 0:
                continue
            b = torch.as_tensor(wl.planted[l][r], dtype=torch.int64)
            t = (b[:, None] * 4 + torch.arange(4)[None, :]).reshape(-1)
            t = t[t < wl.ctxs[r]]
            idx.append(((h.index * wl.n_layers + l) * c.ctx_capacity) + t)
    flat = torch.cat(idx).to(c.slot_table.device)
    return int((c.slot_table.view(-1)[flat] == -1).sum())


def _drift_levels(wl, graph, dev, args, churns, seed):
    """Time the captured step `graph` of wl at each selection-drift level:
    before each step a fraction `churn` of every unit's cold planted blocks
    moves elsewhere (outside the timed region), then one replay is timed
    with CUDA events on the launching stream."""
    from sparse_attention_decode_qsa_gb300 import synth
    stream = torch.cuda.current_stream(dev)
    units = wl.n_req * wl.n_layers
    levels, k = [], 0
    for f in churns:
        for _ in range(args.warmup):
            k += 1
            if f:
                wl.drift(f, synth.mix_seed(seed, k))
            graph.replay()
        torch.cuda.synchronize(dev)
        total_ms, cold = 0.0, 0
        for _ in range(args.steps):
            k += 1
            if f:
                wl.drift(f, synth.mix_seed(seed, k))
            cold += _cold_selected_rows(wl)
            torch.cuda.synchronize(dev)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            graph.replay()
            e1.record(stream)
            torch.cuda.synchronize(dev)
            total_ms += e0.elapsed_time(e1)
        st, det = wl.cache.poll_error()
        step_s = total_ms / 1e3 / args.steps
        lv = {"churn": f, "ms_per_step": round(step_s * 1e3, 4),
              "layer_steps_per_s": round(units / step_s, 1),
              "host_rows_per_step": round(cold / args.steps, 1),
              "host_gbs": round(cold / args.steps * ROW / step_s / 1e9, 1)}
        if st != 0:       # recorded, not raised: a slow host-memory state can run out a bounded wait
            lv["device_error"] = {"status": st, "detail": det}
        levels.append(lv)
    return levels


def drift_timing(dev, args, churns=(0.0, 0.1, 0.25, 1.0)):
    """The benchmark step when the selection drifts between steps (churn =
    fraction of each unit's cold planted blocks moved before each step; 1.0
    makes every cold block new at every step), in four forms:
      - the measured step as it is: cold rows read zero-copy every step from
        the pinned (registered) host history;
      - on host histories in host NUMA memory mapped into the GPU's page
        tables (qsa_host_alloc): zero-copy; and in a cache with BUDGET hot
        rows per request and layer, whose step copies the cold selected rows
        into them first (qsa_hot_cache_fetch), or plans them and lets the
        attention copy them as it reads them (qsa_hot_cache_plan).
    Runs after the other legs: drift on registered pages leaves them slow."""
    from sparse_attention_decode_qsa_gb300 import workloads

    def hot_levels(w, fold, seed):
        hw = workloads.with_hot_rows(w, BUDGET, fold_fill=fold)
        try:
            g = hw.capture(args.groups)
            lv = _drift_levels(hw, g, dev, args, churns, seed)
            del g
        finally:
            hw.close()
        return lv

    wl = workloads.c256k_x8(device=dev, n_layers=args.layers, n_req=args.requests)
    try:
        graph = wl.capture(args.groups)
        zero_copy = _drift_levels(wl, graph, dev, args, churns, 77)
        del graph
    finally:
        wl.close()
    w3 = workloads.c256k_x8(device=dev, n_layers=args.layers, n_req=args.requests, host_memory="vmm")
    try:
        g3 = w3.capture(args.groups)
        vmm_zero_copy = _drift_levels(w3, g3, dev, args, churns, 80)
        del g3
    except Exception:
        w3.close()
        raise
    vmm_fetch = hot_levels(w3, False, 81)           # consumes w3
    w4 = workloads.c256k_x8(device=dev, n_layers=args.layers, n_req=args.requests, host_memory="vmm")
    vmm_plan = hot_levels(w4, True, 82)
    return {"what": "steps whose selection drifts: churn = fraction of each unit's cold planted "
                    "blocks moved before each step; host_rows_per_step = selected rows cold at "
                    "the start of the step",
            "zero_copy": zero_copy,
            "host_numa_memory": {"what": "host histories from qsa_host_alloc (host NUMA pages in "
                                         "the GPU's page tables); the hot cache has BUDGET rows per "
                                         "request and layer",
                                 "hot_rows": BUDGET,
                                 "zero_copy": vmm_zero_copy,
                                 "hot_cache_fetch": vmm_fetch,
                                 "hot_cache_plan_in_attention": vmm_plan}}


def run_ours(args, rank, world):
    from sparse_attention_decode_qsa_gb300 import workloads

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    hbm_peak, peak_kind = peaks()
    wl = workloads.c256k_x8(device=dev, n_layers=args.layers, n_req=args.requests)
    stream = torch.cuda.current_stream(dev)
    R, L = wl.n_req, wl.n_layers
    units = R * L
    kinds = ["index_score", "select_topk", "sparse_attn"]
    # ---- kernel breakdown: for each kernel kind, the 12 layers' launches of
    # one step captured as their own CUDA graph (no host launch gaps), replayed
    # args.steps times between CUDA events on the launching stream
    for _ in range(args.warmup):
        wl.step(stream)
    torch.cuda.synchronize(dev)
    st, det = wl.cache.poll_error()
    if st != 0:
        raise RuntimeError(f"device error word {st} ({det}) after warm-up")
    c, hs = wl.cache, wl.handles
    calls = {
        "index_score": lambda l, sl, s: c.index_score(hs, l, 1, wl.q_idx[sl], wl.w[sl], wl.blk[sl], s),
        "select_topk": lambda l, sl, s: c.select_c4_topk(hs, l, 1, wl.blk[sl], BUDGET, wl.sel[sl],
                                                         wl.nsel[sl], s),
        "sparse_attn": lambda l, sl, s: c.sparse_decode_attn(hs, l, 1, wl.q[sl], wl.sel[sl], wl.nsel[sl],
                                                             BUDGET, None, wl.softmax_scale,
                                                             wl.out[sl], wl.lse[sl], s),
    }
    per_kind, launches = {}, {}
    for kind, fn in calls.items():
        g = torch.cuda.CUDAGraph()
        cs = torch.cuda.Stream()
        cs.wait_stream(stream)
        with torch.cuda.graph(g, stream=cs):
            for l in range(L):
                fn(l, slice(l * R, (l + 1) * R), cs)
        torch.cuda.synchronize(dev)
        g.replay()
        torch.cuda.synchronize(dev)
        k0, k1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        k0.record(stream)
        for _ in range(args.steps):
            g.replay()
        k1.record(stream)
        torch.cuda.synchronize(dev)
        per_kind[kind] = k0.elapsed_time(k1)
        launches[kind] = args.steps * L
        del g
    e0_, e1_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0_.record(stream)
    for _ in range(args.steps):
        wl.step(stream)
    e1_.record(stream)
    torch.cuda.synchronize(dev)
    ms_eager = e0_.elapsed_time(e1_)

    # ---- the measured step: request groups on their own streams, captured
    # once as a CUDA graph and replayed
    graph = wl.capture(args.groups)
    # an event after every replay gives the per-step spread (no extra syncs)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    with quiet_host(), Clocks(dev.index, busy=graph.replay, dev=dev) as clk:
        for _ in range(args.warmup):
            graph.replay()
        torch.cuda.synchronize(dev)
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(dev)
        ev[0].record(stream)
        for i in range(args.steps):
            graph.replay()
            ev[i + 1].record(stream)
        torch.cuda.synchronize(dev)
    ms = ev[0].elapsed_time(ev[-1])
    per_step = sorted(ev[i].elapsed_time(ev[i + 1]) for i in range(args.steps))
    pct = lambda q: per_step[min(len(per_step) - 1, int(round(q * (len(per_step) - 1))))]

    # ---- end to end: per-step queries from pinned host, outputs back to pinned host
    hq_idx = wl.q_idx.cpu().pin_memory()
    hw = wl.w.cpu().pin_memory()
    hq = wl.q.cpu().pin_memory()
    hout = torch.empty_like(wl.out, device="cpu").pin_memory()
    hlse = torch.empty_like(wl.lse, device="cpu").pin_memory()
    h2d = hq_idx.numel() * 4 + hw.numel() * 4 + hq.numel() * 2
    d2h = hout.numel() * 4 + hlse.numel() * 4

    def e2e_step():
        wl.q_idx.copy_(hq_idx, non_blocking=True)
        wl.w.copy_(hw, non_blocking=True)
        wl.q.copy_(hq, non_blocking=True)
        graph.replay()
        hout.copy_(wl.out, non_blocking=True)
        hlse.copy_(wl.lse, non_blocking=True)

    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with quiet_host():
        for _ in range(args.warmup):
            e2e_step()
        torch.cuda.synchronize(dev)
        e0.record(stream)
        for _ in range(args.steps):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize(dev)
    ms_e2e = e0.elapsed_time(e1)
    st, det = wl.cache.poll_error()
    if st != 0:
        raise RuntimeError(f"device error word {st} ({det}) after timing")
    del graph
    wl.close()
    del wl
    all_legs = args.legs == "all"
    append_us = append_timing(dev) if all_legs else None
    fp8_step_ms, fp8_attn_us, fp8_err = fp8_timing(dev, args) if all_legs else (None, None, None)
    hbm_res = hbm_resident_timing(dev, args) if all_legs else None
    link_copy = host_link_peak(dev)
    link_zc = zero_copy_peak(dev)
    link_peak = max(link_copy, link_zc)
    host_only = host_only_timing(dev, args, link_peak) if all_legs else None
    ragged = ragged_timing(dev, args, link_peak) if all_legs else None
    drift = drift_timing(dev, args) if all_legs else None

    ms_max, ms_e2e_max = max_over_ranks([ms, ms_e2e], world)
    if rank != 0:
        return None

    step_s = ms_max / 1e3 / args.steps
    value = whole_job_rate(units, world, step_s)
    idx_b = IDX_BYTES * CTX          # algorithmic bytes per unit: index keys
    rows_b = BUDGET * ROW            # selected rows per unit
    hot_b = rows_b // 2              # half of them from the HBM tail ring
    hbm_step = units * (idx_b + hot_b)
    host_step = units * (rows_b - hot_b)
    avg = {k: per_kind[k] / launches[k] for k in kinds}          # ms per launch (8 units)
    k1_bytes = R * idx_b
    attn_hbm, attn_host = R * hot_b, R * (rows_b - hot_b)
    dominant = max(kinds, key=lambda k: per_kind[k])
    k1_gbs = k1_bytes / (avg["index_score"] * 1e-3) / 1e9
    attn_link_gbs = attn_host / (avg["sparse_attn"] * 1e-3) / 1e9
    roofs = {
        "index_score": {"bound": "hbm", "achieved": round(k1_gbs, 1), "peak": hbm_peak,
                        "unit": "GB/s", "frac": round(k1_gbs / hbm_peak, 4),
                        "traffic": measured_traffic("index_score"),
                        "bytes_per_launch": k1_bytes,
                        "avg_launch_us": round(avg["index_score"] * 1e3, 2)},
        "sparse_attn": {"bound": "host_link", "achieved": round(attn_link_gbs, 1),
                        "peak": round(link_peak, 1), "unit": "GB/s",
                        "frac": round(attn_link_gbs / link_peak, 4),
                        "traffic": measured_traffic("sparse_attn"),
                        "bytes_per_launch": attn_hbm + attn_host,
                        "host_bytes_per_launch": attn_host,
                        "avg_launch_us": round(avg["sparse_attn"] * 1e3, 2)},
        "select_topk": {"bound": "latency", "avg_launch_us": round(avg["select_topk"] * 1e3, 2),
                        "traffic": measured_traffic("select_topk")},
        # producer side: per launch 8 units (one layer) of key quantisation,
        # row store and slot update; not part of the timed decode step
        "append_token": {"bound": "latency", "avg_launch_us": round(append_us, 2),
                         "units_per_launch": 8, "traffic": measured_traffic("append_token")}
        if append_us is not None else None,
        # FP8 KV variant (1040-byte rows) of the same attention launch; not
        # part of the timed decode step, whose rows are BF16 (the whole FP8
        # step is reported under "fp8_kv")
        "sparse_attn_fp8": {"bound": "host_link",
                            "achieved": round(R * (BUDGET // 2) * ROW_FP8 / (fp8_attn_us * 1e-6) / 1e9, 1),
                            "peak": round(link_peak, 1), "unit": "GB/s",
                            "frac": round(R * (BUDGET // 2) * ROW_FP8 / (fp8_attn_us * 1e-6) / 1e9 / link_peak, 4),
                            "host_bytes_per_launch": R * (BUDGET // 2) * ROW_FP8,
                            "traffic": measured_traffic("sparse_attn_fp8"),
                            "avg_launch_us": round(fp8_attn_us, 2)}
        if fp8_attn_us is not None else None,
    }
    dom = dict(roofs[dominant])
    dom["kernel"] = dominant
    cfg = config_block()
    cfg["qsa_layers"], cfg["requests"] = L, R
    cfg["micro_batches"] = args.groups
    cfg["cuda_graph"] = True
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "layer-steps/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(step_s * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "e4m3/bf16->f32",
        "data": "synthetic (seeded; no public dataset)", "config": cfg,
        "impl": "ours",
        "hbm_gbs": round(hbm_step / step_s / 1e9, 1), "hbm_peak_gbs": hbm_peak,
        "hbm_frac": round(hbm_step / step_s / 1e9 / hbm_peak, 4), "peak_kind": peak_kind,
        "host_link_gbs": round(host_step / step_s / 1e9, 1),
        "host_link_peak_gbs": round(link_peak, 1),
        "host_link_peak_parts": {"pinned_h2d_copy_gbs": round(link_copy, 1),
                                 "zero_copy_gather_gbs": round(link_zc, 1)},
        "host_link_frac": round(host_step / step_s / 1e9 / link_peak, 4),
        "eager_sequential_ms_per_step": round(ms_eager / args.steps, 4),
        "step_ms_p10_p50_p90": [round(pct(0.1), 4), round(pct(0.5), 4), round(pct(0.9), 4)],
        "roofline": dom, "kernels": roofs, "selection_drift": drift, "hbm_resident": hbm_res,
        "host_only_1m": host_only, "ragged_batch": ragged,
        "fp8_kv": None if fp8_step_ms is None else {"what": "the same step over FP8 KV rows (1040 bytes: E4M3 K and V codes, fp16 "
                           "scales per head); BF16 queries, fp32 outputs",
                   "ms_per_step": round(fp8_step_ms, 4),
                   "layer_steps_per_s": round(units / (fp8_step_ms / 1e3), 1),
                   "host_gbs": round(units * (BUDGET // 2) * ROW_FP8 / (fp8_step_ms / 1e3) / 1e9, 1),
                   "device_error": fp8_err},
        "gpu_launches": args.steps * L * args.groups * 4,
        "clocks": clk.summary,
        "e2e": {"value": round(units * world / (ms_e2e_max / 1e3 / args.steps), 1),
                "unit": "layer-steps/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
    }
    line["cpu_baseline"] = cpu_baseline(seconds=args.cpu_seconds)
    return line


def _oracle_sample(seconds, budget_units=None, seed_base=1234):
    """Time the fp64 oracle on decode units of the benchmark's workload,
    drawn on the CPU with the same recipe (one unit = one request at one
    layer: 262144 tokens; host rows drawn only for the tokens it selects)."""
    from oracle import qsa_oracle as O
    from sparse_attention_decode_qsa_gb300 import synth

    n = CTX
    done, t_total = 0, 0.0
    while (done == 0 or t_total < seconds) and (budget_units is None or done < budget_units):
        seed = synth.mix_seed(seed_base, done)
        planted = synth.planted_hot_cold(n // 4, 512, RING // 4, synth.mix_seed(seed, 9))
        u = synth.unit_inputs(n, seed, planted, device="cpu")
        codes = u.codes.numpy()
        scales = u.scales.view(torch.int16).numpy().view(np.uint16)
        qb = u.q.view(torch.int16).numpy().view(np.uint16)
        slot = O.ring_slot_row(n, 0, 0, RING)
        rows = synth.kv_rows(BUDGET, synth.mix_seed(seed, 4)).numpy()

        class Rows:   # rows of the selected tokens only (the rest are never read)
            def __init__(self):
                self.m = {}

            def __getitem__(self, t):
                return self.m.setdefault(int(t), rows[len(self.m) % BUDGET])

        host, pool = Rows(), Rows()
        t = time.perf_counter()
        O.layer_step(codes, scales, u.q_idx.numpy(), u.w.numpy(), qb, slot, pool, host, BUDGET,
                     1 / math.sqrt(128))
        t_total += time.perf_counter() - t
        done += 1
    return done, t_total


_ONE_THREAD = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "NUMEXPR_NUM_THREADS")


def _oracle_worker(job):
    seconds, seed_base = job
    return _oracle_sample(seconds, seed_base=seed_base)


def cpu_baseline(seconds=15.0):
    """The oracle on every host core: one spawned process per core, each
    with one math thread, each timing independent decode units for about
    `seconds`; rate = units / the longest worker's compute time.  Falls back
    to one process if the pool cannot run."""
    workers = os.cpu_count() or 1
    sample = (f"decode units (1 request x 1 layer, 262144 tokens each) of the {WORKLOAD} recipe, "
              f"fp64 numpy oracle")
    try:
        pool = _spawn_oracle_pool(workers)
        if pool is None:
            raise RuntimeError("no process pool")
        try:
            res = pool.map_async(_oracle_worker, [(seconds, 1234 + 7919 * i) for i in range(workers)]
                                 ).get(timeout=8 * seconds + 180)
        finally:
            pool.terminate()
        done = sum(d for d, _ in res)
        t = max(tt for _, tt in res)
        return {"value": round(done / t, 3), "unit": "layer-steps/s", "cores": workers, "kind": "oracle",
                "sample": f"{done} {sample}, {workers} processes with one thread each, "
                          f"{t:.1f} s of compute in the longest"}
    except Exception as e:  # noqa: BLE001 - the baseline must not stop the benchmark
        done, t = _oracle_sample(seconds)
        return {"value": round(done / t, 3), "unit": "layer-steps/s", "cores": 1, "kind": "oracle",
                "sample": f"{done} {sample}, one process ({type(e).__name__} from the process pool), "
                          f"{t:.1f} s of CPU work"}


def _oracle_unit_job(seed_base):
    return _oracle_sample(0.0, budget_units=1, seed_base=seed_base)


def _spawn_oracle_pool(workers):
    """A spawned pool of oracle workers with one math thread each, or None."""
    import multiprocessing as mp
    saved = {k: os.environ.get(k) for k in _ONE_THREAD}
    os.environ.update({k: "1" for k in _ONE_THREAD})     # inherited by the spawned workers
    try:
        return mp.get_context("spawn").Pool(workers)
    except Exception:  # noqa: BLE001 - fall back to one process
        return None
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v


def run_reference(args, rank, world):
    """The fp64 oracle as the reference arm: each step is one decode unit of
    the benchmark's workload on every host core (one spawned process with one
    math thread per core); a step's time is the longest worker's oracle time
    (input generation excluded); one process if the pool cannot run."""
    if rank != 0:
        return None
    workers = os.cpu_count() or 1
    pool = _spawn_oracle_pool(workers)

    def step(k):
        if pool is not None:
            try:
                res = pool.map_async(_oracle_unit_job, [1234 + 7919 * (k * workers + i) for i in range(workers)]
                                     ).get(timeout=600)
                return sum(d for d, _ in res), max(t for _, t in res), workers
            except Exception:  # noqa: BLE001 - fall back to one process
                pass
        d, t = _oracle_sample(0.0, budget_units=1, seed_base=1234 + k)
        return d, t, 1

    try:
        for k in range(args.warmup):
            step(k)
        total_units, total_t, cores = 0, 0.0, workers
        for k in range(args.steps):
            d, t, c = step(args.warmup + k)
            total_units += d
            total_t += t
            cores = min(cores, c)
    finally:
        if pool is not None:
            pool.terminate()
    value = total_units / total_t
    sample = (f"{args.steps} timed steps of {total_units // max(1, args.steps)} decode units each "
              f"(1 request x 1 layer, 262144 tokens, one per process) of the {WORKLOAD} recipe; "
              f"fp64 numpy oracle on {cores} processes with one thread each")
    return {
        "metric": METRIC, "value": round(value, 3), "unit": "layer-steps/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * total_t / args.steps, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded; no public dataset)", "config": config_block(),
        "impl": "reference",
        "cpu_baseline": {"value": round(value, 3), "unit": "layer-steps/s",
                         "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 3), "unit": "layer-steps/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


PROFILE_CASES = ("hbm_attn", "step_1layer", "fp8_1layer", "hot_plan_1layer", "c1m_1layer")


def run_profile_case(name, args):
    """One small run of a named case, for ncu captures of single kernels
    (each case's last launches are the ones to capture):
      hbm_attn         1 request x 12 layers x 131072 tokens in HBM: one
                       decode step, then one attention launch over the 12
                       units (HBM rows only)
      step_1layer      8 requests x 1 layer x 262144 tokens, host history +
                       tail ring: warm-up steps, then one step
      fp8_1layer       the same with FP8 KV rows
      hot_plan_1layer  the same requests on host NUMA memory with a 2048-row
                       hot cache planned before attention: warm-up steps,
                       then one step
      c1m_1layer       4 requests x 1 layer x 1048576 tokens, every row in
                       host memory: warm-up steps, then one step"""
    from sparse_attention_decode_qsa_gb300 import workloads
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    if name == "hbm_attn":
        wl = workloads.c128k(device=dev)
        wl.step()
        torch.cuda.synchronize(dev)
        wl.cache.sparse_decode_attn(wl.handles, 0, wl.n_layers, wl.q, wl.sel, wl.nsel, BUDGET, None,
                                    wl.softmax_scale, wl.out, wl.lse)
    else:
        if name == "step_1layer":
            wl = workloads.c256k_x8(device=dev, n_layers=1)
        elif name == "fp8_1layer":
            import sparse_attention_decode_qsa_gb300 as Q
            wl = workloads.c256k_x8(device=dev, n_layers=1, kv_format=Q.KV_FP8)
        elif name == "hot_plan_1layer":
            wl = workloads.with_hot_rows(workloads.c256k_x8(device=dev, n_layers=1, host_memory="vmm"),
                                         BUDGET, fold_fill=True)
        else:
            wl = workloads.c1m_x4(device=dev, n_layers=1)
        for _ in range(args.warmup + 1):
            wl.step()
    torch.cuda.synchronize(dev)
    st, det = wl.cache.poll_error()
    wl.close()
    print(json.dumps({"profile_case": name, "device_error": st, "detail": det}), flush=True)
    if st != 0:
        raise RuntimeError(f"device error word {st} ({det}) in profile case {name}")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--layers", type=int, default=N_LAYERS,
                    help="QSA layers (fewer only for profiling captures)")
    ap.add_argument("--requests", type=int, default=N_REQ)
    ap.add_argument("--groups", type=int, default=2,
                    help="request micro-batches, each on its own stream")
    ap.add_argument("--legs", choices=["all", "headline"], default="all",
                    help="headline: only the measured 256K step (for quick runs and launch lists)")
    ap.add_argument("--profile-case", choices=PROFILE_CASES, default=None,
                    help="run one small named case once (for ncu captures) and exit")
    args = ap.parse_args()
    if args.profile_case:
        run_profile_case(args.profile_case, args)
        return
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1:
        torch.distributed.init_process_group("gloo")
    line = run_reference(args, rank, world) if args.impl == "reference" else run_ours(args, rank, world)
    if line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
