"""Synthetic decode-step workloads on one GPU: a Cache filled with seeded
inputs (index keys, KV rows in HBM and/or pinned host memory, queries), plus
the per-unit output buffers of one decode step.

Recipes (per-layer shapes and distributions as in synth.py):
  tiny      1 layer, 1 request, 8192 tokens, KV in HBM, 512 planted blocks.
  c128k     12 layers, 1 request, 131072 tokens, KV in HBM.
  c256k_x8  12 layers, 8 requests x 262144 tokens; full history in pinned host
            memory plus a 4096-token HBM tail ring per request and layer;
            shared staging 2048 x 12 rows; half of the planted blocks inside
            the tail ring (HBM), half in the cold history (host).
  c1m_x4    12 layers, 4 requests x 1048576 tokens; KV only in pinned host
            memory; planted blocks: sinks 0..3 plus a recency-Zipf(1.1) /
            uniform mixture.
  ragged    64 requests, contexts log-uniform in [4096, 262144] (multiples of
            4); KV in HBM under 32768 tokens, host + tail ring above.
Everything is drawn from seeds; nothing here computes the method.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

from . import _native as N
from . import synth
from .api import Cache, HostMemory

# Host memory for the histories of offloaded requests:
#   "vmm"         qsa_host_alloc: pages on the GPU's host NUMA node, in the
#                 GPU's own page tables (2 MiB entries)
#   "registered"  ordinary pages page-locked with cudaHostRegister
HOST_MEMORY_KINDS = ("vmm", "registered")
DEFAULT_HOST_MEMORY = "registered"


def register_pinned(t: torch.Tensor):
    """Page-lock an existing CPU tensor in place (exact size, mapped for the GPU)."""
    err = torch.cuda.cudart().cudaHostRegister(t.data_ptr(), t.numel() * t.element_size(), 3)
    if int(err) != 0:
        raise RuntimeError(f"cudaHostRegister failed: {err}")
    return t


def unregister_pinned(t: torch.Tensor):
    torch.cuda.cudart().cudaHostUnregister(t.data_ptr())


def alloc_host(shape, device, kind: str = None) -> torch.Tensor:
    """A uint8 CPU tensor of `shape` in host memory the GPU reads directly."""
    kind = kind or DEFAULT_HOST_MEMORY
    if kind not in HOST_MEMORY_KINDS:
        raise ValueError(f"unknown host memory kind {kind}")
    if kind == "registered":
        return register_pinned(torch.empty(tuple(shape), dtype=torch.uint8))
    n = 1
    for x in shape:
        n *= int(x)
    dev = torch.device(device)
    return HostMemory(n, device=dev.index if dev.index is not None else torch.cuda.current_device()).cpu(shape)


def free_host(t: torch.Tensor):
    m = getattr(t, "_qsa_host_memory", None)
    if m is not None:
        m.free()
    else:
        unregister_pinned(t)


def device_view(t: torch.Tensor) -> torch.Tensor:
    """A tensor the GPU's copy kernels can write into: the CUDA view of
    qsa_host_alloc memory, else the pinned CPU tensor itself."""
    m = getattr(t, "_qsa_host_memory", None)
    return m.cuda(t.shape) if m is not None else t


@dataclass
class Workload:
    cache: Cache
    handles: list
    n_layers: int
    ctxs: list
    placements: list
    host: list               # per request: uint8 [L][n][2048] registered pinned, or None
    q_idx: torch.Tensor      # fp32 [L*R][8][64], unit u = l*R + r
    w: torch.Tensor          # fp32 [L*R][8]
    q: torch.Tensor          # bf16 [L*R][16][128]
    planted: list            # [L][R] int64 block ids
    budget: int
    blk: torch.Tensor = None
    sel: torch.Tensor = None
    nsel: torch.Tensor = None
    out: torch.Tensor = None
    lse: torch.Tensor = None
    softmax_scale: float = 1.0 / math.sqrt(128)
    seeds: dict = field(default_factory=dict)
    planting: object = None
    host_memory: str = None
    # with hot rows: plan the hot rows before attention and let the attention
    # copy the misses (qsa_hot_cache_plan), instead of a separate fetch
    fold_fill: bool = False

    @property
    def n_req(self):
        return len(self.handles)

    def unit(self, l, r):
        return l * self.n_req + r

    def layer_slice(self, t: torch.Tensor, l: int):
        return t[l * self.n_req:(l + 1) * self.n_req]

    def reissue(self, r: int, n: int, placement: int, seed: int):
        """Finish request r and admit a new request (new lease, new
        generation) in its place, with freshly drawn inputs."""
        self.cache.request_end(self.handles[r])
        old = self.host[r]
        if old is not None and (placement == N.KV_HBM or old.shape[1] != n):
            free_host(old)
            old = None
        if placement != N.KV_HBM and old is None:
            old = alloc_host((self.n_layers, n, self.cache.row_bytes), self.cache.pool.device,
                             self.host_memory)
        self.host[r] = old
        self.ctxs[r], self.placements[r] = n, placement
        self.handles[r] = self.cache.request_begin(n, placement, host_rows=old)
        _fill_request(self, r, seed, self.planting)
        return self.handles[r]

    def drift(self, frac: float, seed: int):
        """Move a fraction frac of every offloaded unit's cold planted blocks
        (blocks wholly before the tail ring) to other cold blocks, so that
        the next step selects them instead: the selection drift of
        consecutive decode steps."""
        c = self.cache
        for l in range(self.n_layers):
            for r, h in enumerate(self.handles):
                p, n = self.placements[r], self.ctxs[r]
                if p == N.KV_HBM:
                    continue
                hi = (n - c.ring_tokens) // 4 if p == N.KV_HOST_RING else (n + 3) // 4
                if hi <= 0:
                    continue
                dropped, added, now = synth.drift_blocks(self.planted[l][r], 0, hi, frac,
                                                         synth.mix_seed(seed, l, r))
                sc = c.index_scales[h.index, l]
                synth.unplant(sc, dropped, n)
                synth.plant(sc, added, n)
                self.planted[l][r] = now

    def close(self):
        for h in self.host:
            if h is not None:
                free_host(h)
        self.host = []
        self.cache.close()

    # ------------------------------------------------------- one step
    def step_layer(self, l: int, stream=None, gathered=None):
        """Index score, top-k and attention for every request at layer l."""
        c, hs, R = self.cache, self.handles, self.n_req
        sl = slice(l * R, (l + 1) * R)
        c.index_score(hs, l, 1, self.q_idx[sl], self.w[sl], self.blk[sl], stream)
        c.select_c4_topk(hs, l, 1, self.blk[sl], self.budget, self.sel[sl], self.nsel[sl], stream)
        self._hot(hs, l, sl, stream)
        c.sparse_decode_attn(hs, l, 1, self.q[sl], self.sel[sl], self.nsel[sl], self.budget,
                             gathered, self.softmax_scale, self.out[sl], self.lse[sl], stream)

    def _hot(self, hs, l, sl, stream):
        c = self.cache
        if not c.hot_rows:
            return
        if self.fold_fill:
            c.hot_cache_plan(hs, l, 1, self.sel[sl], self.nsel[sl], self.budget, stream)
        else:
            c.hot_cache_fetch(hs, l, 1, self.sel[sl], self.nsel[sl], self.budget, stream)

    def step(self, stream=None):
        for l in range(self.n_layers):
            self.step_layer(l, stream)

    def score_group_layer(self, r0: int, r1: int, l: int, stream):
        """Index score and top-k of requests r0..r1-1 at layer l."""
        c, R = self.cache, self.n_req
        hs = self.handles[r0:r1]
        sl = slice(l * R + r0, l * R + r1)
        c.index_score(hs, l, 1, self.q_idx[sl], self.w[sl], self.blk[sl], stream)
        c.select_c4_topk(hs, l, 1, self.blk[sl], self.budget, self.sel[sl], self.nsel[sl], stream)

    def attn_group_layer(self, r0: int, r1: int, l: int, stream):
        """Attention of requests r0..r1-1 at layer l over their selection."""
        c, R = self.cache, self.n_req
        hs = self.handles[r0:r1]
        sl = slice(l * R + r0, l * R + r1)
        self._hot(hs, l, sl, stream)
        c.sparse_decode_attn(hs, l, 1, self.q[sl], self.sel[sl], self.nsel[sl], self.budget,
                             None, self.softmax_scale, self.out[sl], self.lse[sl], stream)

    def step_pipelined(self, streams, stagger: bool = True):
        """One decode step with the requests split into len(streams) groups
        (micro-batches); streams[g] = (score stream, attention stream) of
        group g.  Each group walks the layers in order: scoring, then its
        attention, then the next layer's scoring.  With stagger, the groups
        also take turns at scoring (group g+1 scores layer l after group g
        has), which puts one group's host-link-bound attention beside another
        group's HBM-bound scoring instead of running all groups in lockstep.
        Forks from and joins back into the current stream."""
        main = torch.cuda.current_stream()
        G = len(streams)
        bounds = [(g * self.n_req // G, (g + 1) * self.n_req // G) for g in range(G)]
        for ss, sa in streams:
            ss.wait_stream(main)
        for l in range(self.n_layers):
            for g, ((r0, r1), (ss, sa)) in enumerate(zip(bounds, streams)):
                if r1 <= r0:
                    continue
                self.score_group_layer(r0, r1, l, ss)
                if stagger and G > 1:
                    streams[(g + 1) % G][0].wait_stream(ss)
                if sa is not ss:
                    sa.wait_stream(ss)
                self.attn_group_layer(r0, r1, l, sa)
                if sa is not ss:
                    ss.wait_stream(sa)   # the next layer of these requests follows it
        for ss, sa in streams:
            main.wait_stream(ss)

    def make_streams(self, n_groups: int, split: bool = True):
        """Per group a scoring stream and a higher-priority attention stream
        (split), so attention CTAs are dispatched ahead of queued scoring
        CTAs; or one stream per group (not split), whose chain of launches
        the library then links by programmatic dependent launch while the
        attention launches still carry the highest priority."""
        if not split:
            return [(s, s) for s in (torch.cuda.Stream() for _ in range(n_groups))]
        try:
            _, hi = torch.cuda.Stream.priority_range()
        except (AttributeError, RuntimeError):
            hi = -1
        return [(torch.cuda.Stream(priority=0), torch.cuda.Stream(priority=hi))
                for _ in range(n_groups)]

    def capture(self, n_groups: int, split: bool = True, stagger: bool = True):
        """Capture step_pipelined into a CUDA graph (after one eager warm-up
        run, which also sets the kernels' launch attributes)."""
        streams = self.make_streams(n_groups, split)
        self.step_pipelined(streams, stagger)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream()
        cap.wait_stream(torch.cuda.current_stream())
        with torch.cuda.graph(g, stream=cap):
            self.step_pipelined(streams, stagger)
        torch.cuda.synchronize()
        self._graph_streams = streams
        return g


def _fill_request(wl: "Workload", r: int, seed: int, planting):
    """Draw and place every layer's inputs of request r (current lease)."""
    cache, h, n, p = wl.cache, wl.handles[r], wl.ctxs[r], wl.placements[r]
    dev = cache.pool.device
    ring = cache.ring_tokens
    info = cache.request_info(h)
    stride = info.max_ctx            # rows per layer of the HBM region / host history
    for l in range(wl.n_layers):
        s = synth.mix_seed(seed, r, l)
        blocks = planting(l, r, n)
        wl.planted[l][r] = torch.as_tensor(blocks, dtype=torch.int64)
        codes, scales = synth.index_keys(n, synth.mix_seed(s, 1), device=dev)
        synth.plant(scales, blocks, n)
        cache.index_keys[h.index, l, :n] = codes
        cache.index_scales[h.index, l, :n] = scales
        qi, wi = synth.index_query(synth.mix_seed(s, 2), device=dev)
        u = wl.unit(l, r)
        wl.q_idx[u], wl.w[u] = qi, wi
        wl.q[u] = synth.attn_query(synth.mix_seed(s, 3), device=dev)
        rows = synth.kv_rows(n, synth.mix_seed(s, 4), device=dev)
        if cache.kv_format == N.KV_FP8:
            rows = synth.fp8_kv_rows(rows)
        if p == N.KV_HBM:
            b0 = info.hbm_row_base + l * stride
            cache.pool[b0:b0 + n] = rows
        else:
            device_view(wl.host[r])[l, :n].copy_(rows)
            if p == N.KV_HOST_RING:
                t = torch.arange(max(0, n - ring), n, device=dev)
                cache.pool[info.hbm_row_base + l * ring + (t % ring)] = rows[t]
        del rows
    torch.cuda.synchronize(dev)


def build(n_layers: int, ctxs, placements, planting, budget: int = 2048, ring: int = 4096,
          staging_rows: int = 2048, seed: int = 0, device="cuda", extra_requests: int = 0,
          spare_rows: int = 0, ctx_capacity: int | None = None, grow: int = 0,
          kv_format: int = N.KV_BF16, hot_rows: int = 0, host_memory: str | None = None) -> Workload:
    """planting(l, r, n) -> block ids to plant for unit (l, r).  grow: tokens
    every request may still append (its max_ctx is ctx + grow).  hot_rows:
    cross-step hot-cache rows per offloaded request and layer (0: none).
    host_memory: kind of the offloaded histories' host memory (see
    HOST_MEMORY_KINDS; None: DEFAULT_HOST_MEMORY)."""
    host_memory = host_memory or DEFAULT_HOST_MEMORY
    ctx_capacity = ctx_capacity or (max(ctxs) + grow)
    dev = torch.device(device)
    R = len(ctxs)
    rows_needed = 0
    for n, p in zip(ctxs, placements):
        rows_needed += n_layers * (n + grow if p == N.KV_HBM else ring if p == N.KV_HOST_RING else 0)
        rows_needed += n_layers * hot_rows if p != N.KV_HBM else 0
    pool_rows = n_layers * staging_rows + rows_needed + spare_rows
    cache = Cache(n_layers=n_layers, max_requests=R + extra_requests, ctx_capacity=ctx_capacity,
                  hbm_pool_rows=pool_rows, budget_tokens=budget, ring_tokens=ring,
                  staging_rows=staging_rows, device=dev, kv_format=kv_format, hot_rows=hot_rows)
    handles, host = [], []
    for r, (n, p) in enumerate(zip(ctxs, placements)):
        hrows = None
        if p != N.KV_HBM:
            hrows = alloc_host((n_layers, n + grow, cache.row_bytes), dev, host_memory)
        host.append(hrows)
        handles.append(cache.request_begin(n, p, host_rows=hrows, max_ctx=n + grow if grow else 0))
    U = n_layers * R
    wl = Workload(cache, handles, n_layers, list(ctxs), list(placements), host,
                  torch.empty(U, 8, 64, dtype=torch.float32, device=dev),
                  torch.empty(U, 8, dtype=torch.float32, device=dev),
                  torch.empty(U, 16, 128, dtype=torch.bfloat16, device=dev),
                  [[None] * R for _ in range(n_layers)], budget)
    wl.planting = planting
    wl.host_memory = host_memory
    for r in range(R):
        _fill_request(wl, r, seed, planting)
    blk_stride = (ctx_capacity + 3) // 4
    wl.blk = torch.empty(U, blk_stride, dtype=torch.float32, device=dev)
    wl.sel = torch.empty(U, budget // 4, dtype=torch.int32, device=dev)
    wl.nsel = torch.empty(U, dtype=torch.int32, device=dev)
    wl.out = torch.empty(U, 16, 128, dtype=torch.float32, device=dev)
    wl.lse = torch.empty(U, 16, dtype=torch.float32, device=dev)
    wl.seeds = dict(seed=seed)
    return wl



def with_hot_rows(wl: Workload, hot_rows: int, fold_fill: bool = False) -> Workload:
    """The same requests and inputs in a new cache whose offloaded requests
    get hot_rows hot rows per layer.  Takes over wl's pinned host histories
    and closes wl's cache (wl is unusable afterwards)."""
    old = wl.cache
    dev = old.pool.device
    n_off = sum(1 for p in wl.placements if p != N.KV_HBM)
    cache = Cache(n_layers=old.n_layers, max_requests=old.max_requests,
                  ctx_capacity=old.ctx_capacity,
                  hbm_pool_rows=old.pool.shape[0] + old.n_layers * hot_rows * n_off,
                  budget_tokens=old.budget_tokens, ring_tokens=old.ring_tokens,
                  staging_rows=old.staging_rows, device=dev, kv_format=old.kv_format,
                  hot_rows=hot_rows)
    handles = []
    for r, h in enumerate(wl.handles):
        info = old.request_info(h)
        nh = cache.request_begin(wl.ctxs[r], wl.placements[r], host_rows=wl.host[r],
                                 max_ctx=int(info.max_ctx))
        ni = cache.request_info(nh)
        cache.index_keys[nh.index] = old.index_keys[h.index]
        cache.index_scales[nh.index] = old.index_scales[h.index]
        rows = info.layer_rows * wl.n_layers
        if rows:
            cache.pool[ni.hbm_row_base:ni.hbm_row_base + rows] = \
                old.pool[info.hbm_row_base:info.hbm_row_base + rows]
        handles.append(nh)
    torch.cuda.synchronize(dev)
    new = Workload(cache, handles, wl.n_layers, list(wl.ctxs), list(wl.placements), wl.host,
                   wl.q_idx, wl.w, wl.q, wl.planted, wl.budget, blk=wl.blk, sel=wl.sel,
                   nsel=wl.nsel, out=wl.out, lse=wl.lse, softmax_scale=wl.softmax_scale,
                   seeds=dict(wl.seeds), planting=wl.planting, host_memory=wl.host_memory,
                   fold_fill=fold_fill)
    wl.host = []
    old.close()
    return new

# ------------------------------------------------------------- recipes

def tiny(device="cuda", seed=0):
    n = 8192
    return build(1, [n], [N.KV_HBM],
                 lambda l, r, n: synth.planted_uniform(n // 4, 512, synth.mix_seed(seed, 90, l, r)),
                 staging_rows=64, seed=seed, device=device)


def c128k(device="cuda", seed=1, n_layers=12):
    n = 131072
    return build(n_layers, [n], [N.KV_HBM],
                 lambda l, r, n: synth.planted_uniform(n // 4, 512, synth.mix_seed(seed, 90, l, r)),
                 staging_rows=64, seed=seed, device=device)


def c256k_x8(device="cuda", seed=2, n_layers=12, n_req=8, n=262144, kv_format=N.KV_BF16,
             host_memory=None):
    return build(n_layers, [n] * n_req, [N.KV_HOST_RING] * n_req,
                 lambda l, r, n: synth.planted_hot_cold(n // 4, 512, 4096 // 4,
                                                        synth.mix_seed(seed, 90, l, r)),
                 seed=seed, device=device, kv_format=kv_format, host_memory=host_memory)


def c1m_x4(device="cuda", seed=3, n_layers=12, n_req=4, n=1048576, host_memory=None):
    return build(n_layers, [n] * n_req, [N.KV_HOST] * n_req,
                 lambda l, r, n: synth.planted_zipf_sinks(n // 4, 512, synth.mix_seed(seed, 90, l, r)),
                 staging_rows=64, seed=seed, device=device, host_memory=host_memory)


def ragged(device="cuda", seed=4, n_layers=12, n_req=64, lo=4096, hi=262144, extra_requests=16,
           spare_rows=0, host_memory=None):
    ctxs = synth.log_uniform_contexts(n_req, lo, hi, synth.mix_seed(seed, 80))
    pl = [N.KV_HBM if n < 32768 else N.KV_HOST_RING for n in ctxs]
    return build(n_layers, ctxs, pl,
                 lambda l, r, n: synth.planted_hot_cold(n // 4, min(512, n // 4), 1024,
                                                        synth.mix_seed(seed, 90, l, r)),
                 seed=seed, device=device, extra_requests=extra_requests, spare_rows=spare_rows,
                 ctx_capacity=hi, host_memory=host_memory)
