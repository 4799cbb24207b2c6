"""CPU tests of the C-ABI library: it loads, exports every entry point that
include/qsa.h declares, and its host-side cache manager (leases, generation
tags, pool row ranges, request recycling) behaves as the pages describe
("双卡RTX4090跑通Qwen3-Next：8并发满血长上下文实测", section
"显存账本：热缓存卸载省下约84%": finished or cancelled requests give back KV
capacity and cache slots, which return to their initial values).

These tests use host-only caches (no device storage), so no GPU is needed.
"""
import ctypes as C
import glob
import os
import random
import re

import pytest

import sparse_attention_decode_qsa_gb300 as Q
from sparse_attention_decode_qsa_gb300 import _native as N
from sparse_attention_decode_qsa_gb300 import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_symbols():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        names |= set(re.findall(r"\b(qsa_\w+)\s*\(", src))
    return names


def test_library_exports_every_declared_symbol():
    L = N.lib()
    declared = _declared_symbols()
    assert len(declared) >= 17
    for name in sorted(declared):
        assert hasattr(L, name), f"{name} declared in include/ but not exported"
        assert name in N.SIGNATURES, f"{name} has no Python binding"
    assert L.qsa_abi_version() == 4


def _host_cache(**kw):
    args = dict(n_layers=12, max_requests=4, ctx_capacity=262144, hbm_pool_rows=200000,
                budget_tokens=2048, ring_tokens=4096, staging_rows=2048, device=None)
    args.update(kw)
    return Q.Cache(**args)


def test_workspace_bytes_and_bad_configs():
    L = N.lib()
    cfg = N.CacheConfig(n_layers=12, max_requests=8, ctx_capacity=262144, budget_tokens=2048,
                        ring_tokens=4096, staging_rows=2048, hbm_pool_rows=1 << 20)
    # error word + 8 req x 12 layers x 64 splits x 2080 floats
    assert L.qsa_workspace_bytes(C.byref(cfg)) == 256 + 8 * 12 * 64 * 2080 * 4 + 8 * 12 * 8
    for field, bad in [("budget_tokens", 6), ("budget_tokens", 0), ("budget_tokens", 16384),
                       ("n_layers", 0), ("ring_tokens", 0), ("ctx_capacity", 0)]:
        c2 = N.CacheConfig.from_buffer_copy(cfg)
        setattr(c2, field, bad)
        assert L.qsa_workspace_bytes(C.byref(c2)) == -1
        h = C.c_void_p()
        assert L.qsa_cache_create(C.byref(c2), C.byref(h)) == N.ERR_INVALID_ARG
    # partial device storage is rejected
    c3 = N.CacheConfig.from_buffer_copy(cfg)
    c3.hbm_pool = 4096
    h = C.c_void_p()
    assert L.qsa_cache_create(C.byref(c3), C.byref(h)) == N.ERR_INVALID_ARG
    assert b"completely" in L.qsa_last_error_string()
    # staging larger than the pool
    c4 = N.CacheConfig.from_buffer_copy(cfg)
    c4.hbm_pool_rows = 100
    assert L.qsa_cache_create(C.byref(c4), C.byref(h)) == N.ERR_CAPACITY


def test_lease_lifecycle_and_generations():
    c = _host_cache()
    s0 = c.stats()
    assert s0["free_request_slots"] == 4 and s0["active_requests"] == 0
    assert s0["staging_rows_total"] == 12 * 2048
    assert s0["free_hbm_rows"] == 200000 - 12 * 2048
    h = c.request_begin(262144, Q.KV_HOST_RING, host_rows=1 << 20)
    assert (h.index, h.generation) == (0, 1)
    info = c.request_info(h)
    assert info.layer_rows == 4096 and info.hbm_row_base == 12 * 2048
    s1 = c.stats()
    assert s1["hbm_kv_bytes_in_use"] == 12 * 4096 * 2048
    c.request_end(h)
    assert c.stats() == s0
    # stale: ended handle, double end, forged generation, index out of range
    for bad in [h, Q.Handle(0, 7), Q.Handle(99, 1)]:
        with pytest.raises(Q.QsaError) as e:
            c.request_end(bad)
        assert e.value.status == Q.ERR_STALE_HANDLE
        with pytest.raises(Q.QsaError) as e:
            c.request_info(bad)
        assert e.value.status == Q.ERR_STALE_HANDLE
    h2 = c.request_begin(1000, Q.KV_HBM)
    assert (h2.index, h2.generation) == (0, 2)      # same slot, new generation
    with pytest.raises(Q.QsaError) as e:
        c.request_info(h)                           # old generation of the same slot
    assert e.value.status == Q.ERR_STALE_HANDLE
    c.request_end(h2)
    assert c.stats() == s0


def test_admission_errors_leave_state_unchanged():
    c = _host_cache(max_requests=2, hbm_pool_rows=12 * 2048 + 12 * 4096 + 10)
    s0 = c.stats()
    cases = [
        (dict(ctx_len=0), Q.ERR_INVALID_ARG),
        (dict(ctx_len=262145), Q.ERR_CAPACITY),
        (dict(ctx_len=100, placement=7), Q.ERR_INVALID_ARG),
        (dict(ctx_len=100, placement=Q.KV_HOST_RING), Q.ERR_INVALID_ARG),     # no host rows
        (dict(ctx_len=100, placement=Q.KV_HBM, host_rows=4096), Q.ERR_INVALID_ARG),
        (dict(ctx_len=100, placement=Q.KV_HOST_RING, host_rows=4097), Q.ERR_INVALID_ARG),  # unaligned
        (dict(ctx_len=5000, placement=Q.KV_HBM), Q.ERR_CAPACITY),             # 60000 rows > pool
    ]
    for kw, status in cases:
        with pytest.raises(Q.QsaError) as e:
            c.request_begin(**kw)
        assert e.value.status == status, kw
        assert c.stats() == s0
    a = c.request_begin(8, Q.KV_HBM)
    b = c.request_begin(8, Q.KV_HBM)
    with pytest.raises(Q.QsaError) as e:
        c.request_begin(8, Q.KV_HBM)
    assert e.value.status == Q.ERR_OUT_OF_SLOTS
    c.request_end(a)
    c.request_end(b)
    assert c.stats() == s0


def test_compute_calls_need_device_storage():
    c = _host_cache()
    h = c.request_begin(100, Q.KV_HBM)
    L = N.lib()
    b = N.Batch(1, 0, 1, 0, C.pointer(N.Handle(h.index, h.generation)))
    st = L.qsa_index_score(c.h, C.byref(b), 16, 16, 16, 100, None)
    assert st == Q.ERR_NO_DEVICE
    st = L.qsa_sparse_decode_attn(c.h, C.byref(b), 16, 16, 16, 2048, None, 0.1, 16, None, None)
    assert st == Q.ERR_NO_DEVICE
    with pytest.raises(Q.QsaError) as e:
        c.slot_table_ptr(h, 0)
    assert e.value.status == Q.ERR_NO_DEVICE
    for name, args in [
        ("qsa_select_c4_topk", (C.byref(b), 16, 100, 2048, 16, 16, None)),
        ("qsa_gather_rows", (C.byref(b), 16, 16, 2048, 16, None, None)),
        ("qsa_append_token", (C.byref(b), 16, 16, None)),
        ("qsa_hot_cache_fetch", (C.byref(b), 16, 16, 2048, None)),
    ]:
        assert getattr(L, name)(c.h, *args) == Q.ERR_NO_DEVICE, name
        assert b"device storage" in L.qsa_last_error_string(), name
    st = L.qsa_staging_ptr(c.h, 0, C.byref(C.c_void_p()))
    assert st == Q.ERR_NO_DEVICE
    st32 = C.c_int32()
    assert L.qsa_poll_error(c.h, None, C.byref(st32), None) == Q.ERR_NO_DEVICE


def test_entry_points_reject_null_and_bad_arguments():
    """Null caches and outputs, bad layers and stale handles are refused with
    a status and a message, and change nothing."""
    L = N.lib()
    c = _host_cache()
    s0 = c.stats()
    h = c.request_begin(100, Q.KV_HBM)
    assert L.qsa_request_end(None, N.Handle(h.index, h.generation)) == Q.ERR_INVALID_ARG
    assert L.qsa_request_info_get(c.h, N.Handle(h.index, h.generation), None) == Q.ERR_INVALID_ARG
    assert L.qsa_cache_stats(c.h, None) == Q.ERR_INVALID_ARG
    assert L.qsa_request_advance(None, N.Handle(h.index, h.generation), 1) == Q.ERR_INVALID_ARG
    assert L.qsa_hot_cache_fetch(None, None, None, None, 2048, None) == Q.ERR_INVALID_ARG
    out = C.c_void_p()
    assert L.qsa_cache_create(None, C.byref(out)) == Q.ERR_INVALID_ARG
    assert L.qsa_cache_create(C.byref(c.cfg), None) == Q.ERR_INVALID_ARG
    stale = N.Handle(h.index, h.generation + 1)
    assert L.qsa_request_advance(c.h, stale, 1) == Q.ERR_STALE_HANDLE
    assert b"stale" in L.qsa_last_error_string()
    c.request_end(h)
    assert c.stats() == s0


def test_free_list_coalesces_after_fragmentation():
    rows = 12 * 2048 + 12 * 10000
    c = _host_cache(max_requests=8, hbm_pool_rows=rows)
    s0 = c.stats()
    hs = [c.request_begin(1000, Q.KV_HBM) for _ in range(8)]
    for i in (1, 3, 5):
        c.request_end(hs[i])
    s = c.stats()
    assert s["free_ranges"] == 4        # three holes + the tail
    for i in (0, 2, 4, 6, 7):
        c.request_end(hs[i])
    s = c.stats()
    assert s == s0 and s["free_ranges"] == 1 and s["largest_free_rows"] == 12 * 10000


def test_ragged_batch_recycling_returns_capacity():
    """64 requests with contexts log-uniform in [4096, 262144] (multiples of
    4): HBM-resident under 32K tokens, host history + 4096-token tail ring
    above.  Finish 16 random requests, reissue 16 new ones under new
    generations, then end everything: every counter returns to its initial
    value, and stale handles of finished requests are rejected."""
    ctxs = synth.log_uniform_contexts(64, 4096, 262144, seed=44)
    rows_needed = sum(12 * (n if n < 32768 else 4096) for n in ctxs)
    c = _host_cache(max_requests=64, hbm_pool_rows=12 * 2048 + rows_needed + 12 * 32768 * 16)
    s0 = c.stats()
    live = {}
    for n in ctxs:
        if n < 32768:
            h = c.request_begin(n, Q.KV_HBM)
        else:
            h = c.request_begin(n, Q.KV_HOST_RING, host_rows=1 << 30)
        live[h.index] = (h, n)
    assert c.stats()["free_request_slots"] == 0
    rng = random.Random(7)
    finished = rng.sample(sorted(live), 16)
    old = [live.pop(i)[0] for i in finished]
    for h in old:
        c.request_end(h)
    new_ctx = synth.log_uniform_contexts(16, 4096, 262144, seed=45)
    for n in new_ctx:
        h = c.request_begin(n, Q.KV_HBM if n < 32768 else Q.KV_HOST_RING,
                            host_rows=None if n < 32768 else 1 << 30)
        assert h.generation == 2
        live[h.index] = (h, n)
    for h in old:
        with pytest.raises(Q.QsaError) as e:
            c.request_end(h)
        assert e.value.status == Q.ERR_STALE_HANDLE
    leased = sum(12 * (n if n < 32768 else 4096) for _, n in live.values())
    assert c.stats()["hbm_kv_bytes_in_use"] == leased * 2048
    for h, _ in list(live.values()):
        c.request_end(h)
    assert c.stats() == s0


def test_request_growth_bookkeeping():
    """max_ctx sizes a resident request's region; qsa_request_advance grows
    ctx_len up to it and no further; bad arguments change nothing."""
    c = _host_cache()
    try:
        s0 = c.stats()
        h = c.request_begin(100, Q.KV_HBM, max_ctx=130)
        info = c.request_info(h)
        assert (info.ctx_len, info.max_ctx, info.layer_rows) == (100, 130, 130)
        assert c.stats()["free_hbm_rows"] == s0["free_hbm_rows"] - c.n_layers * 130
        c.advance(h, 25)
        c.advance(h)
        assert c.request_info(h).ctx_len == 126
        with pytest.raises(Q.QsaError) as e:
            c.advance(h, 5)
        assert e.value.status == Q.ERR_CAPACITY
        with pytest.raises(Q.QsaError) as e:
            c.advance(h, 0)
        assert e.value.status == Q.ERR_INVALID_ARG
        assert c.request_info(h).ctx_len == 126
        c.advance(h, 4)
        assert c.request_info(h).ctx_len == 130
        h2 = c.request_begin(10, Q.KV_HOST, host_rows=0x1000, max_ctx=20)
        assert c.request_info(h2).max_ctx == 20 and c.request_info(h2).layer_rows == 0
        with pytest.raises(Q.QsaError) as e:
            c.request_begin(10, Q.KV_HBM, max_ctx=5)          # max_ctx below ctx_len
        assert e.value.status == Q.ERR_INVALID_ARG
        with pytest.raises(Q.QsaError) as e:
            c.request_begin(10, Q.KV_HBM, max_ctx=c.ctx_capacity + 1)
        assert e.value.status == Q.ERR_CAPACITY
        c.request_end(h)
        with pytest.raises(Q.QsaError) as e:
            c.advance(h)
        assert e.value.status == Q.ERR_STALE_HANDLE
        c.request_end(h2)
        assert c.stats() == s0
    finally:
        c.close()


def test_hot_rows_config_workspace_and_leases():
    """Caches with a cross-step hot cache: hot_rows must be 0 or in
    [budget_tokens, QSA_MAX_HOT_ROWS]; the workspace grows by the hot-cache
    state; offloaded requests lease hot_rows rows per layer after their ring
    rows, HBM requests none; everything returns on request_end."""
    L = N.lib()
    cfg = N.CacheConfig(n_layers=12, max_requests=8, ctx_capacity=262144, budget_tokens=2048,
                        ring_tokens=4096, staging_rows=2048, hbm_pool_rows=1 << 20)
    base = L.qsa_workspace_bytes(C.byref(cfg))
    c2 = N.CacheConfig.from_buffer_copy(cfg)
    c2.hot_rows = 4096
    units = 8 * 12
    # fill list {token, row} per budget token, its length, the cursor, one owner per row,
    # the plan's pending row per budget token and its flag
    assert L.qsa_workspace_bytes(C.byref(c2)) == base + units * (2048 * 8 + 4 + 4 + 4096 * 4 + 2048 * 4 + 4)
    h = C.c_void_p()
    for field, bad in [("hot_rows", 2047), ("hot_rows", N.MAX_HOT_ROWS + 1), ("hot_rows", -4),
                       ("reserved1", 1)]:
        c3 = N.CacheConfig.from_buffer_copy(c2)
        setattr(c3, field, bad)
        assert L.qsa_workspace_bytes(C.byref(c3)) == -1
        assert L.qsa_cache_create(C.byref(c3), C.byref(h)) == N.ERR_INVALID_ARG

    c = _host_cache(hot_rows=2048)
    s0 = c.stats()
    ring = c.request_begin(262144, Q.KV_HOST_RING, host_rows=1 << 20)
    host = c.request_begin(262144, Q.KV_HOST, host_rows=1 << 22)
    hbm = c.request_begin(1000, Q.KV_HBM)
    ir, ih, ib = c.request_info(ring), c.request_info(host), c.request_info(hbm)
    assert ir.layer_rows == 4096 and ir.hot_row_base == ir.hbm_row_base + 12 * 4096
    assert ih.layer_rows == 0 and ih.hot_row_base == ih.hbm_row_base
    assert ib.hot_row_base == -1
    s1 = c.stats()
    assert s1["free_hbm_rows"] == s0["free_hbm_rows"] - 12 * (4096 + 2048) - 12 * 2048 - 12 * 1000
    assert s1["hbm_kv_bytes_in_use"] == (12 * (4096 + 2048) + 12 * 2048 + 12 * 1000) * 2048
    for hd in (ring, host, hbm):
        c.request_end(hd)
    assert c.stats() == s0
    with pytest.raises(Q.QsaError) as e:
        c.hot_cache_fetch([ring], 0, 1, None, None, 2048)
    assert e.value.status in (Q.ERR_NO_DEVICE, Q.ERR_STALE_HANDLE)


def test_header_is_plain_c():
    """include/qsa.h compiles as C99 (not only C++), with every declared
    entry point referenced, so C callers can use the ABI as declared."""
    import shutil
    import subprocess
    import tempfile
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    names = sorted(_declared_symbols())
    src = ("#include <qsa.h>\ntypedef void (*any_fn)(void);\n"
           + "\n".join(f"any_fn ref_{n} = (any_fn)&{n};" for n in names) + "\n")
    with tempfile.TemporaryDirectory() as d:
        path = os.path.join(d, "use_qsa.c")
        with open(path, "w") as f:
            f.write(src)
        r = subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-fsyntax-only",
                            "-I", os.path.join(ROOT, "include"), path], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


_C_PROGRAM = r"""
#include <qsa.h>
#include <stdio.h>
#include <string.h>

int main(void) {
  qsa_cache_config cfg;
  memset(&cfg, 0, sizeof cfg);
  cfg.n_layers = 12; cfg.max_requests = 4; cfg.ctx_capacity = 262144;
  cfg.budget_tokens = 2048; cfg.ring_tokens = 4096; cfg.staging_rows = 2048;
  cfg.kv_format = QSA_KV_BF16; cfg.hbm_pool_rows = 200000; cfg.hot_rows = 2048;
  if (qsa_abi_version() != QSA_ABI_VERSION) return 10;
  if (qsa_workspace_bytes(&cfg) <= 0) return 11;
  qsa_cache* c = NULL;
  if (qsa_cache_create(&cfg, &c) != QSA_OK || !c) return 12;
  qsa_stats s0, s1;
  if (qsa_cache_stats(c, &s0) != QSA_OK) return 13;
  qsa_request_desc d;
  memset(&d, 0, sizeof d);
  d.ctx_len = 262144; d.placement = QSA_KV_HOST_RING; d.host_rows = (const void*)(size_t)(1u << 20);
  qsa_handle h;
  if (qsa_request_begin(c, &d, NULL, &h) != QSA_OK) return 14;
  qsa_request_info info;
  if (qsa_request_info_get(c, h, &info) != QSA_OK) return 15;
  if (info.layer_rows != 4096 || info.hot_row_base != info.hbm_row_base + 12 * 4096) return 16;
  if (qsa_cache_stats(c, &s1) != QSA_OK || s1.free_hbm_rows != s0.free_hbm_rows - 12 * (4096 + 2048)) return 17;
  qsa_handle stale = h;
  stale.generation += 1;
  if (qsa_request_end(c, stale) != QSA_ERR_STALE_HANDLE) return 18;
  if (strlen(qsa_last_error_string()) == 0) return 19;
  if (qsa_request_end(c, h) != QSA_OK) return 20;
  if (qsa_cache_stats(c, &s1) != QSA_OK || memcmp(&s0, &s1, sizeof s0) != 0) return 21;
  if (qsa_cache_destroy(c) != QSA_OK) return 22;
  printf("c abi ok\n");
  return 0;
}
"""


def test_c_program_drives_the_host_bookkeeping():
    """A C program linked against libqsa_gb300.so leases, inspects and ends a
    request on a host-only cache (hot rows included) through the C ABI alone,
    and capacity returns to its initial value."""
    import shutil
    import subprocess
    import tempfile
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    libdir = os.path.dirname(N.LIB_PATH)
    with tempfile.TemporaryDirectory() as d:
        src, exe = os.path.join(d, "host_abi.c"), os.path.join(d, "host_abi")
        with open(src, "w") as f:
            f.write(_C_PROGRAM)
        r = subprocess.run([cc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), src,
                            "-o", exe, "-L", libdir, "-lqsa_gb300", f"-Wl,-rpath,{libdir}"],
                           capture_output=True, text=True)
        assert r.returncode == 0, r.stderr
        r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and "c abi ok" in r.stdout, (r.returncode, r.stdout, r.stderr)


class _PoolModel:
    """First-fit row ranges with coalescing, lowest free request slot, and
    the rows each placement leases: the allocation contract of the cache."""

    def __init__(self, pool_rows, staging, n_layers, ring, hot_rows, max_requests):
        self.free = [(staging, pool_rows - staging)] if pool_rows > staging else []
        self.n_layers, self.ring, self.hot = n_layers, ring, hot_rows
        self.slots = [None] * max_requests
        self.gen = [0] * max_requests

    def rows(self, n, placement):
        L = self.n_layers
        if placement == Q.KV_HBM:
            return L * n
        hot = L * self.hot
        return (L * self.ring if placement == Q.KV_HOST_RING else 0) + hot

    def begin(self, n, placement):
        """-> (slot, base) or an error status"""
        try:
            slot = self.slots.index(None)
        except ValueError:
            return Q.ERR_OUT_OF_SLOTS
        need = self.rows(n, placement)
        base = 0
        if need > 0:
            for i, (s, length) in enumerate(self.free):
                if length >= need:
                    base = s
                    self.free[i] = (s + need, length - need)
                    if self.free[i][1] == 0:
                        del self.free[i]
                    break
            else:
                return Q.ERR_CAPACITY
        self.slots[slot] = (base, need)
        self.gen[slot] += 1
        return slot, base

    def end(self, slot):
        base, n = self.slots[slot]
        self.slots[slot] = None
        if n == 0:
            return
        self.free.append((base, n))
        self.free.sort()
        merged = []
        for s, length in self.free:
            if merged and merged[-1][0] + merged[-1][1] == s:
                merged[-1] = (merged[-1][0], merged[-1][1] + length)
            else:
                merged.append((s, length))
        self.free = merged


@pytest.mark.parametrize("hot_rows", [0, 2048])
def test_pool_allocation_follows_first_fit_model(hot_rows):
    """Random admissions and finishes (all three placements, sizes up to the
    pool) on a host-only cache: every lease's pool base, every refusal and
    the free-capacity counters equal those of a first-fit model with
    coalescing; generations advance per slot."""
    rng = random.Random(17 + hot_rows)
    L, ring, staging, pool, maxr = 4, 512, 256, 60000, 6
    c = Q.Cache(n_layers=L, max_requests=maxr, ctx_capacity=20000, hbm_pool_rows=pool,
                budget_tokens=2048, ring_tokens=ring, staging_rows=staging, device=None, hot_rows=hot_rows)
    m = _PoolModel(pool, L * staging, L, ring, hot_rows, maxr)
    live = {}
    for step in range(400):
        if live and (rng.random() < 0.45 or len(live) == maxr):
            slot = rng.choice(sorted(live))
            c.request_end(live.pop(slot))
            m.end(slot)
        else:
            placement = rng.choice([Q.KV_HBM, Q.KV_HBM, Q.KV_HOST_RING, Q.KV_HOST])
            n = rng.randint(1, 20000) if placement != Q.KV_HBM else rng.randint(1, 6000)
            host = None if placement == Q.KV_HBM else 1 << 20
            want = m.begin(n, placement)
            if isinstance(want, tuple):
                h = c.request_begin(n, placement, host_rows=host)
                slot, base = want
                assert (h.index, h.generation) == (slot, m.gen[slot]), step
                info = c.request_info(h)
                if m.slots[slot][1] > 0:
                    assert info.hbm_row_base == base, step
                live[slot] = h
            else:
                with pytest.raises(Q.QsaError) as e:
                    c.request_begin(n, placement, host_rows=host)
                assert e.value.status == want, step
        st = c.stats()
        assert st["free_hbm_rows"] == sum(length for _, length in m.free), step
        assert st["free_ranges"] == len(m.free), step
        assert st["largest_free_rows"] == max((length for _, length in m.free), default=0), step
        assert st["active_requests"] == len(live), step
    for slot in sorted(live):
        c.request_end(live.pop(slot))
    assert c.stats()["free_hbm_rows"] == pool - L * staging


_C_DECODE_STEP = r"""
#include <cuda_runtime.h>
#include <qsa.h>
#include <stdio.h>
#include <string.h>

#define CK(x) do { if ((x) != cudaSuccess) return 1; } while (0)
#define QK(x) do { if ((x) != QSA_OK) { fprintf(stderr, "%s\n", qsa_last_error_string()); return 2; } } while (0)

/* One decode step of one HBM-resident request at one layer, from C with
   plain device pointers: score, select, attend, check the error word. */
int main(void) {
  const int n = 8192, budget = 2048, L = 1;
  qsa_cache_config cfg;
  memset(&cfg, 0, sizeof cfg);
  cfg.n_layers = L; cfg.max_requests = 1; cfg.ctx_capacity = n; cfg.budget_tokens = budget;
  cfg.ring_tokens = 4096; cfg.staging_rows = 0; cfg.kv_format = QSA_KV_BF16; cfg.hbm_pool_rows = n;
  CK(cudaMalloc(&cfg.hbm_pool, (size_t)n * QSA_ROW_BYTES));
  CK(cudaMalloc((void**)&cfg.index_keys, (size_t)n * QSA_INDEX_DIM));
  CK(cudaMalloc((void**)&cfg.index_scales, (size_t)n * 2));
  CK(cudaMalloc((void**)&cfg.slot_table, (size_t)n * 4));
  cfg.workspace_bytes = qsa_workspace_bytes(&cfg);
  CK(cudaMalloc(&cfg.workspace, (size_t)cfg.workspace_bytes));
  CK(cudaMemset(cfg.index_keys, 0x38, (size_t)n * QSA_INDEX_DIM));   /* e4m3 1.0 */
  CK(cudaMemset(cfg.index_scales, 0, (size_t)n * 2));
  CK(cudaMemset(cfg.hbm_pool, 0, (size_t)n * QSA_ROW_BYTES));
  qsa_cache* c = NULL;
  QK(qsa_cache_create(&cfg, &c));
  qsa_request_desc d;
  memset(&d, 0, sizeof d);
  d.ctx_len = n; d.placement = QSA_KV_HBM;
  qsa_handle h;
  QK(qsa_request_begin(c, &d, NULL, &h));
  float *q_idx, *w, *blk, *out, *lse;
  uint16_t* q;
  int32_t *sel, *nsel;
  CK(cudaMalloc((void**)&q_idx, 8 * 64 * 4)); CK(cudaMemset(q_idx, 0, 8 * 64 * 4));
  CK(cudaMalloc((void**)&w, 8 * 4)); CK(cudaMemset(w, 0, 8 * 4));
  CK(cudaMalloc((void**)&blk, (size_t)(n / 4) * 4));
  CK(cudaMalloc((void**)&sel, (size_t)(budget / 4) * 4));
  CK(cudaMalloc((void**)&nsel, 4));
  CK(cudaMalloc((void**)&q, 16 * 128 * 2)); CK(cudaMemset(q, 0, 16 * 128 * 2));
  CK(cudaMalloc((void**)&out, 16 * 128 * 4));
  CK(cudaMalloc((void**)&lse, 16 * 4));
  qsa_batch b = {1, 0, 1, 0, &h};
  QK(qsa_index_score(c, &b, q_idx, w, blk, n / 4, NULL));
  QK(qsa_select_c4_topk(c, &b, blk, n / 4, budget, sel, nsel, NULL));
  QK(qsa_sparse_decode_attn(c, &b, q, sel, nsel, budget, NULL, 0.0883883f, out, lse, NULL));
  int32_t st = -1;
  QK(qsa_poll_error(c, NULL, &st, NULL));
  if (st != QSA_OK) return 3;
  QK(qsa_request_end(c, h));
  QK(qsa_cache_destroy(c));
  printf("decode step ok\n");
  return 0;
}
"""


def test_c_decode_step_compiles_and_links():
    """A whole decode step written in C against the CUDA runtime (device
    buffers from cudaMalloc, no PyTorch) compiles and links against the
    library as declared."""
    import shutil
    import subprocess
    import tempfile
    cc = shutil.which("gcc") or shutil.which("cc")
    cuda = "/usr/local/cuda"
    if cc is None or not os.path.exists(os.path.join(cuda, "include", "cuda_runtime.h")):
        pytest.skip("no C compiler or CUDA headers")
    libdir = os.path.dirname(N.LIB_PATH)
    cudalib = next((p for p in (os.path.join(cuda, "lib64"), os.path.join(cuda, "lib"))
                    if os.path.isdir(p)), None)
    if cudalib is None:
        pytest.skip("no CUDA runtime library directory")
    with tempfile.TemporaryDirectory() as d:
        src, exe = os.path.join(d, "decode_step.c"), os.path.join(d, "decode_step")
        with open(src, "w") as f:
            f.write(_C_DECODE_STEP)
        r = subprocess.run([cc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                            "-I", os.path.join(cuda, "include"), src, "-o", exe, "-L", libdir,
                            "-lqsa_gb300", "-L", cudalib, "-lcudart", f"-Wl,-rpath,{libdir}"],
                           capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_host_memory_entry_points_check_their_arguments():
    """qsa_host_alloc refuses a null output and a non-positive size before it
    touches the driver; qsa_host_free accepts NULL and refuses an address it
    did not return (both without a GPU)."""
    L = N.lib()
    out = C.c_void_p()
    assert L.qsa_host_alloc(0, -1, 4096, None) == N.ERR_INVALID_ARG
    assert L.qsa_host_alloc(0, -1, 0, C.byref(out)) == N.ERR_INVALID_ARG
    assert L.qsa_host_alloc(0, -1, -5, C.byref(out)) == N.ERR_INVALID_ARG
    assert out.value is None
    assert L.qsa_host_free(None) == N.OK
    assert L.qsa_host_free(0x10000) == N.ERR_INVALID_ARG
    assert b"qsa_host_alloc" in L.qsa_last_error_string()


def test_workloads_refuse_an_unknown_host_memory_kind():
    from sparse_attention_decode_qsa_gb300 import workloads
    with pytest.raises(ValueError):
        workloads.alloc_host((1, 4, 2048), "cpu", "paged")
    assert set(workloads.HOST_MEMORY_KINDS) == {"vmm", "registered"}
