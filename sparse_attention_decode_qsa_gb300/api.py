"""Python binding of the QSA decode-step library: same names as the C ABI
(include/qsa.h), argument marshalling only.  Every step of the decode path
runs in the CUDA library; PyTorch only allocates the device and pinned host
buffers and supplies the stream.
"""
from __future__ import annotations

import ctypes as C

import torch

from . import _native as N
from ._native import QsaError, check  # noqa: F401  (re-exported)


def _ptr(t) -> int | None:
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream if torch.cuda.is_available() else None
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _batch(handles, layer0: int, n_layers: int):
    arr = (N.Handle * len(handles))(*[N.Handle(h.index, h.generation) for h in handles])
    b = N.Batch(len(handles), layer0, n_layers, 0, C.cast(arr, C.POINTER(N.Handle)))
    b._keep = arr
    return b


class HostMemory:
    """Host memory from qsa_host_alloc: pages on a host NUMA node, mapped into
    the device's page tables and the host's at one address.  Pass
    .cpu(shape) as a request's host_rows; .cuda(shape) is a view of the same
    bytes for device-side copies.  Freed by free() (or when collected)."""

    def __init__(self, nbytes: int, device: int = 0, numa_node: int = -1):
        self.L = N.lib()
        out = C.c_void_p()
        check(self.L.qsa_host_alloc(int(device), int(numa_node), int(nbytes), C.byref(out)),
              "qsa_host_alloc")
        self.ptr, self.nbytes, self.device = out.value, int(nbytes), int(device)

    def cpu(self, shape) -> torch.Tensor:
        import numpy as np
        n = 1
        for x in shape:
            n *= int(x)
        if n > self.nbytes:
            raise ValueError("view larger than the allocation")
        arr = np.ctypeslib.as_array((C.c_uint8 * n).from_address(self.ptr)).reshape(tuple(shape))
        t = torch.from_numpy(arr)
        t._qsa_host_memory = self          # the view keeps the allocation alive
        return t

    def cuda(self, shape) -> torch.Tensor:
        n = 1
        for x in shape:
            n *= int(x)
        if n > self.nbytes:
            raise ValueError("view larger than the allocation")

        class _View:
            __cuda_array_interface__ = {"shape": tuple(int(x) for x in shape), "typestr": "|u1",
                                        "data": (self.ptr, False), "version": 3, "strides": None}
        t = torch.as_tensor(_View(), device=torch.device("cuda", self.device))
        t._qsa_host_memory = self
        return t

    def free(self):
        if getattr(self, "ptr", None):
            check(self.L.qsa_host_free(self.ptr), "qsa_host_free")
            self.ptr = None

    def __del__(self):
        try:
            self.free()
        except Exception:
            pass


class Cache:
    """A qsa_cache plus the device storage it runs on.

    With device=None the cache is host-only (bookkeeping without a GPU).
    Storage layout (all owned here, passed to the library as raw pointers):
      pool         uint8 [hbm_pool_rows][row_bytes] (2048 BF16 rows, 1040 FP8 rows)
      index_keys   uint8 [max_requests][n_layers][ctx_capacity][64]
      index_scales fp16  [max_requests][n_layers][ctx_capacity]
      slot_table   int32 [max_requests][n_layers][ctx_capacity]
      workspace    uint8 [qsa_workspace_bytes]
    hot_rows > 0 gives every offloaded request that many hot rows per layer
    (the cross-step hot cache filled by hot_cache_fetch).
    """

    def __init__(self, n_layers: int, max_requests: int, ctx_capacity: int,
                 hbm_pool_rows: int, budget_tokens: int = 2048, ring_tokens: int = 4096,
                 staging_rows: int = 2048, device="cuda", kv_format: int = N.KV_BF16,
                 hot_rows: int = 0):
        self.L = N.lib()
        cfg = N.CacheConfig()
        cfg.n_layers = n_layers
        cfg.max_requests = max_requests
        cfg.ctx_capacity = ctx_capacity
        cfg.budget_tokens = budget_tokens
        cfg.ring_tokens = ring_tokens
        cfg.staging_rows = staging_rows
        cfg.hbm_pool_rows = hbm_pool_rows
        cfg.kv_format = kv_format
        cfg.hot_rows = hot_rows
        self.kv_format = kv_format
        self.hot_rows = hot_rows
        self.row_bytes = N.ROW_BYTES_FP8 if kv_format == N.KV_FP8 else N.ROW_BYTES
        self.n_layers, self.max_requests, self.ctx_capacity = n_layers, max_requests, ctx_capacity
        self.budget_tokens, self.ring_tokens, self.staging_rows = budget_tokens, ring_tokens, staging_rows
        self.device = device
        if device is not None:
            ws = self.L.qsa_workspace_bytes(C.byref(cfg))
            if ws < 0:
                raise QsaError(N.ERR_INVALID_ARG, "qsa_workspace_bytes", "bad config")
            self.pool = torch.empty(hbm_pool_rows, self.row_bytes, dtype=torch.uint8, device=device)
            self.index_keys = torch.zeros(max_requests, n_layers, ctx_capacity, N.INDEX_DIM,
                                          dtype=torch.uint8, device=device)
            self.index_scales = torch.zeros(max_requests, n_layers, ctx_capacity,
                                            dtype=torch.float16, device=device)
            self.slot_table = torch.empty(max_requests, n_layers, ctx_capacity,
                                          dtype=torch.int32, device=device)
            self.workspace = torch.empty(ws, dtype=torch.uint8, device=device)
            cfg.hbm_pool = self.pool.data_ptr()
            cfg.index_keys = self.index_keys.data_ptr()
            cfg.index_scales = self.index_scales.data_ptr()
            cfg.slot_table = self.slot_table.data_ptr()
            cfg.workspace = self.workspace.data_ptr()
            cfg.workspace_bytes = ws
        self.cfg = cfg
        h = C.c_void_p()
        check(self.L.qsa_cache_create(C.byref(cfg), C.byref(h)), "qsa_cache_create")
        self.h = h
        self._host = {}

    def close(self):
        if getattr(self, "h", None):
            self.L.qsa_cache_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # ------------------------------------------------------- bookkeeping
    def request_begin(self, ctx_len: int, placement: int = N.KV_HBM, host_rows=None,
                      stream=None, max_ctx: int = 0) -> N.Handle:
        """Lease a request of ctx_len tokens that may grow to max_ctx (0: no
        growth).  host_rows: pinned host history [n_layers][max(ctx_len,
        max_ctx)][2048] for the host placements."""
        d = N.RequestDesc(ctx_len, placement, max_ctx, None)
        if host_rows is not None:
            d.host_rows = host_rows.data_ptr() if isinstance(host_rows, torch.Tensor) else int(host_rows)
        out = N.Handle()
        check(self.L.qsa_request_begin(self.h, C.byref(d), _stream(stream) if self.device else None,
                                       C.byref(out)), "qsa_request_begin")
        if isinstance(host_rows, torch.Tensor):
            self._host[out.index] = host_rows
        return out

    def request_end(self, handle: N.Handle):
        check(self.L.qsa_request_end(self.h, handle), "qsa_request_end")
        self._host.pop(handle.index, None)

    def request_info(self, handle: N.Handle) -> N.RequestInfo:
        out = N.RequestInfo()
        check(self.L.qsa_request_info_get(self.h, handle, C.byref(out)), "qsa_request_info_get")
        return out

    def advance(self, handle: N.Handle, n_new: int = 1):
        """Reserve the positions of n_new new tokens (ctx_len grows by n_new)."""
        check(self.L.qsa_request_advance(self.h, handle, n_new), "qsa_request_advance")

    def stats(self) -> dict:
        out = N.Stats()
        check(self.L.qsa_cache_stats(self.h, C.byref(out)), "qsa_cache_stats")
        return out.as_dict()

    def slot_table_ptr(self, handle: N.Handle, layer: int) -> int:
        out = C.c_void_p()
        check(self.L.qsa_slot_table_ptr(self.h, handle, layer, C.byref(out)), "qsa_slot_table_ptr")
        return out.value

    def slot_table_set(self, handle: N.Handle, layer: int, tokens, slots, stream=None):
        check(self.L.qsa_slot_table_set(self.h, handle, layer, _ptr(tokens), _ptr(slots),
                                        int(tokens.numel()), _stream(stream)), "qsa_slot_table_set")

    def staging_ptr(self, layer: int) -> int:
        out = C.c_void_p()
        check(self.L.qsa_staging_ptr(self.h, layer, C.byref(out)), "qsa_staging_ptr")
        return out.value

    def poll_error(self, stream=None):
        st, det = C.c_int32(), C.c_int64()
        check(self.L.qsa_poll_error(self.h, _stream(stream), C.byref(st), C.byref(det)),
              "qsa_poll_error")
        return st.value, det.value

    # ------------------------------------------------------ producer side
    def append_token(self, handles, layer0, n_layers, k_new, kv_new, stream=None):
        """Store each unit's newest token: k_new fp32 [units][64] index keys,
        kv_new uint8 [units][2048] KV rows (unit u = i_layer * n_req + i_req)."""
        b = _batch(handles, layer0, n_layers)
        check(self.L.qsa_append_token(self.h, C.byref(b), _ptr(k_new), _ptr(kv_new),
                                      _stream(stream)), "qsa_append_token")

    # ---------------------------------------------------------- hot path
    def index_score(self, handles, layer0, n_layers, q_idx, w, blk_scores, stream=None):
        b = _batch(handles, layer0, n_layers)
        check(self.L.qsa_index_score(self.h, C.byref(b), _ptr(q_idx), _ptr(w), _ptr(blk_scores),
                                     blk_scores.shape[-1], _stream(stream)), "qsa_index_score")

    def select_c4_topk(self, handles, layer0, n_layers, blk_scores, budget_tokens, sel_blocks,
                       n_sel, stream=None):
        b = _batch(handles, layer0, n_layers)
        check(self.L.qsa_select_c4_topk(self.h, C.byref(b), _ptr(blk_scores), blk_scores.shape[-1],
                                        budget_tokens, _ptr(sel_blocks), _ptr(n_sel),
                                        _stream(stream)), "qsa_select_c4_topk")

    def gather_rows(self, handles, layer0, n_layers, sel_blocks, n_sel, budget_tokens, rows_out,
                    n_rows=None, stream=None):
        b = _batch(handles, layer0, n_layers)
        out_ptr = rows_out if isinstance(rows_out, int) else _ptr(rows_out)
        check(self.L.qsa_gather_rows(self.h, C.byref(b), _ptr(sel_blocks), _ptr(n_sel),
                                     budget_tokens, out_ptr, _ptr(n_rows), _stream(stream)),
              "qsa_gather_rows")

    def hot_cache_fetch(self, handles, layer0, n_layers, sel_blocks, n_sel, budget_tokens,
                        stream=None):
        b = _batch(handles, layer0, n_layers)
        check(self.L.qsa_hot_cache_fetch(self.h, C.byref(b), _ptr(sel_blocks), _ptr(n_sel),
                                         budget_tokens, _stream(stream)), "qsa_hot_cache_fetch")

    def hot_cache_plan(self, handles, layer0, n_layers, sel_blocks, n_sel, budget_tokens,
                       stream=None):
        b = _batch(handles, layer0, n_layers)
        check(self.L.qsa_hot_cache_plan(self.h, C.byref(b), _ptr(sel_blocks), _ptr(n_sel),
                                        budget_tokens, _stream(stream)), "qsa_hot_cache_plan")

    def sparse_decode_attn(self, handles, layer0, n_layers, q, sel_blocks, n_sel, budget_tokens,
                           gathered, softmax_scale, out, lse=None, stream=None):
        b = _batch(handles, layer0, n_layers)
        g = gathered if (gathered is None or isinstance(gathered, int)) else _ptr(gathered)
        check(self.L.qsa_sparse_decode_attn(self.h, C.byref(b), _ptr(q.view(torch.int16)),
                                            _ptr(sel_blocks), _ptr(n_sel), budget_tokens, g,
                                            float(softmax_scale), _ptr(out), _ptr(lse),
                                            _stream(stream)), "qsa_sparse_decode_attn")
