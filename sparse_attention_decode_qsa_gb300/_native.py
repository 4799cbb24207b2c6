"""ctypes declarations of the C ABI in include/qsa.h.

Loading fails loudly: there is no fallback path.  Build the library first
(python -m sparse_attention_decode_qsa_gb300.build, or __graft_entry__.build()).
"""
from __future__ import annotations

import ctypes as C
import os

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libqsa_gb300.so")

INDEX_HEADS = 8
INDEX_DIM = 64
KV_HEADS = 4
HEAD_DIM = 128
Q_HEADS = 16
ROW_BYTES = 2048
ROW_BYTES_FP8 = 1040
KV_BF16 = 0
KV_FP8 = 1
MAX_UNITS = 256
MAX_BUDGET_TOKENS = 8192
MAX_HOT_ROWS = 65536
STATIC_MAX_UNITS = 16
STATIC_MAX_ROWS = 2048

STATUS = {
    0: "QSA_OK", 1: "QSA_ERR_INVALID_ARG", 2: "QSA_ERR_CUDA", 3: "QSA_ERR_STALE_HANDLE",
    4: "QSA_ERR_OUT_OF_SLOTS", 5: "QSA_ERR_CAPACITY", 6: "QSA_ERR_BAD_SLOT",
    7: "QSA_ERR_TIMEOUT", 8: "QSA_ERR_BAD_BLOCK", 9: "QSA_ERR_NO_DEVICE",
}
OK, ERR_INVALID_ARG, ERR_CUDA, ERR_STALE_HANDLE, ERR_OUT_OF_SLOTS, ERR_CAPACITY, \
    ERR_BAD_SLOT, ERR_TIMEOUT, ERR_BAD_BLOCK, ERR_NO_DEVICE = range(10)

KV_HBM = 0
KV_HOST_RING = 1
KV_HOST = 2


class CacheConfig(C.Structure):
    _fields_ = [
        ("n_layers", C.c_int32), ("max_requests", C.c_int32), ("ctx_capacity", C.c_int64),
        ("budget_tokens", C.c_int32), ("ring_tokens", C.c_int32), ("staging_rows", C.c_int32),
        ("kv_format", C.c_int32), ("hbm_pool_rows", C.c_int64),
        ("hbm_pool", C.c_void_p), ("index_keys", C.c_void_p), ("index_scales", C.c_void_p),
        ("slot_table", C.c_void_p), ("workspace", C.c_void_p), ("workspace_bytes", C.c_int64),
        ("hot_rows", C.c_int32), ("reserved1", C.c_int32),
    ]


class Handle(C.Structure):
    _fields_ = [("index", C.c_uint32), ("generation", C.c_uint32)]

    def __repr__(self):
        return f"Handle(index={self.index}, generation={self.generation})"


class RequestDesc(C.Structure):
    _fields_ = [("ctx_len", C.c_int64), ("placement", C.c_int32), ("max_ctx", C.c_int32),
                ("host_rows", C.c_void_p)]


class RequestInfo(C.Structure):
    _fields_ = [("ctx_len", C.c_int64), ("placement", C.c_int32), ("layer_rows", C.c_int32),
                ("hbm_row_base", C.c_int64), ("host_rows", C.c_void_p), ("max_ctx", C.c_int64),
                ("hot_row_base", C.c_int64)]


class Stats(C.Structure):
    _fields_ = [
        ("max_requests", C.c_int32), ("active_requests", C.c_int32),
        ("free_request_slots", C.c_int32), ("free_ranges", C.c_int32),
        ("hbm_pool_rows", C.c_int64), ("free_hbm_rows", C.c_int64),
        ("largest_free_rows", C.c_int64), ("staging_rows_total", C.c_int64),
        ("hbm_kv_bytes_in_use", C.c_int64),
    ]

    def as_dict(self):
        return {f: getattr(self, f) for f, _ in self._fields_}


class Batch(C.Structure):
    _fields_ = [("n_req", C.c_int32), ("layer0", C.c_int32), ("n_layers", C.c_int32),
                ("reserved0", C.c_int32), ("requests", C.POINTER(Handle))]


# name -> (restype, argtypes); every entry point declared in include/qsa.h
SIGNATURES = {
    "qsa_abi_version": (C.c_int32, []),
    "qsa_last_error_string": (C.c_char_p, []),
    "qsa_workspace_bytes": (C.c_int64, [C.POINTER(CacheConfig)]),
    "qsa_cache_create": (C.c_int, [C.POINTER(CacheConfig), C.POINTER(C.c_void_p)]),
    "qsa_cache_destroy": (C.c_int, [C.c_void_p]),
    "qsa_request_begin": (C.c_int, [C.c_void_p, C.POINTER(RequestDesc), C.c_void_p, C.POINTER(Handle)]),
    "qsa_request_end": (C.c_int, [C.c_void_p, Handle]),
    "qsa_request_info_get": (C.c_int, [C.c_void_p, Handle, C.POINTER(RequestInfo)]),
    "qsa_cache_stats": (C.c_int, [C.c_void_p, C.POINTER(Stats)]),
    "qsa_request_advance": (C.c_int, [C.c_void_p, Handle, C.c_int32]),
    "qsa_append_token": (C.c_int, [C.c_void_p, C.POINTER(Batch), C.c_void_p, C.c_void_p, C.c_void_p]),
    "qsa_slot_table_ptr": (C.c_int, [C.c_void_p, Handle, C.c_int32, C.POINTER(C.c_void_p)]),
    "qsa_slot_table_set": (C.c_int, [C.c_void_p, Handle, C.c_int32, C.c_void_p, C.c_void_p,
                                     C.c_int32, C.c_void_p]),
    "qsa_staging_ptr": (C.c_int, [C.c_void_p, C.c_int32, C.POINTER(C.c_void_p)]),
    "qsa_poll_error": (C.c_int, [C.c_void_p, C.c_void_p, C.POINTER(C.c_int32), C.POINTER(C.c_int64)]),
    "qsa_index_score": (C.c_int, [C.c_void_p, C.POINTER(Batch), C.c_void_p, C.c_void_p,
                                  C.c_void_p, C.c_int64, C.c_void_p]),
    "qsa_select_c4_topk": (C.c_int, [C.c_void_p, C.POINTER(Batch), C.c_void_p, C.c_int64,
                                     C.c_int32, C.c_void_p, C.c_void_p, C.c_void_p]),
    "qsa_gather_rows": (C.c_int, [C.c_void_p, C.POINTER(Batch), C.c_void_p, C.c_void_p,
                                  C.c_int32, C.c_void_p, C.c_void_p, C.c_void_p]),
    "qsa_hot_cache_fetch": (C.c_int, [C.c_void_p, C.POINTER(Batch), C.c_void_p, C.c_void_p,
                                      C.c_int32, C.c_void_p]),
    "qsa_hot_cache_plan": (C.c_int, [C.c_void_p, C.POINTER(Batch), C.c_void_p, C.c_void_p,
                                     C.c_int32, C.c_void_p]),
    "qsa_sparse_decode_attn": (C.c_int, [C.c_void_p, C.POINTER(Batch), C.c_void_p, C.c_void_p,
                                         C.c_void_p, C.c_int32, C.c_void_p, C.c_float,
                                         C.c_void_p, C.c_void_p, C.c_void_p]),
    "qsa_host_alloc": (C.c_int, [C.c_int32, C.c_int32, C.c_int64, C.POINTER(C.c_void_p)]),
    "qsa_host_free": (C.c_int, [C.c_void_p]),
    "qsa_sparse_decode_attn_noalloc": (C.c_int, [C.c_void_p, C.c_void_p, C.c_void_p, C.c_int32,
                                                 C.c_int32, C.c_float, C.c_void_p, C.c_void_p,
                                                 C.c_void_p]),
}

_lib = None


def lib() -> C.CDLL:
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"QSA CUDA library not built: {LIB_PATH} is missing "
                               "(run python -m sparse_attention_decode_qsa_gb300.build)")
        L = C.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


class QsaError(RuntimeError):
    def __init__(self, status: int, func: str, msg: str):
        self.status = status
        super().__init__(f"{func} -> {STATUS.get(status, status)}: {msg}")


def check(status: int, func: str):
    if status != OK:
        raise QsaError(status, func, lib().qsa_last_error_string().decode(errors="replace"))
