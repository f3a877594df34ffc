"""GB300 multi-adapter LoRA projection: Python binding over liblora.so (C ABI in include/lora.h).

Every function here has the name of the C entry point it wraps and only
marshals arguments: device pointers may be given as ints or as objects with a
``data_ptr()`` method (PyTorch tensors), host arrays as NumPy arrays, streams
as ``cudaStream_t`` ints (default: PyTorch's current stream).  A non-zero
status raises :class:`LoraError` carrying the code and ``lora_last_error()``.

The library must be built first (``adapter_gemm_lora_gb300.build.build()``);
there is no fallback implementation: if the shared library is missing, loading
it raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "liblora.so")

LORA_OK = 0
LORA_EINVAL = -1
LORA_ENOPAGES = -2
LORA_EUNKNOWN_ADAPTER = -3
LORA_ERANK = -4
LORA_EEXIST = -5
LORA_ECUDA = -6
LORA_EDEVICE = -7
LORA_EBUSY = -8
LORA_EVICT_LOAD_ORDER = 0
LORA_EVICT_LRU = 1
LORA_EVICT_FARTHEST = 2
LORA_MAX_RANK = 64
LORA_MAX_ADAPTERS = 16384
LORA_MAX_TOKENS = 65536
LORA_MAX_GROUP = 4
LORA_NOALLOC_MAX_TOKENS = 128
LORA_NOALLOC_MAX_H = 8192
LORA_NOALLOC_SCRATCH_BYTES = 17 * 1024 * 1024

EXPORTED = ["lora_pool_create", "lora_pool_reserve", "lora_pool_release", "lora_adapter_load",
            "lora_adapter_unload", "lora_segments_size", "lora_segments_init", "lora_segments_build",
            "lora_linear_forward", "lora_status", "lora_pool_stats", "lora_last_error", "lora_pool_destroy",
            "lora_profile_enable", "lora_profile_read", "lora_linear_forward_noalloc",
            "lora_segments_size_group", "lora_segments_init_group", "lora_linear_forward_group",
            "lora_adapter_acquire", "lora_adapter_release", "lora_adapter_refs", "lora_pool_evict_idle",
            "lora_adapter_ensure", "lora_pool_set_eviction", "lora_adapter_packed_size", "lora_adapter_pack",
            "lora_adapter_load_packed", "lora_adapter_wait", "lora_kv_grow", "lora_kv_free", "lora_kv_length",
            "lora_kv_table", "lora_kv_batch_table", "lora_attention_decode"]
KINDS = ("segments", "delta", "gemm", "scatter", "shrink", "attention")


class LoraError(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(f"[{code}] {message}")
        self.code = code
        self.message = message


class lora_segments(ctypes.Structure):
    _fields_ = [("T_max", ctypes.c_int32), ("T", ctypes.c_int32), ("max_seg", ctypes.c_int32), ("H", ctypes.c_int32),
                ("perm", ctypes.c_void_p), ("seg_off", ctypes.c_void_p), ("seg_adapter", ctypes.c_void_p),
                ("n_seg", ctypes.c_void_p), ("tok_adapter", ctypes.c_void_p), ("units", ctypes.c_void_p),
                ("n_units", ctypes.c_void_p), ("unit_cap", ctypes.c_int32), ("delta_slots", ctypes.c_int32),
                ("delta", ctypes.c_void_p), ("gemm_partials", ctypes.c_void_p),
                ("n_tiles_max", ctypes.c_int32), ("tile_plan", ctypes.c_void_p), ("entries", ctypes.c_void_p),
                ("n_entries", ctypes.c_void_p), ("units_rest", ctypes.c_void_p), ("n_units_rest", ctypes.c_void_p),
                ("s_lora", ctypes.c_void_p), ("shrink_scratch", ctypes.c_void_p)]


class lora_pool_stats_t(ctypes.Structure):
    _fields_ = [("num_pages", ctypes.c_int64), ("free_pages", ctypes.c_int64), ("adapter_pages", ctypes.c_int64),
                ("reserved_pages", ctypes.c_int64), ("resident_adapters", ctypes.c_int32),
                ("max_adapters", ctypes.c_int32)]


_lib = None


def _load():
    global _lib
    if _lib is not None:
        return _lib
    path = os.environ.get("LORA_LIB", LIB_PATH)
    if not os.path.exists(path):
        raise RuntimeError(f"liblora.so not found at {path}; build it with adapter_gemm_lora_gb300.build.build()")
    lib = ctypes.CDLL(path)
    P, I32, I64, VP = ctypes.POINTER, ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p
    sig = {
        "lora_pool_create": (I32, [VP, I64, I32, I32, I32, VP, P(VP)]),
        "lora_pool_reserve": (I32, [VP, I64, VP]),
        "lora_pool_release": (I32, [VP, I64, VP]),
        "lora_adapter_load": (I32, [VP, I32, I32, VP, VP, VP, VP]),
        "lora_adapter_unload": (I32, [VP, I32, VP]),
        "lora_segments_size": (I64, [VP, I32]),
        "lora_segments_init": (I32, [VP, VP, I64, I32, P(lora_segments)]),
        "lora_segments_build": (I32, [VP, VP, I32, P(lora_segments), VP]),
        "lora_linear_forward": (I32, [VP, P(lora_segments), I32, VP, VP, VP, VP, VP]),
        "lora_status": (I32, [VP, VP]),
        "lora_pool_stats": (None, [VP, P(lora_pool_stats_t)]),
        "lora_last_error": (ctypes.c_char_p, []),
        "lora_pool_destroy": (None, [VP]),
        "lora_profile_enable": (I32, [VP, I32]),
        "lora_profile_read": (I32, [VP, I32, VP, VP, I32]),
        "lora_linear_forward_noalloc": (I32, [VP, VP, I32, I32, VP, VP, VP, VP]),
        "lora_segments_size_group": (I64, [VP, I32, I32]),
        "lora_segments_init_group": (I32, [VP, VP, I64, I32, I32, P(lora_segments)]),
        "lora_linear_forward_group": (I32, [VP, P(lora_segments), I32, VP, VP, VP, VP, VP, VP]),
        "lora_adapter_acquire": (I32, [VP, I32]),
        "lora_adapter_release": (I32, [VP, I32]),
        "lora_adapter_refs": (I32, [VP, I32]),
        "lora_pool_evict_idle": (I32, [VP, I64, VP, VP, VP]),
        "lora_adapter_ensure": (I32, [VP, I32, I32, VP, VP, VP, VP, VP, VP, VP]),
        "lora_pool_set_eviction": (I32, [VP, I32, VP, I64, I32]),
        "lora_adapter_packed_size": (I64, [VP, I32, VP]),
        "lora_adapter_pack": (I32, [VP, I32, VP, VP, VP, I64]),
        "lora_adapter_load_packed": (I32, [VP, I32, I32, VP, VP, I64, VP, VP]),
        "lora_adapter_wait": (I32, [VP, I32, VP]),
        "lora_kv_grow": (I32, [VP, I64, I32, I32, VP]),
        "lora_kv_free": (I32, [VP, I64]),
        "lora_kv_length": (I64, [VP, I64]),
        "lora_kv_table": (I32, [VP, I64, I32, VP]),
        "lora_kv_batch_table": (I32, [VP, VP, I32, I32, VP, VP, VP]),
        "lora_attention_decode": (I32, [VP, I32, VP, VP, I32, I32, I32, VP, VP, I32, VP]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def library():
    """The loaded ctypes library (loads it on first use)."""
    return _load()


def _ptr(obj) -> Optional[int]:
    if obj is None:
        return None
    if isinstance(obj, int):
        return obj
    if hasattr(obj, "data_ptr"):
        return obj.data_ptr()
    if isinstance(obj, np.ndarray):
        return obj.ctypes.data
    raise TypeError(f"cannot take a pointer of {type(obj)!r}")


def _stream(stream) -> Optional[int]:
    if stream is not None:
        return int(stream) if not hasattr(stream, "cuda_stream") else stream.cuda_stream
    import torch
    return torch.cuda.current_stream().cuda_stream


def _check(rc: int) -> None:
    if rc != LORA_OK:
        raise LoraError(rc, lora_last_error())


def lora_last_error() -> str:
    return _load().lora_last_error().decode()


def lora_pool_create(pool_dev, num_pages: int, H: int, n_slots: int, max_adapters: int,
                     page_order: Optional[np.ndarray] = None) -> ctypes.c_void_p:
    """Create a pool over device bf16 storage [num_pages][H] (None: planning pool)."""
    order = None if page_order is None else np.ascontiguousarray(page_order, dtype=np.int64)
    out = ctypes.c_void_p()
    _check(_load().lora_pool_create(_ptr(pool_dev), num_pages, H, n_slots, max_adapters, _ptr(order),
                                    ctypes.byref(out)))
    return out


def lora_pool_reserve(pool, n: int) -> np.ndarray:
    ids = np.zeros(max(n, 1), dtype=np.int64)
    _check(_load().lora_pool_reserve(pool, n, _ptr(ids)))
    return ids[:n]


def lora_pool_release(pool, ids) -> None:
    ids = np.ascontiguousarray(ids, dtype=np.int64)
    _check(_load().lora_pool_release(pool, ids.size, _ptr(ids) if ids.size else None))


def lora_adapter_load(pool, adapter_id: int, rank: int, A_host: Optional[Sequence], B_host: Optional[Sequence],
                      n_slots: int, stream=None, planning: bool = False) -> np.ndarray:
    """Load one adapter; A_host[slot] bf16 bits [H, rank] (None: no LoRA there), B_host[slot] [rank, H].

    Returns the page table int32 [n_slots, 2, rank].
    """
    keep = []

    def arr(seq):
        if seq is None:
            return None
        a = (ctypes.c_void_p * n_slots)()
        for i, m in enumerate(seq):
            if m is None:
                a[i] = None
            else:
                m = np.ascontiguousarray(m, dtype=np.uint16)
                keep.append(m)
                a[i] = m.ctypes.data
        return a

    a_arr, b_arr = arr(A_host), arr(B_host)
    table = np.zeros((n_slots, 2, rank), dtype=np.int32)
    st = 0 if planning else _stream(stream)
    rc = _load().lora_adapter_load(pool, adapter_id, rank, ctypes.cast(a_arr, ctypes.c_void_p) if a_arr else None,
                                   ctypes.cast(b_arr, ctypes.c_void_p) if b_arr else None, st, _ptr(table))
    _check(rc)
    return table


def lora_adapter_unload(pool, adapter_id: int, stream=None, planning: bool = False) -> None:
    _check(_load().lora_adapter_unload(pool, adapter_id, 0 if planning else _stream(stream)))


def lora_adapter_acquire(pool, adapter_id: int) -> None:
    _check(_load().lora_adapter_acquire(pool, adapter_id))


def lora_adapter_release(pool, adapter_id: int) -> None:
    _check(_load().lora_adapter_release(pool, adapter_id))


def lora_pool_set_eviction(pool, policy: int, future=None, lookahead: int = 0) -> None:
    """Eviction rule for idle adapters; `future` = upcoming adapter requests (farthest-future rule)."""
    fut = np.ascontiguousarray(np.zeros(0) if future is None else future, dtype=np.int32)
    _check(_load().lora_pool_set_eviction(pool, policy, _ptr(fut) if fut.size else None, fut.size, lookahead))


def _present(present, n_slots):
    return None if present is None else np.ascontiguousarray([1 if p else 0 for p in present], dtype=np.int32)


def lora_adapter_packed_size(pool, rank: int, present=None, n_slots: int = 0) -> int:
    pr = _present(present, n_slots)
    n = _load().lora_adapter_packed_size(pool, rank, _ptr(pr))
    if n < 0:
        raise LoraError(int(n), lora_last_error())
    return int(n)


def lora_adapter_pack(pool, rank: int, A_host: Sequence, B_host: Sequence, packed_host, packed_bytes: int) -> None:
    """Pack an adapter's factors (bf16 bits; A_host[slot] [H, rank] or None) into page rows in `packed_host`."""
    n = len(A_host)
    keep = []
    a_arr, b_arr = (ctypes.c_void_p * n)(), (ctypes.c_void_p * n)()
    for i in range(n):
        if A_host[i] is not None:
            a = np.ascontiguousarray(A_host[i], dtype=np.uint16)
            b = np.ascontiguousarray(B_host[i], dtype=np.uint16)
            keep += [a, b]
            a_arr[i], b_arr[i] = a.ctypes.data, b.ctypes.data
    _check(_load().lora_adapter_pack(pool, rank, ctypes.cast(a_arr, ctypes.c_void_p), ctypes.cast(b_arr, ctypes.c_void_p),
                                     _ptr(packed_host), packed_bytes))


def lora_adapter_load_packed(pool, adapter_id: int, rank: int, packed_pinned, packed_bytes: int, n_slots: int,
                             present=None, copy_stream=None) -> np.ndarray:
    """Load from a packed buffer in pinned host memory on `copy_stream`, without synchronising."""
    pr = _present(present, n_slots)
    table = np.zeros((n_slots, 2, rank), dtype=np.int32)
    _check(_load().lora_adapter_load_packed(pool, adapter_id, rank, _ptr(pr), _ptr(packed_pinned), packed_bytes,
                                            _stream(copy_stream), _ptr(table)))
    return table


def lora_adapter_wait(pool, adapter_id: int, stream=None) -> None:
    _check(_load().lora_adapter_wait(pool, adapter_id, _stream(stream)))


def lora_kv_grow(pool, request_id: int, n_tokens: int, layers: int) -> list:
    """KV pages for n_tokens new tokens of a request (2 * layers per token); returns their ids."""
    ids = np.zeros(max(2 * layers * n_tokens, 1), dtype=np.int32)
    _check(_load().lora_kv_grow(pool, request_id, n_tokens, layers, _ptr(ids)))
    return ids[:2 * layers * n_tokens].tolist()


def lora_kv_free(pool, request_id: int) -> None:
    _check(_load().lora_kv_free(pool, request_id))


def lora_kv_length(pool, request_id: int) -> int:
    return int(_load().lora_kv_length(pool, request_id))


def lora_kv_table(pool, request_id: int, layer: int) -> np.ndarray:
    """int32 [tokens, 2]: the (K page, V page) of every cached token of a request at one layer."""
    n = lora_kv_length(pool, request_id)
    if n < 0:
        raise LoraError(LORA_EINVAL, f"request {request_id} holds no KV pages")
    out = np.zeros((max(n, 1), 2), dtype=np.int32)
    _check(_load().lora_kv_table(pool, request_id, layer, _ptr(out)))
    return out[:n]


def lora_kv_batch_table(pool, request_ids, max_len: int, table_dev, seq_len_dev, stream=None) -> None:
    """Every request's KV page list (as lora_kv_grow took it) into table_dev, lengths into seq_len_dev."""
    ids = np.ascontiguousarray(request_ids, dtype=np.int64)
    _check(_load().lora_kv_batch_table(pool, _ptr(ids) if ids.size else None, ids.size, max_len, _ptr(table_dev),
                                       _ptr(seq_len_dev), _stream(stream)))


def lora_attention_decode(pool, n_req: int, table_dev, seq_len_dev, max_len: int, layers: int, layer: int, q_dev,
                          out_dev, n_heads: int, stream=None) -> None:
    """Decode attention of one new token per request over its KV pages at `layer`."""
    _check(_load().lora_attention_decode(pool, n_req, _ptr(table_dev), _ptr(seq_len_dev), max_len, layers, layer,
                                         _ptr(q_dev), _ptr(out_dev), n_heads, _stream(stream)))


def lora_adapter_refs(pool, adapter_id: int) -> int:
    """Active requests of a resident adapter, -1 if it is not resident."""
    return int(_load().lora_adapter_refs(pool, adapter_id))


def lora_pool_evict_idle(pool, need: int, max_adapters: int, stream=None, planning: bool = False) -> list:
    """Evict idle adapters (earliest load first) until `need` pages are free; returns their ids."""
    ev = np.zeros(max(max_adapters, 1), dtype=np.int32)
    n = ctypes.c_int32(0)
    _check(_load().lora_pool_evict_idle(pool, need, 0 if planning else _stream(stream), _ptr(ev), ctypes.byref(n)))
    return ev[:n.value].tolist()


def lora_adapter_ensure(pool, adapter_id: int, rank: int, A_host: Optional[Sequence], B_host: Optional[Sequence],
                        n_slots: int, max_adapters: int, stream=None, planning: bool = False):
    """Make an adapter resident with one more active request (loading it, after evicting idle
    adapters, if needed).  Returns (page table int32 [n_slots, 2, rank], loaded, evicted ids)."""
    keep = []

    def arr(seq):
        if seq is None:
            return None
        a = (ctypes.c_void_p * n_slots)()
        for i, m in enumerate(seq):
            if m is not None:
                m = np.ascontiguousarray(m, dtype=np.uint16)
                keep.append(m)
                a[i] = m.ctypes.data
        return a

    a_arr, b_arr = arr(A_host), arr(B_host)
    table = np.zeros((n_slots, 2, max(rank, 1)), dtype=np.int32)
    loaded = ctypes.c_int32(0)
    ev = np.zeros(max(max_adapters, 1), dtype=np.int32)
    n = ctypes.c_int32(0)
    st = 0 if planning else _stream(stream)
    _check(_load().lora_adapter_ensure(pool, adapter_id, rank, ctypes.cast(a_arr, ctypes.c_void_p) if a_arr else None,
                                       ctypes.cast(b_arr, ctypes.c_void_p) if b_arr else None, st, _ptr(table),
                                       ctypes.byref(loaded), _ptr(ev), ctypes.byref(n)))
    return table, bool(loaded.value), ev[:n.value].tolist()


def lora_segments_size(pool, T_max: int) -> int:
    n = _load().lora_segments_size(pool, T_max)
    if n < 0:
        raise LoraError(int(n), lora_last_error())
    return int(n)


def lora_segments_init(pool, workspace_dev, workspace_bytes: int, T_max: int) -> lora_segments:
    seg = lora_segments()
    _check(_load().lora_segments_init(pool, _ptr(workspace_dev), workspace_bytes, T_max, ctypes.byref(seg)))
    return seg


def lora_segments_size_group(pool, T_max: int, max_group: int) -> int:
    n = _load().lora_segments_size_group(pool, T_max, max_group)
    if n < 0:
        raise LoraError(int(n), lora_last_error())
    return int(n)


def lora_segments_init_group(pool, workspace_dev, workspace_bytes: int, T_max: int, max_group: int) -> lora_segments:
    seg = lora_segments()
    _check(_load().lora_segments_init_group(pool, _ptr(workspace_dev), workspace_bytes, T_max, max_group,
                                            ctypes.byref(seg)))
    return seg


def lora_segments_build(pool, token_adapter_dev, T: int, seg: lora_segments, stream=None) -> None:
    _check(_load().lora_segments_build(pool, _ptr(token_adapter_dev), T, ctypes.byref(seg), _stream(stream)))


def lora_linear_forward(pool, seg: lora_segments, slot: int, x_dev, W_dev, y_dev, delta_dbg_dev=None,
                        stream=None) -> None:
    _check(_load().lora_linear_forward(pool, ctypes.byref(seg), slot, _ptr(x_dev), _ptr(W_dev), _ptr(y_dev),
                                       _ptr(delta_dbg_dev), _stream(stream)))


def lora_linear_forward_group(pool, seg: lora_segments, slots: Sequence[int], x_dev, W_devs, y_devs,
                              delta_dbg_devs=None, stream=None) -> None:
    """Several slots that read the same x (q, k, v of a layer): one LoRA-delta launch for all."""
    n = len(slots)
    sl = np.ascontiguousarray(slots, dtype=np.int32)
    Ws = (ctypes.c_void_p * n)(*[_ptr(w) for w in W_devs])
    ys = (ctypes.c_void_p * n)(*[_ptr(v) for v in y_devs])
    ds = None if delta_dbg_devs is None else (ctypes.c_void_p * n)(*[_ptr(d) for d in delta_dbg_devs])
    _check(_load().lora_linear_forward_group(pool, ctypes.byref(seg), n, _ptr(sl), _ptr(x_dev),
                                             ctypes.cast(Ws, ctypes.c_void_p), ctypes.cast(ys, ctypes.c_void_p),
                                             ctypes.cast(ds, ctypes.c_void_p) if ds is not None else None,
                                             _stream(stream)))


def lora_status(pool, stream=None) -> None:
    _check(_load().lora_status(pool, _stream(stream)))


def lora_pool_stats(pool) -> dict:
    s = lora_pool_stats_t()
    _load().lora_pool_stats(pool, ctypes.byref(s))
    return {"num_pages": s.num_pages, "free": s.free_pages, "adapter": s.adapter_pages,
            "reserved": s.reserved_pages, "resident_adapters": s.resident_adapters, "max_adapters": s.max_adapters}


def lora_pool_destroy(pool) -> None:
    _load().lora_pool_destroy(pool)


def lora_profile_enable(pool, enable: bool = True) -> None:
    _check(_load().lora_profile_enable(pool, 1 if enable else 0))


def lora_profile_read(pool, reset: bool = True) -> dict:
    """Per kernel kind: launches and summed device ms of the recorded launches."""
    n = len(KINDS)
    launches = np.zeros(n, dtype=np.int64)
    ms = np.zeros(n, dtype=np.float64)
    _check(_load().lora_profile_read(pool, n, _ptr(launches), _ptr(ms), 1 if reset else 0))
    return {k: {"launches": int(launches[i]), "ms": float(ms[i])} for i, k in enumerate(KINDS)}


def lora_linear_forward_noalloc(pool, token_adapter_dev, T: int, slot: int, x_dev, W_dev, y_dev, stream=None) -> None:
    """One projection slot without a caller workspace: the library's static device scratch is used.

    For callers that cannot allocate device memory; at most LORA_NOALLOC_MAX_TOKENS tokens and
    H <= LORA_NOALLOC_MAX_H.  Calls that overlap on the GPU share the scratch and race.
    """
    _check(_load().lora_linear_forward_noalloc(pool, _ptr(token_adapter_dev), T, slot, _ptr(x_dev), _ptr(W_dev),
                                               _ptr(y_dev), _stream(stream)))
