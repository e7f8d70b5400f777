"""ctypes binding of libkvi (include/kvi.h): argument marshalling only.

Every function here has the name of the C entry point it calls and does no
arithmetic of the method: it turns torch tensors into device pointers,
Python numbers into C scalars, and raises KviError when the library returns
a non-zero status.  All compute runs in libkvi's CUDA kernels.  There is no
fallback: if the library is missing or fails to load, the import of this
module's functions raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Sequence

from . import build as _build

LIB_PATH = _build.LIB_PATH

OK = 0
ERR_INVALID_ARG = 1
ERR_OUT_OF_RANGE = 2
ERR_CAPACITY = 3
ERR_CUDA = 4
ERR_TIMEOUT = 5
ERR_IO = 6
MAX_REQUESTS = 4096

MAX_LAYERS = 128
MAX_K = 256
MAX_INJECT_FACTS = 4096

EXPORTED_SYMBOLS = (
    "kvi_store_layout", "kvi_prepare_rope", "kvi_workspace_bytes", "kvi_retrieve_topk",
    "kvi_place", "kvi_inject_paged", "kvi_retrieve_and_inject", "kvi_trace_stages",
    "kvi_status_str", "kvi_last_error", "kvi_retrieve_topk_noalloc", "kvi_prepare_rope_ex",
    "kvi_inject_paged_ex", "kvi_retrieve_and_inject_ex", "kvi_workspace_bytes_shared",
    "kvi_retrieve_topk_shared", "kvi_retrieve_and_inject_shared", "kvi_plan_create_fused",
    "kvi_plan_launch", "kvi_plan_destroy", "kvi_plan_create_fused_io", "kvi_store_save",
    "kvi_store_file_info_read", "kvi_store_load", "kvi_graph_build_workspace_bytes",
    "kvi_graph_build", "kvi_graph_search_workspace_bytes", "kvi_graph_search",
    "kvi_graph_retrieve_and_inject_workspace_bytes", "kvi_graph_retrieve_and_inject",
    "kvi_selftest_bounded_wait", "kvi_selftest_stream_read",
)
MAX_GRAPH_DEGREE = 128
MAX_GRAPH_BEAM = 256
MAX_GRAPH_FRONTIER = 512
MAX_SHARED_QUERIES = 256
NOALLOC_MAX_FACTS = 65536


class KviError(RuntimeError):
    def __init__(self, status: int, where: str, message: str):
        super().__init__(f"{where}: status {status} ({message})")
        self.status = status


class Geometry(ctypes.Structure):
    _fields_ = [("layers", ctypes.c_int32), ("kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("embed_dim", ctypes.c_int32)]


STORE_KV_HOST = 1


class StoreView(ctypes.Structure):
    _fields_ = [("g", Geometry), ("n_facts", ctypes.c_int64), ("n_tokens", ctypes.c_int64),
                ("kv", ctypes.c_void_p), ("emb", ctypes.c_void_p),
                ("fact_start", ctypes.c_void_p), ("fact_len", ctypes.c_void_p),
                ("flags", ctypes.c_uint32), ("reserved", ctypes.c_uint32)]


class StoreSizes(ctypes.Structure):
    _fields_ = [("n_tokens", ctypes.c_int64), ("kv_bytes", ctypes.c_size_t),
                ("emb_bytes", ctypes.c_size_t), ("offsets_bytes", ctypes.c_size_t)]


ROPE_PAIR_HALF, ROPE_PAIR_INTERLEAVED = 0, 1
ROPE_SCALE_NONE, ROPE_SCALE_LLAMA3 = 0, 1


class Rope(ctypes.Structure):
    """kvi_rope: rotary variant (pairing, Llama 3.1 scaling, caller table)."""
    _fields_ = [("theta", ctypes.c_double), ("pairing", ctypes.c_int32),
                ("scaling", ctypes.c_int32), ("factor", ctypes.c_double),
                ("low_freq_factor", ctypes.c_double), ("high_freq_factor", ctypes.c_double),
                ("original_max_positions", ctypes.c_double),
                ("cos_table", ctypes.c_void_p), ("sin_table", ctypes.c_void_p),
                ("table_positions", ctypes.c_int32), ("table_id", ctypes.c_int64)]


class StoreFileInfo(ctypes.Structure):
    _fields_ = [("g", Geometry), ("n_facts", ctypes.c_int64), ("n_tokens", ctypes.c_int64),
                ("kv_bytes", ctypes.c_size_t), ("emb_bytes", ctypes.c_size_t)]


class GraphSearchParams(ctypes.Structure):
    _fields_ = [("beam", ctypes.c_int32), ("width", ctypes.c_int32), ("max_iters", ctypes.c_int32),
                ("n_seeds", ctypes.c_int32)]


class PagedCache(ctypes.Structure):
    _fields_ = [("layer_base", ctypes.POINTER(ctypes.c_void_p)), ("layers", ctypes.c_int32),
                ("num_blocks", ctypes.c_int32), ("block_size", ctypes.c_int32)]


_lib = None


def load_library(path: str | None = None):
    """Load libkvi.so (built by pre_rope_kv_gb300.build.build())."""
    global _lib
    if _lib is not None:
        return _lib
    _lib = open_library(path or LIB_PATH)
    return _lib


def open_library(path: str):
    """Load and configure the library at `path` without making it the one
    the functions of this module call (see use_library)."""
    if not os.path.exists(path):
        raise RuntimeError(f"libkvi is not built ({path} missing): run pre_rope_kv_gb300.build.build()")
    lib = ctypes.CDLL(path)
    P, i32, i64, f64, sz = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_double,
                           ctypes.c_size_t)
    S = ctypes.c_int
    sig = {
        "kvi_store_layout": (S, [ctypes.POINTER(Geometry), P, i64, P, ctypes.POINTER(StoreSizes)]),
        "kvi_prepare_rope": (S, [f64, i32, i32]),
        "kvi_workspace_bytes": (sz, [i32, i64, i32]),
        "kvi_retrieve_topk": (S, [ctypes.POINTER(StoreView), P, i32, P, P, P, sz, P, P]),
        "kvi_place": (S, [ctypes.POINTER(StoreView), P, i32, i32, P, P, P]),
        "kvi_inject_paged": (S, [ctypes.POINTER(StoreView), P, P, i32, P, i32,
                                 ctypes.POINTER(PagedCache), f64, P, P]),
        "kvi_retrieve_and_inject": (S, [ctypes.POINTER(Geometry), i32, P, i64, P, i32, P, P, P,
                                        i32, ctypes.POINTER(PagedCache), f64, P, P, P, P, sz,
                                        P, P]),
        "kvi_trace_stages": (S, [P, i32]),
        "kvi_prepare_rope_ex": (S, [ctypes.POINTER(Rope), i32, i32]),
        "kvi_workspace_bytes_shared": (sz, [i32, i64, i32]),
        "kvi_plan_create_fused": (S, [P, ctypes.POINTER(Geometry), i32, P, i64, P, i32, P, P, P, i32,
                                      ctypes.POINTER(PagedCache), ctypes.POINTER(Rope), P, P, P, P,
                                      sz, P]),
        "kvi_plan_create_fused_io": (S, [P, ctypes.POINTER(Geometry), i32, P, i64, P, i32, P, P, P,
                                         i32, ctypes.POINTER(PagedCache), ctypes.POINTER(Rope), P, P,
                                         P, P, sz, P, P, P, sz, P, P, sz]),
        "kvi_plan_launch": (S, [P, P]),
        "kvi_plan_destroy": (S, [P]),
        "kvi_retrieve_topk_shared": (S, [ctypes.POINTER(StoreView), i32, P, i32, P, P, P, sz, P, P]),
        "kvi_retrieve_and_inject_shared": (S, [ctypes.POINTER(StoreView), i32, P, i32, P, P, P, i32,
                                               ctypes.POINTER(PagedCache), ctypes.POINTER(Rope), P,
                                               P, P, P, sz, P, P]),
        "kvi_inject_paged_ex": (S, [ctypes.POINTER(StoreView), P, P, i32, P, i32,
                                    ctypes.POINTER(PagedCache), ctypes.POINTER(Rope), P, P]),
        "kvi_retrieve_and_inject_ex": (S, [ctypes.POINTER(Geometry), i32, P, i64, P, i32, P, P,
                                           P, i32, ctypes.POINTER(PagedCache),
                                           ctypes.POINTER(Rope), P, P, P, P, sz, P, P]),
        "kvi_retrieve_topk_noalloc": (S, [ctypes.POINTER(StoreView), P, i32, P, P, P, P]),
        "kvi_store_save": (S, [ctypes.c_char_p, ctypes.POINTER(StoreView)]),
        "kvi_store_file_info_read": (S, [ctypes.c_char_p, ctypes.POINTER(StoreFileInfo)]),
        "kvi_store_load": (S, [ctypes.c_char_p, P, P, P, P, ctypes.c_uint32]),
        "kvi_graph_build_workspace_bytes": (sz, [i64, i32]),
        "kvi_graph_build": (S, [ctypes.POINTER(StoreView), i32, P, P, sz, P, P]),
        "kvi_graph_search_workspace_bytes": (sz, [i32, i64]),
        "kvi_graph_search": (S, [ctypes.POINTER(StoreView), P, i32, i32, P, P,
                                 ctypes.POINTER(GraphSearchParams), i32, P, P, P, P, P, sz, P, P]),
        "kvi_graph_retrieve_and_inject_workspace_bytes": (sz, [i32, i64, i32, i32]),
        "kvi_graph_retrieve_and_inject": (S, [ctypes.POINTER(StoreView), P, i32, i32, P, P,
                                              ctypes.POINTER(GraphSearchParams), i32, P, P, P, i32,
                                              ctypes.POINTER(PagedCache), ctypes.POINTER(Rope), P, P,
                                              P, P, sz, P, P]),
        "kvi_selftest_bounded_wait": (S, [ctypes.c_uint64, P, P, P]),
        "kvi_selftest_stream_read": (S, [P, sz, i32, P, P]),
        "kvi_status_str": (ctypes.c_char_p, [S]),
        "kvi_last_error": (ctypes.c_char_p, []),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if hasattr(lib, "kvi_debug_stall_scorer_row"):  # debug build only
        lib.kvi_debug_stall_scorer_row.restype = S
        lib.kvi_debug_stall_scorer_row.argtypes = [i64]
        lib.kvi_debug_stall_coarse_chunk.restype = S
        lib.kvi_debug_stall_coarse_chunk.argtypes = [ctypes.c_int32, ctypes.c_int32]
    return lib


class use_library:
    """Context manager: the functions of this module call `lib` (from
    open_library, e.g. the debug build) inside the block."""

    def __init__(self, lib):
        self.lib = lib
        self.saved = None

    def __enter__(self):
        global _lib
        self.saved = _lib
        _lib = self.lib
        return self.lib

    def __exit__(self, *exc):
        global _lib
        _lib = self.saved
        return False


def kvi_selftest_stream_read(src_ptr: int, nbytes: int, ctas_per_sm: int, sum_out, stream=None) -> None:
    """Diagnostic: the SMs read nbytes at src_ptr (device or pinned host
    memory); one checksum goes to sum_out (a device uint64 tensor)."""
    _check(load_library().kvi_selftest_stream_read(int(src_ptr), int(nbytes), int(ctas_per_sm),
                                                   _ptr(sum_out), _stream(stream)),
           "kvi_selftest_stream_read")


def kvi_debug_stall_scorer_row(row: int) -> None:
    """Debug build only (include/kvi_debug.h): make the scoring kernel skip
    the copy of one flat row, so that a bounded wait runs out."""
    lib = load_library()
    if not hasattr(lib, "kvi_debug_stall_scorer_row"):
        raise RuntimeError("kvi_debug_stall_scorer_row needs the debug build (build(debug=True))")
    _check(lib.kvi_debug_stall_scorer_row(int(row)), "kvi_debug_stall_scorer_row")


def kvi_debug_stall_coarse_chunk(cta: int, chunk: int) -> None:
    """Debug build only (include/kvi_debug.h): make the shared-store path's
    tensor-core kernel load nothing for K chunk `chunk` in CTA `cta`, so
    that the waits on that stage run out (cta < 0: off)."""
    lib = load_library()
    if not hasattr(lib, "kvi_debug_stall_coarse_chunk"):
        raise RuntimeError("kvi_debug_stall_coarse_chunk needs the debug build (build(debug=True))")
    _check(lib.kvi_debug_stall_coarse_chunk(int(cta), int(chunk)), "kvi_debug_stall_coarse_chunk")


def _check(status: int, where: str):
    if status != OK:
        lib = load_library()
        raise KviError(status, where, lib.kvi_last_error().decode() or
                       lib.kvi_status_str(status).decode())


def _ptr(t) -> int | None:
    """Device (or host) address of a tensor, or None."""
    if t is None:
        return None
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


# ----------------------------------------------------------------- helpers

def geometry(layers: int, kv_heads: int, head_dim: int, embed_dim: int) -> Geometry:
    return Geometry(layers, kv_heads, head_dim, embed_dim)


def store_view(g: Geometry, kv, emb, fact_start, fact_len, n_tokens: int | None = None,
               kv_host: bool = False) -> StoreView:
    """Describe a store held in torch tensors (kv bf16 [L][2][T][H][D],
    emb float32 [N][E], fact_start int64 [N], fact_len int32 [N]).
    kv_host: kv is a pinned host tensor the GPU reads in place."""
    n_facts = (emb.shape[0] if emb is not None else fact_len.shape[0])
    T = n_tokens if n_tokens is not None else (kv.shape[2] if kv is not None else 0)
    return StoreView(g, n_facts, T, _ptr(kv), _ptr(emb), _ptr(fact_start), _ptr(fact_len),
                     STORE_KV_HOST if kv_host else 0, 0)


def pack_store_views(views: Sequence[StoreView]) -> bytes:
    """Bytes of an array of kvi_store_view, to copy into device memory for
    kvi_retrieve_and_inject."""
    arr = (StoreView * len(views))(*views)
    return ctypes.string_at(ctypes.addressof(arr), ctypes.sizeof(arr))


class _Cache:
    """Keeps the host array of layer pointers alive next to the struct."""

    def __init__(self, layer_tensors, block_size: int):
        ptrs = [t.data_ptr() for t in layer_tensors]
        self._arr = (ctypes.c_void_p * len(ptrs))(*ptrs)
        nb = layer_tensors[0].shape[1]
        self.struct = PagedCache(ctypes.cast(self._arr, ctypes.POINTER(ctypes.c_void_p)),
                                 len(ptrs), nb, block_size)
        self.layer_tensors = list(layer_tensors)


def paged_cache(layer_tensors, block_size: int) -> _Cache:
    """Describe a paged pool: one bf16 tensor [2][num_blocks][B][H][D] per layer."""
    return _Cache(layer_tensors, block_size)


# ------------------------------------------------------------- entry points

def kvi_store_layout(g: Geometry, fact_len):
    """Host-only CSR layout: returns (token_offsets list[int], StoreSizes)."""
    lib = load_library()
    n = len(fact_len)
    lens = (ctypes.c_int32 * max(n, 1))(*[int(x) for x in fact_len])
    offs = (ctypes.c_int64 * (n + 1))()
    sizes = StoreSizes()
    _check(lib.kvi_store_layout(ctypes.byref(g), lens, n, offs, ctypes.byref(sizes)),
           "kvi_store_layout")
    return list(offs), sizes


def kvi_prepare_rope(rope_theta: float, head_dim: int, max_position: int) -> None:
    _check(load_library().kvi_prepare_rope(float(rope_theta), int(head_dim), int(max_position)),
           "kvi_prepare_rope")


def rope(theta: float = 0.0, pairing: int = ROPE_PAIR_HALF, llama3=None, cos_table=None,
         sin_table=None, table_id: int = 0) -> Rope:
    """A kvi_rope.  llama3 = (factor, low_freq_factor, high_freq_factor,
    original_max_positions).  cos_table / sin_table: contiguous host float32
    arrays [positions][D/2] (numpy or CPU torch), kept alive by the caller for
    the call that first uses table_id."""
    r = Rope()
    r.theta = float(theta)
    r.pairing = int(pairing)
    if llama3 is not None:
        r.scaling = ROPE_SCALE_LLAMA3
        r.factor, r.low_freq_factor, r.high_freq_factor, r.original_max_positions = map(float, llama3)
    if cos_table is not None:
        r.cos_table = _host_ptr(cos_table)
        r.sin_table = _host_ptr(sin_table)
        r.table_positions = int(cos_table.shape[0])
        r.table_id = int(table_id)
    return r


def _host_ptr(a) -> int:
    if hasattr(a, "data_ptr"):
        return a.data_ptr()
    return a.ctypes.data


def kvi_prepare_rope_ex(spec: Rope, head_dim: int, max_position: int) -> None:
    _check(load_library().kvi_prepare_rope_ex(ctypes.byref(spec), int(head_dim), int(max_position)),
           "kvi_prepare_rope_ex")


def kvi_workspace_bytes(R: int, max_facts: int, k: int) -> int:
    return int(load_library().kvi_workspace_bytes(int(R), int(max_facts), int(k)))


def kvi_retrieve_topk(store: StoreView, query, k: int, ids, scores, ws, status,
                      stream=None) -> None:
    _check(load_library().kvi_retrieve_topk(
        ctypes.byref(store), _ptr(query), int(k), _ptr(ids), _ptr(scores), _ptr(ws),
        ws.numel() * ws.element_size(), _ptr(status), _stream(stream)), "kvi_retrieve_topk")


def kvi_retrieve_topk_noalloc(store: StoreView, query, k: int, ids, scores, status,
                              stream=None) -> None:
    """kvi_retrieve_topk without a workspace: the scratch is a fixed array of
    the library (see include/kvi.h for who needs this and its limits)."""
    _check(load_library().kvi_retrieve_topk_noalloc(
        ctypes.byref(store), _ptr(query), int(k), _ptr(ids), _ptr(scores), _ptr(status),
        _stream(stream)), "kvi_retrieve_topk_noalloc")


def kvi_place(store: StoreView, ids, n: int, start: int, pos, status=None, stream=None) -> None:
    _check(load_library().kvi_place(ctypes.byref(store), _ptr(ids), int(n), int(start), _ptr(pos),
                                    _ptr(status), _stream(stream)), "kvi_place")


def kvi_inject_paged(store: StoreView, fact_ids, start_pos, n: int, block_table, table_len: int,
                     cache: _Cache, rope_theta: float, status=None, stream=None) -> None:
    _check(load_library().kvi_inject_paged(
        ctypes.byref(store), _ptr(fact_ids), _ptr(start_pos), int(n), _ptr(block_table),
        int(table_len), ctypes.byref(cache.struct), float(rope_theta), _ptr(status),
        _stream(stream)), "kvi_inject_paged")


def kvi_inject_paged_ex(store: StoreView, fact_ids, start_pos, n: int, block_table, table_len: int,
                        cache: _Cache, spec: Rope, status=None, stream=None) -> None:
    _check(load_library().kvi_inject_paged_ex(
        ctypes.byref(store), _ptr(fact_ids), _ptr(start_pos), int(n), _ptr(block_table),
        int(table_len), ctypes.byref(cache.struct), ctypes.byref(spec), _ptr(status),
        _stream(stream)), "kvi_inject_paged_ex")


def kvi_retrieve_and_inject_ex(g: Geometry, R: int, stores_dev, max_facts: int, queries, k: int,
                               start_pos, block_tables, table_lens, max_blocks: int, cache: _Cache,
                               spec: Rope, ids, scores, pos, ws, status=None, stream=None) -> None:
    _check(load_library().kvi_retrieve_and_inject_ex(
        ctypes.byref(g), int(R), _ptr(stores_dev), int(max_facts), _ptr(queries), int(k),
        _ptr(start_pos), _ptr(block_tables), _ptr(table_lens), int(max_blocks),
        ctypes.byref(cache.struct), ctypes.byref(spec), _ptr(ids), _ptr(scores), _ptr(pos),
        _ptr(ws), ws.numel() * ws.element_size(), _ptr(status), _stream(stream)),
        "kvi_retrieve_and_inject_ex")


def kvi_workspace_bytes_shared(R: int, n_facts: int, k: int) -> int:
    return int(load_library().kvi_workspace_bytes_shared(int(R), int(n_facts), int(k)))


def kvi_retrieve_topk_shared(store: StoreView, R: int, queries, k: int, ids, scores, ws,
                             status=None, stream=None) -> None:
    _check(load_library().kvi_retrieve_topk_shared(
        ctypes.byref(store), int(R), _ptr(queries), int(k), _ptr(ids), _ptr(scores), _ptr(ws),
        ws.numel() * ws.element_size(), _ptr(status), _stream(stream)), "kvi_retrieve_topk_shared")


def kvi_retrieve_and_inject_shared(store: StoreView, R: int, queries, k: int, start_pos,
                                   block_tables, table_lens, max_blocks: int, cache: _Cache,
                                   spec: Rope, ids, scores, pos, ws, status=None,
                                   stream=None) -> None:
    _check(load_library().kvi_retrieve_and_inject_shared(
        ctypes.byref(store), int(R), _ptr(queries), int(k), _ptr(start_pos), _ptr(block_tables),
        _ptr(table_lens), int(max_blocks), ctypes.byref(cache.struct), ctypes.byref(spec),
        _ptr(ids), _ptr(scores), _ptr(pos), _ptr(ws), ws.numel() * ws.element_size(),
        _ptr(status), _stream(stream)), "kvi_retrieve_and_inject_shared")


class Plan:
    """A fused call recorded once (kvi_plan_create_fused) and replayed with
    launch(); the tensors it was created with must stay alive."""

    def __init__(self, handle: int, keep):
        self.handle = handle
        self._keep = keep

    def launch(self, stream=None) -> None:
        _check(load_library().kvi_plan_launch(self.handle, _stream(stream)), "kvi_plan_launch")

    def close(self) -> None:
        if self.handle:
            _check(load_library().kvi_plan_destroy(self.handle), "kvi_plan_destroy")
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def kvi_plan_create_fused(g: Geometry, R: int, stores_dev, max_facts: int, queries, k: int,
                          start_pos, block_tables, table_lens, max_blocks: int, cache: _Cache,
                          spec: Rope, ids, scores, pos, ws, status=None, io=None) -> Plan:
    """io = (h_in, d_in, d_out, h_out): pinned host and device byte tensors
    whose copies the plan records around the fused call (optional)."""
    h = ctypes.c_void_p()
    lib = load_library()
    common = (ctypes.byref(h), ctypes.byref(g), int(R), _ptr(stores_dev), int(max_facts), _ptr(queries),
              int(k), _ptr(start_pos), _ptr(block_tables), _ptr(table_lens), int(max_blocks),
              ctypes.byref(cache.struct), ctypes.byref(spec), _ptr(ids), _ptr(scores), _ptr(pos),
              _ptr(ws), ws.numel() * ws.element_size(), _ptr(status))
    if io is None:
        _check(lib.kvi_plan_create_fused(*common), "kvi_plan_create_fused")
    else:
        h_in, d_in, d_out, h_out = io
        _check(lib.kvi_plan_create_fused_io(*common, _ptr(h_in), _ptr(d_in), d_in.numel(),
                                            _ptr(d_out), _ptr(h_out), d_out.numel()),
               "kvi_plan_create_fused_io")
    return Plan(h.value, (g, stores_dev, queries, start_pos, block_tables, table_lens, cache, spec,
                          ids, scores, pos, ws, status, io))


def kvi_retrieve_and_inject(g: Geometry, R: int, stores_dev, max_facts: int, queries, k: int,
                            start_pos, block_tables, table_lens, max_blocks: int, cache: _Cache,
                            rope_theta: float, ids, scores, pos, ws, status=None,
                            stream=None) -> None:
    _check(load_library().kvi_retrieve_and_inject(
        ctypes.byref(g), int(R), _ptr(stores_dev), int(max_facts), _ptr(queries), int(k),
        _ptr(start_pos), _ptr(block_tables), _ptr(table_lens), int(max_blocks),
        ctypes.byref(cache.struct), float(rope_theta), _ptr(ids), _ptr(scores), _ptr(pos),
        _ptr(ws), ws.numel() * ws.element_size(), _ptr(status), _stream(stream)),
        "kvi_retrieve_and_inject")


def kvi_store_save(path: str, store: StoreView) -> None:
    lib = load_library()
    _check(lib.kvi_store_save(os.fsencode(path), ctypes.byref(store)), "kvi_store_save")


def kvi_store_file_info_read(path: str) -> StoreFileInfo:
    lib = load_library()
    info = StoreFileInfo()
    _check(lib.kvi_store_file_info_read(os.fsencode(path), ctypes.byref(info)),
           "kvi_store_file_info_read")
    return info


def kvi_store_load(path: str, kv, emb, fact_start, fact_len, kv_host: bool = False) -> None:
    lib = load_library()
    _check(lib.kvi_store_load(os.fsencode(path), _ptr(kv), _ptr(emb), _ptr(fact_start),
                              _ptr(fact_len), STORE_KV_HOST if kv_host else 0), "kvi_store_load")


def load_store(path: str, kv_host: bool = False):
    """Allocate torch buffers for the store file at path and load it:
    returns (Geometry, kv, emb, fact_start, fact_len); kv is a pinned host
    tensor when kv_host, else on the current CUDA device."""
    import torch
    info = kvi_store_file_info_read(path)
    g = info.g
    shape = (g.layers, 2, info.n_tokens, g.kv_heads, g.head_dim)
    if kv_host:
        kv = torch.empty(shape, dtype=torch.bfloat16).pin_memory()
    else:
        kv = torch.empty(shape, dtype=torch.bfloat16, device="cuda")
    emb = torch.empty((info.n_facts, g.embed_dim), dtype=torch.float32, device="cuda")
    fs = torch.empty(info.n_facts, dtype=torch.int64, device="cuda")
    fl = torch.empty(info.n_facts, dtype=torch.int32, device="cuda")
    kvi_store_load(path, kv, emb, fs, fl, kv_host=kv_host)
    return Geometry(g.layers, g.kv_heads, g.head_dim, g.embed_dim), kv, emb, fs, fl


def kvi_graph_build_workspace_bytes(n_facts: int, degree: int) -> int:
    return load_library().kvi_graph_build_workspace_bytes(int(n_facts), int(degree))


def kvi_graph_build(store: StoreView, degree: int, graph, ws, status=None, stream=None) -> None:
    lib = load_library()
    nb = ws.numel() * ws.element_size()
    _check(lib.kvi_graph_build(ctypes.byref(store), int(degree), _ptr(graph), _ptr(ws), nb,
                               _ptr(status), _stream(stream)), "kvi_graph_build")


def kvi_graph_search_workspace_bytes(R: int, n_facts: int) -> int:
    return load_library().kvi_graph_search_workspace_bytes(int(R), int(n_facts))


def graph_search_params(beam: int = 64, width: int = 1, max_iters: int = 1000,
                        n_seeds: int = 64) -> GraphSearchParams:
    return GraphSearchParams(int(beam), int(width), int(max_iters), int(n_seeds))


def kvi_graph_search(store: StoreView, graph, degree: int, R: int, queries, seeds,
                     params: GraphSearchParams, k: int, ids, scores, ws, count=None, stats=None,
                     status=None, stream=None) -> None:
    lib = load_library()
    nb = ws.numel() * ws.element_size()
    _check(lib.kvi_graph_search(ctypes.byref(store), _ptr(graph), int(degree), int(R),
                                _ptr(queries), _ptr(seeds), ctypes.byref(params), int(k),
                                _ptr(ids), _ptr(scores), _ptr(count), _ptr(stats), _ptr(ws), nb,
                                _ptr(status), _stream(stream)), "kvi_graph_search")


def kvi_graph_retrieve_and_inject_workspace_bytes(R: int, n_facts: int, beam: int, k: int) -> int:
    return load_library().kvi_graph_retrieve_and_inject_workspace_bytes(int(R), int(n_facts),
                                                                        int(beam), int(k))


def kvi_graph_retrieve_and_inject(store: StoreView, graph, degree: int, R: int, queries, seeds,
                                  params: GraphSearchParams, k: int, start_pos, block_tables,
                                  table_lens, max_blocks: int, cache, rope: Rope, ids, scores, pos,
                                  ws, status=None, stream=None) -> None:
    lib = load_library()
    c = cache.struct if hasattr(cache, "struct") else cache
    _check(lib.kvi_graph_retrieve_and_inject(
        ctypes.byref(store), _ptr(graph), int(degree), int(R), _ptr(queries), _ptr(seeds),
        ctypes.byref(params), int(k), _ptr(start_pos), _ptr(block_tables), _ptr(table_lens),
        int(max_blocks), ctypes.byref(c), ctypes.byref(rope), _ptr(ids), _ptr(scores), _ptr(pos),
        _ptr(ws), ws.numel() * ws.element_size(), _ptr(status), _stream(stream)),
        "kvi_graph_retrieve_and_inject")


def kvi_selftest_bounded_wait(limit_ns: int, status, elapsed_ns=None, stream=None) -> None:
    _check(load_library().kvi_selftest_bounded_wait(int(limit_ns), _ptr(status), _ptr(elapsed_ns),
                                                    _stream(stream)), "kvi_selftest_bounded_wait")


def kvi_trace_stages(events) -> None:
    """events: three torch.cuda.Event (enable_timing=True), or [] to stop."""
    lib = load_library()
    if not events:
        _check(lib.kvi_trace_stages(None, 0), "kvi_trace_stages")
        return
    handles = (ctypes.c_void_p * 3)(*[e.cuda_event for e in events])
    _check(lib.kvi_trace_stages(handles, 3), "kvi_trace_stages")


def kvi_status_str(status: int) -> str:
    return load_library().kvi_status_str(int(status)).decode()


def kvi_last_error() -> str:
    return load_library().kvi_last_error().decode()
