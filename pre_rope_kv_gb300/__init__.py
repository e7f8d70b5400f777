"""GB300 (sm_103a) retrieve-and-inject library for pre-RoPE KV facts.

Serving-time path of "InferScale: GPU-Native KV Injection for Personalized
LLM Serving": exact top-k retrieval of memory facts by embedding similarity
(Figure 2 caption), Chunked RoPE rotation of their pre-RoPE keys to the
prompt positions they take (Section 5.1 / Theorem 6), and scatter-copy of K/V
into a vLLM-style paged KV cache through a block table (Section 3.4).

The compute is in ``libkvi.so`` (hand-written CUDA for sm_103a, C ABI in
``include/kvi.h``); this package is a ctypes binding with the same function
names.  Build the library with ``pre_rope_kv_gb300.build.build()``.
"""
from ._binding import (  # noqa: F401
    EXPORTED_SYMBOLS, ERR_CAPACITY, ERR_CUDA, ERR_INVALID_ARG, ERR_OUT_OF_RANGE, ERR_TIMEOUT,
    LIB_PATH, MAX_REQUESTS,
    MAX_INJECT_FACTS, MAX_K, MAX_LAYERS, OK, Geometry, KviError, PagedCache, StoreSizes,
    StoreView, geometry, kvi_inject_paged, kvi_last_error, kvi_place, kvi_prepare_rope,
    kvi_retrieve_and_inject, kvi_retrieve_topk, kvi_retrieve_topk_noalloc, kvi_status_str,
    kvi_store_layout, NOALLOC_MAX_FACTS,
    kvi_trace_stages, kvi_workspace_bytes, load_library, pack_store_views, paged_cache,
    store_view, Rope, rope, kvi_prepare_rope_ex, kvi_inject_paged_ex, kvi_retrieve_and_inject_ex,
    ROPE_PAIR_HALF, ROPE_PAIR_INTERLEAVED, ROPE_SCALE_NONE, ROPE_SCALE_LLAMA3,
    MAX_SHARED_QUERIES, kvi_workspace_bytes_shared, kvi_retrieve_topk_shared,
    kvi_retrieve_and_inject_shared, STORE_KV_HOST, Plan, kvi_plan_create_fused,
    ERR_IO, StoreFileInfo, kvi_store_save, kvi_store_file_info_read, kvi_store_load, load_store,
    MAX_GRAPH_DEGREE, MAX_GRAPH_BEAM, MAX_GRAPH_FRONTIER, GraphSearchParams,
    kvi_graph_build_workspace_bytes, kvi_graph_build, kvi_graph_search_workspace_bytes,
    kvi_graph_search, graph_search_params, kvi_graph_retrieve_and_inject_workspace_bytes,
    kvi_graph_retrieve_and_inject, kvi_selftest_bounded_wait, open_library, use_library,
    kvi_debug_stall_scorer_row, kvi_debug_stall_coarse_chunk, kvi_selftest_stream_read,
)
