"""GPU parity of the next paths at the bench's full size.

The Llama-3-8B KV workload (10k facts of 12-48 tokens, 1024-d embeddings,
k = 50; "InferScale: GPU-Native KV Injection for Personalized LLM
Serving" serving setting) through the paths beside the plain fused call:
the rotary variants (Section 5.1 under the engines' conventions), the K/V
store in pinned host memory (review Summary: offload to host DRAM) and 64
or 256 concurrent queries over the one store (Section 6.4).  Every injected
element is compared with the float64 oracle (V bit-exact, K within
2^-8|x| + 1e-6) and every other pool row must keep its canary, as in
tests/test_gpu_configs.py.
"""
import dataclasses
import gc
import types

import numpy as np
import pytest
import torch

import oracle
import pre_rope_kv_gb300 as kvi
from tests import kvi_check as kc
from tests import synth

pytestmark = pytest.mark.gpu

K = 50


@pytest.fixture(scope="module")
def b():
    kc.ensure_built()
    built = synth.build_workload(synth.WORKLOADS["llama3_8b_10k"])
    yield built
    del built
    gc.collect()
    torch.cuda.empty_cache()


def _check(b, f, label, ospec=None):
    ids, scores, pos, status = f.results()
    assert status == 0, f"device status {status}"
    orc = kc.oracle_select(b, K)
    kc.check_selection(ids, scores, pos, orc)
    place = kc.placements_from_oracle(orc)
    kc.check_pool_exhaustive(b, place, rope=ospec, label=label)
    kc.check_canaries_by_row(b, place)


def _engine_table(w, positions):
    # an engine's own float32 cos/sin cache, angles computed in float32
    inv = 1.0 / np.power(np.float32(w.rope_theta),
                         np.arange(0, w.head_dim, 2, dtype=np.float32) / np.float32(w.head_dim))
    ang = np.arange(positions, dtype=np.float32)[:, None] * inv.astype(np.float32)[None, :]
    return np.cos(ang).astype(np.float32), np.sin(ang).astype(np.float32)


@pytest.mark.parametrize("variant", ["interleaved", "llama3_scaling", "engine_table"])
def test_rope_variants_full_size(b, variant):
    w = b.w
    if variant == "interleaved":
        spec = kvi.rope(w.rope_theta, kvi.ROPE_PAIR_INTERLEAVED)
        ospec = oracle.rope_spec(w.rope_theta, w.head_dim, oracle.PAIR_INTERLEAVED)
    elif variant == "llama3_scaling":
        ll = (8.0, 1.0, 4.0, 8192.0)
        spec = kvi.rope(w.rope_theta, llama3=ll)
        ospec = oracle.rope_spec(w.rope_theta, w.head_dim, llama3=ll)
    else:
        c, s = _engine_table(w, b.max_blocks * w.block_size)
        spec = kvi.rope(cos_table=c, sin_table=s, table_id=777001)
        ospec = oracle.rope_spec(w.rope_theta, w.head_dim, cos_table=c, sin_table=s)
    synth.fill_canary(b.pool)
    f = kc.Fused(b, K, rope=spec)
    f()
    _check(b, f, f"llama3_8b_10k k={K} {variant}", ospec)


def test_host_resident_store_full_size(b):
    # the 39 GB K/V store in pinned host memory, read in place by the inject
    # kernel over the host link
    host = torch.empty(b.kv.shape, dtype=b.kv.dtype, pin_memory=True)
    host.copy_(b.kv)
    torch.cuda.synchronize()
    g = kc.geometry_of(b.w)
    st = b.stores[0]
    view = kvi.store_view(g, host, st.emb, st.fact_start, st.fact_len, n_tokens=b.kv.shape[2],
                          kv_host=True)
    synth.fill_canary(b.pool)
    f = kc.Fused(b, K)
    f.d_views = kc.device_views([view])
    f()
    _check(b, f, f"llama3_8b_10k k={K} host-resident K/V")
    del host


@pytest.mark.parametrize("R", [64, 256])
def test_shared_store_queries_full_size(b, R):
    # R requests over the one 10k-fact store: tensor-core coarse scores (64:
    # the cluster form; 256: facts on M), exact rescoring, and the R
    # injections into one pool
    w = b.w
    st = b.stores[0]
    view = kc.views_of(b)[0]
    rng = np.random.default_rng(w.seed + 31)
    q_np = synth.query_rows(rng, R, w.embed_dim)
    q = torch.from_numpy(q_np).cuda()
    tl = int(b.table_lens[0])
    L, H, D, B = w.layers, w.kv_heads, w.head_dim, w.block_size
    pool = torch.empty((L, 2, R * tl, B, H, D), dtype=torch.bfloat16, device="cuda")
    synth.fill_canary(pool)
    tables = rng.permutation(R * tl).astype(np.int32).reshape(R, tl)
    start = np.full(R, int(b.start_pos[0]), np.int32)
    ids = torch.empty((R, K), dtype=torch.int32, device="cuda")
    sc = torch.empty((R, K), dtype=torch.float32, device="cuda")
    pos = torch.empty((R, K), dtype=torch.int32, device="cuda")
    ws = torch.empty(kvi.kvi_workspace_bytes_shared(R, w.n_facts, K), dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    cache = kvi.paged_cache([pool[l] for l in range(L)], B)
    kvi.kvi_retrieve_and_inject_shared(
        view, R, q, K, torch.from_numpy(start).cuda(), torch.from_numpy(tables).cuda(),
        torch.full((R,), tl, dtype=torch.int32, device="cuda"), tl, cache, kvi.rope(w.rope_theta),
        ids, sc, pos, ws, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    # the same requests as R separate stores of one workload, for the checks
    sb = types.SimpleNamespace(
        w=dataclasses.replace(w, requests=R), kv=b.kv, stores=[st] * R, queries_np=q_np,
        start_pos=start, block_tables=tables, table_lens=np.full(R, tl, np.int32), pool=pool,
        num_blocks=R * tl)
    orc = []
    for r in range(R):
        s = oracle.scores(q_np[r], st.emb_np)
        sel = oracle.topk(s, K)
        p_, T = oracle.place(sel, st.len_np, int(start[r]))
        orc.append((s, sel, p_, T))
    kc.check_selection(ids.cpu().numpy(), sc.cpu().numpy(), pos.cpu().numpy(), orc)
    place = kc.placements_from_oracle(orc)
    kc.check_pool_exhaustive(sb, place, label=f"llama3_8b_10k shared store, {R} queries, k={K}")
    kc.check_canaries_by_row(sb, place)
    del pool
