"""GPU parity with the K/V store in host memory (KVI_STORE_KV_HOST).

"InferScale: GPU-Native KV Injection for Personalized LLM Serving" keeps a
store that outgrows HBM in host DRAM at the cost of a few milliseconds of
TTFT (review Summary).  Here kv is a pinned host tensor that the inject
kernel reads in place over the host link; embeddings and extents stay in
device memory.  Same bar as the device path: ids, positions and V bits
exact, K within 2^-8|x| + 1e-6 of the float64 oracle.
"""
import numpy as np
import pytest
import torch

import oracle
import pre_rope_kv_gb300 as kvi
from tests import kvi_check as kc
from tests import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    kc.ensure_built()


def W(**kw):
    base = dict(name="host", layers=2, kv_heads=4, head_dim=128, rope_theta=5e5, block_size=16,
                n_facts=400, len_lo=1, len_hi=40, len_dist="uniform", embed_dim=256, requests=1,
                k=25, start=3, start_hi=0, seed=800, store="dense")
    base.update(kw)
    return synth.Workload(**base)


def host_views(b, which):
    """Views of b's stores with kv in pinned host memory for requests in `which`."""
    g = kc.geometry_of(b.w)
    kv_host = b.kv.cpu().pin_memory()
    views = []
    for r, st in enumerate(b.stores):
        host = r in which
        views.append(kvi.store_view(g, kv_host if host else b.kv, st.emb, st.fact_start, st.fact_len,
                                    n_tokens=b.kv.shape[2], kv_host=host))
    return views, kv_host


@pytest.mark.parametrize("pairing", [0, 1])
def test_fused_with_host_store(pairing):
    w = W(seed=801 + pairing)
    b = synth.build_workload(w)
    views, keep = host_views(b, {0})
    f = kc.Fused(b, rope=kvi.rope(w.rope_theta, pairing))
    f.d_views = kc.device_views(views)
    f()
    ids, scores, pos, status = f.results()
    assert status == 0
    orc = kc.oracle_select(b)
    kc.check_selection(ids, scores, pos, orc)
    kc.check_pool_full(b, kc.placements_from_oracle(orc),
                       rope=oracle.rope_spec(w.rope_theta, w.head_dim, pairing))
    del keep


def test_mixed_host_and_device_stores():
    # three requests: the middle one's store is host-resident
    w = W(requests=3, n_facts=300, k=12, seed=810)
    b = synth.build_workload(w)
    views, keep = host_views(b, {1})
    f = kc.Fused(b)
    f.d_views = kc.device_views(views)
    f()
    ids, scores, pos, status = f.results()
    assert status == 0
    orc = kc.oracle_select(b)
    kc.check_selection(ids, scores, pos, orc)
    kc.check_pool_full(b, kc.placements_from_oracle(orc))
    del keep


def test_split_inject_from_host_store():
    w = W(seed=820, k=18, block_size=32)
    b = synth.build_workload(w)
    views, keep = host_views(b, {0})
    orc = kc.oracle_select(b)
    sel, opos = orc[0][1], orc[0][2]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ids = torch.from_numpy(np.ascontiguousarray(sel, np.int32)).cuda()
    starts = torch.from_numpy(np.ascontiguousarray(opos, np.int32)).cuda()
    tl = int(b.table_lens[0])
    bt = torch.from_numpy(b.block_tables[0, :tl].copy()).cuda()
    kvi.kvi_inject_paged(views[0], ids, starts, ids.shape[0], bt, tl, kc.cache_of(b), w.rope_theta, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    kc.check_pool_full(b, kc.placements_from_oracle(orc))
    del keep


def test_shared_store_path_with_host_kv():
    # many queries over one host-resident store (tensor-core retrieval from
    # device embeddings, injection from host K/V)
    R = 4
    w = W(requests=R, n_facts=500, k=10, seed=830)
    b = synth.build_workload(w)
    b.stores = [b.stores[0]] * R
    views, keep = host_views(b, {0})
    k = w.k
    ids = torch.empty((R, k), dtype=torch.int32, device="cuda")
    sc = torch.empty((R, k), dtype=torch.float32, device="cuda")
    pos = torch.empty((R, k), dtype=torch.int32, device="cuda")
    ws = torch.empty(kvi.kvi_workspace_bytes_shared(R, w.n_facts, k), dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvi.kvi_retrieve_and_inject_shared(
        views[0], R, b.queries, k, torch.from_numpy(b.start_pos).cuda(),
        torch.from_numpy(b.block_tables).cuda(), torch.from_numpy(b.table_lens).cuda(),
        b.max_blocks, kc.cache_of(b), kvi.rope(w.rope_theta), ids, sc, pos, ws, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    orc = kc.oracle_select(b)
    kc.check_selection(ids.cpu().numpy(), sc.cpu().numpy(), pos.cpu().numpy(), orc)
    kc.check_pool_full(b, kc.placements_from_oracle(orc))
    del keep
