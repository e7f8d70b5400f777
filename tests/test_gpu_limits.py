"""GPU parity at the library's limits and degenerate inputs.

Embedding sizes above 2048 (the scoring kernel without the shared-memory
ring) up to the maximum 8192; the maximum number of requests in one fused
call (4096) and of facts in one split inject (4096); facts of length 0;
the maximum head size.  Oracle: "InferScale: GPU-Native KV Injection for
Personalized LLM Serving" as restated in oracle/ (Figure 2 caption, Section
5.1 / Theorem 6, Section 3.4).
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
    base = dict(name="limits", layers=1, kv_heads=1, head_dim=16, rope_theta=1e4, block_size=16,
                n_facts=200, len_lo=1, len_hi=8, len_dist="uniform", embed_dim=64, requests=1,
                k=10, start=2, start_hi=0, seed=900, store="dense")
    base.update(kw)
    return synth.Workload(**base)


def fused_and_check(b, k=None):
    ids, scores, pos, status = kc.run_fused(b, k)
    assert status == 0, kvi.kvi_status_str(status)
    orc = kc.oracle_select(b, k)
    kc.check_selection(ids, scores, pos, orc)
    kc.check_pool_full(b, kc.placements_from_oracle(orc))


@pytest.mark.parametrize("E", [2052, 4096, 8192])
def test_large_embeddings(E):
    fused_and_check(synth.build_workload(W(embed_dim=E, n_facts=300, k=17, seed=900 + E)))


@pytest.mark.parametrize("E", [4096, 8192])
def test_large_embeddings_shared_store(E):
    w = W(embed_dim=E, n_facts=500, seed=901 + E)
    b = synth.build_workload(w, with_pool=False)
    st = b.stores[0]
    R, k = 5, 12
    q = synth.query_rows(np.random.default_rng(E), R, E)
    view = kc.views_of(b)[0]
    ids = torch.empty((R, k), dtype=torch.int32, device="cuda")
    sc = torch.empty((R, k), dtype=torch.float32, device="cuda")
    ws = torch.empty(kvi.kvi_workspace_bytes_shared(R, w.n_facts, k), dtype=torch.uint8, device="cuda")
    kvi.kvi_retrieve_topk_shared(view, R, torch.from_numpy(q).cuda(), k, ids, sc, ws)
    torch.cuda.synchronize()
    for r in range(R):
        assert np.array_equal(ids.cpu().numpy()[r], oracle.topk(oracle.scores(q[r], st.emb_np), k))


def test_maximum_requests_in_one_call():
    # 4096 requests over small stores of their own, every one checked in full
    R = kvi.MAX_REQUESTS
    w = W(requests=R, n_facts=12, k=2, len_hi=3, seed=910)
    fused_and_check(synth.build_workload(w))


def test_maximum_facts_in_one_split_inject():
    n = kvi.MAX_INJECT_FACTS
    w = W(n_facts=n, len_lo=1, len_hi=2, k=1, seed=920, block_size=8)
    b = synth.build_workload(w, tokens_needed=[n * 2 + 8])
    lens = b.stores[0].len_np
    ids_np = np.random.default_rng(920).permutation(n).astype(np.int32)
    starts_np = (2 + np.concatenate([[0], np.cumsum(lens[ids_np])[:-1]])).astype(np.int32)
    view = kc.views_of(b)[0]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    tl = int(b.table_lens[0])
    kvi.kvi_inject_paged(view, torch.from_numpy(ids_np).cuda(), torch.from_numpy(starts_np).cuda(), n,
                         torch.from_numpy(b.block_tables[0, :tl].copy()).cuda(), tl, kc.cache_of(b),
                         w.rope_theta, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    kc.check_pool_full(b, [(ids_np, starts_np.astype(np.int64))])


def test_zero_length_facts():
    # lengths 0..6: empty facts take a rank and inject nothing
    w = W(len_lo=0, len_hi=6, n_facts=300, k=40, seed=930)
    b = synth.build_workload(w)
    assert (b.stores[0].len_np == 0).sum() > 10
    fused_and_check(b)


def test_maximum_head_dim_interleaved():
    w = W(head_dim=512, kv_heads=2, n_facts=100, k=6, seed=940)
    b = synth.build_workload(w)
    spec = kvi.rope(w.rope_theta, kvi.ROPE_PAIR_INTERLEAVED)
    ids, scores, pos, status = kc.run_fused(b, rope=spec)
    assert status == 0
    orc = kc.oracle_select(b)
    kc.check_selection(ids, scores, pos, orc)
    kc.check_pool_full(b, kc.placements_from_oracle(orc),
                       rope=oracle.rope_spec(w.rope_theta, 512, oracle.PAIR_INTERLEAVED))
