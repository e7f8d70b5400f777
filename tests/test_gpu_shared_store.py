"""GPU parity of the shared-store path (many queries, one store).

"InferScale: GPU-Native KV Injection for Personalized LLM Serving",
Section 6.4: concurrent users query one conversation's memory.  The library
scores all queries against the store on the tensor cores and rescores the
facts that can reach the top k exactly, so the bar is the plain one: ids and
positions bit-exact with the float64 oracle, scores within 1e-4, K within
2^-8|x| + 1e-6, V bits exact.  One white-box check reads the tensor-core
intervals from the workspace and checks that each contains the oracle's
exact score.
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
    base = dict(name="shared", layers=2, kv_heads=2, head_dim=64, rope_theta=5e5, block_size=16,
                n_facts=1000, len_lo=1, len_hi=24, len_dist="uniform", embed_dim=256, requests=1,
                k=20, start=5, start_hi=0, seed=700, store="dense")
    base.update(kw)
    return synth.Workload(**base)


def shared_case(R, seed, **kw):
    """One store (request 0 of a workload) and R queries."""
    w = W(seed=seed, **kw)
    b = synth.build_workload(w, with_pool=False)
    st = b.stores[0]
    rng = np.random.default_rng(seed + 1)
    q = synth.query_rows(rng, R, w.embed_dim)
    return w, b, st, q


def run_topk(w, b, st, q, k):
    R = q.shape[0]
    view = kc.views_of(b)[0]
    dq = torch.from_numpy(np.ascontiguousarray(q, np.float32)).cuda()
    ids = torch.empty((R, k), dtype=torch.int32, device="cuda")
    sc = torch.empty((R, k), dtype=torch.float32, device="cuda")
    ws = torch.empty(kvi.kvi_workspace_bytes_shared(R, w.n_facts, k), dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvi.kvi_retrieve_topk_shared(view, R, dq, k, ids, sc, ws, status)
    torch.cuda.synchronize()
    return ids.cpu().numpy(), sc.cpu().numpy(), int(status.item()), ws


def check_topk(st, q, k, ids, sc):
    for r in range(q.shape[0]):
        s = oracle.scores(q[r], st.emb_np)
        sel = oracle.topk(s, k)
        assert np.array_equal(ids[r], sel), f"query {r}: {ids[r].tolist()} vs {sel.tolist()}"
        ref = s[sel]
        assert np.all(np.abs(sc[r].astype(np.float64) - ref) <= kc.S_REL * np.abs(ref) + kc.S_ABS)


@pytest.mark.parametrize("N,E,R,k", [(1000, 256, 1, 10), (3000, 1024, 64, 50), (777, 100, 17, 33),
                                     (5000, 384, 256, 256), (200, 64, 5, 200), (129, 32, 16, 7),
                                     # enough tiles for two accumulators (256 facts) per CTA
                                     (40000, 128, 64, 50), (50001, 96, 3, 20), (39000, 64, 256, 8),
                                     # up to 128 queries: K split over clusters of 2 and of 3
                                     # CTAs; 128 queries fill the M tile; 129 take the other form
                                     (15000, 256, 100, 40), (10000, 512, 128, 64), (20000, 64, 129, 10),
                                     # the widest and the narrowest embeddings: 256 chunks of
                                     # K split over 4 CTAs; one partial chunk of 4 floats
                                     (3000, 8192, 64, 20), (500, 4, 10, 5), (600, 4, 200, 5)])
def test_shared_topk_matches_oracle(N, E, R, k):
    w, b, st, q = shared_case(R, seed=N + E + R + k, n_facts=N, embed_dim=E)
    ids, sc, status, _ = run_topk(w, b, st, q, k)
    assert status == 0
    check_topk(st, q, k, ids, sc)


@pytest.mark.parametrize("N,E,R,k", [(2000, 1024, 48, 30), (40000, 256, 40, 30), (3000, 256, 200, 20)])
def test_tensor_core_intervals_contain_exact_scores(N, E, R, k):
    # white box: the workspace holds the plain regions, then lo and hi
    # planes [R][key_stride] float32 (256-byte aligned regions); 40k facts
    # take the split form without a cluster, 200 queries the form with facts
    # on M
    w, b, st, q = shared_case(R, seed=711, n_facts=N, embed_dim=E)
    ids, sc, status, ws = run_topk(w, b, st, q, k)
    assert status == 0
    stride = (N + 31) // 32 * 32
    base = kvi.kvi_workspace_bytes(R, N, k)
    plane = (R * stride * 4 + 255) // 256 * 256
    raw = ws.cpu().numpy()
    lo = raw[base:base + R * stride * 4].view(np.float32).reshape(R, stride)[:, :N].astype(np.float64)
    hi = raw[base + plane:base + plane + R * stride * 4].view(np.float32).reshape(R, stride)[:, :N].astype(np.float64)
    for r in range(R):
        s = oracle.scores(q[r], st.emb_np)
        assert np.all(lo[r] <= s) and np.all(s <= hi[r]), f"query {r}: an interval misses its score"
        assert np.all(hi[r] - lo[r] < 0.05)  # and the intervals are tight enough to matter
    check_topk(st, q, k, ids, sc)


def test_ties_and_all_equal_keys():
    # planted duplicates tie to the lower id; with every embedding equal all
    # facts are candidates and the selector's histogram fallback runs
    w, b, st, q = shared_case(6, seed=720, n_facts=1500, embed_dim=128)
    emb = st.emb_np.copy()
    emb[700:710] = emb[3]
    q[0] = emb[3]
    st.emb_np = emb
    st.emb = torch.from_numpy(emb).cuda()
    ids, sc, status, _ = run_topk(w, b, st, q, 12)
    assert status == 0
    check_topk(st, q, 12, ids, sc)
    w, b, st, q = shared_case(3, seed=721, n_facts=3000, embed_dim=64)
    emb = np.tile(st.emb_np[:1], (3000, 1))
    st.emb_np = emb
    st.emb = torch.from_numpy(emb).cuda()
    ids, sc, status, _ = run_topk(w, b, st, q, 40)
    assert status == 0
    assert all(ids[r].tolist() == list(range(40)) for r in range(3))


def test_same_ids_as_the_plain_path():
    w, b, st, q = shared_case(9, seed=730, n_facts=2500, embed_dim=512)
    k = 25
    ids, sc, status, _ = run_topk(w, b, st, q, k)
    view = kc.views_of(b)[0]
    for r in range(q.shape[0]):
        dq = torch.from_numpy(np.ascontiguousarray(q[r], np.float32)).cuda()
        pid = torch.empty(k, dtype=torch.int32, device="cuda")
        psc = torch.empty(k, dtype=torch.float32, device="cuda")
        pws = torch.empty(kvi.kvi_workspace_bytes(1, w.n_facts, k), dtype=torch.uint8, device="cuda")
        pst = torch.zeros(1, dtype=torch.int32, device="cuda")
        kvi.kvi_retrieve_topk(view, dq, k, pid, psc, pws, pst)
        torch.cuda.synchronize()
        assert int(pst.item()) == 0
        assert np.array_equal(pid.cpu().numpy(), ids[r])
        np.testing.assert_array_equal(psc.cpu().numpy(), sc[r])


@pytest.mark.parametrize("R,pairing", [(8, 0), (3, 1)])
def test_shared_retrieve_and_inject_full_pool(R, pairing):
    # R requests over one store, each injected through its own block table
    w = W(requests=R, n_facts=600, k=15, seed=740 + R)
    b = synth.build_workload(w)
    b.stores = [b.stores[0]] * R  # every request reads request 0's store
    view = kc.views_of(b)[0]
    spec = kvi.rope(w.rope_theta, pairing)
    ospec = oracle.rope_spec(w.rope_theta, w.head_dim, pairing)
    k = w.k
    ids = torch.empty((R, k), dtype=torch.int32, device="cuda")
    sc = torch.empty((R, k), dtype=torch.float32, device="cuda")
    pos = torch.empty((R, k), dtype=torch.int32, device="cuda")
    ws = torch.empty(kvi.kvi_workspace_bytes_shared(R, w.n_facts, k), dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvi.kvi_retrieve_and_inject_shared(
        view, R, b.queries, k, torch.from_numpy(b.start_pos).cuda(),
        torch.from_numpy(b.block_tables).cuda(), torch.from_numpy(b.table_lens).cuda(),
        b.max_blocks, kc.cache_of(b), spec, ids, sc, pos, ws, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    orc = kc.oracle_select(b)
    kc.check_selection(ids.cpu().numpy(), sc.cpu().numpy(), pos.cpu().numpy(), orc)
    kc.check_pool_full(b, kc.placements_from_oracle(orc), rope=ospec)
