"""GPU parity of the graph index against the oracle.

kvi_graph_build must write exactly the oracle's graph (each fact's degree
most similar other facts, ties to the lower id), and kvi_graph_search must
reproduce the oracle's search step for step on the same graph and seeds:
the same ids in the same order, the same result count, the same number of
iterations and of facts scored, and scores within 1e-4 relative + 1e-7 of
the oracle's float64 values.  A large case (200k facts, 1024-d) checks
sampled graph rows and sampled queries one by one.
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


_EXTENTS = {}


def _view(emb_d):
    # retrieval validates each fact's extent: empty facts (start 0, length 0)
    n = emb_d.shape[0]
    if n not in _EXTENTS:
        _EXTENTS[n] = (torch.zeros(n, dtype=torch.int64, device="cuda"),
                       torch.zeros(n, dtype=torch.int32, device="cuda"))
    fs, fl = _EXTENTS[n]
    g = kvi.geometry(1, 1, 16, emb_d.shape[1])
    return g, kvi.store_view(g, None, emb_d, fs, fl, n_tokens=0)


def gpu_graph(emb_np, degree):
    emb_d = torch.from_numpy(emb_np).cuda()
    _, view = _view(emb_d)
    n = emb_np.shape[0]
    graph = torch.full((n, degree), -7, dtype=torch.int32, device="cuda")
    ws = torch.empty(kvi.kvi_graph_build_workspace_bytes(n, degree), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvi.kvi_graph_build(view, degree, graph, ws, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return graph.cpu().numpy(), emb_d


def gpu_search(emb_d, graph_np, queries_np, seeds_np, beam, width, max_iters, k):
    _, view = _view(emb_d)
    R = queries_np.shape[0]
    graph = torch.from_numpy(np.ascontiguousarray(graph_np, np.int32)).cuda()
    q = torch.from_numpy(queries_np).cuda()
    seeds = torch.from_numpy(np.ascontiguousarray(seeds_np, np.int32)).cuda()
    ids = torch.empty((R, k), dtype=torch.int32, device="cuda")
    sc = torch.empty((R, k), dtype=torch.float32, device="cuda")
    cnt = torch.empty(R, dtype=torch.int32, device="cuda")
    stats = torch.empty((R, 2), dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.empty(kvi.kvi_graph_search_workspace_bytes(R, emb_d.shape[0]), dtype=torch.uint8,
                     device="cuda")
    params = kvi.graph_search_params(beam, width, max_iters, seeds_np.shape[1])
    kvi.kvi_graph_search(view, graph, graph_np.shape[1], R, q, seeds, params, k, ids, sc, ws, cnt,
                         stats, st)
    torch.cuda.synchronize()
    return (ids.cpu().numpy(), sc.cpu().numpy(), cnt.cpu().numpy(), stats.cpu().numpy(),
            int(st.item()))


def check_search(emb_np, graph_np, q_np, seeds_np, out, beam, width, max_iters, k, queries=None):
    ids, sc, cnt, stats, status = out
    assert status == 0
    for r in (range(q_np.shape[0]) if queries is None else queries):
        o_ids, o_sc, o_cnt, o_it, o_scored = oracle.graph_search(
            q_np[r], emb_np, graph_np, seeds_np[r], beam, width, max_iters, k)
        assert cnt[r] == o_cnt, r
        assert np.array_equal(ids[r], o_ids), (r, ids[r], o_ids)
        assert (stats[r, 0], stats[r, 1]) == (o_it, o_scored), r
        m = o_cnt
        assert np.all(np.abs(sc[r, :m] - o_sc[:m]) <= 1e-4 * np.abs(o_sc[:m]) + 1e-7), r
        assert np.all(np.isnan(sc[r, m:]))


@pytest.mark.parametrize("n,e,degree,seed", [(300, 64, 8, 0), (700, 128, 64, 1), (257, 32, 1, 2),
                                            (513, 100, 7, 4), (260, 1028, 128, 5)])
def test_graph_build_matches_the_oracle(n, e, degree, seed):
    rng = np.random.default_rng(seed)
    emb = synth.clustered_rows(rng, n, e, clusters=12)
    g, _ = gpu_graph(emb, degree)
    assert np.array_equal(g, oracle.graph_build(emb, degree))


def test_graph_build_exact_ties_go_to_the_lower_id():
    # integer-valued embeddings: many exactly equal scores
    rng = np.random.default_rng(3)
    emb = rng.integers(-2, 3, (300, 16)).astype(np.float32)
    emb[50:60] = emb[7]  # duplicates of fact 7
    g, _ = gpu_graph(emb, 12)
    assert np.array_equal(g, oracle.graph_build(emb, 12))


@pytest.mark.parametrize("beam,width,max_iters,n_seeds,k", [
    (64, 1, 1000, 16, 10), (64, 1, 1000, 64, 50), (32, 4, 20, 8, 32), (128, 2, 1000, 40, 50),
    (256, 8, 6, 512, 64)])
def test_graph_search_matches_the_oracle(beam, width, max_iters, n_seeds, k):
    rng = np.random.default_rng(10 + beam + width)
    n, e, degree = 3000, 128, 32 if width <= 4 else 64
    emb = synth.clustered_rows(rng, n, e, clusters=30)
    graph = oracle.graph_build(emb, degree)
    q = synth.near_queries(rng, emb, 12)
    seeds = synth.graph_seeds(rng, n, 12, n_seeds)
    emb_d = torch.from_numpy(emb).cuda()
    out = gpu_search(emb_d, graph, q, seeds, beam, width, max_iters, k)
    check_search(emb, graph, q, seeds, out, beam, width, max_iters, k)


@pytest.mark.parametrize("e", [100, 36, 2052])
def test_graph_search_odd_widths_match_the_oracle(e):
    # embedding widths that are not a multiple of a warp's float4 row (a
    # ragged last chunk, and more than one chunk per lane at 2052)
    rng = np.random.default_rng(50 + e)
    n, degree = 1200, 12
    emb = synth.clustered_rows(rng, n, e, clusters=6)
    graph = oracle.graph_build(emb, degree)
    q = synth.near_queries(rng, emb, 6)
    seeds = synth.graph_seeds(rng, n, 6, 5)
    emb_d = torch.from_numpy(emb).cuda()
    out = gpu_search(emb_d, graph, q, seeds, 24, 2, 500, 20)
    check_search(emb, graph, q, seeds, out, 24, 2, 500, 20)


def test_graph_search_batch_variant_matches_the_oracle():
    # more queries than SMs: the 256-thread variant (fewer queries use 512)
    rng = np.random.default_rng(40)
    n, e, degree, R = 2000, 64, 32, 160
    emb = synth.clustered_rows(rng, n, e, clusters=10)
    graph = oracle.graph_build(emb, degree)
    q = synth.near_queries(rng, emb, R)
    seeds = synth.graph_seeds(rng, n, R, 12)
    emb_d = torch.from_numpy(emb).cuda()
    out = gpu_search(emb_d, graph, q, seeds, 48, 2, 1000, 40)
    check_search(emb, graph, q, seeds, out, 48, 2, 1000, 40, queries=range(0, R, 7))


def test_graph_search_edge_cases():
    rng = np.random.default_rng(20)
    n, e = 400, 64
    emb = synth.clustered_rows(rng, n, e, clusters=5)
    graph = oracle.graph_build(emb, 6)
    q = synth.near_queries(rng, emb, 4)
    emb_d = torch.from_numpy(emb).cuda()
    # no iterations: the best seeds
    seeds = synth.graph_seeds(rng, n, 4, 9)
    out = gpu_search(emb_d, graph, q, seeds, 8, 1, 0, 5)
    check_search(emb, graph, q, seeds, out, 8, 1, 0, 5)
    # a graph whose component holds fewer facts than k: a short result
    small = np.array([[(i + 1) % 3 + 0] for i in range(3)] + [[3 + (i + 1) % 5] for i in range(n - 3)],
                     np.int32)
    seeds = np.zeros((4, 1), np.int32)  # fact 0: component {0, 1, 2}
    out = gpu_search(emb_d, small, q, seeds, 8, 1, 100, 5)
    check_search(emb, small, q, seeds, out, 8, 1, 100, 5)
    assert list(out[2]) == [3, 3, 3, 3]
    # repeated seeds are scored once
    seeds = np.full((4, 6), 17, np.int32)
    out = gpu_search(emb_d, graph, q, seeds, 8, 1, 3, 4)
    check_search(emb, graph, q, seeds, out, 8, 1, 3, 4)


def test_graph_search_records_a_bad_seed_and_skips_it():
    rng = np.random.default_rng(21)
    n, e = 200, 32
    emb = synth.clustered_rows(rng, n, e, clusters=4)
    graph = oracle.graph_build(emb, 5)
    q = synth.near_queries(rng, emb, 2)
    seeds = np.array([[3, n + 5, 9], [n, 1, 2]], np.int32)
    emb_d = torch.from_numpy(emb).cuda()
    ids, sc, cnt, stats, status = gpu_search(emb_d, graph, q, seeds, 8, 1, 50, 4)
    assert status == kvi.ERR_OUT_OF_RANGE
    # the remaining seeds give the oracle's search from those seeds
    for r, good in enumerate([[3, 9], [1, 2]]):
        o = oracle.graph_search(q[r], emb, graph, good, 8, 1, 50, 4)
        assert np.array_equal(ids[r], o[0]) and (stats[r, 0], stats[r, 1]) == (o[3], o[4])


def test_graph_search_rejects_bad_parameters():
    rng = np.random.default_rng(22)
    emb = synth.clustered_rows(rng, 100, 16, clusters=3)
    emb_d = torch.from_numpy(emb).cuda()
    graph = torch.zeros((100, 8), dtype=torch.int32, device="cuda")
    _, view = _view(emb_d)
    q = torch.zeros((1, 16), dtype=torch.float32, device="cuda")
    seeds = torch.zeros((1, 4), dtype=torch.int32, device="cuda")
    ids = torch.empty((1, 8), dtype=torch.int32, device="cuda")
    sc = torch.empty((1, 8), dtype=torch.float32, device="cuda")
    ws = torch.empty(kvi.kvi_graph_search_workspace_bytes(1, 100), dtype=torch.uint8, device="cuda")
    bad = [dict(beam=4), dict(beam=300), dict(width=0), dict(width=65), dict(max_iters=-1),
           dict(n_seeds=0), dict(n_seeds=513)]
    for kw in bad:
        p = dict(beam=16, width=1, max_iters=5, n_seeds=4)
        p.update(kw)
        with pytest.raises(kvi.KviError) as e:
            kvi.kvi_graph_search(view, graph, 8, 1, q, seeds, kvi.graph_search_params(**p), 8, ids, sc,
                                 ws)
        assert e.value.status == kvi.ERR_INVALID_ARG, kw
    with pytest.raises(kvi.KviError):
        kvi.kvi_graph_build(view, 100, graph, ws)  # degree >= n_facts


def test_graph_large_store_sampled_rows_and_queries():
    # 200k facts of 1024-d: the build runs 782 shared-store batches; three
    # rows are checked against the oracle's exact scores over all facts and
    # four queries against the oracle's search on the GPU's graph
    rng = np.random.default_rng(30)
    n, e, degree = 200_000, 1024, 64
    emb = synth.clustered_rows(rng, n, e, clusters=2000)
    graph, emb_d = gpu_graph(emb, degree)
    for i in (0, 123_457, n - 1):
        s = oracle.scores(emb[i], emb)
        top = oracle.topk(s, degree + 1)
        assert list(graph[i]) == [int(j) for j in top if j != i][:degree], i
    R = 64
    q = synth.near_queries(rng, emb, R)
    seeds = synth.graph_seeds(rng, n, R, 64)
    out = gpu_search(emb_d, graph, q, seeds, 64, 1, 1000, 50)
    check_search(emb, graph, q, seeds, out, 64, 1, 1000, 50, queries=[0, 17, 40, 63])


def test_graph_retrieval_through_placement_and_injection():
    # the approximate index serves the whole path: the graph search's ids go
    # through kvi_place and kvi_inject_paged, and the pool must equal the
    # oracle's injection of the oracle's search result at its positions
    w = synth.Workload(name="graph_inject", layers=2, kv_heads=4, head_dim=128, rope_theta=5e5,
                       block_size=16, n_facts=800, len_lo=1, len_hi=30, len_dist="uniform",
                       embed_dim=128, requests=1, k=20, start=7, start_hi=0, seed=950, store="dense")
    b = synth.build_workload(w)
    st = b.stores[0]
    emb = st.emb_np
    graph = oracle.graph_build(emb, 16)
    rng = np.random.default_rng(951)
    seeds = synth.graph_seeds(rng, w.n_facts, 1, 16)
    k = w.k
    view = kc.views_of(b)[0]
    ids = torch.empty((1, k), dtype=torch.int32, device="cuda")
    sc = torch.empty((1, k), dtype=torch.float32, device="cuda")
    ws = torch.empty(kvi.kvi_graph_search_workspace_bytes(1, w.n_facts), dtype=torch.uint8,
                     device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    d_graph = torch.from_numpy(graph).cuda()
    d_seeds = torch.from_numpy(seeds).cuda()
    kvi.kvi_graph_search(view, d_graph, 16, 1, b.queries, d_seeds, kvi.graph_search_params(32, 1, 500, 16),
                         k, ids, sc, ws, status=status)
    pos = torch.empty(k, dtype=torch.int32, device="cuda")
    start = int(b.start_pos[0])
    kvi.kvi_place(view, ids[0], k, start, pos, status)
    tl = int(b.table_lens[0])
    bt = torch.from_numpy(b.block_tables[0, :tl].copy()).cuda()
    kvi.kvi_inject_paged(view, ids[0], pos, k, bt, tl, kc.cache_of(b), w.rope_theta, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    o_ids = oracle.graph_search(b.queries_np[0], emb, graph, seeds[0], 32, 1, 500, k)[0]
    assert np.array_equal(ids.cpu().numpy()[0], o_ids)
    o_pos, _ = oracle.place(o_ids, st.len_np, start)
    assert np.array_equal(pos.cpu().numpy(), o_pos)
    kc.check_pool_full(b, [(o_ids, o_pos)])


@pytest.mark.parametrize("R,pairing,width", [(5, 0, 1), (3, 1, 2)])
def test_fused_graph_retrieve_and_inject_full_pool(R, pairing, width):
    # R requests over one store through kvi_graph_retrieve_and_inject: ids,
    # scores and positions as the oracle's search and placement give them,
    # and the whole pool as the oracle's injection of those facts
    w = synth.Workload(name="graph_fused", layers=2, kv_heads=4, head_dim=64, rope_theta=5e5,
                       block_size=16, n_facts=900, len_lo=1, len_hi=25, len_dist="uniform",
                       embed_dim=128, requests=R, k=18, start=5, start_hi=0, seed=960 + R,
                       store="dense")
    b = synth.build_workload(w)
    b.stores = [b.stores[0]] * R  # every request reads request 0's store
    st = b.stores[0]
    emb = st.emb_np
    degree, beam, k = 24, 40, w.k
    graph = oracle.graph_build(emb, degree)
    rng = np.random.default_rng(961 + R)
    seeds = synth.graph_seeds(rng, w.n_facts, R, 10)
    view = kc.views_of(b)[0]
    params = kvi.graph_search_params(beam, width, 300, 10)
    ids = torch.empty((R, k), dtype=torch.int32, device="cuda")
    sc = torch.empty((R, k), dtype=torch.float32, device="cuda")
    pos = torch.empty((R, k), dtype=torch.int32, device="cuda")
    ws = torch.empty(kvi.kvi_graph_retrieve_and_inject_workspace_bytes(R, w.n_facts, beam, k),
                     dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvi.kvi_graph_retrieve_and_inject(
        view, torch.from_numpy(graph).cuda(), degree, R, b.queries, torch.from_numpy(seeds).cuda(),
        params, k, torch.from_numpy(b.start_pos).cuda(), torch.from_numpy(b.block_tables).cuda(),
        torch.from_numpy(b.table_lens).cuda(), b.max_blocks, kc.cache_of(b),
        kvi.rope(w.rope_theta, pairing), ids, sc, pos, ws, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    g_ids, g_sc, g_pos = ids.cpu().numpy(), sc.cpu().numpy(), pos.cpu().numpy()
    placements = []
    for r in range(R):
        o_ids, o_sc, o_cnt, _, _ = oracle.graph_search(b.queries_np[r], emb, graph, seeds[r], beam,
                                                       width, 300, k)
        assert o_cnt == k
        assert np.array_equal(g_ids[r], o_ids), r
        assert np.all(np.abs(g_sc[r] - o_sc) <= 1e-4 * np.abs(o_sc) + 1e-7), r
        o_pos, _ = oracle.place(o_ids, st.len_np, int(b.start_pos[r]))
        assert np.array_equal(g_pos[r], o_pos), r
        placements.append((o_ids, o_pos))
    kc.check_pool_full(b, placements, rope=oracle.rope_spec(w.rope_theta, w.head_dim, pairing))


def test_fused_graph_path_with_more_requests_than_sms():
    # 200 requests over one store: the search runs its batch variant and the
    # selector and inject kernels place and inject every request's facts
    R = 200
    w = synth.Workload(name="graph_many", layers=1, kv_heads=2, head_dim=64, rope_theta=1e4,
                       block_size=16, n_facts=500, len_lo=1, len_hi=6, len_dist="uniform",
                       embed_dim=64, requests=R, k=6, start=2, start_hi=0, seed=970, store="dense")
    b = synth.build_workload(w)
    b.stores = [b.stores[0]] * R
    st = b.stores[0]
    emb = st.emb_np
    graph = oracle.graph_build(emb, 10)
    rng = np.random.default_rng(971)
    seeds = synth.graph_seeds(rng, w.n_facts, R, 6)
    view = kc.views_of(b)[0]
    k, beam = w.k, 16
    ids = torch.empty((R, k), dtype=torch.int32, device="cuda")
    sc = torch.empty((R, k), dtype=torch.float32, device="cuda")
    pos = torch.empty((R, k), dtype=torch.int32, device="cuda")
    ws = torch.empty(kvi.kvi_graph_retrieve_and_inject_workspace_bytes(R, w.n_facts, beam, k),
                     dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvi.kvi_graph_retrieve_and_inject(
        view, torch.from_numpy(graph).cuda(), 10, R, b.queries, torch.from_numpy(seeds).cuda(),
        kvi.graph_search_params(beam, 1, 200, 6), k, torch.from_numpy(b.start_pos).cuda(),
        torch.from_numpy(b.block_tables).cuda(), torch.from_numpy(b.table_lens).cuda(), b.max_blocks,
        kc.cache_of(b), kvi.rope(w.rope_theta), ids, sc, pos, ws, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    g_ids, g_pos = ids.cpu().numpy(), pos.cpu().numpy()
    placements = []
    for r in range(R):
        o_ids = oracle.graph_search(b.queries_np[r], emb, graph, seeds[r], beam, 1, 200, k)[0]
        assert np.array_equal(g_ids[r], o_ids), r
        o_pos, _ = oracle.place(o_ids, st.len_np, int(b.start_pos[r]))
        assert np.array_equal(g_pos[r], o_pos), r
        placements.append((o_ids, o_pos))
    kc.check_pool_full(b, placements)
