"""The debug build (include/kvi_debug.h) on the GPU.

1. kvi_inject_paged reports two facts placed over the same positions as
   KVI_ERR_INVALID_ARG ("InferScale: GPU-Native KV Injection for
   Personalized LLM Serving", Section 5.1: each fact gets positions of its
   own); without an overlap it reports nothing and matches the oracle.
2. Failure detection without a fault: the scoring kernel is told to skip one
   row's copy, so the consumer waiting for it gives up after the kernel's
   one-second bound.  The status word of kvi_retrieve_topk (and of the fused
   call) then reads KVI_ERR_TIMEOUT, and the next call on the same context
   matches the oracle again.
3. The same for the shared-store path's tensor-core kernels: one CTA loads
   nothing for one K chunk, in the cluster form (up to 128 queries) and in
   the form with facts on M (more queries).
"""
import time

import numpy as np
import pytest
import torch

import oracle
import pre_rope_kv_gb300 as kvi
from pre_rope_kv_gb300 import build as kbuild
from tests import kvi_check as kc
from tests import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dbg():
    kc.ensure_built()
    lib = kvi.open_library(kbuild.build(debug=True))
    with kvi.use_library(lib):
        yield lib
        kvi.kvi_debug_stall_scorer_row(-1)
        kvi.kvi_debug_stall_coarse_chunk(-1, -1)


def _w(seed, **kw):
    d = dict(name="dbg", layers=2, kv_heads=2, head_dim=64, rope_theta=1e4, block_size=16, n_facts=400,
             len_lo=2, len_hi=10, len_dist="uniform", embed_dim=128, requests=1, k=6, start=0,
             start_hi=0, seed=seed, store="dense")
    d.update(kw)
    return synth.Workload(**d)


def _inject(b, ids, starts):
    view = kc.views_of(b)[0]
    cache = kc.cache_of(b)
    tl = int(b.table_lens[0])
    bt = torch.from_numpy(b.block_tables[0, :tl].copy()).cuda()
    d_ids = torch.from_numpy(np.ascontiguousarray(ids, np.int32)).cuda()
    d_pos = torch.from_numpy(np.ascontiguousarray(starts, np.int32)).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvi.kvi_inject_paged(view, d_ids, d_pos, len(ids), bt, tl, cache, b.w.rope_theta, status)
    torch.cuda.synchronize()
    return int(status.item())


def test_overlapping_starts_are_reported(dbg):
    b = synth.build_workload(_w(71))
    lens = b.stores[0].len_np
    ids = np.array([3, 17, 42], np.int64)
    # back to back: no overlap, no status, and the pool is the oracle's
    starts = np.array([0, int(lens[3]), int(lens[3] + lens[17])])
    assert _inject(b, ids, starts) == 0
    kc.check_pool_full(b, [(ids, starts)])
    # the third fact starts one position inside the second
    synth.fill_canary(b.pool)
    starts[2] -= 1
    assert _inject(b, ids, starts) == kvi.ERR_INVALID_ARG
    # two facts at the same start
    synth.fill_canary(b.pool)
    assert _inject(b, np.array([5, 6]), np.array([7, 7])) == kvi.ERR_INVALID_ARG
    # an empty fact never overlaps; touching ranges do not overlap
    synth.fill_canary(b.pool)
    starts = np.array([0, int(lens[3]), int(lens[3] + lens[17])])
    assert _inject(b, ids, starts) == 0


def _retrieve(b, k, ws):
    view = kc.views_of(b)[0]
    ids = torch.empty(k, dtype=torch.int32, device="cuda")
    sc = torch.empty(k, dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvi.kvi_retrieve_topk(view, b.queries[0], k, ids, sc, ws, status)
    torch.cuda.synchronize()
    return ids.cpu().numpy(), sc.cpu().numpy(), int(status.item())


def test_a_scorer_wait_that_runs_out_surfaces_in_the_retrieval_status(dbg):
    b = synth.build_workload(_w(72, n_facts=3000, embed_dim=1024), with_pool=False)
    k = 20
    ws = torch.zeros(kvi.kvi_workspace_bytes(1, b.w.n_facts, k), dtype=torch.uint8, device="cuda")
    want = oracle.topk(oracle.scores(b.queries_np[0], b.stores[0].emb_np), k)
    ids, _sc, status = _retrieve(b, k, ws)
    assert status == 0 and np.array_equal(ids, want)
    kvi.kvi_debug_stall_scorer_row(1234)
    t0 = time.perf_counter()
    _ids, _sc, status = _retrieve(b, k, ws)
    waited = time.perf_counter() - t0
    assert status == kvi.ERR_TIMEOUT
    assert 0.9 < waited < 30.0, waited  # the one-second bound, not a hang
    kvi.kvi_debug_stall_scorer_row(-1)
    ids, _sc, status = _retrieve(b, k, ws)
    assert status == 0 and np.array_equal(ids, want)


def test_a_scorer_timeout_in_the_fused_call_injects_nothing_unscored(dbg):
    # the rows the timed-out consumer did not score are marked invalid, so
    # the inject kernel never trusts their stale lengths
    b = synth.build_workload(_w(73, n_facts=2500, embed_dim=512, k=30))
    f = kc.Fused(b)
    f.ws.zero_()
    kvi.kvi_debug_stall_scorer_row(0)
    f()
    _ids, _sc, _pos, status = f.results()
    assert status == kvi.ERR_TIMEOUT
    kvi.kvi_debug_stall_scorer_row(-1)
    synth.fill_canary(b.pool)
    f.status.zero_()
    f()
    ids, scores, pos, status = f.results()
    assert status == 0
    orc = kc.oracle_select(b)
    kc.check_selection(ids, scores, pos, orc)
    kc.check_pool_full(b, kc.placements_from_oracle(orc))


@pytest.mark.parametrize("R", [64, 200])
def test_a_coarse_kernel_wait_that_runs_out_surfaces_in_the_shared_status(dbg, R):
    # 3000 facts, E = 1024: 64 queries take the cluster form (12 tiles of
    # 256 facts, K split over 4 CTAs: CTA 0 owns chunks 0-7); 200 take the
    # form with facts on M (24 CTAs, all 32 chunks each)
    b = synth.build_workload(_w(74, n_facts=3000, embed_dim=1024), with_pool=False)
    st = b.stores[0]
    q = synth.query_rows(np.random.default_rng(75), R, b.w.embed_dim)
    k = 16
    view = kc.views_of(b)[0]
    dq = torch.from_numpy(np.ascontiguousarray(q, np.float32)).cuda()
    ids = torch.empty((R, k), dtype=torch.int32, device="cuda")
    sc = torch.empty((R, k), dtype=torch.float32, device="cuda")
    ws = torch.empty(kvi.kvi_workspace_bytes_shared(R, b.w.n_facts, k), dtype=torch.uint8, device="cuda")

    def call():
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        kvi.kvi_retrieve_topk_shared(view, R, dq, k, ids, sc, ws, status)
        torch.cuda.synchronize()
        return int(status.item())

    def matches():
        got = ids.cpu().numpy()
        return all(np.array_equal(got[r], oracle.topk(oracle.scores(q[r], st.emb_np), k)) for r in range(R))

    assert call() == 0 and matches()
    kvi.kvi_debug_stall_coarse_chunk(0, 1)
    t0 = time.perf_counter()
    status = call()
    waited = time.perf_counter() - t0
    assert status == kvi.ERR_TIMEOUT
    assert 0.9 < waited < 60.0, waited  # the one-second bounds, not a hang
    kvi.kvi_debug_stall_coarse_chunk(-1, -1)
    assert call() == 0 and matches()
