"""Plans: one fused call recorded into a CUDA graph and replayed.

Each replay reads the current contents of the plan's buffers, so a serving
loop writes a new query, start and block table and launches again.  Checked
against the float64 oracle after every launch, exactly as the direct call
("InferScale: GPU-Native KV Injection for Personalized LLM Serving", Figure 2
serving path).
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


@pytest.mark.parametrize("pairing", [0, 1])
def test_plan_replays_with_new_inputs(pairing):
    w = synth.Workload(name="plan", layers=2, kv_heads=2, head_dim=64, rope_theta=5e5, block_size=16,
                       n_facts=600, len_lo=1, len_hi=30, len_dist="uniform", embed_dim=256,
                       requests=2, k=15, start=4, start_hi=0, seed=950 + pairing, store="dense")
    b = synth.build_workload(w)
    f = kc.Fused(b)
    spec = kvi.rope(w.rope_theta, pairing)
    ospec = oracle.rope_spec(w.rope_theta, w.head_dim, pairing)
    q_dev = b.queries.clone()
    plan = kvi.kvi_plan_create_fused(f.g, w.requests, f.d_views, w.n_facts, q_dev, f.k, f.start, f.bt,
                                     f.tl, b.max_blocks, f.cache, spec, f.ids, f.scores, f.pos, f.ws,
                                     f.status)
    rng = np.random.default_rng(951)
    for rep in range(3):
        if rep:
            # new requests: new queries written into the plan's query buffer
            b.queries_np = synth.query_rows(rng, w.requests, w.embed_dim)
            b.queries = torch.from_numpy(b.queries_np).cuda()
            q_dev.copy_(b.queries)
            synth.fill_canary(b.pool)
        f.status.zero_()
        plan.launch()
        ids, scores, pos, status = f.results()
        assert status == 0
        orc = kc.oracle_select(b)
        kc.check_selection(ids, scores, pos, orc)
        kc.check_pool_full(b, kc.placements_from_oracle(orc), rope=ospec)
    plan.close()


def test_plan_refuses_bad_arguments():
    # argument errors surface when the plan is created, before any recording
    w = synth.Workload(name="p", layers=1, kv_heads=1, head_dim=16, rope_theta=1e4, block_size=16,
                       n_facts=10, len_lo=1, len_hi=2, len_dist="uniform", embed_dim=16, requests=1,
                       k=1, start=0, start_hi=0, seed=1, store="dense")
    b = synth.build_workload(w)
    f = kc.Fused(b)
    for R, k in [(0, 1), (1, 0), (1, kvi.MAX_K + 1)]:
        with pytest.raises(kvi.KviError):
            kvi.kvi_plan_create_fused(f.g, R, f.d_views, w.n_facts, b.queries, k, f.start, f.bt, f.tl,
                                      b.max_blocks, f.cache, kvi.rope(1e4), f.ids, f.scores, f.pos,
                                      f.ws, f.status)


def test_plan_with_request_copies():
    # the plan also records the request's packed input copy (query | start |
    # block table) and output copy (ids | scores | positions | status)
    w = synth.Workload(name="planio", layers=2, kv_heads=2, head_dim=64, rope_theta=5e5, block_size=16,
                       n_facts=400, len_lo=1, len_hi=20, len_dist="uniform", embed_dim=128,
                       requests=1, k=9, start=6, start_hi=0, seed=960, store="dense")
    b = synth.build_workload(w)
    f = kc.Fused(b)
    E, k, tl = w.embed_dim, w.k, int(b.block_tables.shape[1])
    s_off, bt_off = E * 4, E * 4 + 16
    in_bytes, out_bytes = bt_off + tl * 4, 12 * k + 4
    d_in = torch.empty(in_bytes, dtype=torch.uint8, device="cuda")
    d_out = torch.zeros(out_bytes, dtype=torch.uint8, device="cuda")
    h_in = torch.zeros(in_bytes, dtype=torch.uint8).pin_memory()
    h_out = torch.zeros(out_bytes, dtype=torch.uint8).pin_memory()
    q = d_in[:s_off].view(torch.float32).view(1, E)
    start = d_in[s_off:s_off + 4].view(torch.int32)
    bt = d_in[bt_off:].view(torch.int32).view(1, tl)
    ids = d_out[:4 * k].view(torch.int32).view(1, k)
    sc = d_out[4 * k:8 * k].view(torch.float32).view(1, k)
    pos = d_out[8 * k:12 * k].view(torch.int32).view(1, k)
    status = d_out[12 * k:].view(torch.int32)
    plan = kvi.kvi_plan_create_fused(f.g, 1, f.d_views, w.n_facts, q, k, start, bt, f.tl, b.max_blocks,
                                     f.cache, kvi.rope(w.rope_theta), ids, sc, pos, f.ws, status,
                                     io=(h_in, d_in, d_out, h_out))
    rng = np.random.default_rng(961)
    hn = h_in.numpy()
    for rep in range(2):
        b.queries_np = synth.query_rows(rng, 1, E)
        hn[:s_off] = b.queries_np.astype(np.float32).view(np.uint8).ravel()
        hn[s_off:s_off + 4] = np.array([b.start_pos[0]], np.int32).view(np.uint8)
        hn[bt_off:] = b.block_tables[0].astype(np.int32).view(np.uint8)
        synth.fill_canary(b.pool)
        plan.launch()
        torch.cuda.synchronize()
        ho = h_out.numpy()
        got_ids = ho[:4 * k].view(np.int32)[None]
        got_sc = ho[4 * k:8 * k].view(np.float32)[None]
        got_pos = ho[8 * k:12 * k].view(np.int32)[None]
        assert int(ho[12 * k:].view(np.int32)[0]) == 0
        orc = kc.oracle_select(b)
        kc.check_selection(got_ids, got_sc, got_pos, orc)
        kc.check_pool_full(b, kc.placements_from_oracle(orc))
    plan.close()


def test_plan_replays_after_the_rope_table_grows():
    # A plan keeps the address of the RoPE table it was recorded with.  A
    # later call that needs more positions replaces the table for later
    # calls; the plan's table must stay valid and the replay must still
    # match the oracle (ids, positions and V bit-exact, K within tolerance).
    w = synth.Workload(name="planrope", layers=2, kv_heads=2, head_dim=64, rope_theta=5e5,
                       block_size=16, n_facts=500, len_lo=1, len_hi=24, len_dist="uniform",
                       embed_dim=128, requests=1, k=12, start=5, start_hi=0, seed=970,
                       store="dense")
    b = synth.build_workload(w)
    f = kc.Fused(b)
    q_dev = b.queries.clone()
    spec = kvi.rope(w.rope_theta)
    plan = kvi.kvi_plan_create_fused(f.g, 1, f.d_views, w.n_facts, q_dev, f.k, f.start, f.bt, f.tl,
                                     b.max_blocks, f.cache, spec, f.ids, f.scores, f.pos, f.ws,
                                     f.status)
    rng = np.random.default_rng(971)
    for grow_to in (b.max_blocks * w.block_size * 8, 1 << 20):
        kvi.kvi_prepare_rope(w.rope_theta, w.head_dim, grow_to)
        b.queries_np = synth.query_rows(rng, 1, w.embed_dim)
        b.queries = torch.from_numpy(b.queries_np).cuda()
        q_dev.copy_(b.queries)
        synth.fill_canary(b.pool)
        f.status.zero_()
        plan.launch()
        ids, scores, pos, status = f.results()
        assert status == 0
        orc = kc.oracle_select(b)
        kc.check_selection(ids, scores, pos, orc)
        kc.check_pool_full(b, kc.placements_from_oracle(orc))
    # a direct call now uses the grown table and agrees as well
    synth.fill_canary(b.pool)
    f.status.zero_()
    f()
    ids, scores, pos, status = f.results()
    assert status == 0
    orc = kc.oracle_select(b)
    kc.check_selection(ids, scores, pos, orc)
    kc.check_pool_full(b, kc.placements_from_oracle(orc))
    plan.close()
