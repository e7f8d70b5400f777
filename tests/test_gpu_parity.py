"""GPU parity of the retrieve-and-inject path against the float64 oracle.

Every case runs the CUDA kernels through the C ABI (ctypes binding) and
compares with the oracle element by element: fact ids, placements and V bits
exactly, rotated K within 2^-8|x| + 1e-6, scores within 1e-4 relative, and
all untouched pool bytes against their canaries.  Sizes span several CTAs,
pages and layer groups with ragged tails.  Method: "InferScale: GPU-Native
KV Injection for Personalized LLM Serving", Figure 2 caption, Section 5.1 /
Theorem 6, Section 3.4.
"""
import dataclasses

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
    base = dict(name="custom", layers=3, kv_heads=4, head_dim=128, rope_theta=5e5, block_size=16,
                n_facts=700, len_lo=1, len_hi=40, len_dist="uniform", embed_dim=256, requests=1,
                k=37, start=5, start_hi=0, seed=123, store="dense")
    base.update(kw)
    return synth.Workload(**base)


def fused_and_check(b, k=None):
    ids, scores, pos, status = kc.run_fused(b, k)
    assert status == 0, kvi.kvi_status_str(status)
    orc = kc.oracle_select(b, k)
    kc.check_selection(ids, scores, pos, orc)
    kc.check_pool_full(b, kc.placements_from_oracle(orc))
    return ids, orc


# ------------------------------------------------------------- fused path

def test_tiny_fused_full_pool():
    b = synth.build_workload(synth.WORKLOADS["tiny"])
    ids, orc = fused_and_check(b)
    assert orc[0][2].tolist() == [0, 16, 32, 48, 64]  # 5 facts of 16 tokens from 0


def test_multi_request_ragged_full_pool():
    w = W(requests=3, n_facts=900, seed=7)
    b = synth.build_workload(w)
    fused_and_check(b)


@pytest.mark.parametrize("R,k,B", [(8, 40, 16), (16, 15, 16), (17, 12, 16), (1, 37, 1), (2, 30, 4)])
def test_fused_staging_limits(R, k, B):
    # small fused calls stage their facts and block tables in shared memory;
    # these straddle the limits (request count, fact slots, table entries) so
    # that both the staged and the global resolution run
    w = W(requests=R, n_facts=300, k=k, block_size=B, layers=2, kv_heads=2, head_dim=64,
          seed=300 + R + k + B)
    fused_and_check(synth.build_workload(w))


def test_selection_streams_large_store():
    # more keys than the selector keeps in registers: both of its passes
    # stream the keys from L2
    w = W(n_facts=15000, k=50, layers=1, kv_heads=1, head_dim=64, embed_dim=64, len_hi=8,
          seed=311)
    fused_and_check(synth.build_workload(w))


@pytest.mark.parametrize("D,H,E,L", [(16, 1, 100, 1), (64, 3, 384, 2), (256, 2, 1536, 9),
                                     (128, 8, 1024, 4), (32, 5, 4, 3), (512, 1, 132, 2)])
def test_geometries(D, H, E, L):
    w = W(head_dim=D, kv_heads=H, embed_dim=E, layers=L, n_facts=300, k=11, seed=D + H + E)
    b = synth.build_workload(w)
    fused_and_check(b)


@pytest.mark.parametrize("k", [1, 2, 31, 32, 33, 64, 256])
def test_k_values(k):
    w = W(layers=1, kv_heads=1, head_dim=64, n_facts=max(300, k), k=k, len_hi=6, seed=1000 + k)
    b = synth.build_workload(w)
    fused_and_check(b)


def test_k_equals_n_and_single_fact_store():
    b = synth.build_workload(W(layers=1, kv_heads=2, head_dim=64, n_facts=40, k=40, seed=5))
    fused_and_check(b)
    b = synth.build_workload(W(layers=1, kv_heads=2, head_dim=64, n_facts=1, k=1, seed=6))
    fused_and_check(b)


def test_block_size_one_and_page_straddles():
    for B, start in [(1, 0), (16, 15), (7, 3), (32, 31)]:
        b = synth.build_workload(W(block_size=B, start=start, n_facts=200, k=9, seed=B))
        fused_and_check(b)


def test_repeated_calls_reuse_workspace():
    b = synth.build_workload(W(requests=2, n_facts=500, k=20, seed=77))
    f = kc.Fused(b)
    f()
    first = f.results()
    synth.fill_canary(b.pool)
    f()
    second = f.results()
    for a, c in zip(first[:3], second[:3]):
        assert np.array_equal(a, c)
    orc = kc.oracle_select(b)
    kc.check_selection(*second[:3], orc)
    kc.check_pool_full(b, kc.placements_from_oracle(orc))


# -------------------------------------------------------- exact selection

def _with_embeddings(b, emb_np, r=0):
    st = b.stores[r]
    st.emb_np = np.ascontiguousarray(emb_np, np.float32)
    st.emb = torch.from_numpy(st.emb_np).cuda()


def test_planted_duplicates_tie_to_lower_id():
    b = synth.build_workload(W(n_facts=2000, k=50, embed_dim=128, seed=31))
    rng = np.random.default_rng(31)
    emb = b.stores[0].emb_np.copy()
    q = synth.planted_query(rng, emb, [10, 500, 1500])
    # copies of the planted rows further down: exact ties in every arithmetic
    for src, dst in [(10, 1999), (500, 20), (1500, 700), (10, 11)]:
        emb[dst] = emb[src]
    _with_embeddings(b, emb)
    b.queries_np[0] = q
    b.queries = torch.from_numpy(b.queries_np).cuda()
    ids, orc = fused_and_check(b)
    assert {10, 11, 1999, 500, 20, 1500, 700} <= set(ids[0].tolist())


def test_all_equal_keys_take_lowest_ids():
    # every key identical: the crowded-bucket radix path runs down to the
    # last digit and the lowest ids win
    b = synth.build_workload(W(n_facts=3000, k=50, embed_dim=128, seed=41))
    emb = np.tile(b.stores[0].emb_np[:1], (3000, 1))
    _with_embeddings(b, emb)
    ids, orc = fused_and_check(b)
    assert ids[0].tolist() == list(range(50))


def test_crowded_bucket_distinct_keys():
    # keys all inside one float32 bucket but distinct in float64: the radix
    # refinement has to separate them
    b = synth.build_workload(W(n_facts=5000, k=40, embed_dim=128, seed=43))
    rng = np.random.default_rng(43)
    base = b.stores[0].emb_np[0].astype(np.float64)
    emb = base[None, :] + 1e-5 * rng.standard_normal((5000, 128))
    _with_embeddings(b, emb.astype(np.float32))
    b.queries_np[0] = base.astype(np.float32)
    b.queries = torch.from_numpy(b.queries_np).cuda()
    fused_and_check(b)


def test_negative_scores_and_zero_query():
    b = synth.build_workload(W(n_facts=400, k=30, seed=47))
    b.queries_np[0] = -b.stores[0].emb_np[3]
    b.queries = torch.from_numpy(b.queries_np).cuda()
    fused_and_check(b)
    b2 = synth.build_workload(W(n_facts=400, k=30, seed=48))
    b2.queries_np[0] = 0.0  # every score is zero: ids 0..k-1
    b2.queries = torch.from_numpy(b2.queries_np).cuda()
    ids, _ = fused_and_check(b2)
    assert ids[0].tolist() == list(range(30))


# -------------------------------------------------------------- split API

def _split(b, k, ids_override=None, starts=None):
    view = kc.views_of(b)[0]
    cache = kc.cache_of(b)
    N = b.w.n_facts
    ids = torch.empty(k, dtype=torch.int32, device="cuda")
    scores = torch.empty(k, dtype=torch.float32, device="cuda")
    ws = torch.empty(kvi.kvi_workspace_bytes(1, N, k), dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvi.kvi_retrieve_topk(view, b.queries[0], k, ids, scores, ws, status)
    pos = torch.empty(k, dtype=torch.int32, device="cuda")
    kvi.kvi_place(view, ids, k, int(b.start_pos[0]), pos, status)
    inj_ids, inj_pos = ids, pos
    if ids_override is not None:
        inj_ids = torch.from_numpy(np.ascontiguousarray(ids_override, np.int32)).cuda()
        inj_pos = torch.from_numpy(np.ascontiguousarray(starts, np.int32)).cuda()
    tl = int(b.table_lens[0])
    bt = torch.from_numpy(b.block_tables[0, :tl].copy()).cuda()
    kvi.kvi_inject_paged(view, inj_ids, inj_pos, inj_ids.shape[0], bt, tl, cache, b.w.rope_theta,
                         status)
    torch.cuda.synchronize()
    return ids.cpu().numpy(), scores.cpu().numpy(), pos.cpu().numpy(), int(status.item())


def test_split_calls_match_oracle():
    b = synth.build_workload(W(n_facts=1500, k=45, seed=51))
    ids, scores, pos, status = _split(b, 45)
    assert status == 0
    orc = kc.oracle_select(b)
    kc.check_selection(ids[None], scores[None], pos[None], orc)
    kc.check_pool_full(b, kc.placements_from_oracle(orc))


@pytest.mark.parametrize("mode", ["reversed", "shuffled", "gaps"])
def test_permuted_placement(mode):
    # Chunked RoPE places any fact at any position: inject the same facts in
    # another order (and with gaps) and compare with the oracle for that order.
    b = synth.build_workload(W(n_facts=600, k=20, seed=61, start=3))
    orc = kc.oracle_select(b)
    sel = orc[0][1]
    lens = b.stores[0].len_np
    rng = np.random.default_rng(61)
    order = sel[::-1] if mode == "reversed" else rng.permutation(sel)
    starts, at = [], 3
    for f in order:
        starts.append(at)
        at += int(lens[f]) + (int(rng.integers(0, 5)) if mode == "gaps" else 0)
    need = at
    synth.attach_pool(b, tokens_needed=[need - 3 + 8], rng=rng)
    _ids, _s, _p, status = _split(b, 20, order, starts)
    assert status == 0
    kc.check_pool_full(b, [(np.ascontiguousarray(order, np.int32), np.asarray(starts, np.int64))])


def test_position_zero_is_bit_identical_including_negative_zero():
    b = synth.build_workload(W(layers=2, kv_heads=2, head_dim=64, n_facts=50, k=3, start=0,
                               seed=71))
    # plant -0.0 and +0.0 in the K rows of every fact's first token
    kv = b.kv_np.copy()
    for f in range(50):
        row = int(b.stores[0].start_np[f])
        kv[:, 0, row, :, ::3] = 0x8000
        kv[:, 0, row, :, 1::3] = 0x0000
    b.kv_np = kv
    b.kv = torch.from_numpy(kv.view(np.int16)).cuda().view(torch.bfloat16)
    orc = kc.oracle_select(b)
    sel = orc[0][1]
    _ids, _s, _p, status = _split(b, 3, sel[:1], [0])
    assert status == 0
    blk = int(b.block_tables[0, 0])
    got = b.pool[:, 0, blk, 0].view(torch.int16).cpu().numpy().view(np.uint16)
    row = int(b.stores[0].start_np[sel[0]])
    assert np.array_equal(got, kv[:, 0, row])


def test_large_positions_theta_1e6():
    # positions up to ~39k at theta = 1e6: float32 angle arithmetic would be
    # off by ~1e-3 rad here; the float64-built table keeps 1 bf16 ulp.
    w = W(layers=2, kv_heads=2, head_dim=128, rope_theta=1e6, block_size=32, n_facts=300,
          len_lo=8, len_hi=128, len_dist="loguniform", k=12, start=0, seed=81)
    b = synth.build_workload(w, with_pool=False)
    rng = np.random.default_rng(81)
    sel = kc.oracle_select(b)[0][1]
    lens = b.stores[0].len_np[sel]
    starts = np.sort(rng.choice(np.arange(0, 39168 - 128, 160), size=12, replace=False))
    starts[-1] = 39168 - int(lens[-1])  # the last token sits at position 39167
    B = 32
    table_len = 39168 // B
    used = sorted({(int(s) + t) // B for s, n in zip(starts, lens) for t in range(int(n))})
    nb = len(used)
    blocks = rng.permutation(nb).astype(np.int32)
    bt = np.full((1, table_len), -1, np.int32)
    bt[0, used] = blocks
    b.pool = torch.empty((2, 2, nb, B, 2, 128), dtype=torch.bfloat16, device="cuda")
    synth.fill_canary(b.pool)
    b.block_tables, b.table_lens = bt, np.array([table_len], np.int32)
    _ids, _s, _p, status = _split(b, 12, sel, starts)
    assert status == 0
    kc.check_pool_full(b, [(sel, starts.astype(np.int64))])


# ---------------------------------------------------- device-side errors

def test_bad_fact_id_is_skipped_and_reported():
    b = synth.build_workload(W(n_facts=300, k=6, seed=91))
    sel = kc.oracle_select(b)[0][1]
    lens = b.stores[0].len_np
    ids = [int(sel[0]), 300, int(sel[1])]  # 300 is out of range
    starts = [5, 5 + int(lens[sel[0]]), 5 + int(lens[sel[0]]) + 1]
    _i, _s, _p, status = _split(b, 6, ids, starts)
    assert status == kvi.ERR_OUT_OF_RANGE
    kc.check_pool_full(b, [(np.array([ids[0], ids[2]], np.int32),
                            np.array([starts[0], starts[2]], np.int64))])


def test_block_outside_pool_and_position_beyond_table():
    b = synth.build_workload(W(n_facts=300, k=4, seed=93, block_size=8, len_lo=8, len_hi=8))
    sel = kc.oracle_select(b)[0][1]
    tl = int(b.table_lens[0])
    b.block_tables[0, 1] = b.num_blocks + 5      # positions 8..15 point outside the pool
    # fact 0 at 0..7 (fine), fact 1 at 8..15 (bad block), fact 2 straddles the table end
    starts = [0, 8, tl * 8 - 4]
    _i, _s, _p, status = _split(b, 4, sel[:3], starts)
    assert status == kvi.ERR_OUT_OF_RANGE
    # the oracle's expectation for what must land: fact 0 whole, fact 2's
    # first 4 tokens
    view_bt = b.block_tables[0, :tl]
    NB, B = b.num_blocks, 8
    bits, vals = kc._pool_arrays(b)
    expect_written = np.zeros(bits.shape, bool)
    st = b.stores[0]
    for f, s0, n in [(sel[0], 0, 8), (sel[2], tl * 8 - 4, 4)]:
        for t in range(n):
            blk, off = oracle.slot(s0 + t, view_bt, B, NB)
            ek, ev = oracle.token_rows(b.kv_np, int(st.start_np[f]) + t, b.w.rope_theta, s0 + t)
            kc.check_k_v(vals[:, 0, blk, off], bits[:, 1, blk, off], ek, ev, f"fact {f} t {t}")
            expect_written[:, :, blk, off] = True
    assert np.all(bits[~expect_written] == synth.CANARY_BITS)


def test_fused_capacity_error_leaves_request_untouched():
    w = W(requests=3, n_facts=400, k=10, seed=95, len_lo=10, len_hi=10)
    b = synth.build_workload(w, with_pool=False)
    synth.attach_pool(b, tokens_needed=[100, 99, 100])  # request 1 lacks one token
    b.table_lens[1] = (5 + 99 + 15) // 16 - 0
    b.table_lens[1] = 6  # 96 slots < 5 + 100 tokens
    f = kc.Fused(b)
    f()
    ids, scores, pos, status = f.results()
    assert status == kvi.ERR_CAPACITY
    orc = kc.oracle_select(b)
    kc.check_selection(ids, scores, pos, orc)
    place = kc.placements_from_oracle(orc)
    place[1] = (np.zeros(0, np.int32), np.zeros(0, np.int64))
    kc.check_pool_full(b, place)


def test_fused_store_with_too_few_facts_is_rejected_on_device():
    w = W(requests=2, n_facts=50, k=10, seed=97)
    b = synth.build_workload(w)
    views = kc.views_of(b)
    views[1].n_facts = 5  # fewer than k
    f = kc.Fused(b)
    f.d_views = kc.device_views(views)
    f()
    ids, scores, pos, status = f.results()
    assert status == kvi.ERR_OUT_OF_RANGE
    assert np.all(ids[1] == -1)
    orc = kc.oracle_select(b)[:1]
    kc.check_selection(ids[:1], scores[:1], pos[:1], orc)
    kc.check_pool_full(b, kc.placements_from_oracle(orc) + [(np.zeros(0, np.int32),
                                                             np.zeros(0, np.int64))])
