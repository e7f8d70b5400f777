"""GPU parity of the rotary variants against the float64 oracle.

Interleaved pairing (2i, 2i+1), the Llama 3.1 frequency scaling and an
engine's own float32 cos/sin table, through kvi_retrieve_and_inject_ex and
kvi_inject_paged_ex.  The paper names only rotary position embedding
("InferScale: GPU-Native KV Injection for Personalized LLM Serving",
Section 5.1 / Theorem 6); these are the conventions of the engines it runs
on.  Same bars as the plain path: ids, positions and V bits exact, K within
2^-8|x| + 1e-6 of the oracle's value.
"""
import itertools

import numpy as np
import pytest
import torch

import oracle
import pre_rope_kv_gb300 as kvi
from tests import kvi_check as kc
from tests import synth

pytestmark = pytest.mark.gpu

LLAMA31 = (8.0, 1.0, 4.0, 8192.0)
_ids = itertools.count(1000)


@pytest.fixture(scope="module", autouse=True)
def _built():
    kc.ensure_built()


def W(**kw):
    base = dict(name="variant", layers=2, kv_heads=3, head_dim=64, rope_theta=5e5, block_size=16,
                n_facts=500, len_lo=1, len_hi=40, len_dist="uniform", embed_dim=128, requests=1,
                k=21, start=7, start_hi=0, seed=501, store="dense")
    base.update(kw)
    return synth.Workload(**base)


def engine_table(theta, D, P):
    """A cos/sin table the way an engine builds one: float32 frequencies and
    float32 angles, cos/sin rounded to float32."""
    inv = (1.0 / np.power(np.float32(theta), np.arange(0, D, 2, dtype=np.float32) / np.float32(D)))
    ang = np.arange(P, dtype=np.float32)[:, None] * inv.astype(np.float32)[None, :]
    return np.cos(ang).astype(np.float32), np.sin(ang).astype(np.float32)


def specs(kind, w, P=None):
    """(kvi.Rope, oracle rope_spec, arrays to keep alive) for a variant."""
    D, theta = w.head_dim, w.rope_theta
    pairing = kvi.ROPE_PAIR_INTERLEAVED if "interleaved" in kind else kvi.ROPE_PAIR_HALF
    if kind.startswith("table"):
        c, s = engine_table(theta, D, P)
        return (kvi.rope(pairing=pairing, cos_table=c, sin_table=s, table_id=next(_ids)),
                oracle.rope_spec(theta, D, pairing, cos_table=c, sin_table=s), (c, s))
    llama3 = LLAMA31 if "llama3" in kind else None
    return (kvi.rope(theta, pairing, llama3=llama3), oracle.rope_spec(theta, D, pairing, llama3), ())


@pytest.mark.parametrize("kind", ["interleaved", "llama3", "llama3_interleaved",
                                  "table_half", "table_interleaved"])
def test_fused_variant_full_pool(kind):
    w = W(seed=500 + len(kind))
    b = synth.build_workload(w)
    spec, ospec, keep = specs(kind, w, P=int(b.max_blocks) * w.block_size)
    ids, scores, pos, status = kc.run_fused(b, rope=spec)
    assert status == 0, kvi.kvi_status_str(status)
    orc = kc.oracle_select(b)
    kc.check_selection(ids, scores, pos, orc)
    kc.check_pool_full(b, kc.placements_from_oracle(orc), rope=ospec)
    del keep


@pytest.mark.parametrize("D,H", [(16, 1), (128, 8), (256, 2)])
def test_interleaved_geometries(D, H):
    w = W(head_dim=D, kv_heads=H, n_facts=200, k=9, seed=D + H)
    b = synth.build_workload(w)
    spec, ospec, _ = specs("interleaved", w)
    ids, scores, pos, status = kc.run_fused(b, rope=spec)
    assert status == 0
    orc = kc.oracle_select(b)
    kc.check_selection(ids, scores, pos, orc)
    kc.check_pool_full(b, kc.placements_from_oracle(orc), rope=ospec)


def test_llama3_scaling_at_large_positions():
    # positions up to ~33k, where every blend regime of the scaling is in use
    w = W(start=None, start_hi=32768, layers=1, kv_heads=2, head_dim=128, n_facts=300, k=12,
          block_size=32, seed=507)
    b = synth.build_workload(w)
    spec, ospec, _ = specs("llama3", w)
    ids, scores, pos, status = kc.run_fused(b, rope=spec)
    assert status == 0
    orc = kc.oracle_select(b)
    kc.check_selection(ids, scores, pos, orc)
    kc.check_pool_full(b, kc.placements_from_oracle(orc), rope=ospec)


@pytest.mark.parametrize("kind", ["interleaved", "table_interleaved", "llama3"])
def test_split_inject_variant(kind):
    w = W(seed=520, k=15)
    b = synth.build_workload(w)
    P = int(b.max_blocks) * w.block_size
    spec, ospec, keep = specs(kind, w, P=P)
    orc = kc.oracle_select(b)
    sel, opos = orc[0][1], orc[0][2]
    view = kc.views_of(b)[0]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ids = torch.from_numpy(np.ascontiguousarray(sel, np.int32)).cuda()
    starts = torch.from_numpy(np.ascontiguousarray(opos, np.int32)).cuda()
    tl = int(b.table_lens[0])
    bt = torch.from_numpy(b.block_tables[0, :tl].copy()).cuda()
    kvi.kvi_inject_paged_ex(view, ids, starts, ids.shape[0], bt, tl, kc.cache_of(b), spec, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    kc.check_pool_full(b, kc.placements_from_oracle(orc), rope=ospec)
    del keep


def test_positions_beyond_a_table_are_reported():
    # a table shorter than the placement: pieces past its end are skipped and
    # KVI_ERR_OUT_OF_RANGE is recorded
    w = W(seed=530, k=20, start=0)
    b = synth.build_workload(w)
    spec, _, keep = specs("table_half", w, P=16)
    _ids, _s, _p, status = kc.run_fused(b, rope=spec)
    assert status == kvi.ERR_OUT_OF_RANGE
    del keep


def test_reused_table_id_keeps_the_first_copy():
    # the library copies a table the first time it sees its id
    w = W(seed=540, k=10)
    b = synth.build_workload(w)
    P = int(b.max_blocks) * w.block_size
    c, s = engine_table(w.rope_theta, w.head_dim, P)
    tid = next(_ids)
    spec = kvi.rope(cos_table=c, sin_table=s, table_id=tid)
    kvi.kvi_prepare_rope_ex(spec, w.head_dim, P)
    garbage = np.full_like(c, 7.0)
    spec2 = kvi.rope(cos_table=garbage, sin_table=garbage, table_id=tid)
    ids, scores, pos, status = kc.run_fused(b, rope=spec2)
    assert status == 0
    orc = kc.oracle_select(b)
    kc.check_pool_full(b, kc.placements_from_oracle(orc),
                       rope=oracle.rope_spec(w.rope_theta, w.head_dim, cos_table=c, sin_table=s))
