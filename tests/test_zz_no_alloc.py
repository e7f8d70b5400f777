"""kvi_retrieve_topk_noalloc against kvi_retrieve_topk, through the C ABI.

The no-allocation entry point serves callers that cannot allocate device
memory where they retrieve (an engine that has handed nearly all GPU memory
to its KV pool, a serving loop that must not call the CUDA allocator, a C
caller with no allocator): it keeps its scratch in a fixed device array of
the library.  It must give the same ids, and scores within the parity
tolerance, as the workspace entry point and as the float64 oracle, call
after call, although every call reuses (and finds the previous call's data
in) the same array.

This file is named to be collected last, so that a run that stops at the
first failure has run every other test before it.
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


def _store(n_facts, embed_dim, seed):
    w = synth.Workload(name="noalloc", layers=2, kv_heads=2, head_dim=64, rope_theta=5e5,
                       block_size=16, n_facts=n_facts, len_lo=1, len_hi=8, len_dist="uniform",
                       embed_dim=embed_dim, requests=1, k=1, start=0, start_hi=0, seed=seed,
                       store="dense")
    b = synth.build_workload(w)
    return b, kc.views_of(b)[0]


def _with_workspace(view, q, k):
    n = int(view.n_facts)
    ids = torch.empty(k, dtype=torch.int32, device="cuda")
    sc = torch.empty(k, dtype=torch.float32, device="cuda")
    ws = torch.empty(kvi.kvi_workspace_bytes(1, n, k), dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvi.kvi_retrieve_topk(view, q, k, ids, sc, ws, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return ids.cpu().numpy(), sc.cpu().numpy()


def _no_alloc(view, q, k, ids, sc, status):
    status.zero_()
    kvi.kvi_retrieve_topk_noalloc(view, q, k, ids, sc, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return ids[:k].cpu().numpy(), sc[:k].cpu().numpy()


def _same(got, want):
    gi, gs = got
    wi, ws = want
    np.testing.assert_array_equal(gi, wi)
    assert np.all(np.abs(gs.astype(np.float64) - ws) <= kc.S_REL * np.abs(ws) + kc.S_ABS)


def _oracle(b, k):
    """The float64 oracle's top-k ids and their exact scores."""
    s = oracle.scores(b.queries_np[0], b.stores[0].emb_np)
    sel = oracle.topk(s, k)
    return sel, s[sel]


def test_two_calls_in_a_row_match_the_workspace_entry_point():
    # a large store first, then a smaller one with another query and k: the
    # second call finds the first call's keys in the shared array
    b1, v1 = _store(20000, 256, seed=901)
    b2, v2 = _store(3001, 128, seed=902)
    ids = torch.full((64,), -7, dtype=torch.int32, device="cuda")
    sc = torch.full((64,), float("nan"), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    want1 = _with_workspace(v1, b1.queries[0], 64)
    want2 = _with_workspace(v2, b2.queries[0], 17)
    got1 = _no_alloc(v1, b1.queries[0], 64, ids, sc, status)
    _same(got1, want1)
    _same(got1, _oracle(b1, 64))
    got2 = _no_alloc(v2, b2.queries[0], 17, ids, sc, status)
    _same(got2, want2)
    _same(got2, _oracle(b2, 17))
    # and once more on the first store: nothing carried over from call two
    _same(_no_alloc(v1, b1.queries[0], 64, ids, sc, status), want1)


def test_largest_store_the_scratch_holds():
    n = kvi.NOALLOC_MAX_FACTS
    b, v = _store(n, 64, seed=903)
    ids = torch.empty(kvi.MAX_K, dtype=torch.int32, device="cuda")
    sc = torch.empty(kvi.MAX_K, dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    want = _with_workspace(v, b.queries[0], kvi.MAX_K)
    _same(_no_alloc(v, b.queries[0], kvi.MAX_K, ids, sc, status), want)
    _same(_no_alloc(v, b.queries[0], kvi.MAX_K, ids, sc, status), _oracle(b, kvi.MAX_K))


def test_larger_store_is_rejected():
    n = kvi.NOALLOC_MAX_FACTS + 1
    b, v = _store(n, 4, seed=904)
    ids = torch.empty(8, dtype=torch.int32, device="cuda")
    sc = torch.empty(8, dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(kvi.KviError, match="KVI_NOALLOC_MAX_FACTS"):
        kvi.kvi_retrieve_topk_noalloc(v, b.queries[0], 8, ids, sc, status)
    assert kvi.kvi_last_error() and "KVI_NOALLOC_MAX_FACTS" in kvi.kvi_last_error()
