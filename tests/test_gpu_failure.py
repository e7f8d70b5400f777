"""Failure detection on the GPU without a fault: a bounded wait that runs out.

Every staging wait in the library is bounded by a time limit.  The
diagnostic kvi_selftest_bounded_wait waits, with the inject kernel's own
helper, on a barrier that nothing completes.  The wait must end near its
limit with KVI_ERR_TIMEOUT in the status word, and the context must stay
usable: a retrieval right after it still matches the oracle."""
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


@pytest.mark.parametrize("limit_ms", [1, 20])
def test_a_wait_that_never_completes_times_out_and_the_context_stays_usable(limit_ms):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    elapsed = torch.zeros(1, dtype=torch.int64, device="cuda")
    kvi.kvi_selftest_bounded_wait(limit_ms * 1_000_000, status, elapsed)
    torch.cuda.synchronize()
    assert int(status.item()) == kvi.ERR_TIMEOUT
    ns = int(elapsed.item())
    assert limit_ms * 1_000_000 <= ns < limit_ms * 1_000_000 + 50_000_000, ns
    # the status word keeps the first error: a second timeout leaves it as is
    kvi.kvi_selftest_bounded_wait(1_000_000, status)
    torch.cuda.synchronize()
    assert int(status.item()) == kvi.ERR_TIMEOUT
    # the context still runs the path
    w = synth.Workload(name="after", layers=2, kv_heads=2, head_dim=64, rope_theta=1e4, block_size=16,
                       n_facts=300, len_lo=1, len_hi=8, len_dist="uniform", embed_dim=128, requests=1,
                       k=10, start=0, start_hi=0, seed=990 + limit_ms, store="dense")
    b = synth.build_workload(w, with_pool=False)
    view = kc.views_of(b)[0]
    ids = torch.empty(10, dtype=torch.int32, device="cuda")
    sc = torch.empty(10, dtype=torch.float32, device="cuda")
    ws = torch.empty(kvi.kvi_workspace_bytes(1, w.n_facts, 10), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvi.kvi_retrieve_topk(view, b.queries[0], 10, ids, sc, ws, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    want = oracle.topk(oracle.scores(b.queries_np[0], b.stores[0].emb_np), 10)
    assert np.array_equal(ids.cpu().numpy(), want)


@pytest.mark.parametrize("where", ["device", "pinned_host"])
def test_stream_read_diagnostic_reads_every_word(where):
    # the read diagnostic the bench uses for the host link's ceiling: its
    # checksum is the wrapping sum of the 32-bit words read
    n = (64 << 20) + 48  # not a multiple of the grid's stride
    g = torch.Generator().manual_seed(5)
    words = torch.randint(0, 2 ** 31 - 1, (n // 4,), generator=g, dtype=torch.int64).to(torch.int32)
    buf = words.cuda() if where == "device" else words.pin_memory()
    out = torch.zeros(1, dtype=torch.int64, device="cuda")
    kvi.kvi_selftest_stream_read(buf.data_ptr(), n, 2, out)
    torch.cuda.synchronize()
    want = int(words.numpy().astype(np.uint32).astype(np.uint64).sum(dtype=np.uint64))
    assert int(out.item()) & (2 ** 64 - 1) == want & (2 ** 64 - 1)
