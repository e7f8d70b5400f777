"""Parity harness: run the CUDA path through the C ABI and compare it with the
float64 oracle, element by element.

Tolerances ("InferScale: GPU-Native KV Injection for Personalized LLM
Serving", Section 5.1 / Theorem 6 make the rotation exact in real
arithmetic; the stored result is bf16):
  - selected fact ids, placements and V rows: bit-exact;
  - rotated K: |gpu - x| <= 2^-8 |x| + 1e-6 per element, x the oracle's
    float64 value (one bf16 rounding of a float32 result that is within a few
    float32 ulps of x);
  - similarity scores: |gpu - s| <= 1e-4 |s| + 1e-7;
  - every pool element the injection must not touch keeps its canary bits.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import pre_rope_kv_gb300 as kvi
from pre_rope_kv_gb300 import build as kvi_build
from tests import synth

K_REL = 2.0 ** -8
K_ABS = 1e-6
S_REL = 1e-4
S_ABS = 1e-7


def ensure_built():
    kvi_build.build()
    kvi.load_library()
    oracle.build()


def geometry_of(w: synth.Workload):
    return kvi.geometry(w.layers, w.kv_heads, w.head_dim, w.embed_dim)


def views_of(b: synth.Built):
    g = geometry_of(b.w)
    return [kvi.store_view(g, b.kv, s.emb, s.fact_start, s.fact_len, n_tokens=b.kv.shape[2])
            for s in b.stores]


def cache_of(b: synth.Built):
    return kvi.paged_cache([b.pool[l] for l in range(b.w.layers)], b.w.block_size)


def device_views(views):
    packed = kvi.pack_store_views(views)
    return torch.frombuffer(bytearray(packed), dtype=torch.uint8).cuda()


class Fused:
    """Device buffers of one kvi_retrieve_and_inject call."""

    def __init__(self, b: synth.Built, k: int | None = None, rope=None):
        w = b.w
        self.b = b
        self.k = k or b.k
        self.rope = rope  # a kvi.Rope for the _ex call, or None for rope_theta
        R = w.requests
        self.g = geometry_of(w)
        self.d_views = device_views(views_of(b))
        self.cache = cache_of(b)
        self.ids = torch.empty((R, self.k), dtype=torch.int32, device="cuda")
        self.scores = torch.empty((R, self.k), dtype=torch.float32, device="cuda")
        self.pos = torch.empty((R, self.k), dtype=torch.int32, device="cuda")
        self.ws = torch.empty(kvi.kvi_workspace_bytes(R, w.n_facts, self.k), dtype=torch.uint8,
                              device="cuda")
        self.status = torch.zeros(1, dtype=torch.int32, device="cuda")
        self.start = torch.from_numpy(b.start_pos).cuda()
        self.bt = torch.from_numpy(b.block_tables).cuda()
        self.tl = torch.from_numpy(b.table_lens).cuda()

    def __call__(self, stream=None):
        w = self.b.w
        if self.rope is not None:
            kvi.kvi_retrieve_and_inject_ex(
                self.g, w.requests, self.d_views, w.n_facts, self.b.queries, self.k, self.start,
                self.bt, self.tl, self.b.max_blocks, self.cache, self.rope, self.ids,
                self.scores, self.pos, self.ws, self.status, stream)
            return
        kvi.kvi_retrieve_and_inject(
            self.g, w.requests, self.d_views, w.n_facts, self.b.queries, self.k, self.start,
            self.bt, self.tl, self.b.max_blocks, self.cache, w.rope_theta, self.ids, self.scores,
            self.pos, self.ws, self.status, stream)

    def results(self):
        torch.cuda.synchronize()
        return (self.ids.cpu().numpy(), self.scores.cpu().numpy(), self.pos.cpu().numpy(),
                int(self.status.item()))


def run_fused(b: synth.Built, k: int | None = None, rope=None):
    f = Fused(b, k, rope)
    f()
    return f.results()


def oracle_select(b: synth.Built, k: int | None = None):
    """Per request: (scores[N] float64, sel[k], pos[k], T) from the oracle."""
    k = k or b.k
    out = []
    for r, st in enumerate(b.stores):
        s = oracle.scores(b.queries_np[r], st.emb_np)
        sel = oracle.topk(s, k)
        pos, T = oracle.place(sel, st.len_np, int(b.start_pos[r]))
        out.append((s, sel, pos, T))
    return out


def check_selection(ids, scores, pos, orc):
    for r, (s, sel, opos, _T) in enumerate(orc):
        if not np.array_equal(ids[r], sel):
            order = np.lexsort((np.arange(s.shape[0]), -s))
            kk = sel.shape[0]
            gap = s[order[kk - 1]] - s[order[kk]] if order.shape[0] > kk else float("inf")
            raise AssertionError(
                f"request {r}: ids differ from the oracle\n gpu    {ids[r].tolist()}\n"
                f" oracle {sel.tolist()}\n k-th/(k+1)-th score gap {gap:.3e}")
        ref = s[sel]
        err = np.abs(scores[r].astype(np.float64) - ref)
        assert np.all(err <= S_REL * np.abs(ref) + S_ABS), f"request {r}: scores off {err.max()}"
        assert np.array_equal(pos[r].astype(np.int64), opos), f"request {r}: positions differ"


def _pool_arrays(b: synth.Built):
    bits = b.pool.view(torch.int16).cpu().numpy().view(np.uint16)
    vals = b.pool.float().cpu().numpy().astype(np.float64)
    return bits, vals


def check_k_v(gk, gv_bits, ek, ev_bits, where=""):
    err = np.abs(gk - ek)
    bad = err > K_REL * np.abs(ek) + K_ABS
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{where}: K off at {tuple(i)}: gpu {gk[tuple(i)]!r} oracle "
                             f"{ek[tuple(i)]!r} ({int(bad.sum())} elements)")
    if not np.array_equal(gv_bits, ev_bits):
        i = np.argwhere(gv_bits != ev_bits)[0]
        raise AssertionError(f"{where}: V bits differ at {tuple(i)}")


def check_pool_full(b: synth.Built, placements, rope: dict | None = None):
    """placements: per request (ids[n], starts[n]) to expect.  Small pools:
    the whole pool is compared with the oracle's expected pool.  rope: the
    oracle's rope_spec for a rotary variant (None: rotate-half, theta)."""
    kv_np = b.kv_np
    if kv_np is None:  # drawn on the device: read the store bits back
        kv_np = b.kv.view(torch.int16).cpu().numpy().view(np.uint16)
    bits, vals = _pool_arrays(b)
    L, _, NB, B, H, D = b.pool.shape
    written_all = np.zeros(bits.shape, np.uint8)
    for r, (ids, starts) in enumerate(placements):
        st = b.stores[r]
        bt = b.block_tables[r, :b.table_lens[r]]
        rc, expect, written = oracle.inject_expected(
            kv_np, st.start_np, st.len_np, ids, starts, bt, NB, B, b.w.rope_theta, rope)
        assert rc == oracle.OK, f"oracle rejected request {r}: {rc}"
        m = written.astype(bool)
        assert not (written_all.astype(bool) & m).any(), "requests overlap"
        written_all |= written
        mk, mv = m[:, 0], m[:, 1]
        ev_bits = (expect[:, 1][mv].astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
        check_k_v(vals[:, 0][mk], bits[:, 1][mv], expect[:, 0][mk], ev_bits, f"request {r}")
    untouched = bits[written_all == 0]
    assert np.all(untouched == synth.CANARY_BITS), \
        f"{int((untouched != synth.CANARY_BITS).sum())} canary elements overwritten"


def token_list(b: synth.Built, placements):
    """Flat arrays over every injected token: request, fact, t, position."""
    rr, ff, tt, pp = [], [], [], []
    for r, (ids, starts) in enumerate(placements):
        lens = b.stores[r].len_np[ids]
        for j in range(len(ids)):
            n = int(lens[j])
            rr.append(np.full(n, r))
            ff.append(np.full(n, ids[j]))
            tt.append(np.arange(n))
            pp.append(int(starts[j]) + np.arange(n))
    cat = lambda x: np.concatenate(x) if x else np.zeros(0, np.int64)
    return cat(rr).astype(np.int64), cat(ff).astype(np.int64), cat(tt), cat(pp).astype(np.int64)


def check_pool_sampled(b: synth.Built, placements, n_samples: int, seed: int = 0,
                       rope: dict | None = None):
    """Large pools: compare sampled tokens' rows (all layers, K and V) with
    the oracle, reading the store bits back from the device."""
    rr, ff, tt, pp = token_list(b, placements)
    assert rr.shape[0] > 0
    rng = np.random.default_rng(seed)
    pick = rng.choice(rr.shape[0], size=min(n_samples, rr.shape[0]), replace=False)
    # always include each request's first and last token
    firsts = np.unique(np.searchsorted(rr, np.arange(b.w.requests)))
    lasts = np.unique(np.searchsorted(rr, np.arange(b.w.requests), side="right") - 1)
    pick = np.unique(np.concatenate([pick, firsts[firsts < rr.shape[0]], lasts[lasts >= 0]]))
    NB, B = b.num_blocks, b.w.block_size
    blk = np.empty(pick.shape[0], np.int32)
    off = np.empty(pick.shape[0], np.int32)
    rows = np.empty(pick.shape[0], np.int64)
    for n, i in enumerate(pick):
        r = int(rr[i])
        sl = oracle.slot(int(pp[i]), b.block_tables[r, :b.table_lens[r]], B, NB)
        assert sl is not None
        blk[n], off[n] = sl
        rows[n] = int(b.stores[r].start_np[ff[i]]) + int(tt[i])
    bi = torch.from_numpy(blk.astype(np.int64)).cuda()
    oi = torch.from_numpy(off.astype(np.int64)).cuda()
    ri = torch.from_numpy(rows).cuda()
    gpu = b.pool[:, :, bi, oi]  # [L][2][S][H][D]
    gbits = gpu.view(torch.int16).cpu().numpy().view(np.uint16)
    gvals = gpu.float().cpu().numpy().astype(np.float64)
    sbits = b.kv[:, :, ri].view(torch.int16).cpu().numpy().view(np.uint16)
    for n, i in enumerate(pick):
        ek, ev = oracle.token_rows_from_rows(sbits[:, 0, n], sbits[:, 1, n], b.w.rope_theta,
                                             int(pp[i]), rope)
        check_k_v(gvals[:, 0, n], gbits[:, 1, n], ek, ev,
                  f"request {rr[i]} fact {ff[i]} token {tt[i]} pos {pp[i]}")
    return pick.shape[0]


# Lines of element counts from the exhaustive checks, printed at the end of
# a pytest session (tests/conftest.py).
PARITY_LOG: list[str] = []


def check_pool_exhaustive(b: synth.Built, placements, rope: dict | None = None,
                          chunk_bytes: int = 1 << 30, label: str = ""):
    """Large pools: every injected token's rows (all layers and heads, K and
    V) compared element by element with the oracle.  Tokens are taken in
    chunks: the pool rows written for them and the store rows they came
    from are gathered on the device, copied to pinned host memory, and the
    oracle's check_rows runs over the chunk on all host cores while the next
    chunk is gathered.  Returns (tokens, elements compared, host threads)."""
    import concurrent.futures as cf
    import os
    rr, ff, tt, pp = token_list(b, placements)
    n_tok = rr.shape[0]
    assert n_tok > 0
    w = b.w
    L, H, D, B = w.layers, w.kv_heads, w.head_dim, w.block_size
    NB = b.num_blocks
    tok_bytes = L * 2 * H * D * 2
    per = max(1, chunk_bytes // tok_bytes)
    slot = np.empty(n_tok, np.int64)
    row = np.empty(n_tok, np.int64)
    for r in range(w.requests):
        m = rr == r
        if not m.any():
            continue
        blk, off = oracle.slots(pp[m], b.block_tables[r, :b.table_lens[r]], B, NB)
        assert np.all(blk >= 0), f"request {r}: a position outside its block table"
        slot[m] = blk.astype(np.int64) * B + off
        row[m] = b.stores[r].start_np[ff[m]] + tt[m]
    pool_v = b.pool.view(torch.int16).view(L * 2, NB * B, H * D)
    kv_v = b.kv.view(torch.int16).view(L * 2, b.kv.shape[2], H * D)
    threads = os.cpu_count() or 1
    bufs = [(torch.empty((L * 2, per, H * D), dtype=torch.int16).pin_memory(),
             torch.empty((L * 2, per, H * D), dtype=torch.int16).pin_memory()) for _ in range(2)]
    slot_d = torch.from_numpy(slot).cuda()
    row_d = torch.from_numpy(row).cuda()

    def check(i, a, n):
        src_h, got_h = bufs[i]
        src = src_h[:, :n].numpy().view(np.uint16).reshape(L, 2, n, H, D)
        got = got_h[:, :n].numpy().view(np.uint16).reshape(L, 2, n, H, D)
        bad_k, bad_v, first = oracle.check_rows(src, got, pp[a:a + n], w.rope_theta, K_REL, K_ABS,
                                                rope, threads=threads)
        if bad_k or bad_v:
            l, c, t, h, e = np.unravel_index(first, (L, 2, n, H, D))
            j = a + t
            raise AssertionError(
                f"{bad_k} K and {bad_v} V elements off the oracle; first: request {rr[j]} fact "
                f"{ff[j]} token {tt[j]} position {pp[j]} layer {l} {'KV'[c]} head {h} elem {e}: "
                f"gpu bits {got[l, c, t, h, e]:#06x}, store bits {src[l, c, t, h, e]:#06x}")

    with cf.ThreadPoolExecutor(max_workers=1) as ex:
        pending = None
        for ci, a in enumerate(range(0, n_tok, per)):
            n = min(per, n_tok - a)
            i = ci % 2
            if pending is not None and pending[1] == i:
                pending[0].result()  # this buffer pair is free again
                pending = None
            src_h, got_h = bufs[i]
            src_h[:, :n].copy_(kv_v.index_select(1, row_d[a:a + n]))
            got_h[:, :n].copy_(pool_v.index_select(1, slot_d[a:a + n]))
            if pending is not None:
                pending[0].result()
            pending = (ex.submit(check, i, a, n), i)
        if pending is not None:
            pending[0].result()
    elements = n_tok * L * 2 * H * D
    PARITY_LOG.append(f"{label or w.name}: {n_tok} tokens, {elements} elements (K and V, all "
                      f"layers and heads) compared with the oracle on {threads} host threads")
    return n_tok, elements, threads


def check_canaries_by_row(b: synth.Built, placements):
    """Every (block, offset) row the oracle's placement maps a token to is
    written in every layer for K and V; every other row keeps its canary."""
    NB, B = b.num_blocks, b.w.block_size
    mask = np.zeros((NB, B), bool)
    total = 0
    for r, (ids, starts) in enumerate(placements):
        lens = b.stores[r].len_np[ids]
        pos = np.concatenate([int(starts[j]) + np.arange(int(lens[j])) for j in range(len(ids))])
        blk, off = oracle.slots(pos, b.block_tables[r, :b.table_lens[r]], B, NB)
        assert np.all(blk >= 0)
        assert not mask[blk, off].any(), "positions overlap"
        mask[blk, off] = True
        total += pos.shape[0]
    assert int(mask.sum()) == total
    m = torch.from_numpy(mask).cuda()
    canary = synth.CANARY_BITS - (1 << 16)
    for l in range(b.w.layers):
        for c in range(2):
            touched = (b.pool[l, c].view(torch.int16) != canary).flatten(2).any(dim=2)
            if not torch.equal(touched, m):
                extra = int((touched & ~m).sum())
                missing = int((~touched & m).sum())
                raise AssertionError(f"layer {l} {'KV'[c]}: {extra} rows touched outside the "
                                     f"placement, {missing} placed rows untouched")


def placements_from_oracle(orc):
    return [(sel, pos) for (_s, sel, pos, _T) in orc]
