"""Store files on the GPU: kvi_store_save writes what the format describes
(read back by tests/store_file.py, which shares no code with the library),
kvi_store_load restores the same bytes into HBM or pinned host memory, a
loaded store passes the oracle's parity bar through the fused call, and
damaged files are refused."""
import os

import numpy as np
import pytest
import torch

import pre_rope_kv_gb300 as kvi
from tests import kvi_check as kc
from tests import store_file as sf
from tests import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    kc.ensure_built()


def W(**kw):
    base = dict(name="file", layers=2, kv_heads=4, head_dim=128, rope_theta=5e5, block_size=16,
                n_facts=200, len_lo=1, len_hi=20, len_dist="uniform", embed_dim=256, requests=1,
                k=20, start=5, start_hi=0, seed=900, store="dense")
    base.update(kw)
    return synth.Workload(**base)


def _view(b, kv=None, kv_host=False):
    st = b.stores[0]
    kv = b.kv if kv is None else kv
    return kvi.store_view(kc.geometry_of(b.w), kv, st.emb, st.fact_start, st.fact_len,
                          n_tokens=kv.shape[2], kv_host=kv_host)


def _bytes(t):
    return t.detach().contiguous().cpu().view(torch.uint8).numpy().tobytes()


def test_save_writes_the_documented_format(tmp_path):
    b = synth.build_workload(W())
    p = os.path.join(str(tmp_path), "s.kvs")
    kvi.kvi_store_save(p, _view(b))
    torch.cuda.synchronize()
    f = sf.read(p)
    w = b.w
    assert f["magic"] == sf.MAGIC and f["version"] == 1 and f["header_bytes"] == 128
    assert f["g"] == (w.layers, w.kv_heads, w.head_dim, w.embed_dim)
    assert f["n"] == w.n_facts and f["t"] == b.kv.shape[2]
    assert f["header_hash_ok"] and f["gaps_zero"] and f["reserved"] == b"\0" * 16
    assert f["size"] == f["layout"]["file"]
    st = b.stores[0]
    assert f["fact_start"] == _bytes(st.fact_start) and f["fact_len"] == _bytes(st.fact_len)
    assert f["emb"] == _bytes(st.emb) and f["kv"] == _bytes(b.kv)
    assert f["extents_hash"] == sf.fnv1a(f["fact_len"], sf.fnv1a(f["fact_start"]))
    assert f["payload_hash"] == sf.payload_hash(f["emb"] + f["kv"])


def test_save_from_a_host_store_writes_the_same_file(tmp_path):
    b = synth.build_workload(W(seed=901))
    p1 = os.path.join(str(tmp_path), "dev.kvs")
    p2 = os.path.join(str(tmp_path), "host.kvs")
    kvi.kvi_store_save(p1, _view(b))
    kv_host = b.kv.cpu().pin_memory()
    kvi.kvi_store_save(p2, _view(b, kv_host, kv_host=True))
    assert open(p1, "rb").read() == open(p2, "rb").read()


@pytest.mark.parametrize("kv_host", [False, True])
def test_loaded_store_round_trips_and_passes_parity(tmp_path, kv_host):
    w = W(seed=902 + kv_host, n_facts=300, k=25)
    b = synth.build_workload(w)
    p = os.path.join(str(tmp_path), "rt.kvs")
    kvi.kvi_store_save(p, _view(b))
    g, kv, emb, fs, fl = kvi.load_store(p, kv_host=kv_host)
    torch.cuda.synchronize()
    st = b.stores[0]
    assert kv.is_cuda != kv_host
    assert torch.equal(kv.cpu().view(torch.int16), b.kv.cpu().view(torch.int16))
    assert torch.equal(emb.cpu(), st.emb.cpu())
    assert torch.equal(fs.cpu(), st.fact_start.cpu()) and torch.equal(fl.cpu(), st.fact_len.cpu())
    # the loaded store through the fused call, against the oracle on the
    # original (byte-identical) store
    view = kvi.store_view(g, kv, emb, fs, fl, n_tokens=kv.shape[2], kv_host=kv_host)
    f = kc.Fused(b)
    f.d_views = kc.device_views([view])
    f()
    ids, scores, pos, status = f.results()
    assert status == 0
    orc = kc.oracle_select(b)
    kc.check_selection(ids, scores, pos, orc)
    kc.check_pool_full(b, kc.placements_from_oracle(orc))
    del kv


def test_many_chunks_round_trip(tmp_path):
    # about 100 MB of K/V: several passes through the 32 MB bounce buffer
    w = W(seed=904, kv_heads=8, n_facts=400, len_lo=12, len_hi=48)
    b = synth.build_workload(w)
    assert b.kv.numel() * 2 > 3 * (32 << 20)
    p = os.path.join(str(tmp_path), "big.kvs")
    kvi.kvi_store_save(p, _view(b))
    g, kv, emb, fs, fl = kvi.load_store(p)
    torch.cuda.synchronize()
    assert torch.equal(kv.view(torch.int16), b.kv.view(torch.int16))
    assert torch.equal(emb, b.stores[0].emb)


def _load_status(p, info):
    g = info.g
    kv = torch.empty((g.layers, 2, info.n_tokens, g.kv_heads, g.head_dim), dtype=torch.bfloat16,
                     device="cuda")
    emb = torch.empty((info.n_facts, g.embed_dim), dtype=torch.float32, device="cuda")
    fs = torch.empty(info.n_facts, dtype=torch.int64, device="cuda")
    fl = torch.empty(info.n_facts, dtype=torch.int32, device="cuda")
    lib = kvi.load_library()
    return lib.kvi_store_load(os.fsencode(p), kv.data_ptr(), emb.data_ptr(), fs.data_ptr(),
                              fl.data_ptr(), 0)


def test_damaged_payload_and_extents_are_refused(tmp_path):
    b = synth.build_workload(W(seed=905, n_facts=50))
    p = os.path.join(str(tmp_path), "d.kvs")
    kvi.kvi_store_save(p, _view(b))
    info = kvi.kvi_store_file_info_read(p)
    good = open(p, "rb").read()
    assert _load_status(p, info) == kvi.OK
    lay = sf.layout((info.g.layers, info.g.kv_heads, info.g.head_dim, info.g.embed_dim),
                    info.n_facts, info.n_tokens)
    # one flipped bit in K/V, then one in an embedding
    for at in (lay["kv"] + lay["kv_bytes"] // 2, lay["emb"] + 5):
        bad = bytearray(good)
        bad[at] ^= 0x10
        open(p, "wb").write(bytes(bad))
        assert _load_status(p, info) == kvi.ERR_IO
        assert "payload hash" in kvi.kvi_last_error()
    # a flipped extent byte: the extents hash no longer matches
    bad = bytearray(good)
    bad[lay["start"] + 8] ^= 0x01
    open(p, "wb").write(bytes(bad))
    assert _load_status(p, info) == kvi.ERR_IO
    assert "extents hash" in kvi.kvi_last_error()
    # a consistent file (hashes recomputed) whose last fact runs past the rows
    f = sf.read(p)
    starts = np.frombuffer(f["fact_start"], "<i8").copy()
    lens = np.frombuffer(f["fact_len"], "<i4").copy()
    starts[1] ^= 1  # undo the flip
    starts[-1] = info.n_tokens - int(lens[-1]) + 1
    open(p, "wb").write(sf.build(f["g"], starts, lens, f["emb"], f["kv"], f["t"]))
    assert _load_status(p, info) == kvi.ERR_IO
    assert "outside the store" in kvi.kvi_last_error()


def test_arena_view_round_trips(tmp_path):
    # extents scattered through more rows than the facts use (an arena
    # stand-in): the file keeps every row and the extents as they are
    b = synth.build_workload(W(seed=906, n_facts=60, len_lo=1, len_hi=6))
    st = b.stores[0]
    T = 400
    rng = np.random.default_rng(907)
    lens = st.len_np.astype(np.int32)
    starts = np.sort(rng.choice(T - 6, size=60, replace=False)).astype(np.int64)
    g = kc.geometry_of(b.w)
    kv = torch.randn((b.w.layers, 2, T, b.w.kv_heads, b.w.head_dim), device="cuda").to(torch.bfloat16)
    fs = torch.from_numpy(starts).cuda()
    fl = torch.from_numpy(lens).cuda()
    view = kvi.store_view(g, kv, st.emb, fs, fl, n_tokens=T)
    p = os.path.join(str(tmp_path), "arena.kvs")
    kvi.kvi_store_save(p, view)
    f = sf.read(p)
    assert f["t"] == T and f["fact_start"] == starts.astype("<i8").tobytes()
    g2, kv2, emb2, fs2, fl2 = kvi.load_store(p)
    torch.cuda.synchronize()
    assert torch.equal(kv2.view(torch.int16), kv.view(torch.int16))
    assert torch.equal(fs2, fs) and torch.equal(fl2, fl) and torch.equal(emb2, st.emb)
