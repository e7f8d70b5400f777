"""Store files without a GPU: kvi_store_file_info_read (host only) against
files written by tests/store_file.py from the format's description, valid
and damaged.  The format's two hashes are pinned by FNV-1a's published test
value, so the writer here and the library cannot share a wrong hash."""
import os

import numpy as np
import pytest

import pre_rope_kv_gb300 as kvi
from pre_rope_kv_gb300 import build as kbuild
from tests import store_file as sf

G = (2, 2, 16, 8)  # L, H, D, E


@pytest.fixture(scope="module")
def lib():
    kbuild.build()
    return kvi.load_library()


def _parts(n=3, t=10, seed=0):
    rng = np.random.default_rng(seed)
    lens = rng.integers(0, 4, n).astype(np.int32)
    starts = np.concatenate([[0], np.cumsum(lens)[:-1]]).astype(np.int64)
    t = max(t, int(lens.sum()))
    emb = rng.standard_normal((n, G[3])).astype(np.float32).tobytes()
    kv = rng.integers(0, 1 << 16, G[0] * 2 * t * G[1] * G[2], dtype=np.uint16).tobytes()
    return starts, lens, emb, kv, t


def _write(tmp_path, name, data):
    p = os.path.join(str(tmp_path), name)
    open(p, "wb").write(data)
    return p


def test_fnv1a_matches_the_published_test_values():
    # FNV-1a 64 of "a" and of "foobar" (the FNV authors' test vectors)
    assert sf.fnv1a(b"") == 0xCBF29CE484222325
    assert sf.fnv1a(b"a") == 0xAF63DC4C8601EC8C
    assert sf.fnv1a(b"foobar") == 0x85944171F73967E8


def test_payload_hash_lanes():
    # one word per lane: each lane is one FNV step from its own basis
    w = [1, 2, 3, 4]
    h = [((sf.FNV_BASIS + j) ^ w[j]) * sf.FNV_PRIME & sf.MASK for j in range(4)]
    rot = lambda x, r: ((x << r) | (x >> (64 - r))) & sf.MASK
    want = h[0] ^ rot(h[1], 16) ^ rot(h[2], 32) ^ rot(h[3], 48)
    assert sf.payload_hash(np.array(w, dtype="<u8").tobytes()) == want


def test_info_of_a_valid_file(lib, tmp_path):
    starts, lens, emb, kv, t = _parts()
    p = _write(tmp_path, "ok.kvs", sf.build(G, starts, lens, emb, kv, t))
    info = kvi.kvi_store_file_info_read(p)
    assert (info.g.layers, info.g.kv_heads, info.g.head_dim, info.g.embed_dim) == G
    assert (info.n_facts, info.n_tokens) == (3, t)
    assert info.kv_bytes == len(kv) and info.emb_bytes == len(emb)


@pytest.mark.parametrize("damage", [
    "magic", "version", "header_hash", "offsets", "reserved", "truncated", "extended",
    "geometry", "no_facts"])
def test_damaged_headers_are_rejected(lib, tmp_path, damage):
    starts, lens, emb, kv, t = _parts()
    g = G
    kw = {}
    if damage == "magic":
        kw["magic"] = b"KVISTORX"
    elif damage == "version":
        kw["version"] = 2
    elif damage == "header_hash":
        kw["header_hash"] = 12345
    elif damage == "offsets":
        lay = sf.layout(G, 3, t)
        kw["offsets"] = [lay["start"], lay["len"], lay["emb"] + 4096, lay["kv"] + 4096, lay["file"] + 4096]
    elif damage == "reserved":
        kw["reserved"] = b"\1" + b"\0" * 15
    elif damage == "geometry":
        g = (2, 2, 10, 8)  # head_dim not a multiple of 16
        kv = b"\0" * sf.layout(g, 3, t)["kv_bytes"]
    data = sf.build(g, starts, lens, emb, kv, t, **kw)
    if damage == "truncated":
        data = data[:-2]
    elif damage == "extended":
        data = data + b"\0" * 16
    elif damage == "no_facts":
        data = sf.build(G, [], np.zeros(0, np.int32), b"", kv, t)
    p = _write(tmp_path, "bad.kvs", data)
    with pytest.raises(kvi.KviError) as e:
        kvi.kvi_store_file_info_read(p)
    assert e.value.status == kvi.ERR_IO


def test_missing_file_and_null_arguments(lib, tmp_path):
    with pytest.raises(kvi.KviError) as e:
        kvi.kvi_store_file_info_read(os.path.join(str(tmp_path), "absent.kvs"))
    assert e.value.status == kvi.ERR_IO
    info = kvi.StoreFileInfo()
    assert lib.kvi_store_file_info_read(None, info) == kvi.ERR_INVALID_ARG
    assert lib.kvi_store_save(None, None) == kvi.ERR_INVALID_ARG
    assert lib.kvi_store_load(None, None, None, None, None, 0) == kvi.ERR_INVALID_ARG
