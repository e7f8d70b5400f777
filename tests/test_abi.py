"""The C ABI without a GPU: the library loads, exports every entry point that
include/kvi.h declares, and rejects bad host arguments before touching CUDA.
Also the host-only store layout call, and that the product package neither
imports the oracle nor falls back to anything when the library is missing."""
import ast
import ctypes
import os
import re

import numpy as np
import pytest

import pre_rope_kv_gb300 as kvi
from pre_rope_kv_gb300 import build as kbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    kbuild.build()
    return kvi.load_library()


def _declared():
    src = open(os.path.join(ROOT, "include", "kvi.h")).read()
    return sorted(set(re.findall(r"KVI_API\s+[\w\s\*]+?\b(kvi_\w+)\s*\(", src)))


def test_header_declares_the_exported_set():
    assert _declared() == sorted(kvi.EXPORTED_SYMBOLS)


def test_library_exports_every_declared_symbol(lib):
    raw = ctypes.CDLL(kvi.LIB_PATH)
    for name in _declared():
        assert hasattr(raw, name), name


def test_only_declared_symbols_are_exported(lib):
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", kvi.LIB_PATH], capture_output=True,
                         text=True).stdout
    exported = {l.split()[-1] for l in out.splitlines() if " T " in l}
    assert exported == set(_declared())


def test_status_strings(lib):
    for s in range(6):
        assert kvi.kvi_status_str(s)
    assert kvi.kvi_status_str(99) == "unknown status"


def test_store_layout_csr(lib):
    g = kvi.geometry(32, 8, 128, 1024)
    lens = [12, 48, 0, 30]
    offs, sizes = kvi.kvi_store_layout(g, lens)
    assert offs == [0, 12, 60, 60, 90]
    assert sizes.n_tokens == 90
    assert sizes.kv_bytes == 32 * 2 * 90 * 8 * 128 * 2
    assert sizes.emb_bytes == 4 * 1024 * 4
    assert sizes.offsets_bytes == 5 * 8


@pytest.mark.parametrize("bad", [
    dict(layers=0), dict(layers=129), dict(kv_heads=0), dict(head_dim=24), dict(head_dim=8),
    dict(head_dim=1024), dict(embed_dim=6), dict(embed_dim=0)])
def test_store_layout_rejects_bad_geometry(lib, bad):
    d = dict(layers=2, kv_heads=2, head_dim=64, embed_dim=384)
    d.update(bad)
    with pytest.raises(kvi.KviError) as e:
        kvi.kvi_store_layout(kvi.geometry(**d), [1, 2])
    assert e.value.status == kvi.ERR_INVALID_ARG


def test_store_layout_rejects_negative_length(lib):
    with pytest.raises(kvi.KviError):
        kvi.kvi_store_layout(kvi.geometry(2, 2, 64, 384), [3, -1])


def test_workspace_bytes(lib):
    a = kvi.kvi_workspace_bytes(1, 10_000, 50)
    b = kvi.kvi_workspace_bytes(64, 10_000, 50)
    assert a > 10_000 * 8 and b > 64 * 10_000 * 8 and a % 256 == 0
    for args in [(0, 10, 5), (1, 0, 5), (1, 10, 0), (1, 10, 257), (70_000, 10, 5)]:
        assert kvi.kvi_workspace_bytes(*args) == 0


class _FakeTensor:
    """Stands in for a tensor where only an address is needed: every call
    below fails validation before any pointer is dereferenced."""

    def __init__(self, addr=0x10000, n=1 << 20):
        self.addr, self.n = addr, n

    def data_ptr(self):
        return self.addr

    def numel(self):
        return self.n

    def element_size(self):
        return 1


def _store(**kw):
    g = kvi.geometry(kw.pop("L", 2), 2, kw.pop("D", 64), 384)
    v = kvi.StoreView(g, kw.pop("n_facts", 100), 1000, 0x20000, 0x30000, 0x40000, 0x50000)
    for k, val in kw.items():
        setattr(v, k, val)
    return v


def _err(fn, *a):
    # stream 0 (the legacy default stream) so that no torch CUDA call is made
    import inspect
    kw = {"stream": 0} if "stream" in inspect.signature(fn).parameters else {}
    with pytest.raises(kvi.KviError) as e:
        fn(*a, **kw)
    return e.value.status


def test_retrieve_topk_host_validation(lib):
    t = _FakeTensor()
    f = kvi.kvi_retrieve_topk
    assert _err(f, _store(), t, 0, t, t, t, t) == kvi.ERR_INVALID_ARG
    assert _err(f, _store(), t, 257, t, t, t, t) == kvi.ERR_INVALID_ARG
    assert _err(f, _store(n_facts=5), t, 6, t, t, t, t) == kvi.ERR_INVALID_ARG
    assert _err(f, _store(), _FakeTensor(0x10004), 5, t, t, t, t) \
        == kvi.ERR_INVALID_ARG                                # misaligned query
    assert _err(f, _store(emb=None), t, 5, t, t, t, t) == kvi.ERR_INVALID_ARG
    small = _FakeTensor(n=16)
    assert _err(f, _store(), t, 5, t, t, small, t) == kvi.ERR_INVALID_ARG
    assert "workspace" in kvi.kvi_last_error()
    # the scoring kernels validate every fact's extent: retrieval needs them
    for missing in ("fact_start", "fact_len"):
        assert _err(f, _store(**{missing: None}), t, 5, t, t, t, t) == kvi.ERR_INVALID_ARG
        assert "fact_start and fact_len" in kvi.kvi_last_error()
    # device-side errors (a selected fact with a bad extent, a scoring wait
    # that gave up) can only be reported through a status word: it is required
    for status in (None, _FakeTensor(0x10002)):
        assert _err(f, _store(), t, 5, t, t, t, status) == kvi.ERR_INVALID_ARG
        assert "status" in kvi.kvi_last_error()


def test_retrieve_topk_noalloc_host_validation(lib):
    t = _FakeTensor()
    f = kvi.kvi_retrieve_topk_noalloc
    assert _err(f, _store(), t, 0, t, t, t) == kvi.ERR_INVALID_ARG
    assert _err(f, _store(n_facts=kvi.NOALLOC_MAX_FACTS + 1), t, 5, t, t, t) == kvi.ERR_INVALID_ARG
    assert "KVI_NOALLOC_MAX_FACTS" in kvi.kvi_last_error()
    for status in (None, _FakeTensor(0x10002)):
        assert _err(f, _store(), t, 5, t, t, status) == kvi.ERR_INVALID_ARG
        assert "status" in kvi.kvi_last_error()


def test_selftest_wait_validation(lib):
    t = _FakeTensor()
    for bad in (0, 999, 1_000_000_001):
        assert _err(kvi.kvi_selftest_bounded_wait, bad, t) == kvi.ERR_INVALID_ARG
    assert lib.kvi_selftest_bounded_wait(1_000_000, None, None, None) == kvi.ERR_INVALID_ARG


def test_graph_host_validation(lib):
    t = _FakeTensor()
    assert _err(kvi.kvi_graph_build, _store(fact_len=None), 8, t, t) == kvi.ERR_INVALID_ARG
    assert _err(kvi.kvi_graph_build, _store(n_facts=8), 8, t, t) == kvi.ERR_INVALID_ARG
    assert _err(kvi.kvi_graph_build, _store(), 129, t, t) == kvi.ERR_INVALID_ARG
    assert _err(kvi.kvi_graph_build, _store(), 8, t, _FakeTensor(n=16)) == kvi.ERR_INVALID_ARG
    assert kvi.kvi_graph_build_workspace_bytes(8, 8) == 0
    assert kvi.kvi_graph_search_workspace_bytes(0, 100) == 0
    p = kvi.graph_search_params(16, 1, 10, 4)
    assert _err(kvi.kvi_graph_search, _store(fact_start=None), t, 8, 1, t, t, p, 8, t, t, t) \
        == kvi.ERR_INVALID_ARG
    assert _err(kvi.kvi_graph_search, _store(), t, 8, 1, t, t, kvi.graph_search_params(4, 1, 10, 4),
                8, t, t, t) == kvi.ERR_INVALID_ARG       # beam < k
    assert _err(kvi.kvi_graph_search, _store(), t, 8, 1, t, t, kvi.graph_search_params(16, 65, 10, 4),
                8, t, t, t) == kvi.ERR_INVALID_ARG       # width * degree > 512


def test_inject_paged_host_validation(lib):
    t = _FakeTensor()

    class L:
        def __init__(self, addr):
            self.a = addr
            self.shape = (2, 8, 16, 2, 64)

        def data_ptr(self):
            return self.a

    cache = kvi.paged_cache([L(0x100000), L(0x200000)], 16)
    bad_cache = kvi.paged_cache([L(0x100000)], 16)           # 1 layer, store has 2
    odd_cache = kvi.paged_cache([L(0x100000), L(0x200008)], 16)  # misaligned layer
    f = kvi.kvi_inject_paged
    assert _err(f, _store(), t, t, 0, t, 4, cache, 1e4) == kvi.ERR_INVALID_ARG
    assert _err(f, _store(), t, t, 4097, t, 4, cache, 1e4) == kvi.ERR_INVALID_ARG
    assert _err(f, _store(), t, t, 3, t, 0, cache, 1e4) == kvi.ERR_INVALID_ARG
    assert _err(f, _store(), t, t, 3, t, 4, bad_cache, 1e4) == kvi.ERR_INVALID_ARG
    assert _err(f, _store(), t, t, 3, t, 4, odd_cache, 1e4) == kvi.ERR_INVALID_ARG
    assert _err(f, _store(), t, t, 3, t, 4, cache, 0.0) == kvi.ERR_INVALID_ARG
    assert _err(f, _store(), t, t, 3, t, 4, cache, float("nan")) == kvi.ERR_INVALID_ARG
    assert _err(f, _store(kv=None), t, t, 3, t, 4, cache, 1e4) == kvi.ERR_INVALID_ARG
    assert _err(f, _store(kv=0x20008), t, t, 3, t, 4, cache, 1e4) == kvi.ERR_INVALID_ARG
    assert _err(f, _store(), None, t, 3, t, 4, cache, 1e4) == kvi.ERR_INVALID_ARG


def test_fused_host_validation(lib):
    t = _FakeTensor()

    class L:
        def __init__(self, addr):
            self.a = addr
            self.shape = (2, 8, 16, 2, 64)

        def data_ptr(self):
            return self.a

    cache = kvi.paged_cache([L(0x100000), L(0x200000)], 16)
    g = kvi.geometry(2, 2, 64, 384)
    f = kvi.kvi_retrieve_and_inject

    def call(**kw):
        a = dict(g=g, R=1, stores=t, max_facts=100, q=t, k=5, start=t, bt=t, tl=t, mb=4,
                 cache=cache, theta=1e4, ids=t, scores=t, pos=t, ws=t)
        a.update(kw)
        return _err(f, a["g"], a["R"], a["stores"], a["max_facts"], a["q"], a["k"], a["start"],
                    a["bt"], a["tl"], a["mb"], a["cache"], a["theta"], a["ids"], a["scores"],
                    a["pos"], a["ws"])

    assert call(R=0) == kvi.ERR_INVALID_ARG
    assert call(k=0) == kvi.ERR_INVALID_ARG
    assert call(max_facts=4) == kvi.ERR_INVALID_ARG
    assert call(mb=0) == kvi.ERR_INVALID_ARG
    assert call(g=kvi.geometry(3, 2, 64, 384)) == kvi.ERR_INVALID_ARG
    assert call(ws=_FakeTensor(n=64)) == kvi.ERR_INVALID_ARG
    assert call(ws=_FakeTensor(addr=0x10010)) == kvi.ERR_INVALID_ARG
    assert call(theta=-1.0) == kvi.ERR_INVALID_ARG
    assert call(mb=1 << 28) == kvi.ERR_INVALID_ARG           # max_blocks * B >= 2^31


def test_trace_stages_validation(lib):
    assert lib.kvi_trace_stages(None, 1) == kvi.ERR_INVALID_ARG
    assert lib.kvi_trace_stages(None, 0) == kvi.OK


def test_place_and_prepare_rope_validation(lib):
    t = _FakeTensor()
    assert _err(kvi.kvi_place, _store(), t, 0, 0, t) == kvi.ERR_INVALID_ARG
    assert _err(kvi.kvi_place, _store(), t, 300, 0, t) == kvi.ERR_INVALID_ARG
    assert _err(kvi.kvi_place, _store(), t, 3, -1, t) == kvi.ERR_INVALID_ARG
    assert _err(kvi.kvi_prepare_rope, 1e4, 24, 10) == kvi.ERR_INVALID_ARG
    assert _err(kvi.kvi_prepare_rope, 1e4, 64, 0) == kvi.ERR_INVALID_ARG
    assert _err(kvi.kvi_prepare_rope, -5.0, 64, 10) == kvi.ERR_INVALID_ARG


def test_product_path_never_imports_the_oracle():
    pkg = os.path.join(ROOT, "pre_rope_kv_gb300")
    for dirpath, _dirs, files in os.walk(pkg):
        for fn in files:
            path = os.path.join(dirpath, fn)
            if fn.endswith(".py"):
                tree = ast.parse(open(path).read())
                for node in ast.walk(tree):
                    if isinstance(node, ast.Import):
                        assert all(not a.name.startswith("oracle") for a in node.names), path
                    if isinstance(node, ast.ImportFrom):
                        assert not (node.module or "").startswith("oracle"), path
            if fn.endswith((".cu", ".cuh", ".h", ".cpp")):
                assert "kvi_oracle" not in open(path).read(), path


def test_missing_library_fails_loudly(tmp_path):
    import subprocess
    import sys
    code = ("import pre_rope_kv_gb300._binding as b\n"
            f"b.LIB_PATH = {str(tmp_path / 'nope.so')!r}\n"
            "try:\n    b.load_library()\nexcept RuntimeError as e:\n    print('raised', e)\n")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True)
    assert "raised" in r.stdout and "not built" in r.stdout


def test_rope_spec_validation():
    import numpy as np
    lib_ok = kvi.load_library()
    assert lib_ok is not None
    bad = [
        kvi.rope(0.0),                                   # theta must be > 0
        kvi.rope(1e4, pairing=2),                        # unknown pairing
        kvi.rope(1e4, llama3=(8.0, 4.0, 1.0, 8192.0)),   # high <= low
        kvi.rope(1e4, llama3=(0.0, 1.0, 4.0, 8192.0)),   # factor <= 0
    ]
    for spec in bad:
        with pytest.raises(kvi.KviError):
            kvi.kvi_prepare_rope_ex(spec, 64, 128)
    c = np.ones((8, 32), np.float32)
    with pytest.raises(kvi.KviError):  # a table needs an id
        kvi.kvi_prepare_rope_ex(kvi.rope(cos_table=c, sin_table=c, table_id=0), 64, 8)
    with pytest.raises(kvi.KviError):  # fewer rows than max_position
        kvi.kvi_prepare_rope_ex(kvi.rope(cos_table=c, sin_table=c, table_id=5), 64, 9)
    spec = kvi.rope(1e4)
    spec.scaling = 3
    with pytest.raises(kvi.KviError):
        kvi.kvi_prepare_rope_ex(spec, 64, 128)


def _declared_in(header):
    src = open(os.path.join(ROOT, "include", header)).read()
    return sorted(set(re.findall(r"KVI_API\s+[\w\s\*]+?\b(kvi_\w+)\s*\(", src)))


def test_debug_build_exports_the_debug_hooks_too():
    # build(debug=True): the same library with -DKVI_DEBUG_CHECKS, which adds
    # exactly the symbols of include/kvi_debug.h; the release build has none
    import subprocess
    path = kbuild.build(debug=True)
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True).stdout
    exported = {l.split()[-1] for l in out.splitlines() if " T " in l}
    assert exported == set(_declared_in("kvi.h")) | set(_declared_in("kvi_debug.h"))
    assert _declared_in("kvi_debug.h") == ["kvi_debug_stall_coarse_chunk", "kvi_debug_stall_scorer_row"]
    raw = ctypes.CDLL(kvi.LIB_PATH)
    assert not hasattr(raw, "kvi_debug_stall_scorer_row")
    assert not hasattr(raw, "kvi_debug_stall_coarse_chunk")
    # the release binding refuses the hooks instead of calling a missing symbol
    with pytest.raises(RuntimeError, match="debug build"):
        kvi.kvi_debug_stall_scorer_row(0)
    with pytest.raises(RuntimeError, match="debug build"):
        kvi.kvi_debug_stall_coarse_chunk(0, 0)


def test_stream_read_validation(lib):
    t = _FakeTensor()
    f = lib.kvi_selftest_stream_read
    assert f(None, 16, 1, t.data_ptr(), None) == kvi.ERR_INVALID_ARG
    assert f(0x10008, 16, 1, t.data_ptr(), None) == kvi.ERR_INVALID_ARG   # misaligned
    assert f(0x10000, 24, 1, t.data_ptr(), None) == kvi.ERR_INVALID_ARG   # not 16-byte words
    assert f(0x10000, 16, 0, t.data_ptr(), None) == kvi.ERR_INVALID_ARG
    assert f(0x10000, 16, 9, t.data_ptr(), None) == kvi.ERR_INVALID_ARG
    assert f(0x10000, 16, 1, None, None) == kvi.ERR_INVALID_ARG
