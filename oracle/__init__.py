"""Float64 CPU oracle for the retrieve-and-inject path (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg import this package.  The product path (``pre_rope_kv_gb300``) never does,
and the two share no code: this module wraps the plain C file
``kvi_oracle.c`` (single thread, float64, no fused multiply-add) with ctypes
and numpy marshalling, nothing else.

Method followed: "InferScale: GPU-Native KV Injection for Personalized LLM
Serving" (pith.science review of arXiv 2607.27090) -- Figure 2 caption
(shared fact_id, top-k retrieval, positioning by Chunked RoPE), Section 5.1 /
Theorem 6 (pre-RoPE keys rotated at injection, R_a^T R_b = R_{b-a}) and the
Section 3.4 premise (scatter-copy into vLLM's paged blocks).  See the C file
for the readings taken where the page is silent.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kvi_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libkvi_oracle.so")

OK, BAD_ARG, OUT_OF_RANGE, CAPACITY = 0, 1, 2, 3
PAIR_HALF, PAIR_INTERLEAVED = 0, 1

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile kvi_oracle.c with gcc into oracle/_build/libkvi_oracle.so."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call([
        "gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math",
        "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        # KVI_ORACLE_LIB lets the mutation tests load a deliberately broken
        # copy of the oracle, to prove that the pins catch it.
        lib = ctypes.CDLL(os.environ.get("KVI_ORACLE_LIB") or build())
        P = ctypes.c_void_p
        i32, i64, f64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_double
        lib.kvo_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.kvo_bf16_to_double.restype = f64
        lib.kvo_scores.argtypes = [P, P, i64, i64, P]
        lib.kvo_scores.restype = None
        lib.kvo_topk.argtypes = [P, i64, i32, P]
        lib.kvo_topk.restype = ctypes.c_int
        lib.kvo_place.argtypes = [P, i32, P, i64, i64, P]
        lib.kvo_place.restype = i64
        lib.kvo_rope_omega.argtypes = [f64, i32, P]
        lib.kvo_rope_omega.restype = None
        lib.kvo_rotate.argtypes = [P, i32, f64, f64, P]
        lib.kvo_rotate.restype = None
        lib.kvo_slot.argtypes = [i64, P, i32, i32, i32, P, P]
        lib.kvo_slot.restype = ctypes.c_int
        lib.kvo_slots.argtypes = [P, i64, P, i32, i32, i32, P, P]
        lib.kvo_slots.restype = None
        lib.kvo_token_rows.argtypes = [P, i32, i32, i32, i64, i64, f64, i64, P, P]
        lib.kvo_token_rows.restype = ctypes.c_int
        lib.kvo_inject_expected.argtypes = [
            P, i32, i32, i32, i64, P, P, i64, P, P, i32, P, i32, i32, i32, f64, P, P]
        lib.kvo_inject_expected.restype = ctypes.c_int
        lib.kvo_request.argtypes = [
            P, P, i64, i64, i32, P, i32, i32, i32, i64, P, P, i64, f64, P, P, P, P, i64]
        lib.kvo_request.restype = i64
        lib.kvo_rotate_pairs.argtypes = [P, i32, P, i32, f64, P]
        lib.kvo_rotate_pairs.restype = None
        lib.kvo_rotate_cs.argtypes = [P, i32, P, P, i32, P]
        lib.kvo_rotate_cs.restype = None
        lib.kvo_rope_omega_llama3.argtypes = [f64, i32, f64, f64, f64, f64, P]
        lib.kvo_rope_omega_llama3.restype = None
        lib.kvo_token_rows_ex.argtypes = [P, i32, i32, i32, i64, i64, P, i32, P, P, i64, i64, P, P]
        lib.kvo_token_rows_ex.restype = ctypes.c_int
        lib.kvo_inject_expected_ex.argtypes = [
            P, i32, i32, i32, i64, P, P, i64, P, P, i32, P, i32, i32, i32, P, i32, P, P, i64,
            P, P]
        lib.kvo_inject_expected_ex.restype = ctypes.c_int
        lib.kvo_check_rows.argtypes = [P, P, i32, i32, i32, i64, i64, i64, P, P, i32, P, P, i64,
                                       f64, f64, P, P, P]
        lib.kvo_check_rows.restype = ctypes.c_int
        lib.kvo_graph_build.argtypes = [P, i64, i64, i32, P]
        lib.kvo_graph_build.restype = ctypes.c_int
        lib.kvo_graph_search.argtypes = [P, P, i64, i64, P, i32, P, i32, i32, i32, i32, i32, P,
                                         P, P]
        lib.kvo_graph_search.restype = i32
        _lib = lib
        return lib


def _c(a: np.ndarray, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def bf16_to_double(bits) -> float:
    return _load().kvo_bf16_to_double(int(bits))


def scores(q: np.ndarray, emb: np.ndarray) -> np.ndarray:
    """s_i = <q, e_i> in float64, sequential sum (float32 inputs)."""
    q = _c(q, np.float32)
    emb = _c(emb, np.float32)
    n, e = emb.shape
    assert q.shape == (e,)
    out = np.empty(n, np.float64)
    _load().kvo_scores(_p(q), _p(emb), n, e, _p(out))
    return out


def topk(s: np.ndarray, k: int) -> np.ndarray:
    """Ids of the k best facts under (score desc, id asc), in rank order."""
    s = _c(s, np.float64)
    sel = np.empty(max(k, 0), np.int32)
    rc = _load().kvo_topk(_p(s), s.shape[0], int(k), _p(sel))
    if rc != OK:
        raise ValueError(f"oracle topk: bad argument (k={k}, n={s.shape[0]})")
    return sel


def place(sel: np.ndarray, fact_len: np.ndarray, start: int):
    """Contiguous rank-order positions; returns (pos[k] int64, total tokens)."""
    sel = _c(sel, np.int32)
    fact_len = _c(fact_len, np.int32)
    pos = np.empty(sel.shape[0], np.int64)
    T = _load().kvo_place(_p(sel), sel.shape[0], _p(fact_len), fact_len.shape[0],
                          int(start), _p(pos))
    if T < 0:
        raise ValueError("oracle place: fact id out of range or negative length")
    return pos, int(T)


def rope_omega(theta: float, d: int) -> np.ndarray:
    out = np.empty(d // 2, np.float64)
    _load().kvo_rope_omega(float(theta), int(d), _p(out))
    return out


def rotate(x: np.ndarray, theta: float, p: float) -> np.ndarray:
    """Rotate one head vector (float64) to position p (rotate-half)."""
    x = _c(x, np.float64)
    y = np.empty_like(x)
    _load().kvo_rotate(_p(x), x.shape[0], float(theta), float(p), _p(y))
    return y


def rope_omega_llama3(theta: float, d: int, factor: float, low: float, high: float,
                      orig: float) -> np.ndarray:
    """Llama 3.1 scaled frequencies (see kvo_rope_omega_llama3)."""
    out = np.empty(d // 2, np.float64)
    _load().kvo_rope_omega_llama3(float(theta), int(d), float(factor), float(low),
                                  float(high), float(orig), _p(out))
    return out


def rotate_pairs(x: np.ndarray, omega: np.ndarray, pairing: int, p: float) -> np.ndarray:
    """Rotate one head vector with explicit frequencies and pairing."""
    x = _c(x, np.float64)
    omega = _c(omega, np.float64)
    y = np.empty_like(x)
    _load().kvo_rotate_pairs(_p(x), x.shape[0], _p(omega), int(pairing), float(p), _p(y))
    return y


def rotate_cs(x: np.ndarray, c: np.ndarray, s: np.ndarray, pairing: int) -> np.ndarray:
    """Rotate one head vector by given cos/sin per pair."""
    x = _c(x, np.float64)
    c = _c(c, np.float64)
    s = _c(s, np.float64)
    y = np.empty_like(x)
    _load().kvo_rotate_cs(_p(x), x.shape[0], _p(c), _p(s), int(pairing), _p(y))
    return y


def rope_spec(theta: float, d: int, pairing: int = PAIR_HALF, llama3=None,
              cos_table=None, sin_table=None) -> dict:
    """How the oracle rotates: frequencies (plain or Llama 3.1 scaled, llama3 =
    (factor, low, high, orig)) or a cos/sin table (float32 [P][D/2]), and the
    pairing."""
    if cos_table is not None:
        return {"omega": np.zeros(d // 2), "pairing": int(pairing),
                "cos": _c(cos_table, np.float32), "sin": _c(sin_table, np.float32)}
    omega = rope_omega_llama3(theta, d, *llama3) if llama3 else rope_omega(theta, d)
    return {"omega": omega, "pairing": int(pairing), "cos": None, "sin": None}


def _rope_args(rope: dict):
    cos, sin = rope["cos"], rope["sin"]
    n = 0 if cos is None else cos.shape[0]
    return (_p(_c(rope["omega"], np.float64)), int(rope["pairing"]),
            None if cos is None else _p(cos), None if sin is None else _p(sin), n)


def slot(p: int, block_table: np.ndarray, block_size: int, num_blocks: int):
    """(block, offset) of position p, or None when out of range."""
    bt = _c(block_table, np.int32)
    blk = ctypes.c_int32()
    off = ctypes.c_int32()
    rc = _load().kvo_slot(int(p), _p(bt), bt.shape[0], int(block_size),
                          int(num_blocks), ctypes.byref(blk), ctypes.byref(off))
    return None if rc != OK else (blk.value, off.value)


def slots(positions, block_table, block_size: int, num_blocks: int):
    """(blk[n], off[n]) int32 arrays for many positions; -1 where out of range."""
    p = _c(positions, np.int64)
    bt = _c(block_table, np.int32)
    blk = np.empty(p.shape[0], np.int32)
    off = np.empty(p.shape[0], np.int32)
    _load().kvo_slots(_p(p), p.shape[0], _p(bt), bt.shape[0], int(block_size),
                      int(num_blocks), _p(blk), _p(off))
    return blk, off


def token_rows(kv_bits: np.ndarray, row: int, theta: float, p: int, rope: dict | None = None):
    """Expected (K float64 [L][H][D], V bits uint16 [L][H][D]) of one token.

    kv_bits: uint16 array shaped [L][2][n_tokens][H][D] (bf16 bit patterns).
    rope: a rope_spec(); None is the plain reading (rotate-half, theta).
    """
    kv_bits = _c(kv_bits, np.uint16)
    L, two, n_tokens, H, D = kv_bits.shape
    assert two == 2
    k_out = np.empty((L, H, D), np.float64)
    v_out = np.empty((L, H, D), np.uint16)
    if rope is None:
        rc = _load().kvo_token_rows(_p(kv_bits), L, H, D, n_tokens, int(row),
                                    float(theta), int(p), _p(k_out), _p(v_out))
    else:
        rc = _load().kvo_token_rows_ex(_p(kv_bits), L, H, D, n_tokens, int(row),
                                       *_rope_args(rope), int(p), _p(k_out), _p(v_out))
    if rc != OK:
        raise ValueError("oracle token_rows: store row out of range")
    return k_out, v_out


def token_rows_from_rows(k_rows: np.ndarray, v_rows: np.ndarray, theta: float, p: int,
                         rope: dict | None = None):
    """Same as token_rows for one token whose K and V rows ([L][H][D] bf16
    bits each) were already gathered from a store too large to pass whole."""
    k_rows = _c(k_rows, np.uint16)
    v_rows = _c(v_rows, np.uint16)
    L, H, D = k_rows.shape
    kv = np.stack([k_rows, v_rows], axis=1).reshape(L, 2, 1, H, D)
    return token_rows(kv, 0, theta, p, rope)


def inject_expected(kv_bits, fact_start, fact_len, ids, starts, block_table,
                    num_blocks: int, block_size: int, theta: float, rope: dict | None = None):
    """Expected pool after injecting facts ids[] at positions starts[].

    rope: a rope_spec(); None is the plain reading (rotate-half, theta).
    Returns (status, expect float64 [L][2][NB][B][H][D], written uint8 same).
    """
    kv_bits = _c(kv_bits, np.uint16)
    L, two, n_tokens, H, D = kv_bits.shape
    fact_start = _c(fact_start, np.int64)
    fact_len = _c(fact_len, np.int32)
    ids = _c(ids, np.int32)
    starts = _c(starts, np.int64)
    bt = _c(block_table, np.int32)
    shape = (L, 2, num_blocks, block_size, H, D)
    expect = np.empty(shape, np.float64)
    written = np.empty(shape, np.uint8)
    if rope is None:
        rc = _load().kvo_inject_expected(
            _p(kv_bits), L, H, D, n_tokens, _p(fact_start), _p(fact_len),
            fact_len.shape[0], _p(ids), _p(starts), ids.shape[0], _p(bt), bt.shape[0],
            int(num_blocks), int(block_size), float(theta), _p(expect), _p(written))
    else:
        rc = _load().kvo_inject_expected_ex(
            _p(kv_bits), L, H, D, n_tokens, _p(fact_start), _p(fact_len),
            fact_len.shape[0], _p(ids), _p(starts), ids.shape[0], _p(bt), bt.shape[0],
            int(num_blocks), int(block_size), *_rope_args(rope), _p(expect), _p(written))
    return rc, expect, written


def request(q, emb, k, kv_bits, fact_start, fact_len, start, theta, max_tokens):
    """Whole request (score, select, place, rotate/copy rows).

    Returns (sel, pos, k_rows [T][L][H][D] float64, v_rows uint16)."""
    q = _c(q, np.float32)
    emb = _c(emb, np.float32)
    kv_bits = _c(kv_bits, np.uint16)
    L, two, n_tokens, H, D = kv_bits.shape
    fact_start = _c(fact_start, np.int64)
    fact_len = _c(fact_len, np.int32)
    sel = np.empty(k, np.int32)
    pos = np.empty(k, np.int64)
    k_out = np.empty((max_tokens, L, H, D), np.float64)
    v_out = np.empty((max_tokens, L, H, D), np.uint16)
    T = _load().kvo_request(
        _p(q), _p(emb), emb.shape[0], emb.shape[1], int(k), _p(kv_bits), L, H, D,
        n_tokens, _p(fact_start), _p(fact_len), int(start), float(theta), _p(sel),
        _p(pos), _p(k_out), _p(v_out), int(max_tokens))
    if T < 0:
        raise ValueError("oracle request failed")
    return sel, pos, k_out[:T], v_out[:T]


def check_rows(src_bits: np.ndarray, got_bits: np.ndarray, pos: np.ndarray, theta: float,
               k_rel: float, k_abs: float, rope: dict | None = None, threads: int = 1):
    """Check T injected tokens against the oracle (see kvo_check_rows).

    src_bits, got_bits: uint16 [L][2][T][H][D] -- the store rows each token
    came from and the pool rows written for it; pos: int64 [T].  The tokens
    are split over `threads` host threads, each running the single-threaded
    C routine on its own range (ctypes releases the interpreter lock).
    Returns (bad K elements, bad V elements, first bad flat index or -1)."""
    src_bits = _c(src_bits, np.uint16)
    got_bits = _c(got_bits, np.uint16)
    pos = _c(pos, np.int64)
    L, two, T, H, D = src_bits.shape
    assert two == 2 and got_bits.shape == src_bits.shape and pos.shape == (T,)
    spec = rope if rope is not None else rope_spec(theta, D)
    omega, pairing, cos_p, sin_p, n_tab = _rope_args(spec)
    lib = _load()
    n = max(1, min(int(threads), T))
    cuts = [T * i // n for i in range(n + 1)]
    res = [None] * n

    def run(i):
        bk, bv, fb = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
        rc = lib.kvo_check_rows(_p(src_bits), _p(got_bits), L, H, D, T, cuts[i], cuts[i + 1],
                                _p(pos), omega, pairing, cos_p, sin_p, n_tab, float(k_rel),
                                float(k_abs), ctypes.byref(bk), ctypes.byref(bv), ctypes.byref(fb))
        res[i] = (rc, bk.value, bv.value, fb.value)

    if n == 1:
        run(0)
    else:
        ts = [threading.Thread(target=run, args=(i,)) for i in range(n)]
        for t in ts:
            t.start()
        for t in ts:
            t.join()
    bad_k = bad_v = 0
    first = -1
    for rc, bk, bv, fb in res:
        if rc != OK:
            raise ValueError(f"oracle check_rows: status {rc}")
        bad_k += bk
        bad_v += bv
        if first < 0 and fb >= 0:
            first = fb
    return bad_k, bad_v, first


def graph_build(emb: np.ndarray, degree: int) -> np.ndarray:
    """Graph index: each fact's `degree` most similar other facts, exact,
    in (score desc, id asc) order -> int32 [N][degree]."""
    emb = _c(emb, np.float32)
    n, e = emb.shape
    nbr = np.empty((n, max(degree, 0)), np.int32)
    rc = _load().kvo_graph_build(_p(emb), n, e, int(degree), _p(nbr))
    if rc != OK:
        raise ValueError(f"oracle graph_build: bad argument (n={n}, degree={degree})")
    return nbr


def graph_search(q: np.ndarray, emb: np.ndarray, nbr: np.ndarray, seeds, beam: int, width: int,
                 max_iters: int, k: int):
    """Best-first beam search of one query over the graph nbr [N][d] from
    the given seed ids.  Returns (ids int32 [k], scores float64 [k], count,
    iterations, facts scored); ids past `count` are -1."""
    q = _c(q, np.float32)
    emb = _c(emb, np.float32)
    nbr = _c(nbr, np.int32)
    seeds = _c(np.atleast_1d(seeds), np.int32)
    n, e = emb.shape
    assert q.shape == (e,) and nbr.shape[0] == n
    sel = np.empty(max(k, 1), np.int32)
    sc = np.empty(max(k, 1), np.float64)
    stats = np.zeros(2, np.int64)
    cnt = _load().kvo_graph_search(_p(q), _p(emb), n, e, _p(nbr), nbr.shape[1], _p(seeds),
                                   seeds.shape[0], int(beam), int(width), int(max_iters), int(k),
                                   _p(sel), _p(sc), _p(stats))
    if cnt < 0:
        raise ValueError("oracle graph_search: bad argument")
    return sel[:k], sc[:k], int(cnt), int(stats[0]), int(stats[1])
