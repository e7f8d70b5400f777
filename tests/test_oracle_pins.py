"""Pins of the float64 oracle against things other than itself.

Each oracle function is checked against a closed form, an invariant, exact
rational arithmetic, brute force, or a hand-worked fixture in tests/golden/,
chosen so that a plausible slip (a dropped term, a flipped sign, a swapped
pairing, a transposed operand, an off-by-one in placement or paging, a
reversed tie-break) fails at least one test.  Method: "InferScale: GPU-Native
KV Injection for Personalized LLM Serving" -- Figure 2 caption, Section 5.1 /
Theorem 6, Section 3.4.
"""
import itertools
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
U64 = 2.0 ** -53  # unit roundoff of float64


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _eval_expr(s):
    return float(eval(s, {"__builtins__": {}}, {"cos": math.cos, "sin": math.sin}))


def _bf16_bits(x):
    """bf16 bits of values that are exactly representable (checked)."""
    a = np.asarray(x, np.float32)
    u = a.view(np.uint32)
    assert np.all((u & 0xFFFF) == 0), "fixture value not exact in bf16"
    return (u >> 16).astype(np.uint16)


# ---------------------------------------------------------------- bf16 decode

def test_bf16_decode_known_patterns():
    # IEEE binary32 upper halves: 0x3F80 = 1.0, 0xC000 = -2.0,
    # 0x3F81 = 1 + 2^-7, 0x0000 = +0, 0x7F80 = +inf.
    assert oracle.bf16_to_double(0x3F80) == 1.0
    assert oracle.bf16_to_double(0xC000) == -2.0
    assert oracle.bf16_to_double(0x3F81) == 1.0 + 2.0 ** -7
    assert oracle.bf16_to_double(0x0000) == 0.0
    assert math.isinf(oracle.bf16_to_double(0x7F80))


# ---------------------------------------------------------------------- scores

def test_scores_basis_embeddings_exact():
    # e_i = unit basis vector i, so s_i = q_i exactly.
    rng = np.random.default_rng(11)
    E = 24
    q = rng.standard_normal(E).astype(np.float32)
    emb = np.eye(E, dtype=np.float32)
    s = oracle.scores(q, emb)
    assert np.array_equal(s, q.astype(np.float64))


def test_scores_against_exact_rationals():
    # Products of float32 values are exact in float64; only the sums round, so
    # |s - exact| <= gamma_{E-1} * sum|q_j e_ij|.  A non-square store catches a
    # transposed operand; an exact rational sum is independent of any rounding.
    rng = np.random.default_rng(12)
    N, E = 7, 37
    q = rng.standard_normal(E).astype(np.float32)
    emb = rng.standard_normal((N, E)).astype(np.float32)
    s = oracle.scores(q, emb)
    g = (E - 1) * U64 / (1 - (E - 1) * U64)
    for i in range(N):
        exact = sum(Fraction(float(q[j])) * Fraction(float(emb[i, j])) for j in range(E))
        bound = g * sum(abs(float(q[j]) * float(emb[i, j])) for j in range(E))
        assert abs(Fraction(s[i]) - exact) <= Fraction(bound)


def test_scores_golden():
    g = _golden("select_place_tiny.json")
    s = oracle.scores(np.array(g["q"]), np.array(g["emb"]))
    assert s.tolist() == g["expected_scores"]


# ----------------------------------------------------------------------- top-k

def _better(a, b):
    # a, b = (score, id): higher score first, lower id on ties
    return a[0] > b[0] or (a[0] == b[0] and a[1] < b[1])


def _brute_force_topk(s, k):
    """The unique k-subset whose every member beats every non-member, in order."""
    n = len(s)
    hits = []
    for sub in itertools.combinations(range(n), k):
        inside = [(s[i], i) for i in sub]
        outside = [(s[i], i) for i in range(n) if i not in sub]
        if all(_better(a, b) for a in inside for b in outside):
            hits.append(sub)
    assert len(hits) == 1
    members = [(s[i], i) for i in hits[0]]
    # order by pairwise comparisons only (selection, no library sort)
    out = []
    while members:
        best = members[0]
        for m in members[1:]:
            if _better(m, best):
                best = m
        out.append(best[1])
        members.remove(best)
    return out


@pytest.mark.parametrize("seed", range(6))
def test_topk_brute_force_with_planted_ties(seed):
    rng = np.random.default_rng(100 + seed)
    n = int(rng.integers(3, 11))
    # few distinct values, so exact ties are common
    s = rng.integers(-3, 4, size=n).astype(np.float64) / 4.0
    for k in range(1, n + 1):
        assert oracle.topk(s, k).tolist() == _brute_force_topk(s.tolist(), k)


def test_topk_golden_and_tie_to_lower_id():
    g = _golden("select_place_tiny.json")
    s = np.array(g["expected_scores"])
    assert oracle.topk(s, g["k"]).tolist() == g["expected_sel"]
    # all equal: the k lowest ids, ascending
    assert oracle.topk(np.zeros(9), 4).tolist() == [0, 1, 2, 3]


def test_topk_invariant_large():
    rng = np.random.default_rng(13)
    n, k = 5000, 50
    s = np.round(rng.standard_normal(n), 3)  # rounding plants many ties
    sel = oracle.topk(s, k)
    chosen = set(sel.tolist())
    assert len(chosen) == k
    worst_in = (s[sel[-1]], sel[-1])
    for i in range(n):
        if i not in chosen:
            assert _better(worst_in, (s[i], i))
    for a, b in zip(sel[:-1], sel[1:]):
        assert _better((s[a], a), (s[b], b))


@pytest.mark.parametrize("k", [0, -1, 7])
def test_topk_rejects_bad_k(k):
    with pytest.raises(ValueError):
        oracle.topk(np.zeros(6), k)


# ------------------------------------------------------------------- placement

def test_place_golden():
    g = _golden("select_place_tiny.json")
    pos, T = oracle.place(np.array(g["expected_sel"]), np.array(g["fact_len"]), g["start"])
    assert pos.tolist() == g["expected_pos"]
    assert T == g["expected_total"]


def test_place_invariants():
    rng = np.random.default_rng(14)
    lens = rng.integers(12, 49, size=300).astype(np.int32)
    sel = rng.permutation(300)[:50].astype(np.int32)
    start = 64
    pos, T = oracle.place(sel, lens, start)
    assert T == int(lens[sel].sum())
    covered = np.zeros(start + T + 5, np.int32)
    for j, f in enumerate(sel):
        covered[pos[j]:pos[j] + lens[f]] += 1
    assert np.all(covered[start:start + T] == 1)   # each position exactly once
    assert covered[:start].sum() == 0 and covered[start + T:].sum() == 0
    assert pos[0] == start and np.all(np.diff(pos) == lens[sel[:-1]])


def test_place_rejects_bad_id():
    with pytest.raises(ValueError):
        oracle.place(np.array([0, 5]), np.array([3, 4]), 0)


# ----------------------------------------------------------------------- RoPE

def test_omega_closed_forms():
    w = oracle.rope_omega(10000.0, 4)
    assert w[0] == 1.0
    assert abs(w[1] - 0.01) <= 1e-17
    w = oracle.rope_omega(500000.0, 128)
    assert w[0] == 1.0
    assert abs(w[32] - 500000.0 ** -0.5) <= 1e-16 * 500000.0 ** -0.5 * 4
    assert np.all(np.diff(w) < 0)


def test_rotate_position_zero_is_identity():
    rng = np.random.default_rng(15)
    for d in (2, 4, 64, 128):
        x = rng.standard_normal(d)
        assert np.array_equal(oracle.rotate(x, 500000.0, 0.0), x)


@pytest.mark.parametrize("p", [1.0, 2.5, 100.0, 39000.0])
def test_rotate_d2_closed_form(p):
    # D = 2: omega_0 = 1, so (1,0) -> (cos p, sin p) and (0,1) -> (-sin p, cos p)
    y = oracle.rotate(np.array([1.0, 0.0]), 10000.0, p)
    assert y.tolist() == pytest.approx([math.cos(p), math.sin(p)], abs=1e-15)
    y = oracle.rotate(np.array([0.0, 1.0]), 10000.0, p)
    assert y.tolist() == pytest.approx([-math.sin(p), math.cos(p)], abs=1e-15)


def test_rotate_d4_pairing_and_frequency():
    # D = 4, theta = 1e4, p = 100: pair (0,2) turns by 100 rad, pair (1,3) by
    # 100 * 0.01 = 1 rad.  Basis inputs expose the pairing (rotate-half, not
    # interleaved) and the sign convention.
    p, th = 100.0, 10000.0
    e = np.eye(4)
    c0, s0, c1, s1 = math.cos(100.0), math.sin(100.0), math.cos(1.0), math.sin(1.0)
    expect = {
        0: [c0, 0.0, s0, 0.0],
        1: [0.0, c1, 0.0, s1],
        2: [-s0, 0.0, c0, 0.0],
        3: [0.0, -s1, 0.0, c1],
    }
    for i in range(4):
        assert oracle.rotate(e[i], th, p).tolist() == pytest.approx(expect[i], abs=1e-13)


def test_rotate_composition():
    rng = np.random.default_rng(16)
    for _ in range(50):
        x = rng.standard_normal(128)
        a, b = rng.integers(0, 20000, size=2).astype(float)
        y = oracle.rotate(oracle.rotate(x, 500000.0, a), 500000.0, b)
        z = oracle.rotate(x, 500000.0, a + b)
        # angle products carry ~1 ulp of 40000 rad, hence the 5e-11 scale
        assert np.max(np.abs(y - z)) <= 5e-11 * np.linalg.norm(x)
    x = rng.standard_normal(64)
    y = oracle.rotate(oracle.rotate(x, 10000.0, 3.0), 10000.0, 4.0)
    assert np.max(np.abs(y - oracle.rotate(x, 10000.0, 7.0))) <= 1e-13


def test_rotate_preserves_pair_norms():
    rng = np.random.default_rng(17)
    for d in (4, 64, 128):
        x = rng.standard_normal(d)
        y = oracle.rotate(x, 1e6, 38000.0)
        h = d // 2
        n_x = np.hypot(x[:h], x[h:])
        n_y = np.hypot(y[:h], y[h:])
        assert np.max(np.abs(n_x - n_y)) <= 1e-14 * np.max(n_x) * 8


def test_relocation_theorem():
    # Theorem 6: <R_m q, R_n k> = <R_{m+s} q, R_{n+s} k> = <R_{m-n} q, k>.
    rng = np.random.default_rng(18)
    for _ in range(40):
        q = rng.standard_normal(128)
        k = rng.standard_normal(128)
        m, n, s = (float(v) for v in rng.integers(0, 40000, size=3))
        base = oracle.rotate(q, 500000.0, m) @ oracle.rotate(k, 500000.0, n)
        shifted = oracle.rotate(q, 500000.0, m + s) @ oracle.rotate(k, 500000.0, n + s)
        rel = oracle.rotate(q, 500000.0, m - n) @ k
        scale = np.linalg.norm(q) * np.linalg.norm(k)
        assert abs(base - shifted) <= 1e-10 * scale
        assert abs(base - rel) <= 1e-10 * scale


def test_rotate_matches_complex_multiplication():
    # Rotate-half RoPE is multiplication of z_i = x_i + 1j*x_{i+D/2} by
    # exp(1j * p * omega_i); numpy's complex exponential is independent of the
    # oracle's real cos/sin arithmetic.
    rng = np.random.default_rng(19)
    D, th, p = 64, 1e6, 12345.0
    x = rng.standard_normal(D)
    h = D // 2
    omega = th ** (-2.0 * np.arange(h) / D)
    z = (x[:h] + 1j * x[h:]) * np.exp(1j * p * omega)
    y = oracle.rotate(x, th, p)
    assert np.max(np.abs(y[:h] - z.real)) <= 1e-11
    assert np.max(np.abs(y[h:] - z.imag)) <= 1e-11


# ------------------------------------------------------------------- paging

def test_slot_mapping_hand_cases():
    bt = np.array([5, 2, 7], np.int32)
    assert oracle.slot(0, bt, 2, 8) == (5, 0)
    assert oracle.slot(1, bt, 2, 8) == (5, 1)
    assert oracle.slot(2, bt, 2, 8) == (2, 0)
    assert oracle.slot(5, bt, 2, 8) == (7, 1)
    assert oracle.slot(6, bt, 2, 8) is None          # beyond the table
    assert oracle.slot(-1, bt, 2, 8) is None
    assert oracle.slot(0, np.array([8]), 2, 8) is None  # block id not in the pool
    assert oracle.slot(37, np.array([0, 1, 9]), 16, 10) == (9, 5)
    blk, off = oracle.slots(np.array([0, 1, 2, 5, 6, -1]), bt, 2, 8)
    assert blk.tolist() == [5, 5, 2, 7, -1, -1] and off.tolist() == [0, 1, 0, 1, -1, -1]


# ----------------------------------------------------------- full expectation

def _golden_store(g):
    k = _bf16_bits(g["store_k"])
    v = _bf16_bits(g["store_v"])
    T = k.shape[0]
    geo = g["geometry"]
    L, H, D = geo["L"], geo["H"], geo["D"]
    kv = np.empty((L, 2, T, H, D), np.uint16)
    kv[0, 0, :, 0, :] = k
    kv[0, 1, :, 0, :] = v
    return kv


@pytest.mark.parametrize("case", [0, 1])
def test_inject_expected_golden(case):
    g = _golden("scatter_tiny.json")
    geo = g["geometry"]
    c = g["cases"][case]
    kv = _golden_store(g)
    rc, expect, written = oracle.inject_expected(
        kv, g["fact_start"], g["fact_len"], g["ids"], c["starts"], c["block_table"],
        geo["num_blocks"], geo["block_size"], geo["theta"])
    assert rc == oracle.OK
    want_written = np.zeros_like(written)
    for tok in c["tokens"]:
        blk, off = tok["slot"]
        kexp = [_eval_expr(e) for e in tok["k"]]
        assert expect[0, 0, blk, off, 0, :] == pytest.approx(kexp, abs=1e-12)
        assert expect[0, 1, blk, off, 0, :].tolist() == [float(v) for v in tok["v"]]
        want_written[0, :, blk, off, 0, :] = 1
    assert np.array_equal(written, want_written)
    if case == 0:  # position 0: K bit-identical to the stored pre-RoPE key
        assert expect[0, 0, 5, 0, 0, :].tolist() == [4.0, -4.0, 0.5, 2.0]


def test_inject_expected_detects_overlap_and_range():
    g = _golden("scatter_tiny.json")
    geo = g["geometry"]
    kv = _golden_store(g)
    # overlapping positions: fact 0 at 0..2 and fact 1 at 2..3
    rc, _, _ = oracle.inject_expected(kv, g["fact_start"], g["fact_len"], [0, 1], [0, 2],
                                      [5, 2, 7], 8, 2, 1e4)
    assert rc == oracle.CAPACITY
    # beyond the block table
    rc, _, _ = oracle.inject_expected(kv, g["fact_start"], g["fact_len"], [0], [5],
                                      [5, 2, 7], 8, 2, 1e4)
    assert rc == oracle.OUT_OF_RANGE
    # fact id out of range
    rc, _, _ = oracle.inject_expected(kv, g["fact_start"], g["fact_len"], [2], [0],
                                      [5, 2, 7], 8, 2, 1e4)
    assert rc == oracle.OUT_OF_RANGE


def test_token_rows_multi_layer_multi_head_layout():
    # Token rows must read kv[l][c][row][h][:] for every layer and head; each
    # (l, h) gets a distinct constant so a stride slip shows up.
    L, H, D, T = 3, 2, 4, 4
    kv = np.zeros((L, 2, T, H, D), np.float32)
    for l in range(L):
        for h in range(H):
            kv[l, 0, 2, h, :] = [l + 1, h + 1, 0, 0]
            kv[l, 1, 2, h, :] = 10 * l + h
    bits = _bf16_bits(kv)
    k_out, v_out = oracle.token_rows(bits, 2, 10000.0, 0)
    for l in range(L):
        for h in range(H):
            assert k_out[l, h].tolist() == [l + 1, h + 1, 0, 0]
            assert [oracle.bf16_to_double(b) for b in v_out[l, h]] == [10 * l + h] * D


def test_request_composes_the_steps():
    rng = np.random.default_rng(20)
    N, E, L, H, D, k = 40, 32, 2, 2, 8, 5
    emb = rng.standard_normal((N, E)).astype(np.float32)
    q = rng.standard_normal(E).astype(np.float32)
    lens = rng.integers(1, 5, size=N).astype(np.int32)
    starts = np.concatenate([[0], np.cumsum(lens)[:-1]]).astype(np.int64)
    T = int(lens.sum())
    kv = _bf16_bits(np.round(rng.standard_normal((L, 2, T, H, D)) * 8) / 8)
    sel, pos, kr, vr = oracle.request(q, emb, k, kv, starts, lens, 7, 1e4, 64)
    s = oracle.scores(q, emb)
    assert sel.tolist() == oracle.topk(s, k).tolist()
    pos2, T2 = oracle.place(sel, lens, 7)
    assert pos.tolist() == pos2.tolist() and kr.shape[0] == T2
    tok = 0
    for j, f in enumerate(sel):
        for t in range(lens[f]):
            k1, v1 = oracle.token_rows(kv, starts[f] + t, 1e4, pos[j] + t)
            assert np.array_equal(kr[tok], k1) and np.array_equal(vr[tok], v1)
            tok += 1


# ------------------------------------------------------- rotary variants
#
# Interleaved pairing (2i, 2i+1), Llama 3.1 frequency scaling and rotation
# by a caller's cos/sin table: the conventions an engine may use other than
# the plain reading.  Pinned by closed forms, regime invariants and
# identities that the plain rotation already satisfies.

def test_interleaved_d2_closed_form():
    # with one pair both pairings coincide: (1, 0) at p -> (cos p, sin p)
    for pairing in (oracle.PAIR_HALF, oracle.PAIR_INTERLEAVED):
        y = oracle.rotate_pairs(np.array([1.0, 0.0]), np.array([1.0]), pairing, 0.7)
        np.testing.assert_allclose(y, [math.cos(0.7), math.sin(0.7)], rtol=0, atol=1e-15)


def test_interleaved_d4_pairs_adjacent_elements():
    # D = 4, omega = (1, 0.01): interleaved pairs are (0, 1) and (2, 3)
    omega = np.array([1.0, 0.01])
    y = oracle.rotate_pairs(np.array([0.0, 0.0, 1.0, 0.0]), omega, oracle.PAIR_INTERLEAVED, 100.0)
    np.testing.assert_allclose(y, [0.0, 0.0, math.cos(1.0), math.sin(1.0)], atol=1e-15)
    y = oracle.rotate_pairs(np.array([0.0, 1.0, 0.0, 0.0]), omega, oracle.PAIR_INTERLEAVED, 2.0)
    np.testing.assert_allclose(y, [-math.sin(2.0), math.cos(2.0), 0.0, 0.0], atol=1e-15)
    # the same inputs under rotate-half pair (0, 2) and (1, 3) instead
    y = oracle.rotate_pairs(np.array([0.0, 0.0, 1.0, 0.0]), omega, oracle.PAIR_HALF, 100.0)
    np.testing.assert_allclose(y, [-math.sin(100.0), 0.0, math.cos(100.0), 0.0], atol=1e-13)


def test_interleaved_is_a_permuted_rotate_half():
    # moving element 2i to i and 2i+1 to i + D/2 turns one pairing into the
    # other: interleaved(x) = P^-1 half(P x)
    rng = np.random.default_rng(17)
    D = 128
    x = rng.standard_normal(D)
    omega = oracle.rope_omega(5e5, D)
    perm = np.concatenate([np.arange(0, D, 2), np.arange(1, D, 2)])  # P x = x[perm]
    for p in (0.0, 3.0, 1234.0, 39167.0):
        yi = oracle.rotate_pairs(x, omega, oracle.PAIR_INTERLEAVED, p)
        yh = oracle.rotate_pairs(x[perm], omega, oracle.PAIR_HALF, p)
        back = np.empty(D)
        back[perm] = yh
        np.testing.assert_allclose(yi, back, rtol=0, atol=1e-14)


def test_rotate_pairs_half_agrees_with_plain_rotation():
    rng = np.random.default_rng(18)
    x = rng.standard_normal(64)
    omega = oracle.rope_omega(1e4, 64)
    for p in (0.0, 1.0, 77.0, 30000.0):
        np.testing.assert_allclose(oracle.rotate_pairs(x, omega, oracle.PAIR_HALF, p),
                                   oracle.rotate(x, 1e4, p), rtol=0, atol=1e-14)


@pytest.mark.parametrize("pairing", [0, 1])
def test_variants_keep_norms_composition_and_relocation(pairing):
    rng = np.random.default_rng(19 + pairing)
    D = 64
    omega = oracle.rope_omega_llama3(5e5, D, 8.0, 1.0, 4.0, 8192.0)
    q, k = rng.standard_normal(D), rng.standard_normal(D)
    a, b, s = 311.0, 9000.0, 20011.0
    # pair norms
    y = oracle.rotate_pairs(k, omega, pairing, a)
    if pairing:
        pn = lambda v: v[0::2] ** 2 + v[1::2] ** 2
    else:
        pn = lambda v: v[:D // 2] ** 2 + v[D // 2:] ** 2
    np.testing.assert_allclose(pn(y), pn(k), rtol=1e-12)
    # composition
    np.testing.assert_allclose(oracle.rotate_pairs(y, omega, pairing, b),
                               oracle.rotate_pairs(k, omega, pairing, a + b), atol=1e-9)
    # relocation: <R_m q, R_n k> depends only on m - n
    d1 = oracle.rotate_pairs(q, omega, pairing, a) @ oracle.rotate_pairs(k, omega, pairing, b)
    d2 = oracle.rotate_pairs(q, omega, pairing, a + s) @ oracle.rotate_pairs(k, omega, pairing, b + s)
    assert abs(d1 - d2) <= 1e-9 * (1 + abs(d1))


def test_llama3_scaling_regimes():
    # Llama 3.1 parameters: theta 5e5, D 128, factor 8, low 1, high 4,
    # original context 8192 -> wavelengths below 2048 keep their frequency,
    # above 8192 are divided by 8, in between lie strictly between the two
    D, theta = 128, 5e5
    base = oracle.rope_omega(theta, D)
    scaled = oracle.rope_omega_llama3(theta, D, 8.0, 1.0, 4.0, 8192.0)
    lam = 2 * math.pi / base
    hi, lo, mid = lam < 2048, lam > 8192, (lam >= 2048) & (lam <= 8192)
    assert hi.sum() > 0 and lo.sum() > 0 and mid.sum() > 0
    np.testing.assert_array_equal(scaled[hi], base[hi])
    np.testing.assert_allclose(scaled[lo], base[lo] / 8.0, rtol=1e-15)
    assert np.all(scaled[mid] < base[mid]) and np.all(scaled[mid] > base[mid] / 8.0)
    assert np.all(np.diff(scaled) < 0)  # still strictly decreasing
    assert scaled[0] == 1.0


def test_llama3_midpoint_closed_form():
    # D = 4: omega_1 = theta^(-1/2).  Choose theta so that omega_1's
    # wavelength is 8192 / 2.5; the blend weight is then exactly 1/2 and
    # omega_1' = omega_1 (1/8 + 1) / 2 = 0.5625 omega_1.
    lam = 8192.0 / 2.5
    w1 = 2 * math.pi / lam
    theta = (1.0 / w1) ** 2
    scaled = oracle.rope_omega_llama3(theta, 4, 8.0, 1.0, 4.0, 8192.0)
    assert scaled[0] == 1.0
    assert abs(scaled[1] - 0.5625 * w1) <= 1e-12 * w1


def test_llama3_is_continuous_at_both_edges():
    # just inside and just outside each edge of the blend region
    for edge, expect in ((8192.0 / 4.0, 1.0), (8192.0 / 1.0, 1.0 / 8.0)):
        ratios = []
        for lam in (edge * (1 - 1e-9), edge * (1 + 1e-9)):
            w1 = 2 * math.pi / lam
            theta = (1.0 / w1) ** 2
            ratios.append(oracle.rope_omega_llama3(theta, 4, 8.0, 1.0, 4.0, 8192.0)[1] / w1)
        assert abs(ratios[0] - expect) < 1e-6 and abs(ratios[1] - expect) < 1e-6


@pytest.mark.parametrize("pairing", [0, 1])
def test_table_rotation_closed_forms(pairing):
    rng = np.random.default_rng(23)
    x = rng.standard_normal(8)
    one, zero = np.ones(4), np.zeros(4)
    np.testing.assert_array_equal(oracle.rotate_cs(x, one, zero, pairing), x)
    y = oracle.rotate_cs(x, zero, one, pairing)  # a quarter turn of every pair
    a, b = (np.arange(0, 8, 2), np.arange(1, 8, 2)) if pairing else (np.arange(4), np.arange(4, 8))
    np.testing.assert_array_equal(y[a], -x[b])
    np.testing.assert_array_equal(y[b], x[a])


def test_table_rows_in_token_rows():
    # a cos/sin table of the exact angles reproduces the computed rotation
    # within float32 rounding of the table; positions beyond it are refused
    rng = np.random.default_rng(29)
    L, H, D, P = 2, 2, 16, 40
    kv = (rng.standard_normal((L, 2, 3, H, D)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    omega = oracle.rope_omega(1e4, D)
    ang = np.arange(P)[:, None] * omega[None, :]
    rope = oracle.rope_spec(1e4, D, oracle.PAIR_INTERLEAVED, cos_table=np.cos(ang), sin_table=np.sin(ang))
    plain = oracle.rope_spec(1e4, D, oracle.PAIR_INTERLEAVED)
    for p in (0, 1, 39):
        kt, vt = oracle.token_rows(kv, 1, 0.0, p, rope)
        kp, vp = oracle.token_rows(kv, 1, 1e4, p, plain)
        np.testing.assert_allclose(kt, kp, atol=1e-6 * np.abs(kp).max())
        np.testing.assert_array_equal(vt, vp)
    with pytest.raises(ValueError):
        oracle.token_rows(kv, 1, 0.0, P, rope)


# ------------------------------------------------------- batched row check

def _rne_bf16_bits(y):
    """float64 -> float32 -> bf16 bits, round to nearest even (numpy)."""
    u = np.asarray(y, np.float64).astype(np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def _check_rows_case(seed, L=3, H=2, D=16, T=7, theta=1e4):
    rng = np.random.default_rng(seed)
    src = _rne_bf16_bits(rng.standard_normal((L, 2, T, H, D)))  # bf16 ~N(0,1), as stored
    pos = rng.integers(0, 40000, size=T).astype(np.int64)
    pos[0] = 0
    want_k = np.empty((L, T, H, D))
    for t in range(T):
        k, v = oracle.token_rows_from_rows(src[:, 0, t], src[:, 1, t], theta, int(pos[t]))
        want_k[:, t] = k
        assert np.array_equal(v, src[:, 1, t])
    return src, pos, want_k


def test_check_rows_agrees_with_token_rows():
    # the batched check computes each token's cos/sin once; its expected
    # values must be those of the per-row routine (pinned above): with the
    # path's result being the RNE bf16 of the expected values, nothing is
    # off within one bf16 ulp, and with a zero tolerance exactly the
    # elements that bf16 cannot hold are off
    src, pos, want_k = _check_rows_case(21)
    got = src.copy()
    got[:, 0] = _rne_bf16_bits(want_k)
    assert oracle.check_rows(src, got, pos, 1e4, 2.0 ** -8, 1e-6) == (0, 0, -1)
    inexact = int(np.sum(np.vectorize(oracle.bf16_to_double)(got[:, 0]) != want_k))
    bad_k, bad_v, first = oracle.check_rows(src, got, pos, 1e4, 0.0, 0.0)
    assert bad_k == inexact and bad_v == 0 and inexact > 0
    # the threaded split gives the same counts
    assert oracle.check_rows(src, got, pos, 1e4, 0.0, 0.0, threads=3)[:2] == (bad_k, 0)


def test_check_rows_position_zero_is_a_copy():
    src, pos, _ = _check_rows_case(22)
    pos[:] = 0
    assert oracle.check_rows(src, src.copy(), pos, 1e4, 0.0, 0.0) == (0, 0, -1)


def test_check_rows_finds_planted_errors():
    src, pos, want_k = _check_rows_case(23)
    good = src.copy()
    good[:, 0] = _rne_bf16_bits(want_k)
    L, _, T, H, D = src.shape
    # a K element moved by 4 bf16 ulps (well outside 2^-8 |x|)
    bad = good.copy()
    l, t, h, i = 2, 5, 1, 9
    bad[l, 0, t, h, i] = bad[l, 0, t, h, i] + 4 if want_k[l, t, h, i] != 0 else 0x3F80
    flat = (((l * 2 + 0) * T + t) * H + h) * D + i
    assert oracle.check_rows(src, bad, pos, 1e4, 2.0 ** -8, 1e-6) == (1, 0, flat)
    # one V bit flipped
    bad = good.copy()
    bad[0, 1, 3, 0, 2] ^= 1
    flat = (((0 * 2 + 1) * T + 3) * H + 0) * D + 2
    assert oracle.check_rows(src, bad, pos, 1e4, 2.0 ** -8, 1e-6) == (0, 1, flat)
    # a wrong position for one token: its K rows fail (nearly) everywhere
    wrong = pos.copy()
    wrong[4] += 1000  # turns even the slowest pair (omega_7 = 10^-3.5) by 0.3 rad
    bk, bv, _ = oracle.check_rows(src, good, wrong, 1e4, 2.0 ** -8, 1e-6)
    assert bv == 0 and bk > L * H * D // 2
    # the wrong pairing fails too
    spec = oracle.rope_spec(1e4, D, oracle.PAIR_INTERLEAVED)
    bk, _, _ = oracle.check_rows(src, good, pos, 1e4, 2.0 ** -8, 1e-6, rope=spec)
    assert bk > (T - 1) * L * H * D // 2


def test_check_rows_with_a_table():
    # a caller's cos/sin table is read at each token's position
    src, pos, _ = _check_rows_case(24, T=5)
    D = src.shape[4]
    P = int(pos.max()) + 1
    ang = np.arange(P)[:, None] * oracle.rope_omega(1e4, D)[None, :]
    spec = oracle.rope_spec(1e4, D, cos_table=np.cos(ang).astype(np.float32),
                            sin_table=np.sin(ang).astype(np.float32))
    got = src.copy()
    for t in range(src.shape[2]):
        k, _ = oracle.token_rows_from_rows(src[:, 0, t], src[:, 1, t], 1e4, int(pos[t]), rope=spec)
        got[:, 0, t] = _rne_bf16_bits(k)
    assert oracle.check_rows(src, got, pos, 1e4, 2.0 ** -8, 1e-6, rope=spec) == (0, 0, -1)
    short = oracle.rope_spec(1e4, D, cos_table=np.ones((1, D // 2), np.float32),
                             sin_table=np.zeros((1, D // 2), np.float32))
    with pytest.raises(ValueError):
        oracle.check_rows(src, got, pos, 1e4, 2.0 ** -8, 1e-6, rope=short)
