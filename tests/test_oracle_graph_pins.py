"""Pins of the oracle's graph index (CPU only).

The graph build is checked against brute force in exact integer arithmetic
(integer-valued embeddings make every score exact in float32 and float64,
so ties are real and the id tie-break is exercised).  The search is checked
on cases whose result follows from its definition by hand: a traced walk
along a path graph, the trap a narrow beam falls into and a wider one
escapes, no iterations (the best seeds), a complete graph (the exact
top-k), and the invariants every result must satisfy.
"""
import numpy as np
import pytest

import oracle


def _int_emb(n, e, seed, lo=-3, hi=4):
    rng = np.random.default_rng(seed)
    return rng.integers(lo, hi, (n, e)).astype(np.float32)


def _exact_order(q_int, emb_int, ids):
    """ids sorted by (exact integer score descending, id ascending)."""
    s = {int(j): int(np.dot(q_int.astype(np.int64), emb_int[j].astype(np.int64))) for j in ids}
    return sorted(ids, key=lambda j: (-s[int(j)], int(j))), s


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_graph_build_brute_force(seed):
    emb = _int_emb(11, 3, seed)
    d = 4
    nbr = oracle.graph_build(emb, d)
    assert nbr.shape == (11, d)
    for i in range(11):
        order, _ = _exact_order(emb[i], emb, [j for j in range(11) if j != i])
        assert list(nbr[i]) == order[:d], i


def test_graph_build_ties_go_to_the_lower_id():
    # facts 1..4 are identical, so fact 0 sees four equal scores
    emb = np.array([[1, 0], [2, 1], [2, 1], [2, 1], [2, 1], [-1, 0]], np.float32)
    nbr = oracle.graph_build(emb, 3)
    assert list(nbr[0]) == [1, 2, 3]
    # fact 2's equal neighbours 1, 3, 4 (score 5 each) in id order, never itself
    assert list(nbr[2]) == [1, 3, 4]


def test_graph_build_closed_form_on_a_circle():
    # unit vectors at angles 2*pi*i/n: the two most similar facts are the
    # adjacent angles, the next two those two steps away (float32 rounding of
    # cos and sin may order each pair either way)
    n = 12
    a = 2 * np.pi * np.arange(n) / n
    emb = np.stack([np.cos(a), np.sin(a)], 1).astype(np.float32)
    nbr = oracle.graph_build(emb, 4)
    for i in range(n):
        assert set(nbr[i][:2].tolist()) == {(i - 1) % n, (i + 1) % n}, i
        assert set(nbr[i][2:].tolist()) == {(i - 2) % n, (i + 2) % n}, i


def test_graph_build_rejects_bad_degrees():
    emb = _int_emb(5, 2, 0)
    for d in (0, 5, 6):
        with pytest.raises(ValueError):
            oracle.graph_build(emb, d)


def _path_graph(n):
    """Each node links to its left then its right neighbour on a line."""
    nbr = np.zeros((n, 2), np.int32)
    for i in range(n):
        nbr[i] = [max(i - 1, 0) if i > 0 else 1, min(i + 1, n - 1) if i < n - 1 else n - 2]
    return nbr


def test_search_traced_walk_along_a_path():
    # scores are the ids (1-d embeddings e_i = i, q = 1); from seed 0 with
    # beam 2 and width 1 the search walks right one node per iteration:
    #   it 1 expands 0 -> scores 1 -> C = [1, 0]
    #   it 2 expands 1 -> scores 2 -> C = [2, 1]     (0 drops out)
    #   ...      it 6 expands 5 -> nothing new; it 7 finds no parent: stop
    n = 6
    emb = np.arange(n, dtype=np.float32)[:, None]
    q = np.ones(1, np.float32)
    nbr = _path_graph(n)
    ids, sc, cnt, iters, scored = oracle.graph_search(q, emb, nbr, [0], beam=2, width=1,
                                                      max_iters=100, k=2)
    assert list(ids) == [5, 4] and list(sc) == [5.0, 4.0] and cnt == 2
    assert iters == 6 and scored == 6
    # stopped after 3 iterations: 0, 1, 2 expanded, C = [3, 2]
    ids, sc, cnt, iters, scored = oracle.graph_search(q, emb, nbr, [0], beam=2, width=1,
                                                      max_iters=3, k=2)
    assert list(ids) == [3, 2] and iters == 3 and scored == 4


def test_search_narrow_beam_is_trapped_wide_beam_escapes():
    # node 0 (seed) links to 1 (score 5) and 2 (score 1); 1 is a dead end
    # back to 0; 2 leads to 3 (score 9).  Beam 1 keeps only 1 and stops;
    # beam 2 keeps 2 as well, expands it and finds 3.
    emb = np.array([[0], [5], [1], [9]], np.float32)
    nbr = np.array([[1, 2], [0, 0], [3, 0], [2, 2]], np.int32)
    q = np.ones(1, np.float32)
    ids, _, _, _, _ = oracle.graph_search(q, emb, nbr, [0], beam=1, width=1, max_iters=50, k=1)
    assert list(ids) == [1]
    ids, _, _, _, _ = oracle.graph_search(q, emb, nbr, [0], beam=2, width=1, max_iters=50, k=2)
    assert list(ids) == [3, 1]
    # width 2 expands 1 and 2 in the same iteration
    ids, _, _, iters, _ = oracle.graph_search(q, emb, nbr, [0], beam=2, width=2, max_iters=50, k=2)
    assert list(ids) == [3, 1] and iters == 3
    # the seeds are cut to the beam before the first expansion: with beam 1
    # only seed 1 is a parent, even at width 2, so 3 is never reached
    ids, _, _, _, scored = oracle.graph_search(q, emb, nbr, [1, 2], beam=1, width=2, max_iters=50,
                                               k=1)
    assert list(ids) == [1] and scored == 3


def test_search_expands_the_best_unexpanded_entry_first():
    # 0 links to 1 (score 5) and 2 (score 1); 1 leads to 3 (score 8), 2 to 4
    # (score 9).  Best first, 1 is expanded, 3 enters the beam of 2 and
    # pushes 2 out before it is expanded, so 4 is never found:
    #   it 1 expands 0 -> C = [1, 2]; it 2 expands 1 -> C = [3, 1];
    #   it 3 expands 3 -> nothing new; it 4 finds no parent: stop
    emb = np.array([[0], [5], [1], [8], [9]], np.float32)
    nbr = np.array([[1, 2], [3, 0], [4, 0], [1, 1], [2, 2]], np.int32)
    ids, _, _, iters, scored = oracle.graph_search(np.ones(1, np.float32), emb, nbr, [0], beam=2,
                                                   width=1, max_iters=50, k=2)
    assert list(ids) == [3, 1] and iters == 3 and scored == 4


@pytest.mark.parametrize("seed", [3, 4])
def test_search_without_iterations_returns_the_best_seeds(seed):
    emb = _int_emb(30, 4, seed)
    q = _int_emb(1, 4, seed + 100)[0]
    nbr = oracle.graph_build(emb, 5)
    seeds = [7, 3, 7, 21, 9, 0, 3, 14]  # repeats are scored once
    ids, sc, cnt, iters, scored = oracle.graph_search(q, emb, nbr, seeds, beam=4, width=1,
                                                      max_iters=0, k=3)
    order, s = _exact_order(q, emb, sorted(set(seeds)))
    assert list(ids) == order[:3] and [int(x) for x in sc] == [s[j] for j in order[:3]]
    assert iters == 0 and scored == len(set(seeds)) and cnt == 3


@pytest.mark.parametrize("seed", [5, 6])
def test_search_on_a_complete_graph_is_the_exact_top_k(seed):
    n = 25
    emb = _int_emb(n, 5, seed)
    q = _int_emb(1, 5, seed + 100)[0]
    nbr = oracle.graph_build(emb, n - 1)
    ids, _, _, _, scored = oracle.graph_search(q, emb, nbr, [n - 1], beam=6, width=1,
                                               max_iters=1, k=6)
    order, _ = _exact_order(q, emb, list(range(n)))
    assert list(ids) == order[:6] and scored == n
    # and it agrees with the exact selection of the scan path
    assert list(ids) == list(oracle.topk(oracle.scores(q, emb), 6))


def test_search_short_beam_reports_fewer_results():
    emb = np.array([[1], [2], [3]], np.float32)
    nbr = np.array([[1], [0], [0]], np.int32)  # fact 2 is unreachable
    ids, sc, cnt, _, scored = oracle.graph_search(np.ones(1, np.float32), emb, nbr, [0], beam=4,
                                                  width=1, max_iters=10, k=3)
    assert cnt == 2 and list(ids) == [1, 0, -1] and scored == 2


@pytest.mark.parametrize("seed", [7, 8, 9])
def test_search_invariants_on_random_graphs(seed):
    rng = np.random.default_rng(seed)
    n, e = 200, 16
    emb = rng.standard_normal((n, e)).astype(np.float32)
    q = rng.standard_normal(e).astype(np.float32)
    nbr = oracle.graph_build(emb, 8)
    seeds = rng.integers(0, n, 6)
    ids, sc, cnt, iters, scored = oracle.graph_search(q, emb, nbr, seeds, beam=16, width=2,
                                                      max_iters=40, k=10)
    assert cnt == 10 and len(set(ids.tolist())) == 10
    exact = oracle.scores(q, emb)
    assert np.array_equal(sc, exact[ids])
    keys = list(zip((-sc).tolist(), ids.tolist()))
    assert keys == sorted(keys)
    # the results lie among the facts reachable from the seeds
    reach = set(int(s) for s in seeds)
    frontier = list(reach)
    while frontier:
        f = frontier.pop()
        for j in nbr[f]:
            if int(j) not in reach:
                reach.add(int(j))
                frontier.append(int(j))
    assert set(ids.tolist()) <= reach
    assert scored <= len(reach)


def test_search_rejects_bad_arguments():
    emb = np.zeros((4, 2), np.float32)
    nbr = np.zeros((4, 1), np.int32)
    q = np.zeros(2, np.float32)
    for kw in (dict(k=0), dict(k=5, beam=4), dict(width=0), dict(max_iters=-1)):
        args = dict(beam=4, width=1, max_iters=3, k=2)
        args.update(kw)
        with pytest.raises(ValueError):
            oracle.graph_search(q, emb, nbr, [0], **args)
    with pytest.raises(ValueError):
        oracle.graph_search(q, emb, nbr, [4], beam=4, width=1, max_iters=3, k=2)
    bad = np.full((4, 1), 9, np.int32)
    with pytest.raises(ValueError):
        oracle.graph_search(q, emb, bad, [0], beam=4, width=1, max_iters=3, k=2)
