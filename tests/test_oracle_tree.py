"""Pins for the best-first draft-tree oracle (CPU only).

SpecPilot (arXiv 2611.02501), news article part "(2) best-first tree
verification" (rank nodes by their log-probability given the parent, keep the
highest cumulative path score first), English summary sections 4.4 (a node
budget shared across requests) and 6.4 (best-first trees on an 8-position
lattice).  The oracle's best-first expansion is checked against:
  * a hand-worked example (tests/golden/worked_tree.txt);
  * brute force: every node of small lattices sorted by the total order,
    first `budget` kept, many ties included;
  * closed cases: a one-candidate chain, all-zero log-probabilities
    (breadth-first order), a budget above the node count (every node);
  * invariants on the 8-position, 8-candidate lattice at 32 and 63 nodes.
"""
import os

import numpy as np
import pytest

from oracle import tree

HERE = os.path.dirname(os.path.abspath(__file__))


def read_worked():
    lines = [l.split("#")[0].strip() for l in open(os.path.join(HERE, "golden", "worked_tree.txt"))]
    lines = [l for l in lines if l]
    R, D, C = map(int, lines[0].split()[1:])
    lp = np.array([[float(x) for x in lines[1 + i].split()] for i in range(R * D)], np.float32).reshape(R, D, C)
    cases, i = [], 1 + R * D
    while i < len(lines):
        _, mode, budget = lines[i].split()
        i += 1
        nodes = []
        while i < len(lines) and not lines[i].startswith("select"):
            r, t, path, s, parent = lines[i].split()
            nodes.append((int(r), int(t), tuple(int(c) for c in path.split(",")), np.float32(s), int(parent)))
            i += 1
        cases.append((mode == "shared", int(budget), nodes))
    return lp, cases


def test_worked_example():
    lp, cases = read_worked()
    for shared, budget, want in cases:
        got = tree.select(lp, budget, shared)
        assert got == want, (shared, got)


@pytest.mark.parametrize("seed", range(40))
def test_equals_bruteforce_on_small_lattices(seed):
    rng = np.random.default_rng(seed)
    R, D, C = int(rng.integers(1, 4)), int(rng.integers(1, 5)), int(rng.integers(1, 4))
    if seed % 2:  # few distinct values: many equal scores, zeros (children tying their parents)
        lp = -rng.integers(0, 3, size=(R, D, C)).astype(np.float32) / 2
    else:
        lp = np.log(rng.dirichlet(np.ones(C), size=(R, D))).astype(np.float32)
    total = R * sum(C ** t for t in range(1, D + 1))
    for budget in (1, 2, 5, total // 2 + 1, total + 3):
        for shared in (False, True):
            assert tree.select(lp, budget, shared) == tree.select_bruteforce(lp, budget, shared)


def test_chain_of_one_candidate():
    lp = np.array([[[-0.5], [-0.25], [-1.0], [-2.0]]], np.float32)
    got = tree.select(lp, 3, False)
    assert [n[2] for n in got] == [(0,), (0, 0), (0, 0, 0)]
    assert [n[3] for n in got] == [np.float32(-0.5), np.float32(-0.75), np.float32(-1.75)]
    assert [n[4] for n in got] == [-1, 0, 1]


def test_zero_logprobs_give_breadth_first_order():
    lp = np.zeros((1, 3, 2), np.float32)
    got = tree.select(lp, 14, False)
    assert [n[2] for n in got] == [(0,), (1,), (0, 0), (0, 1), (1, 0), (1, 1),
                                   (0, 0, 0), (0, 0, 1), (0, 1, 0), (0, 1, 1), (1, 0, 0), (1, 0, 1), (1, 1, 0),
                                   (1, 1, 1)]


def test_budget_above_node_count_keeps_every_node():
    rng = np.random.default_rng(7)
    lp = np.log(rng.dirichlet(np.ones(3), size=(2, 3))).astype(np.float32)
    got = tree.select(lp, 1000, True)
    assert len(got) == 2 * (3 + 9 + 27)
    assert sorted((n[0], n[2]) for n in got) == sorted((n[0], n[2]) for n in tree.all_nodes(lp))


@pytest.mark.parametrize("budget", [32, 63])
@pytest.mark.parametrize("shared", [False, True])
def test_invariants_on_the_8_position_lattice(budget, shared):
    rng = np.random.default_rng(budget)
    lp = np.log(rng.dirichlet(np.full(8, 0.3), size=(3, 8))).astype(np.float32)
    got = tree.select(lp, budget, shared)
    assert len(got) == (budget if shared else 3 * budget)
    keys = [tree.order_key(s, t, r, p) for r, t, p, s, _ in got]
    for i, (r, t, path, s, parent) in enumerate(got):
        if t == 1:
            assert parent == -1 and s == lp[r, 0, path[0]]
        else:
            pr, pt, ppath, ps, _ = got[parent]
            assert parent < i and pr == r and pt == t - 1 and ppath == path[:-1]
            assert s == np.float32(ps + lp[r, t - 1, path[-1]])
    groups = [keys] if shared else [keys[i * budget:(i + 1) * budget] for i in range(3)]
    for g in groups:
        assert g == sorted(g)


def test_pack_path():
    assert tree.pack_path((3, 0, 15, 1)) == 3 | (15 << 8) | (1 << 12)
