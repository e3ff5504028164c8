"""GPU best-first draft-tree node selection (w12_tree_select) against the oracle.

SpecPilot (arXiv 2611.02501), news article part "(2) best-first tree
verification", English summary sections 4.4 (node budget shared across
requests) and 6.4 (best-first trees on an 8-position lattice).  The kept
nodes, their order, paths, FP32 scores and parent links must equal the
oracle's exactly (integers and orders are exact; both sides add the
log-probabilities in FP32 in the same order).
"""
import numpy as np
import pytest
import torch

from oracle import tree

pytestmark = pytest.mark.gpu


def gpu_select(w12lib, lp, budget, shared):
    out = w12lib.w12_tree_select(torch.from_numpy(lp).cuda(), budget, shared)
    torch.cuda.synchronize()
    o = {k: v.cpu().numpy() for k, v in out.items()}
    R = lp.shape[0]
    nodes = []
    if shared:
        for i in range(int(o["count"][0])):
            nodes.append((int(o["req"][i]), int(o["depth"][i]), int(o["path"][i]), np.float32(o["score"][i]),
                          int(o["parent"][i])))
        return nodes
    # segments of `budget` entries per request -> the oracle's compact order
    off = np.concatenate([[0], np.cumsum(o["count"])])
    for r in range(R):
        for i in range(int(o["count"][r])):
            p = int(o["parent"][r, i])
            if p >= 0:
                assert p // budget == r
                p = int(off[r]) + p % budget
            nodes.append((int(o["req"][r, i]), int(o["depth"][r, i]), int(o["path"][r, i]),
                          np.float32(o["score"][r, i]), p))
    return nodes


def oracle_select(lp, budget, shared):
    return [(r, t, tree.pack_path(path), s, p) for r, t, path, s, p in tree.select(lp, budget, shared)]


def check(w12lib, lp, budget, shared):
    want = oracle_select(lp, budget, shared)
    got = gpu_select(w12lib, lp, budget, shared)
    assert len(got) == len(want)
    for i, (g, w) in enumerate(zip(got, want)):
        assert g[:3] == w[:3] and g[4] == w[4], (i, g, w)
        assert g[3] == w[3] and np.signbit(g[3]) == np.signbit(w[3]), (i, g, w)


def lattice(rng, R, D, C, kind):
    if kind == "dirichlet":
        return np.log(rng.dirichlet(np.full(C, 0.3), size=(R, D))).astype(np.float32)
    if kind == "ties":  # few distinct values, zeros included: equal scores everywhere
        return (-rng.integers(0, 3, size=(R, D, C)) / 2).astype(np.float32)
    return np.zeros((R, D, C), np.float32)


@pytest.mark.parametrize("R,D,C,budget", [(1, 8, 8, 32), (1, 16, 8, 63), (3, 16, 8, 256), (64, 8, 8, 32),
                                          (5, 1, 16, 20), (4, 4, 1, 6), (2, 16, 16, 200), (7, 3, 5, 64)])
@pytest.mark.parametrize("kind", ["dirichlet", "ties"])
@pytest.mark.parametrize("shared", [False, True])
def test_tree_select_parity(R, D, C, budget, kind, shared, w12lib):
    rng = np.random.default_rng(R * 1000 + D * 10 + C + budget)
    check(w12lib, lattice(rng, R, D, C, kind), budget, shared)


@pytest.mark.parametrize("shared", [False, True])
def test_tree_select_zero_logprobs_and_small_lattices(shared, w12lib):
    rng = np.random.default_rng(5)
    check(w12lib, lattice(rng, 3, 3, 2, "zeros"), 256, shared)  # 14 nodes per request: every node, BFS order
    check(w12lib, lattice(rng, 2, 2, 2, "dirichlet"), 5, shared)


def test_tree_select_shared_budget_over_many_requests(w12lib):
    rng = np.random.default_rng(11)
    check(w12lib, lattice(rng, 96, 8, 8, "dirichlet"), 256, True)


def test_tree_select_worked_example(w12lib):
    import test_oracle_tree
    lp, cases = test_oracle_tree.read_worked()
    for shared, budget, want in cases:
        got = gpu_select(w12lib, lp, budget, shared)
        assert got == [(r, t, tree.pack_path(p), s, pa) for r, t, p, s, pa in want]


def test_tree_select_shared_budget_falls_back_when_one_request_dominates(w12lib):
    """Request 0's log-probabilities are near 0, the others' near -10: the whole shared budget
    goes to request 0, past its first-pass list (2*ceil(256/8) + 4 = 68 nodes), so the second
    pass with full lists must run."""
    rng = np.random.default_rng(12)
    lp = np.log(rng.dirichlet(np.full(8, 0.3), size=(8, 16))).astype(np.float32) - 10
    lp[0] = -rng.random((16, 8)).astype(np.float32) * 0.01
    want = oracle_select(lp, 256, True)
    assert all(n[0] == 0 for n in want)
    check(w12lib, lp, 256, True)
    # and the next call on the same lattice shape (first pass enough) is still right
    check(w12lib, lattice(rng, 8, 16, 8, "dirichlet"), 256, True)


@pytest.mark.parametrize("shared", [False, True])
def test_tree_select_signed_zero_scores(shared, w12lib):
    """-0.0 log-probabilities: scores keep the sign of zero of the FP32 sums, and -0 ties +0."""
    lp = np.array([[[-0.0, 0.0, -1.0], [-0.0, -0.5, 0.0]], [[0.0, -0.0, -2.0], [-0.25, -0.0, 0.0]]], np.float32)
    check(w12lib, lp, 8, shared)
