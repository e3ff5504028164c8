"""Best-first draft-tree node selection: plain CPU reference.

TEST INFRASTRUCTURE ONLY.  Only the test suite and the benchmark's CPU legs
may import this module; the product path never calls it.

SpecPilot (arXiv 2611.02501), the news article's part "(2) best-first tree
verification" and the English summary's section 6.4 bullet (best-first trees
on the 8-position lattice, 32 and 63 nodes) and section 4.4 bullet (a node
budget shared across requests):
  * a drafter proposes, for every request r, position d and candidate c, a
    log-probability lp[r][d][c] of that candidate given the prefix before it
    (the lattice of a block drafter: the distribution at position d does not
    depend on which candidates were picked before it);
  * a node is a path (c_0, ..., c_{t-1}) from the root, depth t >= 1; its
    score is the cumulative log-probability of the path, summed left to
    right in FP32: score(child) = score(parent) + lp[r][t-1][c_{t-1}];
  * best-first: starting from the root, repeatedly keep the frontier node
    (a child of a kept node, or of the root) with the highest score, and add
    its children to the frontier, until the node budget is spent.  With a
    shared budget the frontier spans all requests.
Ties (the pages give no rule) are broken by the total order
    score descending, depth ascending, request ascending, path ascending
    (lexicographic on candidate indices).
A child never comes before its parent in this order (its score is at most
the parent's, and on a tie its depth is larger), so the kept set is always
a tree and equals the first `budget` nodes of the whole lattice in this
order; `select_bruteforce` checks that on small lattices.

Each function states the passage it follows; scores are numpy float32, so
every addition is one FP32 rounding, as on the GPU.
"""
from __future__ import annotations

import itertools

import numpy as np


def order_key(score, depth, req, path):
    """Sort key of a node: smaller is kept first (score descending, depth,
    request, path ascending)."""
    return (-float(score), int(depth), int(req), tuple(int(c) for c in path))


def select(lp: np.ndarray, budget: int, shared: bool):
    """Best-first selection (news article part (2), summary sections 4.4 and 6.4).

    lp: float32 [R, D, C].  shared=False: `budget` nodes per request, each
    request on its own; shared=True: `budget` nodes over all requests.
    Returns a list of nodes (req, depth, path tuple, score float32, parent
    index in the returned list or -1) in selection order; with shared=False
    the requests follow one another (request 0's nodes first).
    """
    lp = np.asarray(lp, dtype=np.float32)
    R, D, C = lp.shape
    groups = [list(range(R))] if shared else [[r] for r in range(R)]
    out = []
    for reqs in groups:
        # frontier entries: (key, req, depth, path, score, parent index in `out`)
        frontier = []
        for r in reqs:
            for c in range(C):
                s = np.float32(lp[r, 0, c])
                frontier.append((order_key(s, 1, r, (c,)), r, 1, (c,), s, -1))
        kept = 0
        while kept < budget and frontier:
            best = min(range(len(frontier)), key=lambda i: frontier[i][0])  # plain linear scan
            _, r, t, path, s, parent = frontier.pop(best)
            me = len(out)
            out.append((r, t, path, s, parent))
            kept += 1
            if t < D:
                for c in range(C):
                    cs = np.float32(s + lp[r, t, c])  # one FP32 addition
                    frontier.append((order_key(cs, t + 1, r, path + (c,)), r, t + 1, path + (c,), cs, me))
    return out


def all_nodes(lp: np.ndarray):
    """Every node of every request's lattice with its FP32 score (small inputs only)."""
    lp = np.asarray(lp, dtype=np.float32)
    R, D, C = lp.shape
    nodes = []
    for r in range(R):
        for t in range(1, D + 1):
            for path in itertools.product(range(C), repeat=t):
                s = np.float32(lp[r, 0, path[0]])
                for i in range(1, t):
                    s = np.float32(s + lp[r, i, path[i]])
                nodes.append((r, t, path, s))
    return nodes


def select_bruteforce(lp: np.ndarray, budget: int, shared: bool):
    """The first `budget` nodes of the whole lattice in the total order, by
    sorting every node (small inputs only).  Same output as `select`."""
    lp = np.asarray(lp, dtype=np.float32)
    R = lp.shape[0]
    nodes = all_nodes(lp)
    groups = [list(range(R))] if shared else [[r] for r in range(R)]
    out = []
    for reqs in groups:
        cand = sorted((n for n in nodes if n[0] in reqs), key=lambda n: order_key(n[3], n[1], n[0], n[2]))
        base = len(out)
        chosen = cand[:budget]
        index = {(n[0], n[2]): base + i for i, n in enumerate(chosen)}
        for r, t, path, s in chosen:
            out.append((r, t, path, s, index[(r, path[:-1])] if t > 1 else -1))
    return out


def pack_path(path) -> int:
    """Candidate indices packed 4 bits per position, position 0 lowest."""
    v = 0
    for i, c in enumerate(path):
        v |= int(c) << (4 * i)
    return v
