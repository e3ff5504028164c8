"""Gated delta rule along the root paths of a draft tree: plain CPU reference.

TEST INFRASTRUCTURE ONLY.  Only the test suite and the benchmark's CPU legs
may import this module; the product path never calls it.

SpecPilot (arXiv 2611.02501): the news article's part (2) (best-first tree
verification on hybrid models whose recurrent layers are Gated DeltaNet) and
the English summary's section 4.2 bullet on hybrid targets.  Together they
fix what is computed, though not the recurrence itself:
  * the recurrent state of a tree node is not stored; it is recomputed from
    the root state along the node's root path (the "path kernel");
  * the WY verify kernel gets the same outputs by turning that chain of
    rank-one state updates into matrix products, and differs from the path
    kernel only in rounding (within one BF16 ulp).
The pages do not write the recurrence out.  The reading taken is the
published gated delta rule of Gated DeltaNet, per head, with the state S a
dv x dk matrix (row = value index, column = key index):
    S_t = alpha_t * S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T
    o_t = S_t q_t
for the nodes t of a root path in root-to-node order, S_0 the state before
the tree (shared by every path).  Each rank-one update is the chain link the
pages speak of.

Two functions compute the per-node outputs:
  * `path_outputs` is the definition: for every node, start from S_0 and
    apply the updates of its root path one by one, in FP64;
  * `wy_outputs` is the matrix form the GPU's WY kernel uses, in FP64: with
    gamma_t the product of alpha along the path down to t, f_t the rank-one
    coefficient vectors and Gamma_tj = gamma_t / gamma_j (the product of
    alpha over the nodes below j down to t, so no division is needed),
        f_t = beta_t (v_t - gamma_t S_0 k_t - sum_{j<t} Gamma_tj (k_t . k_j) f_j)
        o_t = gamma_t S_0 q_t + sum_{j<=t} Gamma_tj (q_t . k_j) f_j
    (j over the ancestors of t and t itself).  S_0 enters only through
    K S_0^T and Q S_0^T, one product over all nodes.
The tests pin `path_outputs` to closed forms (pure decay, the delta rule
writing v at a unit key, linearity) and to the composition of the per-step
affine maps, and pin `wy_outputs` to `path_outputs`.
"""
from __future__ import annotations

import numpy as np


def depths(parent) -> np.ndarray:
    """Depth of every node (children of the root have depth 1); parent[i] < i."""
    parent = np.asarray(parent, dtype=np.int64)
    d = np.zeros(len(parent), dtype=np.int64)
    for i, p in enumerate(parent):
        if not (-1 <= p < i):
            raise ValueError(f"parent[{i}] = {p} is not in [-1, {i})")
        d[i] = 1 if p < 0 else d[p] + 1
    return d


def root_path(parent, i: int) -> list:
    """The nodes from the root's child down to node i, root side first."""
    path = []
    while i >= 0:
        path.append(int(i))
        i = int(parent[i])
    return path[::-1]


def path_outputs(S0, q, k, v, alpha, beta, parent) -> np.ndarray:
    """Per-node outputs by the definition: the gated delta rule applied along
    each node's root path, one rank-one update at a time, in FP64.

    S0: [H, dv, dk]; q, k: [n, H, dk]; v: [n, H, dv]; alpha, beta: [n, H];
    parent: [n] with parent[i] in [-1, i).  Returns o: [n, H, dv] float64.
    """
    S0 = np.asarray(S0, np.float64)
    q, k, v = (np.asarray(x, np.float64) for x in (q, k, v))
    alpha, beta = np.asarray(alpha, np.float64), np.asarray(beta, np.float64)
    n, H = q.shape[0], S0.shape[0]
    depths(parent)  # checks the tree
    o = np.zeros((n, H, S0.shape[1]))
    for i in range(n):
        path = root_path(parent, i)
        for h in range(H):
            S = S0[h].copy()
            for t in path:
                kt = k[t, h]
                # S <- alpha S (I - beta k k^T) + beta v k^T
                S = alpha[t, h] * (S - beta[t, h] * np.outer(S @ kt, kt)) + beta[t, h] * np.outer(v[t, h], kt)
            o[i, h] = S @ q[i, h]
    return o


def composite_outputs(S0, q, k, v, alpha, beta, parent) -> np.ndarray:
    """The same outputs through explicit matrices: every update is the affine
    map S -> S M_t + C_t with M_t = alpha_t (I - beta_t k_t k_t^T) and
    C_t = beta_t v_t k_t^T; a path composes them as S_0 (M_1 ... M_L) plus the
    carried C terms (library matrix products, small inputs only)."""
    S0 = np.asarray(S0, np.float64)
    q, k, v = (np.asarray(x, np.float64) for x in (q, k, v))
    alpha, beta = np.asarray(alpha, np.float64), np.asarray(beta, np.float64)
    n, H, dk = k.shape
    o = np.zeros((n, H, S0.shape[1]))
    for i in range(n):
        path = root_path(parent, i)
        for h in range(H):
            P = np.eye(dk)
            C = np.zeros_like(S0[h])
            for t in path:
                M = alpha[t, h] * (np.eye(dk) - beta[t, h] * np.outer(k[t, h], k[t, h]))
                P = P @ M
                C = C @ M + beta[t, h] * np.outer(v[t, h], k[t, h])
            o[i, h] = (S0[h] @ P + C) @ q[i, h]
    return o


def wy_outputs(S0, q, k, v, alpha, beta, parent) -> np.ndarray:
    """Per-node outputs through the matrix form (module docstring), FP64:
    one product of all keys and queries with S_0, then the coefficient
    vectors f in node order (ancestors come first since parent[i] < i)."""
    S0 = np.asarray(S0, np.float64)
    q, k, v = (np.asarray(x, np.float64) for x in (q, k, v))
    alpha, beta = np.asarray(alpha, np.float64), np.asarray(beta, np.float64)
    n, H = q.shape[0], S0.shape[0]
    depths(parent)
    KS = np.einsum("nhk,hvk->nhv", k, S0)  # k_t S_0^T for every node
    QS = np.einsum("nhk,hvk->nhv", q, S0)
    f = np.zeros((n, H, S0.shape[1]))
    o = np.zeros_like(f)
    for i in range(n):
        path = root_path(parent, i)  # root side first, ends with i
        for h in range(H):
            # ratio[j] = Gamma_ij: the product of alpha over the path nodes after j, up to i
            ratio = {}
            r = 1.0
            for j in reversed(path):
                ratio[j] = r
                r *= alpha[j, h]
            gamma = r  # alpha multiplied over the whole path
            acc = v[i, h] - gamma * KS[i, h]
            for j in path[:-1]:
                acc = acc - ratio[j] * (k[i, h] @ k[j, h]) * f[j, h]
            f[i, h] = beta[i, h] * acc
            out = gamma * QS[i, h]
            for j in path:
                out = out + ratio[j] * (q[i, h] @ k[j, h]) * f[j, h]
            o[i, h] = out
    return o


def abs_terms(S0, q, k, v, alpha, beta, parent) -> np.ndarray:
    """A bound on the magnitudes summed into each output: the path recurrence
    run on |S_0|, |q|, |k|, |v| with every subtraction turned into an addition.
    Rounding errors of any evaluation order are a small multiple of unit
    roundoff times this (used for the tolerance)."""
    S0 = np.abs(np.asarray(S0, np.float64))
    q, k, v = (np.abs(np.asarray(x, np.float64)) for x in (q, k, v))
    alpha, beta = np.abs(np.asarray(alpha, np.float64)), np.abs(np.asarray(beta, np.float64))
    n, H = q.shape[0], S0.shape[0]
    o = np.zeros((n, H, S0.shape[1]))
    for i in range(n):
        path = root_path(parent, i)
        for h in range(H):
            S = S0[h].copy()
            for t in path:
                kt = k[t, h]
                S = alpha[t, h] * (S + beta[t, h] * np.outer(S @ kt, kt)) + beta[t, h] * np.outer(v[t, h], kt)
            o[i, h] = S @ q[i, h]
    return o
