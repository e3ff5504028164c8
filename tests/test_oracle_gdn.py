"""Pins for the gated-delta-rule tree oracle (CPU only).

SpecPilot (arXiv 2611.02501), news article part (2) (tree verification on
hybrid models with Gated DeltaNet layers) and English summary section 4.2
(the state is recomputed along each root path; the WY kernel turns the chain
of rank-one updates into matrix products).  The definition
(`path_outputs`) is checked against:
  * hand-worked examples (tests/golden/worked_gdn.json);
  * closed forms: beta = 0 leaves only the decay (o = gamma S_0 q); with
    beta = 1 and a unit key the update stores v at that key (S k = v), for any
    alpha; the output is linear in (S_0, v) jointly;
  * the composition of explicit per-step affine maps (library matrix
    products), with dk != dv so that a transposed state shows;
  * prefix independence: a node's output does not depend on other branches.
The matrix form (`wy_outputs`) is checked against the definition.
"""
import json
import os

import numpy as np
import pytest

from oracle import gdn

HERE = os.path.dirname(os.path.abspath(__file__))


def random_tree(rng, n, max_depth=16):
    parent = np.full(n, -1, np.int64)
    depth = np.zeros(n, np.int64)
    for i in range(n):
        cand = [j for j in range(i) if depth[j] < max_depth]
        p = -1 if (i == 0 or rng.random() < 0.2) else int(rng.choice(cand))
        parent[i] = p
        depth[i] = 1 if p < 0 else depth[p] + 1
    return parent


def random_case(rng, n, H, dk, dv, parent=None, unit_keys=True):
    S0 = rng.normal(size=(H, dv, dk))
    q = rng.normal(size=(n, H, dk))
    k = rng.normal(size=(n, H, dk))
    if unit_keys:  # the model L2-normalises its keys
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.normal(size=(n, H, dv))
    alpha = rng.uniform(0.05, 1.0, size=(n, H))
    beta = rng.uniform(0.0, 1.0, size=(n, H))
    if parent is None:
        parent = random_tree(rng, n)
    return S0, q, k, v, alpha, beta, parent


def test_worked_examples():
    cases = json.load(open(os.path.join(HERE, "golden", "worked_gdn.json")))["cases"]
    for c in cases:
        args = [np.array(c[x], np.float64) for x in ("S0", "q", "k", "v", "alpha", "beta")]
        parent = np.array(c["parent"], np.int64)
        o = gdn.path_outputs(*args, parent)
        np.testing.assert_array_equal(o, np.array(c["o"]), err_msg=c["name"])
        np.testing.assert_allclose(gdn.wy_outputs(*args, parent), np.array(c["o"]), rtol=0, atol=1e-13)


def test_beta_zero_is_pure_decay():
    rng = np.random.default_rng(1)
    S0, q, k, v, alpha, beta, parent = random_case(rng, 20, 2, 6, 4)
    beta[:] = 0.0
    o = gdn.path_outputs(S0, q, k, v, alpha, beta, parent)
    for i in range(len(parent)):
        gamma = np.prod([alpha[t] for t in gdn.root_path(parent, i)], axis=0)  # [H]
        for h in range(S0.shape[0]):
            np.testing.assert_allclose(o[i, h], gamma[h] * (S0[h] @ q[i, h]), rtol=1e-12, atol=1e-14)


def test_delta_rule_stores_value_at_unit_key():
    # beta = 1, |k| = 1: S_t k_t = alpha S k - alpha S k (k.k) + v (k.k) = v, whatever alpha and the history
    rng = np.random.default_rng(2)
    S0, q, k, v, alpha, beta, parent = random_case(rng, 24, 3, 8, 5)
    beta[:] = 1.0
    q = k.copy()
    o = gdn.path_outputs(S0, q, k, v, alpha, beta, parent)
    np.testing.assert_allclose(o, v, rtol=0, atol=1e-12)


def test_linear_in_state_and_values():
    rng = np.random.default_rng(3)
    S0, q, k, v, alpha, beta, parent = random_case(rng, 15, 2, 5, 7)
    S0b, vb = rng.normal(size=S0.shape), rng.normal(size=v.shape)
    oa = gdn.path_outputs(S0, q, k, v, alpha, beta, parent)
    ob = gdn.path_outputs(S0b, q, k, vb, alpha, beta, parent)
    oab = gdn.path_outputs(S0 + S0b, q, k, v + vb, alpha, beta, parent)
    np.testing.assert_allclose(oab, oa + ob, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("dk,dv", [(5, 3), (3, 6), (4, 4)])
def test_matches_composed_affine_maps(dk, dv):
    rng = np.random.default_rng(10 + dk * 7 + dv)
    case = random_case(rng, 18, 2, dk, dv, unit_keys=False)
    o = gdn.path_outputs(*case)
    np.testing.assert_allclose(gdn.composite_outputs(*case), o, rtol=1e-11, atol=1e-11)


def test_prefix_independence():
    rng = np.random.default_rng(4)
    S0, q, k, v, alpha, beta, parent = random_case(rng, 30, 2, 6, 6)
    o = gdn.path_outputs(S0, q, k, v, alpha, beta, parent)
    for i in (5, 17, 29):
        path = gdn.root_path(parent, i)
        sub_parent = np.array([-1] + list(range(len(path) - 1)), np.int64)  # the path as a chain
        sub = [x[path] for x in (q, k, v, alpha, beta)]
        o_sub = gdn.path_outputs(S0, *sub, sub_parent)
        np.testing.assert_array_equal(o_sub[-1], o[i])


@pytest.mark.parametrize("seed", range(4))
def test_wy_form_matches_definition(seed):
    rng = np.random.default_rng(100 + seed)
    dk, dv = [(8, 8), (6, 9), (16, 4), (7, 7)][seed]
    case = random_case(rng, 40, 2, dk, dv, unit_keys=seed % 2 == 0)
    S0, q, k, v, alpha, beta, parent = case
    if seed == 3:
        alpha[:] = rng.uniform(0.0, 0.02, size=alpha.shape)  # strong decay, gamma far below 1
        alpha[::5] = 0.0  # a full reset on some nodes
    o = gdn.path_outputs(*case)
    scale = gdn.abs_terms(*case)
    np.testing.assert_array_less(np.abs(gdn.wy_outputs(*case) - o), 1e-12 * scale + 1e-300)
    assert np.all(np.abs(o) <= scale * (1 + 1e-12))


def test_depth_limit_and_bad_parent():
    chain = np.array([-1] + list(range(15)), np.int64)
    assert gdn.depths(chain).max() == 16
    with pytest.raises(ValueError):
        gdn.depths(np.array([-1, 1, 0]))
    with pytest.raises(ValueError):
        gdn.depths(np.array([-2]))
