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
The matrix form (`wy_outputs`) is checked against the definition.  Copies of
the recurrence with a planted mistake (a sign, a missing decay or write
strength, the decay on the wrong term, the key projection missing or on the
wrong side, the output taken before the update, the path applied leaf first)
must each fail at least one of the pins.
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


# ---- the pins catch plausible mistakes: each planted in a copy of the oracle's recurrence ----

def _path_variant(step, out_before=False, leaf_first=False):
    """path_outputs with the update `step(S, k, v, alpha, beta)` swapped in."""
    def fn(S0, q, k, v, alpha, beta, parent):
        S0 = np.asarray(S0, np.float64)
        q, k, v = (np.asarray(x, np.float64) for x in (q, k, v))
        alpha, beta = np.asarray(alpha, np.float64), np.asarray(beta, np.float64)
        o = np.zeros((q.shape[0], S0.shape[0], S0.shape[1]))
        for i in range(q.shape[0]):
            path = gdn.root_path(parent, i)
            if leaf_first:
                path = path[::-1]
            for h in range(S0.shape[0]):
                S = S0[h].copy()
                for t in path:
                    if out_before and t == i:
                        o[i, h] = S @ q[i, h]
                    S = step(S, k[t, h], v[t, h], alpha[t, h], beta[t, h])
                if not out_before:
                    o[i, h] = S @ q[i, h]
        return o
    return fn


def _right(S, k, v, a, b):
    return a * (S - b * np.outer(S @ k, k)) + b * np.outer(v, k)


MUTANTS = {
    "sign of the erase term": lambda S, k, v, a, b: a * (S + b * np.outer(S @ k, k)) + b * np.outer(v, k),
    "decay missing on the erase term": lambda S, k, v, a, b: a * S - b * np.outer(S @ k, k) + b * np.outer(v, k),
    "decay applied after the write": lambda S, k, v, a, b: a * (S - b * np.outer(S @ k, k) + b * np.outer(v, k)),
    "write strength missing on the value": lambda S, k, v, a, b: a * (S - b * np.outer(S @ k, k)) + np.outer(v, k),
    "erase term without the key projection": lambda S, k, v, a, b: a * (S - b * S) + b * np.outer(v, k),
    "erase term with the key on the wrong side": lambda S, k, v, a, b: _left_erase(S, k, v, a, b),
}


def _left_erase(S, k, v, a, b):
    """(I - b k k^T) S instead of S (I - b k k^T); only defined for square states."""
    if S.shape[0] != S.shape[1]:
        raise ValueError("left erase needs dv == dk")
    return a * (S - b * np.outer(k, k @ S)) + b * np.outer(v, k)


def _pins_pass(fn):
    """True when `fn` passes every pin of this file (shapes as in the tests above)."""
    ok = True
    try:
        cases = json.load(open(os.path.join(HERE, "golden", "worked_gdn.json")))["cases"]
        for c in cases:
            args = [np.array(c[x], np.float64) for x in ("S0", "q", "k", "v", "alpha", "beta")]
            ok &= np.allclose(fn(*args, np.array(c["parent"])), np.array(c["o"]), rtol=0, atol=1e-12)
        rng = np.random.default_rng(2)
        S0, q, k, v, alpha, beta, parent = random_case(rng, 24, 3, 8, 5)
        beta[:] = 1.0
        ok &= np.allclose(fn(S0, k.copy(), k, v, alpha, beta, parent), v, rtol=0, atol=1e-12)
        for dk, dv in [(5, 3), (3, 6), (4, 4)]:
            case = random_case(np.random.default_rng(10 + dk * 7 + dv), 18, 2, dk, dv, unit_keys=False)
            ok &= np.allclose(fn(*case), gdn.composite_outputs(*case), rtol=1e-11, atol=1e-11)
    except (ValueError, IndexError):  # a shape error is a failed pin too
        return False
    return bool(ok)


def test_pins_accept_the_oracle():
    assert _pins_pass(_path_variant(_right))
    assert _pins_pass(gdn.path_outputs)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_reject_planted_update_mistakes(name):
    assert not _pins_pass(_path_variant(MUTANTS[name])), name


def test_pins_reject_output_before_update_and_reversed_order():
    assert not _pins_pass(_path_variant(_right, out_before=True))
    assert not _pins_pass(_path_variant(_right, leaf_first=True))
