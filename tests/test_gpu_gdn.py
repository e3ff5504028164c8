"""Parity of the gated-delta-rule tree kernels (path and WY) with the oracle.

SpecPilot (arXiv 2611.02501), news article part (2) and English summary
section 4.2: every node's recurrent state is recomputed along its root path;
the WY kernel gets the same outputs through matrix products and may differ
from the path kernel only in rounding (within one BF16 ulp).

Tolerance.  Each output is a sum reached through at most 16 rank-one updates,
each with dot products of length D, in FP32 (plus S_0 split into two BF16
parts in the WY product, 2^-17 relative).  With N = 16 (D + 4) + D roundings
on the longest chain, |gpu - exact| <= (N 2^-24 + 2^-16) * A, where A is the
oracle's magnitude bound (the recurrence on absolute values).  The WY and
path outputs must also agree within one BF16 ulp of the path output, or
within that same bound where cancellation makes the output tiny.
"""
import numpy as np
import pytest
import torch

import lossless_bit_weight_02_gb300 as w12
from lossless_bit_weight_02_gb300 import synth
from oracle import gdn as ref

pytestmark = pytest.mark.gpu

MODES = (w12.W12_GDN_PATH, w12.W12_GDN_WY)


def f32_of_bits(b):
    return (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32)


def device_args(S0, q, k, v, alpha, beta, parent, req, use_req=True):
    bf = lambda b: torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).cuda()  # noqa
    t = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()  # noqa
    return (t(S0), bf(q), bf(k), bf(v), t(alpha), t(beta), t(parent), t(req) if use_req else None)


def oracle_of(S0, q, k, v, alpha, beta, parent, req):
    n, H, D = q.shape
    out = np.zeros((n, H, D))
    bound = np.zeros((n, H, D))
    qf, kf, vf = f32_of_bits(q), f32_of_bits(k), f32_of_bits(v)
    for r in np.unique(req):  # one request at a time (its nodes form their own tree)
        idx = np.flatnonzero(req == r)
        remap = {int(j): x for x, j in enumerate(idx)}
        par = np.array([remap[int(parent[j])] if parent[j] >= 0 else -1 for j in idx], np.int64)
        args = (S0[r], qf[idx], kf[idx], vf[idx], alpha[idx], beta[idx], par)
        out[idx] = ref.path_outputs(*args)
        bound[idx] = ref.abs_terms(*args)
    return out, bound


def tol_of(bound, D):
    N = 16 * (D + 4) + D
    return (N * 2.0 ** -24 + 2.0 ** -16) * bound


def bf16_ulp(x):
    x = np.abs(np.asarray(x, np.float32))
    e = np.floor(np.log2(np.maximum(x, np.float32(2.0 ** -126))))
    return 2.0 ** (e - 7)


def run(mode, args):
    call = w12.GdnCall(*args, mode=mode)
    out = call().clone()
    torch.cuda.synchronize()
    return out.cpu().numpy().astype(np.float64), call.status()


def check_case(inputs, use_req=True):
    S0, q, k, v, alpha, beta, parent, req = inputs
    D = q.shape[2]
    args = device_args(*inputs, use_req=use_req)
    want, bound = oracle_of(*inputs)
    tol = tol_of(bound, D)
    outs = {}
    for mode in MODES:
        o, st = run(mode, args)
        assert st == w12.W12_OK
        err = np.abs(o - want)
        assert np.all(err <= tol), (mode, float(np.max(err / np.maximum(tol, 1e-300))))
        o2, _ = run(mode, args)
        assert np.array_equal(o.view(np.int64), o2.view(np.int64)), "not deterministic"
        outs[mode] = o
    path, wy = outs[w12.W12_GDN_PATH], outs[w12.W12_GDN_WY]
    diff = np.abs(wy - path)
    assert np.all((diff <= bf16_ulp(path)) | (diff <= tol))
    return outs


@pytest.mark.parametrize("n,H,D,R,seed", [(1, 1, 64, 1, 0), (37, 3, 64, 1, 1), (63, 4, 128, 1, 2),
                                         (100, 2, 128, 3, 3), (129, 2, 64, 5, 4)])
def test_parity_random_trees(n, H, D, R, seed):
    check_case(synth.gdn_inputs(n, H, D, seed=seed, R=R))


def test_parity_without_req_array():
    inputs = synth.gdn_inputs(40, 2, 128, seed=11, R=1)
    check_case(inputs, use_req=False)


def test_chain_of_maximum_depth():
    parent = np.arange(-1, 15, dtype=np.int32)  # one chain of 16 nodes
    check_case(synth.gdn_inputs(16, 2, 128, seed=12, parent=parent))


def test_depth_over_limit_and_bad_parents_are_flagged():
    parent = np.arange(-1, 17, dtype=np.int32)  # 18 nodes: the last two are deeper than 16
    inputs = synth.gdn_inputs(18, 2, 64, seed=13, parent=parent)
    args = device_args(*inputs)
    want, bound = oracle_of(*[x[:16] if i else x for i, x in enumerate(inputs[:6])], parent[:16], inputs[7][:16])
    for mode in MODES:
        o, st = run(mode, args)
        assert st == w12.W12_ERR_INVALID
        assert np.all(np.isnan(o[16:])) and not np.any(np.isnan(o[:16]))
        assert np.all(np.abs(o[:16] - want) <= tol_of(bound, 64))
    # a parent that is not an earlier node, a child in another request, a bad request id
    for bad in ("forward", "cross", "range"):
        S0, q, k, v, alpha, beta, parent, req = synth.gdn_inputs(12, 1, 64, seed=14, R=2,
                                                                 parent=np.array([-1, 0, 1, -1, 3, 4, 0, 6, 7, 8, -1, 10],
                                                                                 np.int32),
                                                                 req=np.array([0, 0, 0, 1, 1, 1, 0, 0, 0, 0, 1, 1],
                                                                              np.int32))
        parent, req = parent.copy(), req.copy()
        if bad == "forward":
            parent[4] = 9
        elif bad == "cross":
            req[5] = 0
        else:
            req[10] = 7
        args = device_args(S0, q, k, v, alpha, beta, parent, req)
        for mode in MODES:
            o, st = run(mode, args)
            assert st == w12.W12_ERR_INVALID, (bad, mode)
            assert np.isnan(o[{"forward": 4, "cross": 5, "range": 10}[bad]]).all()
            assert not np.isnan(o[:3]).any()


def test_closed_forms_on_gpu():
    """beta = 0: o = gamma S_0 q (gamma = alpha multiplied along the path);
    beta = 1 with a one-hot key and q = k: the update stores v, so o = v."""
    S0, q, k, v, alpha, beta, parent, req = synth.gdn_inputs(30, 2, 128, seed=15)
    gamma = np.ones_like(alpha, dtype=np.float64)
    for i in range(30):
        gamma[i] = np.prod([alpha[t].astype(np.float64) for t in ref.root_path(parent, i)], axis=0)
    args = device_args(S0, q, k, v, alpha, np.zeros_like(beta), parent, req)
    qf = f32_of_bits(q).astype(np.float64)
    S0d = S0[0].astype(np.float64)
    want = gamma[:, :, None] * np.einsum("hvk,nhk->nhv", S0d, qf)
    bound = gamma[:, :, None] * np.einsum("hvk,nhk->nhv", np.abs(S0d), np.abs(qf))
    for mode in MODES:
        o, _ = run(mode, args)
        assert np.all(np.abs(o - want) <= 2.0 ** -15 * bound + 1e-30), mode
    onehot = np.zeros(q.shape, np.float32)
    hot = np.random.default_rng(21).integers(0, 128, size=q.shape[:2])
    np.put_along_axis(onehot, hot[:, :, None], 1.0, axis=2)
    kb = synth._to_bf16_bits(onehot)
    args = device_args(S0, kb, kb, v, alpha, np.ones_like(beta), parent, req)
    vf = f32_of_bits(v).astype(np.float64)
    for mode in MODES:
        o, _ = run(mode, args)
        np.testing.assert_allclose(o, vf, rtol=2.0 ** -20, atol=1e-6)


def test_empty_tree():
    inputs = synth.gdn_inputs(0, 2, 64, seed=16, parent=np.zeros(0, np.int32))
    for mode in MODES:
        o, st = run(mode, device_args(*inputs))
        assert o.shape == (0, 2, 64) and st == w12.W12_OK


def test_selected_tree_feeds_the_recurrence():
    """Best-first selection output (shared budget over 4 requests) as the tree."""
    rng = np.random.default_rng(17)
    R, Dp, C, B = 4, 8, 8, 63
    lp = torch.from_numpy(np.log(rng.dirichlet(np.full(C, 0.3), size=(R, Dp))).astype(np.float32)).cuda()
    sel = w12.w12_tree_select(lp, B, True)
    torch.cuda.synchronize()
    n = int(sel["count"][0])
    parent = sel["parent"][:n].cpu().numpy().astype(np.int32)
    req = sel["req"][:n].cpu().numpy().astype(np.int32)
    check_case(synth.gdn_inputs(n, 2, 128, seed=18, R=R, parent=parent, req=req))


def test_maximum_nodes():
    """1024 nodes (the limit) over 2 requests, 4 heads, D = 128."""
    check_case(synth.gdn_inputs(1024, 4, 128, seed=19, R=2))


@pytest.mark.parametrize("seed", range(10))
def test_random_shapes_and_gates(seed):
    """Seeded draws of size, heads, dimension, requests and tree shape, with
    decay and write strength over the whole [0, 1] (exact 0 and 1 included)."""
    rng = np.random.default_rng(900 + seed)
    n = int(rng.integers(1, 200))
    H = int(rng.integers(1, 4))
    D = int(rng.choice([64, 128]))
    R = int(rng.integers(1, 5))
    parent = synth.random_tree(n, seed=950 + seed, max_depth=int(rng.integers(1, 17)),
                               new_root=float(rng.uniform(0.02, 0.5)))
    S0, q, k, v, alpha, beta, parent, req = synth.gdn_inputs(n, H, D, seed=970 + seed, R=R, parent=parent)
    alpha = rng.uniform(0.0, 1.0, size=alpha.shape).astype(np.float32)
    beta = rng.uniform(0.0, 1.0, size=beta.shape).astype(np.float32)
    pick = rng.random(alpha.shape)
    alpha[pick < 0.05] = 0.0
    alpha[pick > 0.9] = 1.0
    beta[pick < 0.1] = 1.0
    beta[(pick > 0.5) & (pick < 0.55)] = 0.0
    check_case((S0, q, k, v, alpha, beta, parent, req))
