"""The seeded GDN tree input generator (CPU only): shapes, types, the tree
rules the library enforces on the device, request inheritance, and seeding."""
import numpy as np
import pytest

from lossless_bit_weight_02_gb300 import synth


def f32(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


@pytest.mark.parametrize("n,max_depth", [(1, 16), (50, 1), (300, 16), (1024, 7)])
def test_random_tree_rules(n, max_depth):
    parent = synth.random_tree(n, seed=n + max_depth, max_depth=max_depth)
    assert parent.dtype == np.int32 and parent.shape == (n,)
    depth = np.zeros(n, np.int64)
    for i, p in enumerate(parent):
        assert -1 <= p < i
        depth[i] = 1 if p < 0 else depth[p] + 1
    assert depth.max() <= max_depth
    if max_depth == 1:
        assert np.all(parent == -1)


def test_gdn_inputs_shapes_and_ranges():
    S0, q, k, v, alpha, beta, parent, req = synth.gdn_inputs(64, 3, 128, seed=5, R=4)
    assert S0.shape == (4, 3, 128, 128) and S0.dtype == np.float32
    for x in (q, k, v):
        assert x.shape == (64, 3, 128) and x.dtype == np.uint16
    assert alpha.shape == beta.shape == (64, 3) and alpha.dtype == beta.dtype == np.float32
    assert np.all((alpha >= 0.85) & (alpha <= 1.0)) and np.all((beta >= 0.1) & (beta <= 0.9))
    # unit-length q and k before the BF16 cast: within the cast's error after it
    for x in (q, k):
        norms = np.linalg.norm(f32(x).astype(np.float64), axis=-1)
        assert np.all(np.abs(norms - 1.0) < 2.0 ** -7)
    assert np.all((req >= 0) & (req < 4))
    for i, p in enumerate(parent):
        if p >= 0:
            assert req[i] == req[p]


def test_gdn_inputs_are_seeded():
    a = synth.gdn_inputs(20, 2, 64, seed=9, R=2)
    b = synth.gdn_inputs(20, 2, 64, seed=9, R=2)
    c = synth.gdn_inputs(20, 2, 64, seed=10, R=2)
    assert all(np.array_equal(x, y) for x, y in zip(a, b))
    assert not np.array_equal(a[1], c[1])


def test_gdn_inputs_keep_a_given_tree():
    parent = np.array([-1, 0, 0, 1, -1, 4], np.int32)
    req = np.array([1, 1, 1, 1, 0, 0], np.int32)
    out = synth.gdn_inputs(6, 1, 64, seed=3, R=2, parent=parent, req=req)
    assert np.array_equal(out[6], parent) and np.array_equal(out[7], req)
