"""Full-size workloads: the 64-layer weight stack and the escape-stress shape.

SpecPilot (arXiv 2611.02501), section 4.1: every decoded tensor is checked bit
for bit at load time, and the verify passes stream every target weight.  The
stack test converts 64 layers of the 27B-class shapes to W12 on the GPU (each
tensor verified bit for bit, the BF16 copy freed), streams the 256 GEMMs at
M = 1 and M = 16, and checks sampled outputs of layers 0 and 63 against the
oracle.  The stress test runs N = 5121, K = 17400 with heavy-tailed weights,
zero rows, denormals and maximum-exponent values at M = 1, 7, 33, each on ten
grid sizes (w12_gemm_opts.max_ctas), bitwise identical.
"""
import numpy as np
import pytest
import torch

from lossless_bit_weight_02_gb300 import synth
from w12_tol import gemm_tolerance_failures

pytestmark = pytest.mark.gpu


def sampled_check(w12lib, oracle, Wd, t, Ad, Y, rng, count=24):
    N = t.N
    M = Ad.shape[0]
    ns = rng.choice(N, size=count, replace=False)
    ms = rng.integers(0, M, size=count)
    Wh = synth.tensor_to_bits(Wd[torch.from_numpy(ns).cuda()])
    st, ref = oracle.encode(Wh)
    st, y, y64, mag = oracle.gemm_sample(synth.tensor_to_bits(Ad), ref, ms, np.arange(count))
    assert st == oracle.OK
    return gemm_tolerance_failures(Y[ms, ns], y, y64, mag).size


def test_stack_of_64_layers(w12lib, oracle):
    layers = []
    keep = {}
    bytes_w12 = 0
    weights = 0
    for layer in range(64):
        for i, (name, N, K) in enumerate(synth.LAYER_SHAPES):
            Wd = synth.dense_weights_device(N, K, seed=3000 * 1 + 16 * layer + i)
            t = w12lib.w12_encode(Wd)
            assert w12lib.w12_verify_roundtrip(Wd, t) == (w12lib.W12_OK, 0)  # load-time check
            if layer in (0, 63):
                keep[(layer, name)] = Wd.cpu()  # for the sampled oracle check
            del Wd
            layers.append((layer, name, t))
            bytes_w12 += t.nbytes()
            weights += N * K
    torch.cuda.empty_cache()
    assert 12.0 < 8 * bytes_w12 / weights < 12.1
    rng = np.random.default_rng(7)
    ws = w12lib.Workspace("cuda", 1 << 24)
    overlap = w12lib.make_opts(flags=w12lib.W12_GEMM_OVERLAP_PREVIOUS)
    for M in (1, 16):
        acts = {K: synth.activations_device(M, K, seed=M * 100 + K) for _, _, K in synth.LAYER_SHAPES}
        outs = {}
        for layer, name, t in layers:
            Y = w12lib.w12_gemm(acts[t.K], t, workspace=ws, opts=overlap)
            if layer in (0, 63):
                outs[(layer, name)] = Y
        torch.cuda.synchronize()
        for (layer, name), Y in outs.items():
            t = next(tt for l, n, tt in layers if l == layer and n == name)
            Wd = keep[(layer, name)].cuda()
            assert sampled_check(w12lib, oracle, Wd, t, acts[t.K], synth.tensor_to_bits(Y), rng) == 0


def test_escape_stress_full_size(w12lib, oracle):
    N, K = 5121, 17400
    W = synth.adversarial_weights(N, K, seed=4)
    Wd = synth.bits_to_tensor(W, "cuda")
    t = w12lib.w12_encode(Wd)
    assert w12lib.w12_verify_roundtrip(Wd, t) == (w12lib.W12_OK, 0)
    assert 0.01 < t.n_esc / (N * K) < 0.06  # 1-5% escapes
    rng = np.random.default_rng(8)
    # ten runs on ten grids (max_ctas 0 = the default grid), bitwise identical;
    # M = 33 takes the tensor-core path, M = 1 and 7 the small-M path
    caps = (0, 1, 7, 76, 152, 304, 3, 64, 760, 2)
    for M in (1, 7, 33):
        Ad = synth.bits_to_tensor(synth.activations(M, K, seed=400 + M), "cuda")
        outs = [synth.tensor_to_bits(w12lib.w12_gemm(Ad, t, opts=w12lib.make_opts(max_ctas=c))) for c in caps]
        for c, o in zip(caps[1:], outs[1:]):
            assert np.array_equal(o, outs[0]), (M, c)
        assert sampled_check(w12lib, oracle, Wd, t, Ad, outs[0], rng, count=48) == 0
