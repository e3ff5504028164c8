"""Seeded synthetic inputs for the W12 tests and benchmark.

This module only draws random numbers and casts them to BF16; it holds none of
the W12 arithmetic.  Both the CUDA path and the CPU oracle are fed from here.

The weight recipe stands in for the dense models of "SpecPilot" (arXiv
2611.02501), section 4.1, which are not available: Gaussian weights with a
log-normal scale per output channel (exponents concentrated inside a row,
which the W12 window relies on), plus exact zeros and large outliers that must
go through the escape list.  The adversarial recipe adds heavy tails, all-zero
rows, denormals and maximum-exponent values.

Host arrays are numpy uint16 holding BF16 bit patterns; device tensors are
torch.bfloat16.  The float -> BF16 cast is torch's round-to-nearest-even.
"""
from __future__ import annotations

import numpy as np
import torch

# 27B-class dense decoder layer: (name, N = output channels, K = input channels)
LAYER_SHAPES = (
    ("qkv", 7168, 5120),
    ("o", 5120, 5120),
    ("gate_up", 34816, 5120),
    ("down", 5120, 17408),
)


def _to_bf16_bits(x: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def bits_to_tensor(bits: np.ndarray, device="cpu") -> torch.Tensor:
    """uint16 BF16 bit array -> torch.bfloat16 tensor (bitwise)."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    return t.to(device)


def tensor_to_bits(t: torch.Tensor) -> np.ndarray:
    """torch.bfloat16 tensor -> uint16 numpy array (bitwise)."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16).copy()


def dense_weights(N: int, K: int, seed: int, zero_frac=1e-3, outlier_frac=5e-4) -> np.ndarray:
    """W = N(0,1) * 0.02 * s_n with s_n ~ LogNormal(0, 0.5) per row; a fraction
    `zero_frac` of positions set to exactly 0 and a further `outlier_frac`
    multiplied by 2^9.  Returns BF16 bits [N,K]."""
    rng = np.random.default_rng(seed)
    s = np.exp(rng.normal(0.0, 0.5, size=N))
    w = rng.normal(0.0, 1.0, size=(N, K)) * 0.02 * s[:, None]
    total = N * K
    nz = int(round(zero_frac * total))
    no = int(round(outlier_frac * total))
    pos = rng.choice(total, size=nz + no, replace=False) if nz + no else np.zeros(0, np.int64)
    flat = w.reshape(-1)
    flat[pos[:nz]] = 0.0
    flat[pos[nz:]] *= 2.0 ** 9
    return _to_bf16_bits(w)


def dense_weights_device(N: int, K: int, seed: int, device="cuda", zero_frac=1e-3,
                         outlier_frac=5e-4) -> torch.Tensor:
    """The dense_weights recipe drawn with torch's generator on `device`
    (for full-size layers).  Returns torch.bfloat16 [N,K]."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    s = torch.exp(torch.randn(N, 1, device=device, generator=g) * 0.5)
    w = torch.randn(N, K, device=device, generator=g).mul_(0.02).mul_(s)
    total = N * K
    nz = int(round(zero_frac * total))
    no = int(round(outlier_frac * total))
    flat = w.view(-1)
    if nz + no:
        pos = torch.randperm(total, device=device, generator=g)[: nz + no]
        flat[pos[:nz]] = 0.0
        flat[pos[nz:]] *= 2.0 ** 9
        del pos
    out = w.to(torch.bfloat16)
    del w
    return out


def random_bits_device(N: int, K: int, seed: int, device="cuda") -> torch.Tensor:
    """Uniformly random 16-bit patterns as torch.bfloat16 [N,K] on `device`
    (every exponent equally likely: about 15 in 16 weights fall outside any
    16-exponent window; zeros, subnormals, infinities and NaNs included)."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return torch.randint(-32768, 32768, (N, K), dtype=torch.int16, device=device, generator=g).view(torch.bfloat16)


def activations(M: int, K: int, seed: int) -> np.ndarray:
    """BF16 activations [M,K] ~ N(0,1).  Returns BF16 bits."""
    rng = np.random.default_rng(seed)
    return _to_bf16_bits(rng.normal(0.0, 1.0, size=(M, K)))


def activations_device(M: int, K: int, seed: int, device="cuda") -> torch.Tensor:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return torch.randn(M, K, device=device, generator=g).to(torch.bfloat16)


def adversarial_weights(N: int, K: int, seed: int) -> np.ndarray:
    """Escape stress: Student-t(3) * 0.02; a random 2% of entries scaled by
    2^(+-20); every 64th row all zero; 0.1% random BF16 denormals; 1% of the
    rows (every 100th, offset 7) carry +-max-exponent values (exponent field
    254) at 1% of their positions.  Returns BF16 bits [N,K]."""
    rng = np.random.default_rng(seed)
    w = rng.standard_t(3.0, size=(N, K)) * 0.02
    total = N * K
    flat = w.reshape(-1)
    big = rng.choice(total, size=int(0.02 * total), replace=False)
    flat[big] *= 2.0 ** (20.0 * rng.choice([-1.0, 1.0], size=big.size))
    bits = _to_bf16_bits(w)
    fb = bits.reshape(-1)
    den = rng.choice(total, size=max(1, int(1e-3 * total)), replace=False)
    fb[den] = (rng.integers(0, 2, den.size) << 15 | rng.integers(1, 128, den.size)).astype(np.uint16)
    for n in range(7, N, 100):
        cols = rng.choice(K, size=max(1, K // 100), replace=False)
        sign = rng.integers(0, 2, cols.size) << 15
        man = rng.integers(0, 128, cols.size)
        bits[n, cols] = (sign | (254 << 7) | man).astype(np.uint16)
    bits[::64, :] = 0
    return bits


def all_patterns(rows: int, seed: int) -> np.ndarray:
    """Every one of the 65536 BF16 bit patterns exactly once, in a seeded random
    order, shaped [rows, 65536/rows]."""
    assert 65536 % rows == 0
    rng = np.random.default_rng(seed)
    return rng.permutation(65536).astype(np.uint16).reshape(rows, 65536 // rows)


# Gated-delta-rule tree inputs (recurrent layers of a hybrid model, tree
# verification).  A GDN layer of a 27B-class hybrid target: 32 heads of
# dimension 128 with unit-length queries and keys, decay near 1, write
# strengths spread over (0, 1), and a root state of a few tenths per entry.
GDN_HEADS, GDN_DIM = 32, 128


def random_tree(n: int, seed: int, max_depth: int = 16, new_root: float = 0.15) -> np.ndarray:
    """parent[i] in [-1, i): each node hangs off a random earlier node whose
    depth is below max_depth, or off the root with probability new_root."""
    rng = np.random.default_rng(seed)
    parent = np.full(n, -1, np.int32)
    depth = np.zeros(n, np.int64)
    for i in range(n):
        if i > 0 and rng.random() >= new_root:
            cand = np.flatnonzero(depth[:i] < max_depth)
            if len(cand):
                parent[i] = int(rng.choice(cand))
        depth[i] = 1 if parent[i] < 0 else depth[parent[i]] + 1
    return parent


def gdn_inputs(n: int, H: int, D: int, seed: int, R: int = 1, parent=None, req=None):
    """Host arrays: S0 float32 [R,H,D,D]; q, k, v BF16 bits [n,H,D] (q and k
    of unit length before the cast); alpha, beta float32 [n,H]; parent int32
    [n]; req int32 [n] (a root child draws its request, children inherit)."""
    rng = np.random.default_rng(seed)
    S0 = (rng.standard_normal((R, H, D, D)) * 0.3).astype(np.float32)
    q = rng.standard_normal((n, H, D))
    k = rng.standard_normal((n, H, D))
    q /= np.linalg.norm(q, axis=-1, keepdims=True)
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((n, H, D))
    alpha = rng.uniform(0.85, 1.0, size=(n, H)).astype(np.float32)
    beta = rng.uniform(0.1, 0.9, size=(n, H)).astype(np.float32)
    if parent is None:
        parent = random_tree(n, seed + 1)
    parent = np.asarray(parent, np.int32)
    if req is None:
        req = np.zeros(n, np.int32)
        for i in range(n):
            req[i] = rng.integers(R) if parent[i] < 0 else req[parent[i]]
    return (S0, _to_bf16_bits(q), _to_bf16_bits(k), _to_bf16_bits(v), alpha, beta, parent,
            np.asarray(req, np.int32))
