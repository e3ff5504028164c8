"""Two ranks on CPU (gloo): the N-sharded W12 GEMM and the benchmark's job timing.

The W12 GEMM shards along N with no exchange: rows [n0, n1) of a W12 tensor
(n0 a multiple of 16) are a W12 tensor of their own (SpecPilot, section 4.1:
the window, records and escape list are all per output channel; this
library groups them by 16-row stripe).  Each rank slices its rows with
W12Tensor.rows (host logic, here on CPU tensors), computes its block of Y
with the oracle, and an all-gather must give exactly the unsharded oracle
result.  The benchmark's whole-job time is the slowest rank's, and its
value counts the bytes of every rank.  The recurrent-layer outputs of draft
trees shard by request and by head, also with no exchange.
"""
import importlib.util
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def load_bench():
    spec = importlib.util.spec_from_file_location("bench_for_test", os.path.join(ROOT, "bench.py"))
    b = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(b)
    return b


def to_tensor(w12, ref):
    """An oracle-encoded tensor as a W12Tensor over CPU torch tensors."""
    return w12.W12Tensor(ref.N, ref.K, torch.from_numpy(ref.hi), torch.from_numpy(ref.lo),
                         torch.from_numpy(ref.base), torch.from_numpy(ref.esc_ptr),
                         torch.from_numpy(ref.esc.view(np.int32)[:ref.n_esc]), ref.n_esc)


def to_ref(oracle, t):
    return oracle.W12Ref(t.N, t.K, t.hi.numpy().copy(), t.lo.numpy().copy(), t.base.numpy().copy(),
                         t.esc_ptr.numpy().copy(), t.esc.numpy().view(np.uint32).copy(), t.n_esc)


def worker(rank, world, port, N, K, M, split, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import sys
        sys.path.insert(0, ROOT)
        sys.path.insert(0, HERE)
        import oracle
        import lossless_bit_weight_02_gb300 as w12
        from lossless_bit_weight_02_gb300 import synth

        W = synth.adversarial_weights(N, K, seed=77)  # every rank draws the same tensor
        A = synth.activations(M, K, seed=78)
        st, ref = oracle.encode(W)
        assert st == oracle.OK
        t = to_tensor(w12, ref)
        n0, n1 = (0, split) if rank == 0 else (split, N)
        part = t.rows(n0, n1)
        st, Y, _, _ = oracle.gemm(A, to_ref(oracle, part))
        assert st == oracle.OK and Y.shape == (M, n1 - n0)
        # gather the column blocks (padded to the largest)
        width = max(split, N - split)
        buf = torch.zeros(M, width, dtype=torch.int32)
        buf[:, :n1 - n0] = torch.from_numpy(Y.astype(np.int32))
        got = [torch.zeros_like(buf) for _ in range(world)]
        dist.all_gather(got, buf)
        full = torch.cat([got[0][:, :split], got[1][:, :N - split]], dim=1).numpy().astype(np.uint16)
        st, Yfull, _, _ = oracle.gemm(A, ref)
        same = bool(np.array_equal(full, Yfull))

        bench = load_bench()
        t_job = bench.job_time_ms(1.5 + rank, world, "cpu")
        v = bench.job_value(1e9, 10, world, t_job)
        q.put((rank, same, t_job, v))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("N,K,M,split", [(400, 700, 5, 208), (130, 257, 17, 64)])
def test_two_ranks_n_sharded_gemm_and_job_time(N, K, M, split, w12lib, oracle):
    ctx = mp.get_context("spawn")
    q = ctx.SimpleQueue()
    port = free_port()
    procs = [ctx.Process(target=worker, args=(r, 2, port, N, K, M, split, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
        assert p.exitcode == 0
    res = sorted(q.get() for _ in range(2))
    for rank, same, t_job, v in res:
        assert same, rank
        assert t_job == 2.5  # the slower rank's 2.5 ms on both
        assert v == pytest.approx(1e9 * 10 * 2 / 2.5e-3 / 1e9)


def gdn_worker(rank, world, port, q):
    """Each rank takes half of the requests of a shared-budget tree and half of
    the heads: its block of the recurrent-layer outputs, computed with the
    oracle on its own nodes and heads, must equal the same block of the
    unsharded result (requests and heads exchange nothing)."""
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import sys
        sys.path.insert(0, ROOT)
        from lossless_bit_weight_02_gb300 import synth
        from oracle import gdn

        n, H, D, R = 48, 4, 8, 4
        S0, qb, kb, vb, alpha, beta, parent, req = synth.gdn_inputs(n, H, D, seed=31, R=R)
        f = lambda b: (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32)  # noqa: E731
        qf, kf, vf = f(qb), f(kb), f(vb)

        def outputs(reqs, heads):
            o = np.zeros((n, len(heads), D))
            for r in reqs:
                idx = np.flatnonzero(req == r)
                remap = {int(j): x for x, j in enumerate(idx)}
                par = np.array([remap[int(parent[j])] if parent[j] >= 0 else -1 for j in idx], np.int64)
                o[idx] = gdn.path_outputs(S0[r][heads], qf[idx][:, heads], kf[idx][:, heads], vf[idx][:, heads],
                                          alpha[idx][:, heads], beta[idx][:, heads], par)
            return o

        mine_r = [r for r in range(R) if r % world == rank]
        mine_h = [h for h in range(H) if h % world == rank]
        block = torch.from_numpy(outputs(mine_r, mine_h))
        got = [torch.zeros_like(block) for _ in range(world)]
        dist.all_gather(got, block)
        full = outputs(range(R), list(range(H)))
        ok = True
        for src in range(world):
            rows = np.isin(req, [r for r in range(R) if r % world == src])
            heads = [h for h in range(H) if h % world == src]
            ok &= bool(np.array_equal(got[src].numpy()[rows], full[rows][:, heads]))
        q.put((rank, ok))
    finally:
        dist.destroy_process_group()


def test_two_ranks_gdn_tree_sharded_by_request_and_head():
    ctx = mp.get_context("spawn")
    q = ctx.SimpleQueue()
    port = free_port()
    procs = [ctx.Process(target=gdn_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
        assert p.exitcode == 0
    res = sorted(q.get() for _ in range(2))
    assert all(ok for _, ok in res), res
