"""The row-parallel (K-sharded) linear on two gloo ranks (CPU, no GPU): the
exchange step that a tensor-parallel row split of the rotated dimension
needs (sglang digest, "风险与影响": each rank's slice of the input features a
whole number of groups). Each rank holds its slice of X and of the prepared
weight, rotates its slice, takes its row maxima, all-reduces them with MAX,
quantizes with the combined maxima, multiplies its slice into int32 partial
sums, all-reduces those with SUM and reconstructs Y. Every step is the
oracle's; rank 0 compares with the oracle on the whole row: codes, scales,
accumulators and Y must be bit-identical."""
import os
import socket
import sys

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _case():
    rng = np.random.default_rng(2024)
    M, K, N, G = 24, 1024, 48, 256
    X = rng.standard_t(3, size=(M, K)) * np.where(rng.random(K) < 0.005, 50.0, 1.0)
    X = torch.from_numpy(X).to(torch.bfloat16).double().numpy()  # bf16 activations, as on the GPU
    W = rng.normal(0, 0.02, size=(N, K))
    b = rng.normal(0, 0.01, size=N)
    return X, W, b, G


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import oracle as O
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        X, W, b, G = _case()
        K = X.shape[1]
        w = K // world
        cols = slice(rank * w, (rank + 1) * w)
        Qw, sw, _ = O.prepare_weights(W, G, "h4")     # offline, on the whole K; each rank keeps its columns
        Xr = O.rotate_rows(X[:, cols], G, "h4")
        amax = torch.from_numpy(O.row_absmax(Xr))
        dist.all_reduce(amax, op=dist.ReduceOp.MAX)
        Q, sx, _, _ = O.quantize_rows_given(Xr, amax.numpy())
        A = torch.from_numpy(O.int_gemm(Q, Qw[:, cols]))
        dist.all_reduce(A, op=dist.ReduceOp.SUM)
        Y = O.reconstruct(A.numpy(), sx, sw, b)
        out[rank] = {"Q": Q, "sx": sx, "A": A.numpy(), "Y": Y}
    finally:
        dist.destroy_process_group()


def test_row_parallel_two_ranks_gloo_is_bit_identical():
    sys.path.insert(0, ROOT)
    import oracle as O
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        mp.start_processes(_worker, args=(2, _free_port(), out), nprocs=2, start_method="spawn")
        res = dict(out)
    X, W, b, G = _case()
    Qw, sw, _ = O.prepare_weights(W, G, "h4")
    whole = O.linear(X, Qw, sw, b, G, "h4")
    w = X.shape[1] // 2
    for rank in (0, 1):
        r = res[rank]
        assert np.array_equal(r["Q"], whole["Qx"][:, rank * w:(rank + 1) * w])
        assert np.array_equal(r["sx"], whole["sx"])
        assert np.array_equal(r["A"], whole["A"])
        assert np.array_equal(r["Y"], whole["Y64"])
