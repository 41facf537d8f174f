"""Multi-rank paths on CPU ranks (gloo, world size 2), no GPU.

* Sequence split across ranks: each rank owns a contiguous piece of every
  head's sequence, forms its piece's state (sum phi(K) V^T, sum phi(K)) --
  the incremental update of "Transformers are RNNs" section 三 run over the
  piece from a zero state -- all-gathers the pieces' states, takes the
  exclusive prefix over ranks and recomputes its outputs from that carried-in
  state.  Concatenated, the ranks' outputs must equal the single-process
  causal forward, and the last rank's final state the full-sequence state.
  The arithmetic is the oracle's; what is tested is the exchange.
* Timing reduction: the bench reports the max over ranks of the timed region.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle

WORLD = 2


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _inputs(nh=3, N=40, D=4, M=3):
    rng = np.random.default_rng(7)
    return (rng.standard_normal((nh, N, D)), rng.standard_normal((nh, N, D)),
            rng.standard_normal((nh, N, M)))


def _worker(rank, port, result_dir):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=WORLD)
    try:
        Q, K, V = _inputs()
        nh, N, D = Q.shape
        M = V.shape[2]
        cuts = np.linspace(0, N, WORLD + 1).astype(int)  # uneven pieces are fine
        a, b = cuts[rank], cuts[rank + 1]
        q, k, v = Q[:, a:b], K[:, a:b], V[:, a:b]
        # 1. this piece's state from a zero state
        _, S_loc, Z_loc = oracle.causal_forward_recurrent(q, k, v)
        mine = torch.from_numpy(np.concatenate([S_loc.reshape(nh, -1), Z_loc], axis=1))
        # 2. exchange: every rank gets every piece's state
        gathered = [torch.empty_like(mine) for _ in range(WORLD)]
        dist.all_gather(gathered, mine)
        # 3. exclusive prefix over ranks (in rank order)
        prefix = torch.zeros_like(mine)
        for r in range(rank):
            prefix += gathered[r]
        S0 = prefix[:, :D * M].reshape(nh, D, M).numpy()
        Z0 = prefix[:, D * M:].numpy()
        O, S_end, Z_end = oracle.causal_forward_recurrent(q, k, v, S0, Z0)
        # 4. bench-style timing reduction: max over ranks
        t = torch.tensor([1.0 + rank])
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        np.savez(os.path.join(result_dir, f"rank{rank}.npz"), O=O, S=S_end, Z=Z_end,
                 tmax=t.numpy(), a=a, b=b)
    finally:
        dist.destroy_process_group()


def test_sequence_split_exchange_matches_single_process(tmp_path):
    port = _free_port()
    mp.spawn(_worker, args=(port, str(tmp_path)), nprocs=WORLD, join=True)
    Q, K, V = _inputs()
    O_ref, S_ref, Z_ref = oracle.causal_forward_recurrent(Q, K, V)
    parts = [np.load(tmp_path / f"rank{r}.npz") for r in range(WORLD)]
    O = np.concatenate([p["O"] for p in parts], axis=1)
    np.testing.assert_allclose(O, O_ref, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(parts[-1]["S"], S_ref, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(parts[-1]["Z"], Z_ref, rtol=1e-13)
    for p in parts:
        assert float(p["tmax"][0]) == float(WORLD)
    assert int(parts[0]["a"]) == 0 and int(parts[-1]["b"]) == Q.shape[1]
