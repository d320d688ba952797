"""The token-sharded QB exchange across processes, on CPU: two gloo ranks,
each holding half of a batch's tokens, run the package's exchange order
(qb_bias_sharded) with torch.distributed's all-reduce summing the digit
histograms.  The per-shard steps are the oracle's (the CUDA kernels need a
GPU; their parity is tests/test_route_ext_gpu.py), so this checks the
exchange itself: both ranks end with the bias of the whole batch's sweep."""
import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")

F32 = np.float32


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


class OracleShard:
    """The per-shard steps of the exchange computed by the CPU oracle, with
    the same interface as quantile_balanced_routing_gb300.sharded.DeviceShards."""

    def __init__(self, s_shard, T_total, k, b0):
        from oracle import qb_oracle as O
        self.O = O
        self.s = s_shard
        self.T = T_total
        self.k = k
        self.b0 = b0
        n = s_shard.shape[1]
        self.hist = torch.zeros((n, 2, 256), dtype=torch.int64)

    def start(self):
        O = self.O
        n = self.s.shape[1]
        self.r = O.qb_targets(self.T, n, self.k)
        self.rank = O.selection_ranks(self.T, self.r)
        self.prefix = np.zeros((n, 2), np.uint32)
        self.keys = O.descending_keys(O.qb_margins(self.s, self.b0, self.k)).T.copy()
        self.hist.zero_()

    def count(self, p):
        self.hist += torch.from_numpy(self.O.shard_digit_histogram(self.keys, self.prefix, p))

    def advance(self, p):
        self.prefix, self.rank = self.O.advance_selection(self.hist.numpy(), self.prefix, self.rank, p)
        self.hist.zero_()

    def bias(self):
        O = self.O
        Ma, Mb = O.margin_of_key(self.prefix[:, 0]), O.margin_of_key(self.prefix[:, 1])
        q = np.where(self.r <= 0, Ma + F32(1), np.where(self.r >= self.T, Ma - F32(1), (Ma + Mb) * F32(0.5)))
        return O.common_offset((-q).astype(F32))


def _problem():
    from oracle import qb_oracle as O
    rng = np.random.default_rng(21)
    T, n, k = 300, 24, 3
    logits = (rng.normal(0, 1, (T, n)) + rng.normal(0, 1.5, n)[None, :]).astype(F32)
    s = O.sigmoid_score(logits)
    b0 = rng.normal(0, 0.02, n).astype(F32)
    return s, b0, k


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from quantile_balanced_routing_gb300.sharded import qb_bias_sharded
    s, b0, k = _problem()
    cut = [0, 113, s.shape[0]]            # uneven shards
    shard = OracleShard(s[cut[rank]:cut[rank + 1]], s.shape[0], k, b0)
    bias = qb_bias_sharded(shard, allreduce=lambda t: dist.all_reduce(t, op=dist.ReduceOp.SUM))
    out[rank] = bias.tobytes()
    dist.destroy_process_group()


def test_two_gloo_ranks_reach_the_whole_batch_bias():
    import torch.multiprocessing as mp
    from oracle import qb_oracle as O
    world, port = 2, _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
    s, b0, k = _problem()
    want = O.qb_sweep_jacobi(s, b0, k)
    for r in range(world):
        assert np.frombuffer(out[r], F32).tobytes() == want.tobytes()


def test_one_process_without_allreduce_matches_too():
    from oracle import qb_oracle as O
    from quantile_balanced_routing_gb300.sharded import qb_bias_sharded
    s, b0, k = _problem()
    b = qb_bias_sharded(OracleShard(s, s.shape[0], k, b0))
    assert b.tobytes() == O.qb_sweep_jacobi(s, b0, k).tobytes()
