"""Token-sharded Quantile Balancing: the order of the histogram exchange.

A batch is split into token shards, on one device or on several (one
process per device).  The bias of a QB sweep needs, per expert, the r-th
and (r+1)-th largest margin over the whole batch; the shards never exchange
margins, only per-expert digit histograms (n x 2 x 256 counts per pass, four
passes), which the library's kernels refine to the exact order statistics.
This module only sequences the library calls and the caller's all-reduce;
every step of the arithmetic runs in the CUDA kernels of libqbmoe.
"""
from __future__ import annotations

from . import QbmoeError, _p, _stream_ptr, load_library

HIST_PASSES = 4
HIST_BINS = 256


class DeviceShards:
    """This device's token shards of one batch (fp32 logits [T_s, n] each).

    ``hist`` is the int32 [n, 2, 256] histogram buffer the exchange sums
    across devices; ``scores[i]`` receives shard i's router scores."""

    def __init__(self, logits_shards, k: int, T_total: int, bias_in=None, stream=None):
        import torch
        self.lib = load_library()
        self.shards = list(logits_shards)
        self.k = k
        self.T_total = T_total
        self.n = self.shards[0].shape[1]
        self.dev = self.shards[0].device
        self.bias_in = bias_in
        self.stream = _stream_ptr(stream)
        for x in self.shards:
            assert x.dtype == torch.float32 and x.is_contiguous() and x.shape[1] == self.n
        n = self.n
        self.state = torch.empty((self.lib.qbmoe_qb_hist_state_bytes(n),), dtype=torch.uint8, device=self.dev)
        self.hist = torch.empty((n, 2, HIST_BINS), dtype=torch.int32, device=self.dev)
        self.scores = [torch.empty_like(x) for x in self.shards]
        self.ws = [torch.empty((self.lib.qbmoe_qb_shard_workspace_bytes(x.shape[0], n, k),), dtype=torch.uint8,
                               device=self.dev) for x in self.shards]

    def _ok(self, rc, what):
        if rc:
            raise QbmoeError(rc, what)

    def start(self):
        """Targets of the whole batch, a zeroed histogram, and every local
        shard's margins under the starting bias."""
        self._ok(self.lib.moe_qb_hist_init(self.T_total, self.n, self.k, _p(self.state), _p(self.hist),
                                           self.stream), "moe_qb_hist_init")
        for x, sc, ws in zip(self.shards, self.scores, self.ws):
            self._ok(self.lib.moe_qb_shard_margins(x.shape[0], self.n, self.k, _p(x), _p(self.bias_in), _p(sc),
                                                   _p(ws), ws.numel(), self.stream), "moe_qb_shard_margins")

    def count(self, p: int):
        """Add every local shard's digit histogram of pass p into hist."""
        for x, ws in zip(self.shards, self.ws):
            self._ok(self.lib.moe_qb_shard_hist(x.shape[0], self.n, p, _p(self.state), _p(ws), _p(self.hist),
                                                self.stream), "moe_qb_shard_hist")

    def advance(self, p: int):
        """Fix pass p's digits from the summed histogram (and zero it)."""
        self._ok(self.lib.moe_qb_hist_advance(self.n, p, _p(self.hist), _p(self.state), self.stream),
                 "moe_qb_hist_advance")

    def bias(self):
        import torch
        b = torch.empty((self.n,), dtype=torch.float32, device=self.dev)
        self._ok(self.lib.moe_qb_hist_bias(self.n, _p(self.state), _p(b), self.stream), "moe_qb_hist_bias")
        return b


def qb_bias_sharded(shards, allreduce=None):
    """One QB sweep's bias over every shard of the batch.

    shards: this process's shards (DeviceShards, or any object with the same
    start/count/advance/bias methods and a ``hist`` buffer).  allreduce: sums
    ``hist`` in place over the processes holding the other shards (e.g.
    ``torch.distributed.all_reduce``); None when every shard is local."""
    shards.start()
    for p in range(HIST_PASSES):
        shards.count(p)
        if allreduce is not None:
            allreduce(shards.hist)
        shards.advance(p)
    return shards.bias()
