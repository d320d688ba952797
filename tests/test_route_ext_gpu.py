"""GPU parity of the QB comparator and of token-sharded QB (through the C ABI).

* moe_route_signsgd: DeepSeek-V3's fixed-step sign rule on the bias (the
  Kimi K3 width page's extended reading on QB vs DeepSeek-V3), bit-exact
  against the oracle's route_signsgd: scores, biases, indices, weights, loads.
* Token-sharded QB: shards of one batch on one device that exchange only
  per-expert digit histograms reach, bit for bit, the bias of the whole
  batch's sweep (moe_route_qb and the oracle), and routing each shard with
  that bias reproduces the whole batch's routing.
"""
import numpy as np
import pytest

import qb_inputs as QI
from oracle import qb_oracle as O

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

F32 = np.float32


def _logits(T, n, seed, offset_var=1.0, ties=False):
    z = QI.normal_f32(seed, QI.TID["logit_noise"], (T, n), 1.0)
    o = QI.normal_f32(seed, QI.TID["router_offset"], (n,), float(np.sqrt(offset_var)))
    lg = (z + o[None, :]).astype(F32)
    if ties:
        lg = (np.round(lg * 4) / 4).astype(F32)
    return lg


def _eq(name, got, want):
    got = np.asarray(got)
    want = np.asarray(want).astype(got.dtype)
    assert got.shape == want.shape, name
    eq = got.view(np.uint32) == want.view(np.uint32) if got.dtype.kind == "f" else got == want
    assert eq.all(), f"{name}: {int((~eq).sum())} mismatches"


SIGN_CASES = [
    # T, n, k, steps, gamma, offset_var, bias_scale
    (4096, 896, 16, 1, 1e-3, 1.0, 0.0),
    (4096, 896, 16, 8, 1e-3, 1.0, 0.0),
    (257, 100, 7, 3, 0.05, 2.0, 0.1),
    (64, 32, 4, 0, 0.01, 0.5, 0.2),
    (1, 8, 3, 2, 0.25, 1.0, 0.0),
    (700, 96, 5, 4, 1.0 / 64, 1.0, 0.0),
]


@pytest.mark.parametrize("T,n,k,steps,gamma,ov,bs", SIGN_CASES)
def test_signsgd_bit_exact(T, n, k, steps, gamma, ov, bs):
    import quantile_balanced_routing_gb300 as Q
    logits = _logits(T, n, seed=T + 3 * n, offset_var=ov)
    b0 = None if bs == 0 else QI.normal_f32(T + n, 77, (n,), bs)
    dev = torch.device("cuda:0")
    g = Q.route_signsgd(torch.from_numpy(logits).to(dev), k, steps, gamma,
                        bias_in=None if b0 is None else torch.from_numpy(b0).to(dev))
    torch.cuda.synchronize()
    o = O.route_signsgd(logits, b0, k, steps, gamma)
    for name, a, b in zip(("scores", "bias", "idx", "w", "loads"), g, o):
        _eq(name, a.cpu().numpy(), b)


def _sharded(logits, k, split, bias_in=None):
    from quantile_balanced_routing_gb300 import sharded as S
    dev = torch.device("cuda:0")
    bounds = np.cumsum([0] + list(split))
    shards = [torch.from_numpy(np.ascontiguousarray(logits[a:b])).to(dev) for a, b in zip(bounds[:-1], bounds[1:])]
    ds = S.DeviceShards(shards, k, logits.shape[0],
                        bias_in=None if bias_in is None else torch.from_numpy(bias_in).to(dev))
    bias = S.qb_bias_sharded(ds)
    torch.cuda.synchronize()
    return ds, bias, shards


SHARD_CASES = [
    # T, n, k, split, offset_var, bias_scale, ties
    (4096, 896, 16, [2048, 2048], 1.0, 0.0, False),
    (4096, 896, 16, [1000, 96, 3000], 2.0, 0.0, False),
    (777, 100, 7, [1, 776], 1.0, 0.1, False),
    (700, 96, 5, [350, 350], 1.0, 0.0, True),
    (5, 7, 3, [2, 3], 1.0, 0.2, False),          # r_j >= T and r_j = 0 targets
]


@pytest.mark.parametrize("T,n,k,split,ov,bs,ties", SHARD_CASES)
def test_sharded_qb_reproduces_the_whole_batch(T, n, k, split, ov, bs, ties):
    import quantile_balanced_routing_gb300 as Q
    logits = _logits(T, n, seed=5 * T + n, offset_var=ov, ties=ties)
    b0 = None if bs == 0 else QI.normal_f32(T * 3 + n, 77, (n,), bs)
    ds, bias, shards = _sharded(logits, k, split, b0)
    o = O.moe_route_qb(logits, b0, k, qb_sweeps=1)
    _eq("bias vs oracle", bias.cpu().numpy(), o[1])
    dev = torch.device("cuda:0")
    whole = Q.route_qb(torch.from_numpy(logits).to(dev), k, qb_sweeps=1,
                       bias_in=None if b0 is None else torch.from_numpy(b0).to(dev))
    _eq("bias vs moe_route_qb", bias.cpu().numpy(), whole[1].cpu().numpy())
    # each shard routes its own tokens with the exchanged bias
    rows = np.cumsum([0] + list(split))
    loads = np.zeros(n, np.int64)
    for i, x in enumerate(shards):
        s, _, idx, w, ld = Q.route_qb(x, k, qb_sweeps=0, bias_in=bias)
        torch.cuda.synchronize()
        a, b = rows[i], rows[i + 1]
        _eq("scores", s.cpu().numpy(), o[0][a:b])
        _eq("shard margins-pass scores", ds.scores[i].cpu().numpy(), o[0][a:b])
        _eq("idx", idx.cpu().numpy(), o[2][a:b])
        _eq("w", w.cpu().numpy(), o[3][a:b])
        loads += ld.cpu().numpy()
    _eq("loads", loads.astype(np.int32), o[4])


def test_sharded_exchange_volume_is_histograms_not_margins():
    from quantile_balanced_routing_gb300 import sharded as S
    import quantile_balanced_routing_gb300 as Q
    lib = Q.load_library()
    n, T = 896, 16384
    per_pass = lib.qbmoe_qb_hist_bytes(n)
    assert per_pass == n * 2 * S.HIST_BINS * 4          # independent of the tokens
    assert S.HIST_PASSES * per_pass <= T * n * 4 / 8    # all passes: an eighth of the margins at 16384 tokens
