"""GPU cyclic coordinate-descent QB (moe_route_qb_gs) against the oracle's
Gauss-Seidel sweep: biases, routing, weights and loads bit-exact; the
"until balanced" mode stops after the same sweep as the oracle."""
import numpy as np
import pytest

import qb_inputs as QI
from oracle import qb_oracle as O

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
F32 = np.float32


def _logits(T, n, seed, ov=1.0, ties=False):
    z = QI.normal_f32(seed, QI.TID["logit_noise"], (T, n), 1.0)
    o = QI.normal_f32(seed, QI.TID["router_offset"], (n,), float(np.sqrt(ov)))
    lg = (z + o[None, :]).astype(F32)
    if ties:
        lg = (np.round(lg * 4) / 4).astype(F32)
    return lg


def _gpu(logits, k, sweeps, stop, bias_in=None):
    import quantile_balanced_routing_gb300 as Q
    lg = torch.from_numpy(logits).cuda()
    b = None if bias_in is None else torch.from_numpy(bias_in).cuda()
    out = Q.route_qb_gs(lg, k, max_sweeps=sweeps, stop_when_balanced=stop, bias_in=b)
    torch.cuda.synchronize()
    return [t.cpu().numpy() for t in out]


def _same(a, b):
    a, b = np.asarray(a), np.asarray(b)
    if a.dtype.kind == "f":
        return np.array_equal(a.view(np.uint32), b.astype(a.dtype).view(np.uint32))
    return np.array_equal(a, b.astype(a.dtype))


@pytest.mark.parametrize("T,n,k,sweeps,ov,ties", [
    (300, 24, 3, 1, 1.5, False),
    (300, 24, 3, 3, 1.5, False),
    (1000, 128, 8, 1, 2.0, False),
    (257, 100, 7, 2, 1.0, False),
    (400, 40, 5, 2, 1.0, True),
    (64, 32, 31, 1, 1.0, False),
])
def test_gauss_seidel_bit_exact(T, n, k, sweeps, ov, ties):
    logits = _logits(T, n, seed=T + n + k, ov=ov, ties=ties)
    g = _gpu(logits, k, sweeps, False)
    o = O.moe_route_qb(logits, None, k, qb_sweeps=sweeps, mode="gauss_seidel")
    for name, a, b in zip(("scores", "bias", "idx", "w", "loads"), g[:5], o):
        assert _same(a, b), name
    assert int(g[5][0]) == sweeps


def test_gauss_seidel_until_balanced():
    T, n, k = 200, 16, 2
    logits = _logits(T, n, seed=5, ov=2.0)
    g = _gpu(logits, k, 60, True)
    done = int(g[5][0])
    r = O.qb_targets(T, n, k)
    assert 1 <= done < 60
    assert np.array_equal(g[4], r)                 # balanced: every load on target
    s = O.sigmoid_score(logits)
    b = np.zeros(n, F32)
    for i in range(done):
        b = O.qb_sweep_gauss_seidel(s, b, k)
        loads = O.route_topk(s, b, k)[2]
        if i < done - 1:
            assert not np.array_equal(loads, r)   # the oracle is not balanced earlier
    assert _same(g[1], b)
    assert np.array_equal(loads, r)


def test_zero_sweeps_is_the_frozen_router():
    logits = _logits(100, 20, seed=9)
    b = QI.normal_f32(3, 77, (20,), 0.1)
    g = _gpu(logits, 4, 0, False, bias_in=b)
    o = O.moe_route_qb(logits, b, 4, qb_sweeps=0)
    for name, a, bb in zip(("scores", "bias", "idx", "w", "loads"), g[:5], o):
        assert _same(a, bb), name


def test_repeated_calls_on_the_same_buffers():
    """Calls that reuse one set of buffers route the logits the buffers hold
    at each call, bit-exact like a fresh call."""
    import quantile_balanced_routing_gb300 as Q
    T, n, k, sweeps = 300, 24, 3, 2
    lib = Q.load_library()
    dev = torch.device("cuda", 0)
    lg = torch.empty((T, n), dtype=torch.float32, device=dev)
    outs = dict(scores=torch.empty((T, n), dtype=torch.float32, device=dev),
                bias=torch.empty((n,), dtype=torch.float32, device=dev),
                idx=torch.empty((T, k), dtype=torch.int32, device=dev),
                w=torch.empty((T, k), dtype=torch.float32, device=dev),
                loads=torch.empty((n,), dtype=torch.int32, device=dev))
    done = torch.zeros((4,), dtype=torch.int32, device=dev)
    ws = torch.empty((lib.qbmoe_route_gs_workspace_bytes(T, n, k),), dtype=torch.uint8, device=dev)
    p = lambda t: t.data_ptr()
    for seed in (11, 12, 13):
        logits = _logits(T, n, seed=seed, ov=1.5)
        lg.copy_(torch.from_numpy(logits))
        rc = lib.moe_route_qb_gs(T, n, k, sweeps, 0, p(lg), None, p(outs["bias"]), p(outs["scores"]), p(outs["idx"]),
                                 p(outs["w"]), p(outs["loads"]), p(done), p(ws), ws.numel(), None)
        assert rc == 0
        torch.cuda.synchronize()
        o = O.moe_route_qb(logits, None, k, qb_sweeps=sweeps, mode="gauss_seidel")
        for name, b in zip(("scores", "bias", "idx", "w", "loads"), o):
            assert _same(outs[name].cpu().numpy(), b), (seed, name)
