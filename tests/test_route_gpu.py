"""GPU parity of moe_route_qb (through the C ABI) against the CPU oracle.

Routing is an integer result decided by fp32 arithmetic that both sides
perform in the same precision and order, so every output must match bit for
bit: scores, QB biases, top-k indices (rank order), weights and loads.
"""
import numpy as np
import pytest

import qb_inputs as QI
from oracle import qb_oracle as O

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

F32 = np.float32


def _logits(T, n, seed, offset_var=1.0, kind="normal"):
    z = QI.normal_f32(seed, QI.TID["logit_noise"], (T, n), 1.0)
    o = QI.normal_f32(seed, QI.TID["router_offset"], (n,), float(np.sqrt(offset_var)))
    lg = (z + o[None, :]).astype(F32)
    if kind == "ties":            # quantised logits: many exact ties in scores and margins
        lg = (np.round(lg * 4) / 4).astype(F32)
    elif kind == "all_equal":
        lg = np.zeros((T, n), F32)
    return lg


def _bias(n, seed, scale):
    if scale == 0:
        return None
    return QI.normal_f32(seed, 77, (n,), scale)


def run_gpu(logits, k, sweeps, bias_in):
    import quantile_balanced_routing_gb300 as Q
    dev = torch.device("cuda:0")
    lg = torch.from_numpy(logits).to(dev)
    b = None if bias_in is None else torch.from_numpy(bias_in).to(dev)
    s, bo, idx, w, loads = Q.route_qb(lg, k, qb_sweeps=sweeps, bias_in=b)
    torch.cuda.synchronize()
    return s.cpu().numpy(), bo.cpu().numpy(), idx.cpu().numpy(), w.cpu().numpy(), loads.cpu().numpy()


def assert_bit_equal(name, got, want):
    got = np.asarray(got)
    want = np.asarray(want)
    assert got.shape == want.shape, name
    if got.dtype.kind == "f":
        eq = got.view(np.uint32) == want.astype(got.dtype).view(np.uint32)
    else:
        eq = got == want.astype(got.dtype)
    if not eq.all():
        bad = np.argwhere(~eq)[:5]
        raise AssertionError(f"{name}: {int((~eq).sum())} mismatches, first at {bad.tolist()}: "
                             f"gpu {got[tuple(bad[0])]!r} oracle {want[tuple(bad[0])]!r}")


CASES = [
    # T, n, k, sweeps, offset_var, bias_scale, kind
    (64, 32, 4, 1, 0.5, 0.0, "normal"),          # tiny workload's routing
    (4096, 896, 16, 1, 1.0, 0.0, "normal"),      # QB routing workload, full size
    (257, 100, 7, 1, 1.0, 0.0, "normal"),        # ragged T, n not a multiple of 32
    (1, 8, 3, 1, 1.0, 0.0, "normal"),            # one token (targets hit r >= T)
    (33, 2, 1, 1, 1.0, 0.0, "normal"),           # two experts
    (500, 64, 1, 2, 2.0, 0.0, "normal"),         # top-1, two sweeps
    (300, 896, 16, 0, 1.0, 0.1, "normal"),       # frozen bias (inference)
    (1000, 1024, 32, 1, 1.0, 0.05, "normal"),    # largest n and k, nonzero bias in
    (700, 96, 5, 1, 1.0, 0.0, "ties"),           # tie-heavy scores
    (129, 40, 6, 1, 1.0, 0.0, "all_equal"),      # every score equal
    (5, 7, 3, 3, 1.0, 0.2, "normal"),            # more sweeps than tokens
]


@pytest.mark.parametrize("T,n,k,sweeps,ov,bs,kind", CASES)
def test_route_bit_exact(T, n, k, sweeps, ov, bs, kind):
    logits = _logits(T, n, seed=T * 7 + n, offset_var=ov, kind=kind)
    bias_in = _bias(n, T + n, bs)
    g = run_gpu(logits, k, sweeps, bias_in)
    o = O.moe_route_qb(logits, bias_in, k, qb_sweeps=sweeps)
    for name, a, b in zip(("scores", "bias", "idx", "w", "loads"), g, o):
        assert_bit_equal(name, a, b)


def test_route_qb_workload_from_router_logits():
    """The QB routing workload as specified: logits = x W_r^T + o at d = 7168."""
    wl = QI.ROUTE_QB
    inp = QI.LayerInputs(wl)
    logits = O.router_logits(inp.values("x"), inp.values("w_router"), inp.values("router_offset"))
    g = run_gpu(logits, wl.k, 1, None)
    o = O.moe_route_qb(logits, None, wl.k, qb_sweeps=1)
    for name, a, b in zip(("scores", "bias", "idx", "w", "loads"), g, o):
        assert_bit_equal(name, a, b)
    # QB moved the loads towards T*k/n (reported balance, not a bit pin)
    _, _, l0 = O.route_topk(o[0], np.zeros(wl.n, F32), wl.k)
    assert g[4].max() < l0.max()


@pytest.mark.slow
def test_route_prefill_size():
    T, n, k = 16384, 896, 16
    logits = _logits(T, n, seed=3, offset_var=2.0)
    g = run_gpu(logits, k, 1, None)
    o = O.moe_route_qb(logits, None, k, qb_sweeps=1)
    for name, a, b in zip(("scores", "bias", "idx", "w", "loads"), g, o):
        assert_bit_equal(name, a, b)


def test_route_repeatable_and_stream_ordered():
    logits = _logits(512, 128, seed=11)
    a = run_gpu(logits, 8, 1, None)
    b = run_gpu(logits, 8, 1, None)
    for x, y in zip(a, b):
        assert np.array_equal(np.asarray(x).view(np.uint8), np.asarray(y).view(np.uint8))


def test_bias_out_may_alias_bias_in():
    import quantile_balanced_routing_gb300 as Q
    logits = _logits(200, 64, seed=5)
    b0 = _bias(64, 9, 0.1)
    dev = torch.device("cuda:0")
    bt = torch.from_numpy(b0.copy()).to(dev)
    lg = torch.from_numpy(logits).to(dev)
    Q.route_qb(lg, 4, qb_sweeps=1, bias_in=bt, bias_out=bt)
    torch.cuda.synchronize()
    want = O.moe_route_qb(logits, b0, 4, qb_sweeps=1)[1]
    assert_bit_equal("bias", bt.cpu().numpy(), want)
