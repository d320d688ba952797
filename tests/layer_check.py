"""Shared checks of the GPU layer against the CPU oracle (used by the GPU tests)."""
from __future__ import annotations

import numpy as np

import qb_inputs as QI
from oracle import qb_oracle as O

F32 = np.float32
TOL = {"f32": 1e-3, "bf16": 2e-2, "mxfp4": 6e-2}


def row_rel_err(got: np.ndarray, want: np.ndarray) -> np.ndarray:
    """Per token row: max_c |got - want| / max_c |want|."""
    num = np.max(np.abs(got.astype(np.float64) - want), axis=1)
    den = np.maximum(np.max(np.abs(want), axis=1), 1e-30)
    return num / den


def tol_of(shape) -> float:
    return TOL["mxfp4"] if shape.wfmt == "mxfp4" else TOL[shape.dtype]


def to_f64(t) -> np.ndarray:
    import torch
    t = t.detach()
    if t.dtype == torch.bfloat16:
        return t.float().cpu().numpy().astype(np.float64)
    return t.cpu().numpy().astype(np.float64)


def bits_equal(a, b) -> np.ndarray:
    a = np.asarray(a)
    b = np.asarray(b).astype(a.dtype)
    if a.dtype.kind == "f":
        return a.view(np.uint32) == b.view(np.uint32)
    return a == b


def check_routing_self_consistent(s, b, idx, w, loads, k):
    """Properties the GPU's own routing must satisfy whatever its scores:
    idx = top-k of fl(s + b) with lower index first on ties, in rank order;
    w = s_idx renormalised (within 2 ulp); loads = route counts."""
    s = np.asarray(s, F32)
    v = (s + np.asarray(b, F32)[None, :]).astype(F32)
    T, n = s.shape
    rows = np.arange(T)[:, None]
    sel_v = v[rows, idx]
    # rank order: non-increasing values, ties by increasing index
    dv = np.diff(sel_v, axis=1)
    assert np.all(dv <= 0)
    assert np.all((dv < 0) | (np.diff(idx, axis=1) > 0))
    # every unchosen expert ranks after the k-th chosen one
    chosen = np.zeros((T, n), bool)
    chosen[rows, idx] = True
    kth_v = sel_v[:, -1][:, None]
    kth_j = idx[:, -1][:, None]
    j = np.arange(n)[None, :]
    after = (v < kth_v) | ((v == kth_v) & (j > kth_j))
    assert np.all(after | chosen)
    sel_s = s[rows, idx].astype(np.float64)
    assert np.allclose(w, sel_s / sel_s.sum(axis=1, keepdims=True), rtol=(k + 2) * 1.2e-7, atol=0)
    assert np.array_equal(np.bincount(idx.ravel(), minlength=n), loads)


def upload_and_run(shape, logits_in=None, layer=None, dev_inputs=None):
    import torch
    from qb_inputs.device import layer_for, upload
    inp = QI.LayerInputs(shape)
    d = dev_inputs or upload(inp, "cuda:0", drop_host=False)
    lay = layer or layer_for(shape)
    w = {kk: vv for kk, vv in d.items() if kk != "x"}
    lay.set_weights(**w)
    lg = None if logits_in is None else torch.from_numpy(np.ascontiguousarray(logits_in, F32)).to("cuda:0")
    out, r = lay.forward(d["x"], logits_in=lg, want_routing=True)
    rc = lay.status()
    assert rc == 0, rc
    torch.cuda.synchronize()
    res = dict(out=to_f64(out), scores=r["scores"].cpu().numpy(), bias=r["bias"].cpu().numpy(),
               idx=r["idx"].cpu().numpy(), w=r["w"].cpu().numpy(), loads=r["loads"].cpu().numpy())
    return inp, res, lay


def compare_fed(shape, tokens=None, qb_mode="jacobi", logits_shape=None):
    """Both sides route from the same fp32 logits (the oracle's router GEMM,
    on logits_shape's inputs if given, else on shape's): routing must be
    bit-exact; outputs within the format's tolerance."""
    from qb_inputs.device import layer_for
    inp = QI.LayerInputs(shape)
    W = O.LayerWeights(inp)
    Wl = W if logits_shape is None else O.LayerWeights(QI.LayerInputs(logits_shape))
    logits = O.router_logits(Wl.dense("x"), Wl.dense("w_router"), Wl.dense("router_offset"))
    _, g, lay = upload_and_run(shape, logits_in=logits, layer=layer_for(shape, qb_mode=qb_mode))
    lay.close()
    o = O.layer_forward(inp, tokens=tokens, logits=logits, weights=W, mode=qb_mode)
    for name in ("scores", "bias", "idx", "w", "loads"):
        eq = bits_equal(g[name], o[name])
        assert eq.all(), f"{name}: {int((~eq).sum())} mismatches"
    tok = o["tokens"]
    err = row_rel_err(g["out"][tok], o["out"])
    assert err.max() <= tol_of(shape), f"max row error {err.max():.3e} > {tol_of(shape)}"
    return err


def compare_own_router(shape, tokens=None, min_agree=0.99):
    """The GPU computes the router logits itself (fp32-accumulated GEMM); the
    oracle computes them in fp64.  Scores agree within tolerance; routing
    agrees except at near-ties; the GPU's routing is self-consistent; outputs
    of tokens routed identically are within tolerance."""
    inp = QI.LayerInputs(shape)
    W = O.LayerWeights(inp)
    _, g, lay = upload_and_run(shape)
    lay.close()
    o = O.layer_forward(inp, tokens=tokens, weights=W)
    s_tol = 2e-6 if shape.dtype == "f32" else 1e-5
    assert np.max(np.abs(g["scores"].astype(np.float64) - o["scores"])) <= s_tol
    assert np.max(np.abs(g["bias"].astype(np.float64) - o["bias"])) <= 5 * s_tol
    check_routing_self_consistent(g["scores"], g["bias"], g["idx"], g["w"], g["loads"], shape.k)
    same = np.all(np.sort(g["idx"], axis=1) == np.sort(o["idx"], axis=1), axis=1)
    assert same.mean() >= min_agree, f"routing agreement {same.mean():.4f}"
    tok = o["tokens"]
    keep = same[tok]
    err = row_rel_err(g["out"][tok][keep], o["out"][keep])
    assert err.max() <= tol_of(shape), f"max row error {err.max():.3e}"
    return err, same.mean()
