"""Upload a workload's seeded inputs to the GPU as torch tensors.

Marshalling only (no arithmetic): host bit patterns are copied as they are.
Returns tensors keyed by the C ABI's qbmoe_weights field names, plus "x".
"""
from __future__ import annotations

import numpy as np

from . import LayerInputs


def _t(a: np.ndarray, device, pinned=False):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a))
    if a.dtype == np.uint16:
        t = t.view(torch.bfloat16)
    if pinned:
        t = t.pin_memory()
    return t.to(device, non_blocking=False)


def upload(inp: LayerInputs, device="cuda", drop_host=True):
    s = inp.shape
    out = {}
    names = ["x", "w_router", "router_offset", "w_down", "gamma", "w_proj_up"]
    if s.m_s:
        names += ["w_shared_gate", "w_shared_up", "w_shared_out"]
    for nm in names:
        key = "rms_gamma" if nm == "gamma" else nm
        out[key] = _t(inp.raw(nm), device)
        if drop_host and nm not in ("x", "router_offset", "gamma"):
            inp.drop(nm)
    for nm, sc in (("w_gate", "s_gate"), ("w_up", "s_up"), ("w_out", "s_out")):
        if s.wfmt == "mxfp4":
            packed, scales = inp.mxfp4(nm)
            out[nm] = _t(packed, device)
            out[sc] = _t(scales, device)
            if drop_host:
                inp.drop(nm + ":mxfp4")
        else:
            out[nm] = _t(inp.raw(nm), device)
        if drop_host:
            inp.drop(nm)
    return out


def layer_for(shape, max_tokens=None, qb_sweeps=None, qb_mode="jacobi"):
    """A LatentMoE context configured for a workload shape."""
    from quantile_balanced_routing_gb300 import LatentMoE
    return LatentMoE(shape.d, shape.latent, shape.n, shape.k, shape.m, shape.m_s, act_dtype=shape.dtype,
                     expert_wfmt=shape.wfmt, qb_sweeps=shape.qb_sweeps if qb_sweeps is None else qb_sweeps,
                     max_tokens=max_tokens or shape.T, qb_mode=qb_mode)
