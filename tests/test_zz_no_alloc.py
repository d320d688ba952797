"""moe_route_qb_noalloc: the router for callers that cannot allocate device
memory (serving paths whose memory is planned up front, plug-ins given only
their inputs and outputs).  Its results must equal moe_route_qb's, bit for bit, on
consecutive calls that reuse its fixed scratch array.  This file is collected
last so that a run stopping at the first failure has run every other test."""
import numpy as np
import pytest

import quantile_balanced_routing_gb300 as Q
import qb_inputs as QI

F32 = np.float32


def test_noalloc_rejects_sizes_beyond_its_scratch_on_the_host():
    lib = Q.load_library()
    cap = lib.qbmoe_route_noalloc_max_bytes()
    assert cap == 32 << 20
    T, n, k = 16384, 896, 16          # needs ~59 MB of scratch
    assert Q.qbmoe_route_workspace_bytes(T, n, k) > cap
    fake = 1 << 20
    rc = Q.moe_route_qb_noalloc(T, n, k, 1, fake, None, fake, fake, fake, fake, fake, None)
    assert rc == Q.QBMOE_EWORKSPACE
    assert Q.moe_route_qb_noalloc(0, n, k, 1, fake, None, fake, fake, fake, fake, fake, None) == Q.QBMOE_EINVAL


def _run_noalloc(logits, k, sweeps, bias_in):
    import torch
    T, n = logits.shape
    dev = logits.device
    scores = torch.empty((T, n), dtype=torch.float32, device=dev)
    idx = torch.empty((T, k), dtype=torch.int32, device=dev)
    w = torch.empty((T, k), dtype=torch.float32, device=dev)
    loads = torch.empty((n,), dtype=torch.int32, device=dev)
    bias_out = torch.empty((n,), dtype=torch.float32, device=dev)
    p = lambda t: None if t is None else t.data_ptr()
    rc = Q.moe_route_qb_noalloc(T, n, k, sweeps, p(logits), p(bias_in), p(bias_out), p(scores), p(idx), p(w),
                                p(loads), torch.cuda.current_stream().cuda_stream or None)
    assert rc == 0, Q.strerror(rc)
    return scores, bias_out, idx, w, loads


@pytest.mark.gpu
def test_noalloc_matches_workspace_router_on_two_calls_in_a_row():
    import torch
    dev = torch.device("cuda:0")
    cases = [(4096, 896, 16, 1, 1.0, 0.0), (777, 100, 7, 2, 2.0, 0.1)]
    for i, (T, n, k, sweeps, ov, bs) in enumerate(cases):
        z = QI.normal_f32(50 + i, QI.TID["logit_noise"], (T, n), 1.0)
        o = QI.normal_f32(50 + i, QI.TID["router_offset"], (n,), float(np.sqrt(ov)))
        logits = torch.from_numpy((z + o[None, :]).astype(F32)).to(dev)
        bias_in = None if bs == 0 else torch.from_numpy(QI.normal_f32(60 + i, 77, (n,), bs)).to(dev)
        got = _run_noalloc(logits, k, sweeps, bias_in)
        want = Q.route_qb(logits, k, qb_sweeps=sweeps, bias_in=bias_in)
        torch.cuda.synchronize()
        for name, a, b in zip(("scores", "bias", "idx", "w", "loads"), got, want):
            a, b = a.cpu().numpy(), b.cpu().numpy()
            assert np.array_equal(a.view(np.uint8), b.view(np.uint8)), name
