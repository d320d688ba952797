"""Python binding of libqbmoe (Stable LatentMoE forward with Quantile Balancing).

Argument marshalling only: every step of the path runs in the library's CUDA
kernels.  PyTorch provides device memory and streams.  There is no CPU
fallback: if ``libqbmoe.so`` is missing, loading it raises.

The C entry points are exposed under their C names (``moe_route_qb``,
``moe_latent_forward``, ``qbmoe_*``) taking plain integers/pointers, plus two
torch conveniences, :func:`route_qb` and :class:`LatentMoE`, that allocate
outputs with torch and call them.
"""
from __future__ import annotations

import ctypes
import os
import re
from typing import Optional

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libqbmoe.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "qbmoe.h")

QBMOE_OK, QBMOE_EINVAL, QBMOE_ENOMEM, QBMOE_ECUDA = 0, -1, -2, -3
QBMOE_EARCH, QBMOE_EWORKSPACE, QBMOE_ETIMEOUT, QBMOE_EDEVICE = -4, -5, -6, -7
QBMOE_F32, QBMOE_BF16 = 0, 1
QBMOE_W_F32, QBMOE_W_BF16, QBMOE_W_MXFP4 = 0, 1, 2
QBMOE_QB_JACOBI, QBMOE_QB_GAUSS_SEIDEL = 0, 1
MAX_EXPERTS, MAX_TOPK = 1024, 32


class QbmoeConfig(ctypes.Structure):
    _fields_ = [("d", ctypes.c_int), ("latent", ctypes.c_int), ("n_experts", ctypes.c_int),
                ("top_k", ctypes.c_int), ("expert_inter", ctypes.c_int), ("shared_inter", ctypes.c_int),
                ("situ_beta1", ctypes.c_float), ("situ_beta2", ctypes.c_float), ("rms_eps", ctypes.c_float),
                ("act_dtype", ctypes.c_int), ("expert_wfmt", ctypes.c_int), ("qb_sweeps", ctypes.c_int),
                ("qb_mode", ctypes.c_int)]


_WEIGHT_FIELDS = ["w_router", "router_offset", "w_down", "w_gate", "w_up", "w_out", "s_gate", "s_up",
                  "s_out", "rms_gamma", "w_proj_up", "w_shared_gate", "w_shared_up", "w_shared_out"]


class QbmoeWeights(ctypes.Structure):
    _fields_ = [(f, ctypes.c_void_p) for f in _WEIGHT_FIELDS]


class QbmoeError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {strerror(code)} ({code})")


_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libqbmoe.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build it with "
                          "`python -m quantile_balanced_routing_gb300._build` (there is no CPU fallback)")
    lib = ctypes.CDLL(path)
    i, vp, sz, f32p = ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p
    lib.qbmoe_route_workspace_bytes.argtypes = [i, i, i]
    lib.qbmoe_route_workspace_bytes.restype = sz
    lib.moe_route_qb.argtypes = [i, i, i, i, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.moe_route_qb.restype = i
    lib.qbmoe_route_gs_workspace_bytes.argtypes = [i, i, i]
    lib.qbmoe_route_gs_workspace_bytes.restype = sz
    lib.moe_route_qb_gs.argtypes = [i, i, i, i, i, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.moe_route_qb_gs.restype = i
    lib.moe_route_qb_noalloc.argtypes = [i, i, i, i, vp, vp, vp, vp, vp, vp, vp, vp]
    lib.moe_route_qb_noalloc.restype = i
    lib.qbmoe_route_noalloc_max_bytes.argtypes = []
    lib.qbmoe_route_noalloc_max_bytes.restype = sz
    lib.qbmoe_route_signsgd_workspace_bytes.argtypes = [i, i, i]
    lib.qbmoe_route_signsgd_workspace_bytes.restype = sz
    lib.moe_route_signsgd.argtypes = [i, i, i, i, ctypes.c_float, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.moe_route_signsgd.restype = i
    for nm in ("qbmoe_qb_hist_state_bytes", "qbmoe_qb_hist_bytes"):
        getattr(lib, nm).argtypes = [i]
        getattr(lib, nm).restype = sz
    lib.qbmoe_qb_shard_workspace_bytes.argtypes = [i, i, i]
    lib.qbmoe_qb_shard_workspace_bytes.restype = sz
    lib.moe_qb_hist_init.argtypes = [i, i, i, vp, vp, vp]
    lib.moe_qb_shard_margins.argtypes = [i, i, i, vp, vp, vp, vp, sz, vp]
    lib.moe_qb_shard_hist.argtypes = [i, i, i, vp, vp, vp, vp]
    lib.moe_qb_hist_advance.argtypes = [i, i, vp, vp, vp]
    lib.moe_qb_hist_bias.argtypes = [i, vp, vp, vp]
    for nm in ("moe_qb_hist_init", "moe_qb_shard_margins", "moe_qb_shard_hist", "moe_qb_hist_advance",
               "moe_qb_hist_bias"):
        getattr(lib, nm).restype = i
    lib.qbmoe_create.argtypes = [ctypes.POINTER(vp), ctypes.POINTER(QbmoeConfig), i]
    lib.qbmoe_create.restype = i
    lib.qbmoe_layer_workspace_bytes.argtypes = [ctypes.POINTER(QbmoeConfig), i]
    lib.qbmoe_layer_workspace_bytes.restype = sz
    lib.qbmoe_set_weights.argtypes = [vp, ctypes.POINTER(QbmoeWeights)]
    lib.qbmoe_set_weights.restype = i
    lib.qbmoe_pack_weights.argtypes = [vp, ctypes.POINTER(QbmoeWeights), vp]
    lib.qbmoe_pack_weights.restype = i
    lib.qbmoe_destroy.argtypes = [vp]
    lib.qbmoe_destroy.restype = i
    lib.moe_latent_forward.argtypes = [vp, i, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
    lib.moe_latent_forward.restype = i
    lib.qbmoe_status.argtypes = [vp, vp]
    lib.qbmoe_status.restype = i
    lib.qbmoe_set_timing.argtypes = [vp, i]
    lib.qbmoe_set_timing.restype = i
    lib.qbmoe_stage_times.argtypes = [vp, ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_char_p), i]
    lib.qbmoe_stage_times.restype = i
    lib.qbmoe_last_launch_count.argtypes = [vp]
    lib.qbmoe_last_launch_count.restype = i
    lib.qbmoe_route_last_launch_count.argtypes = []
    lib.qbmoe_route_last_launch_count.restype = i
    lib.qbmoe_set_wait_limit.argtypes = [vp, ctypes.c_longlong]
    lib.qbmoe_set_wait_limit.restype = i
    lib.qbmoe_debug_stall.argtypes = [vp, i]
    lib.qbmoe_debug_stall.restype = i
    lib.qbmoe_uses_tensor_cores.argtypes = [vp]
    lib.qbmoe_uses_tensor_cores.restype = i
    lib.qbmoe_mma_probe.argtypes = [i, i, ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_double)]
    lib.qbmoe_mma_probe.restype = i
    lib.qbmoe_strerror.argtypes = [i]
    lib.qbmoe_strerror.restype = ctypes.c_char_p
    _lib = lib
    return lib


def declared_functions(header: str = HEADER):
    """Names of the functions include/qbmoe.h declares."""
    text = open(header).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(?:int|size_t|const char\*)\s+\**\s*(\w+)\s*\(", text)))


def strerror(code: int) -> str:
    return load_library().qbmoe_strerror(code).decode()


def _p(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream_ptr(stream) -> Optional[int]:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream or None


# ---------------------------------------------------------------------------
# C entry points (thin, same names)
# ---------------------------------------------------------------------------

def qbmoe_route_workspace_bytes(T: int, n: int, k: int) -> int:
    return load_library().qbmoe_route_workspace_bytes(T, n, k)


def moe_route_qb(T, n, k, qb_sweeps, logits, bias_in, bias_out, scores, topk_idx, topk_w, loads,
                 workspace, workspace_bytes, stream) -> int:
    return load_library().moe_route_qb(T, n, k, qb_sweeps, logits, bias_in, bias_out, scores, topk_idx,
                                       topk_w, loads, workspace, workspace_bytes, stream)


def moe_route_qb_noalloc(T, n, k, qb_sweeps, logits, bias_in, bias_out, scores, topk_idx, topk_w, loads,
                         stream) -> int:
    return load_library().moe_route_qb_noalloc(T, n, k, qb_sweeps, logits, bias_in, bias_out, scores, topk_idx,
                                               topk_w, loads, stream)


def moe_latent_forward(ctx, T, x, logits_in, bias_in, bias_out, out, scores, idx, w, loads, stream) -> int:
    return load_library().moe_latent_forward(ctx, T, x, logits_in, bias_in, bias_out, out, scores, idx, w,
                                             loads, stream)


def qbmoe_status(ctx, stream) -> int:
    return load_library().qbmoe_status(ctx, stream)


# ---------------------------------------------------------------------------
# torch conveniences (allocation through torch; compute in the library)
# ---------------------------------------------------------------------------

def route_qb(logits, k: int, qb_sweeps: int = 1, bias_in=None, bias_out=None, workspace=None, stream=None):
    """Route fp32 logits [T, n] on the GPU.  Returns (scores, bias, idx, w, loads)."""
    import torch
    T, n = logits.shape
    dev = logits.device
    assert logits.dtype == torch.float32 and logits.is_contiguous() and dev.type == "cuda"
    scores = torch.empty((T, n), dtype=torch.float32, device=dev)
    idx = torch.empty((T, k), dtype=torch.int32, device=dev)
    w = torch.empty((T, k), dtype=torch.float32, device=dev)
    loads = torch.empty((n,), dtype=torch.int32, device=dev)
    if bias_out is None:
        bias_out = torch.empty((n,), dtype=torch.float32, device=dev)
    need = qbmoe_route_workspace_bytes(T, n, k)
    if workspace is None or workspace.numel() < need:
        workspace = torch.empty((max(need, 256),), dtype=torch.uint8, device=dev)
    rc = moe_route_qb(T, n, k, qb_sweeps, _p(logits), _p(bias_in), _p(bias_out), _p(scores), _p(idx), _p(w),
                      _p(loads), _p(workspace), workspace.numel(), _stream_ptr(stream))
    if rc:
        raise QbmoeError(rc, "moe_route_qb")
    return scores, bias_out, idx, w, loads


def route_qb_gs(logits, k: int, max_sweeps: int = 1, stop_when_balanced: bool = False, bias_in=None,
                stream=None):
    """Cyclic coordinate-descent QB on fp32 logits [T, n] (moe_route_qb_gs).
    Returns (scores, bias, idx, w, loads, sweeps_done)."""
    import torch
    T, n = logits.shape
    dev = logits.device
    assert logits.dtype == torch.float32 and logits.is_contiguous() and dev.type == "cuda"
    scores = torch.empty((T, n), dtype=torch.float32, device=dev)
    idx = torch.empty((T, k), dtype=torch.int32, device=dev)
    w = torch.empty((T, k), dtype=torch.float32, device=dev)
    loads = torch.empty((n,), dtype=torch.int32, device=dev)
    bias_out = torch.empty((n,), dtype=torch.float32, device=dev)
    done = torch.zeros((4,), dtype=torch.int32, device=dev)
    lib = load_library()
    need = lib.qbmoe_route_gs_workspace_bytes(T, n, k)
    ws = torch.empty((max(need, 256),), dtype=torch.uint8, device=dev)
    rc = lib.moe_route_qb_gs(T, n, k, max_sweeps, int(stop_when_balanced), _p(logits), _p(bias_in), _p(bias_out),
                             _p(scores), _p(idx), _p(w), _p(loads), _p(done), _p(ws), ws.numel(),
                             _stream_ptr(stream))
    if rc:
        raise QbmoeError(rc, "moe_route_qb_gs")
    return scores, bias_out, idx, w, loads, done[:1]


QBMOE_PROBE_BF16, QBMOE_PROBE_MXF4F8 = 0, 1


def mma_probe(kind: str, iters: int = 20000):
    """(milliseconds, flops) of one run of the library's tensor-core rate
    probe for kind "bf16" (kind::f16) or "mxf8f6f4" (block-scaled E2M1 x
    E4M3)."""
    code = {"bf16": QBMOE_PROBE_BF16, "mxf8f6f4": QBMOE_PROBE_MXF4F8}[kind]
    ms, fl = ctypes.c_float(), ctypes.c_double()
    rc = load_library().qbmoe_mma_probe(code, iters, ctypes.byref(ms), ctypes.byref(fl))
    if rc:
        raise QbmoeError(rc, "qbmoe_mma_probe")
    return ms.value, fl.value


def mma_peak_tflops(kind: str, runs: int = 3, iters: int = 20000) -> float:
    """Best TFLOP/s of `runs` probe runs of one MMA kind on the current GPU."""
    best = 0.0
    for _ in range(runs):
        ms, fl = mma_probe(kind, iters)
        best = max(best, fl / (ms * 1e-3) / 1e12)
    return best


def route_signsgd(logits, k: int, steps: int, gamma: float, bias_in=None, stream=None):
    """DeepSeek-V3's sign rule on fp32 logits [T, n] (moe_route_signsgd).
    Returns (scores, bias, idx, w, loads)."""
    import torch
    T, n = logits.shape
    dev = logits.device
    assert logits.dtype == torch.float32 and logits.is_contiguous() and dev.type == "cuda"
    scores = torch.empty((T, n), dtype=torch.float32, device=dev)
    idx = torch.empty((T, k), dtype=torch.int32, device=dev)
    w = torch.empty((T, k), dtype=torch.float32, device=dev)
    loads = torch.empty((n,), dtype=torch.int32, device=dev)
    bias_out = torch.empty((n,), dtype=torch.float32, device=dev)
    lib = load_library()
    need = lib.qbmoe_route_signsgd_workspace_bytes(T, n, k)
    ws = torch.empty((max(need, 256),), dtype=torch.uint8, device=dev)
    rc = lib.moe_route_signsgd(T, n, k, steps, gamma, _p(logits), _p(bias_in), _p(bias_out), _p(scores), _p(idx),
                               _p(w), _p(loads), _p(ws), ws.numel(), _stream_ptr(stream))
    if rc:
        raise QbmoeError(rc, "moe_route_signsgd")
    return scores, bias_out, idx, w, loads


class LatentMoE:
    """One Stable LatentMoE layer bound to a libqbmoe context on the current device."""

    def __init__(self, d, latent, n_experts, top_k, expert_inter, shared_inter, act_dtype="bf16",
                 expert_wfmt="bf16", qb_sweeps=1, max_tokens=256, situ_beta1=4.0, situ_beta2=25.0,
                 rms_eps=1e-6, qb_mode="jacobi"):
        self.lib = load_library()
        self.cfg = QbmoeConfig(d, latent, n_experts, top_k, expert_inter, shared_inter, situ_beta1,
                               situ_beta2, rms_eps, QBMOE_BF16 if act_dtype == "bf16" else QBMOE_F32,
                               {"f32": QBMOE_W_F32, "bf16": QBMOE_W_BF16, "mxfp4": QBMOE_W_MXFP4}[expert_wfmt],
                               qb_sweeps,
                               {"jacobi": QBMOE_QB_JACOBI, "gauss_seidel": QBMOE_QB_GAUSS_SEIDEL}[qb_mode])
        self.ctx = ctypes.c_void_p()
        rc = self.lib.qbmoe_create(ctypes.byref(self.ctx), ctypes.byref(self.cfg), max_tokens)
        if rc:
            raise QbmoeError(rc, "qbmoe_create")
        self.max_tokens = max_tokens
        self._weights = {}

    def close(self):
        if self.ctx:
            self.lib.qbmoe_destroy(self.ctx)
            self.ctx = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def set_weights(self, **tensors):
        """Tensors by qbmoe_weights field name; the layer keeps references."""
        self._weights = dict(tensors)
        w = QbmoeWeights(*[_p(tensors.get(f)) for f in _WEIGHT_FIELDS])
        rc = self.lib.qbmoe_set_weights(self.ctx, ctypes.byref(w))
        if rc:
            raise QbmoeError(rc, "qbmoe_set_weights")

    def pack_weights(self, stream=None, **tensors):
        """Copy the tensors (by qbmoe_weights field name) into memory the
        context owns (qbmoe_pack_weights); the caller's tensors may then go."""
        w = QbmoeWeights(*[_p(tensors.get(f)) for f in _WEIGHT_FIELDS])
        rc = self.lib.qbmoe_pack_weights(self.ctx, ctypes.byref(w), _stream_ptr(stream))
        if rc:
            raise QbmoeError(rc, "qbmoe_pack_weights")
        self._weights = {}

    def forward(self, x, logits_in=None, bias_in=None, bias_out=None, out=None, want_routing=False, stream=None):
        import torch
        T = x.shape[0]
        dev = x.device
        n, k = self.cfg.n_experts, self.cfg.top_k
        if out is None:
            out = torch.empty((T, self.cfg.d), dtype=x.dtype, device=dev)
        r = {}
        if want_routing:
            r = dict(scores=torch.empty((T, n), dtype=torch.float32, device=dev),
                     idx=torch.empty((T, k), dtype=torch.int32, device=dev),
                     w=torch.empty((T, k), dtype=torch.float32, device=dev),
                     loads=torch.empty((n,), dtype=torch.int32, device=dev))
            if bias_out is None:
                bias_out = torch.empty((n,), dtype=torch.float32, device=dev)
        rc = self.lib.moe_latent_forward(self.ctx, T, _p(x), _p(logits_in), _p(bias_in), _p(bias_out), _p(out),
                                         _p(r.get("scores")), _p(r.get("idx")), _p(r.get("w")),
                                         _p(r.get("loads")), _stream_ptr(stream))
        if rc:
            raise QbmoeError(rc, "moe_latent_forward")
        if want_routing:
            r["bias"] = bias_out
            return out, r
        return out

    def status(self, stream=None) -> int:
        return self.lib.qbmoe_status(self.ctx, _stream_ptr(stream))

    def set_timing(self, slots: int):
        """Record per-stage events for the next `slots` forwards (0 = off)."""
        rc = self.lib.qbmoe_set_timing(self.ctx, int(slots))
        if rc:
            raise QbmoeError(rc, "qbmoe_set_timing")

    def stage_times(self):
        ms = (ctypes.c_float * 16)()
        names = (ctypes.c_char_p * 16)()
        n = self.lib.qbmoe_stage_times(self.ctx, ms, names, 16)
        return [(names[i].decode(), ms[i]) for i in range(max(n, 0))]

    def last_launch_count(self) -> int:
        return self.lib.qbmoe_last_launch_count(self.ctx)

    def set_wait_limit(self, iterations: int):
        return self.lib.qbmoe_set_wait_limit(self.ctx, iterations)

    def debug_stall(self, on: bool):
        return self.lib.qbmoe_debug_stall(self.ctx, int(on))

    @property
    def uses_tensor_cores(self) -> bool:
        return bool(self.lib.qbmoe_uses_tensor_cores(self.ctx))
