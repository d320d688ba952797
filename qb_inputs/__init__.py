"""Seeded synthetic inputs for the Stable LatentMoE layer and its QB router.

The one source of inputs for both the CPU oracle and the CUDA path.  It holds
none of the method's arithmetic: it draws seeded tensors (see ``qbgen.c`` for
the generator's definition), converts between storage formats, and describes
the workloads by their sizes and value distributions.

Workload recipe (every weight is drawn with standard deviation 1/sqrt(fan_in);
"N(0, v)" below means variance v):

* x ~ N(0, 1); W_r [n, d], W_down [latent, d], W_gate/W_up [n, m, latent],
  W_out [n, latent, m], W_proj_up [d, latent], W_shared_gate/up [m_s, d],
  W_shared_out [d, m_s] ~ N(0, 1/fan_in); router offsets o [n] ~ N(0, v_off);
  RMSNorm gain gamma = 1 + N(0, 0.01).
* Draws are Gaussian (Box-Muller from two SplitMix64 uniforms, untruncated
  tails; see qbgen.c); weights are rounded to the workload's storage type.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass, field, replace

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qbgen.c")
_LIB = os.path.join(_HERE, "libqbgen.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the generator with gcc (OpenMP) into ``libqbgen.so``."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared",
                               "-ffp-contract=off", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            u64, i64, f32 = ctypes.c_uint64, ctypes.c_int64, ctypes.c_float
            vp = ctypes.c_void_p
            lib.qbgen_normal_f32.argtypes = [u64, u64, i64, i64, f32, vp]
            lib.qbgen_normal_bf16.argtypes = [u64, u64, i64, i64, f32, vp]
            lib.qbgen_quantize_mxfp4.argtypes = [vp, i64, i64, vp, vp]
            for f in (lib.qbgen_normal_f32, lib.qbgen_normal_bf16, lib.qbgen_quantize_mxfp4):
                f.restype = None
            _lib = lib
    return _lib


# Tensor ids of the generator streams (fixed: changing one changes the data).
TID = dict(x=1, w_router=2, router_offset=3, w_down=4, w_gate=5, w_up=6, w_out=7,
           gamma=8, w_proj_up=9, w_shared_gate=10, w_shared_up=11, w_shared_out=12,
           logit_noise=13)


def normal_f32(seed: int, tid: int, shape, sigma: float, offset: int = 0) -> np.ndarray:
    """fp32 draws of elements [offset, offset + prod(shape)) of stream (seed, tid)."""
    out = np.empty(shape, dtype=np.float32)
    _load().qbgen_normal_f32(seed, tid, offset, out.size, float(sigma), out.ctypes.data)
    return out


def normal_bf16(seed: int, tid: int, shape, sigma: float, offset: int = 0) -> np.ndarray:
    """bf16 draws (as uint16 bit patterns) of the same stream elements."""
    out = np.empty(shape, dtype=np.uint16)
    _load().qbgen_normal_bf16(seed, tid, offset, out.size, float(sigma), out.ctypes.data)
    return out


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp32 values."""
    return (bits.astype(np.uint32) << 16).view(np.float32)


def quantize_mxfp4(bits: np.ndarray):
    """bf16 bits [rows, K] -> (packed E2M1 [rows, K/2] u8, E8M0 scales [rows, K/32] u8)."""
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    *lead, K = bits.shape
    rows = int(np.prod(lead)) if lead else 1
    assert K % 32 == 0
    packed = np.empty((*lead, K // 2), dtype=np.uint8)
    scales = np.empty((*lead, K // 32), dtype=np.uint8)
    _load().qbgen_quantize_mxfp4(bits.ctypes.data, rows, K, packed.ctypes.data, scales.ctypes.data)
    return packed, scales


@dataclass(frozen=True)
class LayerShape:
    """Sizes and distributions of one Stable LatentMoE workload."""
    name: str
    T: int              # tokens
    d: int              # model width
    latent: int         # latent width (d / 2 on the pages' model)
    n: int              # routed experts
    k: int              # experts per token
    m: int              # expert GLU intermediate
    m_s: int            # merged shared-expert intermediate (0 = none)
    dtype: str          # storage type of activations and dense weights: "f32" | "bf16"
    wfmt: str           # routed-expert weights: "f32" | "bf16" | "mxfp4"
    offset_var: float   # variance of the per-expert router offsets
    seed: int = 0
    qb_sweeps: int = 1
    # Scale of the latent activations: x is drawn with standard deviation
    # h_scale (so h = x W_down^T grows by it) and the expert gate/up weights
    # with their usual deviation / h_scale, which leaves the expert's GLU
    # inputs as they were.  1 for every workload; large values exercise the
    # block scales of E4M3 token rows.
    h_scale: float = 1.0

    def with_(self, **kw) -> "LayerShape":
        return replace(self, **kw)


# The five workloads.  The model-level sizes (896 experts, 16 active, width
# 7168 -> latent 3584, merged shared expert 6144) are the ones the pages give.
TINY_F32 = LayerShape("tiny_f32", T=64, d=256, latent=128, n=32, k=4, m=64, m_s=0,
                      dtype="f32", wfmt="f32", offset_var=0.5)
ROUTE_QB = LayerShape("route_qb_T4096", T=4096, d=7168, latent=3584, n=896, k=16, m=1024,
                      m_s=6144, dtype="f32", wfmt="f32", offset_var=1.0)
DECODE = LayerShape("k3_decode_T256", T=256, d=7168, latent=3584, n=896, k=16, m=1024,
                    m_s=6144, dtype="bf16", wfmt="bf16", offset_var=1.0)
PREFILL = LayerShape("k3_prefill_T16384", T=16384, d=7168, latent=3584, n=896, k=16, m=1024,
                     m_s=6144, dtype="bf16", wfmt="bf16", offset_var=2.0)
PREFILL_MXFP4 = PREFILL.with_(name="k3_prefill_mxfp4_T16384", wfmt="mxfp4")
# The decode shape with the deployment weight format (routed experts MXFP4).
DECODE_MXFP4 = DECODE.with_(name="k3_decode_mxfp4_T256", wfmt="mxfp4")

WORKLOADS = {w.name: w for w in (TINY_F32, ROUTE_QB, DECODE, PREFILL, PREFILL_MXFP4, DECODE_MXFP4)}


def _sig(fan_in: int) -> float:
    return float(np.float32(1.0 / np.sqrt(fan_in)))


# Whole tensors drawn once per process and shared by every workload that
# draws the same stream with the same shape, spread and storage (decode and
# prefill shapes share all their weights), least recently used first out
# beyond QB_INPUTS_CACHE_GB (default 48).
_shared = {}
_shared_order = []
_shared_lock = threading.Lock()


def _shared_draw(key, make):
    with _shared_lock:
        if key in _shared:
            _shared_order.remove(key)
            _shared_order.append(key)
            return _shared[key]
    a = make()
    cap = float(os.environ.get("QB_INPUTS_CACHE_GB", "48")) * 2 ** 30
    with _shared_lock:
        _shared[key] = a
        _shared_order.append(key)
        total = sum(v.nbytes for v in _shared.values())
        while total > cap and len(_shared_order) > 1:
            old = _shared_order.pop(0)
            total -= _shared.pop(old).nbytes
    return a


def _shared_get(key):
    with _shared_lock:
        return _shared.get(key)


def clear_shared_draws():
    with _shared_lock:
        _shared.clear()
        _shared_order.clear()


class LayerInputs:
    """Host-side inputs of one workload, drawn lazily per tensor.

    Dense tensors come back as storage bit patterns (uint16 for bf16) or fp32;
    ``values(name)`` widens them to fp32 exactly.  Expert tensors can be drawn
    one expert at a time (``expert(name, e)``) so that an oracle check of a few
    tokens at full size never materialises all experts.
    """

    def __init__(self, shape: LayerShape):
        self.shape = shape
        s = shape
        self.specs = {
            "x": ((s.T, s.d), float(s.h_scale), s.dtype),
            "w_router": ((s.n, s.d), _sig(s.d), s.dtype),
            "router_offset": ((s.n,), float(np.sqrt(s.offset_var)), "f32"),
            "w_down": ((s.latent, s.d), _sig(s.d), s.dtype),
            "w_gate": ((s.n, s.m, s.latent), _sig(s.latent) / float(s.h_scale), s.wfmt),
            "w_up": ((s.n, s.m, s.latent), _sig(s.latent) / float(s.h_scale), s.wfmt),
            "w_out": ((s.n, s.latent, s.m), _sig(s.m), s.wfmt),
            "gamma": ((s.latent,), 0.1, "f32"),
            "w_proj_up": ((s.d, s.latent), _sig(s.latent), s.dtype),
        }
        if s.m_s:
            self.specs.update({
                "w_shared_gate": ((s.m_s, s.d), _sig(s.d), s.dtype),
                "w_shared_up": ((s.m_s, s.d), _sig(s.d), s.dtype),
                "w_shared_out": ((s.d, s.m_s), _sig(s.m_s), s.dtype),
            })
        self._cache = {}

    def _draw(self, name, shape, sigma, fmt, offset=0):
        tid = TID[name]
        if fmt == "f32":
            a = normal_f32(self.shape.seed, tid, shape, sigma, offset)
        else:  # bf16 storage, and the bf16 master copy of MXFP4 weights
            a = normal_bf16(self.shape.seed, tid, shape, sigma, offset)
        if name == "gamma":
            a = (np.float32(1.0) + a).astype(np.float32)
        return a

    def _key(self, name):
        shape, sigma, fmt = self.specs[name]
        return (self.shape.seed, name, tuple(shape), float(sigma), "f32" if fmt == "f32" else "bf16")

    def raw(self, name):
        """Whole tensor in its storage form (bf16 bits / fp32 / bf16 master of MXFP4)."""
        if name not in self._cache:
            shape, sigma, fmt = self.specs[name]
            self._cache[name] = _shared_draw(self._key(name), lambda: self._draw(name, shape, sigma, fmt))
        return self._cache[name]

    def drop(self, name):
        self._cache.pop(name, None)

    def values(self, name) -> np.ndarray:
        """fp32 values of a dense tensor (exact widening of its storage)."""
        a = self.raw(name)
        return bf16_bits_to_f32(a) if a.dtype == np.uint16 else a

    def expert_raw(self, name, e: int):
        """Storage form of expert e's slice of an expert tensor (a view of the
        whole tensor when it has been drawn, else drawn alone)."""
        shape, sigma, fmt = self.specs[name]
        whole = self._cache.get(name)
        if whole is None:
            whole = _shared_get(self._key(name))
        if whole is not None:
            return whole[int(e)]
        per = int(shape[1]) * int(shape[2])
        return self._draw(name, shape[1:], sigma, fmt, offset=int(e) * per)

    def mxfp4(self, name):
        """(packed, scales) of an expert tensor quantised to MXFP4."""
        key = name + ":mxfp4"
        if key not in self._cache:
            self._cache[key] = quantize_mxfp4(self.raw(name))
        return self._cache[key]

    def expert_mxfp4(self, name, e: int):
        return quantize_mxfp4(self.expert_raw(name, e))
