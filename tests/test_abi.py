"""The C-ABI library: it loads, exports what include/qbmoe.h declares, and
rejects bad arguments on the host before touching a device (no GPU needed)."""
import ctypes

import pytest

import quantile_balanced_routing_gb300 as Q


@pytest.fixture(scope="module")
def lib():
    return Q.load_library()


def test_every_declared_function_is_exported(lib):
    names = Q.declared_functions()
    for must in ("moe_route_qb", "moe_latent_forward", "qbmoe_create", "qbmoe_destroy", "qbmoe_set_weights",
                 "qbmoe_pack_weights", "qbmoe_status", "qbmoe_route_workspace_bytes"):
        assert must in names
    for nm in names:
        assert hasattr(lib, nm), nm


def test_strerror(lib):
    assert Q.strerror(0) == "ok"
    assert "workspace" in Q.strerror(Q.QBMOE_EWORKSPACE)
    assert Q.strerror(-99) == "unknown status"


def test_route_workspace_size(lib):
    assert Q.qbmoe_route_workspace_bytes(0, 8, 2) == 0
    a = Q.qbmoe_route_workspace_bytes(4096, 896, 16)
    assert a >= 4096 * 896 * 4
    assert Q.qbmoe_route_workspace_bytes(8192, 896, 16) > a


FAKE = 1 << 20   # 256-aligned fake device address: never dereferenced by the host checks


@pytest.mark.parametrize("T,n,k,sweeps", [(0, 8, 2, 1), (4, 1, 1, 1), (4, 8, 8, 1), (4, 8, 0, 1),
                                          (4, 2000, 4, 1), (4, 64, 33, 1), (4, 8, 2, -1)])
def test_route_rejects_bad_sizes(lib, T, n, k, sweeps):
    rc = lib.moe_route_qb(T, n, k, sweeps, FAKE, None, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 30, None)
    assert rc == Q.QBMOE_EINVAL


def test_route_rejects_null_misaligned_and_small_workspace(lib):
    args = [8, 16, 2, 1, FAKE, None, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 30, None]
    bad = list(args)
    bad[4] = None
    assert lib.moe_route_qb(*bad) == Q.QBMOE_EINVAL
    bad = list(args)
    bad[7] = FAKE + 4
    assert lib.moe_route_qb(*bad) == Q.QBMOE_EINVAL
    bad = list(args)
    bad[11] = FAKE + 16    # workspace must be 256-byte aligned
    assert lib.moe_route_qb(*bad) == Q.QBMOE_EINVAL
    bad = list(args)
    bad[12] = 64
    assert lib.moe_route_qb(*bad) == Q.QBMOE_EWORKSPACE


def _cfg(**kw):
    base = dict(d=256, latent=128, n_experts=32, top_k=4, expert_inter=64, shared_inter=0, situ_beta1=4.0,
                situ_beta2=25.0, rms_eps=1e-6, act_dtype=Q.QBMOE_F32, expert_wfmt=Q.QBMOE_W_F32, qb_sweeps=1,
                qb_mode=Q.QBMOE_QB_JACOBI)
    base.update(kw)
    return Q.QbmoeConfig(**base)


@pytest.mark.parametrize("kw", [dict(top_k=32), dict(n_experts=1), dict(n_experts=4096), dict(d=0),
                                dict(act_dtype=7), dict(expert_wfmt=Q.QBMOE_W_MXFP4),
                                dict(act_dtype=Q.QBMOE_BF16, expert_wfmt=Q.QBMOE_W_F32),
                                dict(act_dtype=Q.QBMOE_BF16, expert_wfmt=Q.QBMOE_W_MXFP4, latent=120),
                                dict(situ_beta1=0.0), dict(qb_sweeps=-1), dict(top_k=40, n_experts=64),
                                dict(act_dtype=Q.QBMOE_BF16, expert_wfmt=Q.QBMOE_W_BF16, d=260),
                                dict(qb_mode=2), dict(qb_mode=-1)])
def test_create_rejects_bad_configs(lib, kw):
    ctx = ctypes.c_void_p()
    cfg = _cfg(**kw)
    assert lib.qbmoe_create(ctypes.byref(ctx), ctypes.byref(cfg), 64) == Q.QBMOE_EINVAL
    assert not ctx.value
    assert lib.qbmoe_layer_workspace_bytes(ctypes.byref(cfg), 64) == 0


def test_layer_workspace_grows_with_tokens(lib):
    cfg = _cfg()
    a = lib.qbmoe_layer_workspace_bytes(ctypes.byref(cfg), 64)
    b = lib.qbmoe_layer_workspace_bytes(ctypes.byref(cfg), 128)
    assert 0 < a < b
    assert lib.qbmoe_create(None, ctypes.byref(cfg), 64) == Q.QBMOE_EINVAL


def test_null_context_calls(lib):
    assert lib.qbmoe_destroy(None) == 0
    assert lib.moe_latent_forward(None, 4, FAKE, None, None, None, FAKE, None, None, None, None, None) == Q.QBMOE_EINVAL
    assert lib.qbmoe_set_weights(None, None) == Q.QBMOE_EINVAL
    assert lib.qbmoe_set_timing(None, 1) == Q.QBMOE_EINVAL
    assert lib.qbmoe_pack_weights(None, None, None) == Q.QBMOE_EINVAL

