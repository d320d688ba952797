"""GPU parity of moe_latent_forward (through the C ABI) against the CPU oracle."""
import numpy as np
import pytest

import qb_inputs as QI
from layer_check import compare_fed, compare_own_router, upload_and_run

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

SMALL_BF16 = QI.LayerShape("small_bf16", T=300, d=512, latent=256, n=64, k=8, m=128, m_s=256,
                           dtype="bf16", wfmt="bf16", offset_var=1.0)
SMALL_MXFP4 = SMALL_BF16.with_(name="small_mxfp4", wfmt="mxfp4")
RAGGED_F32 = QI.LayerShape("ragged_f32", T=77, d=96, latent=64, n=10, k=3, m=40, m_s=48,
                           dtype="f32", wfmt="f32", offset_var=1.0)
FROZEN_BF16 = SMALL_BF16.with_(name="frozen_bf16", T=129, qb_sweeps=0)
ONE_TOKEN = SMALL_BF16.with_(name="one_token", T=1)
# tensor-core tilings: ~8 tokens per expert (16-token tiles), ~525 per expert
# (256-token tiles plus ragged tails), dense GEMMs with 256-token tiles and tails
TC_DECODE_LIKE = SMALL_BF16.with_(name="tc_decode_like", T=64)
TC_PREFILL_LIKE = QI.LayerShape("tc_prefill_like", T=2100, d=512, latent=256, n=32, k=8, m=128, m_s=512,
                                dtype="bf16", wfmt="bf16", offset_var=2.0)
# MXFP4 expert weights on the tensor-core path (K multiples of 512 for the
# scale loads): 64-, 16- and 160-row token tiles
TC_MXFP4 = QI.LayerShape("tc_mxfp4", T=300, d=1024, latent=512, n=64, k=8, m=512, m_s=512,
                         dtype="bf16", wfmt="mxfp4", offset_var=1.0)
TC_MXFP4_DECODE_LIKE = TC_MXFP4.with_(name="tc_mxfp4_decode_like", T=64)
TC_MXFP4_PREFILL_LIKE = TC_MXFP4.with_(name="tc_mxfp4_prefill_like", T=1200, n=32, offset_var=2.0)
# edge cases of the tensor-core tilings: one token (a 1-row tile through the
# stacked block-scaled MMA), two tokens on bf16 weights
TC_MXFP4_ONE_TOKEN = TC_MXFP4.with_(name="tc_mxfp4_one_token", T=1)
TC_TWO_TOKENS = TC_DECODE_LIKE.with_(name="tc_two_tokens", T=2)


@pytest.mark.parametrize("shape", [QI.TINY_F32, RAGGED_F32, SMALL_BF16, SMALL_MXFP4, FROZEN_BF16, ONE_TOKEN,
                                   TC_DECODE_LIKE, TC_PREFILL_LIKE, TC_MXFP4, TC_MXFP4_DECODE_LIKE,
                                   TC_MXFP4_PREFILL_LIKE, TC_MXFP4_ONE_TOKEN, TC_TWO_TOKENS],
                         ids=lambda s: s.name)
def test_layer_fed_logits(shape):
    compare_fed(shape)


@pytest.mark.parametrize("shape", [TC_MXFP4_DECODE_LIKE, TC_MXFP4_PREFILL_LIKE, TC_MXFP4_ONE_TOKEN],
                         ids=lambda s: s.name)
def test_mxfp4_large_latent_activations(shape):
    """Latent activations a thousand times larger (|h| in the thousands, far
    past E4M3's largest finite value, 448) with gate/up weights a thousand
    times smaller, so the experts' GLU inputs are as usual: the per-32 block
    scales of the E4M3 token rows keep the block-scaled experts within the
    MXFP4 tolerance.  Routing comes from the unscaled workload's logits."""
    big = shape.with_(name=shape.name + "_h1000", h_scale=1000.0)
    compare_fed(big, logits_shape=shape)


def test_mxfp4_layers_run_on_tensor_cores():
    from qb_inputs.device import layer_for
    lay = layer_for(TC_MXFP4)
    assert lay.uses_tensor_cores
    lay.close()
    lay = layer_for(SMALL_MXFP4)      # latent 256: scale rows too short for the scale loads
    assert not lay.uses_tensor_cores
    lay.close()


def test_mxfp4_weights_need_32_byte_alignment():
    """Packed E2M1 weights are read by unpacking TMA copies that need 32-byte
    aligned bases: qbmoe_set_weights refuses a base that is only 16-byte
    aligned (a host-side check; the layer is not run)."""
    import quantile_balanced_routing_gb300 as Q
    from qb_inputs.device import layer_for, upload
    d = upload(QI.LayerInputs(TC_MXFP4), "cuda:0")
    w = {k: v for k, v in d.items() if k != "x"}
    lay = layer_for(TC_MXFP4)
    lay.set_weights(**w)
    w["w_up"] = w["w_up"].view(torch.uint8).flatten()[16:]    # base 16 bytes past a 32-byte boundary
    with pytest.raises(Q.QbmoeError) as err:
        lay.set_weights(**w)
    assert err.value.code == Q.QBMOE_EINVAL
    lay.close()


@pytest.mark.parametrize("shape", [TC_DECODE_LIKE, TC_TWO_TOKENS, QI.DECODE], ids=lambda s: s.name)
def test_gathered_token_rows_match_the_copied_ones(shape, monkeypatch):
    """Decode-sized token tiles gather their rows from h by route (TMA
    four-row gathers); QBMOE_NO_GATHER=1 makes the same launch read an
    expert-ordered copy instead.  The same bytes reach shared memory, so the
    outputs are identical."""
    from qb_inputs.device import layer_for, upload
    d = upload(QI.LayerInputs(shape), "cuda:0")
    outs = []
    for env in ("0", "1"):
        monkeypatch.setenv("QBMOE_NO_GATHER", env)
        lay = layer_for(shape)
        lay.set_weights(**{k: v for k, v in d.items() if k != "x"})
        o = lay.forward(d["x"])
        torch.cuda.synchronize()
        assert lay.status() == 0
        outs.append(o.clone())
        lay.close()
    assert torch.equal(outs[0], outs[1])


@pytest.mark.parametrize("shape", [TC_PREFILL_LIKE], ids=lambda s: s.name)
def test_paired_m_tiles_match_single_ones(shape, monkeypatch):
    """Prefill-sized bf16 token tiles run the expert gate/up in units of two
    m-tiles that share each stage's token tile; QBMOE_NO_MPAIR=1 runs the
    same launch one m-tile at a time.  Every output element sums the same
    products in the same K order either way, so the outputs are identical."""
    from qb_inputs.device import layer_for, upload
    d = upload(QI.LayerInputs(shape), "cuda:0")
    outs = []
    for env in ("0", "1"):
        monkeypatch.setenv("QBMOE_NO_MPAIR", env)
        lay = layer_for(shape)
        lay.set_weights(**{k: v for k, v in d.items() if k != "x"})
        o = lay.forward(d["x"])
        torch.cuda.synchronize()
        assert lay.status() == 0
        outs.append(o.clone())
        lay.close()
    assert torch.equal(outs[0], outs[1])


def test_bf16_layers_run_on_tensor_cores(monkeypatch):
    from qb_inputs.device import layer_for
    lay = layer_for(SMALL_BF16)
    assert lay.uses_tensor_cores
    lay.close()
    lay = layer_for(QI.TINY_F32)
    assert not lay.uses_tensor_cores
    lay.close()
    monkeypatch.setenv("QBMOE_DISABLE_TC", "1")
    lay = layer_for(SMALL_BF16)
    assert not lay.uses_tensor_cores
    lay.close()


@pytest.mark.parametrize("shape", [SMALL_BF16, TC_PREFILL_LIKE], ids=lambda s: s.name)
def test_layer_cuda_core_path_matches_oracle(shape, monkeypatch):
    """The CUDA-core GEMMs (used for fp32 and untiled shapes) on bf16 shapes."""
    monkeypatch.setenv("QBMOE_DISABLE_TC", "1")
    compare_fed(shape)


@pytest.mark.parametrize("shape", [TC_MXFP4_DECODE_LIKE, TC_MXFP4_PREFILL_LIKE], ids=lambda s: s.name)
def test_mxfp4_decode_to_bf16_path_matches_oracle(shape, monkeypatch):
    """MXFP4 experts on the alternative tensor-core path: converter warps
    decode E2M1 x E8M0 to bf16 in SMEM for the kind::f16 MMA (bf16 tokens)."""
    monkeypatch.setenv("QBMOE_MX_DECODE", "1")
    compare_fed(shape)


def test_two_sm_kernel_on_prefill_tiles_matches_oracle(monkeypatch):
    """The prefill-size GEMMs on the 2-SM (cta_group::2) kernel, grouped ones
    included (opt-in): 256-row weight tiles across a CTA pair, 160- and
    256-row token tiles."""
    monkeypatch.setenv("QBMOE_ENABLE_2SM", "1")
    compare_fed(TC_PREFILL_LIKE)


def test_one_cta_kernel_on_dense_prefill_tiles_matches_oracle(monkeypatch):
    """The dense 256-row GEMMs on the one-CTA kernel (the 2-SM kernel runs
    them by default)."""
    monkeypatch.setenv("QBMOE_DISABLE_2SM", "1")
    compare_fed(TC_PREFILL_LIKE)


def test_bounded_wait_expires_and_context_stays_usable():
    """A tensor-core kernel whose accumulator hand-off never arrives gives up
    after its bounded wait, reports QBMOE_ETIMEOUT, and the context runs the
    next forward correctly."""
    import quantile_balanced_routing_gb300 as Q
    from qb_inputs.device import layer_for, upload
    from oracle import qb_oracle as O
    from layer_check import row_rel_err, to_f64
    shape = TC_DECODE_LIKE
    inp = QI.LayerInputs(shape)
    d = upload(inp, "cuda:0", drop_host=False)
    lay = layer_for(shape)
    assert lay.uses_tensor_cores
    lay.set_weights(**{k: v for k, v in d.items() if k != "x"})
    lay.set_wait_limit(200)
    lay.debug_stall(True)
    lay.forward(d["x"])
    assert lay.status() == Q.QBMOE_ETIMEOUT
    lay.debug_stall(False)
    lay.set_wait_limit(0)
    W = O.LayerWeights(inp)
    logits = O.router_logits(W.dense("x"), W.dense("w_router"), W.dense("router_offset"))
    out = lay.forward(d["x"], logits_in=torch.from_numpy(logits).cuda())
    assert lay.status() == 0
    ref = O.layer_forward(inp, logits=logits, weights=W)
    assert row_rel_err(to_f64(out), ref["out"]).max() <= 2e-2
    lay.close()


@pytest.mark.parametrize("shape", [QI.TINY_F32, RAGGED_F32, SMALL_BF16, TC_PREFILL_LIKE], ids=lambda s: s.name)
def test_layer_own_router(shape):
    compare_own_router(shape, min_agree=0.95)


@pytest.mark.parametrize("shape", [SMALL_BF16.with_(name="gs_bf16", T=150), RAGGED_F32.with_(name="gs_f32", qb_sweeps=2)],
                         ids=lambda s: s.name)
def test_layer_gauss_seidel_mode(shape):
    """qb_mode = QBMOE_QB_GAUSS_SEIDEL: the layer's QB sweeps are cyclic
    (each expert's step sees the latest biases); routing bit-exact against
    the oracle's cyclic sweep, outputs within tolerance."""
    compare_fed(shape, qb_mode="gauss_seidel")


@pytest.mark.parametrize("shape", [TC_DECODE_LIKE, TC_MXFP4_DECODE_LIKE], ids=lambda s: s.name)
def test_packed_weights_give_identical_outputs(shape):
    """qbmoe_pack_weights copies the weights into the context: the forward
    gives the same bits as with the caller's tensors, and keeps doing so once
    the caller's tensors are freed."""
    from qb_inputs.device import layer_for, upload
    d = upload(QI.LayerInputs(shape), "cuda:0")
    x = d.pop("x")
    a = layer_for(shape)
    a.set_weights(**d)
    want = a.forward(x).clone()
    b = layer_for(shape)
    b.pack_weights(**d)
    got1 = b.forward(x).clone()
    assert b.status() == 0 and a.status() == 0
    a.close()
    del d
    torch.cuda.empty_cache()
    junk = torch.full((64 << 20,), 7, dtype=torch.uint8, device="cuda")   # reuse the freed memory
    got2 = b.forward(x)
    assert b.status() == 0
    del junk
    assert torch.equal(got1.view(torch.int16), want.view(torch.int16))
    assert torch.equal(got2.view(torch.int16), want.view(torch.int16))
    b.close()


def test_pack_weights_rejects_a_nan_scale():
    """An E8M0 scale byte of 0xFF (NaN) is not a weight scale: packing fails
    with QBMOE_EINVAL and the context keeps its previous weights."""
    import quantile_balanced_routing_gb300 as Q
    from qb_inputs.device import layer_for, upload
    shape = TC_MXFP4_DECODE_LIKE
    d = upload(QI.LayerInputs(shape), "cuda:0")
    x = d.pop("x")
    lay = layer_for(shape)
    lay.pack_weights(**d)
    want = lay.forward(x).clone()
    bad = dict(d)
    bad["s_up"] = d["s_up"].clone()
    bad["s_up"].view(-1)[12345] = 0xFF
    with pytest.raises(Q.QbmoeError) as e:
        lay.pack_weights(**bad)
    assert e.value.code == Q.QBMOE_EINVAL
    got = lay.forward(x)
    assert lay.status() == 0
    assert torch.equal(got.view(torch.int16), want.view(torch.int16))
    lay.close()


def test_layer_reuses_context_and_bias_chains():
    """Two forwards in a row through one context; the second starts from the
    first's QB bias (the caller carries it between batches)."""
    from qb_inputs.device import layer_for, upload
    from oracle import qb_oracle as O
    shape = SMALL_BF16.with_(T=200)
    inp = QI.LayerInputs(shape)
    d = upload(inp, "cuda:0", drop_host=False)
    lay = layer_for(shape)
    lay.set_weights(**{k: v for k, v in d.items() if k != "x"})
    W = O.LayerWeights(inp)
    logits = O.router_logits(W.dense("x"), W.dense("w_router"), W.dense("router_offset"))
    lg = torch.from_numpy(logits).cuda()
    b = torch.zeros(shape.n, dtype=torch.float32, device="cuda")
    outs = []
    for _ in range(2):
        out, r = lay.forward(d["x"], logits_in=lg, bias_in=b, bias_out=b, want_routing=True)
        outs.append((out.float().cpu().numpy(), r["idx"].cpu().numpy()))
    assert lay.status() == 0
    b_ref = O.moe_route_qb(logits, None, shape.k, 1)[1]
    b_ref2 = O.moe_route_qb(logits, b_ref, shape.k, 1)[1]
    assert np.array_equal(b.cpu().numpy().view(np.uint32), b_ref2.view(np.uint32))
    lay.close()


def test_layer_launch_count_and_timing():
    from qb_inputs.device import layer_for, upload
    shape = QI.TINY_F32
    inp = QI.LayerInputs(shape)
    d = upload(inp, "cuda:0", drop_host=False)
    lay = layer_for(shape)
    lay.set_weights(**{k: v for k, v in d.items() if k != "x"})
    lay.set_timing(4)
    lay.forward(d["x"])
    assert lay.status() == 0
    st = lay.stage_times()
    assert len(st) >= 5 and all(ms >= 0 for _, ms in st)
    assert lay.last_launch_count() >= 8
    lay.close()


def test_forward_rejects_too_many_tokens():
    import quantile_balanced_routing_gb300 as Q
    from qb_inputs.device import layer_for, upload
    shape = QI.TINY_F32
    d = upload(QI.LayerInputs(shape), "cuda:0")
    lay = layer_for(shape, max_tokens=32)
    lay.set_weights(**{k: v for k, v in d.items() if k != "x"})
    with pytest.raises(Q.QbmoeError) as e:
        lay.forward(d["x"])
    assert e.value.code == Q.QBMOE_EWORKSPACE
    lay.close()


def _full_size_tokens(shape, n_prefill=512):
    """Tokens whose layer outputs a full-size test compares: every token of
    a decode batch (256), a seeded subset of 512 tokens of a prefill batch
    (routing is still checked on every token)."""
    if shape.T <= 256:
        return np.arange(shape.T)
    rng = np.random.default_rng(0)
    return np.sort(rng.choice(shape.T, n_prefill, replace=False))


@pytest.mark.slow
@pytest.mark.parametrize("shape", [QI.DECODE, QI.PREFILL, QI.PREFILL_MXFP4, QI.DECODE_MXFP4],
                         ids=lambda s: s.name)
def test_full_size_workload_sampled_tokens(shape):
    """The full K3-shape workloads (20 GB of bf16 or 5.2 GB of MXFP4 expert
    weights, up to 16384 tokens) in the launch configuration the bench times:
    routing of every token bit-exact against the oracle (fed the oracle's
    router logits), layer outputs within tolerance on all 256 decode tokens
    and on 512 seeded tokens of the 16384-token prefill batches."""
    err = compare_fed(shape, tokens=_full_size_tokens(shape))
    assert err.shape[0] == min(shape.T, 512)


@pytest.mark.slow
@pytest.mark.parametrize("shape", [QI.DECODE, QI.PREFILL], ids=lambda s: s.name)
def test_full_size_own_router(shape):
    """The layer's own router at full size: the K = 7168 router sub-GEMM of
    the fused x-side launch (2-SM tiles at prefill, as the bench runs it)
    and its logit + offset epilogue.  Scores within 1e-5 of the oracle's
    fp64 router, the GPU's routing self-consistent, at least 99% of tokens
    routed identically, and outputs of identically routed tokens within
    tolerance (32 seeded tokens)."""
    rng = np.random.default_rng(1)
    tokens = np.sort(rng.choice(shape.T, 32, replace=False))
    err, agree = compare_own_router(shape, tokens=tokens, min_agree=0.99)
    assert agree >= 0.99
