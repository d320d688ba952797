"""Pins of the CPU oracle against facts fixed outside it.

Each test checks the oracle against something other than itself: the pages'
printed constants, hand-worked examples (tests/golden), closed forms, brute
force over all assignments, LP duality, and textbook routines.  They are
chosen so that a plausible slip (a dropped term, a swapped sign, index or
operand) fails at least one of them; test_planted_mistakes_are_caught plants
such slips in copies of the oracle and checks that the pins notice.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

from oracle import qb_oracle as O

F32 = np.float32
GOLD = os.path.join(os.path.dirname(__file__), "golden")


def load(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def ulp_diff(a, b):
    ai = np.asarray(a, F32).view(np.int32).astype(np.int64)
    bi = np.asarray(b, F32).view(np.int32).astype(np.int64)
    return np.abs(ai - bi)


# --------------------------------------------------------------------------
# Router score
# --------------------------------------------------------------------------

def test_sigmoid_within_two_ulp_of_correctly_rounded():
    x = np.linspace(-80, 80, 1_600_001).astype(F32)
    exact = (1.0 / (1.0 + np.exp(-x.astype(np.float64)))).astype(F32)
    s = O.sigmoid_score(x)
    d = ulp_diff(s, exact)
    assert d.max() <= 2
    assert (d == 0).mean() > 0.75


def test_sigmoid_special_values_and_symmetry():
    assert O.sigmoid_score(np.array([0.0], F32))[0] == F32(0.5)
    x = np.random.default_rng(1).normal(0, 3, 100_000).astype(F32)
    s, sm = O.sigmoid_score(x), O.sigmoid_score(-x)
    assert np.max(np.abs(s.astype(np.float64) + sm - 1.0)) < 3e-7
    assert O.sigmoid_score(np.array([200.0], F32))[0] == F32(1.0)
    assert 0 < O.sigmoid_score(np.array([-200.0], F32))[0] < 1e-34


def test_sigmoid_monotone_on_dense_grid():
    x = np.sort(np.random.default_rng(2).uniform(-30, 30, 2_000_000).astype(F32))
    assert np.all(np.diff(O.sigmoid_score(x)) >= 0)


def test_router_logits_hand_worked():
    """x . W_r^T + o on a hand-worked dyadic example (tests/golden): the
    offset belongs to the expert (a column), the weights are [experts, width]."""
    g = load("router_logits_hand.json")
    x, w, o = (np.array(g[k], np.float64) for k in ("x", "w_router", "offset"))
    got = O.router_logits(x, w, o)
    assert got.shape == (x.shape[0], w.shape[0])
    assert got.dtype == F32
    assert np.array_equal(got, np.array(g["logits"], F32))
    assert np.array_equal(O.router_logits(x, w, None), np.array(g["dots"], F32))


def test_router_logits_equal_a_loop_dot_product_with_the_offset():
    """Per token and expert, a plain Python sum over the width plus the
    expert's offset (one fp32 rounding of the fp64 value)."""
    rng = np.random.default_rng(15)
    T, d, n = 5, 19, 7
    x, w, o = rng.normal(0, 1, (T, d)), rng.normal(0, 0.3, (n, d)), rng.normal(0, 1, n)
    got = O.router_logits(x, w, o)
    assert got.shape == (T, n)
    for t in range(T):
        for j in range(n):
            want = math.fsum(float(x[t, c]) * float(w[j, c]) for c in range(d)) + float(o[j])
            assert abs(float(got[t, j]) - want) <= 6e-8 * max(1.0, abs(want))


# --------------------------------------------------------------------------
# QB on hand-worked examples
# --------------------------------------------------------------------------

@pytest.mark.parametrize("name", ["qb_hand_k1.json", "qb_hand_k2.json"])
def test_hand_worked_qb(name):
    g = load(name)
    s = np.array(g["scores"], F32)
    k = g["k"]
    T, n = s.shape
    b0 = np.array(g["bias_in"], F32)
    assert list(O.qb_targets(T, n, k)) == g["targets"]
    _, _, loads0 = O.route_topk(s, b0, k)
    assert list(loads0) == g["loads_before"]
    m = O.qb_margins(s, b0, k)
    assert np.array_equal(m, np.array(g["margins"], F32))
    r = O.qb_targets(T, n, k)
    braw = np.array([O.qb_coordinate_bias(m[:, j], int(r[j])) for j in range(n)], F32)
    assert np.array_equal(braw, np.array(g["bias_raw"], F32))
    b = O.qb_sweep_jacobi(s, b0, k)
    assert np.array_equal(b, np.array(g["bias_out"], F32))
    assert np.array_equal(braw - b, np.full(n, F32(g["offset"])))
    idx, w, loads = O.route_topk(s, b, k)
    assert idx.tolist() == g["idx"]
    assert list(loads) == g["loads"]
    if "weights" in g:
        assert np.array_equal(w, np.array(g["weights"], F32))
    else:
        want = np.array([[F32(Fraction(p, q)) for p, q in row] for row in g["weights_fraction"]], F32)
        assert np.array_equal(w, want)


# --------------------------------------------------------------------------
# Ranking, margins and targets against their definitions
# --------------------------------------------------------------------------

def test_rank_is_textbook_sort_with_index_ties():
    rng = np.random.default_rng(3)
    for _ in range(20):
        T, n = 7, int(rng.integers(3, 40))
        v = (rng.integers(0, 6, (T, n)) / 8.0).astype(F32)   # many exact ties
        order = O.rank_experts(v)
        for t in range(T):
            want = sorted(range(n), key=lambda j: (-float(v[t, j]), j))
            assert order[t].tolist() == want


def test_margin_tau_equals_kth_best_among_other_experts():
    rng = np.random.default_rng(4)
    for trial in range(30):
        T, n = 5, int(rng.integers(3, 12))
        k = int(rng.integers(1, n))
        s = (rng.integers(0, 16, (T, n)) / 16.0).astype(F32)   # tie-heavy
        b = (rng.integers(-4, 5, n) / 32.0).astype(F32)
        m = O.qb_margins(s, b, k)
        v = O.biased(s, b)
        for t in range(T):
            for j in range(n):
                others = sorted((float(v[t, l]) for l in range(n) if l != j), reverse=True)
                tau = F32(others[k - 1])
                want = F32(s[t, j] - tau)
                assert m[t, j] == want and not (m[t, j] == 0 and np.signbit(m[t, j]))


def test_targets_sum_and_spread():
    for T, n, k in [(64, 32, 4), (4096, 896, 16), (256, 896, 16), (16384, 896, 16), (5, 7, 3), (1, 4, 3)]:
        r = O.qb_targets(T, n, k)
        assert r.sum() == T * k and r.max() - r.min() <= (1 if (T * k) % n else 0)
        assert r.min() == (T * k) // n


def test_printed_model_constants():
    c = load("k3_printed_constants.json")["constants"]
    import qb_inputs as Q
    for wl in (Q.DECODE, Q.PREFILL, Q.PREFILL_MXFP4):
        assert wl.n == c["n_routed_experts"]["value"] and wl.k == c["experts_per_token"]["value"]
        assert wl.d == c["model_width"]["value"] and wl.latent == c["latent_width"]["value"]
        assert wl.m_s == c["shared_intermediate"]["value"] == c["n_shared_experts"]["value"] * c["shared_intermediate"]["per_expert"]
    # the page prints 1.78% for 16/896 = 1.7857% (truncated, not rounded)
    assert abs(100 * 16 / 896 - c["activation_ratio_percent"]["value"]) < 0.01
    # every expert's target is within one token of T*k/n
    r = O.qb_targets(4096, 896, 16)
    assert np.all(np.abs(r - 4096 * 16 / 896) < 1)


# --------------------------------------------------------------------------
# QB properties
# --------------------------------------------------------------------------

def _scores(rng, T, n, skew=1.0):
    logits = rng.normal(0, 1, (T, n)) + rng.normal(0, skew, n)[None, :]
    return O.sigmoid_score(logits.astype(F32))


def test_coordinate_step_admits_exactly_the_target():
    """After expert j's Gauss-Seidel coordinate step, j's actual load (by the
    real top-k selection) equals r_j on tie-free data."""
    rng = np.random.default_rng(5)
    T, n, k = 200, 24, 3
    s = _scores(rng, T, n, 1.5)
    r = O.qb_targets(T, n, k)
    b = np.zeros(n, F32)
    for j in range(n):
        v = O.biased(s, b)
        v[:, j] = -np.inf
        tau = -np.sort(-v, axis=1)[:, k - 1]
        m = (s[:, j] - tau).astype(F32)
        b[j] = O.qb_coordinate_bias(m, int(r[j]))
        _, _, loads = O.route_topk(s, b, k)
        assert loads[j] == r[j]


def test_signsgd_direction():
    """The exact coordinate minimiser moves each unbalanced expert's bias in
    the direction of DeepSeek-V3's sign step (K3 page: SignSGD on the same
    dual gives that rule)."""
    rng = np.random.default_rng(6)
    T, n, k = 300, 40, 4
    s = _scores(rng, T, n, 1.0)
    b_old = rng.normal(0, 0.05, n).astype(F32)
    _, _, loads = O.route_topk(s, b_old, k)
    r = O.qb_targets(T, n, k)
    m = O.qb_margins(s, b_old, k)
    braw = np.array([O.qb_coordinate_bias(m[:, j], int(r[j])) for j in range(n)], F32)
    unbalanced = loads != r
    assert unbalanced.sum() > 10
    assert np.all(np.sign(braw - b_old)[unbalanced] == -np.sign(loads - r)[unbalanced])


def test_gauss_seidel_steps_never_raise_the_dual():
    rng = np.random.default_rng(7)
    T, n, k = 60, 10, 2
    s = _scores(rng, T, n, 1.0)
    r = O.qb_targets(T, n, k)
    b = np.zeros(n, F32)
    d_prev = O.dual_objective(s, b, k, r)
    for _ in range(3):
        for j in range(n):
            v = O.biased(s, b)
            v[:, j] = -np.inf
            tau = -np.sort(-v, axis=1)[:, k - 1]
            m = (s[:, j] - tau).astype(F32)
            b[j] = O.qb_coordinate_bias(m, int(r[j]))
            d = O.dual_objective(s, b, k, r)
            assert d <= d_prev + 1e-5
            d_prev = d


@pytest.mark.parametrize("T,n,k,seed", [(6, 4, 2, 0), (8, 4, 1, 1), (6, 4, 2, 2), (7, 5, 2, 3)])
def test_balanced_qb_assignment_is_the_brute_force_optimum(T, n, k, seed):
    """Once QB balances the loads, its assignment maximises the total score
    among all assignments with the same per-token k and per-expert loads
    (LP duality; the K3 page frames QB as the balanced assignment problem's
    dual).  Checked against exhaustive search."""
    rng = np.random.default_rng(seed)
    s = _scores(rng, T, n, 1.0)
    r = O.qb_targets(T, n, k)
    b = np.zeros(n, F32)
    for _ in range(200):
        b = O.qb_sweep_gauss_seidel(s, b, k)
        idx, _, loads = O.route_topk(s, b, k)
        if np.array_equal(loads, r):
            break
    assert np.array_equal(loads, r)
    best, _ = O.brute_force_assignment(s, k, r)
    got = float(sum(float(s[t, j]) for t in range(T) for j in idx[t]))
    assert got == pytest.approx(best, abs=1e-9)


def test_one_sweep_improves_balance_on_skewed_scores():
    rng = np.random.default_rng(8)
    T, n, k = 2048, 128, 8
    s = _scores(rng, T, n, 2.0 ** 0.5)
    _, _, l0 = O.route_topk(s, np.zeros(n, F32), k)
    b = O.qb_sweep_jacobi(s, np.zeros(n, F32), k)
    _, _, l1 = O.route_topk(s, b, k)
    mean = T * k / n
    assert l1.max() / mean < 0.5 * (l0.max() / mean)
    assert l1.max() / mean < 1.5


def test_offset_is_zero_mean_and_selection_invariant_to_a_common_shift():
    rng = np.random.default_rng(9)
    T, n, k = 50, 20, 3
    s = (rng.integers(1, 256, (T, n)) / 256.0).astype(F32)      # dyadic: shifts are exact
    b = (rng.integers(-32, 33, n) / 256.0).astype(F32)
    out = O.common_offset(b)
    assert abs(math.fsum(out.astype(np.float64))) < n * 1e-7
    for c in (F32(0.5), F32(-0.25), F32(1.0 / 64)):
        i1, w1, _ = O.route_topk(s, b, k)
        i2, w2, _ = O.route_topk(s, (b + c).astype(F32), k)
        assert np.array_equal(i1, i2) and np.array_equal(w1, w2)


def test_weights_are_raw_scores_renormalised_not_biased_scores():
    rng = np.random.default_rng(10)
    T, n, k = 100, 30, 4
    s = _scores(rng, T, n)
    b = rng.normal(0, 0.2, n).astype(F32)
    idx, w, _ = O.route_topk(s, b, k)
    sel = s[np.arange(T)[:, None], idx].astype(np.float64)
    want = sel / sel.sum(axis=1, keepdims=True)
    assert np.max(np.abs(w - want)) < 4e-7
    assert np.max(np.abs(w.astype(np.float64).sum(axis=1) - 1)) < k * 1.2e-7
    # the bias changed the selection but not the weights' formula
    idx0, _, _ = O.route_topk(s, np.zeros(n, F32), k)
    assert not np.array_equal(idx, idx0)


def test_frozen_bias_is_passed_through():
    rng = np.random.default_rng(11)
    logits = rng.normal(0, 1, (40, 16)).astype(F32)
    b = rng.normal(0, 0.1, 16).astype(F32)
    _, bout, idx, _, _ = O.moe_route_qb(logits, b, 2, qb_sweeps=0)
    assert np.array_equal(bout, b)
    assert np.array_equal(idx, O.route_topk(O.sigmoid_score(logits), b, 2)[0])


def test_degenerate_targets():
    # r_j = 0 admits nobody; r_j >= T admits everybody
    m = np.array([0.5, -0.25, 0.125], F32)
    b0 = O.qb_coordinate_bias(m, 0)
    assert np.sum(m + b0 > 0) == 0
    bT = O.qb_coordinate_bias(m, 3)
    assert np.sum(m + bT > 0) == 3


# --------------------------------------------------------------------------
# DeepSeek-V3's sign rule (the comparator) and token-sharded QB
# --------------------------------------------------------------------------

def test_signsgd_hand_worked():
    g = load("signsgd_hand_k1.json")
    s = np.array(g["scores"], F32)
    k = g["k"]
    assert list(O.route_topk(s, np.zeros(3, F32), k)[2]) == g["loads_at_zero_bias"]
    assert list(O.qb_targets(*s.shape, k)) == g["targets"]
    for run in g["runs"]:
        b = np.zeros(3, F32)
        for st in run["steps"]:
            b = O.signsgd_bias_step(s, b, k, run["gamma"])
            assert np.array_equal(b, np.array(st["bias"], F32)), run["gamma"]
            idx, _, loads = O.route_topk(s, b, k)
            assert idx.tolist() == st["idx"] and list(loads) == st["loads"]


def test_signsgd_moves_like_the_exact_coordinate_step():
    """SignSGD on the dual and QB's exact coordinate minimiser move every
    unbalanced expert's bias the same way (the page: both work on one dual;
    QB jumps to the minimiser, the sign rule takes a fixed step)."""
    rng = np.random.default_rng(17)
    T, n, k = 400, 32, 4
    s = _scores(rng, T, n, 1.0)
    b_old = rng.normal(0, 0.05, n).astype(F32)
    _, _, loads = O.route_topk(s, b_old, k)
    r = O.qb_targets(T, n, k)
    m = O.qb_margins(s, b_old, k)
    braw = np.array([O.qb_coordinate_bias(m[:, j], int(r[j])) for j in range(n)], F32)
    b_sign = O.signsgd_bias_step(s, b_old, k, 1.0 / 64)
    unbalanced = loads != r
    assert unbalanced.sum() > 10
    assert np.array_equal(np.sign(b_sign - b_old)[unbalanced], np.sign(braw - b_old)[unbalanced])
    assert np.array_equal(b_sign[~unbalanced], b_old[~unbalanced])


def test_one_qb_sweep_balances_better_than_sign_steps():
    """On skewed scores one QB sweep leaves a lower max/mean load than the
    same number of sign steps of any of a range of step sizes."""
    rng = np.random.default_rng(18)
    T, n, k = 2048, 64, 4
    s = _scores(rng, T, n, 2.0 ** 0.5)
    mean = T * k / n
    b = O.qb_sweep_jacobi(s, np.zeros(n, F32), k)
    qb = O.route_topk(s, b, k)[2].max() / mean
    for gamma in (1e-3, 1e-2, 1e-1):
        bs = O.signsgd_bias_step(s, np.zeros(n, F32), k, gamma)
        assert O.route_topk(s, bs, k)[2].max() / mean > qb


def test_descending_keys_order_and_round_trip():
    m = np.array([0.0, -0.0, 1.5, -1.5, 1e-40, -1e-40, 3.4e38, -3.4e38, 0.25, -0.25], F32)
    m[m == 0] = F32(0.0)
    key = O.descending_keys(m)
    assert np.array_equal(O.margin_of_key(key).view(np.uint32), m.view(np.uint32))
    order = np.argsort(key, kind="stable")
    assert np.all(np.diff(m[order].astype(np.float64)) <= 0)     # ascending key = descending margin


@pytest.mark.parametrize("split", [[300], [100, 200], [1, 150, 149], [37, 0, 263]])
def test_histogram_selection_is_an_exact_order_statistic(split):
    """Four exchanged 8-bit digit histograms pin down the exact r-th and
    (r+1)-th largest margin of every expert, whatever the token split:
    checked against a textbook sort of the whole column (ties included)."""
    rng = np.random.default_rng(sum(split) + len(split))
    n, T = 6, sum(split)
    m = (rng.integers(-40, 40, (T, n)) / 64.0).astype(F32)   # many exact ties
    m[m == 0] = F32(0.0)
    keys = O.descending_keys(m).T.copy()
    r = np.array([0, 1, 17, 150, T - 1, T])
    ranks = O.selection_ranks(T, r)
    prefix = np.zeros((n, 2), np.uint32)
    bounds = np.cumsum([0] + split)
    for p in range(O.HIST_PASSES):
        parts = [O.shard_digit_histogram(keys[:, a:b], prefix, p) for a, b in zip(bounds[:-1], bounds[1:])]
        prefix, ranks = O.advance_selection(np.sum(parts, axis=0), prefix, ranks, p)
    for j in range(n):
        desc = np.sort(m[:, j].astype(np.float64))[::-1]
        want = O.selection_ranks(T, r)[j]
        assert O.margin_of_key(prefix[j, 0]) == desc[want[0] - 1]
        assert O.margin_of_key(prefix[j, 1]) == desc[want[1] - 1]


@pytest.mark.parametrize("name,split", [("qb_hand_k1.json", [1, 3]), ("qb_hand_k2.json", [2, 2]),
                                         ("qb_hand_k2.json", [3, 1])])
def test_sharded_sweep_reproduces_the_hand_worked_biases(name, split):
    g = load(name)
    s = np.array(g["scores"], F32)
    b0 = np.array(g["bias_in"], F32)
    shards = np.split(s, np.cumsum(split)[:-1])
    b = O.qb_sweep_jacobi_sharded(shards, b0, g["k"])
    assert np.array_equal(b, np.array(g["bias_out"], F32))


def test_sharded_sweep_equals_whole_batch_sweep():
    rng = np.random.default_rng(19)
    T, n, k = 500, 40, 5
    s = _scores(rng, T, n, 1.5)
    s[::7] = (np.round(s[::7] * 32) / 32).astype(F32)      # some tied scores
    b0 = rng.normal(0, 0.02, n).astype(F32)
    want = O.qb_sweep_jacobi(s, b0, k)
    for split in ([250, 250], [1, 499], [123, 77, 300]):
        shards = np.split(s, np.cumsum(split)[:-1])
        assert np.array_equal(O.qb_sweep_jacobi_sharded(shards, b0, k), want)


# --------------------------------------------------------------------------
# SiTU-GLU, RMSNorm, shared expert, MXFP4
# --------------------------------------------------------------------------

def test_situ_bound_and_limits():
    g = np.concatenate([np.linspace(-60, 60, 4001), [-1e30, 1e30]])
    u = np.concatenate([np.linspace(-400, 400, 4001), [-1e30, 1e30]])
    G, U = np.meshgrid(g, u)
    out = O.situ_glu(G, U)
    assert np.all(np.abs(out) <= 100.0)                      # printed bound beta1*beta2
    sup = 4.0 / (1.0 + math.exp(-4.0)) * 25.0                # closed-form supremum
    assert np.max(np.abs(out)) == pytest.approx(sup, rel=1e-12)
    assert O.situ_glu(-1e30, 1e30) == pytest.approx(-4.0 / (1.0 + math.exp(4.0)) * 25.0, rel=1e-12)
    assert np.array_equal(O.situ_glu(G, -U), -out)           # odd in the up branch


def test_situ_matches_swiglu_near_zero():
    rng = np.random.default_rng(12)
    g = rng.uniform(-0.1, 0.1, 10000)
    u = rng.uniform(-0.1, 0.1, 10000)
    swiglu = g / (1.0 + np.exp(-g)) * u
    rel = np.abs(O.situ_glu(g, u) - swiglu) / np.maximum(np.abs(swiglu), 1e-300)
    assert rel.max() < 2e-3


def test_rmsnorm_scale_invariance_and_unit_rms():
    rng = np.random.default_rng(13)
    y = rng.normal(0, 3, (10, 64))
    gamma = np.ones(64)
    z = O.rmsnorm(y, gamma, 0.0)
    assert np.allclose(np.sqrt(np.mean(z * z, axis=1)), 1.0, rtol=1e-12)
    assert np.allclose(O.rmsnorm(7.5 * y, gamma, 1e-6), O.rmsnorm(y, gamma, 1e-6), rtol=1e-6)
    g2 = rng.normal(1, 0.1, 64)
    assert np.allclose(O.rmsnorm(y, g2, 0.0), z * g2, rtol=1e-12)


def test_merged_shared_expert_is_sum_of_two_halves():
    rng = np.random.default_rng(14)
    d, half = 48, 24
    x = rng.normal(0, 1, (5, d))
    wg, wu = rng.normal(0, 0.2, (2 * half, d)), rng.normal(0, 0.2, (2 * half, d))
    wo = rng.normal(0, 0.2, (d, 2 * half))
    merged = O.shared_mlp(x, wg, wu, wo, "f32")
    parts = (O.shared_mlp(x, wg[:half], wu[:half], wo[:, :half], "f32")
             + O.shared_mlp(x, wg[half:], wu[half:], wo[:, half:], "f32"))
    assert np.allclose(merged, parts, rtol=1e-12, atol=1e-12)


def test_shared_expert_is_odd_in_its_up_branch_only():
    """SiTU-GLU's up factor b = 25 tanh(u / 25) is odd and its gate factor
    a sigma(a) is not, so negating the up weights negates the shared
    expert's output exactly, while negating the gate weights does not (the
    gate and up matrices are not interchangeable)."""
    rng = np.random.default_rng(16)
    d, m_s = 24, 16
    x = rng.normal(0, 1, (6, d))
    wg, wu, wo = rng.normal(0, 0.5, (m_s, d)), rng.normal(0, 0.5, (m_s, d)), rng.normal(0, 0.3, (d, m_s))
    base = O.shared_mlp(x, wg, wu, wo, "f32")
    assert np.array_equal(O.shared_mlp(x, wg, -wu, wo, "f32"), -base)
    flipped_gate = O.shared_mlp(x, -wg, wu, wo, "f32")
    assert np.max(np.abs(flipped_gate + base)) > 0.1 * np.max(np.abs(base))
    # a saturated gate (a -> beta1 = 4) leaves 4 sigma(4) times the capped up branch
    big = O.shared_mlp(x, wg * 1e6, wu, np.eye(m_s, m_s)[:, :m_s], "f32")
    up = x @ wu.T
    sgn = np.sign(x @ wg.T)
    a = 4.0 * sgn
    want = O.round_to(a / (1.0 + np.exp(-a)) * 25.0 * np.tanh(up / 25.0), "f32")
    assert np.allclose(big, want, rtol=1e-6, atol=1e-6)


def test_mxfp4_decode_against_ocp_table():
    # OCP MX v1.0 E2M1: codes 0..7 -> 0, 0.5, 1, 1.5, 2, 3, 4, 6; bit 3 = sign
    table = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0]
    codes = np.arange(16, dtype=np.uint8)
    packed = np.zeros((1, 16), np.uint8)
    packed[0, :8] = codes[0::2] | (codes[1::2] << 4)
    packed[0, 8:] = packed[0, :8]
    for e8, mult in ((127, 1.0), (128, 2.0), (120, 2.0 ** -7), (0, 2.0 ** -127), (254, 2.0 ** 127)):
        got = O.mxfp4_decode(packed, np.array([[e8]], np.uint8))
        assert got[0, :16].tolist() == [t * mult for t in table]
    with pytest.raises(ValueError):
        O.mxfp4_decode(packed, np.array([[255]], np.uint8))


def test_mxfp4_roundtrip_of_the_input_quantiser_is_close():
    import qb_inputs as Q
    bits = Q.normal_bf16(0, 99, (8, 256), 0.05)
    packed, scales = Q.quantize_mxfp4(bits)
    back = O.mxfp4_decode(packed, scales)
    ref = Q.bf16_bits_to_f32(bits).astype(np.float64)
    blocks = np.abs(ref).reshape(8, 8, 32).max(axis=2)
    err = np.abs(back - ref).reshape(8, 8, 32).max(axis=2)
    assert np.all(err <= 0.25 * blocks + 1e-12)    # half a step at the top binade, saturation at 6


def test_round_to_bf16_is_nearest_even():
    vals = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 1.0 + 2 ** -9, -2.5, 3.0 + 2 ** -20])
    want = [1.0, 1.0, 1.0 + 2 ** -6, 1.0, -2.5, 3.0]
    assert O.round_to(vals, "bf16").tolist() == want


# --------------------------------------------------------------------------
# Whole layer: reductions to simpler computations
# --------------------------------------------------------------------------

def _tiny(**kw):
    import qb_inputs as Q
    return Q.LayerInputs(Q.TINY_F32.with_(**kw))


def test_layer_with_identical_experts_is_a_dense_chain():
    """With every expert equal, routing cannot matter (the weights sum to 1),
    so the routed branch is one dense MLP chain computed without routing."""
    import qb_inputs as Q
    inp = _tiny(T=24, m_s=32)
    W = O.LayerWeights(inp)
    e0 = {nm: W.expert(nm, 0) for nm in ("w_gate", "w_up", "w_out")}
    W.expert = lambda nm, e: e0[nm]
    res = O.layer_forward(inp, weights=W)
    X = W.dense("x")
    h = O.round_to(X @ W.dense("w_down").T, "f32")
    act = O.round_to(O.situ_glu(h @ e0["w_gate"].T, h @ e0["w_up"].T), "f32")
    e = O.round_to(act @ e0["w_out"].T, "f32")
    wsum = res["w"].astype(np.float64).sum(axis=1, keepdims=True)
    z = O.round_to(O.rmsnorm(e * wsum, W.dense("gamma"), 1e-6), "f32")
    shared = O.shared_mlp(X, W.dense("w_shared_gate"), W.dense("w_shared_up"), W.dense("w_shared_out"), "f32")
    out = O.round_to(z @ W.dense("w_proj_up").T + shared, "f32")
    assert np.allclose(res["out"], out, rtol=1e-5, atol=1e-6)


def test_routed_branch_is_insensitive_to_expert_output_scale():
    inp = _tiny(T=16)
    W = O.LayerWeights(inp)
    base = O.layer_forward(inp, weights=W)["out"]
    W2 = O.LayerWeights(inp)
    orig = W2.expert
    W2.expert = lambda nm, e: orig(nm, e) * (8.0 if nm == "w_out" else 1.0)
    scaled = O.layer_forward(inp, weights=W2)["out"]
    assert np.allclose(scaled, base, rtol=2e-5, atol=2e-6)


@pytest.mark.parametrize("m_s", [0, 8], ids=["routed_only", "with_shared_expert"])
def test_layer_matches_per_token_loop_on_tiny_case(m_s):
    """Independent per-token, per-route restatement with python loops; the
    shared expert's gate (w_shared_gate, capped at 4, through the sigmoid)
    and up (w_shared_up, capped at 25) branches are named explicitly."""
    inp = _tiny(T=6, n=8, k=2, d=32, latent=16, m=8, m_s=m_s)
    W = O.LayerWeights(inp)
    res = O.layer_forward(inp, weights=W)
    X = W.dense("x")
    for t in range(6):
        shared = [0.0] * 32
        if m_s:
            sg, su, so = W.dense("w_shared_gate"), W.dense("w_shared_up"), W.dense("w_shared_out")
            act_s = []
            for q in range(m_s):
                gate = sum(X[t, c] * sg[q, c] for c in range(32))
                up = sum(X[t, c] * su[q, c] for c in range(32))
                a = 4 * math.tanh(gate / 4)
                act_s.append(float(np.float32(a / (1 + math.exp(-a)) * 25 * math.tanh(up / 25))))
            shared = [sum(act_s[q] * so[c, q] for q in range(m_s)) for c in range(32)]
        h = [float(np.float32(sum(X[t, c] * W.dense("w_down")[r, c] for c in range(32)))) for r in range(16)]
        y = [0.0] * 16
        for i in range(2):
            e = int(res["idx"][t, i])
            wg, wu, wo = W.expert("w_gate", e), W.expert("w_up", e), W.expert("w_out", e)
            act = []
            for q in range(8):
                g = sum(h[c] * wg[q, c] for c in range(16))
                u = sum(h[c] * wu[q, c] for c in range(16))
                a = 4 * math.tanh(g / 4)
                act.append(float(np.float32(a / (1 + math.exp(-a)) * 25 * math.tanh(u / 25))))
            for r in range(16):
                y[r] += float(res["w"][t, i]) * float(np.float32(sum(act[q] * wo[r, q] for q in range(8))))
        rms = math.sqrt(sum(v * v for v in y) / 16 + 1e-6)
        z = [float(np.float32(y[r] / rms * W.dense("gamma")[r])) for r in range(16)]
        for c in range(32):
            o = float(np.float32(sum(z[r] * W.dense("w_proj_up")[c, r] for r in range(16)) + shared[c]))
            assert res["out"][t, c] == pytest.approx(o, rel=1e-5, abs=1e-6)


# --------------------------------------------------------------------------
# The pins catch plausible slips planted in the oracle (CPU only)
# --------------------------------------------------------------------------

def _margins_vs_biased_score(s, b, k):
    return (_ORIG["qb_margins"](s, b, k) + np.asarray(b, F32)[None, :]).astype(F32)


def _quantile_off_by_one(m, r):
    M = np.sort(np.asarray(m, F32))[::-1]
    if 2 <= r < len(M):
        return F32(-((M[r - 2] + M[r - 1]) * F32(0.5)))
    return _ORIG["qb_coordinate_bias"](m, r)


def _weights_from_biased(s, b, k):
    idx, _, loads = _ORIG["route_topk"](s, b, k)
    v = O.biased(s, b)
    sel = v[np.arange(v.shape[0])[:, None], idx].astype(np.float64)
    return idx, (sel / sel.sum(axis=1, keepdims=True)).astype(F32), loads


def _offset_added(b):
    out = _ORIG["common_offset"](b)
    return (2 * np.asarray(b, F32) - out).astype(F32)


def _situ_betas_swapped(g, u, beta1=4.0, beta2=25.0):
    return _ORIG["situ_glu"](g, u, beta2, beta1)


def _rank_high_index_first(v):
    n = v.shape[1]
    return (n - 1 - np.argsort(-v[:, ::-1], axis=1, kind="stable"))


def _tau_ignores_membership(s, b, k):
    v = O.biased(s, b)
    order = O.rank_experts(v)
    vk = v[np.arange(v.shape[0]), order[:, k - 1]]
    m = (np.asarray(s, F32) - vk[:, None]).astype(F32)
    m[m == 0] = F32(0)
    return m


def _rms_without_sqrt(y, gamma, eps):
    y = np.asarray(y, np.float64)
    return y / (np.mean(y * y, axis=-1, keepdims=True) + eps) * gamma


def _sigmoid_wrong_sign(x):
    return _ORIG["sigmoid_score"](-np.asarray(x, F32))


def _logits_without_offset(x, w_router, offset):
    return _ORIG["router_logits"](x, w_router, None)


def _logits_offset_subtracted(x, w_router, offset):
    return _ORIG["router_logits"](x, w_router, None if offset is None else -np.asarray(offset))


def _shared_gate_up_swapped(x, w_gate, w_up, w_out, dtype):
    return _ORIG["shared_mlp"](x, w_up, w_gate, w_out, dtype)


def _sign_step_reversed(s, b, k, gamma):
    return _ORIG["signsgd_bias_step"](s, b, k, -gamma)


def _digit_off_by_one(hist, prefix, rank, n_pass):
    shift = 32 - O.HIST_DIGIT_BITS * (n_pass + 1)
    prefix = np.array(prefix, dtype=np.uint32, copy=True)
    rank = np.array(rank, dtype=np.int64, copy=True)
    for j in range(hist.shape[0]):
        for a in range(2):
            c = np.cumsum(hist[j, a])
            d = min(int(np.searchsorted(c, rank[j, a], side="right")), 255)
            rank[j, a] -= int(c[d - 1]) if d > 0 else 0
            prefix[j, a] = np.uint32(prefix[j, a] | np.uint32(d << shift))
    return prefix, rank


def _histogram_ignores_prefix(keys_shard, prefix, n_pass):
    return _ORIG["shard_digit_histogram"](keys_shard, np.zeros_like(prefix), n_pass)


_ORIG = {nm: getattr(O, nm) for nm in ("qb_margins", "qb_coordinate_bias", "route_topk", "common_offset",
                                       "situ_glu", "rank_experts", "rmsnorm", "sigmoid_score", "router_logits",
                                       "shared_mlp", "signsgd_bias_step", "advance_selection",
                                       "shard_digit_histogram")}

_PLANTS = [
    ("qb_margins", _margins_vs_biased_score, [test_margin_tau_equals_kth_best_among_other_experts]),
    ("qb_margins", _tau_ignores_membership, [test_margin_tau_equals_kth_best_among_other_experts]),
    ("qb_coordinate_bias", _quantile_off_by_one, [lambda: test_hand_worked_qb("qb_hand_k1.json")]),
    ("route_topk", _weights_from_biased, [test_weights_are_raw_scores_renormalised_not_biased_scores]),
    ("common_offset", _offset_added, [lambda: test_hand_worked_qb("qb_hand_k1.json")]),
    ("situ_glu", _situ_betas_swapped, [test_situ_bound_and_limits]),
    ("rank_experts", _rank_high_index_first, [test_rank_is_textbook_sort_with_index_ties]),
    ("rmsnorm", _rms_without_sqrt, [test_rmsnorm_scale_invariance_and_unit_rms]),
    ("sigmoid_score", _sigmoid_wrong_sign, [test_sigmoid_special_values_and_symmetry]),
    ("router_logits", _logits_without_offset,
     [test_router_logits_hand_worked, test_router_logits_equal_a_loop_dot_product_with_the_offset]),
    ("router_logits", _logits_offset_subtracted, [test_router_logits_hand_worked]),
    ("shared_mlp", _shared_gate_up_swapped,
     [test_shared_expert_is_odd_in_its_up_branch_only,
      lambda: test_layer_matches_per_token_loop_on_tiny_case(8)]),
    ("signsgd_bias_step", _sign_step_reversed,
     [test_signsgd_hand_worked, test_signsgd_moves_like_the_exact_coordinate_step]),
    ("advance_selection", _digit_off_by_one, [lambda: test_histogram_selection_is_an_exact_order_statistic([300]),
                                              lambda: test_sharded_sweep_reproduces_the_hand_worked_biases(
                                                  "qb_hand_k1.json", [1, 3])]),
    ("shard_digit_histogram", _histogram_ignores_prefix,
     [lambda: test_histogram_selection_is_an_exact_order_statistic([100, 200])]),
]


@pytest.mark.parametrize("i", range(len(_PLANTS)), ids=[f"{p[0]}:{p[1].__name__}" for p in _PLANTS])
def test_planted_mistakes_are_caught(i, monkeypatch):
    name, bad, pins = _PLANTS[i]
    monkeypatch.setattr(O, name, bad)
    for pin in pins:
        with pytest.raises(AssertionError):
            pin()


def test_expert_slices_match_the_whole_tensor_at_large_indices():
    """Expert e's slice drawn alone equals rows e of the whole tensor (the
    offset arithmetic must not overflow 32 bits for 896 experts x 3.7M)."""
    import qb_inputs as QI
    shape = QI.DECODE
    inp = QI.LayerInputs(shape)
    per = shape.m * shape.latent
    e = np.int32(895)
    sl = inp.expert_raw("w_gate", e)
    first = QI.normal_bf16(shape.seed, QI.TID["w_gate"], (4,), float(np.float32(1 / np.sqrt(shape.latent))),
                           offset=895 * per)
    assert np.array_equal(sl.ravel()[:4], first)
    assert 895 * per > 2 ** 31
