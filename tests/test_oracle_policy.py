"""Pins of the elementwise PPO / TIS / mismatch oracle.

* The masked-fraction-vs-eps curve ("IPO (INTELLECT Policy Optimization)", "Choosing
  eps") and the IcePop band fraction on the 1.8M-token synthetic replay are checked
  against the closed form of the generating distribution (1-D Gauss-Hermite over the
  inference logit, the Gaussian trainer noise integrated exactly), within 4 binomial
  standard deviations.
* mis_kl and mis_k3_kl ("Rollout Correction Methods", "Mismatch Metrics") against 2-D
  quadrature of the same distribution, within a 4-sigma CLT bound.
* PPO clip / dual-clip special cases with hand-worked values ("10-KL-clip-entropy",
  section 2; "Rollout Correction Methods", standard and decoupled PPO).
* Central finite differences of the per-token losses with respect to lp_theta.
"""
import math

import numpy as np
import pytest
from scipy.special import expit, logit, log_expit
from scipy.stats import norm

import oracle
import workloads
from oracle import PolicyParams, policy_loss_elementwise

X_MEAN, X_STD, NOISE = -1.0, 2.5, 0.3


def _hermite(n=160):
    x, w = np.polynomial.hermite_e.hermegauss(n)     # weight exp(-x^2/2)
    return x, w / math.sqrt(2 * math.pi)


def _curve_closed_form(eps):
    """P(|sigmoid(x + e) - sigmoid(x)| > eps), x ~ N(-1, 2.5), e ~ N(0, 0.3)."""
    nodes, wts = _hermite()
    tot = 0.0
    for s, w in zip(nodes, wts):
        x = X_MEAN + X_STD * s
        p = expit(x)
        pr = 0.0
        if p + eps < 1:
            pr += norm.sf((logit(p + eps) - x) / NOISE)
        if p - eps > 0:
            pr += norm.cdf((logit(p - eps) - x) / NOISE)
        tot += w * pr
    return tot


def _icepop_closed_form(lo, hi):
    """P(sigmoid(x + e) / sigmoid(x) outside [lo, hi])."""
    nodes, wts = _hermite()
    tot = 0.0
    for s, w in zip(nodes, wts):
        x = X_MEAN + X_STD * s
        p = expit(x)
        pr = norm.cdf((logit(lo * p) - x) / NOISE)
        if hi * p < 1:
            pr += norm.sf((logit(hi * p) - x) / NOISE)
        tot += w * pr
    return tot


def _moment_2d(f):
    nodes, wts = _hermite(96)
    tot = tot2 = 0.0
    for s, w in zip(nodes, wts):
        x = X_MEAN + X_STD * s
        for s2, w2 in zip(nodes, wts):
            v = f(x, NOISE * s2)
            tot += w * w2 * v
            tot2 += w * w2 * v * v
    return tot, math.sqrt(max(tot2 - tot * tot, 0.0))


@pytest.fixture(scope="module")
def c5():
    case = workloads.make_policy_case()
    out = policy_loss_elementwise(case.lp_theta, case.lp_old, case.lp_samp, case.adv, case.mask,
                                  PolicyParams())
    return case, out


def test_c5_shape(c5):
    case, out = c5
    assert int(case.mask.sum()) == 1_800_000 == out["metrics"]["n_valid"]
    assert case.seq_lens.min() >= 1 and case.seq_lens.max() <= 4096


def test_ipo_curve_matches_closed_form(c5):
    case, out = c5
    n = out["metrics"]["n_valid"]
    for eps, cnt in zip(oracle.IPO_CURVE_EPS, out["metrics"]["ipo_curve"]):
        pc = _curve_closed_form(eps)
        sigma = math.sqrt(max(pc * (1 - pc), 1.0 / n) / n)
        assert abs(cnt / n - pc) <= 4 * sigma + 2e-6, (eps, cnt / n, pc)
    curve = out["metrics"]["ipo_curve"]
    assert all(a >= b for a, b in zip(curve, curve[1:]))      # monotone in eps


def test_icepop_band_matches_closed_form(c5):
    case, out = c5
    n = out["metrics"]["n_valid"]
    pc = _icepop_closed_form(0.5, 2.0)
    frac = (out["metrics"]["icepop_low"] + out["metrics"]["icepop_high"]) / n
    assert abs(frac - pc) <= 4 * math.sqrt(pc * (1 - pc) / n)


def test_mismatch_kl_and_k3_match_quadrature(c5):
    case, out = c5
    n = out["metrics"]["n_valid"]
    # d = log pi_train - log pi_rollout with pi_train = sigmoid(x + e), pi_rollout = sigmoid(x)
    kl_mean, kl_sd = _moment_2d(lambda x, e: log_expit(x) - log_expit(x + e))
    k3_mean, k3_sd = _moment_2d(lambda x, e: math.exp(log_expit(x + e) - log_expit(x))
                                - (log_expit(x + e) - log_expit(x)) - 1.0)
    assert abs(out["metrics"]["mis_kl"] / n - kl_mean) <= 4 * kl_sd / math.sqrt(n) + 1e-6
    assert abs(out["metrics"]["k3"] / n - k3_mean) <= 4 * k3_sd / math.sqrt(n) + 1e-6


def _one(lt, lo, ls, A, pp=None):
    out = policy_loss_elementwise(np.array([lt]), np.array([lo]), np.array([ls]), np.array([A]),
                                  np.array([1], dtype=np.uint8), pp or PolicyParams())
    return {k: (v[0] if isinstance(v, np.ndarray) else v) for k, v in out.items()}


def test_ppo_clip_and_dual_clip_worked_values():
    # r = 1: the surrogate is -A, gradient -A, nothing clipped
    o = _one(-1.0, -1.0, -1.0, 0.5)
    assert abs(o["loss_ppo"] + 0.5) < 1e-15 and abs(o["grad_ppo"] + 0.5) < 1e-15
    assert o["metrics"]["n_clip"] == 0
    # A > 0, r = 2: clipped at 1.2 -> -1.2 A, no gradient, counted as clipped
    o = _one(math.log(2.0), 0.0, 0.0, 1.0)
    assert abs(o["loss_ppo"] + 1.2) < 1e-12 and o["grad_ppo"] == 0.0
    assert o["metrics"]["n_clip"] == 1 and o["metrics"]["n_clip_lower"] == 0
    # A < 0, r = 5: max(5|A|, 1.2|A|) = 5|A| is capped by the dual clip at 3|A|
    o = _one(math.log(5.0), 0.0, 0.0, -2.0)
    assert abs(o["loss_ppo"] - 6.0) < 1e-12 and o["grad_ppo"] == 0.0
    assert o["metrics"]["n_clip_lower"] == 1
    # A < 0, r = 0.5: max(0.5|A|, 0.8|A|) = 0.8|A|, the clipped branch, no gradient
    o = _one(math.log(0.5), 0.0, 0.0, -1.0)
    assert abs(o["loss_ppo"] - 0.8) < 1e-12 and o["grad_ppo"] == 0.0
    # A < 0, r = 1.1 inside the band: -A r, gradient -A r
    o = _one(math.log(1.1), 0.0, 0.0, -1.0)
    assert abs(o["loss_ppo"] - 1.1) < 1e-12 and abs(o["grad_ppo"] - 1.1) < 1e-12


def test_decoupled_reduces_to_clipped_surrogate_without_mismatch():
    """pi_old = pi_rollout: the TIS weight is 1 and the decoupled loss is the clipped
    surrogate (no dual clip in the decoupled formula)."""
    rng = np.random.default_rng(3)
    lt, lo, A = rng.normal(-1, 0.3, 50), rng.normal(-1, 0.3, 50), rng.normal(0, 1, 50)
    out = policy_loss_elementwise(lt, lo, lo, A, np.ones(50, np.uint8), PolicyParams(clip_ratio_c=1e9))
    np.testing.assert_allclose(out["loss_dec"], out["loss_ppo"], rtol=1e-14)
    # TIS weight truncation: pi_old / pi_rollout = e^2 > 2 is truncated to 2
    o = _one(-1.0, -1.0, -3.0, 1.0)
    assert abs(o["loss_dec"] - 2.0 * o["loss_ppo"]) < 1e-12 and o["metrics"]["n_tis_trunc"] == 1


def test_policy_gradients_by_finite_differences():
    rng = np.random.default_rng(4)
    T = 400
    lt = rng.normal(-1, 0.5, T)
    lo = lt + rng.normal(0, 0.3, T)
    ls = lo + rng.normal(0, 0.5, T)
    A = rng.normal(0, 1, T)
    pp = PolicyParams()
    out = policy_loss_elementwise(lt, lo, ls, A, np.ones(T, np.uint8), pp)
    h = 1e-7
    up = policy_loss_elementwise(lt + h, lo, ls, A, np.ones(T, np.uint8), pp)
    dn = policy_loss_elementwise(lt - h, lo, ls, A, np.ones(T, np.uint8), pp)
    r = np.exp(lt - lo)
    away = (np.abs(r - 0.8) > 1e-4) & (np.abs(r - 1.2) > 1e-4) & (np.abs(r * np.abs(A) - 3 * np.abs(A)) > 1e-4)
    for k in ("ppo", "dec"):
        fd = (up["loss_" + k] - dn["loss_" + k]) / (2 * h)
        np.testing.assert_allclose(fd[away], out["grad_" + k][away], rtol=1e-5, atol=1e-7)


def test_masked_tokens_contribute_nothing():
    rng = np.random.default_rng(5)
    T = 100
    m = (rng.random(T) < 0.6).astype(np.uint8)
    args = (rng.normal(-1, 0.3, T), rng.normal(-1, 0.3, T), rng.normal(-1, 0.3, T), rng.normal(0, 1, T))
    a = policy_loss_elementwise(*args, m, PolicyParams())
    b = policy_loss_elementwise(*(x[m == 1] for x in args), np.ones(int(m.sum()), np.uint8), PolicyParams())
    assert a["metrics"]["n_valid"] == b["metrics"]["n_valid"]
    assert abs(a["metrics"]["loss_ppo"] - b["metrics"]["loss_ppo"]) < 1e-12
    assert np.all(a["loss_ppo"][m == 0] == 0)


def test_nonfinite_padding_changes_nothing():
    """NaN / inf in padded slots: every output and metric equals the run with finite
    padding (padding does not count at all)."""
    rng = np.random.default_rng(6)
    T = 200
    m = (rng.random(T) < 0.5).astype(np.uint8)
    args = [rng.normal(-1, 0.3, T), rng.normal(-1, 0.3, T), rng.normal(-1, 0.3, T), rng.normal(0, 1, T)]
    a = policy_loss_elementwise(*args, m, PolicyParams())
    bad = [x.copy() for x in args]
    for x in bad:
        x[m == 0] = rng.choice([np.nan, np.inf, -np.inf], int((m == 0).sum()))
    with np.errstate(invalid="ignore", over="ignore"):
        b = policy_loss_elementwise(*bad, m, PolicyParams())
    for k in ("loss_ppo", "loss_dec", "grad_ppo", "grad_dec"):
        assert np.array_equal(a[k], b[k]), k
    assert a["metrics"] == b["metrics"]
