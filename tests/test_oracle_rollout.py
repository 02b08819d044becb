"""Pins of the rollout-correction oracle ("Rollout Correction Methods": "Importance
Sampling", "Rejection Sampling", "Veto Mechanism", "Config keys", "Mismatch Metrics").

Each check is fixed by the page's definitions or by mathematics, not by re-typing the
oracle's formulas:
  * the sequence weight equals the product of the token probability ratios and the
    geometric weight their geometric mean, computed from probabilities (not log-ratios);
  * sequence-level rejection uses the arithmetic mean of the token weights: a sequence
    whose arithmetic mean is out of bounds while its geometric mean is inside (AM >= GM)
    is rejected at one level and kept at the other;
  * the veto drops a whole sequence for one catastrophic token, with RS off;
  * truncate / clip / mask bound the weights as named; batch normalisation gives mean 1;
  * chi^2 estimated under the rollout policy converges to the exact chi^2 divergence of
    two small categorical distributions, and mis_kl / k3 to their closed forms;
  * a constant log-prob log(1/V) has perplexity V; identical policies give zero mismatch.
"""
import math

import numpy as np
import pytest

from oracle.rollout import (LEVEL_GEOMETRIC, LEVEL_SEQUENCE, LEVEL_TOKEN, TIS_CLIP, TIS_MASK, TIS_TRUNCATE,
                            RolloutParams, rollout_correction, rollout_metrics_named)


def _probs_case():
    # two sequences of probabilities under the two policies
    p_train = [np.array([0.5, 0.2, 0.9]), np.array([0.05, 0.6])]
    p_roll = [np.array([0.25, 0.4, 0.3]), np.array([0.5, 0.6])]
    lt = np.log(np.concatenate(p_train))
    lr = np.log(np.concatenate(p_roll))
    off = np.array([0, 3, 5])
    return p_train, p_roll, lt, lr, off


def test_token_sequence_geometric_weights_from_probabilities():
    p_train, p_roll, lt, lr, off = _probs_case()
    m = np.ones(5, np.uint8)
    big = RolloutParams(tis_lower_bound=0.0, tis_upper_bound=1e9)        # no bounding
    tok = rollout_correction(lt, lr, m, off, big)["weights"]
    np.testing.assert_allclose(tok, np.concatenate([a / b for a, b in zip(p_train, p_roll)]), rtol=1e-12)
    seq = rollout_correction(lt, lr, m, off, RolloutParams(tis_lower_bound=0.0, tis_upper_bound=1e9,
                                                           tis_level=LEVEL_SEQUENCE))["weights"]
    prod = [np.prod(a / b) for a, b in zip(p_train, p_roll)]             # 2 * 0.5 * 3 = 3, 0.1 * 1
    np.testing.assert_allclose(prod, [3.0, 0.1], rtol=1e-12)
    np.testing.assert_allclose(seq, [3.0] * 3 + [0.1] * 2, rtol=1e-12)
    geo = rollout_correction(lt, lr, m, off, RolloutParams(tis_lower_bound=0.0, tis_upper_bound=1e9,
                                                           tis_level=LEVEL_GEOMETRIC))["weights"]
    np.testing.assert_allclose(geo, [3.0 ** (1 / 3)] * 3 + [0.1 ** 0.5] * 2, rtol=1e-12)


def test_masked_tokens_leave_the_sequence_statistics():
    p_train, p_roll, lt, lr, off = _probs_case()
    m = np.array([1, 0, 1, 1, 1], np.uint8)       # drop the 0.2 / 0.4 token
    r = rollout_correction(lt, lr, m, off, RolloutParams(tis_lower_bound=0.0, tis_upper_bound=1e9,
                                                         tis_level=LEVEL_SEQUENCE))
    np.testing.assert_allclose(r["weights"], [6.0, 0.0, 6.0, 0.1, 0.1], rtol=1e-12)   # 2 * 3
    assert r["keep"].tolist() == [1, 0, 1, 1, 1]


@pytest.mark.parametrize("mode", [TIS_TRUNCATE, TIS_CLIP, TIS_MASK])
def test_bounding_modes(mode):
    w = np.array([0.1, 0.5, 1.0, 2.0, 3.0])
    lt, lr = np.log(w), np.zeros(5)
    r = rollout_correction(lt, lr, np.ones(5, np.uint8), [0, 5],
                           RolloutParams(tis_mode=mode, tis_lower_bound=0.5, tis_upper_bound=2.0))
    want = {TIS_TRUNCATE: [0.1, 0.5, 1.0, 2.0, 2.0],      # upper bound only
            TIS_CLIP: [0.5, 0.5, 1.0, 2.0, 2.0],          # both bounds
            TIS_MASK: [0.0, 0.5, 1.0, 2.0, 0.0]}[mode]    # zero outside, bounds kept
    np.testing.assert_allclose(r["weights"], want, rtol=1e-12)
    mt = r["metrics"]
    assert (mt["n_tis_low"], mt["n_tis_high"]) == (1, 1)
    named = rollout_metrics_named(mt, RolloutParams(tis_mode=mode))
    key = {TIS_TRUNCATE: "tis_truncate_fraction", TIS_CLIP: "tis_clip_fraction_high",
           TIS_MASK: "tis_mask_fraction_high"}[mode]
    assert named[key] == pytest.approx(0.2)


def test_rs_sequence_uses_the_arithmetic_mean_geometric_the_geometric():
    # token weights 4 and 0.25: arithmetic mean 2.125, geometric mean 1
    lt = np.log([4.0, 0.25, 1.0, 1.0])
    lr = np.zeros(4)
    off = [0, 2, 4]
    m = np.ones(4, np.uint8)
    seq = rollout_correction(lt, lr, m, off, RolloutParams(use_rs=True, rs_level=LEVEL_SEQUENCE,
                                                           rs_lower_bound=0.5, rs_upper_bound=2.0))
    geo = rollout_correction(lt, lr, m, off, RolloutParams(use_rs=True, rs_level=LEVEL_GEOMETRIC,
                                                           rs_lower_bound=0.5, rs_upper_bound=2.0))
    tok = rollout_correction(lt, lr, m, off, RolloutParams(use_rs=True, rs_level=LEVEL_TOKEN,
                                                           rs_lower_bound=0.5, rs_upper_bound=2.0))
    assert seq["keep"].tolist() == [0, 0, 1, 1]
    assert seq["metrics"]["n_rs_high"] == 2 and seq["metrics"]["n_rs_low"] == 0
    assert geo["keep"].tolist() == [1, 1, 1, 1]
    assert tok["keep"].tolist() == [0, 0, 1, 1]
    assert (tok["metrics"]["n_rs_low"], tok["metrics"]["n_rs_high"]) == (1, 1)
    # unset RS bounds fall back to the tis bounds ("Config keys")
    fb = rollout_correction(lt, lr, m, off, RolloutParams(use_rs=True, rs_level=LEVEL_SEQUENCE,
                                                          tis_lower_bound=0.5, tis_upper_bound=2.2))
    assert fb["keep"].tolist() == [1, 1, 1, 1]


def test_veto_drops_the_whole_sequence_without_rs():
    lt = np.log([1e-7, 0.5, 0.9, 0.8, 0.7])
    lr = np.log([0.5, 0.5, 0.9, 0.8, 0.7])        # token 0: ratio 2e-7 < 1e-6
    off = [0, 2, 5]
    r = rollout_correction(lt, lr, np.ones(5, np.uint8), off, RolloutParams(rs_veto_threshold=1e-6))
    assert r["keep"].tolist() == [0, 0, 1, 1, 1]
    assert r["weights"][:2].tolist() == [0.0, 0.0]
    mt = r["metrics"]
    assert (mt["n_cat_tokens"], mt["n_cat_seqs"], mt["n_kept"]) == (1, 1, 3)
    nm = rollout_metrics_named(mt, RolloutParams(rs_veto_threshold=1e-6))
    assert nm["rs_catastrophic_token_fraction"] == pytest.approx(0.2)
    assert nm["rs_catastrophic_seq_fraction"] == pytest.approx(0.5)


def test_threshold_equality_is_kept():
    lt = np.log([0.5, 2.0])
    r = rollout_correction(lt, np.zeros(2), np.ones(2, np.uint8), [0, 2],
                           RolloutParams(tis_mode=TIS_MASK, use_rs=True, rs_lower_bound=0.5, rs_upper_bound=2.0))
    assert r["keep"].tolist() == [1, 1]
    np.testing.assert_allclose(r["weights"], [0.5, 2.0], rtol=1e-15)


def test_batch_normalisation_gives_mean_one():
    rng = np.random.default_rng(3)
    T = 1000
    lt = rng.normal(-1, 0.5, T)
    lr = lt + rng.normal(0, 0.4, T)
    m = (rng.random(T) < 0.9).astype(np.uint8)
    off = np.arange(0, T + 1, 100)
    rp = RolloutParams(tis_mode=TIS_CLIP, tis_batch_normalize=True, use_rs=True, rs_lower_bound=0.3,
                       rs_upper_bound=3.0)
    r = rollout_correction(lt, lr, m, off, rp)
    k = r["keep"].astype(bool)
    assert k.sum() > 500
    assert r["weights"][k].mean() == pytest.approx(1.0, rel=1e-12)
    assert np.all(r["weights"][~k] == 0)
    nm = rollout_metrics_named(r["metrics"], rp)
    assert nm["is_ratio_mean_final"] == pytest.approx(1.0, rel=1e-12)
    assert nm["batch_norm_factor"] == pytest.approx(1.0 / nm["is_ratio_mean_after_tis_rs"], rel=1e-12)


def test_identical_policies_have_no_mismatch():
    rng = np.random.default_rng(4)
    lp = np.log(rng.random(300) * 0.9 + 0.05)
    off = [0, 100, 250, 300]
    r = rollout_correction(lp, lp, np.ones(300, np.uint8), off,
                           RolloutParams(use_rs=True, rs_level=LEVEL_GEOMETRIC, rs_veto_threshold=1e-4,
                                         tis_batch_normalize=True))
    assert np.all(r["weights"] == 1.0) and np.all(r["keep"] == 1)
    nm = rollout_metrics_named(r["metrics"], RolloutParams(rs_veto_threshold=1e-4))
    for k in ("kl", "k3_kl", "log_ppl_diff", "log_ppl_abs_diff", "chi2_token", "chi2_seq",
              "train_rollout_logprob_abs_diff", "tis_truncate_fraction", "rs_catastrophic_token_fraction"):
        assert nm[k] == pytest.approx(0.0, abs=1e-12), k
    assert nm["ppl_ratio"] == pytest.approx(1.0)
    assert nm["training_log_ppl"] == pytest.approx(nm["rollout_log_ppl"])


def test_perplexity_of_a_uniform_policy_is_its_vocabulary():
    V = 37
    lp = np.full(50, -math.log(V))
    r = rollout_correction(lp, lp, np.ones(50, np.uint8), [0, 20, 50], RolloutParams())
    nm = rollout_metrics_named(r["metrics"], RolloutParams())
    assert nm["training_ppl"] == pytest.approx(V, rel=1e-12)
    assert nm["rollout_log_ppl"] == pytest.approx(math.log(V), rel=1e-12)


def test_chi2_kl_k3_converge_to_the_divergences_of_two_categoricals():
    """Tokens drawn from the rollout distribution q; the estimators converge to
    chi2(p||q) = sum p^2/q - 1, KL(q||p) = sum q log(q/p) (mis_kl = E_q[log q - log p]),
    and E_q[p/q - log(p/q) - 1] = KL(q||p) (k3 is unbiased for it)."""
    p = np.array([0.1, 0.2, 0.3, 0.4])
    q = np.array([0.25, 0.25, 0.25, 0.25])
    rng = np.random.default_rng(5)
    n = 400_000
    v = rng.choice(4, size=n, p=q)
    lt, lr = np.log(p[v]), np.log(q[v])
    r = rollout_correction(lt, lr, np.ones(n, np.uint8), [0, n], RolloutParams())
    nm = rollout_metrics_named(r["metrics"], RolloutParams())
    chi2 = float((p ** 2 / q).sum() - 1.0)
    kl_qp = float((q * np.log(q / p)).sum())
    w = p[v] / q[v]
    sd = lambda x: float(np.std(x)) / math.sqrt(n)
    assert abs(nm["chi2_token"] - chi2) <= 5 * sd(w ** 2)
    assert abs(nm["kl"] - kl_qp) <= 5 * sd(np.log(w))
    assert abs(nm["k3_kl"] - kl_qp) <= 5 * sd(w - np.log(w) - 1)
    assert nm["train_rollout_logprob_abs_diff"] == pytest.approx(float((q * np.abs(np.log(p / q))).sum()), abs=0.01)


def test_log_perplexity_is_a_mean_over_sequences():
    """Reading RC3: per-sequence log-perplexity averaged over sequences, not a token mean.
    Sequence A: 10 tokens at log p = -1; sequence B: 30 tokens at -3 (rollout side equal
    to training, shifted by -0.5 on B only)."""
    lt = np.array([-1.0] * 10 + [-3.0] * 30)
    lr = np.array([-1.0] * 10 + [-3.5] * 30)
    r = rollout_correction(lt, lr, np.ones(40, np.uint8), [0, 10, 40], RolloutParams())
    nm = rollout_metrics_named(r["metrics"], RolloutParams())
    assert nm["training_log_ppl"] == pytest.approx((1.0 + 3.0) / 2)          # token mean would be 2.5
    assert nm["rollout_log_ppl"] == pytest.approx((1.0 + 3.5) / 2)
    assert nm["log_ppl_diff"] == pytest.approx((0.0 - 0.5) / 2)
    assert nm["log_ppl_abs_diff"] == pytest.approx(0.5 / 2)
    assert nm["ppl_ratio"] == pytest.approx((1.0 + math.exp(-0.5)) / 2)
    assert nm["training_ppl"] == pytest.approx(math.exp(2.0))
    # chi2_seq with the sequence weights exp(0) and exp(30 * 0.5)
    assert nm["chi2_seq"] == pytest.approx((1.0 + math.exp(30.0)) / 2 - 1.0)


def test_nonfinite_padding_changes_nothing():
    """NaN / inf in masked slots: weights, keep flags and metrics equal the run with
    finite values there (padding does not count at all)."""
    rng = np.random.default_rng(14)
    lens = [7, 0, 12, 5]
    T = sum(lens)
    off = np.concatenate([[0], np.cumsum(lens)])
    lr = np.log(rng.random(T) * 0.9 + 0.05)
    lt = np.minimum(lr + rng.normal(0, 0.3, T), 0.0)
    m = (rng.random(T) < 0.6).astype(np.uint8)
    bad_t, bad_r = lt.copy(), lr.copy()
    pad = m == 0
    bad_t[pad] = rng.choice([np.nan, np.inf, -np.inf], int(pad.sum()))
    bad_r[pad] = rng.choice([np.nan, np.inf, -np.inf], int(pad.sum()))
    for rp in (RolloutParams(tis_mode=TIS_CLIP, tis_lower_bound=0.5, tis_upper_bound=2.0, tis_level=LEVEL_SEQUENCE,
                             tis_batch_normalize=True, use_rs=True, rs_level=LEVEL_GEOMETRIC, rs_lower_bound=0.5,
                             rs_upper_bound=2.0, rs_veto_threshold=1e-3),
               RolloutParams(tis_lower_bound=0.5, tis_upper_bound=2.0, use_rs=True, rs_level=LEVEL_TOKEN,
                             rs_lower_bound=0.5, rs_upper_bound=2.0)):
        a = rollout_correction(lt, lr, m, off, rp)
        with np.errstate(invalid="ignore", over="ignore"):
            b = rollout_correction(bad_t, bad_r, m, off, rp)
        np.testing.assert_array_equal(a["weights"], b["weights"])
        np.testing.assert_array_equal(a["keep"], b["keep"])
        assert a["metrics"] == b["metrics"]


def test_named_metrics_follow_the_emitted_when_column():
    """"IS/RS Correction Metrics", "Emitted when": the weight statistics need use_tis, a
    mode's fractions that mode, the RS fractions use_rs, the catastrophic fractions a veto
    threshold; the monitoring metrics are always there."""
    rng = np.random.default_rng(6)
    lr = np.log(rng.random(200) * 0.9 + 0.05)
    lt = np.minimum(lr + rng.normal(0, 0.3, 200), 0.0)
    m = np.ones(200, np.uint8)
    always = {"training_log_ppl", "training_ppl", "rollout_log_ppl", "rollout_ppl", "kl", "k3_kl", "log_ppl_diff",
              "log_ppl_abs_diff", "ppl_ratio", "chi2_token", "chi2_seq", "train_rollout_logprob_abs_diff"}
    weights = {"tis_weight_before_bound", "tis_weight_after_bound", "is_ratio_mean_after_tis_rs",
               "batch_norm_factor", "is_ratio_mean_final", "is_ratio_min_final", "is_ratio_max_final"}
    for rp, extra in ((RolloutParams(use_tis=False), set()),
                      (RolloutParams(), weights | {"tis_truncate_fraction"}),
                      (RolloutParams(tis_mode=TIS_CLIP, use_rs=True), weights | {
                          "tis_clip_fraction_low", "tis_clip_fraction_high", "rs_mask_fraction_low",
                          "rs_mask_fraction_high"}),
                      (RolloutParams(tis_mode=TIS_MASK, use_tis=False, rs_veto_threshold=1e-3), {
                          "rs_catastrophic_token_fraction", "rs_catastrophic_seq_fraction"}),
                      (RolloutParams(tis_mode=TIS_MASK, rs_veto_threshold=1e-3), weights | {
                          "tis_mask_fraction_low", "tis_mask_fraction_high", "rs_catastrophic_token_fraction",
                          "rs_catastrophic_seq_fraction"})):
        r = rollout_correction(lt, lr, m, [0, 80, 200], rp)
        assert set(rollout_metrics_named(r["metrics"], rp)) == always | extra
