"""Pins of the fp64 head oracle against what the pages and the mathematics fix.

Each test names the fact it pins.  None of them re-types the oracle's own formula:
they use worked examples from the pages (tests/golden/), closed forms (softmax
cross-entropy gradient, KL, entropy through scipy), brute-force enumeration on tiny
vocabularies, CLT bounds for the K-draw estimator, and central finite differences.
"""
import math
import os

import numpy as np
import pytest
import scipy.special
import scipy.stats

import oracle
from oracle import HeadParams, LOSS_IPO, LOSS_ICEPOP, LOSS_REINFORCE, KL_EXACT, KL_K1

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    rows = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            parts = line.split()
            rows[parts[0]] = parts[1:]
    return rows


def identity_case(z_rows, labels, label_logq, supports, replayed, adv=None, age=None,
                  loss_mask=None):
    """Inputs with W = I (H = V) so hidden rows are the logits and dX is dloss/dz."""
    z_rows = np.asarray(z_rows, dtype=np.float64)
    N, V = z_rows.shape
    offsets = np.zeros(N + 1, dtype=np.int64)
    ids, logq = [], []
    for t, (i, lq) in enumerate(supports):
        ids.extend(i)
        logq.extend(lq)
        offsets[t + 1] = offsets[t] + len(i)
    return dict(hidden=z_rows, W=np.eye(V), labels=np.asarray(labels, dtype=np.int64),
                label_logq=np.asarray(label_logq, dtype=np.float64),
                adv=np.ones(N) if adv is None else np.asarray(adv, dtype=np.float64),
                loss_mask=np.ones(N, dtype=np.uint8) if loss_mask is None else np.asarray(loss_mask),
                age=np.zeros(N, dtype=np.int64) if age is None else np.asarray(age),
                replayed=np.asarray(replayed, dtype=np.uint8), offsets=offsets,
                ids=np.asarray(ids, dtype=np.int64), logq=np.asarray(logq, dtype=np.float64))


# --------------------------------------------------------------------------------------
# "IPO (INTELLECT Policy Optimization)", "Masking by Probability, Not Ratio"
# --------------------------------------------------------------------------------------
def _two_outcome_mask(pi_infer, pi_train, p):
    """Vocabulary of two outcomes {token, rest}; trainer logits give pi_train."""
    z = np.log([[pi_train, 1.0 - pi_train]])
    inp = identity_case(z, [0], [math.log(pi_infer)],
                        [([1], [math.log(1.0 - pi_infer)])], [0])
    out = oracle.head_forward(inp, p)
    return int(out["mask_label"][0]), out


def test_two_outcome_examples_from_page():
    g = _golden("two_outcome_examples.txt")
    rare = [float(x) for x in g["rare_token"]]
    likely = [float(x) for x in g["likely_token"]]
    eps = float(_golden("default_constants.txt")["ipo_eps"][0])
    ipo = HeadParams(loss_type=LOSS_IPO, eps=eps)
    # IPO eps=0.3 keeps the rare token (moved 0.05) and masks the likely one (moved 0.70)
    assert _two_outcome_mask(rare[0], rare[1], ipo)[0] == 1
    assert _two_outcome_mask(likely[0], likely[1], ipo)[0] == 0
    # the printed ratios and moved masses
    assert round(rare[1] / rare[0]) == rare[2]
    assert round(likely[1] / likely[0], 2) == likely[2]
    assert abs(abs(rare[1] - rare[0]) - rare[3]) < 1e-12
    assert abs(abs(likely[1] - likely[0]) - likely[3]) < 1e-12
    # a ratio band with beta < 6 masks the rare token, the configs' [0.5, 2] included
    for beta in (2.0, 3.0, 5.9):
        icepop = HeadParams(loss_type=LOSS_ICEPOP, icepop_low=0.5, icepop_high=beta)
        m, out = _two_outcome_mask(rare[0], rare[1], icepop)
        assert m == 0
        assert out["metrics"]["masked_high"] == 1
    # the page's "IcePop keeps it" for 0.90 -> 0.20 needs alpha <= 0.222 (reading R16)
    wide = HeadParams(loss_type=LOSS_ICEPOP, icepop_low=0.2, icepop_high=5.0)
    assert _two_outcome_mask(likely[0], likely[1], wide)[0] == 1
    narrow = HeadParams(loss_type=LOSS_ICEPOP, icepop_low=0.5, icepop_high=2.0)
    m, out = _two_outcome_mask(likely[0], likely[1], narrow)
    assert m == 0 and out["metrics"]["masked_low"] == 1


@pytest.mark.parametrize("pi_infer,pi_train", [(0.01, 0.06), (0.9, 0.2), (0.4, 0.7), (0.3, 0.3)])
def test_ipo_mask_is_two_outcome_total_variation(pi_infer, pi_train):
    """|pi_train - pi_infer| is the TV distance on the split {token, rest}."""
    tv = 0.5 * (abs(pi_train - pi_infer) + abs((1 - pi_train) - (1 - pi_infer)))
    for eps in (0.05, 0.2, 0.3, 0.5):
        m, _ = _two_outcome_mask(pi_infer, pi_train, HeadParams(loss_type=LOSS_IPO, eps=eps))
        assert m == (1 if tv <= eps + 1e-12 else 0)


def test_default_constants():
    d = _golden("default_constants.txt")
    hp = HeadParams()
    pp = oracle.PolicyParams()
    assert hp.eps == float(d["ipo_eps"][0])
    assert hp.kl_coeff == float(d["kl_coeff"][0])
    assert pp.clip_ratio_low == float(d["clip_ratio_low"][0])
    assert pp.clip_ratio_high == float(d["clip_ratio_high"][0])
    assert pp.clip_ratio_c == float(d["clip_ratio_c"][0])


# --------------------------------------------------------------------------------------
# Textbook special cases
# --------------------------------------------------------------------------------------
def _softmax(z):
    return scipy.special.softmax(np.asarray(z, dtype=np.float64))


@pytest.mark.parametrize("loss_type", [LOSS_IPO, LOSS_ICEPOP, LOSS_REINFORCE])
def test_q_equals_p_full_replay(loss_type):
    """q = p, replay over the whole vocabulary: w = 1, nothing masked, no mismatch,
    support mass 1, KL 0, and loss = -A (log p(a) + H(p))."""
    rng = np.random.default_rng(1)
    V = 16
    z = rng.normal(0, 1.5, size=(3, V))
    labels = [2, 7, 15]
    adv = [0.7, -1.3, 2.0]
    sup = []
    lab_lq = []
    for t in range(3):
        p = _softmax(z[t])
        sup.append((list(range(V)), list(np.log(p))))
        lab_lq.append(math.log(p[labels[t]]))
    inp = identity_case(z, labels, lab_lq, sup, [1, 1, 1], adv=adv)
    hp = HeadParams(loss_type=loss_type, kl_coeff=0.3, kl_estimator=KL_EXACT)
    out = oracle.head_forward(inp, hp)
    met = out["metrics"]
    assert met["masked"] == 0 and abs(met["mismatch_kl"]) < 1e-12
    assert abs(met["support_mass"] - 3.0) < 1e-12
    assert abs(met["kl"]) < 1e-12 and abs(met["mask_tv"]) < 1e-12
    assert np.all(out["mask_support"] == 1)
    for t in range(3):
        p = _softmax(z[t])
        expect = -adv[t] * (math.log(p[labels[t]]) + scipy.stats.entropy(p))
        assert abs(out["loss"][t] - expect) < 1e-12
        assert abs(out["entropy"][t] - scipy.stats.entropy(p)) < 1e-12


def test_reinforce_full_replay_gradient_is_label_minus_q():
    """reinforce, replay with S = V, u = q: d loss / d z = -adv_tau A (onehot(a) - q),
    independent of the trainer's p."""
    rng = np.random.default_rng(2)
    V = 12
    z = rng.normal(0, 1, size=(2, V))
    qz = rng.normal(0, 1, size=(2, V))
    labels = [3, 9]
    adv = [1.5, -0.4]
    sup, lab_lq = [], []
    for t in range(2):
        q = _softmax(qz[t])
        sup.append((list(range(V)), list(np.log(q))))
        lab_lq.append(math.log(q[labels[t]]))
    inp = identity_case(z, labels, lab_lq, sup, [1, 1], adv=adv)
    hp = HeadParams(loss_type=LOSS_REINFORCE, adv_tau=0.8)
    dX, dW = oracle.head_backward(inp, hp, np.ones(2))
    for t in range(2):
        q = _softmax(qz[t])
        onehot = np.eye(V)[labels[t]]
        np.testing.assert_allclose(dX[t], -0.8 * adv[t] * (onehot - q), atol=1e-13)


@pytest.mark.parametrize("estimator", [KL_EXACT, KL_K1])
def test_kl_full_replay_matches_dense_kl_and_xent_gradient(estimator):
    """Exact KL over S = V is KL(q||p) and its gradient is p - q (the softmax
    cross-entropy gradient); k1 is log q(a) - log p(a) with gradient p - onehot(a)."""
    rng = np.random.default_rng(3)
    V = 10
    z = rng.normal(0, 1, size=(2, V))
    qz = rng.normal(0, 1, size=(2, V))
    labels = [1, 6]
    sup, lab_lq = [], []
    for t in range(2):
        q = _softmax(qz[t])
        sup.append((list(range(V)), list(np.log(q))))
        lab_lq.append(math.log(q[labels[t]]))
    inp = identity_case(z, labels, lab_lq, sup, [1, 1], adv=[0.0, 0.0])
    beta = 0.25
    hp = HeadParams(loss_type=LOSS_IPO, kl_coeff=beta, kl_estimator=estimator)
    out = oracle.head_forward(inp, hp)
    dX, _ = oracle.head_backward(inp, hp, np.ones(2))
    for t in range(2):
        p, q = _softmax(z[t]), _softmax(qz[t])
        if estimator == KL_EXACT:
            assert abs(out["kl"][t] - scipy.stats.entropy(q, p)) < 1e-12
            np.testing.assert_allclose(dX[t], beta * (p - q), atol=1e-13)
        else:
            assert abs(out["kl"][t] - (math.log(q[labels[t]]) - math.log(p[labels[t]]))) < 1e-12
            np.testing.assert_allclose(dX[t], beta * (p - np.eye(V)[labels[t]]), atol=1e-13)
        assert abs(out["loss"][t] - beta * out["kl"][t]) < 1e-14


def test_gradient_lies_on_label_and_support_when_sparse_eligible():
    """reinforce without KL on K draws, and any loss on a replayed support: the logit
    gradient is zero off label + support (pull request #4233, sparse LM-head backward)."""
    rng = np.random.default_rng(4)
    V, K = 40, 6
    z = rng.normal(0, 1, size=(2, V))
    q0 = _softmax(z[0] + rng.normal(0, 0.3, V))
    draws = sorted(rng.choice(V, size=K, replace=True, p=q0))
    S = sorted(rng.choice(V, size=9, replace=False))
    qS = _softmax(z[1, S] + rng.normal(0, 0.3, len(S)))
    lab1 = S[4]
    inp = identity_case(z, [5, lab1], [math.log(q0[5]), math.log(qS[4])],
                        [(draws, list(np.log(q0[draws]))), (S, list(np.log(qS)))], [0, 1],
                        adv=[1.2, -0.7])
    for hp in (HeadParams(loss_type=LOSS_REINFORCE),):
        dX, _ = oracle.head_backward(inp, hp, np.ones(2))
        off0 = np.setdiff1d(np.arange(V), np.r_[draws, 5])
        assert np.max(np.abs(dX[0, off0])) < 1e-15
    for hp in (HeadParams(loss_type=LOSS_IPO, kl_coeff=0.1), HeadParams(loss_type=LOSS_ICEPOP)):
        dX, _ = oracle.head_backward(inp, hp, np.ones(2))
        off1 = np.setdiff1d(np.arange(V), S)
        assert np.max(np.abs(dX[1, off1])) == 0.0
        # not eligible on the untruncated row: the dense softmax term is there
        assert np.min(np.abs(dX[0])) > 0.0 or hp.loss_type == LOSS_REINFORCE


# --------------------------------------------------------------------------------------
# Brute force on tiny vocabularies
# --------------------------------------------------------------------------------------
def _keep_w(P, q, hp):
    """Independent restatement of the three weights for enumerated (P, q) pairs."""
    if hp.loss_type == LOSS_REINFORCE:
        return 1.0
    r = P / q
    if hp.loss_type == LOSS_IPO:
        return min(r, hp.max_importance_ratio) if abs(P - q) <= hp.eps else 0.0
    return r if hp.icepop_low <= r <= hp.icepop_high else 0.0


@pytest.mark.parametrize("loss_type", [LOSS_IPO, LOSS_ICEPOP, LOSS_REINFORCE])
def test_exact_centering_equals_dense_expectation(loss_type):
    """Replayed support: sum_v u_v w_v log P_v equals E_q[w log P] enumerated over the
    whole vocabulary with q = 0 off S (pull request #4233: truncated sampling, u = q,
    centering is exact)."""
    rng = np.random.default_rng(5)
    V = 24
    z = rng.normal(0, 2.0, size=V)
    S = sorted(rng.choice(V, size=7, replace=False))
    qS = _softmax(z[S] + rng.normal(0, 0.8, len(S)))
    q_dense = np.zeros(V)
    q_dense[S] = qS
    P_dense = np.zeros(V)
    P_dense[S] = _softmax(z[S])
    hp = HeadParams(loss_type=loss_type, eps=0.1, max_importance_ratio=1.5, icepop_low=0.7,
                    icepop_high=1.4)
    expect = 0.0
    for v in range(V):
        if q_dense[v] > 0:
            expect += q_dense[v] * _keep_w(P_dense[v], q_dense[v], hp) * math.log(P_dense[v])
    inp = identity_case(z[None], [S[0]], [math.log(qS[0])], [(S, list(np.log(qS)))], [1])
    out = oracle.head_forward(inp, hp)
    assert abs(out["center"][0] - expect) < 1e-12
    if loss_type == LOSS_REINFORCE:
        # E_q[log P] = -(H(q) + KL(q||P)), through scipy
        alt = -(scipy.stats.entropy(qS) + scipy.stats.entropy(qS, P_dense[S]))
        assert abs(out["center"][0] - alt) < 1e-12


@pytest.mark.parametrize("K", [16, 256, 4096, 16384])
def test_k_draw_estimator_converges_to_exact_centre(K):
    """u = 1/K over K i.i.d. draws from q estimates E_q[w log p] and KL(q||p) within a
    4 sigma / sqrt(K) CLT bound (pull request #4233, untruncated sampling)."""
    rng = np.random.default_rng(1000 + K)
    V = 32
    z = rng.normal(0, 1.0, size=V)
    q = _softmax(z + rng.normal(0, 0.4, V))
    p = _softmax(z)
    hp = HeadParams(loss_type=LOSS_IPO, eps=0.02, max_importance_ratio=1.3,
                    kl_coeff=0.0, kl_estimator=KL_EXACT)
    f = np.array([_keep_w(p[v], q[v], hp) * math.log(p[v]) for v in range(V)])
    g = np.log(q) - np.log(p)
    Ef, Eg = float(q @ f), float(scipy.stats.entropy(q, p))
    sf = math.sqrt(float(q @ (f - Ef) ** 2))
    sg = math.sqrt(float(q @ (g - Eg) ** 2))
    draws = np.sort(rng.choice(V, size=K, replace=True, p=q))
    inp = identity_case(z[None], [0], [math.log(q[0])], [(draws, list(np.log(q[draws])))], [0])
    out = oracle.head_forward(inp, hp)
    assert abs(out["center"][0] - Ef) <= 4 * sf / math.sqrt(K)
    assert abs(out["kl"][0] - Eg) <= 4 * sg / math.sqrt(K)


def test_support_mass_and_mismatch_kl_against_enumeration():
    """support_mass = E_q[p/q] over the support with the full-vocab p (reading R8)
    equals the trainer mass on S for a replayed support; mismatch KL at the label is
    log q(a) - log P(a)."""
    rng = np.random.default_rng(6)
    V = 30
    z = rng.normal(0, 1.0, size=V)
    S = sorted(rng.choice(V, size=11, replace=False))
    qS = _softmax(z[S] + rng.normal(0, 0.5, len(S)))
    inp = identity_case(z[None], [S[2]], [math.log(qS[2])], [(S, list(np.log(qS)))], [1])
    out = oracle.head_forward(inp, HeadParams(loss_type=LOSS_REINFORCE))
    p = _softmax(z)
    assert abs(out["metrics"]["support_mass"] - p[S].sum()) < 1e-12
    PS = _softmax(z[S])
    assert abs(out["metrics"]["mismatch_kl"] - (math.log(qS[2]) - math.log(PS[2]))) < 1e-12


# --------------------------------------------------------------------------------------
# Finite differences with w held constant (the sg[] of the loss)
# --------------------------------------------------------------------------------------
def _random_case(rng, N=6, H=5, V=9, mixed=True):
    X = rng.normal(0, 1, size=(N, H))
    W = rng.normal(0, 0.6, size=(V, H))
    T = 0.7
    z = X @ W.T / T
    labels, lab_lq, sup, rep = [], [], [], []
    for t in range(N):
        q = _softmax(z[t] + rng.normal(0, 0.4, V))
        if mixed and t % 2 == 1:
            S = sorted(rng.choice(V, size=4, replace=False))
            qS = q[S] / q[S].sum()
            a = S[int(rng.integers(0, 4))]
            labels.append(a)
            lab_lq.append(math.log(qS[S.index(a)]))
            sup.append((S, list(np.log(qS))))
            rep.append(1)
        else:
            d = sorted(rng.choice(V, size=5, replace=True, p=q))
            a = int(rng.integers(0, V))
            labels.append(a)
            lab_lq.append(math.log(q[a]))
            sup.append((d, list(np.log(q[d]))))
            rep.append(0)
    inp = identity_case(np.zeros((N, V)), labels, lab_lq, sup, rep,
                        adv=rng.normal(0, 1, N), age=rng.integers(0, 5, N))
    inp["hidden"], inp["W"] = X, W
    return inp, T


@pytest.mark.parametrize("loss_type,est,stale,ent", [
    (LOSS_IPO, KL_EXACT, oracle.STALE_INV_SQRT, 0.0),
    (LOSS_ICEPOP, KL_K1, oracle.STALE_NONE, 0.0),
    (LOSS_REINFORCE, KL_EXACT, oracle.STALE_NONE, 0.0),
    (LOSS_IPO, KL_EXACT, oracle.STALE_NONE, 0.05),     # with the entropy regulariser
])
def test_finite_differences(loss_type, est, stale, ent):
    rng = np.random.default_rng(7 + loss_type)
    inp, T = _random_case(rng)
    hp = HeadParams(loss_type=loss_type, eps=0.15, max_importance_ratio=1.4, icepop_low=0.8,
                    icepop_high=1.25, adv_tau=0.9, temperature=T, kl_coeff=0.07,
                    kl_estimator=est, kl_staleness=stale, entropy_coeff=ent)
    N = inp["hidden"].shape[0]
    dloss = rng.normal(0, 1, N)
    base = oracle.head_forward(inp, hp)
    off = inp["offsets"]
    frozen = {t: (base["w_label"][t], base["w_support"][off[t]:off[t + 1]]) for t in range(N)}
    dX, dW = oracle.head_backward(inp, hp, dloss)
    h = 1e-6
    for name, grad in (("hidden", dX), ("W", dW)):
        A = inp[name]
        for idx in [(0, 0), (1, 3), (2, 4), (min(A.shape[0] - 1, 5), 2)]:
            old = A[idx]
            A[idx] = old + h
            lp = oracle.head_loss_total(inp, hp, dloss, frozen)
            A[idx] = old - h
            lm = oracle.head_loss_total(inp, hp, dloss, frozen)
            A[idx] = old
            fd = (lp - lm) / (2 * h)
            assert abs(fd - grad[idx]) <= 1e-7 * max(1.0, abs(grad[idx])), (name, idx, fd, grad[idx])


def test_loss_mask_zero_tokens_have_no_loss_or_gradient():
    rng = np.random.default_rng(8)
    inp, T = _random_case(rng)
    inp["loss_mask"] = np.array([1, 0, 1, 0, 1, 1], dtype=np.uint8)
    hp = HeadParams(temperature=T, kl_coeff=0.1)
    out = oracle.head_forward(inp, hp)
    dX, _ = oracle.head_backward(inp, hp, np.ones(6))
    assert out["loss"][1] == 0.0 and out["loss"][3] == 0.0
    assert np.all(dX[1] == 0) and np.all(dX[3] == 0)
    assert out["metrics"]["n_rl"] == 4


def test_temperature_is_a_logit_scale():
    """z = W h / T: doubling W and T leaves every forward output unchanged."""
    rng = np.random.default_rng(9)
    inp, T = _random_case(rng)
    hp = HeadParams(temperature=T, kl_coeff=0.05)
    a = oracle.head_forward(inp, hp)
    inp2 = dict(inp)
    inp2["W"] = 2.0 * inp["W"]
    b = oracle.head_forward(inp2, HeadParams(temperature=2 * T, kl_coeff=0.05))
    np.testing.assert_allclose(a["loss"], b["loss"], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(a["logp_support"], b["logp_support"], rtol=1e-12)


def test_entropy_regulariser_closed_forms():
    """"10-KL-clip-entropy", section 3: loss -= entropy_coeff * entropy.  Uniform logits:
    the entropy is log V and a maximum (zero gradient), so the regulariser shifts the loss
    by -c log V and adds nothing to the gradient; with non-uniform logits it adds
    c p (log p + H), which sums to zero over the vocabulary (a softmax gradient)."""
    V = 11
    z = np.zeros(V)
    base = dict(label=2, label_logq=math.log(1 / V), adv=0.7, age=0, ids=np.array([1, 2, 5]),
                logq=np.log(np.full(3, 1 / V)), replayed=False)
    p0 = HeadParams(kl_coeff=0.0)
    p1 = HeadParams(kl_coeff=0.0, entropy_coeff=0.3)
    f0 = oracle.token_forward(z, p=p0, **base)
    f1 = oracle.token_forward(z, p=p1, **base)
    assert f1["entropy"] == pytest.approx(math.log(V))
    assert f1["loss"] - f0["loss"] == pytest.approx(-0.3 * math.log(V))
    g0 = oracle.rl_head.token_grad_z(z, 2, 0.7, base["ids"], False, f0, p0)
    g1 = oracle.rl_head.token_grad_z(z, 2, 0.7, base["ids"], False, f1, p1)
    np.testing.assert_allclose(g1, g0, atol=1e-15)
    z2 = np.linspace(-1.0, 2.0, V)
    f0 = oracle.token_forward(z2, p=p0, **base)
    f1 = oracle.token_forward(z2, p=p1, **base)
    g0 = oracle.rl_head.token_grad_z(z2, 2, 0.7, base["ids"], False, f0, p0)
    g1 = oracle.rl_head.token_grad_z(z2, 2, 0.7, base["ids"], False, f1, p1)
    d = g1 - g0
    pf = np.exp(z2 - f1["lse"])
    assert abs(d.sum()) < 1e-14
    # the entropy gradient points away from the most likely id (lowering its logit raises H)
    assert d[np.argmax(pf)] > 0 > d[np.argmin(pf)]


# --------------------------------------------------------------------------------------
# mask_tv (reading R9) and the inv_sqrt staleness (reading R6)
# --------------------------------------------------------------------------------------
def _tv_mask_removes(P, keep):
    """Total variation between P and P conditioned on the kept set, by enumeration."""
    P = np.asarray(P, np.float64)
    Pk = np.where(keep, P, 0.0)
    Pk = Pk / Pk.sum()
    return 0.5 * float(np.abs(P - Pk).sum())


@pytest.mark.parametrize("loss_type,knobs", [(LOSS_IPO, dict(eps=0.04)),
                                             (LOSS_ICEPOP, dict(icepop_low=0.7, icepop_high=1.3))])
def test_mask_tv_is_the_total_variation_the_mask_removes_under_exact_replay(loss_type, knobs):
    """Under exact replay (u = q over the support S), mask_tv of a token equals
    TV(P, P | kept entries): the trainer mass the mask takes off the centering support.
    P, q and the masks are enumerated here from their definitions on a 24-id vocabulary
    (truncated supports of 9..24 ids)."""
    rng = np.random.default_rng(21)
    V = 24
    p = HeadParams(loss_type=loss_type, **knobs)
    for trial in range(12):
        z = rng.normal(0, 1.2, size=(1, V))
        k = int(rng.integers(9, V + 1))
        S = np.sort(rng.choice(V, size=k, replace=False))
        qs = scipy.special.softmax(z[0, S] + rng.normal(0, 0.6, size=k))     # sampler, renormalised on S
        label = int(S[int(rng.integers(k))])
        inp = identity_case(z, [label], [math.log(qs[list(S).index(label)])], [(list(S), list(np.log(qs)))], [1])
        out = oracle.head_forward(inp, p)
        PS = scipy.special.softmax(z[0, S])                                   # trainer, renormalised on S
        if loss_type == LOSS_IPO:
            keep = np.abs(PS - qs) <= p.eps
        else:
            keep = (PS / qs >= p.icepop_low) & (PS / qs <= p.icepop_high)
        if keep.all() or not keep.any():
            assert out["metrics"]["mask_tv"] == pytest.approx(0.0 if keep.all() else 1.0, abs=1e-12)
            continue
        assert out["metrics"]["mask_tv"] == pytest.approx(_tv_mask_removes(PS, keep), rel=1e-12)


def test_mask_tv_with_draws_estimates_the_masked_trainer_mass():
    """With K i.i.d. draws from q (u = 1/K), mask_tv is the importance-weighted estimate
    of the full-vocabulary trainer mass the mask removes, sum_v p_v 1(v masked) =
    TV(p, p | kept): within 5 sigma (CLT) for K = 20000, sigma from the exact variance of
    (1 - m) p / q under q."""
    rng = np.random.default_rng(22)
    V = 20
    z = rng.normal(0, 1.0, size=(1, V))
    pf = scipy.special.softmax(z[0])
    q = scipy.special.softmax(z[0] + rng.normal(0, 0.7, size=V))
    p = HeadParams(loss_type=LOSS_IPO, eps=0.02)
    keep = np.abs(pf - q) <= p.eps
    assert 0 < keep.sum() < V
    K = 20000
    draws = np.sort(rng.choice(V, size=K, p=q))
    inp = identity_case(z, [int(draws[0])], [math.log(q[draws[0]])], [(list(draws), list(np.log(q[draws])))], [0])
    got = oracle.head_forward(inp, p)["metrics"]["mask_tv"]
    f = (~keep) * pf / q
    mean = float((q * f).sum())
    sd = math.sqrt(float((q * f ** 2).sum()) - mean ** 2) / math.sqrt(K)
    assert mean == pytest.approx(_tv_mask_removes(pf, keep), rel=1e-12)
    assert abs(got - mean) <= 5 * sd


def test_inv_sqrt_beta_follows_its_stated_properties():
    """Reading R6: age 0 takes the full kl_coeff, beta falls strictly with the policy age,
    and halves by age 3; no staleness leaves kl_coeff at every age."""
    c = 0.04
    stale = HeadParams(kl_coeff=c, kl_staleness=oracle.STALE_INV_SQRT)
    betas = [oracle.rl_head.kl_beta(a, stale) for a in range(12)]
    assert betas[0] == c
    assert all(b1 < b0 for b0, b1 in zip(betas, betas[1:]))
    assert betas[3] == pytest.approx(c / 2, rel=1e-15)
    assert all(oracle.rl_head.kl_beta(a, HeadParams(kl_coeff=c)) == c for a in range(12))
    # and beta scales the KL term of the loss: the loss moves by (beta_1 - beta_0) KL
    z = np.array([[0.3, -0.2, 1.1, 0.0]])
    q = scipy.special.softmax([0.1, 0.0, 0.9, 0.2])
    sup = ([0, 1, 2, 3], list(np.log(q)))
    l0 = oracle.head_forward(identity_case(z, [2], [math.log(q[2])], [sup], [1], age=[0]), stale)
    l1 = oracle.head_forward(identity_case(z, [2], [math.log(q[2])], [sup], [1], age=[1]), stale)
    kl = float((q * (np.log(q) - np.log(scipy.special.softmax(z[0])))).sum())
    assert l1["loss"][0] - l0["loss"][0] == pytest.approx((c / math.sqrt(2) - c) * kl, rel=1e-10)


# --------------------------------------------------------------------------------------
# Sampler-evidence validation (pull request #4233, GPU validation of the CSR entries)
# --------------------------------------------------------------------------------------
def _valid_case():
    rng = np.random.default_rng(23)
    V = 50
    z = rng.normal(0, 1, size=(4, V))
    sup, lq = [], []
    for t in range(4):
        if t % 2 == 0:                          # replayed, renormalised q, label inside
            S = np.sort(rng.choice(V, size=8, replace=False))
            q = scipy.special.softmax(rng.normal(0, 1, 8))
            sup.append((list(S), list(np.log(q))))
            lq.append(float(np.log(q[3])))
        else:                                   # draws, duplicates allowed, ascending
            d = np.sort(rng.integers(0, V, 6))
            sup.append((list(d), list(np.log(np.full(6, 0.02)))))
            lq.append(math.log(0.05))
    labels = [int(sup[0][0][3]), 7, int(sup[2][0][3]), 9]
    return identity_case(z, labels, lq, sup, [1, 0, 1, 0]), V


def test_validation_accepts_a_clean_batch_and_names_each_fault():
    inp, V = _valid_case()
    check = lambda d: oracle.validate_support(d, V)
    assert check(inp) == 0
    S = oracle.rl_head

    def mod(**kw):
        d = {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in inp.items()}
        for k, f in kw.items():
            f(d[k])
        return d

    def setitem(i, v):
        def f(a):
            a[i] = v
        return f
    assert check(mod(offsets=setitem(0, 1))) & S.STATUS_OFFSETS
    assert check(mod(offsets=setitem(2, 3))) & S.STATUS_OFFSETS           # decreasing: row 1 bad
    assert check(mod(offsets=setitem(4, 99))) == S.STATUS_OFFSETS         # past nnz, last row skipped
    assert check(mod(ids=setitem(7, V))) == S.STATUS_ID_RANGE            # last of its row: order kept
    assert check(mod(labels=setitem(1, -1))) == S.STATUS_ID_RANGE
    assert check(mod(logq=setitem(9, 0.5))) == S.STATUS_LOGQ              # log q > 1e-6
    assert check(mod(logq=setitem(9, np.nan))) == S.STATUS_LOGQ
    assert check(mod(label_logq=setitem(1, np.inf))) == S.STATUS_LOGQ
    row0 = list(inp["ids"][:8])
    missing = next(v for v in range(V) if v not in row0)
    assert check(mod(labels=setitem(0, missing))) == S.STATUS_LABEL_MISSING
    assert check(mod(logq=lambda a: a.__setitem__(slice(0, 8), a[:8] + math.log(0.9)))) == S.STATUS_SUPPORT_MASS
    assert check(mod(ids=lambda a: a.__setitem__(slice(2, 4), a[2:4][::-1].copy()))) == S.STATUS_ROW_ORDER
    # a draw row may repeat an id (ascending, not strictly); a replayed row may not
    dup = mod(ids=lambda a: a.__setitem__(9, a[8]))
    assert check(dup) == 0
    assert check(mod(ids=lambda a: a.__setitem__(1, a[0]))) & S.STATUS_ROW_ORDER
    # an RL token with an empty row; a non-RL one may have it
    e = dict(inp, offsets=np.array([0, 8, 8, 16, 22]), ids=np.concatenate([inp["ids"][:8], inp["ids"][14:]]),
             logq=np.concatenate([inp["logq"][:8], inp["logq"][14:]]))
    assert check(e) == S.STATUS_EMPTY_ROW
    assert check(dict(e, loss_mask=np.array([1, 0, 1, 1], np.uint8))) == 0


def test_vocab_shard_statistics_combine_to_the_full_vocabulary():
    """Split by vocabulary into three ranges, the shard statistics combine (max shift, sum)
    to the full logsumexp and entropy of the plain forward, and every label / support
    logit is owned by exactly one shard."""
    rng = np.random.default_rng(24)
    V = 40
    z = rng.normal(0, 2.0, size=(5, V))
    sup = [(sorted(rng.choice(V, 6, replace=False).tolist()), list(np.log(np.full(6, 1 / 6)))) for _ in range(5)]
    inp = identity_case(z, [3, 11, 25, 39, 0], [math.log(0.1)] * 5, sup, [0] * 5)
    p = HeadParams()
    full = oracle.head_forward(inp, p)
    parts = [oracle.vocab_shard_stats(inp, p, a, b) for a, b in ((0, 16), (16, 32), (32, 40))]
    M = np.max([q["m"] for q in parts], axis=0)
    S = sum(q["s"] * np.exp(q["m"] - M) for q in parts)
    U = sum((q["u"] + q["s"] * (q["m"] - M)) * np.exp(q["m"] - M) for q in parts)
    lse = M + np.log(S)
    np.testing.assert_allclose(lse, full["lse"], rtol=1e-13)
    np.testing.assert_allclose(np.log(S) - U / S, full["entropy"], rtol=1e-12, atol=1e-12)
    zlab = sum(q["zlab"] for q in parts)
    np.testing.assert_allclose(zlab - lse, full["logp_label"], rtol=1e-12, atol=1e-12)
    zsup = sum(q["zsup"] for q in parts)
    np.testing.assert_allclose(zsup, z[np.repeat(np.arange(5), 6), inp["ids"]], rtol=0, atol=0)
