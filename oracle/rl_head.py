"""fp64 oracle of the fused LM head + unified RL loss (forward, backward, metrics).

TEST INFRASTRUCTURE: see the package docstring.  Written from prime-rl pull request
#4233 (the loss_t equation; the estimator rules for u; "What changes"), with the mask
sense from "IPO (INTELLECT Policy Optimization)", "Masking by Probability, Not Ratio".

Per RL token t (loss_mask = 1), with z_t = W h_t / T:

  log p_t(v)    = z_tv - logsumexp_v' z_tv'                    (full-vocab trainer p)
  log P_t(v)    = z_tv - logsumexp_{v' in S_t} z_tv'  if replayed, else log p_t(v)  (READING R1)
  u_e           = q_e (= exp logq_e) on a replayed support, 1/K_t on K i.i.d. draws
  r             = P / q,   w = ipo:     1(|P - q| <= eps) * min(r, max_importance_ratio)
                               icepop:  1(low <= r <= high) * r
                               reinforce: 1
  loss_t        = -adv_tau * A_t * (w_a log P(a) - sum_e sg[u_e w_e] log P(v_e)) + beta_t KL_t
  KL_t          = exact: sum_e u_e (log q_e - log P(v_e));  k1: log q(a) - log P(a)  (READING R5)
  beta_t        = kl_coeff * (1 or 1/sqrt(1 + age_t))                               (READING R6)

w and u are held constant in the gradient (the sg[] of the equation; READING R4).
Nothing here is blocked, fused or reordered beyond "one token row at a time".
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

LOSS_IPO, LOSS_ICEPOP, LOSS_REINFORCE = 0, 1, 2
KL_EXACT, KL_K1 = 0, 1
STALE_NONE, STALE_INV_SQRT = 0, 1


@dataclasses.dataclass
class HeadParams:
    """Knobs of the unified loss (pull request #4233, "What changes")."""
    loss_type: int = LOSS_IPO
    eps: float = 0.3                   # ipo band half-width in probability
    max_importance_ratio: float = 10.0  # ipo ratio cap
    icepop_low: float = 0.5
    icepop_high: float = 2.0
    adv_tau: float = 1.0
    temperature: float = 1.0
    kl_coeff: float = 0.0
    kl_estimator: int = KL_EXACT
    kl_staleness: int = STALE_NONE
    entropy_coeff: float = 0.0          # "10-KL-clip-entropy" section 3: loss -= coeff * entropy


def _logsumexp(x: np.ndarray) -> float:
    m = float(np.max(x))
    return m + math.log(float(np.sum(np.exp(x - m))))


def rl_weight(logP: np.ndarray, logq: np.ndarray, p: HeadParams):
    """Per-token importance weight w and keep bit for each (P, q) pair.

    ipo:       1(|P - q| <= eps) * min(P/q, max_importance_ratio)
    icepop:    1(low <= P/q <= high) * P/q
    reinforce: 1
    (pull request #4233, "What changes", first item; the probability-difference mask is
    the one of "Masking by Probability, Not Ratio").  Threshold equality keeps the
    token (READING R15).  Returns (w, keep, low_side, high_side), where the sides say
    on which side of the band a masked token fell (P below / above q's band).
    """
    logP = np.asarray(logP, dtype=np.float64)
    logq = np.asarray(logq, dtype=np.float64)
    ratio = np.exp(logP - logq)
    if p.loss_type == LOSS_IPO:
        diff = np.exp(logP) - np.exp(logq)
        keep = np.abs(diff) <= p.eps
        w = np.where(keep, np.minimum(ratio, p.max_importance_ratio), 0.0)
        low = ~keep & (diff < 0)
        high = ~keep & (diff > 0)
    elif p.loss_type == LOSS_ICEPOP:
        keep = (ratio >= p.icepop_low) & (ratio <= p.icepop_high)
        w = np.where(keep, ratio, 0.0)
        low = ratio < p.icepop_low
        high = ratio > p.icepop_high
    elif p.loss_type == LOSS_REINFORCE:
        keep = np.ones_like(ratio, dtype=bool)
        w = np.ones_like(ratio)
        low = np.zeros_like(keep)
        high = np.zeros_like(keep)
    else:
        raise ValueError(f"unknown loss type {p.loss_type}")
    return w, keep, low, high


def kl_beta(age: int, p: HeadParams) -> float:
    """beta_t = kl_coeff * s(age_t): s = 1 (none) or 1/sqrt(1 + age) (inv_sqrt, READING R6)."""
    if p.kl_staleness == STALE_NONE:
        return float(p.kl_coeff)
    if p.kl_staleness == STALE_INV_SQRT:
        return float(p.kl_coeff) / math.sqrt(1.0 + float(age))
    raise ValueError(f"unknown staleness {p.kl_staleness}")


def token_forward(z: np.ndarray, label: int, label_logq: float, adv: float, age: int,
                  ids: np.ndarray, logq: np.ndarray, replayed: bool, p: HeadParams,
                  w_frozen=None) -> dict:
    """Loss and diagnostics of one RL token from its fp64 logits row z (already / T).

    ``w_frozen = (w_label, w_entries)`` overrides the weights (finite-difference checks
    hold w constant, as the sg[] in the loss says).
    """
    z = np.asarray(z, dtype=np.float64)
    ids = np.asarray(ids, dtype=np.int64)
    logq = np.asarray(logq, dtype=np.float64)
    lse = _logsumexp(z)
    logp_full = z - lse
    pf = np.exp(logp_full)
    entropy = float(-np.sum(pf * logp_full))
    K = ids.shape[0]
    if replayed:
        lse_s = _logsumexp(z[ids])            # READING R1: renormalised over S
        logP_lab = float(z[label] - lse_s)
        logP_ent = z[ids] - lse_s
        u = np.exp(logq)                      # u_v = q_v on a replayed support
    else:
        lse_s = lse
        logP_lab = float(logp_full[label])
        logP_ent = logp_full[ids]
        u = np.full(K, 1.0 / K) if K > 0 else np.zeros(0)   # u = 1/K for K i.i.d. draws
    w_lab, keep_lab, low_lab, high_lab = rl_weight(np.array([logP_lab]), np.array([label_logq]), p)
    w_lab, keep_lab = float(w_lab[0]), bool(keep_lab[0])
    w_ent, keep_ent, _, _ = rl_weight(logP_ent, logq, p)
    if w_frozen is not None:
        w_lab = float(w_frozen[0])
        w_ent = np.asarray(w_frozen[1], dtype=np.float64)
    c = u * w_ent                              # sg[u_v * w_v]
    center = float(np.sum(c * logP_ent))
    if p.kl_estimator == KL_EXACT:
        kl = float(np.sum(u * (logq - logP_ent)))
    elif p.kl_estimator == KL_K1:
        kl = float(label_logq - logP_lab)
    else:
        raise ValueError(f"unknown kl estimator {p.kl_estimator}")
    beta = kl_beta(age, p)
    loss = -p.adv_tau * adv * (w_lab * logP_lab - center) + beta * kl
    # exploration regulariser ("10-KL-clip-entropy", section 3): policy_loss -= entropy_coeff
    # * entropy, the token entropy of the full-vocabulary softmax of the logits
    loss -= p.entropy_coeff * entropy
    ratio_ent = np.exp(logP_ent - logq)
    return dict(
        loss=loss, lse=lse, lse_s=lse_s, entropy=entropy, logp_label=logP_lab,
        logp_support=logP_ent, w_label=w_lab, keep_label=keep_lab, low_label=bool(low_lab[0]),
        high_label=bool(high_lab[0]), w_support=w_ent, keep_support=keep_ent, u=u, c=c,
        center=center, kl=kl, beta=beta,
        # metrics (pull request #4233 "What changes", metrics item; READINGS R7-R9)
        mismatch_kl=float(label_logq - logP_lab),
        support_mass=float(np.sum(u * np.exp(logp_full[ids] - logq))),
        mask_tv=float(np.sum(u * (~keep_ent) * ratio_ent)),
        # the row's largest logit magnitude: the scale of the rounding an fp32 evaluation
        # of these logits carries (what a finite-precision result is compared against)
        zmax=float(np.max(np.abs(z))),
    )


def token_grad_z(z: np.ndarray, label: int, adv: float, ids: np.ndarray, replayed: bool,
                 fwd: dict, p: HeadParams, want_abs: bool = False):
    """d loss_t / d z_t over the whole vocabulary, with w, c, u held constant.

    d log P(v) / d z_j = delta_vj - P_j, where P is the full softmax of z, or for a
    replayed token the softmax restricted to S (zero off S).  The sum over entries uses
    np.add.at so duplicate draw ids each contribute.

    ``want_abs`` also returns the sum of the magnitudes of the terms that make up each
    component (the scale a finite-precision evaluation of the gradient is measured
    against; the terms can cancel in the gradient itself).
    """
    z = np.asarray(z, dtype=np.float64)
    ids = np.asarray(ids, dtype=np.int64)
    V = z.shape[0]
    if replayed:
        P = np.zeros(V)
        P[ids] = np.exp(z[ids] - fwd["lse_s"])
    else:
        P = np.exp(z - fwd["lse"])

    def dlogP(v):
        g = -P.copy()
        g[v] += 1.0
        return g

    # sum_e c_e d log P(v_e) = sum_e c_e onehot(v_e) - (sum_e c_e) P
    sum_c_onehot = np.zeros(V)
    np.add.at(sum_c_onehot, ids, fwd["c"])
    d_center = sum_c_onehot - float(np.sum(fwd["c"])) * P
    grad = -p.adv_tau * adv * (fwd["w_label"] * dlogP(label) - d_center)
    if fwd["beta"] != 0.0:
        if p.kl_estimator == KL_EXACT:
            sum_u_onehot = np.zeros(V)
            np.add.at(sum_u_onehot, ids, fwd["u"])
            d_kl = -(sum_u_onehot - float(np.sum(fwd["u"])) * P)
        else:
            d_kl = -dlogP(label)
        grad = grad + fwd["beta"] * d_kl
    # d(-c H)/dz_j = c p_j (log p_j + H), p the full softmax (dH/dz_j = -p_j (log p_j + H))
    logp_full = z - fwd["lse"]
    pf = np.exp(logp_full)
    if p.entropy_coeff != 0.0:
        grad = grad + p.entropy_coeff * pf * (logp_full + fwd["entropy"])
    if not want_abs:
        return grad
    onehot_abs_c = np.zeros(V)
    np.add.at(onehot_abs_c, ids, np.abs(fwd["c"]))
    sum_abs_c = float(np.sum(np.abs(fwd["c"])))
    at = abs(p.adv_tau * adv)
    mag = at * (abs(fwd["w_label"]) * P + onehot_abs_c + sum_abs_c * P)
    mag[label] += at * abs(fwd["w_label"])
    if fwd["beta"] != 0.0:
        if p.kl_estimator == KL_EXACT:
            onehot_u = np.zeros(V)
            np.add.at(onehot_u, ids, fwd["u"])
            mag = mag + fwd["beta"] * (onehot_u + float(np.sum(fwd["u"])) * P)
        else:
            mag = mag + fwd["beta"] * P
            mag[label] += fwd["beta"]
    if p.entropy_coeff != 0.0:
        mag = mag + p.entropy_coeff * pf * (np.abs(logp_full) + fwd["entropy"])
    return grad, mag


STATUS_OFFSETS, STATUS_ID_RANGE, STATUS_LOGQ, STATUS_LABEL_MISSING = 0x1, 0x2, 0x4, 0x8
STATUS_SUPPORT_MASS, STATUS_EMPTY_ROW, STATUS_ROW_ORDER = 0x10, 0x20, 0x40


def validate_support(inputs: dict, V: int) -> int:
    """The sampler-evidence checks of pull request #4233 ("What changes": the CSR entries
    are validated on the GPU once per step, before the optimizer), as status bits:

      OFFSETS        offsets[0] != 0, offsets[N] != nnz, or a row whose bounds are
                     negative, decreasing or past nnz (such a row is not looked into)
      ID_RANGE       a label or a support id outside [0, V)
      LOGQ           a log q (label or entry) that is not finite or is above 1e-6
      LABEL_MISSING  a replayed RL row that does not hold its label
      SUPPORT_MASS   a replayed RL row whose q does not sum to 1 within 1e-3 (READING R2)
      EMPTY_ROW      an RL token with no support entry
      ROW_ORDER      ids not ascending within a row (strictly ascending when replayed;
                     repeated draws are adjacent, READING R3)
    """
    off = np.asarray(inputs["offsets"], dtype=np.int64)
    ids = np.asarray(inputs["ids"], dtype=np.int64)
    logq = np.asarray(inputs["logq"], dtype=np.float64)
    N = off.shape[0] - 1
    nnz = ids.shape[0]
    rl_mask = inputs.get("loss_mask")
    bits = 0
    if N > 0 and (off[0] != 0 or off[N] != nnz):
        bits |= STATUS_OFFSETS
    for t in range(N):
        b, e = int(off[t]), int(off[t + 1])
        if b < 0 or e < b or e > nnz:
            bits |= STATUS_OFFSETS
            continue
        rl = True if rl_mask is None else bool(rl_mask[t])
        rep = bool(inputs["replayed"][t])
        label = int(inputs["labels"][t])
        llq = float(inputs["label_logq"][t])
        if not 0 <= label < V:
            bits |= STATUS_ID_RANGE
        if not math.isfinite(llq) or llq > 1e-6:
            bits |= STATUS_LOGQ
        if rl and e == b:
            bits |= STATUS_EMPTY_ROW
        row, lq = ids[b:e], logq[b:e]
        if np.any((row < 0) | (row >= V)):
            bits |= STATUS_ID_RANGE
        if np.any(~np.isfinite(lq) | (lq > 1e-6)):
            bits |= STATUS_LOGQ
        steps = np.diff(row)
        if np.any(steps <= 0) if rep else np.any(steps < 0):
            bits |= STATUS_ROW_ORDER
        if rep and rl:
            if label not in set(row.tolist()):
                bits |= STATUS_LABEL_MISSING
            with np.errstate(over="ignore", invalid="ignore"):
                mass = float(np.sum(np.exp(lq)))
            if not abs(mass - 1.0) <= 1e-3:
                bits |= STATUS_SUPPORT_MASS
    return bits


def _rows(inputs: dict):
    off = np.asarray(inputs["offsets"], dtype=np.int64)
    return off


def head_token_logits(inputs: dict, rows, temperature: float) -> np.ndarray:
    """z = hidden[rows] @ W^T / T in fp64 (a library matmul as one step)."""
    X = np.asarray(inputs["hidden"], dtype=np.float64)[rows]
    W = np.asarray(inputs["W"], dtype=np.float64)
    return (X @ W.T) / temperature


def head_forward(inputs: dict, p: HeadParams, rows=None, chunk: int = 64) -> dict:
    """Forward over tokens ``rows`` (default: all).  ``inputs`` holds numpy arrays:
    hidden [N,H], W [V,H] (fp64 copies of the bf16 values), labels, label_logq, adv,
    loss_mask, age, replayed, offsets [N+1], ids, logq.

    Returns per-token arrays (indexed like ``rows``), per-entry arrays (in the entries
    of those rows, concatenated in row order) and metric sums over the RL tokens.
    """
    off = _rows(inputs)
    N = off.shape[0] - 1
    rows = np.arange(N) if rows is None else np.asarray(rows, dtype=np.int64)
    n = rows.shape[0]
    out = {k: np.zeros(n) for k in ("loss", "lse", "lse_s", "entropy", "logp_label", "w_label",
                                    "kl", "beta", "center", "zmax")}
    out["mask_label"] = np.zeros(n, dtype=np.uint8)
    ent_lp, ent_mask, ent_w, ent_c, ent_u = [], [], [], [], []
    met = dict(n_rl=0, loss=0.0, mismatch_kl=0.0, masked=0, masked_low=0, masked_high=0, support_mass=0.0,
               mask_tv=0.0, kl=0.0, beta=0.0, kl_age0=0.0, n_age0=0, entropy=0.0)
    for c0 in range(0, n, chunk):
        rr = rows[c0:c0 + chunk]
        Z = head_token_logits(inputs, rr, p.temperature)
        for j, t in enumerate(rr):
            i = c0 + j
            s, e = int(off[t]), int(off[t + 1])
            fw = token_forward(Z[j], int(inputs["labels"][t]), float(inputs["label_logq"][t]),
                               float(inputs["adv"][t]), int(inputs["age"][t]),
                               inputs["ids"][s:e], inputs["logq"][s:e],
                               bool(inputs["replayed"][t]), p)
            rl = bool(inputs["loss_mask"][t])
            out["loss"][i] = fw["loss"] if rl else 0.0
            for k in ("lse", "lse_s", "entropy", "logp_label", "w_label", "kl", "beta", "center", "zmax"):
                out[k][i] = fw[k]
            out["mask_label"][i] = 1 if fw["keep_label"] else 0
            ent_lp.append(fw["logp_support"])
            ent_mask.append(fw["keep_support"].astype(np.uint8))
            ent_w.append(fw["w_support"])
            ent_c.append(fw["c"])
            ent_u.append(fw["u"])
            if rl:
                met["n_rl"] += 1
                met["loss"] += fw["loss"]
                met["mismatch_kl"] += fw["mismatch_kl"]
                met["masked"] += 0 if fw["keep_label"] else 1
                met["masked_low"] += int(fw["low_label"])
                met["masked_high"] += int(fw["high_label"])
                met["support_mass"] += fw["support_mass"]
                met["mask_tv"] += fw["mask_tv"]
                met["kl"] += fw["kl"]
                met["beta"] += fw["beta"]
                met["entropy"] += fw["entropy"]
                if int(inputs["age"][t]) == 0:
                    met["kl_age0"] += fw["kl"]
                    met["n_age0"] += 1
    cat = lambda xs, dt=np.float64: np.concatenate(xs).astype(dt) if xs else np.zeros(0, dt)
    out["logp_support"] = cat(ent_lp)
    out["mask_support"] = cat(ent_mask, np.uint8)
    out["w_support"] = cat(ent_w)
    out["c_support"] = cat(ent_c)
    out["u_support"] = cat(ent_u)
    out["metrics"] = met
    return out


def head_backward(inputs: dict, p: HeadParams, dloss: np.ndarray, chunk: int = 64,
                  rows=None, want_dW: bool = True, want_bounds: bool = False, want_dX: bool = True,
                  vrows=None, vcols=None):
    """dX [N,H] and dW [V,H] of sum_t dloss_t * loss_t, fp64, by the chain rule:
    G_tj = dloss_t / T * d loss_t / d z_tj;  dX = G W;  dW = G^T X.

    ``rows`` restricts dX to those tokens (dW then sums over those tokens only).
    ``vrows`` keeps only those vocabulary rows of dW (in that order); ``want_dX=False``
    skips dX (and its bounds), returning None for it; ``vcols`` restricts dX to the part
    that flows through those vocabulary ids, G[:, vcols] W[vcols] (one rank's share when W
    is split by vocabulary).
    ``want_bounds`` also returns the magnitudes a finite-precision evaluation is measured
    against, as a dict: ``X`` = |G| |W| and ``W`` = |G|^T |X| with |G| the sum of the
    magnitudes of the terms forming each G entry, and ``zX`` / ``zW`` the same products
    with each |G| entry of token t weighted by max_j |z_tj| (an error in token t's logits
    of that relative size moves G_t by as much).
    """
    off = _rows(inputs)
    N = off.shape[0] - 1
    rows = np.arange(N) if rows is None else np.asarray(rows, dtype=np.int64)
    W = np.asarray(inputs["W"], dtype=np.float64)
    Xall = np.asarray(inputs["hidden"], dtype=np.float64)
    V, H = W.shape
    vsel = np.arange(V) if vrows is None else np.asarray(vrows, dtype=np.int64)
    dX = np.zeros((rows.shape[0], H)) if want_dX else None
    dW = np.zeros((vsel.shape[0], H)) if want_dW else None
    bnd = {}
    if want_bounds:
        if want_dX:
            bnd["X"] = np.zeros((rows.shape[0], H))
            bnd["zX"] = np.zeros((rows.shape[0], H))
        if want_dW:
            bnd["W"] = np.zeros((vsel.shape[0], H))
            bnd["zW"] = np.zeros((vsel.shape[0], H))
    for c0 in range(0, rows.shape[0], chunk):
        rr = rows[c0:c0 + chunk]
        Z = head_token_logits(inputs, rr, p.temperature)
        G = np.zeros_like(Z)
        Gm = np.zeros_like(Z) if want_bounds else None
        Zm = np.zeros_like(Z) if want_bounds else None
        for j, t in enumerate(rr):
            if not inputs["loss_mask"][t] or dloss[t] == 0.0:
                continue
            s, e = int(off[t]), int(off[t + 1])
            ids = inputs["ids"][s:e]
            fw = token_forward(Z[j], int(inputs["labels"][t]), float(inputs["label_logq"][t]),
                               float(inputs["adv"][t]), int(inputs["age"][t]), ids,
                               inputs["logq"][s:e], bool(inputs["replayed"][t]), p)
            scale = float(dloss[t]) / p.temperature
            res = token_grad_z(Z[j], int(inputs["labels"][t]), float(inputs["adv"][t]), ids,
                               bool(inputs["replayed"][t]), fw, p, want_abs=want_bounds)
            if want_bounds:
                G[j] = scale * res[0]
                Gm[j] = abs(scale) * res[1]
                Zm[j] = fw["zmax"]
            else:
                G[j] = scale * res
        if want_dX:
            if vcols is None:
                dX[c0:c0 + rr.shape[0]] = G @ W
            else:
                vc = np.asarray(vcols, dtype=np.int64)
                dX[c0:c0 + rr.shape[0]] = G[:, vc] @ W[vc]
        if want_dW:
            dW += G[:, vsel].T @ Xall[rr]
        if want_bounds:
            aX = np.abs(Xall[rr])
            if want_dX:
                aW = np.abs(W)
                bnd["X"][c0:c0 + rr.shape[0]] = Gm @ aW
                bnd["zX"][c0:c0 + rr.shape[0]] = (Gm * Zm) @ aW
            if want_dW:
                bnd["W"] += Gm[:, vsel].T @ aX
                bnd["zW"] += (Gm * Zm)[:, vsel].T @ aX
    if want_bounds:
        return dX, dW, bnd
    return dX, dW


def head_loss_total(inputs: dict, p: HeadParams, dloss: np.ndarray, frozen=None) -> float:
    """sum_t dloss_t * loss_t over RL tokens; ``frozen`` maps t -> (w_label, w_entries)."""
    off = _rows(inputs)
    N = off.shape[0] - 1
    Z = head_token_logits(inputs, np.arange(N), p.temperature)
    tot = 0.0
    for t in range(N):
        if not inputs["loss_mask"][t]:
            continue
        s, e = int(off[t]), int(off[t + 1])
        fw = token_forward(Z[t], int(inputs["labels"][t]), float(inputs["label_logq"][t]),
                           float(inputs["adv"][t]), int(inputs["age"][t]), inputs["ids"][s:e],
                           inputs["logq"][s:e], bool(inputs["replayed"][t]), p,
                           w_frozen=None if frozen is None else frozen[t])
        tot += float(dloss[t]) * fw["loss"]
    return tot


def vocab_shard_stats(inputs: dict, p: HeadParams, v0: int, v1: int) -> dict:
    """Per-token statistics of the logits over the vocabulary columns [v0, v1) alone (one
    rank's rows of W when the head is split by vocabulary), fp64, from their definitions:
    m = max_j z_j, s = sum_j e^(z_j - m), u = sum_j e^(z_j - m) (z_j - m) over the range;
    and the label / support logits whose id lies in the range (0 for the others).
    Combined over the ranges (logsumexp = M + log sum_r s_r e^(m_r - M)) they give the
    full-vocabulary logsumexp and entropy of head_forward."""
    off = _rows(inputs)
    N = off.shape[0] - 1
    W = np.asarray(inputs["W"], dtype=np.float64)[v0:v1]
    X = np.asarray(inputs["hidden"], dtype=np.float64)
    Z = (X @ W.T) / p.temperature
    m = Z.max(axis=1)
    e = np.exp(Z - m[:, None])
    s = e.sum(axis=1)
    u = (e * (Z - m[:, None])).sum(axis=1)
    labels = np.asarray(inputs["labels"], dtype=np.int64)
    ids = np.asarray(inputs["ids"], dtype=np.int64)
    rows = np.repeat(np.arange(N), np.diff(off))
    own_l = (labels >= v0) & (labels < v1)
    own_s = (ids >= v0) & (ids < v1)
    zlab = np.where(own_l, Z[np.arange(N), np.clip(labels - v0, 0, v1 - v0 - 1)], 0.0)
    zsup = np.where(own_s, Z[rows, np.clip(ids - v0, 0, v1 - v0 - 1)], 0.0)
    return dict(m=m, s=s, u=u, zlab=zlab, zsup=zsup)
