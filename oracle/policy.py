"""fp64 oracle of the elementwise PPO / dual-clip / decoupled-TIS losses and the
mismatch statistics on per-token log-probabilities.

TEST INFRASTRUCTURE: see the package docstring.  Sources:
  * "Rollout Correction Methods", "Algorithms": standard PPO (ratio pi_theta/pi_old,
    clip to [1 - eps, 1 + eps]); bypass PPO (pi_old := rollout, an input choice);
    decoupled 3-policy PPO (the clipped surrogate times pi_old / pi_rollout).
  * "Rollout Correction Methods", "Mismatch Metrics": mis_kl = E[log pi_rollout -
    log pi_train]; mis_k3_kl = E[exp(r) - r - 1], r = log pi_train - log pi_rollout.
  * "10-KL-clip-entropy", section 2: ratio = exp(log_prob - old_log_prob), clamp to
    [1 - clip_ratio_low, 1 + clip_ratio_high], the dual-clip branch for negative
    advantages (clip_ratio_c), and the pg_clipfrac / ppo_kl / pg_clipfrac_lower
    metrics; defaults 0.2 / 0.2 / 3.0.
  * "IPO (INTELLECT Policy Optimization)", "Masking by Probability, Not Ratio" and
    "Choosing eps": the IPO mask |pi_train - pi_infer| > eps swept over eps, against
    the IcePop ratio band [alpha, beta].
"""
from __future__ import annotations

import dataclasses

import numpy as np

IPO_CURVE_EPS = tuple(round(0.05 * k, 2) for k in range(1, 11))   # 0.05 .. 0.50


@dataclasses.dataclass
class PolicyParams:
    clip_ratio_low: float = 0.2
    clip_ratio_high: float = 0.2
    clip_ratio_c: float = 3.0
    tis_upper: float = 2.0          # READING R11: token-level truncation bound
    icepop_low: float = 0.5
    icepop_high: float = 2.0
    curve_eps: tuple = IPO_CURVE_EPS


def policy_loss_elementwise(lp_theta, lp_old, lp_samp, adv, mask, pp: PolicyParams) -> dict:
    """Per-token losses/gradients and masked sums/counts (token-mean is sum / n_valid)."""
    lt = np.asarray(lp_theta, dtype=np.float64)
    lo = np.asarray(lp_old, dtype=np.float64)
    ls = np.asarray(lp_samp, dtype=np.float64)
    A = np.asarray(adv, dtype=np.float64)
    valid = np.asarray(mask).astype(bool)

    r = np.exp(lt - lo)
    l1 = -A * r                                                   # unclipped surrogate
    l2 = -A * np.clip(r, 1.0 - pp.clip_ratio_low, 1.0 + pp.clip_ratio_high)
    lc = np.maximum(l1, l2)                                       # pessimistic of the two
    l3 = -A * pp.clip_ratio_c                                     # dual-clip cap, A < 0 only
    dual = (A < 0) & (l3 < lc)
    loss_ppo = np.where(A < 0, np.minimum(lc, l3), lc)
    # d/d lp_theta of the active branch: -A r on the unclipped branch, 0 when clipped
    # or capped (the clipped branch differs from l1 only outside the band).
    g_c = np.where(l1 >= l2, -A * r, 0.0)
    grad_ppo = np.where(dual, 0.0, g_c)

    rho_raw = np.exp(lo - ls)                                     # pi_old / pi_rollout
    rho = np.minimum(rho_raw, pp.tis_upper)
    loss_dec = rho * lc                                           # -rho * min(rA, clip(r)A)
    grad_dec = rho * g_c

    p_old = np.exp(lo)
    p_samp = np.exp(ls)
    d = lo - ls                                                   # log pi_train - log pi_rollout
    zero = lambda x: np.where(valid, x, 0.0)
    out = dict(loss_ppo=zero(loss_ppo), loss_dec=zero(loss_dec), grad_ppo=zero(grad_ppo),
               grad_dec=zero(grad_dec))
    v = valid
    out["metrics"] = dict(
        n_valid=int(v.sum()),
        loss_ppo=float(loss_ppo[v].sum()),
        loss_dec=float(loss_dec[v].sum()),
        n_clip=int(((l2 > l1) & v).sum()),
        ppo_kl=float((lo - lt)[v].sum()),
        n_clip_lower=int((dual & v).sum()),
        ipo_curve=[int(((np.abs(p_old - p_samp) > e) & v).sum()) for e in pp.curve_eps],
        icepop_low=int(((rho_raw < pp.icepop_low) & v).sum()),
        icepop_high=int(((rho_raw > pp.icepop_high) & v).sum()),
        mis_kl=float((ls - lo)[v].sum()),
        k3=float((np.exp(d) - d - 1.0)[v].sum()),
        tis_sum=float(rho[v].sum()),
        n_tis_trunc=int(((rho_raw > pp.tis_upper) & v).sum()),
    )
    return out
