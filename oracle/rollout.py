"""fp64 oracle of the rollout-correction weights (truncated / clipped / masked importance
sampling at token, sequence or geometric level, rejection sampling, the veto, batch
normalisation) and the mismatch-monitoring metrics, over a batch of sequences.

TEST INFRASTRUCTURE: see the package docstring.  Source: "Rollout Correction Methods"
(miles docs):
  * "Config keys": tis_mode (truncate / clip / mask), tis_lower_bound / tis_upper_bound,
    tis_level (token / sequence / geometric), tis_batch_normalize (weights scaled to mean
    1 over the batch); use_rs with rs_lower_bound / rs_upper_bound (falling back to the
    tis bounds), rs_level and rs_veto_threshold.  Rejected tokens or sequences leave the
    loss average.
  * "Importance Sampling": token weight exp(log pi_train - log pi_rollout); sequence
    weight exp(sum of the token log-ratios); geometric weight exp(mean of them).
  * "Rejection Sampling": token level rejects a token whose weight is outside the
    bounds; sequence level rejects a sequence whose MEAN token weight is outside them;
    geometric level one whose geometric-mean weight is; the veto rejects a whole sequence
    holding a token with weight below the veto threshold, whatever the IS/RS settings.
  * "Mismatch Metrics": training / rollout log-perplexity and perplexity, mis_kl,
    mis_k3_kl, the log-perplexity difference and its absolute value, the perplexity
    ratio, token- and sequence-level chi^2, the token-level absolute log-prob difference;
    and the IS/RS metrics (weights before / after bounding, the truncated / clipped /
    masked fractions, the RS fractions, catastrophic token / sequence fractions, the mean
    after TIS and RS, the batch normalisation factor, final mean / min / max).

Readings where the page is silent (each marked READING below):
  * RC1 "out of threshold" keeps a weight equal to a bound (lower <= w <= upper is kept).
  * RC2 truncate bounds from above only (w -> min(w, upper)); clip clamps to [lower, upper];
    mask zeroes a weight outside [lower, upper] (the token stays in the average).
  * RC3 the expectations E[.] of the mismatch table are token means over the response
    mask, except: the log-perplexities are per sequence (mean of -log pi over its
    tokens) averaged over sequences; perplexity = exp(that mean); the log-ppl difference,
    its absolute value and the perplexity ratio are per-sequence quantities averaged
    over sequences; chi^2_seq uses the sequence weight exp(sum log-ratio).
  * RC4 chi^2 between the two policies, estimated under the rollout policy, is
    E[w^2] - 1.
  * RC5 batch normalisation divides the kept tokens' bounded weights by their token mean
    (factor 1 if that mean is 0 or nothing is kept); the min / max / mean "final"
    statistics are over kept tokens.
  * RC6 a sequence counts for the sequence metrics when it holds at least one response
    token; the fractions of tokens are over response tokens.
  * RC7 with use_tis off the weights are 1 on kept tokens (RS, veto and metrics only).
Sums whose value decides a sequence's weight or rejection are exactly rounded
(math.fsum), so those decisions are the definition's up to one rounding.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

TIS_TRUNCATE, TIS_CLIP, TIS_MASK = "truncate", "clip", "mask"
LEVEL_TOKEN, LEVEL_SEQUENCE, LEVEL_GEOMETRIC = "token", "sequence", "geometric"


@dataclasses.dataclass
class RolloutParams:
    use_tis: bool = True
    tis_mode: str = TIS_TRUNCATE
    tis_lower_bound: float = 0.5
    tis_upper_bound: float = 2.0
    tis_level: str = LEVEL_TOKEN
    tis_batch_normalize: bool = False
    use_rs: bool = False
    rs_lower_bound: Optional[float] = None      # None: the tis bound
    rs_upper_bound: Optional[float] = None
    rs_level: str = LEVEL_TOKEN
    rs_veto_threshold: Optional[float] = None   # None: no veto


def _segments(seq_offsets, T):
    off = np.asarray(seq_offsets, dtype=np.int64)
    assert off.ndim == 1 and off[0] == 0 and off[-1] == T and np.all(np.diff(off) >= 0)
    return off


def rollout_correction(lp_train, lp_rollout, mask, seq_offsets, rp: RolloutParams) -> dict:
    """Per-token final IS weights and keep mask, and the batch's metric sums / counts.

    lp_train: log pi_train per token (the trainer's recomputed log-probs, pi_old);
    lp_rollout: log pi_rollout (the inference engine's); mask: response mask;
    seq_offsets [B+1]: sequence b holds tokens [seq_offsets[b], seq_offsets[b+1]).
    A weight past the double range is inf (as its definition overflows)."""
    with np.errstate(over="ignore"):
        return _rollout_correction(lp_train, lp_rollout, mask, seq_offsets, rp)


def _rollout_correction(lp_train, lp_rollout, mask, seq_offsets, rp: RolloutParams) -> dict:
    lt = np.asarray(lp_train, dtype=np.float64)
    lr = np.asarray(lp_rollout, dtype=np.float64)
    valid = np.asarray(mask).astype(bool)
    T = lt.shape[0]
    off = _segments(seq_offsets, T)
    B = off.shape[0] - 1
    L, U = float(rp.tis_lower_bound), float(rp.tis_upper_bound)
    rs_L = L if rp.rs_lower_bound is None else float(rp.rs_lower_bound)    # "Config keys"
    rs_U = U if rp.rs_upper_bound is None else float(rp.rs_upper_bound)

    delta = lt - lr                       # log pi_train - log pi_rollout
    w_tok = np.exp(delta)                 # token IS weight ("Importance Sampling")
    w_raw = np.zeros(T)                   # IS weight at tis_level
    keep = valid.copy()
    catastrophic = np.zeros(T, dtype=bool)
    rs_low = np.zeros(T, dtype=bool)
    rs_high = np.zeros(T, dtype=bool)
    n_seq = 0
    n_cat_seq = 0
    seq_stats = []                        # per sequence with tokens: (train_lppl, rollout_lppl, S)
    for b in range(B):
        idx = np.arange(off[b], off[b + 1])
        idx = idx[valid[idx]]
        n = idx.shape[0]
        if n == 0:
            continue
        n_seq += 1
        S = math.fsum(delta[idx])         # exactly rounded sum of the log-ratios
        if rp.tis_level == LEVEL_TOKEN:
            w_raw[idx] = w_tok[idx]
        elif rp.tis_level == LEVEL_SEQUENCE:
            w_raw[idx] = np.exp(S)             # inf past the double range
        elif rp.tis_level == LEVEL_GEOMETRIC:
            w_raw[idx] = math.exp(S / n)
        else:
            raise ValueError(rp.tis_level)
        # rejection sampling ("Rejection Sampling")
        if rp.use_rs:
            if rp.rs_level == LEVEL_TOKEN:
                lo_t = w_tok[idx] < rs_L
                hi_t = w_tok[idx] > rs_U
                rs_low[idx] = lo_t
                rs_high[idx] = hi_t
            else:
                if rp.rs_level == LEVEL_SEQUENCE:
                    stat = math.fsum(w_tok[idx]) / n          # mean token weight
                elif rp.rs_level == LEVEL_GEOMETRIC:
                    stat = math.exp(S / n)                    # geometric mean weight
                else:
                    raise ValueError(rp.rs_level)
                if stat < rs_L:                               # READING RC1
                    rs_low[idx] = True
                elif stat > rs_U:
                    rs_high[idx] = True
        # veto ("Veto Mechanism"): independent of the IS / RS settings
        if rp.rs_veto_threshold is not None:
            cat = w_tok[idx] < float(rp.rs_veto_threshold)
            catastrophic[idx] = cat
            if cat.any():
                n_cat_seq += 1
                keep[idx] = False
        tr = -math.fsum(lt[idx]) / n      # per-sequence log-perplexities (READING RC3)
        ro = -math.fsum(lr[idx]) / n
        seq_stats.append((tr, ro, S))
    keep &= ~(rs_low | rs_high)

    # bounding by tis_mode (READING RC2)
    t_low = valid & (w_raw < L)
    t_high = valid & (w_raw > U)
    if not rp.use_tis:
        w_b = np.ones(T)                                  # READING RC7
    elif rp.tis_mode == TIS_TRUNCATE:
        w_b = np.minimum(w_raw, U)
    elif rp.tis_mode == TIS_CLIP:
        w_b = np.clip(w_raw, L, U)
    elif rp.tis_mode == TIS_MASK:
        w_b = np.where((w_raw >= L) & (w_raw <= U), w_raw, 0.0)
    else:
        raise ValueError(rp.tis_mode)
    w_b = np.where(valid, w_b, 0.0)
    kept_sum = float(w_b[keep].sum())
    n_kept = int(keep.sum())
    factor = 1.0
    if rp.use_tis and rp.tis_batch_normalize and n_kept > 0 and kept_sum > 0:
        factor = n_kept / kept_sum                         # READING RC5
    w_final = np.where(keep, w_b * factor, 0.0)

    v = valid
    dv = delta[v]
    st = np.array(seq_stats) if seq_stats else np.zeros((0, 3))
    m = dict(
        n_valid=int(v.sum()), n_seq=n_seq, n_kept=n_kept,
        # IS / RS correction metrics (sums and counts; means are sum / count)
        w_before_sum=float(w_raw[v].sum()), w_after_sum=float(w_b[v].sum()),
        n_tis_low=int(t_low.sum()), n_tis_high=int(t_high.sum()),
        n_rs_low=int((rs_low & v).sum()), n_rs_high=int((rs_high & v).sum()),
        n_cat_tokens=int((catastrophic & v).sum()), n_cat_seqs=n_cat_seq,
        kept_w_sum=kept_sum, batch_norm_factor=factor,
        final_sum=float(w_final[keep].sum()),
        final_min=float(w_final[keep].min()) if n_kept else 0.0,
        final_max=float(w_final[keep].max()) if n_kept else 0.0,
        # mismatch-monitoring sums (READING RC3, RC4)
        mis_kl_sum=float((-dv).sum()), k3_sum=float((np.exp(dv) - dv - 1.0).sum()),
        abs_diff_sum=float(np.abs(dv).sum()), chi2_token_sum=float(np.exp(2.0 * dv).sum()),
        train_lppl_sum=float(st[:, 0].sum()), rollout_lppl_sum=float(st[:, 1].sum()),
        lppl_diff_sum=float((st[:, 0] - st[:, 1]).sum()),
        lppl_abs_diff_sum=float(np.abs(st[:, 0] - st[:, 1]).sum()),
        ppl_ratio_sum=float(np.exp(st[:, 0] - st[:, 1]).sum()),
        chi2_seq_sum=float(np.exp(2.0 * st[:, 2]).sum()),
    )
    return dict(weights=w_final, keep=keep.astype(np.uint8), metrics=m)


def rollout_metrics_named(m: dict, rp: RolloutParams) -> dict:
    """The page's metric names from the sums and counts ("Mismatch Metrics" tables), for
    the metrics those settings emit: the monitoring metrics always; the IS/RS metrics by
    the "Emitted when" column of the "IS/RS Correction Metrics" table (use_tis for the
    weight statistics, the tis_mode for its fractions, use_rs, a set veto threshold).
    A mean over an empty set is 0."""
    nv, ns, nk = max(m["n_valid"], 1), max(m["n_seq"], 1), max(m["n_kept"], 1)
    train_lppl = m["train_lppl_sum"] / ns
    rollout_lppl = m["rollout_lppl_sum"] / ns
    out = {
        "training_log_ppl": train_lppl, "training_ppl": math.exp(train_lppl),
        "rollout_log_ppl": rollout_lppl, "rollout_ppl": math.exp(rollout_lppl),
        "kl": m["mis_kl_sum"] / nv, "k3_kl": m["k3_sum"] / nv,
        "log_ppl_diff": m["lppl_diff_sum"] / ns, "log_ppl_abs_diff": m["lppl_abs_diff_sum"] / ns,
        "ppl_ratio": m["ppl_ratio_sum"] / ns,
        "chi2_token": m["chi2_token_sum"] / nv - 1.0 if m["n_valid"] else 0.0,
        "chi2_seq": m["chi2_seq_sum"] / ns - 1.0 if m["n_seq"] else 0.0,
        "train_rollout_logprob_abs_diff": m["abs_diff_sum"] / nv,
    }
    if rp.use_tis:
        out.update({
            "tis_weight_before_bound": m["w_before_sum"] / nv, "tis_weight_after_bound": m["w_after_sum"] / nv,
            "is_ratio_mean_after_tis_rs": m["kept_w_sum"] / nk, "batch_norm_factor": m["batch_norm_factor"],
            "is_ratio_mean_final": m["final_sum"] / nk, "is_ratio_min_final": m["final_min"],
            "is_ratio_max_final": m["final_max"]})
        lo, hi = m["n_tis_low"] / nv, m["n_tis_high"] / nv
        if rp.tis_mode == TIS_TRUNCATE:
            out["tis_truncate_fraction"] = hi
        elif rp.tis_mode == TIS_CLIP:
            out["tis_clip_fraction_low"], out["tis_clip_fraction_high"] = lo, hi
        else:
            out["tis_mask_fraction_low"], out["tis_mask_fraction_high"] = lo, hi
    if rp.use_rs:
        out["rs_mask_fraction_low"] = m["n_rs_low"] / nv
        out["rs_mask_fraction_high"] = m["n_rs_high"] / nv
    if rp.rs_veto_threshold is not None and rp.rs_veto_threshold > 0:
        out["rs_catastrophic_token_fraction"] = m["n_cat_tokens"] / nv
        out["rs_catastrophic_seq_fraction"] = m["n_cat_seqs"] / ns
    return out
