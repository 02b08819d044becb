"""Tolerances and comparison helpers for the GPU-vs-oracle parity tests.

The bars (stated for this path): logprobs within 1e-5 absolute (fp32 accumulate); loss
within 1e-4 relative; masks, gathers and masked counts bit-exact; gradients within 2
bf16 ulp of the oracle rounded to bf16.

Log-prob bar.  A logit z_tj is an fp32 accumulation of H bf16 products; its rounding is
modelled as 2^-24 sqrt(H) times the row's largest logit magnitude Z_t = max_j |z_tj| (the
random-walk growth of H fp32 roundings of partial sums no larger than about Z_t), taken
twice: once for the gathered logit, once for the logsumexp it is measured against (a
p-weighted mean of the same logit errors).  The logsumexp itself and the subtraction
z - lse each round to fp32 once more: two ulps of lse.  So
    |gpu - ref| <= 1e-5 + 2 * 2^-24 sqrt(H) Z_t + 2 ulp_fp32(lse_t).
At H = 2048 with Z_t ~ 4.5 (the literal c2-c4 scales) that is 1e-5 + 2.4e-5 + 2e-6.

Readings of the gradient bar (a row is one token of dX or one vocabulary id of dW):
  element   |gpu - bf16(ref)| <= 2 ulp(max(|ref|, 2^-8 * rowmax|ref|))  (grad_precision SPLIT)
  row       max_h |gpu - bf16(ref)| <= 2 ulp(rowmax|ref|)              (grad_precision BF16)
and, reported as diagnostics only (not asserted):
  operand   |gpu - bf16(ref)| <= 2 ulp(ref) + 2^-8 * bound             (one bf16 GEMM operand
            rounded; bound = sum of term magnitudes)
  operand2  |gpu - bf16(ref)| <= 2 ulp(ref) + 2^-7 * bound             (both operands rounded)
2^-8 is bf16's unit roundoff.  Every reading first subtracts the logits' fp32
accumulation allowance carried into G (acc_tol of the |G| Z_t-weighted magnitudes).
"""
import math

import numpy as np
import torch

import lm_head_gb300 as rh
import oracle

LOGP_TOL = 1e-5
LOSS_REL = 1e-4
EPS32 = 2.0 ** -24


def acc_tol(H: int, zmax):
    """fp32-accumulation allowance of logits built from H bf16 products, for a row whose
    largest logit magnitude is zmax: 2^-24 sqrt(H) zmax, twice (the gathered logit and
    the logsumexp it is taken against)."""
    return 2.0 * EPS32 * np.sqrt(H) * np.asarray(zmax, dtype=np.float64)


def ulp32(x):
    x = np.abs(np.asarray(x, dtype=np.float64))
    return 2.0 ** (np.floor(np.log2(np.maximum(x, 2.0 ** -126))) - 23)


def logp_tol(H: int, zmax, lse):
    """Log-prob bar of a token whose largest logit magnitude is zmax and whose logsumexp
    (full, or over the replayed support) is lse: 1e-5 + acc_tol + 2 fp32 ulps of lse."""
    return LOGP_TOL + acc_tol(H, zmax) + 2.0 * ulp32(lse)


def f32(x):
    return float(np.float32(x))


def oracle_params(hp: rh.HeadParams) -> oracle.HeadParams:
    """The oracle sees the knobs exactly as the GPU does (fp32-rounded)."""
    return oracle.HeadParams(loss_type=hp.loss_type, eps=f32(hp.eps),
                             max_importance_ratio=f32(hp.max_importance_ratio),
                             icepop_low=f32(hp.icepop_low), icepop_high=f32(hp.icepop_high),
                             adv_tau=f32(hp.adv_tau), temperature=f32(hp.temperature),
                             kl_coeff=f32(hp.kl_coeff), kl_estimator=hp.kl_estimator,
                             kl_staleness=hp.kl_staleness, entropy_coeff=f32(hp.entropy_coeff))


def ulp_bf16(x):
    x = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(x, 2.0 ** -126)))
    return 2.0 ** (e - 7)


def to_bf16(x):
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).double().numpy()


def grad_check(gpu, ref, reading: str, what: str, bounds=None, key="X", H=2048, block=8192, strict=True):
    """Row-blocked grad_check_block (bounded host memory for [V, H] arrays).  ``bounds`` is
    the oracle's dict (keys X / zX for dX, W / zW for dW; ``key`` names the first).
    ``strict=False`` only measures (a diagnostic reading)."""
    worst = 0.0
    n = np.asarray(ref).shape[0]
    b = None if bounds is None else np.asarray(bounds[key])
    zb = None if bounds is None else np.asarray(bounds["z" + key])
    for r0 in range(0, max(n, 1), block):
        sl = slice(r0, min(n, r0 + block))
        worst = max(worst, grad_check_block(np.asarray(gpu)[sl], np.asarray(ref)[sl], reading, what,
                                            None if b is None else b[sl], None if zb is None else zb[sl], H,
                                            strict))
    return worst


def grad_check_block(gpu, ref, reading: str, what: str, bound=None, zbound=None, H=2048, strict=True):
    """Assert the gradient bar (unless ``strict`` is False); returns the worst ratio
    err / allowed.

    readings: "element" (2 ulp of max(|ref|, 2^-8 rowmax)), "row" (2 ulp of the row max),
    "operand" (2 ulp of |ref| plus 2^-8 of the magnitude bound |G||W| / |G|^T|X|),
    "operand2" (2^-7 of the bound: both operands of each product rounded to bf16).
    Every reading also carries the logits' fp32-accumulation allowance carried into G
    (acc_tol on zbound, the |G| Z_t-weighted magnitude)."""
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    rb = to_bf16(ref)
    err = np.abs(gpu - rb)
    zallow = 0.0 if zbound is None else acc_tol(H, zbound)
    err = np.maximum(err - zallow, 0.0)
    rowmax = np.max(np.abs(ref), axis=1, keepdims=True)
    if reading in ("operand", "operand2"):
        frac = 2.0 ** -8 if reading == "operand" else 2.0 ** -7
        allowed = 2 * ulp_bf16(ref) * (ref != 0) + frac * np.asarray(bound, np.float64)
        ratio = np.where(allowed > 0, err / np.maximum(allowed, 1e-300), np.where(err > 0, np.inf, 0.0))
        worst = float(np.max(ratio)) if ratio.size else 0.0
        assert worst <= 1.0 or not strict, f"{what}: worst err/allowed = {worst:.3f} ({reading} reading)"
        return worst
    if reading == "element":
        allowed = 2 * ulp_bf16(np.maximum(np.abs(ref), 2.0 ** -8 * rowmax))
        ratio = err / allowed
    else:
        allowed = 2 * ulp_bf16(rowmax)
        ratio = np.max(err, axis=1, keepdims=True) / allowed
    ratio = np.where(rowmax > 0, ratio, np.where(np.max(err, axis=1, keepdims=True) > 0, np.inf, 0.0))
    worst = float(np.max(ratio)) if ratio.size else 0.0
    assert worst <= 1.0 or not strict, f"{what}: worst err/allowed = {worst:.3f} ({reading} reading)"
    return worst


def loss_prop_tol(ref: dict, inp: dict, op: oracle.HeadParams):
    """Per-token loss bar: the token's log-prob bar (logp_tol) carried through the loss to
    first order, |d loss_t| <= |adv_tau A_t| (|w_a| + sum_e |c_e|) lp_t + beta_t (sum_e u_e
    or 1) lp_t (+ entropy_coeff times the entropy's bar), doubled.  (A per-token loss is a
    difference of O(1) log-prob terms, so where it cancels a relative bar alone cannot
    hold.)"""
    off = np.asarray(inp["offsets"], np.int64)
    abs_c = np.add.reduceat(np.abs(ref["c_support"]), off[:-1]) if ref["c_support"].size else np.zeros(len(off) - 1)
    sum_u = np.add.reduceat(ref["u_support"], off[:-1]) if ref["u_support"].size else np.zeros(len(off) - 1)
    empty = off[1:] == off[:-1]
    abs_c = np.where(empty, 0.0, abs_c)
    sum_u = np.where(empty, 0.0, sum_u)
    kl_w = sum_u if op.kl_estimator == oracle.KL_EXACT else np.ones_like(sum_u)
    A = np.abs(op.adv_tau * np.asarray(inp["adv"], np.float64))
    H = np.asarray(inp["hidden"]).shape[1]
    lp = logp_tol(H, ref["zmax"], ref["lse_s"])
    ent = op.entropy_coeff * logp_tol(H, ref["zmax"], ref["lse"]) if op.entropy_coeff else 0.0
    return 2 * (lp * (A * (np.abs(ref["w_label"]) + abs_c) + np.asarray(ref["beta"]) * kl_w) + ent)


def loss_check(gpu, ref, prop_tol=None, what="loss"):
    """Aggregate loss within 1e-4 relative; per token within 1e-4 relative plus the
    propagated log-prob bar."""
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    tol = LOSS_REL * np.abs(ref) + (0.0 if prop_tol is None else np.asarray(prop_tol, np.float64))
    worst = float(np.max(np.abs(gpu - ref) / np.maximum(tol, 1e-30))) if ref.size else 0.0
    assert worst <= 1.0, f"{what}: worst err/allowed {worst:.3e}"
    tot_g, tot_r = float(gpu.sum()), float(ref.sum())
    assert abs(tot_g - tot_r) <= LOSS_REL * max(abs(tot_r), 1e-12) + 1e-6, (tot_g, tot_r)
    return worst


def weight_keep_fp64(logP, logq, op: oracle.HeadParams):
    """fp64 keep predicate of the oracle, evaluated on given (fp32) log-probs."""
    _, keep, _, _ = oracle.rl_head.rl_weight(np.asarray(logP, np.float64), np.asarray(logq, np.float64), op)
    return keep.astype(np.uint8)


def margin(logP, logq, op: oracle.HeadParams):
    """Distance of each pair from its nearest mask threshold (in the predicate's units)."""
    logP = np.asarray(logP, np.float64)
    logq = np.asarray(logq, np.float64)
    if op.loss_type == oracle.LOSS_IPO:
        return np.abs(np.abs(np.exp(logP) - np.exp(logq)) - op.eps)
    if op.loss_type == oracle.LOSS_ICEPOP:
        r = np.exp(logP - logq)
        return np.minimum(np.abs(r - op.icepop_low), np.abs(r - op.icepop_high)) / np.maximum(r, 1e-30)
    return np.full(logP.shape, np.inf)
