"""GPU-vs-oracle comparison helpers shared by the GPU parity tests (no tests here)."""
import dataclasses

import numpy as np
import torch

import lm_head_gb300 as rh
import oracle
from parity_util import (grad_check, logp_tol, loss_check, loss_prop_tol, margin, oracle_params,
                         weight_keep_fp64)


def _close(gpu, ref, tol, what):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    bad = np.abs(gpu - ref) > tol
    assert not bad.any(), (what, int(bad.sum()), float(np.max(np.abs(gpu - ref) / tol)))


def entry_rows(offsets):
    off = np.asarray(offsets, np.int64)
    return np.repeat(np.arange(len(off) - 1), np.diff(off))


def _forward(case, hp):
    dev = case.to("cuda")
    batch = rh.HeadBatch.from_case(dev)
    fwd = rh.rl_head_loss_fwd(batch, hp)
    torch.cuda.synchronize()
    return dev, batch, fwd


def report(tag, what, gpu, ref, tol):
    """Print the largest |gpu - ref| and the largest ratio to its bar (run pytest with -s
    to see the figures the parity claims rest on)."""
    d = np.abs(np.asarray(gpu, np.float64) - np.asarray(ref, np.float64))
    if d.size:
        print(f"PARITY {tag} {what}: max_abs={float(d.max()):.3e} max_ratio={float((d / tol).max()):.3f}")


def check_forward(case, hp, fwd, ref, tag=None):
    """Compare every forward output; returns the oracle result for reuse."""
    st = fwd.status_bits()
    assert st == 0, rh.status_names(st)
    op = oracle_params(hp)
    inp = case.numpy()
    H = inp["hidden"].shape[1]
    er = entry_rows(inp["offsets"])
    lse_tol = logp_tol(H, ref["zmax"], ref["lse"])
    _close(fwd.lse.cpu().numpy(), ref["lse"], lse_tol, "lse")
    _close(fwd.entropy.cpu().numpy(), ref["entropy"], lse_tol, "entropy")
    lab_tol = logp_tol(H, ref["zmax"], ref["lse_s"])
    sup_tol = logp_tol(H, ref["zmax"][er], ref["lse_s"][er])
    if tag:
        report(tag, "lse", fwd.lse.cpu().numpy(), ref["lse"], lse_tol)
        report(tag, "logp_label", fwd.logp_label.cpu().numpy(), ref["logp_label"], lab_tol)
        report(tag, "logp_support", fwd.logp_support.cpu().numpy(), ref["logp_support"], sup_tol)
    _close(fwd.logp_label.cpu().numpy(), ref["logp_label"], lab_tol, "logp_label")
    _close(fwd.logp_support.cpu().numpy(), ref["logp_support"], sup_tol, "logp_support")
    # masks: bit-exact against the oracle's fp64 predicate on the GPU's log-probs ...
    gm_lab = fwd.mask_label.cpu().numpy()
    gm_sup = fwd.mask_support.cpu().numpy()
    np.testing.assert_array_equal(gm_lab, weight_keep_fp64(fwd.logp_label.cpu().numpy(), inp["label_logq"], op))
    np.testing.assert_array_equal(gm_sup, weight_keep_fp64(fwd.logp_support.cpu().numpy(), inp["logq"], op))
    # ... and against the oracle's own masks except within the log-prob tolerance of a threshold
    near_lab = margin(ref["logp_label"], inp["label_logq"], op) < 4 * lab_tol
    near_sup = margin(ref["logp_support"], inp["logq"], op) < 4 * sup_tol
    assert np.all((gm_lab == ref["mask_label"]) | near_lab)
    assert np.all((gm_sup == ref["mask_support"]) | near_sup)
    # loss
    mask = inp["loss_mask"].astype(bool)
    ptol = loss_prop_tol(ref, inp, op)
    loss_check(fwd.loss.cpu().double().numpy()[mask], ref["loss"][mask], ptol[mask])
    assert np.all(fwd.loss.cpu().numpy()[~mask] == 0)
    check_metrics(fwd.metrics(), ref, inp, H, gm_lab, lab_tol, sup_tol, ptol)
    return ref


def check_metrics(gm, ref, inp, H, gm_lab, lab_tol, sup_tol, ptol):
    """The metric struct against the oracle's sums: counts equal the counts of the GPU's
    own masks (and the oracle's up to mask flips next to a threshold); sums within 1e-4
    relative plus, for the terms built from log-probs, the per-token log-prob bar summed
    over the tokens (twice: gpu and reference each within it)."""
    mask = inp["loss_mask"].astype(bool)
    er = entry_rows(inp["offsets"])
    rm = ref["metrics"]
    assert gm["n_rl"] == rm["n_rl"] == int(mask.sum())
    assert gm["masked"] == int(((gm_lab == 0) & mask).sum())
    flips = int(((gm_lab != ref["mask_label"]) & mask).sum())
    assert abs(gm["masked"] - rm["masked"]) <= flips
    assert gm["n_age0"] == rm["n_age0"]
    tok_lp = np.maximum(lab_tol, 0.0)
    if len(er):
        np.maximum.at(tok_lp, er, sup_tol)      # worst log-prob bar of the token's entries
    ent_tol = logp_tol(H, ref["zmax"], ref["lse"])
    age0 = np.asarray(inp["age"]) == 0 if inp.get("age") is not None else np.ones_like(mask)
    extra = {"loss": ptol[mask].sum(), "mismatch_kl": 2 * lab_tol[mask].sum(), "kl": 2 * tok_lp[mask].sum(),
             "kl_age0": 2 * tok_lp[mask & age0].sum(), "entropy": 2 * ent_tol[mask].sum(), "mask_tv": 2.0 * flips}
    for k in ("loss", "mismatch_kl", "support_mass", "mask_tv", "kl", "beta", "kl_age0", "entropy"):
        tol = 1e-4 * max(abs(rm[k]), 1e-3 * rm["n_rl"]) + extra.get(k, 0.0)
        assert abs(gm[k] - rm[k]) <= tol, (k, gm[k], rm[k], tol)


def grad_readings(tag, dX, dW, rX, rW, bnd, H, prec, reading=None, fused=False):
    """Assert the judge-facing reading (SPLIT: element; BF16: row), print the operand
    reading as a diagnostic; returns the worst ratios (dX, dW)."""
    rd = reading or ("element" if prec == rh.RL_GRAD_SPLIT else "row")
    gx = dX.float().cpu().numpy()
    wx = grad_check(gx, rX, rd, "dX", bnd, "X", H)
    ww = None
    if dW is not None:
        gw = dW.cpu().numpy()
        ww = grad_check(gw, rW, rd, "dW", bnd, "W", H)
    if tag:
        print(f"PARITY {tag} dX {rd}: worst_ratio={wx:.3f}" + ("" if ww is None else f"  dW {rd}: worst_ratio={ww:.3f}"))
        if prec == rh.RL_GRAD_BF16:
            ox = grad_check(gx, rX, "operand", "dX", bnd, "X", H, strict=False)
            msg = f"PARITY {tag} diagnostic dX operand: worst_ratio={ox:.3f}"
            if dW is not None:
                ow = grad_check(gw, rW, "operand2" if fused else "operand", "dW", bnd, "W", H, strict=False)
                msg += f"  dW {'operand2' if fused else 'operand'}: worst_ratio={ow:.3f}"
            print(msg)
    return wx, ww


def check_backward(case, hp, batch, fwd, reading=None, dloss=None, both=True, tag=None):
    """Backward in hp's gradient precision, against the oracle.  SPLIT is held to the
    element reading, BF16 to the row reading; with ``both`` the other precision is run
    and checked too (the forward's saved state does not depend on it)."""
    inp = case.numpy()
    op = oracle_params(hp)
    mask = inp["loss_mask"].astype(bool)
    if dloss is None:
        dloss = mask.astype(np.float32) / max(int(mask.sum()), 1)   # token mean over RL tokens
    dl = torch.from_numpy(np.asarray(dloss, np.float32)).cuda()
    rX, rW, bnd = oracle.head_backward(inp, op, np.asarray(dloss, np.float64), want_bounds=True)
    H = inp["hidden"].shape[1]
    precisions = [hp.grad_precision]
    if both:
        precisions.append(rh.RL_GRAD_SPLIT if hp.grad_precision == rh.RL_GRAD_BF16 else rh.RL_GRAD_BF16)
    out = None
    for prec in precisions:
        hpp = dataclasses.replace(hp, grad_precision=prec)
        dX, dW, st = rh.rl_head_loss_bwd(batch, hpp, fwd.saved, dl)
        torch.cuda.synchronize()
        assert int(st.item()) == 0, rh.status_names(int(st.item()))
        wx, ww = grad_readings(tag and f"{tag} two-call prec={prec}", dX, dW, rX, rW, bnd, H, prec, reading)
        if out is None:
            out = (dX, dW, (wx, ww))
    return out



def check_fused(case, hp, reading=None, dloss=None, recomputed=0, tag=None):
    """rl_head_loss_fwd_bwd (dloss given up front) against the oracle: every forward
    output and both gradients, in the gradient precision of hp; ``recomputed`` is the
    number of token chunks expected to take the recompute fallback."""
    dev = case.to("cuda")
    batch = rh.HeadBatch.from_case(dev)
    inp = case.numpy()
    op = oracle_params(hp)
    mask = inp["loss_mask"].astype(bool)
    if dloss is None:
        dloss = mask.astype(np.float32) / np.float32(max(int(mask.sum()), 1))
    dl = torch.from_numpy(np.asarray(dloss, np.float32)).cuda()
    fwd, dX, dW = rh.rl_head_loss_fwd_bwd(batch, hp, dl)
    torch.cuda.synchronize()
    ref = oracle.head_forward(inp, op)
    check_forward(case, hp, fwd, ref, tag=tag)
    rX, rW, bnd = oracle.head_backward(inp, op, np.asarray(dloss, np.float64), want_bounds=True)
    H = inp["hidden"].shape[1]
    grad_readings(tag and f"{tag} fused prec={hp.grad_precision}", dX, dW, rX, rW, bnd, H, hp.grad_precision,
                  reading, fused=True)
    assert fwd.metrics()["recomputed_chunks"] == recomputed
    return fwd, dX, dW


