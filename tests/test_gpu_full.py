"""GPU parity at the full head shapes (H=2048, V=151936) and at the full 64k-token batch.

* c2 / c3 / c4 shaped batches with ~300 tokens (ragged tail, several 256-row pair tiles,
  the 594 vocabulary tiles): every output element against the fp64 oracle.
* The full c4 batch (65536 tokens) in the launch configuration bench.py times (the fused
  call, default token chunk, default GEMM mode): sampled tokens' outputs and dX rows
  against the oracle one by one; counts that hold at any size; the identity
  <dW, W> = <dX, X> (both equal T * sum G*z); the fused backward against the two-call
  (recompute) backward.
* The full c2 (4096 tokens) and c3 (16384 tokens) batches the same way; c3's sparse CSR
  backward against its dense backward over the whole batch.
* Degenerate cases: empty batch, one token, no RL tokens, one draw per row, a vocabulary
  that is not a multiple of the tile width, the smallest hidden size.
"""
import numpy as np
import pytest
import torch

import lm_head_gb300 as rh
import oracle
import workloads
import oracle_pool
from gpu_checks import _forward, check_backward, check_forward, check_fused, grad_readings, report
from parity_util import grad_check, logp_tol, loss_check, loss_prop_tol, margin, oracle_params, weight_keep_fp64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from lm_head_gb300 import build
    build.build()
    rh.load()


def _hp_c2(**kw):
    return rh.HeadParams(loss_type=rh.RL_LOSS_ICEPOP, icepop_low=0.5, icepop_high=2.0, kl_coeff=0.0,
                         bwd_mode=rh.RL_BWD_DENSE, **kw)


def _hp_c3(**kw):
    return rh.HeadParams(loss_type=rh.RL_LOSS_IPO, eps=0.3, max_importance_ratio=10.0, kl_coeff=0.0, **kw)


def _hp_c4(**kw):
    return rh.HeadParams(loss_type=rh.RL_LOSS_IPO, eps=0.3, max_importance_ratio=10.0, kl_coeff=0.01,
                         kl_estimator=rh.RL_KL_EXACT, kl_staleness=rh.RL_STALE_INV_SQRT, **kw)


@pytest.mark.parametrize("variant", ["literal", "pages"])
def test_c2_shapes_replay_top_p(variant):
    """Replayed top-p 0.97 supports (literal scales keep ~127k ids per token), icepop."""
    case = workloads.make_head_case("c2", n_tokens=264, device="cuda", variant=variant, chunk=132)
    hp = _hp_c2(all_replayed=0)
    check_fused(case, hp, tag=f"c2-shape-{variant}")
    dev, batch, fwd = _forward(case, hp)
    check_backward(case, hp, batch, fwd, both=False, tag=f"c2-shape-{variant}")


def test_c3_shapes_sparse_backward_against_dense_and_oracle():
    case = workloads.make_head_case("c3", n_tokens=300, device="cuda", variant="pages", chunk=150)
    hp_s = _hp_c3(all_replayed=1)                        # AUTO -> sparse CSR matmul
    hp_d = _hp_c3(bwd_mode=rh.RL_BWD_DENSE)
    fs, dXs, dWs = check_fused(case, hp_s, reading="element", tag="c3-shape-sparse")
    fd, dXd, dWd = check_fused(case, hp_d, tag="c3-shape-dense")
    torch.testing.assert_close(dWs, dWd, rtol=1e-5, atol=1e-9)
    torch.testing.assert_close(dXs.float(), dXd.float(), rtol=1e-2, atol=1e-8)


@pytest.mark.parametrize("prec", [rh.RL_GRAD_BF16, rh.RL_GRAD_SPLIT])
def test_c4_shapes_draws_exact_kl(prec):
    """K=16 untruncated draws, exact KL with inv_sqrt staleness: the dense softmax part is
    live on every row, across two 256-row GEMM tiles and a ragged tail."""
    case = workloads.make_head_case("c4", n_tokens=300, device="cuda", chunk=300)
    hp = _hp_c4(bwd_mode=rh.RL_BWD_DENSE, grad_precision=prec)
    check_fused(case, hp, tag="c4-shape")
    if prec == rh.RL_GRAD_BF16:
        dev, batch, fwd = _forward(case, hp)
        check_backward(case, hp, batch, fwd, both=False, tag="c4-shape")


def _sampled_rows(N, seed):
    """Tile edges (128-row halves, 256-row pairs, 8k / 16k chunks), the ends, random rows."""
    rng = np.random.default_rng(seed)
    fixed = [r for r in (0, 1, 127, 128, 255, 256, 8191, 8192, 16383, 16384, 32767, 49152, N // 2, N - 1)
             if r < N]
    return np.unique(np.r_[fixed, rng.integers(0, N, 13)]).astype(np.int64)


def _check_sampled_rows(case, hp, fwd, dX, dloss_t, rows, reading=None, tag=None):
    """Sampled tokens' forward outputs and dX rows against the oracle, one by one."""
    N, H = case.N, case.H
    inp = case.numpy()
    op = oracle_params(hp)
    ref = oracle.head_forward(inp, op, rows=rows, chunk=8)
    off = inp["offsets"]
    ent = np.concatenate([np.arange(off[t], off[t + 1]) for t in rows])
    ltol = logp_tol(H, ref["zmax"], ref["lse"])
    assert np.all(np.abs(fwd.lse.cpu().double().numpy()[rows] - ref["lse"]) <= ltol)
    assert np.all(np.abs(fwd.entropy.cpu().double().numpy()[rows] - ref["entropy"]) <= ltol)
    lab_tol = logp_tol(H, ref["zmax"], ref["lse_s"])
    assert np.all(np.abs(fwd.logp_label.cpu().double().numpy()[rows] - ref["logp_label"]) <= lab_tol)
    er = np.repeat(np.arange(len(rows)), off[rows + 1] - off[rows])
    sup_tol = logp_tol(H, ref["zmax"][er], ref["lse_s"][er])
    assert np.all(np.abs(fwd.logp_support.cpu().double().numpy()[ent] - ref["logp_support"]) <= sup_tol)
    if tag:
        report(tag, "lse", fwd.lse.cpu().numpy()[rows], ref["lse"], ltol)
        report(tag, "logp_label", fwd.logp_label.cpu().numpy()[rows], ref["logp_label"], lab_tol)
        report(tag, "logp_support", fwd.logp_support.cpu().numpy()[ent], ref["logp_support"], sup_tol)
    # masks: bit-exact against the fp64 predicate on the GPU's log-probs, and equal to the
    # oracle's own except within the log-prob tolerance of a threshold
    gm_lab = fwd.mask_label.cpu().numpy()[rows]
    gm_sup = fwd.mask_support.cpu().numpy()[ent]
    np.testing.assert_array_equal(gm_lab, weight_keep_fp64(fwd.logp_label.cpu().numpy()[rows],
                                                           inp["label_logq"][rows], op))
    np.testing.assert_array_equal(gm_sup, weight_keep_fp64(fwd.logp_support.cpu().numpy()[ent], inp["logq"][ent], op))
    assert np.all((gm_lab == ref["mask_label"]) | (margin(ref["logp_label"], inp["label_logq"][rows], op) < 4 * lab_tol))
    sub = {k: (v[rows] if isinstance(v, np.ndarray) and v.shape[:1] == (N,) else v) for k, v in inp.items()}
    ptol = loss_prop_tol(dict(ref, c_support=ref["c_support"], u_support=ref["u_support"]),
                         dict(sub, offsets=np.r_[0, np.cumsum(off[rows + 1] - off[rows])]), op)
    loss_check(fwd.loss.cpu().double().numpy()[rows], ref["loss"], ptol)
    dl = dloss_t.cpu().double().numpy()
    rX, _, bnd = oracle.head_backward(inp, op, dl, rows=rows, want_dW=False, want_bounds=True, chunk=8)
    grad_readings(tag, dX[rows], None, rX, None, bnd, H, hp.grad_precision, reading)
    return inp


def test_c4_full_size_sampled():
    """The 64k-token batch exactly as bench.py runs it; sampled outputs vs the oracle."""
    case = workloads.make_head_case("c4", device="cuda", seed=workloads.BASE_SEED + 4)
    N = case.N
    hp = _hp_c4(bwd_mode=rh.RL_BWD_DENSE)
    batch = rh.HeadBatch.from_case(case)
    dloss_t = (case.loss_mask.float() / case.loss_mask.float().sum()).contiguous()
    fwd, dX, dW = rh.rl_head_loss_fwd_bwd(batch, hp, dloss_t)
    torch.cuda.synchronize()
    assert fwd.status_bits() == 0, rh.status_names(fwd.status_bits())
    # dX rows against the oracle (row reading of the bf16 bar)
    inp = _check_sampled_rows(case, hp, fwd, dX, dloss_t, _sampled_rows(N, 7), tag="c4-full")
    H = case.H
    # sampled vocabulary rows of dW, accumulated over the eight 8k-token chunks, against
    # the oracle's dW over the whole batch (its full-vocabulary logsumexp of every token:
    # about 4e13 fp64 flop, spread over the host's cores)
    ids = case.ids.cpu().numpy()
    counts = np.bincount(ids, minlength=case.V)
    rng = np.random.default_rng(17)
    vrows = np.unique(np.r_[0, 1, 255, 256, 257, case.V // 2, case.V - 257, case.V - 1,
                            np.argsort(counts)[-6:],                      # the most-drawn ids
                            np.flatnonzero(counts == 0)[:4],              # never drawn: dense part only
                            rng.integers(0, case.V, 12)]).astype(np.int64)
    op = oracle_params(hp)
    rWv, bw = oracle_pool.dW_rows(inp, op, dloss_t.cpu().double().numpy(), vrows)
    gW = dW[torch.from_numpy(vrows).cuda()]
    grad_readings("c4-full dW-rows", gW, None, rWv, None, {"X": bw["W"], "zX": bw["zW"]}, H,
                  hp.grad_precision, fused=True)
    # counts that hold at any size
    m = fwd.metrics()
    assert m["n_rl"] == N
    assert m["masked"] == int((fwd.mask_label == 0).sum().item())
    assert m["n_age0"] == int((case.age == 0).sum().item())
    # <dW, W> = <dX, X> = T sum G z
    Wd = case.W.double()
    Xd = case.hidden.double()
    lhs = float((dW.double() * Wd).sum())
    rhs = float((dX.double() * Xd).sum())
    mag = float((dX.double() * Xd).abs().sum())
    assert abs(lhs - rhs) <= 1e-2 * mag, (lhs, rhs, mag)
    # the fused backward agrees with the two-call (recompute) backward
    f2 = rh.rl_head_loss_fwd(batch, hp)
    dX2, dW2, st = rh.rl_head_loss_bwd(batch, hp, f2.saved, dloss_t)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    # same arithmetic, but the fused call runs the forward per 8k-token chunk (its own
    # vocabulary split count), so the logsumexp partials combine in another order: each
    # call's log-probs lie within logp_tol of the oracle, so per token the two losses differ
    # by at most that bar twice, carried through |dloss/dlogP| <= |adv_tau A| (w + sum|c|)
    # + beta sum u <= |adv_tau A| 2 cap + beta (ipo: w <= cap; K draws: sum u = 1).  Z_t
    # is bounded here by Cauchy-Schwarz, |z_tj| <= |h_t| max_j |W_j|.
    zb = (case.hidden.double().norm(dim=1) * case.W.double().norm(dim=1).max()).cpu().numpy()
    lse2 = f2.lse.cpu().double().numpy()
    np.testing.assert_array_less(np.abs(lse2 - fwd.lse.cpu().double().numpy()), 2 * logp_tol(H, zb, lse2))
    gain = np.abs(hp.adv_tau * inp["adv"]) * 2 * hp.max_importance_ratio + hp.kl_coeff
    l1, l2 = fwd.loss.cpu().double().numpy(), f2.loss.cpu().double().numpy()
    np.testing.assert_array_less(np.abs(l1 - l2), gain * 2 * logp_tol(H, zb, lse2) + 1e-4 * np.abs(l2))
    scale = dW2.abs().max().item()
    assert (dW - dW2).abs().max().item() <= 2 ** -7 * scale
    assert (dX.float() - dX2.float()).abs().max().item() <= 2 ** -7 * dX2.float().abs().max().item()


def test_c2_full_size_sampled():
    """The 4096-token replayed top-p 0.97 batch (the pages' sharp rows), icepop, through
    the fused call in its default launch shape: sampled outputs and dX rows vs the oracle,
    <dW, W> = <dX, X>."""
    case = workloads.make_head_case("c2", device="cuda", variant="pages")
    assert case.N == 4096
    hp = _hp_c2(all_replayed=0)
    batch = rh.HeadBatch.from_case(case)
    dloss_t = (case.loss_mask.float() / case.loss_mask.float().sum()).contiguous()
    fwd, dX, dW = rh.rl_head_loss_fwd_bwd(batch, hp, dloss_t)
    torch.cuda.synchronize()
    assert fwd.status_bits() == 0, rh.status_names(fwd.status_bits())
    _check_sampled_rows(case, hp, fwd, dX, dloss_t, _sampled_rows(case.N, 8), tag="c2-full")
    lhs = float((dW.double() * case.W.double()).sum())
    rhs = float((dX.double() * case.hidden.double()).sum())
    assert abs(lhs - rhs) <= 1e-2 * float((dX.double() * case.hidden.double()).abs().sum())


def test_c3_full_size_sparse_against_dense():
    """The 16384-token replayed top-p batch with exact centering, ipo: the deterministic
    CSR sparse backward against the dense backward over the whole batch (dW and dX), and
    the sparse call's sampled outputs and dX rows vs the oracle (element reading: the
    sparse gradient is formed in fp32)."""
    case = workloads.make_head_case("c3", device="cuda", variant="pages")
    assert case.N == 16384
    batch = rh.HeadBatch.from_case(case)
    dloss_t = (case.loss_mask.float() / case.loss_mask.float().sum()).contiguous()
    hp_s = _hp_c3(all_replayed=1)                        # AUTO -> sparse CSR matmul
    hp_d = _hp_c3(bwd_mode=rh.RL_BWD_DENSE)
    fs, dXs, dWs = rh.rl_head_loss_fwd_bwd(batch, hp_s, dloss_t)
    fd, dXd, dWd = rh.rl_head_loss_fwd_bwd(batch, hp_d, dloss_t)
    torch.cuda.synchronize()
    assert fs.status_bits() == 0 and fd.status_bits() == 0
    torch.testing.assert_close(fs.loss, fd.loss, rtol=1e-5, atol=1e-6)   # the same forward arithmetic
    torch.testing.assert_close(dWs, dWd, rtol=1e-5, atol=1e-9)
    torch.testing.assert_close(dXs.float(), dXd.float(), rtol=1e-2, atol=1e-8)
    _check_sampled_rows(case, hp_s, fs, dXs, dloss_t, _sampled_rows(case.N, 9), reading="element",
                        tag="c3-full-sparse")
    _check_sampled_rows(case, hp_d, fd, dXd, dloss_t, _sampled_rows(case.N, 9), tag="c3-full-dense")


def _small(N, V=1000, H=64, **kw):
    return workloads.make_head_case("c1", n_tokens=N, H=H, V=V, hidden_scale=4.0, noise=0.5, **kw)


def test_empty_batch():
    case = _small(8)
    dev = case.to("cuda")
    z = lambda t: t[:0]
    batch = rh.HeadBatch(z(dev.hidden), dev.W, z(dev.labels), z(dev.label_logq), z(dev.adv), dev.offsets[:1] * 0,
                         z(dev.ids), z(dev.logq), z(dev.replayed))
    hp = rh.HeadParams(bwd_mode=rh.RL_BWD_DENSE)
    dW = torch.full((case.V, case.H), 7.0, device="cuda")
    fwd, dX, dW = rh.rl_head_loss_fwd_bwd(batch, hp, torch.zeros(0, device="cuda"), dW=dW)
    torch.cuda.synchronize()
    assert fwd.status_bits() == 0 and float(dW.abs().max()) == 0.0


@pytest.mark.parametrize("N,V,H,K", [(1, 1000, 64, 16), (77, 1000, 64, 1), (130, 1024, 128, 3)])
def test_small_and_ragged_shapes(N, V, H, K):
    case = _small(N, V=V, H=H, K=K, loss_mask_frac=0.2, age_max=3, seed=N + K)
    hp = _hp_c4(bwd_mode=rh.RL_BWD_DENSE)
    check_fused(case, hp)
    dev, batch, fwd = _forward(case, hp)
    check_backward(case, hp, batch, fwd)


def test_no_rl_tokens():
    case = _small(64, loss_mask_frac=1.0)
    assert int(case.loss_mask.sum()) == 0
    hp = _hp_c4(bwd_mode=rh.RL_BWD_DENSE)
    dev = case.to("cuda")
    batch = rh.HeadBatch.from_case(dev)
    fwd, dX, dW = rh.rl_head_loss_fwd_bwd(batch, hp, torch.zeros(case.N, device="cuda"))
    torch.cuda.synchronize()
    assert float(fwd.loss.abs().max()) == 0.0 and float(dX.float().abs().max()) == 0.0
    assert float(dW.abs().max()) == 0.0 and fwd.metrics()["n_rl"] == 0


def test_sampler_equals_trainer_and_zero_advantages():
    """q = p (sampler logits = trainer logits, no noise) and A = 0 on every third token:
    every weight is 1 up to rounding, nothing is masked, the mismatch KL vanishes to the
    log-prob bar, and tokens with A = 0 keep only their KL part (the oracle agrees)."""
    case = workloads.make_head_case("c1", n_tokens=200, H=128, V=1024, hidden_scale=4.0, noise=0.0, age_max=2,
                                    seed=77)
    case.adv[::3] = 0.0
    hp = _hp_c4(bwd_mode=rh.RL_BWD_DENSE)
    fwd, dX, dW = check_fused(case, hp)
    m = fwd.metrics()
    assert m["masked"] == 0
    assert abs(m["mismatch_kl"]) <= 1e-4 * m["n_rl"]
    dev, batch, fwd2 = _forward(case, hp)
    check_backward(case, hp, batch, fwd2)
