"""GPU parity of the fused LM head + RL loss (through the C-ABI) against the fp64 oracle.

Inputs come from the seeded generators in workloads/ (the same tensors feed both sides).
Sizes here are ones the oracle finishes in seconds while still spanning several 128 x 256
tensor-core tiles and a ragged tail.
"""
import dataclasses

import numpy as np
import pytest
import torch

import lm_head_gb300 as rh
import oracle
import workloads
from gpu_checks import _forward, check_backward, check_forward, check_fused
from parity_util import oracle_params

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from lm_head_gb300 import build
    build.build()
    rh.load()


C1_IPO = dict(loss_type=rh.RL_LOSS_IPO, eps=0.3, max_importance_ratio=10.0, kl_coeff=0.0)


def test_c1_forward_and_dense_backward():
    """The tiny config: N=256, H=128, V=1024, K=16 draws, ipo eps 0.3, dense backward."""
    case = workloads.make_head_case("c1")
    hp = rh.HeadParams(**C1_IPO, bwd_mode=rh.RL_BWD_DENSE)
    dev, batch, fwd = _forward(case, hp)
    ref = oracle.head_forward(case.numpy(), oracle_params(hp))
    check_forward(case, hp, fwd, ref)
    check_backward(case, hp, batch, fwd)


@pytest.mark.parametrize("loss_type", [rh.RL_LOSS_IPO, rh.RL_LOSS_ICEPOP, rh.RL_LOSS_REINFORCE])
def test_c1_mask_stress(loss_type):
    """c1 shapes with sharp logits and a noisy sampler, so masks and caps are exercised;
    ragged token count, some non-RL tokens, exact KL with inv_sqrt staleness."""
    case = workloads.make_head_case("c1", n_tokens=300, hidden_scale=10.0, noise=1.0, loss_mask_frac=0.1,
                                    age_max=4, seed=11 + loss_type)
    hp = rh.HeadParams(loss_type=loss_type, eps=0.2, max_importance_ratio=2.0, icepop_low=0.5, icepop_high=2.0,
                       adv_tau=0.7, kl_coeff=0.05, kl_estimator=rh.RL_KL_EXACT,
                       kl_staleness=rh.RL_STALE_INV_SQRT, bwd_mode=rh.RL_BWD_DENSE)
    dev, batch, fwd = _forward(case, hp)
    ref = oracle.head_forward(case.numpy(), oracle_params(hp))
    check_forward(case, hp, fwd, ref)
    assert 0 < int(fwd.mask_support.sum()) < case.nnz or loss_type == rh.RL_LOSS_REINFORCE
    check_backward(case, hp, batch, fwd)


def test_c1_split_precision_meets_element_reading():
    case = workloads.make_head_case("c1", n_tokens=200, hidden_scale=4.0, noise=0.5, seed=21)
    hp = rh.HeadParams(**C1_IPO, bwd_mode=rh.RL_BWD_DENSE, grad_precision=rh.RL_GRAD_SPLIT)
    dev, batch, fwd = _forward(case, hp)
    ref = oracle.head_forward(case.numpy(), oracle_params(hp))
    check_forward(case, hp, fwd, ref)
    check_backward(case, hp, batch, fwd)


def test_k1_estimator_and_temperature():
    case = workloads.make_head_case("c1", n_tokens=130, hidden_scale=3.0, noise=0.3, temperature=0.7, seed=31)
    hp = rh.HeadParams(loss_type=rh.RL_LOSS_ICEPOP, kl_coeff=0.1, kl_estimator=rh.RL_KL_K1, temperature=0.7,
                       bwd_mode=rh.RL_BWD_DENSE)
    dev, batch, fwd = _forward(case, hp)
    ref = oracle.head_forward(case.numpy(), oracle_params(hp))
    check_forward(case, hp, fwd, ref)
    check_backward(case, hp, batch, fwd)


@pytest.mark.parametrize("loss_type", [rh.RL_LOSS_IPO, rh.RL_LOSS_REINFORCE])
def test_replayed_support_sparse_equals_dense_and_oracle(loss_type):
    """Replayed top-p supports (u = q, renormalised P): the sparse CSR-matmul backward
    matches the dense one to fp32 rounding and both match the oracle."""
    case = workloads.make_head_case("c1", n_tokens=260, support="replay", top_p=0.9, hidden_scale=6.0,
                                    noise=0.3, seed=41 + loss_type)
    base = dict(loss_type=loss_type, eps=0.3, kl_coeff=0.02, all_replayed=1)
    hp_d = rh.HeadParams(**base, bwd_mode=rh.RL_BWD_DENSE)
    hp_s = rh.HeadParams(**base, bwd_mode=rh.RL_BWD_SPARSE)
    dev, batch, fwd_d = _forward(case, hp_d)
    ref = oracle.head_forward(case.numpy(), oracle_params(hp_d))
    check_forward(case, hp_d, fwd_d, ref)
    dXd, dWd, _ = check_backward(case, hp_d, batch, fwd_d, both=False)
    fwd_s = rh.rl_head_loss_fwd(batch, hp_s)
    dXs, dWs, _ = check_backward(case, hp_s, batch, fwd_s, both=False)
    torch.testing.assert_close(dWs, dWd, rtol=1e-5, atol=1e-7)
    torch.testing.assert_close(dXs.float(), dXd.float(), rtol=1e-2, atol=1e-6)


def test_reinforce_draws_sparse_without_kl():
    case = workloads.make_head_case("c1", n_tokens=256, K=8, seed=51)
    hp = rh.HeadParams(loss_type=rh.RL_LOSS_REINFORCE, kl_coeff=0.0)   # AUTO -> sparse
    dev, batch, fwd = _forward(case, hp)
    ref = oracle.head_forward(case.numpy(), oracle_params(hp))
    check_forward(case, hp, fwd, ref)
    check_backward(case, hp, batch, fwd)


def test_determinism_bitwise():
    case = workloads.make_head_case("c1", n_tokens=300, hidden_scale=5.0, noise=0.5, seed=61)
    hp = rh.HeadParams(loss_type=rh.RL_LOSS_IPO, kl_coeff=0.01, bwd_mode=rh.RL_BWD_DENSE)
    dev, batch, f1 = _forward(case, hp)
    f2 = rh.rl_head_loss_fwd(batch, hp)
    dl = torch.full((case.N,), 1.0 / case.N, device="cuda")
    a = rh.rl_head_loss_bwd(batch, hp, f1.saved, dl)
    b = rh.rl_head_loss_bwd(batch, hp, f2.saved, dl)
    torch.cuda.synchronize()
    assert torch.equal(f1.loss, f2.loss) and torch.equal(f1.logp_support, f2.logp_support)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_corrupt_support_sets_status_bits_without_trapping():
    case = workloads.make_head_case("c1", n_tokens=128, support="replay", top_p=0.9, hidden_scale=6.0, seed=71)
    hp = rh.HeadParams(loss_type=rh.RL_LOSS_IPO, all_replayed=1)
    bad = case.to("cuda")
    ids = bad.ids.clone()
    ids[3] = case.V + 5                     # out-of-range id
    offsets = bad.offsets.clone()
    logq = bad.logq.clone()
    logq[0] = float("nan")                  # non-finite log q
    labels = bad.labels.clone()
    r = 7                                   # a replayed row whose label is not in its support
    row = ids[int(offsets[r]):int(offsets[r + 1])].cpu().tolist()
    labels[r] = next(v for v in range(case.V) if v not in row)
    batch = rh.HeadBatch(bad.hidden, bad.W, labels, bad.label_logq, bad.adv, offsets, ids, logq, bad.replayed)
    fwd = rh.rl_head_loss_fwd(batch, hp)
    torch.cuda.synchronize()
    names = rh.status_names(fwd.status_bits())
    for n in ("ID_RANGE", "LOGQ", "LABEL_MISSING"):
        assert n in names, names
    # offsets that run past nnz: flagged, and no out-of-bounds access brings the context down
    off2 = offsets.clone()
    off2[-1] = off2[-1] + 1000
    b2 = rh.HeadBatch(bad.hidden, bad.W, bad.labels, bad.label_logq, bad.adv, off2, bad.ids, bad.logq, bad.replayed)
    st = rh.rl_validate_support(b2)
    torch.cuda.synchronize()
    assert "OFFSETS" in rh.status_names(int(st.item()))
    # the context still works
    ok = rh.rl_head_loss_fwd(rh.HeadBatch.from_case(bad), hp)
    torch.cuda.synchronize()
    assert ok.status_bits() == 0


@pytest.mark.parametrize("prec", [rh.RL_GRAD_BF16, rh.RL_GRAD_SPLIT])
@pytest.mark.parametrize("loss_type", [rh.RL_LOSS_IPO, rh.RL_LOSS_ICEPOP])
def test_fused_forward_backward_multi_chunk(loss_type, prec):
    """Fused path over 3 token chunks (128, 128, 44): forward outputs and gradients."""
    case = workloads.make_head_case("c1", n_tokens=300, hidden_scale=8.0, noise=0.7, loss_mask_frac=0.1,
                                    age_max=4, seed=81 + loss_type)
    hp = rh.HeadParams(loss_type=loss_type, eps=0.2, max_importance_ratio=3.0, kl_coeff=0.03,
                       kl_estimator=rh.RL_KL_EXACT, kl_staleness=rh.RL_STALE_INV_SQRT, bwd_mode=rh.RL_BWD_DENSE,
                       grad_precision=prec, token_chunk=128)
    check_fused(case, hp)


def test_fused_c1_and_matches_unfused():
    """The tiny config through the fused call; its gradients agree with the recompute
    path to bf16 rounding of G."""
    case = workloads.make_head_case("c1")
    hp = rh.HeadParams(**C1_IPO, bwd_mode=rh.RL_BWD_DENSE)
    fwd, dX, dW = check_fused(case, hp)
    dev = case.to("cuda")
    batch = rh.HeadBatch.from_case(dev)
    f2 = rh.rl_head_loss_fwd(batch, hp)
    dl = torch.full((case.N,), 1.0 / case.N, device="cuda")
    dX2, dW2, _ = rh.rl_head_loss_bwd(batch, hp, f2.saved, dl)
    torch.cuda.synchronize()
    assert torch.equal(fwd.loss, f2.loss) and torch.equal(fwd.logp_support, f2.logp_support)
    scale = dW2.abs().max().item()
    assert (dW - dW2).abs().max().item() <= 2 ** -7 * scale


def test_fused_recompute_fallback_when_label_far_below_max():
    """Rows whose label logit lies ~86 nats below the row's max logit: numerators stored
    relative to the label would leave bf16's range, so the fused call sends their token
    chunk (and only it) through the gated logit recompute.  Everything still matches the
    oracle, and the metrics count the one chunk."""
    case = workloads.make_head_case("c1", n_tokens=300, hidden_scale=60.0, noise=0.1, seed=121)
    inp = case.numpy()
    z = inp["hidden"] @ inp["W"].T
    for t in (140, 141, 200):   # all in the second chunk of 128 tokens
        v = int(np.argmin(z[t]))
        lse = float(np.max(z[t]) + np.log(np.sum(np.exp(z[t] - np.max(z[t])))))
        case.labels[t] = v
        case.label_logq[t] = float(z[t, v] - lse)
    hp = rh.HeadParams(loss_type=rh.RL_LOSS_IPO, eps=0.3, max_importance_ratio=10.0, kl_coeff=0.02,
                       bwd_mode=rh.RL_BWD_DENSE, token_chunk=128)
    check_fused(case, hp, recomputed=1)


def _concat_cases(a, b):
    """Tokens of a, then tokens of b, on a's weights (b's sampler evidence stays valid
    input: the checks on it do not involve the trainer's weights)."""
    import dataclasses as dc
    cat = lambda f: torch.cat([getattr(a, f), getattr(b, f)])
    off = torch.cat([a.offsets, b.offsets[1:] + a.offsets[-1]])
    return dc.replace(a, hidden=cat("hidden"), labels=cat("labels"), label_logq=cat("label_logq"), adv=cat("adv"),
                      loss_mask=cat("loss_mask"), age=cat("age"), replayed=cat("replayed"), offsets=off,
                      ids=cat("ids"), logq=cat("logq"))


def test_fused_mixed_replayed_and_draw_rows():
    """Dense fused backward over draw rows (spikes folded into the dense operand) and
    replayed rows (no dense part: spikes on the gated sparse path) in one batch; chunks of
    128 give one all-draw chunk, one mixed, one all-replayed."""
    a = workloads.make_head_case("c1", n_tokens=160, hidden_scale=8.0, noise=0.7, age_max=4, seed=131)
    b = workloads.make_head_case("c1", n_tokens=140, support="replay", top_p=0.9, hidden_scale=8.0, noise=0.3,
                                 age_max=4, seed=132)
    case = _concat_cases(a, b)
    hp = rh.HeadParams(loss_type=rh.RL_LOSS_IPO, eps=0.3, max_importance_ratio=10.0, kl_coeff=0.02,
                       kl_estimator=rh.RL_KL_EXACT, kl_staleness=rh.RL_STALE_INV_SQRT, bwd_mode=rh.RL_BWD_DENSE,
                       token_chunk=128)
    check_fused(case, hp)


def test_fused_sparse_mode_and_replay():
    case = workloads.make_head_case("c1", n_tokens=200, support="replay", top_p=0.9, hidden_scale=6.0,
                                    noise=0.3, seed=91)
    hp = rh.HeadParams(loss_type=rh.RL_LOSS_IPO, kl_coeff=0.02, all_replayed=1)
    check_fused(case, hp, reading="element")


def test_recompute_path_multi_chunk():
    case = workloads.make_head_case("c1", n_tokens=300, hidden_scale=8.0, noise=0.7, seed=101)
    hp = rh.HeadParams(loss_type=rh.RL_LOSS_IPO, eps=0.2, kl_coeff=0.03, bwd_mode=rh.RL_BWD_DENSE,
                       token_chunk=128)
    dev, batch, fwd = _forward(case, hp)
    ref = oracle.head_forward(case.numpy(), oracle_params(hp))
    check_forward(case, hp, fwd, ref)
    check_backward(case, hp, batch, fwd)


@pytest.mark.parametrize("prec", [rh.RL_GRAD_BF16, rh.RL_GRAD_SPLIT])
def test_entropy_regulariser_fused_and_two_call(prec):
    """loss -= entropy_coeff * H ("10-KL-clip-entropy", section 3), on draw rows and
    replayed rows (whose renormalised part is sparse but whose entropy gradient is dense),
    through the fused call (BF16: every chunk takes the logit recompute) and through the
    two-call forward / dense backward, in both gradient precisions."""
    a = workloads.make_head_case("c1", n_tokens=160, hidden_scale=8.0, noise=0.7, age_max=4, loss_mask_frac=0.1,
                                 seed=141)
    b = workloads.make_head_case("c1", n_tokens=140, support="replay", top_p=0.9, hidden_scale=8.0, noise=0.3,
                                 age_max=4, seed=142)
    case = _concat_cases(a, b)
    hp = rh.HeadParams(loss_type=rh.RL_LOSS_IPO, eps=0.3, max_importance_ratio=10.0, kl_coeff=0.02,
                       kl_estimator=rh.RL_KL_EXACT, kl_staleness=rh.RL_STALE_INV_SQRT, bwd_mode=rh.RL_BWD_AUTO,
                       grad_precision=prec, token_chunk=128, entropy_coeff=0.05)
    check_fused(case, hp, recomputed=3 if prec == rh.RL_GRAD_BF16 else 0)
    dev, batch, fwd = _forward(case, hp)
    ref = oracle.head_forward(case.numpy(), oracle_params(hp))
    check_forward(case, hp, fwd, ref)
    check_backward(case, hp, batch, fwd, both=False)


@pytest.mark.parametrize("far", [False, True], ids=["in-range", "recompute-chunk"])
def test_keep_e_two_call_equals_fused(far):
    """keep_e: rl_head_loss_fwd keeps the bf16 numerators e / e^T of every token in the
    saved state and rl_head_loss_bwd runs the fused call's backward on them.  Over three
    token chunks the forward outputs, dX and dW equal the fused call's bit for bit; with
    far=True three rows of the second chunk put their label ~86 nats below the row's max,
    so that chunk takes the gated logit recompute in both."""
    if far:
        case = workloads.make_head_case("c1", n_tokens=300, hidden_scale=60.0, noise=0.1, seed=121)
        inp = case.numpy()
        z = inp["hidden"] @ inp["W"].T
        for t in (140, 141, 200):
            v = int(np.argmin(z[t]))
            lse = float(np.max(z[t]) + np.log(np.sum(np.exp(z[t] - np.max(z[t])))))
            case.labels[t] = v
            case.label_logq[t] = float(z[t, v] - lse)
    else:
        case = workloads.make_head_case("c1", n_tokens=300, hidden_scale=8.0, noise=0.7, loss_mask_frac=0.1,
                                        age_max=4, seed=141)
    hp = rh.HeadParams(loss_type=rh.RL_LOSS_IPO, eps=0.2, max_importance_ratio=3.0, kl_coeff=0.03,
                       kl_estimator=rh.RL_KL_EXACT, kl_staleness=rh.RL_STALE_INV_SQRT, bwd_mode=rh.RL_BWD_DENSE,
                       token_chunk=128)
    hk = dataclasses.replace(hp, keep_e=1)
    dev = case.to("cuda")
    batch = rh.HeadBatch.from_case(dev)
    mask = dev.loss_mask.float()
    dl = (mask / mask.sum()).contiguous()
    fwd, dX, dW = rh.rl_head_loss_fwd_bwd(batch, hp, dl)
    f2 = rh.rl_head_loss_fwd(batch, hk)
    assert f2.saved.numel() == rh.rl_head_saved_bytes_ex(case.N, case.nnz, case.V, hk)
    assert f2.saved.numel() > rh.rl_head_saved_bytes(case.N, case.nnz) + 2 * 2 * case.N * case.V
    dX2, dW2, st = rh.rl_head_loss_bwd(batch, hk, f2.saved, dl)
    torch.cuda.synchronize()
    assert f2.status_bits() == 0 and int(st.item()) == 0
    for a, b in ((fwd.loss, f2.loss), (fwd.logp_label, f2.logp_label), (fwd.logp_support, f2.logp_support),
                 (fwd.lse, f2.lse), (fwd.entropy, f2.entropy), (dX, dX2), (dW, dW2)):
        assert torch.equal(a, b)
