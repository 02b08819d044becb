"""Device-side failure reporting, through the C ABI (pull request #4233: the sampler
evidence is validated on the GPU once per step, before the optimizer).

* Each sampler-evidence check on its own: a clean batch with one fault put in on the host
  (offsets, an id or label out of range, a non-finite or positive log q, a replayed row
  without its label or whose q does not sum to 1, an empty RL row, ids out of order).  The
  device's status bits equal the oracle's statement of the checks bit for bit, the
  forward on the corrupt batch reports them without faulting, and a clean call afterwards
  returns status 0.
* The bits the loss kernels raise: a sparse backward asked for where a token's gradient
  has a dense part (SPARSE_INELIGIBLE), a non-finite hidden row (NONFINITE).
* The bounded waits: a wait on an mbarrier nothing signals runs out after the runtime
  limit and reports RL_STATUS_TIMEOUT; kernels run under a limit of a microsecond either
  finish or unwind with that bit; the next call under the default limit is correct.
* The standalone rl_mismatch_metrics against the oracle's metric sums.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

import lm_head_gb300 as rh
import oracle
import workloads
from gpu_checks import check_metrics, entry_rows
from parity_util import logp_tol, loss_prop_tol, oracle_params

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from lm_head_gb300 import build
    build.build()
    rh.load()
    yield
    rh.rl_set_option(rh.RL_OPT_WAIT_LIMIT_US, 1_000_000)


def _replay():
    return workloads.make_head_case("c1", n_tokens=96, support="replay", top_p=0.9, hidden_scale=6.0, seed=91)


def _draws():
    return workloads.make_head_case("c1", n_tokens=96, seed=92, loss_mask_frac=0.1)


def _row(case, t):
    return int(case.offsets[t]), int(case.offsets[t + 1])


def _rl_row(case, want_len=2, replayed=None):
    for t in range(case.N):
        b, e = _row(case, t)
        if e - b >= want_len and bool(case.loss_mask[t]) and (replayed is None or bool(case.replayed[t]) == replayed):
            if len(set(case.ids[b:e].tolist())) == e - b:
                return t
    raise AssertionError("no suitable row")


def _clone(case):
    """A host copy that shares no tensor with `case` (Tensor.to on the same device would)."""
    import dataclasses
    kw = {f.name: getattr(case, f.name) for f in dataclasses.fields(case)}
    return type(case)(**{k: (v.detach().cpu().clone() if isinstance(v, torch.Tensor) else v) for k, v in kw.items()})


def f_offsets_past_nnz(c):
    c.offsets[-1] += 5


def f_offsets_decreasing(c):
    c.offsets[3] = c.offsets[4] + 1


def f_id_out_of_range(c):
    t = _rl_row(c, 2, replayed=False) if not bool(c.replayed.all()) else _rl_row(c, 2)
    b, e = _row(c, t)
    if int(c.labels[t]) == int(c.ids[e - 1]):
        c.labels[t] = int(c.ids[b])
    c.ids[e - 1] = c.V + 3                        # last entry of its row: the order holds


def f_label_out_of_range(c):
    c.labels[4] = c.V


def f_logq_nan(c):
    c.logq[2] = float("nan")


def f_logq_positive(c):
    c.logq[5] = 0.5


def f_label_logq_inf(c):
    c.label_logq[6] = float("inf")


def f_label_missing(c):
    t = _rl_row(c, 2, replayed=True)
    b, e = _row(c, t)
    row = set(c.ids[b:e].tolist())
    c.labels[t] = next(v for v in range(c.V) if v not in row)


def f_support_mass(c):
    t = _rl_row(c, 2, replayed=True)
    b, e = _row(c, t)
    c.logq[b:e] += math.log(0.9)


def f_empty_row(c):
    t = _rl_row(c, 1)
    b, e = _row(c, t)
    c.ids = torch.cat([c.ids[:b], c.ids[e:]])
    c.logq = torch.cat([c.logq[:b], c.logq[e:]])
    c.offsets[t + 1:] -= e - b


def f_row_order(c):
    t = _rl_row(c, 2)
    b, e = _row(c, t)
    c.ids[b], c.ids[b + 1] = int(c.ids[b + 1]), int(c.ids[b])


def f_replayed_duplicate(c):
    t = _rl_row(c, 3, replayed=True)
    b, e = _row(c, t)
    if int(c.labels[t]) == int(c.ids[b + 1]):
        c.labels[t] = int(c.ids[b + 2])
    c.ids[b + 1] = int(c.ids[b])


FAULTS = [("replay", f) for f in (f_offsets_past_nnz, f_offsets_decreasing, f_id_out_of_range, f_label_out_of_range,
                                 f_logq_nan, f_logq_positive, f_label_logq_inf, f_label_missing, f_support_mass,
                                 f_row_order, f_replayed_duplicate, f_empty_row)] + \
         [("draws", f) for f in (f_offsets_past_nnz, f_id_out_of_range, f_logq_nan, f_logq_positive, f_empty_row,
                                f_row_order)]


@pytest.mark.parametrize("kind,fault", FAULTS, ids=[f"{k}-{f.__name__}" for k, f in FAULTS])
def test_each_evidence_check_against_the_oracle(kind, fault):
    clean = _replay() if kind == "replay" else _draws()
    bad = _clone(clean)
    fault(bad)
    want = oracle.validate_support(bad.numpy(), bad.V)
    assert want != 0
    dev = bad.to("cuda")
    batch = rh.HeadBatch.from_case(dev)
    st = rh.rl_validate_support(batch)
    torch.cuda.synchronize()
    assert int(st.item()) == want, (rh.status_names(int(st.item())), rh.status_names(want))
    hp = rh.HeadParams(loss_type=rh.RL_LOSS_IPO, bwd_mode=rh.RL_BWD_DENSE, kl_coeff=0.01)
    fwd = rh.rl_head_loss_fwd(batch, hp)               # runs the same checks, then the loss on clamped indices
    torch.cuda.synchronize()
    assert fwd.status_bits() & want == want
    ok = rh.rl_head_loss_fwd(rh.HeadBatch.from_case(clean.to("cuda")), hp)
    torch.cuda.synchronize()
    assert ok.status_bits() == 0


def test_sparse_backward_asked_for_a_dense_gradient():
    case = _draws().to("cuda")
    batch = rh.HeadBatch.from_case(case)
    for hp, want in ((rh.HeadParams(loss_type=rh.RL_LOSS_IPO, bwd_mode=rh.RL_BWD_SPARSE), 0x80),
                     (rh.HeadParams(loss_type=rh.RL_LOSS_REINFORCE, bwd_mode=rh.RL_BWD_SPARSE, kl_coeff=0.02), 0x80),
                     (rh.HeadParams(loss_type=rh.RL_LOSS_REINFORCE, bwd_mode=rh.RL_BWD_SPARSE), 0)):
        fwd = rh.rl_head_loss_fwd(batch, hp)
        dl = torch.full((case.N,), 1.0 / case.N, device="cuda")
        f2, _, _ = rh.rl_head_loss_fwd_bwd(batch, hp, dl)
        torch.cuda.synchronize()
        assert fwd.status_bits() == want and f2.status_bits() == want, (rh.status_names(fwd.status_bits()), want)
    rep = _replay().to("cuda")
    f3 = rh.rl_head_loss_fwd(rh.HeadBatch.from_case(rep), rh.HeadParams(bwd_mode=rh.RL_BWD_SPARSE))
    torch.cuda.synchronize()
    assert f3.status_bits() == 0


def test_nonfinite_hidden_row_is_reported():
    case = _draws()
    case.hidden[7] = float("nan")
    dev = case.to("cuda")
    fwd = rh.rl_head_loss_fwd(rh.HeadBatch.from_case(dev), rh.HeadParams(bwd_mode=rh.RL_BWD_DENSE))
    torch.cuda.synchronize()
    assert fwd.status_bits() == 0x100, rh.status_names(fwd.status_bits())
    assert math.isnan(float(fwd.lse[7])) and bool(torch.isfinite(fwd.lse[8:]).all())


def test_a_wait_nothing_signals_runs_out_and_the_context_survives():
    for limit_us in (5, 200_000):
        rh.rl_set_option(rh.RL_OPT_WAIT_LIMIT_US, limit_us)
        st = rh.rl_wait_selftest()
        torch.cuda.synchronize()
        assert int(st.item()) == 0x200
    rh.rl_set_option(rh.RL_OPT_WAIT_LIMIT_US, 1_000_000)
    st = rh.rl_wait_selftest()                # the default: 1 s
    torch.cuda.synchronize()
    assert int(st.item()) == 0x200
    case = _draws().to("cuda")
    ok = rh.rl_head_loss_fwd(rh.HeadBatch.from_case(case), rh.HeadParams(bwd_mode=rh.RL_BWD_DENSE))
    torch.cuda.synchronize()
    assert ok.status_bits() == 0


@pytest.mark.parametrize("pair", [1, 0])
def test_kernels_under_a_one_microsecond_limit_finish_or_unwind(pair):
    """A limit far below a DRAM round trip: the tensor-core GEMM (pair or single-SM
    pipeline) and the elementwise pass either finish or give up with RL_STATUS_TIMEOUT,
    draining their own copies and MMAs before they leave; then, under the default limit,
    the same calls are correct again."""
    g = torch.Generator(device="cuda").manual_seed(5)
    A = torch.randn(2048, 2048, device="cuda", generator=g).to(torch.bfloat16)
    B = torch.randn(4096, 2048, device="cuda", generator=g).to(torch.bfloat16)
    pc = workloads.make_policy_case(total_tokens=400_000, seed=3)
    t = [torch.from_numpy(np.ascontiguousarray(x)).cuda() for x in (pc.lp_theta, pc.lp_old, pc.lp_samp, pc.adv, pc.mask)]
    old = rh.rl_get_option(rh.RL_OPT_GEMM_PAIR)
    rh.rl_set_option(rh.RL_OPT_GEMM_PAIR, pair)
    try:
        ref = rh.rl_policy_loss_elementwise(*t, rh.PgParams())
        torch.cuda.synchronize()
        seen = 0
        rh.rl_set_option(rh.RL_OPT_WAIT_LIMIT_US, 1)
        for _ in range(3):
            D, st = rh.rl_gemm_bf16_tn(A, B)
            out = rh.rl_policy_loss_elementwise(*t, rh.PgParams())
            torch.cuda.synchronize()
            assert int(st.item()) in (0, 0x200)
            ps = rh.pg_metrics(out[4])["status"]
            assert ps in (0, 0x200)
            seen |= int(st.item()) | ps
        rh.rl_set_option(rh.RL_OPT_WAIT_LIMIT_US, 1_000_000)
        D, st = rh.rl_gemm_bf16_tn(A, B)
        out = rh.rl_policy_loss_elementwise(*t, rh.PgParams())
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        want = A.float() @ B.float().T
        assert float((D - want).abs().max()) <= 1e-3 * float(want.abs().max())
        for a, b in zip(ref, out):
            assert torch.equal(a, b)
        print(f"short-limit runs with pair={pair}: timeout bit seen={bool(seen & 0x200)}")
    finally:
        rh.rl_set_option(rh.RL_OPT_WAIT_LIMIT_US, 1_000_000)
        rh.rl_set_option(rh.RL_OPT_GEMM_PAIR, old)


@pytest.mark.parametrize("kind", ["draws", "replay"])
def test_standalone_mismatch_metrics_against_the_oracle(kind):
    case = (workloads.make_head_case("c1", n_tokens=256, hidden_scale=10.0, noise=1.0, age_max=3, seed=93,
                                     loss_mask_frac=0.2) if kind == "draws" else
            workloads.make_head_case("c1", n_tokens=256, support="replay", top_p=0.9, hidden_scale=6.0, noise=1.0,
                                     age_max=3, seed=94, loss_mask_frac=0.2))
    hp = rh.HeadParams(loss_type=rh.RL_LOSS_IPO, eps=0.05, max_importance_ratio=3.0, kl_coeff=0.02,
                       kl_staleness=rh.RL_STALE_INV_SQRT, bwd_mode=rh.RL_BWD_DENSE)
    dev = case.to("cuda")
    batch = rh.HeadBatch.from_case(dev)
    fwd = rh.rl_head_loss_fwd(batch, hp, want_metrics=False)
    m = rh.rl_mismatch_metrics(batch, fwd.saved, hp)
    torch.cuda.synchronize()
    assert fwd.status_bits() == 0
    op = oracle_params(hp)
    inp = case.numpy()
    ref = oracle.head_forward(inp, op)
    H = case.H
    er = entry_rows(inp["offsets"])
    lab_tol = logp_tol(H, ref["zmax"], ref["lse_s"])
    sup_tol = logp_tol(H, ref["zmax"][er], ref["lse_s"][er])
    check_metrics(m, ref, inp, H, fwd.mask_label.cpu().numpy(), lab_tol, sup_tol, loss_prop_tol(ref, inp, op))
    assert m["masked"] > 0 and m["n_age0"] > 0
    f2 = rh.rl_head_loss_fwd(batch, hp)                 # the forward's own metrics: the same bits
    torch.cuda.synchronize()
    assert f2.metrics() == m
