"""The allocation-free elementwise entry point (rl_policy_loss_elementwise_noalloc), for
callers that hold only their input and output buffers and cannot allocate device memory
(for example a loss or metrics hook inside an engine whose memory is reserved up front
by its own pool).  It must give the same results as the workspace entry point, within
the tolerances the other elementwise tests use, on two calls in a row (its static
scratch keeps the previous call's contents).  This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

import lm_head_gb300 as rh
import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from lm_head_gb300 import build
    build.build()
    rh.load()


def _dev(case):
    return [torch.from_numpy(np.ascontiguousarray(x)).cuda()
            for x in (case.lp_theta, case.lp_old, case.lp_samp, case.adv, case.mask)]


def _compare(ref, got):
    (rl, rd, rg, rgd, rm), (gl, gd, gg, ggd, gm) = ref, got
    for a, b in ((rl, gl), (rd, gd), (rg, gg), (rgd, ggd)):
        a = a.double().cpu().numpy()
        b = b.double().cpu().numpy()
        scale = np.maximum(np.abs(a), 1e-3 * max(float(np.mean(np.abs(a))), 1e-30))
        assert float(np.max(np.abs(a - b) / scale)) <= 1e-4
    ma, mb = rh.pg_metrics(rm), rh.pg_metrics(gm)
    for k in ("n_valid", "n_clip", "n_clip_lower", "icepop_low", "icepop_high", "n_tis_trunc", "ipo_curve"):
        assert ma[k] == mb[k], k
    n = max(ma["n_valid"], 1)
    for k in ("loss_ppo", "loss_dec", "tis_sum", "ppo_kl", "mis_kl", "k3"):
        assert abs(ma[k] - mb[k]) <= 1e-4 * max(abs(ma[k]), 1e-3 * n) + 2e-6 * n, k


def test_noalloc_matches_workspace_entry_on_two_calls_in_a_row():
    pp = rh.PgParams()
    for total, seed in ((300_000, 7), (123_457, 8)):     # second call: other sizes, stale scratch
        case = workloads.make_policy_case(total_tokens=total, seed=seed)
        t = _dev(case)
        ref = rh.rl_policy_loss_elementwise(*t, pp)
        T = t[0].numel()
        outs = tuple(torch.full((T,), float("nan"), device="cuda") for _ in range(4))
        met = torch.full((ctypes.sizeof(rh.RlPgMetrics),), 0xFF, dtype=torch.uint8, device="cuda")
        got = rh.rl_policy_loss_elementwise_noalloc(*t, pp, outputs=outs, metrics_dev=met)
        torch.cuda.synchronize()
        _compare(ref, got)
