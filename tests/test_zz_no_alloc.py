"""The allocation-free elementwise entry point (rl_policy_loss_elementwise_noalloc), for
callers that hold only their input and output buffers and cannot allocate device memory
(for example a loss or metrics hook inside an engine whose memory is reserved up front
by its own pool).  It runs the same kernel as the workspace entry point on the same
inputs, with the same deterministic reduction of the blocks' records, so its outputs and
its metrics struct must equal that entry point's bit for bit, on several calls in a row:
its static scratch keeps the previous call's contents, so each call here changes the
size, the knobs (curve length and eps values, clip bounds) or puts huge terms in the sums,
which a stale arrival count, record or curve count would all show.  This file is
collected last on purpose."""
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


def _dev(case, big_adv_every=0):
    t = [torch.from_numpy(np.ascontiguousarray(x)).cuda()
         for x in (case.lp_theta, case.lp_old, case.lp_samp, case.adv, case.mask)]
    if big_adv_every:
        t[3][::big_adv_every] = 1e12      # huge loss terms in the sums
    return t


def _equal(ref, got):
    for a, b in zip(ref[:4], got[:4]):
        assert torch.equal(a, b)
    assert torch.equal(ref[4], got[4])   # the raw metrics struct, every byte


CALLS = [
    (300_000, 7, rh.PgParams(), 0),
    (123_457, 8, rh.PgParams(clip_ratio_low=0.1, clip_ratio_high=0.3, clip_ratio_c=2.5, tis_upper=1.5,
                             curve_eps=(0.25, 0.05, 0.4, 0.1, 0.15)), 0),
    (200_001, 9, rh.PgParams(curve_eps=(0.3, 0.02)), 9973),
    (77_777, 10, rh.PgParams(), 0),
]


def test_noalloc_matches_workspace_entry_on_calls_in_a_row():
    for total, seed, pp, big in CALLS:
        case = workloads.make_policy_case(total_tokens=total, seed=seed)
        t = _dev(case, big)
        ref = rh.rl_policy_loss_elementwise(*t, pp)
        T = t[0].numel()
        outs = tuple(torch.full((T,), float("nan"), device="cuda") for _ in range(4))
        met = torch.full((ctypes.sizeof(rh.RlPgMetrics),), 0xFF, dtype=torch.uint8, device="cuda")
        got = rh.rl_policy_loss_elementwise_noalloc(*t, pp, outputs=outs, metrics_dev=met)
        torch.cuda.synchronize()
        _equal(ref, got)
        m = rh.pg_metrics(got[4], len(pp.curve_eps))
        assert m["status"] == 0 and m["n_valid"] == int(case.mask.astype(bool).sum())
