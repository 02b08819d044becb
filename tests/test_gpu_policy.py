"""GPU parity of the elementwise PPO / decoupled-TIS / mismatch path (through the C-ABI)
against the fp64 oracle, on the 1.8M-token synthetic replay and on edge cases."""
import numpy as np
import pytest
import torch

import lm_head_gb300 as rh
import oracle
import workloads
from parity_util import f32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from lm_head_gb300 import build
    build.build()
    rh.load()


def _oracle_pp(pp: rh.PgParams):
    return oracle.PolicyParams(clip_ratio_low=f32(pp.clip_ratio_low), clip_ratio_high=f32(pp.clip_ratio_high),
                               clip_ratio_c=f32(pp.clip_ratio_c), tis_upper=f32(pp.tis_upper),
                               icepop_low=f32(pp.icepop_low), icepop_high=f32(pp.icepop_high),
                               curve_eps=tuple(f32(e) for e in pp.curve_eps))


def _dev(x, offset):
    """x on the device, starting offset elements past the start of its allocation."""
    x = np.ascontiguousarray(x)
    buf = torch.empty(x.size + offset, dtype=torch.from_numpy(x[:0]).dtype, device="cuda")
    view = buf[offset:]
    view.copy_(torch.from_numpy(x))
    return view


def _run(lt, lo, ls, A, m, pp, offset=0):
    """m None: packed input (no mask; every slot valid)."""
    d = [_dev(x, offset) for x in (lt, lo, ls, A)] + [None if m is None else _dev(m, offset)]
    out = rh.rl_policy_loss_elementwise(*d, pp)
    torch.cuda.synchronize()
    return [o.cpu().double().numpy() for o in out[:4]], rh.pg_metrics(out[4], len(pp.curve_eps))


def _compare(lt, lo, ls, A, m, pp, offset=0):
    (lp, ld, gp, gd), gm = _run(lt, lo, ls, A, m, pp, offset)
    assert gm["status"] == 0
    ref = oracle.policy_loss_elementwise(lt, lo, ls, A, np.ones(len(lt), np.uint8) if m is None else m,
                                         _oracle_pp(pp))
    rm = ref["metrics"]
    for g, k in ((lp, "loss_ppo"), (ld, "loss_dec"), (gp, "grad_ppo"), (gd, "grad_dec")):
        r = ref[k]
        scale = np.maximum(np.abs(r), 1e-3 * max(float(np.mean(np.abs(r))), 1e-30))
        assert float(np.max(np.abs(g - r) / scale)) <= 1e-4, k
    for k in ("n_valid", "n_clip", "n_clip_lower", "icepop_low", "icepop_high", "n_tis_trunc"):
        assert gm[k] == rm[k], (k, gm[k], rm[k])
    assert gm["ipo_curve"] == rm["ipo_curve"]
    n = max(rm["n_valid"], 1)
    for k in ("loss_ppo", "loss_dec", "tis_sum"):
        assert abs(gm[k] - rm[k]) <= 1e-4 * max(abs(rm[k]), 1e-3 * n), (k, gm[k], rm[k])
    for k in ("ppo_kl", "mis_kl", "k3"):
        assert abs(gm[k] - rm[k]) <= 1e-4 * abs(rm[k]) + 2e-6 * n, (k, gm[k], rm[k])
    return gm, rm


def test_c5_full_size():
    """1.8M valid tokens, sequences 64-4096 padded to 4096: curve, IcePop band, PPO
    clip + dual clip, decoupled TIS, mismatch KL."""
    c = workloads.make_policy_case()
    gm, rm = _compare(c.lp_theta, c.lp_old, c.lp_samp, c.adv, c.mask, rh.PgParams())
    assert gm["n_valid"] == 1_800_000


def test_c5_packed():
    """The same 1.8M valid tokens laid end to end with no mask (the packed layout):
    against the oracle, and every count equal to the padded run's."""
    c = workloads.make_policy_case()
    p = c.packed()
    gm, rm = _compare(p["lp_theta"], p["lp_old"], p["lp_samp"], p["adv"], None, rh.PgParams())
    assert gm["n_valid"] == 1_800_000 == len(p["lp_theta"])
    _, gpad = _run(c.lp_theta, c.lp_old, c.lp_samp, c.adv, c.mask, rh.PgParams())
    for k in ("n_valid", "n_clip", "n_clip_lower", "icepop_low", "icepop_high", "n_tis_trunc", "ipo_curve"):
        assert gm[k] == gpad[k], k


@pytest.mark.parametrize("T,offset", [(1, 0), (17, 0), (5000, 1), (1024 * 304 * 3 + 7, 0), (300_001, 3)])
def test_packed_ragged_and_unaligned(T, offset):
    """Packed input of every length class, aligned (streaming pass) and not (exact pass)."""
    rng = np.random.default_rng(T + offset)
    lt = rng.normal(-1, 0.5, T).astype(np.float32)
    lo = (lt + rng.normal(0, 0.3, T)).astype(np.float32)
    ls = (lo + rng.normal(0, 0.5, T)).astype(np.float32)
    A = rng.normal(0, 1, T).astype(np.float32)
    gm, _ = _compare(lt, lo, ls, A, None, rh.PgParams(), offset)
    assert gm["n_valid"] == T


@pytest.mark.parametrize("T", [1, 3, 5, 16, 1001, 1024 * 304 * 3 + 7])
def test_ragged_and_scalar_path(T):
    """Lengths below one 16-slot group, a ragged tail after whole groups, and several ring
    stages per block of the streaming pass."""
    rng = np.random.default_rng(T)
    lt = rng.normal(-1, 0.5, T).astype(np.float32)
    lo = (lt + rng.normal(0, 0.3, T)).astype(np.float32)
    ls = (lo + rng.normal(0, 0.5, T)).astype(np.float32)
    A = rng.normal(0, 1, T).astype(np.float32)
    m = (rng.random(T) < 0.8).astype(np.uint8)
    _compare(lt, lo, ls, A, m, rh.PgParams())


def test_exact_threshold_ties_are_bit_exact():
    """Ratios placed exactly on / one ulp around every threshold."""
    vals = []
    for r in (0.8, 1.2, 2.0, 0.5, 3.0):
        for d in (-1, 0, 1):
            x = np.float32(np.log(r))
            x = np.nextafter(x, np.float32(np.inf) if d > 0 else np.float32(-np.inf)) if d else x
            vals.append(x)
    vals = np.array(vals, dtype=np.float32)
    T = len(vals)
    lo = np.full(T, -1.0, np.float32)
    lt = (lo + vals).astype(np.float32)
    ls = (lo - vals).astype(np.float32)
    for A in (1.0, -1.0, 0.0):
        _compare(lt, lo, ls, np.full(T, A, np.float32), np.ones(T, np.uint8), rh.PgParams())


def _band_case(T, frac, seed):
    """Random tokens, with a fraction frac placed on the clip boundary r = 1 - 0.2 (within
    fp32 rounding), where every decision is re-taken exactly."""
    rng = np.random.default_rng(seed)
    ls = np.log(1.0 / (1.0 + np.exp(-rng.normal(-1, 2.5, T)))).astype(np.float32)
    lo = (ls + rng.normal(0, 0.3, T)).astype(np.float32)
    lo = np.minimum(lo, -1e-6).astype(np.float32)
    lt = (lo + rng.normal(0, 0.1, T)).astype(np.float32)
    on = rng.random(T) < frac
    lt[on] = (lo[on].astype(np.float64) + np.log(0.8) + rng.normal(0, 2e-7, int(on.sum()))).astype(np.float32)
    A = rng.normal(0, 1, T).astype(np.float32)
    m = (rng.random(T) < 0.9).astype(np.uint8)
    return lt, lo, ls, A, m


def test_many_band_tokens_fixup_path():
    """About 10% of 20000 tokens sit on a clip threshold: each is re-decided exactly by
    the thread that meets it, and every count stays exact."""
    _compare(*_band_case(20000, 0.1, 5), rh.PgParams())


def test_half_the_tokens_in_a_band():
    """Half of 200000 tokens on a clip threshold: the exact re-decisions dominate the pass
    (a worst case for its time, not its results); results equal the oracle's."""
    _compare(*_band_case(200_000, 0.5, 6), rh.PgParams())


def test_curve_band_tokens_exact():
    """About 10% of 20000 tokens with |p_old - p_samp| within fp32 rounding of one of the
    curve's eps values: the curve counts re-taken exactly equal the oracle's."""
    rng = np.random.default_rng(9)
    T = 20000
    ls = np.log(1.0 / (1.0 + np.exp(-rng.normal(-1, 2.5, T))))
    eps = np.asarray(rh.PgParams().curve_eps, np.float64)
    po = np.exp(ls) + eps[rng.integers(0, len(eps), T)] + rng.normal(0, 3e-8, T)
    po = np.clip(po, 1e-6, 1 - 1e-6)
    lo = np.log(po)
    far = rng.random(T) > 0.1
    lo[far] = ls[far] + rng.normal(0, 0.3, int(far.sum()))
    lo = np.minimum(lo, -1e-6)
    lt = lo + rng.normal(0, 0.1, T)
    A = rng.normal(0, 1, T)
    m = (rng.random(T) < 0.9).astype(np.uint8)
    f = lambda x: np.asarray(x, np.float32)
    _compare(f(lt), f(lo), f(ls), f(A), m, rh.PgParams())


@pytest.mark.parametrize("offset", [1, 2])
def test_unaligned_inputs_take_the_exact_pass(offset):
    """Inputs that start 4 or 8 bytes past a 16-byte boundary cannot be bulk-copied: the
    scalar pass with exact decisions in the bands takes them, with the same results."""
    rng = np.random.default_rng(40 + offset)
    T = 50_001
    lt = rng.normal(-1, 0.5, T).astype(np.float32)
    lo = (lt + rng.normal(0, 0.3, T)).astype(np.float32)
    ls = (lo + rng.normal(0, 0.5, T)).astype(np.float32)
    A = rng.normal(0, 1, T).astype(np.float32)
    m = (rng.random(T) < 0.8).astype(np.uint8)
    _compare(lt, lo, ls, A, m, rh.PgParams(), offset=offset)


@pytest.mark.parametrize("packed", [False, True], ids=["padded", "packed"])
def test_huge_sum_terms(packed):
    """A few tokens with log pi_old - log pi_rollout = 30 (k3 terms near e^30, beside terms
    of order 1): past the range of the 2^-24 fixed-point accumulators, so the last block
    redoes the batch's metrics with exact decisions; outputs and metrics still match the
    oracle, on the padded pass and on the packed one."""
    rng = np.random.default_rng(21)
    T = 100_000
    ls = np.log(rng.random(T) * 0.9 + 0.05).astype(np.float32)
    lo = (ls + rng.normal(0, 0.2, T)).astype(np.float32)
    lo = np.minimum(lo, -1e-6).astype(np.float32)
    ls[::9999] = (lo[::9999] - 30.0).astype(np.float32)
    lt = (lo + rng.normal(0, 0.1, T)).astype(np.float32)
    A = rng.normal(0, 1, T).astype(np.float32)
    m = None if packed else np.ones(T, np.uint8)
    gm, rm = _compare(lt, lo, ls, A, m, rh.PgParams())
    assert rm["k3"] > 1e13


def _padding_case(seed):
    """Masks that leave whole 512-slot stages empty, put single valid tokens on stage
    edges (their pair partner is padding), valid prefixes of random length, a ragged
    16-slot group and a scalar tail; every padded slot holds NaN or +-inf."""
    rng = np.random.default_rng(seed)
    T = 512 * 303 * 5 + 512 * 7 + 48 + 5
    lt = rng.normal(-1, 0.5, T).astype(np.float32)
    lo = (lt + rng.normal(0, 0.3, T)).astype(np.float32)
    ls = (lo + rng.normal(0, 0.5, T)).astype(np.float32)
    A = rng.normal(0, 1, T).astype(np.float32)
    m = np.zeros(T, np.uint8)
    for k in range((T + 511) // 512):
        b = 512 * k
        kind = k % 5
        if kind == 1:
            m[b:b + 512] = 1
        elif kind == 2:
            m[b] = 1
        elif kind == 3:
            m[min(b + 511, T - 1)] = 1
        elif kind == 4:
            m[b:b + int(rng.integers(1, 512))] = 1
    m[-3:] = (1, 0, 7)          # any nonzero mask byte is a valid token
    pad = m == 0
    for x in (lt, lo, ls, A):
        x[pad] = rng.choice(np.array([np.nan, np.inf, -np.inf], np.float32), int(pad.sum()))
    return lt, lo, ls, A, m


def test_padding_stages_and_nonfinite_padding():
    """Whole 512-slot stages of padding, and valid tokens whose neighbour in the same
    two-slot step is padding: the values in padded slots (here NaN and inf) reach
    neither the outputs nor the sums."""
    lt, lo, ls, A, m = _padding_case(12)
    with np.errstate(invalid="ignore", over="ignore"):
        gm, rm = _compare(lt, lo, ls, A, m, rh.PgParams())
    assert gm["n_valid"] == int((m != 0).sum())
    for k in ("loss_ppo", "loss_dec", "tis_sum", "ppo_kl", "mis_kl", "k3"):
        assert np.isfinite(gm[k]), k


def test_all_padding():
    """No valid token at all, every input NaN: zero outputs, zero counts and sums."""
    T = 512 * 400 + 16 + 3
    nan = np.full(T, np.nan, np.float32)
    pp = rh.PgParams()
    (lp, ld, gp, gd), gm = _run(nan, nan, nan, nan, np.zeros(T, np.uint8), pp)
    assert gm["status"] == 0 and gm["n_valid"] == 0
    for o in (lp, ld, gp, gd):
        assert not np.any(o)
    for k in ("loss_ppo", "loss_dec", "tis_sum", "ppo_kl", "mis_kl", "k3"):
        assert gm[k] == 0.0, k
    for k in ("n_clip", "n_clip_lower", "icepop_low", "icepop_high", "n_tis_trunc"):
        assert gm[k] == 0, k
    assert gm["ipo_curve"] == [0] * len(pp.curve_eps)


@pytest.mark.parametrize("packed", [False, True], ids=["padded", "packed"])
def test_bitwise_reproducible(packed):
    """Three c5 passes give identical bytes: metrics and outputs.  The blocks add integer
    partials (order-free); in the packed pass the stages go to whichever block claims them
    first, and each thread's four-token stage sum enters the fixed point on its own, so the
    assignment does not show in the bits."""
    c = workloads.make_policy_case()
    if packed:
        p = c.packed()
        arrays = (p["lp_theta"], p["lp_old"], p["lp_samp"], p["adv"])
    else:
        arrays = (c.lp_theta, c.lp_old, c.lp_samp, c.adv, c.mask)
    d = [torch.from_numpy(np.ascontiguousarray(x)).cuda() for x in arrays] + ([None] if packed else [])
    runs = []
    for _ in range(3):
        out = rh.rl_policy_loss_elementwise(*d, rh.PgParams())
        torch.cuda.synchronize()
        runs.append((bytes(out[4].cpu().numpy().tobytes()), [o.cpu().numpy().tobytes() for o in out[:4]]))
    for r in runs[1:]:
        assert r[0] == runs[0][0]
        assert r[1] == runs[0][1]


def test_one_workspace_across_calls():
    """A workspace zeroed once serves calls of different sizes, layouts and knobs in a row
    (each call's last block leaves the arrival counter at zero): every call equals the
    same call on a fresh workspace, byte for byte."""
    ws = torch.zeros(rh.rl_policy_workspace_bytes(0), dtype=torch.uint8, device="cuda")
    c = workloads.make_policy_case(total_tokens=250_000, seed=31)
    p = c.packed()
    cases = [((c.lp_theta, c.lp_old, c.lp_samp, c.adv, c.mask), rh.PgParams()),
             ((p["lp_theta"], p["lp_old"], p["lp_samp"], p["adv"], None), rh.PgParams(curve_eps=(0.2, 0.1))),
             ((c.lp_theta[:1001], c.lp_old[:1001], c.lp_samp[:1001], c.adv[:1001], c.mask[:1001]), rh.PgParams()),
             ((p["lp_theta"][1:], p["lp_old"][1:], p["lp_samp"][1:], p["adv"][1:], None), rh.PgParams())]
    for arrays, pp in cases * 2:
        d = [None if x is None else torch.from_numpy(np.ascontiguousarray(x)).cuda() for x in arrays]
        fresh = rh.rl_policy_loss_elementwise(*d, pp)
        reused = rh.rl_policy_loss_elementwise(*d, pp, ws=ws)
        torch.cuda.synchronize()
        for a, b in zip(fresh, reused):
            assert torch.equal(a, b)
