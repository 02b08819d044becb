"""GPU parity of the rollout-correction path (IS / RS weights at token, sequence and
geometric level, the veto, batch normalisation, mismatch metrics) through the C ABI,
against the fp64 oracle, on the 1.8M-token synthetic replay (padded rows as sequences)
and on packed, ragged and degenerate layouts.

Bars: keep flags and every count bit-exact (the decisions are exact predicates on the
fp32 inputs on both sides); weights within 4e-6 relative (an fp32 exponential of an
exact log-ratio, times an fp32 factor); sums within 1e-5 relative plus 1e-6 per term
(fp32 terms summed per sequence, then in fp64)."""
import math

import numpy as np
import pytest
import torch

import lm_head_gb300 as rh
import workloads
from oracle.rollout import RolloutParams, rollout_correction, rollout_metrics_named

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from lm_head_gb300 import build
    build.build()
    rh.load()


def _oracle_params(p: rh.RcParams) -> RolloutParams:
    f = lambda x: None if x is None else float(np.float32(x))
    return RolloutParams(use_tis=p.use_tis, tis_mode=p.tis_mode, tis_lower_bound=f(p.tis_lower_bound),
                         tis_upper_bound=f(p.tis_upper_bound), tis_level=p.tis_level,
                         tis_batch_normalize=p.tis_batch_normalize, use_rs=p.use_rs,
                         rs_lower_bound=f(p.rs_lower_bound), rs_upper_bound=f(p.rs_upper_bound),
                         rs_level=p.rs_level, rs_veto_threshold=f(p.rs_veto_threshold))


def _run(lt, lr, m, off, p):
    d = [torch.from_numpy(np.ascontiguousarray(x)).cuda() for x in (lt, lr, m, np.asarray(off, np.int64))]
    w, k, met = rh.rl_rollout_correction(*d, p)
    torch.cuda.synchronize()
    return w.cpu().double().numpy(), k.cpu().numpy(), rh.rc_metrics(met)


def _compare(lt, lr, m, off, p):
    w, k, gm = _run(lt, lr, m, off, p)
    ref = rollout_correction(lt, lr, m, off, _oracle_params(p))
    rm = ref["metrics"]
    assert gm["status"] == 0
    np.testing.assert_array_equal(k, ref["keep"])
    rw = ref["weights"]
    assert np.all(np.abs(w - rw) <= 4e-6 * np.abs(rw) + 1e-30), float(np.max(np.abs(w - rw) / np.maximum(np.abs(rw), 1e-30)))
    for key in ("n_valid", "n_seq", "n_kept", "n_tis_low", "n_tis_high", "n_rs_low", "n_rs_high", "n_cat_tokens",
                "n_cat_seqs"):
        assert gm[key] == rm[key], (key, gm[key], rm[key])
    nv, ns = max(rm["n_valid"], 1), max(rm["n_seq"], 1)
    tok_terms = ("w_before_sum", "w_after_sum", "kept_w_sum", "final_sum", "mis_kl_sum", "k3_sum", "abs_diff_sum",
                 "chi2_token_sum")
    seq_terms = ("train_lppl_sum", "rollout_lppl_sum", "lppl_diff_sum", "lppl_abs_diff_sum", "ppl_ratio_sum",
                 "chi2_seq_sum")
    for key in tok_terms + seq_terms:
        n = nv if key in tok_terms else ns
        g, r = gm[key], rm[key]
        if math.isinf(r):
            assert g == r, key
            continue
        assert abs(g - r) <= 1e-5 * abs(r) + 1e-6 * n, (key, g, r)
    for key in ("batch_norm_factor", "final_min", "final_max"):
        assert gm[key] == pytest.approx(rm[key], rel=4e-6, abs=1e-30), key
    return gm, rm


def _c5():
    c = workloads.make_policy_case()
    B = len(c.seq_lens)
    off = np.arange(B + 1, dtype=np.int64) * c.max_len
    return c.lp_old, c.lp_samp, c.mask, off


SETTINGS = [
    rh.RcParams(),                                                            # token, truncate
    rh.RcParams(tis_mode="clip", tis_level="sequence", tis_lower_bound=0.1, tis_upper_bound=10.0,
                tis_batch_normalize=True, use_rs=True, rs_level="geometric", rs_lower_bound=0.9,
                rs_upper_bound=1.1, rs_veto_threshold=1e-4),
    rh.RcParams(tis_mode="mask", tis_level="geometric", tis_lower_bound=0.95, tis_upper_bound=1.05,
                use_rs=True, rs_level="sequence", rs_lower_bound=0.8, rs_upper_bound=1.3, rs_veto_threshold=1e-3),
    rh.RcParams(use_tis=False, use_rs=True, rs_level="token", rs_lower_bound=0.5, rs_upper_bound=2.0),
    rh.RcParams(tis_mode="clip", tis_batch_normalize=True, rs_veto_threshold=0.05),
]


@pytest.mark.parametrize("cfg", range(len(SETTINGS)))
def test_c5_full_size(cfg):
    """879 padded rows of up to 4096 tokens, 1.8M response tokens, five knob settings."""
    gm, rm = _compare(*_c5(), SETTINGS[cfg])
    assert gm["n_valid"] == 1_800_000


def test_packed_ragged_sequences_and_empty_ones():
    """Packed layout (cumulative lengths), lengths 0..700 with empty and fully masked
    sequences, T not a multiple of anything in particular."""
    rng = np.random.default_rng(11)
    lens = rng.integers(0, 700, size=97)
    lens[[3, 40, 41]] = 0
    T = int(lens.sum())
    off = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    lr = np.log(rng.random(T) * 0.98 + 0.01).astype(np.float32)
    lt = (lr + rng.normal(0, 0.2, T)).astype(np.float32)
    lt = np.minimum(lt, 0).astype(np.float32)
    m = (rng.random(T) < 0.85).astype(np.uint8)
    m[off[10]:off[11]] = 0
    for p in SETTINGS:
        _compare(lt, lr, m, off, p)


def test_exact_bounds_and_single_long_sequence():
    """Token log-ratios on and one float step around ln(bound) for every bound, in one
    sequence of 40000 tokens (one block walks it)."""
    vals = []
    for bnd in (0.5, 2.0, 0.9, 1.1):
        x = np.float32(np.log(bnd))
        vals += [np.nextafter(x, np.float32(-np.inf)), x, np.nextafter(x, np.float32(np.inf))]
    T = 40000
    rng = np.random.default_rng(12)
    d = rng.normal(0, 0.3, T).astype(np.float32)
    d[:len(vals)] = vals
    lr = np.full(T, -2.0, np.float32)
    lt = (lr + d).astype(np.float32)
    m = np.ones(T, np.uint8)
    for p in (rh.RcParams(tis_mode="mask"), rh.RcParams(use_rs=True, rs_lower_bound=0.9, rs_upper_bound=1.1),
              rh.RcParams(tis_mode="clip", tis_level="geometric", use_rs=True, rs_level="sequence")):
        _compare(lt, lr, m, [0, T], p)


def test_bad_offsets_set_the_status_bit():
    T = 1000
    lt = np.zeros(T, np.float32)
    off = torch.tensor([0, 600, 400, T], dtype=torch.int64, device="cuda")   # decreasing
    w, k, met = rh.rl_rollout_correction(torch.zeros(T, device="cuda"), torch.zeros(T, device="cuda"),
                                         torch.ones(T, dtype=torch.uint8, device="cuda"), off, rh.RcParams())
    torch.cuda.synchronize()
    assert rh.rc_metrics(met)["status"] & 0x1


def test_nonfinite_padding():
    """NaN / inf in every masked slot of the c5 rows (their padding and the masked tokens
    inside): results equal the oracle's, which ignores them."""
    lt, lr, m, off = (np.array(x) for x in _c5())
    rng = np.random.default_rng(15)
    pad = m == 0
    lt[pad] = rng.choice(np.array([np.nan, np.inf, -np.inf], np.float32), int(pad.sum()))
    lr[pad] = rng.choice(np.array([np.nan, np.inf, -np.inf], np.float32), int(pad.sum()))
    with np.errstate(invalid="ignore", over="ignore"):
        for cfg in (1, 2, 3):
            _compare(lt, lr, m, off, SETTINGS[cfg])


def test_normalisation_past_the_integer_totals_range():
    """Batch normalisation whose kept weights reach ~2e17 (log-ratios of 40; e^(2 x 40)
    still fits the fp32 chi^2 terms): a sequence's kept-weight sum is past the range of
    the integer totals the factor normally comes from, so the factor is taken from the
    records reduced in sequence order instead; the results equal the oracle's either way."""
    rng = np.random.default_rng(16)
    lens = np.array([300, 500, 200])
    T = int(lens.sum())
    off = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    lr = np.log(rng.random(T) * 0.9 + 0.05)
    lt = np.minimum(lr + rng.normal(0, 0.3, T), 0.0)
    lr[::97] = -52.0
    lt[::97] = -12.0
    m = np.ones(T, np.uint8)
    for p in (rh.RcParams(tis_mode="truncate", tis_upper_bound=1e30, tis_batch_normalize=True),
              rh.RcParams(tis_mode="clip", tis_lower_bound=0.1, tis_upper_bound=10.0, tis_batch_normalize=True)):
        _compare(lt.astype(np.float32), lr.astype(np.float32), m, off, p)


def _named_tolerance(key, rm, rn):
    """Bar of a named metric, from the bars of the sums it is formed from (1e-5 relative
    plus 1e-6 per term, divided by the count it is a mean over); counts are bit-exact, so
    the fractions are equal outright; the factor and the min / max to 4e-6 relative."""
    nv, ns, nk = max(rm["n_valid"], 1), max(rm["n_seq"], 1), max(rm["n_kept"], 1)
    tok = {"kl": "mis_kl_sum", "k3_kl": "k3_sum", "train_rollout_logprob_abs_diff": "abs_diff_sum",
           "chi2_token": "chi2_token_sum", "tis_weight_before_bound": "w_before_sum",
           "tis_weight_after_bound": "w_after_sum"}
    seq = {"training_log_ppl": "train_lppl_sum", "rollout_log_ppl": "rollout_lppl_sum", "log_ppl_diff": "lppl_diff_sum",
           "log_ppl_abs_diff": "lppl_abs_diff_sum", "ppl_ratio": "ppl_ratio_sum", "chi2_seq": "chi2_seq_sum"}
    kept = {"is_ratio_mean_after_tis_rs": "kept_w_sum", "is_ratio_mean_final": "final_sum"}
    if key in tok:
        return (1e-5 * abs(rm[tok[key]]) + 1e-6 * nv) / nv
    if key in seq:
        return (1e-5 * abs(rm[seq[key]]) + 1e-6 * ns) / ns
    if key in kept:
        return (1e-5 * abs(rm[kept[key]]) + 1e-6 * nv) / nk
    if key in ("training_ppl", "rollout_ppl"):
        base = "training_log_ppl" if key == "training_ppl" else "rollout_log_ppl"
        return 1.01 * rn[key] * _named_tolerance(base, rm, rn)
    if key in ("batch_norm_factor", "is_ratio_min_final", "is_ratio_max_final"):
        return 4e-6 * abs(rn[key])
    return 0.0                                          # fractions of exact counts


def _named_compare(lt, lr, m, off, p):
    d = [torch.from_numpy(np.ascontiguousarray(x)).cuda() for x in (lt, lr, m, np.asarray(off, np.int64))]
    _, _, met = rh.rl_rollout_correction(*d, p)
    named = rh.rl_rollout_metrics_named(met, p)
    torch.cuda.synchronize()
    op = _oracle_params(p)
    ref = rollout_correction(lt, lr, m, off, op)
    rn = rollout_metrics_named(ref["metrics"], op)
    assert set(named) == set(rn), (set(named) ^ set(rn))
    for k, r in rn.items():
        g = named[k]
        if math.isinf(r):
            assert g == r, k
            continue
        assert abs(g - r) <= _named_tolerance(k, ref["metrics"], rn), (k, g, r)


@pytest.mark.parametrize("cfg", range(len(SETTINGS)))
def test_named_metrics_c5_against_the_oracle(cfg):
    """The page's named metrics, formed on the device from the sums, against the oracle's
    named metrics: the emitted set per the "Emitted when" column, and every value."""
    _named_compare(*_c5(), SETTINGS[cfg])


def test_named_metrics_ragged_against_the_oracle():
    rng = np.random.default_rng(19)
    lens = rng.integers(0, 500, size=61)
    lens[[2, 30]] = 0
    T = int(lens.sum())
    off = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    lr = np.log(rng.random(T) * 0.98 + 0.01).astype(np.float32)
    lt = np.minimum(lr + rng.normal(0, 0.25, T), 0).astype(np.float32)
    m = (rng.random(T) < 0.8).astype(np.uint8)
    for p in SETTINGS + [rh.RcParams(use_tis=False, rs_veto_threshold=1e-3),
                         rh.RcParams(tis_mode="mask", tis_lower_bound=0.8, tis_upper_bound=1.25)]:
        _named_compare(lt, lr, m, off, p)


def test_repeated_calls_are_bitwise_identical():
    """Sums in a fixed order (records by groups of 32 in sequence order, then the groups in
    order, whichever block finishes last): three calls on one workspace, zeroed once, give
    the same bits: weights, keep flags and the metrics struct."""
    lt, lr, m, off = _c5()
    d = [torch.from_numpy(np.ascontiguousarray(x)).cuda() for x in (lt, lr, m, np.asarray(off, np.int64))]
    B = len(off) - 1
    ws = torch.zeros(rh.rl_rollout_correction_workspace_bytes(B), dtype=torch.uint8, device="cuda")
    outs = []
    for _ in range(3):
        w, k, met = rh.rl_rollout_correction(*d, SETTINGS[1], ws=ws)
        torch.cuda.synchronize()
        outs.append((w.cpu().numpy().tobytes(), k.cpu().numpy().tobytes(), met.cpu().numpy().tobytes()))
    assert outs[0] == outs[1] == outs[2]
    assert rh.rc_metrics(met)["status"] == 0


def test_unaligned_arrays_take_the_chunked_staging():
    """The arrays one element past a 16-byte boundary: sequences of up to 4096 tokens are then
    staged with plain loads instead of bulk copies; the results still equal the oracle's."""
    rng = np.random.default_rng(17)
    lens = rng.integers(1, 3000, size=40)
    T = int(lens.sum())
    off = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    lr = np.log(rng.random(T) * 0.98 + 0.01).astype(np.float32)
    lt = np.minimum(lr + rng.normal(0, 0.2, T), 0).astype(np.float32)
    m = (rng.random(T) < 0.9).astype(np.uint8)
    d = []
    for x in (lt, lr, m):
        buf = torch.zeros(T + 1, dtype=torch.from_numpy(x).dtype, device="cuda")
        buf[1:] = torch.from_numpy(x).cuda()
        d.append(buf[1:])
    assert d[0].data_ptr() % 16 != 0
    offs = torch.from_numpy(off).cuda()
    for p in SETTINGS:
        w, k, met = rh.rl_rollout_correction(*d, offs, p)
        torch.cuda.synchronize()
        ref = rollout_correction(lt, lr, m, off, _oracle_params(p))
        np.testing.assert_array_equal(k.cpu().numpy(), ref["keep"])
        rw = ref["weights"]
        wg = w.cpu().double().numpy()
        assert np.all(np.abs(wg - rw) <= 4e-6 * np.abs(rw) + 1e-30)
        gm = rh.rc_metrics(met)
        assert gm["status"] == 0
        for key in ("n_valid", "n_kept", "n_rs_low", "n_rs_high", "n_cat_tokens"):
            assert gm[key] == ref["metrics"][key], key
