"""CPU checks of the C-ABI library: it loads, exports every function include/rlhead.h
declares, sizes its workspaces, and rejects bad host-side arguments before touching a
GPU (no compute call is made here)."""
import ctypes
import os
import re

import pytest

import lm_head_gb300 as rh

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if not fn.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", fn)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w \*]*?\b(rl_\w+)\s*\(", text, flags=re.M):
            names.append(m.group(1))
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    from lm_head_gb300 import build
    build.build()
    return rh.load()


def test_header_declares_the_boundary():
    names = _declared_functions()
    for n in ("rl_head_loss_fwd", "rl_head_loss_bwd", "rl_mismatch_metrics", "rl_policy_loss_elementwise",
              "rl_validate_support", "rl_status_read"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    raw = ctypes.CDLL(rh.LIB_PATH)
    missing = [n for n in _declared_functions() if not hasattr(raw, n)]
    assert not missing, missing


def test_struct_sizes_match_the_header_layout():
    assert ctypes.sizeof(rh.RlParams) == 16 * 4
    assert ctypes.sizeof(rh.RlHeadMetrics) == 8 * 8 + 6 * 8
    assert ctypes.sizeof(rh.RlPgMetrics) == 6 * 8 + 6 * 8 + 16 * 8 + 8   # ..., ipo_curve[16], status


def test_workspace_queries(lib):
    p = rh.HeadParams()
    assert rh.rl_head_saved_bytes(256, 4096) >= 256 * 4 * 4 + 4096 * 4 + 256 * 32
    f = rh.rl_head_fwd_workspace_bytes(65536, 2048, 151936, 1 << 20, p)
    assert f >= (65536 * 3 * 4) + (1 << 20) * 4
    dense = rh.rl_head_bwd_workspace_bytes(65536, 2048, 151936, 1 << 20, rh.HeadParams(bwd_mode=rh.RL_BWD_DENSE))
    sparse = rh.rl_head_bwd_workspace_bytes(65536, 2048, 151936, 1 << 20, rh.HeadParams(bwd_mode=rh.RL_BWD_SPARSE))
    assert dense > 151936 * 2048 * 2 > sparse > 0
    assert rh.rl_policy_workspace_bytes(3_600_000) > 0


def _batch(N=256, H=128, V=1024, nnz=10):
    fake = 1 << 20   # never dereferenced: the host checks fail first
    sup = rh.RlSupport(fake, fake, fake, fake, nnz)
    return rh.RlHeadBatch(fake, fake, N, H, V, fake, fake, fake, None, None, sup)


def _fwd(lib, batch, params, ws_bytes=1 << 40):
    outs = rh.RlHeadOutputs(1 << 20, None, None, None, None, None, None, None)
    return lib.rl_head_loss_fwd(ctypes.byref(batch) if batch is not None else None,
                                ctypes.byref(params) if params is not None else None, ctypes.byref(outs),
                                ctypes.c_void_p(1 << 20), ctypes.c_void_p(1 << 20), ws_bytes,
                                ctypes.c_void_p(1 << 20), None)


def test_bad_arguments_are_rejected_on_the_host(lib):
    good = rh.HeadParams().c()
    assert _fwd(lib, None, good) == rh.RL_ERR_ARG
    assert _fwd(lib, _batch(), None) == rh.RL_ERR_ARG
    assert _fwd(lib, _batch(H=100), good) == rh.RL_ERR_UNSUPPORTED
    assert _fwd(lib, _batch(V=1001), good) == rh.RL_ERR_UNSUPPORTED
    assert _fwd(lib, _batch(N=-1), good) == rh.RL_ERR_ARG
    for field, val in (("temperature", 0.0), ("eps", -0.1), ("loss_type", 7), ("icepop_low", 3.0),
                       ("token_chunk", 100), ("kl_coeff", -1.0), ("entropy_coeff", -0.5)):
        bad = rh.HeadParams().c()
        setattr(bad, field, val)
        assert _fwd(lib, _batch(), bad) == rh.RL_ERR_ARG, field
    assert _fwd(lib, _batch(), good, ws_bytes=16) == rh.RL_ERR_WORKSPACE
    sparse_ent = rh.HeadParams(bwd_mode=rh.RL_BWD_SPARSE, entropy_coeff=0.01).c()
    assert _fwd(lib, _batch(), sparse_ent) == rh.RL_ERR_ARG     # the entropy gradient is dense
    assert lib.rl_status_read(None, None) == rh.RL_ERR_ARG
    assert lib.rl_error_string(rh.RL_ERR_WORKSPACE) == b"workspace too small"
    pp = rh.PgParams(clip_ratio_c=0.5).c()
    assert lib.rl_policy_loss_elementwise(None, None, None, None, None, 10, ctypes.byref(pp), None, None, None,
                                          None, None, None, 0, None) == rh.RL_ERR_ARG
    rp = rh.RcParams().c()
    ws = ctypes.create_string_buffer(4096)
    # tokens but no sequence: nothing could assign them a weight
    assert lib.rl_rollout_correction(None, None, None, None, 0, 5, ctypes.byref(rp), None, None, None, ws,
                                     4096, None) == rh.RL_ERR_ARG
    bad = rh.RcParams(tis_lower_bound=2.0, tis_upper_bound=1.0).c()
    assert lib.rl_rollout_correction(None, None, None, None, 0, 0, ctypes.byref(bad), None, None, None, ws,
                                     4096, None) == rh.RL_ERR_ARG


def _declared_arity():
    """Number of parameters of each rl_* function declared in include/*.h."""
    out = {}
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if not fn.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", fn)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"\b(rl_\w+)\s*\(([^;{]*?)\)\s*;", text, flags=re.S):
            args = m.group(2).strip()
            out[m.group(1)] = 0 if args in ("", "void") else args.count(",") + 1
    return out


def test_binding_signatures_match_header_arity():
    declared = _declared_arity()
    for name, (_, args) in rh._SIGS.items():
        assert name in declared, name
        assert len(args) == declared[name], (name, len(args), declared[name])


def test_options_and_new_entry_points_check_their_arguments(lib):
    assert lib.rl_get_option(rh.RL_OPT_WAIT_LIMIT_US) == 1_000_000          # 1 s by default
    for bad in (0, -5, 10_000_001):
        assert lib.rl_set_option(rh.RL_OPT_WAIT_LIMIT_US, bad) == rh.RL_ERR_ARG
    assert lib.rl_set_option(rh.RL_OPT_WAIT_LIMIT_US, 2500) == rh.RL_OK
    assert lib.rl_get_option(rh.RL_OPT_WAIT_LIMIT_US) == 2500
    assert lib.rl_set_option(rh.RL_OPT_WAIT_LIMIT_US, 1_000_000) == rh.RL_OK
    assert lib.rl_set_option(99, 1) == rh.RL_ERR_ARG and lib.rl_get_option(99) == -1
    assert lib.rl_wait_selftest(None, None) == rh.RL_ERR_ARG
    rp = rh.RcParams().c()
    assert lib.rl_rollout_metrics_named(None, ctypes.byref(rp), ctypes.c_void_p(1 << 20), None) == rh.RL_ERR_ARG
    bad = rh.RcParams().c()
    bad.tis_mode = 5
    assert lib.rl_rollout_metrics_named(ctypes.c_void_p(1 << 20), ctypes.byref(bad), ctypes.c_void_p(1 << 20),
                                        None) == rh.RL_ERR_ARG
    assert ctypes.sizeof(rh.RlRcNamed) == 28 * 8


def test_saved_bytes_ex_grows_only_where_keep_e_applies():
    """The saved state holds the kept numerators (2 N V bf16 and a little more) exactly when
    keep_e can take effect: a dense backward, BF16 gradients, no entropy term."""
    N, nnz, V = 1000, 5000, 4096
    base = rh.rl_head_saved_bytes(N, nnz)
    on = rh.HeadParams(bwd_mode=rh.RL_BWD_DENSE, keep_e=1)
    assert rh.rl_head_saved_bytes_ex(N, nnz, V, on) >= base + 2 * 2 * N * V
    for p in (rh.HeadParams(bwd_mode=rh.RL_BWD_DENSE),
              rh.HeadParams(bwd_mode=rh.RL_BWD_DENSE, keep_e=1, grad_precision=rh.RL_GRAD_SPLIT),
              rh.HeadParams(bwd_mode=rh.RL_BWD_SPARSE, keep_e=1),
              rh.HeadParams(bwd_mode=rh.RL_BWD_DENSE, keep_e=1, entropy_coeff=0.1)):
        assert rh.rl_head_saved_bytes_ex(N, nnz, V, p) == base
    assert rh.rl_head_bwd_workspace_bytes(N, 2048, V, nnz, on) < rh.rl_head_fwd_bwd_workspace_bytes(N, 2048, V, nnz, on)


def test_shard_entry_points_refuse_keep_e():
    """The vocabulary-split forward writes no kept numerators, so a backward told to use them
    would read past the saved state: both shard entry points refuse keep_e on the host,
    before touching the device."""
    lib = rh.load()
    fake = 1 << 20   # 16-byte aligned, never dereferenced: the call fails before any device work
    sup = rh.RlSupport(fake, fake, fake, fake, 8)
    b = rh.RlHeadBatch(fake, fake, 4, 128, 1024, fake, fake, fake, None, None, sup)
    p = rh.HeadParams(bwd_mode=rh.RL_BWD_DENSE, keep_e=1).c()
    st = ctypes.c_void_p(fake)
    assert lib.rl_head_shard_stats(ctypes.byref(b), ctypes.byref(p), fake, fake, fake, fake, 1 << 40, st,
                                   None) == rh.RL_ERR_ARG
    assert lib.rl_head_loss_from_shard_stats(ctypes.byref(b), ctypes.byref(p), 2, fake, fake, fake, None, fake,
                                             fake, 1 << 40, st, None) == rh.RL_ERR_ARG
    assert b"keep_e" in lib.rl_last_error()
