"""Thin Python binding of librlhead (include/rlhead.h), GB300 / sm_103a.

Argument marshalling only: every step of the computation runs in the library's CUDA
kernels.  PyTorch provides device memory and the current stream.  There is no CPU
fallback: if the extension is missing or no sm_100-family GPU is present, calls raise.

Functions carry the C names:
  head:        rl_validate_support, rl_head_loss_fwd, rl_head_loss_bwd,
               rl_head_loss_fwd_bwd (one call when dloss is known before the forward),
               rl_mismatch_metrics; vocabulary shards: rl_head_shard_remap,
               rl_head_shard_stats, rl_head_loss_from_shard_stats (rank logic in
               lm_head_gb300.vocab_parallel)
  elementwise: rl_policy_loss_elementwise (+ rl_policy_loss_elementwise_noalloc in C)
  rollout:     rl_rollout_correction (IS / RS weights, veto, batch normalisation, metric
               sums), rl_rollout_metrics_named (the page's named metrics from those sums)
  utilities:   rl_gemm_bf16, rl_gemm_bf16_tn, rl_status_read, rl_wait_selftest,
               rl_set_option / rl_get_option, rl_profile_enable / rl_profile_read,
               rl_kernel_launch_count, the *_workspace_bytes queries

Typical use (device tensors; see the tests for every option):
  batch = HeadBatch.from_case(case)                 # hidden, W, labels, CSR support, ...
  hp = HeadParams(loss_type=RL_LOSS_IPO, eps=0.3, max_importance_ratio=10.0)
  fwd, dX, dW = rl_head_loss_fwd_bwd(batch, hp, dloss)   # fused forward + backward
  fwd = rl_head_loss_fwd(batch, hp)                 # or: forward now ...
  dX, dW, status = rl_head_loss_bwd(batch, hp, fwd.saved, dloss)   # ... backward later
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "librlhead.so")

RL_OK, RL_ERR_ARG, RL_ERR_WORKSPACE, RL_ERR_UNSUPPORTED, RL_ERR_CUDA = 0, 1, 2, 3, 4
RL_LOSS_IPO, RL_LOSS_ICEPOP, RL_LOSS_REINFORCE = 0, 1, 2
RL_KL_EXACT, RL_KL_K1 = 0, 1
RL_STALE_NONE, RL_STALE_INV_SQRT = 0, 1
RL_BWD_AUTO, RL_BWD_DENSE, RL_BWD_SPARSE = 0, 1, 2
RL_GRAD_BF16, RL_GRAD_SPLIT = 0, 1
STATUS_BITS = {
    0x0001: "OFFSETS", 0x0002: "ID_RANGE", 0x0004: "LOGQ", 0x0008: "LABEL_MISSING",
    0x0010: "SUPPORT_MASS", 0x0020: "EMPTY_ROW", 0x0040: "ROW_ORDER",
    0x0080: "SPARSE_INELIGIBLE", 0x0100: "NONFINITE", 0x0200: "TIMEOUT",
}
RL_PG_MAX_CURVE = 16


class RlParams(ctypes.Structure):
    _fields_ = [("loss_type", ctypes.c_int32), ("kl_estimator", ctypes.c_int32),
                ("kl_staleness", ctypes.c_int32), ("bwd_mode", ctypes.c_int32),
                ("grad_precision", ctypes.c_int32), ("all_replayed", ctypes.c_int32),
                ("eps", ctypes.c_float), ("max_importance_ratio", ctypes.c_float),
                ("icepop_low", ctypes.c_float), ("icepop_high", ctypes.c_float),
                ("adv_tau", ctypes.c_float), ("temperature", ctypes.c_float),
                ("kl_coeff", ctypes.c_float), ("token_chunk", ctypes.c_int32),
                ("entropy_coeff", ctypes.c_float), ("keep_e", ctypes.c_int32)]


class RlSupport(ctypes.Structure):
    _fields_ = [("offsets", ctypes.c_void_p), ("ids", ctypes.c_void_p), ("logq", ctypes.c_void_p),
                ("replayed", ctypes.c_void_p), ("nnz", ctypes.c_int64)]


class RlHeadBatch(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_void_p), ("weight", ctypes.c_void_p), ("N", ctypes.c_int64),
                ("H", ctypes.c_int64), ("V", ctypes.c_int64), ("labels", ctypes.c_void_p),
                ("label_logq", ctypes.c_void_p), ("adv", ctypes.c_void_p),
                ("loss_mask", ctypes.c_void_p), ("age", ctypes.c_void_p), ("support", RlSupport)]


class RlHeadMetrics(ctypes.Structure):
    _fields_ = [(k, ctypes.c_double) for k in ("loss", "mismatch_kl", "support_mass", "mask_tv", "kl",
                                               "beta", "kl_age0", "entropy")] + \
               [(k, ctypes.c_int64) for k in ("n_rl", "masked", "masked_low", "masked_high", "n_age0",
                                              "recomputed_chunks")]


class RlHeadOutputs(ctypes.Structure):
    _fields_ = [("loss", ctypes.c_void_p), ("logp_label", ctypes.c_void_p),
                ("logp_support", ctypes.c_void_p), ("entropy", ctypes.c_void_p),
                ("lse", ctypes.c_void_p), ("mask_label", ctypes.c_void_p),
                ("mask_support", ctypes.c_void_p), ("metrics", ctypes.c_void_p)]


class RlPgParams(ctypes.Structure):
    _fields_ = [("clip_ratio_low", ctypes.c_float), ("clip_ratio_high", ctypes.c_float),
                ("clip_ratio_c", ctypes.c_float), ("tis_upper", ctypes.c_float),
                ("icepop_low", ctypes.c_float), ("icepop_high", ctypes.c_float),
                ("n_curve", ctypes.c_int32), ("curve_eps", ctypes.c_float * RL_PG_MAX_CURVE)]


class RlPgMetrics(ctypes.Structure):
    _fields_ = [(k, ctypes.c_double) for k in ("loss_ppo", "loss_dec", "ppo_kl", "mis_kl", "k3",
                                               "tis_sum")] + \
               [(k, ctypes.c_int64) for k in ("n_valid", "n_clip", "n_clip_lower", "icepop_low",
                                              "icepop_high", "n_tis_trunc")] + \
               [("ipo_curve", ctypes.c_int64 * RL_PG_MAX_CURVE), ("status", ctypes.c_int64)]


class RlRcParams(ctypes.Structure):
    _fields_ = [("use_tis", ctypes.c_int32), ("tis_mode", ctypes.c_int32), ("tis_level", ctypes.c_int32),
                ("tis_batch_normalize", ctypes.c_int32), ("tis_lower_bound", ctypes.c_float),
                ("tis_upper_bound", ctypes.c_float), ("use_rs", ctypes.c_int32), ("rs_level", ctypes.c_int32),
                ("rs_lower_bound", ctypes.c_float), ("rs_upper_bound", ctypes.c_float),
                ("rs_veto_threshold", ctypes.c_float)]


class RlRcMetrics(ctypes.Structure):
    _fields_ = [(k, ctypes.c_double) for k in (
        "w_before_sum", "w_after_sum", "kept_w_sum", "batch_norm_factor", "final_sum", "final_min", "final_max",
        "mis_kl_sum", "k3_sum", "abs_diff_sum", "chi2_token_sum", "train_lppl_sum", "rollout_lppl_sum",
        "lppl_diff_sum", "lppl_abs_diff_sum", "ppl_ratio_sum", "chi2_seq_sum")] + \
               [(k, ctypes.c_int64) for k in (
                   "n_valid", "n_seq", "n_kept", "n_tis_low", "n_tis_high", "n_rs_low", "n_rs_high",
                   "n_cat_tokens", "n_cat_seqs", "status")]


class RlRcNamed(ctypes.Structure):
    _fields_ = [(k, ctypes.c_double) for k in (
        "training_log_ppl", "training_ppl", "rollout_log_ppl", "rollout_ppl", "kl", "k3_kl", "log_ppl_diff",
        "log_ppl_abs_diff", "ppl_ratio", "chi2_token", "chi2_seq", "train_rollout_logprob_abs_diff",
        "tis_weight_before_bound", "tis_weight_after_bound", "tis_truncate_fraction", "tis_clip_fraction_low",
        "tis_clip_fraction_high", "tis_mask_fraction_low", "tis_mask_fraction_high", "rs_mask_fraction_low",
        "rs_mask_fraction_high", "rs_catastrophic_token_fraction", "rs_catastrophic_seq_fraction",
        "is_ratio_mean_after_tis_rs", "batch_norm_factor", "is_ratio_mean_final", "is_ratio_min_final",
        "is_ratio_max_final")]


_lib = None

_SIGS = {
    "rl_head_saved_bytes": (ctypes.c_size_t, [ctypes.c_int64, ctypes.c_int64]),
    "rl_head_saved_bytes_ex": (ctypes.c_size_t, [ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                                 ctypes.POINTER(RlParams)]),
    "rl_head_token_chunk": (ctypes.c_int64, [ctypes.c_int64, ctypes.c_int64, ctypes.POINTER(RlParams)]),
    "rl_head_fwd_workspace_bytes": (ctypes.c_size_t, [ctypes.c_int64] * 4 + [ctypes.c_void_p]),
    "rl_head_bwd_workspace_bytes": (ctypes.c_size_t, [ctypes.c_int64] * 4 + [ctypes.c_void_p]),
    "rl_validate_support": (ctypes.c_int, [ctypes.c_void_p] * 3),
    "rl_head_loss_fwd": (ctypes.c_int, [ctypes.c_void_p] * 5 + [ctypes.c_size_t] + [ctypes.c_void_p] * 2),
    "rl_head_loss_bwd": (ctypes.c_int, [ctypes.c_void_p] * 6 + [ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t,
                                                                ctypes.c_void_p, ctypes.c_void_p]),
    "rl_mismatch_metrics": (ctypes.c_int, [ctypes.c_void_p] * 4 + [ctypes.c_size_t, ctypes.c_void_p]),
    "rl_head_shard_remap": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                           ctypes.c_void_p, ctypes.c_void_p]),
    "rl_head_shard_stats": (ctypes.c_int, [ctypes.c_void_p] * 6 + [ctypes.c_size_t, ctypes.c_void_p, ctypes.c_void_p]),
    "rl_head_loss_from_shard_stats": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32]
                                      + [ctypes.c_void_p] * 6 + [ctypes.c_size_t, ctypes.c_void_p, ctypes.c_void_p]),
    "rl_head_fwd_bwd_workspace_bytes": (ctypes.c_size_t, [ctypes.c_int64] * 4 + [ctypes.c_void_p]),
    "rl_head_loss_fwd_bwd": (ctypes.c_int, [ctypes.c_void_p] * 6 + [ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                                                                    ctypes.c_size_t, ctypes.c_void_p,
                                                                    ctypes.c_void_p]),
    "rl_policy_workspace_bytes": (ctypes.c_size_t, [ctypes.c_int64]),
    "rl_rollout_correction_workspace_bytes": (ctypes.c_size_t, [ctypes.c_int64]),
    "rl_rollout_metrics_named": (ctypes.c_int, [ctypes.c_void_p] * 4),
    "rl_rollout_correction": (ctypes.c_int, [ctypes.c_void_p] * 4 + [ctypes.c_int64] * 2 + [ctypes.c_void_p] * 5
                              + [ctypes.c_size_t, ctypes.c_void_p]),
    "rl_policy_loss_elementwise": (ctypes.c_int, [ctypes.c_void_p] * 5 + [ctypes.c_int64] + [ctypes.c_void_p] * 7
                                   + [ctypes.c_size_t, ctypes.c_void_p]),
    "rl_policy_loss_elementwise_noalloc": (ctypes.c_int, [ctypes.c_void_p] * 5 + [ctypes.c_int64]
                                           + [ctypes.c_void_p] * 7),
    "rl_status_read": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p]),
    "rl_wait_selftest": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p]),
    "rl_gemm_bf16_tn": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p] + [ctypes.c_int64] * 3
                        + [ctypes.c_void_p] * 3),
    "rl_gemm_bf16": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_int]
                     + [ctypes.c_int64] * 3 + [ctypes.c_void_p] * 3),
    "rl_kernel_launch_count": (ctypes.c_int64, []),
    "rl_set_option": (ctypes.c_int, [ctypes.c_int, ctypes.c_int]),
    "rl_get_option": (ctypes.c_int, [ctypes.c_int]),
    "rl_profile_enable": (ctypes.c_int, [ctypes.c_int]),
    "rl_profile_read": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p]),
    "rl_profile_kind_name": (ctypes.c_char_p, [ctypes.c_int]),
    "rl_error_string": (ctypes.c_char_p, [ctypes.c_int]),
    "rl_last_error": (ctypes.c_char_p, []),
}


def load(path: Optional[str] = None):
    """Load librlhead.so (built by lm_head_gb300.build).  Raises if it is missing."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"librlhead.so not built at {p}; run lm_head_gb300.build.build()")
    lib = ctypes.CDLL(p)
    for name, (res, args) in _SIGS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path is None:
        _lib = lib
    return lib


class RLHeadError(RuntimeError):
    pass


def _check(rc: int):
    if rc != RL_OK:
        lib = load()
        raise RLHeadError(f"{lib.rl_error_string(rc).decode()}: {lib.rl_last_error().decode()}")


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _require_cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise RLHeadError("librlhead takes device tensors; got a CPU tensor")


@dataclasses.dataclass
class HeadParams:
    """Knobs of rl_params (defaults from the pages: eps 0.3, kl_coeff 0)."""
    loss_type: int = RL_LOSS_IPO
    eps: float = 0.3
    max_importance_ratio: float = 10.0
    icepop_low: float = 0.5
    icepop_high: float = 2.0
    adv_tau: float = 1.0
    temperature: float = 1.0
    kl_coeff: float = 0.0
    kl_estimator: int = RL_KL_EXACT
    kl_staleness: int = RL_STALE_NONE
    bwd_mode: int = RL_BWD_AUTO
    grad_precision: int = RL_GRAD_BF16
    all_replayed: int = 0
    token_chunk: int = 0
    entropy_coeff: float = 0.0
    keep_e: int = 0

    def c(self) -> RlParams:
        return RlParams(self.loss_type, self.kl_estimator, self.kl_staleness, self.bwd_mode,
                        self.grad_precision, self.all_replayed, self.eps, self.max_importance_ratio,
                        self.icepop_low, self.icepop_high, self.adv_tau, self.temperature,
                        self.kl_coeff, self.token_chunk, self.entropy_coeff, self.keep_e)


@dataclasses.dataclass
class HeadBatch:
    """Device tensors of one batch (see include/rlhead.h, rl_head_batch)."""
    hidden: torch.Tensor        # [N, H] bf16
    weight: torch.Tensor        # [V, H] bf16
    labels: torch.Tensor        # [N] int32
    label_logq: torch.Tensor    # [N] fp32
    adv: torch.Tensor           # [N] fp32
    offsets: torch.Tensor       # [N+1] int64
    ids: torch.Tensor           # [nnz] int32
    logq: torch.Tensor          # [nnz] fp32
    replayed: torch.Tensor      # [N] uint8
    loss_mask: Optional[torch.Tensor] = None   # [N] uint8
    age: Optional[torch.Tensor] = None         # [N] int32

    @property
    def N(self):
        return int(self.hidden.shape[0])

    @property
    def H(self):
        return int(self.hidden.shape[1])

    @property
    def V(self):
        return int(self.weight.shape[0])

    @property
    def nnz(self):
        return int(self.ids.shape[0])

    def c(self, V: Optional[int] = None) -> RlHeadBatch:
        """The C struct; V overrides the vocabulary size (the whole vocabulary when `weight`
        holds only one rank's rows)."""
        _require_cuda(self.hidden, self.weight, self.labels, self.label_logq, self.adv, self.offsets,
                      self.ids, self.logq, self.replayed, self.loss_mask, self.age)
        for name, t, dt in (("hidden", self.hidden, torch.bfloat16), ("weight", self.weight, torch.bfloat16),
                            ("labels", self.labels, torch.int32), ("label_logq", self.label_logq, torch.float32),
                            ("adv", self.adv, torch.float32), ("offsets", self.offsets, torch.int64),
                            ("ids", self.ids, torch.int32), ("logq", self.logq, torch.float32),
                            ("replayed", self.replayed, torch.uint8)):
            if t.dtype != dt or not t.is_contiguous():
                raise RLHeadError(f"{name}: expected contiguous {dt}, got {t.dtype}")
        sup = RlSupport(self.offsets.data_ptr(), self.ids.data_ptr() if self.nnz else None,
                        self.logq.data_ptr() if self.nnz else None, self.replayed.data_ptr(), self.nnz)
        return RlHeadBatch(self.hidden.data_ptr(), self.weight.data_ptr(), self.N, self.H, self.V if V is None else V,
                           self.labels.data_ptr(), self.label_logq.data_ptr(), self.adv.data_ptr(),
                           None if self.loss_mask is None else self.loss_mask.data_ptr(),
                           None if self.age is None else self.age.data_ptr(), sup)

    @staticmethod
    def from_case(case) -> "HeadBatch":
        """From a workloads.HeadCase already on the device."""
        return HeadBatch(case.hidden, case.W, case.labels, case.label_logq, case.adv, case.offsets,
                         case.ids, case.logq, case.replayed, case.loss_mask, case.age)


@dataclasses.dataclass
class HeadForward:
    loss: torch.Tensor
    logp_label: torch.Tensor
    logp_support: torch.Tensor
    entropy: torch.Tensor
    lse: torch.Tensor
    mask_label: torch.Tensor
    mask_support: torch.Tensor
    metrics_dev: torch.Tensor
    saved: torch.Tensor
    status: torch.Tensor

    def metrics(self) -> dict:
        m = RlHeadMetrics.from_buffer_copy(bytes(self.metrics_dev.cpu().numpy().tobytes()))
        return {f: getattr(m, f) for f, _ in RlHeadMetrics._fields_}

    def status_bits(self) -> int:
        return int(self.status.item())


def _u8(n, device):
    return torch.empty(max(int(n), 1), dtype=torch.uint8, device=device)


def rl_head_saved_bytes(N: int, nnz: int) -> int:
    return int(load().rl_head_saved_bytes(N, nnz))


def rl_head_token_chunk(N: int, H: int, params: HeadParams) -> int:
    p = params.c()
    return int(load().rl_head_token_chunk(N, H, ctypes.byref(p)))


def rl_head_saved_bytes_ex(N: int, nnz: int, V: int, params: HeadParams) -> int:
    p = params.c()
    return int(load().rl_head_saved_bytes_ex(N, nnz, V, ctypes.byref(p)))


def rl_head_fwd_workspace_bytes(N, H, V, nnz, params: HeadParams) -> int:
    p = params.c()
    return int(load().rl_head_fwd_workspace_bytes(N, H, V, nnz, ctypes.byref(p)))


def rl_head_bwd_workspace_bytes(N, H, V, nnz, params: HeadParams) -> int:
    p = params.c()
    return int(load().rl_head_bwd_workspace_bytes(N, H, V, nnz, ctypes.byref(p)))


def rl_validate_support(batch: HeadBatch, status: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    lib = load()
    dev = batch.hidden.device
    st = torch.zeros(1, dtype=torch.int32, device=dev) if status is None else status
    cb = batch.c()
    _check(lib.rl_validate_support(ctypes.byref(cb), _ptr(st), _stream(stream)))
    return st


def rl_head_loss_fwd(batch: HeadBatch, params: HeadParams, *, ws: Optional[torch.Tensor] = None,
                     saved: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None,
                     want_metrics: bool = True, stream=None) -> HeadForward:
    lib = load()
    dev = batch.hidden.device
    N, nnz = batch.N, batch.nnz
    f32 = dict(dtype=torch.float32, device=dev)
    out = HeadForward(
        loss=torch.empty(N, **f32), logp_label=torch.empty(N, **f32),
        logp_support=torch.empty(max(nnz, 1), **f32)[:nnz], entropy=torch.empty(N, **f32),
        lse=torch.empty(N, **f32), mask_label=torch.empty(N, dtype=torch.uint8, device=dev),
        mask_support=torch.empty(max(nnz, 1), dtype=torch.uint8, device=dev)[:nnz],
        metrics_dev=torch.zeros(ctypes.sizeof(RlHeadMetrics), dtype=torch.uint8, device=dev),
        saved=saved if saved is not None else _u8(rl_head_saved_bytes_ex(N, nnz, batch.V, params), dev),
        status=torch.zeros(1, dtype=torch.int32, device=dev) if status is None else status)
    wsb = rl_head_fwd_workspace_bytes(N, batch.H, batch.V, nnz, params)
    if ws is None:
        ws = _u8(wsb, dev)
    p = params.c()
    cb = batch.c()
    co = RlHeadOutputs(out.loss.data_ptr(), out.logp_label.data_ptr(),
                       out.logp_support.data_ptr() if nnz else None, out.entropy.data_ptr(),
                       out.lse.data_ptr(), out.mask_label.data_ptr(),
                       out.mask_support.data_ptr() if nnz else None,
                       out.metrics_dev.data_ptr() if want_metrics else None)
    _check(lib.rl_head_loss_fwd(ctypes.byref(cb), ctypes.byref(p), ctypes.byref(co), _ptr(out.saved),
                                _ptr(ws), ws.numel(), _ptr(out.status), _stream(stream)))
    return out


def rl_head_loss_bwd(batch: HeadBatch, params: HeadParams, saved: torch.Tensor, dloss: torch.Tensor, *,
                     dhidden: Optional[torch.Tensor] = None, dW: Optional[torch.Tensor] = None,
                     accumulate_dW: bool = False, ws: Optional[torch.Tensor] = None,
                     status: Optional[torch.Tensor] = None, stream=None):
    lib = load()
    dev = batch.hidden.device
    _require_cuda(dloss)
    if dloss.dtype != torch.float32 or dloss.numel() != batch.N:
        raise RLHeadError("dloss must be fp32 [N]")
    if dhidden is None:
        dhidden = torch.empty(batch.N, batch.H, dtype=torch.bfloat16, device=dev)
    if dW is None:
        dW = torch.empty(batch.V, batch.H, dtype=torch.float32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev) if status is None else status
    if ws is None:
        ws = _u8(rl_head_bwd_workspace_bytes(batch.N, batch.H, batch.V, batch.nnz, params), dev)
    p = params.c()
    cb = batch.c()
    _check(lib.rl_head_loss_bwd(ctypes.byref(cb), ctypes.byref(p), _ptr(saved), _ptr(dloss), _ptr(dhidden),
                                _ptr(dW), int(bool(accumulate_dW)), _ptr(ws), ws.numel(), _ptr(st),
                                _stream(stream)))
    return dhidden, dW, st


def rl_head_fwd_bwd_workspace_bytes(N, H, V, nnz, params: HeadParams) -> int:
    p = params.c()
    return int(load().rl_head_fwd_bwd_workspace_bytes(N, H, V, nnz, ctypes.byref(p)))


def rl_head_loss_fwd_bwd(batch: HeadBatch, params: HeadParams, dloss: torch.Tensor, *,
                         dhidden: Optional[torch.Tensor] = None, dW: Optional[torch.Tensor] = None,
                         accumulate_dW: bool = False, ws: Optional[torch.Tensor] = None,
                         saved: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None,
                         want_metrics: bool = True, stream=None):
    """Forward + backward in one call (dloss known up front).  Returns (HeadForward, dhidden, dW)."""
    lib = load()
    dev = batch.hidden.device
    _require_cuda(dloss)
    if dloss.dtype != torch.float32 or dloss.numel() != batch.N:
        raise RLHeadError("dloss must be fp32 [N]")
    N, nnz = batch.N, batch.nnz
    f32 = dict(dtype=torch.float32, device=dev)
    out = HeadForward(
        loss=torch.empty(N, **f32), logp_label=torch.empty(N, **f32),
        logp_support=torch.empty(max(nnz, 1), **f32)[:nnz], entropy=torch.empty(N, **f32),
        lse=torch.empty(N, **f32), mask_label=torch.empty(N, dtype=torch.uint8, device=dev),
        mask_support=torch.empty(max(nnz, 1), dtype=torch.uint8, device=dev)[:nnz],
        metrics_dev=torch.zeros(ctypes.sizeof(RlHeadMetrics), dtype=torch.uint8, device=dev),
        saved=saved if saved is not None else _u8(rl_head_saved_bytes(N, nnz), dev),
        status=torch.zeros(1, dtype=torch.int32, device=dev) if status is None else status)
    if dhidden is None:
        dhidden = torch.empty(N, batch.H, dtype=torch.bfloat16, device=dev)
    if dW is None:
        dW = torch.empty(batch.V, batch.H, dtype=torch.float32, device=dev)
    if ws is None:
        ws = _u8(rl_head_fwd_bwd_workspace_bytes(N, batch.H, batch.V, nnz, params), dev)
    p = params.c()
    cb = batch.c()
    co = RlHeadOutputs(out.loss.data_ptr(), out.logp_label.data_ptr(),
                       out.logp_support.data_ptr() if nnz else None, out.entropy.data_ptr(),
                       out.lse.data_ptr(), out.mask_label.data_ptr(),
                       out.mask_support.data_ptr() if nnz else None,
                       out.metrics_dev.data_ptr() if want_metrics else None)
    _check(lib.rl_head_loss_fwd_bwd(ctypes.byref(cb), ctypes.byref(p), ctypes.byref(co), _ptr(dloss), _ptr(dhidden),
                                    _ptr(dW), int(bool(accumulate_dW)), _ptr(out.saved), _ptr(ws), ws.numel(),
                                    _ptr(out.status), _stream(stream)))
    return out, dhidden, dW


def rl_mismatch_metrics(batch: HeadBatch, saved: torch.Tensor, params: HeadParams, *,
                        ws: Optional[torch.Tensor] = None, stream=None) -> dict:
    lib = load()
    dev = batch.hidden.device
    m = torch.zeros(ctypes.sizeof(RlHeadMetrics), dtype=torch.uint8, device=dev)
    if ws is None:
        ws = _u8(rl_head_fwd_workspace_bytes(batch.N, batch.H, batch.V, batch.nnz, params), dev)
    cb = batch.c()
    _check(lib.rl_mismatch_metrics(ctypes.byref(cb), _ptr(saved), _ptr(m), _ptr(ws), ws.numel(), _stream(stream)))
    mm = RlHeadMetrics.from_buffer_copy(bytes(m.cpu().numpy().tobytes()))
    return {f: getattr(mm, f) for f, _ in RlHeadMetrics._fields_}


def rl_head_shard_remap(ids: torch.Tensor, vocab_begin: int, vocab_end: int, out: Optional[torch.Tensor] = None,
                        stream=None) -> torch.Tensor:
    """Global ids (int32, device) in the local numbering of the vocabulary rows
    [vocab_begin, vocab_end): -1 below, vocab_end - vocab_begin above (include/rlhead.h)."""
    _require_cuda(ids)
    out = torch.empty_like(ids) if out is None else out
    _check(load().rl_head_shard_remap(_ptr(ids), int(ids.numel()), int(vocab_begin), int(vocab_end), _ptr(out),
                                      _stream(stream)))
    return out


def rl_head_shard_stats(shard: HeadBatch, params: HeadParams, *, ws: Optional[torch.Tensor] = None,
                        status: Optional[torch.Tensor] = None, stream=None):
    """One rank's logsumexp statistics [3, N] (m, s, u) and owned label / support logits."""
    lib = load()
    dev = shard.hidden.device
    N, nnz = shard.N, shard.nnz
    stats = torch.empty(3, N, dtype=torch.float32, device=dev)
    zlab = torch.empty(N, dtype=torch.float32, device=dev)
    zsup = torch.empty(max(nnz, 1), dtype=torch.float32, device=dev)[:nnz]
    st = torch.zeros(1, dtype=torch.int32, device=dev) if status is None else status
    if ws is None:
        ws = _u8(rl_head_fwd_workspace_bytes(N, shard.H, shard.V, nnz, params), dev)
    p = params.c()
    cb = shard.c()
    _check(lib.rl_head_shard_stats(ctypes.byref(cb), ctypes.byref(p), _ptr(stats), _ptr(zlab),
                                   _ptr(zsup) if nnz else None, _ptr(ws), ws.numel(), _ptr(st), _stream(stream)))
    return stats, zlab, zsup


def rl_head_loss_from_shard_stats(batch: HeadBatch, params: HeadParams, stats_all: torch.Tensor, zlab: torch.Tensor,
                                  zsup: torch.Tensor, *, V: int, ws: Optional[torch.Tensor] = None,
                                  status: Optional[torch.Tensor] = None, want_metrics: bool = True,
                                  stream=None) -> HeadForward:
    """The forward's outputs from the ranks' gathered statistics [R, 3, N] and the summed
    owned logits; `batch` in global numbering, V the whole vocabulary."""
    lib = load()
    _require_cuda(stats_all, zlab, zsup)
    dev = batch.hidden.device
    N, nnz = batch.N, batch.nnz
    f32 = dict(dtype=torch.float32, device=dev)
    out = HeadForward(
        loss=torch.empty(N, **f32), logp_label=torch.empty(N, **f32),
        logp_support=torch.empty(max(nnz, 1), **f32)[:nnz], entropy=torch.empty(N, **f32),
        lse=torch.empty(N, **f32), mask_label=torch.empty(N, dtype=torch.uint8, device=dev),
        mask_support=torch.empty(max(nnz, 1), dtype=torch.uint8, device=dev)[:nnz],
        metrics_dev=torch.zeros(ctypes.sizeof(RlHeadMetrics), dtype=torch.uint8, device=dev),
        saved=_u8(rl_head_saved_bytes(N, nnz), dev),
        status=torch.zeros(1, dtype=torch.int32, device=dev) if status is None else status)
    if ws is None:
        ws = _u8(rl_head_fwd_workspace_bytes(N, batch.H, V, nnz, params), dev)
    p = params.c()
    cb = batch.c(V=V)
    co = RlHeadOutputs(out.loss.data_ptr(), out.logp_label.data_ptr(),
                       out.logp_support.data_ptr() if nnz else None, out.entropy.data_ptr(),
                       out.lse.data_ptr(), out.mask_label.data_ptr(),
                       out.mask_support.data_ptr() if nnz else None,
                       out.metrics_dev.data_ptr() if want_metrics else None)
    R = int(stats_all.shape[0])
    _check(lib.rl_head_loss_from_shard_stats(ctypes.byref(cb), ctypes.byref(p), R, _ptr(stats_all.contiguous()),
                                             _ptr(zlab), _ptr(zsup) if nnz else None, ctypes.byref(co),
                                             _ptr(out.saved), _ptr(ws), ws.numel(), _ptr(out.status),
                                             _stream(stream)))
    return out


@dataclasses.dataclass
class PgParams:
    clip_ratio_low: float = 0.2
    clip_ratio_high: float = 0.2
    clip_ratio_c: float = 3.0
    tis_upper: float = 2.0
    icepop_low: float = 0.5
    icepop_high: float = 2.0
    curve_eps: tuple = tuple(round(0.05 * k, 2) for k in range(1, 11))

    def c(self) -> RlPgParams:
        arr = (ctypes.c_float * RL_PG_MAX_CURVE)(*([float(e) for e in self.curve_eps]
                                                   + [0.0] * (RL_PG_MAX_CURVE - len(self.curve_eps))))
        return RlPgParams(self.clip_ratio_low, self.clip_ratio_high, self.clip_ratio_c, self.tis_upper,
                          self.icepop_low, self.icepop_high, len(self.curve_eps), arr)


def rl_policy_workspace_bytes(T: int) -> int:
    return int(load().rl_policy_workspace_bytes(T))


def rl_policy_loss_elementwise(lp_theta, lp_old, lp_samp, adv, mask, params: PgParams, *, outputs=None,
                               ws: Optional[torch.Tensor] = None, metrics_dev: Optional[torch.Tensor] = None,
                               stream=None):
    """Returns (loss_ppo, loss_dec, grad_ppo, grad_dec, metrics_dev); metrics via pg_metrics()."""
    """mask None: packed input, every slot a valid token."""
    lib = load()
    _require_cuda(lp_theta, lp_old, lp_samp, adv, mask)
    T = int(lp_theta.numel())
    dev = lp_theta.device
    if outputs is None:
        outputs = tuple(torch.empty(T, dtype=torch.float32, device=dev) for _ in range(4))
    if metrics_dev is None:
        metrics_dev = torch.zeros(ctypes.sizeof(RlPgMetrics), dtype=torch.uint8, device=dev)
    if ws is None:   # zeroed once before its first use (include/rlhead.h)
        ws = torch.zeros(rl_policy_workspace_bytes(T), dtype=torch.uint8, device=dev)
    p = params.c()
    _check(lib.rl_policy_loss_elementwise(_ptr(lp_theta), _ptr(lp_old), _ptr(lp_samp), _ptr(adv), _ptr(mask), T,
                                          ctypes.byref(p), *[_ptr(o) for o in outputs], _ptr(metrics_dev),
                                          _ptr(ws), ws.numel(), _stream(stream)))
    return (*outputs, metrics_dev)


def rl_policy_loss_elementwise_noalloc(lp_theta, lp_old, lp_samp, adv, mask, params: PgParams, *, outputs,
                                       metrics_dev, stream=None):
    """rl_policy_loss_elementwise without a workspace, for callers that cannot allocate
    device memory: the library's scratch is a static device array (see include/rlhead.h).
    The caller passes every buffer, outputs and the metrics struct included."""
    lib = load()
    _require_cuda(lp_theta, lp_old, lp_samp, adv, mask, metrics_dev, *[o for o in outputs if o is not None])
    T = int(lp_theta.numel())
    p = params.c()
    _check(lib.rl_policy_loss_elementwise_noalloc(_ptr(lp_theta), _ptr(lp_old), _ptr(lp_samp), _ptr(adv),
                                                  _ptr(mask), T, ctypes.byref(p), *[_ptr(o) for o in outputs],
                                                  _ptr(metrics_dev), _stream(stream)))
    return (*outputs, metrics_dev)


RL_TIS_TRUNCATE, RL_TIS_CLIP, RL_TIS_MASK = 0, 1, 2
RL_LEVEL_TOKEN, RL_LEVEL_SEQUENCE, RL_LEVEL_GEOMETRIC = 0, 1, 2
_TIS_MODES = {"truncate": RL_TIS_TRUNCATE, "clip": RL_TIS_CLIP, "mask": RL_TIS_MASK}
_LEVELS = {"token": RL_LEVEL_TOKEN, "sequence": RL_LEVEL_SEQUENCE, "geometric": RL_LEVEL_GEOMETRIC}


@dataclasses.dataclass
class RcParams:
    """Rollout-correction knobs ("Rollout Correction Methods", "Config keys")."""
    use_tis: bool = True
    tis_mode: str = "truncate"
    tis_lower_bound: float = 0.5
    tis_upper_bound: float = 2.0
    tis_level: str = "token"
    tis_batch_normalize: bool = False
    use_rs: bool = False
    rs_lower_bound: Optional[float] = None      # None: the tis bound
    rs_upper_bound: Optional[float] = None
    rs_level: str = "token"
    rs_veto_threshold: Optional[float] = None   # None: no veto

    def c(self) -> RlRcParams:
        nan = float("nan")
        return RlRcParams(int(self.use_tis), _TIS_MODES[self.tis_mode], _LEVELS[self.tis_level],
                          int(self.tis_batch_normalize), self.tis_lower_bound, self.tis_upper_bound,
                          int(self.use_rs), _LEVELS[self.rs_level],
                          nan if self.rs_lower_bound is None else self.rs_lower_bound,
                          nan if self.rs_upper_bound is None else self.rs_upper_bound,
                          nan if self.rs_veto_threshold is None else self.rs_veto_threshold)


def rl_rollout_correction_workspace_bytes(B: int) -> int:
    return int(load().rl_rollout_correction_workspace_bytes(B))


def rl_rollout_correction(lp_train, lp_rollout, mask, seq_offsets, params: RcParams, *, outputs=None,
                          ws: Optional[torch.Tensor] = None, metrics_dev: Optional[torch.Tensor] = None,
                          stream=None):
    """Returns (weights [T] fp32, keep [T] uint8, metrics_dev); metrics via rc_metrics()."""
    lib = load()
    _require_cuda(lp_train, lp_rollout, mask, seq_offsets)
    T = int(lp_train.numel())
    B = int(seq_offsets.numel()) - 1
    dev = lp_train.device
    if outputs is None:
        outputs = (torch.empty(T, dtype=torch.float32, device=dev), torch.empty(T, dtype=torch.uint8, device=dev))
    if metrics_dev is None:
        metrics_dev = torch.zeros(ctypes.sizeof(RlRcMetrics), dtype=torch.uint8, device=dev)
    if ws is None:   # zeroed once: the library leaves its counters at zero after each call
        ws = torch.zeros(max(rl_rollout_correction_workspace_bytes(B), 1), dtype=torch.uint8, device=dev)
    p = params.c()
    _check(lib.rl_rollout_correction(_ptr(lp_train), _ptr(lp_rollout), _ptr(mask), _ptr(seq_offsets), B, T,
                                     ctypes.byref(p), _ptr(outputs[0]), _ptr(outputs[1]), _ptr(metrics_dev),
                                     _ptr(ws), ws.numel(), _stream(stream)))
    return (*outputs, metrics_dev)


def rc_metrics(metrics_dev: torch.Tensor) -> dict:
    m = RlRcMetrics.from_buffer_copy(bytes(metrics_dev.cpu().numpy().tobytes()))
    return {f: getattr(m, f) for f, _ in RlRcMetrics._fields_}


def rl_rollout_metrics_named(metrics_dev: torch.Tensor, params: RcParams, stream=None) -> dict:
    """The named metrics of "Mismatch Metrics" (include/rlhead.h, rl_rc_named), formed on
    the device by the library from the sums and counts of rl_rollout_correction; the
    metrics these settings do not emit are NaN there and left out here."""
    import math
    _require_cuda(metrics_dev)
    out = torch.empty(ctypes.sizeof(RlRcNamed), dtype=torch.uint8, device=metrics_dev.device)
    p = params.c()
    _check(load().rl_rollout_metrics_named(_ptr(metrics_dev), ctypes.byref(p), _ptr(out), _stream(stream)))
    n = RlRcNamed.from_buffer_copy(bytes(out.cpu().numpy().tobytes()))
    return {f: getattr(n, f) for f, _ in RlRcNamed._fields_ if not math.isnan(getattr(n, f))}


def pg_metrics(metrics_dev: torch.Tensor, n_curve: int = 10) -> dict:
    m = RlPgMetrics.from_buffer_copy(bytes(metrics_dev.cpu().numpy().tobytes()))
    d = {f: getattr(m, f) for f, _ in RlPgMetrics._fields_ if f != "ipo_curve"}
    d["ipo_curve"] = [int(m.ipo_curve[k]) for k in range(n_curve)]
    return d


def rl_gemm_bf16_tn(A: torch.Tensor, B: torch.Tensor, D: Optional[torch.Tensor] = None,
                    status: Optional[torch.Tensor] = None, stream=None):
    """D[M, N] fp32 = A[M, K] @ B[N, K]^T on the tcgen05 path (bf16 inputs)."""
    _require_cuda(A, B)
    M, K = A.shape
    N = B.shape[0]
    if D is None:
        D = torch.empty(M, N, dtype=torch.float32, device=A.device)
    st = torch.zeros(1, dtype=torch.int32, device=A.device) if status is None else status
    _check(load().rl_gemm_bf16_tn(_ptr(A), _ptr(B), M, N, K, _ptr(D), _ptr(st), _stream(stream)))
    return D, st


def rl_gemm_bf16(A: torch.Tensor, a_mn_major: bool, B: torch.Tensor, b_mn_major: bool,
                 D: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None, stream=None):
    """D[M, N] fp32 = A B^T with A given as [M, K] or ([K, M], a_mn_major) and B as [N, K]
    or ([K, N], b_mn_major)."""
    _require_cuda(A, B)
    M = A.shape[1] if a_mn_major else A.shape[0]
    K = A.shape[0] if a_mn_major else A.shape[1]
    N = B.shape[1] if b_mn_major else B.shape[0]
    if D is None:
        D = torch.empty(M, N, dtype=torch.float32, device=A.device)
    st = torch.zeros(1, dtype=torch.int32, device=A.device) if status is None else status
    _check(load().rl_gemm_bf16(_ptr(A), int(bool(a_mn_major)), _ptr(B), int(bool(b_mn_major)), M, N, K, _ptr(D),
                               _ptr(st), _stream(stream)))
    return D, st


def rl_status_read(status: torch.Tensor) -> int:
    out = ctypes.c_int32(0)
    _check(load().rl_status_read(_ptr(status), ctypes.byref(out)))
    return int(out.value)


def rl_wait_selftest(status: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """A wait on an mbarrier nothing signals: runs out after RL_OPT_WAIT_LIMIT_US and sets
    RL_STATUS_TIMEOUT in the returned device status word."""
    st = torch.zeros(1, dtype=torch.int32, device="cuda") if status is None else status
    _require_cuda(st)
    _check(load().rl_wait_selftest(_ptr(st), _stream(stream)))
    return st


def rl_kernel_launch_count() -> int:
    return int(load().rl_kernel_launch_count())


RL_PROF_KINDS = 18


def rl_profile_enable(on: bool = True) -> None:
    _check(load().rl_profile_enable(int(bool(on))))


def rl_profile_read() -> dict:
    """{kind name: (total device ms, launches)} for kinds with launches; syncs on the events."""
    lib = load()
    ms = (ctypes.c_double * RL_PROF_KINDS)()
    n = (ctypes.c_int64 * RL_PROF_KINDS)()
    _check(lib.rl_profile_read(ctypes.cast(ms, ctypes.c_void_p), ctypes.cast(n, ctypes.c_void_p)))
    return {lib.rl_profile_kind_name(k).decode(): (float(ms[k]), int(n[k]))
            for k in range(RL_PROF_KINDS) if n[k] > 0}


RL_OPT_GEMM_PAIR = 1
RL_OPT_WAIT_LIMIT_US = 2


def rl_set_option(key: int, value: int) -> None:
    _check(load().rl_set_option(int(key), int(value)))


def rl_get_option(key: int) -> int:
    return int(load().rl_get_option(int(key)))


def status_names(bits: int):
    return [n for b, n in STATUS_BITS.items() if bits & b]
