"""Benchmark of the fused LM head + unified RL loss, forward + backward, on one GB300.

Contract: `python bench.py --gpus N --steps K --warmup W [--impl reference]` prints ONE
JSON line (rank 0).  A step is one forward + backward of the whole hot path
(validation, tensor-core logits with online logsumexp and support gather, per-token
loss / weights / KL / metrics, dense softmax-gradient backward with the sparse spike
terms) over one batch of the 64k-token workload: N=65536 tokens (128 sequences of
512), H=2048, V=151936, K=16 untruncated sampler draws per token, ipo eps=0.3 with
max_importance_ratio 10, exact KL(q||p) with kl_coeff 0.01 and inv_sqrt staleness over
ages 0..4, dense backward, bf16 operands with fp32 accumulation.

`value` is tokens/s with inputs resident in device memory; `e2e` is the same metric
through the public API with the batch copied from pinned host memory and the loss and
metrics read back every step.  Under torchrun each rank runs its own batch (weak
scaling, replicas: the head's per-token work has no exchange step); rank 0 prints the
max-over-ranks time.  `--impl reference` times the fp64 CPU oracle on a bounded sample
of the same workload instead.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "LM-head+RLLoss fwd+bwd tokens/s at 64k tok, V=152k; % of bf16 TC peak"
WORKLOAD = ("c4: N=65536 tokens (128 seq x 512), H=2048, V=151936, K=16 untruncated sampler "
            "draws/token, ipo eps=0.3 cap 10, exact KL(q||p) kl_coeff=0.01 inv_sqrt age U{0..4}, "
            "dense backward")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                  "source": "fallback"}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        d["source"] = "measured"
        return d
    except Exception:
        return dict(FALLBACK_PEAKS)


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def aggregate(local_ms: float, local_tokens: int, world: int, group=None):
    """Max of step time and sum of tokens over ranks -> (ms, tokens, tokens/s)."""
    import torch
    import torch.distributed as dist
    if world > 1:
        dev = "cuda" if dist.get_backend(group) == "nccl" else "cpu"
        t = torch.tensor([local_ms], dtype=torch.float64, device=dev)
        n = torch.tensor([float(local_tokens)], dtype=torch.float64, device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
        dist.all_reduce(n, op=dist.ReduceOp.SUM, group=group)
        local_ms, tokens = float(t.item()), int(n.item())
    else:
        tokens = local_tokens
    return local_ms, tokens, tokens / (local_ms / 1e3)


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms while running."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        rows = []
        try:
            with open(self.path) as f:
                for line in f:
                    parts = [x.strip() for x in line.split(",")]
                    if len(parts) >= 9:
                        rows.append(parts)
        except Exception:
            pass
        finally:
            if self.path and os.path.exists(self.path):
                os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        pw = [num(r[3]) for r in rows if num(r[3]) is not None]
        reasons = set()
        for r in rows:
            for name, v in (("hw_slowdown", r[5]), ("hw_thermal_slowdown", r[6]),
                            ("sw_thermal_slowdown", r[7]), ("sw_power_cap", r[8])):
                if v.lower().startswith("active"):
                    reasons.add(name)
        top = max(sm) if sm else 0
        loaded = [s for s in sm if s >= 0.5 * top] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(mx) if mx else None, "power_w_max": max(pw) if pw else None,
                "reasons": sorted(reasons), "samples": len(rows)}


def head_params(rh, grad_precision: str):
    return rh.HeadParams(loss_type=rh.RL_LOSS_IPO, eps=0.3, max_importance_ratio=10.0, kl_coeff=0.01,
                         kl_estimator=rh.RL_KL_EXACT, kl_staleness=rh.RL_STALE_INV_SQRT,
                         bwd_mode=rh.RL_BWD_DENSE,
                         grad_precision=rh.RL_GRAD_SPLIT if grad_precision == "split" else rh.RL_GRAD_BF16)


def cpu_baseline(case_host: dict, n_tokens: int, threads: int):
    """Time the fp64 oracle's forward + backward on the first n_tokens of the batch."""
    import numpy as np
    import oracle
    sub = dict(case_host)
    N = n_tokens
    off = case_host["offsets"][:N + 1].copy()
    sub["offsets"] = off
    for k in ("hidden", "labels", "label_logq", "adv", "loss_mask", "age", "replayed"):
        sub[k] = case_host[k][:N]
    sub["ids"] = case_host["ids"][:off[-1]]
    sub["logq"] = case_host["logq"][:off[-1]]
    op = oracle.HeadParams(loss_type=oracle.LOSS_IPO, eps=float(np.float32(0.3)), max_importance_ratio=10.0,
                           kl_coeff=float(np.float32(0.01)), kl_estimator=oracle.KL_EXACT,
                           kl_staleness=oracle.STALE_INV_SQRT)
    t0 = time.perf_counter()
    oracle.head_forward(sub, op, chunk=16)
    oracle.head_backward(sub, op, np.full(N, 1.0 / case_host["hidden"].shape[0]), chunk=16)
    dt = time.perf_counter() - t0
    return {"value": N / dt, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": f"first {N} tokens of the 64k-token batch (full H=2048, V=151936), fp64 "
                      f"forward + backward incl. dW; {dt:.1f} s"}


def _rotating_sets(torch, dev, arrays, min_bytes):
    """Copies of the input arrays, enough of them that one round over the copies moves
    more than min_bytes (so a pass never finds its inputs in L2 from the previous round)."""
    one = sum(a.nbytes for a in arrays if a is not None)
    n = max(2, -(-int(min_bytes) // max(one, 1)))
    return [[None if a is None else torch.from_numpy(a).to(dev) for a in arrays] for _ in range(n)]


def _time_back_to_back(torch, calls, passes):
    """Average device time per call over `passes` calls back to back between one pair of
    CUDA events: one round over the input sets is captured in a CUDA graph and the graph
    replayed, so the host's per-call cost (the Python binding takes longer than a call's
    device time) does not leave gaps between the launches."""
    g = torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    with torch.cuda.graph(g):
        for c in calls:
            c()
    g.replay()
    torch.cuda.synchronize()
    rounds = max(1, passes // len(calls))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(rounds):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    del g
    return e0.elapsed_time(e1) / (rounds * len(calls))


def _copy_floor(torch, dev, nbytes: int, n_sets: int, passes: int) -> float:
    """Average time per call (ms) of a plain streaming kernel that moves nbytes (half read,
    half written: dst = src * 1 in fp32, torch's vectorised elementwise kernel on the SMs,
    not the driver's memcpy, whose path changes with the size), timed as the pass it
    stands beside: back to back in a CUDA graph over n_sets rotating sources and as many
    destinations (a destination written again on the next pass would take its writes in
    L2).  At a few tens of MB a kernel's start and drain are a large part of its time, so
    this is the floor a pass of that size meets, next to the peak measured on GB-sized
    copies."""
    half = (nbytes // 2 + 15) // 16 * 4
    srcs = [torch.ones(half, dtype=torch.float32, device=dev) for _ in range(n_sets)]
    dsts = [torch.empty(half, dtype=torch.float32, device=dev) for _ in range(n_sets)]
    calls = [(lambda a=a, d=d: torch.mul(a, 1.0, out=d)) for a, d in zip(srcs, dsts)]
    for c in calls:
        c()
    torch.cuda.synchronize()
    ms = _time_back_to_back(torch, calls, passes)
    del srcs, dsts
    return ms


def elementwise_side(rh, torch, dev, steps: int, warmup: int, peaks: dict, flush_mb: int = 4096, packed: bool = True):
    """The elementwise PPO / dual-clip / decoupled-TIS / mismatch path on its own workload,
    1.8M valid tokens in sequences of 64..4096, against the HBM roofline.

    packed (the default and the roofline line): the valid tokens end to end, no mask; per
    token 16 B read (four fp32 inputs) and 16 B written (four fp32 outputs).  Otherwise the
    sequences padded to 4096 slots with a response mask: 17 B read and 16 B written per slot.

    Timing: `passes` calls back to back (a CUDA graph of one round over rotating copies of
    the inputs whose total is more than twice L2, so no pass finds its inputs in L2,
    replayed between one event pair); per call that is the kernel launch, the figure the
    roofline divides by.  The library's own per-launch event pairs (rl_profile) time single calls after an
    L2-flushing memset as well (kernel_us_single_launch), a figure that includes an event
    pair's own ~2 us."""
    import numpy as np
    import workloads
    c = workloads.make_policy_case()
    if packed:
        p = c.packed()
        arrays = [p["lp_theta"], p["lp_old"], p["lp_samp"], p["adv"], None]
    else:
        arrays = [c.lp_theta, c.lp_old, c.lp_samp, c.adv, c.mask]
    T = int(arrays[0].shape[0])
    pp = rh.PgParams()
    sets = _rotating_sets(torch, dev, arrays, 2 * 129 * 2 ** 20 + 1)
    # outputs rotate with the inputs: a pass never writes lines the previous passes left in L2
    out_sets = [tuple(torch.empty(T, dtype=torch.float32, device=dev) for _ in range(4)) for _ in sets]
    met = torch.zeros(rh.ctypes.sizeof(rh.RlPgMetrics), dtype=torch.uint8, device=dev)
    ws = torch.zeros(rh.rl_policy_workspace_bytes(T), dtype=torch.uint8, device=dev)   # zeroed once
    calls = [(lambda ins=ins, outs=outs: rh.rl_policy_loss_elementwise(*ins, pp, outputs=outs, ws=ws, metrics_dev=met))
             for ins, outs in zip(sets, out_sets)]
    for i in range(max(warmup, 3)):
        calls[i % len(calls)]()
    torch.cuda.synchronize()
    passes = max(steps, 10) * len(calls)
    ms = _time_back_to_back(torch, calls, passes)
    # single calls after an L2 flush, each timed by the library's event pairs
    big = torch.empty(flush_mb << 20, dtype=torch.uint8, device=dev)
    kern = []
    for i in range(max(steps, 10)):
        big.zero_()
        rh.rl_profile_enable(True)
        calls[i % len(calls)]()
        prof = rh.rl_profile_read()
        rh.rl_profile_enable(False)
        kern.append(sum(t for k, (t, _) in prof.items() if k == "policy"))
    del big
    kms = statistics.median(kern)
    n_valid = int(c.mask.sum())
    nbytes = T * (16 + (0 if packed else 1)) + T * 16
    gbs = nbytes / (ms / 1e3) / 1e9
    copy_ms = _copy_floor(torch, dev, nbytes, len(sets), passes)
    # the same pass on the inputs tiled eight times (14.4M tokens, 461 MB packed): a pass
    # long enough for the launch and drain to amortise, against a copy of its bytes
    big_arrays = [None if x is None else np.tile(x, 8) for x in arrays]
    Tb = int(big_arrays[0].shape[0])
    bsets = _rotating_sets(torch, dev, big_arrays, 2 * 129 * 2 ** 20 + 1)
    bout_sets = [tuple(torch.empty(Tb, dtype=torch.float32, device=dev) for _ in range(4)) for _ in bsets]
    bcalls = [(lambda ins=ins, outs=outs: rh.rl_policy_loss_elementwise(*ins, pp, outputs=outs, ws=ws, metrics_dev=met))
              for ins, outs in zip(bsets, bout_sets)]
    for c_ in bcalls:
        c_()
    torch.cuda.synchronize()
    bpasses = 10 * len(bcalls)
    bms = _time_back_to_back(torch, bcalls, bpasses)
    bbytes = 8 * nbytes
    bcopy_ms = _copy_floor(torch, dev, bbytes, len(bsets), bpasses)
    del bsets, bout_sets, bcalls
    torch.cuda.empty_cache()
    peak = float(peaks["hbm_gbs"])
    layout = (f"packed: {n_valid} valid tokens end to end, no mask" if packed else
              f"padded: {len(c.seq_lens)} sequences of 64..4096 padded to {c.max_len} (T={T} slots) with a mask")
    return {"workload": f"c5 {layout}; PPO clip 0.2/0.2 + dual clip 3, decoupled TIS, 10-point IPO curve, "
                        "IcePop band, mismatch KL",
            "us_per_call_back_to_back": ms * 1e3, "kernel_us_single_launch": kms * 1e3,
            "tokens_per_s": n_valid / (ms / 1e3), "passes": passes, "input_sets": len(sets),
            "device_copy_same_bytes": {"us_per_call_back_to_back": copy_ms * 1e3, "pass_over_copy": ms / copy_ms,
                                       "frac_of_hbm_peak": nbytes / (copy_ms / 1e3) / 1e9 / float(peaks["hbm_gbs"])},
            "tiled_x8": {"tokens": 8 * n_valid if packed else None, "slots": Tb, "bytes_per_pass": bbytes,
                         "us_per_call_back_to_back": bms * 1e3,
                         "frac_of_hbm_peak": bbytes / (bms / 1e3) / 1e9 / float(peaks["hbm_gbs"]),
                         "device_copy_same_bytes_us": bcopy_ms * 1e3,
                         "copy_frac_of_hbm_peak": bbytes / (bcopy_ms / 1e3) / 1e9 / float(peaks["hbm_gbs"])},
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak,
                         "traffic": None, "algorithmic_bytes_per_pass": nbytes,
                         "duration": "average per call, back to back in a CUDA graph (one kernel launch per call)",
                         "peak_kind": f"hbm_gbs ({peaks['source']})"},
            "l2": f"{len(sets)} rotating input sets of {sum(a.nbytes for a in arrays if a is not None) >> 20} MB "
                  "(more than 2x L2 per round), each with its own output buffers"}


def rollout_side(rh, torch, dev, steps: int, warmup: int, peaks: dict, flush_mb: int = 4096, packed: bool = True):
    """Rollout correction (IS / RS weights over sequences, veto, batch normalisation,
    mismatch metrics) on the elementwise workload: lp_old is the trainer's log-probs,
    lp_samp the rollout engine's; packed (the default): the 879 sequences end to end
    (cumulative lengths, every mask byte 1), else the padded rows.  Knobs: sequence-level
    TIS clipped to [0.1, 10] with batch normalisation, geometric RS in [0.9, 1.1], veto
    1e-4.  Timed as elementwise_side (per call: the sequence kernel, whose last block writes
    the metrics and the factor, then the scaling kernel).  Algorithmic bytes per slot: two
    fp32 inputs and the mask read, the fp32 weight and the keep byte written (14 B), plus
    the weight read and written again by the normalisation (8 B): the factor needs every
    token first.  Beside it: a device copy of the same bytes timed the same way, and the
    same call on the batch tiled eight times (7032 sequences, 14.4M tokens)."""
    import numpy as np
    import workloads
    c = workloads.make_policy_case()
    B = len(c.seq_lens)
    if packed:
        p = c.packed()
        arrays = [p["lp_old"], p["lp_samp"], np.ones(len(p["lp_old"]), np.uint8)]
        off_h = p["cu_seqlens"]
    else:
        arrays = [c.lp_old, c.lp_samp, c.mask]
        off_h = np.arange(B + 1, dtype=np.int64) * c.max_len
    off = torch.from_numpy(off_h).to(dev)
    T = int(arrays[0].shape[0])
    rp = rh.RcParams(tis_mode="clip", tis_level="sequence", tis_lower_bound=0.1, tis_upper_bound=10.0,
                     tis_batch_normalize=True, use_rs=True, rs_level="geometric", rs_lower_bound=0.9,
                     rs_upper_bound=1.1, rs_veto_threshold=1e-4)
    sets = _rotating_sets(torch, dev, arrays, 2 * 129 * 2 ** 20 + 1)
    out_sets = [(torch.empty(T, dtype=torch.float32, device=dev), torch.empty(T, dtype=torch.uint8, device=dev))
                for _ in sets]   # rotating with the inputs
    met = torch.zeros(rh.ctypes.sizeof(rh.RlRcMetrics), dtype=torch.uint8, device=dev)
    ws = torch.zeros(rh.rl_rollout_correction_workspace_bytes(B), dtype=torch.uint8, device=dev)   # zeroed once
    calls = [(lambda ins=ins, outs=outs: rh.rl_rollout_correction(*ins, off, rp, outputs=outs, ws=ws, metrics_dev=met))
             for ins, outs in zip(sets, out_sets)]
    for i in range(max(warmup, 3)):
        calls[i % len(calls)]()
    torch.cuda.synchronize()
    passes = max(steps, 10) * len(calls)
    ms = _time_back_to_back(torch, calls, passes)
    big = torch.empty(flush_mb << 20, dtype=torch.uint8, device=dev)
    kern = []
    for i in range(max(steps, 10)):
        big.zero_()
        rh.rl_profile_enable(True)
        calls[i % len(calls)]()
        prof = rh.rl_profile_read()
        rh.rl_profile_enable(False)
        kern.append(sum(t for k, (t, _) in prof.items() if k == "rollout"))
    del big
    kms = statistics.median(kern)
    nbytes = T * (4 + 4 + 1) + T * (4 + 1) + T * 8
    gbs = nbytes / (ms / 1e3) / 1e9
    peak = float(peaks["hbm_gbs"])
    n_valid = int(c.mask.sum())
    copy_ms = _copy_floor(torch, dev, nbytes, len(sets), passes)
    # the same call on the batch tiled eight times (8 x 879 sequences, 14.4M tokens): more
    # sequences than resident blocks, so the block scheduler balances the SMs as it goes
    big_arrays = [np.tile(x, 8) for x in arrays]
    Tb = int(big_arrays[0].shape[0])
    off_b = np.concatenate([off_h[:-1] + k * T for k in range(8)] + [np.array([8 * T], np.int64)]).astype(np.int64)
    offb = torch.from_numpy(off_b).to(dev)
    bsets = _rotating_sets(torch, dev, big_arrays, 2 * 129 * 2 ** 20 + 1)
    bout_sets = [(torch.empty(Tb, dtype=torch.float32, device=dev), torch.empty(Tb, dtype=torch.uint8, device=dev))
                 for _ in bsets]
    bws = torch.zeros(rh.rl_rollout_correction_workspace_bytes(8 * B), dtype=torch.uint8, device=dev)
    bcalls = [(lambda ins=ins, outs=outs: rh.rl_rollout_correction(*ins, offb, rp, outputs=outs, ws=bws, metrics_dev=met))
              for ins, outs in zip(bsets, bout_sets)]
    for c_ in bcalls:
        c_()
    torch.cuda.synchronize()
    bpasses = 10 * len(bcalls)
    bms = _time_back_to_back(torch, bcalls, bpasses)
    bbytes = 8 * nbytes
    bcopy_ms = _copy_floor(torch, dev, bbytes, len(bsets), bpasses)
    del bsets, bout_sets, bcalls, bws
    torch.cuda.empty_cache()
    layout = (f"{B} sequences packed end to end (T={T} tokens, mask all 1)" if packed else
              f"{B} padded rows of {c.max_len} (T={T} slots, {n_valid} response tokens)")
    return {"workload": f"c5 as {layout}; sequence-level TIS clip [0.1, 10] + batch normalisation, geometric RS "
                        "[0.9, 1.1], veto 1e-4, mismatch metrics",
            "us_per_call_back_to_back": ms * 1e3, "kernel_us_single_launch": kms * 1e3,
            "tokens_per_s": n_valid / (ms / 1e3), "passes": passes, "input_sets": len(sets),
            "device_copy_same_bytes": {"us_per_call_back_to_back": copy_ms * 1e3, "call_over_copy": ms / copy_ms,
                                       "frac_of_hbm_peak": nbytes / (copy_ms / 1e3) / 1e9 / peak},
            "tiled_x8": {"sequences": 8 * B, "tokens": Tb, "bytes_per_call": bbytes, "us_per_call_back_to_back": bms * 1e3,
                         "frac_of_hbm_peak": bbytes / (bms / 1e3) / 1e9 / peak,
                         "device_copy_same_bytes_us": bcopy_ms * 1e3,
                         "copy_frac_of_hbm_peak": bbytes / (bcopy_ms / 1e3) / 1e9 / peak},
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak,
                         "traffic": None, "algorithmic_bytes_per_pass": nbytes,
                         "duration": "average per call, back to back in a CUDA graph (the sequence kernel, then the scaling kernel)",
                         "peak_kind": f"hbm_gbs ({peaks['source']})"},
            "l2": f"{len(sets)} rotating input sets (more than 2x L2 per round), each with its own output buffers"}


def time_head_config(rh, torch, dev, case, hp, steps: int, warmup: int, peaks: dict, what: str) -> dict:
    """One side configuration of the head path: the fused forward + backward step timed as
    the headline (CUDA events around each step, a 256 MB memset between steps), with the
    memory it holds beyond its inputs (workspace, saved state, outputs, gradients) and its
    roofline: 6 N H V flop at the burst bf16 peak for a dense backward; for the sparse
    backward the forward's 2 N H V flop at that peak plus, at the HBM peak, the bytes the
    step must move (W and X read once, the W rows and X rows each label / support entry
    gathers, dX and the overwritten dW written)."""
    N, H, V, nnz = case.N, case.H, case.V, case.nnz
    batch = rh.HeadBatch.from_case(case)
    dloss = (case.loss_mask.float() / case.loss_mask.float().sum()).contiguous()
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    torch.cuda.reset_peak_memory_stats(dev)
    base = torch.cuda.memory_allocated(dev)
    ws = torch.empty(rh.rl_head_fwd_bwd_workspace_bytes(N, H, V, nnz, hp), dtype=torch.uint8, device=dev)
    saved = torch.empty(rh.rl_head_saved_bytes(N, nnz), dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    dX = torch.empty(N, H, dtype=torch.bfloat16, device=dev)
    dW = torch.empty(V, H, dtype=torch.float32, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    step = lambda: rh.rl_head_loss_fwd_bwd(batch, hp, dloss, dhidden=dX, dW=dW, ws=ws, saved=saved, status=status)[0]
    for _ in range(max(warmup, 2)):
        f = step()
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError(f"{what}: device status {rh.status_names(int(status.item()))}")
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    rh.rl_profile_enable(True)
    for a, b in ev:
        flush.zero_()
        a.record()
        f = step()
        b.record()
    torch.cuda.synchronize()
    prof = rh.rl_profile_read()
    rh.rl_profile_enable(False)
    ms = statistics.median(a.elapsed_time(b) for a, b in ev)
    held = (torch.cuda.max_memory_allocated(dev) - base - flush.numel()) / 2 ** 30
    m = f.metrics()
    burst = float(peaks["bf16_tflops"])
    hbm = float(peaks["hbm_gbs"])
    out = {"workload": what, "N": N, "nnz": nnz, "ms_per_step": ms, "tokens_per_s": N / (ms / 1e3),
           "token_chunk": rh.rl_head_token_chunk(N, case.H, hp),
           "grad_precision": "split" if hp.grad_precision == rh.RL_GRAD_SPLIT else "bf16",
           "held_gib": held, "recomputed_chunks": int(m["recomputed_chunks"]),
           "kernels_ms_per_step": {k: t / steps for k, (t, n) in sorted(prof.items(), key=lambda kv: -kv[1][0])}}
    sparse = hp.bwd_mode == rh.RL_BWD_SPARSE or (hp.bwd_mode == rh.RL_BWD_AUTO and hp.all_replayed)
    if sparse:
        flop = 2.0 * N * H * V
        nbytes = V * H * 2 + N * H * 2 + 2 * (nnz + N) * H * 2 + V * H * 4 + N * H * 2
        t_roof = flop / (burst * 1e12) + nbytes / (hbm * 1e9)
        out["roofline"] = {"bound": "tensor+hbm", "algorithmic_flops": flop, "algorithmic_bytes": nbytes,
                           "roofline_ms": t_roof * 1e3, "frac": t_roof * 1e3 / ms,
                           "peak": f"bf16_tflops {burst} + hbm_gbs {hbm} ({peaks['source']})"}
        for k, kb in (("sparse_dx", (nnz + N) * H * 2 + N * H * 2), ("sparse_dw", (nnz + N) * H * 2 + V * H * 4)):
            if k in prof:
                t, n = prof[k]
                out.setdefault("hbm_kernels", {})[k] = {"ms_per_step": t / steps, "algorithmic_bytes": kb,
                                                       "gbs": kb / (t / steps / 1e3) / 1e9,
                                                       "frac": kb / (t / steps / 1e3) / 1e9 / hbm}
    else:
        tf = 6.0 * N * H * V / (ms / 1e3) / 1e12
        out["roofline"] = {"bound": "tensor", "step_tflops_6NHV": tf, "peak": burst, "frac": tf / burst,
                           "peak_kind": f"bf16_tflops ({peaks['source']})"}
        if hp.grad_precision == rh.RL_GRAD_SPLIT:
            out["roofline"]["tensor_work_tflops_10NHV"] = 10.0 * N * H * V / (ms / 1e3) / 1e12
    del ws, saved, dX, dW, flush
    torch.cuda.empty_cache()
    return out


def side_configs(rh, torch, dev, case4, steps: int, warmup: int, peaks: dict) -> dict:
    """The other configurations of the head path, each timed as the headline: c4 with the
    hi/lo (SPLIT) gradient operand, c4 at token chunks 4096 / 8192 / 16384 / 32768 (time
    against memory), c2 (4096 tokens, replayed top-p 0.97, icepop, dense), c3 (16384 tokens,
    replayed top-p 0.97, ipo) with the sparse CSR backward and with the dense one."""
    import dataclasses
    import workloads
    steps = max(3, min(steps, 8))
    base = head_params(rh, "bf16")
    out = {"c4_split": time_head_config(rh, torch, dev, case4, dataclasses.replace(base, grad_precision=rh.RL_GRAD_SPLIT),
                                        steps, warmup, peaks, "c4, grad_precision SPLIT (bf16 hi + lo operand)")}
    out["c4_chunks"] = [time_head_config(rh, torch, dev, case4, dataclasses.replace(base, token_chunk=c), steps, warmup,
                                         peaks, f"c4, token_chunk {c}") for c in (4096, 8192, 9728, 16384, 32768)]
    c2 = workloads.make_head_case("c2", device=dev, variant="pages")
    hp2 = rh.HeadParams(loss_type=rh.RL_LOSS_ICEPOP, icepop_low=0.5, icepop_high=2.0, bwd_mode=rh.RL_BWD_DENSE)
    out["c2"] = time_head_config(rh, torch, dev, c2, hp2, steps, warmup, peaks,
                                 "c2: N=4096 (16 x 256), replayed top-p 0.97 (pages-shaped kept counts), icepop "
                                 "[0.5, 2], dense backward")
    del c2
    c3 = workloads.make_head_case("c3", device=dev, variant="pages")
    hp3 = rh.HeadParams(loss_type=rh.RL_LOSS_IPO, eps=0.3, max_importance_ratio=10.0, all_replayed=1)
    what3 = "c3: N=16384 (64 x 256), replayed top-p 0.97 (pages-shaped kept counts), ipo 0.3 cap 10"
    out["c3_sparse"] = time_head_config(rh, torch, dev, c3, hp3, steps, warmup, peaks, what3 + ", sparse CSR backward")
    out["c3_dense"] = time_head_config(rh, torch, dev, c3, dataclasses.replace(hp3, all_replayed=0,
                                                                                bwd_mode=rh.RL_BWD_DENSE),
                                       steps, warmup, peaks, what3 + ", dense backward")
    del c3
    torch.cuda.empty_cache()
    return out


def host_inputs(case):
    """The batch as numpy (fp64 copies of bf16 values) for the oracle."""
    return case.numpy()


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import numpy as np
    import torch
    import workloads
    threads = os.cpu_count() or 1
    torch.set_num_threads(threads)
    # the same seeded batch as the GPU arm, generated on the host (first tokens only)
    n_sample = args.ref_tokens
    case = workloads.make_head_case("c4", n_tokens=max(n_sample, 128), device="cpu")
    host = host_inputs(case)
    import oracle  # noqa: F401  (the reference arm is the oracle)
    per = []
    for i in range(args.warmup + args.steps):
        r = cpu_baseline(host, n_sample, threads)
        if i >= args.warmup:
            per.append(n_sample / r["value"])
    ms = 1e3 * statistics.mean(per)
    val = n_sample / (ms / 1e3)
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "sample_tokens": n_sample},
            "cpu_baseline": {"value": val, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                             "sample": f"first {n_sample} tokens of the 64k-token batch per step"},
            "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_elementwise_only(args):
    """The elementwise paths alone (profiling runs): one JSON line with their side figures."""
    import torch

    import lm_head_gb300 as rh
    from lm_head_gb300 import build

    dev = torch.device("cuda", torch.cuda.current_device())
    build.build()
    rh.load()
    ew = elementwise_side(rh, torch, dev, args.steps, args.warmup, load_peaks(), args.flush_mb)
    ewp = elementwise_side(rh, torch, dev, args.steps, args.warmup, load_peaks(), args.flush_mb, packed=False)
    rc = rollout_side(rh, torch, dev, args.steps, args.warmup, load_peaks(), args.flush_mb)
    print(json.dumps({"elementwise": ew, "elementwise_padded": ewp, "rollout_correction": rc,
                      "gpu_launches_total": int(rh.rl_kernel_launch_count())}), flush=True)
    return 0


def run_ours(args):
    import numpy as np
    import torch
    import torch.distributed as dist

    import lm_head_gb300 as rh
    import workloads
    from lm_head_gb300 import build

    rank, world, local = dist_env()
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", torch.cuda.current_device())
    build.build()
    rh.load()
    if args.gemm_pair is not None:
        rh.rl_set_option(rh.RL_OPT_GEMM_PAIR, args.gemm_pair)
    peaks = load_peaks()

    t_gen = time.perf_counter()
    # the replayed top-p configurations with the pages' kept counts, as in the side figures
    case = workloads.make_head_case(args.config, device=dev, seed=workloads.BASE_SEED + 4 + 1000 * rank,
                                    n_tokens=args.tokens,
                                    variant="pages" if args.config in ("c2", "c3") else "literal")
    torch.cuda.synchronize()
    t_gen = time.perf_counter() - t_gen
    N, H, V, nnz = case.N, case.H, case.V, case.nnz
    hp = head_params(rh, args.grad_precision)
    if args.sparse:
        hp = rh.HeadParams(loss_type=rh.RL_LOSS_IPO, eps=0.3, max_importance_ratio=10.0, all_replayed=1)
    batch = rh.HeadBatch.from_case(case)
    torch.cuda.reset_peak_memory_stats(dev)
    base_mem = torch.cuda.memory_allocated(dev)
    ws_fb = torch.empty(rh.rl_head_fwd_bwd_workspace_bytes(N, H, V, nnz, hp), dtype=torch.uint8, device=dev)
    saved = torch.empty(rh.rl_head_saved_bytes(N, nnz), dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    dloss = (case.loss_mask.float() / case.loss_mask.float().sum()).contiguous()   # token mean
    dX = torch.empty(N, H, dtype=torch.bfloat16, device=dev)
    dW = torch.empty(V, H, dtype=torch.float32, device=dev)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)     # > 2x L2

    def step(b=batch, st=status):
        # one forward + backward of the head over the batch: the fused entry point (the
        # token-mean weights are known before the forward)
        f, _, _ = rh.rl_head_loss_fwd_bwd(b, hp, dloss, dhidden=dX, dW=dW, ws=ws_fb, saved=saved, status=st)
        return f

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {rh.status_names(int(status.item()))}")

    # ---- timed region: device-resident inputs ----
    rh.rl_profile_enable(True)
    n0 = rh.rl_kernel_launch_count()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(dev.index if dev.index is not None else 0) as clk:
        for i in range(args.steps):
            flush.zero_()                      # L2 flush between steps (outside the events)
            starts[i].record()
            f = step()
            ends[i].record()
        torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    launches = rh.rl_kernel_launch_count() - n0
    prof = rh.rl_profile_read()
    rh.rl_profile_enable(False)
    local_ms = sum(s.elapsed_time(e) for s, e in zip(starts, ends)) / args.steps
    ms, tokens, value = aggregate(local_ms, N, world)
    clocks = clk.summary()
    peak_gib = (torch.cuda.max_memory_allocated(dev)) / 2 ** 30
    work_gib = (torch.cuda.max_memory_allocated(dev) - base_mem) / 2 ** 30

    # ---- side figure: the two-call path (forward, then backward with logit recompute) ----
    unfused_ms = kept_ms = kept_gib = None
    if not args.no_unfused:
        del ws_fb
        torch.cuda.empty_cache()
        ws_f = torch.empty(rh.rl_head_fwd_workspace_bytes(N, H, V, nnz, hp), dtype=torch.uint8, device=dev)
        ws_b = torch.empty(rh.rl_head_bwd_workspace_bytes(N, H, V, nnz, hp), dtype=torch.uint8, device=dev)
        for i in range(2 + min(args.steps, 3)):
            if i == 2:
                torch.cuda.synchronize()
                e0 = torch.cuda.Event(enable_timing=True)
                e0.record()
            rh.rl_head_loss_fwd(batch, hp, ws=ws_f, saved=saved, status=status)
            rh.rl_head_loss_bwd(batch, hp, saved, dloss, dhidden=dX, dW=dW, ws=ws_b, status=status)
        e1 = torch.cuda.Event(enable_timing=True)
        e1.record()
        torch.cuda.synchronize()
        unfused_ms = e0.elapsed_time(e1) / min(args.steps, 3)
        del ws_f, ws_b
        torch.cuda.empty_cache()
        # the same two calls with the numerators kept by the forward (keep_e: 2 N V bf16 in
        # the saved state, no logit recompute in the backward)
        import dataclasses
        hk = dataclasses.replace(hp, keep_e=1)
        saved_k = torch.empty(rh.rl_head_saved_bytes_ex(N, nnz, V, hk), dtype=torch.uint8, device=dev)
        ws_f = torch.empty(rh.rl_head_fwd_workspace_bytes(N, H, V, nnz, hk), dtype=torch.uint8, device=dev)
        ws_b = torch.empty(rh.rl_head_bwd_workspace_bytes(N, H, V, nnz, hk), dtype=torch.uint8, device=dev)
        for i in range(2 + min(args.steps, 3)):
            if i == 2:
                torch.cuda.synchronize()
                e0 = torch.cuda.Event(enable_timing=True)
                e0.record()
            rh.rl_head_loss_fwd(batch, hk, ws=ws_f, saved=saved_k, status=status)
            rh.rl_head_loss_bwd(batch, hk, saved_k, dloss, dhidden=dX, dW=dW, ws=ws_b, status=status)
        e1 = torch.cuda.Event(enable_timing=True)
        e1.record()
        torch.cuda.synchronize()
        kept_ms = e0.elapsed_time(e1) / min(args.steps, 3)
        kept_gib = (saved_k.numel() + ws_f.numel() + ws_b.numel()) / 2 ** 30
        if int(status.item()) != 0:
            raise RuntimeError(f"device status {rh.status_names(int(status.item()))}")
        del ws_f, ws_b, saved_k
        torch.cuda.empty_cache()
        ws_fb = torch.empty(rh.rl_head_fwd_bwd_workspace_bytes(N, H, V, nnz, hp), dtype=torch.uint8, device=dev)

    # ---- e2e: same step through the public API from pinned host buffers ----
    pin = {k: getattr(case, k).cpu().pin_memory() for k in
           ("hidden", "labels", "label_logq", "adv", "loss_mask", "age", "replayed", "offsets", "ids", "logq")}
    dbuf = {k: torch.empty_like(getattr(case, k)) for k in pin}
    e_batch = rh.HeadBatch(dbuf["hidden"], case.W, dbuf["labels"], dbuf["label_logq"], dbuf["adv"],
                           dbuf["offsets"], dbuf["ids"], dbuf["logq"], dbuf["replayed"], dbuf["loss_mask"],
                           dbuf["age"])
    h2d = sum(t.numel() * t.element_size() for t in pin.values())
    out_host = torch.empty(N, dtype=torch.float32).pin_memory()
    met_host = torch.empty(ctypes_metrics_size(rh), dtype=torch.uint8).pin_memory()
    d2h = out_host.numel() * 4 + met_host.numel()
    e_steps = max(1, min(args.steps, 5))
    for _ in range(2):
        for k in pin:
            dbuf[k].copy_(pin[k], non_blocking=True)
        f = step(e_batch)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    t0 = time.perf_counter()
    for _ in range(e_steps):
        for k in pin:
            dbuf[k].copy_(pin[k], non_blocking=True)
        f = step(e_batch)
        out_host.copy_(f.loss, non_blocking=True)
        met_host.copy_(f.metrics_dev, non_blocking=True)
        torch.cuda.synchronize()
    e_ms = (time.perf_counter() - t0) * 1e3 / e_steps
    e_ms, _, e_value = aggregate(e_ms, N, world)

    # ---- roofline of the dominant kernel (live CUDA-event times from the timed region) ----
    # per step the forward GEMM does 2 N H V flop, dX and dW 2 N H V each (twice that with the
    # hi/lo operand), spread over one launch per token chunk
    per_step = {"gemm_fwd_stats": 2.0 * N * H * V}
    for k in ("gemm_bwd_dx", "gemm_bwd_dw"):
        per_step[k] = 2.0 * N * H * V * (2 if args.grad_precision == "split" else 1)
    flops_per_launch = {k: v / (prof[k][1] / args.steps) for k, v in per_step.items() if k in prof}
    # the logit-recompute GEMM is gated on the device: it does its 2 chunk H V flop only for
    # the chunks whose range flag was raised (the metrics' recomputed_chunks), else exits
    recomputed = int(f.metrics()["recomputed_chunks"])
    if recomputed and "gemm_bwd_grad" in prof:
        n_chunks = prof["gemm_fwd_stats"][1] / args.steps
        flops_per_launch["gemm_bwd_grad"] = 2.0 * N * H * V / n_chunks * recomputed / (prof["gemm_bwd_grad"][1] / args.steps)
    # the captured per-launch traffic holds for the dense path at the default 8192-token chunk
    chunk = rh.rl_head_token_chunk(N, H, hp)
    traffic_ok = (not args.sparse and chunk == TRAFFIC_CHUNK and N >= chunk and args.grad_precision == "bf16")
    dom = max(prof.items(), key=lambda kv: kv[1][0])
    dom_name, (dom_ms, dom_n) = dom
    peak_sus = float(peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"]))
    peak_burst = float(peaks["bf16_tflops"])
    roof = None
    if dom_name in flops_per_launch:
        ach = flops_per_launch[dom_name] / ((dom_ms / dom_n) / 1e3) / 1e12
        roof = {"kernel": dom_name, "bound": "tensor", "achieved": ach, "peak": peak_sus, "unit": "TFLOP/s",
                "frac": ach / peak_sus, "traffic": TRAFFIC.get(dom_name) if traffic_ok else None,
                "traffic_source": TRAFFIC_SOURCE if traffic_ok and dom_name in TRAFFIC else None,
                "peak_kind": f"bf16_tflops_sustained ({peaks['source']})",
                "frac_of_burst": ach / peak_burst,
                "algorithmic_flops_per_launch": flops_per_launch[dom_name]}
    kernels = {}
    for k, (t, n) in sorted(prof.items(), key=lambda kv: -kv[1][0]):
        d = {"ms_per_step": t / args.steps, "launches_per_step": n / args.steps, "share": t / sum(v[0] for v in prof.values())}
        if k in flops_per_launch:
            d["tflops"] = flops_per_launch[k] / ((t / n) / 1e3) / 1e12
        kernels[k] = d
    step_tflops = 6.0 * N * H * V / (ms / 1e3) / 1e12

    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": WORKLOAD if args.config == "c4" and not args.sparse else
                       f"{args.config} shapes ({'sparse CSR backward, ipo 0.3 cap 10' if args.sparse else 'the c4 loss'}; "
                       "a profiling run)", "N": N, "H": H, "V": V, "nnz": nnz,
                       "grad_precision": args.grad_precision, "parallelism": f"replicas x{world}",
                       "gemm": "sm-pair (cta_group::2, 256x256)" if rh.rl_get_option(rh.RL_OPT_GEMM_PAIR) else
                               "single-sm (128x256)",
                       "l2": "inputs larger than L2 (W 622 MB); 256 MB flush between timed steps"},
            "tc_peak_frac": step_tflops / peak_burst,
            "step_tflops_6NHV": step_tflops,
            "peak_gib": peak_gib, "workspace_peak_gib": work_gib,
            "two_call_ms_per_step": unfused_ms,
            "two_call_keep_e": None if kept_ms is None else
                {"ms_per_step": kept_ms, "held_gib": kept_gib,
                 "note": "rl_head_loss_fwd then rl_head_loss_bwd with keep_e=1: the forward keeps e / e^T of every token"},
            "roofline": roof, "kernels": kernels,
            "e2e": {"value": e_value, "unit": "tokens/s", "ms_per_step": e_ms, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h},
            "clocks": clocks, "gpu_launches": int(launches), "input_gen_s": t_gen,
            "recomputed_chunks_per_step": recomputed}
    if not args.no_side_configs:
        del ws_fb
        torch.cuda.empty_cache()
        line["configs"] = side_configs(rh, torch, dev, case, args.steps, args.warmup, peaks)
    if not args.no_elementwise:
        line["elementwise"] = elementwise_side(rh, torch, dev, max(args.steps, 10), args.warmup, peaks)
        line["elementwise_padded"] = elementwise_side(rh, torch, dev, max(args.steps, 10), args.warmup, peaks,
                                                      packed=False)
        line["rollout_correction"] = rollout_side(rh, torch, dev, max(args.steps, 10), args.warmup, peaks)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        host = host_inputs(case_first(case, args.cpu_tokens))
        line["cpu_baseline"] = cpu_baseline(host, args.cpu_tokens, os.cpu_count() or 1)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


# dram__bytes_read.sum + dram__bytes_write.sum per launch of each kernel, from the ncu
# capture of the kernel as it stands (one launch at the library's default chunk on this
# part, 9728 tokens), summarised in profiles/gemm_pair_dram_traffic_9728_chunk.md.
TRAFFIC_CHUNK = 9728
TRAFFIC = {"gemm_fwd_stats": 1061985536 + 5871818752,
           "gemm_bwd_dx": 11018044928 + 34386176,
           "gemm_bwd_dw": 7238419712 + 1228881152}
TRAFFIC_SOURCE = "ncu capture at the 9728-token chunk, profiles/gemm_pair_dram_traffic_9728_chunk.md (not measured in this run)"


def ctypes_metrics_size(rh):
    import ctypes
    return ctypes.sizeof(rh.RlHeadMetrics)


def case_first(case, n):
    """The first n tokens of a HeadCase (host copy) for the CPU baseline."""
    import dataclasses
    import torch
    off = case.offsets[:n + 1].cpu()
    nnz = int(off[-1])
    kw = {f.name: getattr(case, f.name) for f in dataclasses.fields(case)}
    for k in ("hidden", "labels", "label_logq", "adv", "loss_mask", "age", "replayed"):
        kw[k] = getattr(case, k)[:n].cpu()
    kw["offsets"] = off
    kw["ids"] = case.ids[:nnz].cpu()
    kw["logq"] = case.logq[:nnz].cpu()
    kw["W"] = case.W.cpu()
    return type(case)(**kw)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="c4")
    ap.add_argument("--grad-precision", choices=["bf16", "split"], default="bf16")
    ap.add_argument("--sparse", action="store_true",
                    help="the sparse-backward configuration's loss (ipo 0.3, cap 10, replayed supports) with the "
                         "sparse CSR backward; for --config c3 (profiling runs)")
    ap.add_argument("--cpu-tokens", type=int, default=128, help="oracle sample for cpu_baseline")
    ap.add_argument("--ref-tokens", type=int, default=32, help="oracle sample per step, --impl reference")
    ap.add_argument("--tokens", type=int, default=None, help="fewer tokens, same shapes (profiling runs)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-unfused", action="store_true", help="skip the two-call side figure")
    ap.add_argument("--no-elementwise", action="store_true", help="skip the elementwise-path side figure")
    ap.add_argument("--no-side-configs", action="store_true",
                    help="skip the c2 / c3 / c4-SPLIT / token-chunk side configurations")
    ap.add_argument("--elementwise-only", action="store_true",
                    help="time only the elementwise path (profiling runs); prints its side figure")
    ap.add_argument("--flush-mb", type=int, default=4096, help="memset before each elementwise pass, MB")
    ap.add_argument("--gemm-pair", type=int, choices=[0, 1], default=None,
                    help="tensor-core GEMMs on SM pairs (1) or single SMs (0); default: library default")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    if args.elementwise_only:
        return run_elementwise_only(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
