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


def elementwise_side(rh, torch, dev, steps: int, warmup: int, peaks: dict, flush_mb: int = 4096):
    """The elementwise PPO / dual-clip / decoupled-TIS / mismatch path on its own workload
    (1.8M valid tokens in sequences of 64..4096, padded to 4096), against the HBM roofline.
    Each pass follows a memset of flush_mb MB (default 4 GB: an L2 flush that keeps the GPU
    busy for about half a millisecond, long enough for the host to queue the pass before
    the GPU reaches it; profiling runs pass a smaller one).  The library's own event pairs
    (rl_profile) time the call in two parts, the 256-byte workspace memset and the kernel
    launch: their sum is the pass (us_per_pass, tokens_per_s), the launch alone
    (kernel_us_per_pass) is what the roofline divides by.
    Algorithmic bytes per slot: four fp32 inputs and the mask byte read, four fp32
    outputs written (33 B)."""
    import workloads
    c = workloads.make_policy_case()
    ins = [torch.from_numpy(x).to(dev) for x in (c.lp_theta, c.lp_old, c.lp_samp, c.adv, c.mask)]
    T = int(ins[0].numel())
    pp = rh.PgParams()
    outs = tuple(torch.empty(T, dtype=torch.float32, device=dev) for _ in range(4))
    met = torch.zeros(rh.ctypes.sizeof(rh.RlPgMetrics), dtype=torch.uint8, device=dev)
    ws = torch.empty(rh.rl_policy_workspace_bytes(T), dtype=torch.uint8, device=dev)
    run = lambda: rh.rl_policy_loss_elementwise(*ins, pp, outputs=outs, ws=ws, metrics_dev=met)
    big = torch.empty(flush_mb << 20, dtype=torch.uint8, device=dev)
    for _ in range(warmup):
        run()
    torch.cuda.synchronize()
    per, kern = [], []
    for _ in range(steps):
        big.zero_()
        rh.rl_profile_enable(True)
        run()
        prof = rh.rl_profile_read()
        rh.rl_profile_enable(False)
        per.append(sum(t for t, _ in prof.values()))
        kern.append(sum(t for k, (t, _) in prof.items() if k == "policy"))
    del big
    ms = statistics.median(per)        # the whole call: workspace memset + kernel launches
    kms = statistics.median(kern)      # the kernel launches alone (the roofline's duration)
    nbytes = T * (4 * 4 + 1) + T * 4 * 4
    gbs = nbytes / (kms / 1e3) / 1e9
    peak = float(peaks["hbm_gbs"])
    n_valid = int(c.mask.sum())
    return {"workload": f"c5: {n_valid} valid tokens, {len(c.seq_lens)} sequences of 64..4096 padded to "
                        f"{c.max_len} (T={T} slots); PPO clip 0.2/0.2 + dual clip 3, decoupled TIS, "
                        "10-point IPO curve, IcePop band, mismatch KL",
            "us_per_pass": ms * 1e3, "kernel_us_per_pass": kms * 1e3, "tokens_per_s": n_valid / (ms / 1e3),
            "passes": steps,
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak,
                         "traffic": None, "algorithmic_bytes_per_pass": nbytes,
                         "peak_kind": f"hbm_gbs ({peaks['source']})"},
            "l2": f"{flush_mb} MB memset before each pass (outside the events)"}


def rollout_side(rh, torch, dev, steps: int, warmup: int, peaks: dict, flush_mb: int = 4096):
    """Rollout correction (IS / RS weights over sequences, veto, batch normalisation,
    mismatch metrics) on the elementwise workload: the 879 padded rows are the sequences,
    lp_old the trainer's log-probs, lp_samp the rollout engine's.  Knobs: sequence-level
    TIS clipped to [0.1, 10] with batch normalisation, geometric RS in [0.9, 1.1], veto
    1e-4.  Timed as elementwise_side.  Algorithmic bytes per slot: two fp32 inputs and the
    mask read, the fp32 weight and the keep byte written (14 B), plus the weight read and
    written again by the normalisation (8 B): the factor needs every token first."""
    import numpy as np
    import workloads
    c = workloads.make_policy_case()
    B = len(c.seq_lens)
    off = torch.arange(B + 1, dtype=torch.int64, device=dev) * c.max_len
    ins = [torch.from_numpy(x).to(dev) for x in (c.lp_old, c.lp_samp, c.mask)]
    T = int(ins[0].numel())
    rp = rh.RcParams(tis_mode="clip", tis_level="sequence", tis_lower_bound=0.1, tis_upper_bound=10.0,
                     tis_batch_normalize=True, use_rs=True, rs_level="geometric", rs_lower_bound=0.9,
                     rs_upper_bound=1.1, rs_veto_threshold=1e-4)
    outs = (torch.empty(T, dtype=torch.float32, device=dev), torch.empty(T, dtype=torch.uint8, device=dev))
    met = torch.zeros(rh.ctypes.sizeof(rh.RlRcMetrics), dtype=torch.uint8, device=dev)
    ws = torch.empty(rh.rl_rollout_correction_workspace_bytes(B), dtype=torch.uint8, device=dev)
    run = lambda: rh.rl_rollout_correction(*ins, off, rp, outputs=outs, ws=ws, metrics_dev=met)
    big = torch.empty(flush_mb << 20, dtype=torch.uint8, device=dev)
    for _ in range(warmup):
        run()
    torch.cuda.synchronize()
    per, kern = [], []
    for _ in range(steps):
        big.zero_()
        rh.rl_profile_enable(True)
        run()
        prof = rh.rl_profile_read()
        rh.rl_profile_enable(False)
        per.append(sum(t for t, _ in prof.values()))
        kern.append(sum(t for k, (t, _) in prof.items() if k == "rollout"))
    del big
    ms = statistics.median(per)        # the whole call: workspace memset + kernel launches
    kms = statistics.median(kern)      # the kernel launches alone (the roofline's duration)
    nbytes = T * (4 + 4 + 1) + T * (4 + 1) + T * 8
    gbs = nbytes / (kms / 1e3) / 1e9
    peak = float(peaks["hbm_gbs"])
    n_valid = int(c.mask.sum())
    return {"workload": f"c5 as {B} sequences (padded rows of {c.max_len}, T={T} slots, {n_valid} response "
                        "tokens); sequence-level TIS clip [0.1, 10] + batch normalisation, geometric RS "
                        "[0.9, 1.1], veto 1e-4, mismatch metrics",
            "us_per_pass": ms * 1e3, "kernel_us_per_pass": kms * 1e3, "tokens_per_s": n_valid / (ms / 1e3),
            "passes": steps,
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak,
                         "traffic": None, "algorithmic_bytes_per_pass": nbytes,
                         "peak_kind": f"hbm_gbs ({peaks['source']})"},
            "l2": f"{flush_mb} MB memset before each pass (outside the events)"}


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
    rc = rollout_side(rh, torch, dev, args.steps, args.warmup, load_peaks(), args.flush_mb)
    print(json.dumps({"elementwise": ew, "rollout_correction": rc,
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
    case = workloads.make_head_case(args.config, device=dev, seed=workloads.BASE_SEED + 4 + 1000 * rank,
                                    n_tokens=args.tokens)
    torch.cuda.synchronize()
    t_gen = time.perf_counter() - t_gen
    N, H, V, nnz = case.N, case.H, case.V, case.nnz
    hp = head_params(rh, args.grad_precision)
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
    unfused_ms = None
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
    chunk = min(16384, (N + 127) // 128 * 128)
    flops_per_launch = {"gemm_fwd_stats": 2.0 * chunk * H * V}     # fused path: one launch per chunk
    for k in ("gemm_bwd_grad", "gemm_bwd_dx", "gemm_bwd_dw"):
        flops_per_launch[k] = 2.0 * chunk * H * V * (2 if (args.grad_precision == "split" and k != "gemm_bwd_grad") else 1)
    dom = max(prof.items(), key=lambda kv: kv[1][0])
    dom_name, (dom_ms, dom_n) = dom
    peak_sus = float(peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"]))
    peak_burst = float(peaks["bf16_tflops"])
    roof = None
    if dom_name in flops_per_launch:
        ach = flops_per_launch[dom_name] / ((dom_ms / dom_n) / 1e3) / 1e12
        roof = {"kernel": dom_name, "bound": "tensor", "achieved": ach, "peak": peak_sus, "unit": "TFLOP/s",
                "frac": ach / peak_sus, "traffic": TRAFFIC.get(dom_name),
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
            "config": {"workload": WORKLOAD, "N": N, "H": H, "V": V, "nnz": nnz,
                       "grad_precision": args.grad_precision, "parallelism": f"replicas x{world}",
                       "gemm": "sm-pair (cta_group::2, 256x256)" if rh.rl_get_option(rh.RL_OPT_GEMM_PAIR) else
                               "single-sm (128x256)",
                       "l2": "inputs larger than L2 (W 622 MB); 256 MB flush between timed steps"},
            "tc_peak_frac": step_tflops / peak_burst,
            "step_tflops_6NHV": step_tflops,
            "peak_gib": peak_gib, "workspace_peak_gib": work_gib,
            "two_call_ms_per_step": unfused_ms,
            "roofline": roof, "kernels": kernels,
            "e2e": {"value": e_value, "unit": "tokens/s", "ms_per_step": e_ms, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h},
            "clocks": clocks, "gpu_launches": int(launches), "input_gen_s": t_gen}
    if not args.no_elementwise:
        line["elementwise"] = elementwise_side(rh, torch, dev, max(args.steps, 10), args.warmup, peaks)
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
# captures summarised under profiles/ (one launch at the bench's 16384-token chunk).
TRAFFIC = {"gemm_fwd_stats": 12292000000 + 9935062272}


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
    ap.add_argument("--cpu-tokens", type=int, default=128, help="oracle sample for cpu_baseline")
    ap.add_argument("--ref-tokens", type=int, default=32, help="oracle sample per step, --impl reference")
    ap.add_argument("--tokens", type=int, default=None, help="fewer tokens, same shapes (profiling runs)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-unfused", action="store_true", help="skip the two-call side figure")
    ap.add_argument("--no-elementwise", action="store_true", help="skip the elementwise-path side figure")
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
