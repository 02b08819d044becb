"""The vocabulary-split head on one GPU, the ranks emulated one after another (their
collectives by stacking and summing on the device): each rank's shard statistics and
owned logits (rl_head_shard_stats on its rows of W), the loss from the gathered statistics
(rl_head_loss_from_shard_stats) and each rank's backward on its rows (rl_head_loss_bwd
with local ids), against the fp64 oracle and against the single-GPU path."""
import dataclasses

import numpy as np
import pytest
import torch

import lm_head_gb300 as rh
import oracle
import workloads
from gpu_checks import check_forward, grad_readings
from lm_head_gb300 import vocab_parallel as vp
from parity_util import oracle_params

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from lm_head_gb300 import build
    build.build()
    rh.load()


class EmulatedExchange:
    """The ranks' collectives in one process: the per-rank values are collected, then
    gathered or summed in rank order."""

    def __init__(self, world):
        self.world = world


def _run_ranks(case, hp, world):
    dev = case.to("cuda")
    batch = rh.HeadBatch.from_case(dev)
    ops = vp.LibraryOps()
    parts = vp.vocab_partition(case.V, world)
    locals_, stats, zlabs, zsups = [], [], [], []
    for r, (a, b) in enumerate(parts):
        local = ops.local_batch(batch, dev.W[a:b].contiguous(), vp.Shard(r, world, a, b))
        st, zl, zs = ops.stats(local, hp)
        locals_.append(local)
        stats.append(st)
        zlabs.append(zl)
        zsups.append(zs)
    stats_all = torch.stack(stats)                         # the all-gather, rank order
    zlab = torch.stack(zlabs).sum(0)                       # the all-reduce of owned logits
    zsup = torch.stack(zsups).sum(0) if case.nnz else zsups[0]
    fwd = ops.loss(batch, hp, stats_all, zlab, zsup, case.V)
    torch.cuda.synchronize()
    mask = case.loss_mask.float()
    dloss = (mask / mask.sum().clamp(min=1)).cuda()
    dXs, dWs = [], []
    for local in locals_:
        dXp, dWp = ops.backward(local, hp, fwd, dloss)
        dXs.append(ops.dx_to_sum(dXp))
        dWs.append(dWp)
    dX = ops.dx_from_sum(torch.stack(dXs).sum(0))          # the all-reduce of the dX parts
    dW = torch.cat(dWs)
    torch.cuda.synchronize()
    return batch, fwd, dX, dW, dloss


@pytest.mark.parametrize("world", [2, 3])
@pytest.mark.parametrize("kind", ["draws", "replay"])
def test_emulated_ranks_against_the_oracle_and_one_gpu(world, kind):
    if kind == "draws":
        case = workloads.make_head_case("c1", n_tokens=200, H=128, V=1024, hidden_scale=6.0, noise=0.7, age_max=3,
                                        loss_mask_frac=0.1, seed=51)
        hp = rh.HeadParams(loss_type=rh.RL_LOSS_IPO, eps=0.1, max_importance_ratio=3.0, kl_coeff=0.02,
                           kl_staleness=rh.RL_STALE_INV_SQRT, bwd_mode=rh.RL_BWD_DENSE)
    else:
        case = workloads.make_head_case("c1", n_tokens=200, H=128, V=1024, support="replay", top_p=0.9,
                                        hidden_scale=6.0, noise=0.7, seed=52)
        hp = rh.HeadParams(loss_type=rh.RL_LOSS_ICEPOP, bwd_mode=rh.RL_BWD_DENSE)
    batch, fwd, dX, dW, dloss = _run_ranks(case, hp, world)
    assert fwd.status_bits() == 0, rh.status_names(fwd.status_bits())
    ref = oracle.head_forward(case.numpy(), oracle_params(hp))
    check_forward(case, hp, fwd, ref, tag=f"vocab-split x{world} {kind}")
    rX, rW, bnd = oracle.head_backward(case.numpy(), oracle_params(hp), dloss.cpu().double().numpy(), want_bounds=True)
    grad_readings(f"vocab-split x{world} {kind}", dX, dW, rX, rW, bnd, case.H, rh.RL_GRAD_BF16)
    # the single-GPU two-call path on the same batch
    f1 = rh.rl_head_loss_fwd(batch, hp)
    dX1, dW1, st = rh.rl_head_loss_bwd(batch, hp, f1.saved, dloss)
    torch.cuda.synchronize()
    torch.testing.assert_close(fwd.lse, f1.lse, rtol=0, atol=2e-6)
    torch.testing.assert_close(fwd.loss, f1.loss, rtol=1e-5, atol=1e-6)
    assert torch.equal(fwd.mask_label, f1.mask_label)
    # the same arithmetic on a bf16 gradient operand whose logsumexp differs in its last
    # bits (the statistics combine over other splits): within two bf16 roundings of the
    # largest element
    assert float((dW - dW1).abs().max()) <= 2 ** -7 * float(dW1.abs().max())
    assert float((dX.float() - dX1.float()).abs().max()) <= 2 ** -7 * float(dX1.float().abs().max())


def test_remap_keeps_rows_ascending():
    ids = torch.tensor([0, 5, 255, 256, 300, 511, 512, 900], dtype=torch.int32, device="cuda")
    loc = rh.rl_head_shard_remap(ids, 256, 512)
    torch.cuda.synchronize()
    assert loc.tolist() == [-1, -1, -1, 0, 44, 255, 256, 256]
