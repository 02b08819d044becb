"""The vocabulary-split head's rank logic (lm_head_gb300.vocab_parallel) on CPU: two gloo
ranks (127.0.0.1), each holding half of W's rows, run the forward and backward steps with
an fp64 stand-in for the per-rank ops (the oracle restricted to the rank's vocabulary
range); the gathered statistics combine to the oracle's full-vocabulary logsumexp and
entropy, every label / support logit arrives from its owner, the summed dX parts equal the
oracle's dX and each rank's dW rows the oracle's.  The GPU ops themselves are checked
against the oracle and the single-GPU path in tests/test_gpu_vocab_parallel.py (one GPU
emulating the ranks)."""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from lm_head_gb300.vocab_parallel import Shard, vocab_partition  # noqa: E402


def test_partition_covers_the_vocabulary_in_tile_multiples():
    for V, world in ((151936, 2), (151936, 8), (1000, 2), (1024, 4), (300, 2), (257, 2)):
        parts = vocab_partition(V, world)
        assert parts[0][0] == 0 and parts[-1][1] == V and len(parts) == world
        for (a, b), (c, d) in zip(parts, parts[1:]):
            assert b == c and a < b and b % 256 == 0
        sizes = [b - a for a, b in parts[:-1]]
        assert max(sizes) - min(sizes) <= 256 if sizes else True
    with pytest.raises(ValueError):
        vocab_partition(300, 3)


class OracleOps:
    """fp64 stand-in for the per-rank GPU steps: the oracle on the rank's range."""

    def __init__(self, inputs, op):
        import oracle
        self.oracle = oracle
        self.inputs = inputs
        self.op = op

    def local_batch(self, batch, w_shard, shard):
        return shard

    def stats(self, shard, params):
        r = self.oracle.vocab_shard_stats(self.inputs, self.op, shard.begin, shard.end)
        t = lambda x: torch.from_numpy(np.ascontiguousarray(x, dtype=np.float64))
        return torch.stack([t(r["m"]), t(r["s"]), t(r["u"])]), t(r["zlab"]), t(r["zsup"])

    def loss(self, batch, params, stats_all, zlab, zsup, V):
        m, s, u = stats_all[:, 0], stats_all[:, 1], stats_all[:, 2]
        M = m.max(dim=0).values
        f = torch.exp(m - M)
        S = (f * s).sum(dim=0)
        U = (f * (u + (m - M) * s)).sum(dim=0)
        return {"lse": M + torch.log(S), "entropy": torch.log(S) - U / S, "zlab": zlab, "zsup": zsup}

    def backward(self, shard, params, fwd, dloss):
        cols = np.arange(shard.begin, shard.end)
        dX, dW = self.oracle.head_backward(self.inputs, self.op, dloss, vcols=cols, vrows=cols)
        return torch.from_numpy(dX), torch.from_numpy(dW)

    def dx_to_sum(self, x):
        return x

    def dx_from_sum(self, x):
        return x


def _case():
    import workloads
    return workloads.make_head_case("c1", n_tokens=64, H=64, V=1000, hidden_scale=4.0, noise=0.5, K=6, seed=41)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import oracle
    from lm_head_gb300 import vocab_parallel as vp
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    case = _case()
    inp = case.numpy()
    op = oracle.HeadParams(kl_coeff=0.02, kl_staleness=oracle.STALE_INV_SQRT)
    begin, end = vp.vocab_partition(case.V, world)[rank]
    shard = vp.Shard(rank, world, begin, end)
    ops = OracleOps(inp, op)
    fwd, local = vp.forward(None, None, shard, case.V, op, ops, vp.TorchExchange())
    dloss = np.full(case.N, 1.0 / case.N)
    dX, dW = vp.backward(local, op, fwd, dloss, ops, vp.TorchExchange())
    np.savez(os.path.join(out_dir, f"rank{rank}.npz"), lse=fwd["lse"].numpy(), entropy=fwd["entropy"].numpy(),
             zlab=fwd["zlab"].numpy(), zsup=fwd["zsup"].numpy(), dX=dX.numpy(), dW=dW.numpy(), begin=begin, end=end)
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_against_the_oracle(tmp_path):
    import oracle
    world = 2
    mp.spawn(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    case = _case()
    inp = case.numpy()
    op = oracle.HeadParams(kl_coeff=0.02, kl_staleness=oracle.STALE_INV_SQRT)
    ref = oracle.head_forward(inp, op)
    rX, rW = oracle.head_backward(inp, op, np.full(case.N, 1.0 / case.N))
    Z = inp["hidden"] @ inp["W"].T
    off = inp["offsets"]
    rows = np.repeat(np.arange(case.N), np.diff(off))
    for rank in range(world):
        d = np.load(tmp_path / f"rank{rank}.npz")
        np.testing.assert_allclose(d["lse"], ref["lse"], rtol=1e-13)
        np.testing.assert_allclose(d["entropy"], ref["entropy"], rtol=1e-11, atol=1e-12)
        np.testing.assert_array_equal(d["zlab"], Z[np.arange(case.N), inp["labels"]])     # from its owner
        np.testing.assert_array_equal(d["zsup"], Z[rows, inp["ids"]])
        np.testing.assert_allclose(d["dX"], rX, rtol=1e-10, atol=1e-15)
        b, e = int(d["begin"]), int(d["end"])
        np.testing.assert_allclose(d["dW"], rW[b:e], rtol=1e-10, atol=1e-15)
    # both ranks hold identical combined results
    a, b = np.load(tmp_path / "rank0.npz"), np.load(tmp_path / "rank1.npz")
    assert np.array_equal(a["lse"], b["lse"]) and np.array_equal(a["dX"], b["dX"])
