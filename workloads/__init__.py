"""Seeded synthetic workloads for the fused LM head + RL loss and the elementwise path.

This module only *synthesises inputs*: hidden states, head weights, the sampler's
distribution and its draws, advantages and masks.  It holds none of the trainer-side
loss arithmetic.  Both the CUDA path (through ``lm_head_gb300``) and the fp64 oracle
(``oracle/``) consume what it returns; neither side imports the other.

The sampler side is the inference engine of the pages ("prime-rl pull request #4233",
"What changes": sampler probabilities, replay masks, K i.i.d. draws).  Its logits are
the trainer logits plus Gaussian noise, as the workload descriptions state, so this
module does compute ``hidden @ W.T`` once, in fp32, to build that *input* distribution.

Shapes (tokens N, hidden H, vocab V):
  c1  N=256   (8 x 32),    H=128,  V=1024,   K=16 draws, noise 0.05, ipo
  c2  N=4096  (16 x 256),  H=2048, V=151936, replayed top-p 0.97, noise 0.1, icepop
  c3  N=16384 (64 x 256),  H=2048, V=151936, replayed top-p 0.97, noise 0.1, ipo, sparse bwd
  c4  N=65536 (128 x 512), H=2048, V=151936, K=16 draws, noise 0.1, ipo + exact KL
  c5  1.8M valid tokens, per-token logprobs for the elementwise PPO/TIS path

``variant="pages"`` scales hidden row t by s_t ~ logUniform[7, 16] so that top-p 0.97
keeps a handful of ids per token (the "real chat kept counts" shape); ``"literal"``
keeps hidden ~ N(0, 1), where top-p 0.97 keeps most of the vocabulary.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch

BASE_SEED = 20261202

HEAD_CONFIGS = {
    "c1": dict(n_seq=8, seq_len=32, H=128, V=1024, support="draws", K=16, noise=0.05,
               top_p=None, loss="ipo", kl_coeff=0.0, age_max=0, bwd="dense"),
    "c2": dict(n_seq=16, seq_len=256, H=2048, V=151936, support="replay", K=None, noise=0.1,
               top_p=0.97, loss="icepop", kl_coeff=0.0, age_max=0, bwd="dense"),
    "c3": dict(n_seq=64, seq_len=256, H=2048, V=151936, support="replay", K=None, noise=0.1,
               top_p=0.97, loss="ipo", kl_coeff=0.0, age_max=0, bwd="sparse"),
    "c4": dict(n_seq=128, seq_len=512, H=2048, V=151936, support="draws", K=16, noise=0.1,
               top_p=None, loss="ipo", kl_coeff=0.01, age_max=4, bwd="dense"),
}
CONFIG_INDEX = {"c1": 1, "c2": 2, "c3": 3, "c4": 4, "c5": 5}


@dataclasses.dataclass
class HeadCase:
    """One batch for the head path.  Tensors live on ``device``.

    hidden    [N, H] bf16          W          [V, H] bf16
    labels    [N]    int32         label_logq [N]    fp32  (sampler log q of the label)
    adv       [N]    fp32          loss_mask  [N]    uint8 (1 = RL token)
    age       [N]    int32         replayed   [N]    uint8
    offsets   [N+1]  int64         ids        [nnz]  int32 (ascending within a row)
    logq      [nnz]  fp32          (sampler log q at each support entry)
    """
    name: str
    hidden: torch.Tensor
    W: torch.Tensor
    labels: torch.Tensor
    label_logq: torch.Tensor
    adv: torch.Tensor
    loss_mask: torch.Tensor
    age: torch.Tensor
    replayed: torch.Tensor
    offsets: torch.Tensor
    ids: torch.Tensor
    logq: torch.Tensor
    temperature: float
    cfg: dict

    @property
    def N(self) -> int:
        return int(self.hidden.shape[0])

    @property
    def H(self) -> int:
        return int(self.hidden.shape[1])

    @property
    def V(self) -> int:
        return int(self.W.shape[0])

    @property
    def nnz(self) -> int:
        return int(self.ids.shape[0])

    def to(self, device) -> "HeadCase":
        kw = {f.name: getattr(self, f.name) for f in dataclasses.fields(self)}
        for k, v in kw.items():
            if isinstance(v, torch.Tensor):
                kw[k] = v.to(device)
        return HeadCase(**kw)

    def numpy(self) -> dict:
        """Host copies as numpy; bf16 tensors become the exact fp64 values they hold."""
        out = {}
        for f in dataclasses.fields(self):
            v = getattr(self, f.name)
            if isinstance(v, torch.Tensor):
                if v.dtype == torch.bfloat16:
                    out[f.name] = v.detach().to("cpu", torch.float64).numpy()
                else:
                    out[f.name] = v.detach().cpu().numpy()
            else:
                out[f.name] = v
        return out


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _sampler_logprobs(hidden, W, rows, temperature, noise, g):
    """Sampler log-probabilities for token rows: log_softmax((x W^T)/T + N(0, noise))."""
    z = (hidden[rows].float() @ W.float().T) / temperature
    z = z + noise * torch.randn(z.shape, generator=g, device=z.device, dtype=z.dtype)
    return torch.log_softmax(z, dim=-1)


def make_head_case(name: str = "c1", *, n_tokens: Optional[int] = None, seed: Optional[int] = None,
                   device="cpu", variant: str = "literal", loss_mask_frac: float = 0.0,
                   chunk: int = 1024, H: Optional[int] = None, V: Optional[int] = None,
                   support: Optional[str] = None, K: Optional[int] = None,
                   top_p: Optional[float] = None, noise: Optional[float] = None,
                   hidden_scale: float = 1.0, temperature: float = 1.0,
                   age_max: Optional[int] = None) -> HeadCase:
    """Build a seeded head batch shaped like config ``name``; keyword args override fields.

    ``n_tokens`` truncates/extends the token count (rounded down to whole sequences when
    larger than one sequence); ``loss_mask_frac`` marks that fraction of tokens non-RL.
    """
    cfg = dict(HEAD_CONFIGS[name])
    if H is not None:
        cfg["H"] = H
    if V is not None:
        cfg["V"] = V
    if support is not None:
        cfg["support"] = support
    if K is not None:
        cfg["K"] = K
    if top_p is not None:
        cfg["top_p"] = top_p
    if noise is not None:
        cfg["noise"] = noise
    if age_max is not None:
        cfg["age_max"] = age_max
    N = cfg["n_seq"] * cfg["seq_len"] if n_tokens is None else int(n_tokens)
    seq_len = min(cfg["seq_len"], N)
    Hd, Vd = cfg["H"], cfg["V"]
    if seed is None:
        seed = BASE_SEED + CONFIG_INDEX[name]
    dev = torch.device(device)
    g = _gen(dev, seed)

    hidden = torch.randn((N, Hd), generator=g, device=dev) * hidden_scale
    if variant == "pages":
        # s_t ~ logUniform[7, 16]: sharp rows, so top-p keeps few ids per token.
        s = torch.exp(math.log(7.0) + (math.log(16.0) - math.log(7.0))
                      * torch.rand((N, 1), generator=g, device=dev))
        hidden = hidden * s
    hidden = hidden.to(torch.bfloat16)
    W = (0.02 * torch.randn((Vd, Hd), generator=g, device=dev)).to(torch.bfloat16)

    labels = torch.empty(N, dtype=torch.int32, device=dev)
    label_logq = torch.empty(N, dtype=torch.float32, device=dev)
    rows_ids, rows_logq, counts = [], [], []
    replayed_flag = 1 if cfg["support"] == "replay" else 0
    for c0 in range(0, N, chunk):
        rows = torch.arange(c0, min(N, c0 + chunk), device=dev)
        lq = _sampler_logprobs(hidden, W, rows, temperature, cfg["noise"], g)
        if cfg["support"] == "draws":
            Kd = int(cfg["K"])
            q = lq.exp()
            draws = torch.multinomial(q, Kd + 1, replacement=True, generator=g)
            lab = draws[:, 0]
            d = torch.sort(draws[:, 1:], dim=1).values
            labels[rows] = lab.to(torch.int32)
            label_logq[rows] = lq.gather(1, lab[:, None])[:, 0]
            rows_ids.append(d.reshape(-1).to(torch.int32))
            rows_logq.append(lq.gather(1, d).reshape(-1))
            counts.append(torch.full((rows.numel(),), Kd, dtype=torch.int64, device=dev))
        else:
            # Replayed truncation: shortest prefix of q (descending, ties by lower id)
            # whose mass reaches top_p, including the crossing token; renormalised.
            top_p_v = float(cfg["top_p"])
            sq, order = torch.sort(lq, dim=1, descending=True, stable=True)
            cum = torch.cumsum(sq.exp().double(), dim=1)
            kept = torch.clamp((cum < top_p_v).sum(dim=1) + 1, max=Vd)
            for i in range(rows.numel()):
                k = int(kept[i])
                ids_i = torch.sort(order[i, :k]).values
                lq_i = lq[i, ids_i]
                lq_i = lq_i - torch.logsumexp(lq_i, dim=0)
                pick = torch.multinomial(lq_i.exp(), 1, generator=g)[0]
                labels[c0 + i] = ids_i[pick].to(torch.int32)
                label_logq[c0 + i] = lq_i[pick]
                rows_ids.append(ids_i.to(torch.int32))
                rows_logq.append(lq_i.float())
            counts.append(kept.to(torch.int64))
        del lq
    counts_t = torch.cat(counts)
    offsets = torch.zeros(N + 1, dtype=torch.int64, device=dev)
    offsets[1:] = torch.cumsum(counts_t, dim=0)
    ids = torch.cat(rows_ids).to(torch.int32)
    logq = torch.cat(rows_logq).to(torch.float32)

    n_seq = (N + seq_len - 1) // seq_len
    adv_seq = torch.randn(n_seq, generator=g, device=dev)
    adv = adv_seq.repeat_interleave(seq_len)[:N].contiguous().float()
    if loss_mask_frac > 0:
        loss_mask = (torch.rand(N, generator=g, device=dev) >= loss_mask_frac).to(torch.uint8)
    else:
        loss_mask = torch.ones(N, dtype=torch.uint8, device=dev)
    amax = int(cfg["age_max"])
    if amax > 0:
        age = torch.randint(0, amax + 1, (N,), generator=g, device=dev, dtype=torch.int64).to(torch.int32)
    else:
        age = torch.zeros(N, dtype=torch.int32, device=dev)
    replayed = torch.full((N,), replayed_flag, dtype=torch.uint8, device=dev)
    return HeadCase(name=name, hidden=hidden, W=W, labels=labels, label_logq=label_logq, adv=adv,
                    loss_mask=loss_mask, age=age, replayed=replayed, offsets=offsets, ids=ids,
                    logq=logq, temperature=float(temperature), cfg=cfg)


@dataclasses.dataclass
class PolicyCase:
    """Elementwise batch: B sequences padded to ``max_len``; flat [T = B*max_len] arrays."""
    lp_theta: np.ndarray   # fp32 trainer (current policy) log-prob of each sampled token
    lp_old: np.ndarray     # fp32 proximal / recomputed-old log-prob
    lp_samp: np.ndarray    # fp32 rollout (sampler) log-prob
    adv: np.ndarray        # fp32 per-token advantage (one value per sequence)
    mask: np.ndarray       # uint8 response mask (1 = valid token)
    seq_lens: np.ndarray   # int64 valid length of each sequence
    max_len: int

    @property
    def T(self) -> int:
        return int(self.lp_theta.shape[0])

    def packed(self) -> dict:
        """The same valid tokens laid end to end (no padding, no mask): lp_theta, lp_old,
        lp_samp, adv as [n_valid] fp32 arrays and the sequences' cumulative lengths
        cu_seqlens [B + 1] int64."""
        keep = self.mask.astype(bool)
        out = {k: np.ascontiguousarray(getattr(self, k)[keep]) for k in ("lp_theta", "lp_old", "lp_samp", "adv")}
        out["cu_seqlens"] = np.concatenate([[0], np.cumsum(self.seq_lens)]).astype(np.int64)
        return out


def make_policy_case(total_tokens: int = 1_800_000, *, min_len: int = 64, max_len: int = 4096,
                     seed: Optional[int] = None, x_mean: float = -1.0, x_std: float = 2.5,
                     old_noise: float = 0.3, theta_noise: float = 0.1) -> PolicyCase:
    """Per-token log-probs for the elementwise path (numpy PCG64, fp32 outputs).

    Sequence lengths ~ U{min_len..max_len} until they sum to ``total_tokens`` (the last
    one is cut).  logit(p_samp) ~ N(x_mean, x_std); the trainer ("old") logit adds
    N(0, old_noise); the current policy adds N(0, theta_noise) on top of that.
    """
    if seed is None:
        seed = BASE_SEED + CONFIG_INDEX["c5"]
    rng = np.random.Generator(np.random.PCG64(seed))
    lens = []
    tot = 0
    while tot < total_tokens:
        L = int(rng.integers(min_len, max_len + 1))
        L = min(L, total_tokens - tot)
        lens.append(L)
        tot += L
    lens = np.asarray(lens, dtype=np.int64)
    B = len(lens)
    T = B * max_len
    mask = (np.arange(max_len)[None, :] < lens[:, None]).reshape(-1).astype(np.uint8)
    x = rng.normal(x_mean, x_std, size=T)
    x_old = x + rng.normal(0.0, old_noise, size=T)
    x_theta = x_old + rng.normal(0.0, theta_noise, size=T)
    # log(sigmoid(x)) = -log1p(exp(-x)), evaluated stably
    def log_sigmoid(v):
        return -np.logaddexp(0.0, -v)
    adv_seq = rng.normal(0.0, 1.0, size=B)
    adv = np.repeat(adv_seq, max_len)
    return PolicyCase(lp_theta=log_sigmoid(x_theta).astype(np.float32),
                      lp_old=log_sigmoid(x_old).astype(np.float32),
                      lp_samp=log_sigmoid(x).astype(np.float32),
                      adv=adv.astype(np.float32), mask=mask, seq_lens=lens, max_len=max_len)
