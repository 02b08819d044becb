"""Plain, slow, fp64 CPU oracle for the fused LM head + unified RL loss and the
elementwise PPO / TIS / mismatch path.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` may import it.  It shares no code with the CUDA path
(``lm_head_gb300``), and the CUDA path never calls it: the product has no CPU fallback.

Every function cites the page and section it restates.  The pages:
  * "IPO (INTELLECT Policy Optimization)" (prime-rl docs): "Masking by Probability,
    Not Ratio", "Choosing eps".
  * "Rollout Correction Methods" (miles docs): "Algorithms" (standard / bypass /
    decoupled 3-policy PPO), "Config keys", "Importance Sampling", "Rejection Sampling",
    "Mismatch Metrics".
  * "10-KL-clip-entropy" (verl blog): section 2 (PPO clip, dual clip, clip metrics,
    default constants).
  * prime-rl pull request #4233 ("One RL loss for ipo, icepop and the new reinforce"):
    the loss_t equation, the two estimator rules for u, "What changes", "Numbers".

Readings where the pages are silent (R1..R20) are marked ``READING`` in the code.

Pinning status: every public function here is pinned by ``tests/test_oracle_*.py``
against closed forms, worked examples from the pages, brute force or finite
differences, except the items listed in ``PARITY_UNPINNED`` (parity unpinned: the value of
the decoupled-TIS bound, reading R11, and the rollout-correction default bounds; the pages
give neither number, and the functions themselves are pinned with explicit values).
"""
from .rl_head import (HeadParams, LOSS_IPO, LOSS_ICEPOP, LOSS_REINFORCE, KL_EXACT, KL_K1,
                      STALE_NONE, STALE_INV_SQRT, head_forward, head_backward, head_loss_total,
                      head_token_logits, token_forward, validate_support, vocab_shard_stats)
from .policy import PolicyParams, policy_loss_elementwise, IPO_CURVE_EPS
from .rollout import RolloutParams, rollout_correction, rollout_metrics_named

PARITY_UNPINNED = (
    "decoupled TIS bound: the pages give no value; reading R11 (token-level truncate at 2.0)",
    "rollout correction defaults: the pages give no bound values; tests set every bound "
    "explicitly, and the defaults (tis bounds [0.5, 2.0]) are a reading only",
)

__all__ = [
    "HeadParams", "LOSS_IPO", "LOSS_ICEPOP", "LOSS_REINFORCE", "KL_EXACT", "KL_K1", "STALE_NONE",
    "STALE_INV_SQRT", "head_forward", "head_backward", "head_loss_total", "head_token_logits",
    "token_forward", "validate_support", "vocab_shard_stats", "PolicyParams", "policy_loss_elementwise", "IPO_CURVE_EPS", "PARITY_UNPINNED",
    "RolloutParams", "rollout_correction", "rollout_metrics_named",
]
