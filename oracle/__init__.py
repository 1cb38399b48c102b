"""Float64 CPU oracle for Selective Attention Freezing (SAF).

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import this
package: only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU
baseline leg (``cpu_baseline`` / ``--impl reference``) use it.  It shares no
code with the CUDA library (no kernels, headers, helpers or tables) and it
imports nothing from ``dynamic_causal_attention_gb300``.

Every function materialises full T x T matrices in float64 and follows the
plain definitions of the method as given in "When Can Attention Heads Be
Statically Defined?" (the close-reading notes of Li, Tai, Fonseca and Cohen):

* dynamic head: §1, the causal softmax attention equation
  A = softmax_causal(Q K^T / sqrt(d_h)), Z = A V;
* static (frozen) head: §3 Eq. (3), P(i,j) = exp(alpha(j) + rho(i-j)) / Z(i)
  for j <= i and 0 for j > i;
* backward: §3.3 / App. D.2 (the static head's attention backward is only
  dV = P^T dZ; the alpha/rho gradients are the plain chain rule of Eq. (3));
* calibration: §3.1, the sample mean A_hat and Eq. (1) s_var, then the global
  ascending sort and the first k = round(r L H) heads;
* compact fit: Eq. (3)/(4) and App. A.2, alpha/rho fitted to A_hat by Adam on
  the row-wise cross-entropy, gated by a mean row KL of 0.2 nat.

Parity status: every function here is pinned by ``tests/test_oracle_*.py``
against closed forms, hand-worked fixtures in ``tests/golden/``, finite
differences, invariants and library routines.  No function is "parity
unpinned".
"""

from .attention import (
    causal_mask,
    dynamic_head_fwd,
    dynamic_head_bwd,
    static_pattern,
    static_log_normaliser,
    static_head_fwd,
    static_head_bwd,
    hybrid_attn_fwd,
    hybrid_attn_bwd,
    gqa_hybrid_attn_fwd,
    gqa_hybrid_attn_bwd,
    dynamic_head_fwd_rows,
    static_head_fwd_rows,
    dynamic_head_bwd_rows,
    static_head_bwd_rows,
)
from .fit import (
    marginals,
    fit_loss,
    fit_gradient,
    mean_row_kl,
    adam_step,
    compact_fit,
    select_fitted,
)
from .calibration import (
    calib_mean,
    calib_svar,
    calib_mean_svar,
    num_select,
    select_heads,
    reconstruction_risk,
    calib_kl_score,
    sharp_mean_pattern,
)

__all__ = [
    "causal_mask",
    "dynamic_head_fwd",
    "dynamic_head_bwd",
    "static_pattern",
    "static_log_normaliser",
    "static_head_fwd",
    "static_head_bwd",
    "hybrid_attn_fwd",
    "hybrid_attn_bwd",
    "gqa_hybrid_attn_fwd",
    "gqa_hybrid_attn_bwd",
    "dynamic_head_fwd_rows",
    "static_head_fwd_rows",
    "dynamic_head_bwd_rows",
    "static_head_bwd_rows",
    "calib_mean",
    "calib_svar",
    "calib_mean_svar",
    "num_select",
    "select_heads",
    "reconstruction_risk",
    "calib_kl_score",
    "sharp_mean_pattern",
    "marginals",
    "fit_loss",
    "fit_gradient",
    "mean_row_kl",
    "adam_step",
    "compact_fit",
    "select_fitted",
]
