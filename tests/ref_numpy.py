"""Independent NumPy (float64) statement of ONE draft-token step of the gated
delta rule, in matrix form, for cross-checking the C oracle.

Written separately from ``oracle/gdn_oracle.c`` (which loops over scalars);
the two share nothing but the definition of the step in the vLLM PR reports
"PR #46090 report" (fla.cpp listing: per (sequence, v-head) gated delta-rule
update with in-kernel q/k L2 normalisation) and "PR #51674 report"
(implementation step 1: gated delta rule, then gated RMSNorm epilogue).
"""
from __future__ import annotations

import numpy as np


def token_step(S, q, k, v, a, b, A_log, dt_bias, *, scale, qk_eps=1e-6, threshold=20.0):
    """S: [K, V] float64 (not modified).  q, k: [K]; v: [V]; scalars a, b,
    A_log, dt_bias.  Returns (S_new [K, V], o [V])."""
    x = a + dt_bias
    sp = x if x > threshold else np.log1p(np.exp(x))
    decay = np.exp(-np.exp(A_log) * sp)
    beta = 1.0 / (1.0 + np.exp(-b))
    kh = k / np.sqrt(k @ k + qk_eps)
    qh = q / np.sqrt(q @ q + qk_eps) * scale
    Sd = decay * S
    vprime = beta * (v - Sd.T @ kh)
    S_new = Sd + np.outer(kh, vprime)
    return S_new, S_new.T @ qh


def gated_rmsnorm(o, z, w, eps):
    """o * rsqrt(mean(o^2) + eps) * w * silu(z), all float64."""
    silu = z * (1.0 / (1.0 + np.exp(-z)))
    return o / np.sqrt(np.mean(o * o) + eps) * w * silu
