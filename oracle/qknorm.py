"""Per-head RMSNorm of q and k ahead of the split-halves rotation, fp64 (oracle; test
infrastructure only -- nothing in the package imports it).

Source: Difflet PR #153, FLUX and Wan split-RoPE commits. The per-head q/k RMSNorm weights
are permuted together with the to_q / to_k channels into the split-halves order, so the norm
acts on q and k in that channel layout, just before the rotation; V and everything after the
attention are untouched.

Readings taken where the pages are silent:

* the norm runs over the D channels of one head (the FLUX passage's "per-head qk RMSNorm");
  one weight vector w [D] serves every head, position and batch;
* y = x / sqrt(mean_d(x_d^2) + eps) * w, eps = 1e-6 by default;
* the channel order of w is the one of x (already permuted, as the pages do at load time).
"""
from __future__ import annotations

import numpy as np


def rms_norm_heads(x, w, eps: float = 1e-6) -> np.ndarray:
    """RMSNorm over the last axis (the head channels) of x [..., D] with weight w [D], fp64."""
    x = np.asarray(x, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    assert w.shape == (x.shape[-1],)
    mean_sq = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(mean_sq + float(eps)) * w
