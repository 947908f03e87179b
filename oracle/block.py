"""CPU oracle for the two steps around the scan in a Mamba-2 block (float64, numpy).

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` use this module; the product never imports it.

``causal_conv1d``  the depthwise causal convolution of the block's input branch, then SiLU.
                   youngju.dev "Mamba / selective SSM" article, the Mamba block listing: a
                   depthwise ``nn.Conv1d`` (groups = channels, kernel d_conv, padding
                   d_conv - 1, bias) whose output is cut to the first L positions ("causal
                   trim"), followed by ``F.silu``.  Qiita "Mamba-2 / SSD" article, section 5.1:
                   the separate causal-conv1d package the scan runs after.  Written out: with
                   width K and the K - 1 inputs before the sequence taken from ``state`` (zeros
                   by default),
                       out[b, t, c] = silu(bias[c] + sum_{k=0..K-1} w[c, k] x[b, t - (K-1) + k, c]).
                   The final state is the last K - 1 inputs (the window the next call starts
                   from), so a sequence split into pieces gives the same result.

``gated_rmsnorm``  the step after the scan: ``y = rmsnorm(y) * silu(z)`` (Qiita "Mamba-2 / SSD"
                   article, section 4.2, step 4), per token over groups of ``group_size``
                   features:
                       out[r, i] = y[r, i] / sqrt(mean_{j in group(i)} y[r, j]^2 + eps)
                                   * w[i] * silu(z[r, i]).
                   The pages fix neither eps nor the weight: eps is a parameter (default
                   1e-5), the weight a per-feature vector (ones when absent), and an absent z
                   means no gate.

silu(v) = v / (1 + exp(-v)).  Inputs of any float dtype (numpy or torch) are upcast to float64.
"""
from __future__ import annotations

import numpy as np

from . import _f64


def silu(v):
    v = np.asarray(v, dtype=np.float64)
    return v / (1.0 + np.exp(-v))


def causal_conv1d(x, w, bias=None, state=None, apply_silu: bool = True):
    """x [b, L, C], w [C, K], bias [C] or None, state [b, K-1, C] or None (zeros).

    Returns (out [b, L, C], final_state [b, K-1, C]), float64.
    """
    x = _f64(x)
    w = _f64(w)
    bsz, L, C = x.shape
    K = w.shape[1]
    if w.shape != (C, K):
        raise ValueError("oracle: w must be [C, K]")
    prev = np.zeros((bsz, K - 1, C)) if state is None else _f64(state)
    if prev.shape != (bsz, K - 1, C):
        raise ValueError("oracle: state must be [b, K-1, C]")
    xp = np.concatenate([prev, x], axis=1)          # position t of x is row t + K - 1 of xp
    acc = np.zeros((bsz, L, C)) if bias is None else np.broadcast_to(_f64(bias), (bsz, L, C)).copy()
    for k in range(K):
        acc += w[:, k][None, None, :] * xp[:, k:k + L, :]
    out = silu(acc) if apply_silu else acc
    final = xp[:, L:L + K - 1, :].copy()            # the last K - 1 inputs
    return out, final


def gated_rmsnorm(y, z=None, w=None, eps: float = 1e-5, group_size: int = None):
    """y, z [rows, D] (or any leading shape with D last), w [D] or None.  Returns float64."""
    y = _f64(y)
    shape = y.shape
    D = shape[-1]
    g = D if group_size is None else int(group_size)
    if D % g != 0:
        raise ValueError("oracle: group_size must divide the feature count")
    yr = y.reshape(-1, D // g, g)
    ms = np.mean(yr * yr, axis=-1, keepdims=True)
    out = (yr / np.sqrt(ms + eps)).reshape(shape)
    if w is not None:
        out = out * _f64(w)
    if z is not None:
        out = out * silu(_f64(z))
    return out
