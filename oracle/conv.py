"""Causal depthwise convolution over the packed [q|k|v] channels -- TEST INFRASTRUCTURE ONLY.

The pages put a short causal convolution in front of the KDA op, with its taps carried
per sequence between calls: CausalConv1dFwd over the packed varlen prompt and
CausalConv1dUpdate for the one-token decode step, the carried conv_state split as
chunk(3) into [q|k|v] (vllm.cpp PR #122 "fold Kimi-Linear onto the shared paged
runner", block B2; vllm.cpp PR #113 "paged-incremental decode", commit body: the
conv-tap carry of the decode regime).  They give neither the width nor the activation;
both are arguments here (width W >= 1, activation none or SiLU).

Definition, per sequence and channel c, with the W - 1 carried taps prepended to the
sequence's inputs (oldest first; zeros when the sequence has no slot):

    xe = [taps_0, .., taps_{W-2}, x_0, .., x_{L-1}]
    y_t = act(bias_c + sum_{j=0}^{W-1} w_{c,j} xe_{t+j})        t = 0 .. L-1
    taps <- the last W - 1 entries of xe

so y_t sees x_t and the W - 1 inputs before it (the carried ones before the first).  The
decode step is the same with L = 1.  act(z) = z, or z / (1 + exp(-z)) for SiLU.
Everything in fp64; the taps are stored as given (no arithmetic touches them).
"""
from __future__ import annotations

import numpy as np

ACT_NONE = 0
ACT_SILU = 1


def _f64(x):
    if hasattr(x, "detach"):  # a torch tensor on the CPU (any dtype)
        x = x.detach().cpu().double().numpy()
    return np.asarray(x, dtype=np.float64)


def _act(z, activation):
    if activation == ACT_SILU:
        return z / (1.0 + np.exp(-z))
    return z


def conv_prefill(x, weight, bias, conv_state, state_idx, cu_seqlens, activation=ACT_NONE):
    """x [T, D]; weight [D, W]; bias [D] or None; conv_state [S, W-1, D] float64 numpy
    array updated IN PLACE at the slots state_idx [N] (None: zero taps, nothing kept);
    cu_seqlens [N+1].  Returns y [T, D] float64 (rows outside every sequence are zero)."""
    x = _f64(x)
    w = _f64(weight)
    D, W = w.shape
    b = np.zeros(D) if bias is None else _f64(bias)
    cu = [int(c) for c in cu_seqlens]
    y = np.zeros_like(x)
    for n in range(len(cu) - 1):
        s, e = cu[n], cu[n + 1]
        slot = None if conv_state is None else int(state_idx[n])
        if slot is not None and not (0 <= slot < conv_state.shape[0]):
            slot = None
        taps = conv_state[slot].copy() if slot is not None else np.zeros((W - 1, D))
        xe = np.concatenate([taps, x[s:e]], axis=0)
        for t in range(e - s):
            acc = b.copy()
            for j in range(W):
                acc = acc + w[:, j] * xe[t + j]
            y[s + t] = _act(acc, activation)
        if slot is not None and W > 1:
            conv_state[slot] = xe[xe.shape[0] - (W - 1):]
    return y


def conv_update(x, weight, bias, conv_state, state_idx, activation=ACT_NONE):
    """One token per sequence: x [N, D]; the taps of slot state_idx[n] are used and
    shifted in place.  Returns y [N, D]."""
    x = _f64(x)
    N = x.shape[0]
    cu = np.arange(N + 1)
    return conv_prefill(x, weight, bias, conv_state, state_idx, cu, activation)
