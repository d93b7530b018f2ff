"""Chunk-ordered fp64 restatement of KDA prefill -- TEST INFRASTRUCTURE ONLY.

The pages name the kernel set of the chunked prompt path (vllm.cpp PR #110,
"chunk_kda prefill AOT port", commit description): an in-chunk gate cumsum, the
intra-chunk decayed k.k^T, a unit-lower-triangular solve, the WY recompute of w/u,
the inter-chunk state propagation h and the output o.  They do not print the
algebra.  This module writes it out from the recurrence

    S_t = (I - beta_t k_t k_t^T) Diag(exp g_t) S_{t-1} + beta_t k_t v_t^T,
    o_t = scale * S_t^T q_t

for one chunk of rows r = 0..L-1 that starts from the state h:

    Gam_r     = sum_{i<=r} g_i                       (per key channel)
    A_kk[r,i] = beta_r sum_c k_rc k_ic exp(Gam_rc - Gam_ic)   for i < r
    A_qk[r,i] =        sum_c q_rc k_ic exp(Gam_rc - Gam_ic)   for i <= r
    T         = (I + A_kk)^-1
    W         = T (beta * (k * exp(Gam)))       U = T (beta * v)
    Delta     = U - W h                          (the corrected values)
    O         = scale (q * exp(Gam)) h + scale A_qk Delta
    h'        = Diag(exp Gam_{L-1}) h + (k * exp(Gam_{L-1} - Gam))^T Delta

In exact arithmetic this equals the token recurrence (derivation: unroll
S_r = Diag(e^{Gam_r}) h + sum_{i<=r} Diag(e^{Gam_r - Gam_i}) k_i Delta_i^T, read
S_{r-1} decayed against k_r to get the triangular system for Delta).  Every
exponential here is evaluated exactly per element, with no factorisation, so this
module pins the chunk algebra, not any particular numerical shortcut.
Library routines used as steps: ``numpy.linalg.solve`` for T.
"""
from __future__ import annotations

import numpy as np


def _chunk(q, k, v, g, beta, h, scale):
    L = q.shape[0]
    gam = np.cumsum(g, axis=0)                                    # [L, K]
    # decay[r, i, c] = exp(Gam_rc - Gam_ic), only used where i <= r
    diff = gam[:, None, :] - gam[None, :, :]
    lower_incl = np.tril(np.ones((L, L), dtype=bool))
    diff = np.where(lower_incl[:, :, None], diff, -np.inf)
    dec = np.exp(diff)
    a_kk = beta[:, None] * np.einsum("rc,ic,ric->ri", k, k, dec)
    a_kk = np.tril(a_kk, -1)
    a_qk = np.tril(np.einsum("rc,ic,ric->ri", q, k, dec))
    eye = np.eye(L)
    k_til = k * np.exp(gam)
    q_til = q * np.exp(gam)
    w = np.linalg.solve(eye + a_kk, beta[:, None] * k_til)
    u = np.linalg.solve(eye + a_kk, beta[:, None] * v)
    delta = u - w @ h
    o = scale * (q_til @ h + a_qk @ delta)
    k_hat = k * np.exp(gam[-1][None, :] - gam)
    h_next = np.exp(gam[-1])[:, None] * h + k_hat.T @ delta
    return o, h_next


def prefill_chunked(q, k, v, g, beta, scale, init_state=None, cu_seqlens=None, chunk=64):
    """Same contract as ``oracle.prefill`` (numpy float64 arrays in and out)."""
    q, k, v, g, beta = (np.asarray(x, dtype=np.float64) for x in (q, k, v, g, beta))
    T, H, K = q.shape
    V = v.shape[-1]
    cu = np.asarray([0, T] if cu_seqlens is None else cu_seqlens, dtype=np.int64)
    N = cu.shape[0] - 1
    out = np.zeros((T, H, V))
    final = np.zeros((N, H, K, V))
    for n in range(N):
        bos, eos = int(cu[n]), int(cu[n + 1])
        for hh in range(H):
            h = (np.zeros((K, V)) if init_state is None
                 else np.array(init_state[n, hh], dtype=np.float64))
            for s in range(bos, eos, chunk):
                e = min(s + chunk, eos)
                o, h = _chunk(q[s:e, hh], k[s:e, hh], v[s:e, hh], g[s:e, hh],
                              beta[s:e, hh], h, scale)
                out[s:e, hh] = o
            final[n, hh] = h
    return out, final


def prefill_segmented(q, k, v, g, beta, scale, init_state=None, cu_seqlens=None, chunk=64,
                      segments=2):
    """Same contract as ``oracle.prefill``, evaluated with each sequence split in time.

    The chunk step above is linear in (h, v).  Each sequence's chunks are split into
    ``segments`` runs of consecutive chunks.  Every run is evaluated on its own, from a
    zero state, carrying next to it a K x K state Phi that starts at the identity and
    takes the same chunk step with v = 0 (the homogeneous part): after chunk n, Phi is
    the map from the run's start state to the state there, and the output that step
    gives for Phi (an L x K matrix Psi_n) maps the run's start state to the part of the
    chunk's output the zero start left out.  Then, in order of the runs,

        h_start(p + 1) = Phi_end(p) h_start(p) + h_end(p),    h_start(0) = init,

    and every chunk's output gains Psi_n h_start(p).  The result is the recurrence's,
    in exact arithmetic, for any split; only the order of evaluation differs.
    """
    q, k, v, g, beta = (np.asarray(x, dtype=np.float64) for x in (q, k, v, g, beta))
    T, H, K = q.shape
    V = v.shape[-1]
    cu = np.asarray([0, T] if cu_seqlens is None else cu_seqlens, dtype=np.int64)
    N = cu.shape[0] - 1
    out = np.zeros((T, H, V))
    final = np.zeros((N, H, K, V))
    for n in range(N):
        bos, eos = int(cu[n]), int(cu[n + 1])
        starts = list(range(bos, eos, chunk))
        runs = [r for r in np.array_split(np.arange(len(starts)), max(1, segments)) if r.size]
        for hh in range(H):
            h_start = (np.zeros((K, V)) if init_state is None
                       else np.array(init_state[n, hh], dtype=np.float64))
            for run in runs:
                h_loc, phi = np.zeros((K, V)), np.eye(K)
                for ci in run:
                    s = starts[ci]
                    e = min(s + chunk, eos)
                    args = (q[s:e, hh], k[s:e, hh])
                    o_loc, h_loc_next = _chunk(*args, v[s:e, hh], g[s:e, hh], beta[s:e, hh], h_loc, scale)
                    psi, phi_next = _chunk(*args, np.zeros((e - s, K)), g[s:e, hh], beta[s:e, hh], phi, scale)
                    out[s:e, hh] = o_loc + psi @ h_start
                    h_loc, phi = h_loc_next, phi_next
                h_start = phi @ h_start + h_loc
            final[n, hh] = h_start
    return out, final
