"""Shared test helpers: moving seeded cases to the GPU and comparing with the oracle."""
from __future__ import annotations

import numpy as np
import torch

import oracle

# Parity bar: max |gpu - oracle| / max |oracle| per tensor.
TOL = {"bf16": 2e-3, "f32": 1e-4}


def dtype_name(t: torch.Tensor) -> str:
    return "bf16" if t.dtype == torch.bfloat16 else "f32"


def rel_err(got, ref) -> float:
    got = np.asarray(got.detach().cpu().double().numpy() if hasattr(got, "detach") else got,
                     dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    denom = np.abs(ref).max()
    return float(np.abs(got - ref).max() / (denom if denom > 0 else 1.0))


def cuda(t):
    return None if t is None else t.to("cuda", non_blocking=False).contiguous()


def oracle_prefill(case, heads=None, seqs=None):
    """Oracle outputs for the given heads / sequences of a PrefillCase.

    Returns (out [T, len(heads), V] for the tokens of `seqs` (others NaN),
             final [len(seqs), len(heads), K, V]).
    """
    heads = list(range(case.H)) if heads is None else list(heads)
    seqs = list(range(case.N)) if seqs is None else list(seqs)
    cu = case.cu_seqlens.tolist()
    out = np.full((case.T, len(heads), case.V), np.nan)
    finals = np.zeros((len(seqs), len(heads), case.K, case.V))
    for si, n in enumerate(seqs):
        s, e = cu[n], cu[n + 1]
        sl = slice(s, e)
        init = None if case.init_state is None else case.init_state[n:n + 1, heads]
        o, f = oracle.prefill(case.q[sl, heads], case.k[sl, heads], case.v[sl, heads],
                              case.g[sl, heads], case.beta[sl, heads], case.scale,
                              init, [0, e - s])
        out[s:e] = o
        finals[si] = f[0]
    return out, finals
