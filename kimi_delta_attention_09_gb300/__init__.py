"""GB300-native Kimi Delta Attention (KDA) hot path: chunked prefill and paged decode.

The computation runs in the in-tree CUDA library ``libkda.so`` (C ABI:
``include/kda.h``).  This package only allocates outputs with torch and passes
pointers; importing the op functions raises if the library is missing.

    out, final_state = chunk_prefill(q, k, v, g, beta, scale, init_state, cu_seqlens)
    out = recurrent_decode(q, k, v, g, beta, state_pool, state_idx, scale)
"""
from __future__ import annotations

__all__ = ["chunk_prefill", "chunk_prefill_paged", "recurrent_decode", "kda_chunk_prefill",
           "kda_chunk_prefill_paged", "kda_recurrent_decode"]


def __getattr__(name):
    if name in ("kda_chunk_prefill", "kda_chunk_prefill_paged", "kda_recurrent_decode",
                "KdaError"):
        from . import _native
        return getattr(_native, name)
    raise AttributeError(name)


def chunk_prefill(q, k, v, g, beta, scale=None, init_state=None, cu_seqlens=None,
                  output_final_state: bool = True, final_state=None, out_dtype=None,
                  stream=None):
    """Chunked KDA prefill of packed sequences (CUDA tensors, layouts of include/kda.h).

    Returns ``(out, final_state)``; ``final_state`` is None when not requested.
    Passing ``final_state=init_state`` carries the state in place.  ``out_dtype``
    defaults to the dtype of ``v``.
    """
    import torch
    from . import _native
    T, H, K = q.shape
    if scale is None:
        scale = K ** -0.5
    if cu_seqlens is None:
        cu_seqlens = torch.tensor([0, T], dtype=torch.int32, device=q.device)
    N = cu_seqlens.numel() - 1
    out = torch.empty(v.shape, dtype=out_dtype or v.dtype, device=v.device)
    if final_state is None and output_final_state:
        final_state = torch.empty(N, H, K, v.shape[-1], dtype=torch.float32, device=q.device)
    _native.kda_chunk_prefill(q, k, v, g, beta, scale, init_state, cu_seqlens, out,
                              final_state, stream)
    return out, final_state


def chunk_prefill_paged(q, k, v, g, beta, state_pool, state_idx, scale=None, cu_seqlens=None,
                        out_dtype=None, stream=None):
    """Chunked prefill with each sequence's state in slot ``state_idx[n]`` of
    ``state_pool`` (read as the initial state, overwritten with the final state)."""
    import torch
    from . import _native
    T, H, K = q.shape
    if scale is None:
        scale = K ** -0.5
    if cu_seqlens is None:
        cu_seqlens = torch.tensor([0, T], dtype=torch.int32, device=q.device)
    out = torch.empty(v.shape, dtype=out_dtype or v.dtype, device=v.device)
    _native.kda_chunk_prefill_paged(q, k, v, g, beta, scale, state_pool, state_idx, cu_seqlens,
                                    out, stream)
    return out


def recurrent_decode(q, k, v, g, beta, state_pool, state_idx, scale=None, out_dtype=None,
                     stream=None):
    """One KDA decode step; ``state_pool`` is updated in place at ``state_idx``."""
    import torch
    from . import _native
    if scale is None:
        scale = q.shape[-1] ** -0.5
    out = torch.empty(v.shape, dtype=out_dtype or v.dtype, device=v.device)
    _native.kda_recurrent_decode(q, k, v, g, beta, scale, state_pool, state_idx, out, stream)
    return out
