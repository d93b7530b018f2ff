"""GB300-native Kimi Delta Attention (KDA) hot path: chunked prefill and paged decode.

The computation runs in the in-tree CUDA library ``libkda.so`` (C ABI:
``include/kda.h``).  This package only allocates outputs with torch and passes
pointers; importing the op functions raises if the library is missing.

    out, final_state = chunk_prefill(q, k, v, g, beta, scale, init_state, cu_seqlens)
    out = recurrent_decode(q, k, v, g, beta, state_pool, state_idx, scale)
"""
from __future__ import annotations

__all__ = ["chunk_prefill", "chunk_prefill_paged", "chunk_prefill_from_host", "recurrent_decode",
           "prefill_workspace", "kda_chunk_prefill", "kda_chunk_prefill_ws",
           "kda_chunk_prefill_paged_ws", "kda_chunk_prefill_noalloc",
           "kda_chunk_prefill_workspace_bytes", "kda_chunk_prefill_paged", "kda_chunk_prefill_status",
           "kda_set_prefill_wait_limit", "kda_recurrent_decode", "kda_recurrent_decode_bf16_state"]


def __getattr__(name):
    if name in ("kda_chunk_prefill", "kda_chunk_prefill_ws", "kda_chunk_prefill_workspace_bytes",
                "kda_chunk_prefill_paged", "kda_chunk_prefill_paged_ws", "kda_chunk_prefill_noalloc",
                "kda_chunk_prefill_status", "kda_set_prefill_wait_limit",
                "kda_recurrent_decode", "kda_recurrent_decode_bf16_state", "KdaError"):
        from . import _native
        return getattr(_native, name)
    raise AttributeError(name)


_WORKSPACES = {}


def prefill_workspace(num_seqs, num_heads, head_dim_k, head_dim_v, dtype, device=None,
                      stream=None):
    """The device workspace ``kda_chunk_prefill_ws`` needs for these sizes (None when it
    needs none), allocated zero-filled with torch and cached per (device, stream): calls
    enqueued on one stream run one after another and can share it; calls on different
    streams get different buffers.  It only grows."""
    import torch
    from . import _native
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    n = _native.kda_chunk_prefill_workspace_bytes(num_seqs, num_heads, head_dim_k, head_dim_v, dtype)
    if n == 0:
        return None
    st = torch.cuda.current_stream(dev) if stream is None else stream
    key = (dev.index, st.cuda_stream)
    ws = _WORKSPACES.get(key)
    if ws is None or ws.numel() < n:
        ws = torch.zeros(n, dtype=torch.uint8, device=dev)
        _WORKSPACES[key] = ws
    return ws


def chunk_prefill(q, k, v, g, beta, scale=None, init_state=None, cu_seqlens=None,
                  output_final_state: bool = True, final_state=None, out_dtype=None,
                  stream=None, workspace=None, qk_l2norm: bool = False):
    """Chunked KDA prefill of packed sequences (CUDA tensors, layouts of include/kda.h).

    Returns ``(out, final_state)``; ``final_state`` is None when not requested.
    Passing ``final_state=init_state`` carries the state in place.  ``out_dtype``
    defaults to the dtype of ``v``.  ``qk_l2norm`` normalises the q and k rows inside
    the kernel.  Runs ``kda_chunk_prefill_ws`` with ``workspace``, or with the cached
    workspace of ``prefill_workspace`` when None.
    """
    import torch
    from . import _native
    T, H, K = q.shape
    V = v.shape[-1]
    if scale is None:
        scale = K ** -0.5
    if cu_seqlens is None:
        cu_seqlens = torch.tensor([0, T], dtype=torch.int32, device=q.device)
    N = cu_seqlens.numel() - 1
    out = torch.empty(v.shape, dtype=out_dtype or v.dtype, device=v.device)
    if final_state is None and output_final_state:
        final_state = torch.empty(N, H, K, V, dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = prefill_workspace(N, H, K, V, q.dtype, q.device, stream)
    _native.kda_chunk_prefill_ws(q, k, v, g, beta, scale, init_state, cu_seqlens, out,
                                 final_state, workspace, stream,
                                 _native.KDA_FLAG_QK_L2NORM if qk_l2norm else 0)
    return out, final_state


def chunk_prefill_paged(q, k, v, g, beta, state_pool, state_idx, scale=None, cu_seqlens=None,
                        out_dtype=None, stream=None, workspace=None, qk_l2norm: bool = False):
    """Chunked prefill with each sequence's state in slot ``state_idx[n]`` of
    ``state_pool`` (read as the initial state, overwritten with the final state).  Runs
    ``kda_chunk_prefill_paged_ws`` with ``workspace`` or the cached one of
    ``prefill_workspace``."""
    import torch
    from . import _native
    T, H, K = q.shape
    if scale is None:
        scale = K ** -0.5
    if cu_seqlens is None:
        cu_seqlens = torch.tensor([0, T], dtype=torch.int32, device=q.device)
    out = torch.empty(v.shape, dtype=out_dtype or v.dtype, device=v.device)
    if workspace is None:
        workspace = prefill_workspace(cu_seqlens.numel() - 1, H, K, v.shape[-1], q.dtype,
                                      q.device, stream)
    _native.kda_chunk_prefill_paged_ws(q, k, v, g, beta, scale, state_pool, state_idx, cu_seqlens,
                                       out, workspace, stream,
                                       _native.KDA_FLAG_QK_L2NORM if qk_l2norm else 0)
    return out


def recurrent_decode(q, k, v, g, beta, state_pool, state_idx, scale=None, out_dtype=None,
                     stream=None, qk_l2norm: bool = False):
    """One KDA decode step; ``state_pool`` is updated in place at ``state_idx``.

    An fp32 pool runs ``kda_recurrent_decode``; a bf16 pool runs
    ``kda_recurrent_decode_bf16_state`` (fp32 step, the stored state rounded to bf16)."""
    import torch
    from . import _native
    if scale is None:
        scale = q.shape[-1] ** -0.5
    out = torch.empty(v.shape, dtype=out_dtype or v.dtype, device=v.device)
    flags = _native.KDA_FLAG_QK_L2NORM if qk_l2norm else 0
    if state_pool.dtype == torch.bfloat16:
        _native.kda_recurrent_decode_bf16_state(q, k, v, g, beta, scale, state_pool, state_idx, out,
                                                stream, flags)
    else:
        _native.kda_recurrent_decode(q, k, v, g, beta, scale, state_pool, state_idx, out, stream, flags)
    return out


def chunk_prefill_from_host(q, k, v, g, beta, scale=None, init_state=None, cu_seqlens=None,
                            out_dtype=None, segments: int = 4, device=None, buffers=None,
                            qk_l2norm: bool = False):
    """Chunked prefill of HOST (pinned) inputs, returning HOST outputs, through the C ABI's
    ``kda_chunk_prefill_host``.

    The library cuts the packed token range into ``segments`` pieces on chunk boundaries
    and overlaps the host-to-device copy of piece s + 1 and the device-to-host copy of the
    output of piece s - 1 with the prefill of piece s; the per-sequence states are carried
    from piece to piece in place (a prefill split at any token and continued from the
    carried state equals the unsplit one).

    q, k, v, g, beta, init_state, cu_seqlens are CPU tensors (pinned memory gives
    asynchronous copies).  Returns ``(out, final_state, buffers)``: pinned CPU tensors,
    valid once the current stream of ``device`` has been synchronised, and the working
    buffers (the device buffer and the pinned outputs), which a later call with the same
    shapes and segments may pass back as ``buffers``; that call then allocates nothing and
    overwrites the returned outputs.
    """
    import torch
    from . import _native
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    T, H, K = q.shape
    V = v.shape[-1]
    if scale is None:
        scale = K ** -0.5
    if cu_seqlens is None:
        cu_seqlens = torch.tensor([0, T], dtype=torch.int32)
    N = cu_seqlens.numel() - 1
    odt = out_dtype or v.dtype
    if buffers is None:
        n = _native.kda_chunk_prefill_host_device_bytes(T, N, H, K, V, q.dtype, odt, segments)
        _native._need(n > 0, "unsupported prefill shape for kda_chunk_prefill_host")
        buffers = {
            "dev": torch.zeros(n, dtype=torch.uint8, device=device),
            "hout": torch.empty(v.shape, dtype=odt).pin_memory(),
            "hfin": torch.empty(N, H, K, V, dtype=torch.float32).pin_memory(),
        }
    hout, hfin = buffers["hout"], buffers["hfin"]
    with torch.cuda.device(device):
        _native.kda_chunk_prefill_host(q, k, v, g, beta, scale, init_state, cu_seqlens.to(torch.int32),
                                       hout, hfin, segments, buffers["dev"],
                                       torch.cuda.current_stream(device),
                                       _native.KDA_FLAG_QK_L2NORM if qk_l2norm else 0)
    return hout, hfin, buffers
