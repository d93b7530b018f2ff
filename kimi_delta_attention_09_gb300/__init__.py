"""GB300-native Kimi Delta Attention (KDA) hot path: chunked prefill and paged decode.

The computation runs in the in-tree CUDA library ``libkda.so`` (C ABI:
``include/kda.h``).  This package only allocates outputs with torch and passes
pointers; importing the op functions raises if the library is missing.

    out, final_state = chunk_prefill(q, k, v, g, beta, scale, init_state, cu_seqlens)
    out = recurrent_decode(q, k, v, g, beta, state_pool, state_idx, scale)
"""
from __future__ import annotations

__all__ = ["chunk_prefill", "chunk_prefill_paged", "chunk_prefill_from_host", "piece_bounds",
           "piece_cu_seqlens", "recurrent_decode",
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


def piece_bounds(total_tokens: int, segments: int, chunk: int = 64):
    """Cut the packed token range [0, total_tokens) into at most ``segments`` pieces:
    bounds[s] .. bounds[s + 1] is piece s, every inner boundary a multiple of ``chunk``,
    the pieces as even in chunks as the count allows.  Host logic only."""
    T = int(total_tokens)
    nch = (T + chunk - 1) // chunk
    segments = max(1, min(int(segments), max(nch, 1)))
    return [chunk * ((nch * s) // segments) for s in range(segments)] + [T]


def piece_cu_seqlens(cu_seqlens, bounds):
    """Per piece, the cu_seqlens of every sequence clipped to the piece and counted from
    its first token (a sequence outside the piece has an empty range), as int32 rows
    padded to 16 bytes.  Host logic only."""
    import torch
    cu = torch.as_tensor(cu_seqlens).to(torch.int64)
    N = cu.numel() - 1
    row = (N + 1 + 3) // 4 * 4
    cu_seg = torch.zeros(len(bounds) - 1, row, dtype=torch.int32)
    for s_, (b0, b1) in enumerate(zip(bounds[:-1], bounds[1:])):
        cu_seg[s_, :N + 1] = (cu - b0).clamp(0, b1 - b0).to(torch.int32)
    return cu_seg


def chunk_prefill_from_host(q, k, v, g, beta, scale=None, init_state=None, cu_seqlens=None,
                            out_dtype=None, segments: int = 4, device=None, buffers=None):
    """Chunked prefill of HOST (pinned) inputs, returning HOST outputs.

    The packed token range is cut into ``segments`` pieces on chunk boundaries; the
    host-to-device copy of piece s + 1 and the device-to-host copy of the output of
    piece s - 1 overlap the prefill of piece s (three CUDA streams).  Each piece is one
    ``kda_chunk_prefill_ws`` call over the tokens of every sequence that fall in it, with
    the per-sequence states carried from piece to piece in place -- a prefill split at
    any token and continued from the carried state equals the unsplit one.

    q, k, v, g, beta, init_state, cu_seqlens are CPU tensors (pinned memory gives
    asynchronous copies).  Returns ``(out, final_state, buffers)``: pinned CPU tensors,
    valid once the current stream of ``device`` has been synchronised, and the working
    buffers (device tensors, pinned output tensors, streams), which a later call with
    the same shapes, cu_seqlens and segments may pass back as ``buffers``; that call
    then allocates nothing and overwrites the returned outputs.
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
    bounds = piece_bounds(T, segments)
    segments = len(bounds) - 1
    if buffers is None:
        # per-piece cu_seqlens, rows padded to 16 bytes (the C ABI wants 16-byte aligned pointers)
        cu_seg = piece_cu_seqlens(cu_seqlens, bounds)
        buffers = {
            "q": torch.empty(q.shape, dtype=q.dtype, device=device),
            "k": torch.empty(k.shape, dtype=k.dtype, device=device),
            "v": torch.empty(v.shape, dtype=v.dtype, device=device),
            "g": torch.empty(g.shape, dtype=g.dtype, device=device),
            "beta": torch.empty(beta.shape, dtype=beta.dtype, device=device),
            "cu": cu_seg.to(device),
            "out": torch.empty(v.shape, dtype=out_dtype or v.dtype, device=device),
            "state": torch.empty(N, H, K, V, dtype=torch.float32, device=device),
            "ws": None,
            "hout": torch.empty(v.shape, dtype=out_dtype or v.dtype).pin_memory(),
            "hfin": torch.empty(N, H, K, V, dtype=torch.float32).pin_memory(),
            "copy": torch.cuda.Stream(device), "back": torch.cuda.Stream(device),
            "events": [torch.cuda.Event() for _ in range(2 * segments)],
        }
        n_ws = _native.kda_chunk_prefill_workspace_bytes(N, H, K, V, q.dtype)
        if n_ws:
            buffers["ws"] = torch.empty(n_ws, dtype=torch.uint8, device=device)
    d = buffers
    hout, hfin = d["hout"], d["hfin"]
    main = torch.cuda.current_stream(device)
    cs, bs = d["copy"], d["back"]
    cs.wait_stream(main)
    bs.wait_stream(main)
    with torch.cuda.stream(cs):
        if init_state is None:
            d["state"].zero_()
        else:
            d["state"].copy_(init_state, non_blocking=True)
        for s, (b0, b1) in enumerate(zip(bounds[:-1], bounds[1:])):
            for name, t in (("q", q), ("k", k), ("v", v), ("g", g), ("beta", beta)):
                d[name][b0:b1].copy_(t[b0:b1], non_blocking=True)
            d["events"][s].record(cs)
    for s, (b0, b1) in enumerate(zip(bounds[:-1], bounds[1:])):
        main.wait_event(d["events"][s])
        _native.kda_chunk_prefill_ws(d["q"][b0:b1], d["k"][b0:b1], d["v"][b0:b1], d["g"][b0:b1],
                                     d["beta"][b0:b1], scale, d["state"], d["cu"][s, :N + 1],
                                     d["out"][b0:b1], d["state"], d["ws"], main)
        ev = d["events"][segments + s]
        ev.record(main)
        bs.wait_event(ev)
        with torch.cuda.stream(bs):
            hout[b0:b1].copy_(d["out"][b0:b1], non_blocking=True)
    with torch.cuda.stream(bs):
        hfin.copy_(d["state"], non_blocking=True)
    main.wait_stream(bs)
    return hout, hfin, buffers
