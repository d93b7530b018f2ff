"""ctypes binding of the in-tree ``libkda.so`` (the C ABI of ``include/kda.h``).

Argument marshalling only: every step of the computation runs in the CUDA
library.  There is no fallback of any kind; if the library is missing or fails to
load, importing this module raises.
"""
from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libkda.so")

KDA_OK = 0
KDA_ERR_INVALID_ARG = -1
KDA_ERR_UNSUPPORTED = -2
KDA_ERR_ALIAS = -3
KDA_ERR_CUDA = -4
KDA_ERR_TIMEOUT = -5
KDA_DTYPE_F32 = 0
KDA_DTYPE_BF16 = 1
KDA_FLAG_QK_L2NORM = 1
KDA_CONV_ACT_NONE = 0
KDA_CONV_ACT_SILU = 1
ABI_VERSION = 5

EXPORTED = ("kda_abi_version", "kda_status_string", "kda_last_cuda_error",
            "kda_chunk_prefill", "kda_chunk_prefill_workspace_bytes", "kda_chunk_prefill_ws",
            "kda_chunk_prefill_noalloc", "kda_chunk_prefill_paged_ws",
            "kda_chunk_prefill_paged", "kda_chunk_prefill_status", "kda_set_prefill_wait_limit",
            "kda_recurrent_decode", "kda_recurrent_decode_bf16_state", "kda_causal_conv1d_fwd",
            "kda_causal_conv1d_update", "kda_chunk_prefill_host_device_bytes",
            "kda_chunk_prefill_host")
KDA_HOST_MAX_PIECES = 16


class KdaError(RuntimeError):
    def __init__(self, fn: str, status: int, detail: str = ""):
        self.status = status
        super().__init__(f"{fn} failed: {status_string(status)} ({status}){detail}")


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            f"{LIB_PATH} is not built; run `python -m kimi_delta_attention_09_gb300.build` "
            "(the KDA ops have no non-CUDA implementation)")
    lib = ctypes.CDLL(LIB_PATH)
    vp, f32, i32, i64 = ctypes.c_void_p, ctypes.c_float, ctypes.c_int32, ctypes.c_int64
    lib.kda_abi_version.argtypes = []
    lib.kda_abi_version.restype = ctypes.c_int
    lib.kda_status_string.argtypes = [ctypes.c_int]
    lib.kda_status_string.restype = ctypes.c_char_p
    lib.kda_last_cuda_error.argtypes = []
    lib.kda_last_cuda_error.restype = ctypes.c_int
    lib.kda_chunk_prefill.argtypes = [vp, vp, vp, vp, vp, f32, vp, vp, vp, vp,
                                      i64, i32, i32, i32, i32, i32, i32, i32, vp]
    lib.kda_chunk_prefill.restype = ctypes.c_int
    lib.kda_chunk_prefill_workspace_bytes.argtypes = [i32, i32, i32, i32, i32]
    lib.kda_chunk_prefill_workspace_bytes.restype = ctypes.c_size_t
    lib.kda_chunk_prefill_ws.argtypes = [vp, vp, vp, vp, vp, f32, vp, vp, vp, vp,
                                         i64, i32, i32, i32, i32, i32, i32, vp, ctypes.c_size_t, i32, vp]
    lib.kda_chunk_prefill_ws.restype = ctypes.c_int
    lib.kda_chunk_prefill_noalloc.argtypes = [vp, vp, vp, vp, vp, f32, vp, vp, vp, vp,
                                              i64, i32, i32, i32, i32, i32, i32, vp]
    lib.kda_chunk_prefill_noalloc.restype = ctypes.c_int
    lib.kda_chunk_prefill_paged.argtypes = [vp, vp, vp, vp, vp, f32, vp, vp, vp, vp,
                                            i64, i32, i32, i32, i32, i32, i32, i32, i32, vp]
    lib.kda_chunk_prefill_paged.restype = ctypes.c_int
    lib.kda_chunk_prefill_paged_ws.argtypes = [vp, vp, vp, vp, vp, f32, vp, vp, vp, vp,
                                               i64, i32, i32, i32, i32, i32, i32, i32, vp,
                                               ctypes.c_size_t, i32, vp]
    lib.kda_chunk_prefill_paged_ws.restype = ctypes.c_int
    lib.kda_chunk_prefill_host_device_bytes.argtypes = [i64, i32, i32, i32, i32, i32, i32, i32]
    lib.kda_chunk_prefill_host_device_bytes.restype = ctypes.c_size_t
    lib.kda_chunk_prefill_host.argtypes = [vp, vp, vp, vp, vp, f32, vp, vp, vp, vp,
                                           i64, i32, i32, i32, i32, i32, i32, i32, vp,
                                           ctypes.c_size_t, i32, vp]
    lib.kda_chunk_prefill_host.restype = ctypes.c_int
    lib.kda_chunk_prefill_status.argtypes = [vp, vp]
    lib.kda_chunk_prefill_status.restype = ctypes.c_int
    lib.kda_set_prefill_wait_limit.argtypes = [ctypes.c_uint64]
    lib.kda_set_prefill_wait_limit.restype = None
    lib.kda_recurrent_decode.argtypes = [vp, vp, vp, vp, vp, f32, vp, vp, vp,
                                         i32, i32, i32, i32, i32, i32, i32, i32, vp]
    lib.kda_recurrent_decode.restype = ctypes.c_int
    lib.kda_recurrent_decode_bf16_state.argtypes = [vp, vp, vp, vp, vp, f32, vp, vp, vp,
                                                    i32, i32, i32, i32, i32, i32, i32, i32, vp]
    lib.kda_recurrent_decode_bf16_state.restype = ctypes.c_int
    lib.kda_causal_conv1d_fwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, i64, i32, i32, i32, i32,
                                          i32, i32, i32, vp]
    lib.kda_causal_conv1d_fwd.restype = ctypes.c_int
    lib.kda_causal_conv1d_update.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32,
                                             i32, vp]
    lib.kda_causal_conv1d_update.restype = ctypes.c_int
    if lib.kda_abi_version() != ABI_VERSION:
        raise RuntimeError(f"libkda.so ABI {lib.kda_abi_version()} != expected {ABI_VERSION}")
    return lib


lib = _load()


def status_string(status: int) -> str:
    return lib.kda_status_string(int(status)).decode()


def _check(fn: str, status: int) -> None:
    if status != KDA_OK:
        detail = f", cudaError {lib.kda_last_cuda_error()}" if status == KDA_ERR_CUDA else ""
        raise KdaError(fn, status, detail)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.bfloat16:
        return KDA_DTYPE_BF16
    if t.dtype == torch.float32:
        return KDA_DTYPE_F32
    raise ValueError(f"unsupported dtype {t.dtype} (bf16 or fp32)")


def _stream_handle(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _need(cond: bool, msg: str):
    if not cond:
        raise ValueError(msg)


def kda_chunk_prefill(q, k, v, g, beta, scale, init_state, cu_seqlens, out, final_state,
                      stream=None, flags=0) -> None:
    """Enqueue ``kda_chunk_prefill`` on ``stream`` (default: torch's current stream).

    Tensors are CUDA tensors laid out as include/kda.h states; shapes and dtypes are
    read from them: q [T, H, K], v [T, H, V], cu_seqlens [N + 1] int32; the dtype of
    ``out`` (fp32 or bf16) selects the output element type.
    """
    T, H, K = q.shape
    V = v.shape[-1]
    N = cu_seqlens.numel() - 1
    for name, t in (("q", q), ("k", k), ("v", v), ("g", g), ("beta", beta), ("out", out),
                    ("cu_seqlens", cu_seqlens), ("init_state", init_state),
                    ("final_state", final_state)):
        if t is not None:
            _need(t.is_cuda and t.is_contiguous(), f"{name} must be a contiguous CUDA tensor")
    _need(k.shape == q.shape and g.shape == q.shape, "q, k, g must be [T, H, K]")
    _need(v.shape[:2] == (T, H) and out.shape == v.shape, "v, out must be [T, H, V]")
    _need(beta.shape == (T, H), "beta must be [T, H]")
    _need(k.dtype == q.dtype and v.dtype == q.dtype, "q, k, v must share one dtype")
    import torch
    _need(g.dtype == torch.float32 and beta.dtype == torch.float32, "g, beta must be fp32")
    _need(cu_seqlens.dtype == torch.int32, "cu_seqlens must be int32")
    for s in (init_state, final_state):
        if s is not None:
            _need(s.dtype == torch.float32 and tuple(s.shape) == (N, H, K, V),
                  "states must be fp32 [N, H, K, V]")
    rc = lib.kda_chunk_prefill(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale),
                               _ptr(init_state), _ptr(cu_seqlens), _ptr(out), _ptr(final_state),
                               T, N, H, K, V, _dtype_code(q), _dtype_code(out), int(flags),
                               _stream_handle(stream))
    _check("kda_chunk_prefill", rc)


def kda_chunk_prefill_workspace_bytes(num_seqs: int, num_heads: int, head_dim_k: int,
                                      head_dim_v: int, dtype) -> int:
    """Workspace bytes ``kda_chunk_prefill_ws`` needs (``dtype``: a torch dtype of q/k/v).
    The workspace must be zero-filled before its first use (``torch.zeros``)."""
    import torch
    code = KDA_DTYPE_BF16 if dtype == torch.bfloat16 else KDA_DTYPE_F32
    return int(lib.kda_chunk_prefill_workspace_bytes(int(num_seqs), int(num_heads), int(head_dim_k),
                                                     int(head_dim_v), code))


def kda_chunk_prefill_ws(q, k, v, g, beta, scale, init_state, cu_seqlens, out, final_state,
                         workspace, stream=None, flags=0) -> None:
    """Enqueue ``kda_chunk_prefill_ws``: as ``kda_chunk_prefill`` plus ``workspace``, a
    contiguous CUDA tensor (any dtype) of at least ``kda_chunk_prefill_workspace_bytes``
    bytes, or None when that is 0."""
    T, H, K = q.shape
    V = v.shape[-1]
    N = cu_seqlens.numel() - 1
    for name, t in (("q", q), ("k", k), ("v", v), ("g", g), ("beta", beta), ("out", out),
                    ("cu_seqlens", cu_seqlens), ("init_state", init_state),
                    ("final_state", final_state), ("workspace", workspace)):
        if t is not None:
            _need(t.is_cuda and t.is_contiguous(), f"{name} must be a contiguous CUDA tensor")
    _need(k.shape == q.shape and g.shape == q.shape, "q, k, g must be [T, H, K]")
    _need(v.shape[:2] == (T, H) and out.shape == v.shape, "v, out must be [T, H, V]")
    _need(beta.shape == (T, H), "beta must be [T, H]")
    _need(k.dtype == q.dtype and v.dtype == q.dtype, "q, k, v must share one dtype")
    import torch
    _need(g.dtype == torch.float32 and beta.dtype == torch.float32, "g, beta must be fp32")
    _need(cu_seqlens.dtype == torch.int32, "cu_seqlens must be int32")
    for s in (init_state, final_state):
        if s is not None:
            _need(s.dtype == torch.float32 and tuple(s.shape) == (N, H, K, V),
                  "states must be fp32 [N, H, K, V]")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = lib.kda_chunk_prefill_ws(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale),
                                  _ptr(init_state), _ptr(cu_seqlens), _ptr(out), _ptr(final_state),
                                  T, N, H, K, V, _dtype_code(q), _dtype_code(out), _ptr(workspace),
                                  ws_bytes, int(flags), _stream_handle(stream))
    _check("kda_chunk_prefill_ws", rc)


def kda_chunk_prefill_host_device_bytes(T: int, N: int, H: int, K: int, V: int, dtype,
                                        out_dtype, pieces: int) -> int:
    """Device bytes ``kda_chunk_prefill_host`` needs (0: unsupported arguments)."""
    code = lambda d: KDA_DTYPE_BF16 if "bfloat16" in str(d) else KDA_DTYPE_F32
    return int(lib.kda_chunk_prefill_host_device_bytes(int(T), int(N), int(H), int(K), int(V),
                                                       code(dtype), code(out_dtype), int(pieces)))


def kda_chunk_prefill_host(q, k, v, g, beta, scale, init_state, cu_seqlens, out, final_state,
                           pieces, device_buffer, stream=None, flags=0) -> None:
    """Enqueue ``kda_chunk_prefill_host``: q, k, v, g, beta, cu_seqlens, init_state (or None)
    and out, final_state (or None) are contiguous CPU tensors (page-locked for asynchronous
    copies) in the layouts of ``kda_chunk_prefill``; ``device_buffer`` is a contiguous CUDA
    tensor of at least ``kda_chunk_prefill_host_device_bytes`` bytes, zero-filled before its
    first use.  The outputs are valid once ``stream`` has been synchronised."""
    T, H, K = q.shape
    V = v.shape[-1]
    N = cu_seqlens.numel() - 1
    for name, t in (("q", q), ("k", k), ("v", v), ("g", g), ("beta", beta), ("out", out),
                    ("cu_seqlens", cu_seqlens), ("init_state", init_state),
                    ("final_state", final_state)):
        if t is not None:
            _need(not t.is_cuda and t.is_contiguous(), f"{name} must be a contiguous CPU tensor")
    _need(device_buffer.is_cuda and device_buffer.is_contiguous(),
          "device_buffer must be a contiguous CUDA tensor")
    _need(k.shape == q.shape and g.shape == q.shape, "q, k, g must be [T, H, K]")
    _need(v.shape[:2] == (T, H) and out.shape == v.shape, "v, out must be [T, H, V]")
    _need(beta.shape == (T, H), "beta must be [T, H]")
    _need(k.dtype == q.dtype and v.dtype == q.dtype, "q, k, v must share one dtype")
    import torch
    _need(g.dtype == torch.float32 and beta.dtype == torch.float32, "g, beta must be fp32")
    _need(cu_seqlens.dtype == torch.int32, "cu_seqlens must be int32")
    for s in (init_state, final_state):
        if s is not None:
            _need(s.dtype == torch.float32 and tuple(s.shape) == (N, H, K, V),
                  "states must be fp32 [N, H, K, V]")
    nbytes = device_buffer.numel() * device_buffer.element_size()
    rc = lib.kda_chunk_prefill_host(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale),
                                    _ptr(init_state), _ptr(cu_seqlens), _ptr(out), _ptr(final_state),
                                    T, N, H, K, V, _dtype_code(q), _dtype_code(out), int(pieces),
                                    _ptr(device_buffer), nbytes, int(flags), _stream_handle(stream))
    _check("kda_chunk_prefill_host", rc)


def kda_chunk_prefill_noalloc(q, k, v, g, beta, scale, init_state, cu_seqlens, out, final_state,
                              stream=None) -> None:
    """Enqueue ``kda_chunk_prefill_noalloc``: the prefill on the library's own static
    device scratch (one call in flight per device at a time)."""
    T, H, K = q.shape
    V = v.shape[-1]
    N = cu_seqlens.numel() - 1
    for name, t in (("q", q), ("k", k), ("v", v), ("g", g), ("beta", beta), ("out", out),
                    ("cu_seqlens", cu_seqlens), ("init_state", init_state),
                    ("final_state", final_state)):
        if t is not None:
            _need(t.is_cuda and t.is_contiguous(), f"{name} must be a contiguous CUDA tensor")
    _need(k.shape == q.shape and g.shape == q.shape, "q, k, g must be [T, H, K]")
    _need(v.shape[:2] == (T, H) and out.shape == v.shape, "v, out must be [T, H, V]")
    _need(beta.shape == (T, H), "beta must be [T, H]")
    _need(k.dtype == q.dtype and v.dtype == q.dtype, "q, k, v must share one dtype")
    import torch
    _need(g.dtype == torch.float32 and beta.dtype == torch.float32, "g, beta must be fp32")
    _need(cu_seqlens.dtype == torch.int32, "cu_seqlens must be int32")
    for s in (init_state, final_state):
        if s is not None:
            _need(s.dtype == torch.float32 and tuple(s.shape) == (N, H, K, V),
                  "states must be fp32 [N, H, K, V]")
    rc = lib.kda_chunk_prefill_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale),
                                       _ptr(init_state), _ptr(cu_seqlens), _ptr(out), _ptr(final_state),
                                       T, N, H, K, V, _dtype_code(q), _dtype_code(out),
                                       _stream_handle(stream))
    _check("kda_chunk_prefill_noalloc", rc)


def kda_chunk_prefill_paged(q, k, v, g, beta, scale, state_pool, state_idx, cu_seqlens, out,
                            stream=None, flags=0) -> None:
    """Enqueue ``kda_chunk_prefill_paged``: as ``kda_chunk_prefill`` with sequence n's
    initial and final state in slot ``state_idx[n]`` of ``state_pool`` [S, H, K, V]."""
    T, H, K = q.shape
    V = v.shape[-1]
    N = cu_seqlens.numel() - 1
    S = state_pool.shape[0]
    for name, t in (("q", q), ("k", k), ("v", v), ("g", g), ("beta", beta), ("out", out),
                    ("cu_seqlens", cu_seqlens), ("state_pool", state_pool),
                    ("state_idx", state_idx)):
        _need(t.is_cuda and t.is_contiguous(), f"{name} must be a contiguous CUDA tensor")
    import torch
    _need(k.shape == q.shape and g.shape == q.shape, "q, k, g must be [T, H, K]")
    _need(v.shape[:2] == (T, H) and out.shape == v.shape, "v, out must be [T, H, V]")
    _need(beta.shape == (T, H), "beta must be [T, H]")
    _need(k.dtype == q.dtype and v.dtype == q.dtype, "q, k, v must share one dtype")
    _need(g.dtype == torch.float32 and beta.dtype == torch.float32, "g, beta must be fp32")
    _need(cu_seqlens.dtype == torch.int32, "cu_seqlens must be int32")
    _need(tuple(state_pool.shape[1:]) == (H, K, V) and state_pool.dtype == torch.float32,
          "state_pool must be fp32 [S, H, K, V]")
    _need(state_idx.dtype == torch.int32 and state_idx.numel() == N, "state_idx must be int32 [N]")
    rc = lib.kda_chunk_prefill_paged(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale),
                                     _ptr(state_pool), _ptr(state_idx), _ptr(cu_seqlens),
                                     _ptr(out), T, N, S, H, K, V, _dtype_code(q), _dtype_code(out),
                                     int(flags), _stream_handle(stream))
    _check("kda_chunk_prefill_paged", rc)


def kda_chunk_prefill_paged_ws(q, k, v, g, beta, scale, state_pool, state_idx, cu_seqlens, out,
                               workspace, stream=None, flags=0) -> None:
    """Enqueue ``kda_chunk_prefill_paged_ws``: ``kda_chunk_prefill_paged`` plus ``workspace``
    (as for ``kda_chunk_prefill_ws``)."""
    T, H, K = q.shape
    V = v.shape[-1]
    N = cu_seqlens.numel() - 1
    S = state_pool.shape[0]
    for name, t in (("q", q), ("k", k), ("v", v), ("g", g), ("beta", beta), ("out", out),
                    ("cu_seqlens", cu_seqlens), ("state_pool", state_pool),
                    ("state_idx", state_idx), ("workspace", workspace)):
        if t is not None:
            _need(t.is_cuda and t.is_contiguous(), f"{name} must be a contiguous CUDA tensor")
    import torch
    _need(k.shape == q.shape and g.shape == q.shape, "q, k, g must be [T, H, K]")
    _need(v.shape[:2] == (T, H) and out.shape == v.shape, "v, out must be [T, H, V]")
    _need(beta.shape == (T, H), "beta must be [T, H]")
    _need(k.dtype == q.dtype and v.dtype == q.dtype, "q, k, v must share one dtype")
    _need(g.dtype == torch.float32 and beta.dtype == torch.float32, "g, beta must be fp32")
    _need(cu_seqlens.dtype == torch.int32, "cu_seqlens must be int32")
    _need(tuple(state_pool.shape[1:]) == (H, K, V) and state_pool.dtype == torch.float32,
          "state_pool must be fp32 [S, H, K, V]")
    _need(state_idx.dtype == torch.int32 and state_idx.numel() == N, "state_idx must be int32 [N]")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = lib.kda_chunk_prefill_paged_ws(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale),
                                        _ptr(state_pool), _ptr(state_idx), _ptr(cu_seqlens),
                                        _ptr(out), T, N, S, H, K, V, _dtype_code(q), _dtype_code(out),
                                        _ptr(workspace), ws_bytes, int(flags), _stream_handle(stream))
    _check("kda_chunk_prefill_paged_ws", rc)


def kda_chunk_prefill_status(workspace=None, stream=None) -> int:
    """Synchronise ``stream`` and return (and clear) the device status of the last
    tensor-core prefill on ``workspace`` (None: the library's scratch): ``KDA_OK`` or
    ``KDA_ERR_TIMEOUT``.  Raises on a CUDA error."""
    rc = lib.kda_chunk_prefill_status(_ptr(workspace), _stream_handle(stream))
    if rc not in (KDA_OK, KDA_ERR_TIMEOUT):
        _check("kda_chunk_prefill_status", rc)
    return int(rc)


def kda_set_prefill_wait_limit(nanoseconds: int) -> None:
    """Limit of every wait inside later tensor-core prefill launches (0: the default)."""
    lib.kda_set_prefill_wait_limit(int(nanoseconds))


def _decode(fn, q, k, v, g, beta, scale, state_pool, state_idx, out, pool_dtype, stream, flags):
    N, H, K = q.shape
    V = v.shape[-1]
    S = state_pool.shape[0]
    for name, t in (("q", q), ("k", k), ("v", v), ("g", g), ("beta", beta), ("out", out),
                    ("state_pool", state_pool), ("state_idx", state_idx)):
        _need(t.is_cuda and t.is_contiguous(), f"{name} must be a contiguous CUDA tensor")
    import torch
    _need(k.shape == q.shape and g.shape == q.shape, "q, k, g must be [N, H, K]")
    _need(v.shape[:2] == (N, H) and out.shape == v.shape, "v, out must be [N, H, V]")
    _need(beta.shape == (N, H), "beta must be [N, H]")
    _need(tuple(state_pool.shape[1:]) == (H, K, V) and state_pool.dtype == pool_dtype,
          f"state_pool must be {pool_dtype} [S, H, K, V]")
    _need(state_idx.dtype == torch.int32 and state_idx.numel() == N, "state_idx must be int32 [N]")
    _need(k.dtype == q.dtype and v.dtype == q.dtype, "q, k, v must share one dtype")
    _need(g.dtype == torch.float32 and beta.dtype == torch.float32, "g, beta must be fp32")
    rc = getattr(lib, fn)(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale),
                          _ptr(state_pool), _ptr(state_idx), _ptr(out),
                          N, S, H, K, V, _dtype_code(q), _dtype_code(out), int(flags),
                          _stream_handle(stream))
    _check(fn, rc)


def kda_recurrent_decode(q, k, v, g, beta, scale, state_pool, state_idx, out,
                         stream=None, flags=0) -> None:
    """Enqueue ``kda_recurrent_decode``: q [N, H, K], v [N, H, V], fp32 pool [S, H, K, V]."""
    import torch
    _decode("kda_recurrent_decode", q, k, v, g, beta, scale, state_pool, state_idx, out,
            torch.float32, stream, flags)


def kda_recurrent_decode_bf16_state(q, k, v, g, beta, scale, state_pool, state_idx, out,
                                    stream=None, flags=0) -> None:
    """Enqueue ``kda_recurrent_decode_bf16_state``: the same step on a bf16 pool [S, H, K, V]."""
    import torch
    _decode("kda_recurrent_decode_bf16_state", q, k, v, g, beta, scale, state_pool, state_idx, out,
            torch.bfloat16, stream, flags)


def _conv_checks(x, weight, bias, conv_state, state_idx, out):
    import torch
    for name, t in (("x", x), ("weight", weight), ("bias", bias), ("conv_state", conv_state),
                    ("state_idx", state_idx), ("out", out)):
        if t is not None:
            _need(t.is_cuda and t.is_contiguous(), f"{name} must be a contiguous CUDA tensor")
    D, W = weight.shape
    _need(weight.dtype == torch.float32, "weight must be fp32 [D, W]")
    _need(x.shape[-1] == D and out.shape == x.shape, "x, out must be [rows, D]")
    _need(bias is None or (bias.dtype == torch.float32 and bias.shape == (D,)), "bias must be fp32 [D]")
    if conv_state is not None:
        _need(conv_state.dtype == x.dtype and tuple(conv_state.shape[1:]) == (W - 1, D),
              "conv_state must be [S, W - 1, D] of x's dtype")
        _need(state_idx is not None and state_idx.dtype == torch.int32, "state_idx must be int32 [N]")
    return D, W


def kda_causal_conv1d_fwd(x, weight, bias, conv_state, state_idx, cu_seqlens, out,
                          activation=KDA_CONV_ACT_NONE, stream=None) -> None:
    """Enqueue ``kda_causal_conv1d_fwd``: x [T, D], weight [D, W] fp32, bias [D] or None,
    conv_state [S, W - 1, D] (x's dtype, updated in place) or None, state_idx [N] int32,
    cu_seqlens [N + 1] int32, out [T, D] (its dtype selects the output element type)."""
    import torch
    D, W = _conv_checks(x, weight, bias, conv_state, state_idx, out)
    _need(cu_seqlens.is_cuda and cu_seqlens.dtype == torch.int32, "cu_seqlens must be int32 on CUDA")
    N = cu_seqlens.numel() - 1
    S = 0 if conv_state is None else conv_state.shape[0]
    rc = lib.kda_causal_conv1d_fwd(_ptr(x), _ptr(weight), _ptr(bias), _ptr(conv_state),
                                   _ptr(state_idx), _ptr(cu_seqlens), _ptr(out), x.shape[0], N, S,
                                   D, W, _dtype_code(x), _dtype_code(out), int(activation),
                                   _stream_handle(stream))
    _check("kda_causal_conv1d_fwd", rc)


def kda_causal_conv1d_update(x, weight, bias, conv_state, state_idx, out,
                             activation=KDA_CONV_ACT_NONE, stream=None) -> None:
    """Enqueue ``kda_causal_conv1d_update``: one token per sequence, x [N, D]."""
    D, W = _conv_checks(x, weight, bias, conv_state, state_idx, out)
    S = 0 if conv_state is None else conv_state.shape[0]
    rc = lib.kda_causal_conv1d_update(_ptr(x), _ptr(weight), _ptr(bias), _ptr(conv_state),
                                      _ptr(state_idx), _ptr(out), x.shape[0], S, D, W,
                                      _dtype_code(x), _dtype_code(out), int(activation),
                                      _stream_handle(stream))
    _check("kda_causal_conv1d_update", rc)
