"""fp64 CPU oracle for Kimi Delta Attention (KDA) -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference legs
of ``bench.py`` may import this package.  The CUDA library never imports it, and
nothing here imports the CUDA library: the two share no code.  Inputs reach both
sides from the seeded generator module (``kimi_delta_attention_09_gb300.inputs``),
which holds none of the method's arithmetic.

Contents
--------
* ``prefill`` / ``decode``: ctypes front-end for ``kda_oracle.c``, the token-by-token
  fp64 recurrence (the plain definition of the gated delta rule with a per-key-channel
  decay; see the header of ``kda_oracle.c`` for the citations and the step order).
* ``decode_bf16_state``: the decode step on a pool stored in bf16 (the state's element
  type as a runner configuration, vllm.cpp PR #122, block B3, kda_state_dtype): the
  fp64 step of ``decode`` on the stored values, the output from the unrounded updated
  state, each updated slot then rounded to the nearest bf16 (``round_to_bf16``).
* ``l2_normalize``: the in-kernel query/key normalisation option, x / sqrt(sum x^2 +
  1e-6) over the key dimension in fp64 (the normalisation of the fused prologue that
  the prompt path of vllm.cpp PR #110 names, chunk_kda_with_fused_gate; its epsilon is
  not on the pages and is read as 1e-6); ``prefill`` / ``decode`` apply it to q and k
  first when ``qk_l2norm`` is set.
* ``chunked.prefill_chunked``: a second statement of the same definition, evaluated
  chunk by chunk (numpy, fp64), used to pin the chunk algebra that a chunked
  implementation relies on.

The shared library is compiled from ``kda_oracle.c`` with the host C compiler on
first use (``build()``), into ``oracle/_build/`` (not committed).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libkda_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``kda_oracle.c`` into a shared library; return its path."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
               "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            dp = ctypes.POINTER(ctypes.c_double)
            ip = ctypes.POINTER(ctypes.c_int64)
            i64 = ctypes.c_int64
            lib.kda_oracle_prefill.argtypes = [
                i64, i64, i64, i64, dp, dp, dp, dp, dp, ctypes.c_double,
                dp, ip, dp, dp, ctypes.c_int]
            lib.kda_oracle_prefill.restype = ctypes.c_int
            lib.kda_oracle_decode.argtypes = [
                i64, i64, i64, i64, i64, dp, dp, dp, dp, dp, ctypes.c_double,
                dp, ip, dp, ctypes.c_int]
            lib.kda_oracle_decode.restype = ctypes.c_int
            _lib = lib
    return _lib


def _f64(x) -> np.ndarray:
    if hasattr(x, "detach"):  # torch tensor on the CPU
        x = x.detach().cpu().double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _i64(x) -> np.ndarray:
    if hasattr(x, "detach"):
        x = x.detach().cpu().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.int64))


def _dptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def default_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return max(1, os.cpu_count() or 1)


QK_L2NORM_EPS = 1e-6


def l2_normalize(x) -> np.ndarray:
    """x / sqrt(sum over the last axis of x^2 + 1e-6), in fp64."""
    x = _f64(x)
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + QK_L2NORM_EPS)


def prefill(q, k, v, g, beta, scale: float, init_state=None, cu_seqlens=None,
            nthreads: int | None = None, qk_l2norm: bool = False):
    """Token-by-token fp64 prefill.

    q, k, g: [T, H, K]; v: [T, H, V]; beta: [T, H]; init_state: [N, H, K, V] or
    None (zeros); cu_seqlens: [N+1] or None (one sequence of length T).  With
    ``qk_l2norm`` the q and k rows are normalised first (``l2_normalize``).
    Returns (out [T, H, V], final_state [N, H, K, V]) as float64 arrays.
    """
    q, k, v, g, beta = (_f64(x) for x in (q, k, v, g, beta))
    if qk_l2norm:
        q, k = l2_normalize(q), l2_normalize(k)
    T, H, K = q.shape
    V = v.shape[-1]
    assert k.shape == (T, H, K) and g.shape == (T, H, K)
    assert v.shape == (T, H, V) and beta.shape == (T, H)
    cu = _i64([0, T] if cu_seqlens is None else cu_seqlens)
    N = cu.shape[0] - 1
    init = None if init_state is None else _f64(init_state)
    if init is not None:
        assert init.shape == (N, H, K, V)
    out = np.zeros((T, H, V), dtype=np.float64)
    final = np.zeros((N, H, K, V), dtype=np.float64)
    rc = _load().kda_oracle_prefill(
        N, H, K, V, _dptr(q), _dptr(k), _dptr(v), _dptr(g), _dptr(beta), float(scale),
        _dptr(init), cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
        _dptr(out), _dptr(final), int(nthreads or default_threads()))
    if rc != 0:
        raise ValueError(f"kda_oracle_prefill failed with status {rc}")
    return out, final


def decode(q, k, v, g, beta, scale: float, pool, state_idx, nthreads: int | None = None,
           qk_l2norm: bool = False):
    """One fp64 decode step for N sequences.

    q, k, g: [N, H, K]; v: [N, H, V]; beta: [N, H]; pool: [S, H, K, V] float64
    numpy array, updated IN PLACE at the slots state_idx [N].  With ``qk_l2norm`` the
    q and k rows are normalised first.  Returns out [N, H, V].
    """
    q, k, v, g, beta = (_f64(x) for x in (q, k, v, g, beta))
    if qk_l2norm:
        q, k = l2_normalize(q), l2_normalize(k)
    N, H, K = q.shape
    V = v.shape[-1]
    if not (isinstance(pool, np.ndarray) and pool.dtype == np.float64
            and pool.flags["C_CONTIGUOUS"]):
        raise TypeError("pool must be a C-contiguous float64 numpy array (updated in place)")
    S = pool.shape[0]
    assert pool.shape == (S, H, K, V)
    idx = _i64(state_idx)
    assert idx.shape == (N,)
    out = np.zeros((N, H, V), dtype=np.float64)
    rc = _load().kda_oracle_decode(
        N, S, H, K, V, _dptr(q), _dptr(k), _dptr(v), _dptr(g), _dptr(beta), float(scale),
        _dptr(pool), idx.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), _dptr(out),
        int(nthreads or default_threads()))
    if rc != 0:
        raise ValueError(f"kda_oracle_decode failed with status {rc}")
    return out


def round_to_bf16(x) -> np.ndarray:
    """Nearest bfloat16 value of each element (8 significant bits, ties to even), computed
    exactly from fp64: with |x| = m 2^e, 1/2 <= m < 1, the bf16 spacing there is 2^(e-8)
    (2^-133 below the smallest normal 2^-126); a result of 2^128 or more (past the
    largest bf16, 2^128 - 2^120) is infinite.  Returned as float64."""
    x = np.asarray(x, dtype=np.float64)
    _, e = np.frexp(x)
    e = np.maximum(e, -125)
    y = np.ldexp(np.rint(np.ldexp(x, 8 - e)), e - 8)
    return np.where(np.abs(y) >= 2.0 ** 128, np.copysign(np.inf, y), y)


def decode_bf16_state(q, k, v, g, beta, scale: float, pool, state_idx, nthreads: int | None = None,
                      qk_l2norm: bool = False):
    """One decode step on a pool stored in bf16.

    pool: [S, H, K, V] float64 numpy array holding bf16 values, updated IN PLACE at the
    slots state_idx: the step of ``decode`` in fp64, then each updated slot rounded to
    the nearest bf16.  The output is read from the unrounded updated state.  Returns
    out [N, H, V].
    """
    out = decode(q, k, v, g, beta, scale, pool, state_idx, nthreads, qk_l2norm)
    for s in np.unique(_i64(state_idx)):
        pool[s] = round_to_bf16(pool[s])
    return out
