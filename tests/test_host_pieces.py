"""The host-to-host prefill (kda_chunk_prefill_host): the rule by which the library cuts
the packed token range into pieces and clips each sequence to a piece, restated here and
checked on the CPU against brute force and, through the oracle, against the unsplit
prefill; and the entry point's argument checks, which run before any CUDA call."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from kimi_delta_attention_09_gb300 import inputs


def piece_bounds(total_tokens: int, segments: int, chunk: int = 64):
    """At most ``segments`` pieces, inner bounds on multiples of ``chunk``, the pieces as
    even in chunks as the count allows (the library's rule)."""
    T = int(total_tokens)
    nch = (T + chunk - 1) // chunk
    segments = max(1, min(int(segments), max(nch, 1)))
    return [chunk * ((nch * s) // segments) for s in range(segments)] + [T]


def piece_cu_seqlens(cu_seqlens, bounds):
    """Per piece, every sequence's range clipped to the piece and counted from its first
    token (empty outside it), int32 rows padded to 16 bytes (the library's rule)."""
    cu = torch.as_tensor(cu_seqlens).to(torch.int64)
    N = cu.numel() - 1
    row = (N + 1 + 3) // 4 * 4
    cu_seg = torch.zeros(len(bounds) - 1, row, dtype=torch.int32)
    for s_, (b0, b1) in enumerate(zip(bounds[:-1], bounds[1:])):
        cu_seg[s_, :N + 1] = (cu - b0).clamp(0, b1 - b0).to(torch.int32)
    return cu_seg


@pytest.mark.parametrize("T,segments", [(0, 4), (1, 4), (64, 4), (65, 4), (4096, 4), (4096, 7),
                                        (1000, 1), (1000, 100), (37517, 4)])
def test_piece_bounds_cover_the_range_on_chunk_boundaries(T, segments):
    b = piece_bounds(T, segments)
    nch = (T + 63) // 64
    assert b[0] == 0 and b[-1] == T
    assert 1 <= len(b) - 1 <= max(1, min(segments, nch))
    assert all(x <= y for x, y in zip(b, b[1:]))
    assert all(x % 64 == 0 for x in b[:-1])
    if T:
        sizes = [(y - x + 63) // 64 for x, y in zip(b, b[1:])]
        assert max(sizes) - min(sizes) <= 1 and all(s > 0 for s in sizes)


def test_piece_cu_seqlens_is_each_sequence_clipped_to_each_piece():
    rng = np.random.default_rng(5)
    lengths = [0, 1, 63, 64, 65, 300, 0, 129, 7]
    cu = np.concatenate([[0], np.cumsum(lengths)])
    T = int(cu[-1])
    for segments in (1, 2, 3, 5, 8):
        b = piece_bounds(T, segments)
        seg = piece_cu_seqlens(torch.tensor(cu, dtype=torch.int32), b)
        assert seg.dtype == torch.int32 and (seg.shape[1] * 4) % 16 == 0
        for s, (b0, b1) in enumerate(zip(b, b[1:])):
            for n in range(len(lengths)):
                lo, hi = max(cu[n], b0), min(cu[n + 1], b1)
                want = (lo - b0, hi - b0) if lo < hi else None
                got = (int(seg[s, n]), int(seg[s, n + 1]))
                if want is None:
                    assert got[0] == got[1]
                else:
                    assert got == want
    del rng


def test_pieces_with_carried_states_equal_the_unsplit_prefill():
    """The oracle run piece by piece on the planned cu_seqlens, each sequence's state
    carried from piece to piece, equals the oracle run on the whole range."""
    case = inputs.prefill_case([5, 130, 1, 200, 64, 77], H=2, K=8, V=8, dtype="f32", seed=9,
                               init_std=0.05)
    ref_out, ref_fin = oracle.prefill(case.q, case.k, case.v, case.g, case.beta, case.scale,
                                      case.init_state, case.cu_seqlens)
    b = piece_bounds(case.T, 3)
    seg = piece_cu_seqlens(case.cu_seqlens, b)
    N = case.N
    state = case.init_state.double().numpy().copy()
    out = np.zeros_like(ref_out)
    for s, (b0, b1) in enumerate(zip(b, b[1:])):
        sl = slice(b0, b1)
        o, state = oracle.prefill(case.q[sl], case.k[sl], case.v[sl], case.g[sl], case.beta[sl],
                                  case.scale, state, seg[s, :N + 1])
        out[b0:b1] = o
    assert np.abs(out - ref_out).max() <= 1e-12 * np.abs(ref_out).max()
    assert np.abs(state - ref_fin).max() <= 1e-12 * np.abs(ref_fin).max()


def _host_call(native, pieces=4, flags=0, device_buffer=None, nbytes=0, out=None):
    case = inputs.prefill_case([70, 30], H=2, K=128, V=128, dtype="bf16", seed=3)
    out = torch.empty(case.T, 2, 128, dtype=torch.float32) if out is None else out
    vp = lambda t: ctypes.c_void_p(t.data_ptr())
    return native.lib.kda_chunk_prefill_host(
        vp(case.q), vp(case.k), vp(case.v), vp(case.g), vp(case.beta), case.scale, None,
        vp(case.cu_seqlens), vp(out), None, case.T, case.N, 2, 128, 128,
        native.KDA_DTYPE_BF16, native.KDA_DTYPE_F32, pieces, device_buffer, nbytes, flags, None)


def test_host_entry_rejects_bad_arguments_before_any_cuda_call():
    from kimi_delta_attention_09_gb300 import _native as native
    assert _host_call(native, pieces=0) == native.KDA_ERR_INVALID_ARG
    assert _host_call(native, pieces=native.KDA_HOST_MAX_PIECES + 1) == native.KDA_ERR_INVALID_ARG
    assert _host_call(native, flags=2) == native.KDA_ERR_INVALID_ARG
    assert _host_call(native, device_buffer=None) == native.KDA_ERR_INVALID_ARG
    fake = ctypes.c_void_p(1 << 20)   # never dereferenced: too small
    assert _host_call(native, device_buffer=fake, nbytes=16) == native.KDA_ERR_INVALID_ARG


def test_host_device_bytes_cover_every_region():
    from kimi_delta_attention_09_gb300 import _native as native
    T, N, H = 4096, 3, 32
    n = native.kda_chunk_prefill_host_device_bytes(T, N, H, 128, 128, torch.bfloat16, torch.float32, 4)
    ws = native.kda_chunk_prefill_workspace_bytes(N, H, 128, 128, torch.bfloat16)
    rows = T * H
    least = ws + rows * 128 * 2 * 3 + rows * 128 * 4 + rows * 4 + rows * 128 * 4 + N * H * 128 * 128 * 4
    assert least <= n <= least + 12 * 256 + 4 * 4 * (N + 4)
    assert n % 256 == 0
    assert native.kda_chunk_prefill_host_device_bytes(T, N, H, 96, 128, torch.bfloat16, torch.float32, 4) == 0
    assert native.kda_chunk_prefill_host_device_bytes(T, N, H, 128, 128, torch.bfloat16, torch.float32, 0) == 0


def test_host_entry_alias_rules():
    """A host output overlapping an input is rejected before any CUDA call; the final state
    may be the initial state's own buffer (the in-place carry), as on the device."""
    from kimi_delta_attention_09_gb300 import _native as native
    case = inputs.prefill_case([70, 30], H=2, K=128, V=128, dtype="bf16", seed=3, init_std=0.02)
    vp = lambda t: ctypes.c_void_p(t.data_ptr())
    state = case.init_state.clone()
    out = torch.empty(case.T, 2, 128, dtype=torch.float32)

    def call(out_t, init_t, fin_t):
        return native.lib.kda_chunk_prefill_host(
            vp(case.q), vp(case.k), vp(case.v), vp(case.g), vp(case.beta), case.scale,
            None if init_t is None else vp(init_t), vp(case.cu_seqlens), vp(out_t),
            None if fin_t is None else vp(fin_t), case.T, case.N, 2, 128, 128,
            native.KDA_DTYPE_BF16, native.KDA_DTYPE_F32, 4, None, 0, 0, None)

    # out over q: alias; final over q: alias
    assert call(case.q, None, None) == native.KDA_ERR_ALIAS
    assert call(out, None, case.q.view(torch.float32)) == native.KDA_ERR_ALIAS
    # the in-place carry passes the alias rules and stops at the (missing) device buffer
    assert call(out, state, state) == native.KDA_ERR_INVALID_ARG
