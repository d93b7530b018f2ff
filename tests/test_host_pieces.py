"""Host logic of the host-to-host prefill (chunk_prefill_from_host): how the packed token
range is cut into pieces and how each sequence is clipped to a piece, checked on the CPU
against brute force and, through the oracle, against the unsplit prefill."""
import numpy as np
import pytest
import torch

import oracle
from kimi_delta_attention_09_gb300 import inputs, piece_bounds, piece_cu_seqlens


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
