"""Paged recurrent decode over a bf16 state pool (kda_recurrent_decode_bf16_state) on
the GPU against the fp64 oracle through the C ABI.

The oracle takes the step in fp64 on the stored bf16 values and rounds each updated
slot to the nearest bf16; the kernel takes it in fp32 and rounds the same way.  The
two stored results can therefore differ only where the fp32 result and the exact one
fall on different sides of a bf16 rounding midpoint: by one bf16 step of the element,
at a small fraction of the elements.  That is the single-step bar.  Over several steps
such differences feed the next steps' reads, so the bar there is a few bf16 steps of
the largest element (2^-6 relative to it); the outputs, read from the unrounded fp32
state, keep the fp32-pool bar (2e-3 for bf16 inputs, 1e-4 for fp32 inputs).
"""
import numpy as np
import pytest
import torch

import oracle
from kimi_delta_attention_09_gb300 import inputs
from _helpers import TOL, cuda, rel_err

pytestmark = pytest.mark.gpu

MULTI_STEP_POOL_TOL = 2.0 ** -6


def _native():
    from kimi_delta_attention_09_gb300 import _native
    return _native


def _bf16_spacing(x: np.ndarray) -> np.ndarray:
    """Distance between consecutive bf16 values at |x| (2^(e-8) for |x| in [2^(e-1), 2^e))."""
    _, e = np.frexp(np.asarray(x, dtype=np.float64))
    return np.ldexp(1.0, np.maximum(e, -125) - 8)


def _run(case, steps, out_dtype=torch.float32):
    nat = _native()
    pool = cuda(case.pool.to(torch.bfloat16))
    idx = cuda(case.state_idx)
    outs = []
    for st in case.steps[:steps]:
        out = torch.empty(st.v.shape, dtype=out_dtype, device="cuda")
        nat.kda_recurrent_decode_bf16_state(cuda(st.q), cuda(st.k), cuda(st.v), cuda(st.g),
                                            cuda(st.beta), case.scale, pool, idx, out)
        outs.append(out)
    torch.cuda.synchronize()
    return [o.cpu() for o in outs], pool.cpu()


def _oracle(case, steps, seqs=None):
    seqs = list(range(case.N)) if seqs is None else list(seqs)
    pool = case.pool.to(torch.bfloat16).double().numpy().copy()
    idx = case.state_idx.long().numpy()[seqs]
    outs = []
    for st in case.steps[:steps]:
        outs.append(oracle.decode_bf16_state(st.q[seqs], st.k[seqs], st.v[seqs], st.g[seqs],
                                             st.beta[seqs], case.scale, pool, idx))
    return outs, pool


def _untouched_bit_identical(case, pool):
    mask = torch.ones(case.pool.shape[0], dtype=torch.bool)
    mask[case.state_idx.long()[(case.state_idx >= 0) & (case.state_idx < case.pool.shape[0])]] = False
    start = case.pool.to(torch.bfloat16)
    return torch.equal(pool[mask].view(torch.int16), start[mask].view(torch.int16))


@pytest.mark.parametrize("dtype,K,V", [("bf16", 128, 128), ("f32", 128, 128), ("bf16", 64, 128),
                                       ("f32", 128, 64), ("bf16", 64, 64)])
def test_one_step_is_the_rounded_step(dtype, K, V):
    case = inputs.decode_case(N=9, S=14, H=3, K=K, V=V, steps=1, dtype=dtype, seed=70 + K + V)
    outs, pool = _run(case, 1)
    ref_outs, ref_pool = _oracle(case, 1)
    assert rel_err(outs[0], ref_outs[0]) <= TOL[dtype]
    used = case.state_idx.long()
    got = pool[used].double().numpy()
    ref = ref_pool[used.numpy()]
    assert np.array_equal(oracle.round_to_bf16(ref), ref)       # the oracle stores bf16 values
    diff = np.abs(got - ref)
    step = _bf16_spacing(np.maximum(np.abs(got), np.abs(ref)))
    assert (diff <= step).all(), float((diff / step).max())       # at most one bf16 step apart
    assert np.count_nonzero(diff) <= 1e-2 * diff.size, np.count_nonzero(diff)
    assert _untouched_bit_identical(case, pool)


def test_several_steps_stay_close():
    case = inputs.decode_case(N=8, S=16, H=4, K=128, V=128, steps=8, dtype="bf16", seed=75)
    outs, pool = _run(case, 8)
    ref_outs, ref_pool = _oracle(case, 8)
    for o, r in zip(outs, ref_outs):
        assert rel_err(o, r) <= TOL["bf16"]
    used = case.state_idx.long()
    assert rel_err(pool[used], ref_pool[used.numpy()]) <= MULTI_STEP_POOL_TOL
    assert _untouched_bit_identical(case, pool)


def test_bf16_output_is_the_rounded_fp32_output():
    case = inputs.decode_case(N=5, S=9, H=2, K=128, V=128, steps=3, dtype="bf16", seed=76)
    o32, p32 = _run(case, 3, torch.float32)
    o16, p16 = _run(case, 3, torch.bfloat16)
    for a, b in zip(o16, o32):
        assert torch.equal(a.view(torch.int16), b.to(torch.bfloat16).view(torch.int16))
    assert torch.equal(p16.view(torch.int16), p32.view(torch.int16))


def test_pool_spans_two_bytes_per_element():
    """The output placed right after the bf16 pool in one allocation is accepted (the
    pool's byte range is S H K V * 2) and the step is unchanged."""
    nat = _native()
    case = inputs.decode_case(N=3, S=5, H=2, K=128, V=128, steps=1, dtype="bf16", seed=77)
    st = case.steps[0]
    S, H, K, V = case.pool.shape
    n_pool = S * H * K * V
    buf = torch.empty(n_pool * 2 + 3 * H * V * 4, dtype=torch.uint8, device="cuda")
    pool = buf[:n_pool * 2].view(torch.bfloat16).view(S, H, K, V)
    pool.copy_(cuda(case.pool.to(torch.bfloat16)))
    out = buf[n_pool * 2:].view(torch.float32).view(3, H, V)
    nat.kda_recurrent_decode_bf16_state(cuda(st.q), cuda(st.k), cuda(st.v), cuda(st.g),
                                        cuda(st.beta), case.scale, pool, cuda(case.state_idx), out)
    torch.cuda.synchronize()
    ref_outs, _ = _oracle(case, 1)
    assert rel_err(out.cpu(), ref_outs[0]) <= TOL["bf16"]


def test_out_of_range_slot_touches_nothing():
    case = inputs.decode_case(N=3, S=4, H=2, K=64, V=64, steps=1, dtype="f32", seed=78)
    case.state_idx = torch.tensor([2, 4, -1], dtype=torch.int32)
    outs, pool = _run(case, 1)
    assert torch.equal(outs[0][1:], torch.zeros_like(outs[0][1:]))
    ref_outs, _ = _oracle(case, 1, seqs=[0])
    assert rel_err(outs[0][:1], ref_outs[0]) <= TOL["f32"]
    for s in (0, 1, 3):
        assert torch.equal(pool[s].view(torch.int16), case.pool[s].to(torch.bfloat16).view(torch.int16))


def test_paged_decode_full_size_sampled():
    """The paged-decode workload (256 sequences x 64 steps, 1024 slots) on a bf16 pool:
    the outputs of 24 sampled sequences and their slots against the oracle, every
    untouched slot bit-exact."""
    case = inputs.paged_decode(steps=64)
    outs, pool = _run(case, 64)
    sample = list(range(0, 256, 11))
    ref_outs, ref_pool = _oracle(case, 64, seqs=sample)
    worst = max(rel_err(o[sample], r) for o, r in zip(outs, ref_outs))
    assert worst <= TOL["bf16"], worst
    slots = case.state_idx.long()[sample]
    assert rel_err(pool[slots], ref_pool[slots.numpy()]) <= MULTI_STEP_POOL_TOL
    assert _untouched_bit_identical(case, pool)
