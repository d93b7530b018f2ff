"""Paged recurrent decode on the GPU against the fp64 oracle (through the C ABI)."""
import numpy as np
import pytest
import torch

import oracle
from kimi_delta_attention_09_gb300 import inputs
from _helpers import TOL, cuda, rel_err

pytestmark = pytest.mark.gpu


def _native():
    from kimi_delta_attention_09_gb300 import _native
    return _native


def _run_steps(case, steps, out_dtype=torch.float32):
    """Decode `steps` tokens on the GPU; returns (outs list, final pool on CPU).
    Parity is judged on fp32 outputs; bf16 outputs are checked to be them rounded."""
    nat = _native()
    pool = cuda(case.pool)
    idx = cuda(case.state_idx)
    outs = []
    for st in case.steps[:steps]:
        out = torch.empty(st.v.shape, dtype=out_dtype, device="cuda")
        nat.kda_recurrent_decode(cuda(st.q), cuda(st.k), cuda(st.v), cuda(st.g), cuda(st.beta),
                                 case.scale, pool, idx, out)
        outs.append(out)
    torch.cuda.synchronize()
    return [o.cpu() for o in outs], pool.cpu()


def _oracle_steps(case, steps, seqs=None):
    seqs = list(range(case.N)) if seqs is None else list(seqs)
    pool = case.pool.double().numpy().copy()
    idx = case.state_idx.long().numpy()[seqs]
    outs = []
    for st in case.steps[:steps]:
        outs.append(oracle.decode(st.q[seqs], st.k[seqs], st.v[seqs], st.g[seqs], st.beta[seqs],
                                  case.scale, pool, idx))
    return outs, pool


@pytest.mark.parametrize("dtype,K,V", [("bf16", 128, 128), ("f32", 128, 128), ("f32", 64, 64),
                                       ("bf16", 64, 128), ("bf16", 128, 64)])
def test_decode_matches_oracle(dtype, K, V):
    case = inputs.decode_case(N=7, S=12, H=3, K=K, V=V, steps=5, dtype=dtype, seed=40 + K + V)
    outs, pool = _run_steps(case, 5)
    ref_outs, ref_pool = _oracle_steps(case, 5)
    tol = TOL[dtype]
    for o, r in zip(outs, ref_outs):
        assert rel_err(o, r) <= tol
    used = case.state_idx.long()
    assert rel_err(pool[used], ref_pool[used.numpy()]) <= tol
    # slots that no sequence selects are bit-identical (integer view)
    mask = torch.ones(case.pool.shape[0], dtype=torch.bool)
    mask[used] = False
    assert torch.equal(pool[mask].view(torch.int32), case.pool[mask].view(torch.int32))


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_bf16_output_is_the_rounded_fp32_output(dtype):
    case = inputs.decode_case(N=5, S=9, H=2, K=128, V=128, steps=3, dtype=dtype, seed=52)
    o32, p32 = _run_steps(case, 3, torch.float32)
    o16, p16 = _run_steps(case, 3, torch.bfloat16)
    for a, b in zip(o16, o32):
        assert torch.equal(a.view(torch.int16), b.to(torch.bfloat16).view(torch.int16))
    assert torch.equal(p16, p32)


def test_decode_writes_each_sequence_to_its_own_slot():
    """Scatter goes to state_idx[n] (not slot 0, not slot n) and is actually written."""
    case = inputs.decode_case(N=4, S=9, H=2, K=128, V=128, steps=1, dtype="f32", seed=50)
    case.state_idx = torch.tensor([8, 0, 5, 2], dtype=torch.int32)
    outs, pool = _run_steps(case, 1)
    ref_outs, ref_pool = _oracle_steps(case, 1)
    for s in (8, 0, 5, 2):
        assert not torch.equal(pool[s], case.pool[s])         # the state was written back
        assert rel_err(pool[s], ref_pool[s]) <= 1e-5
    for s in (1, 3, 4, 6, 7):
        assert torch.equal(pool[s].view(torch.int32), case.pool[s].view(torch.int32))
    assert rel_err(outs[0], ref_outs[0]) <= 1e-5


def test_decode_out_of_range_slot_touches_nothing():
    """An index outside [0, S) gives zero outputs and leaves every slot unchanged
    (the kernel's own bounds check; no access is made for that sequence)."""
    case = inputs.decode_case(N=3, S=4, H=2, K=64, V=64, steps=1, dtype="f32", seed=51)
    case.state_idx = torch.tensor([1, 4, -1], dtype=torch.int32)
    outs, pool = _run_steps(case, 1)
    assert torch.equal(outs[0][1:], torch.zeros_like(outs[0][1:]))
    ref_outs, ref_pool = _oracle_steps(case, 1, seqs=[0])
    assert rel_err(outs[0][:1], ref_outs[0]) <= 1e-5
    for s in (0, 2, 3):
        assert torch.equal(pool[s].view(torch.int32), case.pool[s].view(torch.int32))


def test_paged_decode_full_size_sampled():
    """256 sequences x 64 steps over a 1024-slot pool (the paged-decode workload);
    every output of 24 sampled sequences and their slots checked against the oracle,
    every untouched slot checked bit-exact."""
    case = inputs.paged_decode(steps=64)
    outs, pool = _run_steps(case, 64)
    sample = list(range(0, 256, 11))
    ref_outs, ref_pool = _oracle_steps(case, 64, seqs=sample)
    tol = TOL["bf16"]
    worst = max(rel_err(o[sample], r) for o, r in zip(outs, ref_outs))
    assert worst <= tol, worst
    slots = case.state_idx.long()[sample]
    assert rel_err(pool[slots], ref_pool[slots.numpy()]) <= tol
    mask = torch.ones(1024, dtype=torch.bool)
    mask[case.state_idx.long()] = False
    assert torch.equal(pool[mask].view(torch.int32), case.pool[mask].view(torch.int32))
    assert all(torch.isfinite(o.float()).all() for o in outs)
