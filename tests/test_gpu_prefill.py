"""Chunked prefill on the GPU against the fp64 oracle (through the C ABI)."""
import numpy as np
import pytest
import torch

import oracle
from kimi_delta_attention_09_gb300 import inputs
from _helpers import TOL, cuda, dtype_name, oracle_prefill, rel_err

pytestmark = pytest.mark.gpu


def run_prefill(case, init_in_place=False, final=True, out_dtype=torch.float32):
    """Run the GPU prefill.  Parity is judged on fp32 outputs (the arithmetic error
    alone); a bf16 output is checked separately to be that fp32 result rounded."""
    from kimi_delta_attention_09_gb300 import _native
    q, k, v, g, beta = (cuda(x) for x in (case.q, case.k, case.v, case.g, case.beta))
    cu = cuda(case.cu_seqlens)
    init = cuda(case.init_state)
    out = torch.full(v.shape, float("nan"), dtype=out_dtype, device="cuda")
    fin = None
    if final:
        fin = init if (init_in_place and init is not None) else torch.full(
            (case.N, case.H, case.K, case.V), float("nan"), device="cuda")
    _native.kda_chunk_prefill(q, k, v, g, beta, case.scale, init, cu, out, fin)
    torch.cuda.synchronize()
    return out.cpu(), (None if fin is None else fin.cpu())


def check_case(case, heads=None, seqs=None, **kw):
    out, fin = run_prefill(case, **kw)
    heads = list(range(case.H)) if heads is None else heads
    seqs = list(range(case.N)) if seqs is None else seqs
    ref_out, ref_fin = oracle_prefill(case, heads, seqs)
    tol = TOL[dtype_name(case.q)]
    rows = np.concatenate([np.arange(int(case.cu_seqlens[n]), int(case.cu_seqlens[n + 1]))
                           for n in seqs]) if seqs else np.zeros(0, dtype=np.int64)
    e_out = rel_err(out[rows][:, heads], ref_out[rows]) if rows.size else 0.0
    e_fin = rel_err(fin[seqs][:, heads], ref_fin)
    assert e_out <= tol, f"out rel err {e_out:.3e} > {tol}"
    assert e_fin <= tol, f"final state rel err {e_fin:.3e} > {tol}"
    return e_out, e_fin


def test_tiny_f32_workload():
    """B=1, H=2, T=128, K=V=64, fp32 -- the oracle-sized case, full comparison."""
    check_case(inputs.tiny_f32())


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("K,V", [(128, 128), (64, 64), (128, 64), (64, 128)])
def test_ragged_varlen_with_initial_state(dtype, K, V):
    """Several chunks, ragged tails (1, 63, 64, 65, 200 tokens), nonzero init."""
    case = inputs.prefill_case([1, 63, 64, 65, 200], H=3, K=K, V=V, dtype=dtype,
                               seed=60 + K + V, init_std=0.02)
    check_case(case)


def test_final_state_in_place_and_empty_sequences():
    """final_state == init_state carries in place; empty sequences return init."""
    case = inputs.prefill_case([0, 130, 0, 5], H=2, K=128, V=128, dtype="bf16", seed=61,
                               init_std=0.05)
    check_case(case, init_in_place=True)
    out, fin = run_prefill(case)
    assert torch.equal(fin[0], case.init_state[0]) and torch.equal(fin[2], case.init_state[2])


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_bf16_output_is_the_rounded_fp32_output(dtype):
    """out_dtype=bf16 stores exactly round-to-nearest(bf16) of the fp32 result."""
    case = inputs.prefill_case([1, 64, 130], H=2, K=128, V=128, dtype=dtype, seed=66,
                               init_std=0.02)
    o32, f32 = run_prefill(case, out_dtype=torch.float32)
    o16, f16 = run_prefill(case, out_dtype=torch.bfloat16)
    assert torch.equal(o16.view(torch.int16), o32.to(torch.bfloat16).view(torch.int16))
    assert torch.equal(f16, f32)


def test_zero_init_and_no_final_state():
    case = inputs.prefill_case([97], H=2, K=128, V=128, dtype="bf16", seed=62)
    out, fin = run_prefill(case, final=False)
    ref, _ = oracle_prefill(case)
    assert fin is None and rel_err(out, ref) <= TOL["bf16"]


def test_split_prefill_carries_state():
    """Prefill [0, T1) then [T1, T) from the returned state = prefill of [0, T)."""
    full = inputs.prefill_case([300], H=2, K=128, V=128, dtype="bf16", seed=63, init_std=0.02)
    T1 = 137
    a = inputs.PrefillCase(name="a", seed=0, q=full.q[:T1], k=full.k[:T1], v=full.v[:T1],
                           g=full.g[:T1], beta=full.beta[:T1],
                           cu_seqlens=torch.tensor([0, T1], dtype=torch.int32),
                           init_state=full.init_state, scale=full.scale)
    out_a, fin_a = run_prefill(a)
    b = inputs.PrefillCase(name="b", seed=0, q=full.q[T1:], k=full.k[T1:], v=full.v[T1:],
                           g=full.g[T1:], beta=full.beta[T1:],
                           cu_seqlens=torch.tensor([0, 300 - T1], dtype=torch.int32),
                           init_state=fin_a, scale=full.scale)
    out_b, fin_b = run_prefill(b)
    ref_out, ref_fin = oracle_prefill(full)
    assert rel_err(torch.cat([out_a, out_b]), ref_out) <= TOL["bf16"]
    assert rel_err(fin_b, ref_fin) <= TOL["bf16"]


def test_strong_gates():
    """Gates down to -5 per step per channel (a naive exp factorisation overflows)."""
    case = inputs.prefill_case([150], H=2, K=128, V=128, dtype="bf16", seed=64)
    gen = torch.Generator().manual_seed(64)
    case.g = (-5.0 * torch.rand(case.g.shape, generator=gen)).float()
    check_case(case)


def test_prefill_then_decode_matches_full_recurrence():
    """Prompt through the chunked prefill, state scattered into a pool slot, then
    token-by-token decode = the oracle over the whole sequence."""
    from kimi_delta_attention_09_gb300 import _native
    T0, steps, H = 200, 6, 2
    full = inputs.prefill_case([T0 + steps], H=H, K=128, V=128, dtype="bf16", seed=65)
    pre = inputs.PrefillCase(name="p", seed=0, q=full.q[:T0], k=full.k[:T0], v=full.v[:T0],
                             g=full.g[:T0], beta=full.beta[:T0],
                             cu_seqlens=torch.tensor([0, T0], dtype=torch.int32),
                             init_state=None, scale=full.scale)
    out_p, fin_p = run_prefill(pre)
    pool = torch.zeros(3, H, 128, 128, device="cuda")
    pool[1] = fin_p[0].cuda()
    idx = torch.tensor([1], dtype=torch.int32, device="cuda")
    outs = []
    for t in range(T0, T0 + steps):
        o = torch.empty(1, H, 128, dtype=torch.float32, device="cuda")
        sl = slice(t, t + 1)
        _native.kda_recurrent_decode(cuda(full.q[sl]), cuda(full.k[sl]), cuda(full.v[sl]),
                                     cuda(full.g[sl]), cuda(full.beta[sl]), full.scale, pool,
                                     idx, o)
        outs.append(o.cpu())
    ref_out, ref_fin = oracle_prefill(full)
    assert rel_err(torch.cat([out_p] + outs), ref_out) <= TOL["bf16"]
    assert rel_err(pool[1].cpu(), ref_fin[0]) <= TOL["bf16"]


# ------------------------------------------------------------ full-size workloads

def test_single_prompt_workload_sampled_heads():
    """B=1, H=32, T=4096, K=V=128 bf16: all outputs and states of 4 sampled heads."""
    check_case(inputs.single_prompt(), heads=[0, 9, 22, 31])


def test_varlen_packed_workload_sampled():
    """8 packed sequences (lengths 256..8192), nonzero init: 3 sequences x 3 heads."""
    case = inputs.varlen_packed()
    check_case(case, heads=[1, 16, 30], seqs=[0, 4, 6])


def test_long_prefill_workload_sampled():
    """B=1, H=32, T=65536: 2 sampled heads, every output and the final state."""
    check_case(inputs.long_prefill(), heads=[5, 27])


# ------------------------------------------------------------ paged (slot-indexed) prefill

def _run_paged(case, pool_cpu, slots, out_dtype=torch.float32):
    from kimi_delta_attention_09_gb300 import _native
    q, k, v, g, beta = (cuda(x) for x in (case.q, case.k, case.v, case.g, case.beta))
    pool = cuda(pool_cpu)
    idx = torch.tensor(slots, dtype=torch.int32, device="cuda")
    out = torch.full(v.shape, float("nan"), dtype=out_dtype, device="cuda")
    _native.kda_chunk_prefill_paged(q, k, v, g, beta, case.scale, pool, idx,
                                    cuda(case.cu_seqlens), out)
    torch.cuda.synchronize()
    return out.cpu(), pool.cpu()


@pytest.mark.parametrize("dtype,K,V", [("bf16", 128, 128), ("f32", 64, 64), ("bf16", 64, 128)])
def test_paged_prefill_reads_and_writes_its_slots(dtype, K, V):
    """Sequence n starts from slot state_idx[n] and its final state lands there (not in
    slot 0, not in slot n); every other slot is bit-identical."""
    case = inputs.prefill_case([70, 1, 130], H=2, K=K, V=V, dtype=dtype, seed=70)
    gen = torch.Generator().manual_seed(71)
    pool0 = (torch.randn(6, 2, K, V, generator=gen) * 0.05).float()
    slots = [4, 0, 2]
    out, pool = _run_paged(case, pool0, slots)
    case.init_state = pool0[slots].clone()
    ref_out, ref_fin = oracle_prefill(case)
    tol = TOL[dtype]
    assert rel_err(out, ref_out) <= tol
    for n, s in enumerate(slots):
        assert rel_err(pool[s], ref_fin[n]) <= tol
        assert not torch.equal(pool[s], pool0[s])
    for s in (1, 3, 5):
        assert torch.equal(pool[s].view(torch.int32), pool0[s].view(torch.int32))


def test_paged_prefill_then_paged_decode():
    """Paged prefill of a prompt, then token-by-token decode on the same pool slot =
    the oracle over the whole sequence (the runner's prompt + decode path)."""
    from kimi_delta_attention_09_gb300 import _native
    T0, steps, H = 150, 5, 2
    full = inputs.prefill_case([T0 + steps], H=H, K=128, V=128, dtype="bf16", seed=72)
    pre = inputs.PrefillCase(name="p", seed=0, q=full.q[:T0], k=full.k[:T0], v=full.v[:T0],
                             g=full.g[:T0], beta=full.beta[:T0],
                             cu_seqlens=torch.tensor([0, T0], dtype=torch.int32),
                             init_state=None, scale=full.scale)
    pool0 = torch.zeros(4, H, 128, 128)
    out_p, pool = _run_paged(pre, pool0, [3])
    pool = pool.cuda()
    idx = torch.tensor([3], dtype=torch.int32, device="cuda")
    outs = [out_p]
    for t in range(T0, T0 + steps):
        o = torch.empty(1, H, 128, dtype=torch.float32, device="cuda")
        sl = slice(t, t + 1)
        _native.kda_recurrent_decode(cuda(full.q[sl]), cuda(full.k[sl]), cuda(full.v[sl]),
                                     cuda(full.g[sl]), cuda(full.beta[sl]), full.scale, pool,
                                     idx, o)
        outs.append(o.cpu())
    ref_out, ref_fin = oracle_prefill(full)
    assert rel_err(torch.cat(outs), ref_out) <= TOL["bf16"]
    assert rel_err(pool[3].cpu(), ref_fin[0]) <= TOL["bf16"]
    assert torch.equal(pool[:3].cpu(), torch.zeros(3, H, 128, 128))


# ------------------------------------------------------------ host-staged (pipelined) prefill

@pytest.mark.parametrize("segments", [1, 3, 4, 16])
def test_prefill_from_host_matches_oracle(segments):
    """Host inputs, pieces cut on 64-token boundaries of the packed range (so sequences
    are split mid-chunk and carried across pieces), nonzero initial states."""
    import kimi_delta_attention_09_gb300 as kda
    case = inputs.prefill_case([1, 63, 150, 65, 230], H=2, K=128, V=128, dtype="bf16", seed=73,
                               init_std=0.02)
    pin = [x.pin_memory() for x in (case.q, case.k, case.v, case.g, case.beta)]
    out, fin, _ = kda.chunk_prefill_from_host(*pin, case.scale, case.init_state.pin_memory(),
                                              case.cu_seqlens, out_dtype=torch.float32,
                                              segments=segments)
    torch.cuda.synchronize()
    ref_out, ref_fin = oracle_prefill(case)
    assert rel_err(out, ref_out) <= TOL["bf16"]
    assert rel_err(fin, ref_fin) <= TOL["bf16"]


def test_prefill_from_host_reuses_buffers():
    """Two calls in a row with the first call's device buffers give the same result."""
    import kimi_delta_attention_09_gb300 as kda
    case = inputs.prefill_case([300], H=2, K=128, V=128, dtype="bf16", seed=74)
    pin = [x.pin_memory() for x in (case.q, case.k, case.v, case.g, case.beta)]
    o1, f1, bufs = kda.chunk_prefill_from_host(*pin, case.scale, None, case.cu_seqlens, segments=3)
    torch.cuda.synchronize()
    o1, f1 = o1.clone(), f1.clone()
    o2, f2, _ = kda.chunk_prefill_from_host(*pin, case.scale, None, case.cu_seqlens, segments=3,
                                            buffers=bufs)
    torch.cuda.synchronize()
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16)) and torch.equal(f1, f2)


def test_host_entry_with_one_piece_is_the_device_prefill():
    """kda_chunk_prefill_host with one piece runs the same kernel on the same values as
    kda_chunk_prefill_ws on device copies: bit-identical outputs and final states."""
    from kimi_delta_attention_09_gb300 import _native
    case = inputs.prefill_case([1, 63, 150, 65, 230], H=2, K=128, V=128, dtype="bf16", seed=75,
                               init_std=0.02)
    host = [x.pin_memory() for x in (case.q, case.k, case.v, case.g, case.beta)]
    hout = torch.empty(case.T, 2, 128, dtype=torch.float32).pin_memory()
    hfin = torch.empty(case.N, 2, 128, 128).pin_memory()
    n = _native.kda_chunk_prefill_host_device_bytes(case.T, case.N, 2, 128, 128, torch.bfloat16,
                                                    torch.float32, 1)
    dev = torch.zeros(n, dtype=torch.uint8, device="cuda")
    _native.kda_chunk_prefill_host(*host, case.scale, case.init_state.pin_memory(), case.cu_seqlens,
                                   hout, hfin, 1, dev)
    q, k, v, g, beta = (cuda(x) for x in (case.q, case.k, case.v, case.g, case.beta))
    out = torch.empty(case.T, 2, 128, device="cuda")
    fin = torch.empty(case.N, 2, 128, 128, device="cuda")
    ws = torch.zeros(_native.kda_chunk_prefill_workspace_bytes(case.N, 2, 128, 128, torch.bfloat16),
                     dtype=torch.uint8, device="cuda")
    _native.kda_chunk_prefill_ws(q, k, v, g, beta, case.scale, cuda(case.init_state),
                                 cuda(case.cu_seqlens), out, fin, ws)
    torch.cuda.synchronize()
    assert _native.kda_chunk_prefill_status(dev) == _native.KDA_OK
    assert torch.equal(hout, out.cpu()) and torch.equal(hfin, fin.cpu())


def test_host_entry_carries_the_state_in_place():
    """final_state == init_state on the host: the initial state is read before the final
    state is written back over it."""
    from kimi_delta_attention_09_gb300 import _native
    case = inputs.prefill_case([1, 63, 150, 65, 230], H=2, K=128, V=128, dtype="bf16", seed=76,
                               init_std=0.02)
    host = [x.pin_memory() for x in (case.q, case.k, case.v, case.g, case.beta)]
    state = case.init_state.clone().pin_memory()
    hout = torch.empty(case.T, 2, 128, dtype=torch.float32).pin_memory()
    n = _native.kda_chunk_prefill_host_device_bytes(case.T, case.N, 2, 128, 128, torch.bfloat16,
                                                    torch.float32, 3)
    dev = torch.zeros(n, dtype=torch.uint8, device="cuda")
    _native.kda_chunk_prefill_host(*host, case.scale, state, case.cu_seqlens, hout, state, 3, dev)
    torch.cuda.synchronize()
    ref_out, ref_fin = oracle_prefill(case)
    assert rel_err(hout, ref_out) <= TOL["bf16"]
    assert rel_err(state, ref_fin) <= TOL["bf16"]
