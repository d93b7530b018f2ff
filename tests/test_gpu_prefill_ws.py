"""kda_chunk_prefill_ws (the tensor-core prefill: the four CTAs of a cluster share each
chunk's operand record through a ring in the caller's workspace) on the GPU against the
fp64 oracle, through the C ABI."""
import numpy as np
import pytest
import torch

from kimi_delta_attention_09_gb300 import inputs
from _helpers import TOL, cuda, dtype_name, oracle_prefill, rel_err

pytestmark = pytest.mark.gpu


def workspace_for(case):
    from kimi_delta_attention_09_gb300 import _native
    n = _native.kda_chunk_prefill_workspace_bytes(case.N, case.H, case.K, case.V, case.q.dtype)
    return None if n == 0 else torch.zeros(n, dtype=torch.uint8, device="cuda")


def run_ws(case, init_in_place=False, final=True, out_dtype=torch.float32, workspace=None):
    from kimi_delta_attention_09_gb300 import _native
    q, k, v, g, beta = (cuda(x) for x in (case.q, case.k, case.v, case.g, case.beta))
    cu = cuda(case.cu_seqlens)
    init = cuda(case.init_state)
    out = torch.full(v.shape, float("nan"), dtype=out_dtype, device="cuda")
    fin = None
    if final:
        fin = init if (init_in_place and init is not None) else torch.full(
            (case.N, case.H, case.K, case.V), float("nan"), device="cuda")
    ws = workspace_for(case) if workspace is None else workspace
    _native.kda_chunk_prefill_ws(q, k, v, g, beta, case.scale, init, cu, out, fin, ws)
    torch.cuda.synchronize()
    return out.cpu(), (None if fin is None else fin.cpu())


def check_case(case, heads=None, seqs=None, **kw):
    out, fin = run_ws(case, **kw)
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
    return out, fin


def test_workspace_size_query():
    from kimi_delta_attention_09_gb300 import _native
    n = _native.kda_chunk_prefill_workspace_bytes(1, 32, 128, 128, torch.bfloat16)
    assert n > 0 and n % 16 == 0
    # bounded by the resident clusters, not by the number of sequences
    assert _native.kda_chunk_prefill_workspace_bytes(4096, 32, 128, 128, torch.bfloat16) <= 64 * n
    assert _native.kda_chunk_prefill_workspace_bytes(1, 32, 128, 128, torch.float32) == 0
    assert _native.kda_chunk_prefill_workspace_bytes(1, 32, 64, 128, torch.bfloat16) == 0
    assert _native.kda_chunk_prefill_workspace_bytes(0, 32, 128, 128, torch.bfloat16) == 0


def test_ragged_varlen_with_initial_state():
    """Several chunks, ragged tails (1, 63, 64, 65, 200 tokens), nonzero init."""
    case = inputs.prefill_case([1, 63, 64, 65, 200], H=3, K=128, V=128, dtype="bf16", seed=160,
                               init_std=0.02)
    check_case(case)


def test_more_work_items_than_clusters():
    """80 (sequence, head) items, empty ones included: each persistent cluster walks
    several items and the record ring wraps many times."""
    case = inputs.prefill_case([0, 5, 64, 130, 1, 200, 0, 77, 300, 65], H=8, K=128, V=128,
                               dtype="bf16", seed=161, init_std=0.02)
    out, fin = check_case(case)
    for n in (0, 6):   # empty sequences return their initial state
        assert torch.equal(fin[n], case.init_state[n])


def test_many_short_ragged_sequences():
    """40 and 70 sequences of ragged lengths (ties and empty ones included): each
    persistent cluster walks several items of different lengths."""
    rng = np.random.default_rng(165)
    for n_seqs in (40, 70):
        lens = [int(x) for x in rng.integers(0, 160, size=n_seqs)]
        lens[3] = lens[5] = 0
        lens[7] = lens[9] = 130
        case = inputs.prefill_case(lens, H=2, K=128, V=128, dtype="bf16", seed=165 + n_seqs,
                                   init_std=0.02)
        check_case(case)


def test_final_state_in_place_and_empty_sequences():
    case = inputs.prefill_case([0, 130, 0, 5], H=2, K=128, V=128, dtype="bf16", seed=162,
                               init_std=0.05)
    check_case(case, init_in_place=True)


def test_bf16_output_is_the_rounded_fp32_output():
    case = inputs.prefill_case([1, 64, 130], H=2, K=128, V=128, dtype="bf16", seed=163,
                               init_std=0.02)
    o32, f32 = run_ws(case, out_dtype=torch.float32)
    o16, f16 = run_ws(case, out_dtype=torch.bfloat16)
    assert torch.equal(o16.view(torch.int16), o32.to(torch.bfloat16).view(torch.int16))
    assert torch.equal(f16, f32)


def test_library_scratch_entry_point_gives_the_same_bits():
    """kda_chunk_prefill (the library's own scratch) runs the same kernel: bit-identical
    outputs and final states."""
    from kimi_delta_attention_09_gb300 import _native
    case = inputs.prefill_case([300, 77], H=4, K=128, V=128, dtype="bf16", seed=164,
                               init_std=0.02)
    o_ws, f_ws = run_ws(case)
    q, k, v, g, beta = (cuda(x) for x in (case.q, case.k, case.v, case.g, case.beta))
    out = torch.empty(v.shape, device="cuda")
    fin = torch.empty(case.N, case.H, 128, 128, device="cuda")
    _native.kda_chunk_prefill(q, k, v, g, beta, case.scale, cuda(case.init_state),
                              cuda(case.cu_seqlens), out, fin)
    torch.cuda.synchronize()
    assert torch.equal(o_ws.view(torch.int32), out.cpu().view(torch.int32))
    assert torch.equal(f_ws.view(torch.int32), fin.cpu().view(torch.int32))


def test_two_calls_with_one_workspace():
    """A workspace is reused without clearing: a second call (and one after a call of
    other sizes) on the earlier calls' leftovers gives the identical result."""
    case = inputs.prefill_case([200, 9], H=3, K=128, V=128, dtype="bf16", seed=165,
                               init_std=0.02)
    other = inputs.prefill_case([64, 1, 500], H=3, K=128, V=128, dtype="bf16", seed=175)
    ws = workspace_for(other)
    o1, f1 = run_ws(case, workspace=ws)
    o2, f2 = run_ws(case, workspace=ws)
    run_ws(other, workspace=ws)
    o3, f3 = run_ws(case, workspace=ws)
    for o, f in ((o2, f2), (o3, f3)):
        assert torch.equal(o1.view(torch.int32), o.view(torch.int32))
        assert torch.equal(f1.view(torch.int32), f.view(torch.int32))


def test_strong_gates():
    """Gates down to -5 per step per channel: the exact-exponential path of the builders."""
    case = inputs.prefill_case([150], H=2, K=128, V=128, dtype="bf16", seed=166)
    gen = torch.Generator().manual_seed(166)
    case.g = (-5.0 * torch.rand(case.g.shape, generator=gen)).float()
    check_case(case)


def test_split_prefill_carries_state():
    full = inputs.prefill_case([300], H=2, K=128, V=128, dtype="bf16", seed=167, init_std=0.02)
    T1 = 137
    a = inputs.PrefillCase(name="a", seed=0, q=full.q[:T1], k=full.k[:T1], v=full.v[:T1],
                           g=full.g[:T1], beta=full.beta[:T1],
                           cu_seqlens=torch.tensor([0, T1], dtype=torch.int32),
                           init_state=full.init_state, scale=full.scale)
    out_a, fin_a = run_ws(a)
    b = inputs.PrefillCase(name="b", seed=0, q=full.q[T1:], k=full.k[T1:], v=full.v[T1:],
                           g=full.g[T1:], beta=full.beta[T1:],
                           cu_seqlens=torch.tensor([0, 300 - T1], dtype=torch.int32),
                           init_state=fin_a, scale=full.scale)
    out_b, fin_b = run_ws(b)
    ref_out, ref_fin = oracle_prefill(full)
    assert rel_err(torch.cat([out_a, out_b]), ref_out) <= TOL["bf16"]
    assert rel_err(fin_b, ref_fin) <= TOL["bf16"]


def test_fast_and_exact_chunks_alternate_in_one_sequence():
    """Chunks whose gate span leaves the fp16 factors' range (exact-exponential path) and
    chunks on the fp16 fast path alternate inside one sequence; ragged tail."""
    case = inputs.prefill_case([64 * 7 + 29], H=2, K=128, V=128, dtype="bf16", seed=176,
                               init_std=0.02)
    gen = torch.Generator().manual_seed(176)
    strong = (-4.0 * torch.rand(case.g.shape, generator=gen)).float()
    chunk = torch.arange(case.T) // 64
    case.g = torch.where((chunk % 2 == 1)[:, None, None], strong, case.g).contiguous()
    check_case(case)


def test_large_state_and_value_magnitudes():
    """Initial states of std 5 and values of std 100 (inputs far from unit scale, still
    inside the fp16 operand range), with weak gates that keep the state long-lived."""
    case = inputs.prefill_case([333, 64], H=2, K=128, V=128, dtype="bf16", seed=177,
                               init_std=5.0, gate_scale=0.02)
    case.v = (case.v.float() * 100.0).to(torch.bfloat16).contiguous()
    check_case(case)


def test_timeout_is_reported_and_the_context_stays_usable():
    """A wait limit of 100 ns makes the kernel's waits run out on purpose: the clusters
    end early, kda_chunk_prefill_status reports KDA_ERR_TIMEOUT (once), and a normal
    launch afterwards on the same workspace is correct."""
    from kimi_delta_attention_09_gb300 import _native
    case = inputs.prefill_case([640, 100], H=4, K=128, V=128, dtype="bf16", seed=178,
                               init_std=0.02)
    ws = workspace_for(case)
    try:
        _native.kda_set_prefill_wait_limit(100)
        run_ws(case, workspace=ws)
    finally:
        _native.kda_set_prefill_wait_limit(0)
    assert _native.kda_chunk_prefill_status(ws) == _native.KDA_ERR_TIMEOUT
    assert _native.kda_chunk_prefill_status(ws) == _native.KDA_OK   # read and cleared
    check_case(case, workspace=ws)
    assert _native.kda_chunk_prefill_status(ws) == _native.KDA_OK


def test_workspace_must_be_device_memory_of_this_device():
    """Pinned host memory as the workspace is refused before anything is enqueued."""
    import ctypes
    from kimi_delta_attention_09_gb300 import _native
    case = inputs.prefill_case([100], H=2, K=128, V=128, dtype="bf16", seed=179)
    q, k, v, g, beta = (cuda(x) for x in (case.q, case.k, case.v, case.g, case.beta))
    cu = cuda(case.cu_seqlens)
    n = _native.kda_chunk_prefill_workspace_bytes(case.N, case.H, 128, 128, torch.bfloat16)
    host_ws = torch.zeros(n, dtype=torch.uint8).pin_memory()
    out = torch.zeros(v.shape, device="cuda")
    vp = ctypes.c_void_p
    rc = _native.lib.kda_chunk_prefill_ws(
        vp(q.data_ptr()), vp(k.data_ptr()), vp(v.data_ptr()), vp(g.data_ptr()),
        vp(beta.data_ptr()), case.scale, None, vp(cu.data_ptr()), vp(out.data_ptr()), None,
        case.T, case.N, case.H, 128, 128, 1, 0, vp(host_ws.data_ptr()), n, 0,
        vp(torch.cuda.current_stream().cuda_stream))
    assert rc == _native.KDA_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert torch.count_nonzero(out) == 0


def test_shapes_without_the_tensor_core_kernel_need_no_workspace():
    """fp32 inputs and K = 64 run the other kernels; workspace None is accepted."""
    for dtype, K, V in (("f32", 128, 128), ("bf16", 64, 128)):
        case = inputs.prefill_case([70, 3], H=2, K=K, V=V, dtype=dtype, seed=168, init_std=0.02)
        check_case(case)


def test_workspace_errors():
    from kimi_delta_attention_09_gb300 import _native
    case = inputs.prefill_case([100], H=2, K=128, V=128, dtype="bf16", seed=169)
    q, k, v, g, beta = (cuda(x) for x in (case.q, case.k, case.v, case.g, case.beta))
    cu = cuda(case.cu_seqlens)
    n = _native.kda_chunk_prefill_workspace_bytes(case.N, case.H, 128, 128, torch.bfloat16)
    out = torch.zeros(v.shape, device="cuda")
    small = torch.empty(n - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(_native.KdaError) as e:
        _native.kda_chunk_prefill_ws(q, k, v, g, beta, case.scale, None, cu, out, None, small)
    assert e.value.status == _native.KDA_ERR_INVALID_ARG
    with pytest.raises(_native.KdaError) as e:
        _native.kda_chunk_prefill_ws(q, k, v, g, beta, case.scale, None, cu, out, None, None)
    assert e.value.status == _native.KDA_ERR_INVALID_ARG
    big = torch.empty(n + v.numel() * 4, dtype=torch.uint8, device="cuda")
    lo = n - 4096   # the output overlaps the last 4 KB the call would use
    out_in_ws = big[lo:lo + v.numel() * 4].view(torch.float32).view(v.shape)
    with pytest.raises(_native.KdaError) as e:
        _native.kda_chunk_prefill_ws(q, k, v, g, beta, case.scale, None, cu, out_in_ws, None, big)
    assert e.value.status == _native.KDA_ERR_ALIAS
    torch.cuda.synchronize()
    assert torch.count_nonzero(out) == 0   # nothing was launched


# ------------------------------------------------------------ full-size workloads

def test_single_prompt_workload_sampled_heads():
    check_case(inputs.single_prompt(), heads=[0, 9, 22, 31])


def test_varlen_packed_workload_sampled():
    case = inputs.varlen_packed()
    check_case(case, heads=[1, 16, 30], seqs=[0, 4, 6])


def test_long_prefill_workload_sampled():
    check_case(inputs.long_prefill(), heads=[5, 27])


# ------------------------------------------------------------ paged (slot-indexed) prefill

def _run_paged_ws(case, pool_cpu, slots, out_dtype=torch.float32):
    from kimi_delta_attention_09_gb300 import _native
    q, k, v, g, beta = (cuda(x) for x in (case.q, case.k, case.v, case.g, case.beta))
    pool = cuda(pool_cpu)
    idx = torch.tensor(slots, dtype=torch.int32, device="cuda")
    out = torch.full(v.shape, float("nan"), dtype=out_dtype, device="cuda")
    _native.kda_chunk_prefill_paged_ws(q, k, v, g, beta, case.scale, pool, idx,
                                       cuda(case.cu_seqlens), out, workspace_for(case))
    torch.cuda.synchronize()
    return out.cpu(), pool.cpu()


def test_paged_ws_reads_and_writes_its_slots():
    """Sequence n starts from slot state_idx[n] and its final state lands there (not in
    slot 0, not in slot n); every other slot is bit-identical."""
    case = inputs.prefill_case([70, 1, 130], H=2, K=128, V=128, dtype="bf16", seed=170)
    gen = torch.Generator().manual_seed(171)
    pool0 = (torch.randn(6, 2, 128, 128, generator=gen) * 0.05).float()
    slots = [4, 0, 2]
    out, pool = _run_paged_ws(case, pool0, slots)
    case.init_state = pool0[slots].clone()
    ref_out, ref_fin = oracle_prefill(case)
    assert rel_err(out, ref_out) <= TOL["bf16"]
    for n, s in enumerate(slots):
        assert rel_err(pool[s], ref_fin[n]) <= TOL["bf16"]
        assert not torch.equal(pool[s], pool0[s])
    for s in (1, 3, 5):
        assert torch.equal(pool[s].view(torch.int32), pool0[s].view(torch.int32))


def test_paged_ws_out_of_range_slot_and_many_items():
    """An index outside [0, S) reads and writes no slot (zero start, final state dropped);
    40 sequences x 3 heads are more work items than clusters."""
    lens = [(37 * i) % 150 for i in range(40)]
    case = inputs.prefill_case(lens, H=3, K=128, V=128, dtype="bf16", seed=172)
    gen = torch.Generator().manual_seed(173)
    S = 48
    pool0 = (torch.randn(S, 3, 128, 128, generator=gen) * 0.05).float()
    slots = [(5 * i + 1) % S for i in range(40)]
    slots[7] = S + 3       # out of range
    slots[11] = -1         # out of range
    out, pool = _run_paged_ws(case, pool0, slots)
    used = [s for s in slots if 0 <= s < S]
    case.init_state = torch.stack([pool0[s] if 0 <= s < S else torch.zeros(3, 128, 128)
                                   for s in slots])
    ref_out, ref_fin = oracle_prefill(case)
    assert rel_err(out, ref_out) <= TOL["bf16"]
    for n, s in enumerate(slots):
        if 0 <= s < S:
            assert rel_err(pool[s], ref_fin[n]) <= TOL["bf16"]
    for s in range(S):
        if s not in used:
            assert torch.equal(pool[s].view(torch.int32), pool0[s].view(torch.int32))


def test_paged_ws_then_paged_decode():
    """The runner's path: a prompt through the paged tensor-core prefill, then token-by-token
    decode on the same slot = the oracle over the whole sequence."""
    from kimi_delta_attention_09_gb300 import _native
    T0, steps, H = 150, 5, 2
    full = inputs.prefill_case([T0 + steps], H=H, K=128, V=128, dtype="bf16", seed=174)
    pre = inputs.PrefillCase(name="p", seed=0, q=full.q[:T0], k=full.k[:T0], v=full.v[:T0],
                             g=full.g[:T0], beta=full.beta[:T0],
                             cu_seqlens=torch.tensor([0, T0], dtype=torch.int32),
                             init_state=None, scale=full.scale)
    out_p, pool = _run_paged_ws(pre, torch.zeros(4, H, 128, 128), [3])
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
