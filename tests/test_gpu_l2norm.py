"""The in-kernel q/k L2 normalisation option (KDA_FLAG_QK_L2NORM) on the GPU against the
fp64 oracle with the same option, through the C ABI: the tensor-core prefill (fast and
exact-exponential chunks), the CUDA-core prefill (fp32, K = 64), the library-scratch
prefill, the paged prefill and both decode steps.  The q and k rows are scaled by
per-row factors in [0.5, 8] so that the normalisation matters."""
import numpy as np
import pytest
import torch

import oracle
from kimi_delta_attention_09_gb300 import inputs
from _helpers import TOL, cuda, dtype_name, rel_err

pytestmark = pytest.mark.gpu


def _unnormalise(case, seed):
    gen = torch.Generator().manual_seed(seed)
    for name in ("q", "k"):
        x = getattr(case, name)
        f = 0.5 + 7.5 * torch.rand(x.shape[:-1] + (1,), generator=gen)
        setattr(case, name, (x.float() * f).to(x.dtype).contiguous())
    return case


def _oracle(case):
    return oracle.prefill(case.q, case.k, case.v, case.g, case.beta, case.scale, case.init_state,
                          case.cu_seqlens, qk_l2norm=True)


def _run(case, entry="ws"):
    from kimi_delta_attention_09_gb300 import _native
    q, k, v, g, beta = (cuda(x) for x in (case.q, case.k, case.v, case.g, case.beta))
    cu, init = cuda(case.cu_seqlens), cuda(case.init_state)
    out = torch.full(v.shape, float("nan"), dtype=torch.float32, device="cuda")
    fin = torch.full((case.N, case.H, case.K, case.V), float("nan"), device="cuda")
    fl = _native.KDA_FLAG_QK_L2NORM
    if entry == "ws":
        n = _native.kda_chunk_prefill_workspace_bytes(case.N, case.H, case.K, case.V, q.dtype)
        ws = torch.zeros(n, dtype=torch.uint8, device="cuda") if n else None
        _native.kda_chunk_prefill_ws(q, k, v, g, beta, case.scale, init, cu, out, fin, ws, flags=fl)
    else:
        _native.kda_chunk_prefill(q, k, v, g, beta, case.scale, init, cu, out, fin, flags=fl)
    torch.cuda.synchronize()
    return out.cpu(), fin.cpu()


def _check(case, entry="ws"):
    out, fin = _run(case, entry)
    ref_out, ref_fin = _oracle(case)
    tol = TOL[dtype_name(case.q)]
    e1, e2 = rel_err(out, ref_out), rel_err(fin, ref_fin)
    assert e1 <= tol and e2 <= tol, (e1, e2)


@pytest.mark.parametrize("dtype,K,V", [("bf16", 128, 128), ("f32", 64, 64), ("bf16", 64, 128),
                                       ("f32", 128, 128)])
def test_prefill_normalises_rows(dtype, K, V):
    case = _unnormalise(inputs.prefill_case([1, 63, 130, 200], H=3, K=K, V=V, dtype=dtype,
                                            seed=950, init_std=0.02), 951)
    _check(case)


def test_prefill_normalises_rows_on_exact_chunks():
    case = inputs.prefill_case([150, 77], H=2, K=128, V=128, dtype="bf16", seed=952)
    gen = torch.Generator().manual_seed(952)
    case.g = (-5.0 * torch.rand(case.g.shape, generator=gen)).float()
    _check(_unnormalise(case, 953))


def test_library_scratch_entry_point_normalises_rows():
    case = _unnormalise(inputs.prefill_case([300, 5], H=4, K=128, V=128, dtype="bf16", seed=954,
                                            init_std=0.02), 955)
    _check(case, entry="static")


def test_flag_equals_normalising_first():
    """The option on un-normalised rows gives what the kernel gives without it on the same
    rows normalised beforehand (fp32 inputs, so that normalising on the host rounds
    nothing that matters)."""
    from kimi_delta_attention_09_gb300 import _native
    case = _unnormalise(inputs.prefill_case([200, 70], H=2, K=128, V=128, dtype="f32", seed=956,
                                            init_std=0.02), 957)
    o1, f1 = _run(case)
    pre_q = torch.from_numpy(oracle.l2_normalize(case.q)).float()
    pre_k = torch.from_numpy(oracle.l2_normalize(case.k)).float()
    q, k, v, g, beta = (cuda(x) for x in (pre_q, pre_k, case.v, case.g, case.beta))
    out = torch.empty(v.shape, device="cuda")
    fin = torch.empty(case.N, case.H, 128, 128, device="cuda")
    _native.kda_chunk_prefill(q, k, v, g, beta, case.scale, cuda(case.init_state),
                              cuda(case.cu_seqlens), out, fin)
    torch.cuda.synchronize()
    assert rel_err(o1, out.cpu().double().numpy()) <= TOL["f32"]
    assert rel_err(f1, fin.cpu().double().numpy()) <= TOL["f32"]


def test_paged_prefill_normalises_rows():
    from kimi_delta_attention_09_gb300 import _native
    case = _unnormalise(inputs.prefill_case([70, 130], H=2, K=128, V=128, dtype="bf16", seed=958), 959)
    gen = torch.Generator().manual_seed(960)
    pool0 = (torch.randn(4, 2, 128, 128, generator=gen) * 0.05).float()
    slots = [3, 1]
    q, k, v, g, beta = (cuda(x) for x in (case.q, case.k, case.v, case.g, case.beta))
    pool = cuda(pool0)
    out = torch.empty(v.shape, device="cuda")
    _native.kda_chunk_prefill_paged(q, k, v, g, beta, case.scale, pool,
                                    torch.tensor(slots, dtype=torch.int32, device="cuda"),
                                    cuda(case.cu_seqlens), out, flags=_native.KDA_FLAG_QK_L2NORM)
    torch.cuda.synchronize()
    case.init_state = pool0[slots].clone()
    ref_out, ref_fin = _oracle(case)
    assert rel_err(out.cpu(), ref_out) <= TOL["bf16"]
    for n, s in enumerate(slots):
        assert rel_err(pool.cpu()[s], ref_fin[n]) <= TOL["bf16"]


@pytest.mark.parametrize("pool_dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dtype,K,V", [("bf16", 128, 128), ("f32", 64, 64)])
def test_decode_normalises_rows(pool_dtype, dtype, K, V):
    from kimi_delta_attention_09_gb300 import _native
    dc = inputs.decode_case(N=6, S=9, H=2, K=K, V=V, steps=3, dtype=dtype, seed=961)
    ref_pool = dc.pool.double().numpy().copy()
    pool = cuda(dc.pool if pool_dtype == "f32" else dc.pool.to(torch.bfloat16))
    if pool_dtype == "bf16":
        ref_pool = oracle.round_to_bf16(ref_pool)
    idx = cuda(dc.state_idx)
    fn = _native.kda_recurrent_decode if pool_dtype == "f32" else _native.kda_recurrent_decode_bf16_state
    ref_step = oracle.decode if pool_dtype == "f32" else oracle.decode_bf16_state
    gen = torch.Generator().manual_seed(962)
    for st in dc.steps:
        fq = 0.5 + 7.5 * torch.rand(st.q.shape[:-1] + (1,), generator=gen)
        fk = 0.5 + 7.5 * torch.rand(st.k.shape[:-1] + (1,), generator=gen)
        q = (st.q.float() * fq).to(st.q.dtype)
        k = (st.k.float() * fk).to(st.k.dtype)
        out = torch.empty(st.v.shape, dtype=torch.float32, device="cuda")
        fn(cuda(q), cuda(k), cuda(st.v), cuda(st.g), cuda(st.beta), dc.scale, pool, idx, out,
           flags=_native.KDA_FLAG_QK_L2NORM)
        ref = ref_step(q, k, st.v, st.g, st.beta, dc.scale, ref_pool, dc.state_idx.long().numpy(),
                       qk_l2norm=True)
        torch.cuda.synchronize()
        assert rel_err(out.cpu(), ref) <= TOL[dtype_name(st.q)]
    tol = TOL[dtype_name(dc.steps[0].q)] if pool_dtype == "f32" else 2.0 ** -6
    used = dc.state_idx.long().numpy()
    assert rel_err(pool.float().cpu().numpy()[used], ref_pool[used]) <= tol


def test_host_entry_normalises_rows():
    """kda_chunk_prefill_host passes the option to every piece's prefill."""
    import kimi_delta_attention_09_gb300 as kda
    case = _unnormalise(inputs.prefill_case([1, 63, 150, 65, 230], H=2, K=128, V=128, dtype="bf16",
                                            seed=958, init_std=0.02), 959)
    pin = [x.pin_memory() for x in (case.q, case.k, case.v, case.g, case.beta)]
    out, fin, _ = kda.chunk_prefill_from_host(*pin, case.scale, case.init_state.pin_memory(),
                                              case.cu_seqlens, out_dtype=torch.float32, segments=3,
                                              qk_l2norm=True)
    torch.cuda.synchronize()
    ref_out, ref_fin = _oracle(case)
    assert rel_err(out, ref_out) <= TOL["bf16"] and rel_err(fin, ref_fin) <= TOL["bf16"]
