"""Calls whose sequences hold no tokens at all (every sequence empty, so T = 0): the
prefill hands each initial state through unchanged, in place or to a separate final
state, on the tensor-core, CUDA-core, paged and host-to-host entry points; the conv keeps
every slot's taps bit-identical.  No kernel may touch q, k, v, g, beta or out (they have
no rows)."""
import pytest
import torch

from kimi_delta_attention_09_gb300 import inputs
from _helpers import cuda

pytestmark = pytest.mark.gpu


def _empty_case(dtype, K):
    return inputs.prefill_case([0, 0, 0], H=2, K=K, V=K, dtype=dtype, seed=601, init_std=0.05)


@pytest.mark.parametrize("dtype,K", [("bf16", 128), ("f32", 64)])
def test_prefill_passes_the_initial_states_through(dtype, K):
    from kimi_delta_attention_09_gb300 import _native
    case = _empty_case(dtype, K)
    assert case.T == 0
    q, k, v, g, beta = (cuda(x) for x in (case.q, case.k, case.v, case.g, case.beta))
    init = cuda(case.init_state)
    out = torch.empty(0, 2, K, device="cuda")
    fin = torch.full_like(init, float("nan"))
    n = _native.kda_chunk_prefill_workspace_bytes(case.N, 2, K, K, q.dtype)
    ws = torch.zeros(n, dtype=torch.uint8, device="cuda") if n else None
    _native.kda_chunk_prefill_ws(q, k, v, g, beta, case.scale, init, cuda(case.cu_seqlens), out, fin, ws)
    _native.kda_chunk_prefill(q, k, v, g, beta, case.scale, init, cuda(case.cu_seqlens), out, init)
    torch.cuda.synchronize()
    assert torch.equal(fin, init) and torch.equal(init.cpu(), case.init_state)


def test_paged_prefill_leaves_the_slots_as_they_are():
    from kimi_delta_attention_09_gb300 import _native
    case = _empty_case("bf16", 128)
    pool0 = torch.randn(5, 2, 128, 128, generator=torch.Generator().manual_seed(602))
    pool = cuda(pool0)
    idx = cuda(torch.tensor([4, 0, 2], dtype=torch.int32))
    q, k, v, g, beta = (cuda(x) for x in (case.q, case.k, case.v, case.g, case.beta))
    out = torch.empty(0, 2, 128, device="cuda")
    _native.kda_chunk_prefill_paged(q, k, v, g, beta, case.scale, pool, idx, cuda(case.cu_seqlens), out)
    torch.cuda.synchronize()
    assert torch.equal(pool.cpu().view(torch.int32), pool0.view(torch.int32))


def test_host_entry_passes_the_initial_states_through():
    from kimi_delta_attention_09_gb300 import _native
    case = _empty_case("bf16", 128)
    host = [x.pin_memory() for x in (case.q, case.k, case.v, case.g, case.beta)]
    init = case.init_state.pin_memory()
    out = torch.empty(0, 2, 128).pin_memory()
    fin = torch.full_like(case.init_state, float("nan")).pin_memory()
    n = _native.kda_chunk_prefill_host_device_bytes(0, case.N, 2, 128, 128, torch.bfloat16, torch.float32, 4)
    dev = torch.zeros(n, dtype=torch.uint8, device="cuda")
    _native.kda_chunk_prefill_host(*host, case.scale, init, case.cu_seqlens, out, fin, 4, dev)
    torch.cuda.synchronize()
    assert torch.equal(fin, case.init_state)


def test_conv_keeps_every_slot():
    from kimi_delta_attention_09_gb300 import _native
    cc = inputs.conv_case([0, 0], D=64, W=4, dtype="bf16", seed=603, slots=3)
    assert cc.x.shape[0] == 0
    taps = cuda(cc.conv_state)
    out = torch.empty(0, 64, dtype=torch.bfloat16, device="cuda")
    _native.kda_causal_conv1d_fwd(cuda(cc.x), cuda(cc.weight), cuda(cc.bias), taps, cuda(cc.state_idx),
                                  cuda(cc.cu_seqlens), out, activation=_native.KDA_CONV_ACT_SILU)
    torch.cuda.synchronize()
    assert torch.equal(taps.cpu().view(torch.int16), cc.conv_state.view(torch.int16))
