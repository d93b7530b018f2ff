"""The calls only enqueue work (no host synchronisation, no allocation), so a serving loop
can capture them in a CUDA graph: a prefill on a caller workspace, a decode step and the
conv passes, captured once and replayed, give the same bits as the same calls run eagerly."""
import pytest
import torch

from kimi_delta_attention_09_gb300 import inputs

from _helpers import cuda

pytestmark = pytest.mark.gpu


def _prefill_args(case):
    from kimi_delta_attention_09_gb300 import _native
    q, k, v, g, beta = (cuda(x) for x in (case.q, case.k, case.v, case.g, case.beta))
    out = torch.empty(case.T, case.H, case.V, device="cuda")
    fin = torch.empty(case.N, case.H, case.K, case.V, device="cuda")
    ws = torch.zeros(_native.kda_chunk_prefill_workspace_bytes(case.N, case.H, case.K, case.V,
                                                               torch.bfloat16),
                     dtype=torch.uint8, device="cuda")
    return (q, k, v, g, beta, case.scale, cuda(case.init_state), cuda(case.cu_seqlens), out, fin, ws)


def test_prefill_decode_and_conv_replay_from_a_graph():
    from kimi_delta_attention_09_gb300 import _native
    case = inputs.prefill_case([150, 70], H=2, K=128, V=128, dtype="bf16", seed=401, init_std=0.02)
    pa = _prefill_args(case)
    dc = inputs.decode_case(N=3, S=6, H=2, K=128, V=128, steps=1, dtype="bf16", seed=402)
    st = dc.steps[0]
    dargs = [cuda(x) for x in (st.q, st.k, st.v, st.g, st.beta)]
    pool0 = cuda(dc.pool)
    idx = cuda(dc.state_idx)
    cc = inputs.conv_case([40, 9], D=96, W=4, dtype="bf16", seed=403, slots=3)
    taps0 = cuda(cc.conv_state)
    cargs = [cuda(x) for x in (cc.x, cc.weight, cc.bias)]
    ccu, cidx = cuda(cc.cu_seqlens), cuda(cc.state_idx)

    def run(pool, taps, dout, cout):
        _native.kda_chunk_prefill_ws(*pa)
        _native.kda_recurrent_decode(*dargs, dc.scale, pool, idx, dout)
        _native.kda_causal_conv1d_fwd(*cargs, taps, cidx, ccu, cout, activation=_native.KDA_CONV_ACT_SILU)

    # eager
    pool_e, taps_e = pool0.clone(), taps0.clone()
    dout_e = torch.empty(st.v.shape, device="cuda")
    cout_e = torch.empty(cc.x.shape, device="cuda")
    run(pool_e, taps_e, dout_e, cout_e)
    torch.cuda.synchronize()
    out_e, fin_e = pa[8].clone(), pa[9].clone()

    # captured once, replayed on fresh copies of the in-place state
    pool_g, taps_g = pool0.clone(), taps0.clone()
    dout_g = torch.empty_like(dout_e)
    cout_g = torch.empty_like(cout_e)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        run(pool_g, taps_g, dout_g, cout_g)   # warm-up outside the capture (first-use setup)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    pool_g.copy_(pool0)
    taps_g.copy_(taps0)
    pa[8].zero_()
    pa[9].zero_()
    with torch.cuda.graph(graph):
        run(pool_g, taps_g, dout_g, cout_g)
    graph.replay()
    torch.cuda.synchronize()
    assert _native.kda_chunk_prefill_status(pa[10]) == _native.KDA_OK
    assert torch.equal(pa[8], out_e) and torch.equal(pa[9], fin_e)
    assert torch.equal(dout_g, dout_e) and torch.equal(pool_g, pool_e)
    assert torch.equal(cout_g, cout_e) and torch.equal(taps_g, taps_e)
