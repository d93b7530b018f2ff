"""The runner's shape of the path, end to end on the GPU through the C ABI: the causal conv
over the packed [q|k|v] channels with taps in slots, the prompt's KDA prefill with its
states written into pool slots (q/k normalised in the kernel), then decode steps that
continue both carried states (conv taps and KDA state).  Each KDA stage is compared with
the fp64 oracle on the values the GPU conv produced (the conv is checked against its own
oracle), and slots no sequence uses stay bit-identical."""
import numpy as np
import pytest
import torch

import oracle
from oracle import conv as oc
from kimi_delta_attention_09_gb300 import inputs
from _helpers import TOL, cuda, rel_err

pytestmark = pytest.mark.gpu

H, K, W = 2, 128, 4
D = 3 * H * K


def _split(y, rows):
    """[rows, 3 H K] -> q, k, v [rows, H, K], contiguous (the chunk(3) view of the channels)."""
    y = y.view(rows, 3, H, K)
    return y[:, 0].contiguous(), y[:, 1].contiguous(), y[:, 2].contiguous()


def test_conv_prefill_then_decode_in_slots():
    from kimi_delta_attention_09_gb300 import _native
    lengths, slots, steps = [70, 1, 130], 6, 2
    N = len(lengths)
    cc = inputs.conv_case(lengths, D=D, W=W, dtype="bf16", seed=501, slots=slots)
    T = int(cc.cu_seqlens[-1])
    gen = torch.Generator().manual_seed(502)
    g = (-0.1 * torch.nn.functional.softplus(torch.randn(T, H, K, generator=gen))).contiguous()
    beta = torch.sigmoid(torch.randn(T, H, generator=gen)).contiguous()
    pool0 = (0.02 * torch.randn(slots, H, K, K, generator=gen)).contiguous()
    idx = cc.state_idx                     # the same slot keys both carried states
    scale = K ** -0.5

    taps = cuda(cc.conv_state)
    pool = cuda(pool0)
    y = torch.empty(T, D, dtype=torch.bfloat16, device="cuda")
    _native.kda_causal_conv1d_fwd(cuda(cc.x), cuda(cc.weight), cuda(cc.bias), taps, cuda(idx),
                                  cuda(cc.cu_seqlens), y, activation=_native.KDA_CONV_ACT_SILU)
    q, k, v = _split(y, T)
    out = torch.empty(T, H, K, dtype=torch.float32, device="cuda")
    _native.kda_chunk_prefill_paged(q, k, v, cuda(g), cuda(beta), scale, pool, cuda(idx),
                                    cuda(cc.cu_seqlens), out, flags=_native.KDA_FLAG_QK_L2NORM)
    torch.cuda.synchronize()

    # oracle: the conv on its own, then KDA on the GPU conv's values, states in slots
    ref_taps = cc.conv_state.double().numpy().copy()
    ref_y = oc.conv_prefill(cc.x, cc.weight, cc.bias, ref_taps, idx.long().numpy(),
                            cc.cu_seqlens.long().numpy(), activation=oc.ACT_SILU)
    assert rel_err(y.float().cpu(), ref_y) <= 2 ** -8   # bf16 output of the conv
    assert torch.equal(taps.cpu().double(), torch.from_numpy(ref_taps))
    qh, kh, vh = (t.cpu() for t in (q, k, v))
    ref_pool = pool0.double().numpy().copy()
    init = ref_pool[idx.long().numpy()]
    ref_out, ref_fin = oracle.prefill(qh, kh, vh, g, beta, scale, init, cc.cu_seqlens, qk_l2norm=True)
    ref_pool[idx.long().numpy()] = ref_fin
    assert rel_err(out.cpu(), ref_out) <= TOL["bf16"]
    assert rel_err(pool.cpu(), ref_pool) <= TOL["bf16"]

    # decode steps: the conv update continues the taps, the KDA step the pool slots
    for s in range(steps):
        x1 = torch.randn(N, D, generator=gen).to(torch.bfloat16)
        g1 = (-0.1 * torch.nn.functional.softplus(torch.randn(N, H, K, generator=gen))).contiguous()
        b1 = torch.sigmoid(torch.randn(N, H, generator=gen)).contiguous()
        y1 = torch.empty(N, D, dtype=torch.bfloat16, device="cuda")
        _native.kda_causal_conv1d_update(cuda(x1), cuda(cc.weight), cuda(cc.bias), taps, cuda(idx),
                                         y1, activation=_native.KDA_CONV_ACT_SILU)
        q1, k1, v1 = _split(y1, N)
        o1 = torch.empty(N, H, K, dtype=torch.float32, device="cuda")
        _native.kda_recurrent_decode(q1, k1, v1, cuda(g1), cuda(b1), scale, pool, cuda(idx), o1,
                                     flags=_native.KDA_FLAG_QK_L2NORM)
        torch.cuda.synchronize()
        ref_y1 = oc.conv_update(x1, cc.weight, cc.bias, ref_taps, idx.long().numpy(),
                                activation=oc.ACT_SILU)
        assert rel_err(y1.float().cpu(), ref_y1) <= 2 ** -8
        assert torch.equal(taps.cpu().double(), torch.from_numpy(ref_taps))
        rq, rk, rv = (t.cpu() for t in (q1, k1, v1))
        ref_o1 = oracle.decode(rq, rk, rv, g1, b1, scale, ref_pool, idx.long().numpy(), qk_l2norm=True)
        assert rel_err(o1.cpu(), ref_o1) <= TOL["bf16"]
        assert rel_err(pool.cpu(), ref_pool) <= TOL["bf16"]
    # slots no sequence uses were never touched
    unused = sorted(set(range(slots)) - set(idx.tolist()))
    assert torch.equal(pool.cpu()[unused].view(torch.int32), pool0[unused].view(torch.int32))
