"""The causal convolution on the GPU through the C ABI against the fp64 oracle: outputs
within the parity bars (fp32 outputs; a bf16 output is exactly the rounded fp32 one),
carried taps bit-identical to the oracle's (they are copies of inputs), untouched slots
bit-identical, prompt-then-decode equal to the longer prompt, every width and both
activations, ragged and empty sequences, and the full-size varlen and decode workloads."""
import numpy as np
import pytest
import torch

from oracle import conv as oc
from kimi_delta_attention_09_gb300 import inputs
from _helpers import TOL, cuda, rel_err

pytestmark = pytest.mark.gpu


def _dname(t):
    return "bf16" if t.dtype == torch.bfloat16 else "f32"


def _run_prefill(case, act, out_dtype=torch.float32, with_state=True):
    from kimi_delta_attention_09_gb300 import _native
    x = cuda(case.x)
    st = cuda(case.conv_state) if with_state else None
    idx = cuda(case.state_idx) if with_state else None
    out = torch.full(x.shape, float("nan"), dtype=out_dtype, device="cuda")
    _native.kda_causal_conv1d_fwd(x, cuda(case.weight), cuda(case.bias), st, idx,
                                  cuda(case.cu_seqlens), out, activation=act)
    torch.cuda.synchronize()
    return out.cpu(), (st.cpu() if with_state else None)


def _oracle_prefill(case, act, with_state=True):
    st = case.conv_state.double().numpy().copy() if with_state else None
    y = oc.conv_prefill(case.x, case.weight, case.bias, st, case.state_idx.numpy(),
                        case.cu_seqlens.numpy(), activation=act)
    return y, st


def _rows(case):
    cu = case.cu_seqlens.tolist()
    return np.concatenate([np.arange(cu[n], cu[n + 1]) for n in range(len(cu) - 1)] + [np.zeros(0, int)])


@pytest.mark.parametrize("W", [1, 2, 3, 4])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("act", [oc.ACT_NONE, oc.ACT_SILU])
def test_prefill_matches_oracle(W, dtype, act):
    case = inputs.conv_case([1, 3, 0, 127, 128, 129, 300], D=264, W=W, dtype=dtype, seed=70 + W,
                            slots=11)
    out, st = _run_prefill(case, act)
    ref, ref_st = _oracle_prefill(case, act)
    rows = _rows(case)
    assert rel_err(out[rows], ref[rows]) <= TOL[dtype]
    # the carried taps are copies of inputs: bit-identical, and the other slots untouched
    assert torch.equal(st.float(), torch.from_numpy(ref_st).float())


def test_bf16_output_is_the_rounded_fp32_output():
    case = inputs.conv_case([50, 77], D=128, W=4, dtype="bf16", seed=80, slots=3)
    o32, _ = _run_prefill(case, oc.ACT_SILU)
    o16, _ = _run_prefill(case, oc.ACT_SILU, out_dtype=torch.bfloat16)
    assert torch.equal(o16.view(torch.int16), o32.to(torch.bfloat16).view(torch.int16))


def test_no_state_means_zero_taps():
    case = inputs.conv_case([40, 9], D=64, W=3, dtype="f32", seed=81)
    out, _ = _run_prefill(case, oc.ACT_NONE, with_state=False)
    ref, _ = _oracle_prefill(case, oc.ACT_NONE, with_state=False)
    assert rel_err(out, ref) <= TOL["f32"]


def test_out_of_range_slot_uses_zero_taps_and_keeps_nothing():
    case = inputs.conv_case([20, 30], D=64, W=4, dtype="bf16", seed=82, slots=4)
    case.state_idx = torch.tensor([9, 2], dtype=torch.int32)
    before = case.conv_state.clone()
    out, st = _run_prefill(case, oc.ACT_NONE)
    ref, ref_st = _oracle_prefill(case, oc.ACT_NONE)
    assert rel_err(out, ref) <= TOL["bf16"]
    for s in (0, 1, 3):
        assert torch.equal(st[s].view(torch.int16), before[s].view(torch.int16))


@pytest.mark.parametrize("W", [2, 4])
def test_prompt_then_decode_equals_the_longer_prompt(W):
    from kimi_delta_attention_09_gb300 import _native
    T0, steps, D = 150, 6, 256
    full = inputs.conv_case([T0 + steps], D=D, W=W, dtype="bf16", seed=83, slots=2)
    ref, ref_st = _oracle_prefill(full, oc.ACT_SILU)
    st = cuda(full.conv_state)
    idx = cuda(full.state_idx)
    w, b = cuda(full.weight), cuda(full.bias)
    x = cuda(full.x)
    out = torch.empty(x.shape, device="cuda")
    _native.kda_causal_conv1d_fwd(x[:T0].contiguous(), w, b, st, idx,
                                  torch.tensor([0, T0], dtype=torch.int32, device="cuda"),
                                  out[:T0], activation=oc.ACT_SILU)
    for t in range(T0, T0 + steps):
        o = torch.empty(1, D, device="cuda")
        _native.kda_causal_conv1d_update(x[t:t + 1].contiguous(), w, b, st, idx, o,
                                         activation=oc.ACT_SILU)
        out[t:t + 1] = o
    torch.cuda.synchronize()
    assert rel_err(out.cpu(), ref) <= TOL["bf16"]
    assert torch.equal(st.cpu().float(), torch.from_numpy(ref_st).float())


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("D,W", [(520, 4), (260, 4), (2056, 3), (12, 2)])
def test_update_matches_oracle(dtype, D, W):
    """8 channels per thread when D is a multiple of 8 (520, 2056: more than one CTA of
    channels), else 4 (260, 12)."""
    from kimi_delta_attention_09_gb300 import _native
    case = inputs.conv_case([1] * 37, D=D, W=W, dtype=dtype, seed=84, slots=64)
    st = cuda(case.conv_state)
    out = torch.empty(case.x.shape, device="cuda")
    _native.kda_causal_conv1d_update(cuda(case.x), cuda(case.weight), cuda(case.bias), st,
                                     cuda(case.state_idx), out, activation=oc.ACT_SILU)
    ref_st = case.conv_state.double().numpy().copy()
    ref = oc.conv_update(case.x, case.weight, case.bias, ref_st, case.state_idx.numpy(),
                         activation=oc.ACT_SILU)
    torch.cuda.synchronize()
    assert rel_err(out.cpu(), ref) <= TOL[dtype]
    assert torch.equal(st.cpu().double(), torch.from_numpy(ref_st))


def test_varlen_workload_full_size():
    case = inputs.conv_varlen()
    out, st = _run_prefill(case, oc.ACT_SILU)
    # the oracle on sampled channels of every sequence (the full size is 37 k x 12 k)
    ch = np.arange(0, case.x.shape[1], 97)
    sub = inputs.ConvCase(name="sub", seed=0, x=case.x[:, ch], weight=case.weight[ch],
                          bias=case.bias[ch], conv_state=case.conv_state[:, :, ch],
                          state_idx=case.state_idx, cu_seqlens=case.cu_seqlens)
    ref, ref_st = _oracle_prefill(sub, oc.ACT_SILU)
    assert rel_err(out[:, ch], ref) <= TOL["bf16"]
    assert torch.equal(st[:, :, ch].float(), torch.from_numpy(ref_st).float())


def test_decode_workload_full_size():
    from kimi_delta_attention_09_gb300 import _native
    case = inputs.conv_decode()
    st = cuda(case.conv_state)
    out = torch.empty(case.x.shape, device="cuda")
    _native.kda_causal_conv1d_update(cuda(case.x), cuda(case.weight), cuda(case.bias), st,
                                     cuda(case.state_idx), out, activation=oc.ACT_SILU)
    ref_st = case.conv_state.double().numpy().copy()
    ref = oc.conv_update(case.x, case.weight, case.bias, ref_st, case.state_idx.numpy(),
                         activation=oc.ACT_SILU)
    torch.cuda.synchronize()
    assert rel_err(out.cpu(), ref) <= TOL["bf16"]
    assert torch.equal(st.cpu().float(), torch.from_numpy(ref_st).float())
