"""Seeded synthetic inputs for the KDA prefill and decode workloads.

This module is the ONLY code that both the CUDA path's tests/benchmark and the CPU
oracle consume.  It draws random numbers and shapes them into the input recipe; it
holds none of the attention method's arithmetic.  Everything is generated on the CPU
with ``torch.Generator`` so that a (workload, seed) pair gives the same bits on any
machine; callers move the tensors to the device themselves.

Input recipe (the same value distributions for every workload):
  * q, k ~ N(0, 1), each L2-normalised over the key dimension (in fp32, then cast);
  * v ~ N(0, 1);
  * log-gate g = -gate_scale * softplus(z), z ~ N(0, 1)  (natural log, fp32);
  * beta = sigmoid(N(0, 1))  (fp32);
  * scale = 1 / sqrt(K);
  * initial / pool states ~ N(0, state_std^2) in fp32 (std 0.02 where nonzero).
Draw order: lengths, q, k, v, z, beta-logits, initial/pool state, decode slot
permutation, then the per-step decode inputs.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional

import torch
import torch.nn.functional as F

DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16}


@dataclass
class PrefillCase:
    name: str
    seed: int
    q: torch.Tensor            # [T, H, K]  dtype
    k: torch.Tensor            # [T, H, K]  dtype
    v: torch.Tensor            # [T, H, V]  dtype
    g: torch.Tensor            # [T, H, K]  fp32 natural-log gate
    beta: torch.Tensor         # [T, H]     fp32
    cu_seqlens: torch.Tensor   # [N+1]      int32
    init_state: Optional[torch.Tensor]  # [N, H, K, V] fp32 or None (zeros)
    scale: float

    @property
    def T(self) -> int:
        return self.q.shape[0]

    @property
    def N(self) -> int:
        return self.cu_seqlens.numel() - 1

    @property
    def H(self) -> int:
        return self.q.shape[1]

    @property
    def K(self) -> int:
        return self.q.shape[2]

    @property
    def V(self) -> int:
        return self.v.shape[2]


@dataclass
class DecodeStep:
    q: torch.Tensor     # [N, H, K]
    k: torch.Tensor     # [N, H, K]
    v: torch.Tensor     # [N, H, V]
    g: torch.Tensor     # [N, H, K] fp32
    beta: torch.Tensor  # [N, H] fp32


@dataclass
class DecodeCase:
    name: str
    seed: int
    pool: torch.Tensor        # [S, H, K, V] fp32
    state_idx: torch.Tensor   # [N] int32, distinct slots
    steps: List[DecodeStep] = field(default_factory=list)
    scale: float = 1.0

    @property
    def N(self) -> int:
        return self.state_idx.numel()


def _unit_rows(x: torch.Tensor) -> torch.Tensor:
    return x / x.norm(dim=-1, keepdim=True).clamp_min(1e-12)


def _draw_token_inputs(gen, T, H, K, V, dtype, gate_scale):
    q = _unit_rows(torch.randn(T, H, K, generator=gen)).to(dtype)
    k = _unit_rows(torch.randn(T, H, K, generator=gen)).to(dtype)
    v = torch.randn(T, H, V, generator=gen).to(dtype)
    z = torch.randn(T, H, K, generator=gen)
    g = (-gate_scale * F.softplus(z)).float().contiguous()
    beta = torch.sigmoid(torch.randn(T, H, generator=gen)).float().contiguous()
    return q.contiguous(), k.contiguous(), v.contiguous(), g, beta


def prefill_case(lengths, H: int, K: int, V: int, dtype: str = "bf16", seed: int = 0,
                 init_std: float = 0.0, gate_scale: float = 0.1,
                 name: str = "custom") -> PrefillCase:
    """Packed prefill inputs for sequences of the given lengths."""
    gen = torch.Generator().manual_seed(seed)
    lengths = [int(x) for x in lengths]
    cu = torch.zeros(len(lengths) + 1, dtype=torch.int32)
    if lengths:
        cu[1:] = torch.cumsum(torch.tensor(lengths, dtype=torch.int64), 0).to(torch.int32)
    T = int(cu[-1])
    q, k, v, g, beta = _draw_token_inputs(gen, T, H, K, V, DTYPES[dtype], gate_scale)
    init = None
    if init_std > 0.0:
        init = (torch.randn(len(lengths), H, K, V, generator=gen) * init_std).float()
    return PrefillCase(name=name, seed=seed, q=q, k=k, v=v, g=g, beta=beta,
                       cu_seqlens=cu, init_state=init, scale=K ** -0.5)


def decode_case(N: int, S: int, H: int, K: int, V: int, steps: int, dtype: str = "bf16",
                seed: int = 4, state_std: float = 0.02, gate_scale: float = 0.1,
                name: str = "custom_decode") -> DecodeCase:
    """Paged decode inputs: a pool of S slots, N distinct slots in use, `steps` tokens."""
    if N > S:
        raise ValueError("need N <= S distinct slots")
    gen = torch.Generator().manual_seed(seed)
    pool = (torch.randn(S, H, K, V, generator=gen) * state_std).float()
    idx = torch.randperm(S, generator=gen)[:N].to(torch.int32)
    case = DecodeCase(name=name, seed=seed, pool=pool, state_idx=idx, scale=K ** -0.5)
    for _ in range(steps):
        q, k, v, g, beta = _draw_token_inputs(gen, N, H, K, V, DTYPES[dtype], gate_scale)
        case.steps.append(DecodeStep(q=q, k=k, v=v, g=g, beta=beta))
    return case


# ---------------------------------------------------------------------------
# The five named workloads.  The seed of each is its index.
# ---------------------------------------------------------------------------

def tiny_f32() -> PrefillCase:
    """B=1, H=2, T=128, K=V=64, fp32, zero initial state."""
    return prefill_case([128], H=2, K=64, V=64, dtype="f32", seed=0, name="tiny_f32_T128_H2_D64")


def single_prompt(T: int = 4096) -> PrefillCase:
    """B=1, H=32, T=4096, K=V=128, bf16 q/k/v, zero initial state."""
    return prefill_case([T], H=32, K=128, V=128, dtype="bf16", seed=1,
                        name=f"single_prompt_T{T}_H32_D128_bf16")


def varlen_packed() -> PrefillCase:
    """8 sequences, lengths ~ U[256, 8192] (seeded), packed; init ~ N(0, 0.02^2)."""
    seed = 2
    gen = torch.Generator().manual_seed(seed)
    lengths = [int(x) for x in torch.randint(256, 8192 + 1, (8,), generator=gen)]
    # the lengths are the first draw; the other inputs continue on the same generator
    return _prefill_after_lengths(gen, lengths, H=32, K=128, V=128, dtype="bf16",
                                  init_std=0.02, seed=seed,
                                  name="varlen_packed_N8_H32_D128_bf16")


def long_prefill(T: int = 65536) -> PrefillCase:
    """B=1, H=32, T=65536, K=V=128, bf16 q/k/v, zero initial state."""
    return prefill_case([T], H=32, K=128, V=128, dtype="bf16", seed=3,
                        name=f"long_prefill_T{T}_H32_D128_bf16")


def paged_decode(steps: int = 64) -> DecodeCase:
    """256 sequences x 1 token, H=32, K=V=128, bf16; pool of 1024 fp32 slots."""
    return decode_case(N=256, S=1024, H=32, K=128, V=128, steps=steps, dtype="bf16",
                       seed=4, state_std=0.02, name="paged_decode_N256_S1024_H32_D128_bf16")


def _prefill_after_lengths(gen, lengths, H, K, V, dtype, init_std, seed, name):
    cu = torch.zeros(len(lengths) + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.tensor(lengths, dtype=torch.int64), 0).to(torch.int32)
    T = int(cu[-1])
    q, k, v, g, beta = _draw_token_inputs(gen, T, H, K, V, DTYPES[dtype], 0.1)
    init = (torch.randn(len(lengths), H, K, V, generator=gen) * init_std).float()
    return PrefillCase(name=name, seed=seed, q=q, k=k, v=v, g=g, beta=beta,
                       cu_seqlens=cu, init_state=init, scale=K ** -0.5)


@dataclass
class ConvCase:
    name: str
    seed: int
    x: torch.Tensor            # [T, D]  dtype (the packed [q|k|v] channels)
    weight: torch.Tensor       # [D, W]  fp32
    bias: torch.Tensor         # [D]     fp32
    conv_state: torch.Tensor   # [S, W-1, D] dtype (carried taps per slot)
    state_idx: torch.Tensor    # [N] int32, distinct slots
    cu_seqlens: torch.Tensor   # [N+1] int32


def conv_case(lengths, D: int, W: int, dtype: str = "bf16", seed: int = 0, slots: int = 0,
              name: str = "custom_conv") -> ConvCase:
    """Causal-conv inputs: x ~ N(0, 1); weight ~ N(0, 1 / W); bias ~ N(0, 0.1^2); a pool
    of max(slots, N) carried-tap slots ~ N(0, 1); N distinct slots drawn by permutation.
    Draw order: x, weight, bias, taps, slot permutation."""
    gen = torch.Generator().manual_seed(seed)
    lengths = [int(x) for x in lengths]
    cu = torch.zeros(len(lengths) + 1, dtype=torch.int32)
    if lengths:
        cu[1:] = torch.cumsum(torch.tensor(lengths, dtype=torch.int64), 0).to(torch.int32)
    T = int(cu[-1])
    S = max(slots, len(lengths))
    x = torch.randn(T, D, generator=gen).to(DTYPES[dtype]).contiguous()
    weight = (torch.randn(D, W, generator=gen) / W ** 0.5).float().contiguous()
    bias = (torch.randn(D, generator=gen) * 0.1).float().contiguous()
    state = torch.randn(S, max(W - 1, 0), D, generator=gen).to(DTYPES[dtype]).contiguous()
    idx = torch.randperm(S, generator=gen)[:len(lengths)].to(torch.int32)
    return ConvCase(name=name, seed=seed, x=x, weight=weight, bias=bias, conv_state=state,
                    state_idx=idx, cu_seqlens=cu)


def conv_varlen(W: int = 4) -> ConvCase:
    """The varlen packed workload's lengths (8 sequences, U[256, 8192], seed 2) over its
    [q|k|v] channels (3 x 32 heads x 128 = 12,288), taps carried in 8 slots, width 4."""
    gen = torch.Generator().manual_seed(2)
    lengths = [int(x) for x in torch.randint(256, 8192 + 1, (8,), generator=gen)]
    return conv_case(lengths, D=3 * 32 * 128, W=W, dtype="bf16", seed=5, slots=8,
                     name=f"conv_varlen_N8_D12288_W{W}_bf16")


def conv_decode(W: int = 4) -> ConvCase:
    """One token for each of 256 sequences over 12,288 channels, taps in 1024 slots."""
    return conv_case([1] * 256, D=3 * 32 * 128, W=W, dtype="bf16", seed=6, slots=1024,
                     name=f"conv_decode_N256_S1024_D12288_W{W}_bf16")


WORKLOADS = {
    "tiny_f32": tiny_f32,
    "single_prompt": single_prompt,
    "varlen_packed": varlen_packed,
    "long_prefill": long_prefill,
    "paged_decode": paged_decode,
}
