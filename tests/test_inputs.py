"""The seeded input generator: determinism, shapes, dtypes and value ranges."""
import torch

from kimi_delta_attention_09_gb300 import inputs


def test_deterministic_and_shaped():
    a = inputs.prefill_case([5, 70, 64], H=3, K=16, V=8, dtype="bf16", seed=9, init_std=0.02)
    b = inputs.prefill_case([5, 70, 64], H=3, K=16, V=8, dtype="bf16", seed=9, init_std=0.02)
    for x, y in [(a.q, b.q), (a.k, b.k), (a.v, b.v), (a.g, b.g), (a.beta, b.beta),
                 (a.init_state, b.init_state), (a.cu_seqlens, b.cu_seqlens)]:
        assert torch.equal(x, y)
    assert a.q.shape == (139, 3, 16) and a.q.dtype == torch.bfloat16
    assert a.v.shape == (139, 3, 8) and a.g.dtype == torch.float32
    assert a.cu_seqlens.tolist() == [0, 5, 75, 139] and a.cu_seqlens.dtype == torch.int32
    assert a.init_state.shape == (3, 3, 16, 8)
    assert abs(a.scale - 16 ** -0.5) < 1e-15


def test_value_ranges():
    c = inputs.tiny_f32()
    assert c.q.dtype == torch.float32 and c.init_state is None
    n = c.k.norm(dim=-1)
    assert torch.allclose(n, torch.ones_like(n), atol=1e-6)
    assert (c.g <= 0).all() and (c.g > -2).all()
    assert (c.beta > 0).all() and (c.beta < 1).all()


def test_varlen_lengths_in_range():
    gen = torch.Generator().manual_seed(2)
    lengths = torch.randint(256, 8193, (8,), generator=gen)
    assert ((lengths >= 256) & (lengths <= 8192)).all()


def test_decode_case_distinct_slots():
    d = inputs.decode_case(N=10, S=16, H=2, K=8, V=4, steps=3, seed=1)
    assert d.state_idx.unique().numel() == 10
    assert (d.state_idx >= 0).all() and (d.state_idx < 16).all()
    assert len(d.steps) == 3 and d.steps[0].q.shape == (10, 2, 8)
