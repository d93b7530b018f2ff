"""CPU pins of the oracle's in-kernel q/k L2 normalisation option (``qk_l2norm``).

The option is x / sqrt(sum_c x_c^2 + 1e-6) over the key dimension of every query and
key row, applied before the recurrence (the in-kernel half of the fused prologue of the
prompt path, vllm.cpp PR #110, commit description: chunk_kda_with_fused_gate; the
epsilon is not on the pages and is read as 1e-6).  Each pin below is a fact of that
definition that does not repeat its code: the closed form of the row norm, scale
invariance per row, no change to unit rows, finite zero rows, and the agreement of the
decode step with a one-token prefill.  Planted mistakes (the wrong axis, one of q and k
left out) fail the scale-invariance pin.
"""
import numpy as np
import pytest

import oracle
from kimi_delta_attention_09_gb300 import inputs


def _case(lens=(70, 33), H=3, K=16, V=8, seed=900):
    c = inputs.prefill_case(list(lens), H=H, K=K, V=V, dtype="f32", seed=seed, init_std=0.05)
    return c


def _row_factors(shape, seed, lo=0.5, hi=8.0):
    rng = np.random.default_rng(seed)
    return rng.uniform(lo, hi, size=shape[:-1] + (1,))


def test_normalised_rows_have_the_closed_form_norm():
    rng = np.random.default_rng(901)
    x = rng.standard_normal((50, 4, 32)) * rng.uniform(1e-3, 1e3, size=(50, 4, 1))
    y = oracle.l2_normalize(x)
    nx = np.linalg.norm(x, axis=-1)
    ny = np.linalg.norm(y, axis=-1)
    np.testing.assert_allclose(ny, nx / np.sqrt(nx ** 2 + 1e-6), rtol=1e-12, atol=0)
    # direction unchanged: y is a positive multiple of x
    cos = np.sum(x * y, axis=-1) / (nx * ny)
    np.testing.assert_allclose(cos, 1.0, rtol=0, atol=1e-12)


def _prefill(case, q, k, l2):
    return oracle.prefill(q, k, case.v, case.g, case.beta, case.scale, case.init_state,
                          case.cu_seqlens, qk_l2norm=l2)


def test_prefill_is_invariant_to_row_scales():
    c = _case()
    q, k = c.q.double().numpy(), c.k.double().numpy()
    o1, f1 = _prefill(c, q, k, True)
    o2, f2 = _prefill(c, q * _row_factors(q.shape, 902), k * _row_factors(k.shape, 903), True)
    # the only difference is eps / |x|^2 <= 1e-6 / 0.25 in each row's scale
    np.testing.assert_allclose(o2, o1, rtol=0, atol=2e-5 * np.abs(o1).max())
    np.testing.assert_allclose(f2, f1, rtol=0, atol=2e-5 * np.abs(f1).max())


def test_unit_rows_are_left_as_they_are():
    c = _case(seed=904)   # the generator's q and k rows are unit vectors
    q, k = c.q.double().numpy(), c.k.double().numpy()
    q = q / np.linalg.norm(q, axis=-1, keepdims=True)
    k = k / np.linalg.norm(k, axis=-1, keepdims=True)
    o1, f1 = _prefill(c, q, k, True)
    o0, f0 = _prefill(c, q, k, False)
    np.testing.assert_allclose(o1, o0, rtol=0, atol=3e-6 * np.abs(o0).max())
    np.testing.assert_allclose(f1, f0, rtol=0, atol=3e-6 * np.abs(f0).max())


def test_zero_rows_stay_zero_and_finite():
    c = _case(seed=905)
    q, k = c.q.double().numpy().copy(), c.k.double().numpy().copy()
    q[5] = 0.0
    k[9] = 0.0
    o1, f1 = _prefill(c, q, k, True)
    assert np.isfinite(o1).all() and np.isfinite(f1).all()
    qn, kn = oracle.l2_normalize(q), oracle.l2_normalize(k)
    assert np.all(qn[5] == 0.0) and np.all(kn[9] == 0.0)
    o0, f0 = _prefill(c, qn, kn, False)
    np.testing.assert_allclose(o1, o0, rtol=0, atol=1e-14)
    np.testing.assert_allclose(f1, f0, rtol=0, atol=1e-14)


def test_decode_step_equals_a_one_token_prefill():
    c = _case(lens=(1, 1, 1), H=2, K=16, V=8, seed=906)
    q = c.q.double().numpy() * _row_factors(c.q.shape, 907)
    k = c.k.double().numpy() * _row_factors(c.k.shape, 908)
    o_p, f_p = _prefill(c, q, k, True)
    pool = c.init_state.double().numpy().copy()
    o_d = oracle.decode(q, k, c.v, c.g, c.beta, c.scale, pool, np.arange(3), qk_l2norm=True)
    np.testing.assert_allclose(o_d, o_p, rtol=0, atol=1e-13)
    np.testing.assert_allclose(pool, f_p, rtol=0, atol=1e-13)


@pytest.mark.parametrize("mistake", ["head_axis", "q_only", "k_only"])
def test_pins_catch_planted_mistakes(mistake, monkeypatch):
    true_norm = oracle.l2_normalize
    calls = {"n": 0}

    def wrong(x):
        calls["n"] += 1
        x = np.asarray(x, dtype=np.float64)
        if mistake == "head_axis":
            return x / np.sqrt(np.sum(x * x, axis=1, keepdims=True) + 1e-6)
        if (mistake == "q_only" and calls["n"] % 2 == 0) or (mistake == "k_only" and calls["n"] % 2 == 1):
            return x
        return true_norm(x)

    monkeypatch.setattr(oracle, "l2_normalize", wrong)
    with pytest.raises(AssertionError):
        test_prefill_is_invariant_to_row_scales()
