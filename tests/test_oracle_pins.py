"""Pins for the fp64 oracle: facts fixed by the mathematics, not by the oracle's code.

Each pin is a function of an oracle implementation ``(prefill, decode)`` so that the
same checks run against the committed oracle and against deliberately broken copies
of it (``test_pins_catch_planted_mistakes``): a plausible mistake anywhere in the
recurrence (a dropped term, a wrong sign, the decay on the wrong axis, a transposed
read, the read-out taken before the write) must fail at least one pin.

The recurrence being pinned (gated delta rule with a per-key-channel decay):
    S_t = (I - beta_t k_t k_t^T) Diag(exp g_t) S_{t-1} + beta_t k_t v_t^T,
    o_t = scale * S_t^T q_t.
"""
import ctypes
import os
import shutil
import subprocess
import tempfile

import numpy as np
import pytest

import oracle
from oracle import chunked

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_example_T2_K2.txt")


def _rand_case(rng, T, H, K, V, unit_k=True, gate=0.3, beta_range=(0.0, 1.0)):
    q = rng.standard_normal((T, H, K))
    k = rng.standard_normal((T, H, K))
    if unit_k:
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
        q /= np.linalg.norm(q, axis=-1, keepdims=True)
    v = rng.standard_normal((T, H, V))
    g = -gate * np.log1p(np.exp(rng.standard_normal((T, H, K))))
    beta = rng.uniform(*beta_range, size=(T, H))
    return q, k, v, g, beta


# ----------------------------------------------------------------------------- pins

def pin_worked_example(prefill, decode):
    """Hand-derived two-token example (exact rationals), tests/golden."""
    vals = {}
    for line in open(GOLDEN):
        line = line.split("#", 1)[0].strip()
        if line:
            key, *nums = line.split()
            vals[key] = np.array([float(x) for x in nums])
    K = V = 2
    q = vals["q"].reshape(2, 1, K)
    k = vals["k"].reshape(2, 1, K)
    v = vals["v"].reshape(2, 1, V)
    g = np.log(vals["gate_exp"]).reshape(2, 1, K)
    beta = vals["beta"].reshape(2, 1)
    init = vals["init"].reshape(1, 1, K, V)
    out, final = prefill(q, k, v, g, beta, float(vals["scale"][0]), init, [0, 2])
    np.testing.assert_allclose(out.reshape(-1), vals["out"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(final.reshape(-1), vals["final"], rtol=0, atol=1e-12)


def pin_bruteforce_transition_products(prefill, decode):
    """S_T = (A_T...A_1) S_0 + sum_s (A_T...A_{s+1}) B_s with explicit matrices."""
    rng = np.random.default_rng(11)
    for (T, K, V) in [(1, 3, 2), (5, 4, 3), (8, 8, 8), (7, 2, 5)]:
        H = 2
        q, k, v, g, beta = _rand_case(rng, T, H, K, V)
        init = rng.standard_normal((1, H, K, V))
        scale = 0.7
        out, final = prefill(q, k, v, g, beta, scale, init, [0, T])
        for h in range(H):
            A = [(np.eye(K) - beta[t, h] * np.outer(k[t, h], k[t, h])) @ np.diag(np.exp(g[t, h]))
                 for t in range(T)]
            B = [beta[t, h] * np.outer(k[t, h], v[t, h]) for t in range(T)]
            for t in range(T):
                # state after token t from the explicit products
                prod_all = np.eye(K)
                for s in range(t + 1):
                    prod_all = A[s] @ prod_all
                S_t = prod_all @ init[0, h]
                for s in range(t + 1):
                    tail = np.eye(K)
                    for r in range(s + 1, t + 1):
                        tail = A[r] @ tail
                    S_t = S_t + tail @ B[s]
                np.testing.assert_allclose(out[t, h], scale * S_t.T @ q[t, h], rtol=0, atol=1e-12)
            np.testing.assert_allclose(final[0, h], S_t, rtol=0, atol=1e-12)


def pin_single_token_from_zero(prefill, decode):
    """From S_0 = 0 one token gives S_1 = beta k v^T and o = scale beta (k.q) v."""
    rng = np.random.default_rng(12)
    q, k, v, g, beta = _rand_case(rng, 1, 3, 6, 5, unit_k=False)
    out, final = prefill(q, k, v, g, beta, 0.3, None, [0, 1])
    for h in range(3):
        np.testing.assert_allclose(final[0, h], beta[0, h] * np.outer(k[0, h], v[0, h]),
                                   rtol=0, atol=1e-13)
        np.testing.assert_allclose(out[0, h], 0.3 * beta[0, h] * (k[0, h] @ q[0, h]) * v[0, h],
                                   rtol=0, atol=1e-13)


def pin_beta_zero_pure_channel_decay(prefill, decode):
    """beta = 0: S_t = Diag(exp(sum_{s<=t} g_s)) S_0 -- the decay acts on key rows."""
    rng = np.random.default_rng(13)
    T, H, K, V = 9, 2, 5, 3   # K != V so a decay on the wrong axis cannot pass
    q, k, v, g, beta = _rand_case(rng, T, H, K, V)
    beta[:] = 0.0
    init = rng.standard_normal((1, H, K, V))
    out, final = prefill(q, k, v, g, beta, 1.3, init, [0, T])
    cum = np.cumsum(g, axis=0)
    for t in range(T):
        for h in range(H):
            S_t = np.exp(cum[t, h])[:, None] * init[0, h]
            np.testing.assert_allclose(out[t, h], 1.3 * S_t.T @ q[t, h], rtol=0, atol=1e-12)
    for h in range(H):
        np.testing.assert_allclose(final[0, h], np.exp(cum[-1, h])[:, None] * init[0, h],
                                   rtol=0, atol=1e-12)


def pin_delta_rule_exact_readback(prefill, decode):
    """g = 0, beta = 1, unit k: right after token t the state returns v_t under k_t."""
    rng = np.random.default_rng(14)
    T, H, K, V = 6, 2, 4, 7
    q, k, v, g, beta = _rand_case(rng, T, H, K, V)
    g[:] = 0.0
    beta[:] = 1.0
    init = rng.standard_normal((1, H, K, V))
    out, _ = prefill(k.copy(), k, v, g, beta, 1.0, init, [0, T])  # query = key
    np.testing.assert_allclose(out, v, rtol=0, atol=1e-12)


def pin_scalar_gate_gauge(prefill, decode):
    """A gate constant over K (GDN's scalar decay) is a gauge of the ungated rule.

    With scalar per-step decay a_t and L_t = a_1...a_t, S_t = L_t R_t where R follows
    the delta rule with g = 0 on values v_t / L_t; hence o_t = L_t * o~_t.
    """
    rng = np.random.default_rng(15)
    T, H, K, V = 10, 2, 4, 3
    q, k, v, g, beta = _rand_case(rng, T, H, K, V)
    a = -rng.uniform(0.05, 0.6, size=(T, H))
    g = np.repeat(a[:, :, None], K, axis=2)
    L = np.exp(np.cumsum(a, axis=0))                   # [T, H]
    out, final = prefill(q, k, v, g, beta, 0.9, None, [0, T])
    out2, final2 = prefill(q, k, v / L[:, :, None], np.zeros_like(g), beta, 0.9, None, [0, T])
    np.testing.assert_allclose(out, L[:, :, None] * out2, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(final[0], L[-1][:, None, None] * final2[0], rtol=1e-12, atol=1e-13)


def pin_contraction(prefill, decode):
    """With unit k, beta in [0,1], g <= 0 and v = 0 the state norm never grows."""
    rng = np.random.default_rng(16)
    T, H, K, V = 12, 1, 6, 4
    q, k, v, g, beta = _rand_case(rng, T, H, K, V, gate=0.05)
    v[:] = 0.0
    S = rng.standard_normal((1, H, K, V))
    prev = np.linalg.norm(S)
    for t in range(T):
        _, S = prefill(q[t:t + 1], k[t:t + 1], v[t:t + 1], g[t:t + 1], beta[t:t + 1],
                       1.0, S, [0, 1])
        cur = np.linalg.norm(S)
        assert cur <= prev * (1 + 1e-14)
        prev = cur
    # and with beta = 1 the component along k_t is removed exactly
    _, S1 = prefill(q[:1], k[:1], v[:1], np.zeros_like(g[:1]), np.ones_like(beta[:1]),
                    1.0, rng.standard_normal((1, H, K, V)), [0, 1])
    np.testing.assert_allclose(S1[0, 0].T @ k[0, 0], np.zeros(V), atol=1e-13)


def pin_split_invariance(prefill, decode):
    """Prefill [0,T1) then [T1,T) from the carried state equals one prefill of [0,T)."""
    rng = np.random.default_rng(17)
    T, H, K, V = 23, 2, 5, 4
    q, k, v, g, beta = _rand_case(rng, T, H, K, V)
    init = rng.standard_normal((1, H, K, V)) * 0.1
    out, final = prefill(q, k, v, g, beta, 0.5, init, [0, T])
    for T1 in (1, 9, 22):
        o1, s1 = prefill(q[:T1], k[:T1], v[:T1], g[:T1], beta[:T1], 0.5, init, [0, T1])
        o2, s2 = prefill(q[T1:], k[T1:], v[T1:], g[T1:], beta[T1:], 0.5, s1, [0, T - T1])
        np.testing.assert_allclose(np.concatenate([o1, o2]), out, rtol=0, atol=1e-12)
        np.testing.assert_allclose(s2, final, rtol=0, atol=1e-12)


def pin_prefill_then_decode(prefill, decode):
    """Prefill a prompt, then decode token by token from a pool slot = full prefill."""
    rng = np.random.default_rng(18)
    T0, steps, H, K, V = 7, 5, 2, 4, 3
    T = T0 + steps
    q, k, v, g, beta = _rand_case(rng, T, H, K, V)
    out, final = prefill(q, k, v, g, beta, 0.8, None, [0, T])
    o_p, s_p = prefill(q[:T0], k[:T0], v[:T0], g[:T0], beta[:T0], 0.8, None, [0, T0])
    pool = rng.standard_normal((4, H, K, V))
    untouched = pool.copy()
    pool[2] = s_p[0]
    for t in range(T0, T):
        o = decode(q[t:t + 1], k[t:t + 1], v[t:t + 1], g[t:t + 1], beta[t:t + 1], 0.8,
                   pool, [2])
        np.testing.assert_allclose(o[0], out[t], rtol=0, atol=1e-12)
    np.testing.assert_allclose(pool[2], final[0], rtol=0, atol=1e-12)
    for s in (0, 1, 3):
        assert np.array_equal(pool[s], untouched[s])


def pin_varlen_and_heads_independent(prefill, decode):
    """Packing sequences and stacking heads changes nothing in each (sequence, head)."""
    rng = np.random.default_rng(19)
    lens = [3, 1, 6, 4]
    cu = np.concatenate([[0], np.cumsum(lens)])
    T, H, K, V = int(cu[-1]), 3, 4, 5
    q, k, v, g, beta = _rand_case(rng, T, H, K, V)
    init = rng.standard_normal((len(lens), H, K, V))
    out, final = prefill(q, k, v, g, beta, 0.6, init, cu)
    for n in range(len(lens)):
        s, e = cu[n], cu[n + 1]
        for h in range(H):
            o1, f1 = prefill(q[s:e, h:h + 1], k[s:e, h:h + 1], v[s:e, h:h + 1],
                             g[s:e, h:h + 1], beta[s:e, h:h + 1], 0.6,
                             init[n:n + 1, h:h + 1], [0, e - s])
            np.testing.assert_allclose(out[s:e, h], o1[:, 0], rtol=0, atol=1e-13)
            np.testing.assert_allclose(final[n, h], f1[0, 0], rtol=0, atol=1e-13)


PINS = [pin_worked_example, pin_bruteforce_transition_products, pin_single_token_from_zero,
        pin_beta_zero_pure_channel_decay, pin_delta_rule_exact_readback, pin_scalar_gate_gauge,
        pin_contraction, pin_split_invariance, pin_prefill_then_decode,
        pin_varlen_and_heads_independent]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_oracle_pin(pin):
    pin(oracle.prefill, oracle.decode)


# ------------------------------------------------------------- chunk-algebra pin

@pytest.mark.parametrize("chunk", [16, 64, 5])
def test_chunked_restatement_equals_recurrence(chunk):
    """The chunk-ordered algebra (gate cumsum, A_kk, solve, W/U, h, o) = the recurrence."""
    rng = np.random.default_rng(20 + chunk)
    lens = [37, 64, 1, 130]
    cu = np.concatenate([[0], np.cumsum(lens)])
    T, H, K, V = int(cu[-1]), 2, 8, 6
    q, k, v, g, beta = _rand_case(rng, T, H, K, V, gate=0.5)
    init = rng.standard_normal((len(lens), H, K, V)) * 0.3
    out, final = oracle.prefill(q, k, v, g, beta, 0.4, init, cu)
    out_c, final_c = chunked.prefill_chunked(q, k, v, g, beta, 0.4, init, cu, chunk=chunk)
    np.testing.assert_allclose(out_c, out, rtol=0, atol=1e-11 * np.abs(out).max())
    np.testing.assert_allclose(final_c, final, rtol=0, atol=1e-11 * np.abs(final).max())


@pytest.mark.parametrize("segments", [1, 2, 3, 5])
def test_segmented_restatement_equals_recurrence(segments):
    """Each sequence split in time into runs evaluated from a zero state, joined by the
    affine combine of their end maps: the recurrence's result for any split."""
    rng = np.random.default_rng(30 + segments)
    lengths = [1, 64, 200, 333, 0, 129]
    T, H, K, V = sum(lengths), 2, 8, 6
    cu = np.concatenate([[0], np.cumsum(lengths)])
    q, k = rng.standard_normal((2, T, H, K))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((T, H, V))
    g = -0.3 * rng.random((T, H, K))
    beta = rng.random((T, H))
    init = 0.1 * rng.standard_normal((len(lengths), H, K, V))
    ref_o, ref_f = oracle.prefill(q, k, v, g, beta, 0.4, init, cu)
    o, f = chunked.prefill_segmented(q, k, v, g, beta, 0.4, init, cu, chunk=16, segments=segments)
    assert np.abs(o - ref_o).max() <= 1e-10 * np.abs(ref_o).max()
    assert np.abs(f - ref_f).max() <= 1e-10 * np.abs(ref_f).max()


def test_chunked_restatement_strong_gates():
    """Gates down to -5 per step: the exact-exponential chunk algebra still agrees."""
    rng = np.random.default_rng(30)
    T, H, K, V = 70, 1, 6, 4
    q, k, v, g, beta = _rand_case(rng, T, H, K, V)
    g = -5.0 * rng.uniform(0, 1, size=g.shape)
    out, final = oracle.prefill(q, k, v, g, beta, 1.0, None, [0, T])
    out_c, final_c = chunked.prefill_chunked(q, k, v, g, beta, 1.0, None, [0, T], chunk=64)
    np.testing.assert_allclose(out_c, out, rtol=0, atol=1e-12 * max(1.0, np.abs(out).max()))
    np.testing.assert_allclose(final_c, final, rtol=0, atol=1e-12)


def test_oracle_thread_count_invariance():
    rng = np.random.default_rng(31)
    T, H, K, V = 40, 5, 8, 8
    q, k, v, g, beta = _rand_case(rng, T, H, K, V)
    o1, f1 = oracle.prefill(q, k, v, g, beta, 0.5, None, [0, 13, 40], nthreads=1)
    o2, f2 = oracle.prefill(q, k, v, g, beta, 0.5, None, [0, 13, 40], nthreads=7)
    assert np.array_equal(o1, o2) and np.array_equal(f1, f2)


def test_oracle_rejects_bad_slot():
    rng = np.random.default_rng(32)
    q, k, v, g, beta = _rand_case(rng, 1, 1, 2, 2)
    pool = np.zeros((3, 1, 2, 2))
    with pytest.raises(ValueError):
        oracle.decode(q, k, v, g, beta, 1.0, pool, [3])


# ----------------------------------------------------- planted mistakes (mutation)

MUTANTS = {
    # name: (text in kda_oracle.c, replacement)
    "decay_on_value_axis": ("const double a = exp(g[c]);\n        for (int64_t j = 0; j < V; ++j) S[c * V + j] *= a;",
                            "for (int64_t j = 0; j < V; ++j) S[c * V + j] *= exp(g[j % K]);"),
    "delta_sign": ("u[j] = beta * (v[j] - u[j]);", "u[j] = beta * (u[j] - v[j]);"),
    "beta_dropped": ("u[j] = beta * (v[j] - u[j]);", "u[j] = (v[j] - u[j]);"),
    "scale_dropped": ("o[j] *= scale;", "o[j] *= 1.0;"),
    "read_transposed": ("u[j] += S[c * V + j] * k[c];", "u[j] += S[(j % K) * V + (c % V)] * k[c];"),
    "decay_not_exponentiated": ("const double a = exp(g[c]);", "const double a = 1.0 + g[c];"),
    "no_decay_before_read": ("const double a = exp(g[c]);", "const double a = 1.0;"),
    "write_dropped": ("S[c * V + j] += k[c] * u[j];", "(void)0;"),
    "readout_uses_key": ("o[j] += S[c * V + j] * q[c];", "o[j] += S[c * V + j] * k[c];"),
    "init_ignored": ("if (J->init_state) memcpy", "if (0) memcpy"),
}


def _build_mutant(src_text, tmpdir, name):
    path = os.path.join(tmpdir, f"{name}.c")
    with open(path, "w") as f:
        f.write(src_text)
    so = os.path.join(tmpdir, f"lib{name}.so")
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-pthread", path, "-o", so,
                    "-lm"], check=True)
    return so


def _wrap(so_path):
    """(prefill, decode) functions with the oracle's Python contract over another .so."""
    lib = ctypes.CDLL(so_path)
    saved = oracle._lib
    dp = ctypes.POINTER(ctypes.c_double)
    ip = ctypes.POINTER(ctypes.c_int64)
    i64 = ctypes.c_int64
    lib.kda_oracle_prefill.argtypes = [i64, i64, i64, i64, dp, dp, dp, dp, dp, ctypes.c_double,
                                       dp, ip, dp, dp, ctypes.c_int]
    lib.kda_oracle_decode.argtypes = [i64, i64, i64, i64, i64, dp, dp, dp, dp, dp,
                                      ctypes.c_double, dp, ip, dp, ctypes.c_int]

    def call(fn, *a, **kw):
        oracle._lib = lib
        try:
            return fn(*a, **kw)
        finally:
            oracle._lib = saved
    return (lambda *a, **kw: call(oracle.prefill, *a, **kw),
            lambda *a, **kw: call(oracle.decode, *a, **kw))


def test_pins_catch_planted_mistakes():
    src = open(os.path.join(os.path.dirname(oracle.__file__), "kda_oracle.c")).read()
    tmpdir = tempfile.mkdtemp(prefix="kda_mutants_")
    try:
        for name, (old, new) in MUTANTS.items():
            assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
            prefill, decode = _wrap(_build_mutant(src.replace(old, new), tmpdir, name))
            caught = []
            for pin in PINS:
                try:
                    pin(prefill, decode)
                except (AssertionError, ValueError):
                    caught.append(pin.__name__)
            assert caught, f"no pin fails for the planted mistake '{name}'"
    finally:
        shutil.rmtree(tmpdir, ignore_errors=True)


# ------------------------------------------------------------------ bf16 state storage

def test_round_to_bf16_equals_the_fp32_to_bf16_conversion():
    """Every fp32 value (normal and subnormal, both signs, ties included) rounds to the
    bf16 value torch's round-to-nearest-even conversion gives."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(11)
    bits = rng.integers(0, 2 ** 32, size=200_000, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    x = x[np.isfinite(x)]
    ties = (np.arange(1, 5000, dtype=np.uint32) << 16 | 0x8000).view(np.float32)   # exact midpoints
    x = np.concatenate([x, ties, -ties, np.float32([0.0, 1e-45, -1e-45, 1.1754944e-38])])
    ref = torch.from_numpy(x.copy()).to(torch.bfloat16).to(torch.float64).numpy()
    got = oracle.round_to_bf16(x.astype(np.float64))
    assert np.array_equal(got, ref)


def test_round_to_bf16_ties_to_even():
    u = 2.0 ** -8   # half the bf16 step at 1
    got = oracle.round_to_bf16(np.array([1 + u, 1 + 3 * u, 1 + 2 * u, -(1 + u), 2 - u, 3.0]))
    assert got.tolist() == [1.0, 1 + 4 * u, 1 + 2 * u, -1.0, 2.0, 3.0]


def _bf16_case(seed, K=8, V=6, S=5):
    rng = np.random.default_rng(seed)
    pool = oracle.round_to_bf16(rng.standard_normal((S, 2, K, V)) * 0.3)
    q, k = rng.standard_normal((2, 2, 2, K))
    v = rng.standard_normal((2, 2, V))
    g = -0.2 * rng.random((2, 2, K))
    beta = rng.random((2, 2))
    return pool, q, k, v, g, beta, np.array([3, 0])


def test_bf16_state_decode_pins():
    # beta = 0, g = 0: the state is left as stored and the output reads it as it is
    pool, q, k, v, g, beta, idx = _bf16_case(1)
    start = pool.copy()
    out = oracle.decode_bf16_state(q, k, v, 0 * g, 0 * beta, 0.5, pool, idx)
    assert np.array_equal(pool, start)
    for n, s in enumerate(idx):
        assert np.allclose(out[n], 0.5 * np.einsum("hkv,hk->hv", start[s], q[n]), rtol=1e-14, atol=1e-14)
    # a unit key with beta = 1 and no decay replaces that key row by v exactly (v on the
    # bf16 grid), every other row and slot untouched
    pool, q, k, v, g, beta, idx = _bf16_case(2)
    start = pool.copy()
    k = np.zeros_like(k)
    k[:, :, 5] = 1.0
    v = oracle.round_to_bf16(v)
    oracle.decode_bf16_state(q, k, v, 0 * g, np.ones_like(beta), 0.5, pool, idx)
    for n, s in enumerate(idx):
        assert np.array_equal(pool[s][:, 5], v[n])
        assert np.array_equal(np.delete(pool[s], 5, axis=1), np.delete(start[s], 5, axis=1))
    for s in (1, 2, 4):
        assert np.array_equal(pool[s], start[s])
    # a general step: the stored state is on the bf16 grid, within half a bf16 step of the
    # fp64 step, and the output is the fp64 step's
    pool, q, k, v, g, beta, idx = _bf16_case(3)
    exact = pool.copy()
    out_exact = oracle.decode(q, k, v, g, beta, 0.5, exact, idx)
    out = oracle.decode_bf16_state(q, k, v, g, beta, 0.5, pool, idx)
    assert np.array_equal(out, out_exact)
    assert np.array_equal(oracle.round_to_bf16(pool), pool)
    _, e = np.frexp(exact)
    half_step = np.ldexp(1.0, np.maximum(e, -125) - 9)
    assert (np.abs(pool - exact) <= half_step).all()
    assert not np.array_equal(pool[idx], exact[idx])   # the rounding did happen
