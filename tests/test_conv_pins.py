"""CPU pins of the causal-convolution oracle (``oracle.conv``), each checked against a
fact of the definition rather than its code: width 1 is a per-channel affine map, an
impulse returns the taps in reverse order, the SiLU closed form, a prompt split anywhere
and continued from its carried taps equals the unsplit prompt (exactly), decode steps
after a prompt equal the longer prompt, and packed sequences do not see each other.
Planted mistakes (an off-by-one window, a non-causal window, taps not carried) fail at
least one pin."""
import numpy as np
import pytest

from oracle import conv as oc


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def test_width_one_is_a_per_channel_affine_map():
    x = _rand((40, 12), 1)
    w = _rand((12, 1), 2)
    b = _rand(12, 3)
    y = oc.conv_prefill(x, w, b, None, None, [0, 40])
    np.testing.assert_array_equal(y, b + w[:, 0] * x)


@pytest.mark.parametrize("W", [2, 3, 4])
def test_impulse_returns_the_taps_reversed(W):
    D, T, t0 = 6, 20, 7
    w = _rand((D, W), 10 + W)
    x = np.zeros((T, D))
    x[t0, 2] = 1.0
    y = oc.conv_prefill(x, w, None, None, None, [0, T])
    for j in range(W):
        assert y[t0 + j, 2] == w[2, W - 1 - j]
    mask = np.ones_like(y, dtype=bool)
    mask[t0:t0 + W, 2] = False
    assert np.all(y[mask] == 0.0)   # causal and depthwise: nothing else moves


def test_silu_closed_form():
    x = np.array([[-3.0], [0.0], [0.5], [4.0]])
    w = np.ones((1, 1))
    y = oc.conv_prefill(x, w, None, None, None, [0, 4], activation=oc.ACT_SILU)
    np.testing.assert_allclose(y[:, 0], x[:, 0] / (1 + np.exp(-x[:, 0])), rtol=1e-15)
    assert y[1, 0] == 0.0


@pytest.mark.parametrize("W", [1, 2, 4])
@pytest.mark.parametrize("split", [1, 2, 5, 37])
def test_split_prompt_with_carried_taps_equals_the_whole(W, split):
    D, T = 8, 60
    x, w, b = _rand((T, D), 20), _rand((D, W), 21), _rand(D, 22)
    s0 = _rand((3, W - 1, D), 23)
    whole = s0.copy()
    y = oc.conv_prefill(x, w, b, whole, [1], [0, T], activation=oc.ACT_SILU)
    part = s0.copy()
    y1 = oc.conv_prefill(x[:split], w, b, part, [1], [0, split], activation=oc.ACT_SILU)
    y2 = oc.conv_prefill(x[split:], w, b, part, [1], [0, T - split], activation=oc.ACT_SILU)
    np.testing.assert_array_equal(np.concatenate([y1, y2]), y)
    np.testing.assert_array_equal(part, whole)
    # the other slots are untouched; the slot holds the last W - 1 inputs
    np.testing.assert_array_equal(whole[[0, 2]], s0[[0, 2]])
    if W > 1:
        np.testing.assert_array_equal(whole[1], x[T - (W - 1):])


def test_decode_steps_after_a_prompt_equal_the_longer_prompt():
    D, W, T0, steps = 8, 4, 9, 5
    x, w, b = _rand((T0 + steps, D), 30), _rand((D, W), 31), _rand(D, 32)
    s0 = _rand((2, W - 1, D), 33)
    whole = s0.copy()
    y = oc.conv_prefill(x, w, b, whole, [0], [0, T0 + steps])
    st = s0.copy()
    ys = [oc.conv_prefill(x[:T0], w, b, st, [0], [0, T0])]
    for t in range(T0, T0 + steps):
        ys.append(oc.conv_update(x[t:t + 1], w, b, st, [0]))
    np.testing.assert_array_equal(np.concatenate(ys), y)
    np.testing.assert_array_equal(st, whole)


def test_short_prompt_keeps_part_of_the_old_taps():
    D, W = 4, 4
    w = _rand((D, W), 40)
    s0 = _rand((1, W - 1, D), 41)
    x = _rand((1, D), 42)
    st = s0.copy()
    oc.conv_prefill(x, w, None, st, [0], [0, 1])
    np.testing.assert_array_equal(st[0], np.concatenate([s0[0, 1:], x]))


def test_packed_sequences_do_not_see_each_other():
    D, W = 5, 3
    lens = [4, 1, 0, 7]
    cu = np.concatenate([[0], np.cumsum(lens)])
    x, w = _rand((cu[-1], D), 50), _rand((D, W), 51)
    s0 = _rand((4, W - 1, D), 52)
    st = s0.copy()
    y = oc.conv_prefill(x, w, None, st, [3, 0, 1, 2], cu)
    for n in range(4):
        one = s0.copy()
        yn = oc.conv_prefill(x[cu[n]:cu[n + 1]], w, None, one, [[3, 0, 1, 2][n]], [0, lens[n]])
        np.testing.assert_array_equal(y[cu[n]:cu[n + 1]], yn)
        np.testing.assert_array_equal(st[[3, 0, 1, 2][n]], one[[3, 0, 1, 2][n]])


def _mutant(kind):
    def conv_prefill(x, weight, bias, conv_state, state_idx, cu_seqlens, activation=oc.ACT_NONE):
        x = np.asarray(x, dtype=np.float64)
        w = np.asarray(weight, dtype=np.float64)
        D, W = w.shape
        b = np.zeros(D) if bias is None else np.asarray(bias, dtype=np.float64)
        y = np.zeros_like(x)
        cu = [int(c) for c in cu_seqlens]
        for n in range(len(cu) - 1):
            s, e = cu[n], cu[n + 1]
            slot = None if conv_state is None else int(state_idx[n])
            taps = conv_state[slot].copy() if slot is not None else np.zeros((W - 1, D))
            xe = np.concatenate([taps, x[s:e], np.zeros((W, D))], axis=0)
            for t in range(e - s):
                acc = b.copy()
                for j in range(W):
                    k = t + j + (1 if kind == "off_by_one" else 0) + (W - 1 if kind == "future" else 0)
                    acc = acc + w[:, j] * xe[k]
                y[s + t] = oc._act(acc, activation)
            if slot is not None and W > 1 and kind != "no_carry":
                conv_state[slot] = xe[(e - s):(e - s) + W - 1]
        return y
    return conv_prefill


@pytest.mark.parametrize("kind", ["off_by_one", "future", "no_carry"])
def test_pins_catch_planted_mistakes(kind, monkeypatch):
    monkeypatch.setattr(oc, "conv_prefill", _mutant(kind))
    failed = 0
    for pin in (lambda: test_impulse_returns_the_taps_reversed(3),
                lambda: test_split_prompt_with_carried_taps_equals_the_whole(4, 5)):
        try:
            pin()
        except AssertionError:
            failed += 1
    assert failed >= 1
