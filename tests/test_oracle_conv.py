"""Pins of the conv-window oracle against numpy.convolve, brute-force
re-computation over the whole token history, and the rollback rule."""
import numpy as np
import pytest

from oracle.conv import ACT_NONE, ACT_SILU, ConvOracle


def _np_causal(seq, w, bias, act):
    """Per channel: numpy.convolve of the whole sequence with the reversed
    kernel, keeping the outputs whose window lies fully inside."""
    K = w.shape[1]
    out = np.zeros((seq.shape[0] - K + 1, seq.shape[1]))
    for c in range(seq.shape[1]):
        out[:, c] = np.convolve(seq[:, c], w[c, ::-1], mode="valid")
    if bias is not None:
        out += bias
    if act == ACT_SILU:
        out = out / (1.0 + np.exp(-out))
    return out


@pytest.mark.parametrize("K", [2, 4])
@pytest.mark.parametrize("act", [ACT_NONE, ACT_SILU])
def test_chain_of_verifies_equals_one_convolution_of_the_accepted_history(K, act):
    rng = np.random.default_rng(10 * K + act)
    D, B, T = 5, 3, 4
    slots = np.array([2, -1, 0])
    w = rng.standard_normal((D, K))
    bias = rng.standard_normal(D)
    win0 = rng.standard_normal((3, K - 1, D))
    orc = ConvOracle(win0, w, bias, act)
    history = {s: [win0[s]] for s in (0, 2)}
    for step in range(6):
        x = rng.standard_normal((B * T, D))
        acc = rng.integers(0, T + 1, B)
        y = orc.window_step(slots, x, T)
        for r, s in enumerate(slots):
            if s < 0:
                assert np.all(np.isnan(y[r * T:(r + 1) * T]))
                continue
            seq = np.concatenate(history[s] + [x[r * T:(r + 1) * T]])
            want = _np_causal(seq, w, bias, act)[-T:]
            np.testing.assert_allclose(y[r * T:(r + 1) * T], want, rtol=0, atol=1e-12)
            history[s].append(x[r * T:r * T + acc[r]])
        orc.commit(slots, acc)
        for s in (0, 2):
            seq = np.concatenate(history[s])
            np.testing.assert_array_equal(orc.window[s], seq[-(K - 1):])


def test_decode_is_a_one_token_window_accepted():
    rng = np.random.default_rng(3)
    D, K = 4, 4
    w = rng.standard_normal((D, K))
    a = ConvOracle(rng.standard_normal((1, K - 1, D)), w, None, ACT_SILU)
    b = ConvOracle(a.window.copy(), w, None, ACT_SILU)
    xs = rng.standard_normal((7, D))
    ya = np.concatenate([a.decode([0], xs[t:t + 1]) for t in range(7)])
    yb = b.window_step([0], xs, 7)
    b.commit([0], [7])
    np.testing.assert_allclose(ya, yb, rtol=0, atol=1e-13)
    np.testing.assert_array_equal(a.window, b.window)


def test_rejecting_everything_keeps_the_window():
    rng = np.random.default_rng(4)
    orc = ConvOracle(rng.standard_normal((2, 3, 6)), rng.standard_normal((6, 4)))
    before = orc.window.copy()
    orc.window_step([1, 0], rng.standard_normal((2 * 5, 6)), 5)
    orc.commit([1, 0], [0, 0])
    np.testing.assert_array_equal(orc.window, before)
