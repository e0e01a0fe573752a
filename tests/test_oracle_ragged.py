"""Pins of the oracle's ragged windows (row r's tokens are
[cu_seqlens[r], cu_seqlens[r+1]) of one packed token list; LightLLM PR #1690,
commit messages on cu_seqlens windows; SGLang fork PR jianc99/sglang#2,
"Related upstream work" on packed ragged verify).

Each row is checked on its own against the pure-Python transition form
S_t = (I - beta k k^T) diag(e^g) S + beta k v^T: the window's outputs are the
chain's outputs from the committed state, and a commit of a tokens leaves the
chain's state after a tokens. Idle rows (no tokens) keep cursor and state.
"""
import numpy as np
import pytest

from oracle import ReplayOracle, ring
from test_oracle_pins import _brute_chain, _rand_tokens


def _row_tokens(toks, lo, hi):
    return [{key: val[t] for key, val in toks.items()} for t in range(lo, hi)]


@pytest.mark.parametrize("algo", ["gdn", "kda"])
@pytest.mark.parametrize("mode", [ring.LAZY, ring.FOLD_EVERY])
def test_ragged_windows_follow_the_transition_form(algo, mode):
    HK, HV, dk, dv, L, maxT, B = 1, 2, 2, 3, 5, 3, 5
    scale = 0.6
    rng = np.random.default_rng(500 + (algo == "kda") + 2 * mode)
    S0 = rng.standard_normal((1, B, HV, dk, dv)) * 0.3
    slots = np.array([2, -1, 0, 4, 1])
    orc = ReplayOracle(algo, 1, B, HK, HV, dk, dv, L, scale, S0)
    committed = {int(s): S0[0, s].tolist() for s in slots if s >= 0}
    for step in range(8):
        lens = rng.integers(0, maxT + 1, B)
        lens[step % B] = 0                       # at least one idle row per step
        cu = np.concatenate([[0], np.cumsum(lens)])
        toks = _rand_tokens(rng, int(cu[-1]), HK, HV, dk, dv, algo)
        force = (rng.random(B) < 0.2).astype(np.uint8)
        cur0 = orc.cursor.copy()
        o, flags = orc.window_ragged(0, slots, toks, cu, force)
        accept = np.array([rng.integers(0, n + 1) for n in lens])
        for r, s in enumerate(slots):
            if s < 0 or lens[r] == 0:
                assert flags[r] == -1
                assert np.all(np.isnan(o[cu[r]:cu[r + 1]]))
                continue
            fold, _ = ring.fold_decision(int(cur0[s]), int(lens[r]), L, bool(force[r]))
            assert flags[r] == int(fold)
            want_o, _ = _brute_chain(committed[s], _row_tokens(toks, cu[r], cu[r + 1]), scale,
                                     algo, HV // HK)
            np.testing.assert_allclose(o[cu[r]:cu[r + 1]], want_o, rtol=0, atol=1e-12)
        orc.commit_ragged(slots, accept, cu, force, mode)
        for r, s in enumerate(slots):
            if s < 0:
                continue
            if lens[r] == 0:
                assert orc.cursor[s] == cur0[s]
                continue
            if accept[r] > 0:
                _, S_new = _brute_chain(committed[s], _row_tokens(toks, cu[r], cu[r] + accept[r]),
                                        scale, algo, HV // HK)
                committed[s] = S_new.tolist()
            np.testing.assert_allclose(orc.S[0, s], np.array(committed[s]), rtol=0, atol=1e-12)
            assert orc.cursor[s] == ring.cursor_after_commit(int(cur0[s]), int(lens[r]), L,
                                                             bool(force[r]), int(accept[r]), mode)


def test_equal_lengths_are_the_uniform_window():
    """Ragged windows that all hold T tokens give the uniform window's results
    bit for bit (same tokens, same order of operations)."""
    HK, HV, dk, dv, L, T, B = 2, 4, 3, 2, 6, 3, 4
    rng = np.random.default_rng(77)
    S0 = rng.standard_normal((1, B, HV, dk, dv))
    slots = np.array([1, 3, -1, 0])
    a, b = (ReplayOracle("gdn", 1, B, HK, HV, dk, dv, L, 0.5, S0) for _ in range(2))
    cu = np.arange(B + 1) * T
    for step in range(5):
        toks = _rand_tokens(rng, B * T, HK, HV, dk, dv, "gdn")
        accept = rng.integers(0, T + 1, B)
        oa, fa = a.window(0, slots, toks, T)
        ob, fb = b.window_ragged(0, slots, toks, cu)
        assert np.array_equal(fa, fb)
        assert np.array_equal(oa, ob, equal_nan=True)
        a.commit(slots, accept, T)
        b.commit_ragged(slots, accept, cu)
        assert np.array_equal(a.S, b.S) and np.array_equal(a.cursor, b.cursor)


def test_ragged_rejects_bad_offsets():
    orc = ReplayOracle("gdn", 1, 2, 1, 1, 2, 2, 4, 1.0, np.zeros((1, 2, 1, 2, 2)))
    toks = _rand_tokens(np.random.default_rng(0), 6, 1, 1, 2, 2, "gdn")
    with pytest.raises(ValueError):
        orc.window_ragged(0, [0, 1], toks, [0, 3, 2])     # decreasing
    with pytest.raises(ValueError):
        orc.window_ragged(0, [0, 1], toks, [0, 5, 6])     # a window longer than L
