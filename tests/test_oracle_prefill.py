"""Pins of the oracle's replay prefill (LightLLM PR #1690, commit messages:
prefill writes the canonical state and leaves the cursor at zero).

Each row is checked against the pure-Python transition form from its
committed state (which may carry ring history), and against the invariant
that splitting a prompt into two prefills changes nothing.
"""
import numpy as np
import pytest

from oracle import ReplayOracle
from test_oracle_pins import _brute_chain, _rand_tokens


@pytest.mark.parametrize("algo", ["gdn", "kda"])
@pytest.mark.parametrize("ckpt_round", [None, "bf16"])
def test_prefill_follows_the_transition_form_from_the_committed_state(algo, ckpt_round):
    HK, HV, dk, dv, L, B = 1, 2, 3, 2, 4, 4
    rng = np.random.default_rng(900 + (algo == "kda") + 2 * (ckpt_round is not None))
    S0 = rng.standard_normal((1, B, HV, dk, dv)) * 0.3
    orc = ReplayOracle(algo, 1, B, HK, HV, dk, dv, L, 0.8, S0, ckpt_round=ckpt_round)
    slots = np.array([3, -1, 0, 2])
    # some decoded history first (rows keep records in their rings)
    for t in range(3):
        orc.decode(0, slots, _rand_tokens(rng, B, HK, HV, dk, dv, algo), advance=True)
    committed = {int(s): orc.S[0, s].copy() for s in slots if s >= 0}
    lens = np.array([5, 2, 0, 1])
    cu = np.concatenate([[0], np.cumsum(lens)])
    toks = _rand_tokens(rng, int(cu[-1]), HK, HV, dk, dv, algo)
    o = orc.prefill(0, slots, toks, cu)
    orc.prefill_done(slots, cu)
    for r, s in enumerate(slots):
        if s < 0:
            assert np.all(np.isnan(o[cu[r]:cu[r + 1]]))
            continue
        if lens[r] == 0:
            assert orc.cursor[s] == 3
            np.testing.assert_array_equal(orc.S[0, s], committed[s])
            continue
        tl = [{key: val[t] for key, val in toks.items()} for t in range(cu[r], cu[r + 1])]
        want_o, want_S = _brute_chain(committed[s].tolist(), tl, 0.8, algo, HV // HK)
        np.testing.assert_allclose(o[cu[r]:cu[r + 1]], want_o, rtol=0, atol=1e-12)
        if ckpt_round is None:
            np.testing.assert_allclose(orc.ckpt[0, s], want_S, rtol=0, atol=1e-12)
        else:   # the checkpoint holds the bf16-rounded result and the chain continues from it
            np.testing.assert_array_equal(orc.ckpt[0, s], orc.S[0, s])
            np.testing.assert_allclose(orc.S[0, s], want_S, rtol=2 ** -8, atol=0)
        assert orc.cursor[s] == 0


def test_a_prompt_split_in_two_prefills_is_one_prefill():
    HK, HV, dk, dv, L = 2, 4, 4, 3, 8
    rng = np.random.default_rng(31)
    S0 = rng.standard_normal((1, 1, HV, dk, dv))
    toks = _rand_tokens(rng, 23, HK, HV, dk, dv, "kda")
    one = ReplayOracle("kda", 1, 1, HK, HV, dk, dv, L, 0.5, S0)
    two = ReplayOracle("kda", 1, 1, HK, HV, dk, dv, L, 0.5, S0)
    o1 = one.prefill(0, [0], toks, [0, 23])
    first = {key: val[:9] for key, val in toks.items()}
    rest = {key: val[9:] for key, val in toks.items()}
    oa = two.prefill(0, [0], first, [0, 9])
    ob = two.prefill(0, [0], rest, [0, 14])
    np.testing.assert_allclose(np.concatenate([oa, ob]), o1, rtol=0, atol=1e-13)
    np.testing.assert_allclose(two.ckpt, one.ckpt, rtol=0, atol=1e-13)
