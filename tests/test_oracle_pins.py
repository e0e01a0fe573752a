"""Pins of the fp64 oracle against closed forms, other formulations and
special cases (none of them retypes the oracle's own update).

* single rank-1 step: S'^T k = (1 - beta) e^g S^T k + beta v for ||k|| = 1;
* the transition-matrix form S_t = (I - beta k k^T) diag(e^g) S + beta k v^T,
  written with pure-Python lists on tiny non-square shapes;
* the window's triangular form (I + A)^-1 R solved by numpy.linalg.solve, the
  form the CUDA path evaluates;
* the replay identity: checkpoint plus ring records reproduce the state;
* ring invariants: no ring (L = inf) == any L, forced folds change nothing,
  rejected drafts are inert;
* special cases: g = 0 and beta = 0 is a pure read; g = -inf forgets history;
  KDA with equal channel gates is GDN; key-head sharing is h // G.
"""
import math

import numpy as np
import pytest

import synth
from oracle import ReplayOracle, ring, token_step


# ----------------------------------------------------------------- utilities
def _rand_tokens(rng, n, HK, HV, dk, dv, algo, beta=None, g=None):
    q = rng.standard_normal((n, HK, dk))
    k = rng.standard_normal((n, HK, dk))
    q /= np.linalg.norm(q, axis=-1, keepdims=True)
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((n, HV, dv))
    b = rng.uniform(0.05, 0.95, (n, HV)) if beta is None else np.full((n, HV), beta)
    gs = (n, HV) if algo == "gdn" else (n, HV, dk)
    gg = -rng.uniform(0.0, 1.5, gs) if g is None else np.full(gs, g)
    return {"q": q, "k": k, "v": v, "beta": b, "g": gg}


def _slice(inp, lo, hi):
    return {key: val[lo:hi] for key, val in inp.items()}


def _brute_chain(S0, toks, scale, algo, G):
    """Transition-matrix form in pure Python; S0 is [HV][dk][dv] lists."""
    HV, dk, dv = len(S0), len(S0[0]), len(S0[0][0])
    S = [[row[:] for row in Sh] for Sh in S0]
    outs = []
    for t in toks:
        o_t = []
        for h in range(HV):
            kh = h // G
            k = list(t["k"][kh])
            q = list(t["q"][kh])
            v = list(t["v"][h])
            beta = float(t["beta"][h])
            if algo == "gdn":
                dec = [math.exp(float(t["g"][h]))] * dk
            else:
                dec = [math.exp(float(x)) for x in t["g"][h]]
            # P = I - beta k k^T ; M = P diag(dec)
            M = [[((1.0 if i == j else 0.0) - beta * k[i] * k[j]) * dec[j]
                  for j in range(dk)] for i in range(dk)]
            MS = [[sum(M[i][m] * S[h][m][j] for m in range(dk)) for j in range(dv)]
                  for i in range(dk)]
            S[h] = [[MS[i][j] + beta * k[i] * v[j] for j in range(dv)] for i in range(dk)]
            o_t.append([scale * sum(S[h][i][j] * q[i] for i in range(dk))
                        for j in range(dv)])
        outs.append(o_t)
    return np.array(outs), np.array(S)


# ------------------------------------------------------ 1. rank-1 closed form
@pytest.mark.parametrize("beta", [0.0, 0.37, 1.0])
def test_single_rank1_closed_form(beta):
    rng = np.random.default_rng(1)
    R, HV, dk, dv = 3, 2, 5, 7
    S = rng.standard_normal((R, HV, dk, dv))
    k = rng.standard_normal((R, HV, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    q = rng.standard_normal((R, HV, dk))
    v = rng.standard_normal((R, HV, dv))
    g = -rng.uniform(0, 2, (R, HV))
    b = np.full((R, HV), beta)
    S1, d, o = token_step(S, q, k, v, b, g, 0.5, "gdn")
    Stk = np.einsum("rhkv,rhk->rhv", S, k)
    want = (1 - beta) * np.exp(g)[..., None] * Stk + beta * v
    np.testing.assert_allclose(np.einsum("rhkv,rhk->rhv", S1, k), want, atol=1e-13)
    if beta == 1.0:   # delta-rule write: reading back along k gives v
        np.testing.assert_allclose(np.einsum("rhkv,rhk->rhv", S1, k), v, atol=1e-13)
    if beta == 0.0:   # pure decay
        np.testing.assert_allclose(S1, np.exp(g)[..., None, None] * S, atol=1e-15)
    np.testing.assert_allclose(o, 0.5 * np.einsum("rhkv,rhk->rhv", S1, q), atol=1e-13)


# ----------------------------------------- 2. transition-matrix brute force
@pytest.mark.parametrize("algo", ["gdn", "kda"])
@pytest.mark.parametrize("dims", [(1, 1), (2, 3), (3, 2), (3, 3)])
def test_brute_force_transition_form(algo, dims):
    dk, dv = dims
    HK, HV, L, steps = 1, 2, 3, 9
    rng = np.random.default_rng(100 + dk * 10 + dv)
    S0 = rng.standard_normal((1, HV, dk, dv)) * 0.3
    toks = _rand_tokens(rng, steps, HK, HV, dk, dv, algo)
    orc = ReplayOracle(algo, 1, 1, HK, HV, dk, dv, L, 0.7, S0)
    outs = []
    for t in range(steps):
        o, _ = orc.decode(0, [0], _slice(toks, t, t + 1), advance=True)
        outs.append(o[0])
    tok_list = [{key: val[t] for key, val in toks.items()} for t in range(steps)]
    want_o, want_S = _brute_chain(S0[0].tolist(), tok_list, 0.7, algo, HV // HK)
    np.testing.assert_allclose(np.array(outs), want_o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(orc.S[0, 0], want_S, rtol=0, atol=1e-12)


# --------------------------------- 3. window triangular form (I + A)^-1 R
def _window_form(Sbar, toks, T, scale, algo, G):
    """Outputs of one window from the state Sbar via the triangular solve."""
    HV, dk, dv = Sbar.shape
    out = np.zeros((T, HV, dv))
    for h in range(HV):
        kh = h // G
        K = toks["k"][:, kh]          # [T, dk]
        Q = toks["q"][:, kh]
        V = toks["v"][:, h]
        b = toks["beta"][:, h]
        g = toks["g"][:, h]
        Gp = np.cumsum(g, axis=0)     # inclusive in-window prefix (T) or (T, dk)
        if algo == "gdn":
            decK = np.exp(Gp)[:, None] * K
            decQ = np.exp(Gp)[:, None] * Q
            W = lambda i, j, x: np.exp(Gp[i] - Gp[j]) * (K[j] @ x)  # noqa: E731
        else:
            decK = np.exp(Gp) * K
            decQ = np.exp(Gp) * Q
            W = lambda i, j, x: np.sum(np.exp(Gp[i] - Gp[j]) * K[j] * x)  # noqa: E731
        A = np.zeros((T, T))
        for i in range(T):
            for j in range(i):
                A[i, j] = b[i] * W(i, j, K[i])
        R = b[:, None] * (V - decK @ Sbar[h])
        D = np.linalg.solve(np.eye(T) + A, R)
        for i in range(T):
            acc = decQ[i] @ Sbar[h]
            for j in range(i + 1):
                acc = acc + W(i, j, Q[i]) * D[j]
            out[i, h] = scale * acc
    return out


@pytest.mark.parametrize("algo", ["gdn", "kda"])
@pytest.mark.parametrize("T", [1, 3, 6])
def test_window_triangular_form(algo, T):
    HK, HV, dk, dv = 2, 4, 5, 3
    rng = np.random.default_rng(7 * T + (algo == "kda"))
    S0 = rng.standard_normal((1, HV, dk, dv)) * 0.2
    orc = ReplayOracle(algo, 1, 1, HK, HV, dk, dv, 8, 0.4, S0)
    # some committed history first
    for t in range(3):
        orc.decode(0, [0], _rand_tokens(rng, 1, HK, HV, dk, dv, algo), advance=True)
    Sbar = orc.S[0, 0].copy()
    toks = _rand_tokens(rng, T, HK, HV, dk, dv, algo)
    o, _ = orc.window(0, [0], toks, T)
    want = _window_form(Sbar, toks, T, 0.4, algo, HV // HK)
    np.testing.assert_allclose(o, want, rtol=0, atol=1e-12)


# ---------------------------------------------------- 4. replay identity
@pytest.mark.parametrize("algo", ["gdn", "kda"])
def test_checkpoint_plus_ring_replays_state(algo):
    """S = e^Gamma ckpt + sum_h e^(Gamma - Gamma_h) k_h d_h^T over the ring,
    with Gamma_h the inclusive prefix of the record gates."""
    HK, HV, dk, dv, L = 1, 2, 4, 3, 6
    rng = np.random.default_rng(11)
    S0 = rng.standard_normal((1, 1, HV, dk, dv))
    orc = ReplayOracle(algo, 1, 1, HK, HV, dk, dv, L, 1.0, S0)
    for t in range(17):   # crosses several folds
        orc.decode(0, [0], _rand_tokens(rng, 1, HK, HV, dk, dv, algo), advance=True)
        c = int(orc.cursor[0])
        for h in range(HV):
            gam = np.cumsum(orc.ring_g[0, 0, h, :c], axis=0)
            total = gam[-1] if c else (0.0 if algo == "gdn" else np.zeros(dk))
            if algo == "gdn":
                S = np.exp(total) * orc.ckpt[0, 0, h]
            else:
                S = np.exp(total)[:, None] * orc.ckpt[0, 0, h]
            for m in range(c):
                km = orc.ring_k[0, 0, h // (HV // HK), m]
                fac = np.exp(total - gam[m])
                kt = fac * km
                S = S + np.outer(kt, orc.ring_d[0, 0, h, m])
            np.testing.assert_allclose(S, orc.S[0, 0, h], rtol=0, atol=1e-12)


# ---------------------------------------------------- 5. ring invariants
def _decode_chain(L, force_seed=None, steps=30, algo="gdn"):
    HK, HV, dk, dv, B = 1, 2, 4, 4, 3
    S0 = synth.initial_state(3, B, HV, dk, dv)
    orc = ReplayOracle(algo, 2, B, HK, HV, dk, dv, L, 0.5, S0)
    outs = []
    for t in range(steps):
        force = None if force_seed is None else synth.force_flags(force_seed + t, B, 0.3)
        for layer in range(2):
            inp = synth.window_inputs(synth.seed_for(9, t, layer), B, 1, HK, HV, dk, dv, algo)
            o, _ = orc.decode(layer, [0, 1, 2], inp, force, advance=(layer == 1))
            outs.append(o)
    return np.array(outs), orc


def test_no_ring_equals_any_ring_and_forced_folds():
    o_inf, orc_inf = _decode_chain(10 ** 6)
    o16, orc16 = _decode_chain(16)
    o3, _ = _decode_chain(3)
    of, _ = _decode_chain(5, force_seed=44)
    for other in (o16, o3, of):
        np.testing.assert_array_equal(o_inf, other)
    assert orc_inf.cursor.max() == 30 and orc16.cursor.max() < 16
    # After a fold the checkpoint is the committed state.
    orc16.fold([0, 1, 2])
    np.testing.assert_array_equal(orc16.ckpt, orc16.S)
    assert not orc16.cursor.any()


@pytest.mark.parametrize("mode", [ring.LAZY, ring.FOLD_EVERY])
def test_rejected_drafts_are_inert(mode):
    HK, HV, dk, dv, B, T, L = 2, 4, 4, 4, 12, 4, 8
    S0 = synth.initial_state(5, B, HV, dk, dv)
    runs = []
    for poisoned in (False, True):
        orc = ReplayOracle("gdn", 1, B, HK, HV, dk, dv, L, 0.5, S0)
        accepted_o = []
        for step in range(6):
            inp = synth.window_inputs(200 + step, B, T, HK, HV, dk, dv)
            acc = synth.accept_lengths(300 + step, B, T)
            if poisoned:
                inp, rows = synth.poison_rejected(inp, acc, T, 0.5, 400 + step)
                assert len(rows)
            o, _ = orc.window(0, np.arange(B), inp, T)
            mask = np.concatenate([np.arange(T) < acc[r] for r in range(B)])
            accepted_o.append(o[mask])
            orc.commit(np.arange(B), acc, T, mode=mode)
        runs.append((np.concatenate(accepted_o), orc.S.copy(), orc.ckpt.copy(),
                     orc.cursor.copy()))
    for a, b in zip(runs[0], runs[1]):
        np.testing.assert_array_equal(a, b)
    assert np.isfinite(runs[1][0]).all() and np.isfinite(runs[1][1]).all()


# ------------------------------------------------------ 6. special cases
def test_pure_read_when_no_decay_and_no_write():
    HK, HV, dk, dv = 2, 4, 3, 5
    rng = np.random.default_rng(5)
    S0 = rng.standard_normal((1, 1, HV, dk, dv))
    orc = ReplayOracle("gdn", 1, 1, HK, HV, dk, dv, 4, 0.3, S0)
    for t in range(7):
        toks = _rand_tokens(rng, 1, HK, HV, dk, dv, "gdn", beta=0.0, g=0.0)
        o, _ = orc.decode(0, [0], toks, advance=True)
        qh = np.repeat(toks["q"], 2, axis=1)[0]
        want = 0.3 * np.einsum("hkv,hk->hv", S0[0, 0], qh)
        np.testing.assert_allclose(o[0], want, atol=1e-14)


@pytest.mark.parametrize("algo", ["gdn", "kda"])
def test_full_forget_gate(algo):
    HK, HV, dk, dv = 1, 1, 4, 3
    rng = np.random.default_rng(6)
    S0 = rng.standard_normal((1, 1, HV, dk, dv))
    orc = ReplayOracle(algo, 1, 1, HK, HV, dk, dv, 4, 1.0, S0)
    orc.decode(0, [0], _rand_tokens(rng, 1, HK, HV, dk, dv, algo), advance=True)
    toks = _rand_tokens(rng, 1, HK, HV, dk, dv, algo, g=-np.inf)
    o, _ = orc.decode(0, [0], toks, advance=True)
    k, q, v, b = toks["k"][0, 0], toks["q"][0, 0], toks["v"][0, 0], toks["beta"][0, 0]
    np.testing.assert_allclose(o[0, 0], b * (k @ q) * v, atol=1e-14)


def test_kda_with_equal_channel_gates_is_gdn():
    HK, HV, dk, dv, B, T = 2, 4, 6, 5, 3, 3
    rng = np.random.default_rng(8)
    S0 = rng.standard_normal((1, B, HV, dk, dv)) * 0.1
    gdn = ReplayOracle("gdn", 1, B, HK, HV, dk, dv, 5, 0.5, S0)
    kda = ReplayOracle("kda", 1, B, HK, HV, dk, dv, 5, 0.5, S0)
    for step in range(5):
        toks = _rand_tokens(rng, B * T, HK, HV, dk, dv, "gdn")
        ktoks = dict(toks, g=np.repeat(toks["g"][:, :, None], dk, axis=2))
        acc = synth.accept_lengths(step, B, T)
        o1, _ = gdn.window(0, np.arange(B), toks, T)
        o2, _ = kda.window(0, np.arange(B), ktoks, T)
        np.testing.assert_allclose(o1, o2, atol=1e-13)
        gdn.commit(np.arange(B), acc, T)
        kda.commit(np.arange(B), acc, T)
    np.testing.assert_allclose(gdn.S, kda.S, atol=1e-13)


def test_key_head_sharing_is_adjacent_value_heads():
    """G = 2 with key heads [kA, kB] equals HK = HV with keys [kA, kA, kB, kB]."""
    HV, dk, dv = 4, 3, 3
    rng = np.random.default_rng(9)
    S0 = rng.standard_normal((1, 1, HV, dk, dv))
    grouped = ReplayOracle("gdn", 1, 1, 2, HV, dk, dv, 4, 1.0, S0)
    flat = ReplayOracle("gdn", 1, 1, 4, HV, dk, dv, 4, 1.0, S0)
    for t in range(6):
        toks = _rand_tokens(rng, 1, 2, HV, dk, dv, "gdn")
        ftoks = dict(toks, q=toks["q"][:, [0, 0, 1, 1]], k=toks["k"][:, [0, 0, 1, 1]])
        o1, _ = grouped.decode(0, [0], toks, advance=True)
        o2, _ = flat.decode(0, [0], ftoks, advance=True)
        np.testing.assert_array_equal(o1, o2)
    # and differs from the interleaved mapping h % HK
    toks = _rand_tokens(rng, 1, 2, HV, dk, dv, "gdn")
    itoks = dict(toks, q=toks["q"][:, [0, 1, 0, 1]], k=toks["k"][:, [0, 1, 0, 1]])
    o1, _ = grouped.decode(0, [0], toks, advance=True)
    o3, _ = flat.decode(0, [0], itoks, advance=True)
    assert not np.allclose(o1, o3)


def test_restore_clears_history():
    """A restored slot starts from its checkpoint with an empty ring."""
    HK, HV, dk, dv, B = 1, 2, 3, 3, 2
    rng = np.random.default_rng(12)
    S0 = rng.standard_normal((1, B, HV, dk, dv))
    orc = ReplayOracle("gdn", 1, B, HK, HV, dk, dv, 8, 1.0, S0)
    for t in range(5):
        orc.decode(0, [0, 1], _rand_tokens(rng, 2, HK, HV, dk, dv, "gdn"), advance=True)
    orc.fold([0])
    orc.load_checkpoint(1, orc.ckpt[:, 0])
    orc.reset_slots([1])
    np.testing.assert_array_equal(orc.S[:, 1], orc.S[:, 0])
    assert orc.cursor[1] == 0


# ---------------------------------------------- 7. bf16 checkpoint rounding
def test_round_bf16_known_values_and_ties():
    from oracle import round_bf16
    one = 1.0
    cases = {
        one: one,
        one + 2.0 ** -9: one,                       # below half an ulp (ulp = 2^-7)
        one + 2.0 ** -8: one,                       # exact tie, mantissa even: down
        one + 3 * 2.0 ** -8: one + 2.0 ** -6,       # exact tie, odd below: up to even
        one + 2.0 ** -7: one + 2.0 ** -7,           # representable
        -3.0 - 2.0 ** -7: -3.0,                     # ulp at 3 is 2^-6
        0.1: 0.10009765625,                         # nearest with 8 significant bits
        2.0 ** 100 * 1.5: 2.0 ** 100 * 1.5,
    }
    for x, want in cases.items():
        assert round_bf16(np.array(x)) == want, x
    nf = round_bf16(np.array([np.inf, -np.inf, np.nan]))
    assert nf[0] == np.inf and nf[1] == -np.inf and np.isnan(nf[2])


def test_round_bf16_matches_torch_on_float32_values():
    import torch
    rng = np.random.default_rng(21)
    x = (rng.standard_normal(20000) * np.exp(rng.uniform(-20, 20, 20000))).astype(np.float32)
    want = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    from oracle import round_bf16
    np.testing.assert_array_equal(round_bf16(x.astype(np.float64)), want)


def test_bf16_checkpoint_mode_rounds_only_at_folds():
    from oracle import round_bf16
    HK, HV, dk, dv, B = 1, 2, 8, 8, 2
    S0 = round_bf16(synth.initial_state(4, B, HV, dk, dv))
    exact = ReplayOracle("gdn", 1, B, HK, HV, dk, dv, 6, 0.5, S0)
    rounded = ReplayOracle("gdn", 1, B, HK, HV, dk, dv, 6, 0.5, S0, ckpt_round="bf16")
    for t in range(20):
        inp = synth.window_inputs(t, B, 1, HK, HV, dk, dv)
        o1, f = exact.decode(0, [0, 1], inp, advance=True)
        o2, _ = rounded.decode(0, [0, 1], inp, advance=True)
        if t < 6:                                 # before the first fold: identical
            np.testing.assert_array_equal(o1, o2)
        np.testing.assert_array_equal(round_bf16(rounded.ckpt), rounded.ckpt)
        assert np.max(np.abs(o1 - o2)) <= 1e-2 * np.max(np.abs(o1))
    assert not np.array_equal(exact.ckpt, rounded.ckpt)


# ------------------------------------------- fp16 delta ring: overflow flag
def test_fp16_delta_overflow_flag_marks_accepted_deltas_beyond_half_range():
    """With S0 = 0, g = 0 and a unit key, the first token's delta is exactly
    beta * v, so the flag is pinned by hand: 65504 (the largest finite fp16
    value) passes, anything beyond it is flagged, rejected drafts never
    count, and an fp32 delta ring is never flagged."""
    HK, HV, dk, dv, L = 1, 2, 4, 3, 4
    S0 = np.zeros((1, HV, dk, dv))

    def tokens(v_rows, beta=1.0):
        n = len(v_rows)
        k = np.zeros((n, HK, dk))
        k[:, :, 0] = 1.0
        v = np.zeros((n, HV, dv))
        for t, val in enumerate(v_rows):
            v[t, 0, 1] = val              # head 0, one value column
        return {"q": k.copy(), "k": k, "v": v, "beta": np.full((n, HV), beta),
                "g": np.zeros((n, HV))}

    # decode, two slots: slot 0 at the bound, slot 1 just past it
    orc = ReplayOracle("gdn", 1, 2, HK, HV, dk, dv, L, 1.0, np.concatenate([S0, S0]),
                       ring_d_dtype="f16")
    orc.decode(0, [0, 1], tokens([65504.0, 65504.5]), advance=True)
    np.testing.assert_array_equal(orc.d_overflow[0], [False, True])
    np.testing.assert_array_equal(orc.ring_d[0, :, 0, 0, 1], [65504.0, 65504.5])
    # beta scales the delta: beta * v = 0.5 * 2e5 = 1e5 > 65504
    orc = ReplayOracle("gdn", 1, 1, HK, HV, dk, dv, L, 1.0, S0, ring_d_dtype="f16")
    orc.decode(0, [0], tokens([2e5], beta=0.5), advance=True)
    assert orc.d_overflow[0, 0]
    # ... and it is the delta, not the value, that is checked: 0.25 * 2e5 = 5e4
    orc = ReplayOracle("gdn", 1, 1, HK, HV, dk, dv, L, 1.0, S0, ring_d_dtype="f16")
    orc.decode(0, [0], tokens([2e5], beta=0.25), advance=True)
    assert not orc.d_overflow[0, 0]
    # verify: a huge delta at a rejected draft does not count, an accepted one does
    for accept, want in ((1, False), (2, True)):
        orc = ReplayOracle("gdn", 1, 1, HK, HV, dk, dv, L, 1.0, S0, ring_d_dtype="f16")
        orc.window(0, [0], tokens([3.0, 1e6]), 2)
        orc.commit([0], [accept], 2)
        assert orc.d_overflow[0, 0] == want, accept
    # an fp32 delta ring is never flagged
    orc = ReplayOracle("gdn", 1, 1, HK, HV, dk, dv, L, 1.0, S0)
    orc.decode(0, [0], tokens([1e6]), advance=True)
    assert not orc.d_overflow.any()
