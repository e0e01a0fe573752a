"""Native fused-recurrent decode (the comparison point of the replay path)
against the oracle's token recurrence, step by step, through the C ABI."""
import numpy as np
import pytest
import torch

import synth
from oracle import round_bf16, token_step
from replay_harness import SENTINEL, TORCH, dev, rel_err
from linear_attention_state_rssm_gb300.store import ReplayStore

pytestmark = pytest.mark.gpu

TOL32, TOL16 = 1e-4, 4e-3


def _expand(x, G):
    """Key-head rows [R, HK, dk] onto value heads [R, HK*G, dk] (h uses h // G)."""
    return np.repeat(x, G, axis=1)


@pytest.mark.parametrize("algo,HK,HV,dk,dv,in_dtype,state_dtype", [
    ("gdn", 2, 4, 32, 32, "f32", "f32"),
    ("gdn", 16, 32, 128, 128, "bf16", "f32"),
    ("gdn", 4, 8, 128, 64, "bf16", "bf16"),
    ("kda", 4, 4, 64, 128, "f32", "f32"),
    ("kda", 2, 4, 128, 128, "bf16", "bf16"),
])
def test_native_decode_matches_token_recurrence(algo, HK, HV, dk, dv, in_dtype, state_dtype):
    B, steps, G = 6, 12, HV // HK
    slots = np.array([3, -1, 0, 5, -1, 1], dtype=np.int32)
    n_slots = 6
    st = ReplayStore(algo, 1, n_slots, HK, HV, dk, dv, 4, 1, in_dtype, state_dtype)
    S0 = synth.initial_state(synth.seed_for(40, 0, 0), n_slots, HV, dk, dv, state_dtype)
    st.state[0].copy_(dev(S0, state_dtype))
    S = S0.copy()
    slot_t = torch.from_numpy(slots).cuda()
    live = slots >= 0
    tol = TOL32 if (in_dtype, state_dtype) == ("f32", "f32") else TOL16
    for step in range(steps):
        inp = synth.window_inputs(synth.seed_for(40, step + 1, 0), B, 1, HK, HV, dk, dv, algo,
                                  in_dtype)
        o = torch.full((B, HV, dv), SENTINEL, dtype=TORCH[in_dtype], device="cuda")
        st.rssm_native_decode(0, dev(inp["q"], in_dtype), dev(inp["k"], in_dtype),
                              dev(inp["v"], in_dtype), dev(inp["beta"], "f32"),
                              dev(inp["g"], "f32"), slot_t, o)
        rows = np.nonzero(live)[0]
        sl = slots[rows]
        S_new, _, o_ref = token_step(S[sl], _expand(inp["q"][rows], G), _expand(inp["k"][rows], G),
                                     inp["v"][rows], inp["beta"][rows], inp["g"][rows],
                                     st.scale, algo)
        S[sl] = round_bf16(S_new) if state_dtype == "bf16" else S_new
        o_gpu = o.double().cpu().numpy()
        assert rel_err(o_gpu[rows], o_ref) <= tol, step
        assert np.all(o_gpu[~live] == SENTINEL), "null rows must be left untouched"
        S_gpu = st.state[0].double().cpu().numpy()
        if state_dtype == "bf16":
            # the chains round every token: where fp32 and fp64 values fall on
            # opposite sides of a rounding boundary they differ by one bf16 ulp,
            # and such a difference can carry into the next token's rounding
            ulp = np.ldexp(1.0, np.frexp(np.abs(S[sl]))[1] - 8)
            assert np.all(np.abs(S_gpu[sl] - S[sl]) <= 2 * ulp + tol * np.abs(S[sl]).max()), step
        else:
            assert rel_err(S_gpu[sl], S[sl]) <= tol, step
    untouched = np.setdiff1d(np.arange(n_slots), slots[live])
    assert np.array_equal(st.state[0].double().cpu().numpy()[untouched], S0[untouched])
    assert st.rssm_get_device_error() == 0


def test_native_decode_equals_replay_decode_on_an_empty_ring():
    """With an empty ring and no fold, one replay decode step and one native
    step compute the same token: outputs agree within the fp32 tolerance and
    the native state equals the replayed one (checkpoint + the new record)."""
    HK, HV, dk, dv, B = 2, 4, 128, 128, 3
    slots = np.array([0, 1, 2], dtype=np.int32)
    S0 = synth.initial_state(synth.seed_for(41, 0, 0), B, HV, dk, dv, "f32")
    inp = synth.window_inputs(synth.seed_for(41, 1, 0), B, 1, HK, HV, dk, dv, "gdn", "f32")
    outs, states = [], []
    for native in (False, True):
        st = ReplayStore("gdn", 1, B, HK, HV, dk, dv, 4, 1, "f32", "f32")
        st.state[0].copy_(dev(S0, "f32"))
        o = torch.empty((B, HV, dv), dtype=torch.float32, device="cuda")
        args = (0, dev(inp["q"], "f32"), dev(inp["k"], "f32"), dev(inp["v"], "f32"),
                dev(inp["beta"], "f32"), dev(inp["g"], "f32"), torch.from_numpy(slots).cuda())
        if native:
            st.rssm_native_decode(*args, o)
            states.append(st.state[0].double().cpu().numpy())
        else:
            st.rssm_decode(*args, o)
            # the replayed state from the checkpoint and the record just written
            k = st.ring_k[0][:, :, 0].double().cpu().numpy()
            d = st.ring_d[0][:, :, 0].double().cpu().numpy()
            g = st.ring_g[0][:, :, 0].double().cpu().numpy()
            states.append(np.exp(g)[..., None, None] * S0 + k[..., :, None] * d[..., None, :])
        outs.append(o.double().cpu().numpy())
    assert rel_err(outs[1], outs[0]) <= TOL32
    assert rel_err(states[1], states[0]) <= TOL32
