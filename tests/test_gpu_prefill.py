"""Replay prefill (prompt -> checkpoint, cursor -> 0): CUDA path vs the fp64
oracle, row by row, then decode on top of the new checkpoint.

Tolerances as for the replay kernel: 1e-4 when everything is fp32, 4e-3 with a
bf16 input or state, over every prompt token of every active row; the
checkpoint against the oracle's (bf16: the chain rounded at the same points,
plus one ulp); cursors bit-exact.
"""
import numpy as np
import pytest
import torch

import synth
from replay_harness import Run, SENTINEL, rel_err

pytestmark = pytest.mark.gpu

TOL32, TOL16 = 1e-4, 4e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from linear_attention_state_rssm_gb300 import build
    build.build()


def _prompt_inputs(run, seed, cu):
    """Packed prompt tokens plus one spare token whose output must stay."""
    return synth.window_inputs(seed, int(cu[-1]) + 1, 1, run.HK, run.HV, run.dk, run.dv,
                               run.algo, run.in_dtype)


def _check_prefill(run, o_gpu, o_orc, cu, tol):
    lens = np.diff(cu)
    active = (run.slots >= 0) & (lens > 0)
    tok = np.zeros(o_gpu.shape[0], dtype=bool)
    for r in np.nonzero(active)[0]:
        tok[cu[r]:cu[r + 1]] = True
    assert np.isfinite(o_gpu[tok]).all()
    assert rel_err(o_gpu[tok], o_orc[tok[:cu[-1]]]) <= tol
    assert np.all(o_gpu[~tok] == SENTINEL), "null, idle and spare rows untouched"


@pytest.mark.parametrize("algo,HK,HV,dk,dv,in_dt,state", [
    ("gdn", 2, 4, 128, 128, "f32", "f32"),
    ("gdn", 2, 4, 128, 128, "bf16", "f32"),
    ("gdn", 2, 4, 64, 32, "bf16", "bf16"),
    ("gdn", 1, 2, 32, 64, "f32", "f32"),
    ("kda", 2, 2, 128, 128, "f32", "f32"),
    ("kda", 2, 2, 64, 128, "bf16", "bf16"),
])
def test_prefill_after_history_then_decode(algo, HK, HV, dk, dv, in_dt, state):
    """Rows decode a few tokens (ring history), then prefill prompts of every
    length class around the 16-token chunk (0, 1, 15, 16, 17, 45) on two
    layers, then decode again from the new checkpoints."""
    slots = np.array([4, 0, -1, 2, 5, 1, 3], dtype=np.int32)
    B, n_layers, L = slots.size, 2, 8
    run = Run(algo=algo, HK=HK, HV=HV, dk=dk, dv=dv, L=L, max_T=1, slots=slots, n_slots=6,
              n_layers=n_layers, in_dtype=in_dt, state_dtype=state, config_id=70)
    tol = TOL32 if (in_dt, state) == ("f32", "f32") else TOL16

    def decode_steps(step0, n):
        for step in range(step0, step0 + n):
            for layer in range(n_layers):
                inp = run.inputs(step, layer, 1)
                _, o_gpu, o_orc, _, _ = run.window(layer, inp, 1, decode=True,
                                                   advance=layer == n_layers - 1)
                live = run.orc_slots >= 0
                assert rel_err(o_gpu[live], o_orc[live]) <= tol, (step, layer)
            run.check_cursors()
            run.check_ring_records()

    decode_steps(0, 3)
    lens = np.array([17, 0, 5, 1, 45, 16, 15])
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    for layer in range(n_layers):
        inp = _prompt_inputs(run, synth.seed_for(70, 100, layer), cu)
        o_gpu, o_orc = run.prefill(layer, inp, cu, reset_cursor=layer == n_layers - 1)
        _check_prefill(run, o_gpu, o_orc, cu, tol)
    run.check_cursors()
    run.check_ring_records()
    cur = run.cursor_gpu()
    assert cur[slots[1]] == 3, "a row without prompt tokens keeps its history"
    assert all(cur[s] == 0 for r, s in enumerate(slots) if s >= 0 and lens[r] > 0)
    assert run.state_err() <= tol
    decode_steps(3, 3)
    assert run.state_err() <= tol
    assert run.store.rssm_get_device_error() == 0


def test_prefill_qwen_shapes():
    """Qwen3.5-4B-shaped GDN heads (HK 16, HV 32, dk = dv = 128), bf16 prompts
    of a few hundred tokens, fp32 checkpoint, from an empty ring."""
    slots = np.array([0, 1, -1, 2], dtype=np.int32)
    run = Run(HK=16, HV=32, dk=128, dv=128, L=16, max_T=1, slots=slots, n_slots=3,
              in_dtype="bf16", config_id=71)
    lens = np.array([301, 64, 9, 0])
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    inp = _prompt_inputs(run, synth.seed_for(71, 0, 0), cu)
    o_gpu, o_orc = run.prefill(0, inp, cu, reset_cursor=True)
    _check_prefill(run, o_gpu, o_orc, cu, TOL16)
    run.check_cursors()
    run.check_ring_records()
    assert run.state_err() <= TOL16
    assert run.store.rssm_get_device_error() == 0


def test_prefill_bad_offsets_set_the_seqlen_bit():
    from linear_attention_state_rssm_gb300 import _lib as lib
    slots = np.arange(3, dtype=np.int32)
    run = Run(HK=2, HV=4, dk=128, dv=128, L=16, max_T=1, slots=slots, n_slots=3, config_id=72)
    cu = np.array([0, 20, 5, 30], dtype=np.int32)         # row 1 decreasing
    inp = synth.window_inputs(synth.seed_for(72, 0, 0), 31, 1, 2, 4, 128, 128, "gdn", "f32")
    S_before = run.store.state.clone()
    q, k, v, beta, g = run._gpu_inputs(inp)
    o = torch.full((31, 4, 128), SENTINEL, dtype=torch.float32, device="cuda")
    run.store.rssm_prefill(0, q, k, v, beta, g, torch.from_numpy(cu).cuda(), run.slot_t, o,
                           reset_cursor=True)
    assert run.store.rssm_get_device_error() == lib.DEVERR["seqlen"]
    assert torch.equal(run.store.state[:, 1], S_before[:, 1])
    o = o.cpu().numpy()
    assert np.all(o[:20] != SENTINEL) and np.all(o[5:30] != SENTINEL)
    assert np.all(o[30] == SENTINEL)
