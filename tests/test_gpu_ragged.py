"""Ragged verify (windows of different lengths packed through cu_seqlens) and
its commit: CUDA path vs the fp64 oracle, row by row.

Tolerances as for the uniform verify: 1e-4 when everything is fp32, 4e-3 with
a bf16 input or state, over every token of every active row (the inputs are
finite). Idle rows (no tokens) and null rows leave outputs, fold flags,
cursors and checkpoints untouched; cursors and fold flags are bit-exact.
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


def _packed_inputs(run, step, cu):
    """Packed tokens of one step, plus one spare token past cu[-1] whose
    output row must stay untouched."""
    n_tok = int(cu[-1]) + 1
    return synth.window_inputs(synth.seed_for(run.config_id, step, 0), n_tok, 1, run.HK,
                               run.HV, run.dk, run.dv, run.algo, run.in_dtype)


@pytest.mark.parametrize("algo,HK,HV,max_T,in_dt,state,mode", [
    ("gdn", 4, 8, 8, "bf16", "f32", "lazy"),
    ("gdn", 4, 8, 3, "f32", "f32", "lazy"),
    ("gdn", 4, 8, 1, "f32", "f32", "lazy"),
    ("gdn", 4, 8, 8, "bf16", "bf16", "fold_every"),
    ("kda", 4, 4, 4, "f32", "f32", "lazy"),
    ("kda", 4, 4, 8, "bf16", "bf16", "fold_every"),
])
def test_ragged_verify_commit_chain(algo, HK, HV, max_T, in_dt, state, mode):
    B, L, steps = 12, 16, 10
    slots = np.arange(B, dtype=np.int32)[::-1].copy()
    slots[[3, 8]] = -1
    run = Run(algo=algo, HK=HK, HV=HV, dk=128, dv=128, L=L, max_T=max_T, slots=slots,
              n_slots=B, in_dtype=in_dt, state_dtype=state, commit_mode=mode, config_id=60)
    tol = TOL32 if (in_dt, state) == ("f32", "f32") else TOL16
    for step in range(steps):
        cu = synth.ragged_lengths(synth.seed_for(60, step, 1), B, max_T)
        lens = np.diff(cu)
        force = synth.force_flags(synth.seed_for(60, step, 2), B, 0.1)
        inp = _packed_inputs(run, step, cu)
        o_gpu, o_orc, f_gpu, f_orc = run.window_ragged(0, inp, cu, max_T, force)
        active = (slots >= 0) & (lens > 0)
        tok_active = np.zeros(o_gpu.shape[0], dtype=bool)
        for r in np.nonzero(active)[0]:
            tok_active[cu[r]:cu[r + 1]] = True
        assert np.isfinite(o_gpu[tok_active]).all()
        assert rel_err(o_gpu[tok_active], o_orc[:cu[-1]][tok_active[:cu[-1]]]) <= tol, step
        assert np.all(o_gpu[~tok_active] == SENTINEL), "idle, null and spare rows untouched"
        np.testing.assert_array_equal(f_gpu[active], f_orc[active])
        assert np.all(f_gpu[~active] == 7)
        cur0 = run.cursor_gpu().copy()
        acc = synth.ragged_accept(synth.seed_for(60, step, 3), cu)
        run.commit_ragged(acc, cu, max_T, force)
        run.check_cursors()
        run.check_ring_records()
        idle_slots = slots[(slots >= 0) & (lens == 0)]
        np.testing.assert_array_equal(run.cursor_gpu()[idle_slots], cur0[idle_slots])
        assert run.state_err() <= tol, step
    assert run.store.rssm_get_device_error() == 0


@pytest.mark.parametrize("T", [2, 3, 8])
def test_equal_lengths_are_the_uniform_verify_bitwise(T):
    """cu_seqlens = r * T gives the uniform verify's outputs, records, fold
    flags and checkpoints bit for bit (the same kernel width, the same work).
    A one-token window is the exception: uniform, it runs the decode width;
    ragged windows start at width 2 (covered against the oracle above)."""
    B, HK, HV, L = 6, 2, 4, 16
    slots = np.array([0, 4, -1, 2, 5, 1], dtype=np.int32)
    runs = [Run(HK=HK, HV=HV, dk=128, dv=128, L=L, max_T=8, slots=slots, n_slots=B,
                in_dtype="bf16", config_id=61) for _ in range(2)]
    cu = (np.arange(B + 1) * T).astype(np.int32)
    for step in range(6):
        inp = runs[0].inputs(step, 0, T)
        acc = synth.accept_lengths(synth.seed_for(61, step, 1), B, T)
        force = synth.force_flags(synth.seed_for(61, step, 2), B, 0.2)
        o_a, _, _, f_a, _ = runs[0].window(0, inp, T, force)
        o_b, _, f_b, _ = runs[1].window_ragged(0, inp, cu, T, force)
        assert np.array_equal(o_a, o_b)
        assert np.array_equal(f_a, f_b)
        runs[0].commit(acc, T, force)
        runs[1].commit_ragged(acc, cu, T, force)
        for name in ("state", "ring_k", "ring_d", "ring_g", "ring_v", "ring_beta", "cursor"):
            a = getattr(runs[0].store, name)
            b = getattr(runs[1].store, name)
            assert torch.equal(a, b), (step, name)


def test_bad_offsets_set_the_seqlen_bit_and_skip_the_row():
    """A window wider than max_T or with decreasing offsets is refused on the
    device: the error word gets its seqlen bit, the row's outputs, cursor and
    checkpoint stay as they were, the other rows are computed."""
    from linear_attention_state_rssm_gb300 import _lib as lib
    B, max_T = 4, 4
    slots = np.arange(B, dtype=np.int32)
    run = Run(HK=2, HV=4, dk=128, dv=128, L=16, max_T=max_T, slots=slots, n_slots=B,
              config_id=62)
    cu = np.array([0, 2, 9, 5, 8], dtype=np.int32)   # row 1: 7 > max_T; row 2: 9 -> 5
    inp = synth.window_inputs(synth.seed_for(62, 0, 0), 10, 1, 2, 4, 128, 128, "gdn", "f32")
    S_before = run.store.state.clone()
    q, k, v, beta, g = run._gpu_inputs(inp)
    o = torch.full((10, 4, 128), SENTINEL, dtype=torch.float32, device="cuda")
    cu_t = torch.from_numpy(cu).cuda()
    run.store.rssm_verify_ragged(0, q, k, v, beta, g, cu_t, run.slot_t, max_T, o)
    acc = torch.tensor([1, 1, 1, 2], dtype=torch.int32, device="cuda")
    run.store.rssm_commit_ragged(run.slot_t, acc, cu_t, max_T)
    word = run.store.rssm_get_device_error()
    assert word == lib.DEVERR["seqlen"]
    o = o.cpu().numpy()
    assert np.all(o[[2, 3, 4, 8, 9]] == SENTINEL)           # only rows 0 and 3 have windows
    cur = run.cursor_gpu()
    assert cur[1] == 0 and cur[2] == 0                      # refused rows: cursor unchanged
    assert cur[0] == 1 and cur[3] == 2                      # good rows committed
    assert torch.equal(run.store.state[:, 1:3], S_before[:, 1:3])
    assert np.all(o[0:2] != SENTINEL) and np.all(o[5:8] != SENTINEL)


def test_host_refuses_bad_ragged_arguments():
    run = Run(HK=2, HV=4, dk=128, dv=128, L=16, max_T=4, slots=np.arange(2, dtype=np.int32),
              n_slots=2, config_id=63)
    from linear_attention_state_rssm_gb300 import _lib as lib
    inp = synth.window_inputs(synth.seed_for(63, 0, 0), 4, 1, 2, 4, 128, 128, "gdn", "f32")
    q, k, v, beta, g = run._gpu_inputs(inp)
    o = torch.empty((4, 4, 128), device="cuda")
    cu_t = torch.tensor([0, 2, 4], dtype=torch.int32, device="cuda")
    for max_T in (0, 5):                                    # outside [1, configured max_T]
        with pytest.raises(lib.RssmError) as e:
            run.store.rssm_verify_ragged(0, q, k, v, beta, g, cu_t, run.slot_t, max_T, o)
        assert e.value.status == 1
    with pytest.raises(lib.RssmError):
        lib.rssm_verify_ragged(run.store.handle, 0, q, k, v, beta, g, None, run.slot_t, None, 2,
                               4, o, None)
    with pytest.raises(lib.RssmError):
        lib.rssm_commit_ragged(run.store.handle, run.slot_t, None,
                               torch.zeros(2, dtype=torch.int32, device="cuda"), None, 2, 4)
