"""CUDA path vs the fp64 oracle on the workloads the pages' models suggest.

Tolerances (max |gpu - oracle| / max |oracle| over live rows and accepted
positions, per step and layer): 1e-4 when everything is fp32, 4e-3 when any
input or the state is bf16. Cursors, fold decisions and written ring positions
are compared bit for bit.
"""
import numpy as np
import pytest
import torch

import synth
from replay_harness import Run, rel_err, SENTINEL

pytestmark = pytest.mark.gpu

TOL32, TOL16 = 1e-4, 4e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from linear_attention_state_rssm_gb300 import build
    build.build()


def _null_slots(B, n_null, seed):
    slots = np.arange(B, dtype=np.int32)
    slots[synth.null_rows(seed, B, n_null)] = -1
    return slots


# --------------------------------------------------------------- decode
def test_tiny_gdn_decode_forty_steps_two_folds():
    """1 layer, batch 2, HK=2, HV=4, dk=dv=32, L=16, T=1, 40 steps, fp32."""
    run = Run(algo="gdn", HK=2, HV=4, dk=32, dv=32, L=16, max_T=1, slots=[0, 1], config_id=0)
    fold_steps = []
    for step in range(40):
        inp = run.inputs(step, 0, 1)
        _, o_gpu, o_orc, f_gpu, f_orc = run.window(0, inp, 1, decode=True, advance=True)
        assert rel_err(o_gpu, o_orc) <= TOL32, step
        np.testing.assert_array_equal(f_gpu, f_orc)
        run.check_cursors()
        run.check_ring_records()
        if f_gpu[0]:
            fold_steps.append(step)
        assert run.state_err() <= TOL32
    assert fold_steps == [16, 32]
    assert run.ring_d_err() <= TOL32
    assert run.store.rssm_get_device_error() == 0


@pytest.mark.parametrize("plan", ["rows", "pipe"])
def test_qwen_shaped_gdn_decode_full_batch(plan):
    """HK=16, HV=32, dk=dv=128, batch 64 with 8 null slots, L=16, bf16 q/k/v,
    fp32 state and deltas, fp16 ring keys; 34 steps (two folds). Every live row
    is compared with the oracle on every step (outputs, fold flags, cursors,
    ring records; checkpoints after each fold), so the decode kernel's
    reordering of folding rows is covered for every row."""
    B = 64
    slots = _null_slots(B, 8, 1001)
    null = np.nonzero(slots < 0)[0]
    live = np.nonzero(slots >= 0)[0]
    run = Run(algo="gdn", HK=16, HV=32, dk=128, dv=128, L=16, max_T=1, slots=slots,
              n_slots=B, in_dtype="bf16", config_id=1, plan=plan)
    folds = 0
    for step in range(34):
        inp = run.inputs(step, 0, 1)
        o_all, o_gpu, o_orc, f_gpu, f_orc = run.window(0, inp, 1, decode=True, advance=True)
        live_tok = run.orc_slots >= 0
        assert rel_err(o_gpu[live_tok], o_orc[live_tok]) <= TOL16, step
        assert np.all(o_all[null] == SENTINEL), "null rows must be left untouched"
        np.testing.assert_array_equal(f_gpu[live_tok], f_orc[live_tok])
        run.check_cursors()
        run.check_ring_records()
        if f_gpu[live_tok].any():
            folds += 1
            assert run.state_err() <= TOL16, step
    assert folds == 2
    cur = run.cursor_gpu()
    assert np.all(cur[null] == 0)
    assert np.all(cur[live] == cur[live[0]])
    assert run.state_err() <= TOL16
    assert run.ring_d_err() <= TOL16
    assert run.store.rssm_get_device_error() == 0


# --------------------------------------------------------------- verify
def _verify_chain(run, T, steps, poison_frac, seed0, check_oracle=True, narrow_to=None,
                  full_steps=4):
    """Chained verify + commit; returns accepted outputs per step (GPU).

    With ``narrow_to``, the run starts on every row and keeps every row until
    at least ``full_steps`` steps, one of them with ring-overflow folds, have
    been compared; then it follows the rows ``narrow_to`` only."""
    accepted = []
    fold_seen = False
    for step in range(steps):
        if narrow_to is not None and step >= full_steps and fold_seen:
            run.narrow(narrow_to)
            narrow_to = None
        inp = run.inputs(step, 0, T)
        acc = synth.accept_lengths(seed0 + step, run.B, T)
        if poison_frac:
            inp, _ = synth.poison_rejected(inp, acc, T, poison_frac, seed0 + 500 + step)
        o_all, o_gpu, o_orc, f_gpu, f_orc = run.window(0, inp, T)
        mask = (np.arange(T)[None, :] < acc[run.sample][:, None]).reshape(-1)
        mask &= np.repeat(run.orc_slots >= 0, T)
        if check_oracle:
            assert np.isfinite(o_gpu[mask]).all()
            assert rel_err(o_gpu[mask], o_orc[mask]) <= run.tol, (step, T)
            live = run.orc_slots >= 0
            np.testing.assert_array_equal(f_gpu[live], f_orc[live])
            # a fold-every commit folds every step (its windows never overflow)
            fold_seen |= bool(f_gpu[live].any()) or run.commit_mode == "fold_every"
        run.commit(acc, T)
        if check_oracle:
            run.check_cursors()
            run.check_ring_records()
            assert run.state_err() <= run.tol
        amask = (np.arange(T)[None, :] < acc[:, None]).reshape(-1)
        amask &= np.repeat(run.slots >= 0, T)
        accepted.append(o_all[amask])
    return accepted


@pytest.mark.parametrize("plan", ["rows", "pipe", "tc"])
@pytest.mark.parametrize("T", [3, 8])
@pytest.mark.parametrize("state,mode", [("f32", "lazy"), ("bf16", "fold_every")])
def test_gdn_verify_commit_with_poisoned_drafts(T, state, mode, plan):
    """HK=16, HV=32, dk=dv=128, batch 128, L=16, accept ~ U[0, T], NaN/Inf at
    rejected positions of 10% of the rows with rejections, 24 chained steps.
    Every row is compared until at least four steps, one with ring-overflow
    folds, have been; then a sample of rows for the rest of the chain."""
    B = 128
    sample = np.array([0, 5, 17, 42, 77, 101, 127])
    run = Run(algo="gdn", HK=16, HV=32, dk=128, dv=128, L=16, max_T=T, slots=np.arange(B),
              in_dtype="bf16", state_dtype=state, commit_mode=mode, config_id=2, plan=plan)
    run.tol = TOL16
    _verify_chain(run, T, 24, 0.10, 7000 + T, narrow_to=sample)
    assert run.ring_d_err() <= TOL16
    assert run.store.rssm_get_device_error() == 0


@pytest.mark.parametrize("plan", ["rows", "pipe", "tc"])
@pytest.mark.parametrize("state,mode", [("f32", "lazy"), ("bf16", "fold_every")])
def test_poisoned_rejected_drafts_are_bitwise_inert(state, mode, plan):
    """Poisoned vs clean rejected positions: accepted outputs, checkpoints,
    accepted ring records and cursors are bitwise identical."""
    B, T = 64, 4
    runs = []
    for poison in (0.0, 0.5):
        run = Run(algo="gdn", HK=4, HV=8, dk=128, dv=128, L=16, max_T=T, slots=np.arange(B),
                  in_dtype="bf16", state_dtype=state, commit_mode=mode, config_id=12,
                  sample=np.array([0]), plan=plan)
        acc = _verify_chain(run, T, 10, poison, 900, check_oracle=False)
        runs.append((run, acc))
    (r0, a0), (r1, a1) = runs
    for x, y in zip(a0, a1):
        assert np.isfinite(y).all()
        np.testing.assert_array_equal(x, y)
    assert torch.equal(r0.store.state, r1.store.state)
    assert torch.equal(r0.store.cursor, r1.store.cursor)
    cur = r0.cursor_gpu()
    for s in range(B):
        c = int(cur[s])
        assert torch.equal(r0.store.ring_d[:, s, :, :c], r1.store.ring_d[:, s, :, :c])
        assert torch.equal(r0.store.ring_k[:, s, :, :c], r1.store.ring_k[:, s, :, :c])


# --------------------------------------------------------------- KDA
@pytest.mark.parametrize("variant", ["bf16_fp16cache", "fp32"])
def test_kda_decode_and_verify_alternating(variant):
    """KDA HK=HV=32, dk=dv=128, batch 64, L=32; decode (T=1) and verify (T=3)
    steps alternate over 64 chained steps."""
    if variant == "fp32":
        kw = dict(in_dtype="f32", state_dtype="f32", ring_k_dtype="f32", ring_d_dtype="f32",
                  commit_mode="lazy")
        tol = TOL32
    else:
        kw = dict(in_dtype="bf16", state_dtype="bf16", ring_k_dtype="f16", ring_d_dtype="f16",
                  commit_mode="fold_every")
        tol = TOL16
    B = 64
    sample = np.array([3, 31, 60])
    run = Run(algo="kda", HK=32, HV=32, dk=128, dv=128, L=32, max_T=3, slots=np.arange(B),
              config_id=3, **kw)
    for step in range(64):
        if step == 8:
            run.narrow(sample)   # every row for the first eight steps
        if step % 2 == 0:
            inp = run.inputs(step, 0, 1)
            _, o_gpu, o_orc, f_gpu, f_orc = run.window(0, inp, 1, decode=True, advance=True)
            assert rel_err(o_gpu, o_orc) <= tol, step
        else:
            T = 3
            inp = run.inputs(step, 0, T)
            acc = synth.accept_lengths(3300 + step, B, T)
            _, o_gpu, o_orc, f_gpu, f_orc = run.window(0, inp, T)
            mask = (np.arange(T)[None, :] < acc[run.sample][:, None]).reshape(-1)
            assert rel_err(o_gpu[mask], o_orc[mask]) <= tol, step
            run.commit(acc, T)
        np.testing.assert_array_equal(f_gpu, f_orc)
        run.check_cursors()
        run.check_ring_records()
        assert run.state_err() <= tol
    assert run.ring_d_err() <= tol
    if variant != "fp32":
        run.check_no_fp16_delta_overflow()
    assert run.store.rssm_get_device_error() == 0
