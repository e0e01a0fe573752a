"""The bounded waits of the replay and fold kernels, made to run out on
purpose through the test hook rssm_debug_withhold: one barrier is promised 16
bytes more than its copies carry, so every wait on it gives up after its
usual 0.5 s.
Nothing faults or hangs (every copy lands; only the count is short). Checked:
the call returns, RSSM_DEVERR_TIMEOUT is set, the row's outputs, records and
checkpoint are as include/rssm.h says, and with the hook off the next call is
clean and matches the oracle."""
import time

import numpy as np
import pytest
import torch

import synth
from replay_harness import Run, rel_err, SENTINEL

pytestmark = pytest.mark.gpu
TOL32 = 1e-4
BUFS = ("state", "ring_k", "ring_d", "ring_g", "ring_v", "ring_beta", "cursor")
ROWS_PER_CHUNK = 16  # fp32 checkpoint rows of 128 values: 8 KB chunks


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from linear_attention_state_rssm_gb300 import build
    build.build()


def _snap(st):
    return {name: getattr(st, name).clone() for name in BUFS}


def _same(st, snap, names=BUFS):
    for name in names:
        assert torch.equal(getattr(st, name), snap[name]), name


def _history(run, steps, T=1):
    for step in range(steps):
        run.window(0, run.inputs(step, 0, T), T, decode=True, advance=True)


def _timed_out_call(run, inp, T, force=None, decode=False):
    """One verify (or decode, cursor left alone) with the hook on; returns
    (o, fold_out, error word, seconds)."""
    q, k, v, beta, g = run._gpu_inputs(inp)
    o = torch.full((run.B * T, run.HV, run.dv), SENTINEL, device="cuda")
    fold_out = torch.full((run.B,), 7, dtype=torch.uint8, device="cuda")
    f = None if force is None else torch.from_numpy(np.asarray(force, np.uint8)).cuda()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    if decode:
        run.store.rssm_decode(0, q, k, v, beta, g, run.slot_t, o, force=f, fold_out=fold_out)
    else:
        run.store.rssm_verify(0, q, k, v, beta, g, run.slot_t, T, o, force=f,
                              fold_out=fold_out)
    err = run.store.rssm_get_device_error()
    return o, fold_out, err, time.perf_counter() - t0


def _clean_step(run, inp, T, step, force=None, decode=False):
    """The same window with the hook off: matches the oracle, no error."""
    run.store.rssm_debug_withhold(-1)
    _, o_gpu, o_orc, f_gpu, f_orc = run.window(0, inp, T, force=force, decode=decode,
                                               advance=decode)
    acc = np.ones(run.B, np.int32) if decode else synth.accept_lengths(7100 + step, run.B, T)
    mask = (np.arange(T)[None, :] < acc[:, None]).reshape(-1)
    assert rel_err(o_gpu[mask], o_orc[mask]) <= TOL32
    np.testing.assert_array_equal(f_gpu, f_orc)
    if not decode:
        run.commit(acc, T, force=force)
    run.check_cursors()
    run.check_ring_records()
    assert run.state_err() <= TOL32
    assert run.store.rssm_get_device_error() == 0


@pytest.mark.parametrize("algo,plan", [("gdn", "rows"), ("gdn", "pipe"), ("gdn", "tc"),
                                       ("kda", "rows")])
@pytest.mark.parametrize("where", ["window", "history", "chunk"])
def test_wait_that_runs_out_leaves_the_row_untouched(algo, where, plan):
    """A verify window (no fold) whose window, history or checkpoint-chunk wait
    runs out writes no output, fold flag, delta, value, checkpoint or cursor;
    keys, gates and betas may be written only at ring positions [c, c + T),
    past the committed history (the window's own wait: nothing at all)."""
    from linear_attention_state_rssm_gb300 import _lib as L_
    T = 3
    run = Run(algo=algo, HK=2, HV=4, dk=128, dv=128, L=8, max_T=T, slots=[0, 2, 1],
              config_id=70, plan=plan)
    _history(run, 2)                                   # cursor 2: 2 + 3 <= 8, no fold
    snap = _snap(run.store)
    barrier = {"window": L_.WITHHOLD["window"], "history": L_.WITHHOLD["history"],
               "chunk": L_.withhold_chunk(5)}[where]
    run.store.rssm_debug_withhold(barrier)
    inp = run.inputs(10, 0, T)
    o, fold_out, err, secs = _timed_out_call(run, inp, T)
    assert err & L_.DEVERR["timeout"]
    assert secs < 30.0
    assert torch.all(o == SENTINEL)
    assert torch.all(fold_out == 7)
    kgb = ("ring_k", "ring_g", "ring_beta")
    _same(run.store, snap, [n for n in BUFS if n not in kgb or where == "window"])
    c = 2
    for name in kgb:
        now, was = getattr(run.store, name), snap[name]
        assert torch.equal(now[:, :, :, :c], was[:, :, :, :c]), name
        assert torch.equal(now[:, :, :, c + T:], was[:, :, :, c + T:]), name
    _clean_step(run, inp, T, 10)


@pytest.mark.parametrize("algo,T,plan", [("gdn", 3, "rows"), ("kda", 3, "rows"),
                                         ("gdn", 1, "rows"), ("gdn", 8, "rows"),
                                         ("gdn", 3, "pipe"), ("gdn", 1, "pipe"),
                                         ("gdn", 8, "pipe"), ("gdn", 3, "tc"),
                                         ("gdn", 8, "tc")])
def test_folding_row_stops_storing_at_the_failed_chunk(algo, T, plan):
    """A forced fold whose checkpoint chunk 5 never completes (verify, or decode
    for T = 1): no output, fold flag or ring record is written, the checkpoint
    rows from chunk 5 on are untouched (the chunks before it may hold the
    folded state); writing the checkpoint back restores the slot, and the next
    clean call matches."""
    from linear_attention_state_rssm_gb300 import _lib as L_
    run = Run(algo=algo, HK=2, HV=4, dk=128, dv=128, L=16, max_T=T, slots=[0, 1],
              config_id=71, plan=plan)
    _history(run, 4)
    snap = _snap(run.store)
    run.store.rssm_debug_withhold(L_.withhold_chunk(5))
    inp = run.inputs(10, 0, T)
    force = np.ones(run.B, np.uint8)
    o, fold_out, err, secs = _timed_out_call(run, inp, T, force, decode=T == 1)
    assert err & L_.DEVERR["timeout"]
    assert secs < 30.0
    assert torch.all(o == SENTINEL)
    assert torch.all(fold_out == 7)
    _same(run.store, snap, [n for n in BUFS if n != "state"])
    r0 = 5 * ROWS_PER_CHUNK
    assert torch.equal(run.store.state[..., r0:, :], snap["state"][..., r0:, :])
    run.store.state.copy_(snap["state"])               # restore the slot
    _clean_step(run, inp, T, 10, force, decode=T == 1)


@pytest.mark.parametrize("plan", ["rows", "tc"])
def test_fold_every_commit_stops_storing_at_the_failed_chunk(plan):
    """The commit's fold kernel: a chunk wait that runs out leaves the
    checkpoint rows from that chunk on untouched and sets the bit."""
    from linear_attention_state_rssm_gb300 import _lib as L_
    T = 3
    run = Run(algo="gdn", HK=2, HV=4, dk=128, dv=128, L=8, max_T=T, slots=[0, 1],
              config_id=72, commit_mode="fold_every", plan=plan)
    inp = run.inputs(0, 0, T)
    run.window(0, inp, T)
    before = run.store.state.clone()
    run.store.rssm_debug_withhold(L_.withhold_chunk(3))
    acc = torch.full((run.B,), T, dtype=torch.int32, device="cuda")
    run.store.rssm_commit(run.slot_t, acc, T)
    assert run.store.rssm_get_device_error() & L_.DEVERR["timeout"]
    r0 = 3 * ROWS_PER_CHUNK
    assert torch.equal(run.store.state[..., r0:, :], before[..., r0:, :])
    # hook off: the same commit folds every chunk and matches the oracle
    run.store.rssm_debug_withhold(-1)
    run.store.state.copy_(before)
    run.store.cursor.zero_()
    run.commit(np.full(run.B, T, np.int32), T)
    run.check_cursors()
    assert run.state_err() <= TOL32
    assert run.store.rssm_get_device_error() == 0


def test_hook_arguments_are_checked():
    from linear_attention_state_rssm_gb300 import RssmError
    run = Run(algo="gdn", HK=1, HV=1, dk=32, dv=32, L=4, max_T=1, slots=[0], config_id=73)
    with pytest.raises(RssmError):
        run.store.rssm_debug_withhold(-2)              # no such barrier
    with pytest.raises(RssmError):
        run.store.rssm_debug_withhold(2 + 256)         # beyond the last chunk
    run.store.rssm_debug_withhold(-1)                  # off is always accepted
