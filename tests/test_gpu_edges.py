"""Edge cases of the CUDA path: forced folds, ring capacity, written positions,
device errors, argument checks, restore, determinism, CUDA graphs, every
supported head size and GQA group, the widest window, explicit folds."""
import numpy as np
import pytest
import torch

import synth
from replay_harness import Run, rel_err, SENTINEL, dev

pytestmark = pytest.mark.gpu
TOL32, TOL16 = 1e-4, 4e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from linear_attention_state_rssm_gb300 import build
    build.build()


def test_forced_folds_ragged_batch():
    B, T = 5, 3
    run = Run(algo="gdn", HK=2, HV=4, dk=64, dv=64, L=8, max_T=T, slots=[4, 0, 2, 1, 3],
              config_id=20)
    for step in range(14):
        inp = run.inputs(step, 0, T)
        force = synth.force_flags(2000 + step, B, 0.3)
        acc = synth.accept_lengths(2100 + step, B, T)
        _, o_gpu, o_orc, f_gpu, f_orc = run.window(0, inp, T, force=force)
        mask = (np.arange(T)[None, :] < acc[:, None]).reshape(-1)
        assert rel_err(o_gpu[mask], o_orc[mask]) <= TOL32, step
        np.testing.assert_array_equal(f_gpu, f_orc)
        run.commit(acc, T, force=force)
        run.check_cursors()
        run.check_ring_records()
        assert run.state_err() <= TOL32
    assert run.ring_d_err() <= TOL32


@pytest.mark.parametrize("algo", ["gdn", "kda"])
def test_ring_capacity_does_not_change_outputs(algo):
    """L = 16 and L = 64 fold at different steps; outputs agree within fp32 tolerance."""
    outs = []
    for L in (16, 64):
        run = Run(algo=algo, HK=2, HV=4, dk=128, dv=128, L=L, max_T=1, slots=[0, 1, 2],
                  config_id=21, sample=np.array([0]))
        seq = []
        for step in range(40):
            o_all, *_ = run.window(0, run.inputs(step, 0, 1), 1, decode=True, advance=True)
            seq.append(o_all)
        outs.append(np.array(seq))
    assert rel_err(outs[0], outs[1]) <= TOL32


def test_written_ring_positions_are_exact():
    """A verify writes exactly positions [base, base+T) of live slots."""
    T, L = 3, 8
    run = Run(algo="gdn", HK=2, HV=4, dk=32, dv=32, L=L, max_T=T, slots=[0, -1, 1, 2],
              n_slots=4, config_id=22)
    for step in range(6):
        inp = run.inputs(step, 0, T)
        acc = synth.accept_lengths(2200 + step, 4, T)
        run.store.ring_d.fill_(SENTINEL)
        run.window(0, inp, T)
        written = (run.store.ring_d[0] != SENTINEL).any(dim=-1).any(dim=1).cpu().numpy()
        for j, s in enumerate(run.orc_gpu_slots):
            np.testing.assert_array_equal(written[s], run.orc.written[0, j])
        assert not written[3].any()                  # slot 3 is never referenced
        run.commit(acc, T)
        run.check_cursors()
        run.check_ring_records()


def test_device_error_word_bad_slot_and_cursor():
    from linear_attention_state_rssm_gb300 import _lib as L_
    run = Run(algo="gdn", HK=1, HV=2, dk=32, dv=32, L=4, max_T=1, slots=[0, 1], config_id=23)
    inp = run.inputs(0, 0, 1)
    q, k, v, beta, g = run._gpu_inputs(inp)
    o = torch.full((2, 2, 32), SENTINEL, device="cuda")
    bad = torch.tensor([0, 9], dtype=torch.int32, device="cuda")        # 9 >= n_slots
    run.store.rssm_decode(0, q, k, v, beta, g, bad, o, advance_cursor=True)
    assert run.store.rssm_get_device_error() & L_.DEVERR["slot"]
    assert torch.all(o[1] == SENTINEL)
    assert run.store.rssm_get_device_error() == 0                        # cleared
    run.store.cursor[1] = 7                                              # > L
    o.fill_(SENTINEL)
    run.store.rssm_decode(0, q, k, v, beta, g, run.slot_t, o)
    assert run.store.rssm_get_device_error() & L_.DEVERR["cursor"]
    assert torch.all(o[1] == SENTINEL) and not torch.all(o[0] == SENTINEL)
    acc = torch.tensor([0, 5], dtype=torch.int32, device="cuda")
    run.store.cursor[1] = 0
    run.store.rssm_commit(run.slot_t, acc, 1)
    assert run.store.rssm_get_device_error() & L_.DEVERR["accept"]


def test_invalid_arguments_are_refused_before_launch():
    from linear_attention_state_rssm_gb300 import RssmError, ReplayStore
    st = ReplayStore("gdn", 2, 4, 1, 2, 32, 32, 8, 4, "f32", "f32")
    q = torch.zeros((4, 1, 32), device="cuda")
    v = torch.zeros((4, 2, 32), device="cuda")
    b = torch.zeros((4, 2), device="cuda")
    slot = torch.zeros(4, dtype=torch.int32, device="cuda")
    with pytest.raises(RssmError):                     # T > max_T
        st.rssm_verify(0, q, q, v, b, b, slot[:1], 5, v)
    with pytest.raises(RssmError):                     # layer out of range
        st.rssm_verify(2, q, q, v, b, b, slot[:1], 1, v)
    with pytest.raises(RssmError):                     # null output
        from linear_attention_state_rssm_gb300 import _lib as L_
        L_.rssm_verify(st.handle, 0, q, q, v, b, b, slot, None, 1, 1, None, None)
    with pytest.raises(RssmError):                     # ring shorter than the window
        ReplayStore("gdn", 1, 1, 1, 1, 32, 32, 4, 8)
    with pytest.raises(RssmError):                     # head size not built
        ReplayStore("gdn", 1, 1, 1, 1, 48, 32, 8, 1)
    empty = torch.zeros(0, dtype=torch.int32, device="cuda")
    st.rssm_verify(0, q, q, v, b, b, empty, 1, v)      # B == 0 is a no-op
    st.rssm_commit(empty, empty, 1)


def test_restore_copy_checkpoint_into_fresh_slot():
    """Fold slot 0, copy its checkpoint to slot 1, reset slot 1: both continue
    bit-identically and match the oracle."""
    run = Run(algo="gdn", HK=2, HV=4, dk=64, dv=64, L=8, max_T=1, slots=[0, 1], config_id=24)
    for step in range(11):
        run.window(0, run.inputs(step, 0, 1), 1, decode=True, advance=True)
    fold_slot = torch.tensor([0], dtype=torch.int32, device="cuda")
    run.store.rssm_fold(fold_slot)
    run.orc.fold([0])
    run.store.state[:, 1].copy_(run.store.state[:, 0])
    run.store.rssm_reset_slots(torch.tensor([1], dtype=torch.int32, device="cuda"))
    run.orc.load_checkpoint(1, run.orc.ckpt[:, 0])
    run.orc.reset_slots([1])
    assert run.state_err() <= TOL32
    for step in range(11, 20):
        inp = run.inputs(step, 0, 1)
        row0 = {key: val[0:1] for key, val in inp.items()}
        same = {key: np.concatenate([row0[key], row0[key]]) for key in inp}
        o_all, o_gpu, o_orc, _, _ = run.window(0, same, 1, decode=True, advance=True)
        np.testing.assert_array_equal(o_all[0], o_all[1])
        assert rel_err(o_gpu, o_orc) <= TOL32
        run.check_cursors()
        run.check_ring_records()


@pytest.mark.parametrize("plan", ["rows", "tc"])
@pytest.mark.parametrize("L,state,ring_k", [(16, "f32", "f32"), (16, "bf16", "f16"),
                                            (32, "f32", "f16"), (8, "f32", "bf16")])
def test_fold_call_of_every_history_length(L, state, ring_k, plan):
    """rssm_fold with 128-wide GDN heads after L decode steps in which row r
    (r < L) was forced to fold at step r: the rows fold histories of every
    length 1..L in one launch; the checkpoint matches the oracle, then the
    decode carries on from it."""
    B = L + 1
    tol = TOL32 if state == "f32" and ring_k == "f32" else TOL16
    run = Run(algo="gdn", HK=1, HV=2, dk=128, dv=128, L=L, max_T=1,
              slots=np.arange(B, dtype=np.int32), n_slots=B, state_dtype=state,
              ring_k_dtype=ring_k, config_id=35, plan=plan)
    for step in range(L):
        force = (np.arange(B) == step).astype(np.uint8)
        run.window(0, run.inputs(step, 0, 1), 1, force=force, decode=True, advance=True)
    np.testing.assert_array_equal(run.cursor_gpu(), [L - r for r in range(L)] + [L])
    run.fold(np.arange(B))
    run.check_cursors()
    assert run.state_err() <= tol
    for step in range(L, L + 3):
        _, o_gpu, o_orc, _, _ = run.window(0, run.inputs(step, 0, 1), 1, decode=True,
                                           advance=True)
        assert rel_err(o_gpu, o_orc) <= tol, step
        run.check_cursors()
    assert run.state_err() <= tol
    assert run.store.rssm_get_device_error() == 0


def test_runs_are_deterministic():
    res = []
    for _ in range(2):
        run = Run(algo="kda", HK=4, HV=4, dk=128, dv=128, L=8, max_T=4, slots=np.arange(6),
                  in_dtype="bf16", config_id=25, sample=np.array([0]))
        outs = []
        for step in range(9):
            o_all, *_ = run.window(0, run.inputs(step, 0, 4), 4)
            run.commit(synth.accept_lengths(2500 + step, 6, 4), 4)
            outs.append(o_all)
        res.append((np.array(outs), run.store.state.clone(), run.store.ring_d.clone()))
    np.testing.assert_array_equal(res[0][0], res[1][0])
    assert torch.equal(res[0][1], res[1][1]) and torch.equal(res[0][2], res[1][2])


def test_cuda_graph_capture_of_a_decode_step():
    """All layers of a decode step plus the cursor advance, captured once and
    replayed, match eager execution bit for bit."""
    from linear_attention_state_rssm_gb300 import ReplayStore
    nl, B = 3, 4
    stores, outs = [], []
    inps = [synth.window_inputs(synth.seed_for(26, 0, l), B, 1, 2, 4, 64, 64, "gdn", "bf16")
            for l in range(nl)]
    dev_inps = [[dev(x[key], "bf16" if key in "qkv" else "f32") for key in
                 ("q", "k", "v", "beta", "g")] for x in inps]
    slot = torch.arange(B, dtype=torch.int32, device="cuda")
    for use_graph in (False, True):
        st = ReplayStore("gdn", nl, B, 2, 4, 64, 64, 4, 1, "bf16", "f32")
        st.state.copy_(dev(np.stack([synth.initial_state(l, B, 4, 64, 64) for l in range(nl)]),
                           "f32"))
        o = torch.zeros((nl, B, 4, 64), dtype=torch.bfloat16, device="cuda")

        def step():
            for l in range(nl):
                st.rssm_decode(l, *dev_inps[l], slot, o[l], advance_cursor=(l == nl - 1))
        seq = []
        if use_graph:
            s = torch.cuda.Stream()
            s.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(s):
                graph = torch.cuda.CUDAGraph()
                with torch.cuda.graph(graph, stream=s):
                    step()
            torch.cuda.current_stream().wait_stream(s)
            for _ in range(7):
                graph.replay()
                seq.append(o.clone())
        else:
            for _ in range(7):
                step()
                seq.append(o.clone())
        torch.cuda.synchronize()
        stores.append(st)
        outs.append(torch.stack(seq))
    assert torch.equal(outs[0], outs[1])
    assert torch.equal(stores[0].state, stores[1].state)
    assert torch.equal(stores[0].cursor, stores[1].cursor)
    assert int(stores[0].cursor[0]) == 3          # 7 steps on L=4: folded once


@pytest.mark.parametrize("algo", ["gdn", "kda"])
@pytest.mark.parametrize("dk,dv,G", [(32, 32, 1), (64, 32, 2), (32, 128, 4), (128, 64, 8),
                                     (64, 64, 1), (64, 128, 16)])
def test_head_sizes_and_groups(algo, dk, dv, G):
    HK = 2
    HV = HK * G
    T = 2
    run = Run(algo=algo, HK=HK, HV=HV, dk=dk, dv=dv, L=5, max_T=T, slots=[1, 0, 2],
              config_id=27)
    for step in range(8):
        inp = run.inputs(step, 0, T)
        acc = synth.accept_lengths(2700 + step, 3, T)
        _, o_gpu, o_orc, f_gpu, f_orc = run.window(0, inp, T)
        mask = (np.arange(T)[None, :] < acc[:, None]).reshape(-1)
        assert rel_err(o_gpu[mask], o_orc[mask]) <= TOL32, step
        np.testing.assert_array_equal(f_gpu, f_orc)
        run.commit(acc, T)
        run.check_cursors()
        run.check_ring_records()
        assert run.state_err() <= TOL32


@pytest.mark.parametrize("algo", ["gdn", "kda"])
def test_widest_window_and_longest_ring(algo):
    """T = 16 windows on an L = 64 ring (long lazy history), fp32."""
    T = 16
    run = Run(algo=algo, HK=1, HV=2, dk=128, dv=128, L=64, max_T=T, slots=[0, 1],
              config_id=28)
    for step in range(7):
        inp = run.inputs(step, 0, T)
        acc = np.array([16, 11 if step % 2 else 16], dtype=np.int32)
        _, o_gpu, o_orc, f_gpu, f_orc = run.window(0, inp, T)
        mask = (np.arange(T)[None, :] < acc[:, None]).reshape(-1)
        assert rel_err(o_gpu[mask], o_orc[mask]) <= TOL32, step
        np.testing.assert_array_equal(f_gpu, f_orc)
        run.commit(acc, T)
        run.check_cursors()
        run.check_ring_records()
    assert run.ring_d_err() <= TOL32


def test_multi_layer_decode_moves_cursor_once_per_step():
    run = Run(algo="gdn", HK=2, HV=4, dk=64, dv=64, L=6, max_T=1, slots=[0, 1], n_layers=3,
              config_id=29)
    for step in range(15):
        for layer in range(3):
            _, o_gpu, o_orc, f_gpu, f_orc = run.window(layer, run.inputs(step, layer, 1), 1,
                                                       decode=True, advance=(layer == 2))
            assert rel_err(o_gpu, o_orc) <= TOL32, (step, layer)
            np.testing.assert_array_equal(f_gpu, f_orc)
        run.check_cursors()
        run.check_ring_records()
    assert run.state_err() <= TOL32


@pytest.mark.parametrize("B", [128, 160])
def test_decode_row_order_either_side_of_the_ranked_batch_limit(B):
    """Decode launches of up to 128 rows start their folding rows first (each
    CTA ranks the rows by fold decision); wider batches keep the grid order.
    On both sides of that limit, with permuted slots, null rows and forced
    folds, every row matches the oracle and null rows stay untouched."""
    rng = np.random.default_rng(31 + B)
    slots = rng.permutation(B + 8)[:B].astype(np.int32)
    null = rng.choice(B, 9, replace=False)
    slots[null] = -1
    run = Run(algo="gdn", HK=1, HV=2, dk=32, dv=32, L=4, max_T=1, slots=slots, n_slots=B + 8,
              config_id=32)
    live_rows = run.orc_slots >= 0
    for step in range(10):
        force = synth.force_flags(3200 + step, B, 0.1)
        o_all, o_gpu, o_orc, f_gpu, f_orc = run.window(0, run.inputs(step, 0, 1), 1, force=force,
                                                       decode=True, advance=True)
        assert rel_err(o_gpu[live_rows], o_orc[live_rows]) <= TOL32, step
        np.testing.assert_array_equal(f_gpu[live_rows], f_orc[live_rows])
        assert np.all(o_all[null] == SENTINEL), "null rows must be left untouched"
        run.check_cursors()
        run.check_ring_records()
    assert run.state_err() <= TOL32
    assert run.ring_d_err() <= TOL32
    assert run.store.rssm_get_device_error() == 0


@pytest.mark.parametrize("algo,HK,HV", [("gdn", 2, 4), ("kda", 2, 2)])
def test_decode_on_a_long_ring(algo, HK, HV):
    """Decode with 128-wide heads on an L = 64 ring (the largest shared-memory
    plan, long histories, the fold at c = 64): staggered cursors from forced
    folds, bf16 inputs, fp32 state; outputs every step, then the checkpoint."""
    B, L = 10, 64
    slots = np.arange(B, dtype=np.int32)[::-1].copy()
    run = Run(algo=algo, HK=HK, HV=HV, dk=128, dv=128, L=L, max_T=1, slots=slots,
              n_slots=B, in_dtype="bf16", config_id=29)
    for step in range(80):
        inp = run.inputs(step, 0, 1)
        force = np.array([1 if step == 5 * r + 3 else 0 for r in range(B)], dtype=np.uint8)
        _, o_gpu, o_orc, f_gpu, f_orc = run.window(0, inp, 1, force=force, decode=True,
                                                   advance=True)
        assert rel_err(o_gpu, o_orc) <= TOL16, step
        np.testing.assert_array_equal(f_gpu, f_orc)
        run.check_cursors()
        run.check_ring_records()
    assert run.state_err() <= TOL16
    assert run.ring_d_err() <= TOL16
    assert run.store.rssm_get_device_error() == 0


@pytest.mark.parametrize("plan", ["rows", "pipe"])
@pytest.mark.parametrize("state,ring_k", [("f32", "f32"), ("bf16", "f16"), ("f32", "bf16")])
def test_decode_fold_of_every_history_length(state, ring_k, plan):
    """GDN decode with 128-wide heads on an L = 16 ring: row r is forced to fold
    at step r, so one launch folds histories of every length 0..16 (then each
    row folds a full ring every 16 steps), for fp32 and bf16 checkpoints and
    fp32, fp16 and bf16 ring keys."""
    B, L = 17, 16
    slots = np.arange(B, dtype=np.int32)
    tol = TOL32 if state == "f32" and ring_k == "f32" else TOL16
    run = Run(algo="gdn", HK=1, HV=2, dk=128, dv=128, L=L, max_T=1, slots=slots, n_slots=B,
              state_dtype=state, ring_k_dtype=ring_k, config_id=33, plan=plan)
    for step in range(36):
        force = (np.arange(B) == step).astype(np.uint8)
        _, o_gpu, o_orc, f_gpu, f_orc = run.window(0, run.inputs(step, 0, 1), 1, force=force,
                                                   decode=True, advance=True)
        assert rel_err(o_gpu, o_orc) <= tol, step
        np.testing.assert_array_equal(f_gpu, f_orc)
        run.check_cursors()
        run.check_ring_records()
        assert run.state_err() <= tol, step
    assert run.ring_d_err() <= tol
    assert run.store.rssm_get_device_error() == 0


@pytest.mark.parametrize("algo,plan", [("gdn", "rows"), ("gdn", "pipe"), ("gdn", "tc"),
                                       ("kda", "rows")])
@pytest.mark.parametrize("T", [1, 2, 3, 8])
@pytest.mark.parametrize("in_dt,ring_k,state", [("f32", "f32", "f32"), ("f32", "bf16", "f32"),
                                                ("bf16", "f32", "bf16"), ("bf16", "f16", "f32")])
def test_verify_across_input_key_and_state_dtypes(in_dt, ring_k, state, T, algo, plan):
    """Three- and eight-token GDN and KDA verify + commit with 128-wide heads
    (fp32 and 16-bit inputs, ring keys and checkpoints), forced folds on top of
    the ring's own, accept lengths U[0, T]: outputs, fold flags, cursors and
    checkpoints vs the oracle."""
    B, L = 12, 16
    tol = TOL32 if (in_dt, ring_k, state) == ("f32", "f32", "f32") else TOL16
    run = Run(algo=algo, HK=1, HV=2, dk=128, dv=128, L=L, max_T=T,
              slots=np.arange(B, dtype=np.int32), n_slots=B, in_dtype=in_dt, state_dtype=state,
              ring_k_dtype=ring_k, config_id=34, plan=plan)
    for step in range(14):
        inp = run.inputs(step, 0, T)
        force = synth.force_flags(3400 + step, B, 0.15)
        acc = synth.accept_lengths(3500 + step, B, T)
        _, o_gpu, o_orc, f_gpu, f_orc = run.window(0, inp, T, force=force)
        mask = (np.arange(T)[None, :] < acc[:, None]).reshape(-1)
        assert rel_err(o_gpu[mask], o_orc[mask]) <= tol, step
        np.testing.assert_array_equal(f_gpu, f_orc)
        run.commit(acc, T, force=force)
        run.check_cursors()
        run.check_ring_records()
        assert run.state_err() <= tol, step
    assert run.ring_d_err() <= tol
    assert run.store.rssm_get_device_error() == 0
