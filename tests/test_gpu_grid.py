"""Every kernel configuration the steady-state throughput grid launches, at
its dtypes (bf16 inputs, fp16 ring keys, fp32 deltas, lazy commit) and head
size (dk = dv = 128): GDN and KDA, ring lengths 16, 32 and 64, windows of 1, 3
and 8 tokens, fp32 and bf16 checkpoints. Each chain runs long enough that the
rows' cursors reach the end of the ring and fold inside the kernel (forced
folds in the first steps stagger them); outputs, fold flags, cursors, ring
records and checkpoints are compared with the fp64 oracle after every step."""
import numpy as np
import pytest
import torch

import synth
from replay_harness import Run, rel_err

pytestmark = pytest.mark.gpu
TOL16 = 4e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from linear_attention_state_rssm_gb300 import build
    build.build()


def _chain(algo, L, T, state, ring_k="f16"):
    B = 5
    HK, HV = (1, 2) if algo == "gdn" else (2, 2)
    run = Run(algo=algo, HK=HK, HV=HV, dk=128, dv=128, L=L, max_T=T,
              slots=np.arange(B, dtype=np.int32), n_slots=B, in_dtype="bf16",
              state_dtype=state, ring_k_dtype=ring_k, config_id=40 + L + T)
    steps = L + 6 if T == 1 else -(-5 * L // (2 * T)) + 4
    folds = np.zeros(B, dtype=np.int64)
    overflow = False
    for step in range(steps):
        inp = run.inputs(step, 0, T)
        force = synth.force_flags(4000 + 97 * L + step, B, 0.3 if step < 4 else 0.0)
        if T == 1:
            _, o_gpu, o_orc, f_gpu, f_orc = run.window(0, inp, 1, force=force, decode=True,
                                                       advance=True)
            assert rel_err(o_gpu, o_orc) <= TOL16, step
        else:
            _, o_gpu, o_orc, f_gpu, f_orc = run.window(0, inp, T, force=force)
            acc = synth.accept_lengths(4100 + 97 * L + step, B, T)
            mask = (np.arange(T)[None, :] < acc[:, None]).reshape(-1)
            assert rel_err(o_gpu[mask], o_orc[mask]) <= TOL16, step
            run.commit(acc, T, force=force)
        np.testing.assert_array_equal(f_gpu, f_orc)
        folds += f_gpu.astype(np.int64)
        overflow |= bool((f_gpu.astype(bool) & ~force.astype(bool)).any())
        run.check_cursors()
        run.check_ring_records()
        assert run.state_err() <= TOL16, step
    assert (folds > 0).all(), "a row never folded"
    assert overflow, "no window folded for lack of ring room"
    assert run.ring_d_err() <= TOL16
    assert run.store.rssm_get_device_error() == 0


@pytest.mark.parametrize("state", ["f32", "bf16"])
@pytest.mark.parametrize("T", [1, 3, 8])
@pytest.mark.parametrize("L", [16, 32, 64])
@pytest.mark.parametrize("algo", ["gdn", "kda"])
def test_grid_configuration(algo, L, T, state):
    _chain(algo, L, T, state)


@pytest.mark.parametrize("state", ["f32", "bf16"])
@pytest.mark.parametrize("L", [32, 64])
def test_long_ring_decode_with_bf16_ring_keys(L, state):
    """GDN decode on long rings with bf16 ring keys: the fold reads the keys as
    they landed, transposed in place (the 16-bit key path of long rings)."""
    _chain("gdn", L, 1, state, ring_k="bf16")
