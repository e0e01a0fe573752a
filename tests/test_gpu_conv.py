"""Conv-state window and rollback: CUDA path vs the fp64 oracle.

Outputs within 1e-5 (fp32) or 4e-3 (bf16, one output rounding) of the largest
oracle output; windows bit-exact (they hold copies of the inputs)."""
import numpy as np
import pytest
import torch

import synth
from oracle.conv import ACT_NONE, ACT_SILU, ConvOracle
from replay_harness import SENTINEL, TORCH, dev, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from linear_attention_state_rssm_gb300 import build
    build.build()


def _draw(rng, shape, dtype):
    return synth.quantize(rng.standard_normal(shape), dtype)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("K,act", [(4, "silu"), (2, "none"), (8, "silu")])
@pytest.mark.parametrize("D", [96, 1040])
def test_conv_decode_verify_commit_chain(dtype, K, act, D):
    from linear_attention_state_rssm_gb300.store import ConvWindows
    rng = np.random.Generator(np.random.PCG64(synth.seed_for(80, K, D)))
    slots = np.array([3, -1, 0, 4, 1], dtype=np.int32)
    B, n_slots, max_T = slots.size, 6, 5
    cw = ConvWindows(n_slots, D, K, max_T, dtype)
    win0 = _draw(rng, (n_slots, K - 1, D), dtype)
    cw.window.copy_(dev(win0, dtype))
    w = rng.standard_normal((D, K)).astype(np.float32).astype(np.float64)
    bias = rng.standard_normal(D).astype(np.float32).astype(np.float64)
    orc = ConvOracle(win0, w, bias, ACT_SILU if act == "silu" else ACT_NONE)
    w_t, b_t = dev(w, "f32"), dev(bias, "f32")
    slot_t = torch.from_numpy(slots).cuda()
    tol = 1e-5 if dtype == "f32" else 4e-3
    live = slots >= 0
    for step in range(8):
        T = 1 if step % 3 == 0 else int(rng.integers(2, max_T + 1))
        x = _draw(rng, (B * T, D), dtype)
        y = torch.full((B * T, D), SENTINEL, dtype=TORCH[dtype], device="cuda")
        decode = T == 1
        cw.rssm_conv_window(dev(x, dtype), w_t, b_t, slot_t, T, y, act=act, commit_now=decode)
        y_orc = orc.decode(slots, x) if decode else orc.window_step(slots, x, T)
        y_gpu = y.double().cpu().numpy()
        tok = np.repeat(live, T)
        assert rel_err(y_gpu[tok], y_orc[tok]) <= tol, step
        assert np.all(y_gpu[~tok] == SENTINEL)
        if not decode:
            acc = rng.integers(0, T + 1, B).astype(np.int32)
            cw.rssm_conv_commit(slot_t, torch.from_numpy(acc).cuda(), T)
            orc.commit(slots, acc)
        np.testing.assert_array_equal(cw.window.double().cpu().numpy(), orc.window)
    assert int(cw.err_word.item()) == 0


def test_conv_commit_refuses_accept_beyond_the_window():
    from linear_attention_state_rssm_gb300 import _lib as lib
    from linear_attention_state_rssm_gb300.store import ConvWindows
    cw = ConvWindows(2, 64, 4, 3, "f32")
    cw.window.normal_()
    before = cw.window.clone()
    slot = torch.tensor([0, 1], dtype=torch.int32, device="cuda")
    x = torch.randn(6, 64, device="cuda")
    y = torch.empty(6, 64, device="cuda")
    cw.rssm_conv_window(x, torch.randn(64, 4, device="cuda"), None, slot, 3, y)
    cw.rssm_conv_commit(slot, torch.tensor([4, 1], dtype=torch.int32, device="cuda"), 3)
    torch.cuda.synchronize()
    assert int(cw.err_word.item()) == lib.DEVERR["accept"]
    assert torch.equal(cw.window[0], before[0])        # refused row kept
    assert torch.equal(cw.window[1, :2], before[1, 1:])  # accepted one token
    assert torch.equal(cw.window[1, 2], x[3])
