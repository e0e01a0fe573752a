"""Drive the CUDA store (through the C ABI) and the fp64 oracle on the same
seeded inputs, and measure their differences. Test-side only."""
from __future__ import annotations

import numpy as np
import torch

import synth
from oracle import ReplayOracle, ring

TORCH = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}
SENTINEL = 12288.0   # exact in fp32, bf16 and fp16


def dev(x, dtype):
    """Exact upload of values already on the dtype grid."""
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float64)).to(
        device="cuda", dtype=TORCH[dtype])


def rel_err(a, b, mask=None):
    """max|a - b| / max|b| over the (masked) elements; both float64."""
    if mask is not None:
        a, b = a[mask], b[mask]
    if b.size == 0:
        return 0.0
    den = np.max(np.abs(b))
    return float(np.max(np.abs(a - b)) / den) if den > 0 else float(np.max(np.abs(a - b)))


class Run:
    """One store on the GPU and its oracle, over rows ``sample`` of the batch."""

    def __init__(self, *, algo="gdn", HK, HV, dk, dv, L, max_T, slots, n_slots=None,
                 n_layers=1, in_dtype="f32", state_dtype="f32", ring_k_dtype=None,
                 ring_d_dtype="f32", commit_mode="lazy", config_id=0, sample=None,
                 plan="auto"):
        from linear_attention_state_rssm_gb300 import ReplayStore
        self.algo, self.HK, self.HV, self.dk, self.dv, self.L = algo, HK, HV, dk, dv, L
        self.in_dtype, self.state_dtype, self.config_id = in_dtype, state_dtype, config_id
        self.commit_mode = commit_mode
        self.slots = np.asarray(slots, dtype=np.int32)
        self.B = self.slots.size
        self.n_slots = int(n_slots if n_slots is not None else max(self.slots.max() + 1, 1))
        self.n_layers = n_layers
        self.store = ReplayStore(algo, n_layers, self.n_slots, HK, HV, dk, dv, L, max_T,
                                 in_dtype, state_dtype, ring_k_dtype, ring_d_dtype, commit_mode)
        self.store.rssm_set_plan(plan)   # which kernel serves decode and verify
        S0 = np.stack([synth.initial_state(synth.seed_for(config_id, 10_000, l), self.n_slots,
                                           HV, dk, dv, state_dtype) for l in range(n_layers)])
        self.store.state.copy_(dev(S0, state_dtype))
        self.slot_t = torch.from_numpy(self.slots).cuda()
        # oracle over the sampled rows' slots (rows are independent)
        self.sample = np.arange(self.B) if sample is None else np.asarray(sample)
        live_slots = sorted({int(self.slots[r]) for r in self.sample if self.slots[r] >= 0})
        self.orc_index = {s: j for j, s in enumerate(live_slots)}
        self.orc_slots = np.array([self.orc_index.get(int(self.slots[r]), -1)
                                   for r in self.sample], dtype=np.int64)
        self.orc_gpu_slots = np.array(live_slots, dtype=np.int64)
        S0o = S0[:, live_slots] if live_slots else S0[:, :1]
        no = max(len(live_slots), 1)
        rd = "f16" if ring_d_dtype == "f16" else "f32"
        self.orc = ReplayOracle(algo, n_layers, no, HK, HV, dk, dv, L, self.store.scale, S0o,
                                ring_d_dtype=rd)
        # A bf16 checkpoint is also checked against a chain that rounds its
        # checkpoint to bf16 at the same folds (outputs use the exact chain).
        self.orc_r = (ReplayOracle(algo, n_layers, no, HK, HV, dk, dv, L, self.store.scale, S0o,
                                   ckpt_round="bf16", ring_d_dtype=rd)
                      if state_dtype == "bf16" else None)

    def narrow(self, sample):
        """From now on the oracle follows (and the checks compare) only rows
        ``sample``, which must be among the rows followed so far."""
        sample = np.asarray(sample)
        live_slots = sorted({int(self.slots[r]) for r in sample if self.slots[r] >= 0})
        keep = [self.orc_index[s] for s in live_slots]
        for orc in (self.orc, self.orc_r):
            if orc is not None:
                orc.select_slots(keep)
        self.sample = sample
        self.orc_index = {s: j for j, s in enumerate(live_slots)}
        self.orc_slots = np.array([self.orc_index.get(int(self.slots[r]), -1)
                                   for r in sample], dtype=np.int64)
        self.orc_gpu_slots = np.array(live_slots, dtype=np.int64)

    # ------------------------------------------------------------------ inputs
    def inputs(self, step, layer, T):
        return synth.window_inputs(synth.seed_for(self.config_id, step, layer), self.B, T,
                                   self.HK, self.HV, self.dk, self.dv, self.algo, self.in_dtype)

    def _sub(self, inp, T):
        tok = (self.sample[:, None] * T + np.arange(T)[None, :]).reshape(-1)
        return {key: val[tok] for key, val in inp.items()}

    def _gpu_inputs(self, inp):
        return (dev(inp["q"], self.in_dtype), dev(inp["k"], self.in_dtype),
                dev(inp["v"], self.in_dtype), dev(inp["beta"], "f32"), dev(inp["g"], "f32"))

    # ------------------------------------------------------------------ steps
    def window(self, layer, inp, T, force=None, decode=False, advance=False):
        """Run one layer's window on both sides. Returns (o_gpu_all, o_gpu,
        o_orc, fold_gpu, fold_orc): the GPU output of every row, then the GPU
        output, oracle output and fold flags of the sampled rows."""
        q, k, v, beta, g = self._gpu_inputs(inp)
        o = torch.full((self.B * T, self.HV, self.dv), SENTINEL, dtype=TORCH[self.in_dtype],
                       device="cuda")
        fold_out = torch.full((self.B,), 7, dtype=torch.uint8, device="cuda")
        force_t = None if force is None else torch.from_numpy(np.asarray(force, np.uint8)).cuda()
        if decode:
            self.store.rssm_decode(layer, q, k, v, beta, g, self.slot_t, o, force=force_t,
                                   fold_out=fold_out, advance_cursor=advance)
        else:
            self.store.rssm_verify(layer, q, k, v, beta, g, self.slot_t, T, o, force=force_t,
                                   fold_out=fold_out)
        sub = self._sub(inp, T)
        fsub = None if force is None else np.asarray(force)[self.sample]
        if decode:
            o_orc, f_orc = self.orc.decode(layer, self.orc_slots, sub, fsub, advance)
            if self.orc_r is not None:
                self.orc_r.decode(layer, self.orc_slots, sub, fsub, advance)
        else:
            o_orc, f_orc = self.orc.window(layer, self.orc_slots, sub, T, fsub)
            if self.orc_r is not None:
                self.orc_r.window(layer, self.orc_slots, sub, T, fsub)
        o_gpu = o.double().cpu().numpy()
        tok = (self.sample[:, None] * T + np.arange(T)[None, :]).reshape(-1)
        return o_gpu, o_gpu[tok], o_orc, fold_out.cpu().numpy()[self.sample], f_orc

    def commit(self, accept, T, force=None):
        acc_t = torch.from_numpy(np.asarray(accept, np.int32)).cuda()
        force_t = None if force is None else torch.from_numpy(np.asarray(force, np.uint8)).cuda()
        self.store.rssm_commit(self.slot_t, acc_t, T, force=force_t)
        mode = ring.FOLD_EVERY if self.commit_mode == "fold_every" else ring.LAZY
        fsub = None if force is None else np.asarray(force)[self.sample]
        self.orc.commit(self.orc_slots, np.asarray(accept)[self.sample], T, fsub, mode)
        if self.orc_r is not None:
            self.orc_r.commit(self.orc_slots, np.asarray(accept)[self.sample], T, fsub, mode)

    # ----------------------------------------------------------- ragged steps
    def window_ragged(self, layer, inp, cu, max_T, force=None):
        """Ragged verify of one layer on both sides (every row is sampled).
        ``inp`` holds the packed tokens (at least cu[-1] of them). Returns
        (o_gpu, o_orc, fold_gpu, fold_orc) over all packed tokens / rows."""
        assert self.sample.size == self.B
        q, k, v, beta, g = self._gpu_inputs(inp)
        n_tok = inp["q"].shape[0]
        o = torch.full((n_tok, self.HV, self.dv), SENTINEL, dtype=TORCH[self.in_dtype],
                       device="cuda")
        fold_out = torch.full((self.B,), 7, dtype=torch.uint8, device="cuda")
        force_t = None if force is None else torch.from_numpy(np.asarray(force, np.uint8)).cuda()
        cu_t = torch.from_numpy(np.asarray(cu, np.int32)).cuda()
        self.store.rssm_verify_ragged(layer, q, k, v, beta, g, cu_t, self.slot_t, max_T, o,
                                      force=force_t, fold_out=fold_out)
        o_orc, f_orc = self.orc.window_ragged(layer, self.orc_slots, inp, cu, force)
        if self.orc_r is not None:
            self.orc_r.window_ragged(layer, self.orc_slots, inp, cu, force)
        return o.double().cpu().numpy(), o_orc, fold_out.cpu().numpy(), f_orc

    def commit_ragged(self, accept, cu, max_T, force=None):
        acc_t = torch.from_numpy(np.asarray(accept, np.int32)).cuda()
        force_t = None if force is None else torch.from_numpy(np.asarray(force, np.uint8)).cuda()
        cu_t = torch.from_numpy(np.asarray(cu, np.int32)).cuda()
        self.store.rssm_commit_ragged(self.slot_t, acc_t, cu_t, max_T, force=force_t)
        mode = ring.FOLD_EVERY if self.commit_mode == "fold_every" else ring.LAZY
        self.orc.commit_ragged(self.orc_slots, accept, cu, force, mode)
        if self.orc_r is not None:
            self.orc_r.commit_ragged(self.orc_slots, accept, cu, force, mode)

    # ---------------------------------------------------------------- prefill
    def prefill(self, layer, inp, cu, reset_cursor):
        """Replay prefill of one layer on both sides (every row sampled);
        returns (o_gpu, o_orc) over the packed tokens (the GPU buffer may hold
        spare tokens past cu[-1])."""
        assert self.sample.size == self.B
        q, k, v, beta, g = self._gpu_inputs(inp)
        n_tok = inp["q"].shape[0]
        o = torch.full((n_tok, self.HV, self.dv), SENTINEL, dtype=TORCH[self.in_dtype],
                       device="cuda")
        cu_t = torch.from_numpy(np.asarray(cu, np.int32)).cuda()
        self.store.rssm_prefill(layer, q, k, v, beta, g, cu_t, self.slot_t, o,
                                reset_cursor=reset_cursor)
        o_orc = self.orc.prefill(layer, self.orc_slots, inp, cu)
        if self.orc_r is not None:
            self.orc_r.prefill(layer, self.orc_slots, inp, cu)
        if reset_cursor:
            self.orc.prefill_done(self.orc_slots, cu)
            if self.orc_r is not None:
                self.orc_r.prefill_done(self.orc_slots, cu)
        return o.double().cpu().numpy(), o_orc

    # ------------------------------------------------------------- inspection
    def fold(self, slots):
        """rssm_fold of the given slots on the GPU and in both oracles."""
        self.store.rssm_fold(torch.as_tensor(np.asarray(slots, dtype=np.int32)).cuda())
        orc_slots = [self.orc_index[int(s)] for s in slots if int(s) in self.orc_index]
        for orc in (self.orc, self.orc_r):
            if orc is not None:
                orc.fold(orc_slots)

    def cursor_gpu(self):
        return self.store.cursor.cpu().numpy()

    def check_cursors(self):
        """GPU cursors of the oracle's slots equal the oracle's, bit for bit."""
        cur = self.cursor_gpu()
        np.testing.assert_array_equal(cur[self.orc_gpu_slots], self.orc.cursor[:len(self.orc_gpu_slots)])

    def state_err(self):
        """Checkpoint (GPU) vs the checkpoint the oracle says it must hold.

        For a bf16 checkpoint the reference is the chain that rounds at the same
        folds, and one bf16 ulp per element is allowed on top: where the fp32
        and fp64 values of an element fall on opposite sides of a rounding
        boundary, the two roundings differ by exactly one ulp."""
        S = self.store.state.double().cpu().numpy()[:, self.orc_gpu_slots]
        n = len(self.orc_gpu_slots)
        if self.orc_r is None:
            return rel_err(S, self.orc.ckpt[:, :n])
        ref = self.orc_r.ckpt[:, :n]
        ulp = np.ldexp(1.0, np.frexp(np.abs(ref))[1] - 8)
        excess = np.maximum(np.abs(S - ref) - ulp, 0.0)
        return float(np.max(excess) / np.max(np.abs(ref)))

    def check_ring_records(self):
        """Ring records k, g, v and beta of the oracle's slots equal the
        oracle's bit for bit (keys after rounding to the ring-key dtype, each
        value head holding its key head's key) at every position the last
        window of each layer wrote and every committed position [0, cursor);
        non-finite values of rejected drafts must match as well."""
        sl = self.orc_gpu_slots
        n = len(sl)
        if n == 0:
            return
        orc, st, G = self.orc, self.store, self.HV // self.HK
        pos = np.arange(self.L)
        mask = orc.written[:, :n] | (pos[None, None, :] < orc.cursor[None, :n, None])
        got = {"k": st.ring_k, "g": st.ring_g, "v": st.ring_v, "beta": st.ring_beta}
        want = {"k": synth.quantize(np.repeat(orc.ring_k[:, :n], G, axis=2), st.ring_k_dtype),
                "g": orc.ring_g[:, :n], "v": orc.ring_v[:, :n], "beta": orc.ring_beta[:, :n]}
        for name in ("k", "g", "v", "beta"):
            a = got[name].double().cpu().numpy()[:, sl]
            b = want[name]
            m = np.broadcast_to(mask[:, :, None, :].reshape(mask.shape[:2] + (1, self.L) +
                                                            (1,) * (a.ndim - 4)), a.shape)
            assert np.array_equal(a[m], b[m], equal_nan=True), (
                f"ring_{name} differs at {np.count_nonzero(~np.isclose(a[m], b[m], equal_nan=True))}"
                f" of {np.count_nonzero(m)} checked values")

    def check_no_fp16_delta_overflow(self):
        """An fp16 delta ring stayed inside the fp16 range (oracle flag)."""
        assert not self.orc.d_overflow.any(), "an accepted delta exceeds the fp16 range"

    def ring_d_err(self):
        """Committed history records d[0, cursor) vs the oracle's."""
        d = self.store.ring_d.double().cpu().numpy()[:, self.orc_gpu_slots]
        mask = np.zeros(d.shape, dtype=bool)
        for j, s in enumerate(self.orc_gpu_slots):
            mask[:, j, :, :int(self.orc.cursor[j])] = True
        return rel_err(d, self.orc.ring_d[:, :len(self.orc_gpu_slots)], mask)
