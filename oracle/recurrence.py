"""fp64 sequential oracle of the ReplaySSM hot path (GDN and KDA).

Test infrastructure only: the CUDA path never imports, links or runs this file.
Only tests, the package's smoke check and the benchmark's CPU-baseline leg use it.

What it computes, restated from the pages:

* The gated delta rule, one token at a time, for every request slot and value
  head (value head h reads key head h // G, adjacent value heads sharing a key
  head: LightLLM PR #1690 "feat: add ReplaySSM state modes for GDN and KDA",
  commit messages on grouped GDN key groups)::

      GDN:  S <- exp(g) * S                 (one log-decay per value head)
      KDA:  S <- diag(exp(g)) @ S            (one log-decay per key channel)
      d    = beta * (v - S^T k)              (the delta; kept fp32 in the ring)
      S   <- S + k d^T
      o    = scale * S^T q

* The exact committed state is carried forward. The oracle never replays: the
  whole point of ReplaySSM is that a checkpoint plus a ring of accepted records
  reproduces this same state, so the oracle keeps the state itself and, beside
  it, the checkpoint value the GPU must hold and the ring records the GPU must
  write (LightLLM PR #1690, PR description: the checkpoint is the canonical SSM
  state, deltas are stored in fp32).
* Ring, cursor and fold decisions follow ``oracle.ring``: a window folds when
  forced or when it would overflow the ring, and the fold makes the checkpoint
  equal to the committed state (in exact arithmetic a fold changes nothing).
* Speculative verify (SGLang fork PR jianc99/sglang#2, commits on the verify
  and the commit): a window of T draft tokens runs from the committed state and
  writes its T records; commit keeps the first ``a`` tokens, trims the rest,
  and in fold-every mode folds them into the checkpoint. Rejected positions
  never reach the committed state: commit re-runs only the accepted tokens.

Inputs are float64 arrays whose values are already the quantised values the
GPU sees (bf16 inputs widened exactly). Layouts are token-major:
q, k [B*T, HK, dk]; v [B*T, HV, dv]; beta [B*T, HV]; g [B*T, HV] (GDN) or
[B*T, HV, dk] (KDA). Row r's token i is index r*T + i; a row whose slot is -1
is a null row and is skipped entirely.
"""
from __future__ import annotations

import numpy as np

from . import ring

__all__ = ["token_step", "ReplayOracle", "round_bf16", "FP16_MAX"]

FP16_MAX = 65504.0  # largest finite IEEE half-precision value


def round_bf16(x):
    """Round float64 values to the nearest bfloat16 value, ties to even.

    bfloat16 keeps 8 significant bits (1 implicit + 7 stored) and the float32
    exponent range. With x = m * 2**e, 0.5 <= |m| < 1, the nearest value is
    rint(m * 2**8) * 2**(e - 8); numpy's rint rounds halves to even. Non-finite
    values pass through. (Values below the float32 normal range, never met
    here, keep 8 bits instead of becoming bfloat16 subnormals.)
    """
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)
    r = np.ldexp(np.rint(np.ldexp(m, 8)), e - 8)
    return np.where(np.isfinite(x), r, x)


def token_step(S, q, k, v, beta, g, scale, algo):
    """Advance states S [R, HV, dk, dv] by one token.

    q, k: [R, HV, dk] (key heads already mapped onto value heads); v: [R, HV, dv];
    beta: [R, HV]; g: [R, HV] (gdn) or [R, HV, dk] (kda). Returns the new
    state, the delta d [R, HV, dv] and the output o [R, HV, dv].
    """
    if algo == "gdn":
        S = np.exp(g)[:, :, None, None] * S
    elif algo == "kda":
        S = np.exp(g)[:, :, :, None] * S
    else:
        raise ValueError(algo)
    Stk = np.matmul(k[:, :, None, :], S)[:, :, 0, :]          # S^T k
    d = beta[:, :, None] * (v - Stk)
    S += k[:, :, :, None] * d[:, :, None, :]                  # S is a fresh array here
    o = scale * np.matmul(q[:, :, None, :], S)[:, :, 0, :]     # S^T q
    return S, d, o


class ReplayOracle:
    """Sequential fp64 model of one ReplaySSM store (all layers, all slots).

    State kept per (layer, slot): ``S`` the exact committed state, ``ckpt`` the
    value the GPU checkpoint must hold, and the ring records each window wrote.
    ``cursor`` is shared by all layers of a slot, as on the GPU.
    """

    def __init__(self, algo, n_layers, n_slots, HK, HV, dk, dv, L, scale, S0,
                 ckpt_round=None, ring_d_dtype="f32"):
        """``ckpt_round="bf16"`` models a bf16 checkpoint: at every fold the
        committed state is rounded to bf16 and the chain continues from the
        rounded value, as the GPU does (vLLM PR #64699, commit message on
        accounting for BF16 state rounding between flushes).

        ``ring_d_dtype="f16"`` models a store that keeps its deltas in fp16,
        against LightLLM PR #1690 (PR description: deltas are kept in fp32
        because fp16 deltas overflow). The recurrence stays fp64; the oracle
        only flags, per (layer, slot), every accepted delta whose magnitude
        exceeds 65504, the largest finite fp16 value (``d_overflow``), so a
        run in that configuration can show it stayed inside the fp16 range."""
        if HV % HK:
            raise ValueError("HV must be a multiple of HK")
        self.algo, self.n_layers, self.n_slots = algo, n_layers, n_slots
        self.HK, self.HV, self.dk, self.dv, self.L = HK, HV, dk, dv, L
        self.G = HV // HK
        self.scale = float(scale)
        if ckpt_round not in (None, "bf16"):
            raise ValueError(ckpt_round)
        self.ckpt_round = ckpt_round
        if ring_d_dtype not in ("f32", "f16"):
            raise ValueError(ring_d_dtype)
        self.ring_d_dtype = ring_d_dtype
        S0 = np.asarray(S0, dtype=np.float64)
        if S0.shape == (n_slots, HV, dk, dv):
            S0 = np.broadcast_to(S0, (n_layers,) + S0.shape)
        assert S0.shape == (n_layers, n_slots, HV, dk, dv)
        self.S = np.array(S0, dtype=np.float64)
        self.ckpt = self.S.copy()
        self.cursor = np.zeros(n_slots, dtype=np.int64)
        ng = () if algo == "gdn" else (dk,)
        nan = np.nan
        self.ring_k = np.full((n_layers, n_slots, HK, L, dk), nan)
        self.ring_d = np.full((n_layers, n_slots, HV, L, dv), nan)
        self.ring_g = np.full((n_layers, n_slots, HV, L) + ng, nan)
        self.ring_v = np.full((n_layers, n_slots, HV, L, dv), nan)
        self.ring_beta = np.full((n_layers, n_slots, HV, L), nan)
        # positions [base, base+T) written by the last window of each layer
        self.written = np.zeros((n_layers, n_slots, L), dtype=bool)
        # accepted deltas outside the fp16 range (only tracked for an fp16 delta ring)
        self.d_overflow = np.zeros((n_layers, n_slots), dtype=bool)
        self._pending: dict[int, dict] = {}
        # rows per batch of work: keeps each temporary near 16 MB
        self._chunk = max(1, (16 << 20) // (HV * dk * dv * 8))

    # ------------------------------------------------------------------ helpers
    def _expand(self, x):
        """[R, HK, dk] -> [R, HV, dk]: value head h uses key head h // G."""
        return np.repeat(x, self.G, axis=1)

    def _decide(self, slots, lens, force):
        B = len(slots)
        fold = np.zeros(B, dtype=bool)
        base = np.zeros(B, dtype=np.int64)
        for r in range(B):
            s = int(slots[r])
            if s < 0 or lens[r] == 0:
                continue
            f, b = ring.fold_decision(int(self.cursor[s]), int(lens[r]), self.L,
                                      bool(force[r]))
            fold[r], base[r] = f, b
        return fold, base

    def _checkpoint(self, layer, slots):
        """Fold: the checkpoint takes the committed state (rounded to the
        checkpoint dtype when modelled; the chain then continues from it)."""
        if self.ckpt_round == "bf16":
            self.S[layer, slots] = round_bf16(self.S[layer, slots])
        self.ckpt[layer, slots] = self.S[layer, slots]

    def _token_inputs(self, inp, idx):
        return (self._expand(inp["q"][idx]), self._expand(inp["k"][idx]),
                inp["v"][idx], inp["beta"][idx], inp["g"][idx])

    # --------------------------------------------------------------- hot path
    def window(self, layer, slots, inp, T, force=None):
        """Run one T-token window (decode: T=1) for every live row of one layer.

        Returns (o, fold): o [B*T, HV, dv] with NaN on null rows; fold [B]
        int8, 1 where the window folded, 0 where not, -1 on null rows.
        """
        B = len(slots)
        if not 1 <= T <= self.L:
            raise ValueError("window must satisfy 1 <= T <= L")
        starts = np.arange(B, dtype=np.int64) * T
        lens = np.full(B, T, dtype=np.int64)
        return self._window(layer, slots, inp, starts, lens, B * T, T, force)

    def window_ragged(self, layer, slots, inp, cu_seqlens, force=None):
        """Windows of different lengths packed into one token list: row r's
        tokens are [cu_seqlens[r], cu_seqlens[r+1]) (LightLLM PR #1690, commit
        messages: request windows read from cu_seqlens over [tokens, heads,
        dim] inputs; SGLang fork PR jianc99/sglang#2, "Related upstream work":
        verify on packed ragged tokens). A row with no tokens is idle this
        step, like a null row: no fold, no output, no record.

        Returns (o, fold) as ``window`` does, o over the packed tokens.
        """
        cu = np.asarray(cu_seqlens, dtype=np.int64)
        lens = np.diff(cu)
        if cu.shape[0] != len(slots) + 1 or np.any(lens < 0) or np.any(lens > self.L):
            raise ValueError("cu_seqlens must be non-decreasing with windows of at most L")
        return self._window(layer, slots, inp, cu[:-1].copy(), lens, int(cu[-1]), None, force)

    def _window(self, layer, slots, inp, starts, lens, n_tok, T, force):
        slots = np.asarray(slots, dtype=np.int64)
        B = slots.shape[0]
        force = np.zeros(B, np.uint8) if force is None else np.asarray(force)
        fold, base = self._decide(slots, lens, force)
        active = (slots >= 0) & (lens > 0)
        live = np.nonzero(active)[0]
        o = np.full((n_tok, self.HV, self.dv), np.nan)
        over = np.zeros((B, int(lens.max()) if B else 0), dtype=bool)
        flags = np.where(active, fold.astype(np.int8), np.int8(-1))
        if live.size:
            sl = slots[live]
            folded = sl[fold[live]]
            # A fold makes the checkpoint the committed state and empties the ring.
            self._checkpoint(layer, folded)
            self.written[layer, sl] = False
            final = np.empty((live.size, self.HV, self.dk, self.dv))
            with np.errstate(all="ignore"):
                for c0 in range(0, live.size, self._chunk):
                    rows = live[c0:c0 + self._chunk]
                    final[c0:c0 + rows.size] = self._run_window(layer, rows, slots, inp, starts,
                                                                lens, base, o, over)
        else:
            final = None
        self._pending[layer] = {"slots": slots.copy(), "inp": inp, "T": T, "starts": starts,
                                "lens": lens, "force": np.asarray(force).copy(), "base": base,
                                "final": final, "over": over}
        return o, flags

    def _run_window(self, layer, rows, slots, inp, starts, lens, base, o, over):
        """Run the window tokens of some live rows; record outputs and ring
        records (and, for an fp16 delta ring, which tokens' deltas leave the
        fp16 range in ``over``); return the rows' states after their windows."""
        sl = slots[rows]
        S = self.S[layer, sl]                     # fancy indexing: a copy
        for i in range(int(lens[rows].max())):
            on = np.nonzero(lens[rows] > i)[0]   # rows whose window has token i
            r_i, s_i = rows[on], sl[on]
            idx = starts[r_i] + i
            q, k, v, beta, g = self._token_inputs(inp, idx)
            S[on], d, oi = token_step(S[on], q, k, v, beta, g, self.scale, self.algo)
            o[idx] = oi
            if self.ring_d_dtype == "f16":
                over[r_i, i] = np.any(np.abs(d) > FP16_MAX, axis=(1, 2))
            pos = base[r_i] + i
            self.ring_k[layer, s_i, :, pos] = inp["k"][idx]
            self.ring_d[layer, s_i, :, pos] = d
            self.ring_g[layer, s_i, :, pos] = inp["g"][idx]
            self.ring_v[layer, s_i, :, pos] = v
            self.ring_beta[layer, s_i, :, pos] = beta
            self.written[layer, s_i, pos] = True
        return S

    def _accept(self, layer, accept):
        """Commit ``accept[r]`` tokens of the pending window of one layer."""
        pend = self._pending.pop(layer)
        slots, inp, final = pend["slots"], pend["inp"], pend["final"]
        starts, lens = pend["starts"], pend["lens"]
        live = np.nonzero((slots >= 0) & (lens > 0))[0]
        a_live = np.asarray(accept)[live]
        # an fp16 delta ring keeps the accepted records: flag the ones out of range
        over = pend["over"]
        for r, a in zip(live, a_live):
            if over[r, :int(a)].any():
                self.d_overflow[layer, slots[r]] = True
        for c0 in range(0, live.size, self._chunk):
            rows = live[c0:c0 + self._chunk]
            a = a_live[c0:c0 + rows.size]
            sl = slots[rows]
            S = self.S[layer, sl]                 # fancy indexing: a copy
            full = a == lens[rows]                # whole window accepted: final state
            S[full] = final[c0:c0 + rows.size][full]
            for i in range(int(lens[rows].max())):
                keep = np.nonzero(~full & (a > i))[0]   # rows that accept token i
                if keep.size == 0:
                    break
                idx = starts[rows[keep]] + i
                q, k, v, beta, g = self._token_inputs(inp, idx)
                S[keep], _, _ = token_step(S[keep], q, k, v, beta, g, self.scale,
                                           self.algo)
            self.S[layer, sl] = S

    def decode(self, layer, slots, inp, force=None, advance=False):
        """Width-1 decode of one layer; the token is accepted at once.

        The cursor (shared by all layers) moves only when ``advance`` is set,
        i.e. after the last layer of the step.
        """
        o, flags = self.window(layer, slots, inp, 1, force)
        B = len(slots)
        self._accept(layer, np.ones(B, dtype=np.int64))
        if advance:
            force = np.zeros(B, np.uint8) if force is None else np.asarray(force)
            for r, s in enumerate(np.asarray(slots)):
                if s >= 0:
                    self.cursor[s] = ring.cursor_after_decode(
                        int(self.cursor[s]), self.L, bool(force[r]))
        return o, flags

    def commit(self, slots, accept, T, force=None, mode=ring.LAZY):
        """Commit the pending verify windows of every layer, then the cursor."""
        for layer in sorted(self._pending):
            if self._pending[layer]["T"] != T:
                raise ValueError("commit T differs from the verified window")
        B = len(slots)
        self._commit(slots, accept, np.full(B, T, dtype=np.int64), force, mode)

    def commit_ragged(self, slots, accept, cu_seqlens, force=None, mode=ring.LAZY):
        """Commit pending ragged windows: row r accepts accept[r] of its
        cu_seqlens[r+1] - cu_seqlens[r] tokens; an idle row (no tokens) keeps
        its cursor and checkpoint."""
        lens = np.diff(np.asarray(cu_seqlens, dtype=np.int64))
        for layer in sorted(self._pending):
            if not np.array_equal(self._pending[layer]["lens"], lens):
                raise ValueError("commit windows differ from the verified ones")
        self._commit(slots, accept, lens, force, mode)

    def _commit(self, slots, accept, lens, force, mode):
        slots = np.asarray(slots, dtype=np.int64)
        B = slots.shape[0]
        force = np.zeros(B, np.uint8) if force is None else np.asarray(force)
        accept = np.asarray(accept, dtype=np.int64)
        for layer in sorted(self._pending):
            self._accept(layer, accept)
        for r, s in enumerate(slots):
            if s < 0 or lens[r] == 0:
                continue
            c = int(self.cursor[s])
            if mode == ring.FOLD_EVERY:
                self._checkpoint(slice(None), s)
            self.cursor[s] = ring.cursor_after_commit(c, int(lens[r]), self.L,
                                                      bool(force[r]), int(accept[r]), mode)

    def prefill(self, layer, slots, inp, cu_seqlens):
        """Replay prefill of one layer (LightLLM PR #1690, commit messages:
        prefill writes the canonical state directly and leaves the cursor at
        zero). Row r's prompt is tokens [cu_seqlens[r], cu_seqlens[r+1]) of
        the packed inputs; it runs token by token from the row's committed
        state (checkpoint plus ring history), and the checkpoint then takes
        the result. Rows with a null slot or no tokens are left as they are.
        The cursor moves in ``prefill_done``, after the last layer.

        Returns o [N, HV, dv] (NaN where no row wrote), N = cu_seqlens[-1].
        """
        slots = np.asarray(slots, dtype=np.int64)
        cu = np.asarray(cu_seqlens, dtype=np.int64)
        lens = np.diff(cu)
        if cu.shape[0] != slots.shape[0] + 1 or np.any(lens < 0) or cu[0] < 0:
            raise ValueError("cu_seqlens must be non-negative and non-decreasing")
        o = np.full((int(cu[-1]), self.HV, self.dv), np.nan)
        with np.errstate(all="ignore"):
            for r, s in enumerate(slots):
                if s < 0 or lens[r] == 0:
                    continue
                S = self.S[layer, s][None]
                for t in range(int(cu[r]), int(cu[r + 1])):
                    q, k, v, beta, g = self._token_inputs(inp, np.array([t]))
                    S, _, o[t:t + 1] = token_step(S, q, k, v, beta, g, self.scale, self.algo)
                self.S[layer, s] = S[0]
                self._checkpoint(layer, [s])
                self.written[layer, s] = False
        return o

    def prefill_done(self, slots, cu_seqlens):
        """After the last layer's prefill: cursor <- 0 for every row that had
        prompt tokens (its history now lives in the checkpoint)."""
        lens = np.diff(np.asarray(cu_seqlens, dtype=np.int64))
        for r, s in enumerate(np.asarray(slots)):
            if s >= 0 and lens[r] > 0:
                self.cursor[s] = 0

    def fold(self, slots):
        """Explicit fold: checkpoint <- committed state, cursor <- 0."""
        for s in np.asarray(slots):
            if s >= 0:
                self._checkpoint(slice(None), s)
                self.cursor[s] = 0

    def load_checkpoint(self, slot, S):
        """Install a checkpoint in a slot (restore / state copy)."""
        self.ckpt[:, slot] = S

    def reset_slots(self, slots):
        """Restore semantics: cursor <- 0, so the slot's state is its checkpoint."""
        for s in np.asarray(slots):
            if s >= 0:
                self.cursor[s] = 0
                self.S[:, s] = self.ckpt[:, s]

    def select_slots(self, idx):
        """Keep only slots ``idx`` (renumbered 0 .. len(idx) - 1), between
        steps; lets a test follow every row for a while and then a sample."""
        if self._pending:
            raise ValueError("select_slots between steps only (a window is pending)")
        idx = np.asarray(idx, dtype=np.int64)
        for name in ("S", "ckpt", "ring_k", "ring_d", "ring_g", "ring_v", "ring_beta",
                     "written", "d_overflow"):
            setattr(self, name, getattr(self, name)[:, idx].copy())
        self.cursor = self.cursor[idx].copy()
        self.n_slots = int(idx.size)

    def accepted_positions(self, slot):
        """Ring positions holding committed history: [0, cursor)."""
        return np.arange(int(self.cursor[slot]))
