"""fp64 oracle of the conv-state window and its rollback — TEST INFRASTRUCTURE ONLY.

The CUDA path never imports, links or runs this file.

The ReplaySSM pages manage a second per-request state beside the SSM: the
window of the layer's short causal convolution, which the commit rolls back
to the accepted tokens (LightLLM PR #1690, commit messages: page save, PD and
DP copy the accepted conv window; SGLang fork PR jianc99/sglang#2, fifth
commit: the GDN ring commit covers the cursor advance, the fold and the conv
rollback). The pages do not print the convolution itself; this oracle takes
the plainest reading, a depthwise causal convolution of width K per channel:

    xp = [window (K-1 rows), x_0, ..., x_{T-1}]         (per request row)
    y_t[c] = act(bias[c] + sum_{i<K} w[c][i] * xp[t + i][c])
    act = identity, or SiLU (u * sigmoid(u))

and the window after accepting the first a of the T tokens is the last K-1
rows of [window, x_0, ..., x_{a-1}]. Decode accepts its token at once.

Layouts: window [n_slots, K-1, D]; x, y [B*T, D] (row r's token t at r*T + t);
w [D, K]; bias [D] or None. Null rows (slot -1) are skipped.
"""
from __future__ import annotations

import numpy as np

__all__ = ["ConvOracle", "ACT_NONE", "ACT_SILU"]

ACT_NONE, ACT_SILU = 0, 1


class ConvOracle:
    """Conv windows of every slot, plus the draft tokens of the last window."""

    def __init__(self, window0, w, bias=None, act=ACT_NONE):
        self.window = np.array(window0, dtype=np.float64)   # [n_slots, K-1, D]
        self.w = np.asarray(w, dtype=np.float64)            # [D, K]
        self.K = self.w.shape[1]
        if self.window.shape[1] != self.K - 1:
            raise ValueError("window must hold K - 1 rows")
        self.bias = None if bias is None else np.asarray(bias, dtype=np.float64)
        self.act = act
        self._draft = {}

    def _conv(self, xp, T):
        """y_t for t < T from the padded sequence xp [K-1+T, D]."""
        y = np.zeros((T, xp.shape[1]))
        for t in range(T):
            acc = np.zeros(xp.shape[1]) if self.bias is None else self.bias.copy()
            for i in range(self.K):
                acc = acc + self.w[:, i] * xp[t + i]
            y[t] = acc
        if self.act == ACT_SILU:
            y = y / (1.0 + np.exp(-y))
        return y

    def window_step(self, slots, x, T):
        """Outputs of a T-token window for every live row; the inputs are kept
        as drafts until ``commit`` (``decode`` commits at once)."""
        slots = np.asarray(slots)
        x = np.asarray(x, dtype=np.float64)
        y = np.full(x.shape, np.nan)
        for r, s in enumerate(slots):
            if s < 0:
                continue
            xs = x[r * T:(r + 1) * T]
            xp = np.concatenate([self.window[s], xs], axis=0)
            y[r * T:(r + 1) * T] = self._conv(xp, T)
            self._draft[int(s)] = xs.copy()
        return y

    def commit(self, slots, accept):
        """The window becomes the last K-1 rows of [window, first a drafts]."""
        for r, s in enumerate(np.asarray(slots)):
            if s < 0:
                continue
            a = int(accept[r])
            xs = self._draft.pop(int(s))
            if not 0 <= a <= xs.shape[0]:
                raise ValueError("accept length outside [0, T]")
            seq = np.concatenate([self.window[s], xs[:a]], axis=0)
            self.window[s] = seq[seq.shape[0] - (self.K - 1):]

    def decode(self, slots, x):
        y = self.window_step(slots, x, 1)
        self.commit(slots, np.ones(len(slots), dtype=np.int64))
        return y
