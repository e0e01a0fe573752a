"""ReplayStore: owns the device buffers of one ReplaySSM store (allocated with
PyTorch, which is used here only for device memory and streams) and forwards
calls to the C ABI with the same names. No arithmetic of the method runs here.
"""
from __future__ import annotations

import torch

from . import _lib

_TORCH = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}


class ReplayStore:
    """Checkpoint, ring and cursor of ``n_slots`` requests over ``n_layers`` layers.

    Buffers (row-major):
      state     [n_layers, n_slots, HV, dk, dv]    state_dtype
      ring_k    [n_layers, n_slots, HV, L, dk]     ring_k_dtype (one copy per value head)
      ring_d    [n_layers, n_slots, HV, L, dv]     ring_d_dtype
      ring_g    [n_layers, n_slots, HV, L] (+ [dk] for KDA)  fp32
      ring_v    [n_layers, n_slots, HV, L, dv]     in_dtype
      ring_beta [n_layers, n_slots, HV, L]         fp32
      cursor    [n_slots] int32, err_word [1] (uint32 bits in an int32 tensor)
    """

    def __init__(self, algo="gdn", n_layers=1, n_slots=1, HK=1, HV=1, dk=128, dv=128, L=16,
                 max_T=1, in_dtype="bf16", state_dtype="f32", ring_k_dtype=None,
                 ring_d_dtype="f32", commit_mode="lazy", scale=None, device="cuda"):
        self.cfg = _lib.make_config(algo, n_layers, n_slots, HK, HV, dk, dv, L, max_T, in_dtype,
                                    state_dtype, ring_k_dtype, ring_d_dtype, commit_mode, scale)
        self.algo, self.n_layers, self.n_slots = algo, n_layers, n_slots
        self.HK, self.HV, self.dk, self.dv, self.L, self.max_T = HK, HV, dk, dv, L, max_T
        self.in_dtype, self.state_dtype = in_dtype, state_dtype
        self.ring_k_dtype = ring_k_dtype or ("f16" if in_dtype == "bf16" else "f32")
        self.ring_d_dtype = ring_d_dtype
        self.commit_mode = commit_mode
        self.scale = self.cfg.scale
        self.device = torch.device(device)
        _lib.rssm_required_bytes(self.cfg)  # validates the configuration
        ls = (n_layers, n_slots)
        ng = () if algo == "gdn" else (dk,)
        dev = self.device
        self.state = torch.zeros(ls + (HV, dk, dv), dtype=_TORCH[state_dtype], device=dev)
        self.ring_k = torch.zeros(ls + (HV, L, dk), dtype=_TORCH[self.ring_k_dtype], device=dev)
        self.ring_d = torch.zeros(ls + (HV, L, dv), dtype=_TORCH[ring_d_dtype], device=dev)
        self.ring_g = torch.zeros(ls + (HV, L) + ng, dtype=torch.float32, device=dev)
        self.ring_v = torch.zeros(ls + (HV, L, dv), dtype=_TORCH[in_dtype], device=dev)
        self.ring_beta = torch.zeros(ls + (HV, L), dtype=torch.float32, device=dev)
        self.cursor = torch.zeros(n_slots, dtype=torch.int32, device=dev)
        self.err_word = torch.zeros(1, dtype=torch.int32, device=dev)
        bufs = _lib.rssm_buffers(*(t.data_ptr() for t in (
            self.state, self.ring_k, self.ring_d, self.ring_g, self.ring_v, self.ring_beta,
            self.cursor, self.err_word)))
        with torch.cuda.device(dev):
            self.handle = _lib.rssm_alloc(self.cfg, bufs)

    # ---------------------------------------------------------------- calls
    def rssm_decode(self, layer, q, k, v, beta, g, slot, o, force=None, fold_out=None,
                    advance_cursor=False, stream=None):
        _lib.rssm_decode(self.handle, layer, q, k, v, beta, g, slot, force, slot.numel(), o,
                         fold_out, advance_cursor, stream)

    def rssm_verify(self, layer, q, k, v, beta, g, slot, T, o, force=None, fold_out=None,
                    stream=None):
        _lib.rssm_verify(self.handle, layer, q, k, v, beta, g, slot, force, slot.numel(), T, o,
                         fold_out, stream)

    def rssm_verify_ragged(self, layer, q, k, v, beta, g, cu_seqlens, slot, max_T, o,
                           force=None, fold_out=None, stream=None):
        """Windows of different lengths: row r's tokens are
        [cu_seqlens[r], cu_seqlens[r+1]) of the packed inputs (int32, B + 1)."""
        _lib.rssm_verify_ragged(self.handle, layer, q, k, v, beta, g, cu_seqlens, slot, force,
                                slot.numel(), max_T, o, fold_out, stream)

    def rssm_prefill(self, layer, q, k, v, beta, g, cu_seqlens, slot, o, reset_cursor=False,
                     stream=None):
        """Prompt of row r = tokens [cu_seqlens[r], cu_seqlens[r+1]); the
        checkpoint takes the state; the cursor clears on the last layer."""
        _lib.rssm_prefill(self.handle, layer, q, k, v, beta, g, cu_seqlens, slot, slot.numel(),
                          o, reset_cursor, stream)

    def rssm_native_decode(self, layer, q, k, v, beta, g, slot, o, stream=None):
        """The per-token state read/write path ReplaySSM replaces (comparison
        point): the checkpoint is the live state; ring and cursor untouched."""
        _lib.rssm_native_decode(self.handle, layer, q, k, v, beta, g, slot, slot.numel(), o,
                                stream)

    def rssm_commit(self, slot, accept_len, T, force=None, stream=None):
        _lib.rssm_commit(self.handle, slot, force, accept_len, slot.numel(), T, stream)

    def rssm_commit_ragged(self, slot, accept_len, cu_seqlens, max_T, force=None, stream=None):
        _lib.rssm_commit_ragged(self.handle, slot, force, accept_len, cu_seqlens, slot.numel(),
                                max_T, stream)

    def rssm_fold(self, slot, stream=None):
        _lib.rssm_fold(self.handle, slot, slot.numel(), stream)

    def rssm_reset_slots(self, slot, stream=None):
        _lib.rssm_reset_slots(self.handle, slot, slot.numel(), stream)

    def rssm_get_device_error(self, clear=True, stream=None) -> int:
        return _lib.rssm_get_device_error(self.handle, clear, stream)

    def rssm_set_plan(self, plan):
        """Kernel family for decode and verify: "auto", "rows" or "pipe"."""
        _lib.rssm_set_plan(self.handle, plan)

    def rssm_debug_withhold(self, barrier):
        """Test hook of the bounded waits (include/rssm.h): later launches of
        this store short-change `barrier` (-1: off)."""
        _lib.rssm_debug_withhold(self.handle, barrier)

    def close(self):
        if getattr(self, "handle", None):
            _lib.rssm_free(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # ------------------------------------------------------------- helpers
    def new_output(self, B, T=1):
        return torch.empty((B * T, self.HV, self.dv), dtype=_TORCH[self.in_dtype],
                           device=self.device)

    def state_bytes_per_row_layer(self) -> int:
        return self.HV * self.dk * self.dv * (4 if self.state_dtype == "f32" else 2)


class ConvWindows:
    """Conv-state windows of ``n_slots`` requests for one convolution of width K
    over D channels, and the draft inputs of the last verify window.

    Buffers: window [n_slots, K-1, D], draft [n_slots, max_T, D] (dtype),
    err_word [1]. Taps w [D, K] and bias [D] are fp32 and passed per call.
    """

    ACT = {"none": 0, "silu": 1}

    def __init__(self, n_slots, D, K, max_T=1, dtype="bf16", device="cuda"):
        self.n_slots, self.D, self.K, self.max_T, self.dtype = n_slots, D, K, max_T, dtype
        dev = torch.device(device)
        self.window = torch.zeros((n_slots, K - 1, D), dtype=_TORCH[dtype], device=dev)
        self.draft = torch.zeros((n_slots, max_T, D), dtype=_TORCH[dtype], device=dev)
        self.err_word = torch.zeros(1, dtype=torch.int32, device=dev)

    def rssm_conv_window(self, x, w, bias, slot, T, y, act="silu", commit_now=False,
                         stream=None):
        if T > self.max_T:
            raise ValueError("window wider than the draft buffer")
        _lib.rssm_conv_window(x, w, bias, self.window, self.draft, slot, slot.numel(), T, self.D,
                              self.K, self.n_slots, self.dtype, self.ACT[act], commit_now, y,
                              self.err_word, stream)

    def rssm_conv_commit(self, slot, accept_len, T, stream=None):
        _lib.rssm_conv_commit(self.window, self.draft, slot, accept_len, slot.numel(), T, self.D,
                              self.K, self.n_slots, self.dtype, self.err_word, stream)
