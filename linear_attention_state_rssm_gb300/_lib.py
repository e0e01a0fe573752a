"""ctypes binding of librssm (include/rssm.h): same names, argument marshalling only.

Every function here converts arguments (torch tensors -> device pointers, the
current CUDA stream -> cudaStream_t) and calls the C ABI; all computation runs
in the library's CUDA kernels. If librssm.so is missing the import of the
binding fails loudly: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "librssm.so")

RSSM_OK = 0
STATUS_NAMES = {0: "RSSM_OK", 1: "RSSM_ERR_INVALID_ARG", 2: "RSSM_ERR_UNSUPPORTED",
                3: "RSSM_ERR_CUDA", 4: "RSSM_ERR_DEVICE"}
ALGO = {"gdn": 0, "kda": 1}
DTYPE = {"f32": 0, "bf16": 1, "f16": 2}
COMMIT = {"lazy": 0, "fold_every": 1}
DEVERR = {"slot": 1, "cursor": 2, "accept": 4, "timeout": 8, "seqlen": 16}

# Every entry point declared in include/rssm.h.
SYMBOLS = ("rssm_required_bytes", "rssm_alloc", "rssm_free", "rssm_decode", "rssm_verify",
           "rssm_verify_ragged", "rssm_prefill", "rssm_native_decode", "rssm_commit",
           "rssm_commit_ragged", "rssm_fold", "rssm_reset_slots", "rssm_conv_window",
           "rssm_conv_commit",
           "rssm_get_device_error", "rssm_set_plan", "rssm_debug_withhold",
           "rssm_status_string", "rssm_version")


class RssmError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}")


class rssm_config(ctypes.Structure):
    _fields_ = [("algo", ctypes.c_int32), ("n_layers", ctypes.c_int32),
                ("n_slots", ctypes.c_int32), ("HK", ctypes.c_int32), ("HV", ctypes.c_int32),
                ("dk", ctypes.c_int32), ("dv", ctypes.c_int32), ("L", ctypes.c_int32),
                ("max_T", ctypes.c_int32), ("in_dtype", ctypes.c_int32),
                ("state_dtype", ctypes.c_int32), ("ring_k_dtype", ctypes.c_int32),
                ("ring_d_dtype", ctypes.c_int32), ("commit_mode", ctypes.c_int32),
                ("scale", ctypes.c_float)]


class rssm_buffers(ctypes.Structure):
    _fields_ = [(name, ctypes.c_void_p) for name in
                ("state", "ring_k", "ring_d", "ring_g", "ring_v", "ring_beta", "cursor",
                 "err_word")]


class rssm_sizes(ctypes.Structure):
    _fields_ = [(name, ctypes.c_size_t) for name in
                ("state", "ring_k", "ring_d", "ring_g", "ring_v", "ring_beta", "cursor",
                 "err_word")]


_P = ctypes.c_void_p
_I = ctypes.c_int32
_lib = None


def load() -> ctypes.CDLL:
    """Load librssm.so (built in-tree by the package's build module)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            f"librssm.so not found at {LIB_PATH}: build it with "
            "linear_attention_state_rssm_gb300.build.build() (nvcc, sm_103a)")
    lib = ctypes.CDLL(LIB_PATH)
    sig = {
        "rssm_required_bytes": ([ctypes.POINTER(rssm_config), ctypes.POINTER(rssm_sizes)], _I),
        "rssm_alloc": ([ctypes.POINTER(rssm_config), ctypes.POINTER(rssm_buffers),
                        ctypes.POINTER(_P)], _I),
        "rssm_free": ([_P], None),
        "rssm_decode": ([_P, _I, _P, _P, _P, _P, _P, _P, _P, _I, _P, _P, _I, _P], _I),
        "rssm_verify": ([_P, _I, _P, _P, _P, _P, _P, _P, _P, _I, _I, _P, _P, _P], _I),
        "rssm_verify_ragged": ([_P, _I, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _P, _P, _P],
                               _I),
        "rssm_prefill": ([_P, _I, _P, _P, _P, _P, _P, _P, _P, _I, _P, _I, _P], _I),
        "rssm_native_decode": ([_P, _I, _P, _P, _P, _P, _P, _P, _I, _P, _P], _I),
        "rssm_commit": ([_P, _P, _P, _P, _I, _I, _P], _I),
        "rssm_commit_ragged": ([_P, _P, _P, _P, _P, _I, _I, _P], _I),
        "rssm_fold": ([_P, _P, _I, _P], _I),
        "rssm_conv_window": ([_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _P, _P,
                              _P], _I),
        "rssm_conv_commit": ([_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P], _I),
        "rssm_reset_slots": ([_P, _P, _I, _P], _I),
        "rssm_get_device_error": ([_P, ctypes.POINTER(ctypes.c_uint32), _I, _P], _I),
        "rssm_set_plan": ([_P, _I], _I),
        "rssm_debug_withhold": ([_P, _I], _I),
        "rssm_status_string": ([_I], ctypes.c_char_p),
        "rssm_version": ([], _I),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _lib = lib
    return lib


def _ptr(x):
    """Device pointer of a tensor (None -> NULL)."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int, where: str):
    if status != RSSM_OK:
        raise RssmError(status, where)


def make_config(algo="gdn", n_layers=1, n_slots=1, HK=1, HV=1, dk=128, dv=128, L=16, max_T=1,
                in_dtype="bf16", state_dtype="f32", ring_k_dtype=None, ring_d_dtype="f32",
                commit_mode="lazy", scale=None) -> rssm_config:
    """Build an rssm_config; ring keys default to fp16 for bf16 inputs, else fp32."""
    if ring_k_dtype is None:
        ring_k_dtype = "f16" if in_dtype == "bf16" else "f32"
    return rssm_config(ALGO[algo], n_layers, n_slots, HK, HV, dk, dv, L, max_T,
                       DTYPE[in_dtype], DTYPE[state_dtype], DTYPE[ring_k_dtype],
                       DTYPE[ring_d_dtype], COMMIT[commit_mode],
                       float(dk ** -0.5 if scale is None else scale))


# ------------------------------------------------------------ C ABI wrappers
def rssm_required_bytes(cfg: rssm_config) -> rssm_sizes:
    out = rssm_sizes()
    _check(load().rssm_required_bytes(ctypes.byref(cfg), ctypes.byref(out)), "rssm_required_bytes")
    return out


def rssm_alloc(cfg: rssm_config, bufs: rssm_buffers) -> int:
    h = _P()
    _check(load().rssm_alloc(ctypes.byref(cfg), ctypes.byref(bufs), ctypes.byref(h)), "rssm_alloc")
    return h.value


def rssm_free(handle: int) -> None:
    load().rssm_free(handle)


def rssm_decode(handle, layer, q, k, v, beta, g, slot, force, B, o, fold_out, advance_cursor,
                stream=None):
    _check(load().rssm_decode(handle, layer, _ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(g),
                              _ptr(slot), _ptr(force), B, _ptr(o), _ptr(fold_out),
                              int(bool(advance_cursor)), _stream(stream)), "rssm_decode")


def rssm_verify(handle, layer, q, k, v, beta, g, slot, force, B, T, o, fold_out, stream=None):
    _check(load().rssm_verify(handle, layer, _ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(g),
                              _ptr(slot), _ptr(force), B, T, _ptr(o), _ptr(fold_out),
                              _stream(stream)), "rssm_verify")


def rssm_verify_ragged(handle, layer, q, k, v, beta, g, cu_seqlens, slot, force, B, max_T, o,
                       fold_out, stream=None):
    _check(load().rssm_verify_ragged(handle, layer, _ptr(q), _ptr(k), _ptr(v), _ptr(beta),
                                     _ptr(g), _ptr(cu_seqlens), _ptr(slot), _ptr(force), B,
                                     max_T, _ptr(o), _ptr(fold_out), _stream(stream)),
           "rssm_verify_ragged")


def rssm_prefill(handle, layer, q, k, v, beta, g, cu_seqlens, slot, B, o, reset_cursor,
                 stream=None):
    _check(load().rssm_prefill(handle, layer, _ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(g),
                               _ptr(cu_seqlens), _ptr(slot), B, _ptr(o),
                               int(bool(reset_cursor)), _stream(stream)), "rssm_prefill")


def rssm_native_decode(handle, layer, q, k, v, beta, g, slot, B, o, stream=None):
    _check(load().rssm_native_decode(handle, layer, _ptr(q), _ptr(k), _ptr(v), _ptr(beta),
                                     _ptr(g), _ptr(slot), B, _ptr(o), _stream(stream)),
           "rssm_native_decode")


def rssm_commit(handle, slot, force, accept_len, B, T, stream=None):
    _check(load().rssm_commit(handle, _ptr(slot), _ptr(force), _ptr(accept_len), B, T,
                              _stream(stream)), "rssm_commit")


def rssm_commit_ragged(handle, slot, force, accept_len, cu_seqlens, B, max_T, stream=None):
    _check(load().rssm_commit_ragged(handle, _ptr(slot), _ptr(force), _ptr(accept_len),
                                     _ptr(cu_seqlens), B, max_T, _stream(stream)),
           "rssm_commit_ragged")


def rssm_conv_window(x, w, bias, window, draft, slot, B, T, D, K, n_slots, dtype, act,
                     commit_now, y, err_word=None, stream=None):
    _check(load().rssm_conv_window(_ptr(x), _ptr(w), _ptr(bias), _ptr(window), _ptr(draft),
                                   _ptr(slot), B, T, D, K, n_slots, DTYPE[dtype], act,
                                   int(bool(commit_now)), _ptr(y), _ptr(err_word),
                                   _stream(stream)), "rssm_conv_window")


def rssm_conv_commit(window, draft, slot, accept_len, B, T, D, K, n_slots, dtype, err_word=None,
                     stream=None):
    _check(load().rssm_conv_commit(_ptr(window), _ptr(draft), _ptr(slot), _ptr(accept_len), B, T,
                                   D, K, n_slots, DTYPE[dtype], _ptr(err_word), _stream(stream)),
           "rssm_conv_commit")


def rssm_fold(handle, slot, B, stream=None):
    _check(load().rssm_fold(handle, _ptr(slot), B, _stream(stream)), "rssm_fold")


def rssm_reset_slots(handle, slot, B, stream=None):
    _check(load().rssm_reset_slots(handle, _ptr(slot), B, _stream(stream)), "rssm_reset_slots")


def rssm_get_device_error(handle, clear=True, stream=None) -> int:
    word = ctypes.c_uint32(0)
    st = load().rssm_get_device_error(handle, ctypes.byref(word), int(bool(clear)),
                                      _stream(stream))
    if st not in (RSSM_OK, 4):
        raise RssmError(st, "rssm_get_device_error")
    return int(word.value)


PLAN = {"auto": 0, "rows": 1, "pipe": 2, "tc": 3}


def rssm_set_plan(handle, plan):
    """Kernel family for decode and verify: "auto", "rows", "pipe" or "tc"."""
    _check(load().rssm_set_plan(handle, PLAN[plan] if isinstance(plan, str) else int(plan)),
           "rssm_set_plan")


# barriers of the bounded-wait test hook (rssm_debug_withhold)
WITHHOLD = {"off": -1, "window": 0, "history": 1}


def withhold_chunk(j: int) -> int:
    """Barrier index of checkpoint chunk j for rssm_debug_withhold."""
    return 2 + int(j)


def rssm_debug_withhold(handle, barrier):
    """Test hook: every later replay/fold launch of this handle short-changes
    `barrier` (see include/rssm.h); barrier -1 turns it off."""
    _check(load().rssm_debug_withhold(handle, int(barrier)), "rssm_debug_withhold")


def rssm_status_string(status: int) -> str:
    return load().rssm_status_string(status).decode()


def rssm_version() -> int:
    return int(load().rssm_version())
