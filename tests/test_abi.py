"""The C ABI library builds, loads and exports every symbol include/rssm.h
declares; host-only entry points work without a GPU."""
import ctypes
import os
import re

import pytest

from linear_attention_state_rssm_gb300 import _lib, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.load()


def _declared():
    with open(os.path.join(ROOT, "include", "rssm.h")) as f:
        text = f.read()
    return sorted(set(re.findall(r"\b(rssm_[a-z_]+)\s*\(", text)))


def test_header_declarations_match_binding():
    assert _declared() == sorted(_lib.SYMBOLS)


def test_every_declared_symbol_is_exported(lib):
    for name in _declared():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_version_and_status_strings(lib):
    assert _lib.rssm_version() == 1
    assert _lib.rssm_status_string(0) == "ok"
    assert _lib.rssm_status_string(2) == "unsupported configuration"


def test_required_bytes_matches_layouts(lib):
    cfg = _lib.make_config("gdn", n_layers=3, n_slots=5, HK=16, HV=32, dk=128, dv=128, L=16,
                           max_T=8, in_dtype="bf16", state_dtype="f32")
    s = _lib.rssm_required_bytes(cfg)
    assert s.state == 3 * 5 * 32 * 128 * 128 * 4
    assert s.ring_k == 3 * 5 * 32 * 16 * 128 * 2          # fp16 keys, one copy per value head
    assert s.ring_d == 3 * 5 * 32 * 16 * 128 * 4
    assert s.ring_g == 3 * 5 * 32 * 16 * 4
    assert s.ring_v == 3 * 5 * 32 * 16 * 128 * 2
    assert s.ring_beta == 3 * 5 * 32 * 16 * 4
    assert s.cursor == 5 * 4 and s.err_word == 4
    kda = _lib.make_config("kda", n_layers=1, n_slots=2, HK=4, HV=4, dk=64, dv=32, L=8,
                           max_T=3, in_dtype="f32", state_dtype="bf16", ring_d_dtype="f16")
    s = _lib.rssm_required_bytes(kda)
    assert s.state == 2 * 4 * 64 * 32 * 2 and s.ring_g == 2 * 4 * 8 * 64 * 4
    assert s.ring_d == 2 * 4 * 8 * 32 * 2


@pytest.mark.parametrize("kw,status", [
    (dict(max_T=17, L=32), 2),           # window wider than built
    (dict(max_T=8, L=4), 1),             # ring shorter than the window
    (dict(dk=96), 2),                    # head size not built
    (dict(HK=3, HV=8), 1),               # HV not a multiple of HK
    (dict(ring_d_dtype="bf16"), 2),      # bf16 deltas not built
    (dict(n_slots=0), 1),
    (dict(L=300, max_T=1), 2),
    (dict(L=65, max_T=1), 2),            # a fold carries at most 64 records
])
def test_host_validation(lib, kw, status):
    base = dict(algo="gdn", n_layers=1, n_slots=2, HK=2, HV=4, dk=64, dv=64, L=8, max_T=2,
                in_dtype="f32", state_dtype="f32")
    base.update(kw)
    cfg = _lib.make_config(**base)
    with pytest.raises(_lib.RssmError) as e:
        _lib.rssm_required_bytes(cfg)
    assert e.value.status == status


def test_longest_ring_is_accepted(lib):
    cfg = _lib.make_config("gdn", 1, 2, 2, 4, 128, 128, 64, 16, "bf16", "f32")
    assert _lib.rssm_required_bytes(cfg).state == 2 * 4 * 128 * 128 * 4


def test_alloc_refuses_bad_buffers_before_touching_the_device(lib):
    cfg = _lib.make_config("gdn", 1, 2, 2, 4, 64, 64, 8, 2, "f32", "f32")
    bufs = _lib.rssm_buffers(0x1000, 0x2000, 0x3000, 0x4000, 0x5000, 0x6000, 0, 0x8000)
    with pytest.raises(_lib.RssmError) as e:              # null cursor
        _lib.rssm_alloc(cfg, bufs)
    assert e.value.status == 1
    bufs = _lib.rssm_buffers(0x1004, 0x2000, 0x3000, 0x4000, 0x5000, 0x6000, 0x7000, 0x8000)
    with pytest.raises(_lib.RssmError) as e:              # misaligned state
        _lib.rssm_alloc(cfg, bufs)
    assert e.value.status == 1


def test_null_handle_is_refused(lib):
    with pytest.raises(_lib.RssmError):
        _lib.rssm_commit(None, None, None, None, 1, 1, stream=0)
    with pytest.raises(_lib.RssmError):
        _lib.rssm_fold(None, None, 1, stream=0)


# Stand-in addresses, 16-byte aligned unless a case offsets one: every case
# below is refused (or is an empty batch) before any CUDA call, so nothing is
# dereferenced and no device is needed. They run only where no GPU is visible,
# so a stand-in address can never reach a kernel.
def _cuda_visible():
    import torch
    return torch.cuda.is_available()


_NO_GPU = pytest.mark.skipif(_cuda_visible(), reason="stand-in addresses: CPU-only hosts")
_A = 0x100000
_CONV = dict(x=_A, w=_A + 0x1000, bias=_A + 0x2000, window=_A + 0x3000, draft=_A + 0x4000,
             slot=_A + 0x5000, B=2, T=4, D=64, K=4, n_slots=3, dtype=1, act=1, commit_now=0,
             y=_A + 0x6000)


@pytest.mark.parametrize("kw,status", [
    (dict(K=1), 2), (dict(K=9), 2),      # convolution width outside 2..8
    (dict(dtype=2), 2),                  # fp16 channels not built
    (dict(D=4), 2),                      # bf16 rows of 8 bytes: not whole 16-byte vectors
    (dict(D=0), 1), (dict(T=0), 1), (dict(n_slots=0), 1), (dict(B=-1), 1),
    (dict(window=_A + 8), 1),            # window not 16-byte aligned
    (dict(x=_A + 4), 1),                 # inputs not 16-byte aligned
    (dict(slot=_A + 2), 1),              # slots not 4-byte aligned
    (dict(act=7), 1),                    # unknown activation
    (dict(y=None), 1),                   # no output buffer
    (dict(draft=None), 1),               # a verify window without a draft buffer
    (dict(y=_A + 8), 1),                 # outputs not 16-byte aligned
    (dict(B=0), 0),                      # an empty batch is a no-op
])
@_NO_GPU
def test_conv_window_host_refusals(lib, kw, status):
    a = {**_CONV, **kw}
    st = lib.rssm_conv_window(a["x"], a["w"], a["bias"], a["window"], a["draft"], a["slot"],
                              a["B"], a["T"], a["D"], a["K"], a["n_slots"], a["dtype"], a["act"],
                              a["commit_now"], a["y"], None, None)
    assert st == status


@pytest.mark.parametrize("kw,status", [
    (dict(accept=None), 1),              # no accepted lengths
    (dict(accept=_A + 0x7002), 1),       # accepted lengths not 4-byte aligned
    (dict(draft=None), 1),               # nothing to roll the window onto
    (dict(K=9), 2), (dict(dtype=2), 2),
    (dict(window=_A + 4), 1),
    (dict(B=0), 0),                      # an empty batch is a no-op
])
@_NO_GPU
def test_conv_commit_host_refusals(lib, kw, status):
    a = {**_CONV, "accept": _A + 0x7000, **kw}
    st = lib.rssm_conv_commit(a["window"], a["draft"], a["slot"], a["accept"], a["B"], a["T"],
                              a["D"], a["K"], a["n_slots"], a["dtype"], None, None)
    assert st == status
