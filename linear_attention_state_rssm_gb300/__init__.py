"""GB300-native ReplaySSM hot path for gated delta-rule linear attention (GDN, KDA).

The compute lives in librssm.so (hand-written CUDA for sm_103a behind the C ABI
of include/rssm.h). This package is the thin Python side: ``_lib`` binds the C
ABI by name, ``store.ReplayStore`` allocates the device buffers with PyTorch and
forwards calls, ``build`` compiles the library in-tree.
"""
from . import _lib  # noqa: F401
from ._lib import (RssmError, rssm_alloc, rssm_commit, rssm_decode, rssm_fold,  # noqa: F401
                   rssm_free, rssm_get_device_error, rssm_required_bytes, rssm_reset_slots,
                   rssm_status_string, rssm_verify, rssm_version)


def ReplayStore(*args, **kwargs):
    """Allocate a store (see store.ReplayStore); imports torch lazily."""
    from .store import ReplayStore as _RS
    return _RS(*args, **kwargs)
