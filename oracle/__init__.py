"""fp64 CPU oracle for the ReplaySSM hot path — TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The CUDA path shares no code with it and
never calls it; there is no CPU fallback anywhere in the product.

* ``oracle.recurrence``: the sequential fp64 gated delta rule (GDN and KDA)
  carrying the exact committed state, the checkpoint the GPU must hold and the
  ring records it must write.
* ``oracle.ring``: the integer ring/cursor/fold rules.
* ``oracle.conv``: the short causal convolution's window and its rollback.

Pins (tests that check the oracle against something other than itself) live
in ``tests/test_oracle_pins.py``, ``tests/test_ring_rules.py`` and the other
``tests/test_oracle_*.py`` files.
"""
from .recurrence import ReplayOracle, round_bf16, token_step  # noqa: F401
from . import conv, ring  # noqa: F401
