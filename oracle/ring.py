"""Integer rules of the ReplaySSM ring and cursor (oracle side).

Test infrastructure only: nothing in the product path imports this module.

Sources, all restated in our own words:

* LightLLM PR #1690 "feat: add ReplaySSM state modes for GDN and KDA", commit
  messages: decode appends into one buffer of cursor length and folds the whole
  prefix only when the next window would no longer fit, or when a fold is
  forced; the fold decision is taken on the device; the cursor is advanced once
  per step, after the last layer; a restored slot has its cursor cleared.
* SGLang fork PR jianc99/sglang#2 (GDN ReplaySSM for DFLASH/DSPARK), first
  commit: a verify writes its draft window at ring positions
  [write_pos, write_pos + T); rows whose state slot is null are skipped by the
  cursor advance; a ring shorter than the draft window is refused up front.
  Fourth commit: commit trims the rejected tail and, in fold-every mode, folds
  the accepted window so the checkpoint is the committed state after each step.
* vLLM PR #64699 "[Feature][MRV2] Enable Qwen3.5 GDN ReplaySSM standard
  decode", commit messages: a per-row forced flush may happen mid-ring.

Reading taken where the pages differ: the fold is decided *before* the window
(c + T > L), not after it; a post-window flush at write_pos == L - 1 is
reachable through the per-row force flag.
"""
from __future__ import annotations

LAZY = 0
FOLD_EVERY = 1


def fold_decision(c: int, T: int, L: int, force: bool) -> tuple[bool, int]:
    """Return (fold, base) for a window of T tokens.

    c is the number of history records held in the ring (the cursor) and L its
    capacity. The window folds the whole history into the checkpoint when it is
    forced or when appending T records would overflow the ring; the window's
    records are then written from position 0, else from position c.
    """
    fold = bool(force) or (c + T > L)
    return fold, (0 if fold else c)


def cursor_after_decode(c: int, L: int, force: bool) -> int:
    """Cursor after a width-1 decode step: the token is always accepted."""
    _, base = fold_decision(c, 1, L, force)
    return base + 1


def cursor_after_commit(c: int, T: int, L: int, force: bool, a: int,
                        mode: int) -> int:
    """Cursor after committing a accepted tokens of a T-token verify window.

    Lazy mode keeps the accepted records as history (the rejected tail is
    trimmed); fold-every mode folds them into the checkpoint and empties the ring.
    """
    if not 0 <= a <= T:
        raise ValueError("accepted length outside [0, T]")
    if mode == FOLD_EVERY:
        return 0
    _, base = fold_decision(c, T, L, force)
    return base + a


def records_to_fold_at_commit(c: int, T: int, L: int, force: bool, a: int) -> int:
    """Number of ring records a fold-every commit folds: base + a."""
    _, base = fold_decision(c, T, L, force)
    return base + a
