"""Pins of the oracle's integer ring/cursor rules against hand-derived tables."""
import os

import numpy as np
import pytest

from oracle import ring, ReplayOracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                yield line


def test_fold_and_cursor_table_L4():
    n = 0
    for line in _rows("ring_rules_L4.txt"):
        head, dec, cur = (part.split() for part in line.split("|"))
        c, T, force = map(int, head)
        fold, base = map(int, dec)
        assert ring.fold_decision(c, T, 4, bool(force)) == (bool(fold), base), line
        lazy = [ring.cursor_after_commit(c, T, 4, bool(force), a, ring.LAZY)
                for a in range(T + 1)]
        assert lazy == list(map(int, cur)), line
        for a in range(T + 1):
            assert ring.cursor_after_commit(c, T, 4, bool(force), a, ring.FOLD_EVERY) == 0
            assert ring.records_to_fold_at_commit(c, T, 4, bool(force), a) == base + a
        n += 1
    assert n == 27


def test_decode_cursor_sequence_tiny_gdn():
    """Decode steps of the tiny GDN workload: cursor, fold and cursor-after."""
    c = 0
    folds = 0
    for line in _rows("decode_cursor_tiny_gdn.txt"):
        step, before, fold, after = map(int, line.split())
        assert c == before, step
        f, _ = ring.fold_decision(c, 1, 16, False)
        assert int(f) == fold, step
        c = ring.cursor_after_decode(c, 16, False)
        assert c == after, step
        folds += f
    assert folds == 2


def test_enumerate_small_rings_properties():
    """Every (c, T, L, a, force) with L <= 8: the window always fits, cursors
    stay in [0, L], a fold starts at 0, and a non-folding window starts at c."""
    for L in range(1, 9):
        for c in range(0, L + 1):
            for T in range(1, L + 1):
                for force in (False, True):
                    fold, base = ring.fold_decision(c, T, L, force)
                    assert base + T <= L
                    assert fold == (force or c + T > L)
                    assert base == (0 if fold else c)
                    for a in range(T + 1):
                        cur = ring.cursor_after_commit(c, T, L, force, a, ring.LAZY)
                        assert 0 <= cur <= L
                        assert cur == base + a
                    with pytest.raises(ValueError):
                        ring.cursor_after_commit(c, T, L, force, T + 1, ring.LAZY)


def test_oracle_cursor_follows_golden_and_skips_null_slots():
    """The oracle's store, run on the tiny decode workload with one null row,
    reproduces the golden cursor sequence and never moves the null slot."""
    B, HK, HV, dk, dv, L = 3, 2, 4, 4, 4, 16
    S0 = synth.initial_state(7, 4, HV, dk, dv)
    orc = ReplayOracle("gdn", 1, 4, HK, HV, dk, dv, L, dk ** -0.5, S0)
    slots = np.array([2, -1, 0])
    rows = list(_rows("decode_cursor_tiny_gdn.txt"))
    for line in rows:
        step, before, fold, after = map(int, line.split())
        inp = synth.window_inputs(step, B, 1, HK, HV, dk, dv)
        _, flags = orc.decode(0, slots, inp, advance=True)
        assert list(flags) == [fold, -1, fold]
        assert orc.cursor[2] == after and orc.cursor[0] == after
        assert orc.cursor[1] == 0 and orc.cursor[3] == 0
