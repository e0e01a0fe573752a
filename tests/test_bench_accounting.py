"""The byte accounting behind the bench's roofline (CPU only).

The algorithmic bytes of one live row in one replay launch are the method's:
the checkpoint tile once, c history records, the window's inputs, the outputs,
the T new records and, on a fold, the checkpoint written back. Checked against
the per-term sizes written out for the Qwen3.5-4B-shaped decode layer
(HK 16, HV 32, dk = dv = 128, fp32 state, bf16 inputs, fp16 keys, fp32 deltas).
"""
import pytest

import bench


def _terms(c, T, fold):
    state = 32 * 128 * 128 * 4                       # 2,097,152
    record = 16 * 128 * 2 + 32 * 128 * 4 + 32 * 4    # key per key head, delta, gate: 20,608
    window = T * (2 * 16 * 128 * 2 + 32 * 128 * 2 + 32 * 2 * 4)   # q, k, v, beta, g: 16,640
    out = T * 32 * 128 * 2                           # 8,192
    written = T * (record + 32 * 128 * 2 + 32 * 4)   # record + v + beta: 28,928
    return state + c * record + window + out + written + (state if fold else 0)


@pytest.mark.parametrize("c,T,fold", [(0, 1, False), (8, 1, False), (15, 1, False),
                                      (16, 1, True), (5, 8, False), (12, 8, True)])
def test_row_bytes_match_the_per_term_sizes(c, T, fold):
    assert bench.row_bytes(c, T, fold, 16, 32, 128, 128, 4, 2, 2, 4) == _terms(c, T, fold)


def test_decode_row_bytes_worked_example():
    # 2,097,152 + 20,608 c + 16,640 + 8,192 + 28,928 (+ 2,097,152 on a fold)
    assert bench.row_bytes(0, 1, False, 16, 32, 128, 128, 4, 2, 2, 4) == 2150912
    assert bench.row_bytes(8, 1, False, 16, 32, 128, 128, 4, 2, 2, 4) == 2150912 + 8 * 20608
    assert bench.row_bytes(16, 1, True, 16, 32, 128, 128, 4, 2, 2, 4) == \
        2150912 + 16 * 20608 + 2097152


@pytest.mark.parametrize("c,T,L,a,want", [(0, 1, 16, 1, (1, False)), (15, 1, 16, 1, (16, False)),
                                          (16, 1, 16, 1, (1, True)), (8, 8, 16, 3, (11, False)),
                                          (8, 8, 16, 0, (8, False)), (9, 8, 16, 5, (5, True))])
def test_cursor_trajectory_rule(c, T, L, a, want):
    """The bench's host copy of the cursor rule: fold when c + T > L, then the
    accepted tokens go after base = fold ? 0 : c."""
    assert bench.advance(c, T, L, a) == want


def test_job_throughput_is_whole_job():
    assert bench.job_throughput(1000.0, 4, 2.0) == 2000.0


def test_commit_bytes_fold_every():
    """A fold-every commit reads and writes the checkpoint once and reads the
    n committed records: 2 * 2,097,152 + n * 20,608 for the decode shapes."""
    assert bench.commit_bytes(0, 16, 32, 128, 128, 4, 2, 4) == 2 * 2097152
    assert bench.commit_bytes(5, 16, 32, 128, 128, 4, 2, 4) == 2 * 2097152 + 5 * 20608
    # KDA: a gate per key channel, bf16 checkpoint, fp16 keys and deltas
    assert bench.commit_bytes(3, 32, 32, 128, 128, 2, 2, 2, 128) == \
        2 * 32 * 128 * 128 * 2 + 3 * (32 * 128 * 2 + 32 * 128 * 2 + 32 * 128 * 4)


@pytest.mark.parametrize("T,nt", [(1, 1), (2, 2), (3, 4), (4, 4), (5, 8), (8, 8), (9, 16)])
def test_window_width_of_the_kernel(T, nt):
    """The verify line names the kernel by its window width: the smallest
    power of two at least T (the library's own choice of instantiation)."""
    assert bench.nt_for(T) == nt


def test_commit_summary_carries_a_roofline_only_for_a_folding_commit():
    v = {"state_dtype": "bf16"}
    lazy = bench.commit_summary(0.001, 10, [0.0, 0.0], False, 6000.0, v, 48)
    assert "roofline" not in lazy and lazy["launch_ms"] == pytest.approx(0.1)
    # 3 MB per step in 60 us per step: 50 GB/s
    fe = bench.commit_summary(0.0006, 10, [3e6, 3e6], True, 6000.0, v, 48)
    assert fe["roofline"]["achieved"] == pytest.approx(50.0)
    assert fe["roofline"]["frac"] == pytest.approx(50.0 / 6000.0)
    assert fe["per_layer_us"] == pytest.approx(60.0 / 48)


def test_full_grid_covers_every_throughput_configuration():
    """--sweep --grid full: GDN and KDA, batch {1, 8, 64, 128, 256}, ring length
    {16, 32, 64}, window {1, 3, 8}, fp32 and bf16 checkpoints, each once."""
    grid = bench.GRID
    assert len(grid) == len(set(grid)) == 2 * 5 * 3 * 3 * 2
    assert {g[0] for g in grid} == {"gdn", "kda"}
    assert {g[1] for g in grid} == {1, 8, 64, 128, 256}
    assert {g[2] for g in grid} == {16, 32, 64}
    assert {g[3] for g in grid} == {1, 3, 8}
    assert {g[4] for g in grid} == {"f32", "bf16"}
    assert all(g[5] == "lazy" and g[3] <= g[2] for g in grid)


def test_grid_summary_rows(monkeypatch):
    """The bench line's grid object: one compact row per grid point, in GRID
    order, device error words OR-ed (sweep_point stubbed: no GPU here)."""
    def fake_point(torch, dev, algo, B, L, T, state, mode, steps, warmup, peak, plan="auto"):
        assert (mode, steps, warmup) == ("lazy", 5, 3)
        return {"algo": algo, "batch": B, "L": L, "T": T, "state_dtype": state,
                "ms_per_layer": 0.001 * L, "frac_of_hbm_peak": 0.5,
                "device_error_word": 8 if (algo, B, L, T) == ("kda", 8, 32, 3) else 0}
    monkeypatch.setattr(bench, "sweep_point", fake_point)
    g = bench.grid_summary()
    assert g["columns"] == ["algo", "batch", "L", "T", "state_dtype", "us_per_layer",
                            "frac_of_hbm_peak"]
    assert [tuple(r[:5]) for r in g["rows"]] == [pt[:5] for pt in bench.GRID]
    assert all(r[5] == r[2] for r in g["rows"])  # 0.001 ms per record -> L us
    assert g["device_error_word"] == 8 and g["commit_mode"] == "lazy"
