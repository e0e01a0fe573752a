"""The replay kernel's shared-memory plan (host logic, CPU only).

`layout_probe.cu` is compiled as a host program against the kernels' own
header and prints the plan for each configuration. Checked: every region is
16-byte aligned and the plan fits the 227 KB a CTA may use; regions follow in
their order; the long-ring decode plan with 16-bit keys has no fp32 key
region and room for the keys transposed in place; and the CTAs per SM that
the kernels' launch bounds and the measurements rely on.
"""
import json
import os
import shutil
import subprocess
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "linear_attention_state_rssm_gb300", "csrc")
GDN, KDA = 0, 1
F32, BF16, F16 = 0, 1, 2
MAX_SMEM = 227 * 1024
ORDER = ("ring", "mbar", "wq", "wk", "wv", "wraw", "wb", "wg", "yk", "yq", "scal", "xh", "xl",
         "am", "fm", "hk", "kl", "hkraw")


def round4(x):
    return (x + 3) & ~3


@pytest.fixture(scope="module")
def probe():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    tmp = tempfile.mkdtemp(prefix="rssm_layout_")
    exe = os.path.join(tmp, "layout_probe")
    subprocess.run([nvcc, "-x", "cu", "-std=c++17", "-I", CSRC,
                    os.path.join(ROOT, "tests", "layout_probe.cu"), "-o", exe],
                   check=True, capture_output=True, timeout=300)

    def run(configs):
        args = [str(x) for c in configs for x in c]
        out = subprocess.run([exe] + args, check=True, capture_output=True, text=True).stdout
        return [json.loads(line) for line in out.splitlines()]

    yield run
    shutil.rmtree(tmp, ignore_errors=True)


def _cfg(algo=GDN, sb=4, NT=1, T=1, L=16, dk=128, dv=128, in_dt=BF16, rk=F16, rd=F32, tc=0):
    return (algo, sb, NT, T, L, dk, dv, in_dt, rk, rd, tc)


GRID = [_cfg(algo, sb, NT, T, L, dk, dv, BF16, rk, rd)
        for algo in (GDN, KDA) for sb in (4, 2) for NT, T in ((1, 1), (4, 3), (8, 8))
        for L in (16, 32, 64) for dk, dv in ((128, 128), (64, 64), (32, 128))
        for rk in (F32, BF16, F16) for rd in (F32, F16)]


def test_every_plan_is_aligned_ordered_and_fits(probe):
    for cfg, m in zip(GRID, probe(GRID)):
        offs = {k: v for k, v in m.items() if k not in ("kip", "ns", "total", "ctas",
                                                        "rank_bytes")}
        assert all(v % 16 == 0 for v in offs.values()), cfg
        assert m["total"] % 16 == 0 and m["total"] <= MAX_SMEM, cfg
        assert m["ring"] == 0 and m["ns"] >= 1 and m["ctas"] >= 1, cfg
        seq = [m[k] for k in ORDER]
        assert seq == sorted(seq), cfg
        assert max(offs.values()) <= m["total"], cfg
        assert m["rank"] + (m["rank_bytes"] if cfg[2] == 1 else 0) <= m["total"], cfg


def test_long_ring_decode_keys_in_place(probe):
    """GDN decode on rings of 17..64 records with 16-bit keys and 128 value
    columns: no fp32 key region, the landing zone holds the keys transposed
    ([dk][round4(L)] 16-bit), and the row order has a region of its own."""
    cfgs = [_cfg(GDN, sb, 1, 1, L, dk, 128, BF16, rk, F32)
            for sb in (4, 2) for L in (17, 20, 32, 48, 63, 64) for dk in (32, 64, 128)
            for rk in (BF16, F16)]
    for cfg, m in zip(cfgs, probe(cfgs)):
        L, dk = cfg[4], cfg[5]
        assert m["kip"] == 1, cfg
        assert m["kl"] == m["hk"], cfg                      # the fp32 key region is empty
        assert m["hd"] - m["hkraw"] >= 2 * round4(L) * dk, cfg
        assert m["rank"] >= m["hdot"], cfg                   # not inside another region
    off = [_cfg(GDN, 4, 1, 1, 16), _cfg(GDN, 4, 1, 1, 65), _cfg(GDN, 4, 1, 1, 32, rk=F32),
           _cfg(GDN, 4, 1, 1, 32, dv=64), _cfg(KDA, 4, 1, 1, 32), _cfg(GDN, 4, 4, 3, 32)]
    for cfg, m in zip(off, probe(off)):
        assert m["kip"] == 0, cfg
        assert m["kl"] > m["hk"] or cfg[10], cfg


@pytest.mark.parametrize("cfg,ctas", [
    (_cfg(GDN, 4, 1, 1, 16), 4),          # the headline decode: 4 CTAs per SM
    (_cfg(GDN, 2, 1, 1, 16), 4),
    (_cfg(GDN, 4, 1, 1, 32), 4),          # long rings with keys in place
    (_cfg(GDN, 4, 1, 1, 64), 3),
    (_cfg(GDN, 4, 1, 1, 32, rk=F32), 3),  # fp32 keys keep the fp32 key region
    (_cfg(GDN, 4, 4, 3, 16), 4),          # verify, three-token windows
    (_cfg(GDN, 4, 8, 8, 16), 3),          # verify, eight-token windows
    (_cfg(KDA, 4, 1, 1, 32), 3),
    (_cfg(KDA, 2, 1, 1, 32, rd=F16), 4),  # bf16 checkpoint, fp16 key/delta cache
])
def test_ctas_per_sm(probe, cfg, ctas):
    assert probe([cfg])[0]["ctas"] == ctas


def _nt_for(T):
    return 1 if T == 1 else 2 if T == 2 else 4 if T <= 4 else 8 if T <= 8 else 16


def test_no_narrower_window_outgrows_the_widest(probe):
    """rssm_alloc checks that the widest window a store allows fits in shared
    memory; no narrower window of the same store may need more than the limit
    (the plans are not monotone in T: eight-token windows drop a ring stage)."""
    cfgs = [(algo, sb, _nt_for(T), T, L, dk, dv, BF16, rk, rd, 0)
            for algo in (GDN, KDA) for sb in (4, 2) for L in (16, 20, 32, 64, 128, 256)
            for dk, dv in ((128, 128), (256, 128), (128, 256), (256, 256))
            for rk in (F32, F16) for rd in (F32, F16) for T in range(1, 17) if T <= L]
    total = {}
    for cfg, m in zip(cfgs, probe(cfgs)):
        total.setdefault(cfg[:2] + cfg[4:], {})[cfg[3]] = m["total"]
    for key, by_t in total.items():
        for max_t, worst in by_t.items():
            if worst <= MAX_SMEM:
                assert all(by_t[t] <= MAX_SMEM for t in by_t if t <= max_t), (key, max_t)
