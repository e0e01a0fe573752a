#!/usr/bin/env python3
"""Throughput of the ReplaySSM hot path on GB300: replayed tokens/s per layer
and achieved HBM bandwidth of the replay kernel against the measured peak.

Workload (N = 1): a Qwen3.5-4B-shaped Gated DeltaNet decode layer (HK = 16 key
heads, HV = 32 value heads, dk = dv = 128, batch 64 with 8 null slots, ring
L = 16, width T = 1, bf16 q/k/v, fp32 checkpoint and deltas, fp16 ring keys),
48 stacked layers with distinct buffers. A step is one decode pass over all 48
layers plus the cursor advance, replayed from a CUDA graph. The checkpoints
(6 GiB) dwarf the 129 MB L2, so nothing is served from cache between steps.
Rows join a few steps apart before timing, so their cursors are staggered and
every step folds about one row in sixteen, as in steady serving.

A second workload, reported under "verify", times speculative verify + commit
(batch 128, T = 8, L = 16, random accept lengths) on the same head shapes; a
third, under "prefill", times the replay prefill of 8 prompts of 4096 tokens
(one layer per launch, checkpoint written, ALU-bound: reported against the
fp32 FMA peak derived from the SM count and clock).

--impl reference times the fp64 oracle (CPU) on a bounded sample of the same
workload. Under torchrun each rank runs an independent replica (no
collective on the data path; weak scaling).
"""
from __future__ import annotations

import argparse
import hashlib
import glob
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "replayed tokens/s per layer (decode & verify) and HBM GB/s vs GB300 peak"
UNIT = "tokens/s/layer"
WL = dict(workload="Qwen3.5-4B-shaped GDN decode layer", algo="gdn", HK=16, HV=32, dk=128,
          dv=128, batch=64, null_slots=8, L=16, T=1, in_dtype="bf16", state_dtype="f32",
          ring_k_dtype="f16", ring_d_dtype="f32", layers=48)
VERIFY = dict(workload="GDN speculative verify+commit", batch=128, T=8, L=16,
              state_dtype="f32", commit_mode="lazy", layers=48, widths=(8, 3))
VERIFY_FE = dict(VERIFY, workload="GDN speculative verify + fold-every commit (bf16 checkpoint)",
                 state_dtype="bf16", commit_mode="fold_every")
ESZ = {"f32": 4, "bf16": 2, "f16": 2}
PREFILL = dict(workload="Qwen3.5-4B-shaped GDN replay prefill", prompts=8, tokens=4096,
               in_dtype="bf16", state_dtype="f32")
FP32_LANES_PER_SM = 128  # fp32 FMA lanes per SM (4 sub-partitions x 32)
KDA = dict(workload="KDA decode+verify (alternating T = 1 / T = 3)", HK=32, HV=32, dk=128, dv=128,
           batch=64, L=32, T=3, layers=8,
           variants=(("bf16 state, fp16 k/delta cache", "bf16", "f16", "f16", "fold_every"),
                     ("fp32 state", "f32", "f16", "f32", "lazy")))
CONV = dict(workload="Qwen3.5-4B-shaped conv window (q, k, v channels) for verify + commit",
            batch=128, T=8, K=4, layers=8, dtype="bf16")


# --------------------------------------------------------------- accounting
def row_bytes(c, T, fold, HK, HV, dk, dv, s_state, s_in, s_k, s_d, n_g=1):
    """Algorithmic HBM bytes of one live row in one replay launch.

    Reads: the checkpoint tile once, c history records (key per key head,
    delta and gate per value head), the window's q/k/v/beta/g. Writes: the
    outputs, T records (key per key head; delta, gate, v, beta per value head)
    and, on a fold, the folded checkpoint.
    """
    state = HV * dk * dv * s_state
    hist = c * (HK * dk * s_k + HV * dv * s_d + HV * n_g * 4)
    win = T * (2 * HK * dk * s_in + HV * dv * s_in + HV * (1 + n_g) * 4)
    out = T * HV * dv * s_in
    rec = T * (HK * dk * s_k + HV * dv * s_d + HV * n_g * 4 + HV * dv * s_in + HV * 4)
    return state + hist + win + out + rec + (state if fold else 0)


def commit_bytes(n, HK, HV, dk, dv, s_state, s_k, s_d, n_g=1):
    """Algorithmic HBM bytes of one live row in a fold-every commit (all of one
    layer): the checkpoint read and written once and the n = base + a
    committed records (key per key head, delta and gate per value head) read."""
    return 2 * HV * dk * dv * s_state + n * (HK * dk * s_k + HV * dv * s_d + HV * n_g * 4)


def max_over_ranks(x: float, world: int, device) -> float:
    """Largest value of x over all ranks (the slowest replica's time)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(tokens_per_rank: float, world: int, t_max_s: float) -> float:
    """Whole-job throughput of `world` independent replicas (weak scaling)."""
    return world * tokens_per_rank / t_max_s


def nt_for(T):
    """The kernel's window width for a verify of T tokens (powers of two)."""
    nt = 1
    while nt < T:
        nt *= 2
    return nt


def advance(c, T, L, a):
    fold = c + T > L
    return (0 if fold else c) + a, fold


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def ncu_traffic(name="replay_gdn_decode_qwen_shapes.md"):
    """Bytes per launch from a committed ncu summary, if its kernel sources
    still hash to what was profiled; else None."""
    path = os.path.join(ROOT, "profiles", name)
    if not os.path.exists(path):
        return None
    vals = {}
    with open(path) as f:
        for line in f:
            if ":" in line and line.startswith("- "):
                k, v = line[2:].split(":", 1)
                vals[k.strip()] = v.strip().strip("`")
    try:
        want = vals["sources_sha256"]
        per_launch = float(vals["dram_bytes_per_launch_full_batch"])
    except (KeyError, ValueError):
        return None
    return per_launch if want == sources_hash() else None


# The files that define the decode launch the ncu summary describes (kernel,
# shared-memory plan, launch); a change to any of them invalidates the traffic.
DECODE_SOURCES = ("replay_impl.cuh", "rssm_history.cuh", "rssm_common.cuh", "rssm_mma.cuh",
                  "rssm_tc.cuh", "replay_launch.cuh",
                  "replay_gdn_f32.cu")


def sources_hash():
    h = hashlib.sha256()
    for name in DECODE_SOURCES:
        f = os.path.join(ROOT, "linear_attention_state_rssm_gb300", "csrc", name)
        h.update(name.encode())
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


# ------------------------------------------------------------------ clocks
class Clocks:
    """nvidia-smi samples of the SM clock and throttle reasons while the GPU is
    loaded. The sampler is started (and its first, idle sample read) before
    the timed region; `keep_loaded` then repeats the timed step, untimed,
    until the sampler has covered at least `min_s` of load."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    INTERVAL_MS = 50

    def __init__(self, index):
        self.index, self.proc, self.t0 = index, None, None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(self.INTERVAL_MS)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.proc.stdout.readline()  # the sampler runs; this sample predates the load
        except OSError:
            self.proc = None
        self.t0 = time.perf_counter()
        return self

    def keep_loaded(self, step, min_s=0.5):
        """Run `step()` (untimed) until min_s has passed since the sampler's
        first sample; returns how many steps ran."""
        n = 0
        while self.proc is not None and time.perf_counter() - self.t0 < min_s:
            step()
            n += 1
        return n

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        rows = []
        for line in (self.out or "").strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                rows.append((float(parts[0]), float(parts[1]), parts[4:8]))
            except ValueError:
                continue
        if not rows:
            return None
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({names[i] for _, _, r in rows for i, x in enumerate(r)
                          if x.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": rows[0][1],
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------- device inputs
def device_inputs(torch, gen, n_layers, B, T, HK, HV, dk, dv, dtype):
    """Seeded synthetic window inputs for every layer, resident in HBM:
    q, k ~ N(0,1) L2-normalised per head, v ~ N(0,1), beta = sigmoid(N(0,1)),
    g = -softplus(N(0,1)); packed so one copy moves a whole step."""
    n = n_layers * B * T
    dev = "cuda"
    q = torch.randn((n, HK, dk), generator=gen, device=dev)
    k = torch.randn((n, HK, dk), generator=gen, device=dev)
    q = q / q.norm(dim=-1, keepdim=True)
    k = k / k.norm(dim=-1, keepdim=True)
    v = torch.randn((n, HV, dv), generator=gen, device=dev)
    beta = torch.sigmoid(torch.randn((n, HV), generator=gen, device=dev))
    g = -torch.nn.functional.softplus(torch.randn((n, HV), generator=gen, device=dev))
    half = torch.cat([q.reshape(-1), k.reshape(-1), v.reshape(-1)]).to(dtype)
    flt = torch.cat([beta.reshape(-1), g.reshape(-1)]).float()
    return half, flt


def views(half, flt, layer, n_layers, B, T, HK, HV, dk, dv):
    nq = n_layers * B * T * HK * dk
    per_q, per_v, per_s = B * T * HK * dk, B * T * HV * dv, B * T * HV
    q = half[layer * per_q:(layer + 1) * per_q].view(B * T, HK, dk)
    k = half[nq + layer * per_q:nq + (layer + 1) * per_q].view(B * T, HK, dk)
    v = half[2 * nq + layer * per_v:2 * nq + (layer + 1) * per_v].view(B * T, HV, dv)
    ns = n_layers * B * T * HV
    beta = flt[layer * per_s:(layer + 1) * per_s].view(B * T, HV)
    g = flt[ns + layer * per_s:ns + (layer + 1) * per_s].view(B * T, HV)
    return q, k, v, beta, g


# ------------------------------------------------------------------- ours
def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist
    from linear_attention_state_rssm_gb300 import build as _build
    _build.build()
    from linear_attention_state_rssm_gb300.store import ReplayStore

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    w = WL
    nl, B, T, L = args.layers, w["batch"], w["T"], w["L"]
    HK, HV, dk, dv = w["HK"], w["HV"], w["dk"], w["dv"]
    gen = torch.Generator(device=dev)
    gen.manual_seed(1000 + rank)

    st = ReplayStore("gdn", nl, B, HK, HV, dk, dv, L, 1, w["in_dtype"], w["state_dtype"],
                     w["ring_k_dtype"], w["ring_d_dtype"], "lazy", device=dev)
    st.rssm_set_plan(args.plan)
    for layer in range(nl):
        st.state[layer].normal_(0.0, 0.1, generator=gen)
    null = torch.randperm(B, generator=torch.Generator().manual_seed(7))[:w["null_slots"]]
    slots = torch.arange(B, dtype=torch.int32)
    slots[null] = -1
    live_rows = [r for r in range(B) if slots[r] >= 0]
    B_live = len(live_rows)
    slot_d = slots.to(dev)
    half, flt = device_inputs(torch, gen, nl, B, T, HK, HV, dk, dv, torch.bfloat16)
    out = torch.empty((nl, B * T, HV, dv), dtype=torch.bfloat16, device=dev)
    lv = [views(half, flt, l, nl, B, T, HK, HV, dk, dv) for l in range(nl)]

    def step(slot_t, events=None):
        for l in range(nl):
            if events is not None:
                events[l].record()
            st.rssm_decode(l, *lv[l], slot_t, out[l], advance_cursor=(l == nl - 1))
        if events is not None:
            events[nl].record()

    # stagger: row r joins at step r % L so cursors spread over [0, L)
    for j in range(L):
        s = slots.clone()
        for r in range(B):
            if r % L > j:
                s[r] = -1
        step(s.to(dev))
    torch.cuda.synchronize()
    cur = st.cursor.cpu().tolist()

    cap = torch.cuda.Stream(device=dev)
    cap.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cap):
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=cap):
            step(slot_d)
    torch.cuda.current_stream().wait_stream(cap)
    torch.cuda.synchronize()

    def host_advance(cur, steps):
        """Cursor trajectory and algorithmic bytes per launch for `steps` steps."""
        per_launch = []
        for _ in range(steps):
            tot = 0
            nxt = list(cur)
            for r in live_rows:
                c = cur[r]
                nxt[r], fold = advance(c, T, L, 1)
                tot += row_bytes(c, T, fold, HK, HV, dk, dv, 4, 2, 2, 4)
            per_launch.append(tot)
            cur = nxt
        return cur, per_launch

    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()
    cur, _ = host_advance(cur, args.warmup)

    # ---- timed region: K steps
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with Clocks(local_rank) as clk:
        e0.record()
        for _ in range(args.steps):
            graph.replay()
        e1.record()
        torch.cuda.synchronize()

        def pad_step():
            for _ in range(16):
                graph.replay()
            torch.cuda.synchronize()
        pad = 16 * clk.keep_loaded(pad_step)
    if world > 1:
        dist.barrier()
    t_ms = e0.elapsed_time(e1)
    cur, bytes_timed = host_advance(cur, args.steps)
    cur, _ = host_advance(cur, pad)  # untimed steps that kept the clock sampler loaded
    t_max = max_over_ranks(t_ms, world, dev)
    value = job_throughput(B_live * T * nl * args.steps, world, t_max / 1e3)
    ms_per_step = t_max / args.steps

    # ---- per-launch duration of the replay kernel: the timed region (CUDA events
    # on the launching stream around K graph replays) per layer launch. The
    # step's cursor kernel (a few microseconds) is charged to the layers, which
    # understates the replay kernel's bandwidth slightly.
    k_ms = ms_per_step / nl
    k_bytes = statistics.mean(bytes_timed)
    achieved = k_bytes / (k_ms / 1e3) / 1e9
    peak, peak_kind = peaks()
    traffic = ncu_traffic()

    # ---- end to end through the C ABI with host buffers. Every step copies its
    # inputs from pinned host memory and reads its outputs back, as a serving
    # loop does, with the copies pipelined against the compute: inputs and
    # outputs are double-buffered (one captured graph per buffer set), step
    # i's inputs go up on a copy stream while step i - 1 computes, and its
    # outputs come down on another while step i + 1 computes. The timed region
    # runs from the first upload to the last read-back.
    half_h = half.cpu().pin_memory()
    flt_h = flt.cpu().pin_memory()
    out_h = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
    half_b = [half, torch.empty_like(half)]
    flt_b = [flt, torch.empty_like(flt)]
    out_b = [out, torch.empty_like(out)]
    lv2 = [views(half_b[1], flt_b[1], l, nl, B, T, HK, HV, dk, dv) for l in range(nl)]
    graphs = [graph, torch.cuda.CUDAGraph()]
    with torch.cuda.stream(cap):
        with torch.cuda.graph(graphs[1], stream=cap):
            for l in range(nl):
                st.rssm_decode(l, *lv2[l], slot_d, out_b[1][l], advance_cursor=(l == nl - 1))
    torch.cuda.current_stream().wait_stream(cap)
    torch.cuda.synchronize()
    comp = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev = lambda: torch.cuda.Event()  # noqa: E731

    def pipelined(n_steps):
        done = [None, None]     # compute of the last step on each buffer set
        read = [None, None]     # read-back of the last step on each buffer set
        for i in range(n_steps):
            b = i % 2
            with torch.cuda.stream(s_in):
                if done[b] is not None:
                    s_in.wait_event(done[b])      # the buffers' last step has run
                half_b[b].copy_(half_h, non_blocking=True)
                flt_b[b].copy_(flt_h, non_blocking=True)
                up = ev()
                up.record(s_in)
            comp.wait_event(up)
            if read[b] is not None:
                comp.wait_event(read[b])          # the outputs' last read-back is done
            graphs[b].replay()
            done[b] = ev()
            done[b].record(comp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(done[b])
                out_h[b].copy_(out_b[b], non_blocking=True)
                read[b] = ev()
                read[b].record(s_out)
        for r in read:
            if r is not None:
                comp.wait_event(r)

    pipelined(2)
    torch.cuda.synchronize()
    cur, _ = host_advance(cur, 2)
    if world > 1:
        dist.barrier()
    e2, e3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2.record(comp)
    s_in.wait_stream(comp)
    pipelined(args.steps)
    e3.record(comp)
    torch.cuda.synchronize()
    cur, _ = host_advance(cur, args.steps)
    te = max_over_ranks(e2.elapsed_time(e3), world, dev)
    e2e = {"value": job_throughput(B_live * T * nl * args.steps, world, te / 1e3), "unit": UNIT,
           "h2d_bytes_per_step": half.numel() * 2 + flt.numel() * 4,
           "d2h_bytes_per_step": out.numel() * 2,
           "copies": "pipelined against compute on two copy streams, double-buffered"}
    err = st.rssm_get_device_error()

    # ---- comparison point: native fused-recurrent decode on the same shapes
    # (the state read and written every token; ring unused), 48 layers per step
    native = None
    if not args.no_native:
        with torch.cuda.stream(cap):
            ngraph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(ngraph, stream=cap):
                for l in range(nl):
                    st.rssm_native_decode(l, *lv[l], slot_d, out[l])
        torch.cuda.current_stream().wait_stream(cap)
        for _ in range(args.warmup):
            ngraph.replay()
        torch.cuda.synchronize()
        n0, n1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n0.record()
        for _ in range(args.steps):
            ngraph.replay()
        n1.record()
        torch.cuda.synchronize()
        tn = n0.elapsed_time(n1) / 1e3
        n_bytes = B_live * (2 * HV * dk * dv * 4 + 2 * HK * dk * 2 + HV * dv * 2 + 2 * HV * 4
                            + HV * dv * 2)
        native = {"kernel": "native_decode_kernel<GDN, f32>",
                  "tokens_per_s_per_layer": B_live * nl * args.steps / tn,
                  "launch_ms": tn * 1e3 / (args.steps * nl),
                  "achieved_gbs": n_bytes * nl * args.steps / tn / 1e9,
                  "bytes_per_launch": n_bytes}
        err |= st.rssm_get_device_error()
        del ngraph
    del graph, st, half, flt, out, lv
    torch.cuda.empty_cache()

    ver = run_verify(args, torch, dev, rank, peak, local_rank) if not args.no_verify else None
    ver3 = (run_verify(args, torch, dev, rank, peak, local_rank, T=VERIFY["widths"][1])
            if not args.no_verify else None)
    ver_fe = (run_verify(args, torch, dev, rank, peak, local_rank, cfg=VERIFY_FE)
              if not args.no_verify else None)
    kda = run_kda(args, torch, dev, rank, peak, local_rank) if not args.no_kda else None
    pre = run_prefill(args, torch, dev, rank) if not args.no_prefill else None
    conv = run_conv(args, torch, dev, rank, peak) if not args.no_conv else None

    res = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded torch RNG on device; distributions of the pages' tiny "
                "GDN workload)",
        "config": bench_config(nl, world),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_kind": f"{peak_kind} (hbm_gbs, burst)",
                     "traffic": traffic, "kernel": "replay_kernel<GDN, f32, 1>",
                     "algorithmic_bytes_per_launch": k_bytes, "launch_ms": k_ms},
        "gpu_launches": args.steps * (nl + 1),  # the timed region: replay layers + cursor
        "e2e": e2e,
        "clocks": clk.summary(),
        "device_error_word": err,
    }
    if native is not None:
        res["native_decode"] = native
    if ver is not None:
        res["verify"] = ver
    if ver3 is not None:
        res["verify_t3"] = ver3
    if ver_fe is not None:
        res["verify_fold_every"] = ver_fe
    if kda is not None:
        res["kda"] = kda
    if pre is not None:
        res["prefill"] = pre
    if conv is not None:
        res["conv"] = conv
    return res


def run_conv(args, torch, dev, rank, peak):
    """Conv window (verify width, drafts kept) and its commit over distinct
    per-layer buffers; HBM-bound."""
    from linear_attention_state_rssm_gb300.store import ConvWindows
    w_, c = WL, CONV
    B, T, K, nl = c["batch"], c["T"], c["K"], c["layers"]
    D = 2 * w_["HK"] * w_["dk"] + w_["HV"] * w_["dv"]
    gen = torch.Generator(device=dev)
    gen.manual_seed(4000 + rank)
    cws = [ConvWindows(B, D, K, T, c["dtype"], device=dev) for _ in range(nl)]
    for cw in cws:
        cw.window.normal_(generator=gen)
    x = torch.randn(nl, B * T, D, generator=gen, device=dev).to(torch.bfloat16)
    y = torch.empty_like(x)
    w = torch.randn(nl, D, K, generator=gen, device=dev)
    bias = torch.randn(nl, D, generator=gen, device=dev)
    slot = torch.arange(B, dtype=torch.int32, device=dev)
    acc = torch.randint(0, T + 1, (B,), generator=gen, device=dev, dtype=torch.int32)
    ew = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    ec = [torch.cuda.Event(enable_timing=True) for _ in range(2)]

    def windows():
        for l in range(nl):
            cws[l].rssm_conv_window(x[l], w[l], bias[l], slot, T, y[l], act="silu")

    def commits():
        for l in range(nl):
            cws[l].rssm_conv_commit(slot, acc, T)

    # one eager pass, then each layer loop as one CUDA graph (as a serving step
    # replays it), so the times are the kernels' and not the host's launch rate
    windows()
    commits()
    torch.cuda.synchronize()
    cap = torch.cuda.Stream(device=dev)
    cap.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cap):
        g_win, g_com = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_win, stream=cap):
            windows()
        with torch.cuda.graph(g_com, stream=cap):
            commits()
    torch.cuda.current_stream().wait_stream(cap)
    t_win = t_com = 0.0
    for it in range(args.warmup + args.steps):
        timed = it >= args.warmup
        if timed:
            ew[0].record()
        g_win.replay()
        if timed:
            ew[1].record()
            ec[0].record()
        g_com.replay()
        if timed:
            ec[1].record()
            torch.cuda.synchronize()
            t_win += ew[0].elapsed_time(ew[1])
            t_com += ec[0].elapsed_time(ec[1])
    err = sum(int(cw.err_word.item()) for cw in cws)
    n = args.steps * nl
    ms_win, ms_com = t_win / n, t_com / n
    # window: read the kept window, x and the taps, write y and the drafts
    bytes_win = B * ((K - 1) * D * 2 + 3 * T * D * 2) + D * (K + 1) * 4
    achieved = bytes_win / (ms_win / 1e3) / 1e9
    del g_win, g_com, cws, x, y
    torch.cuda.empty_cache()
    return {"workload": c["workload"], "batch": B, "T": T, "K": K, "channels": D,
            "layers": nl, "dtype": c["dtype"], "cuda_graph": True, "window_launch_ms": ms_win,
            "commit_launch_ms": ms_com,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "bytes_per_launch": bytes_win,
                         "kernel": "conv_window_kernel<4>"},
            "device_error_word": err}


def run_prefill(args, torch, dev, rank):
    """Replay prefill of PREFILL's prompts into one layer's checkpoints; the
    prefill kernel is ALU-bound (fp32 FMA on CUDA cores)."""
    from linear_attention_state_rssm_gb300.store import ReplayStore
    w, pf = WL, PREFILL
    B, N = args.prefill_prompts, args.prefill_tokens
    HK, HV, dk, dv = w["HK"], w["HV"], w["dk"], w["dv"]
    gen = torch.Generator(device=dev)
    gen.manual_seed(3000 + rank)
    st = ReplayStore("gdn", 1, B, HK, HV, dk, dv, w["L"], 1, pf["in_dtype"], pf["state_dtype"],
                     "f16", "f32", "lazy", device=dev)
    st.state.normal_(0.0, 0.1, generator=gen)
    tot = B * N
    nrm = torch.nn.functional.normalize
    q = nrm(torch.randn(tot, HK, dk, device=dev, generator=gen), dim=-1).to(torch.bfloat16)
    k = nrm(torch.randn(tot, HK, dk, device=dev, generator=gen), dim=-1).to(torch.bfloat16)
    v = torch.randn(tot, HV, dv, device=dev, generator=gen).to(torch.bfloat16)
    beta = torch.sigmoid(torch.randn(tot, HV, device=dev, generator=gen))
    g = -torch.nn.functional.softplus(torch.randn(tot, HV, device=dev, generator=gen))
    cu = torch.arange(B + 1, dtype=torch.int32, device=dev) * N
    slot = torch.arange(B, dtype=torch.int32, device=dev)
    o = torch.empty(tot, HV, dv, dtype=torch.bfloat16, device=dev)
    for _ in range(args.warmup):
        st.rssm_prefill(0, q, k, v, beta, g, cu, slot, o, reset_cursor=True)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        st.rssm_prefill(0, q, k, v, beta, g, cu, slot, o, reset_cursor=True)
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / args.steps
    err = st.rssm_get_device_error()
    props = torch.cuda.get_device_properties(dev)
    sm_mhz = max_sm_mhz(dev.index if dev.index is not None else 0)
    peak = props.multi_processor_count * FP32_LANES_PER_SM * 2 * sm_mhz * 1e6 / 1e12
    flops = 6.0 * dk * dv * HV * tot  # the token recurrence: S^T k, rank-1 update, S^T q
    achieved = flops / (ms / 1e3) / 1e12
    del st, q, k, v, beta, g, o
    torch.cuda.empty_cache()
    return {"workload": pf["workload"], "prompts": B, "tokens_per_prompt": N,
            "in_dtype": pf["in_dtype"], "state_dtype": pf["state_dtype"],
            "tokens_per_s_per_layer": tot / (ms / 1e3), "launch_ms": ms,
            "roofline": {"bound": "alu", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                         "frac": achieved / peak,
                         "peak_kind": f"derived fp32 FMA peak: {props.multi_processor_count} SMs"
                                      f" x {FP32_LANES_PER_SM} lanes x 2 flop x {sm_mhz} MHz "
                                      "(the scan runs on CUDA cores, the chunk products on "
                                      "the tensor cores)",
                         "flops_per_launch": flops,
                         "kernel": "prefill_kernel<GDN, f32, 64, bf16>"},
            "gpu_launches_per_step": 2, "device_error_word": err}


def max_sm_mhz(index):
    """Maximum SM clock of the GPU (nvidia-smi), 2070 MHz if it cannot be read."""
    try:
        out = subprocess.run(["nvidia-smi", "-i", str(index), "--query-gpu=clocks.max.sm",
                              "--format=csv,noheader,nounits"], capture_output=True, text=True,
                             timeout=30).stdout.strip()
        return int(float(out.splitlines()[0]))
    except (OSError, ValueError, IndexError, subprocess.TimeoutExpired):
        return 2070


def commit_summary(t_com, steps, com_bytes, fold_every, peak, v, nl):
    """The commit's own line: one rssm_commit per step (every layer's fold and
    the cursor kernel for a fold-every store; the cursor kernel alone for a
    lazy one), timed between CUDA events around its graph."""
    launch_ms = t_com * 1e3 / steps
    res = {"launch_ms": launch_ms, "algorithmic_bytes_per_launch": statistics.mean(com_bytes),
           "covers": "one rssm_commit (every layer)"}
    if not fold_every:
        res["note"] = "lazy commit: the cursor kernel only (no state bytes)"
        return res
    achieved = statistics.mean(com_bytes) / (launch_ms / 1e3) / 1e9
    res["note"] = "fold kernel over all layers + cursor kernel"
    res["per_layer_us"] = launch_ms * 1e3 / nl
    res["roofline"] = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                       "frac": achieved / peak, "traffic": None,
                       "kernel": "fold_kernel<GDN, %s, 16>" % v["state_dtype"],
                       "bytes": "per row with n = base + a > 0 records: checkpoint read and "
                                "written once + n records (key, delta, gate) read"}
    return res


def run_verify(args, torch, dev, rank, peak, clk_index, T=None, cfg=None):
    """Speculative verify (T = 8, or 3) + lazy commit over 48 layers, batch 128. The
    verify launches and the commit are captured in two CUDA graphs and timed
    apart (CUDA events between them), so the verify kernel's own launch time
    and bandwidth come out; the host follows the rows' cursors to count each
    launch's algorithmic bytes."""
    from linear_attention_state_rssm_gb300.store import ReplayStore
    w, v = WL, (VERIFY if cfg is None else cfg)
    nl, B, L = args.layers, v["batch"], v["L"]
    T = v["T"] if T is None else T
    HK, HV, dk, dv = w["HK"], w["HV"], w["dk"], w["dv"]
    gen = torch.Generator(device=dev)
    gen.manual_seed(2000 + rank)
    st = ReplayStore("gdn", nl, B, HK, HV, dk, dv, L, T, "bf16", v["state_dtype"], "f16", "f32",
                     v["commit_mode"], device=dev)
    st.rssm_set_plan(args.plan)
    for layer in range(nl):
        st.state[layer].normal_(0.0, 0.1, generator=gen)
    slot = torch.arange(B, dtype=torch.int32, device=dev)
    half, flt = device_inputs(torch, gen, nl, B, T, HK, HV, dk, dv, torch.bfloat16)
    out = torch.empty((nl, B * T, HV, dv), dtype=torch.bfloat16, device=dev)
    lv = [views(half, flt, l, nl, B, T, HK, HV, dk, dv) for l in range(nl)]
    n_acc = args.warmup + args.steps + 1
    acc = torch.randint(0, T + 1, (n_acc, B), generator=gen, device=dev, dtype=torch.int32)
    acc_h = acc.cpu().tolist()
    acc_cur = torch.empty(B, dtype=torch.int32, device=dev)
    s_state = ESZ[v["state_dtype"]]
    fold_every = v["commit_mode"] == "fold_every"

    cap = torch.cuda.Stream(device=dev)
    cap.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cap):
        g_ver, g_com = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_ver, stream=cap):
            for l in range(nl):
                st.rssm_verify(l, *lv[l], slot, T, out[l])
        with torch.cuda.graph(g_com, stream=cap):
            st.rssm_commit(slot, acc_cur, T)
    torch.cuda.current_stream().wait_stream(cap)

    cur = [0] * B
    ver_bytes, com_bytes = [], []

    def host_step(i):
        tot, ctot = 0, 0
        for r in range(B):
            c = cur[r]
            nxt, fold = advance(c, T, L, acc_h[i][r])
            tot += row_bytes(c, T, fold, HK, HV, dk, dv, s_state, 2, 2, 4)
            if fold_every and nxt > 0:  # the commit folds every layer (rows with records)
                ctot += nl * commit_bytes(nxt, HK, HV, dk, dv, s_state, 2, 4)
            cur[r] = 0 if fold_every else nxt
        return tot, ctot

    def step(i):
        acc_cur.copy_(acc[i])
        g_ver.replay()
        g_com.replay()

    for i in range(args.warmup):
        step(i)
        host_step(i)
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    with Clocks(clk_index) as clk:
        for j in range(args.steps):
            i = args.warmup + j
            acc_cur.copy_(acc[i])
            ev[j][0].record()
            g_ver.replay()
            ev[j][1].record()
            g_com.replay()
            ev[j][2].record()
            b, cb = host_step(i)
            ver_bytes.append(b)
            com_bytes.append(cb)
        torch.cuda.synchronize()
        # keep the GPU loaded (untimed) until the clock sampler has seen it
        extra = [0]

        def pad():
            step(n_acc - 1)
            extra[0] += 1
            torch.cuda.synchronize()
        clk.keep_loaded(pad)
    t_ver = sum(e[0].elapsed_time(e[1]) for e in ev) / 1e3
    t_com = sum(e[1].elapsed_time(e[2]) for e in ev) / 1e3
    err = st.rssm_get_device_error()
    del g_ver, g_com, st
    torch.cuda.empty_cache()
    launches = args.steps * nl
    launch_ms = t_ver * 1e3 / launches
    bytes_launch = statistics.mean(ver_bytes)
    achieved = bytes_launch / (launch_ms / 1e3) / 1e9
    acc_sum = sum(sum(acc_h[args.warmup + j]) for j in range(args.steps))
    res = {"workload": v["workload"], "batch": B, "T": T, "L": L, "layers": nl,
           "state_dtype": v["state_dtype"], "commit_mode": v["commit_mode"],
           "replayed_tokens_per_s_per_layer": B * T * launches / t_ver,
           "accepted_tokens_per_s_per_layer": acc_sum * nl / (t_ver + t_com),
           "ms_per_step": (t_ver + t_com) * 1e3 / args.steps,
           "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                        "frac": achieved / peak,
                        "traffic": (ncu_traffic("replay_gdn_verify_t8_qwen_shapes.md")
                                    if T == 8 and v["state_dtype"] == "f32" else None),
                        "kernel": "replay_kernel<GDN, %s, %d>" % (v["state_dtype"], nt_for(T)),
                        "algorithmic_bytes_per_launch": bytes_launch, "launch_ms": launch_ms},
           "commit": commit_summary(t_com, args.steps, com_bytes, fold_every, peak, v, nl),
           "clocks": clk.summary(), "device_error_word": err}
    return res


def run_kda(args, torch, dev, rank, peak, clk_index):
    """KDA decode + verify (HK = HV = 32, dk = dv = 128, batch 64, ring 32):
    decode (T = 1) and verify (T = 3, accept ~ U[0, 3]) steps alternate over
    KDA["layers"] stacked layers, in two variants (bf16 checkpoint with fp16 key
    and delta cache, committed fold-every; fp32 checkpoint, fp16 keys, fp32
    deltas, lazy). Decode launches, verify launches and the commit are timed
    apart; each kind's bytes per launch follow the rows' cursors."""
    from linear_attention_state_rssm_gb300.store import ReplayStore
    k_ = KDA
    nl, B, L, T = k_["layers"], k_["batch"], k_["L"], k_["T"]
    HK, HV, dk, dv = k_["HK"], k_["HV"], k_["dk"], k_["dv"]
    out_all = []
    for vi, (name, sdt, rk, rd, mode) in enumerate(k_["variants"]):
        gen = torch.Generator(device=dev)
        gen.manual_seed(6000 + 10 * rank + vi)
        st = ReplayStore("kda", nl, B, HK, HV, dk, dv, L, T, "bf16", sdt, rk, rd, mode,
                         device=dev)
        for layer in range(nl):
            st.state[layer].normal_(0.0, 0.1, generator=gen)
        slot = torch.arange(B, dtype=torch.int32, device=dev)
        nrm = torch.nn.functional.normalize

        def inputs(Tw):
            n = nl * B * Tw
            q = nrm(torch.randn(n, HK, dk, generator=gen, device=dev), dim=-1).to(torch.bfloat16)
            kk = nrm(torch.randn(n, HK, dk, generator=gen, device=dev), dim=-1).to(torch.bfloat16)
            vv = torch.randn(n, HV, dv, generator=gen, device=dev).to(torch.bfloat16)
            beta = torch.sigmoid(torch.randn(n, HV, generator=gen, device=dev))
            g = -torch.nn.functional.softplus(torch.randn(n, HV, dk, generator=gen, device=dev))
            o = torch.empty(n, HV, dv, dtype=torch.bfloat16, device=dev)
            per = B * Tw
            return [tuple(x[l * per:(l + 1) * per] for x in (q, kk, vv, beta, g, o))
                    for l in range(nl)]
        dec_in, ver_in = inputs(1), inputs(T)
        n_acc = args.warmup + args.steps + 1
        acc = torch.randint(0, T + 1, (n_acc, B), generator=gen, device=dev, dtype=torch.int32)
        acc_h = acc.cpu().tolist()
        acc_cur = torch.empty(B, dtype=torch.int32, device=dev)
        cap = torch.cuda.Stream(device=dev)
        cap.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(cap):
            g_dec, g_ver, g_com = (torch.cuda.CUDAGraph() for _ in range(3))
            with torch.cuda.graph(g_dec, stream=cap):
                for l in range(nl):
                    q, kk, vv, beta, g, o = dec_in[l]
                    st.rssm_decode(l, q, kk, vv, beta, g, slot, o, advance_cursor=l == nl - 1)
            with torch.cuda.graph(g_ver, stream=cap):
                for l in range(nl):
                    q, kk, vv, beta, g, o = ver_in[l]
                    st.rssm_verify(l, q, kk, vv, beta, g, slot, T, o)
            with torch.cuda.graph(g_com, stream=cap):
                st.rssm_commit(slot, acc_cur, T)
        torch.cuda.current_stream().wait_stream(cap)
        s_state, s_d = ESZ[sdt], ESZ[rd]
        fold_every = mode == "fold_every"
        cur = [0] * B
        byt = {"decode": [], "verify": [], "commit": []}

        def host_pair(i, record):
            d = vb = cb = 0
            for r in range(B):
                c = cur[r]
                nxt, fold = advance(c, 1, L, 1)
                d += row_bytes(c, 1, fold, HK, HV, dk, dv, s_state, 2, 2, s_d, dk)
                c = nxt
                nxt, fold = advance(c, T, L, acc_h[i][r])
                vb += row_bytes(c, T, fold, HK, HV, dk, dv, s_state, 2, 2, s_d, dk)
                if fold_every and nxt > 0:  # the commit folds every layer (rows with records)
                    cb += nl * commit_bytes(nxt, HK, HV, dk, dv, s_state, 2, s_d, dk)
                cur[r] = 0 if fold_every else nxt
            if record:
                byt["decode"].append(d)
                byt["verify"].append(vb)
                byt["commit"].append(cb)

        for i in range(args.warmup):
            acc_cur.copy_(acc[i])
            g_dec.replay()
            g_ver.replay()
            g_com.replay()
            host_pair(i, False)
        torch.cuda.synchronize()
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
        with Clocks(clk_index) as clk:
            for j in range(args.steps):
                i = args.warmup + j
                acc_cur.copy_(acc[i])
                ev[j][0].record()
                g_dec.replay()
                ev[j][1].record()
                g_ver.replay()
                ev[j][2].record()
                g_com.replay()
                ev[j][3].record()
                host_pair(i, True)
            torch.cuda.synchronize()
            def pad():
                acc_cur.copy_(acc[n_acc - 1])
                g_dec.replay()
                g_ver.replay()
                g_com.replay()
                torch.cuda.synchronize()
            clk.keep_loaded(pad)
        t = [sum(e[a].elapsed_time(e[a + 1]) for e in ev) / 1e3 for a in range(3)]
        err = st.rssm_get_device_error()
        del g_dec, g_ver, g_com, st, dec_in, ver_in
        torch.cuda.empty_cache()
        launches = args.steps * nl
        res = {"variant": name, "state_dtype": sdt, "ring_k_dtype": rk, "ring_d_dtype": rd,
               "commit_mode": mode, "clocks": clk.summary(), "device_error_word": err}
        for kind, tk, width in (("decode", t[0], 1), ("verify", t[1], T)):
            ms = tk * 1e3 / launches
            bl = statistics.mean(byt[kind])
            ach = bl / (ms / 1e3) / 1e9
            res[kind] = {"T": width, "launch_ms": ms,
                         "replayed_tokens_per_s_per_layer": B * width * launches / tk,
                         "roofline": {"bound": "hbm", "achieved": ach, "peak": peak,
                                      "unit": "GB/s", "frac": ach / peak,
                                      "algorithmic_bytes_per_launch": bl,
                                      "kernel": f"replay_kernel<KDA, {sdt}, {1 if width == 1 else 4}>"}}
        cms = t[2] * 1e3 / args.steps
        cbl = statistics.mean(byt["commit"])
        res["commit"] = {"launch_ms": cms, "algorithmic_bytes_per_launch": cbl,
                         "note": "one rssm_commit: the fold kernel over every layer, then the "
                                 "cursor kernel" if mode == "fold_every" else
                                 "lazy commit: the cursor kernel only (no state bytes)"}
        if cbl > 0:
            ach = cbl / (cms / 1e3) / 1e9
            res["commit"]["roofline"] = {"bound": "hbm", "achieved": ach, "peak": peak,
                                         "unit": "GB/s", "frac": ach / peak,
                                         "kernel": f"fold_kernel<KDA, {sdt}, 32>"}
        out_all.append(res)
    return {"workload": k_["workload"], "batch": B, "L": L, "HK": HK, "HV": HV, "dk": dk,
            "dv": dv, "layers": nl, "in_dtype": "bf16",
            "chained_steps": 2 * (args.warmup + args.steps), "variants": out_all}


# ------------------------------------------------------------ CPU oracle
def oracle_sample(rows, steps, seed=0):
    """Time the fp64 oracle on `rows` rows of the decode workload (1 layer)."""
    import numpy as np
    import synth
    from oracle import ReplayOracle
    w = WL
    HK, HV, dk, dv, L = w["HK"], w["HV"], w["dk"], w["dv"], w["L"]
    S0 = synth.initial_state(seed + 1, rows, HV, dk, dv)
    orc = ReplayOracle("gdn", 1, rows, HK, HV, dk, dv, L, dk ** -0.5, S0)
    inps = [synth.window_inputs(seed * 1000 + s, rows, 1, HK, HV, dk, dv, "gdn", "bf16")
            for s in range(steps)]
    slots = np.arange(rows)
    orc.decode(0, slots, inps[0], advance=True)            # warm the allocator
    c0, t0 = time.process_time(), time.perf_counter()
    for s in range(steps):
        orc.decode(0, slots, inps[s], advance=True)
    wall = time.perf_counter() - t0
    cpu = time.process_time() - c0
    return rows * steps / wall, wall, max(1, round(cpu / wall))


def _oracle_worker(job):
    """One process of the all-cores oracle sample: wait for the common start
    time, then run its own rows (rows are independent)."""
    rows, steps, seed, t_start = job
    import numpy  # noqa: F401  (imported before the start time)
    import oracle  # noqa: F401
    time.sleep(max(0.0, t_start - time.time()))
    t0 = time.time()
    oracle_sample(rows, steps, seed)
    return rows * steps, t0, time.time()


class OraclePool:
    """The oracle on every host core: one single-threaded process per core
    (started with spawn, BLAS held to one thread each), each on its own rows
    of the decode workload, all starting at the same moment."""

    def __init__(self):
        import multiprocessing as mp
        self.n = os.cpu_count() or 1
        keep = {k: os.environ.get(k) for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS",
                                               "MKL_NUM_THREADS")}
        for k in keep:
            os.environ[k] = "1"
        try:
            self.pool = mp.get_context("spawn").Pool(self.n)
            self.pool.map(_oracle_worker, [(2, 2, i, 0.0) for i in range(self.n)])  # warm
        finally:
            for k, v in keep.items():
                if v is None:
                    os.environ.pop(k, None)
                else:
                    os.environ[k] = v

    def run(self, rows, steps):
        """(tokens/s over all processes, wall seconds): tokens of every
        process over the span from the common start to the last finish."""
        t_start = time.time() + 1.0
        res = self.pool.map(_oracle_worker, [(rows, steps, 100 + i, t_start)
                                             for i in range(self.n)])
        toks = sum(r[0] for r in res)
        span = max(r[2] for r in res) - min(r[1] for r in res)
        return toks / span, span

    def close(self):
        self.pool.close()
        self.pool.join()


def cpu_baseline():
    """The oracle as it stands, timed on a bounded sample of the decode
    workload: in one process (its own threads), and on every host core."""
    v1, wall1, cores1 = oracle_sample(8, 20)
    pool = OraclePool()
    try:
        vn, walln = pool.run(8, 20)
    finally:
        pool.close()
    return {"value": vn, "unit": UNIT, "cores": pool.n, "kind": "oracle",
            "sample": f"{pool.n} processes x 8 live rows x 1 layer x 20 decode steps of the "
                      f"same workload, all started together ({walln:.1f} s wall)",
            "host_cores": os.cpu_count(),
            "single_process": {"value": v1, "cores": cores1,
                               "sample": f"8 live rows x 1 layer x 20 decode steps "
                                         f"({wall1:.1f} s wall)"}}


def bench_config(nl, world):
    """The decode workload both arms report (the reference arm times a bounded
    sample of it, described in its cpu_baseline)."""
    w = WL
    return {"workload": w["workload"], "algo": "gdn", "HK": w["HK"], "HV": w["HV"],
            "dk": w["dk"], "dv": w["dv"], "batch": w["batch"],
            "live_rows": w["batch"] - w["null_slots"], "L": w["L"], "T": w["T"], "layers": nl,
            "in_dtype": w["in_dtype"], "state_dtype": w["state_dtype"],
            "ring_k_dtype": w["ring_k_dtype"], "ring_d_dtype": w["ring_d_dtype"],
            "cuda_graph": True, "replicas": world,
            "l2": f"inputs larger than L2 ({nl} distinct layers of checkpoints)"}


def run_reference(args):
    """The reference arm: the fp64 oracle on every host core (one process per
    core over independent rows), each bench step a bounded sample of the
    decode workload."""
    rows, per_step = 8, 10
    pool = OraclePool()
    t_total, toks = 0.0, 0
    try:
        for _ in range(args.warmup):
            pool.run(rows, per_step)
        for _ in range(args.steps):
            v, span = pool.run(rows, per_step)
            t_total += span
            toks += v * span
    finally:
        pool.close()
    value = toks / t_total
    sample = (f"{pool.n} processes x {rows} rows x 1 layer x {per_step} decode steps per bench "
              "step, fp64 numpy oracle, all processes started together")
    return {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * t_total / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference",
            "config": bench_config(args.layers, 1),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": pool.n, "kind": "oracle",
                             "sample": sample, "host_cores": os.cpu_count()},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


# ----------------------------------------------------------------- sweep
SWEEP = [  # (algo, B, L, T, state dtype, commit mode); decode when T == 1
    ("gdn", 1, 16, 1, "f32", "lazy"), ("gdn", 8, 16, 1, "f32", "lazy"),
    ("gdn", 64, 16, 1, "f32", "lazy"), ("gdn", 128, 16, 1, "f32", "lazy"),
    ("gdn", 256, 16, 1, "f32", "lazy"), ("gdn", 64, 32, 1, "f32", "lazy"),
    ("gdn", 64, 64, 1, "f32", "lazy"), ("gdn", 64, 16, 1, "bf16", "lazy"),
    ("gdn", 64, 16, 3, "f32", "lazy"), ("gdn", 128, 16, 8, "f32", "lazy"),
    ("gdn", 128, 16, 8, "bf16", "fold_every"),
    ("kda", 64, 32, 1, "f32", "lazy"), ("kda", 64, 32, 1, "bf16", "lazy"),
    ("kda", 64, 32, 3, "f32", "lazy"),
]


# the full throughput grid: GDN and KDA x batch x ring length x window width x
# checkpoint dtype, lazy commit
GRID = [(algo, B, L, T, st, "lazy") for algo in ("gdn", "kda") for st in ("f32", "bf16")
        for L in (16, 32, 64) for T in (1, 3, 8) for B in (1, 8, 64, 128, 256)]


def sweep_point(torch, dev, algo, B, L, T, state_dtype, mode, steps, warmup, peak, plan="auto"):
    """Steady-state decode (T = 1) or verify + commit (T > 1) over enough
    stacked layers that the checkpoints exceed L2; per-layer time from CUDA
    events around CUDA-graph replays, algorithmic bytes of the replay launches
    from the rows' cursor trajectory (the commit's own work is timed with them)."""
    from linear_attention_state_rssm_gb300.store import ReplayStore
    HK, HV, dk, dv = (16, 32, 128, 128) if algo == "gdn" else (32, 32, 128, 128)
    n_g = 1 if algo == "gdn" else dk
    s_state = ESZ[state_dtype]
    layer_state = B * HV * dk * dv * s_state
    nl = int(min(256, max(4, -(-(512 << 20) // layer_state))))
    gen = torch.Generator(device=dev)
    gen.manual_seed(5000 + B + 7 * T + L)
    st = ReplayStore(algo, nl, B, HK, HV, dk, dv, L, T, "bf16", state_dtype, "f16", "f32", mode,
                     device=dev)
    if algo == "gdn" and L <= 16:
        st.rssm_set_plan(plan)
    for layer in range(nl):
        st.state[layer].normal_(0.0, 0.1, generator=gen)
    cur0 = [r % L for r in range(B)]  # staggered rows, as in steady serving
    st.cursor.copy_(torch.tensor(cur0, dtype=torch.int32))
    n = nl * B * T
    nrm = torch.nn.functional.normalize
    q = nrm(torch.randn(n, HK, dk, generator=gen, device=dev), dim=-1).to(torch.bfloat16)
    k = nrm(torch.randn(n, HK, dk, generator=gen, device=dev), dim=-1).to(torch.bfloat16)
    v = torch.randn(n, HV, dv, generator=gen, device=dev).to(torch.bfloat16)
    beta = torch.sigmoid(torch.randn(n, HV, generator=gen, device=dev))
    gshape = (n, HV) if algo == "gdn" else (n, HV, dk)
    g = -torch.nn.functional.softplus(torch.randn(gshape, generator=gen, device=dev))
    out = torch.empty(n, HV, dv, dtype=torch.bfloat16, device=dev)
    slot = torch.arange(B, dtype=torch.int32, device=dev)
    per = B * T
    acc_all = torch.randint(0, T + 1, (warmup + steps, B), generator=gen, device=dev,
                            dtype=torch.int32)
    acc_cur = torch.empty(B, dtype=torch.int32, device=dev)

    def lv(layer):
        a, b = layer * per, (layer + 1) * per
        return q[a:b], k[a:b], v[a:b], beta[a:b], g[a:b]

    def step():
        for layer in range(nl):
            if T == 1:
                st.rssm_decode(layer, *lv(layer), slot, out[layer * per:(layer + 1) * per],
                               advance_cursor=layer == nl - 1)
            else:
                st.rssm_verify(layer, *lv(layer), slot, T, out[layer * per:(layer + 1) * per])
        if T > 1:
            st.rssm_commit(slot, acc_cur, T)

    cap = torch.cuda.Stream(device=dev)
    cap.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cap):
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=cap):
            step()
    torch.cuda.current_stream().wait_stream(cap)
    # host copy of the cursor trajectory for the byte count (capture ran nothing)
    cur = list(cur0)
    acc_h = acc_all.cpu().tolist()
    total_bytes = 0
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for i in range(warmup + steps):
        if i == warmup:
            torch.cuda.synchronize()
            e0.record()
        acc_cur.copy_(acc_all[i])
        graph.replay()
        a_row = [1] * B if T == 1 else acc_h[i]
        for r in range(B):
            c = cur[r]
            nxt, fold = advance(c, T, L, a_row[r])
            if i >= warmup:
                total_bytes += nl * row_bytes(c, T, fold, HK, HV, dk, dv, s_state, 2, 2, 4, n_g)
            cur[r] = 0 if (T > 1 and mode == "fold_every") else nxt
    e1.record()
    torch.cuda.synchronize()
    ms_layer = e0.elapsed_time(e1) / (steps * nl)
    gbs = total_bytes / (steps * nl) / (ms_layer / 1e3) / 1e9
    err = st.rssm_get_device_error()
    del graph, st, q, k, v, beta, g, out
    torch.cuda.empty_cache()
    return {"algo": algo, "batch": B, "L": L, "T": T, "state_dtype": state_dtype,
            "commit_mode": mode, "layers": nl, "ms_per_layer": ms_layer, "plan": plan,
            "replayed_tokens_per_s_per_layer": B * T / (ms_layer / 1e3),
            "replay_gbs": gbs, "frac_of_hbm_peak": gbs / peak, "device_error_word": err}


def grid_summary():
    """The full throughput grid (GRID: GDN and KDA x batch x ring length x
    window x checkpoint dtype, lazy commit), five timed steps after three
    warm-up steps per point, as compact rows for the bench line."""
    import torch
    dev = torch.device("cuda", 0)
    peak, peak_kind = peaks()
    rows, err = [], 0
    for pt in GRID:
        p = sweep_point(torch, dev, *pt, steps=5, warmup=3, peak=peak)
        rows.append([p["algo"], p["batch"], p["L"], p["T"], p["state_dtype"],
                     round(p["ms_per_layer"] * 1e3, 2), round(p["frac_of_hbm_peak"], 4)])
        err |= p["device_error_word"]
    return {"columns": ["algo", "batch", "L", "T", "state_dtype", "us_per_layer",
                        "frac_of_hbm_peak"],
            "rows": rows, "commit_mode": "lazy", "steps": 5, "warmup": 3, "peak_gbs": peak,
            "peak_kind": peak_kind, "device_error_word": err,
            "note": "per-layer time includes the step's cursor advance or commit; bytes count "
                    "the replay launches"}


def run_sweep(args):
    """--sweep: a steady-state grid of decode and verify launches over batch,
    ring length, window width, state dtype, and GDN and KDA heads."""
    import torch
    from linear_attention_state_rssm_gb300 import build as _build
    _build.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    peak, peak_kind = peaks()
    pts = []
    for pt in (GRID if args.grid == "full" else SWEEP):
        pts.append(sweep_point(torch, dev, *pt, steps=args.steps, warmup=args.warmup, peak=peak,
                               plan=args.plan))
        print(json.dumps(pts[-1]), file=sys.stderr, flush=True)  # progress
    return {"sweep": pts, "peak_gbs": peak, "peak_kind": peak_kind,
            "note": "per-layer time includes the step's cursor advance (decode) or commit "
                    "(verify); bytes count the replay launches only"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--layers", type=int, default=WL["layers"])
    ap.add_argument("--no-verify", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-native", action="store_true",
                    help="skip the native fused-recurrent decode comparison line")
    ap.add_argument("--no-prefill", action="store_true", help="skip the replay prefill line")
    ap.add_argument("--no-conv", action="store_true", help="skip the conv window line")
    ap.add_argument("--no-kda", action="store_true", help="skip the KDA decode+verify line")
    ap.add_argument("--no-grid", action="store_true",
                    help="skip the full throughput grid summary (N = 1 only)")
    ap.add_argument("--plan", default="auto", choices=["auto", "rows", "pipe", "tc"],
                    help="kernel family for GDN decode/verify (rssm_set_plan)")
    ap.add_argument("--sweep", action="store_true",
                    help="print the steady-state grid (batch, L, T, state dtype, GDN/KDA)")
    ap.add_argument("--grid", default="short", choices=["short", "full"],
                    help="--sweep over the short list or the full batch x L x T x dtype grid")
    ap.add_argument("--prefill-prompts", type=int, default=PREFILL["prompts"])
    ap.add_argument("--prefill-tokens", type=int, default=PREFILL["tokens"])
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.sweep:
        print(json.dumps(run_sweep(args)), flush=True)
        return

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return

    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    res = run_ours(args, rank, world, local_rank)
    if rank == 0:
        if world == 1 and not args.no_grid:
            try:
                res["grid"] = grid_summary()
            except Exception as e:  # the headline line stands on its own
                res["grid"] = {"error": f"{type(e).__name__}: {e}"}
        if world == 1 and not args.no_cpu_baseline:
            res["cpu_baseline"] = cpu_baseline()
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
