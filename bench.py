"""Benchmark of the CSA2 decode step on GB300.

Workload (default): one decoder CSA2 group of 4 layers (1 Full + 3 Reuse), batch 64, context
131072 per sequence, compression ratio 1, FP4 main KV (E2M1 + E4M3 per 16 channels), 128-token
bf16 window per layer, indexer Q 4x128 bf16 + fp32 weights, main Q 16x512 bf16, Top-512.
A step = append of the new token (FP4 quantise + indexer-K row) -> indexer scores over all
131072 keys -> exact Top-512 -> four layers of split-KV sparse attention (+ combine), issued as
one `csa2_group_step` C-ABI call.  Inputs are synthetic N(0, 1) (torch's CUDA generator, seed 0)
and resident in HBM; the 2.1 GB indexer-K scan per step is larger than L2, so no flush is needed.

Prints one JSON line.  `value` = decode tokens/s over all ranks (64 sequences per GPU per step),
`e2e` = the same through host buffers (per-step H2D of the step's inputs from pinned memory,
D2H of the four layers' outputs, double-buffered so that they overlap the neighbouring steps),
`roofline` = the indexer-score kernel against the measured HBM
copy bandwidth, `cpu_baseline` = the oracle on the host cores on a bounded sample.
`--impl reference` times the oracle (the CPU reference of this method) instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

B_PER_GPU, T_CTX, N_LAYERS, K_SEL, W_WIN = 64, 131072, 4, 512, 128
WORKLOAD = "csa2_decode_group_1full_3reuse_b64_t131072"
METRIC = "CSA2 decode tokens/s and KV HBM GB/s at 128K ctx; % of GB300 HBM roofline"
# algorithmic bytes per sequence per step: indexer-K scan + 4 layers x (512 FP4 rows of 288 B +
# 128 bf16 window rows of 1 KiB + Q and O of 16 KiB each) + the append (bf16 row in, FP4 out, KI row)
BYTES_KI_PER_SEQ = T_CTX * 128 * 2
BYTES_ATTN_PER_SEQ_LAYER = K_SEL * 288 + W_WIN * 1024 + 2 * 16 * 512 * 2
BYTES_APPEND_PER_SEQ = 512 * 2 + 288 + 2 * 128 * 2
BYTES_PER_SEQ = BYTES_KI_PER_SEQ + N_LAYERS * BYTES_ATTN_PER_SEQ_LAYER + BYTES_APPEND_PER_SEQ
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "index_score_decode_b64_t131072.md")
SCORE_SRC = os.path.join(ROOT, "compressed_sparse_attention_step_gb300", "csrc", "index_score.cu")


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def profiled_traffic():
    """Per-launch DRAM bytes of the score kernel from the committed ncu summary, if the kernel
    source is unchanged since the capture (its sha256 is recorded in the summary)."""
    try:
        txt = open(PROFILE_SUMMARY).read()
        src = hashlib.sha256(open(SCORE_SRC, "rb").read()).hexdigest()[:16]
        vals = {}
        for line in txt.splitlines():
            if ":" in line:
                k, v = line.split(":", 1)
                vals[k.strip().strip("`- ")] = v.strip().strip("`")
        if vals.get("kernel_source_sha256") != src:
            return None
        return int(float(vals["traffic_bytes_per_launch"]))
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi sampling in the background; samples are time-stamped on arrival."""

    QUERY = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
             "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
             "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.samples = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(index), f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.th = threading.Thread(target=self._read, daemon=True)
            self.th.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [x.strip() for x in line.split(",")]))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0, t1):
        inside = [s for (t, s) in self.samples if t0 <= t <= t1]
        near = inside or [s for (t, s) in self.samples if t0 - 0.5 <= t <= t1 + 0.5]
        if not near:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(s[0]) for s in near if num(s[0]) is not None]
        mx = [num(s[1]) for s in near if num(s[1]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for s in near for i in range(4) if len(s) > 4 + i and s[4 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(inside), "samples_near": len(near),
                "power_w_max": max((num(s[2]) or 0.0) for s in near)}


# ----------------------------------------------------------------------------------------------
# oracle (CPU baseline / reference arm)
# ----------------------------------------------------------------------------------------------
def oracle_inputs(n_seq, seed=0):
    """A bounded sample of the workload for the oracle: n_seq sequences at the full context.
    Indexer keys, queries, weights and windows are the seeded N(0, 1) draws; the FP4 cache rows
    are random code bytes with scales in the range N(0, 1) rows quantise to (only the 512
    selected rows per layer are read, so their values do not change the work)."""
    import csa2_synth as syn
    g = np.random.default_rng(seed)
    codes = g.integers(0, 256, (n_seq, T_CTX, 256), dtype=np.uint8)
    scales = g.integers(0x2C, 0x3C, (n_seq, T_CTX, 32), dtype=np.uint8)
    KI = np.stack([syn.normal_bf16(seed, syn.T_KI, b, (T_CTX, 128)) for b in range(n_seq)])
    L = N_LAYERS
    q = np.stack([np.stack([syn.normal_bf16(seed, syn.T_Q + l, b, (1, 16, 512)) for b in range(n_seq)]) for l in range(L)])
    qI = np.stack([np.stack([syn.normal_bf16(seed, syn.T_QI + l, b, (1, 4, 128)) for b in range(n_seq)]) for l in range(L)])
    w = np.stack([np.stack([syn.normal_f32(seed, syn.T_W + l, b, (1, 4)) for b in range(n_seq)]) for l in range(L)])
    swa = np.stack([np.stack([syn.normal_bf16(seed, syn.T_SWA + l, b, (W_WIN, 512)) for b in range(n_seq)]) for l in range(L)])
    return codes, scales, KI, q, qI, w, swa


def oracle_step(orc, inp, threads):
    codes, scales, KI, q, qI, w, swa = inp
    n = codes.shape[0]
    orc.group_step([0, 2, 2, 2], [T_CTX] * n, codes, scales, KI, q, qI, w, swa, np.full(n, W_WIN, np.int32),
                   threads=threads)


def cpu_threads():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def run_reference(args, rank, world):
    """The oracle as it stands, on the host cores, same workload and metric (bounded sample)."""
    if rank != 0:
        return
    import oracle as orc
    orc.build()
    threads = cpu_threads()
    n_seq = min(64, 2 * threads)         # two sequences per host thread per step
    inp = oracle_inputs(n_seq)
    for _ in range(min(args.warmup, 1)):
        oracle_step(orc, inp, threads)
    budget = 150.0
    times = []
    t_start = time.time()
    for i in range(args.steps):
        t0 = time.perf_counter()
        oracle_step(orc, inp, threads)
        times.append(time.perf_counter() - t0)
        if time.time() - t_start + times[-1] > budget:
            break
    ms = 1e3 * statistics.mean(times)
    val = n_seq / (ms / 1e3)
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": len(times), "steps_requested": args.steps, "warmup": min(args.warmup, 1),
            "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32/f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "global_batch": n_seq, "seq_len": T_CTX, "parallelism": "host threads",
                       "l2": "n/a (CPU)"},
            "cpu_baseline": {"value": val, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                             "sample": f"{n_seq} sequences x {T_CTX} context, 4 layers (1 Full + 3 Reuse) per step"},
            "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------------------------
# GPU arm
# ----------------------------------------------------------------------------------------------
def build_workload(torch, c, syn, dev):
    B, T, L = B_PER_GPU, T_CTX, N_LAYERS
    seed = syn.SEEDS["decode_group_1f3r_b64_t131072"]
    codes = torch.empty((B, T, 256), dtype=torch.uint8, device=dev)
    scales = torch.empty((B, T, 32), dtype=torch.uint8, device=dev)
    for b in range(B):   # the library's own quantiser fills the FP4 cache, one sequence at a time
        kv = syn.device_normal_bf16((1, T, 512), seed, syn.T_KV * 1000 + b, device=dev)
        c.csa2_fp4_quantize_append(kv, codes[b:b + 1], scales[b:b + 1])
        del kv
    KI = syn.device_normal_bf16((B, T, 128), seed, syn.T_KI * 1000, device=dev)
    q = [syn.device_normal_bf16((B, 1, 16, 512), seed, syn.T_Q + l, device=dev) for l in range(L)]
    qI = [syn.device_normal_bf16((B, 1, 4, 128), seed, syn.T_QI + l, device=dev) for l in range(L)]
    w = [syn.device_normal_bf16((B, 1, 4), seed, syn.T_W + l, device=dev).float() for l in range(L)]
    swa = [syn.device_normal_bf16((B, W_WIN, 512), seed, syn.T_SWA + l, device=dev) for l in range(L)]
    kv_new = syn.device_normal_bf16((B, 1, 512), seed, syn.T_KV_NEW, device=dev)
    ki_new = syn.device_normal_bf16((B, 1, 128), seed, syn.T_KI_NEW, device=dev)
    lens = torch.full((B,), T, dtype=torch.int32, device=dev)
    swa_len = torch.full((B,), W_WIN, dtype=torch.int32, device=dev)
    out = [torch.empty((B, 1, 16, 512), dtype=torch.bfloat16, device=dev) for _ in range(L)]
    idx = [torch.empty((B, K_SEL), dtype=torch.int32, device=dev), None, None, None]
    ws = torch.empty(c.group_workspace_size(B, 1, T, K_SEL, W_WIN, n_split=N_SPLIT), dtype=torch.uint8, device=dev)
    return dict(codes=codes, scales=scales, KI=KI, q=q, qI=qI, w=w, swa=swa, kv_new=kv_new, ki_new=ki_new,
                lens=lens, swa_len=swa_len, out=out, idx=idx, ws=ws)


N_SPLIT = 0   # attention split-KV factor (0: the library's choice)
SCORE_EVERY = 4  # timed steps per step whose score kernel is bracketed by events


def make_desc(c, wl, events=None, q=None, qI=None, w=None, kv_new=None, ki_new=None, out=None):
    return c.make_group_desc(
        [c.MODE_FULL, c.MODE_REUSE, c.MODE_REUSE, c.MODE_REUSE], B=B_PER_GPU, Nq=1, cap=T_CTX, lens=wl["lens"],
        codes=wl["codes"], scales=wl["scales"], KI=wl["KI"], q=q or wl["q"], qI=qI or wl["qI"], w=w or wl["w"],
        swa=wl["swa"], swa_len=wl["swa_len"], out=out or wl["out"], idx=wl["idx"], K=K_SEL, W=W_WIN,
        kv_new=kv_new if kv_new is not None else wl["kv_new"], ki_new=ki_new if ki_new is not None else wl["ki_new"],
        events=events, n_split=N_SPLIT)


def launches_per_step(c):
    # the append (quantise the new KV row, copy the new indexer-K row: one launch) + score + Top-K
    # (row histogram, filter, select) + one attention launch for the four layers (they attend the
    # same selected rows; split partials are merged inside that launch)
    return 6


def max_over_ranks(torch, dist, value, world, device):
    """The largest of a rank's `value` (a timed region in ms) over all ranks; every rank gets it."""
    if world <= 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def throughput(units_per_rank, world, ms_per_step):
    """Whole-job rate: the units all ranks processed in one step over the (max-over-ranks) step time."""
    return units_per_rank * world / (ms_per_step / 1e3)


def run_gpu(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    import csa2_synth as syn
    import compressed_sparse_attention_step_gb300 as c
    from compressed_sparse_attention_step_gb300 import _build

    if not os.path.exists(_build.LIB):
        raise RuntimeError("libcsa2.so is not built: run `python -c 'import __graft_entry__ as g; g.build()'`")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    c.lib()
    wl = build_workload(torch, c, syn, dev)
    stream = torch.cuda.current_stream()
    K, Wm = args.steps, args.warmup

    def barrier():
        if world > 1:
            dist.barrier()

    # ---- device-resident step --------------------------------------------------------------------
    # The score kernel's duration is taken on every SCORE_EVERY-th timed step: the event pair the
    # library records around the scan breaks the overlap of programmatic launches on both sides of
    # it, so the other steps run without it.
    n_scored = (K + SCORE_EVERY - 1) // SCORE_EVERY
    ev_pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_scored)]
    for a, b in ev_pairs:   # materialise the event handles
        a.record()
        b.record()
    plain = make_desc(c, wl)
    descs = [make_desc(c, wl, events=ev_pairs[i // SCORE_EVERY]) if i % SCORE_EVERY == 0 else plain for i in range(K)]
    for _ in range(Wm):
        c.csa2_group_step(plain, wl["ws"])
    torch.cuda.synchronize()
    sampler = ClockSampler(local_rank) if rank == 0 else None
    time.sleep(0.1)
    barrier()
    torch.cuda.synchronize()
    t_wall0 = time.time()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(K):
        c.csa2_group_step(descs[i], wl["ws"])
    e1.record()
    torch.cuda.synchronize()
    t_wall1 = time.time()
    barrier()
    ms_total = e0.elapsed_time(e1)
    score_ms = [a.elapsed_time(b) for a, b in ev_pairs]
    clocks = sampler.summary(t_wall0, t_wall1) if sampler else None
    ms_total = max_over_ranks(torch, dist, ms_total, world, dev)

    # ---- end to end through host buffers ---------------------------------------------------------
    # Every step copies its inputs from pinned host memory (one packed block: the 4 layers' Q, the
    # Full layer's qI and w, the new KV and KI rows) and reads the 4 layers' outputs back (one
    # packed block).  Two sets of device buffers let step i+1's upload and step i-1's read-back run
    # on their own streams while step i computes, as a serving loop would; the timed region runs
    # from before the first upload to the end of the last read-back.
    L = N_LAYERS
    in_src = list(wl["q"]) + [wl["qI"][0], wl["w"][0], wl["kv_new"], wl["ki_new"]]
    offs, total_in = [], 0
    for x in in_src:
        offs.append(total_in)
        total_in += (x.numel() * x.element_size() + 255) // 256 * 256
    h_in = torch.empty(total_in, dtype=torch.uint8).pin_memory()
    for x, o in zip(in_src, offs):
        h_in[o:o + x.numel() * x.element_size()].copy_(x.contiguous().view(-1).view(torch.uint8).cpu())
    d_in = [torch.empty(total_in, dtype=torch.uint8, device=dev) for _ in range(2)]
    d_out = [torch.empty((L,) + tuple(wl["out"][0].shape), dtype=torch.bfloat16, device=dev) for _ in range(2)]
    h_out = [torch.empty(d_out[0].shape, dtype=torch.bfloat16).pin_memory() for _ in range(2)]

    def views(buf):
        return [buf[o:o + x.numel() * x.element_size()].view(x.dtype).view(x.shape) for x, o in zip(in_src, offs)]

    e2e_descs = []
    for s in range(2):
        v = views(d_in[s])
        e2e_descs.append(make_desc(c, wl, q=v[:L], qI=[v[L], None, None, None], w=[v[L + 1], None, None, None],
                                   kv_new=v[L + 2], ki_new=v[L + 3], out=[d_out[s][l] for l in range(L)]))
    h2d = total_in
    d2h = h_out[0].numel() * h_out[0].element_size()
    comp = torch.cuda.current_stream()
    s_up, s_down = torch.cuda.Stream(), torch.cuda.Stream()
    ev_up = [torch.cuda.Event() for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_down = [torch.cuda.Event() for _ in range(2)]

    def e2e_step(i):
        s = i & 1
        with torch.cuda.stream(s_up):
            if i >= 2:
                s_up.wait_event(ev_comp[s])     # step i-2 has consumed this input set
            d_in[s].copy_(h_in, non_blocking=True)
            ev_up[s].record(s_up)
        comp.wait_event(ev_up[s])
        if i >= 2:
            comp.wait_event(ev_down[s])         # step i-2's outputs in this set have been read back
        c.csa2_group_step(e2e_descs[s], wl["ws"])
        ev_comp[s].record(comp)
        with torch.cuda.stream(s_down):
            s_down.wait_event(ev_comp[s])
            h_out[s].copy_(d_out[s], non_blocking=True)
            ev_down[s].record(s_down)

    def e2e_run(n):
        start = torch.cuda.Event()
        start.record(comp)
        s_up.wait_event(start)
        for i in range(n):
            e2e_step(i)
        for s in range(min(n, 2)):
            comp.wait_event(ev_down[s])

    e2e_run(max(Wm, 2))
    torch.cuda.synchronize()
    barrier()
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record()
    e2e_run(K)
    f1.record()
    torch.cuda.synchronize()
    barrier()
    e2e_ms = f0.elapsed_time(f1)
    e2e_ms = max_over_ranks(torch, dist, e2e_ms, world, dev)
    # the read-back holds the device outputs of the last step
    assert torch.equal(h_out[(K - 1) & 1].to(dev), d_out[(K - 1) & 1])
    if sampler:
        sampler.stop()
    if rank != 0:
        return

    ms_step = ms_total / K
    tokens = B_PER_GPU * world
    value = throughput(B_PER_GPU, world, ms_step)
    kv_gbs = BYTES_PER_SEQ * B_PER_GPU * world / (ms_step / 1e3) / 1e9
    peak, peak_kind = peaks()
    score_avg = statistics.mean(score_ms)
    score_bytes = B_PER_GPU * BYTES_KI_PER_SEQ
    achieved = score_bytes / (score_avg / 1e3) / 1e9
    traffic = profiled_traffic()

    # ---- CPU baseline: the oracle on a bounded sample --------------------------------------------
    cpu = None
    if not args.no_cpu_baseline:
        import oracle as orc
        orc.build()
        threads = cpu_threads()
        n_seq = min(64, 2 * threads)
        inp = oracle_inputs(n_seq)
        times = []
        while not times or (sum(times) * threads < 10.0 and len(times) < 20):   # ~10 s of CPU work
            t0 = time.perf_counter()
            oracle_step(orc, inp, threads)
            times.append(time.perf_counter() - t0)
        dt = statistics.mean(times)
        cpu = {"value": n_seq / dt, "unit": "tokens/s", "cores": threads, "kind": "oracle",
               "sample": f"{len(times)} steps over {n_seq} of the 64 sequences at full context ({T_CTX}), "
                         f"1 Full + 3 Reuse, {dt:.2f} s wall per step on {threads} threads"}

    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K, "warmup": Wm,
        "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16/fp4 in, fp32 accumulate", "data": "synthetic",
        "config": {"workload": WORKLOAD, "global_batch": tokens, "seq_len": T_CTX, "parallelism": f"replicas x{world}",
                   "layers": "1 Full + 3 Reuse", "top_k": K_SEL, "window": W_WIN,
                   "l2": "inputs larger than L2 (2.1 GB indexer-K scan per step)"},
        "kv_gbs": kv_gbs, "hbm_frac_step": kv_gbs / peak, "bytes_per_step": BYTES_PER_SEQ * B_PER_GPU * world,
        "roofline": {"kernel": "index_score_stream_kernel", "bound": "hbm", "achieved": achieved, "peak": peak,
                     "unit": "GB/s", "frac": achieved / peak, "peak_kind": f"{peak_kind} (hbm copy)",
                     "traffic": traffic, "algorithmic_bytes": score_bytes, "avg_launch_ms": score_avg,
                     "launches_timed": len(score_ms), "timed_every": SCORE_EVERY},
        "e2e": {"value": throughput(B_PER_GPU, world, e2e_ms / K), "unit": "tokens/s", "h2d_bytes_per_step": h2d * world,
                "d2h_bytes_per_step": d2h * world, "ms_per_step": e2e_ms / K,
                "copies": "one packed H2D and one packed D2H per step, double-buffered on their own streams "
                          "(step i+1's upload and step i-1's read-back overlap step i)"},
        "gpu_launches": launches_per_step(c) * K,
        "clocks": clocks,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------------------------
# other workloads (`--workload`): the 20-layer decoder stack and the encoder prefill chunk
# ----------------------------------------------------------------------------------------------
def bf16_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return 1900.0, "fallback"


def time_steps(torch, fn, K, Wm):
    for _ in range(Wm):
        fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(K):
        fn()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / K


def run_stack20(args):
    """One token through the 20-layer decoder: 5 groups of 4 (Full + 3 Reuse, then 4 x Reindex +
    3 Reuse) over one cache, B = 64, T = 131072; one csa2_stack_step per step."""
    import torch

    import csa2_synth as syn
    import compressed_sparse_attention_step_gb300 as c
    dev = torch.device("cuda")
    wl = build_workload(torch, c, syn, dev)
    seed = syn.SEEDS["decode_group_1f3r_b64_t131072"]
    B, T = B_PER_GPU, T_CTX
    descs = [make_desc(c, wl)]
    keep = []
    for g in range(1, 5):
        L0 = 4 * g
        q = [syn.device_normal_bf16((B, 1, 16, 512), seed, syn.T_Q + L0 + l, device=dev) for l in range(4)]
        qI = [syn.device_normal_bf16((B, 1, 4, 128), seed, syn.T_QI + L0, device=dev), None, None, None]
        w = [syn.device_normal_bf16((B, 1, 4), seed, syn.T_W + L0, device=dev).float(), None, None, None]
        swa = [syn.device_normal_bf16((B, W_WIN, 512), seed, syn.T_SWA + L0 + l, device=dev) for l in range(4)]
        out = [torch.empty((B, 1, 16, 512), dtype=torch.bfloat16, device=dev) for _ in range(4)]
        idx = [torch.empty((B, K_SEL), dtype=torch.int32, device=dev), None, None, None]
        keep += [q, qI, w, swa, out, idx]
        descs.append(c.make_group_desc(
            [c.MODE_REINDEX, c.MODE_REUSE, c.MODE_REUSE, c.MODE_REUSE], B=B, Nq=1, cap=T, lens=wl["lens"],
            codes=wl["codes"], scales=wl["scales"], KI=wl["KI"], q=q, qI=qI, w=w, swa=swa, swa_len=wl["swa_len"],
            out=out, idx=idx, K=K_SEL, W=W_WIN))
    ms = time_steps(torch, lambda: c.csa2_stack_step(descs, wl["ws"]), args.steps, max(args.warmup, 3))
    # algorithmic bytes: 5 indexer-K scans + 20 layers of attention + the append, per sequence
    per_seq = 5 * BYTES_KI_PER_SEQ + 20 * BYTES_ATTN_PER_SEQ_LAYER + BYTES_APPEND_PER_SEQ
    peak, kind = peaks()
    gbs = per_seq * B / (ms / 1e3) / 1e9
    return {"metric": "CSA2 20-layer decoder stack tokens/s at 128K ctx", "value": B / (ms / 1e3),
            "unit": "tokens/s", "ms_per_step": ms, "higher_is_better": True,
            "config": {"workload": "csa2_decoder_stack_5x4_b64_t131072", "global_batch": B, "seq_len": T,
                       "layers": "Full+3 Reuse, then 4 x (Reindex + 3 Reuse)", "top_k": K_SEL, "window": W_WIN},
            "kv_gbs": gbs, "hbm_frac_step": gbs / peak, "peak_kind": f"{kind} (hbm copy)",
            # group 1: append + score + Top-K (3) + attention; groups 2-5: score + Top-K (3) + attention
            "gpu_launches": (6 + 4 * 5) * args.steps}


def run_prefill(args):
    """The encoder prefill chunk: 2048 queries at the end of 262144 tokens (131072 compressed
    entries, ratio 2), 1 Full + 5 Reuse, Top-512, 128-token window; one csa2_group_step per step."""
    import torch

    import csa2_synth as syn
    import compressed_sparse_attention_step_gb300 as c
    dev = torch.device("cuda")
    seed = syn.SEEDS["prefill_group_1f5r_ratio2_q2048"]
    T, Nq, L = 131072, 2048, 6
    codes = torch.empty((1, T, 256), dtype=torch.uint8, device=dev)
    scales = torch.empty((1, T, 32), dtype=torch.uint8, device=dev)
    kv = syn.device_normal_bf16((1, T, 512), seed, syn.T_KV * 1000, device=dev)
    c.csa2_fp4_quantize_append(kv, codes, scales)
    del kv
    KI = syn.device_normal_bf16((1, T, 128), seed, syn.T_KI * 1000, device=dev)
    q = [syn.device_normal_bf16((1, Nq, 16, 512), seed, syn.T_Q + l, device=dev) for l in range(L)]
    qI = [syn.device_normal_bf16((1, Nq, 4, 128), seed, syn.T_QI, device=dev)] + [None] * (L - 1)
    w = [syn.device_normal_bf16((1, Nq, 4), seed, syn.T_W, device=dev).float()] + [None] * (L - 1)
    swa = [syn.device_normal_bf16((1, W_WIN - 1 + Nq, 512), seed, syn.T_SWA + l, device=dev) for l in range(L)]
    out = [torch.empty((1, Nq, 16, 512), dtype=torch.bfloat16, device=dev) for _ in range(L)]
    idx = [torch.empty((Nq, K_SEL), dtype=torch.int32, device=dev)] + [None] * (L - 1)
    lens = torch.tensor([T], dtype=torch.int32, device=dev)
    swa_len = torch.tensor([W_WIN - 1 + Nq], dtype=torch.int32, device=dev)
    q_pos = torch.arange(2 * T - Nq, 2 * T, dtype=torch.int32, device=dev)
    d = c.make_group_desc([c.MODE_FULL] + [c.MODE_REUSE] * (L - 1), B=1, Nq=Nq, cap=T, lens=lens, codes=codes,
                          scales=scales, KI=KI, q=q, qI=qI, w=w, swa=swa, swa_len=swa_len, out=out, idx=idx,
                          K=K_SEL, W=W_WIN, ratio=2, q_pos=q_pos)
    ws = torch.empty(c.group_workspace_size(1, Nq, T, K_SEL, W_WIN), dtype=torch.uint8, device=dev)
    ms = time_steps(torch, lambda: c.csa2_group_step(d, ws), args.steps, max(args.warmup, 3))
    # dense work: the indexer contraction over each query's visible entries (1024 flop per pair)
    # and 6 layers of attention (2 x 16 heads x 512 x 640 rows x 2 flop per query)
    vis = (np.arange(2 * T - Nq, 2 * T) + 1) // 2
    gflop = (float(vis.sum()) * 1024 + L * Nq * 2 * 16 * 512 * (K_SEL + W_WIN) * 2) / 1e9
    peak, kind = bf16_peak()
    tflops = gflop / ms
    return {"metric": "CSA2 encoder prefill chunk queries/s (2048 q x 131072 entries, 6 layers)",
            "value": Nq / (ms / 1e3), "unit": "queries/s", "ms_per_step": ms, "higher_is_better": True,
            "config": {"workload": "csa2_prefill_1f5r_ratio2_q2048_t131072", "global_batch": Nq, "seq_len": 2 * T,
                       "layers": "1 Full + 5 Reuse", "top_k": K_SEL, "window": W_WIN},
            "dense_gflop_per_step": gflop, "tflops_step": tflops, "bf16_peak_tflops": peak,
            "frac_of_bf16_peak": tflops / peak, "peak_kind": kind,
            # key norms, two tensor-core passes, threshold, count, order, rescore/select, attention
            "gpu_launches": 8 * args.steps}


def run_fp8win(args):
    """The decode workload with 8-bit windows: the same group step, every layer's 128 window rows
    held as E4M3 bytes (csa2_fp8_quantize at set-up)."""
    import torch

    import csa2_synth as syn
    import compressed_sparse_attention_step_gb300 as c
    dev = torch.device("cuda")
    wl = build_workload(torch, c, syn, dev)
    swa8 = []
    for x in wl["swa"]:
        y = torch.empty(x.shape, dtype=torch.uint8, device=dev)
        c.csa2_fp8_quantize(x, y)
        swa8.append(y)
    d = c.make_group_desc(
        [c.MODE_FULL, c.MODE_REUSE, c.MODE_REUSE, c.MODE_REUSE], B=B_PER_GPU, Nq=1, cap=T_CTX, lens=wl["lens"],
        codes=wl["codes"], scales=wl["scales"], KI=wl["KI"], q=wl["q"], qI=wl["qI"], w=wl["w"], swa=swa8,
        swa_len=wl["swa_len"], out=wl["out"], idx=wl["idx"], K=K_SEL, W=W_WIN, kv_new=wl["kv_new"],
        ki_new=wl["ki_new"], swa_fp8=True)
    ms = time_steps(torch, lambda: c.csa2_group_step(d, wl["ws"]), args.steps, max(args.warmup, 3))
    per_seq = BYTES_PER_SEQ - N_LAYERS * W_WIN * 512   # window rows of 512 B instead of 1 KiB
    peak, kind = peaks()
    gbs = per_seq * B_PER_GPU / (ms / 1e3) / 1e9
    return {"metric": "CSA2 decode tokens/s at 128K ctx with 8-bit (E4M3) windows", "value": B_PER_GPU / (ms / 1e3),
            "unit": "tokens/s", "ms_per_step": ms, "higher_is_better": True,
            "config": {"workload": "csa2_decode_group_1full_3reuse_b64_t131072_fp8win", "global_batch": B_PER_GPU,
                       "seq_len": T_CTX, "layers": "1 Full + 3 Reuse", "top_k": K_SEL, "window": W_WIN,
                       "window_format": "E4M3, one byte per channel"},
            "kv_gbs": gbs, "hbm_frac_step": gbs / peak, "bytes_per_step": per_seq * B_PER_GPU,
            "peak_kind": f"{kind} (hbm copy)", "gpu_launches": launches_per_step(c) * args.steps}


def run_hier1m(args):
    """The hierarchical indexer at 1M context: batch 8, T = 2^20, ratio 1; Full (top 2048 blocks of 8
    by block key, then Top-512 in the 16384-position pool) + Reindex (the same pool, its own indexer
    Q) + 3 Reuse; each step appends the new token (refreshing the block it completes)."""
    import torch

    import csa2_synth as syn
    import compressed_sparse_attention_step_gb300 as c
    dev = torch.device("cuda")
    seed = syn.SEEDS["hier_decode_b8_t1m"]
    B, T, L, keep = 8, 1 << 20, 5, 2048
    codes = torch.empty((B, T, 256), dtype=torch.uint8, device=dev)
    scales = torch.empty((B, T, 32), dtype=torch.uint8, device=dev)
    for b in range(B):
        kv = syn.device_normal_bf16((1, T, 512), seed, syn.T_KV * 1000 + b, device=dev)
        c.csa2_fp4_quantize_append(kv, codes[b:b + 1], scales[b:b + 1])
        del kv
    KI = syn.device_normal_bf16((B, T, 128), seed, syn.T_KI * 1000, device=dev)
    lens = torch.full((B,), T, dtype=torch.int32, device=dev)
    block_keys = torch.empty((B, T // 8, 128), dtype=torch.bfloat16, device=dev)
    c.csa2_block_keys_build(KI, lens, block_keys)
    q = [syn.device_normal_bf16((B, 1, 16, 512), seed, syn.T_Q + l, device=dev) for l in range(L)]
    qI = [syn.device_normal_bf16((B, 1, 4, 128), seed, syn.T_QI + l, device=dev) if l < 2 else None for l in range(L)]
    w = [syn.device_normal_bf16((B, 1, 4), seed, syn.T_W + l, device=dev).float() if l < 2 else None for l in range(L)]
    swa = [syn.device_normal_bf16((B, W_WIN, 512), seed, syn.T_SWA + l, device=dev) for l in range(L)]
    out = [torch.empty((B, 1, 16, 512), dtype=torch.bfloat16, device=dev) for _ in range(L)]
    idx = [torch.empty((B, K_SEL), dtype=torch.int32, device=dev) if l < 2 else None for l in range(L)]
    swa_len = torch.full((B,), W_WIN, dtype=torch.int32, device=dev)
    pool = torch.empty((B, keep * 8), dtype=torch.int32, device=dev)
    pool_len = torch.empty((B,), dtype=torch.int32, device=dev)
    kv_new = syn.device_normal_bf16((B, 1, 512), seed, syn.T_KV_NEW, device=dev)
    ki_new = syn.device_normal_bf16((B, 1, 128), seed, syn.T_KI_NEW, device=dev)
    d = c.make_group_desc([c.MODE_FULL, c.MODE_REINDEX, c.MODE_REUSE, c.MODE_REUSE, c.MODE_REUSE], B=B, Nq=1, cap=T,
                          lens=lens, codes=codes, scales=scales, KI=KI, q=q, qI=qI, w=w, swa=swa, swa_len=swa_len,
                          out=out, idx=idx, K=K_SEL, W=W_WIN, hierarchical=True, keep=keep, block_keys=block_keys,
                          pool=pool, pool_len=pool_len, kv_new=kv_new, ki_new=ki_new)
    ws = torch.empty(c.group_workspace_size(B, 1, T, K_SEL, W_WIN, hierarchical=True, keep=keep), dtype=torch.uint8,
                     device=dev)
    ms = time_steps(torch, lambda: c.csa2_group_step(d, ws), args.steps, max(args.warmup, 3))
    # algorithmic bytes per sequence: the block-key scan, the pool's indexer keys for Full and Reindex,
    # five layers of attention, the append
    per_seq = (T // 8) * 256 + 2 * keep * 8 * 256 + L * BYTES_ATTN_PER_SEQ_LAYER + BYTES_APPEND_PER_SEQ
    peak, kind = peaks()
    gbs = per_seq * B / (ms / 1e3) / 1e9
    return {"metric": "CSA2 hierarchical decode tokens/s at 1M ctx", "value": B / (ms / 1e3), "unit": "tokens/s",
            "ms_per_step": ms, "higher_is_better": True,
            "config": {"workload": "csa2_hier_decode_full_reindex_3reuse_b8_t1m", "global_batch": B, "seq_len": T,
                       "layers": "Full + Reindex + 3 Reuse", "blocks_kept": keep, "pool": keep * 8, "top_k": K_SEL,
                       "window": W_WIN},
            "kv_gbs": gbs, "hbm_frac_step": gbs / peak, "bytes_per_step": per_seq * B, "peak_kind": f"{kind} (hbm copy)"}


def run_extra(args):
    import torch
    torch.cuda.set_device(0)
    fn = {"decoder_stack_20": run_stack20, "prefill_chunk": run_prefill,
          "decode_group_fp8win": run_fp8win, "hier_decode_1m": run_hier1m}[args.workload]
    line = fn(args)
    line.update({"n_gpus": 1, "steps": args.steps, "warmup": max(args.warmup, 3), "scaling": "weak",
                 "vs_baseline": None, "dtype": "bf16/fp4 in, fp32 accumulate", "data": "synthetic",
                 "cpu_baseline": None})
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--batch", type=int, default=64,
                    help="sequences per GPU (64 is the workload; smaller values are for profiling)")
    ap.add_argument("--n-split", type=int, default=0, help="force the attention split-KV factor (profiling)")
    ap.add_argument("--workload", default="decode_group",
                    choices=["decode_group", "decoder_stack_20", "prefill_chunk", "decode_group_fp8win",
                             "hier_decode_1m"],
                    help="decode_group (default): the headline line; the others print their own line on one GPU")
    args = ap.parse_args()
    global B_PER_GPU, N_SPLIT
    B_PER_GPU = args.batch
    N_SPLIT = args.n_split
    args.warmup = max(args.warmup, 3) if args.impl == "ours" else args.warmup
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if args.workload != "decode_group":
        if rank == 0:
            run_extra(args)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    run_gpu(args, rank, world, local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
