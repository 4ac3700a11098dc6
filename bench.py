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

`--workload` selects one of the other configurations, each printing its own line with a live
roofline of its dominant kernel and the oracle timed beside it on a bounded sample:
  full_layer_decode    one Full layer, batch 1, 4096 entries (L2 flushed before every step)
  fp4_roundtrip        FP4 quantise and dequantise of 64 x 8192 x 512 bf16 rows (1% outliers x20)
  prefill_chunk        2048 queries over 131072 entries (ratio 2), 1 Full + 5 Reuse
  hier_decode_1m       batch 8 at 2^20 entries, hierarchical pool, Full + Reindex + 3 Reuse
  decoder_stack_20     five groups of four layers over one 128K cache, batch 64
  decode_group_fp8win  the headline workload with 8-bit window rows
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
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
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")
CSRC = os.path.join(ROOT, "compressed_sparse_attention_step_gb300", "csrc")
NOMINAL_HBM_GBS = 8000.0   # GB300 HBM3e nominal bandwidth, for the fraction reported beside the measured one


def peaks():
    """HBM peak (GB/s) for the roofline: the measured copy bandwidth, else the fallback."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def kernel_body_hash(kernel):
    """sha256 (first 16 hex digits) of a kernel's source text, from `__global__` to the closing
    brace of its body, in the library source that defines it; None if not found."""
    for fn in sorted(os.listdir(CSRC)):
        if not fn.endswith(".cu"):
            continue
        src = open(os.path.join(CSRC, fn)).read()
        m = re.search(r"__global__[^;{]*?\b" + re.escape(kernel) + r"\s*\(", src)
        if not m:
            continue
        depth = 0
        for j in range(src.index("{", m.end()), len(src)):
            if src[j] == "{":
                depth += 1
            elif src[j] == "}":
                depth -= 1
                if depth == 0:
                    return hashlib.sha256(src[m.start():j + 1].encode()).hexdigest()[:16]
    return None


def profiled_traffic(kernel, workload):
    """DRAM bytes (read + write) of one launch of `kernel` in `workload`, from the ncu capture
    recorded in profiles/traffic.json; None when there is none or when the kernel's body changed
    since that capture."""
    try:
        with open(TRAFFIC_FILE) as f:
            e = json.load(f)[kernel][workload]
    except Exception:
        return None
    if e.get("kernel_sha256") != kernel_body_hash(kernel):
        return None
    return int(e["bytes_per_launch"])


def roofline(kernel, workload, bound, work, avg_ms, launches, peak, peak_kind):
    """The roofline object of a kernel: `work` algorithmic bytes (hbm) or flops (tensor) per launch
    over its average event-timed launch duration, against the measured peak."""
    if bound == "hbm":
        achieved, unit = work / (avg_ms / 1e3) / 1e9, "GB/s"
    else:
        achieved, unit = work / (avg_ms / 1e3) / 1e12, "TFLOP/s"
    r = {"kernel": kernel, "bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
         "frac": achieved / peak, "peak_kind": peak_kind, "traffic": profiled_traffic(kernel, workload),
         ("algorithmic_bytes" if bound == "hbm" else "algorithmic_flops"): work, "avg_launch_ms": avg_ms,
         "launches_timed": launches}
    if bound == "hbm":
        r["frac_of_nominal_8tbs"] = achieved / NOMINAL_HBM_GBS
    return r


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
    # at least three warm-up steps, as many as asked while they take under a minute
    warm, t_warm = 0, time.time()
    while warm < max(args.warmup, 3) and (warm < 3 or time.time() - t_warm < 60.0):
        oracle_step(orc, inp, threads)
        warm += 1
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
            "steps": len(times), "steps_requested": args.steps, "warmup": warm,
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
    # (one cluster launch for rows of up to 131072 entries) + one attention launch for the four layers
    # (they attend the same selected rows; split partials are merged inside that launch)
    return 4


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
        "kv_gbs": kv_gbs, "hbm_frac_step": kv_gbs / peak, "hbm_frac_step_nominal_8tbs": kv_gbs / NOMINAL_HBM_GBS,
        "bytes_per_step": BYTES_PER_SEQ * B_PER_GPU * world,
        "roofline": dict(roofline("index_score_stream_kernel", f"decode_group_b{B_PER_GPU}_t{T_CTX}", "hbm",
                                  score_bytes, score_avg, len(score_ms), peak, f"{peak_kind} (hbm copy)"),
                         timed_every=SCORE_EVERY),
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
# other workloads (`--workload`): one line each on one GPU, device-resident inputs, CUDA events
# ----------------------------------------------------------------------------------------------
def bf16_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return 1900.0, "fallback"


class Pairs:
    """Event pairs handed to the library (score scan, first attention launch), one per timed step."""

    def __init__(self, torch, n):
        self.p = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        for a, b in self.p:    # materialise the event handles
            a.record()
            b.record()

    def ms(self):
        return [a.elapsed_time(b) for a, b in self.p]


def timed_loop(torch, step, K, Wm, flush=None, sampler=None):
    """Wm untimed steps, then K steps.  Without `flush`: K steps back to back between two events.
    With `flush` (a buffer larger than L2): the buffer is overwritten before every step and each
    step is bracketed by its own events.  Returns (ms per step, wall-clock start, end)."""
    for i in range(Wm):
        if flush is not None:
            flush.zero_()
        step(None)
    torch.cuda.synchronize()
    time.sleep(0.05)
    t0 = time.time()
    if flush is None:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for i in range(K):
            step(i)
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / K
    else:
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
        for i in range(K):
            flush.zero_()
            ev[i][0].record()
            step(i)
            ev[i][1].record()
        torch.cuda.synchronize()
        ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    return ms, t0, time.time()


def oracle_cpu_baseline(fn, units, unit_name, sample, threads, min_cpu_s=10.0, max_wall_s=60.0, per_unit=True):
    """The oracle on the host cores: repeat fn() until about min_cpu_s of CPU work (wall x threads).
    Returns the cpu_baseline object (value = units per second, or milliseconds per call)."""
    import oracle as orc
    orc.build()
    times = []
    t_start = time.time()
    while not times or (sum(times) * threads < min_cpu_s and time.time() - t_start < max_wall_s):
        t0 = time.perf_counter()
        fn()
        times.append(time.perf_counter() - t0)
    dt = statistics.mean(times)
    value = units / dt if per_unit else dt * 1e3
    return {"value": value, "unit": unit_name, "cores": threads, "kind": "oracle",
            "sample": f"{sample}; {len(times)} runs, {dt:.3f} s wall each on {threads} threads"}


def host_inputs(n_seq, T, L, seed, Nq=1, W=W_WIN, fp8=False):
    """Oracle inputs for a bounded sample: n_seq sequences of T entries.  Indexer keys, queries,
    weights and windows are the seeded N(0, 1) draws; the FP4 cache rows are random code bytes with
    scales in the range N(0, 1) rows quantise to (the oracle reads only the rows it selects, so their
    values do not change its work)."""
    import csa2_synth as syn
    g = np.random.default_rng(seed)
    codes = g.integers(0, 256, (n_seq, T, 256), dtype=np.uint8)
    scales = g.integers(0x2C, 0x3C, (n_seq, T, 32), dtype=np.uint8)
    KI = np.stack([syn.normal_bf16(seed, syn.T_KI, b, (T, 128)) for b in range(n_seq)])

    def per_layer(tid, shape, f=syn.normal_bf16):
        return np.stack([np.stack([f(seed, tid + l, b, shape) for b in range(n_seq)]) for l in range(L)])
    q = per_layer(syn.T_Q, (Nq, 16, 512))
    qI = per_layer(syn.T_QI, (Nq, 4, 128))
    w = per_layer(syn.T_W, (Nq, 4), syn.normal_f32)
    swa = per_layer(syn.T_SWA, (W - 1 + Nq, 512))
    if fp8:
        swa = g.integers(0, 0x78, swa.shape, dtype=np.uint8) | (g.integers(0, 2, swa.shape, dtype=np.uint8) << 7)
    return codes, scales, KI, q, qI, w, swa


def device_cache(torch, c, syn, B, T, seed, dev):
    """FP4 main KV filled by the library's own quantiser from N(0, 1) rows, one sequence at a time,
    and the indexer keys."""
    codes = torch.empty((B, T, 256), dtype=torch.uint8, device=dev)
    scales = torch.empty((B, T, 32), dtype=torch.uint8, device=dev)
    for b in range(B):
        kv = syn.device_normal_bf16((1, T, 512), seed, syn.T_KV * 1000 + b, device=dev)
        c.csa2_fp4_quantize_append(kv, codes[b:b + 1], scales[b:b + 1])
        del kv
    KI = syn.device_normal_bf16((B, T, 128), seed, syn.T_KI * 1000, device=dev)
    return codes, scales, KI


def run_full_layer(args, torch, c, syn, dev, sampler):
    """A single Full-layer decode step: batch 1, 4096 entries; append, score, Top-512, attention over
    the 512 rows plus 128 window rows.  L2 is flushed before every step."""
    B, T = 1, 4096
    seed = syn.SEEDS["full_layer_decode_b1_t4096"]
    codes, scales, KI = device_cache(torch, c, syn, B, T, seed, dev)
    q = [syn.device_normal_bf16((B, 1, 16, 512), seed, syn.T_Q, device=dev)]
    qI = [syn.device_normal_bf16((B, 1, 4, 128), seed, syn.T_QI, device=dev)]
    w = [syn.device_normal_bf16((B, 1, 4), seed, syn.T_W, device=dev).float()]
    swa = [syn.device_normal_bf16((B, W_WIN, 512), seed, syn.T_SWA, device=dev)]
    kv_new = syn.device_normal_bf16((B, 1, 512), seed, syn.T_KV_NEW, device=dev)
    ki_new = syn.device_normal_bf16((B, 1, 128), seed, syn.T_KI_NEW, device=dev)
    lens = torch.full((B,), T, dtype=torch.int32, device=dev)
    swa_len = torch.full((B,), W_WIN, dtype=torch.int32, device=dev)
    out = [torch.empty((B, 1, 16, 512), dtype=torch.bfloat16, device=dev)]
    idx = [torch.empty((B, K_SEL), dtype=torch.int32, device=dev)]
    ws = torch.empty(c.group_workspace_size(B, 1, T, K_SEL, W_WIN), dtype=torch.uint8, device=dev)
    K = args.steps
    sc, at = Pairs(torch, K), Pairs(torch, K)

    def desc(i):
        return c.make_group_desc([c.MODE_FULL], B=B, Nq=1, cap=T, lens=lens, codes=codes, scales=scales, KI=KI,
                                 q=q, qI=qI, w=w, swa=swa, swa_len=swa_len, out=out, idx=idx, K=K_SEL, W=W_WIN,
                                 kv_new=kv_new, ki_new=ki_new, events=None if i is None else sc.p[i],
                                 attn_events=None if i is None else at.p[i])
    descs = [desc(i) for i in range(K)]
    plain = desc(None)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    ms, t0, t1 = timed_loop(torch, lambda i: c.csa2_group_step(plain if i is None else descs[i], ws), K,
                            args.warmup, flush=flush)
    score_ms, attn_ms = statistics.mean(sc.ms()), statistics.mean(at.ms())
    bytes_step = T * 256 + BYTES_ATTN_PER_SEQ_LAYER + BYTES_APPEND_PER_SEQ
    peak, kind = peaks()
    # the dominant kernel of the step, by its event-timed duration
    if score_ms >= attn_ms:
        rl = roofline("index_score_stream_kernel", "full_layer_decode_b1_t4096", "hbm", T * 256, score_ms, K, peak,
                      f"{kind} (hbm copy)")
    else:
        rl = roofline("sparse_attn_ws_kernel", "full_layer_decode_b1_t4096", "hbm", BYTES_ATTN_PER_SEQ_LAYER, attn_ms, K,
                      peak, f"{kind} (hbm copy)")
    cpu = None
    if not args.no_cpu_baseline:
        import oracle as orc
        inp = host_inputs(1, T, 1, seed)
        cpu = oracle_cpu_baseline(
            lambda: orc.group_step([0], [T], *inp, np.full(1, W_WIN, np.int32), threads=1),
            1, "ms per step", "the same Full-layer step (1 sequence, 4096 entries, Top-512 + 128 window rows)",
            1, per_unit=False)
    return {"metric": "CSA2 single Full-layer decode step latency (batch 1, 4096 entries)", "value": ms * 1e3,
            "unit": "us per step", "ms_per_step": ms, "higher_is_better": False,
            "config": {"workload": "csa2_full_layer_decode_b1_t4096", "global_batch": B, "seq_len": T,
                       "layers": "1 Full", "top_k": K_SEL, "window": W_WIN,
                       "l2": "flushed (256 MiB written) before every step; each step timed by its own events"},
            "tokens_per_s": B / (ms / 1e3), "kv_gbs": bytes_step / (ms / 1e3) / 1e9, "bytes_per_step": bytes_step,
            "hbm_frac_step": bytes_step / (ms / 1e3) / 1e9 / peak,
            "kernel_ms": {"index_score_stream_kernel": score_ms, "sparse_attn_ws_kernel": attn_ms},
            # the append, the score scan, Top-K (one launch for rows of at most 8192 entries), attention
            "roofline": rl, "cpu_baseline": cpu, "gpu_launches": 4 * K,
            "clocks": sampler.summary(t0, t1) if sampler else None}


def run_fp4_roundtrip(args, torch, c, syn, dev, sampler):
    """FP4 quantise (bf16 -> E2M1 codes + E4M3 scales) and dequantise (back to bf16) of 64 x 8192 x
    512 rows drawn N(0, 1) with 1% of the entries scaled by 20; each direction timed on its own.
    Inputs (537 MB) exceed L2."""
    S, T = 64, 8192
    seed = syn.SEEDS["fp4_roundtrip_64x8192x512"]
    x = syn.device_outlier_bf16((S, T, 512), seed, syn.T_X, device=dev)
    codes = torch.empty((S, T, 256), dtype=torch.uint8, device=dev)
    scales = torch.empty((S, T, 32), dtype=torch.uint8, device=dev)
    out = torch.empty((S, T, 512), dtype=torch.bfloat16, device=dev)
    K = args.steps
    tq, t0, _ = timed_loop(torch, lambda i: c.csa2_fp4_quantize_append(x, codes, scales), K, args.warmup)
    tdq, _, t1 = timed_loop(torch, lambda i: c.csa2_fp4_dequantize(codes, scales, out), K, args.warmup)
    rows = S * T
    bytes_dir = rows * (1024 + 288)       # bf16 row one way, 256 code bytes + 32 scale bytes the other
    peak, kind = peaks()
    rq = roofline("fp4_quantize_kernel", "fp4_roundtrip_64x8192x512", "hbm", bytes_dir, tq, K, peak, f"{kind} (hbm copy)")
    rd = roofline("fp4_dequantize_kernel", "fp4_roundtrip_64x8192x512", "hbm", bytes_dir, tdq, K, peak,
                  f"{kind} (hbm copy)")
    cpu = None
    if not args.no_cpu_baseline:
        import oracle as orc
        threads = cpu_threads()
        n = 256 * threads
        xs = syn.outlier_bf16(seed, syn.T_X, 0, (n, 512))

        def rt():
            cq, sq = orc.fp4_quantize(xs, threads=threads)
            orc.fp4_dequantize(cq, sq)
        cpu = oracle_cpu_baseline(rt, 2 * n * (1024 + 288) / 1e9, "GB/s",
                                  f"{n} of the {rows} rows, quantised ({threads} threads) and dequantised (1 thread)",
                                  threads)
    gbs = 2 * bytes_dir / ((tq + tdq) / 1e3) / 1e9
    return {"metric": "FP4 KV quantise + dequantise round trip GB/s (64 x 8192 x 512 bf16, 1% outliers x20)",
            "value": gbs, "unit": "GB/s", "ms_per_step": tq + tdq, "higher_is_better": True,
            "config": {"workload": "fp4_roundtrip_64x8192x512", "rows": rows, "channels": 512,
                       "l2": "inputs larger than L2 (537 MB of bf16 rows)"},
            "bytes_per_direction": bytes_dir,
            "quantize": {"ms": tq, "gbs": rq["achieved"], "frac": rq["frac"], "frac_of_nominal_8tbs": rq["frac_of_nominal_8tbs"]},
            "dequantize": {"ms": tdq, "gbs": rd["achieved"], "frac": rd["frac"],
                           "frac_of_nominal_8tbs": rd["frac_of_nominal_8tbs"]},
            "roofline": rq if tq >= tdq else rd, "roofline_other": rd if tq >= tdq else rq,
            "cpu_baseline": cpu, "gpu_launches": 2 * K, "clocks": sampler.summary(t0, t1) if sampler else None}


def run_stack20(args, torch, c, syn, dev, sampler):
    """One token through the 20-layer decoder: 5 groups of 4 (Full + 3 Reuse, then 4 x Reindex +
    3 Reuse) over one cache, B = 64, T = 131072; one csa2_stack_step per step."""
    wl = build_workload(torch, c, syn, dev)
    seed = syn.SEEDS["decode_group_1f3r_b64_t131072"]
    B, T, K = B_PER_GPU, T_CTX, args.steps
    sc = Pairs(torch, K)
    first = [make_desc(c, wl, events=sc.p[i]) for i in range(K)]
    rest = []
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
        rest.append(c.make_group_desc(
            [c.MODE_REINDEX, c.MODE_REUSE, c.MODE_REUSE, c.MODE_REUSE], B=B, Nq=1, cap=T, lens=wl["lens"],
            codes=wl["codes"], scales=wl["scales"], KI=wl["KI"], q=q, qI=qI, w=w, swa=swa, swa_len=wl["swa_len"],
            out=out, idx=idx, K=K_SEL, W=W_WIN))
    plain = [make_desc(c, wl)] + rest
    ms, t0, t1 = timed_loop(torch, lambda i: c.csa2_stack_step(plain if i is None else [first[i]] + rest, wl["ws"]),
                            K, max(args.warmup, 3))
    # algorithmic bytes: 5 indexer-K scans + 20 layers of attention + the append, per sequence
    per_seq = 5 * BYTES_KI_PER_SEQ + 20 * BYTES_ATTN_PER_SEQ_LAYER + BYTES_APPEND_PER_SEQ
    peak, kind = peaks()
    gbs = per_seq * B / (ms / 1e3) / 1e9
    cpu = None
    if not args.no_cpu_baseline:
        import oracle as orc
        threads = cpu_threads()
        n = min(B, threads)
        inp = host_inputs(n, T, 20, seed)
        modes = ([0, 2, 2, 2] + [1, 2, 2, 2] * 4)
        cpu = oracle_cpu_baseline(lambda: orc.group_step(modes, [T] * n, *inp, np.full(n, W_WIN, np.int32),
                                                         threads=threads),
                                  n, "tokens/s", f"{n} of the 64 sequences at full context, 20 layers", threads)
    return {"metric": "CSA2 20-layer decoder stack tokens/s at 128K ctx", "value": B / (ms / 1e3),
            "unit": "tokens/s", "ms_per_step": ms, "higher_is_better": True,
            "config": {"workload": "csa2_decoder_stack_5x4_b64_t131072", "global_batch": B, "seq_len": T,
                       "layers": "Full+3 Reuse, then 4 x (Reindex + 3 Reuse)", "top_k": K_SEL, "window": W_WIN,
                       "l2": "inputs larger than L2 (five 2.1 GB indexer-K scans per step)"},
            "kv_gbs": gbs, "hbm_frac_step": gbs / peak, "hbm_frac_step_nominal_8tbs": gbs / NOMINAL_HBM_GBS,
            "roofline": roofline("index_score_stream_kernel", f"decode_group_b{B}_t{T}", "hbm", B * BYTES_KI_PER_SEQ,
                                 statistics.mean(sc.ms()), K, peak, f"{kind} (hbm copy)"),
            "cpu_baseline": cpu,
            # group 1: append + score + Top-K + attention; groups 2-5: score + Top-K + attention
            "gpu_launches": (4 + 3 * 4) * K, "clocks": sampler.summary(t0, t1) if sampler else None}


def run_prefill(args, torch, c, syn, dev, sampler):
    """The encoder prefill chunk: 2048 queries at the end of 262144 tokens (131072 compressed
    entries, ratio 2), 1 Full + 5 Reuse, Top-512, 128-token window; one csa2_group_step per step."""
    seed = syn.SEEDS["prefill_group_1f5r_ratio2_q2048"]
    T, Nq, L = 131072, 2048, 6
    codes, scales, KI = device_cache(torch, c, syn, 1, T, seed, dev)
    q = [syn.device_normal_bf16((1, Nq, 16, 512), seed, syn.T_Q + l, device=dev) for l in range(L)]
    qI = [syn.device_normal_bf16((1, Nq, 4, 128), seed, syn.T_QI, device=dev)] + [None] * (L - 1)
    w = [syn.device_normal_bf16((1, Nq, 4), seed, syn.T_W, device=dev).float()] + [None] * (L - 1)
    swa = [syn.device_normal_bf16((1, W_WIN - 1 + Nq, 512), seed, syn.T_SWA + l, device=dev) for l in range(L)]
    out = [torch.empty((1, Nq, 16, 512), dtype=torch.bfloat16, device=dev) for _ in range(L)]
    idx = [torch.empty((Nq, K_SEL), dtype=torch.int32, device=dev)] + [None] * (L - 1)
    lens = torch.tensor([T], dtype=torch.int32, device=dev)
    swa_len = torch.tensor([W_WIN - 1 + Nq], dtype=torch.int32, device=dev)
    q_pos = torch.arange(2 * T - Nq, 2 * T, dtype=torch.int32, device=dev)
    K = args.steps
    at = Pairs(torch, K)

    def desc(i):
        return c.make_group_desc([c.MODE_FULL] + [c.MODE_REUSE] * (L - 1), B=1, Nq=Nq, cap=T, lens=lens,
                                 codes=codes, scales=scales, KI=KI, q=q, qI=qI, w=w, swa=swa, swa_len=swa_len,
                                 out=out, idx=idx, K=K_SEL, W=W_WIN, ratio=2, q_pos=q_pos,
                                 attn_events=None if i is None else at.p[i])
    descs = [desc(i) for i in range(K)]
    plain = desc(None)
    ws = torch.empty(c.group_workspace_size(1, Nq, T, K_SEL, W_WIN), dtype=torch.uint8, device=dev)
    ms, t0, t1 = timed_loop(torch, lambda i: c.csa2_group_step(plain if i is None else descs[i], ws), K,
                            max(args.warmup, 3))
    # dense work: the indexer contraction over each query's visible entries (1024 flop per pair)
    # and 6 layers of attention (2 x 16 heads x 512 x 640 rows x 2 flop per query)
    vis = (np.arange(2 * T - Nq, 2 * T) + 1) // 2
    attn_flop = L * Nq * 2 * 16 * 512 * (K_SEL + W_WIN) * 2
    gflop = (float(vis.sum()) * 1024 + attn_flop) / 1e9
    peak, kind = bf16_peak()
    tflops = gflop / ms
    cpu = None
    if not args.no_cpu_baseline:
        import oracle as orc
        threads = cpu_threads()
        n = 2 * threads        # the chunk's last n queries, every layer
        inp = host_inputs(1, T, L, seed, Nq=n)
        qp = np.arange(2 * T - n, 2 * T, dtype=np.int32)[None]
        cpu = oracle_cpu_baseline(
            lambda: orc.group_step([0] + [2] * (L - 1), [T], *inp, np.array([W_WIN - 1 + n], np.int32), Nq=n,
                                   ratio=2, q_pos=qp, threads=threads),
            n, "queries/s", f"the last {n} of the 2048 queries, 6 layers", threads)
    return {"metric": "CSA2 encoder prefill chunk queries/s (2048 q x 131072 entries, 6 layers)",
            "value": Nq / (ms / 1e3), "unit": "queries/s", "ms_per_step": ms, "higher_is_better": True,
            "config": {"workload": "csa2_prefill_1f5r_ratio2_q2048_t131072", "global_batch": Nq, "seq_len": 2 * T,
                       "layers": "1 Full + 5 Reuse", "top_k": K_SEL, "window": W_WIN,
                       "l2": "no flush: the chunk's selection streams 33.5 MB of keys twice and 2048 x 512 "
                             "gathered rows; steps run back to back"},
            "dense_gflop_per_step": gflop, "tflops_step": tflops, "bf16_peak_tflops": peak,
            "frac_of_bf16_peak": tflops / peak, "peak_kind": kind,
            "roofline": roofline("sparse_attn_pair_kernel", "prefill_chunk_q2048_t131072", "tensor", attn_flop,
                                 statistics.mean(at.ms()), K, peak, f"{kind} (bf16 dense, burst)"),
            "cpu_baseline": cpu,
            # counters cleared, key norms, two tensor-core passes, threshold, count, order,
            # rescore/select, attention
            "gpu_launches": 9 * K, "clocks": sampler.summary(t0, t1) if sampler else None}


def run_fp8win(args, torch, c, syn, dev, sampler):
    """The decode workload with 8-bit windows: the same group step, every layer's 128 window rows
    held as E4M3 bytes (csa2_fp8_quantize at set-up)."""
    wl = build_workload(torch, c, syn, dev)
    swa8 = []
    for x in wl["swa"]:
        y = torch.empty(x.shape, dtype=torch.uint8, device=dev)
        c.csa2_fp8_quantize(x, y)
        swa8.append(y)
    K = args.steps
    sc = Pairs(torch, K)

    def desc(i):
        return c.make_group_desc(
            [c.MODE_FULL, c.MODE_REUSE, c.MODE_REUSE, c.MODE_REUSE], B=B_PER_GPU, Nq=1, cap=T_CTX, lens=wl["lens"],
            codes=wl["codes"], scales=wl["scales"], KI=wl["KI"], q=wl["q"], qI=wl["qI"], w=wl["w"], swa=swa8,
            swa_len=wl["swa_len"], out=wl["out"], idx=wl["idx"], K=K_SEL, W=W_WIN, kv_new=wl["kv_new"],
            ki_new=wl["ki_new"], swa_fp8=True, events=None if i is None or i % SCORE_EVERY else sc.p[i])
    descs = [desc(i) for i in range(K)]
    plain = desc(None)
    ms, t0, t1 = timed_loop(torch, lambda i: c.csa2_group_step(plain if i is None else descs[i], wl["ws"]), K,
                            max(args.warmup, 3))
    per_seq = BYTES_PER_SEQ - N_LAYERS * W_WIN * 512   # window rows of 512 B instead of 1 KiB
    peak, kind = peaks()
    gbs = per_seq * B_PER_GPU / (ms / 1e3) / 1e9
    cpu = None
    if not args.no_cpu_baseline:
        import oracle as orc
        threads = cpu_threads()
        n = min(64, 2 * threads)
        inp = host_inputs(n, T_CTX, N_LAYERS, 0, fp8=True)
        cpu = oracle_cpu_baseline(lambda: orc.group_step([0, 2, 2, 2], [T_CTX] * n, *inp, np.full(n, W_WIN, np.int32),
                                                         threads=threads, swa_fp8=True),
                                  n, "tokens/s", f"{n} of the 64 sequences at full context, 8-bit windows", threads)
    score_ms = [m for i, m in enumerate(sc.ms()) if i % SCORE_EVERY == 0]
    return {"metric": "CSA2 decode tokens/s at 128K ctx with 8-bit (E4M3) windows", "value": B_PER_GPU / (ms / 1e3),
            "unit": "tokens/s", "ms_per_step": ms, "higher_is_better": True,
            "config": {"workload": "csa2_decode_group_1full_3reuse_b64_t131072_fp8win", "global_batch": B_PER_GPU,
                       "seq_len": T_CTX, "layers": "1 Full + 3 Reuse", "top_k": K_SEL, "window": W_WIN,
                       "window_format": "E4M3, one byte per channel",
                       "l2": "inputs larger than L2 (2.1 GB indexer-K scan per step)"},
            "kv_gbs": gbs, "hbm_frac_step": gbs / peak, "hbm_frac_step_nominal_8tbs": gbs / NOMINAL_HBM_GBS,
            "bytes_per_step": per_seq * B_PER_GPU,
            "roofline": dict(roofline("index_score_stream_kernel", f"decode_group_b{B_PER_GPU}_t{T_CTX}", "hbm",
                                      B_PER_GPU * BYTES_KI_PER_SEQ, statistics.mean(score_ms), len(score_ms), peak,
                                      f"{kind} (hbm copy)"), timed_every=SCORE_EVERY),
            "cpu_baseline": cpu, "gpu_launches": launches_per_step(c) * K,
            "clocks": sampler.summary(t0, t1) if sampler else None}


def run_hier1m(args, torch, c, syn, dev, sampler):
    """The hierarchical indexer at 1M context: batch 8, T = 2^20, ratio 1; Full (top 2048 blocks of 8
    by block key, then Top-512 in the 16384-position pool) + Reindex (the same pool, its own indexer
    Q) + 3 Reuse; each step appends the new token (refreshing the block it completes).  L2 is
    flushed before every step."""
    seed = syn.SEEDS["hier_decode_b8_t1m"]
    B, T, L, keep = min(args.batch, 8), 1 << 20, 5, 2048    # batch 8 is the workload (smaller for profiling)
    codes, scales, KI = device_cache(torch, c, syn, B, T, seed, dev)
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
    K = args.steps
    sc = Pairs(torch, K)

    def desc(i):
        return c.make_group_desc([c.MODE_FULL, c.MODE_REINDEX, c.MODE_REUSE, c.MODE_REUSE, c.MODE_REUSE], B=B, Nq=1,
                                 cap=T, lens=lens, codes=codes, scales=scales, KI=KI, q=q, qI=qI, w=w, swa=swa,
                                 swa_len=swa_len, out=out, idx=idx, K=K_SEL, W=W_WIN, hierarchical=True, keep=keep,
                                 block_keys=block_keys, pool=pool, pool_len=pool_len, kv_new=kv_new, ki_new=ki_new,
                                 events=None if i is None else sc.p[i])
    descs = [desc(i) for i in range(K)]
    plain = desc(None)
    ws = torch.empty(c.group_workspace_size(B, 1, T, K_SEL, W_WIN, hierarchical=True, keep=keep), dtype=torch.uint8,
                     device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    ms, t0, t1 = timed_loop(torch, lambda i: c.csa2_group_step(plain if i is None else descs[i], ws), K,
                            max(args.warmup, 3), flush=flush)
    # algorithmic bytes per sequence: the block-key scan, the pool's indexer keys for Full and Reindex,
    # five layers of attention, the append
    per_seq = (T // 8) * 256 + 2 * keep * 8 * 256 + L * BYTES_ATTN_PER_SEQ_LAYER + BYTES_APPEND_PER_SEQ
    peak, kind = peaks()
    gbs = per_seq * B / (ms / 1e3) / 1e9
    cpu = None
    if not args.no_cpu_baseline:
        import oracle as orc
        threads = cpu_threads()
        n = 2
        inp = host_inputs(n, T, L, seed)
        cpu = oracle_cpu_baseline(
            lambda: orc.group_step([0, 1, 2, 2, 2], [T] * n, *inp, np.full(n, W_WIN, np.int32), hierarchical=True,
                                   keep=keep, threads=threads),
            n, "tokens/s", f"{n} of the 8 sequences at 2^20 entries (block keys, pool, 5 layers)", threads)
    return {"metric": "CSA2 hierarchical decode tokens/s at 1M ctx", "value": B / (ms / 1e3), "unit": "tokens/s",
            "ms_per_step": ms, "higher_is_better": True,
            "config": {"workload": f"csa2_hier_decode_full_reindex_3reuse_b{B}_t1m", "global_batch": B, "seq_len": T,
                       "layers": "Full + Reindex + 3 Reuse", "blocks_kept": keep, "pool": keep * 8, "top_k": K_SEL,
                       "window": W_WIN, "l2": "flushed (256 MiB written) before every step; each step timed by its "
                                              "own events"},
            "kv_gbs": gbs, "hbm_frac_step": gbs / peak, "hbm_frac_step_nominal_8tbs": gbs / NOMINAL_HBM_GBS,
            "bytes_per_step": per_seq * B,
            "roofline": roofline("index_score_stream_kernel", f"hier_decode_b{B}_t1m", "hbm", B * (T // 8) * 256,
                                 statistics.mean(sc.ms()), K, peak, f"{kind} (hbm copy)"),
            "cpu_baseline": cpu,
            # the append (with the completed block's key), the block scan, Top-2048, then for Full and
            # Reindex each a pool scan and Top-512, and one attention launch for the five layers
            "gpu_launches": 8 * K, "clocks": sampler.summary(t0, t1) if sampler else None}


EXTRA = {"full_layer_decode": run_full_layer, "fp4_roundtrip": run_fp4_roundtrip, "prefill_chunk": run_prefill,
         "hier_decode_1m": run_hier1m, "decoder_stack_20": run_stack20, "decode_group_fp8win": run_fp8win}


def run_extra(args):
    import torch

    import csa2_synth as syn
    import compressed_sparse_attention_step_gb300 as c
    from compressed_sparse_attention_step_gb300 import _build
    if not os.path.exists(_build.LIB):
        raise RuntimeError("libcsa2.so is not built: run `python -c 'import __graft_entry__ as g; g.build()'`")
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    c.lib()
    sampler = ClockSampler(0)
    try:
        line = EXTRA[args.workload](args, torch, c, syn, dev, sampler)
    finally:
        sampler.stop()
    line.update({"n_gpus": 1, "steps": args.steps, "warmup": max(args.warmup, 3), "scaling": "weak",
                 "vs_baseline": None, "dtype": "bf16/fp4 in, fp32 accumulate", "data": "synthetic"})
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
    ap.add_argument("--workload", default="decode_group", choices=["decode_group"] + sorted(EXTRA),
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
