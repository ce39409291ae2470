"""Benchmark of the TurboQuant compressed-KV path on B300: prefill quantize + decode steps.

One step = the whole hot path over one batch of the long-context workload (batch 4, 8 KV
heads, 32 query heads, head_dim 128, b=3, 131,072 cached tokens per sequence):
  1. tq_quantize_kv of the full prefill (524,288 tokens x 8 KV heads, K and V);
  2. 64 decode steps, each appending one token per (sequence, KV head) with
     tq_quantize_kv and then running tq_attn_decode for all 32 query heads.

Printed (rank 0, one JSON line):
  value       compressed-KV decode GB/s: algorithmic bytes of the 64 decode steps (the
              compressed pages attended, plus q and out) over the device time of the decode
              phase (appends included), summed over all ranks' work / max-over-ranks time;
  quantize_mtok_s  prefill tokens (all KV heads of a token) per second;
  roofline    the decode kernel's algorithmic GB/s against the measured HBM copy peak;
  e2e         the same decode bytes over the whole step measured through the API with host
              buffers: the prefill K/V and every decode step's inputs copied in from pinned
              host memory, every output read back, prefill quantize and decode included;
  cpu_baseline  the fp64 oracle on a bounded sample of the same workload, on one host thread
              (its page unpacking is plain Python), with the figure at the BLAS pool size beside.

roofline.traffic is the DRAM traffic of one decode-kernel launch from a committed ncu summary
(profiles/), used only while the summary's recorded source fingerprint matches the kernel
source being run; otherwise null.

--impl reference times the oracle alone (there is no other implementation of this path).
--sweep prints one line per (d, b) point of the bit/dim sweep instead.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "compressed-KV decode GB/s & % HBM roofline; quantize Mtokens/s (d=128, b=3)"
UNIT = "GB/s"
DTYPE = ("decode: e2m1 operand pieces (signed bit planes x fixed-point / e2m1 pieces), fp32 accumulate; "
         "quantize: bf16 hi/lo MMAs, fp32 accumulate; cache: packed bit planes + fp32 norms")
DECODE_KERNEL = "decode_f4_kernel"
DECODE_SOURCES = ["kv_cache_vector_19_b300/csrc/decode_f4.cuh", "kv_cache_vector_19_b300/csrc/dev_common.cuh"]
TRAFFIC_PROFILE = "profiles/decode_f4_kernel_longctx.md"


def source_fingerprint():
    """sha256 (first 16 hex digits) of the decode kernel's sources, as recorded in profiles."""
    import hashlib
    h = hashlib.sha256()
    for rel in DECODE_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def committed_traffic():
    """DRAM bytes per decode launch from the committed ncu summary, if it was taken on the
    kernel source being run (its 'source fingerprint:' line matches), else None."""
    import re
    try:
        text = open(os.path.join(ROOT, TRAFFIC_PROFILE)).read()
    except OSError:
        return None
    fp = re.search(r"source fingerprint:\s*([0-9a-f]{16})", text)
    tb = re.search(r"traffic bytes per launch:\s*([0-9]+)", text)
    if not fp or not tb or fp.group(1) != source_fingerprint():
        return None
    return int(tb.group(1))


def bpt(d, b, m):
    """Compressed bytes per token per KV head (keys + values)."""
    return (b - 1) * d // 8 + m // 8 + 8 + b * d // 8 + 4


def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return float(pk["hbm_gbs"]), "measured"
    except Exception:
        return 6400.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            out, _ = self.proc.communicate(timeout=10)
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def max_over_ranks(times_ms, world, device):
    """Each timing as the maximum over the ranks (the slowest rank sets the job's time)."""
    if world <= 1:
        return list(times_ms)
    import torch
    import torch.distributed as dist
    t = torch.tensor(list(times_ms), device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def job_gbs(world, bytes_per_rank, t_ms):
    """Whole-job GB/s: every rank processes bytes_per_rank of its own sequences (replicas) in
    the max-over-ranks time t_ms."""
    return world * bytes_per_rank / (t_ms * 1e-3) / 1e9


def _oracle_sample(w, seed):
    """The oracle's packed pages of a 1024-token sample of workload w (one KV head) and G query
    rows: what the CPU baseline decodes."""
    import numpy as np
    import torch

    from oracle import pagefmt, params, quant

    rng = np.random.default_rng(seed)
    d, b, m, G = w.d, w.b, w.m, w.group
    T = 1024
    p = params.make(d, b, m, seed=w.seed)
    X = rng.standard_normal((2, T, d)).astype(np.float32)
    X = torch.from_numpy(X).to(torch.bfloat16).double().numpy()
    t0 = time.perf_counter()
    ok = quant.quantize_keys(X[0], p.Pi, p.S, p.cb_k)
    ov = quant.quantize_values(X[1], p.Pi, p.cb_v)
    t_quant = time.perf_counter() - t0
    pages = []
    for pg in range(T // 128):
        sl = slice(pg * 128, (pg + 1) * 128)
        pages.append(pagefmt.pack_page(d, b, m, ok["idx"][sl], ok["sigma"][sl], ok["n"][sl], ok["gamma"][sl],
                                       ov["idx"][sl], ov["n"][sl]))
    return dict(p=p, cache=np.concatenate(pages), q=rng.standard_normal((G, d)), T=T, t_quant=t_quant)


def _oracle_decode(w, smp, limit_s, reps_max):
    """Repeats the oracle decode of the sample (unpack + route A for the G query heads) for
    ~limit_s seconds; returns (reps, seconds)."""
    import numpy as np

    from oracle import decode as odec
    from oracle import pagefmt

    d, b, m, G, T, p = w.d, w.b, w.m, w.group, smp["T"], smp["p"]
    reps, t_dec = 0, 0.0
    while t_dec < limit_s and reps < reps_max:
        t0 = time.perf_counter()
        tok = pagefmt.unpack_tokens(d, b, m, smp["cache"], T // 128, 0, 0, T, 1)
        tk = dict(idx=tok["kidx"], n=tok["nk"].astype(np.float64), sigma=tok["sigma"],
                  gamma=tok["gamma"].astype(np.float64))
        tv = dict(idx=tok["vidx"], n=tok["nv"].astype(np.float64))
        for h in range(G):
            odec.attend_route_a(smp["q"][h], tk, tv, p.Pi, p.S, p.cb_k, p.cb_v)
        t_dec += time.perf_counter() - t0
        reps += 1
    return reps, t_dec


def _oracle_worker(job):
    """One process of the multi-process CPU baseline: (workload name, seed, seconds) ->
    (GB/s, reps, seconds) of the oracle decode on one thread of its own."""
    name, seed, seconds = job
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[var] = "1"   # before numpy loads its BLAS in this fresh process
    from kv_cache_vector_19_b300 import workloads
    w = workloads.preset(name)
    smp = _oracle_sample(w, seed)
    reps, t = _oracle_decode(w, smp, seconds, 10 ** 6)
    return reps * smp["T"] * bpt(w.d, w.b, w.m) / t / 1e9, reps, t


def cpu_oracle_sample(w, seconds=12.0, reps_max=1000, processes=0):
    """The oracle's own decode over packed pages (unpack + route A for the G query heads of one
    KV head) on a 1024-token sample of the workload: ~seconds / 2 on one thread, ~seconds / 2
    with the BLAS pool, and, with processes > 1, the same sample in that many spawned processes
    at once (one thread each; started before any GPU work).  Returns (GB/s, Mtokens/s quantized,
    threads of the GB/s figure, description, GB/s on one thread, GB/s with the BLAS pool, pool
    size)."""
    smp = _oracle_sample(w, 1234)
    T = smp["T"]
    per_rep = T * bpt(w.d, w.b, w.m)
    try:
        from threadpoolctl import threadpool_info, threadpool_limits
        pool = max([i.get("num_threads", 1) for i in threadpool_info()] + [1])
        with threadpool_limits(1):
            reps1, t1 = _oracle_decode(w, smp, seconds / 2, reps_max)
    except ImportError:   # no pool control: the run below is the only figure
        threadpool_limits, pool = None, 1
    reps, t_dec = _oracle_decode(w, smp, seconds / 2 if threadpool_limits else seconds, reps_max)
    if threadpool_limits is None:
        reps1, t1 = reps, t_dec
    gbs1, gbs = reps1 * per_rep / t1 / 1e9, reps * per_rep / t_dec / 1e9
    value, threads = gbs1, 1
    head = f"oracle decode of 1 KV head x {T} tokens ({T // 128} packed pages) for {w.group} query heads: "
    if threadpool_limits is not None:
        desc = head + (f"{reps1} reps in {t1:.1f} s on 1 thread; {reps} reps in {t_dec:.1f} s with a {pool}-thread "
                       f"BLAS pool ({gbs:.4f} GB/s; page unpacking is single-threaded Python either way)")
    else:
        desc = head + (f"{reps} reps in {t_dec:.1f} s in this process (BLAS threads not controlled here: "
                       f"threadpoolctl is not importable)")
    if processes > 1:
        import multiprocessing
        with multiprocessing.get_context("spawn").Pool(processes) as mp:
            res = mp.map(_oracle_worker, [(w.name, 1234 + i, seconds / 2) for i in range(processes)])
        value, threads = sum(r[0] for r in res), processes   # the processes ran at the same time
        desc += (f"; {processes} spawned processes at once, one thread each, {sum(r[1] for r in res)} reps "
                 f"in ~{max(r[2] for r in res):.1f} s: {value:.4f} GB/s together")
    desc += f"; oracle quantize of {T} K+V vectors in {smp['t_quant']:.2f} s"
    return value, T / smp["t_quant"] / 1e6, threads, desc, gbs1, gbs, pool


def run_reference(args, w):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    # the oracle on the host's cores: min(16, cores) spawned processes, one BLAS thread each, each
    # step a bounded sample decoded in every process at once (the sum of their rates)
    import multiprocessing
    sample_s = 2.0
    threads = min(16, os.cpu_count() or 1)
    _, mtok, _, _, _, _, _ = cpu_oracle_sample(w, seconds=sample_s / 4, reps_max=1)
    with multiprocessing.get_context("spawn").Pool(threads) as mp:
        for i in range(args.warmup):
            mp.map(_oracle_worker, [(w.name, 99 + j, sample_s / 4) for j in range(threads)])
        vals, reps, t_all = [], 0, time.perf_counter()
        for i in range(args.steps):
            res = mp.map(_oracle_worker, [(w.name, 1234 + j, sample_s) for j in range(threads)])
            vals.append(sum(r[0] for r in res))
            reps += sum(r[1] for r in res)
        elapsed = time.perf_counter() - t_all
    value = statistics.mean(vals)
    desc = (f"oracle decode of 1 KV head x 1024 tokens (8 packed pages) for {w.group} query heads in {threads} "
            f"spawned processes at once, one BLAS thread each, ~{sample_s:.0f} s per step ({reps} reps in all)")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": elapsed / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "quantize_mtok_s": mtok,
            "config": {"workload": w.name, "batch": w.batch, "kv_heads": w.kv_heads, "q_heads": w.q_heads,
                       "tokens": w.tokens, "head_dim": w.d, "bits": w.b, "decode_steps": w.decode_steps,
                       "sample": "bounded CPU sample per step (see cpu_baseline)"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": desc},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args, w):
    import torch
    import torch.distributed as dist

    import kv_cache_vector_19_b300 as tq
    from kv_cache_vector_19_b300 import workloads

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world != args.gpus:
        raise SystemExit(f"--gpus {args.gpus} but WORLD_SIZE={world}")

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_oracle_sample(w, processes=min(16, os.cpu_count() or 1))   # before any GPU work

    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    wl = workloads.preset(w.name, seed=w.seed + rank)
    data = workloads.generate(wl)
    B, H, Hq, T, d, S = wl.batch, wl.kv_heads, wl.q_heads, wl.tokens, wl.d, wl.decode_steps
    appends = S > 1
    maxT = wl.max_tokens
    dev = torch.device("cuda", local)

    # pinned host copies (end-to-end leg) and device-resident copies (kernel leg)
    h_k, h_v, h_q = data["k"].pin_memory(), data["v"].pin_memory(), data["q"].pin_memory()
    k, v, q = h_k.to(dev), h_v.to(dev), h_q.to(dev)
    if appends:
        h_kn, h_vn = data["k_new"].pin_memory(), data["v_new"].pin_memory()
        kn, vn = h_kn.to(dev), h_vn.to(dev)
    del data

    ctx = tq.Context(d, wl.b, seed=wl.seed, device=local)
    cache = ctx.alloc_cache(B, H, maxT)
    ws = ctx.alloc_workspace(B, Hq, H, maxT)
    out = torch.empty(S, B, Hq, d, device=dev)
    h_out = torch.empty(S, B, Hq, d).pin_memory()
    zero = torch.zeros(B, dtype=torch.int32, device=dev)
    pos = torch.tensor([[T + s] * B for s in range(S)], dtype=torch.int32, device=dev)
    lens = pos + 1 if appends else torch.full((1, B), T, dtype=torch.int32, device=dev)

    tev = lambda: torch.cuda.Event(enable_timing=True)
    xev = lambda: torch.cuda.Event(enable_timing=True, external=True)
    call_ev = [(xev(), xev()) for _ in range(S)]

    # end-to-end prefill: batch row b's K/V copy from pinned memory runs on a copy stream while
    # row b - 1 is quantized (one tq_quantize_kv call per row, into that row's cache slice)
    copy_stream = torch.cuda.Stream(dev)
    row_ready = [torch.cuda.Event() for _ in range(B)]
    row_bytes = cache.numel() // B
    per_row = B > 1 and row_bytes % 256 == 0

    def prefill(copies):
        if not copies:
            ctx.quantize_kv(k, v, zero, cache, maxT)
            return
        if not per_row:
            k.copy_(h_k, non_blocking=True)
            v.copy_(h_v, non_blocking=True)
            ctx.quantize_kv(k, v, zero, cache, maxT)
            return
        cur = torch.cuda.current_stream(dev)
        copy_stream.wait_stream(cur)   # the previous step's readers of k and v are done
        for b in range(B):
            with torch.cuda.stream(copy_stream):
                k[b].copy_(h_k[b], non_blocking=True)
                v[b].copy_(h_v[b], non_blocking=True)
                row_ready[b].record(copy_stream)
            cur.wait_event(row_ready[b])
            ctx.quantize_kv(k[b:b + 1], v[b:b + 1], zero[b:b + 1], cache[b * row_bytes:(b + 1) * row_bytes], maxT)

    def decode_phase(copies, events):
        for s in range(S):
            if copies:
                q[s].copy_(h_q[s], non_blocking=True)
                if appends:
                    kn[s].copy_(h_kn[s], non_blocking=True)
                    vn[s].copy_(h_vn[s], non_blocking=True)
            if appends:
                ctx.quantize_kv(kn[s], vn[s], pos[s], cache, maxT)
            if events:
                call_ev[s][0].record()
            ctx.attn_decode(q[s], cache, lens[s], H, maxT, out[s], ws)
            if events:
                call_ev[s][1].record()
            if copies:
                h_out[s].copy_(out[s], non_blocking=True)

    # the decode phase is launch-bound from Python, so each variant is one CUDA graph
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):
        prefill(False)
        decode_phase(False, False)
    torch.cuda.current_stream(dev).wait_stream(side)
    torch.cuda.synchronize()
    g_dec, g_e2e = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_dec):
        decode_phase(False, True)
    with torch.cuda.graph(g_e2e):
        decode_phase(True, False)

    def barrier():
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    e_q0, e_q1, e_d1 = tev(), tev(), tev()

    def step():
        e_q0.record()
        prefill(False)
        e_q1.record()
        g_dec.replay()
        e_d1.record()

    for _ in range(args.warmup):
        step()
    st = ctx.device_status()
    if st != tq.TQ_OK:
        raise SystemExit(f"device status after warm-up: {tq.tq_status_string(st)}")

    q_ms, dphase_ms, dcall_ms = [], [], []
    barrier()
    t_start, t_end = tev(), tev()
    with ClockSampler(local) as clk:
        t_start.record()
        for _ in range(args.steps):
            step()
            torch.cuda.synchronize()     # read this step's events; a step is several ms
            q_ms.append(e_q0.elapsed_time(e_q1))
            dphase_ms.append(e_q1.elapsed_time(e_d1))
            dcall_ms.extend(a.elapsed_time(b) for a, b in call_ev)
        t_end.record()
        barrier()
    total_ms = t_start.elapsed_time(t_end)

    # end-to-end leg: the step's inputs come from pinned host memory and its outputs are
    # read back, inside the timed region
    e2e_steps = max(1, min(args.steps, 5))
    prefill(True)
    g_e2e.replay()
    barrier()
    e0, e1, e2 = tev(), tev(), tev()
    e2e_q, e2e_d = [], []
    for _ in range(e2e_steps):
        e0.record()
        prefill(True)
        e1.record()
        g_e2e.replay()
        e2.record()
        torch.cuda.synchronize()
        e2e_q.append(e0.elapsed_time(e1))
        e2e_d.append(e1.elapsed_time(e2))
    barrier()
    st = ctx.device_status()
    if st != tq.TQ_OK:
        raise SystemExit(f"device status after timing: {tq.tq_status_string(st)}")

    per_token = bpt(d, wl.b, wl.m)
    seq = [int(x) for x in lens[:, 0].tolist()]
    dec_bytes = sum(B * H * n * per_token + 2 * B * Hq * d * 4 for n in seq)
    per_launch_bytes = dec_bytes / S
    mean = lambda xs: sum(xs) / len(xs)
    t_dphase, t_q, t_call = mean(dphase_ms), mean(q_ms), mean(dcall_ms)
    t_e2e_d, t_e2e_q = mean(e2e_d), mean(e2e_q)
    t_dphase, t_q, t_call, total_ms, t_e2e_d, t_e2e_q = max_over_ranks(
        [t_dphase, t_q, t_call, total_ms, t_e2e_d, t_e2e_q], world, dev)
    value = job_gbs(world, dec_bytes, t_dphase)
    peak, peak_kind = read_peaks()
    achieved = per_launch_bytes / (t_call * 1e-3) / 1e9
    h2d = (h_k.numel() + h_v.numel()) * 2 + h_q.numel() * 4 + ((h_kn.numel() + h_vn.numel()) * 2 if appends else 0)
    d2h = h_out.numel() * 4
    launches_per_step = tq.binding.QUANTIZE_LAUNCHES * (1 + (S if appends else 0)) + tq.binding.DECODE_LAUNCHES * S
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": DTYPE,
        "data": "synthetic (seeded bf16 K/V, fp32 queries; no model weights)",
        "config": {"workload": f"{wl.name}: batch {B}, {H} KV / {Hq} query heads, head_dim {d}, b={wl.b}, "
                               f"{T} prefill tokens + {S} decode step(s)",
                   "batch": B, "kv_heads": H, "q_heads": Hq, "tokens": T, "head_dim": d, "bits": wl.b,
                   "decode_steps": S, "parallelism": f"replicas x{world} (independent sequences per GPU)",
                   "l2": "inputs larger than L2 (compressed cache and bf16 K/V are each > 126 MB)"},
        "quantize_mtok_s": world * B * T / (t_q * 1e-3) / 1e6,
        "quantize_ms": t_q,
        "decode_us_per_step": t_dphase / S * 1e3,
        "decode_call_us": t_call * 1e3,
        "roofline": {"bound": "hbm", "kernel": f"tq_attn_decode ({DECODE_KERNEL} + prologue + combine)",
                     "achieved": achieved, "peak": peak,
                     "unit": "GB/s", "frac": achieved / peak, "peak_kind": peak_kind,
                     "traffic": committed_traffic(), "traffic_source": TRAFFIC_PROFILE,
                     "source_fingerprint": source_fingerprint(), "algorithmic_bytes_per_launch": per_launch_bytes},
        "e2e": {"value": job_gbs(world, dec_bytes, t_e2e_q + t_e2e_d), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": t_e2e_q + t_e2e_d,
                "note": f"decode bytes over the whole step: prefill K/V copy + quantize (the copy of batch row "
                        f"b + 1 overlapping the quantize of row b), then {S} x (copies, append, decode, read-back)",
                "decode_phase_gbs": job_gbs(world, dec_bytes, t_e2e_d),
                "quantize_mtok_s": world * B * T / (t_e2e_q * 1e-3) / 1e6},
        "gpu_launches": args.steps * launches_per_step,
        "clocks": clk.summary(),
    }
    if cpu is not None:
        gbs, mtok, threads, desc, gbs1, gbs_pool, pool = cpu
        line["cpu_baseline"] = {"value": gbs, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": desc,
                                "quantize_mtok_s": mtok, "value_1_thread": gbs1, "value_blas_pool": gbs_pool,
                                "blas_pool_threads": pool}
    if rank == 0:
        print(json.dumps(line), flush=True)
    del g_dec, g_e2e
    ctx.close()
    if world > 1:
        dist.destroy_process_group()
    return 0


def run_sweep(args):
    """Per (d, b) point of the bit/dim sweep (1 KV head, 65,536 tokens, 16 queries): quantize
    Mtokens/s, decode us and GB/s, normalized reconstruction MSE of keys and values (from
    tq_dequantize_kv) and the bias / RMS of the inner-product error <q, k^> - <q, k>."""
    import torch

    import kv_cache_vector_19_b300 as tq
    from kv_cache_vector_19_b300 import workloads

    for d in (64, 128, 256):
        for b in (2, 3, 4, 5):
            w = workloads.sweep_point(d, b)
            data = workloads.generate(w)
            T, nq = w.tokens, w.extra["n_queries"]
            ctx = tq.Context(d, b, seed=w.seed)
            cache = ctx.alloc_cache(1, 1, T)
            ws = ctx.alloc_workspace(1, nq, 1, T)
            k, v = data["k"].cuda(), data["v"].cuda()
            q = data["q"][0].cuda().reshape(1, nq, d).contiguous()
            out = torch.empty_like(q)
            zero = torch.zeros(1, dtype=torch.int32, device="cuda")
            lens = torch.full((1,), T, dtype=torch.int32, device="cuda")
            e = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
            for _ in range(args.warmup):
                ctx.quantize_kv(k, v, zero, cache, T)
                ctx.attn_decode(q, cache, lens, 1, T, out, ws)
            torch.cuda.synchronize()
            e[0].record()
            for _ in range(args.steps):
                ctx.quantize_kv(k, v, zero, cache, T)
            e[1].record()
            for _ in range(args.steps):
                ctx.attn_decode(q, cache, lens, 1, T, out, ws)
            e[2].record()
            torch.cuda.synchronize()
            tq_ms = e[0].elapsed_time(e[1]) / args.steps
            td_ms = e[1].elapsed_time(e[2]) / args.steps
            nbytes = T * bpt(d, b, d)
            # reconstruction and inner-product error of the cached vectors (tq_dequantize_kv)
            khat = torch.empty(1, 1, T, d, device="cuda")
            vhat = torch.empty(1, 1, T, d, device="cuda")
            ctx.dequantize_kv(cache, zero, 1, 1, T, T, khat, vhat)
            kx, vx = k[0, 0].float(), v[0, 0].float()
            kh, vh = khat[0, 0], vhat[0, 0]
            nmse_k = ((kh - kx).pow(2).sum(-1) / kx.pow(2).sum(-1).clamp_min(1e-30)).mean().item()
            nmse_v = ((vh - vx).pow(2).sum(-1) / vx.pow(2).sum(-1).clamp_min(1e-30)).mean().item()
            qq = q[0].float()                      # [nq, d]
            exact = kx @ qq.t()                    # <q, k> for every token and query
            err = kh @ qq.t() - exact
            st = ctx.device_status()
            if st != tq.TQ_OK:
                raise SystemExit(f"device status in sweep d={d} b={b}: {tq.tq_status_string(st)}")
            print(json.dumps({"sweep_point": f"d{d}_b{b}", "head_dim": d, "bits": b, "tokens": T,
                              "queries": nq, "quantize_mtok_s": T / tq_ms / 1e3, "decode_us": td_ms * 1e3,
                              "decode_gbs": nbytes / td_ms / 1e6, "compressed_bytes": nbytes,
                              "bytes_per_token": bpt(d, b, d), "compression_vs_bf16": 4 * d / bpt(d, b, d),
                              "recon_nmse_k": nmse_k, "recon_nmse_v": nmse_v,
                              "ip_bias": err.mean().item(), "ip_rms": err.pow(2).mean().sqrt().item(),
                              "ip_rms_rel": (err.pow(2).mean() / exact.pow(2).mean()).sqrt().item()}),
                  flush=True)
            ctx.close()
    return 0


def run_case(args, w):
    """One kernel of the workload, alone, at a reduced prefill length: the cases the ncu
    summaries under profiles/ are taken on.  --kernel-case quantize runs tq_quantize_kv of the
    prefill; decode runs tq_attn_decode over it; scan runs tq_ip_topk (top --topk keys per query
    head) over it.  warmup + steps calls; prints the mean device time of the timed calls (CUDA
    events on the launching stream), no JSON line."""
    import torch

    import kv_cache_vector_19_b300 as tq
    from kv_cache_vector_19_b300 import workloads

    wl = workloads.preset(w.name, tokens=args.tokens or w.tokens, decode_steps=1)
    data = workloads.generate(wl)
    B, H, Hq, T, d = wl.batch, wl.kv_heads, wl.q_heads, wl.tokens, wl.d
    ctx = tq.Context(d, wl.b, seed=wl.seed, decode_path=args.decode_path)
    if args.sparse_v:
        ctx.set_sparse_v(args.sparse_v)
    k, v = data["k"].cuda(), data["v"].cuda()
    if args.token_major:   # a prefill projection's [B, T, H, d], quantized through strides
        k = k.permute(0, 2, 1, 3).contiguous().permute(0, 2, 1, 3)
        v = v.permute(0, 2, 1, 3).contiguous().permute(0, 2, 1, 3)
    zero = torch.zeros(B, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()
    if args.paged:   # a pool of blocks in a seeded random order, one table row per sequence
        max_blocks = (T + 127) // 128
        n_blocks = B * max_blocks
        perm = torch.randperm(n_blocks, generator=torch.Generator().manual_seed(wl.seed + 1))
        table = perm.to(torch.int32).reshape(B, max_blocks).cuda()
        cache = ctx.alloc_pool(H, n_blocks)
        T = 128 * max_blocks

        def quantize():
            if args.token_major:
                ctx.quantize_kv_paged_strided(k, v, zero, cache, n_blocks, table)
            else:
                ctx.quantize_kv_paged(k, v, zero, cache, n_blocks, table)
    else:
        cache = ctx.alloc_cache(B, H, T)

        def quantize():
            if args.token_major:
                ctx.quantize_kv_strided(k, v, zero, cache, T)
            else:
                ctx.quantize_kv(k, v, zero, cache, T)
    if args.kernel_case == "quantize":
        call = quantize
    elif args.kernel_case == "append":   # one token per sequence into the last slot of the prefill
        quantize()
        kn = torch.randn(B, H, 1, d, generator=torch.Generator().manual_seed(wl.seed + 2)).to(torch.bfloat16).cuda()
        vn = torch.randn(B, H, 1, d, generator=torch.Generator().manual_seed(wl.seed + 3)).to(torch.bfloat16).cuda()
        at = torch.full((B,), wl.tokens - 1, dtype=torch.int32, device="cuda")

        def call():
            if args.paged:
                ctx.quantize_kv_paged(kn, vn, at, cache, n_blocks, table)
            else:
                ctx.quantize_kv(kn, vn, at, cache, T)
    else:
        quantize()
        q = (data["q"][0] * args.q_scale).cuda().contiguous()
        lens = torch.full((B,), wl.tokens, dtype=torch.int32, device="cuda")
        if args.kernel_case == "decode":
            ws = ctx.alloc_workspace(B, Hq, H, T)
            out = torch.empty_like(q)
            if args.paged:
                def call():
                    ctx.attn_decode_paged(q, cache, n_blocks, table, lens, H, out, ws)
            else:
                def call():
                    ctx.attn_decode(q, cache, lens, H, T, out, ws)
        else:
            if args.paged:
                raise SystemExit("--paged applies to the quantize and decode cases")
            kk = args.topk
            ws = ctx.alloc_topk_workspace(B, Hq, H, T)
            oi = torch.empty(B, Hq, kk, dtype=torch.int32, device="cuda")
            osc = torch.empty(B, Hq, kk, dtype=torch.float32, device="cuda")

            def call():
                ctx.ip_topk(q, cache, lens, H, T, kk, out_idx=oi, out_score=osc, workspace=ws)
    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        call()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / max(args.steps, 1)
    st = ctx.device_status()
    cache_mb = cache.numel() * cache.element_size() / 1e6
    ctx.close()
    if st != tq.TQ_OK:
        raise SystemExit(f"device status: {tq.tq_status_string(st)}")
    extra = (" (paged pool)" if args.paged else "") + (f" (sparse V {args.sparse_v:g})" if args.sparse_v else "")
    extra += (f" (queries x{args.q_scale:g})" if args.q_scale != 1.0 else "")
    extra += (f" ({args.decode_path} decode)" if args.decode_path != "auto" else "")
    extra += (" (token-major K/V through strides)" if args.token_major else "")
    print(f"{args.kernel_case} case{extra}: {w.name}, {wl.tokens} tokens, "
          f"{args.warmup + args.steps} calls, status ok, "
          f"{ms * 1e3:.1f} us per call (back to back, cache {cache_mb:.0f} MB)", flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="longctx", choices=["longctx", "llama8b", "llama70b", "tiny"])
    ap.add_argument("--sweep", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--kernel-case", choices=["quantize", "decode", "scan", "append"], default=None,
                    help="run one kernel of the workload alone (profiling case), no JSON line")
    ap.add_argument("--tokens", type=int, default=0, help="prefill length of --kernel-case (default: workload's)")
    ap.add_argument("--topk", type=int, default=100, help="k of --kernel-case scan")
    ap.add_argument("--sparse-v", type=float, default=0.0, help="Sparse V threshold of the kernel cases")
    ap.add_argument("--q-scale", type=float, default=1.0,
                    help="query scale of the kernel cases (larger: more peaked attention)")
    ap.add_argument("--decode-path", default="auto", choices=["auto", "simt", "mma", "tc", "tc4"],
                    help="decode kernel of the kernel cases")
    ap.add_argument("--token-major", action="store_true",
                    help="kernel cases: K/V stored [B, T, H, d] and quantized through strides")
    ap.add_argument("--paged", action="store_true",
                    help="--kernel-case quantize / decode on a block pool through a shuffled block table")
    args = ap.parse_args()
    if args.warmup < 3 and not args.sweep:
        args.warmup = 3
    from kv_cache_vector_19_b300 import workloads
    w = workloads.preset(args.workload)
    if args.impl == "reference":
        return run_reference(args, w)
    if args.sweep:
        return run_sweep(args)
    if args.kernel_case:
        return run_case(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
