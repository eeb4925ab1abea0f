#!/usr/bin/env python
"""Decode-step benchmark of the 4-bit paged KV cache on GB300.

One step is the whole decode hot path for one batch: each request's new
token quantised into the NVFP4 pool and decode attention (split-KV kernel +
log-sum-exp combine) over every request's full context, in one
kv4_decode_step call (the decode kernel writes the new tokens itself; the
same step as kv4_write + kv4_decode_attention, which is timed beside it).  The
headline workload is a Qwen3.8-27B-shaped full-attention layer at 32K
context (4 KV heads, 24 query heads, head dim 256, batch 16, lengths uniform
in [24576, 32768], 64-token pages); the pool (about 0.53 GB) is far larger
than L2, so every step streams it from HBM.

Printed: one JSON line on rank 0 with the metric (achieved HBM GB/s of the
step's algorithmic bytes), the roofline of the decode kernel, an end-to-end
figure through the public API with host buffers (every step's inputs
copied in and its output copied back, on copy streams that overlap the
kernels of the neighbouring steps), the oracle timed on the host cores, clock samples, and per-workload lines for 160K, 1M, the INT4
lane and the prefix dequant under "workloads".

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl kv4|reference]
Multi-GPU runs (torchrun) are independent replicas (weak scaling): each rank
decodes its own batch; only the timing is reduced (max over ranks).
"""
import argparse
import hashlib
import re
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "NVFP4 decode-attn achieved HBM GB/s (% of peak) at 32K/160K/1M ctx"
FALLBACK_BF16_TFLOPS = 1900.0
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 1024 * 1024


# ----------------------------------------------------------------------------- helpers
def algorithmic_decode_bytes(w, lens, fmt=None):
    """Bytes a decode call must move: every cached token's K and V codes and
    scales for every kv head, plus q in and out (fp32) out."""
    fmt = fmt or w.fmt
    D = w.head_dim
    per_token_head = {"nvfp4": 2 * (D // 2 + D // 16), "int4": 2 * (D // 2 + 4), "fp8": 2 * D}[fmt]
    kv = int(np.sum(lens, dtype=np.int64)) * w.num_kv_heads * per_token_head
    return kv + len(lens) * w.num_q_heads * D * (2 + 4)


def algorithmic_write_bytes(w, T, in_bytes=2):
    """Bytes of one write of T tokens: K and V in (in_bytes per element: 2 for
    bf16, 1 for FP8), the pool rows out, and the slot mapping."""
    D = w.head_dim
    per_row = {"nvfp4": 2 * (D // 2 + D // 16), "int4": 2 * (D // 2 + 4), "fp8": 2 * D}[w.fmt]
    return T * w.num_kv_heads * (2 * D * in_bytes + per_row) + T * 8


def read_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def read_tensor_peak():
    """(dense f16/bf16 tensor TFLOP/s burst, source).  kind::f16 runs f16 and
    bf16 operands at the same rate, so the measured bf16 GEMM peak serves."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["bf16_tflops"]), "measured bf16_tflops (burst)"
    except Exception:
        return FALLBACK_BF16_TFLOPS, "fallback"


DECODE_SOURCES = ("kv4_decode4.cu", "kv4_decode.cu", "kv4_device.cuh")


def decode_source_hash():
    """Hash of the decode kernels' code (the NVFP4 / INT4 / k8v4 kernel, the
    FP8 split kernel and combine, their device helpers) with comments and
    blank space removed, so a recorded ncu traffic figure survives comment
    edits but not code changes."""
    h = hashlib.sha256()
    for f in DECODE_SOURCES:
        with open(os.path.join(ROOT, "bit_paged_kv_kv4_gb300", "csrc", f)) as fh:
            src = fh.read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        src = re.sub(r"//[^\n]*", "", src)
        h.update("".join(src.split()).encode())
    return h.hexdigest()[:16]


def recorded_ncu(workload):
    """The ncu capture of one decode launch recorded in profiles/ (DRAM bytes,
    duration under ncu), if it was taken on the current decode source; else
    None."""
    p = os.path.join(ROOT, "profiles", "decode_traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
        e = d.get(workload)
        if e and e.get("source_hash") == decode_source_hash():
            return e
    except Exception:
        pass
    return None


def recorded_traffic(workload):
    """ncu DRAM bytes per decode launch (read + write), or None."""
    e = recorded_ncu(workload)
    return float(e["dram_bytes_per_launch"]) if e else None


def recorded_ncu_gbs(workload):
    """ncu DRAM bytes / ncu kernel duration of the recorded launch, GB/s."""
    e = recorded_ncu(workload)
    if not e or not e.get("gpu_time_duration_ns_under_ncu"):
        return None
    return float(e["dram_bytes_per_launch"]) / float(e["gpu_time_duration_ns_under_ncu"])


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"kv4_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None:
            return None
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        try:
            for line in open(self.path):
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        except OSError:
            return None
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


# ----------------------------------------------------------------------------- device setup
class Setup:
    """A workload's pool filled through kv4_write, plus one decode step's inputs.
    keep_kv=True keeps every request's bf16 K/V on the device (for tests)."""

    def __init__(self, w, device, seed_offset=0, num_splits=None, keep_kv=False, fill=None):
        import torch
        import bit_paged_kv_kv4_gb300 as K
        self.w, self.K, self.torch = w, K, torch
        self.device = device
        self.lens = w.seq_lens()
        self.num_pages, self.table = w.block_table(self.lens)
        B, Hkv, Hq, D, P = w.batch, w.num_kv_heads, w.num_q_heads, w.head_dim, w.page_size
        self.pool = K.Pool(w.fmt, self.num_pages, P, Hkv, D, device=device)
        if fill is not None:
            self.pool.buffer.fill_(fill)
        kvs = []
        amax = torch.zeros(2, device=device)
        for b in range(B):
            kv = W.device_kv(w, b, int(self.lens[b]), device)
            amax = torch.maximum(amax, kv.abs().amax(dim=(1, 2, 3)).float())
            kvs.append(kv)
        am = amax.cpu().numpy()
        scale_of = W.fp8_scale_from_amax if w.fmt == "fp8" else W.global_scale_from_amax
        self.g_host = np.array([scale_of(am[0]), scale_of(am[1])], np.float32)
        self.g = torch.from_numpy(self.g_host).to(device)
        for b in range(B):
            L = int(self.lens[b])
            slots = torch.from_numpy(W.slots_for(self.table[b], P, np.arange(L))).to(device)
            K.kv4_write(kvs[b][0], kvs[b][1], slots, self.pool, self.g)
        self.kv = kvs if keep_kv else None
        del kvs
        torch.cuda.empty_cache()
        # the step's inputs: q, and each request's newest token (position L-1)
        self.q, self.k_new, self.v_new = W.device_q(w, device, salt=seed_offset)
        self.slot_new = torch.from_numpy(np.array(
            [W.slots_for(self.table[b], P, [int(self.lens[b]) - 1])[0] for b in range(B)],
            np.int64)).to(device)
        self.d_table = torch.from_numpy(self.table).to(device)
        self.d_lens = torch.from_numpy(self.lens).to(device)
        self.splits = num_splits if num_splits is not None else w.num_splits
        self.ws = K.alloc_workspace(B, Hq, D, self.splits, device=device)
        self.out = torch.empty((B, Hq, D), dtype=torch.float32, device=device)
        self.sm = float(w.sm_scale())
        torch.cuda.synchronize()
        assert K.kv4_device_error() == 0

    def write(self):
        self.K.kv4_write(self.k_new, self.v_new, self.slot_new, self.pool, self.g)

    def decode(self):
        self.K.kv4_decode_attention(self.q, self.pool, self.g, self.d_table, self.d_lens, self.sm,
                                    self.out, num_splits=self.splits, workspace=self.ws)

    @property
    def fused(self):
        """NVFP4 and INT4 have the one-call step; the FP8 comparison format not."""
        return self.w.fmt != "fp8"

    def step(self):
        """write() + decode(), in one kv4_decode_step call where the format has
        it (the decode kernel quantises the new tokens)."""
        if not self.fused:
            self.write()
            self.decode()
            return
        self.K.kv4_decode_step(self.q, self.k_new, self.v_new, self.pool, self.g, self.d_table, self.d_lens,
                               self.sm, self.out, num_splits=self.splits, workspace=self.ws)

    def launches_per_step(self):
        return (0 if self.fused else 1) + 1 + (0 if self.splits == 1 else 1)


def time_calls(run, iters, rounds=3):
    """Mean GPU time of one call: `iters` back-to-back calls between two CUDA
    events on the launching stream, after 3 warm-up calls; the median over
    `rounds` such runs.  A bounded GPU delay (a fixed number of clock cycles,
    about 75 us per call) is queued before the first event, so the host has
    issued every call before the clock starts and no host time between calls
    is counted."""
    import torch
    for _ in range(3):
        run()
    torch.cuda.synchronize()
    sleep = getattr(torch.cuda, "_sleep", None)
    means = []
    for _ in range(rounds):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if sleep is not None:
            sleep(int(1_000_000 + 150_000 * iters))
        a.record()
        for _ in range(iters):
            run()
        b.record()
        torch.cuda.synchronize()
        means.append(a.elapsed_time(b) * 1e-3 / iters)
    return statistics.median(means)


def time_decode_only(s, iters):
    torch = s.torch
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(iters)]
    for _ in range(3):
        s.decode()
    torch.cuda.synchronize()
    for a, b in ev:
        a.record()
        s.decode()
        b.record()
    torch.cuda.synchronize()
    return [a.elapsed_time(b) * 1e-3 for a, b in ev]


# ----------------------------------------------------------------------------- CPU oracle
def cpu_oracle_sample(name, seconds, max_steps=None):
    """Time the oracle's FP64 decode attention on one request and kv head of
    the workload (its whole context), repeated for about `seconds`.
    Returns dict(value GB/s, steps, seconds_per_step, tokens)."""
    import oracle
    from oracle import pool as OP
    w = W.ALL[name]
    lens = w.seq_lens()
    b, h = 0, 0
    L = int(lens[b])
    k, v = w.kv_request(b, h, L)
    g = np.array([W.global_scale_from_amax(np.abs(W.bf16_bits_to_f32(k)).max()),
                  W.global_scale_from_amax(np.abs(W.bf16_bits_to_f32(v)).max())], np.float32)
    P = w.page_size
    npg = (L + P - 1) // P
    spec = OP.PoolSpec(w.fmt, npg, P, 1, w.head_dim)
    pool = OP.new_pool(spec)
    table = np.arange(npg, dtype=np.int32)[None]
    OP.write(pool, spec, k[:, None], v[:, None], W.slots_for(table[0], P, np.arange(L)), g)
    q = w.q()[b:b + 1, h * w.group:(h + 1) * w.group]
    one = W.Workload(w.name, w.fmt, 1, w.group, w.head_dim, 1, P, L, L)
    bytes_per = algorithmic_decode_bytes(one, [L])
    times = []
    t_end = time.perf_counter() + seconds
    while (max_steps is None and (time.perf_counter() < t_end or len(times) < 2)) or \
            (max_steps is not None and len(times) < max_steps):
        t0 = time.perf_counter()
        oracle.attention.decode_attention(q, pool, spec, g, table, np.array([L], np.int32), w.sm_scale())
        times.append(time.perf_counter() - t0)
    per = statistics.median(times)
    return {"value": bytes_per / per / 1e9, "steps": len(times), "seconds_per_step": per,
            "tokens": L, "bytes_per_step": bytes_per, "times": times}


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def run_cpu_oracle_subprocess(name, seconds, max_steps=None, threads=1):
    n = str(threads)
    env = dict(os.environ, OMP_NUM_THREADS=n, OPENBLAS_NUM_THREADS=n, MKL_NUM_THREADS=n,
               CUDA_VISIBLE_DEVICES="")
    code = ("import json,sys; sys.path.insert(0, %r); import bench; "
            "r = bench.cpu_oracle_sample(%r, %r, %r); r.pop('times'); print(json.dumps(r))"
            % (ROOT, name, seconds, max_steps))
    out = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                         timeout=max(600, 20 * seconds))
    if out.returncode != 0:
        raise RuntimeError(out.stderr[-2000:])
    return json.loads(out.stdout.strip().splitlines()[-1])


def _oracle_unit_worker(name, b, h, seconds, barrier, queue):
    """One process of the all-cores oracle baseline: unit (request b, kv
    head h) of the workload, its decode attention repeated for `seconds`
    after every process has built its pool (the barrier)."""
    import oracle
    from oracle import pool as OP
    w = W.ALL[name]
    L = int(w.seq_lens()[b])
    k, v = w.kv_request(b, h, L)
    g = np.array([W.global_scale_from_amax(np.abs(W.bf16_bits_to_f32(k)).max()),
                  W.global_scale_from_amax(np.abs(W.bf16_bits_to_f32(v)).max())], np.float32)
    P = w.page_size
    npg = (L + P - 1) // P
    spec = OP.PoolSpec(w.fmt, npg, P, 1, w.head_dim)
    pool = OP.new_pool(spec)
    table = np.arange(npg, dtype=np.int32)[None]
    OP.write(pool, spec, k[:, None], v[:, None], W.slots_for(table[0], P, np.arange(L)), g)
    q = w.q()[b:b + 1, h * w.group:(h + 1) * w.group]
    one = W.Workload(w.name, w.fmt, 1, w.group, w.head_dim, 1, P, L, L)
    bytes_per = algorithmic_decode_bytes(one, [L])
    barrier.wait(timeout=600)
    steps, t0 = 0, time.perf_counter()
    while steps < 1 or time.perf_counter() - t0 < seconds:
        oracle.attention.decode_attention(q, pool, spec, g, table, np.array([L], np.int32), w.sm_scale())
        steps += 1
    queue.put((bytes_per * steps, time.perf_counter() - t0, steps))


def cpu_oracle_all_cores(name, seconds, procs):
    """The oracle on `procs` host cores at once: one single-threaded process
    per (request, kv head) unit of the workload (units taken in order), all
    timing together.  Spawned processes (never forked after CUDA start-up).
    Returns the summed rate and what was run."""
    import multiprocessing as mp
    w = W.ALL[name]
    units = [(b, h) for b in range(w.batch) for h in range(w.num_kv_heads)][:procs]
    ctx = mp.get_context("spawn")
    barrier, queue = ctx.Barrier(len(units)), ctx.Queue()
    saved = {k: os.environ.get(k) for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS",
                                             "CUDA_VISIBLE_DEVICES")}
    os.environ.update(OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
                      CUDA_VISIBLE_DEVICES="")
    try:
        ps = [ctx.Process(target=_oracle_unit_worker, args=(name, b, h, seconds, barrier, queue))
              for b, h in units]
        for p in ps:
            p.start()
        res, t_give_up = [], time.time() + max(600, 20 * seconds)
        while len(res) < len(ps):
            try:
                res.append(queue.get(timeout=1.0))
            except Exception:       # queue.Empty: check the workers are still alive
                if any(p.exitcode not in (None, 0) for p in ps) or time.time() > t_give_up:
                    for p in ps:
                        if p.is_alive():
                            p.terminate()
                    raise RuntimeError("an oracle worker process failed or ran out of time")
        for p in ps:
            p.join(timeout=60)
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    rate = sum(nbytes / dt for nbytes, dt, _ in res)
    return {"value": rate / 1e9, "procs": len(units), "steps": sum(st for _, _, st in res),
            "units": units}


# ----------------------------------------------------------------------------- arms
def dist_setup(args):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1:
        import torch.distributed as dist
        import torch
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
        pg = dist
    return rank, world, local, pg


def barrier(pg, device=None):
    if pg is not None:
        import torch
        if device is not None and pg.get_backend() == "nccl":
            pg.barrier(device_ids=[device.index])
        else:
            pg.barrier()


def max_over_ranks(pg, x, device=None):
    if pg is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device if pg.get_backend() == "nccl" else "cpu")
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def step_config(w, lens, splits, pool_bytes, world):
    """The bench line's `config` for workload w (both arms print the same)."""
    dec_bytes = algorithmic_decode_bytes(w, lens)
    return {"workload": f"{w.name}: " + w.notes, "kv_heads": w.num_kv_heads, "q_heads": w.num_q_heads,
            "head_dim": w.head_dim, "batch": w.batch, "page_size": w.page_size,
            "seq_lens": [int(x) for x in lens], "num_splits": splits,
            "kv_bytes_per_step": dec_bytes, "step_bytes": dec_bytes + algorithmic_write_bytes(w, w.batch),
            "l2": "inputs larger than L2: the pool is %.0f MB vs 129 MB L2" % (pool_bytes / 1e6),
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}


def reference_arm(args):
    rank, world, local, pg = dist_setup(args)
    if rank != 0:
        return 0
    w = W.ALL[args.workload]
    lens = w.seq_lens()
    num_pages, _ = w.block_table(lens)
    # the pool's bytes: num_pages chunks of P tokens per kv head
    pool_bytes = num_pages * w.page_size * (algorithmic_decode_bytes(w, [1]) - w.num_q_heads * w.head_dim * 6)
    r = cpu_oracle_sample(w.name, 0, max_steps=args.warmup + args.steps)
    times = r["times"][args.warmup:]
    per = statistics.mean(times)
    value = r["bytes_per_step"] / per / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": per * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": step_config(w, lens, w.num_splits, pool_bytes, world),
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": f"one request x one kv head of {w.name} (request 0, kv head 0, "
                                   f"{w.group} query heads, {r['tokens']} tokens), {args.steps} timed steps"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def kv4_arm(args):
    import torch
    import bit_paged_kv_kv4_gb300 as K
    rank, world, local, pg = dist_setup(args)
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    K.load(build_if_missing=True)

    w = W.ALL[args.workload]
    s = Setup(w, device, seed_offset=rank)
    B, Hkv, Hq, D = w.batch, w.num_kv_heads, w.num_q_heads, w.head_dim
    dec_bytes = algorithmic_decode_bytes(w, s.lens)
    step_bytes = dec_bytes + algorithmic_write_bytes(w, B)

    # ---- device-resident timed region -----------------------------------
    for _ in range(args.warmup):
        s.step()
    torch.cuda.synchronize()
    # The decode call's own average duration (the roofline's kernel time): the
    # same kv4_decode_attention call back to back between two events, at least
    # 200 times (a run's start-up, about one call's host time before the first
    # launch, spread over fewer calls would read as kernel time).
    n_roof = max(args.steps, 200)
    d_start = torch.cuda.Event(enable_timing=True)
    d_end = torch.cuda.Event(enable_timing=True)
    # The timed steps: K kv4_decode_step calls back to back (the value).
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    # The same K steps as two calls each, kv4_write then kv4_decode_attention.
    u_start = torch.cuda.Event(enable_timing=True)
    u_end = torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    with clocks:
        barrier(pg, device)
        torch.cuda.synchronize()
        d_start.record()
        for i in range(n_roof):
            s.decode()
        d_end.record()
        torch.cuda.synchronize()
        barrier(pg, device)
        t_start.record()
        for i in range(args.steps):
            s.step()
        t_end.record()
        torch.cuda.synchronize()
        barrier(pg, device)
        u_start.record()
        for i in range(args.steps):
            s.write()
            s.decode()
        u_end.record()
        torch.cuda.synchronize()
        barrier(pg, device)
    total = t_start.elapsed_time(t_end) * 1e-3
    total = max_over_ranks(pg, total, device)
    dec_avg = max_over_ranks(pg, d_start.elapsed_time(d_end) * 1e-3 / n_roof, device)
    split_step = max_over_ranks(pg, u_start.elapsed_time(u_end) * 1e-3 / args.steps, device)
    err = K.kv4_device_error()
    if err != 0:
        raise SystemExit(f"device error {err} during the timed region")
    per_step = total / args.steps
    value = step_bytes * world / per_step / 1e9

    peak, peak_src = read_peaks()
    achieved = dec_bytes / dec_avg / 1e9

    # ---- end to end through the public API, host buffers ----------------
    # The step's inputs (q, the new K/V, the lengths) sit in one
    # pinned host staging buffer and go over in one copy per step into a
    # device buffer, of which the library's arguments are views (each part
    # 256-byte aligned); the step's output comes back into pinned host memory.
    # The copies run on their own streams, as a serving loop would run them:
    # step k+1's inputs go over while step k computes, step k's output comes
    # back while step k+1 computes (two device input buffers and two outputs,
    # each reused only after the copy or the kernels that used it are done).
    parts = [s.q, s.k_new, s.v_new, s.d_lens] + ([] if s.fused else [s.slot_new])
    offs, at = [], 0
    for t in parts:
        offs.append(at)
        at += (t.numel() * t.element_size() + 255) // 256 * 256
    h_in = torch.empty(at, dtype=torch.uint8).pin_memory()
    d_in = [torch.empty(at, dtype=torch.uint8, device=device) for _ in range(2)]
    views = [[], []]
    for t, o in zip(parts, offs):
        n = t.numel() * t.element_size()
        h_in[o:o + n].copy_(t.contiguous().view(torch.uint8).reshape(-1).cpu())
        for j in range(2):
            views[j].append(d_in[j][o:o + n].view(t.dtype).view(t.shape))
    d_out = [torch.empty_like(s.out) for _ in range(2)]
    h_out = [torch.empty((B, Hq, D), dtype=torch.float32).pin_memory() for _ in range(2)]
    h2d = h_in.numel()                       # the staging buffer, alignment padding included
    d2h = h_out[0].numel() * h_out[0].element_size()
    main = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def e2e_step(k):
        j = k % 2
        d_q, d_k, d_v, d_lens = views[j][:4]
        if k >= 2:
            s_in.wait_event(ev_done[j])          # step k-2's kernels are done with d_in[j]
        with torch.cuda.stream(s_in):
            d_in[j].copy_(h_in, non_blocking=True)
        ev_in[j].record(s_in)
        main.wait_event(ev_in[j])
        if k >= 2:
            main.wait_event(ev_out[j])           # step k-2's output has left d_out[j]
        if s.fused:
            K.kv4_decode_step(d_q, d_k, d_v, s.pool, s.g, s.d_table, d_lens, s.sm, d_out[j],
                              num_splits=s.splits, workspace=s.ws, stream=main)
        else:
            K.kv4_write(d_k, d_v, views[j][4], s.pool, s.g, stream=main)
            K.kv4_decode_attention(d_q, s.pool, s.g, s.d_table, d_lens, s.sm, d_out[j],
                                   num_splits=s.splits, workspace=s.ws, stream=main)
        ev_done[j].record(main)
        s_out.wait_event(ev_done[j])
        with torch.cuda.stream(s_out):
            h_out[j].copy_(d_out[j], non_blocking=True)
        ev_out[j].record(s_out)

    def e2e_run(n):
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        start.record(main)
        s_in.wait_event(start)
        s_out.wait_event(start)
        for k in range(n):
            e2e_step(k)
        main.wait_stream(s_in)
        main.wait_stream(s_out)                  # the last output is back
        end.record(main)
        return start, end

    e2e_run(args.warmup)
    torch.cuda.synchronize()
    barrier(pg, device)
    e0, e1 = e2e_run(args.steps)
    torch.cuda.synchronize()
    # the output read back is the decode of the same inputs over the same pool
    if not torch.equal(h_out[(args.steps - 1) % 2], s.out.cpu()):
        raise SystemExit("the end-to-end output differs from the device-timed decode of the same inputs")
    e2e_total = max_over_ranks(pg, e0.elapsed_time(e1) * 1e-3, device)
    e2e_value = step_bytes * world / (e2e_total / args.steps) / 1e9

    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": per_step * 1e3,
        "step": ("kv4_decode_step (new-token write inside the decode kernel) + combine" if s.fused
                 else "kv4_write + kv4_decode_attention"),
        "ms_per_step_as_write_then_decode": split_step * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16*f16+f32 (nvfp4 cache)",
        "data": "synthetic",
        "config": step_config(w, s.lens, s.splits, s.pool.nbytes, world),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": recorded_traffic(w.name),
                     "ncu_dram_gbs": recorded_ncu_gbs(w.name),
                     "kernel": "decode4_kernel<256, NVFP4> + combine_kernel (kv4_decode_attention)",
                     "peak_source": f"{peak_src} hbm_gbs", "decode_us": dec_avg * 1e6,
                     "decode_timing": f"mean of {n_roof} back-to-back kv4_decode_attention calls between "
                                      "two CUDA events on the launching stream, before the timed steps",
                     "tokens_per_s_16_layers": B / (16 * dec_avg)},
        "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_total / args.steps * 1e3},
        "gpu_launches": args.steps * s.launches_per_step(),
        "clocks": clocks.summary(),
    }
    # back-to-back decode calls of the same workload, for the FP8 comparison
    dec_b2b = statistics.median(time_decode_only(s, 20)) if (rank == 0 and not args.no_extra) else None
    del s
    torch.cuda.empty_cache()

    # ---- the other workloads of the metric (one GPU, rank 0) -------------
    if rank == 0 and not args.no_extra:
        extra = {}
        for name in ("nvfp4_160k", "nvfp4_1m", "int4_220k", "fp8_32k"):
            wx = W.ALL[name]
            sx = Setup(wx, device)
            ts = time_decode_only(sx, max(5, min(args.steps, 20)))
            bx = algorithmic_decode_bytes(wx, sx.lens)
            med = statistics.median(ts)
            extra[name] = {"decode_us": med * 1e6, "gbs": bx / med / 1e9, "frac": bx / med / 1e9 / peak,
                           "num_splits": sx.splits, "kv_bytes": bx, "traffic": recorded_traffic(name),
                           "ncu_dram_gbs": recorded_ncu_gbs(name),
                           "tokens_per_s_16_layers": wx.batch / (16 * med)}
            if name == "fp8_32k":
                # the comparison the pages draw: same shapes and lengths as the
                # headline workload, FP8 E4M3 per tensor instead of NVFP4
                extra[name]["nvfp4_32k_decode_us"] = dec_b2b * 1e6
                extra[name]["nvfp4_32k_speedup"] = med / dec_b2b
            if name == "nvfp4_160k":
                extra["dequant_prefix_160k"], ws = time_prefix(sx, wx, peak, keep=True)
                extra["extend_160k"] = time_extend(device, wx, ws, read_tensor_peak()[0])
                del ws
                extra["write_prefill_8k"] = time_write_prefill(sx, wx, peak)
                extra["write_prefill_128k"] = time_write_prefill(sx, wx, peak, T=131072)
            del sx
            torch.cuda.empty_cache()
        extra["calibrate_64k"] = time_calibrate(device, peak)
        extra["write_prefill_8k_int4"] = time_write_int4(device, peak)
        extra["write_prefill_256k_int4"] = time_write_int4(device, peak, T=262144)
        # the k8v4 variant on the headline shapes: FP8 keys, 4-bit values, rotated
        extra["k8v4_32k"] = time_k8v4(device, W.ALL["nvfp4_32k"], peak)
        extra["k8v4_32k"]["traffic"] = recorded_traffic("k8v4_32k")
        extra["k8v4_32k"]["ncu_dram_gbs"] = recorded_ncu_gbs("k8v4_32k")
        extra["k8v4_write_128k"] = time_k8v4_write(device, peak)
        torch.cuda.empty_cache()
        line["workloads"] = extra

    if rank == 0 and not args.no_cpu:
        try:
            r = run_cpu_oracle_subprocess(w.name, args.cpu_seconds)
            line["cpu_baseline"] = {"value": r["value"], "unit": "GB/s", "cores": 1, "kind": "oracle",
                                    "sample": f"request 0 x kv head 0 of {w.name} ({r['tokens']} tokens, "
                                              f"{w.group} query heads), {r['steps']} repeats, FP64 numpy, "
                                              "one thread"}
        except Exception as e:  # the baseline is reported, never required
            line["cpu_baseline"] = {"value": None, "unit": "GB/s", "cores": 1, "kind": "oracle",
                                    "sample": f"failed: {str(e)[-200:]}"}
        try:
            # every host core: one single-threaded oracle process per
            # (request, kv head) unit, all timed together
            nc = host_cores()
            r = cpu_oracle_all_cores(w.name, args.cpu_seconds, nc)
            one = line["cpu_baseline"]["value"]
            line["cpu_baseline"]["all_cores"] = {
                "value": r["value"], "unit": "GB/s", "cores": r["procs"],
                "sample": f"units (request, kv head) {r['units'][0]}..{r['units'][-1]} of {w.name}, "
                          f"one process each, {r['steps']} decode calls in all, FP64 numpy",
                "speedup_over_one_core": (r["value"] / one) if one else None}
        except Exception as e:
            line["cpu_baseline"]["all_cores"] = {"value": None, "failed": str(e)[-200:]}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if pg is not None:
        pg.destroy_process_group()
    return 0


def time_prefix(s, w, peak, keep=False):
    import torch
    K = s.K
    prefix = np.array([max(int(s.lens[0]) - w.prefix_chunk, 0)], np.int32)
    cu = np.array([0, prefix[0]], np.int64)
    n = int(prefix[0])
    wk = torch.empty((n, w.num_kv_heads, w.head_dim), dtype=torch.uint8, device=s.device)
    wv = torch.empty_like(wk)
    s8 = (6 * s.g).contiguous()
    d_prefix = torch.from_numpy(prefix).to(s.device)
    d_cu = torch.from_numpy(cu).to(s.device)
    table0 = s.d_table[:1].contiguous()

    def run():
        K.kv4_dequant_prefix(s.pool, s.g, table0, d_prefix, d_cu, n, s8, wk, wv)

    med = time_calls(run, 10)
    D = w.head_dim
    byts = n * w.num_kv_heads * (2 * (D // 2 + D // 16) + 2 * D)
    r = {"prefix_tokens": n, "us": med * 1e6, "gbs": byts / med / 1e9, "frac": byts / med / 1e9 / peak}
    return (r, (wk, wv, s8)) if keep else r


def extend_flops(Lp, C, Hq, D):
    """Algorithmic FLOPs of extend attention: per query row i and head,
    2*D*(Lp+i+1) for Q.K and the same for P.V."""
    return 4 * D * Hq * (C * Lp + C * (C + 1) // 2)


def time_extend(device, w, ws, tpeak, reps=5):
    """Chunked-prefill attention of an 8192-token chunk over the dequantised
    prefix of request 0 (the kv4_dequant_prefix workspace) plus the chunk's own
    FP8 K/V, on the tensor cores: TFLOP/s of algorithmic work."""
    import torch
    import bit_paged_kv_kv4_gb300 as K
    wk, wv, s8 = ws
    Lp, C = int(wk.shape[0]), w.prefix_chunk
    Hq, Hkv, D = w.num_q_heads, w.num_kv_heads, w.head_dim
    chunk, _ = W.fp8_kv_codes(w.seed, C, Hkv, D, device, scales=s8.cpu().numpy())
    ck, cv = chunk[0].contiguous(), chunk[1].contiguous()
    q = W.extend_q(w.seed, C, Hq, D, device)
    out = torch.empty((C, Hq, D), dtype=torch.bfloat16, device=device)
    i32 = lambda x: torch.tensor(x, dtype=torch.int32, device=device)
    i64 = lambda x: torch.tensor(x, dtype=torch.int64, device=device)
    pl, cp, cl, cc = i32([Lp]), i64([0, Lp]), i32([C]), i64([0, C])

    ws_ext = K.alloc_extend_workspace(1, C, Hq, D, device=device)

    def run():
        K.kv4_extend_attention(q, ck, cv, wk, wv, s8, pl, cp, cl, cc, C, w.sm_scale(), out, workspace=ws_ext)

    med = time_calls(run, reps)
    fl = extend_flops(Lp, C, Hq, D)
    return {"prefix_tokens": Lp, "chunk_tokens": C, "ms": med * 1e3, "tflops": fl / med / 1e12,
            "frac": fl / med / 1e12 / tpeak, "unit": "TFLOP/s", "bound": "tensor",
            "peak": tpeak, "flops": fl}


def time_k8v4(device, w, peak, reps=20):
    """Decode over a k8v4 pool (FP8 keys, INT4 values, Hadamard-rotated) with
    the shapes, lengths and values of workload w: HBM GB/s of pool bytes."""
    import torch
    import bit_paged_kv_kv4_gb300 as K
    lens = w.seq_lens()
    num_pages, table = w.block_table(lens)
    B, Hkv, Hq, D, P = w.batch, w.num_kv_heads, w.num_q_heads, w.head_dim, w.page_size
    pool = K.Pool("k8v4", num_pages, P, Hkv, D, device=device)
    kvs, amax = [], torch.zeros((), device=device)
    for b in range(B):
        kv = W.device_kv(w, b, int(lens[b]), device)
        amax = torch.maximum(amax, kv[0].abs().amax().float())
        kvs.append(kv)
    s_k = torch.tensor([W.fp8_scale_from_amax(float(amax))], dtype=torch.float32, device=device)
    for b in range(B):
        slots = torch.from_numpy(W.slots_for(table[b], P, np.arange(int(lens[b])))).to(device)
        K.kv4_k8v4_write(kvs[b][0], kvs[b][1], slots, pool, s_k)
    del kvs
    torch.cuda.empty_cache()
    q, _, _ = W.device_q(w, device)
    out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device=device)
    chunks = 1           # one split range per unit: the persistent CTAs balance the tiles
    ws = torch.empty(K.kv4_k8v4_workspace_bytes(B, Hkv, D, chunks), dtype=torch.uint8, device=device)
    d_table, d_lens = torch.from_numpy(table).to(device), torch.from_numpy(lens).to(device)

    def run():
        K.kv4_k8v4_decode_attention(q, pool, s_k, d_table, d_lens, w.sm_scale(), out, chunks, ws)

    med = time_calls(run, reps)
    if K.kv4_device_error() != 0:
        raise RuntimeError("k8v4 decode flagged a device error")
    byts = int(np.sum(lens)) * Hkv * (D + D // 2 + 4) + 2 * B * Hq * D * 2
    return {"decode_us": med * 1e6, "gbs": byts / med / 1e9, "frac": byts / med / 1e9 / peak,
            "num_chunks": chunks, "kv_bytes": byts, "tokens_per_s_16_layers": B / (16 * med)}


def time_k8v4_write(device, peak, T=131072, Hkv=4, D=256, P=64):
    """Prefill write of T bf16 tokens into a k8v4 pool (Hadamard rotation,
    FP8 keys, INT4 values): time_calls over 10 back-to-back calls; bytes =
    bf16 K and V in + the pool rows out + the slots."""
    import torch
    import bit_paged_kv_kv4_gb300 as K
    gen = torch.Generator(device=device).manual_seed(11)
    k = torch.randn((T, Hkv, D), generator=gen, device=device).to(torch.bfloat16)
    v = torch.randn((T, Hkv, D), generator=gen, device=device).to(torch.bfloat16)
    pool = K.Pool("k8v4", (T + P - 1) // P, P, Hkv, D, device=device)
    slots = torch.arange(T, dtype=torch.int64, device=device)
    s_k = torch.tensor([W.fp8_scale_from_amax(float(k.abs().amax().float()))], dtype=torch.float32, device=device)
    med = time_calls(lambda: K.kv4_k8v4_write(k, v, slots, pool, s_k), 10)
    if K.kv4_device_error() != 0:
        raise RuntimeError("k8v4 write flagged a device error")
    byts = T * Hkv * (2 * D * 2 + D + D // 2 + 4) + T * 8
    return {"tokens": T, "us": med * 1e6, "gbs": byts / med / 1e9, "frac": byts / med / 1e9 / peak,
            "note": f"{T * Hkv * D * 4 / 1e6:.0f} MB in, {T * Hkv * (D + D // 2 + 4) / 1e6:.1f} MB out: larger than L2"}


def time_write_int4(device, peak, T=8192):
    """Prefill write of T bf16 tokens into an INT4 per-token-head pool with the
    shapes of the 220K INT4 workload (Hkv 2, D 256, 1600-token pages)."""
    import torch
    import bit_paged_kv_kv4_gb300 as K
    w = W.ALL["int4_220k"]
    gen = torch.Generator(device=device).manual_seed(13)
    k = torch.randn((T, w.num_kv_heads, w.head_dim), generator=gen, device=device).to(torch.bfloat16)
    v = torch.randn((T, w.num_kv_heads, w.head_dim), generator=gen, device=device).to(torch.bfloat16)
    pool = K.Pool("int4", (T + w.page_size - 1) // w.page_size, w.page_size, w.num_kv_heads, w.head_dim,
                  device=device)
    slots = torch.arange(T, dtype=torch.int64, device=device)
    med = time_calls(lambda: K.kv4_write(k, v, slots, pool, None), 10)
    byts = algorithmic_write_bytes(w, T)
    in_mb = T * w.num_kv_heads * w.head_dim * 2 * 2 / 1e6
    out_mb = (byts - T * w.num_kv_heads * w.head_dim * 2 * 2) / 1e6
    l2 = "smaller than L2, so this is an L2-warm figure" if in_mb + out_mb < 129 else "larger than L2"
    return {"tokens": T, "us": med * 1e6, "gbs": byts / med / 1e9, "frac": byts / med / 1e9 / peak,
            "note": f"{in_mb:.0f} MB in, {out_mb:.1f} MB out: {l2}"}


def time_calibrate(device, peak, T=65536, Hkv=4, D=256):
    """Serving-time NVFP4 global-scale calibration over the K and V of T
    tokens (bf16, 2 x 134 MB: larger than L2, so an HBM figure)."""
    import torch
    import bit_paged_kv_kv4_gb300 as K
    gen = torch.Generator(device=device).manual_seed(11)
    k = torch.randn((T, Hkv, D), generator=gen, device=device).to(torch.bfloat16)
    v = torch.randn((T, Hkv, D), generator=gen, device=device).to(torch.bfloat16)
    out = torch.empty(2, dtype=torch.float32, device=device)
    med = time_calls(lambda: K.kv4_calibrate_global_scale(k, v, out), 10)
    byts = 2 * T * Hkv * D * 2 + 8
    return {"tokens": T, "us": med * 1e6, "gbs": byts / med / 1e9, "frac": byts / med / 1e9 / peak}


def time_write_prefill(s, w, peak, T=None):
    """Prefill write of T tokens (default: the workload's 8K chunk) of bf16
    K/V into a scratch pool of the workload's geometry, then the same from
    FP8 K/V: time_calls over 10 back-to-back calls each."""
    import torch
    K = s.K
    T = T or w.prefix_chunk
    gen = torch.Generator(device=s.device).manual_seed(7)
    k = torch.randn((T, w.num_kv_heads, w.head_dim), generator=gen, device=s.device).to(torch.bfloat16)
    v = torch.randn((T, w.num_kv_heads, w.head_dim), generator=gen, device=s.device).to(torch.bfloat16)
    # scratch pool of the same geometry, so the measured pool stays intact
    pool = K.Pool(w.fmt, (T + w.page_size - 1) // w.page_size, w.page_size, w.num_kv_heads, w.head_dim,
                  device=s.device)
    slots = torch.arange(T, dtype=torch.int64, device=s.device)
    med = time_calls(lambda: K.kv4_write(k, v, slots, pool, s.g), 10)
    byts = algorithmic_write_bytes(w, T)
    # the same write fed with FP8 K/V (the engine's form), per-tensor input scales
    codes, s_in = W.fp8_kv_codes(w.seed, T, w.num_kv_heads, w.head_dim, s.device)
    k8, v8 = codes[0].contiguous(), codes[1].contiguous()
    d_in = torch.from_numpy(s_in).to(s.device)
    m8 = time_calls(lambda: K.kv4_write_fp8(k8, v8, d_in, slots, pool, s.g), 10)
    b8 = algorithmic_write_bytes(w, T, in_bytes=1)
    in_mb = T * w.num_kv_heads * w.head_dim * 2 * 2 / 1e6
    out_mb = (byts - T * w.num_kv_heads * w.head_dim * 2 * 2) / 1e6
    l2 = "smaller than L2, so these are L2-warm figures" if in_mb + out_mb < 129 else "larger than L2"
    return {"tokens": T, "us": med * 1e6, "gbs": byts / med / 1e9, "frac": byts / med / 1e9 / peak,
            "fp8_input_us": m8 * 1e6, "fp8_input_gbs": b8 / m8 / 1e9, "fp8_input_frac": b8 / m8 / 1e9 / peak,
            "note": f"{in_mb:.0f} MB in ({in_mb / 2:.0f} MB with FP8 input), {out_mb:.1f} MB out: {l2}"}


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("kv4", "reference"), default="kv4")
    ap.add_argument("--workload", default="nvfp4_32k", choices=sorted(W.ALL))
    ap.add_argument("--no-extra", action="store_true", help="skip the 160K / 1M / INT4 lines")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--only", choices=("prefix", "write", "extend", "k8v4", "calibrate"),
                    help="time just the 160K prefix dequant or the 8K prefill write and print "
                         "its line (for profiling one kernel)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        return reference_arm(args)
    if args.only:
        return only_arm(args)
    return kv4_arm(args)


def only_arm(args):
    import torch
    import bit_paged_kv_kv4_gb300 as K
    K.load(build_if_missing=True)
    device = torch.device("cuda", 0)
    w = W.ALL["nvfp4_160k"]
    peak, _ = read_peaks()
    if args.only == "prefix":
        r = time_prefix(Setup(w, device), w, peak)
    elif args.only == "k8v4":
        r = time_k8v4(device, W.ALL["nvfp4_32k"], peak)
        r["write_128k"] = time_k8v4_write(device, peak)
    elif args.only == "calibrate":
        r = time_calibrate(device, peak)
    elif args.only == "extend":
        r, ws = time_prefix(Setup(w, device), w, peak, keep=True)
        r = time_extend(device, w, ws, read_tensor_peak()[0], reps=args.steps)
    else:
        # the prefill write needs no filled pool: a device, a pair of global scales
        # of the workload's magnitude and the library
        import types
        lite = types.SimpleNamespace(device=device, K=K,
                                     g=torch.tensor([1.0 / (6 * 448)] * 2, dtype=torch.float32, device=device))
        r = time_write_prefill(lite, w, peak)
        r["128k"] = time_write_prefill(lite, w, peak, T=131072)
        r["int4"] = time_write_int4(device, peak)
        r["int4_256k"] = time_write_int4(device, peak, T=262144)
    if K.kv4_device_error() != 0:
        raise SystemExit(f"device error {K.kv4_device_error()}")
    print(json.dumps({"only": args.only, "workload": w.name, **r}))
    return 0


if __name__ == "__main__":
    sys.exit(main())
