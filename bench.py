#!/usr/bin/env python
"""Benchmark of the FusedKV decode hot path on GB300.

A step is one attention-only decode step of the 332M-shaped model (12 layers,
storage layers 1-6, 16 Q / 8 KV heads, D=64, bf16 caches, batch 32, 8192
cached tokens per sequence), as the FusedKV Table 1 accounting counts it:
  * fkv_append_kv of the new token's K/V into every layer that stores
    (layers 1-6; all 12 in vanilla mode), then
  * fkv_decode_attn for layers 1..12 in order (upper layers in the mode under
    test: vanilla reads their own cache, lite K^6/V^1, fused K^1,K^6,V^1,V^6).
`value` is fused-mode decode tokens/s (batch / step time) with every input
resident in HBM; `modes` holds all three modes; `e2e` repeats the fused step
through the same C-ABI calls with the per-step inputs copied from pinned host
memory and the outputs read back inside the timed region.  The same step is
timed on the 1.5B-shaped (24 layers, ragged lengths up to 32768) and 4B-shaped
(36 layers, S=131072) workloads in every mode (`decode_steps_other_workloads`),
beside the 650M causal prefill and the 4-bit decode calls; each section
carries its own clock record.  `cpu_baseline` (and `--impl reference`) time
the float64 oracle on whole fused steps, one single-threaded worker process
per host core.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
For N > 1 (torchrun) every rank runs an independent replica (the path shards
by sequence with no exchange), rank 0 prints the max-over-ranks timing.
"""

from __future__ import annotations

import os

# Each oracle worker process runs single-threaded (one per host core), so
# that `cores` is exact.
for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import argparse
import hashlib
import json
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = ("decode tokens/s & KV GB/s (% of 8 TB/s HBM) for fused/lite/vanilla; "
          "prefill TFLOP/s")
HBM_REF_GBS = 8000.0

# DRAM traffic (read + write bytes per launch) of the fused split kernel on
# this workload, from one ncu capture, and the source hash of the kernel it was
# taken on; reported only while the kernel is unchanged.
NCU_TRAFFIC = {"bytes_per_launch": 1073992704 + 2834944, "kernel_sha": "b10f3f3fb27d3bd1",
               "profile": "profiles/decode_split_fused_332M.md"}


def _kernel_sha():
    h = hashlib.sha256()
    for f in ("decode_impl.cuh", "fkv_device.cuh"):
        with open(os.path.join(ROOT, "cross_layer_kv_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
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
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in getattr(self, "lines", []):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# the decode model (caches for all 12 layers so vanilla can run)
# ---------------------------------------------------------------------------

class DecodeModel:
    """Caches of every layer (so that vanilla can run), per-step inputs and
    outputs of one attention-only decode step of a workload.  Sequences are
    full (S rows) or, for ragged workloads, of their drawn lengths; each step
    writes the new token at row len - 1 and attends over len rows, so the
    step's shape stays fixed from step to step."""

    def __init__(self, w, device, seed=0):
        import cross_layer_kv_gb300 as fkv
        from cross_layer_kv_gb300 import synth
        self.w = w
        self.dev = device
        L, n = w.num_layers, w.n
        self.ctx = fkv.Context(L, w.batch, w.seq, w.q_heads, w.kv_heads, w.head_dim, w.dtype,
                               store_upper=True)
        self.caches = {}
        for l in range(1, L + 1):
            k, v = synth.make_cache(w, l, seed, device)
            self.caches[l] = (k, v)
            self.ctx.fkv_bind_layer_cache(l, k, v)
        self.weights = {}
        for l in range(n + 1, L + 1):
            self.weights[l] = synth.make_weights(w, l, seed, device)
            self.ctx.fkv_set_fusion_weights(l, *self.weights[l])
        # per-step inputs: queries of every layer, the new token's K/V per layer
        self.q = torch.stack([synth.make_query(w, l, seed + 1, device) for l in range(1, L + 1)])
        g = torch.Generator(device=device).manual_seed(seed + 2)
        shape = (L, w.batch, w.kv_heads, 1, w.head_dim)
        self.k_new = torch.randn(shape, generator=g, device=device).to(w.torch_dtype)
        self.v_new = torch.randn(shape, generator=g, device=device).to(w.torch_dtype)
        self.lens = synth.make_seq_lens(w, seed, device)
        self.pos = (self.lens - 1).to(torch.int32)
        self.rows = int(self.lens.sum())
        self.out = torch.empty_like(self.q)
        self.ws = self.ctx.workspace(device)

    def appended_layers(self, mode):
        return range(1, self.w.num_layers + 1) if mode == "vanilla" else range(1, self.w.n + 1)

    def launches_per_step(self, mode):
        from cross_layer_kv_gb300.fusedkv import DECODE_LAUNCHES_PER_CALL
        return len(self.appended_layers(mode)) + DECODE_LAUNCHES_PER_CALL * self.w.num_layers

    def step(self, mode, stream, upper_events=None):
        c = self.ctx
        for l in self.appended_layers(mode):
            c.fkv_append_kv(l, self.k_new[l - 1], self.v_new[l - 1], self.pos, 1, stream)
        for l in range(1, self.w.num_layers + 1):
            ev = upper_events is not None and l > self.w.n
            if ev:
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
            c.fkv_decode_attn(self.q[l - 1], l, mode, self.lens, self.out[l - 1], self.ws, stream)
            if ev:
                e1.record(stream)
                upper_events.append((e0, e1))

    def call_bytes(self, layer, mode):
        """Algorithmic cache bytes one decode call reads (K and V sources)."""
        w = self.w
        nsrc = 2 if (layer > w.n and mode == "fused") else 1
        return 2 * nsrc * w.kv_heads * self.rows * w.head_dim * w.elem_bytes

    def step_bytes(self, mode):
        return sum(self.call_bytes(l, mode) for l in range(1, self.w.num_layers + 1))

    def close(self):
        self.ctx.close()
        self.caches.clear()


def _barrier(dist_on):
    if dist_on:
        torch.distributed.barrier()


def _max_over_ranks(x, dist_on, device):
    if not dist_on:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def time_steps(model, mode, K, W, stream, dist_on, device, collect_upper=False):
    """K steps after W warm-up steps, bracketed by barrier + synchronize; the
    max over ranks of their CUDA-event time.  With collect_upper, a second
    run of K steps records events around every upper-layer call (kept out of
    the step timing, since an event between two calls breaks their
    programmatic-dependent-launch overlap) and returns their mean duration."""
    for _ in range(W):
        model.step(mode, stream)
    torch.cuda.synchronize()
    _barrier(dist_on)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(K):
        model.step(mode, stream)
    e1.record(stream)
    torch.cuda.synchronize()
    _barrier(dist_on)
    ms = _max_over_ranks(e0.elapsed_time(e1), dist_on, device)
    upper_ms = None
    if collect_upper:
        upper = []
        for _ in range(K):
            model.step(mode, stream, upper)
        torch.cuda.synchronize()
        upper_ms = statistics.fmean(a.elapsed_time(b) for a, b in upper)
    return ms, upper_ms


def time_e2e(model, K, W, stream, dist_on, device, graph=False):
    """Fused step through the C ABI with per-step inputs from pinned host
    memory and the step's outputs read back, all inside the timed region.
    graph: the step (copies in, kernels, copy out) is captured once in a CUDA
    graph, and each step replays it; the host still waits every step."""
    q_h = model.q.cpu().pin_memory()
    kn_h = model.k_new.cpu().pin_memory()
    vn_h = model.v_new.cpu().pin_memory()
    out_h = torch.empty(model.out.shape, dtype=model.out.dtype).pin_memory()
    n = model.w.n

    def body():
        model.q.copy_(q_h, non_blocking=True)
        model.k_new[:n].copy_(kn_h[:n], non_blocking=True)
        model.v_new[:n].copy_(vn_h[:n], non_blocking=True)
        model.step("fused", stream)
        out_h.copy_(model.out, non_blocking=True)

    if graph:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            body()

        def one():
            with torch.cuda.stream(stream):
                g.replay()
            stream.synchronize()
    else:
        def one():
            with torch.cuda.stream(stream):
                body()
            stream.synchronize()

    for _ in range(W):
        one()
    torch.cuda.synchronize()
    _barrier(dist_on)
    t0 = time.perf_counter()
    for _ in range(K):
        one()
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    _barrier(dist_on)
    dt = _max_over_ranks(dt, dist_on, device)
    h2d = q_h.numel() * q_h.element_size() + 2 * kn_h[:n].numel() * kn_h.element_size()
    d2h = out_h.numel() * out_h.element_size()
    return dt, h2d, d2h


# ---------------------------------------------------------------------------
# oracle timing (cpu_baseline and --impl reference): whole attention-only
# decode steps of the 332M workload in fused mode, the batch's sequences
# spread over a spawn pool of one single-threaded process per host core
# ---------------------------------------------------------------------------

_ORACLE = {}


def host_cores() -> int:
    """Cores this process may run on (the affinity mask, else the CPU count)."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def _oracle_worker_init(wname, seed):
    """Pool initializer (untimed): one synthetic sequence of the workload --
    the same recipe, seeded per worker -- as float64 arrays: the caches of the
    storage layers, the fusion weights of the upper layers, a query per layer."""
    import oracle as O
    from cross_layer_kv_gb300 import synth
    torch.set_num_threads(1)
    w = synth.WORKLOADS[wname]
    one = synth.Workload(w.name, w.num_layers, 1, w.seq, w.q_heads, w.kv_heads, w.head_dim,
                         w.dtype)
    seed = seed + 1000 * (os.getpid() % 1000)
    L, n = w.num_layers, w.n
    kc, vc, weights, qs = {}, {}, {}, {}
    for l in range(1, n + 1):
        k, v = synth.make_cache(one, l, seed, "cpu")
        kc[l], vc[l] = k.double().numpy(), v.double().numpy()
    for l in range(n + 1, L + 1):
        weights[l] = tuple(x.double().numpy() for x in synth.make_weights(one, l, seed, "cpu"))
    for l in range(1, L + 1):
        qs[l] = synth.make_query(one, l, seed, "cpu").double().numpy()
    _ORACLE.update(O=O, L=L, S=w.seq, kc=kc, vc=vc, weights=weights, qs=qs)


def _oracle_sequence(_):
    """The oracle's fused decode step of one sequence: all L layers in order."""
    st = _ORACLE
    O, L = st["O"], st["L"]
    for l in range(1, L + 1):
        O.decode_attn(st["qs"][l], l, L, O.FUSED, st["kc"], st["vc"], [st["S"]],
                      weights=st["weights"])
    return 1


class OraclePool:
    """A spawn pool (safe after CUDA initialisation) of host_cores() workers,
    capped at the batch size; BLAS stays at one thread per process."""

    def __init__(self, w, seed=0, workers=0):
        import multiprocessing as mp
        self.w = w
        self.workers = max(1, min(workers or host_cores(), w.batch))
        self.pool = mp.get_context("spawn").Pool(self.workers, initializer=_oracle_worker_init,
                                                 initargs=(w.name, seed))

    def step(self, rows):
        """One step over `rows` sequences; returns its wall time in seconds."""
        t0 = time.perf_counter()
        done = sum(self.pool.map(_oracle_sequence, range(rows), chunksize=1))
        assert done == rows
        return time.perf_counter() - t0

    def close(self):
        self.pool.close()
        self.pool.join()


def oracle_baseline(w, budget_s=4.0, workers=0):
    """cpu_baseline leg: whole fused decode steps of the workload's batch on the
    oracle pool, one warm-up step, then steps until `budget_s` of wall time."""
    pool = OraclePool(w, workers=workers)
    try:
        pool.step(pool.workers)          # every worker built its inputs
        pool.step(w.batch)               # warm-up step
        steps, el = 0, 0.0
        while el < budget_s or steps < 1:
            el += pool.step(w.batch)
            steps += 1
    finally:
        pool.close()
    sample = ("%d whole fused decode step(s) of %d sequences x %d layers (S=%d) on %d "
              "single-threaded worker processes, %.1f s wall" % (
                  steps, w.batch, w.num_layers, w.seq, pool.workers, el))
    return steps * w.batch / el, pool.workers, sample


def workload_label(w) -> str:
    """The config.workload string both arms report."""
    return ("%s (%d layers, storage 1-%d, B=%d, S=%d, %d/%d heads, D=%d, %s), attention-only "
            "decode step, fused mode" % (w.name, w.num_layers, w.n, w.batch, w.seq, w.q_heads,
                                         w.kv_heads, w.head_dim, w.dtype))


def run_reference(args, rank, dist_on):
    """The reference arm: the oracle, as it stands, timing whole steps."""
    from cross_layer_kv_gb300 import synth
    w = synth.M332
    if rank != 0:
        return
    pool = OraclePool(w, workers=args.oracle_workers)
    try:
        pool.step(pool.workers)
        rows = args.ref_rows or w.batch
        t_full = pool.step(rows)                     # first warm-up step
        # each step processes the whole batch unless K such steps would take
        # more than ~150 s; then a bounded sample of the batch's sequences
        if args.steps * t_full > 150.0:
            rows = max(1, int(rows * 150.0 / (args.steps * t_full)))
        for _ in range(args.warmup - 1):
            pool.step(rows)
        total = 0.0
        for _ in range(args.steps):
            total += pool.step(rows)
    finally:
        pool.close()
    ms = total * 1e3 / args.steps
    val = args.steps * rows / total
    sample = ("%d steps of %d sequence(s) x %d layers (fused decode, S=%d) on %d single-"
              "threaded worker processes" % (args.steps, rows, w.num_layers, w.seq, pool.workers))
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": workload_label(w), "global_batch": w.batch * args.gpus,
                       "seq_len": w.seq, "parallelism": "replicas" if args.gpus > 1 else "single",
                       "rows_per_step": rows},
            "cpu_baseline": {"value": val, "unit": "tokens/s", "cores": pool.workers,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def measure_modes(model, K, W, stream, dist_on, device, local, peaks, world):
    """Decode steps of a model in each mode: tokens/s, step time and GB/s, and
    the mean upper-layer call.  The clocks are sampled over the fused mode's
    timed steps."""
    w = model.w
    modes = {}
    clocks = None
    for mode in ("vanilla", "lite", "fused"):
        if mode == "fused":
            with ClockSampler(local) as cs:
                ms, up = time_steps(model, mode, K, W, stream, dist_on, device,
                                    collect_upper=True)
            clocks = cs.summary()
        else:
            ms, up = time_steps(model, mode, K, W, stream, dist_on, device, collect_upper=True)
        step_ms = ms / K
        gb = model.step_bytes(mode) / 1e9
        ub = model.call_bytes(w.num_layers, mode) / 1e9
        modes[mode] = {
            "upper_call_us": up * 1e3,
            "upper_call_GBps": ub / (up / 1e3),
            "upper_call_pct_of_8TBps": 100.0 * ub / (up / 1e3) / HBM_REF_GBS,
            "upper_call_pct_of_measured_hbm": 100.0 * ub / (up / 1e3) / peaks["hbm_gbs"],
            "tokens_per_s": w.batch * world / (step_ms / 1e3),
            "step_ms": step_ms,
            "step_bytes_GB": gb,
            "GBps": gb / (step_ms / 1e3),
            "pct_of_8TBps": 100.0 * gb / (step_ms / 1e3) / HBM_REF_GBS,
            "pct_of_measured_hbm": 100.0 * gb / (step_ms / 1e3) / peaks["hbm_gbs"],
        }
    return modes, clocks


# ---------------------------------------------------------------------------

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=4.0,
                    help="wall seconds of oracle steps for cpu_baseline (after a warm-up step)")
    ap.add_argument("--ref-rows", type=int, default=0,
                    help="sequences per reference step (0: the whole batch, unless K such "
                         "steps would take over ~150 s)")
    ap.add_argument("--oracle-workers", type=int, default=0,
                    help="oracle worker processes (0: one per host core, at most the batch)")
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--no-other-decode", action="store_true",
                    help="skip the decode steps of the 1.5B and 4B workloads and the 4-bit calls")
    ap.add_argument("--profile", default=None,
                    help="run one call type only, e.g. decode:fused:332M-decode, "
                         "decode:fused:332M-decode:q4 or prefill:fused:650M-prefill "
                         "(for ncu captures)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist_on = world > 1
    if args.impl == "reference":
        if dist_on:
            torch.distributed.init_process_group("gloo")
        run_reference(args, rank, dist_on)
        if dist_on:
            torch.distributed.destroy_process_group()
        return

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if args.profile:
        run_profile_case(args, device)
        return
    if dist_on:
        torch.distributed.init_process_group("nccl", device_id=device)

    from cross_layer_kv_gb300 import synth
    import cross_layer_kv_gb300 as fkv
    fkv.load()
    w = synth.M332
    model = DecodeModel(w, device)
    stream = torch.cuda.Stream(device)
    peaks = _peaks()
    K, W = args.steps, args.warmup

    modes, clocks = measure_modes(model, K, W, stream, dist_on, device, local, peaks, world)
    launches = K * model.launches_per_step("fused")
    upper_ms = modes["fused"]["upper_call_us"] / 1e3

    # dominant kernel: the fused upper-layer decode call
    call_bytes = model.call_bytes(w.num_layers, "fused")
    achieved = call_bytes / (upper_ms / 1e3) / 1e9
    traffic = NCU_TRAFFIC["bytes_per_launch"] if NCU_TRAFFIC["kernel_sha"] == _kernel_sha() else None
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"], "traffic": traffic,
                "kernel": "fused upper-layer fkv_decode_attn (decode_split_kernel, in-kernel merge)",
                "algorithmic_bytes_per_launch": call_bytes, "avg_launch_us": upper_ms * 1e3,
                "peak_source": peaks["source"] + " (MEASURED_PEAKS.json hbm_gbs, copy)"}

    e2e_steps = max(20, K // 5)
    e2e_s, h2d, d2h = time_e2e(model, e2e_steps, W, stream, dist_on, device)
    g_s, _, _ = time_e2e(model, e2e_steps, W, stream, dist_on, device, graph=True)
    eager = {"value": w.batch * world * e2e_steps / e2e_s, "unit": "tokens/s",
             "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
             "note": "fused step via the C ABI, each call launched from the host; per-step q "
                     "and new K/V from pinned host memory, all 12 layer outputs read back, "
                     "host sync every step"}
    e2e = {"value": w.batch * world * e2e_steps / g_s, "unit": "tokens/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
           "note": "the same step through the C ABI, captured once in a CUDA graph (copies in, "
                   "6 appends, 12 decode calls, copy out) and replayed every step, host sync "
                   "every step",
           "eager": eager}

    model.close()
    del model
    torch.cuda.empty_cache()

    prefill = None
    if not args.no_prefill:
        with ClockSampler(local) as cs:
            prefill = bench_prefill(device, stream, peaks, W)
        prefill["clocks"] = cs.summary()
    other_decode = None
    q4 = None
    if not args.no_other_decode:
        other_decode = {}
        for wo in (synth.B1_5, synth.B4):
            m = DecodeModel(wo, device)
            Ko = max(5, min(K, 20))
            om, ocl = measure_modes(m, Ko, W, stream, dist_on, device, local, peaks, world)
            other_decode[wo.name] = {
                "workload": workload_label(wo).replace(", fused mode", ", each mode"),
                "steps": Ko, "modes": om, "clocks": ocl,
                "fused_over_vanilla_step_time": om["fused"]["step_ms"] / om["vanilla"]["step_ms"],
                "lite_over_vanilla_step_time": om["lite"]["step_ms"] / om["vanilla"]["step_ms"]}
            m.close()
            del m
            torch.cuda.empty_cache()
        with ClockSampler(local) as cs:
            q4 = bench_q4_calls(device, stream, peaks, W)
        q4["clocks"] = cs.summary()
        # the 4B shape (D = 80: a row spans 5 lanes of the 4-bit kernel)
        with ClockSampler(local) as cs:
            q4_4b = bench_q4_calls(device, stream, peaks, W, reps=10, w=synth.B4)
        q4_4b["clocks"] = cs.summary()

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        val, cores, sample = oracle_baseline(w, budget_s=args.cpu_budget,
                                             workers=args.oracle_workers)
        cpu = {"value": val, "unit": "tokens/s", "cores": cores, "kind": "oracle",
               "sample": sample}

    fused = modes["fused"]
    if rank == 0:
        line = {
            "metric": METRIC,
            "value": fused["tokens_per_s"],
            "unit": "tokens/s",
            "n_gpus": world,
            "steps": K,
            "warmup": W,
            "ms_per_step": fused["step_ms"],
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": workload_label(w),
                       "global_batch": w.batch * world, "seq_len": w.seq,
                       "parallelism": "replicas" if world > 1 else "single",
                       "l2": "inputs larger than L2 (every call reads >= 0.5 GB)"},
            "modes": modes,
            "fused_over_vanilla_step_time": modes["fused"]["step_ms"] / modes["vanilla"]["step_ms"],
            "roofline": roofline,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": launches,
            "clocks": clocks,
        }
        if prefill is not None:
            line["prefill"] = prefill
        if other_decode is not None:
            line["decode_steps_other_workloads"] = other_decode
        if q4 is not None:
            line["decode_q4_332M"] = q4
            line["decode_q4_4B"] = q4_4b
        print(json.dumps(line), flush=True)
    if dist_on:
        torch.distributed.destroy_process_group()


class SingleCall:
    """Buffers for one call type of a workload: only the layers it reads
    (4-bit caches with ``q4``, quantised by the library's own append)."""

    def __init__(self, kind, mode, w, device, stream, q4=False):
        import cross_layer_kv_gb300 as fkv
        from cross_layer_kv_gb300 import synth
        self.w, self.kind, self.mode = w, kind, mode
        layer = w.num_layers
        need = [layer] if mode == "vanilla" else sorted({1, w.n})
        self.ctx = fkv.Context(w.num_layers, w.batch, w.seq, w.q_heads, w.kv_heads, w.head_dim,
                               w.dtype, store_upper=(mode == "vanilla"))
        self.keep = []
        for l in need:
            k, v = synth.make_cache(w, l, 0, device)
            if q4:
                kr, vr = self.ctx.q4_cache(device), self.ctx.q4_cache(device)
                self.ctx.fkv_bind_layer_cache_q4(l, kr, vr)
                pos0 = torch.zeros(w.batch, dtype=torch.int32, device=device)
                self.ctx.fkv_append_kv(l, k, v, pos0, w.seq, stream)
                torch.cuda.synchronize()
                self.keep.append((kr, vr))
                del k, v
            else:
                self.keep.append((k, v))
                self.ctx.fkv_bind_layer_cache(l, k, v)
        wts = synth.make_weights(w, layer, 0, device)
        self.keep.append(wts)
        self.ctx.fkv_set_fusion_weights(layer, *wts)
        ctx = self.ctx
        if kind == "decode":
            q = synth.make_query(w, layer, 0, device)
            out = torch.empty_like(q)
            lens = synth.make_seq_lens(w, 0, device)
            ws = ctx.workspace(device)
            self.keep += [q, out, lens, ws]
            self.call = lambda: ctx.fkv_decode_attn(q, layer, mode, lens, out, ws, stream)
            nsrc = 2 if mode == "fused" else 1
            row = ctx.fkv_q4_row_bytes() if q4 else w.head_dim * w.elem_bytes
            self.bytes = 2 * nsrc * w.kv_heads * int(lens.sum()) * row
            self.flops = 0
        else:
            q = synth.make_query(w, layer, 0, device, positions=w.seq)
            out = torch.empty_like(q)
            self.keep += [q, out]
            self.call = lambda: ctx.fkv_prefill_attn(q, layer, mode, w.seq, out, stream)
            self.bytes = 0
            self.flops = 4.0 * w.batch * w.q_heads * w.head_dim * w.seq * (w.seq + 1) / 2

    def time_us(self, stream, steps, warmup):
        for _ in range(warmup):
            self.call()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            self.call()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) * 1e3 / steps

    def close(self):
        self.ctx.close()
        self.keep.clear()


def run_profile_case(args, device):
    """One call type on its own, W warm-up calls then K timed calls; prints
    the mean call time.  Used for ncu captures of a single kernel."""
    from cross_layer_kv_gb300 import synth
    parts = args.profile.split(":")
    kind, mode, wname = parts[:3]
    q4 = len(parts) > 3 and parts[3] == "q4"
    stream = torch.cuda.Stream(device)
    sc = SingleCall(kind, mode, synth.WORKLOADS[wname], device, stream, q4=q4)
    us = sc.time_us(stream, args.steps, args.warmup)
    res = {"profile": args.profile, "call_us": us}
    if sc.bytes:
        res["GBps"] = sc.bytes / (us * 1e-6) / 1e9
        res["bytes"] = sc.bytes
    else:
        res["TFLOPs"] = sc.flops / (us * 1e-6) / 1e12
    print(json.dumps(res), flush=True)
    sc.close()


def bench_q4_calls(device, stream, peaks, W, reps=20, w=None):
    """4-bit caches: one upper-layer decode call per mode of a workload (the
    332M-shaped one by default); GB/s over the 4-bit bytes."""
    from cross_layer_kv_gb300 import synth
    w = w or synth.M332
    res = {"workload": w.name + " with 4-bit caches (16-channel groups, bf16 scale/min)"}
    for mode in ("vanilla", "lite", "fused"):
        sc = SingleCall("decode", mode, w, device, stream, q4=True)
        us = sc.time_us(stream, reps, W)
        gbs = sc.bytes / (us * 1e-6) / 1e9
        res[mode] = {"upper_call_us": us, "bytes": sc.bytes, "GBps": gbs,
                     "pct_of_measured_hbm": 100.0 * gbs / peaks["hbm_gbs"]}
        sc.close()
        del sc
        torch.cuda.empty_cache()
    return res


def bench_prefill(device, stream, peaks, W):
    """Causal prefill of the 650M-shaped workload (B=4, S=8192, 16/8 heads,
    D=96), one upper-layer call per mode; TFLOP/s counts unmasked work."""
    import cross_layer_kv_gb300 as fkv
    from cross_layer_kv_gb300 import synth
    w = synth.M650_PREFILL
    ctx = fkv.Context(w.num_layers, w.batch, w.seq, w.q_heads, w.kv_heads, w.head_dim, "bf16",
                      store_upper=True)
    layer = w.num_layers
    keep = []
    for l in sorted({1, w.n, layer}):
        k, v = synth.make_cache(w, l, 0, device)
        keep.append((k, v))
        ctx.fkv_bind_layer_cache(l, k, v)
    wts = synth.make_weights(w, layer, 0, device)
    ctx.fkv_set_fusion_weights(layer, *wts)
    q = synth.make_query(w, layer, 0, device, positions=w.seq)
    out = torch.empty_like(q)
    flops = 4.0 * w.batch * w.q_heads * w.head_dim * w.seq * (w.seq + 1) / 2
    res = {"workload": w.name + " (B=4, S=8192, 16/8 heads, D=96, bf16, causal)"}
    try:
        for mode in ("vanilla", "lite", "fused"):
            for _ in range(W):
                ctx.fkv_prefill_attn(q, layer, mode, w.seq, out, stream)
            torch.cuda.synchronize()
            reps = 10
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(reps):
                ctx.fkv_prefill_attn(q, layer, mode, w.seq, out, stream)
            e1.record(stream)
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1) / reps
            tf = flops / (ms / 1e3) / 1e12
            res[mode] = {"ms": ms, "TFLOPs": tf,
                         "frac_of_bf16_peak": tf / peaks["bf16_tflops"],
                         "peak": peaks["bf16_tflops"], "peak_source": peaks["source"] + " burst"}
    except fkv.FkvError as e:
        res["unavailable"] = str(e)
    ctx.close()
    if "fused" in res and "vanilla" in res:
        res["fused_over_vanilla_time"] = res["fused"]["ms"] / res["vanilla"]["ms"]
    return res


if __name__ == "__main__":
    main()
