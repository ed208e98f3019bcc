#!/usr/bin/env python3
"""Benchmark of the ResidualKV cache-write path (and its sparse read) on GB300.

One step = the whole hot path over the Llama-3.1-8B KV-shape workload: for all 32
layers x 8192 tokens, build the reference pool, compress every token (retrieval,
reference mean, SwiGLU residual code, group quantisation), then one decode-style
sparse read per layer (30% random tokens plus the last 512).  Inputs are resident in
HBM when the timed region starts; `e2e` repeats the step with the host->device copy
of the step's input (every token's kv) and the device->host copy of its product (the
compressed cache: codes, group extremes, reference slots and the stored pool) inside
the timing (layers in chunks, copies overlapped with the compute).  The compressor
weights are model parameters that stay resident across steps, and the sparse read's
outputs are consumed on the device (by the restore and attention), so neither crosses
the host link in a step.

Prints ONE JSON line (rank 0).  `--impl reference` times the fp64 oracle instead on
a bounded sample of the same workload, on this host's CPU.
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import json
import math
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import rkv_workload as wl  # noqa: E402

WORKLOAD = "llama3.1-8b-kv"
METRIC = "tokens compressed/sec (Llama-3.1-8B KV shape) and % of bf16 tensor roofline"
UNIT = "tokens/s"


# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) per launch of a kernel on
# this workload, from one `ncu --set full` capture of the 4-layer case scaled to 32
# layers by the units processed (its traffic grows in proportion).  Set an entry to None
# when its kernel changes.
# layers per chunk of the end-to-end step (copies of one chunk overlap another's compute)
E2E_CHUNK_LAYERS = 2

NCU_DRAM_BYTES = {"umma_swiglu_diff": 8 * (183.950080e6 + 91.849984e6),
                  "umma_distance_topk": 8 * (164.111872e6 + 4.239872e6),
                  "umma_z_quant": 8 * (121.788416e6 + 3.854080e6),
                  "umma_ref_proj": 8 * (50.373120e6 + 2.918656e6)}


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            m = json.load(f)
        return (float(m["hbm_gbs"]), float(m["bf16_tflops"]), float(m["bf16_tflops_sustained"]),
                "measured")
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


def _dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    return int(os.environ.get("RANK", "0")), ws, int(os.environ.get("LOCAL_RANK", "0"))


def max_over_ranks(x: float, ws: int, device=None) -> float:
    """The largest value of x over the ranks (the job's time is its slowest rank's)."""
    if ws <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(ms_local: float, units_per_rank: float, ws: int, device=None):
    """(ms, units per second of the whole job): every rank processes units_per_rank in
    its ms_local; the job's time is the slowest rank's."""
    ms = max_over_ranks(ms_local, ws, device)
    return ms, units_per_rank * ws / (ms / 1e3)


def workload_description(cfg: wl.Config) -> dict:
    return {
        "workload": "%s: %d layers x %d seq x %d tokens, kv width %d (N=%d, D=%d), d_ff=%d, "
                    "d_c=%d, k=%d, stride %d, INT%d, %s kv/%s refs; step = pool + compress of "
                    "all layers + one sparse read per layer (30%% random + last %d)" % (
                        cfg.name, cfg.L, cfg.B, cfg.T, cfg.W, cfg.N, cfg.D, cfg.d_ff, cfg.d_c,
                        cfg.k, cfg.stride, cfg.bits, cfg.kv_dtype, cfg.ref_dtype, cfg.gather_tail),
        "layers": cfg.L, "seqs": cfg.B, "tokens": cfg.T, "kv_width": cfg.W, "d_ff": cfg.d_ff,
        "d_c": cfg.d_c, "bits": cfg.bits, "stride": cfg.stride,
        "l2": "inputs (%.2f GB kv) exceed the 129 MB L2; no flush" % (
            cfg.L * cfg.B * cfg.T * cfg.W * 2 / 1e9),
        "parallelism": "replicas (one independent workload per GPU)",
    }


def algorithmic(cfg: wl.Config):
    """Algorithmic work of one step (per layer-sequence x L*B): the flops the method
    needs (distances over the causal pool, the first compressor layer once per token
    and once per reference, W_c3 once per token) and the read's bytes."""
    T, s, W, F, C = cfg.T, cfg.stride, cfg.W, cfg.d_ff, cfg.d_c
    ref_pos = np.arange(cfg.first, T, s)
    n_ref = ref_pos.size
    n_non = T - n_ref
    t = np.arange(T)
    pool = np.searchsorted(ref_pos, t, side="left")
    is_ref = np.zeros(T, bool)
    is_ref[ref_pos] = True
    pairs = int(pool[~is_ref].sum())
    LB = cfg.L * cfg.B
    fl = {
        "umma_distance_topk": LB * pairs * 2.0 * W,
        "umma_swiglu_diff": LB * n_non * 4.0 * W * F,
        "umma_ref_proj": LB * n_ref * 4.0 * W * F,
        "umma_z_quant": LB * n_non * 2.0 * F * C,
    }
    return fl, n_ref, n_non, pairs


def restore_bytes_per_token(cfg, out_bytes=2):
    """Algorithmic HBM bytes of restoring one selected token: its codes, group extremes,
    reference slots and index, and the K and V rows written (the pool and W_d are read
    once per call and stay in L2)."""
    return cfg.d_c * cfg.bits // 8 + (cfg.d_c // 32) * 8 + 16 + 4 + cfg.W * out_bytes


def gather_bytes_per_token(cfg, out_bytes=2):
    return (cfg.d_c * cfg.bits // 8 + (cfg.d_c // 32) * 8 + 16 + 4 + cfg.d_c * out_bytes
            + cfg.W * out_bytes)


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed region runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), "--query-gpu=" + self.Q, "--format=csv,noheader",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1].split()[0]))
                mx.append(float(f[2].split()[0]))
            except Exception:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(mx)),
                "reasons": sorted(reasons), "samples": len(sm)}


def _gen_inputs(cfg, threads=16):
    with cf.ThreadPoolExecutor(max_workers=threads) as ex:
        kv = list(ex.map(lambda l: wl.layer_kv(cfg, l), range(cfg.L)))
        w = list(ex.map(lambda l: wl.layer_weights(cfg, l), range(cfg.L)))
    return kv, w


def _oracle_tokens(cfg, layer):
    """Inputs of the oracle for one layer-sequence, and its non-reference tokens in a
    fixed pseudo-random order."""
    import oracle
    kv = wl.layer_kv(cfg, layer)[0]
    w = wl.layer_weights(cfg, layer)
    non = np.nonzero((np.arange(cfg.T) - cfg.first) % cfg.stride != 0)[0]
    order = np.random.default_rng(12345).permutation(non).astype(np.int32)
    kv64 = wl.stored_to_f64(kv, cfg.kv_dtype)
    ref_pos = oracle.schedule(cfg)
    refs64, _ = oracle.stored_refs(cfg, kv, ref_pos)
    return kv, kv64, ref_pos, refs64, oracle.weights_f64(cfg, w), order


def _oracle_run(cfg, inputs, tokens, budget_s):
    """Run the oracle's write path on `tokens` in growing batches until about budget_s
    seconds have passed; returns (tokens done, seconds)."""
    import oracle
    kv, kv64, ref_pos, refs64, w64, _ = inputs
    done, dt, batch = 0, 0.0, 16
    while dt < budget_s and done < tokens.size:
        toks = tokens[done:done + batch]
        t0 = time.perf_counter()
        oracle.compress_tokens(cfg, kv, w64, toks, kv64=kv64, refs64=refs64, ref_pos=ref_pos)
        dt += time.perf_counter() - t0
        done += toks.size
        batch = min(512, batch * 2)
    return done, dt


def _oracle_shard(cfg_name, layer, shard, n_shards, budget_s, barrier, results):
    """One process of the all-core oracle run: its share of the tokens, started together
    with the others (input generation is outside the timing)."""
    cfg = wl.CONFIGS[cfg_name]
    inputs = _oracle_tokens(cfg, layer)
    toks = inputs[-1][shard::n_shards]
    barrier.wait()
    t0 = time.perf_counter()
    done, _ = _oracle_run(cfg, inputs, toks, budget_s)
    results.put((done, time.perf_counter() - t0))


def cpu_baseline(cfg, budget_s=10.0, layer=0):
    """The oracle as it stands (plain single-threaded fp64 C), on this host: (1) one
    core on random non-reference tokens of one layer for about budget_s seconds; (2)
    the same binary sharded over every host core, one spawned process per core, each
    on its share of the tokens for about budget_s seconds, reporting the job's tokens
    per wall second and the wall time a full parity run of the workload would take at
    that rate (an extrapolation, stated as such)."""
    import multiprocessing as mp
    import oracle
    oracle.build()
    inputs = _oracle_tokens(cfg, layer)
    done, dt = _oracle_run(cfg, inputs, inputs[-1], budget_s)
    single = done / dt
    cores = os.cpu_count() or 1
    ctx = mp.get_context("spawn")
    barrier, results = ctx.Barrier(cores), ctx.Queue()
    procs = [ctx.Process(target=_oracle_shard, args=(cfg.name, layer, i, cores, budget_s, barrier, results))
             for i in range(cores)]
    for p_ in procs:
        p_.start()
    out = [results.get(timeout=600) for _ in procs]
    for p_ in procs:
        p_.join(timeout=60)
    wall = max(t for _, t in out)
    multi = sum(n for n, _ in out) / wall
    n_tok = cfg.L * cfg.B * cfg.T
    return {"value": multi, "unit": UNIT, "cores": cores, "kind": "oracle",
            "host_cores": cores, "single_core_value": single,
            "full_parity_run_s_extrapolated": n_tok / multi,
            "sample": "%d processes (one per host core, os.cpu_count() = %d), each the single-threaded "
                      "fp64 C oracle on its share of the random non-reference tokens of layer %d of %s "
                      "(T=%d), full write path per token (retrieval over the causal pool, mean, f_c "
                      "twice, quantise), %.0f s wall: %d tokens; single core alone: %d tokens in %.1f s. "
                      "full_parity_run_s_extrapolated = all %d tokens of the workload at the all-core rate"
                      % (cores, cores, layer, cfg.name, cfg.T, wall, sum(n for n, _ in out), done, dt,
                         n_tok)}


def run_reference(args, cfg):
    rank, ws, _ = _dist_env()
    if rank != 0:
        return
    import oracle
    kv = wl.layer_kv(cfg, 0)[0]
    w = wl.layer_weights(cfg, 0)
    kv64 = wl.stored_to_f64(kv, cfg.kv_dtype)
    ref_pos = oracle.schedule(cfg)
    refs64, _ = oracle.stored_refs(cfg, kv, ref_pos)
    w64 = oracle.weights_f64(cfg, w)
    per_step = 48
    rng = np.random.default_rng(0)
    times = []
    for step in range(args.warmup + args.steps):
        toks = np.sort(rng.choice(np.nonzero(np.arange(cfg.T) % cfg.stride)[0], per_step, replace=False))
        t0 = time.perf_counter()
        oracle.compress_tokens(cfg, kv, w64, toks.astype(np.int32), kv64=kv64, refs64=refs64,
                               ref_pos=ref_pos)
        if step >= args.warmup:
            times.append(time.perf_counter() - t0)
    tot = sum(times)
    value = per_step * len(times) / tot
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot / len(times),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_description(cfg),
            "cpu_baseline": {"kind": "oracle", "cores": 1, "value": value, "unit": UNIT,
                             "sample": "per step %d random non-reference tokens of layer 0, full "
                                       "write path, single-threaded fp64 C" % per_step},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def read_path(dev, steps=256, reps=3):
    """The sparse read on the long-context workload (131072 tokens, FP8 references):
    `steps` decode steps, each reading 30% random tokens plus the last 512, captured in
    one CUDA graph; plus that workload's compress rate, the restore and attention of the
    same selections, and the decode loop (append + gather + restore + attention per
    step).  Inputs are device-resident."""
    import torch
    from reference_residual_kv_gb300 import rkv
    cfg = wl.CONFIGS["long-131k-fp8ref"]
    kv = torch.from_numpy(wl.layer_kv(cfg, 0)[None].view(np.int16)).view(torch.bfloat16).to(dev)
    w = wl.layer_weights(cfg, 0)
    G = torch.from_numpy(np.stack([w[0][None], w[1][None]]).view(np.int16)).view(torch.bfloat16).to(dev)
    W1, W2 = G[0], G[1]
    W3 = torch.from_numpy(w[2][None].view(np.int16)).view(torch.bfloat16).to(dev)
    p = rkv.params_from_config(cfg)
    bufs = rkv.Buffers(p, device=dev)
    stream = torch.cuda.current_stream(dev)
    bufs.build_ref_pool(kv, stream)
    bufs.compress(kv, W1, W2, W3, stream)
    torch.cuda.synchronize(dev)
    # compress rate of this workload (pool + compress, 5 reps), with per-kernel times
    rkv.rkv_profile_enable(True)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(5):
        bufs.build_ref_pool(kv, stream)
        bufs.compress(kv, W1, W2, W3, stream)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    c_ms = e0.elapsed_time(e1) / 5
    c_prof = {n: round(t / c, 4) for n, (t, c) in rkv.rkv_profile_collect().items()}
    rkv.rkv_profile_enable(False)
    sels = [torch.from_numpy(wl.gather_selection(cfg, s)).to(dev) for s in range(steps)]
    nmax = max(x.numel() for x in sels)
    oz = torch.empty((1, nmax, cfg.d_c), dtype=torch.bfloat16, device=dev)
    om = torch.empty((1, nmax, cfg.W), dtype=torch.bfloat16, device=dev)
    side = torch.cuda.Stream(dev)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        for s_ in sels[:2]:
            bufs.gather(s_.view(1, -1), oz, om, stream=side)
    side.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        for s_ in sels:
            bufs.gather(s_.view(1, -1), oz, om, stream=side)
    g.replay()
    torch.cuda.synchronize(dev)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(reps):
        g.replay()
    b.record(stream)
    torch.cuda.synchronize(dev)
    ms = a.elapsed_time(b) / (reps * steps)
    st = bufs.device_status()
    n_tok = sum(x.numel() for x in sels) / steps
    # restore (decoder + mean + RoPE) of the same selections, fewer steps per graph
    r_steps = min(32, steps)
    Wd = torch.from_numpy(wl.decoder_weights(cfg, 0)[None].view(np.int16)).view(torch.bfloat16).to(dev)
    dk = cfg.N * cfg.D
    ok_ = torch.empty((1, nmax, dk), dtype=torch.bfloat16, device=dev)
    ov_ = torch.empty_like(ok_)
    with torch.cuda.stream(side):
        for s_ in sels[:2]:
            bufs.restore(Wd, s_.view(1, -1), ok_, ov_, cfg.rope_base, stream=side)
    side.synchronize()
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr, stream=side):
        for s_ in sels[:r_steps]:
            bufs.restore(Wd, s_.view(1, -1), ok_, ov_, cfg.rope_base, stream=side)
    gr.replay()
    torch.cuda.synchronize(dev)
    a.record(stream)
    for _ in range(reps):
        gr.replay()
    b.record(stream)
    torch.cuda.synchronize(dev)
    r_ms = a.elapsed_time(b) / (reps * r_steps)
    r_tok = sum(x.numel() for x in sels[:r_steps]) / r_steps
    r_flops = 2.0 * r_tok * cfg.d_c * cfg.W
    r_bytes = r_tok * restore_bytes_per_token(cfg) + bufs.n_ref * cfg.W * 1
    _, tf_burst, tf_sust, _ = _peaks()
    # sparse attention of the same steps over the restored K^, V^ (32 query heads)
    qs = [torch.from_numpy(wl.decode_queries(cfg, 0, st_).view(np.int16)).view(torch.bfloat16).to(dev)
          for st_ in range(r_steps)]
    ao = torch.empty((1, cfg.H, cfg.D), dtype=torch.float32, device=dev)
    with torch.cuda.stream(side):
        bufs.attend(cfg.H, qs[0], ok_, ov_, sels[0].view(1, -1), ao, stream=side)
    side.synchronize()
    ga = torch.cuda.CUDAGraph()
    with torch.cuda.graph(ga, stream=side):
        for st_ in range(r_steps):
            bufs.attend(cfg.H, qs[st_], ok_, ov_, sels[st_].view(1, -1), ao, stream=side)
    ga.replay()
    torch.cuda.synchronize(dev)
    a.record(stream)
    for _ in range(reps):
        ga.replay()
    b.record(stream)
    torch.cuda.synchronize(dev)
    a_ms = a.elapsed_time(b) / (reps * r_steps)
    a_bytes = r_tok * (2 * dk * 2 + 4) + cfg.H * cfg.D * (2 + 4)
    attention = {"ms_per_step": a_ms, "steps": r_steps, "query_heads": cfg.H,
                 "bytes_per_step": a_bytes, "achieved_gbs": a_bytes / (a_ms / 1e3) / 1e9,
                 "frac_of_hbm": a_bytes / (a_ms / 1e3) / 1e9 / _peaks()[0]}
    restore = {"tokens_per_s": r_tok / (r_ms / 1e3), "ms_per_step": r_ms, "steps": r_steps,
               "flops_per_step": r_flops, "achieved_tflops": r_flops / (r_ms / 1e3) / 1e12,
               "frac_of_burst": r_flops / (r_ms / 1e3) / 1e12 / tf_burst,
               "frac_of_sustained": r_flops / (r_ms / 1e3) / 1e12 / tf_sust,
               "bytes_per_step": r_bytes, "achieved_gbs": r_bytes / (r_ms / 1e3) / 1e9,
               "device_status": bufs.device_status()}
    # the decode loop: each of `steps` steps appends the next token (the last `steps`
    # positions of the sequence, encoded against the pool before them), gathers the
    # step's selection, restores its K^ and V^ and attends over them; one CUDA graph
    t0 = cfg.T - steps
    kv_rows = kv.view(cfg.T, -1)
    xs = [kv_rows[t0 + s_].view(1, -1).contiguous() for s_ in range(steps)]

    def decode_step(s_):
        sl = sels[s_].view(1, -1)
        bufs.append(xs[s_], t0 + s_, W1, W2, W3, stream=side)
        bufs.gather(sl, oz, om, stream=side)
        bufs.restore(Wd, sl, ok_, ov_, cfg.rope_base, stream=side)
        bufs.attend(cfg.H, qs[s_ % r_steps], ok_, ov_, sl, ao, stream=side)

    with torch.cuda.stream(side):
        decode_step(0)
    side.synchronize()
    gd = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gd, stream=side):
        for s_ in range(steps):
            decode_step(s_)
    gd.replay()
    torch.cuda.synchronize(dev)
    d_reps = 2
    a.record(stream)
    for _ in range(d_reps):
        gd.replay()
    b.record(stream)
    torch.cuda.synchronize(dev)
    d_ms = a.elapsed_time(b) / (d_reps * steps)
    decode_loop = {"workload": "long-131k-fp8ref: %d decode steps, each: append token t (the last %d "
                               "positions), gather ~%d selected tokens, restore their K^/V^ (RoPE), "
                               "attention of %d query heads; one CUDA graph" % (steps, steps, int(n_tok), cfg.H),
                   "ms_per_step": d_ms, "steps_per_s": 1e3 / d_ms, "device_status": bufs.device_status()}
    per_tok = gather_bytes_per_token(cfg)
    ref_bytes = bufs.n_ref * cfg.W * 1
    bytes_step = n_tok * per_tok + ref_bytes
    hbm, _, _, src = _peaks()
    gbs = bytes_step / (ms / 1e3) / 1e9
    return {"workload": "long-131k-fp8ref: 1 layer x 131072 tokens, FP8 references; %d decode steps of "
                        "~%d selected tokens (30%% random + last 512), one CUDA graph, device-resident"
                        % (steps, int(n_tok)),
            "gathered_tokens_per_s": n_tok / (ms / 1e3), "ms_per_step": ms,
            "bytes_per_step": bytes_step, "bytes_per_token": per_tok, "achieved": gbs, "peak": hbm,
            "unit": "GB/s", "frac": gbs / hbm, "peak_source": "%s HBM copy bandwidth" % src,
            "device_status": st,
            "compress_tokens_per_s": cfg.T / (c_ms / 1e3), "compress_ms": c_ms,
            "compress_kernels_ms": c_prof, "compress": compress_line(cfg, c_ms),
            "restore": restore, "attention": attention,
            "decode_loop": decode_loop}


def compress_line(cfg, ms, kernels_ms=None):
    """Tokens compressed per second and the algorithmic-FLOP fraction of the bf16 burst
    peak for one workload's pool build + compress (all layers and sequences)."""
    fl, n_ref, n_non, pairs = algorithmic(cfg)
    f_alg = sum(fl.values())
    _, tf_burst, tf_sust, src = _peaks()
    ach = f_alg / (ms / 1e3) / 1e12
    out = {"workload": "%s: %d layers x %d seq x %d tokens, kv width %d, d_ff=%d, d_c=%d, stride %d, "
                       "INT%d, %s kv / %s refs" % (cfg.name, cfg.L, cfg.B, cfg.T, cfg.W, cfg.d_ff,
                                                   cfg.d_c, cfg.stride, cfg.bits, cfg.kv_dtype,
                                                   cfg.ref_dtype),
           "tokens_per_s": cfg.L * cfg.B * cfg.T / (ms / 1e3), "ms_per_call": ms,
           "algorithmic_flops": f_alg, "achieved_tflops": ach, "frac_of_burst": ach / tf_burst,
           "frac_of_sustained": ach / tf_sust, "peak_source": "%s bf16 (MEASURED_PEAKS.json)" % src}
    if kernels_ms is not None:
        out["kernels_ms"] = kernels_ms
    return out


def compress_config(name, dev, reps=10):
    """Pool build + compress of every layer of workload `name` with its inputs resident in
    HBM: `reps` calls after 3 warm-ups, CUDA events on the launch stream, per-kernel times
    from the library's own event timing."""
    import torch
    from reference_residual_kv_gb300 import rkv
    cfg = wl.CONFIGS[name]
    kv, w = _gen_inputs(cfg)
    kv_d = torch.from_numpy(np.stack(kv).view(np.int16)).view(torch.bfloat16).to(dev)
    G = torch.from_numpy(np.stack([np.stack([x[0] for x in w]), np.stack([x[1] for x in w])])
                         .view(np.int16)).view(torch.bfloat16).to(dev)
    W3 = torch.from_numpy(np.stack([x[2] for x in w]).view(np.int16)).view(torch.bfloat16).to(dev)
    del kv, w
    bufs = rkv.Buffers(rkv.params_from_config(cfg), device=dev)
    stream = torch.cuda.current_stream(dev)
    for _ in range(3):
        bufs.build_ref_pool(kv_d, stream)
        bufs.compress(kv_d, G[0], G[1], W3, stream)
    torch.cuda.synchronize(dev)
    if bufs.device_status() != 0:
        raise RuntimeError("device status %d in %s" % (bufs.device_status(), name))
    rkv.rkv_profile_enable(True)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        bufs.build_ref_pool(kv_d, stream)
        bufs.compress(kv_d, G[0], G[1], W3, stream)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    prof = {n: round(t / c, 4) for n, (t, c) in rkv.rkv_profile_collect().items()}
    rkv.rkv_profile_enable(False)
    ms = e0.elapsed_time(e1) / reps
    line = compress_line(cfg, ms, prof)
    line["device_status"] = bufs.device_status()
    line["l2"] = "kv %.2f GB > 129 MB L2; no flush" % (kv_d.numel() * 2 / 1e9)
    del kv_d, G, W3, bufs
    torch.cuda.empty_cache()
    return line


def decode_write(cfg, bufs, kv_d, W1, W2, W3, dev, calls=20, reps=3):
    """The write side of one decode step: the token at the last position of every layer
    appended with rkv_append_token (one call for all layers), `calls` calls in one CUDA
    graph.  Bytes per call: W_c1, W_c2, W_c3 of every layer and the pool rows the exact
    distances read; inputs device-resident."""
    import torch
    LB, t = cfg.L * cfg.B, cfg.T - 1
    x = kv_d.view(LB, cfg.T, -1)[:, t].contiguous()
    stream = torch.cuda.current_stream(dev)
    side = torch.cuda.Stream(dev)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        bufs.append(x, t, W1, W2, W3, stream=side)
    side.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        for _ in range(calls):
            bufs.append(x, t, W1, W2, W3, stream=side)
    g.replay()
    torch.cuda.synchronize(dev)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(reps):
        g.replay()
    b.record(stream)
    torch.cuda.synchronize(dev)
    ms = a.elapsed_time(b) / (reps * calls)
    pool = int(bufs.pool_size[t].item())
    w_bytes = cfg.L * (2 * cfg.d_ff * cfg.W + cfg.d_c * cfg.d_ff) * 2
    p_bytes = LB * pool * cfg.W * (1 if cfg.ref_dtype == "fp8" else 2)
    hbm = _peaks()[0]
    by = w_bytes + p_bytes
    return {"workload": "%s: token %d of each of the %d layer-sequences appended in one call "
                        "(pool of %d references)" % (cfg.name, t, LB, pool),
            "ms_per_call": ms, "tokens_per_s": LB / (ms / 1e3), "bytes_per_call": by,
            "achieved_gbs": by / (ms / 1e3) / 1e9, "frac_of_hbm": by / (ms / 1e3) / 1e9 / hbm,
            "device_status": bufs.device_status()}


def run_ours(args, cfg):
    import torch
    rank, ws, local = _dist_env()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    from reference_residual_kv_gb300 import build as rkv_build
    from reference_residual_kv_gb300 import rkv
    rkv_build.build()
    rkv.lib()
    if args.read_path_only:
        # the long-context read path alone (small cases for a profiler)
        print(json.dumps({"read_path": read_path(dev, steps=args.read_steps)}), flush=True)
        return

    kv, w = _gen_inputs(cfg)
    kv_h = torch.from_numpy(np.stack(kv).view(np.int16)).view(torch.bfloat16).pin_memory()
    # W_c1 and W_c2 of all layers in one allocation [2][L][d_ff][W] (the library loads a
    # stage's two gate halves as one tile when W_c2 follows W_c1)
    G_h = torch.from_numpy(np.stack([np.stack([x[0] for x in w]), np.stack([x[1] for x in w])])
                           .view(np.int16)).view(torch.bfloat16).pin_memory()
    W3_h = torch.from_numpy(np.stack([x[2] for x in w]).view(np.int16)).view(torch.bfloat16).pin_memory()
    del kv, w
    kv_d, G, W3 = (t.to(dev) for t in (kv_h, G_h, W3_h))
    W1, W2 = G[0], G[1]

    p = rkv.params_from_config(cfg)
    bufs = rkv.Buffers(p, device=dev)
    LB = cfg.L * cfg.B
    # one decode step's index set, read from every layer (as a filter layer's
    # selection serves the sparse layers that follow it)
    sel1 = wl.gather_selection(cfg, 0, 0)
    sel = torch.from_numpy(np.ascontiguousarray(np.broadcast_to(sel1, (LB, sel1.size)))).to(dev)
    n_sel = sel.shape[1]
    out_z = torch.empty((LB, n_sel, cfg.d_c), dtype=torch.bfloat16, device=dev)
    out_m = torch.empty((LB, n_sel, cfg.W), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        bufs.build_ref_pool(kv_d, stream)
        bufs.compress(kv_d, W1, W2, W3, stream)
        bufs.gather(sel, out_z, out_m, stream=stream)

    def barrier():
        if ws > 1:
            import torch.distributed as dist
            dist.barrier()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    st = bufs.device_status()
    if st != 0:
        raise RuntimeError("device status %d (%s)" % (st, rkv.rkv_status_string(st)))

    # ---- timed region: inputs resident in HBM
    barrier()
    torch.cuda.synchronize(dev)
    rkv.rkv_profile_enable(True)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        e0.record(stream)
        for _ in range(args.steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize(dev)
    prof = rkv.rkv_profile_collect()
    rkv.rkv_profile_enable(False)
    barrier()
    tokens_per_step = cfg.L * cfg.B * cfg.T
    ms, value = job_rate(e0.elapsed_time(e1) / args.steps, tokens_per_step, ws, dev)

    # ---- end to end: kv in from pinned host memory, compressed cache out.  The layers
    # go through in chunks on three streams: chunk c's host->device copy of its kv
    # overlaps chunk c-1's pool build, compress and sparse read and chunk c-2's
    # device->host copy of its records and pool.  The weights stay resident (model
    # parameters); the read's outputs stay on the device (consumed there).
    e2e = None
    if not args.no_e2e:
        C = args.e2e_chunk_layers if cfg.L % args.e2e_chunk_layers == 0 else cfg.L
        nch = cfg.L // C
        pc = rkv.params_from_config(cfg.replace(L=C))
        cbufs = [rkv.Buffers(pc, device=dev) for _ in range(nch)]
        CB = C * cfg.B
        kv_dc = kv_d.view(cfg.L, -1)
        kv_hc = kv_h.view(cfg.L, -1)
        res = []      # per chunk: (device tensor, pinned host tensor) pairs
        for c, cb in enumerate(cbufs):
            pairs = [(t, torch.empty(t.shape, dtype=t.dtype, pin_memory=True))
                     for t in (cb.codes, cb.hdr, cb.ref_idx, cb.ref_vec, cb.ref_sqnorm)]
            res.append(pairs)
        h2d = kv_h.numel() * kv_h.element_size()
        d2h = sum(h.numel() * h.element_size() for pr in res for _, h in pr)
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ev_in = [torch.cuda.Event() for _ in range(nch)]
        ev_done = [torch.cuda.Event() for _ in range(nch)]

        def e2e_step():
            s_in.wait_stream(stream)
            for c in range(nch):
                lc = slice(c * C, (c + 1) * C)
                with torch.cuda.stream(s_in):
                    kv_dc[lc].copy_(kv_hc[lc], non_blocking=True)
                    ev_in[c].record(s_in)
                stream.wait_event(ev_in[c])
                kvc = kv_dc[lc]
                cbufs[c].build_ref_pool(kvc, stream)
                cbufs[c].compress(kvc, G[0][lc], G[1][lc], W3[lc], stream)
                cbufs[c].gather(sel[c * CB:(c + 1) * CB], out_z[c * CB:(c + 1) * CB],
                                out_m[c * CB:(c + 1) * CB], stream=stream)
                ev_done[c].record(stream)
                s_out.wait_event(ev_done[c])
                with torch.cuda.stream(s_out):
                    for d_, h_ in res[c]:
                        h_.copy_(d_, non_blocking=True)
            stream.wait_stream(s_out)

        e2e_step()
        torch.cuda.synchronize(dev)
        st = max(cb.device_status() for cb in cbufs)
        if st != 0:
            raise RuntimeError("device status %d in the end-to-end step" % st)
        barrier()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n_e2e = max(2, min(args.steps, 5))
        a.record(stream)
        for _ in range(n_e2e):
            e2e_step()
        b.record(stream)
        torch.cuda.synchronize(dev)
        ms_e2e, v_e2e = job_rate(a.elapsed_time(b) / n_e2e, tokens_per_step, ws, dev)
        e2e = {"value": v_e2e, "unit": UNIT,
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "ms_per_step": ms_e2e, "chunk_layers": C,
               "note": "per step: every token's kv in from pinned host memory, the compressed cache "
                       "(codes, group extremes, reference slots, stored pool and norms) out to pinned "
                       "host memory; weights resident (model parameters), read outputs consumed on "
                       "the device; layers in chunks of %d, copies overlapped with the compute on "
                       "separate streams" % C}
    if rank != 0:
        return

    hbm, tf_burst, tf_sust, src = _peaks()
    fl, n_ref, n_non, pairs = algorithmic(cfg)
    kernels = {}
    for name, (tot, cnt) in prof.items():
        ent = {"ms_per_launch": tot / cnt, "launches": cnt, "share": None}
        if name in fl:
            ent["tflops"] = fl[name] / (tot / cnt / 1e3) / 1e12
        kernels[name] = ent
    tot_all = sum(v[0] for v in prof.values())
    for name in kernels:
        kernels[name]["share"] = prof[name][0] / tot_all
    dom = max((n for n in prof if n in fl), key=lambda n: prof[n][0])
    dom_ms = prof[dom][0] / prof[dom][1]
    achieved = fl[dom] / (dom_ms / 1e3) / 1e12
    f_alg = sum(fl.values())
    g_ms = prof.get("gather_dequant", (float("nan"), 1))
    # the write path's share of the step: step time less the read's kernel time
    compress_ms = ms - g_ms[0] / g_ms[1]
    kernel_sum_ms = sum(prof[n][0] / args.steps for n in prof if n != "gather_dequant")
    g_bytes = LB * n_sel * gather_bytes_per_token(cfg) + LB * n_ref * cfg.W * 2
    g_gbs = g_bytes / (g_ms[0] / g_ms[1] / 1e3) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded; random-init weights)",
        "config": workload_description(cfg),
        "roofline": {"bound": "tensor", "kernel": dom, "achieved": achieved, "peak": tf_burst,
                     "unit": "TFLOP/s", "frac": achieved / tf_burst,
                     "traffic": NCU_DRAM_BYTES.get(dom) if cfg.L == 32 else None,
                     "peak_source": "%s bf16 burst (MEASURED_PEAKS.json): the timed step is a few "
                                    "ms, not a seconds-long loop" % src,
                     "frac_of_sustained": achieved / tf_sust,
                     "algorithmic_flops_per_launch": fl[dom]},
        "compress_roofline": {"flops_per_step": f_alg, "ms_per_step": compress_ms,
                              "kernel_sum_ms": kernel_sum_ms,
                              "achieved_tflops": f_alg / (compress_ms / 1e3) / 1e12,
                              "frac_of_sustained": f_alg / (compress_ms / 1e3) / 1e12 / tf_sust,
                              "frac_of_burst": f_alg / (compress_ms / 1e3) / 1e12 / tf_burst},
        "gather_roofline": {"bound": "hbm", "tokens_per_launch": LB * n_sel,
                            "bytes_per_launch": g_bytes, "achieved": g_gbs, "peak": hbm,
                            "unit": "GB/s", "frac": g_gbs / hbm,
                            "gathered_tokens_per_s": LB * n_sel / (g_ms[0] / g_ms[1] / 1e3)},
        "kernels": kernels,
        "gpu_launches": int(sum(v[1] for v in prof.values())),
        "clocks": clk.summary(),
        "e2e": e2e,
    }
    line["compress_configs"] = {cfg.name: compress_line(cfg, compress_ms, {
        n: round(prof[n][0] / prof[n][1], 4) for n in prof if n != "gather_dequant"})}
    if not args.no_read_path:
        line["decode_write"] = decode_write(cfg, bufs, kv_d, W1, W2, W3, dev)
    del kv_d, G, W1, W2, W3, bufs, out_z, out_m
    torch.cuda.empty_cache()
    if not args.no_read_path:
        line["read_path"] = read_path(dev, steps=args.read_steps)
        line["compress_configs"][line["read_path"]["compress"]["workload"].split(":")[0]] = \
            line["read_path"]["compress"]
    if not args.no_configs:
        for name in ("qwen2.5-7b-kv", "multimodal-8x4096-int2"):
            line["compress_configs"][name] = compress_config(name, dev)
    if not args.no_cpu_baseline and ws >= 1:
        line["cpu_baseline"] = cpu_baseline(cfg)
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default=WORKLOAD, choices=list(wl.CONFIGS))
    ap.add_argument("--layers", type=int, default=0,
                    help="use only this many layers (small profiling cases; 0 = all)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-read-path", action="store_true",
                    help="skip the long-context sparse-read measurement")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the compress measurements of the other workloads")
    ap.add_argument("--read-path-only", action="store_true",
                    help="run only the long-context sparse-read measurement")
    ap.add_argument("--read-steps", type=int, default=256,
                    help="decode steps of the sparse-read measurement")
    ap.add_argument("--e2e-chunk-layers", type=int, default=E2E_CHUNK_LAYERS,
                    help="layers per chunk of the end-to-end step")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    cfg = wl.CONFIGS[args.config]
    if args.layers > 0:
        cfg = cfg.replace(L=args.layers)
    if cfg.gather_steps == 0:
        cfg = cfg.replace(gather_steps=1)
    if args.impl == "reference":
        run_reference(args, cfg)
    else:
        run_ours(args, cfg)


if __name__ == "__main__":
    main()
