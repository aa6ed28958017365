"""Benchmark of the KVarN hot path on GB300.

One step = one decode step of a batch at a tile boundary: every (sequence,
KV head) commits the tile its newest token just filled (kvarn_encode_tiles on
that tile, K and V) and then every sequence decodes one query token over its
whole context (kvarn_decode). Workload: 32 sequences, 64 query heads on 8 KV
heads, head_dim 128, 16384 tokens, 16-token pages under a random block
table, k4v2 with 128-token tiles (the dense-32B-layer workload).

Prints one JSON line. `value` is packed-KV bytes read by the step's decode
divided by the step time (GB/s); decode tokens/s, the encode throughput of a
full-context encode, and the fp16-KV decode built on the same kernel skeleton
are reported beside it. `--impl reference` times the CPU oracle instead.
"""
from __future__ import annotations

import argparse
import json
import math
import multiprocessing as mp
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode attn packed-KV GB/s (% of HBM peak), tokens/s; encode tokens/s"
WORKLOAD = "dense32b"


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def _workload_desc(wl):
    return (f"{wl.name}: B{wl.num_seqs} Hq{wl.num_q_heads} Hkv{wl.num_kv_heads} D{wl.head_dim} "
            f"L{wl.context} N{wl.tile_tokens} P{wl.page_tokens} K{wl.k_bits}V{wl.v_bits} T{wl.norm_iters}")


# ----------------------------------------------------------------- clocks
class ClockSampler:
    def __init__(self, index: int):
        self.proc = None
        self.path = os.path.join(ROOT, "gpurun_out", f"clocks_{os.getpid()}.csv")
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        self.proc.wait()
        self.f.close()
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for n, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------- oracle (CPU) leg
def _oracle_unit(args):
    """One (sequence, KV head) of the step on the CPU oracle: encode the
    just-filled tile, decode the group's query heads. Returns seconds."""
    os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")
    import numpy as np
    from oracle import attention, codec, layout
    k, v, q, sm, N = args
    lay = layout.DenseLayout(k.shape[-1], N)
    L = k.shape[0]
    tiles = L // N
    ppt = N // 16
    cache = np.zeros((tiles * ppt, 1, lay.page_bytes), np.uint8)
    bt = np.arange(tiles * ppt)[None, :]
    # untimed: the cache as it stood before the step
    attention.encode_into_cache(cache, lay, k[None, None, :(tiles - 1) * N], v[None, None, :(tiles - 1) * N],
                                bt, [0])
    t0 = time.perf_counter()
    ek = codec.encode_tile(k[(tiles - 1) * N:], 4, 2)
    ev = codec.encode_tile(v[(tiles - 1) * N:], 2, 2)
    layout.write_tile(cache, lay, list(range((tiles - 1) * ppt, tiles * ppt)), 0, ek, ev)
    attention.decode(q[None], cache, lay, bt, [L], sm)
    return time.perf_counter() - t0


def oracle_inputs(case, wl, pairs):
    """Host float64 copies of the sampled (b, kvh) inputs."""
    G = wl.group
    work = []
    for b, h in pairs:
        k = case.k[b, h].double().cpu().numpy()
        v = case.v[b, h].double().cpu().numpy()
        q = case.q[b, h * G:(h + 1) * G].double().cpu().numpy()
        work.append((k, v, q, 1 / math.sqrt(wl.head_dim), wl.tile_tokens))
    return work


def oracle_pool(n):
    """Single-threaded spawn workers, one per host core used."""
    cores = min(n, os.cpu_count() or 1)
    os.environ["OPENBLAS_NUM_THREADS"] = "1"
    os.environ["OMP_NUM_THREADS"] = "1"
    return mp.get_context("spawn").Pool(cores), cores


def oracle_time(pool, cores, work):
    """Seconds the sample takes on `cores` cores: the sum of the units' timed
    sections (commit + decode; the cache preparation is not timed) divided
    by the cores working on them."""
    return sum(pool.map(_oracle_unit, work)) / cores


def _pairs(wl, n):
    allp = [(b, h) for b in range(wl.num_seqs) for h in range(wl.num_kv_heads)]
    step = max(1, len(allp) // n)
    return allp[::step][:n]


# ---------------------------------------------------------------- main arm
def run_kvarn(args):
    import torch
    import torch.distributed as dist

    import quantized_kv_cache_kvarn_gb300 as kv
    from quantized_kv_cache_kvarn_gb300 import build as kvbuild
    from quantized_kv_cache_kvarn_gb300 import workloads as W

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0:
        kvbuild.build()
    if world > 1:
        dist.barrier()
    kv.lib()

    wl = W.WORKLOADS[args.workload]
    if args.num_seqs:
        wl = wl.with_(num_seqs=args.num_seqs)
    case = W.make_dense(wl, device=dev, seed=wl.seed + 7919 * rank)
    B, Hq, Hkv, D, L, N = wl.num_seqs, wl.num_q_heads, wl.num_kv_heads, wl.head_dim, wl.context, wl.tile_tokens
    dt = kv.BF16 if wl.dtype == "bf16" else kv.FP16
    lay = kv.dense_layout(D, N, Hkv, case.num_pages, dt, wl.norm_iters)
    cache = kv.alloc_cache(lay, dev)
    err = kv.new_error_word(dev)
    bt = case.block_table
    zeros = torch.zeros(B, dtype=torch.int32, device=dev)
    tiles = L // N
    # untimed: cache as it stood before the step (all tiles but the last)
    kv.encode_tiles(case.k, case.v, lay, zeros, bt, cache, err, chunk_tokens=(tiles - 1) * N)
    last = torch.full((B,), tiles - 1, dtype=torch.int32, device=dev)
    k_last = case.k[:, :, (tiles - 1) * N:]
    v_last = case.v[:, :, (tiles - 1) * N:]
    out = torch.empty((B, Hq, D), dtype=torch.float32, device=dev)
    ws = torch.empty(kv.decode_workspace_bytes(lay, B, Hq, L), dtype=torch.uint8, device=dev)
    sm = W.default_sm_scale(wl)
    stream = torch.cuda.current_stream()

    def step():
        kv.encode_tiles(k_last, v_last, lay, last, bt, cache, err, chunk_tokens=N)
        kv.decode(case.q, lay, cache, bt, case.seq_lens, L, out, ws, err, sm)

    if args.only == "decode":
        # profiling mode: warm-up and timed launches of the decode call alone
        for _ in range(args.warmup + args.steps):
            kv.decode(case.q, lay, cache, bt, case.seq_lens, L, out, ws, err, sm)
        torch.cuda.synchronize()
        assert kv.read_error_flags(err) == 0
        return
    if args.only == "encode":
        for _ in range(args.warmup + args.steps):
            kv.encode_tiles(k_last, v_last, lay, last, bt, cache, err, chunk_tokens=N)
        torch.cuda.synchronize()
        assert kv.read_error_flags(err) == 0
        return

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert kv.read_error_flags(err) == 0, "device error during warm-up"

    # timed region: per-step events around the step and around the decode call
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    clocks = ClockSampler(local) if rank == 0 else None
    time.sleep(0.3 if clocks else 0)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for i in range(args.steps):
        e0, e1, e2 = ev[i]
        e0.record(stream)
        kv.encode_tiles(k_last, v_last, lay, last, bt, cache, err, chunk_tokens=N)
        e1.record(stream)
        kv.decode(case.q, lay, cache, bt, case.seq_lens, L, out, ws, err, sm)
        e2.record(stream)
    stop.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clk = clocks.stop() if clocks else None
    total_ms = start.elapsed_time(stop)
    dec_ms = statistics.mean(e1_.elapsed_time(e2_) for _, e1_, e2_ in ev)
    enc_ms = statistics.mean(e0_.elapsed_time(e1_) for e0_, e1_, _ in ev)
    t = torch.tensor([total_ms], dtype=torch.float64, device=dev)
    if world > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    total_ms = float(t.item())
    assert kv.read_error_flags(err) == 0, "device error in the timed region"

    packed = B * Hkv * L * kv.page_bytes(lay) // 16        # decode: packed bytes read
    ms_step = total_ms / args.steps
    value = world * packed / (ms_step * 1e-3) / 1e9
    peak, peak_kind = _peaks()
    dec_gbs = packed / (dec_ms * 1e-3) / 1e9

    # full-context encode throughput (prefill of the whole cache), same run
    enc_reps = 3
    torch.cuda.synchronize()
    a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(enc_reps):
        kv.encode_tiles(case.k, case.v, lay, zeros, bt, cache, err, chunk_tokens=tiles * N)
    b_.record(stream)
    torch.cuda.synchronize()
    enc_full_ms = a.elapsed_time(b_) / enc_reps
    encode_tok_s = B * tiles * N / (enc_full_ms * 1e-3)

    # fp16-KV decode on the same skeleton (bypass), same workload
    lay16 = kv.dense_layout(D, N, Hkv, case.num_pages, dt, wl.norm_iters)
    cache16 = kv.alloc_fp16_cache(lay16, dev)
    kv.store_fp16(case.k, case.v, lay16, 0, L, bt, cache16, err)
    for _ in range(3):
        kv.decode_fp16(case.q, lay16, cache16, bt, case.seq_lens, L, out, ws, err, sm)
    torch.cuda.synchronize()
    a.record(stream)
    for _ in range(args.steps):
        kv.decode_fp16(case.q, lay16, cache16, bt, case.seq_lens, L, out, ws, err, sm)
    b_.record(stream)
    torch.cuda.synchronize()
    fp16_ms = a.elapsed_time(b_) / args.steps
    del cache16
    fp16_bytes = B * Hkv * L * D * 2 * 2

    # end to end through the public API with host buffers: per step the
    # query, the newest token's K and V and the lengths come from pinned host
    # memory and the output goes back to the host
    q_h = case.q.cpu().pin_memory()
    tok_k = case.k[:, :, L - 1].cpu().pin_memory()
    tok_v = case.v[:, :, L - 1].cpu().pin_memory()
    lens_h = case.seq_lens.cpu().pin_memory()
    out_h = torch.empty((B, Hq, D), dtype=torch.float32).pin_memory()
    q_d = torch.empty_like(case.q)
    lens_d = torch.empty_like(case.seq_lens)

    def e2e_step():
        q_d.copy_(q_h, non_blocking=True)
        lens_d.copy_(lens_h, non_blocking=True)
        case.k[:, :, L - 1].copy_(tok_k, non_blocking=True)
        case.v[:, :, L - 1].copy_(tok_v, non_blocking=True)
        kv.encode_tiles(k_last, v_last, lay, last, bt, cache, err, chunk_tokens=N)
        kv.decode(q_d, lay, cache, bt, lens_d, L, out, ws, err, sm)
        out_h.copy_(out, non_blocking=True)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    a.record(stream)
    for _ in range(args.steps):
        e2e_step()
    b_.record(stream)
    torch.cuda.synchronize()
    e2e_ms = a.elapsed_time(b_) / args.steps
    h2d = q_h.numel() * 2 + lens_h.numel() * 4 + 2 * tok_k.numel() * 2
    d2h = out_h.numel() * 4

    if rank != 0:
        dist.destroy_process_group()
        return

    traffic = None
    try:
        with open(os.path.join(ROOT, "profiles", "decode_dense32b_traffic.json")) as f:
            tr = json.load(f)
        traffic = tr.get("bytes_per_launch") if tr.get("valid") else None
    except Exception:
        pass

    cpu = None
    if world == 1 and not args.no_cpu:
        pairs = _pairs(wl, max(4, min(16, os.cpu_count() or 4)))
        pool, cores = oracle_pool(len(pairs))
        with pool:
            wall = oracle_time(pool, cores, oracle_inputs(case, wl, pairs))
        frac = len(pairs) / (B * Hkv)
        cpu = {"value": round(frac * packed / wall / 1e9, 6), "unit": "GB/s", "cores": cores,
               "kind": "oracle",
               "sample": f"{len(pairs)} of {B * Hkv} (sequence, KV head) units of one step: commit the "
                         f"last tile and decode its {wl.group} query heads over {L} tokens",
               "decode_tokens_per_s": round(frac * B / wall, 4)}

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32 (codes u4/u2; fp16 hi/lo mma operands)", "data": "synthetic",
        "config": {"workload": _workload_desc(wl),
                   "step": "commit the just-filled tile of every (seq, KV head), then decode 1 token per seq",
                   "l2": "inputs larger than L2 (503 MB of packed KV read per step)",
                   "parallelism": f"dp{world} (independent batches per GPU)"},
        "decode_tokens_per_s": round(world * B / (ms_step * 1e-3), 1),
        "decode_gbs": round(dec_gbs, 2), "decode_ms": round(dec_ms, 5),
        "hbm_frac_of_step": round(value / world / peak, 4),
        "commit_ms": round(enc_ms, 5),
        "encode_tokens_per_s": round(encode_tok_s, 1),
        "encode_full_context_ms": round(enc_full_ms, 4),
        "fp16_kv_decode": {"tokens_per_s": round(B / (fp16_ms * 1e-3), 1), "ms": round(fp16_ms, 5),
                           "gbs": round(fp16_bytes / (fp16_ms * 1e-3) / 1e9, 2),
                           "kvarn_speedup": round(fp16_ms / dec_ms, 3)},
        "roofline": {"bound": "hbm", "achieved": round(dec_gbs, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(dec_gbs / peak, 4), "traffic": traffic,
                     "kernel": "kvarn_decode (split kernel + merge), CUDA events on its stream",
                     "peak_kind": peak_kind},
        "e2e": {"value": round(world * packed / (e2e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
                "ms_per_step": round(e2e_ms, 5), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": 3 * args.steps,
        "clocks": clk,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_reference(args):
    """The CPU oracle as the reference arm: each step is a bounded sample of
    the same step (a few (sequence, KV head) units) on the host cores."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import torch
    from quantized_kv_cache_kvarn_gb300 import workloads as W
    wl = W.WORKLOADS[args.workload]
    case = W.make_dense(wl.with_(num_seqs=2), device="cpu")
    pairs = [(b, h) for b in range(2) for h in range(wl.num_kv_heads)][: max(2, min(8, os.cpu_count() or 2))]
    packed = wl.num_seqs * wl.num_kv_heads * wl.context * 120
    work = oracle_inputs(case, wl, pairs)
    pool, cores = oracle_pool(len(pairs))
    with pool:
        oracle_time(pool, cores, work[:cores])  # warm-up: workers import numpy
        times = [oracle_time(pool, cores, work) for _ in range(args.steps)]
    frac = len(pairs) / (wl.num_seqs * wl.num_kv_heads)
    per_step = statistics.mean(times) / frac  # seconds for a whole step
    val = packed / per_step / 1e9
    line = {"metric": METRIC, "value": round(val, 6), "unit": "GB/s", "impl": "reference",
            "n_gpus": int(os.environ.get("WORLD_SIZE", "1")), "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(per_step * 1e3, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": _workload_desc(wl),
                       "step": "commit the just-filled tile of every (seq, KV head), then decode 1 token per seq"},
            "cpu_baseline": {"value": round(val, 6), "unit": "GB/s", "cores": cores, "kind": "oracle",
                             "sample": f"{len(pairs)} of {wl.num_seqs * wl.num_kv_heads} units per step, "
                                       "scaled to the whole step"},
            "e2e": {"value": round(val, 6), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="kvarn", choices=["kvarn", "reference"])
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--no-cpu", action="store_true", help="skip the oracle CPU baseline leg")
    ap.add_argument("--num-seqs", type=int, default=0, help="override the batch (profiling a small case)")
    ap.add_argument("--only", choices=["decode", "encode"], default=None,
                    help="run only warm-up + timed launches of one call, print nothing (for ncu)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_kvarn(args)


if __name__ == "__main__":
    main()
