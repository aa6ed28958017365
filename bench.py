"""Benchmark of the KVarN hot path on GB300.

One step = one decode step of a batch: the cache is brought up to date
(kvarn_encode_tiles on the tiles that step commits) and every sequence
decodes one query token over its whole context (kvarn_decode). The default
workload is the dense-32B layer: 32 sequences, 64 query heads on 8 KV heads,
head_dim 128, 16384 tokens, 16-token pages under a random block table, k4v2
with 128-token tiles; its step commits the tile the newest token just filled
in every (sequence, KV head). Other workloads (--workload):
  toy     1 sequence, 1024 tokens: commit the last tile, decode
  g64     64-token tiles, lengths 2K-32K, fp16 tails: re-commit the last full
          tile of every sequence (one call), decode with the tails
  hybrid  head_dim 256, 65536 tokens: encode the 4096-token prefill chunk
          (tiles 480..511), decode
  mla     64 sequences x 128 heads on a 512-wide int4 latent + fp16 rope:
          commit the last latent tile, decode

Prints one JSON line. `value` = packed-KV bytes the step's decode reads,
divided by the step time (GB/s). Decode tokens/s, a full-context encode
(tokens/s), the fp16-KV decode on the same kernel skeleton (fp16 dense
workloads) and an end-to-end figure with host buffers are reported beside
it. `--impl reference` times the CPU oracle on a bounded sample instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import multiprocessing as mp
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode attn packed-KV GB/s (% of HBM peak), tokens/s; encode tokens/s"
WORKLOAD = "dense32b"
# decode calls timed back to back for the roofline figure (about 25 ms of
# work on the dense-32B workload, so that clock samples fall inside it)
DECODE_CALLS = 200
# workloads measured beside the main one in a default run (each its own
# step, decode call and roofline)
EXTRA_WORKLOADS = ("toy", "g64", "hybrid", "mla")
# the dense-32B workload through the affine comparison codec (gmlx page: an
# fp16 scale and offset per group of 64; compared at 4 and 8 bits)
EXTRA_AFFINE = (4, 8)
# speculative verification (query tokens per sequence) and the raw-record
# window (sink, recent) on the default workload
EXTRA_VERIFY = (("verify4", 4, 0, 0), ("window", 1, 128, 1024))
L2_BYTES = 129 * 1024 * 1024
DECODE_SOURCES = {"dense": ["kvarn_decode.cu", "kvarn_decode_kernel.cuh", "kvarn_common.cuh", "kvarn_merge.cuh"],
                  "mla": ["kvarn_mla.cu", "kvarn_tcgen05.cuh", "kvarn_common.cuh", "kvarn_merge.cuh"]}


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def _tensor_peak():
    """Dense bf16 tensor peak (TFLOP/s), burst: the decode is timed alone.
    fp16 has the same nominal dense rate as bf16."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return 1900.0, "fallback"


def rank_seed(seed: int, rank: int) -> int:
    """Seed of a rank's own synthetic batch: every rank decodes a different
    batch of the same shape (weak scaling, no exchange between ranks)."""
    return seed + 7919 * rank


def max_over_ranks(x: float, device) -> float:
    """The largest of the ranks' values (the slowest rank's time); the value
    itself when no process group is running."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def decode_source_digest(kind="dense"):
    h = hashlib.sha256()
    for f in DECODE_SOURCES[kind]:
        with open(os.path.join(ROOT, "quantized_kv_cache_kvarn_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def _workload_desc(wl):
    s = (f"{wl.name}: B{wl.num_seqs} Hq{wl.num_q_heads} Hkv{wl.num_kv_heads} D{wl.head_dim} "
         f"L{wl.context} N{wl.tile_tokens} P{wl.page_tokens} K{wl.k_bits}"
         f"{'' if wl.rope_dim else 'V%d' % wl.v_bits} T{wl.norm_iters} {wl.dtype}")
    if wl.rope_dim:
        s += f" rope{wl.rope_dim}"
    if wl.var_lengths:
        s += f" lengths U[{wl.min_context},{wl.context}]"
    return s


# ----------------------------------------------------------------- clocks
class E2E:
    """One step end to end: its inputs copied from pinned host memory, the
    step through the public API, its output copied back. The copies run on
    their own streams, double-buffered on the device, so that a step's input
    copy overlaps the step before and its output copy the step after; every
    step still moves its own bytes both ways.

    ins: (pinned host tensor, [device buffer of slot 0, of slot 1]);
    outs: ([device buffer of slot 0, of slot 1], [pinned host buffers]);
    step(slot): the step on the current stream, reading ins[...][1][slot],
    writing outs[...][0][slot]."""

    def __init__(self, ins, outs, step):
        import torch
        self.ins, self.outs, self.step = ins, outs, step
        self.h2d_bytes = sum(h.numel() * h.element_size() for h, _ in ins)
        self.d2h_bytes = sum(d[0].numel() * d[0].element_size() for d, _ in outs)
        self.up, self.down = torch.cuda.Stream(), torch.cuda.Stream()
        ev = torch.cuda.Event
        self.ev_in, self.ev_done, self.ev_out = [ev(), ev()], [ev(), ev()], [ev(), ev()]

    @staticmethod
    def inp(src, dev=None):
        import torch
        dev = src.device if dev is None else dev
        host = src.detach().cpu().contiguous().pin_memory()
        return host, [torch.empty(host.shape, dtype=host.dtype, device=dev) for _ in range(2)]

    @staticmethod
    def outp(like):
        import torch
        return ([like, torch.empty_like(like)],
                [torch.empty(like.shape, dtype=like.dtype).pin_memory() for _ in range(2)])

    def run(self, steps, stream):
        """`steps` steps; everything they issue is ordered before the next
        work recorded on `stream`."""
        import torch
        start = torch.cuda.Event()
        start.record(stream)
        self.up.wait_event(start)
        self.down.wait_event(start)
        for t in range(steps):
            s = t % 2
            with torch.cuda.stream(self.up):
                if t >= 2:
                    self.up.wait_event(self.ev_done[s])  # step t - 2 has read slot s
                for h, d in self.ins:
                    d[s].copy_(h, non_blocking=True)
                self.ev_in[s].record(self.up)
            stream.wait_event(self.ev_in[s])
            if t >= 2:
                stream.wait_event(self.ev_out[s])  # slot s's output of step t - 2 has left
            with torch.cuda.stream(stream):
                self.step(s)
            self.ev_done[s].record(stream)
            with torch.cuda.stream(self.down):
                self.down.wait_event(self.ev_done[s])
                for d, h in self.outs:
                    h[s].copy_(d[s], non_blocking=True)
                self.ev_out[s].record(self.down)
        for s in range(min(2, steps)):
            stream.wait_event(self.ev_out[s])


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed
    region (read-only queries)."""

    def __init__(self):
        self.proc = None
        self.path = os.path.join(tempfile.gettempdir(), f"kvarn_clocks_{os.getpid()}.csv")
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={q}", "--format=csv,noheader,nounits",
                                          "-lms", "50"], stdout=self.f, stderr=subprocess.DEVNULL)
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
    """One unit of the step on the CPU oracle; returns the seconds of its
    timed part (the cache as it stood before the step is prepared untimed).

    dense: (sequence, KV head): commit the step's tile, decode the group.
    mla:   (sequence, 16-head group): commit the last tile, decode the group.
    """
    os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")
    import numpy as np
    from oracle import attention, codec, layout, mla
    kind = args[0]
    if kind == "dense":
        _, k, v, q, sm, N, L, kb, vb, sb = args
        lay = layout.DenseLayout(k.shape[-1], N, kb, vb, sb)
        tiles = L // N
        ppt = N // 16
        cache = np.zeros((max(1, tiles) * ppt, 1, lay.page_bytes), np.uint8)
        bt = np.arange(max(1, tiles) * ppt)[None, :]
        if tiles > 1:
            attention.encode_into_cache(cache, lay, k[None, None, :(tiles - 1) * N],
                                        v[None, None, :(tiles - 1) * N], bt, [0])
        tail = L - tiles * N
        tk = np.zeros((1, 1, N, k.shape[-1]))
        tv = np.zeros_like(tk)
        tk[0, 0, :tail] = k[tiles * N:L]
        tv[0, 0, :tail] = v[tiles * N:L]
        t0 = time.perf_counter()
        if tiles:
            ek = codec.encode_tile(k[(tiles - 1) * N:tiles * N], kb, 2)
            ev = codec.encode_tile(v[(tiles - 1) * N:tiles * N], vb, 2)
            layout.write_tile(cache, lay, list(range((tiles - 1) * ppt, tiles * ppt)), 0, ek, ev)
        attention.decode(q[None], cache, lay, bt, [L], sm, tk, tv)
        return time.perf_counter() - t0
    if kind == "verify":
        _, k, v, q, sm, N, L, Q = args
        lay = layout.DenseLayout(k.shape[-1], N)
        C = attention.verify_committed(L, Q, N)
        tiles = C // N
        ppt = N // 16
        cache = np.zeros((max(1, tiles) * ppt, 1, lay.page_bytes), np.uint8)
        bt = np.arange(max(1, tiles) * ppt)[None, :]
        if tiles > 1:
            attention.encode_into_cache(cache, lay, k[None, None, :(tiles - 1) * N],
                                        v[None, None, :(tiles - 1) * N], bt, [0])
        tk = np.zeros((1, 1, N + Q - 2, k.shape[-1]))
        tv = np.zeros_like(tk)
        tk[0, 0, :L - C] = k[C:L]
        tv[0, 0, :L - C] = v[C:L]
        t0 = time.perf_counter()
        if tiles:
            ek = codec.encode_tile(k[(tiles - 1) * N:tiles * N], 4, 2)
            ev = codec.encode_tile(v[(tiles - 1) * N:tiles * N], 2, 2)
            layout.write_tile(cache, lay, list(range((tiles - 1) * ppt, tiles * ppt)), 0, ek, ev)
        attention.decode_verify(q[None], cache, lay, bt, [L], sm, tk, tv)
        return time.perf_counter() - t0
    _, lat, rope, ql, qr, sm, L = args
    lay = layout.LatentLayout(512, 64, 128)
    tiles = L // 128
    cache = np.zeros((tiles * 8, lay.page_bytes), np.uint8)
    bt = np.arange(tiles * 8)[None, :]
    if tiles > 1:
        mla.encode_into_cache(cache, lay, lat[None, :(tiles - 1) * 128], rope[None, :(tiles - 1) * 128], bt, [0])
    t0 = time.perf_counter()
    enc = codec.encode_tile(lat[(tiles - 1) * 128:tiles * 128], 4, 2)
    mla.write_tile(cache, lay, list(range((tiles - 1) * 8, tiles * 8)), enc, rope[(tiles - 1) * 128:tiles * 128])
    mla.decode(ql[None], qr[None], cache, lay, bt, [L], sm)
    return time.perf_counter() - t0


def oracle_pool(n):
    """Single-threaded spawn workers, one per host core used."""
    cores = min(n, os.cpu_count() or 1)
    os.environ["OPENBLAS_NUM_THREADS"] = "1"
    os.environ["OMP_NUM_THREADS"] = "1"
    return mp.get_context("spawn").Pool(cores), cores


def oracle_time(pool, cores, work):
    """Seconds the sample takes on `cores` cores: the sum of the units' timed
    sections divided by the cores working on them."""
    return sum(pool.map(_oracle_unit, work)) / cores


def oracle_work(wl, case, n, queries=1, qv=None, widths=(4, 2, 4)):
    """Host float64 inputs of n sampled units of the step, and the fraction
    of the whole step they are."""
    if wl.rope_dim:
        units = [(b, hg) for b in range(wl.num_seqs) for hg in range(wl.num_q_heads // 16)]
        step = max(1, len(units) // n)
        pick = units[::step][:n]
        work = []
        for b, hg in pick:
            L = int(case.seq_lens[b])
            work.append(("mla", case.latent[b, :L].double().cpu().numpy(), case.rope[b, :L].double().cpu().numpy(),
                         case.q_latent[b, hg * 16:(hg + 1) * 16].double().cpu().numpy(),
                         case.q_rope[b, hg * 16:(hg + 1) * 16].double().cpu().numpy(),
                         1 / math.sqrt(wl.head_dim + wl.rope_dim), L))
        return work, len(pick) / len(units)
    units = [(b, h) for b in range(wl.num_seqs) for h in range(wl.num_kv_heads)]
    step = max(1, len(units) // n)
    pick = units[::step][:n]
    G = wl.group
    work = []
    for b, h in pick:
        L = int(case.seq_lens[b])
        k, v = case.k[b, h, :L].double().cpu().numpy(), case.v[b, h, :L].double().cpu().numpy()
        if queries > 1:
            work.append(("verify", k, v, qv[b, :, h * G:(h + 1) * G].double().cpu().numpy(),
                         1 / math.sqrt(wl.head_dim), wl.tile_tokens, L, queries))
        else:
            work.append(("dense", k, v, case.q[b, h * G:(h + 1) * G].double().cpu().numpy(),
                         1 / math.sqrt(wl.head_dim), wl.tile_tokens, L) + tuple(widths))
    return work, len(pick) / len(units)


# -------------------------------------------------------------- harnesses
class DenseHarness:
    """Dense (GQA) workloads: the cache, the step's commit and the decode.
    codec "affine": the same workload through the affine comparison codec
    (keys and values at widths[0] bits) on the same decode skeleton."""

    def __init__(self, kv, W, wl, dev, rank, widths=(4, 2, 4), codec="kvarn"):
        import torch
        self.kv, self.wl, self.dev = kv, wl, dev
        self.case = case = W.make_dense(wl, device=dev, seed=rank_seed(wl.seed, rank))
        B, Hkv, D, N = wl.num_seqs, wl.num_kv_heads, wl.head_dim, wl.tile_tokens
        self.dt = kv.BF16 if wl.dtype == "bf16" else kv.FP16
        if codec == "affine":
            self.lay = kv.affine_layout(Hkv, case.num_pages, widths[0], self.dt)
            self.cache = kv.alloc_affine_cache(self.lay, dev)
            self._enc, self._dec = kv.affine_encode_tiles, kv.affine_decode
            self._wsb, self._pb = kv.affine_decode_workspace_bytes, kv.affine_page_bytes
        else:
            self.lay = kv.dense_layout(D, N, Hkv, case.num_pages, self.dt, wl.norm_iters, k_bits=widths[0],
                                       v_bits=widths[1], fp16_scales=widths[2] == 2)
            self.cache = kv.alloc_cache(self.lay, dev)
            self._enc, self._dec = kv.encode_tiles, kv.decode
            self._wsb, self._pb = kv.decode_workspace_bytes, kv.page_bytes
        self.err = kv.new_error_word(dev)
        lens = case.seq_lens.cpu().tolist()
        self.lens = lens
        self.Lmax = max(lens)
        zeros1 = torch.zeros(1, dtype=torch.int32, device=dev)
        # untimed: the cache as it stood before the step; `commit` lists the
        # encode calls of the step
        self.commit = []
        if wl.encode_chunk:
            C = wl.encode_chunk
            start = self.Lmax - C
            self._enc(case.k, case.v, self.lay, torch.zeros(B, dtype=torch.int32, device=dev),
                            case.block_table, self.cache, self.err, chunk_tokens=start)
            ts = torch.full((B,), start // N, dtype=torch.int32, device=dev)
            self.commit.append((case.k[:, :, start:], case.v[:, :, start:], ts, case.block_table, C))
            self.encode_tokens = B * C
        elif len(set(lens)) == 1:
            T = lens[0] // N
            if T > 1:
                self._enc(case.k, case.v, self.lay, torch.zeros(B, dtype=torch.int32, device=dev),
                                case.block_table, self.cache, self.err, chunk_tokens=(T - 1) * N)
            ts = torch.full((B,), T - 1, dtype=torch.int32, device=dev)
            self.commit.append((case.k[:, :, (T - 1) * N:], case.v[:, :, (T - 1) * N:], ts, case.block_table, N))
            self.encode_tokens = B * N
        else:
            # variable lengths: every sequence's last full tile is re-committed
            # in one call, from a [B, Hkv, N, D] buffer of those tiles' raw
            # tokens (where a serving engine keeps the tile that just filled);
            # a sequence without a full tile gets tile_start -1 (skipped)
            ts, src_k, src_v = [], [], []
            for b, L in enumerate(lens):
                T = L // N
                if T > 1:
                    self._enc(case.k[b:b + 1], case.v[b:b + 1], self.lay, zeros1, case.block_table[b:b + 1],
                                    self.cache, self.err, chunk_tokens=(T - 1) * N)
                ts.append(T - 1 if T else -1)
                c0 = max(T - 1, 0) * N
                src_k.append(case.k[b:b + 1, :, c0:c0 + N])
                src_v.append(case.v[b:b + 1, :, c0:c0 + N])
            ck, cv = torch.cat(src_k).contiguous(), torch.cat(src_v).contiguous()
            self.commit.append((ck, cv, torch.tensor(ts, dtype=torch.int32, device=dev), case.block_table, N))
            self.encode_tokens = sum(1 for L in lens if L // N) * N
        # fp16 tails of the partial last tiles
        self.tail_k = self.tail_v = None
        if any(L % N for L in lens):
            self.tail_k = torch.zeros((B, Hkv, N, D), dtype=case.k.dtype, device=dev)
            self.tail_v = torch.zeros_like(self.tail_k)
            for b, L in enumerate(lens):
                c = (L // N) * N
                if L > c:
                    self.tail_k[b, :, :L - c] = case.k[b, :, c:L]
                    self.tail_v[b, :, :L - c] = case.v[b, :, c:L]
        self.out = torch.empty((B, wl.num_q_heads, D), dtype=torch.float32, device=dev)
        self.ws = torch.empty(self._wsb(self.lay, B, wl.num_q_heads, self.Lmax),
                              dtype=torch.uint8, device=dev)
        self.sm = W.default_sm_scale(wl)
        pb = self._pb(self.lay)
        self.packed = sum(Hkv * ((L // N) * N * pb // 16 + (L % N) * D * 2 * 2) for L in lens)
        self.launches = len(self.commit) + 2

    def use_append(self):
        """The step's commit as kvarn_append of each sequence's newest token
        (position len - 1): it completes the last tile in uniform-length
        workloads, which the same launch encodes; the raw tail holds the
        tile's other tokens."""
        import torch
        c, N = self.case, self.wl.tile_tokens
        B, Hkv, D = self.wl.num_seqs, self.wl.num_kv_heads, self.wl.head_dim
        self.ap_tail_k = torch.zeros((B, Hkv, N, D), dtype=c.k.dtype, device=self.dev)
        self.ap_tail_v = torch.zeros_like(self.ap_tail_k)
        for b, L in enumerate(self.lens):
            c0 = ((L - 1) // N) * N
            self.ap_tail_k[b, :, :L - 1 - c0] = c.k[b, :, c0:L - 1]
            self.ap_tail_v[b, :, :L - 1 - c0] = c.v[b, :, c0:L - 1]
        pos = torch.tensor([L - 1 for L in self.lens], device=self.dev)
        ar = torch.arange(B, device=self.dev)
        self.ap_k = c.k[ar, :, pos].contiguous()
        self.ap_v = c.v[ar, :, pos].contiguous()
        self.appending = True
        self.encode_tokens = sum(1 for L in self.lens if L % N == 0) * N

    def encode(self):
        if getattr(self, "appending", False):
            self.kv.append(self.ap_k, self.ap_v, self.case.seq_lens, self.Lmax, self.ap_tail_k, self.ap_tail_v,
                           self.case.block_table, self.lay, self.cache, self.err)
            return
        for k, v, ts, bt, C in self.commit:
            self._enc(k, v, self.lay, ts, bt, self.cache, self.err, chunk_tokens=C)

    def decode(self, q=None, lens=None):
        c = self.case
        self._dec(c.q if q is None else q, self.lay, self.cache, c.block_table,
                       c.seq_lens if lens is None else lens, self.Lmax, self.out, self.ws, self.err, self.sm,
                       self.tail_k, self.tail_v)

    def full_encode(self):
        """Encode every committed tile of the batch (prefill of the cache)."""
        import torch
        c, N = self.case, self.wl.tile_tokens
        if len(set(self.lens)) == 1:
            self._enc(c.k, c.v, self.lay,
                                 torch.zeros(self.wl.num_seqs, dtype=torch.int32, device=self.dev),
                                 c.block_table, self.cache, self.err, chunk_tokens=(self.lens[0] // N) * N)
            return self.wl.num_seqs * (self.lens[0] // N) * N
        zeros1 = torch.zeros(1, dtype=torch.int32, device=self.dev)
        for b, L in enumerate(self.lens):
            if L // N:
                self._enc(c.k[b:b + 1], c.v[b:b + 1], self.lay, zeros1, c.block_table[b:b + 1],
                                     self.cache, self.err, chunk_tokens=(L // N) * N)
        return sum((L // N) * N for L in self.lens)

    def fp16_decode_setup(self):
        """The uncompressed cache on the same skeleton (fp16 workloads)."""
        if self.dt != self.kv.FP16:
            return None
        import torch
        c, wl = self.case, self.wl
        P = 16
        max_pages = (self.Lmax + P - 1) // P
        num_pages = wl.num_seqs * max_pages
        lay16 = self.kv.dense_layout(wl.head_dim, wl.tile_tokens, wl.num_kv_heads, num_pages, self.dt)
        g = torch.Generator(device=self.dev)
        g.manual_seed(wl.seed + 17)
        bt16 = torch.randperm(num_pages, generator=g, device=self.dev).to(torch.int32).reshape(wl.num_seqs, max_pages)
        cache16 = self.kv.alloc_fp16_cache(lay16, self.dev)
        self.kv.store_fp16(c.k, c.v, lay16, 0, (c.k.shape[2] // P) * P, bt16, cache16, self.err)
        ws = torch.empty(self.kv.decode_workspace_bytes(lay16, wl.num_seqs, wl.num_q_heads, self.Lmax),
                         dtype=torch.uint8, device=self.dev)

        def run():
            self.kv.decode_fp16(c.q, lay16, cache16, bt16, c.seq_lens, self.Lmax, self.out, ws, self.err, self.sm)
        fp16_bytes = sum(wl.num_kv_heads * L * wl.head_dim * 2 * 2 for L in self.lens)
        return run, fp16_bytes, (cache16, ws, bt16)

    def e2e_setup(self):
        """Per step from pinned host memory: the queries, the newest token's K
        and V (written into its slot) and the lengths; the output goes back.
        Device copies of the inputs and outputs are double-buffered (E2E)."""
        import torch
        c = self.case
        pos = [L - 1 for L in self.lens]
        tok_k = torch.stack([c.k[b, :, p] for b, p in enumerate(pos)]).cpu().pin_memory()
        tok_v = torch.stack([c.v[b, :, p] for b, p in enumerate(pos)]).cpu().pin_memory()
        ins = [E2E.inp(c.q), E2E.inp(c.seq_lens), E2E.inp(tok_k, self.dev), E2E.inp(tok_v, self.dev)]
        outs = [E2E.outp(self.out)]
        same = len(set(pos)) == 1
        bidx = torch.arange(len(pos), device=self.dev)
        pidx = torch.tensor(pos, device=self.dev)

        def step(slot):
            q_d, lens_d, tk, tv = (x[1][slot] for x in ins)
            if same:
                c.k[:, :, pos[0]] = tk
                c.v[:, :, pos[0]] = tv
            else:
                c.k[bidx, :, pidx] = tk
                c.v[bidx, :, pidx] = tv
            self.encode()
            self.out = outs[0][0][slot]
            self.decode(q_d, lens_d)
        return E2E(ins, outs, step)


class VerifyHarness(DenseHarness):
    """Dense workloads under speculative verification and/or raw records: the
    last Q tokens of every sequence are under verification, the first S
    tokens and the newest R accepted tokens stay raw (S = R = 0: plain
    commit rule). A step commits one compressed tile per (sequence, KV head)
    and runs one kvarn_decode_window (kvarn_decode_verify when S = R = 0)
    over Q query tokens per sequence."""

    def __init__(self, kv, W, wl, dev, rank, Q, S=0, R=0):
        import torch
        self.kv, self.wl, self.dev, self.Q, self.S, self.R = kv, wl, dev, Q, S, R
        self.case = case = W.make_dense(wl, device=dev, seed=rank_seed(wl.seed, rank))
        B, Hkv, D, N = wl.num_seqs, wl.num_kv_heads, wl.head_dim, wl.tile_tokens
        self.dt = kv.BF16 if wl.dtype == "bf16" else kv.FP16
        self.lay = kv.dense_layout(D, N, Hkv, case.num_pages, self.dt, wl.norm_iters)
        self.cache = kv.alloc_cache(self.lay, dev)
        self._enc, self._dec = kv.encode_tiles, kv.decode
        self._wsb, self._pb = kv.decode_workspace_bytes, kv.page_bytes
        self.err = kv.new_error_word(dev)
        lens = case.seq_lens.cpu().tolist()
        self.lens, self.Lmax = lens, max(lens)
        committed = [max(S, (max(0, L - Q + 1 - R) // N) * N) for L in lens]
        ts, src_k, src_v = [], [], []
        for b, C in enumerate(committed):
            T = C // N
            T0 = S // N  # first compressed tile
            if T - 1 > T0:
                kv.encode_tiles(case.k[b:b + 1, :, S:], case.v[b:b + 1, :, S:], self.lay,
                                torch.full((1,), T0, dtype=torch.int32, device=dev), case.block_table[b:b + 1],
                                self.cache, self.err, chunk_tokens=(T - 1 - T0) * N)
            ts.append(T - 1 if T > T0 else -1)
            c0 = max(T - 1, 0) * N
            src_k.append(case.k[b:b + 1, :, c0:c0 + N])
            src_v.append(case.v[b:b + 1, :, c0:c0 + N])
        self.commit = [(torch.cat(src_k).contiguous(), torch.cat(src_v).contiguous(),
                        torch.tensor(ts, dtype=torch.int32, device=dev), case.block_table, N)]
        self.encode_tokens = sum(1 for C in committed if C > S) * N
        cap = R + N + Q - 2
        self.sink_k = self.sink_v = None
        if S:
            self.sink_k = case.k[:, :, :S].contiguous()
            self.sink_v = case.v[:, :, :S].contiguous()
        self.tail_k = torch.zeros((B, Hkv, cap, D), dtype=case.k.dtype, device=dev)
        self.tail_v = torch.zeros_like(self.tail_k)
        for b, (L, C) in enumerate(zip(lens, committed)):
            self.tail_k[b, :, :L - C] = case.k[b, :, C:L]
            self.tail_v[b, :, :L - C] = case.v[b, :, C:L]
        self.qv = W.verify_queries(wl, Q, device=dev, seed=rank_seed(wl.seed, rank))
        self.out = torch.empty((B, Q, wl.num_q_heads, D), dtype=torch.float32, device=dev)
        self.ws = torch.empty(kv.decode_window_workspace_bytes(self.lay, B, wl.num_q_heads, Q, self.Lmax, S, R),
                              dtype=torch.uint8, device=dev)
        self.sm = W.default_sm_scale(wl)
        pb = kv.page_bytes(self.lay)
        self.packed = sum(Hkv * ((C - S) * pb // 16 + (min(S, L) + L - C) * D * 2 * 2)
                          for L, C in zip(lens, committed))
        self.launches = 3
        self.tokens_per_step = B * Q

    def decode(self, q=None, lens=None):
        c = self.case
        args = (self.qv if q is None else q, self.lay, self.cache, c.block_table,
                c.seq_lens if lens is None else lens, self.Lmax, self.out, self.ws, self.err, self.sm)
        if self.S or self.R:
            self.kv.decode_window(*args, sink_k=self.sink_k, sink_v=self.sink_v, recent_tokens=self.R,
                                  tail_k=self.tail_k, tail_v=self.tail_v)
        else:
            self.kv.decode_verify(*args, self.tail_k, self.tail_v)

    def full_encode(self):
        return DenseHarness.full_encode(self)

    def fp16_decode_setup(self):
        return None

    def e2e_setup(self):
        """Per step from pinned host memory: the Q query rows and the lengths;
        the Q outputs go back."""
        ins = [E2E.inp(self.qv), E2E.inp(self.case.seq_lens)]
        outs = [E2E.outp(self.out)]

        def step(slot):
            self.encode()
            self.out = outs[0][0][slot]
            self.decode(ins[0][1][slot], ins[1][1][slot])
        return E2E(ins, outs, step)


class LatentHarness:
    """The MLA workload: latent cache, the step's commit, MLA decode."""

    def __init__(self, kv, W, wl, dev, rank):
        import torch
        self.kv, self.wl, self.dev = kv, wl, dev
        self.case = case = W.make_latent(wl, device=dev, seed=rank_seed(wl.seed, rank))
        B, L = wl.num_seqs, wl.context
        self.lay = kv.latent_layout(case.num_pages, kv.BF16, wl.norm_iters)
        self.cache = kv.alloc_cache(self.lay, dev)
        self.err = kv.new_error_word(dev)
        T = L // 128
        kv.encode_latent(case.latent, case.rope, self.lay, torch.zeros(B, dtype=torch.int32, device=dev),
                         case.block_table, self.cache, self.err, chunk_tokens=(T - 1) * 128)
        self.ts = torch.full((B,), T - 1, dtype=torch.int32, device=dev)
        self.lat_last = case.latent[:, (T - 1) * 128:]
        self.rope_last = case.rope[:, (T - 1) * 128:]
        self.lens = [L] * B
        self.Lmax = L
        self.out = torch.empty((B, wl.num_q_heads, 512), dtype=torch.float32, device=dev)
        self.ws = torch.empty(kv.decode_workspace_bytes(self.lay, B, wl.num_q_heads, L), dtype=torch.uint8,
                              device=dev)
        self.sm = W.default_sm_scale(wl)
        self.packed = B * L * kv.page_bytes(self.lay) // 16
        self.encode_tokens = B * 128
        self.launches = 3

    def encode(self):
        self.kv.encode_latent(self.lat_last, self.rope_last, self.lay, self.ts, self.case.block_table, self.cache,
                              self.err, chunk_tokens=128)

    def decode(self, q=None, lens=None):
        c = self.case
        self.kv.decode_mla(c.q_latent if q is None else q, c.q_rope, self.lay, self.cache, c.block_table,
                           c.seq_lens if lens is None else lens, self.Lmax, self.out, self.ws, self.err, self.sm)

    def full_encode(self):
        import torch
        c = self.case
        self.kv.encode_latent(c.latent, c.rope, self.lay,
                              torch.zeros(self.wl.num_seqs, dtype=torch.int32, device=self.dev),
                              c.block_table, self.cache, self.err, chunk_tokens=self.Lmax)
        return self.wl.num_seqs * self.Lmax

    def fp16_decode_setup(self):
        return None

    def e2e_setup(self):
        """Per step from pinned host memory: the latent queries, the newest
        token's latent (written into its slot) and the lengths; the output
        goes back."""
        c = self.case
        ins = [E2E.inp(c.q_latent), E2E.inp(c.seq_lens), E2E.inp(c.latent[:, self.Lmax - 1].contiguous())]
        outs = [E2E.outp(self.out)]

        def step(slot):
            q_d, lens_d, tok_d = (x[1][slot] for x in ins)
            c.latent[:, self.Lmax - 1].copy_(tok_d)
            self.encode()
            self.out = outs[0][0][slot]
            self.decode(q_d, lens_d)
        return E2E(ins, outs, step)


# ---------------------------------------------------------------- main arm
def roofline_of(H, wl, dec_ms, traffic=None, kernel=None):
    """Roofline object of a decode call of `dec_ms` ms: HBM for the dense
    workloads (packed bytes read), bf16 tensor peak for MLA (algorithmic
    flops: 2 per multiply-add of the scores, latent + rope width, and of the
    output, latent width, per sequence, head and token)."""
    peak, peak_kind = _peaks()
    gbs = H.packed / (dec_ms * 1e-3) / 1e9
    if wl.rope_dim:
        flops = 2.0 * sum(H.lens) * wl.num_q_heads * (2 * wl.head_dim + wl.rope_dim)
        tpk, tpk_kind = _tensor_peak()
        tf = flops / (dec_ms * 1e-3) / 1e12
        return {"bound": "tensor", "achieved": round(tf, 2), "peak": tpk, "unit": "TFLOP/s",
                "frac": round(tf / tpk, 4), "traffic": traffic, "kernel": kernel, "peak_kind": tpk_kind,
                "flops_per_launch": flops, "hbm_gbs": round(gbs, 2), "hbm_frac": round(gbs / peak, 4)}
    return {"bound": "hbm", "achieved": round(gbs, 2), "peak": peak, "unit": "GB/s", "frac": round(gbs / peak, 4),
            "traffic": traffic, "kernel": kernel, "peak_kind": peak_kind, "bytes_per_launch": H.packed}


def captured_traffic(wl):
    """DRAM bytes per decode launch of workload `wl` at its preset widths, one
    query token and no raw records, from the committed ncu capture, while
    the decode kernel's sources hash to the captured digest; else None."""
    try:
        with open(os.path.join(ROOT, "profiles", "decode_traffic.json")) as fh:
            entry = json.load(fh).get(wl.name)
        kind = "mla" if wl.rope_dim else "dense"
        if entry and entry.get("source_digest") == decode_source_digest(kind):
            return entry.get("bytes_per_launch")
    except Exception:
        pass
    return None


def measure_extra(kv, W, name, dev, rank, steps, warmup, codec="kvarn", bits=4, queries=1, sink=0, recent=0):
    """One more workload in the same run: its step (commit + decode, K back
    to back), its decode call (DECODE_CALLS back to back) and its commit,
    with the roofline of the decode call. A workload whose packed reads fit
    in L2 (toy) is timed one step at a time with L2 flushed between steps
    (outside the timed events)."""
    import torch
    wl = W.WORKLOADS[name]
    if codec == "affine":
        H = DenseHarness(kv, W, wl, dev, rank, widths=(bits, bits, 2), codec="affine")
    elif queries > 1 or sink or recent:
        H = VerifyHarness(kv, W, wl, dev, rank, queries, sink, recent)
    else:
        H = LatentHarness(kv, W, wl, dev, rank) if wl.rope_dim else DenseHarness(kv, W, wl, dev, rank)
    stream = torch.cuda.current_stream()
    ev = lambda: torch.cuda.Event(enable_timing=True)
    for _ in range(warmup):
        H.encode()
        H.decode()
    torch.cuda.synchronize()
    small = H.packed < L2_BYTES
    if small:
        flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
        times, dtimes, ctimes = [], [], []
        for _ in range(steps):
            flush.fill_(1.0)
            a, b_ = ev(), ev()
            a.record(stream)
            H.encode()
            H.decode()
            b_.record(stream)
            flush.fill_(2.0)
            c0, c1, c2 = ev(), ev(), ev()
            c0.record(stream)
            H.encode()
            c1.record(stream)
            flush.fill_(3.0)
            c2.record(stream)
            d0, d1 = ev(), ev()
            d0.record(stream)
            H.decode()
            d1.record(stream)
            torch.cuda.synchronize()
            times.append(a.elapsed_time(b_))
            ctimes.append(c0.elapsed_time(c1))
            dtimes.append(d0.elapsed_time(d1))
        ms_step, dec_ms, com_ms = statistics.median(times), statistics.median(dtimes), statistics.median(ctimes)
        del flush
    else:
        a, b_ = ev(), ev()
        a.record(stream)
        for _ in range(steps):
            H.encode()
            H.decode()
        b_.record(stream)
        d0, d1 = ev(), ev()
        d0.record(stream)
        for _ in range(DECODE_CALLS):
            H.decode()
        d1.record(stream)
        cs = []
        for _ in range(steps):
            c0, c1 = ev(), ev()
            c0.record(stream)
            H.encode()
            c1.record(stream)
            H.decode()
            cs.append((c0, c1))
        torch.cuda.synchronize()
        ms_step = a.elapsed_time(b_) / steps
        dec_ms = d0.elapsed_time(d1) / DECODE_CALLS
        com_ms = statistics.mean(x.elapsed_time(y) for x, y in cs)
    assert kv.read_error_flags(H.err) == 0, f"device error in the {name} workload"
    desc = _workload_desc(wl)
    if codec == "affine":
        desc = desc.replace("K4V2", f"affine K{bits}V{bits} (groups of 64, fp16 scale and offset)")
    if queries > 1:
        desc += f", {queries} query tokens per sequence (kvarn_decode_verify)"
    if sink or recent:
        desc += f", raw sink {sink} + recent {recent} (kvarn_decode_window)"
    out = {"workload": desc, "ms_per_step": round(ms_step, 5),
           "value": round(H.packed / (ms_step * 1e-3) / 1e9, 2), "unit": "GB/s",
           "decode_ms": round(dec_ms, 5), "commit_ms": round(com_ms, 5), "commit_tokens": H.encode_tokens,
           "decode_tokens_per_s": round(wl.num_seqs * queries / (ms_step * 1e-3), 1),
           "l2": ("packed reads fit in L2: one step per timing, L2 flushed between steps (median of K)" if small
                  else f"inputs larger than L2 ({H.packed / 1e6:.0f} MB of packed KV read per step)"),
           "roofline": roofline_of(H, wl, dec_ms,
                                   traffic=(captured_traffic(wl) if codec == "kvarn" and queries == 1
                                            and not (sink or recent) else None),
                                   kernel=f"decode call, {'median of K single' if small else str(DECODE_CALLS) + ' back-to-back'} calls")}
    del H
    torch.cuda.empty_cache()
    return out


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
    widths = (args.kbits, args.vbits, 2 if args.fp16_scales else 4)
    if widths != (4, 2, 4):
        if wl.rope_dim or args.queries > 1 or args.sink or args.recent or args.append:
            raise SystemExit("--kbits/--vbits/--fp16-scales apply to the plain dense step")
        wl = wl.with_(k_bits=args.kbits, v_bits=args.vbits)
    if args.queries > 1 or args.sink or args.recent:
        if wl.rope_dim:
            raise SystemExit("--queries, --sink and --recent apply to the dense workloads")
        H = VerifyHarness(kv, W, wl, dev, rank, args.queries, args.sink, args.recent)
    elif wl.rope_dim:
        H = LatentHarness(kv, W, wl, dev, rank)
    elif args.codec == "affine":
        H = DenseHarness(kv, W, wl, dev, rank, (args.kbits, args.kbits, 2), codec="affine")
    else:
        H = DenseHarness(kv, W, wl, dev, rank, widths)
    if args.append:
        if wl.rope_dim or args.queries > 1 or args.sink or args.recent or wl.encode_chunk:
            raise SystemExit("--append applies to the plain dense step")
        H.use_append()
    stream = torch.cuda.current_stream()
    B = wl.num_seqs

    def ev():
        return torch.cuda.Event(enable_timing=True)

    if args.only == "decode":
        # profiling mode: warm-up and timed launches of the decode call alone
        for _ in range(args.warmup + args.steps):
            H.decode()
        torch.cuda.synchronize()
        assert kv.read_error_flags(H.err) == 0
        return
    if args.only == "encode":
        for _ in range(args.warmup + args.steps):
            H.encode()
        torch.cuda.synchronize()
        assert kv.read_error_flags(H.err) == 0
        return
    if args.only == "full-encode":
        for _ in range(args.warmup + args.steps):
            H.full_encode()
        torch.cuda.synchronize()
        assert kv.read_error_flags(H.err) == 0
        return

    # the clock sampler starts first, so that the warm-up steps run right
    # before the timed region (an idle GPU lowers its clocks within a few
    # hundred milliseconds)
    clocks = ClockSampler() if rank == 0 else None
    time.sleep(0.3 if clocks else 0)
    for _ in range(args.warmup):
        H.encode()
        H.decode()
    torch.cuda.synchronize()
    assert kv.read_error_flags(H.err) == 0, "device error during warm-up"

    # timed region: the K steps back to back, events only at its two ends (an
    # event recorded between two kernels holds the second one back by a few
    # microseconds, about 12 us per step with three of them)
    evs = [(ev(), ev(), None) for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    start, stop = ev(), ev()
    start.record(stream)
    for _ in range(args.steps):
        H.encode()
        H.decode()
    stop.record(stream)
    torch.cuda.synchronize()
    # the same K steps again with events around each commit (its duration),
    # then K decode calls back to back: the decode call's average duration,
    # which the roofline uses (its packed reads exceed the L2 as in the step)
    for e0, e1, _ in evs:
        e0.record(stream)
        H.encode()
        e1.record(stream)
        H.decode()
    d0, d1 = ev(), ev()
    d0.record(stream)
    for _ in range(DECODE_CALLS):
        H.decode()
    d1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clk = clocks.stop() if clocks else None
    total_ms = start.elapsed_time(stop)
    dec_ms = d0.elapsed_time(d1) / DECODE_CALLS
    enc_ms = statistics.mean(a.elapsed_time(b) for a, b, _ in evs)
    total_ms = max_over_ranks(total_ms, dev)
    assert kv.read_error_flags(H.err) == 0, "device error in the timed region"

    ms_step = total_ms / args.steps
    value = world * H.packed / (ms_step * 1e-3) / 1e9
    peak, peak_kind = _peaks()
    dec_gbs = H.packed / (dec_ms * 1e-3) / 1e9

    # full-context encode throughput (prefill of the whole cache), same run
    torch.cuda.synchronize()
    a, b_ = ev(), ev()
    reps = 3
    a.record(stream)
    for _ in range(reps):
        enc_tokens = H.full_encode()
    b_.record(stream)
    torch.cuda.synchronize()
    enc_full_ms = a.elapsed_time(b_) / reps
    encode_tok_s = enc_tokens / (enc_full_ms * 1e-3)

    # fp16-KV decode on the same kernel skeleton
    fp16 = None
    f = H.fp16_decode_setup()
    if f is not None:
        run16, bytes16, keep = f
        for _ in range(3):
            run16()
        torch.cuda.synchronize()
        a.record(stream)
        for _ in range(args.steps):
            run16()
        b_.record(stream)
        torch.cuda.synchronize()
        ms16 = a.elapsed_time(b_) / args.steps
        fp16 = {"tokens_per_s": round(B / (ms16 * 1e-3), 1), "ms": round(ms16, 5),
                "gbs": round(bytes16 / (ms16 * 1e-3) / 1e9, 2), "kvarn_decode_speedup": round(ms16 / dec_ms, 3)}
        del keep, run16

    # end to end through the public API with host buffers
    e2e = H.e2e_setup()
    e2e.run(3, stream)
    torch.cuda.synchronize()
    a.record(stream)
    e2e.run(args.steps, stream)
    b_.record(stream)
    torch.cuda.synchronize()
    e2e_ms = a.elapsed_time(b_) / args.steps
    h2d, d2h = e2e.h2d_bytes, e2e.d2h_bytes

    # the same K steps captured once in a CUDA graph and replayed (every
    # launch takes host sizes and pointers, so the graph replays the step as
    # issued; a serving loop would run it this way)
    graph_ms = None
    try:
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(side):
            H.encode()
            H.decode()
            side.synchronize()
            with torch.cuda.graph(g, stream=side):
                for _ in range(args.steps):
                    H.encode()
                    H.decode()
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        a.record(stream)
        g.replay()
        b_.record(stream)
        torch.cuda.synchronize()
        graph_ms = a.elapsed_time(b_) / args.steps
        assert kv.read_error_flags(H.err) == 0, "device error in the graph replay"
        del g
    except RuntimeError as exc:
        print(f"graph replay not timed: {exc}", file=sys.stderr)

    if rank != 0:
        dist.destroy_process_group()
        return

    # the capture is of the workload's own decode: the preset widths, one
    # query token, no raw records (the append step decodes the same pages)
    same = widths == (4, 2, 4) and args.queries == 1 and not (args.sink or args.recent) and args.codec == "kvarn"
    traffic = captured_traffic(wl) if same and not args.num_seqs else None

    cpu = None
    if world == 1 and not args.no_cpu and not (args.sink or args.recent) and args.codec == "kvarn":
        n = max(4, min(16, os.cpu_count() or 4))
        work, frac = oracle_work(wl, H.case, n, args.queries, getattr(H, "qv", None), widths)
        pool, cores = oracle_pool(len(work))
        with pool:
            wall = oracle_time(pool, cores, work)
        # the same oracle on one core: two of the sampled units
        one = work[:2]
        pool1, _ = oracle_pool(1)
        with pool1:
            wall1 = oracle_time(pool1, 1, one)
        frac1 = frac * len(one) / len(work)
        unit = "(sequence, 16-head group)" if wl.rope_dim else "(sequence, KV head)"
        cpu = {"value": round(frac * H.packed / wall / 1e9, 6), "unit": "GB/s", "cores": cores, "kind": "oracle",
               "sample": f"{len(work)} {unit} units of one step ({frac:.4f} of it): commit and decode, "
                         f"float64 oracle on {cores} single-threaded host processes",
               "decode_tokens_per_s": round(frac * B * args.queries / wall, 4),
               "single_core": {"value": round(frac1 * H.packed / wall1 / 1e9, 6), "unit": "GB/s", "cores": 1,
                               "sample": f"{len(one)} of the same units on one single-threaded process"}}

    kernel_desc = (f"decode call (split kernel + merge kernel): {DECODE_CALLS} calls back to back after the timed "
                   "steps, CUDA events on its stream")
    roofline = roofline_of(H, wl, dec_ms, traffic, kernel_desc)
    # the full-context encode against HBM: its fp16/bf16 K and V read once
    # and its pages written once (algorithmic bytes)
    enc_bytes = enc_tokens * wl.num_kv_heads * (2 * 2 * wl.head_dim if not wl.rope_dim else 2 * (wl.head_dim + wl.rope_dim))
    enc_bytes += H.packed
    enc_gbs = enc_bytes / (enc_full_ms * 1e-3) / 1e9
    encode_roofline = {"bound": "hbm", "achieved": round(enc_gbs, 2), "peak": peak, "unit": "GB/s",
                       "frac": round(enc_gbs / peak, 4), "bytes_per_launch": enc_bytes,
                       "kernel": "full-context encode (encode_tiles over every committed tile), 3 calls",
                       "note": "ALU- and latency-bound, not HBM-bound: issue-slot use from ncu in profiles/"}
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": (f"f32 (codes u{args.kbits}/u{args.vbits}, {'fp16' if args.fp16_scales else 'fp32'} scales; "
                  f"fp16 hi/lo mma operands)"), "data": "synthetic",
        "config": {"workload": _workload_desc(wl) + (" fp16-scales" if args.fp16_scales else ""),
                   "step": (f"commit one compressed tile per (seq, KV head), then {args.queries} query token(s) "
                            f"per seq, raw sink {args.sink} + recent {args.recent} (kvarn_decode_window)"
                            if args.sink or args.recent else
                            f"commit one accepted tile per (seq, KV head), then verify {args.queries} tokens "
                            f"per seq (kvarn_decode_verify)" if args.queries > 1 else
                            "kvarn_append of the newest token (commits the tile it fills), then decode 1 token per seq"
                            if args.append else
                            "encode the 4096-token prefill chunk, then decode 1 token per seq" if wl.encode_chunk
                            else "commit one tile per (seq, KV head), then decode 1 token per seq"),
                   "l2": f"inputs larger than L2 ({H.packed / 1e6:.0f} MB of packed KV read per step)",
                   "parallelism": f"dp{world} (independent batches per GPU)"},
        "decode_tokens_per_s": round(world * B * args.queries / (ms_step * 1e-3), 1),
        "decode_gbs": round(dec_gbs, 2), "decode_ms": round(dec_ms, 5),
        "commit_ms": round(enc_ms, 5), "commit_tokens": H.encode_tokens,
        "encode_tokens_per_s": round(encode_tok_s, 1), "encode_full_context_ms": round(enc_full_ms, 4),
        "fp16_kv_decode": fp16,
        "roofline": roofline,
        "encode_roofline": encode_roofline,
        "e2e": {"value": round(world * H.packed / (e2e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
                "ms_per_step": round(e2e_ms, 5), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "copies": "from and to pinned host memory every step, on their own streams, double-buffered on "
                          "the device: a step's input copy overlaps the step before, its output copy the step after"},
        "gpu_launches": H.launches * args.steps,
        "graph": None if graph_ms is None else {
            "ms_per_step": round(graph_ms, 5),
            "value": round(world * H.packed / (graph_ms * 1e-3) / 1e9, 2), "unit": "GB/s"},
        "clocks": clk,
        "cpu_baseline": cpu,
    }
    plain = not (args.num_seqs or args.queries > 1 or args.sink or args.recent or args.append
                 or widths != (4, 2, 4) or args.no_extra or args.codec != "kvarn")
    if plain and world == 1 and args.workload == WORKLOAD:
        # the other workloads of the same family, each measured on its own
        del H, e2e, f
        torch.cuda.empty_cache()
        line["workloads"] = {}
        for name in EXTRA_WORKLOADS:
            line["workloads"][name] = measure_extra(kv, W, name, dev, rank, args.steps, args.warmup)
        for bits in EXTRA_AFFINE:
            line["workloads"][f"affine{bits}"] = measure_extra(kv, W, WORKLOAD, dev, rank, args.steps, args.warmup,
                                                               codec="affine", bits=bits)
        for key, q, sk, rc in EXTRA_VERIFY:
            line["workloads"][key] = measure_extra(kv, W, WORKLOAD, dev, rank, args.steps, args.warmup,
                                                   queries=q, sink=sk, recent=rc)
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_reference(args):
    """The CPU oracle as the reference arm: each step is a bounded sample of
    the same step on the host cores, scaled to the whole step."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from quantized_kv_cache_kvarn_gb300 import workloads as W
    wl = W.WORKLOADS[args.workload]
    small = wl.with_(num_seqs=min(2, wl.num_seqs))
    case = (W.make_latent if wl.rope_dim else W.make_dense)(small, device="cpu")
    n = max(2, min(8, os.cpu_count() or 2))
    work, _ = oracle_work(small, case, n)
    units_total = (wl.num_seqs * wl.num_q_heads // 16) if wl.rope_dim else (wl.num_seqs * wl.num_kv_heads)
    frac = len(work) / units_total
    lens = case.seq_lens.tolist()
    mean_len = sum(lens) / len(lens)
    if wl.rope_dim:
        packed = wl.num_seqs * wl.context * 6528 // 16
    else:
        page = 12 * wl.head_dim + 256 + 8 * wl.head_dim * 16 // wl.tile_tokens
        packed = int(wl.num_seqs * wl.num_kv_heads * mean_len * page / 16)
    pool, cores = oracle_pool(len(work))
    with pool:
        oracle_time(pool, cores, work[:cores])  # warm-up: workers import numpy
        times = [oracle_time(pool, cores, work) for _ in range(args.steps)]
    per_step = statistics.mean(times) / frac
    val = packed / per_step / 1e9
    line = {"metric": METRIC, "value": round(val, 6), "unit": "GB/s", "impl": "reference",
            "n_gpus": int(os.environ.get("WORLD_SIZE", "1")), "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(per_step * 1e3, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": _workload_desc(wl) + (" fp16-scales" if args.fp16_scales else ""),
                       "step": "commit one tile per (seq, KV head), then decode 1 token per seq"},
            "cpu_baseline": {"value": round(val, 6), "unit": "GB/s", "cores": cores, "kind": "oracle",
                             "sample": f"{len(work)} of {units_total} units per step, scaled to the whole step"},
            "e2e": {"value": round(val, 6), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="kvarn", choices=["kvarn", "reference"])
    ap.add_argument("--workload", default=WORKLOAD, choices=["toy", "dense32b", "g64", "hybrid", "mla"])
    ap.add_argument("--no-cpu", action="store_true", help="skip the oracle CPU baseline leg")
    ap.add_argument("--num-seqs", type=int, default=0, help="override the batch (profiling a small case)")
    ap.add_argument("--queries", type=int, default=1,
                    help="query tokens per sequence under speculative verification (dense workloads)")
    ap.add_argument("--kbits", type=int, default=4, help="key code width (2, 3, 4, 5, 6, 8)")
    ap.add_argument("--vbits", type=int, default=2, help="value code width (2, 3, 4, 5, 6, 8)")
    ap.add_argument("--fp16-scales", action="store_true", help="fp16 scales in the page (else fp32)")
    ap.add_argument("--codec", choices=["kvarn", "affine"], default="kvarn",
                    help="affine: the comparison codec (keys and values at --kbits) on the same skeleton")
    ap.add_argument("--append", action="store_true",
                    help="commit through kvarn_append of the newest token (fused append + commit)")
    ap.add_argument("--sink", type=int, default=0, help="raw sink tokens (a multiple of the tile)")
    ap.add_argument("--recent", type=int, default=0, help="newest accepted tokens kept raw")
    ap.add_argument("--no-extra", action="store_true",
                    help="measure only the named workload (a default run adds the toy, g64, hybrid and MLA "
                         "workloads as extra keys)")
    ap.add_argument("--only", choices=["decode", "encode", "full-encode"], default=None,
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
