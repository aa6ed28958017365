"""Seeded synthetic inputs shaped like the workloads the KVarN pages describe.

This module holds shapes, random draws, block tables and sequence lengths
only: none of the codec's or the attention's arithmetic lives here, so both
the CUDA path and the CPU oracle can take their inputs from it.

The five named workloads follow the problem statement of the KVarN
vLLM-fork review ("KVarN ... KV cache quantization", paragraphs on the
k4v2_g128 preset, the 64-token variant, MLA and hybrid models):

* ``toy``      1 sequence, GQA 4 (4 query heads on 1 KV head), head_dim 128,
               1024 tokens (8 tiles of 128), fp16 N(0,1) with channels
               {7, 31, 64, 100} scaled x20 in K and V.
* ``dense32b`` 32 sequences, 64 query heads on 8 KV heads, head_dim 128,
               16384 tokens, 16-token pages under a random block table,
               fp16 N(0,1) where each (head, channel) is an outlier channel
               with probability 0.01, holding 10 x Student-t(3) draws.
* ``g64``      as ``dense32b`` with 64-token tiles and lengths drawn
               uniformly from 2048..32768; the partial last tile stays fp16.
* ``hybrid``   8 sequences, 24 query heads on 4 KV heads, head_dim 256,
               65536 tokens, bf16 N(0,1) times a per-(head, channel)
               log-normal scale exp(N(0,1)); a 4096-token chunk is encoded
               during the step.
* ``mla``      64 sequences, 128 query heads on one shared 512-wide latent
               plus a 64-wide fp16 rope part, 8192 tokens, latent bf16
               N(0,1) with 2% outlier channels x15.

Everything is drawn with ``torch.Generator`` on the requested device, so a
case can be built directly in device memory at full size, or on the host
for the small cases the oracle checks.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    context: int              # tokens per sequence (the maximum when lengths vary)
    tile_tokens: int
    page_tokens: int
    dtype: str                # "fp16" or "bf16": storage type of K/V (latent) and q
    k_bits: int = 4
    v_bits: int = 2
    norm_iters: int = 2
    rope_dim: int = 0         # > 0 only for the MLA latent cache
    var_lengths: bool = False  # lengths ~ U{min_context..context}
    min_context: int = 0
    encode_chunk: int = 0     # tokens encoded inside the timed step (0: one tile)
    seed: int = 0

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    "toy": Workload("toy", 1, 4, 1, 128, 1024, 128, 16, "fp16", seed=1001),
    "dense32b": Workload("dense32b", 32, 64, 8, 128, 16384, 128, 16, "fp16", seed=1002),
    "g64": Workload("g64", 32, 64, 8, 128, 32768, 64, 16, "fp16", var_lengths=True,
                    min_context=2048, seed=1003),
    "hybrid": Workload("hybrid", 8, 24, 4, 256, 65536, 128, 16, "bf16", encode_chunk=4096,
                       seed=1004),
    "mla": Workload("mla", 64, 128, 1, 512, 8192, 128, 16, "bf16", rope_dim=64, seed=1005),
}

TORCH_DTYPE = {"fp16": torch.float16, "bf16": torch.bfloat16}

# Student-t draws are clipped to this magnitude so that 10 x t(3) stays finite
# in fp16 (max 65504); the probability of reaching it is below 1e-8 per draw.
T3_CLIP = 1000.0


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _student_t3(shape, g, device) -> torch.Tensor:
    z = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    chi2 = torch.randn((3,) + tuple(shape), generator=g, device=device,
                       dtype=torch.float32).square_().sum(0)
    return (z / torch.sqrt(chi2 / 3.0)).clamp_(-T3_CLIP, T3_CLIP)


@dataclasses.dataclass
class DenseCase:
    """Inputs of one dense (GQA) workload.

    k, v        [B, Hkv, L, D] storage dtype, every token of every sequence
                (positions >= seq_lens[b] are unused)
    q           [B, Hq, D] storage dtype, one decode query per sequence
    seq_lens    [B] int32
    block_table [B, max_pages] int32, logical page -> physical page, -1 unused
    num_pages   physical pages in the cache
    """
    wl: Workload
    k: torch.Tensor
    v: torch.Tensor
    q: torch.Tensor
    seq_lens: torch.Tensor
    block_table: torch.Tensor
    num_pages: int


@dataclasses.dataclass
class LatentCase:
    """Inputs of the MLA latent workload.

    latent   [B, L, Dl] bf16      rope    [B, L, R] fp16
    q_latent [B, H, Dl] bf16      q_rope  [B, H, R] bf16
    """
    wl: Workload
    latent: torch.Tensor
    rope: torch.Tensor
    q_latent: torch.Tensor
    q_rope: torch.Tensor
    seq_lens: torch.Tensor
    block_table: torch.Tensor
    num_pages: int


def _seq_lens(wl: Workload, g, device) -> torch.Tensor:
    if not wl.var_lengths:
        return torch.full((wl.num_seqs,), wl.context, dtype=torch.int32, device=device)
    return torch.randint(wl.min_context, wl.context + 1, (wl.num_seqs,), generator=g,
                         device=device, dtype=torch.int64).to(torch.int32)


def _block_table(wl: Workload, seq_lens: torch.Tensor, g, device):
    """Random physical placement of every committed page (a random permutation
    of all physical pages, handed out sequence by sequence)."""
    P, N = wl.page_tokens, wl.tile_tokens
    lens = seq_lens.to("cpu").tolist()
    pages_per_seq = [((L // N) * N) // P for L in lens]
    max_pages = max(1, (wl.context // N) * N // P)
    num_pages = max(1, sum(pages_per_seq))
    perm = torch.randperm(num_pages, generator=g, device=device).to(torch.int32)
    bt = torch.full((wl.num_seqs, max_pages), -1, dtype=torch.int32, device=device)
    off = 0
    for b, n in enumerate(pages_per_seq):
        bt[b, :n] = perm[off:off + n]
        off += n
    return bt, num_pages


def make_dense(wl: Workload, device="cpu", seed: Optional[int] = None) -> DenseCase:
    g = _gen(device, wl.seed if seed is None else seed)
    B, H, L, D = wl.num_seqs, wl.num_kv_heads, wl.context, wl.head_dim
    dt = TORCH_DTYPE[wl.dtype]
    seq_lens = _seq_lens(wl, g, device)
    out = []
    for _ in range(2):  # K then V
        x = torch.randn((B, H, L, D), generator=g, device=device, dtype=torch.float32)
        if wl.name == "toy":
            for ch in (7, 31, 64, 100):
                x[..., ch] *= 20.0
        elif wl.name in ("dense32b", "g64"):
            mask = torch.rand((H, D), generator=g, device=device) < 0.01
            idx = mask.nonzero()
            if idx.numel():
                t = _student_t3((B, idx.shape[0], L), g, device) * 10.0
                x[:, idx[:, 0], :, idx[:, 1]] = t.permute(1, 0, 2)
        elif wl.name == "hybrid":
            scale = torch.exp(torch.randn((H, D), generator=g, device=device))
            x *= scale[None, :, None, :]
        out.append(x.to(dt))
        del x
    q = torch.randn((B, wl.num_q_heads, D), generator=g, device=device).to(dt)
    bt, num_pages = _block_table(wl, seq_lens, g, device)
    return DenseCase(wl, out[0], out[1], q, seq_lens, bt, num_pages)


def verify_queries(wl: Workload, num_queries: int, device="cpu", seed: Optional[int] = None) -> torch.Tensor:
    """Query rows of the tokens under speculative verification: [B, Q, Hq, D]
    N(0,1) in the workload's dtype."""
    g = _gen(device, (wl.seed if seed is None else seed) + 104729)
    return torch.randn((wl.num_seqs, num_queries, wl.num_q_heads, wl.head_dim), generator=g,
                       device=device).to(TORCH_DTYPE[wl.dtype])


def make_latent(wl: Workload, device="cpu", seed: Optional[int] = None) -> LatentCase:
    g = _gen(device, wl.seed if seed is None else seed)
    B, L, Dl, R = wl.num_seqs, wl.context, wl.head_dim, wl.rope_dim
    seq_lens = _seq_lens(wl, g, device)
    lat = torch.randn((B, L, Dl), generator=g, device=device)
    mask = torch.rand((Dl,), generator=g, device=device) < 0.02
    lat[..., mask] *= 15.0
    latent = lat.to(torch.bfloat16)
    del lat
    rope = torch.randn((B, L, R), generator=g, device=device).to(torch.float16)
    q_latent = torch.randn((B, wl.num_q_heads, Dl), generator=g, device=device).to(torch.bfloat16)
    q_rope = torch.randn((B, wl.num_q_heads, R), generator=g, device=device).to(torch.bfloat16)
    bt, num_pages = _block_table(wl, seq_lens, g, device)
    return LatentCase(wl, latent, rope, q_latent, q_rope, seq_lens, bt, num_pages)


def small(name: str, **kw) -> Workload:
    """A reduced copy of a named workload, for cases the oracle finishes fast."""
    return WORKLOADS[name].with_(**kw)


def default_sm_scale(wl: Workload) -> float:
    return 1.0 / math.sqrt(wl.head_dim + wl.rope_dim)
