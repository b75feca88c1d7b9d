"""Seeded synthetic inputs shared by the CUDA path's tests, the oracle's tests and the bench.

This module only draws numbers and lays out index tables.  It holds none of the
attention arithmetic (no RoPE, no softmax, no merge): both sides of every parity
check receive the same bits from here and compute independently.

Workloads follow the shapes the pages discuss:
  * causal GQA with 64 query heads sharing 8 KV heads, head_dim 128 ("Ulysses
    sequence parallelism for inference", sections 3.2 and 2.2);
  * 8K to 128K token contexts (same page, section 4.1; "Flash Attention and
    distributed parallelism", section 18.2 uses N = 8K);
  * chunked prefill over a paged cache (SGLang partitioning page, section 2.2);
  * split-KV decode over a head-major paged cache (Ulysses page, section 2.3).
Values are N(0, 1) or N(0, 1)/sqrt(2) as the workload table states; every
random draw comes from a torch CPU generator seeded per tensor.
"""
from __future__ import annotations

import math
from dataclasses import dataclass
from typing import Optional

import numpy as np
import torch

PAGE = 64  # tokens per KV-cache page

_CHUNK = 1 << 26  # draw in slices so the fp32 temporaries stay small


def randn(shape, seed: int, std: float = 1.0, dtype=torch.bfloat16, device="cpu") -> torch.Tensor:
    """N(0, std^2) samples of `shape`, drawn in fp32 and rounded once to `dtype`.

    The stream of numbers depends on (seed, shape, device): a CPU draw and a
    CUDA draw with the same seed differ, but each is reproducible.  Large
    workloads are drawn on the GPU and copied back for whatever part the CPU
    checks need."""
    n = int(np.prod(shape)) if len(shape) else 1
    dev = torch.device(device)
    out = torch.empty(n, dtype=dtype, device=dev)
    g = torch.Generator(device=dev).manual_seed(int(seed))
    for s in range(0, n, _CHUNK):
        e = min(n, s + _CHUNK)
        x = torch.randn(e - s, generator=g, dtype=torch.float32, device=dev)
        if std != 1.0:
            x.mul_(std)
        out[s:e] = x.to(dtype)
    return out.view(*shape)


def randint8(shape, seed: int, device="cpu") -> torch.Tensor:
    """Uniform integers in [-127, 127] as int8 (the symmetric code range of an
    INT8 cache), seeded like `randn`."""
    n = int(np.prod(shape)) if len(shape) else 1
    dev = torch.device(device)
    out = torch.empty(n, dtype=torch.int8, device=dev)
    g = torch.Generator(device=dev).manual_seed(int(seed))
    for s in range(0, n, _CHUNK):
        e = min(n, s + _CHUNK)
        out[s:e] = torch.randint(-127, 128, (e - s,), generator=g, dtype=torch.int16, device=dev).to(torch.int8)
    return out.view(*shape)


def uniform(shape, seed: int, lo: float, hi: float, device="cpu") -> torch.Tensor:
    """U[lo, hi) fp32 samples of `shape`, seeded like `randn`."""
    dev = torch.device(device)
    g = torch.Generator(device=dev).manual_seed(int(seed))
    return torch.rand(tuple(shape), generator=g, dtype=torch.float32, device=dev).mul_(hi - lo).add_(lo)


def as_f64(t: torch.Tensor) -> np.ndarray:
    """Exact fp64 copy of a bf16/fp32 tensor (every bf16/fp32 value is an fp64 value)."""
    return t.to(torch.float64).numpy()


def cu_seqlens(lens) -> np.ndarray:
    c = np.zeros(len(lens) + 1, dtype=np.int32)
    c[1:] = np.cumsum(lens)
    return c


def positions(lens, starts=None) -> np.ndarray:
    """Absolute token positions: sequence b covers starts[b] .. starts[b]+lens[b]-1."""
    starts = [0] * len(lens) if starts is None else starts
    return np.concatenate([np.arange(s, s + n, dtype=np.int32) for s, n in zip(starts, lens)]) \
        if len(lens) else np.zeros(0, np.int32)


def shuffled_page_table(ctx_lens, seed: int, page: int = PAGE, max_pages: Optional[int] = None):
    """Page table for a paged cache whose physical pages are a seeded permutation.

    Request b owns ceil(ctx_b/page) logical pages; all logical pages of all
    requests are laid out in order and then mapped through one Fisher-Yates
    permutation of the physical ids.  Unused table slots hold -1.
    Returns (page_table [B, max_pages] int32, num_pages).
    """
    npg = [(int(c) + page - 1) // page for c in ctx_lens]
    total = int(sum(npg))
    mp = max(npg) if max_pages is None else max_pages
    perm = np.random.default_rng(seed).permutation(total).astype(np.int32)
    table = np.full((len(ctx_lens), max(mp, 1)), -1, dtype=np.int32)
    o = 0
    for b, n in enumerate(npg):
        table[b, :n] = perm[o:o + n]
        o += n
    return table, total


def shard_rows(seq_len: int, world: int, rank: int, kind: str) -> np.ndarray:
    """Token rows that rank `rank` of `world` holds when one sequence is split
    along the sequence axis (SGLang partitioning page, section 3.5):

      contiguous  rows [rank*c, (rank+1)*c), c = seq_len / world;
      striped     rows rank, rank + world, rank + 2*world, ...;
      zigzag      the sequence cut into 2*world chunks of c = seq_len / (2*world)
                  rows; rank r holds chunks r and 2*world-1-r, so every rank
                  gets one early and one late chunk of the causal triangle.

    Rows come back sorted, so their positions stay non-decreasing."""
    if kind == "contiguous":
        c = seq_len // world
        return np.arange(rank * c, (rank + 1) * c, dtype=np.int64)
    if kind == "striped":
        return np.arange(rank, seq_len, world, dtype=np.int64)
    if kind == "zigzag":
        c = seq_len // (2 * world)
        a, b = rank, 2 * world - 1 - rank
        return np.concatenate([np.arange(a * c, (a + 1) * c), np.arange(b * c, (b + 1) * c)]).astype(np.int64)
    raise ValueError(f"unknown partition {kind!r}")


def sample_rows(seq_len: int, n: int, seed: int) -> np.ndarray:
    """`n` distinct sorted rows of [0, seq_len), always holding the first and last
    row and the rows on either side of the first few 128-row tile edges."""
    must = {0, seq_len - 1}
    for e in (127, 128, 255, 256, 383, 384):
        if e < seq_len:
            must.add(e)
    rng = np.random.default_rng(seed)
    rest = rng.choice(seq_len, size=min(seq_len, n + len(must)), replace=False)
    rows = list(must)
    for r in rest:
        if len(rows) >= n:
            break
        if int(r) not in must:
            rows.append(int(r))
    return np.array(sorted(rows[:n]), dtype=np.int64)


# --------------------------------------------------------------------------- workloads

@dataclass
class Prefill:
    """Causal GQA prefill over packed [tokens, heads, head_dim] tensors."""
    name: str
    batch: int
    seq: int
    hq: int
    hkv: int
    d: int
    dtype: torch.dtype
    std: float
    seed: int
    base: float = 10000.0
    q_start: int = 0          # absolute position of the first query token
    head_ranges: tuple = ()   # extra (h_lo, h_hi) calls the workload runs
    rows_per_head: Optional[int] = None  # oracle row sample (None = all rows)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def tokens(self) -> int:
        return self.batch * self.seq

    def flops(self, h_lo: int = 0, h_hi: Optional[int] = None) -> float:
        """4*d per visible (query, key) pair: QK^T and PV each 2*d."""
        h_hi = self.hq if h_hi is None else h_hi
        pairs = self.seq * (self.seq + 1) // 2
        return 4.0 * self.d * pairs * self.batch * (h_hi - h_lo)

    def make(self, device="cpu"):
        T = self.tokens
        q = randn((T, self.hq, self.d), self.seed * 16 + 1, self.std, self.dtype, device)
        k = randn((T, self.hkv, self.d), self.seed * 16 + 2, self.std, self.dtype, device)
        v = randn((T, self.hkv, self.d), self.seed * 16 + 3, self.std, self.dtype, device)
        lens = [self.seq] * self.batch
        pos = positions(lens, [self.q_start] * self.batch)
        cu = cu_seqlens(lens)
        return dict(q=q, k=k, v=v, pos=torch.from_numpy(pos).to(device), cu=torch.from_numpy(cu).to(device))


@dataclass
class ChunkedPaged:
    """A new chunk of `chunk` tokens per request, appended after a cached prefix of
    `prefix` tokens held in a head-major paged cache with shuffled pages."""
    name: str
    batch: int
    prefix: int
    chunk: int
    hq: int
    hkv: int
    d: int
    seed: int
    std: float = 1.0 / math.sqrt(2.0)
    base: float = 10000.0
    rows_per_head: Optional[int] = None

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    def flops(self) -> float:
        causal = self.chunk * (self.chunk + 1) // 2
        return 4.0 * self.d * self.hq * self.batch * (causal + self.chunk * self.prefix)

    def make(self, device="cpu"):
        B, P = self.batch, PAGE
        table, num_pages = shuffled_page_table([self.prefix] * B, self.seed * 16 + 9)
        kc = randn((self.hkv, num_pages, P, self.d), self.seed * 16 + 4, self.std, device=device)
        vc = randn((self.hkv, num_pages, P, self.d), self.seed * 16 + 5, self.std, device=device)
        T = B * self.chunk
        q = randn((T, self.hq, self.d), self.seed * 16 + 1, self.std, device=device)
        k = randn((T, self.hkv, self.d), self.seed * 16 + 2, self.std, device=device)
        v = randn((T, self.hkv, self.d), self.seed * 16 + 3, self.std, device=device)
        qpos = positions([self.chunk] * B, [self.prefix] * B)
        kpos_prefix = positions([self.prefix] * B)
        return dict(q=q, k=k, v=v, k_cache=kc, v_cache=vc,
                    page_table=torch.from_numpy(table).to(device), num_pages=num_pages,
                    q_pos=torch.from_numpy(qpos).to(device),
                    prefix_pos=torch.from_numpy(kpos_prefix).to(device),
                    cu_q=torch.from_numpy(cu_seqlens([self.chunk] * B)).to(device),
                    cu_prefix=torch.from_numpy(cu_seqlens([self.prefix] * B)).to(device),
                    prefix_lens=torch.full((B,), self.prefix, dtype=torch.int32).to(device))


@dataclass
class Decode:
    """One new query token per request against a head-major paged cache."""
    name: str
    batch: int
    ctx_lo: int
    ctx_hi: int
    hq: int
    hkv: int
    d: int
    splits: int
    seed: int
    q_std: float = 1.0 / math.sqrt(2.0)
    kv_std: float = 1.0
    base: float = 10000.0
    ctx_fixed: Optional[list] = None
    int8: bool = False  # INT8 cache: int8 codes + one fp32 scale per (KV head, token)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    def ctx_lens(self) -> np.ndarray:
        if self.ctx_fixed is not None:
            return np.asarray(self.ctx_fixed, dtype=np.int32)
        rng = np.random.default_rng(self.seed * 16 + 7)
        return rng.integers(self.ctx_lo, self.ctx_hi + 1, size=self.batch).astype(np.int32)

    def kv_bytes(self) -> int:
        """Cache bytes one decode step reads: K and V of every cached token of every KV
        head (bf16: 2 bytes per value; INT8: 1 byte per value + a 4-byte scale per row)."""
        per_row = self.d + 4 if self.int8 else 2 * self.d
        return int(self.ctx_lens().astype(np.int64).sum()) * self.hkv * per_row * 2

    def make(self, device="cpu"):
        ctx = self.ctx_lens()
        table, num_pages = shuffled_page_table(ctx, self.seed * 16 + 8)
        shape = (self.hkv, max(num_pages, 1), PAGE, self.d)
        q = randn((self.batch, self.hq, self.d), self.seed * 16 + 1, self.q_std, device=device)
        qpos = (ctx - 1).astype(np.int32)
        out = dict(q=q, page_table=torch.from_numpy(table).to(device), num_pages=num_pages,
                   ctx_lens=torch.from_numpy(ctx).to(device), q_pos=torch.from_numpy(qpos).to(device))
        if self.int8:
            # codes uniform in [-127, 127] (std 73.3); scales near 1/73.3 so the
            # cached values have about unit variance, like the bf16 workload
            out["k_cache"] = randint8(shape, self.seed * 16 + 4, device)
            out["v_cache"] = randint8(shape, self.seed * 16 + 5, device)
            out["k_scale"] = uniform(shape[:-1], self.seed * 16 + 10, 0.8 / 73.3, 1.2 / 73.3, device)
            out["v_scale"] = uniform(shape[:-1], self.seed * 16 + 11, 0.8 / 73.3, 1.2 / 73.3, device)
        else:
            out["k_cache"] = randn(shape, self.seed * 16 + 4, self.kv_std, device=device)
            out["v_cache"] = randn(shape, self.seed * 16 + 5, self.kv_std, device=device)
        return out


TINY = Prefill("tiny causal GQA: B1 S64 (4x16-token segments) 8/2 heads d64 fp32",
               batch=1, seq=64, hq=8, hkv=2, d=64, dtype=torch.float32, std=1.0, seed=1235)
PREFILL_8K = Prefill("causal GQA prefill: B1 S8192 64/8 heads d128 bf16",
                     batch=1, seq=8192, hq=64, hkv=8, d=128, dtype=torch.bfloat16,
                     std=1.0 / math.sqrt(2.0), seed=1236)
PREFILL_64K = Prefill("long-context causal GQA prefill: B2 S65536 64/8 heads d128 bf16",
                      batch=2, seq=65536, hq=64, hkv=8, d=128, dtype=torch.bfloat16,
                      std=1.0 / math.sqrt(2.0), seed=1237, head_ranges=((16, 32), (0, 64)),
                      rows_per_head=512)
CHUNKED = ChunkedPaged("chunked prefill: B4 x (57344 paged prefix + 8192 chunk) 64/8 heads d128",
                       batch=4, prefix=57344, chunk=8192, hq=64, hkv=8, d=128, seed=1238,
                       rows_per_head=512)
DECODE = Decode("paged decode: B32 ctx U[16384,131072] 64/8 heads d128, 16 splits",
                batch=32, ctx_lo=16384, ctx_hi=131072, hq=64, hkv=8, d=128, splits=16, seed=1239)
DECODE_INT8 = Decode("paged decode, INT8 cache: B32 ctx U[16384,131072] 64/8 heads d128, 16 splits",
                     batch=32, ctx_lo=16384, ctx_hi=131072, hq=64, hkv=8, d=128, splits=16, seed=1239, int8=True)

WORKLOADS = [TINY, PREFILL_8K, PREFILL_64K, CHUNKED, DECODE, DECODE_INT8]
