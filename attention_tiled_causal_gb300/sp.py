"""Sequence parallelism around the attention kernels, as host code over
torch.distributed (any backend with all_to_all_single and isend/irecv: NCCL
between GPUs, gloo between CPU processes).

Device tensors exchanged over a gloo group (which moves host tensors only) go
through host memory; over NCCL they move device to device.

Two ways of spreading one long sequence over P ranks:

  * Ulysses ("Ulysses sequence parallelism for inference", sections 2.1-2.2):
    every rank holds a slice of the tokens with all heads, [T/P, H, d].  One
    all-to-all re-lays Q, K and V out as the full sequence with H/P heads,
    [T, H/P, d]; each rank runs attention for its heads (the head-range call of
    the kernels is exactly this computation); a second all-to-all brings the
    output back to [T/P, H, d].  GQA stays whole: rank r gets query heads
    [r*Hq/P, (r+1)*Hq/P) and KV heads [r*Hkv/P, (r+1)*Hkv/P), which are the KV
    heads of those query heads when Hkv is a multiple of P.
  * Ring context parallelism (SGLang partitioning page, section 3.5): every
    rank keeps its query shard; the key/value shards travel round the ring of
    ranks, each rank sending its current shard to the next rank while it
    computes against it and receiving the previous rank's; after P steps every
    query has met every key, and the P partial results are combined by the
    log-sum-exp merge.  Shards are contiguous blocks, round-robin stripes
    (token % P) or zigzag blocks (block r and block 2P-1-r of 2P), the last two
    balancing the causal triangle between ranks.

Positions are absolute throughout (Ulysses page, section 5.3): RoPE is applied
before the exchange at each token's own position, and the causal mask of every
partial compares absolute positions, so shards with gaps between their
positions need nothing special.

The per-rank computations are callables.  The defaults run the library's CUDA
kernels (attn_prefill with fp32 partial output, attn_lse_merge); any callable
with the same signature can stand in.
"""
from __future__ import annotations

from typing import Callable, Optional, Sequence, Tuple

import numpy as np
import torch
import torch.distributed as dist

from . import _binding as _b

Tensor = torch.Tensor
AttnFn = Callable[[Tensor, Tensor, Tensor, Tensor], Tuple[Tensor, Tensor]]
PartialFn = Callable[[Tensor, Tensor, Tensor, Tensor, Tensor], Tuple[Tensor, Tensor]]
MergeFn = Callable[[Tensor, Tensor], Tuple[Tensor, Tensor]]


# ------------------------------------------------------------------ partitions

def shard_rows(seq_len: int, world: int, rank: int, kind: str = "contiguous") -> np.ndarray:
    """Rows of one sequence that rank `rank` of `world` holds (SGLang page,
    section 3.5): "contiguous" blocks of seq_len/world rows; "striped", rows
    with row % world == rank (round-robin split); "zigzag", blocks rank and
    2*world-1-rank of 2*world equal blocks (in-sequence split).  Sorted."""
    if not 0 <= rank < world:
        raise ValueError("rank out of range")
    if kind == "contiguous":
        if seq_len % world:
            raise ValueError("contiguous shards need seq_len % world == 0")
        c = seq_len // world
        return np.arange(rank * c, (rank + 1) * c, dtype=np.int64)
    if kind == "striped":
        if seq_len % world:
            raise ValueError("striped shards need seq_len % world == 0")
        return np.arange(rank, seq_len, world, dtype=np.int64)
    if kind == "zigzag":
        if seq_len % (2 * world):
            raise ValueError("zigzag shards need seq_len % (2 * world) == 0")
        c = seq_len // (2 * world)
        lo, hi = rank, 2 * world - 1 - rank
        return np.concatenate([np.arange(lo * c, (lo + 1) * c), np.arange(hi * c, (hi + 1) * c)]).astype(np.int64)
    raise ValueError(f"unknown shard kind {kind!r}")


# ------------------------------------------------------------------ Ulysses exchange

def _world(group) -> Tuple[int, int]:
    if not dist.is_available() or not dist.is_initialized():
        return 1, 0
    return dist.get_world_size(group), dist.get_rank(group)


def _host_staged(group, t: Tensor) -> bool:
    """gloo moves host tensors only: device tensors go through host memory."""
    return t.is_cuda and dist.get_backend(group) == "gloo"


def _all_to_all(recv: Tensor, send: Tensor, out_splits, in_splits, group) -> None:
    if _host_staged(group, send):
        rh = torch.empty(recv.shape, dtype=recv.dtype)
        dist.all_to_all_single(rh, send.cpu(), output_split_sizes=out_splits, input_split_sizes=in_splits,
                               group=group)
        recv.copy_(rh)
    else:
        dist.all_to_all_single(recv, send, output_split_sizes=out_splits, input_split_sizes=in_splits, group=group)


def _all_gather(out: Tensor, t: Tensor, group) -> None:
    if _host_staged(group, t):
        oh = torch.empty(out.shape, dtype=out.dtype)
        dist.all_gather_into_tensor(oh, t.cpu(), group=group)
        out.copy_(oh)
    else:
        dist.all_gather_into_tensor(out, t, group=group)


def _counts(n_local: int, group, device) -> list:
    """Every rank's local token count, in rank order."""
    world, _ = _world(group)
    if world == 1:
        return [n_local]
    out = torch.zeros(world, dtype=torch.int64, device=device)
    _all_gather(out, torch.tensor([n_local], dtype=torch.int64, device=device), group)
    return [int(c) for c in out.cpu()]


def seq_to_heads(x: Tensor, group=None, counts: Optional[Sequence[int]] = None) -> Tensor:
    """[T_local, H, ...] on every rank (its tokens, all heads) -> [sum(T_r), H/P, ...]:
    every rank's tokens, in rank order, for this rank's H/P heads (heads
    [rank*H/P, (rank+1)*H/P)).  The first all-to-all of the Ulysses page,
    section 2.2."""
    world, _ = _world(group)
    if world == 1:
        return x
    T, H = x.shape[0], x.shape[1]
    if H % world:
        raise ValueError(f"{H} heads do not split over {world} ranks")
    rest = tuple(x.shape[2:])
    hp = H // world
    counts = list(counts) if counts is not None else _counts(T, group, x.device)
    # per destination rank r: this rank's tokens for heads [r*hp, (r+1)*hp), contiguous
    send = x.reshape(T, world, hp, *rest).transpose(0, 1).contiguous().reshape(world * T, hp, *rest)
    recv = torch.empty((sum(counts), hp) + rest, dtype=x.dtype, device=x.device)
    _all_to_all(recv, send, counts, [T] * world, group)
    return recv


def heads_to_seq(y: Tensor, counts: Sequence[int], group=None) -> Tensor:
    """The inverse of seq_to_heads: [sum(T_r), H/P, ...] (every rank's tokens in
    rank order, this rank's heads) -> [T_local, H, ...] (this rank's tokens, all
    heads).  `counts` are the ranks' local token counts.  The second all-to-all
    of the Ulysses page, section 2.2."""
    world, rank = _world(group)
    if world == 1:
        return y
    hp = y.shape[1]
    rest = tuple(y.shape[2:])
    T = counts[rank]
    recv = torch.empty((world * T, hp) + rest, dtype=y.dtype, device=y.device)
    _all_to_all(recv, y.contiguous(), [T] * world, list(counts), group)
    # recv block r: this rank's tokens for rank r's heads
    return recv.reshape(world, T, hp, *rest).transpose(0, 1).reshape(T, world * hp, *rest)


def gather_positions(pos: Tensor, counts: Sequence[int], group=None) -> Tensor:
    """Every rank's absolute positions, concatenated in rank order."""
    world, _ = _world(group)
    if world == 1:
        return pos
    n = max(counts)
    pad = torch.zeros(n, dtype=pos.dtype, device=pos.device)
    pad[:pos.numel()] = pos
    allp = torch.zeros(world * n, dtype=pos.dtype, device=pos.device)
    _all_gather(allp, pad, group)
    return torch.cat([allp[r * n:r * n + c] for r, c in enumerate(counts)])


def ulysses_attention(q: Tensor, k: Tensor, v: Tensor, pos: Tensor, attn: Optional[AttnFn] = None,
                      group=None) -> Tuple[Tensor, Tensor]:
    """Attention over the whole sequence for tokens spread over the ranks as
    [T_r, H, d] slices (rank order = sequence order, positions non-decreasing):
    q [T_local, Hq, d] and k, v [T_local, Hkv, d], already rotated at their
    absolute positions `pos` [T_local].  Returns (out [T_local, Hq, d],
    lse [T_local, Hq]) for this rank's tokens.  `attn(q, k, v, pos)` computes
    causal attention of one full sequence for the heads it is given (default:
    the tensor-core kernel, kernel_attention)."""
    world, _ = _world(group)
    Hq, Hkv = q.shape[1], k.shape[1]
    if Hq % world or Hkv % world:
        raise ValueError(f"Ulysses needs the query ({Hq}) and KV ({Hkv}) head counts divisible by {world} ranks")
    attn = attn or kernel_attention
    counts = _counts(q.shape[0], group, q.device)
    pos_full = gather_positions(pos, counts, group)
    qh, kh, vh = (seq_to_heads(t, group, counts) for t in (q, k, v))
    out_h, lse_h = attn(qh, kh, vh, pos_full)
    return heads_to_seq(out_h, counts, group), heads_to_seq(lse_h, counts, group)


# ------------------------------------------------------------------ ring exchange

def ring_attention(q: Tensor, k: Tensor, v: Tensor, q_pos: Tensor, k_pos: Tensor,
                   partial: Optional[PartialFn] = None, merge: Optional[MergeFn] = None,
                   group=None) -> Tuple[Tensor, Tensor]:
    """Ring context parallelism (SGLang page, section 3.5): this rank's queries
    q [Tq, Hq, d] at positions q_pos against every rank's keys and values.  Each
    step computes the partial result of the local queries against the K/V shard
    in hand while that shard goes to rank+1 and the next one arrives from
    rank-1 (both transfers posted before the compute and waited after it); after
    P steps the partials are merged by log-sum-exp.  Every rank's k, v [Tk, Hkv,
    d] and k_pos [Tk] must have the same shapes.  Returns (out, lse) of the
    local queries; partials are fp32, so out is fp32."""
    world, rank = _world(group)
    partial = partial or kernel_partial
    merge = merge or kernel_merge
    cur = [k.contiguous(), v.contiguous(), k_pos.contiguous()]
    nxt = [torch.empty_like(t) for t in cur] if world > 1 else None
    staged = world > 1 and _host_staged(group, k)
    outs, lses = [], []
    for step in range(world):
        reqs = []
        if step < world - 1:
            dst, src = (rank + 1) % world, (rank - 1) % world
            # through host buffers when the backend moves host tensors only
            send = [t.cpu() for t in cur] if staged else cur
            recv = [torch.empty(t.shape, dtype=t.dtype) for t in nxt] if staged else nxt
            ops = [dist.P2POp(dist.irecv, t, src, group) for t in recv] + \
                  [dist.P2POp(dist.isend, t, dst, group) for t in send]
            reqs = dist.batch_isend_irecv(ops)
        o, l = partial(q, cur[0], cur[1], q_pos, cur[2])
        outs.append(o)
        lses.append(l)
        for r in reqs:
            r.wait()
        if step < world - 1:
            if staged:
                for d, h in zip(nxt, recv):
                    d.copy_(h)
            cur, nxt = nxt, cur
    return merge(torch.stack(outs), torch.stack(lses))


# ------------------------------------------------------------------ kernel callables

def _single_seq(n: int, device) -> Tensor:
    return torch.tensor([0, n], dtype=torch.int32, device=device)


def kernel_attention(q: Tensor, k: Tensor, v: Tensor, pos: Tensor) -> Tuple[Tensor, Tensor]:
    """Causal attention of one sequence on the library's kernels: q [T, Hq, d],
    k, v [T, Hkv, d] (rotated), pos [T] int32 non-decreasing."""
    cu = _single_seq(q.shape[0], q.device)
    return _b.prefill(q.contiguous(), k.contiguous(), v.contiguous(), cu, pos, q.shape[0], cu_k=cu, k_pos=pos)


def kernel_partial(q: Tensor, k: Tensor, v: Tensor, q_pos: Tensor, k_pos: Tensor) -> Tuple[Tensor, Tensor]:
    """One ring step on the library's kernels: causal attention of the queries
    against one key shard (positions with gaps allowed), fp32 output for the
    merge; rows that see no key of the shard get O = 0, LSE = -inf."""
    cu_q = _single_seq(q.shape[0], q.device)
    cu_k = _single_seq(k.shape[0], k.device)
    return _b.prefill(q, k, v, cu_q, q_pos, q.shape[0], out_dtype=torch.float32, cu_k=cu_k, k_pos=k_pos)


def kernel_merge(part_out: Tensor, part_lse: Tensor) -> Tuple[Tensor, Tensor]:
    """The log-sum-exp merge of stacked partials [P, T, H, d] / [P, T, H] on the
    library's kernel (fp32 out)."""
    out = torch.empty(part_out.shape[1:], dtype=torch.float32, device=part_out.device)
    lse = torch.empty(part_lse.shape[1:], dtype=torch.float32, device=part_lse.device)
    _b.attn_lse_merge(part_out, part_lse, out, lse)
    return out, lse
