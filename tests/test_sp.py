"""The sequence-parallel host code (attention_tiled_causal_gb300.sp) as gloo
ranks on the CPU: the partitions of the SGLang page, section 3.5, the Ulysses
re-layout of the Ulysses page, section 2.2 (exact, integer-coded values), and
ring / Ulysses attention with the fp64 oracle standing in for the per-rank
kernels, compared with the oracle's unsplit result."""
import json
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from attention_tiled_causal_gb300 import sp
import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "sp_partitions.json")


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _spawn(target, world, *args):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=target, args=(r, world, port, q) + args) for r in range(world)]
    for p in procs:
        p.start()
    got = {}
    for _ in range(world):
        r, payload = q.get(timeout=300)
        got[r] = payload
    for p in procs:
        p.join(60)
        assert p.exitcode == 0
    return got


def _init(rank, world, port):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)


# ------------------------------------------------------------------ partitions

def test_shard_rows_follow_the_pages_examples():
    g = json.load(open(GOLDEN))
    for r, want in enumerate(g["striped_16_over_4"]):
        assert sp.shard_rows(16, 4, r, "striped").tolist() == want
    order = g["zigzag_block_order_8"]          # blocks as laid out rank by rank, two per rank
    for r in range(4):
        blocks = sorted(order[2 * r:2 * r + 2])
        assert sp.shard_rows(16, 4, r, "zigzag").tolist() == [b * 2 + i for b in blocks for i in range(2)]
    for kind in ("contiguous", "striped", "zigzag"):
        rows = np.concatenate([sp.shard_rows(48, 3, r, kind) for r in range(3)])
        assert sorted(rows.tolist()) == list(range(48))
        assert all((np.diff(sp.shard_rows(48, 3, r, kind)) > 0).all() for r in range(3))
    with pytest.raises(ValueError):
        sp.shard_rows(10, 3, 0, "zigzag")


# ------------------------------------------------------------------ Ulysses re-layout

def _code(T, H, d):
    """Integer-coded values: token t, head h, element i -> t*10000 + h*100 + i."""
    t = np.arange(T)[:, None, None] * 10000.0
    h = np.arange(H)[None, :, None] * 100.0
    i = np.arange(d)[None, None, :]
    return torch.from_numpy(t + h + i)


def _relayout_rank(rank, world, port, q, T, H, d):
    _init(rank, world, port)
    full = _code(T, H, d)
    n = T // world
    local = full[rank * n:(rank + 1) * n].clone()
    heads = sp.seq_to_heads(local)
    back = sp.heads_to_seq(heads, [n] * world)
    q.put((rank, (heads.numpy(), back.numpy())))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 4])
def test_ulysses_relayout_is_exact(world):
    """[T/P, H, d] -> [T, H/P, d] and back, bit for bit.  At P = 4 this is the
    page's own example: 4 segments of 16 tokens, 8 heads, rank r ends up with
    heads 2r and 2r+1 of all 64 tokens."""
    g = json.load(open(GOLDEN))["ulysses_sp4"]
    T, H, d = g["tokens"], g["heads"], 16
    got = _spawn(_relayout_rank, world, T, H, d)
    full = _code(T, H, d).numpy()
    hp = H // world
    for r in range(world):
        heads, back = got[r]
        assert np.array_equal(heads, full[:, r * hp:(r + 1) * hp])
        assert np.array_equal(back, full[r * (T // world):(r + 1) * (T // world)])
        if world == 4:
            assert list(range(r * hp, (r + 1) * hp)) == g["heads_of_rank"][r]


# ------------------------------------------------------------------ attention across ranks

def _inputs(T, hq, hkv, d, seed):
    q = synth.randn((T, hq, d), seed, 0.7071, torch.float32)
    k = synth.randn((T, hkv, d), seed + 1, 0.7071, torch.float32)
    v = synth.randn((T, hkv, d), seed + 2, 0.7071, torch.float32)
    pos = np.arange(T, dtype=np.int32) + 3
    qr = oracle.rope(synth.as_f64(q), pos)
    kr = oracle.rope(synth.as_f64(k), pos)
    return qr, kr, synth.as_f64(v), pos


def _oracle_full(q, k, v, pos):
    T = q.shape[0]
    p = pos.numpy()
    o, l = oracle.attention(q.numpy(), np.zeros(T, np.int32), p, k.numpy(), v.numpy(), [0, T], p,
                            q.shape[2] ** -0.5)
    return torch.from_numpy(o), torch.from_numpy(l)


def _oracle_partial(q, k, v, q_pos, k_pos):
    o, l = oracle.attention(q.numpy(), np.zeros(q.shape[0], np.int32), q_pos.numpy(), k.numpy(), v.numpy(),
                            [0, k.shape[0]], k_pos.numpy(), q.shape[2] ** -0.5)
    return torch.from_numpy(o), torch.from_numpy(l)


def _oracle_merge(po, pl):
    o, l = oracle.lse_merge(po.numpy(), pl.numpy())
    return torch.from_numpy(o), torch.from_numpy(l)


def _ulysses_rank(rank, world, port, q_out, T, hq, hkv, d):
    _init(rank, world, port)
    qr, kr, v, pos = _inputs(T, hq, hkv, d, 1300)
    n = T // world
    sl = slice(rank * n, (rank + 1) * n)
    out, lse = sp.ulysses_attention(torch.from_numpy(qr[sl]), torch.from_numpy(kr[sl]), torch.from_numpy(v[sl]),
                                    torch.from_numpy(pos[sl]), attn=_oracle_full)
    q_out.put((rank, (out.numpy(), lse.numpy())))
    dist.barrier()
    dist.destroy_process_group()


def test_ulysses_attention_equals_all_heads_oracle():
    """Two ranks, 64 tokens, 8/2 heads: each rank attends the full sequence for
    its heads after the all-to-all; after the inverse all-to-all its tokens'
    outputs equal the oracle's all-heads result bit for bit (the oracle's heads
    are independent computations)."""
    T, hq, hkv, d, world = 64, 8, 2, 64, 2
    got = _spawn(_ulysses_rank, world, T, hq, hkv, d)
    qr, kr, v, pos = _inputs(T, hq, hkv, d, 1300)
    wo, wl = oracle.attention(qr, np.zeros(T, np.int32), pos, kr, v, [0, T], pos, d ** -0.5)
    n = T // world
    for r in range(world):
        o, l = got[r]
        assert np.array_equal(o, wo[r * n:(r + 1) * n]) and np.array_equal(l, wl[r * n:(r + 1) * n])


def _ring_rank(rank, world, port, q_out, T, hq, hkv, d, kind):
    _init(rank, world, port)
    qr, kr, v, pos = _inputs(T, hq, hkv, d, 1310)
    rows = sp.shard_rows(T, world, rank, kind)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a))
    out, lse = sp.ring_attention(t(qr[rows]), t(kr[rows]), t(v[rows]), t(pos[rows]), t(pos[rows]),
                                 partial=_oracle_partial, merge=_oracle_merge)
    q_out.put((rank, (rows, out.numpy(), lse.numpy())))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("kind,world", [("contiguous", 2), ("striped", 2), ("zigzag", 2), ("zigzag", 3)])
def test_ring_attention_equals_unsplit_oracle(kind, world):
    """Ring context parallelism: each rank's queries against every rank's key
    shard as the shards travel round the ring, merged by log-sum-exp, equal the
    oracle's unsplit causal attention for those queries (fp64, to 1e-12)."""
    T, hq, hkv, d = 96 if world == 3 else 64, 8, 2, 64
    got = _spawn(_ring_rank, world, T, hq, hkv, d, kind)
    qr, kr, v, pos = _inputs(T, hq, hkv, d, 1310)
    wo, wl = oracle.attention(qr, np.zeros(T, np.int32), pos, kr, v, [0, T], pos, d ** -0.5)
    seen = []
    for r in range(world):
        rows, o, l = got[r]
        assert np.abs(o - wo[rows]).max() < 1e-12
        assert np.abs(l - wl[rows]).max() < 1e-12
        seen += rows.tolist()
    assert sorted(seen) == list(range(T))
