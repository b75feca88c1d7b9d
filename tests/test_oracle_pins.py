"""Pins for the fp64 CPU oracle: each test checks it against something other than
itself — a library routine, a different algorithm from the pages, a closed form,
an invariant, or a hand-worked case — so that a dropped term, a wrong sign or
index, or a transposed operand in oracle.c fails at least one of them."""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_worked.json")
_ENV = {k: getattr(math, k) for k in ("log", "exp", "cos", "sin", "sqrt", "e", "pi", "inf")}


def _ev(x):
    if isinstance(x, list):
        return [_ev(y) for y in x]
    return float(eval(str(x).replace("-inf", "-inf_"), {"__builtins__": {}},
                      dict(_ENV, inf_=math.inf)))


def _rand(shape, seed, std=1.0):
    return np.random.default_rng(seed).normal(0.0, std, size=shape)


# ------------------------------------------------------------------ bf16 rounding

def test_round_bf16_matches_torch_conversion():
    """RNE to bf16 equals torch's float32 -> bfloat16 conversion (a library routine)
    on random fp32 values, exact ties, subnormals and overflow."""
    rng = np.random.default_rng(0)
    x = np.concatenate([
        rng.normal(0, 1, 20000), rng.normal(0, 1e-3, 2000), rng.normal(0, 1e30, 2000),
        rng.uniform(-1e-38, 1e-38, 2000),
    ]).astype(np.float32)
    # exact ties: midpoints between neighbouring bf16 values are fp32 values
    b = torch.from_numpy(rng.normal(0, 1, 4000).astype(np.float32)).to(torch.bfloat16)
    lo = b.view(torch.int16).to(torch.int32)
    nxt = (lo + 1).to(torch.int16).view(torch.bfloat16)
    mid = ((b.to(torch.float64) + nxt.to(torch.float64)) / 2).to(torch.float32).numpy()
    x = np.concatenate([x, mid, np.array([3.4e38, -3.4e38, 1.0 + 2**-8, 1.0 + 3 * 2**-8],
                                         dtype=np.float32)])
    want = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    got = oracle.round_bf16(x.astype(np.float64))
    np.testing.assert_array_equal(got, want)


# ------------------------------------------------------------------ RoPE

def test_rope_position_zero_is_identity():
    x = _rand((5, 3, 16), 1)
    np.testing.assert_array_equal(oracle.rope(x, np.zeros(5, np.int32)), x)


def test_rope_d2_is_plane_rotation_by_position():
    """d = 2: theta_0 = base^0 = 1, so (1, 0) at position p becomes (cos p, sin p)."""
    p = np.array([0, 1, 2, 7, 1000, 65535], np.int32)
    x = np.zeros((len(p), 1, 2))
    x[:, 0, 0] = 1.0
    y = oracle.rope(x, p)
    np.testing.assert_allclose(y[:, 0, 0], np.cos(p), atol=1e-12)
    np.testing.assert_allclose(y[:, 0, 1], np.sin(p), atol=1e-12)


def test_rope_equals_complex_multiplication():
    """Half-split RoPE is z_i * exp(i p theta_i) with z_i = x_i + i x_{i+d/2}."""
    T, H, d, base = 9, 2, 32, 10000.0
    x = _rand((T, H, d), 2)
    p = np.array([0, 1, 5, 17, 100, 4096, 8191, 65535, 131071], np.int32)
    half = d // 2
    theta = base ** (-(2.0 * np.arange(half)) / d)
    z = (x[..., :half] + 1j * x[..., half:]) * np.exp(1j * p[:, None, None] * theta[None, None, :])
    want = np.concatenate([z.real, z.imag], axis=-1)
    np.testing.assert_allclose(oracle.rope(x, p, base), want, atol=1e-10, rtol=0)


def test_rope_preserves_pair_norms():
    x = _rand((7, 4, 64), 3)
    p = np.arange(7, dtype=np.int32) * 1000
    y = oracle.rope(x, p)
    n0 = x[..., :32] ** 2 + x[..., 32:] ** 2
    n1 = y[..., :32] ** 2 + y[..., 32:] ** 2
    np.testing.assert_allclose(n1, n0, rtol=1e-12)


def test_golden_rope():
    for c in json.load(open(GOLDEN))["rope"]:
        x = np.array(_ev(c["x"]))[None, None, :]
        y = oracle.rope(x, np.array([c["pos"]], np.int32), c["base"])
        np.testing.assert_allclose(y[0, 0], _ev(c["out"]), atol=1e-13)


# ------------------------------------------------------------------ attention

def _varlen_case(seed, lens_q, lens_k, q_start, hq, hkv, d, k_start=None):
    rng = np.random.default_rng(seed)
    B = len(lens_q)
    k_start = [0] * B if k_start is None else k_start
    q = rng.normal(0, 1, (sum(lens_q), hq, d))
    k = rng.normal(0, 1, (sum(lens_k), hkv, d))
    v = rng.normal(0, 1, (sum(lens_k), hkv, d))
    q_seq = np.concatenate([np.full(n, b, np.int32) for b, n in enumerate(lens_q)])
    q_pos = synth.positions(lens_q, q_start)
    k_pos = synth.positions(lens_k, k_start)
    cu_k = synth.cu_seqlens(lens_k)
    return q, k, v, q_seq, q_pos, k_pos, cu_k


def _torch_reference(q, k, v, q_seq, q_pos, k_pos, cu_k, scale, causal):
    """torch SDPA (float64, CPU) with an explicit visibility mask; GQA by repeating
    each KV head for its group of query heads."""
    hq, hkv = q.shape[1], k.shape[1]
    G = hq // hkv
    out = np.zeros_like(q)
    lse = np.zeros(q.shape[:2])
    for b in range(len(cu_k) - 1):
        rows = np.nonzero(q_seq == b)[0]
        kr = slice(cu_k[b], cu_k[b + 1])
        Q = torch.from_numpy(q[rows]).permute(1, 0, 2)                       # [hq, nq, d]
        K = torch.from_numpy(k[kr]).permute(1, 0, 2).repeat_interleave(G, 0)  # [hq, nk, d]
        V = torch.from_numpy(v[kr]).permute(1, 0, 2).repeat_interleave(G, 0)
        vis = torch.ones(len(rows), K.shape[1], dtype=torch.bool)
        if causal:
            vis = torch.from_numpy(k_pos[kr][None, :] <= q_pos[rows][:, None])
        O = torch.nn.functional.scaled_dot_product_attention(Q, K, V, attn_mask=vis, scale=scale)
        S = (Q @ K.transpose(1, 2)) * scale
        L = torch.logsumexp(S.masked_fill(~vis, -math.inf), dim=-1)
        out[rows] = O.permute(1, 0, 2).numpy()
        lse[rows] = L.permute(1, 0).numpy()
    return out, lse


@pytest.mark.parametrize("hq,hkv", [(4, 2), (8, 2), (6, 6), (4, 1)])
def test_attention_matches_torch_sdpa(hq, hkv):
    lens = [13, 40, 1]
    q, k, v, q_seq, q_pos, k_pos, cu_k = _varlen_case(10 + hq, lens, lens, [0, 5, 1000], hq, hkv, 8,
                                                      k_start=[0, 5, 1000])
    scale = 0.37
    o, l = oracle.attention(q, q_seq, q_pos, k, v, cu_k, k_pos, scale)
    wo, wl = _torch_reference(q, k, v, q_seq, q_pos, k_pos, cu_k, scale, True)
    np.testing.assert_allclose(o, wo, atol=1e-12, rtol=1e-10)
    np.testing.assert_allclose(l, wl, atol=1e-12, rtol=1e-10)


def test_attention_non_causal_and_chunk_offset_matches_torch():
    """Queries of a chunk at positions 20..29 against 30 keys at 0..29 (the chunked
    prefill shape), and the same without a mask."""
    q, k, v, q_seq, q_pos, k_pos, cu_k = _varlen_case(5, [10], [30], [20], 4, 2, 16)
    for causal in (True, False):
        o, l = oracle.attention(q, q_seq, q_pos, k, v, cu_k, k_pos, 0.25, causal=causal)
        wo, wl = _torch_reference(q, k, v, q_seq, q_pos, k_pos, cu_k, 0.25, causal)
        np.testing.assert_allclose(o, wo, atol=1e-12)
        np.testing.assert_allclose(l, wl, atol=1e-12)


def _online_softmax(q, k, v, q_pos, k_pos, scale, block):
    """The blockwise recurrence of the Flash Attention page, section 18.3: per K/V block,
    m_new = max(m_old, rowmax S); O <- O e^{m_old - m_new} + e^{S - m_new} V;
    l <- l e^{m_old - m_new} + sum e^{S - m_new}; finally O / l."""
    nq, hq, d = q.shape
    G = hq // k.shape[1]
    out = np.zeros_like(q)
    lse = np.zeros((nq, hq))
    for h in range(hq):
        Kh, Vh = k[:, h // G], v[:, h // G]
        for r in range(nq):
            m, l, O = -np.inf, 0.0, np.zeros(d)
            for j0 in range(0, len(Kh), block):
                Kb, Vb, pb = Kh[j0:j0 + block], Vh[j0:j0 + block], k_pos[j0:j0 + block]
                s = (Kb @ q[r, h]) * scale
                s = np.where(pb <= q_pos[r], s, -np.inf)
                if np.all(s == -np.inf):
                    continue
                m_new = max(m, s.max())
                a = math.exp(m - m_new) if m != -np.inf else 0.0
                p = np.exp(s - m_new)
                O = O * a + p @ Vb
                l = l * a + p.sum()
                m = m_new
            out[r, h] = O / l
            lse[r, h] = m + math.log(l)
    return out, lse


@pytest.mark.parametrize("block", [1, 7, 16, 64])
def test_online_softmax_recurrence_equals_three_pass(block):
    """The method's tiled recurrence gives the same result as the oracle's three
    passes, as section 18.3 of the Flash Attention page states."""
    q, k, v, q_seq, q_pos, k_pos, cu_k = _varlen_case(7, [70], [70], [0], 4, 2, 16)
    o, l = oracle.attention(q, q_seq, q_pos, k, v, cu_k, k_pos, 0.3)
    oo, ll = _online_softmax(q, k, v, q_pos, k_pos, 0.3, block)
    np.testing.assert_allclose(o, oo, atol=1e-12)
    np.testing.assert_allclose(l, ll, atol=1e-12)


def test_uniform_scores_give_causal_prefix_mean():
    """q = 0 makes every visible score 0: O_i = mean(V[0..i]), LSE_i = ln(i + 1)."""
    S, hq, hkv, d = 50, 4, 2, 8
    q = np.zeros((S, hq, d))
    k = _rand((S, hkv, d), 11)
    v = _rand((S, hkv, d), 12)
    pos = np.arange(S, dtype=np.int32)
    o, l = oracle.attention(q, np.zeros(S, np.int32), pos, k, v, [0, S], pos, 0.5)
    G = hq // hkv
    for h in range(hq):
        want = np.cumsum(v[:, h // G], axis=0) / np.arange(1, S + 1)[:, None]
        np.testing.assert_allclose(o[:, h], want, atol=1e-13)
        np.testing.assert_allclose(l[:, h], np.log(np.arange(1, S + 1)), atol=1e-13)


def test_causal_row_zero_is_v0():
    """The first row sees only key 0: O_0 = V[0] exactly, LSE_0 = scale q0.k0."""
    S, hq, hkv, d = 20, 8, 2, 16
    q, k, v = _rand((S, hq, d), 21), _rand((S, hkv, d), 22), _rand((S, hkv, d), 23)
    pos = np.arange(S, dtype=np.int32)
    o, l = oracle.attention(q, np.zeros(S, np.int32), pos, k, v, [0, S], pos, 0.25)
    for h in range(hq):
        np.testing.assert_array_equal(o[0, h], v[0, h // 4])
        assert abs(l[0, h] - 0.25 * float(q[0, h] @ k[0, h // 4])) < 1e-14


def test_head_mapping_is_consecutive_groups():
    """With K/V heads made distinguishable (head g's V is constant g), query head h
    reads KV head h // (hq / hkv)."""
    S, hq, hkv, d = 6, 8, 2, 4
    q, k = _rand((S, hq, d), 31), _rand((S, hkv, d), 32)
    v = np.zeros((S, hkv, d))
    v[:, 1] = 1.0
    pos = np.arange(S, dtype=np.int32)
    o, _ = oracle.attention(q, np.zeros(S, np.int32), pos, k, v, [0, S], pos, 0.5)
    np.testing.assert_allclose(o[:, :4], 0.0, atol=0)
    np.testing.assert_allclose(o[:, 4:], 1.0, atol=1e-14)


def test_fully_masked_row_is_zero_with_minus_inf_lse():
    q, k, v, q_seq, q_pos, k_pos, cu_k = _varlen_case(41, [3], [5], [0], 2, 1, 4, k_start=[10])
    o, l = oracle.attention(q, q_seq, q_pos, k, v, cu_k, k_pos, 1.0)
    assert np.all(o == 0.0) and np.all(l == -np.inf)


def test_rope_shift_invariance_of_attention():
    """RoPE scores depend on position differences only: adding the same offset to every
    query and key position leaves O and LSE unchanged (Ulysses page, 3.5, second check)."""
    S, hq, hkv, d = 40, 4, 2, 32
    q, k, v = _rand((S, hq, d), 51), _rand((S, hkv, d), 52), _rand((S, hkv, d), 53)
    pos = np.arange(S, dtype=np.int32)
    res = []
    for shift in (0, 1000, 57344):
        p = pos + shift
        res.append(oracle.attention(oracle.rope(q, p), np.zeros(S, np.int32), p,
                                    oracle.rope(k, p), v, [0, S], p, d ** -0.5))
    for o, l in res[1:]:
        np.testing.assert_allclose(o, res[0][0], atol=1e-11)
        np.testing.assert_allclose(l, res[0][1], atol=1e-11)


def test_head_slices_concatenate_to_full_call():
    """Ulysses page, 2.2: four shards of 16 tokens and 8 heads; after the all-to-all
    each rank computes 2 heads over all 64 tokens.  Those slices put together equal
    the all-heads result bit for bit."""
    g = json.load(open(GOLDEN))["ulysses_head_shards"]
    S = g["sp"] * g["tokens_per_shard"]
    H = g["heads"]
    q, k, v = _rand((S, H, 16), 61), _rand((S, H, 16), 62), _rand((S, H, 16), 63)
    pos = np.arange(S, dtype=np.int32)
    seq = np.zeros(S, np.int32)
    full_o, full_l = oracle.attention(q, seq, pos, k, v, [0, S], pos, 0.25)
    cat_o = np.full_like(full_o, np.nan)
    cat_l = np.full_like(full_l, np.nan)
    for heads in g["heads_of_rank"]:
        o, l = oracle.attention(q, seq, pos, k, v, [0, S], pos, 0.25, h_lo=heads[0], h_hi=heads[-1] + 1)
        cat_o[:, heads] = o[:, heads]
        cat_l[:, heads] = l[:, heads]
    np.testing.assert_array_equal(cat_o, full_o)
    np.testing.assert_array_equal(cat_l, full_l)


# ------------------------------------------------------------------ merge

def _key_partitions(n, parts):
    idx = np.arange(n)
    contiguous = np.array_split(idx, parts)
    striped = [idx[r::parts] for r in range(parts)]
    # zigzag: 2*parts blocks, part r takes blocks r and 2*parts-1-r
    blocks = np.array_split(idx, 2 * parts)
    zigzag = [np.concatenate([blocks[r], blocks[2 * parts - 1 - r]]) for r in range(parts)]
    return {"contiguous": contiguous, "striped": striped, "zigzag": zigzag}


@pytest.mark.parametrize("kind", ["contiguous", "striped", "zigzag"])
def test_merge_of_key_partitions_equals_unsplit(kind):
    """Attention over disjoint key sets, merged through the LSE, equals attention over
    all keys (the ring / striped / zigzag splits of the SGLang page, section 3.5)."""
    S, hq, hkv, d, parts = 64, 4, 2, 16, 4
    q, k, v = _rand((S, hq, d), 71), _rand((S, hkv, d), 72), _rand((S, hkv, d), 73)
    pos = np.arange(S, dtype=np.int32)
    seq = np.zeros(S, np.int32)
    full_o, full_l = oracle.attention(q, seq, pos, k, v, [0, S], pos, 0.25)
    po, pl = [], []
    for ids in _key_partitions(S, parts)[kind]:
        o, l = oracle.attention(q, seq, pos, k[ids], v[ids], [0, len(ids)], pos[ids], 0.25)
        po.append(o)
        pl.append(l)
    mo, ml = oracle.lse_merge(np.stack(po), np.stack(pl))
    np.testing.assert_allclose(mo, full_o, atol=1e-12)
    np.testing.assert_allclose(ml, full_l, atol=1e-12)


def test_golden_merge():
    for c in json.load(open(GOLDEN))["merge"]:
        o = np.array(_ev(c["o"]))[:, None, :]
        l = np.array(_ev(c["lse"]))[:, None]
        mo, ml = oracle.lse_merge(o, l)
        np.testing.assert_allclose(mo[0], _ev(c["out"]), atol=1e-14)
        assert abs(ml[0] - _ev(c["out_lse"])) < 1e-14


def test_merge_all_empty_parts():
    o = np.ones((3, 2, 4))
    l = np.full((3, 2), -np.inf)
    mo, ml = oracle.lse_merge(o, l)
    assert np.all(mo == 0.0) and np.all(ml == -np.inf)


def test_golden_attention():
    for c in json.load(open(GOLDEN))["attention"]:
        q = np.array(_ev(c["q"]))[:, None, :]
        k = np.array(_ev(c["k"]))[:, None, :]
        v = np.array(_ev(c["v"]))[:, None, :]
        qp = np.array(c["q_pos"], np.int32)
        kp = np.array(c["k_pos"], np.int32)
        qr, kr = oracle.rope(q, qp, c["base"]), oracle.rope(k, kp, c["base"])
        o, l = oracle.attention(qr, np.zeros(len(qp), np.int32), qp, kr, v, [0, len(kp)], kp,
                                c["scale"])
        np.testing.assert_allclose(o[:, 0], _ev(c["out"]), atol=1e-14)
        np.testing.assert_allclose(l[:, 0], _ev(c["lse"]), atol=1e-14)


# ------------------------------------------------------------------ paged decode

def _decode_case(seed, ctx, hq=8, hkv=2, d=16, page=4):
    table, num_pages = synth.shuffled_page_table(ctx, seed, page=page)
    rng = np.random.default_rng(seed)
    kc = rng.normal(0, 1, (hkv, num_pages, page, d))
    vc = rng.normal(0, 1, (hkv, num_pages, page, d))
    q = rng.normal(0, 1, (len(ctx), hq, d))
    return q, kc, vc, table, num_pages


def test_gather_pages_bit_exact():
    ctx = [9, 1, 16, 5]
    q, kc, vc, table, num_pages = _decode_case(81, ctx)
    for b, c in enumerate(ctx):
        for g in range(kc.shape[0]):
            want = np.stack([kc[g, table[b, j // 4], j % 4] for j in range(c)])
            np.testing.assert_array_equal(oracle.gather_pages(kc, table, num_pages, g, b, c), want)


def test_gather_rejects_bad_page_id():
    q, kc, vc, table, num_pages = _decode_case(82, [8])
    table = table.copy()
    table[0, 1] = num_pages
    with pytest.raises(ValueError):
        oracle.gather_pages(kc, table, num_pages, 0, 0, 8)


def test_decode_equals_attention_over_gathered_keys():
    """Decode at position ctx-1 over the paged cache equals causal attention of that
    one query over the keys gathered (here by numpy indexing) in logical order."""
    ctx = [7, 12, 1, 30]
    q, kc, vc, table, num_pages = _decode_case(83, ctx)
    o, l = oracle.decode_paged(q, kc, vc, table, ctx, num_pages, 0.25)
    hkv = kc.shape[0]
    for b, c in enumerate(ctx):
        j = np.arange(c)
        K = kc[:, table[b, j // 4], j % 4].transpose(1, 0, 2)  # [c, hkv, d]
        V = vc[:, table[b, j // 4], j % 4].transpose(1, 0, 2)
        wo, wl = oracle.attention(q[b:b + 1], np.zeros(1, np.int32), np.array([c - 1], np.int32),
                                  K, V, [0, c], j.astype(np.int32), 0.25)
        np.testing.assert_array_equal(o[b], wo[0])
        np.testing.assert_array_equal(l[b], wl[0])
        wo2, wl2 = _torch_reference(q[b:b + 1], K, V, np.zeros(1, np.int32),
                                    np.array([c - 1], np.int32), j.astype(np.int32), [0, c], 0.25, True)
        np.testing.assert_allclose(o[b], wo2[0], atol=1e-12)


def test_decode_invariant_under_page_permutation_and_request_order():
    """Moving pages to other physical slots, or reordering requests, changes no output
    bit (Ulysses page, 3.5, third check: reuse of the cache with a permuted batch)."""
    ctx = [7, 12, 5, 30]
    q, kc, vc, table, num_pages = _decode_case(84, ctx)
    o, l = oracle.decode_paged(q, kc, vc, table, ctx, num_pages, 0.25)
    perm = np.random.default_rng(1).permutation(num_pages)
    inv = np.argsort(perm)
    kc2, vc2 = kc[:, perm], vc[:, perm]
    table2 = np.where(table >= 0, inv[np.maximum(table, 0)], -1).astype(np.int32)
    o2, l2 = oracle.decode_paged(q, kc2, vc2, table2, ctx, num_pages, 0.25)
    np.testing.assert_array_equal(o2, o)
    np.testing.assert_array_equal(l2, l)
    order = np.array([2, 0, 3, 1])
    o3, l3 = oracle.decode_paged(q[order], kc, vc, table[order], np.array(ctx)[order], num_pages, 0.25)
    np.testing.assert_array_equal(o3, o[order])
    np.testing.assert_array_equal(l3, l[order])


# ------------------------------------------------------------ append to the paged cache

def _append_case(seed, T=3, H=2, d=4, pages=3, page=2):
    rng = np.random.default_rng(seed)
    kn = rng.normal(0, 1, (T, H, d))
    vn = rng.normal(0, 1, (T, H, d))
    kc = np.full((H, pages, page, d), 7.0)
    vc = np.full((H, pages, page, d), -7.0)
    return kn, vn, kc, vc


def test_kv_append_places_rows_by_slot_and_skips_minus_one():
    """Hand placement, base 0 (plain copy): slot s of head h is row s of that
    head's pool; slot -1 leaves the cache alone; every other row keeps its value."""
    kn, vn, kc, vc = _append_case(90)
    k2, v2, bad = oracle.kv_append(kn, vn, None, [5, -1, 0], kc, vc, base=0.0)
    assert bad == 0
    want_k, want_v = kc.copy(), vc.copy()
    for h in range(2):
        want_k[h, 2, 1] = kn[0, h]   # slot 5 = page 2, offset 1
        want_v[h, 2, 1] = vn[0, h]
        want_k[h, 0, 0] = kn[2, h]   # slot 0 = page 0, offset 0
        want_v[h, 0, 0] = vn[2, h]
    np.testing.assert_array_equal(k2, want_k)
    np.testing.assert_array_equal(v2, want_v)


def test_kv_append_counts_and_skips_out_of_range_slots():
    kn, vn, kc, vc = _append_case(91)
    k2, v2, bad = oracle.kv_append(kn, vn, None, [6, -2, 3], kc, vc, base=0.0)
    assert bad == 2
    want_k = kc.copy()
    want_k[:, 1, 1] = kn[2]
    np.testing.assert_array_equal(k2, want_k)
    np.testing.assert_array_equal(v2[:, 1, 1], vn[2])


def test_kv_append_d2_key_is_bf16_of_plane_rotation():
    """d = 2: the stored key is the plane rotation of (x, y) by the position
    (theta_0 = 1), rounded to bf16 by torch's own conversion."""
    rng = np.random.default_rng(92)
    T = 6
    kn = rng.normal(0, 1, (T, 1, 2))
    vn = rng.normal(0, 1, (T, 1, 2))
    pos = np.array([0, 1, 5, 17, 1000, 65535], np.int32)
    kc = np.zeros((1, 2, 4, 2))
    k2, v2, bad = oracle.kv_append(kn, vn, pos, np.arange(T, dtype=np.int32), kc, kc, base=10000.0)
    assert bad == 0
    for t in range(T):
        x, y, p = kn[t, 0, 0], kn[t, 0, 1], float(pos[t])
        rot = torch.tensor([x * math.cos(p) - y * math.sin(p), y * math.cos(p) + x * math.sin(p)],
                           dtype=torch.float64).to(torch.bfloat16).double().numpy()
        np.testing.assert_array_equal(k2.reshape(-1, 2)[t], rot)
        np.testing.assert_array_equal(v2.reshape(-1, 2)[t], vn[t, 0])


def test_kv_append_then_gather_returns_the_chunk_in_order():
    """A chunk appended after a prefix through a shuffled page table comes back,
    token by token, from the page gather of that request."""
    P, C, H, d, page = 5, 11, 2, 8, 4
    table, num_pages = synth.shuffled_page_table([P + C], 93, page=page)
    rng = np.random.default_rng(94)
    kc = rng.normal(0, 1, (H, num_pages, page, d))
    vc = rng.normal(0, 1, (H, num_pages, page, d))
    kn = rng.normal(0, 1, (C, H, d))
    vn = rng.normal(0, 1, (C, H, d))
    pos = np.arange(P, P + C, dtype=np.int32)
    slots = np.array([table[0, p // page] * page + p % page for p in pos], np.int32)
    k2, v2, bad = oracle.kv_append(kn, vn, pos, slots, kc, vc, base=0.0)
    assert bad == 0
    for g in range(H):
        gk = oracle.gather_pages(k2, table, num_pages, g, 0, P + C)
        gv = oracle.gather_pages(v2, table, num_pages, g, 0, P + C)
        np.testing.assert_array_equal(gk[P:], kn[:, g])
        np.testing.assert_array_equal(gv[P:], vn[:, g])
        np.testing.assert_array_equal(gk[:P], oracle.gather_pages(kc, table, num_pages, g, 0, P))


# ------------------------------------------------------------ INT8 cache values

def test_dequant_int8_hand_values():
    codes = np.array([[[1, -1, 127, -127], [0, 5, -6, 64]]], np.int8)       # [1 head][2 tokens][d = 4]
    scales = np.array([[0.5, 0.125]], np.float32)
    want = np.array([[[0.5, -0.5, 63.5, -63.5], [0.0, 0.625, -0.75, 8.0]]])
    np.testing.assert_array_equal(oracle.dequant_int8(codes, scales), want)


def test_dequant_int8_is_exact_product():
    """Every value is code * scale exactly: an 8-bit integer times an fp32 scale
    needs at most 32 significant bits, so fp64 holds it without rounding."""
    rng = np.random.default_rng(96)
    codes = rng.integers(-127, 128, (3, 5, 16)).astype(np.int8)
    scales = rng.uniform(1e-3, 2.0, (3, 5)).astype(np.float32)
    got = oracle.dequant_int8(codes, scales)
    from fractions import Fraction
    for idx in [(0, 0, 0), (1, 2, 3), (2, 4, 15), (0, 3, 7)]:
        assert Fraction(got[idx]) == Fraction(int(codes[idx])) * Fraction(float(scales[idx[:2]]))


def test_decode_over_unit_scale_int8_cache_is_decode_over_the_codes():
    """With every scale 1 the INT8 cache holds the codes themselves: decode over
    the dequantised cache equals decode over the codes as numbers."""
    ctx = [70, 3]
    q, kc, vc, table, num_pages = _decode_case(97, ctx)
    rng = np.random.default_rng(98)
    kq = rng.integers(-127, 128, kc.shape).astype(np.int8)
    vq = rng.integers(-127, 128, vc.shape).astype(np.int8)
    ones = np.ones(kc.shape[:-1], np.float32)
    a = oracle.decode_paged(q / 64.0, oracle.dequant_int8(kq, ones), oracle.dequant_int8(vq, ones), table,
                            np.array(ctx, np.int32), num_pages, 0.1)
    b = oracle.decode_paged(q / 64.0, kq.astype(np.float64), vq.astype(np.float64), table,
                            np.array(ctx, np.int32), num_pages, 0.1)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


# ------------------------------------------------------------ INT8 append (quantisation)

def _q_case(rows_k, rows_v=None):
    """One token, one head: k_new / v_new rows given explicitly; 1 page of 2 slots."""
    k = np.asarray(rows_k, np.float64)[None, None, :]
    v = np.asarray(rows_v if rows_v is not None else rows_k, np.float64)[None, None, :]
    d = k.shape[-1]
    z8 = np.zeros((1, 1, 2, d), np.int8)
    zs = np.zeros((1, 1, 2), np.float32)
    return k, v, z8, zs


def test_int8_append_hand_quantisation():
    """max|x| = 2.54 -> scale 0.02 (fp32); 2.54 -> 127, -1.27 -> -63.5 -> -64 (ties to even),
    0.01 -> 0.5 -> 0, 0.03 -> 1.5 -> 2."""
    row = [2.54, -1.27, 0.01, 0.03]
    k, v, z8, zs = _q_case(row)
    kc, vc, ks, vs, bad = oracle.kv_append_int8(k, v, None, [1], z8, z8, zs, zs, base=0.0)
    s = np.float32(2.54) / np.float32(127.0)
    assert ks[0, 0, 1] == s and vs[0, 0, 1] == s
    want = [int(np.rint(np.float32(x) / s)) for x in row]
    assert want[0] == 127
    np.testing.assert_array_equal(kc[0, 0, 1], want)
    np.testing.assert_array_equal(vc[0, 0, 1], want)
    np.testing.assert_array_equal(kc[0, 0, 0], 0)  # slot 0 untouched
    assert bad == 0


def test_int8_append_zero_row_and_error_bound():
    k, v, z8, zs = _q_case([0.0, 0.0, 0.0, 0.0], [0.5, -0.25, 3.0, 1e-3])
    kc, vc, ks, vs, _ = oracle.kv_append_int8(k, v, None, [0], z8, z8, zs, zs, base=0.0)
    assert ks[0, 0, 0] == 0 and (kc[0, 0, 0] == 0).all()
    # any row: |code * scale - x| <= scale / 2, and the largest |x| maps to +-127
    rng = np.random.default_rng(99)
    for _ in range(50):
        row = rng.normal(0, rng.uniform(0.01, 10), 16).astype(np.float32).astype(np.float64)
        k, v, z8, zs = _q_case(row)
        kc, vc, ks, vs, _ = oracle.kv_append_int8(k, v, None, [0], z8, z8, zs, zs, base=0.0)
        s = float(ks[0, 0, 0])
        back = kc[0, 0, 0].astype(np.float64) * s
        # half a step, plus the fp32 rounding of x / scale near a .5 boundary (a few ulps of x)
        assert (np.abs(back - row) <= s / 2 + np.abs(row) * 2.0 ** -22).all()
        assert np.abs(kc[0, 0, 0]).max() == 127


def test_int8_append_keys_are_quantised_bf16_rotations():
    """With rotation, the key codes are the quantisation of what the bf16 append
    stores: the two appends agree after dequantisation within half a step."""
    rng = np.random.default_rng(100)
    T, H, d = 5, 2, 8
    kn = rng.normal(0, 1, (T, H, d))
    vn = rng.normal(0, 1, (T, H, d))
    pos = np.array([0, 3, 77, 1000, 65535], np.int32)
    slots = np.arange(T, dtype=np.int32)
    z = np.zeros((H, 2, 4, d))
    kb, vb, _ = oracle.kv_append(kn, vn, pos, slots, z, z)
    kc, vc, ks, vs, _ = oracle.kv_append_int8(kn, vn, pos, slots, np.zeros((H, 2, 4, d), np.int8),
                                              np.zeros((H, 2, 4, d), np.int8), np.zeros((H, 2, 4), np.float32),
                                              np.zeros((H, 2, 4), np.float32))
    kd = oracle.dequant_int8(kc, ks)
    assert np.all(np.abs(kd - kb) <= ks[..., None].astype(np.float64) / 2 + np.abs(kb) * 2.0 ** -22)


# ------------------------------------------------------------ FP8 (e4m3)

def test_round_e4m3_matches_torch_conversion():
    """Every e4m3 value and every midpoint between neighbours (ties to even),
    against torch's float8_e4m3fn conversion."""
    codes = torch.arange(0, 256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).float()
    vals = codes[torch.isfinite(codes)].double().unique().numpy()
    mids = (vals[:-1] + vals[1:]) / 2
    rng = np.random.default_rng(101)
    rand = rng.uniform(-448, 448, 2000) * rng.choice([1, 1e-1, 1e-2, 1e-3], 2000)
    x = np.concatenate([vals, mids, -mids, rand]).astype(np.float32).astype(np.float64)
    want = torch.from_numpy(x).float().to(torch.float8_e4m3fn).float().double().numpy()
    np.testing.assert_array_equal(oracle.round_e4m3(x), want)


def test_round_e4m3_saturates_and_keeps_signed_zero():
    got = oracle.round_e4m3(np.array([448.0, 449.0, 479.0, 1e6, -1e6, 0.0, -0.0, 2.0 ** -10, 2.0 ** -9]))
    np.testing.assert_array_equal(got[:5], [448.0, 448.0, 448.0, 448.0, -448.0])
    assert got[5] == 0.0 and np.signbit(got[6])
    assert got[7] == 0.0 and got[8] == 2.0 ** -9   # 2^-10 is a tie between 0 and 2^-9: even is 0


def test_quant_e4m3_groups_and_scale():
    """One scale per group (max|x| / 448 in fp32): the largest |x| of a group maps
    to +-448, every value is within half an e4m3 step (relative 2^-4) of x / scale,
    and a zero group has scale 0."""
    rng = np.random.default_rng(102)
    x = rng.normal(0, 1, (3, 5, 32)).astype(np.float32).astype(np.float64)
    x[2, 4] = 0.0
    codes, scales = oracle.quant_e4m3(x, [0, 1])
    assert scales.shape == (3, 5) and scales[2, 4] == 0 and (codes[2, 4] == 0).all()
    for i in range(3):
        for j in range(5):
            if scales[i, j] == 0:
                continue
            s = np.float32(np.abs(x[i, j]).max().astype(np.float32) / np.float32(448.0))
            assert scales[i, j] == s
            assert np.abs(codes[i, j]).max() == 448.0
            ref = (x[i, j].astype(np.float32) / s).astype(np.float64)
            assert np.all(np.abs(codes[i, j] - ref) <= np.maximum(np.abs(ref) * 2.0 ** -4, 2.0 ** -10))
    # group axes in another order: per column group
    c2, s2 = oracle.quant_e4m3(x, [2])
    assert s2.shape == (32,)
    np.testing.assert_array_equal(s2, (np.abs(x).max(axis=(0, 1)).astype(np.float32) / np.float32(448.0)))



def test_quant_e4m3_decides_codes_in_fp32():
    """The code of x is e4m3(x / scale) with the quotient rounded to fp32 first.
    For a group with maximum 400 (scale = 400/448 in fp32), x = 1.171875 gives the
    fp32 quotient 1.3125 exactly: the midpoint between the e4m3 values 1.25 and
    1.375, which ties to even, 1.25.  The exact quotient is 1.3125000125..., which
    would round up to 1.375.  The expected value comes from numpy's fp32 division
    and torch's float8_e4m3fn conversion, not from the oracle."""
    x = np.array([[400.0, 1.171875, -1.171875]])
    codes, scales = oracle.quant_e4m3(x, [0])
    s32 = np.float32(400.0) / np.float32(448.0)
    assert scales[0] == s32
    q32 = np.float32(1.171875) / s32
    assert float(q32) == 1.3125
    want = torch.tensor([float(q32)]).to(torch.float8_e4m3fn).float().item()
    assert want == 1.25
    np.testing.assert_array_equal(codes[0], [448.0, 1.25, -1.25])



def test_int8_codes_are_decided_on_the_fp32_quotient():
    """Row maximum 37.5 (scale = 37.5/127 in fp32) and x = 18.75: the fp32
    quotient is exactly 63.5, which rounds to the even 64; the exact quotient is
    63.49999823..., which would round to 63.  The expectation comes from numpy's
    fp32 division and rint, not from the oracle."""
    row = [37.5, 18.75, -18.75, 0.0]
    k, v, z8, zs = _q_case(row)
    kc, vc, ks, vs, _ = oracle.kv_append_int8(k, v, None, [0], z8, z8, zs, zs, base=0.0)
    s = np.float32(37.5) / np.float32(127.0)
    q = np.float32(18.75) / s
    assert float(q) == 63.5 and np.rint(q) == 64
    assert abs(18.75 / float(s) - 63.5) > 1e-7
    np.testing.assert_array_equal(vc[0, 0, 0], [127, 64, -64, 0])
    np.testing.assert_array_equal(kc[0, 0, 0], [127, 64, -64, 0])
