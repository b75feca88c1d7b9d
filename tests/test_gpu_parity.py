"""CUDA path vs the fp64 CPU oracle, element by element, on seeded inputs.

Tolerances (bf16 inputs, fp32 accumulation): max |dO| <= 1e-2, mean |dO| <= 1e-3,
max |dLSE| <= 1e-3.  fp32 inputs (CUDA-core path): 1e-5.  Integer work (page
gather, positions) is checked bit-exactly through invariance tests.

The path stores RoPE's output in the tensor's dtype, so attention consumes
bf16-rounded rotated Q/K; the oracle models that step by rounding its own fp64
rotation to bf16 (ties to even) before its three-pass attention.
"""
import math

import numpy as np
import pytest
import torch

import attention_tiled_causal_gb300 as atc
import oracle
import synth

pytestmark = pytest.mark.gpu
DEV = "cuda"
TOL_MAX, TOL_MEAN, TOL_LSE = 1e-2, 1e-3, 1e-3
TOL_F32 = 1e-5


def check(out, lse, want_o, want_l, tol_max=TOL_MAX, tol_mean=TOL_MEAN, tol_lse=TOL_LSE, what=""):
    o = out.float().cpu().numpy() if torch.is_tensor(out) else out
    d = np.abs(o - want_o)
    assert np.isfinite(o).all(), f"{what}: non-finite output"
    assert d.max() <= tol_max, f"{what}: max |dO| = {d.max():.3g}"
    assert d.mean() <= tol_mean, f"{what}: mean |dO| = {d.mean():.3g}"
    if lse is not None:
        l = lse.cpu().numpy() if torch.is_tensor(lse) else lse
        inf = np.isinf(want_l)
        assert np.array_equal(np.isinf(l), inf), f"{what}: -inf LSE pattern differs"
        if (~inf).any():
            dl = np.abs(l[~inf] - want_l[~inf]).max()
            assert dl <= tol_lse, f"{what}: max |dLSE| = {dl:.3g}"


def rotated_bf16(x, pos, base=10000.0):
    return oracle.round_bf16(oracle.rope(synth.as_f64(x), np.asarray(pos)))


def seq_ids(lens):
    return np.repeat(np.arange(len(lens), dtype=np.int32), lens)


@pytest.fixture(autouse=True)
def _clean_device_status():
    atc.attn_device_status(clear=True)
    yield
    atc.attn_device_status(clear=True)


# ------------------------------------------------------------------ RoPE

def test_rope_bf16_matches_oracle_within_one_ulp():
    T, H, d = 1500, 8, 128
    x = synth.randn((T, H, d), 101, 0.7071)
    pos = np.sort(np.random.default_rng(1).integers(0, 131072, T)).astype(np.int32)
    pos[:4] = [0, 1, 65535, 131071]
    xd = x.to(DEV)
    atc.rope_apply(xd, torch.from_numpy(pos).to(DEV))
    got = synth.as_f64(xd.cpu())
    want = rotated_bf16(x, pos)
    # one bf16 ulp of the result, plus the absolute error of an fp32 rotation
    # (terms of size |x| ~ 4 cancel to tiny results: ~2^-24 * |x| each)
    bound = np.abs(want) * 2.0 ** -7 + 2e-6
    diff = np.abs(got - want)
    worst = np.unravel_index(np.argmax(diff - bound), diff.shape)
    assert (diff <= bound).all(), f"diff {diff[worst]:.3g} at {worst} (want {want[worst]:.6g})"
    assert (diff > 0).mean() < 0.01, f"{(diff > 0).mean():.3%} of elements differ by one ulp"
    np.testing.assert_array_equal(got[pos == 0], synth.as_f64(x)[pos == 0])  # position 0: identity


def test_rope_fp32_matches_oracle():
    T, H, d = 333, 2, 64
    x = synth.randn((T, H, d), 102, 1.0, torch.float32)
    pos = np.arange(T, dtype=np.int32) * 97
    xd = x.to(DEV)
    atc.rope_apply(xd, torch.from_numpy(pos).to(DEV))
    want = oracle.rope(synth.as_f64(x), pos)
    assert np.abs(xd.cpu().double().numpy() - want).max() < 2e-6



@pytest.mark.parametrize("dtype,d,H", [(torch.bfloat16, 96, 40), (torch.float32, 40, 3), (torch.bfloat16, 224, 5)])
def test_rope_head_dims_with_odd_chunk_counts(dtype, d, H):
    """Head sizes whose half is not a power-of-two number of 16-byte chunks (6, 5
    and 14 chunks) and head counts that leave partial passes: the kernels walk
    (chunk, head, token) by constant steps, which must match the oracle here too."""
    T = 203
    x = synth.randn((T, H, d), 104 + d, 0.7071, dtype=dtype)
    pos = np.arange(T, dtype=np.int32) * 31 + 7
    xd = x.to(DEV)
    atc.rope_apply(xd, torch.from_numpy(pos).to(DEV))
    atc.attn_device_status()
    got = synth.as_f64(xd.cpu())
    if dtype == torch.bfloat16:
        want = rotated_bf16(x, pos)
        assert (np.abs(got - want) <= np.abs(want) * 2.0 ** -7 + 2e-6).all()
    else:
        assert np.abs(got - oracle.rope(synth.as_f64(x), pos)).max() < 2e-6


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_rope_apply_qk_equals_two_rope_apply_calls(dtype):
    """Queries and keys rotated in one launch equal two rope_apply calls bit for
    bit, for the 64/8 layout (4 tokens per block) and a few-head one (16 per
    block), with a ragged token count."""
    for T, hq, hk, seed in ((301, 64, 8, 760), (77, 8, 2, 761)):
        q = synth.randn((T, hq, 128), seed, 0.7071, dtype=dtype).to(DEV)
        k = synth.randn((T, hk, 128), seed + 1, 0.7071, dtype=dtype).to(DEV)
        pos = torch.from_numpy(synth.positions([T], [123456])).to(DEV)
        q2, k2 = q.clone(), k.clone()
        atc.rope_apply_qk(q, k, pos)
        atc.rope_apply(q2, pos)
        atc.rope_apply(k2, pos)
        atc.attn_device_status()
        assert torch.equal(q, q2) and torch.equal(k, k2)

def test_rope_strided_token_rows():
    """Rotating a [T, H, d] view of a wider buffer touches only that view."""
    T, H, d = 64, 4, 128
    big = synth.randn((T, 2 * H, d), 103, 1.0).to(DEV)
    before = big.clone()
    pos = torch.arange(T, dtype=torch.int32, device=DEV) + 7
    atc.rope_apply(big[:, :H], pos)
    assert torch.equal(big[:, H:], before[:, H:])
    want = rotated_bf16(before[:, :H].cpu(), pos.cpu().numpy())
    assert np.abs(synth.as_f64(big[:, :H].cpu()) - want).max() <= 2.0 ** -7 * 4


@pytest.mark.parametrize("hq,hk,d,dtype", [(64, 8, 128, torch.bfloat16), (5, 1, 64, torch.bfloat16),
                                           (3, 1, 32, torch.float32), (100, 20, 256, torch.bfloat16)])
def test_rope_apply_qk_long_equals_strided_calls(hq, hk, d, dtype):
    """rope_apply_qk on long contiguous Q and K (one launch for both tensors)
    equals, bit for bit, the same rows rotated one tensor at a time through
    strided views of wider buffers, and stays within one ulp of the oracle's
    rounded rotation on sampled tokens; bf16 and fp32, several head counts and
    head dims."""
    T = 20011 if hq < 100 else 3001
    q = synth.randn((T, hq, d), 900 + hq, 0.7071, dtype)
    k = synth.randn((T, hk, d), 901 + hq, 0.7071, dtype)
    pos = (np.arange(T, dtype=np.int32) * 3 + 11).astype(np.int32)
    posd = torch.from_numpy(pos).to(DEV)
    qd, kd = q.to(DEV), k.to(DEV)
    atc.rope_apply_qk(qd, kd, posd)
    # the same rows as strided views of wider buffers: the unstaged kernel
    qw = torch.zeros((T, hq + 1, d), dtype=dtype, device=DEV)
    kw = torch.zeros((T, hk + 1, d), dtype=dtype, device=DEV)
    qw[:, :hq] = q.to(DEV)
    kw[:, :hk] = k.to(DEV)
    atc.rope_apply(qw[:, :hq], posd)
    atc.rope_apply(kw[:, :hk], posd)
    atc.attn_device_status()
    assert torch.equal(qd, qw[:, :hq]) and torch.equal(kd, kw[:, :hk])
    rows = np.unique(np.concatenate([[0, 1, T // 2, T - 1], np.random.default_rng(hq).integers(0, T, 60)]))
    for x, xd in ((q, qd), (k, kd)):
        got = synth.as_f64(xd[torch.from_numpy(rows).to(DEV)].cpu())
        if dtype == torch.bfloat16:
            want = rotated_bf16(x[torch.from_numpy(rows)], pos[rows])
            assert (np.abs(got - want) <= np.abs(want) * 2.0 ** -7 + 2e-6).all()
        else:
            want = oracle.rope(synth.as_f64(x[torch.from_numpy(rows)]), pos[rows])
            assert np.abs(got - want).max() < 2e-6


@pytest.mark.parametrize("which,code", [(0, 0x102), (1, 0x105)])
def test_bounded_wait_runs_out_records_its_code_and_the_context_stays_usable(which, code):
    """A kernel waits on an mbarrier that nothing completes (no fault, no trap):
    the wait gives up after its limit, the code is reported by the next status
    read, and the next call on the same context runs and matches the oracle."""
    atc.attn_device_status(clear=True)
    atc.attn_selftest_wait_timeout(which)
    with pytest.raises(atc.AttnError) as e:
        atc.attn_device_status(clear=True)
    assert e.value.status == 6 and f"0x{code:x}" in str(e.value)
    atc.attn_device_status(clear=True)
    x = synth.randn((64, 2, 128), 990, 0.7071)
    pos = np.arange(64, dtype=np.int32)
    xd = x.to(DEV)
    atc.rope_apply(xd, torch.from_numpy(pos).to(DEV))
    atc.attn_device_status()
    want = rotated_bf16(x, pos)
    assert (np.abs(synth.as_f64(xd.cpu()) - want) <= np.abs(want) * 2.0 ** -7 + 2e-6).all()


# ------------------------------------------------------------------ LSE merge

@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("P", [1, 2, 3, 5, 16, 40])
def test_lse_merge_matches_oracle(out_dtype, P):
    """Part counts that take each merge kernel (2 or fewer, 4 or fewer, 32 or
    fewer, more), a ragged number of (row, head) items, an empty part whose
    output rows hold NaN (a part with LSE -inf contributes nothing, whatever its
    rows hold) and a row with no part at all."""
    R, H, d = 37, 6, 128
    rng = np.random.default_rng(7 + P)
    po = rng.normal(0, 1, (P, R, H, d)).astype(np.float32)
    pl = rng.normal(0, 3, (P, R, H)).astype(np.float32)
    pl[P // 2, :, 0] = -np.inf      # an empty part
    pl[:, 3, 2] = -np.inf          # a row with no part at all
    want_o, want_l = oracle.lse_merge(po.astype(np.float64), pl.astype(np.float64))
    po_gpu = po.copy()
    po_gpu[P // 2, :, 0] = np.nan   # never read into the sum
    po_gpu[:, 3, 2] = np.nan
    out = torch.empty((R, H, d), dtype=out_dtype, device=DEV)
    lse = torch.empty((R, H), dtype=torch.float32, device=DEV)
    atc.attn_lse_merge(torch.from_numpy(po_gpu).to(DEV), torch.from_numpy(pl).to(DEV), out, lse)
    # bf16 output: rounding to nearest costs at most half an ulp, 2^-8 of |O| (relative to its binade)
    tol = 1e-5 if out_dtype == torch.float32 else 2.0 ** -8 * np.abs(want_o).max() + 1e-5
    check(out, lse, want_o, want_l, tol_max=tol, tol_mean=tol, tol_lse=1e-5, what=f"merge P={P}")
    assert torch.all(out[3, 2] == 0)


def test_lse_merge_strided_split_layout():
    """Partials laid out [rows, H, splits, d] (the decode workspace) via strides."""
    R, H, S, d = 9, 4, 16, 128
    rng = np.random.default_rng(8)
    po = rng.normal(0, 1, (R, H, S, d)).astype(np.float32)
    pl = rng.normal(0, 1, (R, H, S)).astype(np.float32)
    pl[:, :, 10:] = -np.inf
    want_o, want_l = oracle.lse_merge(po.transpose(2, 0, 1, 3), pl.transpose(2, 0, 1))
    po_d = torch.from_numpy(po).to(DEV)
    pl_d = torch.from_numpy(pl).to(DEV)
    out = torch.empty((R, H, d), dtype=torch.float32, device=DEV)
    lse = torch.empty((R, H), dtype=torch.float32, device=DEV)
    atc.attn_lse_merge(po_d.permute(2, 0, 1, 3), pl_d.permute(2, 0, 1), out, lse)
    check(out, lse, want_o, want_l, tol_max=1e-5, tol_mean=1e-6, tol_lse=1e-5, what="strided merge")


# ------------------------------------------------------------------ prefill: fp32 tiny (CUDA cores)

def _tiny_run(w, inp, h_lo=0, h_hi=None, key_rows=None):
    q, k, v = inp["q"].clone().to(DEV), inp["k"].clone().to(DEV), inp["v"].to(DEV)
    pos = inp["pos"].to(DEV)
    atc.rope_apply(q, pos)
    atc.rope_apply(k, pos)
    cu = inp["cu"].to(DEV)
    if key_rows is not None:
        idx = torch.from_numpy(key_rows).to(DEV)
        k, v, kpos = k[idx].contiguous(), v[idx].contiguous(), pos[idx].contiguous()
        cu_k = torch.tensor([0, len(key_rows)], dtype=torch.int32, device=DEV)
    else:
        kpos, cu_k = pos, cu
    out = torch.full(q.shape, float("nan"), dtype=torch.float32, device=DEV)
    lse = torch.full(q.shape[:2], float("nan"), dtype=torch.float32, device=DEV)
    atc.attn_prefill(q, k, v, out, lse, cu, pos, w.seq, cu_k=cu_k, k_pos=kpos, h_lo=h_lo, h_hi=h_hi)
    atc.attn_device_status()
    return out, lse


def test_tiny_fp32_causal_gqa_matches_oracle():
    w = synth.TINY
    inp = w.make()
    out, lse = _tiny_run(w, inp)
    pos = inp["pos"].numpy()
    qr = oracle.rope(synth.as_f64(inp["q"]), pos)
    kr = oracle.rope(synth.as_f64(inp["k"]), pos)
    want_o, want_l = oracle.attention(qr, seq_ids([w.seq]), pos, kr, synth.as_f64(inp["v"]), inp["cu"].numpy(),
                                      pos, w.scale)
    check(out, lse, want_o, want_l, TOL_F32, TOL_F32, TOL_F32, "tiny fp32")


def test_tiny_fp32_head_slices_and_key_chunks_recombine():
    """Ulysses page, 2.2 (4 segments of 16 tokens): two head slices of one KV group
    each equal the all-heads call, and four key chunks merged by LSE equal it too."""
    w = synth.TINY
    inp = w.make()
    full_o, full_l = _tiny_run(w, inp)
    G = w.hq // w.hkv
    for lo in range(0, w.hq, G):
        o, l = _tiny_run(w, inp, lo, lo + G)
        assert torch.equal(o[:, lo:lo + G], full_o[:, lo:lo + G])
        assert torch.equal(l[:, lo:lo + G], full_l[:, lo:lo + G])
        assert torch.isnan(o[:, :lo]).all() and torch.isnan(o[:, lo + G:]).all()  # other heads untouched
    po, pl = [], []
    for c in range(4):
        o, l = _tiny_run(w, inp, key_rows=np.arange(16 * c, 16 * c + 16))
        po.append(o)
        pl.append(l)
    out = torch.empty_like(full_o)
    lse = torch.empty_like(full_l)
    atc.attn_lse_merge(torch.stack(po), torch.stack(pl), out, lse)
    check(out, lse, full_o.cpu().numpy(), full_l.cpu().numpy(), 1e-5, 1e-6, 1e-5, "chunks merged")


# ------------------------------------------------------------------ prefill: bf16, tensor cores

def _bf16_case(lens, hq, hkv, starts, seed, d=128):
    T = sum(lens)
    q = synth.randn((T, hq, d), seed, 0.7071)
    k = synth.randn((T, hkv, d), seed + 1, 0.7071)
    v = synth.randn((T, hkv, d), seed + 2, 0.7071)
    pos = synth.positions(lens, starts)
    cu = synth.cu_seqlens(lens)
    return q, k, v, pos, cu


def _run_prefill(q, k, v, pos, cu, lens, causal=True, h_lo=0, h_hi=None, out_dtype=None):
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    posd, cud = torch.from_numpy(pos).to(DEV), torch.from_numpy(cu).to(DEV)
    atc.rope_apply(qd, posd)
    atc.rope_apply(kd, posd)
    out = torch.full(q.shape, float("nan"), dtype=out_dtype or q.dtype, device=DEV)
    lse = torch.full(q.shape[:2], float("nan"), dtype=torch.float32, device=DEV)
    atc.attn_prefill(qd, kd, vd, out, lse, cud, posd, max(lens), cu_k=cud, k_pos=posd, h_lo=h_lo, h_hi=h_hi,
                     causal=causal)
    atc.attn_device_status()
    return out, lse


def _oracle_prefill(q, k, v, pos, cu, lens, scale, causal=True, h_lo=0, h_hi=None):
    qr, kr = rotated_bf16(q, pos), rotated_bf16(k, pos)
    return oracle.attention(qr, seq_ids(lens), pos, kr, synth.as_f64(v), cu, pos, scale, causal=causal,
                            h_lo=h_lo, h_hi=h_hi)


CASES = [
    ([300], 16, 2, [0]),                 # several tiles and a ragged tail
    ([1, 129, 513, 256], 16, 2, [5, 0, 100000, 7]),  # varlen batch, offsets, 1-token sequence
    ([700], 64, 8, [0]),                 # the 64/8 head layout
    ([255, 257], 8, 8, [0, 40]),         # MHA, tile edges off by one
]


@pytest.mark.parametrize("lens,hq,hkv,starts", CASES)
def test_prefill_tc_causal_matches_oracle(lens, hq, hkv, starts):
    q, k, v, pos, cu = _bf16_case(lens, hq, hkv, starts, 200 + hq + len(lens))
    out, lse = _run_prefill(q, k, v, pos, cu, lens)
    want_o, want_l = _oracle_prefill(q, k, v, pos, cu, lens, 128 ** -0.5)
    check(out, lse, want_o, want_l, what=f"tc causal {lens}")


def test_prefill_tc_non_causal_and_fp32_output():
    lens = [200, 333]
    q, k, v, pos, cu = _bf16_case(lens, 16, 2, [0, 0], 301)
    out, lse = _run_prefill(q, k, v, pos, cu, lens, causal=False, out_dtype=torch.float32)
    want_o, want_l = _oracle_prefill(q, k, v, pos, cu, lens, 128 ** -0.5, causal=False)
    check(out, lse, want_o, want_l, what="tc non-causal fp32 out")


@pytest.mark.parametrize("d", [64, 256])
def test_prefill_simt_bf16_matches_oracle(d):
    """bf16 at head sizes other than 128 runs on the CUDA-core kernel."""
    lens = [150, 77]
    q, k, v, pos, cu = _bf16_case(lens, 16, 2, [0, 3], 302, d=d)
    out, lse = _run_prefill(q, k, v, pos, cu, lens)
    want_o, want_l = _oracle_prefill(q, k, v, pos, cu, lens, d ** -0.5)
    check(out, lse, want_o, want_l, what=f"simt bf16 d{d}")


def test_prefill_tc_head_slices_are_bit_identical_to_full_call():
    lens = [600]
    q, k, v, pos, cu = _bf16_case(lens, 64, 8, [0], 303)
    full_o, full_l = _run_prefill(q, k, v, pos, cu, lens)
    for lo, hi in ((16, 32), (0, 8), (56, 64)):
        o, l = _run_prefill(q, k, v, pos, cu, lens, h_lo=lo, h_hi=hi)
        assert torch.equal(o[:, lo:hi], full_o[:, lo:hi])
        assert torch.equal(l[:, lo:hi], full_l[:, lo:hi])
        assert torch.isnan(o[:, :lo].float()).all() and torch.isnan(o[:, hi:].float()).all()


def test_prefill_long_sequence_head_slices_are_bit_identical_and_match_oracle():
    """A 20000-token causal prefill (ragged last tile pair): one-group head
    slices equal the full call's heads bit for bit, and sampled rows of the
    full call match the oracle."""
    lens = [20000]
    q, k, v, pos, cu = _bf16_case(lens, 64, 8, [0], 311)
    full_o, full_l = _run_prefill(q, k, v, pos, cu, lens)
    for lo, hi in ((0, 8), (24, 32), (56, 64)):
        o, l = _run_prefill(q, k, v, pos, cu, lens, h_lo=lo, h_hi=hi)
        assert torch.equal(o[:, lo:hi], full_o[:, lo:hi])
        assert torch.equal(l[:, lo:hi], full_l[:, lo:hi])
    rows = np.unique(np.concatenate([[0, 1, 127, 128, 9999, 19999], synth.sample_rows(20000, 10, 312)]))
    qr, kr = rotated_bf16(q, pos), rotated_bf16(k, pos)
    wo, wl = oracle.attention(qr[rows], np.zeros(len(rows), np.int32), pos[rows], kr, synth.as_f64(v),
                              np.array([0, 20000], np.int32), pos, 128 ** -0.5)
    check(full_o[torch.from_numpy(rows).to(DEV)], full_l[torch.from_numpy(rows).to(DEV)], wo, wl,
          what="20000-token prefill")


def _growing_scores_case(T, seed, sign=1.0):
    """Scores that rise along the keys at a rate set per query head: q_h =
    noise + a_h u and k_j = noise + (j / 128) u with u all ones, so head h's
    score grows by about 11.3 a_h (natural units) per 128-key tile.  With a_h =
    0.15 h, heads 0-3 stay under the kernels' 2^8 rescale threshold and heads
    4-7 cross it on every tile: each tile moves the row max, O is rescaled in
    TMEM (bf16) and the e4m3 kernel's lazy check sends the warp back for the
    row max.  With sign -1 the scores fall instead: the row max is set on the
    first tile and later weights underflow towards zero.  No RoPE (the kernels
    take the inputs as given)."""
    hq, hkv, d = 8, 1, 128
    a = (torch.arange(hq, dtype=torch.float32) * 0.15)[None, :, None]
    ramp = sign * (torch.arange(T, dtype=torch.float32) / 128.0)[:, None, None]
    q = (synth.randn((T, hq, d), seed, 0.3).float() + a).to(torch.bfloat16)
    k = (synth.randn((T, hkv, d), seed + 1, 0.3).float() + ramp).to(torch.bfloat16)
    v = synth.randn((T, hkv, d), seed + 2, 0.7071)
    return q, k, v


@pytest.mark.parametrize("sign", [1.0, -1.0])
def test_prefill_tc_scores_growing_along_the_keys(sign):
    """Row maxima that grow on every key tile (O rescaled in TMEM tile after
    tile) and ones that never cross the threshold, in one call -- or, falling,
    a max fixed on the first tile and weights that underflow -- against the
    oracle at the bf16 tolerances."""
    lens = [700]
    q, k, v = _growing_scores_case(700, 320, sign)
    pos, cu = synth.positions(lens, [0]), synth.cu_seqlens(lens)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    posd, cud = torch.from_numpy(pos).to(DEV), torch.from_numpy(cu).to(DEV)
    out, lse = atc.prefill(qd, kd, vd, cud, posd, 700, cu_k=cud, k_pos=posd)
    atc.attn_device_status()
    want_o, want_l = oracle.attention(synth.as_f64(q), seq_ids(lens), pos, synth.as_f64(k), synth.as_f64(v), cu, pos,
                                      128 ** -0.5)
    if sign > 0:
        assert want_l[-1, 7] - want_l[-1, 0] > 30  # the steep heads' scores are far above the flat ones'
    check(out, lse, want_o, want_l, what=f"growing scores, sign {sign}")


@pytest.mark.parametrize("sign", [1.0, -1.0])
def test_prefill_fp8_scores_growing_along_the_keys(sign):
    """The same inputs through the e4m3 kernel, against the oracle on the
    dequantised inputs.  Its steep heads' rows are dominated by a few keys, so
    the rounding of the largest weights to e4m3 (relative error up to 2^-4)
    reaches O without averaging: the bound is the worst case, 2^-4 max|v| per
    element and 2^-4 mean|v| on average; the scores are exact, so the LSE bound
    stays 1e-3."""
    lens = [704]
    q, k, v = _growing_scores_case(704, 330, sign)
    pos, cu = synth.positions(lens, [0]), synth.cu_seqlens(lens)
    out, lse = _run_fp8(q, k, v, pos, cu, lens)
    want_o, want_l, vh = _fp8_oracle(q, k, v, pos, cu, lens)
    check(out, lse, want_o, want_l, tol_max=_fp8_max_tol(vh), tol_mean=2.0 ** -4 * np.abs(vh).mean(),
          what=f"fp8 growing scores, sign {sign}")


def test_prefill_fully_masked_rows_give_zero_and_minus_inf():
    """Queries at positions 0..9 against keys at positions 50..249: nothing visible."""
    d, hq, hkv = 128, 8, 1
    q = synth.randn((10, hq, d), 304, 0.7).to(DEV)
    k = synth.randn((200, hkv, d), 305, 0.7).to(DEV)
    v = synth.randn((200, hkv, d), 306, 0.7).to(DEV)
    qpos = torch.arange(10, dtype=torch.int32, device=DEV)
    kpos = torch.arange(50, 250, dtype=torch.int32, device=DEV)
    out, lse = atc.prefill(q, k, v, torch.tensor([0, 10], dtype=torch.int32, device=DEV), qpos, 10,
                           cu_k=torch.tensor([0, 200], dtype=torch.int32, device=DEV), k_pos=kpos)
    atc.attn_device_status()
    assert torch.all(out == 0) and torch.all(lse == -math.inf)


def test_prefill_zero_length_sequence_in_batch():
    lens = [0, 130, 0]
    q, k, v, pos, cu = _bf16_case(lens, 8, 1, [0, 0, 0], 307)
    out, lse = _run_prefill(q, k, v, pos, cu, lens)
    want_o, want_l = _oracle_prefill(q, k, v, pos, cu, lens, 128 ** -0.5)
    check(out, lse, want_o, want_l, what="zero-length sequences")


# ------------------------------------------------------------------ chunked prefill over a paged prefix

def _chunked_case(prefix, chunk, B, hq, hkv, seed, d=128):
    table, num_pages = synth.shuffled_page_table([prefix] * B, seed)
    kc = synth.randn((hkv, num_pages, 64, d), seed + 1, 0.7071)
    vc = synth.randn((hkv, num_pages, 64, d), seed + 2, 0.7071)
    q = synth.randn((B * chunk, hq, d), seed + 3, 0.7071)
    k = synth.randn((B * chunk, hkv, d), seed + 4, 0.7071)
    v = synth.randn((B * chunk, hkv, d), seed + 5, 0.7071)
    return table, num_pages, kc, vc, q, k, v


def _chunked_gpu(prefix, chunk, B, table, num_pages, kc, vc, q, k, v):
    qpos = torch.from_numpy(synth.positions([chunk] * B, [prefix] * B)).to(DEV)
    cu = torch.from_numpy(synth.cu_seqlens([chunk] * B)).to(DEV)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    atc.rope_apply(qd, qpos)
    atc.rope_apply(kd, qpos)
    T, hq, d = q.shape
    po = torch.empty((2, T, hq, d), dtype=torch.float32, device=DEV)
    pl = torch.empty((2, T, hq), dtype=torch.float32, device=DEV)
    atc.attn_prefill(qd, kc.to(DEV), vc.to(DEV), po[0], pl[0], cu, qpos, chunk,
                     page_table=torch.from_numpy(table).to(DEV),
                     k_lens=torch.full((B,), prefix, dtype=torch.int32, device=DEV), num_pages=num_pages)
    atc.attn_prefill(qd, kd, vd, po[1], pl[1], cu, qpos, chunk, cu_k=cu, k_pos=qpos)
    out = torch.empty((T, hq, d), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((T, hq), dtype=torch.float32, device=DEV)
    atc.attn_lse_merge(po, pl, out, lse)
    atc.attn_device_status()
    return out, lse


def _chunked_oracle(prefix, chunk, B, table, num_pages, kc, vc, q, k, v, rows=None):
    """Oracle: one causal attention of each chunk query over [prefix ; chunk] keys,
    the prefix gathered from the paged cache in logical order."""
    hkv = kc.shape[0]
    qpos = synth.positions([chunk] * B, [prefix] * B)
    qr = rotated_bf16(q, qpos)
    kr = rotated_bf16(k, qpos)
    kcf, vcf = synth.as_f64(kc), synth.as_f64(vc)
    keys, vals, kpos = [], [], []
    for b in range(B):
        kb = np.stack([oracle.gather_pages(kcf, table, num_pages, g, b, prefix) for g in range(hkv)], 1)
        vb = np.stack([oracle.gather_pages(vcf, table, num_pages, g, b, prefix) for g in range(hkv)], 1)
        keys += [kb, kr[b * chunk:(b + 1) * chunk]]
        vals += [vb, synth.as_f64(v[b * chunk:(b + 1) * chunk])]
        kpos += [np.arange(prefix, dtype=np.int32), qpos[b * chunk:(b + 1) * chunk]]
    K, V, KP = np.concatenate(keys), np.concatenate(vals), np.concatenate(kpos)
    cu_k = synth.cu_seqlens([prefix + chunk] * B)
    sel = np.arange(B * chunk) if rows is None else rows
    o, l = oracle.attention(qr[sel], seq_ids([chunk] * B)[sel], qpos[sel], K, V, cu_k, KP, 128 ** -0.5)
    return o, l, sel


def test_chunked_prefill_over_shuffled_paged_prefix_matches_oracle():
    prefix, chunk, B, hq, hkv = 1000, 200, 2, 16, 2
    case = _chunked_case(prefix, chunk, B, hq, hkv, 400)
    out, lse = _chunked_gpu(prefix, chunk, B, *case)
    o, l, _ = _chunked_oracle(prefix, chunk, B, *case)
    check(out, lse, o, l, what="chunked paged prefill")


def test_paged_prefill_invariant_under_page_permutation():
    """Moving the prefix pages to other physical slots changes no output bit."""
    prefix, chunk, B, hq, hkv = 640, 130, 2, 8, 1
    table, num_pages, kc, vc, q, k, v = _chunked_case(prefix, chunk, B, hq, hkv, 401)
    out1, lse1 = _chunked_gpu(prefix, chunk, B, table, num_pages, kc, vc, q, k, v)
    perm = np.random.default_rng(3).permutation(num_pages)
    inv = np.argsort(perm)
    table2 = np.where(table >= 0, inv[np.maximum(table, 0)], -1).astype(np.int32)
    out2, lse2 = _chunked_gpu(prefix, chunk, B, table2, num_pages, kc[:, perm].contiguous(),
                              vc[:, perm].contiguous(), q, k, v)
    assert torch.equal(out1, out2) and torch.equal(lse1, lse2)


# ------------------------------------------------------------------ decode

def _decode(wl, inp, splits):
    g = {k: (t.to(DEV) if torch.is_tensor(t) else t) for k, t in inp.items()}
    q = g["q"].clone()
    atc.rope_apply(q, g["q_pos"])
    po, pl = atc.decode_workspace(wl.batch, wl.hq, splits, wl.d, DEV)
    out = torch.empty((wl.batch, wl.hq, wl.d), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((wl.batch, wl.hq), dtype=torch.float32, device=DEV)
    atc.attn_decode_paged(q, g["k_cache"], g["v_cache"], g["page_table"], g["ctx_lens"], splits, po, pl, out, lse)
    atc.attn_device_status()
    return out, lse, po, pl


def _decode_oracle(wl, inp):
    qr = rotated_bf16(inp["q"], inp["q_pos"].numpy())
    return oracle.decode_paged(qr, synth.as_f64(inp["k_cache"]), synth.as_f64(inp["v_cache"]),
                               inp["page_table"].numpy(), inp["ctx_lens"].numpy(), inp["num_pages"], wl.scale)


@pytest.mark.parametrize("splits", [1, 4, 16])
def test_decode_matches_oracle(splits):
    ctx = [1, 63, 64, 65, 700, 2049, 130]
    wl = synth.Decode("decode small", batch=len(ctx), ctx_lo=0, ctx_hi=0, hq=16, hkv=2, d=128, splits=splits,
                      seed=500 + splits, ctx_fixed=ctx)
    inp = wl.make()
    out, lse, _, _ = _decode(wl, inp, splits)
    want_o, want_l = _decode_oracle(wl, inp)
    check(out, lse, want_o, want_l, what=f"decode splits={splits}")


def test_decode_64_8_heads_zero_context_request():
    ctx = [0, 3000, 5]
    wl = synth.Decode("decode 64/8", batch=3, ctx_lo=0, ctx_hi=0, hq=64, hkv=8, d=128, splits=16, seed=510,
                      ctx_fixed=ctx)
    inp = wl.make()
    out, lse, _, _ = _decode(wl, inp, 16)
    want_o, want_l = _decode_oracle(wl, inp)
    check(out, lse, want_o, want_l, what="decode 64/8")
    assert torch.all(out[0] == 0) and torch.all(lse[0] == -math.inf)


def test_decode_invariant_under_page_permutation_and_request_order():
    """Ulysses page, 3.5, third check: reusing the cache with pages moved and the
    batch reordered changes no output bit."""
    ctx = [100, 1000, 64, 333]
    wl = synth.Decode("decode perm", batch=4, ctx_lo=0, ctx_hi=0, hq=16, hkv=2, d=128, splits=4, seed=520,
                      ctx_fixed=ctx)
    inp = wl.make()
    out, lse, _, _ = _decode(wl, inp, 4)
    n = inp["num_pages"]
    perm = np.random.default_rng(2).permutation(n)
    inv = np.argsort(perm)
    t = inp["page_table"].numpy()
    inp2 = dict(inp)
    inp2["k_cache"] = inp["k_cache"][:, perm].contiguous()
    inp2["v_cache"] = inp["v_cache"][:, perm].contiguous()
    inp2["page_table"] = torch.from_numpy(np.where(t >= 0, inv[np.maximum(t, 0)], -1).astype(np.int32))
    out2, lse2, _, _ = _decode(wl, inp2, 4)
    assert torch.equal(out, out2) and torch.equal(lse, lse2)
    order = [2, 0, 3, 1]
    inp3 = dict(inp)
    for key in ("q", "page_table", "ctx_lens", "q_pos"):
        inp3[key] = inp[key][order].contiguous()
    out3, lse3, _, _ = _decode(wl, inp3, 4)
    assert torch.equal(out3, out[order]) and torch.equal(lse3, lse[order])


def test_decode_bad_page_id_is_reported_not_faulted():
    """A page-table entry outside the cache is caught on the device: the kernel
    reads page 0 instead, records the fault, and the host reports it."""
    ctx = [200]
    wl = synth.Decode("decode bad page", batch=1, ctx_lo=0, ctx_hi=0, hq=8, hkv=1, d=128, splits=2, seed=530,
                      ctx_fixed=ctx)
    inp = wl.make()
    inp["page_table"] = inp["page_table"].clone()
    inp["page_table"][0, 1] = inp["num_pages"] + 5
    g = {k: (t.to(DEV) if torch.is_tensor(t) else t) for k, t in inp.items()}
    po, pl = atc.decode_workspace(1, 8, 2, 128, DEV)
    atc.attn_decode_paged(g["q"], g["k_cache"], g["v_cache"], g["page_table"], g["ctx_lens"], 2, po, pl)
    with pytest.raises(atc.AttnError) as e:
        atc.attn_device_status(clear=True)
    assert e.value.status == 6
    atc.attn_device_status(clear=True)  # cleared


def test_prefill_tc_is_deterministic_across_runs():
    """Repeated calls on the same inputs give bit-identical O and LSE: no part of the
    pipeline (TMA ring, TMEM score/accumulator reuse, P hand-off) races."""
    lens = [2048, 700]
    q, k, v, pos, cu = _bf16_case(lens, 64, 8, [0, 3], 308)
    first = _run_prefill(q, k, v, pos, cu, lens)
    for _ in range(3):
        o, l = _run_prefill(q, k, v, pos, cu, lens)
        assert torch.equal(o, first[0]) and torch.equal(l, first[1])


# ------------------------------------------------------------------ append to the paged cache

def _slots_for(table, b, positions, page=64):
    return np.array([table[b, p // page] * page + p % page for p in positions], np.int32)


def _append_inputs(prefix, chunk, hkv, d, seed, pad=0):
    table, num_pages = synth.shuffled_page_table([p + c for p, c in zip(prefix, chunk)], seed)
    kc0 = synth.randn((hkv, num_pages, 64, d), seed + 1, 0.7071)
    vc0 = synth.randn((hkv, num_pages, 64, d), seed + 2, 0.7071)
    T = sum(chunk) + pad
    kn = synth.randn((T, hkv, d), seed + 3, 0.7071)
    vn = synth.randn((T, hkv, d), seed + 4, 0.7071)
    pos, slots = [], []
    for b, (p, c) in enumerate(zip(prefix, chunk)):
        pp = np.arange(p, p + c, dtype=np.int32)
        pos.append(pp)
        slots.append(_slots_for(table, b, pp))
    pos.append(np.zeros(pad, np.int32))
    slots.append(np.full(pad, -1, np.int32))
    return table, num_pages, kc0, vc0, kn, vn, np.concatenate(pos), np.concatenate(slots)


def test_kv_append_matches_oracle_and_rope_apply():
    """A 3-request chunk plus 3 padding tokens (slot -1), appended after prefixes of
    64, 130 and 0 tokens through a shuffled page table.  Values land bit-exactly,
    keys within one bf16 ulp of the oracle's rounded rotation and bit-identical
    to rope_apply; every other cache row is untouched."""
    hkv, d = 8, 128
    table, num_pages, kc0, vc0, kn, vn, pos, slots = _append_inputs([64, 130, 0], [100, 1, 260], hkv, d, 95, pad=3)
    T = kn.shape[0]
    kc, vc = kc0.to(DEV), vc0.to(DEV)
    ko = torch.full((T, hkv, d), float("nan"), dtype=torch.bfloat16, device=DEV)
    posd, slotd = torch.from_numpy(pos).to(DEV), torch.from_numpy(slots).to(DEV)
    atc.attn_kv_append_paged(kn.to(DEV), vn.to(DEV), posd, slotd, kc, vc, k_rot_out=ko)
    atc.attn_device_status()
    wk, wv, bad = oracle.kv_append(synth.as_f64(kn), synth.as_f64(vn), pos, slots, synth.as_f64(kc0),
                                   synth.as_f64(vc0))
    assert bad == 0
    np.testing.assert_array_equal(synth.as_f64(vc.cpu()), wv)
    got = synth.as_f64(kc.cpu()).reshape(hkv, -1, d)
    want = wk.reshape(hkv, -1, d)
    written = np.zeros(got.shape[1], bool)
    written[slots[slots >= 0]] = True
    np.testing.assert_array_equal(got[:, ~written], want[:, ~written])
    diff = np.abs(got[:, written] - want[:, written])
    bound = np.abs(want[:, written]) * 2.0 ** -7 + 2e-6
    assert (diff <= bound).all()
    assert (diff > 0).mean() < 0.01
    kr = kn.to(DEV).clone()
    atc.rope_apply(kr, posd)
    valid = torch.from_numpy(slots >= 0).to(DEV)
    assert torch.equal(ko[valid], kr[valid])
    assert torch.isnan(ko[~valid].float()).all()
    rows = torch.from_numpy(slots[slots >= 0].astype(np.int64)).to(DEV)
    assert torch.equal(kc.reshape(hkv, -1, d)[:, rows].permute(1, 0, 2), kr[valid])


@pytest.mark.parametrize("hkv,d,tokens", [(8, 128, 20011), (3, 64, 30011), (40, 96, 6007), (1, 16, 70001),
                                          (64, 256, 2003)])
def test_kv_append_many_groups_matches_oracle_and_rope_apply(hkv, d, tokens):
    """A chunk long enough that the append's blocks each take many groups of
    tokens in turn, over head counts and head dims whose groups hold 4, 21, 1
    and 256 tokens, and one (64 heads of 256) past what the staged path takes.
    The slots are a shuffled set of cache rows with two padding tokens (-1) and
    one slot past the cache. The bad slot is recorded and skipped. Values land
    bit-exactly, keys bit-identical to rope_apply and within one bf16 ulp of the
    oracle's rounded rotation, and every other cache row is untouched."""
    num_pages = (tokens + 63) // 64 + 2
    rows = num_pages * 64
    table, _ = synth.shuffled_page_table([rows], 800 + hkv)
    slots = (table[0][np.arange(tokens) // 64] * 64 + np.arange(tokens) % 64).astype(np.int32)
    slots[tokens // 3] = rows          # past the cache
    slots[[5, tokens - 2]] = -1        # padding
    pos = np.arange(tokens, dtype=np.int32) + 3000
    kn = synth.randn((tokens, hkv, d), 810 + hkv, 0.7071)
    vn = synth.randn((tokens, hkv, d), 820 + hkv, 0.7071)
    kc0 = synth.randn((hkv, num_pages, 64, d), 830 + hkv, 0.7071)
    vc0 = synth.randn((hkv, num_pages, 64, d), 840 + hkv, 0.7071)
    kc, vc = kc0.to(DEV), vc0.to(DEV)
    ko = torch.full((tokens, hkv, d), float("nan"), dtype=torch.bfloat16, device=DEV)
    posd, slotd = torch.from_numpy(pos).to(DEV), torch.from_numpy(slots).to(DEV)
    atc.attn_kv_append_paged(kn.to(DEV), vn.to(DEV), posd, slotd, kc, vc, k_rot_out=ko)
    with pytest.raises(atc.AttnError) as e:
        atc.attn_device_status(clear=True)
    assert e.value.status == 6
    atc.attn_device_status(clear=True)
    wk, wv, bad = oracle.kv_append(synth.as_f64(kn), synth.as_f64(vn), pos, slots, synth.as_f64(kc0),
                                   synth.as_f64(vc0))
    assert bad == 1
    np.testing.assert_array_equal(synth.as_f64(vc.cpu()), wv)
    got = synth.as_f64(kc.cpu()).reshape(hkv, -1, d)
    want = wk.reshape(hkv, -1, d)
    valid_np = (slots >= 0) & (slots < rows)
    written = np.zeros(got.shape[1], bool)
    written[slots[valid_np]] = True
    np.testing.assert_array_equal(got[:, ~written], want[:, ~written])
    diff = np.abs(got[:, written] - want[:, written])
    assert (diff <= np.abs(want[:, written]) * 2.0 ** -7 + 2e-6).all()
    assert (diff > 0).mean() < 0.01
    kr = kn.to(DEV).clone()
    atc.rope_apply(kr, posd)
    valid = torch.from_numpy(valid_np).to(DEV)
    assert torch.equal(ko[valid], kr[valid])
    assert torch.isnan(ko[~valid].float()).all()
    written_rows = torch.from_numpy(slots[valid_np].astype(np.int64)).to(DEV)
    assert torch.equal(kc.reshape(hkv, -1, d)[:, written_rows].permute(1, 0, 2), kr[valid])


def test_kv_append_reports_slot_outside_the_cache():
    """A slot past the cache is not written; the device records it and the host
    reports it.  The other tokens are written (base 0: a plain copy)."""
    hkv, d = 2, 128
    kc = torch.zeros((hkv, 2, 64, d), dtype=torch.bfloat16, device=DEV)
    vc = torch.zeros_like(kc)
    kn = synth.randn((3, hkv, d), 540, 0.7071).to(DEV)
    vn = synth.randn((3, hkv, d), 541, 0.7071).to(DEV)
    slots = torch.tensor([5, 128, 7], dtype=torch.int32, device=DEV)  # 128 = num_pages * page_size
    atc.attn_kv_append_paged(kn, vn, None, slots, kc, vc, base=0.0)
    with pytest.raises(atc.AttnError) as e:
        atc.attn_device_status(clear=True)
    assert e.value.status == 6
    atc.attn_device_status(clear=True)
    flat_k, flat_v = kc.reshape(hkv, -1, d), vc.reshape(hkv, -1, d)
    assert torch.equal(flat_k[:, 5], kn[0]) and torch.equal(flat_k[:, 7], kn[2])
    assert torch.equal(flat_v[:, 5], vn[0]) and torch.equal(flat_v[:, 7], vn[2])
    written = torch.zeros(flat_k.shape[1], dtype=torch.bool, device=DEV)
    written[[5, 7]] = True
    assert (flat_k[:, ~written] == 0).all() and (flat_v[:, ~written] == 0).all()


def test_chunked_prefill_through_append_is_one_paged_call():
    """Chunked prefill as a serving engine runs it: append the chunk's K/V to the
    paged cache, then one paged causal call over prefix + chunk (cached token j
    sits at position j).  Matches the oracle over the gathered keys, and the
    two-call (paged prefix + contiguous chunk) + LSE merge path."""
    prefix, chunk, hq, hkv, d = [100, 300], [150, 64], 16, 2, 128
    table, num_pages, kc0, vc0, kn, vn, pos, slots = _append_inputs(prefix, chunk, hkv, d, 550)
    T = kn.shape[0]
    q = synth.randn((T, hq, d), 556, 0.7071)
    posd, slotd = torch.from_numpy(pos).to(DEV), torch.from_numpy(slots).to(DEV)
    cu_q = torch.from_numpy(synth.cu_seqlens(chunk)).to(DEV)
    tabled = torch.from_numpy(table).to(DEV)
    kc, vc = kc0.to(DEV), vc0.to(DEV)
    qd = q.to(DEV)
    atc.rope_apply(qd, posd)
    kr = torch.empty((T, hkv, d), dtype=torch.bfloat16, device=DEV)
    atc.attn_kv_append_paged(kn.to(DEV), vn.to(DEV), posd, slotd, kc, vc, k_rot_out=kr)
    out = torch.empty((T, hq, d), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((T, hq), dtype=torch.float32, device=DEV)
    full = torch.tensor([p + c for p, c in zip(prefix, chunk)], dtype=torch.int32, device=DEV)
    atc.attn_prefill(qd, kc, vc, out, lse, cu_q, posd, max(chunk), page_table=tabled, k_lens=full,
                     num_pages=num_pages)
    # the same through the two-call path: paged prefix only, then the contiguous chunk, then a merge
    po = torch.empty((2, T, hq, d), dtype=torch.float32, device=DEV)
    pl = torch.empty((2, T, hq), dtype=torch.float32, device=DEV)
    pre = torch.tensor(prefix, dtype=torch.int32, device=DEV)
    atc.attn_prefill(qd, kc, vc, po[0], pl[0], cu_q, posd, max(chunk), page_table=tabled, k_lens=pre,
                     num_pages=num_pages)
    atc.attn_prefill(qd, kr, vn.to(DEV), po[1], pl[1], cu_q, posd, max(chunk), cu_k=cu_q, k_pos=posd)
    out2 = torch.empty_like(out)
    lse2 = torch.empty_like(lse)
    atc.attn_lse_merge(po, pl, out2, lse2)
    atc.attn_device_status()
    # oracle: the appended cache (oracle's own append), gathered in logical order
    wk, wv, _ = oracle.kv_append(synth.as_f64(kn), synth.as_f64(vn), pos, slots, synth.as_f64(kc0),
                                 synth.as_f64(vc0))
    qr = rotated_bf16(q, pos)
    want_o = np.empty((T, hq, d))
    want_l = np.empty((T, hq))
    o0 = 0
    for b, (p, c) in enumerate(zip(prefix, chunk)):
        K = np.stack([oracle.gather_pages(wk, table, num_pages, g, b, p + c) for g in range(hkv)], 1)
        V = np.stack([oracle.gather_pages(wv, table, num_pages, g, b, p + c) for g in range(hkv)], 1)
        o, l = oracle.attention(qr[o0:o0 + c], np.zeros(c, np.int32), pos[o0:o0 + c], K, V, [0, p + c],
                                np.arange(p + c, dtype=np.int32), d ** -0.5)
        want_o[o0:o0 + c], want_l[o0:o0 + c] = o, l
        o0 += c
    check(out, lse, want_o, want_l, what="append + one paged call")
    check(out2, lse2, want_o, want_l, what="two calls + merge")


def _growing_decode_case(splits, int8, seed, sign=1.0):
    """Decode inputs whose scores rise along each request's context at a rate
    set per query head: cached key j (logical, through the shuffled page table)
    is noise + (j / 64) u and query head h is noise + a_h u (u all ones, a_h =
    0.15 (h mod 8)), so the heads' scores grow by about 11.3 a_h per 64-token
    page -- the row max moves page after page in the steep heads and hardly in
    the flat ones.  The query is used as given (no RoPE)."""
    ctx = [700, 2049, 130, 1]
    wl = synth.Decode("decode growing", batch=len(ctx), ctx_lo=0, ctx_hi=0, hq=16, hkv=2, d=128, splits=splits,
                      seed=seed, ctx_fixed=ctx, int8=int8)
    inp = wl.make()
    table = inp["page_table"].numpy()
    npg = inp["num_pages"]
    logical = np.full((npg, 64), -1.0)
    for b, c in enumerate(ctx):
        j = np.arange(c)
        logical[table[b, j // 64], j % 64] = j
    ramp = sign * torch.from_numpy(np.where(logical >= 0, logical / 64.0, 0.0)).float()[None, :, :, None]
    k = synth.randn((2, npg, 64, 128), seed + 1, 0.3).float() + ramp
    a = (torch.arange(16) % 8).float()[None, :, None] * 0.15
    inp["q"] = (synth.randn((len(ctx), 16, 128), seed + 2, 0.3).float() + a).to(torch.bfloat16)
    if int8:  # symmetric int8 codes of the keys, one fp32 scale per row
        amax = k.abs().amax(-1)
        sc = (amax / 127.0).float()
        inp["k_cache"] = torch.round(k / sc[..., None]).clamp(-127, 127).to(torch.int8)
        inp["k_scale"] = sc
    else:
        inp["k_cache"] = k.to(torch.bfloat16)
    return wl, inp


@pytest.mark.parametrize("sign", [1.0, -1.0])
@pytest.mark.parametrize("int8", [False, True])
@pytest.mark.parametrize("splits", [1, 16])
def test_decode_scores_growing_along_the_context(splits, int8, sign):
    """Split-KV decode with row maxima that move on every page in the steep
    heads, over a bf16 and an INT8 cache, against the oracle (on the cache's
    exact values) at the bf16 tolerances; the merge of the splits combines
    partials whose LSEs differ by hundreds."""
    wl, inp = _growing_decode_case(splits, int8, 580 + splits + 10 * int8, sign)
    g = {k: (t.to(DEV) if torch.is_tensor(t) else t) for k, t in inp.items()}
    po, pl = atc.decode_workspace(wl.batch, wl.hq, splits, wl.d, DEV)
    out = torch.empty((wl.batch, wl.hq, wl.d), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((wl.batch, wl.hq), dtype=torch.float32, device=DEV)
    if int8:
        atc.attn_decode_paged_int8(g["q"], g["k_cache"], g["v_cache"], g["k_scale"], g["v_scale"], g["page_table"],
                                   g["ctx_lens"], splits, po, pl, out, lse)
        kc = oracle.dequant_int8(inp["k_cache"].numpy(), inp["k_scale"].numpy())
        vc = oracle.dequant_int8(inp["v_cache"].numpy(), inp["v_scale"].numpy())
    else:
        atc.attn_decode_paged(g["q"], g["k_cache"], g["v_cache"], g["page_table"], g["ctx_lens"], splits, po, pl,
                              out, lse)
        kc, vc = synth.as_f64(inp["k_cache"]), synth.as_f64(inp["v_cache"])
    atc.attn_device_status()
    want_o, want_l = oracle.decode_paged(synth.as_f64(inp["q"]), kc, vc, inp["page_table"].numpy(),
                                         inp["ctx_lens"].numpy(), inp["num_pages"], wl.scale)
    if sign > 0:
        assert want_l[1, 7] - want_l[1, 0] > 100  # the steep heads' scores are far above the flat ones'
    check(out, lse, want_o, want_l, what=f"growing decode splits={splits} int8={int8} sign={sign}")


# ------------------------------------------------------------------ decode over an INT8 cache

def _decode_int8(wl, inp, splits):
    g = {k: (t.to(DEV) if torch.is_tensor(t) else t) for k, t in inp.items()}
    q = g["q"].clone()
    atc.rope_apply(q, g["q_pos"])
    po, pl = atc.decode_workspace(wl.batch, wl.hq, splits, wl.d, DEV)
    out = torch.empty((wl.batch, wl.hq, wl.d), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((wl.batch, wl.hq), dtype=torch.float32, device=DEV)
    atc.attn_decode_paged_int8(q, g["k_cache"], g["v_cache"], g["k_scale"], g["v_scale"], g["page_table"],
                               g["ctx_lens"], splits, po, pl, out, lse)
    return out, lse


def _decode_int8_oracle(wl, inp):
    """The oracle's decode over the exact cache values code * scale."""
    qr = rotated_bf16(inp["q"], inp["q_pos"].numpy())
    kc = oracle.dequant_int8(inp["k_cache"].numpy(), inp["k_scale"].numpy())
    vc = oracle.dequant_int8(inp["v_cache"].numpy(), inp["v_scale"].numpy())
    return oracle.decode_paged(qr, kc, vc, inp["page_table"].numpy(), inp["ctx_lens"].numpy(), inp["num_pages"],
                               wl.scale)


@pytest.mark.parametrize("splits", [1, 4, 16])
def test_decode_int8_matches_oracle(splits):
    ctx = [1, 63, 64, 65, 700, 2049, 130, 0]
    wl = synth.Decode("decode int8 small", batch=len(ctx), ctx_lo=0, ctx_hi=0, hq=16, hkv=2, d=128, splits=splits,
                      seed=560 + splits, ctx_fixed=ctx, int8=True)
    inp = wl.make()
    out, lse = _decode_int8(wl, inp, splits)
    atc.attn_device_status()
    want_o, want_l = _decode_int8_oracle(wl, inp)
    check(out, lse, want_o, want_l, what=f"int8 decode splits={splits}")
    assert torch.all(out[-1] == 0) and torch.all(lse[-1] == -math.inf)  # empty context


def test_decode_int8_64_8_heads_long_contexts():
    ctx = [9000, 131, 4097]
    wl = synth.Decode("decode int8 64/8", batch=3, ctx_lo=0, ctx_hi=0, hq=64, hkv=8, d=128, splits=16, seed=570,
                      ctx_fixed=ctx, int8=True)
    inp = wl.make()
    out, lse = _decode_int8(wl, inp, 16)
    atc.attn_device_status()
    want_o, want_l = _decode_int8_oracle(wl, inp)
    check(out, lse, want_o, want_l, what="int8 decode 64/8")


def test_decode_int8_power_of_two_scales_match_bf16_decode():
    """With every scale 2^-6 the cached values code / 64 are exact in bf16 (at most
    8 significant bits): the INT8 path and the bf16 path decode the same numbers."""
    ctx = [300, 77]
    wl = synth.Decode("decode int8 pow2", batch=2, ctx_lo=0, ctx_hi=0, hq=16, hkv=2, d=128, splits=4, seed=580,
                      ctx_fixed=ctx, int8=True)
    inp = wl.make()
    inp["k_scale"] = torch.full_like(inp["k_scale"], 2.0 ** -6)
    inp["v_scale"] = torch.full_like(inp["v_scale"], 2.0 ** -6)
    o8, l8 = _decode_int8(wl, inp, 4)
    bf = dict(inp, k_cache=(inp["k_cache"].float() * 2.0 ** -6).to(torch.bfloat16),
              v_cache=(inp["v_cache"].float() * 2.0 ** -6).to(torch.bfloat16))
    assert torch.equal(bf["k_cache"].float(), inp["k_cache"].float() / 64.0)  # exact
    o16, l16, _, _ = _decode(wl, bf, 4)
    atc.attn_device_status()
    check(o8, l8, o16.float().cpu().numpy(), l16.cpu().numpy(), what="int8 vs bf16 path on code / 64")


def test_decode_int8_value_beyond_fp16_is_reported():
    """A query element beyond the fp16 range is caught on the device and reported."""
    ctx = [100]
    wl = synth.Decode("decode int8 range", batch=1, ctx_lo=0, ctx_hi=0, hq=8, hkv=1, d=128, splits=2, seed=590,
                      ctx_fixed=ctx, int8=True)
    inp = wl.make()
    g = {k: (t.to(DEV) if torch.is_tensor(t) else t) for k, t in inp.items()}
    q = g["q"].clone()
    q[0, 3, 17] = 1.0e6
    po, pl = atc.decode_workspace(1, 8, 2, 128, DEV)
    atc.attn_decode_paged_int8(q, g["k_cache"], g["v_cache"], g["k_scale"], g["v_scale"], g["page_table"],
                               g["ctx_lens"], 2, po, pl)
    with pytest.raises(atc.AttnError) as e:
        atc.attn_device_status(clear=True)
    assert e.value.status == 6
    atc.attn_device_status(clear=True)


# ------------------------------------------------------------------ query RoPE fused into prefill

def test_rope_table_matches_the_angles():
    T, d = 700, 128
    pos = np.sort(np.random.default_rng(4).integers(0, 131072, T)).astype(np.int32)
    pos[:3] = [0, 1, 131071]
    tab = atc.rope_table(torch.from_numpy(pos).to(DEV), d).cpu().numpy().astype(np.float64)
    ang = pos[:, None].astype(np.float64) * (10000.0 ** (-2.0 * np.arange(d // 2) / d))[None, :]
    assert np.abs(tab[..., 0] - np.cos(ang)).max() < 2e-6
    assert np.abs(tab[..., 1] - np.sin(ang)).max() < 2e-6
    np.testing.assert_array_equal(tab[0, :, 0], 1.0)   # position 0: cos 1, sin 0
    np.testing.assert_array_equal(tab[0, :, 1], 0.0)


@pytest.mark.parametrize("lens,hq,hkv,starts", CASES)
def test_prefill_fused_query_rope_equals_rope_apply_then_prefill(lens, hq, hkv, starts):
    """The kernel rotates the unrotated queries itself, with rope_apply's cos/sin
    and rounding: outputs and LSE are bit-identical, and q is left unrotated."""
    q, k, v, pos, cu = _bf16_case(lens, hq, hkv, starts, 600 + hq + len(lens))
    out_ref, lse_ref = _run_prefill(q, k, v, pos, cu, lens)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    posd, cud = torch.from_numpy(pos).to(DEV), torch.from_numpy(cu).to(DEV)
    atc.rope_apply(kd, posd)
    tab = atc.rope_table(posd, q.shape[2])
    out = torch.full(q.shape, float("nan"), dtype=q.dtype, device=DEV)
    lse = torch.full(q.shape[:2], float("nan"), dtype=torch.float32, device=DEV)
    atc.attn_prefill(qd, kd, vd, out, lse, cud, posd, max(lens), cu_k=cud, k_pos=posd, q_rope_cs=tab)
    atc.attn_device_status()
    assert torch.equal(out, out_ref) and torch.equal(lse, lse_ref)
    assert torch.equal(qd.cpu(), q)  # the caller's q is not modified
    want_o, want_l = _oracle_prefill(q, k, v, pos, cu, lens, 128 ** -0.5)
    check(out, lse, want_o, want_l, what=f"fused query RoPE {lens}")


def test_prefill_fused_query_rope_head_slices_and_paged_source():
    """Head slices of the fused call equal the all-heads call; the paged source
    (chunk over a cached prefix) takes the fused rotation too."""
    lens = [600]
    q, k, v, pos, cu = _bf16_case(lens, 64, 8, [0], 610)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    posd, cud = torch.from_numpy(pos).to(DEV), torch.from_numpy(cu).to(DEV)
    atc.rope_apply(kd, posd)
    tab = atc.rope_table(posd, 128)
    full_o, full_l = atc.prefill(qd, kd, vd, cud, posd, 600, cu_k=cud, k_pos=posd, q_rope_cs=tab)
    for lo, hi in ((16, 32), (56, 64)):
        o, l = atc.prefill(qd, kd, vd, cud, posd, 600, cu_k=cud, k_pos=posd, q_rope_cs=tab, h_lo=lo, h_hi=hi)
        assert torch.equal(o[:, lo:hi], full_o[:, lo:hi]) and torch.equal(l[:, lo:hi], full_l[:, lo:hi])
    # paged: the chunk's queries over a cache that holds prefix + chunk
    prefix, chunk, hq2, hkv2, d = [100, 300], [150, 64], 16, 2, 128
    table, num_pages, kc0, vc0, kn, vn, ppos, slots = _append_inputs(prefix, chunk, hkv2, d, 620)
    T = kn.shape[0]
    q2 = synth.randn((T, hq2, d), 626, 0.7071).to(DEV)
    pposd = torch.from_numpy(ppos).to(DEV)
    kc, vc = kc0.to(DEV), vc0.to(DEV)
    atc.attn_kv_append_paged(kn.to(DEV), vn.to(DEV), pposd, torch.from_numpy(slots).to(DEV), kc, vc)
    cu_q = torch.from_numpy(synth.cu_seqlens(chunk)).to(DEV)
    klens = torch.tensor([p + c for p, c in zip(prefix, chunk)], dtype=torch.int32, device=DEV)
    tabled = torch.from_numpy(table).to(DEV)
    o_f, l_f = atc.prefill(q2, kc, vc, cu_q, pposd, max(chunk), page_table=tabled, k_lens=klens,
                           num_pages=num_pages, q_rope_cs=atc.rope_table(pposd, d))
    q2r = q2.clone()
    atc.rope_apply(q2r, pposd)
    o_r, l_r = atc.prefill(q2r, kc, vc, cu_q, pposd, max(chunk), page_table=tabled, k_lens=klens,
                           num_pages=num_pages)
    atc.attn_device_status()
    assert torch.equal(o_f, o_r) and torch.equal(l_f, l_r)


def test_prefill_fused_query_rope_needs_the_tensor_core_path():
    q = torch.zeros((8, 8, 64), dtype=torch.float32, device=DEV)
    pos = torch.arange(8, dtype=torch.int32, device=DEV)
    cu = torch.tensor([0, 8], dtype=torch.int32, device=DEV)
    with pytest.raises(atc.AttnError) as e:
        atc.prefill(q, q[:, :2].contiguous(), q[:, :2].contiguous(), cu, pos, 8, cu_k=cu, k_pos=pos,
                    q_rope_cs=atc.rope_table(pos, 64))
    assert e.value.status == 4


# ------------------------------------------------------------------ append into an INT8 cache

def _int8_cache(hkv, num_pages, seed):
    kc = synth.randint8((hkv, num_pages, 64, 128), seed)
    vc = synth.randint8((hkv, num_pages, 64, 128), seed + 1)
    ks = synth.uniform((hkv, num_pages, 64), seed + 2, 0.01, 0.02)
    vs = synth.uniform((hkv, num_pages, 64), seed + 3, 0.01, 0.02)
    return kc, vc, ks, vs


@pytest.mark.parametrize("rotate", [False, True])
def test_kv_append_int8_matches_oracle(rotate):
    """Codes and scales as the oracle decides them in fp32.  Unrotated rows and all
    value rows are bit-exact; rotated key codes follow the bf16 rotation, which
    may differ from the oracle's by one ulp in rare elements, so their codes are
    within one step and almost all equal.  Other cache rows stay untouched."""
    hkv, d = 8, 128
    table, num_pages, _, _, kn, vn, pos, slots = _append_inputs([64, 130, 0], [100, 1, 260], hkv, d, 640, pad=3)
    kc0, vc0, ks0, vs0 = _int8_cache(hkv, num_pages, 650)
    kc, vc, ks, vs = kc0.to(DEV), vc0.to(DEV), ks0.to(DEV), vs0.to(DEV)
    base = 10000.0 if rotate else 0.0
    ko = torch.empty(kn.shape, dtype=torch.bfloat16, device=DEV)
    atc.attn_kv_append_paged_int8(kn.to(DEV), vn.to(DEV), torch.from_numpy(pos).to(DEV),
                                  torch.from_numpy(slots).to(DEV), kc, vc, ks, vs, k_rot_out=ko, base=base)
    atc.attn_device_status()
    wkc, wvc, wks, wvs, bad = oracle.kv_append_int8(synth.as_f64(kn), synth.as_f64(vn), pos, slots, kc0.numpy(),
                                                    vc0.numpy(), ks0.numpy(), vs0.numpy(), base=base)
    assert bad == 0
    np.testing.assert_array_equal(vc.cpu().numpy(), wvc)
    np.testing.assert_array_equal(vs.cpu().numpy(), wvs)
    gk, gs = kc.cpu().numpy().astype(np.int32), ks.cpu().numpy()
    if not rotate:
        np.testing.assert_array_equal(gk, wkc)
        np.testing.assert_array_equal(gs, wks)
        assert torch.equal(ko[torch.from_numpy(slots >= 0).to(DEV)], kn.to(DEV)[torch.from_numpy(slots >= 0).to(DEV)])
    else:
        diff = np.abs(gk - wkc.astype(np.int32))
        assert diff.max() <= 1 and (diff > 0).mean() < 0.01
        assert np.allclose(gs, wks, rtol=2 ** -7, atol=0)
        # the bf16 rotated keys it also wrote are rope_apply's, bit for bit
        kr = kn.to(DEV).clone()
        atc.rope_apply(kr, torch.from_numpy(pos).to(DEV))
        valid = torch.from_numpy(slots >= 0).to(DEV)
        assert torch.equal(ko[valid], kr[valid])


@pytest.mark.parametrize("hkv", [8, 3, 9, 40, 96])
def test_kv_append_int8_many_groups_matches_oracle(hkv):
    """A chunk long enough that the append's blocks each take many groups of
    tokens in turn (so each staging buffer is refilled several times), at head
    counts whose groups hold 4, 10 and 1 token(s), and at one above what the
    staged path takes.  The slots are a shuffled set of cache rows, with two
    padding tokens (-1) and one slot past the cache in the middle. The bad slot
    is recorded and skipped, and every other row is written as the oracle writes
    it (keys rotated)."""
    d = 128
    tokens = {8: 20011, 3: 40003, 9: 30011, 40: 6007, 96: 2003}[hkv]
    num_pages = (tokens + 63) // 64 + 2
    rows = num_pages * 64
    table, _ = synth.shuffled_page_table([rows], 700 + hkv)
    slots = (table[0][np.arange(tokens) // 64] * 64 + np.arange(tokens) % 64).astype(np.int32)
    slots[tokens // 3] = rows          # past the cache
    slots[[5, tokens - 2]] = -1        # padding
    pos = np.arange(tokens, dtype=np.int32) + 1000
    kn = synth.randn((tokens, hkv, d), 710 + hkv, 0.7071)
    vn = synth.randn((tokens, hkv, d), 720 + hkv, 0.7071)
    kc0, vc0, ks0, vs0 = _int8_cache(hkv, num_pages, 730 + hkv)
    kc, vc, ks, vs = kc0.to(DEV), vc0.to(DEV), ks0.to(DEV), vs0.to(DEV)
    ko = torch.empty(kn.shape, dtype=torch.bfloat16, device=DEV)
    atc.attn_kv_append_paged_int8(kn.to(DEV), vn.to(DEV), torch.from_numpy(pos).to(DEV),
                                  torch.from_numpy(slots).to(DEV), kc, vc, ks, vs, k_rot_out=ko, base=10000.0)
    with pytest.raises(atc.AttnError) as e:
        atc.attn_device_status(clear=True)
    assert e.value.status == 6
    atc.attn_device_status(clear=True)
    wkc, wvc, wks, wvs, bad = oracle.kv_append_int8(synth.as_f64(kn), synth.as_f64(vn), pos, slots, kc0.numpy(),
                                                    vc0.numpy(), ks0.numpy(), vs0.numpy(), base=10000.0)
    assert bad == 1
    np.testing.assert_array_equal(vc.cpu().numpy(), wvc)
    np.testing.assert_array_equal(vs.cpu().numpy(), wvs)
    diff = np.abs(kc.cpu().numpy().astype(np.int32) - wkc.astype(np.int32))
    assert diff.max() <= 1 and (diff > 0).mean() < 0.01
    assert np.allclose(ks.cpu().numpy(), wks, rtol=2 ** -7, atol=0)
    valid = torch.from_numpy((slots >= 0) & (slots < rows)).to(DEV)
    kr = kn.to(DEV).clone()
    atc.rope_apply(kr, torch.from_numpy(pos).to(DEV))
    assert torch.equal(ko[valid], kr[valid])


def test_kv_append_int8_row_scales_across_the_bf16_range():
    """Rows whose max |x| runs over the whole bf16 range (each token's rows
    scaled by 2^e, e = -133 .. 125, plus an all-zero token), unrotated: every
    scale is max|x| / 127 rounded in fp32, and every code the fp32 quotient
    rounded, bit for bit as the oracle decides them -- through both the
    one-correction division and the full one, for scales and for codes."""
    hkv, d = 2, 128
    exps = np.arange(-133, 126)
    tokens = len(exps) + 1
    num_pages = (tokens + 63) // 64
    slots = np.arange(tokens, dtype=np.int32)
    scale = torch.from_numpy(np.concatenate([np.exp2(exps.astype(np.float64)), [0.0]]).astype(np.float32))
    kn = (synth.randn((tokens, hkv, d), 760, 1.0).float() * scale[:, None, None]).to(torch.bfloat16)
    vn = (synth.randn((tokens, hkv, d), 761, 1.0).float() * scale[:, None, None]).to(torch.bfloat16)
    assert torch.isfinite(kn.float()).all() and torch.isfinite(vn.float()).all()
    kc0, vc0, ks0, vs0 = _int8_cache(hkv, num_pages, 770)
    kc, vc, ks, vs = kc0.to(DEV), vc0.to(DEV), ks0.to(DEV), vs0.to(DEV)
    atc.attn_kv_append_paged_int8(kn.to(DEV), vn.to(DEV), None, torch.from_numpy(slots).to(DEV), kc, vc, ks, vs,
                                  base=0.0)
    atc.attn_device_status()
    wkc, wvc, wks, wvs, bad = oracle.kv_append_int8(synth.as_f64(kn), synth.as_f64(vn), np.zeros(tokens, np.int32),
                                                    slots, kc0.numpy(), vc0.numpy(), ks0.numpy(), vs0.numpy(),
                                                    base=0.0)
    assert bad == 0
    np.testing.assert_array_equal(kc.cpu().numpy(), wkc)
    np.testing.assert_array_equal(vc.cpu().numpy(), wvc)
    np.testing.assert_array_equal(ks.cpu().numpy(), wks)
    np.testing.assert_array_equal(vs.cpu().numpy(), wvs)
    assert (wks.reshape(hkv, -1)[:, tokens - 1] == 0).all()
    assert wks.reshape(hkv, -1)[:, 0].max() < 2.0 ** -90 < wks.reshape(hkv, -1)[:, tokens - 2].min()


def test_decode_over_int8_append_matches_oracle():
    """Serving flow on an INT8 cache: the chunk appended (rotated, quantised), then
    the decode of the last position of each request over the whole cache."""
    hkv, hq, d = 2, 16, 128
    prefix, chunk = [300, 64], [40, 1]
    table, num_pages, _, _, kn, vn, pos, slots = _append_inputs(prefix, chunk, hkv, d, 660)
    kc0, vc0, ks0, vs0 = _int8_cache(hkv, num_pages, 670)
    kc, vc, ks, vs = kc0.to(DEV), vc0.to(DEV), ks0.to(DEV), vs0.to(DEV)
    atc.attn_kv_append_paged_int8(kn.to(DEV), vn.to(DEV), torch.from_numpy(pos).to(DEV),
                                  torch.from_numpy(slots).to(DEV), kc, vc, ks, vs)
    ctx = np.array([p + c for p, c in zip(prefix, chunk)], np.int32)
    q = synth.randn((2, hq, d), 680, 0.7071)
    qpos = (ctx - 1).astype(np.int32)
    qr = q.to(DEV).clone()
    atc.rope_apply(qr, torch.from_numpy(qpos).to(DEV))
    po, pl = atc.decode_workspace(2, hq, 4, d, DEV)
    out = torch.empty((2, hq, d), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((2, hq), dtype=torch.float32, device=DEV)
    atc.attn_decode_paged_int8(qr, kc, vc, ks, vs, torch.from_numpy(table).to(DEV), torch.from_numpy(ctx).to(DEV),
                               4, po, pl, out, lse)
    atc.attn_device_status()
    wkc, wvc, wks, wvs, _ = oracle.kv_append_int8(synth.as_f64(kn), synth.as_f64(vn), pos, slots, kc0.numpy(),
                                                  vc0.numpy(), ks0.numpy(), vs0.numpy())
    want_o, want_l = oracle.decode_paged(rotated_bf16(q, qpos), oracle.dequant_int8(wkc, wks),
                                         oracle.dequant_int8(wvc, wvs), table, ctx, num_pages, d ** -0.5)
    check(out, lse, want_o, want_l, what="decode over the INT8 append")


# ------------------------------------------------------------------ FP8 quantisation

def test_quant_fp8_rows_and_heads_match_oracle():
    """e4m3 codes and fp32 scales exactly as the oracle decides them in fp32, for
    one group per (token, head) row, per head, and per head with the transposed
    [heads][128][t_stride] layout of the values."""
    T, H = 333, 8
    x = synth.randn((T, H, 128), 700, 0.7071)
    x[5, 3] = 0                                  # an all-zero row
    xd = x.to(DEV)
    c_r, s_r = atc.quant_fp8_rows(xd)
    c_h, s_h = atc.quant_fp8_heads(xd)
    c_t, s_t = atc.quant_fp8_heads(xd, transposed=True)
    atc.attn_device_status()
    xf = synth.as_f64(x)
    want_r, ws_r = oracle.quant_e4m3(xf, [0, 1])
    want_h, ws_h = oracle.quant_e4m3(xf, [1])
    np.testing.assert_array_equal(c_r.float().cpu().numpy(), want_r)
    np.testing.assert_array_equal(s_r.cpu().numpy(), ws_r)
    np.testing.assert_array_equal(c_h.float().cpu().numpy(), want_h)
    np.testing.assert_array_equal(s_h.cpu().numpy(), ws_h)
    np.testing.assert_array_equal(s_t.cpu().numpy(), ws_h)
    assert c_t.shape == (H, 128, 336)
    np.testing.assert_array_equal(c_t.float().cpu().numpy()[:, :, :T], np.transpose(want_h, (1, 2, 0)))
    assert (c_t.view(torch.uint8)[:, :, T:] == 0).all()   # the padding columns are zero codes




def test_quant_fp8_codes_over_group_maxima_across_the_fp32_range():
    """e4m3 codes bit-exact with the oracle's fp32 division x / scale over group
    maxima spread across 2^-130..2^127 (the three-instruction division serves
    scales from 2^-90 up, the full division below), with every other value a
    random bf16 number no larger than the row's maximum, some of them subnormal."""
    rows = 4096
    g = torch.Generator().manual_seed(740)
    expo = torch.randint(-130, 127, (rows, 1), generator=g).float()
    amax = (torch.rand((rows, 1), generator=g) + 1.0) * torch.pow(2.0, expo)
    frac = torch.rand((rows, 128), generator=g) * 2 - 1
    frac[:, ::7] *= torch.pow(2.0, -torch.randint(0, 40, (rows, 19), generator=g).float())
    x = (frac * amax).to(torch.bfloat16)
    x[:, 0] = amax[:, 0].to(torch.bfloat16)
    x = x.view(rows // 8, 8, 128)
    codes, scales = atc.quant_fp8_rows(x.to(DEV))
    atc.attn_device_status()
    want, wsc = oracle.quant_e4m3(synth.as_f64(x), [0, 1])
    np.testing.assert_array_equal(scales.cpu().numpy(), wsc)
    np.testing.assert_array_equal(codes.float().cpu().numpy(), want)

def test_rope_quant_fp8_equals_rope_then_quant_and_matches_oracle():
    """The fused RoPE + e4m3 quantisation equals rope_apply followed by
    quant_fp8_rows / quant_fp8_heads bit for bit, leaves its input alone, and is
    within one e4m3 step of the oracle's quantisation of its own rotation (the
    rotations differ by at most one bf16 ulp in under 1% of elements)."""
    T, H = 301, 8
    x = synth.randn((T, H, 128), 720, 0.7071)
    pos = synth.positions([T], [99000])
    xd, posd = x.to(DEV), torch.from_numpy(pos).to(DEV)
    x0 = xd.clone()
    c_r, s_r = atc.rope_quant_fp8_rows(xd, posd)
    c_h, s_h = atc.rope_quant_fp8_heads(xd, posd)
    atc.attn_device_status()
    assert torch.equal(xd, x0)
    xr = xd.clone()
    atc.rope_apply(xr, posd)
    w_r, ws_r = atc.quant_fp8_rows(xr)
    w_h, ws_h = atc.quant_fp8_heads(xr)
    assert torch.equal(c_r.view(torch.uint8), w_r.view(torch.uint8)) and torch.equal(s_r, ws_r)
    assert torch.equal(c_h.view(torch.uint8), w_h.view(torch.uint8)) and torch.equal(s_h, ws_h)
    rot = rotated_bf16(x, pos)
    for (codes, sc), axes in (((c_r, s_r), [0, 1]), ((c_h, s_h), [1])):
        want, wsc = oracle.quant_e4m3(rot, axes)
        got_sc = sc.cpu().numpy().astype(np.float64)
        np.testing.assert_allclose(got_sc, wsc, rtol=2.0 ** -7)
        shape = (T, H, 1) if axes == [0, 1] else (1, H, 1)
        got_v = codes.float().cpu().numpy() * got_sc.reshape(shape)
        want_v = want * wsc.astype(np.float64).reshape(shape)
        step = 2.0 ** -3 * np.maximum(np.abs(got_v), np.abs(want_v)) + 2.0 ** -9 * wsc.reshape(shape)
        assert (np.abs(got_v - want_v) <= step).all()
        assert (codes.float().cpu().numpy() != want).mean() < 0.03


# ------------------------------------------------------------------ FP8 (e4m3) prefill

def _fp8_case(lens, hq, hkv, starts, seed, zero_k=False):
    """Already-rotated bf16 Q/K/V; every sequence but the last is a multiple of 16
    tokens long, so every key sequence starts on a 16-token boundary."""
    T = sum(lens)
    q = synth.randn((T, hq, 128), seed, 0.7071)
    k = torch.zeros((T, hkv, 128), dtype=torch.bfloat16) if zero_k else synth.randn((T, hkv, 128), seed + 1, 0.7071)
    v = synth.randn((T, hkv, 128), seed + 2, 0.7071)
    return q, k, v, synth.positions(lens, starts), synth.cu_seqlens(lens)


def _run_fp8(q, k, v, pos, cu, lens, causal=True, h_lo=0, h_hi=None, out_dtype=torch.bfloat16):
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    cq, sq = atc.quant_fp8_rows(qd)
    ck, sk = atc.quant_fp8_heads(kd)
    cv, sv = atc.quant_fp8_heads(vd, transposed=True)
    posd, cud = torch.from_numpy(pos).to(DEV), torch.from_numpy(cu).to(DEV)
    out = torch.full(q.shape, float("nan"), dtype=out_dtype, device=DEV)
    lse = torch.full(q.shape[:2], float("nan"), dtype=torch.float32, device=DEV)
    atc.attn_prefill_fp8(cq, sq, ck, sk, cv, sv, out, lse, cud, posd, max(lens), cud, posd, h_lo=h_lo, h_hi=h_hi,
                         causal=causal)
    atc.attn_device_status()
    return out, lse


def _fp8_oracle(q, k, v, pos, cu, lens, causal=True, h_lo=0, h_hi=None):
    """Attention in fp64 over the values the e4m3 codes stand for (code x group scale)."""
    cq, sq = oracle.quant_e4m3(synth.as_f64(q), [0, 1])
    ck, sk = oracle.quant_e4m3(synth.as_f64(k), [1])
    cv, sv = oracle.quant_e4m3(synth.as_f64(v), [1])
    qh = cq * sq.astype(np.float64)[:, :, None]
    kh = ck * sk.astype(np.float64)[None, :, None]
    vh = cv * sv.astype(np.float64)[None, :, None]
    o, l = oracle.attention(qh, seq_ids(lens), pos, kh, vh, cu, pos, 128 ** -0.5, causal=causal, h_lo=h_lo,
                            h_hi=h_hi)
    return o, l, vh


# The FP8 path rounds each softmax weight p (0 <= p <= 256 with the lazy
# rescale) to e4m3 before P V, while l sums the unrounded weights.  A normal
# e4m3 value carries relative error <= 2^-4, so |dO| <= 2^-4 max|v| per row plus
# at most 2^-10 per subnormal weight (p < 2^-6), which l >= 1 divides.  The
# rounding errors are zero-mean and independent: with RMS relative error about
# 2^-4 / sqrt(3) and softmax rows over n ~ U[1, N] keys of std 0.71, the mean
# |dO| is about 0.8 * 0.036 * 0.71 * 2 / sqrt(N), 2e-3 at N = 300; the mean
# bound below is twice that, and the max bound adds the subnormal term for the
# few keys a row can see with non-negligible weight.  The scores are exact
# products of e4m3 codes summed in fp32, so the LSE bound stays 1e-3.
FP8_MEAN = 4e-3


def _fp8_max_tol(vh):
    return 2.0 ** -4 * np.abs(vh).max() + 32 * 2.0 ** -10 * np.abs(vh).max()


FP8_CASES = [
    ([300], 16, 2, [0]),                      # several tiles and a ragged tail
    ([256, 144, 512, 1], 16, 2, [0, 5, 100000, 7]),  # varlen, offsets, a 1-token sequence
    ([160, 333], 8, 1, [0, 0]),               # MQA, ragged last sequence
    ([704], 64, 8, [0]),                      # the 64/8 head layout
]


@pytest.mark.parametrize("lens,hq,hkv,starts", FP8_CASES)
def test_prefill_fp8_matches_oracle_on_dequantised_inputs(lens, hq, hkv, starts):
    q, k, v, pos, cu = _fp8_case(lens, hq, hkv, starts, 900 + hq + len(lens))
    out, lse = _run_fp8(q, k, v, pos, cu, lens)
    want_o, want_l, vh = _fp8_oracle(q, k, v, pos, cu, lens)
    check(out, lse, want_o, want_l, tol_max=_fp8_max_tol(vh), tol_mean=FP8_MEAN, what=f"fp8 {lens}")


def test_prefill_fp8_uniform_weights_are_exact():
    """Zero keys make every visible score 0, so each weight is exactly 1 in e4m3 and
    O is the plain mean of the visible dequantised values: the P V side (V^T
    layout, value scale, masking, the e4m3 P tile) is checked to fp32 rounding."""
    lens = [256, 77]
    q, k, v, pos, cu = _fp8_case(lens, 16, 2, [0, 3], 910, zero_k=True)
    out, lse = _run_fp8(q, k, v, pos, cu, lens, out_dtype=torch.float32)
    want_o, want_l, vh = _fp8_oracle(q, k, v, pos, cu, lens)
    check(out, lse, want_o, want_l, tol_max=1e-5, tol_mean=1e-6, tol_lse=1e-5, what="fp8 uniform")


def test_prefill_fp8_non_causal_head_slice_fp32_out():
    lens = [192, 200]
    q, k, v, pos, cu = _fp8_case(lens, 16, 2, [0, 0], 911)
    out, lse = _run_fp8(q, k, v, pos, cu, lens, causal=False, h_lo=8, h_hi=16, out_dtype=torch.float32)
    want_o, want_l, vh = _fp8_oracle(q, k, v, pos, cu, lens, causal=False, h_lo=8, h_hi=16)
    check(out[:, 8:], lse[:, 8:], want_o[:, 8:], want_l[:, 8:], tol_max=_fp8_max_tol(vh), tol_mean=FP8_MEAN,
          what="fp8 non-causal")
    assert torch.isnan(out[:, :8]).all()


def test_prefill_fp8_is_deterministic():
    lens = [1024, 320]
    q, k, v, pos, cu = _fp8_case(lens, 64, 8, [0, 9], 912)
    first = _run_fp8(q, k, v, pos, cu, lens)
    for _ in range(2):
        o, l = _run_fp8(q, k, v, pos, cu, lens)
        assert torch.equal(o, first[0]) and torch.equal(l, first[1])


def test_prefill_fp8_misaligned_key_sequence_is_reported():
    """A key sequence starting off a 16-token boundary is refused by its CTAs
    (recorded device error, nothing written); the aligned sequence is computed."""
    lens = [8, 200]
    q, k, v, pos, cu = _fp8_case(lens, 8, 1, [0, 0], 913)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    cq, sq = atc.quant_fp8_rows(qd)
    ck, sk = atc.quant_fp8_heads(kd)
    cv, sv = atc.quant_fp8_heads(vd, transposed=True)
    posd, cud = torch.from_numpy(pos).to(DEV), torch.from_numpy(cu).to(DEV)
    out = torch.full(q.shape, float("nan"), dtype=torch.bfloat16, device=DEV)
    atc.attn_prefill_fp8(cq, sq, ck, sk, cv, sv, out, None, cud, posd, 200, cud, posd)
    with pytest.raises(atc.AttnError) as e:
        atc.attn_device_status(clear=True)
    assert "0x204" in str(e.value)
    assert torch.isnan(out[8:].float()).all()
    assert not torch.isnan(out[:8].float()).any()


def test_prefill_fp8_zero_length_sequences_and_masked_rows():
    """Zero-length sequences in the batch, and queries placed before every key
    (no visible key: O = 0, LSE = -inf), on the e4m3 path."""
    lens = [0, 160, 0, 37]
    q, k, v, pos, cu = _fp8_case(lens, 8, 1, [0, 0, 0, 0], 914)
    out, lse = _run_fp8(q, k, v, pos, cu, lens)
    want_o, want_l, vh = _fp8_oracle(q, k, v, pos, cu, lens)
    check(out, lse, want_o, want_l, tol_max=_fp8_max_tol(vh), tol_mean=FP8_MEAN, what="fp8 zero-length")

    qd = synth.randn((10, 8, 128), 915, 0.7).to(DEV)
    kd = synth.randn((208, 1, 128), 916, 0.7).to(DEV)
    vd = synth.randn((208, 1, 128), 917, 0.7).to(DEV)
    cq, sq = atc.quant_fp8_rows(qd)
    ck, sk = atc.quant_fp8_heads(kd)
    cv, sv = atc.quant_fp8_heads(vd, transposed=True)
    qpos = torch.arange(10, dtype=torch.int32, device=DEV)
    kpos = torch.arange(50, 258, dtype=torch.int32, device=DEV)
    out = torch.full((10, 8, 128), float("nan"), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((10, 8), dtype=torch.float32, device=DEV)
    atc.attn_prefill_fp8(cq, sq, ck, sk, cv, sv, out, lse, torch.tensor([0, 10], dtype=torch.int32, device=DEV),
                         qpos, 10, torch.tensor([0, 208], dtype=torch.int32, device=DEV), kpos)
    atc.attn_device_status()
    assert torch.all(out == 0) and torch.all(lse == -math.inf)


@pytest.mark.parametrize("d", [64, 30])
def test_lse_merge_other_head_sizes(d):
    """Head sizes that take the general merge kernels: 64 (16-byte vectors, not
    the 128-wide kernel) and 30 (scalar), with an empty part and a row with none."""
    P, R, H = 3, 21, 5
    rng = np.random.default_rng(30 + d)
    po = rng.normal(0, 1, (P, R, H, d)).astype(np.float32)
    pl = rng.normal(0, 2, (P, R, H)).astype(np.float32)
    pl[1, :, 1] = -np.inf
    pl[:, 4, 3] = -np.inf
    want_o, want_l = oracle.lse_merge(po.astype(np.float64), pl.astype(np.float64))
    out = torch.empty((R, H, d), dtype=torch.float32, device=DEV)
    lse = torch.empty((R, H), dtype=torch.float32, device=DEV)
    atc.attn_lse_merge(torch.from_numpy(po).to(DEV), torch.from_numpy(pl).to(DEV), out, lse)
    check(out, lse, want_o, want_l, tol_max=1e-5, tol_mean=1e-6, tol_lse=1e-5, what=f"merge d={d}")
    assert torch.all(out[4, 3] == 0)


def test_paged_prefill_fp32_output_head_slice_matches_oracle():
    """The paged (prefix) source with fp32 output for query heads 8..15 only: the
    prefix part of chunked prefill on one rank of a head split."""
    prefix, chunk, B, hq, hkv = 300, 130, 2, 16, 2
    table, num_pages, kc, vc, q, k, v = _chunked_case(prefix, chunk, B, hq, hkv, 930)
    qpos = synth.positions([chunk] * B, [prefix] * B)
    qd = q.to(DEV)
    atc.rope_apply(qd, torch.from_numpy(qpos).to(DEV))
    out = torch.full((B * chunk, hq, 128), float("nan"), dtype=torch.float32, device=DEV)
    lse = torch.full((B * chunk, hq), float("nan"), dtype=torch.float32, device=DEV)
    atc.attn_prefill(qd, kc.to(DEV), vc.to(DEV), out, lse, torch.from_numpy(synth.cu_seqlens([chunk] * B)).to(DEV),
                     torch.from_numpy(qpos).to(DEV), chunk, page_table=torch.from_numpy(table).to(DEV),
                     k_lens=torch.full((B,), prefix, dtype=torch.int32, device=DEV), num_pages=num_pages,
                     h_lo=8, h_hi=16)
    atc.attn_device_status()
    qr = rotated_bf16(q, qpos)
    kcf, vcf = synth.as_f64(kc), synth.as_f64(vc)
    keys = [np.stack([oracle.gather_pages(kcf, table, num_pages, g, b, prefix) for g in range(hkv)], 1)
            for b in range(B)]
    vals = [np.stack([oracle.gather_pages(vcf, table, num_pages, g, b, prefix) for g in range(hkv)], 1)
            for b in range(B)]
    kpos = np.concatenate([np.arange(prefix, dtype=np.int32)] * B)
    want_o, want_l = oracle.attention(qr, seq_ids([chunk] * B), qpos, np.concatenate(keys), np.concatenate(vals),
                                      synth.cu_seqlens([prefix] * B), kpos, 128 ** -0.5, causal=False,
                                      h_lo=8, h_hi=16)
    check(out[:, 8:16], lse[:, 8:16], want_o[:, 8:16], want_l[:, 8:16], what="paged fp32 head slice")
    assert torch.isnan(out[:, :8]).all() and torch.isnan(lse[:, 8:16]).sum() == 0


# ------------------------------------------------------------------ key shards with position gaps

def _shard_case(T, hq, hkv, seed):
    q = synth.randn((T, hq, 128), seed, 0.7071)
    k = synth.randn((T, hkv, 128), seed + 1, 0.7071)
    v = synth.randn((T, hkv, 128), seed + 2, 0.7071)
    return q, k, v, np.arange(T, dtype=np.int32)


def _rows_call(fn, q, k, v, pos, qrows, krows, out_dtype=torch.float32):
    """One attn_prefill(-like) call of the queries `qrows` against the keys
    `krows` of one sequence (both sorted), at their absolute positions."""
    i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(DEV)
    qi, ki = torch.from_numpy(qrows).to(DEV), torch.from_numpy(krows).to(DEV)
    cu_q, cu_k = i32([0, len(qrows)]), i32([0, len(krows)])
    return fn(q[qi].contiguous(), k[ki].contiguous(), v[ki].contiguous(), cu_q, i32(pos[qrows]), len(qrows), cu_k,
              i32(pos[krows]), out_dtype)


def _bf16_call(q, k, v, cu_q, qpos, maxq, cu_k, kpos, out_dtype):
    out = torch.full(q.shape, float("nan"), dtype=out_dtype, device=DEV)
    lse = torch.full(q.shape[:2], float("nan"), dtype=torch.float32, device=DEV)
    atc.attn_prefill(q, k, v, out, lse, cu_q, qpos, maxq, cu_k=cu_k, k_pos=kpos)
    atc.attn_device_status()
    return out, lse


@pytest.mark.parametrize("kind,world", [("striped", 2), ("zigzag", 2), ("striped", 3), ("zigzag", 3)])
def test_prefill_tc_key_shards_with_position_gaps(kind, world):
    """Ring-attention steps (SGLang page, section 3.5): the queries of one rank's
    shard against the keys of every rank's shard, striped (token % N) or zigzag
    (blocks r and 2N-1-r of 2N).  Key positions jump inside 128-key tiles, so the
    kernel's extent search leaves its consecutive-position guess for the
    warp-wide search and the per-tile mask meets the gaps; some shard pairs leave
    rows with no visible key.  Every partial matches the oracle on the same rows
    and keys, and the shards' partials merged by attn_lse_merge match the oracle's
    unsplit result for those queries."""
    T = 2 * world * 300  # zigzag blocks of 300 rows: a gap falls inside a key tile
    q, k, v, pos = _shard_case(T, 16, 2, 1200 + world)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    posd = torch.from_numpy(pos).to(DEV)
    atc.rope_apply_qk(qd, kd, posd)
    qr, kr, vf = rotated_bf16(q, pos), rotated_bf16(k, pos), synth.as_f64(v)
    for rq in range(world):
        qrows = synth.shard_rows(T, world, rq, kind)
        po, pl = [], []
        for rk in range(world):
            krows = synth.shard_rows(T, world, rk, kind)
            o, l = _rows_call(_bf16_call, qd, kd, vd, pos, qrows, krows)
            wo, wl = oracle.attention(qr[qrows], np.zeros(len(qrows), np.int32), pos[qrows], kr[krows], vf[krows],
                                      [0, len(krows)], pos[krows], 128 ** -0.5)
            check(o, l, wo, wl, what=f"{kind} q{rq} k{rk}")
            po.append(o)
            pl.append(l)
        out = torch.empty_like(po[0])
        lse = torch.empty_like(pl[0])
        atc.attn_lse_merge(torch.stack(po), torch.stack(pl), out, lse)
        atc.attn_device_status()
        wo, wl = oracle.attention(qr[qrows], np.zeros(len(qrows), np.int32), pos[qrows], kr, vf, [0, T], pos,
                                  128 ** -0.5)
        check(out, lse, wo, wl, what=f"{kind} q{rq} merged over {world} key shards")


def test_prefill_tc_gapped_shards_in_one_varlen_call():
    """Two sequences in one call, each a different rank's shard with gaps (a
    striped one, then a zigzag one whose key count is not a multiple of 128), so
    the search runs on a key range that starts inside the packed buffer."""
    T = 1320
    q, k, v, pos = _shard_case(T, 64, 8, 1210)
    s_rows = synth.shard_rows(T, 4, 1, "striped")
    z_rows = synth.shard_rows(T, 2, 1, "zigzag")
    qrows = np.concatenate([s_rows, z_rows])
    krows = np.concatenate([synth.shard_rows(T, 4, 3, "striped"), synth.shard_rows(T, 2, 0, "zigzag")])
    nq = [len(s_rows), len(z_rows)]
    nk = [len(krows) - len(z_rows), len(z_rows)]
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    posd = torch.from_numpy(pos).to(DEV)
    atc.rope_apply_qk(qd, kd, posd)
    qi, ki = torch.from_numpy(qrows).to(DEV), torch.from_numpy(krows).to(DEV)
    cu_q, cu_k = synth.cu_seqlens(nq), synth.cu_seqlens(nk)
    i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(DEV)
    out, lse = _bf16_call(qd[qi].contiguous(), kd[ki].contiguous(), vd[ki].contiguous(), i32(cu_q), i32(pos[qrows]),
                          max(nq), i32(cu_k), i32(pos[krows]), torch.bfloat16)
    qr, kr = rotated_bf16(q, pos), rotated_bf16(k, pos)
    wo, wl = oracle.attention(qr[qrows], seq_ids(nq), pos[qrows], kr[krows], synth.as_f64(v)[krows], cu_k,
                              pos[krows], 128 ** -0.5)
    check(out, lse, wo, wl, what="gapped shards, varlen")


def _fp8_call(q, k, v, cu_q, qpos, maxq, cu_k, kpos, out_dtype):
    cq, sq = atc.quant_fp8_rows(q)
    ck, sk = atc.quant_fp8_heads(k)
    cv, sv = atc.quant_fp8_heads(v, transposed=True)
    out = torch.full(q.shape, float("nan"), dtype=out_dtype, device=DEV)
    lse = torch.full(q.shape[:2], float("nan"), dtype=torch.float32, device=DEV)
    atc.attn_prefill_fp8(cq, sq, ck, sk, cv, sv, out, lse, cu_q, qpos, maxq, cu_k, kpos)
    atc.attn_device_status()
    return out, lse


@pytest.mark.parametrize("kind", ["striped", "zigzag"])
def test_prefill_fp8_key_shards_with_position_gaps(kind):
    """The striped / zigzag ring steps on the e4m3 kernel: each shard's rotated
    Q, K, V quantised on their own (a key shard has its own per-head scales),
    compared with the oracle over the dequantised shard inputs; the merged shards
    equal the oracle over every shard's dequantised keys and values at once."""
    world, T = 2, 1200
    q, k, v, pos = _shard_case(T, 16, 2, 1220)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    posd = torch.from_numpy(pos).to(DEV)
    atc.rope_apply_qk(qd, kd, posd)
    qb, kb, vb = (synth.as_f64(t.cpu()) for t in (qd, kd, vd))  # the rotated bf16 inputs both sides quantise
    deq = {}
    for r in range(world):
        rows = synth.shard_rows(T, world, r, kind)
        ck, sk = oracle.quant_e4m3(kb[rows], [1])
        cv, sv = oracle.quant_e4m3(vb[rows], [1])
        deq[r] = (rows, ck * sk.astype(np.float64)[None, :, None], cv * sv.astype(np.float64)[None, :, None])
    for rq in range(world):
        qrows = synth.shard_rows(T, world, rq, kind)
        cq, sq = oracle.quant_e4m3(qb[qrows], [0, 1])
        qh = cq * sq.astype(np.float64)[:, :, None]
        po, pl = [], []
        for rk in range(world):
            krows, kh, vh = deq[rk]
            o, l = _rows_call(_fp8_call, qd, kd, vd, pos, qrows, krows)
            wo, wl = oracle.attention(qh, np.zeros(len(qrows), np.int32), pos[qrows], kh, vh, [0, len(krows)],
                                      pos[krows], 128 ** -0.5)
            check(o, l, wo, wl, tol_max=_fp8_max_tol(vh), tol_mean=FP8_MEAN, what=f"fp8 {kind} q{rq} k{rk}")
            po.append(o)
            pl.append(l)
        out = torch.empty_like(po[0])
        lse = torch.empty_like(pl[0])
        atc.attn_lse_merge(torch.stack(po), torch.stack(pl), out, lse)
        atc.attn_device_status()
        krows = np.concatenate([deq[r][0] for r in range(world)])
        kh = np.concatenate([deq[r][1] for r in range(world)])
        vh = np.concatenate([deq[r][2] for r in range(world)])
        order = np.argsort(krows, kind="stable")
        wo, wl = oracle.attention(qh, np.zeros(len(qrows), np.int32), pos[qrows], kh[order], vh[order], [0, T],
                                  pos[krows[order]], 128 ** -0.5)
        check(out, lse, wo, wl, tol_max=_fp8_max_tol(vh), tol_mean=FP8_MEAN, what=f"fp8 {kind} q{rq} merged")


# ------------------------------------------------------------------ sequence-parallel callables

def test_sp_kernel_callables_single_rank():
    """attention_tiled_causal_gb300.sp on one rank (no exchange): Ulysses with the
    tensor-core kernel as its per-rank attention, and the ring with the kernel's
    fp32 partials and the merge kernel, over a zigzag shard's queries, match the
    oracle."""
    from attention_tiled_causal_gb300 import sp
    T = 600
    q, k, v, pos = _shard_case(T, 16, 2, 1230)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    posd = torch.from_numpy(pos).to(DEV)
    atc.rope_apply_qk(qd, kd, posd)
    out, lse = sp.ulysses_attention(qd, kd, vd, posd)
    atc.attn_device_status()
    qr, kr, vf = rotated_bf16(q, pos), rotated_bf16(k, pos), synth.as_f64(v)
    wo, wl = oracle.attention(qr, np.zeros(T, np.int32), pos, kr, vf, [0, T], pos, 128 ** -0.5)
    check(out, lse, wo, wl, what="sp.ulysses_attention, one rank")
    rows = sp.shard_rows(T, 2, 1, "zigzag")
    ri = torch.from_numpy(rows).to(DEV)
    out, lse = sp.ring_attention(qd[ri].contiguous(), kd, vd, posd[ri].contiguous(), posd)
    atc.attn_device_status()
    check(out, lse, wo[rows], wl[rows], what="sp.ring_attention, one rank")


def test_prefill_fused_query_rope_on_gapped_shards():
    """The fused query RoPE on a zigzag query shard against the other rank's zigzag
    key shard (SGLang page, section 3.5): positions jump inside both the query and
    the key tiles.  Bit-identical to rope_apply followed by attn_prefill, and
    within tolerance of the oracle."""
    T, world = 1200, 2
    q, k, v, pos = _shard_case(T, 16, 2, 1240)
    qrows = synth.shard_rows(T, world, 1, "zigzag")
    krows = synth.shard_rows(T, world, 0, "zigzag")
    qs, ks, vs = q[qrows].contiguous(), k[krows].contiguous(), v[krows].contiguous()
    i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(DEV)
    qpos, kpos = i32(pos[qrows]), i32(pos[krows])
    cu_q, cu_k = i32([0, len(qrows)]), i32([0, len(krows)])
    kd = ks.to(DEV)
    atc.rope_apply(kd, kpos)
    vd = vs.to(DEV)
    qr = qs.to(DEV)
    atc.rope_apply(qr, qpos)
    ref_o, ref_l = atc.prefill(qr, kd, vd, cu_q, qpos, len(qrows), cu_k=cu_k, k_pos=kpos)
    qd = qs.to(DEV)
    tab = atc.rope_table(qpos, 128)
    out, lse = atc.prefill(qd, kd, vd, cu_q, qpos, len(qrows), cu_k=cu_k, k_pos=kpos, q_rope_cs=tab)
    atc.attn_device_status()
    assert torch.equal(out, ref_o) and torch.equal(lse, ref_l)
    wo, wl = oracle.attention(rotated_bf16(qs, pos[qrows]), np.zeros(len(qrows), np.int32), pos[qrows],
                              rotated_bf16(ks, pos[krows]), synth.as_f64(vs), [0, len(krows)], pos[krows],
                              128 ** -0.5)
    check(out, lse, wo, wl, what="fused query RoPE, zigzag shards")
