"""Parity at the full workload sizes, in the launch configuration bench.py times.

The CUDA path runs the whole problem; the fp64 oracle checks every row where it
finishes in seconds (8K prefill; all 32 requests of the decode over the bf16
and over the INT8 cache), 1024 seeded rows of the 8K FP8 prefill, and seeded
samples elsewhere: 512 rows per sequence for the 2 x 64K prefill and 512 rows
per request for chunked prefill over the 57K-token paged prefix.  The 8K
prefill is also measured against the unrounded definition (rotation kept in
fp64), within a bound derived from one bf16 rounding of each rotated element.
Inputs are drawn on the GPU by the seeded generators and copied back for the
oracle before any kernel touches them.
"""
import math

import numpy as np
import pytest
import torch

import attention_tiled_causal_gb300 as atc
import oracle
import synth

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
DEV = "cuda"
TOL_MAX, TOL_MEAN, TOL_LSE = 1e-2, 1e-3, 1e-3


def check(out, lse, want_o, want_l, what):
    o = out.float().cpu().numpy() if torch.is_tensor(out) else out
    l = lse.cpu().numpy() if torch.is_tensor(lse) else lse
    d = np.abs(o - want_o)
    assert np.isfinite(o).all(), f"{what}: non-finite output"
    assert d.max() <= TOL_MAX, f"{what}: max |dO| = {d.max():.3g}"
    assert d.mean() <= TOL_MEAN, f"{what}: mean |dO| = {d.mean():.3g}"
    dl = np.abs(l - want_l).max()
    assert dl <= TOL_LSE, f"{what}: max |dLSE| = {dl:.3g}"


def rot(x, pos):
    return oracle.round_bf16(oracle.rope(synth.as_f64(x), np.asarray(pos)))


@pytest.fixture(autouse=True)
def _status():
    atc.attn_device_status(clear=True)
    yield
    torch.cuda.empty_cache()


def _rounding_bounds(qr, kr, v, qpos, kpos, scale):
    """Per (row, head): eps = scale * (2u + u^2) * max_j sum_i |q_i| |k_ji| over
    the row's visible keys, u = 2^-8 + 2^-22 (one bf16 rounding of an element
    rotated in fp32), bounds |s' - s| for every score when each rotated element
    is perturbed by at most u of its size.  Softmax then moves each weight by a
    factor within [e^-2eps, e^2eps], so |dLSE| <= eps and
    |dO| <= (e^(2 eps) - 1) max|v|.  Returns (eps [rows, hq], max|v|)."""
    u = 2.0 ** -8 + 2.0 ** -22
    n, hq, d = qr.shape
    G = hq // kr.shape[1]
    aq, ak = np.abs(qr), np.abs(kr)
    hidden = qpos[:, None] < kpos[None, :]
    eps = np.empty((n, hq))
    for h in range(hq):
        m = aq[:, h, :] @ ak[:, h // G, :].T          # [rows, keys]
        m[hidden] = 0.0
        eps[:, h] = m.max(axis=1)
    return scale * (2 * u + u * u) * eps, np.abs(v).max()


def test_prefill_8k_all_rows():
    """Every row of the 8K workload against the oracle over bf16-rounded rotated
    Q/K (what the path consumes), and against the plain definition (rotation in
    fp64, unrounded): the distance to the latter is printed and must stay within
    the kernel tolerance plus the bound one bf16 rounding per rotated element
    allows (_rounding_bounds)."""
    w = synth.PREFILL_8K
    inp = w.make(DEV)
    q_raw, k_raw, v = inp["q"].cpu(), inp["k"].cpu(), inp["v"].cpu()
    pos, cu = inp["pos"], inp["cu"]
    atc.rope_apply(inp["q"], pos)
    atc.rope_apply(inp["k"], pos)
    out, lse = atc.prefill(inp["q"], inp["k"], inp["v"], cu, pos, w.seq, cu_k=cu, k_pos=pos)
    atc.attn_device_status()
    p = pos.cpu().numpy()
    vf = synth.as_f64(v)
    wo, wl = oracle.attention(rot(q_raw, p), np.zeros(w.seq, np.int32), p, rot(k_raw, p), vf,
                              cu.cpu().numpy(), p, w.scale)
    check(out, lse, wo, wl, "8K prefill, all rows")
    del wo, wl
    qx, kx = oracle.rope(synth.as_f64(q_raw), p), oracle.rope(synth.as_f64(k_raw), p)
    uo, ul = oracle.attention(qx, np.zeros(w.seq, np.int32), p, kx, vf, cu.cpu().numpy(), p, w.scale)
    o = out.float().cpu().numpy()
    l = lse.cpu().numpy()
    do, dl = np.abs(o - uo), np.abs(l - ul)
    eps, vmax = _rounding_bounds(qx, kx, vf, p, p, w.scale)
    print(f"\n8K prefill vs the unrounded definition: max|dO| {do.max():.3e} mean|dO| {do.mean():.3e} "
          f"max|dLSE| {dl.max():.3e} mean|dLSE| {dl.mean():.3e}; rows 0-127: max|dLSE| {dl[:128].max():.3e}; "
          f"bound eps: median {np.median(eps):.3e} max {eps.max():.3e}")
    assert (dl <= TOL_LSE + eps).all(), "LSE beyond the one-rounding bound"
    assert (do.max(axis=2) <= TOL_MAX + np.expm1(2 * eps) * vmax).all(), "O beyond the one-rounding bound"
    assert do.mean() <= TOL_MEAN


def test_prefill_fp8_8k_sampled_rows():
    """The FP8 prefill on the 8K workload's inputs taken as already rotated (the
    quantisers are bit-exact with the oracle's, so the codes on both sides are
    equal) over 1024 seeded query rows, all 64 heads, against the fp64 oracle over
    the dequantised values; bounds as for the small FP8 cases."""
    w = synth.PREFILL_8K
    inp = w.make(DEV)
    q_raw, k_raw, v_raw = inp["q"].cpu(), inp["k"].cpu(), inp["v"].cpu()
    pos, cu = inp["pos"], inp["cu"]
    cq, sq = atc.quant_fp8_rows(inp["q"])
    ck, sk = atc.quant_fp8_heads(inp["k"])
    cv, sv = atc.quant_fp8_heads(inp["v"], transposed=True)
    out = torch.empty(inp["q"].shape, dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(inp["q"].shape[:2], dtype=torch.float32, device=DEV)
    atc.attn_prefill_fp8(cq, sq, ck, sk, cv, sv, out, lse, cu, pos, w.seq, cu, pos)
    atc.attn_device_status()
    rows = synth.sample_rows(w.seq, 1024, 90)
    p = pos.cpu().numpy()
    oq, osq = oracle.quant_e4m3(synth.as_f64(q_raw[rows]), [0, 1])
    ok, osk = oracle.quant_e4m3(synth.as_f64(k_raw), [1])
    ov, osv = oracle.quant_e4m3(synth.as_f64(v_raw), [1])
    vh = ov * osv.astype(np.float64)[None, :, None]
    wo, wl = oracle.attention(oq * osq.astype(np.float64)[:, :, None], np.zeros(len(rows), np.int32), p[rows],
                              ok * osk.astype(np.float64)[None, :, None], vh, cu.cpu().numpy(), p, w.scale)
    o = out[torch.from_numpy(rows).to(DEV)].float().cpu().numpy()
    l = lse[torch.from_numpy(rows).to(DEV)].cpu().numpy()
    d = np.abs(o - wo)
    assert np.isfinite(o).all()
    tol_max = (2.0 ** -4 + 32 * 2.0 ** -10) * np.abs(vh).max()
    assert d.max() <= tol_max, f"fp8 8K: max |dO| = {d.max():.3g} > {tol_max:.3g}"
    assert d.mean() <= 4e-3, f"fp8 8K: mean |dO| = {d.mean():.3g}"
    assert np.abs(l - wl).max() <= TOL_LSE, f"fp8 8K: max |dLSE| = {np.abs(l - wl).max():.3g}"

def test_prefill_64k_x2_head_slice_and_all_heads():
    w = synth.PREFILL_64K
    inp = w.make(DEV)
    pos, cu = inp["pos"], inp["cu"]
    rows = np.concatenate([synth.sample_rows(w.seq, 512, 50 + b) + b * w.seq for b in range(w.batch)])
    q_raw = inp["q"][torch.from_numpy(rows).to(DEV)].cpu()
    k_raw, v = inp["k"].cpu(), inp["v"].cpu()
    atc.rope_apply(inp["q"], pos)
    atc.rope_apply(inp["k"], pos)
    out, lse = atc.prefill(inp["q"], inp["k"], inp["v"], cu, pos, w.seq, cu_k=cu, k_pos=pos)
    out_s = torch.full_like(out, float("nan"))
    lse_s = torch.full_like(lse, float("nan"))
    atc.attn_prefill(inp["q"], inp["k"], inp["v"], out_s, lse_s, cu, pos, w.seq, cu_k=cu, k_pos=pos, h_lo=16,
                     h_hi=32)
    atc.attn_device_status()
    # the Ulysses-style head slice equals its part of the all-heads call bit for bit
    assert torch.equal(out_s[:, 16:32], out[:, 16:32]) and torch.equal(lse_s[:, 16:32], lse[:, 16:32])
    assert torch.isnan(out_s[:, :16].float()).all() and torch.isnan(out_s[:, 32:].float()).all()
    p = pos.cpu().numpy()
    idx = torch.from_numpy(rows).to(DEV)
    wo, wl = oracle.attention(rot(q_raw, p[rows]), (rows // w.seq).astype(np.int32), p[rows], rot(k_raw, p),
                              synth.as_f64(v), cu.cpu().numpy(), p, w.scale)
    check(out[idx], lse[idx], wo, wl, "2 x 64K prefill, 512 rows per sequence, all heads")


def test_chunked_prefill_over_57k_paged_prefix():
    w = synth.CHUNKED
    inp = w.make(DEV)
    B, P, C = w.batch, w.prefix, w.chunk
    rows = np.concatenate([synth.sample_rows(C, 512, 70 + b) + b * C for b in range(B)])
    q_raw = inp["q"][torch.from_numpy(rows).to(DEV)].cpu()
    k_raw, v_new = inp["k"].cpu(), inp["v"].cpu()
    table = inp["page_table"].cpu().numpy()
    atc.rope_apply(inp["q"], inp["q_pos"])
    atc.rope_apply(inp["k"], inp["q_pos"])
    T, hq, d = inp["q"].shape
    po = torch.empty((2, T, hq, d), dtype=torch.float32, device=DEV)
    pl = torch.empty((2, T, hq), dtype=torch.float32, device=DEV)
    atc.attn_prefill(inp["q"], inp["k_cache"], inp["v_cache"], po[0], pl[0], inp["cu_q"], inp["q_pos"], C,
                     page_table=inp["page_table"], k_lens=inp["prefix_lens"], num_pages=inp["num_pages"])
    atc.attn_prefill(inp["q"], inp["k"], inp["v"], po[1], pl[1], inp["cu_q"], inp["q_pos"], C, cu_k=inp["cu_q"],
                     k_pos=inp["q_pos"])
    out = torch.empty((T, hq, d), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((T, hq), dtype=torch.float32, device=DEV)
    atc.attn_lse_merge(po, pl, out, lse)
    atc.attn_device_status()
    # oracle: each sampled chunk query over [gathered prefix ; causal chunk]
    kcf, vcf = synth.as_f64(inp["k_cache"].cpu()), synth.as_f64(inp["v_cache"].cpu())
    qpos = inp["q_pos"].cpu().numpy()
    krot = rot(k_raw, qpos)
    want_o = np.empty((len(rows), hq, d))
    want_l = np.empty((len(rows), hq))
    for b in range(B):
        sel = np.nonzero((rows // C) == b)[0]
        kb = np.stack([oracle.gather_pages(kcf, table, inp["num_pages"], g, b, P) for g in range(w.hkv)], 1)
        vb = np.stack([oracle.gather_pages(vcf, table, inp["num_pages"], g, b, P) for g in range(w.hkv)], 1)
        K = np.concatenate([kb, krot[b * C:(b + 1) * C]])
        V = np.concatenate([vb, synth.as_f64(v_new[b * C:(b + 1) * C])])
        KP = np.concatenate([np.arange(P, dtype=np.int32), qpos[b * C:(b + 1) * C]])
        o, l = oracle.attention(rot(q_raw[sel], qpos[rows[sel]]), np.zeros(len(sel), np.int32), qpos[rows[sel]], K,
                                V, [0, P + C], KP, w.scale)
        want_o[sel], want_l[sel] = o, l
        del kb, vb, K, V
    idx = torch.from_numpy(rows).to(DEV)
    check(out[idx], lse[idx], want_o, want_l, "chunked prefill, 512 rows per request")


def test_decode_b32_16_splits_all_requests():
    w = synth.DECODE
    inp = w.make(DEV)
    q_raw = inp["q"].cpu()
    q = inp["q"].clone()
    atc.rope_apply(q, inp["q_pos"])
    po, pl = atc.decode_workspace(w.batch, w.hq, w.splits, w.d, DEV)
    out = torch.empty((w.batch, w.hq, w.d), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((w.batch, w.hq), dtype=torch.float32, device=DEV)
    atc.attn_decode_paged(q, inp["k_cache"], inp["v_cache"], inp["page_table"], inp["ctx_lens"], w.splits, po, pl,
                          out, lse)
    atc.attn_device_status()
    ctx = inp["ctx_lens"].cpu().numpy()
    table = inp["page_table"].cpu().numpy()
    qpos = inp["q_pos"].cpu().numpy()
    for b in range(w.batch):
        n = (int(ctx[b]) + 63) // 64
        pages = torch.from_numpy(table[b, :n].astype(np.int64)).to(DEV)
        kc = inp["k_cache"][:, pages].cpu()  # this request's pages, in logical order
        vc = inp["v_cache"][:, pages].cpu()
        ident = np.arange(n, dtype=np.int32)[None, :]
        wo, wl = oracle.decode_paged(rot(q_raw[b:b + 1], qpos[b:b + 1]), synth.as_f64(kc), synth.as_f64(vc), ident,
                                     ctx[b:b + 1], n, w.scale)
        check(out[b:b + 1], lse[b:b + 1], wo, wl, f"decode request {b} (ctx {ctx[b]})")
        del kc, vc


def test_decode_int8_b32_16_splits_all_requests():
    """The INT8-cache decode at the full 32-request size (4.59 GB of codes and
    scales), every request checked against the oracle's decode over the exact
    cached values code * scale."""
    w = synth.DECODE_INT8
    inp = w.make(DEV)
    q_raw = inp["q"].cpu()
    q = inp["q"].clone()
    atc.rope_apply(q, inp["q_pos"])
    po, pl = atc.decode_workspace(w.batch, w.hq, w.splits, w.d, DEV)
    out = torch.empty((w.batch, w.hq, w.d), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((w.batch, w.hq), dtype=torch.float32, device=DEV)
    atc.attn_decode_paged_int8(q, inp["k_cache"], inp["v_cache"], inp["k_scale"], inp["v_scale"], inp["page_table"],
                               inp["ctx_lens"], w.splits, po, pl, out, lse)
    atc.attn_device_status()
    ctx = inp["ctx_lens"].cpu().numpy()
    table = inp["page_table"].cpu().numpy()
    qpos = inp["q_pos"].cpu().numpy()
    for b in range(w.batch):
        n = (int(ctx[b]) + 63) // 64
        pages = torch.from_numpy(table[b, :n].astype(np.int64)).to(DEV)
        kc = oracle.dequant_int8(inp["k_cache"][:, pages].cpu().numpy(), inp["k_scale"][:, pages].cpu().numpy())
        vc = oracle.dequant_int8(inp["v_cache"][:, pages].cpu().numpy(), inp["v_scale"][:, pages].cpu().numpy())
        ident = np.arange(n, dtype=np.int32)[None, :]
        wo, wl = oracle.decode_paged(rot(q_raw[b:b + 1], qpos[b:b + 1]), kc, vc, ident, ctx[b:b + 1], n, w.scale)
        check(out[b:b + 1], lse[b:b + 1], wo, wl, f"INT8 decode request {b} (ctx {ctx[b]})")
        del kc, vc
