"""attn_decode_paged_noalloc, the decode entry point for callers that cannot
allocate device memory (an engine whose KV-cache pool already holds all free
HBM, a plugin inside another framework's caching allocator, a latency-critical
path where cudaMalloc would synchronise the device).  It keeps the split
partials in a scratch array the library holds statically, and must give the
same answer as attn_decode_paged with a caller-supplied workspace -- also on a
second call, after the first call has left its own data in that scratch.

This file is named to be collected last, so a run that stops at the first
failure has run every other test before it.  One test repeats the two-call
check in a fresh Python process, so the entry point's first call on a device
(the scratch address lookup) is covered without anything loaded before it.
"""
import ctypes as C
import os
import subprocess
import sys

import pytest
import torch

import attention_tiled_causal_gb300 as atc
import synth

pytestmark = pytest.mark.gpu
DEV = "cuda"
TOL_MAX, TOL_MEAN, TOL_LSE = 1e-2, 1e-3, 1e-3   # the bf16 tolerance of the parity tests


def _entry():
    lib = atc.library()
    f = lib.attn_decode_paged_noalloc
    P, I32, I64, F32 = C.c_void_p, C.c_int, C.c_int64, C.c_float
    f.argtypes = [P, P, P, P, P, I32, I32, I32, I64, I32, I32, I32, I32, F32, P, I32, P, P]
    f.restype = I32
    return lib, f


def _case(ctx, hq, hkv, splits, seed):
    wl = synth.Decode("no-alloc decode", batch=len(ctx), ctx_lo=0, ctx_hi=0, hq=hq, hkv=hkv, d=128,
                      splits=splits, seed=seed, ctx_fixed=ctx)
    inp = wl.make(DEV)
    q = inp["q"].clone()
    atc.rope_apply(q, inp["q_pos"])
    return wl, inp, q


def _reference(wl, inp, q):
    po, pl = atc.decode_workspace(wl.batch, wl.hq, wl.splits, wl.d, DEV)
    out = torch.empty((wl.batch, wl.hq, wl.d), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((wl.batch, wl.hq), dtype=torch.float32, device=DEV)
    atc.attn_decode_paged(q, inp["k_cache"], inp["v_cache"], inp["page_table"], inp["ctx_lens"], wl.splits, po, pl,
                          out, lse)
    return out, lse


def _noalloc(f, lib, wl, inp, q):
    out = torch.full((wl.batch, wl.hq, wl.d), float("nan"), dtype=torch.bfloat16, device=DEV)
    lse = torch.full((wl.batch, wl.hq), float("nan"), dtype=torch.float32, device=DEV)
    table = inp["page_table"]
    st = f(q.data_ptr(), inp["k_cache"].data_ptr(), inp["v_cache"].data_ptr(), table.data_ptr(),
           inp["ctx_lens"].data_ptr(), wl.batch, table.shape[1], 64, inp["num_pages"], wl.hq, wl.hkv, wl.d,
           wl.splits, wl.scale, out.data_ptr(), 0, lse.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == 0, lib.attn_last_error().decode()
    return out, lse


def _close(out, lse, ref_o, ref_l):
    d = (out.float() - ref_o.float()).abs()
    assert torch.isfinite(out.float()).all()
    assert d.max().item() <= TOL_MAX and d.mean().item() <= TOL_MEAN
    inf = torch.isinf(ref_l)
    assert torch.equal(torch.isinf(lse), inf)
    assert (lse[~inf] - ref_l[~inf]).abs().max().item() <= TOL_LSE


def _two_calls_in_a_row():
    atc.attn_device_status(clear=True)
    lib, f = _entry()
    # first call: many splits over long contexts fills a large part of the scratch
    wl1, inp1, q1 = _case([5000, 300, 12000, 64], 64, 8, 16, 700)
    # second call: fewer requests and splits, a zero-length context and an
    # empty-split request; stale partials from the first call must not leak in
    wl2, inp2, q2 = _case([1, 0, 777], 16, 2, 4, 701)
    for wl, inp, q in ((wl1, inp1, q1), (wl2, inp2, q2)):
        ref_o, ref_l = _reference(wl, inp, q)
        out, lse = _noalloc(f, lib, wl, inp, q)
        atc.attn_device_status()
        _close(out, lse, ref_o, ref_l)


def test_noalloc_decode_matches_workspace_decode_on_two_calls_in_a_row():
    _two_calls_in_a_row()


def test_noalloc_decode_in_a_fresh_process():
    """The same two calls as the first thing a new process does on the GPU."""
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    code = ("import sys; sys.path.insert(0, %r); sys.path.insert(0, %r); "
            "import test_zz_no_alloc as t; t._two_calls_in_a_row(); print('fresh ok')"
            % (root, os.path.join(root, "tests")))
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and "fresh ok" in r.stdout, r.stdout[-2000:] + r.stderr[-2000:]


def test_noalloc_decode_allocates_no_device_memory():
    """After a first call (module load, scratch address lookup), further calls
    leave both the caching allocator's count and the device's free memory as
    they were: the entry point calls no allocator."""
    lib, f = _entry()
    wl, inp, q = _case([3000, 64, 9000], 64, 8, 16, 703)
    out = torch.empty((wl.batch, wl.hq, wl.d), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((wl.batch, wl.hq), dtype=torch.float32, device=DEV)
    table = inp["page_table"]
    args = (q.data_ptr(), inp["k_cache"].data_ptr(), inp["v_cache"].data_ptr(), table.data_ptr(),
            inp["ctx_lens"].data_ptr(), wl.batch, table.shape[1], 64, inp["num_pages"], wl.hq, wl.hkv, wl.d,
            wl.splits, wl.scale, out.data_ptr(), 0, lse.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert f(*args) == 0, lib.attn_last_error().decode()
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    alloc0 = torch.cuda.memory_allocated()
    for _ in range(3):
        assert f(*args) == 0, lib.attn_last_error().decode()
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert torch.cuda.memory_allocated() == alloc0
    assert free1 == free0, f"device free memory changed by {free0 - free1} bytes"
    atc.attn_device_status()


def test_noalloc_decode_rejects_calls_beyond_the_static_scratch():
    lib, f = _entry()
    wl, inp, q = _case([64] * 33, 64, 8, 16, 702)   # 33 * 64 * 16 = 33792 > 32768 partial rows
    out = torch.zeros((wl.batch, wl.hq, wl.d), dtype=torch.bfloat16, device=DEV)
    table = inp["page_table"]
    st = f(q.data_ptr(), inp["k_cache"].data_ptr(), inp["v_cache"].data_ptr(), table.data_ptr(),
           inp["ctx_lens"].data_ptr(), wl.batch, table.shape[1], 64, inp["num_pages"], wl.hq, wl.hkv, wl.d,
           wl.splits, wl.scale, out.data_ptr(), 0, None, torch.cuda.current_stream().cuda_stream)
    assert st == 1
    assert b"scratch" in lib.attn_last_error()
    torch.cuda.synchronize()
    assert torch.all(out == 0)   # nothing was launched
