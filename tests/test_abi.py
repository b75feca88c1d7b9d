"""The C-ABI library loads and exports every function include/attn_gb300.h declares,
and its host-side argument checks reject bad calls before touching a GPU."""
import ctypes as C
import os
import re

import pytest

import attention_tiled_causal_gb300 as atc

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn_gb300.h")

ERR_ARG, ERR_SHAPE, ERR_ALIGN, ERR_UNSUPPORTED = 1, 2, 3, 4


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*ATTN_API\s+(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", text, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    from attention_tiled_causal_gb300 import build
    build.build()
    return atc.library()


def test_header_declares_the_hot_path_calls():
    names = declared_functions()
    for n in ("rope_apply", "attn_prefill", "attn_decode_paged", "attn_lse_merge", "attn_last_error",
              "attn_device_status"):
        assert n in names, n


def test_library_exports_every_declared_symbol(lib):
    for n in declared_functions():
        assert hasattr(lib, n), f"libattn_gb300.so does not export {n}"


def test_only_the_c_abi_is_exported(lib):
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", atc.lib_path()], capture_output=True, text=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    ours = {s for s in exported if s.startswith(("attn_", "rope_", "quant_"))}
    assert ours == set(declared_functions())


def _prefill(lib, **kw):
    a = dict(q=16, k=16, v=16, out=16, out_dtype=0, lse=None, dtype=0, batch=1, cu_q=16, q_pos=16, total_q=4,
             max_seqlen_q=4, cu_k=16, k_pos=16, total_k=4, page_table=None, k_lens=None, max_pages=0,
             page_size=0, num_pages=0, hq=8, hkv=2, d=128, h_lo=0, h_hi=8, scale=0.1, causal=1, stream=None)
    a.update(kw)
    return lib.attn_prefill(*a.values())


def test_prefill_rejects_bad_arguments(lib):
    assert _prefill(lib, h_lo=2) == ERR_SHAPE            # not a whole GQA group
    assert _prefill(lib, h_hi=9) == ERR_SHAPE
    assert _prefill(lib, hq=6, hkv=4) == ERR_SHAPE       # 6 % 4 != 0
    assert _prefill(lib, d=96) == ERR_SHAPE
    assert _prefill(lib, dtype=1, out_dtype=0) == ERR_UNSUPPORTED
    assert _prefill(lib, batch=-1) == ERR_ARG
    assert _prefill(lib, q=None) == ERR_ARG
    assert _prefill(lib, q=8) == ERR_ALIGN               # misaligned device pointer
    assert _prefill(lib, scale=0.0) == ERR_ARG
    assert _prefill(lib, cu_k=None) == ERR_ARG           # contiguous source needs cu_k
    assert _prefill(lib, page_table=16, k_lens=16) == ERR_ARG   # paged source takes no cu_k/k_pos
    assert b"GQA" in lib.attn_last_error() or len(lib.attn_last_error()) > 0


def test_prefill_empty_problem_is_a_no_op(lib):
    assert _prefill(lib, batch=0) == 0
    assert _prefill(lib, h_lo=4, h_hi=4) == 0
    assert _prefill(lib, max_seqlen_q=0) == 0


def test_decode_rejects_bad_arguments(lib):
    base = dict(q=16, kc=16, vc=16, table=16, ctx=16, batch=2, max_pages=4, page=64, num_pages=8, hq=64, hkv=8,
                d=128, splits=16, scale=0.1, po=16, pl=16, out=16, odt=0, lse=None, stream=None)

    def call(**kw):
        a = dict(base)
        a.update(kw)
        return lib.attn_decode_paged(*a.values())

    assert call(hq=32) == ERR_SHAPE
    assert call(d=64) == ERR_SHAPE
    assert call(page=32) == ERR_SHAPE
    assert call(splits=0) == ERR_ARG
    assert call(splits=257) == ERR_ARG
    assert call(table=None) == ERR_ARG
    assert call(kc=24) == ERR_ALIGN
    assert call(batch=0) == 0


def test_rope_and_merge_reject_bad_arguments(lib):
    assert lib.rope_apply(16, 0, 4, 2, 100, 200, 16, 1e4, None) == ERR_SHAPE   # 50 not a multiple of 8
    assert lib.rope_apply(16, 0, 4, 2, 128, 100, 16, 1e4, None) == ERR_ARG     # stride < heads*d
    assert lib.rope_apply(8, 0, 4, 2, 128, 256, 16, 1e4, None) == ERR_ALIGN
    assert lib.rope_apply(16, 0, 0, 2, 128, 256, 16, 1e4, None) == 0          # nothing to do
    assert lib.attn_lse_merge(16, 16, 0, 4, 2, 128, 0, 0, 0, 0, 0, 0, 16, 0, None, None) == ERR_ARG
    assert lib.attn_lse_merge(16, 16, 2, 0, 2, 128, 0, 0, 0, 0, 0, 0, 16, 0, None, None) == 0


def test_kv_append_rejects_bad_arguments(lib):
    base = dict(kn=16, vn=16, pos=16, slots=16, T=4, H=8, d=128, kc=16, vc=16, pages=10, page=64, ko=None,
                rope_base=1e4, stream=None)

    def call(**kw):
        a = dict(base)
        a.update(kw)
        f = lib.attn_kv_append_paged
        f.argtypes = [C.c_void_p] * 4 + [C.c_int64, C.c_int, C.c_int, C.c_void_p, C.c_void_p, C.c_int64, C.c_int,
                                         C.c_void_p, C.c_double, C.c_void_p]
        return f(*a.values())

    assert call(d=100) == ERR_SHAPE          # half of 100 is not a multiple of 8
    assert call(d=512) == ERR_SHAPE
    assert call(rope_base=-1.0) == ERR_ARG
    assert call(T=-1) == ERR_ARG
    assert call(slots=None) == ERR_ARG
    assert call(pos=None) == ERR_ARG         # rotation needs positions
    assert call(pages=0) == ERR_ARG
    assert call(kc=24) == ERR_ALIGN
    assert call(ko=8) == ERR_ALIGN
    assert call(T=0) == 0
    assert call(H=0) == 0


def test_decode_int8_rejects_bad_arguments(lib):
    base = dict(q=16, kc=16, vc=16, ks=16, vs=16, table=16, ctx=16, batch=2, max_pages=4, page=64, num_pages=8,
                hq=64, hkv=8, d=128, splits=16, scale=0.1, po=16, pl=16, out=16, odt=0, lse=None, stream=None)

    def call(**kw):
        a = dict(base)
        a.update(kw)
        return lib.attn_decode_paged_int8(*a.values())

    assert call(hq=32) == ERR_SHAPE
    assert call(d=64) == ERR_SHAPE
    assert call(page=32) == ERR_SHAPE
    assert call(splits=0) == ERR_ARG
    assert call(ks=None) == ERR_ARG
    assert call(vs=8) == ERR_ALIGN
    assert call(kc=24) == ERR_ALIGN
    assert call(batch=0) == 0


def test_rope_table_and_fused_prefill_reject_bad_arguments(lib):
    assert lib.rope_table(16, 4, 127, 1e4, 16, None) == ERR_SHAPE     # odd head_dim
    assert lib.rope_table(16, 4, 128, 0.0, 16, None) == ERR_ARG       # base
    assert lib.rope_table(None, 4, 128, 1e4, 16, None) == ERR_ARG
    assert lib.rope_table(16, 4, 128, 1e4, 8, None) == ERR_ALIGN
    assert lib.rope_table(16, 0, 128, 1e4, None, None) == 0
    a = dict(q=16, k=16, v=16, out=16, out_dtype=0, lse=None, dtype=0, batch=1, cu_q=16, q_pos=16, total_q=4,
             max_seqlen_q=4, cu_k=16, k_pos=16, total_k=4, page_table=None, k_lens=None, max_pages=0,
             page_size=0, num_pages=0, hq=8, hkv=2, d=128, h_lo=0, h_hi=8, scale=0.1, causal=1)
    f = lib.attn_prefill_rope_q
    assert f(*a.values(), None, None) == ERR_ARG      # no table
    assert f(*a.values(), 8, None) == ERR_ALIGN       # misaligned table
    a["d"] = 96
    assert f(*a.values(), 16, None) == ERR_SHAPE      # prefill's own checks still apply


def test_kv_append_int8_rejects_bad_arguments(lib):
    base = dict(kn=16, vn=16, pos=16, slots=16, T=4, H=8, d=128, kc=16, vc=16, ks=16, vs=16, pages=10, page=64,
                ko=None, rope_base=1e4, stream=None)

    def call(**kw):
        a = dict(base)
        a.update(kw)
        return lib.attn_kv_append_paged_int8(*a.values())

    assert call(d=64) == ERR_SHAPE
    assert call(rope_base=-1.0) == ERR_ARG
    assert call(ks=None) == ERR_ARG
    assert call(vs=8) == ERR_ALIGN
    assert call(T=0) == 0


def test_quant_fp8_and_fp8_prefill_reject_bad_arguments(lib):
    assert lib.quant_fp8_rows(16, 4, 2, 64, 16, 16, None) == ERR_SHAPE
    assert lib.quant_fp8_rows(8, 4, 2, 128, 16, 16, None) == ERR_ALIGN
    assert lib.quant_fp8_heads(16, 4, 2, 128, 16, 16, 16, 1, 8, None) == ERR_ARG     # t_stride < tokens
    assert lib.quant_fp8_heads(16, 4, 2, 128, 16, 16, 16, 1, 20, None) == ERR_ARG    # not a multiple of 16
    assert lib.quant_fp8_rows(16, 0, 2, 128, None, None, None) == 0
    a = dict(q=16, qs=16, k=16, ks=16, vt=16, vs=16, vts=16, out=16, odt=0, lse=None, batch=1, cu_q=16, q_pos=16,
             total_q=4, max_q=4, cu_k=16, k_pos=16, total_k=4, hq=8, hkv=2, d=128, h_lo=0, h_hi=8, scale=0.1,
             causal=1, stream=None)

    def call(**kw):
        b = dict(a)
        b.update(kw)
        return lib.attn_prefill_fp8(*b.values())

    assert call(d=64) == ERR_SHAPE
    assert call(h_lo=1) == ERR_SHAPE
    assert call(vts=8) == ERR_ARG          # v_t_stride < total_k
    assert call(vts=24) == ERR_ARG         # not a multiple of 16
    assert call(qs=None) == ERR_ARG
    assert call(vt=8) == ERR_ALIGN
    assert call(scale=0.0) == ERR_ARG
    assert call(odt=7) == ERR_UNSUPPORTED
    assert call(batch=0) == 0


def test_rope_quant_fp8_rejects_bad_arguments(lib):
    assert lib.rope_quant_fp8_rows(16, 4, 2, 64, 16, 1e4, 16, 16, None) == ERR_SHAPE
    assert lib.rope_quant_fp8_rows(16, 4, 2, 128, 16, 0.0, 16, 16, None) == ERR_ARG   # base
    assert lib.rope_quant_fp8_rows(16, 4, 2, 128, None, 1e4, 16, 16, None) == ERR_ARG  # positions
    assert lib.rope_quant_fp8_rows(16, 4, 2, 128, 16, 1e4, 8, 16, None) == ERR_ALIGN
    assert lib.rope_quant_fp8_rows(16, 0, 2, 128, None, 1e4, None, None, None) == 0
    assert lib.rope_quant_fp8_heads(16, 4, 300, 128, 16, 1e4, 16, 16, 16, None) == ERR_SHAPE   # > 256 heads
    assert lib.rope_quant_fp8_heads(16, 4, 8, 128, 16, 1e4, 16, 16, None, None) == ERR_ARG    # no scratch


def test_rope_apply_qk_rejects_bad_arguments(lib):
    f = lib.rope_apply_qk
    assert f(16, 8, 1024, 16, 2, 256, 0, 4, 100, 16, 1e4, None) == ERR_SHAPE     # 50 not a multiple of 8
    assert f(16, 8, 100, 16, 2, 256, 0, 4, 128, 16, 1e4, None) == ERR_ARG       # q stride < heads * d
    assert f(16, 8, 1024, 8, 2, 256, 0, 4, 128, 16, 1e4, None) == ERR_ALIGN     # misaligned k
    assert f(16, 8, 1024, 16, 2, 256, 0, 4, 128, None, 1e4, None) == ERR_ARG    # no positions
    assert f(16, 8, 1024, 16, 2, 256, 0, 4, 128, 16, 0.0, None) == ERR_ARG      # base
    assert f(16, 8, 1024, 16, 2, 256, 5, 4, 128, 16, 1e4, None) == ERR_UNSUPPORTED
    assert f(None, 0, 0, None, 0, 0, 0, 4, 128, 16, 1e4, None) == 0              # nothing to rotate
