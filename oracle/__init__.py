"""Python face of the fp64 CPU oracle (oracle.c).

TEST INFRASTRUCTURE.  Only the tests, `__graft_entry__.smoke()` and the bench's
CPU-baseline leg may import this package.  It shares no code with the CUDA
library and never imports it.

Every function takes and returns numpy float64 arrays; bf16/fp32 inputs are
first widened exactly (`synth.as_f64`).  `build()` compiles oracle.c with gcc
and OpenMP into liboracle.so next to this file.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
# A test that plants a mistake in a copy of oracle.c points this at the mutant build.
_OVERRIDE = os.environ.get("ORACLE_LIB")
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (plain C, -O2, IEEE arithmetic, OpenMP)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
                               _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        if _OVERRIDE:
            lib = C.CDLL(_OVERRIDE)
        else:
            build()
            lib = C.CDLL(_LIB_PATH)
        D, I64, I32, P = C.c_double, C.c_int64, C.c_int, C.c_void_p
        lib.oracle_rope.argtypes = [P, I64, I32, I32, P, D]
        lib.oracle_round_bf16.argtypes = [P, I64]
        lib.oracle_attention.argtypes = [P, I64, P, P, P, P, I32, P, P, I32, I32, I32, I32, I32,
                                         D, I32, P, P]
        lib.oracle_attention.restype = I32
        lib.oracle_gather_pages.argtypes = [P, P, I32, I32, I64, I32, I32, I32, I32, P]
        lib.oracle_gather_pages.restype = I32
        lib.oracle_decode_paged.argtypes = [P, P, P, P, P, I32, I32, I32, I64, I32, I32, I32, D, P, P]
        lib.oracle_decode_paged.restype = I32
        lib.oracle_lse_merge.argtypes = [P, P, I32, I64, I32, P, P]
        lib.oracle_kv_append.argtypes = [P, P, P, P, I64, I32, I32, P, P, I64, D]
        lib.oracle_kv_append.restype = I32
        lib.oracle_dequant_int8.argtypes = [P, P, I64, I32, P]
        lib.oracle_kv_append_int8.argtypes = [P, P, P, P, I64, I32, I32, P, P, P, P, I64, D]
        lib.oracle_kv_append_int8.restype = I32
        lib.oracle_round_e4m3.argtypes = [P, I64]
        lib.oracle_quant_e4m3.argtypes = [P, I64, I64, P, P]
        lib.oracle_num_threads.restype = I32
        lib.oracle_set_num_threads.argtypes = [I32]
        _lib = lib
    return _lib


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64)


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.int32)


def _p(a: np.ndarray):
    return a.ctypes.data_as(C.c_void_p)


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def set_num_threads(n: int) -> None:
    _load().oracle_set_num_threads(int(n))


def rope(x, pos, base: float = 10000.0) -> np.ndarray:
    """Rotated copy of x [tokens, heads, d] at absolute positions pos [tokens]."""
    y = _f64(x).copy()
    p = _i32(pos)
    T, H, d = y.shape
    assert p.shape == (T,) and d % 2 == 0
    _load().oracle_rope(_p(y), T, H, d, _p(p), float(base))
    return y


def round_bf16(x) -> np.ndarray:
    """Copy of x rounded to the bf16 grid, ties to even."""
    y = _f64(x).copy()
    _load().oracle_round_bf16(_p(y), y.size)
    return y


def attention(q, q_seq, q_pos, k, v, cu_k, k_pos, scale: float, causal: bool = True,
              h_lo: int = 0, h_hi=None):
    """Three-pass softmax attention for the query rows given.

    q [nq, hq, d]; row r belongs to sequence q_seq[r] at position q_pos[r].
    k, v [Tk, hkv, d]; sequence b owns key rows cu_k[b]..cu_k[b+1]-1 at k_pos.
    Returns (out [nq, hq, d], lse [nq, hq]); heads outside [h_lo, h_hi) are NaN.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    q_seq, q_pos, cu_k, k_pos = _i32(q_seq), _i32(q_pos), _i32(cu_k), _i32(k_pos)
    nq, hq, d = q.shape
    Tk, hkv, dk = k.shape
    assert dk == d and v.shape == k.shape and q_seq.shape == (nq,) and q_pos.shape == (nq,)
    assert k_pos.shape == (Tk,) and cu_k[-1] == Tk
    h_hi = hq if h_hi is None else h_hi
    out = np.full((nq, hq, d), np.nan)
    lse = np.full((nq, hq), np.nan)
    rc = _load().oracle_attention(_p(q), nq, _p(q_seq), _p(q_pos), _p(k), _p(v), len(cu_k) - 1,
                                  _p(cu_k), _p(k_pos), hq, hkv, d, h_lo, h_hi, float(scale),
                                  int(bool(causal)), _p(out), _p(lse))
    if rc != 0:
        raise ValueError("oracle_attention: bad arguments")
    return out, lse


def gather_pages(cache, page_table, num_pages: int, g: int, b: int, ctx: int) -> np.ndarray:
    """Tokens 0..ctx-1 of request b, KV head g, in logical order: [ctx, d]."""
    cache = _f64(cache)
    table = _i32(page_table)
    hkv, npg, page, d = cache.shape
    dst = np.empty((max(ctx, 0), d))
    rc = _load().oracle_gather_pages(_p(cache), _p(table), table.shape[1], page, num_pages, d,
                                     g, b, ctx, _p(dst))
    if rc != 0:
        raise ValueError("oracle_gather_pages: page id out of range")
    return dst


def decode_paged(q, k_cache, v_cache, page_table, ctx_lens, num_pages: int, scale: float):
    """Decode attention for q [B, hq, d] at positions ctx-1 over a paged cache
    [hkv, num_pages, page, d].  Returns (out [B, hq, d], lse [B, hq])."""
    q, kc, vc = _f64(q), _f64(k_cache), _f64(v_cache)
    table, ctx = _i32(page_table), _i32(ctx_lens)
    B, hq, d = q.shape
    hkv, npg, page, dk = kc.shape
    assert dk == d and vc.shape == kc.shape and ctx.shape == (B,)
    out = np.empty((B, hq, d))
    lse = np.empty((B, hq))
    rc = _load().oracle_decode_paged(_p(q), _p(kc), _p(vc), _p(table), _p(ctx), B, table.shape[1],
                                     page, num_pages, hq, hkv, d, float(scale), _p(out), _p(lse))
    if rc != 0:
        raise ValueError("oracle_decode_paged: bad page table or arguments")
    return out, lse


def lse_merge(part_o, part_lse):
    """part_o [P, ..., d], part_lse [P, ...] -> (out [..., d], lse [...])."""
    po, pl = _f64(part_o), _f64(part_lse)
    P = po.shape[0]
    lead = pl.shape[1:]
    assert po.shape[:-1] == pl.shape
    n = int(np.prod(lead)) if len(lead) else 1
    d = po.shape[-1]
    out = np.empty(lead + (d,))
    lse = np.empty(lead)
    _load().oracle_lse_merge(_p(po), _p(pl), P, n, d, _p(out), _p(lse))
    return out, lse


def kv_append(k_new, v_new, pos, slots, k_cache, v_cache, base: float = 10000.0):
    """New tokens' keys (rotated at `pos`, rounded to bf16) and values into copies of
    the head-major paged caches [heads][num_pages][page_size][d] at `slots`
    (page * page_size + offset; -1 skips).  Returns (k_cache, v_cache, n_bad_slots)."""
    k_new, v_new = _f64(k_new), _f64(v_new)
    T, H, d = k_new.shape
    kc, vc = np.array(k_cache, dtype=np.float64, copy=True), np.array(v_cache, dtype=np.float64, copy=True)
    rows = kc.shape[1] * kc.shape[2]
    pos = _i32(pos if pos is not None else np.zeros(T, np.int32))
    slots = _i32(slots)
    bad = _load().oracle_kv_append(_p(k_new), _p(v_new), _p(pos), _p(slots), T, H, d, _p(kc), _p(vc), rows,
                                   float(base))
    if bad < 0:
        raise MemoryError("oracle_kv_append: out of memory")
    return kc, vc, bad


def dequant_int8(codes, scales) -> np.ndarray:
    """Exact values of an INT8 cache: codes [..., d] int8 times scales [...] fp32
    (one scale per cached token of a KV head)."""
    codes = np.ascontiguousarray(codes, dtype=np.int8)
    scales = np.ascontiguousarray(scales, dtype=np.float32)
    if codes.shape[:-1] != scales.shape:
        raise ValueError("scales must have the codes' shape without the last axis")
    d = codes.shape[-1]
    rows = int(np.prod(codes.shape[:-1]))
    out = np.empty(codes.shape, dtype=np.float64)
    _load().oracle_dequant_int8(_p(codes), _p(scales), rows, d, _p(out))
    return out


def kv_append_int8(k_new, v_new, pos, slots, k_codes, v_codes, k_scale, v_scale, base: float = 10000.0):
    """kv_append into an INT8 cache: keys rotated at `pos` and rounded to bf16, then
    every key and value row quantised (scale = max|x| / 127 in fp32, codes rounded
    to nearest even).  Returns copies (k_codes, v_codes, k_scale, v_scale, n_bad)."""
    k_new, v_new = _f64(k_new), _f64(v_new)
    T, H, d = k_new.shape
    kc = np.array(k_codes, dtype=np.int8, copy=True)
    vc = np.array(v_codes, dtype=np.int8, copy=True)
    ks = np.array(k_scale, dtype=np.float32, copy=True)
    vs = np.array(v_scale, dtype=np.float32, copy=True)
    rows = kc.shape[1] * kc.shape[2]
    pos = _i32(pos if pos is not None else np.zeros(T, np.int32))
    bad = _load().oracle_kv_append_int8(_p(k_new), _p(v_new), _p(pos), _p(_i32(slots)), T, H, d, _p(kc), _p(vc),
                                        _p(ks), _p(vs), rows, float(base))
    if bad < 0:
        raise MemoryError("oracle_kv_append_int8: out of memory")
    return kc, vc, ks, vs, bad


def round_e4m3(x) -> np.ndarray:
    """Nearest e4m3 values (ties to even, saturating at +-448)."""
    out = np.array(x, dtype=np.float64, copy=True)
    _load().oracle_round_e4m3(_p(out), out.size)
    return out


def quant_e4m3(x, group_axes):
    """Quantise x to e4m3 with one fp32 scale per group: a group is one index of
    the leading `group_axes` axes of x (after moving them to the front, in
    order); scale = max|x| / 448, value = e4m3(x / scale) decided in fp32.
    Returns (values with x's shape, scales with the group axes' shape)."""
    x = _f64(x)
    axes = list(group_axes)
    rest = [a for a in range(x.ndim) if a not in axes]
    xt = np.ascontiguousarray(np.transpose(x, axes + rest))
    gshape = xt.shape[:len(axes)]
    groups = int(np.prod(gshape))
    n = int(np.prod(xt.shape[len(axes):]))
    codes = np.empty(xt.shape, dtype=np.float64)
    scales = np.empty(gshape, dtype=np.float32)
    _load().oracle_quant_e4m3(_p(xt), groups, n, _p(codes), _p(scales))
    inv = np.argsort(axes + rest)
    return np.transpose(codes, inv), scales
