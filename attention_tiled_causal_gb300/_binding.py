"""ctypes marshalling for libattn_gb300.so (see include/attn_gb300.h for the contracts)."""
from __future__ import annotations

import ctypes as C
import math
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libattn_gb300.so")

ATTN_BF16 = 0
ATTN_FP32 = 1

_lib = None


class AttnError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"status {status}: {msg}")
        self.status = status


def lib_path() -> str:
    return _LIB_PATH


def library():
    """Load the shared library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise ImportError(f"{_LIB_PATH} is missing: build it with `python -c \"import __graft_entry__ as g; "
                          f"g.build()\"` (nvcc, sm_103a)")
    lib = C.CDLL(_LIB_PATH)
    P, I32, I64, F32, F64 = C.c_void_p, C.c_int, C.c_int64, C.c_float, C.c_double
    lib.attn_last_error.restype = C.c_char_p
    lib.attn_device_status.argtypes = [I32]
    lib.attn_device_status.restype = I32
    lib.attn_selftest_wait_timeout.argtypes = [I32, P]
    lib.attn_selftest_wait_timeout.restype = I32
    lib.rope_apply.argtypes = [P, I32, I64, I32, I32, I64, P, F64, P]
    lib.rope_apply.restype = I32
    lib.rope_table.argtypes = [P, I64, I32, F64, P, P]
    lib.rope_apply_qk.argtypes = [P, I32, I64, P, I32, I64, I32, I64, I32, P, F64, P]
    lib.rope_apply_qk.restype = I32
    lib.rope_table.restype = I32
    lib.attn_prefill_rope_q.argtypes = [P, P, P, P, I32, P, I32, I32, P, P, I64, I32, P, P, I64, P, P, I32, I32,
                                        I64, I32, I32, I32, I32, I32, F32, I32, P, P]
    lib.attn_prefill_rope_q.restype = I32
    lib.attn_prefill_fp8.argtypes = [P, P, P, P, P, P, I64, P, I32, P, I32, P, P, I64, I32, P, P, I64, I32, I32,
                                     I32, I32, I32, F32, I32, P]
    lib.attn_prefill_fp8.restype = I32
    lib.quant_fp8_rows.argtypes = [P, I64, I32, I32, P, P, P]
    lib.rope_quant_fp8_rows.argtypes = [P, I64, I32, I32, P, F64, P, P, P]
    lib.rope_quant_fp8_rows.restype = I32
    lib.rope_quant_fp8_heads.argtypes = [P, I64, I32, I32, P, F64, P, P, P, P]
    lib.rope_quant_fp8_heads.restype = I32
    lib.quant_fp8_rows.restype = I32
    lib.quant_fp8_heads.argtypes = [P, I64, I32, I32, P, P, P, I32, I64, P]
    lib.quant_fp8_heads.restype = I32
    lib.attn_kv_append_paged_int8.argtypes = [P, P, P, P, I64, I32, I32, P, P, P, P, I64, I32, P, F64, P]
    lib.attn_kv_append_paged_int8.restype = I32
    lib.attn_kv_append_paged.argtypes = [P, P, P, P, I64, I32, I32, P, P, I64, I32, P, F64, P]
    lib.attn_kv_append_paged.restype = I32
    lib.attn_prefill.argtypes = [P, P, P, P, I32, P, I32, I32, P, P, I64, I32, P, P, I64, P, P, I32, I32, I64,
                                 I32, I32, I32, I32, I32, F32, I32, P]
    lib.attn_prefill.restype = I32
    lib.attn_decode_paged.argtypes = [P, P, P, P, P, I32, I32, I32, I64, I32, I32, I32, I32, F32, P, P, P, I32,
                                      P, P]
    lib.attn_decode_paged.restype = I32
    lib.attn_decode_paged_int8.argtypes = [P, P, P, P, P, P, P, I32, I32, I32, I64, I32, I32, I32, I32, F32, P, P,
                                           P, I32, P, P]
    lib.attn_decode_paged_int8.restype = I32
    lib.attn_lse_merge.argtypes = [P, P, I32, I64, I32, I32, I64, I64, I64, I64, I64, I64, P, I32, P, P]
    lib.attn_lse_merge.restype = I32
    _lib = lib
    return lib


def _check(status: int):
    if status != 0:
        raise AttnError(status, library().attn_last_error().decode())


def _stream(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensors passed to the library must live on a CUDA device")
    return t.data_ptr()


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return ATTN_BF16
    if t.dtype == torch.float32:
        return ATTN_FP32
    raise ValueError(f"unsupported dtype {t.dtype}")


def _i32(t: Optional[torch.Tensor], name: str) -> Optional[torch.Tensor]:
    if t is None:
        return None
    if t.dtype != torch.int32 or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous int32 tensor")
    return t


def attn_device_status(clear: bool = True) -> None:
    """Synchronise and raise if a kernel recorded a device-side fault."""
    _check(library().attn_device_status(1 if clear else 0))


def attn_selftest_wait_timeout(which: int, stream=None) -> None:
    """Launch the bounded-wait check: a wait on a barrier nothing completes runs
    out after about 2 s and records its code (which 0: 0x102, 1: 0x105), which
    the next attn_device_status() raises."""
    _check(library().attn_selftest_wait_timeout(int(which), _stream(stream)))


def rope_apply(x: torch.Tensor, positions: torch.Tensor, base: float = 10000.0, stream=None) -> torch.Tensor:
    """Rotate x [tokens, heads, head_dim] in place at absolute `positions` [tokens]."""
    if x.dim() != 3 or x.stride(2) != 1 or x.stride(1) != x.shape[2]:
        raise ValueError("x must be [tokens, heads, head_dim] with heads and head_dim packed")
    positions = _i32(positions, "positions")
    if positions.numel() != x.shape[0]:
        raise ValueError("positions must hold one entry per token")
    _check(library().rope_apply(_ptr(x), _dt(x), x.shape[0], x.shape[1], x.shape[2], x.stride(0),
                                _ptr(positions), float(base), _stream(stream)))
    return x


def rope_apply_qk(q: torch.Tensor, k: torch.Tensor, positions: torch.Tensor, base: float = 10000.0,
                  stream=None) -> None:
    """rope_apply on q [tokens, Hq, d] and k [tokens, Hkv, d] (same dtype and d) in one
    launch, in place, at the same absolute positions."""
    for t, n in ((q, "q"), (k, "k")):
        if t.dim() != 3 or t.stride(2) != 1 or t.stride(1) != t.shape[2]:
            raise ValueError(f"{n} must be [tokens, heads, head_dim] with heads and head_dim packed")
    if q.dtype != k.dtype or q.shape[0] != k.shape[0] or q.shape[2] != k.shape[2]:
        raise ValueError("q and k must share dtype, token count and head_dim")
    T, Hq, d = q.shape
    positions = _i32(positions, "positions")
    if positions.numel() != T:
        raise ValueError("positions must hold one entry per token")
    _check(library().rope_apply_qk(_ptr(q), Hq, q.stride(0), _ptr(k), k.shape[1], k.stride(0), _dt(q), T, d,
                                   _ptr(positions), float(base), _stream(stream)))


def attn_kv_append_paged(k_new, v_new, positions, slots, k_cache, v_cache, *, k_rot_out=None,
                         base: float = 10000.0, stream=None) -> None:
    """Write new tokens' K (rotated at `positions`) and V [tokens, Hkv, d] bf16 into the
    head-major paged caches [Hkv, num_pages, page_size, d] at `slots` [tokens]
    (page * page_size + offset; -1 skips).  k_rot_out [tokens, Hkv, d] also receives
    the rotated keys if given.  base = 0 copies the keys unrotated."""
    for t, n in ((k_new, "k_new"), (v_new, "v_new"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        if not t.is_contiguous() or t.dtype != torch.bfloat16:
            raise ValueError(f"{n} must be contiguous bf16")
    T, hkv, d = k_new.shape
    if tuple(v_new.shape) != (T, hkv, d):
        raise ValueError("v_new must have k_new's shape")
    if k_cache.dim() != 4 or tuple(k_cache.shape) != tuple(v_cache.shape) or k_cache.shape[0] != hkv \
            or k_cache.shape[3] != d:
        raise ValueError("caches must be [num_kv_heads, num_pages, page_size, head_dim], alike")
    if k_rot_out is not None and (tuple(k_rot_out.shape) != (T, hkv, d) or not k_rot_out.is_contiguous()
                                  or k_rot_out.dtype != torch.bfloat16):
        raise ValueError("k_rot_out must be contiguous bf16 shaped like k_new")
    slots = _i32(slots, "slots")
    if slots.numel() != T:
        raise ValueError("slots must hold one entry per token")
    pos_ptr = None
    if base > 0:
        positions = _i32(positions, "positions")
        if positions.numel() != T:
            raise ValueError("positions must hold one entry per token")
        pos_ptr = _ptr(positions)
    _check(library().attn_kv_append_paged(_ptr(k_new), _ptr(v_new), pos_ptr, _ptr(slots), T, hkv, d,
                                          _ptr(k_cache), _ptr(v_cache), k_cache.shape[1], k_cache.shape[2],
                                          _ptr(k_rot_out) if k_rot_out is not None else None, float(base),
                                          _stream(stream)))


def rope_table(positions, head_dim: int, base: float = 10000.0, out=None, stream=None) -> torch.Tensor:
    """cos and sin of every RoPE angle at absolute `positions` [tokens]: a float32
    [tokens, head_dim/2, 2] table, the numbers rope_apply rotates with."""
    positions = _i32(positions, "positions")
    T = positions.numel()
    if out is None:
        out = torch.empty((T, head_dim // 2, 2), dtype=torch.float32, device=positions.device)
    elif out.dtype != torch.float32 or tuple(out.shape) != (T, head_dim // 2, 2) or not out.is_contiguous():
        raise ValueError("out must be a contiguous float32 [tokens, head_dim/2, 2] tensor")
    _check(library().rope_table(_ptr(positions), T, int(head_dim), float(base), _ptr(out), _stream(stream)))
    return out


def attn_kv_append_paged_int8(k_new, v_new, positions, slots, k_cache, v_cache, k_scale, v_scale, *,
                              k_rot_out=None, base: float = 10000.0, stream=None) -> None:
    """attn_kv_append_paged into an INT8 cache: code caches [Hkv, num_pages, page, 128]
    int8 and scales [Hkv, num_pages, page] fp32; keys rotated and rounded to bf16,
    then every row quantised (scale = max|x| / 127)."""
    for t, n in ((k_new, "k_new"), (v_new, "v_new")):
        if not t.is_contiguous() or t.dtype != torch.bfloat16:
            raise ValueError(f"{n} must be contiguous bf16")
    T, hkv, d = k_new.shape
    if tuple(v_new.shape) != (T, hkv, d):
        raise ValueError("v_new must have k_new's shape")
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        if t.dtype != torch.int8 or not t.is_contiguous() or t.dim() != 4 or t.shape[0] != hkv or t.shape[3] != d:
            raise ValueError(f"{n} must be a contiguous int8 [Hkv, num_pages, page, d] tensor")
    for t, n in ((k_scale, "k_scale"), (v_scale, "v_scale")):
        if t.dtype != torch.float32 or not t.is_contiguous() or tuple(t.shape) != tuple(k_cache.shape[:3]):
            raise ValueError(f"{n} must be a contiguous float32 [Hkv, num_pages, page] tensor")
    if k_rot_out is not None and (tuple(k_rot_out.shape) != (T, hkv, d) or not k_rot_out.is_contiguous()
                                  or k_rot_out.dtype != torch.bfloat16):
        raise ValueError("k_rot_out must be contiguous bf16 shaped like k_new")
    slots = _i32(slots, "slots")
    if slots.numel() != T:
        raise ValueError("slots must hold one entry per token")
    pos_ptr = None
    if base > 0:
        positions = _i32(positions, "positions")
        if positions.numel() != T:
            raise ValueError("positions must hold one entry per token")
        pos_ptr = _ptr(positions)
    _check(library().attn_kv_append_paged_int8(
        _ptr(k_new), _ptr(v_new), pos_ptr, _ptr(slots), T, hkv, d, _ptr(k_cache), _ptr(v_cache), _ptr(k_scale),
        _ptr(v_scale), k_cache.shape[1], k_cache.shape[2], _ptr(k_rot_out) if k_rot_out is not None else None,
        float(base), _stream(stream)))


def quant_fp8_rows(x, stream=None):
    """e4m3 codes of x [tokens, heads, 128] bf16 with one scale per (token, head) row:
    returns (codes as torch.float8_e4m3fn [tokens, heads, 128], scales [tokens, heads])."""
    if x.dtype != torch.bfloat16 or not x.is_contiguous() or x.dim() != 3:
        raise ValueError("x must be a contiguous bf16 [tokens, heads, head_dim] tensor")
    T, H, d = x.shape
    codes = torch.empty((T, H, d), dtype=torch.uint8, device=x.device)
    scales = torch.empty((T, H), dtype=torch.float32, device=x.device)
    _check(library().quant_fp8_rows(_ptr(x), T, H, d, _ptr(codes), _ptr(scales), _stream(stream)))
    return codes.view(torch.float8_e4m3fn), scales


def quant_fp8_heads(x, transposed: bool = False, stream=None):
    """e4m3 codes of x [tokens, heads, 128] bf16 with one scale per head: returns (codes,
    scales [heads]); codes are [tokens, heads, 128], or [heads, 128, t_stride] with
    t_stride = tokens rounded up to 16 when transposed (the layout the FP8 prefill
    reads its values in)."""
    if x.dtype != torch.bfloat16 or not x.is_contiguous() or x.dim() != 3:
        raise ValueError("x must be a contiguous bf16 [tokens, heads, head_dim] tensor")
    T, H, d = x.shape
    t_stride = (T + 15) // 16 * 16
    shape = (H, d, t_stride) if transposed else (T, H, d)
    codes = torch.empty(shape, dtype=torch.uint8, device=x.device)
    scales = torch.empty((H,), dtype=torch.float32, device=x.device)
    scratch = torch.empty((H,), dtype=torch.int32, device=x.device)
    _check(library().quant_fp8_heads(_ptr(x), T, H, d, _ptr(codes), _ptr(scales), _ptr(scratch),
                                     1 if transposed else 0, t_stride, _stream(stream)))
    return codes.view(torch.float8_e4m3fn), scales


def rope_quant_fp8_rows(x, positions, base: float = 10000.0, stream=None):
    """RoPE at `positions` fused into quant_fp8_rows (x is not modified): returns
    (codes float8_e4m3fn [tokens, heads, 128], scales [tokens, heads])."""
    if x.dtype != torch.bfloat16 or not x.is_contiguous() or x.dim() != 3:
        raise ValueError("x must be a contiguous bf16 [tokens, heads, head_dim] tensor")
    T, H, d = x.shape
    codes = torch.empty((T, H, d), dtype=torch.uint8, device=x.device)
    scales = torch.empty((T, H), dtype=torch.float32, device=x.device)
    _check(library().rope_quant_fp8_rows(_ptr(x), T, H, d, _ptr(_i32(positions, "positions")), float(base),
                                         _ptr(codes), _ptr(scales), _stream(stream)))
    return codes.view(torch.float8_e4m3fn), scales


def rope_quant_fp8_heads(x, positions, base: float = 10000.0, stream=None):
    """RoPE at `positions` fused into quant_fp8_heads, row layout (x is not modified):
    returns (codes float8_e4m3fn [tokens, heads, 128], scales [heads])."""
    if x.dtype != torch.bfloat16 or not x.is_contiguous() or x.dim() != 3:
        raise ValueError("x must be a contiguous bf16 [tokens, heads, head_dim] tensor")
    T, H, d = x.shape
    codes = torch.empty((T, H, d), dtype=torch.uint8, device=x.device)
    scales = torch.empty((H,), dtype=torch.float32, device=x.device)
    scratch = torch.empty((H,), dtype=torch.int32, device=x.device)
    _check(library().rope_quant_fp8_heads(_ptr(x), T, H, d, _ptr(_i32(positions, "positions")), float(base),
                                          _ptr(codes), _ptr(scales), _ptr(scratch), _stream(stream)))
    return codes.view(torch.float8_e4m3fn), scales


def attn_prefill(q, k, v, out, lse, cu_q, q_pos, max_seqlen_q: int, *, cu_k=None, k_pos=None,
                 page_table=None, k_lens=None, num_pages: int = 0, h_lo: int = 0,
                 h_hi: Optional[int] = None, scale: Optional[float] = None, causal: bool = True,
                 q_rope_cs=None, stream=None) -> None:
    """Tiled causal GQA attention.  q [Tq, Hq, d]; contiguous k/v [Tk, Hkv, d] with
    cu_k/k_pos, or head-major paged caches [Hkv, num_pages, page, d] with
    page_table [B, max_pages] and k_lens [B].  Writes out [Tq, Hq, d] and lse [Tq, Hq]
    (if given) for query heads [h_lo, h_hi).  With q_rope_cs (from rope_table over
    q_pos) q holds unrotated queries and the kernel rotates them itself
    (attn_prefill_rope_q)."""
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (out, "out")):
        if not t.is_contiguous():
            raise ValueError(f"{n} must be contiguous")
    Tq, hq, d = q.shape
    paged = page_table is not None
    if paged:
        hkv, npg, page, dk = k.shape
        max_pages = page_table.shape[1]
        num_pages = num_pages or npg
        total_k = 0
    else:
        Tk, hkv, dk = k.shape
        page, max_pages, total_k = 0, 0, Tk
    if dk != d or v.shape != k.shape or out.shape != q.shape:
        raise ValueError("inconsistent q/k/v/out shapes")
    if lse is not None and (lse.dtype != torch.float32 or tuple(lse.shape) != (Tq, hq) or not lse.is_contiguous()):
        raise ValueError("lse must be a contiguous float32 [Tq, Hq] tensor")
    if q.dtype != k.dtype or q.dtype != v.dtype:
        raise ValueError("q, k and v must share a dtype")
    h_hi = hq if h_hi is None else h_hi
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    cu_q = _i32(cu_q, "cu_q")
    B = cu_q.numel() - 1
    args = [_ptr(q), _ptr(k), _ptr(v), _ptr(out), _dt(out), _ptr(lse), _dt(q), B, _ptr(cu_q),
            _ptr(_i32(q_pos, "q_pos")), Tq, int(max_seqlen_q), _ptr(_i32(cu_k, "cu_k")),
            _ptr(_i32(k_pos, "k_pos")), total_k, _ptr(_i32(page_table, "page_table")),
            _ptr(_i32(k_lens, "k_lens")), max_pages, page, int(num_pages), hq, hkv, d, int(h_lo),
            int(h_hi), float(scale), 1 if causal else 0]
    if q_rope_cs is None:
        _check(library().attn_prefill(*args, _stream(stream)))
    else:
        if q_rope_cs.dtype != torch.float32 or tuple(q_rope_cs.shape) != (Tq, d // 2, 2) \
                or not q_rope_cs.is_contiguous():
            raise ValueError("q_rope_cs must be a contiguous float32 [Tq, d/2, 2] table (rope_table)")
        _check(library().attn_prefill_rope_q(*args, _ptr(q_rope_cs), _stream(stream)))


def attn_prefill_fp8(q, q_scale, k, k_scale, v_t, v_scale, out, lse, cu_q, q_pos, max_seqlen_q: int, cu_k, k_pos,
                     *, h_lo: int = 0, h_hi: Optional[int] = None, scale: Optional[float] = None,
                     causal: bool = True, stream=None) -> None:
    """Tiled causal GQA attention on e4m3 codes (quant_fp8_rows for q, quant_fp8_heads for
    k and, transposed, v).  q [Tq, Hq, 128] with q_scale [Tq, Hq]; k [Tk, Hkv, 128] with
    k_scale [Hkv]; v_t [Hkv, 128, t_stride] with v_scale [Hkv].  Every key sequence must
    start at a multiple of 16 tokens.  Writes out [Tq, Hq, 128] (bf16 or fp32) and lse."""
    for t, n in ((q, "q"), (k, "k"), (v_t, "v_t"), (out, "out"), (q_scale, "q_scale"), (k_scale, "k_scale"),
                 (v_scale, "v_scale")):
        if not t.is_contiguous():
            raise ValueError(f"{n} must be contiguous")
    for t, n in ((q, "q"), (k, "k"), (v_t, "v_t")):
        if t.dtype not in (torch.float8_e4m3fn, torch.uint8):
            raise ValueError(f"{n} must hold e4m3 codes (float8_e4m3fn or uint8)")
    for t, n in ((q_scale, "q_scale"), (k_scale, "k_scale"), (v_scale, "v_scale")):
        if t.dtype != torch.float32:
            raise ValueError(f"{n} must be float32")
    Tq, hq, d = q.shape
    Tk, hkv, dk = k.shape
    if dk != d or out.shape != q.shape or tuple(v_t.shape[:2]) != (hkv, d) or v_t.dim() != 3:
        raise ValueError("inconsistent q/k/v_t/out shapes")
    if tuple(q_scale.shape) != (Tq, hq) or tuple(k_scale.shape) != (hkv,) or tuple(v_scale.shape) != (hkv,):
        raise ValueError("q_scale must be [Tq, Hq]; k_scale and v_scale [Hkv]")
    if lse is not None and (lse.dtype != torch.float32 or tuple(lse.shape) != (Tq, hq) or not lse.is_contiguous()):
        raise ValueError("lse must be a contiguous float32 [Tq, Hq] tensor")
    h_hi = hq if h_hi is None else h_hi
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    cu_q = _i32(cu_q, "cu_q")
    _check(library().attn_prefill_fp8(
        _ptr(q), _ptr(q_scale), _ptr(k), _ptr(k_scale), _ptr(v_t), _ptr(v_scale), v_t.shape[2], _ptr(out),
        _dt(out), _ptr(lse), cu_q.numel() - 1, _ptr(cu_q), _ptr(_i32(q_pos, "q_pos")), Tq, int(max_seqlen_q),
        _ptr(_i32(cu_k, "cu_k")), _ptr(_i32(k_pos, "k_pos")), Tk, hq, hkv, d, int(h_lo), int(h_hi), float(scale),
        1 if causal else 0, _stream(stream)))


def prefill(q, k, v, cu_q, q_pos, max_seqlen_q: int, out_dtype=None, with_lse: bool = True, **kw):
    """attn_prefill with freshly allocated out (dtype of q unless given) and lse."""
    out = torch.empty(q.shape, dtype=out_dtype or q.dtype, device=q.device)
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device=q.device) if with_lse else None
    attn_prefill(q, k, v, out, lse, cu_q, q_pos, max_seqlen_q, **kw)
    return out, lse


def decode_workspace(batch: int, num_q_heads: int, num_splits: int, head_dim: int, device):
    """Partial-output workspaces for attn_decode_paged."""
    return (torch.empty((batch, num_q_heads, num_splits, head_dim), dtype=torch.float32, device=device),
            torch.empty((batch, num_q_heads, num_splits), dtype=torch.float32, device=device))


def attn_decode_paged(q, k_cache, v_cache, page_table, ctx_lens, num_splits: int, part_out, part_lse,
                      out=None, lse=None, scale: Optional[float] = None, stream=None) -> None:
    """Split-KV decode.  q [B, Hq, d] bf16 (rotated); caches [Hkv, num_pages, page, d] bf16;
    page_table [B, max_pages]; ctx_lens [B]; partial workspaces from decode_workspace()."""
    B, hq, d = q.shape
    hkv, npg, page, dk = k_cache.shape
    if dk != d or v_cache.shape != k_cache.shape:
        raise ValueError("inconsistent cache shapes")
    for t, n in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache"), (part_out, "part_out"),
                 (part_lse, "part_lse")):
        if not t.is_contiguous():
            raise ValueError(f"{n} must be contiguous")
    if tuple(part_out.shape) != (B, hq, num_splits, d) or tuple(part_lse.shape) != (B, hq, num_splits):
        raise ValueError("workspace shapes must be [B, Hq, splits, d] and [B, Hq, splits]")
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    page_table = _i32(page_table, "page_table")
    _check(library().attn_decode_paged(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(page_table), _ptr(_i32(ctx_lens, "ctx_lens")), B,
        page_table.shape[1], page, npg, hq, hkv, d, int(num_splits), float(scale), _ptr(part_out),
        _ptr(part_lse), _ptr(out), _dt(out) if out is not None else 0, _ptr(lse), _stream(stream)))


def attn_decode_paged_int8(q, k_cache, v_cache, k_scale, v_scale, page_table, ctx_lens, num_splits: int,
                           part_out, part_lse, out=None, lse=None, scale: Optional[float] = None,
                           stream=None) -> None:
    """Split-KV decode over an INT8 cache.  q [B, Hq, d] bf16 (rotated); code caches
    [Hkv, num_pages, page, d] int8 and scales [Hkv, num_pages, page] fp32 (value =
    code * scale); page_table [B, max_pages]; ctx_lens [B]; partial workspaces from
    decode_workspace()."""
    B, hq, d = q.shape
    hkv, npg, page, dk = k_cache.shape
    if dk != d or v_cache.shape != k_cache.shape:
        raise ValueError("inconsistent cache shapes")
    if k_cache.dtype != torch.int8 or v_cache.dtype != torch.int8:
        raise ValueError("code caches must be int8")
    for t, n in ((k_scale, "k_scale"), (v_scale, "v_scale")):
        if t.dtype != torch.float32 or tuple(t.shape) != (hkv, npg, page) or not t.is_contiguous():
            raise ValueError(f"{n} must be a contiguous float32 [Hkv, num_pages, page] tensor")
    for t, n in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache"), (part_out, "part_out"),
                 (part_lse, "part_lse")):
        if not t.is_contiguous():
            raise ValueError(f"{n} must be contiguous")
    if tuple(part_out.shape) != (B, hq, num_splits, d) or tuple(part_lse.shape) != (B, hq, num_splits):
        raise ValueError("workspace shapes must be [B, Hq, splits, d] and [B, Hq, splits]")
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    page_table = _i32(page_table, "page_table")
    _check(library().attn_decode_paged_int8(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale), _ptr(page_table),
        _ptr(_i32(ctx_lens, "ctx_lens")), B, page_table.shape[1], page, npg, hq, hkv, d, int(num_splits),
        float(scale), _ptr(part_out), _ptr(part_lse), _ptr(out), _dt(out) if out is not None else 0, _ptr(lse),
        _stream(stream)))


def attn_lse_merge(part_out, part_lse, out, lse=None, stream=None) -> None:
    """Merge partials part_out [P, rows, H, d] / part_lse [P, rows, H] (any strides, fp32)
    into out [rows, H, d] and lse [rows, H]."""
    P, rows, H, d = part_out.shape
    if tuple(part_lse.shape) != (P, rows, H) or part_out.stride(3) != 1:
        raise ValueError("part_lse must be [P, rows, H] and part_out's last dim contiguous")
    if part_out.dtype != torch.float32 or part_lse.dtype != torch.float32:
        raise ValueError("partials must be float32")
    if not out.is_contiguous() or tuple(out.shape) != (rows, H, d):
        raise ValueError("out must be a contiguous [rows, H, d] tensor")
    so, sl = part_out.stride(), part_lse.stride()
    _check(library().attn_lse_merge(_ptr(part_out), _ptr(part_lse), P, rows, H, d, so[0], so[1], so[2], sl[0],
                                    sl[1], sl[2], _ptr(out), _dt(out), _ptr(lse), _stream(stream)))
