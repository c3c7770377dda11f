"""fp64 CPU oracle for the decode-attention path -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  The CUDA
library never calls it and shares no code with it; the product path fails
loudly when its extension is missing instead of falling back to this.

The arithmetic lives in ``gqaq_oracle.c`` (plain C, fp64, single thread).
This module compiles it with gcc, loads it with ctypes and marshals numpy
arrays in and out, one sequence at a time.  fp16 inputs are decoded by the
C file's own bit-field routine.

Sources: "Core ML Decode Optimization: Removing the 1.9 GiB Per-Token Copy
Caused by GQA repeat_kv" (OptAI), sections 2-3 (repeat_kv and Q folding);
"Quest: Query-Aware Sparsity for Efficient Long-Context LLM Inference"
(reviewer's summary), the page-score, token-budget and bytes-model sections.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gqaq_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

_dp = ctypes.POINTER(ctypes.c_double)
_ip = ctypes.POINTER(ctypes.c_int32)
_up = ctypes.POINTER(ctypes.c_uint16)


def build(force: bool = False) -> str:
    """Compile the C oracle into ``oracle/liboracle.so`` (gcc, no CUDA)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call([
            "gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fPIC", "-shared",
            _SRC, "-o", tmp, "-lm",
        ])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        i64, i32, dbl = ctypes.c_int64, ctypes.c_int, ctypes.c_double
        lib.oracle_f16_to_f64.argtypes = [ctypes.c_uint16]
        lib.oracle_f16_to_f64.restype = dbl
        lib.oracle_f16_array_to_f64.argtypes = [_up, _dp, i64]
        lib.oracle_f16_array_to_f64.restype = None
        u8p = ctypes.POINTER(ctypes.c_uint8)
        lib.oracle_e4m3_array_to_f64.argtypes = [u8p, _dp, i64]
        lib.oracle_e4m3_array_to_f64.restype = None
        lib.oracle_f32_array_to_e4m3.argtypes = [ctypes.POINTER(ctypes.c_float), u8p, i64]
        lib.oracle_f32_array_to_e4m3.restype = None
        for name in ("oracle_attn_repeat_kv", "oracle_attn_folded"):
            fn = getattr(lib, name)
            fn.argtypes = [i32, i32, i32, i64, i64, _dp, _dp, _dp, dbl, _dp]
            fn.restype = i32
        fp = ctypes.POINTER(ctypes.c_float)
        lib.oracle_int4_quantize_rows.argtypes = [fp, i64, i32, u8p, fp]
        lib.oracle_int4_quantize_rows.restype = None
        lib.oracle_int4_dequantize_rows.argtypes = [u8p, fp, i64, i32, _dp]
        lib.oracle_int4_dequantize_rows.restype = None
        lib.oracle_prefill_repeat_kv.argtypes = [i32, i32, i32, i64, i32, i64, _dp, _dp, _dp, dbl, _dp]
        lib.oracle_prefill_repeat_kv.restype = i32
        lib.oracle_page_minmax.argtypes = [i32, i32, i64, i64, i32, _dp, _dp]
        lib.oracle_page_minmax.restype = i32
        lib.oracle_page_minmax_e4m3.argtypes = [i32, i32, i64, i64, i32, u8p, u8p]
        lib.oracle_page_minmax_e4m3.restype = i32
        lib.oracle_page_scores.argtypes = [i32, i32, i32, i64, i64, _dp, _dp, _dp]
        lib.oracle_page_scores.restype = i32
        lib.oracle_topk_pages.argtypes = [i32, i64, i64, i32, _dp, _ip]
        lib.oracle_topk_pages.restype = i32
        lib.oracle_sparse_attn.argtypes = [i32, i32, i32, i64, i64, i32, i32,
                                           _dp, _dp, _dp, _ip, dbl, _dp]
        lib.oracle_sparse_attn.restype = i32
        _lib = lib
    return _lib


def _dptr(a: np.ndarray):
    assert a.dtype == np.float64 and a.flags.c_contiguous
    return a.ctypes.data_as(_dp)


def _iptr(a: np.ndarray):
    assert a.dtype == np.int32 and a.flags.c_contiguous
    return a.ctypes.data_as(_ip)


def _check(rc: int, what: str):
    if rc != 0:
        raise ValueError(f"oracle {what} rejected its arguments (rc={rc})")


# --------------------------------------------------------------------------
# fp16 decoding (the C file's own bit-field routine)
# --------------------------------------------------------------------------
def f16_to_f64(a) -> np.ndarray:
    """Decode an fp16 array (np.float16 or raw uint16 bits) to float64."""
    a = np.ascontiguousarray(a)
    bits = a.view(np.uint16) if a.dtype == np.float16 else a.astype(np.uint16, copy=False)
    bits = np.ascontiguousarray(bits)
    out = np.empty(bits.shape, dtype=np.float64)
    _load().oracle_f16_array_to_f64(bits.ctypes.data_as(_up), _dptr(out), bits.size)
    return out


def e4m3_to_f64(codes) -> np.ndarray:
    """Decode E4M3 codes (uint8) to float64 (the fp8 KV-cache variant)."""
    c = np.ascontiguousarray(np.asarray(codes, dtype=np.uint8))
    out = np.empty(c.shape, dtype=np.float64)
    _load().oracle_e4m3_array_to_f64(c.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8)), _dptr(out), c.size)
    return out


def quantize_e4m3(x, inv_scale: float) -> np.ndarray:
    """E4M3 codes of fp16 values x: round(fp32(x) * fp32(inv_scale)) to the
    nearest E4M3 value (ties to even), magnitudes above 448 saturated. The
    product is taken in fp32, as the GPU takes it, so both sides round the
    same value."""
    y = np.ascontiguousarray(_as_f64(x).astype(np.float32) * np.float32(inv_scale), dtype=np.float32)
    out = np.empty(y.shape, dtype=np.uint8)
    _load().oracle_f32_array_to_e4m3(y.ctypes.data_as(ctypes.POINTER(ctypes.c_float)),
                                     out.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8)), y.size)
    return out


def quantize_int4(x):
    """4-bit KV rows: x [..., D] (fp16 or fp32) -> (codes [..., D/2] uint8, scales [...] fp32).
    Symmetric INT4 per row: scale = amax / 7, q = clamp(rne(x / scale), -7, 7),
    nibble q + 8 (channel 2i in the low nibble of byte i); fp32 arithmetic."""
    y = np.ascontiguousarray(_as_f64(x).astype(np.float32))
    D = y.shape[-1]
    rows = y.size // D
    codes = np.empty(y.shape[:-1] + (D // 2,), dtype=np.uint8)
    scales = np.empty(y.shape[:-1], dtype=np.float32)
    fp = ctypes.POINTER(ctypes.c_float)
    _load().oracle_int4_quantize_rows(y.ctypes.data_as(fp), rows, D,
                                      codes.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8)), scales.ctypes.data_as(fp))
    return codes, scales


def dequantize_int4(codes, scales) -> np.ndarray:
    """(codes [..., D/2], scales [...]) -> values (nibble - 8) * scale, float64 [..., D]."""
    c = np.ascontiguousarray(np.asarray(codes, dtype=np.uint8))
    sc = np.ascontiguousarray(np.asarray(scales, dtype=np.float32))
    D = c.shape[-1] * 2
    out = np.empty(c.shape[:-1] + (D,), dtype=np.float64)
    fp = ctypes.POINTER(ctypes.c_float)
    _load().oracle_int4_dequantize_rows(c.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8)), sc.ctypes.data_as(fp),
                                        sc.size, D, _dptr(out))
    return out


def attn_int4(q, k_codes, k_scales, v_codes, v_scales, valid_len, scale):
    """fp64 decode attention over a 4-bit KV cache: dequantize, then attn_repeat_kv."""
    return attn_repeat_kv(q, dequantize_int4(k_codes, k_scales), dequantize_int4(v_codes, v_scales), valid_len, scale)


def _as_f64(a) -> np.ndarray:
    a = np.asarray(a)
    if a.dtype == np.float16:
        return f16_to_f64(a)
    return np.ascontiguousarray(a, dtype=np.float64)


# --------------------------------------------------------------------------
# Dense decode attention: explicit repeat_kv, and the folded form
# --------------------------------------------------------------------------
def _attn(fn_name, q, k, v, valid_len, scale):
    q = np.asarray(q); k = np.asarray(k); v = np.asarray(v)
    B, Hq, D = q.shape
    _, Hkv, Lmax, _ = k.shape
    out = np.empty((B, Hq, D), dtype=np.float64)
    fn = getattr(_load(), fn_name)
    for b in range(B):
        qb, kb, vb = _as_f64(q[b]), _as_f64(k[b]), _as_f64(v[b])
        ob = np.empty((Hq, D), dtype=np.float64)
        _check(fn(Hq, Hkv, D, Lmax, int(valid_len[b]), _dptr(qb), _dptr(kb), _dptr(vb),
                  float(scale), _dptr(ob)), fn_name)
        out[b] = ob
    return out


def attn_repeat_kv(q, k, v, valid_len, scale):
    """fp64 decode attention with an explicit repeat_kv copy per query head.

    q [B,Hq,D], k/v [B,Hkv,Lmax,D] (fp16 or fp64), valid_len [B] -> [B,Hq,D] fp64.
    """
    return _attn("oracle_attn_repeat_kv", q, k, v, valid_len, scale)


def attn_e4m3(q, k_codes, v_codes, k_scale: float, v_scale: float, valid_len, scale):
    """fp64 decode attention over an E4M3 KV cache: keys and values are the
    decoded codes times their per-tensor scales; then as attn_repeat_kv."""
    k = e4m3_to_f64(k_codes) * float(k_scale)
    v = e4m3_to_f64(v_codes) * float(v_scale)
    return attn_repeat_kv(q, k, v, valid_len, scale)


def prefill_attn(q, k, v, start, scale):
    """fp64 causal attention of a chunk of q_len new tokens per sequence
    ("Prefill Needs Separate Design": the group axis merged into the sequence
    axis, each row with its own mask), explicit repeat_kv.

    q [B,Hq,q_len,D]; k/v [B,Hkv,Lmax,D] already holding the chunk at rows
    start[b] .. start[b]+q_len-1; token t attends to rows 0 .. start[b]+t.
    Returns [B,Hq,q_len,D] fp64."""
    q = np.asarray(q); k = np.asarray(k); v = np.asarray(v)
    B, Hq, q_len, D = q.shape
    _, Hkv, Lmax, _ = k.shape
    out = np.empty((B, Hq, q_len, D), dtype=np.float64)
    lib = _load()
    for b in range(B):
        qb, kb, vb = _as_f64(q[b]), _as_f64(k[b]), _as_f64(v[b])
        ob = np.empty((Hq, q_len, D), dtype=np.float64)
        _check(lib.oracle_prefill_repeat_kv(Hq, Hkv, D, Lmax, q_len, int(start[b]), _dptr(qb), _dptr(kb), _dptr(vb),
                                            float(scale), _dptr(ob)), "oracle_prefill_repeat_kv")
        out[b] = ob
    return out


def attn_folded(q, k, v, valid_len, scale):
    """fp64 decode attention with Q read as [Hkv, G, D] (no KV copy)."""
    return _attn("oracle_attn_folded", q, k, v, valid_len, scale)


# --------------------------------------------------------------------------
# Quest: page metadata, page scores, top-K, sparse attention
# --------------------------------------------------------------------------
def num_pages(length: int, page_size: int) -> int:
    return (int(length) + page_size - 1) // page_size


def page_minmax(k, valid_len, page_size):
    """Per-page per-channel key min/max -> [B,Hkv,Pmax,2,D] fp64 (NaN where no valid token)."""
    k = np.asarray(k)
    B, Hkv, Lmax, D = k.shape
    pmax = num_pages(Lmax, page_size)
    out = np.full((B, Hkv, pmax, 2, D), np.nan, dtype=np.float64)
    for b in range(B):
        kb = _as_f64(k[b])
        mb = np.full((Hkv, pmax, 2, D), np.nan, dtype=np.float64)
        _check(_load().oracle_page_minmax(Hkv, D, Lmax, int(valid_len[b]), page_size,
                                          _dptr(kb), _dptr(mb)), "page_minmax")
        out[b] = mb
    return out


def page_minmax_e4m3(k_codes, valid_len, page_size):
    """Per-page per-channel min/max of an E4M3 key cache, as E4M3 codes
    [B,Hkv,Pmax,2,D] uint8 (compared by value; a zero bound is the code 0x00;
    pages with no valid token hold 0x7F, the NaN code)."""
    k = np.ascontiguousarray(np.asarray(k_codes, dtype=np.uint8))
    B, Hkv, Lmax, D = k.shape
    pmax = num_pages(Lmax, page_size)
    out = np.full((B, Hkv, pmax, 2, D), 0x7F, dtype=np.uint8)
    u8p = ctypes.POINTER(ctypes.c_uint8)
    for b in range(B):
        kb = np.ascontiguousarray(k[b])
        mb = np.ascontiguousarray(out[b])
        _check(_load().oracle_page_minmax_e4m3(Hkv, D, Lmax, int(valid_len[b]), page_size,
                                               kb.ctypes.data_as(u8p), mb.ctypes.data_as(u8p)), "page_minmax_e4m3")
        out[b] = mb
    return out


def page_scores(q, meta, valid_len, page_size):
    """U(p,q) per KV head (max over the G folded query heads) -> [B,Hkv,Pmax] fp64."""
    q = np.asarray(q)
    meta = np.ascontiguousarray(meta, dtype=np.float64)
    B, Hq, D = q.shape
    _, Hkv, pmax, _, _ = meta.shape
    out = np.empty((B, Hkv, pmax), dtype=np.float64)
    for b in range(B):
        qb = _as_f64(q[b])
        mb = np.ascontiguousarray(meta[b])
        sb = np.empty((Hkv, pmax), dtype=np.float64)
        _check(_load().oracle_page_scores(Hq, Hkv, D, pmax, num_pages(valid_len[b], page_size),
                                          _dptr(qb), _dptr(mb), _dptr(sb)), "page_scores")
        out[b] = sb
    return out


def topk_pages(scores, valid_len, page_size, k):
    """Sort-based top-K: [B,Hkv,Pmax] scores -> [B,Hkv,K] int32, ascending, -1 padded."""
    scores = np.ascontiguousarray(scores, dtype=np.float64)
    B, Hkv, pmax = scores.shape
    out = np.empty((B, Hkv, k), dtype=np.int32)
    for b in range(B):
        sb = np.ascontiguousarray(scores[b])
        ib = np.empty((Hkv, k), dtype=np.int32)
        _check(_load().oracle_topk_pages(Hkv, pmax, num_pages(valid_len[b], page_size), int(k),
                                         _dptr(sb), _iptr(ib)), "topk_pages")
        out[b] = ib
    return out


def sparse_attn(q, k, v, valid_len, page_idx, page_size, scale):
    """fp64 attention over the tokens of the listed pages only -> [B,Hq,D]."""
    q = np.asarray(q); k = np.asarray(k); v = np.asarray(v)
    page_idx = np.ascontiguousarray(page_idx, dtype=np.int32)
    B, Hq, D = q.shape
    _, Hkv, Lmax, _ = k.shape
    kp = page_idx.shape[2]
    out = np.empty((B, Hq, D), dtype=np.float64)
    for b in range(B):
        qb, kb, vb = _as_f64(q[b]), _as_f64(k[b]), _as_f64(v[b])
        ib = np.ascontiguousarray(page_idx[b])
        ob = np.empty((Hq, D), dtype=np.float64)
        _check(_load().oracle_sparse_attn(Hq, Hkv, D, Lmax, int(valid_len[b]), page_size, kp,
                                          _dptr(qb), _dptr(kb), _dptr(vb), _iptr(ib),
                                          float(scale), _dptr(ob)), "sparse_attn")
        out[b] = ob
    return out


# --------------------------------------------------------------------------
# Bytes model ("how the bytes read shrink"): M bytes per key or value vector
# --------------------------------------------------------------------------
def bytes_full(M: int, L: int) -> int:
    """D_full = 2 M L: reading every key and value once."""
    return 2 * M * L


def bytes_meta(M: int, L: int, S: int) -> float:
    """D_metadata ~ 2 M L / S: one min and one max vector per page."""
    return 2 * M * L / S


def bytes_selected(M: int, K: int, S: int) -> int:
    """D_selected ~ 2 M K S: keys and values of K full pages."""
    return 2 * M * K * S


def token_budget(K: int, S: int) -> int:
    """B = K S tokens for K full pages of S tokens."""
    return K * S


def quest_read_ratio(L: int, S: int, K: int) -> float:
    """D_Quest / D_full ~ 1/S + K S / L."""
    return 1.0 / S + K * S / L
