"""GB300 (sm_103a) decode attention: GQA query-head folding + Quest page sparsity.

A thin ctypes binding over the C ABI in ``include/gqaq.h`` (``libgqaq.so``).
Every function here only marshals arguments: it reads shapes and pointers
from torch tensors, builds a ``gqaq_dims``, passes
``torch.cuda.current_stream()`` and raises ``GqaqError`` on a non-zero status.
All arithmetic runs in the library's CUDA kernels. When the library is
missing, the import still succeeds but every call raises: there is no CPU
fallback.

Function names follow the C ABI: gqa_decode_attn, quest_append_kv,
quest_update_meta, quest_score_pages, quest_topk_pages, quest_sparse_attn,
quest_decode_attn, the 8-bit cache calls gqa_decode_attn_e4m3 /
kv_append_e4m3 and their Quest counterparts (quest_append_kv_e4m3,
quest_update_meta_e4m3, quest_score_pages_e4m3, quest_sparse_attn_e4m3), the
4-bit pair and prefill.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libgqaq.so")

GQAQ_OK = 0
GQAQ_ERR_INVALID_ARG = 1
GQAQ_ERR_UNSUPPORTED = 2
GQAQ_ERR_WORKSPACE = 3
GQAQ_ERR_CUDA = 4
GQAQ_ERR_TIMEOUT = 5

GQAQ_DEV_TIMEOUT = 1
GQAQ_DEV_BAD_LEN = 2
GQAQ_DEV_BAD_PAGE = 4
GQAQ_DEV_BAD_POS = 8

GQAQ_OPT_MAX_CTAS = 1
GQAQ_OPT_WAIT_TIMEOUT_NS = 2
GQAQ_OPT_TEST_STALL = 3
GQAQ_OPT_CLUSTER_SIZE = 4
GQAQ_OPT_PDL = 5
GQAQ_OPT_QUEST_KERNEL = 6
GQAQ_OPT_PREFILL_SPLITS = 7
GQAQ_OPT_PREFILL_KERNEL = 8
GQAQ_OPT_QUEST_EARLY_META = 9
GQAQ_OPT_DENSE_EARLY_KV = 10

PAGE_SIZE = 16


class GqaqError(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn} failed: {msg} ({status})")
        self.status = status


class Dims(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int), ("num_q_heads", ctypes.c_int),
                ("num_kv_heads", ctypes.c_int), ("head_dim", ctypes.c_int),
                ("max_len", ctypes.c_int), ("page_size", ctypes.c_int)]


# Exported symbols, in the order include/gqaq.h declares them.
EXPORTS = ("gqaq_workspace_bytes", "gqa_decode_attn", "quest_append_kv", "quest_update_meta",
           "quest_score_pages", "quest_topk_pages", "quest_sparse_attn", "quest_decode_attn",
           "gqa_decode_attn_noalloc", "gqa_decode_attn_e4m3", "kv_append_e4m3",
           "quest_append_kv_e4m3", "quest_update_meta_e4m3", "quest_score_pages_e4m3", "quest_sparse_attn_e4m3",
           "quest_decode_attn_e4m3",
           "gqa_decode_attn_int4", "kv_append_int4",
           "gqaq_prefill_workspace_bytes", "gqa_prefill_attn",
           "gqaq_status_string", "gqaq_set_option", "gqaq_device_status", "gqaq_version")

_lib = None


def lib():
    """Load ``libgqaq.so`` (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, dp = ctypes.c_void_p, ctypes.c_int, ctypes.POINTER(Dims)
        L.gqaq_workspace_bytes.argtypes = [dp, i32]
        L.gqaq_workspace_bytes.restype = ctypes.c_size_t
        L.gqa_decode_attn.argtypes = [dp, vp, vp, vp, vp, ctypes.c_float, vp, vp, ctypes.c_size_t, vp]
        L.quest_append_kv.argtypes = [dp, vp, vp, vp, vp, vp, vp, vp]
        L.quest_update_meta.argtypes = [dp, vp, vp, vp, i32, i32, vp]
        L.quest_score_pages.argtypes = [dp, vp, vp, vp, vp, vp]
        L.quest_topk_pages.argtypes = [dp, vp, vp, i32, vp, vp, ctypes.c_size_t, vp]
        L.quest_sparse_attn.argtypes = [dp, vp, vp, vp, vp, vp, i32, ctypes.c_float, vp, vp,
                                        ctypes.c_size_t, vp]
        L.quest_decode_attn.argtypes = [dp, vp, vp, vp, vp, vp, vp, vp, vp, i32, ctypes.c_float, vp, vp, vp,
                                        vp, ctypes.c_size_t, vp]
        L.gqa_decode_attn_noalloc.argtypes = [dp, vp, vp, vp, vp, ctypes.c_float, vp, vp]
        f32 = ctypes.c_float
        L.gqa_decode_attn_e4m3.argtypes = [dp, vp, vp, vp, f32, f32, vp, f32, vp, vp, ctypes.c_size_t, vp]
        L.kv_append_e4m3.argtypes = [dp, vp, vp, vp, vp, vp, f32, f32, vp]
        L.quest_append_kv_e4m3.argtypes = [dp, vp, vp, vp, vp, vp, vp, f32, f32, vp]
        L.quest_update_meta_e4m3.argtypes = [dp, vp, vp, vp, i32, i32, vp]
        L.quest_score_pages_e4m3.argtypes = [dp, vp, vp, f32, vp, vp, vp]
        L.quest_sparse_attn_e4m3.argtypes = [dp, vp, vp, vp, f32, f32, vp, vp, i32, f32, vp, vp, ctypes.c_size_t, vp]
        L.quest_decode_attn_e4m3.argtypes = [dp, vp, vp, vp, vp, vp, vp, vp, f32, f32, f32, f32, vp, i32, f32, vp, vp,
                                             vp, vp]
        L.gqa_decode_attn_int4.argtypes = [dp, vp, vp, vp, vp, vp, vp, f32, vp, vp, ctypes.c_size_t, vp]
        L.kv_append_int4.argtypes = [dp, vp, vp, vp, vp, vp, vp, vp, vp]
        L.gqaq_prefill_workspace_bytes.argtypes = [dp, i32]
        L.gqaq_prefill_workspace_bytes.restype = ctypes.c_size_t
        L.gqa_prefill_attn.argtypes = [dp, i32, vp, vp, vp, vp, f32, vp, vp, ctypes.c_size_t, vp]
        L.gqaq_status_string.argtypes = [i32]
        L.gqaq_status_string.restype = ctypes.c_char_p
        L.gqaq_set_option.argtypes = [i32, ctypes.c_int64]
        L.gqaq_device_status.argtypes = [ctypes.POINTER(ctypes.c_int), i32]
        L.gqaq_version.argtypes = []
        for name in EXPORTS:
            if name not in ("gqaq_workspace_bytes", "gqaq_status_string", "gqaq_prefill_workspace_bytes"):
                getattr(L, name).restype = ctypes.c_int
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().gqaq_status_string(int(status)).decode()


def _check(fn: str, status: int):
    if status != GQAQ_OK:
        raise GqaqError(fn, status, status_string(status))


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(t: torch.Tensor):
    return ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)


def _need(t: torch.Tensor, name: str, dtype, ndim: int):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (the library has no CPU path)")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _shape(t: torch.Tensor, name: str, shape):
    """The library reads and writes whole buffers of these shapes: refuse any other."""
    if tuple(t.shape) != tuple(int(x) for x in shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def _meta_shape(meta, B, Hkv, Lmax, D, page_size):
    _shape(meta, "meta", (B, Hkv, num_pages(Lmax, page_size), 2, D))


def _new_rows(k_new, v_new, pos, B, Hkv, D):
    _shape(k_new, "k_new", (B, Hkv, D))
    _shape(v_new, "v_new", (B, Hkv, D))
    _shape(pos, "pos", (B,))


def make_dims(batch, num_q_heads, num_kv_heads, head_dim, max_len, page_size=PAGE_SIZE) -> Dims:
    return Dims(int(batch), int(num_q_heads), int(num_kv_heads), int(head_dim), int(max_len),
                int(page_size))


def dims_of(q: torch.Tensor, k_cache: torch.Tensor, page_size: int = PAGE_SIZE) -> Dims:
    B, Hq, D = q.shape
    _, Hkv, Lmax, _ = k_cache.shape
    return make_dims(B, Hq, Hkv, D, Lmax, page_size)


def set_option(option: int, value: int):
    _check("gqaq_set_option", lib().gqaq_set_option(int(option), int(value)))


def device_status(reset: bool = True) -> int:
    """Return the current device's GQAQ_DEV_* flags (synchronises the device)."""
    flags = ctypes.c_int(0)
    rc = lib().gqaq_device_status(ctypes.byref(flags), 1 if reset else 0)
    if rc not in (GQAQ_OK, GQAQ_ERR_TIMEOUT):
        _check("gqaq_device_status", rc)
    return flags.value


def workspace_bytes(dims: Dims, max_selected_pages: int = 0) -> int:
    n = lib().gqaq_workspace_bytes(ctypes.byref(dims), int(max_selected_pages))
    if n == 0:
        raise GqaqError("gqaq_workspace_bytes", GQAQ_ERR_UNSUPPORTED, "dims rejected")
    return int(n)


def alloc_workspace(dims: Dims, device, max_selected_pages: int = 0) -> torch.Tensor:
    """Workspace for gqa_decode_attn / quest_sparse_attn, and with
    max_selected_pages = k also for quest_decode_attn's work-queue kernel.
    Zero-filled once, as the library asks; every call leaves its counters at
    zero again."""
    return torch.zeros(workspace_bytes(dims, max_selected_pages), dtype=torch.uint8, device=device)


def workspace_zero_bytes(dims: Dims) -> int:
    """Leading bytes of a workspace that hold counters and flags (zero between calls)."""
    return (256 + 12 * dims.batch * dims.num_kv_heads + 255) // 256 * 256


def num_pages(max_len: int, page_size: int = PAGE_SIZE) -> int:
    return (int(max_len) + page_size - 1) // page_size


# ---------------------------------------------------------------------------
# Entry points
# ---------------------------------------------------------------------------
def gqa_decode_attn(q, k_cache, v_cache, valid_len, scale: float, out=None, workspace=None):
    """Dense folded-GQA decode attention. q [B,Hq,D], caches [B,Hkv,Lmax,D] fp16."""
    _need(q, "q", torch.float16, 3)
    _need(k_cache, "k_cache", torch.float16, 4)
    _need(v_cache, "v_cache", torch.float16, 4)
    _need(valid_len, "valid_len", torch.int32, 1)
    d = dims_of(q, k_cache)
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", torch.float16, 3)
    if workspace is None:
        workspace = alloc_workspace(d, q.device)
    _check("gqa_decode_attn", lib().gqa_decode_attn(
        ctypes.byref(d), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(valid_len), float(scale),
        _ptr(out), _ptr(workspace), workspace.numel(), _stream(q)))
    return out


def quest_decode_attn(q, k_cache, v_cache, meta, valid_len, k: int, scale: float, k_new=None, v_new=None,
                      pos=None, out=None, scores=None, page_idx=None, page_size: int = PAGE_SIZE,
                      workspace=None):
    """Fused Quest step in one launch: optional append (k_new, v_new at pos),
    page scores, top-k pages and attention over them. scores/page_idx are
    optional outputs. With a workspace (alloc_workspace(dims, device, k)) the
    step runs as one GPU-wide work queue; without, one cluster per unit."""
    _need(q, "q", torch.float16, 3)
    _need(k_cache, "k_cache", torch.float16, 4)
    _need(v_cache, "v_cache", torch.float16, 4)
    _need(meta, "meta", torch.float16, 5)
    _need(valid_len, "valid_len", torch.int32, 1)
    if pos is not None:
        _need(k_new, "k_new", torch.float16, 3)
        _need(v_new, "v_new", torch.float16, 3)
        _need(pos, "pos", torch.int32, 1)
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", torch.float16, 3)
    if scores is not None:
        _need(scores, "scores", torch.float32, 3)
    if page_idx is not None:
        _need(page_idx, "page_idx", torch.int32, 3)
    d = dims_of(q, k_cache, page_size)
    _meta_shape(meta, d.batch, d.num_kv_heads, d.max_len, d.head_dim, page_size)
    _shape(valid_len, "valid_len", (d.batch,))
    _shape(v_cache, "v_cache", tuple(k_cache.shape))
    if pos is not None:
        _new_rows(k_new, v_new, pos, d.batch, d.num_kv_heads, d.head_dim)
    if scores is not None:
        _shape(scores, "scores", (d.batch, d.num_kv_heads, num_pages(d.max_len, page_size)))
    if page_idx is not None:
        _shape(page_idx, "page_idx", (d.batch, d.num_kv_heads, int(k)))
    _check("quest_decode_attn", lib().quest_decode_attn(
        ctypes.byref(d), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(meta), _ptr(k_new), _ptr(v_new),
        _ptr(pos), _ptr(valid_len), int(k), float(scale), _ptr(out), _ptr(scores), _ptr(page_idx),
        _ptr(workspace), 0 if workspace is None else workspace.numel(), _stream(q)))
    return out


def gqa_decode_attn_noalloc(q, k_cache, v_cache, valid_len, scale: float, out):
    """gqa_decode_attn without a workspace, for callers that cannot allocate
    device memory (the library keeps the scratch in its own fixed 1 MiB array).
    ``out`` must be given. Overlapping calls race on the shared scratch."""
    _need(q, "q", torch.float16, 3)
    _need(k_cache, "k_cache", torch.float16, 4)
    _need(v_cache, "v_cache", torch.float16, 4)
    _need(valid_len, "valid_len", torch.int32, 1)
    _need(out, "out", torch.float16, 3)
    d = dims_of(q, k_cache)
    _check("gqa_decode_attn_noalloc", lib().gqa_decode_attn_noalloc(
        ctypes.byref(d), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(valid_len), float(scale),
        _ptr(out), _stream(q)))
    return out


def gqa_decode_attn_e4m3(q, k_cache, v_cache, k_scale: float, v_scale: float, valid_len, scale: float,
                         out=None, workspace=None):
    """Dense folded-GQA decode attention over an E4M3 cache: k_cache / v_cache
    [B,Hkv,Lmax,D] uint8 codes, dequantized as code value * k_scale (v_scale)."""
    _need(q, "q", torch.float16, 3)
    _need(k_cache, "k_cache", torch.uint8, 4)
    _need(v_cache, "v_cache", torch.uint8, 4)
    _need(valid_len, "valid_len", torch.int32, 1)
    d = dims_of(q, k_cache)
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", torch.float16, 3)
    if workspace is None:
        workspace = alloc_workspace(d, q.device)
    _check("gqa_decode_attn_e4m3", lib().gqa_decode_attn_e4m3(
        ctypes.byref(d), _ptr(q), _ptr(k_cache), _ptr(v_cache), float(k_scale), float(v_scale), _ptr(valid_len),
        float(scale), _ptr(out), _ptr(workspace), workspace.numel(), _stream(q)))
    return out


def kv_append_e4m3(k_cache, v_cache, k_new, v_new, pos, k_inv_scale: float, v_inv_scale: float):
    """Quantize k_new/v_new [B,Hkv,D] fp16 to E4M3 (x * inv_scale, nearest-even,
    saturating) and write the codes at row pos[b] of the uint8 caches."""
    _need(k_cache, "k_cache", torch.uint8, 4)
    _need(v_cache, "v_cache", torch.uint8, 4)
    _need(k_new, "k_new", torch.float16, 3)
    _need(v_new, "v_new", torch.float16, 3)
    _need(pos, "pos", torch.int32, 1)
    B, Hkv, Lmax, D = k_cache.shape
    d = make_dims(B, Hkv, Hkv, D, Lmax)
    _check("kv_append_e4m3", lib().kv_append_e4m3(
        ctypes.byref(d), _ptr(k_cache), _ptr(v_cache), _ptr(k_new), _ptr(v_new), _ptr(pos), float(k_inv_scale),
        float(v_inv_scale), _stream(k_cache)))


def new_meta_e4m3(batch: int, num_kv_heads: int, max_len: int, head_dim: int, device,
                  page_size: int = PAGE_SIZE) -> torch.Tensor:
    """Allocate E4M3 page bounds [B,Hkv,Pmax,2,D] uint8 (contents undefined)."""
    return torch.empty(batch, num_kv_heads, num_pages(max_len, page_size), 2, head_dim, dtype=torch.uint8,
                       device=device)


def quest_append_kv_e4m3(k_cache, v_cache, meta, k_new, v_new, pos, k_inv_scale: float, v_inv_scale: float,
                         page_size: int = PAGE_SIZE):
    """kv_append_e4m3 plus the page's E4M3 bounds (meta [B,Hkv,Pmax,2,D] uint8)."""
    _need(k_cache, "k_cache", torch.uint8, 4)
    _need(v_cache, "v_cache", torch.uint8, 4)
    _need(meta, "meta", torch.uint8, 5)
    _need(k_new, "k_new", torch.float16, 3)
    _need(v_new, "v_new", torch.float16, 3)
    _need(pos, "pos", torch.int32, 1)
    B, Hkv, Lmax, D = k_cache.shape
    _shape(v_cache, "v_cache", tuple(k_cache.shape))
    _meta_shape(meta, B, Hkv, Lmax, D, page_size)
    _new_rows(k_new, v_new, pos, B, Hkv, D)
    d = make_dims(B, Hkv, Hkv, D, Lmax, page_size)
    _check("quest_append_kv_e4m3", lib().quest_append_kv_e4m3(
        ctypes.byref(d), _ptr(k_cache), _ptr(v_cache), _ptr(meta), _ptr(k_new), _ptr(v_new), _ptr(pos),
        float(k_inv_scale), float(v_inv_scale), _stream(k_cache)))


def quest_update_meta_e4m3(k_cache, valid_len, meta, page_begin: int = 0, page_end: Optional[int] = None,
                           page_size: int = PAGE_SIZE):
    """Rebuild the E4M3 page bounds of pages [page_begin, page_end) from the cache codes."""
    _need(k_cache, "k_cache", torch.uint8, 4)
    _need(valid_len, "valid_len", torch.int32, 1)
    _need(meta, "meta", torch.uint8, 5)
    B, Hkv, Lmax, D = k_cache.shape
    _meta_shape(meta, B, Hkv, Lmax, D, page_size)
    _shape(valid_len, "valid_len", (B,))
    d = make_dims(B, Hkv, Hkv, D, Lmax, page_size)
    if page_end is None:
        page_end = num_pages(Lmax, page_size)
    _check("quest_update_meta_e4m3", lib().quest_update_meta_e4m3(
        ctypes.byref(d), _ptr(k_cache), _ptr(valid_len), _ptr(meta), int(page_begin), int(page_end),
        _stream(k_cache)))
    return meta


def quest_score_pages_e4m3(q, meta, k_scale: float, valid_len, max_len: int, scores=None,
                           page_size: int = PAGE_SIZE):
    """k_scale * U(p,q) from E4M3 page bounds -> scores [B,Hkv,Pmax] fp32."""
    _need(q, "q", torch.float16, 3)
    _need(meta, "meta", torch.uint8, 5)
    _need(valid_len, "valid_len", torch.int32, 1)
    B, Hq, D = q.shape
    Hkv = meta.shape[1]
    d = make_dims(B, Hq, Hkv, D, max_len, page_size)
    _meta_shape(meta, B, Hkv, max_len, D, page_size)
    _shape(valid_len, "valid_len", (B,))
    if scores is None:
        scores = torch.empty(B, Hkv, num_pages(max_len, page_size), dtype=torch.float32, device=q.device)
    _need(scores, "scores", torch.float32, 3)
    _shape(scores, "scores", (B, Hkv, num_pages(max_len, page_size)))
    _check("quest_score_pages_e4m3", lib().quest_score_pages_e4m3(
        ctypes.byref(d), _ptr(q), _ptr(meta), float(k_scale), _ptr(valid_len), _ptr(scores), _stream(q)))
    return scores


def quest_sparse_attn_e4m3(q, k_cache, v_cache, k_scale: float, v_scale: float, valid_len, page_idx, scale: float,
                           out=None, workspace=None, page_size: int = PAGE_SIZE):
    """Attention over the selected pages of an E4M3 cache (page_idx [B,Hkv,k])."""
    _need(q, "q", torch.float16, 3)
    _need(k_cache, "k_cache", torch.uint8, 4)
    _need(v_cache, "v_cache", torch.uint8, 4)
    _need(valid_len, "valid_len", torch.int32, 1)
    _need(page_idx, "page_idx", torch.int32, 3)
    d = dims_of(q, k_cache, page_size)
    _shape(v_cache, "v_cache", tuple(k_cache.shape))
    _shape(valid_len, "valid_len", (d.batch,))
    _shape(page_idx, "page_idx", (d.batch, d.num_kv_heads, page_idx.shape[2]))
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", torch.float16, 3)
    if workspace is None:
        workspace = alloc_workspace(d, q.device)
    _check("quest_sparse_attn_e4m3", lib().quest_sparse_attn_e4m3(
        ctypes.byref(d), _ptr(q), _ptr(k_cache), _ptr(v_cache), float(k_scale), float(v_scale), _ptr(valid_len),
        _ptr(page_idx), int(page_idx.shape[2]), float(scale), _ptr(out), _ptr(workspace), workspace.numel(),
        _stream(q)))
    return out


def quest_decode_attn_e4m3(q, k_cache, v_cache, meta, valid_len, k: int, scale: float, k_scale: float,
                           v_scale: float, k_new=None, v_new=None, pos=None, k_inv_scale: float = 1.0,
                           v_inv_scale: float = 1.0, out=None, scores=None, page_idx=None,
                           page_size: int = PAGE_SIZE):
    """quest_decode_attn over an E4M3 cache (codes [B,Hkv,Lmax,D] uint8, bounds
    [B,Hkv,Pmax,2,D] uint8) in one launch; the optional append quantizes
    k_new/v_new with k_inv_scale / v_inv_scale."""
    _need(q, "q", torch.float16, 3)
    _need(k_cache, "k_cache", torch.uint8, 4)
    _need(v_cache, "v_cache", torch.uint8, 4)
    _need(meta, "meta", torch.uint8, 5)
    _need(valid_len, "valid_len", torch.int32, 1)
    d = dims_of(q, k_cache, page_size)
    _shape(v_cache, "v_cache", tuple(k_cache.shape))
    _meta_shape(meta, d.batch, d.num_kv_heads, d.max_len, d.head_dim, page_size)
    _shape(valid_len, "valid_len", (d.batch,))
    if pos is not None:
        _need(k_new, "k_new", torch.float16, 3)
        _need(v_new, "v_new", torch.float16, 3)
        _need(pos, "pos", torch.int32, 1)
        _new_rows(k_new, v_new, pos, d.batch, d.num_kv_heads, d.head_dim)
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", torch.float16, 3)
    if scores is not None:
        _need(scores, "scores", torch.float32, 3)
        _shape(scores, "scores", (d.batch, d.num_kv_heads, num_pages(d.max_len, page_size)))
    if page_idx is not None:
        _need(page_idx, "page_idx", torch.int32, 3)
        _shape(page_idx, "page_idx", (d.batch, d.num_kv_heads, int(k)))
    _check("quest_decode_attn_e4m3", lib().quest_decode_attn_e4m3(
        ctypes.byref(d), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(meta), _ptr(k_new), _ptr(v_new), _ptr(pos),
        float(k_inv_scale), float(v_inv_scale), float(k_scale), float(v_scale), _ptr(valid_len), int(k),
        float(scale), _ptr(out), _ptr(scores), _ptr(page_idx), _stream(q)))
    return out


def prefill_workspace_bytes(dims: Dims, q_len: int) -> int:
    n = lib().gqaq_prefill_workspace_bytes(ctypes.byref(dims), int(q_len))
    if n == 0:
        raise GqaqError("gqaq_prefill_workspace_bytes", GQAQ_ERR_UNSUPPORTED, "dims rejected")
    return int(n)


def alloc_prefill_workspace(dims: Dims, q_len: int, device) -> torch.Tensor:
    """Zero-filled workspace for gqa_prefill_attn (its counters stay zero between calls)."""
    return torch.zeros(prefill_workspace_bytes(dims, q_len), dtype=torch.uint8, device=device)


def gqa_prefill_attn(q, k_cache, v_cache, start, scale: float, out=None, workspace=None):
    """Causal attention of a chunk: q [B,Hq,q_len,D], caches [B,Hkv,Lmax,D]
    holding the chunk at rows start[b] .. start[b]+q_len-1; token t attends to
    rows 0 .. start[b]+t. The G heads and q_len tokens of a KV head are one
    folded row block."""
    _need(q, "q", torch.float16, 4)
    _need(k_cache, "k_cache", torch.float16, 4)
    _need(v_cache, "v_cache", torch.float16, 4)
    _need(start, "start", torch.int32, 1)
    B, Hq, q_len, D = q.shape
    _, Hkv, Lmax, _ = k_cache.shape
    d = make_dims(B, Hq, Hkv, D, Lmax)
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", torch.float16, 4)
    if workspace is None:
        workspace = alloc_prefill_workspace(d, q_len, q.device)
    _check("gqa_prefill_attn", lib().gqa_prefill_attn(
        ctypes.byref(d), int(q_len), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(start), float(scale), _ptr(out),
        _ptr(workspace), workspace.numel(), _stream(q)))
    return out


def gqa_decode_attn_int4(q, k_codes, k_scales, v_codes, v_scales, valid_len, scale: float, out=None,
                         workspace=None):
    """Dense folded-GQA decode attention over a 4-bit cache: codes
    [B,Hkv,Lmax,D/2] uint8 (two levels + 8 per byte, low nibble first), scales
    [B,Hkv,Lmax] fp32 (value = level * scale). Lmax must be a multiple of 4."""
    _need(q, "q", torch.float16, 3)
    for name, t in (("k_codes", k_codes), ("v_codes", v_codes)):
        _need(t, name, torch.uint8, 4)
    for name, t in (("k_scales", k_scales), ("v_scales", v_scales)):
        _need(t, name, torch.float32, 3)
    _need(valid_len, "valid_len", torch.int32, 1)
    B, Hq, D = q.shape
    _, Hkv, Lmax, _ = k_codes.shape
    d = make_dims(B, Hq, Hkv, D, Lmax)
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", torch.float16, 3)
    if workspace is None:
        workspace = alloc_workspace(d, q.device)
    _check("gqa_decode_attn_int4", lib().gqa_decode_attn_int4(
        ctypes.byref(d), _ptr(q), _ptr(k_codes), _ptr(k_scales), _ptr(v_codes), _ptr(v_scales), _ptr(valid_len),
        float(scale), _ptr(out), _ptr(workspace), workspace.numel(), _stream(q)))
    return out


def kv_append_int4(k_codes, k_scales, v_codes, v_scales, k_new, v_new, pos):
    """Quantize k_new/v_new [B,Hkv,D] fp16 rows to INT4 (scale = amax / 7 per
    row) and write codes and scales at row pos[b]."""
    for name, t in (("k_codes", k_codes), ("v_codes", v_codes)):
        _need(t, name, torch.uint8, 4)
    for name, t in (("k_scales", k_scales), ("v_scales", v_scales)):
        _need(t, name, torch.float32, 3)
    _need(k_new, "k_new", torch.float16, 3)
    _need(v_new, "v_new", torch.float16, 3)
    _need(pos, "pos", torch.int32, 1)
    B, Hkv, Lmax, _ = k_codes.shape
    D = k_new.shape[2]
    d = make_dims(B, Hkv, Hkv, D, Lmax)
    _check("kv_append_int4", lib().kv_append_int4(
        ctypes.byref(d), _ptr(k_codes), _ptr(k_scales), _ptr(v_codes), _ptr(v_scales), _ptr(k_new), _ptr(v_new),
        _ptr(pos), _stream(k_codes)))


def quest_append_kv(k_cache, v_cache, meta, k_new, v_new, pos, page_size: int = PAGE_SIZE):
    """Write k_new/v_new [B,Hkv,D] at row pos[b] and update that page's min/max."""
    _need(k_cache, "k_cache", torch.float16, 4)
    _need(v_cache, "v_cache", torch.float16, 4)
    _need(meta, "meta", torch.float16, 5)
    _need(k_new, "k_new", torch.float16, 3)
    _need(v_new, "v_new", torch.float16, 3)
    _need(pos, "pos", torch.int32, 1)
    B, Hkv, Lmax, D = k_cache.shape
    _shape(v_cache, "v_cache", tuple(k_cache.shape))
    _meta_shape(meta, B, Hkv, Lmax, D, page_size)
    _new_rows(k_new, v_new, pos, B, Hkv, D)
    d = make_dims(B, Hkv, Hkv, D, Lmax, page_size)
    _check("quest_append_kv", lib().quest_append_kv(
        ctypes.byref(d), _ptr(k_cache), _ptr(v_cache), _ptr(meta), _ptr(k_new), _ptr(v_new),
        _ptr(pos), _stream(k_cache)))


def quest_update_meta(k_cache, valid_len, meta, page_begin: int = 0, page_end: Optional[int] = None,
                      page_size: int = PAGE_SIZE):
    """Rebuild page min/max [B,Hkv,Pmax,2,D] for pages [page_begin, page_end)."""
    _need(k_cache, "k_cache", torch.float16, 4)
    _need(valid_len, "valid_len", torch.int32, 1)
    _need(meta, "meta", torch.float16, 5)
    B, Hkv, Lmax, D = k_cache.shape
    _meta_shape(meta, B, Hkv, Lmax, D, page_size)
    _shape(valid_len, "valid_len", (B,))
    d = make_dims(B, Hkv, Hkv, D, Lmax, page_size)
    if page_end is None:
        page_end = num_pages(Lmax, page_size)
    _check("quest_update_meta", lib().quest_update_meta(
        ctypes.byref(d), _ptr(k_cache), _ptr(valid_len), _ptr(meta), int(page_begin), int(page_end),
        _stream(k_cache)))
    return meta


def quest_score_pages(q, meta, valid_len, max_len: int, scores=None, page_size: int = PAGE_SIZE):
    """U(p,q) per KV head (max over its G folded query rows) -> scores [B,Hkv,Pmax] fp32."""
    _need(q, "q", torch.float16, 3)
    _need(meta, "meta", torch.float16, 5)
    _need(valid_len, "valid_len", torch.int32, 1)
    B, Hq, D = q.shape
    Hkv = meta.shape[1]
    d = make_dims(B, Hq, Hkv, D, max_len, page_size)
    _meta_shape(meta, B, Hkv, max_len, D, page_size)
    _shape(valid_len, "valid_len", (B,))
    if scores is None:
        scores = torch.empty(B, Hkv, num_pages(max_len, page_size), dtype=torch.float32, device=q.device)
    _need(scores, "scores", torch.float32, 3)
    _shape(scores, "scores", (B, Hkv, num_pages(max_len, page_size)))
    _check("quest_score_pages", lib().quest_score_pages(
        ctypes.byref(d), _ptr(q), _ptr(meta), _ptr(valid_len), _ptr(scores), _stream(q)))
    return scores


def quest_topk_pages(scores, valid_len, k: int, max_len: int, page_idx=None, page_size: int = PAGE_SIZE):
    """Top-k pages per (b, kv) -> page_idx [B,Hkv,k] int32, ascending, -1 padded."""
    _need(scores, "scores", torch.float32, 3)
    _need(valid_len, "valid_len", torch.int32, 1)
    B, Hkv, _ = scores.shape
    _shape(scores, "scores", (B, Hkv, num_pages(max_len, page_size)))
    _shape(valid_len, "valid_len", (B,))
    d = make_dims(B, Hkv, Hkv, 64, max_len, page_size)
    if page_idx is None:
        page_idx = torch.empty(B, Hkv, int(k), dtype=torch.int32, device=scores.device)
    _need(page_idx, "page_idx", torch.int32, 3)
    _shape(page_idx, "page_idx", (B, Hkv, int(k)))
    _check("quest_topk_pages", lib().quest_topk_pages(
        ctypes.byref(d), _ptr(scores), _ptr(valid_len), int(k), _ptr(page_idx), None, 0,
        _stream(scores)))
    return page_idx


def quest_sparse_attn(q, k_cache, v_cache, valid_len, page_idx, scale: float, out=None, workspace=None,
                      page_size: int = PAGE_SIZE):
    """Attention over the selected pages only (page_idx [B,Hkv,k])."""
    _need(q, "q", torch.float16, 3)
    _need(k_cache, "k_cache", torch.float16, 4)
    _need(v_cache, "v_cache", torch.float16, 4)
    _need(valid_len, "valid_len", torch.int32, 1)
    _need(page_idx, "page_idx", torch.int32, 3)
    d = dims_of(q, k_cache, page_size)
    _shape(v_cache, "v_cache", tuple(k_cache.shape))
    _shape(valid_len, "valid_len", (d.batch,))
    _shape(page_idx, "page_idx", (d.batch, d.num_kv_heads, page_idx.shape[2]))
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", torch.float16, 3)
    if workspace is None:
        workspace = alloc_workspace(d, q.device)
    _check("quest_sparse_attn", lib().quest_sparse_attn(
        ctypes.byref(d), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(valid_len), _ptr(page_idx),
        int(page_idx.shape[2]), float(scale), _ptr(out), _ptr(workspace), workspace.numel(), _stream(q)))
    return out


def new_meta(batch: int, num_kv_heads: int, max_len: int, head_dim: int, device,
             page_size: int = PAGE_SIZE) -> torch.Tensor:
    """Allocate a metadata buffer [B,Hkv,Pmax,2,D] fp16 (contents undefined)."""
    return torch.empty(batch, num_kv_heads, num_pages(max_len, page_size), 2, head_dim,
                       dtype=torch.float16, device=device)
