"""One decode step over a stack of attention layers, through the C ABI.

Layer policy ("Quest: Query-Aware Sparsity ..." review, the note that the
first two attention layers keep full attention): layers with index below
``dense_layers`` run dense folded-GQA attention over every valid token.
Later layers run the Quest path: score every page from its key min/max,
pick the top ``k_pages``, and attend over those pages only. When a step
carries a new token, every layer first appends it (``quest_append_kv``), so
each layer's page metadata stays current whatever path reads it.

With ``kv="e4m3"`` the caches hold 8-bit E4M3 codes with one fp32 scale per
tensor (``Layer.k_scale`` / ``v_scale``): appends quantize
(``kv_append_e4m3``, or ``quest_append_kv_e4m3`` when the layer keeps page
bounds), dense layers read them through ``gqa_decode_attn_e4m3`` and Quest
layers over E4M3 page bounds run as one ``quest_decode_attn_e4m3`` launch
(or, with ``fused=False``, ``quest_score_pages_e4m3``, ``quest_topk_pages``
and ``quest_sparse_attn_e4m3``). With ``kv="int4"`` they hold 4-bit
levels ``[B,Hkv,Lmax,D/2]`` with one fp32 scale per token row
(``Layer.k_scales`` / ``v_scales``), through ``kv_append_int4`` and
``gqa_decode_attn_int4``; an INT4 stack must be all dense.

By default a Quest layer is one fused launch (``quest_decode_attn``: append,
score, top-K and sparse attention in one kernel); the library picks its
kernel (GQAQ_OPT_QUEST_KERNEL), and the stack's workspace covers both. With
``fused=False`` the same layer runs as the four step-by-step calls.

This module only sequences library calls and owns the scratch buffers they
share. Every arithmetic step runs in the CUDA kernels.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional

import torch

from . import (alloc_workspace, gqa_decode_attn, gqa_decode_attn_e4m3, gqa_decode_attn_int4, kv_append_e4m3,
               kv_append_int4, make_dims, new_meta, new_meta_e4m3, num_pages, quest_append_kv, quest_append_kv_e4m3,
               quest_decode_attn, quest_decode_attn_e4m3, quest_score_pages, quest_score_pages_e4m3, quest_sparse_attn, quest_sparse_attn_e4m3,
               quest_topk_pages, quest_update_meta, quest_update_meta_e4m3)


@dataclasses.dataclass
class Layer:
    """Device tensors of one attention layer for one step."""
    q: torch.Tensor                       # [B,Hq,D] fp16
    k_cache: torch.Tensor                 # [B,Hkv,Lmax,D] fp16 (uint8 E4M3 codes with kv="e4m3")
    v_cache: torch.Tensor
    valid_len: torch.Tensor               # [B] int32 (tokens attended after the append)
    out: torch.Tensor                     # [B,Hq,D] fp16
    meta: Optional[torch.Tensor] = None   # [B,Hkv,Pmax,2,D] fp16 (uint8 E4M3 bounds with kv="e4m3")
    k_new: Optional[torch.Tensor] = None  # [B,Hkv,D] fp16
    v_new: Optional[torch.Tensor] = None
    pos: Optional[torch.Tensor] = None    # [B] int32 row the new token goes to
    k_scale: float = 1.0                  # E4M3 caches: value = code value * scale
    v_scale: float = 1.0
    k_scales: Optional[torch.Tensor] = None  # INT4 caches: [B,Hkv,Lmax] fp32 per-token scales
    v_scales: Optional[torch.Tensor] = None
    page_idx: Optional[torch.Tensor] = None  # [B,Hkv,K] int32: when set, Quest layers also write their page lists


def layer_plan(layer: int, k_pages: Optional[int], dense_layers: int, fused: bool, append: bool):
    """Names of the library calls layer ``layer`` makes in one step, in order.

    Layers below ``dense_layers`` (or every layer when ``k_pages`` is None) are
    dense: "append" (when the step carries a token) then "dense". Later layers
    run Quest: one "quest" call (the fused step, which appends itself) or,
    unfused, "append", "score", "topk", "sparse"."""
    dense = k_pages is None or layer < dense_layers
    calls = []
    if append and (dense or not fused):
        calls.append("append")
    if dense:
        calls.append("dense")
    elif fused:
        calls.append("quest")
    else:
        calls += ["score", "topk", "sparse"]
    return tuple(calls)


class DecodeStack:
    def __init__(self, batch: int, num_q_heads: int, num_kv_heads: int, head_dim: int, max_len: int,
                 k_pages: Optional[int], dense_layers: int, device, page_size: int = 16, fused: bool = True,
                 kv: str = "f16", num_layers: Optional[int] = None):
        if kv not in ("f16", "e4m3", "int4"):
            raise ValueError(f"kv must be 'f16', 'e4m3' or 'int4', got {kv!r}")
        if kv == "int4" and k_pages is not None and (num_layers is None or num_layers > dense_layers):
            raise ValueError("a 4-bit cache runs dense layers only")
        self.fused, self.kv = fused, kv
        self.batch, self.num_q_heads, self.num_kv_heads = batch, num_q_heads, num_kv_heads
        self.head_dim, self.max_len, self.page_size = head_dim, max_len, page_size
        self.k_pages, self.dense_layers = k_pages, dense_layers
        self.scale = 1.0 / math.sqrt(head_dim)
        self.device = torch.device(device)
        dims = make_dims(batch, num_q_heads, num_kv_heads, head_dim, max_len, page_size)
        self.workspace = alloc_workspace(dims, self.device, k_pages or 0)
        pmax = num_pages(max_len, page_size)
        self.scores = torch.empty(batch, num_kv_heads, pmax, dtype=torch.float32, device=self.device)
        self.page_idx = (torch.empty(batch, num_kv_heads, k_pages, dtype=torch.int32, device=self.device)
                         if k_pages else None)

    def is_dense(self, layer: int) -> bool:
        return "dense" in layer_plan(layer, self.k_pages, self.dense_layers, self.fused, False)

    def new_meta(self) -> torch.Tensor:
        alloc = new_meta_e4m3 if self.kv == "e4m3" else new_meta
        return alloc(self.batch, self.num_kv_heads, self.max_len, self.head_dim, self.device, self.page_size)

    def build_meta(self, layer: Layer, valid_len: torch.Tensor):
        """Metadata of the pages already in the cache (after a prefill)."""
        build = quest_update_meta_e4m3 if self.kv == "e4m3" else quest_update_meta
        build(layer.k_cache, valid_len, layer.meta, page_size=self.page_size)

    def append(self, L: Layer):
        if self.kv == "e4m3" and L.meta is not None:
            quest_append_kv_e4m3(L.k_cache, L.v_cache, L.meta, L.k_new, L.v_new, L.pos, 1.0 / L.k_scale,
                                 1.0 / L.v_scale, self.page_size)
        elif self.kv == "e4m3":
            kv_append_e4m3(L.k_cache, L.v_cache, L.k_new, L.v_new, L.pos, 1.0 / L.k_scale, 1.0 / L.v_scale)
        elif self.kv == "int4":
            kv_append_int4(L.k_cache, L.k_scales, L.v_cache, L.v_scales, L.k_new, L.v_new, L.pos)
        else:
            quest_append_kv(L.k_cache, L.v_cache, L.meta, L.k_new, L.v_new, L.pos, self.page_size)

    def dense(self, L: Layer):
        if self.kv == "e4m3":
            gqa_decode_attn_e4m3(L.q, L.k_cache, L.v_cache, L.k_scale, L.v_scale, L.valid_len, self.scale,
                                 out=L.out, workspace=self.workspace)
        elif self.kv == "int4":
            gqa_decode_attn_int4(L.q, L.k_cache, L.k_scales, L.v_cache, L.v_scales, L.valid_len, self.scale,
                                 out=L.out, workspace=self.workspace)
        else:
            gqa_decode_attn(L.q, L.k_cache, L.v_cache, L.valid_len, self.scale, out=L.out,
                            workspace=self.workspace)

    def calls(self, layer: int, L: Layer):
        """The library calls of one layer in launch order, as (family, thunk) pairs."""
        out = []
        for name in layer_plan(layer, self.k_pages, self.dense_layers, self.fused, L.k_new is not None):
            out.append((name, self._thunk(name, L)))
        return out

    def _thunk(self, name: str, L: Layer):
        if name == "append":
            return lambda: self.append(L)
        if name == "dense":
            return lambda: self.dense(L)
        if name == "quest" and self.kv == "e4m3":
            return lambda: quest_decode_attn_e4m3(L.q, L.k_cache, L.v_cache, L.meta, L.valid_len, self.k_pages,
                                                  self.scale, L.k_scale, L.v_scale, k_new=L.k_new, v_new=L.v_new,
                                                  pos=L.pos, k_inv_scale=1.0 / L.k_scale, v_inv_scale=1.0 / L.v_scale,
                                                  out=L.out, page_idx=L.page_idx, page_size=self.page_size)
        if name == "quest":
            return lambda: quest_decode_attn(L.q, L.k_cache, L.v_cache, L.meta, L.valid_len, self.k_pages,
                                             self.scale, k_new=L.k_new, v_new=L.v_new, pos=L.pos, out=L.out,
                                             page_idx=L.page_idx, page_size=self.page_size,
                                             workspace=self.workspace)
        if name == "score" and self.kv == "e4m3":
            return lambda: quest_score_pages_e4m3(L.q, L.meta, L.k_scale, L.valid_len, self.max_len,
                                                  scores=self.scores, page_size=self.page_size)
        if name == "score":
            return lambda: quest_score_pages(L.q, L.meta, L.valid_len, self.max_len, scores=self.scores,
                                             page_size=self.page_size)
        idx = self.page_idx if L.page_idx is None else L.page_idx
        if name == "topk":
            return lambda: quest_topk_pages(self.scores, L.valid_len, self.k_pages, self.max_len, page_idx=idx,
                                            page_size=self.page_size)
        if name == "sparse" and self.kv == "e4m3":
            return lambda: quest_sparse_attn_e4m3(L.q, L.k_cache, L.v_cache, L.k_scale, L.v_scale, L.valid_len, idx,
                                                  self.scale, out=L.out, workspace=self.workspace,
                                                  page_size=self.page_size)
        if name == "sparse":
            return lambda: quest_sparse_attn(L.q, L.k_cache, L.v_cache, L.valid_len, idx, self.scale, out=L.out,
                                             workspace=self.workspace, page_size=self.page_size)
        raise ValueError(name)

    def families(self, layers: List[Layer]):
        """The library calls of one step, grouped by kind: name -> list of thunks."""
        fam = {}
        for i, L in enumerate(layers):
            for name, fn in self.calls(i, L):
                fam.setdefault(name, []).append(fn)
        return fam

    @staticmethod
    def kernels_per_call(name: str, k_pages: Optional[int]) -> int:
        """Kernel launches behind one call of a family."""
        return 1                           # split units are merged inside the attention kernel

    def launches_per_step(self, layers: List[Layer]) -> int:
        return sum(len(v) * self.kernels_per_call(k, self.k_pages) for k, v in self.families(layers).items())

    def step(self, layers: List[Layer]):
        for i, L in enumerate(layers):
            for _, fn in self.calls(i, L):
                fn()
