"""Seeded synthetic inputs for the decode-attention path.

This module is shared by the tests, the smoke check and the bench, on both
sides of every parity check (the CUDA library and the CPU oracle).  It holds
none of the method's arithmetic: it only draws random caches and queries with
the shapes and value structure of the five workloads below and returns them.

Workloads (shapes from the two source pages' models and experiments):
  1  dense GQA decode, one layer, batch 1: Hq=32, Hkv=8, D=64, L=4096
     (EXAONE 4.0 1.2B attention shape; "Core ML Decode Optimization ...",
     section 1).
  2  dense GQA decode, 30 layers, Hq=32, Hkv=8, D=64, allocated length 4096,
     valid lengths uniform in [1024, 4096] per layer and sequence, batch 1/32.
  3  Quest on a Llama-2-7B shape: 32 layers, MHA 32 heads, D=128, L=32768,
     S=16, K=128 pages (2048-token budget), layers 0-1 dense, batch 1, 8
     planted pages per head ("Quest ..." review, kernel-comparison setting).
  4  Quest with GQA: Hq=32, Hkv=8, D=128, L=65536, S=16, K=256 (4096-token
     budget), one layer, one appended token per step, batch 1/4/8.
  5  long context: 32 heads MHA, D=128, L=131072, S=16, budgets 2048 / 8192
     tokens (K=128 / 512), batch 1/16, 1% planted pages.

Planted pages ("keys shifted +2 sigma along a random direction shared with
q"), per (layer, sequence, KV head): draw a unit vector u; every folded query
row of that head is z + sqrt(D) u with z ~ N(0, I); choose n_plant distinct
pages uniformly; add 2u to every key of those pages.  Values stay N(0, 1).
Everything is drawn in fp32 and rounded to fp16 once.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

BASE_SEED = 20261202


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic decode workload (all layers of one step)."""
    id: int
    name: str
    batch: int
    num_layers: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    max_len: int
    page_size: int = 16
    k_pages: Optional[int] = None      # Quest K (pages); None = dense only
    dense_layers: int = 0              # leading layers kept dense when k_pages is set
    valid_lo: Optional[int] = None     # valid lengths uniform in [valid_lo, max_len]; None = full
    n_plant: int = 0                   # planted pages per KV head
    append: bool = False               # one token appended per step (pos = max_len - 1)

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def pages_max(self) -> int:
        return (self.max_len + self.page_size - 1) // self.page_size

    def layer_is_dense(self, layer: int) -> bool:
        return self.k_pages is None or layer < self.dense_layers

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


def _plant_count(pages: int, frac: float) -> int:
    return max(1, int(round(frac * pages)))


WORKLOADS = {
    1: Workload(1, "dense-gqa-exaone-1layer", batch=1, num_layers=1, num_q_heads=32,
                num_kv_heads=8, head_dim=64, max_len=4096),
    2: Workload(2, "dense-gqa-exaone-30layer", batch=32, num_layers=30, num_q_heads=32,
                num_kv_heads=8, head_dim=64, max_len=4096, valid_lo=1024),
    3: Workload(3, "quest-llama2-7b-32k", batch=1, num_layers=32, num_q_heads=32,
                num_kv_heads=32, head_dim=128, max_len=32768, k_pages=128, dense_layers=2,
                n_plant=8, append=True),
    4: Workload(4, "quest-gqa-64k", batch=8, num_layers=1, num_q_heads=32, num_kv_heads=8,
                head_dim=128, max_len=65536, k_pages=256, n_plant=8, append=True),
    5: Workload(5, "long-ctx-128k", batch=16, num_layers=1, num_q_heads=32, num_kv_heads=32,
                head_dim=128, max_len=131072, k_pages=128,
                n_plant=_plant_count(131072 // 16, 0.01), append=True),
}


def layer_seed(w: Workload, layer: int, salt: int = 0) -> int:
    return BASE_SEED + 1000 * w.id + layer + 100003 * salt


def valid_lengths(w: Workload, layer: int) -> torch.Tensor:
    """Valid token count per sequence for one layer (int32, CPU)."""
    if w.valid_lo is None:
        return torch.full((w.batch,), w.max_len, dtype=torch.int32)
    g = torch.Generator(device="cpu").manual_seed(layer_seed(w, layer, salt=1))
    return torch.randint(w.valid_lo, w.max_len + 1, (w.batch,), generator=g,
                         dtype=torch.int64).to(torch.int32)


def make_layer(w: Workload, layer: int = 0, device="cpu", seed: Optional[int] = None):
    """Draw one layer's q, k_cache, v_cache (fp16) and, with append, k_new/v_new.

    Returns a dict of torch tensors on ``device``:
      q [B,Hq,D], k_cache/v_cache [B,Hkv,Lmax,D], valid_len [B] int32,
      and when ``w.append``: k_new/v_new [B,Hkv,D], pos [B] int32 (= Lmax-1).
    """
    device = torch.device(device)
    B, Hq, Hkv, D, Lmax, S = (w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim,
                              w.max_len, w.page_size)
    G = Hq // Hkv
    g = torch.Generator(device=device).manual_seed(layer_seed(w, layer) if seed is None else seed)
    q = torch.randn(B, Hkv, G, D, generator=g, device=device, dtype=torch.float32)
    k = torch.empty(B, Hkv, Lmax, D, device=device, dtype=torch.float16)
    v = torch.empty(B, Hkv, Lmax, D, device=device, dtype=torch.float16)
    pages = (Lmax + S - 1) // S
    for b in range(B):  # one sequence at a time keeps the fp32 temporaries small
        kb = torch.randn(Hkv, Lmax, D, generator=g, device=device, dtype=torch.float32)
        vb = torch.randn(Hkv, Lmax, D, generator=g, device=device, dtype=torch.float32)
        if w.n_plant > 0:
            u = torch.randn(Hkv, D, generator=g, device=device, dtype=torch.float32)
            u = u / u.norm(dim=-1, keepdim=True)
            q[b] += math.sqrt(D) * u[:, None, :]
            n_plant = min(w.n_plant, pages)
            order = torch.rand(Hkv, pages, generator=g, device=device).argsort(dim=-1)
            chosen = order[:, :n_plant]                              # [Hkv, n_plant]
            tok_mask = torch.zeros(Hkv, pages * S, device=device, dtype=torch.bool)
            for j in range(S):
                tok_mask.scatter_(1, chosen * S + j, True)
            tok_mask = tok_mask[:, :Lmax]
            kb += 2.0 * tok_mask[:, :, None].to(torch.float32) * u[:, None, :]
        k[b] = kb.to(torch.float16)
        v[b] = vb.to(torch.float16)
        del kb, vb
    out = {
        "q": q.reshape(B, Hq, D).to(torch.float16),
        "k_cache": k,
        "v_cache": v,
        "valid_len": valid_lengths(w, layer).to(device),
    }
    if w.append:
        out["k_new"] = torch.randn(B, Hkv, D, generator=g, device=device).to(torch.float16)
        out["v_new"] = torch.randn(B, Hkv, D, generator=g, device=device).to(torch.float16)
        out["pos"] = torch.full((B,), Lmax - 1, dtype=torch.int32, device=device)
    return out


def make_prefill_layer(w: Workload, layer: int, q_len: int, device="cpu", seed: Optional[int] = None):
    """One layer's inputs for a prefill chunk: the workload's caches, a chunk
    of q_len query tokens per head, q [B,Hq,q_len,D] ~ N(0,1) fp16, and start
    [B] int32 = valid_len - q_len (the chunk is the last q_len valid tokens,
    already in the cache). The decode-only planted pages are not drawn."""
    x = make_layer(w.with_(n_plant=0, append=False), layer, device=device, seed=seed)
    g = torch.Generator(device=torch.device(device)).manual_seed(layer_seed(w, layer, salt=2) if seed is None else seed + 1)
    q = torch.randn(w.batch, w.num_q_heads, q_len, w.head_dim, generator=g, device=device).to(torch.float16)
    start = (x["valid_len"] - q_len).clamp(min=0).to(torch.int32)
    return {"q": q, "k_cache": x["k_cache"], "v_cache": x["v_cache"], "start": start}


def small(w: Workload, **overrides) -> Workload:
    """A reduced copy of a workload with the same structure (for oracle-sized tests)."""
    return w.with_(**overrides)
