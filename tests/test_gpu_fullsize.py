"""Parity at the workloads' full sizes, in the launch configuration the bench
times (default grid and kernel choice, fused Quest layers with the decode
stack's workspace; the work-queue kernel once, at the Llama-2 shape).

The GPU runs every (sequence, KV head) unit; the fp64 oracle checks sampled
units one by one: page metadata bit-exact, the selected page set against the
oracle's own top-K (near-ties exempt), and the attention output within the
fp16 tolerance.
"""
import math

import numpy as np
import pytest
import torch

import gqa_head_folding_gb300 as g
import oracle
import workloads
from _util import assert_attn_close, check_topk, to64

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def unit_arrays(x, b, kv, G):
    q = x["q"][b, kv * G:(kv + 1) * G].unsqueeze(0).cpu().numpy()
    k = x["k_cache"][b, kv].unsqueeze(0).unsqueeze(0).cpu().numpy()
    v = x["v_cache"][b, kv].unsqueeze(0).unsqueeze(0).cpu().numpy()
    return q, k, v


def sample_units(B, Hkv, n, seed=0):
    rng = np.random.default_rng(seed)
    units = [(b, kv) for b in range(B) for kv in range(Hkv)]
    pick = rng.choice(len(units), size=min(n, len(units)), replace=False)
    return [units[i] for i in sorted(pick)]


def check_quest_layer(w, seed_layer=2, n_units=3, kernel="auto"):
    x = workloads.make_layer(w, seed_layer, device=DEV)
    B, Hkv, Lmax, D = x["k_cache"].shape
    G, S, K = w.group, w.page_size, w.k_pages
    meta = g.new_meta(B, Hkv, Lmax, D, DEV)
    g.quest_update_meta(x["k_cache"], x["valid_len"] - 1, meta)
    idx = torch.empty(B, Hkv, K, dtype=torch.int32, device=DEV)
    scale = 1.0 / math.sqrt(D)
    ws = g.alloc_workspace(g.dims_of(x["q"], x["k_cache"]), DEV, K)
    g.set_option(g.GQAQ_OPT_QUEST_KERNEL, 2 if kernel == "queue" else 0)
    try:
        out = g.quest_decode_attn(x["q"], x["k_cache"], x["v_cache"], meta, x["valid_len"], K, scale,
                                  k_new=x["k_new"], v_new=x["v_new"], pos=x["pos"], page_idx=idx, workspace=ws)
    finally:
        g.set_option(g.GQAQ_OPT_QUEST_KERNEL, 0)
    torch.cuda.synchronize()
    assert g.device_status() == 0
    assert int(ws[:g.workspace_zero_bytes(g.dims_of(x["q"], x["k_cache"]))].count_nonzero()) == 0
    vl = x["valid_len"].cpu().numpy()
    for (b, kv) in sample_units(B, Hkv, n_units, seed=D + K):
        q, k, v = unit_arrays(x, b, kv, G)          # caches already hold the appended token
        L = [int(vl[b])]
        ref_meta = oracle.page_minmax(k, L, S)
        P = (L[0] + S - 1) // S
        assert np.array_equal(to64(meta[b, kv, :P]), ref_meta[0, 0, :P]), f"meta ({b},{kv})"
        ref_scores = oracle.page_scores(q, ref_meta, L, S)
        sel = idx[b, kv].cpu().numpy()[None, None]
        check_topk(sel, ref_scores, L, S, K)
        ref = oracle.sparse_attn(q, k, v, L, sel, S, scale)
        assert_attn_close(out[b, kv * G:(kv + 1) * G].unsqueeze(0), ref, f"unit ({b},{kv})")
    del x, meta


def check_dense_layer(w, layer=0, n_units=3):
    x = workloads.make_layer(w, layer, device=DEV)
    B, Hkv, Lmax, D = x["k_cache"].shape
    G = w.group
    scale = 1.0 / math.sqrt(D)
    out = g.gqa_decode_attn(x["q"], x["k_cache"], x["v_cache"], x["valid_len"], scale)
    torch.cuda.synchronize()
    vl = x["valid_len"].cpu().numpy()
    for (b, kv) in sample_units(B, Hkv, n_units, seed=layer + D):
        q, k, v = unit_arrays(x, b, kv, G)
        ref = oracle.attn_repeat_kv(q, k, v, [int(vl[b])], scale)
        assert_attn_close(out[b, kv * G:(kv + 1) * G].unsqueeze(0), ref, f"unit ({b},{kv})")
    del x


def test_llama2_7b_quest_stack_layers():
    # 32 heads, D=128, L=32768, K=128: one dense layer and one Quest layer at full size
    w = workloads.WORKLOADS[3]
    check_dense_layer(w, layer=0)
    check_quest_layer(w, seed_layer=2)
    check_quest_layer(w, seed_layer=3, n_units=2, kernel="queue")


def test_exaone_dense_batch_32():
    check_dense_layer(workloads.WORKLOADS[2], layer=5, n_units=4)


@pytest.mark.parametrize("batch", [1, 8])
def test_gqa_quest_64k(batch):
    check_quest_layer(workloads.WORKLOADS[4].with_(batch=batch), seed_layer=0, n_units=3)


@pytest.mark.parametrize("k_pages", [128, 512])
def test_long_context_128k_quest(k_pages):
    check_quest_layer(workloads.WORKLOADS[5].with_(batch=1, k_pages=k_pages), seed_layer=0, n_units=2)


def test_long_context_128k_dense_batch_16():
    check_dense_layer(workloads.WORKLOADS[5], layer=0, n_units=2)
