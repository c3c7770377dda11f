"""GPU parity of the Quest path at page sizes S in {8, 16, 32, 64} (the
page-size trade-off the Quest review discusses), against the fp64 oracle.

Each case builds the page metadata, appends a token, scores, selects and
attends, through the step-by-step calls and through quest_decode_attn on
both of its kernels, on ragged lengths whose last page is partial. At
S = 8 a consumer warp holds one page; at S = 32 and 64 a page spans two and
four warps, so the valid-row bookkeeping of every gather is exercised.
"""
import math

import numpy as np
import pytest
import torch

import gqa_head_folding_gb300 as g
import oracle
import workloads
from _util import assert_attn_close, check_topk, score_tolerance, to64

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(autouse=True)
def _reset_options():
    yield
    g.set_option(g.GQAQ_OPT_QUEST_KERNEL, 0)
    g.set_option(g.GQAQ_OPT_MAX_CTAS, 0)


def make_case(S, D, G, B=3, Hkv=2, seed=0):
    Lmax = S * 45 + 3
    valid = [Lmax, S * 23 + 5, 2 * S + 1][:B]
    w = workloads.Workload(0, "pages", batch=B, num_layers=1, num_q_heads=G * Hkv, num_kv_heads=Hkv,
                           head_dim=D, max_len=Lmax, page_size=S, n_plant=3, append=True)
    x = workloads.make_layer(w, 0, device="cpu", seed=seed)
    vl = np.array(valid)
    kc = x["k_cache"].numpy().copy()
    vc = x["v_cache"].numpy().copy()
    for b in range(B):                        # the caches after the append at pos = valid - 1
        kc[b, :, vl[b] - 1] = x["k_new"][b].numpy()
        vc[b, :, vl[b] - 1] = x["v_new"][b].numpy()
    return x, vl, kc, vc, Lmax


def check_result(S, x, vl, kc, vc, out, idx, K, scale, meta=None):
    q = x["q"].numpy()
    ref_meta = oracle.page_minmax(kc, vl, S)
    if meta is not None:
        got = to64(meta)
        for b in range(len(vl)):
            P = (vl[b] + S - 1) // S
            assert np.array_equal(got[b, :, :P], ref_meta[b, :, :P]), f"meta b={b}"
    ref_scores = oracle.page_scores(q, ref_meta, vl, S)
    sel = idx.cpu().numpy()
    check_topk(sel, ref_scores, vl, S, K)
    assert_attn_close(out, oracle.sparse_attn(q, kc, vc, vl, sel, S, scale))
    return ref_scores


@pytest.mark.parametrize("S", [8, 32, 64])
@pytest.mark.parametrize("D,G", [(128, 1), (64, 4)])
def test_step_by_step_calls_at_page_size(S, D, G):
    x, vl, kc, vc, Lmax = make_case(S, D, G, seed=S + D + G)
    B, Hkv = kc.shape[0], kc.shape[1]
    K = 9
    kd, vd = x["k_cache"].to(DEV), x["v_cache"].to(DEV)
    vld = torch.tensor(vl, dtype=torch.int32, device=DEV)
    meta = g.new_meta(B, Hkv, Lmax, D, DEV, page_size=S)
    g.quest_update_meta(kd, vld - 1, meta, page_size=S)
    g.quest_append_kv(kd, vd, meta, x["k_new"].to(DEV), x["v_new"].to(DEV), vld - 1, page_size=S)
    q = x["q"].to(DEV)
    scores = g.quest_score_pages(q, meta, vld, Lmax, page_size=S)
    idx = g.quest_topk_pages(scores, vld, K, Lmax, page_size=S)
    scale = 1.0 / math.sqrt(D)
    out = g.quest_sparse_attn(q, kd, vd, vld, idx, scale, page_size=S)
    torch.cuda.synchronize()
    assert g.device_status() == 0
    assert np.array_equal(kd.cpu().numpy(), kc) and np.array_equal(vd.cpu().numpy(), vc)
    ref_scores = check_result(S, x, vl, kc, vc, out, idx, K, scale, meta)
    tol = score_tolerance(oracle.f16_to_f64(x["q"].numpy()), oracle.page_minmax(kc, vl, S), G)
    got = scores.cpu().numpy().astype(np.float64)
    for b in range(B):
        P = (vl[b] + S - 1) // S
        assert np.all(np.abs(got[b, :, :P] - ref_scores[b, :, :P]) <= tol[b, :, :P])


@pytest.mark.parametrize("S", [8, 16, 32, 64])
@pytest.mark.parametrize("kernel,ctas", [("cluster", 0), ("queue", 0), ("queue", 3)])
def test_fused_step_at_page_size(S, kernel, ctas):
    D, G = 128, 4
    x, vl, kc, vc, Lmax = make_case(S, D, G, seed=3 * S + ctas)
    B, Hkv = kc.shape[0], kc.shape[1]
    K = 7
    kd, vd = x["k_cache"].to(DEV), x["v_cache"].to(DEV)
    vld = torch.tensor(vl, dtype=torch.int32, device=DEV)
    meta = g.new_meta(B, Hkv, Lmax, D, DEV, page_size=S)
    g.quest_update_meta(kd, vld - 1, meta, page_size=S)
    g.set_option(g.GQAQ_OPT_QUEST_KERNEL, 1 if kernel == "cluster" else 2)
    g.set_option(g.GQAQ_OPT_MAX_CTAS, ctas)
    ws = g.alloc_workspace(g.dims_of(x["q"], x["k_cache"], S), DEV, K)
    idx = torch.empty(B, Hkv, K, dtype=torch.int32, device=DEV)
    scale = 1.0 / math.sqrt(D)
    out = g.quest_decode_attn(x["q"].to(DEV), kd, vd, meta, vld, K, scale, k_new=x["k_new"].to(DEV),
                              v_new=x["v_new"].to(DEV), pos=vld - 1, page_idx=idx, page_size=S, workspace=ws)
    torch.cuda.synchronize()
    assert g.device_status() == 0
    assert int(ws[:g.workspace_zero_bytes(g.dims_of(x["q"], x["k_cache"], S))].count_nonzero()) == 0
    check_result(S, x, vl, kc, vc, out, idx, K, scale, meta)


@pytest.mark.parametrize("S", [8, 32, 64])
def test_every_page_selected_equals_dense_at_page_size(S):
    D, G, B, Hkv = 64, 2, 2, 2
    Lmax = S * 10 + 3
    w = workloads.Workload(0, "pages", batch=B, num_layers=1, num_q_heads=G * Hkv, num_kv_heads=Hkv,
                           head_dim=D, max_len=Lmax, page_size=S)
    x = workloads.make_layer(w, 0, device=DEV, seed=S)
    vl = torch.tensor([Lmax, S + 1], dtype=torch.int32, device=DEV)
    meta = g.new_meta(B, Hkv, Lmax, D, DEV, page_size=S)
    g.quest_update_meta(x["k_cache"], vl, meta, page_size=S)
    out = g.quest_decode_attn(x["q"], x["k_cache"], x["v_cache"], meta, vl, 64, 0.1, page_size=S)
    ref = oracle.attn_repeat_kv(x["q"].cpu().numpy(), x["k_cache"].cpu().numpy(), x["v_cache"].cpu().numpy(),
                                vl.cpu().numpy(), 0.1)
    assert_attn_close(out, ref)
