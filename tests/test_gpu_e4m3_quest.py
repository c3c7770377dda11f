"""GPU parity of the Quest calls over an 8-bit (E4M3) KV cache against the fp64
oracle ("Quest: Query-Aware Sparsity ..." review: page-score section and
flowchart, with the E4M3 format of the low-bit cache variant).

- quest_append_kv_e4m3 / quest_update_meta_e4m3: codes and page bounds bit
  exact against the oracle's quantizer and page_minmax_e4m3, after every one
  of a run of appends that crosses page starts;
- quest_score_pages_e4m3: within the fp32 summation bound of the oracle's U
  over the dequantized bounds (k_scale * value);
- quest_topk_pages on those scores: the oracle's set up to near-ties;
- quest_sparse_attn_e4m3: within the attention tolerance of the oracle's
  sparse attention over the dequantized cache, on the GPU's page list, over
  D, G and page sizes, and equal to dense E4M3 attention when every page is
  selected.
"""
import math

import numpy as np
import pytest
import torch

import gqa_head_folding_gb300 as g
import oracle
import workloads
from _util import assert_attn_close, check_topk, score_tolerance

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def e4m3_layer(B, G, Hkv, D, Lmax, seed, n_plant=3, S=16):
    w = workloads.Workload(0, "e4m3", batch=B, num_layers=1, num_q_heads=G * Hkv, num_kv_heads=Hkv, head_dim=D,
                           max_len=Lmax, page_size=S, n_plant=n_plant, append=True)
    x = workloads.make_layer(w, 0, device="cpu", seed=seed)
    ks = float(x["k_cache"].float().abs().max()) / 448.0
    vs = float(x["v_cache"].float().abs().max()) / 448.0
    kc = oracle.quantize_e4m3(x["k_cache"].numpy(), 1.0 / ks)
    vc = oracle.quantize_e4m3(x["v_cache"].numpy(), 1.0 / vs)
    return x, kc, vc, ks, vs


def test_appends_write_codes_and_bounds_bit_exact():
    B, Hkv, D, S = 2, 3, 128, 16
    Lmax = 16 * 9
    x, kc, vc, ks, vs = e4m3_layer(B, 1, Hkv, D, Lmax, seed=1)
    start = np.array([16 * 2 - 1, 16 * 5 + 3])
    kd, vd = dev(kc), dev(vc)
    meta = g.new_meta_e4m3(B, Hkv, Lmax, D, DEV).fill_(0x55)
    g.quest_update_meta_e4m3(kd, dev(start.astype(np.int32)), meta)
    gen = torch.Generator().manual_seed(5)
    k_host, v_host = kc.copy(), vc.copy()
    for step in range(2 * S + 3):
        pos = start + step
        kn = (torch.randn(B, Hkv, D, generator=gen) * 2).to(torch.float16)
        vn = torch.randn(B, Hkv, D, generator=gen).to(torch.float16)
        kn[0, 0, :4] = torch.tensor([0.0, -0.0, 448.0 * ks * 4, -1e-9])  # zero, -0, saturation, underflow
        g.quest_append_kv_e4m3(kd, vd, meta, kn.to(DEV), vn.to(DEV), dev(pos.astype(np.int32)), 1.0 / ks, 1.0 / vs)
        for b in range(B):
            k_host[b, :, pos[b]] = oracle.quantize_e4m3(kn[b].numpy(), 1.0 / ks)
            v_host[b, :, pos[b]] = oracle.quantize_e4m3(vn[b].numpy(), 1.0 / vs)
        torch.cuda.synchronize()
        assert g.device_status() == 0
        valid = pos + 1
        ref = oracle.page_minmax_e4m3(k_host, valid, S)
        got = meta.cpu().numpy()
        for b in range(B):
            P = (valid[b] + S - 1) // S
            assert np.array_equal(got[b, :, :P], ref[b, :, :P]), f"bounds step {step} b={b}"
    assert np.array_equal(kd.cpu().numpy(), k_host) and np.array_equal(vd.cpu().numpy(), v_host)


@pytest.mark.parametrize("D", [64, 128])
def test_update_meta_range_and_untouched_pages(D):
    B, Hkv, S, Lmax = 2, 2, 16, 16 * 11 + 5
    x, kc, vc, ks, vs = e4m3_layer(B, 1, Hkv, D, Lmax, seed=2 + D)
    kc[0, 0, 7, :8] = 0x80                               # -0 codes: bounds become +0
    valid = np.array([Lmax, 16 * 3 + 1])
    meta = g.new_meta_e4m3(B, Hkv, Lmax, D, DEV).fill_(0xA5)
    g.quest_update_meta_e4m3(dev(kc), dev(valid.astype(np.int32)), meta, page_begin=2, page_end=9)
    torch.cuda.synchronize()
    got = meta.cpu().numpy()
    ref = oracle.page_minmax_e4m3(kc, valid, S)
    assert np.array_equal(got[0, :, 2:9], ref[0, :, 2:9])
    assert np.array_equal(got[1, :, 2:4], ref[1, :, 2:4])   # sequence 1 has 4 valid pages
    assert np.all(got[1, :, 4:9] == 0xA5) and np.all(got[:, :, :2] == 0xA5) and np.all(got[:, :, 9:] == 0xA5)


@pytest.mark.parametrize("D,G,S", [(128, 1, 16), (128, 4, 16), (64, 8, 16), (64, 2, 8), (128, 4, 32), (128, 2, 64)])
def test_scores_topk_and_sparse_attention(D, G, S):
    B, Hkv, K = 3, 2, 9
    Lmax = S * 40 + 5
    x, kc, vc, ks, vs = e4m3_layer(B, G, Hkv, D, Lmax, seed=10 * D + G + S, S=S)
    valid = np.array([Lmax, S * 17 + 3, S * 5 - 1])
    vl = dev(valid.astype(np.int32))
    kd, vd = dev(kc), dev(vc)
    meta = g.new_meta_e4m3(B, Hkv, Lmax, D, DEV, page_size=S)
    g.quest_update_meta_e4m3(kd, vl, meta, page_size=S)
    scores = g.quest_score_pages_e4m3(x["q"].to(DEV), meta, ks, vl, Lmax, page_size=S)
    idx = g.quest_topk_pages(scores, vl, K, Lmax, page_size=S)
    scale = 1.0 / math.sqrt(D)
    out = g.quest_sparse_attn_e4m3(x["q"].to(DEV), kd, vd, ks, vs, vl, idx, scale, page_size=S)
    torch.cuda.synchronize()
    assert g.device_status() == 0
    q = x["q"].numpy()
    bounds = oracle.e4m3_to_f64(oracle.page_minmax_e4m3(kc, valid, S)) * ks
    ref_scores = oracle.page_scores(q, bounds, valid, S)
    tol = score_tolerance(oracle.f16_to_f64(q), np.nan_to_num(bounds), G)
    got = scores.cpu().numpy().astype(np.float64)
    for b in range(B):
        P = (valid[b] + S - 1) // S
        assert np.all(np.abs(got[b, :, :P] - ref_scores[b, :, :P]) <= tol[b, :, :P]), f"scores b={b}"
    sel = idx.cpu().numpy()
    check_topk(sel, ref_scores, valid, S, K)
    kdq, vdq = oracle.e4m3_to_f64(kc) * ks, oracle.e4m3_to_f64(vc) * vs
    assert_attn_close(out, oracle.sparse_attn(q, kdq, vdq, valid, sel, S, scale))


def test_every_page_selected_equals_dense_e4m3_attention():
    B, G, Hkv, D, S = 2, 4, 2, 128, 16
    Lmax = 16 * 12 + 5
    x, kc, vc, ks, vs = e4m3_layer(B, G, Hkv, D, Lmax, seed=21)
    valid = np.array([Lmax, 33])
    vl = dev(valid.astype(np.int32))
    idx = torch.full((B, Hkv, 20), -1, dtype=torch.int32)
    for b in range(B):
        P = (valid[b] + S - 1) // S
        idx[b, :, :P] = torch.arange(P, dtype=torch.int32)
    sp = g.quest_sparse_attn_e4m3(x["q"].to(DEV), dev(kc), dev(vc), ks, vs, vl, idx.to(DEV), 0.1)
    dn = g.gqa_decode_attn_e4m3(x["q"].to(DEV), dev(kc), dev(vc), ks, vs, vl, 0.1)
    torch.cuda.synchronize()
    ref = oracle.attn_e4m3(x["q"].numpy(), kc, vc, ks, vs, valid, 0.1)
    assert_attn_close(sp, ref)
    assert_attn_close(dn, ref)


def test_sparse_attention_split_over_small_grids():
    # forced small grids: a unit's page tiles split over CTAs and merged in-kernel
    B, G, Hkv, D, S, K = 2, 2, 3, 64, 16, 40
    Lmax = 16 * 60
    x, kc, vc, ks, vs = e4m3_layer(B, G, Hkv, D, Lmax, seed=31)
    valid = np.array([Lmax, 16 * 47 + 9])
    rng = np.random.default_rng(3)
    sel = np.full((B, Hkv, K), -1, np.int32)
    for b in range(B):
        P = (valid[b] + S - 1) // S
        for h in range(Hkv):
            sel[b, h] = np.sort(rng.choice(P, K, replace=False))
    ref = oracle.sparse_attn(x["q"].numpy(), oracle.e4m3_to_f64(kc) * ks, oracle.e4m3_to_f64(vc) * vs, valid, sel, S,
                             0.125)
    try:
        for ctas in (1, 2, 5, 0):
            g.set_option(g.GQAQ_OPT_MAX_CTAS, ctas)
            out = g.quest_sparse_attn_e4m3(x["q"].to(DEV), dev(kc), dev(vc), ks, vs, dev(valid.astype(np.int32)),
                                           dev(sel), 0.125)
            torch.cuda.synchronize()
            assert g.device_status() == 0
            assert_attn_close(out, ref, f"{ctas} CTAs")
    finally:
        g.set_option(g.GQAQ_OPT_MAX_CTAS, 0)


def test_invalid_arguments_are_rejected():
    B, Hkv, D, Lmax = 1, 1, 64, 64
    d = torch.zeros(B, Hkv, Lmax, D, dtype=torch.uint8, device=DEV)
    meta = g.new_meta_e4m3(B, Hkv, Lmax, D, DEV)
    q = torch.zeros(B, Hkv, D, dtype=torch.float16, device=DEV)
    vl = torch.ones(B, dtype=torch.int32, device=DEV)
    for bad in (0.0, -1.0, float("inf")):
        with pytest.raises(g.GqaqError) as e:
            g.quest_score_pages_e4m3(q, meta, bad, vl, Lmax)
        assert e.value.status == g.GQAQ_ERR_INVALID_ARG
    with pytest.raises(g.GqaqError):
        g.quest_update_meta_e4m3(d, vl, meta, page_begin=3, page_end=2)


@pytest.fixture
def _reset_cluster():
    yield
    g.set_option(g.GQAQ_OPT_CLUSTER_SIZE, 0)
    g.set_option(g.GQAQ_OPT_QUEST_EARLY_META, 0)


@pytest.mark.parametrize("D,G,K,csize,S", [
    (128, 4, 8, 0, 16), (128, 1, 16, 4, 16), (128, 4, 16, 2, 16), (64, 2, 40, 8, 16), (128, 8, 3, 1, 16),
    (64, 8, 7, 4, 16), (128, 2, 12, 2, 8), (128, 4, 6, 4, 32), (64, 1, 5, 2, 64),
])
def test_fused_step_over_an_e4m3_cache(D, G, K, csize, S, _reset_cluster):
    """quest_decode_attn_e4m3: append (codes and bounds bit exact), scores
    (times the K scale), page list and attention in one launch, cluster sizes
    1-8 forced, page sizes 8-64, a decode loop of three steps with early
    metadata reads crossing page starts."""
    g.set_option(g.GQAQ_OPT_CLUSTER_SIZE, csize)
    g.set_option(g.GQAQ_OPT_QUEST_EARLY_META, 1)
    B, Hkv = 3, 2
    Lmax = S * 45 + 3
    x, kc, vc, ks, vs = e4m3_layer(B, G, Hkv, D, Lmax, seed=D + 7 * G + K + csize + S, S=S)
    valid0 = np.array([S * 30 - 1, S * 23 + 1, 20])
    kd, vd = dev(kc), dev(vc)
    meta = g.new_meta_e4m3(B, Hkv, Lmax, D, DEV, page_size=S)
    g.quest_update_meta_e4m3(kd, dev((valid0 - 1).astype(np.int32)), meta, page_size=S)
    gen = torch.Generator().manual_seed(D + G)
    scale = 1.0 / math.sqrt(D)
    q = x["q"].numpy()
    Pm = g.num_pages(Lmax, S)
    for step in range(3):
        vl = valid0 + step
        kn = torch.randn(B, Hkv, D, generator=gen).to(torch.float16)
        vn = torch.randn(B, Hkv, D, generator=gen).to(torch.float16)
        scores = torch.full((B, Hkv, Pm), float("nan"), dtype=torch.float32, device=DEV)
        idx = torch.full((B, Hkv, K), -7, dtype=torch.int32, device=DEV)
        out = g.quest_decode_attn_e4m3(x["q"].to(DEV), kd, vd, meta, dev(vl.astype(np.int32)), K, scale, ks, vs,
                                       k_new=kn.to(DEV), v_new=vn.to(DEV), pos=dev((vl - 1).astype(np.int32)),
                                       k_inv_scale=1.0 / ks, v_inv_scale=1.0 / vs, scores=scores, page_idx=idx,
                                       page_size=S)
        torch.cuda.synchronize()
        assert g.device_status() == 0
        for b in range(B):
            kc[b, :, vl[b] - 1] = oracle.quantize_e4m3(kn[b].numpy(), 1.0 / ks)
            vc[b, :, vl[b] - 1] = oracle.quantize_e4m3(vn[b].numpy(), 1.0 / vs)
        assert np.array_equal(kd.cpu().numpy(), kc) and np.array_equal(vd.cpu().numpy(), vc)
        ref_meta = oracle.page_minmax_e4m3(kc, vl, S)
        got_meta = meta.cpu().numpy()
        bounds = oracle.e4m3_to_f64(ref_meta) * ks
        ref_scores = oracle.page_scores(q, bounds, vl, S)
        tol = score_tolerance(oracle.f16_to_f64(q), np.nan_to_num(bounds), G)
        got = scores.cpu().numpy().astype(np.float64)
        for b in range(B):
            P = (vl[b] + S - 1) // S
            assert np.array_equal(got_meta[b, :, :P], ref_meta[b, :, :P]), f"bounds step {step} b={b}"
            assert np.all(np.abs(got[b, :, :P] - ref_scores[b, :, :P]) <= tol[b, :, :P]), f"scores step {step} b={b}"
        sel = idx.cpu().numpy()
        check_topk(sel, ref_scores, vl, S, K)
        assert_attn_close(out, oracle.sparse_attn(q, oracle.e4m3_to_f64(kc) * ks, oracle.e4m3_to_f64(vc) * vs, vl,
                                                  sel, S, scale), f"step {step}")


def test_sparse_attention_above_the_fused_page_limit():
    # k > 1024 selected pages: the split-context kernel gathers E4M3 page boxes
    B, G, Hkv, D, S, K = 1, 4, 2, 64, 16, 1100
    Lmax = 16 * 1200
    x, kc, vc, ks, vs = e4m3_layer(B, G, Hkv, D, Lmax, seed=41, n_plant=0)
    rng = np.random.default_rng(4)
    sel = np.sort(np.stack([rng.choice(1200, K, replace=False) for _ in range(Hkv)]), axis=1)[None].astype(np.int32)
    valid = np.array([Lmax])
    out = g.quest_sparse_attn_e4m3(x["q"].to(DEV), dev(kc), dev(vc), ks, vs, dev(valid.astype(np.int32)), dev(sel),
                                   0.125)
    torch.cuda.synchronize()
    assert g.device_status() == 0
    ref = oracle.sparse_attn(x["q"].numpy(), oracle.e4m3_to_f64(kc) * ks, oracle.e4m3_to_f64(vc) * vs, valid, sel, S,
                             0.125)
    assert_attn_close(out, ref)
