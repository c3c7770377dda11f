"""GPU parity of the Quest path against the fp64 oracle.

- metadata (append and rebuild): bit-exact min/max against the oracle's
  definition, after every append of a run that crosses page boundaries;
- page scores: within the fp32 rounding bound of the fp64 U(p,q);
- top-K: bit-exact on given fp32 scores against numpy's lexsort, and, on
  the full pipeline, equal to the oracle's selection except for near-ties;
- sparse attention: within the output tolerance of the oracle's attention
  over the same pages; with every page selected it equals dense attention.
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
S = 16


@pytest.fixture(autouse=True)
def _reset_options():
    yield
    g.set_option(g.GQAQ_OPT_MAX_CTAS, 0)


def small(B, Hq, Hkv, D, Lmax, n_plant=3, K=8, seed=1):
    w = workloads.Workload(0, "case", batch=B, num_layers=1, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D,
                           max_len=Lmax, k_pages=K, n_plant=n_plant, append=True)
    return w, workloads.make_layer(w, 0, device="cpu", seed=seed)


@pytest.mark.parametrize("D", [64, 128])
def test_append_keeps_exact_page_bounds(D):
    B, Hkv, Lmax = 2, 3, 80
    w, x = small(B, 2 * Hkv, Hkv, D, Lmax)
    k = x["k_cache"].clone(); v = x["v_cache"].clone()
    start = [5, 16]                                  # one run starts mid-page, one on a page start
    vl0 = torch.tensor(start, dtype=torch.int32)
    kd, vd = k.to(DEV), v.to(DEV)
    meta = g.new_meta(B, Hkv, Lmax, D, DEV)
    g.quest_update_meta(kd, vl0.to(DEV), meta)
    gen = torch.Generator().manual_seed(3)
    n_app = 2 * S + 3
    for step in range(n_app):
        pos = torch.tensor([start[0] + step, start[1] + step], dtype=torch.int32)
        kn = torch.randn(B, Hkv, D, generator=gen).to(torch.float16)
        vn = torch.randn(B, Hkv, D, generator=gen).to(torch.float16)
        g.quest_append_kv(kd, vd, meta, kn.to(DEV), vn.to(DEV), pos.to(DEV))
        for b in range(B):
            k[b, :, pos[b]] = kn[b]; v[b, :, pos[b]] = vn[b]
        vl = (pos + 1).numpy()
        ref = oracle.page_minmax(k.numpy(), vl, S)
        got = to64(meta)
        for b in range(B):
            P = (vl[b] + S - 1) // S
            assert np.array_equal(got[b, :, :P], ref[b, :, :P]), f"step {step} b {b}"
    assert torch.equal(kd.cpu(), k) and torch.equal(vd.cpu(), v)


@pytest.mark.parametrize("D", [64, 128])
def test_update_meta_matches_definition(D):
    B, Hkv, Lmax = 3, 2, 203
    w, x = small(B, 4 * Hkv, Hkv, D, Lmax)
    vl = [203, 17, 1]
    meta = g.new_meta(B, Hkv, Lmax, D, DEV)
    meta.fill_(7.0)
    g.quest_update_meta(x["k_cache"].to(DEV), torch.tensor(vl, dtype=torch.int32).to(DEV), meta, 0, 10)
    g.quest_update_meta(x["k_cache"].to(DEV), torch.tensor(vl, dtype=torch.int32).to(DEV), meta, 10, 13)
    ref = oracle.page_minmax(x["k_cache"].numpy(), vl, S)
    got = to64(meta)
    for b in range(B):
        P = (vl[b] + S - 1) // S
        assert np.array_equal(got[b, :, :P], ref[b, :, :P])
        assert np.all(got[b, :, P:] == 7.0)                 # pages with no valid token untouched


@pytest.mark.parametrize("D,G", [(64, 1), (64, 4), (128, 1), (128, 2), (128, 4), (128, 8), (64, 8)])
def test_scores_match_oracle(D, G):
    B, Hkv, Lmax = 2, 2, 16 * 150 + 5
    w, x = small(B, G * Hkv, Hkv, D, Lmax, n_plant=4)
    vl = [Lmax, 16 * 70 + 1]
    vld = torch.tensor(vl, dtype=torch.int32).to(DEV)
    meta = g.new_meta(B, Hkv, Lmax, D, DEV)
    g.quest_update_meta(x["k_cache"].to(DEV), vld, meta)
    scores = g.quest_score_pages(x["q"].to(DEV), meta, vld, Lmax)
    ref_meta = oracle.page_minmax(x["k_cache"].numpy(), vl, S)
    ref = oracle.page_scores(x["q"].numpy(), ref_meta, vl, S)
    tol = score_tolerance(oracle.f16_to_f64(x["q"].numpy()), ref_meta, G)
    got = scores.cpu().numpy().astype(np.float64)
    for b in range(B):
        P = (vl[b] + S - 1) // S
        err = np.abs(got[b, :, :P] - ref[b, :, :P])
        assert np.all(err <= tol[b, :, :P]), f"b={b}: max err {err.max():.3e}"


def test_topk_exact_on_given_scores():
    B, Hkv, Pmax = 3, 4, 300
    rng = np.random.default_rng(5)
    s = rng.standard_normal((B, Hkv, Pmax)).astype(np.float32)
    s[0, 0, 10:20] = 2.5                      # ties straddling the cut
    s[1, 1, :] = 0.0
    s[1, 2, ::2] = -0.0                       # signed zeros tie with +0
    s[2, 3, :] = np.float32(1e-30) * rng.integers(-3, 3, Pmax)
    vl = [300 * S, 200 * S - 3, 57]
    for K in (1, 7, 64, 250):
        idx = g.quest_topk_pages(torch.from_numpy(s).to(DEV), torch.tensor(vl, dtype=torch.int32).to(DEV), K,
                                 Pmax * S).cpu().numpy()
        for b in range(B):
            P = (vl[b] + S - 1) // S
            n = min(K, P)
            for h in range(Hkv):
                sc = s[b, h, :P].astype(np.float64)
                ref = np.sort(np.lexsort((np.arange(P), -sc))[:n])
                assert np.array_equal(idx[b, h, :n], ref), (K, b, h)
                assert np.all(idx[b, h, n:] == -1)


@pytest.mark.parametrize("D,G,K", [(128, 4, 8), (128, 1, 16), (64, 4, 5), (64, 2, 40), (128, 8, 3)])
@pytest.mark.parametrize("max_ctas", [0, 5])
def test_quest_pipeline(D, G, K, max_ctas):
    g.set_option(g.GQAQ_OPT_MAX_CTAS, max_ctas)
    B, Hkv, Lmax = 2, 2, 16 * 40
    w, x = small(B, G * Hkv, Hkv, D, Lmax, n_plant=3, K=K, seed=D + G + K)
    vl = np.array([Lmax, 16 * 23 + 7])
    pos = torch.tensor(vl - 1, dtype=torch.int32)
    kd, vd = x["k_cache"].to(DEV), x["v_cache"].to(DEV)
    vld = torch.tensor(vl, dtype=torch.int32).to(DEV)
    meta = g.new_meta(B, Hkv, Lmax, D, DEV)
    g.quest_update_meta(kd, vld - 1, meta)
    g.quest_append_kv(kd, vd, meta, x["k_new"].to(DEV), x["v_new"].to(DEV), pos.to(DEV))
    scores = g.quest_score_pages(x["q"].to(DEV), meta, vld, Lmax)
    idx = g.quest_topk_pages(scores, vld, K, Lmax)
    scale = 1.0 / math.sqrt(D)
    out = g.quest_sparse_attn(x["q"].to(DEV), kd, vd, vld, idx, scale)
    torch.cuda.synchronize()
    assert g.device_status() == 0

    kc = x["k_cache"].numpy().copy(); vc = x["v_cache"].numpy().copy()
    for b in range(B):
        kc[b, :, vl[b] - 1] = x["k_new"][b].numpy(); vc[b, :, vl[b] - 1] = x["v_new"][b].numpy()
    ref_meta = oracle.page_minmax(kc, vl, S)
    got_meta = to64(meta)
    for b in range(B):
        P = (vl[b] + S - 1) // S
        assert np.array_equal(got_meta[b, :, :P], ref_meta[b, :, :P])
    ref_scores = oracle.page_scores(x["q"].numpy(), ref_meta, vl, S)
    sel = idx.cpu().numpy()
    check_topk(sel, ref_scores, vl, S, K)
    ref = oracle.sparse_attn(x["q"].numpy(), kc, vc, vl, sel, S, scale)
    assert_attn_close(out, ref)


@pytest.mark.parametrize("D,G", [(128, 4), (64, 1)])
def test_sparse_with_every_page_equals_dense(D, G):
    B, Hkv, Lmax = 2, 3, 16 * 33
    w, x = small(B, G * Hkv, Hkv, D, Lmax, seed=4)
    vl = np.array([Lmax, 100])
    K = 40                                         # >= P for both sequences
    vld = torch.tensor(vl, dtype=torch.int32).to(DEV)
    idx = torch.full((B, Hkv, K), -1, dtype=torch.int32)
    for b in range(B):
        P = (vl[b] + S - 1) // S
        idx[b, :, :P] = torch.arange(P, dtype=torch.int32)
    q, kd, vd = x["q"].to(DEV), x["k_cache"].to(DEV), x["v_cache"].to(DEV)
    sp = g.quest_sparse_attn(q, kd, vd, vld, idx.to(DEV), 0.09)
    dn = g.gqa_decode_attn(q, kd, vd, vld, 0.09)
    ref = oracle.attn_repeat_kv(x["q"].numpy(), x["k_cache"].numpy(), x["v_cache"].numpy(), vl, 0.09)
    assert_attn_close(sp, ref, "sparse(all pages)")
    assert_attn_close(dn, ref, "dense")
    # the top-K call with K >= P selects every page
    scores = torch.zeros(B, Hkv, (Lmax + S - 1) // S, dtype=torch.float32, device=DEV)
    sel = g.quest_topk_pages(scores, vld, K, Lmax).cpu()
    assert torch.equal(sel, idx)


def test_sparse_skips_padding_and_bad_indices():
    B, Hkv, D, Lmax = 1, 2, 128, 16 * 10
    w, x = small(B, 4 * Hkv, Hkv, D, Lmax, seed=8)
    vl = np.array([16 * 9 + 3])
    idx = torch.tensor([[[0, 3, -1, 9, 77], [2, -5, 4, -1, -1]]], dtype=torch.int32)
    g.device_status(reset=True)
    out = g.quest_sparse_attn(x["q"].to(DEV), x["k_cache"].to(DEV), x["v_cache"].to(DEV),
                              torch.tensor(vl, dtype=torch.int32).to(DEV), idx.to(DEV), 0.1)
    assert g.device_status(reset=True) & g.GQAQ_DEV_BAD_PAGE
    ref = oracle.sparse_attn(x["q"].numpy(), x["k_cache"].numpy(), x["v_cache"].numpy(), vl,
                             idx.numpy(), S, 0.1)
    assert_attn_close(out, ref)


def test_append_out_of_range_position_is_skipped():
    B, Hkv, D, Lmax = 2, 2, 64, 32
    w, x = small(B, 2 * Hkv, Hkv, D, Lmax, seed=2)
    kd, vd = x["k_cache"].to(DEV), x["v_cache"].to(DEV)
    meta = g.new_meta(B, Hkv, Lmax, D, DEV)
    g.quest_update_meta(kd, torch.tensor([Lmax, Lmax], dtype=torch.int32).to(DEV), meta)
    before_k, before_m = kd.clone(), meta.clone()
    g.device_status(reset=True)
    g.quest_append_kv(kd, vd, meta, x["k_new"].to(DEV), x["v_new"].to(DEV),
                      torch.tensor([Lmax, -1], dtype=torch.int32).to(DEV))
    assert g.device_status(reset=True) & g.GQAQ_DEV_BAD_POS
    assert torch.equal(kd, before_k) and torch.equal(meta, before_m)


def test_quest_step_graph_replay_matches_eager():
    w = workloads.WORKLOADS[4].with_(batch=2, max_len=16 * 200)
    x = workloads.make_layer(w, 0, device=DEV)
    B, Hkv, Lmax, D = x["k_cache"].shape
    meta = g.new_meta(B, Hkv, Lmax, D, DEV)
    g.quest_update_meta(x["k_cache"], x["valid_len"] - 1, meta)
    d = g.dims_of(x["q"], x["k_cache"])
    ws = g.alloc_workspace(d, DEV)
    scores = torch.empty(B, Hkv, g.num_pages(Lmax), dtype=torch.float32, device=DEV)
    idx = torch.empty(B, Hkv, 64, dtype=torch.int32, device=DEV)
    out = torch.empty_like(x["q"])

    def step():
        g.quest_append_kv(x["k_cache"], x["v_cache"], meta, x["k_new"], x["v_new"], x["pos"])
        g.quest_score_pages(x["q"], meta, x["valid_len"], Lmax, scores=scores)
        g.quest_topk_pages(scores, x["valid_len"], 64, Lmax, page_idx=idx)
        g.quest_sparse_attn(x["q"], x["k_cache"], x["v_cache"], x["valid_len"], idx, 0.088, out=out, workspace=ws)

    step()
    eager_out, eager_idx = out.clone(), idx.clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            step()
    torch.cuda.current_stream().wait_stream(s)
    out.zero_(); idx.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(idx, eager_idx)
    assert torch.equal(out, eager_out)


def test_wait_timeout_is_reported_and_context_survives():
    # the producer issues nothing, so every consumer wait runs out after 1 ms
    w = workloads.Workload(0, "case", batch=1, num_layers=1, num_q_heads=8, num_kv_heads=2, head_dim=128,
                           max_len=512)
    x = workloads.make_layer(w, 0, device=DEV, seed=3)
    args = (x["q"], x["k_cache"], x["v_cache"], x["valid_len"])
    ws = g.alloc_workspace(g.dims_of(x["q"], x["k_cache"]), DEV)
    g.device_status(reset=True)
    try:
        g.set_option(g.GQAQ_OPT_WAIT_TIMEOUT_NS, 1_000_000)
        g.set_option(g.GQAQ_OPT_TEST_STALL, 1)
        g.set_option(g.GQAQ_OPT_MAX_CTAS, 5)         # every unit split: counters in use
        g.gqa_decode_attn(*args, 0.1, workspace=ws)
        flags = g.device_status(reset=True)
    finally:
        g.set_option(g.GQAQ_OPT_TEST_STALL, 0)
        g.set_option(g.GQAQ_OPT_WAIT_TIMEOUT_NS, 2_000_000_000)
        g.set_option(g.GQAQ_OPT_MAX_CTAS, 0)
    assert flags & g.GQAQ_DEV_TIMEOUT
    torch.cuda.synchronize()
    assert int(ws[:256].count_nonzero()) == 0      # arrival counters back at zero
    out = g.gqa_decode_attn(*args, 0.1, workspace=ws)   # the context and the workspace are still usable
    ref = oracle.attn_repeat_kv(x["q"].cpu().numpy(), x["k_cache"].cpu().numpy(), x["v_cache"].cpu().numpy(),
                                x["valid_len"].cpu().numpy(), 0.1)
    assert_attn_close(out, ref)
    assert g.device_status(reset=True) == 0
