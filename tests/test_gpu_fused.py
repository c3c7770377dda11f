"""GPU parity of quest_decode_attn, the fused Quest step (append, page scores,
top-K, sparse attention in one launch), against the fp64 oracle, for both of
its kernels.

Cluster kernel (no workspace): cluster sizes 1, 2, 4 and 8 are forced so the
cross-CTA paths (radix threshold from summed histograms, page-list
compaction, log-sum-exp merge through distributed shared memory) all run,
including CTAs whose page range or page share is empty.

Work-queue kernel (with a workspace): grids are forced down to 1..7 CTAs so
one CTA holds many items, waits for page lists that its own ring has still
to select, and merges partials that other CTAs wrote; the workspace's
counters and flags must be back at zero after every call.
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
    g.set_option(g.GQAQ_OPT_CLUSTER_SIZE, 0)
    g.set_option(g.GQAQ_OPT_MAX_CTAS, 0)
    g.set_option(g.GQAQ_OPT_QUEST_KERNEL, 0)
    g.set_option(g.GQAQ_OPT_QUEST_EARLY_META, 0)


def use_queue_kernel():
    g.set_option(g.GQAQ_OPT_QUEST_KERNEL, 2)


def zero_region_clear(ws, B, Hkv):
    torch.cuda.synchronize()
    return int(ws[:g.workspace_zero_bytes(g.make_dims(B, Hkv, Hkv, 64, 16))].count_nonzero()) == 0


def run_fused(D, G, K, csize, B=3, Hkv=2, Lmax=16 * 45 + 3, valid=(16 * 45 + 3, 16 * 23 + 7, 20), seed=0,
              append=True, queue_ctas=None):
    """csize: forced cluster size (cluster kernel). queue_ctas: when not None,
    run the work-queue kernel on that many CTAs (0 = the full grid)."""
    g.set_option(g.GQAQ_OPT_CLUSTER_SIZE, csize)
    ws = None
    if queue_ctas is not None:
        use_queue_kernel()
        g.set_option(g.GQAQ_OPT_MAX_CTAS, queue_ctas)
        ws = g.alloc_workspace(g.make_dims(B, G * Hkv, Hkv, D, Lmax), DEV, K)
    w = workloads.Workload(0, "fused", batch=B, num_layers=1, num_q_heads=G * Hkv, num_kv_heads=Hkv,
                           head_dim=D, max_len=Lmax, k_pages=K, n_plant=3, append=True)
    x = workloads.make_layer(w, 0, device="cpu", seed=seed)
    vl = np.array(valid[:B])
    kd, vd = x["k_cache"].to(DEV), x["v_cache"].to(DEV)
    vld = torch.tensor(vl, dtype=torch.int32, device=DEV)
    meta = g.new_meta(B, Hkv, Lmax, D, DEV)
    pos = torch.tensor(vl - 1, dtype=torch.int32)
    g.quest_update_meta(kd, vld - 1 if append else vld, meta)
    scores = torch.full((B, Hkv, g.num_pages(Lmax)), float("nan"), dtype=torch.float32, device=DEV)
    idx = torch.full((B, Hkv, K), -7, dtype=torch.int32, device=DEV)
    scale = 1.0 / math.sqrt(D)
    kw = dict(k_new=x["k_new"].to(DEV), v_new=x["v_new"].to(DEV), pos=pos.to(DEV)) if append else {}
    out = g.quest_decode_attn(x["q"].to(DEV), kd, vd, meta, vld, K, scale, scores=scores, page_idx=idx,
                              workspace=ws, **kw)
    torch.cuda.synchronize()
    assert g.device_status() == 0
    if ws is not None:
        assert zero_region_clear(ws, B, Hkv)

    kc = x["k_cache"].numpy().copy(); vc = x["v_cache"].numpy().copy()
    if append:
        for b in range(B):
            kc[b, :, vl[b] - 1] = x["k_new"][b].numpy(); vc[b, :, vl[b] - 1] = x["v_new"][b].numpy()
    assert np.array_equal(kd.cpu().numpy(), kc) and np.array_equal(vd.cpu().numpy(), vc)
    ref_meta = oracle.page_minmax(kc, vl, S)
    got_meta = to64(meta)
    ref_scores = oracle.page_scores(x["q"].numpy(), ref_meta, vl, S)
    tol = score_tolerance(oracle.f16_to_f64(x["q"].numpy()), ref_meta, G)
    got_scores = scores.cpu().numpy().astype(np.float64)
    for b in range(B):
        P = (vl[b] + S - 1) // S
        assert np.array_equal(got_meta[b, :, :P], ref_meta[b, :, :P]), f"meta b={b}"
        assert np.all(np.abs(got_scores[b, :, :P] - ref_scores[b, :, :P]) <= tol[b, :, :P]), f"scores b={b}"
    sel = idx.cpu().numpy()
    check_topk(sel, ref_scores, vl, S, K)
    ref = oracle.sparse_attn(x["q"].numpy(), kc, vc, vl, sel, S, scale)
    assert_attn_close(out, ref)
    return out, sel


@pytest.mark.parametrize("D,G,K,csize", [
    (128, 4, 8, 0), (128, 4, 8, 1), (128, 4, 8, 2), (128, 4, 16, 4), (128, 1, 16, 8),
    (64, 4, 5, 2), (64, 2, 40, 0), (128, 8, 3, 2), (64, 8, 7, 4), (64, 1, 12, 1), (128, 2, 30, 8),
])
def test_fused_matches_oracle(D, G, K, csize):
    run_fused(D, G, K, csize, seed=D + 10 * G + K + csize)


@pytest.mark.parametrize("csize", [1, 4])
def test_fused_without_append(csize):
    run_fused(128, 4, 9, csize, append=False, seed=77)


@pytest.mark.parametrize("D,G,K,ctas", [
    (128, 4, 8, 0), (128, 1, 16, 1), (128, 4, 16, 2), (64, 4, 5, 2), (64, 2, 40, 0), (128, 8, 3, 3),
    (64, 8, 7, 5), (64, 1, 12, 1), (128, 2, 30, 7), (128, 1, 200, 4),
])
def test_queue_kernel_matches_oracle(D, G, K, ctas):
    run_fused(D, G, K, 0, seed=D + 10 * G + K + ctas, queue_ctas=ctas)


@pytest.mark.parametrize("ctas", [0, 1])
def test_queue_kernel_without_append(ctas):
    run_fused(128, 4, 9, 0, append=False, seed=78, queue_ctas=ctas)


@pytest.mark.parametrize("ctas", [0, 3])
def test_queue_kernel_long_ragged_batch(ctas):
    # more metadata tiles per sequence than one score item holds, ragged lengths
    run_fused(128, 2, 24, 0, B=4, Hkv=3, Lmax=16 * 700 + 9, valid=(16 * 700 + 9, 16 * 301, 130, 16 * 129 + 1),
              seed=91, queue_ctas=ctas)


def test_queue_kernel_more_than_1024_pages():
    # k beyond the cluster kernel's limit
    run_fused(64, 4, 1100, 0, B=1, Hkv=2, Lmax=16 * 1500, valid=(16 * 1500 - 3,), seed=5, queue_ctas=0)


def test_default_kernel_choice_by_k():
    # automatic choice: k <= 1024 needs no workspace (cluster kernel); k > 1024
    # takes the work queue and so a workspace
    B, Hkv, D, G, Lmax = 1, 2, 64, 4, 16 * 1300
    w = workloads.Workload(0, "big-k", batch=B, num_layers=1, num_q_heads=G * Hkv, num_kv_heads=Hkv,
                           head_dim=D, max_len=Lmax)
    x = workloads.make_layer(w, 0, device=DEV, seed=8)
    meta = g.new_meta(B, Hkv, Lmax, D, DEV)
    g.quest_update_meta(x["k_cache"], x["valid_len"], meta)
    args = (x["q"], x["k_cache"], x["v_cache"], meta, x["valid_len"])
    g.quest_decode_attn(*args, 1024, 0.1)
    with pytest.raises(g.GqaqError):
        g.quest_decode_attn(*args, 1025, 0.1)
    ws = g.alloc_workspace(g.dims_of(x["q"], x["k_cache"]), DEV, 1025)
    idx = torch.empty(B, Hkv, 1025, dtype=torch.int32, device=DEV)
    out = g.quest_decode_attn(*args, 1025, 0.1, page_idx=idx, workspace=ws)
    torch.cuda.synchronize()
    assert g.device_status() == 0
    vl = x["valid_len"].cpu().numpy()
    q, kc, vc = x["q"].cpu().numpy(), x["k_cache"].cpu().numpy(), x["v_cache"].cpu().numpy()
    sel = idx.cpu().numpy()
    check_topk(sel, oracle.page_scores(q, oracle.page_minmax(kc, vl, S), vl, S), vl, S, 1025)
    assert_attn_close(out, oracle.sparse_attn(q, kc, vc, vl, sel, S, 0.1))


def test_queue_kernel_empty_sequence_gives_zeros():
    B, Hkv, D, G, Lmax, K = 3, 2, 128, 4, 16 * 40, 6
    w = workloads.Workload(0, "fused", batch=B, num_layers=1, num_q_heads=G * Hkv, num_kv_heads=Hkv,
                           head_dim=D, max_len=Lmax)
    x = workloads.make_layer(w, 0, device=DEV, seed=12)
    vl = torch.tensor([16 * 40, 0, 77], dtype=torch.int32, device=DEV)
    use_queue_kernel()
    meta = g.new_meta(B, Hkv, Lmax, D, DEV)
    g.quest_update_meta(x["k_cache"], vl, meta)
    ws = g.alloc_workspace(g.make_dims(B, G * Hkv, Hkv, D, Lmax), DEV, K)
    g.device_status(reset=True)
    out = g.quest_decode_attn(x["q"], x["k_cache"], x["v_cache"], meta, vl, K, 0.09, workspace=ws)
    assert g.device_status(reset=True) & g.GQAQ_DEV_BAD_LEN
    assert zero_region_clear(ws, B, Hkv)
    assert bool((out[1] == 0).all())
    keep = [0, 2]
    idx = torch.empty(B, Hkv, K, dtype=torch.int32, device=DEV)
    out2 = g.quest_decode_attn(x["q"], x["k_cache"], x["v_cache"], meta, vl, K, 0.09, page_idx=idx, workspace=ws)
    assert torch.equal(out, out2)
    vk = vl.cpu().numpy()[keep]
    sel = idx.cpu().numpy()[keep]
    q = x["q"].cpu().numpy()[keep]; kc = x["k_cache"].cpu().numpy()[keep]; vc = x["v_cache"].cpu().numpy()[keep]
    ref_scores = oracle.page_scores(q, oracle.page_minmax(kc, vk, S), vk, S)
    check_topk(sel, ref_scores, vk, S, K)
    assert_attn_close(out[keep], oracle.sparse_attn(q, kc, vc, vk, sel, S, 0.09))


def test_queue_kernel_repeatable_and_graph_capturable():
    w = workloads.WORKLOADS[4].with_(batch=3, max_len=16 * 300)
    x = workloads.make_layer(w, 0, device=DEV)
    B, Hkv, Lmax, D = x["k_cache"].shape
    meta = g.new_meta(B, Hkv, Lmax, D, DEV)
    g.quest_update_meta(x["k_cache"], x["valid_len"] - 1, meta)
    out = torch.empty_like(x["q"])
    idx = torch.empty(B, Hkv, 64, dtype=torch.int32, device=DEV)
    ws = g.alloc_workspace(g.dims_of(x["q"], x["k_cache"]), DEV, 64)
    use_queue_kernel()

    def step():
        g.quest_decode_attn(x["q"], x["k_cache"], x["v_cache"], meta, x["valid_len"], 64, 0.088,
                            k_new=x["k_new"], v_new=x["v_new"], pos=x["pos"], out=out, page_idx=idx, workspace=ws)

    step()
    first_out, first_idx = out.clone(), idx.clone()
    for _ in range(3):
        step()                                          # re-appending the same token is idempotent
        assert torch.equal(out, first_out) and torch.equal(idx, first_idx)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            step()
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(3):
        out.zero_(); idx.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, first_out) and torch.equal(idx, first_idx)
    assert zero_region_clear(ws, B, Hkv)
    # the cluster kernel (no workspace) selects the same pages
    g.set_option(g.GQAQ_OPT_QUEST_KERNEL, 0)
    idx2 = torch.empty_like(idx)
    g.quest_decode_attn(x["q"], x["k_cache"], x["v_cache"], meta, x["valid_len"], 64, 0.088, page_idx=idx2)
    assert torch.equal(idx2, first_idx)


def test_queue_kernel_timeout_is_reported_and_context_survives():
    # the producers issue nothing, so every consumer wait runs out after 1 ms
    B, Hkv, D, G, Lmax, K = 2, 2, 128, 2, 16 * 64, 8
    w = workloads.Workload(0, "fused", batch=B, num_layers=1, num_q_heads=G * Hkv, num_kv_heads=Hkv,
                           head_dim=D, max_len=Lmax)
    x = workloads.make_layer(w, 0, device=DEV, seed=4)
    meta = g.new_meta(B, Hkv, Lmax, D, DEV)
    g.quest_update_meta(x["k_cache"], x["valid_len"], meta)
    ws = g.alloc_workspace(g.make_dims(B, G * Hkv, Hkv, D, Lmax), DEV, K)
    args = (x["q"], x["k_cache"], x["v_cache"], meta, x["valid_len"], K, 0.1)
    use_queue_kernel()
    g.device_status(reset=True)
    try:
        g.set_option(g.GQAQ_OPT_WAIT_TIMEOUT_NS, 1_000_000)
        g.set_option(g.GQAQ_OPT_TEST_STALL, 1)
        g.quest_decode_attn(*args, workspace=ws)
        flags = g.device_status(reset=True)
    finally:
        g.set_option(g.GQAQ_OPT_TEST_STALL, 0)
        g.set_option(g.GQAQ_OPT_WAIT_TIMEOUT_NS, 2_000_000_000)
    assert flags & g.GQAQ_DEV_TIMEOUT
    ws.zero_()                                           # the documented reset after a timeout
    idx = torch.empty(B, Hkv, K, dtype=torch.int32, device=DEV)
    out = g.quest_decode_attn(*args, page_idx=idx, workspace=ws)
    assert g.device_status(reset=True) == 0
    vl = x["valid_len"].cpu().numpy()
    q, kc, vc = x["q"].cpu().numpy(), x["k_cache"].cpu().numpy(), x["v_cache"].cpu().numpy()
    sel = idx.cpu().numpy()
    check_topk(sel, oracle.page_scores(q, oracle.page_minmax(kc, vl, S), vl, S), vl, S, K)
    assert_attn_close(out, oracle.sparse_attn(q, kc, vc, vl, sel, S, 0.1))


@pytest.mark.parametrize("csize", [2, 8])
def test_fused_with_every_page_selected_equals_dense(csize):
    B, Hkv, D, G, Lmax = 2, 2, 128, 4, 16 * 12 + 5
    g.set_option(g.GQAQ_OPT_CLUSTER_SIZE, csize)
    w = workloads.Workload(0, "fused", batch=B, num_layers=1, num_q_heads=G * Hkv, num_kv_heads=Hkv,
                           head_dim=D, max_len=Lmax)
    x = workloads.make_layer(w, 0, device=DEV, seed=5)
    vl = torch.tensor([Lmax, 33], dtype=torch.int32, device=DEV)
    meta = g.new_meta(B, Hkv, Lmax, D, DEV)
    g.quest_update_meta(x["k_cache"], vl, meta)
    idx = torch.empty(B, Hkv, 20, dtype=torch.int32, device=DEV)
    sp = g.quest_decode_attn(x["q"], x["k_cache"], x["v_cache"], meta, vl, 20, 0.1, page_idx=idx)
    ref = oracle.attn_repeat_kv(x["q"].cpu().numpy(), x["k_cache"].cpu().numpy(), x["v_cache"].cpu().numpy(),
                                vl.cpu().numpy(), 0.1)
    assert_attn_close(sp, ref)
    for b, P in enumerate([13, 3]):
        assert idx[b, :, :P].tolist() == [list(range(P))] * Hkv
        assert bool((idx[b, :, P:] == -1).all())


def test_fused_repeatable_and_graph_capturable():
    w = workloads.WORKLOADS[4].with_(batch=3, max_len=16 * 300)
    x = workloads.make_layer(w, 0, device=DEV)
    B, Hkv, Lmax, D = x["k_cache"].shape
    meta = g.new_meta(B, Hkv, Lmax, D, DEV)
    g.quest_update_meta(x["k_cache"], x["valid_len"] - 1, meta)
    out = torch.empty_like(x["q"])
    idx = torch.empty(B, Hkv, 64, dtype=torch.int32, device=DEV)

    def step():
        g.quest_decode_attn(x["q"], x["k_cache"], x["v_cache"], meta, x["valid_len"], 64, 0.088,
                            k_new=x["k_new"], v_new=x["v_new"], pos=x["pos"], out=out, page_idx=idx)

    step()
    first_out, first_idx = out.clone(), idx.clone()
    step()                                              # re-appending the same token is idempotent
    assert torch.equal(out, first_out) and torch.equal(idx, first_idx)
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
    assert torch.equal(out, first_out) and torch.equal(idx, first_idx)


def test_sparse_call_above_the_fused_page_limit():
    # k > 1024 selected pages goes through the split-context kernel + combine
    B, Hkv, D, G, Lmax = 1, 2, 64, 4, 16 * 1200
    w = workloads.Workload(0, "big-k", batch=B, num_layers=1, num_q_heads=G * Hkv, num_kv_heads=Hkv,
                           head_dim=D, max_len=Lmax)
    x = workloads.make_layer(w, 0, device=DEV, seed=2)
    K = 1100
    rng = np.random.default_rng(0)
    sel = np.sort(np.stack([rng.choice(1200, K, replace=False) for _ in range(Hkv)]), axis=1)[None].astype(np.int32)
    vl = x["valid_len"]
    out = g.quest_sparse_attn(x["q"], x["k_cache"], x["v_cache"], vl, torch.from_numpy(sel).to(DEV), 0.125)
    ref = oracle.sparse_attn(x["q"].cpu().numpy(), x["k_cache"].cpu().numpy(), x["v_cache"].cpu().numpy(),
                             vl.cpu().numpy(), sel, S, 0.125)
    assert_attn_close(out, ref)
    with pytest.raises(g.GqaqError):              # the cluster kernel stops at 1024 pages
        meta = g.new_meta(B, Hkv, Lmax, D, DEV)
        g.quest_decode_attn(x["q"], x["k_cache"], x["v_cache"], meta, vl, K, 0.125)


@pytest.mark.parametrize("csize,valid0", [(1, (16 * 30 - 1, 16 * 23 + 15, 17)), (4, (16 * 44 - 2, 16 * 8, 33)),
                                          (8, (16 * 45 + 1, 16 * 16 - 1, 2))])
def test_fused_early_metadata_decode_loop(csize, valid0):
    """GQAQ_OPT_QUEST_EARLY_META: two layers, three decode steps, every call
    launched right behind the other layer's (programmatic launch), as a decode
    loop does. Steps cross page boundaries (pos % S == 0, the case where the
    previous step wrote the page before the appended one); each output and
    page list is checked against the oracle replaying the appends."""
    g.set_option(g.GQAQ_OPT_CLUSTER_SIZE, csize)
    g.set_option(g.GQAQ_OPT_QUEST_EARLY_META, 1)
    B, Hkv, G, D, K = 3, 2, 4, 128, 8
    Lmax, nsteps, nl = 16 * 45 + 3, 3, 2
    w = workloads.Workload(0, "fused", batch=B, num_layers=nl, num_q_heads=G * Hkv, num_kv_heads=Hkv,
                           head_dim=D, max_len=Lmax, k_pages=K, n_plant=3, append=True)
    xs = [workloads.make_layer(w, l, device="cpu", seed=50 + csize + l) for l in range(nl)]
    gen = torch.Generator().manual_seed(90 + csize)
    knew = torch.randn(nsteps, nl, B, Hkv, D, generator=gen).to(torch.float16)
    vnew = torch.randn(nsteps, nl, B, Hkv, D, generator=gen).to(torch.float16)
    vls = [np.array(valid0) + s for s in range(nsteps)]
    vld = [torch.tensor(v, dtype=torch.int32, device=DEV) for v in vls]       # made before the loop:
    posd = [torch.tensor(v - 1, dtype=torch.int32, device=DEV) for v in vls]  # no kernel writes them in it
    kd = [x["k_cache"].to(DEV) for x in xs]
    vd = [x["v_cache"].to(DEV) for x in xs]
    qd = [x["q"].to(DEV) for x in xs]
    metas = [g.new_meta(B, Hkv, Lmax, D, DEV) for _ in range(nl)]
    for l in range(nl):
        g.quest_update_meta(kd[l], vld[0] - 1, metas[l])
    kn, vn = knew.to(DEV), vnew.to(DEV)
    outs = torch.empty(nsteps, nl, B, G * Hkv, D, dtype=torch.float16, device=DEV)
    idx = torch.full((nsteps, nl, B, Hkv, K), -7, dtype=torch.int32, device=DEV)
    scale = 1.0 / math.sqrt(D)
    torch.cuda.synchronize()
    for s in range(nsteps):
        for l in range(nl):
            g.quest_decode_attn(qd[l], kd[l], vd[l], metas[l], vld[s], K, scale, k_new=kn[s, l], v_new=vn[s, l],
                                pos=posd[s], out=outs[s, l], page_idx=idx[s, l])
    torch.cuda.synchronize()
    assert g.device_status() == 0
    for l in range(nl):
        kc = xs[l]["k_cache"].numpy().copy(); vc = xs[l]["v_cache"].numpy().copy()
        q = xs[l]["q"].numpy()
        for s in range(nsteps):
            vl = vls[s]
            for b in range(B):
                kc[b, :, vl[b] - 1] = knew[s, l, b].numpy(); vc[b, :, vl[b] - 1] = vnew[s, l, b].numpy()
            ref_meta = oracle.page_minmax(kc, vl, S)
            ref_scores = oracle.page_scores(q, ref_meta, vl, S)
            sel = idx[s, l].cpu().numpy()
            check_topk(sel, ref_scores, vl, S, K)
            assert_attn_close(outs[s, l], oracle.sparse_attn(q, kc, vc, vl, sel, S, scale), f"step {s} layer {l}")
        assert np.array_equal(kd[l].cpu().numpy(), kc) and np.array_equal(vd[l].cpu().numpy(), vc)
        got_meta = to64(metas[l])
        for b in range(B):
            P = (vls[-1][b] + S - 1) // S
            assert np.array_equal(got_meta[b, :, :P], ref_meta[b, :, :P]), f"meta layer {l} b={b}"
