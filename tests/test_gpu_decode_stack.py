"""GPU parity of one decode step over a layer stack, launched the way the
decode benchmark launches it, against the fp64 oracle layer by layer.

"Quest: Query-Aware Sparsity ..." review: the first two attention layers keep
full attention; every later layer appends the token, scores each page from its
key min/max, keeps the top-K pages and attends over them (the flowchart).

The stack runs as one CUDA graph of ``DecodeStack.step`` with programmatic
dependent launch and both early-read options on, so a Quest layer's kernel
starts reading metadata while the dense layer ahead of it drains, and each
dense layer reads its first K/V tiles while its own append runs. The graph is
replayed for three decode steps whose appended rows cross page starts (and
reach the last allocated row). Each layer's output, metadata and page list is
checked after every step against the oracle replaying the same appends.

Each case runs twice on the same inputs: once exactly as the benchmark builds
the stack (no page lists written), once with the Quest layers also writing
their page lists. The two must agree bit for bit; the second is then checked
against the oracle (the sparse output over the GPU's validated page set).
"""
import math

import numpy as np
import pytest
import torch

import bench
import gqa_head_folding_gb300 as g
import oracle
import workloads
from _util import assert_attn_close, check_topk, to64
from gqa_head_folding_gb300.decode import DecodeStack, Layer

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
S = 16
LMAX = 16 * 300
NSTEPS = 3
# valid length of each (layer, sequence) before the first step; step s appends
# at row valid + s - 1. Chosen so appends land on page starts (pos % 16 == 0)
# at steps 0, 1 and 2, reach the last allocated row, and one sequence of a
# Quest layer has fewer pages than K (every page selected: equals dense).
VALID0 = [
    [16 * 250 - 1, 16 * 140 + 16],
    [16 * 37 + 1, LMAX - 2],
    [16 * 299 - 1, 16 * 12 + 15],
    [16 * 200 + 1, 16 * 100 - 1],
    [LMAX - 2, 16 * 64 - 1],
]


@pytest.fixture(autouse=True)
def _options():
    g.set_option(g.GQAQ_OPT_PDL, 1)
    g.set_option(g.GQAQ_OPT_QUEST_EARLY_META, 1)
    g.set_option(g.GQAQ_OPT_DENSE_EARLY_KV, 1)
    yield
    g.set_option(g.GQAQ_OPT_QUEST_EARLY_META, 0)
    g.set_option(g.GQAQ_OPT_DENSE_EARLY_KV, 0)


def draw(G, Hkv=4, B=2, D=128, K=16):
    nl = len(VALID0)
    w = workloads.Workload(0, "stack", batch=B, num_layers=nl, num_q_heads=G * Hkv, num_kv_heads=Hkv,
                           head_dim=D, max_len=LMAX, k_pages=K, dense_layers=2, n_plant=3, append=True)
    xs = [workloads.make_layer(w, l, device="cpu", seed=300 + 10 * G + l) for l in range(nl)]
    gen = torch.Generator().manual_seed(400 + G)
    knew = torch.randn(NSTEPS, nl, B, Hkv, D, generator=gen).to(torch.float16)
    vnew = torch.randn(NSTEPS, nl, B, Hkv, D, generator=gen).to(torch.float16)
    vls = np.array([[np.array(VALID0[l]) + s for l in range(nl)] for s in range(NSTEPS)], dtype=np.int32)
    return w, xs, knew, vnew, vls


def run_stack(w, xs, knew, vnew, vls, fused, record):
    """Graph-replay NSTEPS steps; return per-step snapshots of out, meta, page lists."""
    stack = DecodeStack(w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim, w.max_len, w.k_pages,
                        w.dense_layers, DEV, S, fused=fused, num_layers=w.num_layers)
    layers = []
    for l, x in enumerate(xs):
        L = Layer(q=x["q"].to(DEV), k_cache=x["k_cache"].to(DEV), v_cache=x["v_cache"].to(DEV),
                  valid_len=torch.from_numpy(vls[0, l].copy()).to(DEV), out=torch.empty_like(x["q"], device=DEV),
                  meta=stack.new_meta().zero_(), k_new=knew[0, l].to(DEV), v_new=vnew[0, l].to(DEV),
                  pos=torch.from_numpy(vls[0, l] - 1).to(DEV))
        stack.build_meta(L, L.valid_len - 1)        # the pages before the first appended token
        # (pages past the valid length are never written; zeroed so the two runs compare whole)
        if record and not stack.is_dense(l):
            L.page_idx = torch.full((w.batch, w.num_kv_heads, w.k_pages), -7, dtype=torch.int32, device=DEV)
        layers.append(L)
    torch.cuda.synchronize()
    graph = bench.capture(lambda: stack.step(layers), torch.device(DEV))  # runs step 0 once eagerly
    snaps = []
    for s in range(NSTEPS):
        for l, L in enumerate(layers):                # inputs of step s, outside the graph
            L.valid_len.copy_(torch.from_numpy(vls[s, l].copy()))
            L.pos.copy_(torch.from_numpy(vls[s, l] - 1))
            L.k_new.copy_(knew[s, l])
            L.v_new.copy_(vnew[s, l])
            L.out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert g.device_status() == 0, f"device status flag after step {s}"
        snaps.append([(L.out.cpu().clone(), L.meta.cpu().clone(),
                       None if L.page_idx is None else L.page_idx.cpu().clone()) for L in layers])
    caches = [(L.k_cache.cpu(), L.v_cache.cpu()) for L in layers]
    return stack, snaps, caches


@pytest.mark.parametrize("fused", [True, False], ids=["fused", "step-by-step"])
@pytest.mark.parametrize("G", [1, 4])
def test_decode_stack_matches_oracle(G, fused):
    w, xs, knew, vnew, vls = draw(G)
    stack, bench_snaps, bench_caches = run_stack(w, xs, knew, vnew, vls, fused, record=False)
    _, snaps, caches = run_stack(w, xs, knew, vnew, vls, fused, record=True)
    # the benchmark's launch (no page lists) computes exactly the recorded run
    for s in range(NSTEPS):
        for l in range(w.num_layers):
            assert torch.equal(bench_snaps[s][l][0], snaps[s][l][0]), f"out step {s} layer {l}"
            assert torch.equal(bench_snaps[s][l][1], snaps[s][l][1]), f"meta step {s} layer {l}"
    for (ka, va), (kb, vb) in zip(bench_caches, caches):
        assert torch.equal(ka, kb) and torch.equal(va, vb)

    scale = 1.0 / math.sqrt(w.head_dim)
    for l, x in enumerate(xs):
        kc, vc, q = x["k_cache"].numpy().copy(), x["v_cache"].numpy().copy(), x["q"].numpy()
        for s in range(NSTEPS):
            vl = vls[s, l]
            for b in range(w.batch):
                kc[b, :, vl[b] - 1] = knew[s, l, b].numpy()
                vc[b, :, vl[b] - 1] = vnew[s, l, b].numpy()
            out, meta, idx = snaps[s][l]
            ref_meta = oracle.page_minmax(kc, vl, S)
            got_meta = to64(meta)
            for b in range(w.batch):
                P = (int(vl[b]) + S - 1) // S
                assert np.array_equal(got_meta[b, :, :P], ref_meta[b, :, :P]), f"meta step {s} layer {l} b={b}"
            if stack.is_dense(l):
                assert idx is None
                assert_attn_close(out, oracle.attn_repeat_kv(q, kc, vc, vl, scale), f"dense step {s} layer {l}")
            else:
                sel = idx.numpy()
                check_topk(sel, oracle.page_scores(q, ref_meta, vl, S), vl, S, w.k_pages)
                assert_attn_close(out, oracle.sparse_attn(q, kc, vc, vl, sel, S, scale),
                                  f"quest step {s} layer {l}")
        assert np.array_equal(caches[l][0].numpy(), kc) and np.array_equal(caches[l][1].numpy(), vc)


def test_benchmark_step_at_full_size_sampled():
    """The benchmark's default stack (Llama-2-7B shape, 32 layers, 32K context,
    K = 128, layers 0-1 dense, batch 1) built by the benchmark's own state
    builder and graph-replayed once with its launch options; sampled (sequence,
    KV head) units of a dense layer and of the first and last Quest layers
    checked against the oracle."""
    w = workloads.WORKLOADS[3]
    stack, layers, lens = bench.build_state(w, torch.device(DEV))
    for L in layers[2:]:
        L.page_idx = torch.full((w.batch, w.num_kv_heads, w.k_pages), -7, dtype=torch.int32, device=DEV)
    graph = bench.capture(lambda: stack.step(layers), torch.device(DEV))
    for L in layers:
        L.out.fill_(float("nan"))
    graph.replay()
    torch.cuda.synchronize()
    assert g.device_status() == 0
    scale = 1.0 / math.sqrt(w.head_dim)
    G = w.group
    for l in (1, 2, w.num_layers - 1):
        L = layers[l]
        vl = np.array(lens[l], dtype=np.int32)
        for kv in (0, 17, w.num_kv_heads - 1):
            q = L.q[:, kv * G:(kv + 1) * G].cpu().numpy()
            k = L.k_cache[:, kv:kv + 1].cpu().numpy()
            v = L.v_cache[:, kv:kv + 1].cpu().numpy()
            out = L.out[:, kv * G:(kv + 1) * G]
            if stack.is_dense(l):
                assert_attn_close(out, oracle.attn_repeat_kv(q, k, v, vl, scale), f"layer {l} kv {kv}")
                continue
            ref_meta = oracle.page_minmax(k, vl, S)
            P = (int(vl[0]) + S - 1) // S
            assert np.array_equal(to64(L.meta[:, kv:kv + 1, :P]), ref_meta[:, :, :P]), f"meta layer {l} kv {kv}"
            sel = L.page_idx[:, kv:kv + 1].cpu().numpy()
            check_topk(sel, oracle.page_scores(q, ref_meta, vl, S), vl, S, w.k_pages)
            assert_attn_close(out, oracle.sparse_attn(q, k, v, vl, sel, S, scale), f"layer {l} kv {kv}")


@pytest.mark.parametrize("fused", [True, False], ids=["fused", "step-by-step"])
@pytest.mark.parametrize("G", [1, 4])
def test_decode_stack_over_an_e4m3_cache_matches_oracle(G, fused):
    """The same stack over an E4M3 cache (per-tensor scales): dense layers
    through gqa_decode_attn_e4m3, Quest layers as one quest_decode_attn_e4m3
    launch or the step-by-step E4M3 calls (appends keep the pages' E4M3
    bounds), graph-replayed three steps with programmatic launch and both
    early-read options."""
    w, xs, knew, vnew, vls = draw(G)
    stack = DecodeStack(w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim, w.max_len, w.k_pages,
                        w.dense_layers, DEV, S, kv="e4m3", num_layers=w.num_layers, fused=fused)
    layers, host = [], []
    for l, x in enumerate(xs):
        ks = float(x["k_cache"].float().abs().max()) / 448.0
        vs = float(x["v_cache"].float().abs().max()) / 448.0
        kc = oracle.quantize_e4m3(x["k_cache"].numpy(), 1.0 / ks)
        vc = oracle.quantize_e4m3(x["v_cache"].numpy(), 1.0 / vs)
        L = Layer(q=x["q"].to(DEV), k_cache=torch.from_numpy(kc).to(DEV), v_cache=torch.from_numpy(vc).to(DEV),
                  valid_len=torch.from_numpy(vls[0, l].copy()).to(DEV), out=torch.empty_like(x["q"], device=DEV),
                  meta=stack.new_meta().zero_(), k_new=knew[0, l].to(DEV), v_new=vnew[0, l].to(DEV),
                  pos=torch.from_numpy(vls[0, l] - 1).to(DEV), k_scale=ks, v_scale=vs)
        stack.build_meta(L, L.valid_len - 1)
        if not stack.is_dense(l):
            L.page_idx = torch.full((w.batch, w.num_kv_heads, w.k_pages), -7, dtype=torch.int32, device=DEV)
        layers.append(L)
        host.append((kc, vc, ks, vs))
    torch.cuda.synchronize()
    graph = bench.capture(lambda: stack.step(layers), torch.device(DEV))
    scale = 1.0 / math.sqrt(w.head_dim)
    for s in range(NSTEPS):
        for l, L in enumerate(layers):
            L.valid_len.copy_(torch.from_numpy(vls[s, l].copy()))
            L.pos.copy_(torch.from_numpy(vls[s, l] - 1))
            L.k_new.copy_(knew[s, l])
            L.v_new.copy_(vnew[s, l])
            L.out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert g.device_status() == 0
        for l, L in enumerate(layers):
            kc, vc, ks, vs = host[l]
            vl = vls[s, l]
            for b in range(w.batch):
                kc[b, :, vl[b] - 1] = oracle.quantize_e4m3(knew[s, l, b].numpy(), 1.0 / ks)
                vc[b, :, vl[b] - 1] = oracle.quantize_e4m3(vnew[s, l, b].numpy(), 1.0 / vs)
            ref_meta = oracle.page_minmax_e4m3(kc, vl, S)
            got_meta = L.meta.cpu().numpy()
            for b in range(w.batch):
                P = (int(vl[b]) + S - 1) // S
                assert np.array_equal(got_meta[b, :, :P], ref_meta[b, :, :P]), f"bounds step {s} layer {l} b={b}"
            q = xs[l]["q"].numpy()
            if stack.is_dense(l):
                assert_attn_close(L.out, oracle.attn_e4m3(q, kc, vc, ks, vs, vl, scale), f"dense step {s} layer {l}")
            else:
                sel = L.page_idx.cpu().numpy()
                bounds = oracle.e4m3_to_f64(ref_meta) * ks
                check_topk(sel, oracle.page_scores(q, bounds, vl, S), vl, S, w.k_pages)
                assert_attn_close(L.out, oracle.sparse_attn(q, oracle.e4m3_to_f64(kc) * ks, oracle.e4m3_to_f64(vc) * vs,
                                                             vl, sel, S, scale), f"quest step {s} layer {l}")
    for l, L in enumerate(layers):
        assert np.array_equal(L.k_cache.cpu().numpy(), host[l][0])
