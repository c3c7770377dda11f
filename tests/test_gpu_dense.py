"""GPU parity of gqa_decode_attn (dense folded-GQA decode) against the fp64
oracle's explicit-repeat_kv attention, element by element.

Covers D in {64, 128}, G in {1, 2, 4, 8}, ragged and tiny valid lengths, an
allocated length that is not a multiple of the tile, persistent grids forced
small (so units split across CTAs and go through the in-kernel log-sum-exp
merge), one unit split over the whole grid, one workspace reused across
shapes, and the first workload at its full size.
"""
import math

import numpy as np
import pytest
import torch

import gqa_head_folding_gb300 as g
import oracle
import workloads
from _util import assert_attn_close

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(autouse=True)
def _reset_options():
    yield
    g.set_option(g.GQAQ_OPT_MAX_CTAS, 0)
    g.set_option(g.GQAQ_OPT_DENSE_EARLY_KV, 0)


def run_case(B, Hq, Hkv, D, Lmax, valid, seed, max_ctas=0):
    w = workloads.Workload(0, "case", batch=B, num_layers=1, num_q_heads=Hq, num_kv_heads=Hkv,
                           head_dim=D, max_len=Lmax)
    x = workloads.make_layer(w, 0, device="cpu", seed=seed)
    vl = torch.tensor(valid, dtype=torch.int32)
    g.set_option(g.GQAQ_OPT_MAX_CTAS, max_ctas)
    scale = 1.0 / math.sqrt(D)
    out = g.gqa_decode_attn(x["q"].to(DEV), x["k_cache"].to(DEV), x["v_cache"].to(DEV), vl.to(DEV), scale)
    torch.cuda.synchronize()
    assert g.device_status() == 0
    ref = oracle.attn_repeat_kv(x["q"].numpy(), x["k_cache"].numpy(), x["v_cache"].numpy(), valid, scale)
    return assert_attn_close(out, ref)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("G", [1, 2, 4, 8])
def test_dense_group_sizes(D, G):
    Hkv = 2 if G == 8 else 3
    run_case(2, Hkv * G, Hkv, D, 700, [700, 333], seed=D * 10 + G)


@pytest.mark.parametrize("max_ctas", [0, 1, 2, 3, 7, 50])
def test_dense_split_and_combine(max_ctas):
    # ragged lengths and a tail tile; small grids force units across CTAs
    run_case(3, 32, 8, 64, 1000, [1000, 129, 1], seed=11, max_ctas=max_ctas)


def test_dense_one_unit_split_over_the_whole_grid():
    # batch 1, one KV head: every CTA of the default grid holds a part of it
    run_case(1, 4, 1, 64, 16 * 2048, [16 * 2048 - 5], seed=21)
    run_case(1, 8, 1, 128, 16 * 1024, [16 * 1024], seed=22)


def test_dense_workspace_reused_across_shapes_and_grids():
    # one zero-filled workspace serves calls of different dims and grids; each
    # call leaves its arrival counters at zero for the next
    cases = [(4, 32, 8, 128, 2048, [2048, 700, 1, 1500], 0), (1, 8, 2, 64, 900, [899], 3),
             (3, 16, 8, 128, 512, [0, 300, 512], 7), (2, 32, 8, 64, 1200, [1200, 45], 0),
             (4, 32, 8, 128, 2048, [5, 2048, 2000, 128], 13)]
    need = max(g.workspace_bytes(g.make_dims(B, Hq, Hkv, D, Lmax)) for (B, Hq, Hkv, D, Lmax, _, _) in cases)
    ws = torch.zeros(need, dtype=torch.uint8, device=DEV)
    for i, (B, Hq, Hkv, D, Lmax, valid, max_ctas) in enumerate(cases):
        w = workloads.Workload(0, "case", batch=B, num_layers=1, num_q_heads=Hq, num_kv_heads=Hkv,
                               head_dim=D, max_len=Lmax)
        x = workloads.make_layer(w, 0, device="cpu", seed=100 + i)
        g.set_option(g.GQAQ_OPT_MAX_CTAS, max_ctas)
        scale = 1.0 / math.sqrt(D)
        out = g.gqa_decode_attn(x["q"].to(DEV), x["k_cache"].to(DEV), x["v_cache"].to(DEV),
                                torch.tensor(valid, dtype=torch.int32, device=DEV), scale, workspace=ws)
        torch.cuda.synchronize()
        flags = g.device_status()
        assert flags in (0, g.GQAQ_DEV_BAD_LEN) and (flags == 0) == (min(valid) >= 1)
        assert int(ws[:256].count_nonzero()) == 0
        keep = [b for b in range(B) if valid[b] >= 1]
        assert all(bool((out[b] == 0).all()) for b in range(B) if valid[b] < 1)   # no valid token -> zeros
        ref = oracle.attn_repeat_kv(x["q"].numpy()[keep], x["k_cache"].numpy()[keep], x["v_cache"].numpy()[keep],
                                    [valid[b] for b in keep], scale)
        assert_attn_close(out[keep], ref)


@pytest.mark.parametrize("valid", [[1], [15], [16], [17], [127], [128], [129], [300]])
def test_dense_edge_lengths(valid):
    run_case(1, 8, 2, 128, 300, valid, seed=valid[0])


def test_dense_first_workload_full_size():
    # 32 query heads on 8 KV heads, D=64, 4096 valid tokens, batch 1
    w = workloads.WORKLOADS[1]
    x = workloads.make_layer(w, 0, device="cpu")
    scale = 1.0 / math.sqrt(w.head_dim)
    out = g.gqa_decode_attn(x["q"].to(DEV), x["k_cache"].to(DEV), x["v_cache"].to(DEV),
                            x["valid_len"].to(DEV), scale)
    ref = oracle.attn_repeat_kv(x["q"].numpy(), x["k_cache"].numpy(), x["v_cache"].numpy(),
                                x["valid_len"].numpy(), scale)
    assert_attn_close(out, ref)


def test_dense_second_workload_two_layers():
    # EXAONE-shaped caches, allocated 4096, valid lengths uniform in [1024, 4096]
    w = workloads.WORKLOADS[2].with_(batch=3)
    scale = 1.0 / math.sqrt(w.head_dim)
    for layer in range(2):
        x = workloads.make_layer(w, layer, device="cpu")
        out = g.gqa_decode_attn(x["q"].to(DEV), x["k_cache"].to(DEV), x["v_cache"].to(DEV),
                                x["valid_len"].to(DEV), scale)
        ref = oracle.attn_repeat_kv(x["q"].numpy(), x["k_cache"].numpy(), x["v_cache"].numpy(),
                                    x["valid_len"].numpy(), scale)
        assert_attn_close(out, ref, f"layer {layer}")


def test_dense_invalid_lengths_are_clamped_and_flagged():
    w = workloads.Workload(0, "case", batch=3, num_layers=1, num_q_heads=8, num_kv_heads=2,
                           head_dim=64, max_len=64)
    x = workloads.make_layer(w, 0, device="cpu", seed=5)
    vl = torch.tensor([0, 64, 500], dtype=torch.int32)
    g.device_status(reset=True)
    out = g.gqa_decode_attn(x["q"].to(DEV), x["k_cache"].to(DEV), x["v_cache"].to(DEV), vl.to(DEV), 0.125)
    flags = g.device_status(reset=True)
    assert flags & g.GQAQ_DEV_BAD_LEN
    o = out.float().cpu()
    assert torch.all(o[0] == 0)                                  # no valid token -> zeros
    ref = oracle.attn_repeat_kv(x["q"].numpy()[1:], x["k_cache"].numpy()[1:], x["v_cache"].numpy()[1:],
                                [64, 64], 0.125)                 # 500 clamps to Lmax = 64
    assert_attn_close(out[1:], ref)


def test_dense_uninitialised_tail_is_never_used():
    # rows past valid_len hold NaN; the output must not see them
    w = workloads.Workload(0, "case", batch=2, num_layers=1, num_q_heads=16, num_kv_heads=4,
                           head_dim=128, max_len=256)
    x = workloads.make_layer(w, 0, device="cpu", seed=9)
    k, v = x["k_cache"].clone(), x["v_cache"].clone()
    valid = [100, 37]
    for b, n in enumerate(valid):
        k[b, :, n:] = float("nan")
        v[b, :, n:] = float("nan")
    out = g.gqa_decode_attn(x["q"].to(DEV), k.to(DEV), v.to(DEV), torch.tensor(valid, dtype=torch.int32).to(DEV),
                            0.1)
    ref = oracle.attn_repeat_kv(x["q"].numpy(), k.numpy(), v.numpy(), valid, 0.1)
    assert_attn_close(out, ref)


def test_dense_repeatable_and_graph_capturable():
    w = workloads.WORKLOADS[2].with_(batch=4)
    x = workloads.make_layer(w, 0, device=DEV)
    args = (x["q"], x["k_cache"], x["v_cache"], x["valid_len"])
    d = g.dims_of(x["q"], x["k_cache"])
    ws = g.alloc_workspace(d, DEV)
    out = torch.empty_like(x["q"])
    g.gqa_decode_attn(*args, 0.125, out=out, workspace=ws)
    first = out.clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            g.gqa_decode_attn(*args, 0.125, out=out, workspace=ws)
    torch.cuda.current_stream().wait_stream(s)
    out.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, first)


@pytest.mark.parametrize("D,max_ctas", [(64, 0), (64, 3), (128, 0), (128, 5)])
def test_dense_early_kv_decode_loop(D, max_ctas):
    """GQAQ_OPT_DENSE_EARLY_KV: two layers, three decode steps of append then
    dense attention, every launch right behind the previous one (programmatic
    launch), as a decode loop does. Lengths cross tile boundaries (the appended
    row opens a new tile, or is a sequence's only tile); forced small grids cut
    units across CTAs. Each output is checked against the oracle replaying the
    appends."""
    g.set_option(g.GQAQ_OPT_DENSE_EARLY_KV, 1)
    g.set_option(g.GQAQ_OPT_MAX_CTAS, max_ctas)
    B, Hkv, G, Lmax, nl, nsteps, S = 3, 2, 4, 700, 2, 3, 16
    w = workloads.Workload(0, "case", batch=B, num_layers=nl, num_q_heads=G * Hkv, num_kv_heads=Hkv,
                           head_dim=D, max_len=Lmax)
    xs = [workloads.make_layer(w, l, device="cpu", seed=70 + D + l) for l in range(nl)]
    gen = torch.Generator().manual_seed(80 + D + max_ctas)
    knew = torch.randn(nsteps, nl, B, Hkv, D, generator=gen).to(torch.float16)
    vnew = torch.randn(nsteps, nl, B, Hkv, D, generator=gen).to(torch.float16)
    vls = [np.array([127, 300, 511]) + s for s in range(nsteps)]
    vld = [torch.tensor(v, dtype=torch.int32, device=DEV) for v in vls]       # made before the loop:
    posd = [torch.tensor(v - 1, dtype=torch.int32, device=DEV) for v in vls]  # no kernel writes them in it
    kd = [x["k_cache"].to(DEV) for x in xs]
    vd = [x["v_cache"].to(DEV) for x in xs]
    qd = [x["q"].to(DEV) for x in xs]
    metas = [g.new_meta(B, Hkv, Lmax, D, DEV) for _ in range(nl)]
    kn, vn = knew.to(DEV), vnew.to(DEV)
    outs = torch.empty(nsteps, nl, B, G * Hkv, D, dtype=torch.float16, device=DEV)
    scale = 1.0 / math.sqrt(D)
    torch.cuda.synchronize()
    for s in range(nsteps):
        for l in range(nl):
            g.quest_append_kv(kd[l], vd[l], metas[l], kn[s, l], vn[s, l], posd[s], S)
            g.gqa_decode_attn(qd[l], kd[l], vd[l], vld[s], scale, out=outs[s, l])
    torch.cuda.synchronize()
    assert g.device_status() == 0
    for l in range(nl):
        kc = xs[l]["k_cache"].numpy().copy(); vc = xs[l]["v_cache"].numpy().copy()
        for s in range(nsteps):
            for b in range(B):
                kc[b, :, vls[s][b] - 1] = knew[s, l, b].numpy(); vc[b, :, vls[s][b] - 1] = vnew[s, l, b].numpy()
            ref = oracle.attn_repeat_kv(xs[l]["q"].numpy(), kc, vc, list(vls[s]), scale)
            assert_attn_close(outs[s, l], ref, f"step {s} layer {l}")
