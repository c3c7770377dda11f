"""GPU parity of the 4-bit (INT4) KV-cache variant against the fp64 oracle.

kv_append_int4 must write exactly the oracle's levels and scales (per-row
scale = amax / 7, levels clamp(rne(x / scale), -7, 7), fp32 arithmetic) and
leave every other row alone. gqa_decode_attn_int4 must match the oracle's
attention over the dequantized cache (level * scale) within the fp16-output
tolerance, over D in {64, 128}, G in {1, 2, 4, 8}, ragged lengths, forced
small grids (split units merged in-kernel), NaN scales and random codes in
rows past the valid length, and two dense workloads at full size on sampled
heads.
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


def int4_case(B, Hq, Hkv, D, Lmax, seed):
    w = workloads.Workload(0, "case", batch=B, num_layers=1, num_q_heads=Hq, num_kv_heads=Hkv,
                           head_dim=D, max_len=Lmax, append=True)
    x = workloads.make_layer(w, 0, device="cpu", seed=seed)
    kc, ks = oracle.quantize_int4(x["k_cache"].numpy())
    vc, vs = oracle.quantize_int4(x["v_cache"].numpy())
    return x, kc, ks, vc, vs


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def run_attn(B, Hq, Hkv, D, Lmax, valid, seed, max_ctas=0, garbage_tail=False):
    x, kc, ks, vc, vs = int4_case(B, Hq, Hkv, D, Lmax, seed)
    if garbage_tail:
        rng = np.random.default_rng(seed)
        for b, L in enumerate(valid):
            kc[b, :, L:] = rng.integers(0, 256, size=kc[b, :, L:].shape, dtype=np.uint8)
            vc[b, :, L:] = rng.integers(0, 256, size=vc[b, :, L:].shape, dtype=np.uint8)
            ks[b, :, L:] = np.nan
            vs[b, :, L:] = np.inf
    g.set_option(g.GQAQ_OPT_MAX_CTAS, max_ctas)
    scale = 1.0 / math.sqrt(D)
    vl = torch.tensor(valid, dtype=torch.int32, device=DEV)
    out = g.gqa_decode_attn_int4(x["q"].to(DEV), dev(kc), dev(ks), dev(vc), dev(vs), vl, scale)
    torch.cuda.synchronize()
    assert g.device_status() == 0
    ref = oracle.attn_int4(x["q"].numpy(), kc, ks, vc, vs, valid, scale)
    return assert_attn_close(out, ref)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("G", [1, 2, 4, 8])
def test_int4_attn_group_sizes(D, G):
    Hkv = 2 if G == 8 else 3
    run_attn(2, Hkv * G, Hkv, D, 700, [700, 333], seed=D * 10 + G)


@pytest.mark.parametrize("valid", [[1, 2], [63, 64], [65, 129], [1000, 7]])
def test_int4_attn_ragged_lengths(valid):
    run_attn(2, 8, 2, 128, 1000, valid, seed=sum(valid))


@pytest.mark.parametrize("max_ctas", [1, 3, 7])
def test_int4_attn_split_merge(max_ctas):
    run_attn(2, 16, 2, 64, 4100, [4100, 2999], seed=max_ctas, max_ctas=max_ctas)


@pytest.mark.parametrize("D", [64, 128])
def test_int4_rows_past_valid_length_are_never_used(D):
    run_attn(2, 8, 2, D, 520, [517, 130], seed=D + 1, garbage_tail=True)


@pytest.mark.parametrize("wid", [2, 3])
def test_int4_attn_full_size_sampled_heads(wid):
    """A dense layer of the 30-layer 4K GQA workload (B=32, ragged lengths)
    and of the 32K Llama-2-7B workload at full size. Any codes with positive
    scales are a valid cache: they are drawn at random on the device."""
    w = workloads.WORKLOADS[wid]
    B, Hkv, L, D = w.batch, w.num_kv_heads, w.max_len, w.head_dim
    gen = torch.Generator(device=DEV).manual_seed(50 + wid)
    q = torch.randn(B, w.num_q_heads, D, generator=gen, device=DEV).to(torch.float16)
    kc = torch.randint(0, 256, (B, Hkv, L, D // 2), generator=gen, device=DEV, dtype=torch.uint8)
    vc = torch.randint(0, 256, (B, Hkv, L, D // 2), generator=gen, device=DEV, dtype=torch.uint8)
    ks = torch.rand(B, Hkv, L, generator=gen, device=DEV) * 0.05 + 0.01
    vs = torch.rand(B, Hkv, L, generator=gen, device=DEV) * 0.2 + 0.05
    vl = workloads.valid_lengths(w, 0).to(DEV)
    scale = 1.0 / math.sqrt(D)
    out = g.gqa_decode_attn_int4(q, kc, ks, vc, vs, vl, scale)
    torch.cuda.synchronize()
    assert g.device_status() == 0
    rng = np.random.default_rng(wid)
    vln = vl.cpu().numpy()
    for _ in range(3):
        b, h = int(rng.integers(B)), int(rng.integers(w.num_q_heads))
        kv = h // w.group
        ref = oracle.attn_int4(q[b:b + 1, h:h + 1].cpu().numpy(), kc[b:b + 1, kv:kv + 1].cpu().numpy(),
                               ks[b:b + 1, kv:kv + 1].cpu().numpy(), vc[b:b + 1, kv:kv + 1].cpu().numpy(),
                               vs[b:b + 1, kv:kv + 1].cpu().numpy(), vln[b:b + 1], scale)
        assert_attn_close(out[b:b + 1, h:h + 1], ref, f"b={b} h={h}")


@pytest.mark.parametrize("D", [64, 128])
def test_int4_append_bit_exact(D):
    B, Hkv, Lmax = 3, 4, 52
    rng = np.random.default_rng(D)
    kc = rng.integers(0, 256, size=(B, Hkv, Lmax, D // 2), dtype=np.uint8)
    vc = rng.integers(0, 256, size=(B, Hkv, Lmax, D // 2), dtype=np.uint8)
    ks = rng.uniform(0, 1, size=(B, Hkv, Lmax)).astype(np.float32)
    vs = rng.uniform(0, 1, size=(B, Hkv, Lmax)).astype(np.float32)
    k_new = (rng.standard_normal((B, Hkv, D)) * 30).astype(np.float16)
    v_new = (rng.standard_normal((B, Hkv, D)) * 0.01).astype(np.float16)
    k_new[0, 0, :8] = [7, 2.5, -2.5, 3.5, 0.5, -0.5, 1.5, -7]   # scale 1: ties to even levels
    k_new[0, 0, 8:] = 0
    v_new[1, 2] = 0                                             # a zero row
    pos = np.array([0, 31, Lmax - 1], dtype=np.int32)
    kd, vd, ksd, vsd = dev(kc), dev(vc), dev(ks), dev(vs)
    g.kv_append_int4(kd, ksd, vd, vsd, dev(k_new), dev(v_new), dev(pos))
    torch.cuda.synchronize()
    assert g.device_status() == 0
    kref, vref, ksref, vsref = kc.copy(), vc.copy(), ks.copy(), vs.copy()
    for b in range(B):
        kref[b, :, pos[b]], ksref[b, :, pos[b]] = oracle.quantize_int4(k_new[b])
        vref[b, :, pos[b]], vsref[b, :, pos[b]] = oracle.quantize_int4(v_new[b])
    assert np.array_equal(kd.cpu().numpy(), kref) and np.array_equal(vd.cpu().numpy(), vref)
    assert np.array_equal(ksd.cpu().numpy(), ksref) and np.array_equal(vsd.cpu().numpy(), vsref)
    assert ksref[0, 0, 0] == 1.0 and vsref[1, 2, pos[1]] == 0.0


def test_int4_append_bad_position_flags_and_skips():
    B, Hkv, D, Lmax = 2, 2, 64, 16
    kd = torch.zeros(B, Hkv, Lmax, D // 2, dtype=torch.uint8, device=DEV)
    vd = torch.zeros_like(kd)
    ks = torch.zeros(B, Hkv, Lmax, device=DEV)
    vs = torch.zeros_like(ks)
    new = torch.ones(B, Hkv, D, dtype=torch.float16, device=DEV)
    g.kv_append_int4(kd, ks, vd, vs, new, new, torch.tensor([3, Lmax], dtype=torch.int32, device=DEV))
    torch.cuda.synchronize()
    assert g.device_status() == g.GQAQ_DEV_BAD_POS
    assert int(kd[0, :, 3].ne(0xFF).sum()) == 0                 # ones: level 7 everywhere (0xF nibbles)
    assert int(kd[1].count_nonzero()) == 0 and int(ks[1].count_nonzero()) == 0


@pytest.mark.parametrize("early", [0, 1])
def test_int4_append_then_attend_matches_oracle(early):
    g.set_option(g.GQAQ_OPT_DENSE_EARLY_KV, early)  # the append is the previous kernel: early reads allowed
    B, Hkv, G, D, Lmax = 2, 2, 4, 128, 300
    x, kc, ks, vc, vs = int4_case(B, Hkv * G, Hkv, D, Lmax, seed=21)
    vl = np.array([Lmax, 150])
    kd, vd, ksd, vsd = dev(kc), dev(vc), dev(ks), dev(vs)
    vld = torch.tensor(vl, dtype=torch.int32, device=DEV)
    g.kv_append_int4(kd, ksd, vd, vsd, x["k_new"].to(DEV), x["v_new"].to(DEV), vld - 1)
    out = g.gqa_decode_attn_int4(x["q"].to(DEV), kd, ksd, vd, vsd, vld, 1.0 / math.sqrt(D))
    torch.cuda.synchronize()
    assert g.device_status() == 0
    for b in range(B):
        kc[b, :, vl[b] - 1], ks[b, :, vl[b] - 1] = oracle.quantize_int4(x["k_new"][b].numpy())
        vc[b, :, vl[b] - 1], vs[b, :, vl[b] - 1] = oracle.quantize_int4(x["v_new"][b].numpy())
    assert np.array_equal(kd.cpu().numpy(), kc) and np.array_equal(ksd.cpu().numpy(), ks)
    assert_attn_close(out, oracle.attn_int4(x["q"].numpy(), kc, ks, vc, vs, vl, 1.0 / math.sqrt(D)))
