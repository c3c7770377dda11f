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


def nibble_rows(D, shift=0):
    """One code row whose channel c holds nibble (c + shift) mod 16, i.e. every
    level -8 .. 7 (nibble - 8), channel 2i in the low nibble of byte i."""
    nib = (np.arange(D) + shift) % 16
    return (nib[0::2] | (nib[1::2] << 4)).astype(np.uint8), nib.astype(np.float64) - 8.0


@pytest.mark.parametrize("D", [64, 128])
def test_every_level_decodes_exactly(D):
    """Each of the 16 nibble values decodes to its level exactly, in V and in K.

    V: with one valid token the output is that token's value row, level * scale;
    the scale is a power of two, so every output is exact in fp16 and must
    equal it bit for bit. K: query head (b, g) is one-hot on channel
    c = b * 8 + g, so its score is a * level(k0[c]) * k_scale against a zero
    second key, and the output over one-hot V rows is (sigmoid, 1 - sigmoid)
    of it: adjacent levels move it by far more than the fp16 tolerance."""
    G = 8
    B = D // G                                    # one query head per channel
    Lmax = 4
    # V decode: one valid token per sequence, every level in every row
    kc = np.zeros((B, 1, Lmax, D // 2), np.uint8)
    vc = np.zeros((B, 1, Lmax, D // 2), np.uint8)
    vlev = np.zeros((B, D))
    for b in range(B):
        vc[b, 0, 0], vlev[b] = nibble_rows(D, shift=b)
    ks = np.full((B, 1, Lmax), 0.25, np.float32)
    vs = np.full((B, 1, Lmax), 0.125, np.float32)
    q = torch.randn(B, G, D, generator=torch.Generator().manual_seed(3)).to(torch.float16)
    vl = torch.ones(B, dtype=torch.int32, device=DEV)
    out = g.gqa_decode_attn_int4(q.to(DEV), dev(kc), dev(ks), dev(vc), dev(vs), vl, 0.125)
    torch.cuda.synchronize()
    want = torch.from_numpy(np.repeat((vlev * 0.125)[:, None, :], G, axis=1)).to(torch.float16)
    assert torch.equal(out.cpu(), want), "V levels decode wrongly"

    # K decode: token 0's key holds every level, token 1's key is all zero
    # (nibble 8); V rows one-hot on channels 0 and 1 with level 1, scale 1
    k0, klev = nibble_rows(D)
    kc = np.zeros((B, 1, Lmax, D // 2), np.uint8)
    kc[:, 0, 0] = k0
    kc[:, 0, 1] = 0x88
    vc = np.full((B, 1, Lmax, D // 2), 0x88, np.uint8)
    vc[:, 0, 0, 0] = 0x89                         # channel 0 = level 1
    vc[:, 0, 1, 0] = 0x98                         # channel 1 = level 1
    vs = np.ones((B, 1, Lmax), np.float32)
    a = 4.0                                       # score = a * level * 0.25 * 0.5 = level / 2
    qn = np.zeros((B, G, D), np.float16)
    for b in range(B):
        for gg in range(G):
            qn[b, gg, b * G + gg] = a
    vl = torch.full((B,), 2, dtype=torch.int32, device=DEV)
    out = g.gqa_decode_attn_int4(dev(qn.reshape(B, G, D)), dev(kc), dev(ks), dev(vc), dev(vs), vl, 0.5)
    torch.cuda.synchronize()
    got = out.float().cpu().numpy().reshape(B * G, D)
    s = klev / 2.0                                # channel c's score against the zero key
    p0 = 1.0 / (1.0 + np.exp(-s))
    assert np.abs(got[:, 0] - p0).max() <= 2e-3 and np.abs(got[:, 1] - (1.0 - p0)).max() <= 2e-3, \
        "K levels decode wrongly"
    ref = oracle.attn_int4(qn.reshape(B, G, D), kc, ks, vc, vs, [2] * B, 0.5)
    assert_attn_close(out, ref)
