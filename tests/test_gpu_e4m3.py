"""GPU parity of the 8-bit (E4M3) KV-cache variant against the fp64 oracle.

kv_append_e4m3 must write exactly the oracle's codes (nearest E4M3 value of
fp32(x) * inv_scale, ties to even, saturating at 448) and leave every other
row alone. gqa_decode_attn_e4m3 must match the oracle's attention over the
decoded cache (code value * scale) within the fp16-output tolerance, over
D in {64, 128}, G in {1, 2, 4, 8}, ragged lengths, forced small grids (split
units merged in-kernel) and two dense workloads at full size on sampled
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


def e4m3_case(B, Hq, Hkv, D, Lmax, seed):
    """A workload layer with its caches quantized by the oracle (per-tensor
    scales amax / 448)."""
    w = workloads.Workload(0, "case", batch=B, num_layers=1, num_q_heads=Hq, num_kv_heads=Hkv,
                           head_dim=D, max_len=Lmax, append=True)
    x = workloads.make_layer(w, 0, device="cpu", seed=seed)
    k, v = x["k_cache"].numpy(), x["v_cache"].numpy()
    ks = float(np.abs(k.astype(np.float32)).max()) / 448.0
    vs = float(np.abs(v.astype(np.float32)).max()) / 448.0
    kc = oracle.quantize_e4m3(k, np.float32(1.0 / ks))
    vc = oracle.quantize_e4m3(v, np.float32(1.0 / vs))
    return x, kc, vc, ks, vs


def run_attn(B, Hq, Hkv, D, Lmax, valid, seed, max_ctas=0):
    x, kc, vc, ks, vs = e4m3_case(B, Hq, Hkv, D, Lmax, seed)
    g.set_option(g.GQAQ_OPT_MAX_CTAS, max_ctas)
    scale = 1.0 / math.sqrt(D)
    vl = torch.tensor(valid, dtype=torch.int32, device=DEV)
    out = g.gqa_decode_attn_e4m3(x["q"].to(DEV), torch.from_numpy(kc).to(DEV), torch.from_numpy(vc).to(DEV),
                                 ks, vs, vl, scale)
    torch.cuda.synchronize()
    assert g.device_status() == 0
    ref = oracle.attn_e4m3(x["q"].numpy(), kc, vc, ks, vs, valid, scale)
    return assert_attn_close(out, ref)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("G", [1, 2, 4, 8])
def test_e4m3_attn_group_sizes(D, G):
    Hkv = 2 if G == 8 else 3
    run_attn(2, Hkv * G, Hkv, D, 700, [700, 333], seed=D * 10 + G)


@pytest.mark.parametrize("valid", [[1, 2], [63, 64], [65, 129], [1000, 7]])
def test_e4m3_attn_ragged_lengths(valid):
    run_attn(2, 8, 2, 128, 1000, valid, seed=sum(valid))


@pytest.mark.parametrize("max_ctas", [1, 3, 7])
def test_e4m3_attn_split_merge(max_ctas):
    run_attn(2, 16, 2, 64, 4100, [4100, 2999], seed=max_ctas, max_ctas=max_ctas)


@pytest.mark.parametrize("wid", [2, 3])
def test_e4m3_attn_full_size_sampled_heads(wid):
    """A dense layer of the 30-layer 4K GQA workload (B=32, ragged lengths)
    and of the 32K Llama-2-7B workload at full size; the oracle checks a
    sample of (sequence, query head) pairs. The caches are quantized on the
    device by torch's own float8 conversion (inputs only)."""
    w = workloads.WORKLOADS[wid]
    x = workloads.make_layer(w, 0, device=DEV, seed=5)
    ks = float(x["k_cache"].abs().max()) / 448.0
    vs = float(x["v_cache"].abs().max()) / 448.0
    kc = (x["k_cache"].float() * (1.0 / ks)).to(torch.float8_e4m3fn).view(torch.uint8)
    vc = (x["v_cache"].float() * (1.0 / vs)).to(torch.float8_e4m3fn).view(torch.uint8)
    vl = x["valid_len"].to(DEV)
    scale = 1.0 / math.sqrt(w.head_dim)
    out = g.gqa_decode_attn_e4m3(x["q"], kc, vc, ks, vs, vl, scale)
    torch.cuda.synchronize()
    assert g.device_status() == 0
    rng = np.random.default_rng(wid)
    vln = vl.cpu().numpy()
    G = w.group
    for _ in range(3):
        b, h = int(rng.integers(w.batch)), int(rng.integers(w.num_q_heads))
        kv = h // G
        ref = oracle.attn_e4m3(x["q"][b:b + 1, h:h + 1].cpu().numpy(), kc[b:b + 1, kv:kv + 1].cpu().numpy(),
                               vc[b:b + 1, kv:kv + 1].cpu().numpy(), ks, vs, vln[b:b + 1], scale)
        assert_attn_close(out[b:b + 1, h:h + 1], ref, f"b={b} h={h}")


@pytest.mark.parametrize("D", [64, 128])
def test_e4m3_append_codes_bit_exact(D):
    B, Hkv, Lmax = 3, 4, 50
    rng = np.random.default_rng(D)
    kc = rng.integers(0, 256, size=(B, Hkv, Lmax, D), dtype=np.uint8)
    vc = rng.integers(0, 256, size=(B, Hkv, Lmax, D), dtype=np.uint8)
    k_new = (rng.standard_normal((B, Hkv, D)) * 30).astype(np.float16)
    v_new = (rng.standard_normal((B, Hkv, D)) * 3).astype(np.float16)
    # exact ties, saturation, zeros and subnormals in the first channels
    k_new[0, 0, :8] = [1.0625, 1.1875, 470, -1000, 2.0 ** -10, 0.0, -0.0, 448]
    pos = np.array([0, 31, Lmax - 1], dtype=np.int32)
    k_inv, v_inv = np.float32(1.0), np.float32(37.5)
    kd, vd = torch.from_numpy(kc).to(DEV), torch.from_numpy(vc).to(DEV)
    g.kv_append_e4m3(kd, vd, torch.from_numpy(k_new).to(DEV), torch.from_numpy(v_new).to(DEV),
                     torch.from_numpy(pos).to(DEV), float(k_inv), float(v_inv))
    torch.cuda.synchronize()
    assert g.device_status() == 0
    kref, vref = kc.copy(), vc.copy()
    for b in range(B):
        kref[b, :, pos[b]] = oracle.quantize_e4m3(k_new[b], k_inv)
        vref[b, :, pos[b]] = oracle.quantize_e4m3(v_new[b], v_inv)
    assert np.array_equal(kd.cpu().numpy(), kref)
    assert np.array_equal(vd.cpu().numpy(), vref)
    assert list(kref[0, 0, pos[0], :8]) == [56, 58, 126, 254, 0, 0, 128, 126]


def test_e4m3_append_bad_position_flags_and_skips():
    B, Hkv, D, Lmax = 2, 2, 64, 16
    kd = torch.zeros(B, Hkv, Lmax, D, dtype=torch.uint8, device=DEV)
    vd = torch.zeros_like(kd)
    new = torch.ones(B, Hkv, D, dtype=torch.float16, device=DEV)
    g.kv_append_e4m3(kd, vd, new, new, torch.tensor([3, Lmax], dtype=torch.int32, device=DEV), 1.0, 1.0)
    torch.cuda.synchronize()
    assert g.device_status() == g.GQAQ_DEV_BAD_POS
    assert int(kd[0, :, 3].ne(56).sum()) == 0 and int(kd[1].count_nonzero()) == 0


@pytest.mark.parametrize("early", [0, 1])
def test_e4m3_append_then_attend_matches_oracle(early):
    """A decode step over the 8-bit cache: append the token, attend over it."""
    g.set_option(g.GQAQ_OPT_DENSE_EARLY_KV, early)  # the append is the previous kernel: early reads allowed
    B, Hkv, G, D, Lmax = 2, 2, 4, 128, 300
    x, kc, vc, ks, vs = e4m3_case(B, Hkv * G, Hkv, D, Lmax, seed=21)
    vl = np.array([Lmax, 150])
    kd, vd = torch.from_numpy(kc).to(DEV), torch.from_numpy(vc).to(DEV)
    k_inv, v_inv = np.float32(1.0 / ks), np.float32(1.0 / vs)
    vld = torch.tensor(vl, dtype=torch.int32, device=DEV)
    g.kv_append_e4m3(kd, vd, x["k_new"].to(DEV), x["v_new"].to(DEV), vld - 1, float(k_inv), float(v_inv))
    out = g.gqa_decode_attn_e4m3(x["q"].to(DEV), kd, vd, ks, vs, vld, 1.0 / math.sqrt(D))
    torch.cuda.synchronize()
    assert g.device_status() == 0
    for b in range(B):
        kc[b, :, vl[b] - 1] = oracle.quantize_e4m3(x["k_new"][b].numpy(), k_inv)
        vc[b, :, vl[b] - 1] = oracle.quantize_e4m3(x["v_new"][b].numpy(), v_inv)
    assert np.array_equal(kd.cpu().numpy(), kc) and np.array_equal(vd.cpu().numpy(), vc)
    assert_attn_close(out, oracle.attn_e4m3(x["q"].numpy(), kc, vc, ks, vs, vl, 1.0 / math.sqrt(D)))
