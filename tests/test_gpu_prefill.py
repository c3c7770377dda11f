"""GPU parity of gqa_prefill_attn (causal chunk attention with the group axis
merged into the row axis) against the fp64 oracle, element by element.

Every case runs on both kernels (tcgen05 / tensor memory, the default, and
warp-level MMA). Covers D in {64, 128}, G in {1, 2, 4, 8}, chunk lengths from 1 to past one
128-row block (so blocks wrap across query heads), chunks starting at zero
and deep in the cache, per-sequence starts, forced context splits (including
more splits than tiles: empty slices), NaN rows past the chunk, a bad start,
the stall/timeout path, workspace reuse, and a 4K-context chunk at the
Llama-2-7B-shaped size on sampled rows.
"""
import math

import numpy as np
import pytest
import torch

import gqa_head_folding_gb300 as g
import oracle
from _util import assert_attn_close

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(autouse=True, params=["tcgen05", "warp_mma"])
def kernel(request):
    """Every case runs on both prefill kernels: tensor memory (default) and warp-level MMA."""
    g.set_option(g.GQAQ_OPT_PREFILL_KERNEL, 1 if request.param == "tcgen05" else 2)
    yield request.param
    g.set_option(g.GQAQ_OPT_PREFILL_KERNEL, 0)


@pytest.fixture(autouse=True)
def _reset_options():
    yield
    g.set_option(g.GQAQ_OPT_PREFILL_SPLITS, 0)
    g.set_option(g.GQAQ_OPT_TEST_STALL, 0)
    g.set_option(g.GQAQ_OPT_WAIT_TIMEOUT_NS, 2_000_000_000)


def make_case(B, Hkv, G, D, Lmax, q_len, seed):
    gen = torch.Generator().manual_seed(seed)
    q = torch.randn(B, Hkv * G, q_len, D, generator=gen).to(torch.float16)
    k = torch.randn(B, Hkv, Lmax, D, generator=gen).to(torch.float16)
    v = torch.randn(B, Hkv, Lmax, D, generator=gen).to(torch.float16)
    return q, k, v


def run(B, Hkv, G, D, Lmax, q_len, starts, seed, splits=0, nan_tail=False):
    q, k, v = make_case(B, Hkv, G, D, Lmax, q_len, seed)
    if nan_tail:
        for b, s in enumerate(starts):
            k[b, :, s + q_len:] = float("nan")
            v[b, :, s + q_len:] = float("nan")
    g.set_option(g.GQAQ_OPT_PREFILL_SPLITS, splits)
    scale = 1.0 / math.sqrt(D)
    st = torch.tensor(starts, dtype=torch.int32, device=DEV)
    out = g.gqa_prefill_attn(q.to(DEV), k.to(DEV), v.to(DEV), st, scale)
    torch.cuda.synchronize()
    assert g.device_status() == 0
    ref = oracle.prefill_attn(q.numpy(), k.numpy(), v.numpy(), starts, scale)
    return assert_attn_close(out, ref)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("G", [1, 2, 4, 8])
def test_prefill_group_sizes(D, G):
    run(2, 2, G, D, 300, 37, [263, 100], seed=D + G)


@pytest.mark.parametrize("q_len", [1, 2, 16, 33, 64, 100, 130])
def test_prefill_chunk_lengths(q_len):
    # G * q_len from 4 to 520 rows: 1 to 5 row blocks, most of them wrapping
    run(2, 2, 4, 64, 400, q_len, [400 - q_len, max(0, 150 - q_len)], seed=q_len)


def test_prefill_from_zero_full_causal():
    run(1, 3, 2, 128, 256, 256, [0], seed=3)


@pytest.mark.parametrize("splits", [1, 2, 3, 7, 32])
def test_prefill_forced_splits(splits):
    # 32 splits of at most 10 tiles: most slices are empty
    run(2, 2, 4, 128, 640, 40, [600, 321], seed=splits, splits=splits)


def test_prefill_nan_rows_past_chunk_are_never_read():
    run(2, 2, 4, 64, 300, 20, [200, 37], seed=9, nan_tail=True)


def test_prefill_one_token_matches_decode():
    B, Hkv, G, D, Lmax = 3, 2, 4, 128, 333
    q, k, v = make_case(B, Hkv, G, D, Lmax, 1, seed=11)
    starts = [332, 100, 0]
    st = torch.tensor(starts, dtype=torch.int32, device=DEV)
    kd, vd = k.to(DEV), v.to(DEV)
    out_p = g.gqa_prefill_attn(q.to(DEV), kd, vd, st, 0.1)
    out_d = g.gqa_decode_attn(q[:, :, 0].contiguous().to(DEV), kd, vd, st + 1, 0.1)
    torch.cuda.synchronize()
    ref = oracle.attn_repeat_kv(q[:, :, 0].numpy(), k.numpy(), v.numpy(), [s + 1 for s in starts], 0.1)
    assert_attn_close(out_p[:, :, 0], ref)
    assert_attn_close(out_d, ref)


def test_prefill_bad_start_flags_and_zeroes():
    B, Hkv, G, D, Lmax, q_len = 2, 2, 2, 64, 100, 10
    q, k, v = make_case(B, Hkv, G, D, Lmax, q_len, seed=12)
    st = torch.tensor([95, 20], dtype=torch.int32, device=DEV)  # 95 + 10 > Lmax
    out = g.gqa_prefill_attn(q.to(DEV), k.to(DEV), v.to(DEV), st, 0.125)
    torch.cuda.synchronize()
    assert g.device_status() == g.GQAQ_DEV_BAD_POS
    assert int(out[0].count_nonzero()) == 0
    ref = oracle.prefill_attn(q[1:].numpy(), k[1:].numpy(), v[1:].numpy(), [20], 0.125)
    assert_attn_close(out[1:], ref)


def test_prefill_workspace_reused_and_left_zero():
    cases = [(2, 2, 4, 64, 300, 37, [263, 100]), (1, 4, 8, 128, 500, 20, [480]), (3, 1, 1, 64, 90, 90, [0, 0, 0])]
    dims = [g.make_dims(B, Hkv * G, Hkv, D, L) for B, Hkv, G, D, L, _, _ in cases]
    for splits in (0, 5):
        g.set_option(g.GQAQ_OPT_PREFILL_SPLITS, splits)
        nbytes = max(g.prefill_workspace_bytes(d, c[5]) for d, c in zip(dims, cases))
        ws = torch.zeros(nbytes, dtype=torch.uint8, device=DEV)
        for rep in range(2):
            for i, (B, Hkv, G, D, L, ql, starts) in enumerate(cases):
                q, k, v = make_case(B, Hkv, G, D, L, ql, seed=20 + i)
                st = torch.tensor(starts, dtype=torch.int32, device=DEV)
                out = g.gqa_prefill_attn(q.to(DEV), k.to(DEV), v.to(DEV), st, 0.2, workspace=ws)
                torch.cuda.synchronize()
                assert g.device_status() == 0
                assert_attn_close(out, oracle.prefill_attn(q.numpy(), k.numpy(), v.numpy(), starts, 0.2))
                items = B * Hkv * ((G * ql + 127) // 128)
                assert int(ws[:items * 4].count_nonzero()) == 0


def test_prefill_stall_times_out_and_recovers():
    B, Hkv, G, D, Lmax, q_len = 1, 2, 4, 64, 512, 32
    q, k, v = make_case(B, Hkv, G, D, Lmax, q_len, seed=30)
    d = g.make_dims(B, Hkv * G, Hkv, D, Lmax)
    g.set_option(g.GQAQ_OPT_PREFILL_SPLITS, 4)
    ws = torch.zeros(g.prefill_workspace_bytes(d, q_len), dtype=torch.uint8, device=DEV)
    st = torch.tensor([480], dtype=torch.int32, device=DEV)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    g.set_option(g.GQAQ_OPT_WAIT_TIMEOUT_NS, 2_000_000)
    g.set_option(g.GQAQ_OPT_TEST_STALL, 1)
    g.gqa_prefill_attn(qd, kd, vd, st, 0.125, workspace=ws)
    torch.cuda.synchronize()
    assert g.device_status() & g.GQAQ_DEV_TIMEOUT
    assert int(ws[:64].count_nonzero()) == 0  # arrivals balanced: counters back at zero
    g.set_option(g.GQAQ_OPT_TEST_STALL, 0)
    out = g.gqa_prefill_attn(qd, kd, vd, st, 0.125, workspace=ws)
    torch.cuda.synchronize()
    assert g.device_status() == 0
    assert_attn_close(out, oracle.prefill_attn(q.numpy(), k.numpy(), v.numpy(), [480], 0.125))


def test_prefill_4k_context_chunk_sampled_rows():
    """A 64-token chunk at the end of a 4K context, Llama-2-7B-shaped heads
    (32 heads, MHA, D=128), batch 2; the oracle checks sampled (head, token) rows."""
    B, Hkv, G, D, Lmax, q_len = 2, 32, 1, 128, 4096, 64
    gen = torch.Generator(device=DEV).manual_seed(40)
    q = torch.randn(B, Hkv * G, q_len, D, generator=gen, device=DEV).to(torch.float16)
    k = torch.randn(B, Hkv, Lmax, D, generator=gen, device=DEV).to(torch.float16)
    v = torch.randn(B, Hkv, Lmax, D, generator=gen, device=DEV).to(torch.float16)
    starts = [Lmax - q_len, 1000]
    st = torch.tensor(starts, dtype=torch.int32, device=DEV)
    out = g.gqa_prefill_attn(q, k, v, st, 1.0 / math.sqrt(D))
    torch.cuda.synchronize()
    assert g.device_status() == 0
    rng = np.random.default_rng(4)
    for _ in range(4):
        b, h = int(rng.integers(B)), int(rng.integers(Hkv * G))
        ref = oracle.prefill_attn(q[b:b + 1, h:h + 1].cpu().numpy(), k[b:b + 1, h // G:h // G + 1].cpu().numpy(),
                                  v[b:b + 1, h // G:h // G + 1].cpu().numpy(), starts[b:b + 1], 1.0 / math.sqrt(D))
        assert_attn_close(out[b:b + 1, h:h + 1], ref, f"b={b} h={h}")
