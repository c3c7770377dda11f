"""Pins for the fp64 CPU oracle, each against something other than the oracle.

The oracle is only trusted as a parity reference once these pass: library
routines (numpy's fp16 decoder, numpy min/max and sorting, torch's fp64
scaled-dot-product attention), the pages' printed worked example and byte
arithmetic, closed forms (L=1, identical keys) and brute force on tiny inputs.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle

RNG = np.random.default_rng(7)


def rand_f16(*shape, scale=1.0, rng=RNG):
    return (rng.standard_normal(shape) * scale).astype(np.float16)


# ---------------------------------------------------------------------------
# fp16 decoding: every bit pattern against numpy's own conversion
# ---------------------------------------------------------------------------
def test_f16_decoder_all_bit_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.f16_to_f64(bits)
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    # the sign of zero survives
    assert np.signbit(ours[0x8000]) and not np.signbit(ours[0x0000])


# ---------------------------------------------------------------------------
# The Quest page's worked example (golden values printed on the page)
# ---------------------------------------------------------------------------
def test_quest_worked_example(golden_dir):
    ex = json.load(open(os.path.join(golden_dir, "quest_worked_example.json")))
    q = np.array(ex["q"], dtype=np.float64)
    keys = np.array(ex["page_A_keys"] + ex["page_B_keys"], dtype=np.float64)  # 3 tokens
    # page size 2: page A = tokens 0-1, page B = token 2 (a partial last page)
    k = np.zeros((1, 1, 4, 3)); k[0, 0, :3] = keys
    meta = oracle.page_minmax(k, [3], page_size=2)
    assert np.array_equal(meta[0, 0, 0, 0], [-0.5, -0.1, -0.3])     # m_A
    assert np.array_equal(meta[0, 0, 0, 1], [0.7, 1.2, 0.9])        # M_A
    assert np.array_equal(meta[0, 0, 1, 0], [1.2, 0.0, 0.0])        # m_B = M_B
    u = oracle.page_scores(q[None, None, :], meta, [3], page_size=2)[0, 0]
    assert u[0] == pytest.approx(ex["U_A"], abs=1e-12)
    assert u[0] == pytest.approx(sum(ex["U_A_terms"]), abs=1e-12)
    assert u[1] == pytest.approx(ex["U_B"], abs=1e-12)
    assert keys[:2] @ q == pytest.approx(ex["dots_A"], abs=1e-12)
    assert keys[2] @ q == pytest.approx(ex["dot_B"], abs=1e-12)
    # A outranks B under U, although B holds the larger true dot product
    top1 = oracle.topk_pages(u[None, None, :], [3], page_size=2, k=1)[0, 0]
    assert list(top1) == [0]
    assert max(keys[:2] @ q) < keys[2] @ q


def test_score_uses_min_channel_for_negative_query():
    # the third channel's term is q_3 * m_3 = (-0.2)(-0.3) = +0.06, not q_3 * M_3
    q = np.array([[[0.0, 0.0, -0.2]]])
    k = np.zeros((1, 1, 2, 3)); k[0, 0, 0] = [-0.5, -0.1, -0.3]; k[0, 0, 1] = [0.7, 1.2, 0.9]
    meta = oracle.page_minmax(k, [2], page_size=2)
    u = oracle.page_scores(q, meta, [2], page_size=2)[0, 0, 0]
    assert u == pytest.approx(0.06, abs=1e-15)


# ---------------------------------------------------------------------------
# Metadata against numpy's min/max; the upper bound q.k <= U by brute force
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("L,Lmax,S", [(37, 40, 4), (16, 16, 16), (1, 8, 4), (50, 64, 16)])
def test_page_minmax_matches_numpy(L, Lmax, S):
    k = rand_f16(2, 3, Lmax, 5)
    meta = oracle.page_minmax(k, [L, max(1, L - 3)], page_size=S)
    k64 = k.astype(np.float64)
    for b, lb in enumerate([L, max(1, L - 3)]):
        P = (lb + S - 1) // S
        for p in range(P):
            rows = k64[b, :, p * S:min(p * S + S, lb)]
            assert np.array_equal(meta[b, :, p, 0], rows.min(axis=1))
            assert np.array_equal(meta[b, :, p, 1], rows.max(axis=1))
        assert np.all(np.isnan(meta[b, :, P:]))


@pytest.mark.parametrize("G", [1, 4])
def test_upper_bound_every_key(G):
    S, Hkv, D, L = 4, 3, 8, 45
    Hq = Hkv * G
    q = rand_f16(1, Hq, D, scale=2.0)
    q[0, 0, :4] = -np.abs(q[0, 0, :4])                 # negative components
    k = rand_f16(1, Hkv, 48, D)
    k[0, 1, 8:12] += np.float16(2.0)                   # a planted page
    meta = oracle.page_minmax(k, [L], page_size=S)
    u = oracle.page_scores(q, meta, [L], page_size=S)
    q64, k64 = q.astype(np.float64), k.astype(np.float64)
    for kv in range(Hkv):
        for t in range(L):
            dots = q64[0, kv * G:(kv + 1) * G] @ k64[0, kv, t]
            assert dots.max() <= u[0, kv, t // S] + 1e-12


def test_score_is_tight_for_single_token_page():
    # with one token per page the bound is attained: U = q.k exactly
    q = rand_f16(1, 2, 8)
    k = rand_f16(1, 2, 5, 8)
    meta = oracle.page_minmax(k, [5], page_size=1)
    u = oracle.page_scores(q, meta, [5], page_size=1)
    dots = np.einsum("hd,htd->ht", q[0].astype(np.float64), k[0].astype(np.float64))
    assert np.allclose(u[0], dots, rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------
# Top-K: against numpy's lexsort; K >= P; scale invariance of the ranking
# ---------------------------------------------------------------------------
def _numpy_topk(scores, P, K):
    order = np.lexsort((np.arange(P), -scores[:P]))   # by -score, then by page index
    return np.sort(order[:min(K, P)])


@pytest.mark.parametrize("P,Pmax,K", [(37, 40, 5), (40, 40, 40), (9, 12, 20), (100, 100, 1)])
def test_topk_against_lexsort(P, Pmax, K):
    rng = np.random.default_rng(P * 31 + K)
    s = rng.standard_normal((2, 3, Pmax))
    s[0, 0, 3] = s[0, 0, 7] = s[0, 0, 11] = 5.0          # exact ties at the top
    s[1, 2, :] = 1.0                                     # all equal
    idx = oracle.topk_pages(s, [P * 16, P * 16], page_size=16, k=K)
    for b in range(2):
        for h in range(3):
            ref = _numpy_topk(s[b, h], P, K)
            n = len(ref)
            assert np.array_equal(idx[b, h, :n], ref)
            assert np.all(idx[b, h, n:] == -1)
    # all-equal scores: ties go to the lowest page indices
    assert np.array_equal(idx[1, 2, :min(K, P)], np.arange(min(K, P)))


def test_topk_ranking_invariant_under_positive_scale():
    S, Hkv, D, L, K = 16, 2, 16, 16 * 30, 7
    q = rand_f16(1, Hkv, D)
    k = rand_f16(1, Hkv, L, D)
    meta = oracle.page_minmax(k, [L], page_size=S)
    base = oracle.topk_pages(oracle.page_scores(q, meta, [L], S), [L], S, K)
    for c in (0.25, 2.0, 8.0):                        # powers of two scale exactly
        qc = (q.astype(np.float64) * c)
        sel = oracle.topk_pages(oracle.page_scores(qc, meta, [L], S), [L], S, K)
        assert np.array_equal(sel, base)


# ---------------------------------------------------------------------------
# Dense attention: repeat_kv form vs torch fp64 SDPA, vs the folded form,
# closed forms, and the head mapping h = G*kv + g
# ---------------------------------------------------------------------------
def _sdpa_reference(q, k, v, valid_len, scale, G):
    out = []
    for b in range(q.shape[0]):
        L = int(valid_len[b])
        qb = torch.from_numpy(q[b].astype(np.float64))[:, None, :]          # [Hq,1,D]
        kb = torch.from_numpy(k[b, :, :L].astype(np.float64)).repeat_interleave(G, dim=0)
        vb = torch.from_numpy(v[b, :, :L].astype(np.float64)).repeat_interleave(G, dim=0)
        o = torch.nn.functional.scaled_dot_product_attention(qb, kb, vb, scale=scale)
        out.append(o[:, 0, :].numpy())
    return np.stack(out)


@pytest.mark.parametrize("B,Hkv,G,D,Lmax", [(2, 3, 4, 8, 37), (1, 2, 1, 16, 20), (2, 1, 8, 4, 9)])
def test_dense_matches_torch_sdpa(B, Hkv, G, D, Lmax):
    q = rand_f16(B, Hkv * G, D)
    k = rand_f16(B, Hkv, Lmax, D)
    v = rand_f16(B, Hkv, Lmax, D)
    valid = np.array([Lmax, max(1, Lmax // 3)][:B])
    scale = 1.0 / np.sqrt(D)
    ours = oracle.attn_repeat_kv(q, k, v, valid, scale)
    ref = _sdpa_reference(q, k, v, valid, scale, G)
    assert np.allclose(ours, ref, rtol=0, atol=1e-13)


@pytest.mark.parametrize("B,Hkv,G,D,Lmax", [(2, 3, 4, 8, 37), (1, 2, 2, 16, 20), (2, 1, 8, 4, 9)])
def test_folded_equals_repeat_kv_bitwise(B, Hkv, G, D, Lmax):
    q = rand_f16(B, Hkv * G, D)
    k = rand_f16(B, Hkv, Lmax, D)
    v = rand_f16(B, Hkv, Lmax, D)
    valid = np.array([Lmax, 5][:B])
    a = oracle.attn_repeat_kv(q, k, v, valid, 0.3)
    f = oracle.attn_folded(q, k, v, valid, 0.3)
    assert np.array_equal(a, f)


def test_head_mapping_contiguous_groups():
    # each KV head's values are one constant, so output row h must equal that
    # constant for kv = h // G; an interleaved mapping (kv = h % Hkv) would not
    Hkv, G, D, L = 3, 4, 8, 11
    q = rand_f16(1, Hkv * G, D)
    k = rand_f16(1, Hkv, L, D)
    v = np.zeros((1, Hkv, L, D), dtype=np.float16)
    for kv in range(Hkv):
        v[0, kv] = np.float16(kv + 1)
    out = oracle.attn_repeat_kv(q, k, v, [L], 0.5)[0]
    for h in range(Hkv * G):
        assert np.allclose(out[h], h // G + 1, rtol=0, atol=1e-14)
        if h % Hkv != h // G:   # the interleaved reading would give another constant
            assert not np.allclose(out[h], h % Hkv + 1, rtol=0, atol=1e-3)


def test_single_token_returns_its_value():
    q = rand_f16(1, 8, 16); k = rand_f16(1, 2, 7, 16); v = rand_f16(1, 2, 7, 16)
    out = oracle.attn_repeat_kv(q, k, v, [1], 0.25)
    for h in range(8):
        assert np.array_equal(out[0, h], v[0, h // 4, 0].astype(np.float64))


def test_identical_keys_average_values():
    q = rand_f16(1, 4, 8)
    k = np.repeat(rand_f16(1, 1, 1, 8), 9, axis=2)
    v = rand_f16(1, 1, 9, 8)
    out = oracle.attn_repeat_kv(q, k, v, [9], 0.35)
    assert np.allclose(out[0], v[0, 0].astype(np.float64).mean(axis=0)[None, :], atol=1e-15)


# ---------------------------------------------------------------------------
# Sparse attention: K >= P equals dense; otherwise SDPA over gathered tokens
# ---------------------------------------------------------------------------
def test_sparse_with_all_pages_equals_dense():
    Hkv, G, D, Lmax, S, L = 2, 4, 8, 70, 16, 67
    q = rand_f16(1, Hkv * G, D); k = rand_f16(1, Hkv, Lmax, D); v = rand_f16(1, Hkv, Lmax, D)
    P = (L + S - 1) // S
    idx = np.full((1, Hkv, P + 3), -1, dtype=np.int32)
    idx[0, :, :P] = np.arange(P)
    sp = oracle.sparse_attn(q, k, v, [L], idx, S, 0.3)
    dn = oracle.attn_repeat_kv(q, k, v, [L], 0.3)
    assert np.array_equal(sp, dn)


def test_sparse_matches_sdpa_on_gathered_tokens():
    Hkv, G, D, Lmax, S, L = 2, 2, 8, 80, 16, 75
    q = rand_f16(1, Hkv * G, D); k = rand_f16(1, Hkv, Lmax, D); v = rand_f16(1, Hkv, Lmax, D)
    idx = np.array([[[0, 2, 4, -1], [1, 3, -1, -1]]], dtype=np.int32)
    sp = oracle.sparse_attn(q, k, v, [L], idx, S, 0.4)
    for kv in range(Hkv):
        toks = [t for p in idx[0, kv] if p >= 0 for t in range(p * S, min(p * S + S, L))]
        kk = k[:, kv:kv + 1, toks]; vv = v[:, kv:kv + 1, toks]
        ref = _sdpa_reference(q[:, kv * G:(kv + 1) * G], kk, vv, [len(toks)], 0.4, G)
        assert np.allclose(sp[0, kv * G:(kv + 1) * G], ref[0], rtol=0, atol=1e-13)


# ---------------------------------------------------------------------------
# Byte arithmetic the pages print
# ---------------------------------------------------------------------------
def test_quest_bytes_model(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "byte_arithmetic.json")))["quest"]
    ex = g["budget_example"]
    assert oracle.token_budget(ex["K"], ex["S"]) == ex["B_tokens"]
    ex = g["ratio_example"]
    assert oracle.token_budget(ex["K"], ex["S"]) == ex["B_tokens"]
    assert oracle.quest_read_ratio(ex["L"], ex["S"], ex["K"]) == ex["ratio"]
    assert ex["B_tokens"] // ex["S"] == ex["pages_for_4k_tokens"]
    M, L, S, K = 256, ex["L"], ex["S"], ex["K"]
    quest = oracle.bytes_meta(M, L, S) + oracle.bytes_selected(M, K, S)
    assert quest / oracle.bytes_full(M, L) == ex["ratio"]


def test_repeat_kv_storage_and_byte_counts(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "byte_arithmetic.json")))["opt"]
    k = torch.zeros(1, *g["layer_cache_shape"], dtype=torch.float16)      # [1,8,4096,64]
    assert k.untyped_storage().nbytes() == g["layer_cache_bytes"]
    e = k[:, :, None].expand(1, 8, 4, 4096, 64)                           # view, stride 0
    assert e.untyped_storage().data_ptr() == k.untyped_storage().data_ptr()
    assert e.untyped_storage().nbytes() == g["expand_storage_bytes"]
    r = e.reshape(1, 32, 4096, 64)                                        # copies
    assert r.untyped_storage().data_ptr() != k.untyped_storage().data_ptr()
    assert r.untyped_storage().nbytes() == g["reshape_storage_bytes"] == g["tile_output_bytes"]
    assert 2 * g["num_layers"] * g["layer_cache_bytes"] == g["all_layers_kv_bytes"]
    assert g["num_layers"] * 2 * 8 * 64 * 2 == g["per_token_write_bytes"]
    assert g["tile_ops"] * g["tile_output_bytes"] == g["tile_outputs_total_bytes"]
    assert 2 * g["tile_outputs_total_bytes"] == g["tile_write_plus_read_bytes"]
    q = torch.zeros(*g["q_decode_shape"], dtype=torch.float16)
    assert q.numel() * 2 == g["q_decode_bytes"]
    assert q.reshape(1, 8, 4, 64).data_ptr() == q.data_ptr()              # the fold is a view


# ---------------------------------------------------------------------------
# E4M3 (the 8-bit KV-cache variant): decoding, quantization, attention
# ---------------------------------------------------------------------------
def test_e4m3_decoder_all_codes_against_torch():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_to_f64(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert list(np.nonzero(nan)[0]) == [0x7F, 0xFF]                 # the only NaNs: S.1111.111
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])


def test_e4m3_decoder_closed_forms():
    v = oracle.e4m3_to_f64(np.array([0x38, 0x7E, 0x08, 0x07, 0x01, 0x80, 0xB8, 0x3C], dtype=np.uint8))
    # 1.0 = 2^(7-7); 448 = 1.75 * 2^8; 2^-6 smallest normal; 7 * 2^-9 largest subnormal
    assert list(v[:5]) == [1.0, 448.0, 2.0 ** -6, 7 * 2.0 ** -9, 2.0 ** -9]
    assert v[5] == 0.0 and np.signbit(v[5])                           # negative zero
    assert v[6] == -1.0 and v[7] == 1.5
    pos = oracle.e4m3_to_f64(np.arange(0, 127, dtype=np.uint8))
    assert np.all(np.diff(pos) > 0)                                   # codes 0..126 increase


def test_e4m3_quantize_against_torch_in_range():
    rng = np.random.default_rng(11)
    x = (rng.standard_normal(200_000) * 60).astype(np.float16)
    x = x[np.abs(x.astype(np.float64)) * 1.5 < 448]
    codes = oracle.quantize_e4m3(x, 1.5)
    ref = (torch.from_numpy(x).float() * 1.5).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(codes, ref)


def test_e4m3_quantize_ties_and_saturation():
    x = np.array([1.0, 1.0625, 1.1875, 448, 470, 1000, -1000, 2.0 ** -10, 1.5 * 2.0 ** -9, 0.0, -0.0],
                 dtype=np.float16)
    codes = oracle.quantize_e4m3(x, 1.0)
    # 1.0625 halfway between 1.0 (56) and 1.125 (57) -> even 56; 1.1875 between 57 and 58 -> 58;
    # above 448 saturates to 448 (126 / 254); 2^-10 halfway between 0 and 2^-9 -> 0;
    # 1.5 * 2^-9 halfway between codes 1 and 2 -> 2; signed zeros keep their sign bit
    assert list(codes) == [56, 56, 58, 126, 126, 126, 254, 0, 2, 0, 128]


def test_e4m3_quantize_then_decode_is_nearest():
    rng = np.random.default_rng(12)
    x = (rng.standard_normal(5000) * 40).astype(np.float16)
    codes = oracle.quantize_e4m3(x, 2.0)
    grid = oracle.e4m3_to_f64(np.arange(256, dtype=np.uint8))
    grid = grid[np.isfinite(grid)]
    y = x.astype(np.float64) * 2.0
    err = np.abs(oracle.e4m3_to_f64(codes) - np.clip(y, -448, 448))
    best = np.min(np.abs(grid[None, :] - np.clip(y, -448, 448)[:, None]), axis=1)
    assert np.array_equal(err, best)


def test_attn_e4m3_matches_sdpa_on_torch_dequantized_cache():
    rng = np.random.default_rng(13)
    B, Hkv, G, D, Lmax = 2, 2, 4, 64, 40
    q = rand_f16(B, Hkv * G, D, rng=rng)
    kc = rng.integers(0, 256, size=(B, Hkv, Lmax, D), dtype=np.uint8)
    kc[(kc & 0x7F) == 0x7F] = 0x38                                    # no NaN codes in a cache
    vc = rng.integers(0, 256, size=(B, Hkv, Lmax, D), dtype=np.uint8)
    vc[(vc & 0x7F) == 0x7F] = 0x30
    vl = [Lmax, 17]
    ks, vs, scale = 0.01, 0.02, 0.125
    got = oracle.attn_e4m3(q, kc, vc, ks, vs, vl, scale)
    k = torch.from_numpy(kc).view(torch.float8_e4m3fn).to(torch.float64) * ks
    v = torch.from_numpy(vc).view(torch.float8_e4m3fn).to(torch.float64) * vs
    qt = torch.from_numpy(q.astype(np.float64))
    for b in range(B):
        L = vl[b]
        kk = k[b, :, :L].repeat_interleave(G, dim=0)
        vv = v[b, :, :L].repeat_interleave(G, dim=0)
        ref = torch.nn.functional.scaled_dot_product_attention(qt[b][:, None, :], kk, vv, scale=scale)[:, 0]
        assert np.allclose(got[b], ref.numpy(), rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------
# Prefill (q_len > 1): causal attention of a chunk, group axis merged into rows
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("G,q_len,start", [(1, 5, 0), (4, 7, 0), (2, 9, 13), (8, 3, 30)])
def test_prefill_matches_sdpa_causal(G, q_len, start):
    rng = np.random.default_rng(G * 100 + q_len)
    B, Hkv, D, Lmax = 2, 2, 32, 48
    q = rand_f16(B, Hkv * G, q_len, D, rng=rng)
    k = rand_f16(B, Hkv, Lmax, D, rng=rng)
    v = rand_f16(B, Hkv, Lmax, D, rng=rng)
    st = [start, max(0, start - 3)]
    got = oracle.prefill_attn(q, k, v, st, 0.2)
    for b in range(B):
        L = st[b] + q_len
        kk = torch.from_numpy(k[b, :, :L].astype(np.float64)).repeat_interleave(G, dim=0)
        vv = torch.from_numpy(v[b, :, :L].astype(np.float64)).repeat_interleave(G, dim=0)
        # row t sees cache rows <= start + t: a bottom-right-aligned causal mask
        mask = torch.arange(L)[None, :] <= (st[b] + torch.arange(q_len))[:, None]
        ref = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(q[b].astype(np.float64)), kk, vv, attn_mask=mask, scale=0.2)
        assert np.allclose(got[b], ref.numpy(), rtol=0, atol=1e-12)


def test_prefill_from_zero_equals_is_causal():
    rng = np.random.default_rng(5)
    G, q_len, D = 4, 12, 16
    q = rand_f16(1, 2 * G, q_len, D, rng=rng)
    k = rand_f16(1, 2, q_len, D, rng=rng)
    v = rand_f16(1, 2, q_len, D, rng=rng)
    got = oracle.prefill_attn(q, k, v, [0], 0.25)[0]
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q[0].astype(np.float64)),
        torch.from_numpy(k[0].astype(np.float64)).repeat_interleave(G, dim=0),
        torch.from_numpy(v[0].astype(np.float64)).repeat_interleave(G, dim=0), is_causal=True, scale=0.25)
    assert np.allclose(got, ref.numpy(), rtol=0, atol=1e-12)


def test_prefill_one_token_is_decode():
    rng = np.random.default_rng(6)
    q = rand_f16(2, 8, 1, 64, rng=rng)
    k = rand_f16(2, 2, 30, 64, rng=rng)
    v = rand_f16(2, 2, 30, 64, rng=rng)
    st = [29, 11]
    got = oracle.prefill_attn(q, k, v, st, 0.125)[:, :, 0]
    ref = oracle.attn_repeat_kv(q[:, :, 0], k, v, [s + 1 for s in st], 0.125)
    assert np.array_equal(got, ref)


def test_prefill_first_row_sees_one_token():
    rng = np.random.default_rng(7)
    q = rand_f16(1, 2, 4, 16, rng=rng)
    k = rand_f16(1, 1, 4, 16, rng=rng)
    v = rand_f16(1, 1, 4, 16, rng=rng)
    got = oracle.prefill_attn(q, k, v, [0], 0.5)
    assert np.array_equal(got[0, :, 0], np.repeat(v[0, :, 0].astype(np.float64), 2, axis=0))


# ---------------------------------------------------------------------------
# INT4 (the 4-bit KV-cache variant): per-row symmetric quantization
# ---------------------------------------------------------------------------
def _nibbles(codes):
    c = np.asarray(codes)
    return np.stack([c & 15, c >> 4], axis=-1).reshape(c.shape[:-1] + (c.shape[-1] * 2,)).astype(np.int64)


def test_int4_codes_are_the_nearest_grid_point():
    rng = np.random.default_rng(21)
    x = (rng.standard_normal((300, 64)) * rng.uniform(0.01, 30, size=(300, 1))).astype(np.float16)
    codes, scales = oracle.quantize_int4(x)
    xf = x.astype(np.float32)
    amax = np.abs(xf).max(axis=1)
    assert np.array_equal(scales, amax / np.float32(7.0))
    q = _nibbles(codes) - 8
    assert q.min() >= -7 and q.max() <= 7
    # brute force over the 15 levels, in the same fp32 units x / scale
    t = xf / scales[:, None]
    grid = np.arange(-7, 8)
    dist = np.abs(t[:, :, None] - grid[None, None, :])
    best = dist.min(axis=2)
    assert np.all(np.abs(t - q) == best)
    # the row maximum lands on +-7
    arg = np.abs(xf).argmax(axis=1)
    assert np.all(np.abs(q[np.arange(300), arg]) == 7)


def test_int4_ties_zero_rows_and_packing():
    x = np.zeros((3, 8), dtype=np.float32)
    x[0] = [7, 2.5, -2.5, 3.5, 0.5, -0.5, 1.5, -7]        # scale 1: ties go to the even level
    x[1] = [14, 5, -5, 1, 0, 0, 0, 0]                    # scale 2: 2.5 -> 2, -2.5 -> -2, 0.5 -> 0
    codes, scales = oracle.quantize_int4(x)
    assert list(scales) == [1.0, 2.0, 0.0]
    assert list(_nibbles(codes)[0] - 8) == [7, 2, -2, 4, 0, 0, 2, -7]
    assert list(_nibbles(codes)[1] - 8) == [7, 2, -2, 0, 0, 0, 0, 0]
    assert list(_nibbles(codes)[2]) == [8] * 8               # an all-zero row: scale 0, level 0
    # channel 2i in the low nibble of byte i
    assert codes[0, 0] == ((2 + 8) << 4) | (7 + 8)


def test_int4_dequantize_closed_form():
    rng = np.random.default_rng(22)
    codes = rng.integers(0, 256, size=(5, 3, 32), dtype=np.uint8)
    scales = rng.uniform(0.001, 3, size=(5, 3)).astype(np.float32)
    got = oracle.dequantize_int4(codes, scales)
    ref = (_nibbles(codes) - 8) * scales[..., None].astype(np.float64)
    assert np.array_equal(got, ref)


def test_attn_int4_matches_sdpa_on_dequantized_cache():
    rng = np.random.default_rng(23)
    B, Hkv, G, D, Lmax = 2, 2, 4, 64, 40
    q = rand_f16(B, Hkv * G, D, rng=rng)
    kc, ks = oracle.quantize_int4(rand_f16(B, Hkv, Lmax, D, rng=rng))
    vc, vs = oracle.quantize_int4(rand_f16(B, Hkv, Lmax, D, rng=rng))
    vl = [Lmax, 9]
    got = oracle.attn_int4(q, kc, ks, vc, vs, vl, 0.125)
    k = torch.from_numpy((_nibbles(kc) - 8) * ks[..., None].astype(np.float64))
    v = torch.from_numpy((_nibbles(vc) - 8) * vs[..., None].astype(np.float64))
    qt = torch.from_numpy(q.astype(np.float64))
    for b in range(B):
        L = vl[b]
        ref = torch.nn.functional.scaled_dot_product_attention(
            qt[b][:, None, :], k[b, :, :L].repeat_interleave(G, dim=0), v[b, :, :L].repeat_interleave(G, dim=0),
            scale=0.125)[:, 0]
        assert np.allclose(got[b], ref.numpy(), rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------
# Page min/max over an E4M3 key cache: the page-score section's m and M of
# the keys' values, kept as E4M3 codes (zero bound stored as +0)
# ---------------------------------------------------------------------------
def _torch_e4m3_values():
    """Value of every code, decoded by torch's float8 type (independent of the oracle)."""
    return torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def _value_to_code(vals):
    table = _torch_e4m3_values()
    lut = {}
    for c in range(256):
        v = table[c]
        if np.isnan(v):
            continue
        if v == 0.0:
            lut[0.0] = 0
        elif v not in lut:
            lut[v] = c
    return np.vectorize(lambda v: lut[float(v)], otypes=[np.uint8])(vals)


def test_page_minmax_e4m3_brute_force_against_torch_decoding():
    rng = np.random.default_rng(11)
    finite = [c for c in range(256) if c not in (0x7F, 0xFF)]
    B, Hkv, Lmax, D, S = 2, 3, 16 * 5 + 7, 8, 16
    codes = rng.choice(finite, size=(B, Hkv, Lmax, D)).astype(np.uint8)
    valid = [Lmax, 16 * 2 + 3]
    meta = oracle.page_minmax_e4m3(codes, valid, S)
    vals = _torch_e4m3_values()[codes]
    for b in range(B):
        P = (valid[b] + S - 1) // S
        for p in range(P):
            rows = vals[b, :, p * S:min(p * S + S, valid[b])]
            assert np.array_equal(meta[b, :, p, 0], _value_to_code(rows.min(axis=1)))
            assert np.array_equal(meta[b, :, p, 1], _value_to_code(rows.max(axis=1)))
        assert np.all(meta[b, :, P:] == 0x7F)          # pages with no valid token are left alone


def test_page_minmax_e4m3_values_equal_fp64_page_minmax_of_dequantized_keys():
    # scale * value(code) is the dequantized bound: the fp64 page min/max of
    # the dequantized cache, exactly (scale > 0 keeps the order)
    rng = np.random.default_rng(12)
    x = rng.normal(size=(1, 2, 16 * 4 + 9, 64)).astype(np.float16)
    scale = float(np.abs(x.astype(np.float32)).max()) / 448.0
    codes = oracle.quantize_e4m3(x, 1.0 / scale)
    valid = [16 * 4 + 9]
    meta = oracle.page_minmax_e4m3(codes, valid, 16)
    deq = oracle.e4m3_to_f64(codes) * scale
    ref = oracle.page_minmax(deq, valid, 16)
    assert np.array_equal(oracle.e4m3_to_f64(meta[:, :, :5]) * scale, ref[:, :, :5])


def test_page_minmax_e4m3_zero_bounds_are_plus_zero():
    codes = np.zeros((1, 1, 16, 4), np.uint8)
    codes[0, 0, :, 0] = 0x80                            # all -0
    codes[0, 0, ::2, 1] = 0x80                          # -0 and +0 mixed
    codes[0, 0, :, 2] = 0x38                            # 1.0 everywhere
    codes[0, 0, 3, 2] = 0x80                            # one -0: the min is zero
    codes[0, 0, :, 3] = 0xB8                            # -1.0 everywhere
    codes[0, 0, 5, 3] = 0x80                            # one -0: the max is zero
    meta = oracle.page_minmax_e4m3(codes, [16], 16)[0, 0, 0]
    assert meta[0].tolist() == [0x00, 0x00, 0x00, 0xB8]
    assert meta[1].tolist() == [0x00, 0x00, 0x38, 0x00]


def test_e4m3_page_bound_holds_for_every_key():
    # q.k <= U(p, q) for every key of every page, U from the scaled E4M3 bounds
    rng = np.random.default_rng(13)
    x = rng.normal(size=(1, 2, 16 * 6, 32)).astype(np.float16)
    codes = oracle.quantize_e4m3(x, 40.0)
    scale = 1.0 / 40.0
    meta = oracle.e4m3_to_f64(oracle.page_minmax_e4m3(codes, [96], 16)) * scale
    q = rng.normal(size=(1, 2, 32)).astype(np.float16)
    U = oracle.page_scores(q, meta, [96], 16)
    k = oracle.e4m3_to_f64(codes) * scale
    qk = np.einsum("hd,htd->ht", oracle.f16_to_f64(q[0]), k[0])
    for p in range(6):
        assert np.all(qk[:, p * 16:(p + 1) * 16] <= U[0, :, p][:, None] * (1 + 1e-12) + 1e-12)
