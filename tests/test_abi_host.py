"""Host-side checks of the C ABI: no GPU and no kernel launch needed.

Loads libgqaq.so, checks that it exports every function include/gqaq.h
declares, and drives the argument validation paths that return before any
CUDA call.
"""
import ctypes
import os
import re

import pytest

import gqa_head_folding_gb300 as g

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gqaq.h")


@pytest.fixture(scope="module")
def L():
    if not os.path.exists(g.LIB_PATH):
        from gqa_head_folding_gb300 import _build
        _build.build()
    return g.lib()


def declared_functions():
    text = open(HEADER).read()
    return re.findall(r"GQAQ_API\s+[\w\s\*]+?\b(\w+)\s*\(", text)


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("gqa_decode_attn", "quest_append_kv", "quest_update_meta", "quest_score_pages",
                     "quest_topk_pages", "quest_sparse_attn"):
        assert required in names
    assert tuple(names) == g.EXPORTS


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), f"libgqaq.so does not export {name}"


def test_status_strings(L):
    assert g.status_string(0) == "GQAQ_OK"
    assert g.status_string(g.GQAQ_ERR_WORKSPACE) == "GQAQ_ERR_WORKSPACE"
    assert g.status_string(99) == "GQAQ_ERR_UNKNOWN"
    assert L.gqaq_version() == 100


FAKE = ctypes.c_void_p(0x10000)        # 16-byte aligned, never dereferenced
MISALIGNED = ctypes.c_void_p(0x10008)


def dims(**kw):
    base = dict(batch=1, num_q_heads=32, num_kv_heads=8, head_dim=64, max_len=4096, page_size=16)
    base.update(kw)
    return g.make_dims(**base)


def decode(L, d, q=FAKE, k=FAKE, v=FAKE, vl=FAKE, scale=0.125, out=FAKE, ws=FAKE, wsb=1 << 20):
    return L.gqa_decode_attn(None if d is None else ctypes.byref(d), q, k, v, vl, scale, out, ws, wsb, None)


def test_decode_rejects_bad_arguments(L):
    assert decode(L, None) == g.GQAQ_ERR_INVALID_ARG
    assert decode(L, dims(num_q_heads=30)) == g.GQAQ_ERR_INVALID_ARG      # Hq % Hkv != 0
    assert decode(L, dims(batch=0)) == g.GQAQ_ERR_INVALID_ARG
    assert decode(L, dims(max_len=0)) == g.GQAQ_ERR_INVALID_ARG
    assert decode(L, dims(), q=None) == g.GQAQ_ERR_INVALID_ARG
    assert decode(L, dims(), k=MISALIGNED) == g.GQAQ_ERR_INVALID_ARG
    assert decode(L, dims(), vl=None) == g.GQAQ_ERR_INVALID_ARG
    assert decode(L, dims(), scale=float("nan")) == g.GQAQ_ERR_INVALID_ARG
    assert decode(L, dims(), ws=None) == g.GQAQ_ERR_WORKSPACE
    assert decode(L, dims(), ws=MISALIGNED) == g.GQAQ_ERR_WORKSPACE


def test_decode_reports_unsupported_shapes(L):
    assert decode(L, dims(head_dim=96)) == g.GQAQ_ERR_UNSUPPORTED
    assert decode(L, dims(num_q_heads=24, num_kv_heads=8)) == g.GQAQ_ERR_UNSUPPORTED   # G = 3
    assert decode(L, dims(num_q_heads=128, num_kv_heads=8)) == g.GQAQ_ERR_UNSUPPORTED  # G = 16
    assert decode(L, dims(batch=4096, num_kv_heads=8, num_q_heads=8, max_len=1 << 17)) == \
        g.GQAQ_ERR_UNSUPPORTED                                                          # > 2^31 rows


def test_quest_calls_reject_bad_arguments(L):
    d = dims(head_dim=128)
    assert L.quest_append_kv(ctypes.byref(d), FAKE, FAKE, FAKE, FAKE, FAKE, None, None) == g.GQAQ_ERR_INVALID_ARG
    for bad_s in (0, 4, 12, 24, 128):               # page sizes 8, 16, 32 and 64 are supported
        expect = g.GQAQ_ERR_INVALID_ARG if bad_s < 1 else g.GQAQ_ERR_UNSUPPORTED
        assert L.quest_append_kv(ctypes.byref(dims(page_size=bad_s)), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                                 None) == expect
    assert L.quest_update_meta(ctypes.byref(d), FAKE, FAKE, FAKE, 3, 2, None) == g.GQAQ_ERR_INVALID_ARG
    assert L.quest_update_meta(ctypes.byref(d), FAKE, FAKE, FAKE, 0, 257, None) == g.GQAQ_ERR_INVALID_ARG
    assert L.quest_score_pages(ctypes.byref(d), FAKE, MISALIGNED, FAKE, FAKE, None) == g.GQAQ_ERR_INVALID_ARG
    assert L.quest_topk_pages(ctypes.byref(d), FAKE, FAKE, 0, FAKE, None, 0, None) == g.GQAQ_ERR_INVALID_ARG
    assert L.quest_topk_pages(ctypes.byref(d), FAKE, FAKE, 70000, FAKE, None, 0, None) == g.GQAQ_ERR_INVALID_ARG
    assert L.quest_sparse_attn(ctypes.byref(d), FAKE, FAKE, FAKE, FAKE, FAKE, 0, 0.1, FAKE, FAKE, 1 << 20,
                               None) == g.GQAQ_ERR_INVALID_ARG
    assert L.quest_sparse_attn(ctypes.byref(d), FAKE, FAKE, FAKE, FAKE, FAKE, 8, 0.1, FAKE, None, 0,
                               None) == g.GQAQ_ERR_WORKSPACE


def test_fused_quest_step_rejects_bad_arguments(L):
    d = g.make_dims(1, 8, 2, 128, 4096)
    args = [ctypes.byref(d)] + [FAKE] * 8
    tail = [0.1, FAKE, None, None]
    assert L.quest_decode_attn(*args, 0, *tail, None, 0, None) == g.GQAQ_ERR_INVALID_ARG
    assert L.quest_decode_attn(*args, 70000, *tail, None, 0, None) == g.GQAQ_ERR_INVALID_ARG
    odd = ctypes.c_void_p(FAKE.value + 4)
    assert L.quest_decode_attn(*args, 8, *tail, odd, 1 << 20, None) == g.GQAQ_ERR_WORKSPACE


def test_e4m3_calls_reject_bad_arguments(L):
    d = dims()
    f = ctypes.c_float
    assert L.gqa_decode_attn_e4m3(ctypes.byref(d), FAKE, FAKE, FAKE, f(1.0), f(1.0), FAKE, f(0.1), FAKE, None, 0,
                                  None) == g.GQAQ_ERR_WORKSPACE
    assert L.gqa_decode_attn_e4m3(ctypes.byref(d), FAKE, MISALIGNED, FAKE, f(1.0), f(1.0), FAKE, f(0.1), FAKE, FAKE,
                                  1 << 20, None) == g.GQAQ_ERR_INVALID_ARG
    assert L.gqa_decode_attn_e4m3(ctypes.byref(d), FAKE, FAKE, FAKE, f(float("inf")), f(1.0), FAKE, f(0.1), FAKE,
                                  FAKE, 1 << 20, None) == g.GQAQ_ERR_INVALID_ARG
    assert L.gqa_decode_attn_e4m3(ctypes.byref(dims(head_dim=96)), FAKE, FAKE, FAKE, f(1.0), f(1.0), FAKE, f(0.1),
                                  FAKE, FAKE, 1 << 20, None) == g.GQAQ_ERR_UNSUPPORTED
    assert L.kv_append_e4m3(ctypes.byref(d), FAKE, FAKE, FAKE, FAKE, None, f(1.0), f(1.0), None) == \
        g.GQAQ_ERR_INVALID_ARG
    assert L.kv_append_e4m3(ctypes.byref(d), FAKE, FAKE, FAKE, FAKE, FAKE, f(float("nan")), f(1.0), None) == \
        g.GQAQ_ERR_INVALID_ARG


def test_int4_calls_reject_bad_arguments(L):
    f = ctypes.c_float

    def call(d, ks=FAKE, ws=FAKE):
        return L.gqa_decode_attn_int4(ctypes.byref(d), FAKE, FAKE, ks, FAKE, FAKE, FAKE, f(0.1), FAKE, ws, 1 << 20,
                                      None)
    assert call(dims(max_len=4098)) == g.GQAQ_ERR_UNSUPPORTED      # scale rows need Lmax % 4 == 0
    assert call(dims(), ks=MISALIGNED) == g.GQAQ_ERR_INVALID_ARG
    assert call(dims(), ws=None) == g.GQAQ_ERR_WORKSPACE
    assert call(dims(head_dim=96)) == g.GQAQ_ERR_UNSUPPORTED
    assert L.kv_append_int4(ctypes.byref(dims()), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, None) == \
        g.GQAQ_ERR_INVALID_ARG


def test_prefill_rejects_bad_arguments(L):
    d = dims(max_len=256)
    f = ctypes.c_float

    def call(dd=d, q_len=16, q=FAKE, k=FAKE, start=FAKE, scale=0.1, ws=FAKE):
        return L.gqa_prefill_attn(None if dd is None else ctypes.byref(dd), q_len, q, k, FAKE, start, f(scale), FAKE,
                                  ws, 1 << 20, None)
    assert call(dd=None) == g.GQAQ_ERR_INVALID_ARG
    assert call(q_len=0) == g.GQAQ_ERR_INVALID_ARG
    assert call(q_len=257) == g.GQAQ_ERR_INVALID_ARG                  # longer than the cache
    assert call(q=None) == g.GQAQ_ERR_INVALID_ARG
    assert call(k=MISALIGNED) == g.GQAQ_ERR_INVALID_ARG
    assert call(start=None) == g.GQAQ_ERR_INVALID_ARG
    assert call(scale=float("nan")) == g.GQAQ_ERR_INVALID_ARG
    assert call(ws=None) == g.GQAQ_ERR_WORKSPACE
    assert call(dd=dims(head_dim=96, max_len=256)) == g.GQAQ_ERR_UNSUPPORTED
    assert call(dd=dims(num_q_heads=24, num_kv_heads=8, max_len=256)) == g.GQAQ_ERR_UNSUPPORTED
    assert L.gqaq_prefill_workspace_bytes(ctypes.byref(d), 0) == 0


def test_options(L):
    assert L.gqaq_set_option(g.GQAQ_OPT_MAX_CTAS, -1) == g.GQAQ_ERR_INVALID_ARG
    assert L.gqaq_set_option(12345, 0) == g.GQAQ_ERR_INVALID_ARG
    assert L.gqaq_set_option(g.GQAQ_OPT_MAX_CTAS, 0) == g.GQAQ_OK
    assert L.gqaq_set_option(g.GQAQ_OPT_WAIT_TIMEOUT_NS, 2_000_000_000) == g.GQAQ_OK
    assert L.gqaq_set_option(g.GQAQ_OPT_TEST_STALL, 0) == g.GQAQ_OK
    assert L.gqaq_set_option(g.GQAQ_OPT_CLUSTER_SIZE, 3) == g.GQAQ_ERR_INVALID_ARG
    for v in (0, 1, 2, 4, 8):
        assert L.gqaq_set_option(g.GQAQ_OPT_CLUSTER_SIZE, v) == g.GQAQ_OK
    assert L.gqaq_set_option(g.GQAQ_OPT_CLUSTER_SIZE, 0) == g.GQAQ_OK
    assert L.gqaq_set_option(g.GQAQ_OPT_PDL, 0) == g.GQAQ_OK
    assert L.gqaq_set_option(g.GQAQ_OPT_PDL, 1) == g.GQAQ_OK
    assert L.gqaq_set_option(g.GQAQ_OPT_QUEST_KERNEL, 3) == g.GQAQ_ERR_INVALID_ARG
    assert L.gqaq_set_option(g.GQAQ_OPT_QUEST_KERNEL, -1) == g.GQAQ_ERR_INVALID_ARG
    for v in (2, 1, 0):
        assert L.gqaq_set_option(g.GQAQ_OPT_QUEST_KERNEL, v) == g.GQAQ_OK
    assert L.gqaq_set_option(g.GQAQ_OPT_PREFILL_KERNEL, 3) == g.GQAQ_ERR_INVALID_ARG
    for v in (1, 2, 0):
        assert L.gqaq_set_option(g.GQAQ_OPT_PREFILL_KERNEL, v) == g.GQAQ_OK
    assert L.gqaq_set_option(g.GQAQ_OPT_DENSE_EARLY_KV, 2) == g.GQAQ_ERR_INVALID_ARG
    for v in (1, 0):
        assert L.gqaq_set_option(g.GQAQ_OPT_DENSE_EARLY_KV, v) == g.GQAQ_OK
    assert L.gqaq_set_option(g.GQAQ_OPT_QUEST_EARLY_META, 2) == g.GQAQ_ERR_INVALID_ARG
    assert L.gqaq_set_option(g.GQAQ_OPT_QUEST_EARLY_META, -1) == g.GQAQ_ERR_INVALID_ARG
    for v in (1, 0):
        assert L.gqaq_set_option(g.GQAQ_OPT_QUEST_EARLY_META, v) == g.GQAQ_OK
    assert L.gqaq_set_option(g.GQAQ_OPT_PREFILL_SPLITS, -1) == g.GQAQ_ERR_INVALID_ARG
    assert L.gqaq_set_option(g.GQAQ_OPT_PREFILL_SPLITS, 33) == g.GQAQ_ERR_INVALID_ARG
    for v in (5, 32, 0):
        assert L.gqaq_set_option(g.GQAQ_OPT_PREFILL_SPLITS, v) == g.GQAQ_OK


def test_binding_refuses_cpu_tensors():
    import torch
    q = torch.zeros(1, 8, 64, dtype=torch.float16)
    k = torch.zeros(1, 2, 16, 64, dtype=torch.float16)
    with pytest.raises(ValueError, match="CUDA tensor"):
        g.gqa_decode_attn(q, k, k, torch.ones(1, dtype=torch.int32), 0.125)
