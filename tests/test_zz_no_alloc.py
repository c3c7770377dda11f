"""gqa_decode_attn_noalloc: the decode attention call for callers that cannot
allocate device memory.

A plugin or custom operator inside a host framework is often handed only its
input and output pointers, because the framework owns every device
allocation. A latency-critical decode loop may also refuse cudaMalloc, since it
can synchronise the device. This entry point keeps its scratch in the
library's own fixed device array instead of a caller workspace. These tests
call it through the C ABI on two calls in a row, with different shapes, so
anything the first call leaves in the shared array would show up in the
second result. Each result must equal gqa_decode_attn's (the entry point that
takes a workspace: the same kernel on the same grid, so bit for bit) and match
the fp64 oracle within the attention tolerance.

This file is named to be collected last and passes in a fresh process too.
"""
import ctypes
import math

import pytest
import torch

import gqa_head_folding_gb300 as g
import oracle
import workloads
from _util import assert_attn_close

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def call_noalloc(q, k, v, vl, scale, out):
    L = g.lib()
    d = g.dims_of(q, k)
    return L.gqa_decode_attn_noalloc(ctypes.byref(d), ctypes.c_void_p(q.data_ptr()),
                                     ctypes.c_void_p(k.data_ptr()), ctypes.c_void_p(v.data_ptr()),
                                     ctypes.c_void_p(vl.data_ptr()), float(scale),
                                     ctypes.c_void_p(out.data_ptr()),
                                     ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


CASES = [
    # (batch, Hq, Hkv, D, Lmax, valid lengths)
    (2, 32, 8, 128, 3000, [3000, 1111]),
    (3, 32, 8, 64, 4096, [4096, 17, 2500]),
]


def test_noalloc_matches_workspace_entry_point_and_oracle_two_calls_in_a_row():
    for i, (B, Hq, Hkv, D, Lmax, valid) in enumerate(CASES):
        w = workloads.Workload(0, "noalloc", batch=B, num_layers=1, num_q_heads=Hq, num_kv_heads=Hkv,
                               head_dim=D, max_len=Lmax)
        x = workloads.make_layer(w, 0, device=DEV, seed=100 + i)
        vl = torch.tensor(valid, dtype=torch.int32, device=DEV)
        scale = 1.0 / math.sqrt(D)
        ref = g.gqa_decode_attn(x["q"], x["k_cache"], x["v_cache"], vl, scale)
        out = torch.full_like(x["q"], float("nan"))
        rc = call_noalloc(x["q"], x["k_cache"], x["v_cache"], vl, scale, out)
        assert rc == g.GQAQ_OK, g.status_string(rc)
        torch.cuda.synchronize()
        assert g.device_status() == 0
        assert torch.equal(out, ref), f"call {i}: differs from gqa_decode_attn"
        want = oracle.attn_repeat_kv(x["q"].cpu().numpy(), x["k_cache"].cpu().numpy(),
                                     x["v_cache"].cpu().numpy(), valid, scale)
        assert_attn_close(out, want, f"call {i}")


def test_noalloc_serves_a_small_shape_with_a_large_group():
    # G = 8, D = 128 at a short context: the grid is capped by the few tiles,
    # so the need is far below the 1 MiB array
    B, Hkv, G, D, Lmax = 1, 4, 8, 128, 64
    w = workloads.Workload(0, "noalloc", batch=B, num_layers=1, num_q_heads=Hkv * G, num_kv_heads=Hkv,
                           head_dim=D, max_len=Lmax)
    x = workloads.make_layer(w, 0, device=DEV, seed=7)
    vl = torch.tensor([50], dtype=torch.int32, device=DEV)
    out = torch.full_like(x["q"], float("nan"))
    assert call_noalloc(x["q"], x["k_cache"], x["v_cache"], vl, 0.125, out) == g.GQAQ_OK
    torch.cuda.synchronize()
    assert torch.equal(out, g.gqa_decode_attn(x["q"], x["k_cache"], x["v_cache"], vl, 0.125))


def test_noalloc_rejects_shapes_beyond_its_scratch():
    # G = 8, D = 128 over 800 tiles of 128 tokens: at least 152 CTAs of 8,320
    # bytes of partials each, more than the 1 MiB array
    B, Hkv, G, D, Lmax = 1, 4, 8, 128, 128 * 200
    q = torch.zeros(B, Hkv * G, D, dtype=torch.float16, device=DEV)
    k = torch.zeros(B, Hkv, Lmax, D, dtype=torch.float16, device=DEV)
    vl = torch.full((B,), Lmax, dtype=torch.int32, device=DEV)
    out = torch.zeros_like(q)
    assert call_noalloc(q, k, k, vl, 0.1, out) == g.GQAQ_ERR_WORKSPACE
