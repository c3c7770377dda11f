"""gqa_decode_attn_noalloc: the decode attention call for callers that cannot
allocate device memory.

A plugin or custom operator inside a host framework is often handed only its
input and output pointers, because the framework owns every device
allocation. A latency-critical decode loop may also refuse cudaMalloc, since it
can synchronise the device. This entry point keeps its scratch in the
library's own fixed device array instead of a caller workspace. These tests
call it through the C ABI and compare it with gqa_decode_attn, the entry point
that takes a workspace, on two calls in a row. The two calls use different
shapes, so anything the first call leaves in the shared array would show up in
the second result.

This file is named to be collected last and passes in a fresh process too.
"""
import ctypes
import math

import pytest
import torch

import gqa_head_folding_gb300 as g
import workloads
from _util import MAX_ABS, MEAN_ABS

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


def test_noalloc_matches_workspace_entry_point_two_calls_in_a_row():
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
        err = (out.double() - ref.double()).abs()
        assert torch.isfinite(out).all()
        assert err.max().item() <= MAX_ABS and err.mean().item() <= MEAN_ABS, f"call {i}"


def test_noalloc_rejects_shapes_beyond_its_scratch():
    # G = 8 at D = 128 needs more than the 1 MiB array on a 152-SM GB300
    B, Hkv, G, D, Lmax = 1, 4, 8, 128, 64
    d = g.make_dims(B, Hkv * G, Hkv, D, Lmax)
    if g.workspace_bytes(d) <= (1 << 20):
        pytest.skip("this device's grid fits the 1 MiB scratch for every supported shape")
    q = torch.zeros(B, Hkv * G, D, dtype=torch.float16, device=DEV)
    k = torch.zeros(B, Hkv, Lmax, D, dtype=torch.float16, device=DEV)
    vl = torch.full((B,), Lmax, dtype=torch.int32, device=DEV)
    out = torch.zeros_like(q)
    assert call_noalloc(q, k, k, vl, 0.1, out) == g.GQAQ_ERR_WORKSPACE
