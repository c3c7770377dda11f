"""Host-side pieces of bench.py: the bytes model against the closed forms the
Quest review prints, and the multi-rank timing reduction on gloo (CPU)."""
import json
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import workloads


def test_bytes_model_matches_quest_closed_forms(golden_dir):
    ex = json.load(open(os.path.join(golden_dir, "byte_arithmetic.json")))["quest"]["ratio_example"]
    L, S, K, D = ex["L"], ex["S"], ex["K"], 128
    full = bench.dense_unit_bytes(D, L)
    quest = bench.meta_unit_bytes(D, L, S) + bench.selected_unit_bytes(D, L, S, K)
    assert quest / full == ex["ratio"] == 1 / S + K * S / L
    assert K * S == ex["B_tokens"]
    # K >= number of pages reads every key and value once
    assert bench.selected_unit_bytes(D, 100, 16, 1000) == 2 * 2 * D * 16 * 7


def test_step_bytes_of_the_workloads():
    # Llama-2-7B-shaped Quest stack: 2 x 512 MiB dense + 30 x (32 MiB meta + 32 MiB selected)
    w = workloads.WORKLOADS[3]
    lens = [[w.max_len]] * w.num_layers
    kv = 2 * bench.roofline_unit_bytes(w, "dense", lens[0])
    q = 30 * (bench.roofline_unit_bytes(w, "score", lens[2]) + bench.roofline_unit_bytes(w, "sparse", lens[2]))
    assert kv + q == 3_087_007_744
    sb = bench.step_bytes(w, lens, fused=False)
    assert sb["launches"] == {"dense": 2, "score": 30, "topk": 30, "sparse": 30, "append": 32}
    assert 0 < sb["total"] - (kv + q) < 0.01 * (kv + q)          # q/out/scores/append are small
    sf = bench.step_bytes(w, lens, fused=True)
    assert sf["launches"] == {"dense": 2, "quest": 30, "append": 2}
    assert 0 < sf["total"] - (kv + q) < sb["total"] - (kv + q)   # no score / page-list traffic
    assert bench.roofline_unit_bytes(w, "quest", lens[2]) == 2 * 2 ** 20 * 32
    # EXAONE-shaped dense: 8 MiB for one full 4096-token layer at batch 1
    w1 = workloads.WORKLOADS[1]
    assert bench.roofline_unit_bytes(w1, "dense", [4096]) == 8 * 2 ** 20
    # GQA Quest at 64K: 32 MiB per sequence per layer (2 MiB metadata... per KV head)
    w4 = workloads.WORKLOADS[4].with_(batch=1)
    assert bench.roofline_unit_bytes(w4, "score", [65536]) + \
        bench.roofline_unit_bytes(w4, "sparse", [65536]) == 32 * 2 ** 20


def test_workload_recipes():
    w = workloads.WORKLOADS[5]
    assert w.n_plant == 82                                          # 1% of 8192 pages
    lens = workloads.valid_lengths(workloads.WORKLOADS[2], 3)
    assert lens.min() >= 1024 and lens.max() <= 4096 and lens.dtype == torch.int32
    assert torch.equal(lens, workloads.valid_lengths(workloads.WORKLOADS[2], 3))   # seeded
    x = workloads.make_layer(w.with_(batch=1, max_len=16 * 50, n_plant=3, num_kv_heads=2, num_q_heads=4),
                             0, "cpu")
    assert x["k_cache"].dtype == torch.float16 and x["pos"].tolist() == [16 * 50 - 1]


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        t = bench.max_over_ranks(0.5 + rank, dist)
        bench.barrier(dist)
        results[rank] = (t, bench.rank_seed(rank))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_world_size_2():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    results = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, results)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert results[0][0] == results[1][0] == 1.5          # every rank sees the slowest rank's time
    assert results[0][1] != results[1][1]                 # ranks draw different sequences


def test_single_rank_needs_no_collective():
    assert bench.max_over_ranks(0.25, None) == 0.25
    bench.barrier(None)


def test_dense_side_and_early_read_flags():
    """--dense runs a Quest workload's caches all dense; the launch string names
    the early reads only for the calls that make them."""
    import argparse
    ns = argparse.Namespace(workload=5, batch=16, k_pages=0, layers=0, page_size=0, budget=0, dense=True)
    w = bench.workload_from_args(ns)
    assert w.k_pages is None and w.batch == 16 and w.max_len == 131072
    c = bench.config_of(w, 1, early_meta=True, early_kv=True)
    assert c["dense_layers"] == 1 and c["k_pages"] is None
    assert "dense: first K/V tiles" in c["launch"] and "Quest:" not in c["launch"]
    w3 = workloads.WORKLOADS[3]
    c3 = bench.config_of(w3, 1, early_meta=True, early_kv=True)
    assert "Quest: first metadata tiles" in c3["launch"] and "dense: first K/V tiles" in c3["launch"]
    assert bench.config_of(w3, 1)["launch"] == "programmatic dependent launch"
    assert bench.config_of(w3, 1, pdl=False)["launch"] == "plain stream order"


def test_captured_traffic_is_near_the_bytes_model():
    """The stored ncu DRAM bytes of the Llama-2-shaped launches sit just above the
    bytes model (nothing read twice), so the bench's `traffic` is a real cross-check."""
    w = workloads.WORKLOADS[3]
    full = [w.max_len]
    quest = bench.roofline_unit_bytes(w, "quest", full)
    dense = bench.roofline_unit_bytes(w, "dense", full)
    assert 1.0 < bench.NCU_TRAFFIC[(3, 1, "quest", "f16", 16)] / quest < 1.02
    assert 1.0 < bench.NCU_TRAFFIC[(3, 1, "dense", "f16", 16)] / dense < 1.02
    pf = bench.prefill_bytes(w.with_(batch=1), [w.max_len - 128], 128)
    assert 1.0 < bench.PREFILL_TRAFFIC[(3, 1, 128)] / pf < 1.03


def test_rotation_covers_four_times_l2():
    l2 = 126 * 2 ** 20
    for nbytes in (8 * 2 ** 20, 32 * 2 ** 20, 157_000_000, 4 * l2 - 1):
        n = bench.rotation_copies(nbytes, l2)
        assert n > 1 and n * nbytes >= 4 * l2 and (n - 1) * nbytes < 4 * l2
        assert "rotation" in bench.l2_note(n, nbytes, l2)
    assert bench.rotation_copies(4 * l2, l2) == 1
    assert bench.rotation_copies(3_087_007_744, l2) == 1
    assert "no rotation" in bench.l2_note(1, 3_087_007_744, l2)
    assert "< 4x L2" in bench.l2_note(0, 8 * 2 ** 20, l2)


def test_default_command_turns_on_by_config_only_for_the_default_workload():
    import argparse
    base = dict(workload=3, batch=0, k_pages=0, layers=0, page_size=0, budget=0, dense=False, unfused=False,
                prefill=0, kv="f16", quest_kernel="cluster")
    assert bench.default_command(argparse.Namespace(**base))
    for k, v in (("workload", 4), ("batch", 2), ("dense", True), ("kv", "e4m3"), ("prefill", 128)):
        assert not bench.default_command(argparse.Namespace(**dict(base, **{k: v})))


def test_reference_arm_never_loads_the_cuda_library():
    """--impl reference times the oracle on host-drawn inputs: the product
    package is never imported, and its config equals the GPU arm's."""
    import subprocess
    import sys
    code = ("import sys, json, io, contextlib, bench\n"
            "buf = io.StringIO()\n"
            "with contextlib.redirect_stdout(buf):\n"
            "    bench.main(['--impl', 'reference', '--workload', '1', '--steps', '1', '--warmup', '0',"
            " '--ref-budget', '0.3'])\n"
            "line = json.loads(buf.getvalue().strip().splitlines()[-1])\n"
            "assert not any(m.startswith('gqa_head_folding_gb300') for m in sys.modules), 'product imported'\n"
            "print(json.dumps(line))\n")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    res = subprocess.run([sys.executable, "-c", code], cwd=root, capture_output=True, text=True, timeout=300)
    assert res.returncode == 0, res.stderr[-2000:]
    line = json.loads(res.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "us/step" and line["value"] > 0
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["extrapolated"] and cb["cores"] >= 1 and cb["one_thread"]["cores"] == 1
    assert line["e2e"] == {"value": line["value"], "unit": "us/step", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    import argparse
    args = argparse.Namespace(workload=1, batch=0, k_pages=0, layers=0, page_size=0, budget=0, dense=False, unfused=False, kv="f16",
              no_pdl=False, quest_kernel="cluster", no_early_meta=False, no_early_kv=False)
    assert line["config"] == bench.arm_config(args, bench.workload_from_args(args), 1)


def test_prefill_roofline_takes_the_binding_peak():
    """A prefill launch below the ridge of the two measured peaks (flops per
    byte) is judged against HBM, above it against the tensor peak; the line
    carries both fractions."""
    peaks = {"hbm_gbs": 6766.0, "tensor_tflops": 1716.6, "source": "measured"}
    ridge = peaks["tensor_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
    w = workloads.WORKLOADS[3].with_(batch=1, num_layers=1)
    for q, bound in ((128, "hbm"), (1024, "tensor")):
        starts = [w.max_len - q]
        flops, nbytes = bench.prefill_flops(w, starts, q), bench.prefill_bytes(w, starts, q)
        assert (flops / nbytes >= ridge) == (bound == "tensor")
        t = 100e-6
        r = bench.prefill_roofline(flops, nbytes, t, peaks)
        assert r["bound"] == bound
        tf, gb = flops / t / 1e12, nbytes / t / 1e9
        assert r["tensor_frac"] == pytest.approx(tf / peaks["tensor_tflops"], rel=1e-3)
        assert r["hbm_frac"] == pytest.approx(gb / peaks["hbm_gbs"], rel=1e-3)
        assert r["frac"] == (r["tensor_frac"] if bound == "tensor" else r["hbm_frac"])
        assert r["unit"] == ("TFLOP/s" if bound == "tensor" else "GB/s")
    pf = bench.prefill_bytes(w, [w.max_len - 1024], 1024)
    assert 1.0 < bench.PREFILL_TRAFFIC[(3, 1, 1024)] / pf < 1.35  # eight 128-row blocks share K/V through L2
