"""Decode-step attention benchmark: dense folded-GQA attention + Quest top-K.

One step = one decode step over every layer of the workload, run through the
library's C ABI:
  - dense layers: attend over every valid token;
  - Quest layers: append the new token and update its page's min/max, score
    every page, pick the top-K pages, attend over them.
The whole step is captured in one CUDA graph and replayed. The default
workload is the Llama-2-7B-shaped Quest stack: 32 layers, 32 heads, D=128,
32768 tokens, 16-token pages, K=128 (a 2048-token budget), layers 0-1 dense,
batch 1. It is the one workload whose single step runs every stage. Each
step streams about 3.1 GB of distinct cache and metadata, far more than the
129 MB L2, so no L2 flush is needed between steps.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--workload 1..5] [--batch B]
                       [--impl ours|reference]
Prints one JSON line (rank 0).
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

import workloads  # noqa: E402

METRIC = "decode-attn µs/step and achieved HBM GB/s vs peak (dense GQA-fold; Quest top-K)"
UNIT = "us/step"


# ---------------------------------------------------------------------------
# Bytes model ("Quest ..." review, bytes-model section): M bytes per key or
# value vector; dense reads 2ML per KV head, Quest reads ~2ML/S of metadata
# plus 2MKS of selected keys and values.
# ---------------------------------------------------------------------------
def kv_vector_bytes(head_dim: int, kv: str = "f16") -> int:
    """M: bytes of one cached key or value vector (fp16; 8-bit E4M3 codes; 4-bit
    levels plus the row's fp32 scale)."""
    if kv == "int4":
        return head_dim // 2 + 4
    return head_dim * (1 if kv == "e4m3" else 2)


def dense_unit_bytes(head_dim: int, length: int, kv: str = "f16") -> int:
    """Keys and values of one (sequence, KV head): 2 M L."""
    return 2 * kv_vector_bytes(head_dim, kv) * length


def meta_unit_bytes(head_dim: int, length: int, page_size: int, kv: str = "f16") -> int:
    """Min and max vectors of every page of one (sequence, KV head): 2 M ceil(L/S)
    (E4M3 bounds: one code byte per channel)."""
    return 2 * kv_vector_bytes(head_dim, kv) * ((length + page_size - 1) // page_size)


def selected_unit_bytes(head_dim: int, length: int, page_size: int, k_pages: int, kv: str = "f16") -> int:
    """Keys and values of the selected pages: 2 M S min(K, P)."""
    pages = (length + page_size - 1) // page_size
    return 2 * kv_vector_bytes(head_dim, kv) * page_size * min(k_pages, pages)


def step_bytes(w: workloads.Workload, lens_per_layer, fused: bool = True, kv: str = "f16") -> dict:
    """Algorithmic bytes of one step, by call family (per-step totals).

    Families follow the calls a step makes: "dense" (dense layers), "append"
    (appends outside the fused call), and either "quest" (one fused call per
    Quest layer) or "score" / "topk" / "sparse" (the step-by-step calls)."""
    M, D, S, G = kv_vector_bytes(w.head_dim), w.head_dim, w.page_size, w.group
    fam, launches = {}, {}

    def add(name, nbytes):
        fam[name] = fam.get(name, 0) + nbytes

    def count(name):
        launches[name] = launches.get(name, 0) + 1

    qo = 2 * G * M                                   # q read + out write per unit
    app_unit = 2 * M + 2 * M + 4 * M                 # new k,v read, row write, page min/max read+write
    if kv != "f16":                                  # new k,v read (fp16), low-bit rows written
        app_unit = 2 * M + 2 * kv_vector_bytes(D, kv)
        if kv == "e4m3" and w.append:                # and the page's E4M3 bounds read and written
            app_unit += 4 * kv_vector_bytes(D, kv)
    for layer, lens in enumerate(lens_per_layer):
        dense = w.layer_is_dense(layer)
        if w.append and (dense or not fused):
            count("append")
            add("append", w.batch * w.num_kv_heads * app_unit)
        if dense:
            count("dense")
            for L in lens:
                add("dense", w.num_kv_heads * (dense_unit_bytes(D, L, kv) + qo))
        elif fused:
            count("quest")
            for L in lens:
                add("quest", w.num_kv_heads * ((app_unit if w.append else 0) + meta_unit_bytes(D, L, S, kv) +
                                               selected_unit_bytes(D, L, S, w.k_pages, kv) + qo))
        else:
            for name in ("score", "topk", "sparse"):
                count(name)
            for L in lens:
                P = (L + S - 1) // S
                n = min(w.k_pages, P)
                add("score", w.num_kv_heads * (meta_unit_bytes(D, L, S, kv) + G * M + 4 * P))
                add("topk", w.num_kv_heads * (4 * P + 4 * w.k_pages))
                add("sparse", w.num_kv_heads * (selected_unit_bytes(D, L, S, w.k_pages, kv) + 4 * n + qo))
    return {"bytes": fam, "launches": launches, "total": sum(fam.values())}


def roofline_unit_bytes(w: workloads.Workload, family: str, lens, kv: str = "f16") -> int:
    """Per-launch bytes of the per-unit figures (K/V, metadata, selected K/V)."""
    D, S = w.head_dim, w.page_size
    if family == "dense":
        return sum(w.num_kv_heads * dense_unit_bytes(D, L, kv) for L in lens)
    if family == "score":
        return sum(w.num_kv_heads * meta_unit_bytes(D, L, S, kv) for L in lens)
    if family == "sparse":
        return sum(w.num_kv_heads * selected_unit_bytes(D, L, S, w.k_pages, kv) for L in lens)
    if family == "quest":
        return roofline_unit_bytes(w, "score", lens, kv) + roofline_unit_bytes(w, "sparse", lens, kv)
    raise ValueError(family)


# ---------------------------------------------------------------------------
# Distributed plumbing (one process per GPU; every rank runs its own
# sequences, so no collective touches the data path)
# ---------------------------------------------------------------------------
def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def init_dist(world: int, backend: str):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)
    return dist if world > 1 else None


def barrier(dist):
    if dist is not None:
        dist.barrier()


def max_over_ranks(value: float, dist, device=None) -> float:
    if dist is None:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def rank_seed(rank: int) -> int:
    return 7919 * rank


# ---------------------------------------------------------------------------
# Clocks sampled during the timed region
# ---------------------------------------------------------------------------
CLOCK_FIELDS = ("clocks.sm,clocks.max.sm,power.draw,utilization.gpu,clocks_event_reasons.hw_slowdown,"
                "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
                "clocks_event_reasons.sw_power_cap")


class ClockSampler:
    def __init__(self, gpu_index: int):
        self.proc = None
        self.gpu = gpu_index

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={CLOCK_FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = []
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 8:
                continue
            try:
                rows.append((float(f[0]), float(f[1]), float(f[2]), float(f[3]), f[4:8]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        busy = [r for r in rows if r[3] >= 50] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in busy for i in range(4) if r[4][i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(r[0] for r in busy), "sm_max_mhz": max(r[1] for r in rows),
                "power_w_max": max(r[2] for r in busy), "reasons": reasons, "samples": len(busy)}


# ---------------------------------------------------------------------------
# Workload state on the device
# ---------------------------------------------------------------------------
def e4m3_cache(x: torch.Tensor):
    """Input preparation for the 8-bit cache: per-tensor scale amax / 448 and
    the E4M3 codes of x / scale (torch's float8 conversion, outside the step)."""
    scale = max(float(x.abs().max()), 1e-6) / 448.0
    return (x.float() * (1.0 / scale)).to(torch.float8_e4m3fn).view(torch.uint8), scale


def int4_cache(x: torch.Tensor):
    """Input preparation for the 4-bit cache: per-row scale amax / 7 and the
    levels clamp(round(x / scale), -7, 7) + 8 packed two per byte (torch ops,
    outside the step)."""
    xf = x.float()
    scale = xf.abs().amax(dim=-1) / 7.0
    lv = torch.where(scale[..., None] > 0, torch.round(xf / scale[..., None].clamp(min=1e-30)), torch.zeros_like(xf))
    nib = (lv.clamp(-7, 7) + 8).to(torch.uint8)
    codes = nib[..., 0::2] | (nib[..., 1::2] << 4)
    return codes.contiguous(), scale.contiguous()


def make_stack(w: workloads.Workload, device, fused: bool = True, kv: str = "f16"):
    from gqa_head_folding_gb300.decode import DecodeStack
    return DecodeStack(w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim, w.max_len, w.k_pages,
                       w.dense_layers, device, w.page_size, fused=fused, kv=kv, num_layers=w.num_layers)


def build_state(w: workloads.Workload, device, seed_offset: int = 0, fused: bool = True, kv: str = "f16"):
    import gqa_head_folding_gb300 as g
    from gqa_head_folding_gb300.decode import Layer
    stack = make_stack(w, device, fused, kv)
    layers, lens = [], []
    for layer in range(w.num_layers):
        x = workloads.make_layer(w, layer, device=device,
                                 seed=workloads.layer_seed(w, layer) + seed_offset if seed_offset else None)
        L = Layer(q=x["q"], k_cache=x["k_cache"], v_cache=x["v_cache"], valid_len=x["valid_len"],
                  out=torch.empty_like(x["q"]))
        if kv == "e4m3":
            L.k_cache, L.k_scale = e4m3_cache(x["k_cache"])
            L.v_cache, L.v_scale = e4m3_cache(x["v_cache"])
            del x["k_cache"], x["v_cache"]
            if w.append or not w.layer_is_dense(layer):
                L.meta = stack.new_meta()
                prefill = x["valid_len"] - 1 if w.append else x["valid_len"]
                g.quest_update_meta_e4m3(L.k_cache, prefill, L.meta, page_size=w.page_size)
        elif kv == "int4":
            L.k_cache, L.k_scales = int4_cache(x["k_cache"])
            L.v_cache, L.v_scales = int4_cache(x["v_cache"])
            del x["k_cache"], x["v_cache"]
        elif w.append or not w.layer_is_dense(layer):
            L.meta = stack.new_meta()
            prefill = x["valid_len"] - 1 if w.append else x["valid_len"]
            g.quest_update_meta(L.k_cache, prefill, L.meta, page_size=w.page_size)
        if w.append:
            L.k_new, L.v_new, L.pos = x["k_new"], x["v_new"], x["pos"]
        layers.append(L)
        lens.append([int(v) for v in x["valid_len"].cpu()])
    torch.cuda.synchronize(device)
    return stack, layers, lens


def clone_layers(layers):
    """An independent copy of a step's device state (same values, new memory)."""
    out = []
    for L in layers:
        kw = {f.name: getattr(L, f.name) for f in dataclasses.fields(L)}
        out.append(type(L)(**{k: (v.clone() if isinstance(v, torch.Tensor) else v) for k, v in kw.items()}))
    return out


# ---------------------------------------------------------------------------
# L2 residency: a step whose distinct bytes are under 4x L2 is timed over
# several independent copies of its state, replayed in rotation, so that the
# bytes touched between two uses of one copy are at least 4x L2.
# ---------------------------------------------------------------------------
L2_FALLBACK_BYTES = 126 * 2 ** 20
MAX_COPIES = 128


def l2_bytes() -> int:
    if torch.cuda.is_available():
        n = int(getattr(torch.cuda.get_device_properties(torch.cuda.current_device()), "L2_cache_size", 0) or 0)
        if n > 0:
            return n
    return L2_FALLBACK_BYTES


def rotation_copies(bytes_per_step: int, l2: int) -> int:
    """Number of state copies n with n x bytes_per_step >= 4 x L2 (1 when one step already is)."""
    if bytes_per_step >= 4 * l2:
        return 1
    return max(1, min(MAX_COPIES, -(-4 * l2 // max(1, bytes_per_step))))


def l2_note(copies: int, bytes_per_step: int, l2: int) -> str:
    """What the timing does about L2 (copies = 0: nothing, for a working set under 4x L2)."""
    mb = bytes_per_step / 1e6
    if copies == 0:
        return f"per-step working set {mb:.1f} MB < 4x L2 ({l2 / 1e6:.1f} MB); no flush, no rotation"
    if copies <= 1:
        return f"per-step working set {mb:.1f} MB >= 4x L2 ({l2 / 1e6:.1f} MB); no flush, no rotation"
    return (f"{copies} independent copies of the step's state replayed in rotation "
            f"({copies} x {mb:.1f} MB >= 4x L2 of {l2 / 1e6:.1f} MB); no flush")


# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one launch, from one ncu
# capture of the kernel as it stands, keyed by (workload id, batch, family, KV format,
# page size). A kernel change makes its entry stale: it is then removed until the capture
# is taken again.
NCU_TRAFFIC = {(3, 1, "quest", "f16", 16): 67_763_456, (3, 1, "quest", "e4m3", 16): 33_683_968,
               (3, 1, "dense", "f16", 16): 539_990_528,
               (2, 32, "dense", "f16", 16): 179_788_800, (2, 32, "dense", "e4m3", 16): 90_756_352,
               (2, 32, "dense", "int4", 16): 50_008_576}
# The same for one prefill launch (one layer), keyed by (workload id, batch, chunk length).
PREFILL_TRAFFIC = {(3, 1, 128): 547_511_296, (3, 1, 1024): 708_610_816}


def capture(fn, device):
    s = torch.cuda.Stream(device)
    s.wait_stream(torch.cuda.current_stream(device))
    with torch.cuda.stream(s):
        fn()                                   # eager call: loads kernels, sets attributes
        torch.cuda.synchronize(device)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            fn()
    torch.cuda.current_stream(device).wait_stream(s)
    torch.cuda.synchronize(device)
    return graph


def time_rotation(graphs, reps: int, device) -> float:
    """Mean seconds per replay over `reps` replays of the graphs in rotation,
    CUDA events on the replay stream."""
    st = torch.cuda.current_stream(device)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(device)
    a.record(st)
    for i in range(reps):
        graphs[i % len(graphs)].replay()
    b.record(st)
    b.synchronize()
    return a.elapsed_time(b) / 1e3 / reps


def family_timings(stack, copies, device, reps: int) -> dict:
    """Per-call time of each family of the step's calls, each replayed alone in
    a graph (one graph per state copy, replayed in rotation)."""
    out = {}
    for name in stack.families(copies[0]):
        graphs, n = [], 0
        for layers in copies:
            fns = stack.families(layers)[name]
            n = len(fns)
            graphs.append(capture(lambda fns=fns: [fn() for fn in fns], device))
        for gr in graphs:
            gr.replay()
        out[name] = {"s_per_launch": time_rotation(graphs, reps, device) / n, "launches": n}
        del graphs
    return out


# ---------------------------------------------------------------------------
# CPU baseline: the fp64 oracle on a bounded sample, scaled to one step
# ---------------------------------------------------------------------------
def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_step_seconds(w: workloads.Workload, unit_source, lens, budget_s: float = 10.0, kv: str = "f16",
                        threads: int = 0, sample_lens=None) -> dict:
    """Time the fp64 oracle per (sequence, KV head) unit on sampled units of one
    dense and one Quest layer, on one thread and on `threads` threads (0 = every
    host core), and scale each per token to the whole step.

    unit_source(layer, b, kv_head) returns that unit's numpy arrays: q [1,G,D],
    k and v [1,1,Lmax,D] and, for a 4-bit cache, their scale rows. The oracle's
    C code runs outside the interpreter lock, so threads over units use every
    core. Half the budget goes to each of the two timings. lens[layer][b] are
    the step's valid lengths; sample_lens (default lens) those of the sampled
    units when they were drawn apart from the step's state."""
    import concurrent.futures as cf

    import numpy as np

    import oracle
    S = w.page_size
    scale = 1.0 / math.sqrt(w.head_dim)
    threads = threads or host_cores()

    def run_unit(kind, u, length):
        if kind == "dense":
            if kv == "e4m3":
                oracle.attn_e4m3(u["q"], u["k"], u["v"], u["k_scale"], u["v_scale"], [length], scale)
            elif kv == "int4":
                oracle.attn_int4(u["q"], u["k"], u["k_scales"], u["v"], u["v_scales"], [length], scale)
            else:
                oracle.attn_repeat_kv(u["q"], u["k"], u["v"], [length], scale)
            return
        e4 = kv == "e4m3"                                   # bounds and pages decoded, times the scales
        bounds = oracle.e4m3_to_f64(u["meta"]) * u["k_scale"] if e4 else u["meta"]
        sc = oracle.page_scores(u["q"], bounds, [length], S)
        if w.append:                                        # the appended token's page, rebuilt and rescored
            p = (length - 1) // S
            rows = u["k"][:, :, p * S:length]
            if e4:
                page = oracle.e4m3_to_f64(oracle.page_minmax_e4m3(rows, [rows.shape[2]], S)[:, :, :1]) * u["k_scale"]
            else:
                page = oracle.page_minmax(rows, [rows.shape[2]], S)[:, :, :1]
            sc[:, :, p] = oracle.page_scores(u["q"], page, [rows.shape[2]], S)[:, :, 0]
        idx = oracle.topk_pages(sc, [length], S, w.k_pages)
        if e4:
            oracle.sparse_attn(u["q"], oracle.e4m3_to_f64(u["k"]) * u["k_scale"],
                               oracle.e4m3_to_f64(u["v"]) * u["v_scale"], [length], idx, S, scale)
        else:
            oracle.sparse_attn(u["q"], u["k"], u["v"], [length], idx, S, scale)

    kinds = []
    for kind in ("dense", "quest"):
        ids = [i for i in range(w.num_layers) if w.layer_is_dense(i) == (kind == "dense")]
        if ids:
            kinds.append((kind, ids[0]))
    sample_lens = lens if sample_lens is None else sample_lens
    nb = min(w.batch, len(sample_lens[0]))
    units = [(b, h) for b in range(nb) for h in range(w.num_kv_heads)]
    order = [units[i] for i in np.random.default_rng(0).permutation(len(units))]
    per_tok_1, per_tok_n, sampled = {}, {}, {}
    for kind, li in kinds:
        pool = []                                           # distinct units, arrays extracted up front
        for (b, h) in order[:max(1, min(len(order), threads))]:
            u = unit_source(li, b, h)
            if kind == "quest":                              # prefill state, not timed
                u["meta"] = (oracle.page_minmax_e4m3 if kv == "e4m3" else oracle.page_minmax)(
                    u["k"], [sample_lens[li][b]], S)
            pool.append((u, sample_lens[li][b]))
        # one thread
        t_spent, toks, n1 = 0.0, 0, 0
        while n1 < 1 or (t_spent < budget_s / (2 * len(kinds)) and n1 < 4 * len(pool)):
            u, length = pool[n1 % len(pool)]
            t0 = time.perf_counter()
            run_unit(kind, u, length)
            t_spent += time.perf_counter() - t0
            toks += length
            n1 += 1
        per_tok_1[kind] = t_spent / toks
        per_unit = t_spent / n1
        # every core: enough jobs to keep each thread busy for its share of the budget
        n_jobs = max(threads, int(budget_s / (2 * len(kinds)) * threads / max(per_unit, 1e-6)))
        n_jobs = min(n_jobs, 64 * threads)
        jobs = [pool[i % len(pool)] for i in range(n_jobs)]
        with cf.ThreadPoolExecutor(max_workers=threads) as ex:
            t0 = time.perf_counter()
            list(ex.map(lambda j: run_unit(kind, j[0], j[1]), jobs))
            wall = time.perf_counter() - t0
        per_tok_n[kind] = wall / sum(j[1] for j in jobs)
        sampled[kind] = {"layer": li, "distinct_units": len(pool), "one_thread_units": n1, "all_core_units": n_jobs}

    def extrapolate(per_tok):
        return sum(per_tok["dense" if w.layer_is_dense(i) else "quest"] * w.num_kv_heads * sum(lens[i])
                   for i in range(w.num_layers))

    desc = ", ".join(f"{k}: {v['one_thread_units']} units on 1 thread and {v['all_core_units']} on {threads} "
                     f"threads, drawn from {v['distinct_units']} (sequence, KV head) units of layer {v['layer']}"
                     for k, v in sampled.items())
    return {"one_thread_s": extrapolate(per_tok_1), "all_cores_s": extrapolate(per_tok_n), "threads": threads,
            "sampled": sampled, "extrapolated": True,
            "sample": f"fp64 oracle ({desc}); time per token scaled to all {w.num_layers} layers x "
                      f"{w.batch * w.num_kv_heads} units of the step"}


def device_unit_source(layers, kv: str):
    """Units of the device state, copied to the host (outside any timing)."""
    def src(li, b, h):
        L = layers[li]
        G = L.q.shape[1] // L.k_cache.shape[1]
        u = {"q": L.q[b, h * G:(h + 1) * G].unsqueeze(0).cpu().numpy(),
             "k": L.k_cache[b, h][None, None].cpu().numpy(), "v": L.v_cache[b, h][None, None].cpu().numpy(),
             "k_scale": L.k_scale, "v_scale": L.v_scale}
        if kv == "int4":
            u["k_scales"] = L.k_scales[b, h][None, None].cpu().numpy()
            u["v_scales"] = L.v_scales[b, h][None, None].cpu().numpy()
        return u
    return src


# ---------------------------------------------------------------------------
# Arms
# ---------------------------------------------------------------------------
def workload_from_args(args) -> workloads.Workload:
    w = workloads.WORKLOADS[args.workload]
    if args.batch:
        w = w.with_(batch=args.batch)
    if args.k_pages:
        w = w.with_(k_pages=args.k_pages)
    if args.layers:
        w = w.with_(num_layers=args.layers)
    if args.page_size:
        w = w.with_(page_size=args.page_size)
    if args.budget:
        if w.k_pages is None:
            raise SystemExit("--budget applies to Quest workloads")
        w = w.with_(k_pages=max(1, args.budget // w.page_size))
    if getattr(args, "dense", False):
        w = w.with_(k_pages=None)
    return w


def config_of(w: workloads.Workload, world: int, fused: bool = True, pdl: bool = True,
              quest_kernel: str = "cluster", kv: str = "f16", early_meta: bool = False,
              early_kv: bool = False, l2: str = "") -> dict:
    return {"workload": f"{w.name} (config {w.id})", "batch_per_gpu": w.batch, "global_batch": w.batch * world,
            "layers": w.num_layers, "dense_layers": w.num_layers if w.k_pages is None else w.dense_layers,
            "num_q_heads": w.num_q_heads, "num_kv_heads": w.num_kv_heads, "head_dim": w.head_dim,
            "max_len": w.max_len, "valid_len": "full" if w.valid_lo is None else f"uniform[{w.valid_lo},{w.max_len}]",
            "page_size": w.page_size, "k_pages": w.k_pages,
            "token_budget": None if w.k_pages is None else w.k_pages * w.page_size,
            "append": w.append, "planted_pages_per_head": w.n_plant, "parallelism": f"replicas x{world}",
            "quest_path": (f"fused (quest_decode_attn, {'GPU-wide work queue' if quest_kernel == 'queue' else 'cluster per unit'})"
                           if fused else "step-by-step calls"),
            "launch": ("programmatic dependent launch" if pdl else "plain stream order")
                      + ("; Quest: first metadata tiles read before the dependency wait"
                         if early_meta and fused and w.k_pages is not None and quest_kernel == "cluster" else "")
                      + ("; dense: first K/V tiles read before the dependency wait"
                         if early_kv and (w.k_pages is None or w.dense_layers > 0) else ""),
            "kv_cache": {"e4m3": "e4m3 codes, per-tensor fp32 scales",
                         "int4": "int4 levels, per-token fp32 scales"}.get(kv, "f16"),
            "l2": l2}


def arm_config(args, w: workloads.Workload, world: int) -> dict:
    """The config dict both arms print for this command line."""
    lens = [[int(v) for v in workloads.valid_lengths(w, i)] for i in range(w.num_layers)]
    nbytes = step_bytes(w, lens, fused=not args.unfused, kv=args.kv)["total"]
    l2 = l2_bytes()
    return config_of(w, world, fused=not args.unfused, pdl=not args.no_pdl, quest_kernel=args.quest_kernel,
                     kv=args.kv, early_meta=not args.no_early_meta, early_kv=not args.no_early_kv,
                     l2=l2_note(rotation_copies(nbytes, l2), nbytes, l2))


def run_reference(args, rank, world):
    """The fp64 CPU oracle as it stands, on the host cores, on this workload.

    Inputs are drawn on the host (the same seeded recipe, a host generator) for
    the sampled sequences of one dense and one Quest layer; the page metadata
    comes from the oracle's own min/max. Nothing here loads the CUDA library."""
    if rank != 0:
        return
    w = workload_from_args(args)
    lens = [[int(v) for v in workloads.valid_lengths(w, i)] for i in range(w.num_layers)]
    w_host = w.with_(batch=min(w.batch, 2))              # sampled sequences only
    drawn = {}

    def unit_source(li, b, h):
        if li not in drawn:
            x = workloads.make_layer(w_host, li, device="cpu")
            if args.kv == "e4m3":
                x["k_cache"], x["k_scale"] = e4m3_cache(x["k_cache"])
                x["v_cache"], x["v_scale"] = e4m3_cache(x["v_cache"])
            elif args.kv == "int4":
                x["k_cache"], x["k_scales"] = int4_cache(x["k_cache"])
                x["v_cache"], x["v_scales"] = int4_cache(x["v_cache"])
            drawn[li] = x
        x = drawn[li]
        G = w.group
        u = {"q": x["q"][b, h * G:(h + 1) * G].unsqueeze(0).numpy(), "k": x["k_cache"][b, h][None, None].numpy(),
             "v": x["v_cache"][b, h][None, None].numpy(), "k_scale": x.get("k_scale", 1.0),
             "v_scale": x.get("v_scale", 1.0)}
        if args.kv == "int4":
            u["k_scales"] = x["k_scales"][b, h][None, None].numpy()
            u["v_scales"] = x["v_scales"][b, h][None, None].numpy()
        return u

    host_lens = [[int(v) for v in workloads.valid_lengths(w_host, i)] for i in range(w.num_layers)]
    per_step, one = [], []
    r = None
    for i in range(args.warmup + args.steps):
        r = oracle_step_seconds(w, unit_source, lens, budget_s=args.ref_budget, kv=args.kv, sample_lens=host_lens)
        if i >= args.warmup:
            per_step.append(r["all_cores_s"])
            one.append(r["one_thread_s"])
    value = statistics.mean(per_step) * 1e6
    sb = step_bytes(w, lens, kv=args.kv)
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": value / 1e3, "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (host-drawn, same recipe)",
            "config": arm_config(args, w, 1),
            "achieved_gbs": round(sb["total"] / (value / 1e6) / 1e9, 3),
            "cpu_baseline": {"value": round(value, 1), "unit": UNIT, "cores": r["threads"], "kind": "oracle",
                             "sample": r["sample"], "extrapolated": True, "sampled": r["sampled"],
                             "one_thread": {"value": round(statistics.mean(one) * 1e6, 1), "unit": UNIT, "cores": 1}},
            "e2e": {"value": round(value, 1), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


NOMINAL_HBM_GBS = 7900.0     # GB300 HBM3e, nominal


def load_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": float(d["hbm_gbs"]), "tensor_tflops": float(d.get("bf16_tflops_sustained", 1700.0)),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "tensor_tflops": 1700.0, "source": "fallback"}


# ---------------------------------------------------------------------------
# Prefill mode: a chunk of q_len new tokens per sequence and layer
# ---------------------------------------------------------------------------
PREFILL_METRIC = "prefill-attn us/step (causal chunk of q_len tokens per sequence per layer) and achieved vs the binding roofline (tensor or HBM)"


def prefill_flops(w: workloads.Workload, starts, q_len: int) -> int:
    """q.k and p.V multiply-adds of one layer: 2 x 2 D flops per (row, attended token)."""
    return sum(4 * w.head_dim * w.num_q_heads * (q_len * s + q_len * (q_len + 1) // 2) for s in starts)


def prefill_roofline(flops: int, nbytes: int, s_per_launch: float, peaks: dict, traffic=None) -> dict:
    """The roofline that binds one prefill launch: tensor when its arithmetic
    intensity (flops per byte of K, V, q and out) reaches the ridge of the two
    measured peaks, HBM below it (a short chunk over a long context reads far
    more K/V per flop). Both fractions are reported; `frac` is the binding one."""
    tflops = flops / s_per_launch / 1e12
    gbs = nbytes / s_per_launch / 1e9
    t_frac = tflops / peaks["tensor_tflops"]
    h_frac = gbs / peaks["hbm_gbs"]
    ridge = peaks["tensor_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9)  # flops per byte
    intensity = flops / max(1, nbytes)
    tensor = intensity >= ridge
    return {"bound": "tensor" if tensor else "hbm", "kernel": "gqa_prefill_attn",
            "achieved": round(tflops if tensor else gbs, 1), "peak": peaks["tensor_tflops"] if tensor else peaks["hbm_gbs"],
            "unit": "TFLOP/s" if tensor else "GB/s", "frac": round(t_frac if tensor else h_frac, 4),
            "peak_source": peaks["source"] + (" (bf16 sustained; fp16 has the same nominal rate)" if tensor
                                              else " (device-to-device copy)"),
            "traffic": traffic, "flops_per_launch": flops, "bytes_per_launch": nbytes,
            "intensity_flops_per_byte": round(intensity, 1), "ridge_flops_per_byte": round(ridge, 1),
            "tensor_tflops": round(tflops, 1), "tensor_frac": round(t_frac, 4),
            "hbm_gbs": round(gbs, 1), "hbm_frac": round(h_frac, 4),
            "us_per_launch": round(s_per_launch * 1e6, 2)}


def prefill_bytes(w: workloads.Workload, starts, q_len: int) -> int:
    """K and V rows read once per KV head (2 M per token), plus q in and out."""
    M = kv_vector_bytes(w.head_dim)
    return sum(w.num_kv_heads * 2 * M * (s + q_len) + 2 * w.num_q_heads * q_len * M for s in starts)


def run_prefill(args, rank, world, local):
    import gqa_head_folding_gb300 as g
    device = torch.device(f"cuda:{local}")
    torch.cuda.set_device(device)
    dist = init_dist(world, "nccl")
    w = workload_from_args(args)
    Q = int(args.prefill)
    g.lib()
    g.set_option(g.GQAQ_OPT_PDL, 0 if args.no_pdl else 1)
    layers = []
    for layer in range(w.num_layers):
        x = workloads.make_prefill_layer(w, layer, Q, device=device,
                                         seed=workloads.layer_seed(w, layer) + rank_seed(rank) if rank else None)
        x["out"] = torch.empty_like(x["q"])
        layers.append(x)
    starts = [[int(v) for v in x["start"].cpu()] for x in layers]
    dims = g.make_dims(w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim, w.max_len)
    ws = g.alloc_prefill_workspace(dims, Q, device)
    scale = 1.0 / math.sqrt(w.head_dim)

    def step():
        for x in layers:
            g.gqa_prefill_attn(x["q"], x["k_cache"], x["v_cache"], x["start"], scale, out=x["out"], workspace=ws)

    graph = capture(step, device)
    for _ in range(max(3, args.warmup)):
        graph.replay()
    torch.cuda.synchronize(device)
    sampler = ClockSampler(local)
    sampler.start()
    t_soak = time.perf_counter()
    while time.perf_counter() - t_soak < args.soak:
        graph.replay()
        torch.cuda.synchronize(device)
    st = torch.cuda.current_stream(device)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(dist)
    torch.cuda.synchronize(device)
    ev0.record(st)
    for _ in range(args.steps):
        graph.replay()
    ev1.record(st)
    torch.cuda.synchronize(device)
    barrier(dist)
    clocks = sampler.stop()
    s_per_step = max_over_ranks(ev0.elapsed_time(ev1) / 1e3 / args.steps, dist, device)
    assert g.device_status() == 0, "prefill raised a device status flag"

    # end to end: q in from pinned host memory, out back, every step
    h_q = [torch.empty(x["q"].shape, dtype=x["q"].dtype, pin_memory=True).copy_(x["q"].cpu()) for x in layers]
    h_o = [torch.empty(x["out"].shape, dtype=x["out"].dtype, pin_memory=True) for x in layers]
    e2e_steps = max(3, min(args.steps, 20))
    torch.cuda.synchronize(device)
    barrier(dist)
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        for x, hq in zip(layers, h_q):
            x["q"].copy_(hq, non_blocking=True)
        graph.replay()
        for x, ho in zip(layers, h_o):
            ho.copy_(x["out"], non_blocking=True)
        torch.cuda.synchronize(device)
    e2e_s = max_over_ranks((time.perf_counter() - t0) / e2e_steps, dist, device)
    if rank != 0:
        return
    peaks = load_peaks()
    flops = sum(prefill_flops(w, s, Q) for s in starts)
    per_launch_flops = prefill_flops(w, starts[0], Q)
    per_launch_bytes = prefill_bytes(w, starts[0], Q)
    achieved = flops / s_per_step / 1e12
    cpu = None
    if not args.no_cpu_baseline:
        import numpy as np

        import oracle
        x = layers[0]
        t0 = time.perf_counter()
        oracle.prefill_attn(x["q"][:1, :w.group].cpu().numpy(), x["k_cache"][:1, :1].cpu().numpy(),
                            x["v_cache"][:1, :1].cpu().numpy(), starts[0][:1], scale)
        unit_s = time.perf_counter() - t0
        unit_flops = prefill_flops(w.with_(num_q_heads=w.group, num_kv_heads=1), starts[0][:1], Q)
        est = unit_s * flops / max(1, unit_flops)
        cpu = {"value": round(est * 1e6, 1), "unit": UNIT, "cores": 1, "kind": "oracle",
               "sample": f"fp64 oracle on one (sequence, KV head) unit of layer 0 ({w.group} query heads x {Q} "
                         f"tokens), scaled by flops to the whole step"}
        del np
    line = {
        "metric": PREFILL_METRIC, "value": round(s_per_step * 1e6, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": s_per_step * 1e3, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16 in/out, f32 accumulate",
        "data": "synthetic (seeded N(0,1) fp16 q and caches)",
        "config": dict(config_of(w, world, pdl=not args.no_pdl,
                                 l2=l2_note(1 if per_launch_bytes >= 4 * l2_bytes() else 0, per_launch_bytes,
                                            l2_bytes())), q_len=Q,
                       chunk="last q_len tokens of each sequence's valid length"),
        "achieved_tflops": round(achieved, 1),
        "roofline": prefill_roofline(per_launch_flops, per_launch_bytes, s_per_step / w.num_layers, peaks,
                                     PREFILL_TRAFFIC.get((w.id, w.batch, Q))),
        "achieved_gbs": round(sum(prefill_bytes(w, s, Q) for s in starts) / s_per_step / 1e9, 1),
        "cpu_baseline": cpu,
        "e2e": {"value": round(e2e_s * 1e6, 2), "unit": UNIT,
                "h2d_bytes_per_step": sum(h.numel() * h.element_size() for h in h_q),
                "d2h_bytes_per_step": sum(h.numel() * h.element_size() for h in h_o)},
        "gpu_launches": w.num_layers * args.steps, "gpu_launches_per_step": w.num_layers,
        "clocks": clocks,
    }
    print(json.dumps(line))


FAMILY_KERNEL = {"dense": "gqa_decode_attn", "score": "quest_score_pages", "sparse": "quest_sparse_attn",
                 "quest": "quest_decode_attn"}  # "_e4m3" appended for the 8-bit cache


def measure(w: workloads.Workload, stack, copies, lens, device, steps: int, warmup: int, kv: str = "f16",
            fused: bool = True, dist=None, soak: float = 0.0, sampler=None, reps: int = 50) -> dict:
    """Time `steps` graph replays of one full step (state copies in rotation),
    then each call family alone; return the step time and the roofline of the
    dominant family."""
    sb = step_bytes(w, lens, fused=fused, kv=kv)
    graphs = [capture(lambda ls=ls: stack.step(ls), device) for ls in copies]
    for i in range(max(3, warmup)):
        graphs[i % len(graphs)].replay()
    torch.cuda.synchronize(device)
    if sampler is not None:
        sampler.start()
    t_soak = time.perf_counter()
    i = 0
    while time.perf_counter() - t_soak < soak:
        for _ in range(8):
            graphs[i % len(graphs)].replay()
            i += 1
        torch.cuda.synchronize(device)
    # timed region: exactly `steps` steps
    st = torch.cuda.current_stream(device)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(dist)
    torch.cuda.synchronize(device)
    ev0.record(st)
    for i in range(steps):
        graphs[i % len(graphs)].replay()
    ev1.record(st)
    torch.cuda.synchronize(device)
    barrier(dist)
    clocks = sampler.stop() if sampler is not None else None
    s_per_step = max_over_ranks(ev0.elapsed_time(ev1) / 1e3 / steps, dist, device)
    del graphs

    fam = family_timings(stack, copies, device, reps=max(3, min(reps, steps)))
    per_step_fam = {k: v["s_per_launch"] * sb["launches"][k] for k, v in fam.items()}
    dominant = max(per_step_fam, key=per_step_fam.get)
    peaks = load_peaks()
    roof = None
    if dominant in FAMILY_KERNEL:
        layer_of = next(i for i in range(w.num_layers)
                        if (stack.is_dense(i) if dominant == "dense" else not stack.is_dense(i)))
        per_launch = roofline_unit_bytes(w, dominant, lens[layer_of], kv=kv)
        achieved = per_launch / fam[dominant]["s_per_launch"] / 1e9
        roof = {"bound": "hbm", "kernel": FAMILY_KERNEL[dominant] + ("" if kv == "f16" else "_" + kv),
                "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(achieved / peaks["hbm_gbs"], 4), "peak_source": peaks["source"] + " copy bandwidth",
                "frac_of_nominal": round(achieved / NOMINAL_HBM_GBS, 4), "nominal_peak": NOMINAL_HBM_GBS,
                "traffic": NCU_TRAFFIC.get((w.id, w.batch, dominant, kv, w.page_size)),
                "bytes_per_launch": per_launch, "us_per_launch": round(fam[dominant]["s_per_launch"] * 1e6, 2)}
    return {"s_per_step": s_per_step, "bytes": sb, "fam": fam, "per_step_fam": per_step_fam, "roofline": roof,
            "clocks": clocks, "peaks": peaks}


# Other workloads measured in the same process for the `by_config` object of the
# default line: (label, workload id, overrides, variants on the same caches).
# A variant is a k_pages value, or None for every layer dense.
BY_CONFIG = [
    ("config 1: EXAONE shape, 1 dense layer, batch 1", 1, {}, ["as-is"]),
    ("config 2: EXAONE shape, 30 dense layers, batch 1", 2, {"batch": 1}, ["as-is"]),
    ("config 2: EXAONE shape, 30 dense layers, batch 32", 2, {"batch": 32}, ["as-is"]),
    ("config 4: GQA Quest 64K, K=256, batch 1", 4, {"batch": 1}, ["as-is", None]),
    ("config 4: GQA Quest 64K, K=256, batch 4", 4, {"batch": 4}, ["as-is"]),
    ("config 4: GQA Quest 64K, K=256, batch 8", 4, {"batch": 8}, ["as-is", None]),
    ("config 5: 128K, batch 1", 5, {"batch": 1}, [128, 512, None]),
    ("config 5: 128K, batch 16", 5, {"batch": 16}, [128, 512, None]),
    ("config 3 over an E4M3 cache: Llama-2-7B shape, 32 layers, 32K, K=128", 3, {"kv": "e4m3"}, ["as-is"]),
]


def run_by_config(args, device) -> dict:
    """Each BY_CONFIG workload: state built once, its variants timed on the same caches."""
    out = {"entries": [], "steps": args.by_config_steps, "warmup": 3}
    sampler = ClockSampler(device.index or 0)
    sampler.start()
    t0 = time.perf_counter()
    l2 = l2_bytes()
    for label, wid, over, variants in BY_CONFIG:
        over = dict(over)
        kv = over.pop("kv", "f16")
        fused = True
        base = workloads.WORKLOADS[wid].with_(**over)
        stack0, layers, lens = build_state(base, device, fused=fused, kv=kv)
        del stack0
        nbytes_min = min(step_bytes(base if v == "as-is" else base.with_(k_pages=v), lens, fused=fused, kv=kv)["total"]
                         for v in variants)
        n = rotation_copies(nbytes_min, l2)
        copies = [layers] + [clone_layers(layers) for _ in range(n - 1)]
        for v in variants:
            w = base if v == "as-is" else base.with_(k_pages=v)
            stack = make_stack(w, device, fused=fused, kv=kv)
            m = measure(w, stack, copies, lens, device, args.by_config_steps, 3, kv=kv, fused=fused)
            nb = m["bytes"]["total"]
            e = {"label": label + ("" if v == "as-is" else (", all dense" if v is None else f", K={v}")),
                 "workload": w.name, "config_id": w.id, "batch": w.batch, "layers": w.num_layers, "kv_cache": kv,
                 "k_pages": w.k_pages, "us_per_step": round(m["s_per_step"] * 1e6, 2), "bytes_per_step": nb,
                 "gbs_step": round(nb / m["s_per_step"] / 1e9, 1),
                 "frac_step": round(nb / m["s_per_step"] / 1e9 / m["peaks"]["hbm_gbs"], 4),
                 "us_per_launch_by_family": {k: round(f["s_per_launch"] * 1e6, 2) for k, f in m["fam"].items()},
                 "l2": l2_note(n, nb, l2)}
            if m["roofline"]:
                r = m["roofline"]
                e["dominant"] = {"kernel": r["kernel"], "us_per_launch": r["us_per_launch"],
                                 "bytes_per_launch": r["bytes_per_launch"], "achieved_gbs": r["achieved"],
                                 "frac": r["frac"], "frac_of_nominal": r["frac_of_nominal"],
                                 "traffic": r["traffic"]}
            out["entries"].append(e)
            del stack
        del copies, layers
        torch.cuda.synchronize(device)
        torch.cuda.empty_cache()
    out["clocks"] = sampler.stop()
    out["seconds"] = round(time.perf_counter() - t0, 1)
    return out


def run_ours(args, rank, world, local):
    import gqa_head_folding_gb300 as g
    device = torch.device(f"cuda:{local}")
    torch.cuda.set_device(device)
    dist = init_dist(world, "nccl")
    w = workload_from_args(args)
    g.lib()
    g.set_option(g.GQAQ_OPT_PDL, 0 if args.no_pdl else 1)
    # every Quest call in the step follows another layer's call, which writes
    # none of this layer's metadata, valid_len or pos
    g.set_option(g.GQAQ_OPT_QUEST_EARLY_META, 0 if args.no_early_meta else 1)
    # and every dense call follows its own layer's append (or another layer's
    # call), which writes no cache row but the appended one
    g.set_option(g.GQAQ_OPT_DENSE_EARLY_KV, 0 if args.no_early_kv else 1)
    if args.quest_kernel == "queue":
        g.set_option(g.GQAQ_OPT_QUEST_KERNEL, 2)
    fused = not args.unfused
    stack, layers, lens = build_state(w, device, seed_offset=rank_seed(rank), fused=fused, kv=args.kv)
    l2 = l2_bytes()
    nbytes = step_bytes(w, lens, fused=fused, kv=args.kv)["total"]
    n_copies = rotation_copies(nbytes, l2)
    copies = [layers] + [clone_layers(layers) for _ in range(n_copies - 1)]
    m = measure(w, stack, copies, lens, device, args.steps, args.warmup, kv=args.kv, fused=fused, dist=dist,
                soak=args.soak, sampler=ClockSampler(local))
    s_per_step, sb = m["s_per_step"], m["bytes"]

    # end to end through the public API: host inputs in, host outputs out, every step
    graphs = [capture(lambda ls=ls: stack.step(ls), device) for ls in copies]
    xfers = []
    for ls in copies:
        h2d = [(L.q, torch.empty(L.q.shape, dtype=L.q.dtype, pin_memory=True)) for L in ls]
        if w.append:
            h2d += [(t, torch.empty(t.shape, dtype=t.dtype, pin_memory=True)) for L in ls for t in (L.k_new, L.v_new)]
        for dst, src in h2d:
            src.copy_(dst.cpu())
        d2h = [(L.out, torch.empty(L.out.shape, dtype=L.out.dtype, pin_memory=True)) for L in ls]
        xfers.append((h2d, d2h))
    h2d_bytes = sum(s.numel() * s.element_size() for _, s in xfers[0][0])
    d2h_bytes = sum(d.numel() * d.element_size() for _, d in xfers[0][1])
    e2e_steps = max(3, args.steps)
    torch.cuda.synchronize(device)
    barrier(dist)
    t0 = time.perf_counter()
    for i in range(e2e_steps):
        h2d, d2h = xfers[i % len(xfers)]
        for dst, src in h2d:
            dst.copy_(src, non_blocking=True)
        graphs[i % len(graphs)].replay()
        for src, dst in d2h:
            dst.copy_(src, non_blocking=True)
        torch.cuda.synchronize(device)
    e2e_s = max_over_ranks((time.perf_counter() - t0) / e2e_steps, dist, device)
    barrier(dist)
    del graphs
    assert g.device_status() == 0, "the step raised a device status flag"

    if rank != 0:
        return
    cpu = None
    if not args.no_cpu_baseline:
        r = oracle_step_seconds(w, device_unit_source(layers, args.kv), lens, budget_s=args.cpu_budget, kv=args.kv)
        cpu = {"value": round(r["all_cores_s"] * 1e6, 1), "unit": UNIT, "cores": r["threads"], "kind": "oracle",
               "sample": r["sample"], "extrapolated": True, "sampled": r["sampled"],
               "one_thread": {"value": round(r["one_thread_s"] * 1e6, 1), "unit": UNIT, "cores": 1}}
    launches = stack.launches_per_step(layers)
    del copies, layers, stack
    torch.cuda.synchronize(device)
    torch.cuda.empty_cache()
    by_config = None
    if world == 1 and args.by_config:
        by_config = run_by_config(args, device)
    peaks = m["peaks"]
    total_bytes = sb["total"] * world
    line = {
        "metric": METRIC, "value": round(s_per_step * 1e6, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": s_per_step * 1e3,
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
        "dtype": "f16 in/out, " + ({"e4m3": "e4m3 KV cache, ", "int4": "int4 KV cache, "}.get(args.kv, "")) +
                 "f32 accumulate",
        "data": "synthetic (seeded N(0,1) fp16 caches, planted pages)",
        "config": arm_config(args, w, world),
        "achieved_gbs": round(total_bytes / s_per_step / 1e9, 1),
        "achieved_frac_of_peak": round(sb["total"] / s_per_step / 1e9 / peaks["hbm_gbs"], 4),
        "achieved_frac_of_nominal": round(sb["total"] / s_per_step / 1e9 / NOMINAL_HBM_GBS, 4),
        "bytes_per_step": total_bytes,
        "bytes_by_family": sb["bytes"],
        "us_per_launch_by_family": {k: round(v["s_per_launch"] * 1e6, 2) for k, v in m["fam"].items()},
        "us_per_step_by_family": {k: round(v * 1e6, 2) for k, v in m["per_step_fam"].items()},
        "timing": "mean over the timed steps (CUDA events around all of them)",
        "roofline": m["roofline"],
        "cpu_baseline": cpu,
        "e2e": {"value": round(e2e_s * 1e6, 2), "unit": UNIT, "h2d_bytes_per_step": h2d_bytes,
                "d2h_bytes_per_step": d2h_bytes},
        "gpu_launches": launches * args.steps,
        "gpu_launches_per_step": launches,
        "clocks": m["clocks"],
    }
    if by_config is not None:
        line["by_config"] = by_config
    print(json.dumps(line))


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", type=int, default=3, choices=sorted(workloads.WORKLOADS))
    ap.add_argument("--batch", type=int, default=0)
    ap.add_argument("--k-pages", type=int, default=0)
    ap.add_argument("--dense", action="store_true",
                    help="run every layer dense on the same caches (the dense side of a Quest workload)")
    ap.add_argument("--layers", type=int, default=0)
    ap.add_argument("--page-size", type=int, default=0, choices=(0, 8, 16, 32, 64),
                    help="Quest page size S (tokens); 0 = the workload's (16)")
    ap.add_argument("--budget", type=int, default=0,
                    help="Quest token budget; sets k_pages = budget / S (page-size sweep at a fixed budget)")
    ap.add_argument("--soak", type=float, default=1.5, help="seconds of untimed replays before timing")
    ap.add_argument("--ref-budget", type=float, default=3.0,
                    help="seconds of oracle work per step of --impl reference")
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--by-config", dest="by_config", action="store_true", default=None,
                    help="also time the other workloads in the same process (default: on for the default workload)")
    ap.add_argument("--no-by-config", dest="by_config", action="store_false")
    ap.add_argument("--by-config-steps", type=int, default=50)
    ap.add_argument("--unfused", action="store_true", help="run Quest layers as the step-by-step calls")
    ap.add_argument("--quest-kernel", choices=("queue", "cluster"), default="cluster",
                    help="fused Quest kernel: one cluster per unit (default) or the GPU-wide work queue")
    ap.add_argument("--no-pdl", action="store_true", help="launch without programmatic stream serialization")
    ap.add_argument("--no-early-meta", action="store_true",
                    help="fused Quest kernel: read no metadata before the wait on the previous kernel")
    ap.add_argument("--no-early-kv", action="store_true",
                    help="dense attention: read no K/V tile before the wait on the previous kernel")
    ap.add_argument("--prefill", type=int, default=0,
                    help="time gqa_prefill_attn on a chunk of this many tokens per sequence and layer instead")
    ap.add_argument("--kv", choices=("f16", "e4m3", "int4"), default="f16",
                    help="KV-cache format; e4m3 (8-bit codes and page bounds, per-tensor scales) or int4 (4-bit "
                         "levels, per-token scales; all-dense stacks only)")
    args = ap.parse_args(argv)
    if args.by_config is None:
        args.by_config = default_command(args)
    if args.kv == "int4":
        w = workload_from_args(args)
        if any(not w.layer_is_dense(i) for i in range(w.num_layers)):
            raise SystemExit("--kv int4 needs a stack of dense layers only (e.g. --workload 2, or --layers 2)")
    rank, world, local = dist_env()
    if args.prefill and args.impl == "ours":
        run_prefill(args, rank, world, local)
    elif args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world, local)


def default_command(args) -> bool:
    """True when the command line picks the default workload with no overrides."""
    return (args.workload == 3 and not (args.batch or args.k_pages or args.layers or args.page_size or args.budget
                                        or args.dense or args.unfused or args.prefill or args.kv != "f16"
                                        or args.quest_kernel != "cluster"))


if __name__ == "__main__":
    main()
