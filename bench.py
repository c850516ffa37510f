"""Benchmark of the DSA lightning-indexer step on GB300.

Headline workload: long-context decode -- 4 requests with 1,048,576 cached
tokens and one new token each, H = 64 indexer heads, index_topk = 2048, a
78-layer stack with 21 F layers (explicit seeded pattern).  One step = one
pass of the whole path over the batch: for every F layer, write the new keys
into the paged FP8 cache, score every query row against its request's cached
keys, select the top-k into the shared buffer (S layers launch nothing).
Metric: query-key pairs per second (sum over F layers of the keys each query
row sees, divided by step time).  `per_config` repeats the measurement on
every workload of the suite (tiny prefill, batched decode, prefix-hit
chunked prefill, mixed batch, long-context decode), each at full size.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload ID] [--configs 0,1,2,3,4|none]

`--impl reference` times the FP64 CPU oracle (the correctness reference) on a
bounded sample of the same workload, on this machine's host cores.
`--gpus N` (N > 1) starts N ranks itself unless it already runs under a
launcher; each rank runs its own batch (weak scaling, no data-path
collective) and rank 0 prints one JSON line.
"""

from __future__ import annotations

import argparse
import csv
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time
from pathlib import Path

ROOT = Path(__file__).resolve().parent
if str(ROOT) not in sys.path:
    sys.path.insert(0, str(ROOT))

import numpy as np  # noqa: E402

import synth  # noqa: E402

METRIC = "DSA indexer score+top-k query-key pairs/s; % of HBM / FP8 roofline"
UNIT = "pairs/s"
BYTES_PER_PAIR = 132 + 4 / 64          # FP8 key + FP32 scale + its share of a block-table entry
L2_FLUSH_BYTES = 256 << 20             # larger than the 129 MB L2
KERNEL_SOURCES = ["score_topk.cuh", "ptx.cuh", "plan.cuh", "kwrite.cuh"]


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", type=int, default=None,
                    help="headline workload id (default 4 = long-context decode)")
    ap.add_argument("--configs", default="0,1,2,3,4",
                    help="workloads measured for per_config (comma list, or 'none')")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--scale", type=float, default=1.0,
                    help="context/row scale of the workload (1 = its stated size; smaller for "
                         "profiling captures)")
    ap.add_argument("--no-graph", action="store_true")
    ap.add_argument("--cpu-budget-s", type=float, default=10.0)
    ap.add_argument("--cpu-budget-per-config-s", type=float, default=4.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--bf16", action="store_true",
                    help="BF16 keys and queries, quantised by the cache-write launch")
    ap.add_argument("--sparse-mla", action="store_true",
                    help="time the consumer instead: sparse MLA attention of every query row over "
                         "its top-k tokens (record write + attention per F layer)")
    ap.add_argument("--mla-heads", type=int, default=128)
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def reduce_over_ranks(times_ms, units, world: int, device=None):
    """Whole-job figures of a replicated run: each time is the maximum over
    the ranks (the job ends with its slowest replica), the units processed are
    summed over the ranks.  With one rank the inputs come back unchanged.  Works
    on any initialised process group (NCCL on GPUs, gloo on CPUs)."""
    times_ms = [float(x) for x in times_ms]
    if world == 1:
        return times_ms, float(units)
    import torch
    import torch.distributed as dist
    t = torch.tensor(times_ms, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    u = torch.tensor([float(units)], dtype=torch.float64, device=device)
    dist.all_reduce(u)
    return t.tolist(), u.item()


def read_peaks() -> dict:
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        d = json.loads(p.read_text())
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


def _code_only(text: str) -> str:
    """Source text without comments and with whitespace collapsed, so that an
    edit to comments or layout leaves the hash (and the counters taken on the
    same code) valid."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        text = (ROOT / "dsa_sparse_attention_fp8_gb300" / "csrc" / name).read_text()
        h.update(_code_only(text).encode())
    return h.hexdigest()[:16]


def profiled_traffic(workload_name: str):
    """DRAM bytes per scoring launch from the committed ncu summary, if it was
    taken on the current kernel source; else None."""
    p = ROOT / "profiles" / f"score_topk_{workload_name}.md"
    if not p.exists():
        return None
    text = p.read_text()
    m_b = re.search(r"dram_bytes_per_launch:\s*([0-9]+)", text)
    m_h = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]+)", text)
    if not m_b or not m_h or m_h.group(1) != kernel_source_hash():
        return None
    return int(m_b.group(1))


class ClockSampler:
    """nvidia-smi clock / throttle sampling while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.file = tempfile.NamedTemporaryFile(mode="w+", suffix=".csv", delete=False)

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.file, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except FileNotFoundError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self) -> dict:
        self.file.flush()
        rows = []
        try:
            with open(self.file.name) as f:
                for r in csv.reader(f):
                    if len(r) >= 9:
                        rows.append([x.strip() for x in r])
        finally:
            os.unlink(self.file.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows)}


# ----------------------------------------------------------------------------
# CPU oracle legs
# ----------------------------------------------------------------------------

def oracle_sample_setup(wl, layer=0, requests=None):
    """Oracle state for timing (not timed): the page pool holding the cached
    prefix of the given requests (all by default), the step's keys and
    quantised queries."""
    import oracle as O
    cache = np.zeros((wl.num_pages, O.PAGE_BYTES), np.uint8)
    for r in (range(wl.R) if requests is None else sorted(set(requests))):
        E = int(wl.prefix_entries[r])
        if E:
            O.write_k_cache(cache, wl.k_prefix(layer, r),
                            O.slot_mapping(np.array([0, E]), np.array([E]), wl.block_table[r:r + 1]))
    qc, qs = O.quantize_blocks(wl.q(layer))
    return cache, wl.k_new(layer), qc, qs, wl.w(layer)


def oracle_time_rows(wl, state, rows):
    """Time one oracle indexer layer (key write + scores + full sort) on `rows`."""
    import oracle as O
    cache, k_new, qc, qs, w = state
    buf = np.full((wl.max_num_batched_tokens, wl.index_topk), -1, np.int32)
    c = cache.copy()
    t0 = time.perf_counter()
    O.indexer_layer(c, k_new, qc, qs, w, wl.query_start_loc, wl.seq_lens, wl.block_table,
                    wl.index_topk, buf, rows=rows, compress_ratio=wl.compress_ratio)
    dt = time.perf_counter() - t0
    _, pos = O.token_positions(wl.query_start_loc, wl.seq_lens)
    pairs = int(sum(int(O.visible_entries(pos[t], wl.compress_ratio)) for t in rows))
    return pairs, dt


def sample_rows(wl, max_pairs: int = 4_000_000):
    """Query rows in order from row 0, as many as keep the sample's pairs (and
    so its oracle time) bounded, at least one; and their requests."""
    import oracle as O
    req, pos = O.token_positions(wl.query_start_loc, wl.seq_lens)
    rows, pairs = [], 0
    for t in range(wl.T):
        n = int(O.visible_entries(pos[t], wl.compress_ratio))
        if rows and pairs + n > max_pairs:
            break
        rows.append(t)
        pairs += n
    return rows, sorted({int(req[t]) for t in rows})


def cpu_cores() -> int:
    return len(os.sched_getaffinity(0))


def cpu_baseline(wl, budget_s: float) -> dict:
    """The oracle on layer 0 of the same workload, on a bounded prefix of its
    query rows (see sample_rows), repeated in chunks until about `budget_s`
    seconds of CPU work are done."""
    rows, reqs = sample_rows(wl)
    state = oracle_sample_setup(wl, requests=reqs)
    done_pairs, done_s, n = 0, 0.0, 0
    chunk = max(1, len(rows) // 16)
    while done_s < budget_s:
        a = n % len(rows)
        sel = rows[a:a + chunk]
        p, dt = oracle_time_rows(wl, state, sel)
        done_pairs += p
        done_s += dt
        n += len(sel)
    return {"value": done_pairs / done_s, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
            "sample": f"layer 0, {n} query rows cycling over rows 0..{len(rows) - 1} of the "
                      f"{wl.T}-row batch ({done_pairs} pairs, {done_s:.1f} s; numpy FP64, BLAS "
                      f"threads per the host default)"}


def run_reference(args, wl):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    rows, reqs = sample_rows(wl, max_pairs=1_200_000)
    state = oracle_sample_setup(wl, requests=reqs)
    rows = rows[:8]
    for _ in range(args.warmup):
        oracle_time_rows(wl, state, rows)
    pairs = secs = 0.0
    for _ in range(args.steps):
        p, dt = oracle_time_rows(wl, state, rows)
        pairs += p
        secs += dt
    value = pairs / secs
    sample = (f"layer 0, query rows 0..{len(rows) - 1} of {wl.T} per step "
              f"({int(pairs / max(1, args.steps))} pairs per step)")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * secs / max(1, args.steps),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": wl.name, **{k: v for k, v in wl.describe().items()
                                                                if k != "workload"}},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------
# Sparse MLA leg (the consumer of the top-k rows)
# ----------------------------------------------------------------------------

MLA_METRIC = "sparse MLA attention (row, selected token) pairs/s; % of BF16 tensor roofline"
MLA_UNIT = "pairs/s"


def mla_oracle_rows(wl, heads, scale, budget_s):
    """The FP64 oracle on layer 0's rows in order until about budget_s seconds."""
    import oracle as O
    cache = np.zeros((wl.num_pages, O.MLA_PAGE_BYTES), np.uint8)
    for r in range(wl.R):
        P = int(wl.prefix_lens[r])
        if P:
            O.mla_write_kv_cache(cache, wl.mla_kv_prefix(0, r),
                                 O.slot_mapping(np.array([0, P]), np.array([P]),
                                                wl.block_table[r:r + 1]))
    O.mla_write_kv_cache(cache, wl.mla_kv_new(0),
                         O.slot_mapping(wl.query_start_loc, wl.seq_lens, wl.block_table))
    q = wl.mla_q(0, heads).astype(np.float64)
    topk = wl.selection_rows(0)
    pairs, secs, n = 0, 0.0, 0
    while secs < budget_s:
        t = n % wl.T
        t0 = time.perf_counter()
        O.sparse_mla_attention(q, cache, wl.query_start_loc, wl.seq_lens, wl.block_table, topk,
                               scale, rows=[t])
        secs += time.perf_counter() - t0
        pairs += int(np.sum(topk[t] >= 0))
        n += 1
    return pairs, secs, n


def run_sparse_mla(args, wl):
    import math
    import torch
    from dsa_sparse_attention_fp8_gb300 import _build, binding, staging

    rank, world, local = dist_env()
    heads, scale = args.mla_heads, 1.0 / math.sqrt(192.0)
    if args.impl == "reference":
        if rank != 0:
            return
        pairs, secs, n = mla_oracle_rows(wl, heads, scale, args.cpu_budget_s)
        value = pairs / secs
        line = {"impl": "reference", "metric": MLA_METRIC, "value": value, "unit": MLA_UNIT,
                "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "config": {"workload": wl.name + "+sparse_mla", "heads": heads},
                "cpu_baseline": {"value": value, "unit": MLA_UNIT, "cores": cpu_cores(),
                                 "kind": "oracle", "sample": f"{n} query rows of layer 0"},
                "e2e": {"value": value, "unit": MLA_UNIT, "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    _build.build_library(quiet=True)
    dev = torch.device("cuda", torch.cuda.current_device())
    meta = staging.stage_metadata(wl, dev)
    full = [binding.layer_is_full(l, wl.pattern, wl.freq, wl.offset) for l in range(wl.num_layers)]
    layers = []
    for l in range(wl.num_layers):
        if full[l]:
            io = staging.stage_mla(wl, l, meta, heads, dev)
            io["kv_new"] = torch.from_numpy(wl.mla_kv_new(l)).to(dev)
            io["out"] = torch.empty((wl.T, heads, 512), dtype=torch.bfloat16, device=dev)
            io["lse"] = torch.empty((wl.T, heads), dtype=torch.float32, device=dev)
            layers.append(io)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    selected = sum(int((io["topk"][:wl.T] >= 0).sum().item()) for io in layers)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def one_step(events=None):
        for j, io in enumerate(layers):
            binding.mla_write_kv(io["kv_new"], meta.query_start_loc, meta.seq_lens,
                                 meta.block_table, io["kv_cache"], status=status)
            if events:
                events[j][0].record(stream)
            binding.sparse_mla_attention(io["q"], io["kv_cache"], meta.query_start_loc,
                                         meta.seq_lens, meta.block_table, io["topk"], scale,
                                         out=io["out"], lse=io["lse"], status=status)
            if events:
                events[j][1].record(stream)

    one_step()
    torch.cuda.synchronize()
    graph = None
    if not args.no_graph:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            one_step()
    run = graph.replay if graph is not None else one_step
    for _ in range(args.warmup):
        run()
    torch.cuda.synchronize()
    assert status.item() == 0, f"device status {status.item()}"
    ev0 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ev1 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_push("timed_steps")
    with ClockSampler(dev.index) as clocks:
        for i in range(args.steps):
            flush.fill_(i & 0xFF)
            ev0[i].record(stream)
            run()
            ev1[i].record(stream)
            ev1[i].synchronize()
        torch.cuda.synchronize()
        torch.cuda.nvtx.range_pop()
        k_ms = []
        for i in range(args.steps):
            flush.fill_(i & 0xFF)
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in layers]
            one_step(evs)
            torch.cuda.synchronize()
            k_ms.extend(a.elapsed_time(b) for a, b in evs)
    if world > 1:
        torch.distributed.barrier()
    ms = sum(a.elapsed_time(b) for a, b in zip(ev0, ev1)) / args.steps
    kms = sum(k_ms) / len(k_ms)

    # end to end: this step's q, top-k rows and new records from pinned host
    # memory, the outputs back
    host = [{k: io[k].cpu().pin_memory() for k in ("q", "topk", "kv_new")} for io in layers]
    outs = [torch.empty_like(io["out"], device="cpu").pin_memory() for io in layers]
    h2d = sum(v.numel() * v.element_size() for h in host for v in h.values())
    d2h = sum(o.numel() * o.element_size() for o in outs)

    def e2e_step():
        for io, h in zip(layers, host):
            for k, v in h.items():
                io[k].copy_(v, non_blocking=True)
        run()
        for io, o in zip(layers, outs):
            o.copy_(io["out"], non_blocking=True)

    for _ in range(max(1, args.warmup)):
        e2e_step()
    torch.cuda.synchronize()
    e0 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    e1 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    for i in range(args.steps):
        flush.fill_(i & 0xFF)
        e0[i].record(stream)
        e2e_step()
        e1[i].record(stream)
        e1[i].synchronize()
    e2e_ms = sum(a.elapsed_time(b) for a, b in zip(e0, e1)) / args.steps
    (ms, e2e_ms), total_selected = reduce_over_ranks([ms, e2e_ms], selected, world, dev)

    peaks = read_peaks()
    per_layer_sel = selected / len(layers)
    flops = per_layer_sel * heads * 2.0 * (576 + 512)          # QK^T and PV, useful work
    bytes_ = per_layer_sel * 656 + wl.T * heads * (576 * 2 + 512 * 2 + 4)
    tflops = flops / (kms * 1e-3) / 1e12
    gbs = bytes_ / (kms * 1e-3) / 1e9
    roof = {"bound": "tensor", "achieved": tflops, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
            "frac": tflops / peaks["bf16_tflops"], "traffic": None,
            "kernel": "sparse_mla_kernel", "kernel_ms": kms, "algorithmic_flops": flops,
            "algorithmic_bytes": bytes_, "peak_source": peaks["source"] + " bf16",
            "executed_flops_note": "each of the 4 CTAs of a row recomputes QK^T: executed tensor "
                                   "work is (4*576 + 512) / (576 + 512) = 2.59x the algorithmic; "
                                   "each CTA gathers every selected record itself",
            "other_bound": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"],
                            "unit": "GB/s", "frac": gbs / peaks["hbm_gbs"]}}
    line = {
        "metric": MLA_METRIC, "value": total_selected / (ms * 1e-3), "unit": MLA_UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16 (fp8 e4m3 records dequantised; fp32 accumulate)", "data": "synthetic",
        "config": {"workload": wl.name + "+sparse_mla", "heads": heads, "index_topk": wl.index_topk,
                   "layers": len(layers), "requests": wl.R, "query_rows": wl.T,
                   "selected_per_step": selected, "softmax_scale": scale,
                   "cuda_graph": graph is not None, "l2": "flushed between timed steps",
                   "parallelism": f"replicas x{world}"},
        "roofline": roof,
        "e2e": {"value": total_selected / (e2e_ms * 1e-3), "unit": MLA_UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
        "clocks": clocks.summary(),
        "gpu_launches": 2 * len(layers) * args.steps,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        pairs, secs, n = mla_oracle_rows(wl, heads, scale, args.cpu_budget_s)
        line["cpu_baseline"] = {"value": pairs / secs, "unit": MLA_UNIT, "cores": cpu_cores(),
                                "kind": "oracle", "sample": f"{n} query rows of layer 0 in order "
                                f"({pairs} pairs, {secs:.1f} s; numpy FP64)"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


# ----------------------------------------------------------------------------
# FP8 dense tensor peak (measured here, next to the driver's BF16 and HBM peaks)
# ----------------------------------------------------------------------------

def fp8_peak_probe(dev, sustain_s: float = 2.0) -> dict:
    """Dense E4M3 GEMM rate of this GPU through cuBLASLt (torch._scaled_mm,
    8192^3, FP32 accumulate, BF16 out): best of 10 back-to-back launches
    (burst) and the mean over a loop of about `sustain_s` seconds (sustained).
    Falls back to the measured BF16 rate x 2 (the nominal FP8:BF16 dense
    ratio) when the probe cannot run."""
    import torch
    peaks = read_peaks()
    fallback = {"fp8_tflops": 2.0 * peaks["bf16_tflops"], "fp8_tflops_sustained": None,
                "source": f"{peaks['source']} bf16 x 2 (nominal fp8:bf16 dense ratio)"}
    try:
        n = 8192
        g = torch.Generator(device=dev).manual_seed(0)
        a = torch.randn((n, n), device=dev, generator=g).to(torch.float8_e4m3fn)
        b = torch.randn((n, n), device=dev, generator=g).to(torch.float8_e4m3fn)
        one = torch.ones((), device=dev, dtype=torch.float32)

        def mm():
            return torch._scaled_mm(a, b.t(), scale_a=one, scale_b=one, out_dtype=torch.bfloat16)

        for _ in range(3):
            mm()
        torch.cuda.synchronize()
        best = float("inf")
        for _ in range(10):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            mm()
            e1.record()
            e1.synchronize()
            best = min(best, e0.elapsed_time(e1))
        flops = 2.0 * n ** 3
        reps = max(10, int(sustain_s * 1e3 / best))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            mm()
        e1.record()
        e1.synchronize()
        sus = e0.elapsed_time(e1) / reps
        del a, b
        return {"fp8_tflops": flops / (best * 1e-3) / 1e12,
                "fp8_tflops_sustained": flops / (sus * 1e-3) / 1e12,
                "source": "measured here: torch._scaled_mm e4m3 8192^3 (cuBLASLt), burst best of 10, "
                          f"sustained mean of {reps}"}
    except Exception as e:  # noqa: BLE001 -- any failure falls back to the nominal ratio
        fallback["probe_error"] = f"{type(e).__name__}: {e}"[:200]
        return fallback


# ----------------------------------------------------------------------------
# GPU leg
# ----------------------------------------------------------------------------

HEADLINE_WORKLOAD = 4           # long-context decode: the largest single-GPU workload
PER_CONFIG_WORKLOADS = (0, 1, 2, 3, 4)


def measure_workload(args, wid: int, dev, peaks: dict, fp8: dict, world: int, rank: int,
                     cpu_budget_s: float) -> dict:
    """Stage workload `wid`, time `args.steps` graph-replayed steps (L2 flushed
    between them), time every scoring + selection launch, the end-to-end path
    from pinned host buffers, and (rank 0, one rank) the oracle on a bounded
    sample.  Returns the workload's JSON fields."""
    import torch
    from dsa_sparse_attention_fp8_gb300 import binding, staging
    from dsa_sparse_attention_fp8_gb300.step import IndexerStep

    wl = synth.make_workload(wid, seed=args.seed + rank, scale=args.scale)
    meta = staging.stage_metadata(wl, dev)
    full = [binding.layer_is_full(l, wl.pattern, wl.freq, wl.offset) for l in range(wl.num_layers)]
    caches, host_layers = [], {}
    for l in range(wl.num_layers):
        if not full[l]:
            caches.append(None)
            continue
        io = staging.stage_layer(wl, l, meta, dev)
        caches.append(io["k_cache"])
        if args.bf16:
            q16 = torch.from_numpy(wl.q(l)).to(dev).bfloat16()
            ins = (io["k"].bfloat16(), q16, io["w"])
        else:
            ins = (io["k"], io["q_fp8"], io["q_scale"], io["w"])
        host_layers[l] = tuple(t.cpu().pin_memory() for t in ins)
        del io
    step = IndexerStep(num_layers=wl.num_layers, pattern=wl.pattern, freq=wl.freq,
                       offset=wl.offset, H=wl.H, index_topk=wl.index_topk, T=wl.T, R=wl.R,
                       max_blocks=wl.max_blocks, num_pages=wl.num_pages,
                       max_num_batched_tokens=wl.max_num_batched_tokens, k_caches=caches,
                       device=dev, time_score_kernels=True, bf16=args.bf16,
                       compress_ratio=wl.compress_ratio)
    host_meta = tuple(torch.from_numpy(np.ascontiguousarray(a)).pin_memory() for a in
                      (wl.query_start_loc, wl.seq_lens.astype(np.int32), wl.block_table))
    host = {"meta": host_meta, "layers": host_layers}
    step.set_metadata(*host_meta)
    for l, io in host_layers.items():
        step.set_layer(l, *io)
    torch.cuda.synchronize()

    n_full = sum(full)
    pairs_per_step = wl.pairs_per_full_layer * n_full
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    # ---- warm-up (eager once, then capture), then timed steps
    step.launch()
    torch.cuda.synchronize()
    if not args.no_graph:
        step.capture()
    for _ in range(args.warmup):
        step.run(timed=False)
        step.run(timed=True)
    torch.cuda.synchronize()
    assert step.status.item() == 0, f"device status {step.status.item()}"
    launches = step.launches_per_step

    ev0 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ev1 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    score_ms = []
    kernel_timing = ("events inside a second captured pass of the timed steps" if not args.no_graph
                     else "events around each launch")
    timing_failed = False
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_push("timed_steps")
    with ClockSampler(dev.index) as clocks:
        for i in range(args.steps):
            flush.fill_(i & 0xFF)                 # evict L2 between timed steps
            ev0[i].record(stream)
            step.run(timed=False)
            ev1[i].record(stream)
            ev1[i].synchronize()
        torch.cuda.synchronize()
        # the same steps again with events around every layer's scoring +
        # selection launches (the roofline's per-launch durations)
        for i in range(args.steps):
            flush.fill_(i & 0xFF)
            step.run(timed=True)
            torch.cuda.synchronize()
            if not timing_failed:
                try:
                    score_ms.extend(step.score_kernel_ms())
                except RuntimeError:
                    timing_failed = True
    torch.cuda.nvtx.range_pop()
    if world > 1:
        torch.distributed.barrier()
    step_ms = [a.elapsed_time(b) for a, b in zip(ev0, ev1)]
    if timing_failed:
        score_ms, kernel_timing = [], "events around each launch, eager steps after the timed region"
        for i in range(args.steps):
            flush.fill_(i & 0xFF)
            step.launch()
            torch.cuda.synchronize()
            score_ms.extend(step.score_kernel_ms())
    ms = sum(step_ms) / len(step_ms)

    # ---- end to end through the public API with host buffers
    out = torch.empty((wl.T, wl.index_topk), dtype=torch.int32).pin_memory()
    h2d = step.host_input_bytes(host)
    d2h = out.numel() * out.element_size()
    for _ in range(max(1, args.warmup)):
        step.run_from_host(host, out)
    torch.cuda.synchronize()
    e0 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    e1 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    for i in range(args.steps):
        flush.fill_(i & 0xFF)
        e0[i].record(stream)
        step.run_from_host(host, out)
        e1[i].record(stream)
        e1[i].synchronize()
    e2e_ms = sum(a.elapsed_time(b) for a, b in zip(e0, e1)) / args.steps

    (ms, e2e_ms), total_pairs = reduce_over_ranks([ms, e2e_ms], pairs_per_step, world, dev)
    clk = clocks.summary()
    uses_rows = step.uses_row_selection()
    del step, caches, flush
    torch.cuda.empty_cache()

    # ---- roofline of the dominant kernel pair (scoring + top-k selection), per layer
    k_ms = sum(score_ms) / len(score_ms)
    rows_bytes = wl.T * (wl.H * (128 + 4 + 4) + wl.index_topk * 4)   # q, q_scale, w in; top-k out
    # every key (cache entry) of a request is read once, whatever the number of
    # its query rows (one row per request in a decode batch: one key per pair)
    key_bytes = float(wl.entries[wl.q_lens > 0].astype(np.int64).sum()) * BYTES_PER_PAIR
    alg_bytes = key_bytes + rows_bytes
    achieved = alg_bytes / (k_ms * 1e-3) / 1e9
    kernel = "score_topk_kernel + rows_topk_kernel" if uses_rows else "score_topk_kernel"
    traffic = profiled_traffic(wl.name) if not uses_rows else None
    fp8_peak = fp8["fp8_tflops"]
    alg_flops = wl.pairs_per_full_layer * 2.0 * wl.H * 128
    tflops = alg_flops / (k_ms * 1e-3) / 1e12
    hbm = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
           "frac": achieved / peaks["hbm_gbs"], "traffic": traffic,
           "peak_source": f"{peaks['source']} copy (MEASURED_PEAKS.json hbm_gbs)"}
    tensor = {"bound": "tensor", "achieved": tflops, "peak": fp8_peak, "unit": "TFLOP/s",
              "frac": tflops / fp8_peak, "traffic": traffic,
              "peak_source": f"fp8 e4m3 dense, burst: {fp8['source']}"}
    # HBM-bound unless the work's FP8 FLOP per algorithmic byte exceed the
    # machine balance (peak FLOP/s over peak bytes/s): prefill chunks reuse each
    # key across many rows, decode batches (also with a few MTP rows) do not
    prefill = alg_flops / alg_bytes > fp8_peak * 1e12 / (peaks["hbm_gbs"] * 1e9)
    roof = dict(tensor if prefill else hbm)
    roof.update({"kernel": kernel, "kernel_ms": k_ms, "algorithmic_bytes": alg_bytes,
                 "algorithmic_flops": alg_flops, "kernel_timing": kernel_timing,
                 "other_bound": {k: v for k, v in (hbm if prefill else tensor).items()
                                 if k != "traffic"}})
    res = {
        "workload": wl.name, "value": total_pairs / (ms * 1e-3), "ms_per_step": ms,
        "tokens_per_s": wl.T * n_full * world / (ms * 1e-3),
        "config": {"workload": wl.name, **{k: v for k, v in wl.describe().items() if k != "workload"},
                   "pairs_per_step": pairs_per_step, "full_layers": n_full,
                   "cuda_graph": not args.no_graph, "l2": "flushed between timed steps",
                   "inputs": ("bf16 keys and queries, quantised in the cache-write launch"
                              if args.bf16 else "fp32 keys, e4m3 queries + fp32 scales"),
                   "parallelism": f"replicas x{world}"},
        "roofline": roof,
        "e2e": {"value": total_pairs / (e2e_ms * 1e-3), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
        "clocks": clk,
        "gpu_launches": launches * args.steps,
    }
    if rank == 0 and world == 1 and cpu_budget_s > 0:
        res["cpu_baseline"] = cpu_baseline(wl, cpu_budget_s)
    return res


def spawn_replicas(args):
    """`--gpus N` with N > 1 outside a launcher: run this command as N local
    ranks under torch.distributed.run (one replica per GPU) and return its exit
    code; None when this process is already a rank or N == 1."""
    if args.gpus <= 1 or "WORLD_SIZE" in os.environ:
        return None
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
           f"--nproc-per-node={args.gpus}", "--master-addr", "127.0.0.1",
           f"--master-port={port}", str(Path(__file__).resolve()), *sys.argv[1:]]
    return subprocess.call(cmd)


def main():
    args = parse()
    rc = spawn_replicas(args)
    if rc is not None:
        sys.exit(rc)
    rank, world, local = dist_env()
    if world != args.gpus:
        sys.exit(f"bench.py: --gpus {args.gpus} but WORLD_SIZE={world}; run with matching "
                 "values (or without a launcher: --gpus N starts N ranks itself)")
    wid = HEADLINE_WORKLOAD if args.workload is None else args.workload
    if args.sparse_mla:
        run_sparse_mla(args, synth.make_workload(1 if args.workload is None else args.workload,
                                                 seed=args.seed + rank, scale=args.scale))
        return
    if args.impl == "reference":
        run_reference(args, synth.make_workload(wid, seed=args.seed + rank, scale=args.scale))
        return

    import torch
    from dsa_sparse_attention_fp8_gb300 import _build

    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    _build.build_library(quiet=True)
    dev = torch.device("cuda", torch.cuda.current_device())
    peaks = read_peaks()
    fp8 = fp8_peak_probe(dev)
    budget = 0.0 if args.no_cpu_baseline else args.cpu_budget_s

    head = measure_workload(args, wid, dev, peaks, fp8, world, rank, budget)
    per_config = {}
    configs = [] if args.configs.strip() in ("", "none") else [int(c) for c in args.configs.split(",")]
    for c in configs:
        if c == wid:
            r = head
        else:
            r = measure_workload(args, c, dev, peaks, fp8, world, rank,
                                 min(budget, args.cpu_budget_per_config_s))
        per_config[r["workload"]] = {k: r[k] for k in ("value", "tokens_per_s", "ms_per_step",
                                                       "roofline", "e2e", "cpu_baseline", "config")
                                     if k in r}

    line = {
        "metric": METRIC, "value": head["value"], "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "fp8_e4m3 (fp32 accumulate)", "data": "synthetic",
        "config": head["config"],
        "tokens_per_s": head["tokens_per_s"],
        "roofline": head["roofline"],
        "e2e": head["e2e"],
        "clocks": head["clocks"],
        "gpu_launches": head["gpu_launches"],
        "peaks": {"hbm_gbs": peaks["hbm_gbs"], "bf16_tflops": peaks["bf16_tflops"],
                  "source": peaks["source"], **fp8},
    }
    if "cpu_baseline" in head:
        line["cpu_baseline"] = head["cpu_baseline"]
    if per_config:
        line["per_config"] = per_config
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
