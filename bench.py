"""Benchmark of the GB300 two-level candidate indexer.

One step = one pass of the whole indexer path over one batch of synthetic
input: the source layer's dense block keys, its published candidate blocks,
its own top-512 and the four consumer layers' top-512.  The headline workload
is the 16384-row prefill chunk at 262144 compressed positions; the decode
batches, the multi-request prefill chunk (with prefill_tail over its
published table) and the headline chunk with MXFP4 index-K pools are reported
as secondary lines in the same JSON object.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

N > 1 runs N independent replicas (one per GPU, launched by torchrun); the
indexer has no exchange step, so no collective touches the data path.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)
# The CPU oracle baseline runs one row per host thread; each numpy BLAS call
# stays on its own thread (set before numpy is first imported, by torch).
for _v in ("OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import torch  # noqa: E402

HEADLINE_CID = 4
METRIC = "indexer ms per 16K-token prefill chunk @262K ctx"
PAGES_LAST_CHUNK_MS = 78.2  # sglang PR #40352 Performance table: PR's indexer kernels, last chunk (4x B200)
L2_FLUSH_BYTES = 256 << 20


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(values, world, device):
    """Element-wise maximum of `values` over all ranks (the slowest replica
    sets the job's time); identity on one rank."""
    values = [float(v) for v in values]
    if world <= 1:
        return values
    t = torch.tensor(values, dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return t.tolist()


def emit_line(line, rank):
    """Rank 0 alone prints the job's JSON line."""
    if rank == 0:
        print(json.dumps(line), flush=True)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


# tcgen05 kind::mxf8f6f4 rate measured by this library's own microbenchmark
# (M = 128, N >= 128, 152 SMs at 2070 MHz): context beside the derived peak.
MXF8F6F4_PROBE_TFLOPS = 4860.0


def tensor_peaks(peaks, src):
    """Block-scaled tensor peaks derived from the measured dense bf16 burst
    rate by the nominal ratios (bf16 2.25, fp8 4.5, fp4 13.5 PFLOP/s): FP8 x 2
    for kind::mxf8f6f4 (MXFP4 queries against FP8 index-K), FP4 x 6 for
    kind::mxf4 (MXFP4 against MXFP4)."""
    bf16 = peaks["bf16_tflops"]
    return {
        "fp8": (2.0 * bf16, f"{src} bf16_tflops (burst) x 2, the fp8 / bf16 nominal ratio (kind::mxf8f6f4)"),
        "fp4": (6.0 * bf16, f"{src} bf16_tflops (burst) x 6, the fp4 / bf16 nominal ratio (kind::mxf4)"),
    }


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in getattr(self, "lines", []):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def algorithmic_counts(wl):
    """FLOPs of the dense pass and bytes of index-K it must read.

    Dense scorer: 2 * H * D flops per (row, position) over rows with more than
    min(K, P + 1) blocks.  Bytes: 132 per position of K (128 e4m3 + 4-byte scale;
    68 for MXFP4 pools: 64 packed bytes + 4 scale bytes) read once per launch --
    the pool of a prefill chunk, every scored row's own positions in decode --
    plus the query and weights of scored rows.
    """
    kpos = k_position_bytes(wl)
    L = wl.seq_len.to(torch.int64).cpu()
    nb = (L + 7) // 8
    scored = nb > min(wl.topk_blocks, wl.topk + 1)
    positions = int(L[scored].sum())
    flops = 2 * 64 * 128 * positions
    if wl.layout == 1:
        kbytes = kpos * (int(L.max()) if bool(scored.any()) else 0)
    else:
        kbytes = kpos * positions
    qbytes = int(scored.sum()) * (64 * 64 + 64 * 4 + 64 * 4)
    return flops, kbytes + qbytes, positions


def k_position_bytes(wl):
    """Index-K bytes per position: 132 for FP8 pages, 68 for MXFP4 pages."""
    return 68 if wl.kv == 1 else 132


def select_work(wl):
    """Algorithmic work of the step's sparse-scorer launches (the source with
    its K' = P + 1 blocks, every consumer with K).

    Returns ``(positions, gathered, other)``: candidate positions scored (each
    2 * 64 * 128 flops), index-K bytes gathered for them (132 per position:
    128 e4m3 + one fp32 scale; 68 for MXFP4 pools), and the per-row bytes
    (query, scales and weights 4608, block ids 4 per block, output positions
    4 per pick).  A row with nb_t <= K' blocks scores all L_t positions;
    otherwise K' - 1 full blocks plus its newest (partial) block.
    """
    L = wl.seq_len.to(torch.int64).cpu()
    nb = (L + 7) // 8
    P, K = wl.topk, wl.topk_blocks

    def one(kb):
        full = nb > kb
        pos = torch.where(full, 8 * (kb - 1) + (L - 8 * (nb - 1)), L)
        blocks = torch.where(full, torch.full_like(nb, kb), nb)
        return int(pos.sum()), int((4608 + 4 * blocks + 4 * P).sum())

    pos0, oth0 = one(P + 1)
    posk, othk = one(K)
    n = len(wl.layers) - 1
    positions = pos0 + n * posk
    return positions, k_position_bytes(wl) * positions, oth0 + n * othk


def select_bytes(wl):
    """Algorithmic bytes of the step's sparse-scorer launches (gathered K plus
    the per-row bytes, see select_work)."""
    _, gathered, other = select_work(wl)
    return gathered + other


def publish_bytes(wl):
    """Algorithmic bytes of the publish launch: 4 per key of every row that
    selects (nb_t > min(K, P + 1)), and the two tables it writes (K and
    P + 1 ids, and a count, per row)."""
    L = wl.seq_len.to(torch.int64).cpu()
    nb = (L + 7) // 8
    K, Kp = wl.topk_blocks, wl.topk + 1
    reads = int((4 * nb[nb > min(K, Kp)]).sum())
    return reads + wl.rows * 4 * (K + Kp + 2)


def time_steps(step, steps, warmup, flush, stream, dense_events=True):
    """Per-step CUDA-event durations (ms) on `stream`, whole step and per
    kernel kind (events recorded between the step's launches)."""
    for _ in range(warmup):
        step.run(stream)
    torch.cuda.synchronize()
    out = {"step": [], "dense": [], "publish": [], "select": []}
    for _ in range(steps):
        with torch.cuda.stream(stream):
            flush.zero_()  # evict L2 between steps (same stream, before the first event: not timed)
        marks = []

        def mark(name):
            ev = torch.cuda.Event(enable_timing=True)
            ev.record(stream)
            marks.append((name, ev))

        mark("start")
        step.run(stream, mark=mark)
        torch.cuda.synchronize()
        per = {"dense": 0.0, "publish": 0.0, "select": 0.0}
        for (_, a), (name, b) in zip(marks, marks[1:]):
            per[name] += a.elapsed_time(b)
        out["step"].append(marks[0][1].elapsed_time(marks[-1][1]))
        for k, v in per.items():
            out[k].append(v)
    return out


def graph_step_ms(step, steps, stream, flush):
    """Mean device time of the step replayed as a CUDA graph (L2 flushed
    before every replay)."""
    graph = step.capture(stream)
    ms = []
    with torch.cuda.stream(stream):
        for i in range(steps + 3):
            flush.fill_(i & 0xFF)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            graph.replay()
            e1.record(stream)
            e1.synchronize()
            if i >= 3:
                ms.append(e0.elapsed_time(e1))
    return statistics.mean(ms)


def e2e_time(step, steps, stream):
    """The same step through the library's public API with host buffers:
    IndexerStep.run_host copies the step's inputs from pinned host memory
    and its results (published blocks, every layer's positions) back to
    pinned host memory, overlapping the copies with the kernels; all of it
    inside the timed region."""
    shared, layers = step.device_inputs()
    host_shared = [t.cpu().pin_memory() for t in shared]
    host_layers = [[t.cpu().pin_memory() for t in l] for l in layers]
    outs = [step.blocks, step.nvalid] + [step.pos[j] for j in range(len(layers))]
    host_out = [torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for o in outs]
    h2d = sum(t.numel() * t.element_size() for t in host_shared + [x for l in host_layers for x in l])
    d2h = sum(t.numel() * t.element_size() for t in host_out)
    times = []
    for _ in range(steps + 1):
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        step.run_host(host_shared, host_layers, host_out, stream)
        stream.synchronize()
        times.append((time.perf_counter() - t0) * 1e3)
    return times[1:], h2d, d2h


def host_threads():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def sample_rows(n, cap=128):
    """All rows when there are at most ``cap``; otherwise the first cap/4, the
    last cap/4 and cap/2 evenly spaced rows between them."""
    if n <= cap:
        return list(range(n))
    q = cap // 4
    mid = [q + round(i * (n - 2 * q - 1) / (cap - 2 * q - 1)) for i in range(cap - 2 * q)]
    return sorted(set(list(range(q)) + mid + list(range(n - q, n))))


def oracle_rows_s(wl, rows, threads):
    """Wall seconds of the oracle as it stands over ``rows`` of workload
    ``wl`` (any device: the rows' operands and the pools are copied to the
    host first, outside the timing), one row per host thread: the source
    layer's dense scores, keys, published blocks and own top-P, then every
    consumer's top-P within the published blocks."""
    import concurrent.futures

    import numpy as np

    from oracle import ci_oracle as O
    from two_level_sparse_gb300 import synth

    idx = torch.tensor(rows, dtype=torch.long, device=wl.seq_len.device)
    layers = [synth.Layer(l.q_fp4[idx].cpu(), l.q_sf[idx].cpu(), l.w[idx].cpu(), l.k_pool.cpu()) for l in wl.layers]
    pt = (wl.page_table[idx] if wl.layout == synth.LAYOUT_DECODE else wl.page_table).cpu().numpy()
    lens = wl.seq_len[idx].cpu().numpy()
    K, P = wl.topk_blocks, wl.topk

    def one(i):
        L = int(lens[i])
        src = O.source_row(layers[0], pt, wl.layout, i, L, max(K, P + 1), P)
        blocks, nv = O.select_blocks(src["keys"], O.num_blocks(L), K)
        for j in range(1, len(layers)):
            O.select_row(layers[j], pt, wl.layout, i, L, blocks, nv, P)

    t0 = time.perf_counter()
    with concurrent.futures.ThreadPoolExecutor(max_workers=threads) as ex:
        list(ex.map(one, range(len(rows))))
    return time.perf_counter() - t0


def cpu_baseline(wl, unit, cap=128, threads=None):
    """The oracle timed on the host cores over a bounded row sample of ``wl``
    (all rows when there are at most ``cap``), in the line's unit: ms per step
    extrapolated linearly to every row (rows are independent), or rows/s."""
    threads = threads or host_threads()
    rows = sample_rows(wl.rows, cap)
    sec = oracle_rows_s(wl, rows, threads)
    per_step_ms = sec * 1e3 * wl.rows / len(rows)
    value = wl.rows / (per_step_ms * 1e-3) if unit == "rows/s" else per_step_ms
    what = "all rows" if len(rows) == wl.rows else (f"{len(rows)} of {wl.rows} rows (first {cap // 4}, last "
                                                    f"{cap // 4}, {cap // 2} evenly spaced), extrapolated linearly")
    return {"value": value, "unit": unit, "cores": threads, "kind": "oracle",
            "sample": f"{what}; all {len(wl.layers)} layers; one row per host thread ({threads} threads), "
                      f"{sec:.1f} s wall"}


def headline_config(wl, world, kv="fp8"):
    return {"workload": wl.name, "rows": wl.rows, "context": wl.max_len, "topk_blocks": wl.topk_blocks,
            "topk": wl.topk, "layers": len(wl.layers), "index_k": kv, "parallelism": f"replicas x{world}",
            "l2": "flushed between timed steps (256 MiB write)"}


REFERENCE_ROWS_PER_STEP = 48


def run_reference(args):
    """The reference arm: the oracle as it stands, on the host cores, timed on
    the headline workload.  Each step is a bounded row sample (the first,
    last and evenly spaced rows, REFERENCE_ROWS_PER_STEP of them) extrapolated
    linearly to the chunk."""
    world, rank, local = dist_env()
    if rank != 0:
        return 0
    from two_level_sparse_gb300 import synth

    kv = getattr(args, "kv", "fp8")
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    wl = synth.config_workload(HEADLINE_CID, device=dev, kv=1 if kv == "mxfp4" else 0)
    threads = host_threads()
    rows = sample_rows(wl.rows, REFERENCE_ROWS_PER_STEP)
    steps = []
    for _ in range(args.warmup + args.steps):
        steps.append(oracle_rows_s(wl, rows, threads) * 1e3 * wl.rows / len(rows))
    value = statistics.mean(steps[args.warmup:]) if args.steps else steps[-1]
    sample = (f"{len(rows)} of {wl.rows} rows per step (first, last and evenly spaced), all {len(wl.layers)} "
              f"layers, one row per host thread, extrapolated linearly to the chunk")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "ms", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": value, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": headline_config(wl, world, kv),
        "cpu_baseline": {"value": value, "unit": "ms", "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "ms", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    emit_line(line, rank)
    return 0


def last_rows(wl, rows):
    from two_level_sparse_gb300 import synth

    if rows <= 0 or rows >= wl.rows:
        return wl
    sl = slice(wl.rows - rows, wl.rows)
    layers = [synth.Layer(l.q_fp4[sl].contiguous(), l.q_sf[sl].contiguous(), l.w[sl].contiguous(), l.k_pool)
              for l in wl.layers]
    pt = wl.page_table[sl].contiguous() if wl.layout == synth.LAYOUT_DECODE else wl.page_table
    return synth.Workload(f"{wl.name}_last{rows}rows", wl.layout, wl.seq_len[sl].contiguous(), pt, layers,
                          wl.topk_blocks, wl.topk)


def measure(cid, steps, warmup, stream, flush, e2e=False, rows=0, wl=None, kv=0):
    from two_level_sparse_gb300 import synth

    from two_level_sparse_gb300.step import IndexerStep

    if wl is None:
        wl = last_rows(synth.config_workload(cid, device="cuda", kv=kv), rows)
    step = IndexerStep(wl)
    times = time_steps(step, steps, warmup, flush, stream)
    res = {"cid": cid, "wl": wl, "step": step, "t_step": times["step"], "t_dense": times["dense"],
           "t_select": times["select"], "t_publish": times["publish"], "launches": step.launches()}
    if e2e:
        res["e2e"] = e2e_time(step, max(2, min(steps, 5)), stream)
    return res


def measure_mxfp4(steps, stream, flush, world, peaks, peak_src):
    """The headline chunk with MXFP4 index-K pools (the pages' use_fp4_cache
    variant): the same step with FP4 x FP4 block-scaled MMAs (kind::mxf4) and
    68-byte K positions."""
    from two_level_sparse_gb300 import synth

    wl = synth.config_workload(HEADLINE_CID, device="cuda", kv=synth.KV_MXFP4)
    r = measure(None, steps, 3, stream, flush, wl=wl)
    mst, msd, mss = (statistics.mean(r[k]) for k in ("t_step", "t_dense", "t_select"))
    flops, _, _ = algorithmic_counts(wl)
    positions, gathered, _ = select_work(wl)
    fp4_peak, fp4_src = tensor_peaks(peaks, peak_src)["fp4"]
    line = {
        "metric": "indexer ms per 16K-token prefill chunk @262K ctx, MXFP4 index-K", "workload": wl.name,
        "value": mst, "unit": "ms", "ms_per_step": mst,
        "kernel_ms": {"dense": msd, "publish": statistics.mean(r["t_publish"]), "select": mss},
        "dense_roofline": tensor_roofline(flops, msd, 1, fp4_peak, fp4_src),
        "select_roofline": tensor_roofline(2 * 64 * 128 * positions, mss, len(wl.layers), fp4_peak, fp4_src),
        "l2_gather": l2_gather(gathered, mss),
        "dev_err": int(r["step"].dev_err.item()),
    }
    del r
    return line


def tensor_roofline(flops_per_step, ms_per_step, launches, peak, peak_source, kernel=None, traffic=None):
    """A scorer against its block-scaled tensor peak: flops per launch over the
    mean launch time (launches that overlap at their edges on side streams
    count the phase / launches)."""
    achieved = flops_per_step / (ms_per_step * 1e-3) / 1e12
    out = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
           "traffic": traffic, "peak_source": peak_source, "flops_per_launch": flops_per_step / launches,
           "launches_per_step": launches, "ms_per_launch": ms_per_step / launches, "ms_per_step": ms_per_step}
    if kernel:
        out = {"kernel": kernel, **out}
    return out


def l2_gather(gathered_bytes, ms):
    return {"gbs": gathered_bytes / (ms * 1e-3) / 1e9, "bytes_per_step": gathered_bytes,
            "note": "candidate index-K gathered by the selects; a prefill chunk's pools (34.6 MB per layer) "
                    "are L2-resident, so these bytes come from L2 and are not a fraction of HBM bandwidth"}


def measure_dcp(steps, stream, flush, world):
    """The headline chunk as ``world`` context shards emulated on this device:
    every shard's dense pass and selects run here, one after another, with
    the two merges in between (on ``world`` devices the shards would run side
    by side and the merges would be collectives).  The outputs equal the
    unsharded step's; the time shows what the sharded form costs on one
    device."""
    from two_level_sparse_gb300 import synth
    from two_level_sparse_gb300.dcp import DcpStep

    wl = synth.config_workload(HEADLINE_CID, device="cuda")
    d = DcpStep(wl, world, with_scores=False)
    ms = []
    with torch.cuda.stream(stream):
        for i in range(steps + 1):
            flush.fill_(i & 0xFF)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            d.run(stream)
            e1.record(stream)
            e1.synchronize()
            if i >= 1:
                ms.append(e0.elapsed_time(e1))
    return {"metric": f"indexer ms per 16K-token prefill chunk @262K ctx, {world} context shards on one GPU",
            "workload": wl.name + f"_dcp{world}", "value": statistics.mean(ms), "unit": "ms",
            "dev_err": int(d.dev_err.item())}


QPROD_TOKENS = 16384


def measure_qprod(steps, stream, flush, peaks):
    """The query producer on a 16384-token chunk (RoPE, MXFP4 quantization,
    weight scaling), inputs resident, L2 flushed before every launch."""
    from two_level_sparse_gb300 import ci

    g = torch.Generator(device="cuda")
    g.manual_seed(11)
    t, max_pos = QPROD_TOKENS, 262144
    q = torch.randn(t, 64, 128, generator=g, device="cuda").to(torch.bfloat16)
    ang = torch.rand(max_pos, 32, generator=g, device="cuda") * 6.2831853
    cos_sin = torch.cat([torch.cos(ang), torch.sin(ang)], 1).contiguous()
    pos = torch.arange(max_pos - t, max_pos, dtype=torch.int32, device="cuda")
    w = torch.randn(t, 64, generator=g, device="cuda")
    q_fp4 = torch.empty(t, 64, 64, dtype=torch.uint8, device="cuda")
    q_sf = torch.empty(t, 64, 4, dtype=torch.uint8, device="cuda")
    w_out = torch.empty(t, 64, dtype=torch.float32, device="cuda")
    ms = []
    with torch.cuda.stream(stream):
        for i in range(steps + 3):
            flush.fill_(i & 0xFF)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            ci.ci_q_rope_quant(pos, q, cos_sin, w, 0.0625, 0.125, True, ci.Q_MXFP4, q_fp4, q_sf, w_out, stream=stream)
            e1.record(stream)
            e1.synchronize()
            if i >= 3:
                ms.append(e0.elapsed_time(e1))
    m = statistics.mean(ms)
    moved = t * 64 * (256 + 4 + 64 + 4 + 4) + t * (4 + 256)  # q, w in; codes, scales, w out; positions, cos/sin rows
    return {"metric": "query producer ms per 16K-token chunk (RoPE + MXFP4 + weights)",
            "workload": f"qprod_{t}tokens_64heads_neox", "value": m, "unit": "ms",
            "roofline": {"bound": "hbm", "achieved": moved / (m * 1e-3) / 1e9, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": moved / (m * 1e-3) / 1e9 / peaks["hbm_gbs"], "bytes": moved}}


VARLEN_TAIL_ROWS = 512  # tail rows kept per request by the prefill_tail timing


def measure_varlen(steps, stream, flush, world):
    """The multi-request prefill chunk (four requests of 4096 rows after 16 K -
    240 K prefixes): the whole step, then prefill_tail over its published
    table keeping the last VARLEN_TAIL_ROWS rows of each request."""
    from two_level_sparse_gb300 import ci, synth

    wl = synth.varlen_chunk_workload(device="cuda")
    r = measure(None, steps, 3, stream, flush, wl=wl)
    step = r["step"]
    nreq = wl.req_start.shape[0] - 1
    tail_len = torch.full((nreq,), VARLEN_TAIL_ROWS, dtype=torch.int32, device="cuda")
    cap = nreq * VARLEN_TAIL_ROWS
    out_row = torch.empty(cap, dtype=torch.int32, device="cuda")
    out_blocks = torch.empty(cap, step.K, dtype=torch.int32, device="cuda")
    out_nvalid = torch.empty(cap, dtype=torch.int32, device="cuda")
    out_count = torch.empty(1, dtype=torch.int32, device="cuda")
    tail_ms = []
    with torch.cuda.stream(stream):
        for i in range(steps + 3):
            flush.fill_(i & 0xFF)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            ci.ci_prefill_tail(wl.req_start, tail_len, step.blocks, step.nvalid, out_row, out_blocks, out_nvalid,
                               out_count, dev_err=step.dev_err, stream=stream)
            e1.record(stream)
            e1.synchronize()
            if i >= 3:
                tail_ms.append(e0.elapsed_time(e1))
    mst = statistics.mean(r["t_step"])
    tail = statistics.mean(tail_ms)
    moved = cap * (step.K + 2) * 4 * 2  # rows read and written, with their count and source row
    return {
        "metric": "multi-request prefill chunk ms", "workload": wl.name, "value": mst, "unit": "ms",
        "rows_per_s": world * wl.rows / (mst * 1e-3), "ms_per_step": mst,
        "kernel_ms": {"dense": statistics.mean(r["t_dense"]), "publish": statistics.mean(r["t_publish"]),
                      "select": statistics.mean(r["t_select"])},
        "prefill_tail": {"ms": tail, "rows_kept": int(out_count.item()), "tail_rows_per_request": VARLEN_TAIL_ROWS,
                         "bytes": moved, "gbs": moved / (tail * 1e-3) / 1e9},
        "dev_err": int(step.dev_err.item()),
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-secondary", action="store_true", help="skip the decode, multi-request and MXFP4 workloads")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end timing")
    ap.add_argument("--rows", type=int, default=0,
                    help="keep only the last ROWS rows of the headline chunk (a smaller case for profilers)")
    ap.add_argument("--kv", default="fp8", choices=["fp8", "mxfp4"],
                    help="index-K page format of the headline chunk (the reported metric is defined on fp8)")
    ap.add_argument("--only", default=None,
                    choices=["qprod", "varlen", "mxfp4", "dcp", "decode4", "decode64", "decode128", "prefill4096"],
                    help="run one secondary workload alone and print its line (a small command for profilers)")
    args = ap.parse_args()
    if args.impl == "reference":
        return run_reference(args)
    args.warmup = max(args.warmup, 3)

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    from two_level_sparse_gb300 import ci  # noqa: F401  (fails loudly without the library)

    stream = torch.cuda.Stream()
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    peaks, peak_src = load_peaks()

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    if args.only is not None:
        steps = max(1, args.steps)
        tpk = tensor_peaks(peaks, peak_src)
        std = {"decode4": 0, "decode64": 1, "decode128": 2, "prefill4096": 3}
        if args.only in std:
            args.no_cpu = True
            one = measure_secondary(std[args.only], args, stream, flush, world, rank, peaks, tpk)
        else:
            one = {"qprod": lambda: measure_qprod(steps, stream, flush, peaks),
                   "varlen": lambda: measure_varlen(steps, stream, flush, world),
                   "mxfp4": lambda: measure_mxfp4(steps, stream, flush, world, peaks, peak_src),
                   "dcp": lambda: measure_dcp(steps, stream, flush, 2)}[args.only]()
        emit_line(one, rank)
        if world > 1:
            torch.distributed.destroy_process_group()
        return 0

    barrier()
    with ClockSampler(local) as clk:
        t0 = time.perf_counter()
        head = measure(HEADLINE_CID, args.steps, args.warmup, stream, flush, e2e=not args.no_e2e, rows=args.rows,
                       kv=1 if args.kv == "mxfp4" else 0)
        barrier()
        wall = time.perf_counter() - t0
    ms_step = statistics.mean(head["t_step"])
    ms_dense = statistics.mean(head["t_dense"])
    ms_select = statistics.mean(head["t_select"])
    ms_publish = statistics.mean(head["t_publish"])
    ms_step, ms_dense, ms_select, ms_publish = max_over_ranks([ms_step, ms_dense, ms_select, ms_publish], world,
                                                              "cuda")
    wl = head["wl"]
    err = int(head["step"].dev_err.item())
    flops, kbytes, positions = algorithmic_counts(wl)
    tpk = tensor_peaks(peaks, peak_src)
    peak, peak_source = tpk["fp4" if args.kv == "mxfp4" else "fp8"]
    sel_positions, sel_gathered, _ = select_work(wl)
    n_select = len(wl.layers)
    e2e_ms, h2d, d2h = head.get("e2e", ([float("nan")], 0, 0))
    e2e_val = statistics.mean(e2e_ms)
    (e2e_val,) = max_over_ranks([e2e_val], world, "cuda")
    cpu_head = None
    if rank == 0 and not args.no_cpu:
        cpu_head = cpu_baseline(wl, "ms")
    config = headline_config(wl, world, args.kv)
    del head
    torch.cuda.empty_cache()

    secondary = []
    if not args.no_secondary:
        for cid in (3, 2, 1, 0):
            secondary.append(measure_secondary(cid, args, stream, flush, world, rank, peaks, tpk))
            torch.cuda.empty_cache()
        secondary.append(measure_varlen(max(3, args.steps // 2), stream, flush, world))
        torch.cuda.empty_cache()
        secondary.append(measure_mxfp4(max(3, args.steps // 2), stream, flush, world, peaks, peak_src))
        torch.cuda.empty_cache()
        secondary.append(measure_qprod(max(3, args.steps // 2), stream, flush, peaks))
        torch.cuda.empty_cache()
        secondary.append(measure_dcp(3, stream, flush, 2))
        torch.cuda.empty_cache()

    value = ms_step / world
    dense_rl = tensor_roofline(flops, ms_dense, 1, peak, peak_source, kernel="dense_amax8_kernel",
                               traffic=recorded_traffic("dense_amax8_kernel"))
    dense_rl["peak_mxf8f6f4_probe"] = MXF8F6F4_PROBE_TFLOPS
    dense_rl["frac_of_probe"] = dense_rl["achieved"] / MXF8F6F4_PROBE_TFLOPS
    select_rl = tensor_roofline(2 * 64 * 128 * sel_positions, ms_select, n_select, peak, peak_source,
                                kernel="select_kernel", traffic=recorded_traffic("select_kernel"))
    select_rl["l2_gather"] = l2_gather(sel_gathered, ms_select)
    pub_b = publish_bytes(wl)
    publish_rl = {"bound": "hbm", "kernel": "publish_kernel", "achieved": pub_b / (ms_publish * 1e-3) / 1e9,
                  "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": pub_b / (ms_publish * 1e-3) / 1e9 / peaks["hbm_gbs"],
                  "traffic": recorded_traffic("publish_kernel"), "bytes_per_launch": pub_b, "ms_per_launch": ms_publish}
    line = {
        "metric": METRIC, "value": value, "unit": "ms", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": False, "scaling": "weak",
        "vs_baseline": value / PAGES_LAST_CHUNK_MS,
        "dtype": ("e2m1xe2m1->f32 (mxf4, ue8m0 scales)" if args.kv == "mxfp4"
                  else "e4m3xe4m3->f32 (mxf8f6f4, ue8m0 scales)"),
        "data": "synthetic",
        "config": config,
        **rooflines(dense_rl, select_rl),
        "roofline_publish": publish_rl,
        "kernel_ms": {"dense": ms_dense, "publish": ms_publish, "select": ms_select},
        "e2e": {"value": e2e_val / world, "unit": "ms", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": head_launches(args.steps, world),
        "clocks": clk.summary(),
        "wall_s": wall,
        "dev_err": err,
        "secondary": secondary,
        "cpu_baseline": cpu_head,
    }
    emit_line(line, rank)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def measure_secondary(cid, args, stream, flush, world, rank, peaks, tpk):
    """One of the standard workloads beside the headline chunk: the decode
    batches (rows/s, HBM-bound: their pools exceed L2) and the 4096-row
    prefill chunk (every row keeps all its blocks: the five layers score
    every position, tensor-bound), each with the oracle's CPU baseline."""
    r = measure(cid, max(3, args.steps // 2), 3, stream, flush)
    wl = r["wl"]
    mst, msd, mss = (statistics.mean(r[k]) for k in ("t_step", "t_dense", "t_select"))
    msg = graph_step_ms(r["step"], max(3, args.steps // 2), stream, flush)
    f, b, _ = algorithmic_counts(wl)
    positions, gathered, other = select_work(wl)
    rows = wl.rows
    line = {"workload": wl.name, "ms_per_step": mst, "dense_ms": msd, "select_ms": mss,
            "graph": {"ms_per_step": msg, "rows_per_s": world * rows / (msg * 1e-3),
                      "note": "the same step replayed as a CUDA graph"}}
    if wl.layout == 0:
        line = {"metric": "decode rows/s", "value": world * rows / (mst * 1e-3), "unit": "rows/s", **line}
        if cid != 0:  # the 4-row batch is latency-bound: no roofline claim
            hbm = peaks["hbm_gbs"]
            line["dense_roofline"] = {"bound": "hbm", "achieved": b / (msd * 1e-3) / 1e9, "peak": hbm,
                                      "unit": "GB/s", "frac": b / (msd * 1e-3) / 1e9 / hbm, "bytes": b}
            sb = gathered + other
            line["select_roofline"] = {"bound": "hbm", "achieved": sb / (mss * 1e-3) / 1e9, "peak": hbm,
                                       "unit": "GB/s", "frac": sb / (mss * 1e-3) / 1e9 / hbm, "bytes": sb,
                                       "launches": r["launches"] - 2,
                                       "note": "candidate K gathered by the five layers' selects (pools larger "
                                               "than L2: from HBM) plus per-row bytes / select time"}
            line["step_roofline"] = {"bound": "hbm", "achieved": (b + sb) / (mst * 1e-3) / 1e9, "peak": hbm,
                                     "unit": "GB/s", "frac": (b + sb) / (mst * 1e-3) / 1e9 / hbm}
        unit = "rows/s"
    else:
        peak, src = tpk["fp8"]
        line = {"metric": "prefill chunk ms", "value": mst, "unit": "ms", "rows_per_s": world * rows / (mst * 1e-3),
                **line}
        line["select_roofline"] = tensor_roofline(2 * 64 * 128 * positions, mss, len(wl.layers), peak, src)
        line["l2_gather"] = l2_gather(gathered, mss)
        unit = "ms"
    line["dev_err"] = int(r["step"].dev_err.item())
    if rank == 0 and not args.no_cpu:
        line["cpu_baseline"] = cpu_baseline(wl, unit)
    del r
    return line


def rooflines(a, b):
    """The kernel with the larger share of the step is "roofline" (the
    dominant kernel), the other "roofline_other"."""
    first, second = (a, b) if a["ms_per_step"] >= b["ms_per_step"] else (b, a)
    return {"roofline": first, "roofline_other": second}


# DRAM bytes (read + write) per launch from ncu captures of the headline chunk
# at full size (one-pass metrics), with the hash of the kernel's sources; a
# figure is reported only while the sources still match.
RECORDED_TRAFFIC = {
    # mean of the five launches of a step: 225.2 MB read (the pool once, queries, ids) + 26.9 MB written
    "select_kernel": {"bytes_per_launch": 252.1e6, "sources": ("sparse_tc.cu", "ci_common.cuh", "sm103_ptx.cuh"),
                      "sha256": "260b09aec96763ecf42d977280a92a910bd2309dad15b89c665636806668752d"},
    # 137.1 MB read (pool, queries) + 2051.5 MB written (keys)
    "dense_amax8_kernel": {"bytes_per_launch": 2188.6e6, "sources": ("dense_tc.cu", "ci_common.cuh", "sm103_ptx.cuh"),
                           "sha256": "e7a0a53ef52619e6c2f869174c0322e76cbccb91a0ee54be08619ca4e673a5da"},
    # 2121.6 MB read (keys) + 238.2 MB written (the two tables, 168 MB, and write-backs)
    "publish_kernel": {"bytes_per_launch": 2359.8e6, "sources": ("publish.cu", "ci_common.cuh", "sm103_ptx.cuh"),
                       "sha256": "6d66dc4b040bae252832b53368b45cd214d0a5a28c7c257b3d2b8fa12b54ba11"},
}


def _sources_sha(files):
    import hashlib

    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "two_level_sparse_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def recorded_traffic(kernel):
    rec = RECORDED_TRAFFIC[kernel]
    if rec["sha256"] is None or rec["sha256"] != _sources_sha(rec["sources"]):
        return None
    return rec["bytes_per_launch"]


def head_launches(steps, world):
    # per step of the 16384-row chunk: dense 1 + publish 1 (K and P + 1 together) + select 5 (one per layer)
    return steps * 7


if __name__ == "__main__":
    sys.exit(main())
