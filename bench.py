"""Benchmark: query rows/s of the fused block-sparse paged decode on one GB300,
and the HBM roofline fraction of its dominant kernel (the index-K scan).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...   # the CPU oracle on the host cores

A step = one msa_decode call (index score -> top-k + page-16 table ->
sparse paged attention) over the whole synthetic batch, inputs resident in
HBM.  L2 is flushed (a 512 MiB write, then a 256 MiB read) between timed
steps, outside the timed events.  Under torchrun each rank runs its own
independent batch (requests are independent; no collective on the data
path) and rank 0 prints one JSON line with the max-over-ranks time.

The line's headline keys are the 64-request decode (the workload the 70 %
roofline target names).  At N = 1 the same line also carries `per_workload`:
every other synthetic workload (tiny, batched, speculative, chunked
prefill, plus the FP8 index-K and sparse-MLA variants) timed the same way,
each with the median and mean of >= 100 graph replays, per-kernel times
and roofline fractions, an end-to-end figure and the oracle on the host
cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "query rows/s for fused index-topk+sparse paged decode; % of HBM roofline"
MLA_METRIC = "query rows/s for sparse MLA decode with sinks; % of HBM roofline"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
# the GB300's nominal HBM3e bandwidth (the "~8 TB/s" roofline); fractions are
# reported against it next to the measured copy rate
NOMINAL_HBM_GBS = 7900.0
L2_FLUSH_BYTES = 512 << 20
MEDIAN_ITERS = 100  # graph replays behind every median
EXTRA_E2E_ITERS = 20
EXTRA_KERNEL_ITERS = 20
EXTRA_CPU_BUDGET_S = 3.0
W_SEED = {"tiny_decode": 1, "batched_decode": 2, "speculative_decode": 3,
          "large_batch_decode": 4, "chunked_prefill": 5, "large_batch_decode_fp8_index": 6,
          "sparse_mla_decode": 7, "sparse_mla_decode_fp8": 8}
MLA_WORKLOADS = {"sparse_mla_decode": W.sparse_mla_decode,
                 "sparse_mla_decode_fp8": W.sparse_mla_decode_fp8}
EXTRA_WORKLOADS = ("tiny_decode", "batched_decode", "speculative_decode", "chunked_prefill",
                   "large_batch_decode_fp8_index", "sparse_mla_decode", "sparse_mla_decode_fp8")


# ---------------------------------------------------------------- bytes model

def algorithmic_bytes(w, topk_idx: np.ndarray) -> dict:
    """Bytes (and FLOPs) the method must move for one call, per kernel and in
    total: index-K read once per request, queries, block tables, the
    selected K/V (+ per-token scales) counted once per request over the
    union of its rows' selected blocks (a block selected by several rows of a
    request is read from HBM once), the tables, O and LSE.  Scores are
    intermediates.  FLOPs: the causal index dot products, and QK^T plus PV
    over each row's selected tokens."""
    seq = w.seq_lens
    nb_req = (seq + 127) // 128
    N = w.num_rows
    if getattr(w, "index_dtype", 0) == W.KV_FP8:  # e4m3 codes (+ fp32 per-token scales)
        idx_k = int(seq.sum()) * w.index_heads * (w.index_dim + (4 if w.idx_k_scale is not None
                                                                   else 0))
    else:
        idx_k = int(seq.sum()) * w.index_heads * w.index_dim * 2
    idx_q = N * w.index_heads * w.index_dim * 2
    bt = int(nb_req.sum()) * 4
    q = N * w.hq * w.head_dim * 2
    kv_elem = 1 if w.kv_dtype == W.KV_FP8 else 2
    toks = 0
    row_tokens = 0  # sum over rows of the tokens each row attends to
    score_flops = 0
    score_reads = 0  # the top-k's reads of each row's candidate scores
    for rq in range(len(seq)):
        r0, r1 = int(w.cu_seqlens_q[rq]), int(w.cu_seqlens_q[rq + 1])
        seen = {}
        for r in range(r0, r1):
            L = int(w.context_lens[rq]) + (r - r0) + 1  # tokens row r sees
            score_flops += 2 * L * w.index_heads * w.index_dim
            score_reads += 4 * ((L + 127) // 128)
            for b in topk_idx[r]:
                if b >= 0:
                    n = min(128, L - 128 * int(b))
                    row_tokens += n
                    seen[int(b)] = max(seen.get(int(b), 0), n)
        toks += sum(seen.values())
    kv = toks * w.hkv * w.head_dim * kv_elem * 2
    if w.scale_mode == W.SCALE_PER_TOKEN_HEAD:
        kv += toks * w.hkv * 4 * 2
    k = w.topk
    tables = N * (k * 4 + 8 * k * 4 + 4)
    out = N * (w.hq * w.head_dim * 2 + w.hq * 4)
    score = idx_k + idx_q + bt  # what the index-score kernel must read
    total = score + q + kv + tables + out
    return dict(score_kernel=score, attention=q + kv + out, topk=score_reads + bt + tables,
                total=total, index_k=idx_k, kv=kv, score_flops=score_flops,
                attn_flops=4 * row_tokens * w.hq * w.head_dim)


# ---------------------------------------------------------------- environment

def read_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return dict(hbm=float(d["hbm_gbs"]), bf16=float(d["bf16_tflops"]),
                    bf16_sustained=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                    source="measured")
    except Exception:
        return dict(hbm=FALLBACK_HBM_GBS, bf16=FALLBACK_BF16_TFLOPS,
                    bf16_sustained=FALLBACK_BF16_TFLOPS, source="fallback")


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "block_sparse_paged_02_gb300", "csrc")
    for name in ("index_score.cu", "msa_internal.cuh"):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def read_traffic(workload: str):
    """dram bytes per launch of the score kernel from the committed ncu
    summary, or None if the kernel changed since it was captured."""
    path = os.path.join(ROOT, "profiles", "score_kernel_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        ent = d.get(workload)
        if ent and ent.get("source_hash") == kernel_source_hash():
            return int(ent["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


# spin-kernel length (SM cycles, ~0.2 ms at 2 GHz) that covers the host's
# enqueue of one call in the per-kernel timing pass
GATE_CYCLES = 400_000


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for name, val in zip(names, parts[4:8]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def rank_seed(workload: str, rank: int) -> int:
    """Seed of a rank's batch: rank 0 draws the named workload itself, every
    other rank an independent batch of the same shape."""
    return W_SEED[workload] + 1000 * rank


def workload_config(w):
    seq = w.seq_lens
    return {"workload": w.name, "requests": w.num_reqs, "rows": w.num_rows,
            "query_heads": w.hq, "kv_heads": w.hkv, "head_dim": w.head_dim,
            "index_dim": w.index_dim, "topk": w.topk,
            "index_k": ("fp8_e4m3" + (" + per-token scales" if w.idx_k_scale is not None else "")
                        if getattr(w, "index_dtype", 0) == W.KV_FP8 else "bf16"),
            "kv": "fp8_e4m3" if w.kv_dtype == W.KV_FP8 else "bf16",
            "scales": ["none", "scalar", "per_token_head"][w.scale_mode],
            "sinks": w.sinks is not None, "context_tokens": int(seq.sum()),
            "median_context": float(np.median(seq)),
            "l2": "flushed between steps (512 MiB write, then 256 MiB read)"}


def mla_config(w):
    counts = np.diff(w.kv_indptr)
    dt = lambda a: "fp8_e4m3 + scalar scale" if a.dtype == np.uint8 else "bf16"
    return {"workload": w.name, "rows": w.num_rows, "heads": w.heads, "dqk": w.dqk, "dv": w.dv,
            "cache_tokens": w.num_tokens, "tokens_per_row": int(np.median(counts)),
            "kv": dt(w.kv_cache), "q": dt(w.q), "sinks": w.sinks is not None,
            "l2": "flushed between steps (512 MiB write, then 256 MiB read)"}


# ------------------------------------------------------------- oracle (CPU)

def cpu_oracle_run(w, budget_s: float = 12.0, max_reps: int = 1 << 20, rows=None):
    """The fp64 C oracle on the host cores over the workload (or a sample of
    its rows, each as a one-row request at its own position), timed."""
    import oracle
    oracle.build()
    threads = oracle.default_threads()
    sub = w if rows is None else W.row_subset(w, rows)
    reps, t0 = 0, time.perf_counter()
    while True:
        oracle.decode(sub, nthreads=threads)
        reps += 1
        el = time.perf_counter() - t0
        if reps >= max_reps or el >= budget_s:
            break
    what = (f"full {w.name} batch ({w.num_rows} rows)" if rows is None else
            f"{sub.num_rows} of the {w.num_rows} rows of {w.name} (every "
            f"{max(1, w.num_rows // sub.num_rows)}th)")
    return dict(value=sub.num_rows * reps / el, unit="rows/s", cores=threads, kind="oracle",
                sample=f"{reps} x {what}, fp64 C oracle, {threads} threads, {el:.2f} s")


def cpu_rows_sample(w):
    """Rows the oracle times for a workload: all of them, except for batches
    of thousands of rows, where an evenly spaced sample keeps it to seconds."""
    if w.num_rows <= 64:
        return None
    return np.arange(0, w.num_rows, w.num_rows // 64)


def mla_bytes(w) -> dict:
    """Bytes and FLOPs of one sparse-MLA call: each row's distinct latent rows
    (1152 B bf16 / 576 B e4m3: read once however often listed), queries,
    token lists, outputs."""
    N, H = w.num_rows, w.heads
    toks = 0
    for r in range(N):
        toks += len(np.unique(w.kv_indices[w.kv_indptr[r]:w.kv_indptr[r + 1]]))
    counts = np.diff(w.kv_indptr).astype(np.int64)
    kv_b = 1 if w.kv_cache.dtype == np.uint8 else 2
    q_b = 1 if w.q.dtype == np.uint8 else 2
    total = (toks * w.dqk * kv_b + N * H * w.dqk * q_b + N * H * (w.dv * 2 + 4)
             + int(counts.sum()) * 4 + (N + 1) * 4)
    flops = int(counts.sum()) * H * (w.dqk + w.dv) * 2
    return dict(total=total, flops=flops)


def mla_cpu_run(w, budget_s: float = 12.0, rows: int = 16):
    import oracle
    oracle.build()
    threads = oracle.default_threads()
    sub = min(rows, w.num_rows)
    ip = w.kv_indptr[: sub + 1]
    reps, t0 = 0, time.perf_counter()
    while True:
        oracle.sparse_mla(w.q[:sub], w.kv_cache, ip, w.kv_indices[: int(ip[-1])], w.dv,
                          sinks=w.sinks, softmax_scale=w.softmax_scale, nthreads=threads,
                          q_scale=w.q_scale, kv_scale=w.kv_scale)
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    return dict(value=sub * reps / el, unit="rows/s", cores=threads, kind="oracle",
                sample=f"{reps} x the first {sub} rows of {w.name}, fp64 C oracle, "
                f"{threads} threads, {el:.2f} s")


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    if args.workload in MLA_WORKLOADS:
        w = MLA_WORKLOADS[args.workload](seed=rank_seed(args.workload, 0))
        run_once = lambda: mla_cpu_run(w, budget_s=0.0, rows=w.num_rows)
        metric, config, rows = MLA_METRIC, mla_config(w), w.num_rows
        sample = f"full {w.name} batch per step ({w.num_rows} rows)"
    else:
        w = W.NAMED[args.workload](seed=rank_seed(args.workload, 0))
        pick = cpu_rows_sample(w)
        run_once = lambda: cpu_oracle_run(w, budget_s=0.0, max_reps=1, rows=pick)
        metric, config = METRIC, workload_config(w)
        rows = w.num_rows if pick is None else len(pick)
        sample = (f"full {w.name} batch per step ({w.num_rows} rows)" if pick is None else
                  f"{rows} evenly spaced rows of {w.name} per step")
    times = []
    for _ in range(args.warmup):
        run_once()
    for _ in range(args.steps):
        t0 = time.perf_counter()
        run_once()
        times.append(time.perf_counter() - t0)
    import oracle
    total = sum(times)
    value = rows * args.steps / total
    line = {"impl": "reference", "metric": metric, "value": value, "unit": "rows/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config,
            "cpu_baseline": {"value": value, "unit": "rows/s", "cores": oracle.default_threads(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


# ------------------------------------------------------------- GPU helpers

class Gpu:
    """The device, stream, L2 flush and event helpers of one rank."""

    def __init__(self, local: int, flush: bool = True):
        import torch
        self.torch = torch
        torch.cuda.set_device(local)
        self.dev = f"cuda:{local}"
        self.local = local
        self.stream = torch.cuda.current_stream()
        self.flush = (torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=self.dev)
                      if flush else None)
        self.rbuf = (torch.ones(L2_FLUSH_BYTES // 2, dtype=torch.uint8, device=self.dev)
                     if flush else None)

    def ev(self):
        return self.torch.cuda.Event(enable_timing=True)

    def flush_l2(self, i):
        # write a buffer larger than L2, then read another one so that no dirty
        # lines are left for the timed kernels to write back
        self.flush.fill_(i & 0xff)
        self.rbuf.sum(dtype=self.torch.int32)

    def capture(self, fn):
        """fn(stream) captured once into a CUDA graph (the library is
        graph-capturable: no host sync, no allocation, no host copy)."""
        torch = self.torch
        s = torch.cuda.Stream(device=self.dev)
        s.wait_stream(torch.cuda.current_stream())
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            fn(s)
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        return g

    def time_steps(self, step, n):
        """Per-step device times (ms) of n calls of step(), L2 flushed before
        each, events on the launching stream."""
        marks = [(self.ev(), self.ev()) for _ in range(n)]
        for i in range(n):
            self.flush_l2(i)
            marks[i][0].record(self.stream)
            step()
            marks[i][1].record(self.stream)
        self.torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in marks]

    def e2e(self, case, host_names, step, steps, warmup):
        """End to end through the public call: the per-step inputs copied in
        from pinned host memory and O/LSE copied back, inside the events.  A
        case with packed step buffers (DeviceCase.pack_step_inputs) moves
        them by one copy each way; otherwise one copy per named tensor."""
        torch = self.torch
        packed = getattr(case, "step_inputs", None) is not None
        if packed:
            ins = [(case.step_inputs, case.step_inputs.cpu().pin_memory())]
            outs = [(case.step_outputs,
                     torch.empty_like(case.step_outputs, device="cpu").pin_memory())]
        else:
            ins = [(getattr(case, n), getattr(case, n).cpu().pin_memory()) for n in host_names]
            outs = [(t, torch.empty_like(t, device="cpu").pin_memory()) for t in (case.out, case.lse)]
        h2d = sum(h.numel() * h.element_size() for _, h in ins)
        d2h = sum(h.numel() * h.element_size() for _, h in outs)
        marks = [(self.ev(), self.ev()) for _ in range(steps)]
        for i in range(warmup + steps):
            self.flush_l2(i)
            if i >= warmup:
                marks[i - warmup][0].record(self.stream)
            for d, h in ins:
                d.copy_(h, non_blocking=True)
            step()
            for d, h in outs:
                h.copy_(d, non_blocking=True)
            if i >= warmup:
                marks[i - warmup][1].record(self.stream)
        torch.cuda.synchronize()
        return sum(a.elapsed_time(b) for a, b in marks), h2d, d2h


    def e2e_pipelined(self, case, step, steps, warmup):
        """End to end through the public call, run as a serving loop runs it:
        the case holds two sets of step buffers (DeviceCase.pack_step_inputs
        (sets=2)); step i's inputs are copied in from pinned host memory on
        one stream while step i - 1 runs, and its O / LSE copied back on
        another while step i + 1 runs, each copy waiting for the step that
        last used its buffer.  Every step moves its own inputs and outputs;
        the time is the whole loop's, from the first copy in to the last copy
        out.  No L2 flush: each step of the 64-request batch streams 407 MB
        of index-K, more than the L2 holds."""
        torch = self.torch
        sets = case._sets
        n = len(sets)
        hin = [st["step_inputs"].cpu().pin_memory() for st in sets]
        hout = [torch.empty_like(st["step_outputs"], device="cpu").pin_memory() for st in sets]
        cin = torch.cuda.Stream(device=self.dev)
        cout = torch.cuda.Stream(device=self.dev)
        s = self.stream
        done = [self.ev() for _ in range(n)]
        arrived = [self.ev() for _ in range(n)]
        read = [self.ev() for _ in range(n)]
        start, end = self.ev(), self.ev()
        total = warmup + steps
        torch.cuda.synchronize()
        for i in range(total):
            b = i % n
            if i == warmup:
                if i > 0:
                    s.wait_event(read[(i - 1) % n])  # the warm-up copies are out
                start.record(s)
                cin.wait_event(start)
            if i >= n:
                cin.wait_event(done[b])  # step i - n has finished with these inputs
            with torch.cuda.stream(cin):
                sets[b]["step_inputs"].copy_(hin[b], non_blocking=True)
            arrived[b].record(cin)
            s.wait_event(arrived[b])
            if i >= n:
                s.wait_event(read[b])  # step i - n's O / LSE have been copied out
            case.use_step_set(b)
            step(s)
            done[b].record(s)
            cout.wait_event(done[b])
            with torch.cuda.stream(cout):
                hout[b].copy_(sets[b]["step_outputs"], non_blocking=True)
            read[b].record(cout)
        s.wait_event(read[(total - 1) % n])
        end.record(s)
        torch.cuda.synchronize()
        case.use_step_set(0)
        h2d = hin[0].numel() * hin[0].element_size()
        d2h = hout[0].numel() * hout[0].element_size()
        return start.elapsed_time(end), h2d, d2h


DECODE_INPUTS = ("q", "idx_q", "cu_q", "cu_k", "ctx", "bt")


def decode_kernel_times(gpu, case, msa, iters):
    """The same step eagerly with events after each stage (events recorded
    inside a graph cannot be timed), and the number of kernels the call
    launches (the library's own count).  When the score kernel selects the
    blocks there is no top-k kernel: its interval is empty and the score
    kernel's includes the selection."""
    e = [gpu.ev() for _ in range(4)]
    trace = msa.make_trace(e[1], e[2], e[3])
    score, topk, attn = [], [], []
    for i in range(iters):
        gpu.flush_l2(i)
        # keep the GPU busy (a spin kernel, no memory traffic) while the host
        # enqueues the call, so that host-side launch time never shows up as
        # a gap inside the first kernel's interval
        gpu.torch.cuda._sleep(GATE_CYCLES)
        e[0].record(gpu.stream)
        case.decode(keep_tables=False, trace=trace)
        gpu.torch.cuda.synchronize()
        score.append(e[0].elapsed_time(e[1]))
        topk.append(e[1].elapsed_time(e[2]))
        attn.append(e[2].elapsed_time(e[3]))
    return {"index_score": score, "topk_table": topk, "sparse_attn": attn}, int(trace.kernels)


def kernel_rooflines(nbytes, kernel_ms, peaks):
    """Per kernel: mean time, algorithmic bytes and FLOPs, and the fraction
    of the measured HBM copy rate and of the bf16 tensor peak (burst) they
    reach; the kernel's bound is the larger fraction."""
    work = {"index_score": (nbytes["score_kernel"], nbytes["score_flops"]),
            "topk_table": (nbytes["topk"], 0),
            "sparse_attn": (nbytes["attention"], nbytes["attn_flops"])}
    out = {}
    for name, (b, f) in work.items():
        ms = statistics.mean(kernel_ms[name])
        if ms < 1e-4:  # no such kernel (the selection ran inside the score kernel)
            out[name] = {"ms": ms, "algorithmic_bytes": b, "flops": f, "fused": True}
            continue
        gbs = b / (ms / 1e3) / 1e9
        tfs = f / (ms / 1e3) / 1e12
        hf, tf = gbs / peaks["hbm"], tfs / peaks["bf16"]
        out[name] = {"ms": ms, "algorithmic_bytes": b, "flops": f, "achieved_gbs": gbs,
                     "achieved_tflops": tfs, "hbm_frac": hf, "tensor_frac": tf,
                     "bound": "tensor" if tf > hf else "hbm"}
    return out


def step_roofline(total_bytes, step_ms, peaks):
    gbs = total_bytes / (step_ms / 1e3) / 1e9
    return {"algorithmic_bytes": total_bytes, "achieved_gbs": gbs, "frac": gbs / peaks["hbm"],
            "frac_nominal": gbs / NOMINAL_HBM_GBS, "nominal_gbs": NOMINAL_HBM_GBS}


def measure_extra_decode(gpu, msa, name):
    """One more decode workload: >= 100 graph replays (median and mean),
    per-kernel times, end to end, oracle on the host cores."""
    w = W.NAMED[name](seed=rank_seed(name, 0))
    case = msa.DeviceCase(w, device=gpu.dev)
    for i in range(3):
        gpu.flush_l2(i)
        case.decode(keep_tables=False)
    gpu.torch.cuda.synchronize()
    if int(case.status.item()) != 0:
        raise RuntimeError(f"{name}: device status {int(case.status.item())}")
    g = gpu.capture(lambda s: case.decode(keep_tables=False, stream=s))
    steps = gpu.time_steps(g.replay, MEDIAN_ITERS)
    kern, nk = decode_kernel_times(gpu, case, msa, EXTRA_KERNEL_ITERS)
    case.decode()
    gpu.torch.cuda.synchronize()
    topk_sel = case.topk_idx[: w.num_rows].cpu().numpy()
    case.pack_step_inputs()  # one copy in and one out per step (after the graph timing)
    e2e_ms, h2d, d2h = gpu.e2e(case, DECODE_INPUTS, lambda: case.decode(keep_tables=False),
                               EXTRA_E2E_ITERS, 3)
    peaks = read_peaks()
    nb = algorithmic_bytes(w, topk_sel)
    mean, med = statistics.mean(steps), statistics.median(steps)
    kr = kernel_rooflines(nb, kern, peaks)
    dom = max(kr, key=lambda k: kr[k]["ms"])
    return {
        "config": workload_config(w),
        "ms_per_step": mean, "ms_per_step_median": med, "iters": len(steps),
        "value": w.num_rows / (mean / 1e3), "value_median": w.num_rows / (med / 1e3),
        "unit": "rows/s",
        "step_roofline": step_roofline(nb["total"], med, peaks),
        "kernels": kr, "dominant_kernel": dom,
        "dominant_kernel_frac": max(kr[dom]["hbm_frac"], kr[dom]["tensor_frac"]),
        "dominant_bound": kr[dom]["bound"],
        "e2e": {"value": w.num_rows * EXTRA_E2E_ITERS / (e2e_ms / 1e3), "unit": "rows/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches_per_step": nk,
        "cpu_baseline": cpu_oracle_run(w, budget_s=EXTRA_CPU_BUDGET_S, rows=cpu_rows_sample(w)),
        "peak_source": peaks["source"],
    }


def measure_mla(gpu, msa, name, seed, steps_n, warmup, cpu_budget):
    """Sparse MLA decode: graph replays, end to end, oracle on the host."""
    w = MLA_WORKLOADS[name](seed=seed)
    case = msa.MlaCase(w, device=gpu.dev)
    for i in range(warmup):
        gpu.flush_l2(i)
        case.decode()
    gpu.torch.cuda.synchronize()
    if int(case.status.item()) != 0:
        raise RuntimeError(f"device status {int(case.status.item())} on a clean workload")
    g = gpu.capture(lambda s: case.decode(stream=s))
    steps = gpu.time_steps(g.replay, steps_n)
    e2e_ms, h2d, d2h = gpu.e2e(case, ("q", "indptr", "indices"), case.decode, steps_n, warmup)
    peaks = read_peaks()
    nb = mla_bytes(w)
    mean, med = statistics.mean(steps), statistics.median(steps)
    achieved = nb["total"] / (med / 1e3) / 1e9
    tflops = nb["flops"] / (med / 1e3) / 1e12
    return w, steps, {
        "config": mla_config(w),
        "ms_per_step": mean, "ms_per_step_median": med, "iters": len(steps),
        "value": w.num_rows / (mean / 1e3), "value_median": w.num_rows / (med / 1e3),
        "unit": "rows/s",
        "roofline": {"bound": "hbm", "kernel": "sparse_mla", "achieved": achieved,
                     "peak": peaks["hbm"], "unit": "GB/s", "frac": achieved / peaks["hbm"],
                     "frac_nominal": achieved / NOMINAL_HBM_GBS, "peak_source": peaks["source"],
                     "traffic": None, "algorithmic_bytes_per_launch": nb["total"],
                     "avg_launch_ms": med},
        "tensor": {"achieved_tflops": tflops, "peak_bf16_tflops": peaks["bf16"],
                   "frac": tflops / peaks["bf16"],
                   "note": "mma.sync m16n8k16 " + ("f16 (e4m3 converted exactly)"
                                                   if w.kv_cache.dtype == np.uint8 else "bf16")},
        "dominant_kernel": "sparse_mla", "dominant_kernel_frac": achieved / peaks["hbm"],
        "e2e": {"value": w.num_rows * steps_n / (e2e_ms / 1e3), "unit": "rows/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches_per_step": 1,
        "cpu_baseline": mla_cpu_run(w, budget_s=cpu_budget),
    }


# ------------------------------------------------------------------- arms

def run_mla_gpu(args):
    import torch.distributed as dist

    import block_sparse_paged_02_gb300 as msa

    ws, rank, local = dist_env()
    if ws > 1:
        dist.init_process_group("nccl")
    gpu = Gpu(local, flush=not args.profile)
    if args.profile:
        # plain run for profilers: warm-up + K steps, nothing else
        w = MLA_WORKLOADS[args.workload](seed=rank_seed(args.workload, rank))
        case = msa.MlaCase(w, device=gpu.dev)
        for _ in range(args.warmup + args.steps):
            case.decode()
        gpu.torch.cuda.synchronize()
        print(json.dumps({"profile_run": w.name, "status": int(case.status.item())}))
        return 0
    with ClockSampler(local) as clocks:
        if ws > 1:
            dist.barrier()
        w, steps, rep = measure_mla(gpu, msa, args.workload, rank_seed(args.workload, rank),
                                    args.steps, args.warmup, 12.0 if rank == 0 else 0.0)
    total_ms = sum(steps)
    if ws > 1:
        t = gpu.torch.tensor([total_ms], device=gpu.dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        total_ms = float(t.item())
        if rank != 0:
            dist.destroy_process_group()
            return 0
    line = {"metric": MLA_METRIC, "value": w.num_rows * ws * args.steps / (total_ms / 1e3),
            "unit": "rows/s", "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": total_ms / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16 / fp32 acc", "data": "synthetic",
            "config": rep["config"], "roofline": rep["roofline"], "tensor": rep["tensor"],
            "e2e": rep["e2e"], "gpu_launches": args.steps, "launch": "cuda_graph",
            "clocks": clocks.summary(), "cpu_baseline": rep["cpu_baseline"]}
    print(json.dumps(line))
    if ws > 1:
        dist.destroy_process_group()
    return 0


def run_gpu(args):
    import torch
    import torch.distributed as dist

    import block_sparse_paged_02_gb300 as msa

    ws, rank, local = dist_env()
    if ws > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    gpu = Gpu(local, flush=not args.profile)
    # weak scaling: every rank owns its own batch of independent requests
    w = W.NAMED[args.workload](seed=rank_seed(args.workload, rank))
    case = msa.DeviceCase(w, device=gpu.dev)

    def barrier():
        if ws > 1:
            dist.barrier()

    if args.profile:
        # plain run for profilers: warm-up + K steps, nothing else
        for _ in range(args.warmup + args.steps):
            case.decode(keep_tables=False)
        torch.cuda.synchronize()
        print(json.dumps({"profile_run": w.name, "status": int(case.status.item())}))
        return 0

    for i in range(args.warmup):
        gpu.flush_l2(i)
        case.decode(keep_tables=False)
    torch.cuda.synchronize()
    if int(case.status.item()) != 0:
        raise RuntimeError(f"device status {int(case.status.item())} on a clean workload")

    launch_mode = "cuda_graph"
    try:
        g_main = gpu.capture(lambda s: case.decode(keep_tables=False, stream=s))
        run_step = g_main.replay
    except Exception as exc:  # graph capture unavailable: time eager launches
        launch_mode = f"eager ({type(exc).__name__})"
        run_step = lambda: case.decode(keep_tables=False)

    # ---- timed: K steps, per-step events on the launching stream
    barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        step_ms = gpu.time_steps(run_step, args.steps)
        barrier()
        # the median behind the headline: >= 100 more replays, timed the same way
        med_ms = gpu.time_steps(run_step, max(MEDIAN_ITERS, args.steps))
    total_ms = sum(step_ms)
    if ws > 1:
        t = torch.tensor([total_ms], device=gpu.dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        total_ms = float(t.item())

    kern, nk = decode_kernel_times(gpu, case, msa, args.steps)
    case.decode()
    torch.cuda.synchronize()
    topk_sel = case.topk_idx[: w.num_rows].cpu().numpy()
    # one copy in and one out per step (after the graph timing): a serving
    # loop's pipeline over two buffer sets, and each step on its own with the
    # L2 flushed before it
    case.pack_step_inputs(sets=2)
    e2e_ms, h2d, d2h = gpu.e2e_pipelined(
        case, lambda s: case.decode(keep_tables=False, stream=s), args.steps, args.warmup)
    e2e_serial_ms, _, _ = gpu.e2e(case, DECODE_INPUTS, lambda: case.decode(keep_tables=False),
                                  args.steps, args.warmup)
    if ws > 1:
        t = torch.tensor([e2e_ms, e2e_serial_ms], device=gpu.dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        e2e_ms, e2e_serial_ms = (float(x) for x in t.tolist())
        if rank != 0:
            dist.destroy_process_group()
            return 0

    rows_total = w.num_rows * ws * args.steps
    value = rows_total / (total_ms / 1e3)
    peaks = read_peaks()
    nbytes = algorithmic_bytes(w, topk_sel)
    kr = kernel_rooflines(nbytes, kern, peaks)
    score_avg = kr["index_score"]["ms"]
    achieved = nbytes["score_kernel"] / (score_avg / 1e3) / 1e9
    step_avg = total_ms / args.steps
    line = {
        "metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": step_avg, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "fp8_e4m3 kv / bf16 q / fp32 acc"
        if w.kv_dtype == W.KV_FP8 else "bf16 / fp32 acc", "data": "synthetic",
        "config": workload_config(w),
        "roofline": {"bound": "hbm", "kernel": "index_score", "achieved": achieved,
                     "peak": peaks["hbm"], "unit": "GB/s", "frac": achieved / peaks["hbm"],
                     "frac_nominal": achieved / NOMINAL_HBM_GBS,
                     "peak_source": peaks["source"], "traffic": read_traffic(w.name),
                     "algorithmic_bytes_per_launch": nbytes["score_kernel"],
                     "avg_launch_ms": score_avg},
        "step_roofline": step_roofline(nbytes["total"], step_avg, peaks),
        "ms_per_step_median": statistics.median(med_ms), "median_iters": len(med_ms),
        "kernel_ms": {k: v["ms"] for k, v in kr.items()},
        "kernels": kr,
        "e2e": {"value": w.num_rows * ws * args.steps / (e2e_ms / 1e3), "unit": "rows/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "mode": "pipelined: step i's copy in and step i-1's copy out overlap a step, "
                        "two buffer sets, no L2 flush (407 MB of index-K per step)",
                "ms_per_step": e2e_ms / args.steps,
                "serial": {"value": w.num_rows * ws * args.steps / (e2e_serial_ms / 1e3),
                           "ms_per_step": e2e_serial_ms / args.steps,
                           "mode": "copy in, step, copy out; L2 flushed before each step"}},
        "gpu_launches": nk * args.steps,
        "launch": launch_mode,
        "clocks": clocks.summary(),
        "cpu_baseline": cpu_oracle_run(w),
    }
    if ws == 1 and not args.headline_only:
        # every other workload, measured the same way (one GPU only: under
        # torchrun the ranks time the headline batch alone)
        per = {}
        with ClockSampler(local) as extra_clocks:
            for name in EXTRA_WORKLOADS:
                if name == w.name:
                    continue
                if name in MLA_WORKLOADS:
                    per[name] = measure_mla(gpu, msa, name, rank_seed(name, 0), MEDIAN_ITERS, 3,
                                            EXTRA_CPU_BUDGET_S)[2]
                else:
                    per[name] = measure_extra_decode(gpu, msa, name)
        line["per_workload"] = per
        line["per_workload_clocks"] = extra_clocks.summary()
    print(json.dumps(line))
    if ws > 1:
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default="large_batch_decode",
                    choices=sorted(W.NAMED) + sorted(MLA_WORKLOADS))
    ap.add_argument("--headline-only", action="store_true",
                    help="time the named workload only (no per_workload section)")
    ap.add_argument("--profile", action="store_true",
                    help="plain warm-up + K decode steps for a profiler (no timing)")
    args = ap.parse_args(argv)
    args.warmup = max(3, args.warmup)  # at least 3 untimed warm-up steps
    if args.impl == "reference":
        return run_reference(args)
    if args.workload in MLA_WORKLOADS:
        return run_mla_gpu(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
