"""Benchmark of the sparse-attention step (metadata -> indexer logits -> top-k +
slot transform -> sparse MLA) on the method's five synthetic workloads; by
default the DeepSeek-V3.2-shaped bf16-KV decode batch (32 requests, seqlens
U{4096..32768}, page 64, indexer 64 heads x 128 e4m3, topk 2048, MLA 128 heads
d_qk 576 / d_v 512).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--config NAME] [--cpu-full]
    python bench.py --kv-write      # the KV-cache write-side kernels instead
    python bench.py --local-attn    # chunk-local dense attention (the second workload)

--config picks one of the five workloads (`workloads.CONFIG_NAMES`).  Every
stage is graded against its binding roofline: HBM bandwidth, or the tensor
cores (fp8 for the indexer, bf16 for the attention) where the stage's flops
take longer at peak than its bytes.  --cpu-full times the oracle on the full
CPU sample of the workload (every row; the chunked extend on its 260 sampled
rows) instead of a ~12 s bounded sample.

Prints ONE JSON line (rank 0).  Under torchrun every rank runs an independent
replica of the workload on its own GPU (replicas only: the path has no
exchange step) and `value` is all ranks' rows / the slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "sparse-MLA decode tokens/s + indexer/top-k µs per step; % of HBM/TC roofline"
WORKLOAD = "v32_decode_bf16"  # the workload the metric is quoted on
WORKLOADS = {
    "tiny_fp32_decode": "tiny fp32 decode: batch 2, seqlens {64,100}, page 16, indexer 4 heads x 32 fp32, topk 32, "
                        "MLA 4 heads kv_lora 64 + rope 16 (d_v 64) fp32, sm_scale 80^-0.5",
    "v32_decode_bf16": "DeepSeek-V3.2-shaped decode, bf16 KV: batch 32, seqlens U{4096..32768}, page 64 in random "
                       "order, indexer 64x128 e4m3 + fp32 row scale, weights N(0,1)/8, topk 2048, MLA 128 heads "
                       "d_qk 576 (512+64) d_v 512 bf16, sm_scale 192^-0.5",
    "fp8kv_decode_h16": "fp8-KV decode, 16 MLA heads: batch 128, seqlen 8192, page 64, indexer 64x128 e4m3, topk 2048, "
                        "latent e4m3 with per-128 fp32 scales + bf16 rope (656-byte rows), 1% latent outliers x20",
    "chunked_extend": "chunked extend: 4 sequences x (8192 prefix + 2048 new tokens), causal rows see 8193..10240 "
                      "tokens (clipped to topk 2048), page 64, indexer 64x128 e4m3, MLA 128 heads 576/512 bf16",
    "verify_long_fp8kv": "speculative target-verify, long context: batch 64 x 4 draft tokens, seqlens log-uniform "
                         "16384..131072, page 64, indexer 64x128 e4m3, topk 2048, MLA 128 heads 576/512 fp8 KV",
}
WORKLOAD_DESC = WORKLOADS[WORKLOAD]
DEFAULT_SEED = {"tiny_fp32_decode": 0, "v32_decode_bf16": 2, "fp8kv_decode_h16": 3, "chunked_extend": 4,
                "verify_long_fp8kv": 5}
L2_FLUSH_BYTES = 512 << 20


class L2Flush:
    """Between timed launches: write a buffer larger than L2 (every input line is
    evicted), then read a second buffer larger than L2, so that the write's dirty
    lines go back to HBM here and not inside the next timed region."""

    def __init__(self, dev):
        import torch
        self.w = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        self.r = torch.zeros(L2_FLUSH_BYTES // 8, dtype=torch.float32, device=dev)
        self.acc = torch.zeros((), dtype=torch.float32, device=dev)

    def zero_(self):
        import torch
        self.w.zero_()
        torch.sum(self.r, dim=0, out=self.acc)


# DRAM traffic per launch (dram__bytes_read.sum + dram__bytes_write.sum) of each
# stage's kernel from one ncu capture of a workload (profiles/ names the command),
# keyed by (workload, stage); a stage of two launches (the chunked top-k) sums them.
# Valid only while the kernel sources (comments aside) hash as they did at capture.
NCU_TRAFFIC = {
    ("v32_decode_bf16", "sparse_mla"): dict(bytes=int((81.312768 + 2.825984) * 1e6), sources=['sparse_mla_tc.cu', 'sm100.cuh'], sha="a9fcea53c576bb02"),
    ("v32_decode_bf16", "indexer"): dict(bytes=int((79.639040 + 1.755392) * 1e6), sources=['indexer_tc.cu', 'sm100.cuh'], sha="b418f8c7433f93b5"),
    ("v32_decode_bf16", "topk"): dict(bytes=int((4.744960) * 1e6), sources=['topk.cu'], sha="4c42535136830aa5"),
    ("v32_decode_bf16", "metadata"): dict(bytes=int((2.001152) * 1e6), sources=['metadata.cu'], sha="c41a2686c52610f5"),
    ("fp8kv_decode_h16", "sparse_mla"): dict(bytes=int((197.520640 + 3.252224) * 1e6), sources=['sparse_mla_tc.cu', 'sm100.cuh'], sha="a9fcea53c576bb02"),
    ("fp8kv_decode_h16", "indexer"): dict(bytes=int((140.075008 + 5.098752) * 1e6), sources=['indexer_tc.cu', 'sm100.cuh'], sha="b418f8c7433f93b5"),
    ("fp8kv_decode_h16", "topk"): dict(bytes=int((8.453888) * 1e6), sources=['topk.cu'], sha="4c42535136830aa5"),
    ("fp8kv_decode_h16", "metadata"): dict(bytes=int((2.157568) * 1e6), sources=['metadata.cu'], sha="c41a2686c52610f5"),
    ("chunked_extend", "indexer"): dict(bytes=int((79.824128 + 245.445888) * 1e6), sources=['indexer_tc.cu', 'sm100.cuh'], sha="b418f8c7433f93b5"),
    ("chunked_extend", "topk"): dict(bytes=int((302.840576 + 51.008768) * 1e6), sources=['topk.cu'], sha="4c42535136830aa5"),
    ("chunked_extend", "sparse_mla"): dict(bytes=int((1323.398 + 1042.790) * 1e6), sources=['sparse_mla_tc.cu', 'sm100.cuh'], sha="a9fcea53c576bb02"),
    ("verify_long_fp8kv", "sparse_mla"): dict(bytes=int((406.372352 + 81.999872) * 1e6), sources=['sparse_mla_tc.cu', 'sm100.cuh'], sha="a9fcea53c576bb02"),
    ("verify_long_fp8kv", "indexer"): dict(bytes=int((468.660224 + 47.524608) * 1e6), sources=['indexer_tc.cu', 'sm100.cuh'], sha="b418f8c7433f93b5"),
    ("verify_long_fp8kv", "topk"): dict(bytes=int((70.563584 + 1.356288 + 17.348608) * 1e6), sources=['topk.cu'], sha="4c42535136830aa5"),
    ("verify_long_fp8kv", "metadata"): dict(bytes=int((16.822528) * 1e6), sources=['metadata.cu'], sha="c41a2686c52610f5"),
    ("local_decode_c8192", "local_attention"): dict(bytes=int((642.419968 + 3.919616) * 1e6),
                                                    sources=["local_attention.cu", "sm100.cuh"], sha="921bc0c500fccc86"),
}


_COMMENT_OR_LITERAL = re.compile(r'//[^\n]*|/\*.*?\*/|"(?:\\.|[^"\\\n])*"|\'(?:\\.|[^\'\\\n])*\'', re.S)


def code_only(text: str) -> str:
    """C/C++/CUDA source without its comments, whitespace runs folded to one space
    (string and character literals kept as written): edits to comments alone do not
    change what a capture measured."""
    text = _COMMENT_OR_LITERAL.sub(lambda m: " " if m.group(0).startswith("/") else m.group(0), text)
    return re.sub(r"\s+", " ", text).strip()


def sources_sha(files) -> str:
    import hashlib
    m = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "deepseek_sparse_mla_indexer_gb300", "csrc", f), encoding="utf-8") as fh:
            m.update(code_only(fh.read()).encode())
    return m.hexdigest()[:16]


def ncu_traffic(workload: str, stage: str):
    """Measured bytes per launch, or None when there is no capture for this
    workload or the kernel has changed since the capture."""
    e = NCU_TRAFFIC.get((workload, stage))
    if e is None:
        return None
    return e["bytes"] if sources_sha(e["sources"]) == e["sha"] else None


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return dict(hbm_gbs=float(d["hbm_gbs"]), bf16_tflops=float(d["bf16_tflops"]),
                    bf16_tflops_sustained=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                    source="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0, source="fallback")


# ---------------------------------------------------------------- algorithmic work per stage

def algorithmic_work(wl, seqlens_expanded: np.ndarray, row_to_req=None, indices=None):
    """Bytes each stage must move and flops it must do, from the shapes alone.

    Data that rows of one request share is counted once: the indexer reads each
    request's key rows once (its longest row's worth) however many of its rows are
    scored against them, and the sparse MLA reads each distinct selected KV row once
    (`indices`, all rows; without it every row's selection is counted).  Flops count
    every row's own products."""
    L = seqlens_expanded.astype(np.int64)
    Lsum = int(L.sum())
    nsel = np.minimum(L, wl.topk)
    ps = wl.page_size
    idx_elem = 1 if wl.idx_dtype == W.DT_E4M3 else 4
    row_bytes = wl.kv_row_bytes
    qb = 2 if wl.q_dtype == W.DT_BF16 else 4
    dq = wl.d_latent + wl.d_rope
    r2q = np.arange(wl.R) if row_to_req is None else np.asarray(row_to_req)
    req_len = np.zeros(int(r2q.max()) + 1 if len(r2q) else 0, np.int64)
    np.maximum.at(req_len, r2q, L)
    if indices is not None:
        sel = np.asarray(indices).reshape(-1)
        kv_rows = int(np.unique(sel[sel >= 0]).size)
    else:
        kv_rows = int(nsel.sum())
    w = {}
    # the step's metadata reads each page's first slot and writes its page id (no copied
    # page_table_1: the top-k reads req_to_token through req_rows), plus the per-request
    # and per-row fields
    w["metadata"] = dict(bytes=wl.B * ((wl.W + ps - 1) // ps) * 4 * 2 + 40 * (wl.B + wl.R) + 4 * wl.B, flops=0)
    w["indexer"] = dict(bytes=int(req_len.sum()) * (wl.Di * idx_elem + 4) + Lsum * 4
                        + wl.R * wl.Hi * (wl.Di * idx_elem + 4) + int(((req_len + ps - 1) // ps).sum()) * 4,
                        flops=2 * wl.Hi * wl.Di * Lsum)
    w["topk"] = dict(bytes=Lsum * 4 + wl.R * wl.topk * 4 + int(nsel.sum()) * 4, flops=0)
    w["sparse_mla"] = dict(bytes=kv_rows * row_bytes + wl.R * wl.H * (dq + wl.d_latent) * qb
                           + wl.R * wl.H * 4 + wl.R * wl.topk * 4,
                           flops=2 * wl.H * int(nsel.sum()) * (dq + wl.d_latent))
    return w


def stage_roofline(wl, stage: str, work: dict, sec: float, peaks: dict) -> dict:
    """A stage's binding roofline: the larger of its bytes at the measured HBM copy
    bandwidth and its flops at the tensor-core peak of the precision it runs in
    (the indexer's e4m3 contraction at 2x the measured bf16 peak, the nominal fp8 to
    bf16 ratio; the attention's bf16 products at the measured bf16 peak).  fp32
    stages (the tiny workload) run on CUDA cores and are graded against HBM."""
    nbytes, flops = work["bytes"], work["flops"]
    t_hbm = nbytes / (peaks["hbm_gbs"] * 1e9)
    tc_name, tc_peak = None, None
    if stage == "indexer" and wl.idx_dtype == W.DT_E4M3:
        tc_name, tc_peak = "fp8 dense (2x measured bf16)", 2.0 * peaks["bf16_tflops"]
    elif stage == "sparse_mla" and wl.q_dtype == W.DT_BF16:
        tc_name, tc_peak = "bf16 dense (measured)", peaks["bf16_tflops"]
    t_tc = flops / (tc_peak * 1e12) if tc_peak else 0.0
    gbs = nbytes / sec / 1e9
    tfl = flops / sec / 1e12
    d = dict(us=round(sec * 1e6, 2), bytes=int(nbytes), flops=int(flops), gbs=round(gbs, 1), tflops=round(tfl, 2),
             hbm_frac=round(gbs / peaks["hbm_gbs"], 4))
    if tc_peak:
        d["tc_peak_tflops"] = round(tc_peak, 1)
        d["tc_frac"] = round(tfl / tc_peak, 4)
    d["bound"] = "tensor" if t_tc > t_hbm else "hbm"
    d["roofline_us"] = round(max(t_hbm, t_tc) * 1e6, 2)
    d["frac"] = round(max(t_hbm, t_tc) / sec, 4)
    return d


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples of SM clock / throttle reasons during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return dict(sm_mhz=None, sm_max_mhz=None, reasons=["nvidia-smi unavailable"], samples=0)
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
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
        return dict(sm_mhz=statistics.median(sm) if sm else None, sm_max_mhz=max(mx) if mx else None,
                    reasons=sorted(reasons), samples=len(sm))


# ---------------------------------------------------------------- timestamps inside a graph

_cudart = None


def record_external(event, stream):
    """Record `event` on `stream` as a timestamp node when the stream is being
    captured (cudaEventRecordWithFlags, cudaEventRecordExternal)."""
    global _cudart
    import ctypes
    if _cudart is None:
        _cudart = ctypes.CDLL("libcudart.so.13")
        _cudart.cudaEventRecordWithFlags.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_uint]
        _cudart.cudaEventRecordWithFlags.restype = ctypes.c_int
    rc = _cudart.cudaEventRecordWithFlags(ctypes.c_void_p(event.cuda_event), ctypes.c_void_p(stream.cuda_stream), 1)
    if rc != 0:
        raise RuntimeError(f"cudaEventRecordWithFlags failed ({rc})")


# ---------------------------------------------------------------- replicas

def replica_seed(rank: int, base: int = 2) -> int:
    """Each rank draws an independent batch of the same workload (rank 0 the
    workload's own seed)."""
    return base + 1000 * rank


def max_over_ranks(values, world: int):
    """Element-wise max of per-rank timings (the slowest rank sets the pace)."""
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64)
    if world > 1:
        import torch.distributed as dist
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t]


def replica_throughput(rows_per_rank: int, world: int, ms_per_step: float) -> float:
    """Rows of all ranks per second of the slowest rank's step."""
    return rows_per_rank * world / (ms_per_step * 1e-3)


# ---------------------------------------------------------------- our arm

def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist
    import deepseek_sparse_mla_indexer_gb300 as nsa
    from deepseek_sparse_mla_indexer_gb300.step import SparseAttentionStep

    name = args.config
    wl = W.config(name, seed=replica_seed(rank, DEFAULT_SEED[name]))  # an independent replica per rank
    # the oracle's CPU time is taken before the first GPU call (its worker threads
    # never share a process with a started CUDA context mid-flight)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(wl, full=args.cpu_full)

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    nsa.load()
    step = SparseAttentionStep(wl, dev)
    stream = torch.cuda.current_stream(dev)
    flush = L2Flush(dev)

    stages = ["metadata", "indexer", "topk", "sparse_mla"]
    calls = [step.metadata, step.indexer, step.topk_transform, step.attention]

    def one_step():
        for fn in calls:
            fn(stream)

    for _ in range(args.warmup):
        flush.zero_()
        one_step()
    torch.cuda.synchronize(dev)
    if step.status_code() != 0:
        raise RuntimeError(f"device status {step.status_code()} after warm-up")

    # The step as one CUDA graph (how a serving loop replays a decode step).  A
    # second graph of the same step carries timestamp nodes between the stages
    # for the per-stage split; the step time comes from the graph without them.
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(len(calls) + 1)]
    for e in ev:
        e.record(stream)  # creates the events before capture
    torch.cuda.synchronize(dev)

    def capture(staged):
        g = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(dev)
        cap.wait_stream(stream)
        with torch.cuda.graph(g, stream=cap):
            for i, fn in enumerate(calls):
                if staged:
                    record_external(ev[i], cap)
                fn(cap)
            if staged:
                record_external(ev[len(calls)], cap)
        stream.wait_stream(cap)
        return g

    graph, graph_staged = capture(False), capture(True)
    for _ in range(args.warmup):
        flush.zero_()
        graph.replay()
        flush.zero_()
        graph_staged.replay()
    torch.cuda.synchronize(dev)
    step_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]

    sampler = ClockSampler(local_rank)
    sampler.start()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    per_stage = {s: [] for s in stages}
    for k in range(args.steps):
        flush.zero_()  # L2 flush between steps, outside the timed events
        step_ev[k][0].record(stream)
        graph.replay()
        step_ev[k][1].record(stream)
    torch.cuda.synchronize(dev)
    totals = [a.elapsed_time(b) for a, b in step_ev]
    for k in range(args.steps):
        flush.zero_()
        graph_staged.replay()
        torch.cuda.synchronize(dev)
        for i, s in enumerate(stages):
            per_stage[s].append(ev[i].elapsed_time(ev[i + 1]))
    if world > 1:
        dist.barrier()
    clocks = sampler.stop()
    ms_step = float(np.mean(totals))
    if step.status_code() != 0:
        raise RuntimeError(f"device status {step.status_code()} after the timed steps")

    # end to end through the public API with host buffers: per step the
    # per-request inputs go host->device from pinned memory, the outputs come back.
    def pinned(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.uint8).reshape(-1)).pin_memory()

    h_md = {k: torch.from_numpy(np.ascontiguousarray(getattr(wl, k))).pin_memory()
            for k in ["seq_lens", "req_pool_indices"]}
    if wl.extend_lens is not None:
        h_md["extend_lens"] = torch.from_numpy(np.ascontiguousarray(wl.extend_lens)).pin_memory()
    h_idx = {k: pinned(getattr(wl, k)) for k in ["q_idx", "weights"]}
    h_q = {k: pinned(getattr(wl, k)) for k in ["q_nope", "q_rope"]}
    h_out = torch.empty(step.out.shape, dtype=step.out.dtype).pin_memory()
    h_lse = torch.empty(step.lse.shape, dtype=torch.float32).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in list(h_md.values()) + list(h_idx.values()) + list(h_q.values()))
    d2h = h_out.numel() * h_out.element_size() + h_lse.numel() * 4

    def dev_bytes(t):
        return t.view(torch.uint8).reshape(-1)

    # the queries go in by the copy engines; the rest of the traffic is done by the
    # kernels themselves reading and writing the pinned host buffers
    ins_idx = [(dev_bytes(step.q_idx), h_idx["q_idx"]), (dev_bytes(step.weights), h_idx["weights"])]
    ins_q = [(dev_bytes(step.q_nope), h_q["q_nope"]), (dev_bytes(step.q_rope), h_q["q_rope"])]
    side = torch.cuda.Stream(dev)
    idx_ready, q_ready = torch.cuda.Event(), torch.cuda.Event()

    def e2e_step(st):
        # the indexer's and the attention's queries travel by the copy engines on a side
        # stream (no SMs taken) while the metadata runs; the metadata kernel reads the
        # per-request lengths and pool rows straight from pinned host memory; each
        # consumer waits only for its own inputs; the attention writes out and lse straight
        # into the pinned host buffers (the device-to-host transfer happens in its epilogue)
        side.wait_stream(st)
        with torch.cuda.stream(side):
            for d, h in ins_idx:
                d.copy_(h, non_blocking=True)
            idx_ready.record(side)
            for d, h in ins_q:
                d.copy_(h, non_blocking=True)
            q_ready.record(side)
        step.metadata(st, **h_md)
        st.wait_event(idx_ready)
        step.indexer(st)
        step.topk_transform(st)
        st.wait_event(q_ready)
        step.attention(st, out=h_out, lse=h_lse)

    # the whole host-to-host step (inputs in, the four calls, results out) replayed as
    # one CUDA graph, as a serving loop runs it
    for _ in range(args.warmup):
        e2e_step(stream)
    torch.cuda.synchronize(dev)
    e2e_graph = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream(dev)
    cap.wait_stream(stream)
    with torch.cuda.graph(e2e_graph, stream=cap):
        e2e_step(cap)
    stream.wait_stream(cap)
    for _ in range(args.warmup):
        e2e_graph.replay()
    torch.cuda.synchronize(dev)
    e2e_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for k in range(args.steps):
        flush.zero_()
        e2e_ev[k][0].record(stream)
        e2e_graph.replay()
        e2e_ev[k][1].record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = float(np.mean([a.elapsed_time(b) for a, b in e2e_ev]))
    if step.status_code() != 0:
        raise RuntimeError(f"device status {step.status_code()} after the timed steps")
    # the end-to-end step computes what the device-resident step computes, bit for bit
    graph.replay()
    torch.cuda.synchronize(dev)
    if not (torch.equal(dev_bytes(h_out), dev_bytes(step.out.cpu())) and torch.equal(h_lse, step.lse.cpu())):
        raise RuntimeError("the end-to-end step's result differs from the device-resident step's")

    ms_step, e2e_ms = max_over_ranks([ms_step, e2e_ms], world)

    _, mla_launches = nsa.nsa_sparse_mla_plan(wl.q_dtype, wl.kv_dtype, wl.R, wl.H, wl.d_latent, wl.d_rope,
                                              wl.topk)
    topk_launches = nsa.nsa_topk_launches(wl.R, step.W, step.score_hist is not None)
    launches_per_step = len(calls) - 2 + topk_launches + mla_launches  # metadata and indexer: one each
    md_len = step.md["seqlens_expanded"].cpu().numpy()
    work = algorithmic_work(wl, md_len, step.md["row_to_req"].cpu().numpy(), step.indices.cpu().numpy())
    peaks = load_peaks()
    stage_ms = {s: float(np.mean(v)) for s, v in per_stage.items()}
    stage_info = {s: stage_roofline(wl, s, work[s], stage_ms[s] * 1e-3, peaks) for s in stages}
    for s in stages:
        stage_info[s]["traffic"] = ncu_traffic(name, s)
    dom = max(stages, key=lambda s: stage_ms[s])
    di = stage_info[dom]
    if di["bound"] == "tensor":
        roof = dict(kernel=dom, bound="tensor", achieved=di["tflops"], peak=di["tc_peak_tflops"], unit="TFLOP/s",
                    frac=di["frac"], traffic=di["traffic"], algorithmic_flops=di["flops"],
                    algorithmic_bytes=di["bytes"], peak_source=peaks["source"] + " (" + (
                        "fp8 = 2x bf16" if dom == "indexer" else "bf16") + ")")
    else:
        roof = dict(kernel=dom, bound="hbm", achieved=di["gbs"], peak=peaks["hbm_gbs"], unit="GB/s",
                    frac=di["frac"], traffic=di["traffic"], algorithmic_bytes=di["bytes"],
                    peak_source=peaks["source"])

    rows_total = wl.R * world
    line = dict(metric=METRIC, value=round(replica_throughput(wl.R, world, ms_step), 1), unit="tokens/s", n_gpus=world,
                steps=args.steps, warmup=args.warmup, ms_per_step=round(ms_step, 5), higher_is_better=True,
                scaling="weak", vs_baseline=None,
                dtype="f32" if wl.kv_dtype == W.DT_F32 else
                ("bf16+e4m3 (f32 accumulate)" if wl.kv_dtype == W.DT_BF16 else "e4m3 KV + bf16 (f32 accumulate)"),
                data="synthetic (seeded; random pages; see workloads/)",
                config=dict(workload=name, description=WORKLOADS[name], global_batch=rows_total,
                            seq_len=int(np.mean(wl.seq_lens)), parallelism=f"replicas x{world}",
                            l2="flushed between steps (512 MB write, then a 256 MB read that retires its dirty lines, outside the timed events)",
                            timing="step replayed as one CUDA graph timed by events around the replay; stage "
                                   "split from a second graph with timestamp nodes between the stages"),
                stages=stage_info, roofline=roof,
                e2e=dict(value=round(rows_total / (e2e_ms * 1e-3), 1), unit="tokens/s",
                         h2d_bytes_per_step=int(h2d), d2h_bytes_per_step=int(d2h),
                         note="per-request inputs host->device from pinned memory and out+lse device->host "
                              "each step (the indexer's and the attention's queries by the copy engines on a side "
                              "stream, overlapping the earlier stages; lengths and pool rows read by the metadata "
                              "kernel from pinned host memory; out and lse written by the attention kernel into "
                              "pinned host memory), the step replayed as one CUDA graph; "
                              "KV / indexer-K caches and the req_to_token pool stay resident"),
                gpu_launches=launches_per_step * args.steps,
                clocks=dict(sm_mhz=clocks["sm_mhz"], sm_max_mhz=clocks["sm_max_mhz"], reasons=clocks["reasons"]))
    if cpu is not None:
        line["cpu_baseline"] = cpu
    return line


# ---------------------------------------------------------------- CPU baseline (the oracle)

def host_cpu() -> dict:
    """Core count and CPU model of this host (lscpu, else /proc/cpuinfo)."""
    n = os.cpu_count() or 1
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.strip().lower().startswith("model name"):
                model = ln.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    if model is None:
        try:
            with open("/proc/cpuinfo") as f:
                for ln in f:
                    if ln.lower().startswith(("model name", "cpu part")):
                        model = ln.split(":", 1)[1].strip()
                        break
        except OSError:
            pass
    return dict(cores=n, model=model or "unknown")


def cpu_sample_rows(wl, full: bool) -> list:
    """Rows of the oracle's CPU sample.  Full: every row, except the chunked extend,
    whose fp64 work (~6 TFLOP) is sampled at every 32nd row of each sequence plus its
    first and last rows.  Bounded: all rows in a seeded random order (the caller stops
    at its time budget)."""
    if full and wl.mode == W.MODE_EXTEND:
        rows, start = set(), 0
        for n in wl.extend_lens:
            n = int(n)
            rows.update(range(start, start + n, 32))
            rows.update([start, start + n - 1])
            start += n
        return sorted(rows)
    if full:
        return list(range(wl.R))
    return [int(r) for r in np.random.default_rng(12345).permutation(wl.R)]


def oracle_metadata_time(wl):
    import oracle
    oracle.num_rows(wl.mode, wl.B, wl.extend_lens, wl.n_draft)  # the library is built and loaded outside the timing
    t0 = time.perf_counter()
    md = oracle.metadata(wl.mode, wl.seq_lens, wl.req_to_token, wl.req_pool_indices, W=wl.W, topk=wl.topk,
                         page_size=wl.page_size, extend_lens=wl.extend_lens, n_draft=wl.n_draft)
    return md, time.perf_counter() - t0


def oracle_row_time(wl, md, r: int) -> float:
    """Seconds for the oracle's indexer, top-k and sparse MLA of one query row."""
    import oracle
    t0 = time.perf_counter()
    lg = oracle.indexer_logits(wl.idx_dtype, wl.q_idx, wl.weights, wl.k_cache, wl.k_scale, md["real_page_table"],
                               md["row_to_req"], md["seqlens_expanded"], rows=[r], width=wl.W)
    idx = oracle.topk_transform(lg, md["seqlens_expanded"], md["row_to_req"], md["page_table_1"], wl.topk,
                                rows=[r], logits_rows_are_subset=True)
    oracle.sparse_mla(wl.q_dtype, wl.kv_dtype, wl.q_nope, wl.q_rope, wl.kv, idx, wl.sm_scale, rows=[r],
                      indices_rows_are_subset=True)
    return time.perf_counter() - t0


def cpu_baseline(wl, full: bool = False, budget_s: float = 12.0) -> dict:
    """The oracle as it stands (single-threaded C, fp64): metadata for the whole
    batch, then indexer + top-k + sparse MLA row by row.  Bounded (default): rows in a
    seeded random order until `budget_s` of row work, the mean row time scaled to all
    rows.  Full: the whole CPU sample of the workload, its rows spread over one worker
    thread per host core (each row runs single-threaded on one core; the oracle's C
    code releases the interpreter lock), the per-row times summed as one core's time."""
    from concurrent.futures import ThreadPoolExecutor
    host = host_cpu()
    md, t_md = oracle_metadata_time(wl)
    rows = cpu_sample_rows(wl, full)
    wall0 = time.perf_counter()
    if full:
        threads = max(1, host["cores"])
        with ThreadPoolExecutor(threads) as ex:
            times = list(ex.map(lambda r: oracle_row_time(wl, md, r), rows))
    else:
        threads = 1
        times = []
        for r in rows:
            times.append(oracle_row_time(wl, md, r))
            if sum(times) >= budget_s:
                break
        rows = rows[: len(times)]
    wall = time.perf_counter() - wall0
    per_row = float(np.sum(times)) / len(times)
    step_s = t_md + per_row * wl.R
    scaled = len(times) < wl.R
    what = ("the workload's full CPU sample" if full else f"a bounded sample (~{budget_s:.0f} s of row work)")
    return dict(value=round(wl.R / step_s, 4), unit="tokens/s", cores=1, kind="oracle",
                host=f"1 of {host['cores']} cores, {host['model']}",
                sample=f"{what}: metadata for all {wl.B} requests ({t_md:.3f} s) + indexer/top-k/sparse MLA for "
                       f"{len(times)} of {wl.R} rows, {per_row:.3f} s per row on one core"
                       + (f" (rows run concurrently on {threads} threads, one core each; {wall:.1f} s wall)"
                          if threads > 1 else "")
                       + ("; per-row time scaled to the full step (extrapolated)" if scaled else "; every row")
                       + "; single-threaded C, fp64",
                step_seconds_one_core=round(step_s, 3), extrapolated=scaled)


def run_reference(args, rank, world):
    """The oracle as the reference implementation: each step its metadata for the
    whole batch plus indexer/top-k/sparse MLA for one query row (cycling through
    the rows), single-threaded on one host core."""
    if rank != 0:
        return None
    name = args.config
    wl = W.config(name, seed=DEFAULT_SEED[name])
    rows = cpu_sample_rows(wl, full=False)
    for k in range(args.warmup):
        md, _ = oracle_metadata_time(wl)
        oracle_row_time(wl, md, rows[k % len(rows)])
    t = []
    for k in range(args.steps):
        md, t_md = oracle_metadata_time(wl)
        t.append(t_md + oracle_row_time(wl, md, rows[(args.warmup + k) % len(rows)]))
    s = float(np.mean(t))
    v = round(1 / s, 4)
    host = host_cpu()
    sample = (f"each step: oracle metadata for the whole batch + indexer/top-k/sparse MLA for 1 of {wl.R} rows "
              "(single-threaded C, fp64)")
    return dict(impl="reference", metric=METRIC, value=v, unit="tokens/s", n_gpus=world, steps=args.steps,
                warmup=args.warmup, ms_per_step=round(s * 1e3, 3), higher_is_better=True, scaling="weak",
                vs_baseline=None, dtype="f64", data="synthetic (seeded; random pages; see workloads/)",
                config=dict(workload=name, description=WORKLOADS[name], global_batch=wl.R,
                            seq_len=int(np.mean(wl.seq_lens)), parallelism="oracle on rank 0"),
                cpu_baseline=dict(value=v, unit="tokens/s", cores=1, kind="oracle",
                                  host=f"1 of {host['cores']} cores, {host['model']}", sample=sample),
                e2e=dict(value=v, unit="tokens/s", h2d_bytes_per_step=0, d2h_bytes_per_step=0))


# ---------------------------------------------------------------- KV-cache write side

def run_kv_write(args):
    """The write-side kernels on this workload's shapes: the step's new tokens
    into the fp8 KV cache and the indexer key cache, the whole bf16 cache to fp8
    (the pages' quantize_k_cache), and the gather of the step's selected rows back
    to bf16 (dequantize_k_cache_paged).  One JSON line, HBM roofline per kernel."""
    import torch
    import deepseek_sparse_mla_indexer_gb300 as nsa
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    nsa.load()
    wl = W.config(WORKLOAD, seed=DEFAULT_SEED[WORKLOAD])
    rng = np.random.default_rng(7)
    n_slots = wl.kv.shape[0]
    kv_bf16 = torch.from_numpy(wl.kv.view(np.int16)).to(dev)
    kv_fp8 = torch.empty((n_slots, 656), dtype=torch.uint8, device=dev)
    k_cache = torch.empty((n_slots, 128), dtype=torch.uint8, device=dev)
    k_scale = torch.empty((n_slots,), dtype=torch.float32, device=dev)
    new = wl.B  # one new token per request in a decode step
    loc = torch.from_numpy(rng.choice(n_slots, size=new, replace=False).astype(np.int32)).to(dev)
    k_nope = torch.randn((new, 512), device=dev).to(torch.bfloat16).view(torch.int16)
    k_rope = torch.randn((new, 64), device=dev).to(torch.bfloat16).view(torch.int16)
    k_idx = torch.randn((new, 128), device=dev).to(torch.bfloat16).view(torch.int16)
    sel = torch.from_numpy(rng.integers(0, n_slots, size=wl.R * wl.topk).astype(np.int32)).to(dev)
    gathered = torch.empty((sel.numel(), 576), dtype=torch.int16, device=dev)
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream(dev)
    kernels = {
        "quantize_kv_cache": (lambda: nsa.nsa_quantize_kv_cache(kv_bf16, kv_fp8), n_slots * (1152 + 656)),
        "dequantize_kv_paged": (lambda: nsa.nsa_dequantize_kv_paged(kv_fp8, sel, gathered),
                                sel.numel() * (656 + 1152 + 4)),
        "set_mla_kv_fp8": (lambda: nsa.nsa_set_mla_kv(nsa.DT_E4M3, k_nope, k_rope, loc, kv_fp8), new * (1152 + 656 + 4)),
        "set_index_k": (lambda: nsa.nsa_set_index_k(k_idx, loc, k_cache, k_scale), new * (256 + 128 + 4 + 4)),
    }
    peaks = load_peaks()
    res = {}
    for name, (fn, nbytes) in kernels.items():
        for _ in range(args.warmup):
            flush.zero_()
            fn()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
        for a, b in ev:
            flush.zero_()
            a.record(stream)
            fn()
            b.record(stream)
        torch.cuda.synchronize(dev)
        us = float(np.median([a.elapsed_time(b) for a, b in ev])) * 1e3
        gbs = nbytes / (us * 1e-6) / 1e9
        res[name] = dict(us=round(us, 2), algorithmic_bytes=int(nbytes), gbs=round(gbs, 1),
                         hbm_frac=round(gbs / peaks["hbm_gbs"], 4))
    q = res["quantize_kv_cache"]
    return dict(metric="KV-cache write side: GB/s of the whole-cache fp8 quantisation (HBM roofline)",
                value=q["gbs"], unit="GB/s", n_gpus=1, steps=args.steps, warmup=args.warmup,
                higher_is_better=True, dtype="bf16 -> e4m3 + f32 scales", data="synthetic (seeded)",
                config=dict(workload=WORKLOAD_DESC, kv_slots=int(n_slots), new_tokens=int(new),
                            gathered_rows=int(sel.numel()), l2="flushed before each launch (512 MB write, then a 256 MB read)"),
                kernels=res, peak_gbs=peaks["hbm_gbs"], peak_source=peaks["source"])


# ---------------------------------------------------------------- chunk-local dense attention

LOCAL_WORKLOAD = "local_decode_c8192"
LOCAL_DESC = ("chunk-local dense attention, decode: 32 requests of lengths U{1..16384}, attention chunk 8192, "
              "40 query heads over 8 key/value heads of 128 dims, bf16 paged K/V (page 64, random page order)")


def local_visible_keys(cu: np.ndarray, sk: np.ndarray) -> int:
    """Keys all query rows see: query i of n_q in a virtual batch with k keys sees k - n_q + i + 1."""
    tot = 0
    for v in range(len(sk)):
        n, k = int(cu[v + 1] - cu[v]), int(sk[v])
        i = np.arange(n)
        tot += int(np.clip(k - n + i + 1, 0, k).sum())
    return tot


def local_algorithmic_bytes(wl, cu, sk) -> int:
    """K and V rows of every visible key (per key/value head), q in, out and lse out,
    plus the virtual batches' tables and lengths."""
    rows = local_visible_keys(cu, sk)
    pages = int(((sk.astype(np.int64) + wl.page_size - 1) // wl.page_size).sum())
    return (rows * wl.Hkv * wl.D * 2 * 2 + wl.total_q * wl.Hq * wl.D * 2 * 2 + wl.total_q * wl.Hq * 4
            + pages * 4 + len(sk) * 8 + 4)


def local_cpu_baseline(wl, max_keys: int = 300000):
    """The oracle as it stands: its virtual batches for the whole batch, then its
    attention on a bounded sample of them, scaled to the whole step by the visible
    keys (its attention time is proportional to them)."""
    import oracle
    t0 = time.perf_counter()
    _, cu, sk, _, bt = oracle.local_virtual_batches(wl.chunk, wl.page_size, wl.cu_seqlens_q, wl.seq_lens,
                                                    wl.block_table)
    t_vb = time.perf_counter() - t0
    order = np.argsort(sk)
    rows, keys = [], 0
    for v in np.concatenate([order[len(order) // 2:], order[: len(order) // 2]]):  # from the median length up
        rows.append(int(v))
        keys += local_visible_keys(cu[[v, v + 1]] - cu[v], sk[[v]])
        if keys >= max_keys:
            break
    sel_q = np.concatenate([np.arange(cu[v], cu[v + 1]) for v in rows])
    cu_s = np.zeros(len(rows) + 1, np.int32)
    cu_s[1:] = np.cumsum([cu[v + 1] - cu[v] for v in rows])
    t0 = time.perf_counter()
    oracle.local_attention(wl.q[sel_q], wl.k_cache, wl.v_cache, bt[rows], cu_s, sk[rows], wl.sm_scale)
    dt = time.perf_counter() - t0
    total = local_visible_keys(cu, sk)
    full_s = t_vb + dt * total / max(1, keys)
    return dict(value=round(wl.total_q / full_s, 3), unit="query tokens/s", cores=1, kind="oracle",
                sample=f"virtual batches for the whole batch, attention for {len(rows)} of {len(sk)} of them "
                       f"({keys} of {total} visible keys) scaled by visible keys; single-threaded C, fp64")


def run_local_attention(args):
    """nsa_local_attention on the chunk-local decode workload: query tokens/s of the
    kernel with inputs resident (L2 flushed between launches), end to end from host
    buffers (the host builds the virtual batches each step, as the pages do), the
    HBM roofline and the oracle's CPU time."""
    import torch
    import deepseek_sparse_mla_indexer_gb300 as nsa
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    nsa.load()
    wl = W.local_config(LOCAL_WORKLOAD)
    _, cu, sk, _, bt = nsa.nsa_local_virtual_batches(wl.chunk, wl.page_size, wl.cu_seqlens_q, wl.seq_lens,
                                                     wl.block_table)
    q = torch.from_numpy(wl.q.view(np.int16)).to(dev).view(torch.bfloat16)
    kc = torch.from_numpy(wl.k_cache.view(np.int16)).to(dev).view(torch.bfloat16)
    vc = torch.from_numpy(wl.v_cache.view(np.int16)).to(dev).view(torch.bfloat16)
    d_cu, d_sk, d_bt = [torch.from_numpy(np.ascontiguousarray(x)).to(dev) for x in (cu, sk, bt)]
    out = torch.empty((wl.total_q, wl.Hq, wl.D), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((wl.total_q, wl.Hq), dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream(dev)

    def call():
        nsa.nsa_local_attention(q, kc, vc, d_bt, d_cu, d_sk, wl.sm_scale, out, lse, status=status, stream=stream)

    for _ in range(args.warmup):
        flush.zero_()
        call()
    torch.cuda.synchronize(dev)
    sampler = ClockSampler(0)
    sampler.start()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for a, b in ev:
        flush.zero_()
        a.record(stream)
        call()
        b.record(stream)
    torch.cuda.synchronize(dev)
    clocks = sampler.stop()
    ms = float(np.mean([a.elapsed_time(b) for a, b in ev]))
    if status.item() != 0:
        raise RuntimeError(f"device status {status.item()} after the timed launches")

    # end to end from host buffers: per step the host builds the virtual batches
    # (library C++), q and the local tables go in, out and lse come back
    h_q = torch.from_numpy(wl.q.view(np.int16)).pin_memory()
    h_cu = torch.empty(len(cu), dtype=torch.int32).pin_memory()
    h_sk = torch.empty(len(sk), dtype=torch.int32).pin_memory()
    h_bt = torch.empty(bt.shape, dtype=torch.int32).pin_memory()
    h_out = torch.empty(out.shape, dtype=torch.int16).pin_memory()
    h_lse = torch.empty(lse.shape, dtype=torch.float32).pin_memory()

    h_cu.numpy()[:] = cu
    h_sk.numpy()[:] = sk
    h_bt.numpy()[:] = bt

    # the device part of a step (inputs in by one copy kernel, the attention writing
    # out and lse straight into the pinned host buffers) replayed as one CUDA graph
    def device_part(st):
        nsa.nsa_copy_buffers([(q.view(torch.int16), h_q), (d_cu, h_cu), (d_sk, h_sk), (d_bt, h_bt)], st)
        nsa.nsa_local_attention(q, kc, vc, d_bt, d_cu, d_sk, wl.sm_scale, h_out.view(torch.bfloat16), h_lse,
                                status=status, stream=st)

    device_part(stream)
    torch.cuda.synchronize(dev)
    graph = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream(dev)
    cap.wait_stream(stream)
    with torch.cuda.graph(graph, stream=cap):
        device_part(cap)
    stream.wait_stream(cap)

    def e2e_step():
        _, c2, s2, _, b2 = nsa.nsa_local_virtual_batches(wl.chunk, wl.page_size, wl.cu_seqlens_q, wl.seq_lens,
                                                         wl.block_table)
        h_cu.numpy()[:] = c2
        h_sk.numpy()[:] = s2
        h_bt.numpy()[:] = b2
        graph.replay()
        torch.cuda.current_stream(dev).synchronize()

    for _ in range(args.warmup):
        e2e_step()
    e2e_t = []
    for _ in range(args.steps):
        flush.zero_()
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        e2e_step()
        e2e_t.append(time.perf_counter() - t0)
    e2e_s = float(np.mean(e2e_t))
    if status.item() != 0:
        raise RuntimeError(f"device status {status.item()} after the end-to-end steps")
    h2d = sum(t.numel() * t.element_size() for t in (h_q, h_cu, h_sk, h_bt))
    d2h = h_out.numel() * 2 + h_lse.numel() * 4

    peaks = load_peaks()
    nbytes = local_algorithmic_bytes(wl, cu, sk)
    achieved = nbytes / (ms * 1e-3) / 1e9
    line = dict(metric="chunk-local attention decode query tokens/s (% of HBM roofline)",
                value=round(wl.total_q / (ms * 1e-3), 1), unit="query tokens/s", n_gpus=1, steps=args.steps,
                warmup=args.warmup, ms_per_step=round(ms, 5), higher_is_better=True, scaling="weak",
                vs_baseline=None, dtype="bf16 (f32 accumulate)", data="synthetic (seeded; random pages; see workloads/)",
                config=dict(workload=LOCAL_DESC, global_batch=int(wl.total_q), virtual_batches=int(len(sk)),
                            seq_len=int(np.mean(wl.seq_lens)), visible_keys=local_visible_keys(cu, sk),
                            parallelism="replicas x1", l2="flushed before each launch (512 MB write, then a 256 MB read that retires its dirty lines, outside the events)"),
                roofline=dict(kernel="local_attention", bound="hbm", achieved=round(achieved, 1), peak=peaks["hbm_gbs"],
                              unit="GB/s", frac=round(achieved / peaks["hbm_gbs"], 4), traffic=ncu_traffic(LOCAL_WORKLOAD, "local_attention"),
                              algorithmic_bytes=int(nbytes), peak_source=peaks["source"]),
                e2e=dict(value=round(wl.total_q / e2e_s, 1), unit="query tokens/s", h2d_bytes_per_step=int(h2d),
                         d2h_bytes_per_step=int(d2h),
                         note="per step: the host builds the virtual batches (library C++), then one CUDA graph: "
                              "q and the local tables host->device by a copy kernel, the attention writing out and "
                              "lse straight into pinned host memory; wall clock to the stream's end"),
                gpu_launches=args.steps,
                clocks=dict(sm_mhz=clocks["sm_mhz"], sm_max_mhz=clocks["sm_max_mhz"], reasons=clocks["reasons"]))
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = local_cpu_baseline(wl)
    return line


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default=WORKLOAD, choices=list(WORKLOADS),
                    help="which of the five workloads to run (default: the one the metric is quoted on)")
    ap.add_argument("--cpu-full", action="store_true",
                    help="time the oracle on the workload's full CPU sample instead of a bounded one")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--kv-write", action="store_true",
                    help="measure the KV-cache write-side kernels instead of the attention step")
    ap.add_argument("--local-attn", action="store_true",
                    help="measure chunk-local dense attention (the second workload) instead of the step")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.kv_write:
        if rank == 0:
            print(json.dumps(run_kv_write(args)), flush=True)
        return
    if args.local_attn:
        if rank == 0:
            print(json.dumps(run_local_attention(args)), flush=True)
        return
    if args.impl == "reference":
        line = run_reference(args, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
    line = run_ours(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
