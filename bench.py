"""Benchmark of the indexer hot path on GB300: one step = K store of the step's new keys,
Q quant, paged MQA-logits scorer and per-query top-k, through the C ABI.

Default workload: MXFP4 decode, B=64 sequences x 1 query, H=32, D=128, 8192 keys each,
page size 128 from a permuted pool of 4608 pages, 1% outlier K rows, top-k 1024. Metric:
K-tokens/s = (query, key) pairs scored per second / 1000 (higher is better).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl reference]

Prints one JSON line (rank 0). Timing: W untimed steps, then exactly K steps between a
barrier + synchronize on both sides, CUDA events on the launching stream, max over ranks.
The L2 (129 MB) is defeated by rotating over enough independent copies of the K cache and
Q inputs that consecutive reuses are more than 4x the L2 size apart. Multi-GPU: one
independent replica per rank (the path needs no exchange), weak scaling.
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

from sparse_attention_indexer_mqa_gb300 import workloads as W  # noqa: E402

L2_BYTES = 129 * 1024 * 1024

# per-config algorithmic bytes of one scorer launch (what the scorer must read + write)
# and of the other kernels, computed from the workload below


def algorithmic_bytes(wl):
    """Bytes the scorer must move in one launch: every visible key once (68 or 132 B), the
    quantised Q (64+4 or 128 B per (t,h)), the weights, page table, lengths and the fp32
    logits it writes."""
    per_tok = 68 if wl.dtype == W.MXFP4 else 132
    per_q = 68 if wl.dtype == W.MXFP4 else 128
    keys = int(wl.seq_lens_k.sum())
    pt = int(sum((int(L) + wl.page_size - 1) // wl.page_size for L in wl.seq_lens_k)) * 4
    return {
        "scorer": keys * per_tok + wl.T * wl.H * (per_q + 4) + pt + 4 * wl.B + 4 * (wl.B + 1)
        + 4 * wl.pairs(),
        "qk_prep": len(wl.step_rows) * (256 + per_tok + 8 + 4) + wl.T * wl.H * (256 + per_q + 4 + 4),
        "topk": 4 * wl.pairs() + 4 * wl.T * wl.topk,
    }


def scorer_flops(wl):
    """Tensor-core work of one scorer launch: 2 * H * D flops per (query, key) pair."""
    return 2.0 * wl.H * 128 * wl.pairs()


def scorer_alu_ops(wl):
    """Epilogue issue work of one scorer launch: per (query, key) pair and head one ReLU
    (max) and one fused multiply-add of the head-weighted sum (thread instructions)."""
    return 2.0 * wl.H * wl.pairs()


# issue rate of the GPU in thread instructions per second: 4 schedulers x 32 lanes per SM per
# clock, 152 SMs, at the measured maximum SM clock (one warp instruction per scheduler per clock)
def alu_peak_ops(peaks):
    return 4 * 32 * 152 * peaks.get("sm_max_mhz", 2070.0) * 1e6


# nominal HBM3e bandwidth of the part (the roofline's peak is the measured copy rate)
HBM_SPEC_GBS = 7900.0

# nominal dense tensor rates relative to bf16 (2.25 PF bf16, 4.5 PF fp8, 13.5 PF fp4)
TENSOR_RATIO = {W.MXFP4: 6.0, W.FP8: 2.0}


def is_decode(wl):
    return int(np.diff(wl.cu_seqlens_q).max()) <= 1


def metric_name(wl):
    kind = "decode" if is_decode(wl) else "prefill"
    dt = "MXFP4" if wl.dtype == W.MXFP4 else "FP8"
    return (f"indexer {kind} K-tokens/s (query-key pairs scored per second / 1e3), {wl.name} "
            f"({dt}, H{wl.H}, page {wl.page_size})")


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def source_sha(paths):
    h = hashlib.sha256()
    for p in paths:
        h.update(open(os.path.join(ROOT, p), "rb").read())
    return h.hexdigest()[:16]


def profile_traffic(kernel_key, sources):
    """dram bytes per launch from the committed ncu summary, if it was taken on the
    current kernel source; else None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p)).get(kernel_key)
    if not d or d.get("source_sha") != source_sha(sources):
        return None
    return d.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except FileNotFoundError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1])); mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------------------

# one library call (one kernel launch) each: the separate calls, and the fused scorer -> top-k
STEP_CALLS = ("qk_prep", "scorer", "topk")
FUSED_STEP_CALLS = ("qk_prep", "scorer_topk")


class Replica:
    """Device state of one workload: R rotating copies of the K cache and Q inputs."""

    def __init__(self, wl, copies, device):
        import torch
        from sparse_attention_indexer_mqa_gb300 import binding as Bn
        self.Bn, self.torch, self.wl = Bn, torch, wl
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(device)
        self.cos_sin = t(wl.cos_sin)
        self.page_table = t(wl.page_table)
        self.seq_lens_k = t(wl.seq_lens_k)
        self.cu = t(wl.cu_seqlens_q)
        self.max_q = int(np.diff(wl.cu_seqlens_q).max())
        self.max_k = int(wl.seq_lens_k.max())
        # the step's new keys (their rows of k / slots / positions)
        sr = wl.step_rows
        self.k_new = t(wl.k[sr].view(np.int16))
        self.slot_new = t(wl.slot_mapping[sr])
        self.pos_new = t(wl.k_positions[sr])
        self.q = [t(wl.q.view(np.int16)) for _ in range(copies)]
        self.qpos = t(wl.q_positions)
        self.w_in = t(wl.w_in)
        T, H = wl.T, wl.H
        Hq = (H + 7) // 8 * 8
        per_q = 64 if wl.dtype == W.MXFP4 else 128
        self.q_codes = torch.zeros((T, Hq, per_q), dtype=torch.uint8, device=device)
        self.q_scales = (torch.zeros((T, 512), dtype=torch.uint8, device=device)
                         if wl.dtype == W.MXFP4 else None)
        self.w = torch.zeros((T, H), dtype=torch.float32, device=device)
        self.logits = torch.empty((T, wl.ld_logits), dtype=torch.float32, device=device)
        self.topk = torch.empty((T, wl.topk), dtype=torch.int32, device=device)
        # the scorer's scheduling workspace (zeroed once; every call leaves it zero)
        self.sched_ws = torch.zeros(Bn.idx_mqa_logits_workspace_bytes(), dtype=torch.uint8, device=device)
        # workspace of the fused scorer -> top-k (zeroed once: its counters start at zero)
        n_ws = Bn.idx_mqa_topk_workspace_bytes(T, H, wl.B, self.max_q, self.max_k)
        self.workspace = torch.zeros(max(n_ws, 256), dtype=torch.uint8, device=device)
        # set-up (untimed): store every key once, then clone the pool R-1 times
        pool0 = torch.zeros(wl.pool_pages * wl.page_stride, dtype=torch.uint8, device=device)
        kall = t(wl.k.view(np.int16))
        Bn.idx_k_store(kall, t(wl.slot_mapping), t(wl.k_positions) if wl.k_rope else None,
                       self.cos_sin if wl.k_rope else None, wl.k_rope, wl.k_norm, wl.dtype, pool0,
                       wl.pool_pages, wl.page_size, wl.page_stride)
        del kall
        self.pools = [pool0] + [pool0.clone() for _ in range(copies - 1)]
        torch.cuda.synchronize()

    def call(self, name, i, inputs=None):
        """One library call of the step on rotation copy i % R."""
        wl, Bn = self.wl, self.Bn
        r = i % len(self.pools)
        pool = self.pools[r]
        inp = inputs or {}
        if name == "qk_prep":  # K store of the step's keys + Q quant, one launch
            Bn.idx_qk_prep(inp.get("k", self.k_new), inp.get("slot", self.slot_new),
                           inp.get("pos", self.pos_new) if wl.k_rope else None, wl.k_rope, wl.k_norm,
                           pool, wl.pool_pages, wl.page_size, wl.page_stride, inp.get("q", self.q[r]),
                           inp.get("qpos", self.qpos) if wl.q_rope else None, wl.q_rope,
                           inp.get("w", self.w_in), wl.softmax_scale, wl.head_scale, self.q_codes,
                           self.q_scales, self.w, self.cos_sin if (wl.k_rope or wl.q_rope) else None,
                           wl.dtype)
        elif name == "scorer":
            Bn.idx_mqa_logits_paged(self.q_codes, self.q_scales, self.w, wl.dtype, pool,
                                    wl.pool_pages, wl.page_size, wl.page_stride, self.page_table,
                                    self.seq_lens_k, self.cu, wl.causal, self.max_q, self.max_k,
                                    self.logits, workspace=self.sched_ws)
        elif name == "scorer_topk":
            Bn.idx_mqa_topk_paged(self.q_codes, self.q_scales, self.w, wl.dtype, pool, wl.pool_pages,
                                  wl.page_size, wl.page_stride, self.page_table, self.seq_lens_k,
                                  self.cu, wl.causal, self.max_q, self.max_k, wl.topk,
                                  inp.get("topk_out", self.topk), self.workspace)
        else:
            Bn.idx_topk(self.logits, self.seq_lens_k, self.cu, wl.causal, self.max_k, wl.topk,
                        inp.get("topk_out", self.topk))

    def step(self, i, inputs=None):
        for n in STEP_CALLS:
            self.call(n, i, inputs)


def working_set_bytes(wl):
    """Bytes a step reads that a rotation copy can hold: the K cache and the bf16 Q."""
    return wl.pool_pages * wl.page_stride + wl.q.nbytes


def capture(torch, fn, n):
    """One CUDA graph holding n calls fn(i) on the capture stream."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(n):
            fn(i)
    return g


def time_graph(torch, g, stream):
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record(stream)
    g.replay()
    e.record(stream)
    torch.cuda.synchronize()
    return s.elapsed_time(e)


def rank_max(x, world, device):
    """Maximum of a per-rank float over all ranks (the slowest rank sets the job's time);
    the value itself when there is one rank. `device` is where the collective's tensor
    lives: the rank's GPU under NCCL, the CPU under gloo."""
    if world <= 1:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_rate(pairs_per_rank, ms_per_step, world):
    """Whole-job throughput in K-tokens/s: every rank scores its own replica's pairs each
    step (weak scaling), in the slowest rank's time."""
    return world * pairs_per_rank / (ms_per_step / 1e3) / 1e3


def run_gpu(args, rank, world):
    import torch
    from sparse_attention_indexer_mqa_gb300 import binding as Bn
    Bn.load()
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    wl = W.make(args.config, seed=args.seed + rank)
    ws = working_set_bytes(wl)
    copies = 1 if ws > 16 * L2_BYTES else (2 if ws > 4 * L2_BYTES else max(2, -(-4 * L2_BYTES // ws)))
    rep = Replica(wl, copies, dev)
    stream = torch.cuda.current_stream()

    # W eager warm-up steps, then the K steps are captured once into a CUDA graph (the
    # library's calls are asynchronous and capturable) so that host launch overhead does
    # not gap the device timeline
    for i in range(args.warmup):
        rep.step(i)
    torch.cuda.synchronize()
    g_step = capture(torch, lambda i: rep.step(args.warmup + i), args.steps)
    g_step.replay()  # upload, untimed
    torch.cuda.synchronize()

    clocks = ClockSampler(dev.index)
    clocks.start()
    t_end = time.time() + 0.6
    while time.time() < t_end:  # keep the GPU loaded while the sampler starts
        g_step.replay()
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    ms = time_graph(torch, g_step, stream)  # the timed region: exactly K steps
    if world > 1:
        torch.distributed.barrier()
    t_end = time.time() + 0.3
    while time.time() < t_end:
        g_step.replay()
        torch.cuda.synchronize()
    clk = clocks.stop()
    ms = rank_max(ms, world, dev)

    # per-kernel device time: each kernel captured K times (same rotation) and timed alone;
    # also the fused scorer -> top-k and the step made with it
    per_kernel_ms = {name: time_calls(torch, rep, (name,), args.warmup, args.steps, stream)
                     for name in STEP_CALLS + ("scorer_topk",)}
    step_fused_ms = time_calls(torch, rep, FUSED_STEP_CALLS, args.warmup, args.steps, stream)

    # end to end through the C ABI with host buffers: H2D of the step's inputs (new K rows,
    # slots, positions, Q, weights) from pinned memory, the four calls, D2H of the top-k
    e2e = run_e2e(rep, args, torch, stream, world, dev)

    pairs = wl.pairs()
    value = job_rate(pairs, ms / args.steps, world)
    ab = algorithmic_bytes(wl)
    peaks, peak_kind = measured_peaks()
    sc_s = per_kernel_ms["scorer"] / 1e3
    if is_decode(wl):
        achieved = ab["scorer"] / sc_s / 1e9
        roof = {"kernel": "scorer", "bound": "hbm", "achieved": round(achieved, 1),
                "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
                "frac_of_spec": round(achieved / HBM_SPEC_GBS, 4),
                "cache_tokens_per_s": round(int(wl.seq_lens_k.sum()) / sc_s, 1),
                "traffic": profile_traffic(f"scorer:{args.config}", DECODE_SOURCES),
                "algorithmic_bytes": ab["scorer"], "peak_source": f"{peak_kind} (hbm_gbs)"}
    else:
        roof = prefill_roofline(wl, per_kernel_ms["scorer"], peaks, peak_kind)
    line = {
        "metric": metric_name(wl),
        "value": round(value, 1),
        "unit": "K-tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms / args.steps, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "mxfp4" if wl.dtype == W.MXFP4 else "fp8e4m3",
        "data": "synthetic (seeded numpy PCG64: bf16 N(0,1) q/k, N(0,1/H) head weights, "
                "permuted physical pages)",
        "config": {**config_of(wl),
                   "l2": f"inputs rotate over {copies} copies of cache+Q "
                         f"({copies * ws / 2**20:.0f} MiB)" if copies > 1 else
                         f"working set {ws / 2**20:.0f} MiB > 16x L2",
                   "step": "qk_prep (K store of the step's keys + Q quant, one launch) + mqa_logits_paged + topk",
                   "launch": "K steps captured in one CUDA graph, replayed once"},
        "kernel_us": {n: round(v * 1e3, 3) for n, v in per_kernel_ms.items()},
        "roofline": roof,
        "gpu_launches": len(STEP_CALLS) * args.steps,
        "clocks": clk,
        "e2e": e2e,
        "fused": {"step_us": round(step_fused_ms * 1e3, 3),
                  "value": round(job_rate(pairs, step_fused_ms, world), 1),
                  "step": "qk_prep + mqa_topk_paged (scorer and top-k in one launch)",
                  "note": "not the headline step: measured slower than the separate calls"},
    }
    if is_decode(wl) and args.config == "decode_b64" and not args.no_prefill:
        line["prefill"] = prefill_block(args, dev, peaks, peak_kind)
        line["qk_prep_sweep"] = qk_prep_sweep(args, dev, peaks)
    if args.config == "decode_b64" and not args.no_compress:
        line["compress"] = compress_block(args, dev, peaks)
    if args.config == "decode_b64" and not args.no_cand:
        line["cand"] = cand_block(args, dev, peaks)
    if not args.no_probe:
        line["tensor_probe"] = tensor_probe(torch, stream)
        if "prefill" in line:
            t = line["prefill"]["roofline"]["tensor"]
            p = line["tensor_probe"]["mxf4_tflops"]
            t["probe_tflops"] = p
            t["frac_of_probe"] = round(t["achieved_tflops"] / p, 4)
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, budget_s=args.cpu_budget,
                                            rows_per_step=None if is_decode(wl) else args.ref_rows)
    return line


def time_calls(torch, rep, calls, first, k, stream):
    """Device ms per step of `calls` (library calls of the replica), K steps in one graph."""
    g = capture(torch, lambda i: [rep.call(n, first + i) for n in calls], k)
    g.replay()
    torch.cuda.synchronize()
    return time_graph(torch, g, stream) / k


def prefill_roofline(wl, scorer_ms, peaks, peak_kind):
    """Prefill scorer against the dense tensor rate of its dtype (the measured bf16 rate times
    the nominal ratio) and against the issue rate of its epilogue."""
    sc_s = scorer_ms / 1e3
    alu = scorer_alu_ops(wl) / sc_s
    tpeak = peaks["bf16_tflops"] * TENSOR_RATIO[wl.dtype]
    return {"kernel": "scorer", "bound": "alu", "achieved": round(alu / 1e12, 2),
            "peak": round(alu_peak_ops(peaks) / 1e12, 2), "unit": "T instr/s",
            "frac": round(alu / alu_peak_ops(peaks), 4),
            "traffic": profile_traffic(f"scorer:{wl_key(wl)}", PREFILL_SOURCES),
            "algorithmic_ops": scorer_alu_ops(wl),
            "peak_source": "issue rate 4x32 lanes x 152 SMs x measured max SM clock",
            "tensor": {"achieved_tflops": round(scorer_flops(wl) / sc_s / 1e12, 1),
                       "peak_tflops": round(tpeak, 1),
                       "frac": round(scorer_flops(wl) / sc_s / 1e12 / tpeak, 4),
                       "peak_source": f"{peak_kind} bf16 x nominal ratio {TENSOR_RATIO[wl.dtype]:g}"},
            "hbm_gbs": round(algorithmic_bytes(wl)["scorer"] / sc_s / 1e9, 1)}


def wl_key(wl):
    return {"decode_mxfp4_b64_h32_8192": "decode_b64", "prefill_mxfp4_8192q_h32": "prefill_8k"}.get(wl.name, wl.name)


def prefill_block(args, dev, peaks, peak_kind):
    """The prefill half of the metric, measured in the default run: causal MXFP4 prefill, 8192
    queries x 8192 keys, H=32 (the pages' isolated prefill scorer shape)."""
    import torch
    wl = W.make("prefill_8k", seed=args.seed)
    ws = working_set_bytes(wl)
    copies = 1 if ws > 16 * L2_BYTES else (2 if ws > 4 * L2_BYTES else max(2, -(-4 * L2_BYTES // ws)))
    rep = Replica(wl, copies, dev)
    stream = torch.cuda.current_stream()
    k = max(3, min(args.steps, 10))
    for i in range(3):
        rep.step(i)
    torch.cuda.synchronize()
    kernel_ms = {n: time_calls(torch, rep, (n,), 3, k, stream) for n in STEP_CALLS + ("scorer_topk",)}
    step_ms = time_calls(torch, rep, STEP_CALLS, 3, k, stream)
    step_fused_ms = time_calls(torch, rep, FUSED_STEP_CALLS, 3, k, stream)
    pairs = wl.pairs()
    out = {"workload": wl.name, "queries": wl.T, "pairs": pairs, "steps": k,
           "step_us": round(step_ms * 1e3, 2), "step_fused_us": round(step_fused_ms * 1e3, 2),
           "value": round(pairs / (step_ms / 1e3) / 1e3, 1), "unit": "K-tokens/s",
           "scorer_k_tokens_per_s": round(pairs / (kernel_ms["scorer"] / 1e3) / 1e3, 1),
           "kernel_us": {n: round(v * 1e3, 2) for n, v in kernel_ms.items()},
           "roofline": prefill_roofline(wl, kernel_ms["scorer"], peaks, peak_kind),
           "l2": f"inputs rotate over {copies} copies of cache+Q"}
    del rep
    torch.cuda.empty_cache()
    return out


# thread instructions of the pooling per (window row, dimension): gate max 1, difference 1,
# exp 14 (product, rint, 2 reduction and 7 Horner fused multiply-adds, 2 to build 2^n, product),
# sum 1, fused multiply-add of the weighted row 1
COMPRESS_OPS_PER_ROW_DIM = 18


def compress_block(args, dev, peaks):
    """The compressed K store (idx_compress_k_store) over whole contexts: 256 sequences of raw
    length uniform in [1024, 9472], ratio 4, RMSNorm, NeoX RoPE, MXFP4 into 64-entry pages.
    Inputs (bf16 K and gate rows, 512 B per raw row) are larger than L2."""
    import torch
    from sparse_attention_indexer_mqa_gb300 import binding as Bn
    cw = W.compress_b256(seed=args.seed)

    def d(a):
        a = np.ascontiguousarray(a)
        return torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).to(dev)

    k_raw, gate = d(cw.k_raw), d(cw.gate)
    bnd, fst, slot, pos = d(cw.boundary), d(cw.first), d(cw.slot_mapping), d(cw.positions)
    cs, gam = d(cw.cos_sin), d(cw.gamma)
    pool = torch.zeros(cw.pool_pages * cw.page_stride, dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()

    def call(i=0):
        Bn.idx_compress_k_store(k_raw, gate, bnd, fst, cw.ratio, slot, pos, cs, cw.rope, cw.norm,
                                cw.dtype, pool, cw.pool_pages, cw.page_size, cw.page_stride,
                                gamma=gam, dev_status=status)

    for i in range(3):
        call()
    torch.cuda.synchronize()
    k = max(3, min(args.steps, 20))
    g = capture(torch, call, k)
    g.replay()
    torch.cuda.synchronize()
    ms = time_graph(torch, g, stream) / k
    n_raw, E = int(cw.k_raw.shape[0]), cw.n_entries
    win_rows = int(np.sum(cw.boundary - np.maximum(cw.first, cw.boundary - 2 * cw.ratio + 1) + 1))
    # every raw row once (K and gate), the entry's indices (slot, boundary, first, position) and
    # its 68 B store; the overlapping windows re-read rows from cache, not from HBM
    ab = n_raw * 512 + E * (8 + 8 + 8 + 4 + 68)
    ops = float(win_rows) * 128 * COMPRESS_OPS_PER_ROW_DIM
    t = ms / 1e3
    out = {"workload": cw.name, "raw_rows": n_raw, "entries": E, "window_rows": win_rows, "steps": k,
           "us": round(ms * 1e3, 2), "entries_per_s": round(E / t, 1),
           "raw_rows_per_s": round(n_raw / t, 1),
           "roofline": {"kernel": "compress", "bound": "alu",
                        "achieved": round(ops / t / 1e12, 2), "peak": round(alu_peak_ops(peaks) / 1e12, 2),
                        "unit": "T instr/s", "frac": round(ops / t / alu_peak_ops(peaks), 4),
                        "algorithmic_ops": ops, "ops_per_row_dim": COMPRESS_OPS_PER_ROW_DIM,
                        "peak_source": "issue rate 4x32 lanes x 152 SMs x measured max SM clock",
                        "hbm": {"achieved_gbs": round(ab / t / 1e9, 1), "peak_gbs": peaks["hbm_gbs"],
                                "frac": round(ab / t / 1e9 / peaks["hbm_gbs"], 4),
                                "algorithmic_bytes": ab},
                        "traffic": profile_traffic("compress:compress_b256", COMPRESS_SOURCES)},
           "status": int(status.item()),
           "l2": f"inputs {2 * n_raw * 256 / 2**20:.0f} MiB > L2"}
    del k_raw, gate, pool, g
    torch.cuda.empty_cache()
    return out


def cand_block(args, dev, peaks):
    """The candidate-pool path (idx_mqa_topk_cand_paged) on the decode shape (B=64, H=32, 8192
    keys, page 128): 16 candidate blocks per query (2048 of its 8192 keys, the last block
    always in), beside the dense scorer + top-k on the same data. Each timed call follows a
    256 MiB write that flushes L2; only the call lies between its events."""
    import torch
    from sparse_attention_indexer_mqa_gb300 import binding as Bn
    wl = W.make("decode_b64", seed=args.seed)
    rep = Replica(wl, 1, dev)
    rep.call("qk_prep", 0)
    torch.cuda.synchronize()
    cand, n_cand, max_cand = W.candidate_blocks(wl, seed=args.seed, n_blocks=16)
    c = torch.from_numpy(cand).to(dev)
    nc = torch.from_numpy(n_cand).to(dev)
    max_k = int(wl.seq_lens_k.max())
    ws = torch.zeros(Bn.idx_mqa_topk_cand_workspace_bytes(wl.T, max_cand, wl.page_size, max_k),
                     dtype=torch.uint8, device=dev)
    out = torch.empty((wl.T, wl.topk), dtype=torch.int32, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()

    def cand_call():
        Bn.idx_mqa_topk_cand_paged(rep.q_codes, rep.q_scales, rep.w, wl.dtype, rep.pools[0],
                                   wl.pool_pages, wl.page_size, wl.page_stride, rep.page_table,
                                   rep.seq_lens_k, rep.cu, wl.causal, 1, max_k, c, nc, max_cand,
                                   wl.topk, out, ws, dev_status=status)

    def dense_call():
        rep.call("scorer", 0)
        rep.call("topk", 0)

    def timed(fn, k):
        for _ in range(3):
            fn()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(k)]
        for s, e in ev:
            flush.fill_(1)
            s.record(stream)
            fn()
            e.record(stream)
        torch.cuda.synchronize()
        return sum(s.elapsed_time(e) for s, e in ev) / k

    k = max(3, min(args.steps, 20))
    cand_ms, dense_ms = timed(cand_call, k), timed(dense_call, k)
    keys = int(sum(min(int(n), 16) for n in n_cand)) * wl.page_size
    out_d = {"workload": wl.name, "candidate_blocks_per_query": 16, "candidate_keys": keys,
             "dense_keys": wl.pairs(), "steps": k, "launches_per_call": 4,
             "cand_us": round(cand_ms * 1e3, 2), "dense_scorer_topk_us": round(dense_ms * 1e3, 2),
             "cand_k_tokens_per_s": round(keys / (cand_ms / 1e3) / 1e3, 1),
             "status": int(status.item()), "l2": "256 MiB write before each timed call"}
    del rep, ws, flush
    torch.cuda.empty_cache()
    return out_d


def qk_prep_sweep(args, dev, peaks):
    """The fused QK pre-processing alone (idx_qk_prep: K LayerNorm + RoPE + FP8 store of T new
    keys, Q RoPE + per-(t,h) FP8 quant with the scale fold for T tokens), FP8, block 64, H=32,
    interleaved RoPE, at the token counts of the pages' fused-preprocessing table."""
    import torch
    stream = torch.cuda.current_stream()
    rows = []
    for T in (1, 8, 32, 64, 256, 1024):
        wl = W.make("prefill_fp8", seed=args.seed, B=1, cached=4096, new=T)
        rep = Replica(wl, 2, dev)
        for i in range(3):
            rep.call("qk_prep", i)
        k = 50
        ms = time_calls(torch, rep, ("qk_prep",), 3, k, stream)
        ab = algorithmic_bytes(wl)["qk_prep"]
        rows.append({"tokens": T, "us": round(ms * 1e3, 2), "bytes": ab,
                     "gbs": round(ab / (ms / 1e3) / 1e9, 1)})
        del rep
    return {"dtype": "fp8e4m3", "block_size": 64, "H": 32, "rope": "interleaved",
            "graph_of": 50, "rows": rows,
            "hbm_frac_at_1024": round(rows[-1]["gbs"] / peaks["hbm_gbs"], 4)}


def tensor_probe(torch, stream, iters=2000):
    """Dense tensor-core rate of tcgen05 kind::mxf4 and kind::f8f6f4 MMAs (M=128, N=256), one
    CTA per SM, timed with CUDA events."""
    from sparse_attention_indexer_mqa_gb300 import binding as Bn
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = {}
    for name, dt in (("mxf4", W.MXFP4), ("f8f6f4", W.FP8)):
        Bn.idx_debug_mma_rate(dt, 50, status)
        torch.cuda.synchronize()
        best = None
        for _ in range(3):
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record(stream)
            f = Bn.idx_debug_mma_rate(dt, iters, status)
            e.record(stream)
            torch.cuda.synchronize()
            t = s.elapsed_time(e) / 1e3
            best = t if best is None else min(best, t)
        out[f"{name}_tflops"] = round(f * sms / best / 1e12, 1)
    out["status"] = int(status.item())
    out["how"] = (f"{iters} x 8 back-to-back MMAs (M=128, N=256, K=64 mxf4 / K=32 e4m3) per SM on zero "
                  "operands into one TMEM accumulator, best of 3 launches")
    return out


def config_of(wl):
    return {"workload": wl.name, "B": wl.B, "H": wl.H, "D": 128,
            "seq_len_k": int(wl.seq_lens_k.max()), "page_size": wl.page_size,
            "topk": wl.topk, "queries": wl.T, "pairs": wl.pairs(), "causal": wl.causal,
            "parallelism": "one independent replica per rank (weak scaling)"}


def run_e2e(rep, args, torch, stream, world, dev):
    """The same step through the C ABI with host buffers: every step copies its inputs (new K
    rows, slots, positions, Q, positions, weights: one packed pinned host buffer) to the device
    in one H2D copy and reads its top-k indices back in one D2H copy.

    Pipelined: uploads and read-backs run on two more streams with two device input buffers
    and two top-k buffers used in turn, so step i+1's upload and step i's read-back overlap each
    other and step i's kernels, which stay in order on the compute stream. Serial: upload,
    kernels and read-back of each step one after the other. Both are timed; the value is the
    faster."""
    wl = rep.wl
    sr = wl.step_rows
    parts = [("k", wl.k[sr].view(np.int16), torch.int16), ("slot", wl.slot_mapping[sr], torch.int64),
             ("pos", wl.k_positions[sr], torch.int32), ("q", wl.q.view(np.int16), torch.int16),
             ("qpos", wl.q_positions, torch.int32), ("w", wl.w_in, torch.float32)]
    offs, o = {}, 0
    for n, a, _ in parts:
        offs[n] = o
        o += (a.nbytes + 255) // 256 * 256
    h_buf = torch.zeros(o, dtype=torch.uint8).pin_memory()
    hb = h_buf.numpy()
    for n, a, _ in parts:
        hb[offs[n]:offs[n] + a.nbytes] = np.ascontiguousarray(a).view(np.uint8).ravel()
    device = rep.q[0].device
    d_bufs = [torch.empty(o, dtype=torch.uint8, device=device) for _ in range(2)]
    tops = [torch.empty(tuple(rep.topk.shape), dtype=torch.int32, device=device) for _ in range(2)]
    dev_in = [dict({n: d[offs[n]:offs[n] + a.nbytes].view(dt).view(a.shape) for n, a, dt in parts},
                   topk_out=tops[j]) for j, d in enumerate(d_bufs)]
    h_tops = [torch.empty(tuple(rep.topk.shape), dtype=torch.int32).pin_memory() for _ in range(2)]
    h2d, d2h = o, h_tops[0].numel() * 4

    def serial(i):
        d_bufs[0].copy_(h_buf, non_blocking=True)
        rep.step(i, inputs=dev_in[0])
        h_tops[0].copy_(tops[0], non_blocking=True)

    up_stream = torch.cuda.Stream(device=device)    # host -> device uploads
    down_stream = torch.cuda.Stream(device=device)  # device -> host read-backs

    def pipelined(first, n):
        """n steps: uploads and read-backs on their own streams (two copy engines); the compute
        stream waits for a step's inputs and for the read-back that last used its top-k
        buffer."""
        comp = torch.cuda.current_stream()
        up_stream.wait_stream(comp)
        down_stream.wait_stream(comp)
        ev_in = [torch.cuda.Event() for _ in range(n)]
        ev_out = [torch.cuda.Event() for _ in range(n)]
        ev_back = [torch.cuda.Event() for _ in range(n)]
        with torch.cuda.stream(up_stream):
            d_bufs[0].copy_(h_buf, non_blocking=True)
            ev_in[0].record(up_stream)
        for i in range(n):
            comp.wait_event(ev_in[i])
            if i >= 2:  # top-k buffer i%2 was read back for step i-2
                comp.wait_event(ev_back[i - 2])
            rep.step(first + i, inputs=dev_in[i % 2])
            ev_out[i].record(comp)
            if i + 1 < n:
                with torch.cuda.stream(up_stream):
                    if i >= 1:  # input buffer (i+1)%2 was read by step i-1
                        up_stream.wait_event(ev_out[i - 1])
                    d_bufs[(i + 1) % 2].copy_(h_buf, non_blocking=True)
                    ev_in[i + 1].record(up_stream)
            with torch.cuda.stream(down_stream):
                down_stream.wait_event(ev_out[i])
                h_tops[i % 2].copy_(tops[i % 2], non_blocking=True)
                ev_back[i].record(down_stream)
        comp.wait_stream(up_stream)
        comp.wait_stream(down_stream)

    def timed(g):
        g.replay()
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        return rank_max(time_graph(torch, g, stream) / args.steps, world, dev)

    for i in range(args.warmup):
        serial(i)
    torch.cuda.synchronize()
    g_serial = capture(torch, lambda i: serial(args.warmup + i), args.steps)
    ms_serial = timed(g_serial)
    pipelined(0, args.warmup)
    torch.cuda.synchronize()
    g_pipe = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_pipe):
        pipelined(args.warmup, args.steps)
    ms = timed(g_pipe)
    # every step has the same inputs: the pipelined read-backs must equal a serial step's
    torch.cuda.synchronize()
    serial(0)
    torch.cuda.synchronize()
    ref = h_tops[0].clone()
    g_pipe.replay()
    torch.cuda.synchronize()
    for h in h_tops[: min(2, args.steps)]:
        if not torch.equal(h, ref):
            raise RuntimeError("pipelined end-to-end steps returned a different top-k")
    # the value is the faster of the two schedules (both copy every step's inputs and results;
    # with very large copies the overlapped one can lose)
    best = min(ms, ms_serial)
    return {"value": round(job_rate(wl.pairs(), best, world), 1), "unit": "K-tokens/s",
            "ms_per_step": round(best, 5), "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h),
            "schedule": "pipelined" if ms <= ms_serial else "serial",
            "pipelined_ms_per_step": round(ms, 5),
            "serial_ms_per_step": round(ms_serial, 5),
            "how": "K steps in one CUDA graph; each step: one packed H2D of its inputs from pinned "
                   "host, 3 library calls, one D2H of its top-k. pipelined: uploads and read-backs "
                   "on their own streams with double-buffered inputs/outputs overlap each other and "
                   "the neighbouring steps' kernels; serial: upload, kernels and read-back one after "
                   "the other; value and ms_per_step: the faster of the two"}


# ----------------------------------------------------------------------------------------
# CPU side: the oracle as it stands, timed on this host's cores

def oracle_step(wl, pool, rows, n_threads):
    """One oracle step on a sample: K store of the step's new keys, Q quant of the sampled
    query rows, fp64 scoring and top-k of those rows. Returns the pairs scored."""
    import oracle as O
    sr = wl.step_rows
    O.k_store(pool, wl.k[sr], wl.slot_mapping[sr], wl.k_positions[sr], wl.cos_sin, wl.k_rope,
              wl.k_norm, wl.dtype, wl.pool_pages, wl.page_size, wl.page_stride)
    qc_s, qs_s, w_s = O.q_quant(wl.q[rows], wl.q_positions[rows], wl.cos_sin, wl.q_rope,
                                wl.w_in[rows], wl.softmax_scale, wl.head_scale, wl.dtype)
    qc = np.zeros((wl.T,) + qc_s.shape[1:], qc_s.dtype)
    qs = np.zeros((wl.T,) + qs_s.shape[1:], qs_s.dtype)
    w = np.zeros((wl.T, wl.H), np.float32)
    qc[rows], qs[rows], w[rows] = qc_s, qs_s, w_s
    lg = O.mqa_logits(qc, qs, w, wl.dtype, pool, wl.pool_pages, wl.page_size, wl.page_stride,
                      wl.page_table, wl.seq_lens_k, wl.cu_seqlens_q, wl.causal, wl.ld_logits,
                      rows=rows, n_threads=n_threads)
    O.topk(np.nan_to_num(lg, nan=-np.inf), wl.seq_lens_k, wl.cu_seqlens_q, wl.causal, wl.topk,
           rows=rows, n_threads=n_threads)
    return int(wl.visible()[rows].sum())


def sample_rows(wl, n):
    """n query rows spread evenly over all queries (all rows if n >= T)."""
    if n is None or n >= wl.T:
        return np.arange(wl.T, dtype=np.int64)
    return np.unique(np.linspace(0, wl.T - 1, n).round().astype(np.int64))


def oracle_pool(wl):
    import oracle as O
    pool = np.zeros(wl.pool_pages * wl.page_stride, np.uint8)
    O.k_store(pool, wl.k, wl.slot_mapping, wl.k_positions, wl.cos_sin, wl.k_rope, wl.k_norm,
              wl.dtype, wl.pool_pages, wl.page_size, wl.page_stride)
    return pool


def cpu_baseline(wl, budget_s=15.0, rows_per_step=None):
    """Oracle step (K store of the new keys, Q quant, scoring + top-k of a sample of query
    rows) on all host cores; value in K-tokens/s."""
    n_threads = os.cpu_count() or 1
    pool = oracle_pool(wl)
    rows = sample_rows(wl, rows_per_step)
    t0 = time.perf_counter()
    pairs = 0
    reps = 0
    while True:
        pairs += oracle_step(wl, pool, rows, n_threads)
        reps += 1
        if time.perf_counter() - t0 > budget_s or reps >= 50:
            break
    dt = time.perf_counter() - t0
    # the same step on one core (one step, or a quarter of the sampled rows when that is long)
    rows1 = rows if len(rows) <= 16 else rows[:: max(1, len(rows) // 16)]
    t1 = time.perf_counter()
    pairs1 = oracle_step(wl, pool, rows1, 1)
    dt1 = time.perf_counter() - t1
    return {"value": round(pairs / dt / 1e3, 3), "unit": "K-tokens/s", "cores": n_threads,
            "kind": "oracle",
            "sample": f"{reps} oracle step(s): K store of {len(wl.step_rows)} new keys, Q quant, "
                      f"fp64 scoring and top-k of {len(rows)} of {wl.T} queries spread evenly "
                      f"({pairs // reps} pairs per step), {dt:.1f} s",
            "single_core": {"value": round(pairs1 / dt1 / 1e3, 3), "unit": "K-tokens/s",
                            "sample": f"one step on one thread, {len(rows1)} query rows, {dt1:.1f} s"}}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    wl = W.make(args.config, seed=args.seed)
    n_threads = os.cpu_count() or 1
    pool = oracle_pool(wl)
    # decode: every query of the step (the GPU arm's exact workload); prefill: an even sample
    rows = sample_rows(wl, None if is_decode(wl) else args.ref_rows)
    for _ in range(args.warmup):
        oracle_step(wl, pool, rows, n_threads)
    t0 = time.perf_counter()
    pairs = 0
    for _ in range(args.steps):
        pairs += oracle_step(wl, pool, rows, n_threads)
    dt = time.perf_counter() - t0
    v = round(pairs / dt / 1e3, 3)
    return {
        "impl": "reference",
        "metric": metric_name(wl),
        "value": v, "unit": "K-tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (same seeded workload as the GPU arm)", "config": config_of(wl),
        "cpu_baseline": {"value": v, "unit": "K-tokens/s", "cores": n_threads, "kind": "oracle",
                         "sample": f"each step: K store of {len(wl.step_rows)} new keys, Q quant, "
                                   f"scoring + top-k of {len(rows)} of {wl.T} queries spread evenly"},
        "e2e": {"value": v, "unit": "K-tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# the sources each kernel is built from (a stored DRAM-traffic figure counts only while they
# are unchanged)
DECODE_SOURCES = ["sparse_attention_indexer_mqa_gb300/csrc/scorer_decode.cu",
                  "sparse_attention_indexer_mqa_gb300/csrc/tc.cuh",
                  "sparse_attention_indexer_mqa_gb300/csrc/common.cuh",
                  "sparse_attention_indexer_mqa_gb300/csrc/select.cuh"]
PREFILL_SOURCES = ["sparse_attention_indexer_mqa_gb300/csrc/scorer_prefill.cu",
                   "sparse_attention_indexer_mqa_gb300/csrc/tc.cuh",
                   "sparse_attention_indexer_mqa_gb300/csrc/common.cuh",
                   "sparse_attention_indexer_mqa_gb300/csrc/select.cuh"]
COMPRESS_SOURCES = ["sparse_attention_indexer_mqa_gb300/csrc/quant.cu",
                    "sparse_attention_indexer_mqa_gb300/csrc/common.cuh"]


def run_block(args):
    """One block of the default run, alone on cuda:0 (for a profiler's launch list)."""
    import torch
    from sparse_attention_indexer_mqa_gb300 import binding as Bn
    Bn.load()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    peaks, peak_kind = measured_peaks()
    if args.only == "compress":
        return compress_block(args, dev, peaks)
    if args.only == "cand":
        return cand_block(args, dev, peaks)
    if args.only == "prefill":
        return prefill_block(args, dev, peaks, peak_kind)
    if args.only == "qk_prep_sweep":
        return qk_prep_sweep(args, dev, peaks)
    return tensor_probe(torch, torch.cuda.current_stream())


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default="decode_b64", choices=sorted(W.BUILDERS))
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ref-rows", type=int, default=8,
                    help="query rows per step of the reference arm on prefill configs (decode: all)")
    ap.add_argument("--no-prefill", action="store_true", help="skip the prefill block of the default run")
    ap.add_argument("--no-probe", action="store_true", help="skip the tensor-core rate probe")
    ap.add_argument("--no-compress", action="store_true", help="skip the compressed K store block")
    ap.add_argument("--no-cand", action="store_true", help="skip the candidate-pool block")
    ap.add_argument("--only", choices=["compress", "cand", "prefill", "qk_prep_sweep", "tensor_probe"],
                    help="run one block of the default run alone and print it (profiling)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        line = run_reference(args, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    if args.only:
        print(json.dumps({"only": args.only, args.only: run_block(args)}), flush=True)
        return
    if world > 1:
        import torch
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        torch.distributed.init_process_group("nccl")
    line = run_gpu(args, rank, world)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
