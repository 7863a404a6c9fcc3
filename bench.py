#!/usr/bin/env python3
"""Benchmark of LazyAttention decode (and prefill) over a paged, position-agnostic KV cache.

Default workload: Llama-3.1-8B-shaped decode, bf16, 32 q / 8 KV heads, d=128,
batch 64, contexts of 8 Zipf(1.0)-drawn 512-token documents from a 256-document
pool plus a 64-token private suffix (4160 tokens), RoPE theta 5e5. One step is
one shared-run decode call (lazy_attn_decode_shared: work-item kernel + combine)
for the whole batch, one layer; the per-sequence entry point (lazy_attn_decode) is
timed beside it.

Prints ONE JSON line (rank 0). ``value`` is logical KV GB/s: K+V bytes of every
token of every context divided by the device time of the decode call, inputs
resident in HBM, L2 flushed between steps (written, then read, so no dirty lines remain). Extra keys carry the roofline against
the unique-block HBM bound, the no-sharing control, the lazy-vs-pre-rotated
overhead, prefill TFLOP/s, an end-to-end figure through host buffers, clocks and
the CPU oracle baseline.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
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

METRIC = "LazyAttn decode KV GB/s (% HBM peak); prefill TFLOP/s; lazy-RoPE overhead %"
WORKLOAD = "llama8b_decode"

# DRAM bytes (read + write) per launch of the shared-run decode kernel on this workload,
# from the ncu capture summarised in profiles/; valid only while the kernel's sources
# hash to the value recorded with it (otherwise the bench reports traffic as null).
NCU_TRAFFIC = {"sources": ["paged_kv_cache_57_gb300/csrc/decode_shared.cu",
                           "paged_kv_cache_57_gb300/csrc/decode_block.cuh",
                           "paged_kv_cache_57_gb300/csrc/common.cuh"],
               "sha16": "54297fb7bc4f9285", "bytes_per_launch": 302164480 + 9733632}


def _traffic_if_current():
    import hashlib
    h = hashlib.sha256()
    try:
        for f in NCU_TRAFFIC["sources"]:
            with open(os.path.join(ROOT, f), "rb") as fh:
                h.update(fh.read())
    except OSError:
        return None
    return NCU_TRAFFIC["bytes_per_launch"] if h.hexdigest()[:16] == NCU_TRAFFIC["sha16"] else None


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), float(j["bf16_tflops"]), float(j.get("bf16_tflops_sustained", j["bf16_tflops"])), \
            "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


# ------------------------------------------------------------------ clocks

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index, self.samples, self.proc = index, [], None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            # nvidia-smi takes a moment to print its first line: wait for it (at most 3 s)
            # so that the samples cover the timed region from its start
            t0 = time.perf_counter()
            while not self.samples and self.proc.poll() is None and time.perf_counter() - t0 < 3.0:
                time.sleep(0.01)
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) == 7:
                self.samples.append(parts)

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.thread.join(timeout=5)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        sm = [float(s[0]) for s in self.samples if s[0].replace(".", "").isdigit()]
        mx = [float(s[1]) for s in self.samples if s[1].replace(".", "").isdigit()]
        reasons = sorted({names[i] for s in self.samples for i in range(4) if s[3 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(self.samples)}


# ------------------------------------------------------------------ multi-rank helpers

def rank_seed(rank: int, base: int = 20260002) -> int:
    """Weak scaling: every rank decodes its own batch, drawn with its own seed."""
    return base + 1000 * rank


def max_over_ranks(t: float, dist=None, device="cpu") -> float:
    """The slowest rank's time (the whole job's time); identity on one rank."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return t
    import torch
    tt = torch.tensor([t], dtype=torch.float64, device=device)
    dist.all_reduce(tt, op=dist.ReduceOp.MAX)
    return float(tt.item())


def whole_job_rate(bytes_per_rank_step: float, world: int, steps: int, t_max: float) -> float:
    """Aggregate GB/s over all ranks: every rank processes the same volume per step."""
    return world * bytes_per_rank_step * steps / t_max / 1e9


# ------------------------------------------------------------------ helpers

def build_device(w, lazy=True, k_pool=None):
    import torch
    from paged_kv_cache_57_gb300 import lazy_attn as L
    p = L.make_params(num_seqs=w.num_seqs, num_q_heads=w.num_q_heads, num_kv_heads=w.num_kv_heads,
                      head_dim=w.head_dim, num_pool_blocks=w.num_pool_blocks,
                      max_blocks_per_seq=max(1, w.max_blocks_per_seq), dtype=w.dtype, rope_theta=w.rope_theta,
                      lazy=lazy)
    c = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()
    words, seq_lens = L.pack_block_words(p, len(w.doc_len), c(w.seg_indptr), c(w.seg_doc), c(w.seg_len),
                                         c(w.seq_pos0), c(w.doc_block_indptr), c(w.doc_blocks))
    d = dict(p=p, q=w.q.cuda(), k=(w.k_pool if k_pool is None else k_pool).cuda(), v=w.v_pool.cuda(), words=words,
             seq_lens=seq_lens, rope=L.rope_table_init(p))
    if w.kind == "decode":
        d["q_pos"] = c(w.q_pos)
        d["ws"] = torch.empty(max(1, L.decode_workspace_bytes(p)), dtype=torch.uint8, device="cuda")
        d["out"] = torch.empty_like(d["q"])
        if w.dtype == "bf16":  # shared-run plan (host planner, copied to the device)
            items, slot_indptr = L.plan_shared_host(p, len(w.doc_len), w.seg_indptr, w.seg_doc, w.seg_len,
                                                    w.doc_block_indptr, w.doc_blocks)
            d["plan"] = L.SharedPlan(items, slot_indptr)
            d["ws_sh"] = torch.empty(max(1, L.decode_shared_workspace_bytes(p, d["plan"].num_slots)),
                                     dtype=torch.uint8, device="cuda")
    else:
        d["cu"] = c(w.cu_seqlens_q)
        d["q_start"] = c(w.q_start)
        d["max_q"] = int(np.diff(w.cu_seqlens_q).max())
        d["out"] = torch.empty_like(d["q"])
        d["ws_pf"] = torch.empty(max(1, L.prefill_workspace_bytes(p, int(d["q"].shape[0]))), dtype=torch.uint8,
                                 device="cuda")
    return d


def run_decode(d, lazy=None, path="shared"):
    """One decode call: ``shared`` = lazy_attn_decode_shared (each cited document chunk read
    once per KV head for the whole batch), ``seq`` = lazy_attn_decode (per sequence)."""
    from paged_kv_cache_57_gb300 import lazy_attn as L
    p = d["p"]
    if lazy is not None:
        p.lazy = int(lazy)
    if path == "shared":
        L.decode_shared(p, d["q"], d["k"], d["v"], d["words"], d["q_pos"], d["rope"], d["plan"], out=d["out"],
                        workspace=d["ws_sh"])
    else:
        L.decode(p, d["q"], d["k"], d["v"], d["words"], d["seq_lens"], d["q_pos"], d["rope"], out=d["out"],
                 workspace=d["ws"])


def run_prefill(d, lazy=None):
    from paged_kv_cache_57_gb300 import lazy_attn as L
    p = d["p"]
    if lazy is not None:
        p.lazy = int(lazy)
    L.prefill(p, d["q"], d["cu"], d["q_start"], d["max_q"], d["k"], d["v"], d["words"], d["seq_lens"], d["rope"],
              out=d["out"], workspace=d["ws_pf"])


class L2Flush:
    """Evicts L2 before a timed step: writes a buffer of twice the L2 size (256 MB at
    least), then reads a second one of the same size. The step then starts with a
    cold L2 that holds no dirty lines: the written buffer's write-back to HBM
    happens during the read pass, outside the timed region, instead of competing
    with the step's own reads."""

    def __init__(self, device):
        import torch
        l2 = torch.cuda.get_device_properties(device).L2_cache_size
        n = max(2 * l2, 256 << 20) // 4
        self.w = torch.empty(n, dtype=torch.float32, device="cuda")
        self.r = torch.zeros(n, dtype=torch.float32, device="cuda")
        self.acc = torch.zeros((), dtype=torch.float32, device="cuda")

    def __call__(self):
        import torch
        self.w.add_(1)
        torch.sum(self.r, dim=0, out=self.acc)


L2_NOTE = "flushed before every step: 2x L2 written, then 2x L2 read (cold L2, no dirty lines)"


def time_steps(fn, steps, warmup, flush):
    """Per-step device time (s) with CUDA events on the launching stream, L2 flushed before each step."""
    import torch
    st = torch.cuda.current_stream()
    for _ in range(warmup):
        flush()
        fn()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for a, b in evs:
        flush()
        a.record(st)
        fn()
        b.record(st)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) * 1e-3 for a, b in evs]


def decode_bytes(w):
    from paged_kv_cache_57_gb300 import workloads as W
    elt = 2 if w.dtype == "bf16" else 4
    io = 2 * w.q.numel() * elt + 4 * w.num_seqs * (max(1, w.max_blocks_per_seq) + 2)
    return dict(logical=W.kv_bytes_logical(w) + io, unique=W.kv_bytes_unique(w) + io, blocks=W.kv_bytes_blocks(w) + io,
                kv_logical=W.kv_bytes_logical(w))


def prefill_flops(w):
    """4 d Hq sum_s (C_s N_ctx,s + C_s (C_s + 1) / 2): exact causal count, no rotation."""
    cu = np.asarray(w.cu_seqlens_q)
    tot = 0
    for s in range(w.num_seqs):
        C = int(cu[s + 1] - cu[s])
        nctx = int(w.tokens_per_seq()[s]) - C
        tot += C * nctx + C * (C + 1) // 2
    return 4 * w.head_dim * w.num_q_heads * tot


# ------------------------------------------------------------------ CPU oracle legs

def oracle_sample_rate(w, budget_s=10.0, seqs_per_call=2):
    """Runs the oracle over consecutive sequences of ``w`` until ``budget_s`` has elapsed;
    returns (logical KV GB/s, seconds, sequences, threads)."""
    import oracle
    oracle.build()
    elt = 2 if w.dtype == "bf16" else 4
    toks = w.tokens_per_seq()
    t0 = time.perf_counter()
    done, nbytes = 0, 0
    while True:
        rows = [(done + i) % w.num_seqs for i in range(seqs_per_call)]
        oracle.attention(w, rows=rows)
        nbytes += int(sum(toks[r] for r in rows)) * w.num_kv_heads * w.head_dim * 2 * elt
        done += seqs_per_call
        el = time.perf_counter() - t0
        if el >= budget_s:
            return nbytes / el / 1e9, el, done, oracle.num_threads()


def _prefill_row_flops(w):
    """Algorithmic FLOPs of each query row of a prefill workload: 4 d Hq x visible keys."""
    toks = w.tokens_per_seq()
    cu = np.asarray(w.cu_seqlens_q)
    keys = np.concatenate([toks[s] - (cu[s + 1] - cu[s]) + np.arange(1, cu[s + 1] - cu[s] + 1)
                           for s in range(w.num_seqs)])
    return 4.0 * w.head_dim * w.num_q_heads * keys


def cpu_baseline_table(budget_s=1.0, workloads=None):
    """The oracle as it stands (fp64, materialised position-adjusted K, one-shot
    softmax) on the host cores, with every thread and with one, on each workload the
    GPU legs run. A cell runs consecutive units (sequences, or prefill query rows)
    until ``budget_s`` has passed (at least one call) and reports the rate in the
    workload's unit; the mixed batch's prefill chunks are sampled at 64 rows per chunk
    and their step time extrapolated from that rate."""
    import oracle
    from paged_kv_cache_57_gb300 import workloads as W
    oracle.build()
    all_threads = oracle.num_threads()
    wl = dict(workloads or {})  # workloads the GPU legs already built, reused
    if "mixed_mqa_decode" not in wl or "mixed_mqa_prefill" not in wl:
        wl["mixed_mqa_decode"], wl["mixed_mqa_prefill"] = W.mixed_mqa()
    for name in ("llama8b_decode", "llama8b_prefill", "llama70b_decode"):
        if name not in wl:
            wl[name] = W.FULL[name]()
    loads = [("tiny_fp32", W.tiny_fp32())] + [(n, wl[n]) for n in ("llama8b_decode", "llama8b_prefill",
                                                                   "llama70b_decode", "mixed_mqa_decode",
                                                                   "mixed_mqa_prefill")]
    out = []
    try:
        for name, w in loads:
            for threads in (all_threads, 1):
                oracle.set_num_threads(threads)
                t0 = time.perf_counter()
                if w.kind == "decode":
                    elt = 2 if w.dtype == "bf16" else 4
                    toks = w.tokens_per_seq()
                    done, nbytes = 0, 0
                    while True:
                        r = done % w.num_seqs
                        oracle.attention(w, rows=[r])
                        nbytes += int(toks[r]) * w.num_kv_heads * w.head_dim * 2 * elt
                        done += 1
                        if time.perf_counter() - t0 >= budget_s:
                            break
                    el = time.perf_counter() - t0
                    rate = nbytes / el / 1e9
                    step_bytes = float(W.kv_bytes_logical(w))
                    out.append({"workload": name, "threads": threads, "value": rate, "unit": "GB/s",
                                "sample": f"{done} sequences, {el:.2f} s", "step_s": step_bytes / 1e9 / rate})
                else:
                    fl = _prefill_row_flops(w)
                    cu = np.asarray(w.cu_seqlens_q)
                    if name == "mixed_mqa_prefill":  # 64 rows spread over each chunk
                        rows = np.concatenate([cu[s] + np.linspace(0, cu[s + 1] - cu[s] - 1, 64).astype(np.int64)
                                               for s in range(w.num_seqs)])
                    else:
                        rows = np.arange(int(cu[-1]))
                    done, flop = 0, 0.0
                    while True:
                        take = rows[done: done + 8]
                        if len(take) == 0:
                            break
                        oracle.attention(w, rows=take.tolist())
                        flop += float(fl[take].sum())
                        done += len(take)
                        if time.perf_counter() - t0 >= budget_s:
                            break
                    el = time.perf_counter() - t0
                    rate = flop / el / 1e9
                    cell = {"workload": name, "threads": threads, "value": rate, "unit": "GFLOP/s",
                            "sample": f"{done} query rows, {el:.2f} s", "step_s": float(fl.sum()) / 1e9 / rate}
                    if name == "mixed_mqa_prefill":
                        cell["step_s_extrapolated"] = True
                    out.append(cell)
    finally:
        oracle.set_num_threads(all_threads)
    return out


def reference_arm(args):
    """The oracle timed on the host cores, as the reference arm: each step is the
    whole headline batch (64 sequences x 32 query heads), as the GPU arm's step."""
    import oracle
    from paged_kv_cache_57_gb300 import workloads as W
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    w = W.FULL[WORKLOAD]()
    oracle.build()
    elt = 2
    toks = w.tokens_per_seq()
    step_bytes = int(toks.sum()) * w.num_kv_heads * w.head_dim * 2 * elt
    times = []
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        oracle.attention(w)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            times.append(dt)
    total = sum(times)
    value = step_bytes * len(times) / total / 1e9
    cores = oracle.num_threads()
    line = {"metric": METRIC, "value": value, "unit": "GB/s", "impl": "reference", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / len(times),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "batch": w.num_seqs, "context": int(toks[0]),
                       "heads": [w.num_q_heads, w.num_kv_heads], "head_dim": w.head_dim,
                       "step": "the whole batch, all heads (the GPU arm's step)"},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle",
                             "sample": f"{args.steps} steps of {w.num_seqs} sequences"},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ our arm

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)  # ~0.5 s timed: several 100 ms clock samples
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true", help="headline decode only (used for ncu launch lists)")
    ap.add_argument("--decode-path", default="shared", choices=["shared", "seq"],
                    help="decode entry point timed by --workload (shared-run or per-sequence)")
    ap.add_argument("--kv-dtype", default="bf16", choices=["bf16", "fp8_e4m3"],
                    help="pools timed by --workload (fp8_e4m3: quantised copies)")
    ap.add_argument("--workload", default=None, choices=sorted(["llama8b_decode", "llama8b_decode_noshare",
                                                                "llama8b_prefill", "llama70b_decode",
                                                                "llama70b_decode_noshare", "mixed_mqa_decode",
                                                                "mixed_mqa_prefill"]),
                    help="time one workload alone and print its own line (used for ncu captures)")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    if args.impl == "reference":
        return reference_arm(args)
    if args.workload:
        return single_workload(args)

    import torch
    import torch.distributed as dist
    from paged_kv_cache_57_gb300 import build
    from paged_kv_cache_57_gb300 import workloads as W

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl")
    if rank == 0:
        build.build()
    if world > 1:
        dist.barrier()
    build.build()  # no-op once built
    from paged_kv_cache_57_gb300 import lazy_attn as L

    hbm, tf_burst, tf_sust, peak_src = _peaks()
    # Weak scaling: each rank decodes its own batch (a different seed), no data exchange.
    w = W.decode_zipf(WORKLOAD, batch=64, hq=32, hkv=8, docs_per_seq=8, doc_tokens=512, pool_docs=256,
                      zipf_s=1.0, suffix_tokens=64, seed=rank_seed(rank))
    d = build_device(w)
    nbytes = decode_bytes(w)
    flush = L2Flush(local)

    clocks = ClockSampler(local)
    clocks.start()
    fn = lambda: run_decode(d, lazy=True)
    for _ in range(args.warmup):
        flush()
        fn()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    launches0 = L.launch_count()
    t_wall0 = time.perf_counter()
    per_step = time_steps(fn, args.steps, 0, flush)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    t_wall = time.perf_counter() - t_wall0
    launches = L.launch_count() - launches0
    clk = clocks.stop()
    t_dev = sum(per_step)
    t_max = max_over_ranks(t_dev, dist if world > 1 else None, device="cuda")
    ms = 1e3 * t_max / args.steps
    value = whole_job_rate(nbytes["kv_logical"], world, args.steps, t_max)
    call_avg = t_dev / args.steps

    # The dominant kernel alone: the same decode as its two calls (work-item kernel,
    # then combine), with CUDA events on the launching stream around the first.
    kern = time_split_phase(d, min(max(20, args.steps), 300), 3, flush)
    k_avg = statistics.mean(kern["partials"])
    achieved = nbytes["unique"] / k_avg / 1e9

    extras, keep = {}, {}
    if not args.no_extras and rank == 0:
        extras, keep = measure_extras(args, d, w, flush, hbm, tf_burst, tf_sust)
    e2e = measure_e2e(args, d, w, nbytes) if rank == 0 else None

    if world > 1:
        dist.barrier()
    if rank != 0:
        dist.destroy_process_group()
        return 0
    lz = extras.get("lazy_overhead_pct", {})
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD, "batch": w.num_seqs, "context": int(w.tokens_per_seq()[0]),
                   "heads": [w.num_q_heads, w.num_kv_heads], "head_dim": w.head_dim, "rope_theta": w.rope_theta,
                   "docs": "8 x 512 Zipf(1.0) of 256 + 64 private", "l2": L2_NOTE,
                   "decode_path": "shared-run (lazy_attn_decode_shared)",
                   "parallelism": f"weak x{world} (independent batches)"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                     "traffic": _traffic_if_current(), "peak_source": peak_src,
                     "kernel": "decode_shared_kernel<128, lazy> alone: mean of CUDA-event durations around "
                               "lazy_attn_decode_shared_partials; bytes = unique K/V blocks + q + out + words",
                     "kernel_ms": 1e3 * k_avg, "bytes_per_launch": nbytes["unique"],
                     "call_ms": 1e3 * call_avg, "call_achieved": nbytes["unique"] / call_avg / 1e9,
                     "call_frac": nbytes["unique"] / call_avg / 1e9 / hbm,
                     "lazy_overhead_pct": lz.get("decode"),
                     "lazy_overhead_pct_per_sequence_path": lz.get("decode_per_sequence_path")},
        "decode": {"tokens_per_s": world * w.num_seqs / (t_max / args.steps),
                   "kv_gbs_logical": value, "kv_gbs_unique": world * nbytes["unique"] * args.steps / t_max / 1e9,
                   "bytes_logical": nbytes["logical"], "bytes_unique": nbytes["unique"],
                   "hbm_frac_unique_of_measured": nbytes["unique"] / call_avg / 1e9 / hbm,
                   "hbm_frac_unique_of_8tbs": nbytes["unique"] / call_avg / 1e9 / 8000.0,
                   "ms_median": 1e3 * statistics.median(per_step),
                   "combine_ms": 1e3 * statistics.mean(kern["combine"])},
        "gpu_launches": launches, "wall_s_timed": t_wall, "clocks": clk, "e2e": e2e,
    }
    line.update(extras)
    if not args.no_cpu_baseline:
        table = cpu_baseline_table(budget_s=0.7, workloads=keep.get("workloads"))
        head = next(c for c in table if c["workload"] == WORKLOAD and c["threads"] > 1)
        line["cpu_baseline"] = {"value": head["value"], "unit": "GB/s", "cores": head["threads"], "kind": "oracle",
                                "sample": f"{WORKLOAD}: {head['sample']}; table: every workload, all threads "
                                          f"and 1", "table": table}
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def time_split_phase(d, steps, warmup, flush):
    """The shared-run decode as its two calls, lazy_attn_decode_shared_partials and
    lazy_attn_decode_shared_combine, with CUDA events on the launching stream before,
    between and after them; L2 flushed before each step. Returns per-step seconds of
    each call. The host issues more per step here (two calls, three events) than in
    the one-call loop; a short device-side wait after each flush keeps the launches
    ahead of the device, so that no event interval includes the device waiting for
    the host."""
    import torch
    from paged_kv_cache_57_gb300 import lazy_attn as L
    st = torch.cuda.current_stream()
    p, plan = d["p"], d["plan"]
    p.lazy = 1

    def run():
        L.decode_shared_partials(p, d["q"], d["k"], d["v"], d["words"], d["q_pos"], d["rope"], plan, d["ws_sh"])

    for _ in range(warmup):
        flush()
        run()
        L.decode_shared_combine(p, plan, d["ws_sh"], d["out"])
    torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    spin = getattr(torch.cuda, "_sleep", None)
    for a, b, c in evs:
        flush()
        if spin is not None:
            spin(100000)  # about 50 us of device time, before the first event
        a.record(st)
        run()
        b.record(st)
        L.decode_shared_combine(p, plan, d["ws_sh"], d["out"])
        c.record(st)
    torch.cuda.synchronize()
    return {"partials": [a.elapsed_time(b) * 1e-3 for a, b, _ in evs],
            "combine": [b.elapsed_time(c) * 1e-3 for _, b, c in evs]}


def single_workload(args):
    """One workload on one GPU, timed alone: the command the ncu captures run."""
    import torch
    from paged_kv_cache_57_gb300 import build
    from paged_kv_cache_57_gb300 import workloads as W
    torch.cuda.set_device(0)
    build.build()
    w = W.FULL[args.workload]()
    d = build_device(w)
    flush = L2Flush(0)
    if w.kind == "decode" and args.kv_dtype == "fp8_e4m3":
        from paged_kv_cache_57_gb300 import lazy_attn as L
        k8, v8, ks, vs = W.fp8_pools(w)
        k8, v8 = k8.cuda(), v8.cuda()
        p8 = L.make_params(num_seqs=w.num_seqs, num_q_heads=w.num_q_heads, num_kv_heads=w.num_kv_heads,
                           head_dim=w.head_dim, num_pool_blocks=w.num_pool_blocks,
                           max_blocks_per_seq=d["p"].max_blocks_per_seq, dtype=w.dtype, rope_theta=w.rope_theta,
                           kv_dtype="fp8_e4m3", k_scale=ks, v_scale=vs)
        if args.decode_path == "shared":  # planned for e4m3 pools (items of at most 64 rows)
            items, slot_indptr = L.plan_shared_host(p8, len(w.doc_len), w.seg_indptr, w.seg_doc, w.seg_len,
                                                    w.doc_block_indptr, w.doc_blocks)
            plan8 = L.SharedPlan(items, slot_indptr)
            ws8 = torch.empty(max(1, L.decode_shared_workspace_bytes(p8, plan8.num_slots)), dtype=torch.uint8,
                              device="cuda")
            fn = lambda: L.decode_shared(p8, d["q"], k8, v8, d["words"], d["q_pos"], d["rope"], plan8, out=d["out"],
                                         workspace=ws8)
        else:
            fn = lambda: L.decode(p8, d["q"], k8, v8, d["words"], d["seq_lens"], d["q_pos"], d["rope"], out=d["out"],
                                  workspace=d["ws"])
        t = time_steps(fn, args.steps, args.warmup, flush)
        v, unit = decode_bytes(w)["kv_logical"] / 2 / statistics.median(t) / 1e9, "GB/s"  # e4m3 bytes
    elif w.kind == "decode":
        t = time_steps(lambda: run_decode(d, lazy=True, path=args.decode_path), args.steps, args.warmup, flush)
        v, unit = decode_bytes(w)["kv_logical"] / statistics.median(t) / 1e9, "GB/s"
    else:
        t = time_steps(lambda: run_prefill(d, lazy=True), args.steps, args.warmup, flush)
        v, unit = prefill_flops(w) / statistics.median(t) / 1e12, "TFLOP/s"
    print(json.dumps({"workload": args.workload, "value": v, "unit": unit, "steps": args.steps,
                      "warmup": args.warmup, "ms_median": 1e3 * statistics.median(t)}), flush=True)
    return 0


def measure_e2e(args, d, w, nbytes):
    """The decode end to end through the public API, as a serving step whose batch
    composition may change every step. Timed on the host clock, per step: the host
    planner (lazy_attn_plan_shared_host) and the host packer
    (lazy_attn_pack_block_words_host) write the plan and the block words into one
    pinned staging buffer that also holds q and the query positions; one host-to-device
    copy; lazy_attn_decode_shared; the output read back; a stream synchronisation.
    The KV pool is the resident cache (it persists across steps), not a per-step
    input. Beside it: the host planner and packer times alone, and the same step with
    the plan and words kept from the previous step (device time between CUDA events)."""
    import torch
    from paged_kv_cache_57_gb300 import lazy_attn as L
    steps = max(3, min(args.steps, 50))
    p, plan = d["p"], d["plan"]
    cap = int(plan.num_items) + 64  # item capacity of the staging buffer
    B = w.num_seqs
    shapes = [("q", d["q"].shape, torch.bfloat16), ("words", (B, p.max_blocks_per_seq), torch.int32),
              ("q_pos", (B,), torch.int32), ("items", (cap, L.PLAN_ITEM_INTS), torch.int32),
              ("slot_indptr", (B + 1,), torch.int32)]
    offs, total = {}, 0
    for name, shp, dt in shapes:  # 256-byte aligned slices of one buffer
        offs[name] = total
        total += (int(np.prod(shp)) * torch.empty((), dtype=dt).element_size() + 255) // 256 * 256
    hbuf = torch.empty(total, dtype=torch.uint8).pin_memory()
    dbuf = torch.empty(total, dtype=torch.uint8, device="cuda")

    def view(buf, name):
        _, shp, dt = next(x for x in shapes if x[0] == name)
        n = int(np.prod(shp)) * torch.empty((), dtype=dt).element_size()
        return buf[offs[name]: offs[name] + n].view(dt).view(shp)
    view(hbuf, "q").copy_(d["q"].cpu())
    view(hbuf, "q_pos").copy_(d["q_pos"].cpu())
    h_items, h_si = view(hbuf, "items").numpy(), view(hbuf, "slot_indptr").numpy()
    h_words = view(hbuf, "words").numpy().view(np.uint32)
    h_lens = np.zeros(B, np.int32)
    counts = np.zeros(2, np.int32)
    q, words, qp, items, slot_indptr = (view(dbuf, n) for n in ("q", "words", "q_pos", "items", "slot_indptr"))
    dplan = L.SharedPlan.__new__(L.SharedPlan)
    dplan.__dict__.update(plan.__dict__)
    dplan.items, dplan.slot_indptr = items, slot_indptr
    hout = torch.empty_like(d["out"], device="cpu").pin_memory()
    st = torch.cuda.current_stream()
    plan_args = (p, len(w.doc_len), w.seg_indptr, w.seg_doc, w.seg_len, w.doc_block_indptr, w.doc_blocks)

    def plan_and_pack():
        L.plan_shared_host(*plan_args, out=(h_items, h_si, counts))
        L.pack_block_words_host(p, len(w.doc_len), w.seg_indptr, w.seg_doc, w.seg_len, w.seq_pos0,
                                w.doc_block_indptr, w.doc_blocks, out=(h_words, h_lens))
        dplan.num_items, dplan.num_slots = int(counts[0]), int(counts[1])

    def step():
        dbuf.copy_(hbuf, non_blocking=True)
        L.decode_shared(p, q, d["k"], d["v"], words, qp, d["rope"], dplan, out=d["out"], workspace=d["ws_sh"])
        hout.copy_(d["out"], non_blocking=True)

    times, t_plan, t_pack = [], [], []
    for i in range(steps + 3):
        t0 = time.perf_counter()
        plan_and_pack()
        step()
        st.synchronize()
        if i >= 3:
            times.append(time.perf_counter() - t0)
    assert int(counts[0]) == plan.num_items and np.array_equal(h_items[: plan.num_items], plan.items_host)
    for _ in range(20):  # the host calls alone
        t0 = time.perf_counter()
        L.plan_shared_host(*plan_args, out=(h_items, h_si, counts))
        t1 = time.perf_counter()
        L.pack_block_words_host(p, len(w.doc_len), w.seg_indptr, w.seg_doc, w.seg_len, w.seq_pos0,
                                w.doc_block_indptr, w.doc_blocks, out=(h_words, h_lens))
        t_plan.append(t1 - t0)
        t_pack.append(time.perf_counter() - t1)
    static = []
    for i in range(steps + 3):  # plan and words kept: device time of copies + decode
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(st)
        step()
        b.record(st)
        b.synchronize()
        if i >= 3:
            static.append(a.elapsed_time(b) * 1e-3)
    h2d = total
    d2h = hout.numel() * hout.element_size()
    mean = statistics.mean(times)
    return {"value": nbytes["kv_logical"] / mean / 1e9, "unit": "GB/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": 1e3 * mean,
            "includes": "host planner + host packer into pinned staging, one H2D copy, decode, D2H of the output, "
                        "stream sync (host clock)",
            "plan_ms": 1e3 * statistics.median(t_plan), "pack_ms": 1e3 * statistics.median(t_pack),
            "plan_kept": {"value": nbytes["kv_logical"] / statistics.mean(static) / 1e9,
                          "ms_per_step": 1e3 * statistics.mean(static)}}


def measure_extras(args, d, w, flush, hbm, tf_burst, tf_sust):
    import torch
    from paged_kv_cache_57_gb300 import lazy_attn as L
    from paged_kv_cache_57_gb300 import workloads as W
    out = {}
    keep = {"workloads": {"llama8b_decode": w}}  # workloads built here, reused by the CPU legs
    n = max(20, min(args.steps, 200))
    nb8 = decode_bytes(w)

    def ab(dd, path):
        """Interleaved A/B: lazy rotation vs the same kernel with rotation compiled out
        (same pool and block table). Returns (median lazy s, median control s)."""
        t1, t0 = [], []
        for _ in range(4):
            t1 += time_steps(lambda: run_decode(dd, lazy=True, path=path), n // 4, 2, flush)
            t0 += time_steps(lambda: run_decode(dd, lazy=False, path=path), n // 4, 2, flush)
        dd["p"].lazy = 1
        return statistics.median(t1), statistics.median(t0)

    sh1, sh0 = ab(d, "shared")
    sq1, sq0 = ab(d, "seq")
    out["lazy_overhead_pct"] = {"decode": 100.0 * (sh1 / sh0 - 1.0), "decode_ms_lazy": 1e3 * sh1,
                                "decode_ms_prerotated": 1e3 * sh0,
                                "decode_per_sequence_path": 100.0 * (sq1 / sq0 - 1.0),
                                "pages_h100_context": {"decode_latency": 0.13, "prefill_flops_m128": 0.59}}
    # ALiBi on both decode paths: the same pool, plan and queries, block words in the
    # key-position form, a zero-rate table and the usual slopes, against the rotating
    # decode just timed.
    try:
        pa = L.make_params(num_seqs=w.num_seqs, num_q_heads=w.num_q_heads, num_kv_heads=w.num_kv_heads,
                           head_dim=w.head_dim, num_pool_blocks=w.num_pool_blocks,
                           max_blocks_per_seq=d["p"].max_blocks_per_seq, dtype=w.dtype, rope_theta=w.rope_theta,
                           key_positions=True)
        c = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()
        wa, _ = L.pack_block_words(pa, len(w.doc_len), c(w.seg_indptr), c(w.seg_doc), c(w.seg_len),
                                   c(w.seq_pos0), c(w.doc_block_indptr), c(w.doc_blocks))
        ra = L.rope_table_init(pa, freqs=np.zeros(w.head_dim // 2))
        sl = torch.from_numpy(L.alibi_slopes(w.num_q_heads)).cuda()
        ta = statistics.median(time_steps(lambda: L.decode_shared(
            pa, d["q"], d["k"], d["v"], wa, d["q_pos"], ra, d["plan"], out=d["out"], workspace=d["ws_sh"],
            alibi_slopes=sl), n, 3, flush))
        tq = statistics.median(time_steps(lambda: L.decode(
            pa, d["q"], d["k"], d["v"], wa, d["seq_lens"], d["q_pos"], ra, out=d["out"], workspace=d["ws"],
            alibi_slopes=sl), n, 3, flush))
        out["alibi_decode"] = {"shared_ms": 1e3 * ta, "shared_vs_rope_pct": 100.0 * (ta / sh1 - 1.0),
                               "per_sequence_ms": 1e3 * tq, "per_sequence_vs_rope_pct": 100.0 * (tq / sq1 - 1.0),
                               "kv_gbs_unique_shared": nb8["unique"] / ta / 1e9}
        del wa, ra, sl
    except L.LazyAttnError as e:
        out["alibi_decode"] = {"unavailable": str(e)}
    # The per-sequence path (lazy_attn_decode) on the same workload, for comparison.
    out["decode_per_sequence_path"] = {"ms_median": 1e3 * sq1, "kv_gbs_logical": nb8["kv_logical"] / sq1 / 1e9,
                                       "kv_gbs_unique": nb8["unique"] / sq1 / 1e9,
                                       "hbm_frac_unique_of_measured": nb8["unique"] / sq1 / 1e9 / hbm}
    # Eager-materialised baseline: per-sequence copies with K at absolute positions
    # (lazy_attn_materialize), then the decode kernel's control path on the copies.
    try:
        k_e, v_e, w_e = L.materialize(d["p"], d["k"], d["v"], d["words"], d["seq_lens"], d["rope"])
        tm = statistics.median(time_steps(lambda: L.materialize(d["p"], d["k"], d["v"], d["words"], d["seq_lens"],
                                                                d["rope"]), max(10, n // 4), 3, flush))
        de = dict(d, k=k_e, v=v_e, words=w_e)
        de["p"] = L.make_params(num_seqs=w.num_seqs, num_q_heads=w.num_q_heads, num_kv_heads=w.num_kv_heads,
                                head_dim=w.head_dim, num_pool_blocks=int(k_e.shape[0]),
                                max_blocks_per_seq=d["p"].max_blocks_per_seq, dtype=w.dtype, rope_theta=w.rope_theta,
                                lazy=False)
        te = statistics.median(time_steps(lambda: run_decode(de, path="seq"), n, 3, flush))
        copies = 2 * k_e.numel() * k_e.element_size()
        out["eager_materialised"] = {
            "materialise_ms": 1e3 * tm, "decode_ms_on_copies": 1e3 * te, "lazy_decode_ms": 1e3 * sh1,
            "copies_gb": copies / 1e9, "lazy_unique_kv_gb": W.kv_bytes_unique(w) / 1e9,
            "lazy_decode_speedup_vs_eager": te / sh1,
            "lazy_vs_eager_decode_overhead_pct": 100.0 * (sh1 / te - 1.0)}
        del k_e, v_e, w_e, de
    except L.LazyAttnError as e:
        out["eager_materialised"] = {"unavailable": str(e)}
    # No-sharing control: logical bytes = unique bytes = DRAM bytes.
    wc = W.FULL["llama8b_decode_noshare"]()
    dc = build_device(wc)
    bc = decode_bytes(wc)
    ctl = {"workload": "llama8b_decode_noshare"}
    for path in ("shared", "seq"):
        tc = statistics.median(time_steps(lambda: run_decode(dc, path=path), n, 3, flush))
        gbs = bc["unique"] / tc / 1e9
        key = "" if path == "shared" else "per_sequence_"
        ctl.update({key + "gbs": gbs, key + "frac_of_measured": gbs / hbm, key + "frac_of_8tbs": gbs / 8000.0,
                    key + "ms_median": 1e3 * tc})
    out["noshare_control"] = ctl
    # FP8 KV (e4m3 codes, per-tensor scales) on both decode paths, the headline and
    # the no-sharing workloads, against the bf16 pools on the same path.
    fp8 = {}
    for tag, ww, dd in (("llama8b_decode", w, d), ("llama8b_decode_noshare", wc, dc)):
        k8, v8, ks, vs = W.fp8_pools(ww)
        k8, v8 = k8.cuda(), v8.cuda()
        p8 = L.make_params(num_seqs=ww.num_seqs, num_q_heads=ww.num_q_heads, num_kv_heads=ww.num_kv_heads,
                           head_dim=ww.head_dim, num_pool_blocks=ww.num_pool_blocks,
                           max_blocks_per_seq=dd["p"].max_blocks_per_seq, dtype=ww.dtype, rope_theta=ww.rope_theta,
                           kv_dtype="fp8_e4m3", k_scale=ks, v_scale=vs)
        items8, si8 = L.plan_shared_host(p8, len(ww.doc_len), ww.seg_indptr, ww.seg_doc, ww.seg_len,
                                         ww.doc_block_indptr, ww.doc_blocks)
        plan8 = L.SharedPlan(items8, si8)
        ws8 = torch.empty(max(1, L.decode_shared_workspace_bytes(p8, plan8.num_slots)), dtype=torch.uint8,
                          device="cuda")
        ub = decode_bytes(ww)["unique"]
        row = {"kv_bytes_ratio": 0.5}
        for path in ("shared", "seq"):
            if path == "shared":
                f8 = lambda: L.decode_shared(p8, dd["q"], k8, v8, dd["words"], dd["q_pos"], dd["rope"], plan8,
                                             out=dd["out"], workspace=ws8)
            else:
                f8 = lambda: L.decode(p8, dd["q"], k8, v8, dd["words"], dd["seq_lens"], dd["q_pos"], dd["rope"],
                                      out=dd["out"], workspace=dd["ws"])
            t8 = statistics.median(time_steps(f8, n, 3, flush))
            t16 = statistics.median(time_steps(lambda: run_decode(dd, path=path), n, 3, flush))
            key = "shared_" if path == "shared" else "per_sequence_"
            row.update({key + "fp8_ms": 1e3 * t8, key + "bf16_ms": 1e3 * t16,
                        key + "fp8_unique_gbs": ub / 2 / t8 / 1e9,
                        key + "fp8_frac_of_measured": ub / 2 / t8 / 1e9 / hbm})
        fp8[tag] = row
        del k8, v8, ws8
    out["fp8_kv_decode"] = fp8
    del dc
    # Prefill (Llama-3.1-8B-shaped, 8 x (6 x 1024 docs + 256-token chunk)).
    try:
        wp = W.FULL["llama8b_prefill"]()
        dp = build_device(wp)
        fl = prefill_flops(wp)
        tp = time_steps(lambda: run_prefill(dp, lazy=True), n, 3, flush)
        tp0 = time_steps(lambda: run_prefill(dp, lazy=False), n, 3, flush)
        tfl = fl / statistics.median(tp) / 1e12
        out["prefill"] = {"workload": "llama8b_prefill", "tflops": tfl, "frac_of_burst": tfl / tf_burst,
                          "frac_of_sustained_context": tfl / tf_sust, "gflop_per_step": fl / 1e9,
                          "ms_median": 1e3 * statistics.median(tp),
                          "lazy_overhead_pct": 100.0 * (statistics.median(tp) / statistics.median(tp0) - 1.0),
                          "prerotated_control_ms": 1e3 * statistics.median(tp0)}
        # ALiBi on the same shapes: key-position words, a zero-rate table, the usual slopes.
        pa = L.make_params(num_seqs=wp.num_seqs, num_q_heads=wp.num_q_heads, num_kv_heads=wp.num_kv_heads,
                           head_dim=wp.head_dim, num_pool_blocks=wp.num_pool_blocks,
                           max_blocks_per_seq=dp["p"].max_blocks_per_seq, dtype=wp.dtype, rope_theta=wp.rope_theta,
                           key_positions=True)
        c = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()
        wa, sla = L.pack_block_words(pa, len(wp.doc_len), c(wp.seg_indptr), c(wp.seg_doc), c(wp.seg_len),
                                     c(wp.seq_pos0), c(wp.doc_block_indptr), c(wp.doc_blocks))
        ra = L.rope_table_init(pa, freqs=np.zeros(wp.head_dim // 2))
        sl = torch.from_numpy(L.alibi_slopes(wp.num_q_heads)).cuda()
        ta = statistics.median(time_steps(lambda: L.prefill(
            pa, dp["q"], dp["cu"], dp["q_start"], dp["max_q"], dp["k"], dp["v"], wa, sla, ra, out=dp["out"],
            workspace=dp["ws_pf"], alibi_slopes=sl), n, 3, flush))
        out["prefill"].update({"alibi_ms": 1e3 * ta, "alibi_tflops": fl / ta / 1e12,
                               "alibi_vs_rope_pct": 100.0 * (ta / statistics.median(tp) - 1.0)})
        del wa, sla, ra, sl
    except L.LazyAttnError as e:
        out["prefill"] = {"unavailable": str(e)}
    keep["workloads"]["llama8b_prefill"] = wp
    del dp
    # Llama-3.1-70B-shaped decode: 32 x 16 x 1024 Zipf(1.0) of 512, pool capped at 1 GiB.
    w4 = W.FULL["llama70b_decode"]()
    d4 = build_device(w4)
    b4 = decode_bytes(w4)
    s41, s40 = ab(d4, "shared")
    q41, _ = ab(d4, "seq")
    keep["workloads"]["llama70b_decode"] = w4
    out["llama70b_decode"] = {"kv_gbs_logical": b4["kv_logical"] / s41 / 1e9,
                              "kv_gbs_unique": b4["unique"] / s41 / 1e9,
                              "hbm_frac_unique_of_measured": b4["unique"] / s41 / 1e9 / hbm,
                              "tokens_per_s": w4.num_seqs / s41, "ms_median": 1e3 * s41,
                              "lazy_overhead_pct": 100.0 * (s41 / s40 - 1.0),
                              "per_sequence_path_ms": 1e3 * q41}
    del d4
    # Mixed continuous batch, MQA 32/1: 48 decode sequences + 4 prefill chunks of 512, one
    # shared pool, both calls on one stream and timed as one step.
    wd, wp = W.mixed_mqa()
    keep["workloads"]["mixed_mqa_decode"], keep["workloads"]["mixed_mqa_prefill"] = wd, wp
    dd = build_device(wd)
    dp5 = build_device(wp, k_pool=None)
    dp5["k"], dp5["v"] = dd["k"], dd["v"]  # the two halves index the same physical pool

    def mixed_step():
        run_decode(dd, lazy=True)
        run_prefill(dp5, lazy=True)
    t5 = time_steps(mixed_step, max(10, n // 2), 3, flush)
    td = time_steps(lambda: run_decode(dd, lazy=True), max(10, n // 2), 3, flush)
    tp = time_steps(lambda: run_prefill(dp5, lazy=True), max(10, n // 2), 3, flush)
    # The same step as one launch (lazy_attn_mixed): decode items and prefill tiles in
    # the prefill kernel's persistent pipeline.
    ws_mix = torch.empty(L.mixed_workspace_bytes(dd["p"], dp5["p"], dd["plan"].num_slots), dtype=torch.uint8,
                         device="cuda")
    tf = time_steps(lambda: L.mixed(dd["p"], dd["q"], dd["words"], dd["q_pos"], dd["plan"], dp5["p"], dp5["q"],
                                    dp5["cu"], dp5["q_start"], dp5["max_q"], dp5["words"], dp5["seq_lens"], dd["k"],
                                    dd["v"], dd["rope"], out_dec=dd["out"], out_pf=dp5["out"], workspace=ws_mix),
                    max(10, n // 2), 3, flush)
    del ws_mix
    b5 = decode_bytes(wd)
    f5 = prefill_flops(wp)
    out["mixed_mqa"] = {"step_ms": 1e3 * statistics.median(t5),
                        "one_launch_step_ms": 1e3 * statistics.median(tf),
                        "decode_ms": 1e3 * statistics.median(td), "prefill_ms": 1e3 * statistics.median(tp),
                        "decode_kv_gbs_logical": b5["kv_logical"] / statistics.median(td) / 1e9,
                        "decode_kv_gbs_unique": b5["unique"] / statistics.median(td) / 1e9,
                        "prefill_tflops": f5 / statistics.median(tp) / 1e12,
                        "decode_tokens": int(wd.tokens_per_seq().sum()), "prefill_gflop": f5 / 1e9}
    # Cache-policy replay (host C++ in the same library): block hit rate of the
    # position-agnostic, position-aware and prefix policies on a RAG-shaped Zipf trace,
    # under 1 GiB of Llama-3.1-8B KV (512 blocks) and with an unbounded pool.
    from paged_kv_cache_57_gb300 import cache as CM
    cp = {"trace": "3000 requests x 5 of 500 docs (128-512 tokens), 64-token prompt, 4 in flight"}
    for s in (0.8, 1.2):
        reqs, pos0 = W.cache_trace(num_requests=3000, pool_docs=500, docs_per_request=5, zipf_s=s,
                                   doc_tokens=(128, 512), prompt_tokens=64, seed=23)
        for budget, tag in ((512, "1gib"), (1 << 30, "unbounded")):
            cp[f"zipf{s}_{tag}"] = {p: round(CM.simulate(p, budget, reqs, pos0, concurrency=4)["hit_rate"], 4)
                                    for p in ("agnostic", "aware", "prefix")}
    out["cache_policies"] = cp
    return out, keep


if __name__ == "__main__":
    sys.exit(main())
