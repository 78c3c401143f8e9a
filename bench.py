"""Benchmark of the Gated DeltaNet recurrence on GB300.

One step = one gdn_prefill call on the 4096-token prompt workload
(B=1, T=4096, 16 key / 32 value heads, d_k = d_v = 128, bf16 q/k/v, fp32 g,
beta and state, zero initial state), inputs resident in HBM; L2 is flushed
(a buffer of twice the L2 size is written) between timed steps.  The decode
half of the headline metric is measured in the same run on the batched decode
workload (256 sequences, one token each, state updated in place) and on the
batch-1 decode through 30 layers (one CUDA graph of 30 calls per step).

Prints ONE JSON line (rank 0).  Under torchrun every rank runs its own replica
(independent prompts; no collective on the data path) and the time is the max
over ranks: weak scaling.

--impl reference times the fp64 CPU oracle (the only reference this build
has) on the host cores for the same workload and metric.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "GDN tokens/s: prefill T=4K (tensor-pipe %) & decode state HBM GB/s (% peak)"
WORKLOAD = "prefill_t4096"
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                  "sm_max_mhz": 2070.0}
NUM_SMS_GB300 = 152
FP32_LANES_PER_SM = 128

# DRAM traffic per launch (dram__bytes_read.sum + dram__bytes_write.sum) from one
# ncu capture of each kernel (summaries under profiles/), valid only while the
# kernel's device sources (the .cu and the device headers it includes, comments
# stripped) hash to the recorded value.
NCU_TRAFFIC = {
    "chunk_split": {"files": ["chunk_split.cu", "chunk_common.cuh", "tc.cuh", "rows.cuh"],
                    "sha256_16": "4dbd7899e795fe3c",
                    "bytes": (68_258_048 + 62_212_608) + (135_572_224 + 13_334_784),
                    "profile": "profiles/chunk_split_t4096.md"},
    "chunk_coop": {"files": ["chunk_split.cu", "chunk_common.cuh", "tc.cuh", "rows.cuh"],
                   "sha256_16": "4dbd7899e795fe3c", "bytes": 69_837_312 + 99_008_000,
                   "profile": "profiles/chunk_coop_t4096.md"},
    "chunk_coop@prefill_t131072": {
        "files": ["chunk_split.cu", "chunk_common.cuh", "tc.cuh", "rows.cuh"],
        "sha256_16": "4dbd7899e795fe3c", "bytes": 4_049_355_008 + 4_838_642_176,
        "profile": "profiles/chunk_coop_t131072.md"},
    "chunk_split@prefill_varlen10": {
        "files": ["chunk_split.cu", "chunk_common.cuh", "tc.cuh", "rows.cuh"],
        "sha256_16": "4dbd7899e795fe3c",
        "bytes": 12_544 + (4_362_177_024 + 7_522_012_928) + (8_666_622_720 + 2_143_017_984),
        "profile": "profiles/chunk_split_varlen10.md"},
    "chunk_prefill": {"files": ["chunk_prefill.cu", "chunk_common.cuh", "tc.cuh", "rows.cuh"],
                      "sha256_16": "f95c4a11744de65c", "bytes": 68_218_112 + 5_280_768,
                      "profile": "profiles/chunk_prefill_t4096.md"},
    "attn_decode": {"files": ["attn_decode.cu", "tc.cuh", "rows.cuh"],
                    "sha256_16": "485f911bcb6786c8",
                    "bytes": (268_509_696 + 3_135_488) + 1_264_896,
                    "profile": "profiles/attn_decode_b1_l131072.md"},
    "decode_step": {"files": ["decode_step.cu", "rows.cuh", "tc.cuh"],
                    "sha256_16": "52eb19cd391aa574", "bytes": 541_265_152 + 480_637_184,
                    "profile": "profiles/decode_step_b256.md"},
}


def source_hash(files):
    """Hash of the kernel sources with comments and blank lines removed, so that
    documentation edits do not invalidate a capture but any code change does."""
    import hashlib
    import re

    m = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "gated_deltanet_linear_recurrence_gb300", "csrc", f)) as fh:
            text = re.sub(r"/\*.*?\*/", "", fh.read(), flags=re.S)
        for line in text.splitlines():
            line = line.split("//", 1)[0].rstrip()
            if line:
                m.update(line.encode() + b"\n")
    return m.hexdigest()[:16]


def ncu_traffic(kernel):
    """Recorded DRAM bytes per launch, or None if the kernel changed since the capture."""
    rec = NCU_TRAFFIC[kernel]
    return rec["bytes"] if source_hash(rec["files"]) == rec["sha256_16"] else None


def make_flush(torch, dev, l2):
    """L2 flush between timed calls: write a buffer of twice the L2 size, then
    read another one, so that no input of the next call is cached and no dirty
    line of the flush is still waiting to be written back when the call starts."""
    n = max(2 * l2, 256 << 20)
    wbuf = torch.empty(n, dtype=torch.uint8, device=dev)
    rbuf = torch.ones(n // 4, dtype=torch.float32, device=dev)  # summed by one reduction kernel

    def flush():
        wbuf.fill_(1)
        rbuf.sum()

    return flush


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        d["source"] = "measured"
        return d
    d = dict(PEAKS_FALLBACK)
    d["source"] = "fallback"
    return d


# ---------------------------------------------------------------- algorithmic work
def prefill_bytes(T, N, h_k, h_v, d_k, d_v, esize, state_in):
    qk = 2 * T * h_k * d_k * esize
    vo = 2 * T * h_v * d_v * esize
    gb = 2 * T * h_v * 4
    st = N * h_v * d_v * d_k * 4 * (2 if state_in else 1)
    return qk + vo + gb + st


def chunked_flops_per_token(h_k, h_v, d_k, d_v, C=64):
    """Dense tensor-core work of the chunked form per token (2 flop per
    multiply-add): per (chunk, key head) K K^T and Q K^T; per (chunk, value
    head) W, U~ and P U (C x C x d products), W S^T, Q S^T and the state update
    (C x d_k x d_v).  This is the GEMM portion the roofline is stated on; the
    triangular solve is counted apart (solve_flops_per_token)."""
    per_key = 2 * (2 * C * C * d_k)
    per_val = 2 * C * C * d_k + 2 * 2 * C * C * d_v + 3 * (2 * C * d_k * d_v)
    return (h_k * per_key + h_v * per_val) / C


def solve_flops_per_token(h_v, C=64):
    """The 64 x 64 unit-lower-triangular inverse per (chunk, value head):
    C^3 / 3 multiply-adds, mostly on CUDA cores."""
    return h_v * (2 * C ** 3 // 3) / C


def scan_flops_per_token(h_v, d_k, d_v):
    """Row identity per (token, value head): s = S k, p = S q and the rank-1
    update, 3 multiply-adds per state element."""
    return 6 * d_k * d_v * h_v


def decode_bytes(B, h_k, h_v, d_k, d_v, esize):
    state = 2 * B * h_v * d_v * d_k * 4
    return state + 2 * B * h_k * d_k * esize + 2 * B * h_v * d_v * esize + 2 * B * h_v * 4


# ---------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.close()
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax = float(parts[2])
                except ValueError:
                    continue
                for name, flag in zip(names, parts[5:9]):
                    if flag.lower() == "active":
                        reasons.add(name)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- reference arm
def run_reference(args):
    import numpy as np
    import oracle
    from gated_deltanet_linear_recurrence_gb300 import inputs

    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    w = inputs.WORKLOADS[WORKLOAD]
    d = inputs.make_prefill(w["lengths"], w["h_k"], w["h_v"], w["d_k"], w["d_v"], w["dtype"],
                            seed=w["seed"])
    T = sum(w["lengths"])
    threads = oracle.default_threads()

    def step():
        oracle.prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], w["h_k"],
                       w["h_v"], w["d_k"], w["d_v"], state_in=None, threads=threads)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    sec = time.perf_counter() - t0
    value = args.steps * T / sec
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tok/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * sec / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{WORKLOAD} (B=1, T=4096, H_k=16, H_v=32, d_k=d_v=128, bf16 "
                               "inputs widened to fp64, zero initial state)",
                   "global_batch": 1, "seq_len": T, "parallelism": "host threads"},
        "cpu_baseline": {"value": value, "unit": "tok/s", "cores": threads, "kind": "oracle",
                         "sample": "the whole workload each step (all 32 heads, 4096 tokens)"},
        "e2e": {"value": value, "unit": "tok/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def cpu_baseline(d, w, budget_s=12.0):
    """The oracle as it stands, on the host cores, over whole-workload passes
    until about budget_s seconds have elapsed (at least one pass)."""
    import oracle

    threads = oracle.default_threads()
    T = sum(w["lengths"])
    reps, t0 = 0, time.perf_counter()
    while True:
        oracle.prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], w["h_k"],
                       w["h_v"], w["d_k"], w["d_v"], state_in=d["state_in"], threads=threads)
        reps += 1
        if time.perf_counter() - t0 > budget_s or reps >= 8:
            break
    sec = time.perf_counter() - t0
    return {"value": reps * T / sec, "unit": "tok/s", "cores": threads, "kind": "oracle",
            "sample": f"{reps} pass(es) over the whole {WORKLOAD} workload ({sec:.1f} s)"}


# ---------------------------------------------------------------- our arm
def max_over_ranks(x, device):
    """Largest value of x over all ranks (timing: the slowest rank sets the step)."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--algo", default="auto",
                    choices=["auto", "scan", "chunked", "chunked_fused", "chunked_split",
                             "chunked_coop"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-attention", action="store_true")
    ap.add_argument("--tokens", type=int, default=0,
                    help="with --kernel-only prefill: the prompt's length instead of 4096")
    ap.add_argument("--no-long-prefill", action="store_true",
                    help="skip the 128K-token and ten-prompt varlen prefill timings")
    ap.add_argument("--sweep", action="store_true",
                    help="time every prefill form over sequence lengths for the shapes of the "
                         "crossover table and print the timings and thresholds as JSON lines")
    ap.add_argument("--stream", action="store_true",
                    help="time the 128K-token prompt as one call and as streamed pieces "
                         "(gdn_prefill_streamed), with the workspace each needs, as JSON lines")
    ap.add_argument("--kernel-only", choices=["prefill", "prefill_t131072", "prefill_varlen10",
                                              "decode_b256", "attn_b1_l131072",
                                              "attn_b64_l8192"], default=None,
                    help="run only this kernel's workload (warmup + steps launches, no JSON); "
                         "for profiler captures")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    if args.kernel_only:
        return run_kernel_only(args)
    if args.sweep:
        return run_sweep(args)
    if args.stream:
        return run_stream(args)

    import torch
    import torch.distributed as dist
    from gated_deltanet_linear_recurrence_gb300 import (_lib, gdn_decode_step, gdn_prefill,
                                                        gdn_prefill_form,
                                                        gdn_prefill_workspace_size,
                                                        gdn_stream_status, inputs)
    from gated_deltanet_linear_recurrence_gb300.shard import seq_shard

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    lib = _lib.load()
    peaks = load_peaks()

    w = inputs.WORKLOADS[WORKLOAD]
    h_k, h_v, d_k, d_v = w["h_k"], w["h_v"], w["d_k"], w["d_v"]
    # weak scaling: a global batch of one prompt per rank, split by sequences
    # (no exchange between ranks); rank r draws its own prompt's inputs
    lengths_all = list(w["lengths"]) * world
    n0, n1 = seq_shard(inputs.cu_from_lengths(lengths_all), rank, world)
    lengths = lengths_all[n0:n1]
    T = sum(lengths)
    d = inputs.make_prefill(lengths, h_k, h_v, d_k, d_v, w["dtype"], seed=w["seed"] + n0)
    x = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
    o = torch.empty((T, h_v, d_v), dtype=torch.bfloat16, device=dev)
    st = torch.empty((1, h_v, d_v, d_k), dtype=torch.float32, device=dev)
    ws_n = gdn_prefill_workspace_size(1, T, h_k, h_v, d_k, d_v, torch.bfloat16, args.algo)
    ws = torch.empty(max(ws_n, 16), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    # the evaluation the call runs (the library's own routing, queried)
    form = gdn_prefill_form(len(lengths), T, h_k, h_v, d_k, d_v, torch.bfloat16, args.algo,
                            ws_n)
    algo_used = form

    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = make_flush(torch, dev, l2)

    def prefill_once():
        gdn_prefill(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu_seqlens"], state_in=None,
                    state_out=st, o=o, algo=args.algo, workspace=ws, stream=stream)

    for _ in range(args.warmup):
        flush()
        prefill_once()
    torch.cuda.synchronize()
    assert gdn_stream_status(stream) == "GDN_OK"

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    clocks = ClockSampler(local)
    clocks.start()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    for i in range(args.steps):
        flush()
        starts[i].record(stream)
        prefill_once()
        ends[i].record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    total_ms = sum(step_ms)
    if world > 1:
        total_ms = max_over_ranks(total_ms, dev)
    ms_per_step = total_ms / args.steps
    value = world * T * args.steps / (total_ms / 1e3)
    # two kernels: prepare + chain; cooperative: one kernel; either plus the chunk-table
    # kernel for more than one sequence; fused or scan: one kernel
    multi = 1 if len(lengths) > 1 else 0
    launches_per_step = {"chunked_split": 2 + multi, "chunked_coop": 1 + multi}.get(form, 1)

    # roofline of the prefill kernel (one launch per step)
    if algo_used.startswith("chunked"):
        flop = chunked_flops_per_token(h_k, h_v, d_k, d_v) * T
        achieved = flop / (ms_per_step / 1e3) / 1e12
        flop_solve = solve_flops_per_token(h_v) * T
        scope, traffic_key = {
            "chunked_coop": ("the whole gdn_prefill call: one cooperative kernel, prepare slots "
                             "and state passes overlapped (profiles/)", "chunk_coop"),
            "chunked_split": ("the whole gdn_prefill call: chunk_prepare + chunk_chain kernels "
                              "(one algorithm split in two; shares in profiles/)", "chunk_split"),
        }.get(form, ("the fused chunk_prefill kernel", "chunk_prefill"))
        roof = {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s", "frac": achieved / peaks["bf16_tflops"],
                "traffic": ncu_traffic(traffic_key), "scope": scope,
                "peak_source": f"{peaks['source']} bf16 dense (burst)",
                "algorithmic_flop_per_launch": flop,
                "flop_count": "GEMM products only, 5,242,880 flop/token at 16/32 heads of 128",
                "frac_with_solve": (flop + flop_solve) / (ms_per_step / 1e3) / 1e12
                / peaks["bf16_tflops"]}
    else:
        flop = scan_flops_per_token(h_v, d_k, d_v) * T
        achieved = flop / (ms_per_step / 1e3) / 1e12
        fp32_peak = NUM_SMS_GB300 * FP32_LANES_PER_SM * 2 * peaks["sm_max_mhz"] * 1e6 / 1e12
        roof = {"bound": "alu", "achieved": achieved, "peak": fp32_peak, "unit": "TFLOP/s",
                "frac": achieved / fp32_peak, "traffic": None,
                "peak_source": "fp32 FMA: 152 SMs x 128 lanes x 2 flop x max SM clock",
                "algorithmic_flop_per_launch": flop}
    hbm_bytes = prefill_bytes(T, 1, h_k, h_v, d_k, d_v, 2, False)
    roof["hbm_gbs_at_algorithmic_bytes"] = hbm_bytes / (ms_per_step / 1e3) / 1e9

    # the same prefill with the in-kernel q/k L2 normalisation, on raw N(0, 1) q and k
    dq = inputs.make_prefill(lengths, h_k, h_v, d_k, d_v, w["dtype"], seed=w["seed"] + n0 + 1,
                             unit_qk=False)
    xq = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in dq.items()}
    # the same evaluation as the step above (AUTO's workspace holds the cooperative form)
    ws_q_algo = args.algo if args.algo != "scan" else "chunked_split"
    ws_q = torch.empty(max(gdn_prefill_workspace_size(1, T, h_k, h_v, d_k, d_v, torch.bfloat16,
                                                      ws_q_algo), 16),
                       dtype=torch.uint8, device=dev)

    def prefill_qk():
        gdn_prefill(xq["q"], xq["k"], xq["v"], xq["g"], xq["beta"], xq["cu_seqlens"],
                    state_in=None, state_out=st, o=o, algo=args.algo, workspace=ws_q,
                    stream=stream, qk_l2norm=True)

    for _ in range(args.warmup):
        flush()
        prefill_qk()
    qk_ms = []
    for _ in range(args.steps):
        flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        prefill_qk()
        b.record(stream)
        torch.cuda.synchronize()
        qk_ms.append(a.elapsed_time(b))
    qk_variant = {"ms_per_step": statistics.median(qk_ms),
                  "tok_s": T / (statistics.median(qk_ms) / 1e3),
                  "vs_without": ms_per_step / statistics.median(qk_ms)}
    del xq, dq, ws_q

    # e2e: host buffers in, results out, through the C ABI's host-memory entry point
    # (gdn_prefill_host: pieces of the prompt with the copies in, the prefill and
    # the copies out overlapped); timed per step, pieces of 512 / 1024 / 2048 tokens
    from gated_deltanet_linear_recurrence_gb300 import (gdn_prefill_host,
                                                        gdn_prefill_host_workspace_size)
    pin = {k: d[k].pin_memory() for k in ("q", "k", "v", "g", "beta")}
    o_host = torch.empty(o.shape, dtype=o.dtype).pin_memory()
    st_host = torch.empty(st.shape, dtype=st.dtype).pin_memory()
    by_piece = {}
    for piece in (512, 1024, 2048):
        ws_h = torch.empty(gdn_prefill_host_workspace_size(piece, h_k, h_v, d_k, d_v),
                           dtype=torch.uint8, device=dev)

        def e2e_once():
            gdn_prefill_host(pin["q"], pin["k"], pin["v"], pin["g"], pin["beta"], piece,
                             state_out=st_host, o=o_host, workspace=ws_h, stream=stream)

        for _ in range(3):
            e2e_once()
        torch.cuda.synchronize()
        e_ms = []
        for _ in range(args.steps):
            flush()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            e2e_once()
            b.record(stream)
            b.synchronize()
            e_ms.append(a.elapsed_time(b))
        by_piece[piece] = world * T / (statistics.mean(e_ms) / 1e3)
        del ws_h
    best = max(by_piece, key=by_piece.get)
    h2d = sum(pin[k].numel() * pin[k].element_size() for k in pin)
    d2h = o_host.numel() * 2 + st_host.numel() * 4
    e2e = {"value": by_piece[best], "unit": "tok/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
           "path": ("gdn_prefill_host: page-locked host inputs and outputs through the C ABI, "
                    f"pieces of {best} tokens, copies in / prefill / copies out overlapped"),
           "piece_tokens": best, "by_piece_tok_s": by_piece}

    # decode half of the metric
    decode = None
    if not args.no_decode:
        decode = bench_decode(torch, gdn_decode_step, inputs, dev, stream, peaks, args, flush)

    attention = None
    if not args.no_attention:
        attention = bench_attention(torch, inputs, dev, stream, peaks, args, flush)

    long_prefill = {}
    if not args.no_long_prefill:
        for name in ("prefill_t131072", "prefill_varlen10"):
            long_prefill[name] = bench_prefill_workload(torch, inputs, name, dev, stream, peaks,
                                                        args, flush)

    clk = clocks.stop()
    assert gdn_stream_status(stream) == "GDN_OK"

    line = {
        "metric": METRIC, "value": value, "unit": "tok/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{WORKLOAD} (B=1, T=4096, H_k=16, H_v=32, d_k=d_v=128, bf16 "
                               "q/k/v, fp32 g/beta/state, zero initial state)",
                   "global_batch": world, "seq_len": T,
                   "parallelism": (f"{world} ranks, one prompt each (sequence shards, no "
                                   "exchange)") if world > 1 else "single GPU",
                   "algo": algo_used,
                   "l2": ("flushed between timed steps: a 2x L2 buffer written, then another "
                          "read, so no input is cached and no dirty line is pending")},
        "roofline": roof,
        "prefill_qk_l2norm": qk_variant,
        "gpu_launches": launches_per_step * args.steps,
        "e2e": e2e,
        "clocks": clk,
        "decode": decode,
        "attn_decode": attention,
        "prefill_t131072": long_prefill.get("prefill_t131072"),
        "prefill_varlen10": long_prefill.get("prefill_varlen10"),
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(d, w)
    if world > 1:
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


def bench_prefill_workload(torch, inputs, name, dev, stream, peaks, args, flush):
    """AUTO on one of the long prefill workloads (the 128K-token prompt with a
    drawn initial state; the ten packed prompts of 256 ... 128K tokens): ms per
    call and tok/s with inputs resident and L2 flushed before each call, the
    form the library ran, and the roofline of that call (survey flop count,
    measured bf16 peak; DRAM traffic from the matching ncu capture while the
    kernels' sources are unchanged, else null)."""
    from gated_deltanet_linear_recurrence_gb300 import (gdn_prefill, gdn_prefill_form,
                                                        gdn_prefill_workspace_size)
    w = inputs.WORKLOADS[name]
    h_k, h_v, d_k, d_v = w["h_k"], w["h_v"], w["d_k"], w["d_v"]
    d = inputs.make_prefill(w["lengths"], h_k, h_v, d_k, d_v, w["dtype"], seed=w["seed"],
                            state_std=w["state_std"])
    x = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
    del d
    T, N = sum(w["lengths"]), len(w["lengths"])
    o = torch.empty((T, h_v, d_v), dtype=torch.bfloat16, device=dev)
    st = torch.empty((N, h_v, d_v, d_k), dtype=torch.float32, device=dev)
    ws_n = gdn_prefill_workspace_size(N, T, h_k, h_v, d_k, d_v, torch.bfloat16, "auto")
    ws = torch.empty(max(ws_n, 16), dtype=torch.uint8, device=dev)
    form = gdn_prefill_form(N, T, h_k, h_v, d_k, d_v, torch.bfloat16, "auto", ws_n)

    def once():
        gdn_prefill(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu_seqlens"],
                    state_in=x["state_in"], state_out=st, o=o, algo="auto", workspace=ws,
                    stream=stream)

    for _ in range(args.warmup):
        flush()
        once()
    ts = []
    for _ in range(max(args.steps // 2, 5)):
        flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        once()
        b.record(stream)
        b.synchronize()
        ts.append(a.elapsed_time(b))
    ms = statistics.median(ts)
    flop = chunked_flops_per_token(h_k, h_v, d_k, d_v) * T
    tflops = flop / (ms / 1e3) / 1e12
    nbytes = prefill_bytes(T, N, h_k, h_v, d_k, d_v, 2, x["state_in"] is not None)
    traffic_key = {"chunked_coop": "chunk_coop", "chunked_split": "chunk_split"}.get(form)
    rec = NCU_TRAFFIC.get(f"{traffic_key}@{name}") if traffic_key else None
    traffic = None
    if rec and source_hash(rec["files"]) == rec["sha256_16"]:
        traffic = rec["bytes"]
    out = {"form": form, "tokens": T, "sequences": N, "ms_per_call": ms,
           "tok_s": T / (ms / 1e3), "tok_s_per_30_layers": T / (ms / 1e3) / 30,
           "workspace_bytes": ws_n,
           "roofline": {"bound": "tensor", "achieved": tflops, "peak": peaks["bf16_tflops"],
                        "unit": "TFLOP/s", "frac": tflops / peaks["bf16_tflops"],
                        "traffic": traffic, "algorithmic_flop_per_launch": flop,
                        "algorithmic_bytes_per_launch": nbytes,
                        "hbm_gbs_at_algorithmic_bytes": nbytes / (ms / 1e3) / 1e9,
                        "peak_source": f"{peaks['source']} bf16 dense (burst)"},
           "l2": "flushed before each call (inputs are larger than L2 as well)"}
    del x, o, st, ws
    torch.cuda.empty_cache()
    return out


def bench_decode(torch, gdn_decode_step, inputs, dev, stream, peaks, args, flush):
    out = {}
    # batched decode: 256 sequences; 1 GiB of state, far above L2
    w = inputs.WORKLOADS["decode_b256"]
    dd = inputs.make_decode(w["batch"], w["h_k"], w["h_v"], w["d_k"], w["d_v"], w["dtype"],
                            seed=w["seed"])
    y = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in dd.items()}
    o = torch.empty_like(y["v"])

    def step():
        gdn_decode_step(y["q"], y["k"], y["v"], y["g"], y["beta"], y["state"], o=o, stream=stream)

    for _ in range(args.warmup):
        step()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    torch.cuda.synchronize()
    for a, b in evs:
        a.record(stream)
        step()
        b.record(stream)
    torch.cuda.synchronize()
    ms = statistics.median([a.elapsed_time(b) for a, b in evs])
    nbytes = decode_bytes(w["batch"], w["h_k"], w["h_v"], w["d_k"], w["d_v"], 2)
    gbs = nbytes / (ms / 1e3) / 1e9
    out["decode_b256"] = {"us_per_step": ms * 1e3, "bytes_per_step": nbytes, "gbs": gbs,
                          "frac_of_measured_hbm": gbs / peaks["hbm_gbs"],
                          "frac_of_8tbs_nominal": gbs / 8000.0,
                          "tok_s": w["batch"] / (ms / 1e3), "l2": "state 1 GiB > L2"}
    out["roofline"] = {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                       "frac": gbs / peaks["hbm_gbs"], "traffic": ncu_traffic("decode_step"),
                       "peak_source": f"{peaks['source']} copy bandwidth"}

    # the same step with the in-kernel q/k L2 normalisation
    def qstep():
        gdn_decode_step(y["q"], y["k"], y["v"], y["g"], y["beta"], y["state"], o=o, stream=stream,
                        qk_l2norm=True)

    for _ in range(args.warmup):
        qstep()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    torch.cuda.synchronize()
    for a, b in evs:
        a.record(stream)
        qstep()
        b.record(stream)
    torch.cuda.synchronize()
    qms = statistics.median([a.elapsed_time(b) for a, b in evs])
    out["decode_b256_qk_l2norm"] = {"us_per_step": qms * 1e3,
                                    "gbs": nbytes / (qms / 1e3) / 1e9,
                                    "frac_of_measured_hbm": nbytes / (qms / 1e3) / 1e9 /
                                    peaks["hbm_gbs"]}

    # the same step with the output RMS normalisation fused in (gdn_decode_step_rmsnorm)
    from gated_deltanet_linear_recurrence_gb300 import gdn_decode_step_rmsnorm
    wn = torch.ones(w["d_v"], dtype=torch.float32, device=dev)

    def nstep():
        gdn_decode_step_rmsnorm(y["q"], y["k"], y["v"], y["g"], y["beta"], y["state"],
                                norm_weight=wn, o=o, stream=stream)

    for _ in range(args.warmup):
        nstep()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    torch.cuda.synchronize()
    for a, b in evs:
        a.record(stream)
        nstep()
        b.record(stream)
    torch.cuda.synchronize()
    nms = statistics.median([a.elapsed_time(b) for a, b in evs])
    out["decode_b256_out_rmsnorm"] = {"us_per_step": nms * 1e3,
                                      "gbs": nbytes / (nms / 1e3) / 1e9,
                                      "frac_of_measured_hbm": nbytes / (nms / 1e3) / 1e9 /
                                      peaks["hbm_gbs"]}

    # the same 256 sequences advanced by 4 tokens in one launch (gdn_decode_multi),
    # without and with the per-token state snapshots
    from gated_deltanet_linear_recurrence_gb300 import gdn_decode_multi
    n_tok, B = 4, w["batch"]
    dm = inputs.make_prefill([n_tok] * B, w["h_k"], w["h_v"], w["d_k"], w["d_v"], w["dtype"],
                             seed=w["seed"] + 7)
    mm = {k: dm[k].to(dev).reshape(B, n_tok, *dm[k].shape[1:]).contiguous()
          for k in ("q", "k", "v", "g", "beta")}
    om = torch.empty((B, n_tok, w["h_v"], w["d_v"]), dtype=torch.bfloat16, device=dev)
    snap = torch.empty((B, n_tok, w["h_v"], w["d_v"], w["d_k"]), dtype=torch.float32, device=dev)
    per_token = nbytes - 2 * y["state"].numel() * 4
    for with_snap in (False, True):
        def mstep():
            gdn_decode_multi(mm["q"], mm["k"], mm["v"], mm["g"], mm["beta"], y["state"], o=om,
                             snapshots=snap if with_snap else False, stream=stream)

        for _ in range(args.warmup):
            mstep()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        torch.cuda.synchronize()
        for a, b in evs:
            a.record(stream)
            mstep()
            b.record(stream)
        torch.cuda.synchronize()
        mms = statistics.median([a.elapsed_time(b) for a, b in evs])
        mbytes = 2 * y["state"].numel() * 4 + n_tok * per_token
        if with_snap:
            mbytes += snap.numel() * 4
        key = "decode_multi_b256_n4" + ("_snapshots" if with_snap else "")
        out[key] = {"us_per_call": mms * 1e3, "tokens_per_call": B * n_tok,
                    "tok_s": B * n_tok / (mms / 1e3), "bytes_per_call": mbytes,
                    "gbs": mbytes / (mms / 1e3) / 1e9,
                    "frac_of_measured_hbm": mbytes / (mms / 1e3) / 1e9 / peaks["hbm_gbs"],
                    "vs_4_single_steps": 4 * ms / mms}
    del y, o, dd, mm, om, snap, dm

    # batch-1 decode through 30 layers: one CUDA graph of 30 calls per step
    w = inputs.WORKLOADS["decode_b1_x30layers"]
    layers = []
    for layer in range(w["layers"]):
        dd = inputs.make_decode(1, w["h_k"], w["h_v"], w["d_k"], w["d_v"], w["dtype"],
                                seed=w["seed"] * 100 + layer)
        layers.append({k: (v.to(dev) if isinstance(v, torch.Tensor) else v)
                       for k, v in dd.items()})
    outs = [torch.empty_like(L["v"]) for L in layers]
    side = torch.cuda.Stream(dev)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        for L, ob in zip(layers, outs):  # warm the launch path outside capture
            gdn_decode_step(L["q"], L["k"], L["v"], L["g"], L["beta"], L["state"], o=ob,
                            stream=side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        for L, ob in zip(layers, outs):
            gdn_decode_step(L["q"], L["k"], L["v"], L["g"], L["beta"], L["state"], o=ob,
                            stream=side)
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()
    ms_list = []
    for _ in range(args.steps):
        flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        graph.replay()
        b.record(stream)
        torch.cuda.synchronize()
        ms_list.append(a.elapsed_time(b))
    ms = statistics.median(ms_list)
    nbytes = w["layers"] * decode_bytes(1, w["h_k"], w["h_v"], w["d_k"], w["d_v"], 2)
    out["decode_b1_x30layers"] = {"us_per_step": ms * 1e3, "us_per_layer": ms * 1e3 / 30,
                                  "bytes_per_step": nbytes,
                                  "gbs": nbytes / (ms / 1e3) / 1e9,
                                  "tok_s": 1 / (ms / 1e3),
                                  "l2": "flushed between steps; 30 calls in one CUDA graph"}
    return out


def attn_bytes(lengths, h_q, h_kv, head_dim):
    """Algorithmic bytes of one decode-attention call: every cached K and V row of
    every sequence once (bf16), q in and o out, and the lengths."""
    cache = sum(lengths) * h_kv * head_dim * 2 * 2
    return cache + 2 * len(lengths) * h_q * head_dim * 2 + 4 * len(lengths)


def attn_device_inputs(torch, inputs, dev, name):
    w = inputs.WORKLOADS[name]
    x = inputs.make_attention(w["batch"], w["h_q"], w["h_kv"], w["head_dim"], w["capacity"],
                              w["lengths"], w["dtype"], seed=w["seed"], poison_tail=False)
    return w, {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in x.items()}


def bench_attention(torch, inputs, dev, stream, peaks, args, flush):
    """Decode attention of the full-attention layers (gdn_attn_decode): the
    library's layout choice, and the general layout beside it, timed with CUDA
    events on the launching stream, L2 flushed before each call."""
    from gated_deltanet_linear_recurrence_gb300 import (gdn_attn_decode,
                                                        gdn_attn_decode_block_keys)

    def timed(fn):
        for _ in range(args.warmup):
            fn()
        ts = []
        for _ in range(max(args.steps, 10)):
            flush()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            b.synchronize()
            ts.append(a.elapsed_time(b))
        return statistics.median(ts)

    def measure(x, layout, lengths):
        B, h_q, D = x["q"].shape
        h_kv, cap = x["k_cache"].shape[1], x["k_cache"].shape[2]
        o = torch.empty_like(x["q"])
        ms = timed(lambda: gdn_attn_decode(x["q"], x["k_cache"], x["v_cache"], x["cache_len"],
                                           o=o, layout=layout, stream=stream))
        nbytes = attn_bytes(lengths, h_q, h_kv, D)
        bk = gdn_attn_decode_block_keys(B, h_q, h_kv, D, cap, layout)
        gbs = nbytes / (ms / 1e3) / 1e9
        return {"us": ms * 1e3, "bytes": nbytes, "gbs": gbs,
                "frac_of_measured_hbm": gbs / peaks["hbm_gbs"], "layout": layout,
                "block_keys": bk, "blocks_per_kv_head": -(-cap // bk)}

    out = {}
    w, x = attn_device_inputs(torch, inputs, dev, "attn_b1_l131072")
    head = measure(x, "auto", w["lengths"])
    out["attn_b1_l131072"] = head
    out["roofline"] = {"bound": "hbm", "achieved": head["gbs"], "peak": peaks["hbm_gbs"],
                       "unit": "GB/s", "frac": head["gbs"] / peaks["hbm_gbs"],
                       "traffic": ncu_traffic("attn_decode"),
                       "scope": "the whole gdn_attn_decode call (attention kernel + combine)",
                       "peak_source": f"{peaks['source']} copy bandwidth",
                       "algorithmic_bytes_per_call": head["bytes"]}
    # the pages' layout question at batch 1: general vs fixed blocks over contexts
    sweep = []
    for L in (4096, 32768, 131072):
        xs = x if L == w["capacity"] else {
            "q": x["q"], "k_cache": x["k_cache"][:, :, :L].contiguous(),
            "v_cache": x["v_cache"][:, :, :L].contiguous(),
            "cache_len": torch.full_like(x["cache_len"], L)}
        gen = measure(xs, "general", [L])
        fix = measure(xs, "fixed_block", [L])
        sweep.append({"keys": L, "general_us": gen["us"], "fixed_block_us": fix["us"],
                      "fixed_block_keys": fix["block_keys"],
                      "fixed_vs_general": gen["us"] / fix["us"]})
        del xs
    out["layouts_b1"] = sweep
    del x
    w, x = attn_device_inputs(torch, inputs, dev, "attn_b64_l8192")
    out["attn_b64_l8192"] = measure(x, "auto", w["lengths"])
    del x
    return out


def sweep_inputs(torch, dev, N, L, h_k, h_v, d_k, d_v, seed):
    """Device-drawn inputs of the workloads' distributions for timing only (unit q,
    k; v ~ N(0, 1); beta = sigmoid(N(0, 1)); g = -softplus(N(0, 1)); zero state):
    nothing here is compared with the oracle."""
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    T = N * L

    def unit(n_heads, d):
        x = torch.randn((T, n_heads, d), generator=g, device=dev)
        return (x / x.norm(dim=-1, keepdim=True)).to(torch.bfloat16)

    x = {"q": unit(h_k, d_k), "k": unit(h_k, d_k),
         "v": torch.randn((T, h_v, d_v), generator=g, device=dev).to(torch.bfloat16),
         "beta": torch.sigmoid(torch.randn((T, h_v), generator=g, device=dev)),
         "g": -torch.nn.functional.softplus(torch.randn((T, h_v), generator=g, device=dev)),
         "cu_seqlens": torch.arange(0, T + 1, L, dtype=torch.int32, device=dev)}
    return x


SWEEP_LENGTHS = (8, 16, 32, 64, 128, 256, 512, 1024, 2048, 4096, 8192)
SWEEP_MAX_TOKENS = 65536


def sweep_thresholds(rows, forms):
    """Per shape, from rows {L: {form: us}}: the smallest swept L from which the
    faster of each pair stays faster at every longer L."""
    Ls = sorted(rows)

    def from_where(better, worse):
        start = None
        for L in Ls:
            r = rows[L]
            if better not in r or worse not in r:
                continue
            if r[better] < r[worse]:
                if start is None:
                    start = L
            else:
                start = None
        return start

    chunked = [f for f in ("chunked_fused", "chunked_split") if f in forms]
    best = {L: min(rows[L][f] for f in chunked if f in rows[L]) for L in Ls
            if any(f in rows[L] for f in chunked)}
    scan_below = None
    for L in Ls:
        if L not in best or "scan" not in rows[L]:
            continue
        if best[L] < rows[L]["scan"]:
            if scan_below is None:
                scan_below = L
        else:
            scan_below = None
    split_from = from_where("chunked_split", "chunked_fused") if "chunked_fused" in forms else 0
    coop_from = from_where("chunked_coop", "chunked_split") if "chunked_coop" in forms else None
    return {"scan_below": scan_below, "split_from_avg": split_from, "coop_from_avg": coop_from}


def run_sweep(args):
    """Every prefill form timed over sequence lengths for each shape of the
    crossover table (d_k 64 / 128, d_v 32 / 64 / 128, 4 / 32 value heads with two
    per key head, 1 / 4 / 16 sequences of equal length), L2 flushed before each
    call; prints one JSON line per (shape, length) and one per shape with the
    thresholds the table takes."""
    import torch
    from gated_deltanet_linear_recurrence_gb300 import (_lib, gdn_prefill, gdn_prefill_workspace_size,
                                                        gdn_stream_status)

    dev = torch.device("cuda", 0)
    flush = make_flush(torch, dev, torch.cuda.get_device_properties(dev).L2_cache_size)
    lib = _lib.load()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    ws = torch.empty(2 << 30, dtype=torch.uint8, device=dev)
    for d_k in (128, 64):
        for d_v in (128, 64, 32):
            for h_v in (32, 4):
                for N in (1, 4, 16):
                    h_k = h_v // 2
                    forms = ["scan", "chunked_split"]
                    if d_k == 128:
                        forms.insert(1, "chunked_fused")
                    coop_ok = d_v % 64 == 0 and N * h_v * (d_v // 64) <= sms * 2 // 3
                    if coop_ok:
                        forms.append("chunked_coop")
                    rows, scan_on = {}, True
                    for L in SWEEP_LENGTHS:
                        if N * L > SWEEP_MAX_TOKENS:
                            break
                        x = sweep_inputs(torch, dev, N, L, h_k, h_v, d_k, d_v, seed=L + N)
                        T = N * L
                        o = torch.empty((T, h_v, d_v), dtype=torch.bfloat16, device=dev)
                        st = torch.empty((N, h_v, d_v, d_k), dtype=torch.float32, device=dev)
                        res = {}
                        for f in forms:
                            if f == "scan" and not scan_on:
                                continue
                            need = gdn_prefill_workspace_size(N, T, h_k, h_v, d_k, d_v,
                                                              torch.bfloat16, f)
                            assert need <= ws.numel()
                            ts = []
                            for i in range(6):
                                flush()
                                a = torch.cuda.Event(enable_timing=True)
                                b = torch.cuda.Event(enable_timing=True)
                                a.record()
                                gdn_prefill(x["q"], x["k"], x["v"], x["g"], x["beta"],
                                            x["cu_seqlens"], state_out=st, o=o, algo=f,
                                            workspace=ws if need else None)
                                b.record()
                                b.synchronize()
                                if i >= 1:
                                    ts.append(a.elapsed_time(b) * 1e3)
                            assert gdn_stream_status() == "GDN_OK"
                            res[f] = statistics.median(ts)
                        chunk_best = min(v for k, v in res.items() if k != "scan")
                        if "scan" in res and res["scan"] > 4 * chunk_best:
                            scan_on = False  # the scan only falls further behind
                        rows[L] = res
                        print(json.dumps({"d_k": d_k, "d_v": d_v, "h_v": h_v, "N": N, "L": L,
                                          "us": {k: round(v, 2) for k, v in res.items()}}),
                              flush=True)
                        del x, o, st
                    th = sweep_thresholds(rows, forms)
                    print(json.dumps({"shape": {"d_k": d_k, "d_v": d_v, "h_v": h_v, "N": N},
                                      "thresholds": th}), flush=True)


def run_stream(args):
    """The 128K-token prompt: one gdn_prefill call against gdn_prefill_streamed with
    pieces of several sizes (CUDA events, L2 flushed before each call)."""
    import torch
    from gated_deltanet_linear_recurrence_gb300 import (gdn_prefill, gdn_prefill_streamed,
                                                        gdn_prefill_streamed_workspace_size,
                                                        gdn_prefill_workspace_size,
                                                        gdn_stream_status, inputs)

    dev = torch.device("cuda", 0)
    flush = make_flush(torch, dev, torch.cuda.get_device_properties(dev).L2_cache_size)
    w = inputs.WORKLOADS["prefill_t131072"]
    d = inputs.make_prefill(w["lengths"], w["h_k"], w["h_v"], w["d_k"], w["d_v"], w["dtype"],
                            seed=w["seed"], state_std=w["state_std"])
    x = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
    T = sum(w["lengths"])
    o = torch.empty((T, w["h_v"], w["d_v"]), dtype=torch.bfloat16, device=dev)
    st = torch.empty((1, w["h_v"], w["d_v"], w["d_k"]), dtype=torch.float32, device=dev)
    shape = (w["h_k"], w["h_v"], w["d_k"], w["d_v"])
    cases = [("whole", None, gdn_prefill_workspace_size(1, T, *shape, algo="chunked_split")),
             ("whole, cooperative", "coop", gdn_prefill_workspace_size(1, T, *shape,
                                                                        algo="chunked_coop"))]
    for piece in (2048, 8192, 32768):
        cases.append((f"pieces of {piece}", piece,
                      gdn_prefill_streamed_workspace_size(piece, *shape)))
    for name, piece, ws_bytes in cases:
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
        ts = []
        for i in range(args.warmup + 5):
            flush()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            if piece is None or piece == "coop":
                gdn_prefill(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu_seqlens"],
                            state_in=x["state_in"], state_out=st, o=o,
                            algo="chunked_split" if piece is None else "chunked_coop",
                            workspace=ws)
            else:
                gdn_prefill_streamed(x["q"], x["k"], x["v"], x["g"], x["beta"], piece,
                                     state_in=x["state_in"], state_out=st, o=o, workspace=ws)
            b.record()
            torch.cuda.synchronize()
            if i >= args.warmup:
                ts.append(a.elapsed_time(b) * 1e3)
        assert gdn_stream_status() == "GDN_OK"
        us = statistics.median(ts)
        print(json.dumps({"case": name, "tokens": T, "us": us, "tok_s": T / (us / 1e6),
                          "workspace_bytes": ws_bytes}), flush=True)
        del ws


def run_kernel_only(args):
    """warmup + steps launches of one kernel's workload, for profiler captures."""
    import torch
    from gated_deltanet_linear_recurrence_gb300 import (gdn_decode_step, gdn_prefill,
                                                        gdn_prefill_workspace_size,
                                                        gdn_stream_status, inputs)

    dev = torch.device("cuda", 0)
    if args.kernel_only.startswith("attn_"):
        from gated_deltanet_linear_recurrence_gb300 import gdn_attn_decode
        _, x = attn_device_inputs(torch, inputs, dev, args.kernel_only)
        o = torch.empty_like(x["q"])
        for _ in range(args.warmup + args.steps):
            gdn_attn_decode(x["q"], x["k_cache"], x["v_cache"], x["cache_len"], o=o)
    elif args.kernel_only == "decode_b256":
        w = inputs.WORKLOADS["decode_b256"]
        d = inputs.make_decode(w["batch"], w["h_k"], w["h_v"], w["d_k"], w["d_v"], w["dtype"],
                               seed=w["seed"])
        y = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
        o = torch.empty_like(y["v"])
        for _ in range(args.warmup + args.steps):
            gdn_decode_step(y["q"], y["k"], y["v"], y["g"], y["beta"], y["state"], o=o)
    else:
        name = WORKLOAD if args.kernel_only == "prefill" else args.kernel_only
        w = dict(inputs.WORKLOADS[name])
        if args.kernel_only == "prefill" and args.tokens > 0:
            w["lengths"] = [args.tokens]  # the same heads and distributions, another length
        d = inputs.make_prefill(w["lengths"], w["h_k"], w["h_v"], w["d_k"], w["d_v"],
                                w["dtype"], seed=w["seed"], state_std=w["state_std"])
        x = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
        T, N = sum(w["lengths"]), len(w["lengths"])
        n = gdn_prefill_workspace_size(N, T, w["h_k"], w["h_v"], w["d_k"], w["d_v"],
                                       torch.bfloat16, args.algo)
        ws = torch.empty(max(n, 16), dtype=torch.uint8, device=dev)
        for _ in range(args.warmup + args.steps):
            gdn_prefill(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu_seqlens"],
                        state_in=x["state_in"], algo=args.algo, workspace=ws)
    torch.cuda.synchronize()
    assert gdn_stream_status() == "GDN_OK"
    print(f"kernel-only {args.kernel_only}: {args.warmup + args.steps} launches ok", flush=True)


if __name__ == "__main__":
    main()
