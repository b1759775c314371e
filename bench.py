#!/usr/bin/env python3
"""MLA decode benchmark on GB300: one decode step of the DeepSeek-V3-shaped
workload (batch 32, q_len 1, 128 heads, d_c 512 + d_R 64, 4096 cached tokens per
sequence, bf16 paged cache, page size 64, shuffled pages) through the C ABI.

A step = append of the step's new tokens + absorb_q + paged decode + out_proj
(mla_decode_out_proj: with 2-4 KV splits the split merge runs inside the
projection kernel). The latent cache (151 MB) is larger than L2, and L2 is
additionally flushed before every timed step, outside the per-step CUDA-event
window, by reading a 256 MiB buffer.

Prints ONE JSON line (rank 0). --impl reference times the fp64 CPU oracle on a
bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "MLA decode latent-cache GB/s & tokens/s at 1 GB300; % of HBM roofline"
UNIT = "GB/s"
DEFAULT_WORKLOAD = "dsv3_bf16"
# The output projection with W_UV folded into W_O (y = W~ u, d_model 7168, the
# DeepSeek-V3-shaped decode batch of 32): its own line, on request only.
FUSED_WORKLOAD = "dsv3_fused_out"
FUSED_METRIC = "MLA fused output projection (W~ = W_O W_UV) weight-stream GB/s at 1 GB300; % of HBM roofline"
# A whole decode layer from the hidden states (front end, append, absorb,
# paged decode, fused output projection) at the DeepSeek-V3 shape: its own line.
LAYER_WORKLOAD = "dsv3_layer"
LAYER_METRIC = "MLA decode layer (front end + latent attention + output projection) tokens/s at 1 GB300"
# Prefill in the MHA form (K and V expanded from the latent rows, causal
# attention) for one DeepSeek-V3-shaped prompt of 4096 tokens: its own line.
PREFILL_WORKLOAD = "dsv3_prefill"
PREFILL_METRIC = "MLA prefill (MHA form: K/V expansion + causal attention) TFLOP/s at 1 GB300; % of bf16 tensor peak"
PREFILL_T = 4096
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
L2_FLUSH_BYTES = 256 << 20  # read (not written) before every timed step


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    # default: enough timed steps that the clock sampler (200 ms) sees the
    # timed region under load for about a second (decode step ~0.13 ms with
    # its L2 flush); fewer for the longer steps of the other lines
    p.add_argument("--steps", type=int, default=None)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--workload", default=DEFAULT_WORKLOAD)
    # decode workloads: override the workload's split count (0 = the library's policy)
    p.add_argument("--num-splits", type=int, default=None)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=12.0)
    a = p.parse_args()
    if a.steps is None:
        a.steps = {FUSED_WORKLOAD: 4000, LAYER_WORKLOAD: 3000, PREFILL_WORKLOAD: 300}.get(a.workload, 8000)
        if a.impl == "reference":
            a.steps = 20
    return a


def dist_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), \
        int(os.environ.get("LOCAL_RANK", "0"))


def max_over_ranks(value: float, world: int, device) -> float:
    """The largest of every rank's value: the job's time is that of its slowest
    rank. Identity on one rank; otherwise an all-reduce over the process group
    (NCCL on the GPU machine, gloo in the CPU tests)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(world: int, units_per_rank: float, ms_per_step: float) -> float:
    """Whole-job throughput: the units every rank processed per second of the
    slowest rank's step (independent replicas, fixed work per rank)."""
    return world * units_per_rank / (ms_per_step * 1e-3)


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return {"hbm_gbs": FALLBACK_HBM_GBS}, "fallback"


def decode_bytes(w) -> int:
    """Algorithmic bytes of one mla_decode_paged call: every visible cached row
    once per sequence (shared by its q_len queries), the queries, u and lse."""
    rows = sum(int(L) for L in w.seq_lens)
    act = 4 if w.act_dtype == "f32" else 2
    q = w.batch * w.q_len * w.heads * (512 + 64) * act
    out = w.batch * w.q_len * w.heads * (512 * act + 4)
    return rows * w.row_bytes() + q + out


def fused_bytes(n_tokens: int, d_model: int, heads: int) -> int:
    """Algorithmic bytes of one mla_out_proj_fused call (bf16): W~ once, u, y."""
    K = heads * 512
    return 2 * (d_model * K + n_tokens * K + n_tokens * d_model)


def recorded_traffic(kernel_src: str, workload: str, prefix: str = "decode"):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current source of the kernel; else None."""
    prof = os.path.join(ROOT, "profiles", f"{prefix}_{workload}.md")
    try:
        txt = open(prof).read()
        src = open(kernel_src, "rb").read()
    except OSError:
        return None
    h = hashlib.sha256(src).hexdigest()[:16]
    m_h = re.search(r"source_sha256_16:\s*([0-9a-f]{16})", txt)
    m_t = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", txt)
    if m_h and m_t and m_h.group(1) == h:
        return float(m_t.group(1))
    return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""

    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, dev: int):
        self.dev = dev
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                                          "-lms", "200", "-i", str(self.dev)], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 7:
                continue
            try:
                sm.append(float(f[0]))
                mx.append(float(f[1]))
            except ValueError:
                continue
            for n, v in zip(names, f[3:7]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------- CPU oracle

def blas_threads() -> int:
    """Threads numpy's BLAS uses: the *_NUM_THREADS limit if one is set, else
    threadpoolctl's report where it is installed, else the host's cores."""
    for v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        if os.environ.get(v, "").isdigit():
            return int(os.environ[v])
    try:
        from threadpoolctl import threadpool_info
        info = threadpool_info()
        if info:
            return max(i.get("num_threads", 1) for i in info)
    except Exception:
        pass
    return os.cpu_count() or 1


def cpu_oracle_run(w, d, seconds: float, absorbed: bool = False):
    """Time the fp64 oracle on a bounded sample of the workload: whole sequences
    with all heads, in order, until `seconds` of oracle work are done (the last
    sequence may stop part-way through its heads). The non-absorbed form (K and
    V materialised, one head at a time) is the oracle's definition; absorbed=True
    times its absorbed form instead (q_lat = W_UK^T q_nope, scores and latent sum
    over the cached rows, all heads at once). Building the oracle's cache is
    set-up, not timed. Returns (GB/s of cache rows processed, sample
    description, threads, seconds)."""
    import numpy as np
    from oracle import mla_oracle as O
    from oracle.harness import f64, oracle_pool, seq_token_mask

    threads = blas_threads()
    q_nope, q_rope, w_uk, w_uv = f64(d["q_nope"]), f64(d["q_rope"]), f64(d["w_uk"]), f64(d["w_uv"])
    bt = d["block_table"].numpy()
    H = w.heads
    elapsed, done_bytes, seqs, partial = 0.0, 0.0, 0, None
    for b in range(w.batch):
        pool, sc = oracle_pool(w, d, token_mask=seq_token_mask(w, [b]))
        L = int(w.seq_lens[b])
        t0 = time.perf_counter()
        rows = O.gather_rows(pool, sc, bt[b], L, w.page_size, w.cache_dtype)
        if absorbed:
            for j in range(w.q_len):
                T = O.visible_tokens(L, w.q_len, j)
                q_lat = O.absorb_q(q_nope[b, j], w_uk)
                u, _ = O.attend_absorbed(q_lat, q_rope[b, j], rows[:T], O.default_scale())
                O.out_proj(u, w_uv)
            elapsed += time.perf_counter() - t0
            done_bytes += L * w.row_bytes()
            seqs += 1
            if elapsed > seconds:
                break
            continue
        hd = 0
        for h in range(H):
            for j in range(w.q_len):
                T = O.visible_tokens(L, w.q_len, j)
                O.attend_nonabsorbed(q_nope[b, j, h:h + 1], q_rope[b, j, h:h + 1], w_uk[h:h + 1],
                                     w_uv[h:h + 1], rows[:T], O.default_scale())
            hd += 1
            if elapsed + time.perf_counter() - t0 > seconds:
                break
        elapsed += time.perf_counter() - t0
        done_bytes += L * w.row_bytes() * hd / H
        seqs += 1
        if hd < H:
            partial = hd
            break
        if elapsed > seconds:
            break
    last = f"the last with {partial}/{H} heads" if partial else "all heads"
    form = "absorbed fp64 oracle, all heads at once" if absorbed else "non-absorbed fp64 oracle, one head at a time"
    sample = f"{seqs} sequence(s) of {w.name} ({last}); {form}"
    return done_bytes / elapsed / 1e9, sample, threads, elapsed


def cpu_variants(workload: str, seconds: float):
    """The oracle's other reported baselines, each in a child process so that
    its BLAS thread count is set before numpy loads: the non-absorbed form on
    one thread, and the absorbed form on one thread and on every thread."""
    out = []
    for absorbed, one in ((False, True), (True, False), (True, True)):
        env = dict(os.environ)
        if one:
            for v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
                env[v] = "1"
        code = ("import json, sys; sys.path.insert(0, %r); import bench; "
                "from mla_latent_kv_16_gb300 import workloads as W; w = W.preset(%r); d = W.make_inputs(w); "
                "v, s, t, e = bench.cpu_oracle_run(w, d, %r, absorbed=%r); "
                "print(json.dumps({'value': v, 'sample': s, 'threads': t, 'seconds': e}))"
                % (ROOT, workload, seconds, absorbed))
        try:
            r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=600)
            res = json.loads(r.stdout.strip().splitlines()[-1])
        except Exception as e:  # reported, not fatal: the main baseline stands
            out.append({"form": "absorbed" if absorbed else "non-absorbed", "error": str(e)[:200]})
            continue
        out.append({"form": "absorbed" if absorbed else "non-absorbed", "value": round(res["value"], 4),
                    "unit": UNIT, "cores": res["threads"], "sample": res["sample"],
                    "seconds": round(res["seconds"], 2)})
    return out


def fused_setup(w, d_model: int):
    """The fused projection's inputs from the seeded generators: W_O, W_UV, u."""
    import torch
    from mla_latent_kv_16_gb300 import workloads as W
    w_o = W.make_out_weight(w, d_model)
    w_uv = W.make_inputs(w, with_context=False)["w_uv"]
    g = torch.Generator().manual_seed(w.seed * 7 + 100)
    u = torch.randn(w.batch, w.q_len, w.heads, 512, generator=g).to(torch.bfloat16)
    return w_o, w_uv, u


def cpu_fused_run(w, d_model: int, seconds: float):
    """Time the oracle's fused projection on a bounded sample: blocks of 64 rows
    of W~ (folded by the oracle and rounded to bf16 as set-up, not timed) against
    the whole batch, until `seconds` of oracle work are done. Returns (GB/s of
    W~ bytes processed, sample description, threads, seconds)."""
    import numpy as np
    from oracle import mla_oracle as O
    from oracle.harness import f64

    threads = os.cpu_count()
    w_o, w_uv, u = fused_setup(w, d_model)
    wo64, wuv64, u64 = f64(w_o), f64(w_uv), f64(u)
    K = w.heads * 512
    elapsed, rows = 0.0, 0
    for r0 in range(0, d_model, 64):
        wf = O.round_bf16(O.fuse_out_weights(wo64[r0:r0 + 64], wuv64))
        t0 = time.perf_counter()
        O.out_proj_fused(u64, wf)
        elapsed += time.perf_counter() - t0
        rows += wf.shape[0]
        if elapsed > seconds:
            break
    sample = f"{rows} of {d_model} rows of W~ against all {w.batch * w.q_len} tokens; fp64 oracle product"
    return rows * K * 2 / elapsed / 1e9, sample, threads, elapsed


# ----------------------------------------------------------------------------- GPU arm

def run_fused(args):
    """One mla_out_proj_fused call per step (W~ already folded and resident)."""
    import torch
    import torch.distributed as dist

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    from mla_latent_kv_16_gb300 import build as B
    if rank == 0 or world == 1:
        B.build()
    if world > 1:
        dist.barrier()
    from mla_latent_kv_16_gb300 import capi, workloads as W
    capi.load()
    w = W.preset(DEFAULT_WORKLOAD)
    d_model, H, n = W.D_MODEL, w.heads, w.batch * w.q_len
    w_o, w_uv, u_h = fused_setup(w, d_model)
    w_f = capi.mla_fuse_out_weights(w_o.cuda(), w_uv.cuda())
    del w_o, w_uv
    u = u_h.cuda()
    y = torch.empty(w.batch, w.q_len, d_model, dtype=torch.bfloat16, device="cuda")
    need = capi.mla_out_proj_fused_workspace_size(n, d_model, H)
    ws = torch.empty(max(need, 16), dtype=torch.uint8, device="cuda")
    splits = max(1, need // (n * d_model * 4)) if need else 1
    flush = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()
    torch.cuda.synchronize()

    def capture(fn):
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            for _ in range(2):
                fn()
        stream.wait_stream(side)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        return g

    g_call = capture(lambda: capi.mla_out_proj_fused(u, w_f, y, ws))

    def timed(graph, k, clk=None):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(k)]
        if clk is not None:
            clk.start()
            time.sleep(0.3)
        for i in range(k):
            flush.sum()
            evs[i][0].record(stream)
            graph.replay()
            evs[i][1].record(stream)
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in evs]

    for _ in range(args.warmup):
        flush.sum()
        g_call.replay()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clk = ClockSampler(local)
    call_ms = timed(g_call, args.steps, clk)
    clocks = clk.stop()
    tot = max_over_ranks(sum(call_ms), world, "cuda")

    host_u = u_h.pin_memory()
    host_y = torch.empty(y.shape, dtype=y.dtype).pin_memory()

    def e2e():
        u.copy_(host_u, non_blocking=True)
        capi.mla_out_proj_fused(u, w_f, y, ws)
        host_y.copy_(y, non_blocking=True)

    g_e2e = capture(e2e)
    for _ in range(args.warmup):
        flush.sum()
        g_e2e.replay()
    e2e_tot = max_over_ranks(sum(timed(g_e2e, args.steps)), world, "cuda")

    nbytes = fused_bytes(n, d_model, H)
    ms = tot / args.steps
    gbs = job_rate(world, nbytes, ms) / 1e9
    peaks, src = measured_peaks()
    peak = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))
    achieved = nbytes / (statistics.mean(call_ms) * 1e-3) / 1e9
    traffic = recorded_traffic(os.path.join(ROOT, "mla_latent_kv_16_gb300", "csrc", "linear.cu"),
                               FUSED_WORKLOAD, prefix="linear")
    out = {
        "metric": FUSED_METRIC, "value": round(gbs, 2), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded W_O ~ N(0,1/sqrt(16384)), W_UV ~ N(0,1/sqrt(512)), u ~ N(0,1))",
        "config": {"workload": FUSED_WORKLOAD, "tokens": n, "heads": H, "d_model": d_model, "k_splits": splits,
                   "l2": "flushed before every timed call by reading a 256 MiB buffer; W~ (940 MB) > L2",
                   "parallelism": f"dp{world} (independent replicas, no collective)"},
        "tokens_per_s": round(job_rate(world, n, ms), 1),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "kernel": "mla_out_proj_fused (tcgen05 GEMM + split sum), algorithmic bytes = W~ + u + y",
                     "peak_source": f"hbm_gbs of {src}"},
        "e2e": {"value": round(job_rate(world, nbytes, e2e_tot / args.steps) / 1e9, 2), "unit": UNIT,
                "ms_per_step": round(e2e_tot / args.steps, 5), "h2d_bytes_per_step": host_u.numel() * 2,
                "d2h_bytes_per_step": host_y.numel() * 2},
        "gpu_launches": (2 if splits > 1 else 1) * args.steps,
        "clocks": clocks,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, sample, thr, el = cpu_fused_run(w, d_model, args.cpu_seconds)
        out["cpu_baseline"] = {"value": round(v, 4), "unit": UNIT, "cores": thr, "kind": "oracle",
                               "sample": sample, "seconds": round(el, 2)}
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_ours(args):
    import torch
    import torch.distributed as dist

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    from mla_latent_kv_16_gb300 import build as B
    if rank == 0 or world == 1:
        B.build()
    if world > 1:
        dist.barrier()
    from mla_latent_kv_16_gb300 import capi, workloads as W
    from mla_latent_kv_16_gb300.engine import build_layer, step_inputs
    capi.load()

    w = W.preset(args.workload, **({} if args.num_splits is None else {"num_splits": args.num_splits}))
    d = W.make_inputs(w)
    layer = build_layer(w, d)
    s = step_inputs(d)
    torch.cuda.synchronize()
    assert layer.device_error() == 0, "device error while filling the cache"
    path = capi.mla_decode_kernel_path(layer.cache, layer.scales, w.page_size, w.heads, w.act_dtype, w.cache_dtype)
    # L2 flush by READING a buffer larger than L2: it evicts the previous step's
    # data and leaves only clean lines (a write would leave dirty lines whose
    # write-back would then compete with the timed step for HBM)
    flush = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()

    # one decode step = append + absorb + decode + out_proj (split merge inside it), replayed
    # as a CUDA graph so that host launch overhead stays out of the step
    def one_step():
        layer.step(**s)

    def decode_only():
        layer.decode(layer.q_lat, s["q_rope"])

    g_step = layer.capture(one_step)
    g_dec = layer.capture(decode_only)

    def timed(graph, n, clk=None):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        if clk is not None:
            clk.start()
            time.sleep(0.3)
        for i in range(n):
            flush.sum()
            evs[i][0].record(stream)
            graph.replay()
            evs[i][1].record(stream)
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in evs]

    for _ in range(args.warmup):
        flush.sum()
        g_step.replay()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clk = ClockSampler(local)
    step_ms = timed(g_step, args.steps, clk)
    clocks = clk.stop()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    tot = max_over_ranks(sum(step_ms), world, "cuda")
    for _ in range(args.warmup):
        flush.sum()
        g_dec.replay()
    dec_ms = timed(g_dec, args.steps)
    assert layer.device_error() == 0

    # end to end through the public API: the step's inputs copied in from pinned
    # host memory and o copied back, inside the timed region (also a graph). The
    # inputs sit packed in one pinned buffer (256-byte aligned pieces), so the
    # step pays for one copy in rather than one per tensor.
    offs, total = {}, 0
    for k, v in s.items():
        offs[k] = total
        total += (v.numel() * v.element_size() + 255) // 256 * 256
    host_in = torch.zeros(total, dtype=torch.uint8).pin_memory()
    dev_in = torch.empty(total, dtype=torch.uint8, device="cuda")
    s_e2e = {}
    for k, v in s.items():
        nb = v.numel() * v.element_size()
        host_in[offs[k]:offs[k] + nb].copy_(v.cpu().contiguous().view(-1).view(torch.uint8))
        s_e2e[k] = dev_in[offs[k]:offs[k] + nb].view(v.dtype).view(v.shape)
    host_out = torch.empty(layer.o.shape, dtype=layer.o.dtype).pin_memory()
    h2d = total
    d2h = host_out.numel() * host_out.element_size()

    def e2e_step():
        dev_in.copy_(host_in, non_blocking=True)
        layer.step(**s_e2e)
        host_out.copy_(layer.o, non_blocking=True)

    g_e2e = layer.capture(e2e_step)
    for _ in range(args.warmup):
        flush.sum()
        g_e2e.replay()
    e2e_ms = timed(g_e2e, args.steps)
    e2e_tot = max_over_ranks(sum(e2e_ms), world, "cuda")

    cache_bytes = sum(int(L) for L in w.seq_lens) * w.row_bytes()
    ms = tot / args.steps
    gbs = job_rate(world, cache_bytes, ms) / 1e9
    tok_s = job_rate(world, w.batch * w.q_len, ms)
    e2e_msps = e2e_tot / args.steps
    dec = statistics.mean(dec_ms)
    peaks, src = measured_peaks()
    peak = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))
    achieved = decode_bytes(w) / (dec * 1e-3) / 1e9
    kernel_src = os.path.join(ROOT, "mla_latent_kv_16_gb300", "csrc",
                              "decode_tc.cu" if (w.heads == 128 and w.act_dtype == "bf16") else "decode_simt.cu")
    traffic = recorded_traffic(kernel_src, w.name)
    splits = layer.splits
    launches_per_step = 4 + capi.merge_kernel_launches(path, splits, with_out_proj=True)
    out = {
        "metric": METRIC, "value": round(gbs, 2), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w.cache_dtype, "data": "synthetic (seeded N(0,1) values, N(0,1/sqrt(512)) weights)",
        "config": {"workload": w.name, "batch": w.batch, "q_len": w.q_len, "heads": w.heads,
                   "seq_len": int(max(w.seq_lens)), "page_size": w.page_size, "cache_dtype": w.cache_dtype,
                   "num_splits": splits, "decode_kernel": {capi.MLA_DECODE_PATH_TENSOR_CORE: "tcgen05",
                                                            capi.MLA_DECODE_PATH_CUDA_CORE: "cuda-core"}.get(path),
                   "l2": "flushed before every timed step by reading a 256 MiB buffer (clean lines); cache > L2",
                   "parallelism": f"dp{world} (independent replicas, no collective)"},
        "tokens_per_s": round(tok_s, 1),
        "decode_call_ms": round(dec, 5),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "kernel": "mla_decode_paged (decode + split merge), algorithmic bytes = cache rows + q + u + lse",
                     "peak_source": f"hbm_gbs of {src}"},
        "e2e": {"value": round(job_rate(world, cache_bytes, e2e_msps) / 1e9, 2), "unit": UNIT,
                "ms_per_step": round(e2e_msps, 5), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, sample, thr, el = cpu_oracle_run(w, d, args.cpu_seconds)
        out["cpu_baseline"] = {"value": round(v, 4), "unit": UNIT, "cores": thr, "kind": "oracle",
                               "sample": sample, "seconds": round(el, 2),
                               "variants": cpu_variants(w.name, max(2.0, args.cpu_seconds / 2))}
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        dist.destroy_process_group()


def layer_bytes(w, d_model: int, d_cq: int, fused: bool = True) -> int:
    """Algorithmic HBM bytes of one layer step (bf16): every weight once (W_DQKV,
    W_UQR, W_UK, and W~ when the output projection is fused, else W_UV and W_O),
    the visible cache rows, and the step's activations (plus o when unfused)."""
    H, n = w.heads, w.batch * w.q_len
    out_w = d_model * H * 512 if fused else H * 128 * 512 + d_model * H * 128
    weights = 2 * ((d_cq + 512 + 64) * d_model + H * 192 * d_cq + H * 128 * 512 + out_w)
    cache = sum(int(L) for L in w.seq_lens) * w.row_bytes()
    acts = 2 * n * (d_model + H * (128 + 64 + 512 + 512) + 576 + d_model + (0 if fused else 2 * H * 128))
    return weights + cache + acts


def cpu_layer_run(w, d, fr, w_o, seconds: float):
    """Time the oracle's whole layer on a bounded sample: the front end for every
    token of the step, then, sequence by sequence, the materialised attention
    (all heads) and W_O over the heads, until `seconds` of oracle work are done.
    The oracle's cache is built as untimed set-up. Returns (tokens/s, sample,
    threads, seconds)."""
    import numpy as np
    from oracle import mla_oracle as O
    from oracle.harness import f64, oracle_pool, seq_token_mask
    from mla_latent_kv_16_gb300 import workloads as W

    pos = d["ctx_positions"][d["new_index"]].numpy()
    t0 = time.perf_counter()
    q_nope, q_rope, c_kv, k_r = O.decode_front(f64(fr["h"]), f64(fr["w_dq"]), f64(fr["g_q"]), f64(fr["w_uq"]),
                                               f64(fr["w_qr"]), f64(fr["w_dkv"]), f64(fr["g_kv"]),
                                               f64(fr["w_kr"]), pos, W.RMS_EPS)
    elapsed = time.perf_counter() - t0
    wo64, wuk, wuv = f64(w_o), f64(d["w_uk"]), f64(d["w_uv"])
    bt = d["block_table"].numpy()
    H, Lq = w.heads, w.q_len
    done = 0
    for b in range(w.batch):
        pool, sc = oracle_pool(w, d, token_mask=seq_token_mask(w, [b]))
        t1 = time.perf_counter()
        full = O.decode_full(q_nope.reshape(w.batch, Lq, H, 128), q_rope.reshape(w.batch, Lq, H, 64), wuk, wuv,
                             pool, sc, bt, d["seq_lens"].numpy(), Lq, w.page_size, w.cache_dtype,
                             O.default_scale(), batch_index=[b])
        O.out_proj_model(full[b][0], wo64)
        elapsed += time.perf_counter() - t1
        done += Lq
        if elapsed > seconds:
            break
    sample = (f"front end for all {w.batch * Lq} tokens, then {done} token(s) of {w.name} through the "
              f"materialised fp64 attention and W_O")
    return done / elapsed, sample, os.cpu_count(), elapsed


def run_layer(args):
    """One whole decode layer step per timed iteration, replayed as a graph."""
    import torch

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    from mla_latent_kv_16_gb300 import build as B
    B.build()
    from mla_latent_kv_16_gb300 import capi, workloads as W
    from mla_latent_kv_16_gb300.engine import build_layer
    capi.load()
    w = W.preset(DEFAULT_WORKLOAD)
    d = W.make_inputs(w)
    d_model, d_cq, H, n = W.D_MODEL, W.D_CQ, w.heads, w.batch * w.q_len
    fr = W.make_front_inputs(w, d_model, d_cq)
    w_o = W.make_out_weight(w, d_model)
    layer = build_layer(w, d)
    ni = d["new_index"]
    pos = d["ctx_positions"][ni].cuda()
    slots = d["ctx_slots"][ni].cuda()
    h = fr["h"].cuda()
    layer.attach_front(fr["w_dq"], fr["w_dkv"], fr["w_kr"], fr["g_q"], fr["g_kv"], fr["w_uq"], fr["w_qr"], W.RMS_EPS)
    # the same layer twice over one cache: the output projection fused, and unfused
    import copy
    unf = copy.copy(layer)
    unf.attach_output(w_o, fused=False)
    layer.attach_output(w_o, fused=True)
    y = layer.y
    flush = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()
    torch.cuda.synchronize()
    assert layer.device_error() == 0

    def step_fused():
        layer.step_from_hidden(h, pos, slots)

    def step_unfused():
        unf.step_from_hidden(h, pos, slots)

    g_fused = layer.capture(step_fused)
    g_unfused = layer.capture(step_unfused)

    def timed(graph, k, clk=None):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(k)]
        if clk is not None:
            clk.start()
            time.sleep(0.3)
        for i in range(k):
            flush.sum()
            evs[i][0].record(stream)
            graph.replay()
            evs[i][1].record(stream)
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in evs]

    for g_ in (g_fused, g_unfused):
        for _ in range(args.warmup):
            flush.sum()
            g_.replay()
    torch.cuda.synchronize()
    # the line reports the faster output projection, as measured here (at a decode
    # batch of 32 the unfused one: W~ is 3.7 times the bytes of W_UV and W_O);
    # the clock samples cover the timed steps of the one reported
    probe_f = statistics.mean(timed(g_fused, 20))
    probe_u = statistics.mean(timed(g_unfused, 20))
    use_fused = probe_f <= probe_u
    clk = ClockSampler(local)
    if use_fused:
        fused_ms = timed(g_fused, args.steps, clk)
        clocks = clk.stop()
        unfused_ms = timed(g_unfused, args.steps)
    else:
        unfused_ms = timed(g_unfused, args.steps, clk)
        clocks = clk.stop()
        fused_ms = timed(g_fused, args.steps)
    assert layer.device_error() == 0

    host_h = fr["h"].pin_memory()
    host_y = torch.empty(y.shape, dtype=y.dtype).pin_memory()

    def e2e():
        h.copy_(host_h, non_blocking=True)
        (step_fused if use_fused else step_unfused)()
        host_y.copy_(layer.y if use_fused else unf.y, non_blocking=True)

    g_e2e = layer.capture(e2e)
    for _ in range(args.warmup):
        flush.sum()
        g_e2e.replay()
    e2e_ms = statistics.mean(timed(g_e2e, args.steps))

    ms = statistics.mean(fused_ms if use_fused else unfused_ms)
    nbytes = layer_bytes(w, d_model, d_cq, use_fused)
    peaks, src = measured_peaks()
    peak = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))
    achieved = nbytes / (ms * 1e-3) / 1e9
    if use_fused:
        out_launches = 2 if capi.mla_out_proj_fused_workspace_size(n, d_model, H) else 1
    else:  # W_UV per head, then W_O over the concatenated heads (+ its split sum)
        out_launches = 1 + (2 if capi.mla_linear_workspace_size(n, d_model, H * 128) else 1)
    path = capi.mla_decode_kernel_path(layer.cache, layer.scales, w.page_size, w.heads, w.act_dtype, w.cache_dtype)
    launches = 4 + 1 + 1 + 1 + capi.merge_kernel_launches(path, layer.splits, with_out_proj=not use_fused) + out_launches
    out = {
        "metric": LAYER_METRIC, "value": round(n / (ms * 1e-3), 1), "unit": "tokens/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded hidden states, N(0,1/sqrt(fan_in)) weights, RMSNorm gains 1 + 0.1 N(0,1))",
        "config": {"workload": LAYER_WORKLOAD, "batch": w.batch, "q_len": w.q_len, "heads": H, "d_model": d_model,
                   "d_cq": d_cq, "seq_len": int(max(w.seq_lens)), "page_size": w.page_size,
                   "num_splits": layer.splits, "output_projection": "fused" if use_fused else "unfused",
                   "l2": "flushed before every timed step by reading a 256 MiB buffer; weights + cache > L2",
                   "parallelism": "dp1 (one replica)"},
        "fused_output_ms_per_step": round(statistics.mean(fused_ms), 5),
        "unfused_output_ms_per_step": round(statistics.mean(unfused_ms), 5),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": None,
                     "kernel": "whole layer step; algorithmic bytes = W_DQKV + W_UQR + W_UK + (W~, or W_UV + W_O) + cache rows + activations",
                     "bytes_per_step": nbytes, "peak_source": f"hbm_gbs of {src}"},
        "e2e": {"value": round(n / (e2e_ms * 1e-3), 1), "unit": "tokens/s", "ms_per_step": round(e2e_ms, 5),
                "h2d_bytes_per_step": host_h.numel() * 2, "d2h_bytes_per_step": host_y.numel() * 2},
        "gpu_launches": launches * args.steps,
        "clocks": clocks,
    }
    if not args.no_cpu_baseline:
        v, sample, thr, el = cpu_layer_run(w, d, fr, w_o, args.cpu_seconds)
        out["cpu_baseline"] = {"value": round(v, 4), "unit": "tokens/s", "cores": thr, "kind": "oracle",
                               "sample": sample, "seconds": round(el, 2)}
    print(json.dumps(out), flush=True)


def prefill_flops(T: int, Tq: int, H: int) -> float:
    """Algorithmic FLOPs of one prefill call: the expansion (K_nope and V, each
    [T x 512] x [512 x 128 H]) and the causal attention (query j sees
    T - Tq + j + 1 keys; 192-wide scores, 128-wide values)."""
    vis = sum(T - Tq + j + 1 for j in range(Tq))
    return 2.0 * 2 * T * 512 * 128 * H + 2.0 * H * vis * (192 + 128)


def cpu_prefill_run(d, seconds: float):
    """The oracle's per-query non-absorbed attention (materialised K/V of the
    visible rows, every head) on queries spread over the prompt, for a bounded
    time; returns (TFLOP/s, sample, threads, seconds)."""
    import numpy as np
    from oracle import mla_oracle as O
    from oracle.harness import f64
    rows = f64(d["rows"])
    qn, qr, wuk, wuv = f64(d["q_nope"]), f64(d["q_rope"]), f64(d["w_uk"]), f64(d["w_uv"])
    T, H = rows.shape[0], qn.shape[1]
    order = np.random.default_rng(7).permutation(T)
    t0 = time.time()
    flops, n = 0.0, 0
    for j in order:
        O.attend_nonabsorbed(qn[j], qr[j], wuk, wuv, rows[:j + 1], O.default_scale())
        flops += 2.0 * H * (j + 1) * (512 * 256 + 192 + 128)
        n += 1
        if time.time() - t0 > seconds:
            break
    el = time.time() - t0
    return flops / el / 1e12, f"{n} queries of the {T}-token prompt (all {H} heads; non-absorbed fp64 oracle, K/V materialised per query)", \
        os.cpu_count() or 1, el


def run_prefill(args):
    """One mla_prefill_mha call per step on a 4096-token prompt (128 heads)."""
    import torch

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    from mla_latent_kv_16_gb300 import build as B
    B.build()
    from mla_latent_kv_16_gb300 import capi, workloads as W
    capi.load()
    T, H = PREFILL_T, 128
    d = W.make_prefill_inputs(T, T, H, seed=1)
    dev = {k: v.cuda() for k, v in d.items()}
    ws = torch.empty(capi.mla_prefill_workspace_size(T, H), dtype=torch.uint8, device="cuda")
    o = torch.empty(T, H, 128, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(T, H, dtype=torch.float32, device="cuda")
    flush = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()

    def call():
        capi.mla_prefill_mha(dev["q_nope"], dev["q_rope"], dev["rows"], dev["w_uk"], dev["w_uv"], workspace=ws,
                             o_out=o, lse_out=lse)

    def capture(fn):
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            for _ in range(2):
                fn()
        stream.wait_stream(side)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        return g

    def timed(graph, k, clk=None):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(k)]
        if clk is not None:
            clk.start()
            time.sleep(0.3)
        for i in range(k):
            flush.sum()
            evs[i][0].record(stream)
            graph.replay()
            evs[i][1].record(stream)
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in evs]

    g_call = capture(call)
    for _ in range(args.warmup):
        flush.sum()
        g_call.replay()
    torch.cuda.synchronize()
    clk = ClockSampler(local)
    call_ms = timed(g_call, args.steps, clk)
    clocks = clk.stop()
    host = {k: d[k].pin_memory() for k in ("q_nope", "q_rope", "rows")}
    host_o = torch.empty(o.shape, dtype=o.dtype).pin_memory()

    def e2e():
        for k in host:
            dev[k].copy_(host[k], non_blocking=True)
        call()
        host_o.copy_(o, non_blocking=True)

    g_e2e = capture(e2e)
    for _ in range(args.warmup):
        flush.sum()
        g_e2e.replay()
    e2e_ms = statistics.mean(timed(g_e2e, args.steps))
    fl = prefill_flops(T, T, H)
    ms = statistics.mean(call_ms)
    tfs = fl / (ms * 1e-3) / 1e12
    peaks, src = measured_peaks()
    peak = float(peaks.get("bf16_tflops", FALLBACK_BF16_TFLOPS))
    out = {
        "metric": PREFILL_METRIC, "value": round(tfs, 2), "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded rows, q ~ N(0,1); W_UK, W_UV ~ N(0,1/sqrt(512)))",
        "config": {"workload": PREFILL_WORKLOAD, "tokens": T, "queries": T, "heads": H,
                   "l2": "flushed before every timed call by reading a 256 MiB buffer",
                   "parallelism": "dp1 (one sequence)"},
        "tokens_per_s": round(T / (ms * 1e-3), 1),
        "roofline": {"bound": "tensor", "achieved": round(tfs, 1), "peak": peak, "unit": "TFLOP/s",
                     "frac": round(tfs / peak, 4),
                     "traffic": recorded_traffic(os.path.join(ROOT, "mla_latent_kv_16_gb300", "csrc", "prefill.cu"),
                                                 PREFILL_WORKLOAD, prefix="prefill_attn"),
                     "kernel": "mla_prefill_mha (2 tcgen05 expansion GEMMs + causal attention), algorithmic FLOPs",
                     "peak_source": f"bf16_tflops of {src}"},
        "e2e": {"value": round(fl / (e2e_ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s", "ms_per_step": round(e2e_ms, 5),
                "h2d_bytes_per_step": sum(v.numel() * v.element_size() for v in host.values()),
                "d2h_bytes_per_step": host_o.numel() * 2},
        "gpu_launches": 3 * args.steps,
        "clocks": clocks,
    }
    if not args.no_cpu_baseline:
        v, sample, thr, el = cpu_prefill_run(d, args.cpu_seconds)
        out["cpu_baseline"] = {"value": round(v, 6), "unit": "TFLOP/s", "cores": thr, "kind": "oracle",
                               "sample": sample, "seconds": round(el, 2)}
    print(json.dumps(out), flush=True)


def run_reference_prefill(args):
    from mla_latent_kv_16_gb300 import workloads as W
    T, H = PREFILL_T, 128
    d = W.make_prefill_inputs(T, T, H, seed=1)
    budget = max(2.0, 150.0 / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        cpu_prefill_run(d, min(budget, 2.0))
    vals, secs, sample, thr = [], 0.0, "", 1
    for _ in range(args.steps):
        v, sample, thr, el = cpu_prefill_run(d, budget)
        vals.append(v)
        secs += el
    value = statistics.mean(vals)
    out = {"impl": "reference", "metric": PREFILL_METRIC, "value": round(value, 6), "unit": "TFLOP/s",
           "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * secs / args.steps, 2),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic (seeded)", "config": {"workload": PREFILL_WORKLOAD, "tokens": T, "queries": T,
                                                     "heads": H},
           "cpu_baseline": {"kind": "oracle", "cores": thr, "sample": sample, "value": round(value, 6),
                            "unit": "TFLOP/s"},
           "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def run_reference_fused(args):
    from mla_latent_kv_16_gb300 import workloads as W
    w = W.preset(DEFAULT_WORKLOAD)
    budget = max(2.0, 150.0 / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        cpu_fused_run(w, W.D_MODEL, min(budget, 2.0))
    vals, secs, sample, thr = [], 0.0, "", 1
    for _ in range(args.steps):
        v, sample, thr, el = cpu_fused_run(w, W.D_MODEL, budget)
        vals.append(v)
        secs += el
    value = statistics.mean(vals)
    out = {"impl": "reference", "metric": FUSED_METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": 1,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * secs / args.steps, 2),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic (seeded)", "config": {"workload": FUSED_WORKLOAD, "tokens": w.batch * w.q_len,
                                                     "heads": w.heads, "d_model": W.D_MODEL},
           "cpu_baseline": {"kind": "oracle", "cores": thr, "sample": sample, "value": round(value, 4), "unit": UNIT},
           "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def run_reference_layer(args):
    from mla_latent_kv_16_gb300 import workloads as W
    w = W.preset(DEFAULT_WORKLOAD)
    d = W.make_inputs(w)
    fr = W.make_front_inputs(w, W.D_MODEL, W.D_CQ)
    w_o = W.make_out_weight(w, W.D_MODEL)
    budget = max(2.0, 150.0 / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        cpu_layer_run(w, d, fr, w_o, min(budget, 2.0))
    vals, secs, sample, thr = [], 0.0, "", 1
    for _ in range(args.steps):
        v, sample, thr, el = cpu_layer_run(w, d, fr, w_o, budget)
        vals.append(v)
        secs += el
    value = statistics.mean(vals)
    out = {"impl": "reference", "metric": LAYER_METRIC, "value": round(value, 4), "unit": "tokens/s", "n_gpus": 1,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * secs / args.steps, 2),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic (seeded)", "config": {"workload": LAYER_WORKLOAD, "batch": w.batch, "q_len": w.q_len,
                                                     "heads": w.heads, "d_model": W.D_MODEL, "d_cq": W.D_CQ},
           "cpu_baseline": {"kind": "oracle", "cores": thr, "sample": sample, "value": round(value, 4),
                            "unit": "tokens/s"},
           "e2e": {"value": round(value, 4), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    if args.workload == FUSED_WORKLOAD:
        return run_reference_fused(args)
    if args.workload == LAYER_WORKLOAD:
        return run_reference_layer(args)
    if args.workload == PREFILL_WORKLOAD:
        return run_reference_prefill(args)
    from mla_latent_kv_16_gb300 import workloads as W
    w = W.preset(args.workload)
    d = W.make_inputs(w)
    budget = max(2.0, 150.0 / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        cpu_oracle_run(w, d, min(budget, 2.0))
    vals, secs = [], 0.0
    sample, thr = "", 1
    for _ in range(args.steps):
        v, sample, thr, el = cpu_oracle_run(w, d, budget)
        vals.append(v)
        secs += el
    value = statistics.mean(vals)
    out = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * secs / args.steps, 2),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic (seeded)", "config": {"workload": w.name, "batch": w.batch, "q_len": w.q_len,
                                                     "heads": w.heads, "seq_len": int(max(w.seq_lens)),
                                                     "page_size": w.page_size, "cache_dtype": w.cache_dtype},
           "cpu_baseline": {"kind": "oracle", "cores": thr, "sample": sample, "value": round(value, 4), "unit": UNIT},
           "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    elif args.workload == FUSED_WORKLOAD:
        run_fused(args)
    elif args.workload == LAYER_WORKLOAD:
        run_layer(args)
    elif args.workload == PREFILL_WORKLOAD:
        run_prefill(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
