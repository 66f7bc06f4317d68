#!/usr/bin/env python
"""Throughput of the YOCO token-mixing hot path on one GB300 (per rank).

One step = one YOCO-3B-shaped 512K-token prompt with early exit (the paper's
Section 2.3, Fig. 3: the cross-decoder runs only for the last prompt token):

  13 x chunkwise gRet over 524288 tokens (24 heads x 128; per-layer q, k, v, logits)
  shared K^/V^ projection of M [524288, 3072] (RMSNorm, W_K/W_V 3072 -> 8 x 128)
  13 x cross attention for the last prompt token (24 q heads, GQA 3:1)

value  = prompt tokens per second over the timed steps (inputs resident in HBM);
e2e    = the same with the step's inputs copied from pinned host memory and the
         cross layers' outputs copied back, inside the timed region;
decode = generated tokens per second at a 1M-token context: 13 recurrent gRet
         steps, a one-slot append and 13 split-KV cross layers per token.
--impl reference times the CPU oracle on a bounded sample of the same step.

Multi-GPU: replicas only (independent requests per GPU); value sums all ranks.
"""
import argparse
import ctypes
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "gRet prefill tok/s + shared-KV decode tok/s (1 GB300), % of TC/HBM roofline"
SEED = 20240509
B, N, H, D = 1, 524288, 24, 128            # the 512K prompt, one sequence
L_SELF, L_CROSS = 13, 13
DM, HKV, HQ = 3072, 8, 24
TAU, EPS = 16.0, 1e-6
CFG = 4                                     # stream-id tag of the 512K prompt's inputs
N_DEC, CFG_DEC = 1048576, 5                 # the 1M-token decode context
N_LAYER = 32768                             # --only: the single 32K-token gRet layer shape
CFG_LAYER = 2

# DRAM bytes of one gRet prefill call on the 512K layer (524288 x 24 x 128, bf16):
# dram__bytes_read.sum + dram__bytes_write.sum of both launches of one call, from
# the capture summarised in profiles/gret_tc_kernel_512k_x24_layer.md (the command
# is given there).  None until a capture of the current kernels exists.
GRET_CALL_DRAM_BYTES = 224734208 + 3112448 + 9726954496 + 3163062272


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=10)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", choices=["yoco", "reference"], default="yoco")
    p.add_argument("--e2e-steps", type=int, default=3)
    p.add_argument("--decode-tokens", type=int, default=20, help="timed tokens of the 1M-context decode")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--chunk", type=int, default=0)
    p.add_argument("--only", choices=["gret", "gret_gn", "gret_gn_unfused", "proj", "append", "cross_decode", "cross_prefill", "swa_prefill",
                                      "swa_decode", "gn_gate", "rope", "qkvg", "gret_decode_unfused",
                                      "gret_decode_gn", "gret_steps", "gret_steps_append"], default=None,
                   help="time one call kind on its own (for profiling)")
    p.add_argument("--n", type=int, default=0, help="--only gret: tokens (default 32768)")
    p.add_argument("--segments", type=int, default=0,
                   help="--only gret: segments per head (test hook; 0 = one CTA per SM over the heads)")
    p.add_argument("--no-decay", action="store_true",
                   help="--only gret: logits +inf (gamma = 1), the case where nothing is left out")
    p.add_argument("--cache-len", type=int, default=0,
                   help="--only cross_decode: cache length (default 32768)")
    p.add_argument("--batch", type=int, default=0, help="--only cross_decode: sequences (default 1)")
    p.add_argument("--splits", type=int, default=0, help="--only cross_decode: key splits (default: automatic)")
    p.add_argument("--workload", choices=list(LONG_WORKLOADS), default=None,
                   help="time one of the decode workloads at the pages' sizes instead of the bench step "
                        "(one JSON line per workload and batch; not the driver's line)")
    p.add_argument("--batches", default="1,8,32", help="--workload decode128k: batch sizes")
    p.add_argument("--rope-base", type=float, default=0.0,
                   help="--only proj/cross_decode/cross_prefill: rotary encoding base of the cache (0: off)")
    return p.parse_args()


def workload_config(chunk_used):
    return {"workload": "yoco3b_prefill512k_early_exit", "B": B, "N": N, "self_layers": L_SELF,
            "gret_heads": H, "d": D, "chunk": chunk_used, "tau": TAU, "cross_layers": L_CROSS,
            "cross_rows": 1, "Hq": HQ, "Hkv": HKV, "d_model": DM, "gate_logits": "N(2,1)",
            "qk": "N(0,1)/sqrt(128)", "v_M_Q": "N(0,1)", "W": "N(0,0.02)",
            "l2": "no flush: each step reads 129 GB of inputs (> 129 MB L2)", "parallelism": "replicas"}


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f)
    except OSError:
        return {}


# ----------------------------------------------------------------- CPU oracle

SAMPLE_TOKENS, SAMPLE_ROWS, SAMPLE_KEYS = 12288, 64, 16384


def _cpu_inputs(tokens, proj_rows, cross_keys):
    """Seeded host inputs of the CPU sample, drawn like the step's (same streams)."""
    import synth
    sid = synth.stream_id
    f = synth.bf16_bits_to_f32
    return dict(
        q=f(synth.normal(SEED, sid(CFG, 0, synth.T_Q), (1, tokens, H, D), "bf16", std=D ** -0.5)),
        k=f(synth.normal(SEED, sid(CFG, 0, synth.T_K), (1, tokens, H, D), "bf16", std=D ** -0.5)),
        v=f(synth.normal(SEED, sid(CFG, 0, synth.T_V), (1, tokens, H, D), "bf16")),
        lg=synth.normal(SEED, sid(CFG, 0, synth.T_LOGIT), (1, tokens, H), "f32", mean=2.0),
        M=f(synth.normal(SEED, sid(CFG, 0, synth.T_M), (proj_rows, DM), "bf16")),
        W=f(synth.normal(SEED, sid(CFG, 0, synth.T_WK), (DM, 2 * HKV * D), "bf16", std=0.02)),
        Kc=f(synth.normal(SEED, sid(CFG, 0, synth.T_CACHE_K), (1, HKV, cross_keys, D), "bf16")),
        Vc=f(synth.normal(SEED, sid(CFG, 0, synth.T_CACHE_V), (1, HKV, cross_keys, D), "bf16")),
        Qx=f(synth.normal(SEED, sid(CFG, 0, synth.T_QX), (1, 1, HQ, D), "bf16")))


def cpu_sample(x, threads=0):
    """Time the oracle, as it stands, on the bounded sample `x` (one gRet layer's
    first SAMPLE_TOKENS tokens x 24 heads, SAMPLE_ROWS projection rows, one cross
    row over SAMPLE_KEYS keys) and scale each part linearly to the whole step.
    threads = 0: all the host cores the process may use.  Returns (seconds per
    step, seconds the sample took, cores used)."""
    import oracle
    cores = threads or len(os.sched_getaffinity(0))
    oracle.set_threads(cores)
    t0 = time.perf_counter()
    oracle.gret_recurrent(x["q"], x["k"], x["v"], x["lg"], TAU)
    t_gret = time.perf_counter() - t0
    t0 = time.perf_counter()
    oracle.rmsnorm_proj(x["M"], x["W"], EPS)
    t_proj = time.perf_counter() - t0
    t0 = time.perf_counter()
    oracle.cross_attn(x["Qx"], x["Kc"], x["Vc"], SAMPLE_KEYS - 1, D ** -0.5)
    t_cross = time.perf_counter() - t0
    step = (L_SELF * t_gret * (N / SAMPLE_TOKENS) + t_proj * (N / SAMPLE_ROWS)
            + L_CROSS * t_cross * (N / SAMPLE_KEYS))
    return step, t_gret + t_proj + t_cross, cores


SAMPLE_DESC = (f"oracle timed on {SAMPLE_TOKENS} tokens x 24 heads of one gRet layer, {SAMPLE_ROWS} projection "
               f"rows and one cross row over {SAMPLE_KEYS} keys; each part scaled linearly to the step "
               f"(13 gRet layers x {N} tokens, {N} projection rows, 13 cross rows over {N} keys)")


def cpu_baseline_block():
    """The oracle on all host cores and on one core, each on the bounded sample."""
    x = _cpu_inputs(SAMPLE_TOKENS, SAMPLE_ROWS, SAMPLE_KEYS)
    step_all, sample_all, cores = cpu_sample(x)
    step_one, sample_one, _ = cpu_sample(x, threads=1)
    return {"value": N / step_all, "unit": "tok/s", "cores": cores, "kind": "oracle", "sample": SAMPLE_DESC,
            "sample_s": round(sample_all, 3), "extrapolated_ms_per_step": round(step_all * 1e3, 1),
            "single_thread": {"value": N / step_one, "unit": "tok/s", "cores": 1, "sample_s": round(sample_one, 3),
                              "extrapolated_ms_per_step": round(step_one * 1e3, 1)}}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    x = _cpu_inputs(SAMPLE_TOKENS, SAMPLE_ROWS, SAMPLE_KEYS)
    times, samples, cores = [], [], 1
    for i in range(args.warmup + args.steps):
        step, sample, cores = cpu_sample(x)
        if i >= args.warmup:
            times.append(step)
            samples.append(sample)
    t = statistics.mean(times)
    value = N / t
    sample_s = statistics.mean(samples)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tok/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": sample_s * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config("auto"),
            "timing": ("each step is the oracle timed on a bounded sample of the workload; ms_per_step is that "
                       "measured time; value is the step's tokens over the sample's time scaled linearly to the "
                       "whole step (extrapolated_ms_per_step)"),
            "extrapolated_ms_per_step": round(t * 1e3, 1),
            "sample_s_per_step": round(sample_s, 3),
            "cpu_baseline": {"value": value, "unit": "tok/s", "cores": cores, "kind": "oracle",
                             "sample": SAMPLE_DESC},
            "e2e": {"value": value, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------- GPU arm

def aggregate_over_ranks(elapsed_s, units_per_rank, dist=None, device="cpu"):
    """Whole-job throughput of independent replicas: the units every rank
    processed over the slowest rank's time.  Returns (units/s, max seconds)."""
    import torch
    world = 1
    if dist is not None and dist.is_initialized():
        world = dist.get_world_size()
        t = torch.tensor([float(elapsed_s)], device=device, dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        elapsed_s = float(t)
    return world * units_per_rank / elapsed_s, elapsed_s


class Clocks:
    """nvidia-smi sampler (every 100 ms) running across the timed region; each line
    is stamped on arrival so the summary keeps the samples taken inside a window."""

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []
        self.thread = None

    def __enter__(self):
        import threading
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={q}", "--format=csv,noheader,nounits",
                                          "-i", str(self.index), "-lms", "100"], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        if self.proc is not None:
            def reader():
                for line in self.proc.stdout:
                    self.lines.append((time.monotonic(), line))
            self.thread = threading.Thread(target=reader, daemon=True)
            self.thread.start()
        return self

    def wait_first(self, timeout=3.0):
        t0 = time.monotonic()
        while self.proc is not None and not self.lines and time.monotonic() - t0 < timeout:
            time.sleep(0.01)

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.proc.wait()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t_lo=None, t_hi=None):
        """Samples stamped in [t_lo, t_hi] (all of them without a window)."""
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ts, line in self.lines:
            if (t_lo is not None and ts < t_lo) or (t_hi is not None and ts > t_hi):
                continue
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, val in zip(names, f[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def run_gpu(args):
    import torch

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")

    import gated_retention_shared_gb300 as Y
    import synth
    L = Y.lib
    dev = torch.device("cuda", local)
    bf, f32 = torch.bfloat16, torch.float32
    sid = synth.stream_id
    seed = SEED + 7919 * rank  # replicas serve different requests

    def normal(shape, dtype, stream, mean=0.0, std=1.0):
        t = torch.empty(shape, dtype=dtype, device=dev)
        return synth.fill_normal_(t, seed, stream, mean, std)

    # ---- the prompt's inputs (HBM resident): 13 layers of q, k, v, logits, M, W, queries
    q = [normal((B, N, H, D), bf, sid(CFG, l, synth.T_Q), std=D ** -0.5) for l in range(L_SELF)]
    k = [normal((B, N, H, D), bf, sid(CFG, l, synth.T_K), std=D ** -0.5) for l in range(L_SELF)]
    v = [normal((B, N, H, D), bf, sid(CFG, l, synth.T_V)) for l in range(L_SELF)]
    lg = [normal((B, N, H), f32, sid(CFG, l, synth.T_LOGIT), mean=2.0) for l in range(L_SELF)]
    M = normal((B, N, DM), bf, sid(CFG, 0, synth.T_M))
    Wk = normal((DM, HKV * D), bf, sid(CFG, 0, synth.T_WK), std=0.02)
    Wv = normal((DM, HKV * D), bf, sid(CFG, 0, synth.T_WV), std=0.02)
    Qx = [normal((B, 1, HQ, D), bf, sid(CFG, l, synth.T_QX)) for l in range(L_CROSS)]
    # ---- outputs and state: each layer's o is consumed before the next layer runs
    o = torch.empty(B, N, H, D, dtype=bf, device=dev)
    S = [torch.zeros(B, H, D, D, dtype=f32, device=dev) for _ in range(L_SELF)]
    Ox = [torch.empty(B, 1, HQ, D, dtype=bf, device=dev) for _ in range(L_CROSS)]
    cache = Y.KVCache(B, HKV, D, N + 16, device=dev)
    cc = ctypes.byref(cache.c)
    ws_n = max(L.yoco_gret_prefill_workspace_size(B, N, H, D, D, args.chunk, Y.YOCO_BF16),
               L.yoco_shared_kv_workspace_size(B, N, DM, cc), L.yoco_cross_attn_workspace_size(B, HQ, 1, cc, 0), 256)
    ws = torch.empty(ws_n, dtype=torch.uint8, device=dev)
    torch.cuda.synchronize()

    P = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    wsp, wsn = P(ws), ws.numel()
    stream = torch.cuda.current_stream(dev)
    stp = ctypes.c_void_p(stream.cuda_stream)

    def check(st, what):
        if st != 0:
            raise RuntimeError(f"{what}: {L.yoco_last_error().decode()}")

    def step(gret_events=None, marks=None, wait_layer=None, wait_rest=None):
        def mark(i):
            if marks is not None:
                marks[i].record(stream)
        for s in S:
            s.zero_()
        cache.len_dev.zero_()
        cache.c.len_host = 0
        mark(0)
        if gret_events is not None:
            gret_events[0].record(stream)  # the gRet phase as a whole: no event between its launches
        for l in range(L_SELF):
            if wait_layer is not None:
                wait_layer(l)  # end to end: this layer's inputs have arrived
            check(L.yoco_gret_prefill_chunkwise(P(q[l]), P(k[l]), P(v[l]), P(lg[l]), TAU, P(o), P(S[l]), B, N, H, D,
                                                D, args.chunk, 1, 1, wsp, wsn, stp), "gret prefill")
        if gret_events is not None:
            gret_events[1].record(stream)
        mark(1)
        if wait_rest is not None:
            wait_rest()
        check(L.yoco_shared_kv_project_append(P(M), None, EPS, P(Wk), P(Wv), N, DM, cc, wsp, wsn, stp), "kv append")
        mark(2)
        for l in range(L_CROSS):
            check(L.yoco_cross_attn_prefill(P(Qx[l]), HQ, 1, N - 1, cc, D ** -0.5, P(Ox[l]), wsp, wsn, stp),
                  "cross prefill")
        mark(3)

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    # the clock sampler starts before the warm-up so that it is sampling when the
    # timed region begins; the summary keeps the samples stamped inside that region
    # (plus one interval on either side, the GPU being busy then too)
    clk = Clocks(local).__enter__()
    clk.wait_first()
    for _ in range(args.warmup):
        step()
    launches0 = L.yoco_launch_count()
    step()
    launches_per_step = L.yoco_launch_count() - launches0
    barrier()

    # ---- timed region: K steps, events around each step's gRet phase (13 calls back to back)
    gret_ev = [[torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)] for _ in range(args.steps)]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    t_lo = time.monotonic()
    e0.record(stream)
    for i in range(args.steps):
        step(gret_ev[i])
    e1.record(stream)
    barrier()
    t_hi = time.monotonic()
    time.sleep(0.12)  # let the sample that closes the region arrive
    clk.__exit__(None, None, None)
    elapsed = e0.elapsed_time(e1) / 1e3
    value, elapsed = aggregate_over_ranks(elapsed, B * N * args.steps, dist, dev)
    ms_step = elapsed / args.steps * 1e3
    # average gRet call: each timed step's 13 back-to-back calls over 13 (events only around the phase)
    gret_ms = statistics.mean(c[0].elapsed_time(c[1]) / L_SELF for c in gret_ev)

    # ---- per-phase split: one more (untimed) step with events between phases
    marks = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    phase_names = ["gret_prefill_x13", "kv_project_512k", "cross_last_row_x13"]
    step(marks=marks)
    torch.cuda.synchronize()
    phases = {n: round(marks[i].elapsed_time(marks[i + 1]), 4) for i, n in enumerate(phase_names)}

    # ---- roofline of the dominant call: chunkwise gRet prefill, one layer
    peaks = load_peaks()
    hbm_peak = peaks.get("hbm_gbs", 6800.0)
    # algorithmic bytes of one call: q, k, v read and o written (bf16), the gate
    # logits (fp32), the state read and written (fp32)
    gret_bytes = 3 * B * N * H * D * 2 + B * N * H * D * 2 + B * N * H * 4 + 2 * B * H * D * D * 4
    achieved = gret_bytes / (gret_ms / 1e3) / 1e9
    roofline = {"bound": "hbm", "kernel": "yoco_gret_prefill_chunkwise (one 524288 x 24 x 128 layer: all of its "
                "launches; average over the 13 back-to-back calls of each timed step)",
                "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s", "frac": round(achieved / hbm_peak, 4),
                "peak_source": ("MEASURED_PEAKS.json hbm_gbs (burst copy; of measured)" if "hbm_gbs" in peaks
                                else "fallback 6.8 TB/s (of fallback)"),
                "algorithmic_bytes_per_launch": gret_bytes, "avg_launch_ms": round(gret_ms, 4),
                "traffic": GRET_CALL_DRAM_BYTES,
                "traffic_unit": "bytes per call (ncu dram read + write, both launches)"}
    # the same call against the tensor cores, on the algorithmic flops at the method's
    # chunk of 64: per token and head the causal half of the chunk's QK^T and PV,
    # 2 d (C + 1), plus the cross-chunk q S and the state update, 4 d^2
    gret_flops = B * N * H * (2 * D * (64 + 1) + 4 * D * D)
    kernel_flops = B * N * H * (2 * D * (128 + 1) + 4 * D * D)  # what the kernel issues at its 128-token chunks
    tc_peak = peaks.get("bf16_tflops_sustained", peaks.get("bf16_tflops", 1700.0)) * 1e12  # inside a long step
    tflops = gret_flops / (gret_ms / 1e3)
    attainable = min(tc_peak, gret_flops / gret_bytes * hbm_peak * 1e9)
    roofline.update({"flops_per_launch": gret_flops, "flops_chunk": 64,
                     "tc_achieved_tflops": round(tflops / 1e12, 1), "tc_peak_tflops": round(tc_peak / 1e12, 1),
                     "tc_frac": round(tflops / tc_peak, 4),
                     "tc_peak_source": ("MEASURED_PEAKS.json bf16_tflops_sustained (of measured)"
                                        if "bf16_tflops_sustained" in peaks else "fallback"),
                     "kernel_flops_per_launch_chunk128": kernel_flops,
                     "kernel_tc_frac_chunk128": round(kernel_flops / (gret_ms / 1e3) / tc_peak, 4),
                     "arithmetic_intensity": round(gret_flops / gret_bytes, 1),
                     "attainable_frac": round(tflops / attainable, 4)})
    proj_flops = 2.0 * N * DM * 2 * HKV * D
    cross_bytes = N * HKV * D * 2 * 2
    roof_step_ms = (L_SELF * gret_bytes / (hbm_peak * 1e9) + proj_flops / (peaks.get("bf16_tflops", 1900.0) * 1e12)
                    + L_CROSS * cross_bytes / (hbm_peak * 1e9)) * 1e3

    # ---- end to end: inputs from pinned host memory, results back to host
    barrier()
    e2e = e2e_measure(args, torch, stream, step, q, k, v, lg, [M] + Qx, Ox)
    if e2e is not None:  # whole job: every rank's prompts over the slowest rank's time
        e2e_s = e2e["ms_per_step"] / 1e3 * e2e["steps"]
        e2e["value"], e2e_s = aggregate_over_ranks(e2e_s, B * N * e2e["steps"], dist, dev)
        e2e["ms_per_step"] = e2e_s / e2e["steps"] * 1e3
    del q, k, v, lg, M, o
    torch.cuda.empty_cache()

    # ---- generation at a 1M-token context
    barrier()
    decode = decode_1m(args, torch, Y, dev, seed, hbm_peak)
    if decode is not None:  # whole job: every rank's generated tokens over the slowest rank's time
        dec_s = decode["ms_per_token"] / 1e3 * decode["tokens"]
        dec_value, dec_s = aggregate_over_ranks(dec_s, decode["tokens"], dist, dev)
        decode["value"] = round(dec_value, 2)
        decode["ms_per_token"] = round(dec_s / decode["tokens"] * 1e3, 4)

    clocks = clk.summary(t_lo - 0.1, t_hi + 0.1)
    clocks["window_ms"] = round((t_hi - t_lo) * 1e3, 1)
    out = {"metric": METRIC, "value": value, "unit": "tok/s", "n_gpus": world, "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
           "config": workload_config(args.chunk if args.chunk else "auto"),
           "roofline": roofline, "step_roofline_ms": round(roof_step_ms, 3),
           "step_frac_of_roofline": round(roof_step_ms / ms_step, 4), "e2e": e2e,
           "gpu_launches": int(launches_per_step * args.steps), "gpu_launches_per_step": int(launches_per_step),
           "clocks": clocks, "phases_ms": phases, "decode": decode}
    if rank == 0 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline_block()
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(out), flush=True)


def e2e_measure(args, torch, stream, step, q, k, v, lg, rest, results):
    """The step with a host->device copy of its inputs and a device->host read of
    its results inside the timed region.  Host memory holds one gRet layer's q, k,
    v and logits (pinned, 9.7 GB) and every layer's device inputs are copied from
    it, so the bytes copied per step are the step's whole input (129 GB) without
    holding 13 layers on the host.  The copies run on a second stream in the order
    the step uses them and each layer's call waits for its own inputs only, so
    later layers' copies overlap earlier layers' compute."""
    if args.e2e_steps <= 0:
        return None
    host_layer = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in (q[0], k[0], v[0], lg[0])]
    for h, t in zip(host_layer, (q[0], k[0], v[0], lg[0])):
        h.copy_(t)
    host_rest = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in rest]
    for h, t in zip(host_rest, rest):
        h.copy_(t)
    res_host = [torch.empty(r.shape, dtype=r.dtype, pin_memory=True) for r in results]
    per_layer = [(q[l], k[l], v[l], lg[l]) for l in range(len(q))]
    h2d = (sum(t.numel() * t.element_size() for grp in per_layer for t in grp)
           + sum(t.numel() * t.element_size() for t in rest))
    d2h = sum(r.numel() * r.element_size() for r in results)
    copy_stream = torch.cuda.Stream()
    ev_layer = [torch.cuda.Event() for _ in per_layer]
    ev_rest = torch.cuda.Event()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.e2e_steps):
        copy_stream.wait_stream(stream)  # the previous step has finished reading its inputs
        with torch.cuda.stream(copy_stream):
            for grp, ev in zip(per_layer, ev_layer):
                for t, h in zip(grp, host_layer):
                    t.copy_(h, non_blocking=True)
                ev.record(copy_stream)
            for t, h in zip(rest, host_rest):
                t.copy_(h, non_blocking=True)
            ev_rest.record(copy_stream)
        step(wait_layer=lambda l: stream.wait_event(ev_layer[l]), wait_rest=lambda: stream.wait_event(ev_rest))
        for h, r in zip(res_host, results):
            h.copy_(r, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    t = e0.elapsed_time(e1) / 1e3 / args.e2e_steps
    return {"value": B * N / t, "unit": "tok/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "steps": args.e2e_steps, "ms_per_step": t * 1e3,
            "h2d": ("pinned host memory (one gRet layer's q, k, v, logits copied into every layer's device "
                    "inputs, plus M and the cross queries), one copy per tensor on a second stream, layer by "
                    "layer ahead of use"),
            "d2h": "the 13 cross layers' last-row outputs"}


def decode_1m(args, torch, Y, dev, seed, hbm_peak):
    """Generated tokens at a 1M-token context, B = 1: per token 13 recurrent gRet
    steps (captured once as a CUDA graph and replayed), a one-slot append of the
    new token's K^/V^, and 13 split-KV cross layers over the whole cache.  The
    cache (4.3 GB) is far larger than L2, so every layer's read comes from HBM."""
    if args.decode_tokens <= 0:
        return None
    import synth
    L = Y.lib
    bf, f32 = torch.bfloat16, torch.float32
    sid = synth.stream_id
    stream = torch.cuda.current_stream(dev)
    stp = ctypes.c_void_p(stream.cuda_stream)
    P = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731

    def normal(shape, dtype, stream_tag, mean=0.0, std=1.0):
        return synth.fill_normal_(torch.empty(shape, dtype=dtype, device=dev), seed, stream_tag, mean, std)

    def check(st, what):
        if st != 0:
            raise RuntimeError(f"{what}: {L.yoco_last_error().decode()}")

    extra = args.warmup + args.decode_tokens + 1
    Kc = normal((1, HKV, N_DEC + extra, D), bf, sid(CFG_DEC, 0, synth.T_CACHE_K))
    Vc = normal((1, HKV, N_DEC + extra, D), bf, sid(CFG_DEC, 0, synth.T_CACHE_V))
    cache = Y.KVCache(1, HKV, D, N_DEC + extra, k=Kc, v=Vc)
    cache.set_length(N_DEC)
    cc = ctypes.byref(cache.c)
    Wk = normal((DM, HKV * D), bf, sid(CFG_DEC, 0, synth.T_WK), std=0.02)
    Wv = normal((DM, HKV * D), bf, sid(CFG_DEC, 0, synth.T_WV), std=0.02)
    M1 = normal((1, 1, DM), bf, sid(CFG_DEC, 0, synth.T_M, 1))
    Qd = [normal((1, HQ, D), bf, sid(CFG_DEC, l, synth.T_QX, 1)) for l in range(L_CROSS)]
    Od = [torch.empty(1, HQ, D, dtype=bf, device=dev) for _ in range(L_CROSS)]
    q1 = [normal((1, H, D), bf, sid(CFG_DEC, l, synth.T_Q, 1), std=D ** -0.5) for l in range(L_SELF)]
    k1 = [normal((1, H, D), bf, sid(CFG_DEC, l, synth.T_K, 1), std=D ** -0.5) for l in range(L_SELF)]
    v1 = [normal((1, H, D), bf, sid(CFG_DEC, l, synth.T_V, 1)) for l in range(L_SELF)]
    lg1 = [normal((1, H), f32, sid(CFG_DEC, l, synth.T_LOGIT, 1), mean=2.0) for l in range(L_SELF)]
    S1 = [normal((1, H, D, D), f32, sid(CFG_DEC, l, synth.T_S0), std=0.05) for l in range(L_SELF)]
    o1 = [torch.empty(1, H, D, dtype=bf, device=dev) for _ in range(L_SELF)]
    ws = torch.empty(max(L.yoco_shared_kv_workspace_size(1, 1, DM, cc),
                         L.yoco_cross_attn_workspace_size(1, HQ, 1, cc, 0), 256), dtype=torch.uint8, device=dev)
    wsp, wsn = P(ws), ws.numel()

    def gret_layers(sp):
        for l in range(L_SELF):
            check(L.yoco_gret_decode_step(P(q1[l]), P(k1[l]), P(v1[l]), P(lg1[l]), TAU, P(S1[l]), P(o1[l]), 1, H, D,
                                          D, 1, 1, sp), "gret decode")

    gret_layers(stp)
    torch.cuda.synchronize()
    cap = torch.cuda.Stream(dev)
    cap.wait_stream(stream)
    graph = torch.cuda.CUDAGraph()
    n0 = L.yoco_launch_count()
    with torch.cuda.graph(graph, stream=cap):
        gret_layers(ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream))
    graph_launches = L.yoco_launch_count() - n0
    stream.wait_stream(cap)
    torch.cuda.synchronize()

    def token(ev=None):
        graph.replay()  # the 13 recurrent gRet steps
        check(L.yoco_shared_kv_project_append(P(M1), None, EPS, P(Wk), P(Wv), 1, DM, cc, wsp, wsn, stp), "append")
        if ev is not None:
            ev[0].record(stream)
        for l in range(L_CROSS):
            check(L.yoco_cross_attn_decode(P(Qd[l]), HQ, cc, D ** -0.5, 0, P(Od[l]), wsp, wsn, stp), "cross decode")
        if ev is not None:
            ev[1].record(stream)

    for _ in range(args.warmup):
        token()
    torch.cuda.synchronize()
    len0 = cache.length
    n0 = L.yoco_launch_count()
    cross_ev = [[torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)]
                for _ in range(args.decode_tokens)]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(args.decode_tokens):
        token(cross_ev[i])
    e1.record(stream)
    torch.cuda.synchronize()
    launches = L.yoco_launch_count() - n0 + graph_launches * args.decode_tokens
    ms = e0.elapsed_time(e1) / args.decode_tokens
    cross_ms = statistics.mean(c[0].elapsed_time(c[1]) / L_CROSS for c in cross_ev)
    ctx = len0 + (args.decode_tokens + 1) / 2  # mean cache length the timed tokens read
    key_bytes = HKV * D * 2 * 2  # K^ and V^ of one position
    tok_bytes = L_CROSS * ctx * key_bytes + 2 * DM * HKV * D * 2 + L_SELF * H * D * D * 4 * 2
    cross_bytes = ctx * key_bytes
    out = {"value": round(1e3 / ms, 2), "unit": "tok/s", "context": N_DEC, "B": 1, "ms_per_token": round(ms, 4),
           "tokens": args.decode_tokens, "gpu_launches_per_token": round(launches / args.decode_tokens, 1),
           "roofline": {"bound": "hbm", "achieved": round(tok_bytes / (ms / 1e3) / 1e9, 1), "peak": hbm_peak,
                        "unit": "GB/s", "frac": round(tok_bytes / (ms / 1e3) / 1e9 / hbm_peak, 4),
                        "algorithmic_bytes_per_token": int(tok_bytes),
                        "note": ("13 cross layers each read the whole shared cache (4.3 GB, far above the "
                                 "129 MB L2, so these bytes come from HBM), the projection weights and the 13 "
                                 "layers' fp32 states in and out")},
           "roofline_cross_decode": {"bound": "hbm", "kernel": "yoco_cross_attn_decode (split + combine)",
                                     "achieved": round(cross_bytes / (cross_ms / 1e3) / 1e9, 1), "peak": hbm_peak,
                                     "unit": "GB/s", "frac": round(cross_bytes / (cross_ms / 1e3) / 1e9 / hbm_peak, 4),
                                     "algorithmic_bytes_per_launch": int(cross_bytes),
                                     "avg_launch_ms": round(cross_ms, 4)}}
    del Kc, Vc, cache
    torch.cuda.empty_cache()
    return out


def run_only(args):
    """One call kind of the step, on its bench shape, for kernel profiling."""
    import torch

    import gated_retention_shared_gb300 as Y
    import synth
    L = Y.lib
    dev = torch.device("cuda", 0)
    sid = synth.stream_id
    bf, f32 = torch.bfloat16, torch.float32

    def normal(shape, dtype, stream, mean=0.0, std=1.0):
        return synth.fill_normal_(torch.empty(shape, dtype=dtype, device=dev), SEED, stream, mean, std)

    P = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    stp = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    N = args.n or N_LAYER      # tokens of the call's shape (the single 32K-token gRet layer by default)
    if args.segments:
        assert L.yoco_test_hook(3, args.segments) == 0, L.yoco_last_error()
    CFG = CFG_LAYER if N == N_LAYER else 4
    if args.only in ("gret", "gret_gn", "gret_gn_unfused"):
        q = normal((B, N, H, D), bf, sid(CFG, 0, synth.T_Q), std=D ** -0.5)
        k = normal((B, N, H, D), bf, sid(CFG, 0, synth.T_K), std=D ** -0.5)
        v = normal((B, N, H, D), bf, sid(CFG, 0, synth.T_V))
        lg = normal((B, N, H), f32, sid(CFG, 0, synth.T_LOGIT), mean=2.0)
        if args.no_decay:
            lg.fill_(float("inf"))
        o = torch.empty_like(v)
        S = torch.zeros(B, H, D, D, dtype=f32, device=dev)
        ws = torch.empty(max(256, L.yoco_gret_prefill_workspace_size(B, N, H, D, D, args.chunk, 1)), dtype=torch.uint8,
                         device=dev)

        g = normal((B, N, H, D), bf, sid(CFG, 0, synth.T_QX)) if args.only != "gret" else None
        z = torch.empty_like(v) if args.only != "gret" else None

        if args.only == "gret":
            def call():
                S.zero_()
                return L.yoco_gret_prefill_chunkwise(P(q), P(k), P(v), P(lg), TAU, P(o), P(S), B, N, H, D, D,
                                                     args.chunk, 1, 1, P(ws), ws.numel(), stp)
        elif args.only == "gret_gn":  # with Eq. 7's GroupNorm and swish gate fused
            def call():
                S.zero_()
                return L.yoco_gret_prefill_chunkwise_gn_gate(P(q), P(k), P(v), P(lg), TAU, P(g), None, None, 1e-5,
                                                             P(z), P(S), B, N, H, D, D, 1, P(ws), ws.numel(), stp)
        else:  # the prefill, then the separate GroupNorm + gate pass
            def call():
                S.zero_()
                st_ = L.yoco_gret_prefill_chunkwise(P(q), P(k), P(v), P(lg), TAU, P(o), P(S), B, N, H, D, D,
                                                    args.chunk, 1, 1, P(ws), ws.numel(), stp)
                return st_ or L.yoco_gret_group_norm_gate(P(o), P(g), None, None, 1e-5, P(z), B, N, H, D, 1, stp)
    elif args.only == "append":  # one generated token's K/V slot into a cache holding the prompt
        M1 = normal((B, 1, DM), bf, sid(CFG, 0, synth.T_M, 1))
        Wk = normal((DM, HKV * D), bf, sid(CFG, 0, synth.T_WK), std=0.02)
        Wv = normal((DM, HKV * D), bf, sid(CFG, 0, synth.T_WV), std=0.02)
        # every call appends one more slot (no length reset, so no host write inside the timed loop)
        cache = Y.KVCache(B, HKV, D, N + args.warmup + args.steps, device=dev)
        cache.set_length(N)
        ws = torch.empty(max(256, L.yoco_shared_kv_workspace_size(B, 1, DM, ctypes.byref(cache.c))),
                         dtype=torch.uint8, device=dev)

        def call():
            return L.yoco_shared_kv_project_append(P(M1), None, EPS, P(Wk), P(Wv), 1, DM, ctypes.byref(cache.c),
                                                   P(ws), ws.numel(), stp)
    elif args.only == "cross_prefill":  # every prompt row over the shared cache (no early exit)
        Tq = args.cache_len or N
        Kc = normal((B, HKV, Tq, D), bf, sid(CFG, 0, synth.T_CACHE_K))
        Vc = normal((B, HKV, Tq, D), bf, sid(CFG, 0, synth.T_CACHE_V))
        cache = Y.KVCache(B, HKV, D, Tq, k=Kc, v=Vc, rope_base=args.rope_base)
        cache.set_length(Tq)
        Qp = normal((B, Tq, HQ, D), bf, sid(CFG, 0, synth.T_QX))
        Op = torch.empty_like(Qp)
        ws = torch.empty(max(256, L.yoco_cross_attn_workspace_size(B, HQ, Tq, ctypes.byref(cache.c), 0)),
                         dtype=torch.uint8, device=dev)

        def call():
            return L.yoco_cross_attn_prefill(P(Qp), HQ, Tq, 0, ctypes.byref(cache.c), D ** -0.5, P(Op), P(ws),
                                             ws.numel(), stp)
    elif args.only in ("swa_prefill", "swa_decode"):
        # a sliding-window self-decoder layer of the 3B shape: 24 heads x 128, window 1024
        Ns = args.cache_len or N
        W = 1024
        qs = normal((B, Ns, H, D), bf, sid(CFG, 0, synth.T_Q))
        ks = normal((B, Ns, H, D), bf, sid(CFG, 0, synth.T_K))
        vs = normal((B, Ns, H, D), bf, sid(CFG, 0, synth.T_V))
        os_ = torch.empty_like(qs)
        ring = Y.SwaRing(B, H, D, W, device=dev)
        ws = torch.empty(max(256, L.yoco_swa_workspace_size(B, H, ctypes.byref(ring.c))), dtype=torch.uint8,
                         device=dev)
        q1s, k1s, v1s = qs[:, 0].contiguous(), ks[:, 0].contiguous(), vs[:, 0].contiguous()
        o1s = torch.empty_like(q1s)

        if args.only == "swa_prefill":
            def call():
                ring.c.pos = 0
                return L.yoco_swa_prefill(P(qs), P(ks), P(vs), H, Ns, D ** -0.5, P(os_), ctypes.byref(ring.c), P(ws),
                                          ws.numel(), stp)
        else:
            ring.c.pos = 0
            assert L.yoco_swa_prefill(P(qs), P(ks), P(vs), H, Ns, D ** -0.5, P(os_), ctypes.byref(ring.c), P(ws),
                                      ws.numel(), stp) == 0

            def call():
                return L.yoco_swa_decode(P(q1s), P(k1s), P(v1s), H, D ** -0.5, P(o1s), ctypes.byref(ring.c), P(ws),
                                         ws.numel(), stp)
    elif args.only == "qkvg":  # a gRet layer's four input projections in one GEMM
        Xg = normal((B, N, DM), bf, sid(CFG, 0, synth.T_M))
        Wg = normal((DM, 3 * H * D + H), bf, sid(CFG, 0, synth.T_WK), std=DM ** -0.5)
        qg = torch.empty(B, N, H, D, dtype=bf, device=dev)
        kg, vg = torch.empty_like(qg), torch.empty_like(qg)
        lgg = torch.empty(B, N, H, dtype=f32, device=dev)
        ws = torch.empty(L.yoco_gret_qkvg_workspace_size(B, N, H, D, args.rope_base), dtype=torch.uint8, device=dev)

        def call():
            return L.yoco_gret_qkvg_project(P(Xg), P(Wg), B, N, DM, H, D, 0, args.rope_base, P(qg), P(kg), P(vg),
                                            P(lgg), P(ws), ws.numel(), stp)
    elif args.only in ("gret_decode_unfused", "gret_decode_gn"):
        # one generated token through a gRet layer's recurrent step and Eq. 7's output:
        # the step then the separate GroupNorm + gate call, or the fused call
        q1 = normal((B, H, D), bf, sid(CFG, 0, synth.T_Q, 1), std=D ** -0.5)
        k1 = normal((B, H, D), bf, sid(CFG, 0, synth.T_K, 1), std=D ** -0.5)
        v1 = normal((B, H, D), bf, sid(CFG, 0, synth.T_V, 1))
        lg1 = normal((B, H), f32, sid(CFG, 0, synth.T_LOGIT, 1), mean=2.0)
        g1 = normal((B, H, D), bf, sid(CFG, 0, synth.T_QX, 1))
        S1 = normal((B, H, D, D), f32, sid(CFG, 0, synth.T_S0), std=0.05)
        o1 = torch.empty(B, H, D, dtype=bf, device=dev)
        z1 = torch.empty_like(o1)

        if args.only == "gret_decode_unfused":
            def call():
                st_ = L.yoco_gret_decode_step(P(q1), P(k1), P(v1), P(lg1), TAU, P(S1), P(o1), B, H, D, D, 1, 1, stp)
                return st_ or L.yoco_gret_group_norm_gate(P(o1), P(g1), None, None, 1e-5, P(z1), B, 1, H, D, 1, stp)
        else:
            def call():
                return L.yoco_gret_decode_step_gn_gate(P(q1), P(k1), P(v1), P(lg1), TAU, P(S1), P(g1), None, None,
                                                       1e-5, P(z1), B, H, D, D, 1, stp)
    elif args.only in ("gret_steps", "gret_steps_append"):
        # a generated token's 13 recurrent gRet steps (one CUDA graph), alone or followed
        # by the one-slot append of its K^/V^: the difference is what the append adds
        # inside a token, where it starts while the steps finish (W is cold in L2 each
        # call: a 200 MB buffer is written between calls, as the cross layers' cache
        # reads would evict it)
        q1 = [normal((B, H, D), bf, sid(CFG, l, synth.T_Q, 1), std=D ** -0.5) for l in range(L_SELF)]
        k1 = [normal((B, H, D), bf, sid(CFG, l, synth.T_K, 1), std=D ** -0.5) for l in range(L_SELF)]
        v1 = [normal((B, H, D), bf, sid(CFG, l, synth.T_V, 1)) for l in range(L_SELF)]
        lg1 = [normal((B, H), f32, sid(CFG, l, synth.T_LOGIT, 1), mean=2.0) for l in range(L_SELF)]
        S1 = [normal((B, H, D, D), f32, sid(CFG, l, synth.T_S0), std=0.05) for l in range(L_SELF)]
        o1 = [torch.empty(B, H, D, dtype=bf, device=dev) for _ in range(L_SELF)]
        M1 = normal((B, 1, DM), bf, sid(CFG, 0, synth.T_M, 1))
        Wk = normal((DM, HKV * D), bf, sid(CFG, 0, synth.T_WK), std=0.02)
        Wv = normal((DM, HKV * D), bf, sid(CFG, 0, synth.T_WV), std=0.02)
        cache = Y.KVCache(B, HKV, D, 16 + args.warmup + args.steps, device=dev)
        wsa = torch.empty(max(256, L.yoco_shared_kv_workspace_size(B, 1, DM, ctypes.byref(cache.c))),
                          dtype=torch.uint8, device=dev)
        flush = torch.empty(200 << 20, dtype=torch.uint8, device=dev)
        sp = torch.cuda.current_stream(dev)

        def steps(st_):
            for l in range(L_SELF):
                assert L.yoco_gret_decode_step(P(q1[l]), P(k1[l]), P(v1[l]), P(lg1[l]), TAU, P(S1[l]), P(o1[l]), B, H,
                                               D, D, 1, 1, st_) == 0
        steps(stp)
        torch.cuda.synchronize()
        cap_s = torch.cuda.Stream(dev)
        cap_s.wait_stream(sp)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=cap_s):
            steps(ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream))
        sp.wait_stream(cap_s)
        torch.cuda.synchronize()
        timed_ms = []

        def call():
            flush.fill_(1)  # evicts W from L2, untimed
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(sp)
            graph.replay()
            st_ = 0
            if args.only == "gret_steps_append":
                st_ = L.yoco_shared_kv_project_append(P(M1), None, EPS, P(Wk), P(Wv), 1, DM, ctypes.byref(cache.c),
                                                      P(wsa), wsa.numel(), stp)
            e1.record(sp)
            timed_ms.append((e0, e1))
            return st_
    elif args.only == "rope":  # rotary encoding of one gRet layer's q in place
        qr = normal((B, N, H, D), bf, sid(CFG, 0, synth.T_Q))

        def call():
            return L.yoco_rope_apply(P(qr), B, N, H, D, 0, args.rope_base or 8e7, 1, stp)
    elif args.only == "gn_gate":  # GroupNorm per head + swish gate over one gRet layer's output
        og = normal((B, N, H, D), bf, sid(CFG, 0, synth.T_V))
        gg = normal((B, N, H, D), bf, sid(CFG, 0, synth.T_Q))
        zg = torch.empty_like(og)

        def call():
            return L.yoco_gret_group_norm_gate(P(og), P(gg), None, None, 1e-5, P(zg), B, N, H, D, 1, stp)
    elif args.only == "proj":
        M = normal((B, N, DM), bf, sid(CFG, 0, synth.T_M))
        Wk = normal((DM, HKV * D), bf, sid(CFG, 0, synth.T_WK), std=0.02)
        Wv = normal((DM, HKV * D), bf, sid(CFG, 0, synth.T_WV), std=0.02)
        cache = Y.KVCache(B, HKV, D, N, device=dev, rope_base=args.rope_base)
        ws = torch.empty(L.yoco_shared_kv_workspace_size(B, N, DM, ctypes.byref(cache.c)), dtype=torch.uint8,
                         device=dev)

        def call():
            cache.len_dev.zero_()
            cache.c.len_host = 0
            return L.yoco_shared_kv_project_append(P(M), None, EPS, P(Wk), P(Wv), N, DM, ctypes.byref(cache.c), P(ws),
                                                   ws.numel(), stp)
    else:
        Bc = args.batch or B
        Nc = args.cache_len or N
        Kc = normal((Bc, HKV, Nc, D), bf, sid(CFG, 0, synth.T_CACHE_K))
        Vc = normal((Bc, HKV, Nc, D), bf, sid(CFG, 0, synth.T_CACHE_V))
        cache = Y.KVCache(Bc, HKV, D, Nc, k=Kc, v=Vc, rope_base=args.rope_base)
        cache.set_length(Nc)
        Qd = normal((Bc, HQ, D), bf, sid(CFG, 0, synth.T_QX, 1))
        Od = torch.empty_like(Qd)
        ws = torch.empty(max(256, L.yoco_cross_attn_workspace_size(Bc, HQ, 1, ctypes.byref(cache.c), args.splits)),
                         dtype=torch.uint8, device=dev)

        def call():
            return L.yoco_cross_attn_decode(P(Qd), HQ, ctypes.byref(cache.c), D ** -0.5, args.splits, P(Od), P(ws),
                                            ws.numel(), stp)
    for _ in range(args.warmup):
        assert call() == 0, L.yoco_last_error()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        assert call() == 0, L.yoco_last_error()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / args.steps
    if args.only in ("gret_steps", "gret_steps_append"):  # events around each call only (the flush is untimed)
        ms = statistics.mean(a.elapsed_time(b) for a, b in timed_ms[args.warmup:])
    line = {"only": args.only, "ms_per_call": ms, "steps": args.steps, "N": N}
    if args.only in ("gret", "gret_gn"):
        # the fused call also reads the gate (bf16, the size of q)
        nbytes = (4 + (args.only == "gret_gn")) * B * N * H * D * 2 + B * N * H * 4 + 2 * B * H * D * D * 4
        line.update({"bytes_per_call": nbytes, "achieved_gbs": round(nbytes / (ms / 1e3) / 1e9, 1),
                     "no_decay": bool(args.no_decay), "segments": args.segments or "auto"})
    if args.only == "qkvg":
        flops = 2.0 * B * N * DM * (3 * H * D + H)
        line.update({"flops_per_call": flops, "achieved_tflops": round(flops / (ms / 1e3) / 1e12, 1)})
    if args.only == "rope":
        nbytes = 2 * B * N * H * D * 2  # read and written once
        line.update({"bytes_per_call": nbytes, "achieved_gbs": round(nbytes / (ms / 1e3) / 1e9, 1)})
    if args.only == "gn_gate":
        nbytes = 3 * B * N * H * D * 2  # o and gate read, z written
        line.update({"bytes_per_call": nbytes, "achieved_gbs": round(nbytes / (ms / 1e3) / 1e9, 1)})
    if args.only == "swa_prefill":
        # row n sees min(n + 1, 1024) keys; QK^T and PV cost 2 d flops per (row, key, head) each
        seen = sum(min(n + 1, 1024) for n in range(Ns))
        flops = 4.0 * D * H * B * seen
        line.update({"rows": Ns, "window": 1024, "flops_per_call": flops,
                     "achieved_tflops": round(flops / (ms / 1e3) / 1e12, 1)})
    if args.only == "swa_decode":
        nbytes = 2 * B * H * 1024 * D * 2  # the full ring read once (after the prefill it is full)
        line.update({"window": 1024, "bytes_per_call": nbytes, "achieved_gbs": round(nbytes / (ms / 1e3) / 1e9, 1)})
    if args.only == "cross_prefill":
        # causal: row t reads t + 1 keys; QK^T and PV cost 2 d flops per (row, key, head) each
        flops = 4.0 * D * HQ * B * Tq * (Tq + 1) / 2
        line.update({"rows": Tq, "flops_per_call": flops, "achieved_tflops": round(flops / (ms / 1e3) / 1e12, 1)})
    if args.only == "cross_decode":
        # every K/V byte of every sequence is read once per call
        nbytes = 2 * Bc * HKV * Nc * D * 2
        line.update({"B": Bc, "cache_len": Nc, "bytes_per_call": nbytes,
                     "achieved_gbs": round(nbytes / (ms / 1e3) / 1e9, 1)})
    print(json.dumps(line))


# ------------------------------------------------- long-context workloads

LONG_WORKLOADS = {
    # 13 cross layers per generated token over a 128K-token shared cache, one
    # append per token, B sequences with their own caches
    "decode128k": 3,
    # 1M-token context: 13 recurrent gRet steps, one append, 13 cross layers per token
    "decode1m": 5,
}


def run_workload(args):
    """Time a long-context workload; prints one JSON line per workload (and batch).

    Roofline time of a step: the bytes every memory-bound call must move at the
    measured HBM copy rate plus the projection's flops at the measured bf16 rate;
    `frac_of_roofline` = that time / the measured step time."""
    import torch

    import gated_retention_shared_gb300 as Y
    import synth
    L = Y.lib
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    bf, f32 = torch.bfloat16, torch.float32
    sid = synth.stream_id
    cfg = LONG_WORKLOADS[args.workload]
    P = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    stream = torch.cuda.current_stream(dev)
    stp = ctypes.c_void_p(stream.cuda_stream)
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peaks = json.load(f)
    except OSError:
        peaks = {}
    hbm = peaks.get("hbm_gbs", 6800.0) * 1e9

    def normal(shape, dtype, stream_tag, mean=0.0, std=1.0):
        return synth.fill_normal_(torch.empty(shape, dtype=dtype, device=dev), SEED, stream_tag, mean, std)

    def check(st, what):
        if st != 0:
            raise RuntimeError(f"{what}: {L.yoco_last_error().decode()}")

    def timed(step, steps, warmup):
        for _ in range(warmup):
            step()
        torch.cuda.synchronize()
        clk = Clocks(0).__enter__()
        clk.wait_first()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t_lo = time.monotonic()
        e0.record(stream)
        for _ in range(steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
        t_hi = time.monotonic()
        time.sleep(0.12)
        clk.__exit__(None, None, None)
        c = clk.summary(t_lo - 0.1, t_hi + 0.1)
        c["window_ms"] = round((t_hi - t_lo) * 1e3, 1)
        return e0.elapsed_time(e1) / steps, c

    lines = []
    cache_bytes_per_key = HKV * D * 2 * 2  # K^ and V^ of one position, bf16
    one_m = args.workload == "decode1m"
    Nc = 1048576 if one_m else 131072
    extra = 256 if one_m else 1024
    batches = [1] if one_m else [int(x) for x in args.batches.split(",")]
    assert args.warmup + args.steps <= extra, "the cache holds the prompt plus this many generated tokens"
    Wk = normal((DM, HKV * D), bf, sid(cfg, 0, synth.T_WK), std=0.02)
    Wv = normal((DM, HKV * D), bf, sid(cfg, 0, synth.T_WV), std=0.02)
    for Bc in batches:
        Kc = normal((Bc, HKV, Nc + extra, D), bf, sid(cfg, 0, synth.T_CACHE_K))
        Vc = normal((Bc, HKV, Nc + extra, D), bf, sid(cfg, 0, synth.T_CACHE_V))
        cache = Y.KVCache(Bc, HKV, D, Nc + extra, k=Kc, v=Vc)
        cache.set_length(Nc)
        cc = ctypes.byref(cache.c)
        M1 = normal((Bc, 1, DM), bf, sid(cfg, 0, synth.T_M, 1))
        Qd = [normal((Bc, HQ, D), bf, sid(cfg, l, synth.T_QX, 1)) for l in range(L_CROSS)]
        Od = [torch.empty(Bc, HQ, D, dtype=bf, device=dev) for _ in range(L_CROSS)]
        ws = torch.empty(max(L.yoco_shared_kv_workspace_size(Bc, 1, DM, cc),
                             L.yoco_cross_attn_workspace_size(Bc, HQ, 1, cc, 0), 256), dtype=torch.uint8,
                         device=dev)
        wsp, wsn = P(ws), ws.numel()
        graph = None
        if one_m:
            q1 = [normal((Bc, H, D), bf, sid(cfg, l, synth.T_Q, 1), std=D ** -0.5) for l in range(L_SELF)]
            k1 = [normal((Bc, H, D), bf, sid(cfg, l, synth.T_K, 1), std=D ** -0.5) for l in range(L_SELF)]
            v1 = [normal((Bc, H, D), bf, sid(cfg, l, synth.T_V, 1)) for l in range(L_SELF)]
            lg1 = [normal((Bc, H), f32, sid(cfg, l, synth.T_LOGIT, 1), mean=2.0) for l in range(L_SELF)]
            S1 = [normal((Bc, H, D, D), f32, sid(cfg, l, synth.T_S0), std=0.05) for l in range(L_SELF)]
            o1 = [torch.empty(Bc, H, D, dtype=bf, device=dev) for _ in range(L_SELF)]

            def gret_layers(sp):
                for l in range(L_SELF):
                    check(L.yoco_gret_decode_step(P(q1[l]), P(k1[l]), P(v1[l]), P(lg1[l]), TAU, P(S1[l]),
                                                  P(o1[l]), Bc, H, D, D, 1, 1, sp), "gret decode")
            gret_layers(stp)
            torch.cuda.synchronize()
            cap = torch.cuda.Stream(dev)
            cap.wait_stream(stream)
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=cap):
                gret_layers(ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream))
            stream.wait_stream(cap)
            torch.cuda.synchronize()

        def step():
            if graph is not None:
                graph.replay()  # the 13 recurrent gRet steps
            check(L.yoco_shared_kv_project_append(P(M1), None, EPS, P(Wk), P(Wv), 1, DM, cc, wsp, wsn, stp),
                  "append")
            for l in range(L_CROSS):
                check(L.yoco_cross_attn_decode(P(Qd[l]), HQ, cc, D ** -0.5, 0, P(Od[l]), wsp, wsn, stp),
                      "cross decode")

        ms, clocks = timed(step, args.steps, args.warmup)
        ctx = Nc + args.warmup + args.steps / 2  # mean cache length over the timed tokens
        step_bytes = L_CROSS * Bc * ctx * cache_bytes_per_key + 2 * DM * HKV * D * 2
        if one_m:
            step_bytes += L_SELF * Bc * H * D * D * 4 * 2
        roof_ms = step_bytes / hbm * 1e3
        lines.append({
            "workload": ("yoco3b_decode1m" if one_m else f"shared_kv_decode128k_b{Bc}"),
            "metric": "generated tok/s", "value": Bc / (ms / 1e3), "unit": "tok/s", "ms_per_step": ms,
            "steps": args.steps, "warmup": args.warmup, "dtype": "bf16", "data": "synthetic",
            "config": {"B": Bc, "context": Nc, "cross_layers": L_CROSS, "Hq": HQ, "Hkv": HKV, "d": D,
                       "self_layers": L_SELF if one_m else 0},
            "roofline": {"bound": "hbm", "achieved": round(step_bytes / (ms / 1e3) / 1e9, 1),
                         "peak": hbm / 1e9, "unit": "GB/s", "frac": round(step_bytes / (ms / 1e3) / hbm, 4),
                         "algorithmic_bytes_per_step": int(step_bytes)},
            "roofline_ms": round(roof_ms, 4), "frac_of_roofline": round(roof_ms / ms, 4), "clocks": clocks})
        del Kc, Vc, cache
        torch.cuda.empty_cache()
    for line in lines:
        print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.workload:
        run_workload(args)
    elif args.only:
        run_only(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
