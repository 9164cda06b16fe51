#!/usr/bin/env python
"""Benchmark: GPU-resident tree-speculative greedy decoding of a Llama-3-8B-shaped
int4-g32 / int8-activation decoder on one GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload llama3-8b-ctx4096|qwen05b-ctx512|tiny] [--no-extras]

One step = one generation of `max_new` tokens (256) from a prefilled 4096-token
motif-repeated context: W-step CUDA-graph windows, two in flight, the device-timed width
controller choosing N in {1, 4, 8, 16} between windows (every row of the hot path:
embedding, RMSNorm+quant, W4A8 matmuls, RoPE/KV, tree attention, SwiGLU+quant, LM head,
argmax, acceptance, KV compaction, n-gram drafting, windows, controller).  `value` is
accepted tokens per second with the context resident in HBM (device events around the
window loop; the prefill runs untimed before each step).  `e2e` times the public
end-to-end call (w4a8_decode: prompt copied from pinned host memory, prefill, windows,
tokens read back) on the host clock.  For N > 1 (torchrun) every rank runs an independent
replica (the method is a single sequence: replicas only) and rank 0 reports the aggregate.

Extra keys of the same line (rank 0; skipped with --no-extras): the standalone W4A8 matmul
sweep over the token counts and shapes of the matmul workload, the Qwen2.5-0.5B-shaped
workload (verification step cost per width, the window-size sweep, decode modes), and the
window test on the 8B-shaped model (a 2048-token prompt, W in {1, 4, 16}, host syncs).

`--impl reference` times the CPU oracle (the test oracle under oracle/) on bounded samples
and prints the same JSON line with "impl": "reference".
"""
from __future__ import annotations

import argparse
import json
import os
import platform
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

MAX_NEW = 256
WIDTHS = [1, 4, 8, 16]
METRIC = "accepted tokens/s (GPU-resident tree-speculative greedy decoding)"

WORKLOADS = {
    # name: (shape name, prompt tokens, motifs, motif length, substitution prob, seed)
    "llama3-8b-ctx4096": ("llama3-8b-shaped", 4096, 4, 16, 0.10, 1004),
    "qwen05b-ctx512": ("qwen2.5-0.5b-shaped", 512, 4, 16, 0.10, 1003),
    "tiny": ("tiny-2L-256h", 64, 4, 16, 0.10, 1001),
}
# the window test: 8B-shaped model, 2048 tokens of 8 motifs of 32 tokens, 30% substitutions
WINDOW_TEST = ("llama3-8b-shaped", 2048, 8, 32, 0.30, 1005)
MATMUL_SHAPES = [(896, 4864), (4864, 896), (4096, 14336), (14336, 4096), (4096, 128256)]
MEM_SUB = 0.30  # replaced fraction of the earlier output held in the window test's session memory
MATMUL_TOKENS = [1, 2, 4, 8, 16]


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="llama3-8b-ctx4096", choices=sorted(WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true", help="skip the extra workloads of the line")
    ap.add_argument("--new-tokens", type=int, default=MAX_NEW,
                    help="tokens generated per step (the workload's figure is %d)" % MAX_NEW)
    ap.add_argument("--matmul", type=int, nargs=3, metavar=("K", "N", "M"),
                    help="time one W4A8 matmul shape through the C ABI instead of the decoding step")
    ap.add_argument("--layers", type=int, default=0,
                    help="decoder layers of the model (0 = the workload's; fewer only for small profiling runs)")
    ap.add_argument("--oracle-worker", choices=["tiny", "sample"], help=argparse.SUPPRESS)
    return ap.parse_args()


# --------------------------------------------------------------------------- clocks

class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons while running."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = str(gpu_index)
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", self.gpu, "--query-gpu=" + self.Q,
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (FileNotFoundError, OSError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# --------------------------------------------------------------------------- model

def build_model(shape, seed):
    import synth
    import synth.cuda as SC
    import w4a8_verify_gb300 as W
    from w4a8_verify_gb300 import models as WM

    def fill(kind, layer, out):
        if kind == W.T_EMBED:
            SC.dense_weight(shape, seed, synth.STREAM_EMBED, shape.vocab, shape.hidden, shape.vocab, shape.hidden, out)
        elif kind == W.T_LM_HEAD:
            SC.dense_weight(shape, seed, synth.STREAM_LM_HEAD, shape.vocab, shape.hidden, shape.vocab, shape.hidden,
                            out)
        else:
            rows, cols, rr, rc = synth.tensor_shape(shape, kind)
            SC.dense_weight(shape, seed, synth.layer_stream(layer, kind), rows, cols, rr, rc, out)

    return WM.build_model(shape.n_layers, shape.hidden, shape.n_heads, shape.n_kv_heads, shape.head_dim, shape.ffn,
                          shape.vocab, shape.tied, fill, shape.rms_eps, shape.rope_base)


def mm_traffic(kernel_src):
    """Per-launch DRAM traffic of the matmul kernel from the committed ncu summary
    (profiles/k_mm_traffic.txt: `kernel_sha256_16:` and `dram_bytes_per_launch_n1:` lines),
    if that summary was taken on the current kernel source (hash match); else None."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "k_mm_traffic.txt")
    try:
        kv = {}
        for ln in open(path):
            if ":" in ln:
                k, v = ln.split(":", 1)
                kv[k.strip()] = v.strip()
        h = hashlib.sha256(open(kernel_src, "rb").read()).hexdigest()[:16]
        if kv.get("kernel_sha256_16") == h:
            return float(kv["dram_bytes_per_launch_n1"])
    except (OSError, ValueError, KeyError):
        pass
    return None


def matmul_bytes(K, N, M):
    """Algorithmic bytes of one W4A8 product: packed weights, fp16 scales, int8 activations
    and their scales, fp32 outputs."""
    return N * K // 2 + N * (K // 32) * 2 + M * K + 4 * M + 4 * M * N


def time_matmul(K, N, M, reps_min=20, trials=5, variant="det"):
    """Device time of one standalone matmul call (activation pass + matmul): a CUDA graph of
    back-to-back calls, weights rotated over copies larger than L2, CUDA events on the launching
    stream, median of the trials.  variant: "det" (w4a8_matmul), "nondet" (w4a8_matmul_nondet,
    slices added with atomics), "per32" (w4a8_matmul_per32, one activation scale per 32 inputs)."""
    import torch
    import w4a8_verify_gb300 as W
    dev = torch.device("cuda")
    call = {"det": W.w4a8_matmul, "nondet": W.w4a8_matmul_nondet, "per32": W.w4a8_matmul_per32}[variant]
    wb, sb = W.w4a8_weight_layout_bytes(N, K)
    copies = max(2, -(-(4 * 135 * 2**20) // (wb + sb)))
    g = torch.Generator(device=dev).manual_seed(7)
    wt = [torch.randint(-2**31, 2**31 - 1, (wb // 4,), dtype=torch.int32, device=dev, generator=g)
          for _ in range(copies)]
    st = [torch.full((sb // 2,), 0x2000, dtype=torch.int16, device=dev) for _ in range(copies)]
    x = torch.randn(M, K, device=dev, generator=g)
    a_q, a_s = W.w4a8_quantize_rows(x, 1 if variant == "per32" else 0)
    ws = torch.zeros(W.w4a8_matmul_workspace_bytes(M, K, N), dtype=torch.uint8, device=dev)
    y = torch.empty(M, N, device=dev)
    s = torch.cuda.Stream()
    reps = max(reps_min, copies)
    times = []
    with torch.cuda.stream(s):
        for i in range(3):
            call(a_q, a_s, wt[i % copies], st[i % copies], N, y=y, workspace=ws)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            for i in range(reps):
                call(a_q, a_s, wt[i % copies], st[i % copies], N, y=y, workspace=ws)
        graph.replay()
        for _ in range(trials):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s)
            graph.replay()
            e1.record(s)
            e1.synchronize()
            times.append(e0.elapsed_time(e1) * 1e3 / reps)
    torch.cuda.synchronize()
    flags = W.w4a8_matmul_check(ws, M, K, N)
    del wt, st, graph
    us = statistics.median(times)
    alg = matmul_bytes(K, N, M)
    return {"K": K, "N": N, "M": M, "us": round(us, 3), "GBs": round(alg / us / 1e3, 1),
            "slices": W.w4a8_matmul_slices(K, N), "flags": flags}


def run_matmul(args):
    K, N, M = args.matmul
    r = time_matmul(K, N, M, reps_min=max(20, args.steps))
    r["includes"] = "activation fragment pass + matmul (2 kernels) per call"
    return r


def aggregate_replicas(local_ms, local_tokens, world, device):
    """Whole-job throughput of `world` independent replicas (one sequence per rank, no data
    exchange): the time is the maximum over ranks of each rank's timed milliseconds, the value
    every rank's tokens over that time.  Returns (max ms, tokens per second)."""
    total_ms = float(local_ms)
    if world > 1:
        import torch
        import torch.distributed as dist
        t = torch.tensor([total_ms], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        total_ms = float(t.item())
        dist.barrier()
    return total_ms, local_tokens * world / (total_ms / 1e3)


def timed_generate(sess, prompt_dev, max_new, stream, **kw):
    """Prefill (untimed), then one generation timed with CUDA events on the launching stream:
    (tokens/s, tokens, report)."""
    import torch
    sess.prefill(prompt_dev, max_new)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    ev0.record(stream)
    toks, rep = sess.generate(max_new, **kw)
    ev1.record(stream)
    ev1.synchronize()
    return len(toks) / (ev0.elapsed_time(ev1) / 1e3), toks, rep


def window_sweep(sess, prompt_dev, stream, widths, t_us, windows, max_new=64, reps=3):
    """Decode time per window size W (median of reps), and the smallest W within 10% of the
    fastest (Feedback Control: the window size is chosen at load time)."""
    res = {}
    for Wn in windows:
        ts = []
        for _ in range(reps):
            v, toks, rep = timed_generate(sess, prompt_dev, max_new, stream, window=Wn, widths=widths, t_us=t_us)
            ts.append(1e3 * len(toks) / v)
        res[Wn] = statistics.median(ts) / max_new
    fastest = min(res.values())
    chosen = min(w for w, t in res.items() if t <= 1.10 * fastest)
    return chosen, {str(w): round(t, 4) for w, t in res.items()}


def decode_modes(sess, prompt_dev, stream, max_new, widths, t_us, window):
    """The decode modes of the pages' comparison on one prompt: greedy with a host read-back
    after every token, the GPU loop at width 1 in windows, and speculation with the controller."""
    out = {}
    for name, kw in (("greedy_host_sync_per_token", dict(window=1, fixed_width=1, in_flight=1)),
                     ("gpu_loop_width1_window8", dict(window=8, fixed_width=1, in_flight=2)),
                     ("spec_controller", dict(window=window, widths=widths, t_us=t_us))):
        try:
            v, toks, rep = timed_generate(sess, prompt_dev, max_new, stream, **kw)
            out[name] = {"tokens_per_s": round(v, 2), "steps": rep.n_steps, "host_syncs": rep.host_syncs,
                         "tau": round(len(toks) / max(1, rep.n_steps), 3)}
        except Exception as exc:  # reported, never fatal to the line
            out[name] = "failed: %s" % exc
    return out


# --------------------------------------------------------------------------- our arm

def run_ours(args, rank, world):
    import torch
    import synth
    import w4a8_verify_gb300 as W

    torch.cuda.set_device(rank % max(1, torch.cuda.device_count()))
    dev = torch.device("cuda")
    shape_name, plen, nmot, mlen, psub, seed = WORKLOADS[args.workload]
    shape = synth.SHAPES[shape_name]
    if args.layers > 0:
        import dataclasses
        shape = dataclasses.replace(shape, name="%s-%dlayer" % (shape.name, args.layers), n_layers=args.layers)
        shape_name = shape.name
    t0 = time.time()
    model = build_model(shape, seed)
    torch.cuda.synchronize()
    t_build = time.time() - t0
    prompt = synth.motif_prompt(seed, plen, nmot, mlen, psub, shape.vocab)
    room = max(MAX_NEW, 64)  # the window-size probe below generates 64 tokens
    kv_cap = plen + room + 32
    ctx_cap = plen + room + 64
    sess = W.Session(model, kv_cap, ctx_cap, max_window=16)
    prompt_dev = torch.from_numpy(prompt).to(dev)
    stream = torch.cuda.current_stream()

    # load-time calibration [Feedback Control]: T(N) per width, then the window size
    sess.prefill(prompt_dev, MAX_NEW)
    t_us = sess.calibrate(WIDTHS, reps=10, trials=5)
    window, _ = window_sweep(sess, prompt_dev, stream, WIDTHS, t_us, (1, 2, 4), reps=1)

    def one_step(timed=False):
        sess.prefill(prompt_dev, MAX_NEW)
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if timed:
            torch.cuda.nvtx.range_push("timed")  # lets a profiler select the timed launches
        ev0.record(stream)
        toks, rep = sess.generate(MAX_NEW, window=window, widths=WIDTHS, t_us=t_us)
        ev1.record(stream)
        ev1.synchronize()
        if timed:
            torch.cuda.nvtx.range_pop()
        return ev0.elapsed_time(ev1), toks, rep

    for _ in range(args.warmup):
        one_step()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    times, reps = [], []
    with ClockSampler(torch.cuda.current_device()) as clk:
        for _ in range(args.steps):
            ms, toks, rep = one_step(timed=True)
            assert len(toks) == MAX_NEW, (len(toks), rep.flags)
            times.append(ms)
            reps.append(rep)
    torch.cuda.synchronize()
    total_ms, value = aggregate_replicas(sum(times), MAX_NEW * args.steps, world, dev)

    # end to end through the public call (host prompt -> tokens on the host)
    prompt_list = prompt.tolist()
    e2e_ms = []
    for i in range(max(1, min(args.steps, 3)) + 1):
        torch.cuda.synchronize()
        a = time.perf_counter()
        toks, rep_e = sess.decode(prompt_list, MAX_NEW, window=window, widths=WIDTHS, t_us=t_us)
        b = time.perf_counter()
        if i > 0:
            e2e_ms.append((b - a) * 1e3)
    e2e_value = MAX_NEW / (statistics.median(e2e_ms) / 1e3)
    d2h = rep_e.n_windows * (32 + window * (12 + 64))
    # one prefill on its own (device events; an NVTX range lets a profiler select its launches)
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.nvtx.range_push("prefill")
    ev0.record(stream)
    sess.prefill(prompt_dev, MAX_NEW)
    ev1.record(stream)
    ev1.synchronize()
    torch.cuda.nvtx.range_pop()
    prefill_ms = ev0.elapsed_time(ev1)
    # time to first token through the public call (prompt upload + prefill + one step + read-back)
    ttft = []
    for _ in range(3):
        torch.cuda.synchronize()
        a = time.perf_counter()
        sess.decode(prompt_list, 1, window=1, fixed_width=1, in_flight=1)
        ttft.append((time.perf_counter() - a) * 1e3)

    # dominant kernel: the W4A8 matmul launches of one verification pass (events over a graph)
    sess.prefill(prompt_dev, MAX_NEW)
    mm = {}
    for N in (1, 8, 16):
        # NVTX ranges "matmul_pass" (1 token) and "matmul_pass_16" let a profiler select launches
        if N in (1, 16):
            torch.cuda.nvtx.range_push("matmul_pass" if N == 1 else "matmul_pass_16")
        us, byts, nl = sess.time_matmuls(N, reps=20)
        if N in (1, 16):
            torch.cuda.nvtx.range_pop()
        mm[N] = (us, byts, nl)
    us1, bytes1, nl = mm[1]
    peaks = {}
    try:
        peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except (OSError, ValueError):
        pass
    peak = float(peaks.get("hbm_gbs", 6800.0))
    achieved = bytes1 / us1 / 1e3
    trf = mm_traffic(os.path.join(ROOT, "w4a8_verify_gb300", "csrc", "matmul.cu"))

    modes = decode_modes(sess, prompt_dev, stream, MAX_NEW, WIDTHS, t_us, window)

    launches = sum(int(r.kernels) for r in reps)  # kernel nodes of the window graphs run while timed
    steps_total = sum(r.n_steps for r in reps)
    wsteps = {w: sum(r.width_steps[w] for r in reps) for w in WIDTHS}
    clocks = clk.summary()
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(total_ms / args.steps, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "int4 weights x int8 activations (exact integer sums), fp32 scales/KV",
        "data": "synthetic: seeded random-init weights N(0,0.02) quantised to int4 g32; motif-repeated prompt",
        "config": {
            "workload": args.workload,
            "model": shape_name,
            "prompt_tokens": plen,
            "new_tokens_per_step": MAX_NEW,
            "widths": WIDTHS,
            "window": window,
            "windows_in_flight": 2,
            "parallelism": "replicas" if world > 1 else "single",
            "l2": "weights %.2f GB %s L2 (129 MB)" % (model.weight_bytes() / 1e9,
                                                      ">>" if model.weight_bytes() > 4 * 129e6 else "vs"),
        },
        "e2e": {"value": round(e2e_value, 2), "unit": "tokens/s", "h2d_bytes_per_step": plen * 4,
                "d2h_bytes_per_step": d2h, "includes": "prompt upload + prefill + decode + token read-back",
                "ttft_ms": round(statistics.median(ttft), 2),
                "prefill_ms": round(prefill_ms, 2), "prefill_tokens_per_s": round((plen - 1) / (prefill_ms / 1e3), 1)},
        "gpu_launches": launches,
        "clocks": clocks,
        "roofline": {
            "bound": "hbm", "kernel": "k_mm (W4A8 matmul, N=1 verification pass)",
            "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "peak_source": "measured (MEASURED_PEAKS.json hbm_gbs)" if peaks else "fallback",
            "traffic": trf,
            "algorithmic_bytes_per_launch": round(bytes1),
            "us_per_launch": round(us1, 3), "launches_per_pass": nl,
            "by_width": {str(N): {"us_per_launch": round(v[0], 3), "GBs": round(v[1] / v[0] / 1e3, 1),
                                  "frac": round(v[1] / v[0] / 1e3 / peak, 4)}
                         for N, v in mm.items()},
        },
        "verify_step_us": {str(w): round(t, 1) for w, t in zip(WIDTHS, t_us)},
        "verify_ratio_8_over_1": round(t_us[2] / t_us[0], 3),
        "decode_modes": modes,
        "tau_tokens_per_step": round(MAX_NEW * args.steps / max(1, steps_total), 3),
        "width_steps": wsteps,
        "host_syncs_per_step": round(sum(r.host_syncs for r in reps) / args.steps, 1),
        "setup_s": round(t_build, 1),
    }
    if rank == 0 and world == 1 and not args.no_extras and args.workload == "llama3-8b-ctx4096" and not args.layers:
        line["extras"] = run_extras(model, torch, stream)
    return line


def run_extras(model8b, torch, stream):
    """The other workloads, each reported beside the headline (not part of `value`)."""
    import synth
    import w4a8_verify_gb300 as W
    out = {}
    dev = torch.device("cuda")
    # matmul workload: every token count and shape, standalone calls through the C ABI
    sweep = []
    for K, N in MATMUL_SHAPES:
        for M in MATMUL_TOKENS:
            try:
                sweep.append(time_matmul(K, N, M))
            except Exception as exc:
                sweep.append({"K": K, "N": N, "M": M, "failed": str(exc)})
    out["matmul_sweep"] = {"unit": "us per call, GB/s algorithmic", "calls": sweep,
                           "includes": "activation fragment pass + matmul (2 kernels) per call"}
    # cost of exactness: the fixed-order (deterministic) product against the variant that adds the
    # K slices with atomics, and the per-32 activation-scale form
    cost = []
    for K, N in MATMUL_SHAPES:
        for M in (1, 16):
            try:
                r = {"K": K, "N": N, "M": M}
                for v in ("det", "nondet", "per32"):
                    r[v + "_us"] = time_matmul(K, N, M, variant=v)["us"]
                r["det_over_nondet"] = round(r["det_us"] / r["nondet_us"], 3)
                r["per32_over_det"] = round(r["per32_us"] / r["det_us"], 3)
                cost.append(r)
            except Exception as exc:
                cost.append({"K": K, "N": N, "M": M, "failed": str(exc)})
    out["exactness_cost"] = {"unit": "us per call", "rows": cost,
                             "note": "nondet: slices combined with float atomics in arrival order"}

    # Qwen2.5-0.5B-shaped workload: 512-token prompt, 256 tokens, widths {1,2,4,8,16}
    sh_name, plen, nmot, mlen, psub, seed = WORKLOADS["qwen05b-ctx512"]
    shape = synth.SHAPES[sh_name]
    m = build_model(shape, seed)
    prompt = synth.motif_prompt(seed, plen, nmot, mlen, psub, shape.vocab)
    pd = torch.from_numpy(prompt).to(dev)
    s = W.Session(m, plen + MAX_NEW + 64, plen + MAX_NEW + 96, max_window=16)
    widths = [1, 2, 4, 8, 16]
    s.prefill(pd, MAX_NEW)
    t_us = s.calibrate(widths, reps=20, trials=5)
    chosen, per_tok = window_sweep(s, pd, stream, widths, t_us, (1, 2, 4, 8, 16), max_new=128, reps=3)
    modes = decode_modes(s, pd, stream, MAX_NEW, widths, t_us, chosen)
    s.prefill(pd, MAX_NEW)
    us1, by1, nl = s.time_matmuls(1, reps=50)
    out["qwen05b-ctx512"] = {
        "model": sh_name, "prompt_tokens": plen, "new_tokens": MAX_NEW,
        "verify_step_us": {str(w): round(t, 1) for w, t in zip(widths, t_us)},
        "verify_ratio_over_1": {str(w): round(t / t_us[0], 3) for w, t in zip(widths, t_us)},
        "window_sweep_ms_per_token": per_tok, "window_chosen": chosen,
        "decode_modes": modes,
        "matmul_pass": {"us_per_launch": round(us1, 3), "GBs": round(by1 / us1 / 1e3, 1), "launches": nl},
    }
    s.close()
    del s, m
    torch.cuda.empty_cache()

    # window test on the 8B-shaped model: 2048 tokens of 32-token motifs, 30% substitutions
    sh_name, plen, nmot, mlen, psub, seed = WINDOW_TEST
    prompt = synth.motif_prompt(seed, plen, nmot, mlen, psub, synth.SHAPES[sh_name].vocab)
    pd = torch.from_numpy(prompt).to(dev)
    new = 512
    s = W.Session(model8b, plen + new + 64, plen + new + 96, max_window=16)
    s.prefill(pd, new)
    t_us = s.calibrate(WIDTHS, reps=10, trials=3)
    runs = {}
    for Wn in (1, 4, 16):
        v, toks, rep = timed_generate(s, pd, new, stream, window=Wn, widths=WIDTHS, t_us=t_us)
        runs[str(Wn)] = {"tokens_per_s": round(v, 2), "steps": rep.n_steps, "windows": rep.n_windows,
                         "host_syncs": rep.host_syncs, "tau": round(len(toks) / max(1, rep.n_steps), 3),
                         "accepted_drafts_per_step": round(rep.accepted_drafts / max(1, rep.n_steps), 3),
                         "width_steps": {str(w): rep.width_steps[w] for w in WIDTHS}}
    # The same test with drafts that can be accepted.  Random-init weights never continue a span
    # of their context, so the drafts come from the session memory instead: it holds this
    # request's own greedy output (an earlier answer) with a fraction MEM_SUB of its tokens
    # replaced by random ones; a draft is accepted up to the next replaced token, so MEM_SUB sets
    # the acceptance.  The output must still be the greedy one.
    import numpy as np
    ref, _ = timed_generate(s, pd, new, stream, window=16, fixed_width=1)[1:]
    rng = np.random.default_rng(seed + 1)
    noisy = np.asarray(ref, dtype=np.int64)
    sub = rng.random(noisy.size) < MEM_SUB
    noisy[sub] = rng.integers(0, synth.SHAPES[sh_name].vocab, size=int(sub.sum()))
    s.close()
    sm = W.Session(model8b, plen + new + 64, plen + new + 96, max_window=16, mem_cap=4096)
    sm.memory_append(noisy.tolist())
    runs_m = {}
    for Wn in (1, 4, 16):
        v, toks, rep = timed_generate(sm, pd, new, stream, window=Wn, widths=WIDTHS, t_us=t_us)
        runs_m[str(Wn)] = {"tokens_per_s": round(v, 2), "steps": rep.n_steps, "windows": rep.n_windows,
                           "host_syncs": rep.host_syncs, "tau": round(len(toks) / max(1, rep.n_steps), 3),
                           "accepted_drafts_per_step": round(rep.accepted_drafts / max(1, rep.n_steps), 3),
                           "width_steps": {str(w): rep.width_steps[w] for w in WIDTHS},
                           "equals_greedy": toks == ref}
    sm.close()
    out["window_test"] = {"model": sh_name, "prompt": "%d tokens, %d motifs x %d, substitution p=%.2f" %
                          (plen, nmot, mlen, psub), "new_tokens": new, "by_window": runs,
                          "with_session_memory": {
                              "memory": "this request's greedy output with %d%% of its tokens replaced" %
                                        round(100 * MEM_SUB), "by_window": runs_m}}
    return out


# --------------------------------------------------------------------------- oracle timing

def cpu_model():
    try:
        out = subprocess.run(["lscpu"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True,
                             timeout=10).stdout
        for ln in out.splitlines():
            if ln.lower().startswith("model name"):
                return "%s (%s)" % (ln.split(":", 1)[1].strip(), platform.machine())
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for ln in open("/proc/cpuinfo"):
            if ln.lower().startswith(("model name", "cpu model")):
                return ln.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.processor() or platform.machine()


def oracle_tiny():
    """The oracle decoding the tiny workload for real: 32 greedy tokens, then 32 speculative
    tokens at width 8, from the 64-token motif prompt."""
    import synth
    from oracle import model as OM
    from oracle import spec as OS
    sh_name, plen, nmot, mlen, psub, seed = WORKLOADS["tiny"]
    ow = OM.build_weights(synth.SHAPES[sh_name], 1000)
    prompt = synth.motif_prompt(seed, plen, nmot, mlen, psub, synth.SHAPES[sh_name].vocab)
    a = time.perf_counter()
    g, _ = OM.greedy_decode(ow, prompt, 32)
    b = time.perf_counter()
    s, st = OS.spec_decode(ow, prompt, 32, 8)
    c = time.perf_counter()
    assert s == g
    return {"greedy_tokens_per_s": round(32 / (b - a), 3), "spec_tokens_per_s": round(32 / (c - b), 3),
            "spec_steps": len(st), "greedy_s": round(b - a, 3), "spec_s": round(c - b, 3)}


def oracle_sample(workload, steps, warmup):
    """Times the CPU oracle on a bounded sample of the workload: one decoding step of one
    decoder layer of the workload's shape (attention over the full prompt-length context)
    plus 1/32 of the LM head rows.  Weights are uniform int4 codes with fp16 scales from the
    seeded generator (the oracle's cost does not depend on the values).  Returns the
    measured sample times and the per-token time scaled to all layers and the full head."""
    import numpy as np
    import synth
    from oracle import model as OM

    shape_name, plen, *_ = WORKLOADS[workload]
    sh = synth.SHAPES[shape_name]
    one = synth.ModelShape(sh.name + "-1layer", 1, sh.hidden, sh.n_heads, sh.n_kv_heads, sh.head_dim, sh.ffn,
                           sh.ffn_real, sh.vocab // 32 // 16 * 16, False)

    def qs(rows, cols, stream):
        q = synth.uniform_codes(7, stream, 0, rows * cols).reshape(rows, cols)
        s = synth.uniform_scales(7, stream + 1, 0, rows * (cols // 32)).reshape(rows, cols // 32)
        return q, s

    layer = {}
    for kind in range(7):
        rows, cols, _, _ = synth.tensor_shape(sh, kind)
        layer[kind] = qs(rows, cols, 10 + 2 * kind)
    emb = qs(one.vocab, sh.hidden, 40)
    w = OM.Weights(one, [layer], emb, emb)
    m = OM.Model(w, plen + 2)
    kv = synth.normal(7, 50, 0, sh.n_kv_heads * plen * sh.head_dim, 1.0).reshape(sh.n_kv_heads, plen, sh.head_dim)
    m.K[0][:, :plen] = kv
    m.V[0][:, :plen] = kv[:, ::-1]
    m.step(3, plen)  # warm the dequantised-weight cache (not timed)
    samples = []
    for i in range(warmup + steps):
        a = time.perf_counter()
        m.forward([3], [plen], [plen], [list(range(plen + 1))])
        if i >= warmup:
            samples.append(time.perf_counter() - a)
    x = np.random.default_rng(0).normal(size=sh.hidden)
    a = time.perf_counter()
    m.linear("lm", w.lm_head, x)
    t_head = time.perf_counter() - a
    t_layer = statistics.median(samples) - t_head
    t_tok = sh.n_layers * t_layer + t_head * (sh.vocab / one.vocab)
    return samples, t_tok


def oracle_worker(kind, workload, steps, warmup):
    """Runs in a child process whose BLAS thread count is set by its environment."""
    if kind == "tiny":
        r = oracle_tiny()
    else:
        samples, t_tok = oracle_sample(workload, steps, warmup)
        r = {"samples_s": [round(x, 4) for x in samples], "t_token_s": t_tok}
    print(json.dumps(r), flush=True)


def run_oracle_child(kind, threads, workload="llama3-8b-ctx4096", steps=2, warmup=1, timeout=600):
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS"):
        env[k] = str(threads)
    env["CUDA_VISIBLE_DEVICES"] = ""
    cmd = [sys.executable, os.path.abspath(__file__), "--oracle-worker", kind, "--workload", workload,
           "--steps", str(steps), "--warmup", str(warmup)]
    r = subprocess.run(cmd, env=env, stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True, timeout=timeout)
    if r.returncode != 0:
        raise RuntimeError("oracle worker failed: %s" % r.stderr[-400:])
    return json.loads(r.stdout.strip().splitlines()[-1])


def cpu_baseline_line(workload):
    cores = len(os.sched_getaffinity(0))
    smp = run_oracle_child("sample", cores, workload, steps=2, warmup=1)
    tiny1 = run_oracle_child("tiny", 1)
    tinyn = run_oracle_child("tiny", cores)
    return {"value": round(1.0 / smp["t_token_s"], 5), "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "cpu": cpu_model(),
            "sample": "timed: %d decoding steps of one full-size decoder layer (attention over the whole "
                      "context) plus 1/32 of the LM head rows (%s s each); value = 1 / (per-token time scaled "
                      "to all layers and the full head)" % (len(smp["samples_s"]), smp["samples_s"]),
            "tiny_decode": {"workload": "tiny (2 layers, hidden 256, 64-token prompt, 32 new tokens)",
                            "threads_1": tiny1, "threads_%d" % cores: tinyn}}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    cores = len(os.sched_getaffinity(0))
    t0 = time.perf_counter()
    smp = run_oracle_child("sample", cores, args.workload, steps=args.steps, warmup=args.warmup,
                           timeout=3000)
    wall = time.perf_counter() - t0
    v = 1.0 / smp["t_token_s"]
    shape_name = WORKLOADS[args.workload][0]
    samples = smp["samples_s"]
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": round(v, 5),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": len(samples),
        "warmup": args.warmup,
        "ms_per_step": round(1e3 * statistics.mean(samples), 1),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "fp64 (oracle)",
        "data": "synthetic",
        "config": {"workload": args.workload, "model": shape_name, "prompt_tokens": WORKLOADS[args.workload][1],
                   "new_tokens_per_step": MAX_NEW, "widths": WIDTHS,
                   "parallelism": "replicas" if world > 1 else "single",
                   "timed_unit": "one sample = one decoding step of one full-size decoder layer (attention over "
                                 "the whole context) + 1/32 of the LM head rows; ms_per_step is per sample",
                   "scaled": "value = 1 / (%d x layer time + 32 x the 1/32-head time) = %.1f s per token"
                             % (synth_layers(shape_name), smp["t_token_s"]),
                   "wall_s": round(wall, 1)},
        "cpu_baseline": {"value": round(v, 5), "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "cpu": cpu_model(),
                         "sample": "%d samples of one layer + 1/32 LM head, scaled to the full model" % len(samples)},
        "e2e": {"value": round(v, 5), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def synth_layers(shape_name):
    import synth
    return synth.SHAPES[shape_name].n_layers


def main():
    global MAX_NEW
    args = parse()
    MAX_NEW = args.new_tokens
    if args.oracle_worker:
        oracle_worker(args.oracle_worker, args.workload, args.steps, args.warmup)
        return
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", str(args.gpus)))
    if args.impl == "reference":
        line = run_reference(args, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        dist.init_process_group("nccl")
    from w4a8_verify_gb300 import build as B
    import synth.cuda as SC
    B.build()
    SC.build()
    if args.matmul:
        if rank == 0:
            print(json.dumps(run_matmul(args)), flush=True)
        return
    line = run_ours(args, rank, world)
    if rank == 0:
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline_line(args.workload)
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
