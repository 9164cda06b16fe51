#!/usr/bin/env python
"""Benchmark: GPU-resident tree-speculative greedy decoding of a Llama-3-8B-shaped
int4-g32 / int8-activation decoder on one GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload llama3-8b-ctx4096|qwen05b-ctx512|tiny]

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

`--impl reference` times the CPU oracle (the test oracle under oracle/) on a bounded sample
of the same workload and prints the same JSON line with "impl": "reference".
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

MAX_NEW = 256
WIDTHS = [1, 4, 8, 16]

WORKLOADS = {
    # name: (shape name, prompt tokens, motifs, motif length, substitution prob, seed)
    "llama3-8b-ctx4096": ("llama3-8b-shaped", 4096, 4, 16, 0.10, 1004),
    "qwen05b-ctx512": ("qwen2.5-0.5b-shaped", 512, 4, 16, 0.10, 1003),
    "tiny": ("tiny-2L-256h", 64, 4, 16, 0.10, 1001),
}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="llama3-8b-ctx4096", choices=sorted(WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--new-tokens", type=int, default=MAX_NEW,
                    help="tokens generated per step (the workload's figure is %d)" % MAX_NEW)
    ap.add_argument("--matmul", type=int, nargs=3, metavar=("K", "N", "M"),
                    help="time one W4A8 matmul shape through the C ABI instead of the decoding step")
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


def run_matmul(args):
    """One W4A8 matmul shape (K, N, M) through the C ABI: fragment pass + matmul per call,
    weights rotated over copies larger than L2, CUDA events on the launching stream."""
    import torch
    import w4a8_verify_gb300 as W
    K, N, M = args.matmul
    dev = torch.device("cuda")
    wb, sb = W.w4a8_weight_layout_bytes(N, K)
    copies = max(2, -(-(4 * 135 * 2**20) // (wb + sb)))
    g = torch.Generator(device=dev).manual_seed(7)
    wt = [torch.randint(-2**31, 2**31 - 1, (wb // 4,), dtype=torch.int32, device=dev, generator=g)
          for _ in range(copies)]
    st = [torch.full((sb // 2,), 0x2000, dtype=torch.int16, device=dev) for _ in range(copies)]
    x = torch.randn(M, K, device=dev, generator=g)
    a_q, a_s = W.w4a8_quantize_rows(x, 0)
    ws = torch.zeros(W.w4a8_matmul_workspace_bytes(M, K, N), dtype=torch.uint8, device=dev)
    y = torch.empty(M, N, device=dev)
    stream = torch.cuda.current_stream()
    for i in range(max(3, args.warmup)):
        W.w4a8_matmul(a_q, a_s, wt[i % copies], st[i % copies], N, y=y, workspace=ws)
    reps = max(args.steps, copies)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for i in range(reps):
        W.w4a8_matmul(a_q, a_s, wt[i % copies], st[i % copies], N, y=y, workspace=ws)
    e1.record(stream)
    e1.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / reps
    alg = N * K // 2 + N * (K // 32) * 2 + M * K + 4 * M * N
    return {"matmul": {"K": K, "N": N, "M": M}, "us_per_call": round(us, 3), "calls": reps,
            "algorithmic_bytes": alg, "GBs": round(alg / us / 1e3, 1), "slices": W.w4a8_matmul_slices(K, N),
            "includes": "activation fragment pass + matmul (2 kernels)"}


# --------------------------------------------------------------------------- our arm

def run_ours(args, rank, world):
    import numpy as np
    import torch
    import synth
    import w4a8_verify_gb300 as W

    torch.cuda.set_device(rank % max(1, torch.cuda.device_count()))
    dev = torch.device("cuda")
    shape_name, plen, nmot, mlen, psub, seed = WORKLOADS[args.workload]
    shape = synth.SHAPES[shape_name]
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
    win_t = {}
    for Wn in (1, 2, 4):
        sess.prefill(prompt_dev, 64)
        torch.cuda.synchronize()
        a = time.perf_counter()
        sess.generate(64, window=Wn, widths=WIDTHS, t_us=t_us)
        win_t[Wn] = time.perf_counter() - a
    fastest = min(win_t.values())
    window = min(w for w, t in win_t.items() if t <= 1.10 * fastest)

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
    total_ms = sum(times)
    if world > 1:
        t = torch.tensor([total_ms], device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        total_ms = float(t.item())
        torch.distributed.barrier()
    tokens = MAX_NEW * args.steps * world
    value = tokens / (total_ms / 1e3)

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

    # dominant kernel: the W4A8 matmul launches of one verification pass (events over a graph)
    sess.prefill(prompt_dev, MAX_NEW)
    mm = {}
    for N in (1, 8, 16):
        if N == 1:
            torch.cuda.nvtx.range_push("matmul_pass")  # lets a profiler select these launches
        us, byts, nl = sess.time_matmuls(N, reps=20)
        if N == 1:
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

    # decode modes of the pages' comparison on the same prompt and token count (not part of
    # `value`): greedy with a host read-back after every token, the GPU loop at width 1 in
    # windows of 8, and the speculation loop with the controller (= value)
    modes = {}
    for name, kw in (("greedy_host_sync_per_token", dict(window=1, fixed_width=1, in_flight=1)),
                     ("gpu_loop_width1_window8", dict(window=8, fixed_width=1, in_flight=2))):
        try:
            sess.prefill(prompt_dev, MAX_NEW)
            ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            ev0.record(stream)
            toks_m, _ = sess.generate(MAX_NEW, **kw)
            ev1.record(stream)
            ev1.synchronize()
            modes[name] = round(len(toks_m) / (ev0.elapsed_time(ev1) / 1e3), 2)
        except Exception as exc:  # reported, never fatal to the line
            modes[name] = "failed: %s" % exc
    modes["spec_controller"] = round(value, 2)

    launches = sum(int(r.kernels) for r in reps)  # kernel nodes of the window graphs run while timed
    mean_rep = reps[-1]
    steps_total = sum(r.n_steps for r in reps)
    wsteps = {w: sum(r.width_steps[w] for r in reps) for w in WIDTHS}
    clocks = clk.summary()
    line = {
        "metric": "accepted tokens/s (GPU-resident tree-speculative greedy decoding)",
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
            "l2": "weights 4.2 GB >> L2 (inputs larger than L2)",
        },
        "e2e": {"value": round(e2e_value, 2), "unit": "tokens/s", "h2d_bytes_per_step": plen * 4,
                "d2h_bytes_per_step": d2h, "includes": "prompt upload + prefill + decode + token read-back"},
        "gpu_launches": launches,
        "clocks": clocks,
        "roofline": {
            "bound": "hbm", "kernel": "k_mm (W4A8 matmul, N=1 verification pass)",
            "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
            "frac": round(achieved / peak, 4), "peak_source": "MEASURED_PEAKS.json hbm_gbs" if peaks else "fallback",
            "traffic": trf,
            "algorithmic_bytes_per_launch": round(bytes1),
            "us_per_launch": round(us1, 3), "launches_per_pass": nl,
            "by_width": {str(N): {"us_per_launch": round(v[0], 3), "GBs": round(v[1] / v[0] / 1e3, 1)}
                         for N, v in mm.items()},
        },
        "verify_step_us": {str(w): round(t, 1) for w, t in zip(WIDTHS, t_us)},
        "decode_modes_tokens_per_s": modes,
        "verify_ratio_8_over_1": round(t_us[2] / t_us[0], 3),
        "tau_tokens_per_step": round(MAX_NEW * args.steps / max(1, steps_total), 3),
        "width_steps": wsteps,
        "host_syncs_per_step": round(sum(r.host_syncs for r in reps) / args.steps, 1),
        "setup_s": round(t_build, 1),
    }
    return line


# --------------------------------------------------------------------------- oracle arm

def oracle_sample(args, steps, warmup):
    """Times the CPU oracle on a bounded sample of the workload: one decoding step of
    one decoder layer of the workload's shape (attention over the full prompt-length
    context) plus 1/32 of the LM head rows; the per-token time is scaled to all layers and
    the full head.  Weights are uniform int4 codes with fp16 scales from the seeded
    generator (the oracle's cost does not depend on the values)."""
    import numpy as np
    import synth
    from oracle import model as OM

    shape_name, plen, *_ = WORKLOADS[args.workload]
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
    cores = len(os.sched_getaffinity(0))
    # warm the dequantised-weight cache (not timed)
    m.step(3, plen)
    per_token = []
    for i in range(warmup + steps):
        a = time.perf_counter()
        tr = {}
        m.forward([3], [plen], [plen], [list(range(plen + 1))], trace=tr)
        t_layer_and_head = time.perf_counter() - a
        if i >= warmup:
            per_token.append(t_layer_and_head)
    # split: time of the 1/32 head alone, to scale layer and head separately
    import numpy as _np
    x = _np.random.default_rng(0).normal(size=sh.hidden)
    a = time.perf_counter()
    m.linear("lm", w.lm_head, x)
    t_head = time.perf_counter() - a
    t_layer = statistics.median(per_token) - t_head
    t_tok = sh.n_layers * t_layer + t_head * (sh.vocab / one.vocab)
    return 1.0 / t_tok, cores, per_token, t_tok


def cpu_baseline_line(args):
    v, cores, samples, t_tok = oracle_sample(args, steps=2, warmup=1)
    return {"value": round(v, 5), "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": "one plain greedy step of one decoder layer (full-context attention) + 1/32 of the LM head, "
                      "scaled to all layers and the full head; %.1f s per token" % t_tok}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    v, cores, samples, t_tok = oracle_sample(args, steps=args.steps, warmup=args.warmup)
    shape_name = WORKLOADS[args.workload][0]
    return {
        "impl": "reference",
        "metric": "accepted tokens/s (GPU-resident tree-speculative greedy decoding)",
        "value": round(v, 5),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(t_tok * 1e3, 1),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "fp64 (oracle)",
        "data": "synthetic",
        "config": {"workload": args.workload, "model": shape_name, "prompt_tokens": WORKLOADS[args.workload][1],
                   "new_tokens_per_step": MAX_NEW, "widths": WIDTHS,
                   "parallelism": "replicas" if world > 1 else "single"},
        "cpu_baseline": {"value": round(v, 5), "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": "one plain greedy step of one decoder layer + 1/32 LM head per step, scaled"},
        "e2e": {"value": round(v, 5), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    global MAX_NEW
    args = parse()
    MAX_NEW = args.new_tokens
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
            line["cpu_baseline"] = cpu_baseline_line(args)
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
