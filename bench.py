"""Benchmark: ternary (T158) Gemma-3-1B-shaped decode step on GB300, plus M=1 GEMV weight GB/s.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl qlin|reference] [--workload ...]

Default workload ("decode"): 26 blocks, hidden 1152, 4 query heads / 1 KV head
of 256, GeGLU 6912, vocab 262144 tied bf16 embedding, ternary weights packed
five per byte, seeded random weights (seed 4); the KV cache is filled to
position 1024 with seeded N(0,1) values and every step decodes one token at a
position cycling through 1024..1087, feeding the greedy token back on the
device.  Weights (744 MB) exceed L2 (126 MB), so every step streams from HBM.

value = tokens/s over all ranks (replicas: one independent decoder per GPU).
Also on the line: M=1 GEMV weight GB/s (T158 K=1152 N=6912 and W8 K=4096
N=11008, rotating weight copies >= 4x L2), the roofline of the dominant
kernel (lm_head), e2e through the C ABI with host buffers, clocks sampled
during the timed region, and the oracle timed on the host cores.
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

METRIC = "M=1 weight GB/s (% of 8 TB/s HBM) and decode tokens/s, Gemma-3-1B-shaped"
NOMINAL_HBM_GBS = 8000.0
POS0, POS_SPAN = 1024, 64
SEED = 4


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["qlin", "reference"], default="qlin")
    p.add_argument("--workload", choices=["decode"], default="decode")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--kernel", choices=["sketch_head", "decode_steps", "lanes_steps", "t158_linears", "t158_calls",
                                        "t158_gemv", "w8_calls"],
                   default=None,
                   help="time one kernel alone on its full-size synthetic inputs (for profiling); no JSON bench line")
    return p.parse_args()


# DRAM traffic of one launch of the fused decode kernel (dram__bytes_read.sum +
# dram__bytes_write.sum from one ncu capture at context `pos`), valid only for
# the kernel sources it was taken on: any change to them reports null.
FUSED_SOURCES = ['decode_fused.cu', 'decode_fused.cuh', 'decode_ops.cuh', 'stream.cuh', 'common.cuh']
FUSED_TRAFFIC = {"sha256": "e1e4bf77c2f314a446fe017f44eca2c0419a5ed3b7c768b6b4b5678a0aa53be8", "bytes": 808881408, "pos": 1024}


def fused_traffic():
    h = hashlib.sha256()
    for f in FUSED_SOURCES:
        with open(os.path.join(ROOT, "weight_streaming_gemv_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return FUSED_TRAFFIC if h.hexdigest() == FUSED_TRAFFIC["sha256"] else None


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# ---------------------------------------------------------------- distributed plumbing
def dist_init(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl" if os.environ.get("BENCH_BACKEND", "nccl") == "nccl" else "gloo")
    return rank, local, world


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def allmax(v, world):
    if world <= 1:
        return v
    import torch
    import torch.distributed as dist

    t = torch.tensor([v], dtype=torch.float64, device="cuda")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- workloads
def decode_cfg(steps, warmup):
    import synth

    return synth.DecoderConfig(max_pos=POS0 + POS_SPAN + 1, **synth.GEMMA3_1B)


def decode_bytes(cfg, pos):
    """Algorithmic HBM bytes of one decode step at `pos`: packed trits at the canonical
    ceil(K/5) pitch, the bf16 lm_head table, the KV cache read (pos+1 positions, k and v), the
    new k/v written, and the small vectors (norm gains, scales, embedding row)."""
    w = sum(cfg.n_layers * n * ((k + 4) // 5) for _, n, k in cfg.matrices())
    lm = cfg.vocab * cfg.dim * 2
    kv_read = cfg.n_layers * 2 * (pos + 1) * cfg.kv_dim * 4
    small = cfg.n_layers * (2 * cfg.dim * 4 + 7 * 4) + cfg.dim * 4 + cfg.dim * 2
    return w + lm + kv_read + small, lm


def run_decode(args, rank, local, world):
    import torch

    import synth
    from weight_streaming_gemv_gb300 import qlin
    from weight_streaming_gemv_gb300.decoder import T158Decoder

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    cfg = decode_cfg(args.steps, args.warmup)
    weights = synth.decoder_weights(cfg, seed=SEED)
    gpu = T158Decoder(cfg, weights, device=dev)
    gpu.kv.copy_(torch.from_numpy(synth.kv_fill(cfg, SEED, POS0)))
    prompt0 = int(synth.prompt_ids(SEED, 1, cfg.vocab)[0])
    gpu.token.fill_(prompt0)
    stream = torch.cuda.current_stream()
    for i in range(max(args.warmup, 3)):
        gpu.step(POS0 + i % POS_SPAN, logits=False)
    gpu.check_status()

    # ---- device-resident timed region
    clocks = ClockSampler(local)
    barrier(world)
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(args.steps):
        gpu.step(POS0 + i % POS_SPAN, logits=False)
    e1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    barrier(world)
    gpu.check_status()
    ms = e0.elapsed_time(e1)
    ms = allmax(ms, world)
    tok_s = world * args.steps / (ms / 1e3)
    mean_pos = POS0 + (POS_SPAN - 1) / 2.0
    step_bytes, lm_bytes = decode_bytes(cfg, int(mean_pos))

    # ---- e2e: host token in, host token out, every step through the C ABI
    pin_in = torch.empty(1, dtype=torch.int32, pin_memory=True)
    pin_out = torch.empty(1, dtype=torch.int32, pin_memory=True)
    pin_in.fill_(prompt0)
    n_e2e = max(1, min(args.steps, 500))
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(n_e2e):
        gpu.token.copy_(pin_in, non_blocking=True)
        gpu.step(POS0 + i % POS_SPAN, logits=False)
        pin_out.copy_(gpu.token, non_blocking=True)
        stream.synchronize()
        pin_in.copy_(pin_out)
    e2e_s = time.perf_counter() - t0
    e2e_s = allmax(e2e_s, world)
    barrier(world)

    # ---- dominant kernel: lm_head (bf16 table GEMV + argmax), timed alone
    x = torch.randn(cfg.dim, dtype=torch.float32, device=dev)
    nxt = torch.zeros(1, dtype=torch.int32, device=dev)
    wsb = qlin.qlin_lm_head_workspace_size(cfg.vocab)
    ws = torch.zeros(wsb, dtype=torch.uint8, device=dev)
    for _ in range(5):
        qlin.qlin_lm_head_argmax(gpu.emb, x, cfg.vocab, cfg.dim, None, nxt, ws, wsb)
    n_lm = 50
    torch.cuda.synchronize()
    a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a0.record(stream)
    for _ in range(n_lm):
        qlin.qlin_lm_head_argmax(gpu.emb, x, cfg.vocab, cfg.dim, None, nxt, ws, wsb)
    a1.record(stream)
    torch.cuda.synchronize()
    lm_ms = a0.elapsed_time(a1) / n_lm
    lm_alg = lm_bytes + cfg.dim * 4 + 8
    peak, peak_kind = peaks()
    lm_gbs = lm_alg / (lm_ms / 1e3) / 1e9
    sketch = sketch_decode(gpu, cfg, args, stream, lm_ms, peak)
    lanes = lanes_decode(gpu, cfg, stream, tok_s)
    gemv = gemv_m1(dev, stream)
    gemv_cfg = gemv_configs(dev, stream, peak)
    prefill = prefill_m512(dev, stream)
    lanes_gemm = lanes_t158(dev, stream)
    step_gbs = step_bytes * args.steps / (ms / 1e3) / 1e9
    traffic = fused_traffic()
    launches_per_step = qlin.decode_step_t158_launches(gpu.model)
    del gpu
    torch.cuda.empty_cache()

    out = {
        "metric": METRIC,
        "value": round(tok_s, 2),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": max(args.warmup, 3),
        "ms_per_step": round(ms / args.steps, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "int8 x ternary -> int32, fp32 (bf16 lm_head)",
        "data": "synthetic (seeded random ternary weights, N(0,1) KV cache filled to 1024)",
        "config": {
            "workload": "decode_step_t158, Gemma-3-1B-shaped ternary decoder, context 1024-1087",
            "n_layers": cfg.n_layers, "dim": cfg.dim, "n_heads": cfg.n_heads, "n_kv_heads": cfg.n_kv_heads,
            "head_dim": cfg.head_dim, "ffn": cfg.ffn, "vocab": cfg.vocab, "pos": [POS0, POS0 + POS_SPAN - 1],
            "global_batch": world, "seq_len": 1, "parallelism": f"replicas x{world}",
            "l2": "inputs larger than L2 (744 MB of weights per step)",
            "hbm_bytes_per_step": step_bytes,
        },
        "step_hbm": {
            "achieved_gbs": round(step_bytes * args.steps / (ms / 1e3) / 1e9, 1),
            "frac_of_8tbs": round(step_bytes * args.steps / (ms / 1e3) / 1e9 / NOMINAL_HBM_GBS, 4),
            "frac_of_peak": round(step_bytes * args.steps / (ms / 1e3) / 1e9 / peak, 4),
        },
        "sketch_head": sketch,
        "lanes_decode": lanes,
        "gemv_m1": gemv,
        "gemv_configs": gemv_cfg,
        "prefill_m512": prefill,
        "lanes_t158": lanes_gemm,
        # the step is one launch of the fused kernel: its algorithmic bytes over
        # its CUDA-event time on the launching stream
        "roofline": {
            "kernel": "decode_fused_kernel",
            "bound": "hbm", "achieved": round(step_gbs, 1), "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
            "frac": round(step_gbs / peak, 4),
            "traffic": traffic["bytes"] if traffic else None,
            "traffic_pos": traffic["pos"] if traffic else None,
            "algorithmic_bytes": step_bytes, "ms_per_launch": round(ms / args.steps, 5),
        },
        "lm_head": {
            "kernel": "lm_head_kernel (standalone, timed alone)",
            "bound": "hbm", "achieved": round(lm_gbs, 1), "peak": peak, "unit": "GB/s",
            "frac": round(lm_gbs / peak, 4), "algorithmic_bytes": lm_alg, "ms_per_launch": round(lm_ms, 5),
        },
        "e2e": {"value": round(world * n_e2e / e2e_s, 2), "unit": "tokens/s", "h2d_bytes_per_step": 4,
                "d2h_bytes_per_step": 4, "steps": n_e2e},
        "gpu_launches": args.steps * launches_per_step,
        "clocks": clk,
    }
    return out, cfg, weights


def sketch_decode(gpu, cfg, args, stream, lm_ms, peak):
    """The output layer as a sketch head: the decode step with it (two launches per
    step, tokens fed back on the device) and the sketch head kernel timed alone after
    an L2 flush, against the exact lm_head kernel's time."""
    import torch

    from weight_streaming_gemv_gb300 import qlin

    K_EXACT, N_CAND = 32, 1024
    gpu.prepare_sketch(k=K_EXACT, n_cand=N_CAND, stream=stream)
    for i in range(max(args.warmup, 3)):
        gpu.step_sketch(POS0 + i % POS_SPAN)
    torch.cuda.synchronize()
    gpu.check_sketch_status()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(args.steps):
        gpu.step_sketch(POS0 + i % POS_SPAN)
    e1.record(stream)
    torch.cuda.synchronize()
    gpu.check_sketch_status()
    ms = e0.elapsed_time(e1) / args.steps

    # the kernel alone: a hidden state with the final norm's sizes, L2 flushed before each call
    V, D = cfg.vocab, cfg.dim
    x = (torch.randn(D, device=gpu.emb.device) * gpu.g_final.abs()).contiguous()
    cand = torch.empty(N_CAND, dtype=torch.int32, device=x.device)
    cl = torch.empty(N_CAND, dtype=torch.float32, device=x.device)
    nx = torch.zeros(1, dtype=torch.int32, device=x.device)
    wsb = qlin.qlin_sketch_workspace_size(V)
    ws = torch.zeros(wsb, dtype=torch.uint8, device=x.device)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=x.device)
    call = lambda: qlin.qlin_sketch_head(gpu.emb, gpu.sk_emb_t, gpu.sk_signs, gpu.sk_perm, gpu.sk_ce, V, D, x,
                                         K_EXACT, N_CAND, None, cand, cl, nx, ws, wsb, stream)
    for _ in range(5):
        call()
    ts = []
    for it in range(40):
        flush.fill_(it & 255)
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        call()
        a1.record(stream)
        torch.cuda.synchronize()
        ts.append(a0.elapsed_time(a1) * 1e3)
    qlin.qlin_sketch_head_status(ws)
    us = float(sorted(ts)[len(ts) // 2])
    nblk = (D + 63) // 64
    alg = V * nblk * 8 + K_EXACT * V * 2 + N_CAND * D * 2 + D * 4
    gbs = alg / (us * 1e-6) / 1e9
    return {
        "decode_tokens_per_s": round(1e3 / ms, 2), "decode_ms_per_step": round(ms, 5), "launches_per_step": 2,
        "k_exact": K_EXACT, "n_cand": N_CAND, "size_order": "|final norm gain|",
        "kernel": "sketch_head_kernel (alone, L2 flushed, median of 40)",
        "us_per_call": round(us, 2), "exact_lm_head_us": round(lm_ms * 1e3, 2),
        "speedup_vs_exact_lm_head": round(lm_ms * 1e3 / us, 2),
        "bound": "hbm", "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s", "frac": round(gbs / peak, 4),
        "algorithmic_bytes": alg,
    }


def lanes_decode(gpu, cfg, stream, single_tok_s):
    """Many users at once: one decode step over U lanes (one token of each of U
    sequences at context 1024), captured in a CUDA graph and replayed; tokens/s
    = U / step time, against the single-user fused step."""
    import torch

    users = (1, 2, 4, 8, 16, 32, 64, 128, 256)
    U_MAX = users[-1]
    gpu.prepare_lanes(n_seqs=U_MAX, max_lanes=U_MAX)
    kv0 = gpu.kv[:, :, :, :].clone()  # the bench's cache: filled to 1024 by the decode run
    for s in range(U_MAX):
        gpu.kv_lanes[s].copy_(kv0)
    gpu.lane_seq.copy_(torch.arange(U_MAX, dtype=torch.int32))
    gpu.lane_tokens.fill_(int(gpu.token.item()))
    gpu.lane_pos.fill_(POS0)
    rows = []
    for U in users:
        gpu.step_lanes(U, stream=stream)
        torch.cuda.synchronize()
        gpu.check_lanes_status()
        g = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream()
        cap.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(cap):
            with torch.cuda.graph(g, stream=cap):
                gpu.step_lanes(U, stream=cap)
        torch.cuda.current_stream().wait_stream(cap)
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        n = 20
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n):
            g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / n
        rows.append((U, ms))
        del g
    gpu.check_lanes_status()
    del gpu.kv_lanes, gpu.lanes_workspace
    torch.cuda.empty_cache()
    return {
        "users": [u for u, _ in rows], "ms_per_step": [round(ms, 4) for _, ms in rows],
        "tokens_per_s": [round(u / ms * 1e3, 1) for u, ms in rows],
        "vs_single_user_fused_step": [round(u / ms * 1e3 / single_tok_s, 2) for u, ms in rows],
        "timing": "CUDA graph of one lanes step, 20 replays; every user at context 1024",
        "launches_per_step": [qlin_launches(gpu, u) for u, _ in rows],
    }


def qlin_launches(gpu, U):
    from weight_streaming_gemv_gb300 import qlin

    return qlin.decode_lanes_t158_launches(gpu.model, U)


def _single_launch_us(fn, stream, n=25):
    """One call alone: an L2 flush (a 256 MB write), then CUDA events around the call on the
    launching stream; the median of n such calls, in microseconds.  A device-side sleep after
    the flush keeps the stream busy while the host queues the events and the call, so the
    interval holds the call's device time, not the host's launch latency."""
    import torch

    flush = torch.empty(256 << 20, dtype=torch.uint8, device=torch.device("cuda", torch.cuda.current_device()))
    for _ in range(3):
        fn()
    ts = []
    for it in range(n):
        flush.fill_(it & 255)
        torch.cuda._sleep(200000)  # about 0.1 ms at 2 GHz
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        fn()
        a1.record(stream)
        torch.cuda.synchronize()
        ts.append(a0.elapsed_time(a1) * 1e3)
    del flush
    return float(np.median(ts))


def _oracle_us(fn, budget_s=1.5, max_calls=200):
    """The oracle's call timed on the host cores: calls until `budget_s` or `max_calls`."""
    fn()
    n, t0 = 0, time.perf_counter()
    while n < max_calls and (n == 0 or time.perf_counter() - t0 < budget_s):
        fn()
        n += 1
    dt = time.perf_counter() - t0
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    return dt / n * 1e6, n, int(os.environ.get("OMP_NUM_THREADS", cores))


def gemv_configs(dev, stream, peak):
    """The GEMV configurations the metric is quoted on, each with weight GB/s over rotating
    weight copies (>= 4x L2, CUDA graph), the fraction of the measured HBM peak, the oracle's
    time for the same call on the host cores, and (configs 1 and 2) the single-launch time:
    * W8 M=1, K=288, N=768 (stories15M FFN w1), seed 0;
    * T158 M=1, K=1152, N=6912 (Gemma-3-1B gate/up), seed 1;
    * W8 at Llama-2-7B shapes (4096->11008, 11008->4096, 4096->4096) x M in {1, 4, 16}, seed 3."""
    import torch

    import oracle
    import synth
    from weight_streaming_gemv_gb300 import qlin

    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 126 * 2 ** 20)
    out = {}

    def w8_point(seed, M, K, N, single):
        d = synth.w8_gemv(seed, M, K, N)
        q_o, s_o = oracle.w8_quantize(d["w"])
        pitch = (K + 15) // 16 * 16
        w8 = np.zeros((N, pitch), np.int8)
        w8[:, :K] = q_o
        w1 = torch.from_numpy(w8).to(dev)
        R = int(np.ceil(4 * l2 / w1.numel()))
        wr = w1.repeat(R, 1)
        x = torch.from_numpy(d["x"]).to(dev)
        y = torch.empty((M, N), dtype=torch.float32, device=dev)
        alg = N * K + 4 * M * K + 4 * M * N
        # M > 1: the workspace entry point (activation terms once per call), its scratch
        # allocated once outside the timed calls
        nb = qlin.qlin_w8_f32_workspace_size(M, K)
        work = torch.empty(max(nb, 16), dtype=torch.uint8, device=dev)

        def call(wt):
            if M == 1:
                qlin.qlin_w8_f32(x, wt, pitch, float(s_o), y, M, N, K)
            else:
                qlin.qlin_w8_f32_ws(x, wt, pitch, float(s_o), y, M, N, K, work, nb)

        r = _time_rotating(lambda i: call(wr[i * N]), R, alg, stream)
        r["api"] = "qlin_w8_f32" if M == 1 else "qlin_w8_f32_ws"
        r["frac"] = round(r["gbs"] / peak, 4)
        if single:
            us1 = _single_launch_us(lambda: call(w1), stream)
            r["single_launch_us"] = round(us1, 2)
            r["single_launch_gbs"] = round(alg / (us1 * 1e-6) / 1e9, 1)
        o_us, o_n, o_thr = _oracle_us(lambda: oracle.w8_linear(d["x"], w8, s_o, K))
        r["cpu_baseline"] = {"us_per_call": round(o_us, 1), "gbs": round(alg / (o_us * 1e-6) / 1e9, 3),
                             "calls": o_n, "cores": o_thr, "kind": "oracle"}
        del w1, wr
        return r

    out["cfg1_w8_m1_k288_n768"] = w8_point(0, 1, 288, 768, True)
    # T158 M=1 (config 2)
    K, N = 1152, 6912
    d = synth.t158_gemv(1, 1, K, N)
    pitch = qlin.t158_pitch(K)
    w1 = torch.from_numpy(qlin.t158_pack(d["trits"], pitch)).to(dev)
    R = int(np.ceil(4 * l2 / w1.numel()))
    wr = w1.repeat(R, 1)
    x = torch.from_numpy(d["x"]).to(dev)
    xq = torch.empty((1, K), dtype=torch.int8, device=dev)
    xs = torch.empty(1, dtype=torch.float32, device=dev)
    y = torch.empty((1, N), dtype=torch.float32, device=dev)
    qlin.qlin_quant_i8(x, xq, xs, 1, K)
    alg = N * ((K + 4) // 5) + K + 4 + N * 4
    r = _time_rotating(lambda i: qlin.qlin_t158_i8(xq, xs, wr[i * N], pitch, d["w_scale"], y, None, 1, N, K), R, alg,
                       stream)
    r["frac"] = round(r["gbs"] / peak, 4)
    us1 = _single_launch_us(lambda: qlin.qlin_t158_i8(xq, xs, w1, pitch, d["w_scale"], y, None, 1, N, K), stream)
    r["single_launch_us"] = round(us1, 2)
    r["single_launch_gbs"] = round(alg / (us1 * 1e-6) / 1e9, 1)
    xq_o, xs_o = oracle.quant_i8(d["x"])
    pk_o = oracle.t158_pack(d["trits"])
    o_us, o_n, o_thr = _oracle_us(lambda: oracle.t158_linear(xq_o, xs_o, pk_o, d["w_scale"], K))
    r["cpu_baseline"] = {"us_per_call": round(o_us, 1), "gbs": round(alg / (o_us * 1e-6) / 1e9, 3), "calls": o_n,
                         "cores": o_thr, "kind": "oracle"}
    out["cfg2_t158_m1_k1152_n6912"] = r
    del w1, wr
    for K, N in ((4096, 11008), (11008, 4096), (4096, 4096)):
        for M in (1, 4, 16):
            out[f"cfg4_w8_m{M}_k{K}_n{N}"] = w8_point(3, M, K, N, True)
    torch.cuda.empty_cache()
    return out


def gemv_m1(dev, stream):
    """M=1 GEMV weight GB/s over rotating weight copies (>= 4x L2), launched back to back."""
    import torch

    import synth
    from weight_streaming_gemv_gb300 import qlin

    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 126 * 2 ** 20)
    res = {}
    # T158, K=1152, N=6912
    K, N = 1152, 6912
    d = synth.t158_gemv(1, 1, K, N)
    pitch = qlin.t158_pitch(K)
    w1 = torch.from_numpy(qlin.t158_pack(d["trits"], pitch)).to(dev)
    R = int(np.ceil(4 * l2 / w1.numel()))
    ws = w1.repeat(R, 1)  # R copies back to back
    x = torch.from_numpy(d["x"]).to(dev)
    xq = torch.empty((1, K), dtype=torch.int8, device=dev)
    xs = torch.empty(1, dtype=torch.float32, device=dev)
    y = torch.empty((1, N), dtype=torch.float32, device=dev)
    qlin.qlin_quant_i8(x, xq, xs, 1, K)
    alg = N * ((K + 4) // 5) + K + 4 + N * 4

    def t158(r):
        qlin.qlin_t158_i8(xq, xs, ws[r * N], pitch, d["w_scale"], y, None, 1, N, K)

    res["t158_k1152_n6912"] = _time_rotating(t158, R, alg, stream)
    del ws
    # W8, K=4096, N=11008
    K, N = 4096, 11008
    wq = torch.randint(-127, 128, (N, K), dtype=torch.int8, device=dev)
    R = int(np.ceil(4 * l2 / wq.numel()))
    ws = wq.repeat(R, 1)
    x = torch.randn((1, K), dtype=torch.float32, device=dev)
    y = torch.empty((1, N), dtype=torch.float32, device=dev)
    alg = N * K + 4 * K + 4 * N

    def w8(r):
        qlin.qlin_w8_f32(x, ws[r * N], K, 0.01, y, 1, N, K)

    res["w8_k4096_n11008"] = _time_rotating(w8, R, alg, stream)
    del ws
    # W8 with one scale per 128 weights, same shape
    G = 128
    s_pitch = (K // G + 3) // 4 * 4
    sc1 = torch.rand((N, s_pitch), dtype=torch.float32, device=dev) * 0.01 + 0.001
    ws = wq.repeat(R, 1)
    scs = sc1.repeat(R, 1)
    alg = N * K + 4 * N * (K // G) + 4 * K + 4 * N

    def w8g(r):
        qlin.qlin_w8g_f32(x, ws[r * N], K, scs[r * N], s_pitch, G, y, 1, N, K)

    res["w8g128_k4096_n11008"] = _time_rotating(w8g, R, alg, stream)
    del ws, scs
    torch.cuda.empty_cache()
    res["zero_skip"] = zero_skip(dev, stream, l2)
    return res


def zero_skip(dev, stream, l2):
    """T158 M = 1 with 80% of the input groups of four zero: the dense kernel on the
    five-trit layout against the kernel that skips zero groups on the group-major
    layout, both over rotating weight copies (>= 4x L2) in a CUDA graph."""
    import torch

    import synth
    from weight_streaming_gemv_gb300 import qlin

    out = {}
    for K, N in ((1152, 6912), (6912, 1152), (16384, 16384)):
        d = synth.t158_gemv(5, 1, K, N)
        x = d["x"].copy()
        G = (K + 3) // 4
        keep = synth.uniform_f32(5, 9, (G,), 0.0, 1.0) >= 0.8
        x[0, :] *= np.repeat(keep, 4)[:K]
        xd = torch.from_numpy(x).to(dev)
        xq = torch.empty((1, K), dtype=torch.int8, device=dev)
        xs = torch.empty(1, dtype=torch.float32, device=dev)
        qlin.qlin_quant_i8(xd, xq, xs, 1, K)
        y = torch.empty((1, N), dtype=torch.float32, device=dev)
        pitch = qlin.t158_pitch(K)
        w1 = torch.from_numpy(qlin.t158_pack(d["trits"], pitch)).to(dev)
        R = int(np.ceil(4 * l2 / w1.numel()))
        wd = w1.repeat(R, 1)
        dense = _time_rotating(lambda r: qlin.qlin_t158_i8(xq, xs, wd[r * N], pitch, d["w_scale"], y, None, 1, N, K),
                               R, N * ((K + 4) // 5) + K + 8 + 4 * N, stream)
        del wd
        gp = qlin.t158_group_pitch(N)
        g1 = torch.from_numpy(qlin.t158_pack_groups(d["trits"], gp)).to(dev)
        Rg = int(np.ceil(4 * l2 / g1.numel()))
        wg = g1.repeat(Rg, 1)
        wsb = qlin.qlin_t158_skip_workspace_size(N)
        wsk = torch.zeros(wsb, dtype=torch.uint8, device=dev)
        nnz = int(keep.sum())
        skip = _time_rotating(lambda r: qlin.qlin_t158_i8_skip(xq, xs, wg[r * G], gp, d["w_scale"], y, None, N, K,
                                                                wsk, wsb), Rg, nnz * N + K + 8 + 4 * N, stream)
        del wg
        out[f"t158_k{K}_n{N}"] = {
            "nonzero_groups": nnz, "groups": G,
            "dense_us": dense["us_per_call"], "skip_us": skip["us_per_call"],
            "speedup": round(dense["us_per_call"] / skip["us_per_call"], 2),
            "skip_weight_bytes_read": nnz * N, "dense_weight_bytes_read": N * ((K + 4) // 5),
        }
    torch.cuda.empty_cache()
    return out


def _time_rotating(fn, R, alg_bytes, stream):
    """Capture R back-to-back calls (one per weight copy) in a CUDA graph and time its replays
    with CUDA events, so the number is the kernels' throughput, not host launch cost."""
    import torch

    for r in range(min(R, 8)):
        fn(r)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cap):
        with torch.cuda.graph(g, stream=cap):
            for r in range(R):
                fn(r)
    torch.cuda.current_stream().wait_stream(cap)
    g.replay()
    torch.cuda.synchronize()
    reps = max(3, 2000 // R)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        g.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    n = reps * R
    us = e0.elapsed_time(e1) * 1e3 / n
    gbs = alg_bytes / (us * 1e-6) / 1e9
    del g
    return {"us_per_call": round(us, 3), "gbs": round(gbs, 1), "frac_of_8tbs": round(gbs / NOMINAL_HBM_GBS, 4),
            "copies": R, "calls": n, "algorithmic_bytes": alg_bytes, "timing": "CUDA graph of the rotating calls"}


def prefill_m512(dev, stream):
    """The two 512-token T158 layers of the prompt (1152->6912, 6912->1152) on the tensor
    cores through qlin_t158_i8_ws (activation tiles converted once per call, inside the
    timed call): a CUDA graph of back-to-back calls over rotating weight copies (>= 4x L2);
    dense fp16 rate (2 M N K flops per call) against the measured bf16 tensor peak (fp16 and
    bf16 share one rate).  `us_no_ws`: the same through qlin_t158_i8 (activations converted
    inside the product for every 128 weight rows)."""
    import torch

    import synth
    from weight_streaming_gemv_gb300 import qlin

    tflops_peak = None
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
            tflops_peak = float(json.load(fh)["bf16_tflops"])
    except (OSError, KeyError, ValueError):
        tflops_peak = 1900.0
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 126 * 2 ** 20)
    res = {}
    M = 512
    for K, N in [(1152, 6912), (6912, 1152)]:
        d = synth.t158_gemv(2, M, K, N)
        pitch = qlin.t158_pitch(K)
        w1 = torch.from_numpy(qlin.t158_pack(d["trits"], pitch)).to(dev)
        R = int(np.ceil(4 * l2 / w1.numel()))
        wr = w1.repeat(R, 1)
        x = torch.from_numpy(d["x"]).to(dev)
        xq = torch.empty((M, K), dtype=torch.int8, device=dev)
        xs = torch.empty(M, dtype=torch.float32, device=dev)
        qlin.qlin_quant_i8(x, xq, xs, M, K)
        y = torch.empty((M, N), dtype=torch.float32, device=dev)
        nb = qlin.qlin_t158_i8_workspace_size(M, K)
        work = torch.empty(nb, dtype=torch.uint8, device=dev)

        def call_ws(r):
            qlin.qlin_t158_i8_ws(xq, xs, wr[r * N], pitch, d["w_scale"], y, None, M, N, K, work, nb)

        def call_plain(r):
            qlin.qlin_t158_i8(xq, xs, wr[r * N], pitch, d["w_scale"], y, None, M, N, K)

        us = _time_rotating(call_ws, R, 0, stream)["us_per_call"]
        us_plain = _time_rotating(call_plain, R, 0, stream)["us_per_call"]
        tf = 2.0 * M * N * K / (us * 1e-6) / 1e12
        res[f"t158_m{M}_k{K}_n{N}"] = {
            "us_per_call": round(us, 2), "bound": "tensor", "tflops": round(tf, 1), "peak_tflops": tflops_peak,
            "frac": round(tf / tflops_peak, 4), "int_ops": 2 * M * N * K, "us_no_ws": round(us_plain, 2),
            "timing": f"CUDA graph of {R} back-to-back calls over rotating weight copies (>= 4x L2)"}
        del w1, wr, x, xq, xs, y, work
    torch.cuda.empty_cache()
    return res


def lanes_t158(dev, stream):
    """Many tokens through one weight pass ([citric] "Many users at once"): the T158
    layers of the decoder at M = 1..64 tokens through qlin_t158_i8_ws, a CUDA graph of
    back-to-back calls over rotating weight copies (>= 4x L2); token-rows per microsecond
    = M / time."""
    import torch

    import synth
    from weight_streaming_gemv_gb300 import qlin

    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 126 * 2 ** 20)
    res = {}
    for K, N in [(1152, 6912), (6912, 1152)]:
        d = synth.t158_gemv(2, 64, K, N)
        pitch = qlin.t158_pitch(K)
        w1 = torch.from_numpy(qlin.t158_pack(d["trits"], pitch)).to(dev)
        R = int(np.ceil(4 * l2 / w1.numel()))
        wr = w1.repeat(R, 1)
        x = torch.from_numpy(d["x"]).to(dev)
        row = {"M": [], "us_per_call": [], "token_rows_per_us": []}
        for M in [1, 2, 4, 8, 16, 32, 64]:
            xq = torch.empty((M, K), dtype=torch.int8, device=dev)
            xs = torch.empty(M, dtype=torch.float32, device=dev)
            qlin.qlin_quant_i8(x[:M].contiguous(), xq, xs, M, K)
            y = torch.empty((M, N), dtype=torch.float32, device=dev)
            nb = qlin.qlin_t158_i8_workspace_size(M, K)
            work = torch.empty(max(nb, 16), dtype=torch.uint8, device=dev)

            def call(r):
                qlin.qlin_t158_i8_ws(xq, xs, wr[r * N], pitch, d["w_scale"], y, None, M, N, K, work, nb)

            us = _time_rotating(call, R, 0, stream)["us_per_call"]
            row["M"].append(M)
            row["us_per_call"].append(round(us, 2))
            row["token_rows_per_us"].append(round(M / us, 3))
        row["timing"] = f"CUDA graph of {R} back-to-back calls over rotating weight copies (>= 4x L2)"
        res[f"t158_k{K}_n{N}"] = row
        del w1, wr, x
    torch.cuda.empty_cache()
    return res


# ---------------------------------------------------------------- oracle on the host cores
def oracle_decode(cfg, weights, steps, warmup, budget_s):
    """The oracle's decode step at the same positions, until `steps` are done or `budget_s` passes."""
    import oracle
    import synth

    orc = oracle.Decoder(cfg, weights)
    kv = synth.kv_fill(cfg, SEED, POS0)
    token = int(synth.prompt_ids(SEED, 1, cfg.vocab)[0])
    for i in range(warmup):
        token, _ = orc.step(kv, token, POS0 + i % POS_SPAN, want_logits=False)
    done = 0
    t0 = time.perf_counter()
    while done < steps and time.perf_counter() - t0 < budget_s:
        token, _ = orc.step(kv, token, POS0 + done % POS_SPAN, want_logits=False)
        done += 1
    dt = time.perf_counter() - t0
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    threads = int(os.environ.get("OMP_NUM_THREADS", cores))
    return done, dt, threads


def kernel_only(name):
    """The sketch head alone on a synthetic 262144 x 1152 table: 5 warm-up calls, then 20 timed
    calls with an L2 flush before each (prints one line of timings)."""
    import numpy as np
    import torch

    import synth
    from weight_streaming_gemv_gb300 import qlin

    dev = torch.device("cuda", 0)
    if name == "t158_linears":
        # the 512-token prompt layers and the 1..64-token layers of the tensor-core T158 linear
        stream = torch.cuda.current_stream(dev)
        print(json.dumps({"kernel": name, "prefill_m512": prefill_m512(dev, stream),
                          "lanes_t158": lanes_t158(dev, stream)}))
        return 0
    if name == "t158_gemv":
        # five plain M=1 calls of qlin_t158_i8 per shape (1152->6912, 6912->1152, 16384->16384, in that
        # order), each shape after one quantiser launch: a short launch list for the profiler
        for K, N in [(1152, 6912), (6912, 1152), (16384, 16384)]:
            d = synth.t158_gemv(3, 1, K, N)
            pitch = qlin.t158_pitch(K)
            w = torch.from_numpy(qlin.t158_pack(d["trits"], pitch)).to(dev)
            xq = torch.empty((1, K), dtype=torch.int8, device=dev)
            xs = torch.empty(1, dtype=torch.float32, device=dev)
            qlin.qlin_quant_i8(torch.from_numpy(d["x"]).to(dev), xq, xs, 1, K)
            y = torch.empty((1, N), dtype=torch.float32, device=dev)
            for _ in range(5):
                qlin.qlin_t158_i8(xq, xs, w, pitch, d["w_scale"], y, None, 1, N, K)
        torch.cuda.synchronize()
        print(json.dumps({"kernel": name}))
        return 0
    if name == "w8_calls":
        # four calls of qlin_w8_f32_ws, then four of qlin_w8_f32, 16 tokens through 4096 -> 11008
        # (config-4 inputs, quantised on the GPU): a short launch list for the profiler
        M, K, N = 16, 4096, 11008
        d = synth.w8_gemv(3, M, K, N)
        w8 = torch.empty((N, K), dtype=torch.int8, device=dev)
        sc = torch.empty(1, dtype=torch.float32, device=dev)
        qlin.qlin_w8_quantize(torch.from_numpy(d["w"]).to(dev), N, K, w8, K, sc)
        s = float(sc.item())
        x = torch.from_numpy(d["x"]).to(dev)
        y = torch.empty((M, N), dtype=torch.float32, device=dev)
        nb = qlin.qlin_w8_f32_workspace_size(M, K)
        work = torch.empty(nb, dtype=torch.uint8, device=dev)
        for _ in range(4):
            qlin.qlin_w8_f32_ws(x, w8, K, s, y, M, N, K, work, nb)
        for _ in range(4):
            qlin.qlin_w8_f32(x, w8, K, s, y, M, N, K)
        torch.cuda.synchronize()
        print(json.dumps({"kernel": name}))
        return 0
    if name == "t158_calls":
        # five plain calls of qlin_t158_i8_ws per shape (512 and 64 tokens through 1152->6912 and
        # 6912->1152, in that order): a short launch list for the profiler
        for M in (512, 64):
            for K, N in [(1152, 6912), (6912, 1152)]:
                d = synth.t158_gemv(2, M, K, N)
                pitch = qlin.t158_pitch(K)
                w = torch.from_numpy(qlin.t158_pack(d["trits"], pitch)).to(dev)
                xq = torch.empty((M, K), dtype=torch.int8, device=dev)
                xs = torch.empty(M, dtype=torch.float32, device=dev)
                qlin.qlin_quant_i8(torch.from_numpy(d["x"]).to(dev), xq, xs, M, K)
                y = torch.empty((M, N), dtype=torch.float32, device=dev)
                nb = qlin.qlin_t158_i8_workspace_size(M, K)
                work = torch.empty(nb, dtype=torch.uint8, device=dev)
                for _ in range(5):
                    qlin.qlin_t158_i8_ws(xq, xs, w, pitch, d["w_scale"], y, None, M, N, K, work, nb)
        torch.cuda.synchronize()
        print(json.dumps({"kernel": name}))
        return 0
    if name == "lanes_steps":
        # three steps of 64 lanes (64 users at context 1024) of the Gemma-shaped decoder
        from weight_streaming_gemv_gb300.decoder import T158Decoder

        cfg = decode_cfg(3, 0)
        gpu = T158Decoder(cfg, synth.decoder_weights(cfg, seed=SEED), device=dev)
        U = 64
        gpu.prepare_lanes(n_seqs=U, max_lanes=U)
        kv0 = torch.from_numpy(synth.kv_fill(cfg, SEED, POS0)).to(dev)
        for s in range(U):
            gpu.kv_lanes[s].copy_(kv0)
        gpu.lane_seq.copy_(torch.arange(U, dtype=torch.int32))
        gpu.lane_tokens.copy_(torch.from_numpy(synth.prompt_ids(SEED, U, cfg.vocab)))
        for i in range(3):
            gpu.lane_pos.fill_(POS0 + i)
            gpu.step_lanes(U)
            gpu.lane_tokens.copy_(gpu.lane_next)
        torch.cuda.synchronize()
        gpu.check_lanes_status()
        print(json.dumps({"kernel": name, "next0": int(gpu.lane_next[0].item())}))
        return 0
    if name == "decode_steps":
        # six exact steps and six sketch-head steps of the Gemma-shaped decoder at context 1024
        from weight_streaming_gemv_gb300.decoder import T158Decoder

        cfg = decode_cfg(6, 0)
        gpu = T158Decoder(cfg, synth.decoder_weights(cfg, seed=SEED), device=dev)
        gpu.kv.copy_(torch.from_numpy(synth.kv_fill(cfg, SEED, POS0)))
        gpu.token.fill_(int(synth.prompt_ids(SEED, 1, cfg.vocab)[0]))
        gpu.prepare_sketch(32, 1024)
        for i in range(6):
            gpu.step(POS0 + i, logits=False)
        for i in range(6):
            gpu.step_sketch(POS0 + i)
        torch.cuda.synchronize()
        gpu.check_status()
        gpu.check_sketch_status()
        print(json.dumps({"kernel": name, "next": int(gpu.token.item())}))
        return 0
    V, D, K_EXACT, N_CAND = 262144, 1152, 32, 1024
    d = synth.sketch_head(SEED, V, D)
    emb = torch.from_numpy(d["emb"].view(np.int16)).to(dev)
    scale = torch.from_numpy(d["scale"]).to(dev)
    emb_t = torch.empty((D, qlin.qlin_sketch_emb_t_pitch(V)), dtype=torch.int16, device=dev)
    signs = torch.empty(qlin.qlin_sketch_signs_bytes(V, D) // 8, dtype=torch.int64, device=dev)
    perm = torch.empty(D, dtype=torch.int32, device=dev)
    c_e = torch.zeros(1, dtype=torch.float32, device=dev)
    qlin.qlin_sketch_prepare(emb, V, D, scale, emb_t, signs, perm, c_e)
    x = torch.from_numpy(synth.sketch_x(SEED, 0, d["scale"])).to(dev)
    cand = torch.empty(N_CAND, dtype=torch.int32, device=dev)
    cl = torch.empty(N_CAND, dtype=torch.float32, device=dev)
    nx = torch.zeros(1, dtype=torch.int32, device=dev)
    wsb = qlin.qlin_sketch_workspace_size(V)
    ws = torch.zeros(wsb, dtype=torch.uint8, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    ts = []
    for it in range(25):
        flush.fill_(it & 255)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        qlin.qlin_sketch_head(emb, emb_t, signs, perm, c_e, V, D, x, K_EXACT, N_CAND, None, cand, cl, nx, ws, wsb)
        e1.record()
        torch.cuda.synchronize()
        if it >= 5:
            ts.append(e0.elapsed_time(e1) * 1e3)
    qlin.qlin_sketch_head_status(ws)
    print(json.dumps({"kernel": name, "us_median": round(float(np.median(ts)), 2), "us_min": round(min(ts), 2),
                      "next": int(nx.item())}))
    return 0


def main():
    args = parse()
    if args.kernel:
        return kernel_only(args.kernel)
    rank, local, world = dist_init(args.gpus)
    if args.impl == "reference":
        if rank != 0:
            return 0
        import synth

        cfg = decode_cfg(args.steps, args.warmup)
        weights = synth.decoder_weights(cfg, seed=SEED)
        done, dt, threads = oracle_decode(cfg, weights, args.steps, min(args.warmup, 2), budget_s=120.0)
        v = done / dt
        line = {
            "impl": "reference", "metric": METRIC, "value": round(v, 4), "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": done, "steps_requested": args.steps, "warmup": min(args.warmup, 2),
            "ms_per_step": round(dt / done * 1e3, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "int64 exact / fp32 / fp64 (oracle)", "data": "synthetic",
            "config": {"workload": "decode step, Gemma-3-1B-shaped ternary decoder, context 1024-1087 (CPU oracle)"},
            "cpu_baseline": {"value": round(v, 4), "unit": "tokens/s", "cores": threads, "kind": "oracle",
                             "sample": f"{done} decode steps (time-capped at 120 s)"},
            "e2e": {"value": round(v, 4), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        }
        print(json.dumps(line))
        return 0

    out, cfg, weights = run_decode(args, rank, local, world)
    if rank == 0 and not args.no_cpu_baseline:
        done, dt, threads = oracle_decode(cfg, weights, 40, 1, budget_s=20.0)
        out["cpu_baseline"] = {"value": round(done / dt, 4), "unit": "tokens/s", "cores": threads, "kind": "oracle",
                               "sample": f"{done} oracle decode steps at context 1024+ on the host cores (~20 s cap)"}
    if rank == 0:
        print(json.dumps(out))
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
