#!/usr/bin/env python3
"""Benchmark of the Gated-DeltaNet mixer on GB300. It prints one JSON line.

The headline workload is batched decode at scale: the 30 GDN layers of the
40-layer stack, each with its own seeded parameters and fp32 states (15 GiB),
run on B=256 sequences. One step is one token for every sequence through all
30 layers, as 30 calls of gdn_decode_step. ``value`` is decode tokens/s: B x
steps / device time, with the inputs already resident in HBM.

The same run also times the T=4096 bf16 prefill (one gdn_prefill call) and
reports it under "prefill".

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

With N>1 (launched with torchrun) every rank runs its own replica of the
workload ("replicas only": the mixer has no exchange step). value is the
total over ranks, divided by the slowest rank's time. ``--impl reference``
times the fp64 CPU oracle on the host cores on a bounded sample of the same
workload, as the reference arm.
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

METRIC = "GDN prefill tok/s @T=4096; decode tok/s @B=256; % of HBM/TC roofline"
I_C_CONV = 8192             # q|k|v conv channels
LAYERS, BATCH, PREFILL_T, CHUNK = 30, 256, 4096, 64
NOMINAL_HBM_GBS = 8000.0

# Algorithmic bytes of one decode token through one layer (bf16 activations,
# fp32 state, bf16 output): the state is read and written once (2 x 32 x 128 x
# 128 x 4), the conv_state is read and written once (2 x 3 x 8192 x 2), and the
# inputs qkv, z, alpha and beta are read and out written once (16384 + 8192 +
# 128 + 8192). The layer's parameters (conv_w 131072, A_log, dt_bias and norm_w
# 768) are read once per launch.
DECODE_STATE_CONV_BYTES = 4_194_304 + 98_304
DECODE_IO_BYTES_PER_TOKEN = 32_896
DECODE_BYTES_PER_TOKEN_LAYER = DECODE_STATE_CONV_BYTES + DECODE_IO_BYTES_PER_TOKEN
DECODE_PARAM_BYTES_PER_LAUNCH = 131_840
# Multi-token decode (gdn_decode_multi): MULTI_T tokens per sequence per call,
# e.g. a speculative step. The state and conv_state cross HBM once per call, the
# per-token inputs and outputs once per token.
MULTI_T = 4
MULTI_TS = (2, 4, 8)        # the multi-token leg runs each; MULTI_T is the one the roofline object names
# Algorithmic FLOPs of the chunked prefill per token: the dense contractions
# K K^T and Q K^T once per K-head; T V, T (Gamma K), W S, Q S, the intra-chunk
# (M o Q K^T) V_new and the state update K^T V_new per V-head, with C=64.
PREFILL_FLOP_PER_TOKEN = 5_242_880

# Decode attention of the full-attention layers (gdn_attn_decode): the 10
# attention layers of the stack, each with its own bf16 KV cache, B=256
# sequences at a 4096-position context. Algorithmic bytes per call: the cache
# read once (B x 2 KV heads x ctx x 256 dims x 2 (K, V) x 2 B), q and z read and
# the bf16 output written once (3 x B x 16 x 256 x 2 B), ctx_len (B x 4 B).
ATTN_LAYERS, ATTN_CTX = 10, 4096
ATTN_BYTES_PER_CALL = BATCH * 2 * ATTN_CTX * 256 * 2 * 2 + 3 * BATCH * 16 * 256 * 2 + BATCH * 4
# Algorithmic bytes of one T=4096 bf16 prefill call: the per-token streams
# (32,896 B per token, as for decode), the final state (32 x 128 x 128 x 4) and
# conv_state (3 x 8192 x 2) written, the layer's parameters read.
PREFILL_IO_BYTES_PER_TOKEN = 32_896
PREFILL_END_STATE_BYTES = 2_097_152 + 49_152
PREFILL_PARAM_BYTES = 131_840

# Measured DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum, one ncu
# capture each, cold L2) per launch or per call, with the source file of the
# kernels it covers and that file's SHA-256 prefix at capture time. A figure
# whose source has changed since is reported as null: the counters no longer
# describe the kernel that ran. The summaries under profiles/ give the
# commands and the per-kernel split.
TRAFFIC = {
    "decode": dict(bytes=555_943_936 + 490_274_304, src="gdn_decode.cu", sha="76721eb1da31064e", profile="profiles/decode_step_kernel_B256.md",
                   per="launch of decode_step_kernel at B=256"),
    "attn": dict(bytes=2_168_676_864 + 18_318_080, src="gdn_attn.cu", sha="c68c58d38f8812f9", profile="profiles/attn_decode_B256_ctx4096.md",
                 per="call (attn_block_kernel + attn_combine_kernel) at B=256, ctx 4096"),
    "multi": dict(bytes=574_936_320 + 495_239_424, src="gdn_decode_multi.cu", sha="f4b811c1579705af", profile="profiles/decode_multi_kernel_B256_T4.md",
                  per="launch of decode_multi_kernel at B=256, T=4"),
    "prefill": dict(bytes=226_213_376 + 202_119_424, src="gdn_chunk.cu", sha="2a906081f77dc1ab", profile="profiles/chunk_prefill_T4096.md",
                    per="gdn_prefill call at T=4096 (all of its kernels)"),
    "varlen": dict(bytes=3_851_810_304 + 3_453_916_416, src="gdn_chunk.cu", sha="2a906081f77dc1ab", profile="profiles/chunk_prefill_varlen8.md",
                   per="gdn_prefill call on the 8-sequence varlen workload (all of its kernels)"),
    "in_proj": dict(bytes=109_801_728 + 76_413_184, src="gdn_gemm.cu", sha="e3474fe40a5549bd", profile="profiles/proj_gemm_M4096.md",
                    per="gdn_in_proj call at M=4096"),
    "out_proj": dict(bytes=50_358_016 + 100_096, src="gdn_gemm.cu", sha="e3474fe40a5549bd", profile="profiles/proj_gemm_M4096.md",
                     per="gdn_out_proj call at M=4096"),
    "gated_out_proj": dict(bytes=83_939_072 + 2_929_408, src="gdn_gated_proj.cu", sha="f20dfeb1dda1398b",
                           profile="profiles/gated_proj_M4096.md",
                           per="gdn_gated_out_proj call at M=4096"),
    "in_proj_conv_prefill": dict(bytes=279_962_112 + 257_320_960, src=("gdn_in_conv.cu", "gdn_chunk.cu"),
                                 sha="53f131d97d3c07f6", profile="profiles/in_proj_conv_T4096.md",
                                 per="gdn_in_proj_conv + gdn_prefill_xhat at T=4096 (all of their kernels)"),
    "out_proj_batch": dict(bytes=18_900_224 + 0, src="gdn_gemm.cu", sha="e3474fe40a5549bd", profile="profiles/proj_gemm_M4096.md",
                           per="gdn_out_proj call at M=256"),
}


def traffic(key):
    """(bytes, note) of a TRAFFIC entry: the bytes only while the kernel source
    is the one the counters were taken on."""
    import hashlib
    t = TRAFFIC[key]
    srcs = t["src"] if isinstance(t["src"], tuple) else (t["src"],)
    h = hashlib.sha256()
    try:
        for src in srcs:                              # one hash over the sources, in order
            with open(os.path.join(ROOT, "gated_deltanet_linear_02_gb300", "csrc", src), "rb") as f:
                h.update(f.read())
        sha = h.hexdigest()[:16]
    except OSError:
        sha = None
    if t["bytes"] is None:
        return None, f"not captured for this kernel version ({t['src']} sha {sha})"
    if sha != t["sha"]:
        return None, f"{t['src']} changed since the capture in {t['profile']} (sha {t['sha']} -> {sha})"
    return t["bytes"], f"ncu, per {t['per']}, {t['profile']}"


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    except (OSError, ValueError, KeyError, TypeError):     # absent or malformed: the recipe's fallback
        return 6800.0, 1900.0, 1700.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms while the GPU works."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.lines = []
        self.windows = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "200", "-i", str(self.idx)], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
            threading.Thread(target=self._read, daemon=True).start()
        except OSError:                                    # no nvidia-smi: no clock record
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, t0, t1):
        self.windows.append((t0, t1))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        rows = []
        for ts, line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((ts, float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        inside = [r for r in rows if any(a <= r[0] <= b for a, b in self.windows)]
        use = inside if inside else rows
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in use for i, v in enumerate(r[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in use), "sm_max_mhz": max(r[2] for r in use),
                "reasons": reasons, "samples": len(use), "in_timed_region": bool(inside)}


# ------------------------------------------------------------------ GPU arm

def setup_decode(torch, I, ops, dev, n_inputs):
    layers = []
    for layer in range(LAYERS):
        seed = I.seed_of(3, layer)
        lp = I.layer_params(seed).to(dev)
        conv, S = I.initial_states(seed, BATCH, torch.bfloat16, device=dev)
        st = I.streams(seed, BATCH, torch.bfloat16, device=dev, lead=(n_inputs,))
        out = torch.empty(BATCH, I.D_INNER, dtype=torch.bfloat16, device=dev)
        layers.append(dict(lp=lp, cp=ops.make_params(lp), conv=conv, S=S, st=st, out=out))
    return layers


def decode_step(ops, layers, i):
    for L in layers:
        st = L["st"]
        ops.decode_step(None, st.qkv[i], st.z[i], st.alpha[i], st.beta[i], L["conv"], L["S"], L["out"],
                        cparams=L["cp"])


def run_gpu(args, rank, world, dev):
    import torch
    import torch.distributed as dist

    from gated_deltanet_linear_02_gb300 import build as gbuild
    from gated_deltanet_linear_02_gb300 import inputs as I
    from gated_deltanet_linear_02_gb300 import ops

    if rank == 0 or not os.path.exists(ops.LIB_PATH):
        gbuild.build()
    if world > 1:
        dist.barrier()
    hbm_peak, tc_peak, tc_sust, peak_src = load_peaks()
    stream = torch.cuda.current_stream()
    sampler = ClockSampler(torch.cuda.current_device() if "CUDA_VISIBLE_DEVICES" not in os.environ
                           else int(os.environ["CUDA_VISIBLE_DEVICES"].split(",")[torch.cuda.current_device()]))
    sampler.start()

    def barrier_sync():
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    from gated_deltanet_linear_02_gb300.replicas import job_rate, slowest_ms

    def max_over_ranks(x: float) -> float:
        return slowest_ms(x, device=dev)

    # ---------------- decode @ B=256 over 30 layers (headline)
    n_inputs = 8
    layers = setup_decode(torch, I, ops, dev, n_inputs)
    for w in range(args.warmup):
        decode_step(ops, layers, w % n_inputs)
    barrier_sync()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_wall0 = time.time()
    ev0.record(stream)
    for k in range(args.steps):
        decode_step(ops, layers, k % n_inputs)
    ev1.record(stream)
    barrier_sync()
    sampler.mark(t_wall0, time.time())
    dec_ms = max_over_ranks(ev0.elapsed_time(ev1))
    launches = LAYERS * args.steps
    per_launch_s = dec_ms / 1e3 / launches
    bytes_per_launch = BATCH * DECODE_BYTES_PER_TOKEN_LAYER + DECODE_PARAM_BYTES_PER_LAUNCH
    achieved = bytes_per_launch / per_launch_s / 1e9
    dec_tok_s = job_rate(BATCH * args.steps, world, dec_ms)

    # ---------------- multi-token decode: T consecutive tokens per sequence
    #                  (gdn_decode_multi) through the same 30 layers and states
    mts = {}
    for MT in MULTI_TS:
        m_streams = [I.streams(I.seed_of(3, 100 + layer), MT, torch.bfloat16, device=dev, lead=(BATCH,))
                     for layer in range(LAYERS)]
        m_out = [torch.empty(BATCH, MT, I.D_INNER, dtype=torch.bfloat16, device=dev) for _ in range(LAYERS)]

        def multi_step():
            for L, ms, mo in zip(layers, m_streams, m_out):
                ops.decode_multi(None, ms.qkv, ms.z, ms.alpha, ms.beta, L["conv"], L["S"], mo, cparams=L["cp"])

        for _ in range(args.warmup):
            multi_step()
        barrier_sync()
        t_wall0 = time.time()
        ev0.record(stream)
        for _ in range(args.steps):
            multi_step()
        ev1.record(stream)
        barrier_sync()
        sampler.mark(t_wall0, time.time())
        mt_ms = max_over_ranks(ev0.elapsed_time(ev1))
        mt_launch_s = mt_ms / 1e3 / (LAYERS * args.steps)
        mt_bytes = BATCH * (DECODE_STATE_CONV_BYTES + MT * DECODE_IO_BYTES_PER_TOKEN) + DECODE_PARAM_BYTES_PER_LAUNCH
        mts[MT] = dict(tok_s=job_rate(BATCH * MT * args.steps, world, mt_ms), launch_s=mt_launch_s, bytes=mt_bytes,
                       achieved=mt_bytes / mt_launch_s / 1e9)
        assert ops.device_error() == ops.GDN_OK
        del m_streams, m_out
    mt = mts[MULTI_T]

    # ---------------- e2e: the same decode through the C ABI from pinned host buffers
    host_in = []
    for L in layers:
        st = L["st"]
        host_in.append([t[0].cpu().pin_memory() for t in (st.qkv, st.z, st.alpha, st.beta)])
    # Device inputs and host outputs are double-buffered by step parity, so that
    # step k's uploads and downloads overlap the kernels of neighbouring steps:
    # the upload stream fills the inputs of step k+1 while step k computes, and
    # the download stream drains step k's outputs while step k+1 computes. Each
    # stream waits on one event per step; the 30 kernels of a step run back to
    # back on the compute stream.
    dev_in = [[[torch.empty_like(t, device=dev) for t in h] for h in host_in] for _ in range(2)]
    dev_out = [[torch.empty(BATCH, I.D_INNER, dtype=torch.bfloat16, device=dev) for _ in layers] for _ in range(2)]
    host_out = [torch.empty(BATCH, I.D_INNER, dtype=torch.bfloat16).pin_memory() for _ in layers]
    h2d = sum(t.numel() * t.element_size() for h in host_in for t in h)
    d2h = sum(t.numel() * t.element_size() for t in host_out)
    up, down = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    uploaded = [torch.cuda.Event() for _ in range(2)]     # inputs of the step with this parity are in
    computed = [torch.cuda.Event() for _ in range(2)]     # kernels of the step with this parity are done
    downloaded = [torch.cuda.Event() for _ in range(2)]   # outputs of the step with this parity are out

    def upload(k):
        up.wait_event(computed[k % 2])                     # step k-2 has finished reading these buffers
        with torch.cuda.stream(up):
            for h, d in zip(host_in, dev_in[k % 2]):
                for src, dst in zip(h, d):
                    dst.copy_(src, non_blocking=True)
            uploaded[k % 2].record(up)

    def e2e_step(k):
        upload(k + 1)
        stream.wait_event(uploaded[k % 2])
        stream.wait_event(downloaded[k % 2])               # step k-2's outputs have left these buffers
        for L, d, o in zip(layers, dev_in[k % 2], dev_out[k % 2]):
            ops.decode_step(None, d[0], d[1], d[2], d[3], L["conv"], L["S"], o, cparams=L["cp"], stream=stream)
        computed[k % 2].record(stream)
        down.wait_event(computed[k % 2])
        with torch.cuda.stream(down):
            for o, ho in zip(dev_out[k % 2], host_out):
                ho.copy_(o, non_blocking=True)
            downloaded[k % 2].record(down)

    upload(0)
    for k in range(max(1, args.warmup)):
        e2e_step(k)
    barrier_sync()
    k0 = max(1, args.warmup)
    ev0.record(stream)
    up.wait_event(ev0)
    down.wait_event(ev0)
    for k in range(k0, k0 + args.steps):
        e2e_step(k)
    stream.wait_stream(up)
    stream.wait_stream(down)
    ev1.record(stream)
    barrier_sync()
    e2e_ms = max_over_ranks(ev0.elapsed_time(ev1))
    e2e_tok_s = job_rate(BATCH * args.steps, world, e2e_ms)
    del layers, host_in, dev_in, dev_out, host_out
    torch.cuda.empty_cache()

    # ---------------- prefill @ T=4096 (bf16, zero initial state)
    seed = I.seed_of(2)
    lp = I.layer_params(seed).to(dev)
    cp = ops.make_params(lp)
    st = I.streams(seed, PREFILL_T, torch.bfloat16, device=dev)
    cu = I.cu_seqlens([PREFILL_T]).to(dev)
    out = torch.empty(PREFILL_T, I.D_INNER, dtype=torch.bfloat16, device=dev)
    cs_out = torch.empty(1, I.KCONV - 1, I.C_CONV, dtype=torch.bfloat16, device=dev)
    S_out = torch.empty(1, I.HV, I.DV, I.DK, dtype=torch.float32, device=dev)
    ws = torch.empty(ops.prefill_workspace_size(1, PREFILL_T, torch.bfloat16, 0), dtype=torch.uint8, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)      # > L2 (129 MB)

    def prefill_call():
        ops.prefill(None, st.qkv, st.z, st.alpha, st.beta, cu, out, None, cs_out, None, S_out, chunk_size=0,
                    workspace=ws, cparams=cp)

    for _ in range(args.warmup):
        prefill_call()
    barrier_sync()
    times = []
    t_wall0 = time.time()
    for _ in range(args.steps):
        flush.fill_(1)                                   # evict L2 between timed calls
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        prefill_call()
        b.record(stream)
        times.append((a, b))
    barrier_sync()
    sampler.mark(t_wall0, time.time())
    pf_ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in times) / len(times))
    assert ops.device_error() == ops.GDN_OK
    pf_tok_s = job_rate(PREFILL_T, world, pf_ms)
    pf_tflops = PREFILL_FLOP_PER_TOKEN * PREFILL_T / (pf_ms / 1e3) / 1e12
    # ---------------- ssm_out projection (gdn_out_proj, tcgen05 GEMM) at the prefill
    #                  size and the decode batch, L2 flushed between timed calls
    w_out = I.out_proj_weight(I.seed_of(2), device=dev)
    op = {}
    for M in (PREFILL_T, BATCH):
        xo = torch.randn(M, I.D_INNER, device=dev).to(torch.bfloat16)
        yo = torch.empty(M, I.N_EMBD, dtype=torch.bfloat16, device=dev)
        for _ in range(args.warmup):
            ops.out_proj(xo, w_out, yo)
        barrier_sync()
        times = []
        t_wall0 = time.time()
        for _ in range(args.steps):
            flush.fill_(1)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            ops.out_proj(xo, w_out, yo)
            b.record(stream)
            times.append((a, b))
        barrier_sync()
        sampler.mark(t_wall0, time.time())
        ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in times) / len(times))
        ob = I.N_EMBD * I.D_INNER * 2 + M * I.D_INNER * 2 + M * I.N_EMBD * 2
        op[M] = dict(us=ms * 1e3, tflops=2.0 * M * I.D_INNER * I.N_EMBD / (ms / 1e3) / 1e12,
                     bytes=ob, gbs=ob / (ms / 1e3) / 1e9)
        # the same projection with the gated norm formed inside the GEMM
        # (gdn_gated_out_proj), from the mixer's y and z
        zo = torch.randn(M, I.D_INNER, device=dev).to(torch.bfloat16)
        for _ in range(args.warmup):
            ops.gated_out_proj(lp.norm_w, lp.norm_eps, xo, zo, w_out, yo)
        barrier_sync()
        times = []
        t_wall0 = time.time()
        for _ in range(args.steps):
            flush.fill_(1)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            ops.gated_out_proj(lp.norm_w, lp.norm_eps, xo, zo, w_out, yo)
            b.record(stream)
            times.append((a, b))
        barrier_sync()
        sampler.mark(t_wall0, time.time())
        gms = max_over_ranks(sum(a.elapsed_time(b) for a, b in times) / len(times))
        gb = ob + M * I.D_INNER * 2
        op[M]["gated"] = dict(us=gms * 1e3, tflops=2.0 * M * I.D_INNER * I.N_EMBD / (gms / 1e3) / 1e12,
                              bytes=gb, gbs=gb / (gms / 1e3) / 1e9)
        del xo, yo, zo
    # ---------------- input projections (gdn_in_proj) at the prefill size
    w_in = torch.cat(I.in_proj_weights(I.seed_of(2), device=dev), dim=0)
    h_in = torch.randn(PREFILL_T, I.N_EMBD, device=dev).to(torch.bfloat16)
    outs_in = [torch.empty(PREFILL_T, n, dtype=torch.bfloat16, device=dev) for n in (I.C_CONV, I.D_INNER, I.HV, I.HV)]
    for _ in range(args.warmup):
        ops.in_proj(h_in, w_in, *outs_in)
    barrier_sync()
    times = []
    t_wall0 = time.time()
    for _ in range(args.steps):
        flush.fill_(1)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        ops.in_proj(h_in, w_in, *outs_in)
        b.record(stream)
        times.append((a, b))
    barrier_sync()
    sampler.mark(t_wall0, time.time())
    ip_ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in times) / len(times))
    ip_bytes = (PREFILL_T * I.N_EMBD + w_in.shape[0] * I.N_EMBD + PREFILL_T * w_in.shape[0]) * 2
    ip = dict(us=ip_ms * 1e3, tflops=2.0 * PREFILL_T * w_in.shape[0] * I.N_EMBD / (ip_ms / 1e3) / 1e12,
              bytes=ip_bytes, gbs=ip_bytes / (ip_ms / 1e3) / 1e9)
    # ---------------- projections + mixer at T=4096: gdn_in_proj then gdn_prefill, against
    #                  gdn_in_proj_conv (conv, SiLU and q/k norms in the GEMM's epilogue)
    #                  then gdn_prefill_xhat; L2 flushed between calls
    xh = torch.empty(PREFILL_T, I.C_CONV, dtype=torch.float16, device=dev)

    def unfused():
        ops.in_proj(h_in, w_in, *outs_in)
        ops.prefill(None, outs_in[0], outs_in[1], outs_in[2], outs_in[3], cu, out, None, cs_out, None, S_out,
                    chunk_size=0, workspace=ws, cparams=cp)

    def fused():
        ops.in_proj_conv(None, h_in, w_in, cu, xh, outs_in[1], outs_in[2], outs_in[3], conv_state_out=cs_out,
                         cparams=cp)
        ops.prefill_xhat(None, xh, outs_in[1], outs_in[2], outs_in[3], cu, out, ssm_state_out=S_out, workspace=ws,
                         cparams=cp)

    f2 = {}
    for name, fn in (("unfused", unfused), ("fused", fused)):
        for _ in range(args.warmup):
            fn()
        barrier_sync()
        times = []
        t_wall0 = time.time()
        for _ in range(args.steps):
            flush.fill_(1)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            times.append((a, b))
        barrier_sync()
        sampler.mark(t_wall0, time.time())
        f2[name] = max_over_ranks(sum(a.elapsed_time(b) for a, b in times) / len(times)) * 1e3
    assert ops.device_error() == ops.GDN_OK
    del xh
    del w_in, h_in, outs_in
    assert ops.device_error() == ops.GDN_OK
    torch.cuda.empty_cache()
    # ---------------- decode attention of the 10 full-attention layers (gdn_attn_decode)
    att = [I.attn_inputs(I.seed_of(5, layer), BATCH, ATTN_CTX, device=dev) for layer in range(ATTN_LAYERS)]
    att_out = [torch.empty(BATCH, 16, 256, dtype=torch.bfloat16, device=dev) for _ in range(ATTN_LAYERS)]
    att_ws = torch.empty(ops.attn_decode_workspace_size(BATCH, ATTN_CTX), dtype=torch.uint8, device=dev)

    def attn_step():
        for a_in, a_out in zip(att, att_out):
            ops.attn_decode(a_in.q, a_in.k_cache, a_in.v_cache, a_in.ctx_len, a_in.z, a_out, workspace=att_ws)

    for _ in range(args.warmup):
        attn_step()
    barrier_sync()
    t_wall0 = time.time()
    ev0.record(stream)
    for _ in range(args.steps):
        attn_step()
    ev1.record(stream)
    barrier_sync()
    sampler.mark(t_wall0, time.time())
    at_ms = max_over_ranks(ev0.elapsed_time(ev1))
    at_call_s = at_ms / 1e3 / (ATTN_LAYERS * args.steps)
    at = dict(tok_s=job_rate(BATCH * args.steps, world, at_ms), call_s=at_call_s,
              achieved=ATTN_BYTES_PER_CALL / at_call_s / 1e9)
    assert ops.device_error() == ops.GDN_OK
    del att, att_out, att_ws
    torch.cuda.empty_cache()
    cfgs = other_configs(args, torch, I, ops, dev, stream, flush, barrier_sync, max_over_ranks, sampler,
                         hbm_peak, tc_peak)
    clocks = sampler.stop()

    return dict(cfgs=cfgs, at=at, ip=ip, op=op, mt=mt, mts=mts, f2=f2, dec_ms=dec_ms, dec_tok_s=dec_tok_s, achieved=achieved, per_launch_s=per_launch_s,
                bytes_per_launch=bytes_per_launch, launches=launches, e2e_tok_s=e2e_tok_s, e2e_ms=e2e_ms,
                h2d=h2d, d2h=d2h, pf_ms=pf_ms, pf_tok_s=pf_tok_s, pf_tflops=pf_tflops, hbm_peak=hbm_peak,
                tc_peak=tc_peak, peak_src=peak_src, clocks=clocks)


def other_configs(args, torch, I, ops, dev, stream, flush, barrier_sync, max_over_ranks, sampler, hbm_peak, tc_peak):
    """The other configurations of the metric, timed beside the headline:
    0) one layer, T=64, fp32, zero states: the prefill (exact scan) and 64
       decode steps; 1) one layer, B=64, 128 sequential decode steps, bf16;
    4) the varlen prefill of 8 sequences (seeded log-uniform lengths in
    [256, 32768]), bf16, random initial states. L2 is flushed before every
    timed call. The decode loops are also timed as a CUDA graph, which takes
    the host's launch cost out of these small, launch-bound steps."""
    reps = max(3, min(args.steps, 10))

    def time_calls(fn):
        for _ in range(2):
            fn()
        barrier_sync()
        times = []
        t_wall0 = time.time()
        for _ in range(reps):
            flush.fill_(1)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            times.append((a, b))
        barrier_sync()
        sampler.mark(t_wall0, time.time())
        return max_over_ranks(sum(a.elapsed_time(b) for a, b in times) / len(times))   # ms per call

    def capture(fn):
        # the library's calls only enqueue work (no synchronisation, no allocation),
        # so a sequence of them records into a CUDA graph as it stands
        side = torch.cuda.Stream(device=dev)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            fn()                                       # warm the lazy set-up outside the capture
        stream.wait_stream(side)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        torch.cuda.synchronize()
        return g

    out = {}
    # ---- config 0
    seed = I.seed_of(0)
    lp = I.layer_params(seed).to(dev)
    cp = ops.make_params(lp)
    st = I.streams(seed, 64, torch.float32, device=dev)
    cu = I.cu_seqlens([64]).to(dev)
    o = torch.empty(64, I.D_INNER, device=dev)
    ws = torch.empty(max(ops.prefill_workspace_size(1, 64, torch.float32, 0), 256), dtype=torch.uint8, device=dev)
    pf_ms = time_calls(lambda: ops.prefill(None, st.qkv, st.z, st.alpha, st.beta, cu, o, workspace=ws, cparams=cp))
    conv, S = I.initial_states(seed, 1, torch.float32, device=dev, zero=True)
    sd = I.streams(seed, 1, torch.float32, device=dev, lead=(64,))
    od = torch.empty(1, I.D_INNER, device=dev)

    def dec0():
        for k in range(64):
            ops.decode_step(None, sd.qkv[k], sd.z[k], sd.alpha[k], sd.beta[k], conv, S, od, cparams=cp)
    dec_ms = time_calls(dec0)
    g0 = capture(dec0)
    dec_g_ms = time_calls(g0.replay)
    out["T64_fp32"] = {"prefill_us_per_call": pf_ms * 1e3, "decode_64_steps_us": dec_ms * 1e3,
                       "decode_us_per_step": dec_ms * 1e3 / 64,
                       "decode_us_per_step_cuda_graph": dec_g_ms * 1e3 / 64, "bound": "latency"}
    del g0
    # ---- config 1
    seed = I.seed_of(1)
    lp = I.layer_params(seed).to(dev)
    cp = ops.make_params(lp)
    conv, S = I.initial_states(seed, 64, torch.bfloat16, device=dev)
    sd = I.streams(seed, 64, torch.bfloat16, device=dev, lead=(128,))
    od = torch.empty(64, I.D_INNER, dtype=torch.bfloat16, device=dev)

    def dec1():
        for k in range(128):
            ops.decode_step(None, sd.qkv[k], sd.z[k], sd.alpha[k], sd.beta[k], conv, S, od, cparams=cp)
    ms = time_calls(dec1)
    g1 = capture(dec1)
    ms_g = time_calls(g1.replay)
    del g1
    step_s = ms / 1e3 / 128
    gbs = (64 * DECODE_BYTES_PER_TOKEN_LAYER + DECODE_PARAM_BYTES_PER_LAUNCH) / step_s / 1e9
    out["decode_B64_128_steps_bf16"] = {"value": 64 * 128 / (ms / 1e3), "unit": "tok/s (one layer)",
                                        "us_per_step": step_s * 1e6, "achieved_GBs": gbs,
                                        "us_per_step_cuda_graph": ms_g * 1e3 / 128,
                                        "note": "state 128 MiB, about the size of L2: steps after the "
                                                "first find part of it there"}
    del conv, S, sd, od
    # ---- config 4
    seed = I.seed_of(4)
    lens = I.varlen_lengths(seed)
    T4 = sum(lens)
    lp = I.layer_params(seed).to(dev)
    cp = ops.make_params(lp)
    st = I.streams(seed, T4, torch.bfloat16, device=dev)
    conv, S = I.initial_states(seed, len(lens), torch.bfloat16, device=dev)
    cu = I.cu_seqlens(lens).to(dev)
    o = torch.empty(T4, I.D_INNER, dtype=torch.bfloat16, device=dev)
    cout, sout = torch.empty_like(conv), torch.empty_like(S)
    ws = torch.empty(ops.prefill_workspace_size(len(lens), T4, torch.bfloat16, 0), dtype=torch.uint8, device=dev)
    ms = time_calls(lambda: ops.prefill(None, st.qkv, st.z, st.alpha, st.beta, cu, o, conv, cout, S, sout,
                                        workspace=ws, cparams=cp))
    tflops = PREFILL_FLOP_PER_TOKEN * T4 / (ms / 1e3) / 1e12
    # streams, states in and out, parameters
    io = T4 * PREFILL_IO_BYTES_PER_TOKEN + len(lens) * DECODE_STATE_CONV_BYTES + PREFILL_PARAM_BYTES
    tr, tr_note = traffic("varlen")
    out["varlen_prefill_8seq_bf16"] = {"lengths": lens, "tokens": T4, "value": T4 / (ms / 1e3), "unit": "tok/s",
                                       "ms_per_call": ms, "tflops": tflops,
                                       "io_GBs": io / (ms / 1e3) / 1e9,
                                       "roofline": {"bound": "tensor", "achieved": tflops, "peak": tc_peak,
                                                    "unit": "TFLOP/s", "frac": tflops / tc_peak,
                                                    "hbm_achieved_GBs": io / (ms / 1e3) / 1e9,
                                                    "hbm_frac": io / (ms / 1e3) / 1e9 / hbm_peak,
                                                    "frac_of_nominal_8TBs": io / (ms / 1e3) / 1e9 / NOMINAL_HBM_GBS,
                                                    "algorithmic_flop_per_call": PREFILL_FLOP_PER_TOKEN * T4,
                                                    "algorithmic_bytes_per_call": io,
                                                    "traffic": tr, "traffic_source": tr_note}}
    del st, conv, S, o, cout, sout, ws
    assert ops.device_error() == ops.GDN_OK
    return out


# ------------------------------------------------------------- CPU oracle

def oracle_decode_sample(n_seq: int, threads: int):
    """The fp64 oracle on a bounded sample of the decode workload: one token for
    n_seq sequences through all 30 layers (each layer with its own seeded
    parameters and random states), threads over sequences. Returns (seconds, tokens)."""
    import numpy as np
    import torch
    from concurrent.futures import ThreadPoolExecutor

    from gated_deltanet_linear_02_gb300 import inputs as I
    from oracle import oracle

    # Timing does not depend on the values, so a few distinct sequences per
    # layer stand in for all n_seq (the oracle copies its inputs on every call).
    nd = min(n_seq, 4)
    per_layer = []
    for layer in range(LAYERS):
        seed = I.seed_of(3, layer)
        lp = I.layer_params(seed)
        P = oracle.Params.of(lp.conv_w, lp.A_log, lp.dt_bias, lp.norm_w, lp.l2_eps, lp.norm_eps)
        conv, S = I.initial_states(seed, nd, torch.bfloat16)
        st = I.streams(seed, nd, torch.bfloat16)
        per_layer.append((P, conv.double().numpy(), np.swapaxes(S.double().numpy(), -1, -2).copy(),
                          [t.double().numpy() for t in (st.qkv, st.z, st.alpha, st.beta)]))

    def one_seq(b):
        b %= nd
        for P, conv, S, (qkv, z, al, be) in per_layer:
            oracle.gdn_sequence(P, qkv[b:b + 1], z[b:b + 1], al[b:b + 1], be[b:b + 1], conv[b], S[b])

    t0 = time.perf_counter()
    with ThreadPoolExecutor(max_workers=threads) as ex:
        list(ex.map(one_seq, range(n_seq)))
    return time.perf_counter() - t0, n_seq


def host_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):                      # no affinity call on this platform
        return os.cpu_count() or 1


def cpu_baseline(n_seq=None):
    from oracle import oracle
    oracle.build()
    threads = host_threads()
    n_seq = n_seq or BATCH                # one whole decode step: ~1 s wall on 16 cores
    secs, toks = oracle_decode_sample(n_seq, threads)
    secs1, toks1 = oracle_decode_sample(8, 1)     # one core, on a smaller sample
    return {"value": toks / secs, "unit": "tok/s", "cores": threads, "kind": "oracle",
            "sample": f"one decode token through all 30 layers for {n_seq} of the {BATCH} sequences "
                      f"(fp64 oracle, {threads} threads over sequences), {secs:.1f} s wall, "
                      f"{secs * threads:.0f} core-seconds",
            "value_one_core": toks1 / secs1,
            "sample_one_core": f"the same for 8 sequences on 1 thread, {secs1:.1f} s"}


# ------------------------------------------------------------------- main

def profile_case(args):
    """A small, self-contained run of one path for profilers: no JSON line, no
    clocks, a few launches on a few GB. ``--case decode``: --layers layers of
    gdn_decode_step on --batch sequences; ``--case multi``: the same with
    gdn_decode_multi, --mt tokens per sequence; ``--case prefill``: gdn_prefill on one
    sequence of --T tokens; ``--case out_proj`` / ``--case in_proj``: the
    projection GEMMs on --T rows; ``--case attn``: gdn_attn_decode on --batch
    sequences with a --T position context; ``--case varlen``: gdn_prefill on
    the 8-sequence varlen workload; ``--case gated_out_proj``: the fused gated
    norm + ssm_out GEMM on --T rows; ``--case in_proj_conv``: gdn_in_proj_conv
    then gdn_prefill_xhat on --T tokens."""
    import torch

    from gated_deltanet_linear_02_gb300 import build as gbuild
    from gated_deltanet_linear_02_gb300 import inputs as I
    from gated_deltanet_linear_02_gb300 import ops
    gbuild.build()
    dev = torch.device("cuda", 0)
    n = args.warmup + args.steps
    if args.case == "decode":
        Ls = []
        for layer in range(args.layers):
            seed = I.seed_of(3, layer)
            lp = I.layer_params(seed).to(dev)
            conv, S = I.initial_states(seed, args.batch, torch.bfloat16, device=dev)
            st = I.streams(seed, args.batch, torch.bfloat16, device=dev, lead=(1,))
            out = torch.empty(args.batch, I.D_INNER, dtype=torch.bfloat16, device=dev)
            Ls.append((ops.make_params(lp), conv, S, st, out))
        for _ in range(n):
            for cp, conv, S, st, out in Ls:
                ops.decode_step(None, st.qkv[0], st.z[0], st.alpha[0], st.beta[0], conv, S, out, cparams=cp)
    elif args.case == "out_proj":
        w = I.out_proj_weight(I.seed_of(2), device=dev)
        x = torch.randn(args.T, I.D_INNER, device=dev).to(torch.bfloat16)
        y = torch.empty(args.T, I.N_EMBD, dtype=torch.bfloat16, device=dev)
        for _ in range(n):
            ops.out_proj(x, w, y)
        assert ops.device_error() == ops.GDN_OK
    elif args.case == "multi":
        Ls = []
        for layer in range(args.layers):
            seed = I.seed_of(3, layer)
            lp = I.layer_params(seed).to(dev)
            conv, S = I.initial_states(seed, args.batch, torch.bfloat16, device=dev)
            st = I.streams(seed, args.mt, torch.bfloat16, device=dev, lead=(args.batch,))
            out = torch.empty(args.batch, args.mt, I.D_INNER, dtype=torch.bfloat16, device=dev)
            Ls.append((ops.make_params(lp), conv, S, st, out))
        for _ in range(n):
            for cp, conv, S, st, out in Ls:
                ops.decode_multi(None, st.qkv, st.z, st.alpha, st.beta, conv, S, out, cparams=cp)
        assert ops.device_error() == ops.GDN_OK
    elif args.case == "attn":
        a_in = I.attn_inputs(I.seed_of(5), args.batch, args.T, device=dev)
        out = torch.empty(args.batch, 16, 256, dtype=torch.bfloat16, device=dev)
        for _ in range(n):
            ops.attn_decode(a_in.q, a_in.k_cache, a_in.v_cache, a_in.ctx_len, a_in.z, out)
        assert ops.device_error() == ops.GDN_OK
    elif args.case == "in_proj":
        w_in = torch.cat(I.in_proj_weights(I.seed_of(2), device=dev), dim=0)
        h = torch.randn(args.T, I.N_EMBD, device=dev).to(torch.bfloat16)
        outs = [torch.empty(args.T, m, dtype=torch.bfloat16, device=dev) for m in (I.C_CONV, I.D_INNER, I.HV, I.HV)]
        for _ in range(n):
            ops.in_proj(h, w_in, *outs)
        assert ops.device_error() == ops.GDN_OK
    elif args.case == "gated_out_proj":
        w = I.out_proj_weight(I.seed_of(2), device=dev)
        lp = I.layer_params(I.seed_of(2)).to(dev)
        y = torch.randn(args.T, I.D_INNER, device=dev).to(torch.bfloat16)
        z = torch.randn(args.T, I.D_INNER, device=dev).to(torch.bfloat16)
        o = torch.empty(args.T, I.N_EMBD, dtype=torch.bfloat16, device=dev)
        for _ in range(n):
            ops.gated_out_proj(lp.norm_w, lp.norm_eps, y, z, w, o)
        assert ops.device_error() == ops.GDN_OK
    elif args.case == "in_proj_conv":
        # gdn_in_proj_conv then gdn_prefill_xhat on one sequence of --T tokens
        w_in = torch.cat(I.in_proj_weights(I.seed_of(2), device=dev), dim=0)
        lp = I.layer_params(I.seed_of(2)).to(dev)
        h = torch.randn(args.T, I.N_EMBD, device=dev).to(torch.bfloat16)
        cu = I.cu_seqlens([args.T]).to(dev)
        xh = torch.empty(args.T, I.C_CONV, dtype=torch.float16, device=dev)
        z, al, be = (torch.empty(args.T, c, dtype=torch.bfloat16, device=dev) for c in (I.D_INNER, I.HV, I.HV))
        cs = torch.empty(1, I.KCONV - 1, I.C_CONV, dtype=torch.bfloat16, device=dev)
        out = torch.empty(args.T, I.D_INNER, dtype=torch.bfloat16, device=dev)
        S = torch.empty(1, I.HV, I.DV, I.DK, device=dev)
        ws = None
        for _ in range(n):
            ops.in_proj_conv(lp, h, w_in, cu, xh, z, al, be, conv_state_out=cs)
            ws = ops.prefill_xhat(lp, xh, z, al, be, cu, out, ssm_state_out=S, workspace=ws)
        assert ops.device_error() == ops.GDN_OK
    elif args.case == "varlen":
        seed = I.seed_of(4)
        lens = I.varlen_lengths(seed)
        T4 = sum(lens)
        lp = I.layer_params(seed).to(dev)
        st = I.streams(seed, T4, torch.bfloat16, device=dev)
        conv, S = I.initial_states(seed, len(lens), torch.bfloat16, device=dev)
        cu = I.cu_seqlens(lens).to(dev)
        out = torch.empty(T4, I.D_INNER, dtype=torch.bfloat16, device=dev)
        cout, sout = torch.empty_like(conv), torch.empty_like(S)
        ws = torch.empty(ops.prefill_workspace_size(len(lens), T4, torch.bfloat16, 0), dtype=torch.uint8, device=dev)
        for _ in range(n):
            ops.prefill(lp, st.qkv, st.z, st.alpha, st.beta, cu, out, conv, cout, S, sout, workspace=ws)
        assert ops.device_error() == ops.GDN_OK
    else:
        seed = I.seed_of(2)
        lp = I.layer_params(seed).to(dev)
        st = I.streams(seed, args.T, torch.bfloat16, device=dev)
        cu = I.cu_seqlens([args.T]).to(dev)
        out = torch.empty(args.T, I.D_INNER, dtype=torch.bfloat16, device=dev)
        S_out = torch.empty(1, I.HV, I.DV, I.DK, device=dev)
        ws = torch.empty(ops.prefill_workspace_size(1, args.T, torch.bfloat16, args.chunk), dtype=torch.uint8,
                         device=dev)
        for _ in range(n):
            ops.prefill(lp, st.qkv, st.z, st.alpha, st.beta, cu, out, ssm_state_out=S_out,
                        chunk_size=args.chunk, workspace=ws)
        assert ops.device_error() == ops.GDN_OK
    torch.cuda.synchronize()
    print(f"profile case {args.case} done: {n} iterations")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--case", choices=["decode", "multi", "prefill", "varlen", "out_proj", "in_proj", "attn",
                                       "gated_out_proj", "in_proj_conv"],
                    default=None,
                    help="profiling run of one path (see profile_case); prints no JSON line")
    ap.add_argument("--batch", type=int, default=64)
    ap.add_argument("--layers", type=int, default=1)
    ap.add_argument("--T", type=int, default=4096)
    ap.add_argument("--chunk", type=int, default=0)
    ap.add_argument("--mt", type=int, default=MULTI_T, help="tokens per sequence of --case multi")
    args = ap.parse_args()
    if args.case is not None:
        profile_case(args)
        return
    if args.warmup < 3:
        args.warmup = 3

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank != 0:
            return
        from oracle import oracle
        oracle.build()
        threads = host_threads()
        n_seq = max(16, 2 * threads)
        for _ in range(args.warmup):
            oracle_decode_sample(n_seq, threads)
        tot_s = tot_tok = 0.0
        for _ in range(args.steps):
            s, t = oracle_decode_sample(n_seq, threads)
            tot_s += s
            tot_tok += t
        v = tot_tok / tot_s
        line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "tok/s", "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": tot_s / args.steps * 1e3,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic",
                "config": {"workload": "decode_30L_B256_bf16", "layers": LAYERS, "batch": BATCH,
                           "parallelism": "replicas"},
                "cpu_baseline": {"value": v, "unit": "tok/s", "cores": threads, "kind": "oracle",
                                 "sample": f"per step: one decode token through all 30 layers for {n_seq} "
                                           f"sequences, {threads} threads"},
                "e2e": {"value": v, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    import torch
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    r = run_gpu(args, rank, world, dev)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    if rank != 0:
        return
    frac = r["achieved"] / r["hbm_peak"]
    dec_tr, dec_tr_note = traffic("decode")
    at_tr, at_tr_note = traffic("attn")
    mt_tr, mt_tr_note = traffic("multi")
    pf_tr, pf_tr_note = traffic("prefill")
    ip_tr, ip_tr_note = traffic("in_proj")
    op_tr, op_tr_note = traffic("out_proj")
    opb_tr, opb_tr_note = traffic("out_proj_batch")
    gp_tr, gp_tr_note = traffic("gated_out_proj")
    f2_tr, f2_tr_note = traffic("in_proj_conv_prefill")
    PREFILL_BYTES = PREFILL_T * PREFILL_IO_BYTES_PER_TOKEN + PREFILL_END_STATE_BYTES + PREFILL_PARAM_BYTES
    pf_gbs = PREFILL_BYTES / (r["pf_ms"] / 1e3) / 1e9
    line = {
        "metric": METRIC, "value": r["dec_tok_s"], "unit": "tok/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": r["dec_ms"] / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": "decode_30L_B256_bf16", "layers": LAYERS, "batch": BATCH,
                   "activations": "bf16", "state": "fp32", "parallelism": f"replicas x{world}",
                   "l2": "inputs larger than L2 (15 GiB of state touched per step)"},
        "roofline": {"bound": "hbm", "achieved": r["achieved"], "peak": r["hbm_peak"], "unit": "GB/s",
                     "frac": frac, "traffic": dec_tr, "traffic_source": dec_tr_note,
                     "kernel": "decode_step_kernel<bf16,bf16>",
                     "peak_source": f"{r['peak_src']} (MEASURED_PEAKS.json hbm_gbs)" if r["peak_src"] == "measured"
                     else "fallback 6.8 TB/s",
                     "algorithmic_bytes_per_launch": r["bytes_per_launch"],
                     "launch_us": r["per_launch_s"] * 1e6,
                     "frac_of_nominal_8TBs": r["achieved"] / NOMINAL_HBM_GBS},
        "cpu_baseline": cpu,
        "e2e": {"value": r["e2e_tok_s"], "unit": "tok/s", "h2d_bytes_per_step": r["h2d"],
                "d2h_bytes_per_step": r["d2h"], "ms_per_step": r["e2e_ms"] / args.steps},
        "gpu_launches": r["launches"],
        "clocks": r["clocks"],
        "prefill": {"workload": "prefill_T4096_bf16", "value": r["pf_tok_s"], "unit": "tok/s",
                    "ms_per_call": r["pf_ms"], "l2": "flushed between timed calls",
                    "roofline": {"bound": "tensor", "achieved": r["pf_tflops"], "peak": r["tc_peak"],
                                 "unit": "TFLOP/s", "frac": r["pf_tflops"] / r["tc_peak"],
                                 "hbm_achieved_GBs": pf_gbs, "hbm_frac": pf_gbs / r["hbm_peak"],
                                 "frac_of_nominal_8TBs": pf_gbs / NOMINAL_HBM_GBS,
                                 "algorithmic_flop_per_call": PREFILL_FLOP_PER_TOKEN * PREFILL_T,
                                 "algorithmic_bytes_per_call": PREFILL_BYTES,
                                 "traffic": pf_tr, "traffic_source": pf_tr_note,
                                 "timed": "whole gdn_prefill call (plan, activation, the cooperative prep + chain + "
                                          "gated norm kernel, conv_state kernels)"}},
        "in_proj": {"workload": f"input_projections_M{PREFILL_T}_bf16", "op": "qkv|z|alpha|beta = h w_in^T, 2048 -> 12352",
                    "us_per_call": r["ip"]["us"], "l2": "flushed between timed calls",
                    "roofline": {"bound": "tensor", "achieved": r["ip"]["tflops"], "peak": r["tc_peak"],
                                 "unit": "TFLOP/s", "frac": r["ip"]["tflops"] / r["tc_peak"],
                                 "hbm_achieved_GBs": r["ip"]["gbs"], "hbm_frac": r["ip"]["gbs"] / r["hbm_peak"],
                                 "algorithmic_bytes_per_call": r["ip"]["bytes"],
                                 "traffic": ip_tr, "traffic_source": ip_tr_note}},
        "in_proj_conv_prefill": {
            "workload": f"input_projections_and_prefill_T{PREFILL_T}_bf16",
            "op": "h -> qkv|z|alpha|beta -> mixer output: gdn_in_proj + gdn_prefill against "
                  "gdn_in_proj_conv (conv, SiLU, q/k norms in the GEMM epilogue) + gdn_prefill_xhat",
            "us_per_call_unfused": r["f2"]["unfused"], "us_per_call_fused": r["f2"]["fused"],
            "hbm_bytes_saved_per_call": 2 * PREFILL_T * I_C_CONV * 2,
            "traffic_fused": f2_tr, "traffic_fused_source": f2_tr_note,
            "traffic_unfused": (None if ip_tr is None or pf_tr is None else ip_tr + pf_tr),
            "bytes_saved": "the raw q|k|v stream [T][8192] bf16, written by the projection and read back "
                           "by the mixer's conv", "l2": "flushed between timed calls"},
        "out_proj": {"workload": f"ssm_out_projection_M{PREFILL_T}_bf16", "op": "y = x w^T, 4096 -> 2048",
                     "us_per_call": r["op"][PREFILL_T]["us"], "l2": "flushed between timed calls",
                     "roofline": {"bound": "tensor", "achieved": r["op"][PREFILL_T]["tflops"], "peak": r["tc_peak"],
                                  "unit": "TFLOP/s", "frac": r["op"][PREFILL_T]["tflops"] / r["tc_peak"],
                                  "hbm_achieved_GBs": r["op"][PREFILL_T]["gbs"],
                                  "hbm_frac": r["op"][PREFILL_T]["gbs"] / r["hbm_peak"],
                                  "algorithmic_bytes_per_call": r["op"][PREFILL_T]["bytes"],
                                  "traffic": op_tr, "traffic_source": op_tr_note},
                     "gated_out_proj": {
                         "op": "out = (gated RMSNorm(y) . silu(z)) w^T, the norm formed inside the GEMM",
                         "us_per_call": {str(m): r["op"][m]["gated"]["us"] for m in (PREFILL_T, BATCH)},
                         "roofline": {"bound": "tensor", "achieved": r["op"][PREFILL_T]["gated"]["tflops"],
                                      "peak": r["tc_peak"], "unit": "TFLOP/s",
                                      "frac": r["op"][PREFILL_T]["gated"]["tflops"] / r["tc_peak"],
                                      "hbm_achieved_GBs": r["op"][PREFILL_T]["gated"]["gbs"],
                                      "hbm_frac": r["op"][PREFILL_T]["gated"]["gbs"] / r["hbm_peak"],
                                      "algorithmic_bytes_per_call": r["op"][PREFILL_T]["gated"]["bytes"],
                                      "traffic": gp_tr, "traffic_source": gp_tr_note}},
                     "decode_batch": {"M": BATCH, "us_per_call": r["op"][BATCH]["us"],
                                      "roofline": {"bound": "hbm", "achieved": r["op"][BATCH]["gbs"],
                                                   "peak": r["hbm_peak"], "unit": "GB/s",
                                                   "frac": r["op"][BATCH]["gbs"] / r["hbm_peak"],
                                                   "tensor_frac": r["op"][BATCH]["tflops"] / r["tc_peak"],
                                                   "algorithmic_bytes_per_call": r["op"][BATCH]["bytes"],
                                                   "traffic": opb_tr, "traffic_source": opb_tr_note}}},
        "attn_decode": {"workload": f"attn_decode_{ATTN_LAYERS}L_B{BATCH}_ctx{ATTN_CTX}_bf16",
                        "op": "GQA 16q/2kv, head_dim 256, softmax(q k^T / 16) v * sigmoid(z)",
                        "value": r["at"]["tok_s"], "unit": "tok/s", "us_per_call": r["at"]["call_s"] * 1e6,
                        "kernels_per_call": 2, "l2": "inputs larger than L2 (2 GiB of cache per call)",
                        "roofline": {"bound": "hbm", "achieved": r["at"]["achieved"], "peak": r["hbm_peak"],
                                     "unit": "GB/s", "frac": r["at"]["achieved"] / r["hbm_peak"],
                                     "algorithmic_bytes_per_call": ATTN_BYTES_PER_CALL,
                                     "hbm_frac": r["at"]["achieved"] / r["hbm_peak"],
                                     "frac_of_nominal_8TBs": r["at"]["achieved"] / NOMINAL_HBM_GBS,
                                     "traffic": at_tr, "traffic_source": at_tr_note,
                                     "kernel": "attn_block_kernel<bf16>",
                                     "timed": "whole call: attn_block_kernel + attn_combine_kernel"}},
        "other_configs": r["cfgs"],
        "decode_multi": {"workload": f"decode_multi_30L_B{BATCH}_T{MULTI_T}_bf16", "value": r["mt"]["tok_s"],
                         "unit": "tok/s", "tokens_per_sequence_per_call": MULTI_T,
                         "launch_us": r["mt"]["launch_s"] * 1e6,
                         "roofline": {"bound": "hbm", "achieved": r["mt"]["achieved"], "peak": r["hbm_peak"],
                                      "unit": "GB/s", "frac": r["mt"]["achieved"] / r["hbm_peak"],
                                      "frac_of_nominal_8TBs": r["mt"]["achieved"] / NOMINAL_HBM_GBS,
                                      "algorithmic_bytes_per_launch": r["mt"]["bytes"],
                                      "traffic": mt_tr, "traffic_source": mt_tr_note},
                         "by_tokens_per_sequence": {
                             str(t): {"value": m["tok_s"], "unit": "tok/s", "launch_us": m["launch_s"] * 1e6,
                                      "achieved_GBs": m["achieved"], "frac": m["achieved"] / r["hbm_peak"],
                                      "frac_of_nominal_8TBs": m["achieved"] / NOMINAL_HBM_GBS,
                                      "algorithmic_bytes_per_launch": m["bytes"]}
                             for t, m in sorted(r["mts"].items())}},
    }
    print(json.dumps(line))


if __name__ == "__main__":
    main()
