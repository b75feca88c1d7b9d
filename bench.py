"""Benchmark of the attention hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload all|prefill|decode|long|chunked|fp8|append] [--no-cpu-baseline]
                    [--decode-requests N] [--chunked-requests N]

Headline (the JSON `value`): causal GQA prefill, batch 1 x 8192 tokens, 64 query /
8 KV heads, head_dim 128, bf16 -- one step = RoPE of Q and K at absolute
positions + tiled causal attention (O and LSE).  TFLOP/s counts 4*d flops per
visible (query, key) pair.  The paged split-KV decode workload (32 requests,
contexts U[16384, 131072], 16 splits + LSE merge) is reported in `decode`,
as KV-cache GB/s.  `prefill_64k` times 2 x 65536-token causal prefill over all
heads and over heads 16..31 alone; `chunked` times chunked prefill of 4 x 8192
new tokens over a 57344-token paged prefix (prefix call + chunk call + merge).
`prefill_fp8` times the 8K prefill in the FP8 mode (e4m3 Q/K/V codes with
per-row / per-head scales; the quantisation is inside the step).  The line ends
with `decode`, the decode half of the metric in brief (GB/s, fraction of the
HBM copy peak, end to end with the queries uploaded and O/LSE read back each
step, the INT8-cache variant, and the oracle's decode on the host cores);
`decode_detail` holds the full decode record.
Inputs are synthetic and seeded (N(0,1)/sqrt(2) bf16).

Timing: W untimed warm-up steps, then K steps each bracketed by CUDA events on
the launching stream, with an L2 flush (a 512 MB write) between steps outside
the events; barrier + synchronize around the timed region, max over ranks.
`--impl reference` times the fp64 CPU oracle on a bounded sample of the same
workload (rank 0 only).  Under torchrun every rank runs an independent replica
(the path needs no exchange between GPUs) and `value` sums the ranks' work.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "prefill attn TFLOP/s (% BF16 peak); decode KV-read GB/s (% HBM peak)"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
PROFILES = os.path.join(ROOT, "profiles")
CSRC = os.path.join(ROOT, "attention_tiled_causal_gb300", "csrc")


# ------------------------------------------------------------------ environment helpers

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            d = json.load(open(p))
            flat = {}

            def walk(x, pre=""):
                if isinstance(x, dict):
                    for k, v in x.items():
                        walk(v, f"{pre}{k}.")
                elif isinstance(x, (int, float)):
                    flat[pre[:-1]] = float(x)
            walk(d)

            def find(*keys):
                for k, v in flat.items():
                    if k.split(".")[-1] in keys:
                        return v
                return None
            hbm = find("hbm_gbs", "hbm_GBs", "copy_gbs")
            bf = find("bf16_tflops", "bf16_TFLOPs")
            bfs = find("bf16_tflops_sustained")
            if hbm and bf:
                return {"hbm_gbs": hbm, "bf16_tflops": bf, "bf16_tflops_sustained": bfs or bf}, "measured"
        except Exception:
            pass
    return dict(FALLBACK_PEAKS), "fallback"


def kernel_sha(fname):
    return hashlib.sha256(open(os.path.join(CSRC, fname), "rb").read()).hexdigest()[:16]


def profiled_traffic(summary_name, kernel_file):
    """DRAM bytes per launch recorded by an ncu capture summary under profiles/,
    or None if there is none or the kernel source changed since it was taken."""
    p = os.path.join(PROFILES, summary_name)
    if not os.path.exists(p):
        return None
    rec = {}
    for line in open(p):
        if ":" in line and line.strip().startswith(("kernel_source_sha256", "dram_bytes_per_launch_full")):
            k, v = line.split(":", 1)
            rec[k.strip()] = v.strip().strip("`")
    if rec.get("kernel_source_sha256") != kernel_sha(kernel_file):
        return None
    try:
        return float(rec["dram_bytes_per_launch_full"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"bench_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc:
            time.sleep(0.3)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if not self.proc or not os.path.exists(self.path):
            return None
        sm, mx, pw, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            try:
                pw.append(float(f[3]))
            except ValueError:
                pw.append(0.0)
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return None
        out = {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons), "samples": len(sm)}
        if max(pw) > 0:  # samples at more than half the window's peak power: the kernels at work
            busy = [c for c, w in zip(sm, pw) if w > 0.5 * max(pw)]
            out.update(sm_mhz_under_load=statistics.median(busy), power_w_max=max(pw), samples_under_load=len(busy))
        return out


# ------------------------------------------------------------------ replicas

def max_over_ranks(ms: float, pg=None, device="cpu") -> float:
    """Slowest rank's time per step (every rank runs an independent replica)."""
    if pg is None:
        return float(ms)
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(work_per_rank: float, world_size: int, ms_max: float) -> float:
    """Units per second of the whole job: every rank's work over the slowest rank's time."""
    return world_size * work_per_rank / (ms_max * 1e-3)


# ------------------------------------------------------------------ our arm

class Timer:
    """Per-step CUDA events on the launching stream, L2 flush outside the events."""

    def __init__(self, flush_bytes=512 << 20):
        self.flush = torch.empty(flush_bytes // 4, dtype=torch.float32, device="cuda")

    def run(self, fn, steps, warmup, inner=None):
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize()
        tot, sub = 0.0, 0.0
        s = torch.cuda.current_stream()
        for _ in range(steps):
            self.flush.fill_(1.0)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            ev = [] if inner is None else [torch.cuda.Event(enable_timing=True) for _ in range(2)]
            e0.record(s)
            fn(ev)
            e1.record(s)
            e1.synchronize()
            tot += e0.elapsed_time(e1)
            if ev:
                sub += ev[0].elapsed_time(ev[1])
        return tot / steps, (sub / steps if inner else None)


def graph_step_ms(timer, fn, steps, warmup):
    """ms per step of `fn` captured once into a CUDA graph and replayed (the
    launches of a step go to the GPU as one unit, with no host work between
    them), timed like an eager step; None if the capture fails."""
    try:
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            fn()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        torch.cuda.synchronize()
    except Exception as e:  # noqa: BLE001 -- reported, and the eager number stands
        print(f"graph capture failed: {e}", file=sys.stderr)
        torch.cuda.synchronize()
        return None
    ms, _ = timer.run(lambda ev=(): g.replay(), steps, warmup)
    del g
    return ms


def short_ms(timer, fn, steps, warmup):
    """ms per call of a short (tens of microseconds) call: graph-replayed, so the
    host's launch latency is not counted; eager if the capture fails."""
    ms = graph_step_ms(timer, fn, steps, warmup)
    if ms is None:
        ms, _ = timer.run(lambda ev=(): fn(), steps, warmup)
    return ms


# Steps of the pipelined end-to-end loop (at least): a step's latency (upload, compute, download, about
# 2.4 ms) exceeds its period (about 1 ms), and the timed window holds one fill and one drain, whose share
# falls with the step count.
E2E_PIPELINE_STEPS = 100


def pipelined_e2e(atc, host_in, host_out, dev, pos, cu, seq, steps, warmup):
    """End-to-end time per step through the public API as a serving loop runs it:
    every step uploads its Q/K/V from pinned host memory, runs RoPE + attention and
    downloads O and LSE, on three streams with two sets of device buffers, so the
    upload of step i+1 and the download of step i-1 overlap the compute of step i.
    Returns ms per step (CUDA events from the first upload to the last download)."""
    hq_, hk_, hv_ = host_in
    ho, hl = host_out
    q0, k0, v0, out0, lse0 = dev
    bufs = [(q0, k0, v0, out0, lse0),
            tuple(torch.empty_like(t) for t in (q0, k0, v0, out0, lse0))]
    s_in, s_cmp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    in_done = [torch.cuda.Event() for _ in range(2)]
    cmp_done = [torch.cuda.Event() for _ in range(2)]
    out_done = [torch.cuda.Event() for _ in range(2)]

    def run(n, first):
        for i in range(n):
            b = i % 2
            q, k, v, out, lse = bufs[b]
            with torch.cuda.stream(s_in):
                if i >= 2 or not first:
                    s_in.wait_event(cmp_done[b])  # this buffer's previous inputs are consumed
                q.copy_(hq_, non_blocking=True)
                k.copy_(hk_, non_blocking=True)
                v.copy_(hv_, non_blocking=True)
                in_done[b].record(s_in)
            with torch.cuda.stream(s_cmp):
                s_cmp.wait_event(in_done[b])
                if i >= 2 or not first:
                    s_cmp.wait_event(out_done[b])  # this buffer's previous outputs are read back
                atc.rope_apply_qk(q, k, pos)
                atc.attn_prefill(q, k, v, out, lse, cu, pos, seq, cu_k=cu, k_pos=pos)
                cmp_done[b].record(s_cmp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(cmp_done[b])
                ho.copy_(out, non_blocking=True)
                hl.copy_(lse, non_blocking=True)
                out_done[b].record(s_out)

    run(warmup, True)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    with torch.cuda.stream(s_cmp):
        s_cmp.wait_event(e0)
    run(steps, False)
    e1.record(s_out)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps


def link_floor_ms(host_in, dev_in, host_out, dev_out, steps=5):
    """Per step, the time of the step's uploads and downloads alone, each direction
    on its own stream and both at once: the least the pipelined schedule can take
    when the host link, not the GPU, is the limit."""
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()

    def once():
        e = torch.cuda.Event()
        e.record()
        with torch.cuda.stream(s_in):
            s_in.wait_event(e)
            for d, h in zip(dev_in, host_in):
                d.copy_(h, non_blocking=True)
        with torch.cuda.stream(s_out):
            s_out.wait_event(e)
            for h, d in zip(host_out, dev_out):
                h.copy_(d, non_blocking=True)
        torch.cuda.current_stream().wait_stream(s_in)
        torch.cuda.current_stream().wait_stream(s_out)

    once()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        once()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps


def prefill_arm(wl, args, timer, peaks, peak_src):
    import attention_tiled_causal_gb300 as atc
    inp = wl.make("cuda")
    q, k, v, pos, cu = inp["q"], inp["k"], inp["v"], inp["pos"], inp["cu"]
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device="cuda")
    launches = 2  # RoPE of Q and K (one launch), prefill

    def step(ev=()):
        atc.rope_apply_qk(q, k, pos)
        if ev:
            ev[0].record()
        atc.attn_prefill(q, k, v, out, lse, cu, pos, wl.seq, cu_k=cu, k_pos=pos)
        if ev:
            ev[1].record()

    ms_eager, ms_kernel = timer.run(step, args.steps, args.warmup, inner=True)
    ms_graph = graph_step_ms(timer, step, args.steps, args.warmup)
    ms = ms_graph if ms_graph is not None else ms_eager
    atc.attn_device_status()
    flops = wl.flops()
    # end to end through the public API: pinned host inputs in, O and LSE back out
    hq_, hk_, hv_ = q.cpu().pin_memory(), k.cpu().pin_memory(), v.cpu().pin_memory()
    ho = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    hl = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()

    def e2e_step(ev=()):
        q.copy_(hq_, non_blocking=True)
        k.copy_(hk_, non_blocking=True)
        v.copy_(hv_, non_blocking=True)
        step()
        ho.copy_(out, non_blocking=True)
        hl.copy_(lse, non_blocking=True)

    ms_e2e_serial, _ = timer.run(e2e_step, args.steps, args.warmup)
    e2e_steps = max(args.steps, E2E_PIPELINE_STEPS)
    ms_e2e = pipelined_e2e(atc, (hq_, hk_, hv_), (ho, hl), (q, k, v, out, lse), pos, cu, wl.seq, e2e_steps,
                           args.warmup)
    ms_link = link_floor_ms((hq_, hk_, hv_), (q, k, v), (ho, hl), (out, lse))
    # RoPE alone (S1), an HBM stream: read + write of Q and of K
    ms_rope = short_ms(timer, lambda ev=(): atc.rope_apply_qk(q, k, pos), args.steps, args.warmup)
    rope_bytes = 2 * (q.numel() + k.numel()) * q.element_size()
    h2d = sum(t.numel() * t.element_size() for t in (hq_, hk_, hv_))
    d2h = ho.numel() * ho.element_size() + hl.numel() * hl.element_size()
    peak = peaks["bf16_tflops"]
    achieved = flops / (ms_kernel * 1e-3) / 1e12
    traffic = profiled_traffic("prefill_tc_causal_8k.md", "prefill_tc.cu")
    res = {
        "ms_per_step": ms, "flops": flops, "tflops": flops / (ms * 1e-3) / 1e12,
        "launch": {"step": "CUDA graph of the step's 2 launches, replayed" if ms_graph is not None
                   else "eager (graph capture failed)",
                   "eager_ms_per_step": round(ms_eager, 4),
                   "graph_ms_per_step": None if ms_graph is None else round(ms_graph, 4)},
        "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak, "unit": "TFLOP/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic, "traffic_scope": "prefill_tc_kernel (ncu)",
                     "kernel": "attn::tc::prefill_tc_kernel", "kernel_ms": round(ms_kernel, 4),
                     "peak_source": f"{peak_src} bf16 dense (burst)"},
        "e2e": {"value": round(flops / (ms_e2e * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(ms_e2e, 4),
                "schedule": "three streams, double-buffered: step i+1's upload and step i-1's download overlap "
                            "step i's compute; inputs (168 MB) exceed L2; timed from the first step's upload to the "
                            "last step's download, so one pipeline fill and drain is spread over the steps",
                "pipelined_steps": e2e_steps,
                "host_link_floor_ms": round(ms_link, 4),
                "frac_of_host_link_floor": round(ms_link / ms_e2e, 4),
                "serial": {"value": round(flops / (ms_e2e_serial * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
                           "ms_per_step": round(ms_e2e_serial, 4),
                           "schedule": "upload, compute and download of each step in turn on one stream"}},
        "launches_per_step": launches,
        "rope": hbm_line("rope_apply_qk (Q and K of the 8K prefill, one launch)", rope_bytes, ms_rope, peaks, peak_src),
        "inputs": (q, k, v, pos, cu),
    }
    return res


def fp8_prefill_arm(wl, args, timer, peaks, peak_src, inputs=None):
    """The 8K prefill in the FP8 mode: e4m3 codes for Q (one scale per token and head)
    and K (one scale per KV head) with RoPE fused into their quantisation, V (one
    scale per KV head, transposed), then attention on the codes.  The tensor-core peak for e4m3 is the measured bf16
    peak times the nominal e4m3 / bf16 ratio (4.5 / 2.25 PFLOP/s dense)."""
    import attention_tiled_causal_gb300 as atc
    if inputs is None:
        inp = wl.make("cuda")
        inputs = (inp["q"], inp["k"], inp["v"], inp["pos"], inp["cu"])
    q, k, v, pos, cu = inputs
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device="cuda")
    codes = {}
    s_k, s_v = torch.cuda.Stream(), torch.cuda.Stream()

    def quant():
        # Q, K and V quantise independently: K and V on side streams, joined
        # before the attention (a graph keeps them as parallel branches)
        cur = torch.cuda.current_stream()
        s_k.wait_stream(cur)
        s_v.wait_stream(cur)
        codes["q"] = atc.rope_quant_fp8_rows(q, pos)
        with torch.cuda.stream(s_k):
            codes["k"] = atc.rope_quant_fp8_heads(k, pos)
        with torch.cuda.stream(s_v):
            codes["v"] = atc.quant_fp8_heads(v, transposed=True)
        cur.wait_stream(s_k)
        cur.wait_stream(s_v)

    def attend():
        (cq, sq), (ck, sk), (cv, sv) = codes["q"], codes["k"], codes["v"]
        atc.attn_prefill_fp8(cq, sq, ck, sk, cv, sv, out, lse, cu, pos, wl.seq, cu, pos)

    def step(ev=()):
        quant()
        if ev:
            ev[0].record()
        attend()
        if ev:
            ev[1].record()

    ms_eager, ms_kernel = timer.run(step, args.steps, args.warmup, inner=True)
    ms_graph = graph_step_ms(timer, step, args.steps, args.warmup)
    ms = ms_graph if ms_graph is not None else ms_eager
    ms_q = graph_step_ms(timer, quant, args.steps, args.warmup)
    if ms_q is None:
        ms_q, _ = timer.run(lambda ev=(): quant(), args.steps, args.warmup)
    atc.attn_device_status()
    flops = wl.flops()
    peak = 2.0 * peaks["bf16_tflops"]
    achieved = flops / (ms_kernel * 1e-3) / 1e12
    # Q: bf16 in, codes and row scales out; K and V: bf16 read twice (max, then codes), codes out
    quant_bytes = 3 * q.numel() + q.numel() // 128 * 4 + 5 * (k.numel() + v.numel())
    return {
        "workload": wl.name + " with e4m3 Q/K/V codes (RoPE fused into the quantisation + attention, O and LSE)",
        "value": round(flops / (ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s", "ms_per_step": round(ms, 4),
        "steps": args.steps, "warmup": args.warmup, "dtype": "e4m3 operands, fp32 accumulation and softmax",
        "launch": {"step": "CUDA graph of the step's 7 launches, replayed" if ms_graph is not None
                   else "eager (graph capture failed)",
                   "eager_ms_per_step": round(ms_eager, 4),
                   "graph_ms_per_step": None if ms_graph is None else round(ms_graph, 4)},
        "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": round(peak, 1), "unit": "TFLOP/s",
                     "frac": round(achieved / peak, 4),
                     "traffic": profiled_traffic("prefill_tc_fp8_causal_8k.md", "prefill_tc.cu"),
                     "traffic_scope": "prefill_tc_kernel<false, true> (ncu)",
                     "kernel": "attn::tc::prefill_tc_kernel<false, true>", "kernel_ms": round(ms_kernel, 4),
                     "peak_source": f"{peak_src} bf16 dense (burst) x 2, the nominal e4m3 / bf16 ratio",
                     "vs_bf16_kernel_peak": round(achieved / peaks["bf16_tflops"], 4)},
        "quantisation": hbm_line("rope_quant_fp8_rows (Q) + rope_quant_fp8_heads (K) + quant_fp8_heads (V^T), "
                                 "Q, K and V on three streams",
                                 quant_bytes, ms_q, peaks, peak_src),
        "gpu_launches_per_step": 1 + 2 + 3 + 1,
    }


def decode_arm(wl, args, timer, peaks, peak_src, cpu=True):
    import attention_tiled_causal_gb300 as atc
    inp = wl.make("cuda")
    q = inp["q"]
    q_raw = q.clone()
    po, pl = atc.decode_workspace(wl.batch, wl.hq, wl.splits, wl.d, "cuda")
    out = torch.empty((wl.batch, wl.hq, wl.d), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((wl.batch, wl.hq), dtype=torch.float32, device="cuda")

    def step(ev=()):
        atc.rope_apply(q, inp["q_pos"])
        if ev:
            ev[0].record()
        atc.attn_decode_paged(q, inp["k_cache"], inp["v_cache"], inp["page_table"], inp["ctx_lens"], wl.splits,
                              po, pl, out, lse)
        if ev:
            ev[1].record()

    ms, ms_kernel = timer.run(step, args.steps, args.warmup, inner=True)
    # end to end through the public API: each step uploads the new tokens' queries
    # from pinned host memory and reads O and LSE back; the cache stays resident
    hq_ = q_raw.cpu().pin_memory()
    ho = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    hl = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()

    def e2e_step(ev=()):
        q.copy_(hq_, non_blocking=True)
        step()
        ho.copy_(out, non_blocking=True)
        hl.copy_(lse, non_blocking=True)

    ms_e2e, _ = timer.run(e2e_step, args.steps, args.warmup)
    # the LSE merge of the 16 splits alone (S7), an HBM stream
    ms_merge = short_ms(timer, lambda ev=(): atc.attn_lse_merge(po.permute(2, 0, 1, 3), pl.permute(2, 0, 1), out, lse),
                            args.steps, args.warmup)
    atc.attn_device_status()
    kv = wl.kv_bytes()
    part = wl.batch * wl.hq * wl.splits * (wl.d + 1) * 4
    qb = wl.batch * wl.hq * wl.d * 2
    outb = wl.batch * wl.hq * (wl.d * 2 + 4)
    alg_step = kv + qb + 2 * part + outb            # cache + q + partials out and back + result
    peak = peaks["hbm_gbs"]
    achieved = alg_step / (ms_kernel * 1e-3) / 1e9  # split + merge kernels (rope of q is ~0.5 MB)
    res = {
        "metric": "decode KV-read GB/s", "unit": "GB/s", "value": round(kv / (ms * 1e-3) / 1e9, 1),
        "ms_per_step": round(ms, 4), "kv_bytes_per_step": kv,
        "workload": wl.name,
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4),
                     "traffic": profiled_traffic("decode_split_paged_b32.md", "decode.cu") if wl.batch == 32 else None,
                     "traffic_scope": "decode_split_kernel (ncu, one pass on the full 32-request workload); merge not included",
                     "kernel": "attn::dec::decode_split_kernel + attn::lse_merge_kernel",
                     "kernel_ms": round(ms_kernel, 4), "peak_source": f"{peak_src} HBM copy"},
        "e2e": {"value": round(kv / (ms_e2e * 1e-3) / 1e9, 1), "unit": "GB/s",
                "h2d_bytes_per_step": hq_.numel() * hq_.element_size(),
                "d2h_bytes_per_step": ho.numel() * ho.element_size() + hl.numel() * hl.element_size(),
                "ms_per_step": round(ms_e2e, 4)},
        "gpu_launches_per_step": 3,
        "merge": hbm_line("attn_lse_merge of the 16 decode splits", part + outb, ms_merge, peaks, peak_src),
    }
    if cpu:
        res["cpu_baseline"] = oracle_decode_baseline(wl, inp, q_raw)
    del inp
    return res


def long_prefill_arm(wl, args, timer, peaks, peak_src, cpu=False):
    """2 x 65536-token causal prefill: all 64 heads, and heads 16..31 alone (one
    Ulysses rank's share of a 4-way head split).  Attention only: RoPE is applied
    once before the timed calls."""
    import attention_tiled_causal_gb300 as atc
    import synth
    inp = wl.make("cuda")
    q, k, v, pos, cu = inp["q"], inp["k"], inp["v"], inp["pos"], inp["cu"]
    sample = None
    if cpu:  # the oracle's inputs, taken before the in-place RoPE
        rows = np.concatenate([synth.sample_rows(wl.seq, 16, 77 + b) + b * wl.seq for b in range(wl.batch)])
        sample = (rows, q[torch.from_numpy(rows).to(q.device)].cpu(), k.cpu(), v.cpu(), pos.cpu().numpy(),
                  cu.cpu().numpy())
    atc.rope_apply(q, pos)
    atc.rope_apply(k, pos)
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device="cuda")
    peak = peaks["bf16_tflops"]
    steps, warmup = min(args.steps, 5), 3
    res = {"workload": wl.name + " (attention only)", "steps": steps, "warmup": warmup}
    for lo, hi in ((0, wl.hq), (16, 32)):
        def step(ev=(), lo=lo, hi=hi):
            atc.attn_prefill(q, k, v, out, lse, cu, pos, wl.seq, cu_k=cu, k_pos=pos, h_lo=lo, h_hi=hi)

        ms, _ = timer.run(step, steps, warmup)
        fl = wl.flops(lo, hi)
        tf = fl / (ms * 1e-3) / 1e12
        res[f"heads_{lo}_{hi}"] = {"flops": fl, "ms": round(ms, 4), "value": round(tf, 2), "unit": "TFLOP/s",
                                   "frac": round(tf / peak, 4), "peak": peak,
                                   "peak_source": f"{peak_src} bf16 dense (burst)",
                                   "frac_of_sustained": round(tf / peaks["bf16_tflops_sustained"], 4)}
    atc.attn_device_status()
    del inp, q, k, v, out
    if sample is not None:
        res["cpu_baseline"] = oracle_long_baseline(wl, *sample)
    return res


def oracle_long_baseline(wl, rows, qs, k, v, pos, cu):
    """The oracle on 16 seeded query rows per sequence of the 2 x 65536-token
    workload, all 64 heads: RoPE of those rows and of every key, bf16 rounding,
    fp64 three-pass attention (input widening outside the timed part)."""
    import oracle
    qf, kf, vf = (t.to(torch.float64).numpy() for t in (qs, k, v))
    t0 = time.perf_counter()
    qr = oracle.round_bf16(oracle.rope(qf, pos[rows], wl.base))
    kr = oracle.round_bf16(oracle.rope(kf, pos, wl.base))
    oracle.attention(qr, (rows // wl.seq).astype(np.int32), pos[rows], kr, vf, cu, pos, wl.scale)
    dt = time.perf_counter() - t0
    flops = 4.0 * wl.d * wl.hq * float(np.sum(pos[rows] + 1))
    return {"value": round(flops / dt / 1e12, 6), "unit": "TFLOP/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{len(rows)} seeded query rows (16 per sequence) x 64 heads of the 2 x 65536-token prefill "
                      f"(RoPE + bf16 rounding + fp64 three-pass attention), {dt:.1f} s"}


def oracle_chunked_baseline(wl, inp, rows, q_raw, k_raw):
    """The oracle on 16 seeded chunk rows per request of the chunked workload,
    all 64 heads: each row over its request's 57344 cached keys (gathered through
    the page table) and the causal part of its chunk; RoPE of the rows and the
    chunk keys, bf16 rounding, fp64 three-pass attention.  Page gathers and input
    widening are outside the timed part."""
    import oracle
    B, P, C = wl.batch, wl.prefix, wl.chunk
    table = inp["page_table"].cpu().numpy()
    qpos = inp["q_pos"].cpu().numpy()
    dt, flops = 0.0, 0.0
    for b in range(B):
        sel = np.nonzero((rows // C) == b)[0]
        n = (P + 63) // 64
        pages = torch.from_numpy(table[b, :n].astype(np.int64)).to(inp["k_cache"].device)
        kc = inp["k_cache"][:, pages].cpu().to(torch.float64).numpy().transpose(1, 2, 0, 3).reshape(n * 64, wl.hkv,
                                                                                                    wl.d)[:P]
        vc = inp["v_cache"][:, pages].cpu().to(torch.float64).numpy().transpose(1, 2, 0, 3).reshape(n * 64, wl.hkv,
                                                                                                    wl.d)[:P]
        kch = k_raw[b * C:(b + 1) * C].to(torch.float64).numpy()
        vch = inp["v"][b * C:(b + 1) * C].cpu().to(torch.float64).numpy()
        qb = q_raw[sel].to(torch.float64).numpy()
        rp = qpos[rows[sel]]
        t0 = time.perf_counter()
        qr = oracle.round_bf16(oracle.rope(qb, rp, wl.base))
        kr = oracle.round_bf16(oracle.rope(kch, qpos[b * C:(b + 1) * C], wl.base))
        K = np.concatenate([kc, kr])
        V = np.concatenate([vc, vch])
        KP = np.concatenate([np.arange(P, dtype=np.int32), qpos[b * C:(b + 1) * C]])
        oracle.attention(qr, np.zeros(len(sel), np.int32), rp, K, V, [0, P + C], KP, wl.scale)
        dt += time.perf_counter() - t0
        flops += 4.0 * wl.d * wl.hq * float(np.sum(rp + 1))
        del kc, vc, K, V
    return {"value": round(flops / dt / 1e12, 6), "unit": "TFLOP/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{len(rows)} seeded chunk rows (16 per request) x 64 heads of the chunked prefill over the "
                      f"57344-token paged prefix (RoPE + bf16 rounding + fp64 three-pass attention), {dt:.1f} s"}


def chunked_arm(wl, args, timer, peaks, peak_src, cpu=False):
    """Chunked prefill: 4 requests, each an 8192-token chunk over a 57344-token
    prefix in a shuffled head-major paged cache.  One step = the paged-prefix
    call + the causal chunk call + the LSE merge of the two partial results.  Also
    timed: the serving flow of appending the chunk to the cache, then one paged
    causal call over prefix + chunk."""
    import attention_tiled_causal_gb300 as atc
    import synth
    inp = wl.make("cuda")
    C = wl.chunk
    q, k, v = inp["q"], inp["k"], inp["v"]
    sample = None
    if cpu:  # the oracle's chunk rows and keys, taken before the in-place RoPE
        rows = np.concatenate([synth.sample_rows(C, 16, 88 + b) + b * C for b in range(wl.batch)])
        sample = (rows, q[torch.from_numpy(rows).to(q.device)].cpu(), k.cpu())
    atc.rope_apply(q, inp["q_pos"])
    atc.rope_apply(k, inp["q_pos"])
    T, hq, d = q.shape
    po = torch.empty((2, T, hq, d), dtype=torch.float32, device="cuda")
    pl = torch.empty((2, T, hq), dtype=torch.float32, device="cuda")
    out = torch.empty((T, hq, d), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((T, hq), dtype=torch.float32, device="cuda")

    def prefix(ev=()):
        atc.attn_prefill(q, inp["k_cache"], inp["v_cache"], po[0], pl[0], inp["cu_q"], inp["q_pos"], C,
                         page_table=inp["page_table"], k_lens=inp["prefix_lens"], num_pages=inp["num_pages"])

    def chunk(ev=()):
        atc.attn_prefill(q, k, v, po[1], pl[1], inp["cu_q"], inp["q_pos"], C, cu_k=inp["cu_q"], k_pos=inp["q_pos"])

    def merge(ev=()):
        atc.attn_lse_merge(po, pl, out, lse)

    def step(ev=()):
        prefix()
        chunk()
        merge()

    steps, warmup = min(args.steps, 10), 3
    ms, _ = timer.run(step, steps, warmup)
    ms_p, _ = timer.run(prefix, steps, warmup)
    ms_c, _ = timer.run(chunk, steps, warmup)
    ms_m = short_ms(timer, merge, steps, warmup)
    merge_bytes = po.numel() * 4 + pl.numel() * 4 + out.numel() * 2 + lse.numel() * 4
    del po, pl
    cpu_res = oracle_chunked_baseline(wl, inp, *sample) if sample is not None else None
    del inp

    # The serving flow: append the chunk's K (rotated) and V to a paged cache that
    # has room for it, then one paged causal call over prefix + chunk.
    B, P = wl.batch, wl.prefix
    table2, npg2 = synth.shuffled_page_table([P + C] * B, wl.seed * 16 + 10)
    kc2 = synth.randn((wl.hkv, npg2, synth.PAGE, wl.d), wl.seed * 16 + 11, wl.std, device="cuda")
    vc2 = synth.randn((wl.hkv, npg2, synth.PAGE, wl.d), wl.seed * 16 + 12, wl.std, device="cuda")
    k_raw = synth.randn((T, wl.hkv, wl.d), wl.seed * 16 + 2, wl.std, device="cuda")  # unrotated chunk keys
    qpos = torch.arange(P, P + C, dtype=torch.int32).repeat(B)
    pages = torch.from_numpy(table2).long()[torch.arange(B).repeat_interleave(C), (qpos // synth.PAGE).long()]
    slots = (pages * synth.PAGE + (qpos % synth.PAGE).long()).to(torch.int32).cuda()
    qposd = qpos.cuda()
    tabled = torch.from_numpy(table2).cuda()
    klens = torch.full((B,), P + C, dtype=torch.int32, device="cuda")

    def append(ev=()):
        atc.attn_kv_append_paged(k_raw, v, qposd, slots, kc2, vc2)

    def fused(ev=()):
        append()
        atc.attn_prefill(q, kc2, vc2, out, lse, inp_cu_q, qposd, C, page_table=tabled, k_lens=klens, num_pages=npg2)

    inp_cu_q = torch.from_numpy(synth.cu_seqlens([C] * B)).cuda()
    ms_f, _ = timer.run(fused, steps, warmup)
    ms_a = short_ms(timer, append, steps, warmup)
    atc.attn_device_status()
    append_bytes = 2 * 2 * k_raw.numel() * 2  # read K and V, write both into the cache
    del kc2, vc2
    # the same chunk into an INT8 cache (codes + one fp32 scale per row)
    kc8 = torch.zeros((wl.hkv, npg2, synth.PAGE, wl.d), dtype=torch.int8, device="cuda")
    vc8 = torch.zeros_like(kc8)
    ks8 = torch.zeros((wl.hkv, npg2, synth.PAGE), dtype=torch.float32, device="cuda")
    vs8 = torch.zeros_like(ks8)

    def append8(ev=()):
        atc.attn_kv_append_paged_int8(k_raw, v, qposd, slots, kc8, vc8, ks8, vs8)

    ms_a8 = short_ms(timer, append8, steps, warmup)
    atc.attn_device_status()
    append8_bytes = 2 * k_raw.numel() * 2 + 2 * (k_raw.numel() + k_raw.numel() // wl.d * 4)
    del kc8, vc8, ks8, vs8, k_raw, q, k, v, out, lse
    peak = peaks["bf16_tflops"]
    fl = wl.flops()
    fl_c = 4.0 * wl.d * wl.hq * wl.batch * (C * (C + 1) // 2)
    fl_p = fl - fl_c
    tf = fl / (ms * 1e-3) / 1e12
    return {"workload": wl.name + " (paged prefix + causal chunk + LSE merge)", "steps": steps, "warmup": warmup,
            "flops": fl, "ms": round(ms, 4), "value": round(tf, 2), "unit": "TFLOP/s", "frac": round(tf / peak, 4),
            "peak": peak, "peak_source": f"{peak_src} bf16 dense (burst)",
            "frac_of_sustained": round(tf / peaks["bf16_tflops_sustained"], 4),
            "paged_prefix": {"ms": round(ms_p, 4), "value": round(fl_p / (ms_p * 1e-3) / 1e12, 2),
                             "unit": "TFLOP/s"},
            "causal_chunk": {"ms": round(ms_c, 4), "value": round(fl_c / (ms_c * 1e-3) / 1e12, 2),
                             "unit": "TFLOP/s"},
            "merge": hbm_line("attn_lse_merge of the two partial results", merge_bytes, ms_m, peaks, peak_src),
            "append_then_one_call": {
                "what": "attn_kv_append_paged of the chunk (K rotated, K/V scattered into pages) + one paged causal "
                        "call over prefix + chunk", "ms": round(ms_f, 4),
                "value": round(fl / (ms_f * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
                "frac": round(fl / (ms_f * 1e-3) / 1e12 / peak, 4),
                "append": hbm_line(f"attn_kv_append_paged ({wl.batch} x {wl.chunk} tokens, {wl.hkv} KV heads)", append_bytes, ms_a, peaks,
                                   peak_src),
                "append_int8": hbm_line("attn_kv_append_paged_int8 (the same chunk into an INT8 cache)",
                                        append8_bytes, ms_a8, peaks, peak_src)},
            **({"cpu_baseline": cpu_res} if cpu_res else {})}


def append_arm(wl, args, timer, peaks, peak_src):
    """The chunked workload's cache appends alone: 4 x 8192 new tokens' keys
    (rotated at positions 57344..65535) and values written through a shuffled
    page table into a bf16 cache (attn_kv_append_paged) and into an INT8 cache
    (attn_kv_append_paged_int8).  Small enough for a profiler capture."""
    import attention_tiled_causal_gb300 as atc
    import synth
    B, P, C = wl.batch, wl.prefix, wl.chunk
    T = B * C
    table, npg = synth.shuffled_page_table([P + C] * B, wl.seed * 16 + 10)
    k_raw = synth.randn((T, wl.hkv, wl.d), wl.seed * 16 + 2, wl.std, device="cuda")
    v = synth.randn((T, wl.hkv, wl.d), wl.seed * 16 + 3, wl.std, device="cuda")
    qpos = torch.arange(P, P + C, dtype=torch.int32).repeat(B)
    pages = torch.from_numpy(table).long()[torch.arange(B).repeat_interleave(C), (qpos // synth.PAGE).long()]
    slots = (pages * synth.PAGE + (qpos % synth.PAGE).long()).to(torch.int32).cuda()
    qposd = qpos.cuda()
    kc = torch.zeros((wl.hkv, npg, synth.PAGE, wl.d), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    kc8 = torch.zeros((wl.hkv, npg, synth.PAGE, wl.d), dtype=torch.int8, device="cuda")
    vc8 = torch.zeros_like(kc8)
    ks8 = torch.zeros((wl.hkv, npg, synth.PAGE), dtype=torch.float32, device="cuda")
    vs8 = torch.zeros_like(ks8)
    ms_a = short_ms(timer, lambda ev=(): atc.attn_kv_append_paged(k_raw, v, qposd, slots, kc, vc), args.steps,
                    args.warmup)
    ms_a8 = short_ms(timer, lambda ev=(): atc.attn_kv_append_paged_int8(k_raw, v, qposd, slots, kc8, vc8, ks8, vs8),
                     args.steps, args.warmup)
    atc.attn_device_status()
    append_bytes = 2 * 2 * k_raw.numel() * 2
    append8_bytes = 2 * k_raw.numel() * 2 + 2 * (k_raw.numel() + k_raw.numel() // wl.d * 4)
    return {"append": hbm_line(f"attn_kv_append_paged ({wl.batch} x {wl.chunk} tokens, {wl.hkv} KV heads)", append_bytes, ms_a, peaks,
                               peak_src),
            "append_int8": hbm_line("attn_kv_append_paged_int8 (the same chunk into an INT8 cache)", append8_bytes,
                                    ms_a8, peaks, peak_src)}


def decode_int8_arm(wl, args, timer, peaks, peak_src):
    """The decode workload over an INT8 cache (codes + one fp32 scale per KV head and
    token): half the bytes per cached token."""
    import attention_tiled_causal_gb300 as atc
    inp = wl.make("cuda")
    q = inp["q"]
    po, pl = atc.decode_workspace(wl.batch, wl.hq, wl.splits, wl.d, "cuda")
    out = torch.empty((wl.batch, wl.hq, wl.d), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((wl.batch, wl.hq), dtype=torch.float32, device="cuda")

    def step(ev=()):
        atc.rope_apply(q, inp["q_pos"])
        if ev:
            ev[0].record()
        atc.attn_decode_paged_int8(q, inp["k_cache"], inp["v_cache"], inp["k_scale"], inp["v_scale"],
                                   inp["page_table"], inp["ctx_lens"], wl.splits, po, pl, out, lse)
        if ev:
            ev[1].record()

    ms, ms_kernel = timer.run(step, args.steps, args.warmup, inner=True)
    atc.attn_device_status()
    kv = wl.kv_bytes()
    part = wl.batch * wl.hq * wl.splits * (wl.d + 1) * 4
    qb = wl.batch * wl.hq * wl.d * 2
    outb = wl.batch * wl.hq * (wl.d * 2 + 4)
    alg_step = kv + qb + 2 * part + outb
    peak = peaks["hbm_gbs"]
    achieved = alg_step / (ms_kernel * 1e-3) / 1e9
    tokens = int(wl.ctx_lens().astype(np.int64).sum())
    del inp
    return {
        "metric": "decode KV-read GB/s", "unit": "GB/s", "value": round(kv / (ms * 1e-3) / 1e9, 1),
        "ms_per_step": round(ms, 4), "kv_bytes_per_step": kv, "workload": wl.name,
        "cached_tokens_per_s": round(tokens / (ms * 1e-3), 0),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4),
                     "traffic": profiled_traffic("decode_int8_paged_b32.md", "decode_int8.cu") if wl.batch == 32 else None,
                     "traffic_scope": "decode_split_int8_kernel (ncu, one pass on the full 32-request workload); merge not included",
                     "kernel": "attn::dec8::decode_split_int8_kernel + attn::lse_merge_kernel",
                     "kernel_ms": round(ms_kernel, 4), "peak_source": f"{peak_src} HBM copy"},
        "gpu_launches_per_step": 3,
    }


def hbm_line(what, nbytes, ms, peaks, peak_src):
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"what": what, "bytes": int(nbytes), "ms": round(ms, 4), "value": round(gbs, 1), "unit": "GB/s",
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": round(gbs / peaks["hbm_gbs"], 4), "peak_source": f"{peak_src} HBM copy"}}


# ------------------------------------------------------------------ oracle timing

def oracle_sample(wl, inputs, n_rows, seed):
    """Time the oracle on n_rows query rows (all heads) of the prefill workload:
    RoPE of those rows and of all keys, bf16 rounding, three-pass attention.
    Returns (seconds, flops of the sample)."""
    import oracle
    q, k, v, pos, cu = inputs
    rows = synth_rows(wl.seq, n_rows, seed)
    qs = q[torch.from_numpy(rows).to(q.device)].cpu()
    kc, vc = k.cpu(), v.cpu()
    posn = pos.cpu().numpy()
    t0 = time.perf_counter()
    qr = oracle.round_bf16(oracle.rope(qs.to(torch.float64).numpy(), posn[rows], wl.base))
    kr = oracle.round_bf16(oracle.rope(kc.to(torch.float64).numpy(), posn, wl.base))
    oracle.attention(qr, np.zeros(len(rows), np.int32), posn[rows], kr, vc.to(torch.float64).numpy(),
                     cu.cpu().numpy(), posn, wl.scale)
    dt = time.perf_counter() - t0
    flops = 4.0 * wl.d * wl.hq * float(np.sum(rows + 1))
    return dt, flops


def synth_rows(seq, n, seed):
    import synth
    return synth.sample_rows(seq, n, seed)


def cpu_baseline(wl, inputs, rows=2048):
    import oracle
    dt, flops = oracle_sample(wl, inputs, rows, 99)
    return {"value": round(flops / dt / 1e12, 6), "unit": "TFLOP/s", "cores": oracle.num_threads(),
            "kind": "oracle",
            "sample": f"{rows} seeded query rows x all 64 heads of the 8192-token prefill "
                      f"(RoPE + bf16 rounding + fp64 three-pass attention), {dt:.1f} s"}


def oracle_decode_baseline(wl, inp, q_raw, n_req=16, seed=31):
    """The oracle's decode on n_req seeded requests of the decode workload: RoPE of
    their queries, bf16 rounding, and the fp64 decode over their pages (gathered
    from the device cache into logical order first, outside the timed part).
    Reported in the metric's unit, KV-cache GB/s (bf16 bytes of the pages read)."""
    import oracle
    ctx = wl.ctx_lens()
    picks = np.sort(np.random.default_rng(seed).choice(wl.batch, min(n_req, wl.batch), replace=False))
    table = inp["page_table"].cpu().numpy()
    qpos = inp["q_pos"].cpu().numpy()
    dt, kv = 0.0, 0
    for b in picks:
        n = (int(ctx[b]) + 63) // 64
        pages = torch.from_numpy(table[b, :n].astype(np.int64)).to(inp["k_cache"].device)
        kc = inp["k_cache"][:, pages].cpu().to(torch.float64).numpy()
        vc = inp["v_cache"][:, pages].cpu().to(torch.float64).numpy()
        qb = q_raw[b:b + 1].cpu().to(torch.float64).numpy()
        t0 = time.perf_counter()
        qr = oracle.round_bf16(oracle.rope(qb, qpos[b:b + 1], wl.base))
        oracle.decode_paged(qr, kc, vc, np.arange(n, dtype=np.int32)[None, :], ctx[b:b + 1], n, wl.scale)
        dt += time.perf_counter() - t0
        kv += int(ctx[b]) * wl.hkv * wl.d * 2 * 2
        del kc, vc
    return {"value": round(kv / dt / 1e9, 3), "unit": "GB/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{len(picks)} seeded requests of the 32 (contexts {', '.join(str(int(ctx[b])) for b in picks)}): "
                      f"RoPE + bf16 rounding of the query, fp64 decode over all their cached tokens, {dt:.1f} s"}


def oracle_tiny_timing(reps=200):
    """The tiny fp32 workload (B1 S64, 8/2 heads, d64), every row, on one thread
    and on all threads, repeated `reps` times: RoPE of Q and K plus the fp64
    three-pass attention."""
    import oracle
    import synth
    w = synth.TINY
    inp = w.make()
    q, k, v = (synth.as_f64(inp[n]) for n in ("q", "k", "v"))
    pos, cu = inp["pos"].numpy(), inp["cu"].numpy()
    seq = np.zeros(w.seq, np.int32)
    out = {}
    nmax = oracle.num_threads()
    for label, n in (("one_thread", 1), ("all_threads", nmax)):
        oracle.set_num_threads(n)
        t0 = time.perf_counter()
        for _ in range(reps):
            oracle.attention(oracle.rope(q, pos, w.base), seq, pos, oracle.rope(k, pos, w.base), v, cu, pos, w.scale)
        dt = time.perf_counter() - t0
        out[label] = {"value": round(w.flops() * reps / dt / 1e9, 3), "unit": "GFLOP/s", "cores": n,
                      "ms_per_pass": round(dt / reps * 1e3, 3)}
    oracle.set_num_threads(nmax)
    out["sample"] = f"all 64 rows x 8 heads of the tiny workload, {reps} passes per thread count"
    return out


def compact_decode(dec):
    """The decode half of the metric in a few keys, for the end of the line."""
    i8 = dec.get("int8_cache", {})
    return {"metric": "decode KV-read GB/s (% HBM peak)", "workload": "B32 ctx U[16K,128K] 64/8 d128, 16 splits",
            "value": dec["value"], "unit": "GB/s", "frac_of_hbm": round(dec["value"] / dec["roofline"]["peak"], 4),
            "ms_per_step": dec["ms_per_step"], "kernel_ms": dec["roofline"]["kernel_ms"],
            "kernel_frac": dec["roofline"]["frac"],
            "e2e": {k: dec["e2e"][k] for k in ("value", "unit", "h2d_bytes_per_step", "d2h_bytes_per_step")},
            "int8_cache": {"value": i8.get("value"), "frac": (i8.get("roofline") or {}).get("frac")},
            "cpu_baseline": dec.get("cpu_baseline")}


# ------------------------------------------------------------------ main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="all", choices=["all", "prefill", "decode", "long", "chunked", "fp8", "append"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--decode-requests", type=int, default=None,
                    help="decode workload with fewer requests (first N of the seeded 32); for small profiler captures")
    ap.add_argument("--chunked-requests", type=int, default=None,
                    help="chunked workload with fewer requests (N of 4, same prefix and chunk lengths); "
                         "for small profiler captures")
    args = ap.parse_args()
    ws, rank, local = dist_env()
    import synth

    if args.impl == "reference":
        if rank != 0:
            return 0
        reference_arm(args, synth)
        return 0

    torch.cuda.set_device(local)
    pg = None
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
        pg = dist
    peaks, peak_src = load_peaks()
    timer = Timer()
    # the oracle baselines run on the host cores once: rank 0 of a single-GPU run
    cpu_leg = not args.no_cpu_baseline and ws == 1 and rank == 0
    wl = synth.PREFILL_8K
    res = None
    if args.workload in ("all", "prefill"):
        if pg:
            pg.barrier()
        torch.cuda.synchronize()
        with ClockSampler(local) as clk:
            res = prefill_arm(wl, args, timer, peaks, peak_src)
        torch.cuda.synchronize()
        if pg:
            pg.barrier()
        clocks = clk.summary()
    dec = None
    if args.workload in ("all", "decode"):
        dwl = synth.DECODE
        if args.decode_requests:
            import dataclasses
            dwl = dataclasses.replace(dwl, batch=args.decode_requests,
                                      name=dwl.name.replace("B32", f"B{args.decode_requests}"))
        dec = decode_arm(dwl, args, timer, peaks, peak_src, cpu=cpu_leg)
        torch.cuda.empty_cache()
        dwl8 = synth.DECODE_INT8
        if args.decode_requests:
            import dataclasses
            dwl8 = dataclasses.replace(dwl8, batch=args.decode_requests,
                                       name=dwl8.name.replace("B32", f"B{args.decode_requests}"))
        dec["int8_cache"] = decode_int8_arm(dwl8, args, timer, peaks, peak_src)
        dec["cached_tokens_per_s"] = round(int(dwl.ctx_lens().astype(np.int64).sum()) / (dec["ms_per_step"] * 1e-3), 0)
        torch.cuda.empty_cache()
    extra = {}
    if args.workload in ("all", "fp8"):
        extra["prefill_fp8"] = fp8_prefill_arm(wl, args, timer, peaks, peak_src, res["inputs"] if res else None)
        torch.cuda.empty_cache()
    # the long and chunked arms keep the GPU under dense load for seconds: their clocks go on record
    # beside them (a power-capped clock is what the sustained peak is measured at)
    if args.workload in ("all", "long"):
        with ClockSampler(local) as clk_l:
            extra["prefill_64k"] = long_prefill_arm(synth.PREFILL_64K, args, timer, peaks, peak_src, cpu=cpu_leg)
        extra["prefill_64k"]["clocks"] = clk_l.summary()
        torch.cuda.empty_cache()
    if args.workload in ("all", "chunked"):
        cwl = synth.CHUNKED
        if args.chunked_requests:
            import dataclasses
            cwl = dataclasses.replace(cwl, batch=args.chunked_requests,
                                      name=cwl.name.replace("B4", f"B{args.chunked_requests}"))
        with ClockSampler(local) as clk_c:
            extra["chunked"] = chunked_arm(cwl, args, timer, peaks, peak_src, cpu=cpu_leg)
        extra["chunked"]["clocks"] = clk_c.summary()
        torch.cuda.empty_cache()
    if args.workload == "append":
        extra["append"] = append_arm(synth.CHUNKED, args, timer, peaks, peak_src)
    if not res and not dec:  # a single secondary workload (profiling): print its own object
        if rank == 0:
            print(json.dumps(extra), flush=True)
        if pg:
            pg.destroy_process_group()
        return 0
    ms = max_over_ranks(res["ms_per_step"] if res else dec["ms_per_step"], pg, "cuda")
    if rank != 0:
        if pg:
            pg.destroy_process_group()
        return 0
    line = {"metric": METRIC}
    if res:
        value = whole_job_rate(res["flops"], ws, ms) / 1e12
        line.update({"value": round(value, 2), "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
                     "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True,
                     "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
                     "config": prefill_config(wl, ws),
                     "roofline": res["roofline"], "e2e": res["e2e"], "clocks": clocks,
                     "launch": res["launch"], "gpu_launches": res["launches_per_step"] * args.steps})
        if cpu_leg:
            line["cpu_baseline"] = cpu_baseline(wl, res["inputs"])
        line["rope"] = res["rope"]
    else:
        line.update({"value": dec["value"], "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
                     "warmup": args.warmup, "ms_per_step": dec["ms_per_step"], "higher_is_better": True,
                     "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
                     "config": {"workload": dec["workload"]}, "roofline": dec["roofline"], "e2e": dec["e2e"],
                     "gpu_launches": dec["gpu_launches_per_step"] * args.steps})
        if "cpu_baseline" in dec:
            line["cpu_baseline"] = dec["cpu_baseline"]
    line.update(extra)
    if dec:
        line["decode_detail"] = dec
    if cpu_leg:
        line["oracle_tiny"] = oracle_tiny_timing()
    if dec:
        line["decode"] = compact_decode(dec)  # last: the decode half of the metric in brief
    print(json.dumps(line), flush=True)
    if pg:
        pg.destroy_process_group()
    return 0


def prefill_config(wl, ws):
    """The headline workload's `config`, the same for both arms."""
    return {"workload": wl.name + " (RoPE of Q and K + attention, O and LSE)", "batch": wl.batch,
            "seq_len": wl.seq, "q_heads": wl.hq, "kv_heads": wl.hkv, "head_dim": wl.d, "flops_per_step": wl.flops(),
            "l2_flush": True, "parallelism": f"replicas x{ws}"}


def reference_arm(args, synth):
    """The fp64 CPU oracle on the host cores, on a bounded sample of the same workload."""
    import oracle
    oracle.build()
    wl = synth.PREFILL_8K
    inp = wl.make("cpu")
    inputs = (inp["q"], inp["k"], inp["v"], inp["pos"], inp["cu"])
    rows = 192
    for i in range(args.warmup):
        oracle_sample(wl, inputs, 16, 1000 + i)
    times, flops = [], 0.0
    for i in range(args.steps):
        dt, fl = oracle_sample(wl, inputs, rows, 2000 + i)
        times.append(dt)
        flops = fl
    tot = sum(times)
    total_flops = flops * args.steps
    value = total_flops / tot / 1e12
    ms = tot / args.steps * 1e3
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 2), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": prefill_config(wl, dist_env()[0]),
            "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": oracle.num_threads(),
                             "kind": "oracle",
                             "sample": f"each step: {rows} seeded query rows x 64 heads of the 8192-token "
                                       f"prefill (RoPE + bf16 rounding + fp64 three-pass attention)"},
            "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    sys.exit(main())
