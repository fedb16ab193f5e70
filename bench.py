#!/usr/bin/env python3
"""Benchmark of the QK-Normed MLA decode path on GB300.

One step = one pass of the whole path over one batch: qkmla_absorb_query,
qkmla_append of the step's new latents, qkmla_decode (with its split-KV
combine).  Inputs are synthetic (seeded), resident in HBM before timing.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload I] [--impl ours|reference]

Under torchrun each rank runs its own copy of the workload (different seeds):
the path shards by sequence with no data-path collective (weak scaling).
Rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 256 << 20          # > 129 MB L2


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", type=int, default=4,
                    help="index into workloads.WORKLOADS (default 4: B=128, s_q=2, the largest single-GPU workload)")
    ap.add_argument("--s-q", type=int, default=0,
                    help="query tokens per sequence in a step (multi-token prediction / chunked prefill); "
                         "0 keeps the workload's own")
    ap.add_argument("--batch", type=int, default=0,
                    help="keep only the first N sequences of the workload (a reduced case for profiling)")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-plain", action="store_true", help="skip the plain-MLA comparator timing")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="target CPU time of the oracle sample")
    return ap.parse_args()


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            d = json.load(open(p))
            return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                    "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"]))}, "measured"
        except Exception:
            pass
    return dict(FALLBACK_PEAKS), "fallback"


def algorithmic(w: W.Workload, lens: np.ndarray, plain: bool = False, alpha_bytes: int = 4):
    """Algorithmic bytes and MMA flops of one decode call.

    Bytes: every cached token's row (latent + RoPE key) once, its G alpha^k
    scalars (not in plain mode), the query side (q~ in the cache dtype, alpha^q,
    q_rope fp32) and the fp32 output + lse.  Flops: for every (query, visible
    token, head) 2*(d_c + d_r) for the logit and 2*d_c for the output.
    """
    cb = 4 if w.cache_dtype == "f32" else 2
    tokens = int(lens.sum())
    kv_bytes = tokens * (w.d_c + w.d_r) * cb + (0 if plain else tokens * w.G * alpha_bytes)
    rows = w.B * w.s_q * w.H
    q_bytes = rows * (w.d_c * cb + 4 + w.d_r * 4)
    o_bytes = rows * (w.d_c * 4 + 4)
    visible = sum(int(L) - w.s_q + i + 1 for L in lens for i in range(w.s_q))
    flops = visible * w.H * 2 * (2 * w.d_c + w.d_r)
    return kv_bytes + q_bytes + o_bytes, flops, kv_bytes


class ClockSampler:
    """nvidia-smi clock / throttle-reason sampling while the timed region runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
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
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.t.join(timeout=2)
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
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def traffic_from_profiles(kernel_sig: str):
    """dram bytes per launch recorded by an ncu capture of the current kernel source."""
    p = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(p):
        return None
    for ln in open(p):
        f = dict(kv.split("=", 1) for kv in ln.split() if "=" in kv)
        if f.get("sig") == kernel_sig and "bytes_per_launch" in f:
            return float(f["bytes_per_launch"])
    return None


DECODE_SOURCES = ("common.cuh", "tc_ptx.cuh", "decode_common.cuh", "decode_sched.cuh", "decode_tc.cu",
                  "decode_pair.cu", "decode_simt.cu")


def code_of(text: str) -> str:
    """C++/CUDA source without comments and with whitespace collapsed."""
    import re
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_signature(csrc=None):
    """Hash of the code (comments and layout aside) the decode kernels are
    compiled from: a traffic figure recorded under another hash belongs to a
    kernel that has changed."""
    import hashlib
    h = hashlib.sha256()
    csrc = csrc or os.path.join(ROOT, "qk_normed_latent_gb300", "csrc")
    for f in DECODE_SOURCES:
        h.update(code_of(open(os.path.join(csrc, f)).read()).encode())
    return h.hexdigest()[:16]


# ----------------------------------------------------------------------------
# CPU oracle timing (baseline; oracle as it stands)
# ----------------------------------------------------------------------------
def cpu_oracle_rate(w: W.Workload, target_s: float):
    """Time the oracle's whole path (absorb, append of the sequence, explicit
    decode) on whole sequences until about target_s seconds of work, in this one
    Python process (numpy; its BLAS may run the matrix products on several
    threads).  Returns (tokens/s, sample description, seconds, threads busy on
    average = process CPU time / wall time)."""
    import oracle as O
    wk, gq, gk, grq, grk = W.weights(w)
    q, qr = W.queries(w)
    lens = W.seq_lens(w)
    order = [int(b) for b in np.argsort(lens)]   # shortest first: bounded sample
    t_total, cpu_total, done, toks = 0.0, 0.0, [], 0
    # passes over the batch (shortest sequence first) until about target_s seconds,
    # at least one sequence step
    while not done or t_total < target_s:
        for b in order:
            c, r = W.sequence(w, b)
            t0 = time.perf_counter()
            c0 = time.process_time()
            ch, rh, ak = O.append_tokens(c, r, wk, grk, w.eps, w.cache_dtype)
            O.absorb_query(q[b].reshape(w.s_q, w.H, w.d_h), gq, gk, wk, w.eps)
            O.decode_explicit(q[b:b + 1], qr[b:b + 1], gq, gk, grq, wk, [(ch, rh)], w.s_q, w.scale, w.eps)
            t_total += time.perf_counter() - t0
            cpu_total += time.process_time() - c0
            done.append(b)
            toks += w.s_q
            if t_total >= target_s:
                break
    ctx = int(sum(int(lens[b]) for b in done))
    sample = (f"{len(done)} sequence steps over the {w.B} sequences ({len(done) / w.B:.2f} passes, {ctx} cached "
              f"tokens in all), whole path: oracle append of the sequence (alpha^k over all groups), absorb, "
              f"explicit decode with materialised keys")
    return toks / t_total, sample, t_total, cpu_total / max(t_total, 1e-9)


def rank_workload(w0: W.Workload, rank: int) -> W.Workload:
    """Each rank decodes its own batch (same shapes, its own seed): the path
    shards by sequence, so ranks share no data and need no collective."""
    return w0.with_(seed=w0.seed + 7919 * rank) if rank else w0


def max_over_ranks(value: float, world: int, device="cpu") -> float:
    """Max of a per-rank timing over all ranks (the job ends with the slowest)."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank_step: int, world: int, total_ms_max: float, steps: int) -> float:
    """Whole-job rate: the units all ranks processed over the slowest rank's time."""
    return units_per_rank_step * world * steps / (total_ms_max / 1e3)


def config_of(w: W.Workload, lens: np.ndarray, world: int) -> dict:
    """The `config` object of the JSON line (the same for both arms)."""
    return {"workload": w.name, "B": w.B, "s_q": w.s_q, "H": w.H, "G": w.G, "d_c": w.d_c,
            "d_h": w.d_h, "d_r": w.d_r, "cache": w.cache_dtype,
            "context_tokens": int(np.asarray(lens).sum()), "n_append_per_seq": w.n_append,
            "page_size": w.page_size, "parallelism": f"dp{world} (replicas, no collective)",
            "l2": "flushed before every step outside the timed intervals: 256 MiB written, then 256 MiB "
                  "of another buffer read, so L2 holds no input and no dirty line"}


def cpu_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


# ----------------------------------------------------------------------------
def main():
    args = parse()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    w0 = W.WORKLOADS[args.workload]
    if 0 < args.batch < w0.B:
        w0 = W.small(w0, args.batch, W.seq_lens(w0)[:args.batch], name=f"{w0.name}_first{args.batch}")
    if args.s_q > 0 and args.s_q != w0.s_q:
        w0 = w0.with_(s_q=args.s_q, n_append=args.s_q, name=f"{w0.name}_sq{args.s_q}")

    if args.impl == "reference":
        if rank != 0:
            return 0
        rate, sample, secs = 0.0, "", 0.0
        step_rates = []
        for _ in range(args.warmup):
            cpu_oracle_rate(W.small(w0, 1, (min(256, int(W.seq_lens(w0).min())),)), 0.0)
        busy = []
        for _ in range(max(1, args.steps)):
            r_, sample, secs, busy_ = cpu_oracle_rate(w0, args.cpu_seconds / max(1, args.steps))
            busy.append(busy_)
            step_rates.append(r_)
        rate = statistics.median(step_rates)
        line = {"impl": "reference", "metric": "decode tokens/s", "value": rate, "unit": "tokens/s",
                "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": 1000.0 * w0.B * w0.s_q / rate, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": config_of(w0, W.seq_lens(w0), args.gpus),
                "cpu_baseline": {"value": rate, "unit": "tokens/s", "cores": max(1, round(statistics.mean(busy))),
                                 "cores_available": cpu_threads(), "kind": "oracle",
                                 "sample": sample + " per step; one Python process (numpy fp64; cores = its "
                                           "CPU time / wall time, the BLAS threads of the matrix products)"},
                "e2e": {"value": rate, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return 0

    import torch
    import torch.distributed as dist
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    w = rank_workload(w0, rank)

    from qk_normed_latent_gb300 import build as B
    B.build()
    import qk_normed_latent_gb300 as Q
    from qk_normed_latent_gb300.pipeline import DeviceState

    st = DeviceState(w)
    stream = torch.cuda.current_stream()
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    sweep = torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.int32, device="cuda")

    def flush_l2(k):
        """Write a buffer larger than L2, then read another one: L2 ends up holding
        only clean lines of the second, so no timed kernel starts with data of its
        own cached nor pays for writing back the first buffer's dirty lines."""
        flush.fill_(k & 0xFF)
        sweep.sum()

    lens = W.seq_lens(w)
    bytes_alg, flops_alg, _ = algorithmic(w, lens)
    pk, pk_kind = peaks()
    for _ in range(max(3, args.warmup)):
        st.step()
    torch.cuda.synchronize()
    if Q.get_device_status() != 0:
        raise RuntimeError("device status error during warm-up")
    kernel = Q.decode_kernel_name(st.args)
    launches_per_step = 1 + (1 if st.c_new is not None else 0) + Q.decode_launch_count(st.args)

    def capture(calls):
        """A CUDA graph of `calls` (library calls on one state).  Kernel arguments and
        tensor maps are fixed at capture; sequence lengths and the split plan are
        read on the device at every replay."""
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            calls()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        with torch.cuda.graph(g, capture_error_mode="thread_local"):
            calls()
        torch.cuda.synchronize()
        return g

    def graphs_of(state):
        step_g = capture(lambda: (state.absorb(), state.append_step(), Q.decode_raw(state.args)))
        dec_g = capture(lambda: Q.decode_raw(state.args))
        return step_g, dec_g

    def timed(graph, K):
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
        for k in range(K):
            flush_l2(k)                                 # a cold, clean L2 before every replay
            ev[k][0].record(stream)
            graph.replay()
            ev[k][1].record(stream)
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in ev]

    step_graph, dec_graph = graphs_of(st)
    for _ in range(max(3, args.warmup)):
        step_graph.replay()
    torch.cuda.synchronize()

    clk = ClockSampler(local)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clk.start()
    time.sleep(0.3)
    step_ms = timed(step_graph, args.steps)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    # the decode call alone (scheduler if any, decode kernel, combine): the roofline's interval
    dec_ms = timed(dec_graph, args.steps)
    clocks = clk.stop()
    total_ms = max_over_ranks(sum(step_ms), world, device="cuda")
    if Q.get_device_status() != 0:
        raise RuntimeError("device status error in the timed region")
    ms_per_step = total_ms / args.steps
    tokens_per_step = w.B * w.s_q
    value = job_throughput(tokens_per_step, world, total_ms, args.steps)
    dec_avg = statistics.mean(dec_ms)

    # roofline of the dominant kernel (the decode call: decode kernel + combine)
    t_hbm = bytes_alg / (pk["hbm_gbs"] * 1e9)
    t_mma = flops_alg / (pk["bf16_tflops"] * 1e12)
    if t_hbm >= t_mma:
        roof = {"bound": "hbm", "achieved": bytes_alg / (dec_avg * 1e-3) / 1e9, "peak": pk["hbm_gbs"],
                "unit": "GB/s"}
    else:
        roof = {"bound": "tensor", "achieved": flops_alg / (dec_avg * 1e-3) / 1e12, "peak": pk["bf16_tflops"],
                "unit": "TFLOP/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"] = traffic_from_profiles(kernel_signature() + ":" + w.name)
    roof["peak_source"] = f"{pk_kind} (MEASURED_PEAKS.json)" if pk_kind == "measured" else "fallback (6.8 TB/s, 1.9 PF/s)"
    roof["kernel"] = f"qkmla_decode[{kernel}]"
    roof["algorithmic_bytes_per_launch"] = bytes_alg
    roof["algorithmic_flops_per_launch"] = flops_alg
    roof["flops_rule"] = "per (query token, visible cached token, head): 2 (d_c + d_r) logit + 2 d_c output"
    if roof["bound"] == "tensor":
        # the decode call is timed alone (graph replays back to back): the burst peak; the
        # sustained figure is given beside it
        roof["frac_of_sustained"] = roof["achieved"] / pk["bf16_tflops_sustained"]
    roof["roofline_us"] = max(t_hbm, t_mma) * 1e6

    # plain-MLA comparator: same kernels with the alpha scaling off; and the same QK-norm
    # path with the scalar cache in fp16 (half the alpha^k bytes)
    plain = None
    alpha_f16 = None
    if not args.no_plain:
        sp = DeviceState(w, plain=True)
        sb = DeviceState(w.with_(alpha_dtype="f16"))
        for _ in range(3):
            sp.step()
            sb.step()
        torch.cuda.synchronize()
        if Q.get_device_status() != 0:
            raise RuntimeError("device status error in the comparator warm-up")
        sp_step_g, sp_dec_g = graphs_of(sp)
        sb_step_g, sb_dec_g = graphs_of(sb)
        kp = min(args.steps, 100)
        # the three variants' replays are interleaved one by one, so drift over the
        # run (and the ~2 us modes of short replays) falls on all three alike
        p_step, q_step, b_step, p_dec, q_dec, b_dec = [], [], [], [], [], []
        for _ in range(kp):
            for g_, out in ((sp_step_g, p_step), (step_graph, q_step), (sb_step_g, b_step),
                            (sp_dec_g, p_dec), (dec_graph, q_dec), (sb_dec_g, b_dec)):
                out += timed(g_, 1)
        med = statistics.median
        plain = {"decode_ms": med(p_dec), "qknorm_decode_ms": med(q_dec),
                 "overhead_pct": 100.0 * (med(q_dec) / med(p_dec) - 1.0),
                 "step_overhead_pct": 100.0 * (med(q_step) / med(p_step) - 1.0)}
        bytes_b, _, _ = algorithmic(w, lens, alpha_bytes=2)
        alpha_f16 = {"decode_ms": med(b_dec), "overhead_vs_plain_pct": 100.0 * (med(b_dec) / med(p_dec) - 1.0),
                      "step_overhead_vs_plain_pct": 100.0 * (med(b_step) / med(p_step) - 1.0),
                      "kv_gbs": bytes_b / (med(b_dec) * 1e-3) / 1e9,
                      "byte_floor_pct": 100.0 * (w.G * 2) / ((w.d_c + w.d_r) * (4 if w.cache_dtype == "f32" else 2))}
        if Q.get_device_status() != 0:
            raise RuntimeError("device status error in the comparator timing")
        del sp_step_g, sp_dec_g, sp, sb_step_g, sb_dec_g, sb

    # the value up-projection of this step's latent output (its own call, timed alone)
    wv = torch.from_numpy(W.value_weights(w)).to("cuda").to(torch.bfloat16)
    v_out = torch.empty((w.B, w.s_q, w.H, wv.shape[2]), dtype=torch.float32, device="cuda")
    up_call = Q.prepare_up_project(st.o, wv, v_out)
    up_g = capture(lambda: up_call())
    up_ms = statistics.median(timed(up_g, min(args.steps, 100)))
    if Q.get_device_status() != 0:
        raise RuntimeError("device status error in the up-projection timing")
    up_rows = w.B * w.s_q * w.H
    up_bytes = up_rows * w.d_c * 4 + wv.numel() * 2 + up_rows * wv.shape[2] * 4
    up_flops = 2 * up_rows * w.d_c * wv.shape[2]
    up_project = {"ms": up_ms, "gbs": up_bytes / (up_ms * 1e-3) / 1e9, "tflops": up_flops / (up_ms * 1e-3) / 1e12,
                  "bound": "hbm", "frac_of_hbm": up_bytes / (up_ms * 1e-3) / 1e9 / pk["hbm_gbs"],
                  "algorithmic_bytes": up_bytes, "algorithmic_flops": up_flops}
    del up_g

    # the query projection from the layer input with its RoPE rotation (its own call, timed
    # alone): d_x = 1536 for the 128-head shape (the DeepSeek-V3 query down-projection
    # width), 4 d_h otherwise
    d_x = 1536 if w.H == 128 else 4 * w.d_h
    xq, wq = W.query_inputs(w, d_x)
    xq_d = torch.from_numpy(xq.reshape(w.rows, d_x)).to("cuda").to(torch.bfloat16)
    wq_d = torch.from_numpy(wq).to("cuda").to(torch.bfloat16)
    pos_d = torch.from_numpy(np.array([int(lens[b]) - w.s_q + i for b in range(w.B) for i in range(w.s_q)],
                                      dtype=np.int32)).to("cuda")
    pq_q = torch.empty((w.rows, w.H, w.d_h), dtype=torch.float32, device="cuda")
    pq_r = torch.empty((w.rows, w.H, w.d_r), dtype=torch.float32, device="cuda")
    pq_call = Q.prepare_project_query(xq_d, wq_d, pos_d, 10000.0, pq_q, pq_r)
    pq_g = capture(lambda: pq_call())
    pq_ms = statistics.median(timed(pq_g, min(args.steps, 100)))
    if Q.get_device_status() != 0:
        raise RuntimeError("device status error in the projection timing")
    pq_flops = 2 * w.rows * d_x * w.H * (w.d_h + w.d_r)
    pq_bytes = w.rows * d_x * 2 + wq.size * 2 + w.rows * w.H * (w.d_h + w.d_r) * 4
    project_query = {"ms": pq_ms, "d_x": d_x, "tflops": pq_flops / (pq_ms * 1e-3) / 1e12,
                     "gbs": pq_bytes / (pq_ms * 1e-3) / 1e9,
                     "frac_of_bf16": pq_flops / (pq_ms * 1e-3) / 1e12 / pk["bf16_tflops"],
                     "frac_of_hbm": pq_bytes / (pq_ms * 1e-3) / 1e9 / pk["hbm_gbs"],
                     "algorithmic_flops": pq_flops, "algorithmic_bytes": pq_bytes}
    del pq_g

    # end to end through the public API with host buffers: H2D of the step's inputs,
    # the three calls, D2H of o and lse, all inside the timed region.  The inputs
    # (q, q_rope and the step's new tokens) live in one pinned host buffer and one
    # device buffer, the results likewise: one copy each way.
    h_in = st.step_in.cpu().pin_memory()
    h_out = torch.empty(st.step_out.shape, dtype=torch.uint8).pin_memory()
    h2d = h_in.numel()
    d2h = h_out.numel()
    K2 = min(args.steps, 100)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K2)]
    for k in range(K2):
        flush_l2(k)
        ev[k][0].record(stream)
        st.step_in.copy_(h_in, non_blocking=True)
        st.step()
        h_out.copy_(st.step_out, non_blocking=True)
        ev[k][1].record(stream)
    torch.cuda.synchronize()
    e2e_ms = sum(a.elapsed_time(b) for a, b in ev) / K2
    e2e = {"value": tokens_per_step * world / (e2e_ms / 1e3), "unit": "tokens/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rate, sample, secs, busy = cpu_oracle_rate(w, args.cpu_seconds)
        cpu = {"value": rate, "unit": "tokens/s", "cores": max(1, round(busy)), "cores_available": cpu_threads(),
               "kind": "oracle",
               "sample": sample + "; one Python process (numpy fp64; cores = its CPU time / wall time, the BLAS "
                                  "threads of the matrix products)",
               "seconds": secs}

    if rank == 0:
        line = {
            "metric": "decode tokens/s", "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.cache_dtype,
            "data": "synthetic",
            "config": config_of(w, lens, world),
            "launch": "each step replays a CUDA graph of absorb, append and the decode call; decode_ms and the "
                      "roofline replay a graph of the decode call alone; e2e drives the Python API call by call",
            "decode_ms": dec_avg,
            "kv_gbs": bytes_alg / (dec_avg * 1e-3) / 1e9,
            "roofline": roof,
            "plain_mla": plain,
            "alpha_f16": alpha_f16,
            "up_project": up_project,
            "project_query": project_query,
            "e2e": e2e,
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clocks,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
