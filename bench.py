"""Benchmark of the streaming-attention hot path on GB300.

One step = one causal GQA prefill of the Llama3-70B-shaped workload (B1 Hq64 Hkv8
S8192 d128, bf16, Q x2) plus one split-KV decode of the Llama3-70B decode workload
(B4 Hq64 Hkv8, 32768 cached keys, 16 splits), both through the C ABI (libgbattn.so).

Printed JSON line (rank 0):
  value      prefill TFLOP/s, FLOPs = 4 B Hq Sq Skv d / 2 (causal), inputs resident in HBM
  decode     the decode half: KV GB/s (algorithmic bytes: K, V, Q, O, LSE) with its roofline
  roofline   prefill kernel: achieved TFLOP/s vs the measured dense bf16 peak
  configs    every one of the five workloads timed on its own (L2 flushed before each
             call, CUDA events): 1 tiny fp32, 2 small causal GQA prefill, 3 and 4 (the
             step's two calls), 5 ragged decode, each with its fraction of the roofline
  e2e        the same metric through attn_fwd_host (and the decode half through
             attn_decode_host): pinned-host inputs copied in and outputs copied out by
             the call (chunked, overlapped with the kernels) inside the timed region,
             every step
  cpu_baseline  the fp64 CPU oracle on a bounded sample of the same workload; the same
             leg compares sampled rows of every timed output with the oracle and fails the
             run on a mismatch
L2 is flushed (a 512 MiB write, then a read of it so no dirty lines remain) before every
timed call, outside the kernels' event windows.

--impl reference times the fp64 CPU oracle instead (a bounded row sample per step).
Multi-GPU (torchrun, N > 1): N independent replicas, weak scaling, no collective on the
data path; the step time is the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np
import torch

import attn_workloads as wl

PREFILL = wl.WORKLOADS[3]
DECODE = wl.WORKLOADS[4]
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
NOMINAL_HBM_GBS = 7900.0          # GB300 HBM3e nominal, for the decode fractions' second reading
L2_FLUSH_BYTES = 512 << 20
METRIC = "prefill attn TFLOP/s & decode KV GB/s at 1 GB300, % of roofline"
CSRC = os.path.join(ROOT, "streaming_attention_flashattention_gb300", "csrc")
# DRAM traffic per launch from the committed ncu summaries: each summary carries a line
#   bench-traffic: bytes_per_launch=<n> sources_sha256=<hash of the kernel's sources>
# and the figure is reported only while the sources still hash to the same value.
TRAFFIC_SOURCES = {
    "prefill": ("prefill_fwd_kernel_llama70b_causal_s8192.md",
                ["prefill_tcgen05.cu", "common.cuh", "kernels.h"]),
    "decode": ("decode_split_kernel_llama70b_l32768.md",
               ["decode_splitkv.cu", "decode_splits.cuh", "common.cuh", "kernels.h"]),
}


def sources_sha256(files) -> str:
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(CSRC, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def committed_traffic(kind: str):
    """(bytes per launch, note) from the ncu summary, or (None, why) when stale or absent."""
    md, files = TRAFFIC_SOURCES[kind]
    path = os.path.join(ROOT, "profiles", md)
    try:
        text = open(path).read()
    except OSError:
        return None, f"no summary {md}"
    m = re.search(r"bench-traffic: bytes_per_launch=(\d+) sources_sha256=([0-9a-f]{64})", text)
    if not m:
        return None, f"{md} has no bench-traffic line"
    if m.group(2) != sources_sha256(files):
        return None, f"kernel sources changed since the capture in {md}"
    return int(m.group(1)), f"ncu capture in profiles/{md}"


def prefill_flops(w: wl.Workload) -> float:
    f = 4.0 * w.B * w.Hq * w.Sq * w.Skv * w.d
    return f / 2 if w.causal else f


def chunk_flops(w: wl.Workload) -> float:
    """4 d B Hq x (visible keys summed over the chunk's rows); chunk at the context's end."""
    ctx = w.len_hi
    if w.causal:
        vis = w.Sq * (ctx - w.Sq) + w.Sq * (w.Sq + 1) / 2
    else:
        vis = w.Sq * ctx
    return 4.0 * w.d * w.B * w.Hq * vis


def decode_bytes(w: wl.Workload, lens) -> float:
    kv = float(sum(int(x) for x in lens)) * w.Hkv * w.d * 2 * 2
    q_o = 2.0 * w.B * w.Hq * w.d * 2
    return kv + q_o + w.B * w.Hq * 4


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return pk, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle samples during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 6:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[2:6]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------------------
# CPU oracle legs (the only places this script runs oracle/)
# ---------------------------------------------------------------------------------------

def oracle_sample_prefill(q_np, k_np, v_np, w: wl.Workload, n_rows: int, seed: int):
    import oracle
    rng = np.random.default_rng(seed)
    rows = rng.integers(0, w.B * w.Hq * w.Sq, n_rows)
    i = rows % w.Sq
    flops = float(np.sum(4.0 * w.d * ((i + 1 + (w.Skv - w.Sq)) if w.causal else np.full_like(i, w.Skv))))
    t0 = time.perf_counter()
    o, lse = oracle.attention(q_np, k_np, v_np, w.scale, w.causal, rows=rows)
    return flops, time.perf_counter() - t0, rows, o, lse


def _check_rows(name, o_gpu, lse_gpu, o_ref, lse_ref, dtype):
    """Max / mean |dO| and max |dLSE| of sampled rows against the oracle; raises past the
    parity bars (bf16: 2e-2 / 2e-3, fp32: 1e-4; LSE 1e-3)."""
    o_gpu = np.asarray(o_gpu, dtype=np.float64)
    err = np.abs(o_gpu - o_ref)
    lerr = float(np.abs(np.asarray(lse_gpu, dtype=np.float64) - lse_ref).max())
    mx, mean = float(err.max()), float(err.mean())
    ok = np.all(np.isfinite(o_gpu)) and lerr <= 1e-3 and (
        mx <= 1e-4 if dtype == "fp32" else (mx <= 2e-2 and mean <= 2e-3))
    rec = {"rows": int(o_ref.reshape(-1, o_ref.shape[-1]).shape[0]), "max_abs": mx,
           "mean_abs": mean, "lse_max_abs": lerr, "ok": bool(ok)}
    if not ok:
        raise RuntimeError(f"parity check failed on {name}: {rec}")
    return rec


def cpu_baseline_and_check(inputs, outputs, target_s: float = 12.0):
    """The fp64 oracle timed on a bounded sample of the prefill workload (the baseline), and
    every timed GPU output compared with the oracle on sampled rows (outside any timing)."""
    import oracle
    w = PREFILL
    q, k, v = inputs[3]
    q_np, k_np, v_np = wl.to_oracle(q), wl.to_oracle(k), wl.to_oracle(v)
    n = 256
    _, dt, _, _, _ = oracle_sample_prefill(q_np, k_np, v_np, w, n, 1)
    n2 = int(min(200000, max(n, n * target_s / max(dt, 1e-3))))
    flops, dt, rows, o_ref, lse_ref = oracle_sample_prefill(q_np, k_np, v_np, w, n2, 2)
    base = {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": oracle.max_threads(),
            "kind": "oracle",
            "sample": f"{n2} random query rows of {w.name} (fp64 two-pass definition, "
                      f"{dt:.1f} s, {flops / 1e9:.1f} GFLOP algorithmic)"}
    checks = {}
    o3, l3 = outputs[3]
    checks["3"] = _check_rows(w.name, o3.reshape(-1, w.d)[rows], l3.reshape(-1)[rows],
                              o_ref, lse_ref, "bf16")
    rng = np.random.default_rng(7)
    for idx in (1, 2):
        wi = wl.WORKLOADS[idx]
        qi, ki, vi = inputs[idx]
        oi, li = outputs[idx]
        n_rows = wi.B * wi.Hq * wi.Sq
        r = np.arange(n_rows) if n_rows <= 512 else rng.integers(0, n_rows, 512)
        o_ref, lse_ref = oracle.attention(wl.to_oracle(qi), wl.to_oracle(ki), wl.to_oracle(vi),
                                          wi.scale, wi.causal, rows=r)
        checks[str(idx)] = _check_rows(wi.name, oi.reshape(-1, wi.d)[r], li.reshape(-1)[r],
                                       o_ref, lse_ref, wi.dtype)
    for idx in (4, 5):
        wi = wl.WORKLOADS[idx]
        qi, kc, vc, kl = inputs[idx]
        oi, li = outputs[idx]
        r = rng.choice(wi.B * wi.Hq, 96, replace=False)
        o_ref, lse_ref = oracle.attention(wl.to_oracle(qi), wl.to_oracle(kc), wl.to_oracle(vc),
                                          wi.scale, False, kv_len=kl.numpy(), rows=r)
        checks[str(idx)] = _check_rows(wi.name, oi.reshape(-1, wi.d)[r], li.reshape(-1)[r],
                                       o_ref, lse_ref, "bf16")
    base["checked"] = checks
    return base


def run_reference(args, rank, world):
    """--impl reference: the fp64 CPU oracle timed on a bounded sample per step."""
    if rank != 0:
        return
    import oracle
    q, k, v = wl.prefill_inputs(PREFILL)
    q_np, k_np, v_np = wl.to_oracle(q), wl.to_oracle(k), wl.to_oracle(v)
    rows_per_step = 2048
    for s in range(args.warmup):
        oracle_sample_prefill(q_np, k_np, v_np, PREFILL, rows_per_step, 100 + s)
    tot_f, tot_t = 0.0, 0.0
    for s in range(args.steps):
        f, t, _, _, _ = oracle_sample_prefill(q_np, k_np, v_np, PREFILL, rows_per_step, 1000 + s)
        tot_f += f
        tot_t += t
    val = tot_f / tot_t / 1e12
    line = {
        "impl": "reference", "metric": METRIC,
        "value": val, "unit": "TFLOP/s", "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": tot_t / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": config_dict(args),
        "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": oracle.max_threads(),
                         "kind": "oracle",
                         "sample": f"{rows_per_step} random query rows of {PREFILL.name} per step"},
        "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def max_over_ranks(values, device=None):
    """Element-wise max of per-rank timings (the slowest rank sets the step time).  A
    no-op when torch.distributed is not initialised (one process)."""
    if not (torch.distributed.is_available() and torch.distributed.is_initialized()):
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return [float(x) for x in t.cpu()]


def config_dict(args):
    return {"workload": f"{PREFILL.name} + {DECODE.name}",
            "prefill": {"B": PREFILL.B, "Hq": PREFILL.Hq, "Hkv": PREFILL.Hkv, "Sq": PREFILL.Sq,
                        "Skv": PREFILL.Skv, "d": PREFILL.d, "causal": PREFILL.causal,
                        "q_scale": PREFILL.q_scale},
            "decode": {"B": DECODE.B, "Hq": DECODE.Hq, "Hkv": DECODE.Hkv, "kv_len": DECODE.len_hi,
                       "d": DECODE.d, "num_splits": DECODE.num_splits},
            "parallelism": f"replicas{args.gpus}",
            "l2": "flushed before every timed call (512 MiB write, then read back)"}


# ---------------------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------------------

def run_gpu(args, rank, world, local_rank):
    import streaming_attention_flashattention_gb300 as gb
    from streaming_attention_flashattention_gb300 import build as gbbuild
    if rank == 0:
        gbbuild.build()
    if world > 1:
        torch.distributed.barrier()
    gb.load_library()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    peaks, peak_src = load_peaks()
    nsm = torch.cuda.get_device_properties(dev).multi_processor_count

    # inputs (seeded, CPU-generated), resident in HBM before timing
    q_c, k_c, v_c = wl.prefill_inputs(PREFILL)
    dq_c, dk_c, dv_c, dl_c = wl.decode_inputs(DECODE)
    q, k, v = q_c.to(dev), k_c.to(dev), v_c.to(dev)
    dq, dk, dv, dl = dq_c.to(dev), dk_c.to(dev), dv_c.to(dev), dl_c.to(dev)
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
    do = torch.empty_like(dq)
    dlse = torch.empty(dq.shape[:2], dtype=torch.float32, device=dev)
    ws = torch.empty(gb.attn_decode_workspace_size(DECODE.B, DECODE.Hq, DECODE.Hkv, DECODE.Skv,
                                                   DECODE.d, DECODE.num_splits),
                     dtype=torch.uint8, device=dev)
    flush_buf = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def flush():
        """Evict L2: write a buffer 4x its size, then read it back so that no dirty lines
        are left for the next timed kernel to write back."""
        flush_buf.zero_()
        flush_buf.sum()

    def step(evs=None):
        flush()
        if evs is not None:
            evs[0].record(stream)
        gb.attn_fwd(q, k, v, causal=PREFILL.causal, scale=PREFILL.scale, out=o, lse=lse)
        if evs is not None:
            evs[1].record(stream)
        # flush again: the prefill's dirty output lines would otherwise be written back
        # inside the decode window
        flush()
        if evs is not None:
            evs[2].record(stream)
        gb.attn_decode_splitkv(dq, dk, dv, dl, num_splits=DECODE.num_splits,
                               scale=DECODE.scale, out=do, lse=dlse, workspace=ws)
        if evs is not None:
            evs[3].record(stream)

    def time_calls(fn, reps):
        """Mean CUDA-event time (ms) of `fn` over `reps` calls, L2 flushed before each."""
        ms = []
        for _ in range(reps):
            flush()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            torch.cuda.synchronize(dev)
            ms.append(e0.elapsed_time(e1))
        return sum(ms) / len(ms)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    st, word = gb.attn_last_device_error()
    if st != 0:
        raise RuntimeError(f"device error word {word} during warm-up")

    # the other three workloads, timed one call at a time (inputs resident, outputs kept
    # for the oracle check)
    extra_in, extra_out, extra_fn = {}, {}, {}
    for idx in (1, 2):
        wi = wl.WORKLOADS[idx]
        qi, ki, vi = wl.prefill_inputs(wi)
        extra_in[idx] = (qi, ki, vi)
        gq, gk, gv = qi.to(dev), ki.to(dev), vi.to(dev)
        go = torch.empty_like(gq)
        gl = torch.empty(gq.shape[:3], dtype=torch.float32, device=dev)
        extra_out[idx] = (go, gl)
        extra_fn[idx] = (lambda gq=gq, gk=gk, gv=gv, go=go, gl=gl, wi=wi:
                         gb.attn_fwd(gq, gk, gv, causal=wi.causal, scale=wi.scale, out=go, lse=gl))
    w5 = wl.WORKLOADS[5]
    q5, k5, v5, l5 = wl.decode_inputs(w5)
    extra_in[5] = (q5, k5, v5, l5)
    g5 = [t.to(dev) for t in (q5, k5, v5, l5)]
    o5 = torch.empty_like(g5[0])
    lse5 = torch.empty(g5[0].shape[:2], dtype=torch.float32, device=dev)
    ws5 = torch.empty(gb.attn_decode_workspace_size(w5.B, w5.Hq, w5.Hkv, w5.Skv, w5.d, w5.num_splits),
                      dtype=torch.uint8, device=dev)
    extra_out[5] = (o5, lse5)
    extra_fn[5] = lambda: gb.attn_decode_splitkv(*g5, num_splits=w5.num_splits, scale=w5.scale,
                                                 out=o5, lse=lse5, workspace=ws5)
    for idx in extra_fn:
        for _ in range(3):
            extra_fn[idx]()
    torch.cuda.synchronize(dev)

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(local_rank) as clk:
        t_wall0 = time.perf_counter()
        for s in range(args.steps):
            step(evs[s])
        torch.cuda.synchronize(dev)
        t_wall = time.perf_counter() - t_wall0
        if world > 1:
            torch.distributed.barrier()
        extra_ms = {idx: time_calls(extra_fn[idx], max(args.steps, 10)) for idx in (1, 2, 5)}
    pre_ms = [e[0].elapsed_time(e[1]) for e in evs]
    dec_ms = [e[2].elapsed_time(e[3]) for e in evs]
    pre_avg = sum(pre_ms) / len(pre_ms)
    dec_avg = sum(dec_ms) / len(dec_ms)
    step_ms = pre_avg + dec_avg
    pre_avg, dec_avg, step_ms = max_over_ranks([pre_avg, dec_avg, step_ms], dev)
    for idx in extra_ms:
        extra_ms[idx] = max_over_ranks([extra_ms[idx]], dev)[0]

    # chunked prefill against a KV cache (a widening beyond the step's two calls)
    chunk = None
    if not args.no_chunk:
        wc = wl.EXTRA_WORKLOADS[6]
        cq, ckc, cvc, cctx = (x.to(dev) if torch.is_tensor(x) else x for x in wl.chunk_inputs(wc))
        co = torch.empty_like(cq)
        clse = torch.empty(cq.shape[:3], dtype=torch.float32, device=dev)
        for _ in range(3):
            gb.attn_prefill_kvcache(cq, ckc, cvc, cctx, causal=wc.causal, scale=wc.scale, out=co, lse=clse)
        cm = max_over_ranks([time_calls(lambda: gb.attn_prefill_kvcache(
            cq, ckc, cvc, cctx, causal=wc.causal, scale=wc.scale, out=co, lse=clse), 10)], dev)[0]
        chunk = {"workload": wc.name, "ms": cm, "value": chunk_flops(wc) / (cm * 1e-3) / 1e12,
                 "unit": "TFLOP/s"}
        del cq, ckc, cvc, co, clse

    # multi-token decode (4 new tokens per sequence)
    mtok = None
    if not args.no_chunk:
        wm = wl.EXTRA_WORKLOADS[7]
        mq, mkc, mvc, mkl_c = wl.multitoken_inputs(wm)
        mq, mkc, mvc, mkl = mq.to(dev), mkc.to(dev), mvc.to(dev), mkl_c.to(dev)
        mo = torch.empty_like(mq)
        mlse = torch.empty(mq.shape[:3], dtype=torch.float32, device=dev)
        mws = torch.empty(gb.load_library().attn_decode_multitoken_workspace_size(
            wm.B, wm.Hq, wm.Hkv, wm.Sq, wm.Skv, wm.d, wm.num_splits), dtype=torch.uint8, device=dev)
        run_m = lambda: gb.attn_decode_multitoken(mq, mkc, mvc, mkl, num_splits=wm.num_splits,
                                                  scale=wm.scale, out=mo, lse=mlse, workspace=mws)
        for _ in range(3):
            run_m()
        mm = max_over_ranks([time_calls(run_m, 10)], dev)[0]
        mbytes = float(mkl_c.sum()) * wm.Hkv * wm.d * 2 * 2 + 2.0 * wm.B * wm.Hq * wm.Sq * wm.d * 2
        mtok = {"workload": wm.name, "ms": mm, "value": mbytes / (mm * 1e-3) / 1e9, "unit": "GB/s"}
        del mq, mkc, mvc, mkl, mo, mlse, mws

    # sequence-parallel pieces: one ring step of the Llama3-70B prefill over 8 ranks (a rank's
    # 8 query heads, all 8192 positions, against KV slice 3 of 8: keys 3072..4095 of its KV
    # head) and the merge of that step into an fp32 accumulator (in place)
    spar = None
    if not args.no_chunk:
        Sr, Lr, kp = PREFILL.Sq, PREFILL.Skv // 8, 3 * (PREFILL.Skv // 8)
        g = torch.Generator().manual_seed(97)
        rq = torch.randn((1, 8, Sr, PREFILL.d), generator=g).to(torch.bfloat16).to(dev)
        rk = torch.randn((1, 1, Lr, PREFILL.d), generator=g).to(torch.bfloat16).to(dev)
        rv = torch.randn((1, 1, Lr, PREFILL.d), generator=g).to(torch.bfloat16).to(dev)
        ro = torch.empty_like(rq)
        rl = torch.empty((1, 8, Sr), dtype=torch.float32, device=dev)
        acc_o = torch.zeros((1, 8, Sr, PREFILL.d), dtype=torch.float32, device=dev)
        acc_l = torch.full((1, 8, Sr), float("-inf"), device=dev)
        run_r = lambda: gb.attn_fwd_positions(rq, rk, rv, 0, kp, scale=PREFILL.scale, out=ro, lse=rl)
        run_g = lambda: gb.attn_merge(acc_o, acc_l, ro, rl, out=acc_o, lse_out=acc_l)
        for _ in range(3):
            run_r(); run_g()
        rm = max_over_ranks([time_calls(run_r, 10)], dev)[0]
        gm = max_over_ranks([time_calls(run_g, 10)], dev)[0]
        vis = sum(min(Lr, max(0, i - kp + 1)) for i in range(Sr))       # visible keys, all rows
        rflops = 4.0 * PREFILL.d * vis * 8
        rows = 8 * Sr
        gbytes = rows * (PREFILL.d * (4 + 2 + 4) + 12)                   # acc in, part in, acc out
        spar = {"ring_step": {"shape": f"q 1x8x{Sr}x{PREFILL.d}, kv slice 1x1x{Lr} at {kp}",
                              "ms": rm, "value": rflops / (rm * 1e-3) / 1e12, "unit": "TFLOP/s"},
                "merge": {"rows": rows, "ms": gm, "value": gbytes / (gm * 1e-3) / 1e9,
                          "unit": "GB/s", "bound": "hbm"}}
        del rq, rk, rv, ro, rl, acc_o, acc_l

    st, word = gb.attn_last_device_error()
    if st != 0:
        raise RuntimeError(f"device error word {word} during the timed steps")

    # outputs of the timed calls, for the oracle check (copied after timing)
    outputs = {3: (o.float().cpu().numpy(), lse.cpu().numpy()),
               4: (do.float().cpu().numpy(), dlse.cpu().numpy())}
    for idx in (1, 2, 5):
        outputs[idx] = (extra_out[idx][0].float().cpu().numpy(), extra_out[idx][1].cpu().numpy())
    del g5, o5, lse5, ws5

    e2e_pre = e2e_dec = float("nan")
    h2d = d2h = 0
    if not args.no_e2e:
        # ---- end to end: pinned host inputs in, results out, every step ----
        hq, hk, hv = q_c.pin_memory(), k_c.pin_memory(), v_c.pin_memory()
        hdq, hdk, hdv, hdl = dq_c.pin_memory(), dk_c.pin_memory(), dv_c.pin_memory(), dl_c.pin_memory()
        ho = torch.empty(o.shape, dtype=o.dtype).pin_memory()
        hlse = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
        hdo = torch.empty(do.shape, dtype=do.dtype).pin_memory()
        hdlse = torch.empty(dlse.shape, dtype=dlse.dtype).pin_memory()
        hws = torch.empty(gb.attn_fwd_host_workspace_size(
            PREFILL.B, PREFILL.Hq, PREFILL.Hkv, PREFILL.Sq, PREFILL.Skv, PREFILL.d), dtype=torch.uint8, device=dev)
        hdws = torch.empty(gb.attn_decode_host_workspace_size(
            DECODE.B, DECODE.Hq, DECODE.Hkv, DECODE.Skv, DECODE.d, DECODE.num_splits),
            dtype=torch.uint8, device=dev)
        h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv, hdq, hdk, hdv, hdl))
        d2h = sum(t.numel() * t.element_size() for t in (ho, hlse, hdo, hdlse))

        def e2e_step(ev=None):
            flush()
            if ev is not None:
                ev[0].record(stream)
            # the C-ABI call on host buffers: inputs copied in, outputs copied back, the
            # copies of neighbouring chunks overlapped with the kernel
            gb.attn_fwd_host(hq, hk, hv, causal=PREFILL.causal, scale=PREFILL.scale, out=ho,
                             lse=hlse, workspace=hws)
            if ev is not None:
                ev[1].record(stream)
            gb.attn_decode_host(hdq, hdk, hdv, hdl, num_splits=DECODE.num_splits,
                                scale=DECODE.scale, out=hdo, lse=hdlse, workspace=hdws)
            if ev is not None:
                ev[2].record(stream)

        e2e_step()
        torch.cuda.synchronize(dev)
        n_e2e = args.steps
        evs2 = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n_e2e)]
        for s in range(n_e2e):
            e2e_step(evs2[s])
        torch.cuda.synchronize(dev)
        e2e_pre = sum(e[0].elapsed_time(e[1]) for e in evs2) / n_e2e
        e2e_dec = sum(e[1].elapsed_time(e[2]) for e in evs2) / n_e2e
        e2e_pre, e2e_dec = max_over_ranks([e2e_pre, e2e_dec], dev)
        ok = bool(torch.isfinite(ho.float()).all()) and bool(torch.isfinite(hdo.float()).all())
        if not ok:
            raise RuntimeError("non-finite output in the end-to-end run")

    if rank != 0:
        return
    flops = prefill_flops(PREFILL)
    dbytes = decode_bytes(DECODE, dl_c.tolist())
    pre_tflops = flops / (pre_avg * 1e-3) / 1e12 * world
    dec_gbs = dbytes / (dec_avg * 1e-3) / 1e9 * world
    peak_tf = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    peak_bw = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    if spar is not None:
        spar["merge"]["peak"] = peak_bw
        spar["merge"]["frac"] = spar["merge"]["value"] / peak_bw
        spar["ring_step"]["frac"] = spar["ring_step"]["value"] / peak_tf
    per_gpu_tf = flops / (pre_avg * 1e-3) / 1e12
    per_gpu_bw = dbytes / (dec_avg * 1e-3) / 1e9
    if chunk is not None:
        chunk["frac"] = chunk["value"] / peak_tf      # per GPU
    if mtok is not None:
        mtok["frac"] = mtok["value"] / peak_bw         # per GPU
    pre_plan = gb.attn_prefill_plan(PREFILL.B, PREFILL.Hq, PREFILL.Hkv, PREFILL.Sq, PREFILL.Skv,
                                    PREFILL.causal, nsm)
    dec_plan = gb.attn_decode_plan(DECODE.B, DECODE.Hq, DECODE.Hkv, 1, DECODE.Skv, DECODE.d,
                                   DECODE.num_splits, nsm)
    launches = (1 + (pre_plan["tail_pairs"] > 0)) + (1 + (dec_plan["merge"] != "single_launch"))
    traffic_pre, traffic_pre_src = committed_traffic("prefill")
    traffic_dec, traffic_dec_src = committed_traffic("decode")

    def prefill_entry(idx, ms):
        wi = wl.WORKLOADS[idx]
        tf = prefill_flops(wi) / (ms * 1e-3) / 1e12
        pl = gb.attn_prefill_plan(wi.B, wi.Hq, wi.Hkv, wi.Sq, wi.Skv, wi.causal, nsm)
        e = {"workload": wi.name, "ms": ms, "value": tf, "unit": "TFLOP/s"}
        if wi.dtype == "fp32":
            e.update({"frac": None, "bound": "fp32 CUDA cores (correctness path, no roofline target)",
                      "kernel": f"attn_fwd_f32_kernel<{wi.d}>"})
        else:
            e.update({"frac": tf / peak_tf, "bound": "tensor", "peak": peak_tf,
                      "kernel": f"prefill_fwd_kernel<{wi.d}> ({pl['mode']})"})
        return e

    def decode_entry(w, lens, ms):
        gbs = decode_bytes(w, lens) / (ms * 1e-3) / 1e9
        pl = gb.attn_decode_plan(w.B, w.Hq, w.Hkv, 1, w.Skv, w.d, w.num_splits, nsm)
        return {"workload": w.name, "ms": ms, "value": gbs, "unit": "GB/s", "frac": gbs / peak_bw,
                "frac_of_nominal_7900": gbs / NOMINAL_HBM_GBS, "bound": "hbm", "peak": peak_bw,
                "kernel": f"decode_split_kernel<{w.d}> ({pl['splits']} splits, {pl['merge']})"}

    configs = {
        "1": prefill_entry(1, extra_ms[1]),
        "2": prefill_entry(2, extra_ms[2]),
        "3": prefill_entry(3, pre_avg),
        "4": decode_entry(DECODE, dl_c.tolist(), dec_avg),
        "5": decode_entry(w5, l5.tolist(), extra_ms[5]),
    }
    line = {
        "metric": METRIC,
        "value": pre_tflops, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": step_ms, "wall_ms_per_step": t_wall / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic", "config": config_dict(args),
        "roofline": {"bound": "tensor", "achieved": per_gpu_tf, "peak": peak_tf,
                     "unit": "TFLOP/s", "frac": per_gpu_tf / peak_tf,
                     "traffic": traffic_pre, "traffic_source": traffic_pre_src,
                     "kernel": f"prefill_fwd_kernel<128> ({pre_plan['mode']})",
                     "ms": pre_avg, "peak_source": f"{peak_src} bf16 burst"},
        "decode": {"value": dec_gbs, "unit": "GB/s", "ms": dec_avg,
                   "roofline": {"bound": "hbm", "achieved": per_gpu_bw, "peak": peak_bw,
                                "unit": "GB/s", "frac": per_gpu_bw / peak_bw,
                                "traffic": traffic_dec, "traffic_source": traffic_dec_src,
                                "kernel": configs["4"]["kernel"] + " + decode_combine_kernel (PDL)",
                                "peak_source": f"{peak_src} HBM copy"}},
        "configs": configs,
        "e2e": {"value": (flops / (e2e_pre * 1e-3) / 1e12 * world) if not args.no_e2e else None,
                "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "decode_gbs": (dbytes / (e2e_dec * 1e-3) / 1e9 * world) if not args.no_e2e else None,
                "ms_per_step": e2e_pre + e2e_dec, "steps": args.steps},
        "gpu_launches": launches * args.steps,
        "chunked_prefill": chunk,
        "multitoken_decode": mtok,
        "sequence_parallel": spar,
        "clocks": clk.summary(),
    }
    if not args.no_cpu_baseline:
        inputs = {3: (q_c, k_c, v_c), 4: (dq_c, dk_c, dv_c, dl_c)}
        inputs.update(extra_in)
        line["cpu_baseline"] = cpu_baseline_and_check(inputs, outputs)
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["gbattn", "reference"], default="gbattn")
    ap.add_argument("--no-cpu-baseline", action="store_true",
                    help="skip the oracle leg (its timing and the check of the outputs)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-chunk", action="store_true",
                    help="skip the chunked-prefill and multi-token measurements")
    args = ap.parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl")
    try:
        run_gpu(args, rank, world, local_rank)
    finally:
        if world > 1:
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
