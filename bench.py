"""Benchmark of the streaming-attention hot path on GB300.

One step = one causal GQA prefill of the Llama3-70B-shaped workload (B1 Hq64 Hkv8
S8192 d128, bf16, Q x2) plus one split-KV decode of the Llama3-70B decode workload
(B4 Hq64 Hkv8, 32768 cached keys, 16 splits), both through the C ABI (libgbattn.so).

Printed JSON line (rank 0):
  value      prefill TFLOP/s, FLOPs = 4 B Hq Sq Skv d / 2 (causal), inputs resident in HBM
  decode     the decode half: KV GB/s (algorithmic bytes: K, V, Q, O, LSE) with its roofline
  roofline   prefill kernel: achieved TFLOP/s vs the measured dense bf16 peak
  e2e        the same metric through attn_fwd_host: pinned-host inputs copied in and
             outputs copied out by the call (chunked, overlapped with the kernel)
             inside the timed region, every step
  cpu_baseline  the fp64 CPU oracle on a bounded sample of the same workload
L2 is flushed (a 512 MiB write, then a read of it so no dirty lines remain) before the
prefill and again before the decode of every step, outside the kernels' event windows.

--impl reference times the fp64 CPU oracle instead (a bounded row sample per step).
Multi-GPU (torchrun, N > 1): N independent replicas, weak scaling, no collective on the
data path; the step time is the max over ranks.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np
import torch

import attn_workloads as wl

PREFILL = wl.WORKLOADS[3]
DECODE = wl.WORKLOADS[4]
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 512 << 20
# DRAM bytes per launch from the committed ncu captures (profiles/); None when the kernel
# changed after the capture.
NCU_TRAFFIC = {"prefill": 275_330_304, "decode": 541_500_672}


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
    oracle.attention(q_np, k_np, v_np, w.scale, w.causal, rows=rows)
    return flops, time.perf_counter() - t0


def cpu_baseline_prefill(q, k, v, w: wl.Workload, target_s: float = 12.0):
    import oracle
    q_np, k_np, v_np = wl.to_oracle(q), wl.to_oracle(k), wl.to_oracle(v)
    n = 256
    flops, dt = oracle_sample_prefill(q_np, k_np, v_np, w, n, 1)
    n2 = int(min(200000, max(n, n * target_s / max(dt, 1e-3))))
    flops, dt = oracle_sample_prefill(q_np, k_np, v_np, w, n2, 2)
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": oracle.max_threads(),
            "kind": "oracle",
            "sample": f"{n2} random query rows of {w.name} (fp64 two-pass definition, "
                      f"{dt:.1f} s, {flops / 1e9:.1f} GFLOP algorithmic)"}


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
        f, t = oracle_sample_prefill(q_np, k_np, v_np, PREFILL, rows_per_step, 1000 + s)
        tot_f += f
        tot_t += t
    val = tot_f / tot_t / 1e12
    line = {
        "impl": "reference", "metric": "prefill attn TFLOP/s & decode KV GB/s at 1 GB300, % of roofline",
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
            "parallelism": f"replicas{args.gpus}", "l2": "flushed before each of the two calls of every step (512 MiB write, then read back)"}


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

    class _Flush:
        """Evict L2: write a buffer 4x its size, then read it back so that no dirty
        lines are left for the next timed kernel to write back."""

        def zero_(self):
            flush_buf.zero_()
            flush_buf.sum()

    flush = _Flush()
    stream = torch.cuda.current_stream(dev)

    def step(evs=None):
        flush.zero_()
        if evs is not None:
            evs[0].record(stream)
        gb.attn_fwd(q, k, v, causal=PREFILL.causal, scale=PREFILL.scale, out=o, lse=lse)
        if evs is not None:
            evs[1].record(stream)
        # flush again: the prefill's dirty output lines would otherwise be written back
        # inside the decode window
        flush.zero_()
        if evs is not None:
            evs[2].record(stream)
        gb.attn_decode_splitkv(dq, dk, dv, dl, num_splits=DECODE.num_splits,
                               scale=DECODE.scale, out=do, lse=dlse, workspace=ws)
        if evs is not None:
            evs[3].record(stream)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    st, word = gb.attn_last_device_error()
    if st != 0:
        raise RuntimeError(f"device error word {word} during warm-up")

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
    pre_ms = [e[0].elapsed_time(e[1]) for e in evs]
    dec_ms = [e[2].elapsed_time(e[3]) for e in evs]
    pre_avg = sum(pre_ms) / len(pre_ms)
    dec_avg = sum(dec_ms) / len(dec_ms)
    step_ms = pre_avg + dec_avg
    pre_avg, dec_avg, step_ms = max_over_ranks([pre_avg, dec_avg, step_ms], dev)

    # chunked prefill against a KV cache (a widening beyond the step's two calls)
    chunk = None
    if not args.no_chunk:
        wc = wl.EXTRA_WORKLOADS[6]
        cq, ckc, cvc, cctx = (x.to(dev) if torch.is_tensor(x) else x for x in wl.chunk_inputs(wc))
        co = torch.empty_like(cq)
        clse = torch.empty(cq.shape[:3], dtype=torch.float32, device=dev)
        for _ in range(3):
            gb.attn_prefill_kvcache(cq, ckc, cvc, cctx, causal=wc.causal, scale=wc.scale, out=co, lse=clse)
        cms = []
        for _ in range(10):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            gb.attn_prefill_kvcache(cq, ckc, cvc, cctx, causal=wc.causal, scale=wc.scale, out=co, lse=clse)
            e1.record(stream)
            torch.cuda.synchronize(dev)
            cms.append(e0.elapsed_time(e1))
        cm = max_over_ranks([sum(cms) / len(cms)], dev)[0]
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
        for _ in range(3):
            gb.attn_decode_multitoken(mq, mkc, mvc, mkl, num_splits=wm.num_splits, scale=wm.scale,
                                      out=mo, lse=mlse, workspace=mws)
        mms = []
        for _ in range(10):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            gb.attn_decode_multitoken(mq, mkc, mvc, mkl, num_splits=wm.num_splits, scale=wm.scale,
                                      out=mo, lse=mlse, workspace=mws)
            e1.record(stream)
            torch.cuda.synchronize(dev)
            mms.append(e0.elapsed_time(e1))
        mm = max_over_ranks([sum(mms) / len(mms)], dev)[0]
        mbytes = float(mkl_c.sum()) * wm.Hkv * wm.d * 2 * 2 + 2.0 * wm.B * wm.Hq * wm.Sq * wm.d * 2
        mtok = {"workload": wm.name, "ms": mm, "value": mbytes / (mm * 1e-3) / 1e9, "unit": "GB/s"}
        del mq, mkc, mvc, mkl, mo, mlse, mws

    st, word = gb.attn_last_device_error()
    if st != 0:
        raise RuntimeError(f"device error word {word} during the timed steps")

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
        h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv, hdq, hdk, hdv, hdl))
        d2h = sum(t.numel() * t.element_size() for t in (ho, hlse, hdo, hdlse))

        def e2e_step(ev=None):
            flush.zero_()
            if ev is not None:
                ev[0].record(stream)
            # the C-ABI call on host buffers: inputs copied in, outputs copied back, the
            # copies of neighbouring chunks overlapped with the kernel
            gb.attn_fwd_host(hq, hk, hv, causal=PREFILL.causal, scale=PREFILL.scale, out=ho,
                             lse=hlse, workspace=hws)
            if ev is not None:
                ev[1].record(stream)
            dq.copy_(hdq, non_blocking=True); dk.copy_(hdk, non_blocking=True)
            dv.copy_(hdv, non_blocking=True); dl.copy_(hdl, non_blocking=True)
            gb.attn_decode_splitkv(dq, dk, dv, dl, num_splits=DECODE.num_splits,
                                   scale=DECODE.scale, out=do, lse=dlse, workspace=ws)
            hdo.copy_(do, non_blocking=True); hdlse.copy_(dlse, non_blocking=True)
            if ev is not None:
                ev[2].record(stream)

        e2e_step()
        torch.cuda.synchronize(dev)
        n_e2e = max(1, min(args.steps, 5))
        evs2 = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n_e2e)]
        for s in range(n_e2e):
            e2e_step(evs2[s])
        torch.cuda.synchronize(dev)
        e2e_pre = sum(e[0].elapsed_time(e[1]) for e in evs2) / n_e2e
        e2e_dec = sum(e[1].elapsed_time(e[2]) for e in evs2) / n_e2e
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
    per_gpu_tf = flops / (pre_avg * 1e-3) / 1e12
    per_gpu_bw = dbytes / (dec_avg * 1e-3) / 1e9
    if chunk is not None:
        chunk["frac"] = chunk["value"] / peak_tf      # per GPU
    if mtok is not None:
        mtok["frac"] = mtok["value"] / peak_bw         # per GPU
    line = {
        "metric": "prefill attn TFLOP/s & decode KV GB/s at 1 GB300, % of roofline",
        "value": pre_tflops, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": step_ms, "wall_ms_per_step": t_wall / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic", "config": config_dict(args),
        "roofline": {"bound": "tensor", "achieved": per_gpu_tf, "peak": peak_tf,
                     "unit": "TFLOP/s", "frac": per_gpu_tf / peak_tf,
                     "traffic": NCU_TRAFFIC["prefill"], "kernel": "prefill_fwd_kernel<128, 0, 0> (pairs)",
                     "ms": pre_avg, "peak_source": f"{peak_src} bf16 burst"},
        "decode": {"value": dec_gbs, "unit": "GB/s", "ms": dec_avg,
                   "roofline": {"bound": "hbm", "achieved": per_gpu_bw, "peak": peak_bw,
                                "unit": "GB/s", "frac": per_gpu_bw / peak_bw,
                                "traffic": NCU_TRAFFIC["decode"],
                                "kernel": "decode_split_kernel<128> + decode_combine_kernel<128> (PDL)",
                                "peak_source": f"{peak_src} HBM copy"}},
        "e2e": {"value": (flops / (e2e_pre * 1e-3) / 1e12 * world) if not args.no_e2e else None,
                "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "decode_gbs": (dbytes / (e2e_dec * 1e-3) / 1e9 * world) if not args.no_e2e else None,
                "ms_per_step": e2e_pre + e2e_dec},
        "gpu_launches": 3 * args.steps,
        "chunked_prefill": chunk,
        "multitoken_decode": mtok,
        "clocks": clk.summary(),
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_prefill(q_c, k_c, v_c, PREFILL)
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["gbattn", "reference"], default="gbattn")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-chunk", action="store_true", help="skip the chunked-prefill measurement")
    ap.add_argument("--prefill", type=int, default=3, help="prefill workload index (1-3)")
    ap.add_argument("--decode", type=int, default=4, help="decode workload index (4-5)")
    args = ap.parse_args()
    global PREFILL, DECODE
    PREFILL = wl.WORKLOADS[args.prefill]
    DECODE = wl.WORKLOADS[args.decode]
    if PREFILL.kind != "prefill" or DECODE.kind != "decode":
        ap.error("--prefill takes a prefill workload, --decode a decode workload")
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
