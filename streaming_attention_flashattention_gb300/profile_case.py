"""Run one workload a few times through the public API, for profiler captures.

A capture wants a small, fixed launch sequence: this module builds the library if needed,
generates one seeded workload (the same generators the tests and the benchmark use), and
calls the library `--reps` times with nothing else on the GPU.  Examples:

    python -m streaming_attention_flashattention_gb300.profile_case prefill --workload 3
    python -m streaming_attention_flashattention_gb300.profile_case decode --workload 4
    python -m streaming_attention_flashattention_gb300.profile_case multitoken --keys 16384 --splits 4
    python -m streaming_attention_flashattention_gb300.profile_case ringstep

`ringstep` is one rank's step of an 8-rank ring-KV prefill of the Llama3-70B shape (8 query
heads x 8192 positions against KV slice 3 of 8, attn_fwd_positions) followed by the merge of
its result into an fp32 accumulator (attn_merge), each call `--reps` times.

`--keys` / `--splits` shrink a decode or multi-token workload (cache length and split count)
so that a full-metric capture stays small.
"""
from __future__ import annotations

import argparse

import torch

import attn_workloads as wl
import streaming_attention_flashattention_gb300 as gb
from streaming_attention_flashattention_gb300 import build


def ring_step(reps: int) -> None:
    w = wl.WORKLOADS[3]
    S, L = w.Sq, w.Skv // 8
    g = torch.Generator().manual_seed(97)
    q = torch.randn((1, 8, S, w.d), generator=g).to(torch.bfloat16).cuda()
    k = torch.randn((1, 1, L, w.d), generator=g).to(torch.bfloat16).cuda()
    v = torch.randn((1, 1, L, w.d), generator=g).to(torch.bfloat16).cuda()
    o = torch.empty_like(q)
    lse = torch.empty((1, 8, S), dtype=torch.float32, device="cuda")
    acc_o = torch.zeros((1, 8, S, w.d), dtype=torch.float32, device="cuda")
    acc_l = torch.full((1, 8, S), float("-inf"), device="cuda")
    for _ in range(reps):
        gb.attn_fwd_positions(q, k, v, 0, 3 * L, scale=w.scale, out=o, lse=lse)
        gb.attn_merge(acc_o, acc_l, o, lse, out=acc_o, lse_out=acc_l)
    torch.cuda.synchronize()
    st, word = gb.attn_last_device_error()
    if st != 0 or not torch.isfinite(acc_o).all():
        raise SystemExit(f"ring step failed: status {st}, word {word}")
    print(f"ok ringstep reps={reps}")


def main() -> None:
    ap = argparse.ArgumentParser()
    ap.add_argument("case", choices=["prefill", "decode", "chunk", "multitoken", "ringstep"])
    ap.add_argument("--workload", type=int, default=None, help="workload index (default per case)")
    ap.add_argument("--keys", type=int, default=0, help="decode / multi-token: cache length override")
    ap.add_argument("--splits", type=int, default=-1, help="decode / multi-token: split count override")
    ap.add_argument("--reps", type=int, default=4)
    args = ap.parse_args()
    build.build()
    gb.load_library()
    if args.case == "ringstep":
        ring_step(args.reps)
        return
    default = {"prefill": 3, "decode": 4, "chunk": 6, "multitoken": 7}[args.case]
    idx = args.workload if args.workload is not None else default
    w = wl.WORKLOADS.get(idx) or wl.EXTRA_WORKLOADS[idx]
    if args.keys > 0:
        w = w.replace(Skv=args.keys, len_lo=min(w.len_lo, args.keys), len_hi=args.keys)
    if args.splits >= 0:
        w = w.replace(num_splits=args.splits)

    if args.case == "prefill":
        q, k, v = (t.cuda() for t in wl.prefill_inputs(w))
        run = lambda: gb.attn_fwd(q, k, v, causal=w.causal, scale=w.scale)
    elif args.case == "chunk":
        q, kc, vc, ctx = wl.chunk_inputs(w)
        q, kc, vc = q.cuda(), kc.cuda(), vc.cuda()
        run = lambda: gb.attn_prefill_kvcache(q, kc, vc, ctx, causal=w.causal, scale=w.scale)
    elif args.case == "decode":
        q, kc, vc, lens = (t.cuda() for t in wl.decode_inputs(w))
        run = lambda: gb.attn_decode_splitkv(q, kc, vc, lens, num_splits=w.num_splits, scale=w.scale)
    else:
        q, kc, vc, lens = (t.cuda() for t in wl.multitoken_inputs(w))
        run = lambda: gb.attn_decode_multitoken(q, kc, vc, lens, num_splits=w.num_splits,
                                                scale=w.scale)
    for _ in range(args.reps):
        out = run()
    torch.cuda.synchronize()
    o = out[0] if isinstance(out, tuple) else out
    print(f"{args.case} {w.name}: {args.reps} calls, mean |O| {float(o.float().abs().mean()):.6f}")


if __name__ == "__main__":
    main()
