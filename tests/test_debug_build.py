"""The debug build (-DGBATTN_DEBUG_CHECKS, libgbattn_debug.so): the same entry points, with
every kernel checking the index of each global store against its buffer (a failed check
records word 8 in the device error word and skips the access; nothing traps).

On CPU: the debug library builds and exports every declared entry point.  On the GPU:
ordinary calls of every kernel path run through the debug library in a fresh process,
match the fp64 oracle within the parity bars, and leave the error word clear."""
import ctypes
import os
import subprocess
import sys
import textwrap

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import streaming_attention_flashattention_gb300 as gb  # noqa: E402
from streaming_attention_flashattention_gb300 import build  # noqa: E402


def test_debug_library_exports_every_entry_point():
    path = build.build(debug=True)
    assert path.endswith("libgbattn_debug.so")
    lib = ctypes.CDLL(path)
    for name in gb.EXPORTS:
        assert hasattr(lib, name), name


SCRIPT = textwrap.dedent(r"""
    import sys
    sys.path.insert(0, {root!r}); sys.path.insert(0, {tests!r})
    import numpy as np, torch
    import attn_workloads as wl, oracle
    import streaming_attention_flashattention_gb300 as gb
    from streaming_attention_flashattention_gb300 import build
    from _parity import compare
    gb.load_library(build.build(debug=True))

    def prefill(B, Hq, Hkv, S, d, causal, dtype="bf16", seed=1, Skv=None):
        w = wl.Workload("dbg", "prefill", B=B, Hq=Hq, Hkv=Hkv, d=d, dtype=dtype, Sq=S,
                        Skv=Skv or S, causal=causal, seed=seed)
        q, k, v = wl.prefill_inputs(w)
        o, lse = gb.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=causal, scale=w.scale)
        torch.cuda.synchronize()
        rows = np.random.default_rng(seed).integers(0, B * Hq * S, 300)
        o_ref, l_ref = oracle.attention(wl.to_oracle(q), wl.to_oracle(k), wl.to_oracle(v),
                                        w.scale, causal, rows=rows)
        compare(o.float().cpu().numpy().reshape(-1, d)[rows], lse.cpu().numpy().reshape(-1)[rows],
                o_ref, l_ref, dtype, "prefill")

    def decode(B, Hq, Hkv, L, ns, Tq=1, seed=2):
        w = wl.Workload("dbg-dec", "decode", B=B, Hq=Hq, Hkv=Hkv, d=128, dtype="bf16", Skv=L,
                        num_splits=ns, len_lo=L // 3, len_hi=L, Sq=Tq, seed=seed)
        if Tq == 1:
            q, kc, vc, kl = wl.decode_inputs(w)
            o, lse = gb.attn_decode_splitkv(q.cuda(), kc.cuda(), vc.cuda(), kl.cuda(),
                                            num_splits=ns, scale=w.scale)
        else:
            q, kc, vc, kl = wl.multitoken_inputs(w)
            o, lse = gb.attn_decode_multitoken(q.cuda(), kc.cuda(), vc.cuda(), kl.cuda(),
                                               num_splits=ns, scale=w.scale)
        torch.cuda.synchronize()
        o_ref, l_ref = oracle.attention(wl.to_oracle(q), wl.to_oracle(kc), wl.to_oracle(vc),
                                        w.scale, Tq > 1, kv_len=kl.numpy())
        compare(o.float().cpu().numpy().reshape(o_ref.shape), lse.cpu().numpy().reshape(l_ref.shape),
                o_ref, l_ref, "bf16", "decode")

    prefill(1, 32, 8, 2560, 128, True)            # pairs of Q tiles
    prefill(1, 32, 8, 4096, 128, False, seed=3)   # pairs plus the KV-split tail launch
    prefill(2, 8, 2, 2048, 128, True, seed=4)     # persistent KV-split tiles
    prefill(1, 4, 2, 300, 64, True, seed=5, Skv=700)
    prefill(1, 2, 1, 128, 64, False, dtype="fp32", seed=6)
    decode(4, 64, 8, 32768, 16)                   # pieces, per-group combine
    decode(1, 64, 8, 4096, 0)                     # single launch
    decode(2, 64, 8, 6000, 3, Tq=4)               # tcgen05 multi-token kernel + combine
    decode(1, 32, 8, 4096, 0, Tq=3)               # 12 rows on the warp-level kernel
    # attn_fwd_positions (rows 0..99 filled, the rest from row 100 on) and attn_merge
    g = np.random.default_rng(9)
    bf = lambda *s: torch.from_numpy(g.standard_normal(s).astype(np.float32)).to(torch.bfloat16)
    q, k, v = bf(1, 4, 300, 128), bf(1, 2, 400, 128), bf(1, 2, 400, 128)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    pa = gb.attn_fwd_positions(qd, kd[:, :, :300].contiguous(), vd[:, :, :300].contiguous(), 0, 100)
    pb = gb.attn_fwd_positions(qd, kd[:, :, 300:].contiguous(), vd[:, :, 300:].contiguous(), 0, 400)
    o, lse = gb.attn_merge(pa[0], pa[1], pb[0], pb[1], out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    kk = k[:, :, :300].contiguous(); vv = v[:, :, :300].contiguous()
    o_ref, l_ref = oracle.attention_at_positions(wl.to_oracle(q), wl.to_oracle(kk), wl.to_oracle(vv),
                                                 1 / 128 ** 0.5, 0, 100)
    compare(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, l_ref, "bf16", "positions+merge")
    st, word = gb.attn_last_device_error()
    assert st == 0 and word == 0, f"error word {{word}}"
    print("debug build ok")
""")


@pytest.mark.gpu
def test_debug_build_runs_every_path_with_the_error_word_clear():
    script = SCRIPT.format(root=ROOT, tests=os.path.join(ROOT, "tests"))
    r = subprocess.run([sys.executable, "-c", script], capture_output=True, text=True,
                       timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    assert "debug build ok" in r.stdout


# ---------------------------------------------------------------------------------------
# the debug build's test hook: a wait that runs out inside a real attention kernel
# ---------------------------------------------------------------------------------------

def test_debug_hook_is_in_the_debug_library_only():
    dbg = ctypes.CDLL(build.build(debug=True))
    assert hasattr(dbg, "attn_debug_skip_fill")
    rel = ctypes.CDLL(build.build())
    assert not hasattr(rel, "attn_debug_skip_fill")


def test_debug_header_compiles_as_c99(tmp_path):
    src = tmp_path / "t.c"
    src.write_text('#include "gbattn_debug.h"\nint main(void) { return GBATTN_DEBUG_MULTITOKEN_DECODE - 1; }\n')
    r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-fsyntax-only", "-I",
                        os.path.join(ROOT, "include"), str(src)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


TIMEOUT_SCRIPT = textwrap.dedent(r"""
    import ctypes, sys, time
    sys.path.insert(0, {root!r}); sys.path.insert(0, {tests!r})
    import numpy as np, torch
    import attn_workloads as wl, oracle
    import streaming_attention_flashattention_gb300 as gb
    from streaming_attention_flashattention_gb300 import build
    from _parity import compare
    lib = gb.load_library(build.build(debug=True))
    skip = lib.attn_debug_skip_fill
    skip.argtypes = [ctypes.c_int, ctypes.c_int]
    skip.restype = ctypes.c_int
    PERSISTENT_PREFILL, MULTITOKEN_DECODE, PAIR_PREFILL, SPLIT_DECODE = 0, 1, 2, 3
    NSM = torch.cuda.get_device_properties(0).multi_processor_count
    assert skip(7, 0) == gb.GBATTN_ERR_INVALID_ARG and skip(0, -2) == gb.GBATTN_ERR_INVALID_ARG

    def prefill(Hq=8, Hkv=2, S=1024, mode="kv_split"):
        w = wl.Workload("dbg-to", "prefill", B=1, Hq=Hq, Hkv=Hkv, d=128, dtype="bf16", Sq=S,
                        Skv=S, causal=True, seed=21)
        assert gb.attn_prefill_plan(1, Hq, Hkv, S, S, True, NSM)["mode"] == mode
        q, k, v = wl.prefill_inputs(w)
        o, lse = gb.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=True, scale=w.scale)
        return w, (q, k, v), o, lse

    def pairs():
        return prefill(Hq=32, Hkv=8, S=2560, mode="pairs")

    def split_decode():
        w = wl.Workload("dbg-to-dec", "decode", B=4, Hq=64, Hkv=8, d=128, dtype="bf16", Skv=8192,
                        num_splits=16, len_lo=6000, len_hi=8192, seed=23)
        assert gb.attn_decode_plan(4, 64, 8, 1, 8192, 128, 16, NSM)["merge"] == "combine_per_group"
        q, kc, vc, kl = wl.decode_inputs(w)
        o, lse = gb.attn_decode_splitkv(q.cuda(), kc.cuda(), vc.cuda(), kl.cuda(), num_splits=16,
                                        scale=w.scale)
        return w, (q, kc, vc, kl), o, lse.unsqueeze(-1)

    def decode():
        w = wl.Workload("dbg-to-mt", "decode", B=2, Hq=16, Hkv=2, d=128, dtype="bf16", Skv=3000,
                        num_splits=2, len_lo=2500, len_hi=3000, Sq=4, seed=22)
        assert gb.attn_decode_plan(2, 16, 2, 4, 3000, 128, 2, NSM)["kernel"] == "tcgen05"
        q, kc, vc, kl = wl.multitoken_inputs(w)
        o, lse = gb.attn_decode_multitoken(q.cuda(), kc.cuda(), vc.cuda(), kl.cuda(),
                                           num_splits=2, scale=w.scale)
        return w, (q, kc, vc, kl), o, lse

    for kernel, call in ((PERSISTENT_PREFILL, prefill), (MULTITOKEN_DECODE, decode),
                         (PAIR_PREFILL, pairs), (SPLIT_DECODE, split_decode)):
        # the wait for the unissued K tile runs out; every role of every CTA gives up and the
        # kernel returns: the host sees GBATTN_ERR_TIMEOUT with the code of a wait
        assert skip(kernel, 3) == 0
        t0 = time.time()
        call()
        st, word = gb.attn_last_device_error()
        elapsed = time.time() - t0
        assert st == gb.GBATTN_ERR_TIMEOUT and word in (1, 2, 3, 4, 7), (kernel, st, word)
        assert elapsed < 60, elapsed
        assert gb.attn_last_device_error() == (0, 0)          # read and cleared
        # the context is still usable: the same call without the hook matches the oracle
        assert skip(kernel, -1) == 0
        w, ins, o, lse = call()
        torch.cuda.synchronize()
        if kernel in (PERSISTENT_PREFILL, PAIR_PREFILL):
            q, k, v = ins
            rows = np.random.default_rng(kernel).integers(0, q.shape[1] * q.shape[2], 2000)
            o_ref, l_ref = oracle.attention(wl.to_oracle(q), wl.to_oracle(k), wl.to_oracle(v),
                                            w.scale, True, rows=rows)
            o, lse = o.reshape(-1, 128)[rows], lse.reshape(-1)[rows]
        else:
            q, kc, vc, kl = ins
            o_ref, l_ref = oracle.attention(wl.to_oracle(q), wl.to_oracle(kc), wl.to_oracle(vc),
                                            w.scale, kernel == MULTITOKEN_DECODE, kv_len=kl.numpy())
        compare(o.float().cpu().numpy(), lse.cpu().numpy().reshape(l_ref.shape), o_ref, l_ref,
                "bf16", f"after {{kernel}}")
        assert gb.attn_last_device_error() == (0, 0)
        print(f"kernel {{kernel}}: gave up with word {{word}} after {{elapsed:.2f}} s, then ran clean")
    print("timeouts ok")
""")


@pytest.mark.gpu
def test_wait_runs_out_inside_real_kernels_and_every_role_exits():
    # A K tile copy that is never issued (debug-build hook) makes the wait for it run out
    # inside each attention kernel (pair and persistent prefill, warp-level and tcgen05
    # decode): the producers drain
    # their copies, the MMA issuer drains its products, TMEM is released, the error word
    # carries the wait's code, and the next call on the same context is correct.  No fault,
    # no trap: the copy is simply not started.
    script = TIMEOUT_SCRIPT.format(root=ROOT, tests=os.path.join(ROOT, "tests"))
    r = subprocess.run([sys.executable, "-c", script], capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    assert "timeouts ok" in r.stdout
    print(r.stdout.strip())
