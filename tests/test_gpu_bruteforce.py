"""Brute-force parity sweep of attn_fwd over tiny and tile-edge shapes, against the fp64 oracle.

Every combination of Sq, Skv in {1, 2, 3, 5, 17, 127, 128, 129, 255}, d in {64, 128},
G = Hq / Hkv in {1, 2, 8}, causal on and off (causal needs Sq <= Skv: bottom-right
alignment) runs through the C ABI on the bf16 tensor-core path and is compared element by
element with the plain two-pass definition ("ADR-0060: AHBM GQA Fused Attention Kernel
(Llama3-70B)", section 11: numeric parity of the fused kernel against an unfused reference
on small shapes).  The sizes straddle the 128-row Q tile and 128-key K/V tile edges, so
single-tile, exact-tile, one-past-a-tile and two-tile cases all occur on both sides of the
causal diagonal.  A subset of the same grid runs on the fp32 path at its 1e-4 bar.

Each parametrised test loops over its grid internally (one GPU context, one library
load); a failure names the exact case.
"""
import itertools

import pytest
import torch

import attn_workloads as wl
import oracle
import streaming_attention_flashattention_gb300 as gb
from _parity import compare

pytestmark = pytest.mark.gpu

SIZES = [1, 2, 3, 5, 17, 127, 128, 129, 255]
FP32_SIZES = [1, 5, 128, 129]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from streaming_attention_flashattention_gb300 import build
    build.build()
    gb.load_library()
    yield
    st, word = gb.attn_last_device_error()
    assert st == 0 and word == 0, f"device error word set: {word}"


def _cases(sizes):
    for Sq, Skv in itertools.product(sizes, sizes):
        for causal in (False, True):
            if causal and Sq > Skv:
                continue
            yield Sq, Skv, causal


def _run(Sq, Skv, d, G, causal, dtype, seed):
    # two KV heads, so that the GQA head map (kv = h / G) is exercised across a boundary
    w = wl.Workload(f"bf-s{Sq}x{Skv}-d{d}-g{G}-{'c' if causal else 'nc'}-{dtype}", "prefill",
                    B=1, Hq=2 * G, Hkv=2, d=d, dtype=dtype, Sq=Sq, Skv=Skv, causal=causal,
                    seed=seed)
    q, k, v = wl.prefill_inputs(w)
    o, lse = gb.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=causal, scale=w.scale)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.attention(wl.to_oracle(q), wl.to_oracle(k), wl.to_oracle(v),
                                      w.scale, causal)
    compare(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, dtype, w.name)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("G", [1, 2, 8])
def test_bruteforce_bf16(d, G):
    n = 0
    for i, (Sq, Skv, causal) in enumerate(_cases(SIZES)):
        _run(Sq, Skv, d, G, causal, "bf16", seed=5000 + 131 * i + 7 * G + d)
        n += 1
    assert n == 81 + 45


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("G", [1, 8])
def test_bruteforce_fp32(d, G):
    for i, (Sq, Skv, causal) in enumerate(_cases(FP32_SIZES)):
        _run(Sq, Skv, d, G, causal, "fp32", seed=6000 + 131 * i + 7 * G + d)
