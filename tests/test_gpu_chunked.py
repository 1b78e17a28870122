"""GPU parity of attn_prefill_kvcache (chunked prefill against a KV cache) with the fp64
oracle; cache rows past the context hold NaN, so reading any of them fails the test."""
import numpy as np
import pytest
import torch

import attn_workloads as wl
import oracle
import streaming_attention_flashattention_gb300 as gb
from _parity import compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from streaming_attention_flashattention_gb300 import build
    build.build()
    gb.load_library()
    yield
    st, word = gb.attn_last_device_error()
    assert st == 0 and word == 0, f"device error word set: {word}"


def run(w: wl.Workload, rows=None):
    q, kc, vc, ctx = wl.chunk_inputs(w)
    o, lse = gb.attn_prefill_kvcache(q.cuda(), kc.cuda(), vc.cuda(), ctx, causal=w.causal,
                                     scale=w.scale)
    torch.cuda.synchronize()
    o = o.float().cpu().numpy()
    lse = lse.cpu().numpy()
    kl = np.full(w.B, ctx, np.int32)
    if rows is None:
        o_ref, lse_ref = oracle.attention(wl.to_oracle(q), wl.to_oracle(kc), wl.to_oracle(vc),
                                          w.scale, w.causal, kv_len=kl)
        return compare(o, lse, o_ref, lse_ref, w.dtype, w.name)
    o_ref, lse_ref = oracle.attention(wl.to_oracle(q), wl.to_oracle(kc), wl.to_oracle(vc),
                                      w.scale, w.causal, kv_len=kl, rows=rows)
    return compare(o.reshape(-1, w.d)[rows], lse.reshape(-1)[rows], o_ref, lse_ref, w.dtype, w.name)


def chunk(B, Hq, Hkv, Sq, ctx, Lmax, d, causal, seed=3):
    return wl.Workload(f"chunk-b{B}-h{Hq}/{Hkv}-q{Sq}-ctx{ctx}-cap{Lmax}-d{d}", "chunk", B=B, Hq=Hq,
                       Hkv=Hkv, d=d, dtype="bf16", Sq=Sq, Skv=Lmax, causal=causal,
                       len_lo=ctx, len_hi=ctx, seed=seed)


@pytest.mark.parametrize("B,Hq,Hkv,Sq,ctx,Lmax,d,causal", [
    (1, 8, 2, 128, 1000, 1536, 128, True),     # chunk at the end of a ragged context
    (2, 4, 4, 200, 700, 700, 128, True),       # cache exactly full
    (1, 16, 2, 64, 4096, 8192, 128, True),     # short chunk, long context
    (1, 4, 1, 300, 513, 1024, 64, False),      # non-causal, d = 64
    (1, 8, 8, 1, 777, 1024, 128, True),        # one-token chunk (decode-like)
])
def test_chunked_prefill_shapes(B, Hq, Hkv, Sq, ctx, Lmax, d, causal):
    run(chunk(B, Hq, Hkv, Sq, ctx, Lmax, d, causal))


def test_chunked_prefill_matches_attn_fwd_on_the_trimmed_cache():
    w = chunk(1, 8, 2, 256, 1280, 2048, 128, True, seed=9)
    q, kc, vc, ctx = wl.chunk_inputs(w)
    o1, l1 = gb.attn_prefill_kvcache(q.cuda(), kc.cuda(), vc.cuda(), ctx)
    o2, l2 = gb.attn_fwd(q.cuda(), kc[:, :, :ctx].contiguous().cuda(),
                         vc[:, :, :ctx].contiguous().cuda(), causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.slow
def test_workload6_llama70b_chunk_sampled():
    w = wl.EXTRA_WORKLOADS[6]
    rng = np.random.default_rng(6)
    rows = np.unique(np.concatenate([rng.integers(0, w.B * w.Hq * w.Sq, 600),
                                     np.arange(0, 130), [w.B * w.Hq * w.Sq - 1]]))
    run(w, rows=rows)
