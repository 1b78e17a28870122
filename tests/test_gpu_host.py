"""GPU parity of attn_fwd_host (host buffers in and out, chunked copies overlapped with the
kernel) with the fp64 oracle and with the device-buffer attn_fwd."""
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


def _w(B, Hq, Hkv, S, d, causal, dtype="bf16", seed=41):
    return wl.Workload(f"host-b{B}-h{Hq}/{Hkv}-s{S}-d{d}-{dtype}", "prefill", B=B, Hq=Hq, Hkv=Hkv,
                       d=d, dtype=dtype, Sq=S, Skv=S, causal=causal, seed=seed)


def test_host_pipeline_matches_oracle_several_chunks():
    # 16 (b, KV head) groups of 64 Q-tile pairs: chunks of 3 groups (one pair per SM), the
    # last of 1, so 6 chunks go through the 3 staging sets and every set is reused
    w = _w(2, 64, 8, 2048, 128, True)
    q, k, v = wl.prefill_inputs(w)
    o, lse = gb.attn_fwd_host(q.pin_memory(), k.pin_memory(), v.pin_memory(), causal=True)
    torch.cuda.synchronize()
    rng = np.random.default_rng(5)
    rows = np.unique(rng.integers(0, w.B * w.Hq * w.Sq, 3000))
    o_ref, lse_ref = oracle.attention(wl.to_oracle(q), wl.to_oracle(k), wl.to_oracle(v), w.scale,
                                      True, rows=rows)
    compare(o.float().numpy().reshape(-1, w.d)[rows], lse.numpy().reshape(-1)[rows], o_ref, lse_ref,
            "bf16", w.name)


def test_host_pipeline_agrees_with_device_call():
    w = _w(2, 16, 4, 1536, 128, False, seed=43)
    q, k, v = wl.prefill_inputs(w)
    o_h, l_h = gb.attn_fwd_host(q.pin_memory(), k.pin_memory(), v.pin_memory(), causal=False)
    o_d, l_d = gb.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=False)
    torch.cuda.synchronize()
    assert (o_h.float() - o_d.float().cpu()).abs().max().item() <= 2e-2
    assert (l_h - l_d.cpu()).abs().max().item() <= 1e-3


def test_host_pipeline_fp32_and_pageable_buffers():
    w = _w(1, 4, 2, 300, 64, True, dtype="fp32", seed=47)
    q, k, v = wl.prefill_inputs(w)           # pageable host memory: copies wait on the host
    o, lse = gb.attn_fwd_host(q, k, v, causal=True)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.attention(wl.to_oracle(q), wl.to_oracle(k), wl.to_oracle(v), w.scale, True)
    compare(o.numpy(), lse.numpy(), o_ref, lse_ref, "fp32", w.name)


def test_host_pipeline_rejects_small_workspace():
    w = _w(1, 8, 2, 256, 128, True)
    q, k, v = wl.prefill_inputs(w)
    ws = torch.empty(64, dtype=torch.uint8, device="cuda")
    with pytest.raises(gb.GbAttnError):
        gb.attn_fwd_host(q, k, v, causal=True, workspace=ws)


@pytest.mark.parametrize("B,Hq,Hkv,L,ns", [(4, 64, 8, 32768, 16),   # workload 4's shape: 4 chunks
                                           (7, 32, 8, 5000, 0),     # chunks of 2, the last of 1
                                           (1, 8, 1, 300, 0)])      # one chunk, one buffer set
def test_decode_host_matches_oracle_and_device_call(B, Hq, Hkv, L, ns):
    w = wl.Workload(f"dhost-b{B}-h{Hq}/{Hkv}-l{L}", "decode", B=B, Hq=Hq, Hkv=Hkv, d=128,
                    dtype="bf16", Skv=L, num_splits=ns, len_lo=L // 4, len_hi=L, Sq=1, seed=61)
    q, kc, vc, kl = wl.decode_inputs(w)
    o, lse = gb.attn_decode_host(q.pin_memory(), kc.pin_memory(), vc.pin_memory(),
                                 kl.pin_memory(), num_splits=ns, scale=w.scale)
    torch.cuda.synchronize()
    assert not o.is_cuda and not lse.is_cuda
    o_ref, l_ref = oracle.attention(wl.to_oracle(q), wl.to_oracle(kc), wl.to_oracle(vc), w.scale,
                                    False, kv_len=kl.numpy())
    compare(o.float().numpy(), lse.numpy(), o_ref, l_ref[..., 0] if l_ref.ndim == 3 else l_ref,
            "bf16", w.name)
    # one chunk holds all sequences: the same kernels and split decisions as the device call
    if B == 1:
        od, ld = gb.attn_decode_splitkv(q.cuda(), kc.cuda(), vc.cuda(), kl.cuda(),
                                        num_splits=ns, scale=w.scale)
        torch.cuda.synchronize()
        assert torch.equal(od.cpu(), o) and torch.equal(ld.cpu(), lse)


def test_decode_host_rejects_a_length_beyond_the_cache():
    q = torch.zeros((2, 8, 1, 128), dtype=torch.bfloat16)
    kc = torch.zeros((2, 1, 256, 128), dtype=torch.bfloat16)
    with pytest.raises(gb.GbAttnError):
        gb.attn_decode_host(q, kc, kc, torch.tensor([10, 300], dtype=torch.int32))
