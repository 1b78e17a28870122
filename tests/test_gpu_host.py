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
    # 8 (b, KV head) groups of 64 Q-tile pairs: chunks of 5 groups, the last one partial
    w = _w(1, 64, 8, 2048, 128, True)
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
