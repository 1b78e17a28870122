"""CUDA graph capture of the library calls.

Every call is a fixed sequence of stream operations (counter clears, kernel launches, the
combine launched as a programmatic dependent), and everything that changes from step to step
(tensor contents, sequence lengths) is read on the device.  So one captured call replays as a
whole decode or prefill step: after new inputs are copied into the captured buffers, a
replay gives exactly what an eager call on those inputs gives.
"""
import pytest
import torch

import streaming_attention_flashattention_gb300 as gb

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from streaming_attention_flashattention_gb300 import build
    build.build()
    gb.load_library()
    yield
    st, word = gb.attn_last_device_error()
    assert st == 0 and word == 0, f"device error word set: {word}"


def _capture(fn) -> torch.cuda.CUDAGraph:
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn()                                   # first-call set-up happens outside the capture
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


def _randn(shape, seed, dtype=torch.bfloat16):
    gen = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=gen).to(dtype).cuda()


@pytest.mark.parametrize("causal", [True, False])
def test_graph_prefill_replays_with_new_inputs(causal):
    B, Hq, Hkv, S, d = 1, 8, 2, 1100, 128
    q, k, v = _randn((B, Hq, S, d), 1), _randn((B, Hkv, S, d), 2), _randn((B, Hkv, S, d), 3)
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, S), dtype=torch.float32, device="cuda")
    g = _capture(lambda: gb.attn_fwd(q, k, v, causal=causal, out=o, lse=lse))
    q2, k2, v2 = _randn(q.shape, 11), _randn(k.shape, 12), _randn(v.shape, 13)
    q.copy_(q2); k.copy_(k2); v.copy_(v2)
    g.replay()
    o_ref, lse_ref = gb.attn_fwd(q2, k2, v2, causal=causal)
    torch.cuda.synchronize()
    assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)


@pytest.mark.parametrize("B,Hq,Hkv,Lmax,ns,lens0,lens1", [
    (4, 64, 8, 9000, 16, [9000, 5000, 1, 4097], [2500, 9000, 0, 64]),   # work queue + combine
    (1, 8, 1, 4096, 8, [4096], [1500]),                               # single launch (one wave)
    (1, 64, 8, 131072, 0, [131072], [90001]),                         # single launch, 2 CTAs per SM
])
def test_graph_decode_replays_as_the_cache_grows(B, Hq, Hkv, Lmax, ns, lens0, lens1):
    d = 128
    q = _randn((B, Hq, 1, d), 4)
    kc, vc = _randn((B, Hkv, Lmax, d), 5), _randn((B, Hkv, Lmax, d), 6)
    lens = torch.tensor(lens0, dtype=torch.int32, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq), dtype=torch.float32, device="cuda")
    ws = torch.empty(gb.attn_decode_workspace_size(B, Hq, Hkv, Lmax, d, ns), dtype=torch.uint8,
                     device="cuda")
    g = _capture(lambda: gb.attn_decode_splitkv(q, kc, vc, lens, num_splits=ns, out=o, lse=lse,
                                                workspace=ws))
    # the next step: a new query and other lengths, through the same graph
    q2 = _randn(q.shape, 14)
    q.copy_(q2)
    lens.copy_(torch.tensor(lens1, dtype=torch.int32))
    g.replay()
    o_ref, lse_ref = gb.attn_decode_splitkv(q2, kc, vc, lens.clone(), num_splits=ns)
    torch.cuda.synchronize()
    assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)


@pytest.mark.parametrize("Tq,Hq,Hkv", [(4, 64, 8), (2, 8, 8)])      # tcgen05 path, warp path
def test_graph_multitoken_decode_replays(Tq, Hq, Hkv):
    B, Lmax, d, ns = 3, 6000, 128, 8
    q = _randn((B, Hq, Tq, d), 7)
    kc, vc = _randn((B, Hkv, Lmax, d), 8), _randn((B, Hkv, Lmax, d), 9)
    lens = torch.tensor([6000, 3001, 130], dtype=torch.int32, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, Tq), dtype=torch.float32, device="cuda")
    need = gb.load_library().attn_decode_multitoken_workspace_size(B, Hq, Hkv, Tq, Lmax, d, ns)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    g = _capture(lambda: gb.attn_decode_multitoken(q, kc, vc, lens, num_splits=ns, out=o,
                                                   lse=lse, workspace=ws))
    q2 = _randn(q.shape, 15)
    q.copy_(q2)
    lens.copy_(torch.tensor([4100, 6000, 2], dtype=torch.int32))
    for _ in range(3):                       # the work queue counter is cleared by every replay
        g.replay()
    o_ref, lse_ref = gb.attn_decode_multitoken(q2, kc, vc, lens.clone(), num_splits=ns)
    torch.cuda.synchronize()
    assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)
