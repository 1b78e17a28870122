"""attn_decode_splitkv_noalloc: the decode entry point for callers that cannot allocate
device memory (no workspace argument; the library's fixed 8 MiB scratch is used).

It is checked through the C ABI against the regular entry point, on two calls in a row
(the second call finds the scratch holding the first call's leftovers), within the
parity tolerances of the other decode tests.  This file is collected last so that a
stop-at-first-failure run has already run every other test; it also passes on its own
in a fresh process.
"""
import numpy as np
import pytest
import torch

import attn_workloads as wl
import streaming_attention_flashattention_gb300 as gb
from _parity import BF16_MAX_ABS, BF16_MEAN_ABS, LSE_MAX_ABS


@pytest.fixture(scope="module")
def lib():
    from streaming_attention_flashattention_gb300 import build
    build.build()
    return gb.load_library()


def test_noalloc_is_declared_and_exported(lib):
    assert hasattr(lib, "attn_decode_splitkv_noalloc")


def test_noalloc_rejects_invalid_arguments(lib):
    # invalid arguments get the same codes as the regular entry point, before any device
    # access
    assert lib.attn_decode_splitkv_noalloc(None, 0x10000, 0x10000, 0x10000, 0x20000, None,
                                           4, 64, 8, 4096, 128, 0.088, 16, None) == -1
    assert lib.attn_decode_splitkv_noalloc(0x10000, 0x10000, 0x10000, 0x10000, 0x20000, None,
                                           4, 64, 8, 4096, 96, 0.088, 16, None) == -2


def _close(a, b):
    a = a.float().cpu().numpy().astype(np.float64)
    b = b.float().cpu().numpy().astype(np.float64)
    err = np.abs(a - b)
    return err.max() <= BF16_MAX_ABS and err.mean() <= BF16_MEAN_ABS


@pytest.mark.gpu
def test_noalloc_rejects_requests_beyond_its_scratch(lib):
    # 16 sequences x 64 heads x 32 automatic splits of a 131072-key cache need ~17 MiB
    need = gb.attn_decode_workspace_size(16, 64, 8, 131072, 128, 0)
    assert need > gb.NOALLOC_SCRATCH_BYTES
    st = lib.attn_decode_splitkv_noalloc(0x10000, 0x10000, 0x10000, 0x10000, 0x20000, None,
                                         16, 64, 8, 131072, 128, 0.088, 0, None)
    assert st == -6


@pytest.mark.gpu
@pytest.mark.parametrize("widx,num_splits", [(4, 16), (4, 0)])
def test_noalloc_matches_regular_entry_point_twice(lib, widx, num_splits):
    w = wl.WORKLOADS[widx]
    q, kc, vc, kl = (t.cuda() for t in wl.decode_inputs(w))
    ref_o, ref_lse = gb.attn_decode_splitkv(q, kc, vc, kl, num_splits=num_splits, scale=w.scale)
    for call in range(2):
        o = torch.full_like(ref_o, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        gb.attn_decode_splitkv_noalloc(q, kc, vc, kl, o, lse, num_splits=num_splits,
                                       scale=w.scale)
        torch.cuda.synchronize()
        assert _close(o, ref_o), f"call {call}: O differs from attn_decode_splitkv"
        assert torch.isfinite(lse).all()
        assert (lse - ref_lse).abs().max().item() <= LSE_MAX_ABS, f"call {call}: LSE differs"
    st, word = gb.attn_last_device_error()
    assert st == 0, f"device error word {word}"


@pytest.mark.gpu
def test_noalloc_second_call_with_other_shape(lib):
    # a different, smaller problem right after: leftovers of the previous call must not leak
    w = wl.Workload("noalloc-small", "decode", B=3, Hq=16, Hkv=2, d=128, dtype="bf16",
                    Skv=5000, num_splits=0, len_lo=100, len_hi=5000, seed=77)
    q, kc, vc, kl = (t.cuda() for t in wl.decode_inputs(w))
    ref_o, ref_lse = gb.attn_decode_splitkv(q, kc, vc, kl, num_splits=3, scale=w.scale)
    for call in range(2):
        o = torch.empty_like(ref_o)
        lse = torch.empty_like(ref_lse)
        gb.attn_decode_splitkv_noalloc(q, kc, vc, kl, o, lse, num_splits=3, scale=w.scale)
        torch.cuda.synchronize()
        assert _close(o, ref_o) and (lse - ref_lse).abs().max().item() <= LSE_MAX_ABS


@pytest.mark.gpu
def test_noalloc_eager_first_call_then_graph_replay(lib):
    # The first call on the device looks up the scratch address (outside any capture);
    # a later call captured in a CUDA graph then replays correctly.  B1 with 4096 keys is
    # a one-wave shape, so the single-launch merge (the group counters in the scratch)
    # runs; each replay must clear those counters again.
    w = wl.Workload("noalloc-graph", "decode", B=1, Hq=64, Hkv=8, d=128, dtype="bf16",
                    Skv=4096, num_splits=0, len_lo=4096, len_hi=4096, seed=78)
    plan = gb.attn_decode_plan(1, 64, 8, 1, 4096, 128, 0, torch.cuda.get_device_properties(0).multi_processor_count)
    assert plan["merge"] == "single_launch"
    q, kc, vc, kl = (t.cuda() for t in wl.decode_inputs(w))
    ref_o, ref_lse = gb.attn_decode_splitkv(q, kc, vc, kl, num_splits=0, scale=w.scale)
    o = torch.empty_like(ref_o)
    lse = torch.empty_like(ref_lse)
    gb.attn_decode_splitkv_noalloc(q, kc, vc, kl, o, lse, num_splits=0, scale=w.scale)
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        gb.attn_decode_splitkv_noalloc(q, kc, vc, kl, o, lse, num_splits=0, scale=w.scale)
    for _ in range(2):
        o.fill_(float("nan"))
        lse.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert _close(o, ref_o), "graph replay: O differs from attn_decode_splitkv"
        assert (lse - ref_lse).abs().max().item() <= LSE_MAX_ABS
    st, word = gb.attn_last_device_error()
    assert st == 0, f"device error word {word}"
