"""Causal tile skipping, checked by counting the work the prefill kernels issue.

"ADR-0060: AHBM GQA Fused Attention Kernel (Llama3-70B)", section 11 asks that a causal
prefill skip every KV tile lying wholly in a query tile's future (section 5.4's "future"
class), so that the number of S = Q K^T tile products is the lower-triangular count and not
the full grid.  attn_fwd_counted adds the S tile products its kernels issue to a device
counter; the expected number is the closed form

    sum over 128-row Q tiles of ceil(visible keys of the tile's last row / 128),

where row i sees min(Skv, i + Skv - Sq + 1) keys when causal (bottom-right) and Skv
otherwise.  The cases cover every prefill work split: KV-split mode (workload 2), pairs of
Q tiles (workload 3), pairs with the KV-split tail launch (non-causal, 56 of 152 in the
last wave), ragged Sq < Skv, G = 1 pairs of consecutive Q blocks.  The counted call must
also give the same bits as attn_fwd.
"""
import math

import pytest
import torch

import attn_workloads as wl
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


def expected_s_tiles(B, Hq, Sq, Skv, causal):
    per_head = 0
    for qb in range(math.ceil(Sq / 128)):
        last = min(qb * 128 + 128, Sq) - 1
        vis = min(Skv, last + Skv - Sq + 1) if causal else Skv
        per_head += math.ceil(vis / 128)
    return B * Hq * per_head


@pytest.mark.parametrize("B,Hq,Hkv,Sq,Skv,causal", [
    (2, 8, 2, 2048, 2048, True),       # workload 2: KV-split mode
    (1, 64, 8, 8192, 8192, True),      # workload 3: pairs of Q tiles
    (1, 4, 2, 100, 300, True),         # ragged, Sq < Skv
    (1, 64, 64, 1100, 1100, True),     # G = 1 pairs of consecutive Q blocks, ragged end
    (1, 32, 8, 4096, 4096, False),     # pairs plus the KV-split tail launch
    (1, 2, 1, 130, 1000, True),        # KV split, two Q tiles of very different extent
])
def test_issued_s_tiles_equal_the_closed_form(B, Hq, Hkv, Sq, Skv, causal):
    w = wl.Workload("tiles", "prefill", B=B, Hq=Hq, Hkv=Hkv, d=128, dtype="bf16", Sq=Sq, Skv=Skv,
                    causal=causal, seed=71)
    q, k, v = (t.cuda() for t in wl.prefill_inputs(w))
    s_tiles = torch.zeros(1, dtype=torch.int32, device="cuda")
    o, lse = gb.attn_fwd_counted(q, k, v, causal, s_tiles)
    o_ref, lse_ref = gb.attn_fwd(q, k, v, causal=causal)
    torch.cuda.synchronize()
    want = expected_s_tiles(B, Hq, Sq, Skv, causal)
    assert int(s_tiles.item()) == want
    if causal and Sq == Skv and Sq > 128:
        # strictly fewer than the full grid of Q tiles x K/V tiles
        assert want < B * Hq * math.ceil(Sq / 128) * math.ceil(Skv / 128)
    assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)


def test_counter_accumulates_over_calls():
    w = wl.Workload("tiles2", "prefill", B=1, Hq=4, Hkv=1, d=64, dtype="bf16", Sq=513, Skv=513,
                    causal=True, seed=72)
    q, k, v = (t.cuda() for t in wl.prefill_inputs(w))
    s_tiles = torch.zeros(1, dtype=torch.int32, device="cuda")
    gb.attn_fwd_counted(q, k, v, True, s_tiles)
    gb.attn_fwd_counted(q, k, v, True, s_tiles)
    torch.cuda.synchronize()
    assert int(s_tiles.item()) == 2 * expected_s_tiles(1, 4, 513, 513, True)
