"""GPU parity of attn_decode_multitoken (Tq new tokens per sequence, causal among them)
with the fp64 oracle: the oracle's bottom-right causal rule with Sq = Tq and the
sequence's length is exactly "token t sees keys <= len - Tq + t"."""
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


def make(B, Hq, Hkv, Tq, Lmax, d, lens, seed=5):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, Hq, Tq, d, generator=g).to(torch.bfloat16)
    kc = torch.full((B, Hkv, Lmax, d), float("nan"), dtype=torch.bfloat16)
    vc = torch.full((B, Hkv, Lmax, d), float("nan"), dtype=torch.bfloat16)
    for b, n in enumerate(lens):
        kc[b, :, :n] = torch.randn(Hkv, n, d, generator=g).to(torch.bfloat16)
        vc[b, :, :n] = torch.randn(Hkv, n, d, generator=g).to(torch.bfloat16)
    return q, kc, vc, torch.tensor(lens, dtype=torch.int32)


def run(B, Hq, Hkv, Tq, Lmax, d, lens, ns, seed=5):
    q, kc, vc, kl = make(B, Hq, Hkv, Tq, Lmax, d, lens, seed)
    scale = d ** -0.5
    o, lse = gb.attn_decode_multitoken(q.cuda(), kc.cuda(), vc.cuda(), kl.cuda(), num_splits=ns,
                                       scale=scale)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.attention(wl.to_oracle(q), wl.to_oracle(kc), wl.to_oracle(vc), scale,
                                      True, kv_len=kl.numpy())
    compare(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, "bf16",
            f"Tq{Tq} G{Hq // Hkv} d{d} ns{ns}")


@pytest.mark.parametrize("B,Hq,Hkv,Tq,Lmax,d,lens,ns", [
    (2, 16, 2, 2, 3000, 128, [3000, 1200], 4),        # G*Tq = 16: two row chunks
    (2, 64, 8, 4, 5000, 128, [5000, 4097], 0),        # Llama3-70B heads, 4 tokens, auto
    (3, 8, 8, 3, 700, 128, [700, 65, 3], 16),         # G = 1, ragged, tiny sequences
    (1, 8, 1, 8, 2048, 64, [2048], 3),                # 64 rows, d = 64
    (2, 4, 2, 5, 300, 128, [2, 300], 2),              # len < Tq: rows with no visible key
    (2, 16, 2, 3, 1500, 128, [1500, 700], 0),         # 3 row chunks: a group of 4 with one empty
    (1, 8, 2, 10, 900, 128, [900], 2),                # 5 row chunks: a second group of one chunk
    (2, 16, 2, 20, 1300, 128, [1300, 555], 3),        # 160 rows per KV head: two 128-row tiles
    (1, 32, 4, 6, 700, 64, [700], 0),                 # 48 rows, d = 64, automatic splits
    (2, 16, 2, 4, 300, 128, [2, 300], 2),             # tcgen05 path with len < Tq: rows see no key
    (3, 16, 2, 2, 500, 128, [0, 500, 17], 4),         # tcgen05 path: an empty sequence, short ones
    (2, 16, 2, 4, 600, 128, [0, 0], 3),               # tcgen05 path: no keys anywhere, no work item
    (1, 16, 2, 64, 900, 128, [900], 3),               # 512 rows per KV head: four 128-row tiles
    (2, 8, 1, 40, 700, 64, [700, 45], 0),             # 320 rows, d = 64, len < T_q, automatic
    (2, 8, 2, 3, 9000, 128, [9000, 4100], 4),         # 12 rows, long splits: tcgen05 path
    (1, 8, 8, 9, 5000, 64, [5000], 2),                # 9 rows, long splits, d = 64: tcgen05 path
])
def test_multitoken_decode_shapes(B, Hq, Hkv, Tq, Lmax, d, lens, ns):
    run(B, Hq, Hkv, Tq, Lmax, d, lens, ns)


def test_tq1_is_single_token_decode_bitwise():
    q, kc, vc, kl = make(2, 64, 8, 1, 9000, 128, [9000, 5000], seed=8)
    args = (q.cuda(), kc.cuda(), vc.cuda(), kl.cuda())
    o1, l1 = gb.attn_decode_multitoken(*args, num_splits=0)
    o2, l2 = gb.attn_decode_splitkv(*args, num_splits=0)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1[..., 0], l2)


def test_each_token_equals_its_own_single_token_decode():
    # token t of Tq equals a single-token decode with len - Tq + t + 1 keys
    Tq = 3
    q, kc, vc, kl = make(1, 16, 2, Tq, 4000, 128, [4000], seed=11)
    o, lse = gb.attn_decode_multitoken(q.cuda(), kc.cuda(), vc.cuda(), kl.cuda(), num_splits=5)
    for t in range(Tq):
        kl_t = torch.tensor([4000 - Tq + t + 1], dtype=torch.int32)
        o_t, l_t = gb.attn_decode_splitkv(q[:, :, t:t + 1].contiguous().cuda(), kc.cuda(), vc.cuda(),
                                          kl_t.cuda(), num_splits=5)
        torch.cuda.synchronize()
        assert (o[:, :, t:t + 1].float() - o_t.float()).abs().max().item() <= 2e-2
        assert (lse[:, :, t] - l_t).abs().max().item() <= 1e-3


@pytest.mark.parametrize("B,Hq,Hkv,Tq,Lmax,d,lens,ns", [
    # hundreds of work items over the persistent CTAs: each takes several, of 1 to 4 key
    # tiles, with a ragged last tile (NaN past len) in most of them
    (4, 16, 8, 8, 8192, 128, [8192, 5000, 1500, 777], 16),
    (4, 32, 8, 4, 6000, 64, [6000, 2500, 128, 4000], 32),
    (6, 16, 2, 16, 3000, 128, [3000, 0, 1, 2999, 130, 1024], 24),
])
def test_multitoken_decode_many_items_per_cta(B, Hq, Hkv, Tq, Lmax, d, lens, ns):
    run(B, Hq, Hkv, Tq, Lmax, d, lens, ns, seed=17)


def test_multitoken_workload7_llama70b_sampled():
    # the 4-token Llama3-70B decode at full size (512 work items), sampled rows
    w = wl.EXTRA_WORKLOADS[7]
    q, kc, vc, kl = wl.multitoken_inputs(w)
    o, lse = gb.attn_decode_multitoken(q.cuda(), kc.cuda(), vc.cuda(), kl.cuda(),
                                       num_splits=w.num_splits, scale=w.scale)
    torch.cuda.synchronize()
    rng = np.random.default_rng(7)
    n = w.B * w.Hq * w.Sq
    rows = np.unique(np.concatenate([rng.integers(0, n, 96), [0, n - 1]]))
    o_ref, lse_ref = oracle.attention(wl.to_oracle(q), wl.to_oracle(kc), wl.to_oracle(vc),
                                      w.scale, True, kv_len=kl.numpy(), rows=rows)
    compare(o.float().cpu().numpy().reshape(-1, w.d)[rows], lse.cpu().numpy().reshape(-1)[rows],
            o_ref, lse_ref, "bf16", w.name)


def test_multitoken_deterministic_repeat():
    # which CTA takes which item varies from call to call; the result may not
    q, kc, vc, kl = make(4, 64, 8, 4, 7000, 128, [7000, 6500, 3000, 7000], seed=23)
    args = (q.cuda(), kc.cuda(), vc.cuda(), kl.cuda())
    o1, l1 = gb.attn_decode_multitoken(*args, num_splits=16)
    o2, l2 = gb.attn_decode_multitoken(*args, num_splits=16)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
