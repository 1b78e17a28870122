"""Seeded random shapes against the fp64 oracle, across the kernels' mode boundaries.

The hand-picked shape lists elsewhere cover named edge cases; here a seeded generator draws
shapes inside classes chosen so that every work split the library plans is hit at ragged,
unaligned sizes: prefill in KV-split mode (persistent CTAs), in pair mode, and in pair mode
with a KV-split tail launch; single-token decode with the single-launch merge and with the
per-group combine, with and without splits cut into pieces; multi-token decode on the warp
kernel (either merge) and on the tcgen05 kernel; chunked prefill against a padded cache.  The plan each shape gets is read
from the library's host-side planners (attn_prefill_plan, attn_decode_plan) for this GPU's SM
count, and the test asserts that every mode was drawn, so a change to the planners cannot
silently shrink the coverage.  Large shapes compare sampled rows (whole heads plus random
rows); the oracle computes those rows one by one.
"""
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


def _nsm() -> int:
    return torch.cuda.get_device_properties(0).multi_processor_count


# ---------------------------------------------------------------------------------------
# shape draws (seeded; independent of the GPU except for the SM count the plan uses)
# ---------------------------------------------------------------------------------------

def prefill_shapes(nsm: int):
    """(B, Hq, Hkv, Sq, Skv, d, causal, plan) for 24 KV-split, 12 pair and 8 tail draws."""
    rng = np.random.default_rng(20261203)
    out = {"kv_split": [], "pairs": [], "tail": []}
    want = {"kv_split": 24, "pairs": 12, "tail": 8}
    for _ in range(5000):
        if all(len(out[c]) >= want[c] for c in out):
            break
        cls = [c for c in out if len(out[c]) < want[c]][0]
        d = int(rng.choice([64, 128]))
        if cls == "kv_split":
            B = int(rng.integers(1, 3))
            Hkv = int(rng.choice([1, 2]))
            Hq = Hkv * int(rng.choice([1, 2, 3, 4]))
            Sq = int(rng.integers(1, 700))
            Skv = int(rng.integers(1, 900))
            causal = bool(rng.integers(0, 2))
        elif cls == "pairs":
            B, Hkv = 1, 8
            Hq = Hkv * int(rng.choice([4, 8]))
            Sq = int(rng.integers(700, 1700))
            Skv = Sq + int(rng.integers(0, 300))
            causal = bool(rng.integers(0, 2))
        else:
            B, Hkv = 1, int(rng.choice([4, 8]))
            Hq = Hkv * 8
            Sq = int(rng.integers(1500, 3500))
            Skv = int(rng.integers(600, 1500))
            causal = False
        if causal and Sq > Skv:
            Sq, Skv = Skv, Sq
        plan = gb.attn_prefill_plan(B, Hq, Hkv, Sq, Skv, causal, nsm)
        got = "tail" if plan["tail_pairs"] > 0 else plan["mode"]
        if got == cls:
            out[cls].append((B, Hq, Hkv, Sq, Skv, d, causal, plan))
    else:
        raise AssertionError(f"prefill draws did not fill every class: { {c: len(v) for c, v in out.items()} }")
    return [s for c in ("kv_split", "pairs", "tail") for s in out[c]]


DECODE_DRAWS = 6
DECODE_KINDS = ("single_launch", "single_launch+two_per_sm", "combine_per_group",
                "combine_per_group+pieces", "mt:single_launch", "mt:combine",
                "mt:tcgen05", "mt:tcgen05+row_tiles")


def decode_kind(Tq: int, plan: dict, nsm: int) -> str:
    """Single-token calls merge in the split kernel (single launch: one CTA per SM in one
    wave, two per SM with more items than SMs) or per group (with or without pieces);
    multi-token calls (mt:) run the warp kernel with either merge, or the tcgen05 kernel (its
    partials counted per 128-row tile; one tile per KV head, or several)."""
    if plan["kernel"] == "tcgen05":
        k = "tcgen05" + ("+row_tiles" if plan["rows_per_kv_head"] > 128 else "")
    else:
        k = plan["merge"] + ("+pieces" if plan["pieces"] > 1 else "")
        if Tq == 1 and plan["merge"] == "single_launch" and plan["items"] > nsm:
            k += "+two_per_sm"
    return ("mt:" + k) if Tq > 1 else k


def decode_shapes(nsm: int):
    """(B, Hq, Hkv, Tq, lens, Lmax, d, num_splits, kind): 6 draws of each kind in DECODE_KINDS."""
    rng = np.random.default_rng(777)
    special = [0, 1, 63, 64, 65, 127, 129, 4095, 4097]
    counts = {k: 0 for k in DECODE_KINDS}
    shapes = []
    for _ in range(5000):
        if min(counts.values()) >= DECODE_DRAWS:
            break
        multi = bool(rng.integers(0, 2))
        B = int(rng.integers(1, 7))
        Hkv = int(rng.choice([1, 2, 4, 8]))
        G = int(rng.choice([1, 2, 4, 8]))
        Tq = int(rng.choice(list(range(2, 13)) + [17, 20, 33])) if multi else 1
        d = int(rng.choice([64, 128]))
        hi = int(rng.choice([600, 5000, 40000]))
        lens = [int(rng.choice(special)) if rng.random() < 0.25 else int(rng.integers(1, hi + 1))
                for _ in range(B)]
        lens = [max(n, Tq) if multi and rng.random() < 0.8 else n for n in lens]
        ns = int(rng.choice([0, 0, 1, 2, 5, 16, 37]))
        Lmax = max(max(lens), Tq, 1) + int(rng.integers(0, 200))
        Hq = Hkv * G
        k = decode_kind(Tq, gb.attn_decode_plan(B, Hq, Hkv, Tq, Lmax, d, ns, nsm), nsm)
        if counts.get(k, DECODE_DRAWS) >= DECODE_DRAWS:
            continue
        counts[k] += 1
        shapes.append((B, Hq, Hkv, Tq, lens, Lmax, d, ns, k))
    else:
        raise AssertionError(f"decode draws did not reach every kind: {counts}")
    return shapes


def chunk_shapes():
    rng = np.random.default_rng(4242)
    shapes = []
    for _ in range(16):
        B = int(rng.integers(1, 3))
        Hkv = int(rng.choice([1, 2, 8]))
        Hq = Hkv * int(rng.choice([1, 2, 4, 8]))
        d = int(rng.choice([64, 128]))
        Sq = int(rng.integers(1, 400))
        ctx = Sq + int(rng.integers(0, 3000))
        Lmax = ctx + int(rng.integers(0, 300))
        causal = bool(rng.integers(0, 4))       # mostly causal
        shapes.append((B, Hq, Hkv, Sq, ctx, Lmax, d, causal))
    return shapes


def _sample_rows(B, Hq, S, rng):
    """All rows of the first and last head plus 1500 random rows (flattened [B, Hq, S])."""
    n = B * Hq * S
    return np.unique(np.concatenate([np.arange(S), (B * Hq - 1) * S + np.arange(S),
                                     rng.choice(n, min(n, 1500), replace=False)]))


# ---------------------------------------------------------------------------------------
# tests
# ---------------------------------------------------------------------------------------

def test_prefill_draws_cover_every_mode():
    modes = {("tail" if s[7]["tail_pairs"] else s[7]["mode"]) for s in prefill_shapes(_nsm())}
    assert modes == {"kv_split", "pairs", "tail"}


@pytest.mark.parametrize("i", range(44))
def test_prefill_random_shape(i):
    B, Hq, Hkv, Sq, Skv, d, causal, plan = prefill_shapes(_nsm())[i]
    w = wl.Workload(f"rand{i}-b{B}-h{Hq}/{Hkv}-s{Sq}x{Skv}-d{d}-{'c' if causal else 'nc'}-{plan['mode']}",
                    "prefill", B=B, Hq=Hq, Hkv=Hkv, d=d, dtype="bf16", Sq=Sq, Skv=Skv,
                    causal=causal, seed=5000 + i)
    q, k, v = wl.prefill_inputs(w)
    o, lse = gb.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=causal, scale=w.scale)
    torch.cuda.synchronize()
    o = o.float().cpu().numpy()
    lse = lse.cpu().numpy()
    args = (wl.to_oracle(q), wl.to_oracle(k), wl.to_oracle(v), w.scale, causal)
    if B * Hq * Sq <= 40_000:
        o_ref, lse_ref = oracle.attention(*args)
        compare(o, lse, o_ref, lse_ref, "bf16", w.name)
    else:
        rows = _sample_rows(B, Hq, Sq, np.random.default_rng(i))
        o_ref, lse_ref = oracle.attention(*args, rows=rows)
        compare(o.reshape(-1, d)[rows], lse.reshape(-1)[rows], o_ref, lse_ref, "bf16", w.name)


def test_decode_draws_cover_every_mode():
    assert sorted(s[8] for s in decode_shapes(_nsm())) == sorted(DECODE_KINDS * DECODE_DRAWS)


@pytest.mark.parametrize("i", range(DECODE_DRAWS * len(DECODE_KINDS)))
def test_decode_random_shape(i):
    B, Hq, Hkv, Tq, lens, Lmax, d, ns, kind = decode_shapes(_nsm())[i]
    g = torch.Generator().manual_seed(9000 + i)
    q = torch.randn(B, Hq, Tq, d, generator=g).to(torch.bfloat16)
    kc = torch.full((B, Hkv, Lmax, d), float("nan"), dtype=torch.bfloat16)
    vc = torch.full((B, Hkv, Lmax, d), float("nan"), dtype=torch.bfloat16)
    for b, n in enumerate(lens):
        kc[b, :, :n] = torch.randn(Hkv, n, d, generator=g).to(torch.bfloat16)
        vc[b, :, :n] = torch.randn(Hkv, n, d, generator=g).to(torch.bfloat16)
    kl = torch.tensor(lens, dtype=torch.int32)
    scale = d ** -0.5
    args = (q.cuda(), kc.cuda(), vc.cuda(), kl.cuda())
    if Tq == 1:
        o, lse = gb.attn_decode_splitkv(*args, num_splits=ns, scale=scale)
        lse = lse[..., None]
    else:
        o, lse = gb.attn_decode_multitoken(*args, num_splits=ns, scale=scale)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.attention(wl.to_oracle(q), wl.to_oracle(kc), wl.to_oracle(vc), scale,
                                      Tq > 1, kv_len=kl.numpy())
    compare(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, "bf16",
            f"rand{i}-{kind}-b{B}-h{Hq}/{Hkv}-t{Tq}-d{d}-ns{ns}-lens{lens}")


@pytest.mark.parametrize("i", range(16))
def test_chunked_prefill_random_shape(i):
    B, Hq, Hkv, Sq, ctx, Lmax, d, causal = chunk_shapes()[i]
    w = wl.Workload(f"rand{i}-chunk-b{B}-h{Hq}/{Hkv}-q{Sq}-ctx{ctx}-cap{Lmax}-d{d}", "chunk", B=B,
                    Hq=Hq, Hkv=Hkv, d=d, dtype="bf16", Sq=Sq, Skv=Lmax, causal=causal,
                    len_lo=ctx, len_hi=ctx, seed=7000 + i)
    q, kc, vc, ctx = wl.chunk_inputs(w)
    o, lse = gb.attn_prefill_kvcache(q.cuda(), kc.cuda(), vc.cuda(), ctx, causal=causal,
                                     scale=w.scale)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.attention(wl.to_oracle(q), wl.to_oracle(kc), wl.to_oracle(vc),
                                      w.scale, causal, kv_len=np.full(B, ctx, np.int32))
    compare(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, "bf16", w.name)
