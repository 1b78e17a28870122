"""GPU parity of attn_decode_splitkv against the fp64 oracle (plain definition with
kv_len); the cache rows past each sequence's length hold NaN, so any read of them that
reaches the output fails the test."""
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


def run_decode(w: wl.Workload, lens=None):
    q, kc, vc, kl = wl.decode_inputs(w)
    if lens is not None:
        kl = torch.tensor(lens, dtype=torch.int32)
        for b, n in enumerate(lens):
            kc[b, :, n:] = float("nan")
            vc[b, :, n:] = float("nan")
    o, lse = gb.attn_decode_splitkv(q.cuda(), kc.cuda(), vc.cuda(), kl.cuda(),
                                    num_splits=w.num_splits, scale=w.scale)
    torch.cuda.synchronize()
    o = o.float().cpu().numpy()[:, :, 0]
    lse = lse.cpu().numpy()
    o_ref, lse_ref = oracle.attention(wl.to_oracle(q), wl.to_oracle(kc), wl.to_oracle(vc),
                                      w.scale, False, kv_len=kl.numpy())
    return compare(o, lse, o_ref[:, :, 0], lse_ref[:, :, 0], w.dtype, w.name)


def small(B, Hq, Hkv, Lmax, d, num_splits, lo, hi, seed=3):
    return wl.Workload(f"dec-b{B}-h{Hq}/{Hkv}-l{Lmax}-d{d}-s{num_splits}", "decode", B=B, Hq=Hq,
                       Hkv=Hkv, d=d, dtype="bf16", Skv=Lmax, num_splits=num_splits,
                       len_lo=lo, len_hi=hi, seed=seed)


@pytest.mark.parametrize("B,Hq,Hkv,Lmax,d,ns,lens", [
    (2, 8, 1, 256, 128, 1, [256, 100]),
    (3, 16, 2, 1000, 128, 3, [1000, 63, 65]),
    (4, 8, 8, 300, 128, 16, [1, 64, 2, 300]),          # G = 1, more splits than tiles
    (2, 16, 1, 5000, 128, 0, [5000, 4097]),           # G = 16 (two head chunks), auto
    (2, 8, 2, 777, 64, 4, [777, 129]),                # d = 64
    (5, 64, 8, 9000, 128, 0, [0, 1, 4096, 8191, 9000]),   # empty sequence, auto splits
])
def test_decode_shapes(B, Hq, Hkv, Lmax, d, ns, lens):
    run_decode(small(B, Hq, Hkv, Lmax, d, ns, Lmax, Lmax), lens=lens)


@pytest.mark.parametrize("B,Hq,Hkv,Lmax,d,ns,lens", [
    (1, 64, 8, 131072, 128, 0, [131072]),             # 8 groups x 32 splits = 256 items
    (2, 64, 8, 65536, 128, 0, [65536, 40000]),        # 16 groups x 16 splits, ragged
    (2, 16, 2, 70000, 64, 64, [70000, 33333]),        # d = 64: 4 groups x 64 splits
])
def test_single_launch_two_ctas_per_sm(B, Hq, Hkv, Lmax, d, ns, lens):
    # single-launch merge with more work items than SMs: two CTAs per SM, 2-stage rings
    import torch
    nsm = torch.cuda.get_device_properties(0).multi_processor_count
    p = gb.attn_decode_plan(B, Hq, Hkv, 1, Lmax, d, ns, nsm)
    assert p["merge"] == "single_launch" and p["items"] > nsm
    run_decode(small(B, Hq, Hkv, Lmax, d, ns, Lmax, Lmax, seed=31), lens=lens)


@pytest.mark.parametrize("ns", [1, 2, 7, 16, 64, 0])
def test_decode_split_count_invariance(ns):
    run_decode(small(2, 64, 8, 6000, 128, ns, 5000, 6000, seed=21))


def test_workload4_llama70b_decode_full():
    run_decode(wl.WORKLOADS[4])


@pytest.mark.slow
def test_workload5_ragged_decode_all_rows():
    # every one of the 16 x 64 output rows against the oracle (lengths 1024 to 131072)
    run_decode(wl.WORKLOADS[5])


def test_decode_deterministic_repeat():
    w = small(4, 64, 8, 20000, 128, 0, 10000, 20000, seed=8)
    q, kc, vc, kl = (t.cuda() for t in wl.decode_inputs(w))
    o1, l1 = gb.attn_decode_splitkv(q, kc, vc, kl)
    o2, l2 = gb.attn_decode_splitkv(q, kc, vc, kl)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_decode_workspace_too_small_is_rejected():
    w = small(1, 8, 1, 128, 128, 1, 128, 128)
    q, kc, vc, kl = (t.cuda() for t in wl.decode_inputs(w))
    ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(gb.GbAttnError):
        gb.attn_decode_splitkv(q, kc, vc, kl, num_splits=1, workspace=ws)
