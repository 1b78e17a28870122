"""GPU parity of attn_fwd (bf16 tcgen05 path and fp32 path) against the fp64 oracle.

All calls go through the C ABI (libgbattn.so) via the Python binding.  Inputs come from
attn_workloads (seeded, CPU-generated); the oracle sees exactly the stored bytes.
"""
import math

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


def run_gpu(q, k, v, causal, scale):
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o, lse = gb.attn_fwd(qd, kd, vd, causal=causal, scale=scale)
    torch.cuda.synchronize()
    return o.float().cpu().numpy(), lse.cpu().numpy()


def check(w: wl.Workload, rows=None):
    q, k, v = wl.prefill_inputs(w)
    o, lse = run_gpu(q, k, v, w.causal, w.scale)
    if rows is None:
        o_ref, lse_ref = oracle.attention(wl.to_oracle(q), wl.to_oracle(k), wl.to_oracle(v),
                                          w.scale, w.causal)
        return compare(o, lse, o_ref, lse_ref, w.dtype, w.name)
    o_ref, lse_ref = oracle.attention(wl.to_oracle(q), wl.to_oracle(k), wl.to_oracle(v),
                                      w.scale, w.causal, rows=rows)
    return compare(o.reshape(-1, w.d)[rows], lse.reshape(-1)[rows], o_ref, lse_ref, w.dtype,
                   w.name)


def small(B, Hq, Hkv, Sq, Skv, d, causal, dtype="bf16", seed=7, q_scale=1.0):
    return wl.Workload(f"b{B}-h{Hq}/{Hkv}-s{Sq}x{Skv}-d{d}-{'c' if causal else 'nc'}-{dtype}",
                       "prefill", B=B, Hq=Hq, Hkv=Hkv, d=d, dtype=dtype, Sq=Sq, Skv=Skv,
                       causal=causal, seed=seed, q_scale=q_scale)


# ---------------------------------------------------------------------------------------
# fp32 path
# ---------------------------------------------------------------------------------------

def test_workload1_tiny_fp32():
    check(wl.WORKLOADS[1])


@pytest.mark.parametrize("B,Hq,Hkv,Sq,Skv,d,causal", [
    (1, 2, 1, 128, 128, 64, True),
    (2, 4, 2, 77, 200, 128, False),
    (2, 4, 2, 77, 200, 128, True),
    (1, 8, 1, 1, 33, 64, True),
    (1, 1, 1, 300, 300, 128, True),
])
def test_fp32_shapes(B, Hq, Hkv, Sq, Skv, d, causal):
    check(small(B, Hq, Hkv, Sq, Skv, d, causal, dtype="fp32"))


# ---------------------------------------------------------------------------------------
# bf16 tcgen05 path
# ---------------------------------------------------------------------------------------

@pytest.mark.parametrize("B,Hq,Hkv,Sq,Skv,d,causal", [
    (1, 2, 1, 128, 128, 128, False),   # one pair of Q tiles, one KV tile
    (1, 2, 1, 128, 128, 128, True),
    (1, 2, 2, 256, 256, 128, True),    # G = 1: pairs are consecutive q blocks
    (1, 8, 2, 384, 384, 128, True),    # GQA G = 4
    (2, 8, 1, 200, 200, 128, True),    # ragged tail, G = 8
    (1, 4, 4, 129, 129, 128, False),   # one row past a tile
    (1, 3, 1, 127, 255, 128, False),   # odd G, Sq != Skv
    (1, 4, 2, 100, 300, 128, True),    # bottom-right causal with Sq < Skv
    (1, 2, 1, 1, 1, 128, False),       # single query, single key
    (1, 2, 1, 1, 517, 128, True),      # one query row at the end of a long context
    (2, 4, 2, 256, 256, 64, True),     # d = 64
    (1, 6, 3, 130, 1000, 64, False),
])
def test_bf16_shapes(B, Hq, Hkv, Sq, Skv, d, causal):
    check(small(B, Hq, Hkv, Sq, Skv, d, causal))


def test_bf16_sharp_softmax_rescale_path():
    # Q scaled up so that the running max moves by more than 2^8 between tiles
    check(small(1, 2, 1, 256, 1024, 128, True, q_scale=6.0, seed=11))


@pytest.mark.parametrize("causal,Hq,Hkv,Sq", [
    (False, 2, 1, 128),      # KV-split mode (persistent CTAs)
    (True, 64, 8, 1024),     # pair mode: 256 pairs of Q tiles
    (False, 64, 8, 1024),
])
def test_bf16_max_moves_in_some_rows_of_a_warp(causal, Hq, Hkv, Sq):
    # Keys 512 + (r mod 128) are aligned with query row r of head 0 for every third row r,
    # so those rows' running max jumps by far more than 2^8 in a later KV tile while most
    # other rows of the same warps keep theirs: within one warp some rows rescale their O
    # accumulator and row sum and the others do not.
    w = small(1, Hq, Hkv, Sq, 1024, 128, causal, seed=13)
    q, k, v = wl.prefill_inputs(w)
    qf = q.float()
    for r in range(0, Sq, 3):
        if causal and 512 + r % 128 > r + (w.Skv - w.Sq):
            continue
        u = qf[0, 0, r] / qf[0, 0, r].norm()
        k[0, 0, 512 + r % 128] = (21.0 * u).to(k.dtype)
    # precondition, in fp32 on the stored values: within one warp of head 0, some rows' max
    # after their first KV tile is exceeded by more than 2^8 later on and some rows' is not
    c = w.scale / math.log(2.0)
    s = (qf[0, 0] @ k[0, 0].float().T) * c
    if causal:
        s = s.masked_fill(torch.ones(w.Sq, w.Skv, dtype=torch.bool).triu(w.Skv - w.Sq + 1), -math.inf)
    first = s[:, :128].max(dim=1).values
    moves = (s[:, 128:].max(dim=1).values > first + 8.0).numpy()
    warps = moves[: Sq // 32 * 32].reshape(-1, 32)
    assert (warps.any(axis=1) & ~warps.all(axis=1)).any()
    o, lse = run_gpu(q, k, v, w.causal, w.scale)
    o_ref, lse_ref = oracle.attention(wl.to_oracle(q), wl.to_oracle(k), wl.to_oracle(v),
                                      w.scale, w.causal)
    compare(o, lse, o_ref, lse_ref, w.dtype, w.name)


def test_workload2_causal_gqa_prefill_full():
    check(wl.WORKLOADS[2])


@pytest.mark.slow
def test_workload3_llama70b_prefill_100k_rows():
    # 100,000 random rows, every row of one whole query head (all 64 Q tiles, the diagonal
    # tile of each), the first Q tile of head 0 and the last rows of the last head
    w = wl.WORKLOADS[3]
    rng = np.random.default_rng(3)
    n_rows = w.B * w.Hq * w.Sq
    rows = np.unique(np.concatenate([
        rng.choice(n_rows, 100_000, replace=False),
        37 * w.Sq + np.arange(w.Sq),                         # head 37, all 8192 rows
        np.arange(0, 128),                                   # head 0, first tile (diagonal)
        (w.Hq - 1) * w.Sq + np.arange(w.Sq - 130, w.Sq),     # last head, last rows
    ]))
    assert rows.size >= 100_000
    check(w, rows=rows)


def test_constant_v_and_causal_row0():
    w = small(1, 4, 2, 256, 256, 128, True, seed=5)
    q, k, v = wl.prefill_inputs(w)
    v[:] = 0.8125                      # exactly representable in bf16
    o, _ = run_gpu(q, k, v, True, w.scale)
    assert np.abs(o - 0.8125).max() <= 1e-2
    v2 = wl.prefill_inputs(w)[2]
    o2, lse2 = run_gpu(q, k, v2, True, w.scale)
    # causal row 0 sees key 0 only: O = V[0] exactly (p = 1), LSE = scale * q0 . k0
    for h in range(4):
        np.testing.assert_array_equal(o2[0, h, 0], v2[0, h // 2, 0].float().numpy())
        dot = float((q[0, h, 0].double() * k[0, h // 2, 0].double()).sum())
        assert abs(lse2[0, h, 0] - w.scale * dot) < 1e-3


def test_deterministic_repeat():
    w = small(1, 8, 2, 512, 512, 128, True, seed=9)
    q, k, v = (t.cuda() for t in wl.prefill_inputs(w))
    o1, l1 = gb.attn_fwd(q, k, v, causal=True)
    o2, l2 = gb.attn_fwd(q, k, v, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_gpu_rejects_bad_arguments_without_launch():
    q = torch.zeros(1, 2, 64, 96, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(gb.GbAttnError):
        gb.attn_fwd(q, q[:, :1], q[:, :1], causal=False)


def test_bounded_wait_expiry_is_reported_and_context_survives():
    """A device wait that can never be satisfied gives up, reports GBATTN_ERR_TIMEOUT with
    the self-test code through the error word, and later work still runs correctly."""
    st, word = gb.attn_last_device_error()
    assert st == 0, f"error word already set: {word}"
    gb.attn_selftest_bounded_wait()
    st, word = gb.attn_last_device_error()
    assert st == gb.GBATTN_ERR_TIMEOUT and word == 6
    st, word = gb.attn_last_device_error()          # read-and-clear
    assert st == 0 and word == 0
    check(small(1, 4, 2, 200, 200, 128, True, seed=13))


def test_bf16_pair_mode_full_compare():
    # 320 pairs of Q tiles (>= 2 per SM): the kernel runs in pair mode (two heads of one
    # KV head per CTA); the small shapes above run in KV-split mode.
    check(small(1, 32, 8, 2560, 2560, 128, True, seed=17))


def test_bf16_pair_mode_between_one_and_two_pairs_per_sm():
    # 256 pairs on 152 SMs (1.7 per SM): pair mode since at least one pair per SM, one wave
    # of 152 CTAs then 104 more (causal, so no KV-split tail)
    check(small(1, 32, 8, 2048, 2048, 128, True, seed=37))


def test_bf16_pair_mode_g1_causal_ragged_odd_tiles():
    # pair mode with G = 1: a CTA's two Q tiles are consecutive q blocks of one head with
    # different causal extents; 9 q blocks per head leave a last CTA with one tile, and
    # Sq = 1100 ends in a ragged tile.
    check(small(1, 64, 64, 1100, 1100, 128, True, seed=23))


def test_bf16_pair_mode_g3_noncausal_ragged():
    # pair mode with G = 3 and 5 q blocks: 15 tiles per KV head, so pairs straddle q blocks
    # and the last pair has one tile; ragged Sq and Skv
    check(small(1, 120, 40, 600, 700, 128, False, seed=29))


def test_bf16_single_sm_pair_mode_d64():
    # d = 64 with >= 2 pairs per SM: the one-SM kernel in pair mode
    check(small(1, 32, 8, 2560, 2560, 64, True, seed=31))


def test_bf16_split_mode_ragged_noncausal_long_kv():
    # few Q tiles and a long KV range: one tile's two KV halves merged in the CTA
    check(small(1, 2, 1, 100, 3000, 128, False, seed=19))


@pytest.mark.parametrize("B,Hq,Hkv,S", [(1, 32, 8, 4096), (2, 32, 8, 3072)])
def test_noncausal_with_split_tail_sampled(B, Hq, Hkv, S):
    # 512 (768) equal pairs on 152 SMs leave a last wave of 56 (8) pairs: those run as single
    # Q tiles in KV-split mode in a second launch (the first Q blocks of every head, since
    # they are the last in the pairs' order); sample rows there and elsewhere
    w = small(B, Hq, Hkv, S, S, 128, False, seed=31)
    rng = np.random.default_rng(31)
    n_rows = B * Hq * S
    heads = np.arange(B * Hq)
    rows = np.unique(np.concatenate([
        (heads[:, None] * S + rng.integers(0, 512, (B * Hq, 4))).reshape(-1),   # tail tiles
        rng.integers(0, n_rows, 200),
        [0, n_rows - 1],
    ]))
    check(w, rows=rows)


def test_noncausal_tail_launch_repeat_and_graph():
    # the two launches of a call with a KV-split tail replay in a CUDA graph as one step
    w = small(1, 32, 8, 4096, 4096, 128, False, seed=33)
    q, k, v = (t.cuda() for t in wl.prefill_inputs(w))
    o1, l1 = gb.attn_fwd(q, k, v, causal=False)
    o = torch.empty_like(o1)
    lse = torch.empty_like(l1)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        gb.attn_fwd(q, k, v, causal=False, out=o, lse=lse)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        gb.attn_fwd(q, k, v, causal=False, out=o, lse=lse)
    o.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(o, o1) and torch.equal(lse, l1)


def test_output_16_byte_aligned_only():
    # an output that is 16- but not 32-byte aligned takes the epilogue's 16-byte stores; the
    # result is the same bits as with an aligned output
    w = small(1, 16, 2, 2048, 2048, 128, True, seed=35)
    q, k, v = (t.cuda() for t in wl.prefill_inputs(w))
    o_ref, l_ref = gb.attn_fwd(q, k, v, causal=True)
    buf = torch.empty(q.numel() + 64, dtype=torch.bfloat16, device="cuda")
    o = buf[8:8 + q.numel()].view(q.shape)          # 16 bytes past a 256-byte boundary
    assert o.data_ptr() % 32 == 16
    _, lse = gb.attn_fwd(q, k, v, causal=True, out=o)
    torch.cuda.synchronize()
    assert torch.equal(o, o_ref) and torch.equal(lse, l_ref)
