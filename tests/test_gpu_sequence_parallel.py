"""GPU parity of the sequence-parallel pieces against the fp64 oracle, through the C ABI:

  * attn_fwd_positions (causal attention at explicit query / key positions) -- rows that see
    no key, all keys, the bottom-right case (bit-identical to attn_fwd), both work modes;
  * attn_merge ("ADR-0060" section 4 log-sum-exp merge) of partials over disjoint key
    ranges, every dtype combination, in place, empty partials;
  * the ring-KV prefill (section 5.5) and the reduce-to-root decode (section 4) of
    sequence_parallel.py, with P ranks emulated as threads on this one GPU: each thread runs
    the schedule with its own inputs, the point-to-point transport is a host queue, and all
    kernels go to one stream (no kernel waits on another rank's).
"""
import math
import queue
import threading

import numpy as np
import pytest
import torch

import attn_workloads as wl
import oracle
import streaming_attention_flashattention_gb300 as gb
from streaming_attention_flashattention_gb300 import sequence_parallel as sp
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


def bf16(shape, seed, scale=1.0):
    g = np.random.default_rng(seed)
    return torch.from_numpy((g.standard_normal(shape) * scale).astype(np.float32)).to(torch.bfloat16)


def positions_case(B, Hq, Hkv, Sq, Skv, d, q_pos0, k_pos0, seed=5, heads=None):
    q, k, v = bf16((B, Hq, Sq, d), seed), bf16((B, Hkv, Skv, d), seed + 1), bf16((B, Hkv, Skv, d), seed + 2)
    scale = 1.0 / math.sqrt(d)
    o, lse = gb.attn_fwd_positions(q.cuda(), k.cuda(), v.cuda(), q_pos0, k_pos0, scale=scale)
    torch.cuda.synchronize()
    o, lse = o.float().cpu().numpy(), lse.cpu().numpy()
    G = Hq // Hkv
    hs = range(Hq) if heads is None else heads
    for h in hs:
        qh = wl.to_oracle(q[:, h:h + 1])
        kh = wl.to_oracle(k[:, h // G:h // G + 1])
        vh = wl.to_oracle(v[:, h // G:h // G + 1])
        o_ref, l_ref = oracle.attention_at_positions(qh, kh, vh, scale, q_pos0, k_pos0)
        compare(o[:, h:h + 1], lse[:, h:h + 1], o_ref, l_ref, "bf16",
                f"positions B{B} H{Hq}/{Hkv} {Sq}x{Skv} d{d} q@{q_pos0} k@{k_pos0} h{h}")
    return o, lse


@pytest.mark.parametrize("B,Hq,Hkv,Sq,Skv,d,q_pos0,k_pos0", [
    (1, 4, 2, 300, 256, 128, 0, 100),       # rows 0..99 see no key, the rest a growing prefix
    (2, 4, 1, 200, 300, 64, 1000, 0),       # every row sees every key
    (1, 8, 2, 257, 129, 128, 5000, 4900),   # diagonal crossing the call, ragged tiles
    (1, 2, 2, 130, 400, 128, 0, -270),      # keys start before the queries
    (1, 4, 4, 129, 127, 64, 37, 37),        # same positions: square causal, Sq > Skv
    (3, 6, 3, 64, 200, 128, 150, 10),       # B > 1, G = 2, Sq < 128
])
def test_positions_parity(B, Hq, Hkv, Sq, Skv, d, q_pos0, k_pos0):
    positions_case(B, Hq, Hkv, Sq, Skv, d, q_pos0, k_pos0)


def test_positions_no_row_sees_a_key():
    q, k, v = bf16((1, 4, 200, 128), 1), bf16((1, 2, 64, 128), 2), bf16((1, 2, 64, 128), 3)
    o = torch.full((1, 4, 200, 128), 7.0, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((1, 4, 200), device="cuda")
    gb.attn_fwd_positions(q.cuda(), k.cuda(), v.cuda(), 0, 200, out=o, lse=lse)
    torch.cuda.synchronize()
    assert torch.all(o == 0).item() and torch.all(torch.isneginf(lse)).item()


def test_positions_bottom_right_is_attn_fwd_bit_for_bit():
    q, k, v = bf16((1, 16, 700, 128), 11).cuda(), bf16((1, 4, 900, 128), 12).cuda(), \
        bf16((1, 4, 900, 128), 13).cuda()
    o1, l1 = gb.attn_fwd(q, k, v, causal=True)
    o2, l2 = gb.attn_fwd_positions(q, k, v, 900 - 700 + 3000, 3000)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_positions_pair_mode_sampled_heads():
    # 48 pairs per KV head group x 8 groups: the pair kernel (not the KV-split one); rows
    # 0..511 see no key
    positions_case(1, 64, 8, 2048, 2048, 128, 0, 512, heads=[0, 9, 63])


def test_positions_split_mode_sampled_heads():
    positions_case(1, 16, 4, 1024, 1024, 128, 512, 1024, heads=[0, 5, 15])


# ---------------------------------------------------------------------------------------
# attn_merge
# ---------------------------------------------------------------------------------------

def _halves(Sq, n, cut, d, Hq=4, Hkv=2, q_pos0=None, seed=20):
    q, k, v = bf16((1, Hq, Sq, d), seed), bf16((1, Hkv, n, d), seed + 1), bf16((1, Hkv, n, d), seed + 2)
    qp = n - Sq if q_pos0 is None else q_pos0
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    pa = gb.attn_fwd_positions(qd, kd[:, :, :cut].contiguous(), vd[:, :, :cut].contiguous(), qp, 0)
    pb = gb.attn_fwd_positions(qd, kd[:, :, cut:].contiguous(), vd[:, :, cut:].contiguous(), qp, cut)
    ref = oracle.attention_at_positions(wl.to_oracle(q), wl.to_oracle(k), wl.to_oracle(v),
                                        1.0 / math.sqrt(d), qp, 0)
    return pa, pb, ref


@pytest.mark.parametrize("a32,b32,out32", [(False, False, False), (False, False, True),
                                          (True, False, True), (True, True, False),
                                          (False, True, True)])
@pytest.mark.parametrize("d", [64, 128])
def test_merge_of_key_halves_equals_whole(a32, b32, out32, d):
    (oa, la), (ob, lb), (o_ref, l_ref) = _halves(300, 700, 333, d)
    oa = oa.float() if a32 else oa
    ob = ob.float() if b32 else ob
    o, l = gb.attn_merge(oa, la, ob, lb, out_dtype=torch.float32 if out32 else torch.bfloat16)
    torch.cuda.synchronize()
    assert o.dtype == (torch.float32 if out32 else torch.bfloat16)
    compare(o.float().cpu().numpy(), l.cpu().numpy(), o_ref, l_ref, "bf16", f"merge d{d}")


def test_merge_in_place_accumulator_and_empty_partials():
    # queries at positions 0..299 against keys 0..699: the second half (keys 333..) is
    # empty for rows 0..332 (LSE -inf), so those rows take the first partial exactly
    (oa, la), (ob, lb), (o_ref, l_ref) = _halves(300, 700, 333, 128, q_pos0=0)
    acc_o, acc_l = oa.float(), la.clone()
    ptr = acc_o.data_ptr()
    gb.attn_merge(acc_o, acc_l, ob, lb, out=acc_o, lse_out=acc_l)
    torch.cuda.synchronize()
    assert acc_o.data_ptr() == ptr
    compare(acc_o.cpu().numpy(), acc_l.cpu().numpy(), o_ref, l_ref, "bf16", "merge in place")
    assert torch.isneginf(lb).all().item()                 # the second half saw no key
    assert torch.equal(acc_o, oa.float()) and torch.equal(acc_l, la)
    # an empty partial is dropped whatever its O holds (NaN here)
    nan_o = torch.full_like(acc_o, float("nan"))
    o2, l2 = gb.attn_merge(acc_o, acc_l, nan_o, lb)
    torch.cuda.synchronize()
    assert torch.equal(o2, acc_o) and torch.equal(l2, acc_l)
    # both partials empty: O = 0, LSE = -inf
    e_o = torch.full_like(acc_o, float("nan"))
    e_l = torch.full_like(acc_l, float("-inf"))
    o, l = gb.attn_merge(e_o, e_l, e_o, e_l)
    torch.cuda.synchronize()
    assert torch.all(o == 0).item() and torch.isneginf(l).all().item()


def test_merge_zero_rows_launches_nothing():
    z = torch.empty((0, 128), device="cuda")
    zl = torch.empty((0,), device="cuda")
    o, l = gb.attn_merge(z, zl, z, zl)
    assert o.shape == (0, 128) and l.shape == (0,)


# ---------------------------------------------------------------------------------------
# the schedules, P ranks as threads on this GPU
# ---------------------------------------------------------------------------------------

class ThreadComm:
    """Point-to-point transport between threads: a sender enqueues a snapshot (a copy made
    on the shared stream), the receiver copies it into its buffer."""

    def __init__(self, rank, world, boxes):
        self.rank, self.world, self.boxes = rank, world, boxes

    def _box(self, src, dst):
        return self.boxes[(src, dst)]

    def exchange(self, sends, recvs, dst, src):
        for t in sends:
            self._box(self.rank, dst).put(t.clone())
        comm = self

        class _H:
            def wait(self_):
                for t in recvs:
                    t.copy_(comm._box(src, comm.rank).get(timeout=120))
        return [_H()]

    def send(self, t, dst):
        self._box(self.rank, dst).put(t.clone())

    def recv(self, t, src):
        t.copy_(self._box(src, self.rank).get(timeout=120))


def run_ranks(world, fn):
    boxes = {(a, b): queue.Queue() for a in range(world) for b in range(world)}
    res, errs = [None] * world, []

    def body(r):
        try:
            res[r] = fn(r, ThreadComm(r, world, boxes))
        except BaseException as e:          # surfaced below
            errs.append(e)

    ts = [threading.Thread(target=body, args=(r,)) for r in range(world)]
    for t in ts:
        t.start()
    for t in ts:
        t.join(timeout=600)
    if errs:
        raise errs[0]
    torch.cuda.synchronize()
    return res


@pytest.mark.parametrize("world,B,Hq,Hkv,L,q_rows,q_pos0", [
    (2, 1, 8, 2, 256, None, 0),
    (4, 1, 8, 2, 192, None, 0),              # heads inside one group per rank
    (4, 2, 16, 4, 128, 300, 100),            # B > 1, a chunk from position 100
    (3, 1, 6, 3, 200, 128, 0),               # the first chunk only: later slices skipped
])
def test_ring_prefill_threads_equal_single_device(world, B, Hq, Hkv, L, q_rows, q_pos0):
    n = L * world
    S = n if q_rows is None else q_rows
    d = 128
    q, k, v = bf16((B, Hq, S, d), 31), bf16((B, Hkv, n, d), 32), bf16((B, Hkv, n, d), 33)
    hr = Hq // world
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()

    def rank_fn(r, comm):
        return sp.ring_prefill(qd[:, r * hr:(r + 1) * hr].contiguous(),
                               kd[:, :, r * L:(r + 1) * L].contiguous(),
                               vd[:, :, r * L:(r + 1) * L].contiguous(),
                               group_size=Hq // Hkv, q_pos0=q_pos0, comm=comm)

    res = run_ranks(world, rank_fn)
    o_ref, l_ref = oracle.attention_at_positions(wl.to_oracle(q), wl.to_oracle(k),
                                                 wl.to_oracle(v), 1.0 / math.sqrt(d), q_pos0, 0)
    for r, (o, l) in enumerate(res):
        assert o.dtype == torch.bfloat16 and o.shape == (B, hr, S, d)
        compare(o.float().cpu().numpy(), l.cpu().numpy(), o_ref[:, r * hr:(r + 1) * hr],
                l_ref[:, r * hr:(r + 1) * hr], "bf16", f"ring P{world} rank {r}")


@pytest.mark.parametrize("placement", ["contiguous", "round_robin"])
@pytest.mark.parametrize("world,root", [(3, 0), (4, 2), (5, 1)])
def test_decode_reduce_threads_equal_single_device(world, root, placement):
    # the cache split along the sequence in contiguous blocks ("ADR-0060" section 2.1), or
    # token by token round robin (position t on rank t mod P, the section's alternative)
    B, Hq, Hkv, d = 4, 64, 8, 128
    lens = [9000, 1, 0, 6000]
    Lmax = 9000
    c = -(-Lmax // world)
    q = bf16((B, Hq, d), 41)
    k, v = bf16((B, Hkv, Lmax, d), 42), bf16((B, Hkv, Lmax, d), 43)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()

    def rank_fn(r, comm):
        ks = torch.zeros((B, Hkv, c, d), dtype=torch.bfloat16, device="cuda")
        vs = torch.zeros_like(ks)
        if placement == "contiguous":
            lo, hi = r * c, min((r + 1) * c, Lmax)
            if hi > lo:
                ks[:, :, :hi - lo] = kd[:, :, lo:hi]
                vs[:, :, :hi - lo] = vd[:, :, lo:hi]
            held = [max(0, min(n - lo, c)) for n in lens]
        else:
            mine = kd[:, :, r::world]
            ks[:, :, :mine.shape[2]] = mine
            vs[:, :, :mine.shape[2]] = vd[:, :, r::world]
            held = [max(0, -(-(n - r) // world)) for n in lens]   # positions r, r + P, ... < n
        lens_r = torch.tensor(held, dtype=torch.int32, device="cuda")
        return sp.decode_reduce(qd, ks, vs, lens_r, root=root, comm=comm)

    res = run_ranks(world, rank_fn)
    o_ref, l_ref = oracle.attention(wl.to_oracle(q)[:, :, None, :], wl.to_oracle(k),
                                    wl.to_oracle(v), 1.0 / math.sqrt(d), False,
                                    kv_len=np.array(lens, np.int32))
    for r, (o, l) in enumerate(res):
        if r != root:
            assert o is None and l is None
            continue
        assert o.dtype == torch.bfloat16
        compare(o.float().cpu().numpy(), l.cpu().numpy(), o_ref[:, :, 0], l_ref[:, :, 0],
                "bf16", f"decode P{world} root {root} {placement}")


@pytest.mark.parametrize("Sq", [1, 5, 128, 129])
@pytest.mark.parametrize("Skv", [1, 5, 128, 129])
@pytest.mark.parametrize("shift", [-200, -3, 0, 2, 300])
def test_positions_grid_against_oracle(Sq, Skv, shift):
    # query i at position shift + i, key j at position j: every mix of rows that see no key,
    # some keys and all keys across the tile edges (d = 64, G = 2)
    q, k, v = bf16((1, 2, Sq, 64), 50 + Sq), bf16((1, 1, Skv, 64), 60 + Skv), bf16((1, 1, Skv, 64), 70 + Skv)
    o, lse = gb.attn_fwd_positions(q.cuda(), k.cuda(), v.cuda(), shift, 0, scale=0.125)
    torch.cuda.synchronize()
    o_ref, l_ref = oracle.attention_at_positions(wl.to_oracle(q), wl.to_oracle(k), wl.to_oracle(v),
                                                 0.125, shift, 0)
    compare(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, l_ref, "bf16",
            f"positions grid {Sq}x{Skv} shift {shift}")


def test_ring_prefill_threads_noncausal():
    world, Hq, Hkv, L, d = 2, 8, 2, 256, 128
    n = L * world
    q, k, v = bf16((1, Hq, n, d), 81), bf16((1, Hkv, n, d), 82), bf16((1, Hkv, n, d), 83)
    hr = Hq // world
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    res = run_ranks(world, lambda r, comm: sp.ring_prefill(
        qd[:, r * hr:(r + 1) * hr].contiguous(), kd[:, :, r * L:(r + 1) * L].contiguous(),
        vd[:, :, r * L:(r + 1) * L].contiguous(), group_size=Hq // Hkv, causal=False, comm=comm))
    o_ref, l_ref = oracle.attention(wl.to_oracle(q), wl.to_oracle(k), wl.to_oracle(v),
                                    1.0 / math.sqrt(d), False)
    for r, (o, l) in enumerate(res):
        compare(o.float().cpu().numpy(), l.cpu().numpy(), o_ref[:, r * hr:(r + 1) * hr],
                l_ref[:, r * hr:(r + 1) * hr], "bf16", f"ring non-causal rank {r}")


def _positions_draws():
    """12 seeded (B, Hq, Hkv, Sq, Skv, d, q_pos0, k_pos0): half of them large enough for the
    pair kernel (many heads), half small (persistent KV-split tiles); the offsets mix rows
    that see no key, some keys and every key."""
    rng = np.random.default_rng(6060)
    out = []
    for i in range(12):
        big = i % 2 == 0
        d = int(rng.choice([64, 128]))
        Hkv = 8 if big else int(rng.choice([1, 2]))
        G = 8 if big else int(rng.choice([1, 2, 4]))
        B = 1 if big else int(rng.integers(1, 3))
        Sq = int(rng.integers(650, 800)) if big else int(rng.integers(1, 400))
        Skv = int(rng.integers(300, 900)) if big else int(rng.integers(1, 500))
        k_pos0 = int(rng.integers(0, 1000))
        # (large draws: at most 100 rows before the first key, so that >= 152 tile pairs remain)
        q_pos0 = k_pos0 + int(rng.integers(-100, 1500)) if big else int(rng.integers(-300, 1500))
        out.append((B, Hkv * G, Hkv, Sq, Skv, d, q_pos0, k_pos0))
    return out


@pytest.mark.parametrize("i", range(12))
def test_positions_random_shapes(i):
    B, Hq, Hkv, Sq, Skv, d, q_pos0, k_pos0 = _positions_draws()[i]
    q, k, v = bf16((B, Hq, Sq, d), 700 + i), bf16((B, Hkv, Skv, d), 800 + i), bf16((B, Hkv, Skv, d), 900 + i)
    scale = d ** -0.5
    o, lse = gb.attn_fwd_positions(q.cuda(), k.cuda(), v.cuda(), q_pos0, k_pos0, scale=scale)
    torch.cuda.synchronize()
    o_ref, l_ref = oracle.attention_at_positions(wl.to_oracle(q), wl.to_oracle(k), wl.to_oracle(v),
                                                 scale, q_pos0, k_pos0)
    compare(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, l_ref, "bf16",
            f"positions b{B} h{Hq}/{Hkv} s{Sq}x{Skv} d{d} q@{q_pos0} k@{k_pos0}")
