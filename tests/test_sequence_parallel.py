"""Sequence-parallel schedules on CPU: the ring-KV prefill and the reduce-to-root decode of
"ADR-0060" sections 5.5 and 4 run as gloo ranks (world sizes 2, 3 and 4), with the kernels
replaced by the fp64 oracle, and must give the single-device result; plus the host-side
schedule rules (ring order, tree shape, head ranges).  The same schedules on the GPU
kernels are checked in test_gpu_sequence_parallel.py."""
import math
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from streaming_attention_flashattention_gb300 import sequence_parallel as sp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


# ---------------------------------------------------------------------------------------
# schedule rules
# ---------------------------------------------------------------------------------------

@pytest.mark.parametrize("world", [1, 2, 3, 4, 7, 8])
def test_ring_schedule_visits_every_slice_once_and_passes_them_on(world):
    for r in range(world):
        sched = sp.ring_schedule(r, world)
        assert sorted(sched) == list(range(world))
        assert sched[0] == r                      # a rank starts on its own slice
        for s in range(1, world):                 # what r holds at s, r - 1 held at s - 1
            assert sched[s] == sp.ring_schedule((r - 1) % world, world)[s - 1]


@pytest.mark.parametrize("world", [1, 2, 3, 5, 8, 9, 16])
def test_binomial_tree_reaches_the_root_in_log_depth(world):
    parent = {c: p for p in range(world) for c in sp.tree_children(p, world)}
    assert sorted(parent) == list(range(1, world))          # every non-root: one parent
    for c, p in parent.items():
        assert sp.tree_parent(c) == p
    depth = max([0] + [bin(c).count("1") for c in range(world)])
    assert depth <= math.ceil(math.log2(world)) if world > 1 else depth == 0
    # a child finishes its own subtree before its parent merges it: children come in
    # increasing subtree size, and every child's subtree is a contiguous block after it
    for p in range(world):
        ch = sp.tree_children(p, world)
        assert ch == sorted(ch)


def test_kv_head_range():
    assert sp.kv_head_range(0, 8, 8) == (0, 1)
    assert sp.kv_head_range(16, 16, 8) == (2, 4)
    assert sp.kv_head_range(4, 4, 8) == (0, 1)        # heads inside one group
    assert sp.kv_head_range(3, 1, 1) == (3, 4)
    with pytest.raises(ValueError):
        sp.kv_head_range(4, 8, 8)                     # straddles two groups, not whole
    with pytest.raises(ValueError):
        sp.kv_head_range(0, 12, 8)


# ---------------------------------------------------------------------------------------
# the schedules over gloo, kernels replaced by the oracle
# ---------------------------------------------------------------------------------------

class OracleBackend:
    """Stand-in for the kernels: fp64 oracle attention, and the section-4 merge on states
    (LSE, 1, O).  Also records which key positions each rank attended to."""

    def __init__(self):
        import oracle
        self.oracle = oracle
        self.k_pos = []

    def attend(self, q, k, v, scale, q_pos0, k_pos0, causal, out=None, lse=None):
        self.k_pos.append(k_pos0)
        qn, kn, vn = q.numpy(), k.contiguous().numpy(), v.contiguous().numpy()
        if causal:
            o, l = self.oracle.attention_at_positions(qn, kn, vn, scale, q_pos0, k_pos0)
        else:
            o, l = self.oracle.attention(qn, kn, vn, scale, False)
        o, l = torch.from_numpy(o), torch.from_numpy(l)
        if out is None:
            return o, l
        out.copy_(o)
        lse.copy_(l)
        return out, lse

    def merge(self, acc, part, final):
        if acc is None:
            return part
        (oa, la), (ob, lb) = acc, part
        la, lb = la.double().numpy(), lb.double().numpy()
        m, l, o = self.oracle.merge(la, np.ones_like(la), oa.double().numpy(),
                                    lb, np.ones_like(lb), ob.double().numpy())
        o, lse = self.oracle.finalize(m, l, o)
        return torch.from_numpy(o), torch.from_numpy(lse)

    def decode(self, q, k, v, kv_lens, scale):
        o, l = self.oracle.attention(q.numpy()[:, :, None, :], k.numpy(), v.numpy(), scale,
                                     False, kv_len=kv_lens.numpy())
        return torch.from_numpy(o[:, :, 0]), torch.from_numpy(l[:, :, 0])

    def payload_dtype(self, merged):
        return torch.float64


def _rnd(shape, seed):
    g = np.random.default_rng(seed)
    return torch.from_numpy(g.standard_normal(shape).astype(np.float32))


# ring prefill cases: (B, Hq, Hkv, L per slice, d, q rows, q_pos0, causal)
RING_CASES = [
    (1, 4, 2, 16, 8, None, 0, True),       # queries over the whole sequence
    (2, 8, 2, 8, 8, None, 0, True),        # B > 1
    (1, 4, 2, 16, 8, 16, 0, True),         # a first chunk: every later slice is skipped
    (1, 4, 2, 16, 8, 10, 20, True),        # a chunk in the middle of the context
    (1, 4, 2, 16, 8, None, 0, False),      # full attention
    (1, 6, 3, 8, 8, None, 0, True),        # three KV heads (whole groups on 3 ranks)
]


def _ring_ok(Hq, Hkv, world):
    """The case splits into whole groups, or heads of one group, per rank."""
    if Hq % world:
        return False
    try:
        for r in range(world):
            sp.kv_head_range(r * (Hq // world), Hq // world, Hq // Hkv)
    except ValueError:
        return False
    return True


def _ring_case_inputs(case, world):
    B, Hq, Hkv, L, d, nq, q_pos0, causal = case
    n = L * world
    nq = n if nq is None else nq
    q = _rnd((B, Hq, nq, d), 1)
    k = _rnd((B, Hkv, n, d), 2)
    v = _rnd((B, Hkv, n, d), 3)
    return q, k, v, q_pos0, causal


# decode cases: (B, Hq, Hkv, Lmax, d, lengths)
DEC_CASES = [
    (2, 4, 2, 48, 8, [48, 7]),
    (3, 8, 1, 30, 16, [0, 29, 30]),
]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from streaming_attention_flashattention_gb300 import sequence_parallel as spw
        res = {}
        for ci, case in enumerate(RING_CASES):
            q, k, v, q_pos0, causal = _ring_case_inputs(case, world)
            Hq, Hkv = q.shape[1], k.shape[1]
            if not _ring_ok(Hq, Hkv, world):
                continue
            hr = Hq // world
            L = k.shape[2] // world
            be = OracleBackend()
            o, l = spw.ring_prefill(q[:, rank * hr:(rank + 1) * hr].contiguous(),
                                    k[:, :, rank * L:(rank + 1) * L].contiguous(),
                                    v[:, :, rank * L:(rank + 1) * L].contiguous(),
                                    group_size=Hq // Hkv, q_pos0=q_pos0, causal=causal,
                                    scale=0.35, backend=be)
            res[("ring", ci)] = (o.numpy(), l.numpy(), sorted(set(be.k_pos)))
        for ci, (B, Hq, Hkv, Lmax, d, lens) in enumerate(DEC_CASES):
            q = _rnd((B, Hq, d), 10)
            k = _rnd((B, Hkv, Lmax, d), 11)
            v = _rnd((B, Hkv, Lmax, d), 12)
            c = -(-Lmax // world)                 # keys per rank block
            ks = torch.zeros((B, Hkv, c, d))
            vs = torch.zeros((B, Hkv, c, d))
            lo, hi = rank * c, min((rank + 1) * c, Lmax)
            if hi > lo:
                ks[:, :, :hi - lo] = k[:, :, lo:hi]
                vs[:, :, :hi - lo] = v[:, :, lo:hi]
            lens_r = torch.tensor([max(0, min(n - lo, c)) for n in lens], dtype=torch.int32)
            root = 1 % world
            o, l = spw.decode_reduce(q, ks, vs, lens_r, root=root, scale=0.3,
                                     backend=OracleBackend())
            res[("dec", ci)] = None if o is None else (o.numpy(), l.numpy())
            # round-robin placement: position t on rank t mod P
            ks = torch.zeros((B, Hkv, c, d))
            vs = torch.zeros((B, Hkv, c, d))
            mine = k[:, :, rank::world]
            ks[:, :, :mine.shape[2]] = mine
            vs[:, :, :mine.shape[2]] = v[:, :, rank::world]
            lens_r = torch.tensor([max(0, -(-(n - rank) // world)) for n in lens], dtype=torch.int32)
            o, l = spw.decode_reduce(q, ks, vs, lens_r, root=root, scale=0.3,
                                     backend=OracleBackend())
            res[("dec_rr", ci)] = None if o is None else (o.numpy(), l.numpy())
        out[rank] = res
    finally:
        dist.destroy_process_group()


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


@pytest.mark.parametrize("world", [2, 3, 4])
def test_schedules_over_gloo_equal_single_device(world):
    import oracle
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world, join=True,
                       start_method="spawn")
    # ring prefill: each rank's heads equal the single-device result
    for ci, case in enumerate(RING_CASES):
        q, k, v, q_pos0, causal = _ring_case_inputs(case, world)
        Hq = q.shape[1]
        if not _ring_ok(Hq, k.shape[1], world):
            continue
        if causal:
            o_ref, l_ref = oracle.attention_at_positions(q.numpy(), k.numpy(), v.numpy(), 0.35,
                                                         q_pos0, 0)
        else:
            o_ref, l_ref = oracle.attention(q.numpy(), k.numpy(), v.numpy(), 0.35, False)
        hr = Hq // world
        L = k.shape[2] // world
        for r in range(world):
            o, l, kpos = out[r][("ring", ci)]
            np.testing.assert_allclose(o, o_ref[:, r * hr:(r + 1) * hr], rtol=0, atol=1e-6)
            np.testing.assert_allclose(l, l_ref[:, r * hr:(r + 1) * hr], rtol=0, atol=1e-6)
            # the causal ring skip: slices wholly after the last query are never attended
            last_q = q_pos0 + q.shape[2] - 1
            want = [s * L for s in range(world) if not causal or s * L <= last_q]
            assert kpos == want
    # decode: the root holds the single-device result, the others nothing
    root = 1 % world
    for ci, (B, Hq, Hkv, Lmax, d, lens) in enumerate(DEC_CASES):
        q = _rnd((B, Hq, d), 10)
        k = _rnd((B, Hkv, Lmax, d), 11)
        v = _rnd((B, Hkv, Lmax, d), 12)
        o_ref, l_ref = oracle.attention(q.numpy()[:, :, None, :], k.numpy(), v.numpy(), 0.3,
                                        False, kv_len=np.array(lens, np.int32))
        for key in ("dec", "dec_rr"):       # contiguous blocks, round-robin tokens
            for r in range(world):
                got = out[r][(key, ci)]
                if r != root:
                    assert got is None
                    continue
                o, l = got
                np.testing.assert_allclose(o, o_ref[:, :, 0], rtol=0, atol=1e-6)
                fin = np.isfinite(l_ref[:, :, 0])
                assert np.array_equal(fin, np.isfinite(l))
                np.testing.assert_allclose(l[fin], l_ref[:, :, 0][fin], rtol=0, atol=1e-6)
