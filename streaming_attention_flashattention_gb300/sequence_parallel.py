"""Sequence-parallel attention across ranks, one GPU per process.

Two schedules from "ADR-0060: AHBM GQA Fused Attention Kernel (Llama3-70B)":

ring_prefill  -- section 5.5, prefill with the sequence split over the ranks (Ring KV):
    head-parallel.  Rank r owns some query heads (all of their query positions) and KV slice
    r (keys [r L, (r + 1) L) of every KV head).  The P slices travel round the ring: at step
    s rank r holds slice (r - s) mod P, sends it on to rank r + 1 and receives the next one
    from rank r - 1 while it folds the slice it holds into its heads' running result.  The
    fold of one slice is attn_fwd_positions (causal attention at the slice's absolute key
    positions; a slice wholly in the future of every query of the rank is skipped, the
    section's causal ring skip) followed by attn_merge into the running result.  Each rank
    ends with its own heads' final rows; there is no reduction across ranks.

decode_reduce -- section 4, decode with the KV cache split along the sequence (KV-parallel):
    every rank holds the same queries (T_q = 1) and a share of each sequence's keys -- a
    contiguous block (section 2.1), or every P-th token round robin (the section's
    alternative; decode attends to every key, so any disjoint split of the positions gives
    the same result) -- and sweeps it with the split-KV decode kernel into a partial
    (O_r, LSE_r); the partials are combined by reduce-to-root over a static binomial tree
    of depth ceil(log2 P): a node merges its children's partials, in a fixed order, as they arrive
    and sends the result to its parent once its own sweep and its children are done; only
    the root holds the answer (section 4: attention is needed in one place, so not an
    all-reduce).  The merge is section 4's log-sum-exp merge, attn_merge.

Transport is torch.distributed point-to-point (DistComm: NCCL between GPUs; the tests run
the same schedules on CPU over gloo).  Every attention step and merge runs in libgbattn's
kernels through the package binding; `backend` exists so that the schedules can be
exercised on CPU with a stand-in for the kernels, and defaults to the CUDA library (which
raises if it is not built); `comm` takes any object with DistComm's four methods.
"""
from __future__ import annotations

import math

import torch
import torch.distributed as dist


class CudaBackend:
    """The kernel calls the schedules make, on libgbattn (bf16 inputs, fp32 accumulators)."""

    def __init__(self):
        from . import load_library
        load_library()                       # raises if the library is missing

    def attend(self, q, k, v, scale, q_pos0, k_pos0, causal, out=None, lse=None):
        from . import attn_fwd, attn_fwd_positions
        if causal:
            return attn_fwd_positions(q, k, v, q_pos0, k_pos0, scale=scale, out=out, lse=lse)
        return attn_fwd(q, k, v, causal=False, scale=scale, out=out, lse=lse)

    def merge(self, acc, part, final):
        """Fold `part` into `acc` (None: `part` is the first); final: return the result in
        the inputs' dtype (bf16)."""
        from . import attn_merge
        if acc is None:
            return part
        o_a, l_a = acc
        o_b, l_b = part
        if final:
            return attn_merge(o_a, l_a, o_b, l_b, out_dtype=torch.bfloat16)
        if o_a.dtype == torch.float32:       # running fp32 accumulator, merged in place
            return attn_merge(o_a, l_a, o_b, l_b, out=o_a, lse_out=l_a)
        return attn_merge(o_a, l_a, o_b, l_b, out_dtype=torch.float32)

    def decode(self, q, k, v, kv_lens, scale):
        from . import attn_decode_splitkv
        o, lse = attn_decode_splitkv(q.unsqueeze(2), k, v, kv_lens, num_splits=0, scale=scale)
        return o.squeeze(2), lse

    def payload_dtype(self, merged):
        """dtype of a decode partial sent up the tree: the kernel's bf16 O for a leaf, the
        fp32 accumulator once something was merged into it."""
        return torch.float32 if merged else torch.bfloat16


class DistComm:
    """Point-to-point transport over a torch.distributed process group (default: world)."""

    def __init__(self, group=None):
        self.group = group
        self.rank = dist.get_rank(group)
        self.world = dist.get_world_size(group)

    def _peer(self, r):
        """Global rank of member r of the group (P2P ops address global ranks)."""
        return r if self.group is None else dist.get_global_rank(self.group, r)

    def exchange(self, sends, recvs, dst, src):
        """Start sending `sends` to member dst and receiving `recvs` from member src;
        returns the handles to wait on."""
        ops = [dist.P2POp(dist.isend, t, self._peer(dst), self.group) for t in sends]
        ops += [dist.P2POp(dist.irecv, t, self._peer(src), self.group) for t in recvs]
        return dist.batch_isend_irecv(ops)

    def send(self, t, dst):
        dist.send(t, self._peer(dst), group=self.group)

    def recv(self, t, src):
        dist.recv(t, self._peer(src), group=self.group)


def kv_head_range(h0: int, n_heads: int, group_size: int):
    """KV heads [kvh0, kvh1) that query heads [h0, h0 + n_heads) use (GQA: query head h reads
    KV head h // group_size), checked so that the local call keeps a uniform group: whole
    groups, or heads inside one group."""
    if n_heads <= 0 or group_size <= 0:
        raise ValueError("n_heads and group_size must be positive")
    kvh0, kvh1 = h0 // group_size, (h0 + n_heads - 1) // group_size + 1
    whole = h0 % group_size == 0 and n_heads % group_size == 0
    inside = kvh1 - kvh0 == 1
    if not (whole or inside):
        raise ValueError(f"query heads [{h0}, {h0 + n_heads}) split a KV head group of "
                         f"{group_size}: give each rank whole groups or heads of one group")
    return kvh0, kvh1


def ring_schedule(rank: int, world: int):
    """The slice rank `rank` folds at each ring step: (r - s) mod P for s = 0 .. P-1."""
    return [(rank - s) % world for s in range(world)]


def ring_prefill(q, k_slice, v_slice, *, group_size: int, head0: int | None = None,
                 q_pos0: int = 0, causal: bool = True, scale: float | None = None,
                 group=None, comm=None, backend=None):
    """Ring-KV sequence-parallel prefill ("ADR-0060" section 5.5); call on every rank.

    q        [B, Hq_r, S, d]   this rank's query heads [head0, head0 + Hq_r), all positions
                               (query i at position q_pos0 + i)
    k_slice  [B, Hkv, L, d]    KV slice `rank` of every KV head: keys at positions
    v_slice                    [rank L, (rank + 1) L); every rank's slice has the same L
    group_size                 query heads per KV head (GQA)
    head0                      first query head of this rank (default rank * Hq_r)
    Returns (O [B, Hq_r, S, d], LSE [B, Hq_r, S]) for this rank's heads.
    """
    backend = backend or CudaBackend()
    comm = comm or DistComm(group)
    rank, world = comm.rank, comm.world
    B, Hq_r, S, d = q.shape
    Bk, Hkv, L, dk = k_slice.shape
    if v_slice.shape != k_slice.shape or Bk != B or dk != d:
        raise ValueError("k_slice and v_slice must be [B, Hkv, L, d] with q's B and d")
    if head0 is None:
        head0 = rank * Hq_r
    kvh0, kvh1 = kv_head_range(head0, Hq_r, group_size)
    if kvh1 > Hkv:
        raise ValueError("the rank's query heads need KV heads beyond the slice")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    whole = kvh0 == 0 and kvh1 == Hkv

    def skipped(idx):                    # every key of the slice after every query
        return causal and idx * L > q_pos0 + S - 1

    def attend(kk, vv, k_pos0, causal_):
        if whole:
            return backend.attend(q, kk, vv, scale, q_pos0, k_pos0, causal_)
        # the rank's KV heads are a contiguous block of each batch entry's heads: one call per
        # batch entry, each writing its rows of the step's output (O in q's dtype, fp32 LSE)
        out = torch.empty_like(q)
        lse = torch.empty(tuple(q.shape[:3]), dtype=torch.float32, device=q.device)
        for b in range(B):
            backend.attend(q[b:b + 1], kk[b:b + 1, kvh0:kvh1], vv[b:b + 1, kvh0:kvh1], scale,
                           q_pos0, k_pos0, causal_, out=out[b:b + 1], lse=lse[b:b + 1])
        return out, lse

    def fold(kk, vv, idx, acc, last):
        part = attend(kk, vv, idx * L, causal)
        return backend.merge(acc, part, final=last and acc is not None)

    schedule = ring_schedule(rank, world)
    folds = [s for s, idx in enumerate(schedule) if not skipped(idx)]
    cur_k, cur_v = k_slice, v_slice
    nxt_k, nxt_v = torch.empty_like(k_slice), torch.empty_like(v_slice)
    acc = None
    for s, idx in enumerate(schedule):
        reqs = []
        if s + 1 < world:                # pass the held slice on while folding it
            reqs = comm.exchange([cur_k, cur_v], [nxt_k, nxt_v], (rank + 1) % world,
                                 (rank - 1) % world)
        if folds and s in folds:
            acc = fold(cur_k, cur_v, idx, acc, last=s == folds[-1])
        for r in reqs:
            r.wait()
        if s + 1 < world:
            cur_k, nxt_k = nxt_k, cur_k
            cur_v, nxt_v = nxt_v, cur_v
    if acc is None:                      # no key visible to any query of the rank
        acc = attend(k_slice, v_slice, q_pos0 + S, True)
    return acc


def tree_children(rel: int, world: int):
    """Children of relative rank `rel` in the binomial reduce-to-root tree over `world`
    ranks (root 0), in the order their partials are merged: rel + 1, rel + 2, rel + 4, ...
    while the offset is below rel's lowest set bit."""
    out = []
    step = 1
    while rel + step < world and (rel == 0 or step < (rel & -rel)):
        out.append(rel + step)
        step <<= 1
    return out


def tree_parent(rel: int):
    """Parent of relative rank rel > 0: rel with its lowest set bit cleared."""
    return rel - (rel & -rel)


def decode_reduce(q, k_shard, v_shard, kv_lens, *, root: int = 0, scale: float | None = None,
                  group=None, comm=None, backend=None):
    """KV-parallel decode with reduce-to-root ("ADR-0060" section 4); call on every rank.

    q        [B, Hq, d]          the same decode queries on every rank
    k_shard  [B, Hkv, Lmax, d]   this rank's keys of each sequence (a contiguous block, or
    v_shard                      round-robin tokens: any disjoint split of the positions)
                                 in the cache layout of attn_decode_splitkv
    kv_lens  [B] int32           valid keys of the shard per sequence (0 allowed)
    Returns (O [B, Hq, d] bf16, LSE [B, Hq]) on `root`, (None, None) on the other ranks.
    """
    backend = backend or CudaBackend()
    comm = comm or DistComm(group)
    rank, world = comm.rank, comm.world
    if scale is None:
        scale = 1.0 / math.sqrt(q.shape[-1])
    rel = (rank - root) % world
    children = tree_children(rel, world)
    acc = backend.decode(q, k_shard, v_shard, kv_lens, scale)
    merged = False
    for i, c in enumerate(children):
        child_merged = len(tree_children(c, world)) > 0
        o_c = torch.empty(acc[0].shape, dtype=backend.payload_dtype(child_merged),
                          device=acc[0].device)
        l_c = torch.empty_like(acc[1])       # LSE: fp32 at every node
        src = (c + root) % world
        comm.recv(o_c, src)
        comm.recv(l_c, src)
        last = rel == 0 and i + 1 == len(children)
        acc = backend.merge(acc, (o_c, l_c), final=last)
        merged = not last
    if rel != 0:
        dst = (tree_parent(rel) + root) % world
        o, l = acc
        if o.dtype != backend.payload_dtype(merged):
            raise RuntimeError("decode partial has an unexpected dtype for the tree")
        comm.send(o, dst)
        comm.send(l, dst)
        return None, None
    return acc
