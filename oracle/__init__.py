"""fp64 CPU oracle for streaming attention -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's ``cpu_baseline`` /
``--impl reference`` legs may import this package.  The product path (the C-ABI library
and its Python binding) never imports, links or executes anything here, and nothing here
imports the product.

Pages cited (by title, with their sections):
  [AttnRegion]  "AttentionRegion Transformation - Deriving FlashAttention via
                Memory-Centric Compilation in AICF" -- section 3 (pattern:
                MatMul, Mask, Softmax, MatMul), section 6 (Streaming Attention Region,
                online softmax update of m and l), section 8 (kernel lowering loop).
  [Pipeline]    "AI Compiler pipeline stages" -- IR Normalization (stable softmax
                canonical form exp(x - max x) / sum exp(x - max x)).
  [ADR-0060]    "ADR-0060: AHBM GQA Fused Attention Kernel (Llama3-70B)" -- section 3
                (per-tile op sequence: scale, additive mask, row max, exp, corr, l and O
                updates), section 4 (log-sum-exp merge of partial (m, l, O), final O / l),
                section 5.2 (decode: T_q = 1, every past key visible, G query heads of a
                KV head stacked), section 5.4 (prefill tile classes: past / future /
                partial), section 2.1 (contiguous KV blocks per shard).

Functions:
  attention(...)            plain definition, two-pass stable softmax, fp64 (C, OpenMP)
  attention_probs(...)      the probability matrix P of the same definition (numpy)
  online_attention(...)     the streaming recurrence of [AttnRegion] s.6 / [ADR-0060] s.3
  attention_at_positions(...)  causal attention with explicit query / key positions
                            ([ADR-0060] s.5.4 tile classes on absolute positions, s.5.5 ring
                            steps), via online_attention on one tile per head pair
  merge(...)                [ADR-0060] s.4 merge of two partial states
  split_bounds(...)         contiguous split chunks (reading: [ADR-0060] s.2.1 blocks)
  splitkv_decode(...)       per-split partial states folded with merge()

Every function here is pinned by tests/test_oracle_pins.py against closed forms, a
library routine (torch scaled_dot_product_attention in float64), brute force on tiny
inputs and invariants.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

IN_F32 = 0
IN_BF16 = 1


def build(force: bool = False) -> str:
    """Compile attn_oracle.c into oracle/liboracle.so with gcc + OpenMP."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            lib.oracle_attention.restype = ctypes.c_int
            lib.oracle_attention.argtypes = [
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                ctypes.c_void_p, ctypes.c_void_p,
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.c_void_p, ctypes.c_int, ctypes.c_double, ctypes.c_int,
                ctypes.c_void_p, ctypes.c_longlong, ctypes.c_int,
            ]
            lib.oracle_max_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def _as_input(x: np.ndarray):
    """Accept float32 arrays, or bf16 bit patterns as uint16 arrays."""
    x = np.ascontiguousarray(x)
    if x.dtype == np.float32:
        return x, IN_F32
    if x.dtype == np.uint16:
        return x, IN_BF16
    if x.dtype == np.float64:
        raise TypeError("oracle.attention takes the stored values: float32 or bf16 bits (uint16)")
    raise TypeError(f"unsupported input dtype {x.dtype}")


def attention(q, k, v, scale: float, causal: bool, kv_len=None, rows=None, nthreads: int = 0):
    """O and LSE of softmax(scale * Q K^T + mask) V, plain two-pass definition in fp64.

    q: [B, Hq, Sq, d]; k, v: [B, Hkv, Skv_max, d] (float32 or uint16 bf16 bits).
    kv_len: optional int array [B] of valid keys per batch entry (others never read).
    rows: optional int64 array of flat row ids (b * Hq + h) * Sq + i; when given, the
    outputs hold only those rows (shape [len(rows), d] and [len(rows)]).
    Returns (O float64 [B,Hq,Sq,d] or [n,d], LSE float64 [B,Hq,Sq] or [n]).
    """
    lib = _load()
    q, dt_q = _as_input(q)
    k, dt_k = _as_input(k)
    v, dt_v = _as_input(v)
    if not (dt_q == dt_k == dt_v):
        raise TypeError("q, k, v must share one storage type")
    B, Hq, Sq, d = q.shape
    Bk, Hkv, Skv, dk = k.shape
    if v.shape != k.shape or Bk != B or dk != d:
        raise ValueError("shape mismatch")
    kl = None
    if kv_len is not None:
        kl = np.ascontiguousarray(np.asarray(kv_len, dtype=np.int32))
        if kl.shape != (B,):
            raise ValueError("kv_len must have shape [B]")
    if rows is not None:
        rr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64)).reshape(-1)
        n = rr.shape[0]
        o = np.empty((n, d), dtype=np.float64)
        lse = np.empty((n,), dtype=np.float64)
    else:
        rr = None
        n = B * Hq * Sq
        o = np.empty((B, Hq, Sq, d), dtype=np.float64)
        lse = np.empty((B, Hq, Sq), dtype=np.float64)
    if n == 0:
        return o, lse
    rc = lib.oracle_attention(
        q.ctypes.data, k.ctypes.data, v.ctypes.data, dt_q,
        o.ctypes.data, lse.ctypes.data,
        B, Hq, Hkv, Sq, Skv,
        kl.ctypes.data if kl is not None else None,
        d, float(scale), 1 if causal else 0,
        rr.ctypes.data if rr is not None else None, n, int(nthreads),
    )
    if rc != 0:
        raise ValueError("oracle_attention rejected its arguments")
    return o, lse


# ----------------------------------------------------------------------------------------
# numpy restatements of the pages' algorithm steps (fp64); inputs as float64 arrays.
# ----------------------------------------------------------------------------------------

def widen(x: np.ndarray) -> np.ndarray:
    """Stored values to float64: float32 as is, uint16 taken as bf16 bit patterns."""
    x = np.asarray(x)
    if x.dtype == np.uint16:
        return (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return x.astype(np.float64)


def _visible(Sq: int, Skv: int, causal: bool) -> np.ndarray:
    """Boolean [Sq, Skv]: key j visible from query i (bottom-right causal reading)."""
    if not causal:
        return np.ones((Sq, Skv), dtype=bool)
    i = np.arange(Sq)[:, None]
    j = np.arange(Skv)[None, :]
    return j <= i + (Skv - Sq)


def attention_probs(q: np.ndarray, k: np.ndarray, scale: float, causal: bool) -> np.ndarray:
    """P = softmax(scale * q k^T + mask) for one head pair: q [Sq,d], k [Skv,d] float64.

    The stable canonical form of [Pipeline] (IR Normalization); fully masked rows give 0.
    """
    s = scale * (q @ k.T)
    vis = _visible(q.shape[0], k.shape[0], causal)
    s = np.where(vis, s, -np.inf)
    m = s.max(axis=1, keepdims=True)
    m_safe = np.where(np.isfinite(m), m, 0.0)
    e = np.exp(s - m_safe)
    e = np.where(vis, e, 0.0)
    l = e.sum(axis=1, keepdims=True)
    return np.divide(e, l, out=np.zeros_like(e), where=l > 0)


def online_attention(q, k, v, scale: float, causal: bool, tile: int,
                     key_offset: int = 0, q_pos0: int | None = None):
    """Unnormalised streaming state (m, l, O) for one head pair, KV tile by KV tile.

    Follows [AttnRegion] s.6 and [ADR-0060] s.3 for each KV tile j:
        S_j   = scale * q K_j^T (+ additive -inf mask on invisible keys)
        m_new = max(m, rowmax S_j)
        P     = exp(S_j - m_new);  corr = exp(m - m_new)
        l     = l * corr + rowsum P
        O     = O * corr + P V_j;  m = m_new
    q [Sq,d], k/v [n,d] float64 (keys at global positions key_offset + 0..n-1).
    q_pos0: global position of query row 0 for the causal test (default: the
    bottom-right reading with Skv = key_offset + n).
    Returns (m [Sq], l [Sq], O [Sq,d]) without the final division by l.
    """
    Sq, d = q.shape
    n = k.shape[0]
    if q_pos0 is None:
        q_pos0 = (key_offset + n) - Sq
    m = np.full(Sq, -np.inf)
    l = np.zeros(Sq)
    O = np.zeros((Sq, d))
    qpos = q_pos0 + np.arange(Sq)[:, None]
    for t0 in range(0, n, tile):
        t1 = min(t0 + tile, n)
        Sj = scale * (q @ k[t0:t1].T)
        if causal:
            kpos = key_offset + np.arange(t0, t1)[None, :]
            Sj = np.where(kpos <= qpos, Sj, -np.inf)
        m_new = np.maximum(m, Sj.max(axis=1))
        # rows that have seen no visible key yet keep m = -inf; exp(-inf - -inf) is taken as 0
        base = np.where(np.isfinite(m_new), m_new, 0.0)
        P = np.exp(Sj - base[:, None])
        corr = np.where(np.isfinite(m), np.exp(m - base), 0.0)
        l = l * corr + P.sum(axis=1)
        O = O * corr[:, None] + P @ v[t0:t1]
        m = m_new
    return m, l, O


def finalize(m, l, O):
    """O / l and LSE = m + ln l (rows with l = 0 give O = 0, LSE = -inf); [ADR-0060] s.4."""
    l = np.asarray(l, dtype=np.float64)
    out = np.divide(O, l[..., None], out=np.zeros_like(O), where=l[..., None] > 0)
    with np.errstate(divide="ignore"):
        lse = np.where(l > 0, m + np.log(np.where(l > 0, l, 1.0)), -np.inf)
    return out, lse


def attention_at_positions(q, k, v, scale: float, q_pos0: int, k_pos0: int):
    """Causal attention with explicit positions: query i sits at q_pos0 + i, key j at
    k_pos0 + j, and a query sees the keys whose position is not after its own ([ADR-0060]
    s.5.4 states its tile classes on such absolute positions; s.5.5 folds each ring step's
    KV slice this way).  Per head pair (GQA: query head h reads KV head h // G) the plain
    definition in fp64: the whole key range as one tile of online_attention, then finalize;
    rows that see no key give O = 0, LSE = -inf.

    q [B, Hq, Sq, d], k / v [B, Hkv, Skv, d] stored values (float32 or bf16 bits as uint16).
    Returns (O float64 [B, Hq, Sq, d], LSE float64 [B, Hq, Sq]).
    """
    qf, kf, vf = widen(q), widen(k), widen(v)
    B, Hq, Sq, d = qf.shape
    Hkv, Skv = kf.shape[1], kf.shape[2]
    G = Hq // Hkv
    O = np.zeros((B, Hq, Sq, d))
    L = np.zeros((B, Hq, Sq))
    for b in range(B):
        for h in range(Hq):
            st = online_attention(qf[b, h], kf[b, h // G], vf[b, h // G], scale, True,
                                  max(Skv, 1), key_offset=k_pos0, q_pos0=q_pos0)
            O[b, h], L[b, h] = finalize(*st)
    return O, L


def merge(m_a, l_a, O_a, m_b, l_b, O_b):
    """Log-sum-exp merge of two partial states ([ADR-0060] s.4 merge()).

    m = max(m_a, m_b); s_a = exp(m_a - m); s_b = exp(m_b - m);
    returns (m, l_a s_a + l_b s_b, O_a s_a + O_b s_b).  An empty state (m = -inf, l = 0)
    is the identity.
    """
    m = np.maximum(m_a, m_b)
    base = np.where(np.isfinite(m), m, 0.0)
    sa = np.where(np.isfinite(m_a), np.exp(m_a - base), 0.0)
    sb = np.where(np.isfinite(m_b), np.exp(m_b - base), 0.0)
    return m, l_a * sa + l_b * sb, O_a * sa[..., None] + O_b * sb[..., None]


def split_bounds(length: int, num_splits: int, align: int = 64):
    """Contiguous split chunks [s*C, min((s+1)*C, length)), C = ceil(length/num_splits)
    rounded up to `align` (reading of [ADR-0060] s.2.1: rank r owns [r*B, (r+1)*B)).
    Trailing splits may be empty."""
    if num_splits <= 0:
        raise ValueError("num_splits must be positive")
    c = -(-length // num_splits) if length > 0 else 0
    c = -(-c // align) * align if c > 0 else align
    return [(min(s * c, length), min((s + 1) * c, length)) for s in range(num_splits)]


def splitkv_decode(q, k, v, scale: float, num_splits: int, tile: int = 64, align: int = 64):
    """Split-KV decode for one KV head group ([ADR-0060] s.4 and s.5.2).

    q [G, d] (the group's query heads stacked, T_q = 1), k/v [n, d] float64.
    Each split streams its contiguous chunk with online_attention (no mask: decode sees
    every past key), giving a partial (m_s, l_s, O_s); the partials are folded with
    merge() and normalised once.  Returns (O [G,d], LSE [G], partials list).
    """
    n = k.shape[0]
    G, d = q.shape
    acc = (np.full(G, -np.inf), np.zeros(G), np.zeros((G, d)))
    parts = []
    for a, b in split_bounds(n, num_splits, align):
        if b > a:
            st = online_attention(q, k[a:b], v[a:b], scale, False, tile)
        else:
            st = (np.full(G, -np.inf), np.zeros(G), np.zeros((G, d)))
        parts.append(st)
        acc = merge(*acc, *st)
    O, lse = finalize(*acc)
    return O, lse, parts


def lse_combine(lse_parts: np.ndarray, o_parts: np.ndarray):
    """Combine normalised split results: lse = ln sum_s e^{lse_s}, O = sum_s e^{lse_s - lse} O_s.

    lse_parts [S], o_parts [S, d] (O_s already divided by l_s).  Equivalent to folding
    merge() over states (lse_s, 1, O_s).  Returns (O [d], lse)."""
    lse_parts = np.asarray(lse_parts, dtype=np.float64)
    mx = np.max(lse_parts) if lse_parts.size else -np.inf
    if not np.isfinite(mx):
        return np.zeros(o_parts.shape[-1]), -np.inf
    w = np.exp(lse_parts - mx)
    tot = w.sum()
    return (w[:, None] * o_parts).sum(axis=0) / tot, mx + math.log(tot)
