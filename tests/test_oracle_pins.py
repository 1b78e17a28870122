"""Pins for the fp64 CPU oracle: it is checked against things other than itself.

Pins (each fails on a plausible mistake in the oracle -- a dropped term, a wrong sign,
a wrong index or a transposed operand):
  * a hand-worked example with closed-form outputs (tests/golden/worked_example_d2.txt);
  * torch.nn.functional.scaled_dot_product_attention in float64 (a library routine);
  * brute force with pure-Python loops on tiny shapes;
  * closed forms: constant V, Q = 0 (uniform attention), Skv = 1, causal row 0;
  * invariants: probability rows sum to 1, joint K/V row permutation (non-causal),
    GQA head h equals MHA with KV head h / G;
  * the streaming recurrence of "AttentionRegion Transformation" section 6 / "ADR-0060"
    section 3 equals the two-pass definition for several tile sizes;
  * split-KV partial states merged with the log-sum-exp merge of "ADR-0060" section 4
    equal the unsplit result, empty splits included;
  * attention at explicit positions: the bottom-right case equals the C definition, all
    keys visible equals torch SDPA, brute force with positions on tiny shapes, a common
    shift of both positions changes nothing, and two key ranges at their positions merged
    equal the whole range.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rnd(shape, seed, scale=1.0):
    g = np.random.default_rng(seed)
    return (g.standard_normal(shape) * scale).astype(np.float32)


# ---------------------------------------------------------------------------------------
# hand-worked example
# ---------------------------------------------------------------------------------------

def _parse_golden(path):
    vals = {}
    with open(path) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            name, expr = (s.strip() for s in line.split("=", 1))
            vals[name] = expr
    env = {"e": math.e, "r": math.sqrt(math.e), "log": math.log, "sqrt": math.sqrt}

    def mat(s):
        return np.array([[float(x) for x in row.split()] for row in s.split(";")], np.float32)

    def ev(s):
        return [eval(p, {"__builtins__": {}}, env) for p in s.split(",")]

    return vals, mat, ev


@pytest.mark.parametrize("causal", [False, True])
def test_worked_example_closed_form(causal):
    vals, mat, ev = _parse_golden(os.path.join(GOLDEN, "worked_example_d2.txt"))
    q = mat(vals["q"])[None, None]
    k = mat(vals["k"])[None, None]
    v = mat(vals["v"])[None, None]
    o, lse = oracle.attention(q, k, v, float(vals["scale"]), causal)
    tag = "causal" if causal else "noncausal"
    for i in range(2):
        np.testing.assert_allclose(o[0, 0, i], ev(vals[f"{tag}.O{i}"]), rtol=0, atol=1e-14)
        assert abs(lse[0, 0, i] - ev(vals[f"{tag}.L{i}"])[0]) < 1e-14


# ---------------------------------------------------------------------------------------
# library routine: torch SDPA in float64
# ---------------------------------------------------------------------------------------

def sdpa_ref(q, k, v, scale, causal):
    """torch SDPA (float64, CPU) with an explicit bottom-right mask and KV heads repeated."""
    qt = torch.from_numpy(q.astype(np.float64))
    kt = torch.from_numpy(k.astype(np.float64))
    vt = torch.from_numpy(v.astype(np.float64))
    G = q.shape[1] // k.shape[1]
    kt = kt.repeat_interleave(G, dim=1)
    vt = vt.repeat_interleave(G, dim=1)
    Sq, Skv = q.shape[2], k.shape[2]
    mask = None
    if causal:
        i = torch.arange(Sq)[:, None]
        j = torch.arange(Skv)[None, :]
        mask = j <= i + (Skv - Sq)
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask, scale=scale)
    s = scale * (qt @ kt.transpose(-1, -2))
    if mask is not None:
        s = s.masked_fill(~mask, float("-inf"))
    lse = torch.logsumexp(s, dim=-1)
    return o.numpy(), lse.numpy()


@pytest.mark.parametrize("B,Hq,Hkv,Sq,Skv,d,causal", [
    (1, 2, 1, 128, 128, 64, False),
    (2, 4, 2, 33, 70, 16, False),
    (2, 4, 2, 33, 70, 16, True),
    (1, 8, 1, 65, 65, 32, True),
    (1, 3, 3, 1, 200, 8, False),
    (1, 2, 2, 129, 257, 128, True),
])
def test_against_torch_sdpa_float64(B, Hq, Hkv, Sq, Skv, d, causal):
    q = rnd((B, Hq, Sq, d), 1)
    k = rnd((B, Hkv, Skv, d), 2)
    v = rnd((B, Hkv, Skv, d), 3)
    scale = 1.0 / math.sqrt(d)
    o, lse = oracle.attention(q, k, v, scale, causal)
    o_ref, lse_ref = sdpa_ref(q, k, v, scale, causal)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref, rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------------------
# brute force (pure Python loops)
# ---------------------------------------------------------------------------------------

def brute(q, k, v, scale, causal):
    B, Hq, Sq, d = q.shape
    Hkv, Skv = k.shape[1], k.shape[2]
    G = Hq // Hkv
    O = [[[[0.0] * d for _ in range(Sq)] for _ in range(Hq)] for _ in range(B)]
    L = [[[0.0] * Sq for _ in range(Hq)] for _ in range(B)]
    for b in range(B):
        for h in range(Hq):
            kv = h // G
            for i in range(Sq):
                ws = []
                for j in range(Skv):
                    if causal and j > i + Skv - Sq:
                        continue
                    s = sum(float(q[b, h, i, c]) * float(k[b, kv, j, c]) for c in range(d))
                    ws.append((j, scale * s))
                if not ws:
                    L[b][h][i] = -math.inf
                    continue
                mx = max(s for _, s in ws)
                z = sum(math.exp(s - mx) for _, s in ws)
                for c in range(d):
                    O[b][h][i][c] = sum(math.exp(s - mx) / z * float(v[b, kv, j, c]) for j, s in ws)
                L[b][h][i] = mx + math.log(z)
    return np.array(O), np.array(L)


@pytest.mark.parametrize("Sq", [1, 2, 3, 5])
@pytest.mark.parametrize("Skv", [1, 2, 3, 5])
@pytest.mark.parametrize("G", [1, 2])
@pytest.mark.parametrize("causal", [False, True])
def test_brute_force_tiny(Sq, Skv, G, causal):
    d = 3
    q = rnd((1, 2 * G, Sq, d), 10 + Sq)
    k = rnd((1, 2, Skv, d), 20 + Skv)
    v = rnd((1, 2, Skv, d), 30 + Skv)
    o, lse = oracle.attention(q, k, v, 0.7, causal)
    o_b, lse_b = brute(q, k, v, 0.7, causal)
    np.testing.assert_allclose(o, o_b, rtol=0, atol=1e-12)
    assert np.array_equal(np.isinf(lse), np.isinf(lse_b))
    fin = np.isfinite(lse_b)
    np.testing.assert_allclose(lse[fin], lse_b[fin], rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------------------
# closed forms and invariants
# ---------------------------------------------------------------------------------------

@pytest.mark.parametrize("causal", [False, True])
def test_constant_v_gives_constant_o(causal):
    q = rnd((2, 4, 50, 16), 5, 3.0)
    k = rnd((2, 2, 80, 16), 6)
    v = np.full((2, 2, 80, 16), 0.375, np.float32)
    o, _ = oracle.attention(q, k, v, 0.25, causal)
    np.testing.assert_allclose(o, 0.375, rtol=0, atol=1e-13)


def test_causal_row0_is_v0():
    q = rnd((1, 4, 64, 32), 7)
    k = rnd((1, 2, 64, 32), 8)
    v = rnd((1, 2, 64, 32), 9)
    scale = 0.3
    o, lse = oracle.attention(q, k, v, scale, True)
    for h in range(4):
        kv = h // 2
        np.testing.assert_allclose(o[0, h, 0], v[0, kv, 0], rtol=0, atol=1e-15)
        dot = float(np.dot(q[0, h, 0].astype(np.float64), k[0, kv, 0].astype(np.float64)))
        assert abs(lse[0, h, 0] - scale * dot) < 1e-13


@pytest.mark.parametrize("causal,Sq,Skv", [(False, 20, 40), (True, 20, 40), (True, 40, 40)])
def test_zero_q_is_uniform_mean(causal, Sq, Skv):
    q = np.zeros((1, 2, Sq, 8), np.float32)
    k = rnd((1, 1, Skv, 8), 11)
    v = rnd((1, 1, Skv, 8), 12)
    o, lse = oracle.attention(q, k, v, 0.5, causal)
    vv = v[0, 0].astype(np.float64)
    for i in range(Sq):
        n = (i + Skv - Sq + 1) if causal else Skv
        np.testing.assert_allclose(o[0, 1, i], vv[:n].mean(axis=0), rtol=0, atol=1e-13)
        assert abs(lse[0, 1, i] - math.log(n)) < 1e-13


def test_single_key_gives_v0():
    q = rnd((1, 2, 9, 16), 13)
    k = rnd((1, 1, 1, 16), 14)
    v = rnd((1, 1, 1, 16), 15)
    o, lse = oracle.attention(q, k, v, 0.25, False)
    np.testing.assert_array_equal(o[0, 0], np.broadcast_to(v[0, 0, 0].astype(np.float64), (9, 16)))
    np.testing.assert_allclose(lse[0, 0], 0.25 * (q[0, 0].astype(np.float64) @ k[0, 0, 0]), atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_probability_rows_sum_to_one_and_o_is_pv(causal):
    q = rnd((1, 1, 30, 8), 16, 2.0)
    k = rnd((1, 1, 45, 8), 17)
    v = rnd((1, 1, 45, 8), 18)
    P = oracle.attention_probs(oracle.widen(q[0, 0]), oracle.widen(k[0, 0]), 0.4, causal)
    np.testing.assert_allclose(P.sum(axis=1), 1.0, rtol=0, atol=1e-13)
    assert (P >= 0).all()
    o, _ = oracle.attention(q, k, v, 0.4, causal)
    np.testing.assert_allclose(o[0, 0], P @ oracle.widen(v[0, 0]), rtol=0, atol=1e-13)


def test_gqa_equals_mha_with_repeated_kv():
    q = rnd((2, 8, 17, 16), 19)
    k = rnd((2, 2, 33, 16), 20)
    v = rnd((2, 2, 33, 16), 21)
    o, lse = oracle.attention(q, k, v, 0.25, True)
    k_rep = np.repeat(k, 4, axis=1)
    v_rep = np.repeat(v, 4, axis=1)
    o2, lse2 = oracle.attention(q, k_rep, v_rep, 0.25, True)
    np.testing.assert_array_equal(o, o2)
    np.testing.assert_array_equal(lse, lse2)


def test_joint_kv_permutation_invariance_noncausal():
    q = rnd((1, 2, 12, 16), 22)
    k = rnd((1, 1, 50, 16), 23)
    v = rnd((1, 1, 50, 16), 24)
    perm = np.random.default_rng(5).permutation(50)
    o, lse = oracle.attention(q, k, v, 0.3, False)
    o2, lse2 = oracle.attention(q, k[:, :, perm], v[:, :, perm], 0.3, False)
    np.testing.assert_allclose(o, o2, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, lse2, rtol=0, atol=1e-13)


def test_rows_without_visible_keys():
    # causal with Sq > Skv: the first Sq - Skv rows see no key -> O = 0, LSE = -inf
    q = rnd((1, 1, 6, 4), 25)
    k = rnd((1, 1, 3, 4), 26)
    v = rnd((1, 1, 3, 4), 27)
    o, lse = oracle.attention(q, k, v, 1.0, True)
    assert np.all(o[0, 0, :3] == 0) and np.all(np.isneginf(lse[0, 0, :3]))
    assert np.all(np.isfinite(lse[0, 0, 3:]))
    np.testing.assert_allclose(o[0, 0, 3], v[0, 0, 0], atol=1e-15)


def test_bf16_bits_widen_exactly():
    x = torch.randn(1, 2, 40, 16, generator=torch.Generator().manual_seed(3)).to(torch.bfloat16)
    kx = torch.randn(1, 1, 40, 16, generator=torch.Generator().manual_seed(4)).to(torch.bfloat16)
    vx = torch.randn(1, 1, 40, 16, generator=torch.Generator().manual_seed(5)).to(torch.bfloat16)
    bits = lambda t: t.view(torch.int16).numpy().view(np.uint16)
    o1, l1 = oracle.attention(bits(x), bits(kx), bits(vx), 0.25, True)
    o2, l2 = oracle.attention(x.float().numpy(), kx.float().numpy(), vx.float().numpy(), 0.25, True)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)
    np.testing.assert_array_equal(oracle.widen(bits(x)), x.double().numpy())


def test_row_subset_matches_full():
    q = rnd((2, 4, 19, 8), 28)
    k = rnd((2, 2, 23, 8), 29)
    v = rnd((2, 2, 23, 8), 30)
    o, lse = oracle.attention(q, k, v, 0.5, True)
    rows = np.array([0, 5, 18, 19, 77, 2 * 4 * 19 - 1])
    o_s, lse_s = oracle.attention(q, k, v, 0.5, True, rows=rows)
    np.testing.assert_array_equal(o_s, o.reshape(-1, 8)[rows])
    np.testing.assert_array_equal(lse_s, lse.reshape(-1)[rows])


def test_kv_len_limits_keys_and_ignores_padding():
    q = rnd((3, 2, 1, 8), 31)
    k = rnd((3, 1, 40, 8), 32)
    v = rnd((3, 1, 40, 8), 33)
    lens = np.array([40, 7, 1], np.int32)
    kp, vp = k.copy(), v.copy()
    for b, n in enumerate(lens):
        kp[b, :, n:] = np.nan
        vp[b, :, n:] = np.nan
    o, lse = oracle.attention(qq := q, kp, vp, 0.5, False, kv_len=lens)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))
    for b, n in enumerate(lens):
        o_b, lse_b = oracle.attention(qq[b:b + 1], k[b:b + 1, :, :n], v[b:b + 1, :, :n], 0.5, False)
        np.testing.assert_array_equal(o[b], o_b[0])
        np.testing.assert_array_equal(lse[b], lse_b[0])


# ---------------------------------------------------------------------------------------
# streaming recurrence and split-KV merge
# ---------------------------------------------------------------------------------------

@pytest.mark.parametrize("tile", [1, 7, 64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_online_recurrence_equals_two_pass(tile, causal):
    q = rnd((1, 1, 37, 16), 40, 2.0)
    k = rnd((1, 1, 150, 16), 41)
    v = rnd((1, 1, 150, 16), 42)
    o, lse = oracle.attention(q, k, v, 0.25, causal)
    st = oracle.online_attention(oracle.widen(q[0, 0]), oracle.widen(k[0, 0]),
                                 oracle.widen(v[0, 0]), 0.25, causal, tile)
    o2, lse2 = oracle.finalize(*st)
    np.testing.assert_allclose(o2, o[0, 0], rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse2, lse[0, 0], rtol=0, atol=1e-12)


@pytest.mark.parametrize("n", [1, 63, 64, 65, 1000])
@pytest.mark.parametrize("num_splits", [1, 2, 3, 16, 64])
def test_splitkv_merge_equals_unsplit(n, num_splits):
    G, d = 8, 32
    q = rnd((1, G, 1, d), 50 + n)
    k = rnd((1, 1, n, d), 51 + n)
    v = rnd((1, 1, n, d), 52 + n)
    o, lse = oracle.attention(q, k, v, 1 / math.sqrt(d), False)
    o2, lse2, parts = oracle.splitkv_decode(oracle.widen(q[0, :, 0]), oracle.widen(k[0, 0]),
                                            oracle.widen(v[0, 0]), 1 / math.sqrt(d), num_splits)
    assert len(parts) == num_splits
    np.testing.assert_allclose(o2, o[0, :, 0], rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse2, lse[0, :, 0], rtol=0, atol=1e-12)
    # the normalised-partials form of the merge (what a combine step receives) agrees too
    lse_p = np.stack([oracle.finalize(*p)[1] for p in parts], axis=1)   # [G, S]
    o_p = np.stack([oracle.finalize(*p)[0] for p in parts], axis=1)     # [G, S, d]
    for g in range(G):
        og, lg = oracle.lse_combine(lse_p[g], o_p[g])
        np.testing.assert_allclose(og, o[0, g, 0], rtol=0, atol=1e-12)
        assert abs(lg - lse[0, g, 0]) < 1e-12


@pytest.mark.parametrize("n", [0, 1, 64, 100, 4096, 131072])
@pytest.mark.parametrize("num_splits", [1, 5, 16, 64])
def test_split_bounds_cover_every_key_once(n, num_splits):
    b = oracle.split_bounds(n, num_splits)
    assert len(b) == num_splits
    cover = np.zeros(n, np.int64)
    for lo, hi in b:
        assert 0 <= lo <= hi <= n
        cover[lo:hi] += 1
        if hi > lo and hi < n:
            assert (hi - lo) % 64 == 0
    assert np.all(cover == 1)
    assert [lo for lo, _ in b] == sorted(lo for lo, _ in b)


def test_merge_is_commutative_and_associative():
    rng = np.random.default_rng(9)
    sts = []
    for _ in range(3):
        m = rng.standard_normal(4) * 3
        l = rng.random(4) + 0.5
        O = rng.standard_normal((4, 6))
        sts.append((m, l, O))
    ab = oracle.merge(*sts[0], *sts[1])
    ba = oracle.merge(*sts[1], *sts[0])
    for x, y in zip(ab, ba):
        np.testing.assert_allclose(x, y, atol=1e-14)
    left = oracle.merge(*ab, *sts[2])
    right = oracle.merge(*sts[0], *oracle.merge(*sts[1], *sts[2]))
    for x, y in zip(oracle.finalize(*left), oracle.finalize(*right)):
        np.testing.assert_allclose(x, y, atol=1e-13)
    empty = (np.full(4, -np.inf), np.zeros(4), np.zeros((4, 6)))
    for x, y in zip(oracle.merge(*sts[0], *empty), sts[0]):
        np.testing.assert_allclose(x, y, atol=0)


# ---------------------------------------------------------------------------------------
# the pins catch planted mistakes (mistakes are planted in a copy of the oracle, on CPU)
# ---------------------------------------------------------------------------------------

def test_planted_missing_correction_is_caught():
    """Dropping the corr rescale of O in the recurrence breaks the online == two-pass pin."""
    q = rnd((1, 1, 16, 8), 60, 2.0)
    k = rnd((1, 1, 64, 8), 61)
    v = rnd((1, 1, 64, 8), 62)
    o, _ = oracle.attention(q, k, v, 0.5, False)
    qf, kf, vf = (oracle.widen(x[0, 0]) for x in (q, k, v))
    m = np.full(16, -np.inf); l = np.zeros(16); O = np.zeros((16, 8))
    for t0 in range(0, 64, 8):
        Sj = 0.5 * qf @ kf[t0:t0 + 8].T
        m_new = np.maximum(m, Sj.max(axis=1))
        P = np.exp(Sj - m_new[:, None])
        corr = np.where(np.isfinite(m), np.exp(m - m_new), 0.0)
        l = l * corr + P.sum(axis=1)
        O = O + P @ vf[t0:t0 + 8]          # planted: O is not rescaled by corr
        m = m_new
    assert np.max(np.abs(O / l[:, None] - o[0, 0])) > 1e-3


def test_planted_transposed_operand_is_caught():
    """Using K^T where V belongs (a transposed/wrong operand) breaks the worked example."""
    vals, mat, ev = _parse_golden(os.path.join(GOLDEN, "worked_example_d2.txt"))
    q = mat(vals["q"])[None, None]
    k = mat(vals["k"])[None, None]
    o_bad, _ = oracle.attention(q, k, k, 0.5, False)
    assert np.max(np.abs(o_bad[0, 0, 0] - ev(vals["noncausal.O0"]))) > 1e-2


# ---------------------------------------------------------------------------------------
# attention at explicit positions
# ---------------------------------------------------------------------------------------

def brute_positions(q, k, v, scale, q_pos0, k_pos0):
    B, Hq, Sq, d = q.shape
    Hkv, Skv = k.shape[1], k.shape[2]
    G = Hq // Hkv
    O = np.zeros((B, Hq, Sq, d))
    L = np.full((B, Hq, Sq), -math.inf)
    for b in range(B):
        for h in range(Hq):
            for i in range(Sq):
                ws = [(j, scale * sum(float(q[b, h, i, c]) * float(k[b, h // G, j, c])
                                      for c in range(d)))
                      for j in range(Skv) if k_pos0 + j <= q_pos0 + i]
                if not ws:
                    continue
                mx = max(s for _, s in ws)
                z = sum(math.exp(s - mx) for _, s in ws)
                for c in range(d):
                    O[b, h, i, c] = sum(math.exp(s - mx) / z * float(v[b, h // G, j, c])
                                        for j, s in ws)
                L[b, h, i] = mx + math.log(z)
    return O, L


@pytest.mark.parametrize("q_pos0,k_pos0", [(0, 0), (4, 0), (0, 3), (2, 5), (-3, -1),
                                           (10, 0), (0, 10), (7, 7)])
def test_positions_brute_force_tiny(q_pos0, k_pos0):
    q = rnd((1, 4, 5, 3), 90)
    k = rnd((1, 2, 6, 3), 91)
    v = rnd((1, 2, 6, 3), 92)
    o, lse = oracle.attention_at_positions(q, k, v, 0.6, q_pos0, k_pos0)
    o_b, lse_b = brute_positions(q, k, v, 0.6, q_pos0, k_pos0)
    np.testing.assert_allclose(o, o_b, rtol=0, atol=1e-12)
    assert np.array_equal(np.isinf(lse), np.isinf(lse_b))
    fin = np.isfinite(lse_b)
    np.testing.assert_allclose(lse[fin], lse_b[fin], rtol=0, atol=1e-12)


@pytest.mark.parametrize("Sq,Skv", [(37, 80), (80, 80), (1, 9)])
def test_positions_bottom_right_equals_c_definition(Sq, Skv):
    q = rnd((2, 4, Sq, 16), 93)
    k = rnd((2, 2, Skv, 16), 94)
    v = rnd((2, 2, Skv, 16), 95)
    o, lse = oracle.attention(q, k, v, 0.3, True)
    for shift in (0, 1000):
        o2, lse2 = oracle.attention_at_positions(q, k, v, 0.3, Skv - Sq + shift, shift)
        np.testing.assert_allclose(o2, o, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse2, lse, rtol=0, atol=1e-12)


def test_positions_all_visible_equals_sdpa_noncausal():
    q = rnd((1, 4, 33, 16), 96)
    k = rnd((1, 2, 50, 16), 97)
    v = rnd((1, 2, 50, 16), 98)
    o_ref, lse_ref = sdpa_ref(q, k, v, 0.25, False)
    o, lse = oracle.attention_at_positions(q, k, v, 0.25, 49, 0)     # row 0 already sees all
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref, rtol=0, atol=1e-12)


def test_positions_no_visible_key():
    q = rnd((1, 2, 10, 8), 99)
    k = rnd((1, 1, 12, 8), 100)
    v = rnd((1, 1, 12, 8), 101)
    o, lse = oracle.attention_at_positions(q, k, v, 0.5, 0, 10)      # keys start after row 9
    assert np.all(o == 0) and np.all(np.isneginf(lse))


@pytest.mark.parametrize("cut", [1, 40, 64, 99])
def test_positions_key_ranges_merge_to_whole(cut):
    """Keys [0, cut) and [cut, n) at their own positions, merged with the section-4 merge,
    equal the whole range: what a ring step and attn_merge compute."""
    Sq, n, d = 30, 100, 16
    q = rnd((1, 2, Sq, d), 102)
    k = rnd((1, 1, n, d), 103)
    v = rnd((1, 1, n, d), 104)
    qp = 70                                   # queries at positions 70 .. 99
    o, lse = oracle.attention_at_positions(q, k, v, 0.2, qp, 0)
    oa, la = oracle.attention_at_positions(q, k[:, :, :cut], v[:, :, :cut], 0.2, qp, 0)
    ob, lb = oracle.attention_at_positions(q, k[:, :, cut:], v[:, :, cut:], 0.2, qp, cut)
    m, l, om = oracle.merge(la, np.ones_like(la), oa, lb, np.ones_like(lb), ob)
    o2, lse2 = oracle.finalize(m, l, om)
    np.testing.assert_allclose(o2, o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse2, lse, rtol=0, atol=1e-12)
