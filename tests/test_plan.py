"""Host-side planning of the library calls, pinned without a GPU.

attn_decode_plan / attn_prefill_plan return what a call decides from its sizes alone (the
split count, the kernel, the merge, the prefill work split); the launch code uses the same
functions.  The expected values restate the rules in the header, on a 152-SM GB300.
"""
import pytest

import streaming_attention_flashattention_gb300 as gb

NSM = 152


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from streaming_attention_flashattention_gb300 import build
    build.build()
    gb.load_library()


def dec(B, Hq, Hkv, Tq, L, ns, d=128):
    return gb.attn_decode_plan(B, Hq, Hkv, Tq, L, d, ns, NSM)


def test_llama70b_decode_16_splits():
    # 512 split items would be 3.37 waves on 152 SMs: two pieces per split, 1024 items
    p = dec(4, 64, 8, 1, 32768, 16)
    assert p == {"splits": 16, "kernel": "warp", "merge": "combine_per_group", "items": 1024,
                 "rows_per_kv_head": 8, "combine_lanes": 4, "pieces": 2}


def test_pieces_rule():
    # the smallest piece count giving >= 6 waves or a last wave >= 3/4 full
    assert dec(16, 64, 8, 1, 131072, 0)["pieces"] == 1          # 4096 items, 27 waves
    assert dec(4, 64, 8, 1, 32768, 19)["pieces"] == 1           # 608 items: exactly 4 waves
    assert dec(4, 64, 8, 1, 32768, 8)["pieces"] == 4            # 256 items: 1.7, 3.4, 5.05, 6.7 waves
    assert dec(4, 64, 8, 4, 32768, 16)["pieces"] == 1           # tcgen05 kernel: whole splits
    # one wave: whole splits (and the single-launch merge)
    p = dec(1, 64, 8, 1, 4096, 0)
    assert p["pieces"] == 1 and p["merge"] == "single_launch"
    # pieces keep at least 512 keys: 64 splits of 512 keys are not cut
    assert dec(4, 64, 8, 1, 32768, 64)["pieces"] == 1
    # at most 256 partials per row
    assert dec(2, 64, 8, 1, 200000, 200)["pieces"] == 1


def test_automatic_splits_fill_one_wave():
    # 8 (sequence, KV head) groups: 152 // 8 = 19 splits, capped by 256 keys per split
    assert dec(1, 64, 8, 1, 4096, 0)["splits"] == 16
    assert dec(1, 64, 8, 1, 16384, 0)["splits"] == 19
    # one split per 4096 keys wins when it is larger
    assert dec(1, 64, 8, 1, 131072, 0)["splits"] == 32
    # 64 groups: 152 // 64 = 2
    assert dec(8, 64, 8, 1, 8192, 0)["splits"] == 2
    # 128 groups: the floor is 1, the per-length rule decides
    assert dec(16, 64, 8, 1, 131072, 0)["splits"] == 32
    # fixed counts are kept
    assert dec(1, 64, 8, 1, 4096, 7)["splits"] == 7


def test_single_launch_merge_rule():
    # one wave of work items: the group's last split merges
    assert dec(1, 64, 8, 1, 4096, 0)["merge"] == "single_launch"          # 128 items
    # few groups with long splits: the same
    p = dec(1, 64, 8, 1, 131072, 0)                                       # 8 groups, 4096 keys
    assert p["items"] > NSM and p["merge"] == "single_launch"
    # other single-token calls: the combine merges each group as soon as its partials are
    # counted in: few groups with short splits (512 keys), many groups
    assert dec(1, 64, 8, 1, 32768, 64)["merge"] == "combine_per_group"
    assert dec(4, 64, 8, 1, 32768, 16)["merge"] == "combine_per_group"
    assert dec(16, 64, 8, 1, 131072, 0)["merge"] == "combine_per_group"
    # more than 8 rows per KV head: the combine waits for the whole split grid (9 to 15 rows
    # on the warp-level kernel)
    assert dec(1, 32, 8, 3, 8192, 0)["merge"] == "combine"


def test_kernel_choice_by_rows_per_kv_head():
    assert dec(4, 64, 8, 4, 32768, 16)["kernel"] == "tcgen05"             # 32 rows
    assert dec(2, 32, 2, 1, 8192, 0)["kernel"] == "tcgen05"               # G = 16
    assert dec(4, 64, 8, 2, 32768, 16)["kernel"] == "tcgen05"             # 16 rows
    assert dec(4, 32, 8, 2, 32768, 16)["kernel"] == "warp"                # 8 rows
    # 9 to 15 rows: tcgen05 only with splits of >= 1024 keys
    assert dec(4, 32, 8, 3, 32768, 16)["kernel"] == "tcgen05"             # 12 rows, 2048 keys
    p = dec(1, 32, 8, 3, 8192, 0)                                         # 12 rows, 19 x 431 keys
    assert p["kernel"] == "warp" and p["splits"] == 19
    # the tcgen05 kernel counts its partials per (sequence, KV head, 128-row tile)
    assert dec(1, 64, 8, 4, 4096, 0)["merge"] == "combine_per_group"     # 32 rows
    p = dec(2, 16, 2, 20, 1300, 3)                                        # 160 rows: 2 tiles
    assert p["kernel"] == "tcgen05" and p["merge"] == "combine_per_group"


def test_combine_lanes_cover_every_split():
    for ns, lanes in [(1, 1), (8, 1), (9, 2), (16, 2), (17, 4), (64, 8), (65, 16), (256, 32)]:
        p = dec(64, 64, 8, 1, 300000, ns)
        assert p["combine_lanes"] == lanes and 8 * lanes >= ns


def test_decode_plan_rejects_what_the_call_rejects():
    for args in [(0, 64, 8, 1, 100, 128, 0), (1, 64, 7, 1, 100, 128, 0), (1, 64, 8, 1, 100, 128, 257)]:
        with pytest.raises(gb.GbAttnError) as e:
            gb.attn_decode_plan(*args, NSM)
        assert e.value.status == -1
    with pytest.raises(gb.GbAttnError) as e:
        gb.attn_decode_plan(1, 64, 8, 1, 100, 96, 0, NSM)
    assert e.value.status == -2


def pre(B, Hq, Hkv, Sq, Skv, causal):
    return gb.attn_prefill_plan(B, Hq, Hkv, Sq, Skv, causal, NSM)


def test_prefill_pairs_and_kv_split_mode():
    # Llama3-70B causal prefill: 2048 pairs, heaviest first, one launch
    assert pre(1, 64, 8, 8192, 8192, True) == {"mode": "pairs", "first_launch_ctas": 2048,
                                               "tail_pairs": 0, "q_tiles": 4096}
    # fewer pairs than SMs (128): single Q tiles with their KV range split over a CTA's
    # two slots, on one persistent CTA per SM
    assert pre(2, 8, 2, 2048, 2048, True) == {"mode": "kv_split", "first_launch_ctas": 152,
                                              "tail_pairs": 0, "q_tiles": 256}
    # one pair per SM or more (256): pairs
    assert pre(1, 32, 8, 2048, 2048, True) == {"mode": "pairs", "first_launch_ctas": 256,
                                               "tail_pairs": 0, "q_tiles": 512}
    assert pre(1, 4, 1, 9728, 9728, True)["mode"] == "pairs"        # exactly 152 pairs
    assert pre(1, 4, 1, 9600, 9600, True)["mode"] == "kv_split"     # 150 pairs
    # fewer Q tiles than SMs: one CTA per tile
    assert pre(1, 8, 2, 1024, 1024, True)["first_launch_ctas"] == 64


def test_prefill_tail_for_equal_pairs():
    # a 2048-query chunk after a 16384-key context: 512 near-equal pairs, last wave of 56
    assert pre(1, 64, 8, 2048, 16384, True) == {"mode": "pairs", "first_launch_ctas": 456,
                                                "tail_pairs": 56, "q_tiles": 1024}
    # non-causal, last wave 56 of 152: tail; last wave 112 (more than half): no tail
    assert pre(1, 32, 8, 4096, 4096, False)["tail_pairs"] == 56
    assert pre(1, 64, 8, 4096, 4096, False)["tail_pairs"] == 0
    # causal over the whole context: weights 1..32 tiles, no tail however the waves fall
    assert pre(1, 32, 8, 4096, 4096, True)["tail_pairs"] == 0
    # a last wave that is exactly full: nothing to move
    assert pre(1, 64, 8, 2432, 2432, False)["tail_pairs"] == 0


def test_prefill_plan_rejects_invalid_sizes():
    with pytest.raises(gb.GbAttnError):
        gb.attn_prefill_plan(1, 64, 8, 4096, 2048, True, NSM)      # causal with Sq > Skv
    with pytest.raises(gb.GbAttnError):
        gb.attn_prefill_plan(1, 64, 7, 128, 128, False, NSM)


def test_plan_agrees_with_workspace_size_and_invariants():
    # seeded random sizes: the workspace the caller sizes holds exactly the plan's splits,
    # items are splits x groups of the chosen kernel, lanes cover every split
    import random
    rng = random.Random(2024)
    for _ in range(400):
        Hkv = rng.choice([1, 2, 4, 8])
        G = rng.choice([1, 2, 4, 8, 16])
        B, Tq = rng.randint(1, 24), rng.choice([1, 1, 2, 3, 4, 5, 8, 16, 40])
        L, d = rng.randint(1, 200000), rng.choice([64, 128])
        ns = rng.choice([0, 0, 1, 3, 16, 64, 256])
        p = gb.attn_decode_plan(B, G * Hkv, Hkv, Tq, L, d, ns, NSM)
        rows = B * G * Hkv * Tq * p["splits"] * p["pieces"]
        n_hc = (G * Tq + 7) // 8
        nci = 4 if n_hc >= 3 else n_hc
        n_hg = (n_hc + nci - 1) // nci
        counters = ((1 + B * Hkv * n_hg) * 4 + 255) // 256 * 256
        expect = counters + (rows * 4 + 255) // 256 * 256 + rows * d * 4
        assert gb.attn_decode_workspace_bytes(B, G * Hkv, Hkv, Tq, L, d, ns, NSM) == expect
        assert 1 <= p["splits"] <= 256 and (ns == 0 or p["splits"] == ns)
        per_split = B * Hkv * ((G * Tq + 127) // 128 if p["kernel"] == "tcgen05" else n_hg)
        assert p["items"] == p["splits"] * p["pieces"] * per_split
        assert p["rows_per_kv_head"] == G * Tq
        parts = p["splits"] * p["pieces"]
        assert 1 <= p["pieces"] <= 4 and parts <= 256
        assert p["pieces"] == 1 or L >= 512 * parts
        lanes = p["combine_lanes"]
        assert lanes & (lanes - 1) == 0 and 8 * lanes >= parts and 8 * (lanes // 2) < max(parts, 2)
        if p["merge"] == "single_launch":
            assert p["pieces"] == 1
        if p["merge"] == "combine_per_group":
            # the warp kernel with one row chunk per KV head, or the tcgen05 kernel
            assert (p["kernel"] == "warp" and G * Tq <= 8) or p["kernel"] == "tcgen05"
        if p["kernel"] == "tcgen05":
            assert p["merge"] == "combine_per_group"
        if p["kernel"] == "warp" and G * Tq <= 8:
            assert p["merge"] in ("single_launch", "combine_per_group")
        if p["merge"] == "single_launch":
            assert p["kernel"] == "warp" and G * Tq <= 8
        if G * Tq >= 16:
            assert p["kernel"] == "tcgen05"
        if G * Tq <= 8:
            assert p["kernel"] == "warp"


def test_decode_work_items_do_not_grow_with_the_group_size():
    # GQA reuse ("ADR-0060: AHBM GQA Fused Attention Kernel (Llama3-70B)", §11): a work item
    # reads its split's K and V once for all G query heads of the KV head (all G * T_q rows on
    # the tcgen05 kernel), so the items -- and the K/V bytes read -- are the same for every G
    base = dec(4, 8, 8, 1, 32768, 16)["items"]
    for G in (2, 4, 8):
        assert dec(4, 8 * G, 8, 1, 32768, 16)["items"] == base
    tc = dec(4, 32, 8, 4, 32768, 16)
    assert tc["kernel"] == "tcgen05"
    for G in (8, 16):
        assert dec(4, 8 * G, 8, 4, 32768, 16)["items"] == tc["items"]
