// prefill_tcgen05.cu -- bf16 streaming attention forward on the 5th-generation tensor
// cores (tcgen05.mma with TMEM accumulators), fed by TMA.
//
// What it computes follows "AttentionRegion Transformation - Deriving FlashAttention via
// Memory-Centric Compilation in AICF", section 8 (a resident Q tile, an inner loop over
// K/V tiles, the score tile never written to memory) with the per-tile operation sequence
// of "ADR-0060: AHBM GQA Fused Attention Kernel (Llama3-70B)", section 3 (scale, additive
// causal mask, row max, exp, corr = exp(m_old - m_new), l and O updates) and the tile
// classes of section 5.4 (KV tiles wholly in a query tile's future are skipped, tiles
// crossing the diagonal are masked, past tiles run unmasked).
//
// GB300 mapping (one CTA per pair of 128-row Q tiles that share a KV head):
//   warp 0      TMA producer: Q tiles once, then K and V tiles (128 keys x d, 128-byte
//               swizzle) into two 2-slot rings with full/empty mbarriers;
//   warp 1      TMEM owner and MMA issuer (one thread): S_t = Q_t K^T (both operands
//               K-major in shared memory) and O_t += P_t V (P from TMEM, V MN-major in
//               shared memory), completions signalled with tcgen05.commit;
//   warps 4-7   softmax warpgroup of Q tile 0, warps 8-11 of Q tile 1: one query row per
//               thread (TMEM lane), row max and sum without shuffles, exp2 with the scale
//               folded into one FMA, P (bf16) written back over S in TMEM, and the O
//               correction (a TMEM read-modify-write) only when the row max moves by
//               more than 2^8 -- a stale max is exact because O and l share it.
// TMEM: S0 | S1 | O0 | O1 (128 + 128 + d + d columns of 512).
//
// GQA head packing: the two Q tiles of a CTA are consecutive entries of the list
// (b, kv head, q block, head in group), so for G >= 2 they are two query heads of one KV
// head at the same query block and share every K/V tile and the same causal extent.
//
// KV-split instance (kSplit): the Q tiles of a pair-mode call's last, partly filled wave,
// launched behind the pair grid as a programmatic dependent.  A CTA takes ONE Q tile and
// gives its two ping-pong slots the two halves of that tile's KV range, [0, n0) and
// [n0, n).  Each slot keeps its own (m, l, O); at the end the two states are merged
// inside the CTA with the log-sum-exp rule of "ADR-0060" section 4 (slot 1's O goes
// through shared memory).  The K ring gets a third slot (the unused second Q buffer)
// because each K/V tile now feeds one S/PV pair instead of two.  (Calls too small for
// pairs run the same split on persistent CTAs: prefill_persist.cu.)
#include "common.cuh"
#include "kernels.h"

namespace gbattn {

namespace {

constexpr int kBlockM = 128;              // query rows per Q tile
constexpr int kBlockN = 128;              // keys per K/V tile
constexpr int kThreads = 12 * 32;
constexpr int kSoftmaxWarp0 = 4;          // warps 4..7 -> tile 0, 8..11 -> tile 1
constexpr float kRescaleThreshold = 8.0f; // log2 units: rescale O only if max grows > 2^8
static_assert(kBlockN == 128, "the softmax row reductions assume 128 columns");
#ifdef GBATTN_DEBUG_CHECKS
// Test hook of the debug build: CTA 0 of the grid does not issue the K fill with this index
// (counted over the CTA's fills; -1: none).  The fill's barrier then never completes, the wait
// for it runs out after its time limit and records its code in the error word, and every role
// of every CTA leaves through its give-up exit.  Set by attn_debug_skip_fill.
__device__ int g_skip_k_fill = -1;
#endif

template <int D>
struct PLayout {
    static constexpr int kBoxes = D / 64;
    static constexpr int kTileBytes = kBlockM * D * 2;      // Q, K or V tile
    static constexpr int kBoxBytes = kBlockM * 128;          // one 64-column swizzled box
    static constexpr int kQ0 = 0;
    static constexpr int kK0 = 2 * kTileBytes;               // 2 K slots
    static constexpr int kV0 = 4 * kTileBytes;               // 2 V slots
    static constexpr int kBar = 6 * kTileBytes;
    static constexpr int kNumBars = 18;
    static constexpr int kXm = kBar + kNumBars * 8;          // split merge: m, l [2 slot][128]
    static constexpr int kTmemSlot = kXm + 4 * 128 * 4;
    static constexpr int kOStride = 129;                     // split merge: slot 1's O in the rings
    static constexpr int kBytes = kTmemSlot + 16;
    static constexpr int kAlloc = kBytes + 1024;
    static constexpr uint32_t kColS0 = 0, kColS1 = 128;
    static constexpr uint32_t kColO0 = 256, kColO1 = 256 + D;
    static constexpr uint32_t kTmemCols = 512;
};

struct TileDesc {
    int present;
    int h;        // query head
    int q0;       // first query row
    int n_kv;     // KV tiles to visit
    int kv0;      // first KV tile (KV-split mode: the second half starts at n0)
};

__device__ __forceinline__ int kv_tiles_of(const PrefillParams& p, int q0) {
    if (!p.causal) return (p.Skv + kBlockN - 1) / kBlockN;
    const int last_row = min(q0 + kBlockM, p.Sq) - 1;
    const int keys = min(p.Skv, last_row + p.diag + 1);
    return (keys + kBlockN - 1) / kBlockN;
}

__device__ __forceinline__ void pair_tiles(const PrefillParams& p, int rank, int& b, int& kvh,
                                           TileDesc (&t)[2]);

// KV-split mode over the last pairs of a pair-mode call: item `rank` is Q tile rank % 2 of
// pair tail0 + rank / 2; slot 0 takes KV tiles [0, n0), slot 1 takes [n0, n).
__device__ __forceinline__ void tail_tiles(const PrefillParams& p, int rank, int& b, int& kvh,
                                           TileDesc (&t)[2]) {
    TileDesc pt[2];
    pair_tiles(p, p.tail0 + rank / 2, b, kvh, pt);
    const TileDesc me = (rank & 1) ? pt[1] : pt[0];
    const int n0 = (me.n_kv + 1) / 2;
    t[0] = me; t[0].n_kv = n0; t[0].kv0 = 0;
    t[1] = me; t[1].present = me.present && me.n_kv - n0 > 0; t[1].n_kv = me.n_kv - n0; t[1].kv0 = n0;
}

__device__ __forceinline__ void pair_tiles(const PrefillParams& p, int rank, int& b, int& kvh,
                                           TileDesc (&t)[2]) {
    const int n_groups = p.B * p.Hkv;
    const int cnt = p.n_qblk * p.G;                 // Q tiles per (b, kv head)
    const int pairs_per_group = (cnt + 1) / 2;
    // heaviest pairs first: descending pair index within a group, groups interleaved
    const int jj = pairs_per_group - 1 - rank / n_groups;
    const int grp = rank % n_groups;
    b = grp / p.Hkv;
    kvh = grp % p.Hkv;
    #pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int u = 2 * jj + i;
        t[i].present = u < cnt;
        const int qb = u / p.G, gi = u % p.G;
        t[i].h = kvh * p.G + gi;
        t[i].q0 = p.row0 + qb * kBlockM;
        t[i].n_kv = t[i].present ? kv_tiles_of(p, t[i].q0) : 0;
        t[i].kv0 = 0;
    }
}

// kSplit: the KV-split tail launch of a pair-mode call (its last pairs' Q tiles)
template <int D, bool kSplit>
__global__ void __launch_bounds__(kThreads, 1)
prefill_fwd_kernel(const __grid_constant__ PrefillParams p) {
    constexpr int KS = kSplit ? 3 : 2;   // K ring slots
    using L = PLayout<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBar);
    uint64_t* q_full = bars + 0;
    uint64_t* k_full = bars + 1;     // [KS]
    uint64_t* k_empty = bars + 4;    // [KS]
    uint64_t* v_full = bars + 7;     // [2]
    uint64_t* v_empty = bars + 9;    // [2]
    uint64_t* s_full = bars + 11;    // [2] per slot
    uint64_t* p_ready = bars + 13;   // [2] per slot
    uint64_t* o_done = bars + 15;    // [2] per slot
    uint64_t* merge_bar = bars + 17; // KV-split mode: the two softmax warpgroups meet
    float* xm = reinterpret_cast<float*>(smem + L::kXm);   // [2][128] m, then [2][128] l
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kTmemSlot);
    uint64_t* mma_idle = reinterpret_cast<uint64_t*>(smem + L::kTmemSlot + 8);  // error exit

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    int b, kvh;
    TileDesc td[2];
    if constexpr (kSplit) {
        tail_tiles(p, blockIdx.x, b, kvh, td);
        if (!td[0].present) return;          // the absent second tile of an odd last pair
    } else {
        pair_tiles(p, blockIdx.x, b, kvh, td);
        // a KV-split launch of the last pairs may start on SMs this grid leaves free
        if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    }
    const int n_kv_max = max(td[0].n_kv, td[1].n_kv);
    // the first K/V fill (the one the producer loop below starts with) exists: it goes out
    // before the block barrier, with Q
    const bool early_kv = kSplit ? td[0].n_kv > 0 : n_kv_max > 0;
    // K ring slot of fill f: with KV split, slot 0 is the unused second Q buffer
    auto k_slot = [&](uint32_t f) -> uint8_t* {
        const uint32_t ks = f % KS;
        if constexpr (kSplit) return ks == 0 ? smem + L::kQ0 + L::kTileBytes
                                             : smem + L::kK0 + (ks - 1) * L::kTileBytes;
        else return smem + L::kK0 + ks * L::kTileBytes;
    };

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        for (int i = 0; i < KS; ++i) {
            mbar_init(&k_full[i], 1);
            mbar_init(&k_empty[i], 1);
        }
        mbar_init(merge_bar, 8);
        mbar_init(mma_idle, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&v_full[i], 1);
            mbar_init(&v_empty[i], 1);
            mbar_init(&s_full[i], 1);
            mbar_init(&p_ready[i], 4);
            mbar_init(&o_done[i], 1);
        }
        fence_barrier_init();
        // Q and the first K and V tiles go out now, under the TMEM allocation and the block
        // barrier (this thread initialised the barriers they complete on)
        const int nq = kSplit ? 1 : (td[1].present ? 2 : 1);
        mbar_arrive_expect_tx(q_full, nq * L::kTileBytes);
        #pragma unroll
        for (int t = 0; t < 2; ++t) {
            if (t >= nq) continue;
            #pragma unroll
            for (int bx = 0; bx < L::kBoxes; ++bx)
                tma_load_3d(smem + L::kQ0 + t * L::kTileBytes + bx * L::kBoxBytes, &p.tmap_q,
                            bx * 64, td[t].q0, b * p.Hq + td[t].h, q_full);
        }
        if (early_kv) {
            const int tile0 = kSplit ? td[0].kv0 : 0;
            mbar_arrive_expect_tx(&k_full[0], L::kTileBytes);
            #pragma unroll
            for (int bx = 0; bx < L::kBoxes; ++bx)
                tma_load_3d(k_slot(0) + bx * L::kBoxBytes, &p.tmap_k, bx * 64, tile0 * kBlockN,
                            b * p.Hkv + kvh, &k_full[0]);
            mbar_arrive_expect_tx(&v_full[0], L::kTileBytes);
            #pragma unroll
            for (int bx = 0; bx < L::kBoxes; ++bx)
                tma_load_3d(smem + L::kV0 + bx * L::kBoxBytes, &p.tmap_v, bx * 64, tile0 * kBlockN,
                            b * p.Hkv + kvh, &v_full[0]);
        }
    }
    if (warp == 1) tmem_alloc(tmem_slot, L::kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ================================ TMA producer ================================
        if (lane == 0) {
            prefetch_tensormap(&p.tmap_q);
            prefetch_tensormap(&p.tmap_k);
            prefetch_tensormap(&p.tmap_v);
            // (Q -- one tile per slot for pairs, one for both slots with KV split -- and the
            // first K and V tiles went out before the block barrier)
            // K/V fills in the order the MMA issuer consumes them: one per KV step for
            // pairs (shared by both slots), slot 0 then slot 1 per step with KV split
            const int zkv = b * p.Hkv + kvh;
            uint32_t nf = 0, nfv = 0;
            bool ok = true;
#ifdef GBATTN_DEBUG_CHECKS
            uint32_t skipped = 0xffffffffu;   // the fill the test hook left out
#endif
            for (int j = 0; j < n_kv_max && ok; ++j) {
                #pragma unroll
                for (int t = 0; t < 2; ++t) {
                    if (!kSplit && t == 1) break;
                    if (kSplit && j >= td[t].n_kv) continue;
                    const int tile = kSplit ? td[t].kv0 + j : j;
                    if (nf == 0 && early_kv) {   // fill 0 of K and V went out before the barrier
                        ++nf;
                        ++nfv;
                        continue;
                    }
                    const uint32_t ks = nf % KS, kph = (nf / KS) & 1;
                    if (!mbar_wait(&k_empty[ks], kph ^ 1u, kErrWaitProducer, p.err)) { ok = false; break; }
#ifdef GBATTN_DEBUG_CHECKS
                    if (blockIdx.x == 0 && (int)nf == g_skip_k_fill) {
                        skipped = nf;
                    } else
#endif
                    {
                        mbar_arrive_expect_tx(&k_full[ks], L::kTileBytes);
                        #pragma unroll
                        for (int bx = 0; bx < L::kBoxes; ++bx)
                            tma_load_3d(k_slot(nf) + bx * L::kBoxBytes, &p.tmap_k, bx * 64,
                                        tile * kBlockN, zkv, &k_full[ks]);
                    }
                    ++nf;
                    const uint32_t vs = nfv & 1, vph = (nfv >> 1) & 1;
                    if (!mbar_wait(&v_empty[vs], vph ^ 1u, kErrWaitProducer, p.err)) { ok = false; break; }
                    mbar_arrive_expect_tx(&v_full[vs], L::kTileBytes);
                    #pragma unroll
                    for (int bx = 0; bx < L::kBoxes; ++bx)
                        tma_load_3d(smem + L::kV0 + vs * L::kTileBytes + bx * L::kBoxBytes,
                                    &p.tmap_v, bx * 64, tile * kBlockN, zkv, &v_full[vs]);
                    ++nfv;
                }
            }
            // drain: the last fills of each slot must land before the CTA can exit
            mbar_wait_drain(q_full, 0, p.err);
            for (uint32_t f = nf >= (uint32_t)KS ? nf - KS : 0; f < nf; ++f) {
#ifdef GBATTN_DEBUG_CHECKS
                if (f == skipped) continue;
#endif
                mbar_wait_drain(&k_full[f % KS], (f / KS) & 1, p.err);
            }
            for (uint32_t f = nfv >= 2 ? nfv - 2 : 0; f < nfv; ++f)
                mbar_wait_drain(&v_full[f & 1], (f >> 1) & 1, p.err);
        }
    } else if (warp == 1) {
        // ================================= MMA issuer =================================
        // Tensor-pipe order (ping-pong between the two Q tiles):
        //   S0(0) S1(0) | PV0(0) S0(1) PV1(0) S1(1) | PV0(1) S0(2) PV1(1) S1(2) | ...
        // While softmax 0 works on S0(j+1) the pipe runs PV1(j) and S1(j+1), and the other
        // way round, so neither softmax leaves the tensor cores idle.  S_t(j+1) overwrites
        // P_t(j) in TMEM; it is issued after PV_t(j), and tcgen05.mma executes in order.
        if (lane == 0) {
            constexpr uint32_t idesc_s = make_idesc_bf16(kBlockM, kBlockN, 0, 0);
            constexpr uint32_t idesc_pv = make_idesc_bf16(kBlockM, D, 0, 1);
            const uint32_t q_base = smem_u32(smem + L::kQ0);
            const uint32_t v_base = smem_u32(smem + L::kV0);
            const int n0 = td[0].n_kv, n1 = td[1].n_kv;

            // Operand descriptors are built once; the start-address field (bits 0-13, in
            // 16-byte units) then advances by a constant per K=16 step, so issuing an MMA
            // costs one add.  Shared addresses stay below 2^18, so the field cannot carry.
            // (kept in registers: selected with ternaries, never indexed at run time)
            const uint64_t dq0 = make_sdesc_sw128(q_base, 16, 1024);
            const uint64_t dq1 = make_sdesc_sw128(q_base + L::kTileBytes, 16, 1024);
            const uint64_t dv0 = make_sdesc_sw128(v_base, L::kBoxBytes, 1024);
            const uint64_t dv1 = make_sdesc_sw128(v_base + L::kTileBytes, L::kBoxBytes, 1024);
            const uint64_t dk0 = make_sdesc_sw128(smem_u32(k_slot(0)), 16, 1024);
            const uint64_t dk1 = make_sdesc_sw128(smem_u32(k_slot(1)), 16, 1024);
            const uint64_t dk2 = make_sdesc_sw128(smem_u32(k_slot(KS - 1)), 16, 1024);

            int n_s = 0;       // S tile products issued (reported through p.tiles_issued)
            // S_t = Q K^T with the K tile of fill f (Q buffer t for pairs, 0 with KV split)
            auto issue_s = [&](int t, uint32_t f) {
                ++n_s;
                const uint64_t a0 = (kSplit || t == 0) ? dq0 : dq1;
                const uint32_t ks = f % KS;
                const uint64_t b0 = ks == 0 ? dk0 : (ks == 1 ? dk1 : dk2);
                const uint32_t dst = tmem + (t == 0 ? L::kColS0 : L::kColS1);
                #pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t off = (uint64_t)(((kk >> 2) * L::kBoxBytes + (kk & 3) * 32) >> 4);
                    mma_bf16_ss(dst, a0 + off, b0 + off, idesc_s, kk > 0);
                }
                mma_commit(&s_full[t]);
            };
            // O_t (+)= P_t V with the V tile of fill f; j = the slot's step (0: overwrite O)
            auto issue_pv = [&](int t, int j, uint32_t f) -> bool {
                if (!mbar_wait(&p_ready[t], j & 1, kErrWaitMma, p.err)) return false;
                tc_fence_after();
                const uint64_t b0 = (f & 1) ? dv1 : dv0;
                const uint32_t col_s = t == 0 ? L::kColS0 : L::kColS1;
                const uint32_t dst = tmem + (t == 0 ? L::kColO0 : L::kColO1);
                #pragma unroll
                for (int kk = 0; kk < kBlockN / 16; ++kk)
                    mma_bf16_ts(dst, tmem + col_s + kk * 8, b0 + (uint64_t)((kk * 16 * 128) >> 4),
                                idesc_pv, (j > 0 || kk > 0) ? 1u : 0u);
                mma_commit(&o_done[t]);
                return true;
            };
            auto wait_k = [&](uint32_t f) -> bool {
                const bool okw = mbar_wait(&k_full[f % KS], (f / KS) & 1, kErrWaitMma, p.err);
                tc_fence_after();
                return okw;
            };
            auto wait_v = [&](uint32_t f) -> bool {
                const bool okw = mbar_wait(&v_full[f & 1], (f >> 1) & 1, kErrWaitMma, p.err);
                tc_fence_after();
                return okw;
            };

            bool ok = mbar_wait(q_full, 0, kErrWaitMma, p.err);
            tc_fence_after();
            if constexpr (!kSplit) {
                // pairs: KV step j is fill j, shared by both slots
                if (ok && n_kv_max > 0 && (ok = wait_k(0))) {
                    if (n0 > 0) issue_s(0, 0);
                    if (n1 > 0) issue_s(1, 0);
                    mma_commit(&k_empty[0]);
                }
                for (int j = 0; j < n_kv_max && ok; ++j) {
                    const bool next = j + 1 < n_kv_max;
                    if (!wait_v(j)) break;
                    if (j < n0 && !issue_pv(0, j, j)) break;
                    if (next) {
                        if (!wait_k(j + 1)) break;
                        if (j + 1 < n0) issue_s(0, j + 1);
                    }
                    if (j < n1 && !issue_pv(1, j, j)) break;
                    mma_commit(&v_empty[j & 1]);
                    if (next) {
                        if (j + 1 < n1) issue_s(1, j + 1);
                        mma_commit(&k_empty[(j + 1) % KS]);
                    }
                }
            } else {
                // KV split: slot 0's step j is fill j + min(j, n1), slot 1's is 2j + 1;
                // every fill feeds one S and one PV, and is released after each
                auto f0 = [&](int j) -> uint32_t { return (uint32_t)(j + min(j, n1)); };
                auto f1 = [&](int j) -> uint32_t { return (uint32_t)(2 * j + 1); };
                if (ok && (ok = wait_k(f0(0)))) {
                    issue_s(0, f0(0));
                    mma_commit(&k_empty[f0(0) % KS]);
                    if (n1 > 0 && (ok = wait_k(f1(0)))) {
                        issue_s(1, f1(0));
                        mma_commit(&k_empty[f1(0) % KS]);
                    }
                }
                for (int j = 0; j < n0 && ok; ++j) {
                    if (!wait_v(f0(j)) || !issue_pv(0, j, f0(j))) break;
                    mma_commit(&v_empty[f0(j) & 1]);
                    if (j + 1 < n0) {
                        if (!wait_k(f0(j + 1))) break;
                        issue_s(0, f0(j + 1));
                        mma_commit(&k_empty[f0(j + 1) % KS]);
                    }
                    if (j < n1) {
                        if (!wait_v(f1(j)) || !issue_pv(1, j, f1(j))) break;
                        mma_commit(&v_empty[f1(j) & 1]);
                    }
                    if (j + 1 < n1) {
                        if (!wait_k(f1(j + 1))) break;
                        issue_s(1, f1(j + 1));
                        mma_commit(&k_empty[f1(j + 1) % KS]);
                    }
                }
            }
            if (p.tiles_issued != nullptr) atomicAdd(p.tiles_issued, n_s);
        }
    } else if (warp >= kSoftmaxWarp0) {
        // =============================== softmax warps ================================
        const int t = (warp - kSoftmaxWarp0) >> 2;     // Q tile of this warpgroup
        const int wq = warp & 3;                        // TMEM lane quadrant
        const TileDesc me = td[t];
        if (me.present) {
            const int r = wq * 32 + lane;               // row within the tile
            const int row = me.q0 + r;                  // query index
            const float c = p.scale_log2;
            int lim = p.Skv;                            // keys [0, lim) visible
            if (p.causal) lim = min(lim, row + p.diag + 1);
            const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
            const uint32_t t_s = tmem + lane_off + (t == 0 ? L::kColS0 : L::kColS1);
            const uint32_t t_o = tmem + lane_off + (t == 0 ? L::kColO0 : L::kColO1);
            float m = -INFINITY, l = 0.f;
            bool ok = true;
            for (int j = 0; j < me.n_kv; ++j) {
                if (!mbar_wait(&s_full[t], j & 1, kErrWaitSoftmax, p.err)) { ok = false; break; }
                tc_fence_after();
                const int kbase = (me.kv0 + j) * kBlockN;
                const bool masked = kbase + kBlockN > lim;
                uint32_t sr[kBlockN];
                tmem_ld128(t_s, sr);
                if (masked) {
                    #pragma unroll
                    for (int e = 0; e < kBlockN; ++e)
                        if (kbase + e >= lim) sr[e] = __float_as_uint(-INFINITY);
                }
                // row max of the raw scores: 4 independent chains of 3-input max, chain k
                // covering columns [32k, 32k + 32)
                float mxc[4];
                #pragma unroll
                for (int k = 0; k < 4; ++k) {
                    float v = fmaxf(__uint_as_float(sr[32 * k]), __uint_as_float(sr[32 * k + 1]));
                    #pragma unroll
                    for (int i = 2; i < 32; i += 2)
                        v = fmax3(v, __uint_as_float(sr[32 * k + i]), __uint_as_float(sr[32 * k + i + 1]));
                    mxc[k] = v;
                }
                const float mx0 = mxc[0], mx1 = mxc[1], mx2 = mxc[2], mx3 = mxc[3];
                const float mx = fmax3(mx0, mx1, fmaxf(mx2, mx3));
                const float mt = mx * c;
                float m_new = m;
                if (mt > m + kRescaleThreshold) m_new = mt;   // also taken when m = -inf
                const float base = (m_new == -INFINITY) ? 0.f : m_new;
                const float corr = (m == -INFINITY) ? 0.f : ex2_approx(m - base);
                const float nb = -base;
                // P = 2^(s*c - m) (packed fp32x2 FMA for the argument), row sum, P -> bf16
                float sum0 = 0.f, sum1 = 0.f;
                uint32_t pk[kBlockN / 2];
                #pragma unroll
                for (int e = 0; e < kBlockN; e += 2) {
                    float a0, a1;
                    fma2(a0, a1, __uint_as_float(sr[e]), __uint_as_float(sr[e + 1]), c, c, nb, nb);
                    const float p0 = ex2_approx(a0);
                    const float p1 = ex2_approx(a1);
                    add2(sum0, sum1, p0, p1);
                    pk[e >> 1] = pack_bf16(p0, p1);
                }
                const float sum = sum0 + sum1;
                tmem_st64(t_s, pk);
                tmem_wait_st();
                l = l * corr + sum;
                m = m_new;
                // correction: O *= corr once the previous P.V has landed
                if (j > 0) {
                    if (!mbar_wait(&o_done[t], (j - 1) & 1, kErrWaitSoftmax, p.err)) { ok = false; break; }
                    tc_fence_after();
                    if (__any_sync(0xffffffffu, corr != 1.0f)) {
                        #pragma unroll 1
                        for (int ch = 0; ch < D / 32; ++ch) {
                            uint32_t rr[32];
                            tmem_ld32(t_o + ch * 32, rr);
                            tmem_wait_ld();
                            #pragma unroll
                            for (int e = 0; e < 32; ++e)
                                rr[e] = __float_as_uint(__uint_as_float(rr[e]) * corr);
                            tmem_st32(t_o + ch * 32, rr);
                        }
                        tmem_wait_st();
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&p_ready[t]);
            }
            // epilogue: O / l -> bf16 -> HBM, LSE
            if (ok && me.n_kv > 0 && mbar_wait(&o_done[t], (me.n_kv - 1) & 1, kErrWaitSoftmax, p.err)) {
                tc_fence_after();
                __nv_bfloat16* orow = p.o + (((long long)b * p.Hq + me.h) * p.Sq + row) * D;
                const bool live = row < p.Sq &&
                                  GBATTN_IN_BOUNDS(((long long)b * p.Hq + me.h) * p.Sq + row,
                                                   (long long)p.B * p.Hq * p.Sq, p.err);
                if (kSplit && td[1].present) {
                    // KV split: merge the two halves' states of this row (log-sum-exp):
                    // O = (a0 O0 + a1 O1) / (a0 l0 + a1 l1), a_t = 2^(m_t - max(m0, m1))
                    float* ms = xm;              // [2][128] running max per slot
                    float* ls = xm + 256;        // [2][128] row sum per slot
                    float* ob = reinterpret_cast<float*>(smem + L::kK0);   // [128][kOStride]
                    ms[t * 128 + r] = m;
                    ls[t * 128 + r] = l;
                    auto meet = [&](uint32_t ph) -> bool {
                        __syncwarp();
                        if (lane == 0) mbar_arrive(merge_bar);
                        return mbar_wait(merge_bar, ph, kErrWaitSoftmax, p.err);
                    };
                    if (meet(0)) {
                        const float m0 = ms[r], m1 = ms[128 + r];
                        const float M = fmaxf(m0, m1);
                        const float a0 = (m0 == -INFINITY) ? 0.f : ex2_approx(m0 - M);
                        const float a1 = (m1 == -INFINITY) ? 0.f : ex2_approx(m1 - M);
                        const float lt = a0 * ls[r] + a1 * ls[128 + r];
                        if (t == 1) {                // slot 1: a1 O1 -> shared memory
                            #pragma unroll 1
                            for (int ch = 0; ch < D / 32; ++ch) {
                                uint32_t rr[32];
                                tmem_ld32(t_o + ch * 32, rr);
                                #pragma unroll
                                for (int e = 0; e < 32; ++e)
                                    ob[r * L::kOStride + ch * 32 + e] = a1 * __uint_as_float(rr[e]);
                            }
                        }
                        if (meet(1) && t == 0) {     // slot 0: a0 O0 + a1 O1, normalise, store
                            const float inv = lt > 0.f ? 1.f / lt : 0.f;
                            #pragma unroll 1
                            for (int ch = 0; ch < D / 32; ++ch) {
                                uint32_t rr[32];
                                tmem_ld32(t_o + ch * 32, rr);
                                if (live) {
                                    float o32[32];
                                    #pragma unroll
                                    for (int e = 0; e < 32; ++e)
                                        o32[e] = (a0 * __uint_as_float(rr[e]) + ob[r * L::kOStride + ch * 32 + e]) * inv;
                                    uint4* dst = reinterpret_cast<uint4*>(orow + ch * 32);
                                    #pragma unroll
                                    for (int q4 = 0; q4 < 4; ++q4) {
                                        uint4 w;
                                        w.x = pack_bf16(o32[8 * q4 + 0], o32[8 * q4 + 1]);
                                        w.y = pack_bf16(o32[8 * q4 + 2], o32[8 * q4 + 3]);
                                        w.z = pack_bf16(o32[8 * q4 + 4], o32[8 * q4 + 5]);
                                        w.w = pack_bf16(o32[8 * q4 + 6], o32[8 * q4 + 7]);
                                        dst[q4] = w;
                                    }
                                }
                            }
                            if (live && p.lse != nullptr)
                                p.lse[((long long)b * p.Hq + me.h) * p.Sq + row] =
                                    lt > 0.f ? (M + __log2f(lt)) * 0.69314718055994531f : -INFINITY;
                        }
                    }
                } else {
                    const float inv = l > 0.f ? 1.f / l : 0.f;
                    #pragma unroll 1
                    for (int ch = 0; ch < D / 32; ++ch) {
                        uint32_t rr[32];
                        tmem_ld32(t_o + ch * 32, rr);
                        if (live) {
                            uint32_t w[16];
                            #pragma unroll
                            for (int e = 0; e < 16; ++e)
                                w[e] = pack_bf16(__uint_as_float(rr[2 * e]) * inv, __uint_as_float(rr[2 * e + 1]) * inv);
                            if (p.o_align32) {          // 32-byte stores: half the store instructions
                                #pragma unroll
                                for (int h = 0; h < 2; ++h)
                                    asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};"
                                                 :: "l"(orow + ch * 32 + h * 16), "r"(w[8 * h]), "r"(w[8 * h + 1]),
                                                    "r"(w[8 * h + 2]), "r"(w[8 * h + 3]), "r"(w[8 * h + 4]),
                                                    "r"(w[8 * h + 5]), "r"(w[8 * h + 6]), "r"(w[8 * h + 7])
                                                 : "memory");
                            } else {
                                uint4* dst = reinterpret_cast<uint4*>(orow + ch * 32);
                                #pragma unroll
                                for (int q4 = 0; q4 < 4; ++q4)
                                    dst[q4] = make_uint4(w[4 * q4], w[4 * q4 + 1], w[4 * q4 + 2], w[4 * q4 + 3]);
                            }
                        }
                    }
                    if (live && p.lse != nullptr)
                        p.lse[((long long)b * p.Hq + me.h) * p.Sq + row] =
                            l > 0.f ? (m + __log2f(l)) * 0.69314718055994531f : -INFINITY;
                }
            }
        }
    }

    // TMEM is released only when no tensor-core work of the CTA can still be running: on
    // success the softmax warps have waited for the last P.V of each slot (the issuer's
    // products complete in issue order); after an error the issuer has drained its
    // products (mma_drain).
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        if (lane == 0 && device_error_set(p.err)) mma_drain(mma_idle, p.err);  // the issuer
        __syncwarp();
        tmem_dealloc(tmem, L::kTmemCols);
    }
    // a tail launch finishes only after the pair-mode grid it overlaps
    if constexpr (kSplit)
        if (blockIdx.x == 0 && threadIdx.x == 0) asm volatile("griddepcontrol.wait;" ::: "memory");
}

template <int D>
cudaError_t launch_pairs(const PrefillParams& p, cudaStream_t stream) {
    constexpr int smem = PLayout<D>::kAlloc;
    cudaError_t err = cudaFuncSetAttribute(prefill_fwd_kernel<D, false>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return err;
    prefill_fwd_kernel<D, false><<<p.n_pairs, kThreads, smem, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

template <int D>
cudaError_t launch_tail(const PrefillParams& p, cudaStream_t stream) {
    constexpr int smem = PLayout<D>::kAlloc;
    cudaError_t err = cudaFuncSetAttribute(prefill_fwd_kernel<D, true>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.n_pairs);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, prefill_fwd_kernel<D, true>, p);
}

cudaError_t launch_attn_fwd_bf16_tail(const PrefillParams& p, int d, cudaStream_t stream) {
    if (p.n_pairs <= 0) return cudaSuccess;
    return d == 128 ? launch_tail<128>(p, stream) : launch_tail<64>(p, stream);
}

cudaError_t launch_attn_fwd_bf16(const PrefillParams& p, int d, cudaStream_t stream) {
    if (p.n_pairs <= 0) return cudaSuccess;
    if (p.kv_split) return cudaErrorInvalidValue;   // small calls run prefill_persist.cu
    return d == 128 ? launch_pairs<128>(p, stream) : launch_pairs<64>(p, stream);
}

#ifdef GBATTN_DEBUG_CHECKS
cudaError_t debug_skip_fill_pairs(int fill) {
    return cudaMemcpyToSymbol(g_skip_k_fill, &fill, sizeof(int));
}
#endif

}  // namespace gbattn
