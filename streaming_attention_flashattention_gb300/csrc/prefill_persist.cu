// prefill_persist.cu -- bf16 prefill for calls too small to fill the GPU with pairs of Q
// tiles: persistent CTAs, one per SM, each running a fixed list of single Q tiles whose KV
// range is split over the CTA's two ping-pong slots.
//
// What it computes is the prefill kernel's (prefill_tcgen05.cu): "AttentionRegion
// Transformation - Deriving FlashAttention via Memory-Centric Compilation in AICF",
// section 8 (a resident Q tile, an inner loop over K/V tiles, the score tile never written to
// memory) with the per-tile operation sequence of "ADR-0060: AHBM GQA Fused Attention Kernel
// (Llama3-70B)", section 3, the tile classes of section 5.4 (KV tiles wholly in a query
// tile's future are never loaded or issued, the diagonal tile and a ragged last tile are
// masked per element) and the log-sum-exp merge of section 4 for the two halves of a Q
// tile's KV range.
//
// Why a second kernel: with one CTA per Q tile, a small call (workload 2: 256 Q tiles on
// 152 SMs) pays a CTA's fixed cost -- a cold Q load, the barrier and TMEM set-up, the merge
// and the output stores -- once per tile, and the CTAs that run two tiles pay it twice on
// the critical path.  Here each SM pays the start-up once, and a tile's merge and stores
// overlap the next tile's loads and S products.
//
// Schedule: the Q tiles are ranked heaviest first (most KV tiles: the last query blocks of
// a causal call) and dealt to the CTAs in snake order -- ranks c, 2G-1-c, 2G+c, ... for CTA c
// of G -- so that a CTA holding one of the heaviest tiles gets one of the lightest next.
// The order is fixed by the sizes alone, so no work counter (and no scratch memory) is
// needed.
//
// Roles (the layout of the multi-token decode kernel, decode_tcgen05.cu):
//   warp 0      Q and K producer: a tile's Q once the previous tile's last S product has read
//               the Q buffer, then its K tiles (slot 0's half and slot 1's half interleaved
//               in the order the MMA issuer consumes them) into a 2-slot ring;
//   warp 2      V producer: the same tiles of V into a 2-slot ring;
//   warp 1      TMEM owner and MMA issuer, one thread: S_t = Q K^T and O_t += P_t V for the
//               two slots in ping-pong order; a tile's first P.V waits until the previous
//               tile's merge has read both O accumulators;
//   warps 4-11  softmax, warpgroup t for slot t, one query row per thread; at the end of a
//               tile the two warpgroups merge the slots straight from TMEM (each takes half
//               of the head dimension) into a bf16 staging tile in shared memory, which one
//               thread writes out with TMA stores while the next tile starts; the LSE is
//               stored directly.
// Shared memory: Q | K x2 | V x2 | O staging (6 tiles of 128 x d bf16).
// TMEM: S0 | S1 | O0 | O1 (128 + 128 + d + d columns of 512).
// Measured on workload 2 (per-CTA %globaltimer stamps): about 0.93 us per 128 x 128 tile
// product in the steady state -- each step brings two K and two V tiles into shared memory
// (one per slot), twice the copies per product of the pair kernel, whose 0.81 us it does not
// reach -- and the same with a 3-slot K or V ring or a single producer thread.
#include "common.cuh"
#include "kernels.h"

namespace gbattn {

namespace {

constexpr int kBlockM = 128;              // query rows per Q tile
constexpr int kBlockN = 128;              // keys per K/V tile
constexpr int kThreads = 12 * 32;
constexpr int kSoftmaxWarp0 = 4;
constexpr int KS = 2;                     // K ring slots
constexpr int VS = 2;                     // V ring slots
constexpr float kRescaleThreshold = 8.0f; // log2 units: move the running max only by > 2^8
constexpr int kStoreThread = kSoftmaxWarp0 * 32;   // issues the O tiles' TMA stores
#ifdef GBATTN_DEBUG_CHECKS
// Test hook of the debug build: CTA 0 of the grid does not issue the K fill with this index
// (counted over the CTA's fills; -1: none).  The fill's barrier then never completes, the wait
// for it runs out after its time limit and records its code in the error word, and every role
// of every CTA leaves through its give-up exit.  Set by attn_debug_skip_fill.
__device__ int g_skip_k_fill = -1;
#endif
static_assert(kBlockN == 128, "the softmax row reductions assume 128 columns");

template <int D>
struct Layout {
    static constexpr int kBoxes = D / 64;
    static constexpr int kTileBytes = 128 * D * 2;          // Q, K or V tile
    static constexpr int kBoxBytes = 128 * 128;              // one 64-column swizzled box
    static constexpr int kQ0 = 0;
    static constexpr int kK0 = kTileBytes;                   // KS K slots
    static constexpr int kV0 = kK0 + KS * kTileBytes;        // VS V slots
    static constexpr int kOst = kV0 + VS * kTileBytes;       // O tile staged for its TMA store
    static constexpr int kBar = kOst + kTileBytes;
    static constexpr int kNumBars = 24;
    static_assert(2 + 2 * KS + 2 * VS + 6 + 4 <= kNumBars, "barrier block");
    static constexpr int kXm = kBar + kNumBars * 8;          // merge: m, l [2 slot][128]
    static constexpr int kTmemSlot = kXm + 4 * 128 * 4;
    static constexpr int kBytes = kTmemSlot + 16;
    static constexpr int kAlloc = kBytes + 1024;
    static constexpr uint32_t kColS0 = 0, kColS1 = 128;
    static constexpr uint32_t kColO0 = 256, kColO1 = 256 + D;
    static constexpr uint32_t kTmemCols = 512;
};

// One Q tile: batch b, query head h, first query row q0, n KV tiles to visit.
struct QTile {
    int b, h, q0, n;
};

// KV tiles a Q tile starting at q0 visits: all of them, or (causal) those up to the last
// row's diagonal (row + diag).
__device__ __forceinline__ int kv_tiles(const PrefillParams& p, int q0) {
    if (!p.causal) return (p.Skv + kBlockN - 1) / kBlockN;
    const int last_row = min(q0 + kBlockM, p.Sq) - 1;
    const int keys = min(p.Skv, last_row + p.diag + 1);
    return (keys + kBlockN - 1) / kBlockN;
}

// The CTA's k-th Q tile (rank >= p.n_pairs: none left).  Ranks are heaviest first: the last
// query block of every (b, h) first, then the one before, ...; CTA c of G takes ranks
// c, 2G-1-c, 2G+c, 4G-1-c, ... (snake order).
__device__ __forceinline__ bool tile_of(const PrefillParams& p, int k, QTile& t) {
    const int G = gridDim.x, c = blockIdx.x;
    const int rank = k * G + ((k & 1) ? G - 1 - c : c);
    if (rank >= p.n_pairs) return false;
    const int bh_count = p.B * p.Hq;
    const int qb = p.n_qblk - 1 - rank / bh_count;
    const int bh = rank % bh_count;
    t.b = bh / p.Hq;
    t.h = bh % p.Hq;
    t.q0 = p.row0 + qb * kBlockM;
    t.n = kv_tiles(p, t.q0);
    return true;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
prefill_persist_kernel(const __grid_constant__ PrefillParams p) {
    using L = Layout<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBar);
    uint64_t* q_full = bars + 0;
    uint64_t* q_empty = bars + 1;          // the tile's last S product has read Q
    uint64_t* k_full = bars + 2;           // [KS]
    uint64_t* k_empty = k_full + KS;       // [KS]
    uint64_t* v_full = k_empty + KS;       // [VS]
    uint64_t* v_empty = v_full + VS;       // [VS]
    uint64_t* s_full = v_empty + VS;       // [2] per slot
    uint64_t* p_ready = s_full + 2;        // [2] per slot
    uint64_t* o_done = p_ready + 2;        // [2] per slot
    uint64_t* merge_bar = o_done + 2;      // the two softmax warpgroups meet
    uint64_t* o_free = merge_bar + 1;      // the merge has read both O accumulators
    uint64_t* mma_idle = o_free + 1;       // error exit: the issuer's products have completed
    uint64_t* staged = mma_idle + 1;       // every merge warp has written its rows of the staging tile
    float* xm = reinterpret_cast<float*>(smem + L::kXm);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kTmemSlot);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // the first tile exists and has KV tiles: its Q and its first K (and V) tile go out before the
    // block barrier, from the thread that initialises the barriers
    QTile it0;
    const bool early_q = tile_of(p, 0, it0);
    const bool early_kv = early_q && it0.n > 0;
    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        mbar_init(q_empty, 1);
        for (int i = 0; i < KS; ++i) {
            mbar_init(&k_full[i], 1);
            mbar_init(&k_empty[i], 1);
        }
        for (int i = 0; i < VS; ++i) {
            mbar_init(&v_full[i], 1);
            mbar_init(&v_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&p_ready[i], 4);
            mbar_init(&o_done[i], 1);
        }
        mbar_init(merge_bar, 8);
        mbar_init(o_free, 8);
        mbar_init(mma_idle, 1);
        mbar_init(staged, 8);
        fence_barrier_init();
        // the first tile's Q and first K tile go out now, under the TMEM allocation and the
        // block barrier (this thread initialised the barriers they complete on)
        if (early_q) {
            mbar_arrive_expect_tx(q_full, L::kTileBytes);
            #pragma unroll
            for (int bx = 0; bx < L::kBoxes; ++bx)
                tma_load_3d(smem + L::kQ0 + bx * L::kBoxBytes, &p.tmap_q, bx * 64, it0.q0,
                            it0.b * p.Hq + it0.h, q_full);
            if (early_kv) {
                mbar_arrive_expect_tx(&k_full[0], L::kTileBytes);
                #pragma unroll
                for (int bx = 0; bx < L::kBoxes; ++bx)
                    tma_load_3d(smem + L::kK0 + bx * L::kBoxBytes, &p.tmap_k, bx * 64, 0,
                                it0.b * p.Hkv + it0.h / p.G, &k_full[0]);
            }
        }
    }
    if (warp == 1) tmem_alloc(tmem_slot, L::kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ============================== Q and K producer ==============================
        if (lane == 0) {
            prefetch_tensormap(&p.tmap_q);
            prefetch_tensormap(&p.tmap_k);
            uint32_t nf = 0;         // K fills so far (all tiles)
            int k = 0;               // Q tiles so far
            bool ok = true;
#ifdef GBATTN_DEBUG_CHECKS
            uint32_t skipped = 0xffffffffu;   // the fill the test hook left out
#endif
            QTile it;
            for (; ok && tile_of(p, k, it); ++k) {
                // Q once the previous tile's last S product has read the buffer (the first
                // tile's Q went out before the block barrier)
                if (k > 0) {
                    if (!(ok = mbar_wait(q_empty, (k - 1) & 1, kErrWaitProducer, p.err))) break;
                    mbar_arrive_expect_tx(q_full, L::kTileBytes);
                    #pragma unroll
                    for (int bx = 0; bx < L::kBoxes; ++bx)
                        tma_load_3d(smem + L::kQ0 + bx * L::kBoxBytes, &p.tmap_q, bx * 64, it.q0,
                                    it.b * p.Hq + it.h, q_full);
                }
                const int n0 = (it.n + 1) / 2, n1 = it.n - n0;
                const int zkv = it.b * p.Hkv + it.h / p.G;
                for (int j = 0; j < n0 && ok; ++j) {
                    for (int t = 0; t < 2 && ok; ++t) {
                        if (t == 1 && j >= n1) continue;
                        const int tile = t == 0 ? j : n0 + j;
                        const uint32_t ks = nf % KS, kph = (nf / KS) & 1;
                        if (nf == 0 && early_kv) {  // went out before the block barrier
                            ++nf;
                            continue;
                        }
                        if (!(ok = mbar_wait(&k_empty[ks], kph ^ 1u, kErrWaitProducer, p.err))) break;
#ifdef GBATTN_DEBUG_CHECKS
                        if (blockIdx.x == 0 && (int)nf == g_skip_k_fill) {
                            skipped = nf++;
                            continue;
                        }
#endif
                        mbar_arrive_expect_tx(&k_full[ks], L::kTileBytes);
                        #pragma unroll
                        for (int bx = 0; bx < L::kBoxes; ++bx)
                            tma_load_3d(smem + L::kK0 + ks * L::kTileBytes + bx * L::kBoxBytes,
                                        &p.tmap_k, bx * 64, tile * kBlockN, zkv, &k_full[ks]);
                        ++nf;
                    }
                }
            }
            // drain: the last fills of Q and of each K slot must land before the CTA exits
            if (k > 0) mbar_wait_drain(q_full, (k - 1) & 1, p.err);
            for (uint32_t f = nf >= (uint32_t)KS ? nf - KS : 0; f < nf; ++f) {
#ifdef GBATTN_DEBUG_CHECKS
                if (f == skipped) continue;
#endif
                mbar_wait_drain(&k_full[f % KS], (f / KS) & 1, p.err);
            }
        }
    } else if (warp == 2) {
        // ================================ V producer =================================
        if (lane == 0) {
            prefetch_tensormap(&p.tmap_v);
            uint32_t nf = 0;
            bool ok = true;
            QTile it;
            for (int k = 0; ok && tile_of(p, k, it); ++k) {
                const int n0 = (it.n + 1) / 2, n1 = it.n - n0;
                const int zkv = it.b * p.Hkv + it.h / p.G;
                for (int j = 0; j < n0 && ok; ++j) {
                    for (int t = 0; t < 2 && ok; ++t) {
                        if (t == 1 && j >= n1) continue;
                        const int tile = t == 0 ? j : n0 + j;
                        const uint32_t vs = nf % VS, vph = (nf / VS) & 1;
                        if (!(ok = mbar_wait(&v_empty[vs], vph ^ 1u, kErrWaitProducer, p.err))) break;
                        mbar_arrive_expect_tx(&v_full[vs], L::kTileBytes);
                        #pragma unroll
                        for (int bx = 0; bx < L::kBoxes; ++bx)
                            tma_load_3d(smem + L::kV0 + vs * L::kTileBytes + bx * L::kBoxBytes,
                                        &p.tmap_v, bx * 64, tile * kBlockN, zkv, &v_full[vs]);
                        ++nf;
                    }
                }
            }
            // drain: the last fill of each V slot must land before the CTA exits
            for (uint32_t f = nf >= (uint32_t)VS ? nf - VS : 0; f < nf; ++f)
                mbar_wait_drain(&v_full[f % VS], (f / VS) & 1, p.err);
        }
    } else if (warp == 1) {
        // ================================ MMA issuer =================================
        // Per step j: PV0(j), S0(j+1), PV1(j), S1(j+1) -- S_t(j+1) overwrites P_t(j) and
        // is issued after PV_t(j) (tcgen05.mma executes in issue order).  A tile's first P.V
        // overwrites O and waits until the previous tile's merge has read both accumulators;
        // its S products do not wait.
        if (lane == 0) {
            constexpr uint32_t idesc_s = make_idesc_bf16(kBlockM, kBlockN, 0, 0);
            constexpr uint32_t idesc_pv = make_idesc_bf16(kBlockM, D, 0, 1);
            // descriptors built once; the start-address field advances by a constant per
            // K = 16 step (shared addresses stay below 2^18, so the field cannot carry)
            const uint64_t dq = make_sdesc_sw128(smem_u32(smem + L::kQ0), 16, 1024);
            const uint64_t dk0 = make_sdesc_sw128(smem_u32(smem + L::kK0), 16, 1024);
            const uint64_t dv0 = make_sdesc_sw128(smem_u32(smem + L::kV0), L::kBoxBytes, 1024);
            uint32_t fbase = 0, cs0 = 0, cs1 = 0;
            int n_s = 0;             // S tile products issued (reported through p.tiles_issued)
            bool ok = true;
            QTile it;
            for (int k = 0; ok && tile_of(p, k, it); ++k) {
                const int n = it.n, n0 = (n + 1) / 2, n1 = n - n0;
                // fill order: slot 0's step j is fill f0(j), slot 1's is f1(j)
                auto f0 = [&](int j) -> uint32_t { return fbase + (uint32_t)(j + min(j, n1)); };
                auto f1 = [&](int j) -> uint32_t { return fbase + (uint32_t)(2 * j + 1); };
                int ns = 0;
                auto issue_s = [&](int t, uint32_t f) {
                    const uint64_t b0 = dk0 + (uint64_t)((f % KS) * (L::kTileBytes >> 4));
                    const uint32_t dst = tmem + (t == 0 ? L::kColS0 : L::kColS1);
                    #pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint64_t off = (uint64_t)(((kk >> 2) * L::kBoxBytes + (kk & 3) * 32) >> 4);
                        mma_bf16_ss(dst, dq + off, b0 + off, idesc_s, kk > 0);
                    }
                    mma_commit(&s_full[t]);
                    mma_commit(&k_empty[f % KS]);
                    if (++ns == n) mma_commit(q_empty);   // the tile's last read of Q
                };
                auto issue_pv = [&](int t, int j, uint32_t f) -> bool {
                    const uint32_t cs = t == 0 ? cs0 : cs1;
                    if (!mbar_wait(&p_ready[t], (cs + j) & 1, kErrWaitMma, p.err)) return false;
                    if (t == 0 && j == 0 && k > 0 && !mbar_wait(o_free, (k - 1) & 1, kErrWaitMma, p.err))
                        return false;
                    const uint32_t vs = f % VS;
                    if (!mbar_wait(&v_full[vs], (f / VS) & 1, kErrWaitMma, p.err)) return false;
                    tc_fence_after();
                    const uint64_t b0 = dv0 + (uint64_t)(vs * (L::kTileBytes >> 4));
                    const uint32_t col_s = t == 0 ? L::kColS0 : L::kColS1;
                    const uint32_t dst = tmem + (t == 0 ? L::kColO0 : L::kColO1);
                    #pragma unroll
                    for (int kk = 0; kk < kBlockN / 16; ++kk)
                        mma_bf16_ts(dst, tmem + col_s + kk * 8, b0 + (uint64_t)((kk * 16 * 128) >> 4),
                                    idesc_pv, (j > 0 || kk > 0) ? 1u : 0u);
                    mma_commit(&o_done[t]);
                    mma_commit(&v_empty[vs]);
                    return true;
                };
                auto wait_k = [&](uint32_t f) -> bool {
                    const bool okw = mbar_wait(&k_full[f % KS], (f / KS) & 1, kErrWaitMma, p.err);
                    tc_fence_after();
                    return okw;
                };
                ok = mbar_wait(q_full, k & 1, kErrWaitMma, p.err);
                tc_fence_after();
                if (ok && (ok = wait_k(f0(0)))) {
                    issue_s(0, f0(0));
                    if (n1 > 0 && (ok = wait_k(f1(0)))) issue_s(1, f1(0));
                }
                for (int j = 0; j < n0 && ok; ++j) {
                    if (!(ok = issue_pv(0, j, f0(j)))) break;
                    if (j + 1 < n0) {
                        if (!(ok = wait_k(f0(j + 1)))) break;
                        issue_s(0, f0(j + 1));
                    }
                    if (j < n1 && !(ok = issue_pv(1, j, f1(j)))) break;
                    if (j + 1 < n1) {
                        if (!(ok = wait_k(f1(j + 1)))) break;
                        issue_s(1, f1(j + 1));
                    }
                }
                n_s += ns;
                fbase += (uint32_t)n;
                cs0 += (uint32_t)n0;
                cs1 += (uint32_t)n1;
            }
            if (p.tiles_issued != nullptr) atomicAdd(p.tiles_issued, n_s);
        }
    } else if (warp >= kSoftmaxWarp0) {
        // =============================== softmax warps ================================
        const int t = (warp - kSoftmaxWarp0) >> 2;     // slot of this warpgroup
        const int wq = warp & 3;                        // TMEM lane quadrant
        const int r = wq * 32 + lane;                   // row within the tile
        const float c = p.scale_log2;
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        const uint32_t t_s = tmem + lane_off + (t == 0 ? L::kColS0 : L::kColS1);
        const uint32_t t_o = tmem + lane_off + (t == 0 ? L::kColO0 : L::kColO1);
        const uint32_t t_o0 = tmem + lane_off + L::kColO0;
        const uint32_t t_o1 = tmem + lane_off + L::kColO1;
        if (threadIdx.x == kStoreThread) prefetch_tensormap(&p.tmap_o);
        const uint32_t ost = smem_u32(smem + L::kOst);   // the staging tile
        float* ms = xm;              // [2][128] running max per slot
        float* ls = xm + 256;        // [2][128] row sum per slot
        uint32_t cs0 = 0, cs1 = 0;
        bool ok = true;
        QTile it;
        for (int k = 0; ok && tile_of(p, k, it); ++k) {
            const int n0 = (it.n + 1) / 2, n1 = it.n - n0;
            const int n_t = t == 0 ? n0 : n1;           // this slot's key tiles
            const uint32_t cs = t == 0 ? cs0 : cs1;
            const int kv0 = t == 0 ? 0 : n0;
            const int row = it.q0 + r;                  // query index
            int lim = p.Skv;                            // keys [0, lim) visible
            if (p.causal) lim = min(lim, row + p.diag + 1);
            float m = -INFINITY, l = 0.f;
            for (int j = 0; j < n_t; ++j) {
                if (!mbar_wait(&s_full[t], (cs + j) & 1, kErrWaitSoftmax, p.err)) { ok = false; break; }
                tc_fence_after();
                const int kbase = (kv0 + j) * kBlockN;
                uint32_t sr[kBlockN];
                tmem_ld128(t_s, sr);
                if (kbase + kBlockN > lim) {
                    #pragma unroll
                    for (int e = 0; e < kBlockN; ++e)
                        if (kbase + e >= lim) sr[e] = __float_as_uint(-INFINITY);
                }
                // row max of the raw scores: 4 independent chains of 3-input max
                float mxc[4];
                #pragma unroll
                for (int q = 0; q < 4; ++q) {
                    float v = fmaxf(__uint_as_float(sr[32 * q]), __uint_as_float(sr[32 * q + 1]));
                    #pragma unroll
                    for (int i = 2; i < 32; i += 2)
                        v = fmax3(v, __uint_as_float(sr[32 * q + i]), __uint_as_float(sr[32 * q + i + 1]));
                    mxc[q] = v;
                }
                const float mt = fmax3(mxc[0], mxc[1], fmaxf(mxc[2], mxc[3])) * c;
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
                tmem_st64(t_s, pk);
                tmem_wait_st();
                l = l * corr + (sum0 + sum1);
                m = m_new;
                // correction: O *= corr once the previous P.V has landed
                if (j > 0) {
                    if (!mbar_wait(&o_done[t], (cs + j - 1) & 1, kErrWaitSoftmax, p.err)) { ok = false; break; }
                    tc_fence_after();
                    if (__any_sync(0xffffffffu, corr != 1.0f)) {
                        #pragma unroll 1
                        for (int ch = 0; ch < D / 32; ++ch) {
                            uint32_t rr[32];
                            tmem_ld32(t_o + ch * 32, rr);
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
            if (!ok) break;
            // ---- end of the tile: merge the two slots, store O and the LSE ----
            // Each warpgroup first waits for its own slot's last P.V; after the meet both
            // accumulators are complete, and warpgroup t merges columns [t D/2, (t+1) D/2)
            // of every row:  O = (a0 O0 + a1 O1) / (a0 l0 + a1 l1),  a_s = 2^(m_s - max m).
            // The bf16 rows go to the staging tile (128-byte swizzle, the layout of the O
            // tensor map's boxes) and one thread stores the tile with TMA, asynchronously:
            // rows past Sq are clipped by the copy, and the next tile's merge only waits
            // until the copy has read the staging tile.
            if (n_t > 0) {
                if (!mbar_wait(&o_done[t], (cs + n_t - 1) & 1, kErrWaitSoftmax, p.err)) break;
                ms[t * 128 + r] = m;
                ls[t * 128 + r] = l;
            }
            __syncwarp();
            if (lane == 0) {
                if (threadIdx.x == kStoreThread) bulk_wait_group_read<0>();   // staging tile free
                mbar_arrive(merge_bar);
            }
            if (!mbar_wait(merge_bar, k & 1, kErrWaitSoftmax, p.err)) break;
            // the other slot's last completion, already seen by its warpgroup
            const int u = 1 - t;
            const int n_u = u == 0 ? n0 : n1;
            if (n_u > 0 && !mbar_wait(&o_done[u], ((u == 0 ? cs0 : cs1) + n_u - 1) & 1,
                                      kErrWaitSoftmax, p.err))
                break;
            tc_fence_after();
            {
                const float m0 = ms[r];
                const float m1 = n1 > 0 ? ms[128 + r] : -INFINITY;
                const float M = fmaxf(m0, m1);
                const float a0 = (m0 == -INFINITY) ? 0.f : ex2_approx(m0 - M);
                const float a1 = (m1 == -INFINITY) ? 0.f : ex2_approx(m1 - M);
                const float lt = a0 * ls[r] + (n1 > 0 ? a1 * ls[128 + r] : 0.f);
                const float inv = lt > 0.f ? 1.f / lt : 0.f;
                #pragma unroll 1
                for (int ch = 0; ch < D / 64; ++ch) {
                    const int col = t * (D / 2) + ch * 32;
                    uint32_t r0[32], r1[32];
                    tmem_ld32(t_o0 + col, r0);
                    // (slot 1 empty: a1 = 0 and its accumulator holds no result; zeroing r1
                    // also keeps it defined on both paths, which the register allocator
                    // otherwise answers with spills)
                    if (n1 > 0) {
                        tmem_ld32(t_o1 + col, r1);
                    } else {
                        #pragma unroll
                        for (int e = 0; e < 32; ++e) r1[e] = 0u;
                    }
                    uint32_t w[16];
                    #pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const float v0 = a0 * __uint_as_float(r0[2 * e]) + a1 * __uint_as_float(r1[2 * e]);
                        const float v1 = a0 * __uint_as_float(r0[2 * e + 1]) + a1 * __uint_as_float(r1[2 * e + 1]);
                        w[e] = pack_bf16(v0 * inv, v1 * inv);
                    }
                    // 16-byte chunk c of row r in its 64-column box sits at chunk c ^ (r & 7)
                    const uint32_t box = ost + (uint32_t)((col >> 6) * L::kBoxBytes + r * 128);
                    const int c0 = (col & 63) >> 3;
                    #pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4)
                        st_shared_v4(box + (uint32_t)(((c0 + q4) ^ (r & 7)) << 4), w[4 * q4],
                                     w[4 * q4 + 1], w[4 * q4 + 2], w[4 * q4 + 3]);
                }
                // the tile's coordinates again, from its index: keeping them in registers
                // through the softmax loop costs spills there
                int k_again;
                asm volatile("mov.b32 %0, %1;" : "=r"(k_again) : "r"(k));
                tile_of(p, k_again, it);
                const int row = it.q0 + r;
                if (t == 0 && row < p.Sq && p.lse != nullptr &&
                    GBATTN_IN_BOUNDS(((long long)it.b * p.Hq + it.h) * p.Sq + row,
                                     (long long)p.B * p.Hq * p.Sq, p.err))
                    p.lse[((long long)it.b * p.Hq + it.h) * p.Sq + row] =
                        lt > 0.f ? (M + __log2f(lt)) * 0.69314718055994531f : -INFINITY;
            }
            // the staged tile is complete once all 8 merge warps have arrived; only the store
            // thread waits (bounded), so a warp that left the loop after an error cannot hold
            // the others at a hardware barrier. A warp arrives for tile k + 1 only after the
            // meet of tile k + 1, which the store thread reaches after this wait: the phases
            // cannot overtake one another.
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(staged);
            if (threadIdx.x == kStoreThread && mbar_wait(staged, k & 1, kErrWaitSoftmax, p.err) &&
                GBATTN_IN_BOUNDS(it.b * p.Hq + it.h, p.B * p.Hq, p.err) &&
                GBATTN_IN_BOUNDS(it.q0, p.Sq, p.err)) {
                #pragma unroll
                for (int bx = 0; bx < L::kBoxes; ++bx)
                    tma_store_3d(&p.tmap_o, smem + L::kOst + bx * L::kBoxBytes, bx * 64, it.q0,
                                 it.b * p.Hq + it.h);
                bulk_commit_group();
            }
            // both accumulators (and m, l above) may now be overwritten by the next tile
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(o_free);
            cs0 += (uint32_t)n0;
            cs1 += (uint32_t)n1;
        }
        // the last tile's stores must complete before the CTA (and its shared memory) ends
        if (threadIdx.x == kStoreThread) bulk_wait_group<0>();
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
}

template <int D>
cudaError_t launch_persist(const PrefillParams& p, int nsm, cudaStream_t stream) {
    constexpr int smem = Layout<D>::kAlloc;
    static_assert(smem <= 227 * 1024, "shared memory budget");
    cudaError_t err = cudaFuncSetAttribute(prefill_persist_kernel<D>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return err;
    prefill_persist_kernel<D><<<min(p.n_pairs, nsm), kThreads, smem, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_fwd_bf16_persistent(const PrefillParams& p, int d, int nsm,
                                            cudaStream_t stream) {
    if (p.n_pairs <= 0) return cudaSuccess;
    return d == 128 ? launch_persist<128>(p, nsm, stream) : launch_persist<64>(p, nsm, stream);
}

#ifdef GBATTN_DEBUG_CHECKS
cudaError_t debug_skip_fill_persist(int fill) {
    return cudaMemcpyToSymbol(g_skip_k_fill, &fill, sizeof(int));
}
#endif

}  // namespace gbattn
