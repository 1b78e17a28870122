// decode_tcgen05.cu -- multi-token split-KV decode on the 5th-generation tensor cores.
//
// "ADR-0060: AHBM GQA Fused Attention Kernel (Llama3-70B)":
//   section 0.5 / 5.2 -- the G query heads of a KV head and their T_q new tokens fold into
//                        one GEMM operand of G * T_q rows ([G, T_q, d] -> [G * T_q, d]);
//                        every K/V tile is read once for all of them;
//   section 3         -- per tile: scale, mask, row max, exp, corr = exp(m - m_new), l and O;
//   section 4 / 2.1   -- contiguous splits whose partial (lse, O) a log-sum-exp merge folds.
// New token t of a sequence with len keys sees keys j <= len - T_q + t (the oracle's
// bottom-right causal rule with Sq = T_q).
//
// GB300 mapping.  With R = G * T_q query rows per KV head (16 to 128) the row operand is
// large enough for tcgen05: a work item (sequence b, KV head, split s, 128-row tile of the
// R rows) runs like one Q tile of the prefill kernel's KV-split mode (prefill_tcgen05.cu).
// The CTAs are persistent, one per SM, and pull items from a device counter:
//   warp 0      work queue and Q/K producer: claims the next item, hands it to the other
//               warps through a two-entry ring in shared memory, then loads the item's rows
//               of Q (its R rows rounded up to 8, at most one 128-row tile: the other rows
//               of the M = 128 operand keep stale data and only yield output rows that are
//               never stored) and the split's K in 128-key tiles into a 2-slot ring.  It
//               moves on to the next item's tiles as soon as ring slots free up, so the loads
//               run on through the item boundaries;
//   warp 2      V producer: the same tiles of V into a 3-slot ring.  A V slot is held until
//               its P.V product completes, long after the K tile's S product, so V gets the
//               deeper ring and its own thread: K loads never wait behind a V slot;
//   warp 1      TMEM owner and MMA issuer: S = Q K^T (M = 128 rows, N = 128 keys) and
//               O += P V (P from TMEM), for the two ping-pong slots, which take the two
//               halves of the split's tiles;
//   warps 4-11  softmax, one row per thread (warps whose 32 rows lie past R only keep the
//               handshakes); the running max moves only when it grows by more than 2^8.
// At the end of an item the two warpgroups merge the two slots straight from TMEM (each
// takes half of the head dimension) and write the split's normalised partial (lse_s, O_s)
// to the workspace (a sequence with a single split writes its final O and LSE); the decode
// combine kernel, launched dependent on this one, folds the partials.  Meanwhile the next
// item's S products are already running.
// Decode reads each K/V byte once for R rows: the MMA work per byte is small enough on
// tcgen05 that the kernel runs at the memory rate even with 9 rows of 128 in use.
#include "common.cuh"
#include "decode_splits.cuh"
#include "kernels.h"

namespace gbattn {

namespace {

constexpr int kRowsT = 128;               // query rows per item (M)
constexpr int kKeysT = 128;               // keys per K/V tile (N of S)
constexpr int kThreads = 12 * 32;
constexpr int kSoftmaxWarp0 = 4;
constexpr int KS = 2;                     // K ring slots
constexpr int VS = 3;                     // V ring slots
constexpr float kRescaleThreshold = 8.0f; // log2 units: move the running max only by > 2^8
constexpr int kPubSlots = 4;              // publisher ring entries (finished partials)
#ifdef GBATTN_DEBUG_CHECKS
// Test hook of the debug build: CTA 0 of the grid does not issue the K fill with this index
// (counted over the CTA's fills; -1: none).  The fill's barrier then never completes, the wait
// for it runs out after its time limit and records its code in the error word, and every role
// of every CTA leaves through its give-up exit.  Set by attn_debug_skip_fill.
__device__ int g_skip_k_fill = -1;
#endif
static_assert(kKeysT == 128, "the softmax row reductions assume 128 columns");

// One work item as the producer hands it to the MMA and softmax warps.
struct MtItem {
    int b, kvh, s, rt;                     // s: the item's partial slot (split * pieces + piece)
    int len, t0, t1, n_ne;
    int done;                              // end-of-work marker
    int direct;                            // the item is its rows' only partial: write O, LSE
    int pad[2];
};

template <int D>
struct Layout {
    static constexpr int kBoxes = D / 64;
    static constexpr int kTileBytes = 128 * D * 2;          // Q, K or V tile
    static constexpr int kBoxBytes = 128 * 128;              // one 64-column swizzled box
    static constexpr int kQ0 = 0;
    static constexpr int kK0 = kTileBytes;                   // KS K slots
    static constexpr int kV0 = kK0 + KS * kTileBytes;        // VS V slots
    static constexpr int kBar = kV0 + VS * kTileBytes;
    static constexpr int kNumBars = 40;
    static_assert(2 + 2 * KS + 3 * VS + 6 + 2 + 4 + 1 + 2 * kPubSlots <= kNumBars, "barrier block");
    static constexpr int kXm = kBar + kNumBars * 8;          // merge: m, l [2 slot][128]
    static constexpr int kInfo = kXm + 4 * 128 * 4;          // MtItem [2]
    static constexpr int kTmemSlot = kInfo + 2 * (int)sizeof(MtItem);
    static constexpr int kPubGroup = kTmemSlot + 16;         // publisher ring: group per entry
    static constexpr int kBytes = kPubGroup + kPubSlots * 4;
    static constexpr int kAlloc = kBytes + 1024;
    static constexpr uint32_t kColS0 = 0, kColS1 = 128;
    static constexpr uint32_t kColO0 = 256, kColO1 = 256 + D;
    static constexpr uint32_t kTmemCols = 512;
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
decode_mt_kernel(const __grid_constant__ DecodeTcParams p) {
    using L = Layout<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBar);
    uint64_t* q_full = bars + 0;
    uint64_t* q_empty = bars + 1;          // the item's last S product has read Q
    uint64_t* k_full = bars + 2;           // [KS]
    uint64_t* k_empty = k_full + KS;       // [KS]
    uint64_t* v_full = k_empty + KS;       // [VS]
    uint64_t* v_empty = v_full + VS;       // [VS]
    uint64_t* s_full = v_empty + VS;       // [2] per slot
    uint64_t* p_ready = s_full + 2;        // [2] per slot
    uint64_t* o_done = p_ready + 2;        // [2] per slot
    uint64_t* merge_bar = o_done + 2;      // the two softmax warpgroups meet
    uint64_t* v_fix = merge_bar + 1;       // [VS] per V slot: the tile crossing len, zeroed
    uint64_t* o_free = v_fix + VS;         // the merge has read both O accumulators
    uint64_t* item_full = o_free + 1;      // [2] item ring
    uint64_t* item_empty = item_full + 2;  // [2]
    uint64_t* mma_idle = item_empty + 2;   // error exit: the issuer's products have completed
    uint64_t* pub_full = mma_idle + 1;     // [kPubSlots] softmax warps -> publisher (partial written)
    uint64_t* pub_empty = pub_full + kPubSlots;   // [kPubSlots] publisher -> softmax warps
    int* pub_group = reinterpret_cast<int*>(smem + L::kPubGroup);   // [kPubSlots]
    float* xm = reinterpret_cast<float*>(smem + L::kXm);
    MtItem* info = reinterpret_cast<MtItem*>(smem + L::kInfo);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kTmemSlot);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr int kConsumers = 1 + 8 + 1;  // MMA issuer, softmax warps, V producer read each item

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
            mbar_init(&v_fix[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&p_ready[i], 4);
            mbar_init(&o_done[i], 1);
            mbar_init(&item_full[i], 1);
            mbar_init(&item_empty[i], kConsumers);
        }
        mbar_init(merge_bar, 8);
        mbar_init(o_free, 8);
        mbar_init(mma_idle, 1);
        for (int i = 0; i < kPubSlots; ++i) {
            mbar_init(&pub_full[i], 8);
            mbar_init(&pub_empty[i], 1);
        }
        fence_barrier_init();
    }
    if (warp == 1) tmem_alloc(tmem_slot, L::kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // =========================== work queue, Q and K producer ===========================
        // Lane 0 claims items, hands each to the other warps and loads its Q and K tiles.
        if (lane == 0) {
            prefetch_tensormap(&p.tmap_q);
            prefetch_tensormap(&p.tmap_k);
        }
        uint32_t nf = 0;         // K fills so far (all items)
        uint32_t k = 0;          // items handed over so far
        uint32_t nq = 0;         // Q fills issued (lane 0)
        bool ok = true;
#ifdef GBATTN_DEBUG_CHECKS
        uint32_t skipped = 0xffffffffu;   // the fill the test hook left out
#endif
        while (ok) {
            int item = 0;
            if (lane == 0) item = atomicAdd(p.counter, 1);
            item = __shfl_sync(0xffffffffu, item, 0);
            if (item >= p.n_items) break;
            int rem = item;
            const int rt = rem % p.n_rt; rem /= p.n_rt;
            const int pc = rem % p.pieces; rem /= p.pieces;     // piece of the split
            const int s = rem % p.n_slots; rem /= p.n_slots;
            const int kvh = rem % p.Hkv;
            const int b = rem / p.Hkv;
            int len = __ldg(&p.kv_lens[b]);
            len = max(0, min(len, p.Lmax));
            const int nb = splits_for(len, p.fixed_splits, p.auto_floor);
            const int n_ne = nonempty_splits(len, nb);
            const long long row0 = ((long long)b * p.Hkv + kvh) * p.R + (long long)rt * kRowsT;
            if (s >= n_ne) {
                // no keys in this split; a sequence with no keys at all gets O = 0, LSE = -inf
                if (s == 0 && pc == 0 && n_ne == 0) {
                    const int nrows = min(kRowsT, p.R - rt * kRowsT);
                    for (int i = lane; i < nrows * (D / 8); i += 32) {
                        const int r = i / (D / 8), c = i % (D / 8);
                        if (!GBATTN_IN_BOUNDS(row0 + r, (long long)p.B * p.Hq * p.Tq, p.err)) continue;
                        reinterpret_cast<uint4*>(p.o + (row0 + r) * D)[c] = make_uint4(0, 0, 0, 0);
                        if (c == 0 && p.lse != nullptr) p.lse[row0 + r] = -INFINITY;
                    }
                }
                continue;
            }
            int t0, t1;
            split_range(len, nb, s, t0, t1);
            piece_range(t0, t1, p.pieces, pc, t0, t1);
            const int part = s * p.pieces + pc;
            if (t0 >= t1) {
                // an empty piece of a non-empty split: a partial that weighs nothing (written
                // by one lane, which then counts it with a release covering its writes)
                if (lane == 0) {
                    const int nrows = min(kRowsT, p.R - rt * kRowsT);
                    for (int i = 0; i < nrows; ++i)
                        if (GBATTN_IN_BOUNDS((row0 + i) * p.n_parts + part, (long long)p.B * p.Hq * p.Tq * p.n_parts, p.err))
                            p.ws_lse[(row0 + i) * p.n_parts + part] = -INFINITY;
                    const long long g = ((long long)b * p.Hkv + kvh) * p.n_rt + rt;
                    if (p.counted && GBATTN_IN_BOUNDS(g, (long long)p.B * p.Hkv * p.n_rt, p.err))
                        counter_add_release(p.group_cnt + g, 1);
                }
                __syncwarp();
                continue;
            }
            const int nt = (t1 - t0 + kKeysT - 1) / kKeysT;
            const int n0 = (nt + 1) / 2, n1 = nt - n0;
            if (lane == 0) {
                // hand the item over, then load its Q once the previous item's last S
                // product has read the buffer
                ok = mbar_wait(&item_empty[k & 1], ((k >> 1) & 1) ^ 1u, kErrWaitProducer, p.err);
                if (ok) {
                    MtItem& it = info[k & 1];
                    it.b = b; it.kvh = kvh; it.s = part; it.rt = rt;
                    it.len = len; it.t0 = t0; it.t1 = t1; it.n_ne = n_ne;
                    it.done = 0;
                    it.direct = (n_ne == 1 && p.pieces == 1) ? 1 : 0;
                    mbar_arrive(&item_full[k & 1]);
                }
                if (ok && k > 0) ok = mbar_wait(q_empty, (k - 1) & 1, kErrWaitProducer, p.err);
                if (ok) {
                    mbar_arrive_expect_tx(q_full, (uint32_t)(L::kBoxes * p.q_rows * 128));
                    #pragma unroll
                    for (int bx = 0; bx < L::kBoxes; ++bx)
                        tma_load_3d(smem + L::kQ0 + bx * L::kBoxBytes, &p.tmap_q, bx * 64, (int)row0, 0, q_full);
                    ++nq;
                }
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            ++k;
            const int zkv = b * p.Hkv + kvh;
            for (int j = 0; j < n0 && ok; ++j) {
                for (int t = 0; t < 2 && ok; ++t) {
                    if (t == 1 && j >= n1) continue;
                    const int key0 = t0 + (t == 0 ? j : n0 + j) * kKeysT;
                    const uint32_t ks = nf % KS, kph = (nf / KS) & 1;
                    if (lane == 0) {
                        ok = mbar_wait(&k_empty[ks], kph ^ 1u, kErrWaitProducer, p.err);
#ifdef GBATTN_DEBUG_CHECKS
                        if (ok && blockIdx.x == 0 && (int)nf == g_skip_k_fill) {
                            skipped = nf;
                        } else
#endif
                        if (ok) {
                            mbar_arrive_expect_tx(&k_full[ks], L::kTileBytes);
                            #pragma unroll
                            for (int bx = 0; bx < L::kBoxes; ++bx)
                                tma_load_3d(smem + L::kK0 + ks * L::kTileBytes + bx * L::kBoxBytes, &p.tmap_k,
                                            bx * 64, key0, zkv, &k_full[ks]);
                        }
                    }
                    ok = __shfl_sync(0xffffffffu, ok, 0);
                    nf += ok ? 1u : 0u;   // (a fill not issued is not drained)
                }
            }
        }
        if (lane == 0) {
            // end-of-work marker
            if (ok && mbar_wait(&item_empty[k & 1], ((k >> 1) & 1) ^ 1u, kErrWaitProducer, p.err)) {
                info[k & 1].done = 1;
                mbar_arrive(&item_full[k & 1]);
            }
            // this CTA takes no more work: the combine grid may start being scheduled
            asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
            // drain: the last fills of Q and of each K slot must land before the CTA exits
            if (nq > 0) mbar_wait_drain(q_full, (nq - 1) & 1, p.err);
            for (uint32_t f = nf >= (uint32_t)KS ? nf - KS : 0; f < nf; ++f) {
#ifdef GBATTN_DEBUG_CHECKS
                if (f == skipped) continue;
#endif
                mbar_wait_drain(&k_full[f % KS], (f / KS) & 1, p.err);
            }
        }
    } else if (warp == 2) {
        // ================================== V producer ==================================
        // Lane 0 loads the V tiles in the same fill order, independently of the K ring.  The
        // V rows of the tile that crosses len are zeroed in shared memory by the whole warp
        // once the tile has landed: cache rows past len are not part of the sequence (they
        // may hold anything, NaN included), and their P is 0 -- but 0 * NaN is not 0 in the
        // P.V product.
        if (lane == 0) prefetch_tensormap(&p.tmap_v);
        uint32_t nf = 0;         // V fills so far (all items)
        uint32_t k = 0;
        bool ok = true;
        while (ok) {
            if (!mbar_wait(&item_full[k & 1], (k >> 1) & 1, kErrWaitProducer, p.err)) break;
            const MtItem it = info[k & 1];
            __syncwarp();
            if (lane == 0) mbar_arrive(&item_empty[k & 1]);
            if (it.done) break;
            ++k;
            const int nt = (it.t1 - it.t0 + kKeysT - 1) / kKeysT;
            const int n0 = (nt + 1) / 2, n1 = nt - n0;
            const int zkv = it.b * p.Hkv + it.kvh;
            for (int j = 0; j < n0 && ok; ++j) {
                for (int t = 0; t < 2 && ok; ++t) {
                    if (t == 1 && j >= n1) continue;
                    const int key0 = it.t0 + (t == 0 ? j : n0 + j) * kKeysT;
                    const uint32_t vs = nf % VS, vph = (nf / VS) & 1;
                    if (lane == 0) {
                        ok = mbar_wait(&v_empty[vs], vph ^ 1u, kErrWaitProducer, p.err);
                        if (ok) {
                            mbar_arrive_expect_tx(&v_full[vs], L::kTileBytes);
                            #pragma unroll
                            for (int bx = 0; bx < L::kBoxes; ++bx)
                                tma_load_3d(smem + L::kV0 + vs * L::kTileBytes + bx * L::kBoxBytes, &p.tmap_v,
                                            bx * 64, key0, zkv, &v_full[vs]);
                        }
                    }
                    ok = __shfl_sync(0xffffffffu, ok, 0);
                    const uint32_t issued = ok ? 1u : 0u;   // (a fill not issued is not drained)
                    if (ok && key0 + kKeysT > it.len) {
                        // the tile crossing len (at most one per split): zero its rows past len
                        bool landed = true;
                        if (lane == 0) landed = mbar_wait(&v_full[vs], vph, kErrWaitProducer, p.err);
                        landed = __shfl_sync(0xffffffffu, landed, 0);
                        if (landed) {
                            uint8_t* vt = smem + L::kV0 + vs * L::kTileBytes;
                            const int first = max(0, it.len - key0);
                            for (int i = first * 8 + lane; i < kKeysT * 8; i += 32) {   // 16-byte chunks
                                #pragma unroll
                                for (int bx = 0; bx < L::kBoxes; ++bx)
                                    *reinterpret_cast<uint4*>(vt + bx * L::kBoxBytes + i * 16) = make_uint4(0, 0, 0, 0);
                            }
                            fence_proxy_async_smem();
                            __syncwarp();
                            if (lane == 0) mbar_arrive(&v_fix[vs]);
                        } else {
                            ok = false;
                        }
                    }
                    nf += issued;
                }
            }
        }
        // drain: the last fill of each V slot must land before the CTA exits
        if (lane == 0)
            for (uint32_t f = nf >= (uint32_t)VS ? nf - VS : 0; f < nf; ++f)
                mbar_wait_drain(&v_full[f % VS], (f / VS) & 1, p.err);
    } else if (warp == 1) {
        // ================================= MMA issuer =================================
        // Per step j: PV0(j), S0(j+1), PV1(j), S1(j+1) -- the ping-pong order of the
        // prefill kernel; S_t(j+1) overwrites P_t(j) and is issued after PV_t(j).  The
        // first P.V of an item overwrites O and waits until the previous item's merge has
        // read both accumulators.
        if (lane == 0) {
            constexpr uint32_t idesc_s = make_idesc_bf16(kRowsT, kKeysT, 0, 0);
            constexpr uint32_t idesc_pv = make_idesc_bf16(kRowsT, D, 0, 1);
            const uint64_t dq = make_sdesc_sw128(smem_u32(smem + L::kQ0), 16, 1024);
            const uint64_t dk0 = make_sdesc_sw128(smem_u32(smem + L::kK0), 16, 1024);
            const uint64_t dv0 = make_sdesc_sw128(smem_u32(smem + L::kV0), L::kBoxBytes, 1024);
            uint32_t k = 0, fbase = 0, cs0 = 0, cs1 = 0;
            uint32_t nfix = 0;       // bit i: parity of V slot i's next ragged-tile fix
            bool ok = true;
            while (ok) {
                if (!mbar_wait(&item_full[k & 1], (k >> 1) & 1, kErrWaitMma, p.err)) break;
                const MtItem it = info[k & 1];
                mbar_arrive(&item_empty[k & 1]);
                if (it.done) break;
                const int nt = (it.t1 - it.t0 + kKeysT - 1) / kKeysT;
                const int n0 = (nt + 1) / 2, n1 = nt - n0;
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
                    if (++ns == nt) mma_commit(q_empty);   // the item's last read of Q
                };
                auto issue_pv = [&](int t, int j, uint32_t f) -> bool {
                    const uint32_t cs = t == 0 ? cs0 : cs1;
                    if (!mbar_wait(&p_ready[t], (cs + j) & 1, kErrWaitMma, p.err)) return false;
                    if (t == 0 && j == 0 && k > 0 && !mbar_wait(o_free, (k - 1) & 1, kErrWaitMma, p.err))
                        return false;
                    const uint32_t vs = f % VS;
                    if (!mbar_wait(&v_full[vs], (f / VS) & 1, kErrWaitMma, p.err)) return false;
                    const int key0 = it.t0 + (t == 0 ? j : n0 + j) * kKeysT;
                    if (key0 + kKeysT > it.len) {
                        if (!mbar_wait(&v_fix[vs], (nfix >> vs) & 1, kErrWaitMma, p.err)) return false;
                        nfix ^= 1u << vs;
                    }
                    tc_fence_after();
                    const uint64_t b0 = dv0 + (uint64_t)(vs * (L::kTileBytes >> 4));
                    const uint32_t col_s = t == 0 ? L::kColS0 : L::kColS1;
                    const uint32_t dst = tmem + (t == 0 ? L::kColO0 : L::kColO1);
                    #pragma unroll
                    for (int kk = 0; kk < kKeysT / 16; ++kk)
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
                fbase += (uint32_t)nt;
                cs0 += (uint32_t)n0;
                cs1 += (uint32_t)n1;
                ++k;
            }
        }
    } else if (warp == 3) {
        // ================================ publisher =================================
        // Counts each finished partial into its (sequence, KV head, 128-row tile) group with a device-scope
        // release, so that the combine, which reads the count with acquire, can merge the group
        // while the grid is still running.  The softmax warps' writes of the partial happen
        // before their arrivals here (CTA-scope mbarrier release / acquire), so the release
        // covers them; it waits for those writes to land, on this otherwise idle warp.
        if (lane == 0 && p.counted) {
            for (uint32_t k = 0;; ++k) {
                const uint32_t ps = k % kPubSlots;
                if (!mbar_wait(&pub_full[ps], (k / kPubSlots) & 1, kErrWaitConsumer, p.err)) break;
                const int g = pub_group[ps];
                if (g < 0) break;                    // the softmax warps are done
                if (GBATTN_IN_BOUNDS(g, (long long)p.B * p.Hkv * p.n_rt, p.err))
                    counter_add_release(p.group_cnt + g, 1);
                mbar_arrive(&pub_empty[ps]);
            }
        }
    } else if (warp >= kSoftmaxWarp0) {
        // =============================== softmax warps ================================
        const int t = (warp - kSoftmaxWarp0) >> 2;     // slot of this warpgroup
        const int wq = warp & 3;                        // TMEM lane quadrant
        const int r = wq * 32 + lane;                   // row within the item
        const float c = p.scale_log2;
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        const uint32_t t_s = tmem + lane_off + (t == 0 ? L::kColS0 : L::kColS1);
        const uint32_t t_o = tmem + lane_off + (t == 0 ? L::kColO0 : L::kColO1);
        const uint32_t t_o0 = tmem + lane_off + L::kColO0;
        const uint32_t t_o1 = tmem + lane_off + L::kColO1;
        float* ms = xm;              // [2][128] running max per slot
        float* ls = xm + 256;        // [2][128] row sum per slot
        uint32_t k = 0, cs0 = 0, cs1 = 0;
        bool ok = true;
        while (ok) {
            if (!mbar_wait(&item_full[k & 1], (k >> 1) & 1, kErrWaitSoftmax, p.err)) break;
            // read from shared memory where used (few registers); released after the merge
            const MtItem& it = info[k & 1];
            if (it.done) {
                // tell the publisher (all eight arrivals from one thread)
                if (p.counted && warp == kSoftmaxWarp0 && lane == 0 &&
                    mbar_wait(&pub_empty[k % kPubSlots], ((k / kPubSlots) & 1) ^ 1u, kErrWaitSoftmax, p.err)) {
                    pub_group[k % kPubSlots] = -1;
                    for (int i = 0; i < 8; ++i) mbar_arrive(&pub_full[k % kPubSlots]);
                }
                break;
            }
            const int nt = (it.t1 - it.t0 + kKeysT - 1) / kKeysT;
            const int n0 = (nt + 1) / 2, n1 = nt - n0;
            const int n_t = t == 0 ? n0 : n1;           // this slot's key tiles
            const uint32_t cs = t == 0 ? cs0 : cs1;
            const int kv0 = t == 0 ? 0 : n0;
            const int nrows = min(kRowsT, p.R - it.rt * kRowsT);
            const bool warp_rows = wq * 32 < nrows;     // any real row in this warp
            // token of this row and the keys it may see: [t0, lim)
            const int tok = (it.rt * kRowsT + r) % p.Tq;
            const int lim = min(it.t1, it.len - p.Tq + tok + 1);
            float m = -INFINITY, l = 0.f;
            for (int j = 0; j < n_t; ++j) {
                if (!mbar_wait(&s_full[t], (cs + j) & 1, kErrWaitSoftmax, p.err)) { ok = false; break; }
                tc_fence_after();
                if (warp_rows) {
                    const int kbase = it.t0 + (kv0 + j) * kKeysT;
                    uint32_t sr[kKeysT];
                    tmem_ld128(t_s, sr);
                    if (kbase + kKeysT > lim) {
                        #pragma unroll
                        for (int e = 0; e < kKeysT; ++e)
                            if (kbase + e >= lim) sr[e] = __float_as_uint(-INFINITY);
                    }
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
                    const float nb2 = -base;
                    float sum0 = 0.f, sum1 = 0.f;
                    uint32_t pk[kKeysT / 2];
                    #pragma unroll
                    for (int e = 0; e < kKeysT; e += 2) {
                        float a0, a1;
                        fma2(a0, a1, __uint_as_float(sr[e]), __uint_as_float(sr[e + 1]), c, c, nb2, nb2);
                        const float p0 = ex2_approx(a0);
                        const float p1 = ex2_approx(a1);
                        add2(sum0, sum1, p0, p1);
                        pk[e >> 1] = pack_bf16(p0, p1);
                    }
                    tmem_st64(t_s, pk);
                    tmem_wait_st();
                    l = l * corr + (sum0 + sum1);
                    m = m_new;
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
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&p_ready[t]);
            }
            if (!ok) break;
            // ---- end of the item: merge the two slots, write the partial (or final) ----
            // Each warpgroup first waits for its own slot's last P.V; after the meet both
            // accumulators are complete, and warpgroup t merges columns [t D/2, (t+1) D/2).
            if (n_t > 0) {
                if (!mbar_wait(&o_done[t], (cs + n_t - 1) & 1, kErrWaitSoftmax, p.err)) break;
                ms[t * 128 + r] = m;
                ls[t * 128 + r] = l;
            }
            __syncwarp();
            if (lane == 0) {
                // the publisher entry of this item: free once the item kPubSlots back has been
                // counted; claimed before the meet, so no warp arrives on it earlier
                if (p.counted && warp == kSoftmaxWarp0) {
                    if (mbar_wait(&pub_empty[k % kPubSlots], ((k / kPubSlots) & 1) ^ 1u, kErrWaitSoftmax, p.err))
                        pub_group[k % kPubSlots] = (it.b * p.Hkv + it.kvh) * p.n_rt + it.rt;
                }
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
            if (warp_rows) {
                const float m0 = ms[r];
                const float m1 = n1 > 0 ? ms[128 + r] : -INFINITY;
                const float M = fmaxf(m0, m1);
                const float a0 = (m0 == -INFINITY) ? 0.f : ex2_approx(m0 - M);
                const float a1 = (m1 == -INFINITY) ? 0.f : ex2_approx(m1 - M);
                const float lt = a0 * ls[r] + (n1 > 0 ? a1 * ls[128 + r] : 0.f);
                const long long row0 = ((long long)it.b * p.Hkv + it.kvh) * p.R + (long long)it.rt * kRowsT;
                const long long row = row0 + r;
                const bool live = r < nrows &&
                                  GBATTN_IN_BOUNDS(row * p.n_parts + it.s,
                                                   (long long)p.B * p.Hq * p.Tq * p.n_parts, p.err);
                const float inv = lt > 0.f ? 1.f / lt : 0.f;
                #pragma unroll 1
                for (int ch = 0; ch < D / 64; ++ch) {
                    const int col = t * (D / 2) + ch * 32;
                    uint32_t r0[32], r1[32];
                    tmem_ld32(t_o0 + col, r0);
                    if (n1 > 0) tmem_ld32(t_o1 + col, r1);
                    float v[32];
                    #pragma unroll
                    for (int e = 0; e < 32; ++e)
                        v[e] = (a0 * __uint_as_float(r0[e]) + (n1 > 0 ? a1 * __uint_as_float(r1[e]) : 0.f)) * inv;
                    if (!live) continue;
                    if (it.direct) {
                        uint4* dst = reinterpret_cast<uint4*>(p.o + row * D + col);
                        #pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4)
                            dst[q4] = make_uint4(pack_bf16(v[8 * q4 + 0], v[8 * q4 + 1]), pack_bf16(v[8 * q4 + 2], v[8 * q4 + 3]),
                                                 pack_bf16(v[8 * q4 + 4], v[8 * q4 + 5]), pack_bf16(v[8 * q4 + 6], v[8 * q4 + 7]));
                    } else {
                        float4* dst = reinterpret_cast<float4*>(p.ws_o + (row * p.n_parts + it.s) * D + col);
                        #pragma unroll
                        for (int q4 = 0; q4 < 8; ++q4)
                            dst[q4] = make_float4(v[4 * q4], v[4 * q4 + 1], v[4 * q4 + 2], v[4 * q4 + 3]);
                    }
                }
                if (live && t == 0) {
                    const float lse2 = lt > 0.f ? M + __log2f(lt) : -INFINITY;
                    if (it.direct) {
                        if (p.lse != nullptr) p.lse[row] = lse2 * 0.69314718055994531f;
                    } else {
                        p.ws_lse[row * p.n_parts + it.s] = lse2;
                    }
                }
            }
            // both accumulators (and m, l above) may now be overwritten by the next item,
            // and the item entry by the one after it
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(o_free);
                if (p.counted) mbar_arrive(&pub_full[k % kPubSlots]);   // this warp's rows are written
                mbar_arrive(&item_empty[k & 1]);
            }
            cs0 += (uint32_t)n0;
            cs1 += (uint32_t)n1;
            ++k;
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
}

template <int D>
cudaError_t launch_mt(const DecodeTcParams& p, int nsm, cudaStream_t stream) {
    constexpr int smem = Layout<D>::kAlloc;
    static_assert(smem <= 227 * 1024, "shared memory budget");
    cudaError_t err = cudaFuncSetAttribute(decode_mt_kernel<D>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return err;
    err = cudaMemsetAsync(p.counter, 0, (p.counted ? 1 + (size_t)p.B * p.Hkv * p.n_rt : 1) * sizeof(int),
                          stream);
    if (err != cudaSuccess) return err;
    decode_mt_kernel<D><<<min(p.n_items, nsm), kThreads, smem, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_multitoken_tc(const DecodeTcParams& p, int d, int nsm, cudaStream_t stream) {
    if (p.n_items <= 0) return cudaSuccess;
    return d == 128 ? launch_mt<128>(p, nsm, stream) : launch_mt<64>(p, nsm, stream);
}

#ifdef GBATTN_DEBUG_CHECKS
cudaError_t debug_skip_fill_multitoken(int fill) {
    return cudaMemcpyToSymbol(g_skip_k_fill, &fill, sizeof(int));
}
#endif

}  // namespace gbattn
