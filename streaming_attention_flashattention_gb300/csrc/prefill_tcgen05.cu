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

template <int D>
struct PLayout {
    static constexpr int kBoxes = D / 64;
    static constexpr int kTileBytes = kBlockM * D * 2;      // Q, K or V tile
    static constexpr int kBoxBytes = kBlockM * 128;          // one 64-column swizzled box
    static constexpr int kQ0 = 0;
    static constexpr int kK0 = 2 * kTileBytes;               // 2 K slots
    static constexpr int kV0 = 4 * kTileBytes;               // 2 V slots
    static constexpr int kBar = 6 * kTileBytes;
    static constexpr int kNumBars = 16;
    static constexpr int kTmemSlot = kBar + kNumBars * 8;
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
};

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
    const int off = p.Skv - p.Sq;
    const int n_all = (p.Skv + kBlockN - 1) / kBlockN;
    #pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int u = 2 * jj + i;
        t[i].present = u < cnt;
        const int qb = u / p.G, gi = u % p.G;
        t[i].h = kvh * p.G + gi;
        t[i].q0 = qb * kBlockM;
        int n = n_all;
        if (p.causal) {
            const int last_row = min(t[i].q0 + kBlockM, p.Sq) - 1;
            const int keys = min(p.Skv, last_row + off + 1);
            n = (keys + kBlockN - 1) / kBlockN;
        }
        t[i].n_kv = t[i].present ? n : 0;
    }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
prefill_fwd_kernel(const __grid_constant__ PrefillParams p) {
    using L = PLayout<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBar);
    uint64_t* q_full = bars + 0;
    uint64_t* k_full = bars + 1;     // [2]
    uint64_t* k_empty = bars + 3;    // [2]
    uint64_t* v_full = bars + 5;     // [2]
    uint64_t* v_empty = bars + 7;    // [2]
    uint64_t* s_full = bars + 9;     // [2] per Q tile
    uint64_t* p_ready = bars + 11;   // [2] per Q tile
    uint64_t* o_done = bars + 13;    // [2] per Q tile
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kTmemSlot);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    int b, kvh;
    TileDesc td[2];
    pair_tiles(p, blockIdx.x, b, kvh, td);
    const int n_kv_max = max(td[0].n_kv, td[1].n_kv);

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&k_full[i], 1);
            mbar_init(&k_empty[i], 1);
            mbar_init(&v_full[i], 1);
            mbar_init(&v_empty[i], 1);
            mbar_init(&s_full[i], 1);
            mbar_init(&p_ready[i], 4);
            mbar_init(&o_done[i], 1);
        }
        fence_barrier_init();
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
            const uint32_t qbytes = (td[1].present ? 2 : 1) * L::kTileBytes;
            mbar_arrive_expect_tx(q_full, qbytes);
            #pragma unroll
            for (int t = 0; t < 2; ++t) {
                if (!td[t].present) continue;
                #pragma unroll
                for (int bx = 0; bx < L::kBoxes; ++bx)
                    tma_load_3d(smem + L::kQ0 + t * L::kTileBytes + bx * L::kBoxBytes, &p.tmap_q,
                                bx * 64, td[t].q0, b * p.Hq + td[t].h, q_full);
            }
            const int zkv = b * p.Hkv + kvh;
            int filled_k = 0, filled_v = 0;
            bool ok = true;
            for (int j = 0; j < n_kv_max && ok; ++j) {
                const int slot = j & 1;
                const uint32_t ph = (j >> 1) & 1;
                if (!mbar_wait(&k_empty[slot], ph ^ 1u, kErrWaitProducer, p.err)) { ok = false; break; }
                mbar_arrive_expect_tx(&k_full[slot], L::kTileBytes);
                #pragma unroll
                for (int bx = 0; bx < L::kBoxes; ++bx)
                    tma_load_3d(smem + L::kK0 + slot * L::kTileBytes + bx * L::kBoxBytes,
                                &p.tmap_k, bx * 64, j * kBlockN, zkv, &k_full[slot]);
                filled_k = j + 1;
                if (!mbar_wait(&v_empty[slot], ph ^ 1u, kErrWaitProducer, p.err)) { ok = false; break; }
                mbar_arrive_expect_tx(&v_full[slot], L::kTileBytes);
                #pragma unroll
                for (int bx = 0; bx < L::kBoxes; ++bx)
                    tma_load_3d(smem + L::kV0 + slot * L::kTileBytes + bx * L::kBoxBytes,
                                &p.tmap_v, bx * 64, j * kBlockN, zkv, &v_full[slot]);
                filled_v = j + 1;
            }
            // drain: the last fills of each slot must land before the CTA can exit
            mbar_wait(q_full, 0, kErrWaitDrain, p.err);
            for (int j = max(0, filled_k - 2); j < filled_k; ++j)
                mbar_wait(&k_full[j & 1], (j >> 1) & 1, kErrWaitDrain, p.err);
            for (int j = max(0, filled_v - 2); j < filled_v; ++j)
                mbar_wait(&v_full[j & 1], (j >> 1) & 1, kErrWaitDrain, p.err);
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
            const uint32_t k_base = smem_u32(smem + L::kK0);
            const uint32_t v_base = smem_u32(smem + L::kV0);
            const int n0 = td[0].n_kv, n1 = td[1].n_kv;

            auto issue_s = [&](int t, int j) {
                const uint32_t qa = q_base + t * L::kTileBytes;
                const uint32_t kb = k_base + (j & 1) * L::kTileBytes;
                const uint32_t dst = tmem + (t == 0 ? L::kColS0 : L::kColS1);
                #pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * L::kBoxBytes + (kk & 3) * 32;
                    mma_bf16_ss(dst, make_sdesc_sw128(qa + off, 16, 1024),
                                make_sdesc_sw128(kb + off, 16, 1024), idesc_s, kk > 0);
                }
                mma_commit(&s_full[t]);
            };
            auto issue_pv = [&](int t, int j) -> bool {
                if (!mbar_wait(&p_ready[t], j & 1, kErrWaitMma, p.err)) return false;
                tc_fence_after();
                const uint32_t vb = v_base + (j & 1) * L::kTileBytes;
                const uint32_t col_s = t == 0 ? L::kColS0 : L::kColS1;
                const uint32_t dst = tmem + (t == 0 ? L::kColO0 : L::kColO1);
                #pragma unroll
                for (int kk = 0; kk < kBlockN / 16; ++kk)
                    mma_bf16_ts(dst, tmem + col_s + kk * 8,
                                make_sdesc_sw128(vb + kk * 16 * 128, L::kBoxBytes, 1024),
                                idesc_pv, (j > 0 || kk > 0) ? 1u : 0u);
                mma_commit(&o_done[t]);
                return true;
            };

            bool ok = mbar_wait(q_full, 0, kErrWaitMma, p.err);
            tc_fence_after();
            if (ok && n_kv_max > 0) {
                ok = mbar_wait(&k_full[0], 0, kErrWaitMma, p.err);
                tc_fence_after();
                if (ok) {
                    if (n0 > 0) issue_s(0, 0);
                    if (n1 > 0) issue_s(1, 0);
                    mma_commit(&k_empty[0]);
                }
            }
            for (int j = 0; j < n_kv_max && ok; ++j) {
                const bool next = j + 1 < n_kv_max;
                if (!mbar_wait(&v_full[j & 1], (j >> 1) & 1, kErrWaitMma, p.err)) break;
                tc_fence_after();
                if (j < n0 && !issue_pv(0, j)) break;
                if (next) {
                    if (!mbar_wait(&k_full[(j + 1) & 1], ((j + 1) >> 1) & 1, kErrWaitMma, p.err)) break;
                    tc_fence_after();
                    if (j + 1 < n0) issue_s(0, j + 1);
                }
                if (j < n1 && !issue_pv(1, j)) break;
                mma_commit(&v_empty[j & 1]);
                if (next) {
                    if (j + 1 < n1) issue_s(1, j + 1);
                    mma_commit(&k_empty[(j + 1) & 1]);
                }
            }
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
            if (p.causal) lim = min(lim, row + (p.Skv - p.Sq) + 1);
            const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
            const uint32_t t_s = tmem + lane_off + (t == 0 ? L::kColS0 : L::kColS1);
            const uint32_t t_o = tmem + lane_off + (t == 0 ? L::kColO0 : L::kColO1);
            float m = -INFINITY, l = 0.f;
            bool ok = true;
            for (int j = 0; j < me.n_kv; ++j) {
                if (!mbar_wait(&s_full[t], j & 1, kErrWaitSoftmax, p.err)) { ok = false; break; }
                tc_fence_after();
                const int kbase = j * kBlockN;
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
                const float inv = l > 0.f ? 1.f / l : 0.f;
                const bool live = row < p.Sq;
                __nv_bfloat16* orow = p.o + (((long long)b * p.Hq + me.h) * p.Sq + row) * D;
                #pragma unroll 1
                for (int ch = 0; ch < D / 32; ++ch) {
                    uint32_t rr[32];
                    tmem_ld32(t_o + ch * 32, rr);
                    tmem_wait_ld();
                    if (live) {
                        uint4* dst = reinterpret_cast<uint4*>(orow + ch * 32);
                        #pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4) {
                            uint4 w;
                            w.x = pack_bf16(__uint_as_float(rr[8 * q4 + 0]) * inv, __uint_as_float(rr[8 * q4 + 1]) * inv);
                            w.y = pack_bf16(__uint_as_float(rr[8 * q4 + 2]) * inv, __uint_as_float(rr[8 * q4 + 3]) * inv);
                            w.z = pack_bf16(__uint_as_float(rr[8 * q4 + 4]) * inv, __uint_as_float(rr[8 * q4 + 5]) * inv);
                            w.w = pack_bf16(__uint_as_float(rr[8 * q4 + 6]) * inv, __uint_as_float(rr[8 * q4 + 7]) * inv);
                            dst[q4] = w;
                        }
                    }
                }
                if (live && p.lse != nullptr)
                    p.lse[((long long)b * p.Hq + me.h) * p.Sq + row] =
                        l > 0.f ? (m + __log2f(l)) * 0.69314718055994531f : -INFINITY;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, L::kTmemCols);
    }
}

}  // namespace

cudaError_t launch_attn_fwd_bf16(const PrefillParams& p, int d, cudaStream_t stream) {
    if (p.n_pairs <= 0) return cudaSuccess;
    cudaError_t err;
    if (d == 128) {
        constexpr int smem = PLayout<128>::kAlloc;
        err = cudaFuncSetAttribute(prefill_fwd_kernel<128>,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (err != cudaSuccess) return err;
        prefill_fwd_kernel<128><<<p.n_pairs, kThreads, smem, stream>>>(p);
    } else {
        constexpr int smem = PLayout<64>::kAlloc;
        err = cudaFuncSetAttribute(prefill_fwd_kernel<64>,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (err != cudaSuccess) return err;
        prefill_fwd_kernel<64><<<p.n_pairs, kThreads, smem, stream>>>(p);
    }
    return cudaGetLastError();
}

}  // namespace gbattn
