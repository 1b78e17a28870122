// decode_splitkv.cu -- single-token GQA decode over a bf16 KV cache: split-KV partial
// attention streamed at HBM rate, then a log-sum-exp combine.
//
// "ADR-0060: AHBM GQA Fused Attention Kernel (Llama3-70B)":
//   section 5.2 -- decode has T_q = 1 and sees every past key, so only a ragged last tile
//                  is masked; the G query heads of one KV head are stacked into one GEMM
//                  operand so that every K/V tile is read once for all G heads;
//   section 3   -- per tile: S = scale * Q K^T, row max, exp, corr = exp(m - m_new),
//                  l = l * corr + sum P, O = O * corr + P V;
//   section 4   -- partial (m, l, O) of independent KV ranges merge associatively with
//                  m = max(m_a, m_b), weights exp(m_a - m), exp(m_b - m); normalise once;
//   section 2.1 -- each range is one contiguous block of the cache.
//
// GB300 mapping.
//   split kernel: persistent CTAs (one per SM) pull work items (sequence b, KV head,
//   group of row chunks, split s) from a device counter.  One producer warp streams the split's
//   K and V through a 5-stage shared-memory ring with 3-D TMA copies (64 keys x d,
//   128-byte swizzle) and mbarrier handoff.  Four consumer warps take 16 keys each per
//   stage and run S^T = K Q^T and O^T += V^T P^T on mma.sync m16n8k16 with the G <= 8
//   query heads in the N = 8 dimension (the MMA's M dimension is filled by keys, so no
//   lane is wasted on padding heads).  The S^T accumulator fragment is turned into the
//   P^T operand fragment in registers with movmatrix.  Each warp keeps its own running
//   (m, l, O); at the end of a split the four states merge through shared memory and the
//   normalised partial (lse_s, O_s / l_s) goes to the workspace; a group with a single
//   split writes its final O and LSE directly.
//   Multi-token decode (T_q > 1) has G * T_q query rows per KV head, in chunks of 8.  An
//   item then takes NCI = 2 or 4 chunks at once, so each split's K and V are read from HBM
//   once for all rows instead of once per chunk.  Eight consumer warps split every stage
//   into 4 key slices x 2 halves of the item's chunks; a warp's chunks sit side by side in
//   the MMA N dimension, so each K and V^T fragment it builds feeds one MMA per chunk.
//   NCI = 1 is the single-token case above.
//   Single-launch mode (single-token items that all fit in one wave): no combine kernel.
//   Each finished split counts itself into a per-(b, KV head, row chunk) counter, and the
//   CTA that completes the group folds all of its partials into the final O and LSE -- the
//   data-driven merge of "ADR-0060" section 4.3, without a grid-wide barrier.  For small
//   batches this saves the second launch; for large ones the fence and atomic at every
//   split end cost more than the launch, so they use the combine kernel.
//   combine kernel: one thread per (b, query head, 4 output columns) folds the partials of
//   the splits.  It is launched with programmatic dependent launch: its CTAs are
//   scheduled while the split kernel drains and wait on the device (griddepcontrol.wait)
//   for the partials, so no launch gap sits between the two.  Keeping the merge out of the
//   split kernel keeps fences and atomics off the consumer warps, whose stalls would stop
//   the TMA ring.
//   Decode is HBM bound (8 flop per byte of KV), so these contractions stay on the
//   warp-level tensor path; the streaming design is what sets the speed.
#include "common.cuh"
#include "kernels.h"
#include "decode_splits.cuh"

namespace gbattn {

namespace {

constexpr int kKeysPerStage = 64;
// Warps and ring depth per kind of work item.  Single-token items (NCI = 1): 4 consumer
// warps of 16 keys each and a 5-stage ring, one CTA per SM -- HBM bound.  Multi-token
// items carry NCI times the math per byte of K/V: 8 consumer warps (4 key slices x 2
// halves of the item's chunks) so that each warp holds fewer chunks' state and more warps
// hide the MMA and shuffle latencies; the ring drops to 4 stages to make room for their
// merge buffers.  Single-launch calls with more items than SMs run two CTAs per SM with
// 2-stage rings (kTwo): while one CTA folds a finished group's partials, the other keeps
// streaming.
template <int NCI, bool kTwo = false>
struct Cfg {
    static constexpr int kCW = NCI == 1 ? 4 : 8;           // consumer warps
    static constexpr int kThreads = (kCW + 1) * 32;
    static constexpr int kStages = kTwo ? 2 : (NCI == 1 ? 5 : 4);
    static constexpr int kPerSM = kTwo ? 2 : 1;             // resident CTAs per SM
};
constexpr int kHeads = 8;                  // query heads per work item (MMA N)
constexpr int kPubSlots = 4;               // publisher ring entries (finished partials)
#ifdef GBATTN_DEBUG_CHECKS
// Test hook of the debug build: CTA 0 of the grid does not issue the stage fill (K, V and Q of 64 keys) with this index
// (counted over the CTA's fills; -1: none).  The fill's barrier then never completes, the wait
// for it runs out after its time limit and records its code in the error word, and every role
// of every CTA leaves through its give-up exit.  Set by attn_debug_skip_fill.
__device__ int g_skip_k_fill = -1;
#endif

// Single-token instances that count their partials (for the combine's per-group wait) have a
// publisher warp after the producer: the consumers hand it each finished partial and it
// issues the device-scope release of the count, off the streaming path.
template <int NCI, bool kFused>
constexpr int split_threads() { return Cfg<NCI>::kThreads + ((NCI == 1 && !kFused) ? 32 : 0); }

struct StageInfo {
    int b, kvh, hc, s;            // s: the item's partial slot (split * pieces + piece)
    int tile, ntok, last, done;
    int n_ne;                     // non-empty splits of the sequence
    int key0;                     // first key of this tile
    int len;                      // keys of the sequence
    int direct;                   // the item is the row's only partial: write O and LSE
};

template <int D, int NCI, bool kTwo = false>
struct Layout {
    static constexpr int kStages = Cfg<NCI, kTwo>::kStages;
    static constexpr int kConsumerWarps = Cfg<NCI>::kCW;
    static constexpr int kBoxes = D / 64;                       // 64-element swizzle boxes
    static constexpr int kKBytes = kKeysPerStage * D * 2;       // K tile
    static constexpr int kVBytes = kKeysPerStage * D * 2;
    static constexpr int kQBytes = kHeads * NCI * D * 2;        // 8 query rows per chunk
    static constexpr int kStageBytes = kKBytes + kVBytes + kQBytes;   // multiple of 1024
    static constexpr int kRingBytes = kStages * kStageBytes;
    static constexpr int kInfoOff = kRingBytes;
    static constexpr int kBarOff = kInfoOff + kStages * (int)sizeof(StageInfo);
    static constexpr int kNumBars = 2 * kStages + 2;
    static constexpr int kRedMOff = kBarOff + kNumBars * 8;
    static constexpr int kRedLOff = kRedMOff + kConsumerWarps * kHeads * 4;
    static constexpr int kRedOOff = kRedLOff + kConsumerWarps * kHeads * 4;
    static constexpr int kFusedOff = kRedOOff + kConsumerWarps * kHeads * D * 4;  // sync_c, flag
    static constexpr int kPubOff = kFusedOff + 16;      // publisher ring: full, empty, group
    static constexpr int kBytes = kPubOff + kPubSlots * (8 + 8 + 4);
    static constexpr int kAlloc = kBytes + 1024;                // slack for 1024-B alignment
    static_assert(kStageBytes % 1024 == 0, "stage must keep 1024-byte alignment");
};

// 16-byte chunk `chunk` of row `row` inside a 128-byte-swizzled box.
__device__ __forceinline__ uint32_t sw128(uint32_t box, int row, int chunk) {
    return box + (uint32_t)row * 128u + ((uint32_t)(chunk ^ (row & 7)) << 4);
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 r;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "r"(addr));
    return r;
}

__device__ __forceinline__ uint32_t word(const uint4& v, int i) {
    return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// bf16 element e of x (low 16 bits) and of y (high 16 bits) packed into one register.
__device__ __forceinline__ uint32_t pair_elem(const uint4& x, const uint4& y, int e) {
    return __byte_perm(word(x, e >> 1), word(y, e >> 1), (e & 1) ? 0x7632 : 0x5410);
}

__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

// Final output of one query row: `per` consecutive columns of O (bf16) starting at
// d0, plus the LSE (natural log) from its log2 value when `with_lse`.
template <int D, int per>
__device__ __forceinline__ void store_final(const DecodeParams& p, long long row, int d0,
                                            const float* ov, bool with_lse, float lse2) {
    if (!GBATTN_IN_BOUNDS(row, (long long)p.B * p.Hq * p.Tq, p.err)) return;
    __nv_bfloat16* dst = p.o + row * D + d0;
    if constexpr (per % 8 == 0) {
        #pragma unroll
        for (int i = 0; i < per; i += 8) {
            uint4 w;
            w.x = pack_bf16(ov[i + 0], ov[i + 1]); w.y = pack_bf16(ov[i + 2], ov[i + 3]);
            w.z = pack_bf16(ov[i + 4], ov[i + 5]); w.w = pack_bf16(ov[i + 6], ov[i + 7]);
            *reinterpret_cast<uint4*>(dst + i) = w;
        }
    } else {
        uint2 w;
        w.x = pack_bf16(ov[0], ov[1]); w.y = pack_bf16(ov[2], ov[3]);
        *reinterpret_cast<uint2*>(dst) = w;
    }
    if (with_lse && p.lse != nullptr) p.lse[row] = lse2 * 0.69314718055994531f;
}

// Final O (columns [d0, d0 + per)) and LSE of one query row from the n_ne partials in
// the workspace: O = sum_s w_s O_s / sum_s w_s, w_s = 2^(lse_s - max lse) ("ADR-0060"
// section 4), 8 partials loaded per batch; partials with lse = -inf (a row that saw no key
// of that split) weigh nothing.
template <int D, int per>
__device__ __forceinline__ void fold_partials(const DecodeParams& p, long long row, int d0,
                                              int n_ne, bool with_lse) {
    if (!GBATTN_IN_BOUNDS(row, (long long)p.B * p.Hq * p.Tq, p.err) ||
        !GBATTN_IN_BOUNDS(n_ne - 1, p.n_parts, p.err))
        return;
    const float* lse_s = p.ws_lse + row * p.n_parts;
    const float* o_s = p.ws_o + row * p.n_parts * D + d0;
    constexpr int kChunk = 8;
    float M = -INFINITY, Ltot = 0.f, acc[per];
    #pragma unroll
    for (int u = 0; u < per; ++u) acc[u] = 0.f;
    for (int s0 = 0; s0 < n_ne; s0 += kChunk) {
        float ls[kChunk];
        float4 ox[kChunk][per / 4];
        #pragma unroll
        for (int i = 0; i < kChunk; ++i) {
            const bool in = s0 + i < n_ne;
            ls[i] = in ? __ldcg(lse_s + s0 + i) : -INFINITY;
            #pragma unroll
            for (int e = 0; e < per / 4; ++e)
                ox[i][e] = in ? __ldcg(reinterpret_cast<const float4*>(o_s + (long long)(s0 + i) * D) + e)
                              : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        float Mc = M;
        #pragma unroll
        for (int i = 0; i < kChunk; ++i) Mc = fmaxf(Mc, ls[i]);
        const float sc = (M == -INFINITY) ? 0.f : ex2_approx(M - Mc);
        Ltot *= sc;
        #pragma unroll
        for (int u = 0; u < per; ++u) acc[u] *= sc;
        #pragma unroll
        for (int i = 0; i < kChunk; ++i) {
            if (ls[i] == -INFINITY) continue;
            const float w = ex2_approx(ls[i] - Mc);
            Ltot += w;
            #pragma unroll
            for (int e = 0; e < per / 4; ++e) {
                acc[4 * e] += w * ox[i][e].x; acc[4 * e + 1] += w * ox[i][e].y;
                acc[4 * e + 2] += w * ox[i][e].z; acc[4 * e + 3] += w * ox[i][e].w;
            }
        }
        M = Mc;
    }
    const float inv = Ltot > 0.f ? 1.f / Ltot : 0.f;
    #pragma unroll
    for (int u = 0; u < per; ++u) acc[u] *= inv;
    store_final<D, per>(p, row, d0, acc, with_lse, Ltot > 0.f ? M + __log2f(Ltot) : -INFINITY);
}

// The merge of a row's partials ("ADR-0060" section 4): O = sum_s w_s O_s / sum_s w_s with
// w_s = 2^(lse_s - max lse) over the non-empty splits (every piece of a split is a partial of
// its own).  Each (row, 4 output columns) piece of the output is shared by p.combine_lanes
// adjacent lanes c (a power of two, at most 32): lane j merges partials [8 j, 8 j + 8) with
// all its loads in flight at once, and the lanes' (max, sum, O) states are then merged with
// shuffles -- one round of partial loads instead of one per 8.  This is lane j's share for
// columns [4 cg, 4 cg + 4) of `row`, which has n_parts partials; every lane of the warp
// calls it (inactive ones with active = false), since all take part in the shuffles.
template <int D>
__device__ __forceinline__ void merge_columns(const DecodeParams& p, long long row, int cg, int j,
                                              int n_parts, bool active) {
    constexpr int kChunk = 8;
    const int c = p.combine_lanes;
    const bool merge = active && n_parts > 1 &&   // (one partial: the split kernel wrote the row)
                       GBATTN_IN_BOUNDS(row, (long long)p.B * p.Hq * p.Tq, p.err) &&
                       GBATTN_IN_BOUNDS(n_parts - 1, p.n_parts, p.err);
    float M = -INFINITY, L = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (merge) {
        const float* lse_s = p.ws_lse + row * p.n_parts;
        const float* o_s = p.ws_o + row * p.n_parts * D + cg * 4;
        const int s0 = j * kChunk;
        float ls[kChunk];
        float4 ox[kChunk];
        #pragma unroll
        for (int i = 0; i < kChunk; ++i) {
            const bool in = s0 + i < n_parts;
            ls[i] = in ? __ldcg(lse_s + s0 + i) : -INFINITY;
            ox[i] = in ? __ldcg(reinterpret_cast<const float4*>(o_s + (long long)(s0 + i) * D))
                       : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        #pragma unroll
        for (int i = 0; i < kChunk; ++i) M = fmaxf(M, ls[i]);
        #pragma unroll
        for (int i = 0; i < kChunk; ++i) {
            if (ls[i] == -INFINITY) continue;     // a split (or piece) this row saw no key of
            const float w = ex2_approx(ls[i] - M);
            L += w;
            acc.x += w * ox[i].x; acc.y += w * ox[i].y; acc.z += w * ox[i].z; acc.w += w * ox[i].w;
        }
    }
    // merge the c lanes' states: (M, L, acc) with L and acc relative to 2^M
    for (int off = 1; off < c; off <<= 1) {
        const float Mo = __shfl_xor_sync(0xffffffffu, M, off);
        const float Lo = __shfl_xor_sync(0xffffffffu, L, off);
        float4 ao;
        ao.x = __shfl_xor_sync(0xffffffffu, acc.x, off);
        ao.y = __shfl_xor_sync(0xffffffffu, acc.y, off);
        ao.z = __shfl_xor_sync(0xffffffffu, acc.z, off);
        ao.w = __shfl_xor_sync(0xffffffffu, acc.w, off);
        const float Mn = fmaxf(M, Mo);
        const float a = (M == -INFINITY) ? 0.f : ex2_approx(M - Mn);
        const float bo = (Mo == -INFINITY) ? 0.f : ex2_approx(Mo - Mn);
        L = L * a + Lo * bo;
        acc.x = acc.x * a + ao.x * bo; acc.y = acc.y * a + ao.y * bo;
        acc.z = acc.z * a + ao.z * bo; acc.w = acc.w * a + ao.w * bo;
        M = Mn;
    }
    if (!merge || j != 0) return;
    const float inv = L > 0.f ? 1.f / L : 0.f;
    uint2 packed;
    packed.x = pack_bf16(acc.x * inv, acc.y * inv);
    packed.y = pack_bf16(acc.z * inv, acc.w * inv);
    *reinterpret_cast<uint2*>(p.o + row * D + cg * 4) = packed;
    if (cg == 0 && p.lse != nullptr)
        p.lse[row] = L > 0.f ? (M + __log2f(L)) * 0.69314718055994531f : -INFINITY;
}

// Partials of a row of sequence b: pieces of its non-empty splits.
__device__ __forceinline__ int row_partials(const DecodeParams& p, int b) {
    int len = __ldg(&p.kv_lens[b]);
    len = max(0, min(len, p.Lmax));
    return nonempty_splits(len, splits_for(len, p.fixed_splits, p.auto_floor)) * p.pieces;
}

template <int D, int NCI, bool kFused, bool kTwo = false>
__global__ void __launch_bounds__(split_threads<NCI, kFused>(), (Cfg<NCI, kTwo>::kPerSM))
decode_split_kernel(const __grid_constant__ DecodeParams p) {
    static_assert(!kFused || NCI == 1, "single-launch mode is for single-token items");
    static_assert(!kTwo || kFused, "two CTAs per SM: single-launch calls only");
    using L = Layout<D, NCI, kTwo>;
    constexpr int kConsumerWarps = Cfg<NCI>::kCW;
    constexpr int kStages = Cfg<NCI, kTwo>::kStages;
    constexpr int W = kConsumerWarps / NCI;       // consumer warps per row chunk
    constexpr int kKeysPerWarp = kKeysPerStage / W;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    StageInfo* info = reinterpret_cast<StageInfo*>(smem + L::kInfoOff);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
    uint64_t* full = bars;                   // [kStages] producer -> consumers (TMA bytes)
    uint64_t* empty = bars + kStages;        // [kStages] consumers -> producer (one per warp)
    uint64_t* sync_a = bars + 2 * kStages;   // consumer-warp rendezvous at a split's end
    uint64_t* sync_b = sync_a + 1;
    float* red_m = reinterpret_cast<float*>(smem + L::kRedMOff);
    float* red_l = reinterpret_cast<float*>(smem + L::kRedLOff);
    float* red_o = reinterpret_cast<float*>(smem + L::kRedOOff);
    uint64_t* sync_c = reinterpret_cast<uint64_t*>(smem + L::kFusedOff);   // single-launch mode
    int* last_flag = reinterpret_cast<int*>(smem + L::kFusedOff + 8);
    constexpr bool kPub = NCI == 1 && !kFused;                              // publisher warp
    uint64_t* pub_full = reinterpret_cast<uint64_t*>(smem + L::kPubOff);  // [kPubSlots]
    uint64_t* pub_empty = pub_full + kPubSlots;                             // [kPubSlots]
    int* pub_group = reinterpret_cast<int*>(pub_empty + kPubSlots);         // [kPubSlots]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kConsumerWarps);
        }
        mbar_init(sync_a, kConsumerWarps);
        mbar_init(sync_b, kConsumerWarps);
        if constexpr (kFused) mbar_init(sync_c, kConsumerWarps);
        if constexpr (kPub) {
            for (int i = 0; i < kPubSlots; ++i) {
                mbar_init(&pub_full[i], 1);
                mbar_init(&pub_empty[i], 1);
            }
        }
        fence_barrier_init();
    }
    __syncthreads();

    if (warp == kConsumerWarps) {
        // ============================== producer warp ==============================
        if (lane == 0) {
            prefetch_tensormap(&p.tmap_k);
            prefetch_tensormap(&p.tmap_v);
            prefetch_tensormap(&p.tmap_q);
            int stage = 0;
            uint32_t phase = 0;
            uint32_t filled = 0, fill_parity = 0;   // per-stage bits for the exit drain
            bool ok = true;
#ifdef GBATTN_DEBUG_CHECKS
            int nfill = 0;                          // stage fills so far (the test hook)
#endif
            // Items are pulled from a device counter, so a CTA that finishes early takes
            // more (a static round-robin measured slower even for equal-size splits).
            for (int item = atomicAdd(p.counter, 1); ok && item < p.n_items;
                 item = atomicAdd(p.counter, 1)) {
                // order: row chunk innermost, then split, then KV head, then sequence,
                // then piece (guided pieces: every split's large first piece before the
                // small ones).  The row chunks of one split (several when G * Tq > 8) read
                // the same K/V tiles and run side by side, so all but the first pass hit L2.
                int rem = item;
                const int hc = rem % p.n_hg; rem /= p.n_hg;         // chunk group
#if GBATTN_GUIDED_PIECES
                const int s = rem % p.n_slots; rem /= p.n_slots;
                const int kvh = rem % p.Hkv; rem /= p.Hkv;
                const int b = rem % p.B;
                const int pc = rem / p.B;                           // piece of the split
#else
                const int pc = rem % p.pieces; rem /= p.pieces;     // piece of the split
                const int s = rem % p.n_slots; rem /= p.n_slots;
                const int kvh = rem % p.Hkv; rem /= p.Hkv;
                const int b = rem;
#endif
                int len = __ldg(&p.kv_lens[b]);
                len = max(0, min(len, p.Lmax));
                const int nb = splits_for(len, p.fixed_splits, p.auto_floor);
                if (s >= nb) continue;
                const int n_ne = nonempty_splits(len, nb);
                // rows of this item: the KV head's G * Tq query rows (head-major, token
                // minor), 8 per chunk, NCI chunks per group
                const long long row0 = ((long long)b * p.Hkv + kvh) * p.R + hc * (kHeads * NCI);
                const int gcnt = min(kHeads * NCI, p.R - hc * (kHeads * NCI));
                if (s >= n_ne) {
                    // empty split: no partial.  A sequence with no keys at all gets
                    // O = 0, LSE = -inf from its split 0.
                    if (s == 0 && pc == 0) {
                        for (int g = 0; g < gcnt; ++g) {
                            if (!GBATTN_IN_BOUNDS(row0 + g, (long long)p.B * p.Hq * p.Tq, p.err)) continue;
                            uint4* dst = reinterpret_cast<uint4*>(p.o + (row0 + g) * D);
                            for (int e = 0; e < D / 8; ++e) dst[e] = make_uint4(0, 0, 0, 0);
                            if (p.lse != nullptr) p.lse[row0 + g] = -INFINITY;
                        }
                    }
                    continue;
                }
                int t0, t1;
                split_range(len, nb, s, t0, t1);
#if GBATTN_GUIDED_PIECES
                piece_range_guided(t0, t1, p.pieces, pc, t0, t1);
#else
                piece_range(t0, t1, p.pieces, pc, t0, t1);
#endif
                const int part = s * p.pieces + pc;
                if (t0 >= t1) {
                    // an empty piece of a non-empty split: a partial that weighs nothing
                    for (int g = 0; g < gcnt; ++g)
                        if (GBATTN_IN_BOUNDS((row0 + g) * p.n_parts + part, (long long)p.B * p.Hq * p.Tq * p.n_parts, p.err))
                            p.ws_lse[(row0 + g) * p.n_parts + part] = -INFINITY;
                    if (p.counted && GBATTN_IN_BOUNDS(((long long)b * p.Hkv + kvh) * p.n_hg + hc,
                                                      (long long)p.B * p.Hkv * p.n_hg, p.err))
                        counter_add_release(p.group_cnt + ((long long)b * p.Hkv + kvh) * p.n_hg + hc, 1);
                    continue;
                }
                const int ntiles = (t1 - t0 + kKeysPerStage - 1) / kKeysPerStage;
                const int zkv = b * p.Hkv + kvh;
                for (int tile = 0; tile < ntiles; ++tile) {
                    if (!mbar_wait(&empty[stage], phase ^ 1u, kErrWaitProducer, p.err)) {
                        ok = false;
                        break;
                    }
                    const int y = t0 + tile * kKeysPerStage;
                    StageInfo& si = info[stage];
                    si.b = b; si.kvh = kvh; si.hc = hc; si.s = part;
                    si.tile = tile;
                    si.ntok = min(kKeysPerStage, t1 - y);
                    si.last = (tile == ntiles - 1);
                    si.done = 0;
                    si.n_ne = n_ne;
                    si.key0 = y;
                    si.len = len;
                    si.direct = (n_ne == 1 && p.pieces == 1) ? 1 : 0;
                    uint8_t* st = smem + stage * L::kStageBytes;
                    // single-token items load Q with their first tile only; stacked
                    // multi-token items re-read it from every stage (no registers to keep
                    // NCI chunks of it)
                    const bool with_q = tile == 0 || NCI > 1;
                    const uint32_t bytes = L::kKBytes + L::kVBytes + (with_q ? L::kQBytes : 0);
#ifdef GBATTN_DEBUG_CHECKS
                    if (blockIdx.x == 0 && nfill++ == g_skip_k_fill) {
                        // left out: the stage's barrier never completes (and is not drained)
                    } else
#endif
                    {
                        mbar_arrive_expect_tx(&full[stage], bytes);
                        #pragma unroll
                        for (int bx = 0; bx < L::kBoxes; ++bx) {
                            tma_load_3d(st + bx * (kKeysPerStage * 128), &p.tmap_k, bx * 64, y, zkv,
                                        &full[stage]);
                            tma_load_3d(st + L::kKBytes + bx * (kKeysPerStage * 128), &p.tmap_v,
                                        bx * 64, y, zkv, &full[stage]);
                        }
                        if (with_q) {
                            #pragma unroll
                            for (int cq = 0; cq < NCI; ++cq)
                                #pragma unroll
                                for (int bx = 0; bx < L::kBoxes; ++bx)
                                    tma_load_3d(st + L::kKBytes + L::kVBytes + bx * (kHeads * NCI * 128) +
                                                    cq * (kHeads * 128),
                                                &p.tmap_q, bx * 64, (int)row0 + cq * kHeads, 0, &full[stage]);
                        }
                        filled |= 1u << stage;
                        fill_parity = (fill_parity & ~(1u << stage)) | (phase << stage);
                    }
                    if (++stage == kStages) { stage = 0; phase ^= 1u; }
                }
            }
            if (ok) {
                // end-of-work marker for the consumers
                if (mbar_wait(&empty[stage], phase ^ 1u, kErrWaitProducer, p.err)) {
                    info[stage].done = 1;
                    mbar_arrive(&full[stage]);
                    // the marker is this stage's newest phase: the drain must wait for it,
                    // not for the older fill (whose parity the barrier has now passed twice)
                    filled |= 1u << stage;
                    fill_parity = (fill_parity & ~(1u << stage)) | (phase << stage);
                }
            }
            // this CTA takes no more work: let the combine grid start being scheduled
            asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
            // drain: never leave the CTA with a TMA copy still writing its shared memory
            for (int i = 0; i < kStages; ++i)
                if (filled & (1u << i)) mbar_wait_drain(&full[i], (fill_parity >> i) & 1u, p.err);
        }
    } else if (warp == kConsumerWarps + 1) {
        // ============================= publisher warp ==============================
        // Counts each finished partial into its (sequence, KV head) group with a device-scope
        // release: the consumers' writes of the partial happen before their hand-over here
        // (CTA-scope mbarrier release / acquire), so the release covers them, and the
        // combine, which reads the count with acquire, sees the whole partial.  The release
        // waits for those writes to land; on this warp that costs the stream nothing.
        if constexpr (kPub) {
            if (lane == 0 && p.counted) {
                for (uint32_t k = 0;; ++k) {
                    const uint32_t ps = k % kPubSlots;
                    if (!mbar_wait(&pub_full[ps], (k / kPubSlots) & 1, kErrWaitConsumer, p.err)) break;
                    const int g = pub_group[ps];
                    if (g < 0) break;                    // the consumers are done
                    if (GBATTN_IN_BOUNDS(g, (long long)p.B * p.Hkv * p.n_hg, p.err))
                        counter_add_release(p.group_cnt + g, 1);
                    mbar_arrive(&pub_empty[ps]);
                }
            }
        }
    } else if constexpr (NCI == 1) {
        // ======================= consumer warps (single token) ======================
        const int g = lane >> 2, c = lane & 3;
        const uint32_t ring = smem_u32(smem);
        const float scale_log2 = p.scale_log2;
        uint4 qf[D / 32];
        float acc[D / 16][4];
        float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
        int lim0 = 0, lim1 = 0;
        int stage = 0;
        uint32_t phase = 0, sync_phase = 0, sync_c_phase = 0;
        const int cw = warp / W;                 // row chunk of this warp within the group
        const int kp0 = (warp % W) * kKeysPerWarp;   // this warp's first key within a stage
        int gcnt = 0;                            // rows of this warp's chunk (<= 0: none)
        uint32_t n_pub = 0;                      // partials handed to the publisher (thread 0)
        // thread 0: hand group g (or -1: no more) to the publisher warp
        auto publish = [&](int g) {
            const uint32_t ps = n_pub % kPubSlots;
            if (mbar_wait(&pub_empty[ps], ((n_pub / kPubSlots) & 1) ^ 1u, kErrWaitConsumer, p.err)) {
                pub_group[ps] = g;
                mbar_arrive(&pub_full[ps]);
            }
            ++n_pub;
        };
        while (true) {
            if (!mbar_wait(&full[stage], phase, kErrWaitConsumer, p.err)) break;
            const StageInfo si = info[stage];
            if (si.done) break;
            const uint32_t kbox = ring + stage * L::kStageBytes;
            const uint32_t vbox = kbox + L::kKBytes;
            const uint32_t qbox = vbox + L::kVBytes;
            const int hc = si.hc * NCI + cw;         // this warp's row chunk in the KV head
            if (si.tile == 0) {
                gcnt = min(kHeads, p.R - hc * kHeads);
                #pragma unroll
                for (int s = 0; s < D / 32; ++s) {
                    uint4 z = make_uint4(0, 0, 0, 0);
                    if (g < gcnt)
                        z = lds128(sw128(qbox + (s >> 1) * (kHeads * NCI * 128), cw * kHeads + g,
                                         2 * c + (s & 1)));
                    qf[s] = z;
                }
                m0 = m1 = -INFINITY;
                l0 = l1 = 0.f;
                // causal limit of my two columns (rows hc*8 + 2c, +1): token t of the
                // Tq new ones sees keys < len - Tq + t + 1 (all keys when Tq = 1)
                lim0 = si.len - p.Tq + ((hc * kHeads + 2 * c) % p.Tq) + 1;
                lim1 = si.len - p.Tq + ((hc * kHeads + 2 * c + 1) % p.Tq) + 1;
                #pragma unroll
                for (int mt = 0; mt < D / 16; ++mt)
                    acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.f;
            }
            const int R0 = kp0;                      // this warp's 16 keys within the stage
            const int nvalid = min(16, si.ntok - R0);
            if (nvalid > 0) {
                // ---- S^T[16 keys x 8 heads] = K Q^T ----
                float sc[4] = {0.f, 0.f, 0.f, 0.f};
                #pragma unroll
                for (int s = 0; s < D / 32; ++s) {
                    const uint32_t kb = kbox + (s >> 1) * (kKeysPerStage * 128);
                    const int ch = 2 * c + (s & 1);
                    const uint4 k0 = lds128(sw128(kb, R0 + g, ch));
                    const uint4 k1 = lds128(sw128(kb, R0 + g + 8, ch));
                    mma16816(sc, k0.x, k1.x, k0.y, k1.y, qf[s].x, qf[s].y);
                    mma16816(sc, k0.z, k1.z, k0.w, k1.w, qf[s].z, qf[s].w);
                }
                // ---- online softmax over the keys (columns = heads 2c, 2c+1) ----
                const bool v_lo = g < nvalid, v_hi = g + 8 < nvalid;
                if (p.Tq == 1) {
                    sc[0] = v_lo ? sc[0] * scale_log2 : -INFINITY;
                    sc[1] = v_lo ? sc[1] * scale_log2 : -INFINITY;
                    sc[2] = v_hi ? sc[2] * scale_log2 : -INFINITY;
                    sc[3] = v_hi ? sc[3] * scale_log2 : -INFINITY;
                } else {
                    const int key_lo = si.key0 + R0 + g, key_hi = key_lo + 8;
                    sc[0] = (v_lo && key_lo < lim0) ? sc[0] * scale_log2 : -INFINITY;
                    sc[1] = (v_lo && key_lo < lim1) ? sc[1] * scale_log2 : -INFINITY;
                    sc[2] = (v_hi && key_hi < lim0) ? sc[2] * scale_log2 : -INFINITY;
                    sc[3] = (v_hi && key_hi < lim1) ? sc[3] * scale_log2 : -INFINITY;
                }
                float mx0 = fmaxf(sc[0], sc[2]), mx1 = fmaxf(sc[1], sc[3]);
                #pragma unroll
                for (int w = 4; w < 32; w <<= 1) {
                    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, w));
                    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, w));
                }
                const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
                const float base0 = mn0 == -INFINITY ? 0.f : mn0;
                const float base1 = mn1 == -INFINITY ? 0.f : mn1;
                const float corr0 = ex2_approx(m0 - base0), corr1 = ex2_approx(m1 - base1);
                const float p00 = ex2_approx(sc[0] - base0), p01 = ex2_approx(sc[1] - base1);
                const float p10 = ex2_approx(sc[2] - base0), p11 = ex2_approx(sc[3] - base1);
                l0 = l0 * corr0 + p00 + p10;
                l1 = l1 * corr1 + p01 + p11;
                m0 = mn0;
                m1 = mn1;
                #pragma unroll
                for (int mt = 0; mt < D / 16; ++mt) {
                    acc[mt][0] *= corr0; acc[mt][1] *= corr1;
                    acc[mt][2] *= corr0; acc[mt][3] *= corr1;
                }
                // ---- P^T operand: transpose the (key x head) 8x8 blocks in registers ----
                const uint32_t b0 = movmatrix_trans(pack_bf16(p00, p01));
                const uint32_t b1 = movmatrix_trans(pack_bf16(p10, p11));
                // ---- O^T[d x 8 heads] += V^T P^T ----
                const int tk[4] = {2 * c, 2 * c + 1, 2 * c + 8, 2 * c + 9};
                if constexpr (D == 128) {
                    uint4 vv[4][2];
                    #pragma unroll
                    for (int i = 0; i < 4; ++i)
                        #pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            uint4 z = make_uint4(0, 0, 0, 0);
                            if (tk[i] < nvalid) z = lds128(sw128(vbox + h * (kKeysPerStage * 128), R0 + tk[i], g));
                            vv[i][h] = z;
                        }
                    #pragma unroll
                    for (int mt = 0; mt < 8; ++mt)
                        mma16816(acc[mt], pair_elem(vv[0][0], vv[1][0], mt),
                                 pair_elem(vv[0][1], vv[1][1], mt),
                                 pair_elem(vv[2][0], vv[3][0], mt),
                                 pair_elem(vv[2][1], vv[3][1], mt), b0, b1);
                } else {
                    uint4 vv[4];
                    #pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        uint4 z = make_uint4(0, 0, 0, 0);
                        if (tk[i] < nvalid) z = lds128(sw128(vbox, R0 + tk[i], g));
                        vv[i] = z;
                    }
                    #pragma unroll
                    for (int mt = 0; mt < 4; ++mt)
                        mma16816(acc[mt], pair_elem(vv[0], vv[1], mt),
                                 pair_elem(vv[0], vv[1], mt + 4),
                                 pair_elem(vv[2], vv[3], mt),
                                 pair_elem(vv[2], vv[3], mt + 4), b0, b1);
                }
            }
        
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[stage]);

            if (si.last) {
                // ---- merge the four warps' states; write the split's partial ----
                float lr0 = l0, lr1 = l1;
                #pragma unroll
                for (int w = 4; w < 32; w <<= 1) {
                    lr0 += __shfl_xor_sync(0xffffffffu, lr0, w);
                    lr1 += __shfl_xor_sync(0xffffffffu, lr1, w);
                }
                if (g == 0) {
                    red_m[warp * kHeads + 2 * c] = m0;
                    red_m[warp * kHeads + 2 * c + 1] = m1;
                    red_l[warp * kHeads + 2 * c] = lr0;
                    red_l[warp * kHeads + 2 * c + 1] = lr1;
                }
                float* ro = red_o + warp * kHeads * D;
                #pragma unroll
                for (int mt = 0; mt < D / 16; ++mt) {
                    const int d_lo = (D == 128) ? 8 * g + mt : 8 * g + mt;
                    const int d_hi = (D == 128) ? 64 + 8 * g + mt : 8 * g + 4 + mt;
                    ro[(2 * c) * D + d_lo] = acc[mt][0];
                    ro[(2 * c + 1) * D + d_lo] = acc[mt][1];
                    ro[(2 * c) * D + d_hi] = acc[mt][2];
                    ro[(2 * c + 1) * D + d_hi] = acc[mt][3];
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(sync_a);
                if (!mbar_wait(sync_a, sync_phase, kErrWaitConsumer, p.err)) break;
                // rows of the group: NCI chunks x 8 heads, each finished by kThrPerRow
                // threads from the states of the W warps of its chunk
                constexpr int kRows = kHeads * NCI;
                constexpr int kThrPerRow = (kConsumerWarps * 32) / kRows;
                constexpr int per = D / kThrPerRow;
                const int t = threadIdx.x;              // 0..127
                const int rloc = t / kThrPerRow;
                const int cr = rloc / kHeads, head = rloc % kHeads;
                const int d0 = (t % kThrPerRow) * per;
                const int hcr = si.hc * NCI + cr;
                const long long row = ((long long)si.b * p.Hkv + si.kvh) * p.R + hcr * kHeads + head;
                if (head < min(kHeads, p.R - hcr * kHeads)) {
                    float M = -INFINITY;
                    #pragma unroll
                    for (int w = cr * W; w < cr * W + W; ++w) M = fmaxf(M, red_m[w * kHeads + head]);
                    float wt[W], Ltot = 0.f;
                    #pragma unroll
                    for (int i = 0; i < W; ++i) {
                        const int w = cr * W + i;
                        const float mw = red_m[w * kHeads + head];
                        wt[i] = (mw == -INFINITY) ? 0.f : ex2_approx(mw - M);
                        Ltot += wt[i] * red_l[w * kHeads + head];
                    }
                    // a row that saw no key in this split (a masked new token) contributes
                    // nothing: O = 0, lse = -inf
                    const float inv = Ltot > 0.f ? 1.f / Ltot : 0.f;
                    const float lse2 = Ltot > 0.f ? M + __log2f(Ltot) : -INFINITY;
                    float ov[per];
                    #pragma unroll
                    for (int u = 0; u < per; ++u) {
                        float sum = 0.f;
                        #pragma unroll
                        for (int i = 0; i < W; ++i)
                            sum += wt[i] * red_o[((cr * W + i) * kHeads + head) * D + d0 + u];
                        ov[u] = sum * inv;
                    }
                    if (si.direct) {
                        store_final<D, per>(p, row, d0, ov, (t % kThrPerRow) == 0, lse2);
                    } else if (GBATTN_IN_BOUNDS(row * p.n_parts + si.s,
                                                (long long)p.B * p.Hq * p.Tq * p.n_parts, p.err)) {
                        const long long slot = row * p.n_parts + si.s;
                        float* dst = p.ws_o + slot * D + d0;
                        #pragma unroll
                        for (int e = 0; e < per; e += 4)
                            *reinterpret_cast<float4*>(dst + e) = make_float4(ov[e], ov[e + 1], ov[e + 2], ov[e + 3]);
                        if ((t % kThrPerRow) == 0) p.ws_lse[slot] = lse2;
                        if constexpr (kFused) __threadfence();   // partial visible before the count
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(sync_b);
                if (!mbar_wait(sync_b, sync_phase, kErrWaitConsumer, p.err)) break;
                sync_phase ^= 1u;
                if constexpr (kPub) {
                    // count the partial in (the combine merges a group's rows once its count
                    // is complete): all of its rows are written -- the rendezvous just passed
                    // orders them before this hand-over -- and the publisher warp releases it
                    if (p.counted && !si.direct && t == 0)
                        publish((int)(((long long)si.b * p.Hkv + si.kvh) * p.n_hg + si.hc));
                }
                if constexpr (kFused) {
                    if (!si.direct) {
                        // count this split in; the CTA that completes the group folds it
                        // (single-launch mode has one piece per split)
                        if (t == 0)
                            *last_flag = atomicAdd(p.group_cnt + ((long long)si.b * p.Hkv + si.kvh) * p.n_hg + si.hc, 1)
                                         == si.n_ne - 1;
                        __syncwarp();
                        if (lane == 0) mbar_arrive(sync_c);
                        if (!mbar_wait(sync_c, sync_c_phase, kErrWaitConsumer, p.err)) break;
                        sync_c_phase ^= 1u;
                        if (*last_flag && head < min(kHeads, p.R - hcr * kHeads)) {
                            __threadfence();
                            fold_partials<D, per>(p, row, d0, si.n_ne, (t % kThrPerRow) == 0);
                        }
                    }
                }
            }
            if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
        if constexpr (kPub)
            if (p.counted && threadIdx.x == 0) publish(-1);   // the publisher may stop
    } else {
        // ================== consumer warps (multi-token: chunks stacked) ==================
        // Warp w takes keys [16 (w % 4), +16) of every stage for chunks
        // (w / 4) * CPW .. + CPW - 1 of the item, side by side in the MMA N dimension: each K
        // fragment and each V^T fragment (the byte permutes included) is built once and
        // feeds CPW MMAs.  Q comes from every stage; per-chunk (m, l, O) stay in registers.
        constexpr int CPW = NCI * 4 / kConsumerWarps;   // row chunks per warp
        const int g = lane >> 2, c = lane & 3;
        const uint32_t ring = smem_u32(smem);
        const float scale_log2 = p.scale_log2;
        float acc[CPW][D / 16][4];
        float m0[CPW], m1[CPW], l0[CPW], l1[CPW];
        int lim0[CPW], lim1[CPW], rows[CPW];
        int stage = 0;
        uint32_t phase = 0, sync_phase = 0;
        const int R0 = (warp & 3) * 16;          // this warp's 16 keys within a stage
        const int qd = warp >> 2;                // which half of the item's chunks
        bool run = true;
        while (run) {
            if (!mbar_wait(&full[stage], phase, kErrWaitConsumer, p.err)) break;
            const StageInfo si = info[stage];
            if (si.done) break;
            const uint32_t kbox = ring + stage * L::kStageBytes;
            const uint32_t vbox = kbox + L::kKBytes;
            const uint32_t qbox = vbox + L::kVBytes;
            if (si.tile == 0) {
                #pragma unroll
                for (int cq = 0; cq < CPW; ++cq) {
                    const int hc = si.hc * NCI + qd * CPW + cq;
                    rows[cq] = min(kHeads, p.R - hc * kHeads);
                    m0[cq] = m1[cq] = -INFINITY;
                    l0[cq] = l1[cq] = 0.f;
                    // causal limit of my two columns (rows hc*8 + 2c, +1)
                    lim0[cq] = si.len - p.Tq + ((hc * kHeads + 2 * c) % p.Tq) + 1;
                    lim1[cq] = si.len - p.Tq + ((hc * kHeads + 2 * c + 1) % p.Tq) + 1;
                    #pragma unroll
                    for (int mt = 0; mt < D / 16; ++mt)
                        acc[cq][mt][0] = acc[cq][mt][1] = acc[cq][mt][2] = acc[cq][mt][3] = 0.f;
                }
            }
            const int nvalid = min(16, si.ntok - R0);
            if (nvalid > 0) {
                // ---- S^T[16 keys x 8 rows] per chunk = K Q^T ----
                float sc[CPW][4];
                #pragma unroll
                for (int cq = 0; cq < CPW; ++cq) sc[cq][0] = sc[cq][1] = sc[cq][2] = sc[cq][3] = 0.f;
                #pragma unroll
                for (int s = 0; s < D / 32; ++s) {
                    const uint32_t kb = kbox + (s >> 1) * (kKeysPerStage * 128);
                    const int ch = 2 * c + (s & 1);
                    const uint4 k0 = lds128(sw128(kb, R0 + g, ch));
                    const uint4 k1 = lds128(sw128(kb, R0 + g + 8, ch));
                    #pragma unroll
                    for (int cq = 0; cq < CPW; ++cq) {
                        if (rows[cq] <= 0) continue;
                        const uint4 qv = lds128(sw128(qbox + (s >> 1) * (kHeads * NCI * 128),
                                                      (qd * CPW + cq) * kHeads + g, ch));
                        mma16816(sc[cq], k0.x, k1.x, k0.y, k1.y, qv.x, qv.y);
                        mma16816(sc[cq], k0.z, k1.z, k0.w, k1.w, qv.z, qv.w);
                    }
                }
                // ---- online softmax per chunk (columns = rows 2c, 2c+1 of the chunk) ----
                const bool v_lo = g < nvalid, v_hi = g + 8 < nvalid;
                const int key_lo = si.key0 + R0 + g, key_hi = key_lo + 8;
                uint32_t pb0[CPW], pb1[CPW];
                #pragma unroll
                for (int cq = 0; cq < CPW; ++cq) {
                    pb0[cq] = pb1[cq] = 0u;
                    if (rows[cq] <= 0) continue;
                    const float s0 = (v_lo && key_lo < lim0[cq]) ? sc[cq][0] * scale_log2 : -INFINITY;
                    const float s1 = (v_lo && key_lo < lim1[cq]) ? sc[cq][1] * scale_log2 : -INFINITY;
                    const float s2 = (v_hi && key_hi < lim0[cq]) ? sc[cq][2] * scale_log2 : -INFINITY;
                    const float s3 = (v_hi && key_hi < lim1[cq]) ? sc[cq][3] * scale_log2 : -INFINITY;
                    float mx0 = fmaxf(s0, s2), mx1 = fmaxf(s1, s3);
                    #pragma unroll
                    for (int w = 4; w < 32; w <<= 1) {
                        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, w));
                        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, w));
                    }
                    const float mn0 = fmaxf(m0[cq], mx0), mn1 = fmaxf(m1[cq], mx1);
                    const float base0 = mn0 == -INFINITY ? 0.f : mn0;
                    const float base1 = mn1 == -INFINITY ? 0.f : mn1;
                    const float corr0 = ex2_approx(m0[cq] - base0), corr1 = ex2_approx(m1[cq] - base1);
                    const float p00 = ex2_approx(s0 - base0), p01 = ex2_approx(s1 - base1);
                    const float p10 = ex2_approx(s2 - base0), p11 = ex2_approx(s3 - base1);
                    l0[cq] = l0[cq] * corr0 + p00 + p10;
                    l1[cq] = l1[cq] * corr1 + p01 + p11;
                    m0[cq] = mn0;
                    m1[cq] = mn1;
                    #pragma unroll
                    for (int mt = 0; mt < D / 16; ++mt) {
                        acc[cq][mt][0] *= corr0; acc[cq][mt][1] *= corr1;
                        acc[cq][mt][2] *= corr0; acc[cq][mt][3] *= corr1;
                    }
                    pb0[cq] = movmatrix_trans(pack_bf16(p00, p01));
                    pb1[cq] = movmatrix_trans(pack_bf16(p10, p11));
                }
                // ---- O^T[d x 8 rows] per chunk += V^T P^T ----
                const int tk[4] = {2 * c, 2 * c + 1, 2 * c + 8, 2 * c + 9};
                if constexpr (D == 128) {
                    uint4 vv[4][2];
                    #pragma unroll
                    for (int i = 0; i < 4; ++i)
                        #pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            uint4 z = make_uint4(0, 0, 0, 0);
                            if (tk[i] < nvalid) z = lds128(sw128(vbox + h * (kKeysPerStage * 128), R0 + tk[i], g));
                            vv[i][h] = z;
                        }
                    #pragma unroll
                    for (int mt = 0; mt < 8; ++mt) {
                        const uint32_t a0 = pair_elem(vv[0][0], vv[1][0], mt);
                        const uint32_t a1 = pair_elem(vv[0][1], vv[1][1], mt);
                        const uint32_t a2 = pair_elem(vv[2][0], vv[3][0], mt);
                        const uint32_t a3 = pair_elem(vv[2][1], vv[3][1], mt);
                        #pragma unroll
                        for (int cq = 0; cq < CPW; ++cq)
                            if (rows[cq] > 0) mma16816(acc[cq][mt], a0, a1, a2, a3, pb0[cq], pb1[cq]);
                    }
                } else {
                    uint4 vv[4];
                    #pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        uint4 z = make_uint4(0, 0, 0, 0);
                        if (tk[i] < nvalid) z = lds128(sw128(vbox, R0 + tk[i], g));
                        vv[i] = z;
                    }
                    #pragma unroll
                    for (int mt = 0; mt < 4; ++mt) {
                        const uint32_t a0 = pair_elem(vv[0], vv[1], mt);
                        const uint32_t a1 = pair_elem(vv[0], vv[1], mt + 4);
                        const uint32_t a2 = pair_elem(vv[2], vv[3], mt);
                        const uint32_t a3 = pair_elem(vv[2], vv[3], mt + 4);
                        #pragma unroll
                        for (int cq = 0; cq < CPW; ++cq)
                            if (rows[cq] > 0) mma16816(acc[cq][mt], a0, a1, a2, a3, pb0[cq], pb1[cq]);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[stage]);

            if (si.last) {
                // ---- CPW rounds; in round r each half merges its chunk r over its four
                // warps (red_* hold every warp's 8 rows) and writes the partial ----
                #pragma unroll
                for (int r = 0; r < CPW; ++r) {
                    if (!run) continue;
                    float lr0 = l0[r], lr1 = l1[r];
                    #pragma unroll
                    for (int w = 4; w < 32; w <<= 1) {
                        lr0 += __shfl_xor_sync(0xffffffffu, lr0, w);
                        lr1 += __shfl_xor_sync(0xffffffffu, lr1, w);
                    }
                    if (g == 0) {
                        red_m[warp * kHeads + 2 * c] = m0[r];
                        red_m[warp * kHeads + 2 * c + 1] = m1[r];
                        red_l[warp * kHeads + 2 * c] = lr0;
                        red_l[warp * kHeads + 2 * c + 1] = lr1;
                    }
                    float* ro = red_o + warp * kHeads * D;
                    #pragma unroll
                    for (int mt = 0; mt < D / 16; ++mt) {
                        const int d_lo = 8 * g + mt;
                        const int d_hi = (D == 128) ? 64 + 8 * g + mt : 8 * g + 4 + mt;
                        ro[(2 * c) * D + d_lo] = acc[r][mt][0];
                        ro[(2 * c + 1) * D + d_lo] = acc[r][mt][1];
                        ro[(2 * c) * D + d_hi] = acc[r][mt][2];
                        ro[(2 * c + 1) * D + d_hi] = acc[r][mt][3];
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(sync_a);
                    if (!mbar_wait(sync_a, sync_phase, kErrWaitConsumer, p.err)) { run = false; continue; }
                    // 256 threads: half hq (threads 128 hq ..) finishes chunk hq*CPW + r,
                    // 16 threads per row
                    const int t = threadIdx.x;
                    const int hq = t >> 7;
                    const int head = (t >> 4) & 7;
                    constexpr int per = D / 16;
                    const int d0 = (t & 15) * per;
                    const int hcr = si.hc * NCI + hq * CPW + r;
                    const long long row = ((long long)si.b * p.Hkv + si.kvh) * p.R + hcr * kHeads + head;
                    if (head < min(kHeads, p.R - hcr * kHeads)) {
                        const int w0 = hq * 4;
                        float M = -INFINITY;
                        #pragma unroll
                        for (int i = 0; i < 4; ++i) M = fmaxf(M, red_m[(w0 + i) * kHeads + head]);
                        float wt[4], Ltot = 0.f;
                        #pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const float mw = red_m[(w0 + i) * kHeads + head];
                            wt[i] = (mw == -INFINITY) ? 0.f : ex2_approx(mw - M);
                            Ltot += wt[i] * red_l[(w0 + i) * kHeads + head];
                        }
                        // a row that saw no key in this split (a masked new token)
                        // contributes nothing: O = 0, lse = -inf
                        const float inv = Ltot > 0.f ? 1.f / Ltot : 0.f;
                        const float lse2 = Ltot > 0.f ? M + __log2f(Ltot) : -INFINITY;
                        float ov[per];
                        #pragma unroll
                        for (int u = 0; u < per; ++u) {
                            float sum = 0.f;
                            #pragma unroll
                            for (int i = 0; i < 4; ++i)
                                sum += wt[i] * red_o[((w0 + i) * kHeads + head) * D + d0 + u];
                            ov[u] = sum * inv;
                        }
                        if (si.direct) {
                            store_final<D, per>(p, row, d0, ov, (t & 15) == 0, lse2);
                        } else if (GBATTN_IN_BOUNDS(row * p.n_parts + si.s,
                                                    (long long)p.B * p.Hq * p.Tq * p.n_parts, p.err)) {
                            const long long slot = row * p.n_parts + si.s;
                            float* dst = p.ws_o + slot * D + d0;
                            #pragma unroll
                            for (int e = 0; e < per; e += 4)
                                *reinterpret_cast<float4*>(dst + e) = make_float4(ov[e], ov[e + 1], ov[e + 2], ov[e + 3]);
                            if ((t & 15) == 0) p.ws_lse[slot] = lse2;
                        }
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(sync_b);
                    if (!mbar_wait(sync_b, sync_phase, kErrWaitConsumer, p.err)) { run = false; continue; }
                    sync_phase ^= 1u;
                }
            }
            if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
    }
    __syncthreads();
}

// The merges as a kernel of their own, launched dependent on the split kernel: one thread
// per (row, 4 columns, lane).  The partials come from the split kernel launched just before
// this one.  When that kernel counts each partial into its group (p.counted: calls with at
// most 8 rows per KV head), a block waits only for its own rows' groups -- its CTAs are
// launched as the split kernel's CTAs run out of work items and sit beside them, so each
// group is merged as soon as its last partial lands instead of after the whole grid;
// otherwise it waits for the split grid to complete.
template <int D>
__global__ void __launch_bounds__(256)
decode_combine_kernel(const __grid_constant__ DecodeParams p) {
    constexpr int kGroups = D / 4;
    const int c = p.combine_lanes;
    const long long rows = (long long)p.B * p.Hq * p.Tq;
    const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const int j = (int)(idx % c);
    const long long piece = idx / c;
    const long long row = piece / kGroups;
    const int cg = (int)(piece % kGroups);
    if (p.counted) {
        // the block's rows [r0, r1] and their counters: one per 128-row tile of a (sequence, KV
        // head) group of R rows, counter (row / R) * ceil(R / 128) + (row % R) / 128 (for the
        // warp-level kernel R <= 8, so simply row / R); a counter is complete once every
        // partial of its rows has been counted in
        const long long per_row = (long long)kGroups * c;
        const long long r0 = (long long)blockIdx.x * blockDim.x / per_row;
        const long long r1 = min(rows - 1, ((long long)blockIdx.x * blockDim.x + blockDim.x - 1) / per_row);
        const long long nrt = (p.R + 127) / 128;
        __shared__ int ok;
        if (threadIdx.x == 0) {
            ok = 1;
            const long long g0 = (r0 / p.R) * nrt + (r0 % p.R) / 128;
            const long long g1 = (r1 / p.R) * nrt + (r1 % p.R) / 128;
            for (long long g = g0; g <= g1 && ok; ++g) {
                const int n = row_partials(p, (int)((g / nrt) * p.R / ((long long)p.Hq * p.Tq)));
                if (n > 1 && !counter_wait_geq(p.group_cnt + g, n, kErrWaitMerge, p.err)) ok = 0;
            }
        }
        __syncthreads();
        if (!ok) return;
    } else {
        asm volatile("griddepcontrol.wait;" ::: "memory");
    }
    // rows past the end, or written directly by the split kernel, merge nothing
    const bool in = row < rows;
    const int n_parts = in ? row_partials(p, (int)(row / ((long long)p.Hq * p.Tq))) : 0;
    merge_columns<D>(p, in ? row : 0, cg, j, n_parts, in);
    // the call ends after both grids: one thread holds this grid open until the split grid
    // has completed
    if (p.counted && blockIdx.x == 0 && threadIdx.x == 0)
        asm volatile("griddepcontrol.wait;" ::: "memory");
}

}  // namespace

int decode_slots(int Lmax, int num_splits, int auto_floor) {
    return splits_for(Lmax, num_splits, auto_floor);
}

size_t decode_counter_bytes(int B, int Hkv, int n_hg) {
    // the work queue counter, then one partial counter per (b, KV head, chunk group)
    return (((size_t)1 + (size_t)B * Hkv * n_hg) * 4 + 255) / 256 * 256;
}

size_t decode_workspace_bytes(int B_rows, int Hq, int kv_groups, int n_hg, int d, int n_parts) {
    const size_t rows = (size_t)B_rows * Hq * n_parts;
    size_t bytes = decode_counter_bytes(kv_groups, 1, n_hg);   // counters
    bytes += ((rows * 4 + 255) / 256) * 256;             // lse partials
    bytes += rows * (size_t)d * 4;                       // O partials
    return bytes;
}

namespace {

template <int D, int NCI, bool kFused = false, bool kTwo = false>
cudaError_t launch_pair(const DecodeParams& p, int num_sms, cudaStream_t stream) {
    constexpr int smem = Layout<D, NCI, kTwo>::kAlloc;
    static_assert(smem * Cfg<NCI, kTwo>::kPerSM <= 227 * 1024, "shared memory budget");
    const int slots = num_sms * Cfg<NCI, kTwo>::kPerSM;
    const int grid = p.n_items < slots ? p.n_items : slots;
    if (grid <= 0) return cudaSuccess;
    cudaError_t err = cudaFuncSetAttribute(decode_split_kernel<D, NCI, kFused, kTwo>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return err;
    decode_split_kernel<D, NCI, kFused, kTwo><<<grid, split_threads<NCI, kFused>(), smem, stream>>>(p);
    err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    if constexpr (kFused) return cudaSuccess;      // merged in the split kernel
    // combine: programmatic dependent launch on the same stream
    const long long threads = (long long)p.B * p.Hq * p.Tq * (D / 4) * p.combine_lanes;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((threads + 255) / 256));
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, decode_combine_kernel<D>, p);
}

template <int D>
cudaError_t launch_combine(const DecodeParams& p, cudaStream_t stream) {
    const long long threads = (long long)p.B * p.Hq * p.Tq * (D / 4) * p.combine_lanes;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((threads + 255) / 256));
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, decode_combine_kernel<D>, p);
}

}  // namespace

cudaError_t launch_decode_combine(const DecodeParams& p, int d, cudaStream_t stream) {
    return d == 128 ? launch_combine<128>(p, stream) : launch_combine<64>(p, stream);
}

cudaError_t launch_decode_splitkv(const DecodeParams& p, int d, int num_sms,
                                  cudaStream_t stream) {
    cudaError_t err = cudaMemsetAsync(p.counter, 0, decode_counter_bytes(p.B, p.Hkv, p.n_hg), stream);
    if (err != cudaSuccess) return err;
    if (p.fused) {
        // more items than SMs: two CTAs per SM (one folds a group while the other streams);
        // one wave: one CTA per SM with the deep ring (measured: B1 with 131072 keys 93.9 ->
        // 88.9 us with two per SM, B1 with 65536 keys in one wave 50.4 -> 58.2 us)
        if (p.n_items > num_sms)
            return d == 128 ? launch_pair<128, 1, true, true>(p, num_sms, stream)
                            : launch_pair<64, 1, true, true>(p, num_sms, stream);
        return d == 128 ? launch_pair<128, 1, true>(p, num_sms, stream)
                        : launch_pair<64, 1, true>(p, num_sms, stream);
    }
    // (16 or more rows per KV head run on the tcgen05 kernel, so NCI <= 2 here)
    if (p.nci > 2) return cudaErrorInvalidValue;
    if (d == 128)
        return p.nci == 2 ? launch_pair<128, 2>(p, num_sms, stream) : launch_pair<128, 1>(p, num_sms, stream);
    return p.nci == 2 ? launch_pair<64, 2>(p, num_sms, stream) : launch_pair<64, 1>(p, num_sms, stream);
}

#ifdef GBATTN_DEBUG_CHECKS
cudaError_t debug_skip_fill_split(int fill) {
    return cudaMemcpyToSymbol(g_skip_k_fill, &fill, sizeof(int));
}
#endif

}  // namespace gbattn
