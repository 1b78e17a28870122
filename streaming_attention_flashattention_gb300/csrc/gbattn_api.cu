// gbattn_api.cu -- the C ABI: argument validation ("AI Compiler pipeline stages",
// Legality Checking: shape, dtype, layout and memory conditions decide whether the fused
// kernel may run; here they turn into status codes), launch planning (TMA descriptors,
// work counts, workspace carving) and the launches themselves.  No device memory is
// allocated per call; the only device state is the error word of bounded waits.
#include <cuda.h>
#include <cuda_runtime.h>

#include <nvtx3/nvToolsExt.h>

#include <algorithm>
#include <mutex>
#include <vector>

#include "common.cuh"
#include "kernels.h"
#ifdef GBATTN_DEBUG_CHECKS
#include "gbattn_debug.h"
#endif

namespace gbattn {

namespace {
__device__ int g_device_error = 0;
}  // namespace

int* device_error_word() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
    static int* cached[64] = {nullptr};
    if (dev >= 0 && dev < 64 && cached[dev]) return cached[dev];
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_device_error) != cudaSuccess) return nullptr;
    if (dev >= 0 && dev < 64) cached[dev] = static_cast<int*>(ptr);
    return static_cast<int*>(ptr);
}

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

// 3-D bf16 tensor map with a 128-byte swizzle: dims innermost first, box (64, rows, 1).
// d1_stride: rows between consecutive d2 planes (>= d1; larger for a cache whose
// capacity exceeds the valid length d1 -- the rows past d1 are then out of bounds).
bool make_map_bf16_3d(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1,
                      uint64_t d2, uint32_t box_rows, uint64_t d1_stride = 0) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    if (d1_stride == 0) d1_stride = d1;
    const cuuint64_t dims[3] = {d0, d1, d2};
    const cuuint64_t strides[2] = {d0 * 2, d0 * d1_stride * 2};
    const cuuint32_t box[3] = {64, box_rows, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
              box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

int sm_count() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    static int cached[64] = {0};
    if (dev >= 0 && dev < 64 && cached[dev] > 0) return cached[dev];
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
    if (dev >= 0 && dev < 64) cached[dev] = n;
    return n;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// One thread waits on an mbarrier that nothing ever arrives on; the bounded wait gives up
// after `limit` cycles, records kErrSelfTest and the kernel returns normally.
__global__ void selftest_wait_kernel(int* err_word, long long limit) {
    __shared__ uint64_t bar;
    mbar_init(&bar, 1);
    fence_barrier_init();
    mbar_wait(&bar, 0, kErrSelfTest, err_word, limit);
}

// An NVTX range around one library call, so that a profiler's timeline shows the call with
// the launches it made (without a profiler attached NVTX does nothing).
struct CallRange {
    explicit CallRange(const char* name) { nvtxRangePushA(name); }
    ~CallRange() { nvtxRangePop(); }
};

constexpr long long kIntMax = 2147483647LL;
constexpr long long kFusedMaxGroups = 16;   // single-launch decode: up to this many groups,
constexpr long long kFusedMinKeys = 1024;   // with splits of at least this many keys
constexpr long long kTcMinKeys = 1024;      // 9-15 rows per KV head: tcgen05 path from this
                                            // many keys per split
constexpr int kMaxPieces = 4;               // pieces per split, at most
constexpr long long kPieceWaves = 6;        // enough waves of work items that the last one
                                            // no longer matters
constexpr long long kPieceMinKeys = 512;    // keys per piece, at least (Lmax / (splits * pieces))

// The work split of a bf16 prefill, from its sizes alone (used by the launch and by
// attn_prefill_plan()).
struct PrefillPlan {
    int n_qblk;
    long long n_pairs, n_tiles;
    bool kv_split;           // one Q tile per CTA, its KV range over the CTA's two slots
    long long first;         // CTAs of the first launch
    long long tail;          // pairs run as KV-split tiles in a second launch
};

// diag: causal diagonal (key j visible to query row i iff j <= i + diag); row0: the first
// query row the Q tiles cover (every row from row0 on sees at least one key).
PrefillPlan prefill_plan(int B, int Hq, int Hkv, int Sq, int Skv, int causal, int nsm,
                         int diag, int row0) {
    PrefillPlan pl{};
    const int G = Hq / Hkv;
    pl.n_qblk = (Sq - row0 + 127) / 128;
    const long long per_group = ((long long)pl.n_qblk * G + 1) / 2;
    pl.n_pairs = per_group * B * Hkv;
    pl.n_tiles = (long long)pl.n_qblk * B * Hq;
    // Pairs of Q tiles keep both ping-pong slots busy with independent work; when there are
    // fewer pairs than SMs, splitting each tile's KV range over the two slots halves the
    // longest item instead, and the tiles run on persistent CTAs (one per SM, heaviest
    // tiles dealt first) so that each SM pays the start-up once.  (Between one and two
    // pairs per SM the pair kernel measured 10-19% faster than the split.)
    pl.kv_split = pl.n_pairs < (long long)nsm;
    // Pairs of nearly equal weight (non-causal, or a chunk at the end of a long context)
    // whose last wave is at most half full: those last pairs run as single Q tiles in
    // KV-split mode, launched behind the pair grid as a programmatic dependent so that they
    // fill SMs as the pair grid drains -- half a pair's time instead of a whole one.
    // (Causal prefill over its whole context has pairs of all weights, heaviest first, and
    // keeps one launch.)
    if (!pl.kv_split) {
        auto kv_tiles = [&](long long q0) {
            if (!causal) return ((long long)Skv + 127) / 128;
            const long long last = std::min<long long>(q0 + 128, Sq) - 1;
            const long long keys = std::min<long long>(Skv, last + diag + 1);
            return (keys + 127) / 128;
        };
        const long long lo = kv_tiles(row0),
                        hi = kv_tiles(row0 + (long long)(pl.n_qblk - 1) * 128);
        const long long rem = pl.n_pairs % nsm;
        if (lo > 0 && 4 * hi <= 5 * lo && rem > 0 && rem <= nsm / 2) pl.tail = rem;
    }
    pl.first = pl.kv_split ? std::min<long long>(pl.n_tiles, nsm) : pl.n_pairs - pl.tail;
    return pl;
}

// bf16 tcgen05 prefill; K/V rows of one head are `kv_stride` rows apart (>= Skv).
// diag, row0: as for prefill_plan (bottom-right causal: Skv - Sq and 0).
// tiles: null, or a device counter that receives the S tile products the kernels issue.
int launch_prefill_bf16(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                        int Hq, int Hkv, int Sq, int Skv, int kv_stride, int d, float scale,
                        int causal, int diag, int row0, cudaStream_t st,
                        int* tiles = nullptr) {
    PrefillParams p{};
    if (!make_map_bf16_3d(&p.tmap_q, q, d, Sq, (uint64_t)B * Hq, 128) ||
        !make_map_bf16_3d(&p.tmap_k, k, d, Skv, (uint64_t)B * Hkv, 128, kv_stride) ||
        !make_map_bf16_3d(&p.tmap_v, v, d, Skv, (uint64_t)B * Hkv, 128, kv_stride) ||
        !make_map_bf16_3d(&p.tmap_o, o, d, Sq, (uint64_t)B * Hq, 128))
        return GBATTN_ERR_CUDA;
    p.o = static_cast<__nv_bfloat16*>(o);
    p.lse = lse;
    p.B = B; p.Hq = Hq; p.Hkv = Hkv; p.Sq = Sq; p.Skv = Skv;
    p.G = Hq / Hkv;
    const int nsm = sm_count();
    if (nsm <= 0) return GBATTN_ERR_CUDA;
    const PrefillPlan pl = prefill_plan(B, Hq, Hkv, Sq, Skv, causal, nsm, diag, row0);
    if (pl.n_pairs > kIntMax || pl.n_tiles > kIntMax) return GBATTN_ERR_TOO_LARGE;
    p.n_qblk = pl.n_qblk;
    p.kv_split = pl.kv_split ? 1 : 0;
    p.n_pairs = (int)(pl.kv_split ? pl.n_tiles : pl.first);
    p.tail0 = -1;
    p.causal = causal;
    p.diag = diag;
    p.row0 = row0;
    p.o_align32 = (reinterpret_cast<uintptr_t>(o) & 31u) == 0 ? 1 : 0;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.err = device_error_word();
    if (!p.err) return GBATTN_ERR_CUDA;
    p.tiles_issued = tiles;
    cudaError_t e = pl.kv_split ? launch_attn_fwd_bf16_persistent(p, d, nsm, st)
                                : launch_attn_fwd_bf16(p, d, st);
    if (e == cudaSuccess && pl.tail > 0) {
        PrefillParams t = p;
        t.kv_split = 1;
        t.tail0 = (int)(pl.n_pairs - pl.tail);
        t.n_pairs = (int)(2 * pl.tail);
        e = launch_attn_fwd_bf16_tail(t, d, st);
    }
    return e == cudaSuccess ? GBATTN_OK : GBATTN_ERR_CUDA;
}

// ---- host-buffer prefill: chunked copies in and out overlapped with the kernel ----------
// The work is cut into chunks of consecutive (batch, KV head) groups -- each a contiguous
// slab of Q/O ([G, Sq, d]), K and V ([Skv, d]) and LSE ([G, Sq]) -- staged through up to
// three device buffer sets.  Chunk i's copy in waits for chunk i-3's copy out (the same
// buffers), its kernel for its copy in, its copy out for its kernel, so chunks i+1 and i+2
// come in and chunk i-1 goes out while chunk i computes.  (With two sets, chunk i's copy in
// waited for chunk i-2's copy out, which itself waits for chunk i-2's kernel: the link sat
// idle in between.)
constexpr int kHostSets = 3;

struct HostPlan {
    int cg;                  // groups per chunk
    int n_chunks;
    int n_bufs;              // buffer sets: min(n_chunks, kHostSets)
    size_t q_off, k_off, v_off, o_off, l_off, set_bytes;   // one buffer set
};

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

HostPlan host_plan(int B, int Hq, int Hkv, int Sq, int Skv, int d, size_t esize, int nsm) {
    HostPlan h{};
    const int G = Hq / Hkv;
    const long long ng = (long long)B * Hkv;
    const long long pairs_per_group = ((long long)((Sq + 127) / 128) * G + 1) / 2;
    // the smallest chunk that keeps the kernel's pair mode (a Q-tile pair per SM): small
    // chunks shorten the first copy in and the last kernel and copy out, which nothing hides
    long long cg = ((long long)nsm + pairs_per_group - 1) / pairs_per_group;
    cg = std::min(std::max(cg, 1LL), ng);
    h.cg = (int)cg;
    h.n_chunks = (int)((ng + cg - 1) / cg);
    h.n_bufs = std::min(h.n_chunks, kHostSets);
    const size_t qb = (size_t)cg * G * Sq * d * esize;
    const size_t kb = (size_t)cg * Skv * d * esize;
    const size_t lb = (size_t)cg * G * Sq * 4;
    h.q_off = 0;
    h.k_off = align256(qb);
    h.v_off = h.k_off + align256(kb);
    h.o_off = h.v_off + align256(kb);
    h.l_off = h.o_off + align256(qb);
    h.set_bytes = h.l_off + align256(lb);
    return h;
}

// Copy streams and events of the current device, created on first use.
struct HostPipe {
    cudaStream_t in = nullptr, out = nullptr;
    cudaEvent_t entry = nullptr, done = nullptr;
    cudaEvent_t ev_in[kHostSets] = {}, ev_comp[kHostSets] = {}, ev_out[kHostSets] = {};
    std::mutex mu;           // one host-buffer call at a time per device
};

HostPipe* host_pipe() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    static HostPipe pipes[64];
    static std::once_flag once[64];
    bool ok = true;
    std::call_once(once[dev], [&] {
        HostPipe& h = pipes[dev];
        ok = cudaStreamCreateWithFlags(&h.in, cudaStreamNonBlocking) == cudaSuccess &&
             cudaStreamCreateWithFlags(&h.out, cudaStreamNonBlocking) == cudaSuccess &&
             cudaEventCreateWithFlags(&h.entry, cudaEventDisableTiming) == cudaSuccess &&
             cudaEventCreateWithFlags(&h.done, cudaEventDisableTiming) == cudaSuccess;
        for (int i = 0; i < kHostSets && ok; ++i)
            ok = cudaEventCreateWithFlags(&h.ev_in[i], cudaEventDisableTiming) == cudaSuccess &&
                 cudaEventCreateWithFlags(&h.ev_comp[i], cudaEventDisableTiming) == cudaSuccess &&
                 cudaEventCreateWithFlags(&h.ev_out[i], cudaEventDisableTiming) == cudaSuccess;
    });
    HostPipe& h = pipes[dev];
    return (h.in && h.out && h.done && h.ev_out[kHostSets - 1]) ? &h : nullptr;
}

// Query rows of a decode call per KV head (G * Tq, chunks of 8) and how work items group
// them: one item serves up to 4 row chunks, so K/V are read once for all of them.
struct DecodeRows {
    int R, n_hc, nci, n_hg;
};
DecodeRows decode_rows(int Hq, int Hkv, int Tq) {
    DecodeRows r;
    r.R = (Hq / Hkv) * Tq;
    r.n_hc = (r.R + 7) / 8;
    r.nci = r.n_hc >= 3 ? 4 : r.n_hc;
    r.n_hg = (r.n_hc + r.nci - 1) / r.nci;
    return r;
}

// Automatic split mode: the most splits per sequence that keep the call within one wave of
// work items on a GPU with nsm SMs (one persistent CTA per SM).  A work item is one split
// of one (sequence, KV head) and one row group: a 128-row tile on the tensor-core path
// (R >= 16), a chunk group on the warp-level path.  Never below one.
int auto_floor(int B, int Hkv, const DecodeRows& dr, int nsm) {
    const long long per_split = (long long)B * Hkv * (dr.R >= 16 ? (dr.R + 127) / 128 : dr.n_hg);
    const long long f = nsm / per_split;
    return (int)(f < 1 ? 1 : (f > kMaxSplits ? kMaxSplits : f));
}

// Pieces per split.  The work queue hands out whole items; when there are a few waves of
// them and the last is mostly idle (workload 4: 512 equal splits on 152 SMs, 3.37 waves),
// each split is cut into P contiguous pieces, each a work item with a partial of its own
// that the combine folds like any other: the smallest P that gives kPieceWaves waves or a
// last wave at least 3/4 full.  Pieces keep at least kPieceMinKeys keys, and a row has at
// most kMaxSplits partials.  Calls within one wave keep whole splits.
int pieces_for(long long items, int n_slots, int Lmax, int nsm) {
    if (items <= nsm) return 1;
    for (int P = 1; P <= kMaxPieces; ++P) {
        if (P > 1 && ((long long)n_slots * P > kMaxSplits ||
                      (long long)Lmax < kPieceMinKeys * n_slots * P))
            return P - 1;
        const long long it = items * P, rem = it % nsm;
        if (it >= kPieceWaves * nsm || rem == 0 || 4 * rem >= 3 * (long long)nsm) return P;
    }
    return kMaxPieces;
}

// Everything a decode call decides from its sizes alone, before any device access: the
// split count and pieces, the kernel, the merge.  The launch code, the workspace size and
// attn_decode_plan() all use it.
struct DecodePlan {
    DecodeRows dr;
    int floor_splits, n_slots;
    int pieces;              // work items per split
    long long n_items;       // work items of the warp-level kernel
    bool tc;                 // the tcgen05 kernel runs the call
    int n_rt, q_rows;        // tcgen05 kernel: 128-row tiles per KV head, Q rows loaded
    long long tc_items;      // tcgen05 kernel: work items
    bool fused;              // warp-level kernel: the group's last split merges it
    bool counted;            // warp-level kernel: partials counted per group, per-group combine
    int combine_lanes;       // combine kernel: lanes per (row, 4 columns)
};

DecodePlan decode_plan(int B, int Hq, int Hkv, int Tq, int Lmax, int num_splits, int nsm) {
    DecodePlan pl{};
    pl.dr = decode_rows(Hq, Hkv, Tq);
    pl.floor_splits = auto_floor(B, Hkv, pl.dr, nsm);
    pl.n_slots = decode_slots(Lmax, num_splits, pl.floor_splits);
    pl.pieces = 1;
    pl.n_items = (long long)pl.n_slots * B * Hkv * pl.dr.n_hg;
    // tcgen05 path: 16 or more query rows per KV head (several new tokens, or G >= 16), or 9
    // to 15 with long splits; 8 rows and fewer, and short splits of 9 to 15 rows, run best on
    // the warp-level kernel, whose work items carry less fixed cost
    const int R = pl.dr.R;
    pl.tc = R >= 16 || (R >= 9 && (long long)Lmax >= kTcMinKeys * pl.n_slots);
    pl.n_rt = (R + 127) / 128;
    // only the item's own rows of Q are loaded (R rounded up to 8); the MMA's other rows of
    // the M = 128 operand hold whatever the buffer held and only produce rows that are never
    // stored (each output row depends on its own query row alone)
    pl.q_rows = R >= 128 ? 128 : (R + 7) / 8 * 8;
    pl.tc_items = (long long)pl.n_slots * B * Hkv * pl.n_rt;
    // single launch (the group's last split merges) when every item runs in the first wave,
    // where the combine's launch is a large part of the call, or when there are few groups
    // with long splits, where the combine's few threads wait on long partial lists; with
    // many groups or short splits the per-split count and rendezvous cost more than the
    // combine
    const long long groups = (long long)B * Hkv * pl.dr.n_hg;
    const bool few_long = groups <= kFusedMaxGroups && (long long)Lmax >= kFusedMinKeys * pl.n_slots;
    pl.fused = !pl.tc && pl.dr.nci == 1 && (pl.n_items <= nsm || few_long);
    // (the tcgen05 kernel's items carry more fixed cost -- a Q tile, two ping-pong slots, a
    // merge from TMEM -- and measured no faster or slower in pieces: it keeps whole splits)
    if (!pl.fused && !pl.tc) {
        pl.pieces = pieces_for(pl.n_items, pl.n_slots, Lmax, nsm);
        pl.n_items *= pl.pieces;
    }
    // calls of the warp-level kernel with one row chunk per KV head (R <= 8) count each
    // partial into its (sequence, KV head) group, and the combine merges a group as soon as
    // its count is complete, overlapping the split kernel's last items, instead of waiting
    // for the whole split grid (that wait and the combine after it cost about 6 us on
    // workload 4)
    // The tcgen05 kernel counts the same way, per (sequence, KV head, 128-row tile), through its
    // otherwise idle fourth warp.
    pl.counted = pl.tc || (!pl.fused && pl.dr.nci == 1);
    pl.combine_lanes = 1;
    while (pl.combine_lanes * 8 < pl.n_slots * pl.pieces) pl.combine_lanes *= 2;   // <= 256 partials: at most 32
    return pl;
}

}  // namespace
}  // namespace gbattn

using namespace gbattn;

extern "C" {

int attn_version(void) { return 100; }

const char* attn_status_string(int status) {
    switch (status) {
        case GBATTN_OK: return "ok";
        case GBATTN_ERR_INVALID_ARG: return "invalid argument";
        case GBATTN_ERR_UNSUPPORTED: return "unsupported configuration";
        case GBATTN_ERR_MISALIGNED: return "pointer not 16-byte aligned";
        case GBATTN_ERR_CUDA: return "CUDA error";
        case GBATTN_ERR_TIMEOUT: return "device bounded wait expired";
        case GBATTN_ERR_WORKSPACE: return "workspace missing or too small";
        case GBATTN_ERR_TOO_LARGE: return "size exceeds kernel indexing range";
        default: return "unknown status";
    }
}

int attn_fwd_counted(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                     int Hq, int Hkv, int Sq, int Skv, int d, float scale, int causal,
                     int* s_tiles, void* stream) {
    CallRange range("attn_fwd_counted");
    if (!s_tiles) return GBATTN_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(s_tiles) & 3u) return GBATTN_ERR_MISALIGNED;
    // the same checks as attn_fwd (bf16)
    if (!q || !k || !v || !o) return GBATTN_ERR_INVALID_ARG;
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || Sq <= 0 || Skv <= 0 || d <= 0)
        return GBATTN_ERR_INVALID_ARG;
    if (Hq % Hkv != 0) return GBATTN_ERR_INVALID_ARG;
    if (!(scale > 0.f) || scale != scale) return GBATTN_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return GBATTN_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return GBATTN_ERR_UNSUPPORTED;
    if (causal && Sq > Skv) return GBATTN_ERR_UNSUPPORTED;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) ||
        (lse && !aligned16(lse)))
        return GBATTN_ERR_MISALIGNED;
    if ((long long)B * Hq > 65535LL * 65535LL || (long long)B * Hq * Sq > kIntMax ||
        (long long)B * Hkv * Skv > kIntMax)
        return GBATTN_ERR_TOO_LARGE;
    return launch_prefill_bf16(q, k, v, o, lse, B, Hq, Hkv, Sq, Skv, Skv, d, scale, causal,
                               Skv - Sq, 0, static_cast<cudaStream_t>(stream), s_tiles);
}

int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
             int Hkv, int Sq, int Skv, int d, float scale, int causal, int dtype,
             void* stream) {
    CallRange range("attn_fwd");
    if (!q || !k || !v || !o) return GBATTN_ERR_INVALID_ARG;
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || Sq <= 0 || Skv <= 0 || d <= 0)
        return GBATTN_ERR_INVALID_ARG;
    if (Hq % Hkv != 0) return GBATTN_ERR_INVALID_ARG;
    if (!(scale > 0.f) || scale != scale) return GBATTN_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return GBATTN_ERR_INVALID_ARG;
    if (dtype != GBATTN_BF16 && dtype != GBATTN_FP32) return GBATTN_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return GBATTN_ERR_UNSUPPORTED;
    if (causal && Sq > Skv) return GBATTN_ERR_UNSUPPORTED;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) ||
        (lse && !aligned16(lse)))
        return GBATTN_ERR_MISALIGNED;
    if ((long long)B * Hq > 65535LL * 65535LL || (long long)B * Hq * Sq > kIntMax ||
        (long long)B * Hkv * Skv > kIntMax)
        return GBATTN_ERR_TOO_LARGE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);

    if (dtype == GBATTN_FP32) {
        if (B > 65535 || Hq > 65535) return GBATTN_ERR_TOO_LARGE;
        int* err = device_error_word();
        if (!err) return GBATTN_ERR_CUDA;
        cudaError_t e = launch_attn_fwd_f32(static_cast<const float*>(q),
                                            static_cast<const float*>(k),
                                            static_cast<const float*>(v), static_cast<float*>(o),
                                            lse, B, Hq, Hkv, Sq, Skv, d, scale, causal, err, st);
        return e == cudaSuccess ? GBATTN_OK : GBATTN_ERR_CUDA;
    }

    return launch_prefill_bf16(q, k, v, o, lse, B, Hq, Hkv, Sq, Skv, Skv, d, scale, causal,
                               Skv - Sq, 0, st);
}

size_t attn_fwd_host_workspace_size(int B, int Hq, int Hkv, int Sq, int Skv, int d, int dtype) {
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || Sq <= 0 || Skv <= 0 || Hq % Hkv != 0) return 0;
    if ((d != 64 && d != 128) || (dtype != GBATTN_BF16 && dtype != GBATTN_FP32)) return 0;
    const int nsm = sm_count();
    if (nsm <= 0) return 0;
    const HostPlan h = host_plan(B, Hq, Hkv, Sq, Skv, d, dtype == GBATTN_BF16 ? 2 : 4, nsm);
    return h.set_bytes * h.n_bufs;
}

int attn_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                  int Hq, int Hkv, int Sq, int Skv, int d, float scale, int causal, int dtype,
                  void* workspace, size_t ws_bytes, void* stream) {
    CallRange range("attn_fwd_host");
    if (!q || !k || !v || !o) return GBATTN_ERR_INVALID_ARG;
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || Sq <= 0 || Skv <= 0 || d <= 0)
        return GBATTN_ERR_INVALID_ARG;
    if (Hq % Hkv != 0) return GBATTN_ERR_INVALID_ARG;
    if (!(scale > 0.f) || scale != scale) return GBATTN_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return GBATTN_ERR_INVALID_ARG;
    if (dtype != GBATTN_BF16 && dtype != GBATTN_FP32) return GBATTN_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return GBATTN_ERR_UNSUPPORTED;
    if (causal && Sq > Skv) return GBATTN_ERR_UNSUPPORTED;
    if ((long long)B * Hq > 65535LL * 65535LL || (long long)B * Hq * Sq > kIntMax ||
        (long long)B * Hkv * Skv > kIntMax)
        return GBATTN_ERR_TOO_LARGE;
    const size_t need = attn_fwd_host_workspace_size(B, Hq, Hkv, Sq, Skv, d, dtype);
    if (need == 0) return GBATTN_ERR_CUDA;
    if (!workspace || ws_bytes < need) return GBATTN_ERR_WORKSPACE;
    if (!aligned16(workspace)) return GBATTN_ERR_MISALIGNED;
    HostPipe* hp = host_pipe();
    if (!hp) return GBATTN_ERR_CUDA;
    int* errw = device_error_word();
    if (!errw) return GBATTN_ERR_CUDA;
    std::lock_guard<std::mutex> lock(hp->mu);

    const size_t es = dtype == GBATTN_BF16 ? 2 : 4;
    const HostPlan h = host_plan(B, Hq, Hkv, Sq, Skv, d, es, sm_count());
    const int G = Hq / Hkv;
    const int ng = B * Hkv;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const char* qh = static_cast<const char*>(q);
    const char* kh = static_cast<const char*>(k);
    const char* vh = static_cast<const char*>(v);
    char* oh = static_cast<char*>(o);
    char* lh = reinterpret_cast<char*>(lse);
    char* ws = static_cast<char*>(workspace);
    const size_t qg = (size_t)G * Sq * d * es, kg = (size_t)Skv * d * es, lg = (size_t)G * Sq * 4;
    auto chk = [](cudaError_t e) { return e == cudaSuccess; };
    bool ok = chk(cudaEventRecord(hp->entry, st));   // the caller's earlier work comes first
    for (int i = 0; ok && i < h.n_chunks; ++i) {
        const int bset = i % h.n_bufs;
        const int g0 = i * h.cg, gn = std::min(h.cg, ng - g0);
        char* base = ws + (size_t)bset * h.set_bytes;
        ok = chk(cudaStreamWaitEvent(hp->in, i >= h.n_bufs ? hp->ev_out[bset] : hp->entry, 0)) &&
             chk(cudaMemcpyAsync(base + h.q_off, qh + g0 * qg, gn * qg, cudaMemcpyHostToDevice, hp->in)) &&
             chk(cudaMemcpyAsync(base + h.k_off, kh + g0 * kg, gn * kg, cudaMemcpyHostToDevice, hp->in)) &&
             chk(cudaMemcpyAsync(base + h.v_off, vh + g0 * kg, gn * kg, cudaMemcpyHostToDevice, hp->in)) &&
             chk(cudaEventRecord(hp->ev_in[bset], hp->in)) &&
             chk(cudaStreamWaitEvent(st, hp->ev_in[bset], 0));
        if (!ok) break;
        float* lse_d = lh ? reinterpret_cast<float*>(base + h.l_off) : nullptr;
        int rc;
        if (dtype == GBATTN_FP32) {
            rc = launch_attn_fwd_f32(reinterpret_cast<const float*>(base + h.q_off),
                                     reinterpret_cast<const float*>(base + h.k_off),
                                     reinterpret_cast<const float*>(base + h.v_off),
                                     reinterpret_cast<float*>(base + h.o_off), lse_d, 1, gn * G, gn,
                                     Sq, Skv, d, scale, causal, errw, st) == cudaSuccess
                     ? GBATTN_OK : GBATTN_ERR_CUDA;
        } else {
            rc = launch_prefill_bf16(base + h.q_off, base + h.k_off, base + h.v_off, base + h.o_off,
                                     lse_d, 1, gn * G, gn, Sq, Skv, Skv, d, scale, causal,
                                     Skv - Sq, 0, st);
        }
        if (rc != GBATTN_OK) return rc;
        ok = chk(cudaEventRecord(hp->ev_comp[bset], st)) &&
             chk(cudaStreamWaitEvent(hp->out, hp->ev_comp[bset], 0)) &&
             chk(cudaMemcpyAsync(oh + g0 * qg, base + h.o_off, gn * qg, cudaMemcpyDeviceToHost, hp->out)) &&
             (!lh || chk(cudaMemcpyAsync(lh + g0 * lg, base + h.l_off, gn * lg, cudaMemcpyDeviceToHost, hp->out))) &&
             chk(cudaEventRecord(hp->ev_out[bset], hp->out));
    }
    // the caller's stream completes after the last copy out
    ok = ok && chk(cudaEventRecord(hp->done, hp->out)) && chk(cudaStreamWaitEvent(st, hp->done, 0));
    return ok ? GBATTN_OK : GBATTN_ERR_CUDA;
}

int attn_prefill_kvcache(const void* q, const void* kcache, const void* vcache, void* o,
                         float* lse, int B, int Hq, int Hkv, int Sq, int Skv, int Lmax, int d,
                         float scale, int causal, void* stream) {
    CallRange range("attn_prefill_kvcache");
    if (!q || !kcache || !vcache || !o) return GBATTN_ERR_INVALID_ARG;
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || Sq <= 0 || Skv <= 0 || Lmax <= 0 || d <= 0)
        return GBATTN_ERR_INVALID_ARG;
    if (Skv > Lmax || Hq % Hkv != 0) return GBATTN_ERR_INVALID_ARG;
    if (!(scale > 0.f) || scale != scale) return GBATTN_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return GBATTN_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return GBATTN_ERR_UNSUPPORTED;
    if (causal && Sq > Skv) return GBATTN_ERR_UNSUPPORTED;
    if (!aligned16(q) || !aligned16(kcache) || !aligned16(vcache) || !aligned16(o) ||
        (lse && !aligned16(lse)))
        return GBATTN_ERR_MISALIGNED;
    if ((long long)B * Hq * Sq > kIntMax || (long long)B * Hkv * Lmax > kIntMax)
        return GBATTN_ERR_TOO_LARGE;
    return launch_prefill_bf16(q, kcache, vcache, o, lse, B, Hq, Hkv, Sq, Skv, Lmax, d, scale,
                               causal, Skv - Sq, 0, static_cast<cudaStream_t>(stream));
}

int attn_fwd_positions(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                       int Hq, int Hkv, int Sq, int Skv, int d, float scale, long long q_pos0,
                       long long k_pos0, void* stream) {
    CallRange range("attn_fwd_positions");
    if (!q || !k || !v || !o) return GBATTN_ERR_INVALID_ARG;
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || Sq <= 0 || Skv <= 0 || d <= 0)
        return GBATTN_ERR_INVALID_ARG;
    if (Hq % Hkv != 0) return GBATTN_ERR_INVALID_ARG;
    if (!(scale > 0.f) || scale != scale) return GBATTN_ERR_INVALID_ARG;
    constexpr long long kPosMax = 1LL << 40;
    if (q_pos0 < -kPosMax || q_pos0 > kPosMax || k_pos0 < -kPosMax || k_pos0 > kPosMax)
        return GBATTN_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return GBATTN_ERR_UNSUPPORTED;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) ||
        (lse && !aligned16(lse)))
        return GBATTN_ERR_MISALIGNED;
    if ((long long)B * Hq > 65535LL * 65535LL || (long long)B * Hq * Sq > kIntMax ||
        (long long)B * Hkv * Skv > kIntMax)
        return GBATTN_ERR_TOO_LARGE;
    // query row i sees key j iff j <= i + diag; beyond [-Sq, Skv] the clamp changes nothing
    // (every row sees all keys, or none)
    const int diag = (int)std::max<long long>(-(long long)Sq,
                                              std::min<long long>(Skv, q_pos0 - k_pos0));
    const int row0 = std::min(Sq, std::max(0, -diag));   // rows [0, row0) see no key
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int nsm = sm_count();
    if (nsm <= 0) return GBATTN_ERR_CUDA;
    int* err = device_error_word();
    if (!err) return GBATTN_ERR_CUDA;
    if (row0 > 0 &&
        launch_fill_empty_rows(static_cast<__nv_bfloat16*>(o), lse, (long long)B * Hq, Sq, row0,
                               d, nsm, err, st) != cudaSuccess)
        return GBATTN_ERR_CUDA;
    if (row0 == Sq) return GBATTN_OK;
    return launch_prefill_bf16(q, k, v, o, lse, B, Hq, Hkv, Sq, Skv, Skv, d, scale, 1, diag, row0,
                               st);
}

int attn_merge(const void* o_a, const float* lse_a, int dtype_a, const void* o_b,
               const float* lse_b, int dtype_b, void* o_out, float* lse_out, int dtype_out,
               long long rows, int d, void* stream) {
    CallRange range("attn_merge");
    auto dtype_ok = [](int t) { return t == GBATTN_BF16 || t == GBATTN_FP32; };
    if (!dtype_ok(dtype_a) || !dtype_ok(dtype_b) || !dtype_ok(dtype_out))
        return GBATTN_ERR_INVALID_ARG;
    if (rows < 0 || d <= 0) return GBATTN_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return GBATTN_ERR_UNSUPPORTED;
    if (rows == 0) return GBATTN_OK;             // nothing to read or write
    if (!o_a || !lse_a || !o_b || !lse_b || !o_out) return GBATTN_ERR_INVALID_ARG;
    if (!aligned16(o_a) || !aligned16(o_b) || !aligned16(o_out) ||
        (reinterpret_cast<uintptr_t>(lse_a) & 3u) || (reinterpret_cast<uintptr_t>(lse_b) & 3u) ||
        (reinterpret_cast<uintptr_t>(lse_out) & 3u))
        return GBATTN_ERR_MISALIGNED;
    if (rows > (1LL << 40)) return GBATTN_ERR_TOO_LARGE;
    const int nsm = sm_count();
    if (nsm <= 0) return GBATTN_ERR_CUDA;
    int* err = device_error_word();
    if (!err) return GBATTN_ERR_CUDA;
    return launch_attn_merge(o_a, lse_a, dtype_a == GBATTN_FP32, o_b, lse_b,
                             dtype_b == GBATTN_FP32, o_out, lse_out, dtype_out == GBATTN_FP32,
                             rows, d, nsm, err, static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? GBATTN_OK
               : GBATTN_ERR_CUDA;
}

size_t attn_decode_workspace_bytes(int B, int Hq, int Hkv, int Tq, int Lmax, int d,
                                   int num_splits, int num_sms) {
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || Tq <= 0 || Lmax <= 0 || (d != 64 && d != 128)) return 0;
    if (num_splits < 0 || num_splits > kMaxSplits || num_sms <= 0) return 0;
    if (Hq % Hkv != 0) return 0;
    if ((long long)B * Hq * Tq > kIntMax) return 0;
    const DecodePlan pl = decode_plan(B, Hq, Hkv, Tq, Lmax, num_splits, num_sms);
    return decode_workspace_bytes(B * Tq, Hq, B * Hkv, pl.dr.n_hg, d, pl.n_slots * pl.pieces);
}

size_t attn_decode_workspace_size(int B, int Hq, int Hkv, int Lmax, int d, int num_splits) {
    return attn_decode_multitoken_workspace_size(B, Hq, Hkv, 1, Lmax, d, num_splits);
}

size_t attn_decode_multitoken_workspace_size(int B, int Hq, int Hkv, int Tq, int Lmax, int d,
                                             int num_splits) {
    const int nsm = sm_count();
    if (nsm <= 0) return 0;
    return attn_decode_workspace_bytes(B, Hq, Hkv, Tq, Lmax, d, num_splits, nsm);
}

int attn_decode_multitoken(const void* q, const void* kcache, const void* vcache,
                           const int* kv_lens, void* o, float* lse, int B, int Hq, int Hkv,
                           int Tq, int Lmax, int d, float scale, int num_splits,
                           void* workspace, size_t ws_bytes, void* stream) {
    CallRange range("attn_decode");
    if (!q || !kcache || !vcache || !kv_lens || !o) return GBATTN_ERR_INVALID_ARG;
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || Tq <= 0 || Lmax <= 0 || d <= 0)
        return GBATTN_ERR_INVALID_ARG;
    if (Hq % Hkv != 0) return GBATTN_ERR_INVALID_ARG;
    if (!(scale > 0.f) || scale != scale) return GBATTN_ERR_INVALID_ARG;
    if (num_splits < 0 || num_splits > kMaxSplits) return GBATTN_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return GBATTN_ERR_UNSUPPORTED;
    if (Tq > 64) return GBATTN_ERR_UNSUPPORTED;
    if (!aligned16(q) || !aligned16(kcache) || !aligned16(vcache) || !aligned16(o) ||
        (lse && !aligned16(lse)) || (reinterpret_cast<uintptr_t>(kv_lens) & 3u))
        return GBATTN_ERR_MISALIGNED;
    if ((long long)B * Hq * Tq > kIntMax / 8) return GBATTN_ERR_TOO_LARGE;
    const int nsm = sm_count();
    if (nsm <= 0) return GBATTN_ERR_CUDA;
    const DecodePlan pl = decode_plan(B, Hq, Hkv, Tq, Lmax, num_splits, nsm);
    const DecodeRows dr = pl.dr;
    const int n_slots = pl.n_slots;
    const int n_parts = pl.n_slots * pl.pieces;
    const size_t need = decode_workspace_bytes(B * Tq, Hq, B * Hkv, dr.n_hg, d, n_parts);
    if (!workspace || ws_bytes < need) return GBATTN_ERR_WORKSPACE;
    if (!aligned16(workspace)) return GBATTN_ERR_MISALIGNED;
    const int G = Hq / Hkv;
    const int R = dr.R, n_hc = dr.n_hc, nci = dr.nci, n_hg = dr.n_hg;
    const long long n_items = pl.n_items;
    if (n_items > kIntMax || (long long)B * Hkv * Lmax > kIntMax) return GBATTN_ERR_TOO_LARGE;

    DecodeParams p{};
    if (!make_map_bf16_3d(&p.tmap_k, kcache, d, Lmax, (uint64_t)B * Hkv, 64) ||
        !make_map_bf16_3d(&p.tmap_v, vcache, d, Lmax, (uint64_t)B * Hkv, 64) ||
        !make_map_bf16_3d(&p.tmap_q, q, d, (uint64_t)B * Hq * Tq, 1, 8))
        return GBATTN_ERR_CUDA;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    const size_t rows = (size_t)B * Hq * Tq * n_parts;
    const size_t cnt_bytes = decode_counter_bytes(B, Hkv, n_hg);
    p.counter = reinterpret_cast<int*>(ws);
    p.group_cnt = p.counter + 1;
    p.ws_lse = reinterpret_cast<float*>(ws + cnt_bytes);
    p.ws_o = reinterpret_cast<float*>(ws + cnt_bytes + ((rows * 4 + 255) / 256) * 256);
    p.kv_lens = kv_lens;
    p.o = static_cast<__nv_bfloat16*>(o);
    p.lse = lse;
    p.B = B; p.Hq = Hq; p.Hkv = Hkv; p.Lmax = Lmax; p.G = G;
    p.Tq = Tq;
    p.R = R;
    p.n_hc = n_hc;
    p.nci = nci;
    p.n_hg = n_hg;
    p.n_slots = n_slots;
    p.pieces = pl.pieces;
    p.n_parts = n_parts;
    p.fixed_splits = num_splits;
    p.auto_floor = pl.floor_splits;
    p.combine_lanes = pl.combine_lanes;
    p.n_items = (int)n_items;
    p.fused = pl.fused ? 1 : 0;
    p.counted = pl.counted ? 1 : 0;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.err = device_error_word();
    if (!p.err) return GBATTN_ERR_CUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (pl.tc) {
        // tcgen05 path: the KV head's rows as the M = 128 operand, each K/V tile read once
        // per 128 rows; the combine folds the partials as for the split kernel
        DecodeTcParams tp{};
        const int q_rows = pl.q_rows;
        if (!make_map_bf16_3d(&tp.tmap_q, q, d, (uint64_t)B * Hq * Tq, 1, (uint32_t)q_rows) ||
            !make_map_bf16_3d(&tp.tmap_k, kcache, d, Lmax, (uint64_t)B * Hkv, 128) ||
            !make_map_bf16_3d(&tp.tmap_v, vcache, d, Lmax, (uint64_t)B * Hkv, 128))
            return GBATTN_ERR_CUDA;
        tp.kv_lens = kv_lens;
        tp.o = p.o;
        tp.lse = lse;
        tp.ws_lse = p.ws_lse;
        tp.ws_o = p.ws_o;
        tp.B = B; tp.Hq = Hq; tp.Hkv = Hkv; tp.Lmax = Lmax; tp.Tq = Tq;
        tp.R = R;
        tp.q_rows = q_rows;
        tp.n_rt = pl.n_rt;
        tp.n_slots = n_slots;
        tp.pieces = pl.pieces;
        tp.n_parts = n_parts;
        tp.fixed_splits = num_splits;
        tp.auto_floor = pl.floor_splits;
        const long long tc_items = pl.tc_items;
        if (tc_items > kIntMax) return GBATTN_ERR_TOO_LARGE;
        tp.n_items = (int)tc_items;
        tp.counter = p.counter;
        tp.group_cnt = p.group_cnt;
        tp.counted = p.counted;
        tp.scale_log2 = p.scale_log2;
        tp.err = p.err;
        cudaError_t e = launch_decode_multitoken_tc(tp, d, nsm, st);
        if (e == cudaSuccess) e = launch_decode_combine(p, d, st);
        return e == cudaSuccess ? GBATTN_OK : GBATTN_ERR_CUDA;
    }
    cudaError_t e = launch_decode_splitkv(p, d, nsm, st);
    return e == cudaSuccess ? GBATTN_OK : GBATTN_ERR_CUDA;
}

int attn_decode_splitkv(const void* q, const void* kcache, const void* vcache,
                        const int* kv_lens, void* o, float* lse, int B, int Hq, int Hkv,
                        int Lmax, int d, float scale, int num_splits, void* workspace,
                        size_t ws_bytes, void* stream) {
    return attn_decode_multitoken(q, kcache, vcache, kv_lens, o, lse, B, Hq, Hkv, 1, Lmax, d,
                                  scale, num_splits, workspace, ws_bytes, stream);
}

// ---- host-buffer decode: the sequences in up to 4 chunks, copies overlapped -------------
// Each chunk is a run of consecutive sequences -- contiguous slabs of q / o ([Hq, d]), the
// caches ([Hkv, Lmax, d]), kv_lens and LSE -- staged through two device buffer sets as in
// attn_fwd_host, and decoded by attn_decode_splitkv on the staged copies with a decode
// workspace shared by the chunks (their decodes run in order on the caller's stream).
struct DecodeHostPlan {
    int cb, n_chunks, n_bufs;
    size_t q_off, k_off, v_off, n_off, o_off, l_off, set_bytes, dec_off, dec_bytes;
};

bool decode_host_plan(int B, int Hq, int Hkv, int Lmax, int d, int num_splits,
                      DecodeHostPlan& h) {
    h.cb = (B + 3) / 4;
    h.n_chunks = (B + h.cb - 1) / h.cb;
    h.n_bufs = h.n_chunks > 1 ? 2 : 1;
    const size_t qb = (size_t)h.cb * Hq * d * 2, kb = (size_t)h.cb * Hkv * Lmax * d * 2;
    h.q_off = 0;
    h.k_off = align256(qb);
    h.v_off = h.k_off + align256(kb);
    h.n_off = h.v_off + align256(kb);
    h.o_off = h.n_off + align256((size_t)h.cb * 4);
    h.l_off = h.o_off + align256(qb);
    h.set_bytes = h.l_off + align256((size_t)h.cb * Hq * 4);
    h.dec_off = h.set_bytes * h.n_bufs;
    const int last = B - (h.n_chunks - 1) * h.cb;
    const size_t w0 = attn_decode_workspace_size(h.cb, Hq, Hkv, Lmax, d, num_splits);
    const size_t w1 = attn_decode_workspace_size(last, Hq, Hkv, Lmax, d, num_splits);
    if (w0 == 0 || w1 == 0) return false;
    h.dec_bytes = std::max(w0, w1);
    return true;
}

size_t attn_decode_host_workspace_size(int B, int Hq, int Hkv, int Lmax, int d, int num_splits) {
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || Lmax <= 0 || Hq % Hkv != 0) return 0;
    if ((d != 64 && d != 128) || num_splits < 0 || num_splits > kMaxSplits) return 0;
    DecodeHostPlan h{};
    if (!decode_host_plan(B, Hq, Hkv, Lmax, d, num_splits, h)) return 0;
    return h.dec_off + h.dec_bytes;
}

int attn_decode_host(const void* q, const void* kcache, const void* vcache, const int* kv_lens,
                     void* o, float* lse, int B, int Hq, int Hkv, int Lmax, int d, float scale,
                     int num_splits, void* workspace, size_t ws_bytes, void* stream) {
    CallRange range("attn_decode_host");
    if (!q || !kcache || !vcache || !kv_lens || !o) return GBATTN_ERR_INVALID_ARG;
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || Lmax <= 0 || d <= 0) return GBATTN_ERR_INVALID_ARG;
    if (Hq % Hkv != 0) return GBATTN_ERR_INVALID_ARG;
    if (!(scale > 0.f) || scale != scale) return GBATTN_ERR_INVALID_ARG;
    if (num_splits < 0 || num_splits > kMaxSplits) return GBATTN_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return GBATTN_ERR_UNSUPPORTED;
    for (int b = 0; b < B; ++b)                  // the lengths are on the host: check them here
        if (kv_lens[b] < 0 || kv_lens[b] > Lmax) return GBATTN_ERR_INVALID_ARG;
    if ((long long)B * Hq > kIntMax / 8 || (long long)B * Hkv * Lmax > kIntMax)
        return GBATTN_ERR_TOO_LARGE;
    const size_t need = attn_decode_host_workspace_size(B, Hq, Hkv, Lmax, d, num_splits);
    if (need == 0) return GBATTN_ERR_CUDA;
    if (!workspace || ws_bytes < need) return GBATTN_ERR_WORKSPACE;
    if (!aligned16(workspace)) return GBATTN_ERR_MISALIGNED;
    HostPipe* hp = host_pipe();
    if (!hp) return GBATTN_ERR_CUDA;
    std::lock_guard<std::mutex> lock(hp->mu);

    DecodeHostPlan h{};
    if (!decode_host_plan(B, Hq, Hkv, Lmax, d, num_splits, h)) return GBATTN_ERR_CUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const char* qh = static_cast<const char*>(q);
    const char* kh = static_cast<const char*>(kcache);
    const char* vh = static_cast<const char*>(vcache);
    const char* nh = reinterpret_cast<const char*>(kv_lens);
    char* oh = static_cast<char*>(o);
    char* lh = reinterpret_cast<char*>(lse);
    char* ws = static_cast<char*>(workspace);
    const size_t qs = (size_t)Hq * d * 2, ks = (size_t)Hkv * Lmax * d * 2, ls = (size_t)Hq * 4;
    auto chk = [](cudaError_t e) { return e == cudaSuccess; };
    bool ok = chk(cudaEventRecord(hp->entry, st));   // the caller's earlier work comes first
    for (int i = 0; ok && i < h.n_chunks; ++i) {
        const int bset = i % h.n_bufs;
        const int b0 = i * h.cb, bn = std::min(h.cb, B - b0);
        char* base = ws + (size_t)bset * h.set_bytes;
        ok = chk(cudaStreamWaitEvent(hp->in, i >= h.n_bufs ? hp->ev_out[bset] : hp->entry, 0)) &&
             chk(cudaMemcpyAsync(base + h.q_off, qh + b0 * qs, bn * qs, cudaMemcpyHostToDevice, hp->in)) &&
             chk(cudaMemcpyAsync(base + h.k_off, kh + b0 * ks, bn * ks, cudaMemcpyHostToDevice, hp->in)) &&
             chk(cudaMemcpyAsync(base + h.v_off, vh + b0 * ks, bn * ks, cudaMemcpyHostToDevice, hp->in)) &&
             chk(cudaMemcpyAsync(base + h.n_off, nh + b0 * 4, bn * 4, cudaMemcpyHostToDevice, hp->in)) &&
             chk(cudaEventRecord(hp->ev_in[bset], hp->in)) &&
             chk(cudaStreamWaitEvent(st, hp->ev_in[bset], 0));
        if (!ok) break;
        const int rc = attn_decode_splitkv(
            base + h.q_off, base + h.k_off, base + h.v_off,
            reinterpret_cast<const int*>(base + h.n_off), base + h.o_off,
            lh ? reinterpret_cast<float*>(base + h.l_off) : nullptr, bn, Hq, Hkv, Lmax, d, scale,
            num_splits, ws + h.dec_off, h.dec_bytes, stream);
        if (rc != GBATTN_OK) return rc;
        ok = chk(cudaEventRecord(hp->ev_comp[bset], st)) &&
             chk(cudaStreamWaitEvent(hp->out, hp->ev_comp[bset], 0)) &&
             chk(cudaMemcpyAsync(oh + b0 * qs, base + h.o_off, bn * qs, cudaMemcpyDeviceToHost, hp->out)) &&
             (!lh || chk(cudaMemcpyAsync(lh + b0 * ls, base + h.l_off, bn * ls, cudaMemcpyDeviceToHost, hp->out))) &&
             chk(cudaEventRecord(hp->ev_out[bset], hp->out));
    }
    // the caller's stream completes after the last copy out
    ok = ok && chk(cudaEventRecord(hp->done, hp->out)) && chk(cudaStreamWaitEvent(st, hp->done, 0));
    return ok ? GBATTN_OK : GBATTN_ERR_CUDA;
}

int attn_decode_plan(int B, int Hq, int Hkv, int Tq, int Lmax, int d, int num_splits,
                     int num_sms, int* plan) {
    if (!plan) return GBATTN_ERR_INVALID_ARG;
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || Tq <= 0 || Lmax <= 0 || num_sms <= 0)
        return GBATTN_ERR_INVALID_ARG;
    if (Hq % Hkv != 0 || num_splits < 0 || num_splits > kMaxSplits) return GBATTN_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return GBATTN_ERR_UNSUPPORTED;
    if (Tq > 64) return GBATTN_ERR_UNSUPPORTED;
    if ((long long)B * Hq * Tq > kIntMax / 8) return GBATTN_ERR_TOO_LARGE;
    const DecodePlan pl = decode_plan(B, Hq, Hkv, Tq, Lmax, num_splits, num_sms);
    const long long items = pl.tc ? pl.tc_items : pl.n_items;
    if (items > kIntMax) return GBATTN_ERR_TOO_LARGE;
    plan[0] = pl.n_slots;
    plan[1] = pl.tc ? 1 : 0;
    plan[2] = pl.fused ? 1 : (pl.counted ? 2 : 0);
    plan[3] = (int)items;
    plan[4] = pl.dr.R;
    plan[5] = pl.combine_lanes;
    plan[6] = pl.pieces;
    return GBATTN_OK;
}

int attn_prefill_plan(int B, int Hq, int Hkv, int Sq, int Skv, int causal, int num_sms,
                      int* plan) {
    if (!plan) return GBATTN_ERR_INVALID_ARG;
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || Sq <= 0 || Skv <= 0 || num_sms <= 0)
        return GBATTN_ERR_INVALID_ARG;
    if (Hq % Hkv != 0) return GBATTN_ERR_INVALID_ARG;
    if (causal && Sq > Skv) return GBATTN_ERR_UNSUPPORTED;
    const PrefillPlan pl = prefill_plan(B, Hq, Hkv, Sq, Skv, causal, num_sms, Skv - Sq, 0);
    if (pl.n_pairs > kIntMax || pl.n_tiles > kIntMax) return GBATTN_ERR_TOO_LARGE;
    plan[0] = pl.kv_split ? 1 : 0;
    plan[1] = (int)pl.first;
    plan[2] = (int)pl.tail;
    plan[3] = (int)pl.n_tiles;
    return GBATTN_OK;
}

#ifdef GBATTN_DEBUG_CHECKS
}  // extern "C"
namespace gbattn {
cudaError_t debug_skip_fill_pairs(int fill);
cudaError_t debug_skip_fill_persist(int fill);
cudaError_t debug_skip_fill_split(int fill);
cudaError_t debug_skip_fill_multitoken(int fill);
}  // namespace gbattn
extern "C" {

int attn_debug_skip_fill(int kernel, int fill) {
    if (fill < -1) return GBATTN_ERR_INVALID_ARG;
    cudaError_t e;
    if (kernel == GBATTN_DEBUG_PERSISTENT_PREFILL)
        e = debug_skip_fill_persist(fill);
    else if (kernel == GBATTN_DEBUG_MULTITOKEN_DECODE)
        e = debug_skip_fill_multitoken(fill);
    else if (kernel == GBATTN_DEBUG_PAIR_PREFILL)
        e = debug_skip_fill_pairs(fill);
    else if (kernel == GBATTN_DEBUG_SPLIT_DECODE)
        e = debug_skip_fill_split(fill);
    else
        return GBATTN_ERR_INVALID_ARG;
    return e == cudaSuccess ? GBATTN_OK : GBATTN_ERR_CUDA;
}
#endif

int attn_selftest_bounded_wait(void* stream) {
    int* err = device_error_word();
    if (!err) return GBATTN_ERR_CUDA;
    selftest_wait_kernel<<<1, 1, 0, static_cast<cudaStream_t>(stream)>>>(err, 2000000LL);
    return cudaGetLastError() == cudaSuccess ? GBATTN_OK : GBATTN_ERR_CUDA;
}

int attn_last_device_error(void* stream, int* detail) {
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return GBATTN_ERR_CUDA;
    int word = 0;
    if (cudaMemcpyFromSymbol(&word, g_device_error, sizeof(int)) != cudaSuccess)
        return GBATTN_ERR_CUDA;
    if (detail) *detail = word;
    if (word != 0) {
        const int zero = 0;
        if (cudaMemcpyToSymbol(g_device_error, &zero, sizeof(int)) != cudaSuccess)
            return GBATTN_ERR_CUDA;
        return GBATTN_ERR_TIMEOUT;
    }
    return GBATTN_OK;
}

}  // extern "C"
