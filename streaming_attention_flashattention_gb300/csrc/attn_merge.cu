// attn_merge.cu -- the log-sum-exp merge of two partial attention results, and the fill of
// query rows that see no key.
//
// Merge: "ADR-0060: AHBM GQA Fused Attention Kernel (Llama3-70B)", section 4 (reduction for
// KV-parallel / sequence-parallel decode): two partial results over disjoint key sets,
// (m_a, l_a, O_a) and (m_b, l_b, O_b), combine associatively and commutatively into the
// result over the union, m = max(m_a, m_b), l = l_a e^(m_a - m) + l_b e^(m_b - m), O likewise,
// normalised once at the end.  The partials here are already normalised and carry their
// log-sum-exp L = m + ln l, so with M = max(L_a, L_b) and w_x = e^(L_x - M):
//     O = (w_a O_a + w_b O_b) / (w_a + w_b),    L = M + ln(w_a + w_b).
// A partial over no key has L = -inf (w = 0) and adds nothing; if both have none the row is
// O = 0, L = -inf.
//
// Layout: rows of d contiguous elements; one warp handles 128 / d rows at a time (d / 4 lanes
// per row, 4 elements per lane).  Out may alias either input (see merge_kernel).
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace gbattn {

namespace {

template <typename T> struct Vec4;
template <> struct Vec4<float> {
    __device__ static void load(const float* p, float (&v)[4]) {
        const float4 x = *reinterpret_cast<const float4*>(p);
        v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
    }
    __device__ static void store(float* p, const float (&v)[4]) {
        *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
    }
};
template <> struct Vec4<__nv_bfloat16> {
    __device__ static void load(const __nv_bfloat16* p, float (&v)[4]) {
        const uint2 x = *reinterpret_cast<const uint2*>(p);
        const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&x.x));
        const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&x.y));
        v[0] = lo.x; v[1] = lo.y; v[2] = hi.x; v[3] = hi.y;
    }
    __device__ static void store(__nv_bfloat16* p, const float (&v)[4]) {
        *reinterpret_cast<uint2*>(p) = make_uint2(pack_bf16(v[0], v[1]), pack_bf16(v[2], v[3]));
    }
};

// Each warp takes kUnroll units (rows-per-warp groups) per pass and issues all their loads --
// both LSE values and both O vectors of every lane -- before any arithmetic, so that one pass
// waits for one memory latency; a partial whose weight is 0 is then ignored by selection
// (never multiplied, so whatever its O holds cannot leak in).  Every lane reads its row's LSE
// values itself; the warp synchronises before the stores, so the merged LSE may overwrite an
// input that other lanes of the row have read.
constexpr int kUnroll = 2;

template <typename TA, typename TB, typename TO>
__global__ void __launch_bounds__(256)
merge_kernel(const TA* oa, const float* la, const TB* ob, const float* lb, TO* oo, float* lo,
             long long rows, int d, int* err) {
    const int lane = threadIdx.x & 31;
    const int lpr = d >> 2;                          // lanes per row
    const int rpw = 32 / lpr;                        // rows per warp unit
    const int sub = lane / lpr, col = (lane % lpr) * 4;
    const long long warps = (long long)gridDim.x * (blockDim.x >> 5);
    const long long units = (rows + rpw - 1) / rpw;
    const long long wid = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    for (long long u0 = wid; u0 < units; u0 += warps * kUnroll) {
        long long row[kUnroll];
        float lsa[kUnroll], lsb[kUnroll], va[kUnroll][4], vb[kUnroll][4];
        #pragma unroll
        for (int x = 0; x < kUnroll; ++x) {
            row[x] = (u0 + x * warps) * rpw + sub;
            lsa[x] = lsb[x] = -INFINITY;
            #pragma unroll
            for (int e = 0; e < 4; ++e) va[x][e] = vb[x][e] = 0.f;
            if (u0 + x * warps < units && row[x] < rows) {
                lsa[x] = la[row[x]];
                lsb[x] = lb[row[x]];
                Vec4<TA>::load(oa + row[x] * d + col, va[x]);
                Vec4<TB>::load(ob + row[x] * d + col, vb[x]);
            }
        }
        __syncwarp();
        #pragma unroll
        for (int x = 0; x < kUnroll; ++x) {
            if (!(u0 + x * warps < units && row[x] < rows)) continue;
            const float M = fmaxf(lsa[x], lsb[x]);
            float w_a = 0.f, w_b = 0.f;
            if (M != -INFINITY) {
                w_a = expf(lsa[x] - M);              // e^-inf = 0 for an empty partial
                w_b = expf(lsb[x] - M);
            }
            const float s = w_a + w_b;
            const float inv = s > 0.f ? 1.f / s : 0.f;
            float r[4];
            #pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float ta = w_a > 0.f ? w_a * va[x][e] : 0.f;
                const float tb = w_b > 0.f ? w_b * vb[x][e] : 0.f;
                r[e] = (ta + tb) * inv;
            }
            if (GBATTN_IN_BOUNDS(row[x] * d + col + 3, rows * d, err))
                Vec4<TO>::store(oo + row[x] * d + col, r);
            if (lo != nullptr && lane % lpr == 0 && GBATTN_IN_BOUNDS(row[x], rows, err))
                lo[row[x]] = s > 0.f ? M + logf(s) : -INFINITY;
        }
    }
}

template <typename TA, typename TB, typename TO>
cudaError_t launch_merge_t(const void* oa, const float* la, const void* ob, const float* lb,
                           void* oo, float* lo, long long rows, int d, int nsm, int* err,
                           cudaStream_t st) {
    constexpr int kThreads = 256;
    const long long units = (rows + (128 / d) - 1) / (128 / d);
    // one wave: as many blocks as fit on the SMs at once (registers decide), so that the
    // grid-stride loop gives every block the same share (a second, partial wave of blocks
    // measured 7-13% slower)
    static int occ = 0;
    if (occ == 0 && cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                        &occ, merge_kernel<TA, TB, TO>, kThreads, 0) != cudaSuccess)
        occ = 4;
    const long long blocks = std::min<long long>((units + 8 * kUnroll - 1) / (8 * kUnroll),
                                                 (long long)nsm * std::max(occ, 1));
    merge_kernel<TA, TB, TO><<<(unsigned)std::max<long long>(blocks, 1), kThreads, 0, st>>>(
        static_cast<const TA*>(oa), la, static_cast<const TB*>(ob), lb, static_cast<TO*>(oo), lo,
        rows, d, err);
    return cudaGetLastError();
}

template <typename TA, typename TB>
cudaError_t launch_merge_ab(const void* oa, const float* la, const void* ob, const float* lb,
                            void* oo, float* lo, bool out_f32, long long rows, int d, int nsm,
                            int* err, cudaStream_t st) {
    return out_f32 ? launch_merge_t<TA, TB, float>(oa, la, ob, lb, oo, lo, rows, d, nsm, err, st)
                   : launch_merge_t<TA, TB, __nv_bfloat16>(oa, la, ob, lb, oo, lo, rows, d, nsm, err,
                                                          st);
}

// Rows [0, row0) of every (batch, head): O = 0, L = -inf.  One thread per 16 bytes of O.
__global__ void __launch_bounds__(256)
fill_empty_rows_kernel(__nv_bfloat16* o, float* lse, long long bh, int Sq, int row0, int d,
                       int* err) {
    const int chunks = d / 8;                        // 16-byte chunks per row
    const long long total = bh * row0 * chunks;
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += stride) {
        const long long r = i / chunks;              // (head, row) pair
        const int c = (int)(i % chunks);
        const long long head = r / row0, row = r % row0;
        const long long g = head * Sq + row;
        if (GBATTN_IN_BOUNDS(g * d + c * 8 + 7, bh * Sq * d, err))
            *reinterpret_cast<uint4*>(o + g * d + c * 8) = make_uint4(0u, 0u, 0u, 0u);
        if (lse != nullptr && c == 0 && GBATTN_IN_BOUNDS(g, bh * Sq, err)) lse[g] = -INFINITY;
    }
}

}  // namespace

cudaError_t launch_attn_merge(const void* oa, const float* la, bool a_f32, const void* ob,
                              const float* lb, bool b_f32, void* oo, float* lo, bool out_f32,
                              long long rows, int d, int nsm, int* err, cudaStream_t st) {
    if (rows <= 0) return cudaSuccess;
    using bf = __nv_bfloat16;
    if (a_f32)
        return b_f32 ? launch_merge_ab<float, float>(oa, la, ob, lb, oo, lo, out_f32, rows, d, nsm,
                                                     err, st)
                     : launch_merge_ab<float, bf>(oa, la, ob, lb, oo, lo, out_f32, rows, d, nsm,
                                                  err, st);
    return b_f32 ? launch_merge_ab<bf, float>(oa, la, ob, lb, oo, lo, out_f32, rows, d, nsm, err, st)
                 : launch_merge_ab<bf, bf>(oa, la, ob, lb, oo, lo, out_f32, rows, d, nsm, err, st);
}

cudaError_t launch_fill_empty_rows(__nv_bfloat16* o, float* lse, long long bh, int Sq, int row0,
                                   int d, int nsm, int* err, cudaStream_t st) {
    if (bh <= 0 || row0 <= 0) return cudaSuccess;
    const long long total = bh * row0 * (d / 8);
    const long long blocks = std::min<long long>((total + 255) / 256, (long long)nsm * 8);
    fill_empty_rows_kernel<<<(unsigned)blocks, 256, 0, st>>>(o, lse, bh, Sq, row0, d, err);
    return cudaGetLastError();
}

}  // namespace gbattn
