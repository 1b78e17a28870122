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
// Layout: rows of d contiguous elements; one warp handles 128 / d rows (d / 4 lanes per row,
// 4 elements per lane), so a row's lanes read its two LSE values and one of them writes the
// merged one after the warp has exchanged them -- out may alias either input.
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

template <typename TA, typename TB, typename TO>
__global__ void __launch_bounds__(256)
merge_kernel(const TA* oa, const float* la, const TB* ob, const float* lb, TO* oo, float* lo,
             long long rows, int d, int* err) {
    const int lane = threadIdx.x & 31;
    const int lpr = d >> 2;                          // lanes per row
    const int rpw = 32 / lpr;                        // rows per warp
    const int sub = lane / lpr, col = (lane % lpr) * 4;
    const long long warps = (long long)gridDim.x * (blockDim.x >> 5);
    const long long units = (rows + rpw - 1) / rpw;
    for (long long u = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); u < units;
         u += warps) {
        const long long row = u * rpw + sub;
        const bool live = row < rows;
        float lsa = -INFINITY, lsb = -INFINITY;
        if (live && lane % lpr == 0) {
            lsa = la[row];
            lsb = lb[row];
        }
        const int leader = sub * lpr;
        lsa = __shfl_sync(0xffffffffu, lsa, leader);
        lsb = __shfl_sync(0xffffffffu, lsb, leader);
        if (!live) continue;
        const float M = fmaxf(lsa, lsb);
        float w_a = 0.f, w_b = 0.f;
        if (M != -INFINITY) {
            w_a = expf(lsa - M);                     // e^-inf = 0 for an empty partial
            w_b = expf(lsb - M);
        }
        const float s = w_a + w_b;
        const float inv = s > 0.f ? 1.f / s : 0.f;
        float va[4] = {0.f, 0.f, 0.f, 0.f}, vb[4] = {0.f, 0.f, 0.f, 0.f}, r[4];
        if (w_a > 0.f) Vec4<TA>::load(oa + row * d + col, va);
        if (w_b > 0.f) Vec4<TB>::load(ob + row * d + col, vb);
        #pragma unroll
        for (int e = 0; e < 4; ++e) r[e] = (w_a * va[e] + w_b * vb[e]) * inv;
        if (GBATTN_IN_BOUNDS(row * d + col + 3, rows * d, err)) Vec4<TO>::store(oo + row * d + col, r);
        if (lo != nullptr && lane % lpr == 0 && GBATTN_IN_BOUNDS(row, rows, err))
            lo[row] = s > 0.f ? M + logf(s) : -INFINITY;
    }
}

template <typename TA, typename TB, typename TO>
cudaError_t launch_merge_t(const void* oa, const float* la, const void* ob, const float* lb,
                           void* oo, float* lo, long long rows, int d, int nsm, int* err,
                           cudaStream_t st) {
    constexpr int kThreads = 256;
    const long long units = (rows + (128 / d) - 1) / (128 / d);
    const long long blocks = std::min<long long>((units + 7) / 8, (long long)nsm * 8);
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
