// attn_f32.cu -- exact-fp32 streaming attention forward on CUDA cores.
//
// Serves GBATTN_FP32 inputs (fp32 Q/K/V/O), where a bf16 or tf32 tensor-core product
// would miss a 1e-4 tolerance.  Same algorithm as the tensor-core path: a resident Q
// tile, K/V tiles streamed through shared memory, and the online softmax update of
// "AttentionRegion Transformation" section 6 / "ADR-0060" section 3 (running max m,
// running sum l, O rescaled by exp(m_old - m_new)), normalised once at the end.
//
// Mapping: a CTA owns 16 query rows of one (b, h); each warp owns 4 rows.  Per 32-key
// tile, lane j computes the score of key j for the warp's row, the warp reduces max and
// sum with shuffles, and each lane accumulates its own d/32 output columns.
#include "common.cuh"
#include "kernels.h"

namespace gbattn {

namespace {

constexpr int kWarps = 4;
constexpr int kRowsPerWarp = 4;
constexpr int kRowsPerCta = kWarps * kRowsPerWarp;
constexpr int kKeysPerTile = 32;

template <int D>
__global__ void __launch_bounds__(kWarps * 32)
attn_fwd_f32_kernel(const float* __restrict__ q, const float* __restrict__ k,
                    const float* __restrict__ v, float* __restrict__ o, float* __restrict__ lse,
                    int Hq, int Hkv, int Sq, int Skv, float scale_log2, int causal,
                    int* err) {
    constexpr int P = D + 1;  // padded row: lane j reading row j is conflict free
    constexpr int C = D / 32; // output columns per lane
    __shared__ float sq[kRowsPerCta][D];
    __shared__ float sk[kKeysPerTile][P];
    __shared__ float sv[kKeysPerTile][P];

    const int b = blockIdx.z, h = blockIdx.y;
    const int row0 = blockIdx.x * kRowsPerCta;
    const int kvh = h / (Hq / Hkv);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long q_base = ((long long)b * Hq + h) * Sq;
    const long long kv_base = ((long long)b * Hkv + kvh) * (long long)Skv * D;
    const int off = Skv - Sq;  // bottom-right causal offset

    // Tiles come in with 16-byte loads, all of a thread's loads issued before its shared
    // stores (a loop that stored each element before loading the next waited one memory
    // round trip per element group: ~60 us on a 128-key call after an L2 flush).
    constexpr int kThreads = kWarps * 32;
    constexpr int kV4 = D / 4;                                // float4 per row
    {
        constexpr int kPer = kRowsPerCta * kV4 / kThreads;
        float4 x[kPer];
#pragma unroll
        for (int it = 0; it < kPer; ++it) {
            const int idx = it * kThreads + threadIdx.x, r = idx / kV4, c4 = idx % kV4;
            x[it] = (row0 + r < Sq) ? reinterpret_cast<const float4*>(q + (q_base + row0 + r) * D)[c4]
                                    : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int it = 0; it < kPer; ++it) {
            const int idx = it * kThreads + threadIdx.x, r = idx / kV4, c4 = idx % kV4;
            sq[r][4 * c4] = x[it].x; sq[r][4 * c4 + 1] = x[it].y;
            sq[r][4 * c4 + 2] = x[it].z; sq[r][4 * c4 + 3] = x[it].w;
        }
    }

    float m[kRowsPerWarp], l[kRowsPerWarp], acc[kRowsPerWarp][C];
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
        m[r] = -INFINITY;
        l[r] = 0.f;
#pragma unroll
        for (int c = 0; c < C; ++c) acc[r][c] = 0.f;
    }

    // keys needed by this CTA: all of them, or up to the last row's causal limit
    int kv_end = Skv;
    if (causal) {
        const int last = min(row0 + kRowsPerCta, Sq) - 1;
        kv_end = min(Skv, last + off + 1);
    }

    for (int t0 = 0; t0 < kv_end; t0 += kKeysPerTile) {
        __syncthreads();
        {
            constexpr int kPer = kKeysPerTile * kV4 / kThreads;
            float4 xk[kPer], xv[kPer];
#pragma unroll
            for (int it = 0; it < kPer; ++it) {
                const int idx = it * kThreads + threadIdx.x, j = idx / kV4, c4 = idx % kV4;
                const bool ok = (t0 + j) < Skv;
                const long long at = kv_base + (long long)(t0 + j) * D;
                xk[it] = ok ? reinterpret_cast<const float4*>(k + at)[c4] : make_float4(0.f, 0.f, 0.f, 0.f);
                xv[it] = ok ? reinterpret_cast<const float4*>(v + at)[c4] : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int it = 0; it < kPer; ++it) {
                const int idx = it * kThreads + threadIdx.x, j = idx / kV4, c4 = idx % kV4;
                sk[j][4 * c4] = xk[it].x; sk[j][4 * c4 + 1] = xk[it].y;
                sk[j][4 * c4 + 2] = xk[it].z; sk[j][4 * c4 + 3] = xk[it].w;
                sv[j][4 * c4] = xv[it].x; sv[j][4 * c4 + 1] = xv[it].y;
                sv[j][4 * c4 + 2] = xv[it].z; sv[j][4 * c4 + 3] = xv[it].w;
            }
        }
        __syncthreads();

#pragma unroll
        for (int r = 0; r < kRowsPerWarp; ++r) {
            const int lr = warp * kRowsPerWarp + r;
            const int i = row0 + lr;
            const int key = t0 + lane;
            float dot = 0.f;
#pragma unroll 16
            for (int c = 0; c < D; ++c) dot = fmaf(sq[lr][c], sk[lane][c], dot);
            bool visible = key < Skv;
            if (causal) visible = visible && (key <= i + off);
            const float s = visible ? dot * scale_log2 : -INFINITY;
            float mt = s;
#pragma unroll
            for (int w = 16; w > 0; w >>= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, w));
            const float m_new = fmaxf(m[r], mt);
            if (m_new == -INFINITY) continue;  // nothing visible yet for this row
            const float corr = exp2f(m[r] - m_new);
            const float p = exp2f(s - m_new);
            float ps = p;
#pragma unroll
            for (int w = 16; w > 0; w >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, w);
            l[r] = l[r] * corr + ps;
            m[r] = m_new;
#pragma unroll
            for (int c = 0; c < C; ++c) acc[r][c] *= corr;
            for (int j = 0; j < kKeysPerTile; ++j) {
                const float pj = __shfl_sync(0xffffffffu, p, j);
#pragma unroll
                for (int c = 0; c < C; ++c) acc[r][c] = fmaf(pj, sv[j][lane + 32 * c], acc[r][c]);
            }
        }
    }

#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
        const int i = row0 + warp * kRowsPerWarp + r;
        if (i >= Sq) continue;
        if (!GBATTN_IN_BOUNDS(q_base + i, (long long)gridDim.z * Hq * Sq, err)) continue;
        const float inv = l[r] > 0.f ? 1.f / l[r] : 0.f;
#pragma unroll
        for (int c = 0; c < C; ++c) o[(q_base + i) * D + lane + 32 * c] = acc[r][c] * inv;
        if (lse != nullptr && lane == 0)
            lse[q_base + i] = l[r] > 0.f ? (m[r] + log2f(l[r])) * 0.69314718055994531f : -INFINITY;
    }
}

}  // namespace

cudaError_t launch_attn_fwd_f32(const float* q, const float* k, const float* v, float* o,
                                float* lse, int B, int Hq, int Hkv, int Sq, int Skv, int d,
                                float scale, int causal, int* err, cudaStream_t stream) {
    const float scale_log2 = scale * 1.4426950408889634f;
    dim3 grid((Sq + kRowsPerCta - 1) / kRowsPerCta, Hq, B);
    dim3 block(kWarps * 32);
    if (d == 64)
        attn_fwd_f32_kernel<64><<<grid, block, 0, stream>>>(q, k, v, o, lse, Hq, Hkv, Sq, Skv,
                                                            scale_log2, causal, err);
    else
        attn_fwd_f32_kernel<128><<<grid, block, 0, stream>>>(q, k, v, o, lse, Hq, Hkv, Sq, Skv,
                                                             scale_log2, causal, err);
    return cudaGetLastError();
}

}  // namespace gbattn
