// kernels.h -- internal launch interface between the C ABI (gbattn_api.cu) and the
// kernel translation units.  Not part of the public ABI.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace gbattn {

// Address of this device's error word (the word itself lives in gbattn_api.cu).
int* device_error_word();

// ---- fp32 CUDA-core path (attn_f32.cu) ------------------------------------------------
cudaError_t launch_attn_fwd_f32(const float* q, const float* k, const float* v, float* o,
                                float* lse, int B, int Hq, int Hkv, int Sq, int Skv, int d,
                                float scale, int causal, int* err, cudaStream_t stream);

// ---- bf16 tcgen05 prefill path (prefill_tcgen05.cu) ------------------------------------
struct PrefillParams {
    CUtensorMap tmap_q;   // 3-D (d, Sq, B*Hq), box (64, 128, 1), 128B swizzle
    CUtensorMap tmap_k;   // 3-D (d, Skv, B*Hkv), box (64, 128, 1), 128B swizzle
    CUtensorMap tmap_v;   // same as K
    CUtensorMap tmap_o;   // 3-D (d, Sq, B*Hq), box (64, 128, 1), 128B swizzle (TMA stores of
                          // the persistent kernel)
    __nv_bfloat16* o;     // [B, Hq, Sq, d]
    float* lse;           // [B, Hq, Sq] or null
    int B, Hq, Hkv, Sq, Skv;
    int G;                // Hq / Hkv
    int n_qblk;           // ceil(Sq / 128)
    int n_pairs;          // work items: pairs of Q tiles, or single Q tiles with kv_split
    int kv_split;         // 1: a CTA splits each of its Q tiles' KV range over its two slots
    int tail0;            // KV split: -1, or the first pair whose two Q tiles the CTAs take
                          // (the last, partly filled wave of a pair-mode call)
    int causal;
    int diag;             // causal: key j is visible to query row i iff j <= i + diag
                          // (bottom-right alignment: diag = Skv - Sq)
    int row0;             // first query row the Q tiles cover (tile q0 = row0 + 128 * block);
                          // rows [0, row0) see no key and are written by the row-fill kernel
    int o_align32;        // o is 32-byte aligned: the epilogue may use 32-byte stores
    float scale_log2;     // scale * log2(e)
    int* err;             // device error word of bounded waits
    int* tiles_issued;    // null, or a device counter the MMA issuer adds its S = Q K^T
                          // tile products to (one atomic per CTA at its end)
};
cudaError_t launch_attn_fwd_bf16(const PrefillParams& p, int d, cudaStream_t stream);
// The Q tiles of pairs [p.tail0, p.tail0 + p.n_pairs / 2) in KV-split mode, launched as a
// programmatic dependent of the pair-mode launch just before it (p.n_pairs = tiles).
cudaError_t launch_attn_fwd_bf16_tail(const PrefillParams& p, int d, cudaStream_t stream);

// ---- bf16 persistent KV-split prefill (prefill_persist.cu) ------------------------------
// p.n_pairs single Q tiles (all of the call's), dealt heaviest first in snake order to
// min(p.n_pairs, nsm) persistent CTAs; each tile's KV range is split over a CTA's two slots.
cudaError_t launch_attn_fwd_bf16_persistent(const PrefillParams& p, int d, int nsm,
                                            cudaStream_t stream);

// ---- log-sum-exp merge and empty-row fill (attn_merge.cu) -------------------------------
// (O_out, L_out) = merge((O_a, L_a), (O_b, L_b)) row by row; each O is rows x d, fp32 or bf16
// as flagged; lo may be null; oo may alias oa or ob, lo may alias la or lb.  d in {64, 128}.
// err: the device error word (debug builds record failed store bounds checks there).
cudaError_t launch_attn_merge(const void* oa, const float* la, bool a_f32, const void* ob,
                              const float* lb, bool b_f32, void* oo, float* lo, bool out_f32,
                              long long rows, int d, int nsm, int* err, cudaStream_t st);
// Rows [0, row0) of each of the bh (batch, head) blocks of Sq rows: O = 0, LSE = -inf.
cudaError_t launch_fill_empty_rows(__nv_bfloat16* o, float* lse, long long bh, int Sq, int row0,
                                   int d, int nsm, int* err, cudaStream_t st);

// ---- bf16 split-KV decode path (decode_splitkv.cu) --------------------------------------
struct DecodeParams {
    CUtensorMap tmap_k;   // 3-D (d, Lmax, B*Hkv), box (64, 64, 1), 128B swizzle
    CUtensorMap tmap_v;
    CUtensorMap tmap_q;   // 2-D (d, B*Hq), box (64, 8), 128B swizzle
    const int* kv_lens;   // [B] device
    __nv_bfloat16* o;     // [B, Hq, d]
    float* lse;           // [B, Hq] or null
    int* counter;         // work queue counter (zeroed before the split kernel)
    int* group_cnt;       // [B, Hkv, n_hg] finished partials per group (single-launch mode and
                          // the counted combine)
    float* ws_lse;        // [B, Hq, Tq, n_parts] log2-domain partial lse
    float* ws_o;          // [B, Hq, Tq, n_parts, d] normalised partial outputs
    int B, Hq, Hkv, Lmax, G;
    int Tq;               // new query tokens per sequence (1: single-token decode)
    int R;                // query rows per KV head: G * Tq (head-major, token-minor)
    int n_hc;             // row chunks of <= 8 rows per KV head: ceil(R / 8)
    int nci;              // row chunks per work item: 1, 2 or 4
    int n_hg;             // chunk groups per KV head: ceil(n_hc / nci)
    int n_slots;          // split slots per sequence
    int pieces;           // work items per split (contiguous pieces, each its own partial)
    int n_parts;          // partial slots per row: n_slots * pieces (split s, piece c: s * pieces + c)
    int fixed_splits;     // > 0 fixed count, 0 automatic
    int auto_floor;       // automatic mode: split count that fills the GPU (see splits_for)
    int combine_lanes;    // combine: lanes per (row, 4 columns), a power of two >= n_parts / 8
    int n_items;          // n_slots * pieces * B * Hkv * n_hg
    int fused;            // 1: single launch, the group's last split merges (single token)
    int counted;          // 1: each partial is counted into group_cnt, and the combine waits
                          // for its rows' groups only (R <= 8, not fused)
    float scale_log2;
    int* err;             // device error word of bounded waits
};
// Split-count rule of the automatic mode: one split per kAutoChunk keys, raised for calls
// with few (sequence, KV head) groups to as many splits as still fit one wave of work items
// (one per SM of the device; the host passes the resulting count as auto_floor), but never
// to fewer than kAutoMinKeys keys per split.
constexpr int kAutoChunk = 4096;
constexpr int kAutoMinKeys = 256;
constexpr int kMaxSplits = 256;
constexpr int kSplitAlign = 64;

size_t decode_counter_bytes(int B, int Hkv, int n_hg);
// B_rows: B * Tq; kv_groups: B * Hkv; n_parts: partial slots per row
size_t decode_workspace_bytes(int B_rows, int Hq, int kv_groups, int n_hg, int d, int n_parts);
int decode_slots(int Lmax, int num_splits, int auto_floor);
cudaError_t launch_decode_splitkv(const DecodeParams& p, int d, int num_sms,
                                  cudaStream_t stream);
// The log-sum-exp combine of the partials in the workspace, launched dependent on the
// kernel before it on `stream`.
cudaError_t launch_decode_combine(const DecodeParams& p, int d, cudaStream_t stream);

// ---- bf16 tcgen05 multi-token decode (decode_tcgen05.cu) ----------------------------------
// Work items (b, KV head, split, 128-row tile of the R = G * Tq rows); partials go to the
// same workspace layout as the split kernel's and are folded by launch_decode_combine.
struct DecodeTcParams {
    CUtensorMap tmap_q;   // 3-D (d, B*Hq*Tq, 1), box (64, q_rows, 1), 128B swizzle
    CUtensorMap tmap_k;   // 3-D (d, Lmax, B*Hkv), box (64, 128, 1), 128B swizzle
    CUtensorMap tmap_v;
    const int* kv_lens;
    __nv_bfloat16* o;     // [B, Hq, Tq, d]
    float* lse;           // [B, Hq, Tq] or null
    float* ws_lse;        // [B, Hq, Tq, n_parts] log2-domain partial lse
    float* ws_o;          // [B, Hq, Tq, n_parts, d]
    int B, Hq, Hkv, Lmax, Tq;
    int R;                // query rows per KV head: G * Tq
    int q_rows;           // Q rows loaded per item: R rounded up to 8, at most 128
    int n_rt;             // 128-row tiles per KV head: ceil(R / 128)
    int n_slots, fixed_splits;
    int pieces, n_parts;  // as in DecodeParams
    int auto_floor;       // automatic mode: split count that fills the GPU (see splits_for)
    int n_items;          // n_slots * pieces * B * Hkv * n_rt
    int* counter;         // work queue counter (zeroed before the kernel)
    int* group_cnt;       // [B, Hkv, n_rt] finished partials per (sequence, KV head, row tile)
    int counted;          // 1: each item's partial is counted into group_cnt, and the combine
                          // merges a row tile's rows once their count is complete
    float scale_log2;
    int* err;
};
cudaError_t launch_decode_multitoken_tc(const DecodeTcParams& p, int d, int nsm,
                                        cudaStream_t stream);

}  // namespace gbattn
