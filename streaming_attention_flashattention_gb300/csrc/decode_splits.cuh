// decode_splits.cuh -- how a sequence's keys are cut into splits for split-KV decode.
//
// "ADR-0060: AHBM GQA Fused Attention Kernel (Llama3-70B)", section 2.1: each split is one
// contiguous block of the cache.  n splits of C keys, C = ceil(len / n) rounded up to
// kSplitAlign.  The automatic mode takes one split per kAutoChunk keys, or more when the
// call has few (sequence, KV head) groups (splits_for).
#pragma once
#include "kernels.h"

namespace gbattn {

// Split bounds of the reading "contiguous blocks": n splits of C keys,
// C = ceil(len / n) rounded up to kSplitAlign.
__device__ __forceinline__ void split_range(int len, int n, int s, int& t0, int& t1) {
    int c = (len + n - 1) / n;
    c = ((c + kSplitAlign - 1) / kSplitAlign) * kSplitAlign;
    if (c == 0) c = kSplitAlign;
    const long long a = (long long)s * c;
    t0 = (int)min((long long)len, a);
    t1 = (int)min((long long)len, a + c);
}

// Number of non-empty splits: the first ceil(len / C) of them.
__device__ __forceinline__ int nonempty_splits(int len, int n) {
    if (len <= 0) return 0;
    int c = (len + n - 1) / n;
    c = ((c + kSplitAlign - 1) / kSplitAlign) * kSplitAlign;
    return (len + c - 1) / c;
}

// Piece pc of P of the split [t0, t1): contiguous sub-ranges of ceil((t1 - t0) / P) keys
// rounded up to kSplitAlign (trailing pieces may be empty).  A split cut into pieces is
// still one contiguous block of keys; its pieces' partial states fold into the same
// log-sum-exp merge as the splits themselves.
__device__ __forceinline__ void piece_range(int t0, int t1, int P, int pc, int& a, int& b) {
    int c = (t1 - t0 + P - 1) / P;
    c = ((c + kSplitAlign - 1) / kSplitAlign) * kSplitAlign;
    a = min(t1, t0 + pc * c);
    b = min(t1, t0 + (pc + 1) * c);
}

// Splits of a sequence of len keys.  Automatic mode: one per kAutoChunk keys, raised to
// auto_floor (the count that gives the call about one work item per SM, chosen on the host)
// as long as each split keeps kAutoMinKeys keys.  Non-decreasing in len, so the host sizes
// the workspace with len = Lmax.
__host__ __device__ __forceinline__ int splits_for(int len, int fixed_splits, int auto_floor) {
    if (fixed_splits > 0) return fixed_splits;
    const int by_len = (len + kAutoChunk - 1) / kAutoChunk;
    const int by_keys = (len + kAutoMinKeys - 1) / kAutoMinKeys;
    const int by_fill = auto_floor < by_keys ? auto_floor : by_keys;
    const int n = by_len > by_fill ? by_len : by_fill;
    return n < 1 ? 1 : (n > kMaxSplits ? kMaxSplits : n);
}


// Guided pieces (the layout the split kernel uses): piece pc of P starts at the fraction
// 1 - 4^-pc of the split (3/4 + 1/4 for two pieces), cut points rounded up to kSplitAlign,
// and the work queue hands out piece 0 of every split before any piece 1.  Large items go
// first and small ones last, so the persistent CTAs run out of work within a small item of
// one another instead of a whole one.  Still contiguous blocks, folded by the same merge.
#ifndef GBATTN_GUIDED_PIECES
#define GBATTN_GUIDED_PIECES 1
#endif
__device__ __forceinline__ void piece_range_guided(int t0, int t1, int P, int pc, int& a,
                                                   int& b) {
    const int n = t1 - t0;
    auto cut = [&](int k) -> int {                 // keys of the split before piece k
        if (k <= 0) return 0;
        if (k >= P) return n;
        long long c = (long long)n - ((long long)n >> (2 * k));
        c = ((c + kSplitAlign - 1) / kSplitAlign) * kSplitAlign;
        return (int)min((long long)n, c);
    };
    a = t0 + cut(pc);
    b = t0 + cut(pc + 1);
}

}  // namespace gbattn
