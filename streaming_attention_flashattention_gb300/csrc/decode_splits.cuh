// decode_splits.cuh -- how a sequence's keys are cut into splits for split-KV decode.
//
// "ADR-0060: AHBM GQA Fused Attention Kernel (Llama3-70B)", section 2.1: each split is one
// contiguous block of the cache.  n splits of C keys, C = ceil(len / n) rounded up to
// kSplitAlign; automatic mode takes one split per kAutoChunk keys.
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

__device__ __forceinline__ int splits_for(int len, int fixed_splits) {
    if (fixed_splits > 0) return fixed_splits;
    int n = (len + kAutoChunk - 1) / kAutoChunk;
    return max(1, min(kMaxSplits, n));
}


}  // namespace gbattn
