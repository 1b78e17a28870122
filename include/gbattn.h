/*
 * gbattn.h -- C ABI of the GB300 streaming-attention library (libgbattn.so).
 *
 * The library computes the fused streaming attention forward
 *     O = softmax(scale * Q K^T + mask) V
 * without materialising the score or probability matrix: Q is tiled, K/V tiles stream
 * through on-chip memory and an online-softmax running state (m, l) rescales the output
 * accumulator.
 *   Definition: "AttentionRegion Transformation - Deriving FlashAttention via
 *   Memory-Centric Compilation in AICF", section 3 (MatMul(Q, K^T) -> Mask -> Softmax ->
 *   MatMul(P, V)), section 6 (streaming region, online update of m and l), section 8
 *   (kernel lowering: Q-tile outer loop, KV-tile inner loop, score never materialised).
 *   Per-tile operation sequence, GQA stacking, split-KV decode and the log-sum-exp merge:
 *   "ADR-0060: AHBM GQA Fused Attention Kernel (Llama3-70B)", sections 3, 4, 5.2, 5.4.
 *   I/O contract (post-RoPE Q and K/V cache in, O out, no S or P out, KV cache read only):
 *   the same ADR, section 0.5.
 *
 * Conventions shared by every entry point
 *  - Pointers named q, k, v, kcache, vcache, o, lse, kv_lens, workspace are DEVICE
 *    pointers (CUDA global memory of the current device).  The caller allocates and owns
 *    every buffer; the library allocates no device memory per call.
 *  - Layouts are contiguous row-major "BHSD": Q and O [B, Hq, Sq, d], K and V
 *    [B, Hkv, Skv, d], LSE [B, Hq, Sq].  Grouped-query attention: query head h reads
 *    KV head h / (Hq / Hkv).
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy default
 *    stream).  Errors that the host can detect are returned before anything is launched.
 *  - LSE is the natural log of sum_j exp(scale * q . k_j) over the visible keys, fp32.
 *  - A row that sees no key (a decode sequence of length 0) gets O = 0, LSE = -inf.
 *  - Causal masking is bottom-right aligned: query i sits at key position i + Skv - Sq and
 *    sees keys j <= i + Skv - Sq (attn_fwd_positions takes the positions explicitly).
 *  - Numerics: bf16 inputs, fp32 scores / running state / accumulators, P rounded to
 *    bf16 for the P.V product, O stored in the input dtype.
 *  - Each compute call is an NVTX range named after it (attn_fwd, attn_fwd_counted,
 *    attn_fwd_positions, attn_merge, attn_fwd_host, attn_prefill_kvcache, attn_decode,
 *    attn_decode_host), visible to a profiler and free without one.
 */
#ifndef GBATTN_H
#define GBATTN_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element type of Q, K, V and O. */
typedef enum {
    GBATTN_BF16 = 0, /* bf16 storage; tcgen05 tensor-core path (d = 64 or 128) */
    GBATTN_FP32 = 1  /* fp32 storage; exact fp32 CUDA-core path (d = 64 or 128) */
} gbattn_dtype_t;

/* Status codes (0 = success, negative = error). */
enum {
    GBATTN_OK = 0,
    GBATTN_ERR_INVALID_ARG = -1,    /* null pointer, non-positive size, Hq % Hkv != 0, ... */
    GBATTN_ERR_UNSUPPORTED = -2,    /* d not in {64,128}, dtype/path combination, causal with Sq > Skv */
    GBATTN_ERR_MISALIGNED = -3,     /* a pointer is not 16-byte aligned */
    GBATTN_ERR_CUDA = -4,           /* a CUDA runtime/driver call or launch failed */
    GBATTN_ERR_TIMEOUT = -5,        /* a device-side bounded wait expired (see attn_last_device_error) */
    GBATTN_ERR_WORKSPACE = -6,      /* workspace null or smaller than attn_decode_workspace_size() */
    GBATTN_ERR_TOO_LARGE = -7       /* a size exceeds what the kernels index (e.g. > 2^31 rows) */
};

/*
 * attn_fwd -- prefill / general attention forward.
 *
 *   q   [B, Hq, Sq, d]  device, dtype        post-RoPE queries
 *   k   [B, Hkv, Skv, d] device, dtype       post-RoPE keys
 *   v   [B, Hkv, Skv, d] device, dtype       values
 *   o   [B, Hq, Sq, d]  device, dtype        output (written)
 *   lse [B, Hq, Sq]     device, fp32         log-sum-exp per row (written); may be NULL
 *   scale                                    softmax scale (typically 1/sqrt(d))
 *   causal                                   0 = full attention, 1 = bottom-right causal
 *   dtype                                    GBATTN_BF16 or GBATTN_FP32
 *   stream                                   cudaStream_t
 *
 * Requirements: B, Hq, Hkv, Sq, Skv >= 1; Hq % Hkv == 0; d in {64, 128};
 * causal requires Sq <= Skv; all pointers 16-byte aligned.
 * Tile classes follow "ADR-0060" section 5.4: KV tiles entirely in a query tile's future
 * are skipped, tiles crossing the diagonal are masked, the rest run unmasked.
 * bf16 work items are pairs of Q tiles (one CTA each), or -- when pairs would not fill the
 * GPU once -- single Q tiles with their KV range split over a CTA's two slots, run by
 * at most one persistent CTA per SM that takes its tiles heaviest first.  When the pairs
 * weigh nearly the same (non-causal calls, or a chunk at the end of a long context) and
 * their last wave is at most half full, that wave's Q tiles run split in a second launch,
 * a programmatic dependent of the first that ends after it.  Stream order and CUDA graph
 * capture see one call either way.
 * Returns GBATTN_OK or a negative status; nothing is launched on error.
 */
int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
             int Hkv, int Sq, int Skv, int d, float scale, int causal, int dtype,
             void* stream);

/*
 * attn_fwd_counted -- attn_fwd (bf16 only) that also reports the work it issued, so that
 * the causal tile skipping can be checked: "ADR-0060" section 11 asks that a causal
 * prefill skip every KV tile wholly in a query tile's future, so that the number of
 * S = Q K^T tile products equals the lower-triangular count, not the full grid.
 *
 *   s_tiles  DEVICE int, 4-byte aligned, owned by the caller: the kernels ADD to it the
 *            number of 128-query x 128-key S tile products they issued (one atomic per
 *            CTA); the caller zeroes it first.  The expected value for a call is
 *            sum over 128-row Q tiles of ceil(visible keys of the tile's last row / 128),
 *            where a row i sees min(Skv, i + Skv - Sq + 1) keys (causal) or Skv keys.
 *
 * Same arguments, numerics, output and status codes as attn_fwd with dtype GBATTN_BF16,
 * plus GBATTN_ERR_INVALID_ARG for a NULL s_tiles.  The counter adds one atomic per CTA;
 * attn_fwd passes no counter and skips it.
 */
int attn_fwd_counted(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                     int Hq, int Hkv, int Sq, int Skv, int d, float scale, int causal,
                     int* s_tiles, void* stream);

/*
 * attn_fwd_host_workspace_size -- device bytes attn_fwd_host needs for these sizes on the
 * current device (up to three staging buffer sets); 0 for invalid sizes.
 */
size_t attn_fwd_host_workspace_size(int B, int Hq, int Hkv, int Sq, int Skv, int d, int dtype);

/*
 * attn_fwd_host -- attn_fwd on HOST buffers: the same operation and kernel, with the inputs
 * copied to the device and the outputs back as part of the call.  Not in the pages (their
 * accelerator has no host link); a library-level addition for callers whose tensors live
 * in host memory.
 *
 *   q, k, v, o, lse      HOST pointers, layouts as for attn_fwd (lse may be NULL); page-locked
 *                        memory gives asynchronous copies, pageable memory works but the
 *                        copies then wait on the host
 *   workspace, ws_bytes  DEVICE scratch of at least attn_fwd_host_workspace_size(...) bytes,
 *                        owned by the caller
 *   stream               the call is ordered after the earlier work on `stream`, and work
 *                        queued on `stream` afterwards runs after its last copy has landed
 *                        in host memory (synchronise on it before reading o / lse)
 *
 * The (batch, KV head) groups are cut into chunks, each the smallest that keeps the
 * kernel's pair mode (a pair of Q tiles per SM), and staged through up to three device
 * buffer sets on internal copy streams: chunks i+1 and i+2 are copied in and chunk i-1
 * copied out while chunk i computes.  Calls on one
 * device are serialised on the host; calls sharing a workspace must be ordered on one
 * stream.  Requirements and status codes as attn_fwd, plus GBATTN_ERR_WORKSPACE.
 */
int attn_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                  int Hq, int Hkv, int Sq, int Skv, int d, float scale, int causal, int dtype,
                  void* workspace, size_t ws_bytes, void* stream);

/*
 * attn_prefill_kvcache -- chunked prefill against a KV cache: a chunk of Sq new queries
 * attends to the first Skv rows of a cache of capacity Lmax (the chunk's own keys are the
 * last Sq of those rows; "ADR-0060" section 0.5.2: T_q = the chunk width for a
 * prefill/chunk launch, and section 5.4 for the tile classes).
 *
 *   q       [B, Hq, Sq, d]      device, bf16    the chunk's post-RoPE queries
 *   kcache  [B, Hkv, Lmax, d]   device, bf16    key cache; rows [0, Skv) are used, rows
 *                                               [Skv, Lmax) are never read
 *   vcache  [B, Hkv, Lmax, d]   device, bf16    value cache, same rows
 *   o       [B, Hq, Sq, d]      device, bf16    output (written)
 *   lse     [B, Hq, Sq]         device, fp32    log-sum-exp (written); may be NULL
 *
 * Same kernel and numerics as attn_fwd (bf16); causal is bottom-right: query i of the chunk
 * sits at position Skv - Sq + i.  Requirements: 1 <= Skv <= Lmax, Hq % Hkv == 0,
 * d in {64, 128}, causal requires Sq <= Skv, pointers 16-byte aligned.
 */
int attn_prefill_kvcache(const void* q, const void* kcache, const void* vcache, void* o,
                         float* lse, int B, int Hq, int Hkv, int Sq, int Skv, int Lmax, int d,
                         float scale, int causal, void* stream);

/*
 * attn_fwd_positions -- causal attention with explicit positions: query i of the call sits
 * at position q_pos0 + i and key j at position k_pos0 + j, and a query sees exactly the keys
 * whose position is not after its own.  "ADR-0060" section 5.4 states the tile classes on
 * such absolute positions (query block [qs, qe) against KV tile [ks, ke)), and section 5.5
 * folds the KV slice of each ring step of a sequence-parallel prefill this way.  attn_fwd's
 * bottom-right causal call is the case q_pos0 = Skv - Sq, k_pos0 = 0.
 *
 *   q, k, v, o, lse   as for attn_fwd, bf16 only (lse may be NULL)
 *   q_pos0, k_pos0    positions of query row 0 and key row 0, each within [-2^40, 2^40];
 *                     only their difference matters
 *
 * A query that sees no key (its position is before k_pos0) gets O = 0 and LSE = -inf, the
 * neutral element of attn_merge.  Those rows (a prefix of the call's rows) are written by a
 * fill kernel; the other rows run on attn_fwd's kernels and numerics.  Requirements and
 * status codes as attn_fwd with dtype GBATTN_BF16, except that Sq > Skv is allowed.
 */
int attn_fwd_positions(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                       int Hq, int Hkv, int Sq, int Skv, int d, float scale, long long q_pos0,
                       long long k_pos0, void* stream);

/*
 * attn_merge -- log-sum-exp merge of two partial attention results over disjoint key sets,
 * row by row ("ADR-0060" section 4: the merge is associative and commutative, so partials
 * can be folded in any order, by a chain or by a tree).  With L the rows' log-sum-exp:
 *     M = max(L_a, L_b),  w_x = e^(L_x - M),
 *     O = (w_a O_a + w_b O_b) / (w_a + w_b),  L = M + ln(w_a + w_b);
 * a partial with L = -inf (no key) contributes nothing, whatever its O holds; if both are
 * -inf the row is O = 0, L = -inf.
 *
 *   o_a, lse_a, dtype_a         first partial: rows x d elements (GBATTN_BF16 or GBATTN_FP32)
 *                               and rows fp32 LSE values, device
 *   o_b, lse_b, dtype_b         second partial, likewise
 *   o_out, lse_out, dtype_out   the merged result (lse_out may be NULL); o_out is o_a, o_b or
 *                               a buffer disjoint from both, and lse_out likewise, so that a
 *                               running accumulator can be merged in place
 *   rows, d                     rows >= 0 (0 launches nothing, and the pointers may then
 *                               be NULL), d in {64, 128}
 *
 * O pointers 16-byte aligned, LSE pointers 4-byte aligned.  An fp32 accumulator keeps a
 * chain of merges at fp32 precision; a bf16 result rounds once.  Returns GBATTN_OK or a
 * negative status (nothing launched on error).
 */
int attn_merge(const void* o_a, const float* lse_a, int dtype_a, const void* o_b,
               const float* lse_b, int dtype_b, void* o_out, float* lse_out, int dtype_out,
               long long rows, int d, void* stream);

/*
 * attn_decode_workspace_size -- bytes of device workspace attn_decode_splitkv needs on the
 * CURRENT device.  Holds the per-split partial results (lse_s and O_s / l_s, fp32), a work
 * counter and one finished-split counter per (sequence, KV head); the counters are cleared
 * on the call's stream at the start of every call, so the caller need not initialise
 * anything.  num_splits > 0: fixed split count; 0: automatic: one split per 4096 keys of a
 * sequence, raised for calls with few (sequence, KV head) groups to the most splits that
 * still fit one wave of work items -- one per SM of the device, so the size depends on the
 * device's SM count (queried here) -- but never below 256 keys per split.  A workspace
 * sized on one device serves calls on devices with the same SM count.
 * Returns 0 for invalid arguments, or when no CUDA device can be queried (use
 * attn_decode_workspace_bytes to size for a given SM count without a device).
 */
size_t attn_decode_workspace_size(int B, int Hq, int Hkv, int Lmax, int d, int num_splits);

/*
 * attn_decode_workspace_bytes -- the workspace of a decode call with Tq new tokens per
 * sequence (Tq = 1: attn_decode_splitkv) on a GPU with num_sms SMs.  Host only: no device
 * access.  attn_decode_workspace_size and attn_decode_multitoken_workspace_size are this
 * function with the current device's SM count.  Returns 0 for invalid arguments.
 */
size_t attn_decode_workspace_bytes(int B, int Hq, int Hkv, int Tq, int Lmax, int d,
                                   int num_splits, int num_sms);

/*
 * attn_decode_splitkv -- single-token (T_q = 1) decode against a KV cache, split-KV with a
 * log-sum-exp merge ("ADR-0060" section 4 merge and section 5.2/5.3 decode).
 *
 *   q       [B, Hq, 1, d]       device, bf16    the step's post-RoPE queries
 *   kcache  [B, Hkv, Lmax, d]   device, bf16    key cache (read only; rows >= kv_lens[b] never read)
 *   vcache  [B, Hkv, Lmax, d]   device, bf16    value cache (read only)
 *   kv_lens [B]                 device, int32   valid keys per sequence, 0 <= kv_lens[b] <= Lmax
 *   o       [B, Hq, 1, d]       device, bf16    output (written)
 *   lse     [B, Hq]             device, fp32    log-sum-exp (written); may be NULL
 *   num_splits                                  > 0 fixed splits per sequence (<= 256),
 *                                               0 = automatic per sequence length and
 *                                               call size (attn_decode_workspace_size)
 *   workspace, ws_bytes                         device scratch of at least
 *                                               attn_decode_workspace_size(...) bytes,
 *                                               owned by the caller; calls that share a
 *                                               workspace must be ordered on one stream
 *
 * Sequence b's keys [0, kv_lens[b]) are cut into contiguous splits of C keys,
 * C = ceil(len / n) rounded up to 64 ("ADR-0060" section 2.1: contiguous blocks); each
 * split streams its chunk once for all G = Hq / Hkv query heads of a KV head (the heads
 * are stacked into one MMA operand, "ADR-0060" section 5.2), and the partial (lse_s, O_s)
 * of the splits are merged ("ADR-0060" section 4; a sequence with one split is written
 * directly).  When the (split, KV head) work items of the warp-level kernel would leave the
 * GPU's last wave mostly idle, each split is processed as up to 4 contiguous pieces (at
 * least 512 keys per piece on average; piece k starts at the fraction 1 - 4^-k of the split,
 * and every split's first piece is handed out before the smaller ones), each with a partial
 * of its own in the same merge: the result is the same up to fp32 rounding, and
 * attn_decode_plan reports the piece count.  When every work item fits in one wave of the GPU, or the call has at most
 * 16 (sequence, KV head) groups with splits of at least 1024 keys (Lmax / splits), the
 * merge is done by the CTA that finishes a group's last split (one launch, "ADR-0060"
 * section 4.3); otherwise a combine kernel, launched dependent on the split kernel, merges.  With G >= 16 query
 * heads per KV head the heads form the M = 128 operand of a tcgen05 kernel instead of
 * the N dimension of warp-level MMAs.  kv_lens values are
 * read on the device; values outside [0, Lmax] are clamped into it.
 * Requirements: d = 128 or 64, G <= 8 per launch group (larger G runs several groups),
 * all pointers 16-byte aligned.  Returns GBATTN_OK or a negative status.
 */
int attn_decode_splitkv(const void* q, const void* kcache, const void* vcache,
                        const int* kv_lens, void* o, float* lse, int B, int Hq, int Hkv,
                        int Lmax, int d, float scale, int num_splits, void* workspace,
                        size_t ws_bytes, void* stream);

/*
 * attn_decode_multitoken -- decode of Tq >= 1 new tokens per sequence at once (for
 * example speculative decoding), split-KV with the same log-sum-exp merge.  The G * Tq
 * query rows of a KV head are stacked into the MMA operand ("ADR-0060" section 0.5:
 * the group's Q [G, T_q, d] folds to [G * T_q, d]).  Up to 8 rows run on warp-level MMAs;
 * 16 or more, or 9 to 15 with splits of at least 1024 keys (Lmax / splits), run as the
 * M = 128 operand of tcgen05 MMAs, each K/V tile read once per 128 rows; other 9 to 15 row
 * calls run 8 rows at a time on warp-level MMAs.
 *
 *   q       [B, Hq, Tq, d]      device, bf16    the new tokens' post-RoPE queries
 *   kcache  [B, Hkv, Lmax, d]   device, bf16    key cache; the new tokens' keys are
 *                                               already its rows [len - Tq, len)
 *   vcache  [B, Hkv, Lmax, d]   device, bf16    value cache, same rows
 *   kv_lens [B]                 device, int32   len: cached keys per sequence, new ones included
 *   o       [B, Hq, Tq, d]      device, bf16    output (written)
 *   lse     [B, Hq, Tq]         device, fp32    log-sum-exp (written); may be NULL
 *   workspace, ws_bytes                         >= attn_decode_multitoken_workspace_size(...)
 *                                               (sized for the current device's SM count)
 *
 * New token t (0-based) sees keys j <= len - Tq + t (causal among the new tokens; every
 * older key).  A row that sees no key (len < Tq) gets O = 0, LSE = -inf.  Requirements
 * as attn_decode_splitkv, plus 1 <= Tq <= 64.  Tq = 1 is exactly attn_decode_splitkv.
 */
size_t attn_decode_multitoken_workspace_size(int B, int Hq, int Hkv, int Tq, int Lmax, int d,
                                             int num_splits);
int attn_decode_multitoken(const void* q, const void* kcache, const void* vcache,
                           const int* kv_lens, void* o, float* lse, int B, int Hq, int Hkv,
                           int Tq, int Lmax, int d, float scale, int num_splits,
                           void* workspace, size_t ws_bytes, void* stream);

/*
 * attn_decode_host_workspace_size -- device bytes attn_decode_host needs for these sizes on
 * the current device (staging buffers and a decode workspace); 0 for invalid sizes.
 */
size_t attn_decode_host_workspace_size(int B, int Hq, int Hkv, int Lmax, int d, int num_splits);

/*
 * attn_decode_host -- attn_decode_splitkv on HOST buffers: the same operation and kernels,
 * with the inputs copied to the device and the outputs back as part of the call.  Not in
 * the pages (their accelerator has no host link); the decode counterpart of attn_fwd_host.
 *
 *   q, kcache, vcache, o, lse   HOST pointers, layouts as for attn_decode_splitkv (lse may
 *                               be NULL); page-locked memory gives asynchronous copies
 *   kv_lens                     HOST int32 [B], each within [0, Lmax] (checked on the host:
 *                               GBATTN_ERR_INVALID_ARG otherwise, nothing launched)
 *   num_splits                  as for attn_decode_splitkv, applied to each chunk
 *   workspace, ws_bytes         DEVICE scratch of at least attn_decode_host_workspace_size(...)
 *                               bytes, owned by the caller
 *   stream                      ordered after the earlier work on `stream`; work queued on
 *                               `stream` afterwards runs after the last copy has landed
 *
 * The sequences are cut into up to 4 chunks of consecutive sequences, staged through two
 * device buffer sets on internal copy streams: chunk i+1 is copied in and chunk i-1 copied
 * out while chunk i decodes.  Calls on one device are serialised on the host.  Status codes
 * as attn_decode_splitkv.
 */
int attn_decode_host(const void* q, const void* kcache, const void* vcache, const int* kv_lens,
                     void* o, float* lse, int B, int Hq, int Hkv, int Lmax, int d, float scale,
                     int num_splits, void* workspace, size_t ws_bytes, void* stream);

/*
 * attn_decode_splitkv_noalloc -- attn_decode_splitkv for callers that cannot allocate
 * device memory, so cannot pass a workspace: a plugin inside a framework that owns all
 * device allocations and offers no scratch, or a serving loop that must not allocate
 * once running because an allocation can synchronise the device.  The pages describe
 * no counterpart; this is a library-level addition.
 *
 * Same arguments, layouts and results as attn_decode_splitkv, without the workspace.
 * The scratch is a fixed 8 MiB array inside the library (reserved on every GPU that
 * loads the library, until the process exits).  The call allocates nothing itself.
 *  - Sizes whose attn_decode_workspace_size(...) exceeds 8 MiB (8388608 bytes) are
 *    rejected with GBATTN_ERR_WORKSPACE before anything is launched.
 *  - The first call on a device looks up the array's device address for that device;
 *    make that first call before any stream capture starts.  If that lookup fails (for
 *    example because the first call was made while a stream was being captured) the call
 *    returns GBATTN_ERR_CUDA, launches nothing and clears the CUDA error it caused; a
 *    later call outside capture repeats the lookup.
 *  - Every call shares the one array: calls whose GPU work may overlap (different
 *    streams, or unordered host threads) race and give wrong results.  The counters
 *    that must start at zero are cleared on `stream` by each call.
 */
int attn_decode_splitkv_noalloc(const void* q, const void* kcache, const void* vcache,
                                const int* kv_lens, void* o, float* lse, int B, int Hq,
                                int Hkv, int Lmax, int d, float scale, int num_splits,
                                void* stream);

/*
 * attn_decode_plan -- what attn_decode_multitoken / attn_decode_splitkv (Tq = 1) decide for
 * these sizes on a GPU with num_sms SMs.  Host only: no device access, for tests and
 * capacity planning.  plan (host, 7 ints) receives:
 *   plan[0]  splits per sequence the workspace holds (the automatic count for Lmax when
 *            num_splits = 0)
 *   plan[1]  kernel: 0 warp-level MMAs (8 query rows at a time), 1 tcgen05 (M = 128 rows)
 *   plan[2]  merge: 0 a dependent combine kernel that waits for the whole split grid, 1 the
 *            CTA that finishes a group's last split merges it (single launch), 2 a dependent
 *            combine kernel that merges each (sequence, KV head) group as soon as all of its
 *            partials are counted in
 *   plan[3]  work items of the kernel
 *   plan[4]  query rows per KV head, G * Tq
 *   plan[5]  combine lanes per (row, 4 columns)
 *   plan[6]  pieces per split (work items, and partials, per split)
 * Returns GBATTN_OK or the status the decode call would return for these sizes.
 */
int attn_decode_plan(int B, int Hq, int Hkv, int Tq, int Lmax, int d, int num_splits,
                     int num_sms, int* plan);

/*
 * attn_prefill_plan -- the work split attn_fwd (bf16) and attn_prefill_kvcache choose for
 * these sizes on a GPU with num_sms SMs.  Host only.  plan (host, 4 ints) receives:
 *   plan[0]  mode of the first launch: 0 pairs of Q tiles per CTA, 1 single Q tiles with
 *            their KV range split over a CTA's two slots, on persistent CTAs (at most one
 *            per SM) that take the tiles heaviest first
 *   plan[1]  CTAs of the first launch
 *   plan[2]  pairs whose Q tiles run KV-split in a second, dependent launch (0: none)
 *   plan[3]  Q tiles in all
 * Returns GBATTN_OK or a negative status for invalid sizes.
 */
int attn_prefill_plan(int B, int Hq, int Hkv, int Sq, int Skv, int causal, int num_sms,
                      int* plan);

/*
 * attn_last_device_error -- synchronise `stream`, then read and clear the device error
 * word that bounded waits inside the kernels set when they give up (they never trap).
 * Returns GBATTN_OK, GBATTN_ERR_TIMEOUT (the word was set) or GBATTN_ERR_CUDA.
 * If detail != NULL it receives the raw word (which wait gave up): 1 producer (free ring
 * slot), 2 consumer (filled slot), 3 MMA issuer, 4 softmax warps, 5 exit drain of
 * in-flight copies, 6 the self-test wait, 7 a decode row's merge waiting for its partials,
 * 8 a bounds check of a debug build (below) failed.
 *
 * Debug build: the library compiled with -DGBATTN_DEBUG_CHECKS (build.py: build(debug=True),
 * libgbattn_debug.so; same entry points) checks, in every kernel, the index of each plain
 * global store -- and of the decode merges' partial loads -- against the extent of its
 * buffer before the access.  A failed check records word 8 and skips that access; nothing
 * traps.  Release builds contain no checks.
 */
int attn_last_device_error(void* stream, int* detail);

/*
 * attn_selftest_bounded_wait -- exercise the failure path of the device-side waits without
 * hanging or faulting the GPU: launches a one-thread kernel on `stream` whose mbarrier
 * wait can never be satisfied; after about 2e6 cycles (~1 ms) the wait gives up, records
 * word 6 in the device error word and the kernel returns normally.  A following
 * attn_last_device_error() then reports GBATTN_ERR_TIMEOUT with detail 6 (and clears
 * the word); the context stays usable.  Returns GBATTN_OK if the kernel was launched.
 */
int attn_selftest_bounded_wait(void* stream);

/* Human-readable text for a status code (static storage, never NULL). */
const char* attn_status_string(int status);

/* Library ABI version (major * 100 + minor). */
int attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GBATTN_H */
