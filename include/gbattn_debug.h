/*
 * gbattn_debug.h -- a test hook of the debug build (libgbattn_debug.so, built with
 * -DGBATTN_DEBUG_CHECKS).  The release library does not export it.
 *
 * Every wait in the kernels is bounded: a wait that runs out records which wait it was in
 * the device error word, and the kernel's roles leave through their give-up exits (TMA
 * copies drained, tensor-core products drained, TMEM released) without trapping.  This hook
 * makes such a wait run out inside a real attention kernel, so that a test can check those
 * exits on the GPU: it leaves one K tile copy unissued, so the wait for it never completes.
 * Nothing faults: the copy is simply never started.
 */
#ifndef GBATTN_DEBUG_H
#define GBATTN_DEBUG_H

#ifdef __cplusplus
extern "C" {
#endif

/* kernels the hook can target */
#define GBATTN_DEBUG_PERSISTENT_PREFILL 0  /* persistent KV-split prefill (small attn_fwd calls) */
#define GBATTN_DEBUG_MULTITOKEN_DECODE 1   /* tcgen05 multi-token decode (16+ rows per KV head) */
#define GBATTN_DEBUG_PAIR_PREFILL 2        /* prefill on pairs of Q tiles (and its tail launch) */
#define GBATTN_DEBUG_SPLIT_DECODE 3        /* warp-level split decode (a stage: 64 keys of K, V) */

/*
 * attn_debug_skip_fill -- from the next launch of `kernel` on the current device, CTA 0 does
 * not issue its K tile copy number `fill` (0-based, counted over the CTA's copies; for the
 * split decode kernel a copy is a ring stage of K and V), until called again with fill = -1.
 * The launch then ends after the bounded wait for that tile has run out (about 2e9 cycles,
 * one second), and attn_last_device_error() reports
 * GBATTN_ERR_TIMEOUT with the code of the wait that gave up first (1 producer, 2 consumer,
 * 3 tensor-core issuer, 4 softmax, 7 a combine block).  The outputs of that call are
 * undefined; later calls are not affected once the hook is cleared.
 * Returns GBATTN_OK, GBATTN_ERR_INVALID_ARG (unknown kernel, fill < -1) or GBATTN_ERR_CUDA.
 */
int attn_debug_skip_fill(int kernel, int fill);

#ifdef __cplusplus
}
#endif

#endif /* GBATTN_DEBUG_H */
