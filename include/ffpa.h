/*
 * ffpa.h: C ABI of a GB300 (sm_103a) fused scaled-dot-product attention
 * library for large head dimensions (D = 64 .. 1024 in steps of 64; the
 * regime the pages study is D = 320 .. 1024, headline D = 512).
 *
 * What it computes (per batch b and query head h, kv head g = h / (Hq/Hkv)):
 *
 *   S   = scale * Q_h K_g^T + bias          scores, never materialised
 *   S_ij = -inf where causal and j > i      top-left causal mask
 *   P   = softmax(S)  (row-wise)
 *   O_h = P V_g,   lse_i = ln sum_j exp(S_ij)
 *
 * This is the "naive_math" definition written out in the attention-kernel-
 * profiler design notes (generate_docs.py, "naive_math"),
 * with the grouped-query mapping of its "gqa_4kv" variant (K/V expanded by
 * repeat_interleave) and the additive key-position bias of the FFPA Attention
 * Benchmark page ("Quick Start": compact [1,1,1,Nkv] bias, or [1,1,Nq,Nkv]).
 * The backward is the one the FFPA Attention Benchmark page describes for
 * SM100 ("More Benchmark"): a preprocess (Delta = rowsum(dO * O)) and then dV,
 * dK and dQ launches.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Tensors are described by ffpa_tensor_t: a data pointer, a dtype, four
 *    sizes and four strides counted in ELEMENTS.  Q/K/V/O/dO/dQ/dK/dV are
 *    [B, H, N, D] with the innermost stride equal to 1.
 *  - Device pointers only.  The caller owns every buffer; the library never
 *    allocates or frees caller memory.  Work is enqueued on `stream` and the
 *    call returns without synchronising (stream-ordered, asynchronous).
 *  - Validation happens on the host before anything is enqueued.  On any
 *    non-zero return from validation nothing was launched and no buffer was
 *    written.
 *  - Each call is independent; the library keeps no per-call state except a
 *    per-device status word that kernels set when a bounded wait times out
 *    (read and cleared by ffpa_check_status).  Calls are thread-safe.
 */
#ifndef FFPA_H_
#define FFPA_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream (layout-compatible with cudaStream_t); NULL = legacy default stream. */
typedef struct CUstream_st* ffpa_stream_t;

enum ffpa_dtype { FFPA_F16 = 0, FFPA_BF16 = 1, FFPA_F32 = 2 };

enum ffpa_status {
  FFPA_OK = 0,
  FFPA_ERR_INVALID_ARG = 1, /* null pointer, shape mismatch, Hq % Hkv != 0, N < 1, bad scale */
  FFPA_ERR_UNSUPPORTED = 2, /* D % 64 != 0 or D outside [64, 1024]; dtype not f16/bf16; bias not f32;
                               innermost stride != 1 */
  FFPA_ERR_ALIGNMENT = 3,   /* base pointer not 16-byte aligned or a row/head/batch stride not a
                               multiple of 8 elements (TMA needs 16-byte strides) */
  FFPA_ERR_CUDA = 4,        /* a CUDA runtime call or kernel launch failed */
  FFPA_ERR_TIMEOUT = 5,     /* a kernel's bounded wait expired (reported by ffpa_check_status) */
  FFPA_ERR_SCRATCH_LIMIT = 6 /* ffpa_fwd_decode_noalloc: the call needs more than the fixed scratch */
};

typedef struct ffpa_tensor {
  void* data;        /* device pointer */
  int32_t dtype;     /* enum ffpa_dtype */
  int32_t reserved;  /* must be 0 */
  int64_t shape[4];  /* [B, H, N, D] (lse: [B, H, N, 1]; bias: [B|1, H|1, Nq|1, Nkv]) */
  int64_t stride[4]; /* in elements */
} ffpa_tensor_t;

/*
 * ffpa_fwd: attention forward, O and the row logsumexp.
 *
 *   q    [B, Hq, Nq, D]   f16 or bf16
 *   k, v [B, Hkv, Nkv, D] same dtype as q; Hkv divides Hq (GQA when Hkv < Hq)
 *   bias nullable.  f32, shape [B|1, Hq|1, Nq|1, Nkv], added to the scaled
 *        scores; a size-1 dimension is broadcast (its stride is ignored).
 *   causal  0 or 1: query i sees keys j <= i (top-left, also when Nq != Nkv)
 *   scale   > 0 and finite; the usual value is 1/sqrt(D)
 *   out  [B, Hq, Nq, D]   same dtype as q, written
 *   lse  nullable.  f32 [B, Hq, Nq, 1], contiguous: written with
 *        ln sum_j exp(S_ij); -inf for a row whose scores are all -inf (whose
 *        O row is then 0).
 *
 * Nq <= 16 takes a split-KV decode path (CUDA-core dot products over slices
 * of the keys, then an lse-weighted merge).  Otherwise one fused tcgen05
 * kernel runs; when its CTA pairs would fill less than half of the GPU (short
 * query sets) the keys are split between pairs and the same merge follows.
 * The partials live in stream-ordered scratch on `stream` from a memory pool
 * the library keeps per device (its blocks stay reserved for later calls).
 * Returns FFPA_OK or an ffpa_status code (see above).
 */
int ffpa_fwd(const ffpa_tensor_t* q, const ffpa_tensor_t* k, const ffpa_tensor_t* v,
             const ffpa_tensor_t* bias, int causal, float scale, const ffpa_tensor_t* out,
             const ffpa_tensor_t* lse, ffpa_stream_t stream);

/*
 * ffpa_bwd: attention backward (FFPA Attention Benchmark page, "More
 * Benchmark": a preprocess, then the key-side gradients dK and dV, then dQ).
 * D <= 256 runs preprocess, dV, dK and dQ as four kernels; D = 320 .. 1024
 * runs preprocess, one fused dK/dV kernel and a dQ kernel.
 *
 *   q, k, v, bias, causal, scale   exactly as passed to ffpa_fwd
 *   out   [B, Hq, Nq, D]  the forward's O
 *   lse   f32 [B, Hq, Nq, 1] the forward's lse (required)
 *   dout  [B, Hq, Nq, D]  gradient of the loss with respect to O
 *   dq    [B, Hq, Nq, D]  written
 *   dk, dv [B, Hkv, Nkv, D] written (summed over the query heads of a group)
 *
 * No gradient is produced for the bias.  Delta and lse in log2 units (f32
 * [B, Hq, Nq] each) live in stream-ordered scratch on `stream` from the
 * library's per-device memory pool.
 */
int ffpa_bwd(const ffpa_tensor_t* q, const ffpa_tensor_t* k, const ffpa_tensor_t* v,
             const ffpa_tensor_t* bias, int causal, float scale, const ffpa_tensor_t* out,
             const ffpa_tensor_t* lse, const ffpa_tensor_t* dout, const ffpa_tensor_t* dq,
             const ffpa_tensor_t* dk, const ffpa_tensor_t* dv, ffpa_stream_t stream);

/*
 * ffpa_fwd_dropout / ffpa_bwd_dropout: ffpa_fwd and ffpa_bwd with dropout on
 * the attention probabilities (the "dropout" rows of the FFPA Attention
 * Benchmark page's "More Benchmark" tables).  Arguments as in ffpa_fwd /
 * ffpa_bwd, plus:
 *   dropout_p  drop probability, 0 <= p < 1 (else FFPA_ERR_INVALID_ARG);
 *              p == 0 is the call without dropout
 *   seed       64-bit generator key
 *   offset     32-bit stream index (e.g. a step counter)
 * The forward computes O = (P * Z) V with Z = keep / (1 - p) and the lse of
 * the undropped scores; the backward, given the same (p, seed, offset),
 * returns the gradients of that function for the same keep mask.  Keep mask:
 * for query row i and key j of query head h in batch b, Philox4x32-10 (ten
 * rounds of four 32-bit words, Salmon et al., SC 2011) runs on counter
 * (j / 8, i, b * Hq + h, offset) with key (seed & 0xffffffff, seed >> 32);
 * score (i, j) reads 16-bit field j % 2 of output word (j % 8) / 2 and is kept
 * when that value is at least t = min(65535, floor(p * 65536 + 1/2)).
 * b and h index the tensors of this call: a caller that splits a problem's
 * batches or heads over several calls (or GPUs) and wants the masks of the
 * unsplit call must pass views whose indices match, or tell the pieces apart
 * with distinct seeds or offsets.
 * The pages give no generator; this contract is the library's.  Dropout runs
 * on the D = 320 .. 1024 kernels only (FFPA_ERR_UNSUPPORTED for D <= 256),
 * with neither the decode path nor key splits (every Nq takes the fused
 * kernel).
 */
int ffpa_fwd_dropout(const ffpa_tensor_t* q, const ffpa_tensor_t* k, const ffpa_tensor_t* v,
                     const ffpa_tensor_t* bias, int causal, float scale, double dropout_p, uint64_t seed,
                     uint32_t offset, const ffpa_tensor_t* out, const ffpa_tensor_t* lse, ffpa_stream_t stream);
int ffpa_bwd_dropout(const ffpa_tensor_t* q, const ffpa_tensor_t* k, const ffpa_tensor_t* v,
                     const ffpa_tensor_t* bias, int causal, float scale, double dropout_p, uint64_t seed,
                     uint32_t offset, const ffpa_tensor_t* out, const ffpa_tensor_t* lse,
                     const ffpa_tensor_t* dout, const ffpa_tensor_t* dq, const ffpa_tensor_t* dk,
                     const ffpa_tensor_t* dv, ffpa_stream_t stream);

/*
 * ffpa_fwd_decode_noalloc: the decode forward (Nq <= 16) without allocating.
 * The pages have no counterpart; it exists for callers that cannot allocate
 * device memory during the call: code running under another framework's
 * memory pool or a serving loop that must not enter the CUDA
 * allocator on its hot path.  ffpa_fwd's decode path takes its slice
 * partials from the library's memory pool; this entry point keeps them in a fixed
 * 8 MiB device array inside the library (held by every GPU that loads the
 * library until the process exits) and calls no allocating routine.
 *
 *   Arguments, layouts, results and validation exactly as ffpa_fwd, plus:
 *   - Nq must be <= 16, else FFPA_ERR_UNSUPPORTED.
 *   - The partials take (D + 2) * 4 bytes per (batch, query head, query row,
 *     slice of keys; slices hold 128 to 256 keys, chosen per call so the
 *     decode CTAs fill whole waves); a call that needs more than 8 MiB returns
 *     FFPA_ERR_SCRATCH_LIMIT and launches nothing (e.g. B=1, Hq=8, Nq=1,
 *     Nkv=8192, D=512 takes 37 slices of 224 keys and needs 0.61 MB).
 *   - The first call on a device looks up the array's device address (one
 *     cudaGetSymbolAddress for that device); make that first call before
 *     any stream capture on the device.
 *   - All calls share the array.  Each call overwrites every partial it
 *     reads, so nothing carries over between calls, but calls whose work
 *     overlaps on the GPU (different streams or host threads) race on it:
 *     order them on one stream or synchronise between them.
 */
int ffpa_fwd_decode_noalloc(const ffpa_tensor_t* q, const ffpa_tensor_t* k, const ffpa_tensor_t* v,
                            const ffpa_tensor_t* bias, int causal, float scale, const ffpa_tensor_t* out,
                            const ffpa_tensor_t* lse, ffpa_stream_t stream);

/* Static text for a status code (never NULL). */
const char* ffpa_status_string(int status);

/*
 * Synchronise `stream`, then read and clear the current device's status word.
 * Returns FFPA_ERR_TIMEOUT if a kernel's bounded wait expired since the last
 * check, FFPA_ERR_CUDA if the synchronisation failed, FFPA_OK otherwise.
 */
int ffpa_check_status(ffpa_stream_t stream);

/*
 * ffpa_set_timing_events: measurement hook (no counterpart on the pages; it
 * exists so a benchmark can time each kernel of a call with CUDA events).
 *
 *   events  array of `count` cudaEvent_t handles created by the caller, or NULL
 *   count   0 disables the hook
 *
 * While set (per calling host thread), every later ffpa_fwd / ffpa_bwd call on
 * this thread records events[0] on its stream before its first kernel launch
 * and events[i] right after its i-th launch, for as many events as given
 * (ffpa_fwd launches 1 kernel on the fused path and 2 on the decode and
 * key-split paths; ffpa_bwd launches 4 for D <= 256 and 3 above).  The caller keeps ownership of
 * the events.  Returns FFPA_ERR_INVALID_ARG if count < 0, count > 8, or
 * events (or one of its first `count` handles) is NULL with count > 0.
 */
int ffpa_set_timing_events(void* const* events, int count);

/*
 * ffpa_selftest_wait_timeout: check of the timeout path (no counterpart on the
 * pages; every kernel's waits go through the same bounded wait).
 *
 * Launches, on `stream`, one warp that initialises an mbarrier nobody arrives
 * on and waits for it with the library's bounded wait.  After the wait limit
 * (250 ms) the kernel records a timeout in the device status word and exits;
 * it issues no TMA copy and no MMA, so nothing is left in flight.  The next
 * ffpa_check_status on the stream then returns FFPA_ERR_TIMEOUT (and clears
 * the word), and the context stays usable.  Returns FFPA_ERR_CUDA if the
 * launch fails, FFPA_OK otherwise.
 */
int ffpa_selftest_wait_timeout(ffpa_stream_t stream);

/* Library version: major * 10000 + minor * 100 + patch. */
int ffpa_version(void);

#ifdef __cplusplus
}
#endif
#endif /* FFPA_H_ */
