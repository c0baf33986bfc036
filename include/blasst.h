/*
 * blasst.h -- C ABI of the GB300 (sm_103a) skip-softmax FlashAttention library.
 *
 * The method (BLASST, "Dynamic BLocked Attention Sparsity via Softmax
 * Thresholding"): in the streaming online-softmax pass over key tiles, a tile
 * whose best score lies more than ln(lambda) below the running maximum in EVERY
 * query row of the tile skips its exponentials, its row sums, its V load and its
 * P.V product.  Definitions followed:
 *   - online-softmax recurrence and tiling: Hitchhiker's Guide Phase 08,
 *     Section 1 ("FlashAttention: IO-Optimal Attention", "FlashAttention Tiling
 *     Strategy");
 *   - the skip test m~ - m < ln(lambda), m the running max after the tile's own
 *     update, required for every row: Skip-Softmax design doc, "Algorithm";
 *     BLASST talk notes, "BLASST algorithm" (Eq. 2);
 *   - lambda = threshold_scale_factor / max_kv_len with the two mutually
 *     exclusive controls: Skip-Softmax design doc, "From configuration to the
 *     kernel threshold";
 *   - prefill skips softmax + PV, decode additionally skips the V load (loads K
 *     tiles first, issues V only for tiles that pass): BLASST talk notes,
 *     "kernel design: skip predicate reduction" (Figs. 3 and 4).
 *
 * Conventions shared by every entry point
 *   - Tensors are dense, row-major, bf16 (uint16 bit pattern), in DEVICE memory
 *     owned by the caller, 16-byte aligned:
 *         q [B, Hq, Lq, d]     k, v [B, Hkv, Lkv, d]     o [B, Hq, Lq, d]
 *     (decode: q and o are [B, Hq, d]).  Query head h reads KV head h / (Hq/Hkv).
 *   - lse is fp32 [B, Hq, Lq] (decode [B, Hq]): m + ln(l) in natural-log units of
 *     the scaled scores; -inf for a row that sees no key (its o row is 0).
 *   - scores are scale * (q . k); scale must be finite and > 0.
 *   - lambda in [0, 1].  0 skips nothing.  Values above 1 are rejected: the test's
 *     left side exp(m~ - m) never exceeds 1, so lambda > 1 would skip every tile
 *     including the first and leave O/l undefined.
 *   - Key/query tiles are 128 x 128.  Causal masking is bottom-right aligned:
 *     key c is visible to query row r iff c <= r + (Lkv - Lq).
 *   - Every call only enqueues work on `stream` (a cudaStream_t; NULL = legacy
 *     default stream) after validating its arguments on the host; nothing is
 *     synchronous.  The library allocates nothing and keeps no state except one
 *     device status word per device (see blasst_device_status).
 *   - Return value: BLASST_OK (0), a positive warning, or a negative error
 *     code; no work is enqueued when an error is returned.
 */
#ifndef BLASST_H
#define BLASST_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* status codes */
#define BLASST_OK 0
#define BLASST_WARN_LAMBDA_GE_1 1        /* blasst_lambda: curve gave lambda > 1 (value still returned) */
#define BLASST_ERR_INVALID_ARG (-1)      /* null required pointer, bad size, lambda/scale out of range */
#define BLASST_ERR_UNSUPPORTED (-2)      /* valid request the library does not support (d, G, alignment,
                                            memory that is not this GPU's on a cluster path) */
#define BLASST_ERR_WORKSPACE_TOO_SMALL (-3)
#define BLASST_ERR_CUDA (-4)             /* a CUDA runtime/driver call failed */
#define BLASST_ERR_TIMEOUT (-5)          /* a device-side wait ran past its limit (see blasst_device_status) */
#define BLASST_ERR_NO_CALIBRATION (-6)   /* target-sparsity mode without finite coefficients a, b */
#define BLASST_ERR_SCRATCH_LIMIT (-7)    /* blasst_decode_noalloc: partials exceed the library's static scratch */
#define BLASST_ERR_PAGE_TABLE (-8)       /* blasst_device_status: a page index or sequence length of a paged
                                            decode was out of range (those keys read as zeros / length clamped) */

/* flags for blasst_prefill_ex */
#define BLASST_PREFILL_ELIDE_V 0x1u      /* default kernel: load V_j only if a query tile of the CTA keeps key tile j */
#define BLASST_PREFILL_P_VIA_SMEM 0x2u   /* one query tile per CTA, P staged in shared memory (results identical) */
#define BLASST_PREFILL_ONE_QTILE 0x4u    /* one query tile per CTA, P in tensor memory (results identical) */
#define BLASST_PREFILL_WIDE 0x8u         /* two query tiles per CTA, two softmax threads per row (results identical) */
#define BLASST_FLAG_TEST_SHORT_WATCHDOG 0x80000000u /* test only: waits give up after 200 us and the MMA issuer
                                                       first waits on a barrier nothing arrives on, so the call
                                                       always ends in BLASST_ERR_TIMEOUT (outputs invalid) */

/*
 * Prefill / non-causal self-attention forward.
 *   q, k, v, o          see conventions; o is written for rows r < Lq only.
 *   lse                 nullable fp32 [B, Hq, Lq].
 *   B, Hq, Hkv          batch, query heads, KV heads (Hq % Hkv == 0).
 *   Lq, Lkv             query / key lengths (>= 1).
 *   d                   head dim: 64 or 128.
 *   causal              0 or 1.
 *   scale, lambda       see conventions.
 *   skipped_tiles_out   nullable device uint64: set to the number of skipped
 *                       (query tile, key tile) pairs over the whole call.
 * The skip unit is 128 query rows of ONE query head x 128 keys.  Key tiles that no
 * row of a query tile can see (causal) are not visited and not counted.
 */
int blasst_prefill(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                   int Lq, int Lkv, int d, int causal, float scale, float lambda,
                   unsigned long long* skipped_tiles_out, void* stream);

/*
 * As blasst_prefill, plus:
 *   skip_map   nullable device uint8 [B, Hq, ceil(Lq/128), ceil(Lkv/128)]:
 *              0 = computed, 1 = skipped, 2 = not visited.
 *   margins    nullable device fp32, same shape: max over the tile's rows of
 *              (m~ - m) in scaled-score units (+inf when a row has no visible key
 *              yet, NaN for tiles not visited).  lambda-independent for lambda <= 1;
 *              a tile is skipped iff margin < ln(lambda).
 *   flags      BLASST_PREFILL_P_VIA_SMEM, BLASST_PREFILL_ONE_QTILE, BLASST_PREFILL_WIDE
 *              (kernel variants with identical results; default: two query tiles per CTA,
 *              one softmax thread per query row), BLASST_FLAG_TEST_SHORT_WATCHDOG.
 *              BLASST_PREFILL_ELIDE_V (default kernel only; with another variant flag:
 *              BLASST_ERR_UNSUPPORTED) also skips the V tile load of a key tile that both
 *              query tiles of a CTA skip.  The BLASST talk notes ("Kernel" Q&A) keep loading
 *              V in prefill; eliding it makes each V load wait for the tile vote, so it
 *              saves L2/HBM bytes at the cost of exposing the load latency.  Results are
 *              identical either way.
 */
int blasst_prefill_ex(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
                      int Hkv, int Lq, int Lkv, int d, int causal, float scale, float lambda,
                      unsigned long long* skipped_tiles_out, unsigned char* skip_map, float* margins,
                      unsigned flags, void* stream);

/*
 * Prefill with a causal sliding window of `window` keys (BLASST talk notes, Q&A: the
 * method carries over to windowed attention; the notes give no definition, and this
 * library takes the causal mask cut to the last `window` keys): query row r sees
 * keys c with r' - window < c <= r', r' = r + Lkv - Lq.  Key tiles outside every
 * row's window are not visited (skip map 2).  Arguments as blasst_prefill_ex with
 * causal implied; window >= 1 (else BLASST_ERR_INVALID_ARG); flags may hold
 * BLASST_PREFILL_ELIDE_V, the other variant flags give BLASST_ERR_UNSUPPORTED.
 */
int blasst_prefill_window(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
                          int Hkv, int Lq, int Lkv, int d, int window, float scale, float lambda,
                          unsigned long long* skipped_tiles_out, unsigned char* skip_map, float* margins,
                          unsigned flags, void* stream);

/*
 * Split-KV plan for decode.  Split s of S covers key tiles
 * [floor(s*nT/S), floor((s+1)*nT/S)), nT = ceil(Lkv/128); each split is an
 * independent pass (its running max starts at -inf), so S changes which tiles are
 * skipped and is part of the result's definition.
 *   requested  0 = choose automatically for this GPU, else 1 <= requested <= nT.
 *   out        receives S.
 */
int blasst_decode_num_splits(int B, int Hq, int Hkv, int Lkv, int d, int requested, int* out);

/* Workspace bytes blasst_decode needs for num_splits splits (0 when num_splits == 1). */
size_t blasst_decode_workspace_size(int B, int Hq, int Hkv, int Lkv, int d, int num_splits);

/*
 * Decode forward: one query token per sequence against a KV cache.
 *   q [B, Hq, d], k_cache/v_cache [B, Hkv, Lkv, d], o [B, Hq, d] bf16; lse nullable fp32 [B, Hq].
 *   d is 64 or 128.  The skip unit is the G = Hq/Hkv query heads that read one KV
 *   head x 128 keys; G must be 1, 2, 4, 8, 16, 32, 64 or 128 (MQA: Hkv = 1).  Above
 *   16 the group runs on a wide-group kernel (a cluster of G/64 CTAs at 128).  V tiles
 *   of skipped key tiles are never loaded.
 *   num_splits   S from blasst_decode_num_splits (explicit: the split plan is part
 *                of the result).
 *   workspace    device memory of at least blasst_decode_workspace_size() bytes,
 *                16-byte aligned (may be NULL when S == 1).  Holds per-split
 *                partial results; a second kernel merges them by log-sum-exp.
 *   skipped_tiles_out  nullable device uint64 (count of skipped (b, hkv, tile)).
 *   skip_map     nullable device uint8 [B, Hkv, nT] (0 computed, 1 skipped).
 *   margins      nullable device fp32 [B, Hkv, nT] (as for prefill).
 */
/*   With 128 heads per KV head (the cluster form) q, k_cache and v_cache must be device
 *   memory of the current GPU: the two CTAs of a cluster share key loads by multicast,
 *   which must read this GPU's own memory.  Host, managed or another GPU's memory
 *   returns BLASST_ERR_UNSUPPORTED. */
int blasst_decode(const void* q, const void* k_cache, const void* v_cache, void* o, float* lse, int B, int Hq,
                  int Hkv, int Lkv, int d, float scale, float lambda, int num_splits, void* workspace,
                  size_t workspace_bytes, unsigned long long* skipped_tiles_out, unsigned char* skip_map,
                  float* margins, void* stream);

/*
 * Decode against a paged KV cache, with a key count per sequence (The Hitchhiker's
 * Guide, Phase 08, Section 3 "Continuous Batching & Paged Attention": key i of
 * sequence b is row i mod page_size of page page_table[b][i / page_size]; the
 * Skip-Softmax design doc, "From configuration to the kernel threshold": lambda is
 * one value per call, resolved against max_kv_len with blasst_lambda).
 *   q [B, Hq, d], o [B, Hq, d] bf16; lse nullable fp32 [B, Hq].
 *   k_pages / v_pages  bf16 page pools of num_pages pages, each page_size keys of
 *                every KV head: token_major = 1: [num_pages][page_size][Hkv][d];
 *                token_major = 0: [num_pages][Hkv][page_size][d].  16-byte aligned.
 *   page_table   device int32 [B, max_pages_per_seq]; entries past a sequence's
 *                last page are never read.  max_pages_per_seq * page_size >= max_kv_len.
 *   seq_lens     nullable device int32 [B]: keys of sequence b, 0 <= seq_lens[b] <=
 *                max_kv_len (NULL: every sequence has max_kv_len keys).  A sequence
 *                of length 0 gives o = 0, lse = -inf.
 *   page_size    8, 16, 32, 64, or a multiple of 128 (else BLASST_ERR_UNSUPPORTED).
 *   G = Hq/Hkv   1, 2, 4, 8 or 16 in this form (else BLASST_ERR_UNSUPPORTED).
 *   window       0, or a sliding window: only the last `window` keys of each
 *                sequence are attended (keys c >= seq_lens[b] - window).
 *   num_splits   as for blasst_decode, planned on max_kv_len (or on the window when
 *                it is shorter): split s of sequence b covers its visited tiles
 *                [lo + floor(s*(nT_b-lo)/S), lo + floor((s+1)*(nT_b-lo)/S)), nT_b =
 *                ceil(seq_lens[b]/128), lo = the tile holding the first key in the
 *                window (0 without one); a split with no tile contributes nothing.
 *   workspace    as for blasst_decode (blasst_decode_workspace_size with max_kv_len).
 *   skip_map / margins  nullable [B, Hkv, ceil(max_kv_len/128)], tiles past a
 *                sequence's end stay "not visited" (2 / NaN).
 *   A page index outside [0, num_pages) or a length outside [0, max_kv_len) is
 *   not trusted: those keys read as zeros (no memory outside the pool is touched),
 *   the length is clamped, and blasst_device_status reports BLASST_ERR_PAGE_TABLE.
 *   Keys past seq_lens[b] on the sequence's last page are loaded but get zero
 *   weight; they must hold finite values (a zeroed or previously written pool).
 */
int blasst_decode_paged(const void* q, const void* k_pages, const void* v_pages, const int* page_table,
                        const int* seq_lens, void* o, float* lse, int B, int Hq, int Hkv, int max_kv_len,
                        int window, int d, int num_pages, int page_size, int max_pages_per_seq, int token_major,
                        float scale, float lambda, int num_splits, void* workspace, size_t workspace_bytes,
                        unsigned long long* skipped_tiles_out, unsigned char* skip_map, float* margins,
                        void* stream);

/*
 * Decode without any device allocation (the pages have no counterpart: this entry
 * point exists for callers that cannot allocate).  Same arguments and results as
 * blasst_decode, minus the workspace: the per-split partials go to a device array
 * of blasst_decode_noalloc_scratch_bytes() bytes (4 MiB) that the library declares
 * statically, so code whose device memory belongs to another allocator, or a serving
 * loop that must not allocate between steps, can still split the key range.
 *   - Requires num_splits * B * Hq * (d + 1) * 4 bytes (rounded as for
 *     blasst_decode_workspace_size) <= the scratch size; larger requests return
 *     BLASST_ERR_SCRATCH_LIMIT before any work is enqueued.
 *   - The array exists once per device, for the life of the process, and every call
 *     on that device shares it: calls that overlap on the GPU race on it.
 *   - The first call on a device (with that device current) looks up the array's
 *     device address; make that first call before any stream capture.
 *   - Allocates nothing and calls no allocating routine.
 */
int blasst_decode_noalloc(const void* q, const void* k_cache, const void* v_cache, void* o, float* lse, int B,
                          int Hq, int Hkv, int Lkv, int d, float scale, float lambda, int num_splits,
                          unsigned long long* skipped_tiles_out, unsigned char* skip_map, float* margins,
                          void* stream);

/* Size in bytes of the static scratch array blasst_decode_noalloc uses. */
size_t blasst_decode_noalloc_scratch_bytes(void);

/*
 * Decode for multi-head latent attention in its absorbed form (the pages name MLA
 * decode as the case where the skipped exponentials and P.V products pay, since it
 * can be compute-bound: Skip-Softmax design doc, "Kernel"; they give no formula).
 * Every cached token holds one row of dk = 576 bf16 values (a 512-value latent
 * vector followed by a 64-value rotary key) shared by all query heads: head h
 * scores it as scale * (q_h . row) over all dk values, and the token's value is the
 * row's first dv = 512 values.  One skip decision covers all Hq heads x 128 keys.
 *   q [B, Hq, dk], o [B, Hq, dv] bf16; lse nullable fp32 [B, Hq].
 *   Hq           1, 2, 4, 8, 16, 32, 64 or 128 query heads (else
 *                BLASST_ERR_UNSUPPORTED); above 64 the heads are spread over a cluster
 *                of Hq / 64 CTAs that share the key loads.  dk must be 576 and dv 512
 *                (else BLASST_ERR_UNSUPPORTED).
 *   kv           page_table NULL: contiguous bf16 [B][max_kv_len][dk];
 *                page_table set: a pool of num_pages pages of page_size rows,
 *                bf16 [num_pages][page_size][dk], row i of sequence b at row
 *                i mod page_size of page page_table[b][i / page_size] (The
 *                Hitchhiker's Guide, Phase 08, Section 3, "Paged Attention");
 *                page_size 8, 16, 32, 64 or a multiple of 128, and
 *                max_pages_per_seq * page_size >= max_kv_len; (num_pages + 1) *
 *                page_size must stay below 2^31 - 128 (else BLASST_ERR_UNSUPPORTED).
 *                16-byte aligned.
 *                (num_pages, page_size, max_pages_per_seq are ignored without a
 *                page table.)
 *   seq_lens     nullable device int32 [B]: rows of sequence b (NULL: max_kv_len
 *                each); a sequence of length 0 gives o = 0, lse = -inf.  Rows past
 *                seq_lens[b] in the sequence's last 128-row tile (or page) are read
 *                but get zero weight: they must hold finite values.
 *   num_splits   1 .. ceil(max_kv_len / 128); blasst_mla_decode_num_splits plans one.
 *                Split s of sequence b covers its tiles [floor(s*nT_b/S),
 *                floor((s+1)*nT_b/S)), nT_b = ceil(seq_lens[b]/128); each split is an
 *                independent pass and the splits are merged by log-sum-exp.
 *   workspace    device memory of blasst_mla_decode_workspace_size bytes when
 *                num_splits > 1 (16-byte aligned), else may be NULL.
 *   skipped_tiles_out  nullable, zeroed then accumulated on the stream.
 *   skip_map / margins nullable [B, ceil(max_kv_len/128)] (0 computed, 1 skipped,
 *                2 not visited / the tile's max over heads of m~ - m, NaN if not
 *                visited).
 *   Out-of-range page indices and lengths are handled as for blasst_decode_paged.
 */
/*   Above 64 heads (the cluster form) q and kv must be device memory of the current GPU
 *   (the CTAs of a cluster share key loads by multicast): anything else returns
 *   BLASST_ERR_UNSUPPORTED. */
int blasst_mla_decode(const void* q, const void* kv, const int* page_table, const int* seq_lens, void* o,
                      float* lse, int B, int Hq, int max_kv_len, int dk, int dv, int num_pages, int page_size,
                      int max_pages_per_seq, float scale, float lambda, int num_splits, void* workspace,
                      size_t workspace_bytes, unsigned long long* skipped_tiles_out, unsigned char* skip_map,
                      float* margins, void* stream);

/* Split count for blasst_mla_decode: `requested` (1 .. ceil(max_kv_len/128)) if
 * positive, else the fewest splits whose B * splits * max(1, Hq/64) CTAs fill the
 * last wave of the GPU's SMs to at least 90 %. */
int blasst_mla_decode_num_splits(int B, int Hq, int max_kv_len, int requested, int* out);

/* Workspace bytes blasst_mla_decode needs for num_splits splits (0 when 1). */
size_t blasst_mla_decode_workspace_size(int B, int Hq, int max_kv_len, int num_splits);

/*
 * Threshold resolution (Skip-Softmax design doc, "From configuration to the
 * kernel threshold"; BLASST talk notes, "threshold calibration", Eq. 3):
 *   mode 0 (threshold):        lambda = threshold           (any Lkv)
 *   mode 1 (target sparsity):  lambda = a * exp(b * s) / Lkv
 * Returns BLASST_ERR_INVALID_ARG for a bad mode, Lkv < 1, a negative or
 * non-finite threshold, or s outside [0, 1]; BLASST_ERR_NO_CALIBRATION when mode 1
 * is asked without finite a and b (use mode 0 instead); BLASST_WARN_LAMBDA_GE_1
 * (with the raw value in *lambda_out) when the result exceeds 1.
 */
int blasst_lambda(int mode, double threshold, double a, double b, double target_sparsity, long long Lkv,
                  double* lambda_out);

/* Read (and with clear != 0, reset) this device's status word after synchronising
 * the device.  Returns BLASST_OK, or BLASST_ERR_TIMEOUT if a kernel of this library
 * gave up a wait since the last clear (its outputs are then invalid). */
int blasst_device_status(int clear);

/* Static English description of a status code. */
const char* blasst_status_string(int status);

#ifdef __cplusplus
}
#endif
#endif /* BLASST_H */
