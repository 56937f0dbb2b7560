/*
 * decode_attn_splitkv.h -- split-KV decode attention (flash-decoding) for
 * NVIDIA GB300 (sm_103a), as a plain C ABI.
 *
 * The operation. One decode step: each of B sequences has one query token
 * with Hq query heads; its KV cache has Hkv heads (Hq % Hkv == 0, group size
 * G = Hq / Hkv) and L_b = cu_seqlens_k[b+1] - cu_seqlens_k[b] keys. Query head
 * h reads KV head h / G (the cur_kv_head rule of the TileLang tutorial page
 * decode_attention_splitkv.py, split segment). With s_j = scale * q_h . k_j,
 *
 *     out[b,h,:] = sum_j softmax(s)_j * v_j                      (j < L_b)
 *
 * (MiniInfer flash_decode_splitk.py, flash_decode_reference). The library
 * computes it the flash-decoding way: each sequence's key range is cut into
 * num_splits proportional pieces, split s covering
 *
 *     [floor(L_b * s / S), floor(L_b * (s+1) / S))
 *
 * (TileLang page, split segment, proportional split bounds). One CTA per
 * (sequence, KV head, split) computes, for every packed query head of that KV
 * head, the normalised partial output o_s and lse_s = ln sum_{j in s} exp(s_j);
 * a combine step then merges them exactly:
 *
 *     lse = ln sum_s exp(lse_s),   out = sum_s exp(lse_s - lse) * o_s
 *
 * (CS349E lecture 11, 04_flash_decoding.py, demo1_exact, first observation;
 * TileLang page, combine segment). An empty split (only possible when a
 * caller forces num_splits > L_b) has lse_s = -inf, o_s = 0 and weight 0, as
 * in the MiniInfer reduce kernel; a sequence with L_b = 0 gets out = 0.
 *
 * Conventions for every entry point below.
 *  - Pointers named "device" must be device memory of the current CUDA
 *    device; nothing is copied or allocated by the library, and nothing is
 *    retained after the call returns.
 *  - `stream` is a cudaStream_t (a CUstream) passed as void*; NULL means the
 *    legacy default stream. Device work is enqueued on it asynchronously; no
 *    entry point synchronises unless it says so.
 *  - Host-side checks run first; a call that returns anything but DA_OK has
 *    enqueued no device work.
 *  - Input and output elements are IEEE binary16 (DA_F16) or bfloat16
 *    (DA_BF16) values; accumulation is float32.
 */
#ifndef DECODE_ATTN_SPLITKV_H
#define DECODE_ATTN_SPLITKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    DA_OK = 0,
    DA_ERR_INVALID_ARG = 1,         /* a size, count or pointer is out of range or NULL */
    DA_ERR_UNSUPPORTED = 2,         /* head_dim other than 64/128, or no sm_103a device */
    DA_ERR_ALIGNMENT = 3,           /* a pointer is not aligned as documented */
    DA_ERR_WORKSPACE_TOO_SMALL = 4, /* workspace_bytes < decode_attn_splitkv_workspace_size() */
    DA_ERR_CUDA = 5,                /* a CUDA runtime or driver call failed */
    DA_ERR_SCRATCH_LIMIT = 6,       /* decode_attn_splitkv_noalloc: the problem needs more scratch
                                       than DA_NOALLOC_SCRATCH_BYTES */
    DA_ERR_DEVICE_TIMEOUT = 7       /* returned by the error readers (decode_attn_splitkv_get_error,
                                       decode_attn_splitkv_noalloc_get_error) when a pipeline wait
                                       of an earlier call on the device timed out
                                       (DA_DEVERR_TIMEOUT): that call's outputs are invalid */
} da_status;

typedef enum { DA_F16 = 0, DA_BF16 = 1 } da_dtype;

typedef enum {
    /* K, V: [kv_rows, Hkv, D] row-major; sequence b owns rows
       cu_seqlens_k[b] .. cu_seqlens_k[b+1]-1 (kv_rows = total_kv). */
    DA_LAYOUT_VARLEN = 0,
    DA_LAYOUT_VARLEN_THD = DA_LAYOUT_VARLEN,   /* the same layout: tokens x heads x dim */
    /* K, V: [B, Hkv, kv_rows, D] row-major; sequence b owns positions
       0 .. L_b-1 of its own [kv_rows, D] slab per KV head (kv_rows is the
       per-sequence capacity; L_b still comes from cu_seqlens_k). */
    DA_LAYOUT_BHSD = 1
} da_layout;

/* Bits of the device error word (see decode_attn_splitkv_get_error). */
#define DA_DEVERR_SEQLENS 0x1u /* a sequence's cu_seqlens_k range fell outside K/V; it was treated as empty */
#define DA_DEVERR_TIMEOUT 0x2u /* a pipeline wait exceeded its time limit; the outputs of that call are
                                  invalid and the workspace must be initialised again before reuse */

/* Largest num_splits accepted. */
#define DA_MAX_SPLITS 1024

/*
 * Workspace layout (all offsets from the workspace base, which must be
 * 256-byte aligned):
 *   [0, 256)            header: uint32 device error word at offset 0, the split step's
 *                       work-queue counters at offsets 64 and 128 (zero between calls:
 *                       each call's last take from the queue, or the last CTA of the
 *                       tcgen05 arm, resets them), rest reserved
 *   [256, 256 + A)      lse_part, float32 [B, Hq, num_splits], natural log of the
 *                       scaled scores, A = round_up(B*Hq*num_splits*4, 256)
 *   [256 + A, total)    o_part, float32 [B, Hq, num_splits, D], normalised per split
 * Returns the total size in bytes, or 0 if an argument is out of range.
 */
size_t decode_attn_splitkv_workspace_size(int B, int Hq, int D, int num_splits);

/* Byte offsets of lse_part and o_part inside the workspace (layout above). */
size_t decode_attn_splitkv_lse_offset(void);
size_t decode_attn_splitkv_opart_offset(int B, int Hq, int num_splits);

/*
 * Zero the workspace header (the device error word and the work-queue
 * counters). Call once on a freshly allocated workspace before its first use,
 * and again after a DA_DEVERR_TIMEOUT. Enqueued on `stream`.
 * Errors: DA_ERR_INVALID_ARG (NULL, or fewer than 256 bytes),
 * DA_ERR_ALIGNMENT (not 256-byte aligned), DA_ERR_CUDA.
 */
da_status decode_attn_splitkv_workspace_init(void* workspace, size_t workspace_bytes, void* stream);

/*
 * Split-count picker (host only, enqueues nothing). Chooses num_splits for a
 * batch whose KV lengths lie in [min_kv, max_kv]. The split step has
 * U * num_splits work items, U = B * Hkv * ceil(G/8), run by R = sm_count *
 * (2 at head_dim 128, 4 at 64) persistent CTAs.
 *   Even lengths (max_kv < 2 * min_kv), U >= 0.8 * sm_count: 1, unless the
 *     K/V stream exceeds 1.5e9 bytes; then round(1.68 * R / U), about 1.7 waves
 *     of items, so the work queue evens out unequal SM rates.
 *   Even lengths, fewer units: about one item per SM, ceil(sm_count / U),
 *     with splits of 256 to 1024 keys.
 *   Ragged lengths: about eight items per SM (splits of at least 64 keys),
 *     raised until the longest sequence's splits are at most twice one CTA's
 *     share of a lower bound of the total keys (max_kv + (B-1) * min_kv); with
 *     16-column items (G > 8, or G * T_q > 8 when Hq is passed as Hq * T_q for
 *     several query tokens) four items per SM and four shares. A batch of at
 *     most 128 sequences in which no sequence holds half of that lower bound is
 *     handed out longest first by the split step and gets fewer, longer
 *     splits: six items per SM and four shares (16-column items: three and
 *     eight).
 * No split is ever empty (num_splits <= min_kv; the TileLang page's scheduling
 * constraint, split kernel docstring). sm_count 0 means: query the current
 * device. Returns a value in [1, DA_MAX_SPLITS]; 1 when min_kv <= 0 or an
 * argument is out of range.
 */
int decode_attn_splitkv_num_splits(int B, int Hq, int Hkv, int D, int min_kv, int max_kv,
                                   int sm_count);

/* Split s of num_splits over a length-L sequence: [*start, *end) (host helper). */
void decode_attn_splitkv_split_range(int64_t L, int num_splits, int s, int64_t* start,
                                     int64_t* end);

/*
 * The whole decode attention: the split step, then the combine step, both on
 * `stream`.
 *   q              device, [B, Hq, D] elements of `dtype`, 16-byte aligned
 *   k, v           device, layout per `layout` (above), 16-byte aligned; may be
 *                  NULL only when kv_rows == 0
 *   cu_seqlens_k   device, int32 [B+1], non-decreasing; 4-byte aligned. Entries
 *                  outside the K/V extent set DA_DEVERR_SEQLENS on the device
 *                  and that sequence is treated as empty (never read out of bounds)
 *   B, Hq, Hkv     >= 1, Hq % Hkv == 0
 *   D              64 or 128
 *   kv_rows        >= 0: total_kv (VARLEN) or the per-sequence capacity (BHSD)
 *   scale          finite; the scores are scale * q . k (1/sqrt(D) is usual)
 *   num_splits     in [1, DA_MAX_SPLITS]; values above a sequence's length
 *                  stay exact (the extra splits are empty)
 *   out            device, [B, Hq, D] elements of `dtype`, 16-byte aligned,
 *                  rounded to nearest-even from float32
 *   workspace      device, >= decode_attn_splitkv_workspace_size(B,Hq,D,num_splits)
 *                  bytes, 256-byte aligned, initialised once (workspace_init);
 *                  after the call it holds the per-split lse_part and o_part
 * Errors (host-side, nothing enqueued): DA_ERR_INVALID_ARG, DA_ERR_UNSUPPORTED,
 * DA_ERR_ALIGNMENT, DA_ERR_WORKSPACE_TOO_SMALL; DA_ERR_CUDA if a launch fails.
 */
da_status decode_attn_splitkv(const void* q, const void* k, const void* v,
                              const int32_t* cu_seqlens_k, int B, int Hq, int Hkv, int D,
                              int kv_rows, da_dtype dtype, da_layout layout, float scale,
                              int num_splits, void* out, void* workspace,
                              size_t workspace_bytes, void* stream);

/*
 * The split step alone: fills lse_part and o_part in the workspace (layout
 * above). Same arguments and errors as decode_attn_splitkv, without `out`.
 */
da_status decode_attn_splitkv_partial(const void* q, const void* k, const void* v,
                                      const int32_t* cu_seqlens_k, int B, int Hq, int Hkv,
                                      int D, int kv_rows, da_dtype dtype, da_layout layout,
                                      float scale, int num_splits, void* workspace,
                                      size_t workspace_bytes, void* stream);

/*
 * The split step with its two products (q.k and p.v) on CUDA-core fp32 FMAs
 * instead of tensor cores: the comparison arm for that design choice (the
 * pages' kernels use tensor-core GEMMs for a packed group; this measures what
 * plain FMAs reach on the same pipeline). Same arguments, workspace results
 * and errors as decode_attn_splitkv_partial, plus DA_ERR_UNSUPPORTED when a KV
 * head serves more than 8 query heads (Hq / Hkv > 8). The library's own calls
 * never use it.
 */
da_status decode_attn_splitkv_partial_cuda_core(const void* q, const void* k, const void* v,
                                                const int32_t* cu_seqlens_k, int B, int Hq, int Hkv,
                                                int D, int kv_rows, da_dtype dtype, da_layout layout,
                                                float scale, int num_splits, void* workspace,
                                                size_t workspace_bytes, void* stream);

/*
 * The combine step alone: merges lse_part/o_part from the workspace into
 * out[B, Hq, D]. The workspace must hold a split step's results for the same
 * B, Hq, D and num_splits. Errors as above.
 */
da_status decode_attn_splitkv_combine(int B, int Hq, int D, int num_splits, da_dtype dtype,
                                      void* out, const void* workspace, size_t workspace_bytes,
                                      void* stream);

/* Largest batch accepted by decode_attn_splitkv_varsplit. */
#define DA_MAX_VARSPLIT_BATCH 1024

/*
 * Per-sequence split counts, for ragged batches. Instead of one num_splits
 * for every sequence, sequence b is cut into
 *
 *     S_b = 1 if L_b = 0, else min(max_splits, ceil(L_b / split_len))
 *
 * proportional splits [floor(L_b*s/S_b), floor(L_b*(s+1)/S_b)), so that work
 * items are about split_len keys long whatever the sequence length, and the
 * work queue balances them. The pages motivate it without specifying it: the
 * TileLang page notes that real frameworks choose the split count in their
 * scheduler (split kernel docstring) and the lecture page that real
 * implementations pick splits from batch, length and SM count
 * (04_flash_decoding.py, demo4_splits observations). No split is ever empty.
 *   split_len      >= 1 keys per split (target); max_splits in [1, DA_MAX_SPLITS]
 *   B              <= DA_MAX_VARSPLIT_BATCH (else DA_ERR_UNSUPPORTED)
 *   workspace      >= decode_attn_splitkv_workspace_size(B, Hq, D, max_splits);
 *                  lse_part/o_part use max_splits as the split stride, and
 *                  entries s >= S_b of a row are left untouched
 * The rows of a sequence with S_b = 1 are written by the split step itself (its
 * one split's weight is exactly 1); the combine step merges only the others, and
 * is not launched when max_splits = 1.
 * Other arguments, results and errors as decode_attn_splitkv.
 */
da_status decode_attn_splitkv_varsplit(const void* q, const void* k, const void* v,
                                       const int32_t* cu_seqlens_k, int B, int Hq, int Hkv,
                                       int D, int kv_rows, da_dtype dtype, da_layout layout,
                                       float scale, int split_len, int max_splits, void* out,
                                       void* workspace, size_t workspace_bytes, void* stream);

/*
 * Picker for decode_attn_splitkv_varsplit (host only): from the batch's
 * total and longest KV length, a split_len (a multiple of 64 keys, at least
 * 256) of about 0.4 of one persistent CTA's share of the keys (R = sm_count *
 * (2 at head_dim 128, 4 at 64) CTAs), raised so that the longest sequence has
 * at most about R / 2 work items, and the max_splits that the longest sequence
 * needs. With several query tokens pass Hq * T_q as Hq (the share then counts
 * each column chunk's pass over the keys). sm_count 0 means: query the current
 * device.
 * Returns 0, or -1 (and 1, 1) if an argument is out of range.
 */
int decode_attn_splitkv_varsplit_plan(int B, int Hq, int Hkv, int D, int64_t total_kv, int max_kv,
                                      int sm_count, int* split_len, int* max_splits);

/* Largest T_q accepted by decode_attn_splitkv_multiquery. */
#define DA_MAX_QUERY_TOKENS 16

/*
 * Several new query tokens per sequence (speculative or multi-token decoding).
 * Each sequence has T_q query tokens whose keys and values are already the
 * last T_q entries of its cache; token t sits at position L_b - T_q + t and
 * attends causally to keys [0, L_b - T_q + t] (a token that sees no key gets
 * out = 0). Splits still cut each sequence's whole range [0, L_b) as in
 * decode_attn_splitkv; a split holding no key a token may see is empty for
 * that token (lse = -inf, weight 0). The (token, head) pairs of one KV head's
 * group are packed together into the tensor-core columns (work items of 8
 * columns, or of 16 when G * T_q > 8), so with G * T_q <= 16 each K/V byte is
 * still read and multiplied once; more columns take several items, whose
 * repeated reads of the same keys come mostly from L2. The pages' split kernel has
 * query blocking only in the official examples it refers to (TileLang page,
 * module docstring item 1); the masking follows its split segment's -inf rule.
 *   q, out         device, [B, T_q, Hq, D] elements of `dtype`, 16-byte aligned
 *   T_q            in [1, DA_MAX_QUERY_TOKENS]
 *   workspace      >= decode_attn_splitkv_workspace_size(B * T_q, Hq, D, num_splits);
 *                  rows of lse_part/o_part are (b * T_q + t) * Hq + h
 * Pick num_splits with decode_attn_splitkv_num_splits(B, Hq * T_q, Hkv, ...).
 * Other arguments, results and errors as decode_attn_splitkv.
 */
da_status decode_attn_splitkv_multiquery(const void* q, const void* k, const void* v,
                                         const int32_t* cu_seqlens_k, int B, int T_q, int Hq,
                                         int Hkv, int D, int kv_rows, da_dtype dtype,
                                         da_layout layout, float scale, int num_splits, void* out,
                                         void* workspace, size_t workspace_bytes, void* stream);

/*
 * Several new query tokens per sequence (as decode_attn_splitkv_multiquery)
 * with per-sequence split counts S_b = 1 if L_b = 0, else min(max_splits,
 * ceil(L_b / split_len)) (as decode_attn_splitkv_varsplit): a ragged batch can
 * split only its long sequences, whose single items would otherwise outlast
 * the rest of the batch, and keep the short ones whole, written by the split
 * step itself with no combine.
 *   q, out         device, [B, T_q, Hq, D] elements of `dtype`, 16-byte aligned
 *   T_q            in [1, DA_MAX_QUERY_TOKENS]
 *   split_len      >= 1; max_splits in [1, DA_MAX_SPLITS]
 *   B              <= DA_MAX_VARSPLIT_BATCH (else DA_ERR_UNSUPPORTED)
 *   workspace      >= decode_attn_splitkv_workspace_size(B * T_q, Hq, D, max_splits);
 *                  rows of lse_part/o_part are (b * T_q + t) * Hq + h, with
 *                  max_splits as the split stride; entries s >= S_b are left untouched
 * Pick split_len and max_splits with decode_attn_splitkv_varsplit_plan(B, Hq * T_q, ...).
 * Other arguments, results and errors as decode_attn_splitkv.
 */
da_status decode_attn_splitkv_multiquery_varsplit(const void* q, const void* k, const void* v,
                                                  const int32_t* cu_seqlens_k, int B, int T_q, int Hq,
                                                  int Hkv, int D, int kv_rows, da_dtype dtype,
                                                  da_layout layout, float scale, int split_len,
                                                  int max_splits, void* out, void* workspace,
                                                  size_t workspace_bytes, void* stream);

/*
 * Comparison arm for the product choice on Blackwell: decode_attn_splitkv_multiquery
 * with the split step on the tcgen05 tensor cores and the accumulators in tensor
 * memory, for G * T_q > 8 and G <= 32 (else DA_ERR_UNSUPPORTED). Per 64-key stage
 * S = Q K^T and O += P V run as tcgen05.mma with M = 128 rows: the item's packed
 * columns (up to 32, whole query tokens of one KV head's group), laid into all four
 * 32-row quarters so that four warps, one per SM sub-partition, each take 16 of the
 * stage's keys; P goes back to tensor memory as the A operand of the PV product.
 * Same arguments, results and errors as decode_attn_splitkv_multiquery; the outputs
 * agree with it to fp16/bf16 rounding (the order of the sums differs). It measures
 * slower than the mma.sync path on every shape tried: with M fixed at 128 the
 * products of a stage cost about as much tensor time as the stage takes to stream,
 * whatever the column count.
 */
da_status decode_attn_splitkv_multiquery_tmem(const void* q, const void* k, const void* v,
                                              const int32_t* cu_seqlens_k, int B, int T_q, int Hq,
                                              int Hkv, int D, int kv_rows, da_dtype dtype,
                                              da_layout layout, float scale, int num_splits, void* out,
                                              void* workspace, size_t workspace_bytes, void* stream);

/*
 * Read and clear the device error word of `workspace`: *device_error_bits gets
 * its DA_DEVERR_* bits (the word can hold more than one, so they are returned
 * apart from the status). Synchronises `stream` first.
 * Returns DA_ERR_DEVICE_TIMEOUT when DA_DEVERR_TIMEOUT is among the bits (the
 * outputs of the call that set it are invalid; initialise the workspace again
 * before reusing it), else DA_OK; a DA_DEVERR_SEQLENS bit alone is reported
 * through the bits with DA_OK (the bad sequences were computed as empty).
 * Errors: DA_ERR_INVALID_ARG, DA_ERR_ALIGNMENT, DA_ERR_CUDA (bits then untouched).
 */
da_status decode_attn_splitkv_get_error(void* workspace, uint32_t* device_error_bits,
                                        void* stream);

/*
 * Diagnostic: launch one CTA that waits on a pipeline barrier nothing will
 * complete, through the same bounded wait the split step uses, with a limit
 * of timeout_us microseconds. It must give up, set DA_DEVERR_TIMEOUT in the
 * workspace's error word and return; the device stays usable. Used by the
 * test-suite to exercise the time-out path without hanging a GPU.
 */
da_status decode_attn_splitkv_selftest_timeout(void* workspace, size_t workspace_bytes,
                                               unsigned timeout_us, void* stream);

/* Size of the library's built-in scratch array used by decode_attn_splitkv_noalloc. */
#define DA_NOALLOC_SCRATCH_BYTES (8u * 1024u * 1024u)

/*
 * decode_attn_splitkv without a caller-supplied workspace, for callers that
 * cannot allocate device memory: code that runs behind a plugin or operator
 * interface which hands it only its input and output buffers and owns every
 * allocation itself, and code on a latency-critical path where cudaMalloc is
 * off limits because it can synchronise the whole device. The pages have no
 * counterpart of this entry point; it is an addition of this library.
 *
 * Instead of a workspace it uses one scratch array compiled into the library
 * (a file-scope __device__ array of DA_NOALLOC_SCRATCH_BYTES = 8 MiB). Every
 * GPU that loads the library holds that array until the process exits. The
 * call itself allocates nothing: no cudaMalloc, no cudaFree, no allocating
 * library routine.
 *   - Arguments, layout and results are those of decode_attn_splitkv, minus
 *     the workspace. The per-split results land in the scratch array, where
 *     the caller cannot read them.
 *   - Problems whose workspace_size(B, Hq, D, num_splits) exceeds
 *     DA_NOALLOC_SCRATCH_BYTES are refused with DA_ERR_SCRATCH_LIMIT and
 *     nothing is enqueued. (For example B=64, Hq=28, D=128 fits up to 9 splits.)
 *   - The argument checks run on the host before anything touches a device,
 *     so a refused call (DA_ERR_INVALID_ARG, DA_ERR_ALIGNMENT, DA_ERR_UNSUPPORTED,
 *     DA_ERR_SCRATCH_LIMIT) makes no CUDA call at all.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current and caches it together
 *     with the id of the CUDA context it belongs to; make that first call
 *     before any stream capture on the device. A later call in another context
 *     of the same device (after cudaDeviceReset, which destroys the context and
 *     the array with it) finds a different id and looks the address up again.
 *   - All calls share the one array, which keeps the previous call's
 *     contents; each call clears the part that must start at zero (the error
 *     word and the work-queue counters) and overwrites the rest before reading
 *     it. Calls that can overlap on the GPU (different streams without ordering
 *     between them, or several host threads) race on the array and corrupt
 *     each other's results: serialise them.
 *   - Device-side error bits (DA_DEVERR_*) of the last call on a device land in
 *     the array's error word: read them with decode_attn_splitkv_noalloc_get_error.
 * Errors: those of decode_attn_splitkv, plus DA_ERR_SCRATCH_LIMIT.
 */
da_status decode_attn_splitkv_noalloc(const void* q, const void* k, const void* v,
                                      const int32_t* cu_seqlens_k, int B, int Hq, int Hkv,
                                      int D, int kv_rows, da_dtype dtype, da_layout layout,
                                      float scale, int num_splits, void* out, void* stream);

/*
 * decode_attn_splitkv_get_error for decode_attn_splitkv_noalloc: read and clear
 * the error word of the built-in scratch array of the current device, after
 * synchronising `stream` (the stream of the noalloc call to diagnose). Like that
 * entry point it has no counterpart on the pages and allocates nothing.
 * Returns DA_ERR_DEVICE_TIMEOUT when DA_DEVERR_TIMEOUT is set, else DA_OK, with
 * the bits in *device_error_bits; DA_ERR_INVALID_ARG (NULL) or DA_ERR_CUDA.
 */
da_status decode_attn_splitkv_noalloc_get_error(uint32_t* device_error_bits, void* stream);

/*
 * Time model of one decode_attn_splitkv (or _multiquery) call on GB300, in
 * microseconds: a restatement of the lecture page's decode time model
 * (04_flash_decoding.py, decode_attention_time, best_splits; its A100/H100
 * constants are not on the page) for this library's persistent kernel:
 *
 *   T = t0 + makespan + kappa * B_max / (bw / min(n_items, R))
 *         + [S > 1] * (t_comb + W_ws / bw_comb)
 *
 * makespan: a processor-sharing run of the n_items work items, in queue order
 * (the sequences of a batch of 2 to 128 longest first, ties by index, as the
 * split step hands out a ragged varlen batch), over R = (2 at D = 128, 4 at
 * D = 64) * sm_count persistent CTAs; before each item a CTA spends t_item,
 * then streams the item's K/V bytes (its keys rounded up to 16, times 4*D) at
 * min(r_cta, bw / number of CTAs streaming). When a KV head's columns take c
 * chunks, each chunk's item is charged 1/c of the bytes at 1/c of the rate
 * (the chunks of a split read its keys once from HBM between them). B_max: the
 * largest item's charged bytes (kappa charges the last item for unequal CTA
 * rates); W_ws = B*T_q*Hq*S*(D+1)*4 workspace bytes combined.
 *   kv_lens   host, int32 [B] sequence lengths (negative counts as 0)
 *   params    host, double[8] {t0 us, t_item us, r_cta B/us, bw B/us, t_comb us,
 *             bw_comb B/us, kappa, r_cta2 B/us}, or NULL for the built-in GB300
 *             calibration; r_cta2 replaces r_cta for items of 16 columns
 *             (G * T_q > 8), which carry twice the products per key
 * Returns the predicted time, or a negative value if an argument is out of range.
 */
double decode_attn_splitkv_model_us(const int32_t* kv_lens, int B, int Hq, int Hkv, int D, int T_q,
                                    int num_splits, int sm_count, const double* params);

/*
 * The same model for a decode_attn_splitkv_varsplit (or _multiquery_varsplit)
 * call: sequence b has S_b = 1 if L_b = 0, else min(max_splits, ceil(L_b /
 * split_len)) splits, the work items go out in sequence order, and the combine
 * reads the rows of the sequences with S_b > 1 (T_q * Hq * S_b * (D + 1) * 4
 * bytes each). split_len >= 1; other arguments as decode_attn_splitkv_model_us.
 * Returns the predicted time, or a negative value if an argument is out of range.
 */
double decode_attn_splitkv_model_varsplit_us(const int32_t* kv_lens, int B, int Hq, int Hkv, int D, int T_q,
                                             int split_len, int max_splits, int sm_count, const double* params);

/*
 * The split count (up to min(shortest length, 256)) that the built-in time model
 * predicts fastest, and the predicted time in *predicted_us (may be NULL): the
 * model-driven counterpart of decode_attn_splitkv_num_splits (the lecture
 * page's best_splits). Returns 1 on out-of-range arguments.
 */
int decode_attn_splitkv_model_best_splits(const int32_t* kv_lens, int B, int Hq, int Hkv, int D,
                                          int T_q, int sm_count, double* predicted_us);

/* Static, human-readable name of a status code. */
const char* decode_attn_splitkv_status_string(da_status status);

#ifdef __cplusplus
}
#endif

#endif /* DECODE_ATTN_SPLITKV_H */
