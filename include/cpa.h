/*
 * cpa.h -- C ABI of the GB300 (sm_103a) paged chunked-prefill attention
 * library (libcpa.so).
 *
 * One step of an LLM serving engine hands the library a mixed batch of
 * active tokens: prefill chunks scheduled under a per-step token budget and
 * single-token decodes.  Request r has num_new_tokens[r] active tokens whose
 * queries attend to cached_seq_len[r] tokens of prior K/V -- held in a
 * block-paged pool and reached through row r of a block table -- and,
 * causally, to the request's own active tokens.  Active token i of request
 * r sits at absolute position cached_seq_len[r] + i.  Its new K/V row is
 * written into the pool slot of that position.
 *
 * Sources (page title, section):
 *   "Prefill Processing" (AWS Neuron vLLM design doc): Key Concepts
 *     (active tokens, cached KV segments, kv_segment_size, cached_seq_len),
 *     Kernel Interface (prior_tokens per request, segment count derived
 *     inside the kernel), Partial KV Segment Handling, Attention Metadata
 *     (block table, slot mapping, block size, max blocks per sequence),
 *     Block Allocation (block table rows, unallocated columns).
 *   "Prefill Optimisation": section 2 (causal equivalence: chunked prefill
 *     equals one-shot causal attention; online-softmax rescaling across
 *     tiles), section 6 (grouped-query attention: H_kv key/value heads for
 *     H_q query heads).
 *   "Chunked Prefill" (blog note): the greedy decode-first token budget and
 *     the absolute position offset of each chunk.
 *
 * Conventions shared by every entry point:
 *   - Element type: CPA_DTYPE_BF16 or CPA_DTYPE_FP32; q, k_new, v_new and
 *     out share it, and so do the pools unless kv_format selects the FP8
 *     cache (below).
 *   - q     [T, H_q, d]   contiguous, rows packed by request (cu_new_tokens).
 *   - k_new [T, H_kv, d]  contiguous; v_new likewise.
 *   - out   [T, H_q, d]   contiguous.
 *   - lse   [T, H_q]      float32, natural log of the softmax denominator of
 *                         the scaled scores (nullable).
 *   - k_cache, v_cache [num_blocks, block_size, H_kv, d] contiguous: the
 *     slot of position p of request r is
 *       block_table[r * max_blocks_per_seq + p / block_size] * block_size
 *       + p % block_size,
 *     and a slot is one row of the pool.
 *   - Query head h reads key/value head h / (H_q / H_kv).
 *   - FP8 cache (kv_format = CPA_KV_FP8_E4M3): the pools hold one byte per
 *     element, an FP8 E4M3 code (OCP format: sign, 4 exponent bits with bias
 *     7, 3 mantissa bits; exponent field 0 holds the subnormals m * 2^-9;
 *     S.1111.111 is NaN; largest finite value 448), with one float scale per
 *     kv head for keys (k_scale) and one for values (v_scale).  Element x of
 *     kv head g is stored as the code nearest to fl32(x / scale[g]), ties to
 *     an even mantissa, saturated to +-448 (NaN stays NaN); a code c stands
 *     for value(c) * scale[g].  Attention reads every key and value -- the
 *     active tokens' own new rows included -- through this encoding, so a
 *     prompt prefilled in chunks over the FP8 cache gives the same result as
 *     in one call (a NaN code inside a request's visible keys gives an
 *     unspecified result).  The scores multiply E4M3 operands: each query
 *     row is scaled by a power of two that puts its largest magnitude in
 *     [2^7, 2^8) and taken as two E4M3 terms, a = E4M3(y) and b = E4M3(y - a)
 *     (within 2^-8 |y| of y, about bf16 precision), against the key codes;
 *     the values multiply in fp16 (every E4M3 value is an fp16 value) with
 *     the probabilities rounded to fp16.
 *     ("Prefill Optimisation", section 3, prefix caching: the KV cache data
 *     type, e.g. FP8 E4M3, and its quantization scales are part of what the
 *     cached KV means; the pages fix nothing further, so the format and this
 *     encoding are the library's.)
 *   - Device pointers must be 16-byte aligned.
 *   - Ownership: the caller allocates and frees every buffer, the workspace
 *     included.  The library never allocates, frees or synchronises; all
 *     work is enqueued on the caller's stream (a cudaStream_t passed as
 *     void*, NULL = legacy default stream) and is asynchronous.
 *   - Errors: return codes, never exceptions or aborts.  Every argument is
 *     checked on the host before anything is launched; a failed check
 *     launches nothing.  Block ids read on the device are range-checked:
 *     an id outside [0, num_blocks) is skipped and recorded, and
 *     cpa_last_device_error reports it.
 *   - The caller guarantees that no two active tokens share a slot and that
 *     no active token's slot lies inside another request's cached range
 *     (shared prefix blocks are read-only).
 */
#ifndef CPA_H_
#define CPA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    CPA_SUCCESS = 0,
    CPA_ERR_INVALID_ARG = 1,     /* a host-side check failed; nothing launched */
    CPA_ERR_UNSUPPORTED = 2,     /* valid, but not built for this dtype / shape / device */
    CPA_ERR_CUDA = 3,            /* a CUDA call or launch failed */
    CPA_ERR_DEVICE_TIMEOUT = 4,  /* a bounded device-side wait ran out (kernel returned early) */
    CPA_ERR_BAD_BLOCK_ID = 5,    /* a block-table entry outside [0, num_blocks) was read */
    CPA_ERR_WORKSPACE = 6        /* workspace missing or smaller than the size query returned */
} cpa_status;

typedef enum { CPA_DTYPE_FP32 = 0, CPA_DTYPE_BF16 = 1 } cpa_dtype;

/* Representation of the K/V pools (cpa_params.kv_format). */
typedef enum {
    CPA_KV_SAME = 0,      /* the pools hold elements of cpa_params.dtype */
    CPA_KV_FP8_E4M3 = 1   /* the pools hold FP8 E4M3 codes with per-kv-head scales (BF16
                             dtype; chunked_prefill_attention also needs head_dim 128 and
                             num_heads_q / num_heads_kv at most 128, else CPA_ERR_UNSUPPORTED) */
} cpa_kv_format;

/* flags (cpa_params.flags) */
#define CPA_FLAG_FUSE_KV_WRITE 0x1u /* attention also writes the new K/V into the pool
                                       (the write of paged_kv_write, done in the
                                       attention kernel's prologue) */
#define CPA_FLAG_FORCE_SIMT 0x2u    /* BF16 only: use the CUDA-core kernel instead of the
                                       tensor-core kernel (cross-checking) */
#define CPA_FLAG_NO_SPLIT 0x4u      /* never split one query tile's keys across CTAs */
#define CPA_FLAG_TAIL_SPLIT 0x8u    /* tensor-core kernel, prefill batches: let the planner cut
                                       the last query tiles into pieces over several CTAs when
                                       its schedule model expects the last wave to end sooner
                                       (off by default: with the current kernel it measured no
                                       faster on 2048-token chunks and slower on long prompts) */
#define CPA_FLAG_TEST_STALL 0x100u  /* testing only: the tensor-core kernel withholds the
                                       copies of one K tile, so its consumers' bounded waits
                                       expire and the launch reports CPA_ERR_DEVICE_TIMEOUT
                                       (use with a small timeout_cycles) */

/* Varlen batch descriptor of one step ("Prefill Processing", Scheduler
 * Output and Attention Metadata).  Device arrays are read by the kernels;
 * the host mirrors are read by the host for checks and launch sizing and
 * must hold the same values as the device arrays. */
typedef struct {
    int32_t num_reqs;               /* requests in the step (>= 0) */
    int32_t max_blocks_per_seq;     /* columns of the block table (>= 1 when num_reqs > 0) */
    int32_t total_new_tokens;       /* T = sum of num_new_tokens */
    const int32_t *cached_seq_len;  /* device [num_reqs]: prior tokens in the pool (C_r) */
    const int32_t *num_new_tokens;  /* device [num_reqs]: active tokens (N_r >= 0) */
    const int32_t *cu_new_tokens;   /* device [num_reqs + 1]: prefix sums of N_r, cu[0] = 0 */
    const int32_t *block_table;     /* device [num_reqs, max_blocks_per_seq], row-major */
    const int32_t *h_cached_seq_len;/* host mirror of cached_seq_len */
    const int32_t *h_num_new_tokens;/* host mirror of num_new_tokens */
} cpa_batch;

/* Shape and options of one attention layer. */
typedef struct {
    int32_t num_heads_q;      /* H_q, a multiple of num_heads_kv */
    int32_t num_heads_kv;     /* H_kv */
    int32_t head_dim;         /* d: 64 or 128 */
    int32_t block_size;       /* tokens per cache block: 16, 32, 64 or 128 */
    int32_t num_blocks;       /* blocks in each pool */
    int32_t kv_segment_size;  /* 0 (library chooses) or 512, 1024, 2048, 4096; a multiple of
                                 block_size ("Prefill Processing", Kernel Interface).  The keys
                                 of single-tile requests (decodes) are walked in pieces of this
                                 size, combined by online-softmax merging.  When the batch has
                                 plenty of work a CTA takes 2, 4 or 8 consecutive pieces (up to
                                 8192 keys, while at least 1024 units remain); the result is the
                                 same up to rounding. */
    float scale;              /* softmax scale applied to q.k, finite and > 0 (usually 1/sqrt(d)) */
    int32_t dtype;            /* cpa_dtype */
    uint32_t flags;           /* CPA_FLAG_* */
    int64_t timeout_cycles;   /* bound of every device-side wait, in SM clock cycles;
                                 0 = library default (2e9, about one second) */
    float rope_theta;         /* 0: q and k_new are used as given (already position-encoded).
                                 > 0: rotary position embedding with this base is applied first:
                                 query and new key of active token i of request r are rotated at
                                 absolute position cached_seq_len[r] + i ("Prefill Optimisation",
                                 section 2: chunk tokens keep their absolute positions), each pair
                                 (x_c, x_{c+d/2}) turned by p * rope_theta^(-2c/d) (rotate-half
                                 form), in fp32 and rounded to the element type.  The rotated keys
                                 are what the K/V write stores.  The caller's q and k_new are not
                                 modified: the rotated keys live in the workspace (the
                                 tensor-core kernel with plain pools rotates the queries in
                                 shared memory in the same launch; the CUDA-core kernel and FP8
                                 pools take rotated query copies from a pre-pass). */
    int32_t kv_format;        /* cpa_kv_format; CPA_KV_SAME for plain pools */
    const float *k_scale;     /* CPA_KV_FP8_E4M3 only: device [H_kv], finite and > 0 (the caller's
                                 guarantee; 4-byte aligned, else CPA_ERR_INVALID_ARG); NULL otherwise */
    const float *v_scale;     /* likewise for the values */
} cpa_params;

/* Bytes of device workspace chunked_prefill_attention needs for this batch
 * on the current device.  The parts, each starting on a 256-byte boundary:
 *   - the split-KV partials of the requests whose keys are cut into pieces,
 *     and (CPA_FLAG_TAIL_SPLIT) of the query tiles cut into tail pieces.
 *     The plan depends on the device's SM count: how many of the last
 *     requests take the shorter pieces of the split plan's last wave, and
 *     the tail cut.  With no device present there is neither;
 *   - when rope_theta > 0 (plain pools): the rotated copy of k_new, and of
 *     q too where a pre-pass rotates it (the CUDA-core kernel, and the
 *     two-pipeline tensor-core kernel that block sizes up to 32 use);
 *   - with the FP8 cache: the two E4M3 planes of q ([2][T, H_q, d] bytes),
 *     its row scales ([T, H_q] x 4 bytes) and the codes of k_new and v_new
 *     ([T, H_kv, d] bytes each);
 *   - when the batch runs on the tensor-core kernel (BF16 with num_heads_q /
 *     num_heads_kv at most 128): that persistent kernel's work counter (a
 *     second one when the planner splits its CTAs into two groups), one
 *     counter per softmax warp of every tail-cut tile, and where the
 *     one-pipeline kernel rotates keys itself (rope_theta > 0, plain pools)
 *     the key rotation's 2 + ceil(T / 128) counters (4 bytes each, rounded
 *     up to 256 bytes).
 * 0 for an empty batch and for a CUDA-core batch with no split.  Reads only
 * host mirrors.  Returns 0 also when the arguments are invalid;
 * chunked_prefill_attention then reports the error. */
size_t chunked_prefill_workspace_size(const cpa_batch *batch, const cpa_params *params);

/* Write the K/V rows of every active token into their pool slots: token i of
 * request r goes to the slot of position cached_seq_len[r] + i
 * ("Prefill Processing", Key Concepts: active tokens write new KV to cache;
 * Attention Metadata: slot_mapping).  A byte-exact copy (with the FP8 cache:
 * the E4M3 codes of the rows, see the conventions above).  k_new/v_new are
 * read, k_cache/v_cache written in place.  Only the slots of active tokens
 * change. */
cpa_status paged_kv_write(const cpa_batch *batch, const cpa_params *params, const void *k_new,
                          const void *v_new, void *k_cache, void *v_cache, void *stream);

/* Attention of every active token over its request's cached K/V and,
 * causally, the request's active tokens ("Prefill Processing", How
 * Segmentation Works with KV Segments and Kernel Interface; "Prefill
 * Optimisation", section 2).  For token i of request r, query head h:
 *   out = sum_j softmax_j(scale * q . k_j) v_j over positions j <= C_r + i,
 * keys j < C_r read from the pool through the block table, keys j >= C_r
 * from k_new / v_new.  The cached keys are walked in kv_segment_size pieces
 * combined by online-softmax merging; the result is the same up to
 * rounding.  With CPA_FLAG_FUSE_KV_WRITE the new K/V rows are also written
 * into the pool (as paged_kv_write) in the same launch; without it the pools
 * are only read.
 * workspace: device memory of at least chunked_prefill_workspace_size()
 * bytes (may be NULL when that size is 0); its contents need not be
 * initialised and are overwritten (the work counter by an asynchronous
 * memset on `stream` before the launch), so two calls in flight at once
 * need two workspaces.  lse may be NULL. */
cpa_status chunked_prefill_attention(const cpa_batch *batch, const cpa_params *params, const void *q,
                                     const void *k_new, const void *v_new, void *k_cache,
                                     void *v_cache, void *out, float *lse, void *workspace,
                                     size_t workspace_bytes, void *stream);

/* Bytes of the static device array behind chunked_prefill_attention_no_alloc. */
#define CPA_NO_ALLOC_WORKSPACE_BYTES (32u << 20)

/* chunked_prefill_attention for callers that cannot allocate device memory.
 * (The pages have no counterpart: this is a calling convenience.)  Some
 * callers cannot call cudaMalloc and have no spare device buffer to lend as
 * workspace -- a plugin inside a host application that owns all device memory
 * through its own pool, or a serving loop that must not call cudaMalloc /
 * cudaFree because they can synchronise the device.  This call takes the same
 * arguments minus the workspace and allocates nothing: the whole workspace
 * that chunked_prefill_workspace_size reports -- split-KV and tail-piece
 * partials, the RoPE / FP8 pre-pass copies of the active rows, the work and
 * tail counters -- goes to one file-scope device array of
 * CPA_NO_ALLOC_WORKSPACE_BYTES that every GPU loading the library holds until
 * the process exits.  The pre-pass copies grow with the active tokens, so
 * RoPE and FP8 batches reach the limit at fewer tokens than plain ones.
 *   - With CPA_FLAG_TAIL_SPLIT, a batch whose workspace does not fit is run
 *     without tail pieces (as if the flag were clear: the same result up to
 *     the order of fp32 sums).  A batch that does not fit without them
 *     returns CPA_ERR_WORKSPACE and launches nothing.
 *   - All calls on a device share the array, which keeps the last call's
 *     contents; the call clears the counters itself (an asynchronous memset
 *     on `stream`) and writes every partial before reading it.  Calls that
 *     overlap on the GPU (e.g. on two streams at once) race on it: serialise
 *     them.
 *   - The first call on a device looks up the array's device address and
 *     caches it; make that first call before any stream capture.  After
 *     cudaDeviceReset the cached addresses are stale: reload the library.
 * Results are bit-identical to chunked_prefill_attention's on the same
 * inputs and flags (whenever the tail pieces fit). */
cpa_status chunked_prefill_attention_no_alloc(const cpa_batch *batch, const cpa_params *params,
                                              const void *q, const void *k_new, const void *v_new,
                                              void *k_cache, void *v_cache, void *out, float *lse,
                                              void *stream);

/* Wait for `stream`, then return and clear the first error recorded by a
 * kernel on the current device since the last call (CPA_SUCCESS if none):
 * CPA_ERR_DEVICE_TIMEOUT or CPA_ERR_BAD_BLOCK_ID.  CPA_ERR_CUDA if the
 * stream itself reports an error.  This call synchronises the stream.  The
 * library caches the error word's device address per device on first use;
 * after cudaDeviceReset that address is stale: reload the library. */
cpa_status cpa_last_device_error(void *stream);

/* Static description of a status code. */
const char *cpa_status_string(cpa_status status);

/* Library version, major * 10000 + minor * 100 + patch. */
int32_t cpa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* CPA_H_ */
