/*
 * cpa_engine.h -- C ABI of the host-side serving harness in libcpa.so: the
 * per-step decisions an engine makes before each chunked_prefill_attention
 * call (which requests run, how many tokens each, and their block tables).
 * Pure host code: no device memory, no CUDA calls.
 *
 * What it does (page title, section):
 *   - Greedy token budget ("Chunked Prefill"; "Prefill Optimisation",
 *     section 2, Mechanics of chunked scheduling): every running decode
 *     claims one token of the step's budget first; the rest goes to prompt
 *     chunks in arrival order, each at most chunk_size tokens.
 *   - Incremental block allocation ("Prefill Processing", Block
 *     Allocation): after a request is given num_new tokens it holds
 *     cdiv(num_computed + num_new, block_size) blocks; cached prefix blocks
 *     are claimed first, then fresh ones.  Block 0 is the null block: it is
 *     never handed out, and every block-table column past a request's blocks
 *     holds 0.
 *   - Prefix hash chain ("Prefill Optimisation", section 3, vLLM block hash
 *     chain): the hash of a full block covers its parent block's hash, its
 *     ordered token ids and the cache scope; a new request reuses its
 *     prompt's leading full blocks while their hashes are cached
 *     (full-block-only), leaving at least one prompt token to compute.
 *
 * Choices the pages leave open, fixed here:
 *   - block hash: 64-bit FNV-1a over the little-endian bytes of (parent
 *     hash, scope_key, the block's token ids as int32); the first block's
 *     parent is 0;
 *   - free blocks form a queue: allocation takes the front; when a request
 *     finishes, its blocks whose reference count drops to 0 go to the back,
 *     last block first, keeping their cached hash until they are taken for
 *     new data; a prefix hit on a free cached block takes it out of the queue;
 *   - a request that cannot get its blocks in a step is skipped in that step
 *     (no preemption);
 *   - after a step, the blocks a request completed are hashed and entered
 *     into the cache unless that hash is already cached; a request whose
 *     prompt is complete appends the caller's sampled token each step and
 *     finishes once it has max_new_tokens outputs, freeing its blocks.
 *
 * Ownership: the engine owns its state and the arrays a plan points to;
 * they stay valid until the next cpa_engine_schedule or cpa_engine_destroy.
 * Errors are status codes (cpa_status), never aborts.  Not thread-safe: one
 * thread drives an engine.
 */
#ifndef CPA_ENGINE_H_
#define CPA_ENGINE_H_

#include <stdint.h>

#include "cpa.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct cpa_engine cpa_engine;  /* opaque */

typedef struct {
    int32_t num_blocks;          /* blocks in the pool, block 0 included (>= 2) */
    int32_t block_size;          /* tokens per block (>= 1) */
    int32_t max_blocks_per_seq;  /* block-table columns (>= 1) */
    int32_t max_batched_tokens;  /* per-step token budget (>= 1) */
    int32_t chunk_size;          /* largest prompt chunk in one step (>= 1) */
    uint64_t scope_key;          /* cache scope (model, adapter, configuration, tenant), in every hash */
} cpa_engine_config;

/* One step's batch, in host memory owned by the engine.  Requests appear
 * decodes first, then prompt chunks, each group in arrival order; the arrays
 * match cpa_batch's host mirrors and device arrays row for row. */
typedef struct {
    int32_t num_reqs;
    int32_t max_blocks_per_seq;
    int32_t total_new_tokens;
    const int64_t *request_ids;     /* [num_reqs] */
    const int32_t *cached_seq_len;  /* [num_reqs] tokens already in the cache */
    const int32_t *num_new_tokens;  /* [num_reqs] tokens computed this step */
    const int32_t *cu_new_tokens;   /* [num_reqs + 1] prefix sums */
    const int32_t *block_table;     /* [num_reqs * max_blocks_per_seq], 0 past each request's blocks */
    const int32_t *token_ids;       /* [total_new_tokens] the tokens computed this step, packed like q */
} cpa_step_plan;

/* CPA_ERR_INVALID_ARG for a bad configuration; *out is NULL on failure. */
cpa_status cpa_engine_create(const cpa_engine_config *config, cpa_engine **out);

void cpa_engine_destroy(cpa_engine *engine);

/* Queue a request (arrival order is call order).  prompt: prompt_len >= 1
 * token ids, copied.  CPA_ERR_INVALID_ARG for a bad length, max_new_tokens
 * < 1 or a request id already known to the engine. */
cpa_status cpa_engine_add_request(cpa_engine *engine, int64_t request_id, const int32_t *prompt,
                                  int32_t prompt_len, int32_t max_new_tokens);

/* Decide the next step and allocate its blocks; fills *plan (num_reqs 0 when
 * nothing can run).  Call cpa_engine_commit before the next schedule. */
cpa_status cpa_engine_schedule(cpa_engine *engine, cpa_step_plan *plan);

/* The last scheduled step has run: advance every scheduled request, cache
 * its completed full blocks, append sampled_tokens[i] (one per plan row,
 * used for rows whose prompt is now complete) and retire finished requests.
 * CPA_ERR_INVALID_ARG if no step is pending or sampled_tokens is NULL while
 * the plan has rows. */
cpa_status cpa_engine_commit(cpa_engine *engine, const int32_t *sampled_tokens);

int32_t cpa_engine_num_free_blocks(const cpa_engine *engine);  /* in the free queue */
int32_t cpa_engine_num_unfinished(const cpa_engine *engine);   /* requests not yet finished */

/* Cached prefix tokens of a queued request that has not started yet, as a
 * prefix hit would claim them now (0 if none or unknown). */
int32_t cpa_engine_prefix_hit_tokens(const cpa_engine *engine, int64_t request_id);

#ifdef __cplusplus
}
#endif

#endif /* CPA_ENGINE_H_ */
