/*
 * libcb host runtime: the paged-KV block allocator and the continuous-batching scheduler that
 * turn a stream of requests into the per-step batch metadata the attention path consumes
 * (cu_seqlens_q, kv_lens, block_table), plus the copy-on-write block copies a step needs.
 *
 * Sources:
 *   - Block allocator: "LLM learning path 3.3 Batching & Memory Management", section "Code"
 *     (a free list, a reference count per physical block, fork shares every block, writing a
 *     token into a block whose count is above 1 first copies it) and section "PagedAttention:
 *     block tables" (copy-on-write as in fork(); only full blocks are shared).
 *   - Schedulers: transformers "Continuous batching architecture" doc, section "Scheduler"
 *     (token budget max_batch_tokens, cache budget = the pages that exist, request cap
 *     max_requests_per_batch; FIFO = active decodes, then active prefills, then waiting
 *     requests in arrival order; PrefillFirst completes split prefills before resuming decode)
 *     and its "Chunked prefill" paragraph (a prompt larger than the remaining budget is
 *     processed as far as it fits and continued on later steps); "LLM learning path 3.3",
 *     section "Chunked prefill" (one token per running decode first, then a chunk of a pending
 *     prefill).
 *
 * Everything here is host code: plain C structs and host pointers, no CUDA calls.  The objects
 * are not thread-safe; one owner drives them.  Errors return a cb_status (cb.h) and leave the
 * object unchanged; cb_last_error_message() describes them.
 */
#ifndef CB_SCHED_H_
#define CB_SCHED_H_

#include <stddef.h>
#include <stdint.h>

#include "cb.h"

#ifdef __cplusplus
extern "C" {
#endif

/* ------------------------------------------------------------------------------ allocator */

typedef struct cb_alloc cb_alloc;  /* opaque */

/*
 * cb_alloc_create -- a pool of `num_blocks` physical blocks of `block_size` (>= 4) tokens.
 * Free blocks form a stack: the next allocation takes the most recently freed block, and a new
 * pool hands out num_blocks-1, num_blocks-2, ... first.  `max_blocks_per_seq` bounds one
 * sequence's block table (the width of the block_table rows the scheduler writes).
 * *out receives the object (owned by the caller; release it with cb_alloc_destroy).
 */
cb_status cb_alloc_create(int32_t num_blocks, int32_t block_size, int32_t max_blocks_per_seq,
                          cb_alloc** out);
void cb_alloc_destroy(cb_alloc* a);

/* A new sequence `seq` holding n_tokens (>= 0) tokens: ceil(n_tokens / block_size) blocks,
 * each with reference count 1.  CB_ERR_INVALID_ARG if seq exists; CB_ERR_OUT_OF_RANGE if the
 * free blocks or max_blocks_per_seq do not suffice (nothing is allocated then). */
cb_status cb_alloc_add_seq(cb_alloc* a, int32_t seq, int32_t n_tokens);

/* Grow `seq` by n_tokens (>= 0).  Tokens that start a new block take a free block; if the
 * first token goes into a partly filled last block shared with another sequence (count > 1),
 * that block is first replaced by a fresh private copy: the pair (old, new) is written to
 * cow_src[0], cow_dst[0] and *n_cow = 1 (else 0); the caller copies the block's K/V data
 * (cb_copy_blocks in cb.h) before the step's append.  cow_src / cow_dst may be NULL when the
 * caller knows no copy can occur.  CB_ERR_OUT_OF_RANGE if the blocks do not suffice. */
cb_status cb_alloc_append(cb_alloc* a, int32_t seq, int32_t n_tokens, int32_t* cow_src,
                          int32_t* cow_dst, int32_t* n_cow);

/* Blocks that cb_alloc_append(seq, n_tokens) would take from the free list (0 for an unknown
 * seq it would create with cb_alloc_add_seq: then ceil(n_tokens / block_size)). */
int32_t cb_alloc_blocks_needed(const cb_alloc* a, int32_t seq, int32_t n_tokens);

/*
 * Prefix caching (transformers "Continuous batching architecture", sections "Prefix caching"
 * and "Eviction"; "LLM learning path 3.3", section "Prefix caching and RadixAttention",
 * hash-based blocks): each completed block of prompt tokens is identified by a 64-bit content
 * hash chained with the hash of every block before it (FNV-1a over the parent hash's 8 bytes
 * and the block's token ids, 4 bytes each, little-endian); a later prompt reuses the longest
 * chain of matching blocks (verified token by token) and skips their prefill.  A freed block
 * keeps its content and hash; it is reused by a match, or, once no block without cached
 * content is left, the most recently initialized free block is demoted (its hash dropped) and
 * handed out.  Off by default; switch it on before the first sequence.
 */
cb_status cb_alloc_set_prefix_caching(cb_alloc* a, int32_t enable);

/* A new sequence `seq` whose prompt has n_tokens (>= 1) token ids: it starts with the longest
 * cached chain of full blocks matching the prompt, at most (n_tokens - 1) / block_size blocks
 * so that at least the last prompt token is computed; *n_cached = the tokens it holds (a
 * multiple of block_size; 0 without a match or with caching off). */
cb_status cb_alloc_add_seq_cached(cb_alloc* a, int32_t seq, const int32_t* tokens,
                                  int32_t n_tokens, int32_t* n_cached);

/* Register the content hashes of seq's full blocks within its first n_tokens positions, whose
 * token ids are tokens[0 .. n_tokens) (n_tokens <= the tokens seq holds).  A block whose
 * content is already cached in another block stays unregistered. */
cb_status cb_alloc_hash_blocks(cb_alloc* a, int32_t seq, const int32_t* tokens, int32_t n_tokens);

/* Blocks with cached content (in use or free). */
int32_t cb_alloc_num_cached(const cb_alloc* a);

/* `child` shares every block of `parent` (each count + 1) and its length. */
cb_status cb_alloc_fork(cb_alloc* a, int32_t parent, int32_t child);

/* Drop `seq`: every block's count - 1; blocks reaching 0 return to the free stack in table
 * order (so the last block of the table is the next one handed out). */
cb_status cb_alloc_free_seq(cb_alloc* a, int32_t seq);

int32_t cb_alloc_num_free(const cb_alloc* a);
int32_t cb_alloc_ref_count(const cb_alloc* a, int32_t block);  /* -1 if out of range */

/* Copy seq's block table (up to `cap` entries) and return its block count and token count. */
cb_status cb_alloc_table(const cb_alloc* a, int32_t seq, int32_t* blocks, int32_t cap,
                         int32_t* n_blocks, int32_t* n_tokens);

/* ------------------------------------------------------------------------------ scheduler */

typedef enum { CB_SCHED_FIFO = 0, CB_SCHED_PREFILL_FIRST = 1 } cb_sched_policy;

typedef struct {
  int32_t max_batch_tokens;        /* token budget: query tokens per step (>= 1) */
  int32_t max_requests_per_batch;  /* request cap: sequences per step (>= 1) */
  int32_t policy;                  /* cb_sched_policy */
} cb_sched_config;

typedef struct cb_sched cb_sched;  /* opaque; uses (does not own) a cb_alloc */

cb_status cb_sched_create(cb_alloc* alloc, const cb_sched_config* cfg, cb_sched** out);
void cb_sched_destroy(cb_sched* s);

/* Queue a request: prompt_len >= 1 prompt tokens, then max_new_tokens >= 1 generated tokens
 * (the first comes from the last prompt position, each later one from a one-token decode
 * step).  The request's sequence id in the allocator is `id`.  CB_ERR_INVALID_ARG for a
 * duplicate id or bad lengths; CB_ERR_UNSUPPORTED if prompt_len + max_new_tokens - 1 tokens
 * cannot fit max_blocks_per_seq. */
cb_status cb_sched_add_request(cb_sched* s, int32_t id, int32_t prompt_len,
                               int32_t max_new_tokens);

/* As cb_sched_add_request, with the prompt's token ids (copied): with prefix caching on in
 * the allocator, the request's first admission reuses the cached blocks of its longest cached
 * prompt prefix and prefills only the rest, and its completed prompt blocks are cached. */
cb_status cb_sched_add_request_tokens(cb_sched* s, int32_t id, const int32_t* tokens,
                                      int32_t prompt_len, int32_t max_new_tokens);

/* Parallel sampling: a new request `child` that continues from `parent` (which must be
 * decoding: its prompt done) with the same tokens so far, sharing all of parent's blocks
 * (cb_alloc_fork), and produces max_new_tokens in all counting the ones parent has produced.
 * The first step that writes into the shared partly filled last block copies it. */
cb_status cb_sched_fork_request(cb_sched* s, int32_t parent, int32_t child,
                                int32_t max_new_tokens);

/*
 * One step's batch, written by cb_sched_step into caller-owned host arrays:
 *   seq_ids       [cap_seqs]                request id of each scheduled sequence, batch order
 *   cu_seqlens_q  [cap_seqs + 1]            prefix sum of the sequences' query lengths
 *   kv_lens       [cap_seqs]                keys visible after this step's append
 *   block_table   [cap_seqs * max_blocks]   row-major, rows padded with -1
 *   cow_src/dst   [cap_cow]                 block copies to run before the append
 * Sequences are ordered as the policy admits them (FIFO: decodes, then continuing prefills,
 * then new requests).  cap_seqs >= max_requests_per_batch and cap_cow >= the same are enough.
 */
typedef struct {
  int32_t num_seqs, num_tokens, num_cow;
  int32_t num_decode;    /* sequences with q_len == 1 that are decoding */
  int32_t num_finished;  /* requests retired at the start of this step */
  int32_t num_cached;    /* prompt tokens reused from the prefix cache by this step's admissions */
  int32_t cap_seqs, cap_cow, max_blocks;
  int32_t* seq_ids;
  int32_t* cu_seqlens_q;
  int32_t* kv_lens;
  int32_t* block_table;
  int32_t* cow_src;
  int32_t* cow_dst;
} cb_batch;

/*
 * Build the next step: retire requests that have produced max_new_tokens (their blocks are
 * freed), then admit work in policy order under the three budgets, allocating (and, for a
 * shared last block, copy-on-write) the slots of every token admitted, and advance each
 * admitted request as if the forward pass ran (prefill progress, one generated token per
 * decode step and per completed prompt).  A step with no admissible work returns
 * num_seqs = 0.  CB_ERR_INVALID_ARG if the arrays are missing or too small.
 */
cb_status cb_sched_step(cb_sched* s, cb_batch* out);

/* Requests not yet retired (waiting, prefilling or decoding). */
int32_t cb_sched_num_active(const cb_sched* s);

#ifdef __cplusplus
}
#endif

#endif /* CB_SCHED_H_ */
