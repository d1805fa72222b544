/*
 * cb.h -- C ABI of libcb: paged KV-append and ragged paged attention on one GB300 (sm_103a).
 *
 * The problem these calls solve is the attention step of a continuous-batching engine:
 * every token of one forward pass (decode tokens and chunked-prefill chunks alike) is packed
 * into a single ragged token axis delimited by cu_seqlens_q, and each sequence's keys and
 * values live in fixed-size blocks of a paged KV cache reached through a per-sequence block
 * table ("LLM learning path 3.3 Batching & Memory Management", sections "Continuous
 * (iteration-level) batching", "PagedAttention: block tables" and "Chunked prefill";
 * "Continuous batching in transformers", section "The paged cache, its two reserved blocks,
 * and the block-size trade"; continuous-batching architecture doc, section "Memory
 * management").
 *
 * Conventions shared by every call
 *   - Every pointer argument is DEVICE memory owned by the caller, C-contiguous, and must stay
 *     valid until the work queued on `stream` has finished.  The library allocates nothing per
 *     call; its only device state is one 32-bit error word per device.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream).  All
 *     calls are asynchronous on that stream unless stated otherwise.
 *   - bf16 tensors are passed as void*; 16-byte alignment is required for every tensor.
 *   - Host-side checks (null pointers, sizes, alignment, unsupported shapes) are made before
 *     anything is queued; a failing check returns an error and queues nothing.
 *     cb_last_error_message() then describes it.
 *   - Device-side checks (metadata that only the GPU reads: block ids, lengths) never trap:
 *     the kernel skips the offending access, its outputs for that sequence are unspecified,
 *     and it records the fault in the device error word; cb_get_device_error() reports it.
 *
 * Shapes (S sequences, T packed tokens, Hq query heads, Hkv KV heads, D head dim,
 *         P pages-blocks in the pool, bs block size, MB max blocks per sequence)
 *   q, out            bf16  [T, Hq, D]
 *   k_new, v_new      bf16  [T, Hkv, D]
 *   k_pages, v_pages  bf16  [P, bs, Hkv, D]   token-major: row (block*bs + offset) of the
 *                                             flattened [P*bs, Hkv, D] tensor is one token
 *   block_table       int32 [S, MB]           entry j = physical block holding tokens
 *                                             [j*bs, (j+1)*bs) of the sequence; unused
 *                                             entries are never read
 *   cu_seqlens_q      int32 [S+1]             cu[0] = 0, non-decreasing, cu[S] <= T; rows
 *                                             cu[S] .. T-1 of q/out/k_new/v_new are padding
 *                                             (never read, never written), so a caller can
 *                                             keep fixed buffer shapes (e.g. in a CUDA graph
 *                                             captured for a padded shape)
 *   kv_lens           int32 [S]               keys visible to sequence s INCLUDING this
 *                                             step's appended tokens (kv_len >= q_len)
 *   lse               fp32  [T, Hq]           optional natural-log softmax normaliser
 * Query token i of sequence s sits at absolute position ctx_s + i, ctx_s = kv_len_s - q_len_s,
 * and attends to keys 0 .. ctx_s + i of its own sequence (causal mask offset by the prior
 * context); query head h reads KV head h / (Hq / Hkv).
 */
#ifndef CB_H_
#define CB_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  CB_OK = 0,
  CB_ERR_INVALID_ARG = 1,   /* null pointer, bad size, misaligned tensor, block_size < 4 */
  CB_ERR_UNSUPPORTED = 2,   /* valid request outside what the kernels implement (e.g. D) */
  CB_ERR_OUT_OF_RANGE = 3,  /* device saw metadata outside the pool / table / lengths     */
  CB_ERR_TIMEOUT = 4,       /* a device-side wait gave up (bounded waits, no hang)        */
  CB_ERR_CUDA = 5           /* a CUDA runtime or driver call failed                       */
} cb_status;

typedef struct {
  int32_t num_seqs;            /* S  >= 0                                           */
  int32_t num_tokens;          /* T  >= cu_seqlens_q[S]: rows of the token tensors  */
  int32_t num_q_heads;         /* Hq >= 1, a multiple of Hkv, Hq / Hkv <= 16        */
  int32_t num_kv_heads;        /* Hkv >= 1                                          */
  int32_t head_dim;            /* D: 64 or 128                                      */
  int32_t num_pages;           /* P  >= 1 blocks in the pool (P * bs < 2^31)        */
  int32_t max_blocks_per_seq;  /* MB >= 1 columns of block_table                    */
} cb_dims;

/*
 * cb_kv_append -- scatter this step's K/V rows into their cache slots.
 *
 * Token i of sequence s (packed row cu[s] + i) has position pos = ctx_s + i and is copied,
 * bit for bit, to flattened page row block_table[s][pos / bs] * bs + pos % bs, for K and for V
 * ("LLM learning path 3.3", section "PagedAttention: block tables": token position p lives
 * in block table[p // bs] at offset p % bs; architecture doc, section "Memory management":
 * the kernels write the blocks a request's table names).  Only those T*Hkv*D elements of
 * each pool are written.
 * Undefined when two tokens map to the same slot or when a written block is shared with
 * another sequence's visible keys (copy-on-write is the block manager's job).
 * Device errors (CB_ERR_OUT_OF_RANGE via cb_get_device_error): kv_len < q_len,
 * pos / bs >= MB, block id outside [0, P), malformed cu_seqlens_q.  The row is skipped.
 */
cb_status cb_kv_append(const void* k_new, const void* v_new, void* k_pages, void* v_pages,
                       const int32_t* block_table, const int32_t* cu_seqlens_q,
                       const int32_t* kv_lens, int32_t block_size, const cb_dims* dims,
                       void* stream);

/*
 * cb_attention_workspace_size -- bytes of device scratch cb_ragged_paged_attention needs.
 * Pure host arithmetic on num_seqs, num_tokens, num_q_heads, num_kv_heads and head_dim (the
 * other fields of dims do not change the size and are not checked here); 0 when dims is NULL
 * or those fields are invalid.  The workspace holds the batch plan (including the
 * longest-first order of the chunk work, one int32 per 128 query tokens plus one per
 * sequence) and the fp32 partial results of split decode sequences; it grows with num_seqs,
 * num_tokens, num_q_heads and head_dim.
 */
size_t cb_attention_workspace_size(const cb_dims* dims);

/*
 * cb_ragged_paged_attention -- one attention forward pass over the ragged batch.
 *
 * out[t, h, :] = sum_j softmax_j(scale * q[t,h,:] . K_s[j,g,:]) * V_s[j,g,:] over the keys
 * j <= ctx_s + i of t's own sequence s, with K_s/V_s gathered through block_table and
 * g = h / (Hq/Hkv).  Inputs are bf16, accumulation is fp32, out is rounded to bf16.
 * Sources: the packed token axis whose tokens attend only within their own sequence is
 * "LLM learning path 3.3", section "Continuous (iteration-level) batching", and the "first
 * principles" summary (attention masks that keep the packed sequences apart); the keys of a
 * sequence are read through its block table ("LLM learning path 3.3", section "PagedAttention:
 * block tables"; architecture doc, section "Memory management"); a chunk's query i sees the
 * prior context plus the chunk's queries up to i ("LLM learning path 3.3", section "Chunked
 * prefill"); decode tokens read the whole cached context every step (same page, section
 * "Common pitfalls / misconceptions").  The query-head to KV-head mapping h / (Hq/Hkv) is not
 * stated on the pages; it is the contiguous grouping of grouped-query attention.
 * If lse is not NULL it receives the natural log of each row's softmax normaliser.
 * Sequences with q_len == 0 are skipped; the pass reads the pages after cb_kv_append wrote
 * them (kv_lens include the appended tokens).  out must not alias q or the pages.
 * workspace: device memory of at least cb_attention_workspace_size(dims) bytes,
 * 256-byte aligned, owned by the caller and not used by other work while this call runs.
 * Device errors as for cb_kv_append, plus CB_ERR_TIMEOUT if a bounded wait expired.
 */
cb_status cb_ragged_paged_attention(const void* q, const void* k_pages, const void* v_pages,
                                    const int32_t* block_table, const int32_t* cu_seqlens_q,
                                    const int32_t* kv_lens, int32_t block_size, float scale,
                                    void* out, float* lse, void* workspace,
                                    size_t workspace_bytes, const cb_dims* dims, void* stream);

/*
 * Options of cb_ragged_paged_attention_ex.  Zero-initialise for defaults.
 *   decode_ctas   number of CTAs the decode pass spreads its key tiles over (0 = one per SM;
 *                 1 forces every decode sequence into a single unsplit pass).  Results for
 *                 different values agree within rounding; at most CB_MAX_DECODE_CTAS.
 *   flags         CB_OPT_SERIAL: run the decode pass and then the chunk pass as two launches
 *                 instead of together in one.
 *   phase_events  NULL, or an array of CB_NUM_PHASE_EVENTS cudaEvent_t (created by the
 *                 caller, passed as void*), all recorded on `stream`: [0] before the planner,
 *                 [1] after it, [2] after the decode pass (which also merges split sequences),
 *                 [3] / [4] before / after the chunk pass.  With both passes in one launch
 *                 (the default) [1] and [3] mark that launch's start and [2] and [4] its end;
 *                 cb_pass_timestamps gives the two passes' own spans inside it.
 *   window        0: full causal attention.  W > 0: sliding-window attention, for models with
 *                 sliding-window layer groups (named in "Continuous batching in transformers",
 *                 paged-cache section, which does not define the mask; this is the common
 *                 definition): the query at absolute position p sees keys j with
 *                 p - W < j <= p, i.e. itself and the W - 1 keys before it.  Keys older than
 *                 the window are not read (neither pass streams them).
 *
 * Concurrency: everything runs on `stream`.  The decode pass (HBM-bound) and the chunk pass
 * (tensor-bound) share one kernel launch: its first CTAs are the decode CTAs, which the block
 * scheduler places first, and the chunk CTAs take the SMs the planner leaves free and then the
 * SMs the decode CTAs free as they finish.
 */
#define CB_NUM_PHASE_EVENTS 5
#define CB_OPT_SERIAL 1
typedef struct {
  int32_t decode_ctas;
  int32_t flags;
  void* const* phase_events;
  int32_t window;        /* > 0: sliding-window attention over the last `window` keys */
  int32_t reserved32;
  int64_t reserved[3];
} cb_options;

#define CB_MAX_DECODE_CTAS 512

cb_status cb_ragged_paged_attention_ex(const void* q, const void* k_pages, const void* v_pages,
                                       const int32_t* block_table, const int32_t* cu_seqlens_q,
                                       const int32_t* kv_lens, int32_t block_size, float scale,
                                       void* out, float* lse, void* workspace,
                                       size_t workspace_bytes, const cb_dims* dims,
                                       const cb_options* options, void* stream);

/*
 * cb_append_attention -- cb_kv_append followed by cb_ragged_paged_attention_ex in one call, with
 * the same arguments and the same results (bit for bit).  The attention pass's planner reads
 * only the metadata, so one launch does both the append and the planning (one CTA plans while
 * the others append), and the attention kernel follows: two launches per step, both on
 * `stream`.  Phase events as in cb_ragged_paged_attention_ex, [0] before and [1] after the
 * append + planner launch.  k_new / v_new as in cb_kv_append; every other argument as in
 * cb_ragged_paged_attention_ex (with CB_OPT_SERIAL the append, the planner, the decode pass
 * and the chunk pass are four launches, one after the other).
 */
cb_status cb_append_attention(const void* k_new, const void* v_new, void* k_pages, void* v_pages,
                              const void* q, const int32_t* block_table,
                              const int32_t* cu_seqlens_q, const int32_t* kv_lens,
                              int32_t block_size, float scale, void* out, float* lse,
                              void* workspace, size_t workspace_bytes, const cb_dims* dims,
                              const cb_options* options, void* stream);

/*
 * cb_pass_timestamps -- device time stamps (%globaltimer, ns) of the two passes of the last
 * attention call that used `workspace`: ts_ns[0] / [1] the first start and the last end of the
 * decode CTAs that had work, ts_ns[2] / [3] the same for the chunk CTAs (the end is the last
 * chunk item's output written); 0 / 0 for a pass that had no work.  Waits for `stream`, then
 * reads 64 bytes of the workspace.  For profiling: inside one launch CUDA events cannot separate
 * the passes.  Errors: CB_ERR_INVALID_ARG (NULL pointer), CB_ERR_CUDA.
 */
cb_status cb_pass_timestamps(const void* workspace, uint64_t* ts_ns, void* stream);

/*
 * cb_ragged_paged_attention_noalloc -- cb_ragged_paged_attention without a workspace argument.
 * (An addition of this library with no counterpart in the pages that describe the method.)
 *
 * For callers that cannot allocate device memory: code that is handed only its input and
 * output buffers by a host framework with no scratch allocator, or a steady-state serving loop
 * that must not call cudaMalloc (which can synchronise the whole device).  The scratch comes
 * from one fixed device array of CB_NOALLOC_SCRATCH_BYTES inside the library, which every GPU
 * that loads the library holds until the process exits.  The call allocates nothing.
 *   - The first call on each device looks up the array's device address (with that device
 *     current) and keeps it with the id of the device's current context; a call made in a
 *     later context of the device (after cudaDeviceReset, say) looks it up again.  Make the
 *     first call on a device before any stream capture.
 *   - All calls share the one array: calls that overlap on the GPU (other streams, or host
 *     threads without ordering between them) race on it.  Each call rewrites every scratch
 *     byte it later reads, so contents left by the previous call do no harm.
 *   - A batch whose scratch need, cb_attention_workspace_size(dims), exceeds
 *     CB_NOALLOC_SCRATCH_BYTES is rejected with CB_ERR_UNSUPPORTED before anything is queued.
 *   - cb_pass_timestamps is not available for these calls: it reads its time stamps from the
 *     caller's workspace, and this entry point has none.
 * Arguments, results and errors are otherwise those of cb_ragged_paged_attention.
 */
#define CB_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)
cb_status cb_ragged_paged_attention_noalloc(const void* q, const void* k_pages,
                                            const void* v_pages, const int32_t* block_table,
                                            const int32_t* cu_seqlens_q, const int32_t* kv_lens,
                                            int32_t block_size, float scale, void* out, float* lse,
                                            const cb_dims* dims, void* stream);

/*
 * cb_copy_blocks -- copy whole KV blocks inside the page pools: for each i < n, block dst[i]
 * of k_pages and of v_pages receives the content of block src[i] (bs * Hkv * D bf16 each).
 * This is the data half of copy-on-write ("LLM learning path 3.3 Batching & Memory
 * Management", section "PagedAttention: block tables": a sequence about to write into a block
 * whose reference count is above 1 first copies it; section "Code": the real engine copies the
 * KV data too); the block allocator (cb_sched.h) decides the pairs.
 *   src, dst  device int32 [n]; k_pages, v_pages as in cb_kv_append (16-byte aligned).
 *   dims      num_kv_heads, head_dim and num_pages are used; the other fields are ignored.
 * Asynchronous on `stream`.  Pairs must not overlap (a block both read and written) — then
 * the result is undefined.  A pair with a block id outside [0, num_pages) is skipped and
 * reported through cb_get_device_error (CB_ERR_OUT_OF_RANGE); src == dst is a no-op.
 */
cb_status cb_copy_blocks(void* k_pages, void* v_pages, const int32_t* src, const int32_t* dst,
                         int32_t n, int32_t block_size, const cb_dims* dims, void* stream);

/*
 * cb_kv_offload -- gather blocks[i] (i < n) of both pools into host_k and host_v, each laid
 * out [n, bs, Hkv, D] bf16 (block i of the list at offset i * bs * Hkv * D); cb_kv_restore
 * is the inverse scatter.  The batched copy of a request's blocks to a CPU tier and back
 * (transformers "Continuous batching architecture", section "Memory management": offloaded
 * requests' blocks go to CPU memory in one batched copy and come back the same way).
 *   blocks           device int32 [n], ids in [0, num_pages)
 *   host_k, host_v   host memory the device can address (pinned: cudaHostAlloc or
 *                    cudaHostRegister), 16-byte aligned; owned by the caller, who must not
 *                    touch it until the work on `stream` has completed.
 * The kernel moves the bytes itself over the CPU-GPU link (no staging buffer, one launch for
 * any number of blocks).  Out-of-range ids are skipped and reported as for cb_copy_blocks.
 */
cb_status cb_kv_offload(const void* k_pages, const void* v_pages, const int32_t* blocks,
                        int32_t n, int32_t block_size, const cb_dims* dims, void* host_k,
                        void* host_v, void* stream);
cb_status cb_kv_restore(void* k_pages, void* v_pages, const int32_t* blocks, int32_t n,
                        int32_t block_size, const cb_dims* dims, const void* host_k,
                        const void* host_v, void* stream);

/*
 * cb_get_device_error -- synchronise `stream`, then read and clear the current device's error
 * word.  Returns CB_OK, CB_ERR_OUT_OF_RANGE, CB_ERR_TIMEOUT (reported first when both were
 * seen) or CB_ERR_CUDA if the synchronisation itself failed.
 */
cb_status cb_get_device_error(void* stream);

/*
 * cb_selftest_wait_timeout -- exercise the failure path every kernel of the library shares,
 * without a fault: one GPU thread waits on an mbarrier phase that nothing completes; after
 * limit_us (1 .. 100000) microseconds of %globaltimer it gives up, records CB_ERR_TIMEOUT in
 * the device error word (read it with cb_get_device_error) and returns, leaving the context
 * usable.  The kernels' own waits give up the same way after 1 s.  waited_ns: NULL or device
 * memory for one uint64, the time the wait lasted.  No counterpart on the pages (a test hook).
 */
cb_status cb_selftest_wait_timeout(int32_t limit_us, unsigned long long* waited_ns, void* stream);

/* Static English name of a status code (never NULL). */
const char* cb_status_string(cb_status status);

/* Description of the last host-side error on the calling thread ("" if none). */
const char* cb_last_error_message(void);

/* Library version, major * 10000 + minor * 100 + patch. */
int32_t cb_version(void);

#ifdef __cplusplus
}
#endif

#endif /* CB_H_ */
