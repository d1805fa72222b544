// Internal launch interface between the C ABI (cb_api.cu) and the kernel translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace cb {

struct AppendArgs {
  const void* k_new;
  const void* v_new;
  void* k_pages;
  void* v_pages;
  const int32_t* block_table;
  const int32_t* cu_seqlens_q;
  const int32_t* kv_lens;
  int S, T, Hkv, D, bs, max_blocks, P;
  uint32_t* err;
};

struct AttnArgs {
  const void* q;
  void* out;
  float* lse;
  const int32_t* block_table;
  const int32_t* cu_seqlens_q;
  const int32_t* kv_lens;
  char* ws;
  uint32_t* err;
  int S, T, Hq, Hkv, G, D, bs, max_blocks, P;
  int KB;              // rows per TMA box on the page pool, decode pass: gcd(bs, 16)
  int KBp;             // rows per TMA box on the page pool, chunk pass: gcd(bs, 128)
  int decode_ctas;     // CTAs of the decode pass per KV-head group (<= CB_MAX_DECODE_CTAS)
  int decode_grid;     // decode-role CTAs of this attention launch (decode_ctas x head groups;
                       // 0 when the launch runs the chunk pass only)
  int decode_auto;     // 1: the planner picks how many of them work (decode / chunk balance)
  int prefill_ctas;    // persistent CTAs of the chunk pass (0 when the launch runs decode only)
  int window;          // > 0: query at position p sees keys (p - window, p]; 0: all <= p
  float scale_log2;    // softmax scale * log2(e)
};

// Block moves: copy (pool -> pool), offload (pool -> linear host buffer), restore (host ->
// pool).  Per pool (K, V) one block is block_bytes contiguous bytes.
enum BlockMoveMode { kMoveCopy = 0, kMoveOffload = 1, kMoveRestore = 2 };
struct BlockMoveArgs {
  const char* src[2];   // K, V: pool (copy, offload) or host buffer (restore)
  char* dst[2];         // K, V: pool (copy, restore) or host buffer (offload)
  const int32_t* src_idx;  // block ids read (copy, offload)
  const int32_t* dst_idx;  // block ids written (copy, restore)
  int n, P, mode;
  long long block_bytes;
  uint32_t* err;
};

// Id of the CUDA context the calling thread's next launch goes to (set by every API entry
// point before it launches; 0 if unknown).
unsigned long long launch_context_id();

cudaError_t launch_kv_append(const AppendArgs& a, cudaStream_t stream);
cudaError_t launch_block_move(const BlockMoveArgs& a, int sm_count, cudaStream_t stream);
cudaError_t launch_wait_selftest(uint32_t* err, uint64_t limit_ns, uint64_t* waited_ns,
                                 cudaStream_t stream);
cudaError_t launch_plan(const AttnArgs& a, cudaStream_t stream);
// The append of a step and the planner of its attention pass in one launch (CTA 0 plans, the
// other CTAs append).
cudaError_t launch_append_plan(const AppendArgs& ap, const AttnArgs& a, cudaStream_t stream);
// Tensor maps of the attention pass: Q, and the page pools as the decode pass reads them
// (box of a page run of all KV heads of a group) and as the chunk pass reads them (one head).
struct AttnMaps {
  CUtensorMap q, k_dec, v_dec, k_chunk, v_chunk;
};
// The attention kernel: a.decode_grid decode-role CTAs, then a.prefill_ctas chunk-role CTAs.
cudaError_t launch_attention(const AttnArgs& a, const AttnMaps& maps, cudaStream_t stream);

}  // namespace cb
