// cb_ragged_paged_attention_noalloc: the attention pass with its scratch memory taken from a
// fixed array that lives inside the library, so the caller never allocates device memory.
//
// Who needs it: some callers are given only their input and output buffers and have no way
// to obtain scratch memory -- a host framework that exposes no device allocator to its plugins,
// or a serving loop that must not call cudaMalloc once it is running (cudaMalloc can
// synchronise the device and stall the other streams).  They cannot provide the `workspace`
// argument of cb_ragged_paged_attention, so this entry point supplies it from a static device
// array instead.
//
// The array is a file-scope __device__ object of kNoAllocScratchBytes; every GPU that loads the
// library holds it until the process exits.  Host code cannot use the array's name as a device
// address, so on the first call on each device (with that device current) the entry point asks
// the runtime for the address with cudaGetSymbolAddress and remembers it; that first call
// should therefore be made before any stream capture.  All calls share the one array: calls
// that overlap on the GPU (different streams, or different host threads without ordering)
// race on it.  Every byte the attention pass reads from the scratch is written earlier in the
// same call (the planner rewrites the plan and resets its work counter each time), so stale
// contents from the previous call are harmless.
#include <cstdio>
#include <mutex>

#include "cb_common.cuh"

namespace cb {
cb_status set_last_error(cb_status st, const char* msg);
}

namespace {

constexpr size_t kNoAllocScratchBytes = CB_NOALLOC_SCRATCH_BYTES;
static_assert(kNoAllocScratchBytes % 256 == 0, "scratch size must keep 256-byte alignment");

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices] = {};
std::mutex g_scratch_mu;

}  // namespace

extern "C" cb_status cb_ragged_paged_attention_noalloc(
    const void* q, const void* k_pages, const void* v_pages, const int32_t* block_table,
    const int32_t* cu_seqlens_q, const int32_t* kv_lens, int32_t block_size, float scale,
    void* out, float* lse, const cb_dims* dims, void* stream) {
  const size_t need = cb_attention_workspace_size(dims, block_size);
  if (need == 0) {
    // invalid dims or block size: let the regular entry point produce the detailed message
    return cb_ragged_paged_attention(q, k_pages, v_pages, block_table, cu_seqlens_q, kv_lens,
                                     block_size, scale, out, lse, nullptr, 0, dims, stream);
  }
  char msg[256];
  if (need > kNoAllocScratchBytes) {
    snprintf(msg, sizeof(msg),
             "this batch needs %zu bytes of scratch; the built-in scratch of "
             "cb_ragged_paged_attention_noalloc holds %zu (use cb_ragged_paged_attention "
             "with a caller-provided workspace)",
             need, kNoAllocScratchBytes);
    return cb::set_last_error(CB_ERR_UNSUPPORTED, msg);
  }
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    snprintf(msg, sizeof(msg), "cudaGetDevice: %s", cudaGetErrorString(e));
    return cb::set_last_error(CB_ERR_CUDA, msg);
  }
  if (dev < 0 || dev >= kMaxDevices) return cb::set_last_error(CB_ERR_UNSUPPORTED, "device id");
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (g_scratch_ptr[dev] == nullptr) {
      // One-time set-up on this device: the array's device address (host code only knows a
      // host-side stand-in for the symbol, which must never be handed to a kernel).
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
      if (e != cudaSuccess || p == nullptr) {
        snprintf(msg, sizeof(msg), "cudaGetSymbolAddress(scratch): %s", cudaGetErrorString(e));
        return cb::set_last_error(CB_ERR_CUDA, msg);
      }
      g_scratch_ptr[dev] = p;
    }
    scratch = g_scratch_ptr[dev];
  }
  return cb_ragged_paged_attention(q, k_pages, v_pages, block_table, cu_seqlens_q, kv_lens,
                                   block_size, scale, out, lse, scratch, kNoAllocScratchBytes,
                                   dims, stream);
}
