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
// the runtime for the address with cudaGetSymbolAddress and remembers it together with the id
// of the context it belongs to; a call in another context (the device's context was destroyed
// and made again, e.g. after cudaDeviceReset) looks the address up again.  That first call
// should therefore be made before any stream capture.  All calls share the one array: calls
// that overlap on the GPU (different streams, or different host threads without ordering)
// race on it.  Every byte the attention pass reads from the scratch is written earlier in the
// same call (the planner rewrites the plan, resets its work counter and the merge counters each
// time), so stale contents from the previous call are harmless.
#include <cstdio>
#include <mutex>

#include "cb_common.cuh"

namespace cb {
cb_status set_last_error(cb_status st, const char* msg);
cb_status current_context_id(unsigned long long* id);
}

namespace {

constexpr size_t kNoAllocScratchBytes = CB_NOALLOC_SCRATCH_BYTES;
static_assert(kNoAllocScratchBytes % 256 == 0, "scratch size must keep 256-byte alignment");

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
struct ScratchAddr {
  unsigned long long ctx_id = 0;  // context the address belongs to (0: not looked up)
  void* ptr = nullptr;
};
ScratchAddr g_scratch[kMaxDevices];
std::mutex g_scratch_mu;

}  // namespace

extern "C" cb_status cb_ragged_paged_attention_noalloc(
    const void* q, const void* k_pages, const void* v_pages, const int32_t* block_table,
    const int32_t* cu_seqlens_q, const int32_t* kv_lens, int32_t block_size, float scale,
    void* out, float* lse, const cb_dims* dims, void* stream) {
  const size_t need = cb_attention_workspace_size(dims);
  if (need == 0) {
    // invalid dims: let the regular entry point produce the detailed message
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
  unsigned long long ctx = 0;
  cb_status st = cb::current_context_id(&ctx);
  if (st != CB_OK) return st;
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    ScratchAddr& sa = g_scratch[dev];
    if (ctx == 0 || sa.ctx_id != ctx) {
      // Set-up on this device (once per context): the array's device address.  Host code only
      // knows a host-side stand-in for the symbol, which must never be handed to a kernel.
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_noalloc_scratch);  // makes the context current if needed
      if (e != cudaSuccess || p == nullptr) {
        snprintf(msg, sizeof(msg), "cudaGetSymbolAddress(scratch): %s", cudaGetErrorString(e));
        return cb::set_last_error(CB_ERR_CUDA, msg);
      }
      if ((st = cb::current_context_id(&ctx)) != CB_OK) return st;
      sa.ptr = p;
      sa.ctx_id = ctx;
    }
    scratch = sa.ptr;
  }
  return cb_ragged_paged_attention(q, k_pages, v_pages, block_table, cu_seqlens_q, kv_lens,
                                   block_size, scale, out, lse, scratch, kNoAllocScratchBytes,
                                   dims, stream);
}
