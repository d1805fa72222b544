// C ABI of libcb (see include/cb.h): host-side validation, TMA descriptor encoding, launches,
// and the per-device error word.
#include <cudaTypedefs.h>

#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "cb_common.cuh"
#include "cb_launch.h"

namespace {

__device__ uint32_t g_cb_error_word;

thread_local std::string t_last_error;

cb_status fail(cb_status st, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
cb_status fail(cb_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  t_last_error = buf;
  return st;
}

cb_status cuda_fail(cudaError_t e, const char* what) {
  return fail(CB_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

struct DeviceState {
  bool ready = false;
  unsigned long long ctx_id = 0;  // context the cached addresses belong to
  int sm_count = 0;
  uint32_t* err = nullptr;
};

constexpr int kMaxDevices = 64;
DeviceState g_dev[kMaxDevices];
std::mutex g_mu;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
PFN_cuCtxGetCurrent_v4000 g_ctx_get_current = nullptr;
PFN_cuCtxGetId_v12000 g_ctx_get_id = nullptr;
std::once_flag g_driver_once;
thread_local unsigned long long t_ctx_id = 0;

// Driver entry points the library calls directly (it links the CUDA runtime only).
void load_driver_entry_points() {
  cudaDriverEntryPointQueryResult q;
  void* fn = nullptr;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                       &q) == cudaSuccess && q == cudaDriverEntryPointSuccess)
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  fn = nullptr;
  if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) ==
          cudaSuccess && q == cudaDriverEntryPointSuccess)
    g_ctx_get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
  fn = nullptr;
  if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) ==
          cudaSuccess && q == cudaDriverEntryPointSuccess)
    g_ctx_get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(fn);
}

// Unique id of the calling thread's current CUDA context (0 when none is current yet).
// Device addresses looked up in one context are meaningless in the next (after a
// cudaDeviceReset, for instance), so every cached address is kept together with this id.
cb_status context_id(unsigned long long* id) {
  std::call_once(g_driver_once, load_driver_entry_points);
  *id = 0;
  if (g_ctx_get_current == nullptr || g_ctx_get_id == nullptr)
    return fail(CB_ERR_CUDA, "cuCtxGetCurrent / cuCtxGetId entry points unavailable");
  CUcontext c = nullptr;
  if (g_ctx_get_current(&c) != CUDA_SUCCESS) return fail(CB_ERR_CUDA, "cuCtxGetCurrent failed");
  if (c != nullptr && g_ctx_get_id(c, id) != CUDA_SUCCESS)
    return fail(CB_ERR_CUDA, "cuCtxGetId failed");
  return CB_OK;
}

cb_status device_state(DeviceState** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(CB_ERR_UNSUPPORTED, "device id %d", dev);
  unsigned long long ctx = 0;
  cb_status cst = context_id(&ctx);
  if (cst != CB_OK) return cst;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceState& st = g_dev[dev];
  if (!st.ready || ctx == 0 || st.ctx_id != ctx) {
    st.ready = false;
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (major != 10 || minor != 3)
      return fail(CB_ERR_UNSUPPORTED, "libcb is built for sm_103a; device %d is sm_%d%d", dev,
                  major, minor);
    e = cudaDeviceGetAttribute(&st.sm_count, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_cb_error_word);  // also makes the device's context current
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(error word)");
    st.err = static_cast<uint32_t*>(p);
    if (g_encode == nullptr)
      return fail(CB_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
    if ((cst = context_id(&ctx)) != CB_OK) return cst;
    st.ctx_id = ctx;
    st.ready = true;
  }
  t_ctx_id = st.ctx_id;
  *out = &st;
  return CB_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int gcd_int(int x, int y) {
  while (y) {
    const int t = x % y;
    x = y;
    y = t;
  }
  return x;
}

cb_status check_dims(const cb_dims* d, int32_t block_size) {
  if (d == nullptr) return fail(CB_ERR_INVALID_ARG, "dims is NULL");
  if (block_size < 4)
    return fail(CB_ERR_INVALID_ARG, "block_size must be at least 4, got %d", block_size);
  if (d->num_seqs < 0 || d->num_tokens < 0)
    return fail(CB_ERR_INVALID_ARG, "negative num_seqs or num_tokens");
  if (d->num_q_heads < 1 || d->num_kv_heads < 1)
    return fail(CB_ERR_INVALID_ARG, "num_q_heads and num_kv_heads must be >= 1");
  if (d->num_q_heads % d->num_kv_heads != 0)
    return fail(CB_ERR_INVALID_ARG, "num_q_heads (%d) is not a multiple of num_kv_heads (%d)",
                d->num_q_heads, d->num_kv_heads);
  if (d->num_pages < 1 || d->max_blocks_per_seq < 1)
    return fail(CB_ERR_INVALID_ARG, "num_pages and max_blocks_per_seq must be >= 1");
  if ((long long)d->num_pages * block_size >= (1LL << 31))
    return fail(CB_ERR_INVALID_ARG, "num_pages * block_size must be < 2^31");
  if ((long long)d->max_blocks_per_seq * block_size >= (1LL << 31))
    return fail(CB_ERR_INVALID_ARG, "max_blocks_per_seq * block_size must be < 2^31");
  if (d->head_dim != 64 && d->head_dim != 128)
    return fail(CB_ERR_UNSUPPORTED, "head_dim %d (supported: 64, 128)", d->head_dim);
  return CB_OK;
}

// 3-D bf16 tensor map with 128-byte swizzle and a box of 64 x box1 x box2 elements.
cb_status encode_map(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                     uint64_t s1_bytes, uint64_t s2_bytes, uint32_t box1, uint32_t box2) {
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {s1_bytes, s2_bytes};
  const cuuint32_t box[3] = {64, box1, box2};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(CB_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return CB_OK;
}

}  // namespace

namespace cb {
// Record a host-side error for cb_last_error_message() from another translation unit.
cb_status set_last_error(cb_status st, const char* msg) {
  t_last_error = msg;
  return st;
}
// Id of the calling thread's current context, for caches of device addresses and per-context
// settings in other translation units (0 when no context is current).
cb_status current_context_id(unsigned long long* id) { return context_id(id); }
// The context of the last device_state() on this thread: the one the next launch goes to.
unsigned long long launch_context_id() { return t_ctx_id; }
}  // namespace cb

extern "C" {

int32_t cb_version(void) { return 100; }

const char* cb_status_string(cb_status s) {
  switch (s) {
    case CB_OK: return "CB_OK";
    case CB_ERR_INVALID_ARG: return "CB_ERR_INVALID_ARG";
    case CB_ERR_UNSUPPORTED: return "CB_ERR_UNSUPPORTED";
    case CB_ERR_OUT_OF_RANGE: return "CB_ERR_OUT_OF_RANGE";
    case CB_ERR_TIMEOUT: return "CB_ERR_TIMEOUT";
    case CB_ERR_CUDA: return "CB_ERR_CUDA";
  }
  return "CB_ERR_UNKNOWN";
}

const char* cb_last_error_message(void) { return t_last_error.c_str(); }

size_t cb_attention_workspace_size(const cb_dims* dims) {
  // The size depends on the sequence, token and query-head counts and the head dim only.
  if (dims == nullptr || dims->num_seqs < 0 || dims->num_tokens < 0 || dims->num_q_heads < 1 ||
      dims->num_kv_heads < 1 || dims->num_q_heads % dims->num_kv_heads != 0 ||
      (dims->head_dim != 64 && dims->head_dim != 128))
    return 0;
  return cb::ws_layout(dims->num_seqs, dims->num_tokens, dims->num_q_heads, dims->head_dim).total;
}

cb_status cb_kv_append(const void* k_new, const void* v_new, void* k_pages, void* v_pages,
                       const int32_t* block_table, const int32_t* cu_seqlens_q,
                       const int32_t* kv_lens, int32_t block_size, const cb_dims* dims,
                       void* stream) {
  t_last_error.clear();
  cb_status st = check_dims(dims, block_size);
  if (st != CB_OK) return st;
  if (dims->num_tokens == 0) return CB_OK;
  if (!k_new || !v_new || !k_pages || !v_pages || !block_table || !cu_seqlens_q || !kv_lens)
    return fail(CB_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_pages) || !aligned16(v_pages))
    return fail(CB_ERR_INVALID_ARG, "K/V tensors must be 16-byte aligned");
  if (dims->num_seqs == 0) return CB_OK;  // every token row is padding
  DeviceState* ds = nullptr;
  st = device_state(&ds);
  if (st != CB_OK) return st;
  cb::AppendArgs a;
  a.k_new = k_new;
  a.v_new = v_new;
  a.k_pages = k_pages;
  a.v_pages = v_pages;
  a.block_table = block_table;
  a.cu_seqlens_q = cu_seqlens_q;
  a.kv_lens = kv_lens;
  a.S = dims->num_seqs;
  a.T = dims->num_tokens;
  a.Hkv = dims->num_kv_heads;
  a.D = dims->head_dim;
  a.bs = block_size;
  a.max_blocks = dims->max_blocks_per_seq;
  a.P = dims->num_pages;
  a.err = ds->err;
  cudaError_t e = cb::launch_kv_append(a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "kv_append launch");
  return CB_OK;
}

// The attention pass on `stream`: the planner, then the attention kernel (decode and chunk
// passes in one launch); with `app` non-NULL the KV-append of the same step shares the
// planner's launch.
static cb_status attention(const void* q, const void* k_pages, const void* v_pages,
                           const int32_t* block_table, const int32_t* cu_seqlens_q,
                           const int32_t* kv_lens, int32_t block_size, float scale, void* out,
                           float* lse, void* workspace, size_t workspace_bytes,
                           const cb_dims* dims, const cb_options* options,
                           const cb::AppendArgs* app, void* stream) {
  cb_status st = check_dims(dims, block_size);
  if (st != CB_OK) return st;
  if (dims->num_tokens == 0) return CB_OK;
  if (dims->num_seqs == 0) return CB_OK;  // every token row is padding
  if (!q || !k_pages || !v_pages || !block_table || !cu_seqlens_q || !kv_lens || !out || !workspace)
    return fail(CB_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned16(q) || !aligned16(k_pages) || !aligned16(v_pages) || !aligned16(out))
    return fail(CB_ERR_INVALID_ARG, "q, pages and out must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return fail(CB_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  if (lse != nullptr && (reinterpret_cast<uintptr_t>(lse) & 3u) != 0)
    return fail(CB_ERR_INVALID_ARG, "lse must be 4-byte aligned");
  if (!(scale > 0.f) || scale != scale)
    return fail(CB_ERR_INVALID_ARG, "scale must be a positive finite number");
  const size_t need = cb::ws_layout(dims->num_seqs, dims->num_tokens, dims->num_q_heads, dims->head_dim).total;
  if (workspace_bytes < need)
    return fail(CB_ERR_INVALID_ARG, "workspace too small: %zu < %zu bytes", workspace_bytes, need);
  const int Hq = dims->num_q_heads, Hkv = dims->num_kv_heads, G = Hq / Hkv;
  if (G > 16) return fail(CB_ERR_UNSUPPORTED, "more than 16 query heads per KV head");
  // KV heads per decode CTA: 8, or 4 when each KV head has more than 8 query heads (two warps
  // per KV head then share its query heads)
  const int dec_heads = G > 8 ? cb::kMaxDecodeHeadsPerCta / 2 : cb::kMaxDecodeHeadsPerCta;
  if (Hkv > dec_heads && Hkv % dec_heads != 0)
    return fail(CB_ERR_UNSUPPORTED, "num_kv_heads > %d must be a multiple of %d", dec_heads,
                dec_heads);
  DeviceState* ds = nullptr;
  st = device_state(&ds);
  if (st != CB_OK) return st;

  cb::AttnArgs a;
  a.q = q;
  a.out = out;
  a.lse = lse;
  a.block_table = block_table;
  a.cu_seqlens_q = cu_seqlens_q;
  a.kv_lens = kv_lens;
  a.ws = static_cast<char*>(workspace);
  a.err = ds->err;
  a.S = dims->num_seqs;
  a.T = dims->num_tokens;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.G = G;
  a.D = dims->head_dim;
  a.bs = block_size;
  a.max_blocks = dims->max_blocks_per_seq;
  a.P = dims->num_pages;
  a.KB = gcd_int(block_size, 16);
  a.KBp = gcd_int(block_size, 128);
  int dctas = options != nullptr ? options->decode_ctas : 0;
  a.decode_auto = dctas <= 0 ? 1 : 0;
  const int head_groups = (Hkv + dec_heads - 1) / dec_heads;
  // by default the decode CTAs of all KV-head groups together take one CTA per SM
  if (dctas <= 0) dctas = ds->sm_count / head_groups > 0 ? ds->sm_count / head_groups : 1;
  if (dctas > CB_MAX_DECODE_CTAS) dctas = CB_MAX_DECODE_CTAS;
  a.decode_ctas = dctas;
  a.prefill_ctas = ds->sm_count;
  a.window = options != nullptr ? options->window : 0;
  if (a.window < 0) return fail(CB_ERR_INVALID_ARG, "window must be >= 0, got %d", a.window);
  a.scale_log2 = scale * 1.4426950408889634f;

  cb::AttnMaps maps;
  const uint64_t D = (uint64_t)a.D;
  const uint64_t rows = (uint64_t)a.P * (uint64_t)block_size;
  // Decode pass: dims (d, token, head) so one box {64, KB tokens, up to 8 heads} lands in shared
  // memory as [head][token] rows; chunk pass: dims (d, head, token), box {64, 1 head, KBp tokens}.
  const uint32_t HB = (uint32_t)(Hkv < dec_heads ? Hkv : dec_heads);
  if ((st = encode_map(&maps.k_dec, k_pages, D, rows, Hkv, D * 2 * Hkv, D * 2, a.KB, HB)) != CB_OK) return st;
  if ((st = encode_map(&maps.v_dec, v_pages, D, rows, Hkv, D * 2 * Hkv, D * 2, a.KB, HB)) != CB_OK) return st;
  if ((st = encode_map(&maps.k_chunk, k_pages, D, Hkv, rows, D * 2, D * 2 * Hkv, 1, a.KBp)) != CB_OK) return st;
  if ((st = encode_map(&maps.v_chunk, v_pages, D, Hkv, rows, D * 2, D * 2 * Hkv, 1, a.KBp)) != CB_OK) return st;
  if ((st = encode_map(&maps.q, q, D, Hq, (uint64_t)a.T, D * 2, D * 2 * Hq, 1, 128)) != CB_OK) return st;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  void* const* ev = options != nullptr ? options->phase_events : nullptr;
  const bool serial = options != nullptr && (options->flags & CB_OPT_SERIAL);
  auto mark = [&](int i) -> cudaError_t {
    return ev != nullptr ? cudaEventRecord(static_cast<cudaEvent_t>(ev[i]), s) : cudaSuccess;
  };
  cudaError_t e = cudaSuccess;
  cb::AppendArgs ap;
  if (app != nullptr) {
    ap = *app;
    ap.err = ds->err;
  }
  if (app != nullptr && !serial) {
    // One launch appends the step's K/V rows and plans the attention pass (which reads only
    // the metadata, not the pages).
    if ((e = mark(0)) != cudaSuccess) return cuda_fail(e, "cudaEventRecord(phase event)");
    if ((e = cb::launch_append_plan(ap, a, s)) != cudaSuccess) return cuda_fail(e, "append + plan launch");
  } else {
    if (app != nullptr && (e = cb::launch_kv_append(ap, s)) != cudaSuccess)
      return cuda_fail(e, "kv_append launch");
    if ((e = mark(0)) != cudaSuccess) return cuda_fail(e, "cudaEventRecord(phase event)");
    if ((e = cb::launch_plan(a, s)) != cudaSuccess) return cuda_fail(e, "plan launch");
  }
  if ((e = mark(1)) != cudaSuccess) return cuda_fail(e, "cudaEventRecord(phase event)");
  if (serial) {
    cb::AttnArgs d = a;
    d.decode_grid = a.decode_ctas * head_groups;
    d.prefill_ctas = 0;
    if ((e = cb::launch_attention(d, maps, s)) != cudaSuccess) return cuda_fail(e, "attention launch");
    if ((e = mark(2)) != cudaSuccess || (e = mark(3)) != cudaSuccess)
      return cuda_fail(e, "cudaEventRecord(phase event)");
    cb::AttnArgs c = a;
    c.decode_grid = 0;
    if ((e = cb::launch_attention(c, maps, s)) != cudaSuccess) return cuda_fail(e, "attention launch");
    if ((e = mark(4)) != cudaSuccess) return cuda_fail(e, "cudaEventRecord(phase event)");
  } else {
    a.decode_grid = a.decode_ctas * head_groups;
    if ((e = mark(3)) != cudaSuccess) return cuda_fail(e, "cudaEventRecord(phase event)");
    if ((e = cb::launch_attention(a, maps, s)) != cudaSuccess) return cuda_fail(e, "attention launch");
    if ((e = mark(2)) != cudaSuccess || (e = mark(4)) != cudaSuccess)
      return cuda_fail(e, "cudaEventRecord(phase event)");
  }
  return CB_OK;
}

cb_status cb_pass_timestamps(const void* workspace, uint64_t* ts_ns, void* stream) {
  t_last_error.clear();
  if (workspace == nullptr || ts_ns == nullptr) return fail(CB_ERR_INVALID_ARG, "null pointer argument");
  cb::PlanHeader h;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(&h, workspace, sizeof(h), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "reading the plan header");
  const bool dec = h.t_dec_end != 0, pf = h.t_pf_end != 0;
  ts_ns[0] = dec ? h.t_dec_start : 0;
  ts_ns[1] = dec ? h.t_dec_end : 0;
  ts_ns[2] = pf ? h.t_pf_start : 0;
  ts_ns[3] = pf ? h.t_pf_end : 0;
  return CB_OK;
}

cb_status cb_ragged_paged_attention_ex(const void* q, const void* k_pages, const void* v_pages,
                                       const int32_t* block_table, const int32_t* cu_seqlens_q,
                                       const int32_t* kv_lens, int32_t block_size, float scale,
                                       void* out, float* lse, void* workspace,
                                       size_t workspace_bytes, const cb_dims* dims,
                                       const cb_options* options, void* stream) {
  t_last_error.clear();
  return attention(q, k_pages, v_pages, block_table, cu_seqlens_q, kv_lens, block_size, scale,
                   out, lse, workspace, workspace_bytes, dims, options, nullptr, stream);
}

cb_status cb_append_attention(const void* k_new, const void* v_new, void* k_pages, void* v_pages,
                              const void* q, const int32_t* block_table,
                              const int32_t* cu_seqlens_q, const int32_t* kv_lens,
                              int32_t block_size, float scale, void* out, float* lse,
                              void* workspace, size_t workspace_bytes, const cb_dims* dims,
                              const cb_options* options, void* stream) {
  t_last_error.clear();
  cb_status st = check_dims(dims, block_size);
  if (st != CB_OK) return st;
  if (dims->num_tokens == 0 || dims->num_seqs == 0) return CB_OK;
  if (!k_new || !v_new) return fail(CB_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned16(k_new) || !aligned16(v_new))
    return fail(CB_ERR_INVALID_ARG, "K/V tensors must be 16-byte aligned");
  cb::AppendArgs ap;
  ap.k_new = k_new;
  ap.v_new = v_new;
  ap.k_pages = k_pages;
  ap.v_pages = v_pages;
  ap.block_table = block_table;
  ap.cu_seqlens_q = cu_seqlens_q;
  ap.kv_lens = kv_lens;
  ap.S = dims->num_seqs;
  ap.T = dims->num_tokens;
  ap.Hkv = dims->num_kv_heads;
  ap.D = dims->head_dim;
  ap.bs = block_size;
  ap.max_blocks = dims->max_blocks_per_seq;
  ap.P = dims->num_pages;
  ap.err = nullptr;  // set to the device's error word at launch
  return attention(q, k_pages, v_pages, block_table, cu_seqlens_q, kv_lens, block_size, scale,
                   out, lse, workspace, workspace_bytes, dims, options, &ap, stream);
}

cb_status cb_ragged_paged_attention(const void* q, const void* k_pages, const void* v_pages,
                                    const int32_t* block_table, const int32_t* cu_seqlens_q,
                                    const int32_t* kv_lens, int32_t block_size, float scale,
                                    void* out, float* lse, void* workspace,
                                    size_t workspace_bytes, const cb_dims* dims, void* stream) {
  return cb_ragged_paged_attention_ex(q, k_pages, v_pages, block_table, cu_seqlens_q, kv_lens,
                                      block_size, scale, out, lse, workspace, workspace_bytes,
                                      dims, nullptr, stream);
}

// Shared host half of the three block-move entry points.
static cb_status block_move(const void* pk, const void* pv, void* dk, void* dv,
                            const int32_t* src_idx, const int32_t* dst_idx, int32_t n,
                            int32_t block_size, const cb_dims* dims, int mode, void* stream) {
  t_last_error.clear();
  if (dims == nullptr) return fail(CB_ERR_INVALID_ARG, "dims is NULL");
  if (block_size < 4)
    return fail(CB_ERR_INVALID_ARG, "block_size must be at least 4, got %d", block_size);
  if (n < 0) return fail(CB_ERR_INVALID_ARG, "negative block count");
  if (dims->num_kv_heads < 1 || dims->num_pages < 1)
    return fail(CB_ERR_INVALID_ARG, "num_kv_heads and num_pages must be >= 1");
  if (dims->head_dim != 64 && dims->head_dim != 128)
    return fail(CB_ERR_UNSUPPORTED, "head_dim %d (supported: 64, 128)", dims->head_dim);
  if (n == 0) return CB_OK;
  if (!pk || !pv || !dk || !dv || (mode != cb::kMoveRestore && !src_idx) ||
      (mode != cb::kMoveOffload && !dst_idx))
    return fail(CB_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned16(pk) || !aligned16(pv) || !aligned16(dk) || !aligned16(dv))
    return fail(CB_ERR_INVALID_ARG, "pools and host buffers must be 16-byte aligned");
  DeviceState* ds = nullptr;
  cb_status st = device_state(&ds);
  if (st != CB_OK) return st;
  cb::BlockMoveArgs a;
  a.src[0] = static_cast<const char*>(pk);
  a.src[1] = static_cast<const char*>(pv);
  a.dst[0] = static_cast<char*>(dk);
  a.dst[1] = static_cast<char*>(dv);
  a.src_idx = src_idx;
  a.dst_idx = dst_idx;
  a.n = n;
  a.P = dims->num_pages;
  a.mode = mode;
  a.block_bytes = (long long)block_size * dims->num_kv_heads * dims->head_dim * 2;
  a.err = ds->err;
  cudaError_t e = cb::launch_block_move(a, ds->sm_count, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "block move launch");
  return CB_OK;
}

cb_status cb_copy_blocks(void* k_pages, void* v_pages, const int32_t* src, const int32_t* dst,
                         int32_t n, int32_t block_size, const cb_dims* dims, void* stream) {
  return block_move(k_pages, v_pages, k_pages, v_pages, src, dst, n, block_size, dims,
                    cb::kMoveCopy, stream);
}

cb_status cb_kv_offload(const void* k_pages, const void* v_pages, const int32_t* blocks,
                        int32_t n, int32_t block_size, const cb_dims* dims, void* host_k,
                        void* host_v, void* stream) {
  return block_move(k_pages, v_pages, host_k, host_v, blocks, nullptr, n, block_size, dims,
                    cb::kMoveOffload, stream);
}

cb_status cb_kv_restore(void* k_pages, void* v_pages, const int32_t* blocks, int32_t n,
                        int32_t block_size, const cb_dims* dims, const void* host_k,
                        const void* host_v, void* stream) {
  return block_move(host_k, host_v, k_pages, v_pages, nullptr, blocks, n, block_size, dims,
                    cb::kMoveRestore, stream);
}

cb_status cb_selftest_wait_timeout(int32_t limit_us, unsigned long long* waited_ns, void* stream) {
  t_last_error.clear();
  if (limit_us < 1 || limit_us > 100000)
    return fail(CB_ERR_INVALID_ARG, "limit_us must be in [1, 100000], got %d", limit_us);
  DeviceState* ds = nullptr;
  cb_status st = device_state(&ds);
  if (st != CB_OK) return st;
  cudaError_t e = cb::launch_wait_selftest(ds->err, (uint64_t)limit_us * 1000ull,
                                           reinterpret_cast<uint64_t*>(waited_ns),
                                           static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "self-test launch");
  return CB_OK;
}

cb_status cb_get_device_error(void* stream) {
  t_last_error.clear();
  DeviceState* ds = nullptr;
  cb_status st = device_state(&ds);
  if (st != CB_OK) return st;
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  uint32_t bits = 0;
  e = cudaMemcpy(&bits, ds->err, sizeof(bits), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "read error word");
  if (bits != 0) {
    const uint32_t zero = 0;
    e = cudaMemcpy(ds->err, &zero, sizeof(zero), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return cuda_fail(e, "clear error word");
  }
  if (bits & cb::kErrTimeout) return fail(CB_ERR_TIMEOUT, "a device-side wait expired");
  if (bits & cb::kErrOutOfRange)
    return fail(CB_ERR_OUT_OF_RANGE, "device saw metadata outside the pool, table or lengths");
  return CB_OK;
}

}  // extern "C"
