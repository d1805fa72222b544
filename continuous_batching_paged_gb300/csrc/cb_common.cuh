// Shared device helpers for libcb: error word, bounded mbarrier waits, TMA, warp MMA and
// tcgen05 (5th-generation tensor core) wrappers.  sm_103a only.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/cb.h"

namespace cb {

// Bits of the per-device error word.
constexpr uint32_t kErrOutOfRange = 1u;
constexpr uint32_t kErrTimeout = 2u;

// A device-side wait gives up after this many nanoseconds of %globaltimer.
constexpr uint64_t kWaitLimitNs = 1000ull * 1000ull * 1000ull;  // 1 s

constexpr int kDecodeTileKeys = 16;     // keys per decode pipeline stage
constexpr int kPrefillTileM = 128;      // queries per prefill tile (TMEM lanes)
constexpr int kChunkKeys = 128;         // keys per K/V tile of the chunk pass
constexpr int kMaxDecodeHeadsPerCta = 8;

// A chunk-pass CTA runs two 128-query tiles A and B against the same K/V tiles.  With an even
// GQA group size they are one query tile under two query heads of one KV group (equal key
// ranges); otherwise two consecutive query tiles under one head.  A "unit" is what one item
// covers under one head (pair): 1 tile or 2 tiles.
__host__ __device__ inline bool pf_pair_heads(int G) { return (G & 1) == 0; }
__host__ __device__ inline int pf_unit_tiles(int G) { return pf_pair_heads(G) ? 1 : 2; }

constexpr int kCostBins = 1024;  // histogram bins of the planner's longest-first unit order

// Sliding window: the first key a query at absolute position p sees (0 without a window).
__host__ __device__ inline int window_first_key(int p, int window) {
  return (window > 0 && p >= window) ? p - window + 1 : 0;
}

// %globaltimer (ns since an arbitrary origin, the same on every SM).
__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Workspace header (int32 words).
struct PlanHeader {
  int32_t n_dec;          // number of decode sequences (q_len == 1)
  int32_t dec_tiles;      // total 16-key tiles over all decode sequences
  int32_t n_pf;           // number of chunk sequences (q_len > 1)
  int32_t pf_qtiles;      // total work units over all chunk sequences (pf_unit_tiles)
  int32_t pf_counter;     // dynamic work counter of the prefill pass (reset by the planner)
  int32_t decode_ctas;    // CTAs the decode pass was planned for
  int32_t pad[2];
  // %globaltimer stamps (ns) of the attention kernel's roles, reset by the planner: first
  // start and last end of the decode CTAs that had work, and of the chunk CTAs.
  unsigned long long t_dec_start, t_dec_end, t_pf_start, t_pf_end;
};

// Byte offsets of the workspace sections (all 256-byte aligned).
struct WsLayout {
  size_t header, dec_seq, dec_prefix, dec_rec, cta_first, pf_seq, pf_prefix, pf_order, merge_cnt,
      part_ml, part_o, total;
};

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

__host__ __device__ inline WsLayout ws_layout(int S, int T, int Hq, int D) {
  WsLayout L;
  size_t off = 0;
  L.header = off;     off = align_up(off + sizeof(PlanHeader), 256);
  L.dec_seq = off;    off = align_up(off + sizeof(int32_t) * (size_t)(S + 1), 256);
  L.dec_prefix = off; off = align_up(off + sizeof(int32_t) * (size_t)(S + 1), 256);
  // per decode sequence (sequence, query token, kv_len, first tile) in one 16-byte record, so
  // that the decode pass gets a sequence's metadata in one load
  L.dec_rec = off;    off = align_up(off + sizeof(int32_t) * 4 * (size_t)(S + 1), 256);
  // per decode CTA of the grid: the decode sequence holding its first tile, -1 if it is idle
  L.cta_first = off;  off = align_up(off + sizeof(int32_t) * (size_t)(CB_MAX_DECODE_CTAS + 1), 256);
  L.pf_seq = off;     off = align_up(off + sizeof(int32_t) * (size_t)(S + 1), 256);
  L.pf_prefix = off;  off = align_up(off + sizeof(int32_t) * (size_t)(S + 1), 256);
  // chunk units, longest first: at most one per 128 query tokens plus one per sequence
  L.pf_order = off;   off = align_up(off + sizeof(int32_t) * ((size_t)S + (size_t)T / kPrefillTileM + 1), 256);
  L.merge_cnt = off;  off = align_up(off + sizeof(int32_t) * (size_t)S * (size_t)Hq, 256);
  const size_t slots = (size_t)CB_MAX_DECODE_CTAS + (size_t)S;
  L.part_ml = off;    off = align_up(off + sizeof(float2) * slots * (size_t)Hq, 256);
  L.part_o = off;     off = align_up(off + sizeof(float) * slots * (size_t)Hq * (size_t)D, 256);
  L.total = off;
  return L;
}

#if defined(__CUDACC__)

// Working index of decode CTA bx of a grid of `grid` decode CTAs when N of them work, -1 if bx
// is idle.  With N below the grid size the working CTAs are spread evenly over the grid, in
// pairs of consecutive CTAs where N and the grid are even: CTA b (or pair b/2) works when it is
// the first with its value of floor(b N / grid), and takes that value's range.  The block
// scheduler puts consecutive CTAs on the two SMs of a TPC and deals TPCs out across the GPCs.
// Measured beside a chunk pass: with the first N CTAs working the decode pass ran ~6% slower;
// with single CTAs spread, decode and chunk CTAs shared TPCs and the chunk pass ran ~5% slower;
// spread pairs ran both at the speed of a launch of exactly N CTAs.
__device__ __forceinline__ int decode_cta_index(int bx, int N, int grid) {
  if (N >= grid) return bx;
  const bool pairs = ((N | grid) & 1) == 0;
  const int units = pairs ? grid / 2 : grid, wanted = pairs ? N / 2 : N;
  const int u = pairs ? bx >> 1 : bx;
  const int cu = (int)((long long)u * wanted / units);
  if (u > 0 && (long long)(u - 1) * wanted / units == cu) return -1;
  return pairs ? 2 * cu + (bx & 1) : cu;
}

__device__ __forceinline__ void report(uint32_t* err, uint32_t bit) { atomicOr(err, bit); }

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ------------------------------------------------------------------------------------------
// mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Non-blocking test: has the phase of parity `parity` completed?
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Wait for the phase of parity `parity` to complete; false after `limit_ns` of %globaltimer.
__device__ __forceinline__ bool mbar_wait_for(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
}
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  return mbar_wait_for(bar, parity, kWaitLimitNs);
}

// ------------------------------------------------------------------------------------------
// TMA (bulk tensor copies global -> shared, completion through an mbarrier transaction count)
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

// The same load with an L2 eviction-priority policy (from l2_policy_evict_first).
__device__ __forceinline__ void tma_load_3d_hint(uint32_t dst, const CUtensorMap* map,
                                                 uint32_t bar, int c0, int c1, int c2,
                                                 uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "l"(policy)
      : "memory");
}

// Bulk prefetch of `bytes` (a multiple of 16) at `p` (16-byte aligned) into L2: a hint, no
// completion to wait for.
__device__ __forceinline__ void l2_prefetch_bulk(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(p)),
               "r"(bytes)
               : "memory");
}

// L2 policy for data read once (streamed K/V of decode tokens): its lines are the first to go,
// so data that other work re-reads stays in L2.
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ------------------------------------------------------------------------------------------
// Warp-level tensor-core helpers (ldmatrix + mma.sync m16n8k16, bf16 in, fp32 accumulate)
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void mma_bf16_16816(float* c, const uint32_t* a, uint32_t b0,
                                               uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// Transpose an 8x8 matrix of 16-bit elements held in the mma fragment layout (thread i: row
// i / 4, columns 2 (i % 4) and 2 (i % 4) + 1) across the warp.
__device__ __forceinline__ uint32_t movm_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
// Hardware base-2 exponential (the MUFU approximation; exp2(-inf) = 0).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// Packed pairs of fp32 values in one 64-bit register, for the paired fp32 instructions
// (fma / add on f32x2), which issue one instruction for two lanes of work.
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
// max of three fp32 values in one instruction
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
// Address of 16-byte chunk `chunk` (0..7) of 128-byte row `row` in a region laid out by TMA
// with the 128-byte swizzle: the chunk index is XORed with the row index modulo 8.
__device__ __forceinline__ uint32_t sw128(uint32_t region, uint32_t row, uint32_t chunk) {
  return region + row * 128u + (((chunk ^ row) & 7u) << 4);
}

// One lane of a fully active warp is elected (the same lane every time); the rest skip.  Used
// so that a warp runs the tcgen05 issue loop with warp-uniform control flow while a single
// thread issues the MMAs and the commits that track them.
__device__ __forceinline__ bool elect_one() {
  uint32_t pred;
  asm volatile(
      "{\n\t.reg .b32 r;\n\t.reg .pred p;\n\t"
      "elect.sync r|p, 0xffffffff;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(pred));
  return pred != 0;
}

// Register reallocation between warpgroups (all four warps of a warpgroup execute it).  The
// counts handed out must add up to no more than what the block was launched with.
template <int N>
__device__ __forceinline__ void regs_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void regs_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

// ------------------------------------------------------------------------------------------
// tcgen05: tensor memory allocation, MMA issue, commit, and TMEM <-> register moves.
__device__ __forceinline__ void tmem_alloc(uint32_t smem_dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_dst),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D[tmem] (+)= A[smem desc] * B[smem desc]
__device__ __forceinline__ void tc_mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem desc]
__device__ __forceinline__ void tc_mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive on an mbarrier once every tcgen05.mma issued so far by this thread has completed.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}
__device__ __forceinline__ void tc_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tc_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

#define CB_R8(i) "=r"(r[i]), "=r"(r[i + 1]), "=r"(r[i + 2]), "=r"(r[i + 3]), "=r"(r[i + 4]), \
                 "=r"(r[i + 5]), "=r"(r[i + 6]), "=r"(r[i + 7])
#define CB_W8(i) "r"(r[i]), "r"(r[i + 1]), "r"(r[i + 2]), "r"(r[i + 3]), "r"(r[i + 4]), \
                 "r"(r[i + 5]), "r"(r[i + 6]), "r"(r[i + 7])

// 32 consecutive 32-bit TMEM columns of this thread's lane -> r[0..31].
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : CB_R8(0), CB_R8(8), CB_R8(16), CB_R8(24)
      : "r"(taddr));
}
// r[0..31] -> 32 consecutive 32-bit TMEM columns of this thread's lane.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(
          taddr),
      CB_W8(0), CB_W8(8), CB_W8(16), CB_W8(24)
      : "memory");
}

// Shared-memory matrix descriptor of the 5th-generation tensor core: start address, leading
// and stride byte offsets (all >> 4), descriptor version 1, and the 128-byte swizzle mode.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((addr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo & 0x3FFFFu) >> 4) << 16;
  d |= (uint64_t)((sbo & 0x3FFFFu) >> 4) << 32;
  d |= (uint64_t)1 << 46;  // version
  d |= (uint64_t)2 << 61;  // 128-byte swizzle
  return d;
}
// Instruction descriptor, kind::f16: fp32 accumulator, bf16 A and B, A K-major, B K-major
// (b_mn_major = 0) or MN-major (1), tile M x N.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, int b_mn_major) {
  return (1u << 4)                      // D format: f32
         | (1u << 7)                    // A format: bf16
         | (1u << 10)                   // B format: bf16
         | ((uint32_t)b_mn_major << 16)  // B major-ness
         | ((uint32_t)(N >> 3) << 17)   // N / 8
         | ((uint32_t)(M >> 4) << 24);  // M / 16
}

#endif  // __CUDACC__

}  // namespace cb
