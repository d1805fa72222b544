// Decode pass of ragged paged attention: every sequence with q_len == 1 attends to all of its
// kv_len keys.  Each decode step streams a sequence's whole cached K/V once for one query token
// (the point "LLM learning path 3.3 Batching & Memory Management" makes in its section "Common
// pitfalls"), so this pass is bound by HBM bandwidth and is built around moving K/V pages at
// full rate:
//
//   * The key tiles of all decode sequences are laid end to end (16 keys per tile) and cut into
//     N equal contiguous ranges (N from the planner, at most `decode_ctas`), one per working
//     CTA: every CTA streams the same number of bytes whatever the length mix.  The CTAs are
//     the first CTAs of the attention kernel (cb_attention.cu); the chunk pass's CTAs follow.  A sequence cut by range boundaries leaves per-CTA partial
//     results (m, l, o) in the workspace; the last warp to finish a (sequence, KV head, group of
//     8 query heads) merges them (an atomic counter per triple decides which): the split-KV scheme with an online
//     softmax and a log-sum-exp merge, without a separate merge launch.
//   * One producer warp walks the range, prefetches block-table entries 32 at a time (and each
//     sequence's query rows into L2), and issues TMA tensor copies (128-byte swizzle) of each
//     (page run, KV head, 64-wide half of D) into a multi-stage shared-memory ring guarded by
//     mbarriers.
//   * One consumer warp per KV head computes S^T = K Q^T and O^T += V^T P^T for the G query heads
//     of its group with mma.sync m16n8k16 (bf16 in, fp32 accumulate; keys as the M side, query
//     heads as N), so the G heads of a GQA group share every K/V byte read from HBM.  It takes
//     the stage's K and V fragments into registers and releases the stage before computing.
//     Softmax state lives in registers; maxima and sums are reduced with warp shuffles.
//
// Online softmax: for each new tile, m' = max(m, max_j x_j), rescale (l, o) by 2^(m - m'),
// then add 2^(x_j - m') and 2^(x_j - m') v_j; x_j = scale * log2(e) * q.k_j.
#pragma once

#include "cb_common.cuh"
#include "cb_launch.h"

namespace cb {

// A CTA covers 8 KV heads, one consumer warp per KV head and up to 8 query heads per warp.
// With more than 8 query heads per KV head (QS = 2) it covers 4 KV heads, two warps per KV
// head, each taking 8 of its query heads: the same per-warp work as a group of 8.
template <int QS>
constexpr int decode_kv_heads() { return kMaxDecodeHeadsPerCta / QS; }
// Stages of the decode ring, about 192 KB in all: a 16-key stage of K and V is 64 KB at
// head_dim 128 with 8 KV heads, and proportionally smaller with head_dim 64 or 4 KV heads, so
// those keep the same bytes in flight per SM with more stages.
template <int D, int QS>
constexpr int decode_stages() { return 3 * QS * (128 / D); }
constexpr uint32_t kInfoFirst = 1u, kInfoLast = 2u, kInfoComplete = 4u;

struct StageInfo {
  int seq;       // sequence id
  int dec;       // index among decode sequences (partial-result slot = cta + dec)
  int tok;       // packed token index of the sequence's query
  int kv;        // kv_len
  int lo;        // first key in the window (0 without a sliding window)
  int key0;      // first key of this tile
  uint32_t flags;
  int p0, p1;    // the sequence's tile range [p0, p1) in the concatenated tile order
};

template <int D, int QS>
struct DecodeSmem {
  static constexpr int kHalves = D / 64;
  static constexpr int kHalfBytes = decode_kv_heads<QS>() * kDecodeTileKeys * 128;  // 16 or 8 KB
  static constexpr int kKVBytes = kHalves * kHalfBytes;                             // K or V
  static constexpr int kStageBytes = 2 * kKVBytes;
  static constexpr int kStages = decode_stages<D, QS>();
  static constexpr int kBarOffset = kStages * kStageBytes;
  static constexpr int kInfoOffset = kBarOffset + 2 * kStages * 8;
  static constexpr int kTotal = kInfoOffset + kStages * (int)sizeof(StageInfo) + 1024;
};

// Largest CTA index c in [0, N) whose range start floor(c * n / N) is <= t.
__device__ __forceinline__ int cta_of_tile(long long t, long long n, int N) {
  int lo = 0, hi = N - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (n * mid / N <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// One warp combines the partial (m, l, o) that CTAs cf..cl wrote for decode sequence `dec`
// and query heads h0 .. h1 - 1 of KV head `kvh`'s group: M = max m_c, w_c = 2^(m_c - M),
// out = sum_c w_c o_c / sum_c w_c l_c, lse = (M + log2 sum_c w_c l_c) * ln 2.
// Other CTAs wrote these parts: they are read through L2 (ld.global.cg), never from a stale L1
// line.  Parts are taken kC at a time for kH heads at once, every (m, l) and o row of such a
// batch loaded before any is used (lane i holds output columns PER i .. PER i + PER - 1), and
// folded in with a running maximum: one L2 round trip per batch, so a sequence cut in two
// merges 4 heads in one round trip.
template <int D>
__device__ __forceinline__ void merge_parts(const AttnArgs& a, const float2* part_ml,
                                            const float* part_o, int dec, int tok, int kvh,
                                            int cf, int cl, int h0, int h1, int lane) {
  constexpr int PER = D / 32;  // output columns per lane: 4 (D = 128) or 2 (D = 64)
  constexpr int kH = 4, kC = 2;  // heads and parts in flight
  __nv_bfloat16* outg = static_cast<__nv_bfloat16*>(a.out);
  const int nparts = cl - cf + 1;
  for (int r0 = h0; r0 < h1; r0 += kH) {
    float M[kH], Lsum[kH], acc[kH][PER];
#pragma unroll
    for (int hh = 0; hh < kH; ++hh) {
      M[hh] = -INFINITY;
      Lsum[hh] = 0.f;
#pragma unroll
      for (int i = 0; i < PER; ++i) acc[hh][i] = 0.f;
    }
    for (int c0 = 0; c0 < nparts; c0 += kC) {
      float v[kH][kC][PER];
      float2 ml[kH][kC];
#pragma unroll
      for (int hh = 0; hh < kH; ++hh)
#pragma unroll
        for (int cc = 0; cc < kC; ++cc) {
          const int head = kvh * a.G + r0 + hh;
          const size_t slot = (size_t)(cf + c0 + cc) + dec;
          ml[hh][cc] = make_float2(-INFINITY, 0.f);
#pragma unroll
          for (int i = 0; i < PER; ++i) v[hh][cc][i] = 0.f;
          if (r0 + hh < h1 && c0 + cc < nparts) {
            ml[hh][cc] = __ldcg(part_ml + slot * a.Hq + head);
            const float* po = part_o + (slot * a.Hq + head) * D + lane * PER;
            if constexpr (PER == 4) {
              const float4 x = __ldcg(reinterpret_cast<const float4*>(po));
              v[hh][cc][0] = x.x; v[hh][cc][1] = x.y; v[hh][cc][2] = x.z; v[hh][cc][3] = x.w;
            } else {
              const float2 x = __ldcg(reinterpret_cast<const float2*>(po));
              v[hh][cc][0] = x.x; v[hh][cc][1] = x.y;
            }
          }
        }
#pragma unroll
      for (int hh = 0; hh < kH; ++hh)
#pragma unroll
        for (int cc = 0; cc < kC; ++cc) {
          if (r0 + hh < h1 && c0 + cc < nparts) {
            // every part holds at least one key of its sequence, so its m is finite
            const float mn = fmaxf(M[hh], ml[hh][cc].x);
            const float sc = fast_exp2(M[hh] - mn), w = fast_exp2(ml[hh][cc].x - mn);
            Lsum[hh] = Lsum[hh] * sc + ml[hh][cc].y * w;
#pragma unroll
            for (int i = 0; i < PER; ++i) acc[hh][i] = acc[hh][i] * sc + v[hh][cc][i] * w;
            M[hh] = mn;
          }
        }
    }
#pragma unroll
    for (int hh = 0; hh < kH; ++hh) {
      if (r0 + hh >= h1) continue;
      const int head = kvh * a.G + r0 + hh;
      const float inv = 1.f / Lsum[hh];
      uint32_t* dst =
          reinterpret_cast<uint32_t*>(outg + ((size_t)tok * a.Hq + head) * D + lane * PER);
#pragma unroll
      for (int i = 0; i < PER / 2; ++i)
        dst[i] = pack_bf16x2(acc[hh][2 * i] * inv, acc[hh][2 * i + 1] * inv);
      if (lane == 0 && a.lse != nullptr)
        a.lse[(size_t)tok * a.Hq + head] = (M[hh] + __log2f(Lsum[hh])) * 0.6931471805599453f;
    }
  }
}

// Consumer warp `warp` of the decode pass: KV head warp / QS of the CTA's group, query heads
// 8 (warp % QS) .. 8 (warp % QS) + 7 of its G (clipped to G), every tile of the CTA's range.  Products are taken with keys as the m16n8k16 M side and query heads as N:
//   S^T (16 keys x 8 heads)  = K (16 keys x 16 d) . Q^T (16 d x 8 heads), over D/16 k-steps;
//   O^T (16 d x 8 heads)    += V^T (16 d x 16 keys) . P^T (16 keys x 8 heads), over D/16 m-tiles.
// P^T is moved from the S^T accumulator layout to the B-operand layout with movmatrix.  The warp
// first loads every K and V fragment of the stage into registers and releases the stage before
// computing, so the producer refills it sooner.
template <int D, int QS>
__device__ __forceinline__ void decode_consume(const AttnArgs& a, uint32_t sbase, uint32_t bar_full,
                                               uint32_t bar_empty, const StageInfo* info, int c,
                                               int hg, int warp, long long n_my, long long ntiles,
                                               int N, const WsLayout& L, int lane) {
  using SM = DecodeSmem<D, QS>;
  constexpr int KS = D / 16;  // k-steps of S^T over the head dim
  constexpr int MT = D / 16;  // m-tiles of O^T over the head dim
  constexpr int NTH = 1;      // groups of 8 query heads per warp
  constexpr bool kPreload = true;
  const int h = warp / QS;                       // KV head within the CTA's group
  const int qoff = (warp % QS) * 8;              // first query head (within the KV head's G)
  const int kvh = hg * decode_kv_heads<QS>() + h;  // global KV head
  const int g = lane >> 2, tq = lane & 3;          // mma fragment coordinates
  float2* part_ml = reinterpret_cast<float2*>(a.ws + L.part_ml);
  float* part_o = reinterpret_cast<float*>(a.ws + L.part_o);
  int32_t* merge_cnt = reinterpret_cast<int32_t*>(a.ws + L.merge_cnt);
  const uint32_t* q32 = static_cast<const uint32_t*>(a.q);
  __nv_bfloat16* outg = static_cast<__nv_bfloat16*>(a.out);
  const float sl2 = a.scale_log2;

  uint32_t qb[NTH][KS][2];
  float o[MT][NTH][4];
  float mrun[NTH][2], lrun[NTH][2];
  // Stage layout of one 64-wide half of K (or V): runs of KB keys, each run [HB heads][KB keys]
  // of 128-byte rows, so key k of this warp's head is row (k / KB) * HB * KB + h * KB + k % KB.
  const int KB = a.KB, HB = a.Hkv < decode_kv_heads<QS>() ? a.Hkv : decode_kv_heads<QS>();
  auto row_of = [&](int k) { return (k / KB) * HB * KB + h * KB + (k % KB); };
  // ldmatrix lane -> (key, 16-byte chunk) of the K (non-transposed) and V (transposed) loads
  const int k_row = row_of((lane & 7) + (((lane >> 3) & 1) << 3)), k_csel = lane >> 4;
  const int v_row = row_of((lane & 7) + ((lane >> 4) << 3)), v_csel = (lane >> 3) & 1;

  for (long long it = 0; it < n_my; ++it) {
    const int stage = (int)(it % SM::kStages);
    const uint32_t phase = (uint32_t)((it / SM::kStages) & 1);
    if (!mbar_wait(bar_full + 8 * stage, phase)) {
      report(a.err, kErrTimeout);
      break;
    }
    const StageInfo si = info[stage];
    if (si.flags & kInfoFirst) {
#pragma unroll
      for (int ht = 0; ht < NTH; ++ht) {
        mrun[ht][0] = mrun[ht][1] = -INFINITY;
        lrun[ht][0] = lrun[ht][1] = 0.f;
        const int hl = qoff + ht * 8 + g;  // query head within the group, column g of Q^T
        const uint32_t* qrow = q32 + (((size_t)si.tok * a.Hq + kvh * a.G + hl) * D) / 2;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
          qb[ht][ks][0] = hl < a.G ? __ldg(qrow + ks * 8 + tq) : 0u;
          qb[ht][ks][1] = hl < a.G ? __ldg(qrow + ks * 8 + 4 + tq) : 0u;
        }
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) o[mt][ht][0] = o[mt][ht][1] = o[mt][ht][2] = o[mt][ht][3] = 0.f;
      }
    }
    const uint32_t kst = sbase + stage * SM::kStageBytes;
    const uint32_t vst = kst + SM::kKVBytes;
    const bool tail = si.key0 + kDecodeTileKeys > si.kv;

    const bool head = si.key0 < si.lo;  // keys before the sliding window in this tile

    // ---- K fragments (A operand of S^T: rows = keys, k = head dim)
    uint32_t kf[KS][4];
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      const int chunk = 2 * ks + k_csel;
      ldsm_x4(sw128(kst + (chunk >> 3) * SM::kHalfBytes, k_row, chunk & 7), kf[ks][0],
              kf[ks][1], kf[ks][2], kf[ks][3]);
    }
    // ---- keys past kv_len: their V rows may hold stale or poison data; P is 0 there, but
    // 0 * NaN is NaN, so zero those rows of this head before they are read.
    if (tail) {
      const int first = si.kv - si.key0;  // 1..15
      const int nrow = kDecodeTileKeys - first;
      for (int i = lane; i < nrow * SM::kHalves * 8; i += 32) {
        const int r = first + i / (SM::kHalves * 8);
        const int rem = i % (SM::kHalves * 8);
        const uint32_t addr = sw128(vst + (rem >> 3) * SM::kHalfBytes, row_of(r), rem & 7);
        asm volatile("st.shared.v4.u32 [%0], {%1,%1,%1,%1};" ::"r"(addr), "r"(0u) : "memory");
      }
      __syncwarp();
    }
    // ---- V fragments (A operand of O^T: rows = head dim, k = keys), loaded transposed
    uint32_t vf[kPreload ? MT : 1][4];
    if constexpr (kPreload) {
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        const int chunk = 2 * mt + v_csel;
        ldsm_x4_t(sw128(vst + (chunk >> 3) * SM::kHalfBytes, v_row, chunk & 7),
                  vf[mt][0], vf[mt][1], vf[mt][2], vf[mt][3]);
      }
      if (tail) fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_empty + 8 * stage);
    }

    // ---- S^T = K Q^T
    float s[NTH][4];
#pragma unroll
    for (int ht = 0; ht < NTH; ++ht) {
      s[ht][0] = s[ht][1] = s[ht][2] = s[ht][3] = 0.f;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) mma_bf16_16816(s[ht], kf[ks], qb[ht][ks][0], qb[ht][ks][1]);
    }
    if (tail || head) {
      const bool dead0 = si.key0 + g >= si.kv || si.key0 + g < si.lo;
      const bool dead1 = si.key0 + g + 8 >= si.kv || si.key0 + g + 8 < si.lo;
#pragma unroll
      for (int ht = 0; ht < NTH; ++ht) {
        if (dead0) s[ht][0] = s[ht][1] = -INFINITY;
        if (dead1) s[ht][2] = s[ht][3] = -INFINITY;
      }
    }
    // ---- online softmax per query head (columns 2 tq and 2 tq + 1), reduced over the 16 keys
    uint32_t pb[NTH][2];
    bool resc = false;
    float al[NTH][2];
#pragma unroll
    for (int ht = 0; ht < NTH; ++ht) {
      float ma = fmaxf(s[ht][0], s[ht][2]), mb = fmaxf(s[ht][1], s[ht][3]);
#pragma unroll
      for (int x = 4; x < 32; x <<= 1) {
        ma = fmaxf(ma, __shfl_xor_sync(0xffffffffu, ma, x));
        mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, x));
      }
      const float na = fmaxf(mrun[ht][0], ma * sl2), nb = fmaxf(mrun[ht][1], mb * sl2);
      al[ht][0] = fast_exp2(mrun[ht][0] - na);
      al[ht][1] = fast_exp2(mrun[ht][1] - nb);
      mrun[ht][0] = na;
      mrun[ht][1] = nb;
      const float p0 = fast_exp2(fmaf(s[ht][0], sl2, -na)), p1 = fast_exp2(fmaf(s[ht][1], sl2, -nb));
      const float p2 = fast_exp2(fmaf(s[ht][2], sl2, -na)), p3 = fast_exp2(fmaf(s[ht][3], sl2, -nb));
      lrun[ht][0] = lrun[ht][0] * al[ht][0] + (p0 + p2);
      lrun[ht][1] = lrun[ht][1] * al[ht][1] + (p1 + p3);
      resc |= (al[ht][0] != 1.f) || (al[ht][1] != 1.f);
      pb[ht][0] = movm_trans(pack_bf16x2(p0, p1));  // keys 0-7:  B[k = 2tq, 2tq+1][n = g]
      pb[ht][1] = movm_trans(pack_bf16x2(p2, p3));  // keys 8-15
    }
    // alpha is exactly 1 while the running max stands (the common case): skip the rescale then
    if (__any_sync(0xffffffffu, resc)) {
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int ht = 0; ht < NTH; ++ht) {
          o[mt][ht][0] *= al[ht][0];
          o[mt][ht][1] *= al[ht][1];
          o[mt][ht][2] *= al[ht][0];
          o[mt][ht][3] *= al[ht][1];
        }
    }
    // ---- O^T += V^T P^T
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      uint32_t va[4];
      if constexpr (kPreload) {
        va[0] = vf[mt][0];
        va[1] = vf[mt][1];
        va[2] = vf[mt][2];
        va[3] = vf[mt][3];
      } else {
        const int chunk = 2 * mt + v_csel;
        ldsm_x4_t(sw128(vst + (chunk >> 3) * SM::kHalfBytes, v_row, chunk & 7), va[0],
                  va[1], va[2], va[3]);
      }
#pragma unroll
      for (int ht = 0; ht < NTH; ++ht) mma_bf16_16816(o[mt][ht], va, pb[ht][0], pb[ht][1]);
    }
    if constexpr (!kPreload) {
      if (tail) fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_empty + 8 * stage);
    }

    if (si.flags & kInfoLast) {
      // A split part: read its counter now (acquire), so that the value is in by the time the
      // part is written.  If every other part has counted already, this warp is the last and
      // merges without an atomic of its own.
      int peek = -1;
      if (!(si.flags & kInfoComplete) && lane == 0)
        asm volatile("ld.acquire.gpu.global.s32 %0, [%1];"
                     : "=r"(peek)
                     : "l"(merge_cnt + ((size_t)si.dec * a.Hkv + kvh) * QS + warp % QS)
                     : "memory");
#pragma unroll
      for (int ht = 0; ht < NTH; ++ht) {
        float la = lrun[ht][0], lb = lrun[ht][1];
#pragma unroll
        for (int x = 4; x < 32; x <<= 1) {
          la += __shfl_xor_sync(0xffffffffu, la, x);
          lb += __shfl_xor_sync(0xffffffffu, lb, x);
        }
        const int ha = qoff + ht * 8 + 2 * tq, hb = ha + 1;  // query heads (within the group) of my columns
        if (si.flags & kInfoComplete) {
          const float ia = 1.f / la, ib = 1.f / lb;
          const int hrow = qoff + ht * 8 + g;  // after the transpose a thread holds query head g
          uint32_t* orow = reinterpret_cast<uint32_t*>(
              outg + ((size_t)si.tok * a.Hq + kvh * a.G + hrow) * D);
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            const uint32_t lo = movm_trans(pack_bf16x2(o[mt][ht][0] * ia, o[mt][ht][1] * ib));
            const uint32_t hi = movm_trans(pack_bf16x2(o[mt][ht][2] * ia, o[mt][ht][3] * ib));
            if (hrow < a.G) {
              orow[(16 * mt + 2 * tq) / 2] = lo;
              orow[(16 * mt + 8 + 2 * tq) / 2] = hi;
            }
          }
          if (a.lse != nullptr && g == 0) {
            if (ha < a.G) a.lse[(size_t)si.tok * a.Hq + kvh * a.G + ha] = (mrun[ht][0] + __log2f(la)) * 0.6931471805599453f;
            if (hb < a.G) a.lse[(size_t)si.tok * a.Hq + kvh * a.G + hb] = (mrun[ht][1] + __log2f(lb)) * 0.6931471805599453f;
          }
        } else {
          const size_t slot = (size_t)c + si.dec;
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            if (ha < a.G) {
              float* po = part_o + (slot * a.Hq + kvh * a.G + ha) * D + 16 * mt + g;
              po[0] = o[mt][ht][0];
              po[8] = o[mt][ht][2];
            }
            if (hb < a.G) {
              float* po = part_o + (slot * a.Hq + kvh * a.G + hb) * D + 16 * mt + g;
              po[0] = o[mt][ht][1];
              po[8] = o[mt][ht][3];
            }
          }
          if (g == 0) {
            if (ha < a.G) part_ml[slot * a.Hq + kvh * a.G + ha] = make_float2(mrun[ht][0], la);
            if (hb < a.G) part_ml[slot * a.Hq + kvh * a.G + hb] = make_float2(mrun[ht][1], lb);
          }
        }
      }
      if (!(si.flags & kInfoComplete)) {
        // Split sequence: the last warp to finish this (sequence, KV head, group of 8 query
        // heads) merges the group's parts.
        const int cf = cta_of_tile(si.p0, ntiles, N), cl = cta_of_tile(si.p1 - 1, ntiles, N);
        // one counter per (sequence, KV head, group of 8 query heads): with QS warps per KV
        // head, the last warp of each group merges that group's heads, the groups in parallel.
        // Counts only grow, so a counter already at parts - 1 leaves this warp the last (the
        // fence makes its own part, read back through L2, visible to all its lanes).
        int last = __shfl_sync(0xffffffffu, peek, 0) == cl - cf ? 1 : 0;
        if (last) {
          __threadfence();
          __syncwarp();
        } else {
          __threadfence();
          __syncwarp();
          if (lane == 0)
            last = atomicAdd(merge_cnt + ((size_t)si.dec * a.Hkv + kvh) * QS + warp % QS, 1) ==
                   cl - cf;
          last = __shfl_sync(0xffffffffu, last, 0);
          if (last) __threadfence();
        }
        if (last)
          merge_parts<D>(a, part_ml, part_o, si.dec, si.tok, kvh, cf, cl, qoff,
                         qoff + 8 < a.G ? qoff + 8 : a.G, lane);
      }
    }
  }
}

// The producer warp of a decode CTA (see decode_cta): walks the CTA's tile range and issues
// the TMA copies of every tile's page runs into the stage ring.
template <int D, int QS>
__device__ __forceinline__ void decode_produce(const AttnArgs& a, const CUtensorMap* kmap,
                                               const CUtensorMap* vmap, uint32_t sbase,
                                               uint32_t bar_full, uint32_t bar_empty,
                                               StageInfo* info, const PlanHeader* hdr,
                                               const int4* dec_rec, int d_first, int c, int hg,
                                               int HB, long long t0, long long t1, int lane) {
  using SM = DecodeSmem<D, QS>;
    // ===================================================================== producer warp
  if (lane == 0) {
    tma_prefetch_desc(kmap);
    tma_prefetch_desc(vmap);
  }
  const int KB = a.KB;
  const int nsb = kDecodeTileKeys / KB;        // page runs (TMA boxes per half and K/V) per tile
  const uint64_t stream_policy = l2_policy_evict_first();  // each K/V row is read once
  const int tiles_per_batch = 32 / nsb;
  int d = d_first;
  long long t = t0;
  long long it = 0;
  bool abort = false;
  while (t < t1 && !abort) {
    if (d >= hdr->n_dec) { report(a.err, kErrOutOfRange); break; }
    // one round trip for the sequence's metadata (the next record's first tile ends its range)
    const int4 rec = dec_rec[d];
    const long long p0 = rec.w, p1 = dec_rec[d + 1].w;
    const int s = rec.x, tok = rec.y, kv = rec.z;
    // with a sliding window the sequence's tiles start at the one holding its first key
    const int lo_key = window_first_key(kv - 1, a.window);
    const int first_tile_key = lo_key / kDecodeTileKeys * kDecodeTileKeys;
    const long long lo = t > p0 ? t : p0;
    const long long hi = t1 < p1 ? t1 : p1;
    const bool complete = p0 >= t0 && p1 <= t1;
    const int32_t* row = a.block_table + (size_t)s * a.max_blocks;
    // The consumers read this sequence's query rows (the CTA's head group) at its first tile,
    // a few stages from now: pull them into L2 so that the read does not wait on HBM.
    if (lane == 0)
      l2_prefetch_bulk(static_cast<const __nv_bfloat16*>(a.q) +
                           ((size_t)tok * a.Hq + (size_t)hg * decode_kv_heads<QS>() * a.G) * D,
                       (uint32_t)(HB * a.G * D * 2));
    for (long long tb = lo; tb < hi && !abort; tb += tiles_per_batch) {
      // Prefetch the block-table entries of up to 32 (tile, sub-box) pairs.
      int entry = -1;
      {
        const long long tile = tb + lane / nsb;
        const int pos = first_tile_key + (int)(tile - p0) * kDecodeTileKeys + (lane % nsb) * KB;
        if (lane < tiles_per_batch * nsb && tile < hi && pos < kv) {
          const int lb = pos / a.bs;
          entry = lb < a.max_blocks ? __ldg(row + lb) : -2;
        }
      }
      const int nb = (int)((hi - tb) < tiles_per_batch ? (hi - tb) : tiles_per_batch);
      for (int tl = 0; tl < nb; ++tl, ++it) {
        const long long tile = tb + tl;
        const int stage = (int)(it % SM::kStages);
        const uint32_t phase = (uint32_t)((it / SM::kStages) & 1);
        if (lane == 0 && !mbar_wait(bar_empty + 8 * stage, phase ^ 1)) {
          report(a.err, kErrTimeout);
          abort = true;
        }
        abort = __shfl_sync(0xffffffffu, abort, 0);
        if (abort) break;
        const int key0 = first_tile_key + (int)(tile - p0) * kDecodeTileKeys;
        // One TMA box per (page run sb, half of D, K or V) covers all HB heads of the run:
        // lane sb handles run sb (nsb <= 16 runs per tile).
        const int e = __shfl_sync(0xffffffffu, entry, tl * nsb + (lane < nsb ? lane : 0));
        const int pos = key0 + lane * KB;
        const bool want = lane < nsb && pos < kv;
        const bool valid = want && e >= 0 && e < a.P;
        if (want && !valid) report(a.err, kErrOutOfRange);
        const uint32_t nvalid = __popc(__ballot_sync(0xffffffffu, valid));
        if (lane == 0) {
          StageInfo& si = info[stage];
          si.seq = s;
          si.dec = d;
          si.tok = tok;
          si.kv = kv;
          si.lo = lo_key;
          si.key0 = key0;
          si.p0 = (int)p0;
          si.p1 = (int)p1;
          si.flags = (tile == lo ? kInfoFirst : 0u) | (tile == hi - 1 ? kInfoLast : 0u) |
                     (complete ? kInfoComplete : 0u);
          mbar_arrive_expect_tx(bar_full + 8 * stage,
                                nvalid * (uint32_t)(2 * SM::kHalves * KB * HB * 128));
        }
        __syncwarp();
        if (valid) {
          const int token = e * a.bs + (pos % a.bs);
          const uint32_t kst = sbase + stage * SM::kStageBytes;
          const uint32_t vst = kst + SM::kKVBytes;
          const uint32_t off = (uint32_t)(lane * HB * KB * 128);  // run sb: [HB heads][KB keys]
#pragma unroll
          for (int half = 0; half < SM::kHalves; ++half) {
            tma_load_3d_hint(kst + half * SM::kHalfBytes + off, kmap, bar_full + 8 * stage,
                             half * 64, token, hg * decode_kv_heads<QS>(), stream_policy);
            tma_load_3d_hint(vst + half * SM::kHalfBytes + off, vmap, bar_full + 8 * stage,
                             half * 64, token, hg * decode_kv_heads<QS>(), stream_policy);
          }
        }
      }
    }
    t = hi;
    ++d;
  }
}

// One CTA of the decode pass: CTA `bx` of the a.decode_ctas CTAs of KV-head group `hg`
// (decode_kv_heads<QS>() KV heads per group).  Runs in the attention kernel (cb_attention.cu)
// with that kernel's dynamic shared memory; uses 32 * (QS * HB + 1) of its threads.
template <int D, int QS>
__device__ __forceinline__ void decode_cta(const AttnArgs& a, const CUtensorMap* kmap,
                                           const CUtensorMap* vmap, uint8_t* smem_raw, int bx,
                                           int hg) {
  using SM = DecodeSmem<D, QS>;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar_full = sbase + SM::kBarOffset;              // kStages x 8 B
  const uint32_t bar_empty = bar_full + SM::kStages * 8;         // kStages x 8 B
  StageInfo* info = reinterpret_cast<StageInfo*>(smem + SM::kInfoOffset);

  const int HB = a.Hkv < decode_kv_heads<QS>() ? a.Hkv : decode_kv_heads<QS>();
  const int n_cons = QS * HB;  // consumer warps; the producer is warp n_cons
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const WsLayout L = ws_layout(a.S, a.T, a.Hq, a.D);
  const PlanHeader* hdr = reinterpret_cast<const PlanHeader*>(a.ws + L.header);
  const int4* dec_rec = reinterpret_cast<const int4*>(a.ws + L.dec_rec);
  const int32_t* cta_first = reinterpret_cast<const int32_t*>(a.ws + L.cta_first);

  // The first sequence comes from the planner's per-grid-CTA table, read in the same round trip
  // as the header (neither depends on the other).
  const int d_first = cta_first[bx];
  const long long ntiles = hdr->dec_tiles;
  const int N = hdr->decode_ctas;  // planner's CTA count: <= a.decode_ctas, every range non-empty
  const int c = decode_cta_index(bx, N, a.decode_ctas);
  if (c < 0 || d_first < 0) return;
  const long long t0 = ntiles * c / N, t1 = ntiles * (c + 1) / N;
  if (t0 >= t1) return;

  if (threadIdx.x == 0) {
    for (int i = 0; i < SM::kStages; ++i) {
      mbar_init(bar_full + 8 * i, 1);
      mbar_init(bar_empty + 8 * i, n_cons);
    }
    fence_barrier_init();
  }
  __syncthreads();

  auto produce = [&]() {
    decode_produce<D, QS>(a, kmap, vmap, sbase, bar_full, bar_empty, info, hdr, dec_rec, d_first,
                          c, hg, HB, t0, t1, lane);
  };
  auto consume = [&]() {
    decode_consume<D, QS>(a, sbase, bar_full, bar_empty, info, c, hg, warp, t1 - t0, ntiles, N,
                           L, lane);
  };
  if (warp == n_cons) produce();
  else if (warp < n_cons) consume();
}

}  // namespace cb
