// Paged KV-append: scatter this step's K/V rows into their cache slots, and the batch planner
// of the attention pass.
//
// Slot rule ("LLM learning path 3.3 Batching & Memory Management", section "PagedAttention:
// block tables"): token position p of a sequence lives in physical block table[p / bs] at
// offset p % bs; with the token-major pool of "Continuous batching in transformers"
// (paged-cache section) that is row table[p / bs] * bs + p % bs of the flattened
// [P * bs, Hkv, D] tensor.  Token i of sequence s has position kv_len_s - q_len_s + i.
#include "cb_common.cuh"
#include "cb_launch.h"

namespace cb {

// One warp per new token: the warp finds the token's sequence with 32-way probes of
// cu_seqlens_q (a few rounds instead of a binary search per 16-byte chunk), then each lane
// moves its share of the token's K row and V row (all KV heads: Hkv * D bf16, contiguous in
// both the input and the token-major pool), issuing every load before the first store.
constexpr int kAppendThreads = 256;
constexpr int kAppendMaxChunks = 8;  // 16-byte chunks per lane and tensor in flight

// Tokens handled by warps first_warp, first_warp + nwarps, ...  kMaxChunks: 16-byte chunks per
// lane and tensor in flight (registers: 8 per chunk pair).
template <int kMaxChunks>
__device__ __forceinline__ void append_tokens(const AppendArgs& a, int first_warp, int nwarps) {
  const int lane = threadIdx.x & 31;
  const int cpr = a.Hkv * a.D / 8;  // 16-byte chunks per token row
  const uint4* kn = static_cast<const uint4*>(a.k_new);
  const uint4* vn = static_cast<const uint4*>(a.v_new);
  uint4* kp = static_cast<uint4*>(a.k_pages);
  uint4* vp = static_cast<uint4*>(a.v_pages);
  // Rows at or past cu_seqlens_q[S] are padding of the token tensors: left untouched.
  const int t_end = min(a.T, __ldg(a.cu_seqlens_q + a.S));
  for (int t = first_warp; t < t_end; t += nwarps) {
    // Sequence of token t: the last s with cu[s] <= t (cu is non-decreasing).  Each round
    // probes 32 increasing positions in (lo, hi]; the lanes whose probe is <= t form a prefix.
    int lo = 0, hi = a.S;
    while (lo < hi) {
      const int span = hi - lo;
      const int p = lo + 1 + (int)((long long)(span - 1) * lane / 31);
      const unsigned le = __ballot_sync(0xffffffffu, __ldg(a.cu_seqlens_q + p) <= t);
      const int k = le ? 31 - __clz(le) : -1;
      const int pk = __shfl_sync(0xffffffffu, p, k < 0 ? 0 : k);
      const int pn = __shfl_sync(0xffffffffu, p, k < 31 ? k + 1 : 31);
      if (k < 0) {
        hi = pk - 1;
      } else {
        lo = pk;
        if (k < 31 && pn - 1 < hi) hi = pn - 1;
      }
    }
    const int s = lo;
    if (s >= a.S) {
      if (lane == 0) report(a.err, kErrOutOfRange);
      continue;
    }
    const int c0 = __ldg(a.cu_seqlens_q + s), c1 = __ldg(a.cu_seqlens_q + s + 1);
    const int q_len = c1 - c0;
    const int kv = __ldg(a.kv_lens + s);
    if (t < c0 || t >= c1 || c1 > a.T || kv < q_len) {
      if (lane == 0) report(a.err, kErrOutOfRange);
      continue;
    }
    const int pos = kv - q_len + (t - c0);
    const int lb = pos / a.bs;
    if (lb >= a.max_blocks) {
      if (lane == 0) report(a.err, kErrOutOfRange);
      continue;
    }
    const int blk = __ldg(a.block_table + (size_t)s * a.max_blocks + lb);
    if (blk < 0 || blk >= a.P) {
      if (lane == 0) report(a.err, kErrOutOfRange);
      continue;
    }
    const long long slot = (long long)blk * a.bs + (pos - lb * a.bs);
    const uint4* ks = kn + (size_t)t * cpr;
    const uint4* vs = vn + (size_t)t * cpr;
    uint4* kd = kp + (size_t)slot * cpr;
    uint4* vd = vp + (size_t)slot * cpr;
    for (int base = 0; base < cpr; base += 32 * kMaxChunks) {
      uint4 kr[kMaxChunks], vr[kMaxChunks];
#pragma unroll
      for (int i = 0; i < kMaxChunks; ++i) {
        const int c = base + lane + 32 * i;
        if (c < cpr) {
          kr[i] = __ldg(ks + c);
          vr[i] = __ldg(vs + c);
        }
      }
#pragma unroll
      for (int i = 0; i < kMaxChunks; ++i) {
        const int c = base + lane + 32 * i;
        if (c < cpr) {
          kd[c] = kr[i];
          vd[c] = vr[i];
        }
      }
    }
  }
}

// Checks of cu_seqlens_q that no token's own search sees (cu[0] = 0, non-decreasing,
// cu[S] <= T), spread over the grid's threads: a token of a malformed range may land in a
// neighbouring sequence's range, so the stand-alone append reports the metadata itself.  (The
// append + planner launch leaves this to the planner, which makes the same checks.)
__device__ __forceinline__ void check_cu_seqlens(const AppendArgs& a) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < a.S; i += gridDim.x * blockDim.x) {
    const int c0 = __ldg(a.cu_seqlens_q + i), c1 = __ldg(a.cu_seqlens_q + i + 1);
    if (c1 < c0 || (i == 0 && c0 != 0) || (i == a.S - 1 && c1 > a.T)) report(a.err, kErrOutOfRange);
  }
}

__global__ void __launch_bounds__(kAppendThreads) kv_append_kernel(AppendArgs a) {
  check_cu_seqlens(a);
  append_tokens<kAppendMaxChunks>(a, blockIdx.x * (kAppendThreads / 32) + (threadIdx.x >> 5),
                                  gridDim.x * (kAppendThreads / 32));
}

cudaError_t launch_kv_append(const AppendArgs& a, cudaStream_t stream) {
  if (a.T == 0) return cudaSuccess;
  const int warps = kAppendThreads / 32;
  long long blocks = ((long long)a.T + warps - 1) / warps;
  if (blocks > 8192) blocks = 8192;
  kv_append_kernel<<<(unsigned)blocks, kAppendThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

// ------------------------------------------------------------------------------------------
// Planner: one CTA classifies every sequence (q_len == 1 -> decode, q_len > 1 -> chunk),
// validates its lengths, and writes the compacted lists and prefix sums the attention passes
// read.  Nothing returns to the host.

constexpr int kPlanThreads = 1024;

// Exclusive block-wide scan of four counters at once; returns the block totals in tot[].
__device__ __forceinline__ void block_scan4(int v[4], int ex[4], int tot[4], int (*sw)[4]) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int inc[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    int x = v[k];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    inc[k] = x;
  }
  if (lane == 31) {
#pragma unroll
    for (int k = 0; k < 4; ++k) sw[warp][k] = inc[k];
  }
  __syncthreads();
  if (warp == 0) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      int x = sw[lane][k];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      sw[lane][k] = x;  // inclusive over warps
    }
  }
  __syncthreads();
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    ex[k] = inc[k] - v[k] + (warp > 0 ? sw[warp - 1][k] : 0);
    tot[k] = sw[31][k];
  }
  __syncthreads();
}

// Decode CTA count for a batch whose chunk pass runs beside the decode pass.  Model, fitted to
// GB300 measurements of these kernels: decode on N SMs streams its bytes at
// BW(N) = ((0.11 N)^-3 + 6.8^-3)^(-1/3) TB/s (linear in N until HBM saturates), taking td; the
// chunk pass runs at ~6.4 TFLOP/s per SM on the other M SMs meanwhile and on every SM
// afterwards.  Chunk CTAs claim whole items (one query tile of one or two heads against its
// whole key range), so the chunk pass ends on item boundaries: if its work W fits in M SMs
// before td it ends near W/M (plus a short longest-first tail); if not, the items still
// unclaimed when decode ends each take a full item time on the newly free SMs, so the step is
// td + (W - M td)/SMs + about half an item.  The choice is the largest N within 1% of the
// modelled minimum, so that the decode pass keeps its bandwidth where the curve is flat --
// unless the minimum lies where the chunk pass is the longer one: there the model is flat in N
// (decode SM time is about constant while it is not bandwidth-bound) and the measured step
// is shortest with few decode CTAs that still finish early (chunk-heavy batch: N = 24..40
// 0.307 ms, N = 56 0.314 ms), so the choice is the smallest N within 1% whose decode pass
// takes at most a quarter of the step.  Without chunk work all CTAs decode.  Called by one
// full warp; candidates
// N = 4, 8, ... are spread over the lanes, in fp32 (the fp64 rate of this part is far too low
// for even this much arithmetic on one thread).
__device__ int choose_decode_ctas(float dec_bytes, float chunk_flops, int chunk_items,
                                  int max_ctas, long long tiles) {
  const int lane = threadIdx.x & 31;
  if (tiles <= 0) return 1;
  const int cap = (int)(tiles < max_ctas ? tiles : max_ctas);
  if (chunk_flops <= 0.f || chunk_items <= 0) return cap;
  const float w_us = chunk_flops * (1.f / 6.4e6f);  // chunk work in SM-microseconds
  const float item_us = w_us / (float)chunk_items;
  const float b_mb = dec_bytes * 1e-6f;             // decode bytes / 1e6: MB / (TB/s) = us
  const int n_cand = (cap + 3) / 4;
  float t[4], td[4];
  bool chunk_bound[4];
  int n[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int i = lane + 32 * k;
    n[k] = 4 * (i + 1) < cap ? 4 * (i + 1) : cap;
    t[k] = 3.4e38f;
    td[k] = 0.f;
    chunk_bound[k] = false;
    if (i < n_cand) {
      const float lin = 0.11f * n[k], sat = 6.8f;
      const float bw = rcbrtf(1.f / (lin * lin * lin) + 1.f / (sat * sat * sat));
      td[k] = b_mb / bw;
      const int m = max_ctas - n[k];
      const float rest = w_us - (float)m * td[k];  // chunk work not done when decode ends
      chunk_bound[k] = rest > 0.f;
      t[k] = rest <= 0.f ? fmaxf(td[k], w_us / (float)m + 0.15f * item_us)
                         : td[k] + rest / (float)max_ctas + 0.5f * item_us;
    }
  }
  float t_min = fminf(fminf(t[0], t[1]), fminf(t[2], t[3]));
  for (int o = 16; o > 0; o >>= 1) t_min = fminf(t_min, __shfl_xor_sync(0xffffffffu, t_min, o));
  bool min_chunk_bound = false;
#pragma unroll
  for (int k = 0; k < 4; ++k) min_chunk_bound |= (t[k] == t_min && chunk_bound[k]);
  min_chunk_bound = __any_sync(0xffffffffu, min_chunk_bound);
  if (min_chunk_bound) {
    int small = cap + 1;
#pragma unroll
    for (int k = 0; k < 4; ++k)
      if (t[k] <= 1.01f * t_min && td[k] <= 0.25f * t[k]) small = small < n[k] ? small : n[k];
    for (int o = 16; o > 0; o >>= 1) small = min(small, __shfl_xor_sync(0xffffffffu, small, o));
    if (small <= cap) return small;
  }
  int best = 1;
#pragma unroll
  for (int k = 0; k < 4; ++k)
    if (t[k] <= 1.01f * t_min) best = best > n[k] ? best : n[k];
  for (int o = 16; o > 0; o >>= 1) best = max(best, __shfl_xor_sync(0xffffffffu, best, o));
  return best;
}

// Histogram bin of chunk unit g (global index in chunk-sequence order): units that stream
// more K/V tiles get lower bins, so an ascending walk over the bins is longest first.
// With `lens` (shared memory: q_len and prior context of the i-th chunk sequence, interleaved)
// the lengths need no global loads.
__device__ int pf_unit_bin(const AttnArgs& a, const int32_t* pf_seq, const int32_t* pf_prefix,
                           const int2* lens, int n_pf, int g) {
  int lo = 0, hi = n_pf - 1;  // largest i with pf_prefix[i] <= g
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (pf_prefix[mid] <= g) lo = mid; else hi = mid - 1;
  }
  const int u = g - pf_prefix[lo];
  int q_len, ctx;
  if (lens != nullptr) {
    q_len = lens[lo].x;
    ctx = lens[lo].y;
  } else {
    const int s = pf_seq[lo];
    q_len = a.cu_seqlens_q[s + 1] - a.cu_seqlens_q[s];
    ctx = a.kv_lens[s] - q_len;
  }
  const int rows = min((u + 1) * pf_unit_tiles(a.G) * kPrefillTileM, q_len);
  const int first = window_first_key(ctx + u * pf_unit_tiles(a.G) * kPrefillTileM, a.window);
  const int tiles = (ctx + rows + kChunkKeys - 1) / kChunkKeys - first / kChunkKeys;
  return kCostBins - 1 - min(tiles, kCostBins - 1);
}

// Batches of up to this many decode (or chunk) sequences keep the planner's prefix arrays in
// shared memory as well, so its binary searches cost no global round trips.
constexpr int kPlanSmemSeqs = 2048;

__device__ __forceinline__ void plan_cta(const AttnArgs& a) {
  static_assert(kCostBins == kPlanThreads, "one histogram bin per planner thread");
  __shared__ int sw[32][4];
  __shared__ int32_t s_dec_prefix[kPlanSmemSeqs + 1], s_pf_prefix[kPlanSmemSeqs + 1];
  __shared__ int32_t s_pf_seq[kPlanSmemSeqs];
  __shared__ int2 s_pf_lens[kPlanSmemSeqs];  // (q_len, prior context) of each chunk sequence
  const WsLayout L = ws_layout(a.S, a.T, a.Hq, a.D);
  PlanHeader* hdr = reinterpret_cast<PlanHeader*>(a.ws + L.header);
  int32_t* dec_seq = reinterpret_cast<int32_t*>(a.ws + L.dec_seq);
  int32_t* dec_prefix = reinterpret_cast<int32_t*>(a.ws + L.dec_prefix);
  int4* dec_rec = reinterpret_cast<int4*>(a.ws + L.dec_rec);
  int32_t* cta_first = reinterpret_cast<int32_t*>(a.ws + L.cta_first);
  int32_t* pf_seq = reinterpret_cast<int32_t*>(a.ws + L.pf_seq);
  int32_t* pf_prefix = reinterpret_cast<int32_t*>(a.ws + L.pf_prefix);
  const int tid = threadIdx.x;
  const long long max_kv = (long long)a.max_blocks * a.bs;

  float my_keys = 0.f, my_pairs = 0.f;  // work estimates for the decode / chunk balance
  bool bad = false;
  const int unit_rows = pf_unit_tiles(a.G) * kPrefillTileM;
  int carry[4] = {0, 0, 0, 0};
  for (int base = 0; base < a.S; base += kPlanThreads) {
    const int s = base + tid;
    int v[4] = {0, 0, 0, 0};
    int tok = 0, kv = 0;
    if (s < a.S) {
      const int c0 = a.cu_seqlens_q[s], c1 = a.cu_seqlens_q[s + 1];
      const int q_len = c1 - c0;
      kv = a.kv_lens[s];
      tok = c0;
      if (s == 0 && c0 != 0) report(a.err, kErrOutOfRange);  // cu_seqlens_q[0] must be 0
      const bool ok = c0 >= 0 && c1 <= a.T && q_len >= 0 && kv >= q_len && kv <= max_kv;
      if (!ok) {
        report(a.err, kErrOutOfRange);
        bad = true;
      } else if (q_len == 1) {
        // tiles from the one holding the window's first key (every key without a window)
        const int first = window_first_key(kv - 1, a.window) / kDecodeTileKeys * kDecodeTileKeys;
        v[0] = 1;
        v[1] = (kv - first + kDecodeTileKeys - 1) / kDecodeTileKeys;
        my_keys += (float)(kv - window_first_key(kv - 1, a.window));
      } else if (q_len > 1) {
        v[2] = 1;
        if (a.window > 0) {  // sum over the chunk's rows of min(position + 1, window)
          const float W = (float)a.window;
          for (int i = 0; i < q_len; i += 64) {
            const int i1 = min(i + 64, q_len);
            const float p0 = (float)(kv - q_len + i + 1), p1 = (float)(kv - q_len + i1);
            my_pairs += (i1 - i) * fminf(0.5f * (p0 + p1), W);
          }
        } else {
          my_pairs += (float)q_len * (float)(kv - q_len) + 0.5f * (float)q_len * (float)(q_len + 1);
        }
        v[3] = (q_len + unit_rows - 1) / unit_rows;  // work units (pf_unit_tiles)
      }
    }
    int ex[4], tot[4];
    block_scan4(v, ex, tot, sw);
    if (v[0]) {
      const int i = carry[0] + ex[0];
      dec_seq[i] = s;
      dec_prefix[i] = carry[1] + ex[1];
      dec_rec[i] = make_int4(s, tok, kv, carry[1] + ex[1]);
      if (i < kPlanSmemSeqs) s_dec_prefix[i] = carry[1] + ex[1];
    }
    if (v[2]) {
      const int i = carry[2] + ex[2];
      pf_seq[i] = s;
      pf_prefix[i] = carry[3] + ex[3];
      if (i < kPlanSmemSeqs) {
        s_pf_seq[i] = s;
        s_pf_prefix[i] = carry[3] + ex[3];
        const int q_len = a.cu_seqlens_q[s + 1] - a.cu_seqlens_q[s];
        s_pf_lens[i] = make_int2(q_len, a.kv_lens[s] - q_len);
      }
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) carry[k] += tot[k];
  }
  // With every length valid the query ranges are disjoint, so the units fit pf_order (at most
  // S + T / 128); after an invalid length the chunk pass is given no work.
  bad = __syncthreads_or(bad) != 0;
  const int n_pf = carry[2];
  const int n_units = bad ? 0 : carry[3];
  if (tid == 0) {
    dec_prefix[carry[0]] = carry[1];
    dec_rec[carry[0]] = make_int4(-1, 0, 0, carry[1]);
    pf_prefix[carry[2]] = carry[3];
    if (carry[0] <= kPlanSmemSeqs) s_dec_prefix[carry[0]] = carry[1];
    if (carry[2] <= kPlanSmemSeqs) s_pf_prefix[carry[2]] = carry[3];
    hdr->n_dec = carry[0];
    hdr->dec_tiles = carry[1];
    hdr->n_pf = n_pf;
    hdr->pf_qtiles = n_units;
    hdr->pf_counter = 0;
    hdr->t_dec_start = hdr->t_pf_start = ~0ull;
    hdr->t_dec_end = hdr->t_pf_end = 0ull;
  }
  __syncthreads();
  // Chunk units longest first (a counting sort on the K/V tiles each streams, descending), so
  // that the chunk CTAs, taking items in this order from a shared counter, schedule them
  // longest-processing-time first.  Units of equal cost land in any order: each item writes
  // its own output rows, so the order never changes a result.  (n_units is the same in every
  // thread, so a batch without chunk work skips the section, barriers included.)
  if (n_units > 0) {
    __shared__ int hist[kCostBins];
    int32_t* pf_order = reinterpret_cast<int32_t*>(a.ws + L.pf_order);
    hist[tid] = 0;
    __syncthreads();
    const bool pf_local = n_pf <= kPlanSmemSeqs;
    const int32_t* ps = pf_local ? s_pf_seq : pf_seq;
    const int32_t* pp = pf_local ? s_pf_prefix : pf_prefix;
    const int2* lens = pf_local ? s_pf_lens : nullptr;
    for (int g = tid; g < n_units; g += kPlanThreads)
      atomicAdd(&hist[pf_unit_bin(a, ps, pp, lens, n_pf, g)], 1);
    __syncthreads();
    int v[4] = {hist[tid], 0, 0, 0}, ex[4], tot[4];
    block_scan4(v, ex, tot, sw);
    hist[tid] = ex[0];
    __syncthreads();
    for (int g = tid; g < n_units; g += kPlanThreads)
      pf_order[atomicAdd(&hist[pf_unit_bin(a, ps, pp, lens, n_pf, g)], 1)] = g;
  }
  // First decode sequence of each decode CTA: CTA c owns tiles [c*n/N, (c+1)*n/N), with N
  // capped at the tile count so that no CTA range is empty.
  const int n_dec = carry[0];
  const long long ntiles = carry[1];
  __shared__ int s_N;
  __shared__ float s_red[2][kPlanThreads / 32];
  // fixed-order reduction, so that the CTA count (and with it the rounding of the split-KV
  // merge) is the same on every call with the same lengths
  for (int o = 16; o > 0; o >>= 1) {
    my_keys += __shfl_xor_sync(0xffffffffu, my_keys, o);
    my_pairs += __shfl_xor_sync(0xffffffffu, my_pairs, o);
  }
  if ((tid & 31) == 0) {
    s_red[0][tid >> 5] = my_keys;
    s_red[1][tid >> 5] = my_pairs;
  }
  __syncthreads();
  if (tid < 32) {
    float keys = 0.f, pairs = 0.f;
    for (int w = 0; w < kPlanThreads / 32; ++w) {
      keys += s_red[0][w];
      pairs += s_red[1][w];
    }
    int n = (int)(ntiles < a.decode_ctas ? (ntiles > 0 ? ntiles : 1) : a.decode_ctas);
    if (a.decode_auto)
      n = choose_decode_ctas(keys * (float)(a.Hkv * a.D * 4), pairs * (float)(4 * a.D * a.Hq),
                             n_units * (pf_pair_heads(a.G) ? a.Hq / 2 : a.Hq), a.decode_ctas,
                             ntiles);
    if (tid == 0) {
      s_N = n;
      hdr->decode_ctas = n;
    }
  }
  __syncthreads();
  const int N = s_N;
  // Merge counters of the decode pass: one per (decode sequence, KV head), zero at start.
  int32_t* merge_cnt = reinterpret_cast<int32_t*>(a.ws + L.merge_cnt);
  // (one per decode sequence, KV head and group of 8 query heads: two groups when G > 8)
  const int head_groups = a.G > 8 ? 2 : 1;
  for (int i = tid; i < n_dec * a.Hkv * head_groups; i += kPlanThreads) merge_cnt[i] = 0;
  // Indexed by the grid's decode CTA, so that a CTA reads its first sequence in the same round
  // trip as the plan header.
  const int32_t* dp = n_dec <= kPlanSmemSeqs ? s_dec_prefix : dec_prefix;
  for (int bx = tid; bx < a.decode_ctas; bx += kPlanThreads) {
    const int c = decode_cta_index(bx, N, a.decode_ctas);
    int lo = -1;
    if (c >= 0 && c < N) {
      const long long t0 = ntiles * c / N;
      lo = 0;
      int hi = n_dec;  // largest d in [0, n_dec] with dec_prefix[d] <= t0
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (dp[mid] <= t0) lo = mid; else hi = mid - 1;
      }
    }
    cta_first[bx] = lo;
  }
}

// Both planner launches let the attention kernel that follows them on the stream start early
// (it is launched as their programmatic dependent and waits for their completion itself).
__device__ __forceinline__ void allow_dependent_launch() {
  asm volatile("griddepcontrol.launch_dependents;");
}

__global__ void __launch_bounds__(kPlanThreads, 1) plan_kernel(AttnArgs a) {
  allow_dependent_launch();
  plan_cta(a);
}

cudaError_t launch_plan(const AttnArgs& a, cudaStream_t stream) {
  plan_kernel<<<1, kPlanThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

// CTA 0 plans the attention pass (it reads only the metadata); CTAs 1.. append this step's
// K/V rows, one warp per token, 32 tokens per CTA at a time.
constexpr int kAppendPlanMaxChunks = 4;  // fits the 64 registers of a 1024-thread CTA
__global__ void __launch_bounds__(kPlanThreads, 1) append_plan_kernel(AppendArgs ap, AttnArgs a) {
  allow_dependent_launch();
  if (blockIdx.x == 0) {
    plan_cta(a);
  } else {
    constexpr int kWarps = kPlanThreads / 32;
    append_tokens<kAppendPlanMaxChunks>(ap, (blockIdx.x - 1) * kWarps + (threadIdx.x >> 5),
                                        (gridDim.x - 1) * kWarps);
  }
}

cudaError_t launch_append_plan(const AppendArgs& ap, const AttnArgs& a, cudaStream_t stream) {
  constexpr int kWarps = kPlanThreads / 32;
  long long blocks = ((long long)ap.T + kWarps - 1) / kWarps;
  if (blocks > 2048) blocks = 2048;
  if (blocks < 1) blocks = 1;
  append_plan_kernel<<<(unsigned)(1 + blocks), kPlanThreads, 0, stream>>>(ap, a);
  return cudaGetLastError();
}

}  // namespace cb
