// Chunk pass of ragged paged attention: sequences with q_len > 1 (chunked prefill).  "The
// prefill chunks make the iteration compute-bound" ("LLM learning path 3.3 Batching & Memory
// Management", section "Chunked prefill"), so this pass runs on the 5th-generation tensor
// cores.  A chunk of queries attends to a cache that already holds the earlier chunks: query i
// of a chunk with prior context ctx sees keys 0 .. ctx + i (same section).
//
// One work item = (chunk sequence, 128-query tile, query head).  Persistent CTAs (one per SM)
// take items from a device counter the planner reset.  Per CTA, warp-specialised:
//   warp 0      TMA producer: the Q tile once per item, then K and V tiles of 128 keys gathered
//               page run by page run through the block table into a 2-stage smem ring
//               (128-byte swizzle, the layout the tensor core descriptors read directly).
//   warp 1      tcgen05 issuer (one thread): S_j = Q K_j^T into one of two TMEM buffers, then
//               O += P_j V_j with P_j read from TMEM; completion is signalled through
//               tcgen05.commit on mbarriers.  Also owns the TMEM allocation.
//   warps 2-5   softmax: thread r owns query row r (TMEM lane r); it loads its 128 scores
//               with tcgen05.ld, applies the causal mask only on tiles that cross the diagonal,
//               keeps the running max m and sum l in registers, writes P (bf16) back over S,
//               and rescales O in TMEM only when m grows by more than 2^8 (otherwise the stale
//               max keeps every p <= 256, which fp32 and bf16 represent exactly as well); the
//               final O / l is written as bf16.
// TMEM columns: [0,128) S/P buffer 0, [128,256) S/P buffer 1, [256, 256+D) O.
#include "cb_common.cuh"
#include "cb_launch.h"

namespace cb {

template <int D>
struct PrefillSmem {
  static constexpr int kHalves = D / 64;
  static constexpr int kHalfBytes = 128 * 128;             // 128 rows of 128 B
  static constexpr int kTileBytes = kHalves * kHalfBytes;  // a Q, K or V tile
  static constexpr int kStages = (D == 128) ? 2 : 4;
  static constexpr int kQ = 0;
  static constexpr int kStage0 = kTileBytes;               // stage i: K at +0, V at +kTileBytes
  static constexpr int kBar = kStage0 + kStages * 2 * kTileBytes;
  // barrier indices (8 bytes each)
  static constexpr int bQFull = 0, bQEmpty = 1, bKFull = 2, bVFull = bKFull + kStages,
                       bKVEmpty = bVFull + kStages, bSFull = bKVEmpty + kStages,
                       bPFull = bSFull + 2, bODone = bPFull + 2, bOFree = bODone + 1,
                       bItemFull = bOFree + 1, bItemEmpty = bItemFull + 2,
                       kNumBars = bItemEmpty + 2;
  static constexpr int kMisc = kBar + kNumBars * 8;        // tmem base, item ids
  static constexpr int kTotal = kMisc + 64 + 1024;
};

constexpr uint32_t kTmemCols = 512;
constexpr int kPrefillThreads = 192;

struct PfItem {
  int s, tok0, rows, ctx, head, kvh, qt, n_keys, n_tiles;
};

__device__ __forceinline__ PfItem pf_decode_item(int item, const AttnArgs& a,
                                                 const int32_t* pf_seq, const int32_t* pf_prefix,
                                                 int n_pf) {
  PfItem it;
  const int qtg = item / a.Hq;
  it.head = item - qtg * a.Hq;
  it.kvh = it.head / a.G;
  int lo = 0, hi = n_pf - 1;  // largest i with pf_prefix[i] <= qtg
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (pf_prefix[mid] <= qtg) lo = mid; else hi = mid - 1;
  }
  it.s = pf_seq[lo];
  const int c0 = a.cu_seqlens_q[it.s];
  const int q_len = a.cu_seqlens_q[it.s + 1] - c0;
  const int kv = a.kv_lens[it.s];
  it.ctx = kv - q_len;
  const int nqt = pf_prefix[lo + 1] - pf_prefix[lo];
  it.qt = nqt - 1 - (qtg - pf_prefix[lo]);  // longest tiles of a chunk first
  it.rows = min(kPrefillTileM, q_len - it.qt * kPrefillTileM);
  it.tok0 = c0 + it.qt * kPrefillTileM;
  it.n_keys = it.ctx + it.qt * kPrefillTileM + it.rows;
  it.n_tiles = (it.n_keys + kPrefillTileN - 1) / kPrefillTileN;
  return it;
}

template <int D>
__global__ void __launch_bounds__(kPrefillThreads, 1)
    prefill_kernel(const AttnArgs a, const __grid_constant__ CUtensorMap qmap,
                   const __grid_constant__ CUtensorMap kmap,
                   const __grid_constant__ CUtensorMap vmap) {
  using SM = PrefillSmem<D>;
  constexpr int NS = SM::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return sbase + SM::kBar + 8 * i; };
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + SM::kMisc);
  volatile int* item_ids = reinterpret_cast<volatile int*>(smem + SM::kMisc + 16);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const WsLayout L = ws_layout(a.S, a.Hq, a.D);
  PlanHeader* hdr = reinterpret_cast<PlanHeader*>(a.ws + L.header);
  const int32_t* pf_seq = reinterpret_cast<const int32_t*>(a.ws + L.pf_seq);
  const int32_t* pf_prefix = reinterpret_cast<const int32_t*>(a.ws + L.pf_prefix);
  const int n_pf = hdr->n_pf;
  const int n_items = hdr->pf_qtiles * a.Hq;
  if (n_items == 0) return;

  if (threadIdx.x == 0) {
    mbar_init(bar(SM::bQFull), 1);
    mbar_init(bar(SM::bQEmpty), 1);
    for (int i = 0; i < NS; ++i) {
      mbar_init(bar(SM::bKFull + i), 1);
      mbar_init(bar(SM::bVFull + i), 1);
      mbar_init(bar(SM::bKVEmpty + i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(SM::bSFull + i), 1);
      mbar_init(bar(SM::bPFull + i), 128);
      mbar_init(bar(SM::bItemFull + i), 1);
      mbar_init(bar(SM::bItemEmpty + i), 5);
    }
    mbar_init(bar(SM::bODone), 1);
    mbar_init(bar(SM::bOFree), 128);
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(const_cast<uint32_t*>(tmem_slot)), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ===================================================================== TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&qmap);
      tma_prefetch_desc(&kmap);
      tma_prefetch_desc(&vmap);
    }
    const int KB = a.KB;
    const int nsb = kPrefillTileN / KB;  // page-run boxes per 128-key tile
    uint32_t g = 0;
    for (uint32_t k = 0;; ++k) {
      const int slot = k & 1;
      int item = -1;
      if (lane == 0) {
        if (!mbar_wait(bar(SM::bItemEmpty + slot), ((k >> 1) & 1) ^ 1)) report(a.err, kErrTimeout);
        item = atomicAdd(&hdr->pf_counter, 1);
        if (item >= n_items) item = -1;
        item_ids[slot] = item;
        mbar_arrive(bar(SM::bItemFull + slot));
      }
      item = __shfl_sync(0xffffffffu, item, 0);
      if (item < 0) break;
      const PfItem it = pf_decode_item(item, a, pf_seq, pf_prefix, n_pf);
      if (lane == 0) {
        if (!mbar_wait(bar(SM::bQEmpty), (k & 1) ^ 1)) report(a.err, kErrTimeout);
        mbar_arrive_expect_tx(bar(SM::bQFull), SM::kTileBytes);
#pragma unroll
        for (int half = 0; half < SM::kHalves; ++half)
          tma_load_3d(sbase + SM::kQ + half * SM::kHalfBytes, &qmap, bar(SM::bQFull), half * 64,
                      it.head, it.tok0);
      }
      const int32_t* row = a.block_table + (size_t)it.s * a.max_blocks;
      for (int j = 0; j < it.n_tiles; ++j, ++g) {
        const int stage = g % NS;
        const uint32_t phase = (g / NS) & 1;
        const int key0 = j * kPrefillTileN;
        // Block-table entries of this tile's page runs (loaded before the wait so the load
        // latency overlaps it).
        int ent[4];
#pragma unroll
        for (int p = 0; p < 4; ++p) {
          const int sb = p * 32 + lane;
          const int pos = key0 + sb * KB;
          ent[p] = -1;
          if (sb < nsb && pos < it.n_keys) {
            const int lb = pos / a.bs;
            ent[p] = lb < a.max_blocks ? __ldg(row + lb) : -2;
          }
        }
        uint32_t nvalid = 0;
#pragma unroll
        for (int p = 0; p < 4; ++p) {
          const int sb = p * 32 + lane;
          const bool want = sb < nsb && key0 + sb * KB < it.n_keys;
          const bool valid = want && ent[p] >= 0 && ent[p] < a.P;
          if (want && !valid) report(a.err, kErrOutOfRange);
          nvalid += __popc(__ballot_sync(0xffffffffu, valid));
        }
        if (lane == 0) {
          if (!mbar_wait(bar(SM::bKVEmpty + stage), phase ^ 1)) report(a.err, kErrTimeout);
          const uint32_t bytes = nvalid * (uint32_t)(SM::kHalves * KB * 128);
          mbar_arrive_expect_tx(bar(SM::bKFull + stage), bytes);
          mbar_arrive_expect_tx(bar(SM::bVFull + stage), bytes);
        }
        __syncwarp();
        const uint32_t kst = sbase + SM::kStage0 + stage * 2 * SM::kTileBytes;
        const uint32_t vst = kst + SM::kTileBytes;
#pragma unroll
        for (int p = 0; p < 4; ++p) {
          const int sb = p * 32 + lane;
          const int pos = key0 + sb * KB;
          if (sb < nsb && pos < it.n_keys && ent[p] >= 0 && ent[p] < a.P) {
            const int token = ent[p] * a.bs + (pos % a.bs);
#pragma unroll
            for (int half = 0; half < SM::kHalves; ++half) {
              tma_load_3d(kst + half * SM::kHalfBytes + sb * KB * 128, &kmap,
                          bar(SM::bKFull + stage), half * 64, it.kvh, token);
              tma_load_3d(vst + half * SM::kHalfBytes + sb * KB * 128, &vmap,
                          bar(SM::bVFull + stage), half * 64, it.kvh, token);
            }
          }
        }
      }
    }
  } else if (warp == 1) {
    // ===================================================================== tcgen05 issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16(kPrefillTileM, kPrefillTileN, 0);
      constexpr uint32_t idesc_o = idesc_bf16(kPrefillTileM, D, 1);
      const uint32_t t_o = tmem + 256;
      uint32_t g = 0;
      bool ok = true;
      auto issue_s = [&](uint32_t gg) {
        const int stage = gg % NS;
        if (!mbar_wait(bar(SM::bKFull + stage), (gg / NS) & 1)) { report(a.err, kErrTimeout); ok = false; }
        tc_fence_after();
        const uint32_t kst = sbase + SM::kStage0 + stage * 2 * SM::kTileBytes;
        const uint32_t d_s = tmem + (gg & 1) * 128;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * SM::kHalfBytes + (kk & 3) * 32;
          tc_mma_ss(d_s, smem_desc_sw128(sbase + SM::kQ + off, 16, 1024),
                    smem_desc_sw128(kst + off, 16, 1024), idesc_s, kk > 0 ? 1u : 0u);
        }
        tc_commit(bar(SM::bSFull + (gg & 1)));
      };
      for (uint32_t k = 0; ok; ++k) {
        const int slot = k & 1;
        if (!mbar_wait(bar(SM::bItemFull + slot), (k >> 1) & 1)) { report(a.err, kErrTimeout); break; }
        const int item = item_ids[slot];
        mbar_arrive(bar(SM::bItemEmpty + slot));
        if (item < 0) break;
        const PfItem it = pf_decode_item(item, a, pf_seq, pf_prefix, n_pf);
        if (!mbar_wait(bar(SM::bQFull), k & 1)) { report(a.err, kErrTimeout); break; }
        tc_fence_after();
        issue_s(g);
        for (int j = 0; j < it.n_tiles && ok; ++j) {
          const uint32_t gj = g + j;
          if (j + 1 < it.n_tiles) issue_s(gj + 1);
          else tc_commit(bar(SM::bQEmpty));
          if (!mbar_wait(bar(SM::bPFull + (gj & 1)), (gj >> 1) & 1)) { report(a.err, kErrTimeout); ok = false; break; }
          const int stage = gj % NS;
          if (!mbar_wait(bar(SM::bVFull + stage), (gj / NS) & 1)) { report(a.err, kErrTimeout); ok = false; break; }
          if (j == 0 && k > 0) {
            if (!mbar_wait(bar(SM::bOFree), (k - 1) & 1)) { report(a.err, kErrTimeout); ok = false; break; }
          }
          tc_fence_after();
          const uint32_t vst = sbase + SM::kStage0 + stage * 2 * SM::kTileBytes + SM::kTileBytes;
          const uint32_t p_t = tmem + (gj & 1) * 128;
#pragma unroll
          for (int kk = 0; kk < kPrefillTileN / 16; ++kk) {
            tc_mma_ts(t_o, p_t + kk * 8, smem_desc_sw128(vst + kk * 2048, SM::kHalfBytes, 1024),
                      idesc_o, (j > 0 || kk > 0) ? 1u : 0u);
          }
          tc_commit(bar(SM::bODone));
          tc_commit(bar(SM::bKVEmpty + stage));
        }
        g += it.n_tiles;
      }
    }
  } else {
    // ===================================================================== softmax warps
    const int quad = warp & 3;                    // TMEM lane quadrant this warp may access
    const int r = quad * 32 + lane;               // query row within the tile
    const uint32_t t_lane = tmem + ((uint32_t)(quad * 32) << 16);
    const float sl2 = a.scale_log2;
    __nv_bfloat16* outg = static_cast<__nv_bfloat16*>(a.out);
    uint32_t g = 0;
    for (uint32_t k = 0;; ++k) {
      const int slot = k & 1;
      if (!mbar_wait(bar(SM::bItemFull + slot), (k >> 1) & 1)) { report(a.err, kErrTimeout); break; }
      const int item = item_ids[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(SM::bItemEmpty + slot));
      if (item < 0) break;
      const PfItem it = pf_decode_item(item, a, pf_seq, pf_prefix, n_pf);
      const int limit = it.ctx + it.qt * kPrefillTileM + r;       // last key row r may see
      const int diag0 = it.ctx + it.qt * kPrefillTileM;           // row 0's last key
      float m_run = -INFINITY, l_run = 0.f;
      bool ok = true;
      for (int j = 0; j < it.n_tiles; ++j) {
        const uint32_t gj = g + j;
        const uint32_t buf = gj & 1;
        if (!mbar_wait(bar(SM::bSFull + buf), (gj >> 1) & 1)) { report(a.err, kErrTimeout); ok = false; break; }
        __syncwarp();
        tc_fence_after();
        uint32_t sr[128];
#pragma unroll
        for (int i = 0; i < 4; ++i) tmem_ld32(t_lane + buf * 128 + i * 32, sr + i * 32);
        tc_wait_ld();
        const int key0 = j * kPrefillTileN;
        float mx = -INFINITY;
        if (key0 + kPrefillTileN - 1 > diag0) {
#pragma unroll
          for (int cidx = 0; cidx < 128; ++cidx) {
            float v = __uint_as_float(sr[cidx]);
            v = (key0 + cidx <= limit) ? v : -INFINITY;
            sr[cidx] = __float_as_uint(v);
            mx = fmaxf(mx, v);
          }
        } else {
#pragma unroll
          for (int cidx = 0; cidx < 128; ++cidx) mx = fmaxf(mx, __uint_as_float(sr[cidx]));
        }
        const float mt = mx * sl2;
        float alpha = 1.f;
        bool resc = false;
        if (j == 0) {
          m_run = mt;
        } else if (mt > m_run + 8.f) {
          alpha = fast_exp2(m_run - mt);
          m_run = mt;
          resc = true;
        }
        float sum = 0.f;
#pragma unroll
        for (int cidx = 0; cidx < 128; cidx += 2) {
          const float p0 = fast_exp2(fmaf(__uint_as_float(sr[cidx]), sl2, -m_run));
          const float p1 = fast_exp2(fmaf(__uint_as_float(sr[cidx + 1]), sl2, -m_run));
          sum += p0 + p1;
          sr[cidx >> 1] = pack_bf16x2(p0, p1);
        }
        l_run = l_run * alpha + sum;
        if (__any_sync(0xffffffffu, resc)) {
          // O holds PV_{j-1}: wait for it, then scale this warp's 32 rows in place.
          if (!mbar_wait(bar(SM::bODone), (gj - 1) & 1)) { report(a.err, kErrTimeout); ok = false; break; }
          __syncwarp();
          tc_fence_after();
#pragma unroll
          for (int ch = 0; ch < D / 32; ++ch) {
            uint32_t ov[32];
            tmem_ld32(t_lane + 256 + ch * 32, ov);
            tc_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
            tmem_st32(t_lane + 256 + ch * 32, ov);
          }
          tc_wait_st();
        }
        if (j == it.n_tiles - 1) {
          // Keys at or past n_keys in the last tile: their V rows hold stale or poison data and
          // P is 0 there, but 0 * NaN is NaN, so zero them before the PV product reads them.
          const int stage = gj % NS;
          const int first = it.n_keys - key0;  // 1..128
          if (first < kPrefillTileN) {
            if (!mbar_wait(bar(SM::bVFull + stage), (gj / NS) & 1)) { report(a.err, kErrTimeout); ok = false; break; }
            const uint32_t vst = sbase + SM::kStage0 + stage * 2 * SM::kTileBytes + SM::kTileBytes;
            const int nchunks = (kPrefillTileN - first) * SM::kHalves * 8;
            for (int i = r; i < nchunks; i += 128) {
              const int rr = first + i / (SM::kHalves * 8);
              const int rem = i % (SM::kHalves * 8);
              const uint32_t addr = sw128(vst + (rem >> 3) * SM::kHalfBytes, rr, rem & 7);
              asm volatile("st.shared.v4.u32 [%0], {%1,%1,%1,%1};" ::"r"(addr), "r"(0u) : "memory");
            }
            fence_proxy_async_smem();
          }
        }
        tmem_st32(t_lane + buf * 128, sr);
        tmem_st32(t_lane + buf * 128 + 32, sr + 32);
        tc_wait_st();
        tc_fence_before();
        mbar_arrive(bar(SM::bPFull + buf));
      }
      if (!ok) break;
      // ---- epilogue: O / l -> bf16
      const uint32_t glast = g + it.n_tiles - 1;
      if (!mbar_wait(bar(SM::bODone), glast & 1)) { report(a.err, kErrTimeout); break; }
      __syncwarp();
      tc_fence_after();
      const float inv = 1.f / l_run;
      const bool store = r < it.rows;
      __nv_bfloat16* orow = outg + ((size_t)(it.tok0 + r) * a.Hq + it.head) * D;
#pragma unroll
      for (int ch = 0; ch < D / 32; ++ch) {
        uint32_t ov[32];
        tmem_ld32(t_lane + 256 + ch * 32, ov);
        tc_wait_ld();
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          pk[i] = pack_bf16x2(__uint_as_float(ov[2 * i]) * inv, __uint_as_float(ov[2 * i + 1]) * inv);
        if (store) {
          uint4* dst = reinterpret_cast<uint4*>(orow + ch * 32);
#pragma unroll
          for (int i = 0; i < 4; ++i) dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
        }
      }
      if (store && a.lse != nullptr)
        a.lse[(size_t)(it.tok0 + r) * a.Hq + it.head] = (m_run + __log2f(l_run)) * 0.6931471805599453f;
      tc_fence_before();
      mbar_arrive(bar(SM::bOFree));
      g += it.n_tiles;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D>
static cudaError_t launch_prefill_d(const AttnArgs& a, const CUtensorMap& qmap,
                                    const CUtensorMap& kmap, const CUtensorMap& vmap,
                                    cudaStream_t stream) {
  using SM = PrefillSmem<D>;
  static int configured_device = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_device != dev) {
    cudaError_t e = cudaFuncSetAttribute(prefill_kernel<D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, SM::kTotal);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  prefill_kernel<D><<<a.prefill_ctas, kPrefillThreads, SM::kTotal, stream>>>(a, qmap, kmap, vmap);
  return cudaGetLastError();
}

cudaError_t launch_prefill(const AttnArgs& a, const CUtensorMap& qmap, const CUtensorMap& kmap,
                           const CUtensorMap& vmap, cudaStream_t stream) {
  if (a.D == 128) return launch_prefill_d<128>(a, qmap, kmap, vmap, stream);
  return launch_prefill_d<64>(a, qmap, kmap, vmap, stream);
}

}  // namespace cb
