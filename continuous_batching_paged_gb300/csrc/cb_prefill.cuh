// Chunk pass of ragged paged attention: sequences with q_len > 1 (chunked prefill).  A chunk's
// many queries reuse each K/V tile, so this part of a step is limited by arithmetic rather than
// by memory ("LLM learning path 3.3 Batching & Memory Management", section "Chunked prefill"),
// and this pass runs on the 5th-generation tensor cores.  A chunk of queries attends to a cache that already holds the earlier chunks: query i
// of a chunk with prior context ctx sees keys 0 .. ctx + i (same section).
//
// One work item = two 128-query tiles A and B that read the same K/V tiles: with an even GQA
// group size, one query tile of a chunk under two query heads of one KV group (equal key
// ranges, so the two softmax groups stay in step); otherwise two consecutive query tiles under
// one head.  Persistent CTAs (one per SM) take items from a device counter the planner reset,
// in the planner's longest-first order of the work units with the query head (pair) fastest,
// so the scheduling is longest-processing-time first and the CTAs working on the heads of one
// KV group at the same time share its K/V tiles through L2.  Per CTA,
// warp-specialised (12 warps, three warpgroups; setmaxnreg moves registers from the first
// warpgroup, which only issues copies and MMAs and claims work, to the two softmax warpgroups:
// 104 + 2 x 200 per thread slot = the 3 x 168 the launch provides):
//   warp 0      TMA producer: Q tiles A and B once per item, then the K and V tiles of 128 keys
//               gathered page run by page run through the block table (staged in shared memory
//               once per item) into a ring of stages, each holding the V tile of one K/V step
//               and the K tile of the next (128-byte swizzle, the layout the tensor-core
//               descriptors read directly).
//   warp 1      tcgen05 issuer (one elected lane of a converged warp): S_t(j) = Q_t K_j^T into
//               TMEM, and O_t += P_t(j) V_j with P read from TMEM, then at once S_t(j+1); the
//               other tile's products keep the tensor core busy while a softmax group runs.
//               Completion is signalled with tcgen05.commit on mbarriers.  Also owns the TMEM
//               allocation.
//   warp 2      item scheduler: claims the next item from the counter when the producer is
//               three stages from the end of the current one, decodes it and publishes it in a
//               shared-memory slot, so that no role starts an item with a chain of global loads.
//   warps 4-7   softmax group A, warps 8-11 softmax group B: thread r owns query row r (TMEM
//               lane r) of its tile; it loads its 128 scores with tcgen05.ld, applies the causal
//               mask only on tiles that cross the diagonal, keeps the running max m and sum l in
//               registers (tree reductions), writes P (bf16) back over S, rescales O in TMEM
//               only when m grows by more than 8 in log2 units (otherwise the stale max keeps
//               every p <= 2^8, exact enough in fp32 and bf16), and writes O / l as bf16
//               through a shared-memory staging buffer (coalesced row stores).
// TMEM columns: [0,128) S/P of A, [128,256) S/P of B, [256,256+D) O of A, then O of B.
#pragma once

#include "cb_common.cuh"
#include "cb_launch.h"

namespace cb {

constexpr int kEntryCache = 1024;  // block-table entries of an item staged in shared memory

template <int D>
struct PrefillSmem {
  static constexpr int kHalves = D / 64;
  static constexpr int kQHalf = kPrefillTileM * 128;        // 128 query rows of 128 B
  static constexpr int kQTile = kHalves * kQHalf;
  static constexpr int kKVHalf = kChunkKeys * 128;          // 128 key rows of 128 B
  static constexpr int kKVTile = kHalves * kKVHalf;         // one K or V tile
  static constexpr int kStages = (D == 128) ? 2 : 4;
  static constexpr int kQ0 = 0;                             // Q_A, then Q_B
  // Ring of kStages slots.  Slot contents for stage m of an item: K tile j0 + m at +0 (m <
  // the item's K/V tile count) and V tile j0 + m - 1 at +kKVTile (m >= 1): the K tile of the
  // next S product travels with the V tile of the PV product issued just before it, so one
  // wait and one release per K/V step cover both.
  static constexpr int kStage0 = 2 * kQTile;
  static constexpr int kStageBytes = 2 * kKVTile;
  static constexpr int kBar = kStage0 + kStages * kStageBytes;
  // barrier indices (8 bytes each); [2] arrays are indexed by the tile (A = 0, B = 1)
  static constexpr int bQFull = 0, bQEmpty = 1, bFull = 2, bEmpty = bFull + kStages,
                       bSFull = bEmpty + kStages, bPFull = bSFull + 2, bOFinal = bPFull + 2,
                       bOFree = bOFinal + 2, bItemFull = bOFree + 2, bItemEmpty = bItemFull + 2,
                       bClaim = bItemEmpty + 2, kNumBars = bClaim + 1;
  static constexpr int kMisc = (kBar + kNumBars * 8 + 127) / 128 * 128;  // tmem base
  static constexpr int kItems = kMisc + 64;                 // two slots of decoded items
  static constexpr int kItemSlot = 128;
  static constexpr int kEntries = kItems + 2 * kItemSlot;   // block-table row of the item
  // Output staging of the epilogue: per softmax warp 32 rows x 32 columns of bf16 (64 B a row),
  // so that the output rows leave in coalesced 64-byte runs instead of one 16-byte piece per
  // row and instruction.
  static constexpr int kStageOut = kEntries + 4 * kEntryCache;
  static constexpr int kStageOutWarp = 32 * 64;
  static constexpr int kTotal = kStageOut + 8 * kStageOutWarp + 1024;
  // 16-byte vector accesses to the item slots' neighbours and the staging buffer
  static_assert(kItems % 16 == 0 && kEntries % 16 == 0 && kStageOut % 16 == 0,
                "shared-memory regions keep 16-byte alignment");
};

constexpr uint32_t kTmemCols = 512;
constexpr int kPrefillThreads = 384;
constexpr int kRegsIssue = 104;    // warpgroup 0 (producer, MMA issuer, two idle warps)
constexpr int kRegsSoftmax = 200;  // warpgroups 1 and 2
static_assert(kRegsIssue + 2 * kRegsSoftmax <= 3 * 168, "register split exceeds the launch");
constexpr int kItemConsumers = 10;  // producer, MMA warp, 4 warps of each softmax group

struct PfItem {
  int item;                                    // claimed item index, -1: no more work
  int s, kvh, ctx;
  int head[2], tok[2], rows[2], nk[2], nt[2];  // per tile: query head, first token, valid rows,
                                               // keys, K/V tiles
  int qoff[2];                                 // per tile: first query's offset in the chunk
  int nt_all, nk_all;                          // K/V tiles loaded and keys covered for the item
  int j0;                                      // first K/V tile (a sliding window skips older)
  int hasB;
};
static_assert(sizeof(PfItem) <= 128, "a decoded item fits its shared-memory slot");

// Query heads (pairs) per unit: items are unit-major with the head (pair) fastest, so the
// CTAs on the heads of one KV group at the same time share its K/V tiles through L2.
__device__ __forceinline__ int pf_heads_per_unit(const AttnArgs& a) {
  return pf_pair_heads(a.G) ? a.Hq / 2 : a.Hq;
}

template <bool kWin>
__device__ __forceinline__ PfItem pf_decode_item(int item, const AttnArgs& a,
                                                 const int32_t* pf_seq, const int32_t* pf_prefix,
                                                 const int32_t* pf_order, int n_pf) {
  PfItem it;
  it.item = item;
  const int hu_n = pf_heads_per_unit(a);
  const int pos = item / hu_n;  // position in the longest-first unit order
  const int hu = item - pos * hu_n;
  const int g = pf_order[pos];  // unit index in chunk-sequence order
  int lo = 0, hi = n_pf - 1;    // largest i with pf_prefix[i] <= g
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (pf_prefix[mid] <= g) lo = mid; else hi = mid - 1;
  }
  it.s = pf_seq[lo];
  const int u = g - pf_prefix[lo];
  const int c0 = a.cu_seqlens_q[it.s];
  const int q_len = a.cu_seqlens_q[it.s + 1] - c0;
  it.ctx = a.kv_lens[it.s] - q_len;
  int qt[2];
  if (pf_pair_heads(a.G)) {  // one query tile, heads 2hu and 2hu+1 of one KV group
    qt[0] = qt[1] = u;
    it.head[0] = 2 * hu;
    it.head[1] = 2 * hu + 1;
    it.hasB = true;
  } else {                   // query tiles 2u and 2u+1, one head
    qt[0] = 2 * u;
    qt[1] = 2 * u + 1;
    it.head[0] = it.head[1] = hu;
    it.hasB = qt[1] * kPrefillTileM < q_len;
  }
  it.kvh = it.head[0] / a.G;
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const bool on = t == 0 || it.hasB;
    it.qoff[t] = qt[t] * kPrefillTileM;
    it.tok[t] = c0 + qt[t] * kPrefillTileM;
    it.rows[t] = on ? min(kPrefillTileM, q_len - qt[t] * kPrefillTileM) : 0;
    it.nk[t] = on ? it.ctx + qt[t] * kPrefillTileM + it.rows[t] : 0;
    it.nt[t] = (it.nk[t] + kChunkKeys - 1) / kChunkKeys;
  }
  it.nk_all = max(it.nk[0], it.nk[1]);
  it.nt_all = max(it.nt[0], it.nt[1]);
  // tile A's first row is the item's earliest query; keys before its window are not needed
  it.j0 = kWin ? window_first_key(it.ctx + qt[0] * kPrefillTileM, a.window) / kChunkKeys : 0;
  return it;
}

// kWin: sliding-window attention (a.window > 0).  The full causal pass is compiled without
// the window's bookkeeping, so it runs exactly the code it ran before windows existed.
// One persistent CTA of the chunk pass (all kPrefillThreads threads).  Runs in the attention
// kernel (cb_attention.cu) with that kernel's dynamic shared memory.
template <int D, bool kWin>
__device__ __forceinline__ void prefill_cta(const AttnArgs& a, const CUtensorMap* qmap,
                                            const CUtensorMap* kmap, const CUtensorMap* vmap,
                                            uint8_t* smem_raw) {
  using SM = PrefillSmem<D>;
  constexpr int NS = SM::kStages;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return sbase + SM::kBar + 8 * i; };
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + SM::kMisc);
  // Decoded items, two slots: the scheduler warp claims and decodes the next item while the
  // current one runs; every role reads it from here (no global-memory chain at an item's start).
  auto item_slot = [&](int slot) { return reinterpret_cast<PfItem*>(smem + SM::kItems + slot * SM::kItemSlot); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const WsLayout L = ws_layout(a.S, a.T, a.Hq, a.D);
  PlanHeader* hdr = reinterpret_cast<PlanHeader*>(a.ws + L.header);
  const int32_t* pf_seq = reinterpret_cast<const int32_t*>(a.ws + L.pf_seq);
  const int32_t* pf_prefix = reinterpret_cast<const int32_t*>(a.ws + L.pf_prefix);
  const int32_t* pf_order = reinterpret_cast<const int32_t*>(a.ws + L.pf_order);
  const int n_pf = hdr->n_pf;
  const int n_items = hdr->pf_qtiles * pf_heads_per_unit(a);
  if (n_items == 0) return;

  if (threadIdx.x == 0) {
    mbar_init(bar(SM::bQFull), 1);
    mbar_init(bar(SM::bQEmpty), 1);
    for (int i = 0; i < NS; ++i) {
      mbar_init(bar(SM::bFull + i), 1);
      mbar_init(bar(SM::bEmpty + i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(SM::bSFull + i), 1);
      mbar_init(bar(SM::bPFull + i), 4);   // one arrival per softmax warp
      mbar_init(bar(SM::bOFinal + i), 1);
      mbar_init(bar(SM::bOFree + i), 4);
      mbar_init(bar(SM::bItemFull + i), 1);
      mbar_init(bar(SM::bItemEmpty + i), kItemConsumers);
    }
    mbar_init(bar(SM::bClaim), 1);
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

  // Each role runs inside the branch that set its register count (no join in between, so the
  // compiler allocates every role's code under that role's own limit).
  if (warp < 4) {
    regs_dec<kRegsIssue>();
    if (warp == 0) {
      // =================================================================== TMA producer
      if (lane == 0) {
        tma_prefetch_desc(qmap);
        tma_prefetch_desc(kmap);
        tma_prefetch_desc(vmap);
      }
      const int KB = a.KBp;
      const int nsb = kChunkKeys / KB;  // page-run boxes per K/V tile (<= 128)
      uint32_t g = 0;
      for (uint32_t k = 0;; ++k) {
        const int slot = k & 1;
        if (!mbar_wait(bar(SM::bItemFull + slot), (k >> 1) & 1)) { report(a.err, kErrTimeout); break; }
        const PfItem it = *item_slot(slot);
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(SM::bItemEmpty + slot));
        if (it.item < 0) break;
        // stage at which the scheduler warp is told to claim the next item
        const int m_claim = max(0, it.nt_all - it.j0 - 3);
        if (lane == 0) {
          if (!mbar_wait(bar(SM::bQEmpty), (k & 1) ^ 1)) report(a.err, kErrTimeout);
          mbar_arrive_expect_tx(bar(SM::bQFull), (it.hasB ? 2 : 1) * SM::kQTile);
#pragma unroll
          for (int half = 0; half < SM::kHalves; ++half)
            tma_load_3d(sbase + SM::kQ0 + half * SM::kQHalf, qmap, bar(SM::bQFull), half * 64,
                        it.head[0], it.tok[0]);
          if (it.hasB) {
#pragma unroll
            for (int half = 0; half < SM::kHalves; ++half)
              tma_load_3d(sbase + SM::kQ0 + SM::kQTile + half * SM::kQHalf, qmap, bar(SM::bQFull),
                          half * 64, it.head[1], it.tok[1]);
          }
        }
        const int32_t* row = a.block_table + (size_t)it.s * a.max_blocks;
        // Stage the item's block-table entries in shared memory with coalesced loads issued
        // back to back, so the per-tile loop below never waits on a global load.
        int* ecache = reinterpret_cast<int*>(smem + SM::kEntries);
        const int e0 = it.j0 * kChunkKeys / a.bs;  // first block the item reads
        const int n_ent =
            max(0, min(min((it.nk_all + a.bs - 1) / a.bs, a.max_blocks) - e0, kEntryCache));
        for (int i = lane; i < n_ent; i += 32) ecache[i] = __ldg(row + e0 + i);
        __syncwarp();
        // Entries of the page runs of K/V tile j (lane = run index mod 32); the previous tile's
        // are kept for its V tile, which travels one stage later.
        auto entries = [&](int j, int (&ent)[4]) {
          const int key0 = j * kChunkKeys;
#pragma unroll
          for (int p = 0; p < 4; ++p) {
            const int sb = p * 32 + lane;
            const int pos = key0 + sb * KB;
            ent[p] = -1;
            if (sb < nsb && pos < it.nk_all) {
              const int lb = pos / a.bs;
              ent[p] = lb >= a.max_blocks ? -2
                                          : (lb - e0 < n_ent ? ecache[lb - e0] : __ldg(row + lb));
            }
          }
        };
        // Number of page runs of tile j this warp loads (a run with a bad block id is skipped
        // and reported).
        auto count = [&](int j, const int (&ent)[4], bool report_bad) -> uint32_t {
          uint32_t n = 0;
#pragma unroll
          for (int p = 0; p < 4; ++p) {
            const int sb = p * 32 + lane;
            const bool want = sb < nsb && j * kChunkKeys + sb * KB < it.nk_all;
            const bool valid = want && ent[p] >= 0 && ent[p] < a.P;
            if (report_bad && want && !valid) report(a.err, kErrOutOfRange);
            n += __popc(__ballot_sync(0xffffffffu, valid));
          }
          return n;
        };
        auto load = [&](int j, const int (&ent)[4], uint32_t dst, const CUtensorMap* map,
                        uint32_t full) {
          const int key0 = j * kChunkKeys;
#pragma unroll
          for (int p = 0; p < 4; ++p) {
            const int sb = p * 32 + lane;
            const int pos = key0 + sb * KB;
            if (sb < nsb && pos < it.nk_all && ent[p] >= 0 && ent[p] < a.P) {
              const int token = ent[p] * a.bs + (pos % a.bs);
#pragma unroll
              for (int half = 0; half < SM::kHalves; ++half)
                tma_load_3d(dst + half * SM::kKVHalf + sb * KB * 128, map, full, half * 64,
                            it.kvh, token);
            }
          }
        };
        int ent_k[4] = {-1, -1, -1, -1}, ent_v[4];
        for (int m = 0; m <= it.nt_all - it.j0; ++m, ++g) {
          const int j = it.j0 + m;           // K tile of this stage (if j < nt_all)
          const int stage = g % NS;
          const uint32_t phase = (g / NS) & 1;
          const bool has_k = j < it.nt_all, has_v = m > 0;
#pragma unroll
          for (int p = 0; p < 4; ++p) ent_v[p] = ent_k[p];   // V of tile j - 1
          if (has_k) entries(j, ent_k);
          const uint32_t runs = (has_k ? count(j, ent_k, true) : 0u) + (has_v ? count(j - 1, ent_v, false) : 0u);
          const uint32_t kst = sbase + SM::kStage0 + stage * SM::kStageBytes;
          const uint32_t full = bar(SM::bFull + stage);
          if (lane == 0) {
            if (!mbar_wait(bar(SM::bEmpty + stage), phase ^ 1)) report(a.err, kErrTimeout);
            mbar_arrive_expect_tx(full, runs * (uint32_t)(SM::kHalves * KB * 128));
          }
          __syncwarp();
          if (has_k) load(j, ent_k, kst, kmap, full);
          if (has_v) load(j - 1, ent_v, kst + SM::kKVTile, vmap, full);
          // The next item is claimed three stages before this item's last: early enough that
          // the claim and its decode are done when the item starts, late enough that the claim
          // order stays the order in which CTAs run out of work (the longest-first schedule
          // depends on it).
          if (m == m_claim && lane == 0) mbar_arrive(bar(SM::bClaim));
        }
      }
    } else if (warp == 2) {
      // =================================================================== item scheduler
      // Claims items from the planner's counter, decodes each into a slot of shared memory
      // (two slots), and claims the next one when the producer signals that the current
      // item's loads are near their end.
      auto claim = [&](uint32_t kc) -> int {
        const int slot = kc & 1;
        int item = -1;
        if (lane == 0) {
          if (!mbar_wait(bar(SM::bItemEmpty + slot), ((kc >> 1) & 1) ^ 1)) report(a.err, kErrTimeout);
          item = atomicAdd(&hdr->pf_counter, 1);
          if (item >= n_items) item = -1;
          if (kc == 0 && item >= 0) atomicMin(&hdr->t_pf_start, global_ns());  // role span
        }
        item = __shfl_sync(0xffffffffu, item, 0);
        PfItem it;
        if (item >= 0) it = pf_decode_item<kWin>(item, a, pf_seq, pf_prefix, pf_order, n_pf);
        it.item = item;
        if (lane == 0) {
          *item_slot(slot) = it;
          mbar_arrive(bar(SM::bItemFull + slot));
        }
        return item;
      };
      int item = claim(0);
      for (uint32_t k = 0; item >= 0; ++k) {
        if (!mbar_wait(bar(SM::bClaim), k & 1)) {
          report(a.err, kErrTimeout);
          break;
        }
        item = claim(k + 1);
      }
    } else if (warp == 1) {
      // =================================================================== tcgen05 issuer
      // The whole warp runs this loop (uniform control flow); one elected lane issues each
      // batch of MMAs together with the commit that tracks it.  An MMA's issue returns only
      // once the tensor core can queue it, about one MMA ahead of the one executing, so every
      // instruction this thread runs between two batches is time the tensor core may sit idle:
      // the loop keeps that work short (per-tile state in scalars, never in arrays indexed at
      // run time, which would live in local memory; the tiles unrolled; descriptors
      // precomputed).
      constexpr uint32_t idesc_s = idesc_bf16(kPrefillTileM, kChunkKeys, 0);
      constexpr uint32_t idesc_o = idesc_bf16(kPrefillTileM, D, 1);
      // Descriptor of the first 16-wide K slice of each operand region; a slice at byte offset
      // `off` is the same descriptor with (off >> 4) added to its start-address field.
      const uint64_t q_desc0 = smem_desc_sw128(sbase + SM::kQ0, 16, 1024);
      const uint64_t k_desc0 = smem_desc_sw128(sbase + SM::kStage0, 16, 1024);
      const uint64_t v_desc0 = smem_desc_sw128(sbase + SM::kStage0 + SM::kKVTile, SM::kKVHalf, 1024);
      uint32_t g = 0;                // K/V tiles consumed so far (position in the stage ring)
      uint32_t gxA = 0, gxB = 0;     // S/P rounds of tile A / tile B so far
      uint32_t kxA = 0, kxB = 0;     // items finished on tile A / tile B
      bool ok = true;
      auto wait = [&](uint32_t b, uint32_t parity) {
        if (ok && !mbar_wait(b, parity)) {
          report(a.err, kErrTimeout);
          ok = false;
        }
      };
      auto commit = [&](uint32_t b) {
        if (elect_one()) tc_commit(b);
        __syncwarp();
      };
      // S_t = Q_t K^T with the K tile of ring slot `stage` (loaded) into tile t's S buffer,
      // then its commit.
      auto mma_s = [&](const int t, const int stage) {
        const uint64_t qd = q_desc0 + ((uint32_t)(t * SM::kQTile) >> 4);
        const uint64_t kd = k_desc0 + ((uint32_t)(stage * SM::kStageBytes) >> 4);
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t qo = ((kk >> 2) * SM::kQHalf + (kk & 3) * 32) >> 4;
            const uint32_t ko = ((kk >> 2) * SM::kKVHalf + (kk & 3) * 32) >> 4;
            tc_mma_ss(tmem + t * 128, qd + qo, kd + ko, idesc_s, kk > 0 ? 1u : 0u);
          }
          tc_commit(bar(SM::bSFull + t));
        }
        __syncwarp();
      };
      // O_t += P_t V with P read from TMEM; `first`: the item's first K/V tile (overwrite O);
      // `last`: its last one for this tile (commit the final O).
      auto mma_pv = [&](const int t, const uint64_t vd, const bool first, const bool last) {
        const uint32_t p_t = tmem + t * 128;
        const uint32_t o_t = tmem + 256 + t * D;
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < kChunkKeys / 16; ++kk)
            tc_mma_ts(o_t, p_t + kk * 8, vd + ((uint32_t)(kk * 2048) >> 4), idesc_o,
                      (!first || kk > 0) ? 1u : 0u);
          if (last) tc_commit(bar(SM::bOFinal + t));
        }
        __syncwarp();
      };
      for (uint32_t k = 0; ok; ++k) {
        const int slot = k & 1;
        wait(bar(SM::bItemFull + slot), (k >> 1) & 1);
        if (!ok) break;
        const PfItem it = *item_slot(slot);
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(SM::bItemEmpty + slot));
        if (it.item < 0) break;
        const int j0 = it.j0, nt_all = it.nt_all;
        const int ntA = it.nt[0], ntB = it.hasB ? it.nt[1] : 0;
        // Stage 0 of the item: K tile j0.  (Waiting on a TMA-completed barrier orders the MMAs'
        // shared-memory reads after the copies; no tensor fence is needed for that.)
        wait(bar(SM::bQFull), k & 1);
        wait(bar(SM::bFull + g % NS), (g / NS) & 1);
        mma_s(0, g % NS);
        if (ntB > 0) mma_s(1, g % NS);
        commit(bar(SM::bEmpty + g % NS));
        // Q is read by the S products only: release it once the item's last ones are issued,
        // so that the next item's Q loads during this item's last K/V step.
        if (nt_all - j0 == 1) commit(bar(SM::bQEmpty));
        for (int j = j0; j < nt_all && ok; ++j) {
          // stage j - j0 + 1: V tile j and K tile j + 1
          const uint32_t gs = g + (uint32_t)(j - j0) + 1;
          const int stage = gs % NS;
          const uint64_t vd = v_desc0 + ((uint32_t)(stage * SM::kStageBytes) >> 4);
          wait(bar(SM::bFull + stage), (gs / NS) & 1);
          if (j < ntA) {
            wait(bar(SM::bPFull + 0), (gxA + (uint32_t)(j - j0)) & 1);
            if (j == j0 && kxA > 0) wait(bar(SM::bOFree + 0), (kxA - 1) & 1);
            tc_fence_after();
            mma_pv(0, vd, j == j0, j == ntA - 1);
            if (j + 1 < ntA) mma_s(0, stage);
          }
          if (j < ntB) {
            wait(bar(SM::bPFull + 1), (gxB + (uint32_t)(j - j0)) & 1);
            if (j == j0 && kxB > 0) wait(bar(SM::bOFree + 1), (kxB - 1) & 1);
            tc_fence_after();
            mma_pv(1, vd, j == j0, j == ntB - 1);
            if (j + 1 < ntB) mma_s(1, stage);
          }
          commit(bar(SM::bEmpty + stage));
          if (j == nt_all - 2) commit(bar(SM::bQEmpty));
        }
        g += (uint32_t)(nt_all - j0) + 1;
        gxA += (uint32_t)(ntA - j0);
        kxA += 1;
        if (ntB > 0) {
          gxB += (uint32_t)(ntB - j0);
          kxB += 1;
        }
      }
    }
  } else {
    regs_inc<kRegsSoftmax>();
    // ===================================================================== softmax groups
    const int t = (warp - 4) >> 2;                // 0: tile A, 1: tile B
    const int quad = warp & 3;                    // TMEM lane quadrant this warp may access
    const int r = quad * 32 + lane;               // query row within the tile
    const uint32_t t_lane = tmem + ((uint32_t)(quad * 32) << 16);
    const uint32_t o_col = 256 + t * D;
    const float sl2 = a.scale_log2;
    __nv_bfloat16* outg = static_cast<__nv_bfloat16*>(a.out);
    uint32_t g = 0, gx = 0, kx = 0;
    for (uint32_t k = 0;; ++k) {
      const int slot = k & 1;
      if (!mbar_wait(bar(SM::bItemFull + slot), (k >> 1) & 1)) { report(a.err, kErrTimeout); break; }
      const PfItem it = *item_slot(slot);
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(SM::bItemEmpty + slot));
      if (it.item < 0) break;
      const uint32_t g_item = g;
      g += it.nt_all - it.j0 + 1;  // ring stages of the item
      if (t == 1 && !it.hasB) continue;
      const int nt = t ? it.nt[1] : it.nt[0];
      const int tok = t ? it.tok[1] : it.tok[0];
      const int rows = t ? it.rows[1] : it.rows[0];
      const int head = t ? it.head[1] : it.head[0];
      const int diag0 = it.ctx + (t ? it.qoff[1] : it.qoff[0]);  // row 0's last key
      const int limit = diag0 + r;                                     // row r's last key
      float m_run = -INFINITY, l_run = 0.f;
      bool ok = true;
      const int W = kWin ? a.window : 0;
      for (int j = it.j0; j < nt; ++j) {
        const uint32_t tt = gx + (j - it.j0);
        const uint32_t s_col = t * 128;
        if (!mbar_wait(bar(SM::bSFull + t), tt & 1)) { report(a.err, kErrTimeout); ok = false; break; }
        __syncwarp();
        tc_fence_after();
        uint32_t sr[128];
#pragma unroll
        for (int i = 0; i < 4; ++i) tmem_ld32(t_lane + s_col + i * 32, sr + i * 32);
        tc_wait_ld();
        const int key0 = j * kChunkKeys;
        // causal edge (keys past the row's position) and, with a sliding window, its lower
        // edge (keys at or before position - W)
        const int lo_r = kWin ? limit - W + 1 : 0;
        if (key0 + kChunkKeys - 1 > diag0 || (kWin && key0 < lo_r)) {
#pragma unroll
          for (int c = 0; c < 128; ++c)
            if (key0 + c > limit || (kWin && key0 + c < lo_r)) sr[c] = __float_as_uint(-INFINITY);
        }
        // row max: 8 independent chains of three-input max over the 128 columns
        float mx8[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
          mx8[i] = fmax3(__uint_as_float(sr[i]), __uint_as_float(sr[8 + i]), __uint_as_float(sr[16 + i]));
#pragma unroll
        for (int c = 24; c < 120; c += 16)
#pragma unroll
          for (int i = 0; i < 8; ++i)
            mx8[i] = fmax3(mx8[i], __uint_as_float(sr[c + i]), __uint_as_float(sr[c + 8 + i]));
#pragma unroll
        for (int i = 0; i < 8; ++i) mx8[i] = fmaxf(mx8[i], __uint_as_float(sr[120 + i]));
        const float mx = fmaxf(fmax3(mx8[0], mx8[1], mx8[2]),
                               fmax3(fmax3(mx8[3], mx8[4], mx8[5]), mx8[6], mx8[7]));
        const float mt = mx * sl2;
        float alpha = 1.f;
        bool resc = false;
        if (j == it.j0) {
          m_run = mt;
        } else if (mt > m_run + 8.f) {
          alpha = fast_exp2(m_run - mt);
          m_run = mt;
          resc = true;
        }
        // A row whose keys so far all lie outside its sliding window has m = -inf: subtract
        // 0 instead (every p is then 0), so that no -inf - (-inf) appears.
        const float m_sub = (kWin && m_run == -INFINITY) ? 0.f : m_run;
        // exponent arguments and row sums two columns per instruction (paired fp32)
        const uint64_t scale2 = f2_pack(sl2, sl2), neg_m2 = f2_pack(-m_sub, -m_sub);
        uint64_t sum2[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) sum2[i] = 0ull;
#pragma unroll
        for (int c = 0; c < 128; c += 2) {
          float x0, x1;
          f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[c]), __uint_as_float(sr[c + 1])), scale2, neg_m2),
                    x0, x1);
          const float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
          sum2[(c >> 1) & 3] = f2_add(sum2[(c >> 1) & 3], f2_pack(p0, p1));
          sr[c >> 1] = pack_bf16x2(p0, p1);
        }
        float sm8[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) f2_unpack(sum2[i], sm8[2 * i], sm8[2 * i + 1]);
        const float sum = ((sm8[0] + sm8[1]) + (sm8[2] + sm8[3])) + ((sm8[4] + sm8[5]) + (sm8[6] + sm8[7]));
        l_run = l_run * alpha + sum;
        if (j == it.nt_all - 1) {
          // Keys at or past the pair's last key in the last K/V tile: their V rows hold stale or
          // poison data and P is 0 there, but 0 * NaN is NaN, so zero them before the PV
          // product reads them (both groups may do it; they write the same zeros).
          const int first = it.nk_all - key0;  // 1..128
          if (first < kChunkKeys) {
            const uint32_t gk = g_item + (j - it.j0) + 1;  // the stage holding V tile j
            const int stage = gk % NS;
            if (!mbar_wait(bar(SM::bFull + stage), (gk / NS) & 1)) { report(a.err, kErrTimeout); ok = false; break; }
            const uint32_t vst = sbase + SM::kStage0 + stage * SM::kStageBytes + SM::kKVTile;
            const int nchunks = (kChunkKeys - first) * SM::kHalves * 8;
            for (int i = r; i < nchunks; i += 128) {
              const int rr = first + i / (SM::kHalves * 8);
              const int rem = i % (SM::kHalves * 8);
              const uint32_t addr = sw128(vst + (rem >> 3) * SM::kKVHalf, rr, rem & 7);
              asm volatile("st.shared.v4.u32 [%0], {%1,%1,%1,%1};" ::"r"(addr), "r"(0u) : "memory");
            }
            fence_proxy_async_smem();
          }
        }
        tmem_st32(t_lane + s_col, sr);
        tmem_st32(t_lane + s_col + 32, sr + 32);
        if (__any_sync(0xffffffffu, resc)) {
          // O holds the products of tiles 0..j-1; they have completed, because S of tile j
          // was issued after them and its commit signalled every earlier MMA done.
#pragma unroll
          for (int ch = 0; ch < D / 32; ++ch) {
            uint32_t ov[32];
            tmem_ld32(t_lane + o_col + ch * 32, ov);
            tc_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
            tmem_st32(t_lane + o_col + ch * 32, ov);
          }
        }
        tc_wait_st();
        tc_fence_before();
        // one arrival per warp once all its lanes have stored P: 4 arrivals on the barrier per
        // tile instead of 128, which would queue in shared memory behind one another
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(SM::bPFull + t));
      }
      if (!ok) break;
      // ---- epilogue: O / l -> bf16
      if (!mbar_wait(bar(SM::bOFinal + t), kx & 1)) { report(a.err, kErrTimeout); break; }
      __syncwarp();
      tc_fence_after();
      const float inv = 1.f / l_run;
      const bool store = r < rows;
      // Each 32-column slice of the warp's 32 rows goes through shared memory: lane = row on
      // the way in (TMEM lane), four lanes per row on the way out, so that every store
      // instruction writes 64 contiguous bytes of 8 rows.  The 16-byte chunks of a row are
      // XOR-swizzled by the row pair so that neither side has bank conflicts.
      const uint32_t stg = sbase + SM::kStageOut + (warp - 4) * SM::kStageOutWarp;
      const int orow_base = quad * 32;
#pragma unroll
      for (int ch = 0; ch < D / 32; ++ch) {
        uint32_t ov[32];
        tmem_ld32(t_lane + o_col + ch * 32, ov);
        tc_wait_ld();
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) {
          uint32_t pk[4];
#pragma unroll
          for (int i = 0; i < 4; ++i)
            pk[i] = pack_bf16x2(__uint_as_float(ov[8 * c4 + 2 * i]) * inv,
                                __uint_as_float(ov[8 * c4 + 2 * i + 1]) * inv);
          const uint32_t addr = stg + lane * 64 + ((c4 ^ ((lane >> 1) & 3)) << 4);
          asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(pk[0]), "r"(pk[1]),
                       "r"(pk[2]), "r"(pk[3]) : "memory");
        }
        __syncwarp();
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int row = (lane >> 2) + 8 * i, c4 = lane & 3;
          uint4 v;
          const uint32_t addr = stg + row * 64 + ((c4 ^ ((row >> 1) & 3)) << 4);
          asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                       : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr) : "memory");
          if (orow_base + row < rows)
            *reinterpret_cast<uint4*>(outg + ((size_t)(tok + orow_base + row) * a.Hq + head) * D +
                                      ch * 32 + c4 * 8) = v;
        }
        __syncwarp();
      }
      if (store && a.lse != nullptr)
        a.lse[(size_t)(tok + r) * a.Hq + head] = (m_run + __log2f(l_run)) * 0.6931471805599453f;
      if (r == 0) atomicMax(&hdr->t_pf_end, global_ns());  // role span: last item's end
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(SM::bOFree + t));
      gx += nt - it.j0;
      kx += 1;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace cb
