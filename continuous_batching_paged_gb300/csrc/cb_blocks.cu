// Whole-block moves of the paged KV cache: copy-on-write block copies inside the pools, and
// the batched offload (gather to host) / restore (scatter from host) of a list of blocks.
// HBM (or CPU-GPU link) bound: 16-byte vector loads, four per thread in flight before the
// stores, K and V of the same chunk together; grid = a few waves of the SMs.
#include "cb_common.cuh"
#include "cb_launch.h"

namespace cb {

constexpr int kMoveThreads = 256;
constexpr int kMoveUnroll = 4;

__global__ void __launch_bounds__(kMoveThreads) block_move_kernel(BlockMoveArgs a) {
  const long long cpb = a.block_bytes / 16;  // 16-byte chunks per block and pool
  const long long total = (long long)a.n * cpb;
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long base = (long long)blockIdx.x * blockDim.x + threadIdx.x; base < total;
       base += stride * kMoveUnroll) {
    uint4 kv[kMoveUnroll][2];
    long long doff[kMoveUnroll];
    bool ok[kMoveUnroll];
#pragma unroll
    for (int u = 0; u < kMoveUnroll; ++u) {
      const long long idx = base + u * stride;
      ok[u] = false;
      if (idx >= total) continue;
      const int i = (int)(idx / cpb);
      const long long c = idx - (long long)i * cpb;
      long long sblk = i, dblk = i;  // linear host position for the host side
      if (a.mode != kMoveRestore) sblk = a.src_idx[i];
      if (a.mode != kMoveOffload) dblk = a.dst_idx[i];
      const bool s_ok = a.mode == kMoveRestore || (sblk >= 0 && sblk < a.P);
      const bool d_ok = a.mode == kMoveOffload || (dblk >= 0 && dblk < a.P);
      if (!s_ok || !d_ok) {
        if (c == 0) report(a.err, kErrOutOfRange);
        continue;
      }
      if (a.mode == kMoveCopy && sblk == dblk) continue;
      const long long soff = sblk * a.block_bytes + c * 16;
      doff[u] = dblk * a.block_bytes + c * 16;
      kv[u][0] = *reinterpret_cast<const uint4*>(a.src[0] + soff);
      kv[u][1] = *reinterpret_cast<const uint4*>(a.src[1] + soff);
      ok[u] = true;
    }
#pragma unroll
    for (int u = 0; u < kMoveUnroll; ++u) {
      if (!ok[u]) continue;
      *reinterpret_cast<uint4*>(a.dst[0] + doff[u]) = kv[u][0];
      *reinterpret_cast<uint4*>(a.dst[1] + doff[u]) = kv[u][1];
    }
  }
}

cudaError_t launch_block_move(const BlockMoveArgs& a, int sm_count, cudaStream_t stream) {
  if (a.n <= 0) return cudaSuccess;
  const long long total = (long long)a.n * (a.block_bytes / 16);
  long long blocks = (total + (long long)kMoveThreads * kMoveUnroll - 1) / ((long long)kMoveThreads * kMoveUnroll);
  const long long cap = (long long)sm_count * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  block_move_kernel<<<(unsigned)blocks, kMoveThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

// Self-test of the bounded wait every kernel of the library uses: one thread waits on an
// mbarrier phase that nothing completes; after limit_ns it gives up, records the timeout in
// the error word and returns, leaving the context usable.
__global__ void wait_selftest_kernel(uint32_t* err, uint64_t limit_ns, uint64_t* waited_ns) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = smem_u32(&bar);
  mbar_init(b, 1);
  fence_barrier_init();
  const uint64_t t0 = globaltimer_ns();
  if (!mbar_wait_for(b, 0, limit_ns)) report(err, kErrTimeout);
  if (waited_ns != nullptr) *waited_ns = globaltimer_ns() - t0;
}

cudaError_t launch_wait_selftest(uint32_t* err, uint64_t limit_ns, uint64_t* waited_ns,
                                 cudaStream_t stream) {
  wait_selftest_kernel<<<1, 1, 0, stream>>>(err, limit_ns, waited_ns);
  return cudaGetLastError();
}

}  // namespace cb
