// The attention kernel: the decode pass and the chunk pass of one step in a single launch.
//
// Its grid is a.decode_grid decode-role CTAs followed by a.prefill_ctas chunk-role CTAs, one
// CTA per SM (each role needs ~200 KB of shared memory).  The block scheduler dispatches CTAs
// in index order, so the decode CTAs take their SMs first; the decode CTAs the planner leaves
// without work exit at once and the chunk CTAs fill those SMs, and the rest of the chunk CTAs
// start on the SMs the decode CTAs free as they finish.  The chunk CTAs claim items from the
// planner's counter, so however many of them start early, every item runs once.  In one launch
// the order of the two passes on the SMs is fixed by construction, where two kernels on two
// streams would race for them: a chunk kernel dispatched first holds every SM until it ends.
#include "cb_decode.cuh"
#include "cb_prefill.cuh"

namespace cb {

constexpr int kAttnThreads = kPrefillThreads;
static_assert(32 * (kMaxDecodeHeadsPerCta + 1) <= kAttnThreads,
              "the decode role fits in the chunk role's CTA");

template <int D, int QS>
struct AttnSmem {
  static constexpr int kTotal = DecodeSmem<D, QS>::kTotal > PrefillSmem<D>::kTotal
                                    ? DecodeSmem<D, QS>::kTotal
                                    : PrefillSmem<D>::kTotal;
};

template <int D, int QS, bool kWin>
__global__ void __launch_bounds__(kAttnThreads, 1)
    attention_kernel(const AttnArgs a, const __grid_constant__ CUtensorMap qmap,
                     const __grid_constant__ CUtensorMap kmap_dec,
                     const __grid_constant__ CUtensorMap vmap_dec,
                     const __grid_constant__ CUtensorMap kmap_chunk,
                     const __grid_constant__ CUtensorMap vmap_chunk) {
  extern __shared__ uint8_t smem_raw[];
  // Launched as a programmatic dependent of the planner: CTAs may start while the planner's
  // launch still runs; everything below reads the plan (and the appended K/V), so wait here
  // for that launch to complete and its writes to be visible.  A no-op without the attribute.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int b = (int)blockIdx.x;
  if (b < a.decode_grid) {
    // Span of the decode role: first start and last end of any warp of a CTA with work (the
    // chunk role stamps its own span inside prefill_cta).
    PlanHeader* hdr = reinterpret_cast<PlanHeader*>(a.ws + ws_layout(a.S, a.T, a.Hq, a.D).header);
    const bool busy = hdr->dec_tiles > 0;
    if (threadIdx.x == 0 && busy) atomicMin(&hdr->t_dec_start, global_ns());
    decode_cta<D, QS>(a, &kmap_dec, &vmap_dec, smem_raw, b % a.decode_ctas, b / a.decode_ctas);
    if ((threadIdx.x & 31) == 0 && busy) atomicMax(&hdr->t_dec_end, global_ns());
    return;
  }
  prefill_cta<D, kWin>(a, &qmap, &kmap_chunk, &vmap_chunk, smem_raw);
}

template <int D, int QS, bool kWin>
static cudaError_t launch_instance(const AttnArgs& a, const AttnMaps& m, cudaStream_t stream) {
  constexpr int kSmem = AttnSmem<D, QS>::kTotal;
  // The shared-memory opt-in is a setting of the context: made again whenever the launch
  // goes to another context than the last one configured.
  static unsigned long long configured_ctx = 0;
  const unsigned long long ctx = launch_context_id();
  if (ctx == 0 || configured_ctx != ctx) {
    const cudaError_t e = cudaFuncSetAttribute(
        attention_kernel<D, QS, kWin>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    configured_ctx = ctx;
  }
  // Programmatic stream serialization: the kernel may launch before the preceding launch on
  // the stream (the planner) ends, and waits for it with griddepcontrol.wait, so its launch
  // latency and CTA dispatch overlap the planner.
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.decode_grid + a.prefill_ctas);
  cfg.blockDim = dim3(kAttnThreads);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, attention_kernel<D, QS, kWin>, a, m.q, m.k_dec, m.v_dec,
                            m.k_chunk, m.v_chunk);
}

template <int D>
static cudaError_t launch_d(const AttnArgs& a, const AttnMaps& m, cudaStream_t stream) {
  const bool win = a.window > 0;
  if (a.G <= 8) {
    return win ? launch_instance<D, 1, true>(a, m, stream) : launch_instance<D, 1, false>(a, m, stream);
  }
  return win ? launch_instance<D, 2, true>(a, m, stream) : launch_instance<D, 2, false>(a, m, stream);
}

cudaError_t launch_attention(const AttnArgs& a, const AttnMaps& maps, cudaStream_t stream) {
  if (a.decode_grid + a.prefill_ctas == 0) return cudaSuccess;
  if (a.D == 128) return launch_d<128>(a, maps, stream);
  return launch_d<64>(a, maps, stream);
}

}  // namespace cb
