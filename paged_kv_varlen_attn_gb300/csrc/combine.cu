// Final combine of the cascade ("FlashAttention 在 vLLM 中的实现分析" §6.3:
// the shared-prefix result and each request's suffix result are merged by
// their LSEs, merge_attn_states).
//
// Both passes of a cascade call leave only partial states; this kernel then
// merges, for every row of the suffix pass, the row's own split states with
// the prefix pass's states of the same row and writes out / lse. Keeping the
// merge out of the passes means no block of the suffix pass waits for the
// prefix pass while it holds an SM.
#include <cuda_runtime.h>

#include "epilogue.cuh"

namespace pa {

// Threads of a block: 256 when the suffix pass has prefill-kernel groups (up
// to 256 rows each), else 128 -- a decode group of G rows has G * D / 4
// four-column units, 128 at G = 4 and D = 128, and the smaller blocks fit
// six to an SM instead of three (one wave for 64 sequences x 8 KV heads).
constexpr int kCombineThreads = 256;
constexpr int kCombineThreadsSmall = 128;

// One block per (row group of the suffix pass, KV head). Blocks [0, gb0)
// take class 0 groups, the rest class 1 groups.
template <int D, bool F16>
__global__ void __launch_bounds__(kCombineThreads)
cascade_combine_kernel(const __grid_constant__ AttnArgs a0, const __grid_constant__ AttnArgs a1,
                       int gb0) {
  // The plan is complete when this grid starts (the first attention kernel
  // of the call lets its successors start only after each of its blocks has
  // waited for the plan), so the group and the prefix pass's records are
  // read before the wait; the partial states are read after it.
  int g = static_cast<int>(blockIdx.x);
  const int cls = g >= gb0 ? 1 : 0;
  if (cls) g -= gb0;
  const AttnArgs& a = cls ? a1 : a0;
  const int hk = blockIdx.y;
  const bool live = g < a.header[4 + cls];
  int4 gr = make_int4(0, 0, 0, 0), sg = gr, sp = gr, pseg = gr, psplit = gr;
  if (live) {
    gr = a.groups[g];
    sg = a.seg[gr.x];
    sp = a.segsplit[gr.x];
    pseg = a.mp_seg[0];
    psplit = a.mp_segsplit[0];
  }
  // Launched as a dependent of the last attention kernel of the call: once
  // the wait returns, every kernel of the call before this one has completed.
  pdl_wait();
  pdl_trigger();
  if (!live || call_aborted(a)) return;
  const int rt = gr.y;
  const int rows_per_item = cls ? tc_item_rows(a.G, D) : kRowsSplit;
  const int row0 = rt * rows_per_item;
  const int R = min(rows_per_item, sg.y * a.G - row0);
  combine_splits<D, F16>(a, sp.y + rt * sp.x, sp.x, hk, R, row0, sg.x, threadIdx.x,
                         static_cast<int>(blockDim.x), pseg, psplit);
}

template <int D, bool F16>
static cudaError_t launch_combine_d(const AttnArgs& a0, const AttnArgs& a1, int gb0, int gb1,
                                    cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(gb0 + gb1), static_cast<unsigned>(a0.H_kv));
  cfg.blockDim = dim3(gb1 > 0 ? kCombineThreads : kCombineThreadsSmall);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, cascade_combine_kernel<D, F16>, a0, a1, gb0);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_cascade_combine(const AttnArgs& a0, const AttnArgs& a1, int gb0, int gb1,
                                   cudaStream_t st) {
  if (gb0 + gb1 <= 0) return cudaSuccess;
  if (a0.f16) {
    if (a0.D == 256) return launch_combine_d<256, true>(a0, a1, gb0, gb1, st);
    if (a0.D == 128) return launch_combine_d<128, true>(a0, a1, gb0, gb1, st);
    return launch_combine_d<64, true>(a0, a1, gb0, gb1, st);
  }
  if (a0.D == 256) return launch_combine_d<256, false>(a0, a1, gb0, gb1, st);
  if (a0.D == 128) return launch_combine_d<128, false>(a0, a1, gb0, gb1, st);
  return launch_combine_d<64, false>(a0, a1, gb0, gb1, st);
}

}  // namespace pa
