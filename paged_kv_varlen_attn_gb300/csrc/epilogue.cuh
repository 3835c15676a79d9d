// Shared epilogue pieces of the attention kernels: the LSE merge with a
// cascade prefix state and the combine of split-KV partial states ("FlashAttention
// 在 vLLM 中的实现分析" §6.3 merge_attn_states, used for num_splits of §1.3).
#pragma once

#include "device_common.cuh"

namespace pa {

// Cascade: merge the state (o[0..n) at columns col.., lse) of row (token tok,
// head h) with the prefix pass's partial states of the same row -- one per
// split of the shared prefix -- weighted by their LSEs. lse becomes the merged
// LSE. The prefix pass planned one segment holding every query token, so the
// row's packed index there is tok * G + (h % G).
__device__ __forceinline__ void merge_prefix(const AttnArgs& a, int h, int tok, int col,
                                             float& lse, float* o, int n) {
  const int4 g0 = a.mp_seg[0];
  const int4 s0 = a.mp_segsplit[0];
  const int cls = g0.w;
  const int rows_per_item = cls ? kRowsTc : kRowsSplit;
  const int G = a.G;
  const int hk = h / G;
  const int pr = tok * G + (h - hk * G);
  const int rt = pr / rows_per_item, rl = pr - rt * rows_per_item;
  const int nsp = s0.x, base = s0.y + rt * nsp;
  const float* plse = a.mp_part_lse[cls];
  const float* po = a.mp_part_o[cls];
  const int64_t srows = a.mp_slot_rows[cls];
  float mx = lse;
  for (int j = 0; j < nsp; ++j)
    mx = fmaxf(mx, __ldcg(plse + (static_cast<int64_t>(base + j) * a.H_kv + hk) * srows + rl));
  if (mx == -INFINITY) {
    for (int i = 0; i < n; ++i) o[i] = 0.f;
    return;
  }
  float tot = fast_exp2((lse - mx) * kLog2e);
  for (int i = 0; i < n; ++i) o[i] *= tot;
  for (int j = 0; j < nsp; ++j) {
    const int64_t row = (static_cast<int64_t>(base + j) * a.H_kv + hk) * srows + rl;
    const float w = fast_exp2((__ldcg(plse + row) - mx) * kLog2e);
    tot += w;
    const float* pj = po + row * a.D + col;
    for (int i = 0; i < n; ++i) o[i] += w * __ldcg(pj + i);
  }
  const float inv = 1.f / tot;
  for (int i = 0; i < n; ++i) o[i] *= inv;
  lse = mx + fast_log2(tot) * kLn2;
}

// Write 4 final values of a row as bf16.
__device__ __forceinline__ void store4(const AttnArgs& a, int64_t obase, const float (&v)[4]) {
  *reinterpret_cast<uint2*>(a.out + obase) = make_uint2(pack_bf16(v[0], v[1]), pack_bf16(v[2], v[3]));
}

// Partial-state slot of (group slot `slot`, KV head hk, row rl).
__device__ __forceinline__ int64_t slot_row(const AttnArgs& a, int slot, int hk, int rl) {
  return (static_cast<int64_t>(slot) * a.H_kv + hk) * a.slot_rows + rl;
}

// The last CTA of a split group merges the nsplit partial states of its R
// rows in split order (deterministic) and writes the final output. Threads
// tid in [0, nthreads) share the work, 4 columns each.
template <int D>
__device__ void combine_splits(const AttnArgs& a, int grp, int nsplit, int hk, int R, int row0,
                               int q_start, int tid, int nthreads) {
  constexpr int C4 = D / 4;
  const int G = a.G;
  for (int idx = tid; idx < R * C4; idx += nthreads) {
    const int rl = idx / C4, c4 = idx - rl * C4;
    const int pr = row0 + rl;
    const int i = pr / G;
    const int tk = q_start + i, hh = hk * G + (pr - i * G);
    float mx = -INFINITY;
    for (int jj = 0; jj < nsplit; ++jj) mx = fmaxf(mx, __ldcg(a.part_lse + slot_row(a, grp + jj, hk, rl)));
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    float lse_r = -INFINITY;
    if (mx != -INFINITY) {
      float sw = 0.f;
      for (int jj = 0; jj < nsplit; ++jj) {
        const int64_t sr = slot_row(a, grp + jj, hk, rl);
        const float w = fast_exp2((__ldcg(a.part_lse + sr) - mx) * kLog2e);
        const float4 v = __ldcg(reinterpret_cast<const float4*>(a.part_o + sr * D) + c4);
        sw += w;
        acc[0] += w * v.x;
        acc[1] += w * v.y;
        acc[2] += w * v.z;
        acc[3] += w * v.w;
      }
      const float inv = 1.f / sw;
#pragma unroll
      for (int x = 0; x < 4; ++x) acc[x] *= inv;
      lse_r = mx + fast_log2(sw) * kLn2;
    }
    const int64_t obase = (static_cast<int64_t>(tk) * a.H + hh) * D + c4 * 4;
    if (a.merge_parts) merge_prefix(a, hh, tk, c4 * 4, lse_r, acc, 4);
    store4(a, obase, acc);
    if (a.lse && c4 == 0) a.lse[static_cast<int64_t>(hh) * a.lse_stride + tk] = lse_r;
  }
}

}  // namespace pa
