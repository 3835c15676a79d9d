// Shared epilogue pieces of the attention kernels: the LSE merge with a
// cascade prefix state and the combine of split-KV partial states ("FlashAttention
// 在 vLLM 中的实现分析" §6.3 merge_attn_states, used for num_splits of §1.3).
#pragma once

#include "device_common.cuh"

namespace pa {

// out <- merge((prefix_o, prefix_lse), (o, lse_nat)) for n consecutive columns
// starting at element obase of a [T, H, D] row; updates lse_nat.
__device__ __forceinline__ void merge_prefix(const AttnArgs& a, int64_t obase, int h, int tok,
                                             float& lse_nat, float* o, int n) {
  const float la = a.merge_lse[static_cast<int64_t>(h) * a.lse_stride + tok];
  const float lb = lse_nat;
  const float m = fmaxf(la, lb);
  if (m == -INFINITY) {
    for (int i = 0; i < n; ++i) o[i] = 0.f;
    return;
  }
  const float wa = fast_exp2((la - m) * kLog2e), wb = fast_exp2((lb - m) * kLog2e);
  const float inv = 1.f / (wa + wb);
  for (int i = 0; i < n; ++i) o[i] = (wa * __ldcg(a.merge_o + obase + i) + wb * o[i]) * inv;
  lse_nat = m + fast_log2(wa + wb) * kLn2;
}

// Write 4 final values of a row (bf16 or fp32 destination).
__device__ __forceinline__ void store4(const AttnArgs& a, int64_t obase, const float (&v)[4]) {
  if (a.out_f32) {
    *reinterpret_cast<float4*>(a.out_f32 + obase) = make_float4(v[0], v[1], v[2], v[3]);
  } else {
    *reinterpret_cast<uint2*>(a.out + obase) =
        make_uint2(pack_bf16(v[0], v[1]), pack_bf16(v[2], v[3]));
  }
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
    if (a.merge_o) merge_prefix(a, obase, hh, tk, lse_r, acc, 4);
    store4(a, obase, acc);
    if (a.lse && c4 == 0) a.lse[static_cast<int64_t>(hh) * a.lse_stride + tk] = lse_r;
  }
}

}  // namespace pa
