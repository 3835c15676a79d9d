// Shared epilogue pieces of the attention kernels: the LSE merge with a
// cascade prefix state and the combine of split-KV partial states ("FlashAttention
// 在 vLLM 中的实现分析" §6.3 merge_attn_states, used for num_splits of §1.3).
#pragma once

#include "device_common.cuh"

namespace pa {

// Partial states are merged in batches of kBatch whose loads are all issued
// before any is used, so a merge costs a few memory latencies rather than one
// per state.
constexpr int kBatch = 4;

// Running LSE-weighted merge of (o[0..4), lse) with one batch of partial
// states given by their LSEs l[] and values v[] (n <= kBatch valid):
// the maximum moves to the batch's, both sides are rescaled, and sw sums the
// weights. o stays unnormalised until the end.
__device__ __forceinline__ void merge_batch(float& mx, float& sw, float (&o)[4],
                                            const float (&l)[kBatch], const float4 (&v)[kBatch],
                                            int n) {
  float bm = -INFINITY;
#pragma unroll
  for (int u = 0; u < kBatch; ++u)
    if (u < n) bm = fmaxf(bm, l[u]);
  if (bm == -INFINITY) return;
  const float nm = fmaxf(mx, bm);
  const float r = mx == -INFINITY ? 0.f : fast_exp2((mx - nm) * kLog2e);
  sw *= r;
#pragma unroll
  for (int x = 0; x < 4; ++x) o[x] *= r;
#pragma unroll
  for (int u = 0; u < kBatch; ++u) {
    if (u >= n) continue;
    const float w = fast_exp2((l[u] - nm) * kLog2e);
    sw += w;
    o[0] += w * v[u].x;
    o[1] += w * v[u].y;
    o[2] += w * v[u].z;
    o[3] += w * v[u].w;
  }
  mx = nm;
}

// Merge the n partial states of one row held at rows row(j) = first + j*step
// of (lse_base, o_base + col) into the running (mx, sw, o).
__device__ __forceinline__ void merge_states(float& mx, float& sw, float (&o)[4],
                                             const float* lse_base, const float* o_base,
                                             int64_t first, int64_t step, int n, int D,
                                             int col) {
  for (int j0 = 0; j0 < n; j0 += kBatch) {
    float l[kBatch];
    float4 v[kBatch];
    const int m = min(kBatch, n - j0);
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      if (u < m) {
        const int64_t row = first + static_cast<int64_t>(j0 + u) * step;
        l[u] = __ldcg(lse_base + row);
        v[u] = __ldcg(reinterpret_cast<const float4*>(o_base + row * D + col));
      }
    }
    merge_batch(mx, sw, o, l, v, m);
  }
}

// Write 4 final values of a row in the output's element type.
template <bool F16>
__device__ __forceinline__ void store4(const AttnArgs& a, int64_t obase, const float (&v)[4]) {
  using E = Elem<F16>;
  *reinterpret_cast<uint2*>(a.out + obase) = make_uint2(E::pack(v[0], v[1]), E::pack(v[2], v[3]));
}

// Partial-state slot of (group slot `slot`, KV head hk, row rl).
__device__ __forceinline__ int64_t slot_row(const AttnArgs& a, int slot, int hk, int rl) {
  return (static_cast<int64_t>(slot) * a.H_kv + hk) * a.slot_rows + rl;
}

// The last CTA of a split group (or the cascade combine kernel) merges the
// nsplit partial states of its R rows -- and, in a cascade, the prefix pass's
// states of the same rows -- and writes the final output. Threads tid in
// [0, nthreads) share the work, 4 columns each. The merge is associative and
// its order is fixed, so results are deterministic.
// In a cascade (a.merge_parts), pseg / psplit are the prefix pass's segment
// and split records (its one segment), read by the caller.
template <int D, bool F16>
__device__ void combine_splits(const AttnArgs& a, int grp, int nsplit, int hk, int R, int row0,
                               int q_start, int tid, int nthreads,
                               int4 pseg = make_int4(0, 0, 0, 0),
                               int4 psplit = make_int4(0, 0, 0, 0)) {
  constexpr int C4 = D / 4;
  const int G = a.G;
  // Prefix pass geometry (cascade): one segment holding every query token.
  int p_nsp = 0, p_base = 0, p_rows = 1, p_cls = 0;
  if (a.merge_parts) {
    p_cls = pseg.w;
    p_rows = p_cls ? tc_item_rows(G, D) : kRowsSplit;
    p_nsp = psplit.x;
    p_base = psplit.y;
  }
  const int64_t own_step = static_cast<int64_t>(a.H_kv) * a.slot_rows;
  for (int idx = tid; idx < R * C4; idx += nthreads) {
    const int rl = idx / C4, c4 = idx - rl * C4;
    const int pr = row0 + rl;
    const int i = pr / G;
    const int tk = q_start + i, hh = hk * G + (pr - i * G);
    float mx = -INFINITY, sw = 0.f;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    merge_states(mx, sw, acc, a.part_lse, a.part_o, slot_row(a, grp, hk, rl), own_step, nsplit,
                 D, c4 * 4);
    if (a.merge_parts) {
      // The row's packed index in the prefix pass is tk * G + (hh % G).
      const int ppr = tk * G + (hh - hk * G);
      const int prt = ppr / p_rows, prl = ppr - prt * p_rows;
      const int64_t srows = a.mp_slot_rows[p_cls];
      const int64_t first = (static_cast<int64_t>(p_base + prt * p_nsp) * a.H_kv + hk) * srows + prl;
      merge_states(mx, sw, acc, a.mp_part_lse[p_cls], a.mp_part_o[p_cls], first,
                   static_cast<int64_t>(a.H_kv) * srows, p_nsp, D, c4 * 4);
    }
    if (a.sinks) {   // the sink: one more state, LSE = its logit, value 0
      const float lsk[kBatch] = {__ldg(a.sinks + hh)};
      const float4 vz[kBatch] = {make_float4(0.f, 0.f, 0.f, 0.f)};
      merge_batch(mx, sw, acc, lsk, vz, 1);
    }
    float lse_r = -INFINITY;
    if (sw > 0.f) {
      const float inv = 1.f / sw;
#pragma unroll
      for (int x = 0; x < 4; ++x) acc[x] *= inv;
      lse_r = mx + fast_log2(sw) * kLn2;
    } else {
#pragma unroll
      for (int x = 0; x < 4; ++x) acc[x] = 0.f;
    }
    const int64_t obase = (static_cast<int64_t>(tk) * a.H + hh) * D + c4 * 4;
    store4<F16>(a, obase, acc);
    if (a.lse && c4 == 0) a.lse[static_cast<int64_t>(hh) * a.lse_stride + tk] = lse_r;
  }
}

}  // namespace pa
