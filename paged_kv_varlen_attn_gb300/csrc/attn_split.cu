// Split-KV attention kernel for decode and short-query segments.
//
// What it computes is the paged varlen attention of "FlashAttention 在 vLLM 中的
// 实现分析" §4 / §5 (block_table[seq][logical block] -> physical page, offset in
// page) with the tiled online softmax of §1.1, split over the keys as in the
// num_splits decode of §1.3, the splits recombined with the LSE-weighted merge
// of §6.3.
//
// Design (GB300):
//  * One CTA per work item (segment, row tile of <= 64 packed query rows,
//    key chunk) and KV head. Packed rows are (query token, head of the GQA
//    group), so the K/V tile read from HBM serves all G heads at once.
//  * Warp 4 is the producer: it prefetches block-table entries a group of
//    boxes ahead and issues TMA tile loads (128-byte swizzled boxes of 16-64
//    page rows x 64 dims) into a multi-stage shared-memory ring guarded by
//    full/empty mbarriers. Every wait is bounded; a timeout sets
//    PA_DEV_TIMEOUT and the call's abort word, and the CTA drains and returns.
//  * Warps 0-3 are consumers. With R packed rows, ceil(R/16) warps (rounded to
//    1, 2 or 4) take 16 rows each and the remaining factor splits every 64-key
//    tile between warps, so a decode item (R <= 16) keeps all four warps busy
//    on different keys. Q.K^T and P.V use the warp-level bf16 MMA
//    (m16n8k16, fp32 accumulate) on ldmatrix fragments; row max/sum use quad
//    shuffles; the warps' partial states are merged through shared memory.
//  * A split item writes its normalised fp32 partial (O, LSE) to the
//    workspace; the last CTA of a (row tile, KV head) group -- found with one
//    atomic counter, no spinning -- merges all splits in a fixed order, so the
//    result is deterministic.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "device_common.cuh"
#include "epilogue.cuh"

namespace pa {

template <int D>
struct SplitCfg {
  static constexpr int BN = kKeyTile;                  // keys per stage
  static constexpr int HALVES = D / 64;                // 64-dim swizzled halves
  static constexpr int HALF_BYTES = BN * 128;          // [64 rows x 128 B]
  static constexpr int TILE_BYTES = HALVES * HALF_BYTES;
  static constexpr int STAGE_BYTES = 2 * TILE_BYTES;   // K and V
  static constexpr int STAGES = D == 128 ? 2 : 6;
  static constexpr int RING_BYTES = STAGES * STAGE_BYTES;
  static constexpr int SMEM_BYTES = RING_BYTES + 1024 /*align*/ + 256 /*barriers*/;
  static constexpr int THREADS = 160;
};

struct SplitShared {
  uint64_t* full;
  uint64_t* empty;
  volatile int* flags;   // [0] abort, [1] last-CTA, [2] tiles issued, [4..7] consumed per warp
};

// ---------------------------------------------------------------------------
// Consumers. RGN = number of 16-row groups (1, 2 or 4); 4 / RGN warps share
// each group and split every key tile between them.
// ---------------------------------------------------------------------------
template <int D, int RGN>
__device__ __forceinline__ void split_consumer(const AttnArgs& a, uint8_t* ring, SplitShared sh,
                                               int hk, int seg, int rt, int j, int q_start,
                                               int q_len, int kv_len, int kb, int ke, int ntiles,
                                               int nsplit, int slot_base) {
  using C = SplitCfg<D>;
  constexpr int KS = 4 / RGN;       // warps per row group
  constexpr int KW = C::BN / KS;    // keys per warp per tile
  // A warp's keys of a tile are processed in chunks of at most 32 (one online
  // softmax step each), so the score fragments of a 64-key slice (RGN = 4)
  // do not push the consumer past its register budget.
  constexpr int KWC = KW < 32 ? KW : 32;   // keys per chunk
  constexpr int NCH = KW / KWC;            // chunks per tile
  constexpr int NT = KWC / 8;              // 8-key n-tiles per chunk
  constexpr int DK = D / 16;        // 16-dim k-steps
  constexpr int DN = D / 8;         // 8-dim n-tiles of O
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rg = warp % RGN, ks = warp / RGN;
  const int G = a.G;
  const int row0 = rt * kRowsSplit;
  const int R = min(kRowsSplit, q_len * G - row0);
  const int gq = lane >> 2, cq = lane & 3;

  // Rows owned by this thread: local rows rg*16 + gq and +8.
  int lim[2];
  bool rvalid[2];
  int tok[2], head[2];
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int rl = rg * 16 + gq + 8 * r;
    rvalid[r] = rl < R;
    const int pr = row0 + (rvalid[r] ? rl : 0);
    const int i = pr / G;
    tok[r] = q_start + i;
    head[r] = hk * G + (pr - i * G);
    lim[r] = !rvalid[r] ? -1 : (a.causal ? kv_len - q_len + i : 0x7fffffff);
  }
  int lim_max = max(lim[0], lim[1]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) lim_max = max(lim_max, __shfl_xor_sync(0xffffffffu, lim_max, o));

  // Q fragments (A operand, 16 x D), loaded once from global memory.
  uint32_t qf[DK][4];
#pragma unroll
  for (int kk = 0; kk < DK; ++kk) {
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      const int r = x & 1;                    // a0,a2: row gq; a1,a3: row gq+8
      const int col = kk * 16 + 2 * cq + (x >> 1) * 8;
      uint32_t v = 0;
      if (rvalid[r]) {
        const __nv_bfloat16* p = a.q + static_cast<int64_t>(tok[r]) * a.q_stride +
                                 static_cast<int64_t>(head[r]) * D + col;
        v = __ldg(reinterpret_cast<const uint32_t*>(p));
      }
      qf[kk][x] = v;
    }
  }

  float o[DN][4];
#pragma unroll
  for (int n = 0; n < DN; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
  const float sl2 = a.scale_log2;
  const int slice0 = ks * KW;
  int consumed = 0;

  for (int t = 0; t < ntiles; ++t) {
    const int s = t % C::STAGES;
    if (!mbar_wait(&sh.full[s], (t / C::STAGES) & 1)) {
      abort_call(a);
      sh.flags[0] = 1;
      break;
    }
    consumed = t + 1;
    uint8_t* ktile = ring + s * C::STAGE_BYTES;
    uint8_t* vtile = ktile + C::TILE_BYTES;
    const int tile_key0 = kb + t * C::BN;
    const int key_base = tile_key0 + slice0;
    if (key_base < ke && key_base <= lim_max) {
      // Keys past the sequence end inside a loaded page hold arbitrary bytes;
      // zero those V rows so 0 * garbage cannot produce NaN.
      if (tile_key0 + slice0 + KW > kv_len) {
        const int first = max(kv_len - tile_key0, slice0);
        const int nrow = slice0 + KW - first;
        for (int idx = lane; idx < nrow * C::HALVES * 8; idx += 32) {
          const int rr = first + idx / (C::HALVES * 8);
          const int rem = idx % (C::HALVES * 8);
          *reinterpret_cast<uint4*>(vtile + (rem >> 3) * C::HALF_BYTES + rr * 128 + (rem & 7) * 16) =
              make_uint4(0, 0, 0, 0);
        }
        // These generic-proxy stores precede the next TMA write of the stage.
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
      }
#pragma unroll
      for (int ch = 0; ch < NCH; ++ch) {
      const int cs = slice0 + ch * KWC;        // first key of the chunk in the tile
      const int ckey = tile_key0 + cs;
      if (ckey >= ke || ckey > lim_max) break;  // later chunks are past the range too
      float sacc[NT][4];
#pragma unroll
      for (int n = 0; n < NT; ++n) sacc[n][0] = sacc[n][1] = sacc[n][2] = sacc[n][3] = 0.f;
      const uint32_t kbase = smem_u32(ktile);
      const int mat = lane >> 3, rr = lane & 7;
#pragma unroll
      for (int kk = 0; kk < DK; ++kk) {
        const int half = kk >> 2, col = (kk & 3) * 16;
#pragma unroll
        for (int np = 0; np < NT / 2; ++np) {
          const int key = cs + np * 16 + rr + ((mat >> 1) << 3);
          const int c = col + ((mat & 1) << 3);
          uint32_t b0, b1, b2, b3;
          ldsm_x4(kbase + half * C::HALF_BYTES + sw128(key, c), b0, b1, b2, b3);
          mma_16816(sacc[2 * np], qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3], b0, b1);
          mma_16816(sacc[2 * np + 1], qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3], b2, b3);
        }
      }
      // Mask, scale into the log2 domain, running max.
      float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
      for (int n = 0; n < NT; ++n) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int key = ckey + n * 8 + 2 * cq + (e & 1);
          const int r = e >> 1;
          const bool ok = key < ke && key <= lim[r];
          const float v = ok ? sacc[n][e] * sl2 : -INFINITY;
          sacc[n][e] = v;
          mx[r] = fmaxf(mx[r], v);
        }
      }
      float alpha[2], muse[2];
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
        mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
        const float mn = fmaxf(m[r], mx[r]);
        muse[r] = mn == -INFINITY ? 0.f : mn;
        alpha[r] = fast_exp2(m[r] - muse[r]);
        m[r] = mn;
        l[r] *= alpha[r];
      }
#pragma unroll
      for (int n = 0; n < DN; ++n) {
        o[n][0] *= alpha[0];
        o[n][1] *= alpha[0];
        o[n][2] *= alpha[1];
        o[n][3] *= alpha[1];
      }
#pragma unroll
      for (int n = 0; n < NT; ++n) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float p = fast_exp2(sacc[n][e] - muse[e >> 1]);
          sacc[n][e] = p;
          l[e >> 1] += p;
        }
      }
      // O += P V.
      const uint32_t vbase = smem_u32(vtile);
#pragma unroll
      for (int kk = 0; kk < NT / 2; ++kk) {
        const uint32_t pa0 = pack_bf16(sacc[2 * kk][0], sacc[2 * kk][1]);
        const uint32_t pa1 = pack_bf16(sacc[2 * kk][2], sacc[2 * kk][3]);
        const uint32_t pa2 = pack_bf16(sacc[2 * kk + 1][0], sacc[2 * kk + 1][1]);
        const uint32_t pa3 = pack_bf16(sacc[2 * kk + 1][2], sacc[2 * kk + 1][3]);
#pragma unroll
        for (int dp = 0; dp < D / 16; ++dp) {
          const int half = dp >> 2, col = (dp & 3) * 16;
          const int key = cs + kk * 16 + rr + ((mat & 1) << 3);
          const int c = col + ((mat >> 1) << 3);
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(vbase + half * C::HALF_BYTES + sw128(key, c), b0, b1, b2, b3);
          mma_16816(o[2 * dp], pa0, pa1, pa2, pa3, b0, b1);
          mma_16816(o[2 * dp + 1], pa0, pa1, pa2, pa3, b2, b3);
        }
      }
      }   // chunk
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sh.empty[s]);
    if (sh.flags[0]) break;
  }
  if (lane == 0) sh.flags[4 + warp] = consumed;
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    l[r] += __shfl_xor_sync(0xffffffffu, l[r], 1);
    l[r] += __shfl_xor_sync(0xffffffffu, l[r], 2);
  }

  // All consumers are done with the ring: drain any load still in flight
  // (only after an abort), then reuse the ring as merge scratch.
  asm volatile("bar.sync 1, 128;" ::: "memory");
  if (threadIdx.x == 0) {
    int cmin = sh.flags[4];
    for (int w = 1; w < 4; ++w) cmin = min(cmin, sh.flags[4 + w]);
    const int issued = sh.flags[2];
    for (int t = cmin; t < issued; ++t)
      if (!mbar_wait(&sh.full[t % C::STAGES], (t / C::STAGES) & 1)) break;
  }
  asm volatile("bar.sync 1, 128;" ::: "memory");

  if constexpr (KS > 1) {
    float* scratch = reinterpret_cast<float*>(ring);
    constexpr int PER_WARP = DN * 4 * 32 + 64;   // O fragments + (m, l) of 16 rows
    if (ks > 0) {
      float* w = scratch + warp * PER_WARP;
#pragma unroll
      for (int n = 0; n < DN; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) w[(n * 4 + e) * 32 + lane] = o[n][e];
      if (cq == 0) {
        w[DN * 128 + gq] = m[0];
        w[DN * 128 + gq + 8] = m[1];
        w[DN * 128 + 16 + gq] = l[0];
        w[DN * 128 + 16 + gq + 8] = l[1];
      }
    }
    asm volatile("bar.sync 1, 128;" ::: "memory");
    if (ks == 0) {
#pragma unroll
    for (int k2 = 1; k2 < KS; ++k2) {
      const float* w = scratch + (rg + k2 * RGN) * PER_WARP;
      float alpha_a[2], alpha_b[2];
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const float mb = w[DN * 128 + gq + 8 * r];
        const float lb = w[DN * 128 + 16 + gq + 8 * r];
        const float mn = fmaxf(m[r], mb);
        const float mu = mn == -INFINITY ? 0.f : mn;
        alpha_a[r] = fast_exp2(m[r] - mu);
        alpha_b[r] = fast_exp2(mb - mu);
        l[r] = l[r] * alpha_a[r] + lb * alpha_b[r];
        m[r] = mn;
      }
#pragma unroll
      for (int n = 0; n < DN; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e)
          o[n][e] = o[n][e] * alpha_a[e >> 1] + w[(n * 4 + e) * 32 + lane] * alpha_b[e >> 1];
    }
    }
  }

  // Epilogue. Warps 0 .. RGN-1 hold the merged rows of their group; all four
  // consumer warps take part in a combine.
  float inv_l[2], lse_nat[2];
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const bool any = l[r] > 0.f;
    inv_l[r] = any ? 1.f / l[r] : 0.f;
    lse_nat[r] = any ? (m[r] + fast_log2(l[r])) * kLn2 : -INFINITY;
  }
  const int H = a.H;
  if (nsplit == 1 && !a.partials_only) {
    if (ks > 0) return;
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      if (!rvalid[r]) continue;
      const int64_t obase = (static_cast<int64_t>(tok[r]) * H + head[r]) * D;
#pragma unroll
      for (int n = 0; n < DN; ++n) {
        const int col = n * 8 + 2 * cq;
        *reinterpret_cast<uint32_t*>(a.out + obase + col) =
            pack_bf16(o[n][2 * r] * inv_l[r], o[n][2 * r + 1] * inv_l[r]);
      }
      if (a.lse && cq == 0) a.lse[static_cast<int64_t>(head[r]) * a.lse_stride + tok[r]] = lse_nat[r];
    }
    return;
  }

  // Publish the normalised partial state; then the last CTA of the group
  // merges every split (and, in a cascade suffix pass, the prefix partials)
  // with coalesced loads by all 128 consumer threads.
  const int slot = slot_base + rt * nsplit + j;
  const int64_t slot_row0 = slot_row(a, slot, hk, 0);
  if (ks == 0) {
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int rl = rg * 16 + gq + 8 * r;
      if (!rvalid[r]) continue;
      float* po = a.part_o + (slot_row0 + rl) * D;
#pragma unroll
      for (int n = 0; n < DN; ++n)
        __stcg(reinterpret_cast<float2*>(po + n * 8 + 2 * cq),
               make_float2(o[n][2 * r] * inv_l[r], o[n][2 * r + 1] * inv_l[r]));
      if (cq == 0) __stcg(a.part_lse + slot_row0 + rl, lse_nat[r]);
    }
  }
  if (a.partials_only) return;   // cascade prefix pass: the suffix pass merges
  __threadfence();
  asm volatile("bar.sync 2, 128;" ::: "memory");
  const int grp = slot_base + rt * nsplit;
  int* counter = a.counters + static_cast<int64_t>(grp) * a.H_kv + hk;
  if (threadIdx.x == 0) sh.flags[1] = (atomicAdd(counter, 1) == nsplit - 1) ? 1 : 0;
  asm volatile("bar.sync 2, 128;" ::: "memory");
  if (!sh.flags[1]) return;
  __threadfence();
  combine_splits<D>(a, grp, nsplit, hk, R, row0, q_start, threadIdx.x, 128);
  if (threadIdx.x == 0) *counter = 0;   // ready for the next call
}

template <int D>
__global__ void __launch_bounds__(SplitCfg<D>::THREADS, 3)
attn_split_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                  const __grid_constant__ AttnArgs a) {
  using C = SplitCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  SplitShared sh;
  sh.full = reinterpret_cast<uint64_t*>(ring + C::RING_BYTES);
  sh.empty = sh.full + C::STAGES;
  sh.flags = reinterpret_cast<volatile int*>(sh.empty + C::STAGES);

  // One block per (work item, KV head), KV head fastest: blocks are
  // dispatched in index order and the planner sorted the items longest first.
  const int item = static_cast<int>(blockIdx.x) / a.H_kv;
  const int hk = static_cast<int>(blockIdx.x) - item * a.H_kv;
  pdl_enter(a.pdl_first);
  if (item >= a.header[0] || call_aborted(a)) return;
  const int4 it = a.items[item];
  const int seg = it.x, rt = it.y, j = it.z;
  const int4 sg = a.seg[seg];
  const int4 sp = a.segsplit[seg];
  const int q_start = sg.x, q_len = sg.y, kv_len = sg.z;
  const int nsplit = sp.x, slot_base = sp.y, chunk = sp.z;
  const int G = a.G;
  const int row0 = rt * kRowsSplit;
  const int R = min(kRowsSplit, q_len * G - row0);
  const int kb = j * chunk;
  int ke = min(kv_len, kb + chunk);
  if (a.causal) {
    const int i_last = (row0 + R - 1) / G;
    ke = min(ke, kv_len - q_len + i_last + 1);
  }
  const int ntiles = ke > kb ? (ke - kb + C::BN - 1) / C::BN : 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&sh.full[s], 1);
      mbar_init(&sh.empty[s], 4);
    }
    for (int f = 0; f < 8; ++f) sh.flags[f] = 0;
    fence_mbar_init();
  }
  __syncthreads();

  const int warp = threadIdx.x >> 5;
  if (warp == 4) {
    if (ntiles > 0) {
      const int32_t* bt_row = a.bt + static_cast<int64_t>(seg) * a.bt_row_stride + a.bt_col_offset;
      produce_kv<C::BN, C::HALVES, C::STAGES>(&tmK, &tmV, a, ring, sh.full, sh.empty,
                                              &sh.flags[0], &sh.flags[2], bt_row, hk, kb, kv_len,
                                              ntiles, threadIdx.x & 31);
    }
    return;
  }
  if (R <= 16)
    split_consumer<D, 1>(a, ring, sh, hk, seg, rt, j, q_start, q_len, kv_len, kb, ke, ntiles,
                         nsplit, slot_base);
  else if (R <= 32)
    split_consumer<D, 2>(a, ring, sh, hk, seg, rt, j, q_start, q_len, kv_len, kb, ke, ntiles,
                         nsplit, slot_base);
  else
    split_consumer<D, 4>(a, ring, sh, hk, seg, rt, j, q_start, q_len, kv_len, kb, ke, ntiles,
                         nsplit, slot_base);
}

template <int D>
static cudaError_t launch_split_d(const CUtensorMap& tmK, const CUtensorMap& tmV,
                                  const AttnArgs& a, int items_bound, cudaStream_t st) {
  using C = SplitCfg<D>;
  // The shared-memory opt-in is a per-device function attribute: set it on
  // the first launch on each device (before any stream capture), not again.
  static bool configured[kMaxDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices || !configured[dev]) {
    e = cudaFuncSetAttribute(attn_split_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < kMaxDevices) configured[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(items_bound) * static_cast<unsigned>(a.H_kv));
  cfg.blockDim = dim3(C::THREADS);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, attn_split_kernel<D>, tmK, tmV, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_attn_split(const CUtensorMap& tmK, const CUtensorMap& tmV, const AttnArgs& a,
                              int items_bound, cudaStream_t st) {
  if (items_bound <= 0) return cudaSuccess;
  if (a.D == 128) return launch_split_d<128>(tmK, tmV, a, items_bound, st);
  return launch_split_d<64>(tmK, tmV, a, items_bound, st);
}

}  // namespace pa
