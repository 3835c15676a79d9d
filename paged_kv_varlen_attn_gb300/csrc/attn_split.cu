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
//  * FP8 (e4m3) pools ("FlashAttention と FlashInfer" 役割 / 境界と失敗: FP8
//    KV cache with per-head quant scales), head size 128: a key row is one
//    128-byte swizzled line, so a 64-key stage is half bf16's bytes (4 stages).
//    Decode items (<= 8 packed rows) run split_consumer_fp8_dec (Q.K^T on the
//    e4m3 MMA). Wider items: each warp widens its slice from the staged bytes
//    into f16 MMA fragments (exact), Q in f16. For Q.K^T the head dimension
//    is permuted -- MMA k-index 16*kk + {2c, 2c+1, 2c+8, 2c+9} of lane quad
//    c is dim 32*c + 4*kk + {0..3} in Q and K -- so a lane's K bytes of a
//    key are 32 contiguous bytes. For P.V the output dimension is permuted --
//    MMA column g of n-tile n is dim 16*g + n -- so a lane reads 16 bytes of
//    each of its four keys and pairs them with byte permutes. k_scale folds
//    into the softmax scale and v_scale into the final normalisation.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>

#include "device_common.cuh"
#include "epilogue.cuh"

namespace pa {

template <int D, bool FP8 = false>
struct SplitCfg {
  static constexpr int BN = kKeyTile;                  // keys per stage
  static constexpr int HALVES = FP8 ? 1 : D / 64;      // 128-byte swizzled row segments
  static constexpr int HALF_BYTES = BN * 128;          // [64 rows x 128 B]
  static constexpr int TILE_BYTES = HALVES * HALF_BYTES;
  static constexpr int STAGE_BYTES = 2 * TILE_BYTES;   // K and V
  // 3 CTAs per SM (128 registers per thread). FP8 stages are half the size,
  // so it keeps 4 of them: 2/3 of bf16's bytes in flight, which its
  // (latency-bound) decode consumer does not need more of; measured, 3 CTAs
  // x 4 stages beat 2 CTAs x 6 stages by 9% on decode.
  static constexpr int STAGES = FP8 ? 4 : (D == 128 ? 2 : 6);
  static constexpr int CTAS_PER_SM = 3;
  static constexpr int RING_BYTES = STAGES * STAGE_BYTES;
  static constexpr int SMEM_BYTES = RING_BYTES + 1024 /*align*/ + 256 /*barriers*/;
  static constexpr int THREADS = 160;
};

struct SplitShared {
  uint64_t* full;
  uint64_t* empty;
  volatile int* flags;   // [0] abort, [1] last-CTA, [2] tiles issued, [4..7] consumed per warp
};

// After all four consumer warps have published their item's partial state:
// the last CTA of the (row tile, KV head) group -- found with one atomic
// counter, no spinning -- merges every split (and, in a cascade, the prefix
// partials) with coalesced loads by all 128 consumer threads.
template <int D, bool F16>
__device__ __forceinline__ void finish_group(const AttnArgs& a, SplitShared sh, int slot_base,
                                             int rt, int nsplit, int hk, int R, int row0,
                                             int q_start) {
  if (a.partials_only) return;   // cascade: the combine kernel merges
  __threadfence();
  asm volatile("bar.sync 2, 128;" ::: "memory");
  const int grp = slot_base + rt * nsplit;
  int* counter = a.counters + static_cast<int64_t>(grp) * a.H_kv + hk;
  if (threadIdx.x == 0) sh.flags[1] = (atomicAdd(counter, 1) == nsplit - 1) ? 1 : 0;
  asm volatile("bar.sync 2, 128;" ::: "memory");
  if (!sh.flags[1]) return;
  __threadfence();
  combine_splits<D, F16>(a, grp, nsplit, hk, R, row0, q_start, threadIdx.x, 128);
  if (threadIdx.x == 0) *counter = 0;   // ready for the next call
}

// After the key loop: record how many tiles this warp consumed, wait until
// every consumer warp is done with the ring and drain any load still in
// flight (only after an abort), so the ring can be reused as scratch.
template <int STAGES>
__device__ __forceinline__ void drain_ring(SplitShared sh, int warp, int lane, int consumed) {
  if (lane == 0) sh.flags[4 + warp] = consumed;
  asm volatile("bar.sync 1, 128;" ::: "memory");
  if (threadIdx.x == 0) {
    int cmin = sh.flags[4];
    for (int w = 1; w < 4; ++w) cmin = min(cmin, sh.flags[4 + w]);
    const int issued = sh.flags[2];
    for (int t = cmin; t < issued; ++t)
      if (!mbar_wait(&sh.full[t % STAGES], (t / STAGES) & 1)) break;
  }
  asm volatile("bar.sync 1, 128;" ::: "memory");
}

// Keys past the sequence end inside a loaded page hold arbitrary bytes: zero
// the V rows [max(kv_len - tile_key0, slice0), slice0 + KW) of this warp's
// slice so that 0 * garbage cannot produce NaN.
template <int KW, int HALVES, int HALF_BYTES>
__device__ __forceinline__ void zero_v_tail(uint8_t* vtile, int tile_key0, int slice0, int kv_len,
                                            int lane) {
  if (tile_key0 + slice0 + KW <= kv_len) return;
  const int first = max(kv_len - tile_key0, slice0);
  const int nrow = slice0 + KW - first;
  for (int idx = lane; idx < nrow * HALVES * 8; idx += 32) {
    const int rr = first + idx / (HALVES * 8);
    const int rem = idx % (HALVES * 8);
    *reinterpret_cast<uint4*>(vtile + (rem >> 3) * HALF_BYTES + rr * 128 + (rem & 7) * 16) =
        make_uint4(0, 0, 0, 0);
  }
  // These generic-proxy stores precede the next TMA write of the stage.
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  __syncwarp();
}

// ---------------------------------------------------------------------------
// Consumers. RGN = number of 16-row groups (1, 2 or 4); 4 / RGN warps share
// each group and split every key tile between them.
// ---------------------------------------------------------------------------
template <int D, int RGN, bool FP8, bool F16>
__device__ __forceinline__ void split_consumer(const AttnArgs& a, uint8_t* ring, SplitShared sh,
                                               int hk, int seg, int rt, int j, int q_start,
                                               int q_len, int kv_len, int kb, int ke, int ntiles,
                                               int nsplit, int slot_base) {
  using C = SplitCfg<D, FP8>;
  using E = Elem<F16>;
  static_assert(!FP8 || D == 128, "FP8 pools: head size 128");
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
  // Smallest limit over the warp's valid rows (rows past R are never written).
  int lim_min = min(rvalid[0] ? lim[0] : 0x7fffffff, rvalid[1] ? lim[1] : 0x7fffffff);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) lim_min = min(lim_min, __shfl_xor_sync(0xffffffffu, lim_min, o));

  // Q fragments (A operand, 16 x D), loaded once from global memory: bf16,
  // or for FP8 pools f16 in the permuted dim order of the K fragments.
  uint32_t qf[DK][4];
#pragma unroll
  for (int kk = 0; kk < DK; ++kk) {
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      const int r = x & 1;                    // a0,a2: row gq; a1,a3: row gq+8
      const int col = FP8 ? cq * 32 + kk * 4 + (x >> 1) * 2 : kk * 16 + 2 * cq + (x >> 1) * 8;
      uint32_t v = 0;
      if (rvalid[r]) {
        const uint16_t* p = a.q + static_cast<int64_t>(tok[r]) * a.q_stride +
                            static_cast<int64_t>(head[r]) * D + col;
        v = __ldg(reinterpret_cast<const uint32_t*>(p));
        if constexpr (FP8 && !F16) {   // the FP8 consumers multiply in f16
          const float2 f = Elem<false>::unpack(v);
          v = pack_f16(f.x, f.y);
        }
      }
      qf[kk][x] = v;
    }
  }

  float o[DN][4];
#pragma unroll
  for (int n = 0; n < DN; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
  // FP8: scores use the stored codes, so k_scale joins the softmax scale;
  // v_scale multiplies the normalised output.
  const float sl2 = FP8 ? a.scale_log2 * __ldg(a.k_scale + hk) : a.scale_log2;
  const float vsc = FP8 ? __ldg(a.v_scale + hk) : 1.f;
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
      zero_v_tail<KW, C::HALVES, C::HALF_BYTES>(vtile, tile_key0, slice0, kv_len, lane);
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
      if constexpr (FP8) {
        // Lane (gq, cq) holds key cs + 8n + gq, bytes 32*cq .. +31 (16-byte
        // granules 2cq, 2cq+1 of the swizzled row); word kk gives b0 (low
        // half) and b1 (high half) of k-step kk.
#pragma unroll
        for (int n = 0; n < NT; ++n) {
          const int key = cs + n * 8 + gq;
          const uint8_t* row = ktile + key * 128;
          const uint4 w0 = *reinterpret_cast<const uint4*>(row + (((2 * cq) ^ (key & 7)) << 4));
          const uint4 w1 = *reinterpret_cast<const uint4*>(row + (((2 * cq + 1) ^ (key & 7)) << 4));
          const uint32_t w[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
          for (int kk = 0; kk < DK; ++kk)
            mma_16816_f16(sacc[n], qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3],
                          e4m3x2_to_f16x2(w[kk]), e4m3x2_to_f16x2(w[kk] >> 16));
        }
      } else {
#pragma unroll
      for (int kk = 0; kk < DK; ++kk) {
        const int half = kk >> 2, col = (kk & 3) * 16;
#pragma unroll
        for (int np = 0; np < NT / 2; ++np) {
          const int key = cs + np * 16 + rr + ((mat >> 1) << 3);
          const int c = col + ((mat & 1) << 3);
          uint32_t b0, b1, b2, b3;
          ldsm_x4(kbase + half * C::HALF_BYTES + sw128(key, c), b0, b1, b2, b3);
          E::mma(sacc[2 * np], qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3], b0, b1);
          E::mma(sacc[2 * np + 1], qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3], b2, b3);
        }
      }
      }
      // Mask, scale into the log2 domain, running max. A chunk inside every
      // valid row's visible range needs no mask.
      float mx[2] = {-INFINITY, -INFINITY};
      if (ckey + KWC <= ke && ckey + KWC - 1 <= lim_min) {
#pragma unroll
        for (int n = 0; n < NT; ++n) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float v = sacc[n][e] * sl2;
            sacc[n][e] = v;
            mx[e >> 1] = fmaxf(mx[e >> 1], v);
          }
        }
      } else {
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
      }
      float alpha[2], muse[2];
      bool grew = false;
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
        mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
        const float mn = fmaxf(m[r], mx[r]);
        grew |= mn != m[r];
        muse[r] = mn == -INFINITY ? 0.f : mn;
        alpha[r] = fast_exp2(m[r] - muse[r]);
        m[r] = mn;
        l[r] *= alpha[r];
      }
      // alpha is exactly 1 for a row whose maximum did not move; skip the
      // rescale unless some row's did.
      if (__any_sync(0xffffffffu, grew)) {
#pragma unroll
      for (int n = 0; n < DN; ++n) {
        o[n][0] *= alpha[0];
        o[n][1] *= alpha[0];
        o[n][2] *= alpha[1];
        o[n][3] *= alpha[1];
      }
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
      if constexpr (FP8) {
        // Lane (gq, cq) needs, for the keys of MMA k-index 2cq, 2cq+1, 2cq+8,
        // 2cq+9 of each 16-key step, the dims 16*gq + n of n-tile n: granule
        // gq of those four rows. prmt pairs byte n of two rows into the
        // (low, high) e4m3 pair of one B register.
#pragma unroll
        for (int kk = 0; kk < NT / 2; ++kk) {
          const uint32_t pa0 = pack_f16(sacc[2 * kk][0], sacc[2 * kk][1]);
          const uint32_t pa1 = pack_f16(sacc[2 * kk][2], sacc[2 * kk][3]);
          const uint32_t pa2 = pack_f16(sacc[2 * kk + 1][0], sacc[2 * kk + 1][1]);
          const uint32_t pa3 = pack_f16(sacc[2 * kk + 1][2], sacc[2 * kk + 1][3]);
          uint4 vr[4];
#pragma unroll
          for (int x = 0; x < 4; ++x) {
            const int key = cs + kk * 16 + 2 * cq + (x & 1) + (x >> 1) * 8;
            vr[x] = *reinterpret_cast<const uint4*>(vtile + key * 128 + ((gq ^ (key & 7)) << 4));
          }
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint32_t x0 = (&vr[0].x)[j], x1 = (&vr[1].x)[j];
            const uint32_t x2 = (&vr[2].x)[j], x3 = (&vr[3].x)[j];
            const uint32_t lo01 = prmt(x0, x1, 0x5140), hi01 = prmt(x0, x1, 0x7362);
            const uint32_t lo23 = prmt(x2, x3, 0x5140), hi23 = prmt(x2, x3, 0x7362);
            mma_16816_f16(o[4 * j], pa0, pa1, pa2, pa3, e4m3x2_to_f16x2(lo01),
                          e4m3x2_to_f16x2(lo23));
            mma_16816_f16(o[4 * j + 1], pa0, pa1, pa2, pa3, e4m3x2_to_f16x2(lo01 >> 16),
                          e4m3x2_to_f16x2(lo23 >> 16));
            mma_16816_f16(o[4 * j + 2], pa0, pa1, pa2, pa3, e4m3x2_to_f16x2(hi01),
                          e4m3x2_to_f16x2(hi23));
            mma_16816_f16(o[4 * j + 3], pa0, pa1, pa2, pa3, e4m3x2_to_f16x2(hi01 >> 16),
                          e4m3x2_to_f16x2(hi23 >> 16));
          }
        }
      } else {
#pragma unroll
      for (int kk = 0; kk < NT / 2; ++kk) {
        const uint32_t pa0 = E::pack(sacc[2 * kk][0], sacc[2 * kk][1]);
        const uint32_t pa1 = E::pack(sacc[2 * kk][2], sacc[2 * kk][3]);
        const uint32_t pa2 = E::pack(sacc[2 * kk + 1][0], sacc[2 * kk + 1][1]);
        const uint32_t pa3 = E::pack(sacc[2 * kk + 1][2], sacc[2 * kk + 1][3]);
#pragma unroll
        for (int dp = 0; dp < D / 16; ++dp) {
          const int half = dp >> 2, col = (dp & 3) * 16;
          const int key = cs + kk * 16 + rr + ((mat & 1) << 3);
          const int c = col + ((mat >> 1) << 3);
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(vbase + half * C::HALF_BYTES + sw128(key, c), b0, b1, b2, b3);
          E::mma(o[2 * dp], pa0, pa1, pa2, pa3, b0, b1);
          E::mma(o[2 * dp + 1], pa0, pa1, pa2, pa3, b2, b3);
        }
      }
      }
      }   // chunk
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sh.empty[s]);
    if (sh.flags[0]) break;
  }
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    l[r] += __shfl_xor_sync(0xffffffffu, l[r], 1);
    l[r] += __shfl_xor_sync(0xffffffffu, l[r], 2);
  }
  // All consumers are done with the ring: reuse it as merge scratch.
  drain_ring<C::STAGES>(sh, warp, lane, consumed);

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
    inv_l[r] = any ? vsc / l[r] : 0.f;
    lse_nat[r] = any ? (m[r] + fast_log2(l[r])) * kLn2 : -INFINITY;
  }
  const int H = a.H;
  if (nsplit == 1 && !a.partials_only) {
    if (ks > 0) return;
    if (a.sinks) {
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        if (!rvalid[r]) continue;
        float mm = m[r], ll = l[r];
        const float f = add_sink(mm, ll, __ldg(a.sinks + head[r]) * kLog2e);
        inv_l[r] = ll > 0.f ? vsc * f / ll : 0.f;
        lse_nat[r] = ll > 0.f ? (mm + fast_log2(ll)) * kLn2 : -INFINITY;
      }
    }
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      if (!rvalid[r]) continue;
      const int64_t obase = (static_cast<int64_t>(tok[r]) * H + head[r]) * D;
      if constexpr (FP8) {
        // Column e of the lane's pair holds dims 16 * (2cq + e) + n, n = 0..15.
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          uint32_t pk[8];
#pragma unroll
          for (int n = 0; n < DN; n += 2)
            pk[n / 2] = E::pack(o[n][2 * r + e] * inv_l[r], o[n + 1][2 * r + e] * inv_l[r]);
          uint4* dst = reinterpret_cast<uint4*>(a.out + obase + 16 * (2 * cq + e));
          dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
          dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
        }
      } else {
#pragma unroll
      for (int n = 0; n < DN; ++n) {
        const int col = n * 8 + 2 * cq;
        *reinterpret_cast<uint32_t*>(a.out + obase + col) =
            E::pack(o[n][2 * r] * inv_l[r], o[n][2 * r + 1] * inv_l[r]);
      }
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
      if constexpr (FP8) {
#pragma unroll
        for (int e = 0; e < 2; ++e)
#pragma unroll
          for (int n = 0; n < DN; n += 4)
            __stcg(reinterpret_cast<float4*>(po + 16 * (2 * cq + e) + n),
                   make_float4(o[n][2 * r + e] * inv_l[r], o[n + 1][2 * r + e] * inv_l[r],
                               o[n + 2][2 * r + e] * inv_l[r], o[n + 3][2 * r + e] * inv_l[r]));
      } else {
#pragma unroll
      for (int n = 0; n < DN; ++n)
        __stcg(reinterpret_cast<float2*>(po + n * 8 + 2 * cq),
               make_float2(o[n][2 * r] * inv_l[r], o[n][2 * r + 1] * inv_l[r]));
      }
      if (cq == 0) __stcg(a.part_lse + slot_row0 + rl, lse_nat[r]);
    }
  }
  finish_group<D, F16>(a, sh, slot_base, rt, nsplit, hk, R, row0, q_start);
}

// ---------------------------------------------------------------------------
// FP8 decode consumer, items of R <= 8 packed rows (decode with GQA <= 8).
// The products are taken transposed, S^T = K Q^T and O^T = V^T P^T: the 16
// keys of a warp's slice are the MMA's M dimension and the <= 8 query rows
// its N = 8, so no MMA work goes to padding rows beyond the 8-row tile, and
// O^T needs half the accumulator registers. Lane (g, c) = (lane / 4,
// lane % 4).
//  * S^T on the e4m3 tensor MMA (m16n8k32): A = K (keys x dims) straight from
//    the staged bytes of rows g and g + 8 of the slice -- no conversion --
//    with the head dimension permuted so that k-indices 32 ks + 4c + {0..3}
//    and 32 ks + 16 + 4c + {0..3} are dims 32 c + 8 ks + {0..7}: a lane's K
//    bytes of a key are 32 contiguous bytes. B = Q^T, column g = packed row
//    g, as two e4m3 terms: with a power-of-two row scale 2^k putting the
//    row's largest |q| in [128, 256), q 2^k = Qh + Ql where Qh = e4m3(q 2^k)
//    and Ql = e4m3(q 2^k - Qh). A bf16 q has 8 significant bits and Qh
//    keeps 4, so the remainder (a multiple of 2^(E-7), at most 2^(E-4) in
//    size) fits e4m3 exactly whenever q 2^k >= 2^-2; smaller elements keep
//    an absolute error below 2^-10 2^-k. 2^-k joins the row's softmax scale.
//    The accumulator holds keys g, g + 8 for rows 2c, 2c + 1.
//  * P^T as the B operand of the second product is the transpose of that
//    accumulator layout: one movmatrix per 8 keys, in f16.
//  * O^T: A = V^T (dims x keys) in f16 with the output dimension permuted --
//    row r of m-tile mt is dim 8 r + mt -- so lane g reads 8 contiguous bytes
//    of each of its four keys twice (dims 8 g .. 8 g + 7 and 64 + 8 g ..),
//    pairs two keys' bytes with byte permutes and widens them (exact).
// The four warps take 16 keys each of every 64-key tile; their states are
// merged through shared memory as in the other consumer.
// ---------------------------------------------------------------------------
template <bool F16>
__device__ __forceinline__ void split_consumer_fp8_dec(const AttnArgs& a, uint8_t* ring,
                                                       SplitShared sh, int hk, int rt, int j,
                                                       int q_start, int q_len, int kv_len, int kb,
                                                       int ke, int ntiles, int nsplit,
                                                       int slot_base) {
  using C = SplitCfg<128, true>;
  constexpr int D = 128;
  constexpr int KW = C::BN / 4;     // keys per warp per tile
  constexpr int MT = D / 16;        // m-tiles of O^T
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int G = a.G;
  const int row0 = rt * kRowsSplit;
  const int R = min(kRowsSplit, q_len * G - row0);

  // Accumulator columns of this lane: packed rows 2c and 2c + 1.
  int lim[2];
  bool rvalid[2];
  int tok[2], head[2];
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    const int rl = 2 * c + e;
    rvalid[e] = rl < R;
    const int pr = row0 + (rvalid[e] ? rl : 0);
    const int i = pr / G;
    tok[e] = q_start + i;
    head[e] = hk * G + (pr - i * G);
    lim[e] = !rvalid[e] ? -1 : (a.causal ? kv_len - q_len + i : 0x7fffffff);
  }
  int lim_max = max(lim[0], lim[1]);
  int lim_min = min(rvalid[0] ? lim[0] : 0x7fffffff, rvalid[1] ? lim[1] : 0x7fffffff);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    lim_max = max(lim_max, __shfl_xor_sync(0xffffffffu, lim_max, o));
    lim_min = min(lim_min, __shfl_xor_sync(0xffffffffu, lim_min, o));
  }

  // Q^T fragments (B operand, e4m3): column g is packed row g; lane (g, c)
  // holds its dims 32c .. 32c + 31 as Qh and Ql bytes (4 per register).
  constexpr int KS8 = D / 32;       // k-steps of S^T
  uint32_t qh[KS8][2], ql[KS8][2];
  float rscale[2];                  // 2^-k of rows 2c and 2c + 1
  {
    const bool qv = g < R;
    int tq = 0, hq = 0;
    if (qv) {
      const int pr = row0 + g;
      const int i = pr / G;
      tq = q_start + i;
      hq = hk * G + (pr - i * G);
    }
    const uint4* qrow = reinterpret_cast<const uint4*>(
        a.q + static_cast<int64_t>(tq) * a.q_stride + static_cast<int64_t>(hq) * D + c * 32);
    float qf[32];
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      const uint4 u = qv ? __ldg(qrow + v) : make_uint4(0, 0, 0, 0);
      const uint32_t uw[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        const float2 f = Elem<F16>::unpack(uw[x]);
        qf[8 * v + 2 * x] = f.x;
        qf[8 * v + 2 * x + 1] = f.y;
      }
    }
    float amax = 0.f;
#pragma unroll
    for (int x = 0; x < 32; ++x) amax = fmaxf(amax, fabsf(qf[x]));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    // 2^k with amax 2^k in [128, 256): k = 7 - floor(log2 amax). A zero or
    // subnormal row maximum takes k = 126 (the row's scores are ~0 anyway).
    const int ebits = (__float_as_int(amax) >> 23) & 0xFF;
    const int kexp = ebits == 0 ? 126 : 134 - ebits;      // in [-120, 133]
    const int kc = max(-126, min(126, kexp));
    const float up = __int_as_float((127 + kc) << 23), down = __int_as_float((127 - kc) << 23);
#pragma unroll
    for (int ks = 0; ks < KS8; ++ks) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t hi = 0, lo = 0;
#pragma unroll
        for (int x = 0; x < 4; x += 2) {
          const float y0 = qf[8 * ks + 4 * h + x] * up, y1 = qf[8 * ks + 4 * h + x + 1] * up;
          const uint32_t hb = f32x2_to_e4m3x2(y0, y1);
          const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(
              static_cast<__nv_fp8x2_storage_t>(hb), __NV_E4M3);
          const float2 hv = __half22float2(*reinterpret_cast<const __half2*>(&hr));
          hi |= hb << (8 * x);
          lo |= f32x2_to_e4m3x2(y0 - hv.x, y1 - hv.y) << (8 * x);
        }
        qh[ks][h] = hi;
        ql[ks][h] = lo;
      }
    }
    // Row 2c + e's scale lives in the lanes of column g = 2c + e.
#pragma unroll
    for (int e = 0; e < 2; ++e) rscale[e] = __shfl_sync(0xffffffffu, down, (2 * c + e) * 4);
  }

  float o[MT][4];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
  float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
  const float ksl2 = a.scale_log2 * __ldg(a.k_scale + hk);
  const float sl2r[2] = {ksl2 * rscale[0], ksl2 * rscale[1]};
  const float vsc = __ldg(a.v_scale + hk);
  const int slice0 = warp * KW;
  int consumed = 0;

  for (int t = 0; t < ntiles; ++t) {
    const int s = t % C::STAGES;
    if (!mbar_wait(&sh.full[s], (t / C::STAGES) & 1)) {
      abort_call(a);
      sh.flags[0] = 1;
      break;
    }
    consumed = t + 1;
    const uint8_t* ktile = ring + s * C::STAGE_BYTES;
    uint8_t* vtile = ring + s * C::STAGE_BYTES + C::TILE_BYTES;
    const int tile_key0 = kb + t * C::BN;
    const int ckey = tile_key0 + slice0;
    if (ckey < ke && ckey <= lim_max) {
      zero_v_tail<KW, C::HALVES, C::HALF_BYTES>(vtile, tile_key0, slice0, kv_len, lane);
      // S^T for keys slice0 + g (rows of a0, a2) and slice0 + g + 8 (a1, a3).
      float st[4] = {0.f, 0.f, 0.f, 0.f};
      {
        const int k0 = slice0 + g, k1 = k0 + 8;
        const uint8_t* r0 = ktile + k0 * 128;
        const uint8_t* r1 = ktile + k1 * 128;
        const uint4 a0 = *reinterpret_cast<const uint4*>(r0 + (((2 * c) ^ (k0 & 7)) << 4));
        const uint4 a1 = *reinterpret_cast<const uint4*>(r0 + (((2 * c + 1) ^ (k0 & 7)) << 4));
        const uint4 b0 = *reinterpret_cast<const uint4*>(r1 + (((2 * c) ^ (k1 & 7)) << 4));
        const uint4 b1 = *reinterpret_cast<const uint4*>(r1 + (((2 * c + 1) ^ (k1 & 7)) << 4));
        const uint32_t wa[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
        const uint32_t wb[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
        for (int ks = 0; ks < KS8; ++ks) {
          mma_16832_e4m3(st, wa[2 * ks], wb[2 * ks], wa[2 * ks + 1], wb[2 * ks + 1], qh[ks][0],
                         qh[ks][1]);
          mma_16832_e4m3(st, wa[2 * ks], wb[2 * ks], wa[2 * ks + 1], wb[2 * ks + 1], ql[ks][0],
                         ql[ks][1]);
        }
      }
      // Mask (keys ckey + g and ckey + g + 8; rows 2c + (e & 1)), scale, max.
      if (ckey + KW <= ke && ckey + KW - 1 <= lim_min) {
#pragma unroll
        for (int e = 0; e < 4; ++e) st[e] *= sl2r[e & 1];
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int key = ckey + g + (e >> 1) * 8;
          const bool ok = key < ke && key <= lim[e & 1];
          st[e] = ok ? st[e] * sl2r[e & 1] : -INFINITY;
        }
      }
      float mx[2] = {fmaxf(st[0], st[2]), fmaxf(st[1], st[3])};
      float alpha[2], muse[2];
      bool grew = false;
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        mx[e] = fmaxf(mx[e], __shfl_xor_sync(0xffffffffu, mx[e], 4));
        mx[e] = fmaxf(mx[e], __shfl_xor_sync(0xffffffffu, mx[e], 8));
        mx[e] = fmaxf(mx[e], __shfl_xor_sync(0xffffffffu, mx[e], 16));
        const float mn = fmaxf(m[e], mx[e]);
        grew |= mn != m[e];
        muse[e] = mn == -INFINITY ? 0.f : mn;
        alpha[e] = fast_exp2(m[e] - muse[e]);
        m[e] = mn;
        l[e] *= alpha[e];
      }
      // alpha is exactly 1 for a row whose maximum did not move.
      if (__any_sync(0xffffffffu, grew)) {
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          o[mt][0] *= alpha[0];
          o[mt][1] *= alpha[1];
          o[mt][2] *= alpha[0];
          o[mt][3] *= alpha[1];
        }
      }
      float p[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        p[e] = fast_exp2(st[e] - muse[e & 1]);
        l[e & 1] += p[e];
      }
      // P^T fragments: transpose of (keys g | rows 2c, 2c+1) for keys 0-7 and 8-15.
      const uint32_t pb0 = movmatrix_trans(pack_f16(p[0], p[1]));
      const uint32_t pb1 = movmatrix_trans(pack_f16(p[2], p[3]));
      // V^T fragments: keys slice0 + 2c + {0, 1, 8, 9}; dims 8g + mt (run A)
      // and 64 + 8g + mt (run B), 8 bytes each.
      uint2 va[4], vb[4];
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        const int key = slice0 + 2 * c + (x & 1) + (x >> 1) * 8;
        const uint8_t* row = vtile + key * 128 + (g & 1) * 8;
        va[x] = *reinterpret_cast<const uint2*>(row + (((g >> 1) ^ (key & 7)) << 4));
        vb[x] = *reinterpret_cast<const uint2*>(row + (((4 + (g >> 1)) ^ (key & 7)) << 4));
      }
      // This warp's reads of the stage are done: release it before the P V
      // products (123.1 us against 124.0 us on the Llama-8B decode batch;
      // releasing it before any arithmetic, with every fragment loaded
      // first, measured 135.7 us).
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.empty[s]);
#pragma unroll
      for (int w = 0; w < 2; ++w) {
        const uint32_t a01 = w ? va[0].y : va[0].x, a01b = w ? va[1].y : va[1].x;
        const uint32_t a23 = w ? va[2].y : va[2].x, a23b = w ? va[3].y : va[3].x;
        const uint32_t b01 = w ? vb[0].y : vb[0].x, b01b = w ? vb[1].y : vb[1].x;
        const uint32_t b23 = w ? vb[2].y : vb[2].x, b23b = w ? vb[3].y : vb[3].x;
        const uint32_t lo_a01 = prmt(a01, a01b, 0x5140), hi_a01 = prmt(a01, a01b, 0x7362);
        const uint32_t lo_b01 = prmt(b01, b01b, 0x5140), hi_b01 = prmt(b01, b01b, 0x7362);
        const uint32_t lo_a23 = prmt(a23, a23b, 0x5140), hi_a23 = prmt(a23, a23b, 0x7362);
        const uint32_t lo_b23 = prmt(b23, b23b, 0x5140), hi_b23 = prmt(b23, b23b, 0x7362);
        mma_16816_f16(o[4 * w], e4m3x2_to_f16x2(lo_a01), e4m3x2_to_f16x2(lo_b01),
                      e4m3x2_to_f16x2(lo_a23), e4m3x2_to_f16x2(lo_b23), pb0, pb1);
        mma_16816_f16(o[4 * w + 1], e4m3x2_to_f16x2(lo_a01 >> 16), e4m3x2_to_f16x2(lo_b01 >> 16),
                      e4m3x2_to_f16x2(lo_a23 >> 16), e4m3x2_to_f16x2(lo_b23 >> 16), pb0, pb1);
        mma_16816_f16(o[4 * w + 2], e4m3x2_to_f16x2(hi_a01), e4m3x2_to_f16x2(hi_b01),
                      e4m3x2_to_f16x2(hi_a23), e4m3x2_to_f16x2(hi_b23), pb0, pb1);
        mma_16816_f16(o[4 * w + 3], e4m3x2_to_f16x2(hi_a01 >> 16), e4m3x2_to_f16x2(hi_b01 >> 16),
                      e4m3x2_to_f16x2(hi_a23 >> 16), e4m3x2_to_f16x2(hi_b23 >> 16), pb0, pb1);
      }
    } else {
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.empty[s]);
    }
    if (sh.flags[0]) break;
  }
  // Row sums over the eight lanes of each column (the key halves).
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    l[e] += __shfl_xor_sync(0xffffffffu, l[e], 4);
    l[e] += __shfl_xor_sync(0xffffffffu, l[e], 8);
    l[e] += __shfl_xor_sync(0xffffffffu, l[e], 16);
  }
  drain_ring<C::STAGES>(sh, warp, lane, consumed);

  // Merge the four warps' states into warp 0 through the ring.
  {
    float* scratch = reinterpret_cast<float*>(ring);
    constexpr int PER_WARP = MT * 4 * 32 + 16;   // O^T fragments + (m, l) of 8 rows
    if (warp > 0) {
      float* w = scratch + warp * PER_WARP;
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int e = 0; e < 4; ++e) w[(mt * 4 + e) * 32 + lane] = o[mt][e];
      if (g == 0) {
        w[MT * 128 + 2 * c] = m[0];
        w[MT * 128 + 2 * c + 1] = m[1];
        w[MT * 128 + 8 + 2 * c] = l[0];
        w[MT * 128 + 8 + 2 * c + 1] = l[1];
      }
    }
    asm volatile("bar.sync 1, 128;" ::: "memory");
    if (warp == 0) {
#pragma unroll
      for (int k2 = 1; k2 < 4; ++k2) {
        const float* w = scratch + k2 * PER_WARP;
        float aa[2], ab[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float mb = w[MT * 128 + 2 * c + e];
          const float lb = w[MT * 128 + 8 + 2 * c + e];
          const float mn = fmaxf(m[e], mb);
          const float mu = mn == -INFINITY ? 0.f : mn;
          aa[e] = fast_exp2(m[e] - mu);
          ab[e] = fast_exp2(mb - mu);
          l[e] = l[e] * aa[e] + lb * ab[e];
          m[e] = mn;
        }
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
          for (int e = 0; e < 4; ++e)
            o[mt][e] = o[mt][e] * aa[e & 1] + w[(mt * 4 + e) * 32 + lane] * ab[e & 1];
      }
    }
  }

  float inv_l[2], lse_nat[2];
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    const bool any = l[e] > 0.f;
    inv_l[e] = any ? vsc / l[e] : 0.f;
    lse_nat[e] = any ? (m[e] + fast_log2(l[e])) * kLn2 : -INFINITY;
  }
  // Column e of the lane holds row 2c + e: dims 8g + mt (o[mt][e]) and
  // 64 + 8g + mt (o[mt][2 + e]), mt = 0..7.
  if (nsplit == 1 && !a.partials_only) {
    if (warp > 0) return;
    if (a.sinks) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        if (!rvalid[e]) continue;
        float mm = m[e], ll = l[e];
        const float f = add_sink(mm, ll, __ldg(a.sinks + head[e]) * kLog2e);
        inv_l[e] = ll > 0.f ? vsc * f / ll : 0.f;
        lse_nat[e] = ll > 0.f ? (mm + fast_log2(ll)) * kLn2 : -INFINITY;
      }
    }
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      if (!rvalid[e]) continue;
      uint16_t* orow = a.out + (static_cast<int64_t>(tok[e]) * a.H + head[e]) * D + 8 * g;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t pk[4];
#pragma unroll
        for (int q = 0; q < 4; ++q)
          pk[q] = Elem<F16>::pack(o[2 * q][2 * half + e] * inv_l[e],
                                  o[2 * q + 1][2 * half + e] * inv_l[e]);
        *reinterpret_cast<uint4*>(orow + 64 * half) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
      }
      if (a.lse && g == 0) a.lse[static_cast<int64_t>(head[e]) * a.lse_stride + tok[e]] = lse_nat[e];
    }
    return;
  }
  const int slot = slot_base + rt * nsplit + j;
  const int64_t slot_row0 = slot_row(a, slot, hk, 0);
  if (warp == 0) {
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      if (!rvalid[e]) continue;
      float* po = a.part_o + (slot_row0 + 2 * c + e) * D + 8 * g;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        __stcg(reinterpret_cast<float4*>(po + 64 * half),
               make_float4(o[0][2 * half + e] * inv_l[e], o[1][2 * half + e] * inv_l[e],
                           o[2][2 * half + e] * inv_l[e], o[3][2 * half + e] * inv_l[e]));
        __stcg(reinterpret_cast<float4*>(po + 64 * half + 4),
               make_float4(o[4][2 * half + e] * inv_l[e], o[5][2 * half + e] * inv_l[e],
                           o[6][2 * half + e] * inv_l[e], o[7][2 * half + e] * inv_l[e]));
      }
      if (g == 0) __stcg(a.part_lse + slot_row0 + 2 * c + e, lse_nat[e]);
    }
  }
  finish_group<D, F16>(a, sh, slot_base, rt, nsplit, hk, R, row0, q_start);
}

template <int D, bool FP8, bool F16>
__global__ void __launch_bounds__(SplitCfg<D, FP8>::THREADS, SplitCfg<D, FP8>::CTAS_PER_SM)
attn_split_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                  const __grid_constant__ AttnArgs a) {
  using C = SplitCfg<D, FP8>;
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
  if constexpr (FP8) {
    if (R <= 8) {
      split_consumer_fp8_dec<F16>(a, ring, sh, hk, rt, j, q_start, q_len, kv_len, kb, ke, ntiles,
                             nsplit, slot_base);
      return;
    }
  }
  if (R <= 16)
    split_consumer<D, 1, FP8, F16>(a, ring, sh, hk, seg, rt, j, q_start, q_len, kv_len, kb, ke,
                              ntiles, nsplit, slot_base);
  else if (R <= 32)
    split_consumer<D, 2, FP8, F16>(a, ring, sh, hk, seg, rt, j, q_start, q_len, kv_len, kb, ke,
                              ntiles, nsplit, slot_base);
  else
    split_consumer<D, 4, FP8, F16>(a, ring, sh, hk, seg, rt, j, q_start, q_len, kv_len, kb, ke,
                              ntiles, nsplit, slot_base);
}

template <int D, bool FP8, bool F16>
static cudaError_t launch_split_d(const CUtensorMap& tmK, const CUtensorMap& tmV,
                                  const AttnArgs& a, int items_bound, cudaStream_t st) {
  using C = SplitCfg<D, FP8>;
  // The shared-memory opt-in is a per-device function attribute: set it on
  // the first launch on each device (before any stream capture), not again.
  // The flags are atomics, so first calls from several host threads are
  // race-free (two threads may both set the attribute, which is harmless).
  static std::atomic<bool> configured[kMaxDevices];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const bool known = dev >= 0 && dev < kMaxDevices;
  if (!known || !configured[dev].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(attn_split_kernel<D, FP8, F16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    if (known) configured[dev].store(true, std::memory_order_release);
  }
  cudaLaunchConfig_t cfg = {};
  // One block per (item, KV head), and one more that has no item (the block
  // that waits for the predecessor grid; see pdl_enter).
  cfg.gridDim = dim3(static_cast<unsigned>(items_bound) * static_cast<unsigned>(a.H_kv) + 1u);
  cfg.blockDim = dim3(C::THREADS);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, attn_split_kernel<D, FP8, F16>, tmK, tmV, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_attn_split(const CUtensorMap& tmK, const CUtensorMap& tmV, const AttnArgs& a,
                              int items_bound, cudaStream_t st) {
  if (items_bound <= 0) return cudaSuccess;
  if (a.D > kMaxHeadSplit) return cudaErrorInvalidValue;   // planned on the prefill kernel only
  if (a.f16) {
    if (a.kv_fp8) return launch_split_d<128, true, true>(tmK, tmV, a, items_bound, st);
    if (a.D == 128) return launch_split_d<128, false, true>(tmK, tmV, a, items_bound, st);
    return launch_split_d<64, false, true>(tmK, tmV, a, items_bound, st);
  }
  if (a.kv_fp8) return launch_split_d<128, true, false>(tmK, tmV, a, items_bound, st);
  if (a.D == 128) return launch_split_d<128, false, false>(tmK, tmV, a, items_bound, st);
  return launch_split_d<64, false, false>(tmK, tmV, a, items_bound, st);
}

}  // namespace pa
