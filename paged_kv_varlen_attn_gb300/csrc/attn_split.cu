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
//    128-byte swizzled line, so a stage holds twice the keys' worth of bytes
//    per barrier round trip. Each warp widens its own slice straight from the
//    staged bytes into f16 MMA fragments (e4m3 -> f16 is exact), with Q in
//    f16. For Q.K^T the head dimension is permuted -- MMA k-index
//    16*kk + {2c, 2c+1, 2c+8, 2c+9} of lane quad c is dim 32*c + 4*kk + {0..3}
//    in both Q and K -- so a lane's K bytes of a key are 32 contiguous bytes.
//    For P.V the output dimension is permuted -- MMA column g of n-tile n is
//    dim 16*g + n -- so a lane reads 16 contiguous bytes of each of its four
//    keys and pairs them with byte permutes. k_scale folds into the softmax
//    scale and v_scale into the final normalisation.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

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
  // FP8 runs 2 CTAs per SM (its consumer needs more than 128 registers)
  // with 6 stages, the same bytes in flight per SM as bf16's 3 x 2 stages.
  static constexpr int STAGES = FP8 ? 6 : (D == 128 ? 2 : 6);
  static constexpr int CTAS_PER_SM = FP8 ? 2 : 3;
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
template <int D, int RGN, bool FP8>
__device__ __forceinline__ void split_consumer(const AttnArgs& a, uint8_t* ring, SplitShared sh,
                                               int hk, int seg, int rt, int j, int q_start,
                                               int q_len, int kv_len, int kb, int ke, int ntiles,
                                               int nsplit, int slot_base) {
  using C = SplitCfg<D, FP8>;
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
        const __nv_bfloat16* p = a.q + static_cast<int64_t>(tok[r]) * a.q_stride +
                                 static_cast<int64_t>(head[r]) * D + col;
        v = __ldg(reinterpret_cast<const uint32_t*>(p));
        if constexpr (FP8) {
          const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v));
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
          mma_16816(sacc[2 * np], qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3], b0, b1);
          mma_16816(sacc[2 * np + 1], qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3], b2, b3);
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
    inv_l[r] = any ? vsc / l[r] : 0.f;
    lse_nat[r] = any ? (m[r] + fast_log2(l[r])) * kLn2 : -INFINITY;
  }
  const int H = a.H;
  if (nsplit == 1 && !a.partials_only) {
    if (ks > 0) return;
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
            pk[n / 2] = pack_bf16(o[n][2 * r + e] * inv_l[r], o[n + 1][2 * r + e] * inv_l[r]);
          uint4* dst = reinterpret_cast<uint4*>(a.out + obase + 16 * (2 * cq + e));
          dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
          dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
        }
      } else {
#pragma unroll
      for (int n = 0; n < DN; ++n) {
        const int col = n * 8 + 2 * cq;
        *reinterpret_cast<uint32_t*>(a.out + obase + col) =
            pack_bf16(o[n][2 * r] * inv_l[r], o[n][2 * r + 1] * inv_l[r]);
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

template <int D, bool FP8>
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
  if (R <= 16)
    split_consumer<D, 1, FP8>(a, ring, sh, hk, seg, rt, j, q_start, q_len, kv_len, kb, ke,
                              ntiles, nsplit, slot_base);
  else if (R <= 32)
    split_consumer<D, 2, FP8>(a, ring, sh, hk, seg, rt, j, q_start, q_len, kv_len, kb, ke,
                              ntiles, nsplit, slot_base);
  else
    split_consumer<D, 4, FP8>(a, ring, sh, hk, seg, rt, j, q_start, q_len, kv_len, kb, ke,
                              ntiles, nsplit, slot_base);
}

template <int D, bool FP8>
static cudaError_t launch_split_d(const CUtensorMap& tmK, const CUtensorMap& tmV,
                                  const AttnArgs& a, int items_bound, cudaStream_t st) {
  using C = SplitCfg<D, FP8>;
  // The shared-memory opt-in is a per-device function attribute: set it on
  // the first launch on each device (before any stream capture), not again.
  static bool configured[kMaxDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices || !configured[dev]) {
    e = cudaFuncSetAttribute(attn_split_kernel<D, FP8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
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
  e = cudaLaunchKernelEx(&cfg, attn_split_kernel<D, FP8>, tmK, tmV, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_attn_split(const CUtensorMap& tmK, const CUtensorMap& tmV, const AttnArgs& a,
                              int items_bound, cudaStream_t st) {
  if (items_bound <= 0) return cudaSuccess;
  if (a.kv_fp8) return launch_split_d<128, true>(tmK, tmV, a, items_bound, st);
  if (a.D == 128) return launch_split_d<128, false>(tmK, tmV, a, items_bound, st);
  return launch_split_d<64, false>(tmK, tmV, a, items_bound, st);
}

}  // namespace pa
