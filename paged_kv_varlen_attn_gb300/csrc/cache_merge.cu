// reshape_and_cache (slot_mapping scatter) and merge_attn_states (LSE-weighted
// combine): the two memory-bound helper kernels of the attention path.
//
// Sources: "FlashAttention 在 vLLM 中的实现分析" §4.2 (do_kv_cache_update ->
// reshape_and_cache_flash writes new K/V into the paged cache by slot_mapping),
// §6.3 step 3 and §8.2 (merge_attn_states combines two (out, lse) states).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "device_common.cuh"

namespace pa {

// ---------------------------------------------------------------------------
// Scatter. One warp per token at a time (warps stride over the tokens): the
// lanes move the token's K row and V row ([H_kv, D], vpt 16-byte vectors
// each) with consecutive lanes on consecutive vectors, so the read of the new
// token and the write into its page row are fully coalesced, and each lane
// keeps up to 2 * kScatterUnroll loads in flight. The source loads do not
// depend on the slot, so they are issued together with the slot load, and
// no per-vector index division is needed.
// ---------------------------------------------------------------------------
constexpr int kScatterThreads = 256;
constexpr int kScatterWarps = kScatterThreads / 32;
constexpr int kScatterUnroll = 4;

__global__ void __launch_bounds__(kScatterThreads)
reshape_and_cache_kernel(const uint4* __restrict__ key, const uint4* __restrict__ value,
                         int64_t kstride_v, int64_t vstride_v, uint4* __restrict__ kc,
                         uint4* __restrict__ vc, int64_t block_stride_v,
                         const int64_t* __restrict__ slots, int num_tokens, int vpt, int bs,
                         int64_t num_slots, int32_t* status) {
  // Launched after the planner inside an update-and-attend call (a no-op
  // otherwise): its inputs predate the planner, so only the last block waits
  // for it, after its own rows, which keeps the grids completing in launch
  // order without delaying any row.
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kScatterWarps;
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * kScatterWarps + (threadIdx.x >> 5);
       t < num_tokens; t += nwarps) {
    const uint4* ksrc = key + t * kstride_v;
    const uint4* vsrc = value + t * vstride_v;
    const int64_t slot = __ldg(slots + t);
    for (int v0 = lane; v0 < vpt; v0 += 32 * kScatterUnroll) {
      uint4 kv[kScatterUnroll], vv[kScatterUnroll];
#pragma unroll
      for (int u = 0; u < kScatterUnroll; ++u) {
        const int i = v0 + u * 32;
        if (i < vpt) {
          kv[u] = __ldcs(ksrc + i);
          vv[u] = __ldcs(vsrc + i);
        }
      }
      if (slot < 0) continue;                  // padding token
      if (slot >= num_slots) {
        if (lane == 0 && v0 == lane) flag_status(status, PA_DEV_BAD_SLOT);
        continue;
      }
      const int64_t page = slot / bs;
      const int64_t row = slot - page * bs;
      uint4* kdst = kc + page * block_stride_v + row * vpt;
      uint4* vdst = vc + page * block_stride_v + row * vpt;
#pragma unroll
      for (int u = 0; u < kScatterUnroll; ++u) {
        const int i = v0 + u * 32;
        if (i < vpt) {
          kdst[i] = kv[u];
          vdst[i] = vv[u];
        }
      }
    }
  }
  pdl_leave();
}

cudaError_t launch_reshape_and_cache(const void* key, const void* value, int64_t kstride,
                                     int64_t vstride, void* kc, void* vc, int64_t block_stride,
                                     const int64_t* slots, int num_tokens, int H_kv, int D, int bs,
                                     int num_blocks, int32_t* status, cudaStream_t st, int sms,
                                     bool pdl) {
  if (num_tokens == 0) return cudaSuccess;
  const int vpt = H_kv * D / 8;
  const int64_t want = (static_cast<int64_t>(num_tokens) + kScatterWarps - 1) / kScatterWarps;
  const int64_t cap = static_cast<int64_t>(sms) * 8;  // 8 CTAs of 256 threads per SM
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(want < cap ? want : cap));
  cfg.blockDim = dim3(kScatterThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  cudaError_t e = cudaLaunchKernelEx(
      &cfg, reshape_and_cache_kernel, static_cast<const uint4*>(key),
      static_cast<const uint4*>(value), kstride / 8, vstride / 8, static_cast<uint4*>(kc),
      static_cast<uint4*>(vc), block_stride / 8, slots, num_tokens, vpt, bs,
      static_cast<int64_t>(num_blocks) * bs, status);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Scatter into an FP8 (e4m3) cache ("FlashAttention と FlashInfer" 役割 and
// 境界と失敗: FP8 KV cache with per-head quant scales). Same warp-per-token
// walk as above; a lane reads 8 bf16 or f16 values (16 bytes) of one head, divides
// them by that KV head's scale (the IEEE float32 quotient, correctly rounded)
// and writes the 8 e4m3 bytes (round to nearest even, saturating at +-448).
// ---------------------------------------------------------------------------
// x / s correctly rounded to float32 wherever the quotient decides an e4m3
// code, from y = RN(1/s): q0 = RN(x y), the remainder r = x - q0 s (exact,
// one FMA) and q = RN(q0 + r y). By Markstein's theorem (y within half an
// ulp of 1/s and q0 within one ulp of x/s make RN(q0 + r y) the correctly
// rounded quotient, as long as r neither underflows nor the quotient
// overflows), q is RN(x/s). Zero, |q0| >= 512, infinite and NaN products
// take q0 (a zero product keeps its sign, which q0 + r y would lose for
// -0; where r = 0 otherwise, q0 + r y is q0 anyway; every quotient of at
// least 464 saturates to the same code). With 2^-32 <= |s| <= 2^32 the
// reciprocal is normal and every quotient of at least 2^-11 (below that the
// code is a signed zero either way) has a normal, hence exact, remainder;
// other scales take the IEEE division. The product and the two FMAs run on
// two values at a time (f32x2): three instructions per pair of values
// besides the selects, instead of two divisions.
struct ScaleDiv {
  float s, ns, y;   // the scale, its negation and RN(1 / s)
  bool fast;        // |s| in [2^-32, 2^32]
};

__device__ __forceinline__ ScaleDiv scale_div(float s) {
  const float as = fabsf(s);
  return {s, -s, __frcp_rn(s), as >= 0x1p-32f && as <= 0x1p32f};
}

__device__ __forceinline__ float pick_quotient(float q0, float q) {
  return (q0 != 0.f && fabsf(q0) < 512.f) ? q : q0;
}

template <bool F16>
__device__ __forceinline__ uint2 quantize8(uint4 x, const ScaleDiv& d) {
  const uint32_t h[4] = {x.x, x.y, x.z, x.w};
  float v[8];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 a = Elem<F16>::unpack(h[k]);
    v[2 * k] = a.x;
    v[2 * k + 1] = a.y;
  }
  if (d.fast) {
#pragma unroll
    for (int k = 0; k < 8; k += 2) {
      float q0a, q0b, ra, rb, qa, qb;
      ffma2(q0a, q0b, v[k], v[k + 1], d.y, d.y, -0.f, -0.f);     // RN(x y)
      ffma2(ra, rb, q0a, q0b, d.ns, d.ns, v[k], v[k + 1]);       // x - q0 s
      ffma2(qa, qb, ra, rb, d.y, d.y, q0a, q0b);                 // q0 + r y
      v[k] = pick_quotient(q0a, qa);
      v[k + 1] = pick_quotient(q0b, qb);
    }
  } else {
#pragma unroll
    for (int k = 0; k < 8; ++k) v[k] = __fdiv_rn(v[k], d.s);
  }
  const uint32_t w0 = f32x2_to_e4m3x2(v[0], v[1]) | (f32x2_to_e4m3x2(v[2], v[3]) << 16);
  const uint32_t w1 = f32x2_to_e4m3x2(v[4], v[5]) | (f32x2_to_e4m3x2(v[6], v[7]) << 16);
  return make_uint2(w0, w1);
}

// Same walk as the 2-byte scatter. The head of vector i is i / (D / 8), a
// shift (D is a power of two); a lane's heads, their scales and reciprocals
// are set up once per 32 * kScatterUnroll-vector chunk of the row and kept
// across tokens (a row of at most that many vectors, H_kv * D <= 1024, needs
// them only once). At most 80 registers, so that three 256-thread CTAs fit
// an SM. Measured on the 16,440 new tokens of the chunked-prefill batch:
// 24.5 us, against 26.7 us for an IEEE division per value, 30.3 us with the
// same code at 86 registers (two CTAs per SM), 24.6 us through shared memory
// with bulk copies (two units in flight per warp) and 29.1 us with two
// tokens per warp step. Between 8,220 and 16,440 tokens the time grows at
// 6.1-6.7 TB/s: past a fixed ~8 us of launch and ramp-up it streams at the
// HBM rate.
template <bool F16>
__global__ void __launch_bounds__(kScatterThreads, 3)
reshape_and_cache_fp8_kernel(const uint4* __restrict__ key, const uint4* __restrict__ value,
                             int64_t kstride_v, int64_t vstride_v, uint2* __restrict__ kc,
                             uint2* __restrict__ vc, int64_t block_stride_v,
                             const int64_t* __restrict__ slots, int num_tokens, int vpt,
                             int vph, int bs, int64_t num_slots,
                             const float* __restrict__ k_scale,
                             const float* __restrict__ v_scale, int32_t* status) {
  pdl_trigger();   // the planner: as in reshape_and_cache_kernel
  const int lane = threadIdx.x & 31;
  const int vsh = __ffs(vph) - 1;   // log2(D / 8)
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kScatterWarps;
  ScaleDiv kd[kScatterUnroll], vd[kScatterUnroll];
  int chunk = -1;   // v0 the scales above belong to
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * kScatterWarps + (threadIdx.x >> 5);
       t < num_tokens; t += nwarps) {
    const uint4* ksrc = key + t * kstride_v;
    const uint4* vsrc = value + t * vstride_v;
    const int64_t slot = __ldg(slots + t);
    for (int v0 = lane; v0 < vpt; v0 += 32 * kScatterUnroll) {
      uint4 kv[kScatterUnroll], vv[kScatterUnroll];
#pragma unroll
      for (int u = 0; u < kScatterUnroll; ++u) {
        const int i = v0 + u * 32;
        if (i < vpt) {
          kv[u] = __ldcs(ksrc + i);
          vv[u] = __ldcs(vsrc + i);
        }
      }
      if (slot < 0) continue;                  // padding token
      if (slot >= num_slots) {
        if (lane == 0 && v0 == lane) flag_status(status, PA_DEV_BAD_SLOT);
        continue;
      }
      if (v0 != chunk) {
        chunk = v0;
#pragma unroll
        for (int u = 0; u < kScatterUnroll; ++u) {
          const int i = v0 + u * 32;
          if (i < vpt) {
            kd[u] = scale_div(__ldg(k_scale + (i >> vsh)));
            vd[u] = scale_div(__ldg(v_scale + (i >> vsh)));
          }
        }
      }
      const int64_t page = slot / bs;
      const int64_t row = slot - page * bs;
      uint2* kdst = kc + page * block_stride_v + row * vpt;
      uint2* vdst = vc + page * block_stride_v + row * vpt;
#pragma unroll
      for (int u = 0; u < kScatterUnroll; ++u) {
        const int i = v0 + u * 32;
        if (i < vpt) {
          kdst[i] = quantize8<F16>(kv[u], kd[u]);
          vdst[i] = quantize8<F16>(vv[u], vd[u]);
        }
      }
    }
  }
  pdl_leave();
}

cudaError_t launch_reshape_and_cache_fp8(const void* key, const void* value, int64_t kstride,
                                         int64_t vstride, void* kc, void* vc,
                                         int64_t block_stride, const int64_t* slots,
                                         int num_tokens, int H_kv, int D, int bs, int num_blocks,
                                         const float* k_scale, const float* v_scale,
                                         int32_t* status, cudaStream_t st, int sms, bool pdl,
                                         int f16) {
  if (num_tokens == 0) return cudaSuccess;
  const int vpt = H_kv * D / 8;
  const int64_t want = (static_cast<int64_t>(num_tokens) + kScatterWarps - 1) / kScatterWarps;
  // One wave: the kernel keeps three CTAs per SM (its launch bounds), and
  // warps stride over the tokens. Measured with L2 flushed: 4,110 tokens
  // 12.3-12.5 us against 14.2 with eight CTAs per SM (2.7 waves); 16,440
  // tokens 24.2-24.5 against 24.6-25.9.
  const int64_t cap = static_cast<int64_t>(sms) * 3;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(want < cap ? want : cap));
  cfg.blockDim = dim3(kScatterThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  cudaError_t e = cudaLaunchKernelEx(
      &cfg, f16 ? reshape_and_cache_fp8_kernel<true> : reshape_and_cache_fp8_kernel<false>,
      static_cast<const uint4*>(key),
      static_cast<const uint4*>(value), kstride / 8, vstride / 8, static_cast<uint2*>(kc),
      static_cast<uint2*>(vc), block_stride / 8, slots, num_tokens, vpt, D / 8, bs,
      static_cast<int64_t>(num_blocks) * bs, k_scale, v_scale, status);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// merge_attn_states. One thread per 8 output elements (one 16-byte vector) of
// a (token, head) row; the two LSEs of the row are read per thread (they hit
// L1). With m = max(a, b): out = (e^(a-m) oa + e^(b-m) ob) / (e^(a-m) + e^(b-m)),
// lse = m + ln(e^(a-m) + e^(b-m)); both -inf gives out 0, lse -inf.
// ---------------------------------------------------------------------------
constexpr int kMergeThreads = 256;

// 8 bf16 or f16 values of a 16-byte vector as floats.
template <bool F16>
__device__ __forceinline__ void x8_to_float(const uint4& v, float (&f)[8]) {
  const uint32_t h[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 x = Elem<F16>::unpack(h[i]);
    f[2 * i] = x.x;
    f[2 * i + 1] = x.y;
  }
}

template <bool F16>
__global__ void __launch_bounds__(kMergeThreads)
merge_attn_states_kernel(uint4* out, float* out_lse, const uint4* __restrict__ a,
                         const float* __restrict__ alse, const uint4* __restrict__ b,
                         const float* __restrict__ blse, int T, int H, int vpr) {
  const int64_t total = static_cast<int64_t>(T) * H * vpr;
  const int64_t step = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
       idx += step) {
    const int64_t row = idx / vpr;            // row = t * H + h
    const int vi = static_cast<int>(idx - row * vpr);
    const int t = static_cast<int>(row / H);
    const int h = static_cast<int>(row - static_cast<int64_t>(t) * H);
    const float la = __ldg(alse + static_cast<int64_t>(h) * T + t);
    const float lb = __ldg(blse + static_cast<int64_t>(h) * T + t);
    const float m = fmaxf(la, lb);
    uint4 res;
    float lse_out;
    if (m == -INFINITY) {
      res = make_uint4(0, 0, 0, 0);
      lse_out = -INFINITY;
    } else {
      const float wa = fast_exp2((la - m) * kLog2e);
      const float wb = fast_exp2((lb - m) * kLog2e);
      const float inv = 1.0f / (wa + wb);
      const float ca = wa * inv, cb = wb * inv;
      float fa[8], fb[8];
      x8_to_float<F16>(__ldcs(a + idx), fa);
      x8_to_float<F16>(__ldcs(b + idx), fb);
      uint32_t* r = reinterpret_cast<uint32_t*>(&res);
#pragma unroll
      for (int i = 0; i < 4; ++i)
        r[i] = Elem<F16>::pack(ca * fa[2 * i] + cb * fb[2 * i],
                               ca * fa[2 * i + 1] + cb * fb[2 * i + 1]);
      lse_out = m + fast_log2(wa + wb) * kLn2;
    }
    out[idx] = res;
    if (out_lse && vi == 0) out_lse[static_cast<int64_t>(h) * T + t] = lse_out;
  }
}

cudaError_t launch_merge(void* out, float* out_lse, const void* a, const float* alse,
                         const void* b, const float* blse, int T, int H, int D, cudaStream_t st,
                         int sms, int f16) {
  if (T == 0) return cudaSuccess;
  const int vpr = D / 8;
  const int64_t total = static_cast<int64_t>(T) * H * vpr;
  const int64_t want = (total + kMergeThreads - 1) / kMergeThreads;
  const int64_t cap = static_cast<int64_t>(sms) * 8;
  const int grid = static_cast<int>(want < cap ? want : cap);
  (f16 ? merge_attn_states_kernel<true> : merge_attn_states_kernel<false>)<<<grid, kMergeThreads, 0, st>>>(
      static_cast<uint4*>(out), out_lse, static_cast<const uint4*>(a), alse,
      static_cast<const uint4*>(b), blse, T, H, vpr);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// n-state merge: the LSE merge of the partial results of n ranks of decode
// context parallelism ("FlashAttention 在 vLLM 中的实现分析" §9) or of any n
// disjoint key sets. One thread per 16-byte vector of a (token, head) row:
// the row's n LSEs (L1 hits after the first thread) give the maximum m, then
// the n vectors are read in batches of kBatchN loads in flight and summed
// with weights e^(lse_r - m); out = sum / sum of weights, lse = m + ln(sum
// of weights), a row whose LSEs are all -inf gets out 0, lse -inf.
// ---------------------------------------------------------------------------
constexpr int kBatchN = 4;

template <bool F16>
__global__ void __launch_bounds__(kMergeThreads)
merge_attn_states_n_kernel(uint4* out, float* out_lse, const uint4* __restrict__ parts,
                           int64_t pstride_v, const float* __restrict__ plse, int64_t lstride,
                           int n, int T, int H, int vpr) {
  const int64_t total = static_cast<int64_t>(T) * H * vpr;
  const int64_t step = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
       idx += step) {
    const int64_t row = idx / vpr;            // row = t * H + h
    const int vi = static_cast<int>(idx - row * vpr);
    const int t = static_cast<int>(row / H);
    const int h = static_cast<int>(row - static_cast<int64_t>(t) * H);
    const float* lp = plse + static_cast<int64_t>(h) * T + t;
    float m = -INFINITY;
    for (int r = 0; r < n; ++r) m = fmaxf(m, __ldg(lp + r * lstride));
    uint4 res = make_uint4(0, 0, 0, 0);
    float lse_out = -INFINITY;
    if (m != -INFINITY) {
      float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      float sw = 0.f;
      for (int r0 = 0; r0 < n; r0 += kBatchN) {
        uint4 v[kBatchN];
        float w[kBatchN];
#pragma unroll
        for (int u = 0; u < kBatchN; ++u) {
          if (r0 + u < n) {
            w[u] = fast_exp2((__ldg(lp + (r0 + u) * lstride) - m) * kLog2e);
            v[u] = __ldcs(parts + (r0 + u) * pstride_v + idx);
          }
        }
#pragma unroll
        for (int u = 0; u < kBatchN; ++u) {
          if (r0 + u >= n) continue;
          float f[8];
          x8_to_float<F16>(v[u], f);
          sw += w[u];
#pragma unroll
          for (int i = 0; i < 8; ++i) acc[i] += w[u] * f[i];
        }
      }
      const float inv = 1.0f / sw;
      uint32_t* rr = reinterpret_cast<uint32_t*>(&res);
#pragma unroll
      for (int i = 0; i < 4; ++i) rr[i] = Elem<F16>::pack(acc[2 * i] * inv, acc[2 * i + 1] * inv);
      lse_out = m + fast_log2(sw) * kLn2;
    }
    out[idx] = res;
    if (out_lse && vi == 0) out_lse[static_cast<int64_t>(h) * T + t] = lse_out;
  }
}

cudaError_t launch_merge_n(void* out, float* out_lse, const void* parts, int64_t part_stride,
                           const float* parts_lse, int64_t lse_stride, int n, int T, int H, int D,
                           cudaStream_t st, int sms, int f16) {
  if (T == 0) return cudaSuccess;
  const int vpr = D / 8;
  const int64_t total = static_cast<int64_t>(T) * H * vpr;
  const int64_t want = (total + kMergeThreads - 1) / kMergeThreads;
  // One wave: four CTAs per SM fit (64 registers a thread), and threads
  // stride over the vectors. Measured on 4 parts x 16,384 tokens x 32 heads:
  // 122.7 us against 125.0 with eight per SM (two waves), 145 with six.
  // (Requesting the first batch of vectors before the LSEs took 80
  // registers; held to 64 for four CTAs per SM it measured 137 us.)
  const int64_t cap = static_cast<int64_t>(sms) * 4;
  const int grid = static_cast<int>(want < cap ? want : cap);
  (f16 ? merge_attn_states_n_kernel<true> : merge_attn_states_n_kernel<false>)<<<grid, kMergeThreads, 0, st>>>(
      static_cast<uint4*>(out), out_lse, static_cast<const uint4*>(parts), part_stride / 8,
      parts_lse, lse_stride, n, T, H, vpr);
  return cudaGetLastError();
}

}  // namespace pa
