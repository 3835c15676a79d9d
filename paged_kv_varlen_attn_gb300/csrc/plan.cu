// Device-side work planner for one attention call.
//
// The idea follows the ahead-of-time scheduling of "FlashAttention 在 vLLM 中的
// 实现分析" §7 (a plan computed before the kernels run makes execution
// deterministic and CUDA-graph capturable) and the num_splits split-KV of §1.3,
// but it runs ON THE DEVICE from cu_seqlens_q / seqused_k, so the host never
// reads a device value and the call needs no synchronisation.
//
// For each segment (a sequence, or the whole batch in the cascade prefix pass)
// the planner picks a class -- 0: the split-KV kernel (at most kTcMinRows = 32
// packed query rows, i.e. decode and short queries; items of up to 64 rows when
// the prefill kernel is not used), 1: the tensor-core prefill kernel -- cuts the
// packed rows into row tiles, and splits the keys into equal chunks so that
// each class has about `target` work items per KV head. Chunk length
//   L = max(min chunk of the class, ceil(W / target)) rounded up to kKeyTile,
// where W = sum over segments of (row tiles x keys). Then
//   sum of items <= target + sum of row tiles, and
//   slots (items of segments split more than once) <= 2 * target,
// which is what the host reserves in the workspace (one slot pool per class;
// a slot holds as many rows as one work item of its class can have).
#include <cuda_runtime.h>

#include "device_common.cuh"

namespace pa {


// Block-wide exclusive scan of four counters; returns the block totals.
__device__ __forceinline__ int4 block_scan4(int4 v, int4& excl, int* sh /* [4 * 32] */) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int4 x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int a = __shfl_up_sync(0xffffffffu, x.x, o);
    const int b = __shfl_up_sync(0xffffffffu, x.y, o);
    const int c = __shfl_up_sync(0xffffffffu, x.z, o);
    const int d = __shfl_up_sync(0xffffffffu, x.w, o);
    if (lane >= o) { x.x += a; x.y += b; x.z += c; x.w += d; }
  }
  if (lane == 31) { sh[warp] = x.x; sh[32 + warp] = x.y; sh[64 + warp] = x.z; sh[96 + warp] = x.w; }
  __syncthreads();
  const int nw = static_cast<int>(blockDim.x) >> 5;
  if (warp == 0) {
    int a = 0, b = 0, c = 0, d = 0;
    if (lane < nw) { a = sh[lane]; b = sh[32 + lane]; c = sh[64 + lane]; d = sh[96 + lane]; }
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int a2 = __shfl_up_sync(0xffffffffu, a, o);
      const int b2 = __shfl_up_sync(0xffffffffu, b, o);
      const int c2 = __shfl_up_sync(0xffffffffu, c, o);
      const int d2 = __shfl_up_sync(0xffffffffu, d, o);
      if (lane >= o) { a += a2; b += b2; c += c2; d += d2; }
    }
    sh[lane] = a; sh[32 + lane] = b; sh[64 + lane] = c; sh[96 + lane] = d;
  }
  __syncthreads();
  int4 before = make_int4(0, 0, 0, 0);
  if (warp > 0) before = make_int4(sh[warp - 1], sh[32 + warp - 1], sh[64 + warp - 1], sh[96 + warp - 1]);
  excl = make_int4(before.x + x.x - v.x, before.y + x.y - v.y, before.z + x.z - v.z,
                   before.w + x.w - v.w);
  const int4 tot = make_int4(sh[nw - 1], sh[31 + nw], sh[63 + nw], sh[95 + nw]);
  __syncthreads();
  return tot;
}

// 256 threads: the planner's phases are barrier- and scan-bound at the
// batch sizes of a serving step (6.6 us per call with 1024 threads on the
// 64-sequence decode batch).
constexpr int kPlanThreads = 256;
constexpr int kSizeBuckets = 1024;
constexpr int kPlanSmemSegs = 1024;   // segment tables kept in shared memory up to this many

// Size bucket of work item (segment s, row tile rt, split j): the number of
// 64-key tiles the attention kernel will process for it (capped).
__device__ __forceinline__ int item_bucket(int s, int rt, int j, int4 g, int chunk, int G, int D,
                                           int causal) {
  const int cls = g.w, q_len = g.y, kv = g.z;
  const int R = cls ? tc_item_rows(G, D) : kRowsSplit;
  const int rows = q_len * G;
  const int last_row = min(rows, (rt + 1) * R) - 1;
  const int kb = j * chunk;
  int ke = min(kv, kb + chunk);
  if (causal) ke = min(ke, kv - q_len + last_row / G + 1);
  const int tiles = ke > kb ? (ke - kb + kKeyTile - 1) / kKeyTile : 0;
  return min(tiles, kSizeBuckets - 1);
}

// Segment owning combined item index idx: the last segment whose first item
// (segsplit.w, items of both classes numbered in segment order) is <= idx.
__device__ __forceinline__ int find_segment(const int4* spl, int nseg, int idx) {
  int lo = 0, hi = nseg - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (spl[mid].w <= idx) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(const __grid_constant__ PlanPasses pp) {
  // The first attention kernel may be scheduled now; its blocks wait for
  // this grid to complete before they read the plan.
  pdl_trigger();
  const PlanArgs& P = pp.p[blockIdx.x];
  __shared__ int sh[128];
  __shared__ unsigned long long shW[2];
  // Items per (class, size in key tiles); turned in place into the placement
  // cursors of the size buckets.
  __shared__ int hist[2][kSizeBuckets];
  // Segment tables of this pass when they fit (else the global copies).
  __shared__ int4 tab_geo[kPlanSmemSegs];
  __shared__ int4 tab_spl[kPlanSmemSegs];
  __shared__ int ngroups[2];
  uint8_t* ws = P.ws;
  int* header = reinterpret_cast<int*>(ws + P.L.header);
  int4* seg = reinterpret_cast<int4*>(ws + P.L.seg);
  int4* segsplit = reinterpret_cast<int4*>(ws + P.L.segsplit);
  int4* items0 = reinterpret_cast<int4*>(ws + P.L.items[0]);
  int4* items1 = reinterpret_cast<int4*>(ws + P.L.items[1]);
  int* counters0 = reinterpret_cast<int*>(ws + P.L.counters[0]);
  int* counters1 = reinterpret_cast<int*>(ws + P.L.counters[1]);
  int4* groups0 = reinterpret_cast<int4*>(ws + P.L.groups[0]);
  int4* groups1 = reinterpret_cast<int4*>(ws + P.L.groups[1]);
  const int nseg = P.single_segment ? 1 : P.num_segs;
  const bool in_smem = nseg <= kPlanSmemSegs;
  int4* geo_tab = in_smem ? tab_geo : seg;
  int4* spl_tab = in_smem ? tab_spl : segsplit;
  const int G = P.G;
  const int tid = threadIdx.x;

  // Inputs of this thread's first segment are fetched before the first
  // barrier, so their latency overlaps the clearing of the histograms.
  int q0 = 0, q1 = 0, used = 0;
  if (!P.single_segment && tid < nseg) {
    q0 = P.cu_seqlens_q[tid];
    q1 = P.cu_seqlens_q[tid + 1];
    used = P.seqused_k[tid];
  }
  if (tid < 2) {
    shW[tid] = 0ull;
    ngroups[tid] = 0;
  }
  for (int i = tid; i < 2 * kSizeBuckets; i += blockDim.x) (&hist[0][0])[i] = 0;
  __syncthreads();

  // Pass 1: segment geometry, validation, class, and total work per class.
  unsigned long long w0 = 0, w1 = 0;
  for (int s = tid; s < nseg; s += blockDim.x) {
    int q_start, q_len, kv;
    int bad = 0;
    if (P.single_segment) {
      q_start = 0;
      q_len = P.total_q;
      kv = P.single_kv_len;
    } else {
      if (s != tid) {
        q0 = P.cu_seqlens_q[s];
        q1 = P.cu_seqlens_q[s + 1];
        used = P.seqused_k[s];
      }
      q_start = q0;
      q_len = q1 - q0;
      if (q0 < 0 || q1 > P.total_q || q_len < 0 || q_len > P.max_q) {
        bad |= PA_DEV_BAD_SEQLEN;
        q_len = 0;
        q_start = 0;
      }
      if (used < 0 || used > P.max_k) bad |= PA_DEV_BAD_SEQLEN;
      kv = used - P.kv_len_offset;
    }
    if (kv < 0) {
      bad |= P.check_cascade ? PA_DEV_CASCADE : PA_DEV_BAD_SEQLEN;
      kv = 0;
    }
    if (kv > P.kv_len_cap) {
      bad |= PA_DEV_BAD_SEQLEN;
      kv = P.kv_len_cap;
    }
    if (P.check_cascade && q_len > kv) bad |= PA_DEV_CASCADE;
    if (bad) flag_status(P.status, bad);
    const int rows = q_len * G;
    const int cls = (P.tc_enabled && rows > P.tc_min_rows) ? 1 : 0;
    const int rpi = cls ? tc_item_rows(G, P.D) : kRowsSplit;
    const int nrt = (rows + rpi - 1) / rpi;
    const unsigned long long w = static_cast<unsigned long long>(nrt) * static_cast<unsigned>(kv);
    if (cls) w1 += w; else w0 += w;
    const int4 g = make_int4(q_start, q_len, kv, cls);
    seg[s] = g;
    if (in_smem) tab_geo[s] = g;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    w0 += __shfl_xor_sync(0xffffffffu, w0, o);
    w1 += __shfl_xor_sync(0xffffffffu, w1, o);
  }
  if ((tid & 31) == 0 && (w0 | w1)) {
    atomicAdd(&shW[0], w0);
    atomicAdd(&shW[1], w1);
  }
  __syncthreads();
  const int target[2] = {P.target0, P.target1};
  int chunk_max[2];
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    const unsigned long long W = shW[c];
    const unsigned tg = target[c] > 0 ? static_cast<unsigned>(target[c]) : 1u;
    // ceil(W / target): a 32-bit division unless W needs more bits (a 64-bit
    // division is a long software sequence).
    unsigned long long L;
    if (W == 0) L = 0;
    else if (W < 0xffffffffull - tg) L = (static_cast<unsigned>(W) + tg - 1) / tg;
    else L = (W + tg - 1) / tg;
    const int min_chunk = c ? P.min_chunk_tc : kMinChunkSplit;
    if (L < static_cast<unsigned long long>(min_chunk)) L = min_chunk;
    L = (L + kKeyTile - 1) / kKeyTile * kKeyTile;
    if (L > 0x40000000ull) L = 0x40000000ull;
    chunk_max[c] = static_cast<int>(L);
  }

  // Pass 2: splits, then item and slot offsets by block scans (in chunks of
  // the block size, carried across chunks). segsplit = (nsplit, first slot,
  // chunk, first item in the numbering of both classes in segment order).
  int4 carry = make_int4(0, 0, 0, 0);
  for (int base = 0; base < nseg; base += blockDim.x) {
    const int s = base + tid;
    int nsplit = 1, chunk = 0, cls = 0;
    int4 v = make_int4(0, 0, 0, 0);
    if (s < nseg) {
      const int4 g = geo_tab[s];
      cls = g.w;
      const int R = cls ? tc_item_rows(G, P.D) : kRowsSplit;
      const int nrt = (g.y * G + R - 1) / R;
      const int kv = g.z;
      const int L = cls ? chunk_max[1] : chunk_max[0];
      if (kv > 0) {
        nsplit = (kv + L - 1) / L;
        chunk = (kv + nsplit - 1) / nsplit;
        chunk = (chunk + kKeyTile - 1) / kKeyTile * kKeyTile;
        nsplit = (kv + chunk - 1) / chunk;
      } else {
        nsplit = 1;
        chunk = kKeyTile;
      }
      const int n_items = nrt * nsplit;
      const int n_slots = (nsplit > 1 || P.partials_only) ? n_items : 0;
      v = cls ? make_int4(0, n_items, 0, n_slots) : make_int4(n_items, 0, n_slots, 0);
    }
    int4 ex;
    const int4 tot = block_scan4(v, ex, sh);
    if (s < nseg) {
      const int slot_base = cls ? carry.w + ex.w : carry.z + ex.z;
      const int first = carry.x + carry.y + ex.x + ex.y;
      const int4 sp = make_int4(nsplit, slot_base, chunk, first);
      segsplit[s] = sp;
      if (in_smem) tab_spl[s] = sp;
    }
    carry.x += tot.x;
    carry.y += tot.y;
    carry.z += tot.z;
    carry.w += tot.w;
  }
  __syncthreads();
  const int n_all = carry.x + carry.y;

  // Pass 3, one thread per work item: size histogram (for the longest-first
  // order), the cleared combine counter of each split group, and (cascade
  // suffix) the list of row groups, one per (segment, row tile).
  for (int idx = tid; idx < n_all; idx += blockDim.x) {
    const int s = find_segment(spl_tab, nseg, idx);
    const int4 sp = spl_tab[s];
    const int4 g = geo_tab[s];
    const int local = idx - sp.w;
    const int rt = local / sp.x, j = local - rt * sp.x;
    atomicAdd(&hist[g.w][item_bucket(s, rt, j, g, sp.z, G, P.D, P.causal)], 1);
    if (j == 0 && (sp.x > 1 || P.partials_only)) {
      const int grp = sp.y + rt * sp.x;
      const int sbound = g.w ? P.slots_bound1 : P.slots_bound0;
      if (grp + sp.x <= sbound)
        for (int hk = 0; hk < P.H_kv; ++hk) (g.w ? counters1 : counters0)[grp * P.H_kv + hk] = 0;
    }
    if (j == 0 && P.make_groups) {
      const int gpos = atomicAdd(&ngroups[g.w], 1);
      if (gpos < (g.w ? P.items_bound1 : P.items_bound0))
        (g.w ? groups1 : groups0)[gpos] = make_int4(s, rt, 0, 0);
    }
  }
  __syncthreads();
  // Longest items first: offsets of the size buckets in descending order
  // (one block scan over the buckets). The hardware dispatches blocks in
  // order, so the last wave holds the shortest items. The order inside a
  // bucket does not affect results.
  {
    constexpr int BPT = kSizeBuckets / kPlanThreads;   // buckets per thread, consecutive
    static_assert(BPT * kPlanThreads == kSizeBuckets, "whole buckets per planner thread");
    int c0[BPT], c1[BPT], s0 = 0, s1 = 0;
#pragma unroll
    for (int k = 0; k < BPT; ++k) {
      const int b = kSizeBuckets - 1 - (tid * BPT + k);
      c0[k] = hist[0][b];
      c1[k] = hist[1][b];
      s0 += c0[k];
      s1 += c1[k];
    }
    int4 ex;
    block_scan4(make_int4(s0, s1, 0, 0), ex, sh);
    int o0 = ex.x, o1 = ex.y;
#pragma unroll
    for (int k = 0; k < BPT; ++k) {
      const int b = kSizeBuckets - 1 - (tid * BPT + k);
      hist[0][b] = o0;
      hist[1][b] = o1;
      o0 += c0[k];
      o1 += c1[k];
    }
  }
  __syncthreads();
  // Pass 4, one thread per work item: place it at its bucket's cursor.
  for (int idx = tid; idx < n_all; idx += blockDim.x) {
    const int s = find_segment(spl_tab, nseg, idx);
    const int4 sp = spl_tab[s];
    const int4 g = geo_tab[s];
    const int local = idx - sp.w;
    const int rt = local / sp.x, j = local - rt * sp.x;
    const int cls = g.w;
    const int pos = atomicAdd(&hist[cls][item_bucket(s, rt, j, g, sp.z, G, P.D, P.causal)], 1);
    if (pos < (cls ? P.items_bound1 : P.items_bound0))
      (cls ? items1 : items0)[pos] = make_int4(s, rt, j, 0);
  }
  if (tid == 0) {
    int n0 = carry.x, n1 = carry.y;
    // Cannot happen for inputs within the stated bounds; refuse the work
    // rather than run past the reserved workspace.
    if (n0 > P.items_bound0 || carry.z > P.slots_bound0) {
      flag_status(P.status, PA_DEV_BAD_SEQLEN);
      n0 = 0;
    }
    if (n1 > P.items_bound1 || carry.w > P.slots_bound1) {
      flag_status(P.status, PA_DEV_BAD_SEQLEN);
      n1 = 0;
    }
    header[0] = n0;
    header[1] = n1;
    header[2] = 0;   // abort word of this call
    header[4] = n0 ? ngroups[0] : 0;
    header[5] = n1 ? ngroups[1] : 0;
  }
}

cudaError_t launch_plan(const PlanPasses& pp, int npasses, cudaStream_t st) {
  plan_kernel<<<npasses, kPlanThreads, 0, st>>>(pp);
  return cudaGetLastError();
}

}  // namespace pa
