// Internal structures shared by the host entry points and the kernels.
// Not part of the public ABI (include/pa.h is).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pa.h"

namespace pa {

// Query rows handled by one work item of each attention kernel. A "row" is
// one (query token, query head) pair of a KV-head group: packed row r of a
// segment is token r / G, head-in-group r % G (GQA heads share the K/V tile).
constexpr int kRowsSplit = 64;     // split-KV kernel (decode and short queries)
// Segments with more packed query rows than this run on the prefill kernel
// (measured on 64-row segments: 3.8 TB/s there against 3.3 TB/s through the
// split kernel's four 16-row groups; 32-row segments stay on the split kernel
// at 5.2 TB/s).
constexpr int kTcMinRows = 32;
constexpr int kTcTileRows = 128;   // TMEM lanes of one prefill Q tile (the MMA M dimension)
// A prefill Q tile holds whole tokens: the largest multiple of G packed rows
// that fits the 128 TMEM lanes (128 rows when G divides 128; 126 for G = 3,
// 7 or 42). A work item is two such tiles, or one at head size 256 (its O
// alone takes 256 of the 512 TMEM columns). Segments of groups wider than
// 128 heads run on the split-KV kernel (tc_tile_rows = 0).
__host__ __device__ constexpr int tc_tile_rows(int G) {
  return G >= 1 && G <= kTcTileRows ? (kTcTileRows / G) * G : 0;
}
__host__ __device__ constexpr int tc_tiles(int D) { return D > 128 ? 1 : 2; }
__host__ __device__ constexpr int tc_item_rows(int G, int D) {
  return tc_tiles(D) * tc_tile_rows(G);
}
// Head size 256 runs every segment on the tensor-core kernel (the split-KV
// kernel's register tiles are sized for head sizes up to 128).
constexpr int kMaxHeadSplit = 128;
constexpr int kKeyTile = 64;       // keys per pipeline stage / split granularity
// Smallest KV split (keys) per class. A split-KV block spends a few
// microseconds before its first tile arrives, about the time it takes to
// stream 8 key tiles, so splits shorter than 512 keys cost more than they
// gain; prefill tiles are compute-bound and split down to 256 keys.
constexpr int kMinChunkSplit = 512;   // split-KV kernel
constexpr int kMinChunkTc = 256;      // prefill kernel
constexpr int kMaxDevices = 64;    // per-device host caches

// Work planned for one pass (one attention launch pair) lives in the
// workspace. Device-side layout, all offsets 256-byte aligned.
struct PassLayout {
  size_t header;       // int[64]: [0] items class 0, [1] items class 1, [2] abort word,
                       // [4], [5]: row groups of class 0 / 1 (when the pass lists them)
  size_t seg;          // int4[num_segs]: q_start, q_len, kv_len, class
  size_t segsplit;     // int4[num_segs]: nsplit, slot_base (in its class pool), chunk,
                       // first item in the numbering of both classes in segment order
  size_t items[2];     // int4[items_bound[c]]: seg, row tile, split index, 0
  size_t groups[2];    // int4[items_bound[c]]: seg, row tile, 0, 0 -- one per row tile
  size_t counters[2];  // int[slots_bound[c] * H_kv]
  size_t part_lse[2];  // float[slots_bound[c] * H_kv * slot_rows[c]]
  size_t part_o[2];    // float[slots_bound[c] * H_kv * slot_rows[c] * D]
  size_t end;
  int items_bound[2];
  int slots_bound[2];
  int slot_rows[2];    // rows a partial slot holds: a bound on rows per work item
  int target[2];       // split target (work items per KV head) per class
};

// Everything the planner kernel needs for one pass.
struct PlanArgs {
  const int32_t* cu_seqlens_q;
  const int32_t* seqused_k;
  int num_segs;          // sequences (or 1 for the cascade prefix pass)
  int single_segment;    // 1: one segment of total_q queries with kv_len = single_kv_len
  int total_q;
  int single_kv_len;
  int kv_len_offset;     // subtracted from seqused_k (cascade suffix pass)
  int kv_len_cap;        // keys addressable through a block_table row
  int max_q, max_k;      // host bounds (for the BAD_SEQLEN check)
  int G, H_kv;
  int D;                 // head size (sets the prefill kernel's rows per item)
  int tc_enabled;
  int tc_min_rows;       // segments with more packed rows take the prefill kernel
  int min_chunk_tc;      // smallest KV split of the prefill kernel's items (keys)
  int causal;
  int target0, target1;
  int items_bound0, items_bound1, slots_bound0, slots_bound1;
  uint8_t* ws;           // pass base
  PassLayout L;
  int32_t* status;
  int check_cascade;     // flag q_len > kv_len (suffix pass of cascade)
  int partials_only;     // every item gets a partial-state slot and a zeroed counter (cascade)
  int make_groups;       // list the (segment, row tile) groups of each class (cascade suffix)
};

struct PlanPasses {
  PlanArgs p[2];
};

// Arguments of the attention kernels (both classes).
struct AttnArgs {
  const uint16_t* q;         // bf16 or f16 elements (raw bits; see f16)
  int64_t q_stride;          // elements between tokens
  const int32_t* bt;         // block_table
  int bt_row_stride;         // 0 for the cascade prefix pass (row 0 only)
  int bt_col_offset;         // first page column (cascade suffix pass)
  int H, H_kv, G, D, bs, num_blocks;
  float scale_log2;          // softmax_scale * log2(e)
  int causal;
  uint16_t* out;             // [T, H, D] bf16 or f16 (final) or NULL
  int f16;                   // element type of q, out and the 2-byte pools: 0 bf16, 1 f16
  float* lse;                // [H, lse_stride] natural log or NULL
  int lse_stride;            // = total_q
  // Cascade. Both passes run with partials_only = 1: every work item writes
  // its partial state to its slot and nothing is combined. The combine
  // kernel then runs with merge_parts = 1: each suffix row's states are
  // merged with the prefix pass's states of the same row (prefix segment 0's
  // split info and slot pools, mp_*).
  int partials_only;
  int merge_parts;
  const int4* mp_seg;
  const int4* mp_segsplit;
  const float* mp_part_lse[2];
  const float* mp_part_o[2];
  int mp_slot_rows[2];
  // plan of this pass
  const int* header;         // [0], [1]: item counts of the two kernels
  int* abort_all;            // header[2]: set by any CTA whose wait timed out
  const int4* seg;
  const int4* segsplit;
  const int4* items;
  const int4* groups;        // this class's row groups (combine kernel)
  int* counters;             // this kernel's class pool
  float* part_lse;
  float* part_o;
  int slot_rows;
  int32_t* status;
  int box_rows;              // rows per TMA box (divides block_size and 64)
  // FP8 pools (split-KV kernel only, head size 128): K/V hold e4m3 codes and
  // a stored value means code * scale[kv head].
  int kv_fp8;
  const float* k_scale;      // [H_kv], device
  const float* v_scale;      // [H_kv], device
  // Attention sinks: one logit per query head (natural-log units of
  // softmax_scale * q.k), an extra key with value zero; NULL for none. Added
  // once per row, where the final output is written.
  const float* sinks;
  // Launch order inside one call. The kernels after the planner are launched
  // as programmatic dependents of the kernel before them, so a grid can start
  // while its predecessor drains. pdl_first = 1 for the first kernel after the
  // planner: each block waits for the planner before reading the plan. For
  // the later kernels the plan is already complete when they start (the first
  // kernel signals its dependents only after its own wait), so only the
  // grid's last block waits, which keeps the grids finishing in launch order.
  int pdl_first;
};

// Host launchers (defined in the kernel translation units).
cudaError_t launch_reshape_and_cache(const void* key, const void* value, int64_t kstride,
                                     int64_t vstride, void* kc, void* vc, int64_t block_stride,
                                     const int64_t* slots, int num_tokens, int H_kv, int D, int bs,
                                     int num_blocks, int32_t* status, cudaStream_t st, int sms,
                                     bool pdl);
// The same scatter into e4m3 pools (kc, vc, block_stride in bytes): each
// value is stored as e4m3(x / scale[kv head]).
// key / value are bf16 (f16 = 0) or f16 (f16 = 1).
cudaError_t launch_reshape_and_cache_fp8(const void* key, const void* value, int64_t kstride,
                                         int64_t vstride, void* kc, void* vc,
                                         int64_t block_stride, const int64_t* slots,
                                         int num_tokens, int H_kv, int D, int bs, int num_blocks,
                                         const float* k_scale, const float* v_scale,
                                         int32_t* status, cudaStream_t st, int sms, bool pdl,
                                         int f16);
// Merges of bf16 (f16 = 0) or f16 (f16 = 1) states.
cudaError_t launch_merge(void* out, float* out_lse, const void* a, const float* alse,
                         const void* b, const float* blse, int T, int H, int D, cudaStream_t st,
                         int sms, int f16);
// n-state merge: part r's out at parts + r * part_stride (elements), its
// LSE at parts_lse + r * lse_stride.
cudaError_t launch_merge_n(void* out, float* out_lse, const void* parts, int64_t part_stride,
                           const float* parts_lse, int64_t lse_stride, int n, int T, int H, int D,
                           cudaStream_t st, int sms, int f16);
cudaError_t launch_plan(const PlanPasses& passes, int npasses, cudaStream_t st);
cudaError_t launch_attn_split(const CUtensorMap& tmK, const CUtensorMap& tmV, const AttnArgs& a,
                              int items_bound, cudaStream_t st);
// Final combine of a cascade: for every row group of the suffix pass (both
// classes), merge its split partial states with the prefix pass's partial
// states and write out / lse. a0, a1: the suffix pass's arguments pointed at
// class 0 / 1 (merge_parts set); gb0, gb1: group bounds per class.
cudaError_t launch_cascade_combine(const AttnArgs& a0, const AttnArgs& a1, int gb0, int gb1,
                                   cudaStream_t st);
cudaError_t launch_attn_tc(const CUtensorMap& tmK, const CUtensorMap& tmV, const CUtensorMap& tmQ,
                           const AttnArgs& a, int items_bound, cudaStream_t st);

}  // namespace pa
