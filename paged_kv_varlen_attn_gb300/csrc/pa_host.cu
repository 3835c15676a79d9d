// C-ABI entry points (include/pa.h): argument validation, workspace layout,
// TMA descriptor encoding and kernel launches. Host code only; every step of
// the computation runs in the kernels of the other translation units.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstring>
#include <mutex>

#include "pa.h"
#include "pa_internal.h"

namespace pa {
namespace {

constexpr int kAbiVersion = 1;
constexpr size_t kAlign = 256;

inline size_t align_up(size_t x, size_t a = kAlign) { return (x + a - 1) / a * a; }
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline int cdiv(long long a, long long b) { return static_cast<int>((a + b - 1) / b); }

// Split targets (work items per KV head) per kernel class, from the SM count:
// the split-KV kernel runs 2 CTAs per SM and aims at ~2 waves; the prefill
// kernel runs 1 CTA per SM.
inline int target_split(int sms, int H_kv) { return cdiv(4LL * sms, H_kv); }
inline int target_tc(int sms, int H_kv) { return cdiv(1LL * sms, H_kv); }

// Segments with more than kRowsSplit packed query rows go to the tcgen05
// prefill kernel; the rest to the split-KV kernel.
constexpr bool kTcAvailable = true;

struct PassDims {
  int num_segs;   // segments planned
  int total_q;
  int max_q;      // host bound of a segment's query length
  bool single;    // one segment of total_q queries (cascade prefix pass)
  int G, H, H_kv, D;
  int sms;
  bool all_partial = false;   // every item keeps a partial-state slot (cascade prefix pass)
  bool kv_fp8 = false;        // FP8 pools (head size 128; the prefill kernel widens them)
  // The prefill kernel takes the row maximum of the raw scores and scales it
  // afterwards, which needs softmax_scale > 0; a zero or negative scale runs
  // every segment on the split-KV kernel (which scales before the maximum).
  bool tc_allowed = true;
  int max_kv = 0x7fffffff;    // host bound of a segment's key count
};

// Which kernels a pass can need, from host-known bounds only.
// Packed rows above which a segment takes the prefill kernel: every segment
// at head sizes the split-KV kernel does not take.
int tc_min_rows(int D) { return D > kMaxHeadSplit ? 0 : kTcMinRows; }
bool pass_has_tc(const PassDims& d) {
  const long long rows = static_cast<long long>(d.single ? d.total_q : d.max_q) * d.G;
  return kTcAvailable && d.tc_allowed && tc_tile_rows(d.G) > 0 && rows > tc_min_rows(d.D);
}
bool pass_has_split(const PassDims& d) {
  return d.D <= kMaxHeadSplit && (!d.single || !pass_has_tc(d));
}

// Workspace layout of one pass starting at byte offset `base`.
PassLayout layout_pass(const PassDims& d, size_t base) {
  PassLayout L{};
  const bool tc = pass_has_tc(d), sp = pass_has_split(d);
  L.target[0] = sp ? target_split(d.sms, d.H_kv) : 0;
  L.target[1] = tc ? target_tc(d.sms, d.H_kv) : 0;
  const long long rows = static_cast<long long>(d.total_q) * d.G;
  L.items_bound[0] = sp ? L.target[0] + d.num_segs + cdiv(rows, kRowsSplit) + 1 : 0;
  L.items_bound[1] = tc ? L.target[1] + d.num_segs + cdiv(rows, tc_item_rows(d.G, d.D)) + 1 : 0;
  // A second bound from the key lengths: a segment splits into at most
  // ceil(max_kv / smallest chunk) items per row tile. Where the keys are
  // short (decode suffixes of a cascade, a prefix of a few thousand keys) it
  // is far below the first, so the launches carry fewer blocks that find no
  // item and return (blocks are dispatched in index order, and a dependent
  // launch starts only once every block of its predecessor has started).
  auto by_keys = [&](int rpi, int min_chunk) {
    const long long seg_rows = static_cast<long long>(d.single ? d.total_q : d.max_q) * d.G;
    long long nrt = static_cast<long long>(d.num_segs) * cdiv(seg_rows, rpi);
    const long long nrt2 = d.num_segs + static_cast<long long>(cdiv(rows, rpi));
    if (nrt2 < nrt) nrt = nrt2;
    const long long nsp = d.max_kv > 0 ? cdiv(d.max_kv, min_chunk) : 1;
    const long long b = nrt * nsp;
    return static_cast<int>(b < 1 ? 1 : (b > 0x7fffffffLL ? 0x7fffffffLL : b));
  };
  if (sp && by_keys(kRowsSplit, kMinChunkSplit) < L.items_bound[0])
    L.items_bound[0] = by_keys(kRowsSplit, kMinChunkSplit);
  if (tc && by_keys(tc_item_rows(d.G, d.D), kMinChunkTc) < L.items_bound[1])
    L.items_bound[1] = by_keys(tc_item_rows(d.G, d.D), kMinChunkTc);
  L.slots_bound[0] = sp ? 2 * L.target[0] + 2 : 0;
  L.slots_bound[1] = tc ? 2 * L.target[1] + 2 : 0;
  if (d.all_partial) {
    L.slots_bound[0] = L.items_bound[0];
    L.slots_bound[1] = L.items_bound[1];
  }
  // A work item holds at most min(rows per item of its kernel, q_len * G) rows.
  const long long rows_bound = static_cast<long long>(d.single ? d.total_q : d.max_q) * d.G;
  auto clamp_rows = [&](int item_rows) {
    return static_cast<int>(rows_bound < item_rows ? (rows_bound > 0 ? rows_bound : 1)
                                                   : item_rows);
  };
  L.slot_rows[0] = clamp_rows(kRowsSplit);
  L.slot_rows[1] = clamp_rows(tc ? tc_item_rows(d.G, d.D) : 1);
  size_t off = align_up(base);
  L.header = off;                 off = align_up(off + 64 * sizeof(int));
  L.seg = off;                    off = align_up(off + static_cast<size_t>(d.num_segs) * 16);
  L.segsplit = off;               off = align_up(off + static_cast<size_t>(d.num_segs) * 16);
  L.items[0] = off;               off = align_up(off + static_cast<size_t>(L.items_bound[0]) * 16);
  L.items[1] = off;               off = align_up(off + static_cast<size_t>(L.items_bound[1]) * 16);
  L.groups[0] = off;              off = align_up(off + static_cast<size_t>(d.all_partial ? L.items_bound[0] : 0) * 16);
  L.groups[1] = off;              off = align_up(off + static_cast<size_t>(d.all_partial ? L.items_bound[1] : 0) * 16);
  for (int c = 0; c < 2; ++c) {
    const size_t slot_rows = static_cast<size_t>(L.slots_bound[c]) * d.H_kv * L.slot_rows[c];
    L.counters[c] = off;          off = align_up(off + static_cast<size_t>(L.slots_bound[c]) * d.H_kv * 4);
    L.part_lse[c] = off;          off = align_up(off + slot_rows * 4);
    L.part_o[c] = off;            off = align_up(off + slot_rows * d.D * 4);
  }
  L.end = off;
  return L;
}

struct CascadeLayout {
  PassLayout prefix, suffix;
  size_t end;
};

// prefix_len < 0 (the size queries, which do not take it): the bound of
// either pass's keys is max_k, which covers every prefix length.
CascadeLayout layout_cascade(int num_seqs, int total_q, int max_q, int max_k, int prefix_len,
                             int G, int H, int H_kv, int D, int sms, bool kv_fp8,
                             bool tc_allowed) {
  CascadeLayout C{};
  PassDims pd{1, total_q, total_q, true, G, H, H_kv, D, sms, true, kv_fp8, tc_allowed};
  pd.max_kv = prefix_len < 0 ? max_k : prefix_len;
  C.prefix = layout_pass(pd, 0);
  PassDims sd{num_seqs, total_q, max_q, false, G, H, H_kv, D, sms, true, kv_fp8, tc_allowed};
  sd.max_kv = prefix_len < 0 ? max_k : (max_k > prefix_len ? max_k - prefix_len : 0);
  C.suffix = layout_pass(sd, C.prefix.end);
  C.end = C.suffix.end;
  return C;
}

// Workspace bytes reported by the size queries: enough for either kernel
// choice (the choice also depends on the sign of softmax_scale, which the
// queries do not take).
size_t varlen_bytes(PassDims d) {
  d.tc_allowed = true;
  const size_t a = layout_pass(d, 0).end;
  d.tc_allowed = false;
  const size_t b = layout_pass(d, 0).end;
  return a > b ? a : b;
}
size_t cascade_bytes(int num_seqs, int total_q, int max_q, int max_k, int G, int H, int H_kv,
                     int D, int sms, bool kv_fp8) {
  const size_t a =
      layout_cascade(num_seqs, total_q, max_q, max_k, -1, G, H, H_kv, D, sms, kv_fp8, true).end;
  const size_t b =
      layout_cascade(num_seqs, total_q, max_q, max_k, -1, G, H, H_kv, D, sms, kv_fp8, false).end;
  return a > b ? a : b;
}

int query_sms(int sm_count) {
  if (sm_count > 0) return sm_count;
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

// Checks shared by the attention entry points that need no device pointer.
pa_status check_shape(int num_seqs, int total_q, int max_seqlen_q, int max_seqlen_k, int H,
                      int H_kv, int D, int bs, int dtype) {
  if (num_seqs < 0 || total_q < 0 || max_seqlen_q < 0 || max_seqlen_k < 0) return PA_ERR_INVALID_ARG;
  if (H <= 0 || H_kv <= 0 || H % H_kv != 0) return PA_ERR_INVALID_ARG;
  if (dtype != PA_BF16 && dtype != PA_F16) return PA_ERR_UNSUPPORTED;
  if (D != 64 && D != 128 && D != 256) return PA_ERR_UNSUPPORTED;
  if (bs <= 0 || bs % 16 != 0 || bs > 1024) return PA_ERR_BLOCK_SIZE;
  return PA_OK;
}

// Element type of the K/V pools: bf16, or e4m3 codes with per-KV-head scales.
struct KvFormat {
  bool fp8;
  const float* k_scale;
  const float* v_scale;
};
constexpr KvFormat kKvBf16{false, nullptr, nullptr};

pa_status check_attn_ptrs(const void* q, int64_t q_stride, const void* kc, const void* vc,
                          int64_t block_stride, const int32_t* cu, const int32_t* lens,
                          const int32_t* bt, int bt_stride, int num_seqs, int total_q,
                          int num_blocks, int H, int H_kv, int D, int bs, float scale, int causal,
                          const void* out, const float* lse, const KvFormat& kv) {
  if (num_seqs > 0 && (!cu || !lens || !bt)) return PA_ERR_INVALID_ARG;
  if (total_q > 0 && (!q || !out)) return PA_ERR_INVALID_ARG;
  if (!kc || !vc) return PA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(kc) || !aligned16(vc) || !aligned16(out)) return PA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(lse) & 3u) != 0) return PA_ERR_INVALID_ARG;
  if (q_stride < static_cast<int64_t>(H) * D || q_stride % 8 != 0) return PA_ERR_INVALID_ARG;
  // Page strides are whole 16-byte units (a TMA rule): 8 bf16 or 16 e4m3 elements.
  if (block_stride < static_cast<int64_t>(bs) * H_kv * D || block_stride % (kv.fp8 ? 16 : 8) != 0)
    return PA_ERR_INVALID_ARG;
  if (kv.fp8) {
    if (D != 128) return PA_ERR_UNSUPPORTED;
    if (!kv.k_scale || !kv.v_scale) return PA_ERR_INVALID_ARG;
    if (((reinterpret_cast<uintptr_t>(kv.k_scale) | reinterpret_cast<uintptr_t>(kv.v_scale)) & 3u) != 0)
      return PA_ERR_INVALID_ARG;
  }
  if (bt_stride < 0 || num_blocks < 0) return PA_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return PA_ERR_INVALID_ARG;
  // Head size 256 runs on the prefill kernel only, which needs a positive
  // scale and groups of at most 128 heads.
  if (D > kMaxHeadSplit && (!(scale > 0.f) || tc_tile_rows(H / H_kv) == 0))
    return PA_ERR_UNSUPPORTED;
  if (causal != 0 && causal != 1) return PA_ERR_INVALID_ARG;
  return PA_OK;
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link
// dependency on libcuda).
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 4-D view of a page pool: (dim, kv head, row in page, page), 128-byte
// swizzled boxes of 128 bytes of dims (64 bf16 or 128 e4m3) x 1 head x
// box_rows rows x 1 page. Coordinates past the pool (a page id == num_blocks)
// read as zeros.
bool encode_pool_map(CUtensorMap* map, const void* base, int D, int H_kv, int bs, int num_blocks,
                     int64_t block_stride, int box_rows, bool fp8, bool f16) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t esz = fp8 ? 1 : 2;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H_kv),
                        static_cast<cuuint64_t>(bs),
                        static_cast<cuuint64_t>(num_blocks > 0 ? num_blocks : 1)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(D) * esz,
                           static_cast<cuuint64_t>(H_kv) * D * esz,
                           static_cast<cuuint64_t>(block_stride) * esz};
  cuuint32_t box[4] = {static_cast<cuuint32_t>(128 / esz), 1, static_cast<cuuint32_t>(box_rows),
                       1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUtensorMapDataType ty = fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                : f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                      : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  CUresult r = fn(map, ty, 4,
                  const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int gcd_int(int a, int b) {
  while (b) {
    int t = a % b;
    a = b;
    b = t;
  }
  return a;
}

struct CommonAttn {
  const void* q;
  int64_t q_stride;
  const void* kc;
  const void* vc;
  int64_t block_stride;
  const int32_t* cu;
  const int32_t* lens;
  const int32_t* bt;
  int bt_stride, num_seqs, total_q, max_q, max_k, H, H_kv, D, bs, num_blocks;
  float scale;
  int32_t* status;
  cudaStream_t st;
  KvFormat kv;
  const float* sinks;   // [H] or NULL
  int dtype;            // PA_BF16 or PA_F16: q, out and the 2-byte pools
};

PlanArgs make_plan(const CommonAttn& c, uint8_t* ws, const PassLayout& L, int single, int single_kv,
                   int kv_off, int kv_cap, int causal, int check_cascade, int partials_only = 0) {
  PlanArgs p{};
  p.cu_seqlens_q = c.cu;
  p.seqused_k = c.lens;
  p.num_segs = c.num_seqs;
  p.single_segment = single;
  p.total_q = c.total_q;
  p.single_kv_len = single_kv;
  p.kv_len_offset = kv_off;
  p.kv_len_cap = kv_cap;
  p.max_q = c.max_q;
  p.max_k = c.max_k;
  p.G = c.H / c.H_kv;
  p.H_kv = c.H_kv;
  p.D = c.D;
  p.tc_enabled = L.items_bound[1] > 0 ? 1 : 0;
  p.tc_min_rows = tc_min_rows(c.D);
  p.min_chunk_tc = kMinChunkTc;
  p.causal = causal;
  p.target0 = L.target[0];
  p.target1 = L.target[1];
  p.items_bound0 = L.items_bound[0];
  p.items_bound1 = L.items_bound[1];
  p.slots_bound0 = L.slots_bound[0];
  p.slots_bound1 = L.slots_bound[1];
  p.ws = ws;
  p.L = L;
  p.status = c.status;
  p.check_cascade = check_cascade;
  p.partials_only = partials_only;
  return p;
}

AttnArgs make_attn(const CommonAttn& c, uint8_t* ws, const PassLayout& L, int bt_row_stride,
                   int bt_col_offset, int causal, void* out, float* lse) {
  AttnArgs a{};
  a.q = static_cast<const uint16_t*>(c.q);
  a.q_stride = c.q_stride;
  a.bt = c.bt;
  a.bt_row_stride = bt_row_stride;
  a.bt_col_offset = bt_col_offset;
  a.H = c.H;
  a.H_kv = c.H_kv;
  a.G = c.H / c.H_kv;
  a.D = c.D;
  a.bs = c.bs;
  a.num_blocks = c.num_blocks;
  a.scale_log2 = c.scale * 1.4426950408889634f;
  a.causal = causal;
  a.out = static_cast<uint16_t*>(out);
  a.f16 = c.dtype == PA_F16 ? 1 : 0;
  a.lse = lse;
  a.lse_stride = c.total_q;
  a.header = reinterpret_cast<const int*>(ws + L.header);
  a.abort_all = reinterpret_cast<int*>(ws + L.header) + 2;
  a.seg = reinterpret_cast<const int4*>(ws + L.seg);
  a.segsplit = reinterpret_cast<const int4*>(ws + L.segsplit);
  a.items = reinterpret_cast<const int4*>(ws + L.items[0]);
  a.status = c.status;
  a.box_rows = gcd_int(c.bs, kKeyTile);
  a.sinks = c.sinks;
  a.kv_fp8 = c.kv.fp8 ? 1 : 0;
  a.k_scale = c.kv.k_scale;
  a.v_scale = c.kv.v_scale;
  return a;
}

// Q viewed as (dim, head, token), boxes of 64 dims x G heads x floor(128/G)
// tokens: exactly the tc_tile_rows(G) packed rows of one prefill Q tile,
// 128-byte swizzled.
bool encode_q_map(CUtensorMap* map, const void* q, int D, int H, int total_q, int64_t q_stride,
                  int G, bool f16) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H),
                        static_cast<cuuint64_t>(total_q > 0 ? total_q : 1)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(q_stride) * 2};
  // G <= 128 here (wider groups never use the prefill kernel).
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(G), static_cast<cuuint32_t>(kTcTileRows / G)};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                  const_cast<void*>(q), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Point a kernel's arguments at its class's work list and partial-slot pool.
void set_class(AttnArgs& a, uint8_t* ws, const PassLayout& L, int c) {
  a.items = reinterpret_cast<const int4*>(ws + L.items[c]);
  a.groups = reinterpret_cast<const int4*>(ws + L.groups[c]);
  a.counters = reinterpret_cast<int*>(ws + L.counters[c]);
  a.part_lse = reinterpret_cast<float*>(ws + L.part_lse[c]);
  a.part_o = reinterpret_cast<float*>(ws + L.part_o[c]);
  a.slot_rows = L.slot_rows[c];
}

// Launch the kernels of one pass. *first is set while no attention kernel of
// the call has been launched since the planner; that kernel waits for the
// plan in every block (see AttnArgs::pdl_first).
pa_status launch_pass(const CommonAttn& c, const CUtensorMap& tmK, const CUtensorMap& tmV,
                      const CUtensorMap& tmQ, const AttnArgs& a, uint8_t* ws,
                      const PassLayout& L, bool* first) {
  if (L.items_bound[1] > 0) {
    AttnArgs a1 = a;
    set_class(a1, ws, L, 1);
    a1.pdl_first = *first ? 1 : 0;
    *first = false;
    if (launch_attn_tc(tmK, tmV, tmQ, a1, L.items_bound[1], c.st) != cudaSuccess)
      return PA_ERR_CUDA;
  }
  if (L.items_bound[0] > 0) {
    AttnArgs a0 = a;
    set_class(a0, ws, L, 0);
    a0.pdl_first = *first ? 1 : 0;
    *first = false;
    if (launch_attn_split(tmK, tmV, a0, L.items_bound[0], c.st) != cudaSuccess)
      return PA_ERR_CUDA;
  }
  return PA_OK;
}

// Checks of pa_reshape_and_cache's arguments (nothing launched).
pa_status check_update(const void* key, const void* value, int64_t key_token_stride,
                       int64_t value_token_stride, const void* key_cache, const void* value_cache,
                       int64_t cache_block_stride, const int64_t* slot_mapping, int num_tokens,
                       int num_kv_heads, int head_size, int block_size, int num_blocks,
                       int dtype, const KvFormat& kv = kKvBf16) {
  if (num_tokens < 0 || num_kv_heads <= 0 || num_blocks < 0) return PA_ERR_INVALID_ARG;
  if (dtype != PA_BF16 && dtype != PA_F16) return PA_ERR_UNSUPPORTED;
  if (head_size != 64 && head_size != 128 && head_size != 256) return PA_ERR_UNSUPPORTED;
  if (kv.fp8 && head_size != 128) return PA_ERR_UNSUPPORTED;
  if (block_size <= 0 || block_size % 16 != 0 || block_size > 1024) return PA_ERR_BLOCK_SIZE;
  if (num_tokens == 0) return PA_OK;
  if (kv.fp8 && (!kv.k_scale || !kv.v_scale ||
                 ((reinterpret_cast<uintptr_t>(kv.k_scale) |
                   reinterpret_cast<uintptr_t>(kv.v_scale)) & 3u) != 0))
    return PA_ERR_INVALID_ARG;
  if (!key || !value || !key_cache || !value_cache || !slot_mapping) return PA_ERR_INVALID_ARG;
  if (!aligned16(key) || !aligned16(value) || !aligned16(key_cache) || !aligned16(value_cache))
    return PA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(slot_mapping) & 7u) != 0) return PA_ERR_INVALID_ARG;
  const int64_t row = static_cast<int64_t>(num_kv_heads) * head_size;
  if (key_token_stride < row || value_token_stride < row || key_token_stride % 8 ||
      value_token_stride % 8)
    return PA_ERR_INVALID_ARG;
  if (cache_block_stride < row * block_size || cache_block_stride % (kv.fp8 ? 16 : 8))
    return PA_ERR_INVALID_ARG;
  return PA_OK;
}

// The scatter of pa_reshape_and_cache(_fp8) for the cache format kv.
cudaError_t launch_scatter(const void* key, const void* value, int64_t kstride, int64_t vstride,
                           void* kc, void* vc, int64_t block_stride, const int64_t* slots,
                           int num_tokens, int H_kv, int D, int bs, int num_blocks,
                           const KvFormat& kv, int32_t* status, cudaStream_t st, int sms,
                           bool pdl, int dtype) {
  if (kv.fp8)
    return launch_reshape_and_cache_fp8(key, value, kstride, vstride, kc, vc, block_stride, slots,
                                        num_tokens, H_kv, D, bs, num_blocks, kv.k_scale,
                                        kv.v_scale, status, st, sms, pdl, dtype == PA_F16);
  return launch_reshape_and_cache(key, value, kstride, vstride, kc, vc, block_stride, slots,
                                  num_tokens, H_kv, D, bs, num_blocks, status, st, sms, pdl);
}

// Validate an optional K/V update of an update-and-attend call.
pa_status check_kv_update(const pa_kv_update* u, const CommonAttn& c, void* key_cache,
                          void* value_cache, int dtype) {
  if (!u || u->num_tokens == 0) return u && u->num_tokens < 0 ? PA_ERR_INVALID_ARG : PA_OK;
  return check_update(u->key, u->value, u->key_token_stride, u->value_token_stride, key_cache,
                      value_cache, c.block_stride, u->slot_mapping, u->num_tokens, c.H_kv, c.D,
                      c.bs, c.num_blocks, dtype, c.kv);
}

// Launch the update's scatter right after the planner, as a programmatic
// dependent: it overlaps the planner (its inputs predate the call), and the
// first attention kernel waits for it before reading the cache.
pa_status launch_kv_update(const pa_kv_update* u, const CommonAttn& c, void* key_cache,
                           void* value_cache, int sms) {
  if (!u || u->num_tokens == 0) return PA_OK;
  return launch_scatter(u->key, u->value, u->key_token_stride, u->value_token_stride, key_cache,
                        value_cache, c.block_stride, u->slot_mapping, u->num_tokens, c.H_kv, c.D,
                        c.bs, c.num_blocks, c.kv, c.status, c.st, sms, true, c.dtype) == cudaSuccess
             ? PA_OK
             : PA_ERR_CUDA;
}

}  // namespace
}  // namespace pa

using namespace pa;

extern "C" {

const char* pa_status_string(pa_status s) {
  switch (s) {
    case PA_OK: return "PA_OK";
    case PA_ERR_INVALID_ARG: return "PA_ERR_INVALID_ARG: invalid argument";
    case PA_ERR_BLOCK_SIZE: return "PA_ERR_BLOCK_SIZE: block size must be a multiple of 16 (<= 1024)";
    case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED: head size or dtype not supported";
    case PA_ERR_WORKSPACE: return "PA_ERR_WORKSPACE: workspace missing, misaligned or too small";
    case PA_ERR_CUDA: return "PA_ERR_CUDA: CUDA launch or query failed";
    case PA_ERR_NOALLOC_LIMIT:
      return "PA_ERR_NOALLOC_LIMIT: the problem needs more scratch than the fixed no-allocation "
             "buffer (PA_NOALLOC_SCRATCH_BYTES) holds; use pa_varlen_fwd with a workspace";
    default: return "PA_ERR_UNKNOWN";
  }
}

int pa_abi_version(void) { return kAbiVersion; }

pa_status pa_reshape_and_cache(const void* key, const void* value, int64_t key_token_stride,
                               int64_t value_token_stride, void* key_cache, void* value_cache,
                               int64_t cache_block_stride, const int64_t* slot_mapping,
                               int num_tokens, int num_kv_heads, int head_size, int block_size,
                               int num_blocks, int dtype, int32_t* dev_status, void* stream) {
  const pa_status st = check_update(key, value, key_token_stride, value_token_stride, key_cache,
                                    value_cache, cache_block_stride, slot_mapping, num_tokens,
                                    num_kv_heads, head_size, block_size, num_blocks, dtype);
  if (st != PA_OK || num_tokens == 0) return st;
  const int sms = query_sms(0);
  if (sms <= 0) return PA_ERR_CUDA;
  cudaError_t e = launch_reshape_and_cache(key, value, key_token_stride, value_token_stride,
                                           key_cache, value_cache, cache_block_stride,
                                           slot_mapping, num_tokens, num_kv_heads, head_size,
                                           block_size, num_blocks, dev_status,
                                           static_cast<cudaStream_t>(stream), sms, false);
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

size_t pa_varlen_fwd_workspace_size(int num_seqs, int total_q, int max_seqlen_q, int max_seqlen_k,
                                    int num_heads, int num_kv_heads, int head_size, int block_size,
                                    int sm_count) {
  if (check_shape(num_seqs, total_q, max_seqlen_q, max_seqlen_k, num_heads, num_kv_heads,
                  head_size, block_size, PA_BF16) != PA_OK)
    return 0;
  const int sms = query_sms(sm_count);
  if (sms <= 0) return 0;
  PassDims d{num_seqs, total_q, max_seqlen_q, false, num_heads / num_kv_heads, num_heads,
             num_kv_heads, head_size, sms};
  d.max_kv = max_seqlen_k;
  return varlen_bytes(d);
}

size_t pa_cascade_fwd_workspace_size(int num_seqs, int total_q, int max_seqlen_q,
                                     int max_seqlen_k, int num_heads, int num_kv_heads,
                                     int head_size, int block_size, int sm_count) {
  if (check_shape(num_seqs, total_q, max_seqlen_q, max_seqlen_k, num_heads, num_kv_heads,
                  head_size, block_size, PA_BF16) != PA_OK)
    return 0;
  const int sms = query_sms(sm_count);
  if (sms <= 0) return 0;
  return cascade_bytes(num_seqs, total_q, max_seqlen_q, max_seqlen_k, num_heads / num_kv_heads,
                       num_heads, num_kv_heads, head_size, sms, false);
}

// pa_varlen_fwd, optionally preceded by a K/V update of the same cache.
static pa_status varlen_impl(const pa_kv_update* upd, const void* q, int64_t q_token_stride,
                             void* key_cache, void* value_cache, int64_t cache_block_stride,
                             const int32_t* cu_seqlens_q, const int32_t* seqused_k,
                             const int32_t* block_table, int bt_stride, int num_seqs, int total_q,
                             int max_seqlen_q, int max_seqlen_k, int num_heads, int num_kv_heads,
                             int head_size, int block_size, int num_blocks, float softmax_scale,
                             int causal, void* out, float* lse, void* workspace,
                             size_t workspace_bytes, int dtype, int32_t* dev_status,
                             void* stream, const KvFormat& kv, const float* sinks = nullptr) {
  pa_status st = check_shape(num_seqs, total_q, max_seqlen_q, max_seqlen_k, num_heads,
                             num_kv_heads, head_size, block_size, dtype);
  if (st != PA_OK) return st;
  st = check_attn_ptrs(q, q_token_stride, key_cache, value_cache, cache_block_stride, cu_seqlens_q,
                       seqused_k, block_table, bt_stride, num_seqs, total_q, num_blocks, num_heads,
                       num_kv_heads, head_size, block_size, softmax_scale, causal, out, lse, kv);
  if (st != PA_OK) return st;
  if ((reinterpret_cast<uintptr_t>(sinks) & 3u) != 0) return PA_ERR_INVALID_ARG;
  CommonAttn c{q, q_token_stride, key_cache, value_cache, cache_block_stride, cu_seqlens_q,
               seqused_k, block_table, bt_stride, num_seqs, total_q, max_seqlen_q, max_seqlen_k,
               num_heads, num_kv_heads, head_size, block_size, num_blocks, softmax_scale,
               dev_status, static_cast<cudaStream_t>(stream), kv, sinks, dtype};
  st = check_kv_update(upd, c, key_cache, value_cache, dtype);
  if (st != PA_OK) return st;
  if (num_seqs == 0 || total_q == 0) {   // nothing to attend: the update alone
    if (!upd || upd->num_tokens == 0) return PA_OK;
    const int sms = query_sms(0);
    if (sms <= 0) return PA_ERR_CUDA;
    return launch_scatter(upd->key, upd->value, upd->key_token_stride, upd->value_token_stride,
                          key_cache, value_cache, cache_block_stride, upd->slot_mapping,
                          upd->num_tokens, num_kv_heads, head_size, block_size, num_blocks, kv,
                          dev_status, c.st, sms, false, dtype) == cudaSuccess
               ? PA_OK
               : PA_ERR_CUDA;
  }
  const int sms = query_sms(0);
  if (sms <= 0) return PA_ERR_CUDA;
  PassDims d{num_seqs, total_q, max_seqlen_q, false, num_heads / num_kv_heads, num_heads,
             num_kv_heads, head_size, sms};
  d.max_kv = max_seqlen_k;
  d.kv_fp8 = kv.fp8;
  d.tc_allowed = softmax_scale > 0.f;
  const PassLayout L = layout_pass(d, 0);
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) % kAlign) != 0 ||
      workspace_bytes < L.end)
    return PA_ERR_WORKSPACE;
  const int box_rows = gcd_int(block_size, kKeyTile);
  CUtensorMap tmK, tmV;
  if (!encode_pool_map(&tmK, key_cache, head_size, num_kv_heads, block_size, num_blocks,
                       cache_block_stride, box_rows, kv.fp8, dtype == PA_F16) ||
      !encode_pool_map(&tmV, value_cache, head_size, num_kv_heads, block_size, num_blocks,
                       cache_block_stride, box_rows, kv.fp8, dtype == PA_F16))
    return PA_ERR_CUDA;
  CUtensorMap tmQ{};
  if (L.items_bound[1] > 0 &&
      !encode_q_map(&tmQ, q, head_size, num_heads, total_q, q_token_stride,
                    num_heads / num_kv_heads, dtype == PA_F16))
    return PA_ERR_CUDA;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const long long cap = static_cast<long long>(bt_stride) * block_size;
  PlanPasses pp{};
  pp.p[0] = make_plan(c, ws, L, 0, 0, 0, cap > 0x7fffffff ? 0x7fffffff : static_cast<int>(cap),
                      causal, 0);
  if (launch_plan(pp, 1, c.st) != cudaSuccess) return PA_ERR_CUDA;
  st = launch_kv_update(upd, c, key_cache, value_cache, sms);
  if (st != PA_OK) return st;
  AttnArgs a = make_attn(c, ws, L, bt_stride, 0, causal, out, lse);
  bool first = true;
  return launch_pass(c, tmK, tmV, tmQ, a, ws, L, &first);
}

pa_status pa_use_cascade_attention(int common_prefix_len, int num_seqs, int num_kv_heads,
                                   int head_size, int split_kv, int* use_cascade) {
  if (!use_cascade || common_prefix_len < 0 || num_seqs < 0 || num_kv_heads <= 0 ||
      head_size <= 0)
    return PA_ERR_INVALID_ARG;
  *use_cascade = 0;
  if (common_prefix_len < 256 || num_seqs < 8) return PA_OK;   // the pages' two thresholds
  if (!split_kv) {
    *use_cascade = 1;
    return PA_OK;
  }
  // Bytes of the shared prefix that flat attention re-reads (K and V, bf16)
  // against the bytes the cascade's fixed cost could have moved.
  const double reread = static_cast<double>(num_seqs - 1) * common_prefix_len * num_kv_heads *
                        head_size * 4.0;
  const double fixed = PA_CASCADE_FIXED_US * 1e-6 * PA_CASCADE_HBM_GBS * 1e9;
  *use_cascade = reread > fixed ? 1 : 0;
  return PA_OK;
}

pa_status pa_varlen_fwd(const void* q, int64_t q_token_stride, const void* key_cache,
                        const void* value_cache, int64_t cache_block_stride,
                        const int32_t* cu_seqlens_q, const int32_t* seqused_k,
                        const int32_t* block_table, int bt_stride, int num_seqs, int total_q,
                        int max_seqlen_q, int max_seqlen_k, int num_heads, int num_kv_heads,
                        int head_size, int block_size, int num_blocks, float softmax_scale,
                        int causal, void* out, float* lse, void* workspace,
                        size_t workspace_bytes, int dtype, int32_t* dev_status, void* stream) {
  return varlen_impl(nullptr, q, q_token_stride, const_cast<void*>(key_cache),
                     const_cast<void*>(value_cache), cache_block_stride, cu_seqlens_q, seqused_k,
                     block_table, bt_stride, num_seqs, total_q, max_seqlen_q, max_seqlen_k,
                     num_heads, num_kv_heads, head_size, block_size, num_blocks, softmax_scale,
                     causal, out, lse, workspace, workspace_bytes, dtype, dev_status, stream,
                     kKvBf16);
}

pa_status pa_varlen_fwd_with_update(const pa_kv_update* update, const void* q,
                                    int64_t q_token_stride, void* key_cache, void* value_cache,
                                    int64_t cache_block_stride, const int32_t* cu_seqlens_q,
                                    const int32_t* seqused_k, const int32_t* block_table,
                                    int bt_stride, int num_seqs, int total_q, int max_seqlen_q,
                                    int max_seqlen_k, int num_heads, int num_kv_heads,
                                    int head_size, int block_size, int num_blocks,
                                    float softmax_scale, int causal, void* out, float* lse,
                                    void* workspace, size_t workspace_bytes, int dtype,
                                    int32_t* dev_status, void* stream) {
  return varlen_impl(update, q, q_token_stride, key_cache, value_cache, cache_block_stride,
                     cu_seqlens_q, seqused_k, block_table, bt_stride, num_seqs, total_q,
                     max_seqlen_q, max_seqlen_k, num_heads, num_kv_heads, head_size, block_size,
                     num_blocks, softmax_scale, causal, out, lse, workspace, workspace_bytes,
                     dtype, dev_status, stream, kKvBf16);
}

pa_status pa_merge_attn_states(void* out, float* out_lse, const void* prefix_out,
                               const float* prefix_lse, const void* suffix_out,
                               const float* suffix_lse, int num_tokens, int num_heads,
                               int head_size, int dtype, void* stream) {
  if (num_tokens < 0 || num_heads <= 0) return PA_ERR_INVALID_ARG;
  if (dtype != PA_BF16 && dtype != PA_F16) return PA_ERR_UNSUPPORTED;
  if (head_size <= 0 || head_size % 8 != 0 || head_size > 256) return PA_ERR_UNSUPPORTED;
  if (num_tokens == 0) return PA_OK;
  if (!out || !prefix_out || !suffix_out || !prefix_lse || !suffix_lse) return PA_ERR_INVALID_ARG;
  if (!aligned16(out) || !aligned16(prefix_out) || !aligned16(suffix_out)) return PA_ERR_INVALID_ARG;
  if (((reinterpret_cast<uintptr_t>(prefix_lse) | reinterpret_cast<uintptr_t>(suffix_lse) |
        reinterpret_cast<uintptr_t>(out_lse)) & 3u) != 0)
    return PA_ERR_INVALID_ARG;
  if (out_lse && (out_lse == prefix_lse || out_lse == suffix_lse)) return PA_ERR_INVALID_ARG;
  const int sms = query_sms(0);
  if (sms <= 0) return PA_ERR_CUDA;
  cudaError_t e = launch_merge(out, out_lse, prefix_out, prefix_lse, suffix_out, suffix_lse,
                               num_tokens, num_heads, head_size,
                               static_cast<cudaStream_t>(stream), sms, dtype == PA_F16);
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

pa_status pa_merge_attn_states_n(void* out, float* out_lse, const void* parts_out,
                                 int64_t part_stride_out, const float* parts_lse,
                                 int64_t part_stride_lse, int num_parts, int num_tokens,
                                 int num_heads, int head_size, int dtype, void* stream) {
  if (num_parts < 1 || num_parts > PA_MERGE_N_MAX || num_tokens < 0 || num_heads <= 0)
    return PA_ERR_INVALID_ARG;
  if (dtype != PA_BF16 && dtype != PA_F16) return PA_ERR_UNSUPPORTED;
  if (head_size <= 0 || head_size % 8 != 0 || head_size > 256) return PA_ERR_UNSUPPORTED;
  if (num_tokens == 0) return PA_OK;
  if (!out || !parts_out || !parts_lse) return PA_ERR_INVALID_ARG;
  if (!aligned16(out) || !aligned16(parts_out)) return PA_ERR_INVALID_ARG;
  if (((reinterpret_cast<uintptr_t>(parts_lse) | reinterpret_cast<uintptr_t>(out_lse)) & 3u) != 0)
    return PA_ERR_INVALID_ARG;
  const int64_t row_elems = static_cast<int64_t>(num_tokens) * num_heads * head_size;
  const int64_t lse_elems = static_cast<int64_t>(num_heads) * num_tokens;
  if (num_parts > 1 && (part_stride_out < row_elems || part_stride_out % 8 != 0 ||
                        part_stride_lse < lse_elems))
    return PA_ERR_INVALID_ARG;
  if (out_lse) {   // out_lse must not overlap any part's LSE (other threads still read them)
    const float* lo = parts_lse;
    const float* hi = parts_lse + (num_parts - 1) * part_stride_lse + lse_elems;
    if (out_lse + lse_elems > lo && out_lse < hi) return PA_ERR_INVALID_ARG;
  }
  const int sms = query_sms(0);
  if (sms <= 0) return PA_ERR_CUDA;
  cudaError_t e = launch_merge_n(out, out_lse, parts_out, part_stride_out, parts_lse,
                                 part_stride_lse, num_parts, num_tokens, num_heads, head_size,
                                 static_cast<cudaStream_t>(stream), sms, dtype == PA_F16);
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

// pa_cascade_fwd, optionally preceded by a K/V update of the same cache.
static pa_status cascade_impl(const pa_kv_update* upd, const void* q, int64_t q_token_stride,
                              void* key_cache, void* value_cache, int64_t cache_block_stride,
                              const int32_t* cu_seqlens_q, const int32_t* seqused_k,
                              const int32_t* block_table, int bt_stride, int num_seqs,
                              int total_q, int max_seqlen_q, int max_seqlen_k, int num_heads,
                              int num_kv_heads, int head_size, int block_size, int num_blocks,
                              float softmax_scale, int common_prefix_len, void* out, float* lse,
                              void* workspace, size_t workspace_bytes, int dtype,
                              int32_t* dev_status, void* stream, const KvFormat& kv,
                              const float* sinks = nullptr) {
  pa_status st = check_shape(num_seqs, total_q, max_seqlen_q, max_seqlen_k, num_heads,
                             num_kv_heads, head_size, block_size, dtype);
  if (st != PA_OK) return st;
  st = check_attn_ptrs(q, q_token_stride, key_cache, value_cache, cache_block_stride, cu_seqlens_q,
                       seqused_k, block_table, bt_stride, num_seqs, total_q, num_blocks, num_heads,
                       num_kv_heads, head_size, block_size, softmax_scale, 1, out, lse, kv);
  if (st != PA_OK) return st;
  if ((reinterpret_cast<uintptr_t>(sinks) & 3u) != 0) return PA_ERR_INVALID_ARG;
  if (st != PA_OK) return st;
  if (common_prefix_len < 0 || common_prefix_len % block_size != 0) return PA_ERR_INVALID_ARG;
  if (static_cast<long long>(common_prefix_len) > static_cast<long long>(bt_stride) * block_size)
    return PA_ERR_INVALID_ARG;
  {
    const CommonAttn cu{q, q_token_stride, key_cache, value_cache, cache_block_stride,
                        cu_seqlens_q, seqused_k, block_table, bt_stride, num_seqs, total_q,
                        max_seqlen_q, max_seqlen_k, num_heads, num_kv_heads, head_size,
                        block_size, num_blocks, softmax_scale, dev_status,
                        static_cast<cudaStream_t>(stream), kv, sinks, dtype};
    st = check_kv_update(upd, cu, key_cache, value_cache, dtype);
    if (st != PA_OK) return st;
  }
  if (num_seqs == 0 || total_q == 0) {   // nothing to attend: the update alone
    if (!upd || upd->num_tokens == 0) return PA_OK;
    const int sms = query_sms(0);
    if (sms <= 0) return PA_ERR_CUDA;
    return launch_scatter(upd->key, upd->value, upd->key_token_stride, upd->value_token_stride,
                          key_cache, value_cache, cache_block_stride, upd->slot_mapping,
                          upd->num_tokens, num_kv_heads, head_size, block_size, num_blocks, kv,
                          dev_status, static_cast<cudaStream_t>(stream), sms, false, dtype) == cudaSuccess
               ? PA_OK
               : PA_ERR_CUDA;
  }
  const int sms = query_sms(0);
  if (sms <= 0) return PA_ERR_CUDA;
  const int G = num_heads / num_kv_heads;
  const CascadeLayout CL = layout_cascade(num_seqs, total_q, max_seqlen_q, max_seqlen_k,
                                          common_prefix_len, G, num_heads, num_kv_heads,
                                          head_size, sms, kv.fp8, softmax_scale > 0.f);
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) % kAlign) != 0 ||
      workspace_bytes < CL.end)
    return PA_ERR_WORKSPACE;
  CommonAttn c{q, q_token_stride, key_cache, value_cache, cache_block_stride, cu_seqlens_q,
               seqused_k, block_table, bt_stride, num_seqs, total_q, max_seqlen_q, max_seqlen_k,
               num_heads, num_kv_heads, head_size, block_size, num_blocks, softmax_scale,
               dev_status, static_cast<cudaStream_t>(stream), kv, sinks, dtype};
  const int box_rows = gcd_int(block_size, kKeyTile);
  CUtensorMap tmK, tmV;
  if (!encode_pool_map(&tmK, key_cache, head_size, num_kv_heads, block_size, num_blocks,
                       cache_block_stride, box_rows, kv.fp8, dtype == PA_F16) ||
      !encode_pool_map(&tmV, value_cache, head_size, num_kv_heads, block_size, num_blocks,
                       cache_block_stride, box_rows, kv.fp8, dtype == PA_F16))
    return PA_ERR_CUDA;
  CUtensorMap tmQ{};
  if ((CL.prefix.items_bound[1] > 0 || CL.suffix.items_bound[1] > 0) &&
      !encode_q_map(&tmQ, q, head_size, num_heads, total_q, q_token_stride, G, dtype == PA_F16))
    return PA_ERR_CUDA;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const int P = common_prefix_len;
  const int pages = P / block_size;
  const long long cap = (static_cast<long long>(bt_stride) - pages) * block_size;
  PlanPasses pp{};
  // Pass A: all queries, one non-causal segment, row 0's first P keys; every
  // work item leaves its partial state in its slot.
  pp.p[0] = make_plan(c, ws, CL.prefix, 1, P, 0, P, 0, 0, 1);
  // The prefix pass's items hold every query row of a KV head, and the two
  // passes run side by side. Over 2-byte pools the suffix pass is the longer
  // and finer prefix chunks only take SMs from it; over e4m3 pools the suffix
  // streams half the bytes and the prefix pass is the longer one. Measured on
  // 64 decode requests sharing 2048 tokens (graph step): 2-byte pools 48.2 us
  // with 512-key chunks, 52.4 with 256; e4m3 pools 50.3 with 512, 46.2 with
  // 256.
  pp.p[0].min_chunk_tc = kv.fp8 ? kMinChunkTc : 2 * kMinChunkTc;
  // Pass B: each sequence, causal, its own keys from position P on; each final
  // row is merged with pass A's partial states of the same row.
  pp.p[1] = make_plan(c, ws, CL.suffix, 0, 0, P,
                      cap > 0x7fffffff ? 0x7fffffff : static_cast<int>(cap), 1, 1, 1);
  pp.p[1].make_groups = 1;
  if (launch_plan(pp, 2, c.st) != cudaSuccess) return PA_ERR_CUDA;
  st = launch_kv_update(upd, c, key_cache, value_cache, sms);
  if (st != PA_OK) return st;
  AttnArgs pa_ = make_attn(c, ws, CL.prefix, 0, 0, 0, nullptr, nullptr);
  pa_.partials_only = 1;
  bool first = true;
  st = launch_pass(c, tmK, tmV, tmQ, pa_, ws, CL.prefix, &first);
  if (st != PA_OK) return st;
  // Pass B: each sequence, causal, its own keys from position P on; every
  // work item leaves its partial state too, so no block of either pass waits
  // for the other.
  AttnArgs pb = make_attn(c, ws, CL.suffix, bt_stride, pages, 1, out, lse);
  pb.partials_only = 1;
  st = launch_pass(c, tmK, tmV, tmQ, pb, ws, CL.suffix, &first);
  if (st != PA_OK) return st;
  // Combine: each row of pass B merges its own partial states with pass A's.
  AttnArgs cb = pb;
  cb.partials_only = 0;
  cb.merge_parts = 1;
  cb.mp_seg = reinterpret_cast<const int4*>(ws + CL.prefix.seg);
  cb.mp_segsplit = reinterpret_cast<const int4*>(ws + CL.prefix.segsplit);
  for (int k = 0; k < 2; ++k) {
    cb.mp_part_lse[k] = reinterpret_cast<const float*>(ws + CL.prefix.part_lse[k]);
    cb.mp_part_o[k] = reinterpret_cast<const float*>(ws + CL.prefix.part_o[k]);
    cb.mp_slot_rows[k] = CL.prefix.slot_rows[k];
  }
  AttnArgs c0 = cb, c1 = cb;
  set_class(c0, ws, CL.suffix, 0);
  set_class(c1, ws, CL.suffix, 1);
  if (launch_cascade_combine(c0, c1, CL.suffix.items_bound[0], CL.suffix.items_bound[1], c.st) !=
      cudaSuccess)
    return PA_ERR_CUDA;
  return PA_OK;
}

pa_status pa_cascade_fwd(const void* q, int64_t q_token_stride, const void* key_cache,
                         const void* value_cache, int64_t cache_block_stride,
                         const int32_t* cu_seqlens_q, const int32_t* seqused_k,
                         const int32_t* block_table, int bt_stride, int num_seqs, int total_q,
                         int max_seqlen_q, int max_seqlen_k, int num_heads, int num_kv_heads,
                         int head_size, int block_size, int num_blocks, float softmax_scale,
                         int common_prefix_len, void* out, float* lse, void* workspace,
                         size_t workspace_bytes, int dtype, int32_t* dev_status, void* stream) {
  return cascade_impl(nullptr, q, q_token_stride, const_cast<void*>(key_cache),
                      const_cast<void*>(value_cache), cache_block_stride, cu_seqlens_q, seqused_k,
                      block_table, bt_stride, num_seqs, total_q, max_seqlen_q, max_seqlen_k,
                      num_heads, num_kv_heads, head_size, block_size, num_blocks, softmax_scale,
                      common_prefix_len, out, lse, workspace, workspace_bytes, dtype, dev_status,
                      stream, kKvBf16);
}

pa_status pa_cascade_fwd_with_update(const pa_kv_update* update, const void* q,
                                     int64_t q_token_stride, void* key_cache, void* value_cache,
                                     int64_t cache_block_stride, const int32_t* cu_seqlens_q,
                                     const int32_t* seqused_k, const int32_t* block_table,
                                     int bt_stride, int num_seqs, int total_q, int max_seqlen_q,
                                     int max_seqlen_k, int num_heads, int num_kv_heads,
                                     int head_size, int block_size, int num_blocks,
                                     float softmax_scale, int common_prefix_len, void* out,
                                     float* lse, void* workspace, size_t workspace_bytes,
                                     int dtype, int32_t* dev_status, void* stream) {
  return cascade_impl(update, q, q_token_stride, key_cache, value_cache, cache_block_stride,
                      cu_seqlens_q, seqused_k, block_table, bt_stride, num_seqs, total_q,
                      max_seqlen_q, max_seqlen_k, num_heads, num_kv_heads, head_size, block_size,
                      num_blocks, softmax_scale, common_prefix_len, out, lse, workspace,
                      workspace_bytes, dtype, dev_status, stream, kKvBf16);
}

// ---------------------------------------------------------------- FP8 cache
static KvFormat fp8_format(const pa_kv_fp8* f) {
  return KvFormat{true, f ? f->k_scale : nullptr, f ? f->v_scale : nullptr};
}

pa_status pa_reshape_and_cache_fp8(const void* key, const void* value, int64_t key_token_stride,
                                   int64_t value_token_stride, void* key_cache, void* value_cache,
                                   int64_t cache_block_stride, const int64_t* slot_mapping,
                                   int num_tokens, int num_kv_heads, int head_size,
                                   int block_size, int num_blocks, const pa_kv_fp8* scales,
                                   int dtype, int32_t* dev_status, void* stream) {
  const KvFormat kv = fp8_format(scales);
  const pa_status st =
      check_update(key, value, key_token_stride, value_token_stride, key_cache, value_cache,
                   cache_block_stride, slot_mapping, num_tokens, num_kv_heads, head_size,
                   block_size, num_blocks, dtype, kv);
  if (st != PA_OK || num_tokens == 0) return st;
  const int sms = query_sms(0);
  if (sms <= 0) return PA_ERR_CUDA;
  return launch_scatter(key, value, key_token_stride, value_token_stride, key_cache, value_cache,
                        cache_block_stride, slot_mapping, num_tokens, num_kv_heads, head_size,
                        block_size, num_blocks, kv, dev_status, static_cast<cudaStream_t>(stream),
                        sms, false, dtype) == cudaSuccess
             ? PA_OK
             : PA_ERR_CUDA;
}

size_t pa_varlen_fwd_fp8kv_workspace_size(int num_seqs, int total_q, int max_seqlen_q,
                                          int max_seqlen_k, int num_heads, int num_kv_heads,
                                          int head_size, int block_size, int sm_count) {
  if (check_shape(num_seqs, total_q, max_seqlen_q, max_seqlen_k, num_heads, num_kv_heads,
                  head_size, block_size, PA_BF16) != PA_OK || head_size != 128)
    return 0;
  const int sms = query_sms(sm_count);
  if (sms <= 0) return 0;
  PassDims d{num_seqs, total_q, max_seqlen_q, false, num_heads / num_kv_heads, num_heads,
             num_kv_heads, head_size, sms};
  d.max_kv = max_seqlen_k;
  d.kv_fp8 = true;
  return varlen_bytes(d);
}

size_t pa_cascade_fwd_fp8kv_workspace_size(int num_seqs, int total_q, int max_seqlen_q,
                                           int max_seqlen_k, int num_heads, int num_kv_heads,
                                           int head_size, int block_size, int sm_count) {
  if (check_shape(num_seqs, total_q, max_seqlen_q, max_seqlen_k, num_heads, num_kv_heads,
                  head_size, block_size, PA_BF16) != PA_OK || head_size != 128)
    return 0;
  const int sms = query_sms(sm_count);
  if (sms <= 0) return 0;
  return cascade_bytes(num_seqs, total_q, max_seqlen_q, max_seqlen_k, num_heads / num_kv_heads,
                       num_heads, num_kv_heads, head_size, sms, true);
}

pa_status pa_varlen_fwd_fp8kv(const pa_kv_update* update, const void* q, int64_t q_token_stride,
                              void* key_cache, void* value_cache, int64_t cache_block_stride,
                              const int32_t* cu_seqlens_q, const int32_t* seqused_k,
                              const int32_t* block_table, int bt_stride, int num_seqs,
                              int total_q, int max_seqlen_q, int max_seqlen_k, int num_heads,
                              int num_kv_heads, int head_size, int block_size, int num_blocks,
                              float softmax_scale, int causal, const pa_kv_fp8* scales, void* out,
                              float* lse, void* workspace, size_t workspace_bytes, int dtype,
                              int32_t* dev_status, void* stream) {
  return varlen_impl(update, q, q_token_stride, key_cache, value_cache, cache_block_stride,
                     cu_seqlens_q, seqused_k, block_table, bt_stride, num_seqs, total_q,
                     max_seqlen_q, max_seqlen_k, num_heads, num_kv_heads, head_size, block_size,
                     num_blocks, softmax_scale, causal, out, lse, workspace, workspace_bytes,
                     dtype, dev_status, stream, fp8_format(scales));
}

pa_status pa_cascade_fwd_fp8kv(const pa_kv_update* update, const void* q,
                               int64_t q_token_stride, void* key_cache, void* value_cache,
                               int64_t cache_block_stride, const int32_t* cu_seqlens_q,
                               const int32_t* seqused_k, const int32_t* block_table,
                               int bt_stride, int num_seqs, int total_q, int max_seqlen_q,
                               int max_seqlen_k, int num_heads, int num_kv_heads, int head_size,
                               int block_size, int num_blocks, float softmax_scale,
                               int common_prefix_len, const pa_kv_fp8* scales, void* out,
                               float* lse, void* workspace, size_t workspace_bytes, int dtype,
                               int32_t* dev_status, void* stream) {
  return cascade_impl(update, q, q_token_stride, key_cache, value_cache, cache_block_stride,
                      cu_seqlens_q, seqused_k, block_table, bt_stride, num_seqs, total_q,
                      max_seqlen_q, max_seqlen_k, num_heads, num_kv_heads, head_size, block_size,
                      num_blocks, softmax_scale, common_prefix_len, out, lse, workspace,
                      workspace_bytes, dtype, dev_status, stream, fp8_format(scales));
}

// ---------------------------------------------------------------- options
pa_status pa_varlen_fwd_ex(const pa_kv_update* update, const void* q, int64_t q_token_stride,
                           void* key_cache, void* value_cache, int64_t cache_block_stride,
                           const int32_t* cu_seqlens_q, const int32_t* seqused_k,
                           const int32_t* block_table, int bt_stride, int num_seqs, int total_q,
                           int max_seqlen_q, int max_seqlen_k, int num_heads, int num_kv_heads,
                           int head_size, int block_size, int num_blocks, float softmax_scale,
                           int causal, const pa_attn_opts* opts, void* out, float* lse,
                           void* workspace, size_t workspace_bytes, int dtype,
                           int32_t* dev_status, void* stream) {
  const KvFormat kv = opts && opts->fp8 ? fp8_format(opts->fp8) : kKvBf16;
  return varlen_impl(update, q, q_token_stride, key_cache, value_cache, cache_block_stride,
                     cu_seqlens_q, seqused_k, block_table, bt_stride, num_seqs, total_q,
                     max_seqlen_q, max_seqlen_k, num_heads, num_kv_heads, head_size, block_size,
                     num_blocks, softmax_scale, causal, out, lse, workspace, workspace_bytes,
                     dtype, dev_status, stream, kv, opts ? opts->sinks : nullptr);
}

pa_status pa_cascade_fwd_ex(const pa_kv_update* update, const void* q, int64_t q_token_stride,
                            void* key_cache, void* value_cache, int64_t cache_block_stride,
                            const int32_t* cu_seqlens_q, const int32_t* seqused_k,
                            const int32_t* block_table, int bt_stride, int num_seqs,
                            int total_q, int max_seqlen_q, int max_seqlen_k, int num_heads,
                            int num_kv_heads, int head_size, int block_size, int num_blocks,
                            float softmax_scale, int common_prefix_len, const pa_attn_opts* opts,
                            void* out, float* lse, void* workspace, size_t workspace_bytes,
                            int dtype, int32_t* dev_status, void* stream) {
  const KvFormat kv = opts && opts->fp8 ? fp8_format(opts->fp8) : kKvBf16;
  return cascade_impl(update, q, q_token_stride, key_cache, value_cache, cache_block_stride,
                      cu_seqlens_q, seqused_k, block_table, bt_stride, num_seqs, total_q,
                      max_seqlen_q, max_seqlen_k, num_heads, num_kv_heads, head_size, block_size,
                      num_blocks, softmax_scale, common_prefix_len, out, lse, workspace,
                      workspace_bytes, dtype, dev_status, stream, kv,
                      opts ? opts->sinks : nullptr);
}

}  // extern "C"
