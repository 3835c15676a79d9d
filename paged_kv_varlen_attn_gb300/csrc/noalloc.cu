// pa_varlen_fwd_noalloc: pa_varlen_fwd with its scratch in a fixed,
// library-owned device buffer instead of a caller workspace, for callers that
// cannot allocate device memory (see include/pa.h).
#include <cuda_runtime.h>

#include <mutex>

#include "pa.h"

namespace {

// The scratch. Every GPU that loads this library holds it until exit. In
// host code the name is only a host-side handle: its device address comes
// from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char pa_noalloc_scratch[PA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
// Per device: the context the address was looked up in, and the address.
// cudaDeviceReset destroys the device's primary context and the module with
// the buffer; the next call then runs in a new context and looks it up again.
void* g_ctx[kMaxDevices] = {};
void* g_ptr[kMaxDevices] = {};

// cuCtxGetCurrent through the runtime's driver entry point (no link
// dependency on libcuda). Returns nullptr if unavailable.
using CtxGetCurrentFn = int (*)(void**);
CtxGetCurrentFn ctx_get_current() {
  static CtxGetCurrentFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(p);
  });
  return fn;
}

// Device address of the scratch on the current device, looked up once per
// device and context with that device current. Returns nullptr on failure,
// leaving no CUDA error pending.
void* scratch_on_current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return nullptr;
  }
  // The context the call's kernels will run in (null before the runtime has
  // made one current on this thread; the symbol lookup below does that).
  CtxGetCurrentFn get = ctx_get_current();
  if (!get) return nullptr;
  void* ctx = nullptr;
  if (get(&ctx) != 0) return nullptr;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!ctx || !g_ptr[dev] || g_ctx[dev] != ctx) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, pa_noalloc_scratch) != cudaSuccess) {
      cudaGetLastError();   // clear it, so a later launch check does not report it
      g_ptr[dev] = nullptr;
      return nullptr;
    }
    if (get(&ctx) != 0 || !ctx) return nullptr;
    g_ptr[dev] = p;
    g_ctx[dev] = ctx;
  }
  return g_ptr[dev];
}

}  // namespace

extern "C" pa_status pa_varlen_fwd_noalloc(
    const void* q, int64_t q_token_stride, const void* key_cache, const void* value_cache,
    int64_t cache_block_stride, const int32_t* cu_seqlens_q, const int32_t* seqused_k,
    const int32_t* block_table, int bt_stride, int num_seqs, int total_q, int max_seqlen_q,
    int max_seqlen_k, int num_heads, int num_kv_heads, int head_size, int block_size,
    int num_blocks, float softmax_scale, int causal, void* out, float* lse, int dtype,
    int32_t* dev_status, void* stream) {
  // Argument checks first, exactly as pa_varlen_fwd does them: with no
  // workspace it returns PA_ERR_WORKSPACE only when everything else is valid
  // (and PA_OK, launching nothing, for an empty batch).
  pa_status st = pa_varlen_fwd(q, q_token_stride, key_cache, value_cache, cache_block_stride,
                               cu_seqlens_q, seqused_k, block_table, bt_stride, num_seqs, total_q,
                               max_seqlen_q, max_seqlen_k, num_heads, num_kv_heads, head_size,
                               block_size, num_blocks, softmax_scale, causal, out, lse, nullptr, 0,
                               dtype, dev_status, stream);
  if (st != PA_ERR_WORKSPACE) return st;
  const size_t need = pa_varlen_fwd_workspace_size(num_seqs, total_q, max_seqlen_q, max_seqlen_k,
                                                   num_heads, num_kv_heads, head_size, block_size,
                                                   0);
  if (need == 0) return PA_ERR_CUDA;
  if (need > PA_NOALLOC_SCRATCH_BYTES) return PA_ERR_NOALLOC_LIMIT;
  void* scratch = scratch_on_current_device();
  if (!scratch) return PA_ERR_CUDA;
  return pa_varlen_fwd(q, q_token_stride, key_cache, value_cache, cache_block_stride,
                       cu_seqlens_q, seqused_k, block_table, bt_stride, num_seqs, total_q,
                       max_seqlen_q, max_seqlen_k, num_heads, num_kv_heads, head_size,
                       block_size, num_blocks, softmax_scale, causal, out, lse, scratch,
                       PA_NOALLOC_SCRATCH_BYTES, dtype, dev_status, stream);
}
