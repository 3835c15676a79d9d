"""Python binding of libpa.so: paged varlen attention for GB300 (sm_103a).

Thin ctypes marshalling over the C ABI in include/pa.h. Torch is used for
device memory (outputs and workspaces are allocated here, on the caller's
side of the ABI) and for the current CUDA stream; every step of the
computation runs in the library's CUDA kernels. There is no CPU fallback: the
functions raise if the library or a GPU is missing.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libpa.so")

PA_OK = 0
PA_ERR_INVALID_ARG = 1
PA_ERR_BLOCK_SIZE = 2
PA_ERR_UNSUPPORTED = 3
PA_ERR_WORKSPACE = 4
PA_ERR_CUDA = 5
PA_ERR_NOALLOC_LIMIT = 6
NOALLOC_SCRATCH_BYTES = 32 << 20
PA_DEV_BAD_PAGE = 1
PA_DEV_BAD_SLOT = 2
PA_DEV_BAD_SEQLEN = 4
PA_DEV_TIMEOUT = 8
PA_DEV_CASCADE = 16
PA_BF16 = 0
PA_F16 = 1

EXPORTS = (
    "pa_status_string",
    "pa_abi_version",
    "pa_reshape_and_cache",
    "pa_varlen_fwd_workspace_size",
    "pa_varlen_fwd",
    "pa_merge_attn_states",
    "pa_cascade_fwd_workspace_size",
    "pa_cascade_fwd",
    "pa_varlen_fwd_noalloc",
    "pa_varlen_fwd_with_update",
    "pa_cascade_fwd_with_update",
    "pa_use_cascade_attention",
    "pa_reshape_and_cache_fp8",
    "pa_varlen_fwd_fp8kv_workspace_size",
    "pa_cascade_fwd_fp8kv_workspace_size",
    "pa_varlen_fwd_fp8kv",
    "pa_cascade_fwd_fp8kv",
    "pa_merge_attn_states_n",
    "pa_varlen_fwd_ex",
    "pa_cascade_fwd_ex",
)

_lib = None

_c = ctypes
_vp, _i64, _i32, _f32, _sz = _c.c_void_p, _c.c_int64, _c.c_int, _c.c_float, _c.c_size_t


class KvUpdate(ctypes.Structure):
    """struct pa_kv_update of include/pa.h."""
    _fields_ = [("key", _vp), ("value", _vp), ("key_token_stride", _i64),
                ("value_token_stride", _i64), ("slot_mapping", _vp), ("num_tokens", _i32)]


class KvFp8(ctypes.Structure):
    """struct pa_kv_fp8 of include/pa.h (device float32 [num_kv_heads] scales)."""
    _fields_ = [("k_scale", _vp), ("v_scale", _vp)]


class AttnOpts(ctypes.Structure):
    """struct pa_attn_opts of include/pa.h."""
    _fields_ = [("sinks", _vp), ("fp8", ctypes.POINTER(KvFp8))]


_ATTN_ARGS = [_vp, _i64, _vp, _vp, _i64, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i32, _i32,
              _i32, _i32, _i32, _f32, _i32, _vp, _vp, _vp, _sz, _i32, _vp, _vp]

_SIGS = {
    "pa_status_string": ([_i32], _c.c_char_p),
    "pa_abi_version": ([], _i32),
    "pa_reshape_and_cache": ([_vp, _vp, _i64, _i64, _vp, _vp, _i64, _vp, _i32, _i32, _i32, _i32,
                              _i32, _i32, _vp, _vp], _i32),
    "pa_varlen_fwd_workspace_size": ([_i32] * 9, _sz),
    "pa_varlen_fwd": ([_vp, _i64, _vp, _vp, _i64, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32,
                       _i32, _i32, _i32, _i32, _i32, _f32, _i32, _vp, _vp, _vp, _sz, _i32, _vp,
                       _vp], _i32),
    "pa_merge_attn_states": ([_vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _vp], _i32),
    "pa_cascade_fwd_workspace_size": ([_i32] * 9, _sz),
    "pa_varlen_fwd_noalloc": ([_vp, _i64, _vp, _vp, _i64, _vp, _vp, _vp, _i32, _i32, _i32, _i32,
                               _i32, _i32, _i32, _i32, _i32, _i32, _f32, _i32, _vp, _vp, _i32, _vp,
                               _vp], _i32),
    "pa_cascade_fwd": ([_vp, _i64, _vp, _vp, _i64, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32,
                        _i32, _i32, _i32, _i32, _i32, _f32, _i32, _vp, _vp, _vp, _sz, _i32, _vp,
                        _vp], _i32),
    "pa_varlen_fwd_with_update": ([ctypes.POINTER(KvUpdate)] + _ATTN_ARGS, _i32),
    "pa_cascade_fwd_with_update": ([ctypes.POINTER(KvUpdate)] + _ATTN_ARGS, _i32),
    "pa_use_cascade_attention": ([_i32, _i32, _i32, _i32, _i32, ctypes.POINTER(_i32)], _i32),
    "pa_reshape_and_cache_fp8": ([_vp, _vp, _i64, _i64, _vp, _vp, _i64, _vp, _i32, _i32, _i32,
                                  _i32, _i32, ctypes.POINTER(KvFp8), _i32, _vp, _vp], _i32),
    "pa_varlen_fwd_fp8kv_workspace_size": ([_i32] * 9, _sz),
    "pa_merge_attn_states_n": ([_vp, _vp, _vp, _i64, _vp, _i64, _i32, _i32, _i32, _i32, _i32, _vp],
                               _i32),
    "pa_varlen_fwd_ex": ([ctypes.POINTER(KvUpdate)] + _ATTN_ARGS[:20] +
                         [ctypes.POINTER(AttnOpts)] + _ATTN_ARGS[20:], _i32),
    "pa_cascade_fwd_ex": ([ctypes.POINTER(KvUpdate)] + _ATTN_ARGS[:20] +
                          [ctypes.POINTER(AttnOpts)] + _ATTN_ARGS[20:], _i32),
    "pa_cascade_fwd_fp8kv_workspace_size": ([_i32] * 9, _sz),
    "pa_varlen_fwd_fp8kv": ([ctypes.POINTER(KvUpdate)] + _ATTN_ARGS[:20] +
                            [ctypes.POINTER(KvFp8)] + _ATTN_ARGS[20:], _i32),
    "pa_cascade_fwd_fp8kv": ([ctypes.POINTER(KvUpdate)] + _ATTN_ARGS[:20] +
                             [ctypes.POINTER(KvFp8)] + _ATTN_ARGS[20:], _i32),
}


def load_library(path: str = LIB_PATH):
    """Load libpa.so (built by ``_build.build()``) and declare its signatures."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"libpa.so not built ({path}); run __graft_entry__.build() "
                           "or python paged_kv_varlen_attn_gb300/_build.py")
    lib = ctypes.CDLL(path)
    for name, (args, res) in _SIGS.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _lib = lib
    return lib


class PAError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        msg = load_library().pa_status_string(code).decode()
        super().__init__(f"{where}: {msg}")


def _check(code: int, where: str):
    if code != PA_OK:
        raise PAError(code, where)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _need_cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("all tensors must be CUDA tensors (no CPU fallback)")


def _dtype_code(*ts):
    """PA_BF16 or PA_F16 for tensors that must all share one 2-byte float type."""
    dts = {t.dtype for t in ts if t is not None}
    if len(dts) != 1:
        raise ValueError(f"tensors must share one element type, got {sorted(map(str, dts))}")
    dt = dts.pop()
    if dt == torch.bfloat16:
        return PA_BF16
    if dt == torch.float16:
        return PA_F16
    raise ValueError(f"unsupported element type {dt} (bfloat16 or float16)")


def _sm_count(device) -> int:
    return torch.cuda.get_device_properties(device).multi_processor_count


def _row_stride(t):
    """Token stride of a [T, heads, D] tensor whose [heads, D] rows are contiguous."""
    if t.dim() != 3 or t.stride(2) != 1 or t.stride(1) != t.shape[2]:
        raise ValueError("tensor must be [tokens, heads, head_size] with contiguous rows")
    return t.stride(0)


def _cache_stride(c):
    if c.dim() != 4 or c.stride(3) != 1 or c.stride(2) != c.shape[3] or \
            c.stride(1) != c.shape[2] * c.shape[3]:
        raise ValueError("cache must be [num_blocks, block_size, num_kv_heads, head_size] with "
                         "contiguous pages")
    return c.stride(0)


# ---------------------------------------------------------------------------
def reshape_and_cache(key, value, key_cache, value_cache, slot_mapping, dev_status=None):
    """Scatter new K/V rows into their pages (in place on the caches)."""
    lib = load_library()
    _need_cuda(key, value, key_cache, value_cache, slot_mapping, dev_status)
    if key_cache.stride(0) != value_cache.stride(0):
        raise ValueError("key and value caches must share the page stride")
    nb, bs, hk, d = key_cache.shape
    dtype = _dtype_code(key, value, key_cache, value_cache)
    code = lib.pa_reshape_and_cache(
        _ptr(key), _ptr(value), _row_stride(key), _row_stride(value), _ptr(key_cache),
        _ptr(value_cache), _cache_stride(key_cache), _ptr(slot_mapping), key.shape[0], hk, d, bs,
        nb, dtype, _ptr(dev_status), _stream(key.device))
    _check(code, "pa_reshape_and_cache")


def varlen_fwd_workspace_size(num_seqs, total_q, max_seqlen_q, max_seqlen_k, num_heads,
                              num_kv_heads, head_size, block_size, sm_count):
    return load_library().pa_varlen_fwd_workspace_size(
        num_seqs, total_q, max_seqlen_q, max_seqlen_k, num_heads, num_kv_heads, head_size,
        block_size, sm_count)


def cascade_fwd_workspace_size(num_seqs, total_q, max_seqlen_q, max_seqlen_k, num_heads,
                               num_kv_heads, head_size, block_size, sm_count):
    return load_library().pa_cascade_fwd_workspace_size(
        num_seqs, total_q, max_seqlen_q, max_seqlen_k, num_heads, num_kv_heads, head_size,
        block_size, sm_count)


def use_cascade_attention(common_prefix_len, num_seqs, num_kv_heads, head_size, split_kv=True):
    """Whether a batch whose sequences share common_prefix_len tokens should
    run as cascade attention (host-side policy, no GPU needed)."""
    out = _i32(0)
    _check(load_library().pa_use_cascade_attention(int(common_prefix_len), int(num_seqs),
                                                   int(num_kv_heads), int(head_size),
                                                   int(bool(split_kv)), ctypes.byref(out)),
           "pa_use_cascade_attention")
    return bool(out.value)


def alloc_workspace(nbytes, device):
    # 256-byte aligned (the caching allocator aligns to 512 bytes).
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def _attn_common(q, key_cache, value_cache, cu_seqlens_q, seqused_k, block_table):
    _need_cuda(q, key_cache, value_cache, cu_seqlens_q, seqused_k, block_table)
    if key_cache.stride(0) != value_cache.stride(0) or key_cache.shape != value_cache.shape:
        raise ValueError("key and value caches must have the same shape and page stride")
    for t, name in ((cu_seqlens_q, "cu_seqlens_q"), (seqused_k, "seqused_k"),
                    (block_table, "block_table")):
        if t.dtype != torch.int32:
            raise ValueError(f"{name} must be int32")
    if block_table.dim() != 2 or block_table.stride(1) != 1:
        raise ValueError("block_table must be [num_seqs, max_blocks] with unit column stride")


def _kv_update(key, value, slot_mapping):
    if key is None:
        return None
    _need_cuda(key, value, slot_mapping)
    return KvUpdate(key.data_ptr(), value.data_ptr(), _row_stride(key), _row_stride(value),
                    slot_mapping.data_ptr(), key.shape[0])


def _attend(entry, update, q, key_cache, value_cache, cu_seqlens_q, seqused_k, block_table,
            max_seqlen_q, max_seqlen_k, softmax_scale, mode_arg, out, lse, return_lse,
            workspace, dev_status, size_fn, fp8=None, sinks=None, update_tensors=None):
    lib = load_library()
    _attn_common(q, key_cache, value_cache, cu_seqlens_q, seqused_k, block_table)
    T, H, D = q.shape
    nb, bs, hk, _ = key_cache.shape
    S = cu_seqlens_q.numel() - 1
    if out is None:
        out = torch.empty((T, H, D), dtype=q.dtype, device=q.device)
    # q, out, the new tokens and (unless they hold e4m3 bytes) the pools share the type
    pools = () if fp8 is not None else (key_cache, value_cache)
    dtype = _dtype_code(q, out, *pools, *((update_tensors or ()) if update is not None else ()))
    if lse is None and return_lse:
        lse = torch.empty((H, T), dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = alloc_workspace(size_fn(S, T, max_seqlen_q, max_seqlen_k, H, hk, D, bs,
                                            _sm_count(q.device)), q.device)
    args = (_ptr(q), _row_stride(q), _ptr(key_cache), _ptr(value_cache), _cache_stride(key_cache),
            _ptr(cu_seqlens_q), _ptr(seqused_k), _ptr(block_table), block_table.stride(0), S, T,
            int(max_seqlen_q), int(max_seqlen_k), H, hk, D, bs, nb, float(softmax_scale),
            int(mode_arg)) + ((ctypes.byref(fp8),) if fp8 is not None else ()) + (
            _ptr(out), _ptr(lse), _ptr(workspace), workspace.numel(), dtype,
            _ptr(dev_status), _stream(q.device))
    upd = ctypes.byref(update) if update is not None else None
    if sinks is not None:
        # Options (attention sinks) go through the _ex entry points.
        _need_cuda(sinks)
        if sinks.dtype != torch.float32 or sinks.shape != (H,) or not sinks.is_contiguous():
            raise ValueError("sinks must be a contiguous float32 tensor of num_heads values")
        opts = AttnOpts(sinks.data_ptr(), ctypes.pointer(fp8) if fp8 is not None else None)
        entry = "pa_varlen_fwd_ex" if entry.startswith("pa_varlen") else "pa_cascade_fwd_ex"
        if fp8 is not None:
            args = args[:20] + args[21:]          # the descriptor travels in opts
        code = getattr(lib, entry)(upd, *args[:20], ctypes.byref(opts), *args[20:])
        _check(code, entry)
        return out, lse
    fn = getattr(lib, entry)
    code = fn(upd, *args) if entry.endswith(("_with_update", "_fp8kv")) else fn(*args)
    _check(code, entry)
    return out, lse


def varlen_fwd(q, key_cache, value_cache, cu_seqlens_q, seqused_k, block_table, max_seqlen_q,
               max_seqlen_k, softmax_scale, causal, out=None, lse=None, return_lse=True,
               workspace=None, dev_status=None, sinks=None):
    """Varlen attention over a paged KV cache. Returns (out, lse or None)."""
    return _attend("pa_varlen_fwd", None, q, key_cache, value_cache, cu_seqlens_q, seqused_k,
                   block_table, max_seqlen_q, max_seqlen_k, softmax_scale, bool(causal), out,
                   lse, return_lse, workspace, dev_status, varlen_fwd_workspace_size, sinks=sinks)


def varlen_fwd_with_update(key, value, slot_mapping, q, key_cache, value_cache, cu_seqlens_q,
                           seqused_k, block_table, max_seqlen_q, max_seqlen_k, softmax_scale,
                           causal, out=None, lse=None, return_lse=True, workspace=None,
                           dev_status=None, sinks=None):
    """One step: scatter the new tokens' K/V (key, value by slot_mapping) into
    the caches, then varlen attention; the planner overlaps the scatter.
    Returns (out, lse or None)."""
    return _attend("pa_varlen_fwd_with_update", _kv_update(key, value, slot_mapping), q,
                   key_cache, value_cache, cu_seqlens_q, seqused_k, block_table, max_seqlen_q,
                   max_seqlen_k, softmax_scale, bool(causal), out, lse, return_lse, workspace,
                   dev_status, varlen_fwd_workspace_size, sinks=sinks,
                   update_tensors=(key, value))


def varlen_fwd_noalloc(q, key_cache, value_cache, cu_seqlens_q, seqused_k, block_table,
                       max_seqlen_q, max_seqlen_k, softmax_scale, causal, out=None, lse=None,
                       return_lse=True, dev_status=None):
    """varlen_fwd without a workspace: the library's fixed 32 MiB scratch is
    used instead (for callers that cannot allocate device memory). Calls that
    overlap on the GPU race on that buffer. Returns (out, lse or None)."""
    lib = load_library()
    _attn_common(q, key_cache, value_cache, cu_seqlens_q, seqused_k, block_table)
    T, H, D = q.shape
    nb, bs, hk, _ = key_cache.shape
    S = cu_seqlens_q.numel() - 1
    if out is None:
        out = torch.empty((T, H, D), dtype=q.dtype, device=q.device)
    if lse is None and return_lse:
        lse = torch.empty((H, T), dtype=torch.float32, device=q.device)
    code = lib.pa_varlen_fwd_noalloc(
        _ptr(q), _row_stride(q), _ptr(key_cache), _ptr(value_cache), _cache_stride(key_cache),
        _ptr(cu_seqlens_q), _ptr(seqused_k), _ptr(block_table), block_table.stride(0), S, T,
        int(max_seqlen_q), int(max_seqlen_k), H, hk, D, bs, nb, float(softmax_scale),
        int(bool(causal)), _ptr(out), _ptr(lse), _dtype_code(q, out, key_cache, value_cache),
        _ptr(dev_status), _stream(q.device))
    _check(code, "pa_varlen_fwd_noalloc")
    return out, lse


def merge_attn_states(prefix_out, prefix_lse, suffix_out, suffix_lse, out=None, out_lse=None,
                      return_lse=True):
    """LSE-weighted combine of two partial attention states. Returns (out, lse or None)."""
    lib = load_library()
    _need_cuda(prefix_out, prefix_lse, suffix_out, suffix_lse)
    T, H, D = prefix_out.shape
    for t in (prefix_out, suffix_out):
        if not t.is_contiguous():
            raise ValueError("outputs must be contiguous [tokens, heads, head_size]")
    if out is None:
        out = torch.empty_like(prefix_out)
    if out_lse is None and return_lse:
        out_lse = torch.empty((H, T), dtype=torch.float32, device=prefix_out.device)
    code = lib.pa_merge_attn_states(
        _ptr(out), _ptr(out_lse), _ptr(prefix_out), _ptr(prefix_lse), _ptr(suffix_out),
        _ptr(suffix_lse), T, H, D, _dtype_code(prefix_out, suffix_out, out),
        _stream(prefix_out.device))
    _check(code, "pa_merge_attn_states")
    return out, out_lse


def merge_attn_states_n(parts_out, parts_lse, out=None, out_lse=None, return_lse=True):
    """LSE-weighted combine of n partial states: parts_out [n, T, H, D] bf16
    (each part contiguous), parts_lse [n, H, T] float32. Returns (out, lse or None)."""
    lib = load_library()
    _need_cuda(parts_out, parts_lse)
    n, T, H, D = parts_out.shape
    if parts_out[0].numel() and not parts_out[0].is_contiguous():
        raise ValueError("each part must be a contiguous [tokens, heads, head_size] tensor")
    if parts_lse.shape != (n, H, T) or (T and parts_lse.stride(2) != 1) or \
            (T and parts_lse.stride(1) != T):
        raise ValueError("parts_lse must be [n, heads, tokens] with contiguous parts")
    if out is None:
        out = torch.empty((T, H, D), dtype=parts_out.dtype, device=parts_out.device)
    if out_lse is None and return_lse:
        out_lse = torch.empty((H, T), dtype=torch.float32, device=parts_out.device)
    code = lib.pa_merge_attn_states_n(
        _ptr(out), _ptr(out_lse), _ptr(parts_out), parts_out.stride(0), _ptr(parts_lse),
        parts_lse.stride(0), n, T, H, D, _dtype_code(parts_out, out), _stream(parts_out.device))
    _check(code, "pa_merge_attn_states_n")
    return out, out_lse


def cascade_fwd(q, key_cache, value_cache, cu_seqlens_q, seqused_k, block_table, max_seqlen_q,
                max_seqlen_k, softmax_scale, common_prefix_len, out=None, lse=None,
                return_lse=True, workspace=None, dev_status=None, sinks=None):
    """Shared-prefix (cascade) attention. Returns (out, lse or None)."""
    return _attend("pa_cascade_fwd", None, q, key_cache, value_cache, cu_seqlens_q, seqused_k,
                   block_table, max_seqlen_q, max_seqlen_k, softmax_scale, common_prefix_len,
                   out, lse, return_lse, workspace, dev_status, cascade_fwd_workspace_size, sinks=sinks)


def cascade_fwd_with_update(key, value, slot_mapping, q, key_cache, value_cache, cu_seqlens_q,
                            seqused_k, block_table, max_seqlen_q, max_seqlen_k, softmax_scale,
                            common_prefix_len, out=None, lse=None, return_lse=True,
                            workspace=None, dev_status=None, sinks=None):
    """One step: scatter the new tokens' K/V into the caches, then cascade
    attention. Returns (out, lse or None)."""
    return _attend("pa_cascade_fwd_with_update", _kv_update(key, value, slot_mapping), q,
                   key_cache, value_cache, cu_seqlens_q, seqused_k, block_table, max_seqlen_q,
                   max_seqlen_k, softmax_scale, common_prefix_len, out, lse, return_lse,
                   workspace, dev_status, cascade_fwd_workspace_size, sinks=sinks,
                   update_tensors=(key, value))


# ---------------------------------------------------------------------------
# FP8 (e4m3) KV cache: uint8 (or float8_e4m3fn) pools of e4m3 codes with one
# scale per KV head; a stored code c means e4m3(c) * scale.
def _fp8_pool(c):
    if c.element_size() != 1:
        raise ValueError("FP8 caches hold one byte per element (uint8 or float8_e4m3fn)")
    return c


def _scales(s, hk, device):
    """Per-KV-head float32 scales on the device: a number, or a tensor of 1 or
    num_kv_heads values."""
    if not torch.is_tensor(s):
        return torch.full((hk,), float(s), dtype=torch.float32, device=device)
    s = s.to(device=device, dtype=torch.float32).reshape(-1)
    if s.numel() == 1:
        s = s.expand(hk)
    if s.numel() != hk:
        raise ValueError(f"expected 1 or {hk} scales, got {s.numel()}")
    return s.contiguous()


def _fp8_desc(k_scale, v_scale, hk, device):
    ks, vs = _scales(k_scale, hk, device), _scales(v_scale, hk, device)
    return KvFp8(ks.data_ptr(), vs.data_ptr()), (ks, vs)


def varlen_fwd_fp8kv_workspace_size(num_seqs, total_q, max_seqlen_q, max_seqlen_k, num_heads,
                                    num_kv_heads, head_size, block_size, sm_count):
    return load_library().pa_varlen_fwd_fp8kv_workspace_size(
        num_seqs, total_q, max_seqlen_q, max_seqlen_k, num_heads, num_kv_heads, head_size,
        block_size, sm_count)


def cascade_fwd_fp8kv_workspace_size(num_seqs, total_q, max_seqlen_q, max_seqlen_k, num_heads,
                                     num_kv_heads, head_size, block_size, sm_count):
    return load_library().pa_cascade_fwd_fp8kv_workspace_size(
        num_seqs, total_q, max_seqlen_q, max_seqlen_k, num_heads, num_kv_heads, head_size,
        block_size, sm_count)


def reshape_and_cache_fp8(key, value, key_cache, value_cache, slot_mapping, k_scale, v_scale,
                          dev_status=None):
    """Quantize new bf16 K/V rows to e4m3 (x / scale of their KV head) and
    scatter them into the FP8 pools (in place)."""
    lib = load_library()
    _need_cuda(key, value, key_cache, value_cache, slot_mapping, dev_status)
    _fp8_pool(key_cache), _fp8_pool(value_cache)
    if key_cache.stride(0) != value_cache.stride(0):
        raise ValueError("key and value caches must share the page stride")
    nb, bs, hk, d = key_cache.shape
    desc, keep = _fp8_desc(k_scale, v_scale, hk, key.device)
    code = lib.pa_reshape_and_cache_fp8(
        _ptr(key), _ptr(value), _row_stride(key), _row_stride(value), _ptr(key_cache),
        _ptr(value_cache), _cache_stride(key_cache), _ptr(slot_mapping), key.shape[0], hk, d, bs,
        nb, ctypes.byref(desc), _dtype_code(key, value), _ptr(dev_status), _stream(key.device))
    _check(code, "pa_reshape_and_cache_fp8")
    del keep


def varlen_fwd_fp8kv(q, key_cache, value_cache, cu_seqlens_q, seqused_k, block_table,
                     max_seqlen_q, max_seqlen_k, softmax_scale, causal, k_scale, v_scale,
                     key=None, value=None, slot_mapping=None, out=None, lse=None,
                     return_lse=True, workspace=None, dev_status=None, sinks=None):
    """Varlen attention over FP8 pools, optionally first quantizing and
    scattering the new tokens' K/V (key, value, slot_mapping). Returns
    (out, lse or None)."""
    _fp8_pool(key_cache), _fp8_pool(value_cache)
    desc, keep = _fp8_desc(k_scale, v_scale, key_cache.shape[2], q.device)
    res = _attend("pa_varlen_fwd_fp8kv", _kv_update(key, value, slot_mapping), q, key_cache,
                  value_cache, cu_seqlens_q, seqused_k, block_table, max_seqlen_q, max_seqlen_k,
                  softmax_scale, bool(causal), out, lse, return_lse, workspace, dev_status,
                  varlen_fwd_fp8kv_workspace_size, fp8=desc, sinks=sinks,
                  update_tensors=(key, value))
    del keep
    return res


def cascade_fwd_fp8kv(q, key_cache, value_cache, cu_seqlens_q, seqused_k, block_table,
                      max_seqlen_q, max_seqlen_k, softmax_scale, common_prefix_len, k_scale,
                      v_scale, key=None, value=None, slot_mapping=None, out=None, lse=None,
                      return_lse=True, workspace=None, dev_status=None, sinks=None):
    """Cascade attention over FP8 pools (optional update as in
    varlen_fwd_fp8kv). Returns (out, lse or None)."""
    _fp8_pool(key_cache), _fp8_pool(value_cache)
    desc, keep = _fp8_desc(k_scale, v_scale, key_cache.shape[2], q.device)
    res = _attend("pa_cascade_fwd_fp8kv", _kv_update(key, value, slot_mapping), q, key_cache,
                  value_cache, cu_seqlens_q, seqused_k, block_table, max_seqlen_q, max_seqlen_k,
                  softmax_scale, common_prefix_len, out, lse, return_lse, workspace, dev_status,
                  cascade_fwd_fp8kv_workspace_size, fp8=desc, sinks=sinks,
                  update_tensors=(key, value))
    del keep
    return res
