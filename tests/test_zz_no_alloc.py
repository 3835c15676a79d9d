"""pa_varlen_fwd_noalloc: the entry point for callers that cannot allocate
device memory (and so cannot pass a workspace), e.g. an engine whose allocator
has reserved all device memory for its page pool. Its scratch is the
library's fixed 32 MiB device buffer. Checked through the C ABI against
pa_varlen_fwd with a caller workspace, on two calls in a row (the buffer keeps
the previous call's contents). Both entry points run the same kernels on the
same plan, only the scratch address differs, so the outputs must agree bit for
bit (which implies the parity tolerances of the other tests).

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test."""
import ctypes

import pytest
import torch

import paged_kv_varlen_attn_gb300 as pa
import workloads as W
from helpers import to_dev

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_varlen_attn_gb300 import _build
    _build.build()
    return pa.load_library()


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _call_noalloc(lib, wl, d, out, lse):
    T, H, D = wl.q.shape
    kc = d["key_cache"]
    return lib.pa_varlen_fwd_noalloc(
        _p(d["q"]), d["q"].stride(0), _p(kc), _p(d["value_cache"]), kc.stride(0),
        _p(d["cu_seqlens_q"]), _p(d["seqused_k"]), _p(d["block_table"]),
        d["block_table"].stride(0), wl.num_seqs, T, wl.max_seqlen_q, wl.max_seqlen_k, H,
        wl.num_kv_heads, D, wl.block_size, wl.num_blocks, wl.softmax_scale, int(wl.causal),
        _p(out), _p(lse), pa.PA_BF16, None,
        ctypes.c_void_p(torch.cuda.current_stream(DEV).cuda_stream))


@pytest.mark.parametrize("make", [
    lambda: W.decode_llama8b(num_seqs=16),                  # decode: split-KV kernel
    lambda: W._build("noalloc_mixed", 301, 8, 4, 64, 16, [1, 3, 40, 1], [682, 80, 628, 584],
                     torch.Generator().manual_seed(301)),       # both kernels (40 x 2 rows > 64)
], ids=["decode", "mixed"])
def test_noalloc_matches_workspace_call_twice(lib, make):
    wl = make()
    d = to_dev(wl, DEV)
    pa.reshape_and_cache(d["k_new"], d["v_new"], d["key_cache"], d["value_cache"],
                         d["slot_mapping"])
    ref_o, ref_l = pa.varlen_fwd(d["q"], d["key_cache"], d["value_cache"], d["cu_seqlens_q"],
                                 d["seqused_k"], d["block_table"], wl.max_seqlen_q,
                                 wl.max_seqlen_k, wl.softmax_scale, wl.causal)
    T, H, D = wl.q.shape
    for _ in range(2):
        out = torch.full((T, H, D), float("nan"), dtype=torch.bfloat16, device=DEV)
        lse = torch.full((H, T), float("nan"), dtype=torch.float32, device=DEV)
        assert _call_noalloc(lib, wl, d, out, lse) == pa.PA_OK
        torch.cuda.synchronize()
        assert torch.equal(out, ref_o)
        # bitwise, -inf rows included (a NaN would fail this too)
        assert torch.equal(lse.view(torch.int32), ref_l.view(torch.int32))


def test_noalloc_rejects_problems_beyond_its_buffer(lib):
    need = pa.varlen_fwd_workspace_size(4096, 4096 * 16, 16, 8192, 32, 8, 128, 16, 0)
    assert need > pa.NOALLOC_SCRATCH_BYTES
    wl = W.decode_llama8b(num_seqs=2)
    d = to_dev(wl, DEV)
    T, H, D = wl.q.shape
    out = torch.empty((T, H, D), dtype=torch.bfloat16, device=DEV)
    # Same tensors, but bounds (and batch shape) that need more scratch than the
    # buffer holds: refused on the host before any launch.
    code = lib.pa_varlen_fwd_noalloc(
        _p(d["q"]), d["q"].stride(0), _p(d["key_cache"]), _p(d["value_cache"]),
        d["key_cache"].stride(0), _p(d["cu_seqlens_q"]), _p(d["seqused_k"]),
        _p(d["block_table"]), d["block_table"].stride(0), 4096, 4096 * 16, 16, 8192, H,
        wl.num_kv_heads, D, wl.block_size, wl.num_blocks, wl.softmax_scale, 1, _p(out), None,
        pa.PA_BF16, None, ctypes.c_void_p(torch.cuda.current_stream(DEV).cuda_stream))
    assert code == pa.PA_ERR_NOALLOC_LIMIT
    assert b"no-allocation" in lib.pa_status_string(code)
