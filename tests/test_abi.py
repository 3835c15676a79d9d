"""C-ABI checks that need no GPU: the library loads, exports every function
include/pa.h declares, and rejects invalid arguments on the host before any
CUDA call (the pages' ValueError for a block size that is not a multiple of
16, head-size and dtype limits -- "FlashAttention と FlashInfer" 境界と失敗,
"AttentionBackend" 境界と失敗)."""
import ctypes
import os
import re

import pytest

import paged_kv_varlen_attn_gb300 as pa
from paged_kv_varlen_attn_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pa.h")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return pa.load_library()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_four_operations():
    names = declared_functions()
    for op in ("pa_reshape_and_cache", "pa_varlen_fwd", "pa_merge_attn_states", "pa_cascade_fwd"):
        assert op in names


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert names, "no declarations parsed"
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) <= set(pa.EXPORTS) | set(names)
    assert set(pa.EXPORTS) == set(names)


def test_abi_version_and_status_strings(lib):
    assert lib.pa_abi_version() == 1
    assert lib.pa_status_string(0) == b"PA_OK"
    assert b"multiple of 16" in lib.pa_status_string(pa.PA_ERR_BLOCK_SIZE)
    assert lib.pa_status_string(99) == b"PA_ERR_UNKNOWN"


def test_workspace_size_pure_host(lib):
    n = lib.pa_varlen_fwd_workspace_size(64, 64, 1, 8192, 32, 8, 128, 16, 152)
    assert n > 0 and n % 256 == 0
    # grows with the batch, and cascade needs more than plain varlen
    assert lib.pa_varlen_fwd_workspace_size(128, 128, 1, 8192, 32, 8, 128, 16, 152) > n
    assert lib.pa_cascade_fwd_workspace_size(64, 64, 1, 8192, 32, 8, 128, 16, 152) > n
    # invalid shapes give 0
    assert lib.pa_varlen_fwd_workspace_size(64, 64, 1, 8192, 32, 7, 128, 16, 152) == 0
    assert lib.pa_varlen_fwd_workspace_size(64, 64, 1, 8192, 32, 8, 96, 16, 152) == 0
    assert lib.pa_varlen_fwd_workspace_size(64, 64, 1, 8192, 32, 8, 128, 24, 152) == 0


FAKE = 0x10000  # 16-byte aligned, never dereferenced: validation fails first


def _varlen(lib, **kw):
    a = dict(q=FAKE, qs=32 * 128, kc=FAKE, vc=FAKE, cbs=16 * 8 * 128, cu=FAKE, lens=FAKE,
             bt=FAKE, bts=4, S=2, T=2, mq=1, mk=64, H=32, Hk=8, D=128, bs=16, nb=10,
             scale=0.088, causal=1, out=FAKE, lse=None, ws=FAKE, wsb=1 << 20, dtype=0)
    a.update(kw)
    return lib.pa_varlen_fwd(a["q"], a["qs"], a["kc"], a["vc"], a["cbs"], a["cu"], a["lens"],
                             a["bt"], a["bts"], a["S"], a["T"], a["mq"], a["mk"], a["H"], a["Hk"],
                             a["D"], a["bs"], a["nb"], a["scale"], a["causal"], a["out"], a["lse"],
                             a["ws"], a["wsb"], a["dtype"], None, None)


@pytest.mark.parametrize("kw,code", [
    (dict(bs=24), pa.PA_ERR_BLOCK_SIZE),
    (dict(bs=0), pa.PA_ERR_BLOCK_SIZE),
    (dict(bs=2048), pa.PA_ERR_BLOCK_SIZE),
    (dict(D=96), pa.PA_ERR_UNSUPPORTED),
    (dict(D=512), pa.PA_ERR_UNSUPPORTED),
    (dict(D=256, qs=32 * 256, cbs=16 * 8 * 256, scale=-0.1),
     pa.PA_ERR_UNSUPPORTED),                            # D 256 runs on the prefill kernel only,
    (dict(D=256, H=200, Hk=1, qs=200 * 256, cbs=16 * 256),
     pa.PA_ERR_UNSUPPORTED),                            # which needs scale > 0 and G <= 128
    (dict(dtype=2), pa.PA_ERR_UNSUPPORTED),             # neither bf16 (0) nor f16 (1)
    (dict(H=32, Hk=6), pa.PA_ERR_INVALID_ARG),          # H % H_kv != 0
    (dict(q=None), pa.PA_ERR_INVALID_ARG),
    (dict(out=None), pa.PA_ERR_INVALID_ARG),
    (dict(kc=FAKE + 2), pa.PA_ERR_INVALID_ARG),         # misaligned
    (dict(qs=32 * 128 + 4), pa.PA_ERR_INVALID_ARG),     # stride not 16-byte multiple
    (dict(qs=16), pa.PA_ERR_INVALID_ARG),               # stride shorter than a row
    (dict(cbs=100), pa.PA_ERR_INVALID_ARG),
    (dict(causal=2), pa.PA_ERR_INVALID_ARG),
    (dict(scale=float("nan")), pa.PA_ERR_INVALID_ARG),
    (dict(scale=float("inf")), pa.PA_ERR_INVALID_ARG),
    (dict(scale=float("-inf")), pa.PA_ERR_INVALID_ARG),
    (dict(S=-1), pa.PA_ERR_INVALID_ARG),
    (dict(S=0, T=0), pa.PA_OK),                         # empty batch: nothing to do
])
def test_varlen_host_validation(lib, kw, code):
    assert _varlen(lib, **kw) == code


@pytest.mark.parametrize("kw", [
    dict(H=24, Hk=8),       # GQA ratio 3: any H % H_kv == 0 is accepted
    dict(H=40, Hk=8),       # ratio 5
    dict(H=28, Hk=4),       # ratio 7
    dict(H=200, Hk=1),      # a group wider than a 128-lane prefill tile
    dict(scale=0.0),        # any finite softmax scale
    dict(scale=-0.1),
    dict(D=256),            # head sizes 64, 128 and 256
    dict(D=256, H=24, Hk=8),
])
def test_varlen_accepts_every_ratio_and_finite_scale(lib, kw):
    """These pass every argument check; with no workspace the call then stops
    at PA_ERR_WORKSPACE (or PA_ERR_CUDA on a machine without a GPU, where the
    SM count cannot be queried) -- either way before anything is launched."""
    D = kw.get("D", 128)
    qs = kw.get("H", 32) * D     # the query row is H x D elements
    assert _varlen(lib, ws=None, wsb=0, qs=qs, cbs=16 * kw.get("Hk", 8) * D, **kw) in (
        pa.PA_ERR_WORKSPACE, pa.PA_ERR_CUDA)
    n = lib.pa_varlen_fwd_workspace_size(2, 2, 1, 64, kw.get("H", 32), kw.get("Hk", 8), D, 16,
                                         152)
    assert n > 0 and n % 256 == 0


def test_cascade_prefix_must_be_page_multiple(lib):
    args = [FAKE, 32 * 128, FAKE, FAKE, 16 * 8 * 128, FAKE, FAKE, FAKE, 200, 2, 2, 1, 64, 32, 8,
            128, 16, 10, 0.088]
    tail = [FAKE, None, FAKE, 1 << 20, 0, None, None]
    assert lib.pa_cascade_fwd(*args, 24, *tail) == pa.PA_ERR_INVALID_ARG   # 24 % 16 != 0
    assert lib.pa_cascade_fwd(*args, -16, *tail) == pa.PA_ERR_INVALID_ARG
    assert lib.pa_cascade_fwd(*args, 16 * 201, *tail) == pa.PA_ERR_INVALID_ARG  # past the row


def test_reshape_and_cache_host_validation(lib):
    f = lib.pa_reshape_and_cache
    ok = [FAKE, FAKE, 1024, 1024, FAKE, FAKE, 16 * 1024, FAKE, 4, 8, 128, 16, 10, 0, None, None]

    def call(i, v):
        a = list(ok)
        a[i] = v
        return f(*a)
    assert call(11, 24) == pa.PA_ERR_BLOCK_SIZE      # the pages' "multiple of 16" rule
    assert call(10, 80) == pa.PA_ERR_UNSUPPORTED     # head size
    assert call(13, 2) == pa.PA_ERR_UNSUPPORTED      # dtype: neither bf16 nor f16
    assert call(0, None) == pa.PA_ERR_INVALID_ARG
    assert call(7, FAKE + 4) == pa.PA_ERR_INVALID_ARG   # int64 slots misaligned
    assert call(2, 512) == pa.PA_ERR_INVALID_ARG     # token stride shorter than a row
    assert call(8, 0) == pa.PA_OK                    # no tokens: nothing to do


def test_merge_host_validation(lib):
    f = lib.pa_merge_attn_states
    base = [FAKE, FAKE + 0x1000, FAKE, FAKE + 0x2000, FAKE, FAKE + 0x3000, 4, 8, 128, 0, None]

    def call(i, v):
        a = list(base)
        a[i] = v
        return f(*a)
    assert call(9, 2) == pa.PA_ERR_UNSUPPORTED
    assert call(2, None) == pa.PA_ERR_INVALID_ARG
    assert call(1, FAKE + 0x2000) == pa.PA_ERR_INVALID_ARG   # out_lse aliases prefix_lse
    assert call(6, 0) == pa.PA_OK


def test_binding_refuses_cpu_tensors():
    import torch
    x = torch.zeros(2, 8, 128, dtype=torch.bfloat16)
    c = torch.zeros(4, 16, 8, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        pa.reshape_and_cache(x, x, c, c, torch.zeros(2, dtype=torch.int64))


def _upd(**kw):
    a = dict(key=FAKE, value=FAKE, ks=1024, vs=1024, slots=FAKE, n=4)
    a.update(kw)
    return pa.KvUpdate(a["key"], a["value"], a["ks"], a["vs"], a["slots"], a["n"])


def _varlen_upd(lib, upd, **kw):
    a = dict(q=FAKE, qs=32 * 128, kc=FAKE, vc=FAKE, cbs=16 * 8 * 128, cu=FAKE, lens=FAKE,
             bt=FAKE, bts=4, S=2, T=2, mq=1, mk=64, H=32, Hk=8, D=128, bs=16, nb=10,
             scale=0.088, causal=1, out=FAKE, lse=None, ws=FAKE, wsb=1 << 20, dtype=0)
    a.update(kw)
    return lib.pa_varlen_fwd_with_update(
        ctypes.byref(upd) if upd is not None else None, a["q"], a["qs"], a["kc"], a["vc"],
        a["cbs"], a["cu"], a["lens"], a["bt"], a["bts"], a["S"], a["T"], a["mq"], a["mk"], a["H"],
        a["Hk"], a["D"], a["bs"], a["nb"], a["scale"], a["causal"], a["out"], a["lse"], a["ws"],
        a["wsb"], a["dtype"], None, None)


def test_update_entry_validation(lib):
    """The K/V update of an update-and-attend call is checked like
    pa_reshape_and_cache's arguments before anything is launched."""
    assert _varlen_upd(lib, _upd(n=-1)) == pa.PA_ERR_INVALID_ARG
    assert _varlen_upd(lib, _upd(key=None)) == pa.PA_ERR_INVALID_ARG
    assert _varlen_upd(lib, _upd(key=FAKE + 2)) == pa.PA_ERR_INVALID_ARG   # misaligned
    assert _varlen_upd(lib, _upd(slots=FAKE + 4)) == pa.PA_ERR_INVALID_ARG
    assert _varlen_upd(lib, _upd(ks=512)) == pa.PA_ERR_INVALID_ARG        # shorter than a row
    assert _varlen_upd(lib, _upd(), bs=24) == pa.PA_ERR_BLOCK_SIZE
    # attention arguments are still checked
    assert _varlen_upd(lib, _upd(), scale=float("nan")) == pa.PA_ERR_INVALID_ARG
    # nothing to do: no update and an empty batch, or an update of zero tokens
    assert _varlen_upd(lib, None, S=0, T=0) == pa.PA_OK
    assert _varlen_upd(lib, _upd(n=0), S=0, T=0) == pa.PA_OK
    args = [ctypes.byref(_upd(n=-1)), FAKE, 32 * 128, FAKE, FAKE, 16 * 8 * 128, FAKE, FAKE, FAKE,
            200, 2, 2, 1, 64, 32, 8, 128, 16, 10, 0.088, 16, FAKE, None, FAKE, 1 << 20, 0, None,
            None]
    assert lib.pa_cascade_fwd_with_update(*args) == pa.PA_ERR_INVALID_ARG


def test_use_cascade_attention_policy(lib):
    """The pages' use_cascade_attention rules (a shared prefix of >= 256
    tokens, >= 8 requests; cascade outright without split-KV), then this
    library's byte estimate: cascade iff re-reading the prefix per sequence
    costs more than the cascade's fixed 20 us at 6.5 TB/s."""
    def use(P, S, Hk=8, D=128, split=1):
        out = ctypes.c_int(-1)
        assert lib.pa_use_cascade_attention(P, S, Hk, D, split, ctypes.byref(out)) == pa.PA_OK
        return out.value
    assert use(255, 64, split=0) == 0          # prefix too short
    assert use(256, 7, split=0) == 0           # too few requests
    assert use(256, 8, split=0) == 1           # no split-KV: cascade outright
    assert use(2048, 64) == 1                  # the shared-prompt workload
    assert use(256, 8) == 0                    # small prefix, few requests: flat
    # boundary of the estimate: (S-1)*P*Hk*D*4 > 20e-6 * 6.5e12 = 1.3e8 bytes
    assert use(4534, 8) == 0                   # 7*4534*4096 = 129,998,848 bytes: just below
    bound = 20e-6 * 6500.0 * 1e9
    for P in (4530, 4531, 4532, 4533, 4534, 4535, 4536):
        assert use(P, 8) == int(7 * P * 8 * 128 * 4 > bound)
    out = ctypes.c_int(0)
    assert lib.pa_use_cascade_attention(-1, 8, 8, 128, 1, ctypes.byref(out)) == \
        pa.PA_ERR_INVALID_ARG
    assert lib.pa_use_cascade_attention(256, 8, 8, 128, 1, None) == pa.PA_ERR_INVALID_ARG
    assert pa.use_cascade_attention(2048, 64, 8, 128) is True


def _fp8(ks=FAKE, vs=FAKE):
    return pa.KvFp8(ks, vs)


def _varlen_fp8(lib, upd, fp8, **kw):
    a = dict(q=FAKE, qs=32 * 128, kc=FAKE, vc=FAKE, cbs=16 * 8 * 128, cu=FAKE, lens=FAKE,
             bt=FAKE, bts=4, S=2, T=2, mq=1, mk=64, H=32, Hk=8, D=128, bs=16, nb=10,
             scale=0.088, causal=1, out=FAKE, lse=None, ws=FAKE, wsb=1 << 20, dtype=0)
    a.update(kw)
    return lib.pa_varlen_fwd_fp8kv(
        ctypes.byref(upd) if upd is not None else None, a["q"], a["qs"], a["kc"], a["vc"],
        a["cbs"], a["cu"], a["lens"], a["bt"], a["bts"], a["S"], a["T"], a["mq"], a["mk"], a["H"],
        a["Hk"], a["D"], a["bs"], a["nb"], a["scale"], a["causal"],
        ctypes.byref(fp8) if fp8 is not None else None, a["out"], a["lse"], a["ws"], a["wsb"],
        a["dtype"], None, None)


def test_fp8_entry_validation(lib):
    """FP8 pools: head size 128 only, scales required (4-byte aligned), page
    stride a multiple of 16 bytes; checked before anything is launched."""
    assert _varlen_fp8(lib, None, _fp8(), D=64, qs=32 * 64, cbs=16 * 8 * 64) == \
        pa.PA_ERR_UNSUPPORTED
    assert _varlen_fp8(lib, None, None) == pa.PA_ERR_INVALID_ARG
    assert _varlen_fp8(lib, None, _fp8(ks=None)) == pa.PA_ERR_INVALID_ARG
    assert _varlen_fp8(lib, None, _fp8(vs=FAKE + 2)) == pa.PA_ERR_INVALID_ARG
    assert _varlen_fp8(lib, None, _fp8(), cbs=16 * 8 * 128 + 8) == pa.PA_ERR_INVALID_ARG
    assert _varlen_fp8(lib, _upd(key=FAKE + 2), _fp8()) == pa.PA_ERR_INVALID_ARG
    assert _varlen_fp8(lib, None, _fp8(), S=0, T=0) == pa.PA_OK
    args = [FAKE, FAKE, 1024, 1024, FAKE, FAKE, 16 * 8 * 128, FAKE, 4, 8, 128, 16, 10]
    assert lib.pa_reshape_and_cache_fp8(*args, None, 0, None, None) == pa.PA_ERR_INVALID_ARG
    bad_d = [FAKE, FAKE, 512, 512, FAKE, FAKE, 16 * 8 * 64, FAKE, 4, 8, 64, 16, 10]
    assert lib.pa_reshape_and_cache_fp8(*bad_d, ctypes.byref(_fp8()), 0, None, None) == \
        pa.PA_ERR_UNSUPPORTED
    bad_stride = args[:6] + [16 * 8 * 128 + 8] + args[7:]
    assert lib.pa_reshape_and_cache_fp8(*bad_stride, ctypes.byref(_fp8()), 0, None, None) == \
        pa.PA_ERR_INVALID_ARG
    zero = args[:8] + [0] + args[9:]
    assert lib.pa_reshape_and_cache_fp8(*zero, None, 0, None, None) == pa.PA_OK
    assert lib.pa_varlen_fwd_fp8kv_workspace_size(2, 2, 1, 64, 32, 8, 64, 16, 152) == 0
    assert lib.pa_varlen_fwd_fp8kv_workspace_size(2, 2, 1, 64, 32, 8, 128, 16, 152) > 0
    assert lib.pa_cascade_fwd_fp8kv_workspace_size(2, 2, 1, 64, 32, 8, 128, 16, 152) > 0


def test_merge_n_validation(lib):
    """pa_merge_attn_states_n checks its arguments before launching."""
    T, H, D = 4, 2, 128
    rowe, lsee = T * H * D, H * T
    args = dict(out=FAKE, olse=None, po=FAKE, ps=rowe, pl=FAKE, pls=lsee, n=3, T=T, H=H, D=D)

    def call(**kw):
        a = dict(args)
        a.update(kw)
        return lib.pa_merge_attn_states_n(a["out"], a["olse"], a["po"], a["ps"], a["pl"], a["pls"],
                                          a["n"], a["T"], a["H"], a["D"], 0, None)
    assert call(n=0) == pa.PA_ERR_INVALID_ARG
    assert call(n=1025) == pa.PA_ERR_INVALID_ARG
    assert call(D=12) == pa.PA_ERR_UNSUPPORTED
    assert call(T=0) == pa.PA_OK
    assert call(ps=rowe - 8) == pa.PA_ERR_INVALID_ARG          # parts overlap
    assert call(ps=rowe + 4) == pa.PA_ERR_INVALID_ARG          # not a 16-byte multiple
    assert call(pls=lsee - 1) == pa.PA_ERR_INVALID_ARG
    assert call(po=FAKE + 8) == pa.PA_ERR_INVALID_ARG          # misaligned
    assert call(olse=FAKE + 4 * lsee) == pa.PA_ERR_INVALID_ARG  # out_lse inside part 1's LSE
    assert call(po=None) == pa.PA_ERR_INVALID_ARG


def test_ex_entry_validation(lib):
    """The option entries: sinks must be 4-byte aligned; NULL options are the
    plain entry; an FP8 descriptor in the options is checked like the FP8
    entry's."""
    a = [FAKE, 32 * 128, FAKE, FAKE, 16 * 8 * 128, FAKE, FAKE, FAKE, 4, 2, 2, 1, 64, 32, 8, 128,
         16, 10, 0.088, 1]
    tail = [FAKE, None, FAKE, 1 << 20, 0, None, None]
    bad = pa.AttnOpts(FAKE + 2, None)
    assert lib.pa_varlen_fwd_ex(None, *a, ctypes.byref(bad), *tail) == pa.PA_ERR_INVALID_ARG
    assert lib.pa_cascade_fwd_ex(None, *a[:19], 16, ctypes.byref(bad), *tail) == \
        pa.PA_ERR_INVALID_ARG
    empty = list(a)
    empty[9], empty[10] = 0, 0          # no sequences, no tokens
    assert lib.pa_varlen_fwd_ex(None, *empty, None, *tail) == pa.PA_OK
    fp8_d64 = list(a)
    fp8_d64[1], fp8_d64[4], fp8_d64[15] = 32 * 64, 16 * 8 * 64, 64
    desc = pa.KvFp8(FAKE, FAKE)
    opts = pa.AttnOpts(None, ctypes.pointer(desc))
    assert lib.pa_varlen_fwd_ex(None, *fp8_d64, ctypes.byref(opts), *tail) == pa.PA_ERR_UNSUPPORTED
