"""Update-and-attend entry points (pa_varlen_fwd_with_update,
pa_cascade_fwd_with_update) through the C ABI: one call that scatters the
step's new K/V and attends must give bitwise the same cache, output and LSE
as pa_reshape_and_cache followed by the attention call (the same kernels run
in the same order of arithmetic; only the planner overlaps the scatter), and
match the oracle."""
import pytest
import torch

import paged_kv_varlen_attn_gb300 as pa
import workloads as W
from helpers import LSE_TOL, OUT_TOL, oracle_full, oracle_pools, to_dev

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_varlen_attn_gb300 import _build
    _build.build()
    pa.load_library()


def _args(wl, d):
    return (d["q"], d["key_cache"], d["value_cache"], d["cu_seqlens_q"], d["seqused_k"],
            d["block_table"], max(wl.max_seqlen_q, 1), wl.max_seqlen_k, wl.softmax_scale)


def _separate(wl, cascade):
    d = to_dev(wl, DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    pa.reshape_and_cache(d["k_new"], d["v_new"], d["key_cache"], d["value_cache"],
                         d["slot_mapping"], dev_status=st)
    if cascade:
        out, lse = pa.cascade_fwd(*_args(wl, d), wl.common_prefix_len, dev_status=st)
    else:
        out, lse = pa.varlen_fwd(*_args(wl, d), wl.causal, dev_status=st)
    torch.cuda.synchronize()
    return out, lse, d, int(st.item())


def _fused(wl, cascade, reps=1):
    d = to_dev(wl, DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    for _ in range(reps):   # repeating the step rewrites the same slots with the same rows
        if cascade:
            out, lse = pa.cascade_fwd_with_update(d["k_new"], d["v_new"], d["slot_mapping"],
                                                  *_args(wl, d), wl.common_prefix_len,
                                                  dev_status=st)
        else:
            out, lse = pa.varlen_fwd_with_update(d["k_new"], d["v_new"], d["slot_mapping"],
                                                 *_args(wl, d), wl.causal, dev_status=st)
    torch.cuda.synchronize()
    return out, lse, d, int(st.item())


@pytest.mark.parametrize("name", ["tiny_mixed", "random_104", "random_109"])
def test_varlen_with_update_equals_separate_calls(name):
    if name == "tiny_mixed":
        wl = W.tiny_mixed()
    elif name == "random_104":
        wl = W.random_case(104, num_seqs=6, num_heads=16, num_kv_heads=2, head_size=64,
                           block_size=64, max_q=20, max_kv=400, decode_frac=0.5)
    else:
        wl = W.random_case(109, num_seqs=2, num_heads=8, num_kv_heads=2, head_size=128,
                           block_size=16, max_q=300, max_kv=1100, decode_frac=0.0)
    o1, l1, d1, s1 = _separate(wl, False)
    o2, l2, d2, s2 = _fused(wl, False, reps=2)
    assert s1 == 0 and s2 == 0
    assert torch.equal(d1["key_cache"], d2["key_cache"])
    assert torch.equal(d1["value_cache"], d2["value_cache"])
    assert torch.equal(o1, o2)
    assert torch.equal(l1, l2)
    kc_ref, vc_ref = oracle_pools(wl)
    assert torch.equal(d2["key_cache"].cpu(), kc_ref)
    ref_o, ref_l = oracle_full(wl)
    fin = torch.isfinite(ref_l)
    assert (o2.cpu().double() - ref_o).abs().max().item() <= OUT_TOL
    assert (l2.cpu().double()[fin] - ref_l[fin]).abs().max().item() <= LSE_TOL


def test_cascade_with_update_equals_separate_calls():
    g = torch.Generator().manual_seed(81)
    S, P, bs = 12, 128, 16
    suffix = [int(x) for x in torch.randint(8, 120, (S,), generator=g)]
    q_lens = [min(int(x), s) for x, s in zip(torch.randint(1, 4, (S,), generator=g), suffix)]
    wl = W._build("cascade_update", 81, 16, 4, 128, bs, q_lens, [P + s for s in suffix], g,
                  shared_prefix_pages=P // bs)
    o1, l1, d1, s1 = _separate(wl, True)
    o2, l2, d2, s2 = _fused(wl, True)
    assert s1 == 0 and s2 == 0
    assert torch.equal(d1["key_cache"], d2["key_cache"])
    assert torch.equal(o1, o2)
    assert torch.equal(l1, l2)
    ref_o, ref_l = oracle_full(wl, cascade=True)
    assert (o2.cpu().double() - ref_o).abs().max().item() <= OUT_TOL


def test_update_without_attention_only_scatters():
    wl = W.tiny_mixed()
    d = to_dev(wl, DEV)
    kc_ref, vc_ref = oracle_pools(wl)
    empty_cu = torch.zeros(1, dtype=torch.int32, device=DEV)
    empty = torch.zeros(0, dtype=torch.int32, device=DEV)
    q = torch.zeros((0, wl.num_heads, wl.head_size), dtype=torch.bfloat16, device=DEV)
    bt = torch.zeros((0, 1), dtype=torch.int32, device=DEV)
    pa.varlen_fwd_with_update(d["k_new"], d["v_new"], d["slot_mapping"], q, d["key_cache"],
                              d["value_cache"], empty_cu, empty, bt, 1, 1, wl.softmax_scale, True)
    torch.cuda.synchronize()
    assert torch.equal(d["key_cache"].cpu(), kc_ref)
    assert torch.equal(d["value_cache"].cpu(), vc_ref)
