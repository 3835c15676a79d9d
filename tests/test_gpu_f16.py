"""GPU parity with IEEE half (f16) inputs and outputs ("FlashAttention 在 vLLM
中的实现分析" §2.1: float16 and bfloat16 are the supported activation types).
The workloads draw the same fp32 values as the bf16 ones and round them to
f16; the oracle reads those f16 values. Scatter bit-exact; f16 outputs within
1e-2 max-abs and LSE within 1e-3 absolute, as for bf16."""
import pytest
import torch

import oracle
import paged_kv_varlen_attn_gb300 as pa
import workloads as W
from helpers import oracle_full, oracle_pools, oracle_sampled, to_dev
from test_gpu_parity import DEV, _sample_rows, assert_close, run_gpu

pytestmark = pytest.mark.gpu
F16 = torch.float16


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_varlen_attn_gb300 import _build
    _build.build()
    pa.load_library()


def test_scatter_bit_exact_f16():
    wl = W.tiny_mixed(dtype=F16)
    kc_ref, vc_ref = oracle_pools(wl)
    d = to_dev(wl, DEV)
    pa.reshape_and_cache(d["k_new"], d["v_new"], d["key_cache"], d["value_cache"],
                         d["slot_mapping"])
    torch.cuda.synchronize()
    assert d["key_cache"].dtype == F16
    assert torch.equal(d["key_cache"].cpu().view(torch.int16), kc_ref.view(torch.int16))
    assert torch.equal(d["value_cache"].cpu().view(torch.int16), vc_ref.view(torch.int16))


CASES = [
    # seed, S, H, Hk, D, bs, max_q, max_kv, causal, decode_frac
    (301, 5, 4, 2, 64, 16, 40, 150, True, 0.3),
    (302, 4, 8, 2, 128, 16, 300, 1100, True, 0.2),     # multi-tile prefill: tensor-core kernel
    (303, 3, 8, 8, 128, 32, 90, 200, False, 0.3),
    (304, 4, 32, 4, 128, 128, 33, 700, True, 0.5),
    (305, 2, 16, 2, 64, 32, 260, 700, False, 0.0),
    (306, 4, 8, 2, 128, 16, 1, 6000, True, 1.0),       # decode with many KV splits
    (307, 3, 24, 8, 128, 16, 150, 400, True, 0.3),     # G = 3
]


@pytest.mark.parametrize("case", CASES, ids=[str(c[0]) for c in CASES])
def test_random_varlen_f16(case):
    seed, S, H, Hk, D, bs, mq, mk, causal, dfrac = case
    wl = W.random_case(seed, num_seqs=S, num_heads=H, num_kv_heads=Hk, head_size=D,
                       block_size=bs, max_q=mq, max_kv=mk, causal=causal, decode_frac=dfrac,
                       dtype=F16)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out, lse, _ = run_gpu(wl, status=status)
    assert out.dtype == F16
    ref_o, ref_l = oracle_full(wl)
    assert_close(out, lse, ref_o, ref_l)
    assert int(status.item()) == 0


def test_tiny_mixed_f16():
    wl = W.tiny_mixed(dtype=F16)
    out, lse, _ = run_gpu(wl)
    ref_o, ref_l = oracle_full(wl)
    assert_close(out, lse, ref_o, ref_l)


def test_cascade_shared_prefix_f16():
    wl = W.cascade_shared_prefix(dtype=F16)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out, lse, _ = run_gpu(wl, cascade=True, status=status)
    ref_o, ref_l = oracle_full(wl, cascade=True)
    assert_close(out, lse, ref_o, ref_l)
    assert int(status.item()) == 0


@pytest.mark.parametrize("name,seqs", [
    ("decode_llama8b", [0, 17, 63]),
    ("chunked_prefill_mix", [0, 7, 8, 40]),
    ("long_context_70b", [0, 32, 35]),
])
def test_full_size_config_sampled_f16(name, seqs):
    wl = W.CONFIGS[name](dtype=F16)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out, lse, _ = run_gpu(wl, status=status)
    ref = oracle_sampled(wl, _sample_rows(wl, seqs))
    for s, (tok, ro, rl) in ref.items():
        assert_close(out, lse, ro, rl, tokens=tok)
    assert int(status.item()) == 0


def test_merges_f16():
    g = torch.Generator().manual_seed(311)
    n, T, H, D = 3, 41, 8, 128
    po = torch.randn((n, T, H, D), generator=g).to(F16)
    pl = torch.randn((n, H, T), generator=g) * 3
    pl[:, 0, :4] = float("-inf")
    ref_o, ref_l = oracle.merge_attn_states(po[0], pl[0], po[1], pl[1])
    out, lse = pa.merge_attn_states(po[0].to(DEV), pl[0].to(DEV), po[1].to(DEV), pl[1].to(DEV))
    torch.cuda.synchronize()
    assert out.dtype == F16
    assert_close(out, lse, ref_o, ref_l)
    ref_o, ref_l = oracle.merge_attn_states_n(po, pl)
    out, lse = pa.merge_attn_states_n(po.to(DEV), pl.to(DEV))
    torch.cuda.synchronize()
    assert_close(out, lse, ref_o, ref_l)


def test_update_entry_f16_equals_separate_calls():
    wl = W.random_case(321, num_seqs=4, num_heads=8, num_kv_heads=2, head_size=128,
                       block_size=16, max_q=150, max_kv=500, decode_frac=0.3, dtype=F16)
    d1, d2 = to_dev(wl, DEV), to_dev(wl, DEV)
    o1, l1, _ = run_gpu(wl, d1)
    o2, l2 = pa.varlen_fwd_with_update(d2["k_new"], d2["v_new"], d2["slot_mapping"], d2["q"],
                                       d2["key_cache"], d2["value_cache"], d2["cu_seqlens_q"],
                                       d2["seqused_k"], d2["block_table"], wl.max_seqlen_q,
                                       wl.max_seqlen_k, wl.softmax_scale, wl.causal)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_sinks_f16():
    wl = W.random_case(331, num_seqs=3, num_heads=8, num_kv_heads=2, head_size=128,
                       block_size=16, max_q=140, max_kv=400, decode_frac=0.3, dtype=F16)
    sinks = torch.linspace(-2.0, 3.0, wl.num_heads, dtype=torch.float32)
    d = to_dev(wl, DEV)
    pa.reshape_and_cache(d["k_new"], d["v_new"], d["key_cache"], d["value_cache"],
                         d["slot_mapping"])
    out, lse = pa.varlen_fwd(d["q"], d["key_cache"], d["value_cache"], d["cu_seqlens_q"],
                             d["seqused_k"], d["block_table"], wl.max_seqlen_q, wl.max_seqlen_k,
                             wl.softmax_scale, wl.causal, sinks=sinks.to(DEV))
    torch.cuda.synchronize()
    kc, vc = oracle_pools(wl)
    ref_o, ref_l = oracle.varlen_attention(wl.q, kc, vc, wl.cu_seqlens_q, wl.seqused_k,
                                           wl.block_table, wl.softmax_scale, wl.causal,
                                           sinks=sinks)
    assert_close(out, lse, ref_o, ref_l)


def test_fp8_pools_with_f16_activations():
    """e4m3 pools, f16 queries, new tokens and outputs: the quantizing scatter
    is bit-exact against the oracle's (which reads the f16 values), and the
    attention matches the oracle over the dequantized pools (decode rows on
    the e4m3 MMA consumer, wider rows on the f16 one)."""
    wl = W.random_case(341, num_seqs=5, num_heads=16, num_kv_heads=2, head_size=128,
                       block_size=16, max_q=60, max_kv=500, decode_frac=0.5, dtype=F16)
    ks, vs = wl.kv_scales(0), wl.kv_scales(1)
    kc_ref, vc_ref = wl.fp8_pool(0), wl.fp8_pool(1)
    oracle.reshape_and_cache_e4m3(wl.k_new, wl.v_new, wl.slot_mapping, kc_ref, vc_ref, ks, vs)
    kc, vc = wl.fp8_pool(0, DEV), wl.fp8_pool(1, DEV)
    out, lse = pa.varlen_fwd_fp8kv(wl.q.to(DEV), kc, vc, wl.cu_seqlens_q.to(DEV),
                                   wl.seqused_k.to(DEV), wl.block_table.to(DEV), wl.max_seqlen_q,
                                   wl.max_seqlen_k, wl.softmax_scale, wl.causal,
                                   torch.tensor(ks, device=DEV), torch.tensor(vs, device=DEV),
                                   key=wl.k_new.to(DEV), value=wl.v_new.to(DEV),
                                   slot_mapping=wl.slot_mapping.to(DEV))
    torch.cuda.synchronize()
    assert out.dtype == F16
    assert torch.equal(kc.cpu(), kc_ref) and torch.equal(vc.cpu(), vc_ref)
    ref_o, ref_l = oracle.varlen_attention_e4m3(wl.q, kc_ref, vc_ref, wl.cu_seqlens_q,
                                                wl.seqused_k, wl.block_table, wl.softmax_scale,
                                                wl.causal, ks, vs)
    assert_close(out, lse, ref_o, ref_l)


def test_mixed_element_types_are_refused():
    wl = W.random_case(351, num_seqs=2, dtype=F16)
    d = to_dev(wl, DEV)
    with pytest.raises(ValueError):
        pa.varlen_fwd(d["q"].to(torch.bfloat16), d["key_cache"], d["value_cache"],
                      d["cu_seqlens_q"], d["seqused_k"], d["block_table"], wl.max_seqlen_q,
                      wl.max_seqlen_k, wl.softmax_scale, wl.causal)
