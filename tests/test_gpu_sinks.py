"""GPU parity of attention sinks ("FlashAttention 在 vLLM 中的实现分析"
§1.2 / §1.3: the s_aux sink token of FA3/FA4) against the fp64 oracle, on
every kernel path that writes final rows: the split-KV kernel (one split and
several, bf16 and both FP8 consumers), the tensor-core prefill kernel (one
split and several) and the cascade's combine."""
import pytest
import torch

import oracle
import paged_kv_varlen_attn_gb300 as pa
import workloads as W
from helpers import LSE_TOL, OUT_TOL, oracle_pools

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_varlen_attn_gb300 import _build
    _build.build()
    pa.load_library()


def check(out, lse, ref_o, ref_l):
    o, l = out.cpu().double(), lse.cpu().double()
    fin = torch.isfinite(ref_l)
    assert torch.equal(fin, torch.isfinite(l))
    assert (o - ref_o).abs().max().item() <= OUT_TOL
    assert (l[fin] - ref_l[fin]).abs().max().item() <= LSE_TOL


def sinks_for(H):
    return torch.linspace(-1.0, 4.0, H, dtype=torch.float32)


CASES = [
    # seed, S, H, Hk, D, bs, max_q, max_kv, causal, decode_frac, empty_ok
    (401, 6, 32, 8, 128, 16, 1, 3000, True, 1.0, False),    # decode, several splits
    (402, 5, 8, 2, 64, 16, 1, 200, True, 1.0, False),       # decode, one split, D 64
    (403, 3, 16, 2, 128, 32, 300, 700, True, 0.0, False),   # prefill on the tensor-core kernel
    (404, 2, 32, 8, 128, 128, 200, 4000, True, 0.0, False), # prefill with KV splits
    (405, 6, 8, 2, 128, 16, 12, 60, True, 0.3, True),       # empty sequences, keyless rows
    (406, 4, 8, 8, 64, 16, 40, 300, False, 0.2, False),     # non-causal
]


@pytest.mark.parametrize("seed,S,H,Hk,D,bs,max_q,max_kv,causal,dfrac,empty", CASES)
def test_sinks_varlen(seed, S, H, Hk, D, bs, max_q, max_kv, causal, dfrac, empty):
    wl = W.random_case(seed, num_seqs=S, num_heads=H, num_kv_heads=Hk, head_size=D,
                       block_size=bs, max_q=max_q, max_kv=max_kv, causal=causal,
                       decode_frac=dfrac, empty_ok=empty)
    sinks = sinks_for(H)
    kc, vc = oracle_pools(wl)
    ref_o, ref_l = oracle.varlen_attention(wl.q, kc, vc, wl.cu_seqlens_q, wl.seqused_k,
                                           wl.block_table, wl.softmax_scale, causal,
                                           sinks=sinks.double())
    out, lse = pa.varlen_fwd(wl.q.to(DEV), kc.to(DEV), vc.to(DEV), wl.cu_seqlens_q.to(DEV),
                             wl.seqused_k.to(DEV), wl.block_table.to(DEV),
                             max(wl.max_seqlen_q, 1), wl.max_seqlen_k, wl.softmax_scale, causal,
                             sinks=sinks.to(DEV))
    torch.cuda.synchronize()
    check(out, lse, ref_o, ref_l)


@pytest.mark.parametrize("seed,H,Hk,max_q,max_kv", [(411, 32, 8, 1, 2500), (412, 32, 2, 1, 600),
                                                   (413, 16, 2, 40, 300)])
def test_sinks_fp8(seed, H, Hk, max_q, max_kv):
    """FP8 pools: the transposed decode consumer (GQA 4), the 16-row consumer
    (GQA 16) and wider rows (GQA 8 with up to 40 queries)."""
    wl = W.random_case(seed, num_seqs=5, num_heads=H, num_kv_heads=Hk, head_size=128,
                       block_size=16, max_q=max_q, max_kv=max_kv, decode_frac=0.5)
    sinks = sinks_for(H)
    kc, vc = wl.fp8_pool(0), wl.fp8_pool(1)
    oracle.reshape_and_cache_e4m3(wl.k_new, wl.v_new, wl.slot_mapping, kc, vc, wl.kv_scales(0),
                                  wl.kv_scales(1))
    kd = oracle.dequantize_e4m3(kc, wl.kv_scales(0))
    vd = oracle.dequantize_e4m3(vc, wl.kv_scales(1))
    ref_o, ref_l = oracle.varlen_attention(wl.q, kd, vd, wl.cu_seqlens_q, wl.seqused_k,
                                           wl.block_table, wl.softmax_scale, True,
                                           sinks=sinks.double())
    kcd, vcd = wl.fp8_pool(0, DEV), wl.fp8_pool(1, DEV)
    out, lse = pa.varlen_fwd_fp8kv(
        wl.q.to(DEV), kcd, vcd, wl.cu_seqlens_q.to(DEV), wl.seqused_k.to(DEV),
        wl.block_table.to(DEV), wl.max_seqlen_q, wl.max_seqlen_k, wl.softmax_scale, True,
        torch.tensor(wl.kv_scales(0), device=DEV), torch.tensor(wl.kv_scales(1), device=DEV),
        key=wl.k_new.to(DEV), value=wl.v_new.to(DEV), slot_mapping=wl.slot_mapping.to(DEV),
        sinks=sinks.to(DEV))
    torch.cuda.synchronize()
    check(out, lse, ref_o, ref_l)


def test_sinks_cascade():
    g = torch.Generator().manual_seed(421)
    S, P = 12, 256
    suffix = [int(x) for x in torch.randint(4, 120, (S,), generator=g)]
    q_lens = [int(x) for x in torch.randint(1, 4, (S,), generator=g)]
    wl = W._build("cascade_sinks", 421, 32, 4, 128, 16, q_lens, [P + s for s in suffix], g,
                  shared_prefix_pages=P // 16)
    sinks = sinks_for(32)
    kc, vc = oracle_pools(wl)
    ref_o, ref_l = oracle.cascade_attention(wl.q, kc, vc, wl.cu_seqlens_q, wl.seqused_k,
                                            wl.block_table, wl.softmax_scale,
                                            wl.common_prefix_len, sinks=sinks.double())
    out, lse = pa.cascade_fwd(wl.q.to(DEV), kc.to(DEV), vc.to(DEV), wl.cu_seqlens_q.to(DEV),
                              wl.seqused_k.to(DEV), wl.block_table.to(DEV), wl.max_seqlen_q,
                              wl.max_seqlen_k, wl.softmax_scale, wl.common_prefix_len,
                              sinks=sinks.to(DEV))
    torch.cuda.synchronize()
    check(out, lse, ref_o, ref_l)


def test_sinks_minus_inf_equals_plain():
    wl = W.random_case(431, num_seqs=5, num_heads=16, num_kv_heads=4, head_size=128,
                       block_size=16, max_q=40, max_kv=900)
    kc, vc = oracle_pools(wl)
    args = (wl.q.to(DEV), kc.to(DEV), vc.to(DEV), wl.cu_seqlens_q.to(DEV), wl.seqused_k.to(DEV),
            wl.block_table.to(DEV), wl.max_seqlen_q, wl.max_seqlen_k, wl.softmax_scale, True)
    o1, l1 = pa.varlen_fwd(*args)
    o2, l2 = pa.varlen_fwd(*args, sinks=torch.full((16,), float("-inf"), device=DEV))
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
