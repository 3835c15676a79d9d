"""GPU parity at head size 256 ("FlashAttention 在 vLLM 中的实现分析" §10: head
sizes up to 256; "AttentionBackend" 境界と失敗: unsupported head sizes are
refused). At this size every segment -- decode rows included -- runs on the
tensor-core kernel with one 128-row Q tile and 64-key K/V tiles. Same oracle
and tolerances as the other parity tests."""
import pytest
import torch

import oracle
import paged_kv_varlen_attn_gb300 as pa
import workloads as W
from helpers import oracle_full, oracle_pools, oracle_sampled, to_dev
from test_gpu_parity import DEV, assert_close, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_varlen_attn_gb300 import _build
    _build.build()
    pa.load_library()


CASES = [
    # seed, S, H, Hk, D, bs, max_q, max_kv, causal, decode_frac, dtype
    (401, 5, 4, 2, 256, 16, 40, 150, True, 0.3, torch.bfloat16),
    (402, 4, 8, 2, 256, 16, 300, 1100, True, 0.2, torch.bfloat16),    # several Q tiles
    (403, 3, 8, 8, 256, 32, 90, 200, False, 0.3, torch.bfloat16),     # G = 1, non-causal
    (404, 4, 32, 4, 256, 128, 33, 700, True, 0.5, torch.bfloat16),
    (405, 3, 16, 2, 256, 64, 200, 500, False, 0.0, torch.float16),
    (406, 4, 8, 2, 256, 16, 1, 6000, True, 1.0, torch.bfloat16),      # decode, many KV splits
    (407, 3, 24, 8, 256, 16, 150, 400, True, 0.3, torch.float16),     # G = 3
    (408, 3, 16, 1, 256, 48, 17, 260, True, 0.0, torch.bfloat16),     # MQA-like, block 48
]


@pytest.mark.parametrize("case", CASES, ids=[str(c[0]) for c in CASES])
def test_random_varlen_d256(case):
    seed, S, H, Hk, D, bs, mq, mk, causal, dfrac, dt = case
    wl = W.random_case(seed, num_seqs=S, num_heads=H, num_kv_heads=Hk, head_size=D,
                       block_size=bs, max_q=mq, max_kv=mk, causal=causal, decode_frac=dfrac,
                       dtype=dt)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out, lse, _ = run_gpu(wl, status=status)
    ref_o, ref_l = oracle_full(wl)
    assert_close(out, lse, ref_o, ref_l)
    assert int(status.item()) == 0


def test_empty_and_keyless_rows_d256():
    g = torch.Generator().manual_seed(411)
    H, Hk, D, bs = 8, 2, 256, 16
    q_lens, kv_lens = [0, 3, 5, 1, 0], [20, 0, 2, 40, 0]
    T, nb = sum(q_lens), 8
    kc = torch.randn(nb, bs, Hk, D, generator=g).to(torch.bfloat16)
    vc = torch.randn(nb, bs, Hk, D, generator=g).to(torch.bfloat16)
    q = torch.randn(T, H, D, generator=g).to(torch.bfloat16)
    bt = torch.tensor([[0, 1, 7], [2, 7, 7], [3, 7, 7], [4, 5, 6], [7, 7, 7]], dtype=torch.int32)
    cu = torch.tensor([0, 0, 3, 8, 9, 9], dtype=torch.int32)
    lens = torch.tensor(kv_lens, dtype=torch.int32)
    ref_o, ref_l = oracle.varlen_attention(q, kc, vc, cu, lens, bt, 0.0625, True)
    out, lse = pa.varlen_fwd(q.to(DEV), kc.to(DEV), vc.to(DEV), cu.to(DEV), lens.to(DEV),
                             bt.to(DEV), 5, 40, 0.0625, True)
    torch.cuda.synchronize()
    assert_close(out, lse, ref_o, ref_l)


def test_cascade_d256():
    g = torch.Generator().manual_seed(421)
    S, P, bs = 24, 256, 16
    suffix = [int(x) for x in torch.randint(5, 120, (S,), generator=g)]
    q_lens = [min(int(x), s) for x, s in zip(torch.randint(1, 4, (S,), generator=g), suffix)]
    wl = W._build("cascade_d256", 421, 16, 4, 256, bs, q_lens, [P + s for s in suffix], g,
                  shared_prefix_pages=P // bs)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out, lse, _ = run_gpu(wl, cascade=True, status=status)
    ref_o, ref_l = oracle_full(wl, cascade=True)
    assert_close(out, lse, ref_o, ref_l)
    assert int(status.item()) == 0


def test_sinks_and_update_entry_d256():
    wl = W.random_case(431, num_seqs=3, num_heads=8, num_kv_heads=2, head_size=256,
                       block_size=16, max_q=140, max_kv=400, decode_frac=0.3)
    sinks = torch.linspace(-2.0, 3.0, wl.num_heads, dtype=torch.float32)
    d = to_dev(wl, DEV)
    out, lse = pa.varlen_fwd_with_update(d["k_new"], d["v_new"], d["slot_mapping"], d["q"],
                                         d["key_cache"], d["value_cache"], d["cu_seqlens_q"],
                                         d["seqused_k"], d["block_table"], wl.max_seqlen_q,
                                         wl.max_seqlen_k, wl.softmax_scale, wl.causal,
                                         sinks=sinks.to(DEV))
    torch.cuda.synchronize()
    kc, vc = oracle_pools(wl)
    ref_o, ref_l = oracle.varlen_attention(wl.q, kc, vc, wl.cu_seqlens_q, wl.seqused_k,
                                           wl.block_table, wl.softmax_scale, wl.causal,
                                           sinks=sinks)
    assert_close(out, lse, ref_o, ref_l)


def test_decode_batch_d256_sampled():
    """A decode batch at head size 256 (64 sequences, KV lengths U[512, 8192],
    32/8 heads), checked on sampled sequences."""
    g = torch.Generator().manual_seed(441)
    kv = [int(x) for x in torch.randint(512, 8193, (64,), generator=g)]
    wl = W._build("decode_d256", 441, 32, 8, 256, 16, [1] * 64, kv, g)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out, lse, _ = run_gpu(wl, status=status)
    ref = oracle_sampled(wl, {0: [0], 21: [0], 63: [0]})
    for s, (tok, ro, rl) in ref.items():
        assert_close(out, lse, ro, rl, tokens=tok)
    assert int(status.item()) == 0


def test_d256_refusals():
    """Head size 256 runs on the prefill kernel only: a non-positive scale or
    a group of more than 128 heads is refused before any launch."""
    wl = W.random_case(451, num_seqs=2, num_heads=4, num_kv_heads=2, head_size=256)
    d = to_dev(wl, DEV)
    for scale in (0.0, -0.5):
        with pytest.raises(pa.PAError) as e:
            pa.varlen_fwd(d["q"], d["key_cache"], d["value_cache"], d["cu_seqlens_q"],
                          d["seqused_k"], d["block_table"], wl.max_seqlen_q, wl.max_seqlen_k,
                          scale, True)
        assert e.value.code == pa.PA_ERR_UNSUPPORTED


@pytest.mark.parametrize("name,seqs", [
    ("decode_d256", {0: [0], 31: [0], 63: [0]}),
    ("prefill_d256", {0: [0, 1, 1023, 2047], 3: [5, 2046]}),
])
def test_d256_bench_workloads_sampled(name, seqs):
    """The head-size-256 workloads the bench times (16/8 heads): the full
    batch on the GPU, sampled query rows against the oracle."""
    wl = W.CONFIGS[name]()
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out, lse, _ = run_gpu(wl, status=status)
    ref = oracle_sampled(wl, seqs)
    for s, (tok, ro, rl) in ref.items():
        assert_close(out, lse, ro, rl, tokens=tok)
    assert int(status.item()) == 0
