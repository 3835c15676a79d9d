"""GPU parity at the edges of the boundary: every GQA ratio the pages allow
(num_heads a multiple of num_kv_heads, "AttentionBackend" 境界と失敗; the
group need not be a power of two) and any finite softmax scale (a caller
argument, zero and negative included). Same oracle and tolerances as the
other parity tests."""
import pytest
import torch

import paged_kv_varlen_attn_gb300 as pa
import workloads as W
from helpers import oracle_full, to_dev
from test_gpu_parity import DEV, assert_close, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_varlen_attn_gb300 import _build
    _build.build()
    pa.load_library()


GQA_CASES = [
    # seed, S, H, Hk, D, bs, max_q, max_kv, causal, decode_frac
    (201, 3, 24, 8, 128, 16, 150, 400, True, 0.3),    # G = 3: 126-row tiles, two items
    (202, 3, 40, 8, 128, 32, 120, 300, True, 0.3),    # G = 5: 125-row tiles
    (203, 2, 28, 4, 64, 16, 100, 300, False, 0.0),    # G = 7, non-causal, D = 64
    (204, 3, 12, 1, 64, 16, 60, 260, True, 0.3),      # G = 12: 120-row tiles
    (205, 2, 48, 1, 64, 16, 40, 300, True, 0.0),      # G = 48: 96-row tiles (2 tokens)
    (206, 2, 200, 1, 64, 16, 6, 200, True, 0.5),      # G = 200 > 128: split-KV kernel only
    (207, 3, 6, 2, 128, 128, 1, 5000, True, 1.0),     # G = 3 decode, long keys, KV splits
]


@pytest.mark.parametrize("case", GQA_CASES, ids=[str(c[0]) for c in GQA_CASES])
def test_any_gqa_ratio(case):
    seed, S, H, Hk, D, bs, mq, mk, causal, dfrac = case
    wl = W.random_case(seed, num_seqs=S, num_heads=H, num_kv_heads=Hk, head_size=D,
                       block_size=bs, max_q=mq, max_kv=mk, causal=causal, decode_frac=dfrac)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out, lse, _ = run_gpu(wl, status=status)
    ref_o, ref_l = oracle_full(wl)
    assert_close(out, lse, ref_o, ref_l)
    assert int(status.item()) == 0


def _case_with_scale(seed, scale, H=8, Hk=2, D=128, q_lens=(1, 90, 3, 200), kv=(300, 260, 40,
                                                                               500)):
    g = torch.Generator().manual_seed(seed)
    return W._build(f"scale_{seed}", seed, H, Hk, D, 16, list(q_lens), list(kv), g, scale=scale)


@pytest.mark.parametrize("scale", [0.0, -0.0884, -0.3, 1e-30])
def test_any_finite_softmax_scale(scale):
    """Zero and negative scales (and a tiny positive one) on a batch with
    decode rows and multi-tile prefill rows."""
    wl = _case_with_scale(211, scale)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out, lse, _ = run_gpu(wl, status=status)
    ref_o, ref_l = oracle_full(wl)
    assert_close(out, lse, ref_o, ref_l)
    assert int(status.item()) == 0


@pytest.mark.parametrize("H,Hk,scale", [(24, 8, 0.0884), (40, 8, 0.0884), (8, 2, -0.2)])
def test_cascade_any_ratio_and_scale(H, Hk, scale):
    """Cascade (prefix pass over every query token, suffix pass, combine) with
    a non-power-of-two group and with a negative scale."""
    g = torch.Generator().manual_seed(221)
    S, P, bs = 40, 256, 16
    suffix = [int(x) for x in torch.randint(5, 120, (S,), generator=g)]
    q_lens = [min(int(x), s) for x, s in zip(torch.randint(1, 5, (S,), generator=g), suffix)]
    wl = W._build("cascade_boundary", 221, H, Hk, 128, bs, q_lens, [P + s for s in suffix], g,
                  shared_prefix_pages=P // bs, scale=scale)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out, lse, _ = run_gpu(wl, cascade=True, status=status)
    ref_o, ref_l = oracle_full(wl, cascade=True)
    assert_close(out, lse, ref_o, ref_l)
    assert int(status.item()) == 0


def test_non_pow2_group_update_entry_matches_separate_calls():
    """The update-and-attend entry with G = 5 equals the scatter followed by
    the attention call, bitwise."""
    wl = W.random_case(231, num_seqs=4, num_heads=40, num_kv_heads=8, head_size=128,
                       block_size=16, max_q=150, max_kv=400, decode_frac=0.3)
    d1, d2 = to_dev(wl, DEV), to_dev(wl, DEV)
    o1, l1, _ = run_gpu(wl, d1)
    o2, l2 = pa.varlen_fwd_with_update(d2["k_new"], d2["v_new"], d2["slot_mapping"], d2["q"],
                                       d2["key_cache"], d2["value_cache"], d2["cu_seqlens_q"],
                                       d2["seqused_k"], d2["block_table"], wl.max_seqlen_q,
                                       wl.max_seqlen_k, wl.softmax_scale, wl.causal)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
