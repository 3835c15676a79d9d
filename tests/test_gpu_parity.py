"""GPU parity: the CUDA path through the C ABI against the fp64 oracle on the
same seeded inputs. Scatter and indexing bit-exact; bf16 outputs within 1e-2
max-abs and LSE within 1e-3 absolute."""
import math

import pytest
import torch

import oracle
import paged_kv_varlen_attn_gb300 as pa
import workloads as W
from helpers import LSE_TOL, OUT_TOL, oracle_full, oracle_pools, oracle_sampled, to_dev

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_varlen_attn_gb300 import _build
    _build.build()
    pa.load_library()


def run_gpu(wl, d=None, causal=None, cascade=False, status=None):
    d = d or to_dev(wl, DEV)
    pa.reshape_and_cache(d["k_new"], d["v_new"], d["key_cache"], d["value_cache"],
                         d["slot_mapping"], dev_status=status)
    args = (d["q"], d["key_cache"], d["value_cache"], d["cu_seqlens_q"], d["seqused_k"],
            d["block_table"], max(wl.max_seqlen_q, 1), wl.max_seqlen_k, wl.softmax_scale)
    if cascade:
        out, lse = pa.cascade_fwd(*args, wl.common_prefix_len, dev_status=status)
    else:
        out, lse = pa.varlen_fwd(*args, wl.causal if causal is None else causal,
                                 dev_status=status)
    torch.cuda.synchronize()
    return out, lse, d


def assert_close(out, lse, ref_o, ref_l, tokens=None):
    o = out.cpu().double()
    l = lse.cpu().double()
    if tokens is not None:
        o, l = o[tokens], l[:, tokens]
    fin = torch.isfinite(ref_l)
    assert torch.equal(fin, torch.isfinite(l)), "rows without keys must have lse = -inf"
    err_o = (o - ref_o).abs().max().item() if o.numel() else 0.0
    err_l = (l[fin] - ref_l[fin]).abs().max().item() if fin.any() else 0.0
    assert err_o <= OUT_TOL, f"out max-abs err {err_o}"
    assert err_l <= LSE_TOL, f"lse abs err {err_l}"
    return err_o, err_l


# ---------------------------------------------------------------- scatter
def test_scatter_bit_exact_tiny_mixed():
    wl = W.tiny_mixed()
    kc_ref, vc_ref = oracle_pools(wl)
    d = to_dev(wl, DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    pa.reshape_and_cache(d["k_new"], d["v_new"], d["key_cache"], d["value_cache"],
                         d["slot_mapping"], dev_status=status)
    torch.cuda.synchronize()
    assert torch.equal(d["key_cache"].cpu(), kc_ref)
    assert torch.equal(d["value_cache"].cpu(), vc_ref)
    assert int(status.item()) == 0


@pytest.mark.parametrize("seed,bs,D,Hk", [(21, 16, 128, 8), (22, 32, 64, 2), (23, 128, 128, 1),
                                          (24, 48, 64, 4)])
def test_scatter_padding_and_canary(seed, bs, D, Hk):
    wl = W.random_case(seed, num_seqs=6, num_heads=Hk * 2, num_kv_heads=Hk, head_size=D,
                       block_size=bs, max_q=50, max_kv=300)
    slots = wl.slot_mapping.clone()
    slots[::3] = -1
    canary = torch.full((wl.num_blocks, bs, Hk, D), -3.5, dtype=torch.bfloat16)
    kc_ref, vc_ref = canary.clone(), canary.clone()
    oracle.reshape_and_cache(wl.k_new, wl.v_new, slots, kc_ref, vc_ref)
    kc, vc = canary.to(DEV), canary.to(DEV)
    pa.reshape_and_cache(wl.k_new.to(DEV), wl.v_new.to(DEV), kc, vc, slots.to(DEV))
    torch.cuda.synchronize()
    assert torch.equal(kc.cpu(), kc_ref) and torch.equal(vc.cpu(), vc_ref)


def test_scatter_combined_kv_layout():
    """K and V as views of one [num_blocks, 2, block_size, H_kv, D] tensor."""
    wl = W.random_case(25, num_seqs=4, num_heads=8, num_kv_heads=4, head_size=128,
                       block_size=16, max_q=30, max_kv=100)
    kc_ref, vc_ref = oracle_pools(wl)
    both = torch.stack([wl.pool(0), wl.pool(1)], dim=1).to(DEV)
    kc, vc = both[:, 0], both[:, 1]
    pa.reshape_and_cache(wl.k_new.to(DEV), wl.v_new.to(DEV), kc, vc, wl.slot_mapping.to(DEV))
    out, lse = pa.varlen_fwd(wl.q.to(DEV), kc, vc, wl.cu_seqlens_q.to(DEV),
                             wl.seqused_k.to(DEV), wl.block_table.to(DEV), wl.max_seqlen_q,
                             wl.max_seqlen_k, wl.softmax_scale, True)
    torch.cuda.synchronize()
    assert torch.equal(kc.cpu(), kc_ref) and torch.equal(vc.cpu(), vc_ref)
    ref_o, ref_l = oracle.varlen_attention(wl.q, kc_ref, vc_ref, wl.cu_seqlens_q, wl.seqused_k,
                                           wl.block_table, wl.softmax_scale, True)
    assert_close(out, lse, ref_o, ref_l)


def test_scatter_bad_slot_is_flagged_and_skipped():
    wl = W.random_case(26, num_seqs=3, num_heads=4, num_kv_heads=2, head_size=64, block_size=16)
    slots = wl.slot_mapping.clone()
    slots[0] = wl.num_blocks * wl.block_size + 5     # past the pool
    kc_ref, vc_ref = wl.pool(0), wl.pool(1)
    ok = slots.clone()
    ok[0] = -1
    oracle.reshape_and_cache(wl.k_new, wl.v_new, ok, kc_ref, vc_ref)
    kc, vc = wl.pool(0).to(DEV), wl.pool(1).to(DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    pa.reshape_and_cache(wl.k_new.to(DEV), wl.v_new.to(DEV), kc, vc, slots.to(DEV),
                         dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & pa.PA_DEV_BAD_SLOT
    assert torch.equal(kc.cpu(), kc_ref) and torch.equal(vc.cpu(), vc_ref)


# ---------------------------------------------------------------- varlen
def test_tiny_mixed_config():
    wl = W.tiny_mixed()
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out, lse, _ = run_gpu(wl, status=status)
    ref_o, ref_l = oracle_full(wl)
    assert_close(out, lse, ref_o, ref_l)
    assert int(status.item()) == 0


CASES = [
    # seed, S, H, Hk, D, bs, max_q, max_kv, causal, decode_frac
    (101, 5, 4, 2, 64, 16, 40, 150, True, 0.3),
    (102, 4, 8, 2, 128, 16, 70, 300, True, 0.5),
    (103, 3, 8, 8, 128, 32, 90, 200, False, 0.3),
    (104, 6, 16, 2, 64, 64, 20, 400, True, 0.5),
    (105, 4, 32, 4, 128, 128, 33, 700, True, 0.5),
    (106, 3, 16, 1, 128, 48, 17, 260, True, 0.0),     # MQA-like group of 16, bs 48
    (107, 5, 8, 4, 64, 16, 130, 260, False, 0.2),
    (108, 4, 4, 4, 128, 80, 65, 500, True, 0.25),     # G = 1, bs 80
    (109, 2, 8, 2, 128, 16, 300, 1100, True, 0.0),    # multi-tile causal prefill, prior context
    (110, 2, 16, 2, 64, 32, 260, 700, False, 0.0),    # multi-tile non-causal, D = 64
    (111, 3, 32, 8, 128, 128, 200, 900, True, 0.0),   # GQA 4, block 128
    (112, 4, 8, 2, 128, 16, 1, 6000, True, 1.0),      # decode, long keys: many KV splits
    (113, 3, 16, 2, 64, 32, 8, 4000, True, 0.0),      # up to 64 packed rows, split KV
]


@pytest.mark.parametrize("case", CASES, ids=[str(c[0]) for c in CASES])
def test_random_varlen_cases(case):
    seed, S, H, Hk, D, bs, mq, mk, causal, dfrac = case
    wl = W.random_case(seed, num_seqs=S, num_heads=H, num_kv_heads=Hk, head_size=D,
                       block_size=bs, max_q=mq, max_kv=mk, causal=causal, decode_frac=dfrac)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out, lse, _ = run_gpu(wl, status=status)
    ref_o, ref_l = oracle_full(wl)
    assert_close(out, lse, ref_o, ref_l)
    assert int(status.item()) == 0


def test_empty_and_keyless_rows():
    """q_len = 0 sequences, kv_len = 0 sequences, and causal rows with no
    visible key (q_len > kv_len) give out 0 and lse -inf."""
    H, Hk, D, bs = 8, 2, 64, 16
    g = torch.Generator().manual_seed(31)
    q_lens = [0, 3, 5, 1, 0]
    kv_lens = [20, 0, 2, 40, 0]
    T = sum(q_lens)
    nb = 8
    kc = torch.randn(nb, bs, Hk, D, generator=g).to(torch.bfloat16)
    vc = torch.randn(nb, bs, Hk, D, generator=g).to(torch.bfloat16)
    q = torch.randn(T, H, D, generator=g).to(torch.bfloat16)
    bt = torch.tensor([[0, 1, 7], [2, 7, 7], [3, 7, 7], [4, 5, 6], [7, 7, 7]], dtype=torch.int32)
    cu = torch.tensor([0, 0, 3, 8, 9, 9], dtype=torch.int32)
    lens = torch.tensor(kv_lens, dtype=torch.int32)
    ref_o, ref_l = oracle.varlen_attention(q, kc, vc, cu, lens, bt, 0.125, True)
    out, lse = pa.varlen_fwd(q.to(DEV), kc.to(DEV), vc.to(DEV), cu.to(DEV), lens.to(DEV),
                             bt.to(DEV), 5, 40, 0.125, True)
    torch.cuda.synchronize()
    assert_close(out, lse, ref_o, ref_l)
    assert bool(torch.isinf(lse[:, :3].cpu()).all())       # seq 1 has no keys


def test_page_permutation_invariance_bitwise():
    wl = W.random_case(41, num_seqs=4, num_heads=8, num_kv_heads=2, head_size=128,
                       block_size=16, max_q=40, max_kv=500)
    kc_ref, vc_ref = oracle_pools(wl)
    out1, lse1 = pa.varlen_fwd(wl.q.to(DEV), kc_ref.to(DEV), vc_ref.to(DEV),
                               wl.cu_seqlens_q.to(DEV), wl.seqused_k.to(DEV),
                               wl.block_table.to(DEV), wl.max_seqlen_q, wl.max_seqlen_k,
                               wl.softmax_scale, True)
    from test_oracle_pins import contiguous_copy
    bt2, kc2, vc2 = contiguous_copy(wl, kc_ref, vc_ref)
    out2, lse2 = pa.varlen_fwd(wl.q.to(DEV), kc2.to(DEV), vc2.to(DEV), wl.cu_seqlens_q.to(DEV),
                               wl.seqused_k.to(DEV), bt2.to(DEV), wl.max_seqlen_q,
                               wl.max_seqlen_k, wl.softmax_scale, True)
    torch.cuda.synchronize()
    assert torch.equal(out1, out2) and torch.equal(lse1, lse2)


def test_deterministic_bitwise():
    wl = W.decode_llama8b(num_seqs=8)
    d = to_dev(wl, DEV)
    o1, l1, d = run_gpu(wl, d)
    args = (d["q"], d["key_cache"], d["value_cache"], d["cu_seqlens_q"], d["seqused_k"],
            d["block_table"], 1, wl.max_seqlen_k, wl.softmax_scale, True)
    o2, l2 = pa.varlen_fwd(*args)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_bad_page_is_flagged_not_read():
    wl = W.random_case(51, num_seqs=3, num_heads=4, num_kv_heads=2, head_size=64,
                       block_size=16, max_q=10, max_kv=60, decode_frac=1.0)
    kc, vc = oracle_pools(wl)
    bt = wl.block_table.clone()
    bt[0, 0] = wl.num_blocks + 1000       # out of the pool
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out, lse = pa.varlen_fwd(wl.q.to(DEV), kc.to(DEV), vc.to(DEV), wl.cu_seqlens_q.to(DEV),
                             wl.seqused_k.to(DEV), bt.to(DEV), wl.max_seqlen_q, wl.max_seqlen_k,
                             wl.softmax_scale, True, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & pa.PA_DEV_BAD_PAGE
    assert bool(torch.isfinite(out.float()).all())


def test_key_bound_sizes_launches_not_results():
    """The caller's key bound only sizes the launches and the workspace; the
    plan follows the lengths themselves. A bound four times too large gives
    bitwise the same outputs, for a cascade over decode suffixes and for a
    decode batch."""
    for wl, cascade in ((W.cascade_shared_prefix(num_seqs=16), True),
                        (W.decode_llama8b(num_seqs=8), False)):
        d = to_dev(wl, DEV)
        pa.reshape_and_cache(d["k_new"], d["v_new"], d["key_cache"], d["value_cache"],
                             d["slot_mapping"])
        res = []
        for max_k in (wl.max_seqlen_k, 4 * wl.max_seqlen_k):
            args = (d["q"], d["key_cache"], d["value_cache"], d["cu_seqlens_q"], d["seqused_k"],
                    d["block_table"], max(wl.max_seqlen_q, 1), max_k, wl.softmax_scale)
            status = torch.zeros(1, dtype=torch.int32, device=DEV)
            if cascade:
                res.append(pa.cascade_fwd(*args, wl.common_prefix_len, dev_status=status))
            else:
                res.append(pa.varlen_fwd(*args, True, dev_status=status))
            torch.cuda.synchronize()
            assert int(status.item()) == 0
        assert torch.equal(res[0][0], res[1][0]) and torch.equal(res[0][1], res[1][1])


def test_back_to_back_calls_share_a_workspace():
    """Calls queued on one stream with one workspace and no host sync between
    them: each call's planner is launched normally, so it starts only once the
    previous call's kernels (chained by programmatic dependent launch inside
    the call) have all completed. A decode batch, a cascade and a mixed batch
    in a row give bitwise the outputs of the same calls made one at a time."""
    sms = torch.cuda.get_device_properties(DEV).multi_processor_count
    wls = [(W.decode_llama8b(num_seqs=8), False),
           (W.cascade_shared_prefix(num_seqs=8), True),
           (W.random_case(53, num_seqs=5, num_heads=8, num_kv_heads=2, head_size=128,
                          block_size=16, max_q=70, max_kv=300, decode_frac=0.4), False)]
    calls, need = [], 0
    for wl, cascade in wls:
        d = to_dev(wl, DEV)
        pa.reshape_and_cache(d["k_new"], d["v_new"], d["key_cache"], d["value_cache"],
                             d["slot_mapping"])
        T, H, D = wl.q.shape
        size = (pa.cascade_fwd_workspace_size if cascade else pa.varlen_fwd_workspace_size)(
            wl.num_seqs, T, max(wl.max_seqlen_q, 1), wl.max_seqlen_k, H, wl.num_kv_heads, D,
            wl.block_size, sms)
        need = max(need, size)
        calls.append((wl, cascade, d))
    ws = pa.alloc_workspace(need, DEV)

    def call(wl, cascade, d):
        args = (d["q"], d["key_cache"], d["value_cache"], d["cu_seqlens_q"], d["seqused_k"],
                d["block_table"], max(wl.max_seqlen_q, 1), wl.max_seqlen_k, wl.softmax_scale)
        if cascade:
            return pa.cascade_fwd(*args, wl.common_prefix_len, workspace=ws)
        return pa.varlen_fwd(*args, wl.causal, workspace=ws)

    alone = []
    for c in calls:
        alone.append(call(*c))
        torch.cuda.synchronize()
    queued = [call(*c) for c in calls]
    torch.cuda.synchronize()
    for (o1, l1), (o2, l2) in zip(alone, queued):
        assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_keys_above_bound_are_flagged():
    """A sequence with more keys than the caller's bound is a caller error
    the planner reports (PA_DEV_BAD_SEQLEN); the block table it reads stays
    within its rows."""
    wl = W.random_case(52, num_seqs=4, num_heads=4, num_kv_heads=2, head_size=64,
                       block_size=16, max_q=1, max_kv=100, decode_frac=1.0)
    d = to_dev(wl, DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    pa.varlen_fwd(d["q"], d["key_cache"], d["value_cache"], d["cu_seqlens_q"], d["seqused_k"],
                  d["block_table"], max(wl.max_seqlen_q, 1), wl.max_seqlen_k - 1,
                  wl.softmax_scale, True, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & pa.PA_DEV_BAD_SEQLEN


def test_workspace_too_small_is_rejected():
    wl = W.tiny_mixed()
    d = to_dev(wl, DEV)
    ws = torch.empty(1024, dtype=torch.uint8, device=DEV)
    with pytest.raises(pa.PAError) as e:
        pa.varlen_fwd(d["q"], d["key_cache"], d["value_cache"], d["cu_seqlens_q"],
                      d["seqused_k"], d["block_table"], wl.max_seqlen_q, wl.max_seqlen_k,
                      wl.softmax_scale, True, workspace=ws)
    assert e.value.code == pa.PA_ERR_WORKSPACE


# ---------------------------------------------------------------- merge
def test_merge_matches_oracle_and_aliases():
    g = torch.Generator().manual_seed(61)
    T, H, D = 37, 8, 128
    oa = torch.randn(T, H, D, generator=g).to(torch.bfloat16)
    ob = torch.randn(T, H, D, generator=g).to(torch.bfloat16)
    a = torch.randn(H, T, generator=g) * 3
    b = torch.randn(H, T, generator=g) * 3
    a[0, :5] = float("-inf")
    b[0, 3:8] = float("-inf")
    ref_o, ref_l = oracle.merge_attn_states(oa, a, ob, b)
    out, lse = pa.merge_attn_states(oa.to(DEV), a.to(DEV), ob.to(DEV), b.to(DEV))
    torch.cuda.synchronize()
    assert_close(out, lse, ref_o, ref_l)
    oad = oa.to(DEV)
    pa.merge_attn_states(oad, a.to(DEV), ob.to(DEV), b.to(DEV), out=oad, return_lse=False)
    torch.cuda.synchronize()
    assert torch.equal(oad, out)


def test_split_kv_states_merge_to_full():
    """Two varlen calls on disjoint key ranges (the second through a shifted
    block table) merged by pa_merge_attn_states equal one call over all keys
    (the DCP-style split of "FlashAttention 在 vLLM 中的实现分析" §9)."""
    wl = W.random_case(62, num_seqs=4, num_heads=8, num_kv_heads=2, head_size=128,
                       block_size=16, max_q=1, max_kv=600, decode_frac=1.0)
    kc, vc = oracle_pools(wl)
    cut_pages = 10
    c = cut_pages * wl.block_size
    lens = wl.seqused_k.clone()
    lens_a = torch.minimum(lens, torch.tensor(c, dtype=torch.int32))
    lens_b = lens - lens_a
    bt_b = torch.full_like(wl.block_table, W.INT32_MAX)
    bt_b[:, :wl.block_table.shape[1] - cut_pages] = wl.block_table[:, cut_pages:]
    dk, dv = kc.to(DEV), vc.to(DEV)
    q, cu = wl.q.to(DEV), wl.cu_seqlens_q.to(DEV)
    oa, la = pa.varlen_fwd(q, dk, dv, cu, lens_a.to(DEV), wl.block_table.to(DEV), 1, c,
                           wl.softmax_scale, False)
    ob, lb = pa.varlen_fwd(q, dk, dv, cu, lens_b.to(DEV), bt_b.to(DEV), 1, wl.max_seqlen_k,
                           wl.softmax_scale, False)
    mo, ml = pa.merge_attn_states(oa, la, ob, lb)
    torch.cuda.synchronize()
    ref_o, ref_l = oracle.varlen_attention(wl.q, kc, vc, wl.cu_seqlens_q, wl.seqused_k,
                                           wl.block_table, wl.softmax_scale, False)
    assert_close(mo, ml, ref_o, ref_l)


# ---------------------------------------------------------------- cascade
def test_cascade_small_matches_flat():
    g = torch.Generator().manual_seed(71)
    S, P, bs = 9, 96, 16
    suffix = [int(x) for x in torch.randint(5, 80, (S,), generator=g)]
    q_lens = [min(int(x), s) for x, s in zip(torch.randint(1, 4, (S,), generator=g), suffix)]
    wl = W._build("cascade_small", 71, 8, 2, 128, bs, q_lens, [P + s for s in suffix], g,
                  shared_prefix_pages=P // bs)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out, lse, _ = run_gpu(wl, cascade=True, status=status)
    ref_o, ref_l = oracle_full(wl, cascade=True)
    assert_close(out, lse, ref_o, ref_l)
    assert int(status.item()) == 0


@pytest.mark.parametrize("seed,S,H,Hk,D,P,qmax,smax", [
    (72, 4, 8, 2, 128, 64, 1, 40),       # prefix pass rows 4*4 = 16: split-KV kernel
    (73, 40, 32, 4, 128, 512, 2, 200),   # prefix rows 61*8 = 488: two 256-row tiles
    (74, 12, 16, 16, 64, 256, 3, 90),    # GQA 1, head 64
    (75, 40, 32, 4, 128, 256, 4, 100),   # prefix rows 99*8 = 792: four row tiles, last partial
])
def test_cascade_prefix_row_tiles(seed, S, H, Hk, D, P, qmax, smax):
    g = torch.Generator().manual_seed(seed)
    suffix = [int(x) for x in torch.randint(qmax + 1, smax, (S,), generator=g)]
    q_lens = [int(x) for x in torch.randint(1, qmax + 1, (S,), generator=g)]
    wl = W._build(f"cascade_{seed}", seed, H, Hk, D, 16, q_lens, [P + s for s in suffix], g,
                  shared_prefix_pages=P // 16)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out, lse, _ = run_gpu(wl, cascade=True, status=status)
    ref_o, ref_l = oracle_full(wl, cascade=True)
    assert_close(out, lse, ref_o, ref_l)
    assert int(status.item()) == 0


def test_cascade_shared_prefix_config():
    wl = W.cascade_shared_prefix()
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out, lse, _ = run_gpu(wl, cascade=True, status=status)
    ref_o, ref_l = oracle_full(wl, cascade=True)
    assert_close(out, lse, ref_o, ref_l)
    assert int(status.item()) == 0


# ---------------------------------------------------------------- full-size configs
def _sample_rows(wl, seqs, per_seq=24, seed=0):
    g = torch.Generator().manual_seed(seed)
    rows = {}
    for s in seqs:
        n = wl.q_lens[s]
        if n <= per_seq:
            rows[s] = list(range(n))
        else:
            pick = {0, n - 1, n // 2, 63, 64, 127, 128}
            pick |= set(int(x) for x in torch.randint(0, n, (per_seq,), generator=g))
            rows[s] = sorted(p for p in pick if p < n)
    return rows


@pytest.mark.parametrize("name,seqs", [
    ("decode_llama8b", [0, 17, 63]),
    ("chunked_prefill_mix", [0, 7, 8, 40, 63]),
    ("long_context_70b", [0, 31, 32, 35]),
])
def test_full_size_config_sampled(name, seqs):
    wl = W.CONFIGS[name]()
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out, lse, _ = run_gpu(wl, status=status)
    rows = _sample_rows(wl, seqs)
    ref = oracle_sampled(wl, rows)
    for s, (tok, ro, rl) in ref.items():
        assert_close(out, lse, ro, rl, tokens=tok)
    assert int(status.item()) == 0


# ---------------------------------------------------------------- size edges
def test_many_sequences_planner_global_tables():
    """More sequences than the planner keeps in shared memory (1,024): its
    segment tables live in the workspace instead; mixed decode and short
    prefill rows, ragged lengths."""
    g = torch.Generator().manual_seed(91)
    S = 1100
    kv = [int(x) for x in torch.randint(1, 160, (S,), generator=g)]
    ql = [1 if float(torch.rand((1,), generator=g)) < 0.8 else min(k, int(torch.randint(2, 24, (1,), generator=g)))
          for k in kv]
    wl = W._build("many_seqs", 91, 8, 2, 64, 16, ql, kv, g)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out, lse, _ = run_gpu(wl, status=status)
    ref_o, ref_l = oracle_full(wl)
    assert_close(out, lse, ref_o, ref_l)
    assert int(status.item()) == 0


def test_long_context_decode_many_splits():
    """Two decode sequences of 131,072 and 65,535 keys: one row tile split
    into many KV chunks whose partial states the last CTA merges."""
    g = torch.Generator().manual_seed(92)
    wl = W._build("long_decode", 92, 32, 8, 128, 16, [1, 1], [131072, 65535], g)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out, lse, _ = run_gpu(wl, status=status)
    ref = oracle_sampled(wl, {0: [0], 1: [0]})
    for s, (tokens, ro, rl) in ref.items():
        assert_close(out, lse, ro, rl, tokens=tokens)
    assert int(status.item()) == 0
