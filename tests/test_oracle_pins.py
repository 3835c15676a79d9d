"""Pins for the fp64 oracle: every function is checked against something other
than itself (hand-derived fixtures, brute-force loops, closed forms, a torch
library routine, invariants). CPU only.

Sources: "FlashAttention 在 vLLM 中的实现分析" (§1.1 online softmax target,
§4.2 scatter, §5 paged addressing, §6.3 cascade and merge) and
"AttentionBackend:アテンションバックエンド抽象レイヤー" (境界と失敗: natural-log
LSE).
"""
import json
import math
import os

import pytest
import torch

import oracle
from oracle import paged_attention as P
import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_examples.json")
F64 = torch.float64


def golden():
    with open(GOLDEN) as f:
        return json.load(f)


def _ln(expr):
    return {"0": 0.0, "ln(3)": math.log(3.0), "ln(4)": math.log(4.0)}[expr]


# ----------------------------------------------------------------------------
# Pin checks, written as functions so the mutation tests below can run them
# against an oracle with a planted mistake.
# ----------------------------------------------------------------------------
def check_golden_merge():
    g = golden()["merge"]
    oa = torch.tensor(g["prefix_out"], dtype=F64).view(1, 1, -1)
    ob = torch.tensor(g["suffix_out"], dtype=F64).view(1, 1, -1)
    a = torch.tensor([[_ln(g["prefix_lse"])]], dtype=F64)
    b = torch.tensor([[_ln(g["suffix_lse"])]], dtype=F64)
    o, l = oracle.merge_attn_states(oa, a, ob, b)
    assert torch.allclose(o.view(-1), torch.tensor(g["expected_out"], dtype=F64), atol=1e-14)
    assert abs(float(l) - _ln(g["expected_lse"])) < 1e-14


def check_golden_two_key():
    g = golden()["two_key_attention"]
    q = torch.tensor(g["q"], dtype=F64).view(1, 1, 2)
    k = torch.tensor(g["k"], dtype=F64).view(2, 1, 2)
    v = torch.tensor(g["v"], dtype=F64).view(2, 1, 2)
    o, l = oracle.attend_dense(q, k, v, g["softmax_scale"], False, 1, 2)
    e4 = math.exp(4.0)
    exp_o = [(1 - e4) / (1 + e4), (3 + 5 * e4) / (1 + e4)]
    assert torch.allclose(o.view(-1), torch.tensor(exp_o, dtype=F64), atol=1e-14)
    assert abs(float(l) - math.log(1 + e4)) < 1e-13


def visible_matrix(q_len, kv_len, causal=True):
    """Which keys each row sees, read off the oracle: with Q = 0 every visible
    key gets the same weight, and V = one-hot key indicators."""
    D = max(kv_len, 1)
    q = torch.zeros((q_len, 1, D), dtype=F64)
    k = torch.randn((kv_len, 1, D), dtype=F64)
    v = torch.eye(kv_len, D, dtype=F64).view(kv_len, 1, D)
    o, _ = oracle.attend_dense(q, k, v, 1.0, causal, q_len, kv_len)
    return (o[:, 0, :kv_len] > 0).to(torch.int64)


def check_golden_causal():
    g = golden()["bottom_right_causal"]
    vis = visible_matrix(g["q_len"], g["kv_len"])
    assert vis.tolist() == g["visible"]


def check_golden_paged_address():
    g = golden()["paged_address"]
    bt = torch.tensor(g["block_table_row"], dtype=torch.int32)
    pages, rows = P.logical_to_physical(bt, g["positions"], g["block_size"])
    assert [[int(p), int(r)] for p, r in zip(pages, rows)] == g["expected_page_row"]


def check_lse_fsum(seed=0):
    """LSE against a direct ln(sum exp) with math.fsum on tiny inputs."""
    torch.manual_seed(seed)
    q_len, kv_len, H, D = 3, 7, 2, 5
    q = torch.randn(q_len, H, D, dtype=F64)
    k = torch.randn(kv_len, 1, D, dtype=F64)
    v = torch.randn(kv_len, 1, D, dtype=F64)
    scale = 0.37
    _, lse = oracle.attend_dense(q, k, v, scale, True, q_len, kv_len)
    for h in range(H):
        for i in range(q_len):
            last = kv_len - q_len + i
            logits = [scale * math.fsum(float(q[i, h, d]) * float(k[j, 0, d]) for d in range(D))
                      for j in range(last + 1)]
            ref = math.log(math.fsum(math.exp(x) for x in logits))
            assert abs(float(lse[h, i]) - ref) < 1e-12, (h, i, float(lse[h, i]), ref)


def brute_attention(q, k, v, scale, causal):
    """Explicit loops over (i, j): the textbook definition, float64."""
    q_len, H, D = q.shape
    kv_len, H_kv, _ = k.shape
    G = H // H_kv
    out = [[[0.0] * D for _ in range(H)] for _ in range(q_len)]
    lse = [[float("-inf")] * q_len for _ in range(H)]
    for i in range(q_len):
        for h in range(H):
            hk = h // G
            js = [j for j in range(kv_len) if (not causal) or j <= kv_len - q_len + i]
            if not js:
                continue
            logits = {j: scale * math.fsum(float(q[i, h, d]) * float(k[j, hk, d])
                                           for d in range(D)) for j in js}
            m = max(logits.values())
            w = {j: math.exp(logits[j] - m) for j in js}
            den = math.fsum(w.values())
            for d in range(D):
                out[i][h][d] = math.fsum(w[j] * float(v[j, hk, d]) for j in js) / den
            lse[h][i] = m + math.log(den)
    return torch.tensor(out, dtype=F64), torch.tensor(lse, dtype=F64)


def check_brute_force(max_len=6, seed=1, H=4, H_kv=2, D=3):
    g = torch.Generator().manual_seed(seed)
    for causal in (True, False):
        for kv_len in range(1, max_len + 1):
            for q_len in range(1, max_len + 1):
                q = torch.randn(q_len, H, D, generator=g, dtype=F64)
                k = torch.randn(kv_len, H_kv, D, generator=g, dtype=F64)
                v = torch.randn(kv_len, H_kv, D, generator=g, dtype=F64)
                o, l = oracle.attend_dense(q, k, v, 0.8, causal, q_len, kv_len)
                bo, bl = brute_attention(q, k, v, 0.8, causal)
                assert torch.allclose(o, bo, atol=1e-12, rtol=0), (causal, q_len, kv_len)
                fin = torch.isfinite(bl)
                assert torch.equal(fin, torch.isfinite(l))
                assert torch.allclose(l[fin], bl[fin], atol=1e-12, rtol=0)


def contiguous_copy(wl, kc, vc):
    """The same batch laid out with sequence s's pages consecutive (identity
    block table). Returns (block_table, key_cache, value_cache)."""
    bs = wl.block_size
    pages = [wl.pages_of(s) for s in range(wl.num_seqs)]
    total = sum(len(p) for p in pages)
    kc2 = torch.zeros((max(total, 1),) + tuple(kc.shape[1:]), dtype=kc.dtype)
    vc2 = torch.zeros_like(kc2)
    bt2 = torch.full_like(wl.block_table, W.INT32_MAX)
    cur = 0
    for s, ps in enumerate(pages):
        for i, p in enumerate(ps):
            kc2[cur] = kc[p]
            vc2[cur] = vc[p]
            bt2[s, i] = cur
            cur += 1
    return bt2, kc2, vc2


def scattered_pools(wl):
    kc, vc = wl.pool(0, threads=1), wl.pool(1, threads=1)
    oracle.reshape_and_cache(wl.k_new, wl.v_new, wl.slot_mapping, kc, vc)
    return kc, vc


def check_sdpa(seed=5, causal=True):
    """Contiguous layout vs torch scaled_dot_product_attention (fp64, GQA via
    the library's enable_gqa, explicit bottom-right boolean mask)."""
    wl = W.random_case(seed, num_seqs=4, num_heads=8, num_kv_heads=2, head_size=32,
                       block_size=16, max_q=20, max_kv=70, causal=causal)
    kc, vc = scattered_pools(wl)
    out, lse = oracle.varlen_attention(wl.q, kc, vc, wl.cu_seqlens_q, wl.seqused_k,
                                       wl.block_table, wl.softmax_scale, causal)
    cu = wl.cu_seqlens_q.tolist()
    for s in range(wl.num_seqs):
        q_len, kv_len = wl.q_lens[s], wl.kv_lens[s]
        if q_len == 0 or kv_len == 0:
            continue
        k = P.gather_kv(kc, wl.block_table[s], kv_len).to(F64)
        v = P.gather_kv(vc, wl.block_table[s], kv_len).to(F64)
        qs = wl.q[cu[s]:cu[s + 1]].to(F64)
        mask = torch.ones(q_len, kv_len, dtype=torch.bool)
        if causal:
            mask = torch.ones(q_len, kv_len, dtype=torch.bool).tril(kv_len - q_len)
        ref = torch.nn.functional.scaled_dot_product_attention(
            qs.transpose(0, 1)[None], k.transpose(0, 1)[None], v.transpose(0, 1)[None],
            attn_mask=mask, scale=wl.softmax_scale, enable_gqa=True)[0].transpose(0, 1)
        assert torch.allclose(out[cu[s]:cu[s + 1]], ref, atol=1e-12, rtol=0), s
        # LSE: logsumexp of the masked logits through torch's own routine
        kk = k.repeat_interleave(wl.num_heads // wl.num_kv_heads, dim=1)
        logits = wl.softmax_scale * torch.einsum("ihd,jhd->hij", qs, kk)
        logits = logits.masked_fill(~mask[None], float("-inf"))
        assert torch.allclose(lse[:, cu[s]:cu[s + 1]], torch.logsumexp(logits, dim=-1),
                              atol=1e-12, rtol=0)


def check_permutation_invariance(seed=7):
    wl = W.random_case(seed, num_seqs=5, num_heads=4, num_kv_heads=2, head_size=16,
                       block_size=16, max_q=30, max_kv=90)
    kc, vc = scattered_pools(wl)
    o1, l1 = oracle.varlen_attention(wl.q, kc, vc, wl.cu_seqlens_q, wl.seqused_k,
                                     wl.block_table, wl.softmax_scale, True)
    bt2, kc2, vc2 = contiguous_copy(wl, kc, vc)
    o2, l2 = oracle.varlen_attention(wl.q, kc2, vc2, wl.cu_seqlens_q, wl.seqused_k,
                                     bt2, wl.softmax_scale, True)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


# ----------------------------------------------------------------------------
# The pins as tests.
# ----------------------------------------------------------------------------
def test_golden_merge():
    check_golden_merge()


def test_golden_two_key_attention():
    check_golden_two_key()


def test_golden_bottom_right_causal():
    check_golden_causal()


def test_golden_paged_address():
    check_golden_paged_address()


def test_golden_scatter_slots():
    g = golden()["scatter_slot"]
    bs = g["block_size"]
    kc = torch.zeros(4, bs, 1, 2)
    vc = torch.zeros(4, bs, 1, 2)
    n = len(g["slots"])
    key = torch.arange(1, n + 1, dtype=torch.float32).view(n, 1, 1).expand(n, 1, 2).clone()
    val = -key
    oracle.reshape_and_cache(key, val, torch.tensor(g["slots"]), kc, vc)
    for t, pr in enumerate(g["expected_page_row"]):
        if pr is None:
            assert not (kc == key[t, 0, 0]).any()
            continue
        assert torch.equal(kc[pr[0], pr[1]], key[t]) and torch.equal(vc[pr[0], pr[1]], val[t])
    assert int((kc != 0).any(dim=-1).sum()) == 3


def test_scatter_brute_force_and_canary():
    """Element-by-element Python reference over nested lists; every slot that no
    token targets keeps its canary value."""
    wl = W.random_case(11, num_seqs=4, num_heads=4, num_kv_heads=2, head_size=8,
                       block_size=16, max_q=20, max_kv=60)
    slots = wl.slot_mapping.clone()
    slots[::5] = -1                                     # padding tokens
    NB, bs, Hk, D = wl.num_blocks, wl.block_size, wl.num_kv_heads, wl.head_size
    canary = torch.full((NB, bs, Hk, D), 7.25, dtype=torch.bfloat16)
    kc, vc = canary.clone(), canary.clone()
    oracle.reshape_and_cache(wl.k_new, wl.v_new, slots, kc, vc)
    ref = [[[[7.25] * D for _ in range(Hk)] for _ in range(bs)] for _ in range(NB)]
    written = set()
    for t, slot in enumerate(slots.tolist()):
        if slot < 0:
            continue
        b, r = divmod(slot, bs)
        written.add((b, r))
        for h in range(Hk):
            for d in range(D):
                ref[b][r][h][d] = float(wl.k_new[t, h, d])
    assert torch.equal(kc.float(), torch.tensor(ref))
    for b in range(NB):
        for r in range(bs):
            if (b, r) not in written:
                assert bool((kc[b, r] == 7.25).all()) and bool((vc[b, r] == 7.25).all())


def test_brute_force_tiny_all_lengths():
    check_brute_force()


def test_lse_fsum():
    check_lse_fsum()


def test_matches_torch_sdpa_causal():
    check_sdpa(causal=True)


def test_matches_torch_sdpa_noncausal():
    check_sdpa(seed=6, causal=False)


def test_page_permutation_invariance():
    check_permutation_invariance()


def test_closed_form_single_visible_key():
    """Causal with q_len == kv_len: row 0 sees only key 0, so O = V[0] and
    LSE = scale * q.k0."""
    torch.manual_seed(3)
    q = torch.randn(4, 2, 8, dtype=F64)
    k = torch.randn(4, 1, 8, dtype=F64)
    v = torch.randn(4, 1, 8, dtype=F64)
    o, l = oracle.attend_dense(q, k, v, 0.3, True, 4, 4)
    for h in range(2):
        assert torch.equal(o[0, h], v[0, 0])
        dot = math.fsum(float(q[0, h, d]) * float(k[0, 0, d]) for d in range(8))
        assert abs(float(l[h, 0]) - 0.3 * dot) < 1e-13


def test_closed_form_constant_v():
    torch.manual_seed(4)
    q = torch.randn(5, 4, 8, dtype=F64)
    k = torch.randn(9, 2, 8, dtype=F64)
    c = torch.randn(1, 2, 8, dtype=F64)
    v = c.expand(9, 2, 8).clone()
    o, _ = oracle.attend_dense(q, k, v, 0.5, True, 5, 9)
    for h in range(4):
        assert torch.allclose(o[:, h], c[0, h // 2].expand(5, 8), atol=1e-14, rtol=0)


def test_closed_form_zero_q():
    """Q = 0: uniform weights over the visible keys -> mean of V, LSE = ln(n)."""
    torch.manual_seed(5)
    q_len, kv_len = 3, 10
    q = torch.zeros(q_len, 2, 4, dtype=F64)
    k = torch.randn(kv_len, 2, 4, dtype=F64)
    v = torch.randn(kv_len, 2, 4, dtype=F64)
    o, l = oracle.attend_dense(q, k, v, 0.9, True, q_len, kv_len)
    for i in range(q_len):
        n = kv_len - q_len + i + 1
        for h in range(2):
            mean = [math.fsum(float(v[j, h, d]) for j in range(n)) / n for d in range(4)]
            assert torch.allclose(o[i, h], torch.tensor(mean, dtype=F64), atol=1e-14)
            assert abs(float(l[h, i]) - math.log(n)) < 1e-14


def test_closed_form_shift_invariance():
    """Adding a vector w to every key adds scale*q.w to a row's logits: O is
    unchanged and the LSE moves by exactly that amount."""
    torch.manual_seed(6)
    q = torch.randn(4, 2, 8, dtype=F64)
    k = torch.randn(11, 1, 8, dtype=F64)
    v = torch.randn(11, 1, 8, dtype=F64)
    w = torch.randn(1, 1, 8, dtype=F64)
    o1, l1 = oracle.attend_dense(q, k, v, 0.4, True, 4, 11)
    o2, l2 = oracle.attend_dense(q, k + w, v, 0.4, True, 4, 11)
    assert torch.allclose(o1, o2, atol=1e-12, rtol=0)
    shift = 0.4 * torch.einsum("ihd,d->hi", q, w[0, 0])
    assert torch.allclose(l2 - l1, shift, atol=1e-12, rtol=0)


def test_rows_without_visible_key():
    """Causal with q_len > kv_len: the first q_len - kv_len rows see nothing."""
    q = torch.randn(5, 2, 4, dtype=F64)
    k = torch.randn(2, 1, 4, dtype=F64)
    v = torch.randn(2, 1, 4, dtype=F64)
    o, l = oracle.attend_dense(q, k, v, 1.0, True, 5, 2)
    assert torch.equal(o[:3], torch.zeros(3, 2, 4, dtype=F64))
    assert bool(torch.isinf(l[:, :3]).all()) and bool((l[:, :3] < 0).all())
    assert bool(torch.isfinite(l[:, 3:]).all())


def test_empty_sequences():
    """q_len = 0 rows produce nothing; kv_len = 0 rows see nothing."""
    q = torch.randn(2, 2, 4, dtype=torch.bfloat16)
    kc = torch.randn(3, 16, 1, 4, dtype=torch.bfloat16)
    vc = torch.randn(3, 16, 1, 4, dtype=torch.bfloat16)
    cu = torch.tensor([0, 0, 2], dtype=torch.int32)
    lk = torch.tensor([5, 0], dtype=torch.int32)
    bt = torch.tensor([[0], [1]], dtype=torch.int32)
    o, l = oracle.varlen_attention(q, kc, vc, cu, lk, bt, 0.5, False)
    assert torch.equal(o, torch.zeros_like(o)) and bool(torch.isinf(l).all())


def test_merge_split_invariance():
    """Attention over keys [0, c) merged with attention over [c, n) equals
    attention over all n keys, for every split point c."""
    torch.manual_seed(8)
    q = torch.randn(3, 4, 8, dtype=F64)
    k = torch.randn(13, 2, 8, dtype=F64)
    v = torch.randn(13, 2, 8, dtype=F64)
    full_o, full_l = oracle.attend_dense(q, k, v, 0.6, False, 3, 13)
    for c in range(1, 13):
        oa, la = oracle.attend_dense(q, k[:c], v[:c], 0.6, False, 3, c)
        ob, lb = oracle.attend_dense(q, k[c:], v[c:], 0.6, False, 3, 13 - c)
        o, l = oracle.merge_attn_states(oa, la, ob, lb)
        assert torch.allclose(o, full_o, atol=1e-12, rtol=0), c
        assert torch.allclose(l, full_l, atol=1e-12, rtol=0), c


def test_merge_identity_commutative_and_empty():
    torch.manual_seed(9)
    oa = torch.randn(4, 3, 5, dtype=F64)
    ob = torch.randn(4, 3, 5, dtype=F64)
    a = torch.randn(3, 4, dtype=F64)
    b = torch.randn(3, 4, dtype=F64)
    ninf = torch.full((3, 4), float("-inf"), dtype=F64)
    o, l = oracle.merge_attn_states(oa, a, ob, ninf)
    assert torch.equal(o, oa) and torch.equal(l, a)
    o1, l1 = oracle.merge_attn_states(oa, a, ob, b)
    o2, l2 = oracle.merge_attn_states(ob, b, oa, a)
    assert torch.allclose(o1, o2, atol=1e-15) and torch.allclose(l1, l2, atol=1e-15)
    o3, l3 = oracle.merge_attn_states(oa, ninf, ob, ninf)
    assert torch.equal(o3, torch.zeros_like(o3)) and bool(torch.isinf(l3).all())


def test_cascade_steps_equal_flat():
    """The pages' three cascade steps reproduce flat causal attention."""
    g = torch.Generator().manual_seed(12)
    S, P, bs = 5, 48, 16
    suffix = [int(x) for x in torch.randint(3, 40, (S,), generator=g)]
    q_lens = [min(int(x), s) for x, s in zip(torch.randint(1, 6, (S,), generator=g), suffix)]
    wl = W._build("cascade_small", 12, 4, 2, 16, bs, q_lens, [P + s for s in suffix], g,
                  shared_prefix_pages=P // bs)
    kc, vc = scattered_pools(wl)
    args = (wl.q, kc, vc, wl.cu_seqlens_q, wl.seqused_k, wl.block_table, wl.softmax_scale)
    flat_o, flat_l = oracle.cascade_attention(*args, P)
    steps_o, steps_l = oracle.cascade_attention_steps(*args, P)
    assert torch.allclose(flat_o, steps_o, atol=1e-12, rtol=0)
    assert torch.allclose(flat_l, steps_l, atol=1e-12, rtol=0)


def test_workload_recipe_is_deterministic():
    a, b = W.tiny_mixed(), W.tiny_mixed()
    assert torch.equal(a.q, b.q) and torch.equal(a.block_table, b.block_table)
    assert torch.equal(a.pool(0, threads=1), b.pool(0, threads=4))
    pages = a.pages_of(3)
    got = a.pool_pages(1, pages)
    full = a.pool(1)
    for p in pages:
        assert torch.equal(got[p], full[p])
    # the tiny config: 166 query tokens, 16 of 64 pages in use
    assert a.total_q == 166 and a.num_blocks == 64
    used = sum(len(a.pages_of(s)) for s in range(a.num_seqs))
    assert used == 16


# ----------------------------------------------------------------------------
# Planted mistakes: each plausible slip in the oracle must fail some pin.
# ----------------------------------------------------------------------------
def _fails(check):
    try:
        check()
    except AssertionError:
        return True
    return False


def test_planted_top_left_causal_is_caught(monkeypatch):
    monkeypatch.setattr(P, "causal_last_visible", lambda q_len, kv_len, i: i)
    assert _fails(check_golden_causal)
    assert _fails(lambda: check_sdpa(causal=True))


def test_planted_gqa_modulo_mapping_is_caught(monkeypatch):
    monkeypatch.setattr(P, "kv_head_of", lambda h, H, H_kv: h % H_kv)
    assert _fails(lambda: check_sdpa(causal=True))
    assert _fails(check_brute_force)


def test_planted_log2_lse_is_caught(monkeypatch):
    monkeypatch.setattr(P, "log_sum_exp_from", lambda m, l: m + torch.log2(l))
    assert _fails(check_lse_fsum)
    assert _fails(check_golden_two_key)


def test_planted_swapped_page_index_is_caught(monkeypatch):
    def swapped(bt_row, positions, bs):
        positions = torch.as_tensor(positions, dtype=torch.long)
        return bt_row[positions % bs % bt_row.numel()].long(), positions // bs
    monkeypatch.setattr(P, "logical_to_physical", swapped)
    assert _fails(check_golden_paged_address)


def test_planted_dropped_scale_is_caught(monkeypatch):
    real = P.attend_dense

    def no_scale(q, k, v, softmax_scale, *a, **kw):
        return real(q, k, v, 1.0, *a, **kw)
    monkeypatch.setattr(oracle, "attend_dense", no_scale)
    assert _fails(check_golden_two_key)


# ----------------------------------------------------------------------------
# FP8 (e4m3) KV cache ("FlashAttention と FlashInfer" 役割 / 境界と失敗: fp8_e4m3
# KV cache with per-head quant scales). The format is the OCP 8-bit floating
# point E4M3 one (bias 7, 3 mantissa bits, max 448, S.1111.111 = NaN).
# ----------------------------------------------------------------------------
E4M3_POINTS = {
    0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9,   # subnormals m/8 * 2^-6
    0x08: 2.0 ** -6,                                   # smallest normal
    0x38: 1.0, 0x39: 1.125, 0x3F: 1.875,               # e = 7: 1 + m/8
    0x77: 240.0, 0x7E: 448.0,                          # e = 14, e = 15 (m <= 6)
    0xB8: -1.0, 0xFE: -448.0,
}


def check_e4m3_points():
    for code, v in E4M3_POINTS.items():
        assert P.e4m3_decode(code) == v, hex(code)
        assert P.e4m3_encode(v) == code, hex(code)
    assert math.isnan(P.e4m3_decode(0x7F)) and math.isnan(P.e4m3_decode(0xFF))
    assert P.e4m3_encode(-0.0) == 0x80


def check_e4m3_round_vs_torch():
    """Every value near a rounding boundary: all e4m3 values, the midpoints
    between neighbours, and one float32 step either side of each, plus a random
    spread; torch's float8_e4m3fn conversion rounds to nearest even (and agrees
    with saturation for |x| < 464)."""
    vals = P.e4m3_table()[:0x7F]
    pts = set(vals.tolist())
    for a, b in zip(vals[:-1].tolist(), vals[1:].tolist()):
        mid = torch.tensor((a + b) / 2, dtype=torch.float32)
        pts.update([float(mid), float(torch.nextafter(mid, torch.tensor(0.0))),
                    float(torch.nextafter(mid, torch.tensor(1e9)))])
    pts.update([452.0, 455.99, 460.0, 463.9])
    g = torch.Generator().manual_seed(7)
    pts.update((torch.randn(2000, generator=g) * 30).tolist())
    pts.update((torch.rand(2000, generator=g) * 2.0 ** -5).tolist())
    x = torch.tensor(sorted(pts), dtype=torch.float32)
    x = torch.cat([x, -x])
    x = x[x.abs() < 464]
    ref = x.to(torch.float8_e4m3fn)
    got_codes = P.quantize_e4m3(x.view(-1, 1, 1), [1.0]).view(-1)
    assert torch.equal(got_codes, ref.view(torch.uint8)), "vector quantizer"
    for xi, ri in zip(x.tolist()[::7], ref.float().tolist()[::7]):
        assert P.e4m3_round(xi) == ri, xi


def test_e4m3_format_points():
    check_e4m3_points()


def test_e4m3_decode_matches_torch():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(F64)
    got = P.e4m3_table()
    nan = torch.isnan(ref)
    assert torch.equal(nan, torch.isnan(got)) and nan.sum() == 2
    assert torch.equal(got[~nan], ref[~nan])


def test_e4m3_round_matches_torch():
    check_e4m3_round_vs_torch()


def test_e4m3_code_roundtrip_and_saturation():
    for c in range(256):
        if c & 0x7F == 0x7F:
            continue
        assert P.e4m3_encode(P.e4m3_decode(c)) == c
    # Beyond the largest finite value the write saturates (torch does not).
    for v, code in ((464.0, 0x7E), (1e6, 0x7E), (math.inf, 0x7E), (-500.0, 0xFE),
                    (-math.inf, 0xFE)):
        assert P.e4m3_encode(v) == code
        assert int(P.quantize_e4m3(torch.tensor([[[v]]]), [1.0])) == code
    assert int(P.quantize_e4m3(torch.tensor([[[math.nan]]]), [1.0])) == 0x7F


def test_e4m3_quotient_is_float32():
    # 5.28125 / 0x1.018618p+0 is 5.25000012 in float64 -- above the midpoint
    # of 5.0 and 5.5 -- but exactly 5.25 in float32, a tie that goes to the
    # even neighbour 5.0 (code 0x4A). The code is decided by the float32
    # quotient, as the kernel computes it.
    s = float.fromhex("0x1.018618p+0")
    x = torch.tensor([[[5.28125]]], dtype=torch.bfloat16)
    assert int(P.quantize_e4m3(x, [s])) == 0x4A
    assert P.e4m3_encode(5.28125 / s) == 0x4B


def test_e4m3_per_head_scale_and_error_bound():
    g = torch.Generator().manual_seed(3)
    x = (torch.randn(6, 4, 16, generator=g) * 3).to(torch.bfloat16)
    sc = [0.5, 1.0, 0.0625, 3.0]
    codes = P.quantize_e4m3(x, sc)
    for h in range(4):
        brute = [P.e4m3_encode(float(torch.tensor(float(v), dtype=torch.float32) /
                                     torch.tensor(sc[h], dtype=torch.float32)))
                 for v in x[:, h].reshape(-1).tolist()]
        assert codes[:, h].reshape(-1).tolist() == brute
    dq = P.dequantize_e4m3(codes, sc)
    xs = x.to(F64)
    s = torch.tensor(sc, dtype=F64)[:, None]
    # Half a unit in the last place: 2^-4 relative in the normal range, and
    # 2^-10 * scale absolute among the subnormals.
    bound = torch.maximum(xs.abs() * 2.0 ** -4, 2.0 ** -10 * s.expand_as(xs))
    assert ((dq - xs).abs() <= bound + 1e-12).all()


def test_e4m3_scatter_brute_force():
    g = torch.Generator().manual_seed(5)
    key = torch.randn(5, 2, 128, generator=g).to(torch.bfloat16)
    value = torch.randn(5, 2, 128, generator=g).to(torch.bfloat16)
    kc = torch.full((3, 16, 2, 128), 0x55, dtype=torch.uint8)
    vc = kc.clone()
    slots = torch.tensor([17, -1, 0, 47, 5], dtype=torch.int64)
    P.reshape_and_cache_e4m3(key, value, slots, kc, vc, [0.25, 2.0], [1.0, 0.5])
    for t, slot in enumerate(slots.tolist()):
        if slot < 0:
            continue
        b, r = divmod(slot, 16)
        for h, (ks, vs) in enumerate(((0.25, 1.0), (2.0, 0.5))):
            assert kc[b, r, h].tolist() == [P.e4m3_encode(float(torch.tensor(float(v)) / ks))
                                            for v in key[t, h].tolist()]
            assert vc[b, r, h].tolist() == [P.e4m3_encode(float(torch.tensor(float(v)) / vs))
                                            for v in value[t, h].tolist()]
    untouched = torch.ones(3 * 16, dtype=torch.bool)
    untouched[[17, 0, 47, 5]] = False
    assert (kc.view(48, -1)[untouched] == 0x55).all()


def test_e4m3_attention_is_attention_of_dequantized_pool():
    # Codes 0x38 (1.0) and 0xB8 (-1.0) with scale 0.5 are keys of +-0.5: two
    # keys whose scores differ by q.(k0 - k1); closed form of a 2-key softmax.
    D = 128
    kc = torch.zeros(1, 16, 1, D, dtype=torch.uint8)
    vc = torch.zeros(1, 16, 1, D, dtype=torch.uint8)
    kc[0, 0, 0, 0] = 0x38
    kc[0, 1, 0, 0] = 0xB8
    vc[0, 0, 0, :] = 0x40          # 2.0
    vc[0, 1, 0, :] = 0x00          # 0.0
    q = torch.zeros(1, 1, D, dtype=torch.bfloat16)
    q[0, 0, 0] = 2.0
    out, lse = P.varlen_attention_e4m3(q, kc, vc, torch.tensor([0, 1]), torch.tensor([2]),
                                       torch.tensor([[0]], dtype=torch.int32), 1.0, False,
                                       [0.5], [3.0])
    s0, s1 = 2.0 * 0.5, 2.0 * -0.5
    w0 = math.exp(s0) / (math.exp(s0) + math.exp(s1))
    assert abs(float(out[0, 0, 5]) - w0 * 6.0) < 1e-12
    assert abs(float(lse[0, 0]) - math.log(math.exp(s0) + math.exp(s1))) < 1e-12


def test_planted_ties_away_is_caught(monkeypatch):
    def away(y):
        a = abs(y)
        if a >= P.E4M3_MAX:
            return math.copysign(P.E4M3_MAX, y)
        E = -6
        while E < 8 and 2.0 ** (E + 1) <= a:
            E += 1
        q = 2.0 ** (E - 3)
        return math.copysign(min(math.floor(a / q + 0.5) * q, P.E4M3_MAX), y)
    monkeypatch.setattr(P, "e4m3_round", away)
    with pytest.raises(AssertionError):
        check_e4m3_round_vs_torch()


def test_planted_exponent_bias_is_caught(monkeypatch):
    orig = P.e4m3_decode
    monkeypatch.setattr(P, "e4m3_decode", lambda c: orig(c) * 2.0 if c & 0x78 else orig(c))
    with pytest.raises(AssertionError):
        check_e4m3_points()


# ----------------------------------------------------------------------------
# n-state merge and decode context parallelism over virtual ranks
# ("FlashAttention 在 vLLM 中的实现分析" §9: each rank attends over its KV shard,
# the partial (out, lse) are merged by LSE).
# ----------------------------------------------------------------------------
def check_merge_n_partition():
    """Attention over a partition of the keys into n interleaved groups,
    merged, equals attention over all keys (attend_dense is pinned by brute
    force and torch SDPA)."""
    g = torch.Generator().manual_seed(12)
    q = torch.randn(3, 4, 8, generator=g, dtype=F64)
    k = torch.randn(17, 2, 8, generator=g, dtype=F64)
    v = torch.randn(17, 2, 8, generator=g, dtype=F64)
    full_o, full_l = oracle.attend_dense(q, k, v, 0.7, False, 3, 17)
    for n in (1, 2, 3, 5):
        outs, lses = [], []
        for r in range(n):
            idx = torch.arange(r, 17, n)
            o, l = oracle.attend_dense(q, k[idx], v[idx], 0.7, False, 3, idx.numel())
            outs.append(o)
            lses.append(l)
        o, l = P.merge_attn_states_n(torch.stack(outs), torch.stack(lses))
        assert torch.allclose(o, full_o, atol=1e-12, rtol=0), n
        assert torch.allclose(l, full_l, atol=1e-12, rtol=0), n


def test_merge_n_partition_invariance():
    check_merge_n_partition()


def test_merge_n_identity_order_and_empty():
    g = torch.Generator().manual_seed(13)
    po = torch.randn(4, 3, 2, 8, generator=g, dtype=F64)
    pl = torch.randn(4, 2, 3, generator=g, dtype=F64) * 3
    o1, l1 = P.merge_attn_states_n(po[:1], pl[:1])
    assert torch.equal(o1, po[0]) and torch.allclose(l1, pl[0], atol=1e-15, rtol=0)
    perm = torch.tensor([2, 0, 3, 1])
    oa, la = P.merge_attn_states_n(po, pl)
    ob, lb = P.merge_attn_states_n(po[perm], pl[perm])
    assert torch.allclose(oa, ob, atol=1e-13, rtol=0) and torch.allclose(la, lb, atol=1e-13, rtol=0)
    # two states: the pinned two-state merge
    o2, l2 = P.merge_attn_states_n(po[:2], pl[:2])
    r2o, r2l = oracle.merge_attn_states(po[0], pl[0], po[1], pl[1])
    assert torch.allclose(o2, r2o, atol=1e-13, rtol=0) and torch.allclose(l2, r2l, atol=1e-13, rtol=0)
    # -inf parts carry no weight; a row with only -inf parts is empty
    pl2 = pl.clone()
    pl2[1:] = float("-inf")
    o3, l3 = P.merge_attn_states_n(po, pl2)
    assert torch.equal(o3, po[0]) and torch.allclose(l3, pl[0], atol=1e-15, rtol=0)
    pl2[0] = float("-inf")
    o4, l4 = P.merge_attn_states_n(po, pl2)
    assert torch.equal(o4, torch.zeros_like(o4)) and torch.isinf(l4).all()


@pytest.mark.parametrize("ranks", [1, 2, 3, 4])
def test_dcp_virtual_ranks_equal_flat_decode(ranks):
    """Decode over R virtual ranks (block b on rank b % R, each rank
    non-causal over its shard, states merged) equals flat causal decode,
    including sequences with fewer blocks than ranks (empty shards)."""
    wl = W.random_case(31 + ranks, num_seqs=5, num_heads=4, num_kv_heads=2, head_size=16,
                       block_size=16, max_q=1, max_kv=90, decode_frac=1.0)
    assert all(q == 1 for q in wl.q_lens)
    kc, vc = wl.pool(0), wl.pool(1)
    oracle.reshape_and_cache(wl.k_new, wl.v_new, wl.slot_mapping, kc, vc)
    ref_o, ref_l = oracle.varlen_attention(wl.q, kc, vc, wl.cu_seqlens_q, wl.seqused_k,
                                           wl.block_table, wl.softmax_scale, True)
    tables, lens = W.dcp_shards(wl, ranks)
    assert [int(sum(l[s] for l in lens)) for s in range(wl.num_seqs)] == wl.kv_lens
    o, l = oracle.dcp_decode_attention(wl.q, kc, vc, wl.cu_seqlens_q, tables, lens,
                                       wl.softmax_scale)
    assert torch.allclose(o, ref_o, atol=1e-12, rtol=0)
    assert torch.allclose(l, ref_l, atol=1e-12, rtol=0)


def test_planted_max_instead_of_logsumexp_is_caught(monkeypatch):
    orig = P.merge_attn_states_n

    def bad(po, pl):
        o, l = orig(po, pl)
        return o, pl.to(F64).max(dim=0).values
    monkeypatch.setattr(P, "merge_attn_states_n", bad)
    with pytest.raises(AssertionError):
        check_merge_n_partition()


# ----------------------------------------------------------------------------
# Attention sinks ("FlashAttention 在 vLLM 中的实现分析" §1.2 / §1.3: the s_aux
# learnable sink token of FA3/FA4): one extra logit per query head with no
# value, in the softmax denominator and the LSE.
# ----------------------------------------------------------------------------
def check_sinks_merge_identity():
    """Attention with sinks = the two-state merge (pinned) of attention
    without them and the state (out 0, lse = sink)."""
    wl = W.random_case(41, num_seqs=4, num_heads=8, num_kv_heads=2, head_size=16,
                       block_size=16, max_q=9, max_kv=40, empty_ok=True)
    kc, vc = wl.pool(0), wl.pool(1)
    oracle.reshape_and_cache(wl.k_new, wl.v_new, wl.slot_mapping, kc, vc)
    sinks = torch.linspace(-2.0, 3.0, 8, dtype=F64)
    args = (wl.q, kc, vc, wl.cu_seqlens_q, wl.seqused_k, wl.block_table, wl.softmax_scale, True)
    o_s, l_s = oracle.varlen_attention(*args, sinks=sinks)
    o, l = oracle.varlen_attention(*args)
    T = wl.q.shape[0]
    mo, ml = oracle.merge_attn_states(o, l, torch.zeros_like(o), sinks[:, None].expand(8, T))
    assert torch.allclose(o_s, mo, atol=1e-12, rtol=0)
    assert torch.allclose(l_s, ml, atol=1e-12, rtol=0)


def test_sinks_merge_identity():
    check_sinks_merge_identity()


def test_sinks_minus_inf_is_no_sink():
    wl = W.random_case(42, num_seqs=3, num_heads=4, num_kv_heads=4, head_size=16, block_size=16)
    kc, vc = wl.pool(0), wl.pool(1)
    args = (wl.q, kc, vc, wl.cu_seqlens_q, wl.seqused_k, wl.block_table, wl.softmax_scale, True)
    o, l = oracle.varlen_attention(*args)
    o2, l2 = oracle.varlen_attention(*args, sinks=torch.full((4,), float("-inf"), dtype=F64))
    assert torch.equal(o, o2) and torch.equal(l, l2)


def test_sinks_as_an_extra_key():
    """A sink of logit s behaves as one more key k* with scale * q.k* = s and
    value 0 (one query row, no GQA, so k* can be built per head)."""
    g = torch.Generator().manual_seed(43)
    H, D, n = 3, 8, 7
    q = torch.randn(1, H, D, generator=g, dtype=F64)
    k = torch.randn(n, H, D, generator=g, dtype=F64)
    v = torch.randn(n, H, D, generator=g, dtype=F64)
    scale = 0.4
    sinks = torch.tensor([0.5, -1.0, 2.5], dtype=F64)
    kx = torch.stack([q[0, h] * (sinks[h] / (scale * q[0, h].dot(q[0, h]))) for h in range(H)])
    k2 = torch.cat([k, kx[None]], dim=0)
    v2 = torch.cat([v, torch.zeros(1, H, D, dtype=F64)], dim=0)
    o_ref, l_ref = oracle.attend_dense(q, k2, v2, scale, False, 1, n + 1)
    o, l = oracle.attend_dense(q, k, v, scale, False, 1, n, sinks=sinks)
    assert torch.allclose(o, o_ref, atol=1e-12, rtol=0)
    assert torch.allclose(l, l_ref, atol=1e-12, rtol=0)


def test_sinks_keyless_rows():
    q = torch.randn(2, 2, 8, dtype=F64)
    k = torch.zeros(0, 2, 8, dtype=F64)
    o, l = oracle.attend_dense(q, k, k, 0.5, True, 2, 0, sinks=torch.tensor([1.5, -0.5]))
    assert torch.equal(o, torch.zeros_like(o))
    assert l[0].tolist() == [1.5, 1.5] and l[1].tolist() == [-0.5, -0.5]


def test_planted_sink_in_lse_only_is_caught(monkeypatch):
    orig = P.attend_dense

    def bad(q, k, v, scale, causal, q_len, kv_len, rows=None, row_chunk=512, sinks=None):
        o, _ = orig(q, k, v, scale, causal, q_len, kv_len, rows=rows, row_chunk=row_chunk)
        _, l = orig(q, k, v, scale, causal, q_len, kv_len, rows=rows, row_chunk=row_chunk,
                    sinks=sinks)
        return o, l                       # the sink missing from the denominator of out
    monkeypatch.setattr(P, "attend_dense", bad)
    with pytest.raises(AssertionError):
        check_sinks_merge_identity()


def test_dcp_shard_layout():
    """Every page of every sequence is on exactly one virtual rank, in
    logical order, and the key counts add up (input layout only)."""
    wl = W.random_case(51, num_seqs=6, num_heads=4, num_kv_heads=2, head_size=16,
                       block_size=16, max_q=1, max_kv=150, decode_frac=1.0)
    for ranks in (1, 2, 3, 5):
        tables, lens = W.dcp_shards(wl, ranks)
        for s in range(wl.num_seqs):
            pages = wl.pages_of(s)
            got = []
            for r in range(ranks):
                nb = (int(lens[r][s]) + wl.block_size - 1) // wl.block_size
                row = [int(x) for x in tables[r][s, :nb]]
                assert row == pages[r::ranks]
                got += row
            assert sorted(got) == sorted(pages)
            assert sum(int(l[s]) for l in lens) == wl.kv_lens[s]


# ---------------------------------------------------------------- f16 inputs
def check_f16_values_read_exactly():
    """f16 keeps 10 fraction bits, bf16 7: 1 + 2^-10, 3 + 2^-9 and
    1 - 2^-11 are f16 values bf16 cannot hold. One sequence with one key: the
    output is that key's value row exactly and the LSE is scale * q.k, both
    from the f16 values themselves ("FlashAttention 在 vLLM 中的实现分析"
    §2.1 lists float16 beside bfloat16)."""
    D, bs = 8, 16
    qv, kv, vv = 3 + 2 ** -9, 1 - 2 ** -11, 1 + 2 ** -10
    q = torch.full((1, 1, D), qv, dtype=torch.float16)
    kc = torch.zeros((1, bs, 1, D), dtype=torch.float16)
    vc = torch.zeros((1, bs, 1, D), dtype=torch.float16)
    kc[0, 0, 0] = kv
    vc[0, 0, 0] = vv
    for t, x in ((q, qv), (kc[0, 0], kv), (vc[0, 0], vv)):
        assert float(t.flatten()[0]) == x                      # exact in f16
    assert float(torch.tensor(vv).to(torch.bfloat16)) != vv    # not in bf16
    o, l = oracle.varlen_attention(q, kc, vc, torch.tensor([0, 1], dtype=torch.int32),
                                   torch.tensor([1], dtype=torch.int32),
                                   torch.tensor([[0]], dtype=torch.int32), 0.25, True)
    assert o.dtype == F64 and bool((o[0, 0] == vv).all())
    assert float(l[0, 0]) == 0.25 * D * qv * kv               # exact: a dyadic product


def test_f16_inputs_are_read_as_f16_values():
    check_f16_values_read_exactly()


def test_planted_bf16_rounding_of_f16_inputs_is_caught(monkeypatch):
    orig = P.attend_dense

    def bad(q, k, v, *args, **kw):
        r = lambda x: x.to(torch.bfloat16).to(F64)
        return orig(r(q), r(k), r(v), *args, **kw)
    monkeypatch.setattr(P, "attend_dense", bad)
    assert _fails(check_f16_values_read_exactly)
