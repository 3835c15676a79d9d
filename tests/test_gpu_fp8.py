"""GPU parity of the FP8 (e4m3) KV cache path ("FlashAttention と FlashInfer"
役割 / 境界と失敗: fp8_e4m3 KV cache with per-head quant scales) against the
fp64 oracle. The quantizing scatter is bit-exact; attention over the e4m3
pools is compared with the oracle's attention over the dequantized pools,
bf16 outputs within 1e-2 max-abs and LSE within 1e-3."""
import pytest
import torch

import oracle
import paged_kv_varlen_attn_gb300 as pa
import workloads as W
from helpers import LSE_TOL, OUT_TOL

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_varlen_attn_gb300 import _build
    _build.build()
    pa.load_library()


def assert_close(out, lse, ref_o, ref_l, tokens=None):
    o, l = out.cpu().double(), lse.cpu().double()
    if tokens is not None:
        o, l = o[tokens], l[:, tokens]
    fin = torch.isfinite(ref_l)
    assert torch.equal(fin, torch.isfinite(l)), "rows without keys must have lse = -inf"
    err_o = (o - ref_o).abs().max().item() if o.numel() else 0.0
    err_l = (l[fin] - ref_l[fin]).abs().max().item() if fin.any() else 0.0
    assert err_o <= OUT_TOL, f"out max-abs err {err_o}"
    assert err_l <= LSE_TOL, f"lse abs err {err_l}"
    return err_o, err_l


def oracle_fp8_pools(wl, slots=None):
    kc, vc = wl.fp8_pool(0), wl.fp8_pool(1)
    oracle.reshape_and_cache_e4m3(wl.k_new, wl.v_new,
                                  wl.slot_mapping if slots is None else slots, kc, vc,
                                  wl.kv_scales(0), wl.kv_scales(1))
    return kc, vc


def run_fp8(wl, cascade=False, status=None, fused=True):
    """GPU: prior e4m3 pools, then (fused or separate) quantizing scatter of
    the new tokens and attention. Returns out, lse, key pool, value pool."""
    kc, vc = wl.fp8_pool(0, DEV), wl.fp8_pool(1, DEV)
    ks = torch.tensor(wl.kv_scales(0), device=DEV)
    vs = torch.tensor(wl.kv_scales(1), device=DEV)
    k_new, v_new, slots = wl.k_new.to(DEV), wl.v_new.to(DEV), wl.slot_mapping.to(DEV)
    upd = dict(key=k_new, value=v_new, slot_mapping=slots) if fused else {}
    if not fused:
        pa.reshape_and_cache_fp8(k_new, v_new, kc, vc, slots, ks, vs, dev_status=status)
    args = (wl.q.to(DEV), kc, vc, wl.cu_seqlens_q.to(DEV), wl.seqused_k.to(DEV),
            wl.block_table.to(DEV), max(wl.max_seqlen_q, 1), wl.max_seqlen_k, wl.softmax_scale)
    if cascade:
        out, lse = pa.cascade_fwd_fp8kv(*args, wl.common_prefix_len, ks, vs, dev_status=status,
                                        **upd)
    else:
        out, lse = pa.varlen_fwd_fp8kv(*args, wl.causal, ks, vs, dev_status=status, **upd)
    torch.cuda.synchronize()
    return out, lse, kc, vc


# ---------------------------------------------------------------- scatter
@pytest.mark.parametrize("seed,bs,Hk", [(201, 16, 8), (202, 32, 2), (203, 128, 1), (204, 48, 4)])
def test_fp8_scatter_bit_exact(seed, bs, Hk):
    wl = W.random_case(seed, num_seqs=6, num_heads=Hk * 2, num_kv_heads=Hk, head_size=128,
                       block_size=bs, max_q=50, max_kv=300)
    k_new, v_new = wl.k_new.clone(), wl.v_new.clone()
    # Saturation, signed zeros, subnormal codes and a float32-decided tie:
    # 5.28125 / 0x1.018618p+0 is exactly 5.25 in float32 (ties to 5.0, code
    # 0x4A) but 5.25000012 in float64.
    k_new[0, 0, :6] = torch.tensor([1000.0, -1000.0, 0.0, -0.0, 1e-4, -3e-3])
    ks = wl.kv_scales(0)
    ks[0] = float.fromhex("0x1.018618p+0")
    k_new[0, 0, 6] = 5.28125
    slots = wl.slot_mapping.clone()
    slots[1::4] = -1
    canary = torch.full((wl.num_blocks, bs, Hk, 128), 0xA5, dtype=torch.uint8)
    kc_ref, vc_ref = canary.clone(), canary.clone()
    oracle.reshape_and_cache_e4m3(k_new, v_new, slots, kc_ref, vc_ref, ks, wl.kv_scales(1))
    kc, vc = canary.to(DEV), canary.to(DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    pa.reshape_and_cache_fp8(k_new.to(DEV), v_new.to(DEV), kc, vc, slots.to(DEV),
                             torch.tensor(ks, device=DEV), torch.tensor(wl.kv_scales(1), device=DEV),
                             dev_status=status)
    torch.cuda.synchronize()
    assert torch.equal(kc.cpu(), kc_ref)
    assert torch.equal(vc.cpu(), vc_ref)
    assert int(status.item()) == 0
    t0 = 0 if int(slots[0]) >= 0 else None
    if t0 is not None:
        b, r = divmod(int(slots[0]), bs)
        assert kc_ref[b, r, 0, :7].tolist() == [0x7E, 0xFE, 0x00, 0x80,
                                                 kc_ref[b, r, 0, 4].item(),
                                                 kc_ref[b, r, 0, 5].item(), 0x4A]


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_fp8_scatter_every_value(dtype):
    """Every bf16 (or f16) value -- zeros, subnormals, infinities and NaNs
    included -- divided by each of 8 KV-head scales: the edges of the range
    the kernel divides by reciprocal and correction (2^-32, 2^32), scales
    outside it (2^-40, 2^40, which divide) and ordinary ones. Bit-exact."""
    Hk, D, bs = 8, 128, 16
    T = 65536 // D
    every = torch.arange(65536, dtype=torch.int32).to(torch.int16).view(dtype)
    g = torch.Generator().manual_seed(241)
    k_new = torch.stack([every[torch.randperm(65536, generator=g)].reshape(T, D)
                         for _ in range(Hk)], dim=1)
    v_new = torch.stack([every[torch.randperm(65536, generator=g)].reshape(T, D)
                         for _ in range(Hk)], dim=1)
    ks = [2.0 ** -32, 2.0 ** 32, 2.0 ** -40, 2.0 ** 40, 0.0123, 1 / 3, 3.7 / 448, 1.0]
    vs = [0.021, 2.0 ** 40, 1 / 7, 2.0 ** -32, 2.0 ** 32, 2.0 ** -40, 0.5, 255.0]
    ks = [float(torch.tensor(x, dtype=torch.float32)) for x in ks]
    vs = [float(torch.tensor(x, dtype=torch.float32)) for x in vs]
    nb = T // bs + 2
    slots = torch.randperm(nb * bs, generator=g)[:T].to(torch.int64)
    kc_ref = torch.zeros((nb, bs, Hk, D), dtype=torch.uint8)
    vc_ref = kc_ref.clone()
    oracle.reshape_and_cache_e4m3(k_new, v_new, slots, kc_ref, vc_ref, ks, vs)
    kc, vc = torch.zeros_like(kc_ref, device=DEV), torch.zeros_like(vc_ref, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    pa.reshape_and_cache_fp8(k_new.to(DEV), v_new.to(DEV), kc, vc, slots.to(DEV),
                             torch.tensor(ks, device=DEV), torch.tensor(vs, device=DEV),
                             dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(kc.cpu(), kc_ref)
    assert torch.equal(vc.cpu(), vc_ref)


def test_fp8_scatter_scalar_scale_and_bad_slot():
    wl = W.random_case(205, num_seqs=3, num_heads=8, num_kv_heads=4, head_size=128,
                       block_size=16, max_q=20, max_kv=60)
    slots = wl.slot_mapping.clone()
    slots[0] = wl.num_blocks * 16 + 3
    ok = slots.clone()
    ok[0] = -1
    kc_ref, vc_ref = wl.fp8_pool(0), wl.fp8_pool(1)
    oracle.reshape_and_cache_e4m3(wl.k_new, wl.v_new, ok, kc_ref, vc_ref, [0.05] * 4, [0.02] * 4)
    kc, vc = wl.fp8_pool(0, DEV), wl.fp8_pool(1, DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    pa.reshape_and_cache_fp8(wl.k_new.to(DEV), wl.v_new.to(DEV), kc, vc, slots.to(DEV), 0.05,
                             0.02, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & pa.PA_DEV_BAD_SLOT
    assert torch.equal(kc.cpu(), kc_ref) and torch.equal(vc.cpu(), vc_ref)


# ---------------------------------------------------------------- attention
CASES = [
    # seed, S, H, Hk, bs, max_q, max_kv, causal, decode_frac
    (211, 5, 8, 8, 16, 40, 300, True, 0.4),      # GQA 1
    (212, 6, 32, 8, 16, 1, 2000, True, 1.0),     # decode, GQA 4, several splits
    (213, 4, 16, 2, 32, 70, 400, True, 0.2),     # GQA 8: 16-64 row items
    (214, 3, 8, 1, 64, 90, 500, False, 0.0),     # non-causal, GQA 8, page 64
    (215, 7, 32, 8, 128, 33, 1500, True, 0.5),   # page 128, ragged
    (216, 5, 16, 16, 48, 20, 200, True, 0.3),    # page 48 (boxes of 16 rows)
    (219, 4, 32, 2, 16, 1, 700, True, 1.0),      # decode, GQA 16: 16-row items
    # prefill segments (more than 32 packed rows): the tensor-core kernel
    # with the e4m3 tiles widened to f16 in shared memory
    (231, 2, 8, 2, 16, 300, 1100, True, 0.0),    # several Q tiles, prior context
    (232, 3, 32, 8, 128, 200, 3000, True, 0.0),  # long keys: KV splits, page 128
    (233, 2, 24, 8, 16, 150, 400, True, 0.0),    # G = 3: 126-row tiles
    (234, 3, 16, 2, 32, 100, 300, False, 0.0),   # non-causal
    (235, 4, 8, 1, 48, 70, 260, True, 0.3),      # G = 8, page 48, with decode rows
]


@pytest.mark.parametrize("seed,S,H,Hk,bs,max_q,max_kv,causal,dfrac", CASES)
def test_fp8_varlen_parity(seed, S, H, Hk, bs, max_q, max_kv, causal, dfrac):
    wl = W.random_case(seed, num_seqs=S, num_heads=H, num_kv_heads=Hk, head_size=128,
                       block_size=bs, max_q=max_q, max_kv=max_kv, causal=causal,
                       decode_frac=dfrac)
    kc_ref, vc_ref = oracle_fp8_pools(wl)
    ref_o, ref_l = oracle.varlen_attention_e4m3(wl.q, kc_ref, vc_ref, wl.cu_seqlens_q,
                                                wl.seqused_k, wl.block_table, wl.softmax_scale,
                                                wl.causal, wl.kv_scales(0), wl.kv_scales(1))
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out, lse, kc, vc = run_fp8(wl, status=status)
    assert torch.equal(kc.cpu(), kc_ref) and torch.equal(vc.cpu(), vc_ref)
    assert_close(out, lse, ref_o, ref_l)
    assert int(status.item()) == 0


def test_fp8_fused_equals_separate():
    wl = W.random_case(217, num_seqs=6, num_heads=32, num_kv_heads=8, head_size=128,
                       block_size=16, max_q=12, max_kv=900)
    o1, l1, k1, v1 = run_fp8(wl, fused=True)
    o2, l2, k2, v2 = run_fp8(wl, fused=False)
    assert torch.equal(k1, k2) and torch.equal(v1, v2)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_fp8_empty_and_keyless_rows():
    wl = W.random_case(218, num_seqs=6, num_heads=8, num_kv_heads=2, head_size=128,
                       block_size=16, max_q=10, max_kv=40, empty_ok=True)
    kc_ref, vc_ref = oracle_fp8_pools(wl)
    ref_o, ref_l = oracle.varlen_attention_e4m3(wl.q, kc_ref, vc_ref, wl.cu_seqlens_q,
                                                wl.seqused_k, wl.block_table, wl.softmax_scale,
                                                wl.causal, wl.kv_scales(0), wl.kv_scales(1))
    out, lse, _, _ = run_fp8(wl)
    assert_close(out, lse, ref_o, ref_l)


@pytest.mark.parametrize("seed,S,H,Hk,P,qmax,smax", [
    (221, 9, 8, 2, 96, 3, 80),
    (222, 40, 32, 4, 512, 2, 200),
])
def test_fp8_cascade_parity(seed, S, H, Hk, P, qmax, smax):
    g = torch.Generator().manual_seed(seed)
    suffix = [int(x) for x in torch.randint(qmax + 1, smax, (S,), generator=g)]
    q_lens = [int(x) for x in torch.randint(1, qmax + 1, (S,), generator=g)]
    wl = W._build(f"cascade_fp8_{seed}", seed, H, Hk, 128, 16, q_lens,
                  [P + s for s in suffix], g, shared_prefix_pages=P // 16)
    kc_ref, vc_ref = oracle_fp8_pools(wl)
    kd = oracle.dequantize_e4m3(kc_ref, wl.kv_scales(0))
    vd = oracle.dequantize_e4m3(vc_ref, wl.kv_scales(1))
    ref_o, ref_l = oracle.cascade_attention(wl.q, kd, vd, wl.cu_seqlens_q, wl.seqused_k,
                                            wl.block_table, wl.softmax_scale,
                                            wl.common_prefix_len)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out, lse, _, _ = run_fp8(wl, cascade=True, status=status)
    assert_close(out, lse, ref_o, ref_l)
    assert int(status.item()) == 0


def test_fp8_cascade_shared_prefix_config():
    """The cascade bench workload (64 requests sharing a 2048-token prefix,
    32/8 heads, page 16) on e4m3 pools, every row against the oracle: the
    prefix pass in 256-key chunks on the tensor-core kernel (Q as two e4m3
    terms), the suffix pass on the split kernel, then the combine."""
    wl = W.cascade_shared_prefix()
    kc_ref, vc_ref = oracle_fp8_pools(wl)
    kd = oracle.dequantize_e4m3(kc_ref, wl.kv_scales(0))
    vd = oracle.dequantize_e4m3(vc_ref, wl.kv_scales(1))
    ref_o, ref_l = oracle.cascade_attention(wl.q, kd, vd, wl.cu_seqlens_q, wl.seqused_k,
                                            wl.block_table, wl.softmax_scale,
                                            wl.common_prefix_len)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out, lse, _, _ = run_fp8(wl, cascade=True, status=status)
    assert_close(out, lse, ref_o, ref_l)
    assert int(status.item()) == 0


def test_fp8_decode_llama8b_sampled():
    """The full-size decode batch (64 sequences, KV 512-8192, 32/8 heads) on
    e4m3 pools, checked on sampled sequences (the oracle regenerates only
    their pages)."""
    wl = W.decode_llama8b()
    out, lse, kc, vc = run_fp8(wl)
    g = torch.Generator().manual_seed(9)
    seqs = sorted(set(int(x) for x in torch.randint(0, wl.num_seqs, (6,), generator=g)))
    seqs = sorted(set(seqs) | {int(torch.tensor(wl.kv_lens).argmax())})
    sub = wl.sub_batch(seqs)
    pages = sorted({p for s in range(sub.num_seqs) for p in sub.pages_of(s)})
    remap = {p: i for i, p in enumerate(pages)}
    kp, vp = wl.fp8_pool_pages(0, pages), wl.fp8_pool_pages(1, pages)
    kc_s = torch.stack([kp[p] for p in pages])
    vc_s = torch.stack([vp[p] for p in pages])
    bt = torch.full_like(sub.block_table, W.INT32_MAX)
    for s in range(sub.num_seqs):
        ps = sub.pages_of(s)
        bt[s, :len(ps)] = torch.tensor([remap[p] for p in ps], dtype=torch.int32)
    bs = wl.block_size
    slots = torch.tensor([remap[int(x) // bs] * bs + int(x) % bs for x in sub.slot_mapping],
                         dtype=torch.int64)
    oracle.reshape_and_cache_e4m3(sub.k_new, sub.v_new, slots, kc_s, vc_s, wl.kv_scales(0),
                                  wl.kv_scales(1))
    ref_o, ref_l = oracle.varlen_attention_e4m3(sub.q, kc_s, vc_s, sub.cu_seqlens_q,
                                                sub.seqused_k, bt, wl.softmax_scale, True,
                                                wl.kv_scales(0), wl.kv_scales(1))
    tokens = torch.tensor([int(wl.cu_seqlens_q[s]) for s in seqs])
    assert_close(out, lse, ref_o, ref_l, tokens=tokens)
    # the fused scatter wrote the sampled sequences' new rows bit-exactly
    for i, s in enumerate(seqs):
        sl = int(wl.slot_mapping[int(wl.cu_seqlens_q[s])])
        b, r = divmod(sl, bs)
        b2, r2 = divmod(int(slots[i]), bs)
        assert torch.equal(kc[b, r].cpu(), kc_s[b2, r2])
        assert torch.equal(vc[b, r].cpu(), vc_s[b2, r2])


def test_fp8_long_context_prefill_sampled():
    """The 70B prefill shape (4 causal x 4096 queries on 28,672 prior keys,
    64/8 heads, page 128) on e4m3 pools: the tensor-core kernel over widened
    tiles, checked on sampled rows of every sequence (first, last, tile
    boundaries and seeded random rows)."""
    wl = W.long_context_70b_prefill()
    out, lse, kc, vc = run_fp8(wl)
    seqs = list(range(wl.num_seqs))
    pages = sorted({p for s in seqs for p in wl.pages_of(s)})
    remap = {p: i for i, p in enumerate(pages)}
    kp, vp = wl.fp8_pool_pages(0, pages), wl.fp8_pool_pages(1, pages)
    kc_s = torch.stack([kp[p] for p in pages])
    vc_s = torch.stack([vp[p] for p in pages])
    bt = torch.full_like(wl.block_table, W.INT32_MAX)
    for s in seqs:
        ps = wl.pages_of(s)
        bt[s, :len(ps)] = torch.tensor([remap[p] for p in ps], dtype=torch.int32)
    bs = wl.block_size
    slots = torch.tensor([remap[int(x) // bs] * bs + int(x) % bs for x in wl.slot_mapping],
                         dtype=torch.int64)
    oracle.reshape_and_cache_e4m3(wl.k_new, wl.v_new, slots, kc_s, vc_s, wl.kv_scales(0),
                                  wl.kv_scales(1))
    g = torch.Generator().manual_seed(17)
    rows = {}
    for s in seqs:
        n = wl.q_lens[s]
        pick = {0, 15, 16, 127, 128, n // 2, n - 1} | set(int(x) for x in
                                                         torch.randint(0, n, (12,), generator=g))
        rows[s] = sorted(pick)
    ref_o, ref_l = oracle.varlen_attention_e4m3(wl.q, kc_s, vc_s, wl.cu_seqlens_q, wl.seqused_k,
                                                bt, wl.softmax_scale, True, wl.kv_scales(0),
                                                wl.kv_scales(1), rows=rows)
    cu = wl.cu_seqlens_q.tolist()
    tokens = torch.tensor([cu[s] + r for s in seqs for r in rows[s]])
    assert_close(out, lse, ref_o[tokens], ref_l[:, tokens], tokens=tokens)
