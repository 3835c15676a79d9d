"""GPU parity of the n-state merge and of decode context parallelism over
virtual ranks ("FlashAttention 在 vLLM 中的实现分析" §9: each rank attends
over its KV shard, non-causal for decode, and the partial (out, lse) are
merged by LSE) against the fp64 oracle."""
import pytest
import torch

import oracle
import paged_kv_varlen_attn_gb300 as pa
import workloads as W
from helpers import LSE_TOL, OUT_TOL, oracle_full, oracle_sampled

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_varlen_attn_gb300 import _build
    _build.build()
    pa.load_library()


def check(out, lse, ref_o, ref_l, tokens=None):
    o, l = out.cpu().double(), lse.cpu().double()
    if tokens is not None:
        o, l = o[tokens], l[:, tokens]
    fin = torch.isfinite(ref_l)
    assert torch.equal(fin, torch.isfinite(l))
    assert (o - ref_o).abs().max().item() <= OUT_TOL
    if fin.any():
        assert (l[fin] - ref_l[fin]).abs().max().item() <= LSE_TOL


@pytest.mark.parametrize("n,T,H,D", [(1, 5, 4, 128), (2, 33, 8, 64), (3, 17, 32, 128),
                                     (7, 9, 4, 128), (33, 6, 2, 64)])
def test_merge_n_matches_oracle(n, T, H, D):
    g = torch.Generator().manual_seed(100 + n)
    # Attention-like parts (outputs are convex combinations of values, O(1)):
    # the 1e-2 max-abs bar is for O(1) outputs; bf16 rounding alone is 1/64
    # for a value in [4, 8).
    po = (torch.randn(n, T, H, D, generator=g) * 0.5).to(torch.bfloat16)
    pl = torch.randn(n, H, T, generator=g) * 4
    pl[0, 0, :] = float("-inf")                 # a part that saw no key for head 0
    if n > 1:
        pl[:, 1 % H, 0] = float("-inf")         # a row that saw no key at all
    ref_o, ref_l = oracle.merge_attn_states_n(po, pl)
    out, lse = pa.merge_attn_states_n(po.to(DEV), pl.to(DEV))
    torch.cuda.synchronize()
    check(out, lse, ref_o, ref_l)
    # and element by element within one bf16 rounding of the exact merge
    err = (out.cpu().double() - ref_o).abs()
    assert (err <= ref_o.abs() * 2.0 ** -8 + 1e-3).all()
    # out may alias a part
    pod = po.to(DEV)
    out2, lse2 = pa.merge_attn_states_n(pod, pl.to(DEV), out=pod[0])
    torch.cuda.synchronize()
    assert torch.equal(out2.cpu(), out.cpu()) and torch.equal(lse2.cpu(), lse.cpu())


def dcp_gpu(wl, ranks, status=None):
    """R virtual ranks: pa_varlen_fwd (non-causal) over each rank's shard into
    one stacked buffer, then the n-state merge."""
    tables, lens = W.dcp_shards(wl, ranks)
    T, H, D = wl.q.shape
    kc, vc = wl.pool(0, device=DEV), wl.pool(1, device=DEV)
    q = wl.q.to(DEV)
    pa.reshape_and_cache(wl.k_new.to(DEV), wl.v_new.to(DEV), kc, vc, wl.slot_mapping.to(DEV))
    parts = torch.empty((ranks, T, H, D), dtype=torch.bfloat16, device=DEV)
    plse = torch.empty((ranks, H, T), dtype=torch.float32, device=DEV)
    cu = wl.cu_seqlens_q.to(DEV)
    for r in range(ranks):
        mk = max(1, int(lens[r].max()))
        pa.varlen_fwd(q, kc, vc, cu, lens[r].to(DEV), tables[r].to(DEV), wl.max_seqlen_q, mk,
                      wl.softmax_scale, False, out=parts[r], lse=plse[r], dev_status=status)
    out, lse = pa.merge_attn_states_n(parts, plse)
    flat_o, flat_l = pa.varlen_fwd(q, kc, vc, cu, wl.seqused_k.to(DEV), wl.block_table.to(DEV),
                                   wl.max_seqlen_q, wl.max_seqlen_k, wl.softmax_scale, True)
    torch.cuda.synchronize()
    return out, lse, flat_o, flat_l


@pytest.mark.parametrize("seed,ranks,Hk,bs", [(301, 2, 8, 16), (302, 4, 2, 32), (303, 3, 4, 16),
                                              (304, 8, 8, 64)])
def test_dcp_virtual_ranks_decode(seed, ranks, Hk, bs):
    wl = W.random_case(seed, num_seqs=7, num_heads=Hk * 4, num_kv_heads=Hk, head_size=128,
                       block_size=bs, max_q=1, max_kv=1500, decode_frac=1.0)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out, lse, flat_o, flat_l = dcp_gpu(wl, ranks, status)
    ref_o, ref_l = oracle_full(wl)
    check(out, lse, ref_o, ref_l)
    check(flat_o, flat_l, ref_o, ref_l)
    assert int(status.item()) == 0


def test_dcp_virtual_ranks_decode_llama8b_sampled():
    """The full-size decode batch over 4 virtual ranks, checked on sampled
    sequences (decode over ranks equals flat causal decode)."""
    wl = W.decode_llama8b()
    out, lse, _, _ = dcp_gpu(wl, 4)
    g = torch.Generator().manual_seed(11)
    seqs = sorted(set(int(x) for x in torch.randint(0, wl.num_seqs, (6,), generator=g)))
    ref = oracle_sampled(wl, {s: [0] for s in seqs})
    for s, (tok, ro, rl) in ref.items():
        check(out, lse, ro, rl, tokens=tok)
