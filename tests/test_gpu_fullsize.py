"""GPU parity at the sizes the benchmark reports: the scatter of the chunked
prefill batch's 16,440 new tokens (bit-exact over the whole pools), and the
two-state and n-state LSE merges of 16,384 tokens x 32 heads x 128 (the
merge is row-independent, so the oracle checks a seeded sample of tokens,
first and last included)."""
import pytest
import torch

import oracle
import paged_kv_varlen_attn_gb300 as pa
import workloads as W
from test_gpu_parity import DEV, assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_varlen_attn_gb300 import _build
    _build.build()
    pa.load_library()


def _sample_tokens(T, n=48, seed=0):
    g = torch.Generator().manual_seed(seed)
    pick = {0, 1, T // 2, T - 2, T - 1}
    pick |= set(int(x) for x in torch.randint(0, T, (n,), generator=g))
    return torch.tensor(sorted(pick), dtype=torch.long)


def test_scatter_bit_exact_chunked_prefill_batch():
    wl = W.chunked_prefill_mix()
    assert wl.k_new.shape[0] == 16440
    kc_ref, vc_ref = wl.pool(0), wl.pool(1)
    kc, vc = kc_ref.to(DEV), vc_ref.to(DEV)
    oracle.reshape_and_cache(wl.k_new, wl.v_new, wl.slot_mapping, kc_ref, vc_ref)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    pa.reshape_and_cache(wl.k_new.to(DEV), wl.v_new.to(DEV), kc, vc, wl.slot_mapping.to(DEV),
                         dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(kc.cpu().view(torch.int16), kc_ref.view(torch.int16))
    assert torch.equal(vc.cpu().view(torch.int16), vc_ref.view(torch.int16))


def _states(g, n, T, H, D):
    # A partial output is a convex combination of value rows, so its entries
    # are O(1) (the tolerance is stated for O(1) inputs): N(0,1) clamped to
    # +-2. Unclamped, 67M draws reach |x| ~ 5.7, where the one bf16 rounding
    # of the result alone is up to 2^-6 = 0.0156.
    o = torch.randn((n, T, H, D), generator=g).clamp_(-2.0, 2.0).to(torch.bfloat16)
    lse = torch.randn((n, H, T), generator=g) * 3
    # rows whose states are all -inf, and rows where one state is -inf
    lse[:, 0, :7] = float("-inf")
    lse[0, 1, 7:40] = float("-inf")
    return o, lse


def test_merge_16k_tokens_sampled():
    T, H, D = 16384, 32, 128
    g = torch.Generator().manual_seed(71)
    o, lse = _states(g, 2, T, H, D)
    out, out_lse = pa.merge_attn_states(o[0].to(DEV), lse[0].to(DEV), o[1].to(DEV),
                                        lse[1].to(DEV))
    torch.cuda.synchronize()
    idx = torch.cat([torch.arange(8), _sample_tokens(T, seed=72)]).unique()
    ref_o, ref_l = oracle.merge_attn_states(o[0][idx], lse[0][:, idx], o[1][idx],
                                            lse[1][:, idx])
    assert_close(out.cpu()[idx], out_lse.cpu()[:, idx], ref_o, ref_l)


def test_merge_n_4parts_16k_tokens_sampled():
    n, T, H, D = 4, 16384, 32, 128
    g = torch.Generator().manual_seed(73)
    o, lse = _states(g, n, T, H, D)
    out, out_lse = pa.merge_attn_states_n(o.to(DEV), lse.to(DEV))
    torch.cuda.synchronize()
    idx = torch.cat([torch.arange(8), _sample_tokens(T, seed=74)]).unique()
    ref_o, ref_l = oracle.merge_attn_states_n(o[:, idx], lse[:, :, idx])
    assert_close(out.cpu()[idx], out_lse.cpu()[:, idx], ref_o, ref_l)
