"""Shared test helpers: run the oracle and the CUDA path on the same seeded
workload. The oracle side never sees a value produced by the CUDA path."""
import torch

import oracle
import workloads as W

OUT_TOL = 1e-2   # max-abs error of bf16 outputs (O(1) inputs)
LSE_TOL = 1e-3   # absolute error of the natural-log LSE


def oracle_pools(wl):
    """Full CPU pools after the oracle's scatter of the new tokens."""
    kc, vc = wl.pool(0), wl.pool(1)
    oracle.reshape_and_cache(wl.k_new, wl.v_new, wl.slot_mapping, kc, vc)
    return kc, vc


def oracle_full(wl, causal=None, cascade=False):
    kc, vc = oracle_pools(wl)
    args = (wl.q, kc, vc, wl.cu_seqlens_q, wl.seqused_k, wl.block_table, wl.softmax_scale)
    if cascade:
        return oracle.cascade_attention(*args, wl.common_prefix_len)
    return oracle.varlen_attention(*args, wl.causal if causal is None else causal)


def oracle_sampled(wl, rows_by_seq, causal=None):
    """Oracle out/lse for selected query rows of a full-size workload.

    Only the pages of the selected sequences are regenerated (from the
    workload's seeds) into a compact CPU pool; the selected sequences' new
    tokens are scattered into it by the oracle. Returns {seq: (global token
    indices, out [n, H, D], lse [H, n])}.
    """
    seqs = sorted(rows_by_seq)
    bs = wl.block_size
    pages = []
    for s in seqs:
        for p in wl.pages_of(s):
            if p not in pages:
                pages.append(p)
    remap = {p: i for i, p in enumerate(pages)}
    kpages, vpages = wl.pool_pages(0, pages), wl.pool_pages(1, pages)
    kc = torch.stack([kpages[p] for p in pages])
    vc = torch.stack([vpages[p] for p in pages])
    cu = wl.cu_seqlens_q.tolist()
    # remapped block table rows and new-token slots of the selected sequences
    bt = torch.full((len(seqs), wl.block_table.shape[1]), W.INT32_MAX, dtype=torch.int32)
    tok_idx = []
    for i, s in enumerate(seqs):
        ps = wl.pages_of(s)
        bt[i, :len(ps)] = torch.tensor([remap[p] for p in ps], dtype=torch.int32)
        tok_idx.append(torch.arange(cu[s], cu[s + 1]))
    tok_idx = torch.cat(tok_idx)
    slots = wl.slot_mapping[tok_idx]
    new_slots = torch.tensor([remap[int(x) // bs] * bs + int(x) % bs for x in slots],
                             dtype=torch.int64)
    oracle.reshape_and_cache(wl.k_new[tok_idx], wl.v_new[tok_idx], new_slots, kc, vc)
    q_lens = [wl.q_lens[s] for s in seqs]
    cu_sub = torch.tensor([0] + list(torch.tensor(q_lens).cumsum(0).tolist()), dtype=torch.int32)
    lens = torch.tensor([wl.kv_lens[s] for s in seqs], dtype=torch.int32)
    rows = {i: rows_by_seq[s] for i, s in enumerate(seqs)}
    out, lse = oracle.varlen_attention(wl.q[tok_idx], kc, vc, cu_sub, lens, bt, wl.softmax_scale,
                                       wl.causal if causal is None else causal, rows=rows)
    res = {}
    for i, s in enumerate(seqs):
        local = torch.as_tensor(rows_by_seq[s], dtype=torch.long)
        sub_idx = int(cu_sub[i]) + local
        res[s] = (cu[s] + local, out[sub_idx], lse[:, sub_idx])
    return res


def to_dev(wl, device):
    """Device copies of everything the CUDA path needs (pool before scatter)."""
    d = {
        "q": wl.q.to(device),
        "k_new": wl.k_new.to(device),
        "v_new": wl.v_new.to(device),
        "slot_mapping": wl.slot_mapping.to(device),
        "cu_seqlens_q": wl.cu_seqlens_q.to(device),
        "seqused_k": wl.seqused_k.to(device),
        "block_table": wl.block_table.to(device),
        "key_cache": wl.pool(0, device=device),
        "value_cache": wl.pool(1, device=device),
    }
    return d
