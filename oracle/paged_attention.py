"""Plain fp64 CPU oracle for varlen attention over a paged KV cache.

TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the benchmark's
CPU-baseline leg may import this module. The product path (the CUDA library
and its Python binding) never calls it and shares no code with it.

Sources (web pages describing vLLM's attention backends; cited by key):
  [FA-vLLM]  "FlashAttention 在 vLLM 中的实现分析" (blog.chen3feng.top,
             vllm-analysis/07), sections 1.1, 4, 4.2, 5, 6.3, 8.2, 9.
  [FA/FI]    "FlashAttention と FlashInfer:2 大 GPU アテンションバックエンド"
             (vllm-arch-zh.pages.dev/ja/attention/flash), sections 役割,
             データフロー, 境界と失敗.
  [Backend]  "AttentionBackend:アテンションバックエンド抽象レイヤー"
             (vllm-arch-zh.pages.dev/ja/attention/backend), section 境界と失敗.

What is computed is the plain definition: every query row attends to the keys
it may see with an exact softmax, in float64, on the bf16 input values. The
tiled online softmax of [FA-vLLM] §1.1 reaches the same numbers up to rounding
order, so the oracle does not tile. Readings of points the pages leave open:
  * causal alignment is bottom-right: query i of a sequence with q_len
    queries and kv_len keys sits at position kv_len - q_len + i and sees the
    keys at positions <= that (a decode query therefore sees every key, as the
    causal suffix pass of [FA-vLLM] §6.3 requires);
  * GQA heads are grouped contiguously: query head h reads KV head
    h // (num_heads / num_kv_heads);
  * the LSE is the natural-log log-sum-exp (the base-e vs base-2 pitfall named
    in [Backend] 境界と失敗), stored [num_heads, num_tokens];
  * a row that sees no key has output 0 and LSE -inf; a slot < 0 is skipped.

Every function here is pinned by tests under tests/ (brute force on tiny
inputs, closed forms, a torch library routine, and invariants); none is
"parity unpinned".
"""
from __future__ import annotations

import math

import torch

F64 = torch.float64
NEG_INF = float("-inf")


# --------------------------------------------------------------------------
# reshape_and_cache: the slot_mapping scatter ([FA-vLLM] §4.2, §8.2;
# [FA/FI] 役割: the KV-cache write is a separate op before attention).
# --------------------------------------------------------------------------
def reshape_and_cache(key, value, slot_mapping, key_cache, value_cache):
    """Write new K/V rows into their pages, in place.

    key, value: [num_tokens, num_kv_heads, head_size]; slot_mapping: int64
    [num_tokens]; key_cache, value_cache: [num_blocks, block_size,
    num_kv_heads, head_size]. Token t goes to page slot // block_size, row
    slot % block_size. A negative slot means "no write" (padding).
    """
    block_size = key_cache.shape[1]
    for t in range(key.shape[0]):
        slot = int(slot_mapping[t])
        if slot < 0:
            continue
        page, row = slot // block_size, slot % block_size
        key_cache[page, row] = key[t]
        value_cache[page, row] = value[t]


# --------------------------------------------------------------------------
# Paged addressing ([FA-vLLM] §5: physical block = block_table[seq][logical
# block], then the offset inside the block).
# --------------------------------------------------------------------------
def logical_to_physical(block_table_row, positions, block_size):
    """(page id, row in page) of each logical key position of one sequence."""
    positions = torch.as_tensor(positions, dtype=torch.long)
    pages = block_table_row[positions // block_size].long()
    return pages, positions % block_size


def gather_kv(cache, block_table_row, kv_len, start=0):
    """Keys [start, kv_len) of one sequence as a dense [n, num_kv_heads, D] tensor."""
    block_size = cache.shape[1]
    pos = torch.arange(start, kv_len, dtype=torch.long)
    pages, rows = logical_to_physical(block_table_row, pos, block_size)
    return cache[pages, rows]


def kv_head_of(h, num_heads, num_kv_heads):
    """GQA: contiguous groups of num_heads / num_kv_heads query heads share a KV head."""
    return h // (num_heads // num_kv_heads)


def causal_last_visible(q_len, kv_len, i):
    """Last key position query row i may see under the bottom-right causal rule."""
    return kv_len - q_len + i


def log_sum_exp_from(m, l):
    """Natural-log LSE from row maxima m and sums l of exp(logit - m) (tensors)."""
    return m + torch.log(l)


# --------------------------------------------------------------------------
# Attention of one sequence ([FA-vLLM] §1.1 target result; §4 varlen call).
# --------------------------------------------------------------------------
def attend_dense(q, k, v, softmax_scale, causal, q_len, kv_len, rows=None, row_chunk=512):
    """Exact softmax attention of query rows against dense keys of one sequence.

    q: [q_len, H, D], k, v: [kv_len, H_kv, D] (any float type; computed in
    float64). ``rows`` selects which of the q_len rows to compute (default all).
    Returns out [n_rows, H, D] float64 and lse [H, n_rows] float64.
    """
    H, D = q.shape[1], q.shape[2]
    H_kv = k.shape[1]
    rows = torch.arange(q_len, dtype=torch.long) if rows is None else \
        torch.as_tensor(rows, dtype=torch.long)
    n = rows.numel()
    out = torch.zeros((n, H, D), dtype=F64)
    lse = torch.full((H, n), NEG_INF, dtype=F64)
    if n == 0 or kv_len == 0:
        return out, lse
    q64, k64, v64 = q.to(F64), k.to(F64), v.to(F64)
    key_pos = torch.arange(kv_len, dtype=torch.long)
    for c0 in range(0, n, row_chunk):
        r = rows[c0:c0 + row_chunk]
        if causal:
            last = torch.tensor([causal_last_visible(q_len, kv_len, int(i)) for i in r],
                                dtype=torch.long)
            visible = key_pos[None, :] <= last[:, None]
        else:
            visible = torch.ones((r.numel(), kv_len), dtype=torch.bool)
        any_visible = visible.any(dim=1)
        for h in range(H):
            hk = kv_head_of(h, H, H_kv)
            logits = softmax_scale * (q64[r, h, :] @ k64[:, hk, :].T)
            logits = logits.masked_fill(~visible, NEG_INF)
            m = torch.where(any_visible, logits.max(dim=1).values, torch.zeros_like(any_visible, dtype=F64))
            p = torch.exp(logits - m[:, None])
            l = p.sum(dim=1)
            safe_l = torch.where(any_visible, l, torch.ones_like(l))
            o = (p @ v64[:, hk, :]) / safe_l[:, None]
            out[c0:c0 + r.numel(), h, :] = torch.where(any_visible[:, None], o, torch.zeros_like(o))
            lse_h = log_sum_exp_from(m, safe_l)
            lse[h, c0:c0 + r.numel()] = torch.where(any_visible, lse_h,
                                                    torch.full_like(lse_h, NEG_INF))
    return out, lse


def varlen_attention(q, key_cache, value_cache, cu_seqlens_q, seqused_k, block_table,
                     softmax_scale, causal, rows=None):
    """Varlen attention over a paged KV cache ([FA-vLLM] §4 and §5).

    q: [T, H, D] packed by cu_seqlens_q [S+1]; seqused_k [S]; block_table
    [S, max_blocks] int32; caches [num_blocks, block_size, H_kv, D].
    ``rows``: optional {seq index: list of local query rows} to compute only
    those rows (others stay out = 0, lse = -inf).
    Returns out [T, H, D] float64 and lse [H, T] float64.
    """
    T, H, D = q.shape
    out = torch.zeros((T, H, D), dtype=F64)
    lse = torch.full((H, T), NEG_INF, dtype=F64)
    cu = [int(x) for x in cu_seqlens_q]
    for s in range(len(cu) - 1):
        if rows is not None and s not in rows:
            continue
        q0, q1 = cu[s], cu[s + 1]
        q_len, kv_len = q1 - q0, int(seqused_k[s])
        if q_len == 0:
            continue
        k = gather_kv(key_cache, block_table[s], kv_len)
        v = gather_kv(value_cache, block_table[s], kv_len)
        local = None if rows is None else torch.as_tensor(rows[s], dtype=torch.long)
        o, l = attend_dense(q[q0:q1], k, v, softmax_scale, causal, q_len, kv_len, rows=local)
        idx = torch.arange(q0, q1) if local is None else q0 + local
        out[idx] = o
        lse[:, idx] = l
    return out, lse


# --------------------------------------------------------------------------
# merge_attn_states ([FA-vLLM] §6.3 step 3 and §8.2: LSE-weighted combine).
# --------------------------------------------------------------------------
def merge_attn_states(prefix_out, prefix_lse, suffix_out, suffix_lse):
    """Combine two partial attention results over disjoint key sets.

    out: [T, H, D]; lse: [H, T] natural log. With m = max(a, b),
    wa = exp(a - m), wb = exp(b - m): out = (wa*oa + wb*ob) / (wa + wb) and
    lse = m + ln(wa + wb). If both LSEs are -inf the row saw no key: out = 0,
    lse = -inf.
    """
    oa, ob = prefix_out.to(F64), suffix_out.to(F64)
    a, b = prefix_lse.to(F64), suffix_lse.to(F64)
    T, H, D = oa.shape
    out = torch.zeros((T, H, D), dtype=F64)
    lse = torch.full((H, T), NEG_INF, dtype=F64)
    for h in range(H):
        for t in range(T):
            la, lb = float(a[h, t]), float(b[h, t])
            m = max(la, lb)
            if m == NEG_INF:
                continue
            wa, wb = math.exp(la - m), math.exp(lb - m)
            out[t, h] = (wa * oa[t, h] + wb * ob[t, h]) / (wa + wb)
            lse[h, t] = m + math.log(wa + wb)
    return out, lse


# --------------------------------------------------------------------------
# Cascade (shared-prefix) attention ([FA-vLLM] §6.3).
# --------------------------------------------------------------------------
def cascade_attention(q, key_cache, value_cache, cu_seqlens_q, seqused_k, block_table,
                      softmax_scale, common_prefix_len, rows=None):
    """What cascade attention computes: flat causal attention over prefix || suffix.

    With every query in the private suffix (kv_len - q_len >= common_prefix_len),
    the bottom-right causal rule makes all prefix keys visible to every query,
    so the result is ordinary causal varlen attention over the whole KV.
    """
    return varlen_attention(q, key_cache, value_cache, cu_seqlens_q, seqused_k, block_table,
                            softmax_scale, causal=True, rows=rows)


def cascade_attention_steps(q, key_cache, value_cache, cu_seqlens_q, seqused_k, block_table,
                            softmax_scale, common_prefix_len):
    """The three steps of [FA-vLLM] §6.3, taken literally.

    1. prefix pass: every query token of the batch, as one non-causal segment,
       against the shared pages of row 0 (block_table[:1], first
       common_prefix_len keys), keeping the LSE;
    2. suffix pass: each sequence, causal, against its own pages from block
       common_prefix_len // block_size on (kv_len - common_prefix_len keys);
    3. merge_attn_states(prefix, suffix).
    """
    T, H, D = q.shape
    bs = key_cache.shape[1]
    P = common_prefix_len
    pfx_k = gather_kv(key_cache, block_table[0], P)
    pfx_v = gather_kv(value_cache, block_table[0], P)
    pfx_out, pfx_lse = attend_dense(q, pfx_k, pfx_v, softmax_scale, False, T, P)
    nb = P // bs
    suf_out = torch.zeros((T, H, D), dtype=F64)
    suf_lse = torch.full((H, T), NEG_INF, dtype=F64)
    cu = [int(x) for x in cu_seqlens_q]
    for s in range(len(cu) - 1):
        q0, q1 = cu[s], cu[s + 1]
        if q1 == q0:
            continue
        kv_len = int(seqused_k[s]) - P
        k = gather_kv(key_cache, block_table[s, nb:], kv_len)
        v = gather_kv(value_cache, block_table[s, nb:], kv_len)
        o, l = attend_dense(q[q0:q1], k, v, softmax_scale, True, q1 - q0, kv_len)
        suf_out[q0:q1] = o
        suf_lse[:, q0:q1] = l
    return merge_attn_states(pfx_out, pfx_lse, suf_out, suf_lse)
