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
it may see with an exact softmax, in float64, on the bf16 or f16 input values. The
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
def attend_dense(q, k, v, softmax_scale, causal, q_len, kv_len, rows=None, row_chunk=512,
                 sinks=None):
    """Exact softmax attention of query rows against dense keys of one sequence.

    q: [q_len, H, D], k, v: [kv_len, H_kv, D] (any float type; computed in
    float64). ``rows`` selects which of the q_len rows to compute (default all).
    ``sinks``: optional per-query-head logits ([FA-vLLM] §1.2 and §1.3: the
    `s_aux` learnable sink token of FA3/FA4), read as one extra key of logit
    sinks[h] (in the units of softmax_scale * q.k) and value zero: it joins
    the softmax denominator and the LSE only.
    Returns out [n_rows, H, D] float64 and lse [H, n_rows] float64.
    """
    H, D = q.shape[1], q.shape[2]
    H_kv = k.shape[1]
    rows = torch.arange(q_len, dtype=torch.long) if rows is None else \
        torch.as_tensor(rows, dtype=torch.long)
    n = rows.numel()
    out = torch.zeros((n, H, D), dtype=F64)
    lse = torch.full((H, n), NEG_INF, dtype=F64)
    if sinks is not None:
        for h in range(H):
            lse[h, :] = float(sinks[h])      # a row with no visible key sees only the sink
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
            if sinks is not None:
                m = torch.where(any_visible, torch.maximum(m, torch.tensor(float(sinks[h]), dtype=F64)), m)
            p = torch.exp(logits - m[:, None])
            l = p.sum(dim=1)
            if sinks is not None:
                l = l + torch.exp(float(sinks[h]) - m)
            safe_l = torch.where(any_visible, l, torch.ones_like(l))
            o = (p @ v64[:, hk, :]) / safe_l[:, None]
            out[c0:c0 + r.numel(), h, :] = torch.where(any_visible[:, None], o, torch.zeros_like(o))
            lse_h = log_sum_exp_from(m, safe_l)
            lse[h, c0:c0 + r.numel()] = torch.where(any_visible, lse_h, lse[h, c0:c0 + r.numel()])
    return out, lse


def varlen_attention(q, key_cache, value_cache, cu_seqlens_q, seqused_k, block_table,
                     softmax_scale, causal, rows=None, sinks=None):
    """Varlen attention over a paged KV cache ([FA-vLLM] §4 and §5).

    q: [T, H, D] packed by cu_seqlens_q [S+1]; seqused_k [S]; block_table
    [S, max_blocks] int32; caches [num_blocks, block_size, H_kv, D].
    ``rows``: optional {seq index: list of local query rows} to compute only
    those rows (others stay out = 0, lse = -inf). ``sinks``: optional [H]
    sink logits (see attend_dense).
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
        o, l = attend_dense(q[q0:q1], k, v, softmax_scale, causal, q_len, kv_len, rows=local,
                            sinks=sinks)
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


def merge_attn_states_n(parts_out, parts_lse):
    """Combine n partial attention results over disjoint key sets ([FA-vLLM]
    §9: DCP merges the ranks' partial results by their LSEs; §6.3 / §8.2 give
    the two-state merge this generalises).

    parts_out: [n, T, H, D]; parts_lse: [n, H, T] natural log. With
    m = max_r lse_r and w_r = exp(lse_r - m): out = sum_r w_r out_r / sum_r w_r,
    lse = m + ln(sum_r w_r). A row whose LSEs are all -inf saw no key: out 0,
    lse -inf.
    """
    po, pl = parts_out.to(F64), parts_lse.to(F64)
    n, T, H, D = po.shape
    out = torch.zeros((T, H, D), dtype=F64)
    lse = torch.full((H, T), NEG_INF, dtype=F64)
    for h in range(H):
        for t in range(T):
            ls = [float(pl[r, h, t]) for r in range(n)]
            m = max(ls)
            if m == NEG_INF:
                continue
            ws = [math.exp(x - m) for x in ls]
            acc = torch.zeros(D, dtype=F64)
            for r in range(n):
                acc += ws[r] * po[r, t, h]
            tot = math.fsum(ws)
            out[t, h] = acc / tot
            lse[h, t] = m + math.log(tot)
    return out, lse


def dcp_decode_attention(q, key_cache, value_cache, cu_seqlens_q, shard_tables, shard_lens,
                         softmax_scale):
    """Decode context parallelism over virtual ranks ([FA-vLLM] §9 and the
    DCP branch of §4): every rank holds some of each sequence's KV blocks;
    each computes the attention of all the queries against its own shard,
    non-causal (the decode query follows every key), and the ranks' partial
    (out, lse) are merged by their LSEs.

    shard_tables[r]: int32 [S, max_blocks] block table of rank r's shard,
    shard_lens[r]: int32 [S] its key counts. Returns the merged (out, lse).
    """
    outs, lses = [], []
    for bt, lens in zip(shard_tables, shard_lens):
        o, l = varlen_attention(q, key_cache, value_cache, cu_seqlens_q, lens, bt,
                                softmax_scale, causal=False)
        outs.append(o)
        lses.append(l)
    return merge_attn_states_n(torch.stack(outs), torch.stack(lses))


# --------------------------------------------------------------------------
# Cascade (shared-prefix) attention ([FA-vLLM] §6.3).
# --------------------------------------------------------------------------
def cascade_attention(q, key_cache, value_cache, cu_seqlens_q, seqused_k, block_table,
                      softmax_scale, common_prefix_len, rows=None, sinks=None):
    """What cascade attention computes: flat causal attention over prefix || suffix.

    With every query in the private suffix (kv_len - q_len >= common_prefix_len),
    the bottom-right causal rule makes all prefix keys visible to every query,
    so the result is ordinary causal varlen attention over the whole KV.
    """
    return varlen_attention(q, key_cache, value_cache, cu_seqlens_q, seqused_k, block_table,
                            softmax_scale, causal=True, rows=rows, sinks=sinks)


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


# --------------------------------------------------------------------------
# FP8 (e4m3) KV cache ([FA/FI] 役割 and 境界と失敗: FlashInfer and FA3 accept an
# fp8 / fp8_e4m3 KV cache with per-head quant scales; [FA-vLLM] §10 lists an FP8
# KV cache among the backends' features). The pools hold e4m3 bytes; a byte c
# of KV head h means e4m3(c) * scale[h], and a new row is written as
# e4m3(x / scale[h]). The pages do not define the format, so it is the OCP
# 8-bit floating point "E4M3" one: 1 sign, 4 exponent bits (bias 7), 3
# mantissa bits; normal values 2^(e-7) * (1 + m/8) for e = 1..15, except the
# all-ones pattern S.1111.111, which is NaN; subnormals 2^-6 * m/8; largest
# finite 448; no infinities. Readings where the pages are silent: rounding is
# to nearest with ties to even, values beyond 448 saturate to +-448, and the
# division x / scale is IEEE float32 (the precision that decides the code
# is the kernel's).
# --------------------------------------------------------------------------
E4M3_MAX = 448.0


def e4m3_decode(code: int) -> float:
    """Value of one e4m3 byte (NaN for S.1111.111)."""
    s = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return s * (m / 8.0) * 2.0 ** -6
    return s * (1.0 + m / 8.0) * 2.0 ** (e - 7)


def e4m3_round(y: float) -> float:
    """Nearest e4m3 value to y (ties to even), saturating at +-448.

    Within [2^E, 2^(E+1)) (E >= -6; E = -6 also covers the subnormals
    [0, 2^-6)) the e4m3 values are the multiples of q = 2^(E-3), so y rounds
    to the nearest multiple of q; on a tie the even multiple wins, which is
    the value whose last mantissa bit is 0.
    """
    if y != y:
        return y
    a = abs(y)
    if a >= E4M3_MAX:
        return math.copysign(E4M3_MAX, y)
    if a == 0.0:
        return math.copysign(0.0, y)
    E = -6
    while E < 8 and 2.0 ** (E + 1) <= a:
        E += 1
    q = 2.0 ** (E - 3)
    n = a / q                  # exact: q is a power of two
    r = math.floor(n)
    frac = n - r
    if frac > 0.5 or (frac == 0.5 and r % 2 == 1):
        r += 1
    return math.copysign(min(r * q, E4M3_MAX), y)


def e4m3_encode(y: float) -> int:
    """The e4m3 byte of e4m3_round(y); NaN encodes as 0x7F."""
    v = e4m3_round(y)
    if v != v:
        return 0x7F
    sign = 0x80 if math.copysign(1.0, v) < 0 else 0
    a = abs(v)
    if a == 0.0:
        return sign
    if a < 2.0 ** -6:                      # subnormal: a = (m/8) * 2^-6
        return sign | int(a / 2.0 ** -9)
    e = 0
    while 2.0 ** (e + 1) <= a:
        e += 1
    while 2.0 ** e > a:
        e -= 1
    m = int((a / 2.0 ** e - 1.0) * 8.0)    # exact: a has at most 4 significant bits
    return sign | ((e + 7) << 3) | m


def e4m3_table():
    """float64 [256]: the value of every e4m3 byte."""
    return torch.tensor([e4m3_decode(c) for c in range(256)], dtype=F64)


def quantize_e4m3(x, scale):
    """e4m3 bytes (uint8, same shape) of x / scale[h] for x [..., H_kv, D].

    x / scale is IEEE float32 division; the quotient then rounds to the
    nearest e4m3 value as in e4m3_round, found here by searching the sorted
    finite non-negative values (codes 0x00 .. 0x7E, increasing with the code):
    the closer neighbour wins, a tie goes to the even code, |y| >= 448 gives
    0x7E, and the sign bit is copied.
    """
    s = torch.as_tensor(scale, dtype=torch.float32).reshape(-1)
    y = (x.to(torch.float32) / s[:, None]).to(F64)          # float32 quotient, exact in f64
    vals = e4m3_table()[:0x7F]                              # 0, 2^-9, ..., 448
    a = y.abs()
    hi = torch.searchsorted(vals, a.contiguous()).clamp(max=0x7E)
    lo = (hi - 1).clamp(min=0)
    dlo, dhi = a - vals[lo], vals[hi] - a
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (hi % 2 == 0))
    code = torch.where(pick_hi, hi, lo)
    code = torch.where(a >= E4M3_MAX, torch.full_like(code, 0x7E), code)
    code = torch.where(torch.signbit(y), code | 0x80, code)
    code = torch.where(torch.isnan(y), torch.full_like(code, 0x7F), code)
    return code.to(torch.uint8)


def dequantize_e4m3(codes, scale):
    """float64 e4m3(codes) * scale[h] for codes [..., H_kv, D]."""
    s = torch.as_tensor(scale, dtype=torch.float32).to(F64).reshape(-1)
    return e4m3_table()[codes.long()] * s[:, None]


def reshape_and_cache_e4m3(key, value, slot_mapping, key_cache, value_cache, k_scale, v_scale):
    """The FP8 cache write: reshape_and_cache of the e4m3 bytes of
    key / k_scale[h] and value / v_scale[h] into uint8 pools."""
    reshape_and_cache(quantize_e4m3(key, k_scale), quantize_e4m3(value, v_scale), slot_mapping,
                      key_cache, value_cache)


def varlen_attention_e4m3(q, key_cache, value_cache, cu_seqlens_q, seqused_k, block_table,
                          softmax_scale, causal, k_scale, v_scale, rows=None):
    """Varlen attention over e4m3 pools: the plain definition applied to the
    dequantized keys and values e4m3(c) * scale[h]."""
    return varlen_attention(q, dequantize_e4m3(key_cache, k_scale),
                            dequantize_e4m3(value_cache, v_scale), cu_seqlens_q, seqused_k,
                            block_table, softmax_scale, causal, rows=rows)
