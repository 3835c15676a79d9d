"""Seeded synthetic inputs for paged varlen attention, shared by the tests, the
benchmark and the smoke check.

This module only draws random numbers and lays out metadata the way a serving
engine's scheduler would hand it to the attention backend (FlashAttention in
vLLM analysis page, section 5 "PagedAttention integration": a K/V page pool
[num_blocks, block_size, num_kv_heads, head_size], an int32 block_table
[num_seqs, max_blocks], seqused_k and cu_seqlens_q). It holds none of the
attention arithmetic: no softmax, no gather, no scatter.

Recipe (every workload):
  * one torch CPU generator seeded with ``seed``; draw order is lengths,
    page permutation, Q, new K, new V;
  * pool contents (the prior context) are N(0,1) drawn per chunk of pages from
    a generator whose seed is a splitmix64 mix of (seed, K|V, chunk index), so
    any page can be regenerated on its own and chunks can be drawn in parallel;
  * pages are handed to sequences in order from a random permutation of the
    pool; unused block_table entries hold INT32_MAX;
  * the new tokens of sequence s are its last q_len[s] positions, and their
    slot is (physical page) * block_size + (position % block_size);
  * all values are drawn in fp32 and rounded to the workload's element type
    (bf16 by default, or f16); both the oracle and the GPU path consume the
    same rounded values.
  * FP8 (e4m3) pools: the prior context of KV head h is the same N(0,1) pages
    divided by the pool's scale for h (kv_scales) and cast by torch to
    float8_e4m3fn (bytes kept as uint8), after clamping to +-448 -- synthetic
    bytes that both sides read as they are. New tokens stay bf16; the oracle
    and the GPU path each quantize them with their own code.
"""
from __future__ import annotations

import math
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import torch

INT32_MAX = 2**31 - 1
PAGES_PER_CHUNK = 64
_MASK64 = (1 << 64) - 1


def _splitmix64(x: int) -> int:
    x = (x + 0x9E3779B97F4A7C15) & _MASK64
    x = ((x ^ (x >> 30)) * 0xBF58476D1CE4E5B9) & _MASK64
    x = ((x ^ (x >> 27)) * 0x94D049BB133111EB) & _MASK64
    return x ^ (x >> 31)


def derived_seed(seed: int, stream: int, index: int) -> int:
    return _splitmix64(_splitmix64(_splitmix64(seed) ^ stream) ^ index) & ((1 << 63) - 1)


@dataclass
class Workload:
    """One synthetic batch. Host (CPU) tensors except where noted."""

    name: str
    seed: int
    num_heads: int
    num_kv_heads: int
    head_size: int
    block_size: int
    num_blocks: int
    softmax_scale: float
    causal: bool
    q_lens: list
    kv_lens: list
    block_table: torch.Tensor          # int32 [S, max_blocks]
    slot_mapping: torch.Tensor         # int64 [T_new]
    q: torch.Tensor                    # bf16 [T, H, D]
    k_new: torch.Tensor                # bf16 [T_new, H_kv, D]
    v_new: torch.Tensor                # bf16 [T_new, H_kv, D]
    common_prefix_len: int = 0
    meta: dict = field(default_factory=dict)
    dtype: torch.dtype = torch.bfloat16      # element type of Q, K/V pools and new tokens

    # ---- derived metadata -------------------------------------------------
    @property
    def num_seqs(self) -> int:
        return len(self.q_lens)

    @property
    def total_q(self) -> int:
        return int(sum(self.q_lens))

    @property
    def cu_seqlens_q(self) -> torch.Tensor:
        cu = [0]
        for n in self.q_lens:
            cu.append(cu[-1] + n)
        return torch.tensor(cu, dtype=torch.int32)

    @property
    def seqused_k(self) -> torch.Tensor:
        return torch.tensor(self.kv_lens, dtype=torch.int32)

    @property
    def max_seqlen_q(self) -> int:
        return max(self.q_lens) if self.q_lens else 0

    @property
    def max_seqlen_k(self) -> int:
        return max(self.kv_lens) if self.kv_lens else 0

    @property
    def page_shape(self):
        return (self.block_size, self.num_kv_heads, self.head_size)

    # ---- pool contents (prior context) ------------------------------------
    def num_chunks(self) -> int:
        return (self.num_blocks + PAGES_PER_CHUNK - 1) // PAGES_PER_CHUNK

    def pool_chunk(self, which: int, chunk: int) -> torch.Tensor:
        """Pages [chunk*64, chunk*64+64) of the K (which=0) or V (which=1) pool."""
        first = chunk * PAGES_PER_CHUNK
        n = min(PAGES_PER_CHUNK, self.num_blocks - first)
        g = torch.Generator().manual_seed(derived_seed(self.seed, 1 + which, chunk))
        x = torch.randn((n,) + self.page_shape, generator=g, dtype=torch.float32)
        return x.to(self.dtype)

    def pool(self, which: int, device="cpu", threads: int = 8) -> torch.Tensor:
        """The whole K or V pool [num_blocks, block_size, H_kv, D] before the scatter."""
        out = torch.empty((self.num_blocks,) + self.page_shape, dtype=self.dtype,
                          device=device)

        def fill(c):
            first = c * PAGES_PER_CHUNK
            chunk = self.pool_chunk(which, c)
            out[first:first + chunk.shape[0]].copy_(chunk)

        if threads > 1 and self.num_chunks() > 1:
            with ThreadPoolExecutor(threads) as ex:
                list(ex.map(fill, range(self.num_chunks())))
        else:
            for c in range(self.num_chunks()):
                fill(c)
        return out

    def pool_pages(self, which: int, pages) -> dict:
        """{page id: bf16 [bs, H_kv, D]} for the given page ids (pre-scatter contents)."""
        by_chunk = {}
        for p in sorted(set(int(p) for p in pages)):
            by_chunk.setdefault(p // PAGES_PER_CHUNK, []).append(p)
        res = {}
        for c, ps in by_chunk.items():
            chunk = self.pool_chunk(which, c)
            for p in ps:
                res[p] = chunk[p - c * PAGES_PER_CHUNK].clone()
        return res

    # ---- FP8 (e4m3) pools ----------------------------------------------------
    def kv_scales(self, which: int) -> list:
        """Per-KV-head e4m3 scales of the K (0) or V (1) pool: amax (4 + (h + which) % 4)
        of an N(0,1) head maps to the largest e4m3 value 448."""
        return [(4 + (h + which) % 4) / 448.0 for h in range(self.num_kv_heads)]

    def fp8_pool_chunk(self, which: int, chunk: int) -> torch.Tensor:
        """uint8 e4m3 pages of chunk ``chunk`` (see the module recipe)."""
        x = self.pool_chunk(which, chunk).to(torch.float32)
        s = torch.tensor(self.kv_scales(which), dtype=torch.float32)[:, None]
        return (x / s).clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)

    def fp8_pool(self, which: int, device="cpu") -> torch.Tensor:
        """The whole e4m3 K or V pool [num_blocks, block_size, H_kv, D] (uint8)."""
        out = torch.empty((self.num_blocks,) + self.page_shape, dtype=torch.uint8,
                          device=device)
        for c in range(self.num_chunks()):
            first = c * PAGES_PER_CHUNK
            chunk = self.fp8_pool_chunk(which, c)
            out[first:first + chunk.shape[0]].copy_(chunk)
        return out

    def fp8_pool_pages(self, which: int, pages) -> dict:
        """{page id: uint8 [bs, H_kv, D]} e4m3 pages (pre-scatter contents)."""
        by_chunk = {}
        for p in sorted(set(int(p) for p in pages)):
            by_chunk.setdefault(p // PAGES_PER_CHUNK, []).append(p)
        res = {}
        for c, ps in by_chunk.items():
            chunk = self.fp8_pool_chunk(which, c)
            for p in ps:
                res[p] = chunk[p - c * PAGES_PER_CHUNK].clone()
        return res

    def pages_of(self, s: int):
        nb = (self.kv_lens[s] + self.block_size - 1) // self.block_size
        return [int(x) for x in self.block_table[s, :nb]]

    def sub_batch(self, seqs) -> "Workload":
        """A batch made of the given sequences only, sharing the same pool.

        The page table rows, lengths, queries and new K/V of the chosen sequences
        are kept unchanged; the pool (num_blocks, seeds) is the same, so pages
        regenerate identically.
        """
        seqs = list(seqs)
        cu = self.cu_seqlens_q.tolist()
        q_rows = torch.cat([torch.arange(cu[s], cu[s + 1]) for s in seqs]) if seqs else \
            torch.zeros(0, dtype=torch.long)
        return Workload(
            name=f"{self.name}[sub]", seed=self.seed, num_heads=self.num_heads,
            num_kv_heads=self.num_kv_heads, head_size=self.head_size,
            block_size=self.block_size, num_blocks=self.num_blocks,
            softmax_scale=self.softmax_scale, causal=self.causal,
            q_lens=[self.q_lens[s] for s in seqs], kv_lens=[self.kv_lens[s] for s in seqs],
            block_table=self.block_table[seqs].clone(),
            slot_mapping=self.slot_mapping[q_rows].clone(),
            q=self.q[q_rows].clone(), k_new=self.k_new[q_rows].clone(),
            v_new=self.v_new[q_rows].clone(),
            common_prefix_len=self.common_prefix_len, meta=dict(self.meta), dtype=self.dtype)


def dcp_shards(wl: "Workload", ranks: int):
    """Block tables of ``ranks`` virtual context-parallel ranks: block b of a
    sequence (its b-th logical page) lives on rank b % ranks. Returns
    ([int32 [S, max_blocks]] per rank, [int32 [S] key counts] per rank); a
    rank's row lists its pages in logical order (INT32_MAX after them), so
    the sequence's partial last page, if it is the rank's, comes last."""
    S, bs = wl.num_seqs, wl.block_size
    width = max(1, (wl.block_table.shape[1] + ranks - 1) // ranks)
    tables, lens = [], []
    for r in range(ranks):
        bt = torch.full((S, width), INT32_MAX, dtype=torch.int32)
        ln = torch.zeros(S, dtype=torch.int32)
        for s in range(S):
            pages = wl.pages_of(s)
            mine = [b for b in range(len(pages)) if b % ranks == r]
            if mine:
                bt[s, :len(mine)] = torch.tensor([pages[b] for b in mine], dtype=torch.int32)
            kv = wl.kv_lens[s]
            ln[s] = sum(min(bs, kv - b * bs) for b in mine)
        tables.append(bt)
        lens.append(ln)
    return tables, lens


def _build(name, seed, H, H_kv, D, bs, q_lens, kv_lens, g, causal=True, scale=None,
           num_blocks=None, shared_prefix_pages=0, pool_slack=1.1, meta=None,
           dtype=torch.bfloat16):
    """Lay out pages, draw Q and new K/V. ``g`` has already drawn the lengths."""
    S = len(q_lens)
    assert all(0 <= q <= k for q, k in zip(q_lens, kv_lens)), "new tokens lie inside the KV"
    pages_needed = [(k + bs - 1) // bs for k in kv_lens]
    private = [max(0, p - shared_prefix_pages) for p in pages_needed]
    used = shared_prefix_pages + sum(private)
    if num_blocks is None:
        num_blocks = max(1, math.ceil(pool_slack * used))
    assert num_blocks >= used, (num_blocks, used)
    perm = torch.randperm(num_blocks, generator=g).to(torch.int32)
    max_blocks = max(pages_needed) if pages_needed else 1
    bt = torch.full((S, max(1, max_blocks)), INT32_MAX, dtype=torch.int32)
    cursor = 0
    shared = perm[:shared_prefix_pages]
    cursor = shared_prefix_pages
    for s in range(S):
        n_sh = min(shared_prefix_pages, pages_needed[s])
        bt[s, :n_sh] = shared[:n_sh]
        n_pr = private[s]
        bt[s, n_sh:n_sh + n_pr] = perm[cursor:cursor + n_pr]
        cursor += n_pr
    T = sum(q_lens)
    q = torch.randn((T, H, D), generator=g, dtype=torch.float32).to(dtype)
    k_new = torch.randn((T, H_kv, D), generator=g, dtype=torch.float32).to(dtype)
    v_new = torch.randn((T, H_kv, D), generator=g, dtype=torch.float32).to(dtype)
    slots = []
    for s in range(S):
        for pos in range(kv_lens[s] - q_lens[s], kv_lens[s]):
            slots.append(int(bt[s, pos // bs]) * bs + pos % bs)
    slot_mapping = torch.tensor(slots, dtype=torch.int64)
    return Workload(name=name, seed=seed, num_heads=H, num_kv_heads=H_kv, head_size=D,
                    block_size=bs, num_blocks=num_blocks,
                    softmax_scale=(1.0 / math.sqrt(D)) if scale is None else scale,
                    causal=causal, q_lens=list(q_lens), kv_lens=list(kv_lens),
                    block_table=bt, slot_mapping=slot_mapping, q=q, k_new=k_new,
                    v_new=v_new, common_prefix_len=shared_prefix_pages * bs,
                    meta=meta or {}, dtype=dtype)


def _uniform_int(g, lo, hi, n):
    """n integers uniform on {lo..hi} (inclusive)."""
    return [int(x) for x in torch.randint(lo, hi + 1, (n,), generator=g)]


def tiny_mixed(seed=1001, dtype=torch.bfloat16):
    """4 seqs, 4 query / 2 KV heads, head_size 64, block_size 16, pool of 64 pages.
    KV lens {17, 33, 64, 100}; seqs 0-1 decode (one query), seqs 2-3 causal
    prefill with query length equal to KV length."""
    g = torch.Generator().manual_seed(seed)
    kv = [17, 33, 64, 100]
    ql = [1, 1, 64, 100]
    return _build("tiny_mixed", seed, 4, 2, 64, 16, ql, kv, g, num_blocks=64,
                  scale=1.0 / 8.0, dtype=dtype)


def decode_llama8b(seed=1002, num_seqs=64, dtype=torch.bfloat16):
    """64 decode seqs x 1 query token, 32/8 heads, head_size 128, block_size 16,
    KV lens uniform on [512, 8192], pool = total pages + 10%."""
    g = torch.Generator().manual_seed(seed)
    kv = _uniform_int(g, 512, 8192, num_seqs)
    return _build("decode_llama8b", seed, 32, 8, 128, 16, [1] * num_seqs, kv, g, dtype=dtype)


def chunked_prefill_mix(seed=1003, n_prefill=8, chunk=2048, n_decode=56, dtype=torch.bfloat16):
    """8 causal prefill chunks of 2048 tokens with prior context uniform on
    [0, 4096], then 56 decode seqs with KV uniform on [1024, 8192]; 32/8 heads,
    head_size 128, block_size 16."""
    g = torch.Generator().manual_seed(seed)
    ctx = _uniform_int(g, 0, 4096, n_prefill)
    dec = _uniform_int(g, 1024, 8192, n_decode)
    ql = [chunk] * n_prefill + [1] * n_decode
    kv = [c + chunk for c in ctx] + dec
    return _build("chunked_prefill_mix", seed, 32, 8, 128, 16, ql, kv, g, dtype=dtype)


def cascade_shared_prefix(seed=1004, num_seqs=64, prefix=2048, dtype=torch.bfloat16):
    """64 requests sharing a 2048-token prefix (128 pages of 16, the same first
    128 block_table entries in every row), each with one query token and a
    private suffix uniform on [64, 512] tokens; 32/8 heads, head_size 128."""
    g = torch.Generator().manual_seed(seed)
    suf = _uniform_int(g, 64, 512, num_seqs)
    kv = [prefix + s for s in suf]
    return _build("cascade_shared_prefix", seed, 32, 8, 128, 16, [1] * num_seqs, kv, g,
                  shared_prefix_pages=prefix // 16, dtype=dtype)


def long_context_70b(seed=1005, n_decode=32, kv_len=32768, n_prefill=4, q_len=4096, dtype=torch.bfloat16):
    """64/8 heads (GQA 8), head_size 128, block_size 128: 32 decode seqs at KV
    32768, then 4 causal prefill seqs of 4096 tokens on 28672 prior tokens."""
    g = torch.Generator().manual_seed(seed)
    ql = [1] * n_decode + [q_len] * n_prefill
    kv = [kv_len] * (n_decode + n_prefill)
    return _build("long_context_70b", seed, 64, 8, 128, 128, ql, kv, g, dtype=dtype)


def long_context_70b_prefill(seed=1015, n_prefill=4, kv_len=32768, q_len=4096, dtype=torch.bfloat16):
    """The prefill side of long_context_70b as a batch of its own: 4 causal
    prefill seqs of 4096 queries on 28672 prior tokens, 64/8 heads, head_size
    128, block_size 128 (the same shapes and FLOPs; its own pool of those
    sequences' pages only, ~0.3 GB per pool)."""
    g = torch.Generator().manual_seed(seed)
    return _build("long_context_70b_prefill", seed, 64, 8, 128, 128, [q_len] * n_prefill,
                  [kv_len] * n_prefill, g, dtype=dtype)


def chunked_prefill_mix_prefill(seed=1003, n_prefill=8, chunk=2048, n_decode=56, dtype=torch.bfloat16):
    """The prefill chunks of chunked_prefill_mix as a batch of their own: the
    same 8 chunks of 2048 causal queries with the same prior-context lengths
    (drawn first from the same seed), 32/8 heads, head_size 128, block_size
    16; a pool of those sequences' pages only."""
    g = torch.Generator().manual_seed(seed)
    ctx = _uniform_int(g, 0, 4096, n_prefill)
    _uniform_int(g, 1024, 8192, n_decode)      # the decode lengths, drawn and dropped
    return _build("chunked_prefill_mix_prefill", seed, 32, 8, 128, 16, [chunk] * n_prefill,
                  [c + chunk for c in ctx], g, dtype=dtype)


def prefill_profile(seed=1006, n_prefill=4, q_len=2048, kv_len=12288, dtype=torch.bfloat16):
    """A small case of the long-context prefill shape for profiler captures:
    64/8 heads, head_size 128, block_size 128, 4 causal prefill sequences of
    2048 queries on 10240 prior tokens (pool ~220 MB, larger than L2)."""
    g = torch.Generator().manual_seed(seed)
    return _build("prefill_profile", seed, 64, 8, 128, 128, [q_len] * n_prefill,
                  [kv_len] * n_prefill, g, dtype=dtype)


def decode_d256(seed=1007, num_seqs=64, dtype=torch.bfloat16):
    """A decode batch at head size 256 (Gemma-2-like heads): 64 sequences x 1
    query, 16/8 heads, block_size 16, KV lengths uniform on [512, 4096]
    (about 1.2 GB of K/V, as the head-size-128 decode batch)."""
    g = torch.Generator().manual_seed(seed)
    kv = _uniform_int(g, 512, 4096, num_seqs)
    return _build("decode_d256", seed, 16, 8, 256, 16, [1] * num_seqs, kv, g, dtype=dtype)


def prefill_d256(seed=1008, n_prefill=4, q_len=2048, kv_len=10240, dtype=torch.bfloat16):
    """A prefill batch at head size 256: 4 causal sequences of 2048 queries on
    8192 prior tokens, 16/8 heads, block_size 16."""
    g = torch.Generator().manual_seed(seed)
    return _build("prefill_d256", seed, 16, 8, 256, 16, [q_len] * n_prefill,
                  [kv_len] * n_prefill, g, dtype=dtype)


CONFIGS = {
    "tiny_mixed": tiny_mixed,
    "decode_llama8b": decode_llama8b,
    "chunked_prefill_mix": chunked_prefill_mix,
    "cascade_shared_prefix": cascade_shared_prefix,
    "long_context_70b": long_context_70b,
    "prefill_profile": prefill_profile,
    "long_context_70b_prefill": long_context_70b_prefill,
    "chunked_prefill_mix_prefill": chunked_prefill_mix_prefill,
    "decode_d256": decode_d256,
    "prefill_d256": prefill_d256,
}


def random_case(seed, num_seqs=3, num_heads=4, num_kv_heads=2, head_size=64,
                block_size=16, max_q=40, max_kv=120, causal=True, decode_frac=0.3,
                empty_ok=False, slack=1.5, dtype=torch.bfloat16):
    """A small random batch: lengths, pages and values all from ``seed``."""
    g = torch.Generator().manual_seed(seed)
    ql, kv = [], []
    for _ in range(num_seqs):
        lo = 0 if empty_ok else 1
        k = int(torch.randint(lo, max_kv + 1, (1,), generator=g))
        if float(torch.rand((1,), generator=g)) < decode_frac:
            q = min(1, k) if not empty_ok else int(torch.randint(0, 2, (1,), generator=g))
        else:
            q = int(torch.randint(lo, max_q + 1, (1,), generator=g))
        q = min(q, k)
        ql.append(q)
        kv.append(k)
    return _build(f"random_{seed}", seed, num_heads, num_kv_heads, head_size, block_size,
                  ql, kv, g, causal=causal, pool_slack=slack, dtype=dtype)
