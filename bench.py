"""Benchmark of the paged varlen attention hot path on GB300.

One step = the whole hot path over one synthetic batch: the slot_mapping
scatter of the batch's new K/V tokens into the page pool, the device-side
work plan, the paged attention (split-KV decode kernel; tensor-core prefill
kernel for long queries) and the split combine.

Default workload: the Llama-3-8B-shaped decode batch (64 sequences x 1 query,
32/8 heads, head_size 128, block_size 16, KV lengths uniform on [512, 8192],
pages randomly permuted). Metric: algorithmic HBM bytes per step / step time
(GB/s). Algorithmic bytes count each visible K/V byte once per step plus Q, O,
LSE, the block-table rows read and the scatter's read+write of the new tokens;
workspace (split partial) traffic is not counted.

With --kv-cache fp8 the page pools hold e4m3 bytes with per-KV-head scales
(the FP8 KV cache of the FlashAttention/FlashInfer backend page): each K/V
byte of the pool counts once, the scatter reads bf16 rows and writes bytes.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                       [--workload NAME] [--kv-cache bf16|fp8]
Under torchrun (N > 1) every rank runs its own replica of the workload (weak
scaling, no collective on the data path); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

import workloads as W  # noqa: E402

METRIC = "paged-attn decode HBM GB/s + prefill TFLOPS on 1 GB300, % of roofline"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
FALLBACK_BF16_SUSTAINED = 1700.0
L2_BYTES = 129 * 1024 * 1024
_CSRC = os.path.join(ROOT, "paged_kv_varlen_attn_gb300", "csrc")
# Sources the split kernel's code comes from; the recorded DRAM traffic is
# valid only while all of them are unchanged.
SPLIT_KERNEL_SRCS = [os.path.join(_CSRC, f) for f in
                     ("attn_split.cu", "device_common.cuh", "epilogue.cuh", "pa_internal.h")]
TC_KERNEL_SRCS = [os.path.join(_CSRC, f) for f in
                  ("attn_tc.cu", "device_common.cuh", "epilogue.cuh", "pa_internal.h")]
KERNEL_SRCS = {"attn_split_kernel<128>": SPLIT_KERNEL_SRCS,
               "attn_split_kernel<128, fp8>": SPLIT_KERNEL_SRCS,
               "attn_tc_kernel<128>": TC_KERNEL_SRCS,
               "attn_tc_kernel<128, fp8>": TC_KERNEL_SRCS}
# The prefill half of the metric: tensor-core prefill sub-launches timed in
# the default run beside the decode step (workload name -> what it is).
PREFILL_LEGS = {
    "long_context_70b_prefill": "long_context_70b's prefill: 4 causal seqs x 4096 queries on "
                                "28,672 prior keys, 64/8 heads, D 128, block 128",
    "chunked_prefill_mix_prefill": "chunked_prefill_mix's prefill chunks: 8 causal seqs x 2048 "
                                   "queries on prior context U[0, 4096], 32/8 heads, D 128, "
                                   "block 16",
}
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")


# ---------------------------------------------------------------------------
def is_prefill(wl, s, fp8=False):
    """Segments with more than 32 packed query rows run on the tensor-core
    kernel (for FP8 pools too; at head size 256 every segment does)."""
    return wl.q_lens[s] * (wl.num_heads // wl.num_kv_heads) > 32


def algorithmic_counts(wl: W.Workload, seqs=None, cascade=False, fp8=False):
    """Bytes and FLOPs of one step by the counting rule in the module docstring.

    Each visible K/V byte counts once per step (for cascade, the shared prefix
    counts once for the whole batch), plus Q, O, LSE and the block-table rows;
    FLOPs are 4 * D * H per visible (query, key) pair.
    """
    H, Hk, D = wl.num_heads, wl.num_kv_heads, wl.head_size
    seqs = range(wl.num_seqs) if seqs is None else seqs
    kv_bytes = {"decode": 0, "prefill": 0}
    flops = {"decode": 0, "prefill": 0}
    T = 0
    bt = 0
    kv_elem = 1 if fp8 else 2
    per_key = Hk * D * 2 * kv_elem
    for s in seqs:
        ql, kl = wl.q_lens[s], wl.kv_lens[s]
        kind = "prefill" if is_prefill(wl, s) else "decode"
        keys = kl - wl.common_prefix_len if cascade else kl
        kv_bytes[kind] += keys * per_key
        if wl.causal:
            pairs = ql * (kl - ql) + ql * (ql + 1) // 2
        else:
            pairs = ql * kl
        flops[kind] += 4 * D * H * pairs
        T += ql
        bt += (kl + wl.block_size - 1) // wl.block_size * 4
    if cascade:
        kv_bytes["decode"] += wl.common_prefix_len * per_key
    qo = 2 * T * H * D * 2
    lse = H * T * 4
    scatter = 2 * T * Hk * D * (2 + kv_elem)   # read bf16 K and V rows, write the pool's
    attn_bytes = kv_bytes["decode"] + kv_bytes["prefill"] + qo + lse + bt
    return {"attn_bytes": attn_bytes, "scatter_bytes": scatter,
            "step_bytes": attn_bytes + scatter, "flops": flops["decode"] + flops["prefill"],
            "kv_bytes": kv_bytes, "flops_by_kind": flops, "qo_lse_bt": qo + lse + bt}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        hbm = p.get("hbm_gbs") or p.get("hbm_GBs")
        bf16 = p.get("bf16_tflops")
        sus = p.get("bf16_tflops_sustained")
        return {"hbm_gbs": float(hbm) if hbm else FALLBACK_HBM_GBS,
                "bf16_tflops": float(bf16) if bf16 else FALLBACK_BF16_TFLOPS,
                "bf16_tflops_sustained": float(sus) if sus else FALLBACK_BF16_SUSTAINED,
                "source": "measured" if hbm else "fallback"}
    return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": FALLBACK_BF16_TFLOPS,
            "bf16_tflops_sustained": FALLBACK_BF16_SUSTAINED, "source": "fallback"}


def sources_sha(paths):
    h = hashlib.sha256()
    for p in paths:
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def load_traffic(kernel, workload):
    """Per-launch DRAM bytes of `kernel` from a committed ncu summary, or None
    when the kernel source changed since the counters were taken."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    with open(TRAFFIC_FILE) as f:
        t = json.load(f)
    e = t.get(kernel, {}).get(workload)
    if not e or e.get("source_sha") != sources_sha(KERNEL_SRCS[kernel]):
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            threading.Thread(target=self._read, daemon=True).start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.05)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 6:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[2:6]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


def hold(step, batch, seconds):
    """Replay `step` on `batch` (untimed) for about `seconds` of wall time."""
    import torch
    t0 = time.time()
    while time.time() - t0 < seconds:
        for _ in range(16):
            step(batch)
        torch.cuda.synchronize()


# ---------------------------------------------------------------------------
def dist_setup(n_gpus):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world, device):
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def run_oracle_sample(wl, max_seconds=12.0, max_seqs=None, fp8=False):
    """Returns (algorithmic bytes covered, flops covered, seconds, description)."""
    import oracle
    torch.set_num_threads(os.cpu_count() or 1)
    cu = wl.cu_seqlens_q.tolist()
    covered_bytes, covered_flops, secs, n = 0, 0, 0.0, 0
    Hk, D, H = wl.num_kv_heads, wl.head_size, wl.num_heads
    order = list(range(wl.num_seqs))
    for s in order:
        if secs >= max_seconds or (max_seqs is not None and n >= max_seqs):
            break
        sub = wl.sub_batch([s])
        pages = sub.pages_of(0)
        if fp8:
            kp, vp = sub.fp8_pool_pages(0, pages), sub.fp8_pool_pages(1, pages)
        else:
            kp, vp = sub.pool_pages(0, pages), sub.pool_pages(1, pages)
        kc = torch.stack([kp[p] for p in pages])
        vc = torch.stack([vp[p] for p in pages])
        bt = torch.arange(len(pages), dtype=torch.int32)[None]
        bs = wl.block_size
        remap = {p: i for i, p in enumerate(pages)}
        slots = torch.tensor([remap[int(x) // bs] * bs + int(x) % bs for x in sub.slot_mapping],
                             dtype=torch.int64)
        ql, kl = sub.q_lens[0], sub.kv_lens[0]
        rows = None
        if ql > 64:
            g = torch.Generator().manual_seed(s)
            rows = {0: sorted(set(int(x) for x in torch.randint(0, ql, (64,), generator=g)))}
        t0 = time.perf_counter()
        if fp8:
            ks, vs = wl.kv_scales(0), wl.kv_scales(1)
            oracle.reshape_and_cache_e4m3(sub.k_new, sub.v_new, slots, kc, vc, ks, vs)
            oracle.varlen_attention_e4m3(sub.q, kc, vc, sub.cu_seqlens_q, sub.seqused_k, bt,
                                         wl.softmax_scale, wl.causal, ks, vs, rows=rows)
        else:
            oracle.reshape_and_cache(sub.k_new, sub.v_new, slots, kc, vc)
            oracle.varlen_attention(sub.q, kc, vc, sub.cu_seqlens_q, sub.seqused_k, bt,
                                    wl.softmax_scale, wl.causal, rows=rows)
        secs += time.perf_counter() - t0
        nrows = ql if rows is None else len(rows[0])
        e = 1 if fp8 else 2
        covered_bytes += kl * Hk * D * 2 * e + 2 * ql * H * D * 2 + H * ql * 4 + 2 * ql * Hk * D * (2 + e)
        covered_flops += 4 * D * H * nrows * kl
        n += 1
    desc = f"{n} of {wl.num_seqs} sequences of {wl.name}{' (e4m3 KV)' if fp8 else ''} " \
           f"(all query rows of decode sequences, 64 seeded rows of longer ones), " \
           f"scatter + attention, fp64 torch CPU"
    return covered_bytes, covered_flops, secs, desc


# ---------------------------------------------------------------------------
def bench_reference(args, rank, world):
    if rank != 0:
        return
    wl = W.CONFIGS[args.workload](dtype=DTYPES[args.dtype])
    times = []
    total_bytes = 0
    desc = ""
    for i in range(args.warmup + args.steps):
        b, f, s, desc = run_oracle_sample(wl, max_seconds=3.0, max_seqs=4,
                                          fp8=args.kv_cache == "fp8")
        if i >= args.warmup:
            times.append(s)
            total_bytes += b
    secs = sum(times)
    value = total_bytes / secs / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * secs / max(1, args.steps), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": wl.name + ("+fp8_kv" if args.kv_cache == "fp8" else ""),
                       "sample": desc},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": torch.get_num_threads(),
                             "kind": "oracle", "sample": desc},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def l2_flush(wbuf, rbuf, i):
    """Flush L2 before a timed launch: write a 256 MB buffer (twice the L2),
    then read another 256 MB so that the flush's own dirty lines are written
    back before the timed region starts rather than inside it."""
    wbuf.fill_(i & 0xff)
    torch.amax(rbuf.view(torch.int32))


def timed_flushed(fn, n, flush, stream, flush_rd):
    """Mean device time (ms) of fn over n launches, L2 flushed before each."""
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(n)]
    for i in range(n):
        l2_flush(flush, flush_rd, i)
        evs[i][0].record(stream)
        fn()
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    return sum(a.elapsed_time(b) for a, b in evs) / n


DTYPES = {"bf16": torch.bfloat16, "fp16": torch.float16}


def prefill_record(pa, name, dev, peaks, steps, min_ms=600.0, dtype=torch.bfloat16, fp8=False):
    """The prefill half of the metric on one prefill-only batch: the attention
    call (planner + tensor-core prefill kernel) timed launch by launch with
    CUDA events on the launching stream, SM clocks sampled over the window.
    FLOPs are 4 * D * H per visible (query, key) pair; the fraction is taken
    against the sustained bf16 peak (the launches run back to back for
    longer than a second), the burst fraction is given beside it. With fp8
    the pools hold e4m3 bytes (the kernel widens them to f16 and multiplies
    at the 16-bit rate, so the same peak applies)."""
    wl = W.CONFIGS[name](dtype=dtype)
    T, H, D = wl.q.shape
    counts = algorithmic_counts(wl, fp8=fp8)
    b = DeviceBatch(wl, dev)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    if fp8:
        kc, vc = wl.fp8_pool(0, dev), wl.fp8_pool(1, dev)
        ksc = torch.tensor(wl.kv_scales(0), device=dev)
        vsc = torch.tensor(wl.kv_scales(1), device=dev)
        pa.reshape_and_cache_fp8(b.d["k_new"], b.d["v_new"], kc, vc, b.d["slot_mapping"], ksc, vsc)
        size_fn = pa.varlen_fwd_fp8kv_workspace_size
    else:
        kc, vc = wl.pool(0, device=dev), wl.pool(1, device=dev)
        pa.reshape_and_cache(b.d["k_new"], b.d["v_new"], kc, vc, b.d["slot_mapping"])
        size_fn = pa.varlen_fwd_workspace_size
    ws = pa.alloc_workspace(size_fn(wl.num_seqs, T, wl.max_seqlen_q, wl.max_seqlen_k, H,
                                    wl.num_kv_heads, D, wl.block_size, sms), dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    # Inputs read per launch (Q, K/V pages) vs L2: flush before each launch
    # when they would fit.
    in_bytes = counts["kv_bytes"]["prefill"] + T * H * D * 2
    flush = flush_rd = None
    if in_bytes < 2 * L2_BYTES:
        flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
        flush_rd = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)

    def attn():
        if fp8:
            pa.varlen_fwd_fp8kv(b.d["q"], kc, vc, b.d["cu_seqlens_q"], b.d["seqused_k"],
                                b.d["block_table"], wl.max_seqlen_q, wl.max_seqlen_k,
                                wl.softmax_scale, wl.causal, ksc, vsc, out=b.out, lse=b.lse,
                                workspace=ws, dev_status=status)
        else:
            pa.varlen_fwd(b.d["q"], kc, vc, b.d["cu_seqlens_q"], b.d["seqused_k"],
                          b.d["block_table"], wl.max_seqlen_q, wl.max_seqlen_k, wl.softmax_scale,
                          wl.causal, out=b.out, lse=b.lse, workspace=ws, dev_status=status)
    for _ in range(3):
        attn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    attn()
    e1.record(stream)
    torch.cuda.synchronize()
    est = e0.elapsed_time(e1)
    n = int(min(100, max(5, min(steps, 50), min_ms / max(est, 1e-3))))
    sampler = ClockSampler(dev.index or 0)
    sampler.start()
    hold(lambda _b: attn(), None, 0.3)   # the clock record under this launch's load
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(n)]
    for i in range(n):
        if flush is not None:
            l2_flush(flush, flush_rd, i)
        ev[i][0].record(stream)
        attn()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    assert int(status.item()) == 0, f"device status bits {int(status.item())}"
    ms = sum(a.elapsed_time(c) for a, c in ev) / n
    tflops = counts["flops"] / (ms * 1e-3) / 1e12
    rec = {"workload": name + ("+fp8_kv" if fp8 else ""), "what": PREFILL_LEGS.get(name, name),
           "dtype": str(dtype)[6:] + (", e4m3 kv widened to f16" if fp8 else ""),
           "kernel": "plan + attn_tc_kernel<128%s>" % (", fp8" if fp8 else ""), "bound": "tensor",
           "flops_per_launch": counts["flops"], "ms_per_launch": ms, "launches": n,
           "tflops": tflops, "unit": "TFLOP/s",
           "peak": peaks["bf16_tflops_sustained"], "peak_kind": "bf16 sustained",
           "frac": tflops / peaks["bf16_tflops_sustained"],
           "frac_burst": tflops / peaks["bf16_tflops"],
           "traffic": load_traffic("attn_tc_kernel<128%s>" % (", fp8" if fp8 else ""),
                                   name + ("+fp8_kv" if fp8 else "")),
           "algorithmic_bytes_per_launch": counts["attn_bytes"],
           "l2": "flushed before every launch" if flush is not None else
                 "inputs larger than L2 (%.2f GB of Q and K/V per launch)" % (in_bytes / 1e9),
           "timing": "CUDA events per launch on the launching stream, after 3 warm-up launches",
           "clocks": clocks, "peak_source": peaks["source"]}
    del kc, vc, b, ws
    torch.cuda.empty_cache()
    return rec


def row_figures(pa, wl, counts, dev, stream, scatter_fn, steps):
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    flush_rd = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    n = max(5, min(50, steps))
    T, H, D = wl.q.shape
    Tn = wl.k_new.shape[0]
    out = {}
    for _ in range(3):
        scatter_fn()
    ms = timed_flushed(scatter_fn, n, flush, stream, flush_rd)
    b = counts["scatter_bytes"] + Tn * 8
    out["reshape_and_cache"] = {"tokens": Tn, "bytes": b, "ms": ms, "gbs": b / (ms * 1e-3) / 1e9}
    g = torch.Generator(device="cpu").manual_seed(7)
    for name, tm in (("merge_attn_states", T), ("merge_attn_states_16k_tokens", 16384)):
        oa = torch.randn((tm, H, D), generator=g).to(torch.bfloat16).to(dev)
        ob = torch.randn((tm, H, D), generator=g).to(torch.bfloat16).to(dev)
        la = (torch.randn((H, tm), generator=g) * 3).to(dev)
        lb = (torch.randn((H, tm), generator=g) * 3).to(dev)
        o = torch.empty_like(oa)
        lo = torch.empty_like(la)

        def merge():
            pa.merge_attn_states(oa, la, ob, lb, out=o, out_lse=lo)
        for _ in range(3):
            merge()
        ms = timed_flushed(merge, n, flush, stream, flush_rd)
        b = 3 * tm * H * D * 2 + 3 * H * tm * 4
        out[name] = {"tokens": tm, "bytes": b, "ms": ms, "gbs": b / (ms * 1e-3) / 1e9}
    # The n-state merge of decode context parallelism: 4 virtual ranks'
    # partial states of a 16,384-token batch.
    nr, tm = 4, 16384
    po = torch.randn((nr, tm, H, D), generator=g).to(torch.bfloat16).to(dev)
    pl = (torch.randn((nr, H, tm), generator=g) * 3).to(dev)
    o = torch.empty((tm, H, D), dtype=torch.bfloat16, device=dev)
    lo = torch.empty((H, tm), dtype=torch.float32, device=dev)

    def merge_n():
        pa.merge_attn_states_n(po, pl, out=o, out_lse=lo)
    for _ in range(3):
        merge_n()
    ms = timed_flushed(merge_n, n, flush, stream, flush_rd)
    b = (nr + 1) * tm * H * D * 2 + (nr + 1) * H * tm * 4
    out["merge_attn_states_n_4parts_16k_tokens"] = {"tokens": tm, "parts": nr, "bytes": b,
                                                    "ms": ms, "gbs": b / (ms * 1e-3) / 1e9}
    return out


class DeviceBatch:
    """Device copies of one batch's per-step inputs, plus its outputs."""

    def __init__(self, wl, dev):
        self.wl = wl
        self.host = {
            "q": wl.q.pin_memory(), "k_new": wl.k_new.pin_memory(),
            "v_new": wl.v_new.pin_memory(), "slot_mapping": wl.slot_mapping.pin_memory(),
            "cu_seqlens_q": wl.cu_seqlens_q.pin_memory(),
            "seqused_k": wl.seqused_k.pin_memory(), "block_table": wl.block_table.pin_memory(),
        }
        self.d = {k: v.to(dev) for k, v in self.host.items()}
        T, H, D = wl.q.shape
        self.out = torch.empty((T, H, D), dtype=wl.q.dtype, device=dev)
        self.lse = torch.empty((H, T), dtype=torch.float32, device=dev)
        self.out_h = torch.empty_like(self.out, device="cpu").pin_memory()
        self.lse_h = torch.empty_like(self.lse, device="cpu").pin_memory()


def bench_ours(args, rank, world, local):
    import paged_kv_varlen_attn_gb300 as pa
    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA GPU (no CPU fallback)")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if rank == 0:
        from paged_kv_varlen_attn_gb300 import _build
        _build.build()
    barrier(world)
    pa.load_library()

    wl = W.CONFIGS[args.workload](dtype=DTYPES[args.dtype])
    cascade = wl.common_prefix_len > 0
    fp8 = args.kv_cache == "fp8"
    counts = algorithmic_counts(wl, cascade=cascade, fp8=fp8)
    if fp8:
        kc0, vc0 = wl.fp8_pool(0, device=dev), wl.fp8_pool(1, device=dev)
        ksc = torch.tensor(wl.kv_scales(0), dtype=torch.float32, device=dev)
        vsc = torch.tensor(wl.kv_scales(1), dtype=torch.float32, device=dev)
    else:
        kc0 = wl.pool(0, device=dev)
        vc0 = wl.pool(1, device=dev)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    T, H, D = wl.q.shape
    if fp8:
        size_fn = pa.cascade_fwd_fp8kv_workspace_size if cascade else \
            pa.varlen_fwd_fp8kv_workspace_size
    else:
        size_fn = pa.cascade_fwd_workspace_size if cascade else pa.varlen_fwd_workspace_size
    ws = pa.alloc_workspace(size_fn(wl.num_seqs, T, wl.max_seqlen_q, wl.max_seqlen_k, H,
                                    wl.num_kv_heads, D, wl.block_size, sms), dev)
    main = DeviceBatch(wl, dev)

    def attention(b, dd=None):
        dd = dd or b.d
        w = b.wl
        args_ = (dd["q"], kc0, vc0, dd["cu_seqlens_q"], dd["seqused_k"], dd["block_table"],
                 w.max_seqlen_q, w.max_seqlen_k, w.softmax_scale)
        if fp8 and cascade:
            pa.cascade_fwd_fp8kv(*args_, w.common_prefix_len, ksc, vsc, out=b.out, lse=b.lse,
                                 workspace=ws, dev_status=status)
        elif fp8:
            pa.varlen_fwd_fp8kv(*args_, w.causal, ksc, vsc, out=b.out, lse=b.lse, workspace=ws,
                                dev_status=status)
        elif cascade:
            pa.cascade_fwd(*args_, w.common_prefix_len, out=b.out, lse=b.lse, workspace=ws,
                           dev_status=status)
        else:
            pa.varlen_fwd(*args_, w.causal, out=b.out, lse=b.lse, workspace=ws,
                          dev_status=status)

    def scatter(b, dd=None):
        dd = dd or b.d
        if fp8:
            pa.reshape_and_cache_fp8(dd["k_new"], dd["v_new"], kc0, vc0, dd["slot_mapping"], ksc,
                                     vsc, dev_status=status)
        else:
            pa.reshape_and_cache(dd["k_new"], dd["v_new"], kc0, vc0, dd["slot_mapping"],
                                 dev_status=status)

    def fused(b, dd=None):
        # One serving step through the public API: the step's new K/V are
        # scattered into the cache and attended in one call (the planner
        # overlaps the scatter).
        dd = dd or b.d
        w = b.wl
        if fp8:
            args_ = (dd["q"], kc0, vc0, dd["cu_seqlens_q"], dd["seqused_k"], dd["block_table"],
                     w.max_seqlen_q, w.max_seqlen_k, w.softmax_scale)
            upd = dict(key=dd["k_new"], value=dd["v_new"], slot_mapping=dd["slot_mapping"],
                       out=b.out, lse=b.lse, workspace=ws, dev_status=status)
            if cascade:
                pa.cascade_fwd_fp8kv(*args_, w.common_prefix_len, ksc, vsc, **upd)
            else:
                pa.varlen_fwd_fp8kv(*args_, w.causal, ksc, vsc, **upd)
            return
        args_ = (dd["k_new"], dd["v_new"], dd["slot_mapping"], dd["q"], kc0, vc0,
                 dd["cu_seqlens_q"], dd["seqused_k"], dd["block_table"], w.max_seqlen_q,
                 w.max_seqlen_k, w.softmax_scale)
        if cascade:
            pa.cascade_fwd_with_update(*args_, w.common_prefix_len, out=b.out, lse=b.lse,
                                       workspace=ws, dev_status=status)
        else:
            pa.varlen_fwd_with_update(*args_, w.causal, out=b.out, lse=b.lse, workspace=ws,
                                      dev_status=status)

    def step(b, dd=None):
        fused(b, dd)

    for _ in range(max(3, args.warmup)):
        step(main)
        attention(main)
    torch.cuda.synchronize()

    graphs = None
    if not args.no_graph:
        # Every C-ABI call is asynchronous, allocation-free and sync-free, so a
        # step is recorded once as a CUDA graph and replayed, as a serving
        # engine replays its decode step. A second graph holds the attention
        # call alone, replayed after the timed steps to time the dominant
        # launch for the roofline.
        g_step, g_at = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_step):
            fused(main)
        with torch.cuda.graph(g_at):
            attention(main)
        torch.cuda.synchronize()
        graphs = (g_step, g_at)

        def step(b, dd=None):  # noqa: F811
            if dd is not None:
                for k, v in dd.items():
                    b.d[k].copy_(v, non_blocking=True)
            g_step.replay()

        for _ in range(3):
            step(main)
        torch.cuda.synchronize()
        stream = torch.cuda.current_stream(dev)

    def attention_only():
        if graphs is not None:
            graphs[1].replay()
        else:
            attention(main)

    # ---- device-resident timing -------------------------------------------
    # The K/V pages read per step exceed the 129 MB L2 for the decode and
    # mixed workloads, so no flush is needed between steps; the cascade
    # workload flushes L2 (a 256 MB write) before every step, outside the
    # per-step attention events.
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev) if cascade else None
    flush_rd = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev) if cascade else None
    sampler = ClockSampler(local)
    sampler.start()
    # The timed region lasts a few milliseconds, shorter than the sampling
    # period, so the GPU is held at this workload's load (untimed replays of
    # the step) for ~0.4 s before it and ~0.2 s after it: the clock record is
    # then the clocks this workload runs at, not those of an idle GPU.
    hold(step, main, 0.4)
    barrier(world)
    torch.cuda.synchronize()
    t_begin = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    step_ms = 0.0
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    if flush is None:
        t_begin.record(stream)
        for i in range(args.steps):
            step(main)
        t_end.record(stream)
        torch.cuda.synchronize()
        step_ms = t_begin.elapsed_time(t_end)
        # The dominant launch alone (attention on the same inputs, whose K/V
        # reads exceed L2), back to back, each launch between its own events.
        for i in range(args.steps):
            ev[i][0].record(stream)
            attention_only()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
    else:
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        for i in range(args.steps):
            l2_flush(flush, flush_rd, i)
            starts[i].record(stream)
            step(main)
            ends[i].record(stream)
        torch.cuda.synchronize()
        step_ms = sum(a.elapsed_time(b) for a, b in zip(starts, ends))
        for i in range(args.steps):
            l2_flush(flush, flush_rd, i)
            ev[i][0].record(stream)
            attention_only()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
    hold(step, main, 0.2)
    barrier(world)
    clocks = sampler.stop()
    attn_ms = sum(x.elapsed_time(y) for x, y in ev)
    total_ms = max_over_ranks(step_ms, world, dev)
    ms_per_step = total_ms / args.steps
    value = world * counts["step_bytes"] / (ms_per_step * 1e-3) / 1e9

    # ---- end-to-end through the API with host buffers ------------------------
    h2d = sum(t.numel() * t.element_size() for t in main.host.values())
    d2h = main.out_h.numel() * main.out_h.element_size() + \
        main.lse_h.numel() * main.lse_h.element_size()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(args.steps):
        if graphs is None:
            dd = {k: v.to(dev, non_blocking=True) for k, v in main.host.items()}
        else:
            dd = main.host   # copied into the graph's input buffers inside step()
        step(main, dd)
        main.out_h.copy_(main.out, non_blocking=True)
        main.lse_h.copy_(main.lse, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, dev) / args.steps
    e2e_value = world * counts["step_bytes"] / (e2e_ms * 1e-3) / 1e9

    # ---- sub-launches of a mixed batch: decode-only and prefill-only ----------
    sub = {}
    kinds = {"prefill": [s for s in range(wl.num_seqs) if is_prefill(wl, s)],
             "decode": [s for s in range(wl.num_seqs) if not is_prefill(wl, s)]}
    if not cascade and kinds["prefill"] and kinds["decode"]:
        for kind, seqs in kinds.items():
            b = DeviceBatch(wl.sub_batch(seqs), dev)
            c = algorithmic_counts(wl, seqs, fp8=fp8)
            for _ in range(3):
                attention(b)
            torch.cuda.synchronize()
            x0 = torch.cuda.Event(enable_timing=True)
            x1 = torch.cuda.Event(enable_timing=True)
            n = max(3, args.steps // 2)
            x0.record(stream)
            for _ in range(n):
                attention(b)
            x1.record(stream)
            torch.cuda.synchronize()
            ms = x0.elapsed_time(x1) / n
            sub[kind] = {"ms": ms, "gbs": c["attn_bytes"] / (ms * 1e-3) / 1e9,
                         "tflops": c["flops"] / (ms * 1e-3) / 1e12, "seqs": len(seqs)}
    # ---- per-step figures of the standalone steps --------------------------
    # The scatter of this step's new tokens (launched alone) and
    # pa_merge_attn_states on partial states of this batch's shape and of a
    # 16,384-token batch, each launch timed alone after an L2 flush.
    rows_fig = row_figures(pa, wl, counts, dev, stream, lambda: scatter(main), args.steps)
    assert int(status.item()) == 0, f"device status bits {int(status.item())}"
    # ---- the prefill half of the metric (same pool format) -------------------
    peaks = load_peaks()
    prefill = {}
    if not args.no_prefill:
        for name in PREFILL_LEGS:
            prefill[name] = prefill_record(pa, name, dev, peaks, args.steps,
                                           dtype=DTYPES[args.dtype], fp8=fp8)

    if rank != 0:
        return
    attn_ms_avg = attn_ms / args.steps
    config = {"workload": wl.name + ("+fp8_kv" if fp8 else ""), "num_seqs": wl.num_seqs,
              "num_heads": H,
              "num_kv_heads": wl.num_kv_heads, "head_size": D, "block_size": wl.block_size,
              "kv_tokens": int(sum(wl.kv_lens)), "query_tokens": T,
              "step_bytes": counts["step_bytes"], "step_flops": counts["flops"],
              "l2": ("L2 flushed before every step (256 MB write, then 256 MB read so the "
                     "flush's dirty lines are written back outside the timed region)" if cascade else
                     "inputs larger than L2: %.2f GB of K/V pages read per step vs 129 MB L2"
                     % (counts["attn_bytes"] / 1e9)),
              "parallelism": f"replicas x{world}"}
    if cascade:
        config["common_prefix_len"] = wl.common_prefix_len
    line = {"metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": ("e4m3 kv (f16 mma), %s q/out" % args.dtype) if fp8 else args.dtype,
            "data": "synthetic",
            "config": config}
    if fp8:
        config["kv_cache"] = ("e4m3 bytes, per-KV-head scales k %s v %s"
                              % (wl.kv_scales(0), wl.kv_scales(1)))
    prefill_heavy = counts["flops_by_kind"]["prefill"] > 0
    if prefill_heavy:
        # Mixed batch: one figure of merit = t_ideal / t_measured, where
        # t_ideal = decode-side bytes / HBM peak + prefill FLOPs / bf16 peak.
        t_ideal = ((counts["step_bytes"] - counts["kv_bytes"]["prefill"]) / (peaks["hbm_gbs"] * 1e9)
                   + counts["flops_by_kind"]["prefill"] / (peaks["bf16_tflops"] * 1e12))
        line["value"] = 100.0 * t_ideal / (ms_per_step * 1e-3)
        line["unit"] = "% of roofline"
        line["e2e"] = {"value": 100.0 * t_ideal / (e2e_ms * 1e-3), "unit": "% of roofline",
                       "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms}
        ach = counts["flops"] / (attn_ms_avg * 1e-3) / 1e12
        line["roofline"] = {"bound": "tensor",
                            "kernel": ("plan + attn_tc_kernel<%d> (every segment)" % D if D > 128
                                       else "plan + attn_tc_kernel<128, fp8> + attn_split_kernel<128, fp8>"
                                       if fp8 else
                                       "plan + attn_tc_kernel<128> + attn_split_kernel<128>"),
                            "achieved": ach, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                            "frac": ach / peaks["bf16_tflops"], "traffic": None,
                            "peak_source": peaks["source"], "attn_ms_per_launch": attn_ms_avg}
    else:
        achieved = counts["attn_bytes"] / (attn_ms_avg * 1e-3) / 1e9
        line["e2e"] = {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                       "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms}
        kname = "attn_split_kernel<128, fp8>" if fp8 else "attn_split_kernel<128>"
        tname = "attn_tc_kernel<128, fp8>" if fp8 else "attn_tc_kernel<128>"
        if D > 128:   # head size 256: every segment on the prefill kernel
            kname = tname = "attn_tc_kernel<%d>" % D
        line["roofline"] = {"bound": "hbm",
                            "kernel": ("plan + %s (prefix) + %s (suffix) + cascade_combine_kernel<%d>"
                                       % (tname, kname, D) if cascade else
                                       "plan + %s (every segment)" % kname if D > 128 else
                                       "plan + %s (+ split combine)" % kname),
                            "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                            "frac": achieved / peaks["hbm_gbs"],
                            "traffic": load_traffic(kname, config["workload"]),
                            "peak_source": peaks["source"], "attn_ms_per_launch": attn_ms_avg}
    line["roofline"]["timing"] = ("the attention call alone (same inputs), replayed once per "
                                  "timed step right after the timed steps, CUDA events per launch")
    line["config"]["step"] = (("cascade_fwd_fp8kv" if cascade else "varlen_fwd_fp8kv") if fp8 else
                              ("cascade_fwd_with_update" if cascade else "varlen_fwd_with_update")) + \
        " (scatter of the new K/V + attention in one call)"
    if sub:
        for kind, r in sub.items():
            r["frac_hbm"] = r["gbs"] / peaks["hbm_gbs"]
            r["frac_bf16"] = r["tflops"] / peaks["bf16_tflops"]
            r["frac_bf16_sustained"] = r["tflops"] / peaks["bf16_tflops_sustained"]
        line["sub_launches"] = sub
    if prefill:
        # The headline's second half: the long-context prefill sub-launch, with
        # the chunked-prefill chunks beside it.
        main_leg = prefill.pop("long_context_70b_prefill", None)
        if main_leg is not None:
            line["prefill"] = main_leg
        for k, v in prefill.items():
            line["prefill_" + k] = v
    # Our kernels per step: scatter, planner, then per attention pass the
    # split-KV kernel and/or the prefill kernel (the host launches a kernel
    # only when some segment can need it).
    G = H // wl.num_kv_heads
    # The prefill kernel takes segments of more than 32 packed rows (every
    # segment at head size 256, where the split-KV kernel is not launched).
    tc_rows = lambda rows: rows > 32 or D > 128
    if cascade:
        # scatter, planner, prefix pass (prefill kernel for more than 32
        # packed rows, else split-KV), suffix pass (split-KV and/or prefill
        # kernel), combine
        per_step = 2 + 1 + 1 + (1 if tc_rows(wl.max_seqlen_q * G) else 0) + 1
    else:
        per_step = 3 + (1 if tc_rows(wl.max_seqlen_q * G) else 0)
    if D > 128:
        per_step -= 1   # no split-KV launch beside the prefill kernel
    line["gpu_launches"] = per_step * args.steps
    for r in rows_fig.values():
        r["frac_hbm"] = r["gbs"] / peaks["hbm_gbs"]
    line["steps_standalone"] = rows_fig
    line["graph"] = graphs is not None
    line["clocks"] = clocks
    if not args.no_cpu_baseline:
        b, f, sec, desc = run_oracle_sample(wl, max_seconds=args.cpu_seconds, fp8=fp8)
        line["cpu_baseline"] = {"value": b / sec / 1e9, "unit": "GB/s",
                                "cores": torch.get_num_threads(), "kind": "oracle",
                                "sample": desc}
    print(json.dumps(line))


def bench_prefill_only(args, rank, world, local):
    """Only the prefill sub-launch records (one line per leg): the command the
    profiler captures of the prefill kernel run."""
    import paged_kv_varlen_attn_gb300 as pa
    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA GPU (no CPU fallback)")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    from paged_kv_varlen_attn_gb300 import _build
    _build.build()
    pa.load_library()
    peaks = load_peaks()
    names = list(PREFILL_LEGS) if args.workload == "decode_llama8b" else [args.workload]
    for name in names:
        rec = prefill_record(pa, name, dev, peaks, args.steps, min_ms=0.0,
                             dtype=DTYPES[args.dtype], fp8=args.kv_cache == "fp8")
        if rank == 0:
            print(json.dumps({"prefill": rec}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="decode_llama8b", choices=sorted(W.CONFIGS))
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--kv-cache", default="bf16", choices=["bf16", "fp8"],
                    help="page pool element type: bf16, or e4m3 bytes with per-KV-head scales")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--dtype", default="bf16", choices=sorted(DTYPES),
                    help="element type of Q, the 2-byte K/V pools and the outputs")
    ap.add_argument("--no-prefill", action="store_true",
                    help="skip the prefill sub-launch records (the metric's prefill half)")
    ap.add_argument("--prefill-only", action="store_true",
                    help="time only the prefill sub-launches (for profiler captures)")
    ap.add_argument("--no-graph", action="store_true",
                    help="launch the C-ABI calls directly instead of replaying CUDA graphs")
    args = ap.parse_args()
    rank, world, local = dist_setup(args.gpus)
    if args.impl == "reference":
        bench_reference(args, rank, world)
    elif args.prefill_only:
        bench_prefill_only(args, rank, world, local)
    else:
        bench_ours(args, rank, world, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
