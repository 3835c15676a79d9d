"""Host logic of bench.py that the reported numbers rest on, on CPU: the
algorithmic byte and FLOP counts (checked against counts worked out by hand
for small batches), the kernel-source hash that keys the committed DRAM
traffic records, and the parsing of the nvidia-smi clock record."""
import types

import bench


def _wl(q_lens, kv_lens, H=4, Hk=2, D=64, bs=16, causal=True, prefix=0):
    return types.SimpleNamespace(num_heads=H, num_kv_heads=Hk, head_size=D, block_size=bs,
                                 q_lens=list(q_lens), kv_lens=list(kv_lens),
                                 num_seqs=len(q_lens), causal=causal,
                                 common_prefix_len=prefix)


def test_decode_counts_by_hand():
    # two decode rows (G = 2: 2 packed rows each, not prefill), 40 and 17 keys
    wl = _wl([1, 1], [40, 17])
    c = bench.algorithmic_counts(wl)
    per_key = 2 * 64 * 2 * 2            # H_kv x D x (K and V) x 2 bytes
    assert c["kv_bytes"] == {"decode": (40 + 17) * per_key, "prefill": 0}
    qo = 2 * 2 * 4 * 64 * 2             # Q and O: T = 2 tokens x H x D x 2 bytes
    lse = 4 * 2 * 4
    bt = (3 + 2) * 4                    # ceil(40/16) + ceil(17/16) table entries
    assert c["qo_lse_bt"] == qo + lse + bt
    assert c["attn_bytes"] == (40 + 17) * per_key + qo + lse + bt
    assert c["scatter_bytes"] == 2 * 2 * 2 * 64 * (2 + 2)
    assert c["flops"] == 4 * 64 * 4 * (40 + 17)   # 4 D H per visible (query, key) pair


def test_causal_prefill_pairs_by_hand():
    # 20 queries (40 packed rows: prefill) ending at key 50: bottom-right mask
    wl = _wl([20], [50])
    c = bench.algorithmic_counts(wl)
    pairs = sum(50 - 20 + i + 1 for i in range(20))
    assert c["flops_by_kind"] == {"decode": 0, "prefill": 4 * 64 * 4 * pairs}
    nc = bench.algorithmic_counts(_wl([20], [50], causal=False))
    assert nc["flops"] == 4 * 64 * 4 * 20 * 50


def test_cascade_counts_the_prefix_once():
    wl = _wl([1, 1, 1], [48, 70, 33], prefix=32)
    c = bench.algorithmic_counts(wl, cascade=True)
    per_key = 2 * 64 * 2 * 2
    assert c["kv_bytes"]["decode"] == (16 + 38 + 1) * per_key + 32 * per_key
    flat = bench.algorithmic_counts(wl)
    assert flat["kv_bytes"]["decode"] - c["kv_bytes"]["decode"] == 2 * 32 * per_key


def test_fp8_counts_one_byte_per_element():
    wl = _wl([1], [40])
    c8 = bench.algorithmic_counts(wl, fp8=True)
    c2 = bench.algorithmic_counts(wl)
    assert 2 * c8["kv_bytes"]["decode"] == c2["kv_bytes"]["decode"]
    assert c8["scatter_bytes"] == 2 * 1 * 2 * 64 * (2 + 1)


def test_traffic_records_are_keyed_by_the_kernel_sources(tmp_path, monkeypatch):
    import json
    rec = {"attn_split_kernel<128>": {"w": {
        "source_sha": bench.sources_sha(bench.KERNEL_SRCS["attn_split_kernel<128>"]),
        "dram_bytes_per_launch": 123}}}
    p = tmp_path / "traffic.json"
    p.write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(p))
    assert bench.load_traffic("attn_split_kernel<128>", "w") == 123
    assert bench.load_traffic("attn_split_kernel<128>", "other") is None
    rec["attn_split_kernel<128>"]["w"]["source_sha"] = "0" * 16   # sources changed since
    p.write_text(json.dumps(rec))
    assert bench.load_traffic("attn_split_kernel<128>", "w") is None


def test_clock_record_parsing():
    s = bench.ClockSampler(0)
    s.proc = types.SimpleNamespace(terminate=lambda: None, wait=lambda timeout=None: 0)
    s.lines = ["2070, 2070, Not Active, Not Active, Not Active, Not Active",
               "2055, 2070, Not Active, Not Active, Not Active, Active",
               "1980, 2070, Not Active, Not Active, Not Active, Active",
               "[N/A], 2070, Not Active, Not Active, Not Active, Not Active",
               "garbage"]
    r = s.stop()
    assert r == {"sm_mhz": 2055.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"],
                 "samples": 3}


def test_committed_traffic_records_name_their_captures():
    """Every committed DRAM-traffic record names the summary under profiles/
    that gives its ncu command, and keys a kernel and a workload the bench
    knows."""
    import json
    import os
    import workloads as W
    with open(bench.TRAFFIC_FILE) as f:
        t = json.load(f)
    for kernel, recs in t.items():
        assert kernel in bench.KERNEL_SRCS
        for workload, e in recs.items():
            assert workload.split("+")[0] in W.CONFIGS
            path = os.path.join(bench.ROOT, e["capture"])
            assert os.path.isfile(path) and e["capture"].startswith("profiles/")
            with open(path) as f:
                assert "ncu " in f.read()
            assert e["dram_bytes_per_launch"] == e["dram_bytes_read"] + e["dram_bytes_write"]
