"""Host-side arithmetic of bench.py (no GPU): the algorithmic byte and flop counts
the roofline divides by, the L2-flush rule, and the traffic record's guard on the
kernel source."""
import json
import os

import numpy as np
import torch

import bench
from mla_paged_kv_02_gb300 import synth


def _small(q_len=3, lens=(5, 64, 130), H=4, **kw):
    return synth.make_inputs("tiny", seed=7, kv_lens=list(lens), q_len=q_len, batch=len(lens), num_heads=H, **kw)


def test_algorithmic_bytes_counts_each_row_once():
    inp = _small()
    rows = 3 * 3 * 4
    kv = (5 + 64 + 130) * 576 * 2
    assert bench.algorithmic_bytes(inp, 2) == kv + rows * 576 * 2 + rows * (512 * 2 + 4)
    assert bench.algorithmic_bytes(inp, 4) == kv + rows * 576 * 2 + rows * (512 * 4 + 4)
    fp8 = _small(kv_fp8=True)
    assert bench.algorithmic_bytes(fp8, 2) == (5 + 64 + 130) * 576 + rows * 576 * 2 + rows * (512 * 2 + 4)


def test_visible_pairs_matches_the_causal_mask_by_enumeration():
    inp = _small()
    L = inp.seq_lens.tolist()
    brute = 0
    for b in range(inp.batch):
        for i in range(inp.q_len):
            for h in range(inp.num_heads):
                for t in range(L[b]):  # query i sits at L - q_len + i and sees [0, that]
                    brute += t <= L[b] - inp.q_len + i
    assert bench.visible_pairs(inp) == brute
    assert bench.algorithmic_flops(inp) == 2176 * brute


def test_l2_flush_rule():
    l2 = 129 << 20
    assert bench.needs_l2_flush(320 << 20, l2)          # plain's 320 MB: under 4x L2
    assert not bench.needs_l2_flush(6 << 30, l2)        # MTP-3's 6 GB streams past L2
    assert bench.needs_l2_flush(6 << 30, l2, "on")
    assert not bench.needs_l2_flush(1 << 20, l2, "off")


def test_recorded_traffic_only_for_the_current_kernel_source():
    path = os.path.join(bench.ROOT, "profiles", "traffic.json")
    with open(path) as f:
        rec = json.load(f)
    sha = bench.kernel_source_sha()
    assert len(sha) == 16
    for w, ent in rec.items():
        got = bench.recorded_traffic(w)
        if ent["kernel_sha"] == sha:
            assert got == ent["dram_bytes_per_launch"]
            # DRAM bytes within a few percent of the algorithmic bytes: no page read twice
            assert 0.9 < ent["dram_bytes_per_launch"] / ent["algorithmic_bytes_per_launch"] < 1.3
        else:
            assert got is None
    assert bench.recorded_traffic("no such workload") is None
