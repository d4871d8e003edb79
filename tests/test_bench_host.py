"""bench.py's host-side logic without a GPU: every committed ncu summary it
reads matches the current kernel sources (else its DRAM traffic figure is
void), and the launch counts it claims follow the library's own rules."""

import os
import re
import types

import pytest

import bench
from mla_latent_kv_03_gb300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("key", sorted(bench.PROFILES))
def test_every_registered_profile_matches_the_current_sources(key):
    fname, sources = bench.PROFILES[key]
    text = open(os.path.join(ROOT, "profiles", fname)).read()
    rec = re.search(r"source_sha256: `(\w+)`", text)
    assert rec, fname
    assert rec.group(1) == bench.source_hash(sources), f"{fname}: sources changed since the capture"
    assert bench.profiled_traffic(*key) > 0


def test_projection_launch_counts_follow_the_split_rule():
    # 64 tokens: too few tiles for 152 SMs, so K splits and a sum kernel follows
    assert bench.proj_launches(64, 16 * 192, 2048, 152) == 2
    assert bench.proj_launches(64, 576, 2048, 152) == 2
    # thousands of tokens: enough tiles, one kernel
    assert bench.proj_launches(4096, 16 * 192, 2048, 152) == 1


def test_decode_launch_counts():
    props = types.SimpleNamespace(multi_processor_count=152)
    serving = W.serving(batch=4, seq_len=64)      # the same layout rules, small draws
    assert bench.decode_call_launches(serving, props) == (True, 2)   # 4 rows: split-heavy
    w = W.make("x", [64] * 64, [1] * 64, 16, 64, "bf16", seed=1)
    assert bench.decode_call_launches(w, props) == (True, 1)         # one fused launch
    mixed = W.mixed()
    d = bench.w_decode_part(mixed)
    assert (d.num_q, d.batch) == (60, 60)
    assert bench.decode_call_launches(d, props) == (True, 1)
