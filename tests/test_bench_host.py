"""bench.py's host-side logic without a GPU: the gate on the committed ncu
summaries (a DRAM traffic figure counts only while the kernel's code is the
code that was captured), and the launch counts it claims follow the library's
own rules."""

import os
import re
import types

import pytest

import bench
from mla_latent_kv_03_gb300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_code_hash_ignores_comments_and_layout_but_not_code():
    a = "int f(int x) {  // add one\n  return x + 1; /* plain */ }\n"
    b = "/* header */ int f(int x)\n{\n    return x + 1;\n}"
    c = "int f(int x) { return x + 2; }"
    assert bench.strip_comments(a) == bench.strip_comments(b)
    assert bench.strip_comments(a) != bench.strip_comments(c)


def test_traffic_is_void_once_the_code_changes(tmp_path, monkeypatch):
    src = tmp_path / "mla_latent_kv_03_gb300" / "csrc"
    src.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    (src / "k.cu").write_text("__global__ void k() { }  // v1\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setitem(bench.PROFILES, ("k", "w"), ("k_w.md", ["k.cu"]))
    h = bench.code_hash(["k.cu"])
    (tmp_path / "profiles" / "k_w.md").write_text(
        f"- code_sha256: `{h}`\n- dram_bytes_per_launch_full_size: `123,456`\n")
    assert bench.profiled_traffic("k", "w") == 123456.0
    (src / "k.cu").write_text("// a new header comment\n__global__ void k() { }\n")
    assert bench.profiled_traffic("k", "w") == 123456.0
    (src / "k.cu").write_text("__global__ void k() { int x = 1; }\n")
    assert bench.profiled_traffic("k", "w") is None
    assert bench.profiled_traffic("other", "w") is None


@pytest.mark.parametrize("key", sorted(bench.PROFILES))
def test_every_registered_profile_is_well_formed(key):
    """Each summary exists, records the command that made it, its code hash
    and its per-launch traffic; the bench uses the figure only while the hash
    matches (a stale summary reads as null, never as a number)."""
    fname, sources = bench.PROFILES[key]
    text = open(os.path.join(ROOT, "profiles", fname)).read()
    assert "ncu " in text and "--clock-control none" in text, fname
    vals = bench.profile_fields(fname)
    assert re.fullmatch(r"[0-9a-f]{16}", vals.get("code_sha256", "")), fname
    assert float(vals["dram_bytes_per_launch_full_size"].replace(",", "")) > 0
    t = bench.profiled_traffic(*key)
    assert t is None or t > 0


def test_projection_launch_counts_follow_the_split_rule():
    # 64 tokens: too few tiles for 152 SMs, so K splits and a sum kernel follows
    assert bench.proj_launches(64, 16 * 192, 2048, 152) == 2
    assert bench.proj_launches(64, 576, 2048, 152) == 2
    # from 256 tokens: one tensor-core kernel, no split
    assert bench.proj_launches(256, 576, 2048, 152) == 1
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
