"""GPU parity: every libmla call against the fp64 oracle, through the C ABI.

Each step is checked in isolation (on the GPU's own inputs to that step) and
end to end (raw inputs -> out, against the naive expanded form), on the
workloads of the problem statement: small cases the oracle finishes in
seconds over every row, the full-size ones on sampled sequences and heads.
"""

import numpy as np
import pytest
import torch

from _helpers import (BF16_MAX_ABS, assert_close, bf16_ulp, errors, ref_cache_rows,
                      ref_o_lat_from, ref_out, ref_q_abs, to_f64)
from mla_latent_kv_03_gb300 import libmla as L
from mla_latent_kv_03_gb300 import workloads as W
from mla_latent_kv_03_gb300.step import MlaDecodeStep
from oracle import mla_oracle as O

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    L.load()


def _sentinel_fill(dtype):
    return float("nan")


# ---------------------------------------------------------------------------
# mla_cache_write
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dtype,bs", [("f32", 16), ("bf16", 16), ("bf16", 32), ("bf16", 64)])
def test_cache_write_placement_is_bit_exact(dtype, bs):
    w = W.make("cw", [7, 33, 64, 65, 130, 1], [1] * 6, 16, bs, dtype, seed=21, extra_blocks=3)
    s = MlaDecodeStep(w, device=DEV)
    itype = torch.int16 if dtype == "bf16" else torch.int32
    pattern = 0x7FC1 if dtype == "bf16" else 0x7FC00123   # a NaN bit pattern
    s.cache.view(itype).fill_(pattern)
    # add padding tokens (slot -1) that must write nothing
    L.mla_cache_write(s.cfg, s.c_kv[:5].contiguous(), s.k_pe[:5].contiguous(),
                      s.kv_positions[:5].contiguous(),
                      torch.full((5,), -1, dtype=torch.int64, device=DEV),
                      s.rms_weight, s.cache, s.status)
    s.populate()
    torch.cuda.synchronize()
    assert L.mla_get_device_status(s.status)[0] == 0
    bits = s.cache.view(itype).cpu().numpy().reshape(-1, 576)
    written = np.zeros(bits.shape[0], dtype=bool)
    written[w.slot_mapping] = True
    assert np.all(bits[~written] == np.array(pattern).astype(bits.dtype)), "bytes outside the slots changed"
    got = to_f64(s.cache).reshape(-1, 576)[w.slot_mapping]
    ref = ref_cache_rows(w)
    if dtype == "bf16":
        assert np.all(np.abs(got - ref) <= bf16_ulp(ref)), "row values beyond 1 bf16 ulp"
    else:
        np.testing.assert_allclose(got, ref, rtol=1e-6, atol=1e-6)


def test_cache_write_bad_slot_sets_status_and_writes_nothing():
    w = W.make("cw_bad", [10], [1], 16, 16, "bf16", seed=22)
    s = MlaDecodeStep(w, device=DEV)
    s.cache.view(torch.int16).fill_(0x7FC1)
    bad = torch.full((10,), w.num_blocks * 16, dtype=torch.int64, device=DEV)
    L.mla_cache_write(s.cfg, s.c_kv, s.k_pe, s.kv_positions, bad, s.rms_weight, s.cache, s.status)
    st, bits = L.mla_get_device_status(s.status)
    assert st == 8 and bits & L.DEV_BAD_SLOT
    assert torch.all(s.cache.view(torch.int16) == 0x7FC1)


# ---------------------------------------------------------------------------
# mla_absorb_q and mla_out_proj
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dtype,nq,heads", [("f32", 3, 16), ("bf16", 1, 16), ("bf16", 37, 32),
                                            ("bf16", 64, 16), ("bf16", 200, 16),
                                            ("bf16", 600, 16), ("bf16", 5, 128)])
def test_absorb_q(dtype, nq, heads):
    w = W.make("aq", [40] * nq, [1] * nq, heads, 64, dtype, seed=23)
    s = MlaDecodeStep(w, device=DEV)
    s.absorb()
    got = to_f64(s.q_abs)
    ref = ref_q_abs(w)
    if dtype == "f32":
        np.testing.assert_allclose(got, ref, rtol=0, atol=2e-5)
    else:
        assert np.all(np.abs(got - ref) <= 2 * bf16_ulp(ref) + 1e-5), "q_abs beyond 2 bf16 ulp"


@pytest.mark.parametrize("dtype,nq,heads", [("f32", 3, 16), ("bf16", 1, 16), ("bf16", 64, 16),
                                            ("bf16", 37, 32), ("bf16", 600, 16), ("bf16", 9, 128)])
def test_out_proj(dtype, nq, heads):
    w = W.make("op", [8] * nq, [1] * nq, heads, 64, dtype, seed=24)
    s = MlaDecodeStep(w, device=DEV)
    o = torch.randn(nq, heads, 512, generator=torch.Generator().manual_seed(5)) / 20
    s.o_lat.copy_(o)
    s.out_proj()
    got = to_f64(s.out)
    ref = O.out_proj(o.double().numpy(), w.W_uv)
    assert_close(got, ref, dtype, "out_proj")


# ---------------------------------------------------------------------------
# mla_decode_paged + mla_combine on the GPU's own cache rows and q_abs
# ---------------------------------------------------------------------------

SMALL = {
    "tiny_fp32": lambda: W.tiny(),
    "ragged_tails_bf16": lambda: W.make("ragged_tails", [1, 63, 64, 65, 127, 128, 129, 1000],
                                        [1] * 8, 16, 64, "bf16", seed=31, extra_blocks=2),
    "bs16_bf16": lambda: W.make("bs16", [5, 40, 200], [1] * 3, 16, 16, "bf16", seed=32),
    "bs32_h32_bf16": lambda: W.make("bs32h32", [33, 97], [1, 1], 32, 32, "bf16", seed=33),
    "h128_bf16": lambda: W.make("h128", [17, 300, 1], [1] * 3, 128, 64, "bf16", seed=34),
    "h64_bf16": lambda: W.make("h64", [70, 2], [1, 1], 64, 64, "bf16", seed=35),
    "prefill_bf16": lambda: W.make("prefill", [150, 64, 20], [40, 1, 20], 16, 64, "bf16", seed=36),
    "empty_seq_bf16": lambda: W.make("empty", [0, 5, 0, 70], [0, 1, 0, 1], 16, 64, "bf16", seed=37),
}


@pytest.mark.parametrize("name", sorted(SMALL))
def test_decode_and_combine_vs_latent_oracle(name):
    w = SMALL[name]()
    s = MlaDecodeStep(w, device=DEV)
    s.populate()
    s.absorb()
    s.decode()
    s.combine()
    torch.cuda.synchronize()
    assert s.device_status()[0][0] == 0
    ref = ref_o_lat_from(w, to_f64(s.cache), to_f64(s.q_abs))
    assert_close(to_f64(s.o_lat), ref, w.dtype, f"o_lat {name}")


@pytest.mark.parametrize("name", sorted(SMALL))
def test_end_to_end_vs_naive_oracle(name):
    w = SMALL[name]()
    s = MlaDecodeStep(w, device=DEV)
    s.populate()
    got = to_f64(s.step())
    torch.cuda.synchronize()
    assert s.device_status()[0][0] == 0
    assert_close(got, ref_out(w), w.dtype, f"out {name}")


@pytest.mark.parametrize("seq_len", [1, 256, 1024])
def test_v2lite_decode(seq_len):
    w = W.v2lite(seq_len)
    s = MlaDecodeStep(w, device=DEV)
    s.populate()
    assert_close(to_f64(s.step()), ref_out(w), "bf16", f"v2lite L={seq_len}")


def test_tiny_fp32_meets_page_bar():
    w = W.tiny()
    s = MlaDecodeStep(w, device=DEV)
    s.populate()
    max_abs, _ = errors(to_f64(s.step()), ref_out(w))
    assert max_abs <= 1e-4


def test_block_table_permutation_gives_identical_bits():
    a = W.make("perm", [300, 129, 64], [1] * 3, 16, 64, "bf16", seed=41, extra_blocks=4)
    b = W.make("perm", [300, 129, 64], [1] * 3, 16, 64, "bf16", seed=41, extra_blocks=4)
    rng = np.random.default_rng(99)
    perm = rng.permutation(b.num_blocks).astype(np.int32)
    bt = b.block_table.copy()
    bt[bt >= 0] = perm[bt[bt >= 0]]
    b.block_table = bt
    b.slot_mapping = bt[b.token_seq, b.kv_positions // 64].astype(np.int64) * 64 + b.kv_positions % 64
    outs = []
    for w in (a, b):
        s = MlaDecodeStep(w, device=DEV, num_ctas=5)
        s.populate()
        outs.append(s.step().clone())
    torch.cuda.synchronize()
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))


@pytest.mark.parametrize("num_ctas", [1, 3, 64, 0, 500])
def test_split_count_does_not_change_the_result(num_ctas):
    w = W.make("splits", [2000, 1, 333, 64], [1, 1, 1, 1], 16, 64, "bf16", seed=42)
    s = MlaDecodeStep(w, device=DEV, num_ctas=num_ctas)
    s.populate()
    got = to_f64(s.step())
    assert_close(got, ref_out(w), "bf16", f"num_ctas={num_ctas}")


# ---------------------------------------------------------------------------
# device-side errors: reported, skipped, no fault
# ---------------------------------------------------------------------------

def test_bad_block_entry_is_reported_and_skipped():
    w = W.make("badblk", [200, 100], [1, 1], 16, 64, "bf16", seed=43)
    s = MlaDecodeStep(w, device=DEV)
    s.populate()
    bt = s.block_table.clone()
    s.block_table[0, 1] = w.num_blocks + 7          # out of range
    s.step()
    (st, bits), _ = s.device_status()
    assert st == 6 and bits & L.DEV_BAD_BLOCK
    got = to_f64(s.out)
    # the untouched sequence is still exact
    assert_close(got[1:2], ref_out(w, seqs=[1])[1:2], "bf16", "other sequence")
    assert np.all(np.isfinite(got))
    s.block_table.copy_(bt)
    s.step()
    assert s.device_status()[0][0] == 0


def test_query_longer_than_sequence_is_reported():
    w = W.make("badseq", [50, 60], [1, 1], 16, 64, "bf16", seed=44)
    s = MlaDecodeStep(w, device=DEV)
    s.populate()
    s.seq_lens[0] = 0                                 # one query row, zero tokens
    s.step()
    (st, bits), _ = s.device_status()
    assert st == 7 and bits & L.DEV_BAD_SEQ
    out = to_f64(s.out)
    assert np.all(out[0] == 0)
    assert_close(out[1:2], ref_out(w, seqs=[1])[1:2], "bf16", "other sequence")


def test_bounded_wait_times_out_and_context_survives():
    word = torch.zeros(1, dtype=torch.int32, device=DEV)
    L.mla_selftest_wait_timeout(word, 20_000_000)    # 20 ms
    st, bits = L.mla_get_device_status(word)
    assert st == 5 and bits == L.DEV_TIMEOUT
    w = W.tiny()
    s = MlaDecodeStep(w, device=DEV)
    s.populate()
    max_abs, _ = errors(to_f64(s.step()), ref_out(w))
    assert max_abs <= 1e-4


# ---------------------------------------------------------------------------
# the self-planned decode: one launch plans, decodes (and merges)
# ---------------------------------------------------------------------------

SELF_CASES = ["bs16_bf16", "bs32_h32_bf16", "empty_seq_bf16", "ragged_tails_bf16"]


def _plan_bytes(s):
    """Header fields, row_info and cta_start of the decode workspace (the
    16-row layout: fixed counters end at 2,304 bytes, then row_info[num_q],
    then cta_start[num_ctas], each 256-byte aligned)."""
    ws = s.workspace.cpu().numpy()
    nq = s.w.num_q
    hdr = ws[4:40].view(np.int32)
    ctas = int(hdr[4])
    ri0 = 2304
    cs0 = ri0 + (nq * 16 + 255) // 256 * 256
    return hdr.copy(), ws[ri0:ri0 + nq * 16].view(np.int32).copy(), ws[cs0:cs0 + ctas * 16].view(np.int32).copy()


@pytest.mark.parametrize("name", SELF_CASES)
@pytest.mark.parametrize("num_ctas", [0, 7, 500])
def test_self_planned_decode_writes_the_plan_kernels_plan(name, num_ctas):
    w = SMALL[name]()
    a = MlaDecodeStep(w, device=DEV, num_ctas=num_ctas)
    b = MlaDecodeStep(w, device=DEV, num_ctas=num_ctas)
    a.populate()
    a.absorb()
    a.decode()                      # one launch: the kernel plans for itself
    b.plan()                        # the plan kernel
    torch.cuda.synchronize()
    assert a.device_status()[0][0] == 0
    for x, y, what in zip(_plan_bytes(a), _plan_bytes(b), ("header", "row_info", "cta_start")):
        assert np.array_equal(x, y), f"{what} differs from the plan kernel's"
    # and the partials it left are the planned decode's, bit for bit
    a.combine()
    o_self = a.o_lat.clone()
    a.decode_planned()
    a.combine()
    torch.cuda.synchronize()
    assert torch.equal(o_self, a.o_lat)


@pytest.mark.parametrize("name", SELF_CASES)
@pytest.mark.parametrize("num_ctas", [0, 7, 500])
def test_decode_paged_combine_matches_oracle_and_repeats(name, num_ctas):
    w = SMALL[name]()
    s = MlaDecodeStep(w, device=DEV, num_ctas=num_ctas)
    s.populate()
    s.absorb()
    outs = []
    for _ in range(3):
        s.o_lat.fill_(float("nan"))                  # rows nobody visits must become 0
        s.decode_paged_combine()
        outs.append(s.o_lat.clone())
    torch.cuda.synchronize()
    assert s.device_status()[0][0] == 0
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[1], outs[2]), "counters not reset"
    fused = to_f64(outs[0])
    ref = ref_o_lat_from(w, to_f64(s.cache), to_f64(s.q_abs))
    empty = np.isnan(ref).all(axis=(1, 2))
    assert np.all(fused[empty] == 0)
    assert_close(fused, ref, w.dtype, f"decode_paged_combine o_lat {name}")
    s.decode_planned()
    s.combine()
    np.testing.assert_allclose(fused, to_f64(s.o_lat), rtol=0, atol=1e-5)


@pytest.mark.parametrize("num_ctas", [0, 40])
def test_decode_paged_combine_serving_shape(num_ctas):
    # 16 rows of 4,096 tokens: every row is cut into several parts (about 7
    # with one CTA per SM, 2 with 40 CTAs), merged by the CTA that finishes last
    w = W.make("srv16", [4096] * 16, [1] * 16, 16, 64, "bf16", seed=47)
    s = MlaDecodeStep(w, device=DEV, num_ctas=num_ctas)
    s.populate()
    s.absorb()
    s.decode_paged_combine()
    s.out_proj()
    torch.cuda.synchronize()
    assert s.device_status()[0][0] == 0
    ref = ref_o_lat_from(w, to_f64(s.cache), to_f64(s.q_abs))
    assert_close(to_f64(s.o_lat), ref, "bf16", f"o_lat, num_ctas={num_ctas}")
    assert_close(to_f64(s.out), ref_out(w), "bf16", f"out, num_ctas={num_ctas}")


def test_decode_paged_combine_many_parts():
    # the 3,000-token row (47 tiles, 2 per CTA) is cut into 24 parts: twelve
    # rounds of two parts in the merging CTA
    lens = [3000] + [1] * 9 + [333, 64]
    w = W.make("many_self", lens, [1] * len(lens), 16, 64, "bf16", seed=48)
    s = MlaDecodeStep(w, device=DEV, num_ctas=40)
    s.populate()
    s.absorb()
    s.decode_paged_combine()
    s.out_proj()
    torch.cuda.synchronize()
    assert s.device_status()[0][0] == 0
    assert_close(to_f64(s.out), ref_out(w), "bf16", "self-planned, 24 parts")


def test_decode_paged_combine_reports_a_bad_sequence():
    w = W.make("badseq_self", [50, 60], [1, 1], 16, 64, "bf16", seed=49)
    s = MlaDecodeStep(w, device=DEV)
    s.populate()
    s.absorb()
    s.seq_lens[0] = 0                                 # one query row, zero tokens
    s.o_lat.fill_(float("nan"))
    s.decode_paged_combine()
    (st, bits), _ = s.device_status()
    assert st == 7 and bits & L.DEV_BAD_SEQ
    got = to_f64(s.o_lat)
    assert np.all(got[0] == 0)
    ref = ref_o_lat_from(w, to_f64(s.cache), to_f64(s.q_abs))
    assert_close(got[1:2], ref[1:2], "bf16", "other sequence")
    L.mla_workspace_init(s.workspace)                 # re-init after a device error


# ---------------------------------------------------------------------------
# mla_decode_combine: the decode kernel merging its own splits
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("name", sorted(SMALL))
@pytest.mark.parametrize("num_ctas", [0, 7, 500])
def test_fused_decode_combine_matches_oracle_and_unfused(name, num_ctas):
    w = SMALL[name]()
    s = MlaDecodeStep(w, device=DEV, num_ctas=num_ctas)
    s.populate()
    s.absorb()
    s.plan()
    s.o_lat.fill_(float("nan"))                      # rows nobody visits must become 0
    s.decode_combine()
    torch.cuda.synchronize()
    assert s.device_status()[0][0] == 0
    fused = to_f64(s.o_lat)
    ref = ref_o_lat_from(w, to_f64(s.cache), to_f64(s.q_abs))
    empty = np.isnan(ref).all(axis=(1, 2))
    assert np.all(fused[empty] == 0)
    assert_close(fused, ref, w.dtype, f"fused o_lat {name}")
    s.decode_planned()
    s.combine()
    unfused = to_f64(s.o_lat)
    tol = 1e-6 if w.dtype == "f32" else 1e-5
    np.testing.assert_allclose(fused, unfused, rtol=0, atol=tol)


def test_fused_merge_of_many_splits():
    # 12 q-tiles over 40 CTAs keeps the merge inside the decode kernel; the
    # 3,000-token row (47 tiles, 2 per CTA) is cut into 24 parts, more than
    # one chunk of staged merge weights
    lens = [3000] + [1] * 9 + [333, 64]
    w = W.make("many", lens, [1] * len(lens), 16, 64, "bf16", seed=45)
    s = MlaDecodeStep(w, device=DEV, num_ctas=40)
    s.populate()
    s.absorb()
    s.plan()
    s.decode_combine()
    s.out_proj()
    assert_close(to_f64(s.out), ref_out(w), "bf16", "fused, 500 CTAs")


def test_fused_decode_combine_repeats_on_one_plan():
    w = W.make("repeat", [700, 1, 129], [1, 1, 1], 16, 64, "bf16", seed=46)
    s = MlaDecodeStep(w, device=DEV, num_ctas=9)
    s.populate()
    s.absorb()
    s.plan()
    outs = []
    for _ in range(3):
        s.o_lat.fill_(float("nan"))
        s.decode_combine()
        outs.append(s.o_lat.clone())
    torch.cuda.synchronize()
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[1], outs[2])
    ref = ref_o_lat_from(w, to_f64(s.cache), to_f64(s.q_abs))
    assert_close(to_f64(outs[2]), ref, "bf16", "third launch on one plan")


@pytest.mark.parametrize("name", sorted(SMALL))
@pytest.mark.parametrize("num_ctas", [0, 7, 500])
def test_combine_out_proj_matches_separate_calls_and_oracle(name, num_ctas):
    w = SMALL[name]()
    s = MlaDecodeStep(w, device=DEV, num_ctas=num_ctas)
    s.populate()
    s.absorb()
    s.plan()
    s.decode_planned()
    s.out.fill_(float("nan"))
    s.combine_out_proj()
    torch.cuda.synchronize()
    fused = to_f64(s.out)
    assert_close(fused, ref_out(w), w.dtype, f"combine_out_proj {name}")
    s.combine()
    s.out_proj()
    sep = to_f64(s.out)
    if w.dtype == "f32":
        np.testing.assert_allclose(fused, sep, rtol=0, atol=1e-6)
    else:  # both round the merged row to bf16 for the mma; the merge order differs
        assert np.max(np.abs(fused - sep)) <= 2e-3


def test_combine_out_proj_many_rows():
    w = W.make("cop_big", [300] * 3 + [1] * 300, [100] * 3 + [1] * 300, 16, 64, "bf16", seed=47)
    s = MlaDecodeStep(w, device=DEV)
    s.populate()
    s.absorb()
    s.plan()
    s.decode_planned()
    s.combine_out_proj()
    assert_close(to_f64(s.out), ref_out(w), "bf16", "combine_out_proj, 600 rows")


# ---------------------------------------------------------------------------
# tensor-core tiles of 128 (row, head) rows: 128 heads, or prefill chunks
# ---------------------------------------------------------------------------

TC_CASES = {
    "h128_bs64": lambda: W.make("tc_h128", [1, 31, 32, 33, 64, 65, 200], [1] * 7, 128, 64, "bf16", seed=61),
    "h128_bs16": lambda: W.make("tc_h128_16", [5, 40, 129], [1] * 3, 128, 16, "bf16", seed=62),
    "h64_bs32": lambda: W.make("tc_h64_32", [70, 2, 97], [1] * 3, 64, 32, "bf16", seed=63),
    "prefill_h16": lambda: W.make("tc_pf16", [300, 77, 40], [120, 9, 40], 16, 64, "bf16", seed=64),
    "prefill_h32_mixed": lambda: W.make("tc_pf32", [150, 10, 64, 1], [37, 10, 1, 1], 32, 64, "bf16", seed=65),
    "bad_and_empty": lambda: W.make("tc_empty", [0, 90, 0, 3], [0, 12, 0, 3], 16, 64, "bf16", seed=66),
}


@pytest.mark.parametrize("name", sorted(TC_CASES))
@pytest.mark.parametrize("num_ctas", [2, 7, 0, 500])
def test_tensor_core_tiles(name, num_ctas):
    w = TC_CASES[name]()
    s = MlaDecodeStep(w, device=DEV, num_ctas=num_ctas)
    s.populate()
    s.absorb()
    s.plan()
    s.o_lat.fill_(float("nan"))
    s.decode_combine()                                  # fused merge
    torch.cuda.synchronize()
    assert s.device_status()[0][0] == 0
    fused = to_f64(s.o_lat)
    ref = ref_o_lat_from(w, to_f64(s.cache), to_f64(s.q_abs))
    empty = np.isnan(ref).all(axis=(1, 2))
    assert np.all(fused[empty] == 0)
    assert_close(fused, ref, "bf16", f"tc fused o_lat {name}")
    s.decode_planned()                                  # partials + merge kernel
    s.combine()
    np.testing.assert_allclose(to_f64(s.o_lat), fused, rtol=0, atol=1e-5)
    s.combine_out_proj()                                # merge inside the projection
    assert_close(to_f64(s.out), ref_out(w), "bf16", f"tc out {name}")


def test_tensor_core_merge_of_many_splits():
    # 41 q-blocks over 40 CTA pairs keeps the merge inside the decode kernel;
    # the 32,000-token row (500 tiles, ~14 per pair) is cut into ~37 parts,
    # more than one pass of staged merge weights
    lens = [32000] + [1] * 38 + [100, 64]
    w = W.make("tc_many", lens, [1] * len(lens), 128, 64, "bf16", seed=67)
    s = MlaDecodeStep(w, device=DEV, num_ctas=80)
    s.populate()
    s.absorb()
    s.plan()
    s.o_lat.fill_(float("nan"))
    s.decode_combine()
    torch.cuda.synchronize()
    assert s.device_status()[0][0] == 0
    fused = to_f64(s.o_lat)
    ref = ref_o_lat_from(w, to_f64(s.cache), to_f64(s.q_abs))
    assert_close(fused, ref, "bf16", "tc fused o_lat, 37 parts")
    s.decode_planned()
    s.combine()
    np.testing.assert_allclose(to_f64(s.o_lat), fused, rtol=0, atol=1e-5)


# ---------------------------------------------------------------------------
# projections for many rows (tcgen05 kernels from 256 rows on)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("rows,heads", [(255, 16), (256, 16), (300, 16), (1000, 32), (257, 128)])
def test_out_proj_many_rows(rows, heads):
    rng = np.random.default_rng(800 + rows + heads)
    cfg = L.make_config(heads, 64, "bf16")
    # latent outputs are convex combinations of normalised rows: |o| well below 1
    o_lat = torch.from_numpy(0.25 * rng.standard_normal((rows, heads, 512)).astype(np.float32)).to(DEV)
    w = W.round_to_dtype(rng.standard_normal((heads, 512, 128)).astype(np.float32) / np.sqrt(512), "bf16")
    W_uv = torch.from_numpy(w).to(DEV).to(torch.bfloat16)
    out = torch.full((rows, heads, 128), float("nan"), dtype=torch.bfloat16, device=DEV)
    L.mla_out_proj(cfg, o_lat, W_uv, out)
    torch.cuda.synchronize()
    ref = O.out_proj(to_f64(o_lat), w.astype(np.float64))
    assert_close(to_f64(out), ref, "bf16", f"out_proj {rows} rows x {heads} heads")


@pytest.mark.parametrize("rows,heads", [(255, 16), (256, 16), (300, 16), (1000, 32), (257, 128)])
def test_absorb_many_rows(rows, heads):
    rng = np.random.default_rng(900 + rows + heads)
    cfg = L.make_config(heads, 64, "bf16")
    qn = W.round_to_dtype(rng.standard_normal((rows, heads, 128)).astype(np.float32), "bf16")
    qp = W.round_to_dtype(rng.standard_normal((rows, heads, 64)).astype(np.float32), "bf16")
    wk = W.round_to_dtype(rng.standard_normal((heads, 512, 128)).astype(np.float32) / np.sqrt(512), "bf16")
    pos = rng.integers(0, 32768, size=rows).astype(np.int32)
    t = lambda a: torch.from_numpy(a).to(DEV).to(torch.bfloat16)
    q_abs = torch.full((rows, heads, 576), float("nan"), dtype=torch.bfloat16, device=DEV)
    L.mla_absorb_q(cfg, t(qn), t(qp), torch.from_numpy(pos).to(DEV), t(wk), q_abs)
    torch.cuda.synchronize()
    ref = O.absorb_q(qn, qp, pos, wk, cfg.rope_base)
    assert_close(to_f64(q_abs), ref, "bf16", f"absorb {rows} rows x {heads} heads")
