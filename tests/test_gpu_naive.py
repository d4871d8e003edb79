"""GPU parity of the pages' other two forms (full key/value cache; latent cache
re-expanded every step) against the fp64 oracle, through the C ABI.

mla_naive_cache_write and mla_latent_expand are checked row by row against
the oracle's naive_kv_rows, mla_naive_decode on the GPU's own expanded rows
against expanded_attention, and all three forms end to end against the naive
form from raw inputs.
"""

import numpy as np
import pytest
import torch

from _helpers import assert_close, bf16_ulp, ref_cache_rows, ref_out, to_f64
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


CASES = {
    "ragged_tails": lambda: W.make("nv_tails", [1, 63, 64, 65, 127, 128, 129, 300], [1] * 8, 16,
                                   64, "bf16", seed=51, extra_blocks=2),
    "bs16_h32": lambda: W.make("nv_bs16", [5, 40, 200], [1] * 3, 32, 16, "bf16", seed=52),
    "bs32_h128": lambda: W.make("nv_h128", [33, 97], [1, 1], 128, 32, "bf16", seed=53),
    "prefill": lambda: W.make("nv_prefill", [150, 64, 20], [40, 1, 20], 16, 64, "bf16", seed=54),
    "empty_seq": lambda: W.make("nv_empty", [0, 5, 0, 70], [0, 1, 0, 1], 16, 64, "bf16", seed=55),
}


def _slots_of(w, b):
    t = np.arange(int(w.seq_lens[b]))
    return w.block_table[b][t // w.block_size].astype(np.int64) * w.block_size + t % w.block_size


def _naive_step(name):
    w = CASES[name]()
    s = MlaDecodeStep(w, device=DEV)
    s.naive_setup()
    return w, s


@pytest.mark.parametrize("name", sorted(CASES))
def test_naive_cache_write_rows_and_placement(name):
    w, s = _naive_step(name)
    s.kv_naive.view(torch.int16).fill_(0x7FC1)              # a NaN bit pattern
    s.naive_populate()
    s.populate()                                            # the latent rows it expands
    torch.cuda.synchronize()
    assert L.mla_get_device_status(s.naive_ws)[0] == 0
    bits = s.kv_naive.view(torch.int16).cpu().numpy().reshape(-1, w.num_heads, 320)
    written = np.zeros(bits.shape[0], dtype=bool)
    written[w.slot_mapping] = True
    assert np.all(bits[~written] == 0x7FC1), "bytes outside the slots changed"
    got = to_f64(s.kv_naive).reshape(-1, w.num_heads, 320)[w.slot_mapping]
    # the latent rows themselves are pinned by the cache-write tests; here the
    # expansion of those bf16 rows by the bf16 weights is one rounding to bf16
    # of the exact product (fp32 accumulation over 512 terms adds ~1e-5)
    lat = to_f64(s.cache).reshape(-1, 576)[w.slot_mapping]
    ref = O.naive_kv_rows(lat[:, :512], lat[:, 512:], to_f64(s.W_uk), to_f64(s.W_uv))
    assert np.array_equal(got[:, :, 128:192], ref[:, :, 128:192]), "rope key not copied exactly"
    err = np.abs(got - ref)
    assert np.all(err <= bf16_ulp(ref) + 1e-4), f"{name}: beyond 1 bf16 ulp, max {err.max():.3g}"
    # and against the oracle from the raw inputs, at the rows' own scale
    rows = ref_cache_rows(w)
    raw = O.naive_kv_rows(rows[:, :512], rows[:, 512:], w.W_uk, w.W_uv)
    rel = np.linalg.norm(got - raw) / np.linalg.norm(raw)
    assert rel <= 5e-3, f"{name}: rel-L2 {rel:.3g} against the raw-input oracle"


@pytest.mark.parametrize("name", ["ragged_tails", "bs16_h32", "bs32_h128"])
def test_latent_expand_equals_the_naive_cache_write(name):
    # version 2 re-expands the latent cache into exactly the rows version 1 caches
    w, s = _naive_step(name)
    s.populate()
    s.naive_populate()
    v1 = s.kv_naive.clone()
    s.kv_naive.view(torch.int16).fill_(0x7FC1)
    s.latent_expand()
    torch.cuda.synchronize()
    assert L.mla_get_device_status(s.naive_ws)[0] == 0
    slots = np.concatenate([_slots_of(w, b) for b in range(w.batch)])
    a = v1.view(torch.int16).reshape(-1, w.num_heads, 320)[torch.from_numpy(slots).to(DEV)]
    b = s.kv_naive.view(torch.int16).reshape(-1, w.num_heads, 320)[torch.from_numpy(slots).to(DEV)]
    assert torch.equal(a, b)
    # the two-part form: weights prepared once (into a fresh workspace), then
    # expanded twice with them -- the same rows, bit for bit
    ws2 = torch.zeros_like(s.naive_ws)
    L.mla_latent_expand_prepare(s.cfg, s.W_uk, s.W_uv, ws2)
    for _ in range(2):
        s.kv_naive.view(torch.int16).fill_(0x7FC1)
        L.mla_latent_expand_prepared(s.cfg, s.cache, s.block_table, s.seq_lens, s.kv_naive, ws2)
        torch.cuda.synchronize()
        assert L.mla_get_device_status(ws2)[0] == 0
        c = s.kv_naive.view(torch.int16).reshape(-1, w.num_heads, 320)[torch.from_numpy(slots).to(DEV)]
        assert torch.equal(a, c)


@pytest.mark.parametrize("name", sorted(CASES))
def test_naive_decode_vs_expanded_oracle(name):
    w, s = _naive_step(name)
    s.naive_populate()
    s.out_naive.fill_(float("nan"))
    s.naive_decode()
    torch.cuda.synchronize()
    assert L.mla_get_device_status(s.naive_ws)[0] == 0
    kv = to_f64(s.kv_naive).reshape(-1, w.num_heads, 320)
    q = np.concatenate([w.q_nope.astype(np.float64),
                        O.rope(w.q_pe, w.q_positions, w.rope_base)], -1)
    ref = np.zeros((w.num_q, w.num_heads, 128))
    for b in range(w.batch):
        qr = w.q_range(b)
        if qr.stop == qr.start:
            continue
        ref[qr] = O.expanded_attention(kv[_slots_of(w, b)], q[qr], w.q_positions[qr],
                                       w.softmax_scale)
    assert_close(to_f64(s.out_naive), ref, "bf16", f"naive decode {name}")


@pytest.mark.parametrize("name", ["ragged_tails", "prefill", "bs32_h128"])
def test_three_forms_agree_with_the_naive_oracle(name):
    w, s = _naive_step(name)
    s.populate()
    absorbed = to_f64(s.step())                 # version 3
    s.naive_populate()
    s.naive_decode()
    full = to_f64(s.out_naive)                  # version 1
    s.kv_naive.view(torch.int16).fill_(0x7FC1)
    s.latent_expand()
    s.naive_decode()
    latent = to_f64(s.out_naive)                # version 2
    torch.cuda.synchronize()
    ref = ref_out(w)
    for got, form in ((absorbed, "absorbed"), (full, "full K/V"), (latent, "latent re-expanded")):
        assert_close(got, ref, "bf16", f"{form} {name}")


def test_v2lite_shapes_every_seq_len():
    for L_ in (1, 256, 1024):
        w = W.v2lite(L_)
        s = MlaDecodeStep(w, device=DEV)
        s.naive_setup()
        s.populate()
        s.latent_expand()
        s.naive_decode()
        torch.cuda.synchronize()
        assert_close(to_f64(s.out_naive), ref_out(w), "bf16", f"v2lite L={L_} latent re-expanded")


def test_bad_block_is_reported_and_skipped():
    w = W.make("nv_bad", [200, 100], [1, 1], 16, 64, "bf16", seed=56)
    s = MlaDecodeStep(w, device=DEV)
    s.naive_setup()
    s.naive_populate()
    s.block_table[0, 1] = w.num_blocks + 3
    s.naive_decode()
    st, bits = L.mla_get_device_status(s.naive_ws)
    assert st == 6 and bits & L.DEV_BAD_BLOCK
    got = to_f64(s.out_naive)
    assert np.all(np.isfinite(got))
    assert_close(got[1:2], ref_out(w, seqs=[1])[1:2], "bf16", "other sequence")


# ---------------------------------------------------------------------------
# mla_naive_prefill: the same attention in 64-row tensor-core tiles
# ---------------------------------------------------------------------------

PREFILL_CASES = dict(CASES)
PREFILL_CASES.update({
    "multi_tile_bs16": lambda: W.make("pf_mt16", [300, 70, 129], [200, 64, 129], 16, 16, "bf16",
                                      seed=57),
    "multi_tile_h32": lambda: W.make("pf_mt32", [600, 5], [260, 5], 32, 64, "bf16", seed=58),
})


def _expanded_ref(w, s):
    kv = to_f64(s.kv_naive).reshape(-1, w.num_heads, 320)
    q = np.concatenate([w.q_nope.astype(np.float64),
                        O.rope(w.q_pe, w.q_positions, w.rope_base)], -1)
    ref = np.zeros((w.num_q, w.num_heads, 128))
    for b in range(w.batch):
        qr = w.q_range(b)
        if qr.stop == qr.start:
            continue
        ref[qr] = O.expanded_attention(kv[_slots_of(w, b)], q[qr], w.q_positions[qr],
                                       w.softmax_scale)
    return ref


@pytest.mark.parametrize("name", sorted(PREFILL_CASES))
def test_naive_prefill_vs_expanded_oracle_and_decode(name):
    w = PREFILL_CASES[name]()
    s = MlaDecodeStep(w, device=DEV)
    s.naive_setup()
    s.naive_populate()
    s.out_naive.fill_(float("nan"))
    s.naive_prefill()
    torch.cuda.synchronize()
    assert L.mla_get_device_status(s.naive_ws)[0] == 0
    first = s.out_naive.clone()
    got = to_f64(first)
    assert_close(got, _expanded_ref(w, s), "bf16", f"naive prefill {name}")
    # the same rows through the split CUDA-core path
    s.naive_decode()
    torch.cuda.synchronize()
    assert_close(got, to_f64(s.out_naive), "bf16", f"prefill vs decode {name}")
    # and a repeated launch agrees bit for bit
    s.naive_prefill()
    torch.cuda.synchronize()
    assert torch.equal(s.out_naive, first)


def test_naive_prefill_interleaved_rope_and_bad_sequence():
    w = W.make("pf_ri", [150, 64, 20], [40, 1, 20], 16, 64, "bf16", seed=59)
    s = MlaDecodeStep(w, device=DEV, rope_interleaved=True)
    s.naive_setup()
    s.naive_populate()
    s.naive_prefill()
    torch.cuda.synchronize()
    kv = to_f64(s.kv_naive).reshape(-1, w.num_heads, 320)
    q = np.concatenate([w.q_nope.astype(np.float64),
                        O.rope(w.q_pe, w.q_positions, w.rope_base, interleaved=True)], -1)
    ref = np.zeros((w.num_q, w.num_heads, 128))
    for b in range(w.batch):
        qr = w.q_range(b)
        ref[qr] = O.expanded_attention(kv[_slots_of(w, b)], q[qr], w.q_positions[qr],
                                       w.softmax_scale)
    assert_close(to_f64(s.out_naive), ref, "bf16", "naive prefill, interleaved RoPE")
    # a query chunk longer than its sequence: status set, its rows zero
    s.seq_lens[1] = 0
    s.out_naive.fill_(float("nan"))
    s.naive_prefill()
    st, bits = L.mla_get_device_status(s.naive_ws)
    assert st == 7 and bits & L.DEV_BAD_SEQ
    got = to_f64(s.out_naive)
    assert np.all(got[w.q_range(1)] == 0)
    assert_close(got[w.q_range(0)], ref[w.q_range(0)], "bf16", "other sequence")


def test_hybrid_step_on_the_mixed_batch_sampled():
    # prefill sequences in the expanded form on tensor cores, decode rows
    # absorbed, concurrently; checked on sampled sequences and heads
    from _helpers import ref_out
    w = W.mixed()
    s = MlaDecodeStep(w, device=DEV)
    s.populate(include_new=False)
    s.hybrid_setup()
    s.out_naive.fill_(float("nan"))
    side = torch.cuda.Stream()
    out = to_f64(s.hybrid_step(side))
    torch.cuda.synchronize()
    (st1, _), (st2, _) = s.device_status()
    assert st1 == 0 and st2 == 0
    assert L.mla_get_device_status(s.naive_ws)[0] == 0
    assert not np.isnan(out).any()
    seqs, heads = [1, 3, 4, 63], [0, 9, 15]
    ref = ref_out(w, seqs=seqs, heads=heads)
    rows = np.concatenate([np.arange(w.q_range(b).start, w.q_range(b).stop) for b in seqs])
    assert_close(out[:, heads][rows], ref[rows], "bf16", "hybrid mixed step")
